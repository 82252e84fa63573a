// lq_aux.cu -- the smaller kernels of the library: dequantization, the
// gate/up row interleave, a plain-load matvec used where the streaming
// kernel's layout conditions do not hold, MoE routing/grouping and the MoE
// weighted combine.
#include "lq_codec.cuh"
#include "lq_internal.h"

namespace lq {
namespace {

__device__ __forceinline__ uint32_t ldg_u16(const uint8_t* p) {
    return __ldg(reinterpret_cast<const unsigned short*>(p));
}

// ---------------------------------------------------------------- dequant
// One thread per 32 consecutive weights of a row (one Q4_K/Q6_K sub-block
// pair half or one Q8_0 block), reading the block with 2-byte loads.
__global__ void dequant_kernel(int fmt, const uint8_t* __restrict__ W, int64_t rows,
                               int64_t cols, float* __restrict__ out) {
    const int64_t per_row = cols / 32;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= rows * per_row) return;
    const int64_t r = idx / per_row;
    const int64_t c32 = idx % per_row;          // 32-weight chunk within the row
    const int64_t rb = cols / block_elems_of(fmt) * block_bytes_of(fmt);
    const uint8_t* row = W + r * rb;
    float* o = out + r * cols + c32 * 32;
    if (fmt == FMT_Q8_0) {
        const uint8_t* bp = row + c32 * 34;
        const float d = half_bits_to_float(ldg_u16(bp));
        for (int i = 0; i < 32; i += 2) {
            const uint32_t v = ldg_u16(bp + 2 + i);
            o[i] = d * (float)(int8_t)(v & 0xFF);
            o[i + 1] = d * (float)(int8_t)(v >> 8);
        }
    } else if (fmt == FMT_Q4_K) {
        const int64_t blk = c32 / 8;
        const int j = (int)(c32 % 8);               // sub-block
        const uint8_t* bp = row + blk * 144;
        const uint32_t dw = ldg_u16(bp) | (ldg_u16(bp + 2) << 16);
        const uint32_t s0 = ldg_u16(bp + 4) | (ldg_u16(bp + 6) << 16);
        const uint32_t s1 = ldg_u16(bp + 8) | (ldg_u16(bp + 10) << 16);
        const uint32_t s2 = ldg_u16(bp + 12) | (ldg_u16(bp + 14) << 16);
        float2 dsc, dm;
        q4k_group_scales(dw, s0, s1, s2, j >> 1, dsc, dm);
        const float sc = (j & 1) ? dsc.y : dsc.x;
        const float mm = (j & 1) ? dm.y : dm.x;
        const uint8_t* qs = bp + 16 + 32 * (j >> 1);
        for (int l = 0; l < 32; l += 2) {
            const uint32_t v = ldg_u16(qs + l);
            const uint32_t q0 = (j & 1) ? ((v >> 4) & 15) : (v & 15);
            const uint32_t q1 = (j & 1) ? ((v >> 12) & 15) : ((v >> 8) & 15);
            o[l] = q4k_weight(sc, mm, (float)q0);
            o[l + 1] = q4k_weight(sc, mm, (float)q1);
        }
    } else {  // Q6_K: chunk c32 = 32 weights = quarter q of half h
        const int64_t blk = c32 / 8;
        const int hq = (int)(c32 % 8), h = hq >> 2, q = hq & 3;
        const uint8_t* bp = row + blk * 210;
        const float d = half_bits_to_float(ldg_u16(bp + 208));
        const uint8_t* ql = bp + 64 * h + (q & 1) * 32;
        const uint8_t* qh = bp + 128 + 32 * h;
        for (int l = 0; l < 32; l += 2) {
            const uint32_t lv = ldg_u16(ql + l), hv = ldg_u16(qh + l);
            for (int e = 0; e < 2; ++e) {
                const uint32_t lb = (lv >> (8 * e)) & 0xFF, hb = (hv >> (8 * e)) & 0xFF;
                const uint32_t nib = q < 2 ? (lb & 15) : (lb >> 4);
                const int code = (int)(nib | (((hb >> (2 * q)) & 3) << 4)) - 32;
                const int sidx = 8 * h + 2 * q + (l + e) / 16;
                const int sc = (int8_t)(ldg_u16(bp + 192 + (sidx & ~1)) >> (8 * (sidx & 1)));
                o[l + e] = (d * (float)sc) * (float)code;
            }
        }
    }
}

// ---------------------------------------------------------------- interleave
__global__ void interleave_rows_kernel(const uint8_t* __restrict__ Wg,
                                       const uint8_t* __restrict__ Wu, int64_t rows,
                                       int64_t rb, uint8_t* __restrict__ out) {
    // 2-byte units; rb is even for every format
    const int64_t n16 = rb / 2;
    const int64_t total = rows * 2 * n16;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t orow = i / n16, c = i % n16;
        const int64_t r = orow >> 1;
        const uint8_t* src = ((orow & 1) ? Wu : Wg) + r * rb;
        reinterpret_cast<uint16_t*>(out + orow * rb)[c] =
            __ldg(reinterpret_cast<const unsigned short*>(src) + c);
    }
}

// ---------------------------------------------------------------- direct matvec
// One warp per output (row or gate/up pair) and batch chunk; lanes over
// 32-weight chunks; weights dequantized exactly and FMA'd with x read from
// global memory.  Per-chunk partials, fixed-order lane sum + butterfly.
__device__ float direct_chunk(int fmt, const uint8_t* row, int64_t c32, const float* xrow) {
    float acc = 0.f;
    if (fmt == FMT_Q8_0) {
        const uint8_t* bp = row + c32 * 34;
        const float d = half_bits_to_float(ldg_u16(bp));
        for (int i = 0; i < 32; i += 2) {
            const uint32_t v = ldg_u16(bp + 2 + i);
            acc = fmaf(d * (float)(int8_t)(v & 0xFF), __ldg(xrow + c32 * 32 + i), acc);
            acc = fmaf(d * (float)(int8_t)(v >> 8), __ldg(xrow + c32 * 32 + i + 1), acc);
        }
    } else if (fmt == FMT_Q4_K) {
        const int64_t blk = c32 / 8;
        const int j = (int)(c32 % 8);
        const uint8_t* bp = row + blk * 144;
        const uint32_t dw = ldg_u16(bp) | (ldg_u16(bp + 2) << 16);
        const uint32_t s0 = ldg_u16(bp + 4) | (ldg_u16(bp + 6) << 16);
        const uint32_t s1 = ldg_u16(bp + 8) | (ldg_u16(bp + 10) << 16);
        const uint32_t s2 = ldg_u16(bp + 12) | (ldg_u16(bp + 14) << 16);
        float2 dsc, dm;
        q4k_group_scales(dw, s0, s1, s2, j >> 1, dsc, dm);
        const float sc = (j & 1) ? dsc.y : dsc.x;
        const float mm = (j & 1) ? dm.y : dm.x;
        const uint8_t* qs = bp + 16 + 32 * (j >> 1);
        const int64_t col0 = blk * 256 + 32 * j;
        for (int l = 0; l < 32; l += 2) {
            const uint32_t v = ldg_u16(qs + l);
            const uint32_t q0 = (j & 1) ? ((v >> 4) & 15) : (v & 15);
            const uint32_t q1 = (j & 1) ? ((v >> 12) & 15) : ((v >> 8) & 15);
            acc = fmaf(q4k_weight(sc, mm, (float)q0), __ldg(xrow + col0 + l), acc);
            acc = fmaf(q4k_weight(sc, mm, (float)q1), __ldg(xrow + col0 + l + 1), acc);
        }
    } else {
        const int64_t blk = c32 / 8;
        const int hq = (int)(c32 % 8), h = hq >> 2, q = hq & 3;
        const uint8_t* bp = row + blk * 210;
        const float d = half_bits_to_float(ldg_u16(bp + 208));
        const uint8_t* ql = bp + 64 * h + (q & 1) * 32;
        const uint8_t* qh = bp + 128 + 32 * h;
        const int64_t col0 = blk * 256 + 128 * h + 32 * q;
        for (int l = 0; l < 32; l += 2) {
            const uint32_t lv = ldg_u16(ql + l), hv = ldg_u16(qh + l);
            for (int e = 0; e < 2; ++e) {
                const uint32_t lb = (lv >> (8 * e)) & 0xFF, hb = (hv >> (8 * e)) & 0xFF;
                const uint32_t nib = q < 2 ? (lb & 15) : (lb >> 4);
                const int code = (int)(nib | (((hb >> (2 * q)) & 3) << 4)) - 32;
                const int sidx = 8 * h + 2 * q + (l + e) / 16;
                const int sc = (int8_t)(ldg_u16(bp + 192 + (sidx & ~1)) >> (8 * (sidx & 1)));
                acc = fmaf((d * (float)sc) * (float)code, __ldg(xrow + col0 + l + e), acc);
            }
        }
    }
    return acc;
}

__device__ float direct_row(int fmt, const uint8_t* row, int64_t cols, const float* xrow,
                            int lane) {
    const int64_t nchunk = cols / 32;
    float acc = 0.f;
    for (int64_t c = lane; c < nchunk; c += 32) acc += direct_chunk(fmt, row, c, xrow);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    return acc;
}

__global__ void direct_mv_kernel(Seg S, int64_t cols, int maxb) {
    const int warp = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp >= S.nout) return;
    int nval = S.bcnt ? (*S.bcnt - S.b0) : S.nbatch;
    nval = nval > maxb ? maxb : nval;
    const int boff = (S.boff ? *S.boff : 0) + S.b0;
    const int64_t rb = cols / block_elems_of(S.fmt) * block_bytes_of(S.fmt);
    for (int b = 0; b < nval; ++b) {
        const int rho = boff + b;
        const float* xrow = S.x + (int64_t)(S.xmap ? S.xmap[rho] : rho) * cols;
        float v;
        if (S.mode == MODE_PLAIN) {
            v = seg_out(S.cap, direct_row(S.fmt, S.w + (int64_t)warp * rb, cols, xrow, lane));
        } else {
            const uint8_t* rg = S.mode == MODE_PAIR_INTERLEAVED ? S.w + (int64_t)(2 * warp) * rb
                                                               : S.w + (int64_t)warp * rb;
            const uint8_t* ru = S.mode == MODE_PAIR_INTERLEAVED ? rg + rb : S.w2 + (int64_t)warp * rb;
            const float g = direct_row(S.fmt, rg, cols, xrow, lane);
            const float u = direct_row(S.fmt, ru, cols, xrow, lane);
            v = act_eval(S.act, g) * u;
        }
        if (lane == 0) S.y[(int64_t)rho * S.ld_y + warp] = v;
    }
}

// ---------------------------------------------------------------- x transforms
// RMS-norm of one row per CTA (256 threads): out = (x * r) * w with
// r = 1 / sqrt(mean(x^2) + eps), the sum of squares in a fixed order (per
// thread over its columns, a butterfly over the warp, the warps in order).
// out may be x itself: every thread reads its own columns again after the
// barrier that ends the sum, then writes them.
__global__ void rmsnorm_kernel(const float* x, const float* __restrict__ w, float eps, float* out, int64_t n) {
    __shared__ float red[8];
    const float* xr = x + (int64_t)blockIdx.x * n;
    float* orow = out + (int64_t)blockIdx.x * n;
    float ss = 0.f;
    for (int64_t j = threadIdx.x; j < n; j += 256) ss = fmaf(xr[j], xr[j], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < 8; ++i) t += red[i];
    const float r = 1.0f / sqrtf(t / (float)n + eps);
    for (int64_t j = threadIdx.x; j < n; j += 256) orow[j] = (xr[j] * r) * __ldg(w + j);
}

// h[i] = act(g_i) * u_i of n (g, u) pairs.
__global__ void act_pairs_kernel(const float* __restrict__ gu, float* __restrict__ h, int64_t n, int act) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        h[i] = act_eval(act, gu[2 * i]) * gu[2 * i + 1];
}

// ---------------------------------------------------------------- MoE routing
// One CTA: router logits (one warp per (token, expert) dot product,
// deterministic), softmax over the experts, top-k by repeated maximum with
// the lower index winning ties, weights renormalised by the selected sum
// (dotLLM PR #320, MoE commit) or, with ws.norm = 0, the selected softmax
// probabilities as they are (norm_topk_prob = false, the Qwen-MoE commit).
// With a shared-expert gate vector g, also sgate[t] = sigmoid(g . x_t), one
// warp per token.  Then groups the (token, slot) pairs by expert in token
// order.
__device__ __forceinline__ float warp_dot(const float* __restrict__ a, const float* __restrict__ b, int64_t n,
                                          int lane) {
    float acc = 0.f;
    for (int64_t j = lane; j < n; j += 32) acc = fmaf(__ldg(a + j), __ldg(b + j), acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    return acc;
}

__global__ void moe_route_kernel(const float* __restrict__ R, int E, int64_t hidden,
                                 const float* __restrict__ X, int ntok, int topk,
                                 const float* __restrict__ gvec, MoeWs ws) {
    extern __shared__ float sh[];
    float* logits = sh;                          // ntok * E
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int p = warp; p < ntok * E; p += nw) {
        const int t = p / E, e = p % E;
        const float acc = warp_dot(R + (int64_t)e * hidden, X + (int64_t)t * hidden, hidden, lane);
        if (lane == 0) logits[p] = acc;
    }
    if (gvec) {
        for (int t = warp; t < ntok; t += nw) {
            const float z = warp_dot(gvec, X + (int64_t)t * hidden, hidden, lane);
            if (lane == 0) ws.sgate[t] = 1.0f / (1.0f + expf(-z));
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < ntok; t += blockDim.x) {
        const float* l = logits + t * E;
        float mx = l[0];
        for (int e = 1; e < E; ++e) mx = fmaxf(mx, l[e]);
        float z = 0.f;
        for (int e = 0; e < E; ++e) z += expf(l[e] - mx);
        uint32_t taken[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // up to 256 experts
        float sel = 0.f;
        for (int k = 0; k < topk; ++k) {
            int best = -1;
            float bp = 0.f;
            for (int e = 0; e < E; ++e) {
                if (taken[e >> 5] & (1u << (e & 31))) continue;
                const float p = expf(l[e] - mx) / z;
                if (best < 0 || p > bp) {
                    best = e;
                    bp = p;
                }
            }
            taken[best >> 5] |= 1u << (best & 31);
            ws.idx[t * topk + k] = best;
            ws.w[t * topk + k] = bp;
            sel += bp;
        }
        if (ws.norm)
            for (int k = 0; k < topk; ++k) ws.w[t * topk + k] = ws.w[t * topk + k] / sel;
    }
    __syncthreads();
    // grouping: expert e's slots in token order (single thread: ntok*topk small)
    if (threadIdx.x == 0) {
        int off = 0;
        for (int e = 0; e < E; ++e) {
            ws.grp_off[e] = off;
            int c = 0;
            for (int s = 0; s < ntok * topk; ++s)
                if (ws.idx[s] == e) {
                    ws.tok_of[off + c] = s / topk;
                    ws.slot_row[s] = off + c;
                    ++c;
                }
            ws.grp_cnt[e] = c;
            off += c;
        }
    }
}

// Y[t] = sum_k w[t][k] * ye[row of (t,k)], k in order, plus the shared
// experts' outputs summed in expert order and scaled by the gate (sgate[t],
// or 1 without a gate vector).
__global__ void moe_combine_kernel(const float* __restrict__ ye, int64_t hidden, int ntok,
                                   int topk, MoeWs ws, bool gated, float* __restrict__ Y) {
    const int64_t total = (int64_t)ntok * hidden;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / hidden);
        const int64_t o = i % hidden;
        float acc = 0.f;
        for (int k = 0; k < topk; ++k) {
            const int s = t * topk + k;
            acc = fmaf(ws.w[s], ye[(int64_t)ws.slot_row[s] * hidden + o], acc);
        }
        if (ws.nshared > 0) {
            float sum = 0.f;
            for (int e = 0; e < ws.nshared; ++e) sum += ws.ysh[((int64_t)e * ntok + t) * hidden + o];
            acc = gated ? fmaf(ws.sgate[t], sum, acc) : acc + sum;
        }
        Y[i] = acc;
    }
}

}  // namespace

// Failure-detection probe: waits on an mbarrier that nothing will complete,
// with the same bounded wait the streaming kernel uses; the wait runs out
// after timeout_ns and the kernel records STATUS_TIMEOUT and returns.
__global__ void timeout_probe_kernel(uint64_t timeout_ns, unsigned* status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0, timeout_ns))
        record_status(status, STATUS_TIMEOUT);
}

cudaError_t launch_timeout_probe(uint64_t timeout_ns, unsigned* status, cudaStream_t st) {
    timeout_probe_kernel<<<1, 32, 0, st>>>(timeout_ns, status);
    return cudaGetLastError();
}

cudaError_t launch_dequant(int fmt, const uint8_t* W, int64_t rows, int64_t cols, float* out,
                           cudaStream_t st) {
    const int64_t n = rows * (cols / 32);
    const int tpb = 256;
    dequant_kernel<<<(unsigned)((n + tpb - 1) / tpb), tpb, 0, st>>>(fmt, W, rows, cols, out);
    return cudaGetLastError();
}

cudaError_t launch_interleave(const uint8_t* Wg, const uint8_t* Wu, int64_t rows, int64_t rb,
                              uint8_t* out, cudaStream_t st) {
    const int64_t n = rows * rb;   // 2-byte units = rows * 2 * rb / 2
    int64_t blocks = (n + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    interleave_rows_kernel<<<(unsigned)blocks, 256, 0, st>>>(Wg, Wu, rows, rb, out);
    return cudaGetLastError();
}

cudaError_t launch_direct(const Seg& S, int64_t cols, int maxb, cudaStream_t st) {
    const int64_t threads = (int64_t)S.nout * 32;
    const int tpb = 256;
    direct_mv_kernel<<<(unsigned)((threads + tpb - 1) / tpb), tpb, 0, st>>>(S, cols, maxb);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const float* x, const float* w, float eps, float* out, int rows, int64_t n,
                           cudaStream_t st) {
    rmsnorm_kernel<<<(unsigned)rows, 256, 0, st>>>(x, w, eps, out, n);
    return cudaGetLastError();
}

cudaError_t launch_act_pairs(const float* gu, float* h, int64_t n, int act, cudaStream_t st) {
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    act_pairs_kernel<<<(unsigned)blocks, 256, 0, st>>>(gu, h, n, act);
    return cudaGetLastError();
}

cudaError_t launch_moe_route(const float* R, int E, int64_t hidden, const float* X, int ntok,
                             int topk, const float* sgate_vec, const MoeWs& ws, cudaStream_t st) {
    const size_t smem = (size_t)ntok * E * sizeof(float);
    moe_route_kernel<<<1, 1024, smem, st>>>(R, E, hidden, X, ntok, topk, sgate_vec, ws);
    return cudaGetLastError();
}

cudaError_t launch_moe_combine(const float* ye, int64_t hidden, int ntok, int topk,
                               const MoeWs& ws, float* Y, cudaStream_t st) {
    const int64_t n = (int64_t)ntok * hidden;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    moe_combine_kernel<<<(unsigned)blocks, 256, 0, st>>>(ye, hidden, ntok, topk, ws, ws.sgate != nullptr, Y);
    return cudaGetLastError();
}

}  // namespace lq
