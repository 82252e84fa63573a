// lq_stream.cu -- the streaming block-quantized matvec kernel.
//
// Computes y = W.x for batch rows of x (larql "Architecture -> Metal shader
// map": q4k_matvec / q6k_matvec rows of the Gemma 3 table; dotLLM PR #320:
// matmul_q8_0 GEMV), optionally fused with the gated-FFN activation over
// gate/up row pairs (larql Gemma 3 table, FFN gate+up + GEGLU rows;
// h = act(gate) * up) and over several weight matrices sharing one x in one
// launch (the mixed Q4_K/Q6_K QKV projection of the same table).
//
// GB300 design:
//  * Row tiles of W (contiguous bytes) stream into a ring of shared-memory
//    stages by 1-D bulk copies (cp.async.bulk, TMA engine) completing on
//    mbarriers; one elected thread issues them, nothing waits on HBM
//    latency but the barrier.  Unaligned or ragged tiles are copied by the
//    threads instead.
//  * Each thread owns a fixed 64/B-column slice of the row ("unit") for the
//    whole kernel and keeps the matching x values (B batch rows) in
//    registers; it dot-products that slice for R rows of every tile.
//  * Partials go to shared memory and are summed per output by a warp in a
//    fixed order (lane-strided, then xor butterfly; lane 0's value), so the
//    result is deterministic and independent of B.
//  * Every mbarrier wait is bounded in time; on expiry the CTA records
//    STATUS_TIMEOUT in the device status word, drains its own copies (also
//    bounded) and returns.
#include "lq_codec.cuh"
#include "lq_internal.h"

namespace lq {

namespace {

__device__ __forceinline__ int seg_of(const StreamParams& P, int t, int hint) {
    int s = hint;
    while (s + 1 < P.nseg && t >= P.seg[s + 1].tile0) ++s;
    return s;
}

// valid batch rows of a segment (0 = nothing to do)
__device__ __forceinline__ int seg_nval(const Seg& S, int B) {
    int n = S.bcnt ? (*S.bcnt - S.b0) : S.nbatch;
    return n < 0 ? 0 : (n > B ? B : n);
}

__device__ __forceinline__ int seg_boff(const Seg& S) { return (S.boff ? *S.boff : 0) + S.b0; }

__device__ __forceinline__ int64_t row_bytes(int fmt, int cols) {
    return (int64_t)(cols / block_elems_of(fmt)) * block_bytes_of(fmt);
}

// Geometry of tile t of segment S.
struct TileGeo {
    const uint8_t* src1;
    const uint8_t* src2;
    uint32_t bytes1, bytes2;    // bytes per copy (bytes2 = 0 unless two-matrix)
    uint32_t dst2;              // stage offset of the second copy
    int n_o;                    // outputs (rows or pairs) in this tile
    int o0;                     // first output index
    bool tma;                   // bulk-copyable
};

__device__ __forceinline__ TileGeo tile_geo(const StreamParams& P, const Seg& S, int t) {
    TileGeo g;
    const int64_t rb = row_bytes(S.fmt, P.cols);
    const int lt = t - S.tile0;
    const int opt = S.mode == MODE_PLAIN ? P.RT : P.RT / 2;
    g.o0 = lt * opt;
    g.n_o = min(opt, S.nout - g.o0);
    g.src2 = nullptr;
    g.bytes2 = 0;
    g.dst2 = 0;
    if (S.mode == MODE_PLAIN) {
        g.src1 = S.w + (int64_t)g.o0 * rb;
        g.bytes1 = (uint32_t)(g.n_o * rb);
    } else if (S.mode == MODE_PAIR_INTERLEAVED) {
        g.src1 = S.w + (int64_t)g.o0 * 2 * rb;
        g.bytes1 = (uint32_t)(2 * g.n_o * rb);
    } else {
        g.src1 = S.w + (int64_t)g.o0 * rb;
        g.bytes1 = (uint32_t)(g.n_o * rb);
        g.src2 = S.w2 + (int64_t)g.o0 * rb;
        g.bytes2 = g.bytes1;
        g.dst2 = (uint32_t)((P.RT / 2) * rb);
    }
    g.tma = ((reinterpret_cast<uintptr_t>(g.src1) | g.bytes1) & 15u) == 0;
    if (S.mode == MODE_PAIR_TWO)
        g.tma = g.tma && ((reinterpret_cast<uintptr_t>(g.src2) | g.bytes2 | g.dst2) & 15u) == 0;
    return g;
}

// next tile of this CTA at or after t (stepping by gridDim) whose segment
// has work; P.ntiles if none.
__device__ __forceinline__ int next_tile(const StreamParams& P, int t, int& hint, int B) {
    while (t < P.ntiles) {
        hint = seg_of(P, t, hint);
        if (seg_nval(P.seg[hint], B) > 0) return t;
        t += gridDim.x;
    }
    return P.ntiles;
}

// copy n bytes global -> shared with plain loads (any 2-byte alignment)
__device__ __forceinline__ void manual_copy(uint8_t* dst, const uint8_t* src, uint32_t n) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(src);
    if ((a & 3u) == 0 && (n & 3u) == 0) {
        const uint32_t* s = reinterpret_cast<const uint32_t*>(src);
        uint32_t* d = reinterpret_cast<uint32_t*>(dst);
        for (uint32_t i = threadIdx.x; i < n / 4; i += blockDim.x) d[i] = __ldg(s + i);
    } else {
        const uint16_t* s = reinterpret_cast<const uint16_t*>(src);
        uint16_t* d = reinterpret_cast<uint16_t*>(dst);
        for (uint32_t i = threadIdx.x; i < n / 2; i += blockDim.x) d[i] = __ldg(s + i);
    }
}

// 32-bit word at a 2-byte-aligned shared address
__device__ __forceinline__ uint32_t lds_u32_any(const uint8_t* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* q = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    return funnel_r(q[0], q[1], (uint32_t)(a & 3u) * 8u);
}

// n consecutive words starting at a 2-byte-aligned shared address
template <int N>
__device__ __forceinline__ void lds_words_any(const uint8_t* p, uint32_t* out) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* q = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    const uint32_t sh = (uint32_t)(a & 3u) * 8u;
    uint32_t w[N + 1];
#pragma unroll
    for (int i = 0; i <= N; ++i) w[i] = q[i];
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = funnel_r(w[i], w[i + 1], sh);
}

// x values of this thread's unit for one segment: xr[b][leaf][pair]
template <int B>
__device__ __forceinline__ void load_x(const StreamParams& P, const Seg& S, int G, int lam0,
                                       float2 (&xr)[B][4 / B][8]) {
    const int nval = seg_nval(S, B);
    const int boff = seg_boff(S);
#pragma unroll
    for (int b = 0; b < B; ++b) {
        const float* xrow = nullptr;
        if (b < nval) {
            const int rho = boff + b;
            const int xr_idx = S.xmap ? S.xmap[rho] : rho;
            xrow = S.x + (int64_t)xr_idx * P.cols;
        }
#pragma unroll
        for (int l = 0; l < 4 / B; ++l)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (xrow) {
                    xr[b][l][i].x = __ldg(xrow + leaf_col(S.fmt, G, lam0 + l, i, 0));
                    xr[b][l][i].y = __ldg(xrow + leaf_col(S.fmt, G, lam0 + l, i, 1));
                } else {
                    xr[b][l][i] = make_float2(0.f, 0.f);
                }
            }
    }
}

// Partial dot products of one row's unit (group G, leaves lam0..lam0+4/B-1)
// for B batch rows; leaves combined as (l0 + l1) + (l2 + l3).
template <int B>
__device__ __forceinline__ void unit_dot(int fmt, const uint8_t* row, int G, int lam0,
                                         const float2 (&xr)[B][4 / B][8], float (&part)[B]) {
    constexpr int NL = 4 / B;
    float lp[NL][B];
    if (fmt == FMT_Q4_K) {
        const uint8_t* bp = row + 144 * (G >> 2);
        const int g = G & 3;
        const uint4 hdr = *reinterpret_cast<const uint4*>(bp);
        float2 dsc, dm;
        q4k_group_scales(hdr.x, hdr.y, hdr.z, hdr.w, g, dsc, dm);
        const uint8_t* qs = bp + 16 + 32 * g + 8 * lam0;
#pragma unroll
        for (int l = 0; l < NL; ++l) {
            const uint2 w = *reinterpret_cast<const uint2*>(qs + 8 * l);
            q4k_leaf<B, NL>(w.x, w.y, dsc, dm, xr, l, lp[l]);
        }
    } else if (fmt == FMT_Q6_K) {
        const uint8_t* bp = row + 210 * (G >> 2);
        const int gm = G & 3, h = gm >> 1, l0 = 16 * (gm & 1);
        uint32_t A[NL], Bw[NL], H[NL], scw[2];
        lds_words_any<NL>(bp + 64 * h + l0 + 4 * lam0, A);
        lds_words_any<NL>(bp + 64 * h + 32 + l0 + 4 * lam0, Bw);
        lds_words_any<NL>(bp + 128 + 32 * h + l0 + 4 * lam0, H);
        lds_words_any<2>(bp + 192 + 8 * h, scw);           // scales 8h .. 8h+7
        const float d = half_bits_to_float(lds_u32_any(bp + 208));
        // quarter q uses scale byte 2q + l0/16 of the 8 loaded
        const uint32_t o = (uint32_t)(l0 >> 4);
        const int sc0 = (int8_t)(scw[0] >> (8 * o));
        const int sc1 = (int8_t)(scw[0] >> (8 * (2 + o)));
        const int sc2 = (int8_t)(scw[1] >> (8 * o));
        const int sc3 = (int8_t)(scw[1] >> (8 * (2 + o)));
        const float2 dsc01 = make_float2(d * (float)sc0, d * (float)sc1);
        const float2 dsc23 = make_float2(d * (float)sc2, d * (float)sc3);
#pragma unroll
        for (int l = 0; l < NL; ++l) q6k_leaf<B, NL>(A[l], Bw[l], H[l], dsc01, dsc23, xr, l, lp[l]);
    } else {
#pragma unroll
        for (int l = 0; l < NL; ++l) {
            const int lam = lam0 + l;
            const uint8_t* bp = row + 34 * (2 * G + (lam >> 1));
            const float d = half_bits_to_float(lds_u32_any(bp));
            uint32_t Q[4];
            lds_words_any<4>(bp + 2 + 16 * (lam & 1), Q);
            q80_leaf<B, NL>(Q, d, xr, l, lp[l]);
        }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
        if (NL == 4) part[b] = (lp[0][b] + lp[1][b]) + (lp[2][b] + lp[3][b]);
        else if (NL == 2) part[b] = lp[0][b] + lp[1 % NL][b];
        else part[b] = lp[0][b];
    }
}

// Fast activation epilogue.  GELU-tanh written as g * sigmoid(2z), which
// is the same function as 0.5 g (1 + tanh z) without the cancellation of
// 1 + tanh z for negative g.
__device__ __forceinline__ float act_apply(int act, float g) {
    if (act == ACT_GEGLU_TANH) {
        const float z = 0.7978845608028654f * fmaf(0.044715f * g, g * g, g);
        return g / (1.0f + expf(-2.0f * z));
    }
    return g / (1.0f + expf(-g));
}

// Sum of one (row, batch) partial vector over all groups in the canonical
// order; the value in lane 0 is the result.
template <int B>
__device__ __forceinline__ float reduce_groups(const float* r, int ngroups, int lane) {
    float acc = 0.f;
    for (int G = lane; G < ngroups; G += 32) {
        float pg;
        if (B == 1) pg = r[G];
        else if (B == 2) pg = r[2 * G] + r[2 * G + 1];
        else pg = (r[4 * G] + r[4 * G + 1]) + (r[4 * G + 2] + r[4 * G + 3]);
        acc += pg;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    return acc;
}

}  // namespace

// Shared memory: [nstages * stage_bytes] stages | red[2][RT*B*U] | mbar[nstages]
template <int B>
__global__ void __launch_bounds__(512, 1) stream_mv_kernel(const __grid_constant__ StreamParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int NL = 4 / B;
    const int tid = threadIdx.x;
    const int NT = blockDim.x;
    const int U = P.ngroups * B;
    const int u = tid % U;
    const int slot = tid / U;
    const int G = u / B;
    const int lam0 = (u % B) * NL;
    const int R = P.RT / P.k;
    const int S_ = P.nstages;
    const int red_stride = P.RT * B * U;

    uint8_t* stages = smem;
    float* red = reinterpret_cast<float*>(smem + (size_t)S_ * P.stage_bytes);
    uint64_t* mbar = reinterpret_cast<uint64_t*>(red + 2 * red_stride);

    if (tid == 0) {
        for (int s = 0; s < S_; ++s) mbar_init(&mbar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    uint64_t policy = 0;
    if (tid == 0) policy = policy_evict_first();

    // ---- producer state (thread 0): next tile to issue, stage ring cursor
    int p_hint = 0;
    int p_tile = next_tile(P, blockIdx.x, p_hint, B);
    uint32_t pending = 0;      // stages with a bulk copy in flight (thread 0)
    auto issue = [&](int stage) {
        const Seg& S = P.seg[p_hint];
        const TileGeo g = tile_geo(P, S, p_tile);
        if (g.tma) {
            uint8_t* dst = stages + (size_t)stage * P.stage_bytes;
            mbar_arrive_expect_tx(&mbar[stage], g.bytes1 + g.bytes2);
            bulk_g2s_stream(dst, g.src1, g.bytes1, &mbar[stage], policy);
            if (g.bytes2) bulk_g2s_stream(dst + g.dst2, g.src2, g.bytes2, &mbar[stage], policy);
            pending |= 1u << stage;
        }
        p_tile = next_tile(P, p_tile + gridDim.x, p_hint, B);
    };
    if (tid == 0) {
        for (int s = 0; s < S_ && p_tile < P.ntiles; ++s) issue(s);
    }

    // ---- consumers (all threads)
    int c_hint = 0;
    int c_tile = next_tile(P, blockIdx.x, c_hint, B);
    int cur_seg = -1;
    uint32_t phase_bits = 0;   // parity of the next completion per stage
    float2 xr[B][NL][8];
    int i = 0;
    int buf = 0;
    while (c_tile < P.ntiles) {
        const int stage = i % S_;
        const Seg& S = P.seg[c_hint];
        const TileGeo g = tile_geo(P, S, c_tile);
        uint8_t* st = stages + (size_t)stage * P.stage_bytes;
        bool bad = false;
        if (g.tma) {
            bad = !mbar_wait_bounded(&mbar[stage], (phase_bits >> stage) & 1u, P.timeout_ns);
            if (!bad) {
                phase_bits ^= 1u << stage;
                pending &= ~(1u << stage);
            }
        } else {
            manual_copy(st, g.src1, g.bytes1);
            if (g.bytes2) manual_copy(st + g.dst2, g.src2, g.bytes2);
            __syncthreads();
        }
        if (c_hint != cur_seg) {   // new matrix: its format / x rows may differ
            load_x<B>(P, S, G, lam0, xr);
            cur_seg = c_hint;
        }
        const int64_t rb = row_bytes(S.fmt, P.cols);
        const int half = P.RT / 2;
        float* rbuf = red + buf * red_stride;
        if (!bad) {
#pragma unroll 1
            for (int j = 0; j < R; ++j) {
                const int rho = slot + P.k * j;
                bool valid;
                if (S.mode == MODE_PLAIN) valid = rho < g.n_o;
                else if (S.mode == MODE_PAIR_INTERLEAVED) valid = rho < 2 * g.n_o;
                else valid = (rho % half) < g.n_o;
                float part[B];
                if (valid) {
                    unit_dot<B>(S.fmt, st + (int64_t)rho * rb, G, lam0, xr, part);
                } else {
#pragma unroll
                    for (int b = 0; b < B; ++b) part[b] = 0.f;
                }
#pragma unroll
                for (int b = 0; b < B; ++b) rbuf[(rho * B + b) * U + u] = part[b];
            }
        }
        const int any_bad = __syncthreads_or(bad ? 1 : 0);
        if (any_bad) {
            if (tid == 0) {
                record_status(P.status, STATUS_TIMEOUT);
                // drain this CTA's bulk copies still in flight (bounded)
                for (int s2 = 0; s2 < S_; ++s2)
                    if (pending & (1u << s2))
                        mbar_wait_bounded(&mbar[s2], (phase_bits >> s2) & 1u, P.timeout_ns);
            }
            return;
        }
        // stage `stage` is free: refill it with the next tile of this CTA
        if (tid == 0 && p_tile < P.ntiles) issue(stage);

        // reduce partials -> outputs
        const int lane = tid & 31, warp = tid >> 5, nw = NT >> 5;
        const int nval = seg_nval(S, B);
        const int boff = seg_boff(S);
        const int n_items = g.n_o * B;
        for (int o = warp; o < n_items; o += nw) {
            const int pi = o / B, b = o % B;
            if (S.mode == MODE_PLAIN) {
                const float v = reduce_groups<B>(rbuf + (pi * B + b) * U, P.ngroups, lane);
                if (lane == 0 && b < nval)
                    S.y[(int64_t)(boff + b) * S.ld_y + g.o0 + pi] = v;
            } else {
                const int rg = S.mode == MODE_PAIR_INTERLEAVED ? 2 * pi : pi;
                const int ru = S.mode == MODE_PAIR_INTERLEAVED ? 2 * pi + 1 : pi + half;
                const float vg = reduce_groups<B>(rbuf + (rg * B + b) * U, P.ngroups, lane);
                const float vu = reduce_groups<B>(rbuf + (ru * B + b) * U, P.ngroups, lane);
                if (lane == 0 && b < nval)
                    S.y[(int64_t)(boff + b) * S.ld_y + g.o0 + pi] = act_apply(S.act, vg) * vu;
            }
        }
        buf ^= 1;
        ++i;
        c_tile = next_tile(P, c_tile + gridDim.x, c_hint, B);
    }
}

// ---- host-side wrappers (the kernel template stays in this translation unit)

cudaError_t stream_set_smem_limit(int bytes) {
    cudaError_t e = cudaFuncSetAttribute(stream_mv_kernel<1>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(stream_mv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(stream_mv_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return e;
}

cudaError_t stream_occupancy(int B, int nt, size_t smem, int* per_sm) {
    if (B == 1) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, stream_mv_kernel<1>, nt, smem);
    if (B == 2) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, stream_mv_kernel<2>, nt, smem);
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, stream_mv_kernel<4>, nt, smem);
}

cudaError_t stream_launch(int B, const StreamParams& P, int grid, int nt, size_t smem,
                          cudaStream_t st) {
    if (B == 1) stream_mv_kernel<1><<<grid, nt, smem, st>>>(P);
    else if (B == 2) stream_mv_kernel<2><<<grid, nt, smem, st>>>(P);
    else stream_mv_kernel<4><<<grid, nt, smem, st>>>(P);
    return cudaGetLastError();
}

}  // namespace lq
