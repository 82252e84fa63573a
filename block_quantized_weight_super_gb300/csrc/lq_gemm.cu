// lq_gemm.cu -- the prefill GEMM: Y[n][r] = sum_j w_rj X[n][j] for many x
// rows n against Q4_K or Q8_0 weights (dotLLM PR #320: the tiled
// matmul_q8_0_gemm for many tokens, and the batched intra-block GEMMs of
// ForwardBatch; larql "Architecture -> Metal shader map" for the Q4_K
// weights).  The same values as lq_matvec's, within the same bound; each
// weight tile is read once per 64 x rows instead of once per 8.
//
// Operands (mma.sync m16n8k16, fp16 in, fp32 accumulate):
//  * A: the exact integer codes of 16 weight rows x 16 columns of one
//    (sub-)block, built in registers from the quantized bytes: a LOP3 ORs
//    two codes into fp16 halves 1024 + q (Q4_K nibbles) or 1152 + q (Q8_0
//    bytes, sign bit flipped), and one fp16x2 subtraction leaves q - qb
//    (Q4_K, re-centred as in the other kernels: qb = round(dmin m / d sc)) or
//    q (Q8_0), exactly.
//  * B: x / s_n in two fp16 pieces (hi = fp16(x / s_n), lo = fp16(x / s_n -
//    hi)), s_n a power of two per x row with |x / s_n| < 2^15, written once
//    per call by gemm_xprep_kernel, together with the 32-column sums of
//    x / s_n (Q4_K).  The pieces carry x to 2^-22 relative (an absolute floor
//    of ~2^-40 max|x| of the row where a value underflows).
//  * Per 32-column (sub-)block the MMAs give P = sum (q - qb) x / s for 16
//    rows x 8 x rows; the epilogue adds d sc P + e sum(x / s) (Q4_K, e = d sc
//    qb - dmin m) or d P (Q8_0) into fp32 accumulators, and the store
//    multiplies by s_n.
//  * k order: within every 16 columns of a block, MMA slot 2t, 2t+1, 2t+8,
//    2t+9 holds column 4t, 4t+2, 4t+1, 4t+3, so a lane's four codes of a row
//    are the four bytes of one 32-bit word; the x pieces are written in the
//    same order.
//
// GB300 structure: a CTA of 8 warps computes 128 weight rows (16 per warp)
// x 64 x rows; every 256 columns a stage of the weight tile (one 16-byte
// cp.async per piece, rows 16-byte aligned) and of the x pieces lands in
// shared memory, two stages in flight.  B fragments come from shared memory
// with ldmatrix (x piece rows padded to 528 bytes: conflict-free), A codes
// with 32-bit loads (row pitch 144 / 272 bytes: 36 / 68 words, the eight
// rows of a quarter-warp in distinct banks).  Consecutive CTAs share a
// weight tile (the x-row tile varies fastest), so a tile comes from HBM once
// and from L2 for the other x-row tiles; the x pieces of a call sit in L2.
// Every output is summed in a fixed order: deterministic, and a row's result
// does not depend on the other x rows of the call.
#include "lq_gv.cuh"
#include "lq_internal.h"

namespace lq {
namespace {

constexpr int GM_THREADS = 256;
constexpr int GM_XP = 528;                 // shared pitch of an x piece row (256 halves + 16 bytes)

// Stage layout for XN x rows per CTA (8 or 4 n-tiles of 8 per warp).
template <int FMT, int XN>
struct GmF {
    static constexpr int WB = FMT == FMT_Q4_K ? 144 : 272;     // weight bytes of a row per stage
    static constexpr int NTL = XN / 8;                         // n-tiles per warp
    static constexpr uint32_t W_OFF = 0;
    static constexpr uint32_t XH_OFF = GEMM_WR * WB;
    static constexpr uint32_t XL_OFF = XH_OFF + XN * GM_XP;
    static constexpr uint32_t XS_OFF = XL_OFF + XN * GM_XP;
    static constexpr uint32_t STAGE = XS_OFF + (FMT == FMT_Q4_K ? XN * 8 * 4 : 0);
};

__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm4(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(a));
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}

// Position of column c (0..15) of a 16-column group in the MMA k order.
__device__ __forceinline__ int gm_slot(int c) {
    const int t = c >> 2, r = c & 3;
    return r == 0 ? 2 * t : r == 2 ? 2 * t + 1 : r == 1 ? 2 * t + 8 : 2 * t + 9;
}

// One CTA per x row: s_n from the row's largest |x|, then per 32-column
// block the pieces of x / s_n (k order of gm_slot) and their fp32 sum.
__global__ void __launch_bounds__(GM_THREADS) gemm_xprep_kernel(const float* __restrict__ X, int64_t K,
                                                                __half* __restrict__ xh, __half* __restrict__ xl,
                                                                float* __restrict__ xs, float* __restrict__ sn) {
    __shared__ float red[GM_THREADS / 32];
    const int64_t n = blockIdx.x;
    const float* x = X + n * K;
    float m = 0.f;
    for (int64_t j = 4 * (int64_t)threadIdx.x; j < K; j += 4 * GM_THREADS) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(x + j));
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = red[0];
    for (int i = 1; i < GM_THREADS / 32; ++i) m = fmaxf(m, red[i]);
    const int E = (int)((__float_as_uint(m) >> 23) & 0xFFu);
    const int es = max(1, E - 14);                                  // s = 2^(es - 127): |x / s| < 2^15
    const float inv = __uint_as_float((uint32_t)(254 - es) << 23);  // 1 / s, exact
    if (threadIdx.x == 0) sn[n] = __uint_as_float((uint32_t)es << 23);
    for (int64_t b = threadIdx.x; b < K / 32; b += GM_THREADS) {
        const float* xb = x + 32 * b;
        float v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 q = __ldg(reinterpret_cast<const float4*>(xb) + i);
            v[4 * i] = q.x * inv;
            v[4 * i + 1] = q.y * inv;
            v[4 * i + 2] = q.z * inv;
            v[4 * i + 3] = q.w * inv;
        }
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) s += v[i];
        xs[n * (K / 32) + b] = s;
#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
            __align__(16) __half hi[16], lo[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float a = v[16 * grp + c];
                const __half h = __float2half_rn(a);
                hi[gm_slot(c)] = h;
                lo[gm_slot(c)] = __float2half_rn(a - __half2float(h));
            }
            uint4* dh = reinterpret_cast<uint4*>(xh + n * K + 32 * b + 16 * grp);
            uint4* dl = reinterpret_cast<uint4*>(xl + n * K + 32 * b + 16 * grp);
            dh[0] = reinterpret_cast<const uint4*>(hi)[0];
            dh[1] = reinterpret_cast<const uint4*>(hi)[1];
            dl[0] = reinterpret_cast<const uint4*>(lo)[0];
            dl[1] = reinterpret_cast<const uint4*>(lo)[1];
        }
    }
}

// 16 rows x 32 columns of one (sub-)block against the NTL x 8 x rows of the
// stage: P[jn] (n-tile jn: x rows 8 jn .. 8 jn + 7) += A . (hi + lo).
// a[h][0..3]: the A registers of the two 16-column halves.
template <int NTL>
__device__ __forceinline__ void gm_block(const uint32_t (&a)[2][4], uint32_t xh_base, uint32_t xl_base, int blk,
                                         int lane, float (&P)[NTL][4]) {
    const int mi = lane >> 3, r8 = lane & 7;
    // lane's ldmatrix row: n-tile (jn + (mi >> 1)), row r8, k half (mi & 1)
    const uint32_t roff = (uint32_t)((8 * (mi >> 1) + r8) * GM_XP + 2 * (32 * blk + 8 * (mi & 1)));
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int jn = 0; jn < NTL; jn += 2) {
            const uint32_t off = roff + (uint32_t)(8 * jn * GM_XP + 2 * 16 * h);
            uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
            ldsm4(xh_base + off, b0, b1, b2, b3);
            ldsm4(xl_base + off, c0, c1, c2, c3);
            mma_h(P[jn], a[h][0], a[h][1], a[h][2], a[h][3], b0, b1);
            mma_h(P[jn], a[h][0], a[h][1], a[h][2], a[h][3], c0, c1);
            mma_h(P[jn + 1], a[h][0], a[h][1], a[h][2], a[h][3], b2, b3);
            mma_h(P[jn + 1], a[h][0], a[h][1], a[h][2], a[h][3], c2, c3);
        }
    }
}

template <int FMT, int XN>
__global__ void __launch_bounds__(GM_THREADS, XN == 32 ? 2 : 1) gemm_kernel(const __grid_constant__ GemmParams P) {
    using F = GmF<FMT, XN>;
    constexpr int NTL = F::NTL;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int mt = blockIdx.x % P.nmt, wt = blockIdx.x / P.nmt;
    const int64_t r0 = (int64_t)wt * GEMM_WR, n0 = (int64_t)mt * XN;
    const int64_t K = P.cols;
    const int nk = (int)(K / 256);
    const uint32_t sbase = smem_u32(smem);

    auto load_stage = [&](int kk, int s) {
        const uint32_t st = sbase + (uint32_t)s * F::STAGE;
        constexpr int WP = F::WB / 16;                  // 16-byte pieces of a row
        for (int p = tid; p < GEMM_WR * WP; p += GM_THREADS) {
            const int rr = p / WP, q = p - rr * WP;
            if (r0 + rr < P.rows)
                cp16(st + F::W_OFF + (uint32_t)(rr * F::WB + 16 * q),
                     P.W + (r0 + rr) * P.rowbytes + (int64_t)kk * F::WB + 16 * q);
        }
        for (int p = tid; p < XN * 32; p += GM_THREADS) {
            const int nn = p >> 5, q = p & 31;
            if (n0 + nn < P.M) {
                const int64_t src = (n0 + nn) * K + (int64_t)kk * 256 + 8 * q;
                cp16(st + F::XH_OFF + (uint32_t)(nn * GM_XP + 16 * q), P.xh + src);
                cp16(st + F::XL_OFF + (uint32_t)(nn * GM_XP + 16 * q), P.xl + src);
            }
        }
        if (FMT == FMT_Q4_K) {
            for (int p = tid; p < XN * 2; p += GM_THREADS) {
                const int nn = p >> 1, q = p & 1;
                if (n0 + nn < P.M) cp16(st + F::XS_OFF + (uint32_t)(nn * 32 + 16 * q), P.xs + (n0 + nn) * (K / 32) + kk * 8 + 4 * q);
            }
        }
    };

    float acc[NTL][4];
#pragma unroll
    for (int j = 0; j < NTL; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    const GvK KC = gv_consts();

    load_stage(0, 0);
    cp_commit();
    for (int kk = 0; kk < nk; ++kk) {
        if (kk + 1 < nk) load_stage(kk + 1, (kk + 1) & 1);
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        const uint32_t st = sbase + (uint32_t)(kk & 1) * F::STAGE;
        const uint32_t rowA = st + F::W_OFF + (uint32_t)((16 * warp + g) * F::WB);
        const uint32_t rowB = rowA + 8 * F::WB;
        const uint32_t xhb = st + F::XH_OFF, xlb = st + F::XL_OFF;
        if constexpr (FMT == FMT_Q4_K) {
            const uint4 hA = lds128(rowA), hB = lds128(rowB);
#pragma unroll 1
            for (int jq = 0; jq < 4; ++jq) {                     // quant group: sub-blocks 2 jq, 2 jq + 1
                const Q4Sel sel = q4_sel(jq);
                const Q4Cent cA = q4k_centres(hA, sel, KC.magic), cB = q4k_centres(hB, sel, KC.magic);
#pragma unroll
                for (int nib = 0; nib < 2; ++nib) {
                    const uint32_t sA = h2dup(1024.0f + (nib ? cA.qb1 : cA.qb0));
                    const uint32_t sB = h2dup(1024.0f + (nib ? cB.qb1 : cB.qb0));
                    uint32_t a[2][4];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t wA = lds32(rowA + 16 + 32 * jq + 16 * h + 4 * t);
                        uint32_t wB = lds32(rowB + 16 + 32 * jq + 16 * h + 4 * t);
                        if (nib) {
                            wA >>= 4;
                            wB >>= 4;
                        }
                        a[h][0] = hsub2_u32(lop_and_or(wA, KC.m4lo, KC.magic), sA);
                        a[h][1] = hsub2_u32(lop_and_or(wB, KC.m4lo, KC.magic), sB);
                        a[h][2] = hsub2_u32(lop_and_or(wA >> 8, KC.m4lo, KC.magic), sA);
                        a[h][3] = hsub2_u32(lop_and_or(wB >> 8, KC.m4lo, KC.magic), sB);
                    }
                    float Pp[NTL][4];
#pragma unroll
                    for (int j = 0; j < NTL; ++j) Pp[j][0] = Pp[j][1] = Pp[j][2] = Pp[j][3] = 0.f;
                    const int blk = 2 * jq + nib;
                    gm_block<NTL>(a, xhb, xlb, blk, lane, Pp);
                    const float dA = nib ? cA.dsc1 : cA.dsc0, dB = nib ? cB.dsc1 : cB.dsc0;
                    const float eA = nib ? cA.e1 : cA.e0, eB = nib ? cB.e1 : cB.e0;
                    const float* xsb = reinterpret_cast<const float*>(smem + (kk & 1) * F::STAGE + F::XS_OFF);
#pragma unroll
                    for (int j = 0; j < NTL; ++j) {
                        const int nl = 8 * j + 2 * t;
                        const float s0 = xsb[nl * 8 + blk], s1 = xsb[(nl + 1) * 8 + blk];
                        acc[j][0] = fmaf(dA, Pp[j][0], fmaf(eA, s0, acc[j][0]));
                        acc[j][1] = fmaf(dA, Pp[j][1], fmaf(eA, s1, acc[j][1]));
                        acc[j][2] = fmaf(dB, Pp[j][2], fmaf(eB, s0, acc[j][2]));
                        acc[j][3] = fmaf(dB, Pp[j][3], fmaf(eB, s1, acc[j][3]));
                    }
                }
            }
        } else {
#pragma unroll 1
            for (int blk = 0; blk < 8; ++blk) {
                // block blk of the stage: 34 bytes at 34 blk; codes start 2 bytes in
                const uint32_t bA = rowA + 34 * blk, bB = rowB + 34 * blk;
                const float dA = half_bits_to_float(lds16(bA)), dB = half_bits_to_float(lds16(bB));
                uint32_t a[2][4];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t oA = bA + 2 + 16 * h + 4 * t, oB = bB + 2 + 16 * h + 4 * t;
                    uint32_t wA, wB;
                    if (blk & 1) {                              // 34 blk + 2 = 0 (mod 4)
                        wA = lds32(oA);
                        wB = lds32(oB);
                    } else {                                    // = 2 (mod 4): two words, funnel shift
                        wA = __funnelshift_r(lds32(oA - 2), lds32(oA + 2), 16);
                        wB = __funnelshift_r(lds32(oB - 2), lds32(oB + 2), 16);
                    }
                    a[h][0] = hsub2_u32(lop_and_xor(wA, KC.m8, KC.x8), KC.s8);
                    a[h][1] = hsub2_u32(lop_and_xor(wB, KC.m8, KC.x8), KC.s8);
                    a[h][2] = hsub2_u32(lop_and_xor(wA >> 8, KC.m8, KC.x8), KC.s8);
                    a[h][3] = hsub2_u32(lop_and_xor(wB >> 8, KC.m8, KC.x8), KC.s8);
                }
                float Pp[NTL][4];
#pragma unroll
                for (int j = 0; j < NTL; ++j) Pp[j][0] = Pp[j][1] = Pp[j][2] = Pp[j][3] = 0.f;
                gm_block<NTL>(a, xhb, xlb, blk, lane, Pp);
#pragma unroll
                for (int j = 0; j < NTL; ++j) {
                    acc[j][0] = fmaf(dA, Pp[j][0], acc[j][0]);
                    acc[j][1] = fmaf(dA, Pp[j][1], acc[j][1]);
                    acc[j][2] = fmaf(dB, Pp[j][2], acc[j][2]);
                    acc[j][3] = fmaf(dB, Pp[j][3], acc[j][3]);
                }
            }
        }
        __syncthreads();                                      // the stage is read; the next load may overwrite it
    }
    cp_wait<0>();
    // y[n][r] = s_n * acc; lane holds rows g, g + 8 and x rows 8 j + 2 t, + 1
    const int64_t ra = r0 + 16 * warp + g, rb = ra + 8;
#pragma unroll
    for (int j = 0; j < NTL; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int64_t n = n0 + 8 * j + 2 * t + e;
            if (n >= P.M) continue;
            const float s = P.sn[n];
            if (ra < P.rows) P.Y[n * P.ld_y + ra] = acc[j][e] * s;
            if (rb < P.rows) P.Y[n * P.ld_y + rb] = acc[j][2 + e] * s;
        }
    }
}

}  // namespace

int gemm_xn(int fmt) { return fmt == FMT_Q4_K ? GEMM_XN_Q4K : GEMM_XN_Q80; }

size_t gemm_smem_bytes(int fmt) {
    return 2 * (size_t)(fmt == FMT_Q4_K ? GmF<FMT_Q4_K, GEMM_XN_Q4K>::STAGE : GmF<FMT_Q8_0, GEMM_XN_Q80>::STAGE);
}

cudaError_t gemm_set_smem() {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<FMT_Q4_K, GEMM_XN_Q4K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)gemm_smem_bytes(FMT_Q4_K));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gemm_kernel<FMT_Q8_0, GEMM_XN_Q80>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)gemm_smem_bytes(FMT_Q8_0));
}

cudaError_t gemm_launch(int fmt, const GemmParams& P, const float* X, cudaStream_t st) {
    gemm_xprep_kernel<<<(unsigned)P.M, GM_THREADS, 0, st>>>(X, P.cols, reinterpret_cast<__half*>(P.xh),
                                                             reinterpret_cast<__half*>(P.xl), P.xs, P.sn);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t nwt = (P.rows + GEMM_WR - 1) / GEMM_WR;
    const int grid = (int)(nwt * P.nmt);
    if (fmt == FMT_Q4_K)
        gemm_kernel<FMT_Q4_K, GEMM_XN_Q4K><<<grid, GM_THREADS, gemm_smem_bytes(fmt), st>>>(P);
    else
        gemm_kernel<FMT_Q8_0, GEMM_XN_Q80><<<grid, GM_THREADS, gemm_smem_bytes(fmt), st>>>(P);
    return cudaGetLastError();
}

}  // namespace lq
