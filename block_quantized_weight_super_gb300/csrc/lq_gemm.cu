// lq_gemm.cu -- the prefill GEMM: Y[n][r] = sum_j w_rj X[n][j] for many x
// rows n against Q4_K or Q8_0 weights (dotLLM PR #320: the tiled
// matmul_q8_0_gemm for many tokens, and the batched intra-block GEMMs of
// ForwardBatch; larql "Architecture -> Metal shader map" for the Q4_K
// weights), on the fifth-generation tensor cores.  The same values as
// lq_matvec's, within the same bound.
//
// tcgen05.mma, fp16 in, fp32 accumulators in tensor memory.  The per-block
// scales are taken out of the MMA's way: every weight is dequantized exactly
// as the library does (w = d sc q - dmin m in one fp32 rounding, or d q) and
// divided by t_r, a power of two per weight row with |w / t_r| < 2^15 (from
// the row's block scales), then split into fp16 pieces hi = fp16(w / t_r)
// and lo = fp16(w / t_r - hi); x / s_n is split the same way (s_n a power
// of two per x row).  The tensor cores form w_hi x_hi, w_lo x_hi and
// w_hi x_lo in fp32 accumulators in tensor memory over the whole row (w_lo
// x_lo is below 2^-22 of |w x| and left out); the epilogue multiplies by t_r
// and s_n (exact, powers of two).  The pieces carry w / t_r and x / s_n to
// 2^-22 relative each (absolute floors ~2^-40 of the row's largest value
// where a value underflows fp16).  gemm_prep_kernel finds s_n and t_r,
// gemm_ximg_kernel writes the x pieces.
//
// Operands, per 32-column step: A = the weight pieces (hi then lo, 128 rows
// each) and B = the x pieces of an x tile (hi then lo, 128 rows each), both
// in shared memory in the K-major core-matrix layout without swizzle (a core
// matrix is 8 rows x 16 bytes; 128 bytes between core matrices along K, 512
// along M / N).  The x pieces are written once per call in exactly that
// layout, 16 KB per 128 x rows and 32 columns, so a stage of B is one bulk
// copy per x tile.  Per 16 columns and x tile two MMAs into the tile's
// accumulator (256 tensor-memory columns): A_hi against all 256 rows of B
// (N = 256: w_hi x_hi in columns 0-127, w_hi x_lo in 128-255) and A_lo
// against B's hi rows (N = 128, into columns 0-127); the epilogue adds the
// two halves.  A CTA takes one or two x tiles (NX): with two, every A stage
// is used twice and the MMAs of the two tiles alternate; each tile's
// accumulator sees the same sequence either way, so a row's result does not
// depend on NX.
//
// Gate / up pairs (the packed matrix of lq_pack_gate_up, rows 2i and 2i + 1
// the gate and up rows of output i): the epilogue scales both sums, the odd
// lane hands its up value to the even one by a shuffle, and the even lane
// stores act(g) * u.
//
// Split K: where the weight matrix has few 128-row tiles the row is cut
// into ksplit ranges of whole 256-column chunks (gemm_tc_ksplit, a
// function of the weight shape alone); each CTA stores its raw partial sums
// and gemm_tc_reduce_kernel adds them in range order and scales.
//
// Warp roles.  A warp's scheduler is its index mod 4; the MMA-issuing
// thread must not share one with the A builders (their ALU work starves its
// issue, halving the MMA rate), so:
//  * warps 0-2, 4-6, 8-9 build A: per 32-column step a thread dequantizes
//    and splits 16 weights of one row (two threads per row) from the staged
//    weight bytes into the step's A stage;
//  * warp 3 owns the tensor memory and one thread issues each step's MMAs
//    once A and B are in, committing them to the stages' "empty" barriers;
//  * warp 7 copies the x pieces of each step (a bulk copy per x tile);
//  * warp 10 copies the weight bytes of each 256-column chunk (one tensor
//    copy of 128 rows), two chunks in flight;
//  * at the end warps 0-7 read the accumulators back (warp w: tensor-memory
//    lanes 32 (w % 4) .. + 31) and store.
// Every wait is bounded: on a timeout the CTA records it, lets its copies
// and MMAs in flight finish (bounded), frees its tensor memory and returns.
#include <algorithm>

#include "lq_codec.cuh"
#include "lq_device.cuh"
#include "lq_internal.h"

namespace lq {
namespace {

constexpr int GT_WR = GEMM_TC_WR;          // weight rows per CTA (MMA M)
constexpr int GT_XN = GEMM_TC_XN;          // x rows per x tile
constexpr int GT_NB = 8;                   // A-building warps
constexpr int GT_THREADS = 11 * 32;
constexpr int GT_MMA_WARP = 3, GT_BLOAD_WARP = 7, GT_WLOAD_WARP = 10;
constexpr uint32_t GT_XSTEP = 16384;       // x image bytes per 128 x rows and 32 columns (hi, lo)
constexpr uint32_t GT_ASTEP = 16384;       // A stage: 128 weight rows x 32 columns (hi, lo)
constexpr uint32_t GT_LBO = 128;           // core matrices adjacent along K
constexpr uint32_t GT_SBO = 512;           // core matrices adjacent along M / N
constexpr int GT_SPLIT_SMS = 152;          // split K below half this many weight tiles (GB300's SM count)

// builder warp index (0-7) of warps 0-2, 4-6, 8-9; -1 for the others
__device__ __forceinline__ int gt_builder(int warp) {
    return (warp & 3) == 3 || warp > 9 ? -1 : warp - (warp >> 2);
}

template <int FMT, int NX>
struct GtF {
    static constexpr int WB = FMT == FMT_Q4_K ? 144 : 272;     // weight bytes of a row per 256 columns
    static constexpr int NSA = NX == 1 ? (FMT == FMT_Q4_K ? 4 : 3) : 3;           // A stages
    static constexpr int NSB = NX == 1 ? (FMT == FMT_Q4_K ? 7 : 6) : (FMT == FMT_Q4_K ? 4 : 3);   // B stages
    static constexpr uint32_t BSTEP = NX * GT_XSTEP;
    static constexpr uint32_t A_OFF = 0;
    static constexpr uint32_t B_OFF = A_OFF + NSA * GT_ASTEP;
    static constexpr uint32_t W_OFF = B_OFF + NSB * BSTEP;
    static constexpr uint32_t WBUF = GT_WR * WB;                // a multiple of 16
    static constexpr uint32_t BAR_OFF = W_OFF + 2 * WBUF;
    // bfull, bempty [NSB]; afull, aempty [NSA]; wfull, wempty [2]; dfull
    static constexpr int NBAR = 2 * NSB + 2 * NSA + 5;
    static constexpr uint32_t TOTAL = BAR_OFF + 8 * NBAR + 16;
    static constexpr uint32_t TMEM_COLS = 256 * NX;
};

__device__ __forceinline__ uint64_t gt_desc(uint32_t addr) {
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((GT_LBO >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((GT_SBO >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;                // descriptor version of this architecture; no swizzle, base offset 0
    return d;
}

// kind::f16 instruction descriptors: fp32 accumulators, fp16 A and B, both
// K-major, M = 128, N = 256 or 128
constexpr uint32_t GT_IDESC256 = (1u << 4) | ((uint32_t)(256 >> 3) << 17) | ((uint32_t)(GT_WR >> 4) << 24);
constexpr uint32_t GT_IDESC128 = (1u << 4) | ((uint32_t)(128 >> 3) << 17) | ((uint32_t)(GT_WR >> 4) << 24);

// D (tensor memory) += A . B, both from shared memory (descriptors)
__device__ __forceinline__ void gt_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                 "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void gt_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Bounded wait on one thread.
__device__ __forceinline__ bool gt_wait1(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    return mbar_wait_bounded(bar, parity, timeout_ns);
}

// Warp-uniform bounded wait: lane 0 polls (32 lanes polling one barrier
// serialize on it), then the warp synchronizes, which orders the other
// lanes' later accesses after lane 0's observation of the phase.
__device__ __forceinline__ bool gt_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = gt_wait1(bar, parity, timeout_ns);
    __syncwarp();
    return __shfl_sync(0xFFFFFFFFu, ok, 0);
}

__device__ __forceinline__ uint32_t h2pk(float2 v) {
    const __half2 h = __floats2half2_rn(v.x, v.y);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// pairs of values (w / t) as packed hi and lo fp16 pieces
template <int N>
__device__ __forceinline__ void gt_split(const float2 (&w)[N], uint32_t (&hi)[N], uint32_t (&lo)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
        hi[i] = h2pk(w[i]);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hi[i]));
        lo[i] = h2pk(__fadd2_rn(w[i], make_float2(-f.x, -f.y)));
    }
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds128u(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
                 "%14, %15}, [%16];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                   "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                 : "r"(taddr));
}

// The two scale passes in one launch.  Blocks [0, mp): s_n of x row
// blockIdx.x (rows M .. mp - 1 of the padded tile get 1), s_n = 2^(e - 14)
// for the binade e of the row's largest |x|.  The blocks after them: 1 / t_r
// per weight row, one warp per row: the row's largest |w| is at most the
// largest over its blocks of |d| * 63 * 15 + |dmin| * 63 (Q4_K) or |d| * 128
// (Q8_0); t_r = 2^(e - 14) for that bound's binade e (at least 2^-126).
template <int FMT>
__global__ void __launch_bounds__(256) gemm_prep_kernel(const float* __restrict__ X, int64_t M, int64_t mp,
                                                        int64_t K, float* __restrict__ sn, const uint8_t* __restrict__ W,
                                                        int64_t rows, int64_t rowbytes, float* __restrict__ tinv) {
    __shared__ float red[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if ((int64_t)blockIdx.x < mp) {
        const int64_t n = blockIdx.x;
        float m = 0.f;
        if (n < M)
            for (int64_t j = 4 * (int64_t)threadIdx.x; j < K; j += 1024) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(X + n * K + j));
                m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) red[warp] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
            const int E = (int)((__float_as_uint(m) >> 23) & 0xFFu);
            const int es = max(1, E - 14);                               // s = 2^(es - 127): |x / s| < 2^15
            sn[n] = n < M ? __uint_as_float((uint32_t)es << 23) : 1.f;
        }
        return;
    }
    const int64_t r = ((int64_t)blockIdx.x - mp) * 8 + warp;
    if (r >= rows) return;
    const uint8_t* row = W + r * rowbytes;
    float bound = 0.f;
    if (FMT == FMT_Q4_K) {
        for (int64_t b = lane; b < K / 256; b += 32) {
            const uint32_t dd = __ldg(reinterpret_cast<const uint32_t*>(row + 144 * b));
            bound = fmaxf(bound, fmaf(fabsf(half_bits_to_float(dd)), 945.0f, 63.0f * fabsf(half_bits_to_float(dd >> 16))));
        }
    } else {
        for (int64_t b = lane; b < K / 32; b += 32) {
            const uint32_t dd = __ldg(reinterpret_cast<const unsigned short*>(row + 34 * b));
            bound = fmaxf(bound, 128.0f * fabsf(half_bits_to_float(dd)));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bound = fmaxf(bound, __shfl_xor_sync(0xFFFFFFFFu, bound, o));
    const int E = (int)((__float_as_uint(bound) >> 23) & 0xFFu);
    const int et = max(1, E - 14);                                       // t = 2^(et - 127)
    if (lane == 0) tinv[r] = __uint_as_float((uint32_t)(254 - et) << 23);   // 1 / t, exact
}

// The x image: for x tile m (128 rows, rows >= M zero) and 32-column step
// s, GT_XSTEP bytes at (m * nsteps + s) * GT_XSTEP: the hi pieces of x / s_n
// in the core-matrix layout, then the lo pieces.  A block does 8 x rows
// (one core-matrix row group) x 256 columns, eight threads writing one
// 128-byte line.
__global__ void __launch_bounds__(256) gemm_ximg_kernel(const float* __restrict__ X, int64_t M, int64_t K,
                                                        const float* __restrict__ sn, uint8_t* __restrict__ img) {
    const int tid = threadIdx.x, i8 = tid & 7;
    const int64_t n = (int64_t)blockIdx.x * 8 + i8;
    const int64_t c8 = (int64_t)blockIdx.y * 32 + (tid >> 3);           // 8-column piece
    const float inv = __uint_as_float((254u << 23) - __float_as_uint(__ldg(sn + n)));   // 1 / s_n, exact
    float2 v[4];
    if (n < M) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(X + n * K + 8 * c8));
        const float4 b = __ldg(reinterpret_cast<const float4*>(X + n * K + 8 * c8 + 4));
        v[0] = make_float2(a.x * inv, a.y * inv);
        v[1] = make_float2(a.z * inv, a.w * inv);
        v[2] = make_float2(b.x * inv, b.y * inv);
        v[3] = make_float2(b.z * inv, b.w * inv);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = make_float2(0.f, 0.f);
    }
    uint32_t hi[4], lo[4];
    gt_split(v, hi, lo);
    const int64_t mt = n >> 7, s = c8 >> 2;
    const int i = (int)(n & 127), kc = (int)(c8 & 3);
    uint8_t* dst = img + (mt * (K / 32) + s) * GT_XSTEP + (i >> 3) * GT_SBO + kc * GT_LBO + (i & 7) * 16;
    *reinterpret_cast<uint4*>(dst) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(dst + GT_XSTEP / 2) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// Y[n][r] = (sum over the ksplit partial sums, in order) * t_r * s_n; a
// block does four columns per thread of one x row (blockIdx.x)
__global__ void __launch_bounds__(256) gemm_tc_reduce_kernel(const float* __restrict__ part, int ksplit, int64_t M,
                                                             int64_t rows, const float* __restrict__ tinv,
                                                             const float* __restrict__ sn, float* __restrict__ Y) {
    const int64_t n = blockIdx.x, r = 4 * ((int64_t)blockIdx.y * blockDim.x + threadIdx.x);
    if (r >= rows) return;
    const int64_t total = M * rows, i = n * rows + r;
    const float s = __ldg(sn + n);
    if (r + 4 <= rows && (rows & 3) == 0 && (reinterpret_cast<uintptr_t>(Y) & 15) == 0) {
        float4 v = __ldg(reinterpret_cast<const float4*>(part + i));
        for (int k = 1; k < ksplit; ++k) {
            const float4 u = __ldg(reinterpret_cast<const float4*>(part + (int64_t)k * total + i));
            v.x += u.x;
            v.y += u.y;
            v.z += u.z;
            v.w += u.w;
        }
        const float4 t = __ldg(reinterpret_cast<const float4*>(tinv + r));
        *reinterpret_cast<float4*>(Y + i) =
            make_float4((v.x * (1.0f / t.x)) * s, (v.y * (1.0f / t.y)) * s, (v.z * (1.0f / t.z)) * s, (v.w * (1.0f / t.w)) * s);
        return;
    }
    for (int64_t e = 0; e < 4 && r + e < rows; ++e) {
        float v = part[i + e];
        for (int k = 1; k < ksplit; ++k) v += part[(int64_t)k * total + i + e];
        Y[i + e] = (v * (1.0f / tinv[r + e])) * s;
    }
}

// The same for gate / up pairs: H[n][i] = act(g) * u with g, u the scaled
// sums of rows 2i and 2i + 1; a thread per output
__global__ void __launch_bounds__(256) gemm_tc_reduce_pairs_kernel(const float* __restrict__ part, int ksplit,
                                                                   int64_t M, int64_t rows, const float* __restrict__ tinv,
                                                                   const float* __restrict__ sn, int act,
                                                                   float* __restrict__ H) {
    const int64_t n = blockIdx.x, i = (int64_t)blockIdx.y * blockDim.x + threadIdx.x, inter = rows / 2;
    if (i >= inter) return;
    const int64_t total = M * rows, o = n * rows + 2 * i;
    float g = part[o], u = part[o + 1];
    for (int k = 1; k < ksplit; ++k) {
        g += part[(int64_t)k * total + o];
        u += part[(int64_t)k * total + o + 1];
    }
    const float s = __ldg(sn + n);
    g = (g * (1.0f / tinv[2 * i])) * s;
    u = (u * (1.0f / tinv[2 * i + 1])) * s;
    H[n * inter + i] = act_eval(act, g) * u;
}

template <int FMT, int NX>
__global__ void __launch_bounds__(GT_THREADS, 1) gemm_tc_kernel(const __grid_constant__ GemmParams P) {
    using F = GtF<FMT, NX>;
    constexpr int NSA = F::NSA, NSB = F::NSB;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // block order: x-tile group fastest, then K range, then weight tile
    const int nxg = (P.nmt + NX - 1) / NX;
    const int xg = blockIdx.x % nxg, ks = (blockIdx.x / nxg) % P.ksplit, wt = blockIdx.x / nxg / P.ksplit;
    const int mt0 = xg * NX;
    const int ntile = min(NX, P.nmt - mt0);                              // x tiles of this CTA (1 or NX)
    const int64_t r0 = (int64_t)wt * GT_WR;
    const int64_t K = P.cols;
    const int nsteps_all = (int)(K / 32), nchunk_all = (int)(K / 256);
    const int c0 = (int)((int64_t)nchunk_all * ks / P.ksplit), c1 = (int)((int64_t)nchunk_all * (ks + 1) / P.ksplit);
    const int nchunk = c1 - c0, nsteps = 8 * nchunk;                     // this CTA's chunks and steps
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bfull = reinterpret_cast<uint64_t*>(smem + F::BAR_OFF);   // [B stage] x pieces landed (tx)
    uint64_t* bempty = bfull + NSB;                                      // [B stage] its MMAs finished
    uint64_t* afull = bempty + NSB;                                      // [A stage] A stored
    uint64_t* aempty = afull + NSA;                                      // [A stage] its MMAs finished
    uint64_t* wfull = aempty + NSA;                                      // [buffer] weight chunk landed (tx)
    uint64_t* wempty = wfull + 2;                                        // [buffer] A built from it
    uint64_t* dfull = wempty + 2;                                        // every MMA finished
    uint32_t* tslot = reinterpret_cast<uint32_t*>(dfull + 1);

    if (tid == 0) {
        for (int i = 0; i < NSB; ++i) {
            mbar_init(&bfull[i], 1);
            mbar_init(&bempty[i], 1);
        }
        for (int i = 0; i < NSA; ++i) {
            mbar_init(&afull[i], GT_NB);
            mbar_init(&aempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&wfull[i], 1);
            mbar_init(&wempty[i], GT_NB);
        }
        mbar_init(dfull, 1);
        fence_mbar_init();
    }
    if (warp == GT_MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "r"(F::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tslot;
    bool ok = true;
    const int bi = gt_builder(warp);

    if (warp == GT_BLOAD_WARP) {
        // ---- x pieces: a bulk copy per step and x tile
        const uint8_t* img = P.ximg + ((int64_t)mt0 * nsteps_all + 8 * c0) * GT_XSTEP;
        int issued = 0;
        for (int s = 0; s < nsteps; ++s) {
            const int sb = s % NSB;
            if (s >= NSB && !(ok = gt_wait(&bempty[sb], (uint32_t)((s / NSB - 1) & 1), P.timeout_ns))) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bfull[sb], (unsigned)ntile * GT_XSTEP);
                for (int t = 0; t < ntile; ++t)
                    bulk_g2s(smem + F::B_OFF + sb * F::BSTEP + t * GT_XSTEP,
                             img + ((int64_t)t * nsteps_all + s) * GT_XSTEP, GT_XSTEP, &bfull[sb]);
            }
            issued = s + 1;
        }
        // the last copy of each stage has landed before the CTA may exit
        for (int s = max(0, issued - NSB); s < issued; ++s)
            gt_wait(&bfull[s % NSB], (uint32_t)((s / NSB) & 1), drain_bound(P.timeout_ns));
    } else if (warp == GT_WLOAD_WARP) {
        // ---- weight bytes: one tensor copy per 256-column chunk (128 rows,
        // rows past the matrix zero-filled)
        if (lane == 0) prefetch_tensormap(&P.tmw);
        int issued = 0;
        for (int c = 0; c < nchunk; ++c) {
            const int b = c & 1;
            if (c >= 2 && !(ok = gt_wait(&wempty[b], (uint32_t)((c / 2 - 1) & 1), P.timeout_ns))) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&wfull[b], F::WBUF);
                tma_load_2d_plain(smem + F::W_OFF + b * F::WBUF, &P.tmw, (c0 + c) * (F::WB / 4), (int)r0, &wfull[b]);
            }
            issued = c + 1;
        }
        for (int c = max(0, issued - 2); c < issued; ++c)
            gt_wait(&wfull[c & 1], (uint32_t)((c / 2) & 1), drain_bound(P.timeout_ns));
    } else if (warp == GT_MMA_WARP) {
        // ---- MMA issue (one thread).  Per tile and 16-column half: A_hi
        // against B (256 rows, hi then lo), then A_lo against B's hi rows.
        if (lane == 0) {
            const uint64_t a0 = gt_desc(sbase + F::A_OFF), b0 = gt_desc(sbase + F::B_OFF);
            for (int s = 0; s < nsteps; ++s) {
                const int sb = s % NSB, sa = s % NSA;
                if (!(ok = gt_wait1(&afull[sa], (uint32_t)((s / NSA) & 1), P.timeout_ns) &&
                           gt_wait1(&bfull[sb], (uint32_t)((s / NSB) & 1), P.timeout_ns)))
                    break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                // descriptor start addresses advance in 16-byte units
                const uint64_t ah = a0 + ((uint64_t)sa * GT_ASTEP >> 4), al = ah + (GT_ASTEP / 2 >> 4);
                const uint64_t bs = b0 + ((uint64_t)sb * F::BSTEP >> 4);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint64_t ko = (uint64_t)h * (2 * GT_LBO >> 4);
                    const uint32_t acc = (s | h) != 0 ? 1u : 0u;
#pragma unroll
                    for (int t = 0; t < NX; ++t)
                        if (t < ntile) gt_mma(tmem + 256u * t, ah + ko, bs + t * (GT_XSTEP >> 4) + ko, GT_IDESC256, acc);
#pragma unroll
                    for (int t = 0; t < NX; ++t)
                        if (t < ntile) gt_mma(tmem + 256u * t, al + ko, bs + t * (GT_XSTEP >> 4) + ko, GT_IDESC128, 1u);
                }
                gt_commit(&bempty[sb]);
                gt_commit(&aempty[sa]);
            }
            gt_commit(dfull);                              // completes once every MMA issued above has
            if (!gt_wait1(dfull, 0, drain_bound(P.timeout_ns))) ok = false;   // before the memory is freed
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    } else if (bi >= 0) {
        // ---- A: thread (row rr, 16-column half hk) per step; rows past the
        // matrix read the tensor copy's zero fill (w = 0)
        const int rr = 16 * bi + (lane & 15), hk = lane >> 4;
        const float tv = r0 + rr < P.rows ? P.tinv[r0 + rr] : 0.f;
        const uint32_t aoff = F::A_OFF + (uint32_t)(rr >> 3) * GT_SBO + (uint32_t)(rr & 7) * 16 + (uint32_t)hk * 2 * GT_LBO;
        for (int c = 0; c < nchunk; ++c) {
            const int b = c & 1;
            if (ok) ok = gt_wait(&wfull[b], (uint32_t)((c / 2) & 1), P.timeout_ns);
            const uint32_t wrow = sbase + F::W_OFF + (uint32_t)b * F::WBUF + (uint32_t)rr * F::WB;
            uint4 hd = make_uint4(0u, 0u, 0u, 0u);
            if (FMT == FMT_Q4_K) hd = lds128u(wrow);
            float2 dsc = make_float2(0.f, 0.f), dm = dsc;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int s = 8 * c + j, sa = s % NSA;
                if (s >= NSA && ok) ok = gt_wait(&aempty[sa], (uint32_t)((s / NSA - 1) & 1), P.timeout_ns);
                float2 w[8];
                if (FMT == FMT_Q4_K) {
                    if ((j & 1) == 0) {
                        q4k_group_scales(hd.x, hd.y, hd.z, hd.w, j >> 1, dsc, dm);
                        dsc = __fmul2_rn(dsc, make_float2(tv, tv));    // exact: powers of two
                        dm = __fmul2_rn(dm, make_float2(tv, tv));
                    }
                    const float a = (j & 1) ? dsc.y : dsc.x, mn = (j & 1) ? dm.y : dm.x;
                    const uint4 qv = lds128u(wrow + 16 + 32 * (j >> 1) + 16 * hk);
                    const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t v = (qw[q] >> (4 * (j & 1))) & 0x0F0F0F0Fu;
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float2 cf = __fadd2_rn(make_float2(__uint_as_float(prmt(v, 0x4B000000u, 0x7440u + 2 * e)),
                                                                     __uint_as_float(prmt(v, 0x4B000000u, 0x7441u + 2 * e))),
                                                         make_float2(-8388608.0f, -8388608.0f));
                            w[2 * q + e] = __ffma2_rn(make_float2(a, a), cf, make_float2(-mn, -mn));
                        }
                    }
                } else {
                    const uint32_t blk = wrow + 34 * (uint32_t)j;
                    const float d = half_bits_to_float(lds32(blk & ~3u) >> ((blk & 2u) * 8)) * tv;
                    const uint32_t off = blk + 2 + 16 * (uint32_t)hk, a4 = off & ~3u, sh = (off & 3u) * 8;
                    uint32_t u[5];
#pragma unroll
                    for (int q = 0; q < 5; ++q) u[q] = lds32(a4 + 4 * q);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t v = funnel_r(u[q], u[q + 1], sh) ^ 0x80808080u;     // code + 128 per byte
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float2 cf = __fadd2_rn(make_float2(__uint_as_float(prmt(v, 0x4B000000u, 0x7440u + 2 * e)),
                                                                     __uint_as_float(prmt(v, 0x4B000000u, 0x7441u + 2 * e))),
                                                         make_float2(-8388736.0f, -8388736.0f));
                            w[2 * q + e] = __fmul2_rn(cf, make_float2(d, d));
                        }
                    }
                }
                uint32_t hi[8], lo[8];
                gt_split(w, hi, lo);
                const uint32_t ab = sbase + (uint32_t)sa * GT_ASTEP + aoff;
                sts128(ab, hi[0], hi[1], hi[2], hi[3]);
                sts128(ab + GT_LBO, hi[4], hi[5], hi[6], hi[7]);
                sts128(ab + GT_ASTEP / 2, lo[0], lo[1], lo[2], lo[3]);
                sts128(ab + GT_ASTEP / 2 + GT_LBO, lo[4], lo[5], lo[6], lo[7]);
                fence_proxy_async_smem();                  // the tensor cores read what was just stored
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&afull[sa]);
                    if (j == 7) mbar_arrive(&wempty[b]);
                }
            }
        }
    }
    // ---- epilogue: warps 0-7; warp w reads accumulator lanes 32 (w % 4) ..
    // + 31 (weight rows): NX = 1: x rows 64 (w / 4) .. + 63; NX = 2: x tile
    // w / 4.  Output = (w_hi x_hi + w_lo x_hi) + w_hi x_lo.
    if (warp < 8) {
        if (ok) ok = gt_wait(dfull, 0u, P.timeout_ns);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const int q4 = warp & 3, lr = 32 * q4 + lane;
        const int t = NX == 1 ? 0 : warp >> 2;                          // x tile
        const int cb = NX == 1 ? 64 * (warp >> 2) : 0, cn = NX == 1 ? 64 : 128;
        const int64_t r = r0 + lr, nb = (int64_t)(mt0 + t) * GT_XN + cb;
        const bool live = r < P.rows && t < ntile;
        const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16) + 256u * (uint32_t)t + (uint32_t)cb;
        if (ok && t < ntile) {
            const float tr = r < P.rows ? 1.0f / P.tinv[r] : 0.f;           // exact: a power of two
            float* part = P.ksplit > 1 ? P.part + (int64_t)ks * P.M * P.rows : nullptr;
#pragma unroll 1
            for (int c = 0; c < cn; c += 16) {
                uint32_t x0[16], x1[16];
                tmem_ld16(tl + (uint32_t)c, x0);
                tmem_ld16(tl + 128u + (uint32_t)c, x1);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int64_t n = nb + c + e;
                    const bool on = live && n < P.M;
                    const float v = __uint_as_float(x0[e]) + __uint_as_float(x1[e]);
                    if (part) {
                        if (on) part[n * P.rows + r] = v;
                    } else if (!P.pairs) {
                        if (on) P.Y[n * P.ld_y + r] = (v * tr) * __ldg(P.sn + n);
                    } else {
                        // gate in the even lane, up in the odd one (rows 2i, 2i + 1)
                        const float sv = on ? (v * tr) * __ldg(P.sn + n) : 0.f;
                        const float up = __shfl_xor_sync(0xFFFFFFFFu, sv, 1);
                        if (on && (lane & 1) == 0) P.Y[n * P.ld_y + (r >> 1)] = act_eval(P.act, sv) * up;
                    }
                }
            }
        }
    }
    if (!ok && lane == 0) record_status(P.status, STATUS_TIMEOUT);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == GT_MMA_WARP) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(F::TMEM_COLS));
    }
}

}  // namespace

cudaError_t gemm_set_smem() {
    cudaError_t e = cudaSuccess;
#define LQ_GT_SMEM(fmt, nx)                                                                               \
    if ((e = cudaFuncSetAttribute(gemm_tc_kernel<fmt, nx>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                  (int)GtF<fmt, nx>::TOTAL)) != cudaSuccess)                              \
        return e;
    LQ_GT_SMEM(FMT_Q4_K, 1)
    LQ_GT_SMEM(FMT_Q4_K, 2)
    LQ_GT_SMEM(FMT_Q8_0, 1)
    LQ_GT_SMEM(FMT_Q8_0, 2)
#undef LQ_GT_SMEM
    return cudaSuccess;
}

int gemm_tc_ksplit(int64_t rows, int64_t cols) {
    const int64_t nwt = (rows + GT_WR - 1) / GT_WR, nchunk = cols / 256;
    if (nwt >= GT_SPLIT_SMS / 2 || nchunk < 4) return 1;
    return (int)std::max<int64_t>(1, std::min<int64_t>({GT_SPLIT_SMS / nwt, nchunk / 2, 8}));
}

size_t gemm_tc_smem_bytes(int fmt) {
    return std::max<size_t>(fmt == FMT_Q4_K ? GtF<FMT_Q4_K, 1>::TOTAL : GtF<FMT_Q8_0, 1>::TOTAL,
                            fmt == FMT_Q4_K ? GtF<FMT_Q4_K, 2>::TOTAL : GtF<FMT_Q8_0, 2>::TOTAL);
}

cudaError_t gemm_tc_launch(int fmt, const GemmParams& P, const float* X, cudaStream_t st) {
    const int64_t nmt = P.nmt, mp = nmt * GT_XN;
    if (P.cols / 256 > 65535) return cudaErrorInvalidValue;
    const unsigned pgrid = (unsigned)(mp + (P.rows + 7) / 8);
    if (fmt == FMT_Q4_K)
        gemm_prep_kernel<FMT_Q4_K><<<pgrid, 256, 0, st>>>(X, P.M, mp, P.cols, P.sn, P.W, P.rows, P.rowbytes, P.tinv);
    else
        gemm_prep_kernel<FMT_Q8_0><<<pgrid, 256, 0, st>>>(X, P.M, mp, P.cols, P.sn, P.W, P.rows, P.rowbytes, P.tinv);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    gemm_ximg_kernel<<<dim3((unsigned)(mp / 8), (unsigned)(P.cols / 256)), 256, 0, st>>>(X, P.M, P.cols, P.sn, P.ximg);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t nwt = (P.rows + GT_WR - 1) / GT_WR;
    const int nx = nmt >= 2 ? 2 : 1;
    const int64_t grid = nwt * P.ksplit * ((nmt + nx - 1) / nx);
    if (grid > INT32_MAX) return cudaErrorInvalidValue;
#define LQ_GT_LAUNCH(f, x) gemm_tc_kernel<f, x><<<(unsigned)grid, GT_THREADS, GtF<f, x>::TOTAL, st>>>(P)
    if (fmt == FMT_Q4_K) {
        if (nx == 2) LQ_GT_LAUNCH(FMT_Q4_K, 2); else LQ_GT_LAUNCH(FMT_Q4_K, 1);
    } else {
        if (nx == 2) LQ_GT_LAUNCH(FMT_Q8_0, 2); else LQ_GT_LAUNCH(FMT_Q8_0, 1);
    }
#undef LQ_GT_LAUNCH
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (P.ksplit > 1) {
        if ((P.rows + 1023) / 1024 > 65535) return cudaErrorInvalidValue;
        if (P.pairs) {
            const dim3 rgrid((unsigned)P.M, (unsigned)((P.rows / 2 + 255) / 256));
            gemm_tc_reduce_pairs_kernel<<<rgrid, 256, 0, st>>>(P.part, P.ksplit, P.M, P.rows, P.tinv, P.sn, P.act,
                                                               P.Y);
        } else {
            const dim3 rgrid((unsigned)P.M, (unsigned)((P.rows + 1023) / 1024));
            gemm_tc_reduce_kernel<<<rgrid, 256, 0, st>>>(P.part, P.ksplit, P.M, P.rows, P.tinv, P.sn, P.Y);
        }
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace lq
