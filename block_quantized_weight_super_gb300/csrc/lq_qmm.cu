// lq_qmm.cu -- tensor-core matvec for a batch of up to eight x rows against
// Q4_K weights (the batched decode / grouped MoE case): Y = X . W^T.
//
// What it computes is the matvec of lq_matvec (larql "Architecture -> Metal
// shader map", Gemma 3 / Llama tables; dotLLM PR #320 MoeSwiGluMlp for the
// grouped experts); the tensor cores only replace the per-x-row multiply-adds.
//
// Each 32-weight Q4_K sub-block is factored as in the CUDA-core kernel
// (lq_group.cuh): sum_k w_k x_k = dsc * sum_k (q_k - qb) x_k + e * sum_k x_k,
// qb = round(dmin*m / dsc) clamped to [-16, 15], e = dsc*qb - dmin*m.
//  * A operand: the codes q - qb, exact in bf16 (|q - qb| <= 31): a LOP3
//    ORs two 4-bit codes into bf16 halves equal to 128 + q (high nibbles
//    shifted down first) and a bf16x2 subtraction of 128 + qb leaves q - qb.
//  * B operand: x = hi + lo with hi = bf16(x), lo = bf16(x - hi); the
//    residual is at most 2^-18 |x|, so the pieces carry x to well inside the
//    1e-5 relative tolerance.  Columns 0..7 of one MMA are the hi pieces of
//    the eight x rows, of a second MMA the lo pieces.
//  * mma.sync m16n8k16 (bf16 in, fp32 accumulate) over the two 16-column
//    slices of a sub-block gives sum (q - qb) x_piece for 16 rows x 8 x rows;
//    the epilogue multiplies by dsc and adds e * sum x into fp32
//    accumulators held in registers.
// The k index inside a 16-column slice is permuted identically for A and B:
// lane (g, c) takes the bytes 4c..4c+3 of a row's 16-byte quant run, bytes
// (0, 2) fill its k pair (2c, 2c+1), bytes (1, 3) the pair (2c+8, 2c+9).
//
// GB300 structure: a CTA has four consumer warps (16 weight rows each) and a
// producer warp.  A tile is 64 weight rows x 512 columns plus the eight x
// rows' 512 columns, streamed into a ring of shared-memory stages by 1-D
// bulk copies (TMA), one per row, on full / empty mbarriers (bounded waits).
// A CTA walks its row blocks one after another, all column chunks of a row
// block in order, so every output's sum runs in a fixed order: the result is
// deterministic.  Matrices with few row blocks (a down projection: 4096 rows
// but 14336 columns) split the columns over the CTAs of a thread-block
// cluster: rank r takes an even share of the column chunks, ranks 1.. store
// their partial sums into rank 0's shared memory (distributed shared memory,
// an mbarrier per direction, bounded waits) and rank 0 adds them in rank
// order and writes the outputs.  Gate / up pairs: the producer lays gate row i and up row i
// of a pair segment out as tile rows 2i and 2i+1 (also for two separate
// matrices), and the activation is applied across that lane pair.
#include "lq_group.cuh"
#include "lq_internal.h"

namespace lq {
namespace {

constexpr int NT = QMM_NT;                 // x rows per pass
constexpr int RT = QMM_RT;                 // weight rows per tile
constexpr int KC = QMM_KC;                 // columns per tile
constexpr int NW = RT / 16;                // consumer warps
constexpr int SB = KC / 32;                // sub-blocks per tile
constexpr int WROW = KC / 256 * 144;       // weight bytes of a row per tile
constexpr int WBYTES = RT * WROW;          // weight bytes per stage
constexpr int XBYTES = NT * KC * 4;        // x bytes per stage
constexpr int STAGE = WBYTES + XBYTES;

__device__ __forceinline__ int seg_nval(const Seg& S) {
    int n = S.bcnt ? (*S.bcnt - S.b0) : S.nbatch;
    return n < 0 ? 0 : (n > NT ? NT : n);
}
__device__ __forceinline__ int seg_boff(const Seg& S) { return (S.boff ? *S.boff : 0) + S.b0; }
// weight rows of a segment (pairs count twice)
__device__ __forceinline__ int seg_rows(const Seg& S) { return S.mode == MODE_PLAIN ? S.nout : 2 * S.nout; }

struct QWalk {
    int rb, step, end, hint;               // row-block index (global over segments)
};

__device__ __forceinline__ void qwalk_fix(const Seg* segs, int nseg, QWalk& w) {
    while (w.rb < w.end) {
        int s = w.hint;
        while (s + 1 < nseg && w.rb >= segs[s + 1].tile0) ++s;
        while (s > 0 && w.rb < segs[s].tile0) --s;
        w.hint = s;
        if (seg_nval(segs[s]) > 0) return;
        w.rb += w.step;
    }
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                         const float (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// bf16x2 (lo = b, hi = a), round to nearest
__device__ __forceinline__ uint32_t bf16x2_pack(float hi, float lo) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
__device__ __forceinline__ float bf16_lo_f(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float act_f(int act, float g) {
    if (act == ACT_GEGLU_TANH) {
        const float z = 0.7978845608028654f * fmaf(0.044715f * g, g * g, g);
        return g / (1.0f + expf(-2.0f * z));
    }
    return g / (1.0f + expf(-g));
}

// Scales of one (row, sub-block): the bf16x2 subtrahend (base + qb term),
// the multiplier of the MMA sum and e.
struct SbScale {
    uint32_t sub;
    float dsc, e, pad;
};

struct Smem {
    uint8_t* stages;
    SbScale* scl;            // [RT][SB]
    uint4* bfr;              // [2*SB k-slices][32 lanes]: b0 hi, b1 hi, b0 lo, b1 lo
    float4* red;             // [csize-1][NW*32] partial sums of ranks 1.. (rank 0 only)
    float* sx;               // [NT][SB] sums of x per sub-block
    Seg* segs;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* red_full;      // rank 0: partials of a row block have arrived
    uint64_t* red_free;      // ranks 1..: rank 0 has read the previous partials
    int* abort_flag;
};

__device__ __forceinline__ void consumer_bar() {
    asm volatile("bar.sync 1, %0;" ::"r"(NW * 32) : "memory");
}

__global__ void __launch_bounds__(32 * (NW + 1), 2) qmm_q4k_kernel(const __grid_constant__ QmmParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_launch_dependents();
    const int S_ = P.nstages;
    Smem sm;
    size_t off = 0;
    sm.stages = smem;
    off += (size_t)S_ * STAGE;
    sm.scl = reinterpret_cast<SbScale*>(smem + off);
    off += sizeof(SbScale) * RT * SB;
    sm.bfr = reinterpret_cast<uint4*>(smem + off);
    off += sizeof(uint4) * 2 * SB * 32;
    const int cs = P.csize;
    sm.red = reinterpret_cast<float4*>(smem + off);
    off += sizeof(float4) * (cs - 1) * NW * 32;
    sm.sx = reinterpret_cast<float*>(smem + off);
    off += sizeof(float) * NT * SB;
    sm.segs = reinterpret_cast<Seg*>(smem + off);
    off += sizeof(Seg) * MAX_SEG;
    sm.full = reinterpret_cast<uint64_t*>(smem + off);
    sm.empty = sm.full + S_;
    sm.red_full = sm.empty + S_;
    sm.red_free = sm.red_full + 1;
    sm.abort_flag = reinterpret_cast<int*>(sm.red_free + 1);
    {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(&P.seg[0]);
        uint32_t* dst = reinterpret_cast<uint32_t*>(sm.segs);
        const int nw = P.nseg * (int)(sizeof(Seg) / 4);
        for (int i = threadIdx.x; i < nw; i += blockDim.x) dst[i] = src[i];
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < S_; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], NW);
        }
        if (cs > 1) {
            mbar_init(sm.red_full, (cs - 1) * NW * 32);
            mbar_init(sm.red_free, NW * 32);
        }
        *sm.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // peers' barriers are initialised before any remote arrive
    if (cs > 1) cluster_sync_all();
    const uint32_t rank = cs > 1 ? cluster_ctarank() : 0u;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nchunk = P.nchunk;
    // this rank's column chunks of every row block
    const int c0 = (int)((int64_t)rank * nchunk / cs), c1 = (int)((int64_t)(rank + 1) * nchunk / cs);
    const int64_t rowb = (int64_t)(P.cols / 256) * 144;
    QWalk w0;
    w0.rb = blockIdx.x / cs;                    // cluster index
    w0.step = gridDim.x / cs;
    w0.end = P.nblocks;
    w0.hint = 0;

    if (warp == NW) {
        // ------------------------------------------------ producer warp
        pdl_wait();                                  // x, row counts: preceding kernel
        const uint64_t policy = policy_evict_first();
        QWalk w = w0;
        qwalk_fix(sm.segs, P.nseg, w);
        uint32_t ephase = 0;
        int last_use[8];
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) last_use[s2] = -1;
        bool ok = true;
        int n = 0, s = 0;
        for (; w.rb < w.end && ok; w.rb += w.step, qwalk_fix(sm.segs, P.nseg, w)) {
            const Seg& S = sm.segs[w.hint];
            const int nval = seg_nval(S), boff = seg_boff(S);
            const int lrb = w.rb - S.tile0;          // row block within the segment
            const int nrow = seg_rows(S);
            for (int c = c0; c < c1; ++c, ++n) {
                if (*reinterpret_cast<volatile int*>(sm.abort_flag)) {
                    ok = false;
                    break;
                }
                if (n >= S_) {
                    if (lane == 0) ok = mbar_wait_bounded(&sm.empty[s], (ephase >> s) & 1u, P.timeout_ns);
                    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                    ephase ^= 1u << s;
                    if (!ok) break;
                }
                uint8_t* dst = sm.stages + (size_t)s * STAGE;
                // bytes of this tile: rows that exist, x rows that are valid
                int nr = 0;
                for (int tr = 0; tr < RT; ++tr) nr += (lrb * RT + tr < nrow) ? 1 : 0;
                if (lane == 0) mbar_arrive_expect_tx(&sm.full[s], (uint32_t)(nr * WROW + nval * KC * 4));
                __syncwarp();
#pragma unroll
                for (int h = 0; h < RT / 32; ++h) {
                    const int tr = lane + 32 * h;        // tile row
                    const int r = lrb * RT + tr;          // weight row of the segment (pairs interleaved)
                    if (r < nrow) {
                        const uint8_t* src;
                        if (S.mode == MODE_PAIR_TWO)
                            src = ((r & 1) ? S.w2 : S.w) + (int64_t)(r >> 1) * rowb;
                        else
                            src = S.w + (int64_t)r * rowb;
                        bulk_g2s_stream(dst + tr * WROW, src + (int64_t)c * WROW, WROW, &sm.full[s], policy);
                    }
                }
                if (lane < nval) {
                    const int rho = boff + lane;
                    const float* xr = S.x + (int64_t)(S.xmap ? S.xmap[rho] : rho) * P.cols + (int64_t)c * KC;
                    bulk_g2s(dst + WBYTES + lane * KC * 4, xr, KC * 4, &sm.full[s]);
                }
                last_use[s] = n / S_;
                if (++s == S_) s = 0;
            }
        }
        if (!ok && lane == 0) {
            record_status(P.status, STATUS_TIMEOUT);
            atomicExch(sm.abort_flag, 1);
        }
        if (lane == 0) {
            for (int s2 = 0; s2 < S_; ++s2)
                if (last_use[s2] >= 0)
                    mbar_wait_bounded(&sm.full[s2], (uint32_t)last_use[s2] & 1u, P.timeout_ns);
        }
        __syncwarp();
        if (cs > 1) cluster_sync_all();         // no CTA leaves while a peer may address it
        return;
    }

    // ---------------------------------------------------- consumer warps
    pdl_wait();
    const int g = lane >> 2, cq = lane & 3;
    const int ct = tid;                          // 0 .. NW*32-1
    QWalk w = w0;
    qwalk_fix(sm.segs, P.nseg, w);
    uint32_t fphase = 0;
    bool aborted = false;
    int s = 0, kb = 0;                           // kb: row blocks done by this CTA
    const uint32_t magic16 = 0x64006400u;        // half2 (1024, 1024), for the scale decode
    for (; w.rb < w.end; w.rb += w.step, qwalk_fix(sm.segs, P.nseg, w)) {
        const Seg& S = sm.segs[w.hint];
        const int nval = seg_nval(S), boff = seg_boff(S);
        float acc_hi[4] = {0.f, 0.f, 0.f, 0.f}, acc_lo[4] = {0.f, 0.f, 0.f, 0.f};
        for (int c = c0; c < c1; ++c) {
            if (!aborted) {
                bool ok = true;
                if (lane == 0) ok = mbar_wait_bounded(&sm.full[s], (fphase >> s) & 1u, P.timeout_ns);
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                if (!ok || *reinterpret_cast<volatile int*>(sm.abort_flag)) {
                    aborted = true;
                    if (lane == 0 && !ok) {
                        record_status(P.status, STATUS_TIMEOUT);
                        atomicExch(sm.abort_flag, 1);
                    }
                }
            }
            fphase ^= 1u << s;
            const uint8_t* st = sm.stages + (size_t)s * STAGE;
            const float* xs = reinterpret_cast<const float*>(st + WBYTES);
            if (!aborted) {
                // ---- phase A (all consumers): scales, x pieces, x sums
                // scales: (tile row, super-block) pairs, all 8 sub-blocks each
                for (int e = ct; e < RT * (SB / 8); e += NW * 32) {
                    const int tr = e / (SB / 8), sbk = e % (SB / 8);
                    const uint4 hdr = *reinterpret_cast<const uint4*>(st + tr * WROW + sbk * 144);
#pragma unroll
                    for (int gq = 0; gq < 4; ++gq) {
                        const Q4Sel sl = q4_sel(gq);
                        const Q4Cent qc = q4k_centres(hdr, sl, magic16);
                        SbScale* o = sm.scl + tr * SB + sbk * 8 + 2 * gq;
                        // codes arrive as 128 + q; subtract 128 + qb (exact in bf16)
                        const uint32_t s0 = bf16x2_pack(128.0f + qc.qb0, 128.0f + qc.qb0);
                        const uint32_t s1 = bf16x2_pack(128.0f + qc.qb1, 128.0f + qc.qb1);
                        o[0] = SbScale{s0, qc.dsc0, qc.e0, 0.f};
                        o[1] = SbScale{s1, qc.dsc1, qc.e1, 0.f};
                    }
                }
                // x pieces in B-fragment order: unit = (k-slice, lane)
                for (int e = ct; e < 2 * SB * 32; e += NW * 32) {
                    const int ks = e >> 5, ln = e & 31, tok = ln >> 2, c4 = ln & 3;
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (tok < nval) {
                        const float4 x = *reinterpret_cast<const float4*>(xs + tok * KC + 16 * ks + 4 * c4);
                        const uint32_t h0 = bf16x2_pack(x.z, x.x);      // (k 2c, 2c+1) = cols (4c, 4c+2)
                        const uint32_t h1 = bf16x2_pack(x.w, x.y);      // (k 2c+8, 2c+9) = cols (4c+1, 4c+3)
                        const uint32_t l0 = bf16x2_pack(x.z - bf16_hi_f(h0), x.x - bf16_lo_f(h0));
                        const uint32_t l1 = bf16x2_pack(x.w - bf16_hi_f(h1), x.y - bf16_lo_f(h1));
                        v = make_uint4(h0, h1, l0, l1);
                    }
                    sm.bfr[e] = v;
                }
                // sums of x per (x row, sub-block), in column order
                for (int e = ct; e < NT * SB; e += NW * 32) {
                    const int tok = e / SB, j = e % SB;
                    float sum = 0.f;
                    if (tok < nval) {
                        const float* xr = xs + tok * KC + 32 * j;
                        for (int i = 0; i < 32; ++i) sum += xr[i];
                    }
                    sm.sx[e] = sum;
                }
            }
            consumer_bar();
            if (!aborted) {
                // ---- phase B: warp rows r0 .. r0+15
                const int r0 = 16 * warp;
                const uint8_t* wg = st + (r0 + g) * WROW;
                const uint8_t* wg8 = st + (r0 + g + 8) * WROW;
#pragma unroll 2
                for (int j = 0; j < SB; ++j) {
                    const int sbk = j >> 3, jj = j & 7;
                    const int qoff = sbk * 144 + 16 + 32 * (jj >> 1) + 4 * cq;
                    const uint32_t nsh = (jj & 1) ? 4u : 0u;  // high nibbles: shift down
                    const SbScale sa = sm.scl[(r0 + g) * SB + j];
                    const SbScale sb = sm.scl[(r0 + g + 8) * SB + j];
                    float dh[4] = {0.f, 0.f, 0.f, 0.f}, dl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int hs = 0; hs < 2; ++hs) {
                        const uint32_t Wa = *reinterpret_cast<const uint32_t*>(wg + qoff + 16 * hs) >> nsh;
                        const uint32_t Wb = *reinterpret_cast<const uint32_t*>(wg8 + qoff + 16 * hs) >> nsh;
                        const uint32_t msk = 0x000F000Fu, mag = 0x43004300u;
                        uint32_t a[4];
                        a[0] = bf16x2_sub(lop_and_or(Wa, msk, mag), sa.sub);
                        a[1] = bf16x2_sub(lop_and_or(Wb, msk, mag), sb.sub);
                        a[2] = bf16x2_sub(lop_and_or(Wa >> 8, msk, mag), sa.sub);
                        a[3] = bf16x2_sub(lop_and_or(Wb >> 8, msk, mag), sb.sub);
                        const uint4 bf = sm.bfr[(2 * j + hs) * 32 + lane];
                        mma_bf16(dh, a, bf.x, bf.y, dh);
                        mma_bf16(dl, a, bf.z, bf.w, dl);
                    }
                    // epilogue: rows g, g+8; x rows 2cq, 2cq+1
                    const float sx0 = sm.sx[(2 * cq) * SB + j], sx1 = sm.sx[(2 * cq + 1) * SB + j];
                    acc_hi[0] = fmaf(sa.e, sx0, fmaf(sa.dsc, dh[0], acc_hi[0]));
                    acc_hi[1] = fmaf(sa.e, sx1, fmaf(sa.dsc, dh[1], acc_hi[1]));
                    acc_hi[2] = fmaf(sb.e, sx0, fmaf(sb.dsc, dh[2], acc_hi[2]));
                    acc_hi[3] = fmaf(sb.e, sx1, fmaf(sb.dsc, dh[3], acc_hi[3]));
                    acc_lo[0] = fmaf(sa.dsc, dl[0], acc_lo[0]);
                    acc_lo[1] = fmaf(sa.dsc, dl[1], acc_lo[1]);
                    acc_lo[2] = fmaf(sb.dsc, dl[2], acc_lo[2]);
                    acc_lo[3] = fmaf(sb.dsc, dl[3], acc_lo[3]);
                }
            }
            // release the stage and the per-tile tables
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
            consumer_bar();
            if (++s == S_) s = 0;
        }
        if (aborted) continue;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = acc_hi[i] + acc_lo[i];
        if (cs > 1) {
            // ---- split columns: partial sums meet in rank 0, added in rank order
            const int k = kb++;
            if (rank != 0) {
                if (k > 0 && !mbar_wait_bounded_cluster(sm.red_free, (uint32_t)(k - 1) & 1u, P.timeout_ns)) {
                    aborted = true;
                    record_status(P.status, STATUS_TIMEOUT);
                    atomicExch(sm.abort_flag, 1);
                    continue;
                }
                const uint32_t slot = smem_u32(sm.red + (size_t)(rank - 1) * NW * 32 + ct);
                st_cluster_f4(mapa_shared(slot, 0), v[0], v[1], v[2], v[3]);
                mbar_arrive_remote(mapa_shared(smem_u32(sm.red_full), 0));
                continue;                        // rank 0 writes the outputs
            }
            if (!mbar_wait_bounded_cluster(sm.red_full, (uint32_t)k & 1u, P.timeout_ns)) {
                aborted = true;
                record_status(P.status, STATUS_TIMEOUT);
                atomicExch(sm.abort_flag, 1);
                continue;
            }
            for (int r = 1; r < cs; ++r) {
                const float4 p = sm.red[(size_t)(r - 1) * NW * 32 + ct];
                v[0] += p.x;
                v[1] += p.y;
                v[2] += p.z;
                v[3] += p.w;
            }
            for (int r = 1; r < cs; ++r) mbar_arrive_remote(mapa_shared(smem_u32(sm.red_free), (uint32_t)r));
        }
        // ---- outputs of this row block: rows r0+g, r0+g+8 x rows 2cq, 2cq+1
        const int lrb = w.rb - S.tile0;
        const int trg = 16 * warp + g;                  // tile row of v[0], v[1]; +8 for v[2], v[3]
        if (S.mode == MODE_PLAIN) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = lrb * RT + trg + (i >> 1) * 8;
                const int tok = 2 * cq + (i & 1);
                if (row < S.nout && tok < nval) S.y[(int64_t)(boff + tok) * S.ld_y + row] = v[i];
            }
        } else {
            // gate rows are even tile rows, up rows odd: partner lane g ^ 1
            float u[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) u[i] = __shfl_xor_sync(0xFFFFFFFFu, v[i], 4);
            if ((g & 1) == 0) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int out = (lrb * RT + trg + (i >> 1) * 8) >> 1;
                    const int tok = 2 * cq + (i & 1);
                    if (out < S.nout && tok < nval)
                        S.y[(int64_t)(boff + tok) * S.ld_y + out] = act_f(S.act, v[i]) * u[i];
                }
            }
        }
    }
    if (cs > 1) cluster_sync_all();
}

}  // namespace

cudaError_t qmm_set_smem(int bytes) {
    return cudaFuncSetAttribute(qmm_q4k_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

size_t qmm_smem_bytes(int nstages, int csize) {
    return (size_t)nstages * STAGE + sizeof(SbScale) * RT * SB + sizeof(uint4) * 2 * SB * 32 +
           sizeof(float4) * (csize - 1) * NW * 32 + sizeof(float) * NT * SB + sizeof(Seg) * MAX_SEG +
           (2 * nstages + 2) * sizeof(uint64_t) + 16;
}

// Clusters of `csize` CTAs that can be resident at once (CTAs for csize 1).
cudaError_t qmm_max_resident(int csize, size_t smem, int sms, int* out) {
    *out = 0;
    if (csize <= 1) {
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qmm_q4k_kernel, 32 * (NW + 1), smem);
        *out = per_sm * sms;
        return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(csize * sms));
    cfg.blockDim = dim3(32 * (NW + 1));
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, reinterpret_cast<void*>(qmm_q4k_kernel), &cfg);
}

cudaError_t qmm_launch(const QmmParams& P, int grid, size_t smem, cudaStream_t st) {
    void* args[1] = {const_cast<QmmParams*>(&P)};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32 * (NW + 1));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (P.csize > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)P.csize;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<void*>(qmm_q4k_kernel), args);
}

}  // namespace lq
