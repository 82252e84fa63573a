// lq_qmm.cu -- tensor-core matvec for a batch of up to eight x rows against
// Q4_K or Q8_0 weights (the batched decode / grouped MoE case): Y = X . W^T.
//
// What it computes is the matvec of lq_matvec (larql "Architecture -> Metal
// shader map", Gemma 3 / Llama tables; dotLLM matmul_q8_0 GEMV and PR #320
// MoeSwiGluMlp for the grouped experts); the tensor cores only replace the
// per-x-row multiply-adds.
//
// Q4_K.  Each 32-weight sub-block is factored as in the CUDA-core kernel
// (lq_group.cuh): sum_k w_k x_k = dsc * sum_k (q_k - qb) x_k + e * sum_k x_k,
// qb = round(dmin*m / dsc) clamped to [-16, 15], e = dsc*qb - dmin*m.
//  * A operand: the codes q - qb, exact in bf16 (|q - qb| <= 31): a LOP3
//    ORs two 4-bit codes into bf16 halves equal to 128 + q (high nibbles
//    shifted down first) and a bf16x2 subtraction of 128 + qb leaves q - qb.
//  * B operand: x = hi + lo with hi = bf16(x), lo = bf16(x - hi); the
//    residual is at most 2^-18 |x|, so the pieces carry x to well inside the
//    1e-5 relative tolerance.  The hi and lo MMAs of a sub-block chain into
//    one fp32 accumulator (exact products, fp32 sums).
//  * mma.sync m16n8k16 (bf16 in, fp32 accumulate) over the two 16-column
//    slices of a sub-block gives sum (q - qb) x for 16 rows x 8 x rows; the
//    epilogue multiplies by dsc and adds e * sum x (packed fp32 FMAs).
// Q8_0 (w = d q, no offset).  A is q itself in fp16: a LOP3 ORs the byte,
// sign bit flipped, into a half equal to 1152 + q and a half2 subtraction
// of 1152 leaves q, exact.  B is x / s in fp16 hi + lo pieces, s a power of
// two per (x row, 32-column block) with |x / s| < 2^15, so the pieces stay
// in fp16 range; the epilogue multiplies a block's MMA sum by d * s.
// The k index of a slice is permuted identically for A and B so that a lane
// loads its codes for both slices (and, Q4_K, both nibbles) of a 32-byte
// quant run with one 8-byte shared load: lane (g, c) takes bytes 8c..8c+7
// of the run; slice h uses bytes 8c+4h..8c+4h+3, whose bytes (0, 2) fill
// its k pair (2c, 2c+1) and bytes (1, 3) the pair (2c+8, 2c+9).
//
// GB300 structure: a CTA has eight consumer warps and a producer warp.
// Tiles are 64 weight rows x 512 (Q4_K) or 256 (Q8_0) columns, streamed
// into a ring of shared-memory stages by 2-D tensor copies (TMA, one box
// per tile, or eight 8-row boxes for gate / up pairs) on full / empty
// mbarriers (bounded waits).  Warps w and w + 4 take the same 16 rows and
// the two halves of every tile, and add their partial sums at the end.  Row
// blocks are dealt to the clusters in units of up to four, round robin; a
// cluster takes the blocks of a unit that read the same x rows as one
// group, and for each column chunk the x rows are staged
// once (their own bulk copies and barriers), converted once into B
// fragments and per-block sums or scales, and used by every row block of
// the group, whose partial sums stay in registers.  Each warp decodes the
// scales of its own 16 rows into a private table, so a tile needs no
// CTA-wide barrier.  Every output's sum runs in a fixed order: the result
// is deterministic.  Matrices with few row blocks (a down projection: 4096
// rows but 14336 columns) split the column chunks over the CTAs of the
// cluster: ranks 1.. store their partial sums into rank 0's shared memory
// (distributed shared memory, tx-counted stores, bounded waits) and rank 0
// adds them in rank order and writes the outputs.  Gate / up pairs: the
// producer lays the gate rows of pairs 8q .. 8q+7 of a tile out as tile
// rows 16q .. 16q+7 and their up rows as 16q+8 .. 16q+15 (an MMA lane holds
// rows g and g + 8), and the activation is applied within the lane that
// holds both.
#include "lq_group.cuh"
#include "lq_internal.h"

namespace lq {
namespace {

constexpr int NT = QMM_NT;                 // x rows per pass
constexpr int RT = QMM_RT;                 // weight rows per tile
constexpr int GR = QMM_GROUP;              // row blocks sharing one staging of x
constexpr int RW = RT / 16;                // warps per column half (16 rows each)
constexpr int NW = 2 * RW;                 // consumer warps: (row quarter, half of the tile's columns)

// Tile geometry per weight format: Q4_K tiles are two super-blocks (512
// columns, 288 bytes of a row), Q8_0 tiles eight blocks (256 columns, 272
// bytes).  A (sub-)block is 32 columns either way.
template <int FMT>
struct QF {
    static constexpr int KC = FMT == FMT_Q4_K ? 512 : 256;    // columns per tile
    static constexpr int WROW = FMT == FMT_Q4_K ? 288 : 272;  // weight bytes of a row per tile
    static constexpr int SB = KC / 32;                        // 32-column blocks per tile
    static constexpr int SBW = SB / 2;                        // blocks per warp
    static constexpr int WSTAGE = RT * WROW;                  // weight bytes per stage
    static constexpr int XSTR = KC * 4 + 16;                  // shared stride of an x row (bank spread)
    static constexpr int SCLB = FMT == FMT_Q4_K ? 16 : 8;     // bytes of a (row, block) scale entry
    static constexpr int SUBB = FMT == FMT_Q4_K ? 4 : 0;      // bytes of a subtrahend entry
};
static_assert(QF<FMT_Q4_K>::KC == QMM_KC && QF<FMT_Q8_0>::KC == QMM_KC8, "tile widths");

// Scales of one (row, sub-block), paired for the packed FMAs of the
// epilogue: (dsc, dsc, e, e).  The bf16x2 subtrahends 128 + qb of rows g and
// g + 8 sit side by side in a separate table (one 8-byte load).
struct SbScale {
    float dsc, dsc2, e, e2;
};

struct Layout {
    size_t wst, xraw, bfr, sx, scl, sub, half, red, bars, total;
};

// red: [csize-1][gmax][RW*32] partial sums of the other ranks (rank 0 only);
// half: [gmax][RW*32] partial sums of the second-half warps.
template <int FMT>
__host__ __device__ inline Layout qmm_layout(int nstages, int csize, int gmax) {
    using F = QF<FMT>;
    Layout L;
    size_t o = 0;
    L.wst = o;  o += (size_t)nstages * F::WSTAGE;
    L.xraw = o; o += (size_t)NT * F::XSTR;
    L.bfr = o;  o += sizeof(uint4) * 2 * F::SB * 32;
    L.sx = o;   o += sizeof(float) * F::SB * NT;
    L.scl = o;  o += (size_t)F::SCLB * NW * F::SBW * 16;
    L.sub = o;  o += (size_t)F::SUBB * NW * F::SBW * 16;
    L.half = o; o += sizeof(float4) * gmax * RW * 32;
    L.red = o;  o += sizeof(float4) * (csize - 1) * gmax * RW * 32;
    L.bars = o; o += sizeof(uint64_t) * (2 * nstages + 4) + 16;
    L.total = o;
    return L;
}

__device__ __forceinline__ int seg_nval(const Seg& S) {
    int n = S.bcnt ? (*S.bcnt - S.b0) : S.nbatch;
    return n < 0 ? 0 : (n > NT ? NT : n);
}
__device__ __forceinline__ int seg_boff(const Seg& S) { return (S.boff ? *S.boff : 0) + S.b0; }
__device__ __forceinline__ bool same_x(const Seg& a, const Seg& b) {
    return a.x == b.x && a.xmap == b.xmap && a.boff == b.boff && a.bcnt == b.bcnt && a.b0 == b.b0 &&
           a.nbatch == b.nbatch;
}

// Row blocks are dealt to the clusters in units of gmax consecutive blocks,
// round robin (unit u goes to cluster u mod ncl), so that blocks with nothing
// to do (a grouped-MoE segment past its expert's token count) spread over
// the clusters.  A group is up to gmax blocks of one unit that have x rows
// to process and read the x rows of the first; segments' tile0 = first row
// block.
struct Group {
    int n;
    int rb[GR];
    int sg[GR];
};

struct Walk {
    int u, pos, end, hint;
};

__device__ __forceinline__ void walk_start(Walk& w, int cid, int gmax, int nblocks) {
    w.u = cid;
    w.pos = cid * gmax;
    w.end = min(nblocks, w.pos + gmax);
    w.hint = 0;
}

__device__ __forceinline__ bool next_group(const Seg* segs, int nseg, int gmax, int nblocks, int ncl, Walk& w,
                                           Group& G) {
    for (;;) {
        if (w.pos >= w.end) {                      // next unit of this cluster
            w.u += ncl;
            w.pos = w.u * gmax;
            if (w.pos >= nblocks) return false;
            w.end = min(nblocks, w.pos + gmax);
        }
        G.n = 0;
        while (w.pos < w.end) {
            int s = w.hint;
            while (s + 1 < nseg && w.pos >= segs[s + 1].tile0) ++s;
            while (s > 0 && w.pos < segs[s].tile0) --s;
            w.hint = s;
            if (seg_nval(segs[s]) <= 0) {          // nothing to do for this segment
                w.pos = min(w.end, segs[s].tile0 + segs[s].ntiles);
                continue;
            }
            if (G.n > 0 && !same_x(segs[G.sg[0]], segs[s])) break;
#pragma unroll
            for (int k = 0; k < GR; ++k)
                if (k == G.n) {
                    G.rb[k] = w.pos;
                    G.sg[k] = s;
                }
            ++G.n;
            ++w.pos;
        }
        if (G.n > 0) return true;
    }
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d = a . b (no accumulator input)
__device__ __forceinline__ void mma_bf16_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// half2 (lo = b, hi = a), round to nearest
__device__ __forceinline__ uint32_t f16x2_pack(float hi, float lo) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
__device__ __forceinline__ float f16_lo_f(uint32_t v) { return half_bits_to_float(v); }
__device__ __forceinline__ float f16_hi_f(uint32_t v) { return half_bits_to_float(v >> 16); }
// fp16 B fragments of (already scaled) x columns (c0, c1, c2, c3) of one k
// slice, hi then lo pieces, in the k order of bf16 ones below
__device__ __forceinline__ uint4 x_frag_h(float4 a) {
    const uint32_t h0 = f16x2_pack(a.z, a.x), h1 = f16x2_pack(a.w, a.y);
    return make_uint4(h0, h1, f16x2_pack(a.z - f16_hi_f(h0), a.x - f16_lo_f(h0)),
                      f16x2_pack(a.w - f16_hi_f(h1), a.y - f16_lo_f(h1)));
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
// bf16x2 (v, v) of a float with at most 8 significant bits (exact: the
// upper half of its fp32 encoding)
__device__ __forceinline__ uint32_t bf16_dup(float v) { return __byte_perm(__float_as_uint(v), 0u, 0x3232); }
__device__ __forceinline__ uint64_t u64_of(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}

__device__ __forceinline__ void consumer_bar() {
    asm volatile("bar.sync 1, %0;" ::"r"(NW * 32) : "memory");
}
// the first super-block warps only
__device__ __forceinline__ void half_bar() {
    asm volatile("bar.sync 2, %0;" ::"r"(RW * 32) : "memory");
}

// bounded wait by lane 0, result broadcast to the warp
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns, int lane) {
    bool ok = true;
    if (lane == 0) ok = mbar_wait_bounded(bar, parity, timeout_ns);
    return __shfl_sync(0xFFFFFFFFu, ok, 0);
}

template <int FMT>
__global__ void __launch_bounds__(32 * (NW + 1), 2) qmm_kernel(const __grid_constant__ QmmParams P) {
    using F = QF<FMT>;
    constexpr int KC = F::KC, WROW = F::WROW, SB = F::SB, SBW = F::SBW, WSTAGE = F::WSTAGE, XSTR = F::XSTR;
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_launch_dependents();
    const int S_ = P.nstages, cs = P.csize, gmax = P.gmax;
    const Layout L = qmm_layout<FMT>(S_, cs, gmax);
    uint8_t* wst = smem + L.wst;
    uint8_t* xraw = smem + L.xraw;
    uint4* bfr = reinterpret_cast<uint4*>(smem + L.bfr);       // [2*SB k-slices][32 lanes]
    float* sxs = reinterpret_cast<float*>(smem + L.sx);        // [SB][NT] Q4_K: sums of x per sub-block; Q8_0: x scales
    uint8_t* sclb = smem + L.scl;                              // [NW][SBW][16 rows] scale entries
    uint32_t* subt = reinterpret_cast<uint32_t*>(smem + L.sub); // [NW][SBW][8][rows g, g+8]
    float4* halfb = reinterpret_cast<float4*>(smem + L.half);  // [gmax][RW*32]
    float4* red = reinterpret_cast<float4*>(smem + L.red);     // [csize-1][gmax][RW*32]
    const Seg* segs = P.seg;                                    // kernel parameter space
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + S_;
    uint64_t* xfull = empty + S_;
    uint64_t* xempty = xfull + 1;
    uint64_t* red_full = xempty + 1;          // rank 0: the other ranks' partial sums of a group have landed
    uint64_t* red_free = red_full + 1;        // ranks 1..: rank 0 has read them
    int* abort_flag = reinterpret_cast<int*>(red_free + 1);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (warp == NW && lane < P.nseg) {
        prefetch_tensormap(&P.tm[lane][0]);
        if (segs[lane].mode != MODE_PLAIN) prefetch_tensormap(&P.tm[lane][1]);
    }
    if (tid == 0) {
        for (int s = 0; s < S_; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        mbar_init(xfull, 1);
        mbar_init(xempty, NW);
        if (cs > 1) {
            mbar_init(red_full, 1);
            mbar_init(red_free, 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // peers' barriers are initialised before any remote access: each thread
    // waits on this arrive before its first one
    bool cw = cs <= 1;
    if (cs > 1) cluster_arrive();
    const uint32_t rank = cs > 1 ? cluster_ctarank() : 0u;

    // this rank's column chunks of every row block
    const int c0 = (int)((int64_t)rank * P.nchunk / cs), c1 = (int)((int64_t)(rank + 1) * P.nchunk / cs);
    // this cluster's units of row blocks
    const int ncl = gridDim.x / cs, cid = blockIdx.x / cs;

    if (warp == NW) {
        // ------------------------------------------------ producer warp
        const uint64_t policy = policy_evict_first();
        // weights do not depend on the preceding kernel: unless the row
        // counts do, the first tiles are requested before waiting for it
        bool waited = P.dev_counts == 0 ? false : (pdl_wait(), true);
        Walk wk;
        walk_start(wk, cid, gmax, P.nblocks);
        Group G{};
        uint32_t ephase = 0;
        int last_use[8];
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) last_use[s2] = -1;
        bool ok = true;
        int n = 0, s = 0, xn = 0;
        auto issue_tile = [&](int k, int c) {
            int rbk = G.rb[0], sgk = G.sg[0];
#pragma unroll
            for (int kk = 1; kk < GR; ++kk)
                if (kk == k) {
                    rbk = G.rb[kk];
                    sgk = G.sg[kk];
                }
            const Seg& S = segs[sgk];
            const int lrb = rbk - S.tile0;                // row block within the segment
            if (n >= S_) {
                ok = warp_wait(&empty[s], (ephase >> s) & 1u, P.timeout_ns, lane);
                ephase ^= 1u << s;
                if (!ok) return;
            }
            uint8_t* dst = wst + (size_t)s * WSTAGE;
            // the whole tile (rows past the matrix are zero filled)
            if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)WSTAGE);
            __syncwarp();
            const int xw = c * (WROW / 4);                   // chunk start, uint32 elements
            if (S.mode == MODE_PLAIN) {
                if (lane == 0) tma_load_2d(dst, &P.tm[sgk][0], xw, lrb * RT, &full[s], policy);
            } else if (lane < 2 * RW) {
                // rows 16q .. 16q+7: gate rows of pairs p0 + 8q ..; 16q+8 ..: their up rows
                const int q = lane >> 1, u = lane & 1;
                tma_load_2d(dst + (16 * q + 8 * u) * WROW, &P.tm[sgk][u], xw, lrb * (RT / 2) + QMM_PAIR_BOX * q,
                            &full[s], policy);
            }
            last_use[s] = n / S_;
            ++n;
            if (++s == S_) s = 0;
        };
        while (ok && next_group(segs, P.nseg, gmax, P.nblocks, ncl, wk, G)) {
            const Seg& S0 = segs[G.sg[0]];
            for (int c = c0; c < c1 && ok; ++c) {
                if (*reinterpret_cast<volatile int*>(abort_flag)) {
                    ok = false;
                    break;
                }
                int k = 0;
                if (!waited) {                   // first chunk: tiles into the free stages first
                    for (; k < G.n && k < S_; ++k) issue_tile(k, c);
                    pdl_wait();
                    waited = true;
                }
                // x rows of this chunk (the buffer is free once converted)
                if (xn > 0 && !(ok = warp_wait(xempty, (uint32_t)(xn - 1) & 1u, P.timeout_ns, lane))) break;
                const int nval = seg_nval(S0), boff = seg_boff(S0);
                if (lane == 0) mbar_arrive_expect_tx(xfull, (uint32_t)(nval * KC * 4));
                __syncwarp();
                if (lane < nval) {
                    const int rho = boff + lane;
                    const float* xr = S0.x + (int64_t)(S0.xmap ? S0.xmap[rho] : rho) * P.cols + (int64_t)c * KC;
                    bulk_g2s(xraw + lane * XSTR, xr, KC * 4, xfull);
                }
                ++xn;
                for (; k < G.n && ok; ++k) issue_tile(k, c);
            }
        }
        if (!waited) pdl_wait();
        if (!ok && lane == 0) {
            record_status(P.status, STATUS_TIMEOUT);
            atomicExch(abort_flag, 1);
        }
        // no copy may still be in flight when the CTA exits
        if (lane == 0) {
            for (int s2 = 0; s2 < S_; ++s2)
                if (last_use[s2] >= 0)
                    mbar_wait_bounded(&full[s2], (uint32_t)last_use[s2] & 1u, drain_bound(P.timeout_ns));
            if (xn > 0) mbar_wait_bounded(xfull, (uint32_t)(xn - 1) & 1u, drain_bound(P.timeout_ns));
        }
        __syncwarp();
        if (cs > 1) {                            // no CTA leaves while a peer may address it
            cluster_wait();
            cluster_sync_all();
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    pdl_wait();
    const int g = lane >> 2, cq = lane & 3;
    const int rq = warp % RW, hb = warp / RW;    // rows 16*rq .. +15, super-block hb of each tile
    const int r0w = 16 * rq;
    const int rt = rq * 32 + lane;               // slot of this lane's partial sums
    Walk wk;
    walk_start(wk, cid, gmax, P.nblocks);
    Group G{};
    uint32_t fphase = 0, xph = 0;
    bool aborted = false;
    int s = 0, grp = 0;
    const uint32_t magic16 = 0x64006400u;        // half2 (1024, 1024), for the scale decode
    SbScale* sw = reinterpret_cast<SbScale*>(sclb + warp * (SBW * 16 * F::SCLB));   // Q4_K: [SBW][16]
    float2* sw8 = reinterpret_cast<float2*>(sclb + warp * (SBW * 16 * F::SCLB));     // Q8_0: [SBW][16] (d, d)
    uint32_t* subw = subt + warp * (SBW * 16);   // [SBW][8][2]
    auto fail = [&](void) {
        aborted = true;
        if (lane == 0) {
            record_status(P.status, STATUS_TIMEOUT);
            atomicExch(abort_flag, 1);
        }
    };
    while (next_group(segs, P.nseg, gmax, P.nblocks, ncl, wk, G)) {
        const int nval = seg_nval(segs[G.sg[0]]);
        float acc[GR][4];
#pragma unroll
        for (int k = 0; k < GR; ++k) acc[k][0] = acc[k][1] = acc[k][2] = acc[k][3] = 0.f;
        for (int c = c0; c < c1; ++c) {
            consumer_bar();                      // B fragments and half slots no longer read
            if (!aborted && !warp_wait(xfull, xph, P.timeout_ns, lane)) fail();
            xph ^= 1u;
            if (!aborted && FMT == FMT_Q8_0) {
                // x chunk -> fp16 B fragments of x / s (hi, lo per k slice), s a
                // power of two per (x row, block) with |x / s| < 2^15: unit
                // (block j, lane (tok, c4)) covers columns 32j + 8c4 .. +7
                const int tok = lane >> 2, c4 = lane & 3;
#pragma unroll
                for (int it = 0; it < (SB + NW - 1) / NW; ++it) {
                    const int j = warp + NW * it;
                    if (j < SB) {
                        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
                        if (tok < nval) {
                            const float* xr = reinterpret_cast<const float*>(xraw + tok * XSTR) + 32 * j + 8 * c4;
                            a = *reinterpret_cast<const float4*>(xr);
                            b = *reinterpret_cast<const float4*>(xr + 4);
                        }
                        float m = fmaxf(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))),
                                        fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w))));
                        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
                        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
                        const int es = max(1, (int)((__float_as_uint(m) >> 23) & 0xFFu) - 14);  // biased exponent of s
                        const float inv = __uint_as_float((uint32_t)(254 - es) << 23);        // 1 / s, exact
                        a = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
                        b = make_float4(b.x * inv, b.y * inv, b.z * inv, b.w * inv);
                        bfr[(2 * j) * 32 + lane] = x_frag_h(a);
                        bfr[(2 * j + 1) * 32 + lane] = x_frag_h(b);
                        if (c4 == 0) sxs[j * NT + tok] = __uint_as_float((uint32_t)es << 23);
                    }
                }
            }
            if (!aborted && FMT == FMT_Q4_K) {
                // x chunk -> B fragments (hi, lo per k slice) and sums per sub-block:
                // unit (sub-block j, lane (tok, c4)) covers columns 32j + 8c4 .. +7
                const int tok = lane >> 2, c4 = lane & 3;
#pragma unroll
                for (int it = 0; it < SB / NW; ++it) {
                    const int j = warp + NW * it;
                    uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
                    float sum = 0.f;
                    if (tok < nval) {
                        const float* xr = reinterpret_cast<const float*>(xraw + tok * XSTR) + 32 * j + 8 * c4;
                        const float4 a = *reinterpret_cast<const float4*>(xr);
                        const float4 b = *reinterpret_cast<const float4*>(xr + 4);
                        uint32_t h0 = bf16x2_pack(a.z, a.x), h1 = bf16x2_pack(a.w, a.y);
                        v0 = make_uint4(h0, h1, bf16x2_pack(a.z - bf16_hi_f(h0), a.x - bf16_lo_f(h0)),
                                        bf16x2_pack(a.w - bf16_hi_f(h1), a.y - bf16_lo_f(h1)));
                        h0 = bf16x2_pack(b.z, b.x);
                        h1 = bf16x2_pack(b.w, b.y);
                        v1 = make_uint4(h0, h1, bf16x2_pack(b.z - bf16_hi_f(h0), b.x - bf16_lo_f(h0)),
                                        bf16x2_pack(b.w - bf16_hi_f(h1), b.y - bf16_lo_f(h1)));
                        sum = ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w));
                    }
                    bfr[(2 * j) * 32 + lane] = v0;
                    bfr[(2 * j + 1) * 32 + lane] = v1;
                    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
                    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
                    if (c4 == 0) sxs[j * NT + tok] = sum;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(xempty);      // raw x may be overwritten
            consumer_bar();                          // B fragments ready
            for (int k = 0; k < G.n; ++k) {
                if (!aborted && !warp_wait(&full[s], (fphase >> s) & 1u, P.timeout_ns, lane)) fail();
                fphase ^= 1u << s;
                const uint8_t* st = wst + (size_t)s * WSTAGE;
                float t[4] = {0.f, 0.f, 0.f, 0.f};
                if (!aborted && FMT == FMT_Q8_0) {
                    // block scales of this warp's 16 rows, blocks 4hb .. 4hb+3:
                    // lane -> (row lane & 15, blocks 2 (lane >> 4) + {0, 1})
                    {
                        const int rr = lane & 15, jq = lane >> 4;
#pragma unroll
                        for (int gi = 0; gi < 2; ++gi) {
                            const int jj = 2 * jq + gi;
                            const uint16_t dh =
                                *reinterpret_cast<const uint16_t*>(st + (r0w + rr) * WROW + 34 * (SBW * hb + jj));
                            const float d = half_bits_to_float(dh);
                            sw8[jj * 16 + rr] = make_float2(d, d);
                        }
                    }
                    __syncwarp();
                    // codes: int8 q as fp16 1152 + q (LOP3 with the byte's sign
                    // bit flipped) minus 1152, exact; one MMA operand per byte
                    const uint8_t* wg = st + (r0w + g) * WROW + 2 + 8 * cq;   // + 34 j: this lane's 8 codes of block j
                    const uint8_t* wg8 = wg + 8 * WROW;
                    uint64_t t01 = pk2(0.f, 0.f), t23 = pk2(0.f, 0.f);
                    const uint4* bfl = bfr + (2 * SBW * hb) * 32 + lane;
                    const float* sxq = sxs + SBW * hb * NT + 2 * cq;
#pragma unroll
                    for (int jj = 0; jj < SBW; ++jj) {
                        uint32_t wa[2], wb[2];
                        lds_words_any2<2>(wg + 34 * (SBW * hb + jj), wa);
                        lds_words_any2<2>(wg8 + 34 * (SBW * hb + jj), wb);
                        const float2 da = sw8[jj * 16 + g], db = sw8[jj * 16 + g + 8];
                        float d[4];
#pragma unroll
                        for (int hs = 0; hs < 2; ++hs) {
                            const uint32_t msk = 0x00FF00FFu, mag = 0x64806480u;   // half2 (1152, 1152)
                            uint32_t a[4];
                            a[0] = hsub2_u32(lop_and_xor(wa[hs], msk, mag), mag);
                            a[1] = hsub2_u32(lop_and_xor(wb[hs], msk, mag), mag);
                            a[2] = hsub2_u32(lop_and_xor(wa[hs] >> 8, msk, mag), mag);
                            a[3] = hsub2_u32(lop_and_xor(wb[hs] >> 8, msk, mag), mag);
                            const uint4 bf = bfl[(2 * jj + hs) * 32];
                            if (hs == 0)
                                mma_f16_z(d, a, bf.x, bf.y);
                            else
                                mma_f16(d, a, bf.x, bf.y);
                            mma_f16(d, a, bf.z, bf.w);
                        }
                        const uint64_t sv = *reinterpret_cast<const uint64_t*>(sxq + jj * NT);   // s of x rows 2cq, 2cq+1
                        const uint64_t z = pk2(0.f, 0.f);
                        t01 = ffma2(ffma2(u64_of(__float_as_uint(da.x), __float_as_uint(da.y)), sv, z), pk2(d[0], d[1]), t01);
                        t23 = ffma2(ffma2(u64_of(__float_as_uint(db.x), __float_as_uint(db.y)), sv, z), pk2(d[2], d[3]), t23);
                    }
                    t[0] = lo_f(t01);
                    t[1] = hi_f(t01);
                    t[2] = lo_f(t23);
                    t[3] = hi_f(t23);
                }
                if (!aborted && FMT == FMT_Q4_K) {
                    // scales of this warp's 16 rows in super-block hb:
                    // lane -> (row lane & 15, sub-block pairs 2 (lane >> 4) + {0, 1})
                    {
                        const int rr = lane & 15, gh = lane >> 4;
                        const uint4 hdr = *reinterpret_cast<const uint4*>(st + (r0w + rr) * WROW + hb * 144);
                        const int si = ((rr & 7) << 1) | (rr >> 3);
#pragma unroll
                        for (int gi = 0; gi < 2; ++gi) {
                            const int gq = 2 * gh + gi;
                            const Q4Cent qc = q4k_centres(hdr, q4_sel(gq), magic16);
                            const int j0 = 2 * gq;
                            sw[j0 * 16 + rr] = SbScale{qc.dsc0, qc.dsc0, qc.e0, qc.e0};
                            sw[(j0 + 1) * 16 + rr] = SbScale{qc.dsc1, qc.dsc1, qc.e1, qc.e1};
                            subw[j0 * 16 + si] = bf16_dup(128.0f + qc.qb0);
                            subw[(j0 + 1) * 16 + si] = bf16_dup(128.0f + qc.qb1);
                        }
                    }
                    __syncwarp();
                    const uint8_t* wg = st + (r0w + g) * WROW + hb * 144 + 16 + 8 * cq;  // this lane's 8 bytes of a run
                    const uint8_t* wg8 = wg + 8 * WROW;
                    uint64_t t01 = pk2(0.f, 0.f), t23 = pk2(0.f, 0.f);   // rows g, g+8 x tokens 2cq, 2cq+1
                    const SbScale* swa = sw + g;
                    const uint2* subg = reinterpret_cast<const uint2*>(subw) + g;
                    const uint4* bfl = bfr + (2 * SBW * hb) * 32 + lane;
                    const float* sxq = sxs + SBW * hb * NT + 2 * cq;
#pragma unroll
                    for (int m = 0; m < SBW / 2; ++m) {                  // sub-block pairs (2m, 2m+1)
                        const uint2 wa = *reinterpret_cast<const uint2*>(wg + 32 * m);
                        const uint2 wb = *reinterpret_cast<const uint2*>(wg8 + 32 * m);
#pragma unroll
                        for (int nib = 0; nib < 2; ++nib) {
                            const int j = 2 * m + nib;                    // sub-block within the warp's half
                            const uint4 sa = *reinterpret_cast<const uint4*>(swa + j * 16);
                            const uint4 sb = *reinterpret_cast<const uint4*>(swa + j * 16 + 8);
                            const uint2 sub = subg[j * 8];                   // rows g, g + 8
                            float d[4];
#pragma unroll
                            for (int hs = 0; hs < 2; ++hs) {
                                const uint32_t Wa = (hs ? wa.y : wa.x) >> (4 * nib);
                                const uint32_t Wb = (hs ? wb.y : wb.x) >> (4 * nib);
                                const uint32_t msk = 0x000F000Fu, mag = 0x43004300u;
                                uint32_t a[4];
                                a[0] = bf16x2_sub(lop_and_or(Wa, msk, mag), sub.x);
                                a[1] = bf16x2_sub(lop_and_or(Wb, msk, mag), sub.y);
                                a[2] = bf16x2_sub(lop_and_or(Wa >> 8, msk, mag), sub.x);
                                a[3] = bf16x2_sub(lop_and_or(Wb >> 8, msk, mag), sub.y);
                                const uint4 bf = bfl[(2 * j + hs) * 32];
                                if (hs == 0)
                                    mma_bf16_z(d, a, bf.x, bf.y);
                                else
                                    mma_bf16(d, a, bf.x, bf.y);
                                mma_bf16(d, a, bf.z, bf.w);
                            }
                            const uint64_t sxv = *reinterpret_cast<const uint64_t*>(sxq + j * NT);
                            t01 = ffma2(u64_of(sa.x, sa.y), pk2(d[0], d[1]), t01);
                            t01 = ffma2(u64_of(sa.z, sa.w), sxv, t01);
                            t23 = ffma2(u64_of(sb.x, sb.y), pk2(d[2], d[3]), t23);
                            t23 = ffma2(u64_of(sb.z, sb.w), sxv, t23);
                        }
                    }
                    t[0] = lo_f(t01);
                    t[1] = hi_f(t01);
                    t[2] = lo_f(t23);
                    t[3] = hi_f(t23);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                if (++s == S_) s = 0;
#pragma unroll
                for (int kk = 0; kk < GR; ++kk)
                    if (kk == k) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[kk][i] += t[i];
                    }
            }
        }
        // ---- outputs of the group (barrier counts are the same for every
        // warp whatever its state, so that none is left waiting)
        if (hb == 1) {
#pragma unroll
            for (int k = 0; k < GR; ++k)
                if (k < G.n) halfb[k * (RW * 32) + rt] = make_float4(acc[k][0], acc[k][1], acc[k][2], acc[k][3]);
        }
        consumer_bar();
        if (hb == 0) {
            // super-block 0 + super-block 1 of every chunk of this rank
#pragma unroll
            for (int k = 0; k < GR; ++k)
                if (k < G.n) {
                    const float4 o = halfb[k * (RW * 32) + rt];
                    acc[k][0] += o.x;
                    acc[k][1] += o.y;
                    acc[k][2] += o.z;
                    acc[k][3] += o.w;
                }
            bool write = !aborted;
            if (cs > 1) {
                // split columns: partial sums meet in rank 0 (tx-counted remote
                // stores), added in rank order
                if (!cw) {
                    cluster_wait();
                    cw = true;
                }
                if (rank != 0) {
                    write = false;
                    if (!aborted && grp > 0 &&
                        !mbar_wait_bounded_cluster(red_free, (uint32_t)(grp - 1) & 1u, P.timeout_ns))
                        fail();
                    if (!aborted) {
                        const uint32_t rbar = mapa_shared(smem_u32(red_full), 0);
#pragma unroll
                        for (int k = 0; k < GR; ++k)
                            if (k < G.n) {
                                const float4* slot = red + ((size_t)(rank - 1) * gmax + k) * (RW * 32) + rt;
                                st_async_f4(mapa_shared(smem_u32(slot), 0),
                                            make_float4(acc[k][0], acc[k][1], acc[k][2], acc[k][3]), rbar);
                            }
                    }
                } else {
                    if (tid == 0)
                        mbar_arrive_expect_tx(red_full, (uint32_t)((cs - 1) * G.n * RW * 32 * sizeof(float4)));
                    if (!aborted && !mbar_wait_bounded_cluster(red_full, (uint32_t)grp & 1u, P.timeout_ns)) fail();
                    if (!aborted) {
                        for (int r = 1; r < cs; ++r) {
#pragma unroll
                            for (int k = 0; k < GR; ++k)
                                if (k < G.n) {
                                    const float4 p = red[((size_t)(r - 1) * gmax + k) * (RW * 32) + rt];
                                    acc[k][0] += p.x;
                                    acc[k][1] += p.y;
                                    acc[k][2] += p.z;
                                    acc[k][3] += p.w;
                                }
                        }
                    }
                    half_bar();                  // every reader is done with the slots
                    if (tid == 0)
                        for (int r = 1; r < cs; ++r) mbar_arrive_remote(mapa_shared(smem_u32(red_free), (uint32_t)r));
                    write = !aborted;
                }
            }
            if (write) {
#pragma unroll
                for (int k = 0; k < GR; ++k) {
                    if (k >= G.n) break;
                    // rows r0w+g, r0w+g+8 of the tile x tokens 2cq, 2cq+1
                    const float* v = acc[k];
                    const Seg& S = segs[G.sg[k]];
                    const int boff = seg_boff(S);
                    const int lrb = G.rb[k] - S.tile0;
                    if (S.mode == MODE_PLAIN) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int row = lrb * RT + r0w + g + (i >> 1) * 8;
                            const int tok = 2 * cq + (i & 1);
                            if (row < S.nout && tok < nval)
                                S.y[(int64_t)(boff + tok) * S.ld_y + row] = seg_out(S.cap, v[i]);
                        }
                    } else {
                        // row g is the gate row of pair p0 + 8 rq + g, row g + 8 its up row
                        const int out = lrb * (RT / 2) + QMM_PAIR_BOX * rq + g;
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            const int tok = 2 * cq + i;
                            if (out < S.nout && tok < nval)
                                S.y[(int64_t)(boff + tok) * S.ld_y + out] = act_eval(S.act, v[i]) * v[2 + i];
                        }
                    }
                }
            }
        }
        ++grp;
    }
    if (cs > 1) {
        if (!cw) cluster_wait();
        cluster_sync_all();
    }
}

}  // namespace

namespace {
const void* qmm_fn(int fmt) {
    return fmt == FMT_Q8_0 ? reinterpret_cast<const void*>(qmm_kernel<FMT_Q8_0>)
                           : reinterpret_cast<const void*>(qmm_kernel<FMT_Q4_K>);
}
}  // namespace

bool qmm_format_ok(int fmt) { return fmt == FMT_Q4_K || fmt == FMT_Q8_0; }
int qmm_kc(int fmt) { return fmt == FMT_Q8_0 ? QF<FMT_Q8_0>::KC : QF<FMT_Q4_K>::KC; }
int qmm_wrow(int fmt) { return fmt == FMT_Q8_0 ? QF<FMT_Q8_0>::WROW : QF<FMT_Q4_K>::WROW; }

cudaError_t qmm_set_smem(int fmt, int bytes) {
    return cudaFuncSetAttribute(qmm_fn(fmt), cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

size_t qmm_smem_bytes(int fmt, int nstages, int csize, int gmax) {
    return fmt == FMT_Q8_0 ? qmm_layout<FMT_Q8_0>(nstages, csize, gmax).total
                           : qmm_layout<FMT_Q4_K>(nstages, csize, gmax).total;
}

// Clusters of `csize` CTAs that can be resident at once (CTAs for csize 1).
cudaError_t qmm_max_resident(int fmt, int csize, size_t smem, int sms, int* out) {
    *out = 0;
    if (csize <= 1) {
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qmm_fn(fmt), 32 * (NW + 1), smem);
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
    return cudaOccupancyMaxActiveClusters(out, qmm_fn(fmt), &cfg);
}

cudaError_t qmm_launch(int fmt, const QmmParams& P, int grid, size_t smem, cudaStream_t st) {
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
    return cudaLaunchKernelExC(&cfg, qmm_fn(fmt), args);
}

}  // namespace lq
