#pragma once
// lq_qmv_impl.cuh -- the quantized matvec kernel (batch 1, 2 or 4 rows of x).
//
// y = W.x for Q4_K / Q6_K / Q8_0 weight rows (larql "Architecture -> Metal
// shader map", Gemma 3 table: q4k_matvec, q6k_matvec, q4k_q6k_qkv_proj,
// q4k_ffn_gate_up + geglu; dotLLM PR #320: matmul_q8_0 GEMV), over a list of
// segments (several matrices sharing x in one launch; gate/up row pairs with
// the activation fused before the store; MoE experts with gathered rows).
//
// GB300 structure:
//  * warp NC (the producer) streams row tiles of W into a ring of shared-
//    memory stages with 1-D bulk copies (TMA) on "full" mbarriers and reuses
//    a stage once its "empty" mbarrier says the consumers are done with it;
//  * warps 0..NC-1 (consumers) never synchronise with each other per tile:
//    each processes a fixed share of work items of every tile (an item = one
//    64-weight group of R consecutive rows, dequantized once and multiplied
//    with B x rows read from shared memory), writes per-group partials, and
//    the warp that finishes a tile last (shared counter) releases the stage
//    and sums that tile's partials in a fixed order into y;
//  * x for the current matrix is staged in shared memory (64-float group
//    slots padded to 68 floats so a warp's 16-byte reads hit distinct banks),
//    with per-sub-block sums of x for the Q4_K re-centred form;
//  * a CTA runs one block format (template), so the hot loop has no format
//    branch; mixed-format launches split the grid into two CTA groups;
//  * every wait is bounded by %globaltimer; on expiry the CTA records
//    STATUS_TIMEOUT, stops waiting, drains its copies (bounded) and exits.
// Results do not depend on B (each (row, x row) dot product is computed by
// the same instruction sequence) and are deterministic.
#include "lq_group.cuh"
#include "lq_internal.h"
#include "lq_qmv.cuh"

namespace lq {
namespace {

// ---------------------------------------------------------------- tiles

__device__ __forceinline__ int qseg_of(const QmvParams& P, int t, int hint) {
    int s = hint;
    while (s + 1 < P.nseg && t >= P.seg[s + 1].tile0) ++s;
    while (s > 0 && t < P.seg[s].tile0) --s;
    return s;
}

__device__ __forceinline__ int qseg_nval(const Seg& S, int B) {
    int n = S.bcnt ? (*S.bcnt - S.b0) : S.nbatch;
    return n < 0 ? 0 : (n > B ? B : n);
}

__device__ __forceinline__ int qseg_boff(const Seg& S) { return (S.boff ? *S.boff : 0) + S.b0; }

__device__ __forceinline__ int64_t qrow_bytes(int fmt, int cols) {
    return (int64_t)(cols / block_elems_of(fmt)) * block_bytes_of(fmt);
}

struct QTile {
    const uint8_t* src1;
    const uint8_t* src2;
    uint32_t bytes1, bytes2, dst2;
    int n_o, o0;
    bool tma;
};

__device__ __forceinline__ QTile qtile(const QGeo& Gm, const Seg& S, int t) {
    QTile g;
    const int64_t rb = qrow_bytes(S.fmt, Gm.cols);
    const int lt = t - S.tile0;
    const int opt = S.mode == MODE_PLAIN ? Gm.RT : Gm.RT / 2;
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
        g.dst2 = (uint32_t)((Gm.RT / 2) * rb);
    }
    g.tma = ((reinterpret_cast<uintptr_t>(g.src1) | g.bytes1) & 15u) == 0;
    if (S.mode == MODE_PAIR_TWO)
        g.tma = g.tma && ((reinterpret_cast<uintptr_t>(g.src2) | g.bytes2 | g.dst2) & 15u) == 0;
    return g;
}

// This CTA's tile walk: t = t0, t0 + step, ... < t_end over tiles of active
// segments (segments whose device-side row count is zero are skipped).
struct Walk {
    int t, step, end, hint;
};

__device__ __forceinline__ int qseg_of_s(const Seg* segs, int nseg, int t, int hint) {
    int s = hint;
    while (s + 1 < nseg && t >= segs[s + 1].tile0) ++s;
    while (s > 0 && t < segs[s].tile0) --s;
    return s;
}

template <int B>
__device__ __forceinline__ void walk_fix(const Seg* segs, int nseg, Walk& w) {
    while (w.t < w.end) {
        w.hint = qseg_of_s(segs, nseg, w.t, w.hint);
        if (qseg_nval(segs[w.hint], B) > 0) return;
        w.t += w.step;
    }
}

// 32 lanes copy n bytes global -> shared with plain loads (2-byte aligned)
__device__ __forceinline__ void warp_copy(uint8_t* dst, const uint8_t* src, uint32_t n, int lane) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(src);
    if ((a & 3u) == 0 && (n & 3u) == 0) {
        const uint32_t* s = reinterpret_cast<const uint32_t*>(src);
        uint32_t* d = reinterpret_cast<uint32_t*>(dst);
        for (uint32_t i = lane; i < n / 4; i += 32) d[i] = __ldg(s + i);
    } else {
        const uint16_t* s = reinterpret_cast<const uint16_t*>(src);
        uint16_t* d = reinterpret_cast<uint16_t*>(dst);
        for (uint32_t i = lane; i < n / 2; i += 32) d[i] = __ldg(s + i);
    }
}

// The CTA's abort flag as lane 0 reads it, for the whole warp: the warp's
// control flow (and the full-mask shuffles after it) stays uniform.
__device__ __forceinline__ bool warp_aborted(const int* flag, int lane) {
    int v = 0;
    if (lane == 0) v = *reinterpret_cast<const volatile int*>(flag);
    return __shfl_sync(0xFFFFFFFFu, v, 0) != 0;
}

__device__ __forceinline__ void consumer_sync(int nct) {
    asm volatile("bar.sync 1, %0;" ::"r"(nct) : "memory");
}

__device__ __forceinline__ float4 lds_f4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// ---------------------------------------------------------------- x staging

// column of x value i (0..63) of group G in the format's group order
template <int FMT>
__device__ __forceinline__ int qxcol(int G, int i) {
    if (FMT == FMT_Q6_K) {
        const int blk = G >> 2, gm = G & 3, h = gm >> 1, l0 = 16 * (gm & 1);
        return 256 * blk + 128 * h + 32 * (i >> 4) + l0 + (i & 15);
    }
    return 64 * G + i;
}

// Stage the B x rows of segment S into xs[(b*U + G)*68 + i] (64-float group
// slots padded to 68 floats) and, for Q4_K, sxs[(b*U + G)*2 + {0,1}] = sums
// of the low / high 32 columns of group G.  A unit is 16 consecutive columns
// (one 64-byte run of x, four float4; x rows are 16-byte aligned: the host
// checks); each thread loads two units before storing, and the sub-block
// sums come from registers: the 16-column sum of a unit (in column order)
// plus that of its neighbour unit (lane ^ 1).  Ends with the consumer barrier;
// the caller brackets it with one before.  COHERENT: x was written by other
// CTAs of this kernel, so it is read through L2 (no read-only path).  NU:
// units each thread loads before storing (all in flight at once).
template <int FMT, int B, bool COHERENT, int NU, bool XACT>
__device__ __forceinline__ void stage_x_body(const QGeo& Gm, const Seg& S, float* xs, float* sxs, int ct, int nct,
                                             bool wout) {
    const int U = Gm.U;
    const int nval = qseg_nval(S, B);
    const int boff = qseg_boff(S);
    const int units = B * U * 4;
    const int wbase = ct & ~31;                  // loop bound uniform over the warp
    const int64_t xstride = (int64_t)Gm.cols * (XACT ? 2 : 1);
    for (int e0 = ct, w0 = wbase; w0 < units; e0 += NU * nct, w0 += NU * nct) {
        float4 v[NU][4];
#pragma unroll
        for (int h = 0; h < NU; ++h) {
            const int e = e0 + h * nct;
            const int b = e / (U * 4), r = e % (U * 4), G = r >> 2, q = r & 3;
            if (e < units && b < nval) {
                const int rho = boff + b;
                const float* xrow = S.x + (int64_t)(S.xmap ? S.xmap[rho] : rho) * xstride;
                const int c0 = qxcol<FMT>(G, 16 * q);
#pragma unroll
                for (int k = 0; k < 4; ++k) v[h][k] = load_x4<COHERENT>(xrow, c0 + 4 * k, XACT ? S.xact : 0);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) v[h][k] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int h = 0; h < NU; ++h) {
            const int e = e0 + h * nct;
            const int b = e / (U * 4), r = e % (U * 4), G = r >> 2, q = r & 3;
            if (e < units) {
                float4* dst = reinterpret_cast<float4*>(xs + (b * U + G) * XS_STRIDE + 16 * q);
#pragma unroll
                for (int k = 0; k < 4; ++k) dst[k] = v[h][k];
                if (XACT && wout && b < nval) {
                    float* o = S.xout + (int64_t)(boff + b) * Gm.cols + qxcol<FMT>(G, 16 * q);
#pragma unroll
                    for (int k = 0; k < 4; ++k) *reinterpret_cast<float4*>(o + 4 * k) = v[h][k];
                }
            }
            if (FMT == FMT_Q4_K) {
                float s16 = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) s16 = ((s16 + v[h][k].x) + v[h][k].y) + v[h][k].z + v[h][k].w;
                const float s32 = s16 + __shfl_xor_sync(0xFFFFFFFFu, s16, 1);
                if (e < units && (q & 1) == 0) sxs[(b * U + G) * 2 + (q >> 1)] = s32;
            }
        }
    }
}

// With S.xact the staged values are act(g) * u of x's (g, u) pairs (one
// unit per thread in flight: the pairs take twice the registers), and when
// wout is set (the CTA staging for the segment's first tile) they are also
// stored to S.xout.
template <int FMT, int B, bool COHERENT = false, int NU = 2>
__device__ void stage_x(const QGeo& Gm, const Seg& S, float* xs, float* sxs, int ct, int nct, bool wout = false) {
    if (S.xact) stage_x_body<FMT, B, COHERENT, 1, true>(Gm, S, xs, sxs, ct, nct, wout);
    else stage_x_body<FMT, B, COHERENT, NU, false>(Gm, S, xs, sxs, ct, nct, false);
    consumer_sync(nct);
}

// Segments reading the same x rows (QKV: Q and K) need no second staging.
__device__ __forceinline__ bool same_xsrc(const Seg& a, const Seg& b) {
    return a.x == b.x && a.xmap == b.xmap && a.boff == b.boff && a.bcnt == b.bcnt && a.b0 == b.b0 &&
           a.nbatch == b.nbatch && a.xact == b.xact;
}

// Stage group G of the B x rows of segment S for the calling thread alone.
// For launches with one consumer thread per group (NCT == U: the down
// projections) every work item of a thread uses the same group, so each
// thread stages only what it reads itself: no barrier before or after, and
// a thread starts its items as soon as its own loads land instead of when the
// whole CTA's x (the L2 bandwidth of all CTAs together) has arrived.  The
// values and the sub-block sums (same order of additions) equal stage_x's.
template <int FMT, int B, bool COHERENT = false>
__device__ __forceinline__ void stage_x_own(const QGeo& Gm, const Seg& S, float* xs, float* sxs, int G,
                                            bool wout = false) {
    const int U = Gm.U;
    const int nval = qseg_nval(S, B);
    const int boff = qseg_boff(S);
    if (S.xact) {
        // act(g) * u of (g, u) pairs, one 16-column quarter at a time (the
        // pairs take twice the registers); the same values and sums
#pragma unroll 1
        for (int b = 0; b < B; ++b) {
            const int rho = boff + b;
            const float* xrow = b < nval ? S.x + (int64_t)(S.xmap ? S.xmap[rho] : rho) * (2 * (int64_t)Gm.cols)
                                         : nullptr;
            float slo = 0.f, shi = 0.f;
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                const int c0 = qxcol<FMT>(G, 16 * q);
                float4 v[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    v[k] = xrow ? load_x4<COHERENT>(xrow, c0 + 4 * k, S.xact) : make_float4(0.f, 0.f, 0.f, 0.f);
                float4* dst = reinterpret_cast<float4*>(xs + (b * U + G) * XS_STRIDE + 16 * q);
#pragma unroll
                for (int k = 0; k < 4; ++k) dst[k] = v[k];
                if (wout && xrow) {
                    float* o = S.xout + (int64_t)rho * Gm.cols + c0;
#pragma unroll
                    for (int k = 0; k < 4; ++k) *reinterpret_cast<float4*>(o + 4 * k) = v[k];
                }
                float s16 = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) s16 = ((s16 + v[k].x) + v[k].y) + v[k].z + v[k].w;
                if (q < 2) slo += s16;
                else shi += s16;
            }
            if (FMT == FMT_Q4_K) {
                sxs[(b * U + G) * 2] = slo;
                sxs[(b * U + G) * 2 + 1] = shi;
            }
        }
        return;
    }
#pragma unroll 1
    for (int b = 0; b < B; ++b) {
        float4 v[4][4];
        if (b < nval) {
            const int rho = boff + b;
            const float* xrow = S.x + (int64_t)(S.xmap ? S.xmap[rho] : rho) * Gm.cols;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4* src = reinterpret_cast<const float4*>(xrow + qxcol<FMT>(G, 16 * q));
#pragma unroll
                for (int k = 0; k < 4; ++k) v[q][k] = COHERENT ? __ldcg(src + k) : __ldg(src + k);
            }
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int k = 0; k < 4; ++k) v[q][k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float4* dst = reinterpret_cast<float4*>(xs + (b * U + G) * XS_STRIDE);
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int k = 0; k < 4; ++k) dst[4 * q + k] = v[q][k];
        if (FMT == FMT_Q4_K) {
            float s16[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                s16[q] = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) s16[q] = ((s16[q] + v[q][k].x) + v[q][k].y) + v[q][k].z + v[q][k].w;
            }
            sxs[(b * U + G) * 2] = s16[0] + s16[1];
            sxs[(b * U + G) * 2 + 1] = s16[2] + s16[3];
        }
    }
}

// ---------------------------------------------------------------- items
//
// An item is one 64-weight group G of R consecutive rows of the stage (row
// pointers rp) against B staged x rows; part[r][b] receives the dot
// product.  Accumulators are fp32 pairs (even / odd code positions of a
// word), combined in a fixed order at the end.

struct Q4Row {
    float c0, c1, dsc0, dsc1, e0, e1;
};

// Scales of quant group g of a Q4_K super-block (see lq_group.cuh) and the
// re-centring constants of its two sub-blocks.
__device__ __forceinline__ Q4Row q4k_row(const uint4 hdr, const Q4Sel& sl, const GroupConsts& K) {
    const Q4Cent c = q4k_centres(hdr, sl, K.magic);
    Q4Row q;
    q.dsc0 = c.dsc0;
    q.dsc1 = c.dsc1;
    q.e0 = c.e0;
    q.e1 = c.e1;
    q.c0 = -1024.0f - c.qb0;
    q.c1 = fmaf(c.qb1, -16.0f, -1024.0f);
    return q;
}

__device__ __forceinline__ uint32_t comp(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ float pair_sum(uint64_t a, uint64_t b) {
    return (lo_f(a) + hi_f(a)) + (lo_f(b) + hi_f(b));
}

// Q4_K: quant bytes 32g'..32g'+31 of the group's super-block hold columns
// l (low nibble) and 32 + l (high nibble, arrives as 16 q).
template <int B, int R>
__device__ __forceinline__ void q4k_item(const uint8_t* const (&rp)[R], int G, const float* xs,
                                         const float* sxs, int U, const Q4Sel& sl,
                                         const GroupConsts& K, float (&part)[R][B]) {
    const int boff = 144 * (G >> 2);
    const int qoff = boff + 16 + 32 * (G & 3);
    Q4Row rc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) rc[r] = q4k_row(*reinterpret_cast<const uint4*>(rp[r] + boff), sl, K);
    uint64_t a[R][B][4];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < B; ++b)
#pragma unroll
            for (int k = 0; k < 4; ++k) a[r][b][k] = 0;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        uint4 q[R];
#pragma unroll
        for (int r = 0; r < R; ++r) q[r] = *reinterpret_cast<const uint4*>(rp[r] + qoff + 16 * hf);
#pragma unroll
        for (int ww = 0; ww < 4; ++ww) {
            const int w = 4 * hf + ww;
            X2 xl[B], xh[B];
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const float* xg = xs + (b * U + G) * XS_STRIDE;
                xl[b] = lds_x2(xg + 4 * w);
                xh[b] = lds_x2(xg + 32 + 4 * w);
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t W = comp(q[r], ww), W8 = W >> 8;
                uint64_t v01, v23, u01, u23;      // u: high nibbles, 16 (q - qb) exactly
                h2f_pairs(lop_and_or(W, K.m4lo, K.magic), lop_and_or(W8, K.m4lo, K.magic), rc[r].c0, v01, v23);
                h2f_pairs(lop_and_or(W, K.m4hi, K.magic), lop_and_or(W8, K.m4hi, K.magic), rc[r].c1, u01, u23);
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    a[r][b][0] = ffma2(v01, xl[b].a, a[r][b][0]);
                    a[r][b][1] = ffma2(v23, xl[b].b, a[r][b][1]);
                    a[r][b][2] = ffma2(u01, xh[b].a, a[r][b][2]);
                    a[r][b][3] = ffma2(u23, xh[b].b, a[r][b][3]);
                }
            }
        }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
        const float sxl = sxs[(b * U + G) * 2], sxh = sxs[(b * U + G) * 2 + 1];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float A = pair_sum(a[r][b][0], a[r][b][1]);
            const float Bs = pair_sum(a[r][b][2], a[r][b][3]) * 0.0625f;   // exact
            part[r][b] = fmaf(rc[r].dsc0, A, fmaf(rc[r].e0, sxl, fmaf(rc[r].dsc1, Bs, rc[r].e1 * sxh)));
        }
    }
}

// Q6_K: group = half h (128 weights) x column run l0..l0+15 (l0 in {0, 16})
// of a super-block, over its four quarters q (column 128h + 32q + l).
// w = d * sc * (code - 32): exact, no cancellation, so the factored form
// sum_q d*sc_q * sum (code - 32) x is within a few gamma_n * sum |w x|.
template <int B, int R>
__device__ __forceinline__ void q6k_item(const uint8_t* const (&rp)[R], int G, const float* xs,
                                         int U, const GroupConsts& K, float (&part)[R][B]) {
    const int gm = G & 3, h = gm >> 1, l0 = 16 * (gm & 1);
    const int boff = 210 * (G >> 2);
    const uint32_t o = (uint32_t)(l0 >> 4);
    const uint32_t sel = 0x7050u | ((2u + o) << 8) | o;
    float ds[R][4];
    uint32_t A[R][4], Bw[R][4], H[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint8_t* bp = rp[r] + boff;
        lds_words_any2<4>(bp + 64 * h + l0, A[r]);
        lds_words_any2<4>(bp + 64 * h + 32 + l0, Bw[r]);
        lds_words_any2<4>(bp + 128 + 32 * h + l0, H[r]);
        uint32_t scw[2];
        lds_words_any2<2>(bp + 192 + 8 * h, scw);
        const uint32_t dw = lds_u32_any2(bp + 208);
        const uint32_t s01 = hsub2_u32(__byte_perm(scw[0], K.magic, sel) ^ 0x00800080u, 0x64806480u);
        const uint32_t s23 = hsub2_u32(__byte_perm(scw[1], K.magic, sel) ^ 0x00800080u, 0x64806480u);
        ds[r][0] = hmul_lo_lo(dw, s01, 0.0f);
        ds[r][1] = hmul_lo_hi(dw, s01, 0.0f);
        ds[r][2] = hmul_lo_lo(dw, s23, 0.0f);
        ds[r][3] = hmul_lo_hi(dw, s23, 0.0f);
    }
    uint64_t a[R][B][4];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < B; ++b)
#pragma unroll
            for (int q = 0; q < 4; ++q) a[r][b][q] = 0;
    const float cq = -1056.0f;                          // -(1024 + 32)
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        X2 xq[B][4];
#pragma unroll
        for (int b = 0; b < B; ++b)
#pragma unroll
            for (int q = 0; q < 4; ++q) xq[b][q] = lds_x2(xs + (b * U + G) * XS_STRIDE + 16 * q + 4 * w);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t c[4] = {(A[r][w] & 0x0F0F0F0Fu) | ((H[r][w] << 4) & 0x30303030u),
                                   (Bw[r][w] & 0x0F0F0F0Fu) | ((H[r][w] << 2) & 0x30303030u),
                                   ((A[r][w] >> 4) & 0x0F0F0F0Fu) | (H[r][w] & 0x30303030u),
                                   ((Bw[r][w] >> 4) & 0x0F0F0F0Fu) | ((H[r][w] >> 2) & 0x30303030u)};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint64_t v01, v23;
                h2f_pairs(lop_and_or(c[q], K.m6, K.magic), lop_and_or(c[q] >> 8, K.m6, K.magic), cq, v01, v23);
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    a[r][b][q] = ffma2(v01, xq[b][q].a, a[r][b][q]);
                    a[r][b][q] = ffma2(v23, xq[b][q].b, a[r][b][q]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < B; ++b) {
            float t[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) t[q] = lo_f(a[r][b][q]) + hi_f(a[r][b][q]);
            part[r][b] = fmaf(ds[r][0], t[0], fmaf(ds[r][1], t[1], fmaf(ds[r][2], t[2], ds[r][3] * t[3])));
        }
}

// Q8_0: group = two consecutive 34-byte blocks (68 bytes, 4-byte aligned in
// the stage).  w = d * q exact; factored per block.
template <int B, int R>
__device__ __forceinline__ void q80_item(const uint8_t* const (&rp)[R], int G, const float* xs,
                                         int U, const GroupConsts& K, float (&part)[R][B]) {
    const float cq = -1152.0f;                          // -(1024 + 128)
    uint64_t a[R][B][2];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < B; ++b) a[r][b][0] = a[r][b][1] = 0;
    float d[R][2];
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        uint32_t wv[R][9];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t* q = reinterpret_cast<const uint32_t*>(rp[r] + 68 * G) + 8 * blk;
#pragma unroll
            for (int i = 0; i < 9; ++i) wv[r][i] = q[i];
            d[r][blk] = blk == 0 ? h2f_lo(wv[r][0], 0.0f) : h2f_hi(wv[r][0], 0.0f);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            X2 xv[B];
#pragma unroll
            for (int b = 0; b < B; ++b) xv[b] = lds_x2(xs + (b * U + G) * XS_STRIDE + 32 * blk + 4 * i);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t Q = blk == 0 ? __funnelshift_r(wv[r][i], wv[r][i + 1], 16) : wv[r][i + 1];
                uint64_t v01, v23;
                h2f_pairs(lop_and_xor(Q, K.m8, K.x8), lop_and_xor(Q >> 8, K.m8, K.x8), cq, v01, v23);
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    a[r][b][blk] = ffma2(v01, xv[b].a, a[r][b][blk]);
                    a[r][b][blk] = ffma2(v23, xv[b].b, a[r][b][blk]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < B; ++b)
            part[r][b] = fmaf(d[r][0], lo_f(a[r][b][0]) + hi_f(a[r][b][0]),
                              d[r][1] * (lo_f(a[r][b][1]) + hi_f(a[r][b][1])));
}

template <int FMT, int B, int R>
__device__ __forceinline__ void run_item(const uint8_t* const (&rp)[R], int G, const float* xs,
                                         const float* sxs, int U, const Q4Sel& sl,
                                         const GroupConsts& K, float (&part)[R][B]) {
    if (FMT == FMT_Q4_K) q4k_item<B, R>(rp, G, xs, sxs, U, sl, K, part);
    else if (FMT == FMT_Q6_K) q6k_item<B, R>(rp, G, xs, U, K, part);
    else q80_item<B, R>(rp, G, xs, U, K, part);
}

// ---------------------------------------------------------------- reduction

// s1 = r[j] + r[j + 8] + r[j + 16] + ... (< U) in that order, and the same
// for r2 when `two`; the loads of a round of eight (both rows) are issued
// before any add, so their latencies overlap (absent terms add +0).
__device__ __forceinline__ void lane_sums(const float* r, const float* r2, bool two, int j, int U,
                                          float& s1, float& s2) {
    s1 = 0.f;
    s2 = 0.f;
    for (int G0 = j; G0 < U; G0 += 64) {
        float v[8], u[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const bool in = G0 + 8 * k < U;
            v[k] = in ? r[G0 + 8 * k] : 0.f;
            u[k] = (in && two) ? r2[G0 + 8 * k] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            s1 += v[k];
            s2 += u[k];
        }
    }
}

// Sum the per-group partials of tile t (segment S) into y, with the gated
// activation for row pairs: passes pass0, pass0 + pstep, ... of four
// outputs each, so the consumer warps share a tile.  8 lanes per output, lane j summing
// groups j, j + 8, ... in order, then a fixed butterfly: the order depends
// only on U, so results do not depend on B or the tile.  Four outputs per
// pass read rows UP floats apart (UP = 8 mod 32): no bank conflicts.
template <int B>
__device__ __forceinline__ void reduce_tile(const QGeo& Gm, const Seg& S, int t, const float* red,
                                            int lane, int pass0, int pstep) {
    const int U = Gm.U, UP = Gm.UP, mode = S.mode;
    const int half = Gm.RT / 2;
    const int lt = t - S.tile0;
    const int opt = mode == MODE_PLAIN ? Gm.RT : half;
    const int o0 = lt * opt;
    const int n_o = min(opt, S.nout - o0);
    const int nval = qseg_nval(S, B);
    const int boff = qseg_boff(S);
    float* y = S.y;
    const int64_t ldy = S.ld_y;
    const int j = lane & 7;
    const int n_out = n_o * B;
    const float* up_plane = red + (size_t)half * B * UP;
    for (int ob = 4 * pass0; ob < n_out; ob += 4 * pstep) {
        const int o = ob + (lane >> 3);
        const bool live = o < n_out;
        const int oo = live ? o : 0;
        const bool pair = mode != MODE_PLAIN;
        float vg, vu;
        lane_sums(red + (size_t)oo * UP, up_plane + (size_t)oo * UP, pair, j, U, vg, vu);
#pragma unroll
        for (int m = 1; m < 8; m <<= 1) {
            vg += __shfl_xor_sync(0xFFFFFFFFu, vg, m);
            vu += __shfl_xor_sync(0xFFFFFFFFu, vu, m);
        }
        const float v = pair ? act_eval(S.act, vg) * vu : seg_out(S.cap, vg);
        const int pi = oo / B, b = oo % B;
        if (live && j == 0 && b < nval) y[(int64_t)(boff + b) * ldy + o0 + pi] = v;
    }
}

// ---------------------------------------------------------------- the CTA

struct Smem {
    const Seg* segs;        // copy of the segment table (parameter reads with a
                            // dynamic index are slow; shared memory is not)
    uint8_t* stages;
    float* xs;
    float* sxs;
    float* red;
    uint64_t* full;
    uint64_t* empty;
    int* cnt;
    int* abort_flag;
};

template <int FMT, int B, int R>
__device__ void qmv_cta(const QmvParams& P, const GroupConsts& K, const Smem& sm, Walk walk0) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NC = (blockDim.x >> 5) - 1;          // consumer warps
    const int NCT = NC * 32;
    const int S_ = P.nstages;
    const QGeo& Gm = P.geo;
    const int U = Gm.U;
    const int red_tile = Gm.RT * B * Gm.UP;
    const int NRED = S_ + 1;             // partial slots

    if (warp == NC) {
        // ------------------------------------------------ producer warp
        // Streams tile n into stage n % S once the consumers released tile
        // n - S, then reduces tile n - S (its partials are complete when that
        // stage's empty barrier completes).  After the last issue it goes on
        // reducing all but the last two tiles, which the consumer warps share.
        const uint64_t policy = policy_evict_first();
        Walk w = walk0;
        // weights do not depend on the preceding kernel: unless the row
        // counts do, the first tiles go into their stages before waiting
        // for it (the CTA starts while that kernel finishes)
        const bool early = !P.dev_counts;
        if (!early) pdl_wait();
        walk_fix<B>(sm.segs, P.nseg, w);
        Walk wr = w;                      // reduction walk, S tiles behind
        uint32_t ephase = 0;
        int last_use[8];                  // last bulk-copied use of each stage (-1: none)
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) last_use[s2] = -1;
        bool ok = true;
        int nr = 0, ntiles = 0;           // tiles reduced / issued
        auto reduce_next = [&]() {
            __syncwarp();
            reduce_tile<B>(Gm, sm.segs[wr.hint], wr.t, sm.red + (size_t)(nr % NRED) * red_tile, lane, 0, 1);
            ++nr;
            wr.t += wr.step;
            walk_fix<B>(sm.segs, P.nseg, wr);
        };
        for (int n = 0, s = 0; w.t < w.end; ++n) {
            if (early && n == S_) pdl_wait();   // stages full: the rest waits
            if (warp_aborted(sm.abort_flag, lane)) break;
            if (n >= S_) {            // wait until the consumers released stage s
                if (lane == 0) ok = mbar_wait_bounded(&sm.empty[s], (ephase >> s) & 1u, P.timeout_ns);
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                ephase ^= 1u << s;
                if (!ok) break;
            }
            const Seg& S = sm.segs[w.hint];
            const QTile g = qtile(Gm, S, w.t);
            uint8_t* dst = sm.stages + (size_t)s * P.stage_bytes;
            if (g.tma) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sm.full[s], g.bytes1 + g.bytes2);
                    bulk_g2s_stream(dst, g.src1, g.bytes1, &sm.full[s], policy);
                    if (g.bytes2) bulk_g2s_stream(dst + g.dst2, g.src2, g.bytes2, &sm.full[s], policy);
                }
                last_use[s] = n / S_;
            } else {
                warp_copy(dst, g.src1, g.bytes1, lane);
                if (g.bytes2) warp_copy(dst + g.dst2, g.src2, g.bytes2, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.full[s]);
            }
            if (n >= S_) reduce_next();   // tile n - S
            w.t += w.step;
            walk_fix<B>(sm.segs, P.nseg, w);
            if (++s == S_) s = 0;
            ntiles = n + 1;
        }
        if (early && ntiles < S_) pdl_wait();
        // tiles before the last two are reduced here while the consumers
        // finish; the consumer warps share the last two
        while (ok && nr < ntiles - 2 && !warp_aborted(sm.abort_flag, lane)) {
            const int s2 = nr % S_;
            if (lane == 0) ok = mbar_wait_bounded(&sm.empty[s2], (ephase >> s2) & 1u, P.timeout_ns);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            ephase ^= 1u << s2;
            if (ok) reduce_next();
        }
        if (!ok && lane == 0) {
            record_status(P.status, STATUS_TIMEOUT);
            atomicExch(sm.abort_flag, 1);
        }
        // never leave a bulk copy in flight: wait (bounded) for the last
        // copy into each stage (already complete unless the CTA aborted)
        if (lane == 0) {
            for (int s2 = 0; s2 < S_; ++s2)
                if (last_use[s2] >= 0)
                    mbar_wait_bounded(&sm.full[s2], (uint32_t)last_use[s2] & 1u, drain_bound(P.timeout_ns));
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    // Per tile: wait for the stage, run the items, write the partials into
    // slot n % (S + 1), release the stage (the producer reduces the tile
    // later).  After the loop the consumer warps share the reduction of the
    // last two tiles.
    Walk w = walk0;
    int cur_seg = -1;
    uint32_t fphase = 0;
    bool aborted = false;
    const int UP = Gm.UP;
    const int half = Gm.RT / 2;
    const int rb = (int)qrow_bytes(FMT, Gm.cols);
    // Item it = tid + q*NCT of every tile covers group it % U of rows
    // (it / U)*R .. +R-1: the same for every tile, so it is stepped, not divided.
    const int G_first = tid % U, row_first = (tid / U) * R;
    const int dG = NCT % U, dRow = (NCT / U) * R;
    pdl_wait();                          // x and device row counts come from the preceding kernel
    walk_fix<B>(sm.segs, P.nseg, w);
    int slot_n = 0, ntl = 0, last_hint = 0, last_t = 0, prev_hint = 0, prev_t = 0;
    for (int n = 0, s = 0; w.t < w.end; ++n) {
        const Seg& S = sm.segs[w.hint];
        if (w.hint != cur_seg) {
            if (cur_seg >= 0 && same_xsrc(sm.segs[cur_seg], S)) {
                // the staged x serves this segment too
            } else if (NCT == U) {
                stage_x_own<FMT, B>(Gm, S, sm.xs, sm.sxs, G_first, S.xout && w.t == S.tile0);
            } else {
                consumer_sync(NCT);      // every consumer is done with the previous x
                stage_x<FMT, B>(Gm, S, sm.xs, sm.sxs, tid, NCT, S.xout && w.t == S.tile0);
            }
            cur_seg = w.hint;
        }
        if (!aborted) {
            bool ok = true;
            if (lane == 0) ok = mbar_wait_bounded(&sm.full[s], (fphase >> s) & 1u, P.timeout_ns);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok || warp_aborted(sm.abort_flag, lane)) {
                aborted = true;
                if (lane == 0 && !ok) {
                    record_status(P.status, STATUS_TIMEOUT);
                    atomicExch(sm.abort_flag, 1);
                }
            }
        }
        fphase ^= 1u << s;
        const int mode = S.mode;
        const uint8_t* st = sm.stages + (size_t)s * P.stage_bytes;
        float* red = sm.red + (size_t)slot_n * red_tile;
        if (!aborted) {
            int G = G_first, row0 = row_first;
            for (int q = 0; q < Gm.ipt; ++q) {
                const uint8_t* rp[R];
#pragma unroll
                for (int r = 0; r < R; ++r) rp[r] = st + (row0 + r) * rb;
                float part[R][B];
                const Q4Sel sel = q4_sel(G & 3);
                run_item<FMT, B, R>(rp, G, sm.xs, sm.sxs, U, sel, K, part);
                // partial row slot: gate rows of interleaved pairs first, then up rows
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int rho = row0 + r;
                    const int slot = mode == MODE_PAIR_INTERLEAVED ? (rho & 1) * half + (rho >> 1) : rho;
#pragma unroll
                    for (int b = 0; b < B; ++b) red[(slot * B + b) * UP + G] = part[r][b];
                }
                G += dG;
                row0 += dRow;
                if (G >= U) {
                    G -= U;
                    row0 += R;
                }
            }
        }
        // release the stage; the empty barrier (all consumer warps, release
        // order) also publishes the partials to whoever reduces the tile
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);
        prev_hint = last_hint;
        prev_t = last_t;
        last_hint = w.hint;
        last_t = w.t;
        w.t += w.step;
        walk_fix<B>(sm.segs, P.nseg, w);
        if (++s == S_) s = 0;
        if (++slot_n == NRED) slot_n = 0;
        ntl = n + 1;
    }
    // the last two tiles, shared by the consumer warps (passes of the second
    // assigned from the last warp down); tile m's partials are complete when
    // the empty barrier of stage m % S completes its use m / S
    for (int k = 0; k < 2 && !aborted; ++k) {
        const int m = ntl - 2 + k;
        if (m < 0) continue;
        bool ok = true;
        if (lane == 0) ok = mbar_wait_bounded(&sm.empty[m % S_], (uint32_t)(m / S_) & 1u, P.timeout_ns);
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) {
            aborted = true;
            if (lane == 0) {
                record_status(P.status, STATUS_TIMEOUT);
                atomicExch(sm.abort_flag, 1);
            }
            break;
        }
        reduce_tile<B>(Gm, sm.segs[k ? last_hint : prev_hint], k ? last_t : prev_t,
                       sm.red + (size_t)(m % NRED) * red_tile, lane, k ? NC - 1 - warp : warp, NC);
    }
}

}  // namespace

// Kernel: B x rows, R rows per work item, MASK = block formats compiled in
// (bit 0 Q4_K, bit 1 Q6_K, bit 2 Q8_0).
template <int B, int R, int MASK>
__global__ void __launch_bounds__(32 * (qmv_max_consumer_warps(R) + 1), B >= 8 ? 1 : 2)
    qmv_kernel(const __grid_constant__ QmvParams P, const GroupConsts K) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_launch_dependents();
    const int S_ = P.nstages;
    const int U = P.geo.U;
    Smem sm;
    size_t off = 0;
    sm.stages = smem;
    off += (size_t)S_ * P.stage_bytes;
    sm.xs = reinterpret_cast<float*>(smem + off);
    off += (size_t)B * U * XS_STRIDE * sizeof(float);
    sm.sxs = reinterpret_cast<float*>(smem + off);
    off += (size_t)B * U * 2 * sizeof(float);
    sm.red = reinterpret_cast<float*>(smem + off);
    off += (size_t)(S_ + 1) * P.geo.RT * B * P.geo.UP * sizeof(float);
    off = (off + 7) & ~size_t(7);
    sm.full = reinterpret_cast<uint64_t*>(smem + off);
    sm.empty = sm.full + S_;
    sm.cnt = reinterpret_cast<int*>(sm.empty + S_);
    sm.abort_flag = sm.cnt + (S_ + 1);
    size_t seg_off = off + (size_t)2 * S_ * sizeof(uint64_t) + (size_t)(S_ + 2) * sizeof(int);
    seg_off = (seg_off + 15) & ~size_t(15);                  // as in qmv_smem_bytes
    Seg* segs = reinterpret_cast<Seg*>(smem + seg_off);
    {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(&P.seg[0]);
        uint32_t* dst = reinterpret_cast<uint32_t*>(segs);
        const int nw = P.nseg * (int)(sizeof(Seg) / 4);
        for (int i = threadIdx.x; i < nw; i += blockDim.x) dst[i] = src[i];
    }
    sm.segs = segs;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S_; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], (blockDim.x >> 5) - 1);   // every consumer warp arrives
        }
        for (int s = 0; s <= S_; ++s) sm.cnt[s] = 0;
        *sm.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const bool g1 = (int)blockIdx.x >= P.cta_split;
    Walk w;
    w.hint = 0;
    if (!g1) {
        w.t = blockIdx.x;
        w.step = P.cta_split;
        w.end = P.tile_split;
    } else {
        w.t = P.tile_split + (blockIdx.x - P.cta_split);
        w.step = gridDim.x - P.cta_split;
        w.end = P.ntiles;
    }
    const int fmt = g1 ? P.fmt1 : P.fmt0;
    if ((MASK & 1) && fmt == FMT_Q4_K) qmv_cta<FMT_Q4_K, B, R>(P, K, sm, w);
    else if ((MASK & 2) && fmt == FMT_Q6_K) qmv_cta<FMT_Q6_K, B, R>(P, K, sm, w);
    else if ((MASK & 4) && fmt == FMT_Q8_0) qmv_cta<FMT_Q8_0, B, R>(P, K, sm, w);
}

inline GroupConsts group_consts() {
    GroupConsts K;
    K.magic = 0x64006400u;
    K.m4lo = 0x000F000Fu;
    K.m4hi = 0x00F000F0u;
    K.m8 = 0x00FF00FFu;
    K.x8 = 0x64806480u;
    K.m6 = 0x003F003Fu;
    return K;
}

// Host-side access to the instantiations of one batch width B.
template <int B>
struct QmvTable {
    template <int MASK>
    static void* fn() {
        return reinterpret_cast<void*>(qmv_kernel<B, qmv_rows_per_item(B, MASK), MASK>);
    }
    static void* get(int mask) {
        switch (mask) {
            case 1: return fn<1>();
            case 2: return fn<2>();
            case 4: return fn<4>();
            case 3: return fn<3>();
            default: return fn<7>();
        }
    }
    static cudaError_t set_smem(int bytes) {
        const int masks[5] = {1, 2, 4, 3, 7};
        for (int m : masks) {
            cudaError_t e = cudaFuncSetAttribute(get(m), cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    static cudaError_t occupancy(int mask, int nt, size_t smem, int* per_sm) {
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, get(mask), nt, smem);
    }
    // Launched with programmatic stream serialization: the kernel may start
    // while the preceding kernel of the stream finishes.  x and device row
    // counts are read only after griddepcontrol.wait; the producer copies its
    // first S weight tiles before that wait (weights do not depend on the
    // preceding kernel) unless the row counts come from the device.
    static cudaError_t launch(int mask, const QmvParams& P, int grid, int nt, size_t smem,
                              cudaStream_t st) {
        const GroupConsts K = group_consts();
        void* args[2] = {const_cast<QmvParams*>(&P), const_cast<GroupConsts*>(&K)};
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(nt);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelExC(&cfg, get(mask), args);
    }
};

}  // namespace lq
