// lq_gv.cu -- the batch-1 tensor-core matvec (one x row): y = W.x for Q4_K
// matrices and for launches that mix Q4_K and Q6_K matrices sharing x (the
// Q4_K Q/K + Q6_K V projection), plain matrices or interleaved gate/up pairs
// with the gated activation fused into the store (larql "Architecture ->
// Metal shader map", Gemma 3 table: q4k_matvec, q4k_q6k_qkv_proj,
// q4k_ffn_gate_up + geglu).  The work units and the operand encoding are in
// lq_gv.cuh.
//
// GB300 structure.
//  * One CTA of 16 warps per SM.  The row blocks (16 matrix rows, or 8
//    gate/up pairs) of all the launch's matrices are split into contiguous
//    ranges of nearly equal weight bytes, one per CTA; a tile is one row block
//    with all of its columns.
//  * A tile's 16 rows are consecutive, so one bulk copy brings it into a
//    shared-memory slot (4-byte cp.async copies when the weights are not
//    16-byte aligned), completion counted on the tile's own single-use
//    mbarrier.  Every tile that has a slot is requested at kernel entry,
//    before griddepcontrol.wait (weights never depend on the preceding
//    kernel); a slot is requested again once every unit of its tile is done.
//  * A tile's units (16 rows x 256 columns) go to the warps in pairs of
//    consecutive units, in order, so all warps work on each tile as it
//    lands: round robin when a CTA has a few pairs per warp, else from a
//    shared counter, so that a warp held up takes fewer pairs.
//  * x (the preceding kernel's output) is read once per CTA after
//    griddepcontrol.wait and turned into the MMA B images, optionally
//    RMS-normalised first (the input norm fused in front of QKV or gate+up)
//    or formed as act(g) * u from (g, u) pairs (the activation fused into
//    the down projection's x-load); CTA 0 stores the resulting row.
//  * Sums: a lane adds its rows' parts of a pair's units in order, the lane
//    quad adds in a fixed butterfly, and the warp that completes a tile adds
//    the tile's pair sums in column order and stores them: every order is
//    fixed by the shapes, so the result is deterministic and does not depend
//    on which warp computed what.
//  * Every mbarrier wait is bounded by %globaltimer; on expiry the warp
//    records STATUS_TIMEOUT and stops computing, and before exit the CTA waits
//    (bounded) for every copy it requested.
#include "lq_internal.h"
#include "lq_gv.cuh"

namespace lq {
namespace {

__device__ __forceinline__ void bulk_s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// The mbarrier also waits for this thread's earlier cp.async copies (the
// pending count is raised now and lowered when they complete).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.shared.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// acquire-release add on a shared counter: the partial sums a warp wrote
// before its add are visible to the warp that sees the completed count
__device__ __forceinline__ int atom_add_acqrel_cta(int* p, int v) {
    int old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_u32(p)), "r"(v) : "memory");
    return old;
}

// Device-scope wrap-around count (atom.inc: the value returned is the count
// before this arrival; reaching lim + 1 leaves 0), acquire-release.
__device__ __forceinline__ unsigned atom_inc_acqrel_gpu(unsigned* p, unsigned lim) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(lim) : "memory");
    return old;
}
__device__ __forceinline__ void st_relaxed_gpu(float* p, float v) {
    asm volatile("st.relaxed.gpu.global.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_relaxed_gpu(const float* p) {
    float v;
    asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t h2pack(__half lo, __half hi) {
    return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// the segment of row block rb (segs: the shared copy of the table)
__device__ __forceinline__ const GvSeg& gv_seg(const GvSeg* segs, int nseg, int rb) {
    int i = 0;
    while (i + 1 < nseg && rb >= segs[i + 1].rb0) ++i;
    return segs[i];
}

// Store the complete sums of row block rb of segment G, MMA rows r and r + 8
// (for gate/up pairs: gate and up of pair r).
__device__ __forceinline__ void gv_store(const GvSeg& G, int rb, int r, float v0, float v1) {
    const int lrb = rb - G.rb0;
    if (G.mode == MODE_PLAIN) {
        const int o = GV_ROWS * lrb + r;
        if (o < G.nout) G.y[o] = seg_out(G.cap, v0);
        if (o + 8 < G.nout) G.y[o + 8] = seg_out(G.cap, v1);
    } else {
        const int o = 8 * lrb + r;
        if (o < G.nout) G.y[o] = act_eval(G.act, v0) * v1;
    }
}

// x chunks per thread in the image build: 32-column blocks bi = 64 it +
// 4 warp + lane / 8 (it < GV_XIT), so rows of up to 24 super-blocks
constexpr int GV_XIT = 3;
static_assert(GV_XIT * GV_NW * 4 * 32 >= GV_MAX_NSB * 256, "image build covers the widest row");

// The raw loads behind four consecutive values of the launch's x row from
// column c: four floats, or with GV_X_ACT the four (g, u) pairs (a, b).
struct GvXRaw {
    float4 a, b;
};
template <class XP>
__device__ __forceinline__ GvXRaw gv_xload(const XP& P, int c) {
    GvXRaw r;
    if (P.xpre == GV_X_ACT) {
        const float* p = P.x + 2 * (int64_t)c;
        if (P.x16) {
            r.a = __ldcg(reinterpret_cast<const float4*>(p));
            r.b = __ldcg(reinterpret_cast<const float4*>(p) + 1);
        } else {
            r.a = make_float4(__ldcg(p), __ldcg(p + 1), __ldcg(p + 2), __ldcg(p + 3));
            r.b = make_float4(__ldcg(p + 4), __ldcg(p + 5), __ldcg(p + 6), __ldcg(p + 7));
        }
        return r;
    }
    const float* p = P.x + c;
    r.a = P.x16 ? __ldcg(reinterpret_cast<const float4*>(p)) : make_float4(__ldcg(p), __ldcg(p + 1), __ldcg(p + 2), __ldcg(p + 3));
    r.b = make_float4(0.f, 0.f, 0.f, 0.f);
    return r;
}

// The four values as the matvec sees them before any norm: the row itself,
// or act(g) * u of its (g, u) pairs (GV_X_ACT).
template <class XP>
__device__ __forceinline__ float4 gv_xval(const XP& P, const GvXRaw& r) {
    if (P.xpre == GV_X_ACT)
        return make_float4(act_eval(P.act, r.a.x) * r.a.y, act_eval(P.act, r.a.z) * r.a.w, act_eval(P.act, r.b.x) * r.b.y,
                           act_eval(P.act, r.b.z) * r.b.w);
    return r.a;
}

// The norm weights of this thread's x chunks (GV_X_NORM).  They never
// depend on the preceding kernel, so they are read before griddepcontrol.wait.
__device__ __forceinline__ void gv_load_nw(const GvParams& P, int nsb, int warp, int lane, float4 (&nwv)[GV_XIT]) {
#pragma unroll
    for (int it = 0; it < GV_XIT; ++it) {
        const int bi = 64 * it + 4 * warp + (lane >> 3);
        nwv[it] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (P.xpre == GV_X_NORM && bi < 8 * nsb) nwv[it] = __ldg(reinterpret_cast<const float4*>(P.nw + 32 * bi + 4 * (lane & 7)));
    }
}

constexpr uint32_t GV_RED_OFF = 384;      // in the parameter area: the warps' sums of squares
constexpr uint32_t GV_NEXT_OFF = GV_RED_OFF + 4 * GV_NW;   // the unit counter
// unit pairs of a CTA from which they are handed out by the counter (the
// layer's gate+up has 45 per CTA, QKV and O at most 15: 2 / 4 warps' worth
// gave gate+up 11.28 / 11.52 us, QKV and O unchanged)
constexpr int GV_DYN_PAIRS = 2 * GV_NW;
// tiles requested before griddepcontrol.wait (the others of the ring once x's
// loads are issued): 0 / 1 / 2 / 3 / 4 / 6 gave a Gemma-3-4B layer of
// 36.4 / 35.3 / 34.5 / 34.9 / 35.1 / 35.5 us
constexpr int GV_EARLY_TILES = 2;
// the column-chunked kernel: 2 / 3 / 4 / 6 gave 35.6 / 35.1 / 34.8 / 34.7 us
constexpr int GVW_EARLY_TILES = GV_MAX_INFLIGHT;
static_assert(GV_MAX_SEG * sizeof(GvSeg) + 8 <= GV_RED_OFF && GV_NEXT_OFF + 4 <= GV_PRM_BYTES,
              "parameter area layout");

// The MMA B images and x tables of the launch's x row (eight threads per
// 32-column block; every thread of the CTA takes part), after the optional
// RMS-norm or activation of x; CTA 0 stores the resulting row to P.xout.
// x is read once, all of a thread's chunks at the same time (one L2 round
// trip after griddepcontrol.wait); nwv holds the norm weights of the chunks.
//   The images cover the nsb super-blocks from super-block sbA of the row
// (the whole row, or the column window of a CTA's chunks); the super-blocks
// [st_lo, st_hi) of the window are also stored to P.xout.  The RMS-norm needs
// the whole row (sbA = 0, nsb = the row's super-blocks).
// `issued` runs once x's loads are issued, before their values are used.
template <int MASK, class XP, class F>
__device__ __forceinline__ void gv_images(const XP& P, const GvLayout& L, uint8_t* smem, int sbA, int nsb, int st_lo,
                                          int st_hi, int tid, int warp, int lane, const float4 (&nwv)[GV_XIT],
                                          F&& issued) {
    const int nblk = 8 * nsb;
    const int c0 = 256 * sbA;
    GvXRaw raw[GV_XIT];
#pragma unroll
    for (int it = 0; it < GV_XIT; ++it) {
        const int bi = 64 * it + 4 * warp + (lane >> 3);
        if (bi < nblk) raw[it] = gv_xload(P, c0 + 32 * bi + 4 * (lane & 7));
    }
    issued();
    float4 xv[GV_XIT];
#pragma unroll
    for (int it = 0; it < GV_XIT; ++it) {
        const int bi = 64 * it + 4 * warp + (lane >> 3);
        xv[it] = bi < nblk ? gv_xval(P, raw[it]) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // RMS-norm: every CTA sums the squares in the same fixed order (per
    // thread over its columns, a butterfly over the warp, then the warps
    // in order), so every CTA scales by the same r
    float rn = 1.0f;
    if (P.xpre == GV_X_NORM) {
        float ss = 0.f;
#pragma unroll
        for (int it = 0; it < GV_XIT; ++it) {
            const float4 v = xv[it];
            ss = fmaf(v.w, v.w, fmaf(v.z, v.z, fmaf(v.y, v.y, fmaf(v.x, v.x, ss))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
        float* red = reinterpret_cast<float*>(smem + L.prm + GV_RED_OFF);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float t = 0.f;
        for (int w = 0; w < GV_NW; ++w) t += red[w];
        rn = 1.0f / sqrtf(t / (float)(256 * nsb) + P.eps);
    }
#pragma unroll
    for (int it = 0; it < GV_XIT; ++it) {
        const int bi = 64 * it + 4 * warp + (lane >> 3), j = lane & 7;
        if (64 * it + 4 * warp >= nblk) break;          // warp-uniform: no block of this warp is left
        const bool valid = bi < nblk;
        const int sb = bi >> 3, blk = bi & 7;
        float4 v = xv[it];
        if (valid) {
            if (P.xpre == GV_X_NORM) {
                const float4 w = nwv[it];
                v = make_float4((v.x * rn) * w.x, (v.y * rn) * w.y, (v.z * rn) * w.z, (v.w * rn) * w.w);
            }
            if (P.xout && sb >= st_lo && sb < st_hi) *reinterpret_cast<float4*>(P.xout + c0 + 32 * bi + 4 * j) = v;
        }
        float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
        const int E = (int)((__float_as_uint(m) >> 23) & 0xFFu);
        const int es = max(1, E - 14);                                  // s = 2^(es - 127): |x / s| < 2^15
        const float inv = __uint_as_float((uint32_t)(254 - es) << 23);  // 1 / s, exact
        const float sc = __uint_as_float((uint32_t)es << 23);
        const float a[4] = {v.x * inv, v.y * inv, v.z * inv, v.w * inv};
        __half hi[4], lo[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            hi[c] = __float2half_rn(a[c]);
            lo[c] = __float2half_rn(a[c] - __half2float(hi[c]));
        }
        const uint2 ph = make_uint2(h2pack(hi[0], hi[2]), h2pack(hi[1], hi[3]));
        const uint2 pl = make_uint2(h2pack(lo[0], lo[2]), h2pack(lo[1], lo[3]));
        float sum = (v.x + v.y) + (v.z + v.w);
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 4);
        if (valid && (MASK & 1)) {
            const int tq = blk >> 1, hf = blk & 1, mm = 8 * hf + j;
            uint8_t* im = smem + L.img4 + sb * GV_BIMG + (2 * tq) * GV_BSLOT + mm * 8;
            *reinterpret_cast<uint2*>(im) = ph;
            *reinterpret_cast<uint2*>(im + GV_BSLOT) = pl;
            if (j == 0) {
                float* tb = reinterpret_cast<float*>(smem + L.tab4) + (sb * 4 + tq) * 4;
                tb[hf] = sum;
                tb[2 + hf] = sc;
            }
        }
        if (valid && (MASK & 2)) {
            const int h = blk >> 2, q = blk & 3, s6 = j >> 2, i = j & 3;
            const int tq = 2 * h + s6, mm = 4 * q + i;
            uint8_t* im = smem + L.img6 + sb * GV_BIMG + (2 * tq) * GV_BSLOT + mm * 8;
            *reinterpret_cast<uint2*>(im) = ph;
            *reinterpret_cast<uint2*>(im + GV_BSLOT) = pl;
            if (j == 0) {
                float* tb = reinterpret_cast<float*>(smem + L.tab6) + (sb * 4 + 2 * h) * 4;
                const float sq = q >= 2 ? sc * 0.0625f : sc;      // quarters 2, 3 arrive as 16 code
                tb[q] = sq;
                tb[4 + q] = sq;
            }
        }
    }
    if (tid < 32) reinterpret_cast<uint32_t*>(smem + L.zero)[tid] = 0u;
}

template <int MASK>
__global__ void __launch_bounds__(GV_NW * 32, 1) gv_kernel(const __grid_constant__ GvParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NS = P.nslots, nsb = P.nsb;
    const uint32_t SLOT = P.slot_bytes;
    const GvLayout L = gv_layout(MASK, NS, SLOT, P.maxtiles, nsb, NS);
    const uint32_t sbase = smem_u32(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);  // [tile] its copy has landed
    int* done = reinterpret_cast<int*>(smem + L.done);          // [tile] units done
    int* reqd = done + P.maxtiles;                               // [tile] requested
    // kernel parameters read with a dynamic index are slow (a chain of
    // constant-cache misses): the segment table and this CTA's row-block
    // range are copied to shared memory with one round of parallel loads
    GvSeg* segs = reinterpret_cast<GvSeg*>(smem + L.prm);
    int* crng = reinterpret_cast<int*>(smem + L.prm + GV_MAX_SEG * sizeof(GvSeg));
    int* nextv = reinterpret_cast<int*>(smem + L.prm + GV_NEXT_OFF);   // the next unit pair to hand out
    {
        const int nw = P.nseg * (int)(sizeof(GvSeg) / 4);
        if (tid < nw) reinterpret_cast<uint32_t*>(segs)[tid] = reinterpret_cast<const uint32_t*>(P.seg)[tid];
        if (tid >= 64 && tid < 66) crng[tid - 64] = P.cta_rb[blockIdx.x + tid - 64];
        if (tid == 96) *nextv = GV_NW;
        for (int i = tid; i < P.maxtiles; i += GV_NW * 32) {
            done[i] = 0;
            reqd[i] = 0;
            mbar_init(&full[i], 1);
        }
        fence_mbar_init();
    }
    const int nseg = P.nseg;
    __syncthreads();
    const int rbA = crng[0], ntile = crng[1] - crng[0];
    const uint64_t policy = policy_evict_first();

    // Request tile i (local row block) into slot i % NS.  Tile row r holds
    // matrix row 16 lrb + r (for gate/up pairs the packed rows: gate, up,
    // gate, ...).
    auto issue_tile = [&](int i) {
        const int rb = rbA + i;
        const GvSeg& G = gv_seg(segs, nseg, rb);
        const int row0 = GV_ROWS * (rb - G.rb0);
        const int nval = min(GV_ROWS, G.nrows - row0);
        const uint32_t dst = sbase + L.slots + (uint32_t)(i % NS) * SLOT;
        uint64_t* bar = &full[i];
        if (lane == 0) reqd[i] = 1;
        if (G.copy == GV_COPY_TILE) {
            // the rows are contiguous and the matrix ends on a 16-byte boundary
            if (lane == 0) {
                const uint32_t bytes = (uint32_t)((nval * G.rowbytes + 15) & ~int64_t(15));
                mbar_arrive_expect_tx(bar, bytes);
                bulk_s(dst, G.w + (int64_t)row0 * G.rowbytes, bytes, bar, policy);
            }
        } else {
            // each row (4-byte aligned, a multiple of 4 bytes) at a pitch of G.pitch
            const int nw = (int)(G.rowbytes >> 2);
            for (int r = 0; r < nval; ++r) {
                const uint8_t* p = G.w + (int64_t)(row0 + r) * G.rowbytes;
                for (int c = lane; c < nw; c += 32) cp_async4(dst + (uint32_t)(r * G.pitch + 4 * c), p + 4 * c);
            }
            cp_async_arrive(bar);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar);
        }
        __syncwarp();
    };

    // the first GV_EARLY_TILES tiles are requested at entry (warp w: tiles
    // w, w + GV_NW, ...), the other tiles that have a slot once the loads of
    // x are issued, so that x is not queued behind them
    const int early = min(ntile, min(NS, GV_EARLY_TILES));
    for (int i = warp; i < early; i += GV_NW) issue_tile(i);
    float4 nwv[GV_XIT];
    gv_load_nw(P, nsb, warp, lane, nwv);
    pdl_wait();

    gv_images<MASK>(P, L, smem, 0, nsb, 0, blockIdx.x == 0 ? nsb : 0, tid, warp, lane, nwv, [&] {
        for (int i = early + warp; i < min(ntile, NS); i += GV_NW) issue_tile(i);
    });
    __syncthreads();

    // ---- the units: unit pairs v = 0, 1, ... in order; pair v is units
    // 2 (v % hp) and 2 (v % hp) + 1 of tile v / hp (hp pairs per tile; the
    // last pair of a tile with an odd unit count has one unit).  Warp w starts
    // with pair w.  A CTA with many pairs hands out the next pair from a
    // shared counter, so a warp held up (waiting for a tile, completing one)
    // takes fewer; one with a few per warp deals them round robin (v + GV_NW),
    // which measured faster for the short launches.
    const GvK K = gv_consts();
    const int g = lane >> 2, t = lane & 3;
    const bool bact = (g >> 1) == t;                       // lanes holding B values
    const uint32_t bslot = (uint32_t)(2 * t + (g & 1)) * GV_BSLOT;
    const uint32_t b4 = bact ? sbase + L.img4 + bslot : sbase + L.zero;
    const uint32_t b6 = bact ? sbase + L.img6 + bslot : sbase + L.zero;
    const uint32_t bstr = bact ? GV_BIMG : 0u;
    const Q4Sel sel4 = q4_sel(t);
    float* part = reinterpret_cast<float*>(smem + L.part);   // [slot][pair][16]
    const int hp = (nsb + 1) / 2;
    int waited = -1;
    bool aborted = false;
    const bool dyn = ntile * hp >= GV_DYN_PAIRS;
    for (int v = warp; v < ntile * hp;) {
        const int i = v / hp, sb0 = 2 * (v % hp);
        const int nun = min(2, nsb - sb0);
        if (i != waited && !aborted) {
            bool ok = true;
            if (lane == 0) ok = mbar_wait_bounded(&full[i], 0u, P.timeout_ns);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
            if (!ok) {
                aborted = true;
                if (lane == 0) record_status(P.status, STATUS_TIMEOUT);
            }
            waited = i;
        }
        const int rb = rbA + i;
        const GvSeg& G = gv_seg(segs, nseg, rb);
        float y0 = 0.f, y1 = 0.f;
        if (!aborted) {
            const uint32_t tb = sbase + L.slots + (uint32_t)(i % NS) * SLOT;
            // tile rows of MMA rows g and g + 8 (pairs: gate row 2g, up row 2g + 1)
            const int ra = G.mode == MODE_PLAIN ? g : 2 * g, rr = G.mode == MODE_PLAIN ? g + 8 : 2 * g + 1;
            const int pitch = G.copy == GV_COPY_TILE ? (int)G.rowbytes : G.pitch;
            const uint32_t r0 = tb + (uint32_t)(ra * pitch), r1 = tb + (uint32_t)(rr * pitch);
            for (int jj = 0; jj < nun; ++jj) {
                const int sb = sb0 + jj;
                if ((MASK & 1) && G.fmt == FMT_Q4_K) {
                    const float4 xs = lds128f(sbase + L.tab4 + (uint32_t)(sb * 4 + t) * 16);
                    q4k_unit(r0 + 144 * sb, r1 + 144 * sb, t, sel4, b4 + sb * bstr, xs, K, y0, y1);
                } else if (MASK & 2) {
                    const float4 xs = lds128f(sbase + L.tab6 + (uint32_t)(sb * 4 + t) * 16);
                    const uint32_t bb = b6 + sb * bstr;
                    // rows start on 4-byte boundaries in shared memory, so
                    // super-block sb is half-word aligned exactly when
                    // 210 sb = 2 (mod 4)
                    if ((210 * sb) & 2) q6k_unit<true>(r0 + 210 * sb, r1 + 210 * sb, t, bb, xs, K, y0, y1);
                    else q6k_unit<false>(r0 + 210 * sb, r1 + 210 * sb, t, bb, xs, K, y0, y1);
                }
            }
        }
        // the pair's row sums (fixed butterfly over the lane quad)
        y0 += __shfl_xor_sync(0xFFFFFFFFu, y0, 1);
        y0 += __shfl_xor_sync(0xFFFFFFFFu, y0, 2);
        y1 += __shfl_xor_sync(0xFFFFFFFFu, y1, 1);
        y1 += __shfl_xor_sync(0xFFFFFFFFu, y1, 2);
        float* pu = part + ((i % NS) * hp + sb0 / 2) * 16;
        if (t == 0) {
            pu[g] = y0;
            pu[g + 8] = y1;
        }
        // the warp that completes the tile adds its pairs in column order,
        // stores, and requests tile i + NS into the slot
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atom_add_acqrel_cta(&done[i], nun) + nun == nsb;
        if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
            const float* pt = part + (i % NS) * hp * 16;
            if (lane < 8) {
                float v0 = 0.f, v1 = 0.f;
                for (int k = 0; k < hp; ++k) {
                    v0 += pt[k * 16 + lane];
                    v1 += pt[k * 16 + lane + 8];
                }
                gv_store(G, rb, lane, v0, v1);
            }
            if (i + NS < ntile && !aborted) {
                __syncwarp();
                if (lane == 0) fence_proxy_async_smem();   // every warp's reads of the slot come first
                __syncwarp();
                issue_tile(i + NS);
            }
        }
        if (dyn) {
            int vn = 0;
            if (lane == 0) vn = atomicAdd(nextv, 1);
            v = __shfl_sync(0xFFFFFFFFu, vn, 0);
        } else {
            v += GV_NW;
        }
    }
    __syncthreads();
    if (tid == 0) {
        // no copy may still be in flight when the CTA exits (every request was
        // waited for unless a warp gave up): wait, bounded, for each requested tile
        for (int i = 0; i < ntile; ++i)
            if (reqd[i]) mbar_wait_bounded(&full[i], 0u, drain_bound(P.timeout_ns));
    }
}

// ---------------------------------------------------------------- column chunks
// gvw_kernel: one plain matrix whose items are (column chunk, row block)
// pieces (the parameter struct describes the numbering), against one x row
// or (Q6_K) up to 8.  The structure is gv_kernel's with two changes: a tile
// is an item (16 rows of ch super-blocks, one bulk copy per row), and the CTA
// stages x only for the column window of its chunks.  Row sums of a row
// block are added across CTAs in chunk order through the scratch set.

// Shared memory of a gvw_kernel CTA: the tile slots, one mbarrier and two
// counters per tile, the parameter area (the RMS-norm's scratch in
// gv_images, unused here), for each of nm x rows the x image and table of
// the window's super-blocks (one format; row m at m * winsb super-blocks), a
// zero B slot, and per slot the 16 row sums of each of its unit pairs (at
// most ch) for each x row.
__host__ __device__ inline GvLayout gvw_layout(int nslots, uint32_t slot_bytes, int maxtiles, int winsb, int ch,
                                               int nm) {
    GvLayout L;
    uint32_t o = 0;
    L.slots = o;
    o += (uint32_t)nslots * slot_bytes;
    o = (o + 127u) & ~127u;
    L.bars = o;
    o += (uint32_t)maxtiles * 8u;
    L.done = o;
    o += (uint32_t)maxtiles * 8u;
    o = (o + 15u) & ~15u;
    L.prm = o;
    o += GV_PRM_BYTES;
    L.img4 = L.img6 = o;
    o += (uint32_t)(nm * winsb) * GV_BIMG;
    L.zero = o;
    o += 128u;
    L.tab4 = L.tab6 = o;
    o += (uint32_t)(nm * winsb) * 64u;
    L.part = o;
    o += (uint32_t)(nslots * ch * nm) * 64u;
    L.total = o;
    return L;
}

// The B images and x tables of M x rows (M > 1, x plain) over the column
// window of nsb super-blocks from sbA: gv_images' arithmetic, with the
// 32-column blocks of all rows numbered together (block vb: row vb / (8 nsb))
// and loaded three per thread at a time.
template <int MASK, class F>
__device__ __forceinline__ void gvw_images_m(const GvwParams& P, const GvLayout& L, uint8_t* smem, int sbA, int nsb,
                                             int M, int tid, int warp, int lane, F&& issued) {
    const int nblk = 8 * nsb, nvb = M * nblk;
    const uint32_t imgrow = (uint32_t)P.winsb * GV_BIMG, tabrow = (uint32_t)P.winsb * 64u;
    const int j = lane & 7;
    for (int base = 0; base < nvb; base += 64 * GV_XIT) {
        float4 xv[GV_XIT];
#pragma unroll
        for (int it = 0; it < GV_XIT; ++it) {
            const int vb = base + 64 * it + 4 * warp + (lane >> 3);
            xv[it] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (vb < nvb) {
                const int m = vb / nblk, bi = vb - m * nblk;
                const float* p = P.x + (int64_t)m * P.ld_x + 256 * sbA + 32 * bi + 4 * j;
                xv[it] = P.x16 ? __ldcg(reinterpret_cast<const float4*>(p))
                               : make_float4(__ldcg(p), __ldcg(p + 1), __ldcg(p + 2), __ldcg(p + 3));
            }
        }
        if (base == 0) issued();
#pragma unroll
        for (int it = 0; it < GV_XIT; ++it) {
            const int vb0 = base + 64 * it + 4 * warp;
            if (vb0 >= nvb) break;                         // warp-uniform: no block of this warp is left
            const int vb = vb0 + (lane >> 3);
            const bool valid = vb < nvb;
            const int m = valid ? vb / nblk : 0, bi = valid ? vb - m * nblk : 0;
            const int sb = bi >> 3, blk = bi & 7;
            const float4 v = xv[it];
            float mx = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
            const int E = (int)((__float_as_uint(mx) >> 23) & 0xFFu);
            const int es = max(1, E - 14);                                  // s = 2^(es - 127): |x / s| < 2^15
            const float inv = __uint_as_float((uint32_t)(254 - es) << 23);  // 1 / s, exact
            const float sc = __uint_as_float((uint32_t)es << 23);
            const float a[4] = {v.x * inv, v.y * inv, v.z * inv, v.w * inv};
            __half hi[4], lo[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                hi[c] = __float2half_rn(a[c]);
                lo[c] = __float2half_rn(a[c] - __half2float(hi[c]));
            }
            const uint2 ph = make_uint2(h2pack(hi[0], hi[2]), h2pack(hi[1], hi[3]));
            const uint2 pl = make_uint2(h2pack(lo[0], lo[2]), h2pack(lo[1], lo[3]));
            float sum = (v.x + v.y) + (v.z + v.w);
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
            sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 4);
            if (valid && (MASK & 1)) {
                const int tq = blk >> 1, hf = blk & 1, mm = 8 * hf + j;
                uint8_t* im = smem + L.img4 + m * imgrow + sb * GV_BIMG + (2 * tq) * GV_BSLOT + mm * 8;
                *reinterpret_cast<uint2*>(im) = ph;
                *reinterpret_cast<uint2*>(im + GV_BSLOT) = pl;
                if (j == 0) {
                    float* tb = reinterpret_cast<float*>(smem + L.tab4 + m * tabrow) + (sb * 4 + tq) * 4;
                    tb[hf] = sum;
                    tb[2 + hf] = sc;
                }
            }
            if (valid && (MASK & 2)) {
                const int h = blk >> 2, q = blk & 3, s6 = j >> 2, i = j & 3;
                const int tq = 2 * h + s6, mm = 4 * q + i;
                uint8_t* im = smem + L.img6 + m * imgrow + sb * GV_BIMG + (2 * tq) * GV_BSLOT + mm * 8;
                *reinterpret_cast<uint2*>(im) = ph;
                *reinterpret_cast<uint2*>(im + GV_BSLOT) = pl;
                if (j == 0) {
                    float* tb = reinterpret_cast<float*>(smem + L.tab6 + m * tabrow) + (sb * 4 + 2 * h) * 4;
                    const float sq = q >= 2 ? sc * 0.0625f : sc;      // quarters 2, 3 arrive as 16 code
                    tb[q] = sq;
                    tb[4 + q] = sq;
                }
            }
        }
    }
    if (tid < 32) reinterpret_cast<uint32_t*>(smem + L.zero)[tid] = 0u;
}

// MASK 1: Q4_K, 2: Q6_K; NM: x rows the kernel is built for (1, or 4 and
// 8 for Q6_K with P.nx <= NM rows; absent rows read the zero slot).
template <int MASK, int NM>
__global__ void __launch_bounds__(GV_NW * 32, 1) gvw_kernel(const __grid_constant__ GvwParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_launch_dependents();
    constexpr int SPAN = MASK == 1 ? 144 : 210;      // bytes of a super-block row
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NS = P.nslots, ch = P.ch, nrb = P.nrb, nsb = P.nsb;
    const uint32_t SLOT = P.slot_bytes;
    const GvLayout L = gvw_layout(NS, SLOT, P.maxtiles, P.winsb, ch, NM);
    const int M = NM == 1 ? 1 : P.nx;
    const uint32_t sbase = smem_u32(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);  // [tile] its copies have landed
    int* done = reinterpret_cast<int*>(smem + L.done);          // [tile] units done
    int* reqd = done + P.maxtiles;                               // [tile] requested
    int* nextu = reinterpret_cast<int*>(smem + L.prm);          // the next unit to hand out
    const int jA = P.cta_j[blockIdx.x], jB = P.cta_j[blockIdx.x + 1], ntile = jB - jA;
    for (int i = tid; i < P.maxtiles; i += GV_NW * 32) {
        done[i] = 0;
        reqd[i] = 0;
        mbar_init(&full[i], 1);
    }
    if (tid == 0) *nextu = GV_NW;
    fence_mbar_init();
    __syncthreads();
    const uint64_t policy = policy_evict_first();

    // Request tile i (item jA + i) into slot i % NS: row r of the item (16
    // row-block rows, fewer in a ragged last block) lands at r * pitch.
    auto issue_tile = [&](int i) {
        const int j = jA + i, c = j / nrb, rb = j - c * nrb;
        const int row0 = GV_ROWS * rb, nval = min(GV_ROWS, P.rows - row0);
        const uint32_t len = (uint32_t)(min(ch, nsb - c * ch) * SPAN);
        const uint32_t dst = sbase + L.slots + (uint32_t)(i % NS) * SLOT;
        uint64_t* bar = &full[i];
        if (lane == 0) {
            reqd[i] = 1;
            mbar_arrive_expect_tx(bar, len * (uint32_t)nval);
        }
        __syncwarp();
        if (lane < nval)
            bulk_s(dst + (uint32_t)(lane * P.pitch), P.w + (int64_t)(row0 + lane) * P.rowbytes + (int64_t)c * ch * SPAN,
                   len, bar, policy);
        __syncwarp();
    };

    const int early = min(ntile, min(NS, GVW_EARLY_TILES));
    for (int i = warp; i < early; i += GV_NW) issue_tile(i);
    float4 nwv[GV_XIT];
#pragma unroll
    for (int it = 0; it < GV_XIT; ++it) nwv[it] = make_float4(0.f, 0.f, 0.f, 0.f);
    pdl_wait();

    // the column window: chunks cA .. cB; x is stored for the chunks whose
    // first item (row block 0) is this CTA's
    const int cA = jA / nrb, cB = (jB - 1) / nrb, sbA = cA * ch;
    const int nsbw = min(nsb, (cB + 1) * ch) - sbA;
    const int cs0 = (jA + nrb - 1) / nrb, cs1 = (jB + nrb - 1) / nrb;
    auto issue_rest = [&] {
        for (int i = early + warp; i < min(ntile, NS); i += GV_NW) issue_tile(i);
    };
    if constexpr (NM == 1)
        gv_images<MASK>(P, L, smem, sbA, nsbw, cs0 * ch - sbA, min(nsb, cs1 * ch) - sbA, tid, warp, lane, nwv,
                        issue_rest);
    else
        gvw_images_m<MASK>(P, L, smem, sbA, nsbw, M, tid, warp, lane, issue_rest);
    __syncthreads();

    // ---- the takes v = 0, 1, ... of the CTA's tiles in order, UT units each
    // (pairs with one x row, single units with several; hpc takes per tile:
    // take v is units UT (v % hpc) .. + UT - 1 of tile v / hpc; the last take
    // of a chunk may be short, and takes past a ragged last chunk's end are
    // skipped).  Warp w starts with take w and then takes the next from a
    // shared counter, so a warp held up (by a tile's completion) takes fewer.
    const GvK K = gv_consts();
    const int g = lane >> 2, t = lane & 3;
    const bool bact = (g >> 1) == t;                       // lanes holding B values
    const uint32_t bslot = (uint32_t)(2 * t + (g & 1)) * GV_BSLOT;
    // x row m's images and tables are imgrow / tabrow bytes after row 0's
    const uint32_t imgrow = (uint32_t)P.winsb * GV_BIMG, tabrow = (uint32_t)P.winsb * 64u;
    const uint32_t bimg = bact ? sbase + L.img4 + bslot : sbase + L.zero;
    const uint32_t bstr = bact ? GV_BIMG : 0u;
    const Q4Sel sel4 = q4_sel(t);
    float* part = reinterpret_cast<float*>(smem + L.part);   // [slot][pair][x row][16]
    constexpr int UT = NM == 1 ? 2 : 1;                    // units per take: pairs, one with several x rows
    const int hpc = (ch + UT - 1) / UT;
    int i = warp / hpc, pr = warp - i * hpc;
    int ti = -1, c = 0, rb = 0, ncb = 0, waited = -1;
    bool aborted = false;
    while (i < ntile) {
        if (i != ti) {
            ti = i;
            const int j = jA + i;
            c = j / nrb;
            rb = j - c * nrb;
            ncb = min(ch, nsb - c * ch);
        }
        const int u0 = UT * pr, nun = min(UT, ncb - u0);
        if (nun > 0) {
            if (i != waited && !aborted) {
                bool ok = true;
                if (lane == 0) ok = mbar_wait_bounded(&full[i], 0u, P.timeout_ns);
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
                if (!ok) {
                    aborted = true;
                    if (lane == 0) record_status(P.status, STATUS_TIMEOUT);
                }
                waited = i;
            }
            float y0[NM], y1[NM];
#pragma unroll
            for (int m = 0; m < NM; ++m) y0[m] = y1[m] = 0.f;
            if (!aborted) {
                for (int uu = 0; uu < nun; ++uu) {
                    const int u = u0 + uu;
                    const uint32_t r0 = sbase + L.slots + (uint32_t)(i % NS) * SLOT + (uint32_t)(g * P.pitch + u * SPAN);
                    const uint32_t r1 = r0 + (uint32_t)(8 * P.pitch);
                    const int sbl = c * ch + u - sbA;             // the unit's super-block in the window
                    if constexpr (NM == 1) {
                        const float4 xs = lds128f(sbase + L.tab4 + (uint32_t)(sbl * 4 + t) * 16);
                        const uint32_t bb = bimg + (uint32_t)sbl * bstr;
                        if constexpr (MASK == 1) {
                            q4k_unit(r0, r1, t, sel4, bb, xs, K, y0[0], y1[0]);
                        } else {
                            // rows start on 4-byte boundaries (pitch 16 ch), so the
                            // unit is half-word aligned exactly when 210 u = 2 (mod 4)
                            if ((SPAN * u) & 2) q6k_unit<true>(r0, r1, t, bb, xs, K, y0[0], y1[0]);
                            else q6k_unit<false>(r0, r1, t, bb, xs, K, y0[0], y1[0]);
                        }
                    } else {
                        static_assert(MASK == 2, "several x rows: Q6_K only");
                        const uint32_t bb = bimg + (uint32_t)sbl * bstr, bs = bact ? imgrow : 0u;
                        const uint32_t tb = sbase + L.tab4 + (uint32_t)(sbl * 4 + t) * 16;
                        // one unit per take (U = 1): the unit's sums are the take's
                        if ((SPAN * u) & 2) q6k_unit_m<true, NM>(r0, r1, t, bb, bs, tb, tabrow, sbase + L.zero, M, K, y0, y1);
                        else q6k_unit_m<false, NM>(r0, r1, t, bb, bs, tb, tabrow, sbase + L.zero, M, K, y0, y1);
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < NM; ++m) {
                float a = y0[m], b = y1[m];
                a += __shfl_xor_sync(0xFFFFFFFFu, a, 1);
                a += __shfl_xor_sync(0xFFFFFFFFu, a, 2);
                b += __shfl_xor_sync(0xFFFFFFFFu, b, 1);
                b += __shfl_xor_sync(0xFFFFFFFFu, b, 2);
                float* pu = part + (((i % NS) * hpc + pr) * NM + m) * 16;
                if (t == 0) {
                    pu[g] = a;
                    pu[g + 8] = b;
                }
            }
            __syncwarp();
            int last = 0;
            if (lane == 0) last = atom_add_acqrel_cta(&done[i], nun) + nun == ncb;
            if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
                // the item's sums, its pairs in column order: value e of this
                // lane is (x row m, row r) = (idx / 16, idx % 16), idx = lane + 32 e
                constexpr int NV = (16 * NM + 31) / 32;
                const float* pt = part + (i % NS) * hpc * NM * 16;
                float v[NV];
#pragma unroll
                for (int e = 0; e < NV; ++e) {
                    const int idx = lane + 32 * e, m = idx >> 4, r = idx & 15;
                    v[e] = 0.f;
                    if (idx < 16 * M)
                        for (int k = 0; k < (ncb + UT - 1) / UT; ++k) v[e] += pt[(k * NM + m) * 16 + r];
                }
                // the slot's next tile first (its reads of the slot are done)
                if (i + NS < ntile && !aborted) {
                    __syncwarp();
                    if (lane == 0) fence_proxy_async_smem();   // every warp's reads of the slot come first
                    __syncwarp();
                    issue_tile(i + NS);
                }
                if (P.nch == 1) {
#pragma unroll
                    for (int e = 0; e < NV; ++e) {
                        const int idx = lane + 32 * e, m = idx >> 4, row = GV_ROWS * rb + (idx & 15);
                        if (idx < 16 * M && row < P.rows) P.y[(int64_t)m * P.ld_y + row] = seg_out(P.cap, v[e]);
                    }
                } else {
                    // publish the item's sums (the warp's stores, then one
                    // lane's acquire-release count: the release covers the
                    // stores the warp barrier ordered before it); the warp
                    // whose item completes the row block adds the chunks in
                    // order
#pragma unroll
                    for (int e = 0; e < NV; ++e) {
                        const int idx = lane + 32 * e, m = idx >> 4, r = idx & 15;
                        if (idx < 16 * M) st_relaxed_gpu(P.part + ((int64_t)(c * nrb + rb) * NM + m) * 16 + r, v[e]);
                    }
                    __syncwarp();
                    unsigned before = 0;
                    if (lane == 0) before = atom_inc_acqrel_gpu(P.cnt + rb, (unsigned)(P.nch - 1));
                    before = __shfl_sync(0xFFFFFFFFu, before, 0);
                    if (before == (unsigned)(P.nch - 1)) {
                        __syncwarp();                      // lane 0's acquire before every lane's loads
#pragma unroll
                        for (int e = 0; e < NV; ++e) {
                            const int idx = lane + 32 * e, m = idx >> 4, r = idx & 15, row = GV_ROWS * rb + r;
                            if (idx < 16 * M) {
                                float sum = 0.f;
                                for (int cc = 0; cc < P.nch; ++cc)
                                    sum += ld_relaxed_gpu(P.part + ((int64_t)(cc * nrb + rb) * NM + m) * 16 + r);
                                if (row < P.rows) P.y[(int64_t)m * P.ld_y + row] = seg_out(P.cap, sum);
                            }
                        }
                    }
                }
            }
        }
        int vn = 0;
        if (lane == 0) vn = atomicAdd(nextu, 1);
        vn = __shfl_sync(0xFFFFFFFFu, vn, 0);
        i = vn / hpc;
        pr = vn - i * hpc;
    }
    __syncthreads();
    if (tid == 0) {
        for (int k = 0; k < ntile; ++k)
            if (reqd[k]) mbar_wait_bounded(&full[k], 0u, drain_bound(P.timeout_ns));
    }
}

void* gv_get(int mask) {
    return mask == 1 ? reinterpret_cast<void*>(gv_kernel<1>) : reinterpret_cast<void*>(gv_kernel<3>);
}

}  // namespace

// the instance for the format and x rows: <1,1>, <2,1>, <2,4>, <2,8>
static void* gvw_get(int fmt, int nm) {
    if (fmt == FMT_Q4_K) return reinterpret_cast<void*>(gvw_kernel<1, 1>);
    return nm == 1 ? reinterpret_cast<void*>(gvw_kernel<2, 1>)
         : nm == 4 ? reinterpret_cast<void*>(gvw_kernel<2, 4>)
                   : reinterpret_cast<void*>(gvw_kernel<2, 8>);
}

cudaError_t gv_set_smem(int bytes) {
    for (int m : {1, 3}) {
        cudaError_t e = cudaFuncSetAttribute(gv_get(m), cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
    }
    for (void* f : {gvw_get(FMT_Q4_K, 1), gvw_get(FMT_Q6_K, 1), gvw_get(FMT_Q6_K, 4), gvw_get(FMT_Q6_K, 8)}) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

size_t gvw_smem_bytes(int nm, int nslots, uint32_t slot_bytes, int maxtiles, int winsb, int ch) {
    return gvw_layout(nslots, slot_bytes, maxtiles, winsb, ch, nm).total;
}


// The scratch sets of the column-chunked kernel: item sums and row-block
// counters.  Device globals start at zero and every launch leaves each
// counter at zero (a wrapping count), so no set needs clearing.
__device__ unsigned g_gvw_cnt[GVW_SLOTS][GVW_MAX_RB];
__device__ float g_gvw_part[GVW_SLOTS][GVW_MAX_PART];

cudaError_t gvw_scratch(unsigned** cnt, float** part) {
    void* a = nullptr;
    void* b = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&a, g_gvw_cnt);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&b, g_gvw_part);
    if (e != cudaSuccess) return e;
    *cnt = static_cast<unsigned*>(a);
    *part = static_cast<float*>(b);
    return cudaSuccess;
}

cudaError_t gvw_launch(int fmt, int nm, const GvwParams& P, int grid, size_t smem, cudaStream_t st) {
    void* args[1] = {const_cast<GvwParams*>(&P)};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(GV_NW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, gvw_get(fmt, nm), args);
}

cudaError_t gv_launch(int mask, const GvParams& P, int grid, size_t smem, cudaStream_t st) {
    void* args[1] = {const_cast<GvParams*>(&P)};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(GV_NW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, gv_get(mask), args);
}

}  // namespace lq
