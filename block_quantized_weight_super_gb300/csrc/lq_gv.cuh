// lq_gv.cuh -- work units of the batch-1 tensor-core matvec (lq_gv.cu).
//
// A unit is 16 weight rows x one 256-column super-block (Q4_K or Q6_K),
// held in shared memory, multiplied with one x row by warp-level MMAs
// (mma.sync m16n8k16, fp16 operands, fp32 accumulation).  What is computed
// is the matvec of larql "Architecture -> Metal shader map" (Gemma 3 table:
// q4k_matvec, q4k_q6k_qkv_proj, q4k_ffn_gate_up + geglu); only the
// multiply-adds move to the tensor cores.
//
// Operands.
//  * A (16 rows x 16 k per MMA) holds exact integer codes as fp16: a LOP3
//    ORs two 4-bit (or 6-bit) codes into the
//    mantissas of an fp16 pair equal to 1024 + code (or 1024 + 16 code for a
//    high nibble, which needs no shift), and one fp16x2 subtraction leaves
//    code - centre exactly.  Q4_K is re-centred per (row, sub-block) on
//    qb = round(dmin m / (d sc)) as in the CUDA-core kernel: every term of
//    sum_k (q_k - qb) x_k is then at most a small multiple of |w_k x_k|.
//    Q6_K codes are centred on 32 (w = d sc (code - 32), exact).
//  * B (16 k x 8 columns) holds x / s split into two fp16 pieces, hi =
//    fp16(x / s) and lo = fp16(x / s - hi), with s a power of two per
//    32-column block chosen so that |x / s| < 2^15: the pieces carry x to
//    2^-22 relative (plus an absolute floor ~2^-40 max|x| of the block).
//  * Column trick: lane quad t (lanes 4g + t) supplies the k slots 2t, 2t+1,
//    2t+8, 2t+9 of every MMA, and the code assignment gives each lane quad
//    one scale group per MMA.  B puts that group's x pieces in columns 2t
//    (hi) and 2t+1 (lo) and zeros elsewhere, so D[row][2t] + D[row][2t+1] is
//    exactly lane quad t's group sum, and it lands in lane (g, t) itself:
//    one MMA serves four scale groups, no lane holds another's sums, and the
//    per-group scaling needs no shuffles.
//
// Column permutation of a super-block (the same for A and B):
//   Q4_K: lane quad t owns columns 64t .. 64t+63; MMA m < 8 takes columns
//     64t + 4m + {0, 2} (k 2t, 2t+1) and {1, 3} (k 2t+8, 2t+9), MMA m >= 8
//     the same 32 columns higher: the low and high nibbles of bytes
//     4m..4m+3 of quant group t (sub-blocks 2t, 2t+1).
//   Q6_K: lane quad t = (h, s) = (t >> 1, t & 1) owns columns
//     128h + 32q + 16s + l (q = 0..3, l = 0..15), scale index 8h + 2q + s;
//     MMA m = 4q + i takes l = 4i + {0, 2} and {1, 3}.
#pragma once
#include "lq_group.cuh"

namespace lq {

// Constants kept in registers.
struct GvK {
    uint32_t magic;    // 0x64006400: fp16 pair (1024, 1024)
    uint32_t m4lo;     // 0x000F000F
    uint32_t m4hi;     // 0x00F000F0
    uint32_t m8;       // 0x00FF00FF
    uint32_t x8;       // 0x64806480: magic with bit 7 of each byte flipped (int8 + 128)
    uint32_t s8;       // 0x64806480 as the subtrahend of an int8 (Q6_K scales): (1152, 1152)
    uint32_t m6lo;     // 0x00300030: Q6_K high bits at mantissa bits 4-5
    uint32_t m6hi;     // 0x03000300: Q6_K high bits at mantissa bits 8-9
    uint32_t s6lo;     // 0x64206420: (1056, 1056) = 1024 + 32
    uint32_t s6hi;     // 0x66006600: (1536, 1536) = 1024 + 16 * 32
};

__host__ __device__ inline GvK gv_consts() {
    GvK k;
    k.magic = 0x64006400u;
    k.m4lo = 0x000F000Fu;
    k.m4hi = 0x00F000F0u;
    k.m8 = 0x00FF00FFu;
    k.x8 = 0x64806480u;
    k.s8 = 0x64806480u;
    k.m6lo = 0x00300030u;
    k.m6hi = 0x03000300u;
    k.s6lo = 0x64206420u;
    k.s6hi = 0x66006600u;
    return k;
}

// Rows of a unit and bytes of one unit's row (one 256-column unit).
constexpr int GV_ROWS = 16;
__host__ __device__ constexpr int gv_span(int fmt) { return fmt == 1 ? 144 : 210; }

// Shared-memory row pitch of a tile whose rows were copied with 4-byte
// cp.async copies: a row of n units rounded to an odd multiple of 16 bytes,
// so that the eight rows a quarter-warp reads sit in distinct banks.
__host__ __device__ inline int gv_row_pitch(int fmt, int n) {
    int p = ((gv_span(fmt) * n + 15) / 16) * 16;
    if (((p / 16) & 1) == 0) p += 16;
    return p;
}

// x image of one super-block for one layout: for each lane quad t and piece
// (hi, lo), the 16 MMAs' B registers (8 bytes each), slots padded to 144 bytes
// so that the eight lanes holding B read distinct banks.
constexpr int GV_BSLOT = 144;
constexpr int GV_BIMG = 8 * GV_BSLOT;     // bytes per super-block

constexpr int GV_NW = 16;                 // warps per CTA (one CTA per SM)
constexpr uint32_t GV_SMEM_MAX = 227u * 1024u;

// Shared memory of a CTA: the weight slots (whole tiles, or the warps'
// unit-pair stages), one mbarrier and two counters per tile (single use: a
// slot's next tile waits on a fresh barrier, so no phase can be mistaken for
// another), the shared copy of the parameters, the x images and per-block x
// tables (layout "4": Q4_K, layout "6": Q6_K) of the nsb super-blocks, a
// zero B slot, and for npart tiles the 16 row sums of each unit pair.
struct GvLayout {
    uint32_t slots, bars, done, prm, img4, img6, zero, tab4, tab6, part, total;
};
constexpr uint32_t GV_PRM_BYTES = 512;     // shared copy of the segment table and the CTA's row-block range
__host__ __device__ inline GvLayout gv_layout(int mask, int nslots, uint32_t slot_bytes, int maxtiles, int nsb,
                                              int npart) {
    GvLayout L;
    uint32_t o = 0;
    L.slots = o;
    o += (uint32_t)nslots * slot_bytes;
    o = (o + 127u) & ~127u;
    L.bars = o;
    o += (uint32_t)maxtiles * 8u;
    L.done = o;
    o += (uint32_t)maxtiles * 8u;          // per tile: units done, requested
    o = (o + 15u) & ~15u;
    L.prm = o;
    o += GV_PRM_BYTES;
    L.img4 = o;
    if (mask & 1) o += (uint32_t)nsb * GV_BIMG;
    L.img6 = o;
    if (mask & 2) o += (uint32_t)nsb * GV_BIMG;
    L.zero = o;
    o += 128u;
    L.tab4 = o;
    if (mask & 1) o += (uint32_t)nsb * 64u;
    L.tab6 = o;
    if (mask & 2) o += (uint32_t)nsb * 64u;
    L.part = o;
    o += (uint32_t)(npart * ((nsb + 1) / 2)) * 64u;
    L.total = o;
    return L;
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}

// D += A.B, m16n8k16, fp16 operands, fp32 accumulators
__device__ __forceinline__ void mma_h(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                      uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t gv_comp(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// fp16 pair (v, v) of a float (round to nearest; exact for the integers used)
__device__ __forceinline__ uint32_t h2dup(float v) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %1;" : "=r"(d) : "f"(v));
    return d;
}

// ---------------------------------------------------------------- Q4_K

// Row part of a Q4_K unit for lane quad t: the scales of sub-blocks 2t, 2t+1
// (exact d*sc, the centre, e = dsc*qb - dmin*m) and the fp16 subtrahends
// (1024 + qb, 1024 + 16 qb).
struct Q4U {
    float dlo, dhi, elo, ehi;
    uint32_t slo, shi;
};

__device__ __forceinline__ Q4U q4u_scales(const uint4 hdr, const Q4Sel& sl, uint32_t magic) {
    const Q4Cent c = q4k_centres(hdr, sl, magic);
    Q4U u;
    u.dlo = c.dsc0;
    u.dhi = c.dsc1;
    u.elo = c.e0;
    u.ehi = c.e1;
    u.slo = h2dup(1024.0f + c.qb0);
    u.shi = h2dup(fmaf(16.0f, c.qb1, 1024.0f));
    return u;
}

// One Q4_K unit: the super-blocks of rows g and g + 8 at shared addresses
// r0, r1 against x image `bimg` (this lane's B slot base for the
// super-block, or the zero slot) and the super-block's x sums / scales of
// lane quad t: xs = (sum x of sub-block 2t, of 2t+1, s of 2t, s of 2t+1).
// Adds the rows' partial dot products (over sub-blocks 2t, 2t+1) to y0, y1.
__device__ __forceinline__ void q4k_unit(uint32_t r0, uint32_t r1, int t, const Q4Sel& sl, uint32_t bimg, float4 xs,
                                         const GvK& K, float& y0, float& y1) {
    const uint4 h0 = lds128(r0), h1 = lds128(r1);
    const uint4 qa0 = lds128(r0 + 16 + 32 * t), qa1 = lds128(r0 + 32 + 32 * t);
    const uint4 qb0 = lds128(r1 + 16 + 32 * t), qb1 = lds128(r1 + 32 + 32 * t);
    const Q4U u0 = q4u_scales(h0, sl, K.magic), u1 = q4u_scales(h1, sl, K.magic);
    float dl[4] = {0.f, 0.f, 0.f, 0.f}, dh[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m2 = 0; m2 < 4; ++m2) {
        const uint4 bl = lds128(bimg + 16 * m2);          // B of lo MMAs 2m2, 2m2+1
        const uint4 bh = lds128(bimg + 64 + 16 * m2);     // B of hi MMAs 2m2, 2m2+1
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int m = 2 * m2 + k;
            const uint32_t wa = gv_comp(m < 4 ? qa0 : qa1, m & 3), wb = gv_comp(m < 4 ? qb0 : qb1, m & 3);
            const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
            mma_h(dl, hsub2_u32(lop_and_or(wa, K.m4lo, K.magic), u0.slo),
                  hsub2_u32(lop_and_or(wb, K.m4lo, K.magic), u1.slo),
                  hsub2_u32(lop_and_or(wa8, K.m4lo, K.magic), u0.slo),
                  hsub2_u32(lop_and_or(wb8, K.m4lo, K.magic), u1.slo), k ? bl.z : bl.x, k ? bl.w : bl.y);
            mma_h(dh, hsub2_u32(lop_and_or(wa, K.m4hi, K.magic), u0.shi),
                  hsub2_u32(lop_and_or(wb, K.m4hi, K.magic), u1.shi),
                  hsub2_u32(lop_and_or(wa8, K.m4hi, K.magic), u0.shi),
                  hsub2_u32(lop_and_or(wb8, K.m4hi, K.magic), u1.shi), k ? bh.z : bh.x, k ? bh.w : bh.y);
        }
    }
    const float sh = xs.w * 0.0625f;                     // high nibbles arrive as 16 q
    const float tl0 = (dl[0] + dl[1]) * xs.z, th0 = (dh[0] + dh[1]) * sh;
    const float tl1 = (dl[2] + dl[3]) * xs.z, th1 = (dh[2] + dh[3]) * sh;
    y0 += fmaf(u0.dlo, tl0, fmaf(u0.elo, xs.x, fmaf(u0.dhi, th0, u0.ehi * xs.y)));
    y1 += fmaf(u1.dlo, tl1, fmaf(u1.elo, xs.x, fmaf(u1.dhi, th1, u1.ehi * xs.y)));
}


// ---------------------------------------------------------------- misaligned shared loads

__device__ __forceinline__ uint32_t fsh16(uint32_t lo, uint32_t hi) { return __funnelshift_r(lo, hi, 16); }

// N words at shared address a, a = 2 (mod 4) when ODD, else a = 0 (mod 4).
template <bool ODD, int N>
__device__ __forceinline__ void ldw(uint32_t a, uint32_t (&out)[N]) {
    if constexpr (!ODD) {
#pragma unroll
        for (int i = 0; i < N; ++i) out[i] = lds32(a + 4 * i);
    } else {
        uint32_t w[N + 1];
#pragma unroll
        for (int i = 0; i <= N; ++i) w[i] = lds32(a - 2 + 4 * i);
#pragma unroll
        for (int i = 0; i < N; ++i) out[i] = fsh16(w[i], w[i + 1]);
    }
}

// ---------------------------------------------------------------- Q6_K

// One Q6_K unit: the super-blocks of rows g and g + 8 at shared addresses
// r0, r1 (both = 2 mod 4 when ODD, else = 0 mod 4).  Lane quad t = (h, s); per row it reads ql run 64h + 16s
// (quarters 0 and 2: low / high nibbles), ql run 64h + 32 + 16s (quarters 1,
// 3), qh run 32h + 16s (two bits per quarter) and the scales 8h + 2q + s.
// Codes of quarters 2 and 3 are built from the nibble in place (16 code),
// the high bits shifted two places further.  xs = (s of the x blocks of
// quarters 0..3 of half h; quarters 2, 3 divided by 16).
template <bool ODD>
__device__ __forceinline__ void q6k_unit(uint32_t r0, uint32_t r1, int t, uint32_t bimg, float4 xs, const GvK& K,
                                         float& y0, float& y1) {
    const int h = t >> 1, s = t & 1;
    uint32_t A0[4], B0[4], H0[4], A1[4], B1[4], H1[4];
    ldw<ODD>(r0 + 64 * h + 16 * s, A0);
    ldw<ODD>(r0 + 64 * h + 32 + 16 * s, B0);
    ldw<ODD>(r0 + 128 + 32 * h + 16 * s, H0);
    ldw<ODD>(r1 + 64 * h + 16 * s, A1);
    ldw<ODD>(r1 + 64 * h + 32 + 16 * s, B1);
    ldw<ODD>(r1 + 128 + 32 * h + 16 * s, H1);
    // scales sc[8h + 2q + s], q = 0..3, as fp16 pairs (q0, q2), (q1, q3); d
    const uint32_t sel = s ? 0x7531u : 0x6420u;
    float ds0[4], ds1[4];
    {
        uint32_t c0[2], c1[2];
        ldw<ODD>(r0 + 192 + 8 * h, c0);
        ldw<ODD>(r1 + 192 + 8 * h, c1);
        const uint32_t d0 = ODD ? lds32(r0 + 206) >> 16 : lds32(r0 + 208);
        const uint32_t d1 = ODD ? lds32(r1 + 206) >> 16 : lds32(r1 + 208);
        const uint32_t p0 = __byte_perm(c0[0], c0[1], sel), p1 = __byte_perm(c1[0], c1[1], sel);
        const uint32_t a02 = hsub2_u32(lop_and_xor(p0, K.m8, K.x8), K.s8), a13 = hsub2_u32(lop_and_xor(p0 >> 8, K.m8, K.x8), K.s8);
        const uint32_t b02 = hsub2_u32(lop_and_xor(p1, K.m8, K.x8), K.s8), b13 = hsub2_u32(lop_and_xor(p1 >> 8, K.m8, K.x8), K.s8);
        ds0[0] = hmul_lo_lo(d0, a02, 0.0f);
        ds0[2] = hmul_lo_hi(d0, a02, 0.0f);
        ds0[1] = hmul_lo_lo(d0, a13, 0.0f);
        ds0[3] = hmul_lo_hi(d0, a13, 0.0f);
        ds1[0] = hmul_lo_lo(d1, b02, 0.0f);
        ds1[2] = hmul_lo_hi(d1, b02, 0.0f);
        ds1[1] = hmul_lo_lo(d1, b13, 0.0f);
        ds1[3] = hmul_lo_hi(d1, b13, 0.0f);
    }
    float acc[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t wa0 = A0[i], wb0 = B0[i], hh0 = H0[i];
        const uint32_t wa1 = A1[i], wb1 = B1[i], hh1 = H1[i];
        const uint32_t wa0s = wa0 >> 8, wb0s = wb0 >> 8, wa1s = wa1 >> 8, wb1s = wb1 >> 8;
        const uint32_t h04 = hh0 << 4, h04r = hh0 >> 4, h02 = hh0 << 2, h06r = hh0 >> 6;
        const uint32_t h14 = hh1 << 4, h14r = hh1 >> 4, h12 = hh1 << 2, h16r = hh1 >> 6;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const bool hn = q >= 2;
            const uint32_t la0 = (q & 1) ? wb0 : wa0, lb0 = (q & 1) ? wb0s : wa0s;
            const uint32_t la1 = (q & 1) ? wb1 : wa1, lb1 = (q & 1) ? wb1s : wa1s;
            const uint32_t ha0 = (q & 1) ? h02 : h04, hb0 = (q & 1) ? h06r : h04r;
            const uint32_t ha1 = (q & 1) ? h12 : h14, hb1 = (q & 1) ? h16r : h14r;
            const uint32_t ml = hn ? K.m4hi : K.m4lo, mh = hn ? K.m6hi : K.m6lo, sb = hn ? K.s6hi : K.s6lo;
            const uint32_t a0 = hsub2_u32(lop_and_or(la0, ml, lop_and_or(ha0, mh, K.magic)), sb);
            const uint32_t a1 = hsub2_u32(lop_and_or(la1, ml, lop_and_or(ha1, mh, K.magic)), sb);
            const uint32_t a2 = hsub2_u32(lop_and_or(lb0, ml, lop_and_or(hb0, mh, K.magic)), sb);
            const uint32_t a3 = hsub2_u32(lop_and_or(lb1, ml, lop_and_or(hb1, mh, K.magic)), sb);
            const uint2 b = lds64(bimg + 32 * q + 8 * i);
            mma_h(acc[q], a0, a1, a2, a3, b.x, b.y);
        }
    }
    const float sx[4] = {xs.x, xs.y, xs.z, xs.w};
    float v0 = 0.f, v1 = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        v0 = fmaf(ds0[q], (acc[q][0] + acc[q][1]) * sx[q], v0);
        v1 = fmaf(ds1[q], (acc[q][2] + acc[q][3]) * sx[q], v1);
    }
    y0 += v0;
    y1 += v1;
}

// The same unit against NM x rows at once: x row m < M has its B slot at
// bimg0 + m bstep and its table entry of the super-block and lane quad (four
// floats: the scales of quarters 0..3, as xs of q6k_unit) at tab0 + m tstep;
// rows m >= M read the zero slot (bstep = 0 with bimg0 the zero slot for
// lanes holding no B values).  Each A fragment is built once and used by one MMA
// per x row; a quarter's code words are loaded when it is reached, to keep
// registers for the NM accumulators.  A row's arithmetic is q6k_unit's in
// the same order (each quarter's four MMAs accumulate i = 0..3, the
// quarters are added q = 0..3); v0[m], v1[m] are set to the row sums.
template <bool ODD, int NM>
__device__ __forceinline__ void q6k_unit_m(uint32_t r0, uint32_t r1, int t, uint32_t bimg0, uint32_t bstep,
                                           uint32_t tab0, uint32_t tstep, uint32_t zero, int M, const GvK& K,
                                           float (&v0)[NM], float (&v1)[NM]) {
    const int h = t >> 1, s = t & 1;
    const uint32_t sel = s ? 0x7531u : 0x6420u;
    float ds0[4], ds1[4];
    {
        uint32_t c0[2], c1[2];
        ldw<ODD>(r0 + 192 + 8 * h, c0);
        ldw<ODD>(r1 + 192 + 8 * h, c1);
        const uint32_t d0 = ODD ? lds32(r0 + 206) >> 16 : lds32(r0 + 208);
        const uint32_t d1 = ODD ? lds32(r1 + 206) >> 16 : lds32(r1 + 208);
        const uint32_t p0 = __byte_perm(c0[0], c0[1], sel), p1 = __byte_perm(c1[0], c1[1], sel);
        const uint32_t a02 = hsub2_u32(lop_and_xor(p0, K.m8, K.x8), K.s8), a13 = hsub2_u32(lop_and_xor(p0 >> 8, K.m8, K.x8), K.s8);
        const uint32_t b02 = hsub2_u32(lop_and_xor(p1, K.m8, K.x8), K.s8), b13 = hsub2_u32(lop_and_xor(p1 >> 8, K.m8, K.x8), K.s8);
        ds0[0] = hmul_lo_lo(d0, a02, 0.0f);
        ds0[2] = hmul_lo_hi(d0, a02, 0.0f);
        ds0[1] = hmul_lo_lo(d0, a13, 0.0f);
        ds0[3] = hmul_lo_hi(d0, a13, 0.0f);
        ds1[0] = hmul_lo_lo(d1, b02, 0.0f);
        ds1[2] = hmul_lo_hi(d1, b02, 0.0f);
        ds1[1] = hmul_lo_lo(d1, b13, 0.0f);
        ds1[3] = hmul_lo_hi(d1, b13, 0.0f);
    }
#pragma unroll
    for (int m = 0; m < NM; ++m) v0[m] = v1[m] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        // quarter q: low codes from ql run 64h + 16s (q even) or 64h + 32 + 16s
        // (q odd), high bits from qh run 32h + 16s
        uint32_t L0[4], L1[4], H0[4], H1[4];
        ldw<ODD>(r0 + 64 * h + 32 * (q & 1) + 16 * s, L0);
        ldw<ODD>(r1 + 64 * h + 32 * (q & 1) + 16 * s, L1);
        ldw<ODD>(r0 + 128 + 32 * h + 16 * s, H0);
        ldw<ODD>(r1 + 128 + 32 * h + 16 * s, H1);
        const bool hn = q >= 2;
        const uint32_t ml = hn ? K.m4hi : K.m4lo, mh = hn ? K.m6hi : K.m6lo, sb = hn ? K.s6hi : K.s6lo;
        float acc[NM][4];
#pragma unroll
        for (int m = 0; m < NM; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t la0 = L0[i], la1 = L1[i];
            const uint32_t lb0 = la0 >> 8, lb1 = la1 >> 8;
            const uint32_t ha0 = (q & 1) ? H0[i] << 2 : H0[i] << 4, hb0 = (q & 1) ? H0[i] >> 6 : H0[i] >> 4;
            const uint32_t ha1 = (q & 1) ? H1[i] << 2 : H1[i] << 4, hb1 = (q & 1) ? H1[i] >> 6 : H1[i] >> 4;
            const uint32_t a0 = hsub2_u32(lop_and_or(la0, ml, lop_and_or(ha0, mh, K.magic)), sb);
            const uint32_t a1 = hsub2_u32(lop_and_or(la1, ml, lop_and_or(ha1, mh, K.magic)), sb);
            const uint32_t a2 = hsub2_u32(lop_and_or(lb0, ml, lop_and_or(hb0, mh, K.magic)), sb);
            const uint32_t a3 = hsub2_u32(lop_and_or(lb1, ml, lop_and_or(hb1, mh, K.magic)), sb);
#pragma unroll
            for (int m = 0; m < NM; ++m) {
                const uint32_t ba = m < M ? bimg0 + m * bstep : zero;
                const uint2 b = lds64(ba + 32 * q + 8 * i);
                mma_h(acc[m], a0, a1, a2, a3, b.x, b.y);
            }
        }
#pragma unroll
        for (int m = 0; m < NM; ++m) {
            const float sx = __uint_as_float(lds32((m < M ? tab0 + m * tstep : zero) + 4 * q));
            v0[m] = fmaf(ds0[q], (acc[m][0] + acc[m][1]) * sx, v0[m]);
            v1[m] = fmaf(ds1[q], (acc[m][2] + acc[m][3]) * sx, v1[m]);
        }
    }
}

}  // namespace lq
