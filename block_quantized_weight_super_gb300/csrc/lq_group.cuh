// lq_group.cuh -- batch-1 dot products of one row's 64-weight "group"
// against x values held in registers, for the three block formats.
//
// Instruction budget (GB300, measured): at HBM speed a Q4_K weight may cost
// about 3.4 issue slots and 1.7 half-rate ALU operations.  So each weight
// is handled by
//   * one LOP3 per two weights: two 4/6/8-bit codes are OR-ed into the
//     mantissas of a half2 whose exponent makes the half equal 1024 + code
//     (exact);
//   * one mixed-precision add (add.rn.f32.f16): float(1024 + code) + c, with
//     c = -(1024 + centre), giving code - centre exactly in fp32;
//   * one FFMA with the fp32 x value.
// Block scales are applied once per 16-32 weights (factored form).
//
// Q4_K: w_j = d*sc*q_j - dmin*m.  The factored sum d*sc*sum(q x) -
// dmin*m*sum(x) cancels when dmin*m ~ d*sc*q_j for all j.  It is re-centred
// on qb = round(dmin*m / (d*sc)) clamped to [-16, 15]:
//     sum_j w_j x_j = dsc * sum_j (q_j - qb) x_j + e * sum_j x_j,
//     e = dsc*qb - dmin*m (one fp32 rounding).
// With |e| <= dsc/2 (or the same sign as every w_j when qb is clamped),
// every term is bounded by a small multiple of |w_j x_j|, so the computed
// sum is within a few gamma_n * sum |w_j x_j| of the exact one for every
// input, like a dot product over the dequantized weights.
#pragma once
#include "lq_codec.cuh"

namespace lq {

// Constants kept in registers (passed as kernel arguments, so the compiler
// cannot turn them into immediates, which costs extra ALU operations).
struct GroupConsts {
    uint32_t magic;     // 0x64006400: half2 (1024, 1024)
    uint32_t m4lo;      // 0x000F000F
    uint32_t m4hi;      // 0x00F000F0
    uint32_t m8;        // 0x00FF00FF
    uint32_t x8;        // 0x64806480: magic with bit 7 of each byte flipped (int8 + 128)
    uint32_t m6;        // 0x003F003F
};

__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t m, uint32_t c) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(m), "r"(c));   // (a & m) | c
    return r;
}
__device__ __forceinline__ uint32_t lop_and_xor(uint32_t a, uint32_t m, uint32_t c) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(a), "r"(m), "r"(c));   // (a & m) ^ c
    return r;
}
// float(low / high half of h) + c, exact when the sum fits in fp32
__device__ __forceinline__ float h2f_lo(uint32_t h, float c) {
    float d;
    asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %1;\n\tadd.rn.f32.f16 %0, l, %2;\n\t}"
        : "=f"(d) : "r"(h), "f"(c));
    return d;
}
__device__ __forceinline__ float h2f_hi(uint32_t h, float c) {
    float d;
    asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %1;\n\tadd.rn.f32.f16 %0, u, %2;\n\t}"
        : "=f"(d) : "r"(h), "f"(c));
    return d;
}
// float(half a) * float(half b) + c in one rounding (products of halves are exact in fp32)
__device__ __forceinline__ float hmul_lo_lo(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{\n\t.reg .b16 al, au, bl, bu;\n\tmov.b32 {al, au}, %1;\n\tmov.b32 {bl, bu}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %3;\n\t}"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float hmul_lo_hi(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{\n\t.reg .b16 al, au, bl, bu;\n\tmov.b32 {al, au}, %1;\n\tmov.b32 {bl, bu}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bu, %3;\n\t}"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float hmul_hi_lo(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{\n\t.reg .b16 al, au, bl, bu;\n\tmov.b32 {al, au}, %1;\n\tmov.b32 {bl, bu}, %2;\n\t"
        "fma.rn.f32.f16 %0, au, bl, %3;\n\t}"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float hmul_hi_hi(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{\n\t.reg .b16 al, au, bl, bu;\n\tmov.b32 {al, au}, %1;\n\tmov.b32 {bl, bu}, %2;\n\t"
        "fma.rn.f32.f16 %0, au, bu, %3;\n\t}"
        : "=f"(d) : "r"(a), "r"(b), "f"(c));
    return d;
}
__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// ---------------------------------------------------------------- Q4_K
// x registers of group G (64 columns): xl[l] = x[64G + l], xh[l] =
// x[64G + 32 + l] / 16 (the high nibble arrives as 16*q).  sxl = sum xl
// over the 32 low columns, sxh = sum of x (unscaled) over the 32 high ones.

// Per-thread selectors of quant group g's scale/min fields in the 12-byte
// scale array: g < 2 reads 6-bit fields of bytes j, j+4; g >= 2 combines the
// low/high nibble of byte j+4 with the top two bits of bytes j-4 / j.
struct Q4Sel {
    uint32_t sh;        // 16 * (g & 1): which byte pair of the scale words
    uint32_t mlo;       // 0x3F3F (g < 2) or 0x0F0F
    uint32_t mhi;       // 0 (g < 2) or 0x3030
    bool hi;            // g >= 2
};

__device__ __forceinline__ Q4Sel q4_sel(int g) {
    Q4Sel s;
    s.sh = (uint32_t)(g & 1) * 16u;
    s.hi = g >= 2;
    s.mlo = s.hi ? 0x0F0Fu : 0x3F3Fu;
    s.mhi = s.hi ? 0x3030u : 0u;
    return s;
}

// Dot product of one Q4_K quant group with x: hdr = the super-block's first
// 16 bytes (d, dmin, scales), qa/qb = the group's 32 quant bytes.
__device__ __forceinline__ float q4k_group_dot(const uint4 hdr, const uint4 qa, const uint4 qb,
                                               const Q4Sel& sl, const float* xl, const float* xh,
                                               float sxl, float sxh, const GroupConsts& K) {
    // 6-bit scales and mins of sub-blocks 2g (byte 0) and 2g+1 (byte 1)
    const uint32_t s_sc = sl.hi ? hdr.w : hdr.y;
    const uint32_t s_m = sl.hi ? (hdr.w >> 4) : hdr.z;
    const uint32_t scw = ((s_sc >> sl.sh) & sl.mlo) | ((hdr.y >> (sl.sh + 2)) & sl.mhi);
    const uint32_t mw = ((s_m >> sl.sh) & sl.mlo) | ((hdr.z >> (sl.sh + 2)) & sl.mhi);
    // as halves (1024 + v) and then exact halves v
    const uint32_t sch = __byte_perm(scw, K.magic, 0x7150);    // (1024+sc0, 1024+sc1)
    const uint32_t mh = __byte_perm(mw, K.magic, 0x7150);
    // d*sc and dmin*m, exact: float(d) * (1024 + sc) - 1024 float(d) ...
    // written as (half d) x (half sc) with sc = (1024+sc) - 1024 in half arithmetic
    const uint32_t sc_h = hsub2_u32(sch, K.magic);
    const uint32_t m_h = hsub2_u32(mh, K.magic);
    const float dsc0 = hmul_lo_lo(hdr.x, sc_h, 0.0f);
    const float dsc1 = hmul_lo_hi(hdr.x, sc_h, 0.0f);
    const float dm0 = hmul_hi_lo(hdr.x, m_h, 0.0f);
    const float dm1 = hmul_hi_hi(hdr.x, m_h, 0.0f);
    // centres
    const float qb0 = rintf(fminf(fmaxf(dm0 * rcp_approx(dsc0), -16.0f), 15.0f));
    const float qb1 = rintf(fminf(fmaxf(dm1 * rcp_approx(dsc1), -16.0f), 15.0f));
    const float e0 = fmaf(dsc0, qb0, -dm0);
    const float e1 = fmaf(dsc1, qb1, -dm1);
    const float c0 = -1024.0f - qb0;                  // exact
    const float c1 = fmaf(qb1, -16.0f, -1024.0f);     // exact
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f, b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f;
    const uint32_t Wv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t W = Wv[w], W8 = W >> 8;
        const uint32_t h0 = lop_and_or(W, K.m4lo, K.magic);    // lo nibbles of bytes 0, 2
        const uint32_t h1 = lop_and_or(W, K.m4hi, K.magic);    // hi nibbles of bytes 0, 2 (x16)
        const uint32_t h2 = lop_and_or(W8, K.m4lo, K.magic);   // lo nibbles of bytes 1, 3
        const uint32_t h3 = lop_and_or(W8, K.m4hi, K.magic);   // hi nibbles of bytes 1, 3
        a0 = fmaf(h2f_lo(h0, c0), xl[4 * w + 0], a0);
        a1 = fmaf(h2f_hi(h0, c0), xl[4 * w + 2], a1);
        a2 = fmaf(h2f_lo(h2, c0), xl[4 * w + 1], a2);
        a3 = fmaf(h2f_hi(h2, c0), xl[4 * w + 3], a3);
        b0 = fmaf(h2f_lo(h1, c1), xh[4 * w + 0], b0);
        b1 = fmaf(h2f_hi(h1, c1), xh[4 * w + 2], b1);
        b2 = fmaf(h2f_lo(h3, c1), xh[4 * w + 1], b2);
        b3 = fmaf(h2f_hi(h3, c1), xh[4 * w + 3], b3);
    }
    const float A = (a0 + a1) + (a2 + a3);
    const float Bs = (b0 + b1) + (b2 + b3);
    return fmaf(dsc0, A, fmaf(e0, sxl, fmaf(dsc1, Bs, e1 * sxh)));
}

}  // namespace lq

namespace lq {

// 32-bit word at a 2-byte-aligned shared address
__device__ __forceinline__ uint32_t lds_u32_any2(const uint8_t* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* q = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    return __funnelshift_r(q[0], q[1], (uint32_t)(a & 3u) * 8u);
}
// N consecutive words starting at a 2-byte-aligned shared address
template <int N>
__device__ __forceinline__ void lds_words_any2(const uint8_t* p, uint32_t* out) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* q = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    const uint32_t sh = (uint32_t)(a & 3u) * 8u;
    uint32_t w[N + 1];
#pragma unroll
    for (int i = 0; i <= N; ++i) w[i] = q[i];
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = __funnelshift_r(w[i], w[i + 1], sh);
}

// ---------------------------------------------------------------- Q6_K
// Group = half h (128 weights) x column run l0..l0+15 (l0 in {0, 16}) of a
// super-block, over its four quarters q (column 128h + 32q + l).
// xr[16q + i] = x[col of quarter q, l = l0 + i].  w = d * sc[i/16] * (code - 32):
// exact, no cancellation, so the factored form sum_q d*sc_q * sum (code-32) x
// is within a few gamma_n * sum |w x|.
__device__ __forceinline__ float q6k_group_dot(const uint8_t* bp, int h, int l0, const float* xr,
                                               const GroupConsts& K) {
    uint32_t A[4], Bw[4], H[4], scw[2];
    lds_words_any2<4>(bp + 64 * h + l0, A);
    lds_words_any2<4>(bp + 64 * h + 32 + l0, Bw);
    lds_words_any2<4>(bp + 128 + 32 * h + l0, H);
    lds_words_any2<2>(bp + 192 + 8 * h, scw);          // scales 8h .. 8h+7
    const uint32_t dw = lds_u32_any2(bp + 208);        // d in the low half
    // quarter q uses scale byte 2q + o, o = l0/16: (q0,q1) from scw[0], (q2,q3) from scw[1]
    const uint32_t o = (uint32_t)(l0 >> 4);
    const uint32_t sel = 0x7050u | ((2u + o) << 8) | o;
    const uint32_t s01 = hsub2_u32(__byte_perm(scw[0], K.magic, sel) ^ 0x00800080u, 0x64806480u);
    const uint32_t s23 = hsub2_u32(__byte_perm(scw[1], K.magic, sel) ^ 0x00800080u, 0x64806480u);
    const float ds0 = hmul_lo_lo(dw, s01, 0.0f);
    const float ds1 = hmul_lo_hi(dw, s01, 0.0f);
    const float ds2 = hmul_lo_lo(dw, s23, 0.0f);
    const float ds3 = hmul_lo_hi(dw, s23, 0.0f);
    const float cq = -1056.0f;                          // -(1024 + 32)
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t c0 = (A[w] & 0x0F0F0F0Fu) | ((H[w] << 4) & 0x30303030u);
        const uint32_t c1 = (Bw[w] & 0x0F0F0F0Fu) | ((H[w] << 2) & 0x30303030u);
        const uint32_t c2 = ((A[w] >> 4) & 0x0F0F0F0Fu) | (H[w] & 0x30303030u);
        const uint32_t c3 = ((Bw[w] >> 4) & 0x0F0F0F0Fu) | ((H[w] >> 2) & 0x30303030u);
        const uint32_t c[4] = {c0, c1, c2, c3};
        float* acc[4] = {&a0, &a1, &a2, &a3};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t hA = lop_and_or(c[q], K.m6, K.magic);        // bytes 0, 2
            const uint32_t hB = lop_and_or(c[q] >> 8, K.m6, K.magic);   // bytes 1, 3
            float t = *acc[q];
            t = fmaf(h2f_lo(hA, cq), xr[16 * q + 4 * w + 0], t);
            t = fmaf(h2f_lo(hB, cq), xr[16 * q + 4 * w + 1], t);
            t = fmaf(h2f_hi(hA, cq), xr[16 * q + 4 * w + 2], t);
            t = fmaf(h2f_hi(hB, cq), xr[16 * q + 4 * w + 3], t);
            *acc[q] = t;
        }
    }
    return fmaf(ds0, a0, fmaf(ds1, a1, fmaf(ds2, a2, ds3 * a3)));
}

// ---------------------------------------------------------------- Q8_0
// Group = two consecutive 34-byte blocks (68 bytes, 4-byte aligned in the
// stage).  xr[i] = x[64G + i].  w = d*q exact; factored per block.
__device__ __forceinline__ float q80_group_dot(const uint8_t* bp, const float* xr,
                                               const GroupConsts& K) {
    const uint32_t* q = reinterpret_cast<const uint32_t*>(bp);
    uint32_t w[17];
#pragma unroll
    for (int i = 0; i < 17; ++i) w[i] = q[i];
    const float cq = -1152.0f;                          // -(1024 + 128)
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t Q = __funnelshift_r(w[i], w[i + 1], 16);     // block 0 quants 4i..4i+3
        const uint32_t hA = lop_and_xor(Q, K.m8, K.x8);
        const uint32_t hB = lop_and_xor(Q >> 8, K.m8, K.x8);
        a0 = fmaf(h2f_lo(hA, cq), xr[4 * i + 0], a0);
        a1 = fmaf(h2f_lo(hB, cq), xr[4 * i + 1], a1);
        a0 = fmaf(h2f_hi(hA, cq), xr[4 * i + 2], a0);
        a1 = fmaf(h2f_hi(hB, cq), xr[4 * i + 3], a1);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t Q = w[9 + i];                                 // block 1 quants 4i..4i+3
        const uint32_t hA = lop_and_xor(Q, K.m8, K.x8);
        const uint32_t hB = lop_and_xor(Q >> 8, K.m8, K.x8);
        b0 = fmaf(h2f_lo(hA, cq), xr[32 + 4 * i + 0], b0);
        b1 = fmaf(h2f_lo(hB, cq), xr[32 + 4 * i + 1], b1);
        b0 = fmaf(h2f_hi(hA, cq), xr[32 + 4 * i + 2], b0);
        b1 = fmaf(h2f_hi(hB, cq), xr[32 + 4 * i + 3], b1);
    }
    const float d0 = h2f_lo(w[0], 0.0f);
    const float d1 = h2f_hi(w[8], 0.0f);
    return fmaf(d0, a0 + a1, d1 * (b0 + b1));
}

}  // namespace lq
