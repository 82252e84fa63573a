// lq_group.cuh -- arithmetic primitives of the quantized matvec work items:
// exact code -> fp32 conversion, packed fp32 pairs, scale decoding.
//
// Instruction budget (GB300, measured): at HBM speed a Q4_K weight may cost
// about 3.4 issue slots.  Each weight is handled by
//   * one LOP3 per two weights: two 4/6/8-bit codes are OR-ed into the
//     mantissas of a half2 whose exponent makes each half equal 1024 + code
//     (exact);
//   * one mixed-precision add (add.rn.f32.f16): float(1024 + code) + c, with
//     c = -(1024 + centre), giving code - centre exactly in fp32;
//   * half of a packed FMA (fma.rn.f32x2) with the fp32 x values: the low
//     halves of the LOP3 results of bytes (0, 2) and (1, 3) of a code word
//     form the pair of columns (0, 1), the high halves (2, 3), matching the
//     two pairs of a 16-byte shared load of x in natural order.
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

// ---------------------------------------------------------------- fp32 pairs

// Two fp32 values in one 64-bit register (low word = first).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ float lo_f(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_f(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
// (a.lo * b.lo + c.lo, a.hi * b.hi + c.hi), each rounded once
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// four consecutive shared floats as two pairs
struct X2 {
    uint64_t a, b;
};
__device__ __forceinline__ X2 lds_x2(const float* p) {       // p 16-byte aligned
    const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(p);
    return X2{v.x, v.y};
}
// Codes of bytes 0..3 of a word, as (code - centre) pairs in column order:
// hA holds bytes 0 and 2 (low / high half), hB bytes 1 and 3, so the low
// halves give columns (0, 1) and the high halves columns (2, 3).
__device__ __forceinline__ void h2f_pairs(uint32_t hA, uint32_t hB, float c, uint64_t& c01,
                                          uint64_t& c23) {
    c01 = pk2(h2f_lo(hA, c), h2f_lo(hB, c));
    c23 = pk2(h2f_hi(hA, c), h2f_hi(hB, c));
}

// ---------------------------------------------------------------- Q4_K

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



// Scales and re-centring of the two sub-blocks (2g, 2g+1) of quant group g
// of a Q4_K super-block (hdr = its first 16 bytes: d, dmin, scales):
// dsc = d*sc and dm = dmin*m exactly in fp32, the centre
// qb = round(dm / dsc) clamped to [-16, 15], and e = dsc*qb - dm (one
// rounding).  magic = 0x64006400 (half2 1024, 1024).
struct Q4Cent {
    float dsc0, dsc1, qb0, qb1, e0, e1;
};

__device__ __forceinline__ Q4Cent q4k_centres(const uint4 hdr, const Q4Sel& sl, uint32_t magic) {
    const uint32_t s_sc = sl.hi ? hdr.w : hdr.y;
    const uint32_t s_m = sl.hi ? (hdr.w >> 4) : hdr.z;
    const uint32_t scw = ((s_sc >> sl.sh) & sl.mlo) | ((hdr.y >> (sl.sh + 2)) & sl.mhi);
    const uint32_t mw = ((s_m >> sl.sh) & sl.mlo) | ((hdr.z >> (sl.sh + 2)) & sl.mhi);
    const uint32_t sc_h = hsub2_u32(__byte_perm(scw, magic, 0x7150), magic);
    const uint32_t m_h = hsub2_u32(__byte_perm(mw, magic, 0x7150), magic);
    Q4Cent q;
    q.dsc0 = hmul_lo_lo(hdr.x, sc_h, 0.0f);
    q.dsc1 = hmul_lo_hi(hdr.x, sc_h, 0.0f);
    const float dm0 = hmul_hi_lo(hdr.x, m_h, 0.0f);
    const float dm1 = hmul_hi_hi(hdr.x, m_h, 0.0f);
    q.qb0 = rintf(fminf(fmaxf(dm0 * rcp_approx(q.dsc0), -16.0f), 15.0f));
    q.qb1 = rintf(fminf(fmaxf(dm1 * rcp_approx(q.dsc1), -16.0f), 15.0f));
    q.e0 = fmaf(q.dsc0, q.qb0, -dm0);
    q.e1 = fmaf(q.dsc1, q.qb1, -dm1);
    return q;
}

// 32-bit word at a 2-byte-aligned shared address
// (the aligned address is formed by pointer arithmetic, not an integer
// round trip, so the compiler keeps the shared address space: LDS, not LD)
__device__ __forceinline__ uint32_t lds_u32_any2(const uint8_t* p) {
    const uint32_t mis = (uint32_t)(reinterpret_cast<uintptr_t>(p) & 3u);
    const uint32_t* q = reinterpret_cast<const uint32_t*>(p - mis);
    return __funnelshift_r(q[0], q[1], mis * 8u);
}
// N consecutive words starting at a 2-byte-aligned shared address
template <int N>
__device__ __forceinline__ void lds_words_any2(const uint8_t* p, uint32_t* out) {
    const uint32_t mis = (uint32_t)(reinterpret_cast<uintptr_t>(p) & 3u);
    const uint32_t* q = reinterpret_cast<const uint32_t*>(p - mis);
    const uint32_t sh = mis * 8u;
    uint32_t w[N + 1];
#pragma unroll
    for (int i = 0; i <= N; ++i) w[i] = q[i];
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = __funnelshift_r(w[i], w[i + 1], sh);
}

}  // namespace lq
