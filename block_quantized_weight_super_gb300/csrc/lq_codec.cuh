// lq_codec.cuh -- in-register unpacking of the three block formats and the
// 16-weight "leaf" dot products the matvec kernels are built from.
//
// Formats (GGUF convention; block sizes from larql "Architecture -> Metal
// shader map", dispatch-predicate table (Q4_K: 144-byte blocks) and dotLLM
// PR #320, Q8_0 GEMV row-stride fix (Q8_0: 34 bytes per 32 weights)):
//   Q4_K 144 B / 256: fp16 d, fp16 dmin, 12 B 6-bit scales/mins, 128 B nibbles
//   Q6_K 210 B / 256: 128 B low nibbles, 64 B high 2-bit, 16 int8 scales, fp16 d
//   Q8_0  34 B /  32: fp16 d, 32 int8
//
// Dequantized weights are exact fp32 values: w = d*sc*q - dmin*m (Q4_K, one
// rounding, both products exact), w = d*sc*q (Q6_K, exact), w = d*q (Q8_0,
// exact).  4- and 6-bit codes become floats without a conversion
// instruction: OR-ing a code into the mantissa of a power of two M gives the
// float M + code, and M is then subtracted exactly.
//
// A "group" is 64 consecutive weights of a row's weight index space grouped
// so one thread can own them: Q4_K group = one 32-byte quant group of a
// super-block (its two 32-weight sub-blocks), Q6_K group = one 16-wide column
// run of one half of a super-block over its four quarters, Q8_0 group = two
// blocks.  A group is four 16-weight leaves.  Every leaf's partial dot product
// is computed by the same code whatever the batch, and partials are combined
// in a fixed tree, so results do not depend on the batch size.
#pragma once
#include "lq_device.cuh"

namespace lq {

enum { FMT_Q4_K = 1, FMT_Q6_K = 2, FMT_Q8_0 = 3 };

__host__ __device__ constexpr int block_bytes_of(int fmt) {
    return fmt == FMT_Q4_K ? 144 : fmt == FMT_Q6_K ? 210 : fmt == FMT_Q8_0 ? 34 : 0;
}
__host__ __device__ constexpr int block_elems_of(int fmt) {
    return fmt == FMT_Q4_K ? 256 : fmt == FMT_Q6_K ? 256 : fmt == FMT_Q8_0 ? 32 : 0;
}

__device__ __forceinline__ float as_f(uint32_t u) { return __uint_as_float(u); }

// float with exponent chosen so that a 4-bit field at bit p of its mantissa
// counts as 1 per unit: value = 2^(23-p) + q.
#define LQ_MG(p) ((uint32_t)(150 - (p)) << 23)

// ---------------------------------------------------------------- Q4_K

// Scale pair of quant group g (sub-blocks 2g, 2g+1) from the three scale
// words s0 = bytes 0..3, s1 = 4..7, s2 = 8..11 of the 12-byte field.
//   j < 4 : sc_j = s[j] & 63,  m_j = s[j+4] & 63
//   j >= 4: sc_j = (s[j+4] & 15) | (s[j-4] >> 6) << 4,
//           m_j  = (s[j+4] >> 4) | (s[j] >> 6) << 4
// Returns (d*sc_2g, d*sc_2g+1) and (dmin*m_2g, dmin*m_2g+1); exact products.
__device__ __forceinline__ void q4k_group_scales(uint32_t dword, uint32_t s0, uint32_t s1,
                                                 uint32_t s2, int g, float2& dsc, float2& dm) {
    const uint32_t sh = (g & 1) * 16;
    const uint32_t a = s0 >> sh, b = s1 >> sh, c = s2 >> sh;
    uint32_t scw, mw;
    if (g < 2) {
        scw = a & 0x3F3Fu;
        mw = b & 0x3F3Fu;
    } else {
        scw = (c & 0x0F0Fu) | ((a >> 2) & 0x3030u);
        mw = ((c >> 4) & 0x0F0Fu) | ((b >> 2) & 0x3030u);
    }
    const float2 sc = __fadd2_rn(make_float2(as_f(prmt(scw, 0x4B000000u, 0x7440u)),
                                             as_f(prmt(scw, 0x4B000000u, 0x7441u))),
                                 make_float2(-8388608.0f, -8388608.0f));
    const float2 m = __fadd2_rn(make_float2(as_f(prmt(mw, 0x4B000000u, 0x7440u)),
                                            as_f(prmt(mw, 0x4B000000u, 0x7441u))),
                                make_float2(-8388608.0f, -8388608.0f));
    const float d = half_bits_to_float(dword);
    const float dmin = half_bits_to_float(dword >> 16);
    dsc = __fmul2_rn(sc, make_float2(d, d));
    dm = __fmul2_rn(m, make_float2(dmin, dmin));
}

// The eight 4-bit quants of one 32-bit word of qs as exact floats, in pairs:
//   lo01 = (lo nibble of byte 0, of byte 1), lo23 = bytes 2, 3; hi01, hi23 the
//   high nibbles.  Low nibbles belong to sub-block 2g, high to 2g+1.
struct Q4Pairs {
    float2 lo01, lo23, hi01, hi23;
};

__device__ __forceinline__ Q4Pairs q4k_word(uint32_t W) {
    const uint32_t Ws = W >> 12;
    Q4Pairs r;
    r.lo01 = __fadd2_rn(make_float2(as_f((W & 0xFu) | LQ_MG(0)), as_f((W & 0xF00u) | LQ_MG(8))),
                        make_float2(-8388608.0f, -32768.0f));
    r.lo23 = __fadd2_rn(
        make_float2(as_f((W & 0xF0000u) | LQ_MG(16)), as_f((Ws & 0xF000u) | LQ_MG(12))),
        make_float2(-128.0f, -2048.0f));
    r.hi01 = __fadd2_rn(make_float2(as_f((W & 0xF0u) | LQ_MG(4)), as_f((W & 0xF000u) | LQ_MG(12))),
                        make_float2(-524288.0f, -2048.0f));
    r.hi23 = __fadd2_rn(
        make_float2(as_f((Ws & 0xF00u) | LQ_MG(8)), as_f((Ws & 0xF0000u) | LQ_MG(16))),
        make_float2(-32768.0f, -128.0f));
    return r;
}

// Leaf = 2 qs words = 8 weights of sub-block 2g (cols c0+0..7) and 8 of
// sub-block 2g+1 (cols c0+32..39).  xr[b][l][0..3] hold the low-nibble columns in
// pairs, xr[b][l][4..7] the high-nibble columns.  Per batch row b, returns the
// leaf's partial dot product.
template <int B, int NL>
__device__ __forceinline__ void q4k_leaf(uint32_t W0, uint32_t W1, float2 dsc, float2 dm,
                                         const float2 (&xr)[B][NL][8], int l, float* out) {
    const float2 slo = make_float2(dsc.x, dsc.x), shi = make_float2(dsc.y, dsc.y);
    const float2 mlo = make_float2(-dm.x, -dm.x), mhi = make_float2(-dm.y, -dm.y);
    float2 alo[B], ahi[B];
#pragma unroll
    for (int b = 0; b < B; ++b) alo[b] = ahi[b] = make_float2(0.f, 0.f);
#pragma unroll
    for (int wi = 0; wi < 2; ++wi) {
        const Q4Pairs q = q4k_word(wi ? W1 : W0);
        const float2 w0 = __ffma2_rn(q.lo01, slo, mlo);
        const float2 w1 = __ffma2_rn(q.lo23, slo, mlo);
        const float2 w2 = __ffma2_rn(q.hi01, shi, mhi);
        const float2 w3 = __ffma2_rn(q.hi23, shi, mhi);
#pragma unroll
        for (int b = 0; b < B; ++b) {
            alo[b] = __ffma2_rn(w0, xr[b][l][2 * wi + 0], alo[b]);
            alo[b] = __ffma2_rn(w1, xr[b][l][2 * wi + 1], alo[b]);
            ahi[b] = __ffma2_rn(w2, xr[b][l][4 + 2 * wi + 0], ahi[b]);
            ahi[b] = __ffma2_rn(w3, xr[b][l][4 + 2 * wi + 1], ahi[b]);
        }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
        const float2 t = __fadd2_rn(alo[b], ahi[b]);
        out[b] = t.x + t.y;
    }
}

// exact dequantized weight of Q4_K
__device__ __forceinline__ float q4k_weight(float dsc, float dm, float q) {
    return fmaf(dsc, q, -dm);
}

// ---------------------------------------------------------------- Q6_K

// Four 6-bit codes per quarter from ql word A (quarters 0 and 2), ql word Bw
// (quarters 1 and 3) and qh word H (2 high bits of each, quarters 0..3 in bit
// pairs 0-1, 2-3, 4-5, 6-7).  Byte k of the result is the code of column k.
__device__ __forceinline__ void q6k_codes(uint32_t A, uint32_t Bw, uint32_t H, uint32_t& c0,
                                          uint32_t& c1, uint32_t& c2, uint32_t& c3) {
    c0 = (A & 0x0F0F0F0Fu) | ((H << 4) & 0x30303030u);
    c1 = (Bw & 0x0F0F0F0Fu) | ((H << 2) & 0x30303030u);
    c2 = ((A >> 4) & 0x0F0F0F0Fu) | (H & 0x30303030u);
    c3 = ((Bw >> 4) & 0x0F0F0F0Fu) | ((H >> 2) & 0x30303030u);
}

// code byte k of c as the exact float (code - 32), paired with byte k of c'.
__device__ __forceinline__ float2 q6k_pair(uint32_t c, uint32_t cp, uint32_t sel) {
    return __fadd2_rn(make_float2(as_f(prmt(c, 0x4B000000u, sel)), as_f(prmt(cp, 0x4B000000u, sel))),
                      make_float2(-8388640.0f, -8388640.0f));
}

// Leaf = one word of each of A, Bw, H: 4 columns in each of the 4 quarters.
// xr[b][l][k] (k < 4) = (col of quarter 0, col of quarter 1) for column k,
// xr[b][l][4+k] = (quarter 2, quarter 3).  dsc01 = (d*sc_q0, d*sc_q1), dsc23 alike.
template <int B, int NL>
__device__ __forceinline__ void q6k_leaf(uint32_t A, uint32_t Bw, uint32_t H, float2 dsc01,
                                         float2 dsc23, const float2 (&xr)[B][NL][8], int l,
                                         float* out) {
    uint32_t c0, c1, c2, c3;
    q6k_codes(A, Bw, H, c0, c1, c2, c3);
    float2 a01[B], a23[B];
#pragma unroll
    for (int b = 0; b < B; ++b) a01[b] = a23[b] = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t sel = 0x7440u | k;
        const float2 q01 = q6k_pair(c0, c1, sel);
        const float2 q23 = q6k_pair(c2, c3, sel);
#pragma unroll
        for (int b = 0; b < B; ++b) {
            a01[b] = __ffma2_rn(q01, xr[b][l][k], a01[b]);
            a23[b] = __ffma2_rn(q23, xr[b][l][4 + k], a23[b]);
        }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
        float2 t = __fmul2_rn(dsc01, a01[b]);
        t = __ffma2_rn(dsc23, a23[b], t);
        out[b] = t.x + t.y;
    }
}

// ---------------------------------------------------------------- Q8_0

__device__ __forceinline__ float2 q80_pair(uint32_t Qb, uint32_t sel0, uint32_t sel1) {
    return __fadd2_rn(make_float2(as_f(prmt(Qb, 0x4B000000u, sel0)), as_f(prmt(Qb, 0x4B000000u, sel1))),
                      make_float2(-8388736.0f, -8388736.0f));
}

// Leaf = 16 int8 quants (4 words) of one block half, scale d.
template <int B, int NL>
__device__ __forceinline__ void q80_leaf(const uint32_t* Q, float d, const float2 (&xr)[B][NL][8],
                                         int l, float* out) {
    float2 a0[B], a1[B];
#pragma unroll
    for (int b = 0; b < B; ++b) a0[b] = a1[b] = make_float2(0.f, 0.f);
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        const uint32_t Qb = Q[wi] ^ 0x80808080u;   // int8 -> unsigned q + 128
        const float2 q01 = q80_pair(Qb, 0x7440u, 0x7441u);
        const float2 q23 = q80_pair(Qb, 0x7442u, 0x7443u);
#pragma unroll
        for (int b = 0; b < B; ++b) {
            a0[b] = __ffma2_rn(q01, xr[b][l][2 * wi + 0], a0[b]);
            a1[b] = __ffma2_rn(q23, xr[b][l][2 * wi + 1], a1[b]);
        }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
        const float2 t = __fadd2_rn(a0[b], a1[b]);
        out[b] = d * (t.x + t.y);
    }
}

// ---------------------------------------------------------------- columns
// Column (within the row) of x pair element e (0 = .x, 1 = .y) of pair i
// (0..7) of leaf lam (0..3) of group G, per format.
__host__ __device__ __forceinline__ int leaf_col(int fmt, int G, int lam, int i, int e) {
    if (fmt == FMT_Q4_K) {
        // group G = block G/4, quant group g = G%4; leaf covers qs bytes
        // 32g + 8lam .. +7: low nibbles -> cols 64G + 8lam + 0..7, high
        // nibbles -> 64G + 32 + 8lam + 0..7.
        const int base = 64 * G + 8 * lam;
        return i < 4 ? base + 2 * i + e : base + 32 + 2 * (i - 4) + e;
    } else if (fmt == FMT_Q6_K) {
        // group G = block G/4, gamma = G%4: half h = gamma/2, l0 = 16*(gamma%2);
        // leaf columns l = l0 + 4lam + k: quarter q -> 128h + 32q + l.
        const int blk = G >> 2, gm = G & 3, h = gm >> 1, l0 = 16 * (gm & 1);
        const int base = 256 * blk + 128 * h + l0 + 4 * lam;
        return i < 4 ? base + 32 * e + i : base + 64 + 32 * e + (i - 4);
    } else {
        // group G = blocks 2G, 2G+1; leaf lam = 16 consecutive columns.
        return 64 * G + 16 * lam + 2 * i + e;
    }
}

}  // namespace lq
