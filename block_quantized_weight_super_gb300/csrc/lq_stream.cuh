// lq_stream.cuh -- segment descriptors of the quantized matvec kernel
// (shared by the kernel translation units and the host launchers).
#pragma once
#include <cmath>
#include <cstdint>

namespace lq {

constexpr int MAX_SEG = 36;

enum { MODE_PLAIN = 0, MODE_PAIR_INTERLEAVED = 1, MODE_PAIR_TWO = 2 };
enum { ACT_NONE = 0, ACT_GEGLU_TANH = 1, ACT_SWIGLU = 2 };

// One weight matrix (or gate/up matrix pair) of a launch, with where its x
// rows come from and where its outputs go.  Batch row b of the segment is
// rho_b = (*boff or 0) + b0 + b; its x row is x + (xmap ? xmap[rho_b] : rho_b)
// * cols and its output row is y + rho_b * ld_y.  With xact set, x rows hold
// (g, u) pairs (2 cols floats, g at even positions) and the matvec's x value
// of column j is act(g_j) * u_j; the CTA that stages the segment for its
// first tile also stores those values to xout + rho_b * cols (if non-null).
struct Seg {
    const uint8_t* w;      // matrix (plain / interleaved pairs) or gate matrix
    const uint8_t* w2;     // up matrix (MODE_PAIR_TWO)
    const float* x;
    const int32_t* xmap;   // optional device gather list
    float* y;
    const int32_t* boff;   // optional device offset of batch row 0
    const int32_t* bcnt;   // optional device count of rows from boff (valid rows: b0 + b < cnt)
    int64_t ld_y;
    int32_t nout;          // output rows (plain) or output pairs (pair modes)
    int32_t fmt;
    int32_t mode;
    int32_t act;
    int32_t b0;
    int32_t nbatch;        // valid batch rows when bcnt is null
    int32_t tile0;         // first global tile index of this segment
    int32_t ntiles;
    float cap;             // > 0: plain outputs are cap * tanh(y / cap) (final-logit soft-cap)
    int32_t xact;          // ACT_NONE, or the activation applied to (g, u) pairs of x
    float* xout;           // with xact: the activated x rows, stored once
};

#ifdef __CUDACC__
// The gated activations of the FFN (larql Gemma 3 table: GEGLU with
// GELU-tanh; dotLLM: SwiGLU with SiLU).  GELU-tanh in the form
// g / (1 + exp(-2z)), z = sqrt(2/pi) (g + 0.044715 g^3), which equals
// 0.5 g (1 + tanh(z)); SiLU g / (1 + exp(-g)).  fp32.
__device__ __forceinline__ float act_eval(int act, float g) {
    if (act == ACT_GEGLU_TANH) {
        const float z = 0.7978845608028654f * fmaf(0.044715f * g, g * g, g);
        return g / (1.0f + expf(-2.0f * z));
    }
    return g / (1.0f + expf(-g));
}

// Four consecutive x values of a row as the matvec sees them: a float4 of
// the row (16-byte aligned), or act(g) * u of four (g, u) pairs.
template <bool COHERENT>
__device__ __forceinline__ float4 load_x4(const float* row, int col, int xact) {
    if (!xact) {
        const float4* p = reinterpret_cast<const float4*>(row + col);
        return COHERENT ? __ldcg(p) : __ldg(p);
    }
    const float4* p = reinterpret_cast<const float4*>(row + 2 * col);
    const float4 a = COHERENT ? __ldcg(p) : __ldg(p), b = COHERENT ? __ldcg(p + 1) : __ldg(p + 1);
    return make_float4(act_eval(xact, a.x) * a.y, act_eval(xact, a.z) * a.w, act_eval(xact, b.x) * b.y,
                       act_eval(xact, b.z) * b.w);
}
#endif

// The stored value of a plain segment's output y (dotLLM PR #255 soft-cap
// s -> softCap * tanh(s / softCap), applied to the logits after the lm_head
// GEMM by PR #274's FinalLogitSoftcap).
__host__ __device__ inline float seg_out(float cap, float y) { return cap > 0.f ? cap * tanhf(y / cap) : y; }

}  // namespace lq
