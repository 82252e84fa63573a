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
// * cols and its output row is y + rho_b * ld_y.
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
};

// The stored value of a plain segment's output y (dotLLM PR #255 soft-cap
// s -> softCap * tanh(s / softCap), applied to the logits after the lm_head
// GEMM by PR #274's FinalLogitSoftcap).
__host__ __device__ inline float seg_out(float cap, float y) { return cap > 0.f ? cap * tanhf(y / cap) : y; }

}  // namespace lq
