/* lq.h -- C ABI of the block-quantized decode matvec library (liblq.so).
 *
 * The library computes the matrix-vector products of LLM decoding against
 * GGUF-style block-quantized weights on one NVIDIA GB300 (sm_103a).  Every
 * call is asynchronous on the caller's CUDA stream, validates its arguments
 * on the host before launching anything, allocates nothing, and returns an
 * lq_status (LQ_OK = 0).  No C++ exception crosses this boundary.
 *
 * Sources of the operations (pages cited by title and section):
 *  - larql "Architecture -> Metal shader map": the Gemma 3 table names the
 *    production kernels of one decode layer -- q4k_q6k_qkv_proj (QKV,
 *    Q4_K Q/K + Q6_K V), q4k_matvec_8sg (O projection), q4k_ffn_gate_up_8sg +
 *    geglu (FFN gate+up, GELU-tanh), q6k_matvec (FFN down), q4k_matvec
 *    (lm_head); the Llama table the SiLU variant; the dispatch-predicate table
 *    the 144-byte Q4_K ("Q4_KF", GGUF-direct) block; the Gemma 4 26B-A4B table
 *    the MoE gate scoring (f32_gemv), per-expert gate_up + down, and combine.
 *  - dotLLM PR #320: the Q8_0 GEMV (matmul_q8_0) and its row-stride fix
 *    (row stride = blocksPerRow * 34 bytes); the LoRA Q8_0 commit (inputs
 *    must be a multiple of the 32-element group, otherwise rejected); the MoE
 *    commit (MoeSwiGluMlp: softmax over experts, top-k with the lower index
 *    winning ties, renormalise by the selected sum, per-expert SwiGLU,
 *    weighted sum); ForwardBatch (batched rows of activations [sum N_i][K]).
 *
 * Layout conventions (all calls):
 *  - W is row-major block rows: row r starts at W + r * lq_row_bytes(fmt, cols)
 *    and holds cols / lq_block_elems(fmt) consecutive blocks.  W must be
 *    2-byte aligned (16-byte alignment is the fast path, not a requirement).
 *  - x is [batch][cols] fp32 row-major, y is [batch][rows] fp32 row-major
 *    (4-byte aligned).
 *  - cols must be a multiple of the format's block (LQ_ESHAPE otherwise);
 *    rows == 0 (or ntok == 0) returns LQ_OK without launching.
 *  - Numerics: dequantized weights are exact fp32 (Q4_K: one rounding of
 *    d*sc*q - dmin*m; Q6_K, Q8_0: exact); dot products accumulate in fp32
 *    with short fixed-order chains; each output is within
 *    1e-5 * sum_j |w_ij x_j| + 1e-6 of the exact value.  Results are
 *    deterministic.  Kernel choice (by shape and alignment only):
 *    batch-1 calls with Q4_K weights (alone, or with Q6_K in one QKV
 *    launch), cols a multiple of 256 and 16-row tiles of at most 48 KB run
 *    on the batch-1 tensor-core kernel; batch-1 calls of one Q4_K or Q6_K
 *    matrix that it does not take, with W 16-byte aligned and rows a
 *    multiple of 16 bytes, run on its column-chunked form (16-row x 7 or 8
 *    super-block items spread evenly over the SMs; a matrix with several
 *    chunks per row and at least 4 row blocks per SM stays on the CUDA-core
 *    kernel), and so do Q6_K calls of 3 to 8 x rows with more than 2048
 *    columns (each weight fragment used by one MMA per x row); Q4_K calls
 *    with batch >= 2 and Q8_0 calls with batch >= 3
 *    whose cols are a multiple of 512 (Q4_K) or 256 (Q8_0), with W and x
 *    16-byte aligned, run on the batched tensor-core kernel (exact bf16 /
 *    fp16 codes times x split into two pieces, fp32 sums); every other call
 *    runs the CUDA-core matvec kernel, or, when x is not 16-byte aligned or
 *    the width cannot be tiled, a plain-load kernel.  Within one kernel row
 *    b of a batch call equals, bit for bit, the same x row in any other
 *    batch width; across kernels results differ only by rounding (all
 *    within the bound).  The grouped MoE expert FFN uses the tensor cores for
 *    Q4_K / Q8_0 when ntok >= 2.
 *  - Streams: calls on different streams may run concurrently.  The
 *    column-chunked batch-1 kernel adds the chunk sums of a row through one
 *    of 4 scratch sets inside the library (static device memory, no
 *    allocation), each bound to the first stream that needs it for the
 *    life of the CUDA context; a call on a fifth stream runs on the CUDA-core
 *    kernel instead.  A captured graph holding such a call must not run
 *    concurrently with other work of the stream it was captured on.
 *  - Pointers are device pointers unless stated; the caller owns all memory.
 *  - stream may be NULL (the legacy default stream).
 */
#ifndef LQ_H_
#define LQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* lq_stream_t; /* a cudaStream_t */

typedef enum { LQ_Q4_K = 1, LQ_Q6_K = 2, LQ_Q8_0 = 3 } lq_fmt;
typedef enum { LQ_ACT_GEGLU_TANH = 1, LQ_ACT_SWIGLU = 2 } lq_act;
typedef enum {
    LQ_OK = 0,
    LQ_EINVAL = 1,      /* null pointer, batch < 1, bad topk, unknown enum      */
    LQ_EALIGN = 2,      /* W not 2-byte aligned, or x / y not 4-byte aligned     */
    LQ_ESHAPE = 3,      /* cols not a multiple of the block, sizes out of range  */
    LQ_EWORKSPACE = 4,  /* workspace smaller than lq_moe_workspace_bytes         */
    LQ_ECUDA = 5,       /* a CUDA launch or query failed (see lq_last_error)     */
    LQ_ETIMEOUT = 6,    /* a kernel's bounded wait ran out (lq_device_status)    */
    LQ_EUNSUPPORTED = 7 /* a combination the library does not implement          */
} lq_status;

/* Format facts.  Q4_K: 144 bytes / 256 weights; Q6_K: 210 / 256; Q8_0: 34 / 32.
 * Unknown formats return 0. */
size_t lq_block_bytes(int fmt);
int lq_block_elems(int fmt);
int64_t lq_row_bytes(int fmt, int64_t cols); /* 0 if cols is not a block multiple */

const char* lq_status_str(int status);
/* Detail of the last failure on the calling thread ("" if none). */
const char* lq_last_error(void);

/* lq_dequant -- out[r][c] = w_rc as fp32 for a rows x cols matrix.
 * Exact: equals the definition bit for bit.  out: [rows][cols] fp32. */
int lq_dequant(int fmt, const void* W, int64_t rows, int64_t cols, float* out,
               lq_stream_t stream);

/* lq_matvec -- y[b][r] = sum_j w_rj x[b][j] for b < batch (batch >= 1).
 * larql Gemma 3 table (q4k_matvec, q6k_matvec); dotLLM matmul_q8_0 GEMV. */
int lq_matvec(int fmt, const void* W, int64_t rows, int64_t cols, const float* x, float* y,
              int batch, lq_stream_t stream);

/* lq_matvec_softcap -- lq_matvec with the final-logit soft-cap fused into the
 * store: y[b][r] = cap * tanh((sum_j w_rj x[b][j]) / cap).  dotLLM PR #255
 * (soft-cap s -> softCap * tanh(s / softCap)) and PR #274 (FinalLogitSoftcap,
 * applied to the logits after the lm_head GEMM; Gemma 4 configs carry
 * final_logit_softcapping = 30).  cap must be finite and > 0 (LQ_EINVAL
 * otherwise).  Every output lies in [-cap, cap]; its error is the matvec
 * bound (the map has slope at most 1) plus a few ulps of the fp32 tanh. */
int lq_matvec_softcap(int fmt, const void* W, int64_t rows, int64_t cols, const float* x, float* y,
                      int batch, float cap, lq_stream_t stream);

/* lq_matvec_act -- y[b][r] = sum_j w_rj h[b][j] with h[b][j] = act(g_j) * u_j
 * formed as the matvec loads its input: the activation fused into the down
 * projection's x-load (larql "Architecture -> Metal shader map", Gemma 4
 * 26B-A4B section, Expert FFN row: q4k_ffn_gate_up followed by
 * q4k_geglu_down).  gu: [batch][2 cols] (g, u) pairs, g at even positions:
 * the output of lq_matvec over an interleaved Wgu (lq_pack_gate_up).
 * h: [batch][cols] (written: the activated input, not overlapping gu),
 * y: [batch][rows].  act as lq_ffn_gate_up_act.  Where the kernel that runs
 * cannot form h while loading (the batched tensor-core kernel, the
 * plain-load kernel), h is formed by a separate launch first; the results
 * are the same within the matvec bound.  rows == 0: nothing is launched. */
int lq_matvec_act(int fmt, const void* W, int64_t rows, int64_t cols, const float* gu, float* h, float* y,
                  int batch, int act, lq_stream_t stream);

/* lq_gemm -- the prefill GEMM: Y[n][r] = sum_j w_rj X[n][j] for M x rows
 * (X: [M][cols] fp32, Y: [M][rows] fp32), the same values as lq_matvec
 * within the same bound.  dotLLM PR #320: the tiled matmul_q8_0_gemm for
 * many tokens (parity over a grid of (M, K, N)) and ForwardBatch's batched
 * GEMMs; Q4_K weights as in the larql tables.  Q4_K and Q8_0 weights with
 * cols a multiple of 256, 16-byte aligned W and X, and M >= LQ_GEMM_MIN_M
 * run on the tcgen05 tensor-core kernel (each weight tile read once per 128
 * or 256 x rows); a row's result depends only on the row, W and its shape,
 * not on M or on the other rows.  Other calls run lq_matvec's batched
 * kernels (a pass over the weights per 8 x rows) and leave the workspace
 * untouched.
 * workspace: lq_gemm_workspace_bytes(M, rows, cols) bytes, 256-byte
 * aligned (LQ_EWORKSPACE / LQ_EALIGN otherwise, checked when the tiled
 * kernel runs): the fp16 pieces of x that the kernel reads, a scale per
 * weight row and, for matrices of few rows, partial sums over K ranges.
 * Sizes < 0 give 0. */
#define LQ_GEMM_MIN_M 32
size_t lq_gemm_workspace_bytes(int64_t M, int64_t rows, int64_t cols);
int lq_gemm(int fmt, const void* W, int64_t rows, int64_t cols, const float* X, float* Y, int64_t M,
            void* workspace, size_t ws_bytes, lq_stream_t stream);

/* lq_gemm_gate_up_act -- the prefill FFN's gate and up GEMMs with the
 * activation fused before the store: H[n][i] = act(g_i . X[n]) * (u_i . X[n])
 * over the packed matrix Wgu of lq_pack_gate_up (rows 2i, 2i + 1 the gate
 * and up rows of output i; [2 inter][cols]) for M x rows (X: [M][cols],
 * H: [M][inter] fp32).  The prefill counterpart of lq_ffn_gate_up_act
 * (larql Gemma 3 table, FFN gate+up row; dotLLM PR #320 ForwardBatch for
 * the many-token form): the same kernel and conditions as lq_gemm, with the
 * x pieces built once for both matrices; other calls run the batched
 * lq_ffn_gate_up_act kernels.  act as lq_ffn_gate_up_act (LQ_EINVAL
 * otherwise).  workspace: lq_gemm_workspace_bytes(M, 2 * inter, cols)
 * bytes, 256-byte aligned.  Each output is within the bound the oracle's
 * gate_up check states for the matvec bounds of g and u. */
int lq_gemm_gate_up_act(int fmt, const void* Wgu, int64_t inter, int64_t cols, const float* X, float* H, int64_t M,
                        int act, void* workspace, size_t ws_bytes, lq_stream_t stream);

/* lq_gemv_f16, lq_gemv_f32 -- y[b][r] = sum_j W[r][j] x[b][j] for a
 * non-quantized W, fp16 or fp32, [rows][cols] row-major, 16-byte aligned:
 * the lm_head fallbacks for a tied embedding that is not block-quantized
 * (larql Gemma 3 table, lm_head row: the f16_gemv / f32_gemv fallback
 * chain).  fp32 accumulation; the results are within the matvec bound.
 * cols a multiple of 8 (fp16) or 4 (fp32); batch 1..8 with batch * cols *
 * 4 <= 200 KB (LQ_ESHAPE / LQ_EINVAL otherwise); x 16-byte aligned. */
int lq_gemv_f16(const void* W, int64_t rows, int64_t cols, const float* x, float* y, int batch, lq_stream_t stream);
int lq_gemv_f32(const float* W, int64_t rows, int64_t cols, const float* x, float* y, int batch, lq_stream_t stream);

/* lq_rmsnorm -- out[t][j] = x[t][j] * w[j] / sqrt(mean_j(x[t][j]^2) + eps)
 * for ntok rows of n values (larql Gemma 3 table, "Input RMS-norm" row;
 * the stored weight already carries any offset, eps from the model config).
 * fp32, the sum of squares in a fixed order; out may equal x. */
int lq_rmsnorm(const float* x, const float* w, float eps, float* out, int ntok, int64_t n, lq_stream_t stream);

/* lq_qkv_mixed -- q = Wq.x, k = Wk.x, v = Wv.x in ONE launch over a shared
 * x (larql q4k_q6k_qkv_proj: Q/K Q4_K and V Q6_K, or uniform formats).
 * Each matrix has its own format and row count; all share cols.
 * q: [batch][nq], k: [batch][nk], v: [batch][nv]. */
int lq_qkv_mixed(int fq, const void* Wq, int64_t nq, int fk, const void* Wk, int64_t nk, int fv,
                 const void* Wv, int64_t nv, int64_t cols, const float* x, float* q, float* k,
                 float* v, int batch, lq_stream_t stream);

/* lq_qkv_mixed_rmsnorm -- lq_qkv_mixed of the RMS-normed input:
 * xn = lq_rmsnorm(x, norm_w, eps), then q, k, v from xn (larql Gemma 3
 * table, "Input RMS-norm" and "QKV projection" rows: the opt-in variant
 * that fuses the norm into the projection).  At batch 1 on the tensor-core
 * kernel every CTA computes the row's norm while it builds its x operand
 * (one launch) and CTA 0 stores xn; elsewhere the norm is a launch of its
 * own.  xn: [batch][cols] (written; must not overlap x), norm_w: [cols],
 * eps finite and >= 0 (LQ_EINVAL otherwise). */
int lq_qkv_mixed_rmsnorm(int fq, const void* Wq, int64_t nq, int fk, const void* Wk, int64_t nk, int fv,
                         const void* Wv, int64_t nv, int64_t cols, const float* x, const float* norm_w, float eps,
                         float* xn, float* q, float* k, float* v, int batch, lq_stream_t stream);

/* lq_pack_gate_up -- one-time repack of separate gate and up matrices
 * (inter x cols each, same format) into the interleaved layout the fused
 * kernel reads: row 2i = gate row i, row 2i+1 = up row i.
 * Wgu_out: 2 * inter * lq_row_bytes(fmt, cols) bytes. */
int lq_pack_gate_up(int fmt, const void* Wg, const void* Wu, int64_t inter, int64_t cols,
                    void* Wgu_out, lq_stream_t stream);

/* lq_ffn_gate_up_act -- h[b][i] = act(g) * u with g = (gate row i).x_b,
 * u = (up row i).x_b, from the interleaved Wgu (lq_pack_gate_up), the
 * activation fused before the store.  act: LQ_ACT_GEGLU_TANH
 * (0.5 g (1 + tanh(sqrt(2/pi)(g + 0.044715 g^3)))) or LQ_ACT_SWIGLU
 * (g / (1 + exp(-g))).  larql q4k_ffn_gate_up_8sg + geglu.  h: [batch][inter]. */
int lq_ffn_gate_up_act(int fmt, const void* Wgu, int64_t inter, int64_t cols, const float* x,
                       float* h, int batch, int act, lq_stream_t stream);

/* lq_ffn_gate_up_act_rmsnorm -- lq_ffn_gate_up_act of the RMS-normed input
 * (the pre-FFN norm), fused as lq_qkv_mixed_rmsnorm fuses the input norm;
 * xn, norm_w, eps as there.  The pages fuse the norm only in front of QKV;
 * this applies the same fusion to the FFN's own input norm. */
int lq_ffn_gate_up_act_rmsnorm(int fmt, const void* Wgu, int64_t inter, int64_t cols, const float* x,
                               const float* norm_w, float eps, float* xn, float* h, int batch, int act,
                               lq_stream_t stream);

/* lq_ffn -- the dense FFN of a decode step: h = act(Wg.x) * (Wu.x) by
 * lq_ffn_gate_up_act (interleaved Wgu, format fmt_gu, inter pairs x hidden
 * columns), then y = Wd.h by lq_matvec (Wd: hidden rows x inter columns,
 * format fmt_down).  larql "Architecture -> Metal shader map", Gemma 3 table:
 * q4k_ffn_gate_up + geglu feeding the Q6_K down projection.
 * x: [batch][hidden], h: [batch][inter] (written: the intermediate), y:
 * [batch][hidden]; h overlaps neither x nor y.  Two launches, on stream.
 * inter == 0 or hidden == 0 -> LQ_ESHAPE. */
int lq_ffn(int fmt_gu, const void* Wgu, int fmt_down, const void* Wd, int64_t inter, int64_t hidden,
           const float* x, float* h, float* y, int batch, int act, lq_stream_t stream);

/* MoE expert FFN (dotLLM MoeSwiGluMlp rule; larql Gemma 4 26B-A4B table).
 * router: [E][hidden] fp32; logits l_e = router_e . x_t, p = softmax(l),
 * top-k experts (lower index wins ties), weights p / sum of selected p;
 * Y_t = sum_k w_tk * W2_e (silu(W1_e x_t) * (W3_e x_t)), e = the k-th pick
 * (W1 = gate, W3 = up: inter x hidden; W2 = down: hidden x inter; all fmt).
 * W1, W3, W2 are HOST arrays of E device pointers.  X, Y: [ntok][hidden].
 * topk_idx / topk_w (optional, may be NULL): [ntok][topk] outputs of the
 * routing.  workspace: device memory of at least lq_moe_workspace_bytes
 * bytes, 256-byte aligned; its contents are scratch. */
size_t lq_moe_workspace_bytes(int n_experts, int topk, int ntok, int64_t hidden, int64_t inter);
int lq_moe_ffn(const float* router, int n_experts, int topk, int fmt, const void* const* W1,
               const void* const* W3, const void* const* W2, int64_t hidden, int64_t inter,
               const float* X, float* Y, int ntok, int32_t* topk_idx, float* topk_w,
               void* workspace, size_t ws_bytes, lq_stream_t stream);

/* lq_moe_ffn_ex -- lq_moe_ffn with the MoE variants of dotLLM PR #320 (the
 * Qwen-MoE commit and its N-shared-experts follow-up):
 *   norm_topk_prob: 1 renormalises the selected weights by their sum (the
 *     lq_moe_ffn rule); 0 keeps the selected softmax probabilities p_e as
 *     they are (norm_topk_prob = false).
 *   n_shared (0..LQ_MOE_MAX_SHARED) shared experts, dense SwiGLU FFNs that
 *     every token passes through: Ws1 (gate), Ws3 (up): inter_s x hidden,
 *     Ws2 (down): hidden x inter_s, format fmt; HOST arrays of n_shared device
 *     pointers (NULL when n_shared == 0).  Their outputs are summed in expert
 *     order and added to the routed sum:
 *       Y_t = sum_k w_tk * E_k(x_t) + gate_t * sum_s S_s(x_t)
 *   shared_gate: optional [hidden] fp32 vector g; gate_t = sigmoid(g . x_t)
 *     scales the sum of the shared experts (NULL: gate_t = 1).  A gate
 *     without shared experts -> LQ_EINVAL.
 * The shared experts run as extra dense segments of the grouped gate/up and
 * down launches (in the same launch when they take the same kernel and, for
 * down, the same width); the gate is computed in the routing launch and
 * applied in the combine.  workspace: lq_moe_ffn_ex_workspace_bytes bytes,
 * 256-byte aligned.  Other arguments, outputs and errors as lq_moe_ffn. */
#define LQ_MOE_MAX_SHARED 16
size_t lq_moe_ffn_ex_workspace_bytes(int n_experts, int topk, int ntok, int64_t hidden, int64_t inter,
                                     int n_shared, int64_t inter_s);
int lq_moe_ffn_ex(const float* router, int n_experts, int topk, int norm_topk_prob, int fmt,
                  const void* const* W1, const void* const* W3, const void* const* W2, int64_t hidden,
                  int64_t inter, int n_shared, const void* const* Ws1, const void* const* Ws3,
                  const void* const* Ws2, int64_t inter_s, const float* shared_gate, const float* X, float* Y,
                  int ntok, int32_t* topk_idx, float* topk_w, void* workspace, size_t ws_bytes,
                  lq_stream_t stream);

/* lq_moe_ffn_static -- lq_moe_ffn without a caller-supplied workspace: the
 * scratch is a static device array of LQ_MOE_STATIC_SCRATCH_BYTES (4 MiB)
 * inside the library, one per device, and the call allocates no device
 * memory (no cudaMalloc / cudaFree or allocating routine, on any call).
 * The method's description has no such call; it is for callers that cannot
 * allocate, e.g. a plain C caller without a device allocator, or a serving
 * process whose device memory is all reserved by another allocator, where a
 * cudaMalloc would fail and a cudaFree would synchronise the device.
 *   Arguments, results and errors are those of lq_moe_ffn (without
 * workspace, ws_bytes).  Shapes whose lq_moe_workspace_bytes exceeds
 * LQ_MOE_STATIC_SCRATCH_BYTES are rejected with LQ_EWORKSPACE (e.g.
 * hidden 4096, inter 14336 fit up to ntok * topk = 56).
 *   The first call on a device does the set-up (looks up the scratch
 * address with that device current) and returns LQ_ECUDA if that fails;
 * make it before any stream capture.  The address is kept per device and
 * CUDA context: after cudaDeviceReset the next call looks it up again.
 * Arguments are validated before the size check (LQ_EINVAL, LQ_ESHAPE,
 * LQ_EALIGN come before LQ_EWORKSPACE).  No part of the scratch needs to start
 * at zero: every word a call reads was written earlier in the same call.
 * All calls on a device share the one scratch: calls that overlap in time
 * (on different streams, or from different host threads without ordering)
 * race on it; calls in order on one stream do not. */
#define LQ_MOE_STATIC_SCRATCH_BYTES (4u << 20)
int lq_moe_ffn_static(const float* router, int n_experts, int topk, int fmt, const void* const* W1,
                      const void* const* W3, const void* const* W2, int64_t hidden, int64_t inter,
                      const float* X, float* Y, int ntok, int32_t* topk_idx, float* topk_w,
                      lq_stream_t stream);

/* lq_device_status -- waits for all work on the current device (every
 * stream: the status word is one per device, shared by every launch of the
 * library, so a bit set by a launch on another stream is reported here
 * too), then reads and clears the word that kernels set when a bounded wait
 * runs out.  *bits = the word (0 = clean).  Returns LQ_ETIMEOUT if the
 * timeout bit was set, LQ_OK otherwise (LQ_ECUDA on a CUDA error).  `stream`
 * is accepted for symmetry with the other calls; the wait covers it. */
int lq_device_status(lq_stream_t stream, uint32_t* bits);

/* lq_set_wait_timeout_ns -- wall-time limit of every bounded wait in later
 * launches (default 1e9 ns).  Process-wide.  The waits with which a CTA lets
 * its own copies and MMAs in flight finish before it exits use at least
 * 10 ms whatever this limit. */
void lq_set_wait_timeout_ns(uint64_t ns);

/* lq_probe_timeout -- failure-detection check: launches a kernel that waits,
 * with the bounded wait, on a barrier nothing completes; after timeout_ns it
 * records the timeout in the device status word and exits.  Follow with
 * lq_device_status to observe LQ_ETIMEOUT. */
int lq_probe_timeout(uint64_t timeout_ns, lq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* LQ_H_ */
