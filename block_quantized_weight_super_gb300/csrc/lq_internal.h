// lq_internal.h -- launchers shared between the library's translation units.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "lq_qmv.cuh"

namespace lq {

// MoE workspace views (device memory carved from the caller's workspace).
struct MoeWs {
    int32_t* idx;        // [ntok*topk] selected experts
    float* w;            // [ntok*topk] renormalised weights
    int32_t* tok_of;     // [ntok*topk] token of each grouped row
    int32_t* slot_row;   // [ntok*topk] grouped row of each (token, slot)
    int32_t* grp_off;    // [E] first grouped row of each expert
    int32_t* grp_cnt;    // [E] grouped rows of each expert
    float* hbuf;         // [ntok*topk][inter] expert hidden activations
    float* ybuf;         // [ntok*topk][hidden] expert outputs
    float* sgate;        // [ntok] shared-expert gate sigmoid(g . x_t) (when a gate vector is given)
    float* hsh;          // [nshared][ntok][inter_s] shared-expert hidden activations
    float* ysh;          // [nshared][ntok][hidden] shared-expert outputs
    int32_t nshared;
    int32_t norm;        // 1: weights renormalised by the selected sum; 0: raw softmax probabilities
};

// tensor-core matvec for up to QMM_NT x rows of Q4_K or Q8_0 (lq_qmm.cu):
// tiles of QMM_RT weight rows x QMM_KC (Q4_K) or QMM_KC8 (Q8_0) columns;
// segments' tile0 = first row block.
// Weights are fetched through 2-D tensor maps (uint32 elements, one row of
// the matrix per tensor row): per segment map 0 is the plain matrix (boxes of
// QMM_RT rows) or the gate rows of a pair segment, map 1 the up rows (boxes
// of 8 rows; packed gate/up matrices use a row stride of two rows).
constexpr int QMM_NT = 8;
constexpr int QMM_RT = 64;
constexpr int QMM_KC = 512;             // Q4_K tile columns (two super-blocks)
constexpr int QMM_KC8 = 256;            // Q8_0 tile columns (eight blocks)
constexpr int QMM_MAX_SEG = 16;
constexpr int QMM_PAIR_BOX = 8;
struct QmmParams {
    CUtensorMap tm[QMM_MAX_SEG][2];
    Seg seg[QMM_MAX_SEG];
    int32_t nseg;
    int32_t nblocks;         // row blocks over all segments
    int32_t cols;
    int32_t nchunk;          // cols / QMM_KC
    int32_t nstages;
    int32_t csize;           // CTAs per cluster splitting a row block's columns (1, 2 or 4)
    int32_t gmax;            // row blocks per group (<= QMM_GROUP): partial-sum slots
    int32_t dev_counts;      // segments read row counts / offsets written by the preceding kernel
    uint64_t timeout_ns;
    unsigned* status;
};
constexpr int QMM_MAX_CSIZE = 4;
constexpr int QMM_GROUP = 4;              // row blocks sharing one staging of x
constexpr int QMM_MIN_BATCH = 2;          // dense Q4_K calls with at least this many x rows
constexpr int QMM_MIN_BATCH_Q8 = 3;       // dense Q8_0 calls
constexpr int QMM_MOE_MIN_TOKENS = 2;     // MoE calls with at least this many tokens
bool qmm_format_ok(int fmt);             // Q4_K, Q8_0
int qmm_kc(int fmt);                     // columns per tile
int qmm_wrow(int fmt);                   // weight bytes of a row per tile
cudaError_t qmm_set_smem(int fmt, int bytes);
size_t qmm_smem_bytes(int fmt, int nstages, int csize, int gmax);
cudaError_t qmm_max_resident(int fmt, int csize, size_t smem, int sms, int* out);
cudaError_t qmm_launch(int fmt, const QmmParams& P, int grid, size_t smem, cudaStream_t st);

// batch-1 tensor-core matvec (lq_gv.cu): one CTA of GV_NW warps per SM;
// segments share x and the column count; row blocks of 16 rows (8 gate/up
// pairs) over all segments are numbered from 0 (seg.rb0 = the first).  CTA k
// takes row blocks [cta_rb[k], cta_rb[k+1]), each as one tile of whole rows
// landing in one of nslots shared-memory slots of slot_bytes: GV_COPY_TILE
// copies the 16 contiguous rows at once (w 16-byte aligned, the matrix a
// multiple of 16 bytes), GV_COPY_CPA uses 4-byte cp.async copies at a row
// pitch of `pitch` (w 4-byte aligned); rows are a multiple of 4 bytes.
// mask: bit 0 Q4_K, bit 1 Q6_K; masks 1 (Q4_K) and 3 (both) are built.
constexpr int GV_MAX_SEG = 4;
constexpr int GV_MAX_CTA = 160;
constexpr int GV_MAX_INFLIGHT = 6;     // tiles in flight per CTA (more delays the first tile)
constexpr int GV_MAX_TILES = 512;
constexpr int GV_MAX_TILE_BYTES = 48 * 1024;
constexpr int GV_MAX_NSB = 24;          // 256-column units per row (the x image build's reach)
enum { GV_COPY_TILE = 0, GV_COPY_CPA = 1 };
struct GvSeg {
    const uint8_t* w;        // plain matrix or interleaved gate/up pairs (row 2i gate, 2i+1 up)
    float* y;
    int64_t rowbytes;
    int32_t fmt, mode, copy, act;
    int32_t nout;            // outputs: rows (plain) or pairs
    int32_t nrows;           // matrix rows
    int32_t rb0, nrb;        // first row block, row blocks
    int32_t pitch;           // shared row pitch of GV_COPY_CPA tiles
    float cap;               // > 0: plain outputs are cap * tanh(y / cap)
};
// GV_X_NORM: x * nw / sqrt(mean(x^2) + eps) (RMS-norm of the row);
// GV_X_ACT: x holds (g, u) pairs (2 cols floats), the value is act(g) * u.
enum { GV_X_PLAIN = 0, GV_X_NORM = 1, GV_X_ACT = 2 };
struct GvParams {
    GvSeg seg[GV_MAX_SEG];
    const float* x;
    uint64_t timeout_ns;
    unsigned* status;
    int32_t nseg;
    int32_t nsb;             // 256-column units per row
    int32_t nslots;          // tile slots per CTA
    uint32_t slot_bytes;
    int32_t maxtiles;        // most tiles (row blocks) of one CTA
    int32_t x16;             // x is 16-byte aligned
    // what the kernel makes of x before the matvec (GV_X_*), and where CTA 0
    // stores the resulting x row (xout, cols floats; null: not stored)
    int32_t xpre;
    int32_t act;             // GV_X_ACT: the activation of the (g, u) pairs
    const float* nw;         // GV_X_NORM: the norm weight [cols]
    float eps;               // GV_X_NORM: epsilon
    float* xout;
    int32_t cta_rb[GV_MAX_CTA + 1];
};
cudaError_t gv_set_smem(int bytes);
cudaError_t gv_launch(int mask, const GvParams& P, int grid, size_t smem, cudaStream_t st);

// batch-1 tensor-core matvec over column chunks (lq_gv.cu, gvw_kernel): one
// plain Q4_K or Q6_K matrix whose rows are too wide for whole-row tiles, or
// Q6_K alone.  Work items are (column chunk c, row block rb) = 16 rows x ch
// super-blocks, numbered j = c * nrb + rb (column-major, so a CTA's items span
// few chunks and it stages x for those only); CTA k takes items
// [cta_j[k], cta_j[k+1]).  Each row is 16-byte aligned and a multiple of
// 16 bytes, so every row of an item comes in by one bulk copy.  With nch > 1
// a row block's chunks are summed across CTAs: each item's 16 sums go to
// part[j][16], the counter cnt[rb] counts the items done (wrapping to 0), and
// the CTA that completes the row block adds the chunks in order c = 0, 1, ...
constexpr int GVW_SLOTS = 4;                 // scratch sets (one per stream in use)
constexpr int GVW_MAX_PART = 1 << 18;        // floats of item sums per scratch set
constexpr int GVW_MAX_RB = 1 << 13;          // row-block counters per scratch set
constexpr int GVW_MAX_RB_PER_SM = 4;         // with nch > 1: fewer row blocks than this per SM
constexpr int GVW_MAX_X = 8;                 // x rows of one launch (Q6_K; one for Q4_K)
struct GvwParams {
    const uint8_t* w;
    float* y;
    const float* x;
    float* part;             // nch > 1: [nch * nrb][NM][16] item sums
    unsigned* cnt;           // nch > 1: [nrb] items done (every entry 0 between launches)
    uint64_t timeout_ns;
    unsigned* status;
    int64_t rowbytes;
    int32_t rows, nsb, ch, nch, nrb;
    int32_t pitch;           // shared row pitch of a tile: ch super-blocks
    uint32_t slot_bytes;
    int32_t nslots, maxtiles;
    int32_t winsb;           // super-blocks of the widest CTA's column window
    int32_t x16, xpre, act;  // xpre: GV_X_PLAIN or GV_X_ACT (one x row)
    int32_t nx;              // x rows (at most the instance's NM; several: x plain, no xout)
    int64_t ld_x, ld_y;      // floats between x rows, between y rows
    const float* nw;         // unused (the RMS-norm needs whole rows)
    float eps;
    float* xout;
    float cap;
    int32_t cta_j[GV_MAX_CTA + 1];
};
cudaError_t gvw_launch(int fmt, int nm, const GvwParams& P, int grid, size_t smem, cudaStream_t st);
size_t gvw_smem_bytes(int nm, int nslots, uint32_t slot_bytes, int maxtiles, int winsb, int ch);
cudaError_t gvw_scratch(unsigned** cnt, float** part);   // the GVW_SLOTS scratch sets of the current device

// quantized matvec kernel (lq_qmv_b{1,2,4,8}.cu); mask = block formats present
cudaError_t qmv1_set_smem(int bytes);
cudaError_t qmv2_set_smem(int bytes);
cudaError_t qmv4_set_smem(int bytes);
cudaError_t qmv8_set_smem(int bytes);
cudaError_t qmv1_occupancy(int mask, int nt, size_t smem, int* per_sm);
cudaError_t qmv2_occupancy(int mask, int nt, size_t smem, int* per_sm);
cudaError_t qmv4_occupancy(int mask, int nt, size_t smem, int* per_sm);
cudaError_t qmv8_occupancy(int mask, int nt, size_t smem, int* per_sm);
cudaError_t qmv1_launch(int mask, const QmvParams& P, int grid, int nt, size_t smem, cudaStream_t st);
cudaError_t qmv2_launch(int mask, const QmvParams& P, int grid, int nt, size_t smem, cudaStream_t st);
cudaError_t qmv4_launch(int mask, const QmvParams& P, int grid, int nt, size_t smem, cudaStream_t st);
cudaError_t qmv8_launch(int mask, const QmvParams& P, int grid, int nt, size_t smem, cudaStream_t st);


cudaError_t launch_dequant(int fmt, const uint8_t* W, int64_t rows, int64_t cols, float* out,
                           cudaStream_t st);
cudaError_t launch_interleave(const uint8_t* Wg, const uint8_t* Wu, int64_t rows, int64_t rb,
                              uint8_t* out, cudaStream_t st);
cudaError_t launch_direct(const Seg& S, int64_t cols, int maxb, cudaStream_t st);
cudaError_t launch_rmsnorm(const float* x, const float* w, float eps, float* out, int rows, int64_t n,
                           cudaStream_t st);
cudaError_t launch_act_pairs(const float* gu, float* h, int64_t n, int act, cudaStream_t st);
cudaError_t launch_moe_route(const float* R, int E, int64_t hidden, const float* X, int ntok,
                             int topk, const float* sgate_vec, const MoeWs& ws, cudaStream_t st);
cudaError_t launch_moe_combine(const float* ye, int64_t hidden, int ntok, int topk,
                               const MoeWs& ws, float* Y, cudaStream_t st);
// prefill GEMM (lq_gemm.cu): Y[n][r] = sum_j w_rj X[n][j], Q4_K or Q8_0 W
// with rows 16-byte aligned and cols a multiple of 256, on tcgen05: CTA
// tiles of GEMM_TC_WR weight rows x one or two x tiles of GEMM_TC_XN rows
// (nmt x tiles).  The x image, s_n, 1 / t_r and the split-K partial sums are
// workspace written by the launch itself.
constexpr int GEMM_TC_WR = 128;
constexpr int GEMM_TC_XN = 128;
struct GemmParams {
    const uint8_t* W;
    int64_t rows, cols, rowbytes, M, ld_y;
    float* sn;               // [nmt * GEMM_TC_XN] x row scales
    float* Y;
    int32_t nmt;
    CUtensorMap tmw;         // W as uint32 elements, boxes of one 256-column chunk x GEMM_TC_WR rows
    uint8_t* ximg;           // the x pieces in the MMA operand layout
    float* tinv;             // [rows] 1 / t_r
    float* part;             // split-K partial sums [ksplit][M][rows] (ksplit > 1)
    int32_t ksplit;          // K ranges per output tile
    int32_t pairs;           // rows 2i, 2i + 1 are gate / up: Y[n][i] = act(gate) * up
    int32_t act;             // with pairs: ACT_GEGLU_TANH or ACT_SWIGLU
    uint64_t timeout_ns;     // bound on every wait
    unsigned* status;
};
cudaError_t gemm_set_smem();
// K ranges per output tile for a weight matrix of this shape (a function of
// the weight shape alone, so a row's result does not depend on M)
int gemm_tc_ksplit(int64_t rows, int64_t cols);
size_t gemm_tc_smem_bytes(int fmt);
cudaError_t gemm_tc_launch(int fmt, const GemmParams& P, const float* X, cudaStream_t st);

// non-quantized GEMV (lq_dense.cu): fp16 (f16) or fp32 W [rows][cols], x
// [batch][cols] 16-byte aligned, y [batch][rows]; batch 1..8
cudaError_t dense_gemv_launch(bool f16, const void* W, int64_t rows, int cols, const float* x, float* y, int batch,
                              int sms, cudaStream_t st);
cudaError_t launch_timeout_probe(uint64_t timeout_ns, unsigned* status, cudaStream_t st);

}  // namespace lq
