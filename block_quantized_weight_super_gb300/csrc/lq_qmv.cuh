// lq_qmv.cuh -- parameters of the quantized matvec kernel (lq_qmv.cu),
// shared with the host launcher.
#pragma once
#include <cstdint>

#include "lq_stream.cuh"

namespace lq {

constexpr int XS_STRIDE = 68;   // floats per 64-value x group slot in shared memory

// Shape of the matrices of one launch.
struct QGeo {
    int32_t cols;
    int32_t U;               // groups of 64 weights per row
    int32_t UP;              // row stride of the per-group partials (qmv_red_stride)
    int32_t RT;              // matrix rows per tile
    int32_t ipt;             // work items per thread per tile
};

struct QmvParams {
    Seg seg[MAX_SEG];
    int32_t nseg;
    int32_t ntiles;          // total tiles (format group 0 first)
    QGeo geo;
    int32_t R;               // rows per work item (interleaved in a thread)
    int32_t nstages;
    int32_t stage_bytes;
    int32_t fmt0, fmt1;      // formats of CTA groups 0 and 1
    int32_t cta_split;       // CTAs [0, cta_split) run format group 0
    int32_t tile_split;      // tiles [0, tile_split) belong to format group 0
    int32_t dev_counts;      // some segment reads its row count / offset from device memory
    uint64_t timeout_ns;
    unsigned* status;
};

// Rows of W per work item for batch width B and block-format mask (bit 0
// Q4_K, bit 1 Q6_K, bit 2 Q8_0): as many as the registers allow.  Batch 1
// Q4_K / Q8_0 items take four rows (x reads shared by more rows); Q6_K items,
// which need more registers per row, two.
__host__ __device__ constexpr int qmv_rows_per_item(int B, int mask) {
    return B == 1 ? ((mask & 2) ? 2 : 4) : 1;
}

// Consumer warps at most: four-row items use 128 registers per thread, so
// their CTAs are limited to 256 threads (two CTAs per SM).
__host__ __device__ constexpr int qmv_max_consumer_warps(int R) { return R == 4 ? 7 : 8; }

// Row stride of the per-group partials: at least U and 8 mod 32, so the
// reduction's four concurrent rows fall in distinct banks.
__host__ __device__ constexpr int qmv_red_stride(int U) { return U + (((8 - U) % 32) + 32) % 32; }

__host__ __device__ inline size_t qmv_smem_bytes(int B, int U, int RT, int nstages, int stage_bytes) {
    size_t off = (size_t)nstages * stage_bytes;
    off += (size_t)B * U * XS_STRIDE * sizeof(float);
    off += (size_t)B * U * 2 * sizeof(float);
    off += (size_t)(nstages + 1) * RT * B * qmv_red_stride(U) * sizeof(float);
    off = (off + 7) & ~size_t(7);
    off += (size_t)2 * nstages * sizeof(uint64_t) + (size_t)(nstages + 2) * sizeof(int);
    off = (off + 15) & ~size_t(15);
    off += (size_t)MAX_SEG * sizeof(Seg);          // shared copy of the segment table
    return off;
}

}  // namespace lq
