// lq_dense.cu -- the non-quantized lm_head fallbacks: y = W.x for an fp16 or
// fp32 weight matrix (larql "Architecture -> Metal shader map", Gemma 3
// table, lm_head row: the f16_gemv / f32_gemv fallback chain for a tied
// embedding that is not block-quantized).  They are the comparison rows for
// the block-quantized lm_head: the same shape, two and four bytes per weight
// instead of 0.5625.
//
// HBM-bound: every weight byte is read once with 16-byte loads, coalesced
// per warp (lane l reads chunks l, l + 32, ... of a row); a warp takes RW
// rows at a time (RW independent loads in flight per lane), the x rows sit
// in shared memory, and each row's dot products are summed in a fixed order
// (per lane in column order, then a butterfly over the warp) in fp32.
#include <algorithm>

#include <cuda_fp16.h>

#include "lq_internal.h"

namespace lq {
namespace {

constexpr int DG_THREADS = 256;
constexpr int DG_RW = 4;           // rows per warp per pass

// 16 bytes of a row as weights: eight fp16 values or four fp32 values
template <bool F16>
__device__ __forceinline__ void unpack16(const uint4& v, float (&w)[F16 ? 8 : 4]) {
    if constexpr (F16) {
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
            w[2 * i] = f.x;
            w[2 * i + 1] = f.y;
        }
    } else {
        w[0] = __uint_as_float(v.x);
        w[1] = __uint_as_float(v.y);
        w[2] = __uint_as_float(v.z);
        w[3] = __uint_as_float(v.w);
    }
}

template <bool F16, int B>
__global__ void __launch_bounds__(DG_THREADS) dense_gemv_kernel(const uint8_t* __restrict__ W, int64_t rows,
                                                                int cols, const float* __restrict__ x,
                                                                float* __restrict__ y) {
    extern __shared__ __align__(16) float xs[];          // [B][cols]
    for (int i = threadIdx.x; i < B * cols / 4; i += DG_THREADS)
        reinterpret_cast<float4*>(xs)[i] = __ldg(reinterpret_cast<const float4*>(x) + i);
    __syncthreads();
    constexpr int EPC = F16 ? 8 : 4;                     // weights per 16-byte chunk
    const int64_t rowbytes = (int64_t)cols * (F16 ? 2 : 4);
    const int nchunk = cols / EPC;
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * (DG_THREADS / 32) + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)gridDim.x * (DG_THREADS / 32);
    for (int64_t r0 = gw * DG_RW; r0 < rows; r0 += nw * DG_RW) {
        float acc[DG_RW][B];
#pragma unroll
        for (int i = 0; i < DG_RW; ++i)
#pragma unroll
            for (int b = 0; b < B; ++b) acc[i][b] = 0.f;
        for (int c = lane; c < nchunk; c += 32) {
            uint4 v[DG_RW];
#pragma unroll
            for (int i = 0; i < DG_RW; ++i)
                v[i] = r0 + i < rows ? __ldcs(reinterpret_cast<const uint4*>(W + (r0 + i) * rowbytes) + c)
                                     : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int i = 0; i < DG_RW; ++i) {
                float w[EPC];
                unpack16<F16>(v[i], w);
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    const float* xb = xs + b * cols + c * EPC;
#pragma unroll
                    for (int e = 0; e < EPC; ++e) acc[i][b] = fmaf(w[e], xb[e], acc[i][b]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < DG_RW; ++i)
#pragma unroll
            for (int b = 0; b < B; ++b) {
                float s = acc[i][b];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
                if (lane == 0 && r0 + i < rows) y[(int64_t)b * rows + r0 + i] = s;
            }
    }
}

template <bool F16, int B>
cudaError_t dense_launch_b(const uint8_t* W, int64_t rows, int cols, const float* x, float* y, int sms,
                           cudaStream_t st) {
    const size_t smem = (size_t)B * cols * sizeof(float);
    auto k = dense_gemv_kernel<F16, B>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, DG_THREADS, smem);
    if (e != cudaSuccess) return e;
    const int64_t warps_needed = (rows + DG_RW - 1) / DG_RW;
    const int64_t blocks_needed = (warps_needed + DG_THREADS / 32 - 1) / (DG_THREADS / 32);
    const int grid = (int)std::min<int64_t>((int64_t)sms * std::max(1, per_sm), blocks_needed);
    k<<<grid, DG_THREADS, smem, st>>>(W, rows, cols, x, y);
    return cudaGetLastError();
}

}  // namespace

cudaError_t dense_gemv_launch(bool f16, const void* W, int64_t rows, int cols, const float* x, float* y, int batch,
                              int sms, cudaStream_t st) {
    const uint8_t* w = static_cast<const uint8_t*>(W);
    switch (batch) {
#define LQ_DG_CASE(b)                                                                       \
    case b:                                                                                 \
        return f16 ? dense_launch_b<true, b>(w, rows, cols, x, y, sms, st)                  \
                   : dense_launch_b<false, b>(w, rows, cols, x, y, sms, st);
        LQ_DG_CASE(1)
        LQ_DG_CASE(2)
        LQ_DG_CASE(3)
        LQ_DG_CASE(4)
        LQ_DG_CASE(5)
        LQ_DG_CASE(6)
        LQ_DG_CASE(7)
        LQ_DG_CASE(8)
#undef LQ_DG_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lq
