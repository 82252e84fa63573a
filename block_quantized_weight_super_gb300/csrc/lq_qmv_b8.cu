// lq_qmv_b8.cu -- instantiations of the quantized matvec kernel for 8 x rows
// (one CTA per SM: its accumulators need more than the two-CTA register share).
#include "lq_qmv_impl.cuh"

namespace lq {

cudaError_t qmv8_set_smem(int bytes) { return QmvTable<8>::set_smem(bytes); }
cudaError_t qmv8_occupancy(int mask, int nt, size_t smem, int* per_sm) {
    return QmvTable<8>::occupancy(mask, nt, smem, per_sm);
}
cudaError_t qmv8_launch(int mask, const QmvParams& P, int grid, int nt, size_t smem, cudaStream_t st) {
    return QmvTable<8>::launch(mask, P, grid, nt, smem, st);
}

}  // namespace lq
