// lq_qmv_b1.cu -- instantiations of the quantized matvec kernel for 1 x row(s).
#include "lq_qmv_impl.cuh"

namespace lq {

cudaError_t qmv1_set_smem(int bytes) { return QmvTable<1>::set_smem(bytes); }
cudaError_t qmv1_occupancy(int mask, int nt, size_t smem, int* per_sm) {
    return QmvTable<1>::occupancy(mask, nt, smem, per_sm);
}
cudaError_t qmv1_launch(int mask, const QmvParams& P, int grid, int nt, size_t smem, cudaStream_t st) {
    return QmvTable<1>::launch(mask, P, grid, nt, smem, st);
}

}  // namespace lq
