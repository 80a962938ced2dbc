// bf16 instantiation of the SpMM / SDDMM / transpose launchers.
#include "spmm.cuh"

namespace snack {

template <>
cudaError_t run_spmm<bf16>(const SpmmParams &p, const BatchGeom &bg, bool gather_val, bool fuse_dw,
                          cudaStream_t s) {
  if (!gather_val) return launch_spmm<bf16, bf16, false, false>(p, bg, s);
  return fuse_dw ? launch_spmm<bf16, bf16, true, true>(p, bg, s) : launch_spmm<bf16, bf16, true, false>(p, bg, s);
}

template <>
cudaError_t run_sddmm<bf16>(int64_t nnz, const int32_t *row, const int32_t *col, int32_t out_f, int32_t in_f,
                          const bf16 *xt, const bf16 *dyt, const BatchGeom &bg, float *dw, int num_sms,
                          cudaStream_t s) {
  return launch_sddmm<bf16>(nnz, row, col, out_f, in_f, xt, dyt, bg, dw, num_sms, s);
}

template <>
cudaError_t run_ell<bf16>(const SpmmParams &p, const BatchGeom &bg, int32_t K, cudaStream_t s) {
  return launch_ell<bf16, bf16>(p, bg, K, s);
}

template <>
cudaError_t run_transpose<bf16>(const bf16 *a, int batch, int n, bf16 *at, int ldx, cudaStream_t s) {
  return launch_transpose<bf16>(a, batch, n, at, ldx, s);
}

template <>
cudaError_t run_colsum<bf16>(const bf16 *a, int batch, int n, float *out, cudaStream_t s) {
  return launch_colsum<bf16>(a, batch, n, out, s);
}

template <>
cudaError_t run_rowsum_t<bf16>(const bf16 *at, int ldx, int batch, int n, float *out, cudaStream_t s) {
  return launch_rowsum_t<bf16>(at, ldx, batch, n, out, s);
}

template <>
cudaError_t run_transpose2<bf16>(const TransposePair<bf16> &tp, int batch, int ldx, cudaStream_t s) {
  return launch_transpose2<bf16>(tp, batch, ldx, s);
}

}  // namespace snack
