// f32 instantiation of the SpMM / SDDMM / transpose launchers.
#include "spmm.cuh"

namespace snack {

template <>
cudaError_t run_spmm<float>(const SpmmParams &p, const BatchGeom &bg, bool gather_val, bool fuse_dw,
                          cudaStream_t s) {
  if (!gather_val) return launch_spmm<float, float, false, false>(p, bg, s);
  return fuse_dw ? launch_spmm<float, float, true, true>(p, bg, s) : launch_spmm<float, float, true, false>(p, bg, s);
}

template <>
cudaError_t run_sddmm<float>(int64_t nnz, const int32_t *row, const int32_t *col, int32_t out_f, int32_t in_f,
                          const float *xt, const float *dyt, const BatchGeom &bg, float *dw, int num_sms,
                          cudaStream_t s) {
  return launch_sddmm<float>(nnz, row, col, out_f, in_f, xt, dyt, bg, dw, num_sms, s);
}

template <>
cudaError_t run_ell<float>(const SpmmParams &p, const BatchGeom &bg, int32_t K, cudaStream_t s) {
  return launch_ell<float, float>(p, bg, K, s);
}

template <>
cudaError_t run_transpose<float>(const float *a, int batch, int n, float *at, int ldx, cudaStream_t s) {
  return launch_transpose<float>(a, batch, n, at, ldx, s);
}

template <>
cudaError_t run_colsum<float>(const float *a, int batch, int n, float *out, cudaStream_t s) {
  return launch_colsum<float>(a, batch, n, out, s);
}

template <>
cudaError_t run_rowsum_t<float>(const float *at, int ldx, int batch, int n, float *out, cudaStream_t s) {
  return launch_rowsum_t<float>(at, ldx, batch, n, out, s);
}

template <>
cudaError_t run_transpose2<float>(const TransposePair<float> &tp, int batch, int ldx, cudaStream_t s) {
  return launch_transpose2<float>(tp, batch, ldx, s);
}

}  // namespace snack
