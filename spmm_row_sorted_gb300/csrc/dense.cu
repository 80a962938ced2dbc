// Dense path for moderately sparse bf16 layers (half or more of the weights
// stored, batch >= 32): there the product is a dense contraction, so the
// stored weights are scattered into a dense bf16 copy of W and the
// contraction runs on the tensor cores through a cuBLASLt GEMM (a plain
// library GEMM; every other step is a kernel of this file).  The weight
// gradient is the dense dY^T X, read back at the stored positions only.
//
//   forward      W_dense = scatter(row, col, val);  Y = X W_dense^T (+ bias)
//   input grad   W_dense as above;                  dX = dY W_dense
//   weight grad  G = dY^T X (fp32);                 dW[k] = G[row_k, col_k]
//
// Results equal the definitions up to the order of the fp32 sums, the same
// contract as the gather kernels.  The kernels here are launched plainly
// (not as dependent launches): they sit next to cuBLASLt's GEMM.
#include <cublasLt.h>

#include "internal.hpp"

namespace snack {

namespace {

constexpr int kDensifyChunk = 8192;  // columns of one row staged in shared memory at a time

// Row r of the dense copy: zeros, then the row's stored weights at their
// columns, written as whole 16-byte vectors.
template <typename I>
__global__ void __launch_bounds__(256) k_densify(const int32_t *__restrict__ rp, const I *__restrict__ col,
                                                 const bf16 *__restrict__ val, int32_t in_f, bf16 *__restrict__ wd) {
  pdl_wait();
  __shared__ __align__(16) bf16 row_buf[kDensifyChunk];
  const int r = blockIdx.x;
  const int64_t k0 = rp[r], k1 = rp[r + 1];
  bf16 *dst = wd + (size_t)r * in_f;
  for (int c0 = 0; c0 < in_f; c0 += kDensifyChunk) {
    const int n = in_f - c0 < kDensifyChunk ? in_f - c0 : kDensifyChunk;
    for (int i = threadIdx.x; i < n; i += blockDim.x) row_buf[i] = __float2bfloat16(0.f);
    __syncthreads();
    for (int64_t kb = k0 + threadIdx.x; kb < k1; kb += 8 * (int64_t)blockDim.x) {
      int c[8];
      bf16 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {  // all loads in flight before the stores
        const int64_t k = kb + u * (int64_t)blockDim.x;
        c[u] = k < k1 ? (int)col[k] - c0 : -1;
        v[u] = k < k1 ? val[k] : __float2bfloat16(0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (c[u] >= 0 && c[u] < n) row_buf[c[u]] = v[u];
    }
    __syncthreads();
    if ((in_f & 7) == 0) {  // rows start on 16 bytes: vector stores
      const uint4 *src4 = reinterpret_cast<const uint4 *>(row_buf);
      uint4 *dst4 = reinterpret_cast<uint4 *>(dst + c0);
      for (int i = threadIdx.x; i < n / 8; i += blockDim.x) dst4[i] = src4[i];
    } else {
      for (int i = threadIdx.x; i < n; i += blockDim.x) dst[c0 + i] = row_buf[i];
    }
    __syncthreads();
  }
}

// dW[k] = G[row_k][col_k], one block per row of G.
__global__ void __launch_bounds__(256) k_gather_dw(const int32_t *__restrict__ rp, const int32_t *__restrict__ col,
                                                   const float *__restrict__ g, int32_t in_f, float *__restrict__ dw) {
  pdl_wait();
  const int r = blockIdx.x;
  const float *gr = g + (size_t)r * in_f;
  const int64_t k1 = rp[r + 1];
  for (int64_t kb = rp[r] + threadIdx.x; kb < k1; kb += 8 * (int64_t)blockDim.x) {
    int c[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t k = kb + u * (int64_t)blockDim.x;
      c[u] = k < k1 ? col[k] : 0;
    }
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldcs(gr + c[u]);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t k = kb + u * (int64_t)blockDim.x;
      if (k < k1) dw[k] = v[u];
    }
  }
}

// y[b][r] = bf16(acc[b][r] + bias[r]): the fp32 product and the bias are
// added before the one rounding to bf16
__global__ void k_bias_round(const float *__restrict__ acc, const float *__restrict__ bias, int batch, int n,
                             bf16 *__restrict__ y) {
  pdl_wait();
  const int64_t total = (int64_t)batch * n;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x)
    y[i] = __float2bfloat16_rn(bias[i % n] + acc[i]);
}

// db[r] = sum_b dy[b][r], b increasing
__global__ void k_colsum_bf16(const bf16 *__restrict__ a, int batch, int n, float *__restrict__ out) {
  pdl_wait();
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= n) return;
  float s = 0.f;
  for (int b = 0; b < batch; ++b) s += __bfloat162float(a[(size_t)b * n + c]);
  out[c] = s;
}

constexpr size_t kLtWorkspace = 32u << 20;

struct DenseWs {
  size_t wd, g, lt, total;
};

// wd: the dense bf16 W; g: the dense fp32 weight gradient, or the forward's
// fp32 sums [batch][out_f] before the bias (so at least max_batch columns)
DenseWs dense_ws(int32_t out_f, int32_t in_f, int32_t max_batch) {
  DenseWs w;
  size_t o = 0;
  w.wd = o;
  o += align_up((size_t)out_f * in_f * sizeof(bf16), kAlign);
  w.g = o;
  o += align_up((size_t)out_f * (in_f > max_batch ? in_f : max_batch) * sizeof(float), kAlign);
  w.lt = o;
  o += kLtWorkspace;
  w.total = o;
  return w;
}

// One GEMM D = op(A) op(B) in column-major terms (m x n, inner k), A/B bf16,
// D bf16 or fp32, fp32 accumulation.
cudaError_t lt_gemm(cublasLtHandle_t lt, cublasOperation_t ta, cublasOperation_t tb, int m, int n, int k,
                    const void *a, int lda, const void *b, int ldb, void *d, int ldd, cudaDataType_t dtype,
                    void *ws, cudaStream_t s) {
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, ld = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  cudaError_t result = cudaErrorUnknown;
  const float alpha = 1.f, beta = 0.f;
  size_t wsb = kLtWorkspace;
  cublasLtMatmulHeuristicResult_t heur;
  int found = 0;
  do {
    if (cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS) break;
    if (cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof(ta)) != CUBLAS_STATUS_SUCCESS) break;
    if (cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof(tb)) != CUBLAS_STATUS_SUCCESS) break;
    const int ar = ta == CUBLAS_OP_N ? m : k, ac = ta == CUBLAS_OP_N ? k : m;
    const int br = tb == CUBLAS_OP_N ? k : n, bc = tb == CUBLAS_OP_N ? n : k;
    if (cublasLtMatrixLayoutCreate(&la, CUDA_R_16BF, ar, ac, lda) != CUBLAS_STATUS_SUCCESS) break;
    if (cublasLtMatrixLayoutCreate(&lb, CUDA_R_16BF, br, bc, ldb) != CUBLAS_STATUS_SUCCESS) break;
    if (cublasLtMatrixLayoutCreate(&ld, dtype, m, n, ldd) != CUBLAS_STATUS_SUCCESS) break;
    if (cublasLtMatmulPreferenceCreate(&pref) != CUBLAS_STATUS_SUCCESS) break;
    if (cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &wsb, sizeof(wsb)) !=
        CUBLAS_STATUS_SUCCESS)
      break;
    if (cublasLtMatmulAlgoGetHeuristic(lt, op, la, lb, ld, ld, pref, 1, &heur, &found) != CUBLAS_STATUS_SUCCESS ||
        found < 1)
      break;
    if (cublasLtMatmul(lt, op, &alpha, a, la, b, lb, &beta, d, ld, d, ld, &heur.algo, ws, wsb, s) !=
        CUBLAS_STATUS_SUCCESS)
      break;
    result = cudaSuccess;
  } while (0);
  if (pref) cublasLtMatmulPreferenceDestroy(pref);
  if (ld) cublasLtMatrixLayoutDestroy(ld);
  if (lb) cublasLtMatrixLayoutDestroy(lb);
  if (la) cublasLtMatrixLayoutDestroy(la);
  if (op) cublasLtMatmulDescDestroy(op);
  return result;
}

unsigned grid_of(int64_t n, int threads) {
  int64_t b = (n + threads - 1) / threads;
  if (b < 1) b = 1;
  if (b > 65535 * 8) b = 65535 * 8;
  return (unsigned)b;
}

// the dense copy of W; columns from the plan's 16-bit copy when there is one
void densify(const snack_layer *h, const int32_t *col, const void *val, bf16 *wd, cudaStream_t s) {
  const bf16 *v = reinterpret_cast<const bf16 *>(val);
  if (h->p.col16)
    k_densify<uint16_t><<<h->out_f, 256, 0, s>>>(h->p.rp, h->p.col16, v, h->in_f, wd);
  else
    k_densify<int32_t><<<h->out_f, 256, 0, s>>>(h->p.rp, col, v, h->in_f, wd);
}

}  // namespace

bool dense_layer(int32_t out_f, int32_t in_f, int64_t nnz, int32_t max_batch, snack_dtype val_t) {
  return val_t == SNACK_BF16 && max_batch >= kDenseMinBatch && (double)nnz >= 0.25 * (double)out_f * (double)in_f &&
         (int64_t)out_f * in_f <= ((int64_t)1 << 31);
}

size_t dense_ws_bytes(int32_t out_f, int32_t in_f, int32_t max_batch) { return dense_ws(out_f, in_f, max_batch).total; }

bool dense_init(snack_layer *h) {
  cublasLtHandle_t lt = nullptr;
  if (cublasLtCreate(&lt) != CUBLAS_STATUS_SUCCESS) return false;
  h->lt = lt;
  return true;
}

void dense_release(snack_layer *h) {
  if (h->lt) cublasLtDestroy(reinterpret_cast<cublasLtHandle_t>(h->lt));
  h->lt = nullptr;
}

snack_status dense_fwd(snack_layer *h, const int32_t *col, const void *val, const void *x, int32_t batch,
                       const float *bias, void *y, void *ws, size_t ws_bytes, cudaStream_t s) {
  const DenseWs W = dense_ws(h->out_f, h->in_f, h->max_batch);
  if (ws_bytes < W.total) return SNACK_ERR_WORKSPACE;
  uint8_t *b = reinterpret_cast<uint8_t *>(ws);
  bf16 *wd = reinterpret_cast<bf16 *>(b + W.wd);
  densify(h, col, val, wd, s);
  if (cudaGetLastError() != cudaSuccess) return SNACK_ERR_CUDA;
  // column-major: Y'(out x B) = Wd'(in x out)^T X'(in x B).  Without a bias
  // the GEMM rounds its fp32 sums to bf16 once; with one, it writes the fp32
  // sums (into the fp32 gradient buffer, unused by the forward) and the bias
  // is added before the single rounding.
  float *acc = reinterpret_cast<float *>(b + W.g);
  if (lt_gemm(reinterpret_cast<cublasLtHandle_t>(h->lt), CUBLAS_OP_T, CUBLAS_OP_N, h->out_f, batch, h->in_f, wd,
              h->in_f, x, h->in_f, bias ? (void *)acc : y, h->out_f, bias ? CUDA_R_32F : CUDA_R_16BF, b + W.lt,
              s) != cudaSuccess)
    return SNACK_ERR_CUDA;
  if (bias) {
    k_bias_round<<<grid_of((int64_t)batch * h->out_f, 256), 256, 0, s>>>(acc, bias, batch, h->out_f,
                                                                         reinterpret_cast<bf16 *>(y));
    if (cudaGetLastError() != cudaSuccess) return SNACK_ERR_CUDA;
  }
  return SNACK_OK;
}

snack_status dense_dx(snack_layer *h, const int32_t *col, const void *val, const void *dy, int32_t batch, void *dx,
                      void *ws, size_t ws_bytes, cudaStream_t s) {
  const DenseWs W = dense_ws(h->out_f, h->in_f, h->max_batch);
  if (ws_bytes < W.total) return SNACK_ERR_WORKSPACE;
  uint8_t *b = reinterpret_cast<uint8_t *>(ws);
  bf16 *wd = reinterpret_cast<bf16 *>(b + W.wd);
  densify(h, col, val, wd, s);
  if (cudaGetLastError() != cudaSuccess) return SNACK_ERR_CUDA;
  // column-major: dX'(in x B) = Wd'(in x out) dY'(out x B)
  if (lt_gemm(reinterpret_cast<cublasLtHandle_t>(h->lt), CUBLAS_OP_N, CUBLAS_OP_N, h->in_f, batch, h->out_f, wd,
              h->in_f, dy, h->out_f, dx, h->in_f, CUDA_R_16BF, b + W.lt, s) != cudaSuccess)
    return SNACK_ERR_CUDA;
  return SNACK_OK;
}

snack_status dense_dw(snack_layer *h, const int32_t *col, const void *x, const void *dy, int32_t batch, float *dw,
                      float *db, void *ws, size_t ws_bytes, cudaStream_t s) {
  const DenseWs W = dense_ws(h->out_f, h->in_f, h->max_batch);
  if (ws_bytes < W.total) return SNACK_ERR_WORKSPACE;
  uint8_t *b = reinterpret_cast<uint8_t *>(ws);
  float *g = reinterpret_cast<float *>(b + W.g);
  if (db) {
    k_colsum_bf16<<<(h->out_f + 255) / 256, 256, 0, s>>>(reinterpret_cast<const bf16 *>(dy), batch, h->out_f, db);
    if (cudaGetLastError() != cudaSuccess) return SNACK_ERR_CUDA;
  }
  if (h->nnz == 0) return SNACK_OK;
  // column-major: G'(in x out) = X'(in x B) dY'(out x B)^T, i.e. row-major G[out][in] = dY^T X
  if (lt_gemm(reinterpret_cast<cublasLtHandle_t>(h->lt), CUBLAS_OP_N, CUBLAS_OP_T, h->in_f, h->out_f, batch, x,
              h->in_f, dy, h->out_f, g, h->in_f, CUDA_R_32F, b + W.lt, s) != cudaSuccess)
    return SNACK_ERR_CUDA;
  k_gather_dw<<<h->out_f, 256, 0, s>>>(h->p.rp, col, g, h->in_f, dw);
  if (cudaGetLastError() != cudaSuccess) return SNACK_ERR_CUDA;
  return SNACK_OK;
}

}  // namespace snack
