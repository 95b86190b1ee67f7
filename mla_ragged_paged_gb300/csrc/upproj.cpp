// Up-projection of gathered latent rows to per-head K_nope or V:
//   out[t, n] = sum_k latent[t, k] * weight[n, k]
// (weight in nn.Linear layout [H * 128, kv_lora_rank]).  A plain dense GEMM,
// so it goes to cuBLASLt: bf16 operands, fp32 accumulation, bf16 output.
#include <cublasLt.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "host_common.h"

namespace mla {
namespace {

std::mutex g_lt_mutex;
cublasLtHandle_t g_lt[64] = {};

const char* lt_error(cublasStatus_t s) {
  switch (s) {
    case CUBLAS_STATUS_NOT_INITIALIZED: return "not initialized";
    case CUBLAS_STATUS_ALLOC_FAILED: return "allocation failed";
    case CUBLAS_STATUS_INVALID_VALUE: return "invalid value";
    case CUBLAS_STATUS_ARCH_MISMATCH: return "architecture mismatch";
    case CUBLAS_STATUS_EXECUTION_FAILED: return "execution failed";
    case CUBLAS_STATUS_NOT_SUPPORTED: return "not supported";
    default: return "error";
  }
}

struct LtObjects {
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t a = nullptr, b = nullptr, c = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  ~LtObjects() {
    if (pref) cublasLtMatmulPreferenceDestroy(pref);
    if (c) cublasLtMatrixLayoutDestroy(c);
    if (b) cublasLtMatrixLayoutDestroy(b);
    if (a) cublasLtMatrixLayoutDestroy(a);
    if (op) cublasLtMatmulDescDestroy(op);
  }
};

}  // namespace
}  // namespace mla

extern "C" mla_status_t mla_up_project(const mla_tensor_t* out, const mla_tensor_t* latent,
                                       const mla_tensor_t* weight, void* workspace,
                                       size_t workspace_bytes, mla_stream_t stream) {
  using namespace mla;
  mla_status_t st;
  if ((st = check_tensor(out, "out", 2, MLA_DTYPE_BF16)) != MLA_OK) return st;
  if ((st = check_tensor(latent, "latent", 2, MLA_DTYPE_BF16)) != MLA_OK) return st;
  if ((st = check_tensor(weight, "weight", 2, MLA_DTYPE_BF16)) != MLA_OK) return st;
  const int64_t M = latent->shape[0], K = latent->shape[1], N = weight->shape[0];
  if (weight->shape[1] != K) return fail(MLA_ERR_INVALID_ARG, "weight must be [N, K] with latent's K");
  if (out->shape[0] != M || out->shape[1] != N) return fail(MLA_ERR_INVALID_ARG, "out must be [rows, N]");
  if (K < 1 || N < 1) return fail(MLA_ERR_INVALID_ARG, "empty projection");
  const mla_tensor_t* ts[3] = {out, latent, weight};
  for (const mla_tensor_t* t : ts) {
    if (!aligned16(t->data) || (t->stride[0] * 2) % 16 != 0)
      return fail(MLA_ERR_INVALID_ARG, "GEMM operands need 16-byte aligned rows");
  }
  if (workspace_bytes && !workspace) return fail(MLA_ERR_INVALID_ARG, "workspace is NULL");
  int dev = 0, sms = 0;
  if ((st = check_device(&dev, &sms)) != MLA_OK) return st;
  if (M == 0) return MLA_OK;
  if (dev >= 64) return fail(MLA_ERR_UNSUPPORTED, "device index %d", dev);
  cublasLtHandle_t lt;
  {
    std::lock_guard<std::mutex> lock(g_lt_mutex);
    if (!g_lt[dev]) {
      cublasStatus_t s = cublasLtCreate(&g_lt[dev]);
      if (s != CUBLAS_STATUS_SUCCESS) return fail(MLA_ERR_CUDA, "cublasLtCreate: %s", lt_error(s));
    }
    lt = g_lt[dev];
  }
  // Column-major view: out^T [N, M] = weight [K, N]^T (op T) x latent^T [K, M].
  LtObjects o;
  cublasStatus_t s = cublasLtMatmulDescCreate(&o.op, CUBLAS_COMPUTE_32F, CUDA_R_32F);
  const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
  if (s == CUBLAS_STATUS_SUCCESS)
    s = cublasLtMatmulDescSetAttribute(o.op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof(ta));
  if (s == CUBLAS_STATUS_SUCCESS)
    s = cublasLtMatmulDescSetAttribute(o.op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof(tb));
  if (s == CUBLAS_STATUS_SUCCESS)
    s = cublasLtMatrixLayoutCreate(&o.a, CUDA_R_16BF, K, N, weight->stride[0]);
  if (s == CUBLAS_STATUS_SUCCESS)
    s = cublasLtMatrixLayoutCreate(&o.b, CUDA_R_16BF, K, M, latent->stride[0]);
  if (s == CUBLAS_STATUS_SUCCESS)
    s = cublasLtMatrixLayoutCreate(&o.c, CUDA_R_16BF, N, M, out->stride[0]);
  if (s == CUBLAS_STATUS_SUCCESS) s = cublasLtMatmulPreferenceCreate(&o.pref);
  if (s == CUBLAS_STATUS_SUCCESS)
    s = cublasLtMatmulPreferenceSetAttribute(o.pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES,
                                             &workspace_bytes, sizeof(workspace_bytes));
  if (s != CUBLAS_STATUS_SUCCESS) return fail(MLA_ERR_CUDA, "cuBLASLt set-up: %s", lt_error(s));
  cublasLtMatmulHeuristicResult_t heur = {};
  int found = 0;
  s = cublasLtMatmulAlgoGetHeuristic(lt, o.op, o.a, o.b, o.c, o.c, o.pref, 1, &heur, &found);
  if (s != CUBLAS_STATUS_SUCCESS || found == 0)
    return fail(MLA_ERR_UNSUPPORTED, "cuBLASLt has no algorithm for this GEMM: %s", lt_error(s));
  const float alpha = 1.f, beta = 0.f;
  s = cublasLtMatmul(lt, o.op, &alpha, weight->data, o.a, latent->data, o.b, &beta, out->data, o.c,
                     out->data, o.c, &heur.algo, workspace, workspace_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
  if (s != CUBLAS_STATUS_SUCCESS) return fail(MLA_ERR_CUDA, "cublasLtMatmul: %s", lt_error(s));
  return MLA_OK;
}
