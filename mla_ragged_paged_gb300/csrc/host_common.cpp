#include "host_common.h"

#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <mutex>

namespace mla {
namespace {

thread_local char g_error[512] = "no error";

constexpr int kMaxDevices = 64;
std::atomic<int> g_num_sms[kMaxDevices];  // 0 = unknown, -1 = unsupported device
std::atomic<int> g_smem_set[kMaxDevices][8];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

}  // namespace

mla_status_t fail(mla_status_t status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_error, sizeof(g_error), fmt, ap);
  va_end(ap);
  return status;
}

mla_status_t ok() { return MLA_OK; }

mla_status_t check_device(int* device_out, int* num_sms_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(MLA_ERR_UNSUPPORTED, "device index %d", dev);
  int sms = g_num_sms[dev].load(std::memory_order_relaxed);
  if (sms == 0) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return fail(MLA_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    if (major != 10 || minor != 3) sms = -1;
    g_num_sms[dev].store(sms, std::memory_order_relaxed);
  }
  if (sms < 0) return fail(MLA_ERR_UNSUPPORTED, "device %d is not compute capability 10.3", dev);
  *device_out = dev;
  *num_sms_out = sms;
  return MLA_OK;
}

mla_status_t encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, void* base,
                          const uint64_t* dims, const uint64_t* strides_bytes,
                          const uint32_t* box, CUtensorMapSwizzle swizzle, const char* what) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], es[5];
  for (uint32_t i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  CUresult r = g_encode(map, dtype, rank, base, d, s, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MLA_ERR_CUDA, "tensor map for %s rejected (CUresult %d)", what, (int)r);
  return MLA_OK;
}

mla_status_t set_max_dynamic_smem(const void* func, int bytes, int device, int slot) {
  std::atomic<int>& cached = g_smem_set[device][slot];
  if (cached.load(std::memory_order_relaxed) >= bytes) return MLA_OK;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess)
    return fail(MLA_ERR_CUDA, "cudaFuncSetAttribute(%d bytes): %s", bytes, cudaGetErrorString(e));
  cached.store(bytes, std::memory_order_relaxed);
  return MLA_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

mla_status_t check_tensor(const mla_tensor_t* t, const char* name, int ndim, mla_dtype_t dtype) {
  if (!t) return fail(MLA_ERR_INVALID_ARG, "%s descriptor is NULL", name);
  if (!t->data) return fail(MLA_ERR_INVALID_ARG, "%s data is NULL", name);
  if (t->ndim != ndim) return fail(MLA_ERR_INVALID_ARG, "%s has ndim %d, expected %d", name, t->ndim, ndim);
  if (t->dtype != dtype)
    return fail(MLA_ERR_INVALID_ARG, "%s has dtype %d, expected %d", name, (int)t->dtype, (int)dtype);
  for (int i = 0; i < ndim; ++i) {
    if (t->shape[i] < 0 || t->shape[i] > 0x7FFFFFFFll)
      return fail(MLA_ERR_INVALID_ARG, "%s shape[%d] = %lld out of range", name, i, (long long)t->shape[i]);
    if (t->stride[i] < 0) return fail(MLA_ERR_INVALID_ARG, "%s stride[%d] is negative", name, i);
  }
  if (t->stride[ndim - 1] != 1) return fail(MLA_ERR_INVALID_ARG, "%s innermost stride must be 1", name);
  return MLA_OK;
}

}  // namespace mla

extern "C" const char* mla_last_error_string(void) { return mla::g_error; }

extern "C" uint32_t mla_prefill_plan_max_rows(uint64_t total_k_upper_bound,
                                              uint32_t buffer_token_size) {
  if (buffer_token_size == 0) return 0;
  uint64_t r = (total_k_upper_bound + buffer_token_size - 1) / buffer_token_size;
  return r > 0xFFFFFFFFull ? 0xFFFFFFFFu : static_cast<uint32_t>(r);
}

extern "C" mla_status_t mla_read_device_status(const void* workspace, uint32_t* status_out,
                                               mla_stream_t stream) {
  if (!workspace || !status_out) return mla::fail(MLA_ERR_INVALID_ARG, "null argument");
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaSuccess)
    e = cudaMemcpy(status_out, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return mla::fail(MLA_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  return MLA_OK;
}
