// Gather of one buffer row out of a paged cache into a contiguous buffer: the
// step the prefill plan exists for (generic_flare_mla_prefill_ragged_paged_plan:
// "gather K/V entries into a contiguous buffer").  Position bro[b] + i of the
// buffer holds context token co[b] + i of sequence b, whose cache row is
// page_table[b, a / P] * P + a % P (a = co[b] + i).
//
// HBM-bound copy: each 16-byte chunk of a cache row is read once and written
// once.  One thread moves one 16-byte chunk; the chunks of a row are adjacent
// threads, so a warp reads and writes whole rows (1152 bytes for a 576-wide
// bf16 latent row).
#include <cuda_runtime.h>

#include <cstdint>

#include "host_common.h"

namespace mla {
namespace {

constexpr int kGatherThreads = 256;

struct GatherParams {
  uint8_t* dst;
  long long dst_row;          // bytes
  const uint8_t* cache;
  long long page_bytes, tok_bytes;
  const uint32_t* page_table;
  long long pt_stride;
  const uint32_t* bro;
  const uint32_t* co;
  uint32_t* status;
  uint32_t B, P, max_pages, num_pages, chunks, rows_cap;
};

__global__ void __launch_bounds__(kGatherThreads) gather_kernel(const GatherParams p) {
  const uint32_t rows = min(p.bro[p.B], p.rows_cap);
  const unsigned long long total = static_cast<unsigned long long>(rows) * p.chunks;
  uint32_t bad = 0;
  for (unsigned long long idx = blockIdx.x * static_cast<unsigned long long>(blockDim.x) + threadIdx.x;
       idx < total; idx += static_cast<unsigned long long>(gridDim.x) * blockDim.x) {
    const uint32_t t = static_cast<uint32_t>(idx / p.chunks);
    const uint32_t c = static_cast<uint32_t>(idx - static_cast<unsigned long long>(t) * p.chunks);
    // Sequence owning buffer position t: the last b with bro[b] <= t (empty
    // windows share their start with the next sequence and are skipped).
    uint32_t lo = 0, hi = p.B;
    while (hi - lo > 1) {
      const uint32_t mid = (lo + hi) >> 1;
      if (p.bro[mid] <= t) lo = mid; else hi = mid;
    }
    const uint32_t a = p.co[lo] + (t - p.bro[lo]);
    const uint32_t col = a / p.P;
    if (col >= p.max_pages) { bad |= MLA_DEVICE_STATUS_BAD_COLUMN; continue; }
    const uint32_t page = p.page_table[lo * p.pt_stride + col];
    if (page >= p.num_pages) { bad |= MLA_DEVICE_STATUS_BAD_PAGE; continue; }
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(
        p.cache + page * p.page_bytes + static_cast<long long>(a - col * p.P) * p.tok_bytes) + c);
    reinterpret_cast<uint4*>(p.dst + t * p.dst_row)[c] = v;
  }
  if (bad && p.status) atomicOr(p.status, bad);
}

}  // namespace
}  // namespace mla

extern "C" mla_status_t mla_gather_rows(const mla_tensor_t* dst, const mla_tensor_t* cache,
                                        const mla_tensor_t* page_table,
                                        const uint32_t* buffer_row_offsets,
                                        const uint32_t* cache_offsets, uint32_t* status,
                                        mla_stream_t stream) {
  using namespace mla;
  mla_status_t st;
  if (!cache) return fail(MLA_ERR_INVALID_ARG, "cache descriptor is NULL");
  const mla_dtype_t dt = cache->dtype;
  if (dt != MLA_DTYPE_BF16 && dt != MLA_DTYPE_FP8_E4M3)
    return fail(MLA_ERR_INVALID_ARG, "cache must be bf16 or fp8");
  if ((st = check_tensor(cache, "cache", 3, dt)) != MLA_OK) return st;
  if ((st = check_tensor(dst, "dst", 2, dt)) != MLA_OK) return st;
  if ((st = check_tensor(page_table, "page_table", 2, MLA_DTYPE_U32)) != MLA_OK) return st;
  if (!buffer_row_offsets || !cache_offsets)
    return fail(MLA_ERR_INVALID_ARG, "buffer_row_offsets / cache_offsets is NULL");
  const int64_t es = dt == MLA_DTYPE_BF16 ? 2 : 1;
  const int64_t W = cache->shape[2], B = page_table->shape[0];
  if (dst->shape[1] != W) return fail(MLA_ERR_INVALID_ARG, "dst rows must be as wide as cache rows");
  if ((W * es) % 16 != 0 || W < 1) return fail(MLA_ERR_INVALID_ARG, "row width must be a positive multiple of 16 bytes");
  if (B < 1 || page_table->shape[1] < 1) return fail(MLA_ERR_INVALID_ARG, "empty page table");
  if (cache->shape[0] < 1 || cache->shape[1] < 1) return fail(MLA_ERR_INVALID_ARG, "empty cache");
  if (cache->shape[0] * cache->shape[1] > 0x7FFFFFFFll) return fail(MLA_ERR_INVALID_ARG, "cache exceeds 2^31 rows");
  if (!aligned16(dst->data) || !aligned16(cache->data))
    return fail(MLA_ERR_INVALID_ARG, "dst / cache data must be 16-byte aligned");
  if ((dst->stride[0] * es) % 16 != 0 || (cache->stride[0] * es) % 16 != 0 || (cache->stride[1] * es) % 16 != 0)
    return fail(MLA_ERR_INVALID_ARG, "dst / cache strides must be multiples of 16 bytes");
  int dev = 0, sms = 0;
  if ((st = check_device(&dev, &sms)) != MLA_OK) return st;
  if (dst->shape[0] == 0) return MLA_OK;

  GatherParams p;
  p.dst = static_cast<uint8_t*>(dst->data);
  p.dst_row = dst->stride[0] * es;
  p.cache = static_cast<const uint8_t*>(cache->data);
  p.page_bytes = cache->stride[0] * es;
  p.tok_bytes = cache->stride[1] * es;
  p.page_table = static_cast<const uint32_t*>(page_table->data);
  p.pt_stride = page_table->stride[0];
  p.bro = buffer_row_offsets;
  p.co = cache_offsets;
  p.status = status;
  p.B = static_cast<uint32_t>(B);
  p.P = static_cast<uint32_t>(cache->shape[1]);
  p.max_pages = static_cast<uint32_t>(page_table->shape[1]);
  p.num_pages = static_cast<uint32_t>(cache->shape[0]);
  p.chunks = static_cast<uint32_t>(W * es / 16);
  p.rows_cap = static_cast<uint32_t>(dst->shape[0]);
  const unsigned long long threads = static_cast<unsigned long long>(dst->shape[0]) * p.chunks;
  const unsigned long long want = (threads + kGatherThreads - 1) / kGatherThreads;
  const int blocks = static_cast<int>(want < 8ull * sms ? want : 8ull * sms);
  gather_kernel<<<blocks, kGatherThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "gather launch: %s", cudaGetErrorString(e));
  return MLA_OK;
}
