// Prefill plan: tiles the batch-order packing of all K contexts into buffer
// rows of buffer_token_size tokens (generic_flare_mla_prefill_ragged_paged_plan,
// summary and Args).  One CTA: a block-wide scan of the context lengths into
// shared memory, then a CTA-stride loop that emits every (row, sequence) entry.
#include <cuda_runtime.h>

#include <cstdint>

#include "host_common.h"

namespace mla {
namespace {

constexpr int kPlanThreads = 1024;
constexpr uint32_t kPlanMaxBatch = 16384;

__device__ __forceinline__ uint64_t warp_inclusive_scan(uint64_t x, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    uint64_t y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  return x;
}

// ctx_start[b] = G_b (start of sequence b's context in the packing), b = 0..B.
__global__ void __launch_bounds__(kPlanThreads, 1)
plan_kernel(const uint32_t* __restrict__ iro, const uint32_t* __restrict__ cache_lens, uint32_t B,
            uint32_t T, uint32_t max_rows, uint32_t* __restrict__ bro, uint32_t* __restrict__ co,
            int32_t* __restrict__ blen, uint32_t* __restrict__ num_rows) {
  extern __shared__ uint32_t ctx_start[];
  __shared__ uint64_t warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Each thread owns a contiguous run of sequences.
  const uint32_t per = (B + kPlanThreads - 1) / kPlanThreads;
  const uint32_t b0 = min(B, tid * per), b1 = min(B, b0 + per);
  uint64_t local = 0;
  bool bad = false;
  for (uint32_t b = b0; b < b1; ++b) {
    const uint32_t lo = iro[b], hi = iro[b + 1];
    bad |= hi < lo;
    local += static_cast<uint64_t>(cache_lens[b]) + (hi - lo);
  }
  // Block-wide exclusive scan of the per-thread sums.
  uint64_t incl = warp_inclusive_scan(local, lane);
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint64_t t = warp_tot[lane];
    uint64_t ti = warp_inclusive_scan(t, lane);
    warp_tot[lane] = ti - t;
  }
  __syncthreads();
  uint64_t run = warp_tot[warp] + incl - local;
  for (uint32_t b = b0; b < b1; ++b) {
    if (run > 0xFFFFFFFFull) bad = true;
    ctx_start[b] = static_cast<uint32_t>(run);
    run += static_cast<uint64_t>(cache_lens[b]) + (iro[b + 1] - iro[b]);
  }
  if (b1 == B && b0 < b1) {
    if (run > 0xFFFFFFFFull) bad = true;
    ctx_start[B] = static_cast<uint32_t>(run);
  }
  if (B == 0 && tid == 0) ctx_start[0] = 0;
  if (__syncthreads_or(bad)) {
    if (tid == 0 && num_rows) *num_rows = 0xFFFFFFFFu;
    return;
  }
  const uint64_t S = ctx_start[B];
  const uint64_t R = (S + T - 1) / T;
  if (tid == 0 && num_rows) *num_rows = static_cast<uint32_t>(R);

  const uint64_t width = static_cast<uint64_t>(B) + 1;
  const uint64_t total = static_cast<uint64_t>(max_rows) * width;
  for (uint64_t idx = tid; idx < total; idx += kPlanThreads) {
    const uint64_t r = idx / width;
    const uint32_t b = static_cast<uint32_t>(idx - r * width);
    const int64_t start = static_cast<int64_t>(r * T);
    const int64_t g = ctx_start[b];
    const int64_t off = min(max(g - start, int64_t(0)), int64_t(T));
    bro[idx] = static_cast<uint32_t>(off);
    if (b < B) {
      const int64_t L = static_cast<int64_t>(ctx_start[b + 1]) - g;
      const int64_t c = min(max(start - g, int64_t(0)), L);
      co[r * B + b] = static_cast<uint32_t>(c);
    } else {
      blen[r] = r < R ? static_cast<int32_t>(min(static_cast<int64_t>(T), static_cast<int64_t>(S) - start))
                      : -1;
    }
  }
}

}  // namespace
}  // namespace mla

extern "C" mla_status_t mla_prefill_plan(const uint32_t* input_row_offsets,
                                         const uint32_t* cache_lens, uint32_t batch,
                                         uint32_t buffer_token_size, uint32_t max_buffer_rows,
                                         uint32_t* buffer_row_offsets, uint32_t* cache_offsets,
                                         int32_t* buffer_lengths, uint32_t* num_rows,
                                         mla_stream_t stream) {
  using namespace mla;
  if (!input_row_offsets) return fail(MLA_ERR_INVALID_ARG, "input_row_offsets is NULL");
  if (batch > 0 && !cache_lens) return fail(MLA_ERR_INVALID_ARG, "cache_lens is NULL");
  if (batch > kPlanMaxBatch)
    return fail(MLA_ERR_INVALID_ARG, "batch %u exceeds %u", batch, kPlanMaxBatch);
  if (buffer_token_size == 0) return fail(MLA_ERR_INVALID_ARG, "buffer_token_size is 0");
  if (max_buffer_rows > 0 && (!buffer_row_offsets || !buffer_lengths || (batch > 0 && !cache_offsets)))
    return fail(MLA_ERR_INVALID_ARG, "plan output pointer is NULL");
  if (static_cast<uint64_t>(max_buffer_rows) * (batch + 1ull) > 0xFFFFFFFFull)
    return fail(MLA_ERR_INVALID_ARG, "max_buffer_rows * (batch + 1) exceeds 32 bits");
  int dev = 0, sms = 0;
  mla_status_t st = check_device(&dev, &sms);
  if (st != MLA_OK) return st;
  const int smem = static_cast<int>((batch + 1) * sizeof(uint32_t));
  if ((st = set_max_dynamic_smem(reinterpret_cast<const void*>(plan_kernel), smem, dev, 0)) != MLA_OK)
    return st;
  plan_kernel<<<1, kPlanThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
      input_row_offsets, cache_lens, batch, buffer_token_size, max_buffer_rows, buffer_row_offsets,
      cache_offsets, buffer_lengths, num_rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "plan launch: %s", cudaGetErrorString(e));
  return MLA_OK;
}
