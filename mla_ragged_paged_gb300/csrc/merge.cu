// Combination of the buffer rows of a chunked prefill: per (token, head),
//   out = sum_r e^(lse_r - m) O_r / sum_r e^(lse_r - m),  m = max_r lse_r,
// over the rows whose window holds keys of the token's sequence and whose lse
// is finite.  HBM-bound: each row's 256-byte output and 4-byte lse are read
// once and the merged row is written once.  Sixteen threads share one
// (token, head) row, 8 columns (16 bytes) each, so a half-warp reads one
// contiguous 256-byte row.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "host_common.h"
#include "sm103.cuh"

namespace mla {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kBatch = 4;  // rows whose loads are in flight together
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint4 ld_nc_v4(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xFFFF0000u);
}

struct MergeParams {
  uint16_t* out;
  long long o_tok, o_head;
  const uint16_t* po;
  long long po_row, po_tok, po_head;
  const float* pl;
  long long pl_row, pl_tok, pl_head;
  const uint32_t* ro;
  const uint32_t* bro;
  uint32_t B, R, H, Tq;
};

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p) {
  const uint32_t t_begin = p.ro[0], t_end = min(p.ro[p.B], p.Tq);
  if (t_end <= t_begin) return;
  const unsigned long long total = static_cast<unsigned long long>(t_end - t_begin) * p.H * 16u;
  for (unsigned long long idx = blockIdx.x * static_cast<unsigned long long>(blockDim.x) + threadIdx.x;
       idx < total; idx += static_cast<unsigned long long>(gridDim.x) * blockDim.x) {
    const uint32_t c = static_cast<uint32_t>(idx & 15u);
    const unsigned long long th = idx >> 4;
    const uint32_t h = static_cast<uint32_t>(th % p.H);
    const uint32_t t = t_begin + static_cast<uint32_t>(th / p.H);
    // Sequence of token t: the last b with ro[b] <= t.
    uint32_t lo = 0, hi = p.B;
    while (hi - lo > 1) {
      const uint32_t mid = (lo + hi) >> 1;
      if (p.ro[mid] <= t) lo = mid; else hi = mid;
    }
    const uint32_t b = lo;
    float m = -INFINITY, den = 0.f, acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    // Rows in batches of kBatch: every load of a batch is issued before any
    // is used, so a thread keeps kBatch 16-byte reads in flight.
    for (uint32_t r0 = 0; r0 < p.R; r0 += kBatch) {
      float ls[kBatch];
      uint4 v[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const uint32_t r = r0 + k;
        ls[k] = -INFINITY;
        v[k] = make_uint4(0u, 0u, 0u, 0u);
        if (r < p.R) {
          const uint32_t* row = p.bro + static_cast<size_t>(r) * (p.B + 1);
          if (row[b + 1] > row[b]) {  // sequence b has keys in row r
            ls[k] = p.pl[r * p.pl_row + t * p.pl_tok + h * p.pl_head];
            v[k] = ld_nc_v4(p.po + r * p.po_row + t * p.po_tok + h * p.po_head + 8 * c);
          }
        }
      }
      float mb = m;
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (ls[k] > mb && ls[k] < INFINITY) mb = ls[k];
      if (mb > m) {
        const float cr = ex2_approx((m - mb) * kLog2e);  // 0 while m = -inf
        den *= cr;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] *= cr;
        m = mb;
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (!(ls[k] > -INFINITY) || !(ls[k] < INFINITY)) continue;
        const float wgt = ex2_approx((ls[k] - m) * kLog2e);
        den += wgt;
        const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x0, x1;
          bf16x2_to_f32(w[e], x0, x1);
          acc[2 * e] = fmaf(wgt, x0, acc[2 * e]);
          acc[2 * e + 1] = fmaf(wgt, x1, acc[2 * e + 1]);
        }
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    uint4 o;
    o.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    o.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    o.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    o.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4*>(p.out + t * p.o_tok + h * p.o_head + 8 * c) = o;
  }
}

}  // namespace
}  // namespace mla

extern "C" mla_status_t mla_prefill_merge(const mla_tensor_t* out, const mla_tensor_t* partial_out,
                                          const mla_tensor_t* partial_lse, const uint32_t* row_offsets,
                                          const uint32_t* buffer_row_offsets, uint32_t batch,
                                          mla_stream_t stream) {
  using namespace mla;
  mla_status_t st;
  if ((st = check_tensor(out, "out", 3, MLA_DTYPE_BF16)) != MLA_OK) return st;
  if ((st = check_tensor(partial_out, "partial_out", 4, MLA_DTYPE_BF16)) != MLA_OK) return st;
  if ((st = check_tensor(partial_lse, "partial_lse", 3, MLA_DTYPE_F32)) != MLA_OK) return st;
  if (!row_offsets || !buffer_row_offsets)
    return fail(MLA_ERR_INVALID_ARG, "row_offsets / buffer_row_offsets is NULL");
  if (batch < 1 || batch > 0x7FFFFFFEu) return fail(MLA_ERR_INVALID_ARG, "batch must be >= 1");
  const int64_t Tq = out->shape[0], H = out->shape[1], R = partial_out->shape[0];
  if (out->shape[2] != 128) return fail(MLA_ERR_INVALID_ARG, "out must be [Tq, H, 128]");
  if (R < 1) return fail(MLA_ERR_INVALID_ARG, "partial_out holds no rows");
  if (partial_out->shape[1] != Tq || partial_out->shape[2] != H || partial_out->shape[3] != 128)
    return fail(MLA_ERR_INVALID_ARG, "partial_out must be [R, Tq, H, 128] matching out");
  if (partial_lse->shape[0] != R || partial_lse->shape[1] != Tq || partial_lse->shape[2] != H)
    return fail(MLA_ERR_INVALID_ARG, "partial_lse must be [R, Tq, H] matching partial_out");
  if (!aligned16(out->data) || !aligned16(partial_out->data))
    return fail(MLA_ERR_INVALID_ARG, "out / partial_out data must be 16-byte aligned");
  for (int d = 0; d < 2; ++d)
    if ((out->stride[d] * 2) % 16 != 0) return fail(MLA_ERR_INVALID_ARG, "out strides must be multiples of 16 bytes");
  for (int d = 0; d < 3; ++d)
    if ((partial_out->stride[d] * 2) % 16 != 0)
      return fail(MLA_ERR_INVALID_ARG, "partial_out strides must be multiples of 16 bytes");
  if (reinterpret_cast<uintptr_t>(partial_lse->data) & 3u)
    return fail(MLA_ERR_INVALID_ARG, "partial_lse data must be 4-byte aligned");
  int dev = 0, sms = 0;
  if ((st = check_device(&dev, &sms)) != MLA_OK) return st;
  if (Tq == 0 || H == 0) return MLA_OK;

  MergeParams p;
  p.out = static_cast<uint16_t*>(out->data);
  p.o_tok = out->stride[0];
  p.o_head = out->stride[1];
  p.po = static_cast<const uint16_t*>(partial_out->data);
  p.po_row = partial_out->stride[0];
  p.po_tok = partial_out->stride[1];
  p.po_head = partial_out->stride[2];
  p.pl = static_cast<const float*>(partial_lse->data);
  p.pl_row = partial_lse->stride[0];
  p.pl_tok = partial_lse->stride[1];
  p.pl_head = partial_lse->stride[2];
  p.ro = row_offsets;
  p.bro = buffer_row_offsets;
  p.B = batch;
  p.R = static_cast<uint32_t>(R);
  p.H = static_cast<uint32_t>(H);
  p.Tq = static_cast<uint32_t>(Tq);
  const unsigned long long threads = static_cast<unsigned long long>(Tq) * H * 16u;
  const unsigned long long want = (threads + kMergeThreads - 1) / kMergeThreads;
  const int blocks = static_cast<int>(want < 8ull * sms ? want : 8ull * sms);
  merge_kernel<<<blocks, kMergeThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "merge launch: %s", cudaGetErrorString(e));
  return MLA_OK;
}
