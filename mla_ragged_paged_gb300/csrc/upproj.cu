// Up-projection of latent cache rows to per-head K_nope and V: the step
// between the buffer-row gather and the attention when the cache holds the
// compressed latent row (c_kv | k_rope) rather than K_nope and V
// (generic_flare_mla_prefill_ragged_paged_plan summary: the plan lets the
// prefill kernel gather K/V entries into a contiguous buffer;
// mla_prefill_v2_ragged Args: v is the nope segment of the latent cache).
//   out[t, n] = sum_k A[t, k] * W[n, k]          (W in nn.Linear layout [N, K])
// A dense bf16 GEMM on the tensor cores (tcgen05.mma, fp32 accumulation in
// tensor memory, bf16 output).  A is either a plain row-major matrix or, fused
// with the gather, the first K columns of a buffer row's cache rows, fetched
// through the page table by TMA row gathers (four rows per instruction).
//
// K is at most 512 (kv_lora_rank), so a 128-row block of A fits in tensor
// memory (256 columns of packed bf16 pairs) and stays there while the CTA
// runs through its output tiles of that block: only the weight tiles stream
// through shared memory, 16 KB per 64-wide K block (64 bytes per tensor-core
// cycle instead of 96 when both operands stream), and A is fetched (or
// gathered) once per 128 rows instead of once per output tile.  A ring slot
// holds two 64-wide K blocks (32 KB), so the one issuing thread waits once
// per eight UMMAs.
//
// Persistent kernel, one CTA of 192 threads per SM; each CTA takes a
// contiguous range of 128 x 128 output tiles, row block by row block:
//   warp 0     producer: TMA of A's K blocks when the row block changes, then
//              per tile its weight K blocks, into a 6-slot ring of 32 KB
//   warp 1     tensor-core thread and tensor-memory owner: copies A's K blocks
//              from shared into tensor memory (tcgen05.cp), then per tile 32
//              UMMAs M128 N128 K16 with A read from tensor memory
//   warps 2-5  epilogue: tensor memory -> bf16 -> 128B-swizzled staging ->
//              TMA tile store; each warp stores its own 32 rows, 64 columns
//              at a time through two 4 KB buffers, with no barrier between
//              the warps
// Tensor memory: A [0, 256), two accumulators [256, 384) and [384, 512), so
// the epilogue of one tile overlaps the main loop of the next.  With two
// weight matrices (K_nope and V from the same latent rows) the tiles of both
// outputs share the resident A.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>

#include "host_common.h"
#include "sm103.cuh"

namespace mla {
namespace {

constexpr int kGM = 128;        // output rows per tile (= tensor-memory lanes)
constexpr int kGN = 128;        // output columns per tile (UMMA N)
constexpr int kGAtom = 64;      // K per 128-byte swizzle atom of bf16
constexpr int kGMaxK = 512;     // A block resident in tensor memory: 128 x 512 bf16
constexpr int kGStages = 6;
constexpr int kGThreads = 192;
constexpr uint32_t kGAtomBytes = 128 * kGAtom * 2;  // 16 KB: 128 rows of one atom
constexpr uint32_t kGChunk = 2 * kGAtomBytes;       // a ring slot: two atoms
constexpr uint32_t kGSlab = 32 * 64 * 2;       // 4 KB: 64 output columns of one warp's 32 rows
constexpr uint32_t kGTmemCols = 512;
constexpr uint32_t kGColAcc = kGMaxK / 2;      // accumulators after A's 256 columns

struct __align__(1024) GemmSmem {
  uint8_t ring[kGStages][kGChunk];
  uint8_t c[4][2][kGSlab];   // per epilogue warp, two staging buffers
  uint64_t full[kGStages], empty[kGStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t a_drain, drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
};
static_assert(sizeof(GemmSmem) + 1024 <= 232448, "up-projection shared memory");

struct GemmParams {
  CUtensorMap tm_a;     // contiguous A [M, K], box 64 x 128; or cache rows [slots, K], box 64 x 1
  CUtensorMap tm_b[2];  // weights [N, K], box 64 x 128
  CUtensorMap tm_c[2];  // outputs [M, N], box 64 x 32
  uint32_t M, k_atoms, m_tiles, n_tiles, num_out;  // k_atoms = ceil(K / 64)
  // Row gather: buffer position t holds context token co[b] + t - bro[b] of
  // the sequence b with bro[b] <= t < bro[b+1]; its cache row (slot) is
  // page_table[b, a / P] * P + a % P.
  uint32_t gather;
  const uint32_t* page_table;
  long long pt_stride;
  const uint32_t* bro;
  const uint32_t* co;
  uint32_t B, P, num_pages, max_pages;
  uint32_t* status;
};

// Tiles in row-block-major order: t = (m * num_out + o) * n_tiles + n.
struct TileIdx {
  uint32_t m, n, o;
};
__device__ __forceinline__ TileIdx tile_of(const GemmParams& p, uint32_t t) {
  TileIdx r;
  const uint32_t per_m = p.n_tiles * p.num_out;
  r.m = t / per_m;
  const uint32_t rest = t - r.m * per_m;
  r.o = rest / p.n_tiles;
  r.n = rest - r.o * p.n_tiles;
  return r;
}
// This CTA's contiguous share of the tiles.
__device__ __forceinline__ void tile_range(const GemmParams& p, uint32_t& t0, uint32_t& t1) {
  const unsigned long long total = static_cast<unsigned long long>(p.m_tiles) * p.n_tiles * p.num_out;
  t0 = static_cast<uint32_t>(total * blockIdx.x / gridDim.x);
  t1 = static_cast<uint32_t>(total * (blockIdx.x + 1) / gridDim.x);
}

// Cache slot of buffer position t (slot 0 for positions past the row's
// tokens or with a bad page, whose outputs are then unspecified).
__device__ __forceinline__ int32_t gather_slot(const GemmParams& p, uint32_t t, uint32_t& bad) {
  if (t >= p.M || t >= p.bro[p.B]) return 0;
  uint32_t lo = 0, hi = p.B;
  while (hi - lo > 1) {
    const uint32_t mid = (lo + hi) >> 1;
    if (p.bro[mid] <= t) lo = mid; else hi = mid;
  }
  const uint32_t a = p.co[lo] + (t - p.bro[lo]);
  const uint32_t col = a / p.P;
  if (col >= p.max_pages) {
    bad |= MLA_DEVICE_STATUS_BAD_COLUMN;
    return 0;
  }
  const uint32_t page = p.page_table[static_cast<long long>(lo) * p.pt_stride + col];
  if (page >= p.num_pages) {
    bad |= MLA_DEVICE_STATUS_BAD_PAGE;
    return 0;
  }
  return static_cast<int32_t>(page * p.P + (a - col * p.P));
}

// One 128-lane x 256-bit copy from shared memory (an operand descriptor) into
// tensor memory: 32 bytes of each of 128 rows.  Ordered with the tcgen05.mma
// instructions the same thread issues afterwards.
__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ void gemm_producer(GemmSmem& s, const GemmParams& p, int lane, volatile uint32_t* abort) {
  uint32_t t0, t1;
  tile_range(p, t0, t1);
  uint32_t pos = 0;                 // ring position (chunks issued)
  uint32_t cur_m = 0xFFFFFFFFu;
  uint32_t bad = 0;
  bool alive = true;
  const uint64_t keep = l2_policy_evict_last();
  // Claim the next ring slot and arm its barrier for `atoms` 16 KB atoms.
  auto acquire = [&](uint32_t atoms, uint32_t& bar, uint32_t& dst) -> bool {
    const uint32_t st = pos % kGStages;
    if (!mbar_wait(smem_u32(&s.empty[st]), ((pos / kGStages) & 1u) ^ 1u, abort)) return false;
    bar = smem_u32(&s.full[st]);
    dst = smem_u32(s.ring[st]);
    if (lane == 0) mbar_arrive_expect_tx(bar, atoms * kGAtomBytes);
    __syncwarp();
    ++pos;
    return true;
  };
  for (uint32_t t = t0; t < t1 && alive; ++t) {
    const TileIdx ti = tile_of(p, t);
    if (ti.m != cur_m) {
      // A's K blocks of the new row block (gather: rows 4*lane .. 4*lane+3
      // of each block, 128 bytes each).
      cur_m = ti.m;
      int32_t rows[4] = {0, 0, 0, 0};
      if (p.gather) {
#pragma unroll
        for (int j = 0; j < 4; ++j) rows[j] = gather_slot(p, ti.m * kGM + lane * 4 + j, bad);
      }
      for (uint32_t a0 = 0; a0 < p.k_atoms && alive; a0 += 2) {
        const uint32_t na = min(2u, p.k_atoms - a0);
        uint32_t bar, dst;
        if (!(alive = acquire(na, bar, dst))) break;
        for (uint32_t a = 0; a < na; ++a) {
          const int32_t x = static_cast<int32_t>((a0 + a) * kGAtom);
          if (p.gather) {
            tma_gather4_2d(dst + a * kGAtomBytes + lane * 512u, &p.tm_a, bar, x, rows[0], rows[1], rows[2], rows[3]);
          } else if (lane == 0) {
            tma_load_2d(dst + a * kGAtomBytes, &p.tm_a, bar, x, static_cast<int32_t>(ti.m * kGM));
          }
        }
      }
    }
    for (uint32_t a0 = 0; a0 < p.k_atoms && alive; a0 += 2) {
      const uint32_t na = min(2u, p.k_atoms - a0);
      uint32_t bar, dst;
      if (!(alive = acquire(na, bar, dst))) break;
      // The weights are read once per row block: keep them in L2 against
      // the streamed output.
      if (lane == 0)
        for (uint32_t a = 0; a < na; ++a)
          tma_load_2d_hint(dst + a * kGAtomBytes, &p.tm_b[ti.o], bar, static_cast<int32_t>((a0 + a) * kGAtom),
                           static_cast<int32_t>(ti.n * kGN), keep);
    }
  }
  for (int o = 16; o; o >>= 1) bad |= __shfl_xor_sync(0xffffffffu, bad, o);
  if (lane == 0 && bad && p.status) atomicOr(p.status, bad);
  if (*abort) {
    // Let the copies still in flight land before the CTA exits.
    const uint32_t n = pos < kGStages ? pos : kGStages;
    for (uint32_t i = 1; i <= n; ++i) {
      const uint32_t q = pos - i;
      const uint64_t t0n = global_timer_ns();
      while (!mbar_try_wait(smem_u32(&s.full[q % kGStages]), (q / kGStages) & 1u))
        if (global_timer_ns() - t0n > kWaitTimeoutNs) break;
    }
  }
}

__device__ void gemm_mma(GemmSmem& s, const GemmParams& p, uint32_t tmem, volatile uint32_t* abort) {
  uint32_t t0, t1;
  tile_range(p, t0, t1);
  const uint32_t idesc = make_idesc(kGM, kGN, 1, false);  // bf16 A and B, both K-major
  uint32_t pos = 0, tl = 0, drains = 0;
  uint32_t cur_m = 0xFFFFFFFFu;
  bool alive = true;
  // Wait for the next ring chunk; returns its shared address.
  auto next_chunk = [&](uint32_t& addr) -> bool {
    const uint32_t st = pos % kGStages;
    if (!mbar_wait(smem_u32(&s.full[st]), (pos / kGStages) & 1u, abort)) return false;
    tc_fence_after();
    addr = smem_u32(s.ring[st]);
    return true;
  };
  auto release = [&]() {
    umma_commit(smem_u32(&s.empty[pos % kGStages]));
    ++pos;
  };
  for (uint32_t t = t0; t < t1 && alive; ++t, ++tl) {
    const TileIdx ti = tile_of(p, t);
    if (ti.m != cur_m) {
      if (cur_m != 0xFFFFFFFFu) {
        // Every UMMA reading the old A must complete before it is overwritten.
        umma_commit(smem_u32(&s.a_drain));
        if (!(alive = mbar_wait(smem_u32(&s.a_drain), drains & 1u, abort))) break;
        ++drains;
        tc_fence_after();
      }
      cur_m = ti.m;
      for (uint32_t a0 = 0; a0 < p.k_atoms && alive; a0 += 2) {
        uint32_t a;
        if (!(alive = next_chunk(a))) break;
        for (uint32_t at = a0; at < a0 + 2 && at < p.k_atoms; ++at) {
          const uint64_t ad = sw128_desc_at(a + (at - a0) * kGAtomBytes);
#pragma unroll
          for (int k = 0; k < kGAtom / 16; ++k) tmem_cp_128x256b(tmem + at * 32 + k * 8, ad + 2 * k);
        }
        release();
      }
      if (!alive) break;
    }
    const uint32_t buf = tl & 1u;
    if (!(alive = mbar_wait(smem_u32(&s.acc_empty[buf]), ((tl >> 1) & 1u) ^ 1u, abort))) break;
    tc_fence_after();
    const uint32_t d = tmem + kGColAcc + buf * kGN;
    for (uint32_t a0 = 0; a0 < p.k_atoms && alive; a0 += 2) {
      uint32_t b;
      if (!(alive = next_chunk(b))) break;
      for (uint32_t at = a0; at < a0 + 2 && at < p.k_atoms; ++at) {
        const uint64_t bd = sw128_desc_at(b + (at - a0) * kGAtomBytes);
#pragma unroll
        for (int k = 0; k < kGAtom / 16; ++k)
          umma_f16_ts(d, tmem + at * 32 + k * 8, bd + 2 * k, idesc, (at | k) != 0);
      }
      release();
    }
    if (alive) umma_commit(smem_u32(&s.acc_full[buf]));
  }
  // No UMMA may still be in flight when tensor memory is released.
  umma_commit(smem_u32(&s.drain));
  const uint64_t tw = global_timer_ns();
  while (!mbar_try_wait(smem_u32(&s.drain), 0))
    if (global_timer_ns() - tw > kWaitTimeoutNs) break;
}

__device__ void gemm_epilogue(GemmSmem& s, const GemmParams& p, uint32_t tmem, int quarter, int lane,
                              volatile uint32_t* abort) {
  uint32_t t0, t1;
  tile_range(p, t0, t1);
  const int r = lane;                                    // row inside this warp's 32-row quarter
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint64_t stream_out = l2_policy_evict_first();
  uint32_t tl = 0, slab = 0;
  for (uint32_t t = t0; t < t1; ++t, ++tl) {
    const TileIdx ti = tile_of(p, t);
    const uint32_t buf = tl & 1u;
    if (!mbar_wait(smem_u32(&s.acc_full[buf]), (tl >> 1) & 1u, abort)) break;
    tc_fence_after();
#pragma unroll 1
    for (int c = 0; c < kGN / 64; ++c, ++slab) {
      uint32_t v0[32], v1[32];
      const uint32_t col = tmem + lane_off + kGColAcc + buf * kGN + c * 64;
      tmem_ld_32x32b_x32(col, v0);
      tmem_ld_32x32b_x32(col + 32, v1);
      tmem_ld_wait();
      if (c == kGN / 64 - 1) {
        // The accumulator is in registers: the next tile may use it.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.acc_empty[buf]));
      }
      uint32_t pk[32];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        pk[e] = pack_bf16x2(__uint_as_float(v0[2 * e]), __uint_as_float(v0[2 * e + 1]));
        pk[16 + e] = pack_bf16x2(__uint_as_float(v1[2 * e]), __uint_as_float(v1[2 * e + 1]));
      }
      // The store that last read this staging buffer (two slabs ago) must be done.
      if (lane == 0) bulk_wait_group_read<1>();
      __syncwarp();
      const uint32_t base = smem_u32(s.c[quarter][slab & 1u]);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t a = base + r * 128 + ((q ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(pk[4 * q]), "r"(pk[4 * q + 1]),
                     "r"(pk[4 * q + 2]), "r"(pk[4 * q + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        // The output is written once and not read here: stream it through L2.
        tma_store_2d_hint(&p.tm_c[ti.o], base, static_cast<int32_t>(ti.n * kGN + c * 64),
                          static_cast<int32_t>(ti.m * kGM + quarter * 32), stream_out);
        bulk_commit_group();
      }
    }
  }
  if (lane == 0) bulk_wait_group_all();
}

__global__ void __launch_bounds__(kGThreads, 1) up_project_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  GemmSmem& s = *reinterpret_cast<GemmSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile uint32_t* abort = &s.abort_flag;
  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    for (int i = 0; i < kGStages; ++i) {
      mbar_init(smem_u32(&s.full[i]), 1);
      mbar_init(smem_u32(&s.empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.acc_full[i]), 1);
      mbar_init(smem_u32(&s.acc_empty[i]), 4);  // the four epilogue warps
    }
    mbar_init(smem_u32(&s.a_drain), 1);
    mbar_init(smem_u32(&s.drain), 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tm_a);
    for (uint32_t o = 0; o < p.num_out; ++o) {
      tma_prefetch_desc(&p.tm_b[o]);
      tma_prefetch_desc(&p.tm_c[o]);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s.tmem_base), kGTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  if (warp == 0) {
    gemm_producer(s, p, lane, abort);
  } else if (warp == 1) {
    if (lane == 0) gemm_mma(s, p, tmem, abort);
    __syncwarp();
  } else {
    gemm_epilogue(s, p, tmem, warp & 3, lane, abort);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kGTmemCols);
  }
  if (threadIdx.x == 0 && s.abort_flag && p.status) atomicOr(p.status, MLA_DEVICE_STATUS_TIMEOUT);
}

// Checks shared by both entry points: a bf16 [rows, cols] matrix with 16-byte
// aligned rows.
mla_status_t check_matrix(const mla_tensor_t* t, const char* name) {
  mla_status_t st = check_tensor(t, name, 2, MLA_DTYPE_BF16);
  if (st != MLA_OK) return st;
  if (!aligned16(t->data) || (t->stride[0] * 2) % 16 != 0 || t->stride[0] * 2 >= (1ll << 40))
    return fail(MLA_ERR_INVALID_ARG, "%s must start 16-byte aligned with a 16-byte-multiple row stride", name);
  return MLA_OK;
}

mla_status_t encode_matrix(CUtensorMap* map, const mla_tensor_t* t, uint64_t cols, uint32_t box_rows,
                           const char* what) {
  uint64_t dims[2] = {cols, static_cast<uint64_t>(t->shape[0])};
  uint64_t str[1] = {static_cast<uint64_t>(t->stride[0]) * 2};
  uint32_t box[2] = {64, box_rows};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, t->data, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B, what);
}

// Weights and outputs of `num_out` projections of the same A ([M, K]).
mla_status_t setup_outputs(GemmParams& p, const mla_tensor_t* const* outs, const mla_tensor_t* const* weights,
                           uint32_t num_out, int64_t M, int64_t K) {
  mla_status_t st;
  if (K > kGMaxK) return fail(MLA_ERR_INVALID_ARG, "K = %lld exceeds %d (the latent width the kernel keeps on chip)",
                              (long long)K, kGMaxK);
  int64_t N = -1;
  for (uint32_t o = 0; o < num_out; ++o) {
    if ((st = check_matrix(outs[o], o ? "v_out" : "out")) != MLA_OK) return st;
    if ((st = check_matrix(weights[o], o ? "w_uv" : "weight")) != MLA_OK) return st;
    if (weights[o]->shape[1] != K) return fail(MLA_ERR_INVALID_ARG, "weight must be [N, K] with K = %lld", (long long)K);
    if (N < 0) N = weights[o]->shape[0];
    if (weights[o]->shape[0] != N) return fail(MLA_ERR_INVALID_ARG, "both weights must have the same N");
    if (outs[o]->shape[0] != M || outs[o]->shape[1] != N)
      return fail(MLA_ERR_INVALID_ARG, "out must be [%lld, %lld]", (long long)M, (long long)N);
    if ((st = encode_matrix(&p.tm_b[o], weights[o], static_cast<uint64_t>(K), kGN, "weight")) != MLA_OK) return st;
    if ((st = encode_matrix(&p.tm_c[o], outs[o], static_cast<uint64_t>(N), 32, "out")) != MLA_OK) return st;
  }
  if (N < 1 || K < 1) return fail(MLA_ERR_INVALID_ARG, "empty projection");
  p.M = static_cast<uint32_t>(M);
  p.k_atoms = static_cast<uint32_t>((K + kGAtom - 1) / kGAtom);
  p.m_tiles = static_cast<uint32_t>((M + kGM - 1) / kGM);
  p.n_tiles = static_cast<uint32_t>((N + kGN - 1) / kGN);
  p.num_out = num_out;
  if (static_cast<uint64_t>(p.m_tiles) * p.n_tiles * num_out > 0xFFFFFFFFull)
    return fail(MLA_ERR_INVALID_ARG, "too many output tiles");
  return MLA_OK;
}

mla_status_t launch(GemmParams& p, uint32_t* status, mla_stream_t stream) {
  int dev = 0, sms = 0;
  mla_status_t st = check_device(&dev, &sms);
  if (st != MLA_OK) return st;
  p.status = status;
  const uint64_t tiles = static_cast<uint64_t>(p.m_tiles) * p.n_tiles * p.num_out;
  if (tiles == 0) return MLA_OK;
  const int smem = static_cast<int>(sizeof(GemmSmem) + 1024);
  if ((st = set_max_dynamic_smem(reinterpret_cast<const void*>(up_project_kernel), smem, dev, 5)) != MLA_OK)
    return st;
  const uint32_t grid = static_cast<uint32_t>(std::min<uint64_t>(tiles, static_cast<uint64_t>(sms)));
  up_project_kernel<<<grid, kGThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "up-projection launch: %s", cudaGetErrorString(e));
  return MLA_OK;
}

}  // namespace
}  // namespace mla

extern "C" mla_status_t mla_up_project(const mla_tensor_t* out, const mla_tensor_t* latent,
                                       const mla_tensor_t* weight, uint32_t* status, mla_stream_t stream) {
  using namespace mla;
  mla_status_t st;
  if ((st = check_matrix(latent, "latent")) != MLA_OK) return st;
  GemmParams p;
  memset(&p, 0, sizeof(p));
  const int64_t M = latent->shape[0], K = latent->shape[1];
  const mla_tensor_t* outs[1] = {out};
  const mla_tensor_t* ws[1] = {weight};
  if ((st = setup_outputs(p, outs, ws, 1, M, K)) != MLA_OK) return st;
  if (M == 0) return MLA_OK;
  if ((st = encode_matrix(&p.tm_a, latent, static_cast<uint64_t>(K), kGM, "latent")) != MLA_OK) return st;
  return launch(p, status, stream);
}

extern "C" mla_status_t mla_gather_up_project(const mla_tensor_t* k_out, const mla_tensor_t* v_out,
                                              const mla_tensor_t* cache, const mla_tensor_t* w_uk,
                                              const mla_tensor_t* w_uv, const mla_tensor_t* page_table,
                                              const uint32_t* buffer_row_offsets,
                                              const uint32_t* cache_offsets, uint32_t kv_lora_rank,
                                              uint32_t* status, mla_stream_t stream) {
  using namespace mla;
  mla_status_t st;
  if ((st = check_tensor(cache, "cache", 3, MLA_DTYPE_BF16)) != MLA_OK) return st;
  if ((st = check_tensor(page_table, "page_table", 2, MLA_DTYPE_U32)) != MLA_OK) return st;
  if (!buffer_row_offsets || !cache_offsets)
    return fail(MLA_ERR_INVALID_ARG, "buffer_row_offsets / cache_offsets is NULL");
  if (!k_out) return fail(MLA_ERR_INVALID_ARG, "k_out descriptor is NULL");
  if ((v_out == nullptr) != (w_uv == nullptr))
    return fail(MLA_ERR_INVALID_ARG, "v_out and w_uv must both be given or both be NULL");
  const int64_t NP = cache->shape[0], P = cache->shape[1], W = cache->shape[2];
  const int64_t B = page_table->shape[0], max_pages = page_table->shape[1];
  if (kv_lora_rank < 1 || static_cast<int64_t>(kv_lora_rank) > W)
    return fail(MLA_ERR_INVALID_ARG, "kv_lora_rank must be in 1..%lld (the cache row width)", (long long)W);
  if (kv_lora_rank % 8 != 0) return fail(MLA_ERR_INVALID_ARG, "kv_lora_rank must be a multiple of 8");
  if (NP < 1 || P < 1 || max_pages < 1 || B < 1) return fail(MLA_ERR_INVALID_ARG, "empty cache or page table");
  if (NP * P > 0x7FFFFFFFll) return fail(MLA_ERR_INVALID_ARG, "cache exceeds 2^31 rows");
  // The rows of all pages form one [num_pages * P, W] matrix for the row gather.
  if (cache->stride[0] != P * cache->stride[1])
    return fail(MLA_ERR_INVALID_ARG, "cache pages must be contiguous (page stride = P x token stride)");
  if (!aligned16(cache->data) || (cache->stride[1] * 2) % 16 != 0 || cache->stride[1] * 2 >= (1ll << 40))
    return fail(MLA_ERR_INVALID_ARG, "cache must start 16-byte aligned with a 16-byte-multiple token stride");
  GemmParams p;
  memset(&p, 0, sizeof(p));
  const int64_t M = k_out->shape[0], K = kv_lora_rank;
  const mla_tensor_t* outs[2] = {k_out, v_out};
  const mla_tensor_t* ws[2] = {w_uk, w_uv};
  if ((st = setup_outputs(p, outs, ws, v_out ? 2u : 1u, M, K)) != MLA_OK) return st;
  if (M == 0) return MLA_OK;
  {
    uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(NP * P)};
    uint64_t str[1] = {static_cast<uint64_t>(cache->stride[1]) * 2};
    uint32_t box[2] = {64, 1};  // row gathers take a one-row box
    if ((st = encode_tiled(&p.tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cache->data, dims, str, box,
                           CU_TENSOR_MAP_SWIZZLE_128B, "cache")) != MLA_OK)
      return st;
  }
  p.gather = 1;
  p.page_table = static_cast<const uint32_t*>(page_table->data);
  p.pt_stride = page_table->stride[0];
  p.bro = buffer_row_offsets;
  p.co = cache_offsets;
  p.B = static_cast<uint32_t>(B);
  p.P = static_cast<uint32_t>(P);
  p.num_pages = static_cast<uint32_t>(NP);
  p.max_pages = static_cast<uint32_t>(max_pages);
  return launch(p, status, stream);
}
