// Ragged causal MLA prefill attention for sm_103a (flare_mla_prefill:
// description and Args; the k_rope_scales overload for fp8 inputs).
//
// Per work item (sequence b, head h, block of 256 query rows split into two
// 128-row tiles Q0/Q1) one CTA streams the sequence's K context in 128-key
// tiles:
//   S_q  = Q_q . [K_nope | K_rope]^T         (UMMA, K = 192, fp32 in TMEM)
//   P_q  = exp2(S_q * scale * log2(e) - m)   (one thread per query row)
//   O_q += P_q . V                           (UMMA, A = P read from TMEM)
// The two Q tiles ping-pong so one tile's softmax overlaps the other tile's
// GEMMs, and a tile's next S is computed while its softmax runs.  K_rope (64
// dims shared by every head) is fetched from the paged pool through the page
// table.
//
// Warp roles (384 threads = three warpgroups, one warp of each per SM
// sub-partition):
//   warp 0      producer: work-item fetch (atomic counter), TMA loads
//   warp 1      UMMA issuer for Q0 (one thread) and tensor-memory owner
//   warp 2      UMMA issuer for Q1 (one thread)
//   warp 3      fp8 inputs only: Q_rope conversion to bf16 (else idle)
//   warps 4-7   softmax + epilogue for Q0
//   warps 8-11  softmax + epilogue for Q1
// A warp may only touch TMEM lanes 32*(warp%4) .. +31, so each softmax
// warpgroup covers the 128 rows of its tile exactly once.  The kernel is
// built for 168 registers per thread; warpgroup 0 then gives registers back
// (setmaxnreg 120) so each softmax thread can hold its whole 128-column S row
// (setmaxnreg 192): 120 + 2 * 192 = 3 * 168 per sub-partition.
// Tensor memory (512 columns): one S region [0,128) that the score tiles of
// Q0 and Q1 take in turn (freed as soon as the softmax has loaded it), P0
// [128,192) and P1 [192,256) (packed bf16, or four e4m3 per column for fp8
// inputs), O0 [256,384), O1 [384,512).
//
// bf16 inputs: Q0/Q1 take 3 x 16 KB each (three 64-dim 128B-swizzled K-major
// atoms); a ring of eight 16 KB chunks carries, per KV tile, K_nope[0:64],
// K_nope[64:128], K_rope, V[:, 0:64], V[:, 64:128] (V MN-major).
// fp8 inputs: Q_nope (e4m3, one 128-byte atom) and Q_rope (converted to bf16)
// take 2 x 16 KB per tile; a ring of ten 16 KB chunks carries, per KV tile,
// K_nope (e4m3), K_rope converted to bf16 as code * s_r[token] / s_k, and
// V (e4m3, MN-major).  S = s_q s_k (q_nope . k_nope [e4m3 UMMA] + q_rope .
// k_rope' [bf16 UMMA]) accumulates both parts in one fp32 tile; P is
// quantised to e4m3 after a 2^6 prescale and P.V runs as an e4m3 UMMA.
// With MLA_FP8_PRECISE (template flag SPLIT) P and K_rope' are each carried
// as a value plus the remainder of its rounding: P's remainder in the next
// 32 columns of its region with a second e4m3 P.V pass, K_rope''s in a third
// ring chunk per KV tile with four more bf16 UMMAs.
//
// Entry points: the full-context call (one window per sequence, its whole
// context), one buffer row of chunked execution (the row's window per
// sequence, optional in-place fold), and all buffer rows at once over their
// stacked K buffers (one window per sequence spanning its rows).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "host_common.h"
#include "sm103.cuh"

namespace mla {
namespace {

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per KV tile
constexpr int kQRows = 2 * kBM;   // query rows per work item
constexpr int kChunk = 16384;     // 128 rows x 128 bytes
constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;  // registers per thread the register split assumes
constexpr uint32_t kTmemCols = 512;
// Tensor-memory columns: one S region [0,128) that the score tiles of both
// query tiles take in turn, P_q [128 + 64q, +64) (packed bf16, or four e4m3
// per column), O_q [256 + 128q, +128).
constexpr uint32_t kColS = 0;
__device__ __forceinline__ uint32_t col_p(int q) { return q ? 192u : 128u; }
__device__ __forceinline__ uint32_t col_o(int q) { return q ? 384u : 256u; }
constexpr uint32_t kMaxBatch = 4096;
constexpr uint64_t kL2GroupBytes = 32ull << 20;  // K/V bytes a head group should keep in L2
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

// Layout and numerics that depend on the input type.
template <bool FP8>
struct Cfg {
  static constexpr int kQChunks = FP8 ? 2 : 3;   // 16 KB chunks per Q tile
  static constexpr int kRing = FP8 ? 10 : 8;     // 16 KB ring slots
  static constexpr int kCPT = FP8 ? 3 : 5;       // ring chunks per KV tile
  // The running max used for the exponentials moves only when a tile's max
  // exceeds it by more than this (log2 units); P <= 2^threshold.
  static constexpr float kThreshold = FP8 ? 2.0f : 8.0f;
  // fp8: P is stored as e4m3(p * 2^6) so that P <= 2^8 stays below 448.
  static constexpr float kPScale = FP8 ? 64.0f : 1.0f;
  static constexpr float kPScaleLog2 = FP8 ? 6.0f : 0.0f;  // the prescale rides in the exponent
};

struct WsHeader {
  uint32_t status;
  uint32_t counter;
  uint32_t total_items;
  uint32_t num_seqs;
  uint32_t pad[60];
};
static_assert(sizeof(WsHeader) == 256, "workspace header");

// One sequence, in scheduling order.  Its keys are the window of W context
// positions starting at co (the whole context, co = 0, for a full-context
// call; one buffer row's share for a chunked call), held at K/V rows
// kv_start .. kv_start + W - 1.  bg = b | (head group size << 16).
struct SeqRec {
  uint32_t q_start, n, prior, kv_start, bg, item_start, W, co;
};

// shift = prior - co: window key j is visible to query i when j <= shift + i.
struct ItemInfo {
  int32_t valid, b, h, q_row0, i0, n, shift, W, kv_row0, n0, n1, nkv0, nkv1, co, pad[2];
};

struct AttnParams {
  CUtensorMap tm_q;
  CUtensorMap tm_qr;          // split Q, bf16: q_rope [Tq, H, 64]
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_rope;
  CUtensorMap tm_rope_lo;     // fp8 with two K_rope' terms: the remainder copy
  uint16_t* out;
  long long out_tok, out_head;
  uint32_t out_v8;            // out rows start 32-byte aligned: the epilogue uses 32-byte stores
  float* lse;                 // chunked calls: [Tq, H] natural-log sum of exp(scores), else NULL
  long long lse_tok, lse_head;
  uint32_t accumulate;        // chunked calls: fold into out / lse of the earlier rows
  const uint32_t* page_table;
  long long pt_stride;
  const uint8_t* rope_base;
  const uint8_t* rope_base_lo;  // fp8 with two K_rope' terms: the remainder copy
  long long rope_tok_bytes, rope_page_bytes;
  uint32_t max_pages, num_pages, page_size, rope_box, rope_manual;
  uint32_t rope_contig;  // K_rope row = K row (no page table)
  // Tests of the timeout path only: the producer leaves the first K group of
  // its first work item unloaded, so the UMMA issuers' wait for it runs out.
  uint32_t test_stall;
  // Tests of the pipeline's ordering only: query tile 1's softmax waits this
  // many nanoseconds before loading each score tile, so it runs well behind
  // tile 0 (results must not change).
  uint32_t test_delay_ns;
  uint32_t H, causal;
  float sl2;
  uint8_t* ws;
  // fp8 inputs only.
  const uint8_t* q_base;
  long long q_tok, q_head;  // byte strides of q
  uint32_t Tq;
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  const float* rope_scales;  // [num_pages * page_size]
  // One K_nope scale per K row ([Sk]) instead of k_scale: the score of key
  // row t is scaled by k_tok_scales[t] in the softmax, and K_rope' (divided by
  // the same scale) is read contiguously at the K row.
  const float* k_tok_scales;
  // Split Q (q_nope and a bf16 q_rope): q_rope rows, byte strides.
  uint32_t q_split;
  const uint8_t* qr_base;
  long long qr_tok, qr_head;
};

template <bool FP8>
struct __align__(1024) Smem {
  uint8_t q[2][Cfg<FP8>::kQChunks][kChunk];
  uint8_t ring[Cfg<FP8>::kRing][kChunk];
  uint64_t item_full[2], item_empty[2];
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[Cfg<FP8>::kRing], kv_empty[Cfg<FP8>::kRing];
  uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
  // Softmax q has loaded its k-th S tile (barrier [q][k & 1], phase k >> 1):
  // the S region may be reused.  Two barriers per query tile, taken in turn,
  // because an issuer may skip one of the other tile's phases (see
  // mma_thread); with parity waits on a single barrier that skip could match
  // a phase two behind.
  uint64_t s_free[2][2];
  uint64_t pv_done[2];  // P_q . V of the previous tile has completed: P_q and O_q are free
  uint64_t drain[2];
  // Per-token K scales: the 128 scales of the KV tile each softmax warpgroup
  // is working on (filled by its threads, one key each), with barriers that
  // count the group's four warps: written, and no longer read.
  uint64_t ks_full[2], ks_free[2];
  alignas(16) float ksc[2][kBN];
  ItemInfo items[2];
  uint32_t tmem_base;
  uint32_t abort_flag;
};
// One CTA per SM: the struct, plus up to 1 KB to align it, within the 227 KB
// a CTA may use.
static_assert(sizeof(Smem<false>) + 1024 <= 232448, "shared memory (bf16)");
static_assert(sizeof(Smem<true>) + 1024 <= 232448, "shared memory (fp8)");

__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitTimeoutNs) return false;
  return true;
}

// ------------------------------------------------------------ scheduler
// One CTA: validates the ragged offsets, orders sequences longest context
// first, picks a head-group size per sequence so a group's K/V fits in L2,
// and writes the per-sequence records the attention kernel decodes work
// items from.  Work item order inside a sequence: head group, then query
// block from last (most keys) to first, then head.
constexpr int kSchedThreads = 1024;

// Chunked execution of all buffer rows in one launch (T != 0): the plan's
// arrays bro [max_rows, B+1] and cof [max_rows, B], R = min(*num_rows,
// max_rows) rows used, each row's K buffer T rows after the previous one.
struct StackedRows {
  const uint32_t* num_rows;
  uint32_t max_rows, T;
};

__device__ __forceinline__ uint32_t block_excl_scan(uint32_t x, uint32_t* warp_tot, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = x;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = warp_tot[lane];
    uint32_t ti = t;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, ti, d);
      if (lane >= d) ti += y;
    }
    warp_tot[lane] = ti - t;
    if (lane == 31) *total = ti;
  }
  __syncthreads();
  uint32_t r = warp_tot[warp] + incl - x;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kSchedThreads, 1)
schedule_kernel(const uint32_t* __restrict__ ro, const uint32_t* __restrict__ cl,
                const uint32_t* __restrict__ bro, const uint32_t* __restrict__ cof, uint32_t B,
                uint32_t H, uint32_t Tq, uint32_t Sk, uint32_t P, uint32_t max_pages,
                uint32_t kv_bytes_per_key_head, StackedRows stk, uint8_t* __restrict__ ws) {
  extern __shared__ uint32_t sm[];
  uint32_t* kv_start = sm;           // [B]
  uint32_t* key = sm + B;            // [B]  keys in the window (0 = no work)
  uint32_t* order = sm + 2 * B;      // [B]  scheduling position -> sequence
  __shared__ uint32_t warp_tot[32];
  __shared__ uint32_t total_s;
  __shared__ uint32_t status_s;
  const int tid = threadIdx.x;
  if (tid == 0) status_s = 0;
  __syncthreads();

  // Context starts: chunked exclusive scan of L_b (64-bit guarded).
  const uint32_t per = (B + kSchedThreads - 1) / kSchedThreads;
  const uint32_t b0 = min(B, tid * per), b1 = min(B, b0 + per);
  uint64_t local = 0;
  uint32_t bad = 0;
  for (uint32_t b = b0; b < b1; ++b) {
    const uint32_t lo = ro[b], hi = ro[b + 1];
    if (hi < lo || hi > Tq) bad |= MLA_DEVICE_STATUS_BAD_OFFSETS;
    local += static_cast<uint64_t>(cl[b]) + (hi >= lo ? hi - lo : 0u);
  }
  const uint32_t local32 = local > 0x7FFFFFFFull ? 0x7FFFFFFFu : static_cast<uint32_t>(local);
  uint32_t run = block_excl_scan(local32, warp_tot, &total_s);
  for (uint32_t b = b0; b < b1; ++b) {
    const uint32_t lo = ro[b], hi = ro[b + 1];
    const uint32_t n = hi >= lo ? hi - lo : 0u;
    const uint64_t L = static_cast<uint64_t>(cl[b]) + n;
    // Window: the whole context at K rows run.., or (chunked call) the
    // buffer row's W keys from context position co at rows bro[b]...
    uint64_t w0 = 0, W = L, start = run;
    bool ok = hi >= lo && hi <= Tq && L <= 0x7FFFFFFFull;
    if (stk.T) {
      // All buffer rows at once, their K buffers stacked T rows apart: the
      // sequence's context sits at plan rows r0..r1, whose windows are then
      // adjacent K rows run.. run + L - 1.  Check the first and the last of
      // those rows against the plan (global packing).
      ok = ok && static_cast<uint64_t>(run) + L <= Sk;
      if (ok && L > 0) {
        const uint32_t R = min(*stk.num_rows, stk.max_rows);
        const uint64_t g = run, T = stk.T, r0 = g / T, r1 = (g + L - 1) / T;
        ok = r1 < R;
        if (ok) {
          const uint32_t* b0r = bro + r0 * (B + 1);
          const uint32_t* b1r = bro + r1 * (B + 1);
          ok = b0r[b] == g - r0 * T && cof[r0 * B + b] == 0 && b1r[b + 1] == g + L - r1 * T &&
               cof[r1 * B + b] == (r1 == r0 ? 0 : r1 * T - g);
        }
      }
    } else if (bro) {
      const uint32_t r0 = bro[b], r1 = bro[b + 1];
      ok = ok && r0 <= r1 && r1 <= Sk;
      w0 = cof[b];
      W = r1 >= r0 ? r1 - r0 : 0u;
      start = r0;
      ok = ok && w0 + W <= L;
    } else {
      ok = ok && static_cast<uint64_t>(run) + L <= Sk;
    }
    uint32_t k = static_cast<uint32_t>(W);
    if (!ok) {
      bad |= MLA_DEVICE_STATUS_BAD_OFFSETS;
      k = 0;
    } else if ((w0 + W + P - 1) / P > max_pages) {
      bad |= MLA_DEVICE_STATUS_BAD_COLUMN;
      k = 0;
    }
    if (n == 0) k = 0;
    kv_start[b] = static_cast<uint32_t>(start);
    key[b] = k;
    run += static_cast<uint32_t>(min(L, static_cast<uint64_t>(0x7FFFFFFFu)));
  }
  if (bad) atomicOr(&status_s, bad);
  __syncthreads();

  // Longest context first (stable); identity order for very large batches.
  for (uint32_t b = tid; b < B; b += kSchedThreads) {
    uint32_t rank = b;
    if (B <= 2048) {
      rank = 0;
      const uint32_t kb = key[b];
      for (uint32_t c = 0; c < B; ++c) {
        const uint32_t kc = key[c];
        rank += (kc > kb) || (kc == kb && c < b);
      }
    }
    order[rank] = b;
  }
  __syncthreads();

  // Item counts in scheduling order, then their exclusive scan.
  uint32_t cnt_local = 0;
  for (uint32_t s = b0; s < b1; ++s) {
    const uint32_t b = order[s];
    const uint32_t n = key[b] ? ro[b + 1] - ro[b] : 0u;
    cnt_local += ((n + kQRows - 1) / kQRows) * H;
  }
  uint32_t item = block_excl_scan(cnt_local, warp_tot, &total_s);
  SeqRec* recs = reinterpret_cast<SeqRec*>(ws + sizeof(WsHeader));
  for (uint32_t s = b0; s < b1; ++s) {
    const uint32_t b = order[s];
    SeqRec r;
    r.q_start = ro[b];
    r.n = key[b] ? ro[b + 1] - ro[b] : 0u;
    r.prior = cl[b];
    r.kv_start = kv_start[b];
    r.W = key[b];
    r.co = bro && !stk.T ? cof[b] : 0u;
    const uint64_t head_bytes = static_cast<uint64_t>(key[b]) * kv_bytes_per_key_head;
    uint64_t g = head_bytes ? kL2GroupBytes / head_bytes : H;
    if (g > H) g = H;
    if (g > 0xFFFF) g = 0xFFFF;
    if (g < 1) g = 1;
    r.bg = b | (static_cast<uint32_t>(g) << 16);
    r.item_start = item;
    recs[s] = r;
    item += ((r.n + kQRows - 1) / kQRows) * H;
  }
  if (tid == 0) {
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    hdr->status = status_s;
    hdr->counter = 0;
    hdr->total_items = total_s;
    hdr->num_seqs = B;
  }
}

// ------------------------------------------------------------ attention
__device__ __forceinline__ ItemInfo decode_item(uint32_t t, const WsHeader* hdr, const SeqRec* recs,
                                                uint32_t H, uint32_t causal) {
  ItemInfo it = {};
  const uint32_t total = hdr->total_items;
  if (t >= total) return it;
  // Last sequence whose first item is <= t (sequences without items share
  // their start with the next one, so they are never selected).
  uint32_t lo = 0, hi = hdr->num_seqs;
  while (hi - lo > 1) {
    const uint32_t mid = (lo + hi) >> 1;
    if (recs[mid].item_start <= t) lo = mid; else hi = mid;
  }
  const SeqRec r = recs[lo];
  const uint32_t nqb = (r.n + kQRows - 1) / kQRows;
  const uint32_t u = t - r.item_start;
  const uint32_t G = r.bg >> 16;
  const uint32_t g = u / (nqb * G);
  const uint32_t rem = u - g * nqb * G;
  const uint32_t Gg = min(G, H - g * G);
  const uint32_t qrev = rem / Gg;
  const uint32_t hh = rem - qrev * Gg;
  const int qblk = static_cast<int>(nqb - 1 - qrev);
  it.valid = 1;
  it.b = static_cast<int>(r.bg & 0xFFFFu);
  it.h = static_cast<int>(g * G + hh);
  it.n = static_cast<int>(r.n);
  it.shift = static_cast<int>(r.prior) - static_cast<int>(r.co);
  it.W = static_cast<int>(r.W);
  it.co = static_cast<int>(r.co);
  it.i0 = qblk * kQRows;
  it.q_row0 = static_cast<int>(r.q_start) + it.i0;
  it.kv_row0 = static_cast<int>(r.kv_start);
  it.n0 = min(kBM, it.n - it.i0);
  it.n1 = max(0, min(kBM, it.n - it.i0 - kBM));
  // KV tiles up to the one holding window key `last` (none if last < 0).
  const int all_tiles = (it.W + kBN - 1) / kBN;
  auto tiles = [&](int last) { return last < 0 ? 0 : min(last / kBN + 1, all_tiles); };
  it.nkv0 = causal ? tiles(it.shift + it.i0 + it.n0 - 1) : all_tiles;
  it.nkv1 = it.n1 > 0 ? (causal ? tiles(it.shift + it.i0 + kBM + it.n1 - 1) : all_tiles) : 0;
  return it;
}

template <int R>
struct Ring {
  uint32_t full, empty, data;  // shared addresses of kv_full[0], kv_empty[0], ring[0]
  __device__ __forceinline__ uint32_t slot(uint32_t pos) const { return pos % R; }
  __device__ __forceinline__ uint32_t phase(uint32_t pos) const { return (pos / R) & 1u; }
  __device__ __forceinline__ uint32_t full_bar(uint32_t pos) const { return full + 8u * slot(pos); }
  __device__ __forceinline__ uint32_t empty_bar(uint32_t pos) const { return empty + 8u * slot(pos); }
  __device__ __forceinline__ uint32_t buf(uint32_t pos) const { return data + kChunk * slot(pos); }
};

template <bool FP8>
__device__ __forceinline__ Ring<Cfg<FP8>::kRing> make_ring(Smem<FP8>& s) {
  return Ring<Cfg<FP8>::kRing>{smem_u32(&s.kv_full[0]), smem_u32(&s.kv_empty[0]),
                               smem_u32(&s.ring[0][0])};
}

// Ring positions of one KV tile.  bf16: K_nope[0:64], K_nope[64:128], K_rope,
// then the V pair; when V[:, 0:64] would land in the last slot the tile skips
// that slot (a pad position that carries no data) so the two V chunks are
// adjacent in shared memory and one N=128 UMMA can span them.  fp8: K_nope,
// K_rope, V.
// Ring placement of one chunk group: a K group (K_nope chunks + K_rope) or a
// V group.  A bf16 V pair never straddles the ring end (one N = 128 UMMA
// spans both chunks): it skips a pad slot, passed through its barriers
// without data.  Producer and UMMA issuers place groups in the same order,
// each K group one tile ahead of V: K(0), K(1), V(0), K(2), V(1), ... (the
// issuers compute the next score tile before the current P.V).
struct GroupPos {
  uint32_t head, pad, next;  // pad == kNoPad when the group has no pad slot
};
constexpr uint32_t kNoPad = 0xFFFFFFFFu;
template <bool FP8, bool SPLIT>
__device__ __forceinline__ GroupPos place_k(uint32_t pos) {
  return {pos, kNoPad, pos + (FP8 ? (SPLIT ? 3u : 2u) : 3u)};
}
template <bool FP8>
__device__ __forceinline__ GroupPos place_v(uint32_t pos) {
  using C = Cfg<FP8>;
  if (FP8) return {pos, kNoPad, pos + 1};
  if (pos % C::kRing == C::kRing - 1) return {pos + 1, pos, pos + 3};
  return {pos, kNoPad, pos + 2};
}

// Reads the next work item from the item ring (every consumer warp reads
// every item; lane 0 releases the slot after the whole warp has read it).
template <bool FP8>
__device__ __forceinline__ bool read_item(Smem<FP8>& s, uint32_t& item_k, int lane, ItemInfo& it,
                                          volatile uint32_t* abort) {
  const uint32_t islot = item_k & 1u;
  if (!mbar_wait(smem_u32(&s.item_full[islot]), (item_k >> 1) & 1u, abort)) return false;
  it = s.items[islot];
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&s.item_empty[islot]));
  ++item_k;
  return true;
}

// Full barriers are per group, not per chunk: every TMA box of a tile's K
// chunks (and of its V pair) signals the full barrier of the group's first
// slot with one expect_tx for the summed bytes, so the UMMA thread waits once
// per group.  A slot's full barrier therefore completes a phase only when the
// slot heads a group; both sides keep one phase bit per slot.  Empty barriers
// stay per chunk (one UMMA commit each).
// One lane's page-table read for a K_rope box: state 0 = no box, 1 = page
// read, 2 = page-table column out of range.
struct RopeFetch {
  uint32_t page, row, state;
};

template <bool FP8, bool SPLIT>
__device__ void producer_warp(Smem<FP8>& s, const AttnParams& p, int lane, volatile uint32_t* abort) {
  using C = Cfg<FP8>;
  WsHeader* hdr = reinterpret_cast<WsHeader*>(p.ws);
  const SeqRec* recs = reinterpret_cast<const SeqRec*>(p.ws + sizeof(WsHeader));
  const auto ring = make_ring(s);
  uint32_t pos = 0, item_k = 0, q_uses[2] = {0, 0};
  uint32_t status = 0;
  uint32_t fph = 0;                  // full-barrier phase bit per slot (flipped per head use)
  uint32_t recent[C::kRing] = {};    // last group heads issued, for the abort drain
  uint32_t nrecent = 0;
  bool alive = true;

  auto acquire = [&](uint32_t ps) -> bool {
    return mbar_wait(ring.empty_bar(ps), ring.phase(ps) ^ 1u, abort);
  };
  auto note_head = [&](uint32_t head) {
    recent[nrecent % C::kRing] = (ring.slot(head) << 1) | ((fph >> ring.slot(head)) & 1u);
    ++nrecent;
    fph ^= 1u << ring.slot(head);
  };
  // TMA of 128 rows (one 16 KB chunk) of k_nope or v into slot `ps`, signalling `bar`.
  auto tma_chunk = [&](const CUtensorMap* map, int x, const ItemInfo& it, int j, uint32_t ps, uint32_t bar) {
    tma_load_3d(ring.buf(ps), map, bar, x, it.h, it.kv_row0 + j * kBN);
  };
  // bf16 K_rope rows into slot `ps`: TMA boxes (one per page segment, lane t
  // owns box t) when page segments are 8-row aligned, else a swizzled row
  // gather.  Window key `key` is context position co + key.  The page-table
  // reads for a tile's boxes are issued one tile ahead (rope_fetch) and only
  // checked when the boxes go out, so their latency hides behind the ring
  // waits in between.
  auto rope_fetch = [&](const ItemInfo& it, int j) -> RopeFetch {
    RopeFetch f = {0u, 0u, 0u};
    const int nbox = kBN / static_cast<int>(p.rope_box);
    if (lane < nbox) {
      const int key = j * kBN + lane * static_cast<int>(p.rope_box);
      if (key < it.W) {
        const uint32_t a = static_cast<uint32_t>(it.co + key);
        const uint32_t col = a / p.page_size;
        f.row = a - col * p.page_size;
        if (col >= p.max_pages) {
          f.state = 2;
        } else {
          f.page = p.page_table[static_cast<long long>(it.b) * p.pt_stride + col];
          f.state = 1;
        }
      }
    }
    return f;
  };
  auto rope_gather = [&](const ItemInfo& it, int j, uint32_t ps, const uint8_t* rope_base) {
    const uint32_t dst = ring.buf(ps);
    for (int r = lane; r < kBN; r += 32) {
      const int key = j * kBN + r;
      if (key >= it.W) continue;
      const uint32_t a = static_cast<uint32_t>(it.co + key);
      const uint32_t col = a / p.page_size;
      if (col >= p.max_pages) { status |= MLA_DEVICE_STATUS_BAD_COLUMN; continue; }
      const uint32_t page = p.page_table[static_cast<long long>(it.b) * p.pt_stride + col];
      if (page >= p.num_pages) { status |= MLA_DEVICE_STATUS_BAD_PAGE; continue; }
      const uint4* src = reinterpret_cast<const uint4*>(
          rope_base + page * p.rope_page_bytes +
          static_cast<long long>(a - col * p.page_size) * p.rope_tok_bytes);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = src[c];
        const uint32_t a = dst + r * 128 + ((c ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
  };
  // The K group of tile j: K_nope chunks (bf16: [0:64] and [64:128] at k,
  // k+1; fp8: one 128-code chunk at k), then the bf16 K_rope chunk (for fp8
  // inputs read from the converted copy of the pool; with two K_rope' terms
  // the remainder chunk follows it).
  auto load_k_group = [&](const ItemInfo& it, int j, uint32_t k, bool boxes, const RopeFetch& rf) -> bool {
    constexpr int kNope = FP8 ? 1 : 2;
    constexpr int kRope = SPLIT ? 2 : 1;
    const uint32_t bar = ring.full_bar(k);
    const uint32_t kr = k + kNope;  // K_rope slot
    for (int c = 0; c < kNope + kRope; ++c)
      if (!acquire(k + c)) return false;
    if (p.rope_contig) {
      // Contiguous K_rope: the tile's 128 rows sit at its K rows.
      if (lane == 0) {
        mbar_arrive_expect_tx(bar, (kNope + kRope) * kChunk);
        for (int c = 0; c < kNope; ++c) tma_chunk(&p.tm_k, 64 * c, it, j, k + c, bar);
        tma_load_2d(ring.buf(kr), &p.tm_rope, bar, 0, it.kv_row0 + j * kBN);
        if (SPLIT) tma_load_2d(ring.buf(kr + 1), &p.tm_rope_lo, bar, 0, it.kv_row0 + j * kBN);
      }
      __syncwarp();
    } else if (boxes) {
      bool issue = false;
      if (rf.state == 2) status |= MLA_DEVICE_STATUS_BAD_COLUMN;
      else if (rf.state == 1 && rf.page >= p.num_pages) status |= MLA_DEVICE_STATUS_BAD_PAGE;
      else issue = rf.state == 1;
      const uint32_t mask = __ballot_sync(0xffffffffu, issue);
      const uint32_t bytes = kNope * kChunk + kRope * __popc(mask) * p.rope_box * 128u;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar, bytes);
        for (int c = 0; c < kNope; ++c) tma_chunk(&p.tm_k, 64 * c, it, j, k + c, bar);
      }
      __syncwarp();
      if (issue) {
        tma_load_3d(ring.buf(kr) + lane * p.rope_box * 128u, &p.tm_rope, bar, 0,
                    static_cast<int>(rf.row), static_cast<int>(rf.page));
        if (SPLIT)
          tma_load_3d(ring.buf(kr + 1) + lane * p.rope_box * 128u, &p.tm_rope_lo, bar, 0,
                      static_cast<int>(rf.row), static_cast<int>(rf.page));
      }
    } else {
      rope_gather(it, j, kr, p.rope_base);
      if (SPLIT) rope_gather(it, j, kr + 1, p.rope_base_lo);
      if (lane == 0) {
        mbar_arrive_expect_tx(bar, kNope * kChunk);
        for (int c = 0; c < kNope; ++c) tma_chunk(&p.tm_k, 64 * c, it, j, k + c, bar);
      }
    }
    note_head(k);
    return true;
  };
  // The V group of tile j: bf16 V[:, 0:64], V[:, 64:128] at v, v+1; fp8 V at v.
  auto load_v_group = [&](const ItemInfo& it, int j, uint32_t v) -> bool {
    const uint32_t bar = ring.full_bar(v);
    if (!acquire(v) || (!FP8 && !acquire(v + 1))) return false;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar, (FP8 ? 1 : 2) * kChunk);
      tma_chunk(&p.tm_v, 0, it, j, v, bar);
      if (!FP8) tma_chunk(&p.tm_v, 64, it, j, v + 1, bar);
    }
    note_head(v);
    return true;
  };
  // bf16: the whole 192-wide Q tile (three 64-dim atoms).  fp8: the 128
  // nope codes only; the converter warp writes the rope part.
  auto load_q = [&](int q, const ItemInfo& it) -> bool {
    const uint32_t bar = smem_u32(&s.q_full[q]);
    if (!mbar_wait(smem_u32(&s.q_empty[q]), (q_uses[q] & 1u) ^ 1u, abort)) return false;
    ++q_uses[q];
    if (lane == 0) {
      mbar_arrive_expect_tx(bar, (FP8 ? 1 : 3) * kChunk);
      for (int a = 0; a < (FP8 ? 1 : 3); ++a) {
        // Split bf16 Q: the rope atom comes from q_rope.
        const bool rope_map = !FP8 && a == 2 && p.q_split;
        tma_load_3d(smem_u32(&s.q[q][a][0]), rope_map ? &p.tm_qr : &p.tm_q, bar, rope_map ? 0 : 64 * a, it.h,
                    it.q_row0 + q * kBM);
      }
    }
    return true;
  };

  // The next item is claimed two KV tiles before the end of the current one,
  // so the counter's round trip overlaps the last loads; lane 0 holds the
  // claimed index until the item starts.
  uint32_t t_claim = 0;
  bool claimed = false;
  while (alive) {
    if (!claimed && lane == 0) t_claim = atomicAdd(&hdr->counter, 1u);
    claimed = false;
    const uint32_t t = __shfl_sync(0xffffffffu, t_claim, 0);
    const ItemInfo it = decode_item(t, hdr, recs, p.H, p.causal);
    const uint32_t islot = item_k & 1u;
    if (!mbar_wait(smem_u32(&s.item_empty[islot]), ((item_k >> 1) & 1u) ^ 1u, abort)) break;
    if (lane == 0) {
      s.items[islot] = it;
      mbar_arrive(smem_u32(&s.item_full[islot]));
    }
    ++item_k;
    if (!it.valid) break;
    const int nkv = it.n1 > 0 ? it.nkv1 : it.nkv0;
    // K_rope by one TMA box per page segment, unless the rows are contiguous
    // or the segments are not 8-row aligned (pages, or a window that starts
    // inside a segment): then the row gather.
    const bool boxes = !p.rope_contig && !p.rope_manual && it.co % static_cast<int>(p.rope_box) == 0;
    RopeFetch rf = {0u, 0u, 0u};
    if (boxes && nkv > 0) rf = rope_fetch(it, 0);
    auto k_group = [&](int j) -> bool {
      const GroupPos g = place_k<FP8, SPLIT>(pos);
      pos = g.next;
      if (p.test_stall && item_k == 1 && j == 0) return true;  // nothing arms this group's barrier
      const bool ok = load_k_group(it, j, g.head, boxes, rf);
      if (boxes && j + 1 < nkv) rf = rope_fetch(it, j + 1);
      return ok;
    };
    auto v_group = [&](int j) -> bool {
      const GroupPos g = place_v<FP8>(pos);
      pos = g.next;
      if (g.pad != kNoPad) {  // pad slot: keeps the V pair adjacent
        if (!acquire(g.pad)) return false;
        if (lane == 0) mbar_arrive(ring.full_bar(g.pad));
        note_head(g.pad);
      }
      return load_v_group(it, j, g.head);
    };
    if (nkv > 0) {
      // Q first: its buffers free up as soon as the previous item's last
      // score tiles are issued, while the K group's ring slots come free only
      // after that item's last P.V; issued after K, the Q copy's latency would
      // fall between the items.  A query tile that sees no key of the window
      // is not loaded.
      alive = (it.nkv0 == 0 || load_q(0, it)) && (it.nkv1 == 0 || load_q(1, it));
      if (alive) alive = k_group(0);
    }
    for (int j = 0; j < nkv && alive; ++j) {
      if (j + 2 == nkv) {
        if (lane == 0) t_claim = atomicAdd(&hdr->counter, 1u);
        claimed = true;
      }
      if (j + 1 < nkv) alive = k_group(j + 1);
      alive = alive && v_group(j);
    }
  }
  if (status) atomicOr(&hdr->status, status);
  if (*abort) {
    // Let every copy this warp started land before the CTA exits.
    const uint32_t n = nrecent < C::kRing ? nrecent : C::kRing;
    for (uint32_t i = 0; i < n; ++i) {
      const uint32_t e = recent[(nrecent - 1 - i) % C::kRing];
      wait_drain(ring.full + 8u * (e >> 1), e & 1u);
    }
    for (int q = 0; q < 2; ++q)
      if (q_uses[q]) wait_drain(smem_u32(&s.q_full[q]), (q_uses[q] - 1) & 1u);
  }
}

// fp8 inputs: warp 3 turns each query tile's 64 rope codes per row into
// bf16 (exact), 128B-swizzled, so q_rope . k_rope' runs as a bf16 UMMA next to
// the e4m3 nope UMMA.  Each lane owns four of the 128 rows; the warp signals
// q_full once its rows are written.  (K_rope' = code * s_r[token] / s_k is
// converted once per call by rope_convert_kernel.)
__device__ __forceinline__ void store_bf16_row(uint32_t dst, int r, const float (&f)[64]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t a = dst + r * 128 + ((c ^ (r & 7)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                 "r"(pack_bf16x2(f[8 * c], f[8 * c + 1])), "r"(pack_bf16x2(f[8 * c + 2], f[8 * c + 3])),
                 "r"(pack_bf16x2(f[8 * c + 4], f[8 * c + 5])), "r"(pack_bf16x2(f[8 * c + 6], f[8 * c + 7]))
                 : "memory");
  }
}
__device__ __forceinline__ void load_e4m3_row(const uint8_t* src, float scale, float (&f)[64]) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v = s4[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float a, b, cc, d;
      e4m3x4_to_f32(w[e], a, b, cc, d);
      f[16 * c + 4 * e] = a * scale;
      f[16 * c + 4 * e + 1] = b * scale;
      f[16 * c + 4 * e + 2] = cc * scale;
      f[16 * c + 4 * e + 3] = d * scale;
    }
  }
}

__device__ __forceinline__ void load_bf16_row(const uint8_t* src, float scale, float (&f)[64]) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 v = s4[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[8 * c + 2 * e] = __uint_as_float(w[e] << 16) * scale;
      f[8 * c + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u) * scale;
    }
  }
}

__device__ void converter_warp(Smem<true>& s, const AttnParams& p, int lane, volatile uint32_t* abort) {
  uint32_t item_k = 0, q_uses[2] = {0, 0};
  const float inv_sq = p.q_split ? 1.f / *p.q_scale : 1.f;
  bool alive = true;
  auto conv_q = [&](int q, const ItemInfo& it) -> bool {
    if (!mbar_wait(smem_u32(&s.q_empty[q]), (q_uses[q] & 1u) ^ 1u, abort)) return false;
    ++q_uses[q];
    const uint32_t dst = smem_u32(&s.q[q][1][0]);
    for (int r = lane; r < kBM; r += 32) {
      const int row = it.q_row0 + q * kBM + r;
      float f[64];
      if (row < static_cast<int>(p.Tq) && p.q_split) {
        // bf16 q_rope in true units, to the units of the e4m3 codes (1 / s_q).
        load_bf16_row(p.qr_base + row * p.qr_tok + it.h * p.qr_head, inv_sq, f);
      } else if (row < static_cast<int>(p.Tq)) {
        load_e4m3_row(p.q_base + row * p.q_tok + it.h * p.q_head + 128, 1.f, f);
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) f[e] = 0.f;
      }
      store_bf16_row(dst, r, f);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s.q_full[q]));
    return true;
  };
  while (alive) {
    ItemInfo it;
    if (!read_item(s, item_k, lane, it, abort) || !it.valid) break;
    alive = (it.nkv0 == 0 || conv_q(0, it)) && (it.nkv1 == 0 || conv_q(1, it));
  }
}

// 64 values as a bf16 row at hi and, when lo != NULL, the remainder of that
// rounding as a second bf16 row at lo (hi + lo carries about 16 significant
// bits).
__device__ __forceinline__ void store_bf16_terms(const float (&f)[64], uint16_t* hi, uint16_t* lo) {
  uint32_t w[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) w[e] = pack_bf16x2(f[2 * e], f[2 * e + 1]);
  uint4* dh = reinterpret_cast<uint4*>(hi);
#pragma unroll
  for (int c = 0; c < 8; ++c) dh[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  if (!lo) return;
  uint4* dl = reinterpret_cast<uint4*>(lo);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t r[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t h = w[4 * c + e];
      const float h0 = __uint_as_float(h << 16), h1 = __uint_as_float(h & 0xFFFF0000u);
      r[e] = pack_bf16x2(f[8 * c + 2 * e] - h0, f[8 * c + 2 * e + 1] - h1);
    }
    dl[c] = make_uint4(r[0], r[1], r[2], r[3]);
  }
}

// fp8 inputs, once per call: K_rope' = e4m3 code * s_r[slot] / s_k in bf16 for
// every pool slot, into the workspace ([num_pages * P] rows of 64 bf16, 128
// bytes each).  The attention kernel then streams it like bf16 K_rope.
__global__ void __launch_bounds__(256) rope_convert_kernel(const uint8_t* __restrict__ pool,
                                                           long long tok_bytes, long long page_bytes,
                                                           uint32_t P, uint32_t slots,
                                                           const float* __restrict__ scales,
                                                           const float* __restrict__ k_scale,
                                                           uint16_t* __restrict__ out, uint16_t* __restrict__ out_lo) {
  const float inv_sk = 1.f / *k_scale;
  for (uint32_t sl = blockIdx.x * blockDim.x + threadIdx.x; sl < slots; sl += gridDim.x * blockDim.x) {
    const uint32_t page = sl / P, row = sl - page * P;
    float f[64];
    load_e4m3_row(pool + page * page_bytes + row * tok_bytes, scales[sl] * inv_sk, f);
    store_bf16_terms(f, out + static_cast<size_t>(sl) * 64, out_lo ? out_lo + static_cast<size_t>(sl) * 64 : nullptr);
  }
}

// fp8 inputs with one K_nope scale per K row: K_rope' = e4m3 code * s_r[slot]
// / s_k[row] for every key row of every sequence's window, written at the K
// row (a contiguous [Sk, 64] bf16 copy, so the attention kernel reads it like
// a contiguous K_rope).  It runs after the scheduler: the records give each
// window's K rows, its context offset and its sequence.  Block (x, y) takes
// records x, x + gridDim.x, ... and, inside each, every gridDim.y-th group of
// blockDim.x keys.
struct RopeRows {
  const uint8_t* pool;            // e4m3 K_rope rows
  long long tok_bytes, page_bytes;
  const uint32_t* page_table;     // NULL: contiguous K_rope, row = K row
  long long pt_stride;
  uint32_t P, num_pages, max_pages, Sk;
  const float* rope_scales;       // [num_pages * P] (contiguous: [Sk])
  const float* k_scales;          // [Sk]
  uint16_t* out;                  // [Sk, 64] bf16
  uint16_t* out_lo;               // NULL, or the remainder term [Sk, 64] bf16
  uint8_t* ws;
};

__global__ void __launch_bounds__(256) rope_convert_rows_kernel(const __grid_constant__ RopeRows a) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
  const SeqRec* recs = reinterpret_cast<const SeqRec*>(a.ws + sizeof(WsHeader));
  const uint32_t nseq = hdr->num_seqs;
  uint32_t bad = 0;
  for (uint32_t si = blockIdx.x; si < nseq; si += gridDim.x) {
    const SeqRec rec = recs[si];
    const uint32_t b = rec.bg & 0xFFFFu;
    for (uint32_t j = blockIdx.y * blockDim.x + threadIdx.x; j < rec.W; j += gridDim.y * blockDim.x) {
      const uint32_t row = rec.kv_start + j;
      if (row >= a.Sk) break;
      uint32_t page = row, prow = 0;  // contiguous: a one-row page per K row
      if (a.page_table) {
        const uint32_t pos = rec.co + j;  // context position of the key
        const uint32_t col = pos / a.P;
        uint32_t pg = 0xFFFFFFFFu;
        if (col < a.max_pages) pg = a.page_table[static_cast<long long>(b) * a.pt_stride + col];
        else bad |= MLA_DEVICE_STATUS_BAD_COLUMN;
        if (pg >= a.num_pages) {
          if (col < a.max_pages) bad |= MLA_DEVICE_STATUS_BAD_PAGE;
          float z[64];
#pragma unroll
          for (int c = 0; c < 64; ++c) z[c] = 0.f;
          store_bf16_terms(z, a.out + static_cast<size_t>(row) * 64,
                           a.out_lo ? a.out_lo + static_cast<size_t>(row) * 64 : nullptr);
          continue;
        }
        page = pg;
        prow = pos - col * a.P;
      }
      const long long slot = static_cast<long long>(page) * a.P + prow;
      float f[64];
      load_e4m3_row(a.pool + page * a.page_bytes + prow * a.tok_bytes, a.rope_scales[slot] / a.k_scales[row], f);
      store_bf16_terms(f, a.out + static_cast<size_t>(row) * 64,
                       a.out_lo ? a.out_lo + static_cast<size_t>(row) * 64 : nullptr);
    }
  }
  if (bad) atomicOr(&hdr->status, bad);
}

// UMMA issue for one query tile.  Warps 1 and 2 each run this for their own
// tile (q = 0, 1): a thread blocked on a barrier wait then no longer holds up
// the other tile's UMMAs.  Both threads walk the same ring and release every
// chunk (empty barriers count two); a thread with no work on a KV tile still
// waits for the tile's groups before releasing them, so no barrier phase can
// be released ahead of its fill.  Per KV tile j a thread issues S_q(j+1) as
// soon as the S region is free (the softmax of the score tile before it has
// loaded it into registers) and then P_q(j) . V(j) once P_q(j) is stored, so
// the next score tile is computed while the softmax works on this one.
template <bool FP8, bool SPLIT>
__device__ void mma_thread(Smem<FP8>& s, uint32_t tmem, int q, volatile uint32_t* abort) {
  using C = Cfg<FP8>;
  const auto ring = make_ring(s);
  // Instruction descriptors (fp32 accumulate): bf16 A/B (format 1) or e4m3 (format 0).
  const uint32_t idS = make_idesc(128, 128, 1, false);     // bf16 S (whole S, or fp8's rope part)
  const uint32_t idS8 = make_idesc(128, 128, 0, false);    // fp8 nope part of S
  const uint32_t idPV = make_idesc(128, 128, 1, true);     // bf16 P.V, N = 128 over the V pair
  const uint32_t idPV8 = make_idesc(128, 128, 0, true);    // fp8 P.V, N = 128
  const uint64_t qd = sw128_desc_at(smem_u32(&s.q[q][0][0]));
  const uint32_t d_s = tmem + kColS, d_p = tmem + col_p(q), d_o = tmem + col_o(q);
  uint32_t pos = 0, item_k = 0, qf = 0, pf = 0, oe = 0;
  // The S region serves the score tiles in the order S0(0), S1(0), S0(1),
  // S1(1), ... over all items.  Both issuers count them: rbase[t] = S tiles of
  // query tile t in earlier items, rlast = query tile of the last one.
  uint32_t rbase[2] = {0u, 0u};
  int rlast = -1;
  bool alive = true;

  uint32_t fph = 0;  // full-barrier phase bit per slot, flipped at each use as a group head
  auto wait_group = [&](uint32_t head) -> bool {
    const uint32_t sl = ring.slot(head);
    if (!mbar_wait(ring.full_bar(head), (fph >> sl) & 1u, abort)) return false;
    fph ^= 1u << sl;
    tc_fence_after();
    return true;
  };
  // S_q = Q_q . [K_nope | K_rope]^T.  bf16: each K chunk's empty barrier is
  // committed right after the UMMAs that read it, so the producer can refill
  // a slot while the rest of the score tile is still being computed (the
  // eight-slot bf16 ring is short of room for the copies in flight; the fp8
  // ring is not, and there the extra commits cost more than they return).
  auto issue_s = [&](uint32_t kpos) {
    if (FP8) {
      // 4 e4m3 K-steps of 32 over the nope atom, then 4 bf16 K-steps of 16 over rope.
      const uint64_t kd = sw128_desc_at(ring.buf(kpos)), rd = sw128_desc_at(ring.buf(kpos + 1));
#pragma unroll
      for (int k = 0; k < 4; ++k) umma_f8_ss(d_s, qd + 2 * k, kd + 2 * k, idS8, k != 0);
#pragma unroll
      for (int k = 0; k < 4; ++k) umma_f16_ss(d_s, qd + (kChunk >> 4) + 2 * k, rd + 2 * k, idS, 1);
      if (SPLIT) {
        // The remainder term of K_rope' (its bf16 rounding), same Q rope atom.
        const uint64_t rl = sw128_desc_at(ring.buf(kpos + 2));
#pragma unroll
        for (int k = 0; k < 4; ++k) umma_f16_ss(d_s, qd + (kChunk >> 4) + 2 * k, rl + 2 * k, idS, 1);
      }
    } else {
      // 3 swizzle atoms x 4 K-steps of 16.
#pragma unroll
      for (int a = 0; a < 3; ++a) {
        const uint64_t kd = sw128_desc_at(ring.buf(kpos + a));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_f16_ss(d_s, qd + a * (kChunk >> 4) + 2 * k, kd + 2 * k, idS, (a | k) != 0);
        umma_commit(ring.empty_bar(kpos + a));
      }
    }
    umma_commit(smem_u32(&s.s_full[q]));
  };
  // O_q (+)= P_q . V, P from TMEM.
  auto issue_pv = [&](uint32_t vpos, bool acc) {
    const uint32_t acc0 = acc ? 1u : 0u;
    if (FP8) {
      // 4 K-steps of 32 keys; P holds four e4m3 per column, V is one MN-major atom.
      const uint64_t v0 = sw128_desc_at(ring.buf(vpos));
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_f8_ts(d_o, d_p + ks * 8, v0 + ks * (4096 >> 4), idPV8, ks ? 1u : acc0);
      if (SPLIT) {
        // The second e4m3 term of P (the remainder of its rounding), in the
        // next 32 columns of the P region, into the same accumulator.
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) umma_f8_ts(d_o, d_p + 32 + ks * 8, v0 + ks * (4096 >> 4), idPV8, 1u);
      }
    } else {
      // 8 K-steps of 16 keys, N = 128: the two V chunks sit in adjacent slots,
      // 16 KB apart (the leading byte offset between the two 64-column atoms).
      const uint64_t v0 = sw128_desc(ring.buf(vpos), kChunk, 1024);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_f16_ts(d_o, d_p + ks * 8, v0 + ks * (2048 >> 4), idPV, ks ? 1u : acc0);
    }
  };
  auto release = [&](uint32_t first, int count) {
    for (int c = 0; c < count; ++c) umma_commit(ring.empty_bar(first + c));
  };
  auto wait_p = [&](bool first_tile) -> bool {
    if (!mbar_wait(smem_u32(&s.p_full[q]), pf & 1u, abort)) return false;
    ++pf;
    if (first_tile) {
      if (!mbar_wait(smem_u32(&s.o_empty[q]), (oe & 1u) ^ 1u, abort)) return false;
      ++oe;
    }
    tc_fence_after();
    return true;
  };
  constexpr int kK = FP8 ? (SPLIT ? 3 : 2) : 3;  // K chunks per tile (ring order: K chunks, then V chunks)
  constexpr int kV = FP8 ? 1 : 2;

  // Wait until the k-th S tile of query tile t has been loaded by its softmax.
  // The waits of one issuer on tile t's loads are not always consecutive: at
  // the end of a causal item query tile 1 usually has one more KV tile than
  // tile 0, so its last two score tiles follow each other in the S region,
  // and the next item's S0(0) waits for the second of them although issuer 0
  // never waited for the first.  The other tile's load count is then one or
  // two ahead of issuer 0's last wait; barrier [t][k & 1] with phase k >> 1
  // tells those cases apart, where one barrier's parity would not.
  auto wait_region = [&](int t, uint32_t k) -> bool {
    if (t < 0) return true;
    if (!mbar_wait(smem_u32(&s.s_free[t][k & 1u]), (k >> 1) & 1u, abort)) return false;
    tc_fence_after();
    return true;
  };

  while (alive) {
    const uint32_t islot = item_k & 1u;
    if (!mbar_wait(smem_u32(&s.item_full[islot]), (item_k >> 1) & 1u, abort)) break;
    const ItemInfo it = s.items[islot];
    mbar_arrive(smem_u32(&s.item_empty[islot]));
    ++item_k;
    if (!it.valid) break;
    const int nkv = it.n1 > 0 ? it.nkv1 : it.nkv0;   // KV tiles the item streams
    if (nkv == 0) continue;                           // no query of the item sees a key
    const int m0 = it.nkv0, m1 = it.n1 > 0 ? it.nkv1 : 0;  // tiles of each query tile (m1 >= m0 if m1 > 0)
    const int mine = q ? m1 : m0;
    // Query tile t and global index k of the score tile that precedes S_q(j)
    // in the S region.
    auto pred = [&](int j, int& t, uint32_t& k) {
      if (q == 0) {
        if (j == 0) { t = rlast; k = t >= 0 ? rbase[t] - 1u : 0u; }
        else if (j - 1 < m1) { t = 1; k = rbase[1] + j - 1; }
        else { t = 0; k = rbase[0] + j - 1; }
      } else {
        if (j < m0) { t = 0; k = rbase[0] + j; }
        else if (j == 0) { t = rlast; k = t >= 0 ? rbase[t] - 1u : 0u; }
        else { t = 1; k = rbase[1] + j - 1; }
      }
    };
    // S_q(j) into the S region once the previous score tile there has been
    // loaded; a tile this query tile does not use only passes its K group back.
    auto do_s = [&](int j) -> bool {
      const GroupPos g = place_k<FP8, SPLIT>(pos);
      pos = g.next;
      if (!wait_group(g.head)) return false;
      if (j < mine) {
        if (j == 0) {
          if (!mbar_wait(smem_u32(&s.q_full[q]), qf & 1u, abort)) return false;
          ++qf;
          tc_fence_after();
        }
        int t;       // query tile and index of the previous S tile in the region
        uint32_t k;
        pred(j, t, k);
        if (!wait_region(t, k)) return false;
        issue_s(g.head);  // bf16: releases the group's chunks
        if (j + 1 == mine) umma_commit(smem_u32(&s.q_empty[q]));  // Q_q no longer read
        if (FP8) release(g.head, kK);
      } else {
        release(g.head, kK);
      }
      return true;
    };
    // O_q (+)= P_q(j) . V(j) once the softmax has stored P_q(j).
    auto do_pv = [&](int j) -> bool {
      const GroupPos g = place_v<FP8>(pos);
      pos = g.next;
      if (g.pad != kNoPad) {  // pass the empty pad slot straight back
        if (!wait_group(g.pad)) return false;
        release(g.pad, 1);
      }
      if (!wait_group(g.head)) return false;
      if (j < mine) {
        if (!wait_p(j == 0)) return false;
        issue_pv(g.head, j > 0);
        umma_commit(smem_u32(&s.pv_done[q]));
        if (j + 1 == mine) umma_commit(smem_u32(&s.o_full[q]));
      }
      release(g.head, kV);
      return true;
    };
    // S_q(j+1) goes ahead of P_q(j) . V(j), so the next score tile is
    // ready when the softmax finishes this one.
    alive = do_s(0);
    for (int j = 0; j < nkv && alive; ++j) {
      if (j + 1 < nkv) alive = do_s(j + 1);
      alive = alive && do_pv(j);
    }
    rbase[0] += static_cast<uint32_t>(m0);
    rbase[1] += static_cast<uint32_t>(m1);
    if (m1 > 0) rlast = 1;
    else if (m0 > 0) rlast = 0;
  }
  // Make sure no UMMA is still in flight before tensor memory is released.
  umma_commit(smem_u32(&s.drain[q]));
  wait_drain(smem_u32(&s.drain[q]), 0);
}

template <bool FP8, bool KTOK, bool SPLIT>
__device__ void softmax_warp(Smem<FP8>& s, const AttnParams& p, uint32_t tmem, int q, int wq,
                             int lane, volatile uint32_t* abort) {
  using C = Cfg<FP8>;
  const int r = wq * 32 + lane;  // query row inside the tile == TMEM lane
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t t_s = tmem + lane_off + kColS;
  const uint32_t t_p = tmem + lane_off + col_p(q);
  const uint32_t t_o = tmem + lane_off + col_o(q);
  // fp8: S in TMEM is in units of s_q * s_k (per-token K scales: s_q * s_k[key],
  // the key's factor applied per column below); P, O and the row sum l carry
  // the kPScale prescale (folded into the exponent), so O / l needs only s_v.
  // Clamped away from 0 (a zero scale) so that a masked -inf score stays -inf
  // after the scaling FMA; any real scale is far above the clamp.
  const float sl2 = fmaxf(FP8 ? p.sl2 * (*p.q_scale) * (KTOK ? 1.f : *p.k_scale) : p.sl2, 1e-30f);
  const float out_scale = FP8 ? *p.v_scale : 1.f;
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  uint32_t item_k = 0, sf = 0, of = 0;
  uint32_t pvc = 0;  // tiles of this query tile so far (= P.V launches that follow them)
  uint32_t kt = 0;   // KV tiles whose key scales this warpgroup has staged
  const uint32_t ks_full = smem_u32(&s.ks_full[q]), ks_free = smem_u32(&s.ks_free[q]);
  const uint32_t ks_row = smem_u32(&s.ksc[q][0]);
  // Scale of window key j * kBN + r (1 past the window: those keys are masked).
  auto key_scale = [&](const ItemInfo& it, int j) -> float {
    const int key = j * kBN + r;
    return key < it.W ? __ldg(p.k_tok_scales + it.kv_row0 + key) : 1.f;
  };

  for (;;) {
    ItemInfo it;
    if (!read_item(s, item_k, lane, it, abort) || !it.valid) return;
    if (q == 1 && it.n1 == 0) continue;
    const int nkv = q ? it.nkv1 : it.nkv0;
    const int i = it.i0 + q * kBM + r;  // query index inside the sequence
    if (nkv == 0) {
      // Chunked call, no query of this tile sees a key of the window.  A
      // folding call leaves the earlier rows' result as it is.
      if (i < it.n && !(p.accumulate && it.co > 0)) {
        const long long row = it.q_row0 + q * kBM + r;
        uint4* dst = reinterpret_cast<uint4*>(p.out + row * p.out_tok + static_cast<long long>(it.h) * p.out_head);
#pragma unroll
        for (int c = 0; c < 16; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
        if (p.lse) p.lse[row * p.lse_tok + static_cast<long long>(it.h) * p.lse_head] = -INFINITY;
      }
      continue;
    }
    const int last_key = it.W - 1;
    const int limit = p.causal ? min(it.shift + i, last_key) : last_key;
    const int tile_limit = p.causal ? min(it.shift + it.i0 + q * kBM, last_key) : last_key;
    float m_used = -INFINITY, l = 0.f;
    float ks_next = KTOK ? key_scale(it, 0) : 1.f;  // this thread's key scale for the next tile

    for (int j = 0; j < nkv; ++j) {
      if (KTOK) {
        // Stage tile j's 128 key scales (thread r holds key r's) once every
        // warp of the group has finished reading tile j-1's; the load for
        // tile j+1 is issued here and consumed a tile later.
        if (kt > 0 && !mbar_wait(ks_free, (kt - 1) & 1u, abort)) return;
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(ks_row + 4u * r), "f"(ks_next * sl2) : "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(ks_full);
        if (!mbar_wait(ks_full, kt & 1u, abort)) return;
        if (j + 1 < nkv) ks_next = key_scale(it, j + 1);
      }
      if (!mbar_wait(smem_u32(&s.s_full[q]), sf & 1u, abort)) return;
      if (q == 1 && p.test_delay_ns) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < p.test_delay_ns) {
        }
      }
      ++sf;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(t_s + 32 * c, sr[c]);
      tmem_ld_wait();
      // The S region is free for the next score tile.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s.s_free[q][(sf - 1) & 1u]));
      // Exponent reference so far (0 before the first visible key).
      float mb = m_used == -INFINITY ? 0.f : m_used;
      if (KTOK) {
        // Per-token K scales: column c's factor sl2 * s_k[key] (a broadcast
        // read: every lane reads the same four) goes into the one FMA that
        // also subtracts the current reference, y = S * factor + 6 - mb; the
        // max below is then taken over y.
        const uint64_t off = f2_pack(C::kPScaleLog2 - mb, C::kPScaleLog2 - mb);
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float k0, k1, k2, k3;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(k0), "=f"(k1), "=f"(k2), "=f"(k3)
                         : "r"(ks_row + 4u * (32 * c + 4 * k)));
            float x0, x1, x2, x3;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c][4 * k]), __uint_as_float(sr[c][4 * k + 1])),
                             f2_pack(k0, k1), off), x0, x1);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c][4 * k + 2]), __uint_as_float(sr[c][4 * k + 3])),
                             f2_pack(k2, k3), off), x2, x3);
            sr[c][4 * k] = __float_as_uint(x0);
            sr[c][4 * k + 1] = __float_as_uint(x1);
            sr[c][4 * k + 2] = __float_as_uint(x2);
            sr[c][4 * k + 3] = __float_as_uint(x3);
          }
        __syncwarp();
        if (lane == 0) mbar_arrive(ks_free);
        ++kt;
      }
      const int key0 = j * kBN;
      const bool masked = key0 + kBN - 1 > tile_limit;
      // Columns c < nvalid are visible to this row.
      const int nvalid = masked ? max(0, min(kBN, limit - key0 + 1)) : kBN;
      if (masked) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (32 * c + e >= nvalid) sr[c][e] = __float_as_uint(-INFINITY);
      }
      float smax = -INFINITY;
      if (KTOK) {
        // Eight independent chains, then a short tree (the 3-input max does
        // not reassociate); measured faster here, neutral elsewhere.
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int c = k >> 1, e0 = (k & 1) * 16;
          mx[k] = max3(__uint_as_float(sr[c][e0]), __uint_as_float(sr[c][e0 + 1]), __uint_as_float(sr[c][e0 + 2]));
#pragma unroll
          for (int e = 3; e < 15; e += 2)
            mx[k] = max3(mx[k], __uint_as_float(sr[c][e0 + e]), __uint_as_float(sr[c][e0 + e + 1]));
          mx[k] = fmaxf(mx[k], __uint_as_float(sr[c][e0 + 15]));
        }
        smax = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            smax = max3(smax, __uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1]));
      }
      const float m_tile = smax == -INFINITY ? -INFINITY
                           : KTOK           ? smax - C::kPScaleLog2 + mb
                                            : smax * sl2;
      const float m_new = fmaxf(m_used, m_tile);
      const bool grow = m_new > m_used + C::kThreshold;
      float alpha = 1.f;
      if (grow) {
        alpha = ex2_approx(m_used - m_new);
        m_used = m_new;
        l *= alpha;
        if (KTOK) {
          // Move this tile's exponents to the new reference.
          const float d = mb - m_used;
          const uint64_t d2 = f2_pack(d, d);
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float x0, x1;
              f2_unpack(f2_add(f2_pack(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])), d2), x0, x1);
              sr[c][e] = __float_as_uint(x0);
              sr[c][e + 1] = __float_as_uint(x1);
            }
        }
      }
      mb = m_used == -INFINITY ? 0.f : m_used;
      const uint64_t negm = f2_pack(C::kPScaleLog2 - mb, C::kPScaleLog2 - mb);
      uint64_t lacc = f2_pack(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float x0, x1;
          if (KTOK) {
            x0 = __uint_as_float(sr[c][2 * e]);
            x1 = __uint_as_float(sr[c][2 * e + 1]);
          } else {
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c][2 * e]), __uint_as_float(sr[c][2 * e + 1])),
                             sl2x2, negm), x0, x1);
          }
          // A masked score is -inf here (sl2 > 0), so its exponential is 0.
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          lacc = f2_add(lacc, f2_pack(p0, p1));
          if (FP8) {
            // 4 codes per column: pairs e (even) and e+1 (odd) share one word.
            const uint32_t two = pack_e4m3x2(p0, p1);
            pk[e >> 1] = (e & 1) ? (pk[e >> 1] | (two << 16)) : two;
            if (SPLIT) {
              // P = e4m3(P) + e4m3(P - e4m3(P)): the rounding remainder as a
              // second term (words 8..15 of pk), about 7 significant bits in all.
              float h0, h1;
              e4m3x2_to_f32(two, h0, h1);
              const uint32_t lo = pack_e4m3x2(p0 - h0, p1 - h1);
              pk[8 + (e >> 1)] = (e & 1) ? (pk[8 + (e >> 1)] | (lo << 16)) : lo;
            }
          } else {
            pk[e] = pack_bf16x2(p0, p1);
          }
        }
        if (c == 0 && pvc > 0) {
          // P_q and O_q are read / written by the previous tile's P.V until it
          // completes.
          if (!mbar_wait(smem_u32(&s.pv_done[q]), (pvc - 1) & 1u, abort)) return;
          tc_fence_after();
        }
        if (FP8) {
          uint32_t w8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) w8[e] = pk[e];
          tmem_st_32x32b_x8(t_p + 8 * c, w8);
          if (SPLIT) {
#pragma unroll
            for (int e = 0; e < 8; ++e) w8[e] = pk[8 + e];
            tmem_st_32x32b_x8(t_p + 32 + 8 * c, w8);
          }
        } else {
          tmem_st_32x32b_x16(t_p + 16 * c, pk);
        }
      }
      float l0, l1;
      f2_unpack(lacc, l0, l1);
      l += l0 + l1;
      ++pvc;
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        // The previous P.V of this tile has completed (see the P stores).  The
        // score registers are free again: the whole O row goes through them
        // in one load, one wait and one store.
        const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(t_o + 32 * c, sr[c]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float x0, x1;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])), a2), x0, x1);
            sr[c][e] = __float_as_uint(x0);
            sr[c][e + 1] = __float_as_uint(x1);
          }
          tmem_st_32x32b_x32(t_o + 32 * c, sr[c]);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&s.p_full[q]));
    }

    // Epilogue: O / l -> bf16 rows of out.
    if (!mbar_wait(smem_u32(&s.o_full[q]), of & 1u, abort)) return;
    ++of;
    tc_fence_after();
    // A row that saw no key (chunked calls only) has l = 0 and O = 0.
    float inv = l > 0.f ? out_scale / l : 0.f;
    const bool store = i < it.n;
    const long long row = it.q_row0 + q * kBM + r;
    uint4* dst = reinterpret_cast<uint4*>(p.out + row * p.out_tok + static_cast<long long>(it.h) * p.out_head);
    // Folding chunked calls: out / lse already hold the result over the
    // sequence's earlier buffer rows (its window does not start at context
    // position 0); combine by log-sum-exp weights, old : new = wo : wn.
    float keep = 0.f;  // weight of the old output row
    if (p.lse && store) {
      float* lp = p.lse + row * p.lse_tok + static_cast<long long>(it.h) * p.lse_head;
      float lse = l > 0.f ? (m_used + __log2f(l) - C::kPScaleLog2) * kLn2 : -INFINITY;
      if (p.accumulate && it.co > 0) {
        const float old = *lp;
        const float mx = fmaxf(old, lse);
        if (mx > -INFINITY) {
          const float wo = ex2_approx((old - mx) * kLog2e), wn = ex2_approx((lse - mx) * kLog2e);
          const float den = 1.f / (wo + wn);
          keep = wo * den;
          inv *= wn * den;
          lse = mx + __log2f(wo + wn) * kLn2;
        }
      }
      *lp = lse;
    }
    const uint64_t inv2 = f2_pack(inv, inv);
    const uint64_t keep2 = f2_pack(keep, keep);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      tmem_ld_32x32b_x32(t_o + 32 * c, o);
      tmem_ld_wait();
      uint32_t pk[16];
      if (keep > 0.f) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 w4 = dst[4 * c + v];
          const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = 4 * v + e;
            const uint64_t prev = f2_pack(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(o[2 * k]), __uint_as_float(o[2 * k + 1])), inv2,
                             f2_mul(prev, keep2)), x0, x1);
            pk[k] = pack_bf16x2(x0, x1);
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float x0, x1;
          f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), inv2), x0, x1);
          pk[e] = pack_bf16x2(x0, x1);
        }
      }
      if (store) {
        if (p.out_v8) {
          // 32-byte stores: whole sectors, half the store instructions.
          st_global_v8(dst + 4 * c, pk);
          st_global_v8(dst + 4 * c + 2, pk + 8);
        } else {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[4 * c + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&s.o_empty[q]));
  }
}

template <bool FP8, bool KTOK, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1) mla_attention_kernel(const __grid_constant__ AttnParams p) {
  using C = Cfg<FP8>;
  extern __shared__ uint8_t smem_raw[];
  Smem<FP8>& s =
      *reinterpret_cast<Smem<FP8>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile uint32_t* abort = &s.abort_flag;

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.item_full[i]), 1);
      // 2 UMMA threads + 8 softmax warps (+ the converter warp for fp8)
      mbar_init(smem_u32(&s.item_empty[i]), FP8 ? 11 : 10);
      mbar_init(smem_u32(&s.q_full[i]), FP8 ? 2 : 1);  // TMA (+ the rope converter warp)
      mbar_init(smem_u32(&s.q_empty[i]), 1);
      mbar_init(smem_u32(&s.s_full[i]), 1);
      mbar_init(smem_u32(&s.p_full[i]), 4);
      mbar_init(smem_u32(&s.o_full[i]), 1);
      mbar_init(smem_u32(&s.o_empty[i]), 4);
      mbar_init(smem_u32(&s.s_free[i][0]), 4);   // the 4 softmax warps of query tile i
      mbar_init(smem_u32(&s.s_free[i][1]), 4);
      mbar_init(smem_u32(&s.pv_done[i]), 1);
      mbar_init(smem_u32(&s.ks_full[i]), 4);
      mbar_init(smem_u32(&s.ks_free[i]), 4);
    }
    for (int i = 0; i < C::kRing; ++i) {
      // Full barriers are per group (see producer_warp).
      mbar_init(smem_u32(&s.kv_full[i]), 1);
      // Both UMMA threads release every chunk.
      mbar_init(smem_u32(&s.kv_empty[i]), 2);
    }
    mbar_init(smem_u32(&s.drain[0]), 1);
    mbar_init(smem_u32(&s.drain[1]), 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    if (!FP8 && !p.rope_manual) tma_prefetch_desc(&p.tm_rope);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 120;" ::: "memory");
    if (warp == 0) {
      producer_warp<FP8, SPLIT>(s, p, lane, abort);
    } else if (warp == 1 || warp == 2) {
      if (lane == 0) mma_thread<FP8, SPLIT>(s, tmem, warp - 1, abort);
      __syncwarp();
    } else if constexpr (FP8) {
      converter_warp(s, p, lane, abort);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
    softmax_warp<FP8, KTOK, SPLIT>(s, p, tmem, (warp - 4) >> 2, warp & 3, lane, abort);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && s.abort_flag)
    atomicOr(&reinterpret_cast<WsHeader*>(p.ws)->status, MLA_DEVICE_STATUS_TIMEOUT);
}

}  // namespace
}  // namespace mla

extern "C" size_t mla_prefill_ragged_workspace_size(uint32_t batch) {
  size_t bytes = sizeof(mla::WsHeader) + static_cast<size_t>(batch) * sizeof(mla::SeqRec);
  return (bytes + 255) & ~size_t(255);
}

extern "C" size_t mla_prefill_ragged_workspace_size_fp8(uint32_t batch, uint64_t pool_slots) {
  // Scheduler records, then the bf16 copy of K_rope' (128 bytes per pool slot).
  return mla_prefill_ragged_workspace_size(batch) + static_cast<size_t>(pool_slots) * 128;
}

namespace mla {
namespace {

// Launches the scheduler, the per-row K_rope conversion (per-token K scales
// only, rows != NULL) and the attention kernel for one input type.
template <bool FP8, bool KTOK, bool SPLIT>
mla_status_t launch_attention(AttnParams& prm, int dev, int sms, const uint32_t* row_offsets,
                              const uint32_t* cache_lens, const uint32_t* buffer_row_offsets,
                              const uint32_t* cache_offsets, uint32_t B, uint32_t H, uint32_t Tq,
                              uint32_t Sk, uint32_t P, uint32_t max_pages, void* workspace,
                              const RopeRows* rows, const StackedRows& stk, cudaStream_t cs) {
  mla_status_t st;
  auto* kernel = mla_attention_kernel<FP8, KTOK, SPLIT>;
  {
    // The register split inside the kernel is only safe when the kernel was
    // built with exactly kLaunchRegs registers per thread.
    static int checked[64] = {0};
    if (dev < 64 && !checked[dev]) {
      cudaFuncAttributes fa;
      cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
      if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "cudaFuncGetAttributes: %s", cudaGetErrorString(e));
      if (fa.numRegs != kLaunchRegs)
        return fail(MLA_ERR_UNSUPPORTED, "attention kernel built with %d registers per thread, expected %d",
                    fa.numRegs, kLaunchRegs);
      checked[dev] = 1;
    }
  }
  const int sched_smem = static_cast<int>(3 * B * sizeof(uint32_t));
  if ((st = set_max_dynamic_smem(reinterpret_cast<const void*>(schedule_kernel), sched_smem, dev, 1)) != MLA_OK)
    return st;
  const int attn_smem = static_cast<int>(sizeof(Smem<FP8>) + 1024);
  // One attribute cache slot per kernel instantiation.
  if ((st = set_max_dynamic_smem(reinterpret_cast<const void*>(kernel), attn_smem, dev,
                                 FP8 ? (SPLIT ? (KTOK ? 7 : 6) : (KTOK ? 4 : 3)) : 2)) != MLA_OK)
    return st;
  const uint32_t elt = FP8 ? 1u : 2u;
  schedule_kernel<<<1, kSchedThreads, sched_smem, cs>>>(row_offsets, cache_lens, buffer_row_offsets,
                                                        cache_offsets, B, H, Tq, Sk, P, max_pages,
                                                        elt * (128 + 128), stk, static_cast<uint8_t*>(workspace));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "scheduler launch: %s", cudaGetErrorString(e));
  if (rows) {
    // About 4 blocks per SM in all, at least one per sequence record.
    const uint32_t gy = std::max<uint32_t>(
        1u, std::min<uint32_t>((Sk + 255) / 256, (4u * static_cast<uint32_t>(sms) + B - 1) / B));
    rope_convert_rows_kernel<<<dim3(B, gy), 256, 0, cs>>>(*rows);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "rope conversion launch: %s", cudaGetErrorString(e));
  }
  kernel<<<sms, kThreads, attn_smem, cs>>>(prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "attention launch: %s", cudaGetErrorString(e));
  return MLA_OK;
}

std::atomic<uint32_t> g_test_stall{0};
std::atomic<uint32_t> g_test_delay_ns{0};

// Full-context call (buffer_row_offsets == NULL) or one buffer row of a
// chunked call (with lse).
// page_table == NULL: K_rope is contiguous, k_rope_pages is [Sk, 64] with row
// r holding the rope part of k_nope row r, and contig_batch gives B.
// q_rope != NULL: split Q, q is q_nope [Tq, H, 128] and q_rope [Tq, H, 64] is bf16.
mla_status_t prefill(const mla_tensor_t* out, const mla_tensor_t* lse, const mla_tensor_t* q,
                     const mla_tensor_t* q_rope, const mla_tensor_t* k_nope, const mla_tensor_t* v, const mla_tensor_t* k_rope_pages,
                     const mla_tensor_t* page_table, uint32_t contig_batch, const uint32_t* row_offsets,
                     const uint32_t* cache_lens, const uint32_t* buffer_row_offsets,
                     const uint32_t* cache_offsets, float scale, mla_mask_t mask, uint32_t flags,
                     void* workspace, size_t workspace_bytes, mla_stream_t stream,
                     const StackedRows& stk = StackedRows{nullptr, 0u, 0u}) {
  mla_status_t st;
  const bool stacked = stk.T != 0;
  const bool chunk = buffer_row_offsets != nullptr && !stacked;
  if (flags & ~(MLA_CHUNK_ACCUMULATE | MLA_FP8_PRECISE)) return fail(MLA_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  if ((flags & MLA_CHUNK_ACCUMULATE) && buffer_row_offsets == nullptr)
    return fail(MLA_ERR_INVALID_ARG, "MLA_CHUNK_ACCUMULATE applies to the per-row chunk calls only");
  const bool fp8_precise = (flags & MLA_FP8_PRECISE) != 0;
  const bool contig = page_table == nullptr;
  if (!q) return fail(MLA_ERR_INVALID_ARG, "q descriptor is NULL");
  const bool fp8 = q->dtype == MLA_DTYPE_FP8_E4M3;
  const mla_dtype_t dt = fp8 ? MLA_DTYPE_FP8_E4M3 : MLA_DTYPE_BF16;
  if (fp8_precise && !fp8) return fail(MLA_ERR_INVALID_ARG, "MLA_FP8_PRECISE needs fp8 inputs");
  if ((st = check_tensor(q, "q", 3, dt)) != MLA_OK) return st;
  if ((st = check_tensor(out, "out", 3, MLA_DTYPE_BF16)) != MLA_OK) return st;
  if ((st = check_tensor(k_nope, "k_nope", 3, dt)) != MLA_OK) return st;
  if ((st = check_tensor(v, "v", 3, dt)) != MLA_OK) return st;
  if ((st = check_tensor(k_rope_pages, contig ? "k_rope" : "k_rope_pages", contig ? 2 : 3, dt)) != MLA_OK)
    return st;
  if (!contig && (st = check_tensor(page_table, "page_table", 2, MLA_DTYPE_U32)) != MLA_OK) return st;
  const bool split = q_rope != nullptr;
  // fp8 K_nope may carry one scale per K row instead of one per tensor.
  const bool ktok = fp8 && k_nope->scale && k_nope->scale_gran == MLA_SCALE_PER_TOKEN;
  if (fp8) {
    const mla_tensor_t* pt[3] = {q, k_nope, v};
    const char* pn[3] = {"q", "k_nope", "v"};
    for (int i = 0; i < 3; ++i) {
      if (i == 1 && ktok) continue;
      // Split Q: v without a scale of its own is dequantised with k's
      // (per-tensor k only).
      if (split && i == 2 && !v->scale && !ktok) continue;
      if (!pt[i]->scale || pt[i]->scale_gran != MLA_SCALE_PER_TENSOR)
        return fail(MLA_ERR_INVALID_ARG, "fp8 %s needs a per-tensor scale%s", pn[i],
                    i == 1 ? " or one scale per row" : "");
    }
    if (!k_rope_pages->scale || k_rope_pages->scale_gran != MLA_SCALE_PER_TOKEN)
      return fail(MLA_ERR_INVALID_ARG, "fp8 k_rope_pages needs per-token scales");
  }
  if (!row_offsets || !cache_lens) return fail(MLA_ERR_INVALID_ARG, "row_offsets / cache_lens is NULL");
  if (mask != MLA_MASK_CAUSAL && mask != MLA_MASK_NULL) return fail(MLA_ERR_INVALID_ARG, "unknown mask %d", (int)mask);
  if (!(scale >= 0.f) || !std::isfinite(scale)) return fail(MLA_ERR_INVALID_ARG, "scale must be finite and >= 0");

  const int64_t Tq = q->shape[0], H = q->shape[1], Sk = k_nope->shape[0];
  // A contiguous K_rope is addressed like a pool of one-row pages whose page
  // id is the K row; the page table is not read.
  const int64_t B = contig ? static_cast<int64_t>(contig_batch) : page_table->shape[0];
  const int64_t max_pages = contig ? 0xFFFFFFFFll : page_table->shape[1];
  const int64_t NP = k_rope_pages->shape[0], P = contig ? 1 : k_rope_pages->shape[1];
  if (split) {
    if (q->shape[2] != 128) return fail(MLA_ERR_INVALID_ARG, "q_nope depth must be 128");
    if ((st = check_tensor(q_rope, "q_rope", 3, MLA_DTYPE_BF16)) != MLA_OK) return st;
    if (q_rope->shape[0] != Tq || q_rope->shape[1] != H || q_rope->shape[2] != 64)
      return fail(MLA_ERR_INVALID_ARG, "q_rope must be [Tq, H, 64] matching q_nope");
    if (!aligned16(q_rope->data) || (q_rope->stride[0] * 2) % 16 != 0 || (q_rope->stride[1] * 2) % 16 != 0)
      return fail(MLA_ERR_INVALID_ARG, "q_rope must be 16-byte aligned with 16-byte-multiple strides");
  } else if (q->shape[2] != 192) {
    return fail(MLA_ERR_INVALID_ARG, "q depth must be 192");
  }
  if (out->shape[0] != Tq || out->shape[1] != H || out->shape[2] != 128)
    return fail(MLA_ERR_INVALID_ARG, "out must be [Tq, H, 128] matching q");
  if (k_nope->shape[1] != H || k_nope->shape[2] != 128) return fail(MLA_ERR_INVALID_ARG, "k_nope must be [Sk, H, 128]");
  if (v->shape[0] != Sk || v->shape[1] != H || v->shape[2] != 128) return fail(MLA_ERR_INVALID_ARG, "v must be [Sk, H, 128] matching k_nope");
  if (contig) {
    if (NP != Sk || k_rope_pages->shape[1] != 64) return fail(MLA_ERR_INVALID_ARG, "k_rope must be [Sk, 64] matching k_nope");
  } else if (k_rope_pages->shape[2] != 64) {
    return fail(MLA_ERR_INVALID_ARG, "k_rope_pages must be [num_pages, P, 64]");
  }
  if (H < 1) return fail(MLA_ERR_INVALID_ARG, "num_heads must be >= 1");
  if (B < 1 || B > kMaxBatch) return fail(MLA_ERR_INVALID_ARG, "batch %lld outside 1..%u", (long long)B, kMaxBatch);
  if (P < 1 || NP < 1 || max_pages < 1) return fail(MLA_ERR_INVALID_ARG, "empty page pool or page table");
  if (NP * P > 0x7FFFFFFFll) return fail(MLA_ERR_INVALID_ARG, "page pool exceeds 2^31 slots");
  if (chunk || lse) {
    if (chunk && !cache_offsets) return fail(MLA_ERR_INVALID_ARG, "cache_offsets is NULL");
    if ((st = check_tensor(lse, "lse", 2, MLA_DTYPE_F32)) != MLA_OK) return st;
    if (lse->shape[0] != Tq || lse->shape[1] != H) return fail(MLA_ERR_INVALID_ARG, "lse must be [Tq, H] matching q");
    if (reinterpret_cast<uintptr_t>(lse->data) & 3u) return fail(MLA_ERR_INVALID_ARG, "lse data must be 4-byte aligned");
  }
  if (stacked) {
    if (!buffer_row_offsets || !cache_offsets || !stk.num_rows)
      return fail(MLA_ERR_INVALID_ARG, "buffer_row_offsets / cache_offsets / num_rows is NULL");
    if (stk.max_rows < 1) return fail(MLA_ERR_INVALID_ARG, "max_rows must be >= 1");
    if (static_cast<uint64_t>(stk.max_rows) * stk.T > 0x7FFFFFFFull)
      return fail(MLA_ERR_INVALID_ARG, "max_rows x buffer_token_size exceeds 2^31 K rows");
    if (Sk < Tq) return fail(MLA_ERR_INVALID_ARG, "k_nope has fewer rows than q");
  } else if (chunk) {
    if (Sk < 1) return fail(MLA_ERR_INVALID_ARG, "the buffer row holds no keys");
  } else if (Sk < Tq) {
    return fail(MLA_ERR_INVALID_ARG, "k_nope has fewer rows than q");
  }
  if ((Tq / kQRows + B + 1) * H > 0x7FFFFFFFll)
    return fail(MLA_ERR_INVALID_ARG, "too many work items (query blocks x heads exceeds 2^31)");
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(MLA_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
  // fp8: the bf16 K_rope' copy has one row per pool slot, or per K row when
  // K scales are per token.
  // With two K_rope' terms the remainder copy follows the first.
  const uint64_t rope_slots = static_cast<uint64_t>(ktok ? Sk : NP * P);
  const size_t ws_need = fp8 ? mla_prefill_ragged_workspace_size_fp8(static_cast<uint32_t>(B),
                                                                     rope_slots * (fp8_precise ? 2u : 1u))
                             : mla_prefill_ragged_workspace_size(static_cast<uint32_t>(B));
  if (workspace_bytes < ws_need)
    return fail(MLA_ERR_INVALID_ARG, "workspace too small: %zu bytes needed", ws_need);
  // TMA and vector-access constraints: 16-byte aligned bases and strides.
  const mla_tensor_t* ts[5] = {q, k_nope, v, k_rope_pages, out};
  const char* names[5] = {"q", "k_nope", "v", "k_rope_pages", "out"};
  for (int i = 0; i < 5; ++i) {
    const int64_t es = (i < 4 && fp8) ? 1 : 2;
    if (!aligned16(ts[i]->data)) return fail(MLA_ERR_INVALID_ARG, "%s data must be 16-byte aligned", names[i]);
    for (int d = 0; d < ts[i]->ndim - 1; ++d)
      if ((ts[i]->stride[d] * es) % 16 != 0 || ts[i]->stride[d] * es >= (1ll << 40))
        return fail(MLA_ERR_INVALID_ARG, "%s stride[%d] must be a multiple of 16 bytes", names[i], d);
  }

  int dev = 0, sms = 0;
  if ((st = check_device(&dev, &sms)) != MLA_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (Tq == 0) {
    cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(WsHeader), cs);
    if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "workspace reset: %s", cudaGetErrorString(e));
    return MLA_OK;
  }

  AttnParams prm;
  memset(&prm, 0, sizeof(prm));
  const int64_t es = fp8 ? 1 : 2;
  const CUtensorMapDataType tdt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // Boxes are 128 bytes wide (one swizzle atom): 64 bf16 or 128 e4m3 codes.
  const uint32_t inner = fp8 ? 128 : 64;
  {
    uint64_t dims[3] = {split ? 128u : 192u, (uint64_t)H, (uint64_t)Tq};
    uint64_t str[2] = {(uint64_t)(q->stride[1] * es), (uint64_t)(q->stride[0] * es)};
    uint32_t box[3] = {inner, 1, kBM};
    if ((st = encode_tiled(&prm.tm_q, tdt, 3, q->data, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B, "q")) != MLA_OK)
      return st;
    if (split) {
      prm.q_split = 1;
      prm.qr_base = static_cast<const uint8_t*>(q_rope->data);
      prm.qr_tok = q_rope->stride[0] * 2;
      prm.qr_head = q_rope->stride[1] * 2;
      uint64_t dr[3] = {64, (uint64_t)H, (uint64_t)Tq};
      uint64_t sr[2] = {(uint64_t)(q_rope->stride[1] * 2), (uint64_t)(q_rope->stride[0] * 2)};
      uint32_t br[3] = {64, 1, kBM};
      if ((st = encode_tiled(&prm.tm_qr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q_rope->data, dr, sr, br,
                             CU_TENSOR_MAP_SWIZZLE_128B, "q_rope")) != MLA_OK)
        return st;
    }
  }
  {
    uint64_t dims[3] = {128, (uint64_t)H, (uint64_t)Sk};
    uint32_t box[3] = {inner, 1, kBN};
    uint64_t str[2] = {(uint64_t)(k_nope->stride[1] * es), (uint64_t)(k_nope->stride[0] * es)};
    if ((st = encode_tiled(&prm.tm_k, tdt, 3, k_nope->data, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B,
                           "k_nope")) != MLA_OK)
      return st;
    uint64_t strv[2] = {(uint64_t)(v->stride[1] * es), (uint64_t)(v->stride[0] * es)};
    if ((st = encode_tiled(&prm.tm_v, tdt, 3, v->data, dims, strv, box, CU_TENSOR_MAP_SWIZZLE_128B, "v")) != MLA_OK)
      return st;
  }
  uint32_t g = 1;
  {
    uint32_t a = static_cast<uint32_t>(P), b = kBN;
    while (b) { uint32_t t = a % b; a = b; b = t; }
    g = a;  // gcd(P, 128): rows per page segment inside a key tile
  }
  // Per-token K scales: the converted K_rope' sits at the K rows, so the
  // kernel reads it like a contiguous K_rope whatever the caller's layout.
  const bool rows_contig = contig || ktok;
  prm.rope_contig = rows_contig;
  prm.rope_manual = !rows_contig && (g % 8u) != 0;
  prm.rope_box = rows_contig ? kBN : g;
  // bf16 K_rope rows: the caller's pool, or for fp8 inputs the converted copy
  // the pre-pass writes after the scheduler records in the workspace.
  const int64_t rope_tok_el = contig ? k_rope_pages->stride[0] : k_rope_pages->stride[1];
  void* rope_rows = k_rope_pages->data;
  uint64_t rope_tok = static_cast<uint64_t>(rope_tok_el) * 2;
  uint64_t rope_page = static_cast<uint64_t>(k_rope_pages->stride[0]) * 2;
  void* rope_rows_lo = nullptr;
  if (fp8) {
    rope_rows = static_cast<uint8_t*>(workspace) + mla_prefill_ragged_workspace_size(static_cast<uint32_t>(B));
    rope_tok = 128;
    rope_page = static_cast<uint64_t>(P) * 128;
    if (fp8_precise) rope_rows_lo = static_cast<uint8_t*>(rope_rows) + rope_slots * 128;
  }
  if (rows_contig) {
    // One 128-row box per KV tile, at the tile's K row.
    uint64_t dims[2] = {64, (uint64_t)(ktok ? Sk : NP)};
    uint64_t str[1] = {rope_tok};
    uint32_t box[2] = {64, kBN};
    if ((st = encode_tiled(&prm.tm_rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rope_rows, dims, str, box,
                           CU_TENSOR_MAP_SWIZZLE_128B, "k_rope")) != MLA_OK)
      return st;
    if (rope_rows_lo && (st = encode_tiled(&prm.tm_rope_lo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rope_rows_lo, dims,
                                           str, box, CU_TENSOR_MAP_SWIZZLE_128B, "k_rope remainder")) != MLA_OK)
      return st;
  } else if (!prm.rope_manual) {
    uint64_t dims[3] = {64, (uint64_t)P, (uint64_t)NP};
    uint64_t str[2] = {rope_tok, rope_page};
    uint32_t box[3] = {64, g, 1};
    if ((st = encode_tiled(&prm.tm_rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, rope_rows, dims, str, box,
                           CU_TENSOR_MAP_SWIZZLE_128B, "k_rope_pages")) != MLA_OK)
      return st;
    if (rope_rows_lo && (st = encode_tiled(&prm.tm_rope_lo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, rope_rows_lo, dims,
                                           str, box, CU_TENSOR_MAP_SWIZZLE_128B, "k_rope remainder")) != MLA_OK)
      return st;
  }
  prm.out = static_cast<uint16_t*>(out->data);
  prm.out_tok = out->stride[0];
  prm.out_head = out->stride[1];
  prm.out_v8 = (reinterpret_cast<uintptr_t>(out->data) % 32u == 0 && (prm.out_tok * 2) % 32 == 0 &&
                (prm.out_head * 2) % 32 == 0)
                   ? 1u
                   : 0u;
  if (chunk || lse) {
    prm.lse = static_cast<float*>(lse->data);
    prm.lse_tok = lse->stride[0];
    prm.lse_head = lse->stride[1];
    prm.accumulate = (flags & MLA_CHUNK_ACCUMULATE) ? 1u : 0u;
  }
  prm.page_table = contig ? nullptr : static_cast<const uint32_t*>(page_table->data);
  prm.pt_stride = contig ? 0 : page_table->stride[0];
  prm.rope_base = static_cast<const uint8_t*>(rope_rows);
  prm.rope_base_lo = static_cast<const uint8_t*>(rope_rows_lo);
  prm.rope_tok_bytes = static_cast<long long>(rope_tok);
  prm.rope_page_bytes = static_cast<long long>(rope_page);
  prm.max_pages = static_cast<uint32_t>(max_pages);
  prm.num_pages = static_cast<uint32_t>(NP);
  prm.page_size = static_cast<uint32_t>(P);
  prm.H = static_cast<uint32_t>(H);
  prm.causal = mask == MLA_MASK_CAUSAL;
  prm.test_stall = g_test_stall.load(std::memory_order_relaxed);
  prm.test_delay_ns = g_test_delay_ns.load(std::memory_order_relaxed);
  prm.sl2 = scale * 1.4426950408889634f;
  prm.ws = static_cast<uint8_t*>(workspace);
  prm.q_base = static_cast<const uint8_t*>(q->data);
  prm.q_tok = q->stride[0] * es;
  prm.q_head = q->stride[1] * es;
  prm.Tq = static_cast<uint32_t>(Tq);
  if (fp8) {
    prm.q_scale = q->scale;
    prm.k_scale = ktok ? nullptr : k_nope->scale;
    prm.k_tok_scales = ktok ? k_nope->scale : nullptr;
    prm.v_scale = v->scale ? v->scale : k_nope->scale;
    prm.rope_scales = k_rope_pages->scale;
  }
  const uint32_t uB = static_cast<uint32_t>(B), uH = static_cast<uint32_t>(H), uTq = static_cast<uint32_t>(Tq),
                 uSk = static_cast<uint32_t>(Sk), uP = static_cast<uint32_t>(P),
                 uMP = static_cast<uint32_t>(max_pages);
  if (ktok) {
    RopeRows rr;
    rr.pool = static_cast<const uint8_t*>(k_rope_pages->data);
    rr.tok_bytes = rope_tok_el;
    rr.page_bytes = k_rope_pages->stride[0];
    rr.page_table = contig ? nullptr : static_cast<const uint32_t*>(page_table->data);
    rr.pt_stride = contig ? 0 : page_table->stride[0];
    rr.P = uP;
    rr.num_pages = static_cast<uint32_t>(NP);
    rr.max_pages = uMP;
    rr.Sk = uSk;
    rr.rope_scales = k_rope_pages->scale;
    rr.k_scales = k_nope->scale;
    rr.out = static_cast<uint16_t*>(rope_rows);
    rr.out_lo = static_cast<uint16_t*>(rope_rows_lo);
    rr.ws = static_cast<uint8_t*>(workspace);
    auto launch_k = fp8_precise ? launch_attention<true, true, true> : launch_attention<true, true, false>;
    return launch_k(prm, dev, sms, row_offsets, cache_lens, buffer_row_offsets,
                                        cache_offsets, uB, uH, uTq, uSk, uP, uMP, workspace, &rr, stk, cs);
  }
  if (fp8) {
    const uint32_t slots = static_cast<uint32_t>(NP * P);
    const int blocks = static_cast<int>(std::min<uint32_t>((slots + 255) / 256, 16u * sms));
    rope_convert_kernel<<<blocks, 256, 0, cs>>>(
        static_cast<const uint8_t*>(k_rope_pages->data), rope_tok_el, k_rope_pages->stride[0],
        static_cast<uint32_t>(P), slots, k_rope_pages->scale, k_nope->scale, static_cast<uint16_t*>(rope_rows),
        static_cast<uint16_t*>(rope_rows_lo));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "rope conversion launch: %s", cudaGetErrorString(e));
  }
  auto launch = !fp8 ? launch_attention<false, false, false>
                     : fp8_precise ? launch_attention<true, false, true> : launch_attention<true, false, false>;
  return launch(prm, dev, sms, row_offsets, cache_lens, buffer_row_offsets, cache_offsets, uB, uH, uTq, uSk,
                uP, uMP, workspace, nullptr, stk, cs);
}

}  // namespace
}  // namespace mla

extern "C" mla_status_t mla_prefill_ragged(const mla_tensor_t* out, const mla_tensor_t* q,
                                           const mla_tensor_t* k_nope, const mla_tensor_t* v,
                                           const mla_tensor_t* k_rope_pages,
                                           const mla_tensor_t* page_table,
                                           const uint32_t* row_offsets, const uint32_t* cache_lens,
                                           float scale, mla_mask_t mask, void* workspace,
                                           size_t workspace_bytes, mla_stream_t stream) {
  if (!page_table) return mla::fail(MLA_ERR_INVALID_ARG, "page_table descriptor is NULL");
  return mla::prefill(out, nullptr, q, nullptr, k_nope, v, k_rope_pages, page_table, 0, row_offsets, cache_lens,
                      nullptr, nullptr, scale, mask, 0u, workspace, workspace_bytes, stream);
}

extern "C" mla_status_t mla_test_inject_stall(uint32_t enable) {
  mla::g_test_stall.store(enable ? 1u : 0u, std::memory_order_relaxed);
  return MLA_OK;
}

extern "C" mla_status_t mla_test_delay_softmax(uint32_t nanoseconds) {
  if (nanoseconds > 100000u) return mla::fail(MLA_ERR_INVALID_ARG, "delay above 100 us");
  mla::g_test_delay_ns.store(nanoseconds, std::memory_order_relaxed);
  return MLA_OK;
}

extern "C" mla_status_t mla_prefill_ragged_split(
    const mla_tensor_t* out, const mla_tensor_t* q_nope, const mla_tensor_t* q_rope, const mla_tensor_t* k_nope,
    const mla_tensor_t* v, const mla_tensor_t* k_rope, const mla_tensor_t* page_table, uint32_t batch,
    const uint32_t* row_offsets, const uint32_t* cache_lens, float scale, mla_mask_t mask, void* workspace,
    size_t workspace_bytes, mla_stream_t stream) {
  if (!q_rope) return mla::fail(MLA_ERR_INVALID_ARG, "q_rope descriptor is NULL");
  if (batch < 1) return mla::fail(MLA_ERR_INVALID_ARG, "batch must be >= 1");
  if (page_table && page_table->shape[0] != static_cast<int64_t>(batch))
    return mla::fail(MLA_ERR_INVALID_ARG, "page_table has %lld rows for batch %u",
                     (long long)page_table->shape[0], batch);
  return mla::prefill(out, nullptr, q_nope, q_rope, k_nope, v, k_rope, page_table, batch, row_offsets,
                      cache_lens, nullptr, nullptr, scale, mask, 0u, workspace, workspace_bytes, stream);
}

extern "C" mla_status_t mla_prefill_ragged_chunk_contiguous(
    const mla_tensor_t* out, const mla_tensor_t* lse, const mla_tensor_t* q, const mla_tensor_t* k_nope,
    const mla_tensor_t* v, const mla_tensor_t* k_rope, const uint32_t* row_offsets,
    const uint32_t* cache_lens, const uint32_t* buffer_row_offsets, const uint32_t* cache_offsets,
    uint32_t batch, float scale, mla_mask_t mask, uint32_t flags, void* workspace,
    size_t workspace_bytes, mla_stream_t stream) {
  if (!buffer_row_offsets) return mla::fail(MLA_ERR_INVALID_ARG, "buffer_row_offsets is NULL");
  if (batch < 1) return mla::fail(MLA_ERR_INVALID_ARG, "batch must be >= 1");
  return mla::prefill(out, lse, q, nullptr, k_nope, v, k_rope, nullptr, batch, row_offsets, cache_lens,
                      buffer_row_offsets, cache_offsets, scale, mask, flags, workspace, workspace_bytes,
                      stream);
}

extern "C" mla_status_t mla_prefill_ragged_contiguous(const mla_tensor_t* out, const mla_tensor_t* q,
                                                      const mla_tensor_t* k_nope, const mla_tensor_t* v,
                                                      const mla_tensor_t* k_rope,
                                                      const uint32_t* row_offsets,
                                                      const uint32_t* cache_lens, uint32_t batch,
                                                      float scale, mla_mask_t mask, void* workspace,
                                                      size_t workspace_bytes, mla_stream_t stream) {
  if (batch < 1) return mla::fail(MLA_ERR_INVALID_ARG, "batch must be >= 1");
  return mla::prefill(out, nullptr, q, nullptr, k_nope, v, k_rope, nullptr, batch, row_offsets, cache_lens,
                      nullptr, nullptr, scale, mask, 0u, workspace, workspace_bytes, stream);
}

extern "C" mla_status_t mla_prefill_ragged_chunked(
    const mla_tensor_t* out, const mla_tensor_t* lse, const mla_tensor_t* q, const mla_tensor_t* k_nope,
    const mla_tensor_t* v, const mla_tensor_t* k_rope_pages, const mla_tensor_t* page_table,
    const uint32_t* row_offsets, const uint32_t* cache_lens, const uint32_t* buffer_row_offsets,
    const uint32_t* cache_offsets, const uint32_t* num_rows, uint32_t max_rows, uint32_t buffer_token_size,
    float scale, mla_mask_t mask, uint32_t flags, void* workspace, size_t workspace_bytes,
    mla_stream_t stream) {
  if (!page_table) return mla::fail(MLA_ERR_INVALID_ARG, "page_table descriptor is NULL");
  if (buffer_token_size < 1) return mla::fail(MLA_ERR_INVALID_ARG, "buffer_token_size must be >= 1");
  if (flags & MLA_CHUNK_ACCUMULATE)
    return mla::fail(MLA_ERR_INVALID_ARG, "MLA_CHUNK_ACCUMULATE applies to the per-row chunk calls only");
  return mla::prefill(out, lse, q, nullptr, k_nope, v, k_rope_pages, page_table, 0, row_offsets, cache_lens,
                      buffer_row_offsets, cache_offsets, scale, mask, flags, workspace, workspace_bytes, stream,
                      mla::StackedRows{num_rows, max_rows, buffer_token_size});
}

extern "C" mla_status_t mla_prefill_ragged_ex(const mla_tensor_t* out, const mla_tensor_t* lse,
                                              const mla_tensor_t* q, const mla_tensor_t* k_nope,
                                              const mla_tensor_t* v, const mla_tensor_t* k_rope_pages,
                                              const mla_tensor_t* page_table, const uint32_t* row_offsets,
                                              const uint32_t* cache_lens, float scale, mla_mask_t mask,
                                              uint32_t flags, void* workspace, size_t workspace_bytes,
                                              mla_stream_t stream) {
  if (!page_table) return mla::fail(MLA_ERR_INVALID_ARG, "page_table descriptor is NULL");
  return mla::prefill(out, lse, q, nullptr, k_nope, v, k_rope_pages, page_table, 0, row_offsets, cache_lens,
                      nullptr, nullptr, scale, mask, flags, workspace, workspace_bytes, stream);
}

extern "C" mla_status_t mla_prefill_ragged_chunk(
    const mla_tensor_t* out, const mla_tensor_t* lse, const mla_tensor_t* q, const mla_tensor_t* k_nope,
    const mla_tensor_t* v, const mla_tensor_t* k_rope_pages, const mla_tensor_t* page_table,
    const uint32_t* row_offsets, const uint32_t* cache_lens, const uint32_t* buffer_row_offsets,
    const uint32_t* cache_offsets, float scale, mla_mask_t mask, uint32_t flags, void* workspace,
    size_t workspace_bytes, mla_stream_t stream) {
  if (!buffer_row_offsets) return mla::fail(MLA_ERR_INVALID_ARG, "buffer_row_offsets is NULL");
  if (!page_table) return mla::fail(MLA_ERR_INVALID_ARG, "page_table descriptor is NULL");
  return mla::prefill(out, lse, q, nullptr, k_nope, v, k_rope_pages, page_table, 0, row_offsets, cache_lens,
                      buffer_row_offsets, cache_offsets, scale, mask, flags, workspace, workspace_bytes,
                      stream);
}

// ------------------------------------------------------------ no-allocation entry point
// Some callers cannot hand this library a workspace: a plug-in whose host
// framework owns every byte of device memory through its own pool and offers
// it no scratch buffer, or code on a latency-critical path where cudaMalloc
// (which may synchronise the device) is not acceptable.  For them the
// scheduler workspace lives in this fixed, file-scope device array instead,
// sized for up to kNoAllocMaxBatch sequences (33,024 bytes).  Every GPU that
// loads the library holds the array until the process exits.
namespace mla {
namespace {
constexpr uint32_t kNoAllocMaxBatch = 1024;
constexpr size_t kNoAllocBytes = sizeof(WsHeader) + kNoAllocMaxBatch * sizeof(SeqRec);
static_assert(kNoAllocBytes % 256 == 0, "workspace size must keep 256-byte granularity");

// The array's device address belongs to the context that loaded the module:
// a cudaDeviceReset (or any other re-creation of the device's primary
// context) moves it.  So the address is cached per device together with the
// id of the context it was looked up in, and looked up again when the
// current context's id differs.
struct NoAllocSlot {
  std::mutex m;
  unsigned long long ctx_id = 0;
  void* addr = nullptr;
};
NoAllocSlot g_noalloc[64];
using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);
PfnCtxGetCurrent g_ctx_get_current = nullptr;
PfnCtxGetId g_ctx_get_id = nullptr;
std::once_flag g_ctx_fn_once;

// Id of the calling thread's current context, 0 if none is current (the
// runtime creates the primary context lazily) or the driver lacks the query.
unsigned long long current_ctx_id() {
  std::call_once(g_ctx_fn_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<PfnCtxGetCurrent>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = reinterpret_cast<PfnCtxGetId>(fn);
  });
  if (!g_ctx_get_current || !g_ctx_get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}
}  // namespace
}  // namespace mla

static __device__ __align__(256) unsigned char g_noalloc_workspace[mla::kNoAllocBytes];

extern "C" mla_status_t mla_prefill_ragged_noalloc(const mla_tensor_t* out, const mla_tensor_t* q,
                                                   const mla_tensor_t* k_nope, const mla_tensor_t* v,
                                                   const mla_tensor_t* k_rope_pages,
                                                   const mla_tensor_t* page_table,
                                                   const uint32_t* row_offsets,
                                                   const uint32_t* cache_lens, float scale,
                                                   mla_mask_t mask, mla_stream_t stream) {
  using namespace mla;
  if (!page_table) return fail(MLA_ERR_INVALID_ARG, "page_table descriptor is NULL");
  if (page_table->shape[0] > static_cast<int64_t>(kNoAllocMaxBatch))
    return fail(MLA_ERR_INVALID_ARG,
                "batch %lld exceeds the %u sequences the built-in workspace of "
                "mla_prefill_ragged_noalloc holds; use mla_prefill_ragged with a workspace",
                (long long)page_table->shape[0], kNoAllocMaxBatch);
  // fp8 inputs convert the whole K_rope pool into the workspace first, which
  // the fixed array has no room for.
  const mla_tensor_t* ins[4] = {q, k_nope, v, k_rope_pages};
  for (const mla_tensor_t* t : ins)
    if (t && t->dtype == MLA_DTYPE_FP8_E4M3)
      return fail(MLA_ERR_INVALID_ARG,
                  "mla_prefill_ragged_noalloc takes bf16 inputs only; fp8 inputs need "
                  "mla_prefill_ragged with a workspace");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MLA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(MLA_ERR_UNSUPPORTED, "device index %d", dev);
  // Set-up, once per device and context (the device is current here): the
  // array's host-side name is only a stand-in, so ask the runtime for its
  // address.
  void* ws = nullptr;
  {
    NoAllocSlot& slot = g_noalloc[dev];
    std::lock_guard<std::mutex> lock(slot.m);
    const unsigned long long id = current_ctx_id();
    if (id != 0 && id == slot.ctx_id && slot.addr) {
      ws = slot.addr;
    } else {
      e = cudaGetSymbolAddress(&ws, g_noalloc_workspace);
      if (e != cudaSuccess || !ws)
        return fail(MLA_ERR_CUDA, "cudaGetSymbolAddress(workspace): %s", cudaGetErrorString(e));
      // The lookup made the primary context current if it was not yet.
      slot.ctx_id = current_ctx_id();
      slot.addr = ws;
    }
  }
  // The scheduler launch inside rewrites every workspace field the attention
  // kernel reads (header, work counter, sequence records) on each call.
  return mla_prefill_ragged(out, q, k_nope, v, k_rope_pages, page_table, row_offsets, cache_lens,
                            scale, mask, ws, kNoAllocBytes, stream);
}
