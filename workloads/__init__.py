"""Seeded synthetic inputs for MLA ragged paged prefill.

This module only draws random numbers and lays them out: ragged lengths, a
shuffled page pool with its page table, and Q / K_nope / V / K_rope values
(bf16, or fp8-e4m3 codes with their fp32 scales).  It holds none of the
attention or plan arithmetic.  Both the CPU oracle and the GPU tests/bench
take their inputs from here.

Shapes follow the flare_mla_prefill page (Args: q, k, v, k_rope):
  q        [total_q_tokens, H, 192]   (128 nope dims then 64 rope dims)
  k_nope   [S_k, H, 128]              (S_k = sum over sequences of prior + new)
  v        [S_k, H, 128]
  k_rope   paged pool [num_pages, page_size, row_width], the 64 rope dims at
           columns [rope_col, rope_col + 64) of each token row
  page_table [B, max_pages] uint32: logical page -> physical page
Sequence b's K context (prior cached tokens followed by its new tokens) sits
in rows [G_b, G_b + L_b) of k_nope / v, with G_b the running sum of L over
earlier sequences.

Recipe: numpy Generator(PCG64(seed)); draw order lengths, priors, page
permutation, Q, K_nope, V, K_rope; standard normal float32 values times
``value_scale``; bf16 by round-to-nearest-even (torch CPU cast).  fp8 inputs
use a per-tensor scale amax/448 for Q, K_nope and V and a per-token scale
amax_row/448 for K_rope, with a saturating round-to-nearest-even cast.  The
pool holds exactly sum(ceil(L_b / P)) pages plus one spare page, in a random
permutation; slack slots, the spare page and any extra row columns are NaN so
that a wrong gather shows up as NaN.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional, Sequence

import numpy as np
import torch

Q_DEPTH = 192
NOPE_DEPTH = 128
ROPE_DEPTH = 64
V_DEPTH = 128
FP8_MAX = 448.0
FP8_NAN_CODE = 0x7F

_CHUNK = 1 << 25


@dataclass(frozen=True)
class Spec:
    name: str
    batch: int
    heads: int
    page_size: int
    buffer_token_size: int
    dtype: str                 # "bf16" or "fp8"
    seed: int
    new_len: tuple             # ("fixed", (..)) | ("uniform", lo, hi) | ("loguniform", lo, hi)
    prior_len: tuple           # ("zero",) | ("fixed", v) | ("uniform", lo, hi)
    value_scale: float = 1.0
    mask: str = "causal"       # "causal" or "null"
    row_width: int = ROPE_DEPTH  # width of one pool token row (>= 64)
    rope_col: int = 0            # column of the first rope dim in a pool row
    description: str = ""


# The five workloads of this library's parity and throughput suite.
CONFIGS = [
    Spec("tiny_bf16", 2, 4, 16, 32, "bf16", 0, ("fixed", (17, 33)), ("zero",),
         description="B=2, n={17,33}, no prior, H=4, P=16, T=32, bf16 N(0,1)"),
    Spec("ragged_chunked_bf16", 4, 16, 128, 1024, "bf16", 1, ("uniform", 1, 512),
         ("uniform", 0, 1024),
         description="B=4, n~U[1,512], prior~U[0,1024], H=16, P=128, T=1024, bf16 N(0,1)"),
    Spec("deepseek_v3_bf16", 8, 128, 128, 4096, "bf16", 2, ("uniform", 512, 4096), ("zero",),
         value_scale=0.5,
         description="B=8, n~U[512,4096], no prior, H=128, P=128, T=4096, bf16 0.5*N(0,1)"),
    Spec("long_context_bf16", 2, 128, 128, 8192, "bf16", 3, ("fixed", (8192, 8192)),
         ("fixed", 32768),
         description="B=2, n=8192, prior=32768, H=128, P=128, T=8192, bf16 N(0,1)"),
    Spec("fp8_e4m3", 16, 128, 128, 8192, "fp8", 4, ("loguniform", 1, 8192), ("uniform", 0, 2048),
         description="B=16, n log-uniform [1,8192], prior~U[0,2048], H=128, P=128, T=8192, "
                     "fp8 e4m3 with per-tensor Q/K/V scales and per-token K_rope scales"),
]
CONFIG_BY_NAME = {c.name: c for c in CONFIGS}


@dataclass
class Workload:
    spec: Spec
    n: np.ndarray              # int64 [B] new tokens per sequence
    prior: np.ndarray          # int64 [B] previously cached tokens per sequence
    row_offsets: np.ndarray    # uint32 [B+1] ragged Q offsets
    cache_lens: np.ndarray     # uint32 [B] prior lengths
    q: torch.Tensor            # [Tq, H, 192] bf16, or uint8 e4m3 codes
    k_nope: torch.Tensor       # [Sk, H, 128]
    v: torch.Tensor            # [Sk, H, 128]
    k_rope_pool: torch.Tensor  # [num_pages, P, row_width]
    page_table: np.ndarray     # uint32 [B, max_pages]
    scale: float               # softmax scale applied to QK^T
    q_scale: Optional[float] = None
    k_scale: Optional[object] = None   # float, or float32 [S_k] (one scale per K row)
    v_scale: Optional[float] = None
    k_rope_scales: Optional[torch.Tensor] = None  # float32 [num_pages, P]
    extra: dict = field(default_factory=dict)

    @property
    def batch(self):
        return self.spec.batch

    @property
    def heads(self):
        return self.spec.heads

    @property
    def page_size(self):
        return self.spec.page_size

    @property
    def total_q(self):
        return int(self.row_offsets[-1])

    @property
    def total_k(self):
        return int((self.n + self.prior).sum())

    @property
    def num_pages(self):
        return int(self.k_rope_pool.shape[0])


def _lengths(rng, recipe, batch, what):
    kind = recipe[0]
    if kind == "zero":
        return np.zeros(batch, dtype=np.int64)
    if kind == "fixed":
        v = recipe[1]
        if isinstance(v, (tuple, list)):
            assert len(v) == batch, f"{what}: {len(v)} fixed values for batch {batch}"
            return np.asarray(v, dtype=np.int64)
        return np.full(batch, int(v), dtype=np.int64)
    if kind == "uniform":
        return rng.integers(recipe[1], recipe[2] + 1, size=batch).astype(np.int64)
    if kind == "loguniform":
        lo, hi = recipe[1], recipe[2]
        u = rng.uniform(math.log(lo), math.log(hi + 1), size=batch)
        return np.clip(np.floor(np.exp(u)), lo, hi).astype(np.int64)
    if kind == "list":
        return np.asarray(recipe[1], dtype=np.int64)
    raise ValueError(f"unknown length recipe {recipe!r}")


def _normal_bf16(rng, numel, value_scale):
    out = torch.empty(numel, dtype=torch.bfloat16)
    for s in range(0, numel, _CHUNK):
        e = min(numel, s + _CHUNK)
        x = rng.standard_normal(e - s, dtype=np.float32)
        if value_scale != 1.0:
            x *= np.float32(value_scale)
        out[s:e] = torch.from_numpy(x).to(torch.bfloat16)
    return out


def _sat_e4m3(x):
    """Saturating round-to-nearest-even cast of float32 numpy values to e4m3 codes."""
    y = np.clip(x, -FP8_MAX, FP8_MAX)
    return torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8)


def _normal_fp8_per_tensor(rng, numel, value_scale):
    """e4m3 codes with one scale amax/448; two passes over the same draws."""
    state = rng.bit_generator.state
    amax = np.float32(0.0)
    for s in range(0, numel, _CHUNK):
        e = min(numel, s + _CHUNK)
        x = rng.standard_normal(e - s, dtype=np.float32) * np.float32(value_scale)
        if e > s:
            amax = max(amax, np.float32(np.abs(x).max()))
    rng.bit_generator.state = state
    sc = np.float32(amax) / np.float32(FP8_MAX) if amax > 0 else np.float32(1.0)
    codes = torch.empty(numel, dtype=torch.uint8)
    for s in range(0, numel, _CHUNK):
        e = min(numel, s + _CHUNK)
        x = rng.standard_normal(e - s, dtype=np.float32) * np.float32(value_scale)
        codes[s:e] = _sat_e4m3(x / sc)
    return codes, float(sc)


def generate(spec: Spec, n: Optional[Sequence[int]] = None,
             prior: Optional[Sequence[int]] = None) -> Workload:
    """Draw one workload.  ``n`` / ``prior`` override the length recipes."""
    rng = np.random.Generator(np.random.PCG64(spec.seed))
    B, H, P = spec.batch, spec.heads, spec.page_size
    n_arr = _lengths(rng, spec.new_len, B, "new_len")
    prior_arr = _lengths(rng, spec.prior_len, B, "prior_len")
    if n is not None:
        n_arr = np.asarray(n, dtype=np.int64)
    if prior is not None:
        prior_arr = np.asarray(prior, dtype=np.int64)
    assert n_arr.shape == (B,) and prior_arr.shape == (B,)
    L = n_arr + prior_arr
    row_offsets = np.zeros(B + 1, dtype=np.uint32)
    row_offsets[1:] = np.cumsum(n_arr).astype(np.uint32)
    cache_lens = prior_arr.astype(np.uint32)

    pages_per_seq = (L + P - 1) // P
    n_pages = int(pages_per_seq.sum())
    perm = rng.permutation(n_pages + 1)
    max_pages = max(int(pages_per_seq.max()) if B else 0, 1)
    page_table = np.zeros((B, max_pages), dtype=np.uint32)
    logical = 0
    for b in range(B):
        for k in range(int(pages_per_seq[b])):
            page_table[b, k] = perm[logical]
            logical += 1

    Tq = int(n_arr.sum())
    Sk = int(L.sum())
    W = spec.row_width
    assert W >= ROPE_DEPTH and 0 <= spec.rope_col <= W - ROPE_DEPTH
    fp8 = spec.dtype == "fp8"
    extra = {}
    if not fp8:
        q = _normal_bf16(rng, Tq * H * Q_DEPTH, spec.value_scale).view(Tq, H, Q_DEPTH)
        k_nope = _normal_bf16(rng, Sk * H * NOPE_DEPTH, spec.value_scale).view(Sk, H, NOPE_DEPTH)
        v = _normal_bf16(rng, Sk * H * V_DEPTH, spec.value_scale).view(Sk, H, V_DEPTH)
        rope_vals = _normal_bf16(rng, Sk * ROPE_DEPTH, spec.value_scale).view(Sk, ROPE_DEPTH)
        pool = torch.full((n_pages + 1, P, W), float("nan"), dtype=torch.bfloat16)
        q_scale = k_scale = v_scale = None
        rope_scales = None
    else:
        qc, q_scale = _normal_fp8_per_tensor(rng, Tq * H * Q_DEPTH, spec.value_scale)
        kc, k_scale = _normal_fp8_per_tensor(rng, Sk * H * NOPE_DEPTH, spec.value_scale)
        vc, v_scale = _normal_fp8_per_tensor(rng, Sk * H * V_DEPTH, spec.value_scale)
        q = qc.view(Tq, H, Q_DEPTH)
        k_nope = kc.view(Sk, H, NOPE_DEPTH)
        v = vc.view(Sk, H, V_DEPTH)
        x = rng.standard_normal(Sk * ROPE_DEPTH, dtype=np.float32).reshape(Sk, ROPE_DEPTH)
        x *= np.float32(spec.value_scale)
        amax = np.abs(x).max(axis=1) if Sk else np.zeros(0, np.float32)
        row_scale = np.where(amax > 0, amax / np.float32(FP8_MAX), np.float32(1.0)).astype(np.float32)
        rope_vals = _sat_e4m3(x / row_scale[:, None]).view(Sk, ROPE_DEPTH)
        pool = torch.full((n_pages + 1, P, W), FP8_NAN_CODE, dtype=torch.uint8)
        rope_scales = torch.full((n_pages + 1, P), float("nan"), dtype=torch.float32)
        extra["rope_row_scale"] = row_scale

    # Scatter each sequence's K_rope rows into its pages.
    flat = pool.view((n_pages + 1) * P, W)
    g = 0
    for b in range(B):
        Lb = int(L[b])
        if Lb == 0:
            continue
        j = np.arange(Lb)
        slots = page_table[b, j // P].astype(np.int64) * P + (j % P)
        idx = torch.from_numpy(slots)
        flat[idx, spec.rope_col:spec.rope_col + ROPE_DEPTH] = rope_vals[g:g + Lb]
        if fp8:
            rope_scales.view(-1)[idx] = torch.from_numpy(extra["rope_row_scale"][g:g + Lb])
        g += Lb

    return Workload(spec=spec, n=n_arr, prior=prior_arr, row_offsets=row_offsets,
                    cache_lens=cache_lens, q=q, k_nope=k_nope, v=v, k_rope_pool=pool,
                    page_table=page_table, scale=1.0 / math.sqrt(Q_DEPTH),
                    q_scale=q_scale, k_scale=k_scale, v_scale=v_scale,
                    k_rope_scales=rope_scales, extra=extra)


def config(name_or_index) -> Spec:
    if isinstance(name_or_index, int):
        return CONFIGS[name_or_index]
    return CONFIG_BY_NAME[name_or_index]


def custom(n, prior, heads=2, page_size=16, dtype="bf16", seed=100, value_scale=1.0,
           mask="causal", row_width=ROPE_DEPTH, rope_col=0, buffer_token_size=64) -> Workload:
    """A small workload with explicit lengths, for edge-case tests."""
    n = list(n)
    prior = list(prior)
    spec = Spec(f"custom_s{seed}", len(n), heads, page_size, buffer_token_size, dtype, seed,
                ("list", n), ("list", prior), value_scale=value_scale, mask=mask,
                row_width=row_width, rope_col=rope_col)
    return generate(spec)


def with_mask(spec: Spec, mask: str) -> Spec:
    return replace(spec, mask=mask)


def device_inputs(w: Workload, device="cuda", pin=False):
    """The workload's tensors on `device` (or pinned host memory when
    device == "cpu" and pin=True): offsets and the page table as int32 holding
    the uint32 values, fp8 scales as float32 tensors."""
    def mv(t):
        t = t.contiguous()
        if device == "cpu":
            return t.pin_memory() if pin else t
        return t.to(device, non_blocking=True)

    d = {
        "q": mv(w.q),
        "k_nope": mv(w.k_nope),
        "v": mv(w.v),
        "k_rope_pool": mv(w.k_rope_pool),
        "page_table": mv(torch.from_numpy(w.page_table.astype(np.int32))),
        "row_offsets": mv(torch.from_numpy(w.row_offsets.astype(np.int32))),
        "cache_lens": mv(torch.from_numpy(w.cache_lens.astype(np.int32))),
    }
    if w.spec.dtype == "fp8":
        d["q_scale"] = mv(torch.tensor([w.q_scale], dtype=torch.float32))
        d["k_scale"] = mv(torch.from_numpy(np.atleast_1d(np.asarray(w.k_scale, dtype=np.float32)).copy()))
        d["v_scale"] = mv(torch.tensor([w.v_scale], dtype=torch.float32))
        d["k_rope_scales"] = mv(w.k_rope_scales)
    return d


def per_token_k(w: Workload, spread_log2: float = 2.0) -> Workload:
    """The fp8 workload `w` with K_nope re-quantised per K row: row t's real
    values (code * k_scale) are multiplied by 2^u_t, u_t ~ U(-spread_log2,
    spread_log2) from a generator of its own (seed + 20011), then cast to e4m3
    with the row's own scale amax_row / 448 (saturating, round to nearest
    even).  Every other tensor is w's.  k_scale becomes float32 [S_k]."""
    assert w.spec.dtype == "fp8", "per-token K scales are for fp8 workloads"
    rng = np.random.Generator(np.random.PCG64(w.spec.seed + 20011))
    Sk = w.total_k
    factor = np.exp2(rng.uniform(-spread_log2, spread_log2, size=Sk)).astype(np.float32)
    real = w.k_nope.view(torch.float8_e4m3fn).float().numpy() * np.float32(w.k_scale)
    real = real.reshape(Sk, -1) * factor[:, None]
    amax = np.abs(real).max(axis=1) if Sk else np.zeros(0, np.float32)
    row_scale = np.where(amax > 0, amax / np.float32(FP8_MAX), np.float32(1.0)).astype(np.float32)
    codes = _sat_e4m3((real / row_scale[:, None]).astype(np.float32)).view(w.k_nope.shape)
    return replace(w, k_nope=codes, k_scale=row_scale)


def contiguous_rope(w: Workload):
    """The same K_rope laid out contiguously, as a cache without pages holds it:
    row G_b + j = the pool row of key j of sequence b (the page table's
    placement undone).  Returns ([S_k, row_width] tensor of the pool's dtype,
    [S_k] float32 per-row scales or None for bf16)."""
    P = w.page_size
    slots = np.empty(w.total_k, dtype=np.int64)
    G = 0
    for b in range(w.batch):
        L = int(w.n[b] + w.prior[b])
        j = np.arange(L)
        slots[G:G + L] = w.page_table[b, j // P].astype(np.int64) * P + j % P
        G += L
    idx = torch.from_numpy(slots)
    rows = w.k_rope_pool.reshape(-1, w.k_rope_pool.shape[-1])[idx].contiguous()
    scales = None
    if w.spec.dtype == "fp8":
        scales = w.k_rope_scales.reshape(-1)[idx].contiguous()
    return rows, scales


KV_LORA_RANK = 512   # latent width of a DeepSeek-V3 MLA cache row (rope dims follow)


def latent_cache(w: Workload, kv_lora_rank: int = KV_LORA_RANK):
    """A paged latent cache for workload `w` (bf16 only): every pool row is
    [c_kv (kv_lora_rank values) | the workload's 64 K_rope values], placed
    through w's page table, plus synthetic up-projection weights W_UK, W_UV of
    shape [H * 128, kv_lora_rank] (nn.Linear layout: output features first).

    Draws from its own generator (seed + 10007).  c_kv ~ value_scale * N(0,1)
    and weights ~ N(0, 1/kv_lora_rank), so the projected K_nope / V entries
    have about the spread of c_kv.  Slack slots and the spare page are NaN.
    Returns (pool [num_pages, P, kv_lora_rank + 64] bf16, w_uk, w_uv)."""
    assert w.spec.dtype == "bf16", "the latent cache is drawn for bf16 workloads"
    rng = np.random.Generator(np.random.PCG64(w.spec.seed + 10007))
    H, P = w.heads, w.page_size
    Sk = w.total_k
    c_kv = _normal_bf16(rng, Sk * kv_lora_rank, w.spec.value_scale).view(Sk, kv_lora_rank)
    std = 1.0 / math.sqrt(kv_lora_rank)
    w_uk = _normal_bf16(rng, H * NOPE_DEPTH * kv_lora_rank, std).view(H * NOPE_DEPTH, kv_lora_rank)
    w_uv = _normal_bf16(rng, H * V_DEPTH * kv_lora_rank, std).view(H * V_DEPTH, kv_lora_rank)
    width = kv_lora_rank + ROPE_DEPTH
    pool = torch.full((w.num_pages, P, width), float("nan"), dtype=torch.bfloat16)
    flat = pool.view(-1, width)
    src = w.k_rope_pool.view(-1, w.k_rope_pool.shape[-1])
    c0 = w.spec.rope_col
    g = 0
    for b in range(w.batch):
        L = int(w.n[b] + w.prior[b])
        j = np.arange(L)
        idx = torch.from_numpy(w.page_table[b, j // P].astype(np.int64) * P + j % P)
        flat[idx, :kv_lora_rank] = c_kv[g:g + L]
        flat[idx, kv_lora_rank:] = src[idx, c0:c0 + ROPE_DEPTH]
        g += L
    return pool, w_uk, w_uv
