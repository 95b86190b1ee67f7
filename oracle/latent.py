"""Gathering buffer rows out of a paged latent cache and up-projecting them
to K_nope / V, in float64 (test infrastructure only).

What the pages fix:
* generic_flare_mla_prefill_ragged_paged_plan exists so that the prefill
  kernel "can gather K/V entries into a contiguous buffer" (summary), one
  buffer row of buffer_token_size tokens at a time, from the paged cache
  collection (Args: kv_collection, buffer_row_offsets, cache_offsets).
* flare_mla_prefill: K_rope is the last q_depth - depth = 64 dims of the
  cache row (Args: k_rope); mla_prefill_v2_ragged calls V "the nope segment
  of the latent cache" (Args: v).

Readings where the pages are silent:
* A cache row is [c_kv (kv_lora_rank = 512) | k_rope (64)], the DeepSeek-V3
  latent layout (576 values).
* Buffer row r holds, at position bro[b] + i, context token co[b] + i of
  sequence b (the same reading as the chunked attention).
* K_nope[t, h, :] = W_UK[h*128:(h+1)*128, :] . c_kv[t] and likewise V with
  W_UV (weights in nn.Linear layout [H*128, 512]); the weights are synthetic.
"""
import numpy as np
import torch

from .attention import DV, NOPE, ROPE, _decode, _raw, attention_rows
from .numerics import decode_bf16


def _pool_rows(pool):
    return decode_bf16(pool.view(torch.int16).numpy().view(np.uint16)).reshape(-1, pool.shape[-1])


def gather_row(pool, page_table, buffer_row_offsets, cache_offsets, page_size):
    """Buffer row [bro[B], width] float64, one token at a time."""
    rows = _pool_rows(pool)
    bro = np.asarray(buffer_row_offsets, dtype=np.int64)
    co = np.asarray(cache_offsets, dtype=np.int64)
    B = co.shape[0]
    out = np.empty((int(bro[B]), rows.shape[1]), dtype=np.float64)
    for b in range(B):
        for i in range(int(bro[b + 1] - bro[b])):
            a = int(co[b]) + i
            slot = int(page_table[b, a // page_size]) * page_size + a % page_size
            out[int(bro[b]) + i] = rows[slot]
    return out


def up_project(c_kv, weight, heads=None):
    """[n, 512] x W[H*128, 512] -> [n, H, 128] (float64 matmuls); with
    `heads`, only those heads' output columns are computed (the others are NaN)."""
    if isinstance(weight, torch.Tensor):
        weight = weight.view(torch.int16).numpy().view(np.uint16)
        wt = None
    else:
        wt = np.asarray(weight, dtype=np.float64)
    n, H = c_kv.shape[0], weight.shape[0] // 128
    out = np.full((n, H, 128), np.nan, dtype=np.float64)
    for h in (range(H) if heads is None else heads):
        wh = wt[h * 128:(h + 1) * 128] if wt is not None else decode_bf16(weight[h * 128:(h + 1) * 128])
        out[:, h, :] = c_kv @ wh.T
    return out


def context_latent(w, pool, b):
    """Cache rows of sequence b's whole context [L_b, width], one token at a time."""
    rows = _pool_rows(pool)
    P = w.page_size
    L = int(w.n[b] + w.prior[b])
    out = np.empty((L, rows.shape[1]), dtype=np.float64)
    for j in range(L):
        out[j] = rows[int(w.page_table[b, j // P]) * P + j % P]
    return out


def reference(w, pool, w_uk, w_uv, heads=None, rows=None, kv_lora_rank=512):
    """Attention output [total_q, H, 128] float64 with K_nope, V up-projected
    from the latent cache and K_rope taken from its last 64 columns (NaN where
    not computed; `heads` / `rows` as in oracle.attention.reference)."""
    H = w.heads
    heads = list(range(H)) if heads is None else list(heads)
    q_raw = _raw(w.q, False)
    out = np.full((w.total_q, H, DV), np.nan, dtype=np.float64)
    for b in range(w.batch):
        n, prior = int(w.n[b]), int(w.prior[b])
        L = n + prior
        sel = np.arange(n) if rows is None else np.asarray(rows.get(b, []), dtype=np.int64)
        if n == 0 or sel.size == 0:
            continue
        lat = context_latent(w, pool, b)
        k_nope = up_project(lat[:, :kv_lora_rank], w_uk, heads)
        v = up_project(lat[:, :kv_lora_rank], w_uv, heads)
        rope = lat[:, kv_lora_rank:kv_lora_rank + ROPE]
        q0 = int(w.row_offsets[b])
        j = np.arange(L)
        for h in heads:
            k = np.concatenate([k_nope[:, h, :], rope], axis=1)
            qh = _decode(q_raw[q0 + sel, h, :], False, None)
            if w.spec.mask == "causal":
                allowed = j[None, :] <= (prior + sel)[:, None]
            else:
                allowed = np.ones((sel.size, L), dtype=bool)
            out[q0 + sel, h, :] = attention_rows(qh, k, v[:, h, :], allowed, w.scale)
    return out
