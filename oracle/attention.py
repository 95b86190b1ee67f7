"""Ragged causal MLA prefill attention in float64 (test infrastructure only).

What is computed, per the flare_mla_prefill page:
* q is [total_q_tokens, num_heads, 192] (Args: q); k (the nope part) and v are
  [cache_len, num_heads, 128] (Args: k, v); the rope part of K is 64 wide,
  lives in the paged cache and is shared by every head (description: the
  missing 64 elements of each K head are "retrieved from the K cache, and
  broadcasted to all the heads"; Args: k_rope).
* Query offsets are cumulative, offsets[b]..offsets[b+1] (Args: valid_length).
* scores = scale * Q K^T (Args: scale), the mask functor applied to the
  scores (Args: mask_functor; "causal / null" on the mla_prefill_v2_ragged
  page, Args: mask_functor), softmax over keys, times V; the output is 128
  wide (description: "output has reduced dimension").
* fp8 inputs are dequantised as code value times scale, K_rope with one scale
  per cached token (the k_rope_scales overload); K_nope with one scale per
  tensor or, where the split-Q overload's k_scales hold one per token, one
  per K row.

Readings where the pages are silent:
* cache_lens[b] is the prior length; the query tokens of sequence b sit at
  absolute positions prior_b .. prior_b + n_b - 1 (mla_prefill_v2_ragged,
  Args: k_nope "supplies cache_length for start_pos"); its K context has
  L_b = prior_b + n_b rows, at rows G_b .. G_b + L_b - 1 of k and v with G_b
  the sum of the earlier L.
* causal: query i of sequence b sees keys j <= prior_b + i; null: all j < L_b.
* The first 128 Q dims pair with the nope K dims, the last 64 with K_rope.
* K_rope of key j of sequence b is row page_table[b, j // P] * P + j % P of
  the pool, at columns rope_col .. rope_col + 63.

For each (sequence, head) the full masked score matrix over the requested
query rows is materialised (in blocks of whole rows when it would not fit in
memory), softmax is taken by subtracting the row maximum, and the output is
P V.  Nothing is fused or reordered beyond that.
"""
import numpy as np
import torch

from .numerics import decode_bf16, decode_e4m3

NOPE, ROPE, DV = 128, 64, 128


def _raw(t: torch.Tensor, fp8: bool) -> np.ndarray:
    if fp8:
        return t.view(torch.uint8).numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def _decode(raw: np.ndarray, fp8: bool, scale) -> np.ndarray:
    """Real values of raw codes: bf16 bits, or e4m3 codes times their scale
    (a number, or one scale per leading row of `raw`)."""
    if fp8:
        s = np.asarray(scale, dtype=np.float64)
        return decode_e4m3(raw) * (s.reshape((-1,) + (1,) * (raw.ndim - 1)) if s.ndim else float(s))
    return decode_bf16(raw)


def k_scale_rows(w, rows):
    """K_nope dequantisation scale of K rows `rows`: the per-tensor scale, or
    (one scale per K row, the split-Q overload's k_scales) the rows' own."""
    if w.k_scale is None or np.ndim(w.k_scale) == 0:
        return w.k_scale
    return np.asarray(w.k_scale, dtype=np.float64).reshape(-1)[rows]


def gather_k_rope(w, b: int) -> np.ndarray:
    """K_rope rows of sequence b's whole context, one token at a time."""
    fp8 = w.spec.dtype == "fp8"
    P = w.page_size
    L = int(w.n[b] + w.prior[b])
    pool = _raw(w.k_rope_pool, fp8).reshape(-1, w.k_rope_pool.shape[-1])
    c0 = w.spec.rope_col
    scales = w.k_rope_scales.numpy().reshape(-1) if fp8 else None
    out = np.empty((L, ROPE), dtype=np.float64)
    for j in range(L):
        page = int(w.page_table[b, j // P])
        slot = page * P + j % P
        row = pool[slot, c0:c0 + ROPE]
        out[j] = _decode(row, fp8, scales[slot] if fp8 else None)
    return out


def attention_rows(q_rows, k_full, v, allowed, scale):
    """softmax(scale * q_rows k_full^T masked) v for one (sequence, head).

    q_rows [m, 192], k_full [L, 192], v [L, 128], allowed bool [m, L]."""
    s = scale * (q_rows @ k_full.T)
    s = np.where(allowed, s, -np.inf)
    s_max = s.max(axis=1, keepdims=True)
    p = np.exp(s - s_max)
    p = p / p.sum(axis=1, keepdims=True)
    return p @ v


def reference(w, heads=None, rows=None, row_block=1024, out=None, q=None):
    """Oracle output [total_q_tokens, H, 128] float64 (NaN where not computed).

    heads: iterable of head indices (default all).
    rows:  optional dict b -> array of local query indices; when given, only
           the sequences it names are computed (default: every row).
    out:   optional preallocated float64 [total_q_tokens, H, 128] to write the
           computed rows into (other entries are left untouched).
    q:     optional float64 [total_q_tokens, H, 192] query values to use
           instead of decoding w.q (Q held in another layout, e.g. split into
           q_nope and q_rope)."""
    fp8 = w.spec.dtype == "fp8"
    H = w.heads
    heads = list(range(H)) if heads is None else list(heads)
    q_raw = _raw(w.q, fp8)
    k_raw = _raw(w.k_nope, fp8)
    v_raw = _raw(w.v, fp8)
    if out is None:
        out = np.full((w.total_q, H, DV), np.nan, dtype=np.float64)
    G = 0
    for b in range(w.batch):
        n = int(w.n[b])
        prior = int(w.prior[b])
        L = prior + n
        q0 = int(w.row_offsets[b])
        if rows is None:
            sel = np.arange(n)
        else:
            sel = np.asarray(rows.get(b, []), dtype=np.int64)
        if n == 0 or sel.size == 0:
            G += L
            continue
        k_rope = gather_k_rope(w, b)
        j = np.arange(L)
        for h in heads:
            k_full = np.empty((L, NOPE + ROPE), dtype=np.float64)
            k_full[:, :NOPE] = _decode(k_raw[G:G + L, h, :], fp8, k_scale_rows(w, np.arange(G, G + L)))
            k_full[:, NOPE:] = k_rope
            v = _decode(v_raw[G:G + L, h, :], fp8, w.v_scale)
            for s0 in range(0, sel.size, row_block):
                idx = sel[s0:s0 + row_block]
                q_rows = (q[q0 + idx, h, :] if q is not None
                          else _decode(q_raw[q0 + idx, h, :], fp8, w.q_scale))
                if w.spec.mask == "causal":
                    allowed = j[None, :] <= (prior + idx)[:, None]
                else:
                    allowed = np.ones((idx.size, L), dtype=bool)
                out[q0 + idx, h, :] = attention_rows(q_rows, k_full, v, allowed, w.scale)
        G += L
    return out

