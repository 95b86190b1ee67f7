"""Chunked execution over the plan's buffer rows, in float64 (test
infrastructure only).

What the pages fix:
* generic_flare_mla_prefill_ragged_paged_plan cuts the K context into buffer
  rows of buffer_token_size tokens and, per row, gives buffer_row_offsets
  (where each sequence's entries start in the row's contiguous K buffer) and
  cache_offsets (where they start in the paged cache);
* flare_mla_prefill takes exactly those two arrays (Args: cache_row_offsets,
  cache_offsets), so one attention call consumes one buffer row.

Readings where the pages are silent:
* Row r holds, for sequence b, W_b = bro[b+1] - bro[b] keys at context
  positions co[b] .. co[b] + W_b - 1.  Position-dependent steps use the
  absolute position: the causal mask (query i of sequence b sees position
  a <= prior_b + i) and the page lookup of K_rope.
* Each call returns the softmax-normalised output over the keys it sees and
  lse = ln sum_j exp(scale * q . k_j) over the same keys; a query row that
  sees none gets output 0 and lse = -inf.  Rows combine by the usual
  log-sum-exp weighting (merge below).

The window function reads K_nope and V at the rows of the full-context layout
(G_b + a), not through the buffer slice the CUDA path is handed, so a test
that compares the two also checks the buffer packing.
"""
import numpy as np

from .attention import DV, NOPE, ROPE, _decode, _raw, gather_k_rope, k_scale_rows


def window_reference(w, buffer_row_offsets, cache_offsets, heads=None):
    """One buffer row.  buffer_row_offsets [B+1], cache_offsets [B].

    Returns (out [total_q, H, 128], lse [total_q, H]) in float64; entries of
    sequences with no key in the row (or no query tokens) are NaN."""
    fp8 = w.spec.dtype == "fp8"
    H = w.heads
    heads = list(range(H)) if heads is None else list(heads)
    bro = np.asarray(buffer_row_offsets, dtype=np.int64)
    co = np.asarray(cache_offsets, dtype=np.int64)
    q_raw, k_raw, v_raw = _raw(w.q, fp8), _raw(w.k_nope, fp8), _raw(w.v, fp8)
    out = np.full((w.total_q, H, DV), np.nan, dtype=np.float64)
    lse = np.full((w.total_q, H), np.nan, dtype=np.float64)
    G = 0
    for b in range(w.batch):
        n, prior = int(w.n[b]), int(w.prior[b])
        L = n + prior
        W = int(bro[b + 1] - bro[b])
        c0 = int(co[b])
        if n == 0 or W == 0:
            G += L
            continue
        assert 0 <= c0 and c0 + W <= L, "window outside the sequence's context"
        a = c0 + np.arange(W)                       # absolute key positions
        rope = gather_k_rope(w, b)[a]
        q0 = int(w.row_offsets[b])
        i = np.arange(n)
        if w.spec.mask == "causal":
            allowed = a[None, :] <= (prior + i)[:, None]
        else:
            allowed = np.ones((n, W), dtype=bool)
        for h in heads:
            k = np.empty((W, NOPE + ROPE), dtype=np.float64)
            k[:, :NOPE] = _decode(k_raw[G + a, h, :], fp8, k_scale_rows(w, G + a))
            k[:, NOPE:] = rope
            v = _decode(v_raw[G + a, h, :], fp8, w.v_scale)
            qh = _decode(q_raw[q0:q0 + n, h, :], fp8, w.q_scale)
            s = np.where(allowed, w.scale * (qh @ k.T), -np.inf)
            seen = allowed.any(axis=1)
            m = np.where(seen, s.max(axis=1), 0.0)
            e = np.exp(s - m[:, None])              # 0 where masked
            tot = e.sum(axis=1)
            o = np.zeros((n, DV), dtype=np.float64)
            o[seen] = (e[seen] @ v) / tot[seen, None]
            out[q0:q0 + n, h, :] = o
            lse[q0:q0 + n, h] = np.where(seen, m + np.log(np.where(seen, tot, 1.0)), -np.inf)
        G += L
    return out, lse


def merge(outs, lses):
    """Combine per-row results: out = sum_r exp(lse_r - m) out_r / sum_r exp(lse_r - m),
    m = max_r lse_r.  NaN entries (sequence absent from a row) are skipped;
    where every row is -inf or absent the result is 0 (-inf rows) or NaN."""
    outs = np.stack(outs)                            # [R, T, H, 128]
    lses = np.stack(lses)                            # [R, T, H]
    present = ~np.isnan(lses)
    finite = present & np.isfinite(lses)
    m = np.where(finite, lses, -np.inf).max(axis=0)  # [T, H]
    m_safe = np.where(np.isfinite(m), m, 0.0)
    wgt = np.exp(np.where(finite, lses, -np.inf) - m_safe[None])   # 0 off the finite rows
    num = (wgt[..., None] * np.where(finite[..., None], outs, 0.0)).sum(axis=0)
    den = wgt.sum(axis=0)
    res = np.where(den[..., None] > 0, num / np.where(den > 0, den, 1.0)[..., None], 0.0)
    res[~present.any(axis=0)] = np.nan
    return res
