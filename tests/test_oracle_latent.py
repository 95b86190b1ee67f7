"""Pins for the latent-cache oracle (gather of buffer rows, up-projection, and
attention over the projected K/V).

* The gather is pinned to the global-packing definition of a buffer row,
  walked one context token at a time without the plan's offsets.
* The up-projection is pinned to an explicit triple loop on a small case.
* The attention over the latent cache is pinned to torch's
  scaled_dot_product_attention in float64 with K/V built by torch.einsum.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import latent as olat
from oracle import plan as oplan
from oracle.numerics import decode_bf16


def _w(mask="causal"):
    w = workloads.custom([5, 0, 9, 3], [4, 2, 0, 11], heads=2, page_size=4, seed=21, mask=mask)
    pool, w_uk, w_uv = workloads.latent_cache(w, kv_lora_rank=32)
    return w, pool, w_uk, w_uv


@pytest.mark.parametrize("T", [1, 5, 8, 100])
def test_gather_rows_follow_global_packing(T):
    w, pool, _, _ = _w()
    rows = decode_bf16(pool.view(torch.int16).numpy().view(np.uint16)).reshape(-1, pool.shape[-1])
    L = (w.n + w.prior).astype(np.int64)
    R = oplan.num_rows(w.row_offsets, w.prior, T)
    bro, co, blen, _ = oplan.plan_formula(w.row_offsets, w.prior, T, R)
    # Global position g of the batch-order packing -> (sequence, context position).
    owner = np.repeat(np.arange(w.batch), L)
    pos = np.concatenate([np.arange(x) for x in L])
    for r in range(R):
        got = olat.gather_row(pool, w.page_table, bro[r], co[r], w.page_size)
        assert got.shape[0] == blen[r]
        for i in range(int(blen[r])):
            g = r * T + i
            b, a = owner[g], pos[g]
            slot = int(w.page_table[b, a // w.page_size]) * w.page_size + a % w.page_size
            assert np.array_equal(got[i], rows[slot], equal_nan=False), (r, i)


def test_up_project_matches_loops():
    rng = np.random.default_rng(1)
    c = rng.normal(size=(3, 16))
    wt = rng.normal(size=(2 * 128, 16))
    got = olat.up_project(c, wt)
    for t in range(3):
        for h in range(2):
            for d in range(0, 128, 17):
                ref = sum(c[t, k] * wt[h * 128 + d, k] for k in range(16))
                assert got[t, h, d] == pytest.approx(ref, rel=1e-12, abs=1e-12)


@pytest.mark.parametrize("mask", ["causal", "null"])
def test_latent_attention_matches_sdpa(mask):
    w, pool, w_uk, w_uv = _w(mask)
    got = olat.reference(w, pool, w_uk, w_uv, kv_lora_rank=32)
    f = lambda t: t.to(torch.float64)
    flat = f(pool).reshape(-1, pool.shape[-1])
    P = w.page_size
    ref = torch.zeros(w.total_q, w.heads, 128, dtype=torch.float64)
    for b in range(w.batch):
        n, prior = int(w.n[b]), int(w.prior[b])
        if n == 0:
            continue
        L = n + prior
        j = torch.arange(L)
        slots = torch.as_tensor(w.page_table[b].astype(np.int64))[j // P] * P + j % P
        lat = flat[slots]
        k_nope = torch.einsum("tc,oc->to", lat[:, :32], f(w_uk)).view(L, w.heads, 128)
        v = torch.einsum("tc,oc->to", lat[:, :32], f(w_uv)).view(L, w.heads, 128)
        k = torch.cat([k_nope, lat[:, None, 32:96].expand(L, w.heads, 64)], dim=-1)
        qb = f(w.q[int(w.row_offsets[b]):int(w.row_offsets[b + 1])])
        m = (j[None, :] <= (prior + torch.arange(n))[:, None]) if mask == "causal" else None
        o = torch.nn.functional.scaled_dot_product_attention(
            qb.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1), attn_mask=m, scale=w.scale)
        ref[int(w.row_offsets[b]):int(w.row_offsets[b + 1])] = o.transpose(0, 1)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-11, atol=1e-12)


def test_latent_pool_rope_columns_are_the_workload_rope():
    w, pool, _, _ = _w()
    flat = pool.view(-1, pool.shape[-1])
    src = w.k_rope_pool.view(-1, w.k_rope_pool.shape[-1])
    P = w.page_size
    for b in range(w.batch):
        L = int(w.n[b] + w.prior[b])
        for j in range(L):
            slot = int(w.page_table[b, j // P]) * P + j % P
            assert torch.equal(flat[slot, 32:96], src[slot, :64])
