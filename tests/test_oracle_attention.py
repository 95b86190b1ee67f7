"""Pins for the float64 attention oracle.

Nothing numeric is printed on the flare_mla_prefill page, so the oracle is
pinned to mathematics and to independent library routines:
* equivalence to standard multi-head attention with a 192-wide key per head
  once K_rope is replicated per head (torch scaled_dot_product_attention in
  float64 on CPU, an explicit bottom-right causal mask, dequantisation by
  torch's own dtype casts),
* closed forms (one key gives V; scale 0 or identical keys give the mean of
  the visible V rows; normalisation),
* invariances (page placement, key order under the null mask, batch order,
  head independence),
* brute force with scalar Python arithmetic on tiny cases.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oatt
from oracle.numerics import decode_bf16, decode_e4m3


def _f64(t):
    return t.to(torch.float64)


def _sdpa_reference(w):
    """Standard MHA (d_qk = 192, d_v = 128) with K_rope copied into every head."""
    fp8 = w.spec.dtype == "fp8"
    P = w.page_size
    if fp8:
        deq = lambda t, s: _f64(t.view(torch.float8_e4m3fn)) * s
        q = deq(w.q, w.q_scale)
        ks = np.asarray(w.k_scale, dtype=np.float64)   # per tensor, or one per K row
        kn = deq(w.k_nope, torch.from_numpy(ks)[:, None, None] if ks.ndim else float(ks))
        v = deq(w.v, w.v_scale)
        pool = _f64(w.k_rope_pool.view(torch.float8_e4m3fn)) * _f64(w.k_rope_scales)[..., None]
    else:
        q, kn, v, pool = _f64(w.q), _f64(w.k_nope), _f64(w.v), _f64(w.k_rope_pool)
    pool = pool[..., w.spec.rope_col:w.spec.rope_col + 64]
    out = torch.zeros(w.total_q, w.heads, 128, dtype=torch.float64)
    G = 0
    for b in range(w.batch):
        n, prior = int(w.n[b]), int(w.prior[b])
        L = n + prior
        if n == 0:
            G += L
            continue
        pages = torch.as_tensor(w.page_table[b].astype(np.int64))
        j = torch.arange(L)
        rope = pool[pages[j // P], j % P]                                   # [L, 64]
        k = torch.cat([kn[G:G + L], rope[:, None, :].expand(L, w.heads, 64)], dim=-1)
        qb = q[int(w.row_offsets[b]):int(w.row_offsets[b + 1])]
        mask = None
        if w.spec.mask == "causal":
            mask = j[None, :] <= (prior + torch.arange(n))[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(
            qb.transpose(0, 1), k.transpose(0, 1), v[G:G + L].transpose(0, 1),
            attn_mask=mask, scale=w.scale)
        out[int(w.row_offsets[b]):int(w.row_offsets[b + 1])] = o.transpose(0, 1)
        G += L
    return out.numpy()


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("mask", ["causal", "null"])
def test_matches_standard_mha_with_replicated_rope(dtype, mask):
    w = workloads.custom([5, 1, 0, 9], [0, 3, 2, 6], heads=3, page_size=4, dtype=dtype,
                         seed=7, mask=mask)
    ref = oatt.reference(w)
    sdpa = _sdpa_reference(w)
    assert np.isfinite(ref).all()
    np.testing.assert_allclose(ref, sdpa, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mask", ["causal", "null"])
def test_per_token_k_scales_match_standard_mha(mask):
    """One K_nope scale per K row (rows re-quantised over a 2^±2 spread): the
    oracle's per-row dequantisation against SDPA on torch-dequantised keys."""
    w = workloads.per_token_k(workloads.custom([5, 1, 0, 9], [0, 3, 2, 6], heads=3, page_size=4,
                                               dtype="fp8", seed=8, mask=mask))
    assert np.ndim(w.k_scale) == 1 and len(np.unique(w.k_scale)) > w.total_k // 2
    np.testing.assert_allclose(oatt.reference(w), _sdpa_reference(w), rtol=1e-12, atol=1e-12)


def test_per_token_k_scales_equal_reduce_to_per_tensor():
    from dataclasses import replace
    w = workloads.custom([7, 3], [2, 5], heads=2, page_size=4, dtype="fp8", seed=9)
    wt = replace(w, k_scale=np.full(w.total_k, w.k_scale, dtype=np.float32))
    assert np.array_equal(oatt.reference(w), oatt.reference(wt))


def test_per_token_k_scale_of_one_row_reaches_only_its_viewers():
    """Changing key row t's scale changes exactly the query rows that see it
    (causal: its own sequence's rows at or after its position)."""
    from dataclasses import replace
    w = workloads.per_token_k(workloads.custom([6, 5], [3, 2], heads=2, page_size=4, dtype="fp8",
                                               seed=10))
    G1 = int(w.n[0] + w.prior[0])
    t = G1 + 4                                  # sequence 1, context position 4
    ks = np.array(w.k_scale, copy=True)
    ks[t] *= 3.0
    a, b = oatt.reference(w), oatt.reference(replace(w, k_scale=ks))
    changed = np.abs(a - b).max(axis=(1, 2)) > 0
    q1 = int(w.row_offsets[1])
    expect = np.zeros(w.total_q, dtype=bool)
    expect[q1 + (4 - int(w.prior[1])):] = True  # query i sees position 4 when prior + i >= 4
    assert np.array_equal(changed, expect)


def test_tiny_config_matches_standard_mha():
    w = workloads.generate(workloads.config("tiny_bf16"))
    np.testing.assert_allclose(oatt.reference(w), _sdpa_reference(w), rtol=1e-12, atol=1e-12)


def test_latent_row_layout_matches_standard_mha():
    # rope dims at the tail of a 576-wide latent row
    w = workloads.custom([6, 3], [2, 0], heads=2, page_size=8, row_width=576, rope_col=512, seed=8)
    np.testing.assert_allclose(oatt.reference(w), _sdpa_reference(w), rtol=1e-12, atol=1e-12)


def test_single_key_returns_v():
    w = workloads.custom([1, 1], [0, 0], heads=2, page_size=16, seed=3)
    ref = oatt.reference(w)
    v = decode_bf16(w.v.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(ref, v)


def test_rows_are_normalised():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((7, 192))
    k = rng.standard_normal((11, 192))
    allowed = np.tril(np.ones((7, 11), bool), k=4)
    out = oatt.attention_rows(q, k, np.ones((11, 128)), allowed, 0.3)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-14)


def _visible_mean_v(w, b, i, h):
    G = int((w.n[:b] + w.prior[:b]).sum())
    prior = int(w.prior[b])
    L = prior + int(w.n[b])
    v = decode_bf16(w.v.view(torch.int16).numpy().view(np.uint16))
    last = prior + i if w.spec.mask == "causal" else L - 1
    return v[G:G + last + 1, h].mean(axis=0)


def test_zero_scale_gives_mean_of_visible_values():
    w = workloads.custom([4, 6], [3, 0], heads=2, page_size=4, seed=11)
    w.scale = 0.0
    ref = oatt.reference(w)
    for b in range(2):
        for i in range(int(w.n[b])):
            for h in range(2):
                np.testing.assert_allclose(ref[int(w.row_offsets[b]) + i, h],
                                           _visible_mean_v(w, b, i, h), rtol=1e-13, atol=1e-13)


def test_identical_keys_give_mean_of_visible_values():
    w = workloads.custom([5], [2], heads=2, page_size=4, seed=12)
    w.k_nope[:] = w.k_nope[0:1]                      # same nope part for every key
    pool = w.k_rope_pool.view(-1, 64)
    first = int(w.page_table[0, 0]) * w.page_size
    for j in range(7):
        slot = int(w.page_table[0, j // 4]) * 4 + j % 4
        pool[slot] = pool[first]
    ref = oatt.reference(w)
    for i in range(5):
        for h in range(2):
            np.testing.assert_allclose(ref[i, h], _visible_mean_v(w, 0, i, h), rtol=1e-12, atol=1e-12)


def test_page_placement_does_not_matter():
    w = workloads.custom([7, 12], [5, 9], heads=2, page_size=4, seed=13)
    ref = oatt.reference(w)
    # move every page to a new physical position and rewrite the table
    rng = np.random.default_rng(5)
    perm = rng.permutation(w.num_pages)                 # old page p -> new page perm[p]
    new_pool = torch.full_like(w.k_rope_pool, float("nan"))
    new_pool[torch.as_tensor(perm)] = w.k_rope_pool
    w.page_table = perm[w.page_table.astype(np.int64)].astype(np.uint32)
    w.k_rope_pool = new_pool
    np.testing.assert_array_equal(oatt.reference(w), ref)


def test_key_order_does_not_matter_under_null_mask():
    w = workloads.custom([6], [5], heads=2, page_size=4, seed=14, mask="null")
    ref = oatt.reference(w)
    L = 11
    perm = np.random.default_rng(3).permutation(L)
    w.k_nope[:L] = w.k_nope[torch.as_tensor(perm)].clone()
    w.v[:L] = w.v[torch.as_tensor(perm)].clone()
    pool = w.k_rope_pool.view(-1, 64)
    slots = [int(w.page_table[0, j // 4]) * 4 + j % 4 for j in range(L)]
    rows = pool[torch.as_tensor(slots)].clone()
    pool[torch.as_tensor(slots)] = rows[torch.as_tensor(perm)]
    np.testing.assert_allclose(oatt.reference(w), ref, rtol=1e-12, atol=1e-12)


def test_batch_order_permutes_outputs():
    w = workloads.custom([3, 5, 2], [1, 0, 4], heads=2, page_size=4, seed=15)
    ref = oatt.reference(w)
    order = [2, 0, 1]
    L = (w.n + w.prior).astype(np.int64)
    G = np.concatenate([[0], np.cumsum(L)])
    ro = w.row_offsets.astype(np.int64)
    w2 = workloads.custom([int(w.n[b]) for b in order], [int(w.prior[b]) for b in order],
                          heads=2, page_size=4, seed=15)
    w2.q = torch.cat([w.q[ro[b]:ro[b + 1]] for b in order])
    w2.k_nope = torch.cat([w.k_nope[G[b]:G[b + 1]] for b in order])
    w2.v = torch.cat([w.v[G[b]:G[b + 1]] for b in order])
    w2.k_rope_pool = w.k_rope_pool
    pt = np.zeros((3, w.page_table.shape[1]), np.uint32)
    for nb, b in enumerate(order):
        pt[nb] = w.page_table[b]
    w2.page_table = pt
    ref2 = oatt.reference(w2)
    np.testing.assert_array_equal(ref2, np.concatenate([ref[ro[b]:ro[b + 1]] for b in order]))


def test_heads_are_independent():
    w = workloads.custom([6, 4], [2, 3], heads=3, page_size=4, seed=16)
    ref = oatt.reference(w)
    w.q[:, 1] = 0
    w.k_nope[:, 1] = 3
    w.v[:, 1] = -2
    ref2 = oatt.reference(w)
    np.testing.assert_array_equal(ref2[:, [0, 2]], ref[:, [0, 2]])
    assert not np.allclose(ref2[:, 1], ref[:, 1])


def test_brute_force_scalar_arithmetic():
    """n, L <= 4 with every sum written out in scalar Python."""
    w = workloads.custom([2, 3], [1, 0], heads=2, page_size=2, seed=17)
    ref = oatt.reference(w)
    q = decode_bf16(w.q.view(torch.int16).numpy().view(np.uint16))
    kn = decode_bf16(w.k_nope.view(torch.int16).numpy().view(np.uint16))
    v = decode_bf16(w.v.view(torch.int16).numpy().view(np.uint16))
    pool = decode_bf16(w.k_rope_pool.view(torch.int16).numpy().view(np.uint16)).reshape(-1, 64)
    G = 0
    for b in range(2):
        n, prior = int(w.n[b]), int(w.prior[b])
        for h in range(2):
            for i in range(n):
                t = int(w.row_offsets[b]) + i
                scores = []
                for j in range(prior + i + 1):
                    slot = int(w.page_table[b, j // 2]) * 2 + j % 2
                    s = 0.0
                    for d in range(128):
                        s += q[t, h, d] * kn[G + j, h, d]
                    for d in range(64):
                        s += q[t, h, 128 + d] * pool[slot, d]
                    scores.append(s * w.scale)
                m = max(scores)
                e = [math.exp(s - m) for s in scores]
                z = sum(e)
                for d in range(128):
                    o = sum(e[j] * v[G + j, h, d] for j in range(len(e))) / z
                    assert abs(o - ref[t, h, d]) <= 1e-12 * max(1.0, abs(o))
        G += n + prior


def test_row_subset_matches_full():
    w = workloads.custom([40, 9], [30, 0], heads=2, page_size=8, seed=18)
    full = oatt.reference(w)
    rows = {0: np.array([0, 17, 39]), 1: np.array([8])}
    part = oatt.reference(w, heads=[1], rows=rows, row_block=2)
    for b, idx in rows.items():
        t = int(w.row_offsets[b]) + idx
        np.testing.assert_allclose(part[t, 1], full[t, 1], rtol=1e-13, atol=1e-13)
    assert np.isnan(part[:, 0]).all()


def test_decoders_match_torch_casts():
    codes = np.arange(256, dtype=np.uint8)
    mine = decode_e4m3(codes)
    theirs = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(theirs))
    ok = ~np.isnan(mine)
    np.testing.assert_array_equal(mine[ok], theirs[ok])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6
    bits = np.random.default_rng(1).integers(0, 1 << 16, size=4096).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]           # drop inf/nan patterns
    mine = decode_bf16(bits)
    theirs = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(mine, theirs)


@pytest.mark.parametrize("name", ["tiny_bf16", "ragged_chunked_bf16"])
def test_generated_configs_are_finite(name):
    w = workloads.generate(workloads.config(name))
    heads = [0, w.heads - 1]
    ref = oatt.reference(w, heads=heads)
    assert np.isfinite(ref[:, heads]).all()


def test_explicit_query_values_replace_decoding():
    w = workloads.custom([6, 3], [2, 5], heads=2, page_size=4, seed=31, dtype="fp8")
    q64 = decode_e4m3(w.q.numpy()) * w.q_scale
    np.testing.assert_array_equal(oatt.reference(w, q=q64), oatt.reference(w))
    q64[:, :, 128:] *= 0.5                     # different rope queries change the result
    assert not np.allclose(oatt.reference(w, q=q64), oatt.reference(w))
