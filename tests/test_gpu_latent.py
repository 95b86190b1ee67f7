"""The latent-cache path on the GPU (mla_prefill_plan, then per buffer row
mla_gather_up_project and mla_prefill_ragged_chunk with K_rope read from the
latent cache, then mla_prefill_merge or the in-place fold) versus the float64
oracle, plus the stand-alone gather (mla_gather_rows) and GEMM (mla_up_project).

* The gather moves bits: compared exactly with the oracle's token-by-token
  gather.
* The up-projections (plain, and fused with the row gather): bf16 output of
  an fp32-accumulated GEMM against the float64 product of the gathered rows,
  |err| <= 1e-2 + 1e-2 |ref| (the bf16 rounding of the output is 2^-9
  relative; the fp32 sum over 512 terms adds far less).
* The merged attention output against the oracle's attention over the
  float64-projected K/V, with the attention tolerance 2e-2 + 2e-2 |ref|.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import latent as olat
from oracle import plan as oplan

pytestmark = pytest.mark.gpu


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _close(got, ref, tol, what):
    sel = ~np.isnan(ref)
    g, r = got[sel], ref[sel]
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - r)
    bad = err > tol + tol * np.abs(r)
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} out of tolerance, max err {err.max():.4g}"


def _setup(n, prior, heads=2, page_size=16, seed=900, mask="causal"):
    w = workloads.custom(n, prior, heads=heads, page_size=page_size, seed=seed, mask=mask)
    pool, w_uk, w_uv = workloads.latent_cache(w)
    return w, pool, w_uk, w_uv


@pytest.mark.parametrize("T,page", [(64, 16), (100, 16), (1000, 128), (37, 12)])
def test_gather_rows_exact(lib, T, page):
    from mla_ragged_paged_gb300 import binding
    w, pool, _, _ = _setup([150, 0, 40, 300], [70, 9, 0, 129], page_size=page, seed=901)
    d = workloads.device_inputs(w)
    cache = pool.cuda()
    R = oplan.num_rows(w.row_offsets, w.prior, T)
    bro, co, blen, _ = oplan.plan_formula(w.row_offsets, w.prior, T, R)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for r in range(R):
        dst = torch.full((T, pool.shape[-1]), float("nan"), dtype=torch.bfloat16, device="cuda")
        b_r = torch.from_numpy(bro[r].astype(np.int32)).cuda()
        c_r = torch.from_numpy(co[r].astype(np.int32)).cuda()
        binding.gather_rows(dst, cache, d["page_table"], b_r, c_r, status)
        got = _f64(dst)
        ref = olat.gather_row(pool, w.page_table, bro[r], co[r], w.page_size)
        assert np.array_equal(got[:blen[r]], ref), f"row {r}"
        assert np.isnan(got[blen[r]:]).all(), f"row {r}: positions past the row were written"
    assert int(status.item()) == 0


def test_gather_bad_page_sets_status(lib):
    from mla_ragged_paged_gb300 import binding
    w, pool, _, _ = _setup([40], [100], seed=902)
    w.page_table[0, 3] = 10 ** 6
    d = workloads.device_inputs(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dst = torch.zeros((140, pool.shape[-1]), dtype=torch.bfloat16, device="cuda")
    bro = torch.tensor([0, 140], dtype=torch.int32, device="cuda")
    co = torch.tensor([0], dtype=torch.int32, device="cuda")
    binding.gather_rows(dst, pool.cuda(), d["page_table"], bro, co, status)
    assert int(status.item()) & 0x1


@pytest.mark.parametrize("rows,heads", [(1, 1), (37, 2), (300, 16), (129, 3), (4096, 128)])
def test_up_project(lib, rows, heads):
    from mla_ragged_paged_gb300 import binding
    w = workloads.custom([rows], [0], heads=heads, page_size=128, seed=903)
    pool, w_uk, _ = workloads.latent_cache(w)
    lat = pool.view(-1, pool.shape[-1])[:rows].cuda()           # rows of the first page(s)
    out = torch.full((rows, heads * 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.up_project(out, lat[:, :512], w_uk.cuda(), status)
    hs = list(range(heads)) if heads <= 16 else [0, 63, 127]
    ref = olat.up_project(_f64(lat[:, :512]), w_uk, hs)
    _close(_f64(out).reshape(rows, heads, 128), ref, 1e-2, "up_project")
    assert int(status.item()) == 0


@pytest.mark.parametrize("T,page,heads", [(64, 16, 1), (100, 16, 3), (1000, 128, 4), (37, 12, 2),
                                          (300, 128, 16), (256, 64, 2)])
def test_gather_up_project_matches_oracle(lib, T, page, heads):
    """K_nope and V of every buffer row, projected from cache rows gathered
    inside the GEMM, against the float64 projection of the oracle's gather."""
    from mla_ragged_paged_gb300 import binding
    w, pool, w_uk, w_uv = _setup([150, 0, 40, 300], [70, 9, 0, 129], heads=heads, page_size=page,
                                 seed=904)
    d = workloads.device_inputs(w)
    cache, uk, uv = pool.cuda(), w_uk.cuda(), w_uv.cuda()
    R = oplan.num_rows(w.row_offsets, w.prior, T)
    bro, co, blen, _ = oplan.plan_formula(w.row_offsets, w.prior, T, R)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for r in range(R):
        k_out = torch.full((T, heads * 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        v_out = torch.full_like(k_out, float("nan"))
        b_r = torch.from_numpy(bro[r].astype(np.int32)).cuda()
        c_r = torch.from_numpy(co[r].astype(np.int32)).cuda()
        binding.gather_up_project(k_out, v_out, cache, uk, uv, d["page_table"], b_r, c_r, 512, status)
        lat = olat.gather_row(pool, w.page_table, bro[r], co[r], w.page_size)[:, :512]
        n = int(blen[r])
        _close(_f64(k_out)[:n].reshape(n, heads, 128), olat.up_project(lat, w_uk), 1e-2, f"K row {r}")
        _close(_f64(v_out)[:n].reshape(n, heads, 128), olat.up_project(lat, w_uv), 1e-2, f"V row {r}")
    assert int(status.item()) == 0


def test_gather_up_project_single_output_and_full_size(lib):
    """DeepSeek-V3 shapes (T = 4096, H = 128): one projection alone, then both,
    on sampled rows and heads; the two launches agree bit for bit on K."""
    from mla_ragged_paged_gb300 import binding
    w = workloads.generate(workloads.config("deepseek_v3_bf16"))
    pool, w_uk, w_uv = workloads.latent_cache(w)
    d = workloads.device_inputs(w)
    cache, uk, uv = pool.cuda(), w_uk.cuda(), w_uv.cuda()
    T = w.spec.buffer_token_size
    R = oplan.num_rows(w.row_offsets, w.prior, T)
    bro, co, blen, _ = oplan.plan_formula(w.row_offsets, w.prior, T, R)
    r = R // 2
    b_r = torch.from_numpy(bro[r].astype(np.int32)).cuda()
    c_r = torch.from_numpy(co[r].astype(np.int32)).cuda()
    H = w.heads
    k1 = torch.empty((T, H * 128), dtype=torch.bfloat16, device="cuda")
    binding.gather_up_project(k1, None, cache, uk, None, d["page_table"], b_r, c_r)
    k2, v2 = torch.empty_like(k1), torch.empty_like(k1)
    binding.gather_up_project(k2, v2, cache, uk, uv, d["page_table"], b_r, c_r)
    torch.cuda.synchronize()
    assert torch.equal(k1, k2)
    rng = np.random.default_rng(905)
    n = int(blen[r])
    sel = np.unique(np.concatenate([[0, 127, 128, n - 1], rng.integers(0, n, 12)]))
    lat = olat.gather_row(pool, w.page_table, bro[r], co[r], w.page_size)[sel, :512]
    hs = [0, 1, 64, 127]
    _close(_f64(k2)[sel].reshape(-1, H, 128), olat.up_project(lat, w_uk, hs), 1e-2, "K full size")
    _close(_f64(v2)[sel].reshape(-1, H, 128), olat.up_project(lat, w_uv, hs), 1e-2, "V full size")


def test_gather_up_project_bad_page_sets_status(lib):
    from mla_ragged_paged_gb300 import binding
    w, pool, w_uk, _ = _setup([40], [100], seed=906)
    w.page_table[0, 3] = 10 ** 6
    d = workloads.device_inputs(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros((140, w.heads * 128), dtype=torch.bfloat16, device="cuda")
    bro = torch.tensor([0, 140], dtype=torch.int32, device="cuda")
    co = torch.tensor([0], dtype=torch.int32, device="cuda")
    binding.gather_up_project(out, None, pool.cuda(), w_uk.cuda(), None, d["page_table"], bro, co, 512,
                              status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x1


def _run_latent(w, pool, w_uk, w_uv, T, fold=False):
    from mla_ragged_paged_gb300 import binding
    d = workloads.device_inputs(w)
    S = w.total_k
    R = max(1, -(-S // T))
    bro, co, blen, nrows = binding.plan(d["row_offsets"], d["cache_lens"], T, R)
    blen_h = blen.cpu().numpy()
    cache, uk, uv = pool.cuda(), w_uk.cuda(), w_uv.cuda()
    bufs = binding.LatentRowBuffers(T, w.heads)
    po, pl = binding.chunked_scratch(R, w.total_q, w.heads)
    ws = binding.alloc_workspace(w.batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask = binding.MLA_MASK_CAUSAL if w.spec.mask == "causal" else binding.MLA_MASK_NULL
    out = torch.full((w.total_q, w.heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.total_q, w.heads), dtype=torch.float32, device="cuda")
    for r in range(R):
        if fold:
            binding.prefill_latent_row(out, lse, d["q"], cache, d["page_table"], d["row_offsets"],
                                       d["cache_lens"], bro[r], co[r], uk, uv, w.scale, bufs,
                                       int(blen_h[r]), mask, ws, status, flags=binding.MLA_CHUNK_ACCUMULATE)
        else:
            binding.prefill_latent_row(po[r], pl[r], d["q"], cache, d["page_table"], d["row_offsets"],
                                       d["cache_lens"], bro[r], co[r], uk, uv, w.scale, bufs,
                                       int(blen_h[r]), mask, ws, status)
        assert binding.device_status(ws) == 0
    if not fold:
        binding.merge(out, po, pl, d["row_offsets"], bro)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return _f64(out)


@pytest.mark.parametrize("fold", [False, True])
@pytest.mark.parametrize("case", ["small_T64", "ragged_T128", "null_T200", "page12_T37"])
def test_latent_chunked_matches_oracle(lib, case, fold):
    cfg = {
        "small_T64": (dict(n=[150, 0, 40], prior=[70, 9, 0]), 64),
        "ragged_T128": (dict(n=[300, 17, 513], prior=[0, 700, 129], heads=4, page_size=128), 128),
        "null_T200": (dict(n=[100, 130], prior=[50, 300], mask="null"), 200),
        "page12_T37": (dict(n=[150, 40], prior=[70, 0], page_size=12), 37),
    }[case]
    kw, T = cfg
    w, pool, w_uk, w_uv = _setup(seed=910 + len(case), **kw)
    got = _run_latent(w, pool, w_uk, w_uv, T, fold)
    _close(got, olat.reference(w, pool, w_uk, w_uv), 2e-2, case)


def test_latent_full_size_sampled(lib):
    """DeepSeek-V3 shapes (B=8, H=128, T=4096), sampled rows and heads."""
    w = workloads.generate(workloads.config("deepseek_v3_bf16"))
    pool, w_uk, w_uv = workloads.latent_cache(w)
    got = _run_latent(w, pool, w_uk, w_uv, w.spec.buffer_token_size, fold=True)
    assert np.isfinite(got).all()
    rng = np.random.default_rng(6)
    rows = {b: np.unique(np.concatenate([[0, int(w.n[b]) - 1], rng.integers(0, int(w.n[b]), 6)]))
            for b in (0, 3, 7)}
    ref = olat.reference(w, pool, w_uk, w_uv, heads=[0, 127], rows=rows)
    _close(got, ref, 2e-2, "deepseek_v3 latent")
