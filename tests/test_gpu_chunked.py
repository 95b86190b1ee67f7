"""Chunked execution on the GPU (mla_prefill_plan, then mla_prefill_ragged_chunk
per buffer row with mla_prefill_merge or the in-place fold, or every row in
one mla_prefill_ragged_chunked call, all through the C ABI) versus the float64
oracle.

Per row: the row's output and lse against the oracle's window function, on
every token of every sequence the row holds keys of (rows of the others must
stay untouched).  Merged: against the full-context oracle.  Tolerances are
those of the full-context call for the outputs (bf16 2e-2 + 2e-2|ref|, fp8
6e-2 + 6e-2|ref|).  lse carries no bf16 rounding (scores accumulate in fp32
from exact products and l sums unrounded exponentials), so bf16 inputs take
1e-3 + 1e-3|ref| on it; fp8 inputs, whose rope scores use K_rope rounded to
bf16 after scaling, take the output tolerance.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oatt
from oracle import chunked as och

pytestmark = pytest.mark.gpu

SENTINEL = 6144.0   # exact in bf16 and float32


def _tols(w):
    if w.spec.dtype == "fp8":
        return (6e-2, 6e-2), (6e-2, 6e-2)
    return (2e-2, 2e-2), (1e-3, 1e-3)


def _close(got, ref, atol, rtol, what):
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} out of tolerance, max err {err.max():.4g}"


def _run_rows(w, T):
    """Plan + one chunk call per row on the GPU.  Returns (bro, co, R, outs, lses, status)."""
    from mla_ragged_paged_gb300 import binding
    d = workloads.device_inputs(w)
    S = int((w.n + w.prior).sum())
    R = max(1, -(-S // T))
    bro, co, blen, nrows = binding.plan(d["row_offsets"], d["cache_lens"], T, R)
    assert int(nrows.cpu()[0]) == R
    pool = d["k_rope_pool"][..., w.spec.rope_col:w.spec.rope_col + 64]
    slots = w.num_pages * w.page_size if w.spec.dtype == "fp8" else None
    ws = binding.alloc_workspace(w.batch, fp8_pool_slots=slots)
    mask = binding.MLA_MASK_CAUSAL if w.spec.mask == "causal" else binding.MLA_MASK_NULL
    po = torch.full((R, w.total_q, w.heads, 128), SENTINEL, dtype=torch.bfloat16, device="cuda")
    pl = torch.full((R, w.total_q, w.heads), SENTINEL, dtype=torch.float32, device="cuda")
    status = 0
    for r in range(R):
        lo, hi = r * T, min((r + 1) * T, S)
        binding.prefill_ragged_chunk(po[r], pl[r], d["q"], d["k_nope"][lo:hi], d["v"][lo:hi], pool,
                                     d["page_table"], d["row_offsets"], d["cache_lens"], bro[r], co[r],
                                     w.scale, mask, ws, q_scale=d.get("q_scale"),
                                     k_scale=d.get("k_scale"), v_scale=d.get("v_scale"),
                                     k_rope_scales=d.get("k_rope_scales"))
        status |= binding.device_status(ws)
    merged = torch.full((w.total_q, w.heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    binding.merge(merged, po, pl, d["row_offsets"], bro)
    torch.cuda.synchronize()
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    return (bro.cpu().numpy().astype(np.int64), co.cpu().numpy().astype(np.int64), R,
            f(po), f(pl), f(merged), status)


def _check_rows(w, bro, co, R, po, pl):
    (oa, orr), (la, lr) = _tols(w)
    for r in range(R):
        ref_o, ref_l = och.window_reference(w, bro[r], co[r])
        held = ~np.isnan(ref_l)                                  # [Tq, H]
        assert np.array_equal(held.any(axis=1), held.all(axis=1))
        assert (po[r][~held] == SENTINEL).all() and (pl[r][~held] == SENTINEL).all(), \
            f"row {r}: tokens of absent sequences were written"
        if not held.any():
            continue
        none = held & np.isneginf(ref_l)
        assert np.isneginf(pl[r][none]).all() and (po[r][none] == 0).all(), f"row {r}: empty rows"
        seen = held & np.isfinite(ref_l)
        _close(po[r][seen], ref_o[seen], oa, orr, f"row {r} out")
        _close(pl[r][seen], ref_l[seen], la, lr, f"row {r} lse")


CASES = {
    "tiny_T32": ("tiny_bf16", None, 32),
    "ragged_T1024": ("ragged_chunked_bf16", None, 1024),
    "ragged_T128": ("ragged_chunked_bf16", None, 128),
    "ragged_T100_gather": ("ragged_chunked_bf16", None, 100),
    "T1_one_key_rows": (None, dict(n=[5, 0, 9], prior=[3, 2, 0], page_size=4), 1),
    "page12_T37": (None, dict(n=[150, 40], prior=[70, 0], page_size=12), 37),
    "null_mask_T200": (None, dict(n=[100, 130], prior=[50, 300], mask="null"), 200),
    "latent576_T64": (None, dict(n=[140, 60], prior=[10, 130], row_width=576, rope_col=512,
                                 page_size=64), 64),
    "long_prior_T300": (None, dict(n=[700, 3], prior=[1100, 900], page_size=128), 300),
    "fp8_T100": (None, dict(n=[300, 17, 513], prior=[0, 700, 129], heads=4, page_size=128,
                            dtype="fp8"), 100),
    "fp8_T256_page16": (None, dict(n=[260, 20, 513], prior=[1, 0, 300], heads=3, page_size=16,
                                   dtype="fp8"), 256),
}


@pytest.mark.parametrize("case", list(CASES))
def test_chunked_rows_and_merge(lib, case):
    name, kw, T = CASES[case]
    if name is not None:
        w = workloads.generate(workloads.config(name))
    else:
        kw = dict(dict(heads=2, page_size=16, seed=700 + list(CASES).index(case)), **kw)
        n, prior = kw.pop("n"), kw.pop("prior")
        w = workloads.custom(n, prior, **kw)
    bro, co, R, po, pl, merged, status = _run_rows(w, T)
    assert status == 0
    _check_rows(w, bro, co, R, po, pl)
    ref = oatt.reference(w)
    (oa, orr), _ = _tols(w)
    assert np.isfinite(merged).all()
    _close(merged, ref, oa, orr, f"{case} merged")


def test_window_outside_context_sets_status(lib):
    from mla_ragged_paged_gb300 import binding
    w = workloads.custom([10, 6], [4, 0], heads=2, page_size=16, seed=720)
    d = workloads.device_inputs(w)
    pool = d["k_rope_pool"][..., :64]
    ws = binding.alloc_workspace(w.batch)
    out = torch.zeros((w.total_q, w.heads, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((w.total_q, w.heads), dtype=torch.float32, device="cuda")
    # Sequence 0 has 14 context tokens; a window of 8 from position 10 leaves it.
    bro = torch.tensor([0, 8, 8], dtype=torch.int32, device="cuda")
    co = torch.tensor([10, 0], dtype=torch.int32, device="cuda")
    binding.prefill_ragged_chunk(out, lse, d["q"], d["k_nope"][:8], d["v"][:8], pool, d["page_table"],
                                 d["row_offsets"], d["cache_lens"], bro, co, w.scale,
                                 binding.MLA_MASK_CAUSAL, ws)
    assert binding.device_status(ws) & 0x4


def _sample_rows(w, per_seq=10, seed=1):
    rng = np.random.default_rng(seed)
    rows = {}
    for b in range(w.batch):
        n = int(w.n[b])
        if n:
            fixed = [0, n - 1] + [x for x in (127, 128, 255, 256) if x < n]
            rows[b] = np.unique(np.concatenate([fixed, rng.integers(0, n, size=per_seq)]))
    return rows


@pytest.mark.parametrize("name", ["deepseek_v3_bf16", "fp8_e4m3"])
def test_full_size_chunked_sampled(lib, name):
    """The chunked path at full size with the configuration's buffer_token_size
    (the plan's rows cut sequences mid-context), sampled against the oracle."""
    from mla_ragged_paged_gb300 import binding
    w = workloads.generate(workloads.config(name))
    d = workloads.device_inputs(w)
    T = w.spec.buffer_token_size
    S = int((w.n + w.prior).sum())
    pool = d["k_rope_pool"][..., w.spec.rope_col:w.spec.rope_col + 64]
    out = torch.full((w.total_q, w.heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    slots = w.num_pages * w.page_size if w.spec.dtype == "fp8" else None
    ws = binding.alloc_workspace(w.batch, fp8_pool_slots=slots)
    binding.prefill_chunked(out, d["q"], d["k_nope"], d["v"], pool, d["page_table"], d["row_offsets"],
                            d["cache_lens"], w.scale, T, -(-S // T), workspace=ws, q_scale=d.get("q_scale"),
                            k_scale=d.get("k_scale"), v_scale=d.get("v_scale"),
                            k_rope_scales=d.get("k_rope_scales"))
    assert binding.device_status(ws) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    heads = [0, w.heads // 2, w.heads - 1]
    ref = oatt.reference(w, heads=heads, rows=_sample_rows(w))
    sel = ~np.isnan(ref)
    (oa, orr), _ = _tols(w)
    _close(got[sel], ref[sel], oa, orr, name)


def _case_workload(case):
    name, kw, T = CASES[case]
    if name is not None:
        return workloads.generate(workloads.config(name)), T
    kw = dict(dict(heads=2, page_size=16, seed=750 + list(CASES).index(case)), **kw)
    n, prior = kw.pop("n"), kw.pop("prior")
    return workloads.custom(n, prior, **kw), T


def _full_window(w):
    from oracle import plan as oplan
    bro, co, _, R = oplan.plan_formula(w.row_offsets, w.prior, max(1, w.total_k), 1)
    assert R == 1
    return bro[0], co[0]


@pytest.mark.parametrize("case", ["tiny_T32", "ragged_T100_gather", "T1_one_key_rows", "page12_T37",
                                  "null_mask_T200", "long_prior_T300", "fp8_T100"])
def test_chunked_fold_in_place(lib, case):
    """MLA_CHUNK_ACCUMULATE: one mla_prefill_ragged_chunk per row, folded into
    out / lse in row order, no merge; out must be the full-context result and
    lse the full-context lse."""
    from mla_ragged_paged_gb300 import binding
    w, T = _case_workload(case)
    d = workloads.device_inputs(w)
    pool = d["k_rope_pool"][..., w.spec.rope_col:w.spec.rope_col + 64]
    slots = w.num_pages * w.page_size if w.spec.dtype == "fp8" else None
    ws = binding.alloc_workspace(w.batch, fp8_pool_slots=slots)
    mask = binding.MLA_MASK_CAUSAL if w.spec.mask == "causal" else binding.MLA_MASK_NULL
    out = torch.full((w.total_q, w.heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.total_q, w.heads), float("nan"), dtype=torch.float32, device="cuda")
    S = w.total_k
    R = -(-S // T)
    bro, co, _, _ = binding.plan(d["row_offsets"], d["cache_lens"], T, R)
    for r in range(R):
        lo, hi = r * T, min((r + 1) * T, S)
        binding.prefill_ragged_chunk(out, lse, d["q"], d["k_nope"][lo:hi], d["v"][lo:hi], pool,
                                     d["page_table"], d["row_offsets"], d["cache_lens"], bro[r], co[r],
                                     w.scale, mask, ws, q_scale=d.get("q_scale"), k_scale=d.get("k_scale"),
                                     v_scale=d.get("v_scale"), k_rope_scales=d.get("k_rope_scales"),
                                     flags=binding.MLA_CHUNK_ACCUMULATE)
        assert binding.device_status(ws) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    got_lse = lse.cpu().numpy().astype(np.float64)
    (oa, orr), (la, lr) = _tols(w)
    assert np.isfinite(got).all() and np.isfinite(got_lse).all()
    _close(got, oatt.reference(w), oa, orr, f"{case} folded out")
    _, ref_lse = och.window_reference(w, *_full_window(w))
    _close(got_lse, ref_lse, la, lr, f"{case} folded lse")


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("spare_rows", [0, 3])
def test_chunked_single_call(lib, case, spare_rows):
    """mla_prefill_ragged_chunked: the plan, then all its rows in one call over
    the rows' K buffers stacked T rows apart; out and lse must be the
    full-context result.  With spare plan capacity (max_rows > R) the unused
    rows are not read."""
    from mla_ragged_paged_gb300 import binding
    w, T = _case_workload(case)
    d = workloads.device_inputs(w)
    pool = d["k_rope_pool"][..., w.spec.rope_col:w.spec.rope_col + 64]
    slots = w.num_pages * w.page_size if w.spec.dtype == "fp8" else None
    ws = binding.alloc_workspace(w.batch, fp8_pool_slots=slots)
    mask = binding.MLA_MASK_CAUSAL if w.spec.mask == "causal" else binding.MLA_MASK_NULL
    out = torch.full((w.total_q, w.heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.total_q, w.heads), float("nan"), dtype=torch.float32, device="cuda")
    R = -(-w.total_k // T)
    binding.prefill_chunked(out, d["q"], d["k_nope"], d["v"], pool, d["page_table"], d["row_offsets"],
                            d["cache_lens"], w.scale, T, R + spare_rows, mask=mask, workspace=ws,
                            q_scale=d.get("q_scale"), k_scale=d.get("k_scale"), v_scale=d.get("v_scale"),
                            k_rope_scales=d.get("k_rope_scales"), lse=lse)
    assert binding.device_status(ws) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    got_lse = lse.cpu().numpy().astype(np.float64)
    (oa, orr), (la, lr) = _tols(w)
    _close(got, oatt.reference(w), oa, orr, f"{case} out")
    _, ref_lse = och.window_reference(w, *_full_window(w))
    _close(got_lse, ref_lse, la, lr, f"{case} lse")


def test_chunked_single_call_checks_the_plan(lib):
    """A plan row that disagrees with the stacked layout, or a row count that
    leaves a sequence's last row out, skips the sequences concerned and sets
    MLA_DEVICE_STATUS_BAD_OFFSETS; the other sequences are still correct."""
    from mla_ragged_paged_gb300 import binding
    w = workloads.custom([150, 40, 90], [70, 0, 30], heads=2, page_size=16, seed=790)
    d = workloads.device_inputs(w)
    T = 64
    R = -(-w.total_k // T)
    bro, co, _, nrows = binding.plan(d["row_offsets"], d["cache_lens"], T, R)
    ws = binding.alloc_workspace(w.batch)
    ref = oatt.reference(w)
    q0 = [int(x) for x in w.row_offsets]
    # Sequence 1 starts inside row 3 (G_1 = 220) at its context position 0:
    # claim position 1 there instead.
    bad_co = co.clone()
    bad_co[3, 1] += 1
    out = torch.full((w.total_q, w.heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    binding.prefill_ragged_chunked(out, d["q"], d["k_nope"], d["v"], d["k_rope_pool"], d["page_table"],
                                   d["row_offsets"], d["cache_lens"], bro, bad_co, nrows, T, w.scale,
                                   workspace=ws)
    assert binding.device_status(ws) & 0x4
    got = out.float().cpu().numpy().astype(np.float64)
    for b in (0, 2):
        sl = slice(q0[b], q0[b + 1])
        _close(got[sl], ref[sl], 2e-2, 2e-2, f"sequence {b}")
    # One row fewer than the plan needs: the last sequence's last row is missing.
    short = torch.tensor([R - 1], dtype=torch.int32, device="cuda")
    out.fill_(float("nan"))
    binding.prefill_ragged_chunked(out, d["q"], d["k_nope"], d["v"], d["k_rope_pool"], d["page_table"],
                                   d["row_offsets"], d["cache_lens"], bro, co, short, T, w.scale,
                                   workspace=ws)
    assert binding.device_status(ws) & 0x4
    got = out.float().cpu().numpy().astype(np.float64)
    for b in (0, 1):
        sl = slice(q0[b], q0[b + 1])
        _close(got[sl], ref[sl], 2e-2, 2e-2, f"sequence {b}")
