"""fp8 K_nope with one scale per K row (the split-Q overload's k_scales, read
as per-token) through every entry point that takes fp8 K, versus the float64
oracle on the same codes and scales.

Inputs: an fp8 workload whose K_nope rows are re-quantised each to its own
amax / 448 after a per-row factor 2^U(-2, 2) (workloads.per_token_k), so that
a scale applied to the wrong key, or not at all, moves scores by up to 16x.
Tolerance as for the per-tensor fp8 path: |gpu - ref| <= 6e-2 + 6e-2 |ref|.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oatt
from oracle import chunked as och
from oracle.numerics import decode_bf16, decode_e4m3

pytestmark = pytest.mark.gpu

TOL = 6e-2


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _close(got, ref, what, tol=TOL):
    sel = ~np.isnan(ref)
    assert sel.any()
    g, r = got[sel], ref[sel]
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - r)
    bad = err > tol + tol * np.abs(r)
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} out of tolerance, max err {err.max():.4g}"


def _workload(n, prior, **kw):
    kw = dict(dict(heads=2, page_size=16, dtype="fp8", seed=1200), **kw)
    return workloads.per_token_k(workloads.custom(n, prior, **kw))


def _mask(w):
    from mla_ragged_paged_gb300 import binding
    return binding.MLA_MASK_CAUSAL if w.spec.mask == "causal" else binding.MLA_MASK_NULL


def run_fused(w):
    from mla_ragged_paged_gb300 import binding
    d = workloads.device_inputs(w)
    assert d["k_scale"].numel() == w.total_k
    out = torch.full((w.total_q, w.heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    pool = d["k_rope_pool"][..., w.spec.rope_col:w.spec.rope_col + 64]
    # Converted K_rope rows at the K rows (a single K row is per-tensor as well:
    # the pool's slots then).
    rows = w.total_k if w.total_k > 1 else w.num_pages * w.page_size
    ws = binding.alloc_workspace(w.batch, fp8_pool_slots=rows)
    binding.prefill_ragged(out, d["q"], d["k_nope"], d["v"], pool, d["page_table"], d["row_offsets"],
                           d["cache_lens"], w.scale, _mask(w), ws, q_scale=d["q_scale"],
                           k_scale=d["k_scale"], v_scale=d["v_scale"], k_rope_scales=d["k_rope_scales"])
    return _f64(out), binding.device_status(ws)


FUSED_CASES = {
    "single_key": dict(n=[1], prior=[0]),
    "ragged_tails": dict(n=[300, 0, 129, 256, 257, 1], prior=[0, 5, 1000, 127, 3, 77]),
    "page_12": dict(n=[150, 40], prior=[70, 0], page_size=12),
    "latent_row_576": dict(n=[140, 60], prior=[10, 130], row_width=576, rope_col=512, page_size=64),
    "null_mask": dict(n=[100, 130], prior=[50, 300], mask="null"),
    "many_heads": dict(n=[260, 20, 513], prior=[1, 0, 2], heads=16),
}


@pytest.mark.parametrize("case", list(FUSED_CASES))
def test_fused_per_token_k(lib, case):
    kw = dict(FUSED_CASES[case])
    n, prior = kw.pop("n"), kw.pop("prior")
    w = _workload(n, prior, seed=1200 + list(FUSED_CASES).index(case), **kw)
    got, status = run_fused(w)
    assert status == 0
    _close(got, oatt.reference(w), case)


def test_per_token_k_scales_are_applied(lib):
    """The same codes with the per-row scales replaced by their mean: the
    output moves well outside the tolerance, so the per-row path is live."""
    from dataclasses import replace
    w = _workload([300, 200], [100, 0], seed=1250)
    flat = replace(w, k_scale=np.full(w.total_k, np.float32(np.mean(w.k_scale)), dtype=np.float32))
    got, status = run_fused(w)
    assert status == 0
    ref = oatt.reference(w)
    _close(got, ref, "per-token")
    assert np.abs(oatt.reference(flat) - ref).max() > 10 * TOL


def test_bad_page_id_sets_status(lib):
    w = _workload([40], [100], seed=1251)
    w.page_table[0, 3] = 10 ** 6          # the row pre-pass skips the page and flags it
    _, status = run_fused(w)
    assert status & 0x1


def _split_inputs(w):
    codes = w.q.view(torch.uint8)
    q_nope = codes[..., :128].contiguous()
    q_rope = torch.from_numpy(decode_e4m3(codes[..., 128:].numpy()) * w.q_scale).to(torch.bfloat16)
    q64 = np.concatenate([decode_e4m3(q_nope.numpy()) * w.q_scale,
                          decode_bf16(q_rope.view(torch.int16).numpy().view(np.uint16))], axis=-1)
    return q_nope, q_rope, q64


def run_split(w, contiguous=False):
    from mla_ragged_paged_gb300 import binding
    d = workloads.device_inputs(w)
    q_nope, q_rope, q64 = _split_inputs(w)
    if contiguous:
        rows, rsc = workloads.contiguous_rope(w)
        k_rope = rows.cuda()[:, w.spec.rope_col:w.spec.rope_col + 64]
        page_table, rope_scales = None, rsc.cuda()
    else:
        k_rope = d["k_rope_pool"][..., w.spec.rope_col:w.spec.rope_col + 64]
        page_table, rope_scales = d["page_table"], d["k_rope_scales"]
    out = torch.full((w.total_q, w.heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = binding.alloc_workspace(w.batch, fp8_pool_slots=w.total_k)
    binding.prefill_ragged_split(out, q_nope.cuda(), q_rope.cuda(), d["k_nope"], d["v"], k_rope, page_table,
                                 d["row_offsets"], d["cache_lens"], w.scale, _mask(w), ws,
                                 q_scale=d["q_scale"], k_scale=d["k_scale"], v_scale=d["v_scale"],
                                 k_rope_scales=rope_scales)
    assert binding.device_status(ws) == 0
    return _f64(out), q64


@pytest.mark.parametrize("case,kw,contiguous", [
    ("paged", dict(n=[300, 17, 513], prior=[0, 700, 129], heads=4), False),
    ("page_12", dict(n=[150, 40], prior=[70, 0], page_size=12), False),
    ("contiguous", dict(n=[260, 20], prior=[1, 300]), True),
    ("null_mask", dict(n=[100, 130], prior=[50, 300], mask="null"), False),
])
def test_split_per_token_k(lib, case, kw, contiguous):
    kw = dict(kw)
    n, prior = kw.pop("n"), kw.pop("prior")
    w = _workload(n, prior, seed=1260 + len(case), **kw)
    got, q64 = run_split(w, contiguous)
    _close(got, oatt.reference(w, q=q64), case)


@pytest.mark.parametrize("fold", [False, True, "single"])
def test_chunked_per_token_k(lib, fold):
    """Plan + one chunk call per buffer row (the row's slice of the per-token
    scales with its K rows), merged or folded, against the window oracle per
    row and the full-context oracle; or all rows in one
    mla_prefill_ragged_chunked call (scales by stacked K row)."""
    from mla_ragged_paged_gb300 import binding
    w = _workload([300, 17, 513], [0, 700, 129], heads=4, page_size=16, seed=1270)
    T = 200
    d = workloads.device_inputs(w)
    S = w.total_k
    R = -(-S // T)
    if fold == "single":
        pool = d["k_rope_pool"][..., :64]
        ws = binding.alloc_workspace(w.batch, fp8_pool_slots=S)
        out = torch.full((w.total_q, w.heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        binding.prefill_chunked(out, d["q"], d["k_nope"], d["v"], pool, d["page_table"], d["row_offsets"],
                                d["cache_lens"], w.scale, T, R, workspace=ws, q_scale=d["q_scale"],
                                k_scale=d["k_scale"], v_scale=d["v_scale"], k_rope_scales=d["k_rope_scales"])
        assert binding.device_status(ws) == 0
        _close(_f64(out), oatt.reference(w), "chunked single call")
        return
    bro, co, _, _ = binding.plan(d["row_offsets"], d["cache_lens"], T, R)
    pool = d["k_rope_pool"][..., :64]
    ws = binding.alloc_workspace(w.batch, fp8_pool_slots=max(T, w.num_pages * w.page_size))
    out = torch.full((w.total_q, w.heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.total_q, w.heads), dtype=torch.float32, device="cuda")
    po = torch.empty((R, w.total_q, w.heads, 128), dtype=torch.bfloat16, device="cuda")
    pl = torch.empty((R, w.total_q, w.heads), dtype=torch.float32, device="cuda")
    kw = dict(q_scale=d["q_scale"], v_scale=d["v_scale"], k_rope_scales=d["k_rope_scales"])
    bro_h, co_h = bro.cpu().numpy().astype(np.int64), co.cpu().numpy().astype(np.int64)
    for r in range(R):
        lo, hi = r * T, min((r + 1) * T, S)
        o_r, l_r, flags = (out, lse, binding.MLA_CHUNK_ACCUMULATE) if fold else (po[r], pl[r], 0)
        binding.prefill_ragged_chunk(o_r, l_r, d["q"], d["k_nope"][lo:hi], d["v"][lo:hi], pool,
                                     d["page_table"], d["row_offsets"], d["cache_lens"], bro[r], co[r],
                                     w.scale, binding.MLA_MASK_CAUSAL, ws, k_scale=d["k_scale"][lo:hi],
                                     flags=flags, **kw)
        assert binding.device_status(ws) == 0
        if not fold:
            ref_o, ref_l = och.window_reference(w, bro_h[r], co_h[r])
            held = ~np.isnan(ref_l)
            _close(_f64(po[r])[held], ref_o[held], f"row {r} output")
            g_l, r_l = _f64(pl[r])[held], ref_l[held]
            none = np.isneginf(r_l)                 # queries that see no key of the row
            assert np.array_equal(np.isneginf(g_l), none), f"row {r}: -inf lse placement"
            _close(g_l[~none], r_l[~none], f"row {r} lse")
    if not fold:
        binding.merge(out, po, pl, d["row_offsets"], bro)
    _close(_f64(out), oatt.reference(w), "chunked fold" if fold else "chunked merge")


def test_full_size_fp8_per_token_sampled(lib):
    """The B=16, H=128 fp8 workload with per-token K scales, sampled rows and heads."""
    w = workloads.per_token_k(workloads.generate(workloads.config("fp8_e4m3")))
    got, status = run_fused(w)
    assert status == 0
    assert np.isfinite(got).all()
    rng = np.random.default_rng(12)
    rows = {b: np.unique(np.concatenate([[0, int(w.n[b]) - 1], rng.integers(0, int(w.n[b]), 6)]))
            for b in range(w.batch)}
    _close(got, oatt.reference(w, heads=[0, 64, 127], rows=rows), "fp8_e4m3 per-token K")


def test_per_tensor_and_per_token_launches_interleave(lib):
    """Alternating launches of the per-tensor and the per-token kernels on one
    workspace: each matches its first result bit for bit."""
    from mla_ragged_paged_gb300 import binding
    w8 = workloads.custom([300, 129], [40, 0], heads=4, page_size=16, dtype="fp8", seed=1280)
    wt = workloads.per_token_k(w8)
    ws = binding.alloc_workspace(w8.batch, fp8_pool_slots=max(w8.total_k, w8.num_pages * w8.page_size))
    dev = {id(w): workloads.device_inputs(w) for w in (w8, wt)}
    first = {}
    for i in range(40):
        w = (w8, wt)[i & 1]
        d = dev[id(w)]
        out = torch.empty((w.total_q, w.heads, 128), dtype=torch.bfloat16, device="cuda")
        binding.prefill_ragged(out, d["q"], d["k_nope"], d["v"], d["k_rope_pool"], d["page_table"],
                               d["row_offsets"], d["cache_lens"], w.scale, binding.MLA_MASK_CAUSAL, ws,
                               q_scale=d["q_scale"], k_scale=d["k_scale"], v_scale=d["v_scale"],
                               k_rope_scales=d["k_rope_scales"])
        assert binding.device_status(ws) == 0, f"launch {i}"
        if i < 2:
            first[i & 1] = out
        else:
            assert torch.equal(out, first[i & 1]), f"launch {i}"
