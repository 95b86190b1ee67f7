"""Split-Q attention (mla_prefill_ragged_split through the C ABI) versus the
float64 oracle.

The split inputs are built from a workload's fused Q: q_nope = Q[..., :128]
(bf16, or the e4m3 codes with the per-tensor scale) and q_rope = Q[..., 128:]
as bf16 real values (for fp8 workloads the dequantised rope codes rounded to
bf16).  The oracle takes exactly those query values (its `q` argument).
Tolerances as for the fused call: bf16 2e-2 + 2e-2|ref|, fp8 6e-2 + 6e-2|ref|.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oatt
from oracle.numerics import decode_bf16, decode_e4m3

pytestmark = pytest.mark.gpu


def _split_inputs(w, views=False):
    """(q_nope, q_rope) CPU tensors and the float64 query values they carry."""
    if w.spec.dtype == "fp8":
        codes = w.q.view(torch.uint8)
        q_nope = codes[..., :128].contiguous()
        rope = torch.from_numpy(decode_e4m3(codes[..., 128:].numpy()) * w.q_scale)
        q_rope = rope.to(torch.bfloat16)
        q64 = np.concatenate([decode_e4m3(q_nope.numpy()) * w.q_scale,
                              decode_bf16(q_rope.view(torch.int16).numpy().view(np.uint16))], axis=-1)
        return q_nope, q_rope, q64
    if views:
        return w.q[..., :128], w.q[..., 128:], None
    return w.q[..., :128].contiguous(), w.q[..., 128:].contiguous(), None


def _close(got, ref, tol, what):
    sel = ~np.isnan(ref)
    g, r = got[sel], ref[sel]
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - r)
    bad = err > tol + tol * np.abs(r)
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} out of tolerance, max err {err.max():.4g}"


def run_split(w, contiguous=False, views=False, v_own_scale=True):
    from mla_ragged_paged_gb300 import binding
    d = workloads.device_inputs(w)
    fp8 = w.spec.dtype == "fp8"
    q_nope, q_rope, q64 = _split_inputs(w, views)
    if views:
        q_nope, q_rope = d["q"][..., :128], d["q"][..., 128:]
    else:
        q_nope, q_rope = q_nope.cuda(), q_rope.cuda()
    if contiguous:
        rows, rsc = workloads.contiguous_rope(w)
        k_rope = rows.cuda()[:, w.spec.rope_col:w.spec.rope_col + 64]
        page_table, k_rope_scales = None, (rsc.cuda() if fp8 else None)
    else:
        k_rope = d["k_rope_pool"][..., w.spec.rope_col:w.spec.rope_col + 64]
        page_table, k_rope_scales = d["page_table"], d.get("k_rope_scales")
    out = torch.full((w.total_q, w.heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    slots = (w.total_k if contiguous else w.num_pages * w.page_size) if fp8 else None
    ws = binding.alloc_workspace(w.batch, fp8_pool_slots=slots)
    mask = binding.MLA_MASK_CAUSAL if w.spec.mask == "causal" else binding.MLA_MASK_NULL
    binding.prefill_ragged_split(out, q_nope, q_rope, d["k_nope"], d["v"], k_rope, page_table,
                                 d["row_offsets"], d["cache_lens"], w.scale, mask, ws,
                                 q_scale=d.get("q_scale"), k_scale=d.get("k_scale"),
                                 v_scale=d.get("v_scale") if v_own_scale else None,
                                 k_rope_scales=k_rope_scales)
    assert binding.device_status(ws) == 0
    return out.float().cpu().numpy().astype(np.float64), q64


CASES = {
    "bf16_paged": (dict(n=[300, 0, 129, 257], prior=[0, 5, 1000, 3]), {}),
    "bf16_views": (dict(n=[140, 60], prior=[10, 130]), dict(views=True)),
    "bf16_contiguous": (dict(n=[200, 33], prior=[0, 260]), dict(contiguous=True)),
    "bf16_null_mask": (dict(n=[100, 130], prior=[50, 300], mask="null"), {}),
    "fp8_paged": (dict(n=[300, 17, 513], prior=[0, 700, 129], heads=4, dtype="fp8"), {}),
    "fp8_page12": (dict(n=[150, 40], prior=[70, 0], page_size=12, dtype="fp8"), {}),
    "fp8_contiguous": (dict(n=[260, 20], prior=[1, 300], dtype="fp8"), dict(contiguous=True)),
    "fp8_v_uses_k_scale": (dict(n=[200, 90], prior=[30, 0], dtype="fp8"), dict(v_own_scale=False)),
}


@pytest.mark.parametrize("case", list(CASES))
def test_split_q(lib, case):
    kw, opts = CASES[case]
    kw = dict(dict(heads=2, page_size=16, seed=950 + list(CASES).index(case)), **kw)
    n, prior = kw.pop("n"), kw.pop("prior")
    w = workloads.custom(n, prior, **kw)
    got, q64 = run_split(w, **opts)
    ref_w = w if opts.get("v_own_scale", True) else replace(w, v_scale=w.k_scale)
    tol = 6e-2 if w.spec.dtype == "fp8" else 2e-2
    _close(got, oatt.reference(ref_w, q=q64), tol, case)


def test_split_q_full_size_fp8_sampled(lib):
    w = workloads.generate(workloads.config("fp8_e4m3"))
    got, q64 = run_split(w)
    assert np.isfinite(got).all()
    rng = np.random.default_rng(8)
    rows = {b: np.unique(np.concatenate([[0, int(w.n[b]) - 1], rng.integers(0, int(w.n[b]), 6)]))
            for b in range(w.batch)}
    ref = oatt.reference(w, heads=[0, 64, 127], rows=rows, q=q64)
    _close(got, ref, 6e-2, "fp8_e4m3 split")
