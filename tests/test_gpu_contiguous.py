"""Contiguous K_rope (mla_prefill_ragged_contiguous through the C ABI) versus the
float64 oracle.  The contiguous tensor holds, at K row G_b + j, the pool row the
page table gives for key j of sequence b, so the paged oracle's result is the
expected output.  Tolerances as for the paged call."""
import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oatt

pytestmark = pytest.mark.gpu


def run_contig(w):
    from mla_ragged_paged_gb300 import binding
    d = workloads.device_inputs(w)
    rows, scales = workloads.contiguous_rope(w)
    rope = rows.cuda()[:, w.spec.rope_col:w.spec.rope_col + 64]
    fp8 = w.spec.dtype == "fp8"
    out = torch.full((w.total_q, w.heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = binding.alloc_workspace(w.batch, fp8_pool_slots=w.total_k if fp8 else None)
    mask = binding.MLA_MASK_CAUSAL if w.spec.mask == "causal" else binding.MLA_MASK_NULL
    binding.prefill_ragged_contiguous(out, d["q"], d["k_nope"], d["v"], rope, d["row_offsets"],
                                      d["cache_lens"], w.scale, mask, ws, q_scale=d.get("q_scale"),
                                      k_scale=d.get("k_scale"), v_scale=d.get("v_scale"),
                                      k_rope_scales=scales.cuda() if fp8 else None)
    status = binding.device_status(ws)
    return out.float().cpu().numpy().astype(np.float64), status


def _close(got, ref, atol, rtol, what):
    sel = ~np.isnan(ref)
    g, r = got[sel], ref[sel]
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - r)
    bad = err > atol + rtol * np.abs(r)
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} out of tolerance, max err {err.max():.4g}"


CASES = {
    "tiny": ("tiny_bf16", None),
    "ragged": ("ragged_chunked_bf16", None),
    "tails": (None, dict(n=[300, 0, 129, 256, 257, 1], prior=[0, 5, 1000, 127, 3, 77])),
    "latent_row_576": (None, dict(n=[140, 60], prior=[10, 130], row_width=576, rope_col=512,
                                  page_size=64)),
    "null_mask": (None, dict(n=[100, 130], prior=[50, 300], mask="null")),
    "fp8": (None, dict(n=[300, 17, 513], prior=[0, 700, 129], heads=4, dtype="fp8")),
    "fp8_latent_row_576": (None, dict(n=[140, 60], prior=[10, 130], row_width=576, rope_col=512,
                                      dtype="fp8")),
}


@pytest.mark.parametrize("case", list(CASES))
def test_contiguous_rope(lib, case):
    name, kw = CASES[case]
    if name:
        w = workloads.generate(workloads.config(name))
    else:
        kw = dict(dict(heads=2, page_size=16, seed=800 + list(CASES).index(case)), **kw)
        n, prior = kw.pop("n"), kw.pop("prior")
        w = workloads.custom(n, prior, **kw)
    got, status = run_contig(w)
    assert status == 0
    tol = 6e-2 if w.spec.dtype == "fp8" else 2e-2
    _close(got, oatt.reference(w), tol, tol, case)


def test_contiguous_full_size_sampled(lib):
    w = workloads.generate(workloads.config("deepseek_v3_bf16"))
    got, status = run_contig(w)
    assert status == 0
    assert np.isfinite(got).all()
    rng = np.random.default_rng(5)
    rows = {b: np.unique(np.concatenate([[0, int(w.n[b]) - 1], rng.integers(0, int(w.n[b]), 10)]))
            for b in range(w.batch)}
    ref = oatt.reference(w, heads=[0, 77, w.heads - 1], rows=rows)
    _close(got, ref, 2e-2, 2e-2, "deepseek_v3_bf16 contiguous")
