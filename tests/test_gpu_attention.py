"""GPU attention (mla_prefill_ragged through the C ABI) versus the float64
oracle, element by element.

Tolerance (bf16 output): |gpu - ref| <= 2e-2 + 2e-2 * |ref| for bf16 inputs and
6e-2 + 6e-2 * |ref| for fp8-e4m3 inputs, the oracle taking the dequantised values.
Small workloads are compared in full; the full-size workloads run in the same
launch configuration as the benchmark and are compared on sampled rows and
heads, which the oracle computes one (sequence, head) at a time.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oatt

pytestmark = pytest.mark.gpu

ATOL = RTOL = 2e-2
ATOL8 = RTOL8 = 6e-2


def run_gpu(w, workspace=None):
    from mla_ragged_paged_gb300 import binding
    d = workloads.device_inputs(w)
    out = torch.full((w.total_q, w.heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    pool = d["k_rope_pool"][..., w.spec.rope_col:w.spec.rope_col + 64]
    slots = w.num_pages * w.page_size if w.spec.dtype == "fp8" else None
    ws = binding.alloc_workspace(w.batch, fp8_pool_slots=slots) if workspace is None else workspace
    mask = binding.MLA_MASK_CAUSAL if w.spec.mask == "causal" else binding.MLA_MASK_NULL
    binding.prefill_ragged(out, d["q"], d["k_nope"], d["v"], pool, d["page_table"],
                           d["row_offsets"], d["cache_lens"], w.scale, mask, ws,
                           q_scale=d.get("q_scale"), k_scale=d.get("k_scale"),
                           v_scale=d.get("v_scale"), k_rope_scales=d.get("k_rope_scales"))
    status = binding.device_status(ws)
    return out.float().cpu().numpy().astype(np.float64), status


def tol(w):
    return (ATOL8, RTOL8) if w.spec.dtype == "fp8" else (ATOL, RTOL)


def assert_close(got, ref, what, atol=ATOL, rtol=RTOL):
    sel = ~np.isnan(ref)
    assert sel.any()
    g, r = got[sel], ref[sel]
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - r)
    bound = atol + rtol * np.abs(r)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements out of tolerance, "
                           f"max err {err.max():.4g}, worst excess {(err - bound).max():.4g}")


@pytest.mark.parametrize("name", ["tiny_bf16", "ragged_chunked_bf16"])
def test_small_workloads_full(lib, name):
    w = workloads.generate(workloads.config(name))
    got, status = run_gpu(w)
    assert status == 0
    assert_close(got, oatt.reference(w), name)


EDGE_CASES = {
    "single_key": dict(n=[1], prior=[0]),
    "ragged_tails": dict(n=[300, 0, 129, 256, 257, 1], prior=[0, 5, 1000, 127, 3, 77]),
    "page_12_row_gather": dict(n=[150, 40], prior=[70, 0], page_size=12),
    "page_24_boxes": dict(n=[200, 33], prior=[0, 260], page_size=24),
    "page_256": dict(n=[300, 90], prior=[200, 0], page_size=256),
    "latent_row_576": dict(n=[140, 60], prior=[10, 130], row_width=576, rope_col=512, page_size=64),
    "null_mask": dict(n=[100, 130], prior=[50, 300], mask="null"),
    "odd_heads": dict(n=[260, 20, 513], prior=[1, 0, 2], heads=3),
    "zero_scale": dict(n=[70], prior=[20], value_scale=1.0),
    # Scores with a standard deviation near 16: peaky rows, many moves of the running max.
    "large_scores": dict(n=[300, 200], prior=[700, 0], value_scale=4.0),
}


@pytest.mark.parametrize("case", list(EDGE_CASES))
def test_edge_cases(lib, case):
    kw = dict(heads=2, page_size=16, seed=300 + list(EDGE_CASES).index(case))
    kw.update(EDGE_CASES[case])
    n, prior = kw.pop("n"), kw.pop("prior")
    w = workloads.custom(n, prior, **kw)
    if case == "zero_scale":
        w.scale = 0.0
    got, status = run_gpu(w)
    assert status == 0
    assert_close(got, oatt.reference(w), case, *tol(w))


def test_many_sequences_random(lib):
    rng = np.random.default_rng(77)
    n = rng.integers(0, 300, size=40)
    prior = rng.integers(0, 400, size=40) * (rng.random(40) < 0.5)
    w = workloads.custom(n.tolist(), prior.tolist(), heads=4, page_size=32, seed=401)
    got, status = run_gpu(w)
    assert status == 0
    assert_close(got, oatt.reference(w), "many_sequences")


def test_repeat_calls_identical(lib):
    w = workloads.custom([333, 77], [12, 500], heads=4, page_size=64, seed=402)
    a, _ = run_gpu(w)
    b, _ = run_gpu(w)
    assert np.array_equal(a, b)


def _sample_rows(w, per_seq=12, seed=0):
    rng = np.random.default_rng(seed)
    rows = {}
    for b in range(w.batch):
        n = int(w.n[b])
        if n == 0:
            continue
        fixed = [0, n - 1] + [x for x in (127, 128, 255, 256, 4095) if x < n]
        rows[b] = np.unique(np.concatenate([fixed, rng.integers(0, n, size=per_seq)]))
    return rows


@pytest.mark.parametrize("name", ["deepseek_v3_bf16", "long_context_bf16", "fp8_e4m3"])
def test_full_size_sampled(lib, name):
    w = workloads.generate(workloads.config(name))
    got, status = run_gpu(w)
    assert status == 0
    assert np.isfinite(got).all(), "every output row must be written and finite"
    heads = [0, w.heads // 3, w.heads - 1]
    ref = oatt.reference(w, heads=heads, rows=_sample_rows(w))
    assert_close(got, ref, name, *tol(w))


FP8_CASES = {
    "fp8_single_key": dict(n=[1], prior=[0]),
    "fp8_ragged_tails": dict(n=[300, 0, 129, 256, 257, 1], prior=[0, 5, 1000, 127, 3, 77]),
    "fp8_page_12": dict(n=[150, 40], prior=[70, 0], page_size=12),
    "fp8_latent_row_576": dict(n=[140, 60], prior=[10, 130], row_width=576, rope_col=512, page_size=64),
    "fp8_null_mask": dict(n=[100, 130], prior=[50, 300], mask="null"),
    "fp8_many_heads": dict(n=[260, 20, 513], prior=[1, 0, 2], heads=16),
    # 1.5x the workload's spread: larger scores and V.  (The e4m3 rounding of P
    # grows with the score range; a float64 model of it stays within the
    # tolerance up to about 1.5x and exceeds it from about 2x.)
    "fp8_large_scores": dict(n=[300, 200], prior=[700, 0], value_scale=1.5),
}


@pytest.mark.parametrize("case", list(FP8_CASES))
def test_fp8_cases(lib, case):
    kw = dict(heads=2, page_size=16, seed=600 + list(FP8_CASES).index(case), dtype="fp8")
    kw.update(FP8_CASES[case])
    n, prior = kw.pop("n"), kw.pop("prior")
    w = workloads.custom(n, prior, **kw)
    got, status = run_gpu(w)
    assert status == 0
    assert_close(got, oatt.reference(w), case, ATOL8, RTOL8)


def test_bad_page_id_sets_status(lib):
    w = workloads.custom([40], [100], heads=2, page_size=16, seed=403)
    w.page_table[0, 3] = 10 ** 6          # no such page: the kernel skips it and flags it
    _, status = run_gpu(w)
    assert status & 0x1


@pytest.mark.parametrize("name,calls", [("tiny_bf16", 400), ("ragged_chunked_bf16", 400),
                                        ("deepseek_v3_bf16", 60)])
def test_many_launches_stable(lib, name, calls):
    """Back-to-back launches: every one completes without a status bit (no
    pipeline wait ever runs out) and gives bit-identical results."""
    from mla_ragged_paged_gb300 import binding
    w = workloads.generate(workloads.config(name))
    d = workloads.device_inputs(w)
    ws = binding.alloc_workspace(w.batch)
    outs = [torch.empty((w.total_q, w.heads, 128), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    for i in range(calls):
        binding.prefill_ragged(outs[i & 1], d["q"], d["k_nope"], d["v"], d["k_rope_pool"], d["page_table"],
                               d["row_offsets"], d["cache_lens"], w.scale, binding.MLA_MASK_CAUSAL, ws)
        # The scheduler of every launch rewrites the status word: read it each time.
        assert binding.device_status(ws) == 0, f"launch {i}"
        if i % 20 == 19:
            assert torch.equal(outs[0], outs[1]), f"launch {i}"


@pytest.mark.parametrize("B,dtype", [(2048, "bf16"), (2049, "fp8"), (4096, "bf16")])
def test_largest_batches(lib, B, dtype):
    """Batch sizes around the scheduler's longest-first sort (up to 2048
    sequences; identity order above) and at the 4096-sequence limit, with
    empty sequences mixed in, every sequence checked."""
    rng = np.random.default_rng(B)
    n = rng.integers(0, 9, size=B)
    prior = rng.integers(0, 21, size=B) * (rng.random(B) < 0.7)
    w = workloads.custom(n.tolist(), prior.tolist(), heads=1, page_size=16, seed=B, dtype=dtype)
    got, status = run_gpu(w)
    assert status == 0
    assert_close(got, oatt.reference(w), f"B={B}", *tol(w))


@pytest.mark.parametrize("offset", [0, 8, 16])
def test_output_alignment(lib, offset):
    """Output rows 32-byte aligned (offset 0 or 16 bf16) take the kernel's
    32-byte store path, rows only 16-byte aligned (offset 8) the 16-byte one;
    both must write exactly the output rows, within tolerance of the oracle."""
    from mla_ragged_paged_gb300 import binding
    w = workloads.custom([200, 37, 129], [0, 50, 300], heads=3, page_size=32, seed=611)
    d = workloads.device_inputs(w)
    # Each (token, head) row sits at `offset` inside a 144-element slot: the row
    # strides (144 and 3 * 144 elements) are 32-byte multiples, so only the
    # base offset decides the alignment.
    buf = torch.full((w.total_q * w.heads * 144 + 16,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[offset:offset + w.total_q * w.heads * 144].view(w.total_q, w.heads, 144)[..., :128]
    ws = binding.alloc_workspace(w.batch)
    binding.prefill_ragged(out, d["q"], d["k_nope"], d["v"], d["k_rope_pool"], d["page_table"],
                           d["row_offsets"], d["cache_lens"], w.scale, binding.MLA_MASK_CAUSAL, ws)
    assert binding.device_status(ws) == 0
    torch.cuda.synchronize()
    slots = buf[offset:offset + w.total_q * w.heads * 144].view(w.total_q, w.heads, 144)
    assert torch.isnan(slots[..., 128:]).all(), "the kernel wrote outside the output rows"
    assert_close(out.float().cpu().numpy().astype(np.float64), oatt.reference(w), f"offset {offset}")
