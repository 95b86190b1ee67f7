"""The allocation-free entry point (mla_prefill_ragged_noalloc) against the
workspace entry point (mla_prefill_ragged) and the oracle, through the C ABI.

mla_prefill_ragged_noalloc serves callers that cannot allocate device memory
(for example a plug-in whose host framework owns all device memory, or a
latency-critical path that may not call cudaMalloc).  It keeps its scheduler
workspace in a fixed array inside the library, shared by every call, so the
tests make calls in a row, a larger batch before a smaller one, and check that
nothing left in the array by one call changes the next: each output must equal
the workspace entry point's bit for bit (both launch the same kernels on the
same inputs) and lie within the attention tolerance of the float64 oracle.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oatt

pytestmark = pytest.mark.gpu

ATOL = RTOL = 2e-2


def _close(got, ref):
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    assert np.isfinite(got).all()
    assert bool((err <= bound).all()), f"max err {err.max():.4g}"


def _args(w, d, binding):
    return (d["q"], d["k_nope"], d["v"], d["k_rope_pool"], d["page_table"], d["row_offsets"],
            d["cache_lens"], w.scale, binding.MLA_MASK_CAUSAL)


def _workspace_result(w, d, binding):
    ref = torch.empty((w.total_q, w.heads, 128), dtype=torch.bfloat16, device="cuda")
    binding.prefill_ragged(ref, *_args(w, d, binding))
    return ref


def _noalloc_result(w, d, binding):
    out = torch.full((w.total_q, w.heads, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    binding.prefill_ragged_noalloc(out, *_args(w, d, binding))
    return out


def test_noalloc_matches_workspace_entry_point_twice(lib):
    from mla_ragged_paged_gb300 import binding
    # A larger batch first, then a smaller one: records and the work counter
    # of the first call stay in the shared array and must not leak into the
    # second.
    big = workloads.custom([300, 0, 129, 257, 40, 3, 77, 511, 1], [0, 5, 1000, 3, 77, 0, 64, 2, 9],
                           heads=4, page_size=32, seed=501)
    small = workloads.custom([65, 200], [7, 0], heads=3, page_size=16, seed=503)
    cases = []
    for w in (big, small, small):
        d = workloads.device_inputs(w)
        got = _noalloc_result(w, d, binding)
        cases.append((w, got, _workspace_result(w, d, binding)))
    torch.cuda.synchronize()
    refs = {}
    for w, got, want in cases:
        assert torch.equal(got, want), "noalloc output differs from the workspace entry point"
        if id(w) not in refs:
            refs[id(w)] = oatt.reference(w)
        _close(got.float().cpu().numpy(), refs[id(w)])


def test_noalloc_accepts_its_maximum_batch(lib):
    from mla_ragged_paged_gb300 import binding
    B = 1024
    rng = np.random.default_rng(504)
    n = rng.integers(0, 4, size=B).tolist()
    w = workloads.custom(n, rng.integers(0, 3, size=B).tolist(), heads=1, page_size=16, seed=504)
    d = workloads.device_inputs(w)
    got = _noalloc_result(w, d, binding)
    want = _workspace_result(w, d, binding)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    _close(got.float().cpu().numpy(), oatt.reference(w))


def test_noalloc_rejects_batch_above_its_workspace(lib):
    from mla_ragged_paged_gb300 import binding
    B = 1025
    w = workloads.custom([1] * B, [0] * B, heads=1, page_size=16, seed=502)
    d = workloads.device_inputs(w)
    out = torch.empty((w.total_q, 1, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.MlaError) as exc:
        binding.prefill_ragged_noalloc(out, *_args(w, d, binding))
    assert exc.value.status == binding.MLA_ERR_INVALID_ARG
    assert "1024" in str(exc.value)


def test_noalloc_rejects_fp8_inputs(lib):
    from mla_ragged_paged_gb300 import binding
    w = workloads.custom([20, 7], [0, 3], heads=2, page_size=16, dtype="fp8", seed=505)
    d = workloads.device_inputs(w)
    out = torch.empty((w.total_q, w.heads, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.MlaError) as exc:
        binding.prefill_ragged_noalloc(out, *_args(w, d, binding))
    assert exc.value.status == binding.MLA_ERR_INVALID_ARG
    assert "bf16" in str(exc.value)
