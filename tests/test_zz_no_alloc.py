"""The allocation-free entry point (mla_prefill_ragged_noalloc) against the
workspace entry point (mla_prefill_ragged), both through the C ABI.

mla_prefill_ragged_noalloc serves callers that cannot allocate device memory
(for example a plug-in whose host framework owns all device memory, or a
latency-critical path that may not call cudaMalloc).  It keeps its scheduler
workspace in a fixed array inside the library, shared by every call, so the
test makes two calls in a row and checks both.  This file is collected last
so that a run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

ATOL = RTOL = 2e-2


def _close(got, ref):
    err = (got - ref).abs()
    bound = ATOL + RTOL * ref.abs()
    assert torch.isfinite(got).all()
    assert bool((err <= bound).all()), f"max err {err.max().item():.4g}"


def test_noalloc_matches_workspace_entry_point_twice(lib):
    from mla_ragged_paged_gb300 import binding
    w = workloads.custom([300, 0, 129, 257, 40], [0, 5, 1000, 3, 77], heads=4, page_size=32,
                         seed=501)
    d = workloads.device_inputs(w)
    args = (d["q"], d["k_nope"], d["v"], d["k_rope_pool"], d["page_table"], d["row_offsets"],
            d["cache_lens"], w.scale, binding.MLA_MASK_CAUSAL)
    shape = (w.total_q, w.heads, 128)
    ref = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    binding.prefill_ragged(ref, *args)
    outs = []
    for _ in range(2):
        out = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        binding.prefill_ragged_noalloc(out, *args)
        outs.append(out)
    torch.cuda.synchronize()
    for out in outs:
        _close(out.float(), ref.float())


def test_noalloc_rejects_batch_above_its_workspace(lib):
    from mla_ragged_paged_gb300 import binding
    B = 1025
    w = workloads.custom([1] * B, [0] * B, heads=1, page_size=16, seed=502)
    d = workloads.device_inputs(w)
    out = torch.empty((w.total_q, 1, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.MlaError) as exc:
        binding.prefill_ragged_noalloc(out, d["q"], d["k_nope"], d["v"], d["k_rope_pool"],
                                       d["page_table"], d["row_offsets"], d["cache_lens"], w.scale)
    assert exc.value.status == binding.MLA_ERR_INVALID_ARG
    assert "1024" in str(exc.value)
