"""The kernel's bounded waits on the GPU: with the test hook enabled, nothing
arms the barrier of one K group per CTA, the UMMA issuers' wait runs out, the
kernel winds down and reports MLA_DEVICE_STATUS_TIMEOUT in the workspace
status word; the context stays usable and the next launch is correct."""
import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oatt

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_wait_timeout_sets_status_and_context_survives(lib, dtype):
    from mla_ragged_paged_gb300 import binding
    w = workloads.custom([200, 40], [30, 0], heads=2, page_size=16, seed=960, dtype=dtype)
    d = workloads.device_inputs(w)
    pool = d["k_rope_pool"][..., :64]
    fp8 = dtype == "fp8"
    ws = binding.alloc_workspace(w.batch, fp8_pool_slots=w.num_pages * w.page_size if fp8 else None)
    out = torch.zeros((w.total_q, w.heads, 128), dtype=torch.bfloat16, device="cuda")
    kw = dict(q_scale=d.get("q_scale"), k_scale=d.get("k_scale"), v_scale=d.get("v_scale"),
              k_rope_scales=d.get("k_rope_scales"))
    binding.test_inject_stall(True)
    try:
        binding.prefill_ragged(out, d["q"], d["k_nope"], d["v"], pool, d["page_table"], d["row_offsets"],
                               d["cache_lens"], w.scale, binding.MLA_MASK_CAUSAL, ws, **kw)
        status = binding.device_status(ws)
    finally:
        binding.test_inject_stall(False)
    assert status & 0x8, f"status {status:#x}"
    # The context is intact: the next launch completes and is correct.
    binding.prefill_ragged(out, d["q"], d["k_nope"], d["v"], pool, d["page_table"], d["row_offsets"],
                           d["cache_lens"], w.scale, binding.MLA_MASK_CAUSAL, ws, **kw)
    assert binding.device_status(ws) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    ref = oatt.reference(w)
    tol = 6e-2 if fp8 else 2e-2
    assert np.all(np.abs(got - ref) <= tol + tol * np.abs(ref))
