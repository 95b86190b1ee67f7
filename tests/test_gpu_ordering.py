"""Pipeline ordering with a slow second query tile.

A test hook delays the softmax of each work item's second query tile before
every score-tile load, so that tile runs well behind the first.  At the end
of a causal item the second tile usually has one more KV tile than the
first; its last two score tiles then follow each other in the shared score
region, and the next item's first score tile waits for the second of them
without the first tile's issuer ever having waited for the first.  The
kernel's alternating region barriers make that skipped wait safe; with a
single parity-tracked barrier the wait could match a phase two behind,
overwrite an unread score tile and stall the pipeline.  Every launch must
finish without a status bit and give output bit-identical to an undelayed
launch.
"""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def _run(binding, w, d, ws, out):
    sc = {k: d.get(k) for k in ("q_scale", "k_scale", "v_scale", "k_rope_scales")}
    binding.prefill_ragged(out, d["q"], d["k_nope"], d["v"], d["k_rope_pool"], d["page_table"],
                           d["row_offsets"], d["cache_lens"], w.scale, binding.MLA_MASK_CAUSAL, ws, **sc)


@pytest.mark.parametrize("name,k_scales,calls", [("deepseek_v3_bf16", "tensor", 6),
                                                 ("fp8_e4m3", "tensor", 3),
                                                 ("fp8_e4m3", "token", 3),
                                                 ("ragged_chunked_bf16", "tensor", 20)])
def test_delayed_second_tile_keeps_results(lib, name, k_scales, calls):
    from mla_ragged_paged_gb300 import binding
    w = workloads.generate(workloads.config(name))
    if k_scales == "token":
        w = workloads.per_token_k(w)
    d = workloads.device_inputs(w)
    fp8 = w.spec.dtype == "fp8"
    slots = (w.total_k if k_scales == "token" else w.num_pages * w.page_size) if fp8 else None
    ws = binding.alloc_workspace(w.batch, fp8_pool_slots=slots)
    ref = torch.empty((w.total_q, w.heads, 128), dtype=torch.bfloat16, device="cuda")
    _run(binding, w, d, ws, ref)
    assert binding.device_status(ws) == 0
    out = torch.empty_like(ref)
    binding.test_delay_softmax(3000)
    try:
        for i in range(calls):
            out.fill_(float("nan"))
            _run(binding, w, d, ws, out)
            assert binding.device_status(ws) == 0, f"launch {i}"
            assert torch.equal(out, ref), f"launch {i}"
    finally:
        binding.test_delay_softmax(0)
