"""GPU plan kernel versus the plan oracle: bit-exact on every workload and on
random ragged edge cases (generic_flare_mla_prefill_ragged_paged_plan)."""
import numpy as np
import pytest
import torch

import workloads
from oracle import plan as oplan

pytestmark = pytest.mark.gpu


def _run(lib_binding, iro, cl, T, R_max):
    from mla_ragged_paged_gb300 import binding
    d_iro = torch.from_numpy(np.asarray(iro, np.uint32).astype(np.int64).astype(np.int32)).cuda()
    d_cl = torch.from_numpy(np.asarray(cl, np.uint32).astype(np.int64).astype(np.int32)).cuda()
    bro, co, blen, nr = binding.plan(d_iro, d_cl, T, R_max)
    torch.cuda.synchronize()
    u32 = lambda t: t.cpu().numpy().view(np.uint32)
    return u32(bro), u32(co), blen.cpu().numpy(), int(u32(nr)[0])


def _compare(lib, iro, cl, T, R_max):
    got = _run(lib, iro, cl, T, R_max)
    want = oplan.plan_formula(iro, cl, T, R_max)
    assert got[3] == want[3]
    for g, w in zip(got[:3], want[:3]):
        assert np.array_equal(g.reshape(w.shape), w.astype(g.dtype)), (g, w)


@pytest.mark.parametrize("name", [c.name for c in workloads.CONFIGS])
def test_plan_matches_oracle_on_workloads(lib, name):
    spec = workloads.config(name)
    rng = np.random.Generator(np.random.PCG64(spec.seed))
    n = workloads._lengths(rng, spec.new_len, spec.batch, "n")
    prior = workloads._lengths(rng, spec.prior_len, spec.batch, "prior")
    iro = np.concatenate([[0], np.cumsum(n)]).astype(np.uint32)
    T = spec.buffer_token_size
    R = oplan.num_rows(iro, prior, T)
    _compare(lib, iro, prior.astype(np.uint32), T, R + 2)


def test_plan_edge_sweep(lib):
    rng = np.random.default_rng(99)
    for trial in range(60):
        B = int(rng.integers(1, 40))
        n = rng.integers(0, 200, size=B)
        prior = rng.integers(0, 300, size=B) * (rng.random(B) < 0.7)
        iro = np.concatenate([[0], np.cumsum(n)]).astype(np.uint32)
        S = int((n + prior).sum())
        T = int(rng.choice([1, 7, 16, 100, 128, max(S, 1), S + 5]))
        R = (S + T - 1) // T
        _compare(lib, iro, prior.astype(np.uint32), T, R + int(rng.integers(0, 3)))


def test_plan_large_batch_and_zero_rows(lib):
    rng = np.random.default_rng(5)
    B = 3000
    n = rng.integers(0, 5, size=B)
    prior = rng.integers(0, 5, size=B)
    iro = np.concatenate([[0], np.cumsum(n)]).astype(np.uint32)
    _compare(lib, iro, prior.astype(np.uint32), 64, oplan.num_rows(iro, prior, 64))
    _compare(lib, np.zeros(4, np.uint32), np.zeros(3, np.uint32), 8, 2)   # empty contexts
    _compare(lib, iro, prior.astype(np.uint32), 64, 0)                     # no room: num_rows only


def test_plan_overflow_reports_sentinel(lib):
    iro = np.array([0, 1, 2], np.uint32)
    cl = np.array([0xFFFFFFF0, 0x100], np.uint32)          # S does not fit in 32 bits
    got = _run(lib, iro, cl, 1024, 1)
    assert got[3] == 0xFFFFFFFF
