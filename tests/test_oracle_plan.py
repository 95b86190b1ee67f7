"""Pins for the plan oracle: hand-worked examples, two independent derivations
agreeing bit for bit, and the tiling invariants of the global-packing reading
of generic_flare_mla_prefill_ragged_paged_plan (Args: buffer_row_offsets,
cache_offsets, buffer_lengths)."""
import json
import os

import numpy as np
import pytest

from oracle import plan as oplan

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "plan_examples.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
@pytest.mark.parametrize("impl", [oplan.plan_formula, oplan.plan_token_walk])
def test_hand_worked_examples(case, impl):
    bro, co, blen, R = impl(case["input_row_offsets"], case["cache_lens"],
                            case["buffer_token_size"], case["max_rows"])
    assert R == case["num_rows"]
    assert bro.dtype == np.uint32 and co.dtype == np.uint32 and blen.dtype == np.int32
    assert bro.tolist() == case["buffer_row_offsets"]
    assert co.tolist() == case["cache_offsets"]
    assert blen.tolist() == case["buffer_lengths"]


def _random_case(rng):
    B = int(rng.integers(1, 9))
    n = rng.integers(0, 33, size=B)
    prior = rng.integers(0, 33, size=B)
    iro = np.concatenate([[0], np.cumsum(n)]).astype(np.uint32)
    S = int((n + prior).sum())
    T = int(rng.choice([1, 3, 7, 32, max(S, 1), S + 1]))
    return iro, prior.astype(np.uint32), T, S


def _check_invariants(iro, cache_lens, T, bro, co, blen, R):
    L = oplan.context_lengths(iro, cache_lens)
    B = L.size
    S = int(L.sum())
    assert R == (S + T - 1) // T
    R_max = bro.shape[0]
    seen = np.zeros(B, dtype=np.int64)
    for r in range(R_max):
        row = bro[r].astype(np.int64)
        assert np.all(np.diff(row) >= 0), "offsets non-decreasing within a row"
        lens = np.diff(row)
        if r < R:
            assert int(row[-1]) == int(blen[r])
            assert blen[r] == (T if r < R - 1 else S - (R - 1) * T)
        else:
            assert blen[r] == -1 and row[-1] == 0
        # each sequence's segments tile [0, L_b) contiguously, in row order
        for b in range(B):
            assert int(co[r, b]) == seen[b]
            seen[b] += int(lens[b])
    assert np.array_equal(seen, L)


def test_formula_equals_token_walk_and_invariants():
    rng = np.random.default_rng(1234)
    for _ in range(300):
        iro, prior, T, S = _random_case(rng)
        R_max = (S + T - 1) // T + int(rng.integers(0, 3))
        a = oplan.plan_formula(iro, prior, T, R_max)
        b = oplan.plan_token_walk(iro, prior, T, R_max)
        assert a[3] == b[3]
        for x, y in zip(a[:3], b[:3]):
            assert x.dtype == y.dtype and np.array_equal(x, y)
        _check_invariants(iro, prior, T, *a)


def test_empty_batch_context():
    iro = np.zeros(4, np.uint32)
    prior = np.zeros(3, np.uint32)
    bro, co, blen, R = oplan.plan_formula(iro, prior, 16, 2)
    assert R == 0 and blen.tolist() == [-1, -1]
    assert not bro.any() and not co.any()


def test_single_token_rows():
    iro = np.array([0, 2, 5], np.uint32)
    prior = np.array([1, 0], np.uint32)
    bro, co, blen, R = oplan.plan_formula(iro, prior, 1, 6)
    assert R == 6 and blen.tolist() == [1] * 6
    # tokens 0..2 belong to sequence 0, tokens 3..5 to sequence 1
    assert [int(x) for x in bro[:, 1]] == [1, 1, 1, 0, 0, 0]
    assert [int(x) for x in co[:, 1]] == [0, 0, 0, 0, 1, 2]
