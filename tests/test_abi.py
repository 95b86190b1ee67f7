"""C-ABI library checks that need no GPU: it loads, exports every entry point
declared in include/*.h, and rejects bad arguments on the host before touching
the device."""
import ctypes
import glob
import os
import re

import pytest

import mla_ragged_paged_gb300 as pkg
from mla_ragged_paged_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pkg.build()
    return binding.load()


def _declared_functions():
    names = set()
    for path in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(mla_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert "mla_prefill_plan" in declared and "mla_prefill_ragged" in declared
    for name in declared:
        assert hasattr(lib, name), f"{name} declared but not exported"
    assert sorted(binding.EXPORTS) == [n for n in declared if n in binding.EXPORTS]


def test_host_helpers(lib):
    assert binding.plan_max_rows(50, 32) == 2
    assert binding.plan_max_rows(0, 32) == 0
    assert binding.plan_max_rows(64, 32) == 2
    assert binding.plan_max_rows(10, 0) == 0
    ws = binding.workspace_size(8)
    assert ws % 256 == 0 and ws >= 256 + 8 * 32
    assert binding.workspace_size(8, fp8_pool_slots=1000) == ws + 1000 * 128


def _desc(shape, dtype=binding.MLA_DTYPE_BF16, ptr=0x10000):
    d = binding.MlaTensor()
    d.data = ptr
    d.dtype = dtype
    d.ndim = len(shape)
    stride = 1
    for i in reversed(range(len(shape))):
        d.shape[i] = shape[i]
        d.stride[i] = stride
        stride *= shape[i]
    return d


def _ragged_args(**over):
    a = dict(out=_desc([10, 2, 128]), q=_desc([10, 2, 192]), k=_desc([20, 2, 128]),
             v=_desc([20, 2, 128]), rope=_desc([4, 16, 64]),
             pt=_desc([2, 2], binding.MLA_DTYPE_U32), ro=0x20000, cl=0x30000, scale=0.07,
             mask=binding.MLA_MASK_CAUSAL, ws=0x40000, ws_bytes=4096)
    a.update(over)
    return a


def _call_ragged(lib, a):
    r = lambda d: None if d is None else ctypes.byref(d)
    return lib.mla_prefill_ragged(r(a["out"]), r(a["q"]), r(a["k"]), r(a["v"]), r(a["rope"]),
                                  r(a["pt"]), a["ro"], a["cl"], a["scale"], a["mask"], a["ws"],
                                  a["ws_bytes"], None)


@pytest.mark.parametrize("change", [
    dict(q=None), dict(out=None), dict(ro=None), dict(cl=None), dict(ws=None),
    dict(q=_desc([10, 2, 128])),                        # q depth must be 192
    dict(out=_desc([10, 2, 64])),                       # output depth 128
    dict(k=_desc([20, 3, 128])),                        # head count mismatch
    dict(v=_desc([19, 2, 128])),                        # v rows differ from k
    dict(rope=_desc([4, 16, 32])),                      # rope depth 64
    dict(rope=_desc([0, 16, 64])),                      # empty pool
    dict(pt=_desc([2, 2], binding.MLA_DTYPE_BF16)),     # page table dtype
    dict(q=_desc([10, 2, 192], binding.MLA_DTYPE_U32)),  # q dtype
    dict(scale=-1.0), dict(scale=float("nan")), dict(mask=7),
    dict(ws=0x40008),                                   # workspace alignment
    dict(ws_bytes=16),                                  # workspace size
    dict(k=_desc([5, 2, 128]), v=_desc([5, 2, 128])),   # fewer K rows than Q rows
    dict(q=_desc([10, 2, 192], ptr=0x10004)),            # unaligned base
])
def test_ragged_rejects_bad_arguments(lib, change):
    assert _call_ragged(lib, _ragged_args(**change)) == binding.MLA_ERR_INVALID_ARG
    assert lib.mla_last_error_string()


def test_fp8_needs_scales(lib):
    fp8 = binding.MLA_DTYPE_FP8_E4M3
    a = _ragged_args(q=_desc([10, 2, 192], fp8), k=_desc([20, 2, 128], fp8),
                     v=_desc([20, 2, 128], fp8), rope=_desc([4, 16, 64], fp8))
    assert _call_ragged(lib, a) == binding.MLA_ERR_INVALID_ARG
    assert b"scale" in lib.mla_last_error_string()
    for t in (a["q"], a["k"], a["v"]):
        t.scale = 0x50000
        t.scale_gran = binding.MLA_SCALE_PER_TENSOR
    assert _call_ragged(lib, a) == binding.MLA_ERR_INVALID_ARG     # rope scales still missing
    assert b"per-token" in lib.mla_last_error_string()
    mixed = _ragged_args(q=_desc([10, 2, 192], fp8))                 # fp8 q with bf16 k
    assert _call_ragged(lib, mixed) == binding.MLA_ERR_INVALID_ARG


def test_fp8_per_token_k_scales(lib):
    """K_nope may carry one scale per K row; the workspace then holds the
    converted K_rope at the K rows (S_k rows, not the pool's slots), and the
    split overload's v needs a scale of its own."""
    fp8 = binding.MLA_DTYPE_FP8_E4M3
    a = _ragged_args(q=_desc([10, 2, 192], fp8), k=_desc([20, 2, 128], fp8),
                     v=_desc([20, 2, 128], fp8), rope=_desc([4, 16, 64], fp8))
    for t, gran in ((a["q"], binding.MLA_SCALE_PER_TENSOR), (a["k"], binding.MLA_SCALE_PER_TOKEN),
                    (a["v"], binding.MLA_SCALE_PER_TENSOR), (a["rope"], binding.MLA_SCALE_PER_TOKEN)):
        t.scale = 0x50000
        t.scale_gran = gran
    a["ws_bytes"] = binding.workspace_size(2, fp8_pool_slots=19)      # one row short of S_k = 20
    assert _call_ragged(lib, a) == binding.MLA_ERR_INVALID_ARG
    assert b"workspace too small" in lib.mla_last_error_string()
    a["ws_bytes"] = binding.workspace_size(2, fp8_pool_slots=20)      # less than the 64 pool slots
    assert _call_ragged(lib, a) != binding.MLA_ERR_INVALID_ARG        # host checks pass
    a["k"].scale_gran = binding.MLA_SCALE_PER_TENSOR                   # per tensor: 64 rows needed
    assert _call_ragged(lib, a) == binding.MLA_ERR_INVALID_ARG
    a["k"].scale_gran = binding.MLA_SCALE_NONE
    assert _call_ragged(lib, a) == binding.MLA_ERR_INVALID_ARG
    assert b"k_nope" in lib.mla_last_error_string()

    # Split Q: per-token k and a v without its own scale.
    a["k"].scale_gran = binding.MLA_SCALE_PER_TOKEN
    a["v"].scale = None
    a["v"].scale_gran = binding.MLA_SCALE_NONE
    r = lambda d: None if d is None else ctypes.byref(d)
    qn, qr = _desc([10, 2, 128], fp8), _desc([10, 2, 64])
    qn.scale, qn.scale_gran = 0x50000, binding.MLA_SCALE_PER_TENSOR
    st = lib.mla_prefill_ragged_split(r(a["out"]), r(qn), r(qr), r(a["k"]), r(a["v"]), r(a["rope"]),
                                      r(a["pt"]), 2, a["ro"], a["cl"], a["scale"], a["mask"], a["ws"],
                                      a["ws_bytes"], None)
    assert st == binding.MLA_ERR_INVALID_ARG
    assert b"fp8 v" in lib.mla_last_error_string()


def test_ragged_rejects_unaligned_stride(lib):
    q = _desc([10, 2, 192])
    q.stride[1] = 196          # 392 bytes: not a multiple of 16
    assert _call_ragged(lib, _ragged_args(q=q)) == binding.MLA_ERR_INVALID_ARG
    assert b"stride" in lib.mla_last_error_string()


def test_plan_rejects_bad_arguments(lib):
    f = lib.mla_prefill_plan
    P = 0x10000
    assert f(None, P, 2, 32, 4, P, P, P, None, None) == binding.MLA_ERR_INVALID_ARG
    assert f(P, None, 2, 32, 4, P, P, P, None, None) == binding.MLA_ERR_INVALID_ARG
    assert f(P, P, 2, 0, 4, P, P, P, None, None) == binding.MLA_ERR_INVALID_ARG
    assert f(P, P, 2, 32, 4, None, P, P, None, None) == binding.MLA_ERR_INVALID_ARG
    assert f(P, P, 1 << 20, 32, 4, P, P, P, None, None) == binding.MLA_ERR_INVALID_ARG
    assert b"buffer_token_size" in lib.mla_last_error_string() or lib.mla_last_error_string()


def _call_chunk(lib, a, lse, bro=0x60000, co=0x70000, flags=0):
    r = lambda d: None if d is None else ctypes.byref(d)
    return lib.mla_prefill_ragged_chunk(r(a["out"]), r(lse), r(a["q"]), r(a["k"]), r(a["v"]),
                                        r(a["rope"]), r(a["pt"]), a["ro"], a["cl"], bro, co,
                                        a["scale"], a["mask"], flags, a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("case", ["no_lse", "lse_shape", "lse_dtype", "lse_unaligned", "no_bro",
                                  "no_co", "empty_row", "q_depth", "flags"])
def test_chunk_rejects_bad_arguments(lib, case):
    a = _ragged_args()
    lse = _desc([10, 2], binding.MLA_DTYPE_F32, ptr=0x80000)
    bro, co = 0x60000, 0x70000
    if case == "no_lse":
        lse = None
    elif case == "lse_shape":
        lse = _desc([10, 3], binding.MLA_DTYPE_F32)
    elif case == "lse_dtype":
        lse = _desc([10, 2], binding.MLA_DTYPE_BF16)
    elif case == "lse_unaligned":
        lse = _desc([10, 2], binding.MLA_DTYPE_F32, ptr=0x80002)
    elif case == "no_bro":
        bro = None
    elif case == "no_co":
        co = None
    elif case == "empty_row":
        a = _ragged_args(k=_desc([0, 2, 128]), v=_desc([0, 2, 128]))
    elif case == "q_depth":
        a = _ragged_args(q=_desc([10, 2, 128]))
    flags = 0x6 if case == "flags" else 0
    assert _call_chunk(lib, a, lse, bro, co, flags) == binding.MLA_ERR_INVALID_ARG
    assert lib.mla_last_error_string()


@pytest.mark.parametrize("case", ["out_depth", "po_rows", "po_shape", "lse_shape", "lse_dtype",
                                  "no_ro", "no_bro", "batch0", "po_unaligned"])
def test_merge_rejects_bad_arguments(lib, case):
    out = _desc([10, 2, 128])
    po = _desc([3, 10, 2, 128], ptr=0x90000)
    pl = _desc([3, 10, 2], binding.MLA_DTYPE_F32, ptr=0xA0000)
    ro, bro, batch = 0x20000, 0x60000, 2
    if case == "out_depth":
        out = _desc([10, 2, 64])
    elif case == "po_rows":
        po, pl = _desc([0, 10, 2, 128]), _desc([0, 10, 2], binding.MLA_DTYPE_F32)
    elif case == "po_shape":
        po = _desc([3, 10, 3, 128])
    elif case == "lse_shape":
        pl = _desc([2, 10, 2], binding.MLA_DTYPE_F32)
    elif case == "lse_dtype":
        pl = _desc([3, 10, 2])
    elif case == "no_ro":
        ro = None
    elif case == "no_bro":
        bro = None
    elif case == "batch0":
        batch = 0
    elif case == "po_unaligned":
        po = _desc([3, 10, 2, 128], ptr=0x90008)
    r = lambda d: None if d is None else ctypes.byref(d)
    assert lib.mla_prefill_merge(r(out), r(po), r(pl), ro, bro, batch, None) == binding.MLA_ERR_INVALID_ARG
    assert lib.mla_last_error_string()


@pytest.mark.parametrize("case", ["rope_3d", "rope_rows", "rope_depth", "batch0", "rope_stride"])
def test_contiguous_rejects_bad_arguments(lib, case):
    a = _ragged_args()
    rope, batch = _desc([20, 64]), 2
    if case == "rope_3d":
        rope = _desc([4, 16, 64])
    elif case == "rope_rows":
        rope = _desc([19, 64])
    elif case == "rope_depth":
        rope = _desc([20, 32])
    elif case == "batch0":
        batch = 0
    elif case == "rope_stride":
        rope.stride[0] = 68       # 136 bytes
    r = ctypes.byref
    st = lib.mla_prefill_ragged_contiguous(r(a["out"]), r(a["q"]), r(a["k"]), r(a["v"]), r(rope),
                                           a["ro"], a["cl"], batch, a["scale"], a["mask"], a["ws"],
                                           a["ws_bytes"], None)
    assert st == binding.MLA_ERR_INVALID_ARG
    assert lib.mla_last_error_string()


def test_gather_rejects_bad_arguments(lib):
    r = ctypes.byref
    dst, cache = _desc([8, 576]), _desc([4, 16, 576])
    pt = _desc([2, 2], binding.MLA_DTYPE_U32)
    f = lib.mla_gather_rows
    ok = binding.MLA_ERR_INVALID_ARG
    assert f(r(_desc([8, 512])), r(cache), r(pt), 0x60000, 0x70000, None, None) == ok   # width
    assert f(r(dst), r(_desc([4, 16, 12])), r(pt), 0x60000, 0x70000, None, None) == ok  # 24-byte rows
    assert f(r(dst), r(cache), r(pt), None, 0x70000, None, None) == ok
    assert f(r(dst), r(cache), r(pt), 0x60000, None, None, None) == ok
    assert f(r(dst), r(cache), r(_desc([2, 2])), 0x60000, 0x70000, None, None) == ok  # table dtype
    assert f(r(dst), r(_desc([4, 16, 576], binding.MLA_DTYPE_U32)), r(pt), 0x60000, 0x70000, None,
             None) == ok


def test_up_project_rejects_bad_arguments(lib):
    r = ctypes.byref
    f = lib.mla_up_project
    bad = binding.MLA_ERR_INVALID_ARG
    out, lat, wt = _desc([8, 256]), _desc([8, 512]), _desc([256, 512])
    assert f(r(_desc([8, 128])), r(lat), r(wt), None, None) == bad       # N mismatch
    assert f(r(_desc([9, 256])), r(lat), r(wt), None, None) == bad       # rows mismatch
    assert f(r(out), r(_desc([8, 500])), r(wt), None, None) == bad       # K mismatch
    assert f(r(out), r(lat), r(_desc([256, 512], binding.MLA_DTYPE_F32)), None, None) == bad
    odd = _desc([8, 512])
    odd.stride[0] = 516                                                  # 1032-byte rows
    assert f(r(out), r(odd), r(wt), None, None) == bad
    unaligned = _desc([8, 512], ptr=0x10008)
    assert f(r(out), r(unaligned), r(wt), None, None) == bad
    assert f(r(out), r(_desc([8, 520])), r(_desc([256, 520])), None, None) == bad   # K above 512


@pytest.mark.parametrize("case", ["page_stride", "rank0", "rank_wide", "rank_odd", "v_without_w",
                                  "w_without_v", "no_bro", "no_co", "table_dtype", "k_rows", "w_k"])
def test_gather_up_project_rejects_bad_arguments(lib, case):
    r = lambda d: None if d is None else ctypes.byref(d)
    k_out, v_out = _desc([100, 256]), _desc([100, 256])
    cache, pt = _desc([4, 16, 576]), _desc([2, 3], binding.MLA_DTYPE_U32)
    w_uk, w_uv = _desc([256, 512]), _desc([256, 512])
    bro, co, rank = 0x60000, 0x70000, 512
    if case == "page_stride":
        cache.stride[0] = 16 * 576 + 64          # padded pages: not one row matrix
    elif case == "rank0":
        rank = 0
    elif case == "rank_wide":
        rank = 584
    elif case == "rank_odd":
        rank = 500
    elif case == "v_without_w":
        w_uv = None
    elif case == "w_without_v":
        v_out = None
    elif case == "no_bro":
        bro = None
    elif case == "no_co":
        co = None
    elif case == "table_dtype":
        pt = _desc([2, 3])
    elif case == "k_rows":
        k_out = _desc([100, 128])
    elif case == "w_k":
        w_uk = _desc([256, 448])
    st = lib.mla_gather_up_project(r(k_out), r(v_out), r(cache), r(w_uk), r(w_uv), r(pt), bro, co, rank,
                                   None, None)
    assert st == binding.MLA_ERR_INVALID_ARG, case
    assert lib.mla_last_error_string()


@pytest.mark.parametrize("case", ["no_q_rope", "q_nope_192", "q_rope_fp8", "q_rope_shape", "batch_rows",
                                  "batch0"])
def test_split_rejects_bad_arguments(lib, case):
    a = _ragged_args()
    qn, qr, batch, pt = _desc([10, 2, 128]), _desc([10, 2, 64]), 2, a["pt"]
    if case == "no_q_rope":
        qr = None
    elif case == "q_nope_192":
        qn = _desc([10, 2, 192])
    elif case == "q_rope_fp8":
        qr = _desc([10, 2, 64], binding.MLA_DTYPE_FP8_E4M3)
    elif case == "q_rope_shape":
        qr = _desc([10, 3, 64])
    elif case == "batch_rows":
        batch = 3
    elif case == "batch0":
        batch = 0
    r = lambda d: None if d is None else ctypes.byref(d)
    st = lib.mla_prefill_ragged_split(r(a["out"]), r(qn), r(qr), r(a["k"]), r(a["v"]), r(a["rope"]), r(pt),
                                      batch, a["ro"], a["cl"], a["scale"], a["mask"], a["ws"],
                                      a["ws_bytes"], None)
    assert st == binding.MLA_ERR_INVALID_ARG
    assert lib.mla_last_error_string()


def test_binding_refuses_host_tensors():
    """A host tensor's address must never reach a kernel: the binding raises
    before any call."""
    import torch
    t = torch.zeros(4, 2, 192, dtype=torch.bfloat16)
    with pytest.raises(binding.MlaError, match="CUDA tensor"):
        binding.describe(t, binding.MLA_DTYPE_BF16)
    with pytest.raises(binding.MlaError, match="CUDA tensor"):
        binding._ptr(torch.zeros(3, dtype=torch.int32))
    assert binding._ptr(None) is None


def test_ragged_rejects_batch_above_limit(lib):
    a = _ragged_args(pt=_desc([4097, 2], binding.MLA_DTYPE_U32))
    assert _call_ragged(lib, a) == binding.MLA_ERR_INVALID_ARG
    assert b"4096" in lib.mla_last_error_string()


def test_binding_k_scale_granularity_and_workspace_rows():
    """Host logic of the binding: a one-float k_scale is per tensor, a longer
    one per K row; fp8 workspaces then hold one converted K_rope row per K row
    instead of one per pool slot."""
    import torch
    k_nope = torch.empty(20, 2, 128, dtype=torch.uint8)
    assert not binding._per_token(None)
    assert not binding._per_token(torch.ones(1))
    assert binding._per_token(torch.ones(20))
    assert binding._rope_rows(k_nope, torch.ones(1), 64) == 64
    assert binding._rope_rows(k_nope, torch.ones(20), 64) == 20
    assert binding.workspace_size(3, fp8_pool_slots=20) == binding.workspace_size(3) + 20 * 128


@pytest.mark.parametrize("case", ["no_bro", "no_co", "no_num_rows", "max_rows0", "T0", "rows_overflow",
                                  "lse_shape", "few_k_rows", "accumulate", "split_bf16", "unknown_flag"])
def test_chunked_single_call_rejects_bad_arguments(lib, case):
    a = _ragged_args()
    bro, co, nrows, max_rows, T, lse, flags = 0x50000, 0x60000, 0x70000, 3, 8, None, 0
    if case == "no_bro":
        bro = None
    elif case == "no_co":
        co = None
    elif case == "no_num_rows":
        nrows = None
    elif case == "max_rows0":
        max_rows = 0
    elif case == "T0":
        T = 0
    elif case == "rows_overflow":
        max_rows, T = 1 << 20, 1 << 12
    elif case == "lse_shape":
        lse = _desc([10, 3], binding.MLA_DTYPE_F32)
    elif case == "few_k_rows":
        a = _ragged_args(k=_desc([5, 2, 128]), v=_desc([5, 2, 128]))
    elif case == "accumulate":
        flags = binding.MLA_CHUNK_ACCUMULATE
    elif case == "split_bf16":
        flags = binding.MLA_FP8_PRECISE
    elif case == "unknown_flag":
        flags = 0x80
    r = lambda d: None if d is None else ctypes.byref(d)
    st = lib.mla_prefill_ragged_chunked(r(a["out"]), r(lse), r(a["q"]), r(a["k"]), r(a["v"]), r(a["rope"]),
                                        r(a["pt"]), a["ro"], a["cl"], bro, co, nrows, max_rows, T, a["scale"],
                                        a["mask"], flags, a["ws"], a["ws_bytes"], None)
    assert st == binding.MLA_ERR_INVALID_ARG, case
    assert lib.mla_last_error_string()


@pytest.mark.parametrize("case", ["split_bf16", "accumulate", "unknown_flag", "lse_shape"])
def test_ragged_ex_rejects_bad_arguments(lib, case):
    a = _ragged_args()
    lse, flags = None, 0
    if case == "split_bf16":
        flags = binding.MLA_FP8_PRECISE
    elif case == "accumulate":
        flags = binding.MLA_CHUNK_ACCUMULATE
    elif case == "unknown_flag":
        flags = 0x40
    elif case == "lse_shape":
        lse = _desc([10, 3], binding.MLA_DTYPE_F32)
    r = lambda d: None if d is None else ctypes.byref(d)
    st = lib.mla_prefill_ragged_ex(r(a["out"]), r(lse), r(a["q"]), r(a["k"]), r(a["v"]), r(a["rope"]), r(a["pt"]),
                                   a["ro"], a["cl"], a["scale"], a["mask"], flags, a["ws"], a["ws_bytes"], None)
    assert st == binding.MLA_ERR_INVALID_ARG, case
    assert lib.mla_last_error_string()
