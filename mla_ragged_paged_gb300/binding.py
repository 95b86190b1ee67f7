"""ctypes binding for libmla_prefill (argument marshalling only).

Every computation happens in the CUDA library; this module turns torch CUDA
tensors into the C descriptors of include/mla_prefill.h and calls the entry
points on torch's current stream.  There is no fallback: if the library is
missing or the device is unsupported the call raises.
"""
import ctypes
import os

import torch

from .buildlib import LIB_PATH

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA = 0, 1, 2, 3
MLA_DTYPE_BF16, MLA_DTYPE_FP8_E4M3, MLA_DTYPE_U32, MLA_DTYPE_F32 = 0, 1, 2, 3
MLA_MASK_CAUSAL, MLA_MASK_NULL = 0, 1
MLA_SCALE_NONE, MLA_SCALE_PER_TENSOR, MLA_SCALE_PER_TOKEN = 0, 1, 2
MLA_CHUNK_ACCUMULATE = 0x1
MLA_FP8_PRECISE = 0x2
STATUS_BITS = {0x1: "BAD_PAGE", 0x2: "BAD_COLUMN", 0x4: "BAD_OFFSETS", 0x8: "TIMEOUT"}

# Names exported by the C ABI (kept in step with include/mla_prefill.h).
EXPORTS = ["mla_prefill_plan", "mla_prefill_plan_max_rows", "mla_prefill_ragged_workspace_size",
           "mla_prefill_ragged_workspace_size_fp8", "mla_prefill_ragged", "mla_prefill_ragged_ex",
           "mla_prefill_ragged_noalloc",
           "mla_prefill_ragged_chunk", "mla_prefill_ragged_chunked", "mla_prefill_merge",
           "mla_prefill_ragged_contiguous",
           "mla_prefill_ragged_chunk_contiguous", "mla_gather_rows", "mla_up_project",
           "mla_gather_up_project",
           "mla_prefill_ragged_split", "mla_test_inject_stall", "mla_test_delay_softmax",
           "mla_read_device_status",
           "mla_last_error_string"]


class MlaError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"libmla_prefill status {status}: {message}")
        self.status = status


class MlaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4),
                ("scale", ctypes.c_void_p), ("scale_gran", ctypes.c_int)]


_lib = None


def load(path=LIB_PATH):
    """Load the library (built beforehand by mla_ragged_paged_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise MlaError(-1, f"{path} is missing; build it with mla_ragged_paged_gb300.build()")
    lib = ctypes.CDLL(path)
    vp, u32, i32 = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int32
    lib.mla_prefill_plan.argtypes = [vp, vp, u32, u32, u32, vp, vp, vp, vp, vp]
    lib.mla_prefill_plan.restype = ctypes.c_int
    lib.mla_prefill_plan_max_rows.argtypes = [ctypes.c_uint64, u32]
    lib.mla_prefill_plan_max_rows.restype = u32
    lib.mla_prefill_ragged_workspace_size.argtypes = [u32]
    lib.mla_prefill_ragged_workspace_size.restype = ctypes.c_size_t
    lib.mla_prefill_ragged_workspace_size_fp8.argtypes = [u32, ctypes.c_uint64]
    lib.mla_prefill_ragged_workspace_size_fp8.restype = ctypes.c_size_t
    pt = ctypes.POINTER(MlaTensor)
    lib.mla_prefill_ragged.argtypes = [pt, pt, pt, pt, pt, pt, vp, vp, ctypes.c_float, ctypes.c_int,
                                       vp, ctypes.c_size_t, vp]
    lib.mla_prefill_ragged.restype = ctypes.c_int
    lib.mla_prefill_ragged_noalloc.argtypes = [pt, pt, pt, pt, pt, pt, vp, vp, ctypes.c_float,
                                               ctypes.c_int, vp]
    lib.mla_prefill_ragged_noalloc.restype = ctypes.c_int
    lib.mla_prefill_ragged_chunk.argtypes = [pt, pt, pt, pt, pt, pt, pt, vp, vp, vp, vp, ctypes.c_float,
                                             ctypes.c_int, u32, vp, ctypes.c_size_t, vp]
    lib.mla_prefill_ragged_chunk.restype = ctypes.c_int
    lib.mla_prefill_ragged_chunked.argtypes = [pt, pt, pt, pt, pt, pt, pt, vp, vp, vp, vp, vp, u32, u32,
                                               ctypes.c_float, ctypes.c_int, u32, vp, ctypes.c_size_t, vp]
    lib.mla_prefill_ragged_ex.argtypes = [pt, pt, pt, pt, pt, pt, pt, vp, vp, ctypes.c_float, ctypes.c_int, u32,
                                          vp, ctypes.c_size_t, vp]
    lib.mla_prefill_ragged_ex.restype = ctypes.c_int
    lib.mla_prefill_ragged_chunked.restype = ctypes.c_int
    lib.mla_prefill_merge.argtypes = [pt, pt, pt, vp, vp, u32, vp]
    lib.mla_prefill_merge.restype = ctypes.c_int
    lib.mla_prefill_ragged_contiguous.argtypes = [pt, pt, pt, pt, pt, vp, vp, u32, ctypes.c_float,
                                                  ctypes.c_int, vp, ctypes.c_size_t, vp]
    lib.mla_prefill_ragged_contiguous.restype = ctypes.c_int
    lib.mla_prefill_ragged_chunk_contiguous.argtypes = [pt, pt, pt, pt, pt, pt, vp, vp, vp, vp, u32,
                                                        ctypes.c_float, ctypes.c_int, u32, vp,
                                                        ctypes.c_size_t, vp]
    lib.mla_prefill_ragged_chunk_contiguous.restype = ctypes.c_int
    lib.mla_prefill_ragged_split.argtypes = [pt, pt, pt, pt, pt, pt, pt, u32, vp, vp, ctypes.c_float,
                                             ctypes.c_int, vp, ctypes.c_size_t, vp]
    lib.mla_prefill_ragged_split.restype = ctypes.c_int
    lib.mla_test_inject_stall.argtypes = [u32]
    lib.mla_test_inject_stall.restype = ctypes.c_int
    lib.mla_test_delay_softmax.argtypes = [u32]
    lib.mla_test_delay_softmax.restype = ctypes.c_int
    lib.mla_gather_rows.argtypes = [pt, pt, pt, vp, vp, vp, vp]
    lib.mla_gather_rows.restype = ctypes.c_int
    lib.mla_up_project.argtypes = [pt, pt, pt, vp, vp]
    lib.mla_up_project.restype = ctypes.c_int
    lib.mla_gather_up_project.argtypes = [pt, pt, pt, pt, pt, pt, vp, vp, u32, vp, vp]
    lib.mla_gather_up_project.restype = ctypes.c_int
    lib.mla_read_device_status.argtypes = [vp, ctypes.POINTER(u32), vp]
    lib.mla_read_device_status.restype = ctypes.c_int
    lib.mla_last_error_string.argtypes = []
    lib.mla_last_error_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status):
    if status != MLA_OK:
        raise MlaError(status, load().mla_last_error_string().decode())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _on_device(t, what="tensor"):
    """Every array the library reads or writes is device memory: a host
    tensor's address handed to a kernel would be an illegal access, so refuse
    it here."""
    if not t.is_cuda:
        raise MlaError(MLA_ERR_INVALID_ARG, f"{what} must be a CUDA tensor (got {t.device})")
    return t


def _ptr(t):
    return None if t is None else ctypes.c_void_p(_on_device(t).data_ptr())


def describe(t, dtype, scale=None, scale_gran=MLA_SCALE_NONE):
    """MlaTensor for a CUDA torch tensor (element strides, up to 4 dims)."""
    _on_device(t)
    if scale is not None:
        _on_device(scale, "scale")
    d = MlaTensor()
    d.data = t.data_ptr()
    d.dtype = dtype
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    d.scale = None if scale is None else scale.data_ptr()
    d.scale_gran = scale_gran
    return d


def _per_token(k_scale):
    """An fp8 k_scale of more than one float holds one scale per K row."""
    return k_scale is not None and k_scale.numel() > 1


def _kdesc(k_nope, k_scale, fp8):
    """k_nope's descriptor: fp8 scale per tensor (one float) or per K row."""
    if not fp8:
        return describe(k_nope, _dtype_code(k_nope))
    gran = MLA_SCALE_PER_TOKEN if _per_token(k_scale) else MLA_SCALE_PER_TENSOR
    return describe(k_nope, _dtype_code(k_nope), k_scale, gran)


def _rope_rows(k_nope, k_scale, pool_slots):
    """Rows of the converted K_rope' an fp8 workspace holds: one per pool slot,
    or one per K row with per-token K scales."""
    return k_nope.shape[0] if _per_token(k_scale) else pool_slots


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return MLA_DTYPE_BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return MLA_DTYPE_FP8_E4M3
    if t.dtype in (torch.int32,) or str(t.dtype) == "torch.uint32":
        return MLA_DTYPE_U32
    if t.dtype == torch.float32:
        return MLA_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def plan_max_rows(total_k_upper_bound, buffer_token_size):
    return int(load().mla_prefill_plan_max_rows(int(total_k_upper_bound), int(buffer_token_size)))


def plan(input_row_offsets, cache_lens, buffer_token_size, max_rows, stream=None, out=None):
    """mla_prefill_plan on device int32/uint32 tensors.  Returns
    (buffer_row_offsets [R_max,B+1], cache_offsets [R_max,B], buffer_lengths [R_max],
    num_rows [1]) as int32 device tensors holding the uint32 / int32 values."""
    lib = load()
    B = input_row_offsets.numel() - 1
    dev = input_row_offsets.device
    if out is None:
        bro = torch.empty((max_rows, B + 1), dtype=torch.int32, device=dev)
        co = torch.empty((max_rows, B), dtype=torch.int32, device=dev)
        blen = torch.empty((max_rows,), dtype=torch.int32, device=dev)
        nrows = torch.empty((1,), dtype=torch.int32, device=dev)
    else:
        bro, co, blen, nrows = out
    _check(lib.mla_prefill_plan(_ptr(input_row_offsets), _ptr(cache_lens), B, int(buffer_token_size),
                                int(max_rows), _ptr(bro), _ptr(co), _ptr(blen), _ptr(nrows),
                                _stream(stream)))
    return bro, co, blen, nrows


def workspace_size(batch, fp8_pool_slots=None):
    """Workspace bytes for `batch` sequences; pass the K_rope pool's slot count
    (num_pages * P) for fp8 inputs."""
    if fp8_pool_slots is not None:
        return int(load().mla_prefill_ragged_workspace_size_fp8(int(batch), int(fp8_pool_slots)))
    return int(load().mla_prefill_ragged_workspace_size(int(batch)))


def alloc_workspace(batch, device="cuda", fp8_pool_slots=None):
    return torch.zeros(workspace_size(batch, fp8_pool_slots), dtype=torch.uint8, device=device)


def prefill_ragged(out, q, k_nope, v, k_rope_pages, page_table, row_offsets, cache_lens, scale,
                   mask=MLA_MASK_CAUSAL, workspace=None, q_scale=None, k_scale=None, v_scale=None,
                   k_rope_scales=None, stream=None):
    """mla_prefill_ragged.  fp8 inputs take per-tensor scale tensors (1 float on
    the device) and a per-token K_rope scale tensor [num_pages, P]."""
    lib = load()
    B = page_table.shape[0]
    fp8 = _dtype_code(q) == MLA_DTYPE_FP8_E4M3
    if workspace is None:
        slots = _rope_rows(k_nope, k_scale, k_rope_pages.shape[0] * k_rope_pages.shape[1]) if fp8 else None
        workspace = alloc_workspace(B, q.device, slots)
    gran_t = MLA_SCALE_PER_TENSOR if fp8 else MLA_SCALE_NONE
    d_out = describe(out, MLA_DTYPE_BF16)
    d_q = describe(q, _dtype_code(q), q_scale if fp8 else None, gran_t)
    d_k = _kdesc(k_nope, k_scale, fp8)
    d_v = describe(v, _dtype_code(v), v_scale if fp8 else None, gran_t)
    d_r = describe(k_rope_pages, _dtype_code(k_rope_pages), k_rope_scales if fp8 else None,
                   MLA_SCALE_PER_TOKEN if fp8 else MLA_SCALE_NONE)
    d_pt = describe(page_table, MLA_DTYPE_U32)
    _check(lib.mla_prefill_ragged(ctypes.byref(d_out), ctypes.byref(d_q), ctypes.byref(d_k),
                                  ctypes.byref(d_v), ctypes.byref(d_r), ctypes.byref(d_pt),
                                  _ptr(row_offsets), _ptr(cache_lens), float(scale), int(mask),
                                  _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def prefill_ragged_ex(out, q, k_nope, v, k_rope_pages, page_table, row_offsets, cache_lens, scale,
                      mask=MLA_MASK_CAUSAL, workspace=None, lse=None, flags=0, q_scale=None, k_scale=None,
                      v_scale=None, k_rope_scales=None, stream=None):
    """mla_prefill_ragged_ex: mla_prefill_ragged with an optional lse [Tq, H]
    float32 output and flags (MLA_FP8_PRECISE)."""
    lib = load()
    B = page_table.shape[0]
    fp8 = _dtype_code(q) == MLA_DTYPE_FP8_E4M3
    if workspace is None:
        slots = _rope_rows(k_nope, k_scale, k_rope_pages.shape[0] * k_rope_pages.shape[1]) if fp8 else None
        if slots is not None and flags & MLA_FP8_PRECISE:
            slots *= 2
        workspace = alloc_workspace(B, q.device, slots)
    d_q, d_k, d_v, d_r, d_pt = _inputs(q, k_nope, v, k_rope_pages, page_table, q_scale, k_scale,
                                       v_scale, k_rope_scales)
    d_out = describe(out, MLA_DTYPE_BF16)
    d_lse = describe(lse, MLA_DTYPE_F32) if lse is not None else None
    _check(lib.mla_prefill_ragged_ex(ctypes.byref(d_out), ctypes.byref(d_lse) if d_lse is not None else None,
                                     ctypes.byref(d_q), ctypes.byref(d_k), ctypes.byref(d_v), ctypes.byref(d_r),
                                     ctypes.byref(d_pt), _ptr(row_offsets), _ptr(cache_lens), float(scale),
                                     int(mask), int(flags), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def _inputs(q, k_nope, v, k_rope_pages, page_table, q_scale, k_scale, v_scale, k_rope_scales):
    fp8 = _dtype_code(q) == MLA_DTYPE_FP8_E4M3
    gran_t = MLA_SCALE_PER_TENSOR if fp8 else MLA_SCALE_NONE
    return (describe(q, _dtype_code(q), q_scale if fp8 else None, gran_t),
            _kdesc(k_nope, k_scale, fp8),
            describe(v, _dtype_code(v), v_scale if fp8 else None, gran_t),
            describe(k_rope_pages, _dtype_code(k_rope_pages), k_rope_scales if fp8 else None,
                     MLA_SCALE_PER_TOKEN if fp8 else MLA_SCALE_NONE),
            describe(page_table, MLA_DTYPE_U32))


def prefill_ragged_chunk(out, lse, q, k_nope, v, k_rope_pages, page_table, row_offsets, cache_lens,
                         buffer_row_offsets, cache_offsets, scale, mask=MLA_MASK_CAUSAL,
                         workspace=None, q_scale=None, k_scale=None, v_scale=None, k_rope_scales=None,
                         stream=None, flags=0):
    """mla_prefill_ragged_chunk: one buffer row.  k_nope / v are the row's K
    buffer; buffer_row_offsets [B+1] and cache_offsets [B] are that row of the
    plan (device int32 views of the uint32 values); lse is float32 [Tq, H].
    flags=MLA_CHUNK_ACCUMULATE folds the row into out / lse."""
    lib = load()
    B = page_table.shape[0]
    fp8 = _dtype_code(q) == MLA_DTYPE_FP8_E4M3
    if workspace is None:
        slots = _rope_rows(k_nope, k_scale, k_rope_pages.shape[0] * k_rope_pages.shape[1]) if fp8 else None
        if slots is not None and flags & MLA_FP8_PRECISE:
            slots *= 2
        workspace = alloc_workspace(B, q.device, slots)
    d_q, d_k, d_v, d_r, d_pt = _inputs(q, k_nope, v, k_rope_pages, page_table, q_scale, k_scale,
                                       v_scale, k_rope_scales)
    d_out = describe(out, MLA_DTYPE_BF16)
    d_lse = describe(lse, MLA_DTYPE_F32)
    _check(lib.mla_prefill_ragged_chunk(ctypes.byref(d_out), ctypes.byref(d_lse), ctypes.byref(d_q),
                                        ctypes.byref(d_k), ctypes.byref(d_v), ctypes.byref(d_r),
                                        ctypes.byref(d_pt), _ptr(row_offsets), _ptr(cache_lens),
                                        _ptr(buffer_row_offsets), _ptr(cache_offsets), float(scale),
                                        int(mask), int(flags), _ptr(workspace), workspace.numel(),
                                        _stream(stream)))
    return out, lse


def prefill_ragged_contiguous(out, q, k_nope, v, k_rope, row_offsets, cache_lens, scale,
                              mask=MLA_MASK_CAUSAL, workspace=None, q_scale=None, k_scale=None,
                              v_scale=None, k_rope_scales=None, stream=None):
    """mla_prefill_ragged_contiguous: k_rope is [Sk, 64], row r the rope part of
    k_nope row r; fp8 inputs take one K_rope scale per row ([Sk] float32)."""
    lib = load()
    B = row_offsets.numel() - 1
    fp8 = _dtype_code(q) == MLA_DTYPE_FP8_E4M3
    if workspace is None:
        workspace = alloc_workspace(B, q.device, _rope_rows(k_nope, k_scale, k_rope.shape[0]) if fp8 else None)
    gran_t = MLA_SCALE_PER_TENSOR if fp8 else MLA_SCALE_NONE
    d_out = describe(out, MLA_DTYPE_BF16)
    d_q = describe(q, _dtype_code(q), q_scale if fp8 else None, gran_t)
    d_k = _kdesc(k_nope, k_scale, fp8)
    d_v = describe(v, _dtype_code(v), v_scale if fp8 else None, gran_t)
    d_r = describe(k_rope, _dtype_code(k_rope), k_rope_scales if fp8 else None,
                   MLA_SCALE_PER_TOKEN if fp8 else MLA_SCALE_NONE)
    _check(lib.mla_prefill_ragged_contiguous(ctypes.byref(d_out), ctypes.byref(d_q), ctypes.byref(d_k),
                                             ctypes.byref(d_v), ctypes.byref(d_r), _ptr(row_offsets),
                                             _ptr(cache_lens), B, float(scale), int(mask),
                                             _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def prefill_ragged_chunk_contiguous(out, lse, q, k_nope, v, k_rope, row_offsets, cache_lens,
                                    buffer_row_offsets, cache_offsets, scale, mask=MLA_MASK_CAUSAL,
                                    workspace=None, q_scale=None, k_scale=None, v_scale=None,
                                    k_rope_scales=None, stream=None, flags=0):
    """mla_prefill_ragged_chunk_contiguous: one buffer row whose K_rope is the
    row's own [S_row, 64] tensor (row t = buffer position t)."""
    lib = load()
    B = row_offsets.numel() - 1
    fp8 = _dtype_code(q) == MLA_DTYPE_FP8_E4M3
    if workspace is None:
        workspace = alloc_workspace(B, q.device, _rope_rows(k_nope, k_scale, k_rope.shape[0]) if fp8 else None)
    gran_t = MLA_SCALE_PER_TENSOR if fp8 else MLA_SCALE_NONE
    d_out, d_lse = describe(out, MLA_DTYPE_BF16), describe(lse, MLA_DTYPE_F32)
    d_q = describe(q, _dtype_code(q), q_scale if fp8 else None, gran_t)
    d_k = _kdesc(k_nope, k_scale, fp8)
    d_v = describe(v, _dtype_code(v), v_scale if fp8 else None, gran_t)
    d_r = describe(k_rope, _dtype_code(k_rope), k_rope_scales if fp8 else None,
                   MLA_SCALE_PER_TOKEN if fp8 else MLA_SCALE_NONE)
    _check(lib.mla_prefill_ragged_chunk_contiguous(
        ctypes.byref(d_out), ctypes.byref(d_lse), ctypes.byref(d_q), ctypes.byref(d_k), ctypes.byref(d_v),
        ctypes.byref(d_r), _ptr(row_offsets), _ptr(cache_lens), _ptr(buffer_row_offsets),
        _ptr(cache_offsets), B, float(scale), int(mask), int(flags), _ptr(workspace), workspace.numel(),
        _stream(stream)))
    return out, lse


def prefill_ragged_split(out, q_nope, q_rope, k_nope, v, k_rope, page_table, row_offsets, cache_lens,
                         scale, mask=MLA_MASK_CAUSAL, workspace=None, q_scale=None, k_scale=None,
                         v_scale=None, k_rope_scales=None, stream=None):
    """mla_prefill_ragged_split: Q as q_nope (bf16, or fp8 with q_scale) plus a
    bf16 q_rope; page_table None means k_rope is contiguous [Sk, 64].  fp8 v
    without v_scale uses k_scale."""
    lib = load()
    B = row_offsets.numel() - 1
    fp8 = _dtype_code(q_nope) == MLA_DTYPE_FP8_E4M3
    if workspace is None:
        slots = (k_rope.shape[0] * k_rope.shape[1] if page_table is not None else k_rope.shape[0]) if fp8 else None
        slots = _rope_rows(k_nope, k_scale, slots) if fp8 else None
        workspace = alloc_workspace(B, q_nope.device, slots)
    gran_t = MLA_SCALE_PER_TENSOR if fp8 else MLA_SCALE_NONE
    d_out = describe(out, MLA_DTYPE_BF16)
    d_qn = describe(q_nope, _dtype_code(q_nope), q_scale if fp8 else None, gran_t)
    d_qr = describe(q_rope, MLA_DTYPE_BF16)
    d_k = _kdesc(k_nope, k_scale, fp8)
    d_v = describe(v, _dtype_code(v), v_scale if fp8 else None, gran_t if v_scale is not None else MLA_SCALE_NONE)
    d_r = describe(k_rope, _dtype_code(k_rope), k_rope_scales if fp8 else None,
                   MLA_SCALE_PER_TOKEN if fp8 else MLA_SCALE_NONE)
    d_pt = describe(page_table, MLA_DTYPE_U32) if page_table is not None else None
    _check(lib.mla_prefill_ragged_split(ctypes.byref(d_out), ctypes.byref(d_qn), ctypes.byref(d_qr),
                                        ctypes.byref(d_k), ctypes.byref(d_v), ctypes.byref(d_r),
                                        ctypes.byref(d_pt) if d_pt is not None else None, B,
                                        _ptr(row_offsets), _ptr(cache_lens), float(scale), int(mask),
                                        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def gather_rows(dst, cache, page_table, buffer_row_offsets, cache_offsets, status=None, stream=None):
    """mla_gather_rows: dst[bro[b] + i] = cache row of context token co[b] + i of sequence b."""
    code = _dtype_code(cache)
    d_dst, d_cache = describe(dst, code), describe(cache, code)
    d_pt = describe(page_table, MLA_DTYPE_U32)
    _check(load().mla_gather_rows(ctypes.byref(d_dst), ctypes.byref(d_cache), ctypes.byref(d_pt),
                                  _ptr(buffer_row_offsets), _ptr(cache_offsets), _ptr(status),
                                  _stream(stream)))
    return dst


def up_project(out, latent, weight, status=None, stream=None):
    """mla_up_project: out [rows, N] = latent [rows, K] x weight [N, K]^T (bf16)."""
    d_out = describe(out, MLA_DTYPE_BF16)
    d_lat = describe(latent, MLA_DTYPE_BF16)
    d_w = describe(weight, MLA_DTYPE_BF16)
    _check(load().mla_up_project(ctypes.byref(d_out), ctypes.byref(d_lat), ctypes.byref(d_w),
                                 _ptr(status), _stream(stream)))
    return out


def gather_up_project(k_out, v_out, cache, w_uk, w_uv, page_table, buffer_row_offsets, cache_offsets,
                      kv_lora_rank=512, status=None, stream=None):
    """mla_gather_up_project: K_nope and V of one buffer row, projected from the
    c_kv columns of its cache rows, gathered through the page table inside the
    GEMM.  k_out / v_out are [rows, N] (or [rows, H, 128]); v_out and w_uv may
    both be None."""
    def flat(t):
        return t.reshape(t.shape[0], -1) if t is not None and t.dim() == 3 else t
    k_out, v_out = flat(k_out), flat(v_out)
    d_k = describe(k_out, MLA_DTYPE_BF16)
    d_v = describe(v_out, MLA_DTYPE_BF16) if v_out is not None else None
    d_c = describe(cache, MLA_DTYPE_BF16)
    d_uk = describe(w_uk, MLA_DTYPE_BF16)
    d_uv = describe(w_uv, MLA_DTYPE_BF16) if w_uv is not None else None
    d_pt = describe(page_table, MLA_DTYPE_U32)
    ref = lambda d: ctypes.byref(d) if d is not None else None
    _check(load().mla_gather_up_project(ctypes.byref(d_k), ref(d_v), ctypes.byref(d_c), ctypes.byref(d_uk),
                                        ref(d_uv), ctypes.byref(d_pt), _ptr(buffer_row_offsets),
                                        _ptr(cache_offsets), int(kv_lora_rank), _ptr(status),
                                        _stream(stream)))


class LatentRowBuffers:
    """Per-row scratch of the latent path: the projected K_nope / V [T, H, 128]."""
    def __init__(self, T, heads, device="cuda"):
        self.k_nope = torch.empty((T, heads, 128), dtype=torch.bfloat16, device=device)
        self.v = torch.empty((T, heads, 128), dtype=torch.bfloat16, device=device)


def latent_rope_pages(cache, kv_lora_rank=512):
    """The K_rope part of a paged latent cache [num_pages, P, W] as a paged
    K_rope view [num_pages, P, 64] (token stride W)."""
    return cache[:, :, kv_lora_rank:kv_lora_rank + 64]


def prefill_latent_row(po, pl, q, cache, page_table, row_offsets, cache_lens, bro_r, co_r, w_uk,
                       w_uv, scale, buffers, rows_in_row, mask=MLA_MASK_CAUSAL, workspace=None,
                       status=None, kv_lora_rank=512, stream=None, flags=0):
    """One buffer row from the paged latent cache: K_nope and V projected from
    the gathered c_kv rows (one launch), then the row's attention with K_rope
    read from the same cache through the page table."""
    n = int(rows_in_row)
    kn, v = buffers.k_nope[:n], buffers.v[:n]
    gather_up_project(kn, v, cache, w_uk, w_uv, page_table, bro_r, co_r, kv_lora_rank, status, stream)
    return prefill_ragged_chunk(po, pl, q, kn, v, latent_rope_pages(cache, kv_lora_rank), page_table,
                                row_offsets, cache_lens, bro_r, co_r, scale, mask, workspace,
                                stream=stream, flags=flags)


def merge(out, partial_out, partial_lse, row_offsets, buffer_row_offsets, stream=None):
    """mla_prefill_merge over rows 0..R-1 (R = partial_out.shape[0]);
    buffer_row_offsets is the plan's [R_max, B+1] array."""
    B = row_offsets.numel() - 1
    if buffer_row_offsets.shape[-1] != B + 1 or (buffer_row_offsets.dim() > 1
                                                  and buffer_row_offsets.stride(0) != B + 1):
        raise MlaError(MLA_ERR_INVALID_ARG, "buffer_row_offsets must hold rows of B+1 packed offsets")
    d_out = describe(out, MLA_DTYPE_BF16)
    d_po = describe(partial_out, MLA_DTYPE_BF16)
    d_pl = describe(partial_lse, MLA_DTYPE_F32)
    _check(load().mla_prefill_merge(ctypes.byref(d_out), ctypes.byref(d_po), ctypes.byref(d_pl),
                                    _ptr(row_offsets), _ptr(buffer_row_offsets), B, _stream(stream)))
    return out


def chunked_scratch(num_rows, total_q, heads, device="cuda"):
    """Per-row partial outputs [R, Tq, H, 128] bf16 and lse [R, Tq, H] float32."""
    return (torch.empty((num_rows, total_q, heads, 128), dtype=torch.bfloat16, device=device),
            torch.empty((num_rows, total_q, heads), dtype=torch.float32, device=device))


def prefill_ragged_chunked(out, q, k_nope, v, k_rope_pages, page_table, row_offsets, cache_lens,
                           buffer_row_offsets, cache_offsets, num_rows, buffer_token_size, scale,
                           mask=MLA_MASK_CAUSAL, workspace=None, lse=None, q_scale=None, k_scale=None,
                           v_scale=None, k_rope_scales=None, stream=None, flags=0):
    """mla_prefill_ragged_chunked: every buffer row of the plan in one call.
    buffer_row_offsets [max_rows, B+1] / cache_offsets [max_rows, B] / num_rows
    [1] are the plan's device outputs; k_nope / v hold the rows' K buffers
    stacked buffer_token_size rows apart."""
    lib = load()
    B = page_table.shape[0]
    fp8 = _dtype_code(q) == MLA_DTYPE_FP8_E4M3
    if workspace is None:
        slots = _rope_rows(k_nope, k_scale, k_rope_pages.shape[0] * k_rope_pages.shape[1]) if fp8 else None
        if slots is not None and flags & MLA_FP8_PRECISE:
            slots *= 2
        workspace = alloc_workspace(B, q.device, slots)
    if buffer_row_offsets.dim() != 2 or buffer_row_offsets.shape[1] != B + 1 or \
            buffer_row_offsets.stride(0) != B + 1 or cache_offsets.dim() != 2 or \
            cache_offsets.shape != (buffer_row_offsets.shape[0], B) or cache_offsets.stride(0) != B:
        raise MlaError(MLA_ERR_INVALID_ARG, "plan arrays must be packed [max_rows, B+1] and [max_rows, B]")
    d_q, d_k, d_v, d_r, d_pt = _inputs(q, k_nope, v, k_rope_pages, page_table, q_scale, k_scale,
                                       v_scale, k_rope_scales)
    d_out = describe(out, MLA_DTYPE_BF16)
    d_lse = describe(lse, MLA_DTYPE_F32) if lse is not None else None
    _check(lib.mla_prefill_ragged_chunked(ctypes.byref(d_out), ctypes.byref(d_lse) if d_lse is not None else None,
                                          ctypes.byref(d_q), ctypes.byref(d_k), ctypes.byref(d_v),
                                          ctypes.byref(d_r), ctypes.byref(d_pt), _ptr(row_offsets),
                                          _ptr(cache_lens), _ptr(buffer_row_offsets), _ptr(cache_offsets),
                                          _ptr(num_rows), int(buffer_row_offsets.shape[0]),
                                          int(buffer_token_size), float(scale), int(mask), int(flags),
                                          _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def prefill_chunked(out, q, k_nope, v, k_rope_pages, page_table, row_offsets, cache_lens, scale,
                    buffer_token_size, max_rows, mask=MLA_MASK_CAUSAL, workspace=None, q_scale=None,
                    k_scale=None, v_scale=None, k_rope_scales=None, stream=None, lse=None, plan_out=None):
    """Chunked execution: mla_prefill_plan, then mla_prefill_ragged_chunked over
    all its rows.  k_nope / v hold the contexts packed in batch order, i.e. the
    rows' K buffers stacked buffer_token_size rows apart; max_rows (host int)
    is the plan's capacity, at least ceil(total context / buffer_token_size)."""
    bro, co, _, nrows = plan(row_offsets, cache_lens, buffer_token_size, max_rows, stream=stream,
                             out=plan_out)
    return prefill_ragged_chunked(out, q, k_nope, v, k_rope_pages, page_table, row_offsets, cache_lens,
                                  bro, co, nrows, buffer_token_size, scale, mask, workspace, lse, q_scale,
                                  k_scale, v_scale, k_rope_scales, stream)


def prefill_ragged_noalloc(out, q, k_nope, v, k_rope_pages, page_table, row_offsets, cache_lens,
                           scale, mask=MLA_MASK_CAUSAL, stream=None):
    """mla_prefill_ragged_noalloc (bf16 inputs): the same attention without a
    caller workspace, for callers that cannot allocate device memory; the
    library's built-in workspace holds up to 1024 sequences and is shared by
    every call, so calls must not overlap on the GPU."""
    lib = load()
    d_out = describe(out, MLA_DTYPE_BF16)
    d_q = describe(q, _dtype_code(q))
    d_k = describe(k_nope, _dtype_code(k_nope))
    d_v = describe(v, _dtype_code(v))
    d_r = describe(k_rope_pages, _dtype_code(k_rope_pages))
    d_pt = describe(page_table, MLA_DTYPE_U32)
    _check(lib.mla_prefill_ragged_noalloc(ctypes.byref(d_out), ctypes.byref(d_q), ctypes.byref(d_k),
                                          ctypes.byref(d_v), ctypes.byref(d_r), ctypes.byref(d_pt),
                                          _ptr(row_offsets), _ptr(cache_lens), float(scale),
                                          int(mask), _stream(stream)))
    return out


def test_inject_stall(enable):
    """mla_test_inject_stall: make attention launches run into their wait
    timeout (tests of the timeout path only)."""
    _check(load().mla_test_inject_stall(1 if enable else 0))


def test_delay_softmax(nanoseconds):
    """mla_test_delay_softmax: delay the second query tile's softmax before
    every score-tile load (tests of the pipeline's ordering only)."""
    _check(load().mla_test_delay_softmax(int(nanoseconds)))


def device_status(workspace, stream=None):
    """Synchronising read of the workspace status word (0 = ok)."""
    val = ctypes.c_uint32(0)
    _check(load().mla_read_device_status(_ptr(workspace), ctypes.byref(val), _stream(stream)))
    return int(val.value)
