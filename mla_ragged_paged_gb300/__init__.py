"""libmla_prefill: MLA ragged paged prefill for one sm_103 GPU.

The compute lives in the CUDA library ``libmla_prefill.so`` (C ABI declared in
include/mla_prefill.h); ``binding`` marshals torch tensors into its calls.
"""
from .buildlib import LIB_PATH, build  # noqa: F401
