// Host-side helpers shared by the entry points: per-thread error text, the
// device capability check and the tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>

#include "../../include/mla_prefill.h"

namespace mla {

// Record a failure for mla_last_error_string() and return `status`.
mla_status_t fail(mla_status_t status, const char* fmt, ...);
mla_status_t ok();

// Current device must be compute capability 10.3.  Fills the SM count.
mla_status_t check_device(int* device_out, int* num_sms_out);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).  Returns MLA_ERR_CUDA when the encoder rejects the map.
mla_status_t encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, void* base,
                          const uint64_t* dims, const uint64_t* strides_bytes,
                          const uint32_t* box, CUtensorMapSwizzle swizzle, const char* what);

bool aligned16(const void* ptr);

// Descriptor checks: non-NULL data, rank, dtype, shapes in [0, 2^31),
// non-negative strides, innermost stride 1.
mla_status_t check_tensor(const mla_tensor_t* t, const char* name, int ndim, mla_dtype_t dtype);

// Allow `bytes` of dynamic shared memory for `func` on `device`, cached per
// (device, slot): each kernel needs a slot of its own, 0..7 (0 plan,
// 1 scheduler, 2 / 3 / 4 attention bf16 / fp8 / fp8 with per-token K scales).
mla_status_t set_max_dynamic_smem(const void* func, int bytes, int device, int slot);

}  // namespace mla
