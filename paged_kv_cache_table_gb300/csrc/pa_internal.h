// Host-side helpers shared by the translation units of the library.
#pragma once

#include <cuda_runtime.h>

#include "pa.h"

namespace pa {

inline int dtype_bytes(pa_dtype t) { return t == PA_BF16 ? 2 : 1; }

inline bool is_quantized(const pa_cache_desc* d) { return d->k_dtype != PA_BF16; }

// Checks a cache description against what the kernels implement.
pa_status validate_desc(const pa_cache_desc* d);

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline pa_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
