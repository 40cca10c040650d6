// pa_common.h -- host-side helpers shared by the library's translation units:
// status reporting (a thread-local detail string) and argument checks.
#pragma once

#include <cmath>
#include <cstdint>
#include <cuda_runtime_api.h>

#include "../../include/pa.h"

namespace pa {

void clear_error();
pa_status fail(pa_status s, const char* what);
pa_status fail_cuda(const char* what, cudaError_t e);

inline bool is_fp8(pa_dtype d) { return d == PA_FP8_E4M3 || d == PA_FP8_E5M2; }
inline bool valid_dtype(pa_dtype d) { return d == PA_F32 || d == PA_F16 || d == PA_BF16 || is_fp8(d); }
inline int dtype_bytes(pa_dtype d) { return d == PA_F32 ? 4 : (is_fp8(d) ? 1 : 2); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool isfinite_host(float x) { return std::isfinite(x); }

}  // namespace pa
