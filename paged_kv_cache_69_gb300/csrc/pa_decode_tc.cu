// pa_decode_tc.cu -- tensor-core (mma.sync m16n8k16, fp32 accumulate)
// instantiations of the paged decode kernel.
#include <cuda.h>

#include "pa_decode_kernel.cuh"
#include "pa_kernels.h"

namespace pa {

const void* decode_kernel_tc(pa_dtype kv, pa_dtype q, int D) {
    if (kv == PA_F16 && q == PA_F16) {
        if (D == 128) return reinterpret_cast<const void*>(&pa_decode_kernel<F16T, F16T, 128, true, 16>);
        if (D == 64) return reinterpret_cast<const void*>(&pa_decode_kernel<F16T, F16T, 64, true, 16>);
    }
    if (kv == PA_BF16 && q == PA_BF16) {
        if (D == 128) return reinterpret_cast<const void*>(&pa_decode_kernel<BF16T, BF16T, 128, true, 16>);
        if (D == 64) return reinterpret_cast<const void*>(&pa_decode_kernel<BF16T, BF16T, 64, true, 16>);
    }
    if (kv == PA_FP8_E4M3 && D == 128) {
        if (q == PA_F16) return reinterpret_cast<const void*>(&pa_decode_kernel<FP8T, F16T, 128, true, 16>);
        if (q == PA_BF16) return reinterpret_cast<const void*>(&pa_decode_kernel<FP8T, BF16T, 128, true, 16>);
    }
    if (kv == PA_FP8_E5M2 && D == 128) {
        if (q == PA_F16) return reinterpret_cast<const void*>(&pa_decode_kernel<E5M2T, F16T, 128, true, 16>);
        if (q == PA_BF16) return reinterpret_cast<const void*>(&pa_decode_kernel<E5M2T, BF16T, 128, true, 16>);
    }
    return nullptr;
}

}  // namespace pa
