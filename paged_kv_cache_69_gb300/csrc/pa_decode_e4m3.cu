// pa_decode_e4m3.cu -- native-fp8 tensor-core instantiations of the paged
// decode kernel (fp8 caches, head_dim 128, 32-token chunks, mma.sync
// m16n8k32: e4m3 query / probability terms times e4m3 or e5m2 K/V bytes,
// fp32 accumulation).
#include <cuda.h>

#include "pa_decode_kernel.cuh"
#include "pa_kernels.h"

namespace pa {

const void* decode_kernel_e4m3(pa_dtype kv, pa_dtype q, int D) {
    if (D != 128) return nullptr;
    if (kv == PA_FP8_E4M3) {
        if (q == PA_F16) return reinterpret_cast<const void*>(&pa_decode_kernel<FP8T, F16T, 128, true, 32>);
        if (q == PA_BF16) return reinterpret_cast<const void*>(&pa_decode_kernel<FP8T, BF16T, 128, true, 32>);
    }
    if (kv == PA_FP8_E5M2) {
        if (q == PA_F16) return reinterpret_cast<const void*>(&pa_decode_kernel<E5M2T, F16T, 128, true, 32>);
        if (q == PA_BF16) return reinterpret_cast<const void*>(&pa_decode_kernel<E5M2T, BF16T, 128, true, 32>);
    }
    return nullptr;
}

const void* decode_kernel_fp8t(pa_dtype kv, pa_dtype q, int D) {
#define PA_T8(KVT, QTT) reinterpret_cast<const void*>(&pa_decode_kernel<KVT, QTT, 128, true, 32, false, true>)
    if (D != 128) return nullptr;
    if (kv == PA_FP8_E4M3) return q == PA_F16 ? PA_T8(FP8T, F16T) : q == PA_BF16 ? PA_T8(FP8T, BF16T) : nullptr;
    if (kv == PA_FP8_E5M2) return q == PA_F16 ? PA_T8(E5M2T, F16T) : q == PA_BF16 ? PA_T8(E5M2T, BF16T) : nullptr;
#undef PA_T8
    return nullptr;
}

}  // namespace pa
