// pa_decode_simt.cu -- CUDA-core (FMA) instantiations of the paged decode
// kernel, and the log-sum-exp reduce kernel.
#include <cuda.h>

#include "pa_decode_kernel.cuh"
#include "pa_kernels.h"

namespace pa {

const void* decode_kernel_simt(pa_dtype kv, pa_dtype q, int D) {
#define PA_SIMT_CASE(KVT, QTT)                                                                  \
    if (D == 128) return reinterpret_cast<const void*>(&pa_decode_kernel<KVT, QTT, 128, false, 16>); \
    if (D == 64) return reinterpret_cast<const void*>(&pa_decode_kernel<KVT, QTT, 64, false, 16>);   \
    return nullptr;
    if (kv == PA_F32 && q == PA_F32) { PA_SIMT_CASE(F32T, F32T) }
    if (kv == PA_F16 && q == PA_F16) { PA_SIMT_CASE(F16T, F16T) }
    if (kv == PA_BF16 && q == PA_BF16) { PA_SIMT_CASE(BF16T, BF16T) }
    if (kv == PA_FP8_E4M3 && q == PA_F16 && D == 128)
        return reinterpret_cast<const void*>(&pa_decode_kernel<FP8T, F16T, 128, false, 16>);
    if (kv == PA_FP8_E4M3 && q == PA_BF16 && D == 128)
        return reinterpret_cast<const void*>(&pa_decode_kernel<FP8T, BF16T, 128, false, 16>);
    if (kv == PA_FP8_E5M2 && q == PA_F16 && D == 128)
        return reinterpret_cast<const void*>(&pa_decode_kernel<E5M2T, F16T, 128, false, 16>);
    if (kv == PA_FP8_E5M2 && q == PA_BF16 && D == 128)
        return reinterpret_cast<const void*>(&pa_decode_kernel<E5M2T, BF16T, 128, false, 16>);
#undef PA_SIMT_CASE
    return nullptr;
}

const void* reduce_kernel(pa_dtype out, int D, bool split_heads) {
#define PA_RED(T) \
    if (D == 128) return split_heads ? reinterpret_cast<const void*>(&pa_reduce_kernel<T, 128, RED_SPLIT_WARPS>) \
                                     : reinterpret_cast<const void*>(&pa_reduce_kernel<T, 128, 1>);          \
    if (D == 64) return split_heads ? reinterpret_cast<const void*>(&pa_reduce_kernel<T, 64, RED_SPLIT_WARPS>)  \
                                    : reinterpret_cast<const void*>(&pa_reduce_kernel<T, 64, 1>);            \
    return nullptr;
    if (out == PA_F32) { PA_RED(float) }
    if (out == PA_F16) { PA_RED(__half) }
    if (out == PA_BF16) { PA_RED(__nv_bfloat16) }
#undef PA_RED
    return nullptr;
}

}  // namespace pa
