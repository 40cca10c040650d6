// pa_attention.cu -- instantiations of the paged attention kernel for
// several query tokens per sequence (causal): the mma.sync variant and the
// tcgen05 variant (accumulators in tensor memory) for 16-bit caches.
#include <cuda.h>

#include "pa_decode_kernel.cuh"
#include "pa_kernels.h"

namespace pa {

const void* decode_kernel_mq(pa_dtype kv, pa_dtype q, int D) {
#define PA_MQ(KVT, QTT, DD) reinterpret_cast<const void*>(&pa_decode_kernel<KVT, QTT, DD, true, 16, true>)
    if (kv == PA_F16 && q == PA_F16) return D == 128 ? PA_MQ(F16T, F16T, 128) : D == 64 ? PA_MQ(F16T, F16T, 64) : nullptr;
    if (kv == PA_BF16 && q == PA_BF16) return D == 128 ? PA_MQ(BF16T, BF16T, 128) : D == 64 ? PA_MQ(BF16T, BF16T, 64) : nullptr;
    if (D != 128) return nullptr;
    if (kv == PA_FP8_E4M3) return q == PA_F16 ? PA_MQ(FP8T, F16T, 128) : q == PA_BF16 ? PA_MQ(FP8T, BF16T, 128) : nullptr;
    if (kv == PA_FP8_E5M2) return q == PA_F16 ? PA_MQ(E5M2T, F16T, 128) : q == PA_BF16 ? PA_MQ(E5M2T, BF16T, 128) : nullptr;
#undef PA_MQ
    return nullptr;
}

const void* decode_kernel_mq_um(pa_dtype kv, pa_dtype q, int D, int CT) {
#define PA_UM(KVT, DD, C) reinterpret_cast<const void*>(&pa_decode_kernel<KVT, KVT, DD, true, C, true, false, true>)
#define PA_UM_CT(KVT, DD) (CT == 32 ? PA_UM(KVT, DD, 32) : nullptr)
    if (kv == PA_F16 && q == PA_F16) return D == 128 ? PA_UM_CT(F16T, 128) : D == 64 ? PA_UM_CT(F16T, 64) : nullptr;
    if (kv == PA_BF16 && q == PA_BF16) return D == 128 ? PA_UM_CT(BF16T, 128) : D == 64 ? PA_UM_CT(BF16T, 64) : nullptr;
#undef PA_UM_CT
#undef PA_UM
    return nullptr;
}

}  // namespace pa
