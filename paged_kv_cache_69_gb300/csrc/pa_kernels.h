// pa_kernels.h -- lookup of the decode kernel instantiations (host side).
#pragma once

#include "../../include/pa.h"

namespace pa {
// Kernel entry for the given cache dtype, query dtype and head_dim, or null.
const void* decode_kernel_tc(pa_dtype kv, pa_dtype q, int D);
const void* decode_kernel_simt(pa_dtype kv, pa_dtype q, int D);
// fp8 cache (e4m3 or e5m2), tensor cores with fp8 operands, 32-token chunks.
const void* decode_kernel_e4m3(pa_dtype kv, pa_dtype q, int D);
// the same for GQA groups of at most 4 heads: keys as the MMA rows.
const void* decode_kernel_fp8t(pa_dtype kv, pa_dtype q, int D);
// several (causal) query tokens per sequence, tensor cores.
const void* decode_kernel_mq(pa_dtype kv, pa_dtype q, int D);
// the same on the 5th-generation tensor cores (tcgen05, accumulators in
// tensor memory), 16-bit caches, more than 16 (token, head) rows per KV
// head; chunks of CT = 32 tokens.
const void* decode_kernel_mq_um(pa_dtype kv, pa_dtype q, int D, int CT);
// Log-sum-exp merge; split_heads: several warps per (sequence, head), for
// partitioned sequences with many partials.
const void* reduce_kernel(pa_dtype out, int D, bool split_heads);
}  // namespace pa
