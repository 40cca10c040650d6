// pa_noalloc.cu -- pa_decode_noalloc: paged decode attention for callers that
// cannot hand the library a workspace buffer.
//
// pa_decode needs a caller-owned device workspace for its split-KV partials.
// Some callers cannot provide one at the call site: a serving loop whose
// device memory is entirely pre-partitioned by its own allocator and which
// forbids further cudaMalloc calls, or a plugin running inside a host
// framework that owns all device memory and gives plugins none.  This entry
// point serves them with scratch memory that lives inside the library: a
// fixed-size array in device global memory, created when the library is
// loaded on a device and kept until the process exits.
//
// Rules for callers:
//  * The first call on each device resolves the array's device address
//    (cudaGetSymbolAddress, with that device current).  Make that first call
//    before any stream capture on the device.
//  * Problems whose partials need more than PA_NOALLOC_SCRATCH_BYTES are
//    rejected with PA_ERR_WORKSPACE; nothing is launched.
//  * Every call on a device shares the one array, and the array keeps what
//    the previous call left in it.  Calls whose GPU work overlaps (other
//    streams, other host threads) race on it and give wrong results; order
//    them on one stream or serialise them.  Nothing in the array has to start
//    at zero: the decode kernels initialise everything they read.
//  * No device memory is allocated or freed by this call.
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "pa_common.h"

namespace pa {

// 32 MiB: enough for the partials of a 64-sequence, 28-head, head_dim-128
// decode batch (about 5.4 MB) or of 8 long sequences with 32 heads.
constexpr size_t kNoallocScratchBytes = PA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch on the current device, resolved once
// per device.
static pa_status noalloc_scratch(void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda("decode_noalloc: cudaGetDevice", e);
    if (dev < 0 || dev >= 64) return fail(PA_ERR_UNSUPPORTED, "decode_noalloc: device ordinal above 63");
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return fail_cuda("decode_noalloc: cudaGetSymbolAddress of the scratch array", e);
        addr[dev] = p;
    }
    *out = addr[dev];
    return PA_OK;
}

}  // namespace pa

using namespace pa;

extern "C" pa_status pa_decode_noalloc(void* out, const void* q, pa_dtype q_dtype, const void* k_cache,
                                       const void* v_cache, pa_dtype kv_dtype, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                       int num_blocks, float scale, float k_scale, float v_scale,
                                       int partition_tokens, int32_t* err_flag, cudaStream_t stream) {
    clear_error();
    if (num_seqs == 0) return PA_OK;
    if (num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 || block_size <= 0 ||
        static_cast<long long>(max_blocks_per_seq) * block_size >= (1LL << 30))
        return fail(PA_ERR_INVALID_ARG, "decode_noalloc: sizes must be positive");
    int dev = 0;
    const cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return fail_cuda("decode_noalloc: no current device", de);
    const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, max_blocks_per_seq * block_size,
                                                 head_dim, partition_tokens);
    if (need == 0) return fail(PA_ERR_INVALID_ARG, "decode_noalloc: invalid sizes for the scratch bound");
    if (need > kNoallocScratchBytes) {
        char msg[200];
        std::snprintf(msg, sizeof msg,
                      "decode_noalloc: this batch needs %zu bytes of scratch but the built-in scratch holds %zu; "
                      "use pa_decode with a caller workspace", need, kNoallocScratchBytes);
        return fail(PA_ERR_WORKSPACE, msg);
    }
    void* scratch = nullptr;
    const pa_status st = noalloc_scratch(&scratch);
    if (st != PA_OK) return st;
    return pa_decode(out, q, q_dtype, k_cache, v_cache, kv_dtype, block_tables, max_blocks_per_seq, seq_lens,
                     num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, k_scale,
                     v_scale, partition_tokens, scratch, kNoallocScratchBytes, err_flag, stream);
}
