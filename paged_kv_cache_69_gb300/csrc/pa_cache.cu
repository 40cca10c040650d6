// pa_cache.cu -- pa_reshape_and_cache and pa_copy_blocks.
//
// reshape_and_cache: token t's K and V rows go to pool slot slot_mapping[t]
// ("vLLM intro part 2", section 3.2; "kv-cache-memory-core", section 3:
// decode appends one slot per step, prefill writes whole blocks).  A token's
// [num_kv_heads, head_dim] row is contiguous in both the source and the
// pool, so one warp moves one token with 16-byte vector accesses.  fp8 pools
// quantise on write ("kv-cache-memory-core", section 4.4): the source value
// widened to float, divided by the per-tensor scale (IEEE division), then
// CUDA's saturating round-to-nearest-even E4M3 conversion.
//
// copy_blocks: copy-on-write copies of whole blocks ("vLLM intro part 2",
// section 5), for one layer's pools or for all layers in one launch; swap:
// the same block copy between a device pool and a host pool (preemption by
// swapping a request's blocks out to CPU memory and back,
// "kv-cache-memory-core", section on preemption).  16-byte vector copies.
#include <cstdint>
#include <cstdio>

#include "pa_common.h"
#include "pa_device.cuh"

namespace pa {

constexpr int VEC = 8;   // elements per lane per step

template <class S, class Dt>
struct Conv;

// same type: move bits
template <class X>
struct Conv<X, X> {
    static __device__ __forceinline__ void run(const uint8_t* src, uint8_t* dst, float) {
        if constexpr (X::bytes == 4) {
            reinterpret_cast<uint4*>(dst)[0] = reinterpret_cast<const uint4*>(src)[0];
            reinterpret_cast<uint4*>(dst)[1] = reinterpret_cast<const uint4*>(src)[1];
        } else if constexpr (X::bytes == 2) {
            reinterpret_cast<uint4*>(dst)[0] = reinterpret_cast<const uint4*>(src)[0];
        } else {
            reinterpret_cast<uint2*>(dst)[0] = reinterpret_cast<const uint2*>(src)[0];
        }
    }
};

// any float source -> e4m3 or e5m2
template <class S, class F8>
struct ConvFp8 {
    static __device__ __forceinline__ void run(const uint8_t* src, uint8_t* dst, float scale) {
        float x[VEC];
        if constexpr (S::code == PA_F32) {
            const float4 a = reinterpret_cast<const float4*>(src)[0];
            const float4 b = reinterpret_cast<const float4*>(src)[1];
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
        } else {
            const uint4 r = reinterpret_cast<const uint4*>(src)[0];
            const typename S::T* e = reinterpret_cast<const typename S::T*>(&r);
#pragma unroll
            for (int k = 0; k < VEC; ++k) x[k] = to_float(e[k]);
        }
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int k = 0; k < VEC; ++k) {
            const uint32_t b = static_cast<uint32_t>(__nv_cvt_float_to_fp8(
                __fdiv_rn(x[k], scale), __NV_SATFINITE, F8::code == PA_FP8_E5M2 ? __NV_E5M2 : __NV_E4M3));
            if (k < 4) lo |= b << (8 * k); else hi |= b << (8 * (k - 4));
        }
        reinterpret_cast<uint2*>(dst)[0] = make_uint2(lo, hi);
    }
};

template <class S> struct Conv<S, FP8T> : ConvFp8<S, FP8T> {};
template <class S> struct Conv<S, E5M2T> : ConvFp8<S, E5M2T> {};

// an already-quantised source: move bytes
template <> struct Conv<FP8T, FP8T> {
    static __device__ __forceinline__ void run(const uint8_t* src, uint8_t* dst, float) {
        reinterpret_cast<uint2*>(dst)[0] = reinterpret_cast<const uint2*>(src)[0];
    }
};
template <> struct Conv<E5M2T, E5M2T> {
    static __device__ __forceinline__ void run(const uint8_t* src, uint8_t* dst, float) {
        reinterpret_cast<uint2*>(dst)[0] = reinterpret_cast<const uint2*>(src)[0];
    }
};

template <class S, class Dt>
__global__ void __launch_bounds__(256)
reshape_and_cache_kernel(uint8_t* __restrict__ kc, uint8_t* __restrict__ vc,
                         const uint8_t* __restrict__ key, const uint8_t* __restrict__ value,
                         const int64_t* __restrict__ slots, int T, int row_elems, int block_size,
                         int64_t nslots, float k_scale, float v_scale, int32_t* err) {
    // a decode launched next may become resident now (it waits for this
    // grid to complete before it reads anything)
    grid_dependents_launch();
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const int64_t slot = slots[t];
    if (slot < 0) return;
    if (slot >= nslots) {
        if (lane == 0) raise_flag(err, PA_ERRBIT_BAD_SLOT);
        return;
    }
    // slot = block * block_size + offset; rows of the pool are ordered the same way
    const size_t drow = static_cast<size_t>(slot) * row_elems;
    const size_t srow = static_cast<size_t>(t) * row_elems;
    for (int e = lane * VEC; e < row_elems; e += 32 * VEC) {
        Conv<S, Dt>::run(key + (srow + e) * S::bytes, kc + (drow + e) * Dt::bytes, k_scale);
        Conv<S, Dt>::run(value + (srow + e) * S::bytes, vc + (drow + e) * Dt::bytes, v_scale);
    }
}

// Whole-block copies between two pools of the same shape, for every layer
// and both K and V: copy-on-write inside one pool (source pool = destination
// pool) and swapping blocks between a device pool and a host pool the
// device can address.  One CTA per (pair, layer, K|V).
constexpr int MAX_LAYERS = 256;
struct BlockCopyArgs {
    uint8_t* dst[2][MAX_LAYERS];           // [K|V][layer]
    const uint8_t* src[2][MAX_LAYERS];
    const int64_t* pairs;                  // (src block, dst block) per pair
    int64_t block_bytes;
    int src_blocks, dst_blocks;
    int32_t* err;
};

__global__ void __launch_bounds__(256)
block_copy_kernel(const __grid_constant__ BlockCopyArgs a) {
    grid_dependents_launch();
    const int p = blockIdx.x, l = blockIdx.y, kv = blockIdx.z;
    const int64_t src = a.pairs[2 * static_cast<int64_t>(p)], dst = a.pairs[2 * static_cast<int64_t>(p) + 1];
    if (src < 0 || src >= a.src_blocks || dst < 0 || dst >= a.dst_blocks) {
        if (threadIdx.x == 0 && l == 0 && kv == 0) raise_flag(a.err, PA_ERRBIT_BAD_PAIR);
        return;
    }
    const uint4* s = reinterpret_cast<const uint4*>(a.src[kv][l] + src * a.block_bytes);
    uint4* d = reinterpret_cast<uint4*>(a.dst[kv][l] + dst * a.block_bytes);
    const int64_t n = a.block_bytes / 16;
    // Up to U vectors per thread are loaded before any is stored: the
    // compiler cannot prove source and destination blocks apart, and would
    // otherwise wait for each load before the next.
    constexpr int U = 8;
    for (int64_t k0 = threadIdx.x; k0 < n; k0 += static_cast<int64_t>(U) * blockDim.x) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = k0 + static_cast<int64_t>(u) * blockDim.x;
            if (k < n) r[u] = s[k];
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = k0 + static_cast<int64_t>(u) * blockDim.x;
            if (k < n) d[k] = r[u];
        }
    }
}

// Validates and launches a block copy over num_layers pools.
static pa_status launch_block_copy(const char* who, void* const* dst_k, void* const* dst_v,
                                   const void* const* src_k, const void* const* src_v, int num_layers,
                                   pa_dtype kv_dtype, const int64_t* pairs, int num_pairs, int num_kv_heads,
                                   int head_dim, int block_size, int src_blocks, int dst_blocks,
                                   int32_t* err_flag, cudaStream_t stream) {
    char msg[128];
    auto bad = [&](pa_status st, const char* what) {
        std::snprintf(msg, sizeof msg, "%s: %s", who, what);
        return fail(st, msg);
    };
    if (num_pairs < 0 || num_layers <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        src_blocks <= 0 || dst_blocks <= 0)
        return bad(PA_ERR_INVALID_ARG, "sizes must be positive (num_pairs >= 0)");
    if (num_layers > MAX_LAYERS) return bad(PA_ERR_UNSUPPORTED, "more than 256 layers");
    if (!valid_dtype(kv_dtype)) return bad(PA_ERR_INVALID_ARG, "unknown dtype");
    if (num_pairs == 0) return PA_OK;
    if (!pairs || !dst_k || !dst_v || !src_k || !src_v) return bad(PA_ERR_INVALID_ARG, "null pointer");
    const int64_t block_bytes = static_cast<int64_t>(block_size) * num_kv_heads * head_dim * dtype_bytes(kv_dtype);
    if (block_bytes % 16 != 0) return bad(PA_ERR_UNSUPPORTED, "block bytes must be a multiple of 16");
    BlockCopyArgs a{};
    for (int l = 0; l < num_layers; ++l) {
        if (!dst_k[l] || !dst_v[l] || !src_k[l] || !src_v[l]) return bad(PA_ERR_INVALID_ARG, "null pool pointer");
        if (!aligned16(dst_k[l]) || !aligned16(dst_v[l]) || !aligned16(src_k[l]) || !aligned16(src_v[l]))
            return bad(PA_ERR_INVALID_ARG, "pools must be 16-byte aligned");
        a.dst[0][l] = static_cast<uint8_t*>(dst_k[l]);
        a.dst[1][l] = static_cast<uint8_t*>(dst_v[l]);
        a.src[0][l] = static_cast<const uint8_t*>(src_k[l]);
        a.src[1][l] = static_cast<const uint8_t*>(src_v[l]);
    }
    a.pairs = pairs;
    a.block_bytes = block_bytes;
    a.src_blocks = src_blocks;
    a.dst_blocks = dst_blocks;
    a.err = err_flag;
    dim3 grid(static_cast<unsigned>(num_pairs), static_cast<unsigned>(num_layers), 2);
    block_copy_kernel<<<grid, 256, 0, stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        std::snprintf(msg, sizeof msg, "%s launch", who);
        return fail_cuda(msg, e);
    }
    return PA_OK;
}

template <class S, class Dt>
static cudaError_t launch_rc(void* kc, void* vc, const void* key, const void* value, const int64_t* slots,
                             int T, int row_elems, int bs, int64_t nslots, float ks, float vs,
                             int32_t* err, cudaStream_t stream) {
    const int warps = 8;
    const unsigned grid = static_cast<unsigned>((static_cast<int64_t>(T) + warps - 1) / warps);
    reshape_and_cache_kernel<S, Dt><<<grid, warps * 32, 0, stream>>>(
        static_cast<uint8_t*>(kc), static_cast<uint8_t*>(vc), static_cast<const uint8_t*>(key),
        static_cast<const uint8_t*>(value), slots, T, row_elems, bs, nslots, ks, vs, err);
    return cudaGetLastError();
}

}  // namespace pa

using namespace pa;

extern "C" pa_status pa_reshape_and_cache(void* k_cache, void* v_cache, pa_dtype kv_dtype,
                                          const void* key, const void* value, pa_dtype src_dtype,
                                          const int64_t* slot_mapping, int num_tokens,
                                          int num_kv_heads, int head_dim, int block_size,
                                          int num_blocks, float k_scale, float v_scale,
                                          int32_t* err_flag, cudaStream_t stream) {
    clear_error();
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARG, "reshape_and_cache: sizes must be positive (num_tokens >= 0)");
    if (num_tokens == 0) return PA_OK;
    if (!k_cache || !v_cache || !key || !value || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "reshape_and_cache: null pointer");
    if (!valid_dtype(kv_dtype) || !valid_dtype(src_dtype))
        return fail(PA_ERR_INVALID_ARG, "reshape_and_cache: unknown dtype");
    const int64_t row_elems = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (row_elems % VEC != 0 || row_elems > (1 << 30))
        return fail(PA_ERR_UNSUPPORTED, "reshape_and_cache: num_kv_heads*head_dim must be a multiple of 8");
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(key) || !aligned16(value))
        return fail(PA_ERR_INVALID_ARG, "reshape_and_cache: caches and sources must be 16-byte aligned");
    const int64_t nslots = static_cast<int64_t>(num_blocks) * block_size;
    cudaError_t e;
    const int re = static_cast<int>(row_elems);
    if (kv_dtype == PA_FP8_E5M2) {
        if (!(k_scale > 0.f) || !(v_scale > 0.f) || !isfinite_host(k_scale) || !isfinite_host(v_scale))
            return fail(PA_ERR_INVALID_ARG, "reshape_and_cache: fp8 scales must be finite and > 0");
        switch (src_dtype) {
            case PA_F32: e = launch_rc<F32T, E5M2T>(k_cache, v_cache, key, value, slot_mapping, num_tokens, re, block_size, nslots, k_scale, v_scale, err_flag, stream); break;
            case PA_F16: e = launch_rc<F16T, E5M2T>(k_cache, v_cache, key, value, slot_mapping, num_tokens, re, block_size, nslots, k_scale, v_scale, err_flag, stream); break;
            case PA_BF16: e = launch_rc<BF16T, E5M2T>(k_cache, v_cache, key, value, slot_mapping, num_tokens, re, block_size, nslots, k_scale, v_scale, err_flag, stream); break;
            case PA_FP8_E5M2: e = launch_rc<E5M2T, E5M2T>(k_cache, v_cache, key, value, slot_mapping, num_tokens, re, block_size, nslots, 1.f, 1.f, err_flag, stream); break;
            default: return fail(PA_ERR_UNSUPPORTED, "reshape_and_cache: e5m2 cache needs an f32, f16, bf16 or e5m2 source");
        }
    } else if (kv_dtype == PA_FP8_E4M3) {
        if (!(k_scale > 0.f) || !(v_scale > 0.f) || !isfinite_host(k_scale) || !isfinite_host(v_scale))
            return fail(PA_ERR_INVALID_ARG, "reshape_and_cache: fp8 scales must be finite and > 0");
        switch (src_dtype) {
            case PA_F32: e = launch_rc<F32T, FP8T>(k_cache, v_cache, key, value, slot_mapping, num_tokens, re, block_size, nslots, k_scale, v_scale, err_flag, stream); break;
            case PA_F16: e = launch_rc<F16T, FP8T>(k_cache, v_cache, key, value, slot_mapping, num_tokens, re, block_size, nslots, k_scale, v_scale, err_flag, stream); break;
            case PA_BF16: e = launch_rc<BF16T, FP8T>(k_cache, v_cache, key, value, slot_mapping, num_tokens, re, block_size, nslots, k_scale, v_scale, err_flag, stream); break;
            case PA_FP8_E4M3: e = launch_rc<FP8T, FP8T>(k_cache, v_cache, key, value, slot_mapping, num_tokens, re, block_size, nslots, 1.f, 1.f, err_flag, stream); break;
            default: return fail(PA_ERR_UNSUPPORTED, "reshape_and_cache: fp8 cache needs an f32, f16 or bf16 source");
        }
    } else {
        if (src_dtype != kv_dtype)
            return fail(PA_ERR_UNSUPPORTED, "reshape_and_cache: source dtype must equal cache dtype");
        switch (kv_dtype) {
            case PA_F32: e = launch_rc<F32T, F32T>(k_cache, v_cache, key, value, slot_mapping, num_tokens, re, block_size, nslots, 1.f, 1.f, err_flag, stream); break;
            case PA_F16: e = launch_rc<F16T, F16T>(k_cache, v_cache, key, value, slot_mapping, num_tokens, re, block_size, nslots, 1.f, 1.f, err_flag, stream); break;
            default: e = launch_rc<BF16T, BF16T>(k_cache, v_cache, key, value, slot_mapping, num_tokens, re, block_size, nslots, 1.f, 1.f, err_flag, stream); break;
        }
    }
    return e == cudaSuccess ? PA_OK : fail_cuda("reshape_and_cache launch", e);
}

extern "C" pa_status pa_copy_blocks(void* k_cache, void* v_cache, pa_dtype kv_dtype,
                                    const int64_t* block_mapping, int num_pairs,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, int32_t* err_flag, cudaStream_t stream) {
    clear_error();
    void* k[1] = {k_cache};
    void* v[1] = {v_cache};
    const void* ks[1] = {k_cache};
    const void* vs[1] = {v_cache};
    if (num_pairs > 0 && (!k_cache || !v_cache || !block_mapping))
        return fail(PA_ERR_INVALID_ARG, "copy_blocks: null pointer");
    return launch_block_copy("copy_blocks", k, v, ks, vs, 1, kv_dtype, block_mapping, num_pairs, num_kv_heads,
                             head_dim, block_size, num_blocks, num_blocks, err_flag, stream);
}

extern "C" pa_status pa_copy_blocks_layers(void* const* k_caches, void* const* v_caches, int num_layers,
                                           pa_dtype kv_dtype, const int64_t* block_mapping, int num_pairs,
                                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                           int32_t* err_flag, cudaStream_t stream) {
    clear_error();
    return launch_block_copy("copy_blocks_layers", k_caches, v_caches,
                             reinterpret_cast<const void* const*>(k_caches),
                             reinterpret_cast<const void* const*>(v_caches), num_layers, kv_dtype,
                             block_mapping, num_pairs, num_kv_heads, head_dim, block_size, num_blocks,
                             num_blocks, err_flag, stream);
}

extern "C" pa_status pa_swap_blocks(void* dst_k, void* dst_v, int dst_num_blocks, const void* src_k,
                                    const void* src_v, int src_num_blocks, pa_dtype kv_dtype,
                                    const int64_t* block_mapping, int num_pairs, int num_kv_heads,
                                    int head_dim, int block_size, int32_t* err_flag, cudaStream_t stream) {
    clear_error();
    void* dk[1] = {dst_k};
    void* dv[1] = {dst_v};
    const void* sk[1] = {src_k};
    const void* sv[1] = {src_v};
    return launch_block_copy("swap_blocks", dk, dv, sk, sv, 1, kv_dtype, block_mapping, num_pairs, num_kv_heads,
                             head_dim, block_size, src_num_blocks, dst_num_blocks, err_flag, stream);
}
