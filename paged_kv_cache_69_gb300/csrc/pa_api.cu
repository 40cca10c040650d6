// pa_api.cu -- host side of pa_decode / pa_decode_simt: argument checks,
// launch planning (heads per CTA, pipeline depth, persistent grid), TMA
// tensor-map encoding, workspace carving and the two launches (main kernel,
// then the log-sum-exp reduce kernel with programmatic dependent launch).
// Also the status strings shared by every entry point.
#include <cuda.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "pa_common.h"
#include "pa_decode_kernel.cuh"
#include "pa_kernels.h"

namespace pa {

// ---------------------------------------------------------------------------
// status reporting
// ---------------------------------------------------------------------------
static thread_local char g_detail[256] = "";

void clear_error() { g_detail[0] = '\0'; }

pa_status fail(pa_status s, const char* what) {
    std::snprintf(g_detail, sizeof g_detail, "%s", what);
    return s;
}

pa_status fail_cuda(const char* what, cudaError_t e) {
    std::snprintf(g_detail, sizeof g_detail, "%s: %s", what, cudaGetErrorString(e));
    return PA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// device facts (cached per device)
// ---------------------------------------------------------------------------
struct DeviceInfo { int sms = 0; int max_smem = 0; };

static bool device_info(DeviceInfo& info) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].sms == 0) {
        int sms = 0, smem = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
        if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
        cache[dev].sms = sms;
        cache[dev].max_smem = smem;
    }
    info = cache[dev];
    return true;
}

// ---------------------------------------------------------------------------
// tensor-map encoding through the driver entry point
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

static CUtensorMapDataType tmap_type(pa_dtype d) {
    switch (d) {
        case PA_F32: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        case PA_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        case PA_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        default: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
    }
}

// One TMA box = `rpb` pool rows x HPC heads x the whole head_dim, placed in
// shared memory as [column block of 128 B][head][row][128 B] with the 128-B
// swizzle.  The 4-D map lists the dimensions in that shared-memory order
// (column-in-block, row, head, column block), so one copy moves the box.
// With one_plane the box holds a single column block (the tcgen05 path places
// each block separately).  Fallback: a 3-D map in the pool's natural order,
// one copy per (column block, head).
static CUresult encode_kv_map(CUtensorMap* m, const void* cache, pa_dtype kvd, int NB, int bs, int Hkv,
                              int D, int HPC, int rpb, bool per_head, bool one_plane) {
    const EncodeTiledFn enc = encode_fn();
    if (!enc) return CUDA_ERROR_NOT_FOUND;
    const int e = dtype_bytes(kvd);
    const cuuint64_t rows = static_cast<cuuint64_t>(NB) * bs;
    const cuuint32_t e128 = 128 / e;
    const cuuint32_t DH = static_cast<cuuint32_t>(D * e / 128);
    if (!per_head) {
        cuuint64_t dims[4] = {e128, rows, static_cast<cuuint64_t>(Hkv), DH};
        cuuint64_t strides[3] = {static_cast<cuuint64_t>(Hkv) * D * e, static_cast<cuuint64_t>(D) * e, 128};
        cuuint32_t box[4] = {e128, static_cast<cuuint32_t>(rpb), static_cast<cuuint32_t>(HPC), one_plane ? 1u : DH};
        cuuint32_t es[4] = {1, 1, 1, 1};
        return enc(m, tmap_type(kvd), 4, const_cast<void*>(cache), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv), rows};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * e, static_cast<cuuint64_t>(Hkv) * D * e};
    cuuint32_t box[3] = {e128, 1, static_cast<cuuint32_t>(rpb)};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, tmap_type(kvd), 3, const_cast<void*>(cache), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// ---------------------------------------------------------------------------
// launch planning
// ---------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static int cdiv_h(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Hq here counts partial rows per slot: query heads x query tokens per sequence.
static size_t workspace_bytes_for(int B, int Hq, int D, int max_seq_len, int partition_tokens, int sms) {
    const long long nr_cap = 2LL * sms;
    const long long units = partition_tokens > 0 ? static_cast<long long>(B) * cdiv_h(max_seq_len, partition_tokens)
                                                 : static_cast<long long>(B);
    const long long slots = nr_cap + units;
    return align256(sizeof(int4) * static_cast<size_t>(B)) + 256 +
           align256(sizeof(float2) * static_cast<size_t>(slots) * Hq) +
           align256(sizeof(float) * static_cast<size_t>(slots) * Hq * D);
}

static int max_slots_for(int B, int max_seq_len, int partition_tokens, int sms) {
    const long long units = partition_tokens > 0 ? static_cast<long long>(B) * cdiv_h(max_seq_len, partition_tokens)
                                                 : static_cast<long long>(B);
    return static_cast<int>(std::min<long long>(2LL * sms + units, 0x7fffffffLL));
}

// q_start == nullptr: one query per sequence (decode); otherwise sequence i
// has q_start[i+1] - q_start[i] <= QL query rows starting at row q_start[i].
static pa_status decode_impl(bool tc, void* out, const void* q, pa_dtype q_dtype, const void* k_cache,
                             const void* v_cache, pa_dtype kv_dtype, const int32_t* block_tables, int MB,
                             const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int bs, int NB,
                             float scale, float k_scale, float v_scale, int partition_tokens,
                             void* workspace, size_t workspace_bytes, int32_t* err_flag, cudaStream_t stream,
                             const int32_t* q_start = nullptr, int QL = 1, int total_q = 0) {
    const bool mq = q_start != nullptr;
    clear_error();
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || bs <= 0 || NB <= 0 || MB <= 0)
        return fail(PA_ERR_INVALID_ARG, "decode: sizes must be positive (num_seqs >= 0)");
    if (B == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens)
        return fail(PA_ERR_INVALID_ARG, "decode: null pointer");
    if (!valid_dtype(q_dtype) || !valid_dtype(kv_dtype)) return fail(PA_ERR_INVALID_ARG, "decode: unknown dtype");
    if (Hq % Hkv != 0) return fail(PA_ERR_INVALID_ARG, "decode: num_q_heads must be a multiple of num_kv_heads");
    if (D != 64 && D != 128) return fail(PA_ERR_UNSUPPORTED, "decode: head_dim must be 64 or 128");
    if (bs != 8 && bs != 16 && bs != 32 && bs != 64 && bs != 128)
        return fail(PA_ERR_UNSUPPORTED, "decode: block_size must be 8, 16, 32, 64 or 128");
    if (Hkv > 256) return fail(PA_ERR_UNSUPPORTED, "decode: num_kv_heads must be <= 256");
    if (partition_tokens < 0 || partition_tokens % 16 != 0)
        return fail(PA_ERR_INVALID_ARG, "decode: partition_tokens must be 0 or a positive multiple of 16");
    if (static_cast<long long>(NB) * bs >= (1LL << 31) || static_cast<long long>(MB) * bs >= (1LL << 30))
        return fail(PA_ERR_UNSUPPORTED, "decode: pool or table too large for 32-bit row coordinates");
    if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "decode: q, out, k_cache and v_cache must be 16-byte aligned");
    if (is_fp8(kv_dtype)) {
        if (q_dtype != PA_F16 && q_dtype != PA_BF16)
            return fail(PA_ERR_UNSUPPORTED, "decode: an fp8 cache needs f16 or bf16 queries");
        if (!(k_scale > 0.f) || !(v_scale > 0.f) || !isfinite_host(k_scale) || !isfinite_host(v_scale))
            return fail(PA_ERR_INVALID_ARG, "decode: fp8 scales must be finite and > 0");
    } else if (q_dtype != kv_dtype) {
        return fail(PA_ERR_UNSUPPORTED, "decode: q dtype must equal the cache dtype (fp8 caches excepted)");
    }
    // f32 caches: the CUDA-core kernel is the only one for that element type
    // (fp32 is no tensor-core operand type here), so pa_decode runs it.
    if (kv_dtype == PA_F32) {
        if (mq) return fail(PA_ERR_UNSUPPORTED, "attention: f32 caches take one query token per sequence (pa_decode)");
        tc = false;
    }
    if (mq && (!tc || QL < 1 || total_q < 0 || static_cast<long long>(QL) * (Hq / Hkv) > 128))
        return fail(PA_ERR_UNSUPPORTED,
                    "attention: several query tokens need the tensor-core path and max_q_len * G <= 128");
    // fp8 caches on the tensor-core path run the native-e4m3 kernel (32-token
    // chunks, GQA groups of up to 8 heads, partitions a multiple of 32
    // tokens); other fp8 shapes convert e4m3 to f16 in registers.
    const bool native8 = !mq && tc && is_fp8(kv_dtype) && D == 128 && Hq / Hkv <= 8 &&
                         partition_tokens % 32 == 0;
    const bool fp8t = native8 && Hq / Hkv <= 4;      // keys as the MMA rows: half the MMAs
    // Several query tokens with 48-128 (token, head) rows per KV head on a
    // 16-bit cache: the tcgen05 kernel.  The rows of UH KV heads, each
    // head's padded to a multiple of 32, fill a 128-row tile with the
    // accumulators in tensor memory; a chunk is 32 tokens of its one or two
    // heads (16-32 KB of K and V per pipeline stage).
    const int um_rows = 32 * cdiv_h(static_cast<long long>(QL) * (Hq / Hkv), 32);
    int UH = 0;
    for (int h = std::min(4, 128 / std::max(1, um_rows)); h >= 1; --h)
        if (Hkv % h == 0) { UH = h; break; }
    const int um_ct = 32;
    // From 48 rows up: with fewer, the per-row softmax of a 16- or 32-token
    // chunk leaves most of the tile idle and the mma.sync kernel is faster.
    const bool um = mq && !is_fp8(kv_dtype) && QL * (Hq / Hkv) >= 48 && um_rows <= 128 && UH > 0 &&
                    partition_tokens % um_ct == 0;
    const int CT = um ? um_ct : native8 ? 32 : 16;
    const void* kern = um      ? decode_kernel_mq_um(kv_dtype, q_dtype, D, CT)
                       : mq    ? decode_kernel_mq(kv_dtype, q_dtype, D)
                       : fp8t  ? decode_kernel_fp8t(kv_dtype, q_dtype, D)
                       : native8 ? decode_kernel_e4m3(kv_dtype, q_dtype, D)
                       : tc    ? decode_kernel_tc(kv_dtype, q_dtype, D)
                               : decode_kernel_simt(kv_dtype, q_dtype, D);
    if (!kern) return fail(PA_ERR_UNSUPPORTED, "decode: no kernel for this dtype / head_dim combination");
    const bool split_heads = partition_tokens > 0;
    const void* rkern = reduce_kernel(q_dtype, D, split_heads);
    if (!rkern) return fail(PA_ERR_UNSUPPORTED, "decode: no reduce kernel for this output dtype");
    DeviceInfo dev;
    if (!device_info(dev)) return fail(PA_ERR_CUDA, "decode: cannot query the current device");

    const int G = Hq / Hkv;
    const int e = dtype_bytes(kv_dtype);
    const int eq = dtype_bytes(q_dtype);
    const int MT = cdiv_h(static_cast<long long>(QL) * G, 16);   // 16-row tiles of (query token, head) rows
    if (MT > 8) return fail(PA_ERR_UNSUPPORTED, "decode: more than 128 query rows per KV head");
    int HPC = 0;
    // several query tokens: at most 4 consumer warps per CTA when the rows
    // take more than one tile, so that two CTAs share an SM
    const int max_warps = (mq && MT > 1) ? 4 : 8;
    // At most 16 KB of keys per stage (HPC heads x one chunk): smaller
    // stages give two CTAs per SM three stages each, 192 KB of K/V in flight
    // per SM, which streamed 6-8% faster than one CTA with two 64 KB stages.
    for (int h = Hkv; h >= 1; --h) {
        if (Hkv % h) continue;
        if (h * MT > std::max(max_warps, MT)) continue;
        if (static_cast<long long>(CT) * h * D * e > 16 * 1024) continue;
        HPC = h;
        break;
    }
    if (um) HPC = UH;                // the KV heads whose row blocks fill the tile
    if (HPC == 0) return fail(PA_ERR_UNSUPPORTED, "decode: no head grouping fits one CTA");
    const int NHG = Hkv / HPC;
    // tcgen05 path: 4 consumer warps (one tile row per thread), the producer
    // warp and the MMA warp
    const int NCW = um ? 4 : HPC * MT;
    const int rpb = std::min(CT, bs);
    const int DH = D * e / 128;
    if (DH < 1 || (D * e) % 128 != 0) return fail(PA_ERR_UNSUPPORTED, "decode: head_dim * elem bytes must be a multiple of 128");

    DecodeParams p{};
    p.out = out; p.q = q; p.block_tables = block_tables; p.seq_lens = seq_lens; p.err_flag = err_flag;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.G = G; p.D = D; p.bs = bs; p.NB = NB; p.MB = MB;
    p.out_bytes = eq;
    p.HPC = HPC; p.NHG = NHG; p.MT = MT; p.NCW = NCW;
    p.ct = CT;
    p.PC = partition_tokens / CT;
    p.q_start = q_start;
    p.QL = QL;
    p.total_q = mq ? total_q : B;
    // Schedule weights: a unit start (query rows loaded, result written)
    // is charged 3/4 of a chunk, which balanced CTA finish times best on
    // length mixes with many short sequences.
    p.WQ = 4;
    p.WS = 3;
    p.rpb = rpb;
    p.box_bytes = static_cast<uint32_t>(rpb * HPC * DH * 128);
    p.kv_bytes = static_cast<uint32_t>(CT * HPC * D * e);
    p.q_bytes = static_cast<uint32_t>(QL * HPC * G * D * eq);
    p.q_slot_bytes = (p.q_bytes + 1023u) & ~1023u;   // swizzled tensor copies need 1024-B alignment
    if (um) {
        // a column plane holds the 128 tile rows (head hl's query rows at row
        // um_rows * hl); the rows between the heads' blocks are never written
        // and reach only tile rows nobody reads
        p.um_rows = um_rows;
        p.q_plane_bytes = 128u * 128u;
        p.q_slot_bytes = static_cast<uint32_t>(DH) * p.q_plane_bytes;
    }
    p.stage_bytes = 2 * p.kv_bytes;
    // CUDA-core variant: private fp32 query rows; transposed fp8: P bytes per warp
    // tcgen05 path: two P buffers of 128 rows x CT tokens per head
    const uint32_t simtq = um ? 2u * static_cast<uint32_t>(HPC) * 128u * static_cast<uint32_t>(CT) * 2u
                         : fp8t ? static_cast<uint32_t>(NCW * 256) : tc ? 0u : static_cast<uint32_t>(NCW * 16 * D * 4);
    const uint32_t extras = 1024;   // barriers, stage descriptors, prologue scratch
    const uint32_t fixed = nq_slots(um) * p.q_slot_bytes + simtq + extras + 1024;   // + base alignment slack
    const int threads = (NCW + (um ? 2 : 1)) * 32;
    // Two co-resident CTAs per SM double the consumer warps that hide the
    // per-chunk MMA/softmax latency; use them when registers and shared
    // memory allow at least 3 stages each, else one CTA with a deeper ring.
    cudaFuncAttributes fa{};
    cudaError_t ce = cudaFuncGetAttributes(&fa, kern);
    if (ce != cudaSuccess) return fail_cuda("decode: kernel attributes", ce);
    const int regs = (fa.numRegs + 7) & ~7;
    const int by_regs = std::max(1, 65536 / std::max(1, regs * threads));
    const long long sm_smem = std::min(dev.max_smem, 227 * 1024) + 1024LL;   // per-SM budget incl. reservation
    int stages = 0;
    // tcgen05 kernels run one CTA per SM (their tensor-memory allocation
    // limits residency): size the ring for one CTA
    if (by_regs >= 2 && !um) {
        const long long per_cta = sm_smem / 2 - 1024 - fixed;
        const int s2 = static_cast<int>(std::min<long long>(MAX_STAGES, per_cta / p.stage_bytes));
        // the multi-token query ring takes more shared memory: two stages
        // per CTA still keep four in flight per SM
        if (s2 >= (mq ? 2 : 3)) stages = s2;
    }
    if (stages == 0) {
        const long long per_cta = std::min(dev.max_smem, 227 * 1024) - static_cast<long long>(fixed);
        stages = static_cast<int>(std::min<long long>(MAX_STAGES, per_cta / p.stage_bytes));
        // roughly 192 KB of K/V in flight per CTA
        const int want = cdiv_h(192 * 1024, p.stage_bytes);
        stages = std::min(stages, std::max(2, want));
    }
    if (stages < 2) return fail(PA_ERR_UNSUPPORTED, "decode: pipeline stages do not fit in shared memory");
    p.stages = stages;
    p.q_off = stages * p.stage_bytes;
    p.simtq_off = p.q_off + nq_slots(um) * p.q_slot_bytes;
    p.bar_off = (p.simtq_off + simtq + 15u) & ~15u;
    const size_t smem = 1024 + p.bar_off + extras;
    const float log2e = 1.4426950408889634f;
    p.qk_scale = scale * log2e * (is_fp8(kv_dtype) ? k_scale : 1.f);
    p.v_scale = is_fp8(kv_dtype) ? v_scale : 1.f;

    // workspace
    const int prow = QL * Hq;                         // partial rows per slot
    const size_t need = workspace_bytes_for(B, prow, D, MB * bs, partition_tokens, dev.sms);
    if (!workspace) return fail(PA_ERR_WORKSPACE, "decode: workspace pointer is null");
    if (workspace_bytes < need) return fail(PA_ERR_WORKSPACE, "decode: workspace smaller than pa_decode_workspace_size()");
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(PA_ERR_WORKSPACE, "decode: workspace must be 256-byte aligned");
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.split_list = reinterpret_cast<int4*>(ws); ws += align256(sizeof(int4) * static_cast<size_t>(B));
    p.totals = reinterpret_cast<int*>(ws); ws += 256;
    p.max_slots = max_slots_for(B, MB * bs, partition_tokens, dev.sms);
    p.part_ml = reinterpret_cast<float2*>(ws); ws += align256(sizeof(float2) * static_cast<size_t>(p.max_slots) * prow);
    p.part_acc = reinterpret_cast<float*>(ws);

    // tensor maps
    alignas(64) CUtensorMap tk, tv;
    p.per_head_copies = 0;
    CUresult r1 = encode_kv_map(&tk, k_cache, kv_dtype, NB, bs, Hkv, D, HPC, rpb, false, um);
    CUresult r2 = r1 == CUDA_SUCCESS ? encode_kv_map(&tv, v_cache, kv_dtype, NB, bs, Hkv, D, HPC, rpb, false, um) : r1;
    if (r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS) {
        p.per_head_copies = 1;
        r1 = encode_kv_map(&tk, k_cache, kv_dtype, NB, bs, Hkv, D, HPC, rpb, true, um);
        r2 = r1 == CUDA_SUCCESS ? encode_kv_map(&tv, v_cache, kv_dtype, NB, bs, Hkv, D, HPC, rpb, true, um) : r1;
        if (r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS) {
            char msg[96];
            std::snprintf(msg, sizeof msg, "decode: cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r1 ? r1 : r2));
            return fail(PA_ERR_CUDA, msg);
        }
    }

    // query rows: a 128-B-swizzled tensor copy [column block][row][128 B] of
    // the CTA's HPC*G rows, so the MMA fragment loads are bank-conflict free
    alignas(64) CUtensorMap tq;
    std::memset(&tq, 0, sizeof tq);
    p.q_tma = 0;
    if (mq) {
        // [column block][token][head][128 B]: QL tokens x HPC*G heads per copy
        const EncodeTiledFn enc = encode_fn();
        const cuuint32_t e128q = static_cast<cuuint32_t>(128 / eq);
        const cuuint32_t dhq = static_cast<cuuint32_t>(D * eq / 128);
        cuuint64_t dims[4] = {e128q, static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(std::max(total_q, 1)), dhq};
        cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * eq, static_cast<cuuint64_t>(Hq) * D * eq, 128};
        // tcgen05 path: one KV head's rows and one column plane per copy
        cuuint32_t box[4] = {e128q, static_cast<cuuint32_t>(um ? G : HPC * G), static_cast<cuuint32_t>(QL),
                             um ? 1u : dhq};
        cuuint32_t es[4] = {1, 1, 1, 1};
        if (!enc || HPC * G > 256 || QL > 256 ||
            enc(&tq, tmap_type(q_dtype), 4, const_cast<void*>(q), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return fail(PA_ERR_CUDA, "attention: query tensor map could not be encoded");
        p.q_tma = 1;
    } else if (tc) {
        const EncodeTiledFn enc = encode_fn();
        const cuuint32_t e128q = static_cast<cuuint32_t>(128 / eq);
        const cuuint32_t dhq = static_cast<cuuint32_t>(D * eq / 128);
        cuuint64_t dims[3] = {e128q, static_cast<cuuint64_t>(B) * Hq, dhq};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * eq, 128};
        cuuint32_t box[3] = {e128q, static_cast<cuuint32_t>(HPC * G), dhq};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc && HPC * G <= 256 &&
            enc(&tq, tmap_type(q_dtype), 3, const_cast<void*>(q), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
            p.q_tma = 1;
    }

    // grid: persistent CTAs, as many as fit, split into ranges x head groups
    ce = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (ce != cudaSuccess) return fail_cuda("decode: set shared memory size", ce);
    int per_sm = 0;
    ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (ce != cudaSuccess) return fail_cuda("decode: occupancy query", ce);
    per_sm = std::max(1, per_sm);
    const long long chunk_bound = static_cast<long long>(B) * cdiv_h(static_cast<long long>(MB) * bs, CT);
    long long NR = std::max(1LL, static_cast<long long>(per_sm) * dev.sms / NHG);
    NR = std::min(NR, 2LL * dev.sms);   // the workspace holds 2 x SMs ranges
    NR = std::min(NR, chunk_bound);
    p.NR = static_cast<int>(NR);

    // Both launches are programmatic dependents of the work before them on
    // the stream; each kernel waits (griddepcontrol.wait) for that work to
    // complete before it reads anything, so only the launch overlaps.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(NR * NHG));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&p, &tk, &tv, &tq};
    ce = cudaLaunchKernelExC(&cfg, kern, args);
    if (ce != cudaSuccess) return fail_cuda("decode: main kernel launch", ce);

    cudaLaunchConfig_t rcfg{};
    const int red_block = red_threads(split_heads ? RED_SPLIT_WARPS : 1);
    {
        // persistent reduce grid: one wave of CTAs striding over the
        // (split sequence, head group) items
        int red_per_sm = 0;
        ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&red_per_sm, rkern, red_block, 0);
        if (ce != cudaSuccess) return fail_cuda("decode: reduce occupancy query", ce);
        const long long items = static_cast<long long>(QL) *
                                (split_heads ? static_cast<long long>(B) * Hq
                                             : static_cast<long long>(B) * ((Hq + RED_THREADS / 32 - 1) / (RED_THREADS / 32)));
        const long long g = std::max(1LL, std::min(items, static_cast<long long>(std::max(1, red_per_sm)) * dev.sms));
        rcfg.gridDim = dim3(static_cast<unsigned>(g));
    }
    rcfg.blockDim = dim3(static_cast<unsigned>(red_block));
    rcfg.dynamicSmemBytes = 0;
    rcfg.stream = stream;
    rcfg.attrs = attr;
    rcfg.numAttrs = 1;
    void* rargs[] = {&p};
    ce = cudaLaunchKernelExC(&rcfg, rkern, rargs);
    if (ce != cudaSuccess) return fail_cuda("decode: reduce kernel launch", ce);
    return PA_OK;
}

}  // namespace pa

using namespace pa;

extern "C" const char* pa_status_string(pa_status s) {
    switch (s) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        default: return "PA_ERR_UNKNOWN";
    }
}

extern "C" const char* pa_last_error_detail(void) { return g_detail; }

extern "C" size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int max_seq_len, int head_dim,
                                           int partition_tokens) {
    if (num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0 || max_seq_len < 0 || partition_tokens < 0)
        return 0;
    DeviceInfo dev;
    if (!device_info(dev)) return 0;
    return workspace_bytes_for(num_seqs, num_q_heads, head_dim, max_seq_len, partition_tokens, dev.sms);
}

extern "C" pa_status pa_decode(void* out, const void* q, pa_dtype q_dtype, const void* k_cache,
                               const void* v_cache, pa_dtype kv_dtype, const int32_t* block_tables,
                               int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                               int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                               int num_blocks, float scale, float k_scale, float v_scale,
                               int partition_tokens, void* workspace, size_t workspace_bytes,
                               int32_t* err_flag, cudaStream_t stream) {
    return decode_impl(true, out, q, q_dtype, k_cache, v_cache, kv_dtype, block_tables, max_blocks_per_seq,
                       seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                       k_scale, v_scale, partition_tokens, workspace, workspace_bytes, err_flag, stream);
}

extern "C" pa_status pa_decode_simt(void* out, const void* q, pa_dtype q_dtype, const void* k_cache,
                                    const void* v_cache, pa_dtype kv_dtype, const int32_t* block_tables,
                                    int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                                    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, float scale, float k_scale, float v_scale,
                                    int partition_tokens, void* workspace, size_t workspace_bytes,
                                    int32_t* err_flag, cudaStream_t stream) {
    return decode_impl(false, out, q, q_dtype, k_cache, v_cache, kv_dtype, block_tables, max_blocks_per_seq,
                       seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                       k_scale, v_scale, partition_tokens, workspace, workspace_bytes, err_flag, stream);
}

extern "C" size_t pa_attention_workspace_size(int num_seqs, int max_q_len, int num_q_heads, int max_seq_len,
                                              int head_dim, int partition_tokens) {
    if (num_seqs < 0 || max_q_len <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_seq_len < 0 ||
        partition_tokens < 0)
        return 0;
    DeviceInfo dev;
    if (!device_info(dev)) return 0;
    return workspace_bytes_for(num_seqs, max_q_len * num_q_heads, head_dim, max_seq_len, partition_tokens, dev.sms);
}

extern "C" pa_status pa_attention(void* out, const void* q, pa_dtype q_dtype, const void* k_cache,
                                  const void* v_cache, pa_dtype kv_dtype, const int32_t* block_tables,
                                  int max_blocks_per_seq, const int32_t* seq_lens, const int32_t* q_start,
                                  int num_seqs, int total_q, int max_q_len, int num_q_heads, int num_kv_heads,
                                  int head_dim, int block_size, int num_blocks, float scale, float k_scale,
                                  float v_scale, int partition_tokens, void* workspace, size_t workspace_bytes,
                                  int32_t* err_flag, cudaStream_t stream) {
    clear_error();
    if (!q_start) return fail(PA_ERR_INVALID_ARG, "attention: q_start is null");
    if (max_q_len < 1 || total_q < 0) return fail(PA_ERR_INVALID_ARG, "attention: max_q_len must be >= 1");
    if (num_seqs > 0 && total_q == 0) return PA_OK;
    return decode_impl(true, out, q, q_dtype, k_cache, v_cache, kv_dtype, block_tables, max_blocks_per_seq,
                       seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                       k_scale, v_scale, partition_tokens, workspace, workspace_bytes, err_flag, stream,
                       q_start, max_q_len, total_q);
}
