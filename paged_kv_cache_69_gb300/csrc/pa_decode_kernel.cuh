// pa_decode_kernel.cuh -- paged decode attention: device code.
//
// What is computed (for every sequence i and query head h, g = h / G):
//   s_t = scale * <q_h, K_t>, p = softmax(s), out_h = sum_t p_t V_t, t < L_i,
// with K_t / V_t read through the block table ("vLLM intro part 2",
// section 4; the PagedAttention note's three kernel steps: look up the block
// table, load block by block, merge across blocks with online softmax).
//
// How (GB300 design):
//  * Work unit = a 16-token chunk (32 on the fp8 and tcgen05 paths) of one
//    sequence for HPC KV heads.  The chunks of all sequences form one stream
//    that is cut into NR ranges of equal cost (a chunk weighs WQ, a segment
//    start WS more), one per persistent CTA (times NHG head groups), so every
//    CTA does the same work whatever the length mix.
//  * One producer warp per CTA walks its range, prefetches block-table
//    entries 32 at a time into registers, and issues TMA tile loads of the
//    K and V rows of each chunk (all HPC heads of a block in one copy, 128-B
//    swizzled in shared memory) plus a copy of the query rows when it starts
//    a sequence (at every segment start on the tcgen05 path), into a ring of
//    stages guarded by full/empty mbarriers.
//  * Consumer warps, one per (KV head, 16-row query tile), keep the GQA
//    group's query heads packed as the M dimension of mma.sync m16n8k16
//    (tensor-core variant) or as register rows (CUDA-core variant) and run
//    online softmax over the chunk in fp32 (log2 domain).  With 48 or more
//    (query token, head) rows per KV head the rows of up to four KV heads
//    fill a 128-row tcgen05 tile instead: one thread issues the MMAs into
//    tensor memory, four warps run the softmax one row per thread.
//  * A segment (the part of one sequence -- or of one partition of it --
//    inside one CTA's range) ends by writing the final output directly when
//    it covers the whole sequence, else an unnormalised partial
//    (acc, m, l) for the log-sum-exp reduce kernel.
// Every wait on an mbarrier is bounded in time; a timeout sets
// PA_ERRBIT_WAIT_TIMEOUT and the CTA drains its outstanding copies and exits.
#pragma once

#include <climits>
#include <cstdint>
#include <type_traits>

#include "pa_device.cuh"

namespace pa {

constexpr int MAX_STAGES = 8;
constexpr int NQ = 2;                // query-row ring slots
// The tcgen05 path's query tile (128 rows x head_dim) is 32 KB: one slot
// there leaves room for one more K/V stage.
constexpr int nq_slots(bool um) { return um ? 1 : NQ; }
constexpr int MAX_WARPS = 9;         // up to 8 consumers + 1 producer

// GAP: this segment ends the CTA's range exactly at a partition end while
// its sequence continues in the next range; the slot after the segment's
// would stay unwritten, so the segment also writes an empty partial there
// (m = -inf, l = 0, acc = 0), keeping every sequence's partials consecutive.
// QLOAD: the segment's query rows were copied into ring slot qslot with this
// chunk.  A partition start inside a sequence that the CTA has already begun
// keeps the query fragments the consumers hold (the tcgen05 path, which reads
// the query from shared memory, always copies).
enum : uint32_t { SEG_START = 1u, SEG_END = 2u, DIRECT = 4u, GAP = 8u, QLOAD = 16u };

struct StageDesc {
    int seq;
    int tok0;
    int slot;
    uint32_t vmask;
    uint32_t flags;          // SEG_* bits; bits 16.. hold the sequence's query count
    int qslot;               // query ring slot of the segment's rows (written at QLOAD chunks)
    int qrow0;               // row of the sequence's first query token in q / out
    int qpos0;               // its position in the sequence (queries are the last tokens)
};
constexpr int QCOUNT_SHIFT = 16;

struct DecodeParams {
    void* out;
    const void* q;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    float* part_acc;          // [max_slots][Hq][D]
    float2* part_ml;          // [max_slots][Hq]  (m in log2 units, l)
    int4* split_list;         // [B] sequences needing a merge: (seq, first slot, slot count, -1) when
                              // their partials are consecutive slots, else (seq, first chunk, first unit, length)
    int* totals;              // [0] chunks, [1] units, [2] entries in split_list
    int32_t* err_flag;
    int B, Hq, Hkv, G, D, bs, NB, MB;
    int out_bytes;            // bytes of one output element
    int HPC, NHG, NR, MT, NCW;
    int ct;                   // tokens per chunk (pipeline stage): 16, or 32 for native e4m3
    int PC;                   // partition length in chunks, 0 = none
    const int32_t* q_start;   // several query tokens per sequence: [B+1] row offsets; null = one each
    int QL;                   // most query tokens of a sequence (1 for decode)
    int total_q;              // query rows in q / out
    int WQ, WS;               // schedule weights of a chunk and of a unit start
    int max_slots;
    float qk_scale;           // scale * log2(e) (* k_scale for fp8)
    float v_scale;            // v_scale for fp8, else 1
    int stages;
    int rpb;                  // rows per TMA box = min(16, bs)
    uint32_t box_bytes;       // bytes of one K (or V) box
    uint32_t kv_bytes;        // bytes of one stage's K (or V) buffer
    uint32_t q_bytes;         // query bytes copied per query load
    uint32_t q_slot_bytes;    // one query ring slot
    uint32_t stage_bytes;     // K + V
    uint32_t q_off;           // offset of the query ring
    uint32_t simtq_off;       // offset of the CUDA-core private query rows
    uint32_t bar_off;         // offset of the barriers
    int per_head_copies;      // 1: one TMA copy per (head, 128-B column block)
    int q_tma;                // 1: query rows arrive by a 128-B-swizzled tensor copy
    uint32_t q_plane_bytes;   // tcgen05 path: distance between the query slot's 128-B column planes
    int um_rows;              // tcgen05 path: tile rows per KV head (its query rows padded to 32)
};

__device__ __forceinline__ int cdiv_i(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ int clamp_len(int L, int maxL) {
    return L < 0 ? 0 : (L > maxL ? maxL : L);
}
__device__ __forceinline__ int n_units(int L, int PC, int ct) {
    const int nch = cdiv_i(L, ct);
    return nch == 0 ? 0 : (PC > 0 ? cdiv_i(nch, PC) : 1);
}
// Query rows [qa, qa + qn) of sequence i: row i in decode, q_start[i] ..
// q_start[i+1] with several query tokens.  Entries that are not increasing
// inside [0, total_q], or give more than QL tokens, make the sequence's query
// count 0 (nothing is read or written for it) and return false.
__device__ __forceinline__ bool query_rows(const DecodeParams& p, int i, int& qa, int& qn) {
    if (!p.q_start) { qa = i; qn = 1; return true; }
    const int a = __ldg(p.q_start + i), b = __ldg(p.q_start + i + 1);
    if (a < 0 || b < a || b > p.total_q || b - a > p.QL) { qa = 0; qn = 0; return false; }
    qa = a; qn = b - a;
    return true;
}

// Cost-weighted chunk stream.  Chunk k (global index) of global unit gu sits
// at position WQ*k + WS*(gu + 1): each chunk weighs WQ and each unit start WS
// more, for the per-segment work (query rows in, result out).  With
// W = WQ*C + WS*Ut over all C chunks and Ut units, range r (one CTA column)
// takes the chunks whose positions lie in [floor(r*W/NR), floor((r+1)*W/NR)):
// contiguous chunk intervals of about equal cost.
__device__ __forceinline__ long long stream_weight(const DecodeParams& p, int C, int Ut) {
    return static_cast<long long>(p.WQ) * C + static_cast<long long>(p.WS) * Ut;
}
__device__ __forceinline__ long long chunk_pos(const DecodeParams& p, int k, int gu) {
    return static_cast<long long>(p.WQ) * k + static_cast<long long>(p.WS) * (gu + 1);
}
// (Divisions run in 32 bits whenever W * NR fits, as it does for any
// realistic batch; 64-bit integer division is several times slower.)
__device__ __forceinline__ bool fits32(long long W, int NR) {
    return W * NR < 0x7fffffffLL;
}
__device__ __forceinline__ long long range_lo(int r, long long W, int NR) {
    if (fits32(W, NR))
        return static_cast<unsigned>(r) * static_cast<unsigned>(W) / static_cast<unsigned>(NR);
    return static_cast<long long>(r) * W / NR;
}
// the range holding weighted position pos: largest r with range_lo(r) <= pos
__device__ __forceinline__ int range_of_pos(long long pos, long long W, int NR) {
    if (fits32(W, NR))
        return static_cast<int>((static_cast<unsigned>(pos + 1) * static_cast<unsigned>(NR) - 1u) /
                                static_cast<unsigned>(W));
    return static_cast<int>(((pos + 1) * NR - 1) / W);
}
// first chunk k in [a, b) of a unit (positions WQ*k + base) with position >= t
__device__ __forceinline__ int first_chunk_from(long long t, int a, long long base, int WQ) {
    const long long d = t - base;
    long long k = 0;
    if (d > 0) k = d < 0x7fffffffLL ? static_cast<long long>((static_cast<unsigned>(d) + WQ - 1) / WQ) : (d + WQ - 1) / WQ;
    return static_cast<int>(k > a ? k : a);
}
// Every range spans at least WQ + WS positions, the largest gap between
// consecutive chunks, so no range is empty.
__device__ __forceinline__ bool dense_ranges(const DecodeParams& p, long long W) {
    return W >= static_cast<long long>(p.WQ + p.WS) * p.NR;
}
// does range r hold a chunk of the unit [a, b) with base offset `base`?
__device__ __forceinline__ bool unit_in_range(int r, int a, int b, long long base, long long W, int NR, int WQ) {
    const int k = first_chunk_from(range_lo(r, W, NR), a, base, WQ);
    return k < b && static_cast<long long>(WQ) * k + base < range_lo(r + 1, W, NR);
}

// ---------------------------------------------------------------------------
// CTA prologue: chunk totals, this CTA's range, and the sequence holding
// the range's first chunk.  CTA 0 also publishes per-sequence prefixes for
// the reduce kernel.
// ---------------------------------------------------------------------------
struct Plan {
    int cs, ce;               // chunk range [cs, ce)
    int seq, S, U;            // first sequence, its first chunk and unit
    int C, Ut;                // totals
};

__device__ __forceinline__ void warp_scan_pair(int& a, int& b) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, a, o);
        const int y = __shfl_up_sync(0xffffffffu, b, o);
        if (lane >= o) { a += x; b += y; }
    }
}

__device__ inline void make_plan(const DecodeParams& p, int range, int2* scratch, int4* s_first, int2* s_tot,
                                 int* s_end, Plan& plan) {
    const int tid = threadIdx.x, nth = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = nth >> 5;
    const int maxL = p.MB * p.bs;
    const int per = cdiv_i(p.B, nth);
    const int i0 = min(p.B, tid * per), i1 = min(p.B, i0 + per);
    int csum = 0, usum = 0;
    bool bad = false;
    int L0raw = 0;                      // the first of the thread's lengths, reused below
    for (int i = i0; i < i1; ++i) {
        const int Lraw = p.seq_lens[i];
        if (i == i0) L0raw = Lraw;
        bad |= (Lraw < 0 || Lraw > maxL);
        const int L = clamp_len(Lraw, maxL);
        csum += cdiv_i(L, p.ct);
        usum += n_units(L, p.PC, p.ct);
    }
    if (bad && blockIdx.x == 0) raise_flag(p.err_flag, PA_ERRBIT_SEQ_TOO_LONG);
    if (blockIdx.x == 0 && tid == 0) p.totals[2] = 0;
    int ci = csum, ui = usum;           // inclusive within the warp
    warp_scan_pair(ci, ui);
    if (lane == 31) scratch[warp] = make_int2(ci, ui);
    if (tid == 0) { *s_first = make_int4(-1, 0, 0, 0); *s_end = INT_MAX; }
    __syncthreads();
    if (warp == 0) {
        int2 v = lane < nwarps ? scratch[lane] : make_int2(0, 0);
        int a = v.x, b = v.y;
        warp_scan_pair(a, b);
        if (lane < nwarps) scratch[lane] = make_int2(a - v.x, b - v.y);   // exclusive
        if (lane == nwarps - 1) *s_tot = make_int2(a, b);
    }
    __syncthreads();
    const int2 wpre = scratch[warp];
    const int cpre = wpre.x + ci - csum, upre = wpre.y + ui - usum;       // exclusive per thread
    const int C = s_tot->x, Ut = s_tot->y;
    const long long W = stream_weight(p, C, Ut);
    // The range starts at the first chunk with position >= lo and ends at
    // the first with position >= hi; the thread whose sequences hold such a
    // chunk records it.
    const long long lo = range_lo(range, W, p.NR), hi = range_lo(range + 1, W, p.NR);
    if (csum > 0) {
        const long long prev_last = cpre > 0 ? chunk_pos(p, cpre - 1, upre - 1) : -1;
        const long long my_last = chunk_pos(p, cpre + csum - 1, upre + usum - 1);
        const bool has_lo = prev_last < lo && lo <= my_last;
        const bool has_hi = prev_last < hi && hi <= my_last;
        if (has_lo || has_hi) {
            int S = cpre, U = upre;
            bool need_lo = has_lo, need_hi = has_hi;
            // the first chunk of sequence (S, U, nch, nu) at or after
            // position t, or -1 if its last chunk lies before t
            auto find = [&](long long t, int S, int U, int nch, int nu) -> int {
                int u = 0;
                if (p.PC > 0 && nu > 1) {
                    // last chunk of unit u < nu-1 sits at
                    // (WQ*PC + WS)*(u+1) + WQ*(S-1) + WS*U
                    const long long step = static_cast<long long>(p.WQ) * p.PC + p.WS;
                    const long long d = t - (static_cast<long long>(p.WQ) * (S - 1) + static_cast<long long>(p.WS) * U);
                    const long long uu = d <= step ? 0 : (d + step - 1) / step - 1;
                    u = static_cast<int>(uu < nu - 1 ? uu : nu - 1);
                }
                const int a = S + (p.PC > 0 ? u * p.PC : 0);
                const int b = p.PC > 0 ? min(a + p.PC, S + nch) : S + nch;
                const long long base = static_cast<long long>(p.WS) * (U + u + 1);
                if (t > static_cast<long long>(p.WQ) * (b - 1) + base) return -1;
                return first_chunk_from(t, a, base, p.WQ);
            };
            for (int i = i0; i < i1 && (need_lo || need_hi); ++i) {
                const int L = clamp_len(i == i0 ? L0raw : p.seq_lens[i], maxL);
                const int nch = cdiv_i(L, p.ct), nu = n_units(L, p.PC, p.ct);
                if (nch > 0) {
                    if (need_lo) {
                        const int k = find(lo, S, U, nch, nu);
                        if (k >= 0) { *s_first = make_int4(i, S, U, k); need_lo = false; }
                    }
                    if (need_hi) {
                        const int k = find(hi, S, U, nch, nu);
                        if (k >= 0) { *s_end = k; need_hi = false; }
                    }
                }
                S += nch;
                U += nu;
            }
        }
    }
    if (blockIdx.x == 0) {
        // Sequences split across ranges or partitions go to the merge list;
        // empty sequences get zero outputs here.
        int S = cpre, U = upre;
        for (int i = i0; i < i1; ++i) {
            const int L = clamp_len(p.seq_lens[i], maxL);
            const int nch = cdiv_i(L, p.ct), nu = n_units(L, p.PC, p.ct);
            if (L == 0) {
                // no keys: zero outputs for every query row of the sequence
                int qa, qn;
                query_rows(p, i, qa, qn);
                uint4* o = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) +
                                                    static_cast<size_t>(qa) * p.Hq * p.D * p.out_bytes);
                for (int k = 0; k < qn * p.Hq * p.D * p.out_bytes / 16; ++k) o[k] = make_uint4(0, 0, 0, 0);
            } else {
                const int r0 = range_of_pos(chunk_pos(p, S, U), W, p.NR);
                const int r1 = range_of_pos(chunk_pos(p, S + nch - 1, U + nu - 1), W, p.NR);
                if (nu > 1 || r0 != r1) {
                    // The partials sit in consecutive slots r0 + U ..
                    // r1 + U + nu - 1 when every range between r0 and r1
                    // holds a chunk of the sequence (GAP segments fill the
                    // slots skipped at range ends that meet partition ends).
                    int4 e = make_int4(i, S, U, L);
                    if ((nu == 1 && C >= p.NR) || dense_ranges(p, W)) {
                        const int first = r0 + U, last = r1 + U + nu - 1;
                        e = make_int4(i, first, min(last - first + 1, p.max_slots - first), -1);
                    }
                    p.split_list[atomicAdd(&p.totals[2], 1)] = e;
                }
            }
            S += nch;
            U += nu;
        }
        if (tid == 0) { p.totals[0] = C; p.totals[1] = Ut; }
        __threadfence();             // the merge kernel reads the list before this grid ends
    }
    __syncthreads();
    const int4 f = *s_first;
    plan.cs = f.x >= 0 ? f.w : C;
    plan.ce = min(*s_end, C);
    plan.seq = f.x; plan.S = f.y; plan.U = f.z;
    plan.C = C; plan.Ut = Ut;
}

// ---------------------------------------------------------------------------
// Shared-memory addressing of one stage's K or V buffer.  A box holds
// `rpb` token rows of all HPC heads, laid out [col_block][head][row][128 B]
// with the 128-B TMA swizzle; a 16-token chunk is 16 / rpb boxes.
// ---------------------------------------------------------------------------
struct KVLayout {
    uint32_t box_bytes, head_stride, dh_stride;
    int rpb;
    __device__ __forceinline__ uint32_t row_base(int tok, int hl) const {
        const int b = tok / rpb, r = tok - b * rpb;
        return b * box_bytes + (hl * rpb + r) * 128u;
    }
    // byte offset of 16-byte column chunk `c` (c = 0 .. D*e/16-1) of token row
    __device__ __forceinline__ uint32_t chunk_addr(uint32_t rowbase, int tok, int c) const {
        return rowbase + (c >> 3) * dh_stride + (((c & 7) ^ (tok & 7)) << 4);
    }
};

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// Four consecutive output values in one vector store.
template <typename T> __device__ __forceinline__ void store4(T* dst, const float (&v)[4]);
template <> __device__ __forceinline__ void store4<float>(float* dst, const float (&v)[4]) {
    *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}
template <> __device__ __forceinline__ void store4<__half>(__half* dst, const float (&v)[4]) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack2(v[0], v[1], false), pack2(v[2], v[3], false));
}
template <> __device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, const float (&v)[4]) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack2(v[0], v[1], true), pack2(v[2], v[3], true));
}

// Barriers and the tensor-memory base of the tcgen05 path (shared memory).
struct UmBars {
    uint64_t sfull[2];        // S of chunk k in tensor-memory buffer k % 2 (MMA commit)
    uint64_t pfull[2];        // P of chunk k in shared-memory buffer k % 2 (one arrival per consumer warp)
    uint64_t pvdone[2];       // P V of chunk k added to O (MMA commit): P buffer k % 2 free again
    uint64_t ofree;           // a segment's O read out (one arrival per consumer warp)
    uint64_t fin;             // every MMA of the CTA complete
    uint32_t tmem;            // tensor-memory base address
};

template <class KV, class QT, int D, bool TC, int CT, bool MQ = false, bool T8 = false, bool UM = false>
struct DecodeKernel {
    using KT = typename KV::T;
    using QE = typename QT::T;
    static constexpr bool FP8 = (KV::bytes == 1);             // e4m3 or e5m2
    // 32-token chunks are the native-e4m3 tensor-core variant (fp8 operands,
    // m16n8k32); every other variant runs 16-token chunks.
    static constexpr bool NATIVE8 = (CT == 32);
    static_assert(CT == 16 || (CT == 32 && ((FP8 && TC && D == 128) || UM)),
                  "32-token chunks: the fp8 tensor-core and the tcgen05 paths only");
    static constexpr bool KV_E5M2 = (KV::code == PA_FP8_E5M2);
    static constexpr int MAXB = CT / 8;       // TMA boxes per chunk at the smallest block size
    static constexpr bool MMA_BF16 = (KV::code == PA_BF16);   // fp8 runs in f16
    static constexpr int NT = D / 8;          // 8-wide output column tiles
    static constexpr int KS = D / 16;         // 16-deep k-steps over head_dim
    static constexpr int ROWB = D * KV::bytes;  // bytes of one K/V row
    static constexpr int CPR = ROWB / 16;     // 16-byte chunks per row
    static_assert(!UM || (MQ && TC && !FP8), "tcgen05 path: several query tokens, 16-bit caches");
    static constexpr int UM_M = 128;          // tcgen05 tile rows: (query token, head) rows of one KV head
    static constexpr int UM_TCOLS = 256;      // tensor-memory columns per CTA: two S buffers, then O
    static constexpr uint32_t UM_PBUF = UM_M * CT * 2;   // bytes of one P buffer (one head, one chunk)

    // ---------------- producer ----------------
    static __device__ void producer(const DecodeParams& p, const Plan& pl, int hg, uint8_t* base,
                                    uint64_t* full, uint64_t* empty, uint64_t* qempty, StageDesc* descs,
                                    const CUtensorMap* tk, const CUtensorMap* tv, const CUtensorMap* tq) {
        const int lane = threadIdx.x & 31;
        const int S = p.stages;
        const int maxL = p.MB * p.bs;
        // Sequence lengths come 32 sequences per warp-wide load, and block
        // table entries in 32-entry windows with the window after the
        // current one always in flight, so neither a change of sequence nor
        // a long sequence stalls the copy issue on a dependent global load.
        int lbase = pl.seq, lval = 0;
        auto load_lens = [&](int first) {
            lbase = first;
            const int ii = first + lane;
            lval = ii < p.B ? clamp_len(__ldg(p.seq_lens + ii), maxL) : 0;
        };
        auto len_of = [&](int ii) -> int {     // warp-uniform
            if (ii >= p.B) return 0;
            if (ii - lbase >= 32) load_lens(ii);
            return __shfl_sync(0xffffffffu, lval, ii - lbase);
        };
        auto load_win = [&](int seq, int wb, int nblk) -> int {
            const int idx = wb + lane;
            return (seq < p.B && idx < nblk) ? __ldg(p.block_tables + static_cast<size_t>(seq) * p.MB + idx) : -1;
        };
        load_lens(pl.seq);
        int i = pl.seq, Si = pl.S, Ui = pl.U;
        int j = pl.cs - Si;
        int wbase = (j * CT) / p.bs;                        // current window: blocks [wbase, wbase+32) of i
        // The first window is bounded by the table row instead of the
        // sequence's block count, so it loads alongside the lengths rather
        // than after them (entries past the sequence are never used).
        int wval = load_win(i, wbase, p.MB);
        int L = len_of(i);
        // first query row and query count of sequence i (one per sequence in decode)
        int qrow_i = i, qn_i = 1;
        auto load_q_rows = [&]() {
            if constexpr (MQ) {
                if (i < p.B) {
                    if (!query_rows(p, i, qrow_i, qn_i) && lane == 0) raise_flag(p.err_flag, PA_ERRBIT_BAD_QUERY);
                } else {
                    qrow_i = 0; qn_i = 0;
                }
            } else {
                qrow_i = i;
            }
        };
        load_q_rows();
        int nch = cdiv_i(L, CT), nbl = cdiv_i(L, p.bs);
        const int nb = p.bs >= CT ? 1 : CT / p.bs;      // boxes per chunk
        int nseq = 0, nbase = 0, nval = -1;                    // its successor
        auto prefetch_next = [&]() {
            if (wbase + 32 < nbl) {
                nseq = i; nbase = wbase + 32; nval = load_win(i, nbase, nbl);
            } else {
                nseq = i + 1; nbase = 0; nval = load_win(i + 1, 0, cdiv_i(len_of(i + 1), p.bs));
            }
        };
        prefetch_next();
        const int hq0 = hg * p.HPC * p.G;
        const int range = blockIdx.x / p.NHG;
        int issued = 0, qcount = 0;
        int slot = 0, qs = 0;                 // issued % S, qcount % NQ
        uint32_t round = 0, qround = 0;       // issued / S, qcount / NQ
        // Chunk j of sequence i is chunk jp of its partition ju (jp = j and
        // ju = 0 without partitions), tracked incrementally: a division by
        // the partition length per chunk, on the path from a stage coming
        // free to its refill, cost 7-10% with 512-token partitions.
        int jp = j, ju = 0;
        if (p.PC > 0) { ju = j / p.PC; jp = j - ju * p.PC; }
        bool ok = true;
        for (int k = pl.cs; k < pl.ce; ++k) {
            while (j >= nch) {
                Si += nch; Ui += n_units(L, p.PC, p.ct); ++i;
                L = len_of(i);
                load_q_rows();
                nch = cdiv_i(L, CT); nbl = cdiv_i(L, p.bs);
                j = 0; jp = 0; ju = 0;
                wbase = 0;
                wval = (nseq == i && nbase == 0) ? nval : load_win(i, 0, nbl);
                prefetch_next();
            }
            const int tok0 = j * CT;
            const int b0 = tok0 / p.bs;
            if (b0 + nb - 1 >= wbase + 32) {                   // step to the successor window
                if (nseq == i && nbase <= b0 && b0 + nb - 1 < nbase + 32) {
                    wbase = nbase; wval = nval;
                } else {
                    wbase = b0; wval = load_win(i, wbase, nbl);
                }
                prefetch_next();
            }
            int blk[MAXB];
#pragma unroll
            for (int b = 0; b < MAXB; ++b) blk[b] = __shfl_sync(0xffffffffu, wval, min(b0 + b - wbase, 31));
            if (lane == 0) {
                if (issued >= S && !mbar_wait_bounded(&empty[slot], (round - 1) & 1u)) {
                    raise_flag(p.err_flag, PA_ERRBIT_WAIT_TIMEOUT);
                    ok = false;
                }
                const bool seg_start = (k == pl.cs) || (jp == 0);
                const bool qload = seg_start && (UM || k == pl.cs || j == 0);
                const int ntok = min(CT, L - tok0);
                const uint32_t vmask_full = CT == 32 ? 0xffffffffu : ((1u << CT) - 1u);
                uint32_t vmask = (ntok >= 32) ? 0xffffffffu : ((1u << ntok) - 1u);
                vmask &= vmask_full;
                uint32_t nbox_issued = 0;
                uint32_t issue_mask = 0;
#pragma unroll
                for (int b = 0; b < MAXB; ++b) {
                    if (b >= nb) break;
                    const int first = b * p.rpb;
                    if (first >= ntok) continue;                 // nothing valid here
                    const int id = blk[b];
                    const uint32_t rows = (p.rpb >= 32 ? 0xffffffffu : ((1u << p.rpb) - 1u)) << first;
                    if (id < 0 || id >= p.NB) {
                        raise_flag(p.err_flag, PA_ERRBIT_BAD_BLOCK);
                        vmask &= ~rows;
                        continue;
                    }
                    issue_mask |= 1u << b;
                    ++nbox_issued;
                }
                const bool part_end = p.PC > 0 && jp == p.PC - 1;
                uint32_t flags = 0;
                if (seg_start) flags |= SEG_START;
                if (qload) flags |= QLOAD;
                if (k == pl.ce - 1 || j == nch - 1 || part_end) flags |= SEG_END;
                if (k == pl.ce - 1 && part_end && j + 1 < nch) flags |= GAP;
                const int nu = n_units(L, p.PC, p.ct);
                if (nu == 1 && Si >= pl.cs && Si + nch <= pl.ce) flags |= DIRECT;
                StageDesc d;
                d.seq = i; d.tok0 = tok0; d.vmask = vmask;
                d.flags = flags | (static_cast<uint32_t>(qn_i) << QCOUNT_SHIFT);
                d.slot = range + Ui + ju;
                d.qslot = qload ? qs : (qs == 0 ? nq_slots(UM) - 1 : qs - 1);
                d.qrow0 = qrow_i;
                d.qpos0 = L - qn_i;
                const uint32_t bytes = nbox_issued * p.box_bytes * 2u + (qload ? p.q_bytes : 0u);
                if (ok && qload && qcount >= nq_slots(UM) && !mbar_wait_bounded(&qempty[qs], (qround - 1) & 1u)) {
                    raise_flag(p.err_flag, PA_ERRBIT_WAIT_TIMEOUT);
                    ok = false;
                }
                if (ok) {
                    uint8_t* kbuf = base + slot * p.stage_bytes;
                    uint8_t* vbuf = kbuf + p.kv_bytes;
                    descs[slot] = d;
                    mbar_arrive_expect_tx(&full[slot], bytes);
#pragma unroll
                    for (int b = 0; b < MAXB; ++b) {
                        if (b >= nb) break;
                        if (!((issue_mask >> b) & 1u)) continue;
                        const int row0 = blk[b] * p.bs + (p.bs > CT ? (tok0 % p.bs) : 0);
                        if constexpr (UM) {
                            // tcgen05 layout: column plane dh of box b at
                            // (dh * nb + b) * pbox, so that one plane's rows of
                            // every box of the chunk are contiguous (the N rows
                            // of one S MMA)
                            const uint32_t pbox = static_cast<uint32_t>(p.HPC * p.rpb) * 128u;
#pragma unroll
                            for (int dh = 0; dh < ROWB / 128; ++dh) {
                                const uint32_t off = static_cast<uint32_t>(dh * nb + b) * pbox;
                                if (!p.per_head_copies) {
                                    tma_load_4d(kbuf + off, tk, &full[slot], 0, row0, hg * p.HPC, dh);
                                    tma_load_4d(vbuf + off, tv, &full[slot], 0, row0, hg * p.HPC, dh);
                                } else {
                                    const int E128 = 128 / KV::bytes;
                                    for (int hl = 0; hl < p.HPC; ++hl) {
                                        const uint32_t o2 = off + static_cast<uint32_t>(hl * p.rpb) * 128u;
                                        tma_load_3d(kbuf + o2, tk, &full[slot], dh * E128, hg * p.HPC + hl, row0);
                                        tma_load_3d(vbuf + o2, tv, &full[slot], dh * E128, hg * p.HPC + hl, row0);
                                    }
                                }
                            }
                            continue;
                        }
                        uint8_t* kd = kbuf + b * p.box_bytes;
                        uint8_t* vd = vbuf + b * p.box_bytes;
                        if (!p.per_head_copies) {
                            tma_load_4d(kd, tk, &full[slot], 0, row0, hg * p.HPC, 0);
                            tma_load_4d(vd, tv, &full[slot], 0, row0, hg * p.HPC, 0);
                        } else {
                            const int DH = ROWB / 128;
                            const int E128 = 128 / KV::bytes;
                            for (int dh = 0; dh < DH; ++dh)
                                for (int hl = 0; hl < p.HPC; ++hl) {
                                    const uint32_t off = ((dh * p.HPC + hl) * p.rpb) * 128u;
                                    tma_load_3d(kd + off, tk, &full[slot], dh * E128, hg * p.HPC + hl, row0);
                                    tma_load_3d(vd + off, tv, &full[slot], dh * E128, hg * p.HPC + hl, row0);
                                }
                        }
                    }
                    if (qload) {
                        const uint8_t* qsrc = static_cast<const uint8_t*>(p.q) +
                            (static_cast<size_t>(i) * p.Hq + hq0) * D * QT::bytes;
                        uint8_t* qdst = base + p.q_off + qs * p.q_slot_bytes;
                        if constexpr (UM) {
                            // per KV head of the CTA and 128-B column plane one
                            // copy of its [token][head] rows, to tile row
                            // um_rows * head; planes q_plane_bytes (a multiple of
                            // 1024) apart, so every swizzle atom starts aligned
                            for (int hl = 0; hl < p.HPC; ++hl)
#pragma unroll
                                for (int dh = 0; dh < ROWB / 128; ++dh)
                                    tma_load_4d(qdst + dh * p.q_plane_bytes + hl * p.um_rows * 128, tq, &full[slot], 0,
                                                hq0 + hl * p.G, qrow_i, dh);
                        } else if constexpr (MQ) {
                            // rows [token][head] of QL tokens x HPC*G heads, one 4-D copy
                            tma_load_4d(qdst, tq, &full[slot], 0, hq0, qrow_i, 0);
                        } else {
                            if (p.q_tma) tma_load_3d(qdst, tq, &full[slot], 0, i * p.Hq + hq0, 0);
                            else bulk_load(qdst, qsrc, p.q_bytes, &full[slot]);
                        }
                        ++qcount;
                        if (++qs == nq_slots(UM)) { qs = 0; ++qround; }
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            ++issued;
            if (++slot == S) { slot = 0; ++round; }
            ++j;
            if (++jp == p.PC) { jp = 0; ++ju; }
        }
        // drain: every copy this CTA issued must land before the CTA exits
        if (lane == 0) {
            const int first = max(0, issued - S);
            for (int st = first; st < issued; ++st) {
                if (!mbar_wait_bounded(&full[st % S], (st / S) & 1u)) {
                    raise_flag(p.err_flag, PA_ERRBIT_WAIT_TIMEOUT);
                    break;
                }
            }
        }
    }

    // ---------------- output of a finished segment ----------------
    template <typename OutT>
    static __device__ __forceinline__ void store_pair(OutT* dst, float a, float b) {
        dst[0] = from_float<OutT>(a);
        dst[1] = from_float<OutT>(b);
    }

    // Two query elements (one 32-bit word of QT) as an f16x2 MMA operand.
    static __device__ __forceinline__ uint32_t to_f16x2(uint32_t w) {
        if constexpr (QT::code == PA_F16) {
            return w;
        } else {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
            return pack2(f.x, f.y, false);
        }
    }

    // Column of accumulator element (tile nt, column pair index within the
    // tile n) in head_dim coordinates.
    static __device__ __forceinline__ int out_col(int nt, int n) {
        if constexpr (FP8) {
            return 16 * (nt >> 1) + 2 * n + (nt & 1);
        } else {
            return nt * 8 + n;
        }
    }

    // The two accumulator rows a lane owns (g4 and g4 + 8 of its 16-row
    // tile): which query token and which head each stands for.  Tile row R
    // of KV head hl is query token R / G, head R % G of the group; decode has
    // one token, so R is the head.
    struct RowInfo {
        int j[2];          // query token index within the sequence
        int head[2];       // query head
        bool in[2];        // inside the group's query rows
    };
    static __device__ __forceinline__ RowInfo row_info(const DecodeParams& p, int hg, int hl, int mt, int lane) {
        RowInfo ri;
        const int rows_total = p.QL * p.G;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int R = 16 * mt + (lane >> 2) + 8 * hh;
            const int jj = R / p.G;
            ri.j[hh] = jj;
            ri.head[hh] = hg * p.HPC * p.G + hl * p.G + (R - jj * p.G);
            ri.in[hh] = R < rows_total;
        }
        return ri;
    }
    // Row of the query ring slot holding tile row R of KV head hl: the slot
    // is [token][HPC * G heads] (one token in decode).
    static __device__ __forceinline__ int q_smem_row(const DecodeParams& p, int hl, int R) {
        const int jj = R / p.G;
        return jj * p.HPC * p.G + hl * p.G + (R - jj * p.G);
    }

    // End of a segment: the normalised output rows when the segment covers
    // the whole sequence (DIRECT), else the unnormalised partial (acc, m, l)
    // for the merge kernel.  Rows g4 and g4 + 8 of the tile, columns from
    // out_col(); rows past the group or past the sequence's query tokens are
    // not stored.
    static __device__ __forceinline__ void finish_segment(const DecodeParams& p, const StageDesc& d,
                                                          const float (&acc)[NT][4], float m0, float m1,
                                                          float l0, float l1, int lane, int rows_valid,
                                                          const RowInfo& ri) {
        const int g4 = lane >> 2, t4 = lane & 3;
        float lt0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
        lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
        float lt1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
        lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
        const bool direct = (d.flags & DIRECT) != 0;
        if (!(direct || d.slot < p.max_slots)) return;
        const int qn = static_cast<int>(d.flags >> QCOUNT_SHIFT);
        float sc0 = p.v_scale, sc1 = p.v_scale;
        if (direct) {
            sc0 = lt0 > 0.f ? p.v_scale / lt0 : 0.f;
            sc1 = lt1 > 0.f ? p.v_scale / lt1 : 0.f;
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            if (hh == 1 && rows_valid <= 8) break;      // rows 8..15 are padding
            const bool ok = ri.in[hh] && ri.j[hh] < qn;
            const float sc = hh ? sc1 : sc0;
            QE* orow = static_cast<QE*>(p.out) +
                       (static_cast<size_t>(d.qrow0 + ri.j[hh]) * p.Hq + ri.head[hh]) * D;
            float* prow = p.part_acc +
                          ((static_cast<size_t>(d.slot) * p.QL + ri.j[hh]) * p.Hq + ri.head[hh]) * D;
            // Each lane stores 4 consecutive columns of a row per pair of
            // column tiles.  With fp8 the permuted head_dim order already
            // gives every lane 4 consecutive columns; otherwise one exchange
            // between lane pairs of a quad assembles them.
#pragma unroll
            for (int q2 = 0; q2 < NT / 2; ++q2) {
                const float a0 = acc[2 * q2][2 * hh] * sc, a1 = acc[2 * q2][2 * hh + 1] * sc;
                const float b0 = acc[2 * q2 + 1][2 * hh] * sc, b1 = acc[2 * q2 + 1][2 * hh + 1] * sc;
                float v[4];
                int col;
                if constexpr (FP8) {
                    v[0] = a0; v[1] = b0; v[2] = a1; v[3] = b1;
                    col = 16 * q2 + 4 * t4;
                } else {
                    const bool odd = (t4 & 1) != 0;
                    const float r0 = __shfl_xor_sync(0xffffffffu, odd ? a0 : b0, 1);
                    const float r1 = __shfl_xor_sync(0xffffffffu, odd ? a1 : b1, 1);
                    if (odd) { v[0] = r0; v[1] = r1; v[2] = b0; v[3] = b1; col = 16 * q2 + 8 + 2 * (t4 - 1); }
                    else     { v[0] = a0; v[1] = a1; v[2] = r0; v[3] = r1; col = 16 * q2 + 2 * t4; }
                }
                if (ok) {
                    if (direct) store4<QE>(orow + col, v);
                    else store4<float>(prow + col, v);
                }
            }
            if (!direct && ok && t4 == 0)
                p.part_ml[(static_cast<size_t>(d.slot) * p.QL + ri.j[hh]) * p.Hq + ri.head[hh]] =
                    make_float2(hh ? m1 : m0, hh ? lt1 : lt0);
        }
        (void)g4;
    }

    // An empty partial (m = -inf, l = 0, acc = 0) at `slot` for every query
    // row of the warp's tile (tile rows 16*mt .. +rows).
    static __device__ __forceinline__ void write_empty_partial(const DecodeParams& p, int slot, int hg, int hl,
                                                               int mt, int rows, int lane) {
        if (slot >= p.max_slots) return;
        for (int r = 0; r < rows; ++r) {
            const int R = 16 * mt + r;
            const int jj = R / p.G;
            const int head = hg * p.HPC * p.G + hl * p.G + (R - jj * p.G);
            const size_t row = (static_cast<size_t>(slot) * p.QL + jj) * p.Hq + head;
            float4* acc = reinterpret_cast<float4*>(p.part_acc + row * D);
            for (int e = lane; e < D / 4; e += 32) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (lane == 0) p.part_ml[row] = make_float2(-INFINITY, 0.f);
        }
    }

    // ---------------- tensor-core consumer ----------------
    static __device__ void consumer_tc(const DecodeParams& p, const Plan& pl, int hg, int w,
                                       uint8_t* base, uint64_t* full, uint64_t* empty, uint64_t* qempty,
                                       const StageDesc* descs) {
        const int lane = threadIdx.x & 31;
        const int g4 = lane >> 2, t4 = lane & 3;
        const int hl = w / p.MT, mt = w - hl * p.MT;
        const int rows_valid = min(16, p.QL * p.G - 16 * mt);
        const int S = p.stages;
        const KVLayout lay{p.box_bytes, static_cast<uint32_t>(p.rpb) * 128u,
                           static_cast<uint32_t>(p.HPC * p.rpb) * 128u, p.rpb};
        // per-lane ldmatrix rows
        const int mi = lane >> 3, r8 = lane & 7;
        const int tokK = (mi >> 1) * 8 + r8;       // K (non-transposed) row
        const int tokV = (mi & 1) * 8 + r8;        // V (transposed) row
        const uint32_t rbK = lay.row_base(tokK, hl), rbV = lay.row_base(tokV, hl);
        const RowInfo ri = row_info(p, hg, hl, mt, lane);

        float acc[NT][4];
        uint32_t qa[KS][4];
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        int lim0 = INT_MAX, lim1 = INT_MAX;         // last key position each row may attend

        for (int st = 0, k = pl.cs; k < pl.ce; ++k, ++st) {
            const int slot = st % S;
            if (!mbar_wait_bounded(&full[slot], (st / S) & 1u)) {
                if (lane == 0) raise_flag(p.err_flag, PA_ERRBIT_WAIT_TIMEOUT);
                return;
            }
            const StageDesc d = descs[slot];
            uint8_t* kbuf = base + slot * p.stage_bytes;
            uint8_t* vbuf = kbuf + p.kv_bytes;
            if (d.flags & SEG_START) {
                if (d.flags & QLOAD) {
                    load_q_frags(qa, base + p.q_off + d.qslot * p.q_slot_bytes, p, hl, mt, rows_valid, lane);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&qempty[d.qslot]);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
                m0 = m1 = -INFINITY; l0 = l1 = 0.f;
                if constexpr (MQ) {
                    // causal: query token j attends keys up to its own position
                    const int qn = static_cast<int>(d.flags >> QCOUNT_SHIFT);
                    lim0 = (ri.in[0] && ri.j[0] < qn) ? d.qpos0 + ri.j[0] : -1;
                    lim1 = (ri.in[1] && ri.j[1] < qn) ? d.qpos0 + ri.j[1] : -1;
                }
            }
            // V fragments of masked token rows are zeroed in registers: the
            // pool may hold NaN there and 0 * NaN would poison the sum.  A
            // fragment register holds token 2t in its low half and 2t+1 in
            // its high half (rows 8+2t, 8+2t+1 for the second k-half).
            const uint32_t vk0 = (((d.vmask >> (2 * t4)) & 1u) ? 0x0000ffffu : 0u) |
                                 (((d.vmask >> (2 * t4 + 1)) & 1u) ? 0xffff0000u : 0u);
            const uint32_t vk1 = (((d.vmask >> (8 + 2 * t4)) & 1u) ? 0x0000ffffu : 0u) |
                                 (((d.vmask >> (9 + 2 * t4)) & 1u) ? 0xffff0000u : 0u);
            // ---- S = Q K^T (16 rows x 16 tokens) ----
            float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            const uint32_t kb = smem_u32(kbuf);
            if constexpr (!FP8) {
                // two accumulator chains per tile (even / odd k-steps) halve the
                // dependent-MMA latency of the chunk
                float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < KS; ks += 2) {
                    uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
                    ldsm_x4(kb + lay.chunk_addr(rbK, tokK, 2 * ks + (mi & 1)), b0, b1, b2, b3);
                    ldsm_x4(kb + lay.chunk_addr(rbK, tokK, 2 * ks + 2 + (mi & 1)), c0, c1, c2, c3);
                    mma_16816<MMA_BF16>(s[0], qa[ks], b0, b1);
                    mma_16816<MMA_BF16>(s[1], qa[ks], b2, b3);
                    mma_16816<MMA_BF16>(s2[0], qa[ks + 1], c0, c1);
                    mma_16816<MMA_BF16>(s2[1], qa[ks + 1], c2, c3);
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[nt][e] += s2[nt][e];
            } else {
                float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < KS; ks += 2) {
                    uint32_t r0, r1, r2, r3;    // (tile0,ks) (tile0,ks+1) (tile1,ks) (tile1,ks+1)
                    ldsm_x4(kb + lay.chunk_addr(rbK, tokK, ks + (mi & 1)), r0, r1, r2, r3);
                    mma_16816<false>(s[0], qa[ks], fp8x2_to_f16x2<KV>(r0), fp8x2_to_f16x2<KV>(r0 >> 16));
                    mma_16816<false>(s2[0], qa[ks + 1], fp8x2_to_f16x2<KV>(r1), fp8x2_to_f16x2<KV>(r1 >> 16));
                    mma_16816<false>(s[1], qa[ks], fp8x2_to_f16x2<KV>(r2), fp8x2_to_f16x2<KV>(r2 >> 16));
                    mma_16816<false>(s2[1], qa[ks + 1], fp8x2_to_f16x2<KV>(r3), fp8x2_to_f16x2<KV>(r3 >> 16));
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[nt][e] += s2[nt][e];
            }
            // ---- online softmax (log2 domain), rows g4 and g4+8 ----
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int col = nt * 8 + 2 * t4 + (e & 1);
                    bool keep = ((d.vmask >> col) & 1u) != 0;
                    if constexpr (MQ) keep = keep && d.tok0 + col <= (e < 2 ? lim0 : lim1);
                    s[nt][e] = keep ? s[nt][e] * p.qk_scale : -INFINITY;
                }
            float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
            float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
            const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
            const float al0 = exp2f(m0 - mu0), al1 = exp2f(m1 - mu1);
            m0 = mn0; m1 = mn1;
            float pr[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                pr[nt][0] = exp2f(s[nt][0] - mu0);
                pr[nt][1] = exp2f(s[nt][1] - mu0);
                pr[nt][2] = exp2f(s[nt][2] - mu1);
                pr[nt][3] = exp2f(s[nt][3] - mu1);
            }
            l0 = l0 * al0 + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
            l1 = l1 * al1 + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
            if (!__all_sync(0xffffffffu, al0 == 1.f && al1 == 1.f)) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    acc[nt][0] *= al0; acc[nt][1] *= al0;
                    acc[nt][2] *= al1; acc[nt][3] *= al1;
                }
            }
            uint32_t pa[4];
            pa[0] = pack2(pr[0][0], pr[0][1], MMA_BF16);
            pa[1] = pack2(pr[0][2], pr[0][3], MMA_BF16);
            pa[2] = pack2(pr[1][0], pr[1][1], MMA_BF16);
            pa[3] = pack2(pr[1][2], pr[1][3], MMA_BF16);
            // ---- acc += P V ----
            const uint32_t vb = smem_u32(vbuf);
            if constexpr (!FP8) {
#pragma unroll
                for (int j2 = 0; j2 < NT / 2; ++j2) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vb + lay.chunk_addr(rbV, tokV, 2 * j2 + (mi >> 1)), b0, b1, b2, b3);
                    mma_16816<MMA_BF16>(acc[2 * j2], pa, b0 & vk0, b1 & vk1);
                    mma_16816<MMA_BF16>(acc[2 * j2 + 1], pa, b2 & vk0, b3 & vk1);
                }
            } else {
#pragma unroll
                for (int c2 = 0; c2 < D / 16; c2 += 2) {
                    uint32_t r0, r1, r2, r3;  // (tok0-7,c) (tok8-15,c) (tok0-7,c+1) (tok8-15,c+1)
                    ldsm_x4_t(vb + lay.chunk_addr(rbV, tokV, c2 + (mi >> 1)), r0, r1, r2, r3);
                    const uint32_t x0 = __byte_perm(r0 & vk0, 0, 0x3120), x1 = __byte_perm(r1 & vk1, 0, 0x3120);
                    const uint32_t x2 = __byte_perm(r2 & vk0, 0, 0x3120), x3 = __byte_perm(r3 & vk1, 0, 0x3120);
                    mma_16816<false>(acc[2 * c2], pa, fp8x2_to_f16x2<KV>(x0), fp8x2_to_f16x2<KV>(x1));
                    mma_16816<false>(acc[2 * c2 + 1], pa, fp8x2_to_f16x2<KV>(x0 >> 16), fp8x2_to_f16x2<KV>(x1 >> 16));
                    mma_16816<false>(acc[2 * c2 + 2], pa, fp8x2_to_f16x2<KV>(x2), fp8x2_to_f16x2<KV>(x3));
                    mma_16816<false>(acc[2 * c2 + 3], pa, fp8x2_to_f16x2<KV>(x2 >> 16), fp8x2_to_f16x2<KV>(x3 >> 16));
                }
            }
            // The stage's shared memory is no longer read: hand it back to
            // the producer before the segment-end epilogue.
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (d.flags & SEG_END) {
                finish_segment(p, d, acc, m0, m1, l0, l1, lane, rows_valid, ri);
                if ((d.flags & GAP) && !(d.flags & DIRECT))
                    write_empty_partial(p, d.slot + 1, hg, hl, mt, rows_valid, lane);
            }
        }
    }

    // ---------------- native-e4m3 tensor-core consumer ----------------
    // fp8 caches, 32-token chunks, GQA groups of at most 8 query heads.  The
    // key and value bytes enter the MMA as stored (m16n8k32, e4m3 x e4m3 ->
    // fp32), so nothing is converted per token.  The query and the softmax
    // weights are each carried as two e4m3 terms, hi = e4m3(x) and
    // lo = e4m3(x - hi) (about 8 significant bits together), placed in the
    // two halves of the 16-row tile: row r < 8 holds the hi term of query
    // head r and row r + 8 its lo term.  A lane owns rows g and g + 8 of
    // every accumulator tile, so hi + lo is a register add: scores after
    // Q K^T, outputs at the end of the segment.  The query tile is scaled by
    // a power of two 2^e putting its largest magnitude in [128, 256) (2^-e
    // goes into the score scale), and the weights are 2^8 * exp2(s - m), in
    // [0, 256]: that factor is common to acc and l and cancels in acc / l
    // and in the log-sum-exp merge.
    static constexpr int KS8 = D / 32;        // 32-deep k-steps over head_dim

    static __device__ __forceinline__ uint32_t token_bytemask(uint32_t x) {
        // bits 0, 1, 8, 9 of x -> bytes 0, 1, 2, 3 (0xff where set)
        const uint32_t y = (x & 1u) | ((x & 2u) << 7) | ((x & 0x100u) << 8) | ((x & 0x200u) << 15);
        return y * 0xffu;
    }

    // (hi, lo) e4m3 byte pairs of two non-negative weights
    static __device__ __forceinline__ void split_e4m3x2(float a, float b, uint32_t& hi, uint32_t& lo) {
        const uint32_t h = f32x2_to_f16x2(a, b);
        hi = f16x2_to_e4m3x2(h);
        lo = f16x2_to_e4m3x2(sub_f16x2(h, e4m3x2_to_f16x2(hi)));
    }

    static __device__ void consumer_e4m3(const DecodeParams& p, const Plan& pl, int hg, int w,
                                         uint8_t* base, uint64_t* full, uint64_t* empty, uint64_t* qempty,
                                         const StageDesc* descs) {
        const int lane = threadIdx.x & 31;
        const int t4 = lane & 3;
        const int hl = w;                           // one tile per KV head (G <= 8)
        const int rows_valid = p.G;
        const int S = p.stages;
        const KVLayout lay{p.box_bytes, static_cast<uint32_t>(p.rpb) * 128u,
                           static_cast<uint32_t>(p.HPC * p.rpb) * 128u, p.rpb};
        const int mi = lane >> 3, r8 = lane & 7;
        // K: ldmatrix matrices (tokens 0-7, k 0-15 | tokens 0-7, k 16-31 |
        // tokens 8-15, k 0-15 | tokens 8-15, k 16-31) of each half-chunk
        const int tokK = (mi >> 1) * 8 + r8;
        const uint32_t rbK0 = lay.row_base(tokK, hl), rbK1 = lay.row_base(tokK + 16, hl);
        // V (transposed): matrix mi holds tokens 8mi .. 8mi+7 of a 16-byte column chunk
        const int tokV = mi * 8 + r8;
        const uint32_t rbV = lay.row_base(tokV, hl);

        float acc[NT][4];
        uint32_t qa[KS8][4];
        float m0 = -INFINITY, l0 = 0.f;
        float qk_scale = p.qk_scale;
        const int qrow_lo = hl * p.G;
        RowInfo ri = row_info(p, hg, hl, 0, lane);
        ri.in[1] = false;                           // rows g4 + 8 hold the lo terms, not outputs

        for (int st = 0, k = pl.cs; k < pl.ce; ++k, ++st) {
            const int slot = st % S;
            if (!mbar_wait_bounded(&full[slot], (st / S) & 1u)) {
                if (lane == 0) raise_flag(p.err_flag, PA_ERRBIT_WAIT_TIMEOUT);
                return;
            }
            const StageDesc d = descs[slot];
            uint8_t* kbuf = base + slot * p.stage_bytes;
            uint8_t* vbuf = kbuf + p.kv_bytes;
            if (d.flags & SEG_START) {
                if (d.flags & QLOAD) {
                    qk_scale = p.qk_scale * load_q_e4m3(qa, base + p.q_off + d.qslot * p.q_slot_bytes, qrow_lo,
                                                        rows_valid, lane, p.q_tma, p.HPC * p.G);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&qempty[d.qslot]);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
                m0 = -INFINITY; l0 = 0.f;
            }
            // ---- S = Q K^T: 16 rows x 32 tokens, four 8-token tiles ----
            float s[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
            const uint32_t kb = smem_u32(kbuf);
#pragma unroll
            for (int ks = 0; ks < KS8; ++ks) {
                uint32_t r0, r1, r2, r3, c0, c1, c2, c3;
                ldsm_x4(kb + lay.chunk_addr(rbK0, tokK, 2 * ks + (mi & 1)), r0, r1, r2, r3);
                ldsm_x4(kb + lay.chunk_addr(rbK1, tokK, 2 * ks + (mi & 1)), c0, c1, c2, c3);
                mma_e4m3_16832<KV_E5M2>(s[0], qa[ks], r0, r1);
                mma_e4m3_16832<KV_E5M2>(s[1], qa[ks], r2, r3);
                mma_e4m3_16832<KV_E5M2>(s[2], qa[ks], c0, c1);
                mma_e4m3_16832<KV_E5M2>(s[3], qa[ks], c2, c3);
            }
            // ---- online softmax (log2 domain) of row g4 over 8 tokens per lane ----
            float x[4][2];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int col = nt * 8 + 2 * t4 + e;
                    x[nt][e] = ((d.vmask >> col) & 1u) ? (s[nt][e] + s[nt][e + 2]) * qk_scale : -INFINITY;
                }
            float mx = fmaxf(fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1])),
                             fmaxf(fmaxf(x[2][0], x[2][1]), fmaxf(x[3][0], x[3][1])));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mn = fmaxf(m0, mx);
            const float mu = (mn == -INFINITY) ? 0.f : mn;
            const float al = exp2f(m0 - mu);
            m0 = mn;
            const float eb = mu - 8.f;                 // weights scaled by 2^8
            float pr[4][2];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                pr[nt][0] = exp2f(x[nt][0] - eb);
                pr[nt][1] = exp2f(x[nt][1] - eb);
            }
            l0 = l0 * al + (((pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1])) +
                            ((pr[2][0] + pr[2][1]) + (pr[3][0] + pr[3][1])));
            if (!__all_sync(0xffffffffu, al == 1.f)) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    acc[nt][0] *= al; acc[nt][1] *= al; acc[nt][2] *= al; acc[nt][3] *= al;
                }
            }
            // ---- weights as A fragments: hi in row g4, lo in row g4 + 8 ----
            // logical k 4*t4 + i <-> tokens (2t4, 2t4+1, 8+2t4, 9+2t4)[i]
            // (+16 for registers 2 and 3), the token order of the S tiles
            uint32_t pa[4];
#pragma unroll
            for (int hk = 0; hk < 2; ++hk) {
                uint32_t h0, q0, h1, q1;
                split_e4m3x2(pr[2 * hk][0], pr[2 * hk][1], h0, q0);
                split_e4m3x2(pr[2 * hk + 1][0], pr[2 * hk + 1][1], h1, q1);
                pa[2 * hk] = h0 | (h1 << 16);
                pa[2 * hk + 1] = q0 | (q1 << 16);
            }
            // ---- acc += P V ----
            // A transposed ldmatrix of token rows gives lane (g4, t4) the
            // byte pairs (dims 2g4, 2g4+1) of tokens 2t4 and 2t4+1 of each
            // 8-token matrix; byte permutes regroup them into the even-dim
            // and odd-dim B fragments in the weights' token order.  Masked
            // token bytes are zeroed: the pool may hold NaN codes there.
            const uint32_t vb = smem_u32(vbuf);
            auto pv = [&](auto masked) {
                uint32_t mk0 = 0xffffffffu, mk1 = 0xffffffffu;
                if constexpr (decltype(masked)::value) {
                    mk0 = token_bytemask(d.vmask >> (2 * t4));
                    mk1 = token_bytemask(d.vmask >> (16 + 2 * t4));
                }
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                    uint32_t r0, r1, r2, r3;     // tokens 0-7, 8-15, 16-23, 24-31 of column chunk c
                    ldsm_x4_t(vb + lay.chunk_addr(rbV, tokV, c), r0, r1, r2, r3);
                    uint32_t e0 = __byte_perm(r0, r1, 0x6420), o0 = __byte_perm(r0, r1, 0x7531);
                    uint32_t e1 = __byte_perm(r2, r3, 0x6420), o1 = __byte_perm(r2, r3, 0x7531);
                    if constexpr (decltype(masked)::value) {
                        e0 &= mk0; o0 &= mk0; e1 &= mk1; o1 &= mk1;
                    }
                    mma_e4m3_16832<KV_E5M2>(acc[2 * c], pa, e0, e1);
                    mma_e4m3_16832<KV_E5M2>(acc[2 * c + 1], pa, o0, o1);
                }
            };
            if (d.vmask == 0xffffffffu) pv(std::false_type{});      // every token of the chunk is valid
            else pv(std::true_type{});
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (d.flags & SEG_END) {
                // hi + lo halves -> rows g4 (rows 8..15 are not stored)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    acc[nt][0] += acc[nt][2];
                    acc[nt][1] += acc[nt][3];
                }
                finish_segment(p, d, acc, m0, -INFINITY, l0, 0.f, lane, rows_valid, ri);
                if ((d.flags & GAP) && !(d.flags & DIRECT))
                    write_empty_partial(p, d.slot + 1, hg, hl, 0, rows_valid, lane);
            }
        }
    }

    // ---------------- transposed native-fp8 consumer (GQA groups of <= 4) ----------------
    // Keys are the M rows of the first product, S^T = K Q^T, with the 2G
    // query columns (the hi and the lo term of each head) as N = 8; the
    // second is O^T = V^T P^T with 16 head-dim rows per tile.  Each product
    // takes half the MMAs of the packed layout.  A lane owns one head (t4) in
    // both products, so its softmax statistics rescale its own accumulators.
    // P reaches the B layout of the second product through 256 bytes of
    // shared memory per warp.
    static __device__ void consumer_fp8t(const DecodeParams& p, const Plan& pl, int hg, int w,
                                         uint8_t* base, uint64_t* full, uint64_t* empty, uint64_t* qempty,
                                         const StageDesc* descs, uint8_t* pt) {
        const int lane = threadIdx.x & 31;
        const int g4 = lane >> 2, t4 = lane & 3;
        const int hl = w;                           // one warp per KV head
        const int S = p.stages;
        const KVLayout lay{p.box_bytes, static_cast<uint32_t>(p.rpb) * 128u,
                           static_cast<uint32_t>(p.HPC * p.rpb) * 128u, p.rpb};
        const int mi = lane >> 3, r8 = lane & 7;
        // K as A: matrix mi holds tokens (mi & 1) * 8 .. of the k-half mi >> 1
        const int tokA = (mi & 1) * 8 + r8;
        const uint32_t rbK0 = lay.row_base(tokA, hl), rbK1 = lay.row_base(tokA + 16, hl);
        // V transposed as A: matrix mi holds tokens 8 mi ..
        const int tokV = mi * 8 + r8;
        const uint32_t rbV = lay.row_base(tokV, hl);
        uint8_t* ptw = pt + w * 256;                // [8 columns][32 logical k] bytes
        const bool head_ok = t4 < p.G;
        const int head = hg * p.HPC * p.G + hl * p.G + t4;
        // logical k of this lane's hi/lo words: even g4 = 2m fills k 4m..4m+3,
        // odd g4 = 2m+1 fills k 16+4m..16+4m+3
        const int kblk = (g4 & 1) ? 16 + 4 * (g4 >> 1) : 4 * (g4 >> 1);

        float acc[8][4];
        uint32_t qb[KS8][2];
        float m = -INFINITY, l = 0.f;
        float qk_scale = p.qk_scale;

        for (int st = 0, k = pl.cs; k < pl.ce; ++k, ++st) {
            const int slot = st % S;
            if (!mbar_wait_bounded(&full[slot], (st / S) & 1u)) {
                if (lane == 0) raise_flag(p.err_flag, PA_ERRBIT_WAIT_TIMEOUT);
                return;
            }
            const StageDesc d = descs[slot];
            uint8_t* kbuf = base + slot * p.stage_bytes;
            uint8_t* vbuf = kbuf + p.kv_bytes;
            if (d.flags & SEG_START) {
                if (d.flags & QLOAD) {
                    qk_scale = p.qk_scale * load_q_fp8t(qb, base + p.q_off + d.qslot * p.q_slot_bytes, hl * p.G,
                                                         p.G, lane, p.q_tma, p.HPC * p.G);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&qempty[d.qslot]);
                }
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
                m = -INFINITY; l = 0.f;
            }
            // ---- S^T = K Q^T: tokens 0-15 and 16-31 x 8 query columns ----
            float s[2][4];
#pragma unroll
            for (int t = 0; t < 2; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
            const uint32_t kb = smem_u32(kbuf);
#pragma unroll
            for (int ks = 0; ks < KS8; ++ks) {
                uint32_t a[4], b[4];
                ldsm_x4(kb + lay.chunk_addr(rbK0, tokA, 2 * ks + (mi >> 1)), a[0], a[1], a[2], a[3]);
                ldsm_x4(kb + lay.chunk_addr(rbK1, tokA, 2 * ks + (mi >> 1)), b[0], b[1], b[2], b[3]);
                mma_fp8_16832<KV_E5M2, false>(s[0], a, qb[ks][0], qb[ks][1]);
                mma_fp8_16832<KV_E5M2, false>(s[1], b, qb[ks][0], qb[ks][1]);
            }
            // ---- online softmax of head t4 over its tokens g4, g4+8, 16+g4, 24+g4 ----
            float x[4];
            x[0] = s[0][0] + s[0][1];       // hi + lo columns of the head
            x[1] = s[0][2] + s[0][3];
            x[2] = s[1][0] + s[1][1];
            x[3] = s[1][2] + s[1][3];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int tok = (a & 1) * 8 + (a >> 1) * 16 + g4;
                x[a] = ((d.vmask >> tok) & 1u) ? x[a] * qk_scale : -INFINITY;
            }
            float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m, mx);
            const float mu = (mn == -INFINITY) ? 0.f : mn;
            const float al = exp2f(m - mu);
            m = mn;
            const float eb = mu - 8.f;                 // weights scaled by 2^8
            float pr[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) pr[a] = exp2f(x[a] - eb);
            l = l * al + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
            if (!__all_sync(0xffffffffu, al == 1.f)) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    acc[c][0] *= al; acc[c][1] *= al; acc[c][2] *= al; acc[c][3] *= al;
                }
            }
            // ---- P^T to the B layout through shared memory ----
            uint32_t h01, l01, h23, l23;
            split_e4m3x2(pr[0], pr[1], h01, l01);
            split_e4m3x2(pr[2], pr[3], h23, l23);
            const uint32_t myhi = h01 | (h23 << 16), mylo = l01 | (l23 << 16);   // bytes: tokens g4, g4+8, 16+g4, 24+g4
            const uint32_t ohi = __shfl_xor_sync(0xffffffffu, myhi, 4);         // partner g4 ^ 1
            const uint32_t olo = __shfl_xor_sync(0xffffffffu, mylo, 4);
            // even g4 = 2m: tokens (2m, 2m+1, 2m+8, 2m+9) = (own, partner, own, partner) of bytes 0, 1;
            // odd g4: tokens 16 + (2m, 2m+1, 2m+8, 2m+9) = (partner, own, partner, own) of bytes 2, 3
            const uint32_t sel = (g4 & 1) ? 0x3726u : 0x5140u;
            const uint32_t whi = __byte_perm(myhi, ohi, sel), wlo = __byte_perm(mylo, olo, sel);
            __syncwarp();                               // the previous chunk's reads are done
            *reinterpret_cast<uint32_t*>(ptw + (2 * t4) * 32 + kblk) = whi;
            *reinterpret_cast<uint32_t*>(ptw + (2 * t4 + 1) * 32 + kblk) = wlo;
            __syncwarp();
            const uint32_t pb0 = *reinterpret_cast<const uint32_t*>(ptw + g4 * 32 + 4 * t4);
            const uint32_t pb1 = *reinterpret_cast<const uint32_t*>(ptw + g4 * 32 + 16 + 4 * t4);
            // ---- O^T += V^T P^T: 8 tiles of 16 head-dim rows (dims 16c + 2r, 16c + 2r + 1) ----
            const uint32_t vb = smem_u32(vbuf);
            auto pv = [&](auto masked) {
                uint32_t mk0 = 0xffffffffu, mk1 = 0xffffffffu;
                if constexpr (decltype(masked)::value) {
                    mk0 = token_bytemask(d.vmask >> (2 * t4));
                    mk1 = token_bytemask(d.vmask >> (16 + 2 * t4));
                }
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                    uint32_t r0, r1, r2, r3;     // tokens 0-7, 8-15, 16-23, 24-31 of column chunk c
                    ldsm_x4_t(vb + lay.chunk_addr(rbV, tokV, c), r0, r1, r2, r3);
                    uint32_t a[4] = {__byte_perm(r0, r1, 0x6420), __byte_perm(r0, r1, 0x7531),
                                     __byte_perm(r2, r3, 0x6420), __byte_perm(r2, r3, 0x7531)};
                    if constexpr (decltype(masked)::value) {
                        a[0] &= mk0; a[1] &= mk0; a[2] &= mk1; a[3] &= mk1;
                    }
                    mma_fp8_16832<KV_E5M2, false>(acc[c], a, pb0, pb1);
                }
            };
            if (d.vmask == 0xffffffffu) pv(std::false_type{});
            else pv(std::true_type{});
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (d.flags & SEG_END) {
                float lt = l + __shfl_xor_sync(0xffffffffu, l, 4);
                lt += __shfl_xor_sync(0xffffffffu, lt, 8);
                lt += __shfl_xor_sync(0xffffffffu, lt, 16);
                const bool direct = (d.flags & DIRECT) != 0;
                if (direct || d.slot < p.max_slots) {
                    const float sc = direct ? (lt > 0.f ? p.v_scale / lt : 0.f) : p.v_scale;
                    if (head_ok) {
                        const size_t row = static_cast<size_t>(d.qrow0) * p.Hq + head;
                        QE* orow = static_cast<QE*>(p.out) + row * D;
                        float* prow = p.part_acc + (static_cast<size_t>(d.slot) * p.QL * p.Hq + head) * D;
#pragma unroll
                        for (int c = 0; c < D / 16; ++c) {
                            const float v0 = (acc[c][0] + acc[c][1]) * sc;    // dim 16c + 2 g4
                            const float v1 = (acc[c][2] + acc[c][3]) * sc;    // dim 16c + 2 g4 + 1
                            const int col = 16 * c + 2 * g4;
                            if (direct) {
                                store_pair(orow + col, v0, v1);
                            } else {
                                *reinterpret_cast<float2*>(prow + col) = make_float2(v0, v1);
                            }
                        }
                        if (!direct && g4 == 0)
                            p.part_ml[static_cast<size_t>(d.slot) * p.QL * p.Hq + head] = make_float2(m, lt);
                    }
                    if (!direct && (d.flags & GAP)) write_empty_partial(p, d.slot + 1, hg, hl, 0, p.G, lane);
                }
            }
        }
    }

    // The query as the B fragments of S^T = K Q^T: column g4 is the hi
    // (g4 even) or lo (g4 odd) e4m3 term of head g4 / 2 of the group, for
    // head dims 32ks + 4t4 .. +3 (register 0) and 16 more (register 1); heads
    // past the group are zero.  Returns 2^-e, the inverse of the tile scale.
    static __device__ __forceinline__ float load_q_fp8t(uint32_t (&qb)[KS8][2], const uint8_t* qbuf, int qrow_lo,
                                                        int G, int lane, int q_tma, int qrows) {
        const int g4 = lane >> 2, t4 = lane & 3;
        auto qaddr = [&](int r, int c) -> uint32_t {
            if (q_tma) {
                const int rr = (c >> 3) * qrows + r;
                return static_cast<uint32_t>(rr * 128 + (((c & 7) ^ (rr & 7)) << 4));
            }
            return static_cast<uint32_t>(r * D * 2 + c * 16);
        };
        const int h = g4 >> 1;
        const int row = qrow_lo + min(h, G - 1);
        auto load4 = [&](int ks, int hk, float (&f)[4]) {
            const int c = 4 * ks + 2 * hk + (t4 >> 1);
            const uint2 u = *reinterpret_cast<const uint2*>(qbuf + qaddr(row, c) + 8 * (t4 & 1));
            float2 f0, f1;
            if constexpr (QT::code == PA_F16) {
                f0 = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
                f1 = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
            } else {
                f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
                f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
            }
            f[0] = f0.x; f[1] = f0.y; f[2] = f1.x; f[3] = f1.y;
        };
        float mx = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS8; ++ks)
#pragma unroll
            for (int hk = 0; hk < 2; ++hk) {
                float f[4];
                load4(ks, hk, f);
                mx = fmaxf(mx, fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3]))));
            }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        int e = 0;
        if (mx > 0.f && mx <= 3.0e38f) {
            const int ex = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 127;   // floor(log2(mx))
            e = max(-60, min(60, 7 - ex));
        }
        const float sc = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
        const bool lo_term = (g4 & 1) != 0, pad = h >= G;
#pragma unroll
        for (int ks = 0; ks < KS8; ++ks)
#pragma unroll
            for (int hk = 0; hk < 2; ++hk) {
                float f[4];
                load4(ks, hk, f);
                const float a0 = f[0] * sc, a1 = f[1] * sc, a2 = f[2] * sc, a3 = f[3] * sc;
                uint32_t v01 = f32x2_to_e4m3x2(a0, a1), v23 = f32x2_to_e4m3x2(a2, a3);
                if (lo_term) {
                    const uint32_t f01 = e4m3x2_to_f16x2(v01), f23 = e4m3x2_to_f16x2(v23);
                    const float2 b01 = __half22float2(*reinterpret_cast<const __half2*>(&f01));
                    const float2 b23 = __half22float2(*reinterpret_cast<const __half2*>(&f23));
                    v01 = f32x2_to_e4m3x2(a0 - b01.x, a1 - b01.y);
                    v23 = f32x2_to_e4m3x2(a2 - b23.x, a3 - b23.y);
                }
                qb[ks][hk] = pad ? 0u : (v01 | (v23 << 16));
            }
        return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    }

    // The query tile as A fragments (m16n8k32 layout, head_dim in natural
    // order): row g4 < G holds e4m3(2^e q) and row g4 + 8 the e4m3 residual;
    // rows past the group are zero.  Returns 2^-e.
    static __device__ __forceinline__ float load_q_e4m3(uint32_t (&qa)[KS8][4], const uint8_t* qbuf,
                                                        int qrow_lo, int rows_valid, int lane, int q_tma,
                                                        int qrows) {
        const int g4 = lane >> 2, t4 = lane & 3;
        auto qaddr = [&](int r, int c) -> uint32_t {
            if (q_tma) {
                const int rr = (c >> 3) * qrows + r;
                return static_cast<uint32_t>(rr * 128 + (((c & 7) ^ (rr & 7)) << 4));
            }
            return static_cast<uint32_t>(r * D * 2 + c * 16);
        };
        const int row = qrow_lo + min(g4, rows_valid - 1);
        // dims 32ks + 16hk + 4t4 .. +3: 8 bytes of the query row
        auto load4 = [&](int ks, int hk, float (&f)[4]) {
            const int c = 4 * ks + 2 * hk + (t4 >> 1);
            const uint2 u = *reinterpret_cast<const uint2*>(qbuf + qaddr(row, c) + 8 * (t4 & 1));
            float2 f0, f1;
            if constexpr (QT::code == PA_F16) {
                f0 = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
                f1 = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
            } else {
                f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
                f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
            }
            f[0] = f0.x; f[1] = f0.y; f[2] = f1.x; f[3] = f1.y;
        };
        // largest magnitude over the group's rows (lanes past it repeat a valid row)
        float mx = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS8; ++ks)
#pragma unroll
            for (int hk = 0; hk < 2; ++hk) {
                float f[4];
                load4(ks, hk, f);
                mx = fmaxf(mx, fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3]))));
            }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        int e = 0;
        if (mx > 0.f && mx <= 3.0e38f) {
            const int ex = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 127;   // floor(log2(mx))
            e = max(-60, min(60, 7 - ex));
        }
        const float sc = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
        const bool pad = g4 >= rows_valid;
#pragma unroll
        for (int ks = 0; ks < KS8; ++ks)
#pragma unroll
            for (int hk = 0; hk < 2; ++hk) {
                float f[4];
                load4(ks, hk, f);
                const float a0 = f[0] * sc, a1 = f[1] * sc, a2 = f[2] * sc, a3 = f[3] * sc;
                const uint32_t h01 = f32x2_to_e4m3x2(a0, a1), h23 = f32x2_to_e4m3x2(a2, a3);
                const uint32_t f01 = e4m3x2_to_f16x2(h01), f23 = e4m3x2_to_f16x2(h23);
                const float2 b01 = __half22float2(*reinterpret_cast<const __half2*>(&f01));
                const float2 b23 = __half22float2(*reinterpret_cast<const __half2*>(&f23));
                const uint32_t l01 = f32x2_to_e4m3x2(a0 - b01.x, a1 - b01.y);
                const uint32_t l23 = f32x2_to_e4m3x2(a2 - b23.x, a3 - b23.y);
                qa[ks][2 * hk] = pad ? 0u : (h01 | (h23 << 16));
                qa[ks][2 * hk + 1] = pad ? 0u : (l01 | (l23 << 16));
            }
        return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    }

    // A fragments of this tile's query rows (16 x D) from the stage's query
    // copy; rows past the group are zero.
    static __device__ __forceinline__ void load_q_frags(uint32_t (&qa)[KS][4], const uint8_t* qbuf,
                                                        const DecodeParams& p, int hl, int mt,
                                                        int rows_valid, int lane) {
        const int g4 = lane >> 2, t4 = lane & 3;
        const int q_tma = p.q_tma;
        const int qrows = p.HPC * p.G * p.QL;       // rows of one 128-B column plane of the slot
        // byte offset of 16-byte column chunk c of query row r in the ring
        // slot: [column block][row][128 B] with the 128-B swizzle when the
        // rows came by tensor copy, plain row-major otherwise
        auto qaddr = [&](int r, int c) -> uint32_t {
            if (q_tma) {
                const int rr = (c >> 3) * qrows + r;
                return static_cast<uint32_t>(rr * 128 + (((c & 7) ^ (rr & 7)) << 4));
            }
            return static_cast<uint32_t>(r * D * 2 + c * 16);
        };
        if constexpr (!FP8) {
            const int mi = lane >> 3, r8 = lane & 7;
            int row = (mi & 1) * 8 + r8;
            if (row >= rows_valid) row = 0;
            const int srow = q_smem_row(p, hl, 16 * mt + row);
            const uint32_t qb = smem_u32(qbuf);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                ldsm_x4(qb + qaddr(srow, 2 * ks + (mi >> 1)), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
            }
        } else {
            // head_dim order inside a 16-wide k-step is permuted to match the
            // byte order of e4m3 key rows: logical k (2t, 2t+1, 2t+8, 2t+9)
            // holds physical dims (4t, 4t+1, 4t+2, 4t+3).
            const int r0 = q_smem_row(p, hl, 16 * mt + min(g4, rows_valid - 1));
            const int r1 = q_smem_row(p, hl, 16 * mt + min(g4 + 8, rows_valid - 1));
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int c = 2 * ks + (t4 >> 1), inner = 8 * (t4 & 1);
                const uint2 u0 = *reinterpret_cast<const uint2*>(qbuf + qaddr(r0, c) + inner);
                const uint2 u1 = *reinterpret_cast<const uint2*>(qbuf + qaddr(r1, c) + inner);
                qa[ks][0] = to_f16x2(u0.x);
                qa[ks][1] = to_f16x2(u1.x);
                qa[ks][2] = to_f16x2(u0.y);
                qa[ks][3] = to_f16x2(u1.y);
            }
        }
        if (g4 >= rows_valid) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) { qa[ks][0] = 0u; qa[ks][2] = 0u; }
        }
        if (g4 + 8 >= rows_valid) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) { qa[ks][1] = 0u; qa[ks][3] = 0u; }
        }
    }

    // ---------------- tcgen05 consumer (several query tokens per KV head) ----------------
    // HPC KV heads per CTA: each head's (query token, head) rows are a block
    // of um_rows rows (its rows padded to a multiple of 32) of the M = 128
    // tile, so every consumer warp owns rows.  Row r is tensor-memory lane r,
    // owned by thread r of the consumer warps 0-3.  Per chunk the MMA warp
    // computes S = Q K^T into one
    // of two S buffers in tensor memory; each row's thread masks (sequence
    // end, causal limit), exponentiates against a reference maximum and
    // writes its weights to a K-major P buffer in shared memory (two,
    // alternating); the MMA warp then adds P V into O (M x D fp32 in tensor
    // memory) with V read in place from the stage as an MN-major operand.
    // A chunk is 32 tokens of one or two heads, so one producer iteration
    // moves 16-32 KB of K and V.
    // The reference maximum moves only when a row's maximum passes it by more
    // than 2^8, and only then is that row of O rescaled (tcgen05.ld / st), so
    // acc, l and m of a partial all refer to it.  V rows of tokens outside the
    // chunk's valid mask are zeroed in shared memory first: the MMA reads
    // every row, and 0 x NaN is NaN.
    static __device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity));
    }

    static __device__ void consumer_um(const DecodeParams& p, const Plan& pl, int hg, int w, uint8_t* base,
                                       uint64_t* full, UmBars* ub, const StageDesc* descs) {
        const int lane = threadIdx.x & 31;
        const int R = w * 32 + lane;                      // tile row = tensor-memory lane
        const int hl = R / p.um_rows;                     // KV head of the CTA owning this row
        const int rr = R - hl * p.um_rows;                // row within that head's block
        const int rows = p.QL * p.G;
        const int jrow = rr / p.G;                        // query token of this row
        const int head = (hg * p.HPC + hl) * p.G + (rr - jrow * p.G);
        const bool row_in = hl < p.HPC && rr < rows;
        const uint32_t trow = ub->tmem + (static_cast<uint32_t>(w * 32) << 16);
        const uint32_t sspan = static_cast<uint32_t>(CT * p.HPC);   // columns of one S buffer
        const uint32_t ocol = 2u * sspan;                          // first column of O
        const int S = p.stages;
        // stage layout of the tcgen05 path: column plane dh of box b at (dh * nbox + b) * pbox
        const uint32_t pbox = static_cast<uint32_t>(p.HPC * p.rpb) * 128u;
        const KVLayout lay{pbox, static_cast<uint32_t>(p.rpb) * 128u,
                           static_cast<uint32_t>(CT / p.rpb) * pbox, p.rpb};
        uint8_t* pbuf0 = base + p.simtq_off;
        constexpr uint32_t FULLM = CT == 32 ? 0xffffffffu : ((1u << CT) - 1u);
        // P buffers start at zero: a head's buffer only ever gets its own
        // rows, so the other heads' rows contribute nothing to its P V
        for (uint32_t i = threadIdx.x; i < 2u * p.HPC * UM_PBUF / 16u; i += UM_M)
            reinterpret_cast<uint4*>(pbuf0)[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
        float m_ref = -INFINITY, l = 0.f;
        bool row_ok = false;
        int lim = -1;
        bool ok = true;
        for (int st = 0, k = pl.cs; k < pl.ce; ++k, ++st) {
            const int slot = st % S;
            if (!(ok = warp_wait(&full[slot], (st / S) & 1u))) break;
            const StageDesc d = descs[slot];
            uint8_t* vbuf = base + slot * p.stage_bytes + p.kv_bytes;
            if (d.flags & SEG_START) {
                const int qn = static_cast<int>(d.flags >> QCOUNT_SHIFT);
                row_ok = row_in && jrow < qn;
                lim = row_ok ? d.qpos0 + jrow : -1;
                m_ref = -INFINITY;
                l = 0.f;
            }
            if ((d.vmask & FULLM) != FULLM) {
                // V rows of tokens outside the valid mask -> 0, every head
                for (int i = R; i < CT * CPR * p.HPC; i += UM_M) {
                    const int t = i / (CPR * p.HPC), r2 = i - t * (CPR * p.HPC);
                    const int h2 = r2 / CPR, c = r2 - h2 * CPR;
                    if (!((d.vmask >> t) & 1u))
                        *reinterpret_cast<uint4*>(vbuf + lay.chunk_addr(lay.row_base(t, h2), t, c)) =
                            make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // ---- this row's scores: token t of the chunk sits in column
            // (t / rpb) * HPC * rpb + head * rpb + t % rpb of the S buffer ----
            if (!(ok = warp_wait(&ub->sfull[st & 1], (st >> 1) & 1u))) break;
            tc05_fence_after();
            float s[CT];
            {
                const uint32_t sb = trow + (st & 1) * sspan;
#pragma unroll
                for (int b8 = 0; b8 < CT / 8; ++b8) {
                    const int t0 = 8 * b8;
                    const int bx = t0 / p.rpb;
                    const uint32_t col = static_cast<uint32_t>((bx * p.HPC + (hl < p.HPC ? hl : 0)) * p.rpb +
                                                               (t0 - bx * p.rpb));
                    float v8[8];
                    tmem_ld8(sb + col, v8);
#pragma unroll
                    for (int i = 0; i < 8; ++i) s[t0 + i] = v8[i];
                }
                tmem_wait_ld();
            }
            float alpha = 1.f;
            bool resc = false;
            if (row_ok) {
                float mx = -INFINITY;
#pragma unroll
                for (int t = 0; t < CT; ++t) {
                    const bool keep = ((d.vmask >> t) & 1u) && d.tok0 + t <= lim;
                    s[t] = keep ? s[t] * p.qk_scale : -INFINITY;
                    mx = fmaxf(mx, s[t]);
                }
                if (mx > m_ref + 8.f) {       // also the first finite maximum (m_ref = -inf: O is zero)
                    if (m_ref != -INFINITY) {
                        alpha = exp2f(m_ref - mx);
                        resc = true;
                        l *= alpha;
                    }
                    m_ref = mx;
                }
                float sum = 0.f;
#pragma unroll
                for (int t = 0; t < CT; ++t) {
                    s[t] = m_ref == -INFINITY ? 0.f : ex2_approx(s[t] - m_ref);
                    sum += s[t];
                }
                l += sum;
            } else {
#pragma unroll
                for (int t = 0; t < CT; ++t) s[t] = 0.f;
            }
            // P buffers st % 2 are free once P V of chunk st - 2 is complete
            if (st >= 2 && !(ok = warp_wait(&ub->pvdone[st & 1], ((st >> 1) - 1) & 1u))) break;
            if (__any_sync(0xffffffffu, resc)) {
                // rescale this warp's rows of O: P V of chunk st - 1 must be complete
                if (!(ok = warp_wait(&ub->pvdone[(st - 1) & 1], ((st - 1) >> 1) & 1u))) break;
                tc05_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 16) {
                    float o[16];
                    tmem_ld16(trow + ocol + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) o[i] *= alpha;
                    tmem_st16(trow + ocol + c0, o);
                }
                tmem_wait_st();
            }
            // ---- P: row R of its head's buffer, CT / 8 core-matrix rows of 8 tokens ----
            if (row_in) {
                uint8_t* pb = pbuf0 + ((st & 1) * p.HPC + hl) * UM_PBUF;
#pragma unroll
                for (int kc = 0; kc < CT / 8; ++kc) {
                    const float* v = s + 8 * kc;
                    *reinterpret_cast<uint4*>(pb + (kc * (UM_M / 8) + (R >> 3)) * 128 + (R & 7) * 16) =
                        make_uint4(pack2(v[0], v[1], MMA_BF16), pack2(v[2], v[3], MMA_BF16),
                                   pack2(v[4], v[5], MMA_BF16), pack2(v[6], v[7], MMA_BF16));
                }
            }
            fence_proxy_async_smem();            // P and zeroed V rows visible to the tensor core
            tc05_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ub->pfull[st & 1]);
            if (d.flags & SEG_END) {
                if (!(ok = warp_wait(&ub->pvdone[st & 1], (st >> 1) & 1u))) break;
                tc05_fence_after();
                finish_segment_um(p, d, trow + ocol, row_ok, jrow, head, m_ref, l);
                tc05_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ub->ofree);
            }
        }
        if (!ok && lane == 0) raise_flag(p.err_flag, PA_ERRBIT_WAIT_TIMEOUT);
    }

    // End of a segment on the tcgen05 path: this thread's row of O (tensor
    // memory at `orow`), normalised into the output when the segment covers
    // the whole sequence, else the unnormalised partial (acc, m, l).
    static __device__ __forceinline__ void finish_segment_um(const DecodeParams& p, const StageDesc& d, uint32_t orow_t,
                                                             bool row_ok, int jrow, int head, float m, float l) {
        const bool direct = (d.flags & DIRECT) != 0;
        const bool store = row_ok && (direct || d.slot < p.max_slots);
        const float sc = direct ? (l > 0.f ? p.v_scale / l : 0.f) : p.v_scale;
        QE* orow = static_cast<QE*>(p.out) + (static_cast<size_t>(d.qrow0 + jrow) * p.Hq + head) * D;
        const size_t prow = (static_cast<size_t>(d.slot) * p.QL + jrow) * p.Hq + head;
        float* pacc = p.part_acc + prow * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
            float o[16];
            tmem_ld16(orow_t + c0, o);
            tmem_wait_ld();
            if (store) {
#pragma unroll
                for (int i = 0; i < 16; ++i) o[i] *= sc;
                if (direct) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + c0);
                    dst[0] = make_uint4(pack2(o[0], o[1], MMA_BF16), pack2(o[2], o[3], MMA_BF16),
                                        pack2(o[4], o[5], MMA_BF16), pack2(o[6], o[7], MMA_BF16));
                    dst[1] = make_uint4(pack2(o[8], o[9], MMA_BF16), pack2(o[10], o[11], MMA_BF16),
                                        pack2(o[12], o[13], MMA_BF16), pack2(o[14], o[15], MMA_BF16));
                } else {
                    float4* dst = reinterpret_cast<float4*>(pacc + c0);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                }
            }
        }
        if (store && !direct) p.part_ml[prow] = make_float2(m, l);
        if (row_ok && !direct && (d.flags & GAP) && d.slot + 1 < p.max_slots) {
            // the slot a range end meeting a partition end skips: an empty partial
            const size_t prow1 = prow + static_cast<size_t>(p.QL) * p.Hq;
            float4* z = reinterpret_cast<float4*>(p.part_acc + prow1 * D);
#pragma unroll 4
            for (int i = 0; i < D / 4; ++i) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            p.part_ml[prow1] = make_float2(-INFINITY, 0.f);
        }
    }

    // The MMA warp's issuing thread.  S of chunk st + 1 is issued before P V
    // of chunk st when its bytes have landed, so the scores of the next chunk
    // are ready when the consumers finish the current one; otherwise P V of
    // chunk st goes first and frees its stage without waiting for memory.
    //   S: with several KV heads per CTA one MMA per box of rpb tokens and
    //   K-step takes the box's rows of every head (N = HPC * rpb, rows 128 B
    //   apart); the products of one head's query rows with another head's keys
    //   land in columns nobody reads.  With one head, one MMA per 16 tokens.
    //   P V: per head, P of that head (its rows only, the rest zero) times
    //   its V, 16 tokens per MMA.
    static __device__ void mma_um(const DecodeParams& p, const Plan& pl, uint8_t* base, uint64_t* full,
                                  uint64_t* empty, uint64_t* qempty, UmBars* ub, const StageDesc* descs) {
        const int S = p.stages;
        const int HPC = p.HPC;
        const uint32_t tm = ub->tmem;
        const uint32_t sspan = static_cast<uint32_t>(CT * HPC);
        const uint32_t ocol = 2u * sspan;
        const int nbox = CT / p.rpb;                      // TMA boxes per chunk
        // Stage layout: column plane dh of box b at (dh * nbox + b) * pbox,
        // so a plane holds the chunk's rows (box, head, row) contiguously and
        // S = Q K^T takes one MMA per k-step with N = CT * HPC.
        const uint32_t pbox = static_cast<uint32_t>(HPC * p.rpb) * 128u;
        const uint32_t dhs = static_cast<uint32_t>(nbox) * pbox;             // 64-element column planes apart
        const uint32_t id_s = umma_idesc_f16(MMA_BF16, UM_M, CT * HPC, false, false);
        const uint32_t id_o = umma_idesc_f16(MMA_BF16, UM_M, D, false, true);
        // 8-token groups of one head's V rows: 1024 B apart inside a box of
        // 16 or more rows, one box (pbox) apart with 8-row boxes
        const uint32_t grp = p.rpb == 8 ? pbox : 1024u;
        const uint32_t pb0 = smem_u32(base + p.simtq_off);
        // byte offset of head h's 16-token group g in a stage's K or V buffer,
        // worked out once: a division per MMA on this single issuing thread
        // would stand between the consumers' P and the P V it waits for
        constexpr int NG = CT / 16;
        uint32_t toff[NG][4];
#pragma unroll
        for (int g = 0; g < NG; ++g)
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int t0 = 16 * g;
                toff[g][h] = static_cast<uint32_t>(t0 / p.rpb) * pbox +
                             static_cast<uint32_t>(h * p.rpb + t0 % p.rpb) * 128u;
            }
        bool ok = true;
        int q_cur = 0;          // query ring slot of the current segment (descriptors name it at its first chunk)
        // S of chunk st, its stage already landed
        auto issue_s_ready = [&](int st) {
            const int slot = st % S;
            const StageDesc d = descs[slot];
            if (d.flags & SEG_START) q_cur = d.qslot;
            const uint32_t qb = smem_u32(base + p.q_off + q_cur * p.q_slot_bytes);
            const uint32_t kb = smem_u32(base + slot * p.stage_bytes);
            const uint32_t sb = tm + (st & 1) * sspan;
            // S column (b * HPC + h) * rpb + r holds token b * rpb + r of head h
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t plane = static_cast<uint32_t>(kk >> 2), within = static_cast<uint32_t>(kk & 3) * 32u;
                umma_f16(sb, umma_desc(qb + plane * p.q_plane_bytes + within, 16u, 1024u, 2u),
                         umma_desc(kb + plane * dhs + within, 16u, 1024u, 2u), id_s, kk > 0);
            }
            umma_commit(&ub->sfull[st & 1]);
            if (d.flags & SEG_END) umma_commit(&qempty[q_cur]);       // the segment's query rows are read
        };
        auto issue_s = [&](int st) -> bool {
            const int slot = st % S;
            if (!mbar_wait_bounded(&full[slot], (st / S) & 1u)) return false;
            tc05_fence_after();
            issue_s_ready(st);
            return true;
        };
        const int n = pl.ce - pl.cs;
        int seg = 0;
        if (n > 0) ok = issue_s(0);
        for (int st = 0; st < n && ok; ++st) {
            const int slot = st % S;
            const StageDesc d = descs[slot];
            // S of the next chunk goes first when its data is already here:
            // P V of this chunk must not wait for the next chunk's bytes
            bool s_next = st + 1 >= n;
            if (!s_next && mbar_test_wait(&full[(st + 1) % S], ((st + 1) / S) & 1u)) {
                tc05_fence_after();
                issue_s_ready(st + 1);
                s_next = true;
            }
            if (!(ok = mbar_wait_bounded(&ub->pfull[st & 1], (st >> 1) & 1u))) break;
            const bool first = (d.flags & SEG_START) != 0;
            if (first && seg > 0 && !(ok = mbar_wait_bounded(&ub->ofree, (seg - 1) & 1u))) break;
            if (first) ++seg;
            tc05_fence_after();
            const uint32_t vb = smem_u32(base + slot * p.stage_bytes + p.kv_bytes);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                if (h >= HPC) break;
                const uint32_t pbh = pb0 + static_cast<uint32_t>((st & 1) * HPC + h) * UM_PBUF;
#pragma unroll
                for (int k16 = 0; k16 < NG; ++k16)
                    umma_f16(tm + ocol,
                             umma_desc(pbh + k16 * 2u * (UM_M / 8) * 128u, (UM_M / 8) * 128u, 128u, 0u),
                             umma_desc(vb + toff[k16][h], dhs, grp, 2u), id_o, !first || h > 0 || k16 > 0);
            }
            umma_commit(&ub->pvdone[st & 1]);
            umma_commit(&empty[slot]);                                 // K and V of the stage are read
            if (!s_next && !(ok = issue_s(st + 1))) break;
        }
        // nothing may still read shared or tensor memory when the CTA frees them
        umma_commit(&ub->fin);
        if (!mbar_wait_bounded(&ub->fin, 0u)) ok = false;
        if (!ok) raise_flag(p.err_flag, PA_ERRBIT_WAIT_TIMEOUT);
    }

    // ---------------- CUDA-core consumer ----------------
    // Lanes (t, half) = (lane & 15, lane >> 4) compute the dot products of
    // token t over half of head_dim for up to 16 query rows; for P*V each
    // lane owns D/32 consecutive columns.
    static __device__ void consumer_simt(const DecodeParams& p, const Plan& pl, int hg, int w,
                                         uint8_t* base, uint64_t* full, uint64_t* empty, uint64_t* qempty,
                                         const StageDesc* descs, float* qpriv) {
        constexpr int R = 16;
        constexpr int VE = 16 / KV::bytes;     // elements per 16-byte chunk
        constexpr int DPL = D / 32;            // columns per lane in P*V
        const int lane = threadIdx.x & 31;
        const int tq = lane & 15, half = lane >> 4;
        const int hl = w / p.MT, mt = w - hl * p.MT;
        const int nr = min(R, p.G - 16 * mt);
        const int S = p.stages;
        const KVLayout lay{p.box_bytes, static_cast<uint32_t>(p.rpb) * 128u,
                           static_cast<uint32_t>(p.HPC * p.rpb) * 128u, p.rpb};
        const int qrow_lo = hl * p.G + 16 * mt;
        const int out_h0 = hg * p.HPC * p.G + qrow_lo;
        float* qp = qpriv + static_cast<size_t>(w) * R * D;   // this warp's query rows, fp32

        float acc[R][DPL];
        float m[R], l[R];
        for (int st = 0, k = pl.cs; k < pl.ce; ++k, ++st) {
            const int slot = st % S;
            if (!mbar_wait_bounded(&full[slot], (st / S) & 1u)) {
                if (lane == 0) raise_flag(p.err_flag, PA_ERRBIT_WAIT_TIMEOUT);
                return;
            }
            const StageDesc d = descs[slot];
            const uint8_t* kbuf = base + slot * p.stage_bytes;
            const uint8_t* vbuf = kbuf + p.kv_bytes;
            if (d.flags & SEG_START) {
                if (d.flags & QLOAD) {
                    const QE* qbuf = reinterpret_cast<const QE*>(base + p.q_off + d.qslot * p.q_slot_bytes);
                    for (int e = lane; e < nr * D; e += 32)
                        qp[e] = to_float(qbuf[static_cast<size_t>(qrow_lo) * D + e]);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&qempty[d.qslot]);
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    m[r] = -INFINITY; l[r] = 0.f;
#pragma unroll
                    for (int c = 0; c < DPL; ++c) acc[r][c] = 0.f;
                }
                __syncwarp();
            }
            // ---- scores of token tq over half of head_dim ----
            float s[R];
#pragma unroll
            for (int r = 0; r < R; ++r) s[r] = 0.f;
            const uint32_t rbk = lay.row_base(tq, hl);
#pragma unroll 2
            for (int c = half * (CPR / 2); c < (half + 1) * (CPR / 2); ++c) {
                const uint4 raw = *reinterpret_cast<const uint4*>(kbuf + lay.chunk_addr(rbk, tq, c));
                float kf[VE];
                unpack16<KV>(raw, kf);
                const int d0 = c * VE;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (r < nr) {
                        const float* qr = qp + r * D + d0;
                        float a = s[r];
#pragma unroll
                        for (int e = 0; e < VE; ++e) a = fmaf(qr[e], kf[e], a);
                        s[r] = a;
                    }
                }
            }
            const bool valid = (d.vmask >> tq) & 1u;
            float p_[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (r < nr) {
                    float x = s[r] + __shfl_xor_sync(0xffffffffu, s[r], 16);
                    x = valid ? x * p.qk_scale : -INFINITY;
                    float cm = x;
                    cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 1));
                    cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 2));
                    cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 4));
                    cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 8));
                    const float mn = fmaxf(m[r], cm);
                    const float mu = (mn == -INFINITY) ? 0.f : mn;
                    const float al = exp2f(m[r] - mu);
                    m[r] = mn;
                    const float pv = exp2f(x - mu);
                    float cs = pv;
                    cs += __shfl_xor_sync(0xffffffffu, cs, 1);
                    cs += __shfl_xor_sync(0xffffffffu, cs, 2);
                    cs += __shfl_xor_sync(0xffffffffu, cs, 4);
                    cs += __shfl_xor_sync(0xffffffffu, cs, 8);
                    l[r] = l[r] * al + cs;
#pragma unroll
                    for (int c = 0; c < DPL; ++c) acc[r][c] *= al;
                    p_[r] = pv;
                }
            }
            // ---- acc += p V over the chunk's valid tokens ----
            const int cidx = (lane * DPL * KV::bytes) / 16;           // 16-byte chunk holding my columns
            const int cbyte = (lane * DPL * KV::bytes) % 16;
            for (int t = 0; t < CT; ++t) {
                if (!((d.vmask >> t) & 1u)) continue;
                const uint8_t* src = vbuf + lay.chunk_addr(lay.row_base(t, hl), t, cidx) + cbyte;
                float vf[DPL];
                load_cols<KV, DPL>(src, vf);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (r < nr) {
                        const float pt = __shfl_sync(0xffffffffu, p_[r], t);
#pragma unroll
                        for (int c = 0; c < DPL; ++c) acc[r][c] = fmaf(pt, vf[c], acc[r][c]);
                    }
                }
            }
            if (d.flags & SEG_END) {
                const int c0 = lane * DPL;
                if (d.flags & DIRECT) {
                    QE* o = static_cast<QE*>(p.out) + static_cast<size_t>(d.seq) * p.Hq * D;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        if (r < nr) {
                            const float inv = l[r] > 0.f ? p.v_scale / l[r] : 0.f;
                            QE* row = o + static_cast<size_t>(out_h0 + r) * D + c0;
#pragma unroll
                            for (int c = 0; c < DPL; ++c) row[c] = from_float<QE>(acc[r][c] * inv);
                        }
                    }
                } else if (d.slot < p.max_slots) {
                    float* pa_ = p.part_acc + static_cast<size_t>(d.slot) * p.Hq * D;
                    float2* ml = p.part_ml + static_cast<size_t>(d.slot) * p.Hq;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        if (r < nr) {
                            float* row = pa_ + static_cast<size_t>(out_h0 + r) * D + c0;
#pragma unroll
                            for (int c = 0; c < DPL; ++c) row[c] = acc[r][c] * p.v_scale;
                            if (lane == 0) ml[out_h0 + r] = make_float2(m[r], l[r]);
                        }
                    }
                    if (d.flags & GAP) write_empty_partial(p, d.slot + 1, hg, hl, mt, nr, lane);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
    }

    template <class K2>
    static __device__ __forceinline__ void unpack16(const uint4 raw, float (&f)[16 / K2::bytes]) {
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        if constexpr (K2::code == PA_F32) {
#pragma unroll
            for (int e = 0; e < 4; ++e) f[e] = __uint_as_float(w[e]);
        } else if constexpr (K2::code == PA_F16) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
                f[2 * e] = x.x; f[2 * e + 1] = x.y;
            }
        } else if constexpr (K2::code == PA_BF16) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
                f[2 * e] = x.x; f[2 * e + 1] = x.y;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t h01 = fp8x2_to_f16x2<K2>(w[e]), h23 = fp8x2_to_f16x2<K2>(w[e] >> 16);
                const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h01));
                const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h23));
                f[4 * e] = a.x; f[4 * e + 1] = a.y; f[4 * e + 2] = b.x; f[4 * e + 3] = b.y;
            }
        }
    }

    template <class K2, int N>
    static __device__ __forceinline__ void load_cols(const uint8_t* src, float (&f)[N]) {
#pragma unroll
        for (int c = 0; c < N; ++c) {
            if constexpr (K2::code == PA_F32) f[c] = reinterpret_cast<const float*>(src)[c];
            else if constexpr (K2::code == PA_F16) f[c] = __half2float(reinterpret_cast<const __half*>(src)[c]);
            else if constexpr (K2::code == PA_BF16) f[c] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(src)[c]);
            else if constexpr (K2::code == PA_FP8_E5M2) f[c] = e5m2_to_float(src[c]);
            else f[c] = fp8_to_float(src[c]);
        }
    }
};

template <class KV, class QT, int D, bool TC, int CT, bool MQ = false, bool T8 = false, bool UM = false>
__global__ void __launch_bounds__(MAX_WARPS * 32, 1)
pa_decode_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tq) {
    using K = DecodeKernel<KV, QT, D, TC, CT, MQ, T8, UM>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(base + p.bar_off);
    uint64_t* empty = full + MAX_STAGES;
    uint64_t* qempty = empty + MAX_STAGES;
    StageDesc* descs = reinterpret_cast<StageDesc*>(qempty + 2 * NQ);
    int2* scratch = reinterpret_cast<int2*>(descs + MAX_STAGES);
    int4* s_first = reinterpret_cast<int4*>(scratch + 32);
    int2* s_tot = reinterpret_cast<int2*>(s_first + 1);
    int* s_end = reinterpret_cast<int*>(s_tot + 1);
    UmBars* ub = reinterpret_cast<UmBars*>((reinterpret_cast<uintptr_t>(s_end + 1) + 15) & ~uintptr_t(15));

    // This kernel is launched as a programmatic dependent of the previous
    // kernel on the stream (typically the cache write): its CTAs may be
    // resident before that grid ends, and wait here until it has completed
    // and its writes are visible.  The merge kernel is in turn launched as a
    // programmatic dependent of this one once every CTA has passed the
    // trigger below: it becomes resident early, reads the merge list (made
    // visible by CTA 0 before its trigger) and then waits for this grid to
    // complete before reading partials.
    grid_dependency_wait();
    const int hg = blockIdx.x % p.NHG;
    const int range = blockIdx.x / p.NHG;
    Plan pl;
    make_plan(p, range, scratch, s_first, s_tot, s_end, pl);
    grid_dependents_launch();
    if (pl.cs >= pl.ce || pl.seq < 0) return;

    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        // on the tcgen05 path one MMA commit frees a stage or a query slot
        const uint32_t frees = UM ? 1u : static_cast<uint32_t>(p.NCW);
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], frees);
        }
        for (int s = 0; s < NQ; ++s) mbar_init(&qempty[s], frees);
        if constexpr (UM) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(&ub->sfull[b], 1);
                mbar_init(&ub->pfull[b], p.NCW);
                mbar_init(&ub->pvdone[b], 1);
            }
            mbar_init(&ub->ofree, p.NCW);
            mbar_init(&ub->fin, 1);
        }
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if constexpr (UM) {
        if (warp == 0) tmem_alloc<K::UM_TCOLS>(&ub->tmem);
        tc05_fence_before();
    }
    __syncthreads();
    if constexpr (UM) {
        tc05_fence_after();
        if (warp == p.NCW) {
            if ((threadIdx.x & 31) == 0) {
                prefetch_tensormap(&tk);
                prefetch_tensormap(&tv);
                prefetch_tensormap(&tq);
            }
            K::producer(p, pl, hg, base, full, empty, qempty, descs, &tk, &tv, &tq);
        } else if (warp == p.NCW + 1) {
            if ((threadIdx.x & 31) == 0) K::mma_um(p, pl, base, full, empty, qempty, ub, descs);
        } else if (warp < p.NCW) {
            K::consumer_um(p, pl, hg, warp, base, full, ub, descs);
        }
        // every role is done: the tensor memory goes back
        tc05_fence_before();
        __syncthreads();
        tc05_fence_after();
        if (warp == 0) tmem_dealloc<K::UM_TCOLS>(ub->tmem);
        return;
    }
    if (warp == p.NCW) {
        if ((threadIdx.x & 31) == 0) {
            prefetch_tensormap(&tk);
            prefetch_tensormap(&tv);
            if (p.q_tma) prefetch_tensormap(&tq);
        }
        K::producer(p, pl, hg, base, full, empty, qempty, descs, &tk, &tv, &tq);
    } else if (warp < p.NCW) {
        if constexpr (T8) {
            K::consumer_fp8t(p, pl, hg, warp, base, full, empty, qempty, descs, base + p.simtq_off);
        } else if constexpr (K::NATIVE8) {
            K::consumer_e4m3(p, pl, hg, warp, base, full, empty, qempty, descs);
        } else if constexpr (TC) {
            K::consumer_tc(p, pl, hg, warp, base, full, empty, qempty, descs);
        } else {
            K::consumer_simt(p, pl, hg, warp, base, full, empty, qempty, descs,
                             reinterpret_cast<float*>(base + p.simtq_off));
        }
    }
}

// ---------------------------------------------------------------------------
// log-sum-exp merge of the partials of sequences split across CTAs or
// partitions:  M = max m_k,  out = sum_k 2^(m_k - M) acc_k / sum_k 2^(m_k - M) l_k.
// One warp per (sequence, head); lanes own head_dim/32 consecutive columns.
// Partials of one sequence lie at slots range + first_unit + unit.
// ---------------------------------------------------------------------------
// Read-only vector loads as ordered inline PTX: a batch of them issues back
// to back instead of being sunk next to each use.
template <int DPL>
struct VecF;
template <> struct VecF<4> {
    static __device__ __forceinline__ void load(const float* p, float (&v)[4]) {
        asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]) : "l"(p));
    }
};
template <> struct VecF<2> {
    static __device__ __forceinline__ void load(const float* p, float (&v)[2]) {
        asm volatile("ld.global.nc.v2.f32 {%0, %1}, [%2];" : "=f"(v[0]), "=f"(v[1]) : "l"(p));
    }
};
__device__ __forceinline__ float2 ldg_f2(const float2* p) {
    float2 v;
    asm volatile("ld.global.nc.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
    return v;
}

constexpr int RED_THREADS = 128;     // 4 warps: one query head each
constexpr int RED_SPLIT_WARPS = 16;  // warps sharing one head's partials

// Threads of a merge CTA with WPI warps per (sequence, head).
__host__ __device__ constexpr int red_threads(int wpi) { return wpi == 1 ? RED_THREADS : 32 * wpi; }

// WPI warps per (sequence, head): 1 when sequences have a handful of
// partials (each warp of a 4-warp CTA takes one head), RED_SPLIT_WARPS when
// partitioned sequences have hundreds (the CTA's warps split one head's
// partials, so that a long sequence's reads are spread over 16 warps, and
// combine their results through shared memory).
template <typename OutT, int D, int WPI>
__global__ void __launch_bounds__(red_threads(WPI))
pa_reduce_kernel(const __grid_constant__ DecodeParams p) {
    constexpr int DPL = D / 32;
    // partials merged per batch, one per lane (8: fewer registers than 16,
    // measured faster whether a warp merges a handful or a share of hundreds)
    constexpr int NB = 8;
    constexpr int NW = red_threads(WPI) / 32;
    constexpr int HPB = NW / WPI;        // heads per CTA
    static_assert(WPI == 1 || HPB == 1, "split heads take the whole CTA");
    static_assert((WPI & (WPI - 1)) == 0, "the combine tree halves the warps");
    __shared__ float comb[WPI > 1 ? NW * 32 * (DPL + 2) : 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = warp % WPI;
    const int HG = cdiv_i(p.Hq, HPB);    // head groups of HPB heads
    const int per_seq = p.QL * HG;       // items of one split sequence: query tokens x head groups
    // The list and its length are final once every CTA of the main grid has
    // passed its trigger, which precedes this grid's start: the first item's
    // entry loads before the wait for the partials.
    int count = *reinterpret_cast<volatile int*>(&p.totals[2]);
    int4 e = __ldcg(&p.split_list[min(static_cast<int>(blockIdx.x) / per_seq, p.B - 1)]);
    grid_dependency_wait();
    for (int item = blockIdx.x;; item += gridDim.x) {
        if (item != static_cast<int>(blockIdx.x)) {
            // the count and this item's list entry load together
            count = *reinterpret_cast<volatile int*>(&p.totals[2]);
            e = __ldcg(&p.split_list[min(item / per_seq, p.B - 1)]);
        }
        if (item >= count * per_seq) break;
        const int jq = (item / HG) % p.QL;                // query token of the sequence
        const int h = (item % HG) * HPB + warp / WPI;
        if (WPI == 1 && h >= p.Hq) continue;
        int qrow = e.x;                                   // row of (sequence, token) in q / out
        if (p.q_start) {
            int a, qn;
            query_rows(p, e.x, a, qn);
            if (jq >= qn) continue;                       // the sequence has fewer query tokens
            qrow = a + jq;
        }
        // partial rows of this (token, head): slot * QL * Hq + jq * Hq + h
        const size_t prow0 = static_cast<size_t>(jq) * p.Hq + h;
        const size_t pstride = static_cast<size_t>(p.QL) * p.Hq;
        OutT* o = static_cast<OutT*>(p.out) + (static_cast<size_t>(qrow) * p.Hq + h) * D + lane * DPL;
        float num[DPL];
#pragma unroll
        for (int c = 0; c < DPL; ++c) num[c] = 0.f;
        float den = 0.f, M = -INFINITY;
        // Merge n <= NB partials; lane t names the slot of partial t.  The
        // (m, l) pair of each partial (one per lane) and every lane's
        // columns of all n partials are independent loads issued together.
        auto merge = [&](int n, int my_slot) {
            float v[NB][DPL];
#pragma unroll
            for (int t = 0; t < NB; ++t) {
                const int st = __shfl_sync(0xffffffffu, my_slot, t);
                if (t < n) {
                    VecF<DPL>::load(p.part_acc + (static_cast<size_t>(st) * pstride + prow0) * D + lane * DPL, v[t]);
                } else {
#pragma unroll
                    for (int c = 0; c < DPL; ++c) v[t][c] = 0.f;
                }
            }
            const float2 ml = lane < n ? ldg_f2(p.part_ml + static_cast<size_t>(my_slot) * pstride + prow0)
                                       : make_float2(-INFINITY, 0.f);
            float bm = ml.x;
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o2));
            const float Mn = fmaxf(M, bm);
            const float Mu = (Mn == -INFINITY) ? 0.f : Mn;
            const float sold = exp2f(M - Mu);
            const float w = lane < n ? exp2f(ml.x - Mu) : 0.f;
            float wl = w * ml.y;
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) wl += __shfl_xor_sync(0xffffffffu, wl, o2);
            den = den * sold + wl;
#pragma unroll
            for (int c = 0; c < DPL; ++c) num[c] *= sold;
#pragma unroll
            for (int t = 0; t < NB; ++t) {
                const float wt = __shfl_sync(0xffffffffu, w, t);
#pragma unroll
                for (int c = 0; c < DPL; ++c) num[c] = fmaf(wt, v[t][c], num[c]);
            }
            M = Mn;
        };
        if (e.w < 0) {
            // consecutive slots e.y .. e.y + e.z - 1, a contiguous share per warp
            const int per = cdiv_i(e.z, WPI), lo = min(e.z, sub * per), hi = min(e.z, lo + per);
            for (int b0 = lo; b0 < hi; b0 += NB) merge(min(NB, hi - b0), e.y + b0 + lane);
        } else if (sub == 0) {
            // Partials of sequence i lie at slot range + first_unit + unit for
            // every range holding chunks of the unit.
            const int S = e.y, U = e.z, L = e.w;
            const int C = p.totals[0], Ut = p.totals[1];
            const int nch = cdiv_i(L, p.ct), nu = n_units(L, p.PC, p.ct);
            const long long W = stream_weight(p, C, Ut);
            int cnt = 0, my_slot = 0;
            for (int u = 0; u < nu; ++u) {
                const int a = S + (p.PC > 0 ? u * p.PC : 0);
                const int b = p.PC > 0 ? min(a + p.PC, S + nch) : S + nch;
                const long long base = static_cast<long long>(p.WS) * (U + u + 1);
                const int r0 = range_of_pos(static_cast<long long>(p.WQ) * a + base, W, p.NR);
                const int r1 = range_of_pos(static_cast<long long>(p.WQ) * (b - 1) + base, W, p.NR);
                for (int r = r0; r <= r1; ++r) {
                    const int slot = r + U + u;
                    // ranges may be empty unless they are dense: skip those
                    // without a chunk of the unit
                    if (slot >= p.max_slots || (!dense_ranges(p, W) && !unit_in_range(r, a, b, base, W, p.NR, p.WQ)))
                        continue;
                    if ((cnt % NB) == lane) my_slot = slot;
                    if ((++cnt % NB) == 0) merge(NB, my_slot);
                }
            }
            if (cnt % NB) merge(cnt % NB, my_slot);
        }
        if constexpr (WPI > 1) {
            // pairwise tree: at stride s, warp w (a multiple of 2s) folds in
            // the running result of warp w + s
            float* mine = comb + (warp * 32 + lane) * (DPL + 2);
#pragma unroll
            for (int s = WPI / 2; s >= 1; s >>= 1) {
                if (sub >= s && sub < 2 * s) {
                    mine[0] = M; mine[1] = den;
#pragma unroll
                    for (int c = 0; c < DPL; ++c) mine[2 + c] = num[c];
                }
                __syncthreads();
                if (sub < s) {
                    const float* o2 = comb + ((warp + s) * 32 + lane) * (DPL + 2);
                    const float M2 = o2[0];
                    const float Mn = fmaxf(M, M2);
                    const float Mu = (Mn == -INFINITY) ? 0.f : Mn;
                    const float s1 = exp2f(M - Mu), s2 = exp2f(M2 - Mu);
                    den = den * s1 + o2[1] * s2;
#pragma unroll
                    for (int c = 0; c < DPL; ++c) num[c] = num[c] * s1 + o2[2 + c] * s2;
                    M = Mn;
                }
                __syncthreads();              // the buffer is reused by the next stride / item
            }
            if (sub != 0) continue;
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
        for (int c = 0; c < DPL; ++c) o[c] = from_float<OutT>(num[c] * inv);
    }
}

}  // namespace pa
