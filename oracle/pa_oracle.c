/*
 * pa_oracle.c -- plain, slow, single-threaded CPU oracle for paged decode
 * attention and its two companion cache operations.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path (the
 * CUDA library under paged_kv_cache_69_gb300/) never links, imports or calls
 * it, and this file shares no code, header, table or constant generator with
 * that path.
 *
 * Every function follows the plain definition the pages give, with no
 * blocking, fusion or reordering beyond it:
 *
 *  - Storage layout of one layer's pool: k_cache and v_cache are separate
 *    arrays of shape [num_blocks, block_size, num_kv_heads, head_dim]
 *    ("kv-cache-memory-core", section 2.2, the single-layer physical layout).
 *  - Logical token t of sequence i lives in physical block
 *    block_tables[i][t / block_size] at offset t % block_size
 *    ("vLLM intro part 2", section 3.2, the block_table worked example).
 *  - slot_mapping holds, for every new token, its absolute position in the
 *    pool, slot = block * block_size + offset (same page, section 3.2).
 *  - Query head h reads KV head h / (num_q_heads / num_kv_heads): consecutive
 *    query heads share one KV head ("kv-cache-memory-core", section 4.2, GQA
 *    figure).
 *  - Decode attention: gather the sequence's K and V through its block table
 *    into contiguous arrays, then s_t = scale * <q, k_t>,
 *    p = exp(s - max s) / sum exp(s - max s), out = sum_t p_t v_t
 *    ("vLLM intro part 2", section 4.2 key formulas; "kv-cache-memory-core",
 *    section 3, attention read pseudo-code).
 *  - fp8 KV: quantise on write, dequantise on read
 *    ("kv-cache-memory-core", section 4.4), E4M3 with 3 mantissa bits or
 *    E5M2 with 2 ("vLLM intro part 2", section 7, which names both).  The
 *    codecs below are written from the OCP FP8 definitions (E4M3: bias 7, no
 *    infinities, S.1111.111 is NaN, largest finite 448; E5M2: bias 15,
 *    IEEE-like infinities and NaNs, largest finite 57344); the per-tensor
 *    scale is an input.
 *  - copy_blocks: copy-on-write copies the whole content of a shared block
 *    into a fresh one before the write ("vLLM intro part 2", section 5;
 *    aibook "显存与 KV 缓存", the five copy-on-write steps).
 *
 * Arithmetic: every stored element is widened exactly to double; dot
 * products, the softmax and the weighted sum accumulate in double; results
 * are returned in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Element type codes, as the library's C interface numbers them. */
enum { PAO_F32 = 0, PAO_F16 = 1, PAO_BF16 = 2, PAO_FP8_E4M3 = 3, PAO_FP8_E5M2 = 4 };

static int pao_is_fp8(int dtype) { return dtype == PAO_FP8_E4M3 || dtype == PAO_FP8_E5M2; }

/* Error codes returned by the oracle (not device flags). */
enum { PAO_OK = 0, PAO_BAD_ARG = -1, PAO_BAD_BLOCK = -2 };

static size_t pao_elem_bytes(int dtype) {
    switch (dtype) {
        case PAO_F32: return 4;
        case PAO_F16: return 2;
        case PAO_BF16: return 2;
        case PAO_FP8_E4M3: return 1;
        case PAO_FP8_E5M2: return 1;
        default: return 0;
    }
}

/* ------------------------------------------------------------------------ */
/* Scalar codecs, each written from its format's definition.                */
/* ------------------------------------------------------------------------ */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double pao_f16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);            /* subnormal: m * 2^-14 * 2^-10 */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32 word. */
double pao_bf16_to_double(uint16_t b) {
    uint32_t w = (uint32_t)b << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits.
 * No infinities; exponent 1111 with fraction 111 is NaN; largest finite
 * value is 1.75 * 2^8 = 448; subnormals are m * 2^-9. */
double pao_e4m3_to_double(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xf;
    int m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) {
        v = ldexp((double)m, -9);
    } else {
        v = ldexp((double)(8 + m), e - 10);  /* (1 + m/8) * 2^(e-7) */
    }
    return sign ? -v : v;
}

/* Round a non-negative double to the nearest integer, ties to even. */
static double pao_round_half_even(double y) {
    double f = floor(y);
    double d = y - f;
    if (d > 0.5) return f + 1.0;
    if (d < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* float -> E4M3 with round-to-nearest-even and saturation to the largest
 * finite value (+-448); NaN maps to the canonical NaN code 0x7F. */
uint8_t pao_float_to_e4m3_satfinite(float x) {
    if (isnan(x)) return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7e;  /* includes +-inf */
    unsigned code;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: value = m * 2^-9, m in [0, 8]; m == 8 is the
         * smallest normal (code 0x08), which the code arithmetic reaches. */
        double m = pao_round_half_even(a * 512.0);
        code = (unsigned)m;
    } else {
        int ex;
        double fr = frexp(a, &ex);        /* a = fr * 2^ex, fr in [0.5, 1) */
        int E = ex - 1;                   /* a = (2*fr) * 2^E, 2*fr in [1,2) */
        double mant = fr * 16.0;          /* (1 + f/8) * 8 in [8, 16) */
        double r = pao_round_half_even(mant);  /* in [8, 16] */
        code = (unsigned)((E + 7) << 3) + (unsigned)(r - 8.0); /* r==16 carries */
    }
    if (code > 0x7e) code = 0x7e;
    return sign | (uint8_t)code;
}

/* OCP FP8 E5M2: 1 sign bit, 5 exponent bits (bias 15), 2 fraction bits,
 * IEEE-like: exponent 11111 is infinity (fraction 0) or NaN; largest finite
 * value 1.75 * 2^15 = 57344; subnormals are m * 2^-16. */
double pao_e5m2_to_double(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 2) & 0x1f;
    int m = b & 3;
    double v;
    if (e == 31) {
        if (m != 0) return NAN;
        v = INFINITY;
    } else if (e == 0) {
        v = ldexp((double)m, -16);
    } else {
        v = ldexp((double)(4 + m), e - 17);  /* (1 + m/4) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* float -> E5M2 with round-to-nearest-even and saturation of overflow and
 * infinities to the largest finite value (+-57344); NaN maps to 0x7F. */
uint8_t pao_float_to_e5m2_satfinite(float x) {
    if (isnan(x)) return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 57344.0) return sign | 0x7b;
    unsigned code;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: value = m * 2^-16, m in [0, 4]; m == 4 is the
         * smallest normal (code 0x04). */
        code = (unsigned)pao_round_half_even(a * 65536.0);
    } else {
        int ex;
        double fr = frexp(a, &ex);        /* a = fr * 2^ex, fr in [0.5, 1) */
        int E = ex - 1;
        double r = pao_round_half_even(fr * 8.0);   /* (1 + f/4) * 4 in [4, 8] */
        code = (unsigned)((E + 15) << 2) + (unsigned)(r - 4.0);   /* r == 8 carries */
    }
    if (code > 0x7b) code = 0x7b;
    return sign | (uint8_t)code;
}

static uint8_t pao_float_to_fp8(int dtype, float x) {
    return dtype == PAO_FP8_E5M2 ? pao_float_to_e5m2_satfinite(x) : pao_float_to_e4m3_satfinite(x);
}

/* Read element idx of a typed array as an exact double. */
static double pao_load(const void* base, int dtype, size_t idx) {
    switch (dtype) {
        case PAO_F32: return (double)((const float*)base)[idx];
        case PAO_F16: return pao_f16_to_double(((const uint16_t*)base)[idx]);
        case PAO_BF16: return pao_bf16_to_double(((const uint16_t*)base)[idx]);
        case PAO_FP8_E4M3: return pao_e4m3_to_double(((const uint8_t*)base)[idx]);
        case PAO_FP8_E5M2: return pao_e5m2_to_double(((const uint8_t*)base)[idx]);
        default: return NAN;
    }
}

/* Bulk helpers so tests can pin the codecs over whole code spaces. */
void pao_decode_array(double* out, const void* in, int dtype, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = pao_load(in, dtype, (size_t)i);
}

void pao_encode_e4m3_array(uint8_t* out, const float* in, int64_t n, float scale) {
    for (int64_t i = 0; i < n; ++i) out[i] = pao_float_to_e4m3_satfinite(in[i] / scale);
}

void pao_encode_e5m2_array(uint8_t* out, const float* in, int64_t n, float scale) {
    for (int64_t i = 0; i < n; ++i) out[i] = pao_float_to_e5m2_satfinite(in[i] / scale);
}

/* ------------------------------------------------------------------------ */
/* Gather: logical tokens [0, L) of one sequence and one KV head, read      */
/* through its block-table row into a contiguous [L, head_dim] array.       */
/* Returns PAO_BAD_BLOCK if a block id the sequence needs is out of range.  */
/* ------------------------------------------------------------------------ */
int pao_gather(double* out, const void* cache, int dtype, const int32_t* bt_row,
               int L, int g, int num_kv_heads, int head_dim, int block_size,
               int num_blocks, double elem_scale) {
    for (int t = 0; t < L; ++t) {
        int32_t blk = bt_row[t / block_size];
        int off = t % block_size;
        if (blk < 0 || blk >= num_blocks) return PAO_BAD_BLOCK;
        size_t row = (((size_t)blk * block_size + off) * num_kv_heads + g) * head_dim;
        for (int d = 0; d < head_dim; ++d) {
            double v = pao_load(cache, dtype, row + d);
            if (pao_is_fp8(dtype)) v *= elem_scale;
            out[(size_t)t * head_dim + d] = v;
        }
    }
    return PAO_OK;
}

/* ------------------------------------------------------------------------ */
/* Textbook softmax(q K^T * scale) V for one sequence i and query head h.   */
/* out_d receives head_dim doubles.  L == 0 yields zeros.                   */
/* ------------------------------------------------------------------------ */
int pao_attend_one(double* out_d, const void* q, int q_dtype,
                   const void* k_cache, const void* v_cache, int kv_dtype,
                   const int32_t* block_tables, int max_blocks_per_seq,
                   const int32_t* seq_lens, int num_seqs, int num_q_heads,
                   int num_kv_heads, int head_dim, int block_size, int num_blocks,
                   float scale, float k_scale, float v_scale, int i, int h) {
    if (i < 0 || i >= num_seqs || h < 0 || h >= num_q_heads) return PAO_BAD_ARG;
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return PAO_BAD_ARG;
    int G = num_q_heads / num_kv_heads;
    int g = h / G;
    int L = seq_lens[i];
    for (int d = 0; d < head_dim; ++d) out_d[d] = 0.0;
    if (L <= 0) return PAO_OK;
    if ((L + block_size - 1) / block_size > max_blocks_per_seq) return PAO_BAD_ARG;

    const int32_t* bt_row = block_tables + (size_t)i * max_blocks_per_seq;
    double* Kc = (double*)malloc((size_t)L * head_dim * sizeof(double));
    double* Vc = (double*)malloc((size_t)L * head_dim * sizeof(double));
    double* s = (double*)malloc((size_t)L * sizeof(double));
    double* qh = (double*)malloc((size_t)head_dim * sizeof(double));
    if (!Kc || !Vc || !s || !qh) {
        free(Kc); free(Vc); free(s); free(qh);
        return PAO_BAD_ARG;
    }
    int rc = pao_gather(Kc, k_cache, kv_dtype, bt_row, L, g, num_kv_heads, head_dim,
                        block_size, num_blocks, (double)k_scale);
    if (rc == PAO_OK)
        rc = pao_gather(Vc, v_cache, kv_dtype, bt_row, L, g, num_kv_heads, head_dim,
                        block_size, num_blocks, (double)v_scale);
    if (rc == PAO_OK) {
        size_t qrow = ((size_t)i * num_q_heads + h) * head_dim;
        for (int d = 0; d < head_dim; ++d) qh[d] = pao_load(q, q_dtype, qrow + d);
        /* logits */
        double mx = -INFINITY;
        for (int t = 0; t < L; ++t) {
            double acc = 0.0;
            for (int d = 0; d < head_dim; ++d) acc += qh[d] * Kc[(size_t)t * head_dim + d];
            s[t] = (double)scale * acc;
            if (s[t] > mx) mx = s[t];
        }
        /* softmax with the maximum subtracted */
        double Z = 0.0;
        for (int t = 0; t < L; ++t) {
            s[t] = exp(s[t] - mx);
            Z += s[t];
        }
        /* weighted sum of V rows */
        for (int t = 0; t < L; ++t) {
            double p = s[t] / Z;
            for (int d = 0; d < head_dim; ++d) out_d[d] += p * Vc[(size_t)t * head_dim + d];
        }
    }
    free(Kc); free(Vc); free(s); free(qh);
    return rc;
}

/* All sequences and heads: out is [num_seqs, num_q_heads, head_dim] doubles.
 * Returns the first non-zero status met (and keeps going). */
int pao_decode(double* out, const void* q, int q_dtype,
               const void* k_cache, const void* v_cache, int kv_dtype,
               const int32_t* block_tables, int max_blocks_per_seq,
               const int32_t* seq_lens, int num_seqs, int num_q_heads,
               int num_kv_heads, int head_dim, int block_size, int num_blocks,
               float scale, float k_scale, float v_scale) {
    int status = PAO_OK;
    for (int i = 0; i < num_seqs; ++i) {
        for (int h = 0; h < num_q_heads; ++h) {
            int rc = pao_attend_one(out + ((size_t)i * num_q_heads + h) * head_dim, q, q_dtype,
                                    k_cache, v_cache, kv_dtype, block_tables,
                                    max_blocks_per_seq, seq_lens, num_seqs, num_q_heads,
                                    num_kv_heads, head_dim, block_size, num_blocks,
                                    scale, k_scale, v_scale, i, h);
            if (rc != PAO_OK && status == PAO_OK) status = rc;
        }
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Cache write: token t's [num_kv_heads, head_dim] rows of key and value go */
/* to pool slot slot_mapping[t].  A negative slot is padding and is skipped; */
/* a slot at or past num_blocks * block_size is skipped and counted.        */
/* Same-type writes copy the element bytes; an fp8 cache stores             */
/* e4m3_satfinite(x / scale) with x widened exactly to float.               */
/* Returns the number of skipped out-of-range slots, or PAO_BAD_ARG.        */
/* ------------------------------------------------------------------------ */
static void pao_store(void* cache, int kv_dtype, size_t idx, const void* src,
                      int src_dtype, size_t sidx, float scale) {
    if (kv_dtype == src_dtype) {
        size_t e = pao_elem_bytes(kv_dtype);
        memcpy((char*)cache + idx * e, (const char*)src + sidx * e, e);
    } else {
        /* only fp8 caches accept another source type */
        float x = (float)pao_load(src, src_dtype, sidx);  /* exact widening */
        ((uint8_t*)cache)[idx] = pao_float_to_fp8(kv_dtype, x / scale);
    }
}

int pao_reshape_and_cache(void* k_cache, void* v_cache, int kv_dtype,
                          const void* key, const void* value, int src_dtype,
                          const int64_t* slot_mapping, int num_tokens,
                          int num_kv_heads, int head_dim, int block_size,
                          int num_blocks, float k_scale, float v_scale) {
    if (kv_dtype != src_dtype && !pao_is_fp8(kv_dtype)) return PAO_BAD_ARG;
    int skipped = 0;
    int64_t nslots = (int64_t)num_blocks * block_size;
    size_t row = (size_t)num_kv_heads * head_dim;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= nslots) { ++skipped; continue; }
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        size_t dst = ((size_t)blk * block_size + (size_t)off) * row;
        for (size_t e = 0; e < row; ++e) {
            pao_store(k_cache, kv_dtype, dst + e, key, src_dtype, (size_t)t * row + e, k_scale);
            pao_store(v_cache, kv_dtype, dst + e, value, src_dtype, (size_t)t * row + e, v_scale);
        }
    }
    return skipped;
}

/* ------------------------------------------------------------------------ */
/* Copy-on-write block copies: for each pair (src, dst) the whole K block   */
/* and V block src are copied onto block dst.  Pairs with an id outside     */
/* [0, num_blocks) are skipped and counted.  Returns the skipped count.     */
/* ------------------------------------------------------------------------ */
int pao_copy_blocks(void* k_cache, void* v_cache, int kv_dtype,
                    const int64_t* block_mapping, int num_pairs,
                    int num_kv_heads, int head_dim, int block_size, int num_blocks) {
    size_t bytes = (size_t)block_size * num_kv_heads * head_dim * pao_elem_bytes(kv_dtype);
    if (bytes == 0) return PAO_BAD_ARG;
    int skipped = 0;
    for (int p = 0; p < num_pairs; ++p) {
        int64_t src = block_mapping[2 * p], dst = block_mapping[2 * p + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) { ++skipped; continue; }
        memmove((char*)k_cache + (size_t)dst * bytes, (char*)k_cache + (size_t)src * bytes, bytes);
        memmove((char*)v_cache + (size_t)dst * bytes, (char*)v_cache + (size_t)src * bytes, bytes);
    }
    return skipped;
}
