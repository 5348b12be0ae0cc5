/*
 * pa_oracle.c -- CPU oracle for the paged-KV hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the tests, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py do.  It shares no code, header,
 * table or helper with the CUDA library.
 *
 * Every routine is the plain definition written out with loops, in the
 * order the pages give the steps, accumulating in double precision:
 *
 *   - slot translation: "分页 KV Cache" (ai-infra handbook), §块表与 slot
 *     mapping and the slot_mapping_for helper of its paged.py listing;
 *     "PagedAttention：分页内存管理" (mini-vllm step 12), §block_table
 *     translation formula.
 *   - write: "分页 KV Cache", paged.py PagedKVCache.write (row scatter, in
 *     index order).
 *   - swap: the xxqk.cn PagedAttention article, §显存不够时的调度 (evicted
 *     blocks go to CPU memory and come back).
 *   - block copy: "分页 KV Cache", exercise 2 answer (copy-on-write copies
 *     the old block's content into the new block); "KV cache：容量推导、分页与
 *     回收", kv_cache.py Sequence.append (allocate(copy of data)).
 *   - attention: "分页 KV Cache", paged.py paged_attention (gather the
 *     first seq_len tokens through the block table, repeat KV heads with
 *     repeat_interleave, scores = q.k * scale, causal mask
 *     tril(diagonal = seq_len - num_new), softmax, P.V).
 *   - quantized cache: "KV cache：容量推导、分页与回收" names a quantized
 *     cache (量化缓存) as something that changes the per-token size, with no
 *     method.  The reading taken here: FP8 E4M3 codes (the OCP 8-bit
 *     floating-point format: 1 sign, 4 exponent bits with bias 7, 3 mantissa
 *     bits, no infinities, S.1111.111 = NaN, largest finite 448) with one
 *     fp32 scale per written (token, KV head) row, scale = max|x| / 448
 *     (1 for an all-zero row), code = x / scale rounded to the nearest code,
 *     ties to the even code, values beyond 448 held at 448.  The division
 *     and the maximum are taken in fp32, the precision the GPU takes the
 *     same decisions in; the attention reads code value x scale exactly.
 *
 * Element types: 0 = fp32, 1 = bf16, 2 = fp16.  Inputs are decoded to double
 * exactly from their bit patterns; results are returned in double.  The
 * page's reference casts the softmax probabilities back to the query dtype
 * before P.V; this oracle keeps them in double (the exact value).
 *
 * Build: gcc -O2 -std=c11 -fopenmp -shared -fPIC (oracle/build.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- element decoding (IEEE 754 binary32 / bfloat16 / binary16) ---------- */

static double dec_f32(uint32_t bits) {
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* bfloat16 is the upper half of a binary32 with the same sign/exponent. */
static double dec_bf16(uint16_t bits) { return dec_f32((uint32_t)bits << 16); }

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double dec_f16(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
    else if (e == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp(1.0 + frac / 1024.0, e - 15);
    return sign ? -mag : mag;
}

static size_t elt_size(int dtype) { return dtype == 0 ? 4 : 2; }

static double load_elt(const void* base, int64_t i, int dtype) {
    if (dtype == 0) {
        uint32_t b;
        memcpy(&b, (const char*)base + 4 * i, 4);
        return dec_f32(b);
    }
    uint16_t h;
    memcpy(&h, (const char*)base + 2 * i, 2);
    return dtype == 1 ? dec_bf16(h) : dec_f16(h);
}

/* Decode n consecutive elements to double (used by tests to read buffers). */
void oracle_decode(const void* src, int64_t n, int dtype, double* dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = load_elt(src, i, dtype);
}

/* ---- slot translation ---------------------------------------------------- */

/* Position p lives in logical block p // block_size at offset p % block_size;
 * the block table maps the logical block to a physical one, and the slot is
 * physical_block * block_size + offset. */
int64_t oracle_slot(const int32_t* block_table, int64_t pos, int32_t block_size) {
    int64_t logical = pos / block_size;
    int64_t offset = pos % block_size;
    return (int64_t)block_table[logical] * block_size + offset;
}

/* One slot per new token: token i belongs to sequence seq_idx[i] (row of the
 * padded [num_seqs, max_blocks] table) at position positions[i].  A negative
 * position marks a padding token and yields slot -1. */
void oracle_slot_mapping(const int32_t* block_tables, int32_t max_blocks,
                         const int32_t* seq_idx, const int64_t* positions, int64_t n,
                         int32_t block_size, int64_t* slot_out) {
    for (int64_t i = 0; i < n; ++i) {
        if (positions[i] < 0) {
            slot_out[i] = -1;
            continue;
        }
        const int32_t* table = block_tables + (int64_t)seq_idx[i] * max_blocks;
        slot_out[i] = oracle_slot(table, positions[i], block_size);
    }
}

/* ---- write ---------------------------------------------------------------- */

/* The cache viewed as [num_blocks * block_size, row] rows; token i's row goes
 * to row slot_mapping[i], tokens taken in index order.  A negative slot is a
 * padding token and is skipped. */
void oracle_write_kv(const void* k, const void* v, const int64_t* slot_mapping, int64_t n,
                     void* k_cache, void* v_cache, int64_t row_bytes) {
    for (int64_t i = 0; i < n; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0) continue;
        memcpy((char*)k_cache + s * row_bytes, (const char*)k + i * row_bytes, (size_t)row_bytes);
        memcpy((char*)v_cache + s * row_bytes, (const char*)v + i * row_bytes, (size_t)row_bytes);
    }
}

/* ---- copy-on-write block copy -------------------------------------------- */

/* For every layer and every (src, dst) pair in order: the whole dst block of K
 * and of V receives the content of the src block. */
void oracle_copy_blocks(void* const* k_caches, void* const* v_caches, int32_t num_layers,
                        const int64_t* block_pairs, int32_t num_pairs, int64_t block_bytes) {
    for (int32_t l = 0; l < num_layers; ++l) {
        for (int32_t p = 0; p < num_pairs; ++p) {
            int64_t src = block_pairs[2 * p], dst = block_pairs[2 * p + 1];
            memcpy((char*)k_caches[l] + dst * block_bytes, (const char*)k_caches[l] + src * block_bytes,
                   (size_t)block_bytes);
            memcpy((char*)v_caches[l] + dst * block_bytes, (const char*)v_caches[l] + src * block_bytes,
                   (size_t)block_bytes);
        }
    }
}

/* Swap: for every layer and pair, block dst of the destination pool receives
 * block src of the source pool (K and V), the pools being different arrays
 * (device pool and host pool in either direction).  "xxqk.cn PagedAttention",
 * §显存不够时的调度: evicted blocks move to CPU memory and back. */
void oracle_swap_blocks(void* const* src_k, void* const* src_v, void* const* dst_k, void* const* dst_v,
                        int32_t num_layers, const int64_t* block_pairs, int32_t num_pairs, int64_t block_bytes) {
    for (int32_t l = 0; l < num_layers; ++l) {
        for (int32_t p = 0; p < num_pairs; ++p) {
            int64_t src = block_pairs[2 * p], dst = block_pairs[2 * p + 1];
            memcpy((char*)dst_k[l] + dst * block_bytes, (const char*)src_k[l] + src * block_bytes, (size_t)block_bytes);
            memcpy((char*)dst_v[l] + dst * block_bytes, (const char*)src_v[l] + src * block_bytes, (size_t)block_bytes);
        }
    }
}

/* ---- FP8 E4M3 codes ------------------------------------------------------- */

/* Value of a code, from the format's definition: exponent field e, mantissa
 * field m: normal (e > 0): (1 + m/8) 2^(e-7) = (8 + m) 2^(e-10); subnormal
 * (e = 0): (m/8) 2^-6 = m 2^-9; e = 15 with m = 7 is NaN. */
double oracle_e4m3_value(uint8_t c) {
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return s ? -v : v;
}

/* Nearest code to x (ties to the code with an even mantissa), |x| >= 448
 * held at +-448, NaN to 0x7F.  The 127 finite non-negative codes have
 * values that increase with the code, so the nearest one is found by
 * bisection for the last code whose value is <= |x|, then comparing it with
 * the next code. */
static double g_e4m3_table[127];
static int g_e4m3_ready = 0;

uint8_t oracle_e4m3_encode(float x) {
    if (!g_e4m3_ready) {
        for (int c = 0; c < 127; ++c) g_e4m3_table[c] = oracle_e4m3_value((uint8_t)c);
        g_e4m3_ready = 1;
    }
    if (isnan(x)) return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    int lo = 0, hi = 0x7E; /* table[lo] <= a < table[hi] */
    while (hi - lo > 1) {
        const int mid = (lo + hi) / 2;
        if (g_e4m3_table[mid] <= a) lo = mid;
        else hi = mid;
    }
    const double dl = a - g_e4m3_table[lo], dh = g_e4m3_table[hi] - a;
    uint8_t best;
    if (dl < dh) best = (uint8_t)lo;
    else if (dh < dl) best = (uint8_t)hi;
    else best = (uint8_t)((lo & 1) == 0 ? lo : hi);
    return sign | best;
}

void oracle_e4m3_encode_array(const float* x, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(const uint8_t* c, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_value(c[i]);
}

/* One row of row_len elements (src in `dtype`) -> codes and its scale. */
static void quant_row(const void* src, int64_t first, int32_t row_len, int dtype, uint8_t* codes, float* scale) {
    float amax = 0.0f;
    for (int32_t e = 0; e < row_len; ++e) {
        const float x = (float)load_elt(src, first + e, dtype);
        amax = fmaxf(amax, fabsf(x));
    }
    const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int32_t e = 0; e < row_len; ++e) {
        const float x = (float)load_elt(src, first + e, dtype);
        codes[e] = oracle_e4m3_encode(x / s);
    }
    *scale = s;
}

/* rows [n_rows, row_len] -> codes [n_rows, row_len], scales [n_rows] */
void oracle_quant_rows(const void* src, int dtype, int64_t n_rows, int32_t row_len, uint8_t* codes, float* scales) {
    for (int64_t r = 0; r < n_rows; ++r)
        quant_row(src, r * row_len, row_len, dtype, codes + r * row_len, scales + r);
}

/* The quantizing write: token i's K and V rows ([n, num_kv_heads, head_dim]
 * in `dtype`) go, one (token, KV head) row at a time, to codes at
 * (slot * num_kv_heads + h) * head_dim -- the cache layout -- and to the
 * scale at ((slot / block_size) * num_kv_heads + h) * block_size +
 * slot % block_size: scales are laid out [num_blocks, num_kv_heads,
 * block_size], so the scales of one KV head within one block are
 * contiguous.  Negative slots are skipped. */
void oracle_write_kv_fp8(const void* k, const void* v, int dtype, const int64_t* slot_mapping, int64_t n,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size, uint8_t* k_codes,
                         uint8_t* v_codes, float* k_scales, float* v_scales) {
    for (int64_t i = 0; i < n; ++i) {
        const int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        const int64_t blk = slot / block_size, off = slot % block_size;
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            const int64_t src = (i * num_kv_heads + h) * head_dim, dst = slot * num_kv_heads + h;
            const int64_t sc = (blk * num_kv_heads + h) * block_size + off;
            quant_row(k, src, head_dim, dtype, k_codes + dst * head_dim, k_scales + sc);
            quant_row(v, src, head_dim, dtype, v_codes + dst * head_dim, v_scales + sc);
        }
    }
}

/* ---- gather --------------------------------------------------------------- */

/* The first seq_len tokens of one sequence in logical order, as double
 * [seq_len, num_kv_heads, head_dim]: blocks = table[:ceil(seq_len/bs)], the
 * blocks' rows concatenated, truncated to seq_len. */
void oracle_gather(const void* cache, const int32_t* block_table, int32_t seq_len,
                   int32_t block_size, int32_t num_kv_heads, int32_t head_dim, int dtype,
                   double* out) {
    int64_t row = (int64_t)num_kv_heads * head_dim;
    int32_t nblk = (seq_len + block_size - 1) / block_size;
    int64_t t = 0;
    for (int32_t b = 0; b < nblk; ++b) {
        int64_t phys = block_table[b];
        for (int32_t o = 0; o < block_size && t < seq_len; ++o, ++t) {
            int64_t src_row = phys * block_size + o;
            for (int64_t e = 0; e < row; ++e) out[t * row + e] = load_elt(cache, src_row * row + e, dtype);
        }
    }
}

/* ---- attention ------------------------------------------------------------ */

/* One request's rows, from its K and V gathered as double [seq_len, num_kv_heads, head_dim]. */
static void attend_request(double* out, const void* q, int q_dtype, const double* k, const double* v,
                           int32_t seq_len, int32_t start, int32_t num_new, int32_t num_heads, int32_t num_kv_heads,
                           int32_t head_dim, double sc, int causal) {
    const int32_t rep = num_heads / num_kv_heads;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    double* p = (double*)malloc(sizeof(double) * (size_t)seq_len);
    double* qv = (double*)malloc(sizeof(double) * (size_t)head_dim);
    for (int32_t j = 0; j < num_new; ++j) {
        const int64_t qrow = start + j;
        const int64_t pos = (int64_t)seq_len - num_new + j;
        const int32_t visible = causal ? (int32_t)(pos + 1) : seq_len;
        for (int32_t h = 0; h < num_heads; ++h) {
            const int32_t kvh = h / rep;
            for (int32_t d = 0; d < head_dim; ++d) qv[d] = load_elt(q, (qrow * num_heads + h) * head_dim + d, q_dtype);
            /* scores over the visible keys */
            double m = -INFINITY;
            for (int32_t s = 0; s < visible; ++s) {
                double dot = 0.0;
                for (int32_t d = 0; d < head_dim; ++d) dot += qv[d] * k[s * row + (int64_t)kvh * head_dim + d];
                p[s] = dot * sc;
                if (p[s] > m) m = p[s];
            }
            /* softmax */
            double denom = 0.0;
            for (int32_t s = 0; s < visible; ++s) {
                p[s] = exp(p[s] - m);
                denom += p[s];
            }
            /* P . V */
            double* o = out + (qrow * num_heads + h) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d) {
                double acc = 0.0;
                for (int32_t s = 0; s < visible; ++s) acc += p[s] * v[s * row + (int64_t)kvh * head_dim + d];
                o[d] = acc / denom;
            }
        }
    }
    free(p);
    free(qv);
}

/*
 * Varlen paged attention, request by request:
 *   q, out:           [total_q, num_heads, head_dim]  (q in `dtype`, out double)
 *   k_cache, v_cache: [num_blocks, block_size, num_kv_heads, head_dim]
 *   block_tables:     [num_seqs, max_blocks] int32
 *   seq_lens:         [num_seqs]  total context after this step
 *   query_start_loc:  [num_seqs + 1]  request i owns q rows [qsl[i], qsl[i+1])
 * New token j of request i sits at position seq_len - num_new + j.  With
 * causal != 0 it sees positions <= that; with causal == 0 it sees all seq_len.
 * Query head h reads KV head h / (num_heads / num_kv_heads).
 * seq_select (may be NULL): only requests with seq_select[i] != 0 are
 * computed; the rows of the others are left untouched.
 */
void oracle_paged_attention(double* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int32_t max_blocks,
                            const int32_t* seq_lens, const int32_t* query_start_loc,
                            int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                            int32_t head_dim, int32_t block_size, float scale, int causal,
                            int dtype, const uint8_t* seq_select, int num_threads) {
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int32_t i = 0; i < num_seqs; ++i) {
        if (seq_select && !seq_select[i]) continue;
        const int32_t seq_len = seq_lens[i];
        const int32_t start = query_start_loc[i], num_new = query_start_loc[i + 1] - start;
        if (seq_len <= 0 || num_new <= 0) continue;
        const int32_t* table = block_tables + (int64_t)i * max_blocks;
        const int64_t row = (int64_t)num_kv_heads * head_dim;
        double* k = (double*)malloc(sizeof(double) * (size_t)(seq_len * row));
        double* v = (double*)malloc(sizeof(double) * (size_t)(seq_len * row));
        oracle_gather(k_cache, table, seq_len, block_size, num_kv_heads, head_dim, dtype, k);
        oracle_gather(v_cache, table, seq_len, block_size, num_kv_heads, head_dim, dtype, v);
        attend_request(out, q, dtype, k, v, seq_len, start, num_new, num_heads, num_kv_heads, head_dim,
                       (double)scale, causal);
        free(k);
        free(v);
    }
}

/* The same over a quantized cache: K and V codes [num_blocks, block_size,
 * num_kv_heads, head_dim] with scales [num_blocks, num_kv_heads, block_size];
 * a key or value element reads code value x its row's scale (exact in
 * double); q (and so the output's element type) is `q_dtype`. */
void oracle_paged_attention_fp8(double* out, const void* q, int q_dtype, const uint8_t* k_codes,
                                const uint8_t* v_codes, const float* k_scales, const float* v_scales,
                                const int32_t* block_tables, int32_t max_blocks, const int32_t* seq_lens,
                                const int32_t* query_start_loc, int32_t num_seqs, int32_t num_heads,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size, float scale,
                                int causal, int num_threads) {
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int32_t i = 0; i < num_seqs; ++i) {
        const int32_t seq_len = seq_lens[i];
        const int32_t start = query_start_loc[i], num_new = query_start_loc[i + 1] - start;
        if (seq_len <= 0 || num_new <= 0) continue;
        const int32_t* table = block_tables + (int64_t)i * max_blocks;
        const int64_t row = (int64_t)num_kv_heads * head_dim;
        double* k = (double*)malloc(sizeof(double) * (size_t)(seq_len * row));
        double* v = (double*)malloc(sizeof(double) * (size_t)(seq_len * row));
        for (int32_t t = 0; t < seq_len; ++t) {
            const int64_t blk = table[t / block_size], off = t % block_size;
            const int64_t slot = blk * block_size + off;
            for (int32_t h = 0; h < num_kv_heads; ++h) {
                const int64_t r = slot * num_kv_heads + h;
                const int64_t sc = (blk * num_kv_heads + h) * block_size + off;
                for (int32_t d = 0; d < head_dim; ++d) {
                    k[t * row + (int64_t)h * head_dim + d] = oracle_e4m3_value(k_codes[r * head_dim + d]) * (double)k_scales[sc];
                    v[t * row + (int64_t)h * head_dim + d] = oracle_e4m3_value(v_codes[r * head_dim + d]) * (double)v_scales[sc];
                }
            }
        }
        attend_request(out, q, q_dtype, k, v, seq_len, start, num_new, num_heads, num_kv_heads, head_dim,
                       (double)scale, causal);
        free(k);
        free(v);
    }
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

size_t oracle_elt_size(int dtype) { return elt_size(dtype); }
