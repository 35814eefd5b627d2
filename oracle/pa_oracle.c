/*
 * pa_oracle.c -- plain, slow fp64 CPU reference for PagedAttention V2 single-query decode
 * over a block-paged KV cache, and for the slot-mapping cache writer.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's CPU baseline
 * call it; the product library never does.  It shares no code, header, table or constant
 * with the CUDA path.
 *
 * Sources (page title, then section/symbol):
 *   "paged_attention_v2_pytorch.py"  paged_attention_v2_pytorch: unused-slot init, empty
 *       sequences, the paged K/V gather, k_scale/v_scale, GQA view, ALiBi with absolute
 *       positions, per-partition max / exp-sum / weighted V, and the phase-2 combine.
 *   "paged_attention_v2_triton.py"   _paged_attn_v2_reduce_kernel: the same phase-2 formula
 *       (global max, weights exp(m_p - g) * l_p normalised by their sum).
 *   "paged_attn.py"                  split_kv_cache (x = 16 / element size and the two
 *       cache views), write_to_paged_cache (reshape_and_cache by slot).
 *
 * Readings where the pages are silent or inconsistent:
 *   - tmp_output holds the partition-NORMALISED output (sum_t e_t v_t / l_p).  The pages'
 *     PyTorch phase 1 stores the un-normalised sum while its phase 2 and the Triton reduce
 *     weight by l_p; only the normalised reading makes that phase 2 a correct
 *     log-sum-exp combine (a one-partition sequence then returns softmax(s) V).
 *   - head h reads kv head h / (H / Hk)   (the [kv_h, gqa, 1, d] view of the query).
 *   - ALiBi adds slope[h] * t with t the absolute position 0 .. L-1.
 *   - k_scale and v_scale always multiply the decoded cache values.
 *   - per-kv-head scales (an extension: the pages pass one float each): with arrays
 *     k_scales[Hk], v_scales[Hk] the keys and values of kv head j are multiplied by
 *     k_scales[j] and v_scales[j] instead, and the writer divides head j's rows by them.
 *   - fp8 cache bytes are OCP e4m3fn codes (bias 7, subnormals, 0x7F/0xFF NaN, no inf).
 *   - writer: fp16/bf16 caches get a bitwise copy; an fp8 cache gets
 *     RNE-satfinite-e4m3( (float)x / k_scale ) with the division in IEEE binary32.
 *   - a negative slot means "skip this token".
 *   - partitions p >= ceil(L / partition_size) keep max_logits = -inf, exp_sums = 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* element formats understood by the oracle */
enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_F32 = 2, ORC_E4M3 = 3 };

/* ---- decoding, written from the format definitions ---------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_dec_f16(uint16_t h) {
    int sign = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-10 * 2^-14 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1.0 + m / 1024.0, e - 15);
    return sign ? -v : v;
}

/* bfloat16: the upper half of binary32 -- 1 sign, 8 exponent bits (bias 127), 7 fraction. */
double orc_dec_bf16(uint16_t b) {
    int sign = (b >> 15) & 1, e = (b >> 7) & 0xff, m = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133); /* subnormal: m * 2^-7 * 2^-126 */
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1.0 + m / 128.0, e - 127);
    return sign ? -v : v;
}

/* OCP 8-bit e4m3fn: 1 sign, 4 exponent bits (bias 7), 3 fraction bits; exponent 15 with
 * fraction 7 is NaN; there is no infinity. */
double orc_dec_e4m3(uint8_t c) {
    int sign = (c >> 7) & 1, e = (c >> 3) & 0xf, m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9); /* subnormal: m * 2^-3 * 2^-6 */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

static double dec_elem(const void* base, int64_t idx, int fmt) {
    switch (fmt) {
        case ORC_F16: return orc_dec_f16(((const uint16_t*)base)[idx]);
        case ORC_BF16: return orc_dec_bf16(((const uint16_t*)base)[idx]);
        case ORC_F32: return (double)((const float*)base)[idx];
        case ORC_E4M3: return orc_dec_e4m3(((const uint8_t*)base)[idx]);
    }
    return NAN;
}

static int elem_bytes(int fmt) { return fmt == ORC_E4M3 ? 1 : (fmt == ORC_F32 ? 4 : 2); }

/* ---- encoding to e4m3fn (writer), from the format definition ------------------------- */

/* Round-to-nearest-even onto the e4m3fn grid, saturating finite values (and infinities)
 * to +-448, NaN to NaN (0x7F with the input's sign bit). */
uint8_t orc_enc_e4m3(float xf) {
    double x = (double)xf;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x))
        return (uint8_t)(sign | 0x7F);
    double a = fabs(x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E); /* 1.75 * 2^8, the largest finite value */
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: grid step 2^-9; q == 8 lands on the smallest normal (code 8) */
        double q = nearbyint(a / ldexp(1.0, -9));
        return (uint8_t)(sign | (uint8_t)q);
    }
    int e;
    frexp(a, &e);          /* a = f * 2^e with f in [0.5, 1) */
    e -= 1;                /* a in [2^e, 2^(e+1)) */
    double step = ldexp(1.0, e - 3);
    double q = nearbyint(a / step); /* in [8, 16] */
    if (q == 16.0) {
        q = 8.0;
        e += 1;
    }
    if (e + 7 > 15 || (e + 7 == 15 && q - 8 > 6)) /* rounding past 448 (cannot happen below 448) */
        return (uint8_t)(sign | 0x7E);
    return (uint8_t)(sign | ((e + 7) << 3) | (int)(q - 8.0));
}

/* ---- decode attention ---------------------------------------------------------------- */

typedef struct {
    const void* query;
    int q_fmt;
    const void* key_cache;
    const void* value_cache;
    int kv_fmt;
    int S, H, Hk, d, bs;
    const int32_t* block_tables;
    int max_blocks_per_seq;
    const int32_t* seq_lens;
    double scale;
    const float* alibi;
    double k_scale, v_scale;
    const float* k_scales; /* [Hk] or NULL: per-kv-head scales replace k_scale */
    const float* v_scales; /* [Hk] or NULL */
    int part;  /* partition size in tokens */
    int Pmax;
} orc_args;

/* key_cache[b][kvh][i / x][o][i % x] */
static double k_at(const orc_args* a, int64_t b, int kvh, int i, int o) {
    int x = 16 / elem_bytes(a->kv_fmt);
    int64_t idx = ((((b * a->Hk + kvh) * (a->d / x) + i / x) * a->bs + o) * x) + i % x;
    return dec_elem(a->key_cache, idx, a->kv_fmt) * (a->k_scales ? (double)a->k_scales[kvh] : a->k_scale);
}

/* value_cache[b][kvh][i][o] */
static double v_at(const orc_args* a, int64_t b, int kvh, int i, int o) {
    int64_t idx = ((b * a->Hk + kvh) * a->d + i) * (int64_t)a->bs + o;
    return dec_elem(a->value_cache, idx, a->kv_fmt) * (a->v_scales ? (double)a->v_scales[kvh] : a->v_scale);
}

/* One (sequence, query head).  Outputs: out[d] (phase 2 of the partitioned pass),
 * out1[d] (one softmax over the whole sequence), ml[Pmax], es[Pmax], tmp[Pmax*d]. */
static void decode_one(const orc_args* a, int s, int h, double* out, double* out1,
                       double* ml, double* es, double* tmp) {
    const int d = a->d;
    for (int p = 0; p < a->Pmax; ++p) {
        ml[p] = -INFINITY;
        es[p] = 0.0;
        for (int i = 0; i < d; ++i) tmp[(int64_t)p * d + i] = 0.0;
    }
    for (int i = 0; i < d; ++i) out[i] = out1[i] = 0.0;
    const int L = a->seq_lens[s];
    if (L <= 0)
        return; /* empty sequence: zero output, statistics untouched */

    const int G = a->H / a->Hk;
    const int kvh = h / G;
    double* q = (double*)malloc(sizeof(double) * d);
    double* sc = (double*)malloc(sizeof(double) * L);
    for (int i = 0; i < d; ++i) q[i] = dec_elem(a->query, ((int64_t)s * a->H + h) * d + i, a->q_fmt);

    /* scores s_t = scale * <q, k_t> + slope_h * t */
    for (int t = 0; t < L; ++t) {
        int64_t b = a->block_tables[(int64_t)s * a->max_blocks_per_seq + t / a->bs];
        int o = t % a->bs;
        double dot = 0.0;
        for (int i = 0; i < d; ++i) dot += q[i] * k_at(a, b, kvh, i, o);
        sc[t] = a->scale * dot + (a->alibi ? (double)a->alibi[h] * (double)t : 0.0);
    }

    /* phase 1: per-partition max, exp-sum and normalised weighted V */
    const int P = (int)(((int64_t)L + a->part - 1) / a->part);
    for (int p = 0; p < P; ++p) {
        int t0 = p * a->part, t1 = (int64_t)t0 + a->part < L ? t0 + a->part : L;
        double m = -INFINITY;
        for (int t = t0; t < t1; ++t) m = sc[t] > m ? sc[t] : m;
        double l = 0.0;
        for (int t = t0; t < t1; ++t) l += exp(sc[t] - m);
        double* tp = tmp + (int64_t)p * d;
        for (int t = t0; t < t1; ++t) {
            double e = exp(sc[t] - m);
            int64_t b = a->block_tables[(int64_t)s * a->max_blocks_per_seq + t / a->bs];
            int o = t % a->bs;
            for (int i = 0; i < d; ++i) tp[i] += e * v_at(a, b, kvh, i, o);
        }
        for (int i = 0; i < d; ++i) tp[i] /= l;
        ml[p] = m;
        es[p] = l;
    }

    /* phase 2: g = max_p m_p, w_p = exp(m_p - g) * l_p, out = sum_p w_p tmp_p / sum_p w_p */
    double g = -INFINITY;
    for (int p = 0; p < P; ++p) g = ml[p] > g ? ml[p] : g;
    double W = 0.0;
    for (int p = 0; p < P; ++p) W += exp(ml[p] - g) * es[p];
    for (int p = 0; p < P; ++p) {
        double w = exp(ml[p] - g) * es[p] / W;
        for (int i = 0; i < d; ++i) out[i] += w * tmp[(int64_t)p * d + i];
    }

    /* one pass: softmax over all L tokens, times V */
    double M = -INFINITY;
    for (int t = 0; t < L; ++t) M = sc[t] > M ? sc[t] : M;
    double Z = 0.0;
    for (int t = 0; t < L; ++t) Z += exp(sc[t] - M);
    for (int t = 0; t < L; ++t) {
        double e = exp(sc[t] - M) / Z;
        int64_t b = a->block_tables[(int64_t)s * a->max_blocks_per_seq + t / a->bs];
        int o = t % a->bs;
        for (int i = 0; i < d; ++i) out1[i] += e * v_at(a, b, kvh, i, o);
    }
    free(q);
    free(sc);
}

/*
 * Decode attention for a list of (sequence, head) pairs.
 *   pairs[2*n], pairs[2*n+1] = (s, h) for n < n_pairs
 *   out, out1: [n_pairs][d]; max_logits, exp_sums: [n_pairs][Pmax]; tmp_out: [n_pairs][Pmax][d]
 * partition_size <= 0 means one partition per sequence.  k_scales / v_scales (NULL, or
 * num_kv_heads floats) replace k_scale / v_scale per kv head.  Returns 0, or -1 on bad sizes.
 */
int pa_oracle_decode(const void* query, int q_fmt, const void* key_cache, const void* value_cache,
                     int kv_fmt, int num_seqs, int num_heads, int num_kv_heads, int head_size,
                     int block_size, const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* seq_lens, float scale, const float* alibi_slopes,
                     float k_scale, float v_scale, const float* k_scales, const float* v_scales,
                     int partition_size, int max_num_partitions, const int32_t* pairs, int n_pairs, double* out, double* out1,
                     double* max_logits, double* exp_sums, double* tmp_out, int num_threads) {
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || head_size <= 0 ||
        block_size <= 0 || max_num_partitions <= 0)
        return -1;
    if (head_size % (16 / elem_bytes(kv_fmt)))
        return -1;
    orc_args a = {query, q_fmt, key_cache, value_cache, kv_fmt, num_seqs, num_heads,
                  num_kv_heads, head_size, block_size, block_tables, max_blocks_per_seq,
                  seq_lens, (double)scale, alibi_slopes, (double)k_scale, (double)v_scale,
                  k_scales, v_scales, partition_size > 0 ? partition_size : 0x7fffffff, max_num_partitions};
    for (int n = 0; n < n_pairs; ++n) {
        int s = pairs[2 * n], h = pairs[2 * n + 1];
        if (s < 0 || s >= num_seqs || h < 0 || h >= num_heads) return -1;
        int L = seq_lens[s];
        if (L > 0 && ((int64_t)L + a.part - 1) / a.part > max_num_partitions) return -1;
        if (L > 0 && (L + block_size - 1) / block_size > max_blocks_per_seq) return -1;
    }
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int n = 0; n < n_pairs; ++n) {
        const int64_t d = head_size, P = max_num_partitions;
        decode_one(&a, pairs[2 * n], pairs[2 * n + 1], out + n * d, out1 + n * d,
                   max_logits + n * P, exp_sums + n * P, tmp_out + n * P * d);
    }
    return 0;
}

/*
 * Slot-mapping cache writer ("paged_attn.py", write_to_paged_cache -> reshape_and_cache).
 * key/value rows: [num_tokens][num_kv_heads][head_size], token stride given in elements.
 * For token t with slot = slot_mapping[t] >= 0, b = slot / block_size, o = slot % block_size:
 *   key_cache[b][h][i / x][o][i % x] = enc(key[t][h][i]),  value_cache[b][h][i][o] = enc(value[t][h][i])
 * k_scales / v_scales (NULL, or num_kv_heads floats) replace k_scale / v_scale per kv head.
 * Returns 0, or -1 on bad arguments.
 */
int pa_oracle_reshape_and_cache(const void* key, const void* value, int src_fmt,
                                int64_t key_stride_t, int64_t value_stride_t, void* key_cache,
                                void* value_cache, int kv_fmt, const int64_t* slot_mapping,
                                int num_tokens, int num_kv_heads, int head_size, int block_size,
                                int num_blocks, float k_scale, float v_scale, const float* k_scales,
                                const float* v_scales) {
    if (src_fmt != ORC_F16 && src_fmt != ORC_BF16) return -1;
    if (kv_fmt != src_fmt && kv_fmt != ORC_E4M3) return -1;
    const int x = 16 / elem_bytes(kv_fmt);
    if (head_size % x) return -1;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t b = slot / block_size;
        int o = (int)(slot % block_size);
        if (b >= num_blocks) return -1;
        for (int h = 0; h < num_kv_heads; ++h) {
            const float kdiv = k_scales ? k_scales[h] : k_scale;
            const float vdiv = v_scales ? v_scales[h] : v_scale;
            for (int i = 0; i < head_size; ++i) {
                int64_t ks = t * key_stride_t + (int64_t)h * head_size + i;
                int64_t vs = t * value_stride_t + (int64_t)h * head_size + i;
                int64_t kd = ((((b * num_kv_heads + h) * (head_size / x) + i / x) * block_size + o) * x) + i % x;
                int64_t vd = ((b * num_kv_heads + h) * head_size + i) * (int64_t)block_size + o;
                if (kv_fmt == ORC_E4M3) {
                    float kx = (float)dec_elem(key, ks, src_fmt);
                    float vx = (float)dec_elem(value, vs, src_fmt);
                    ((uint8_t*)key_cache)[kd] = orc_enc_e4m3(kx / kdiv);
                    ((uint8_t*)value_cache)[vd] = orc_enc_e4m3(vx / vdiv);
                } else {
                    ((uint16_t*)key_cache)[kd] = ((const uint16_t*)key)[ks];
                    ((uint16_t*)value_cache)[vd] = ((const uint16_t*)value)[vs];
                }
            }
        }
    }
    return 0;
}

/* Decode every code of a format into doubles (n = 65536 for 16-bit formats, 256 for e4m3). */
int pa_oracle_decode_table(int fmt, double* out) {
    if (fmt == ORC_F16 || fmt == ORC_BF16) {
        for (int c = 0; c < 65536; ++c) out[c] = fmt == ORC_F16 ? orc_dec_f16((uint16_t)c) : orc_dec_bf16((uint16_t)c);
        return 65536;
    }
    if (fmt == ORC_E4M3) {
        for (int c = 0; c < 256; ++c) out[c] = orc_dec_e4m3((uint8_t)c);
        return 256;
    }
    return -1;
}

/* Encode float32 values to e4m3fn codes (the writer's quantiser), for pinning. */
void pa_oracle_encode_e4m3(const float* x, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_enc_e4m3(x[i]);
}

/*
 * Block moves ("paged_attn.py", copy_blocks / swap_blocks): for each pair n in order,
 * dst block mapping[2n+1] receives src block mapping[2n] (block_bytes bytes each).
 * Returns 0, or -1 for an id outside its cache.
 */
int pa_oracle_copy_blocks(void* dst, const void* src, const int64_t* mapping, int num_pairs,
                          int64_t block_bytes, int src_num_blocks, int dst_num_blocks) {
    for (int n = 0; n < num_pairs; ++n) {
        int64_t s = mapping[2 * n], d = mapping[2 * n + 1];
        if (s < 0 || s >= src_num_blocks || d < 0 || d >= dst_num_blocks) return -1;
        memcpy((char*)dst + d * block_bytes, (const char*)src + s * block_bytes, (size_t)block_bytes);
    }
    return 0;
}

/*
 * Chunked-prefix attention ("paged_attn.py", _forward_prefix_pytorch): sequence i has
 * ctx = context_lens[i] tokens already in the paged cache and q_len = qsl[i+1] - qsl[i] new
 * tokens whose rows are query/key/value[qsl[i] + j].  Query j of head h (absolute position
 * ctx + j) attends to every context token and to new tokens 0..j:
 *   s = scale * <q, k> over those keys, out = softmax(s) . v,   kv head = h / (H / Hk).
 * Rows: query [T][H][d], key/value [T][Hk][d] (contiguous), cache views as for decode.
 * rows: optional list of (token, head) pairs; out then holds one d-vector per pair, else
 * out is [T][H][d].  All in fp64.  Returns 0, or -1 on bad sizes.
 */
int pa_oracle_prefix(const void* query, const void* key, const void* value, int fmt,
                     const void* key_cache, const void* value_cache, int num_seqs, int num_heads,
                     int num_kv_heads, int head_size, int block_size, const int32_t* block_tables,
                     int max_blocks_per_seq, const int32_t* query_start_loc,
                     const int32_t* context_lens, float scale, const int32_t* rows, int num_rows,
                     double* out, int num_threads) {
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || head_size % 8) return -1;
    if (fmt != ORC_F16 && fmt != ORC_BF16) return -1;
    orc_args a = {NULL, fmt, key_cache, value_cache, fmt, num_seqs, num_heads, num_kv_heads,
                  head_size, block_size, block_tables, max_blocks_per_seq, NULL, (double)scale,
                  NULL, 1.0, 1.0, NULL, NULL, 0x7fffffff, 1};
    const int H = num_heads, Hk = num_kv_heads, d = head_size, G = H / Hk;
    for (int i = 0; i < num_seqs; ++i) {
        int ctx = context_lens[i];
        if (ctx < 0 || (ctx + block_size - 1) / block_size > max_blocks_per_seq) return -1;
        if (query_start_loc[i + 1] < query_start_loc[i]) return -1;
    }
    const int T = query_start_loc[num_seqs];
    const int64_t n = rows ? (int64_t)num_rows : (int64_t)T * H;
    for (int64_t r = 0; rows && r < n; ++r)
        if (rows[2 * r] < 0 || rows[2 * r] >= T || rows[2 * r + 1] < 0 || rows[2 * r + 1] >= H) return -1;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < n; ++r) {
        {
            const int tq = rows ? rows[2 * r] : (int)(r / H);
            const int h = rows ? rows[2 * r + 1] : (int)(r % H);
            int i = 0;
            while (query_start_loc[i + 1] <= tq) ++i;
            const int q0 = query_start_loc[i], j = tq - q0, ctx = context_lens[i];
            const int kvh = h / G;
            const int nk = ctx + j + 1;
            double* sc = (double*)malloc(sizeof(double) * nk);
            double M = -INFINITY;
            for (int t = 0; t < nk; ++t) {
                double dot = 0.0;
                for (int e = 0; e < d; ++e) {
                    double qv = dec_elem(query, ((int64_t)tq * H + h) * d + e, fmt), kv;
                    if (t < ctx) {
                        int64_t b = block_tables[(int64_t)i * max_blocks_per_seq + t / block_size];
                        kv = k_at(&a, b, kvh, e, t % block_size);
                    } else {
                        kv = dec_elem(key, ((int64_t)(q0 + t - ctx) * Hk + kvh) * d + e, fmt);
                    }
                    dot += qv * kv;
                }
                sc[t] = (double)scale * dot;
                M = sc[t] > M ? sc[t] : M;
            }
            double Z = 0.0;
            for (int t = 0; t < nk; ++t) Z += exp(sc[t] - M);
            double* o = out + r * d;
            for (int e = 0; e < d; ++e) o[e] = 0.0;
            for (int t = 0; t < nk; ++t) {
                const double w = exp(sc[t] - M) / Z;
                for (int e = 0; e < d; ++e) {
                    double vv;
                    if (t < ctx) {
                        int64_t b = block_tables[(int64_t)i * max_blocks_per_seq + t / block_size];
                        vv = v_at(&a, b, kvh, e, t % block_size);
                    } else {
                        vv = dec_elem(value, ((int64_t)(q0 + t - ctx) * Hk + kvh) * d + e, fmt);
                    }
                    o[e] += w * vv;
                }
            }
            free(sc);
        }
    }
    return 0;
}
