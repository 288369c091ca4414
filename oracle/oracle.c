/*
 * oracle.c -- plain fp64 CPU oracle for attention forward over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header or table with the CUDA
 * library.
 *
 * What it computes (the plain definition, evaluated directly):
 *   out[i, h] = sum_j softmax_j(scale * <q[i, h], k_j>) * v_j
 *   lse[i, h] = log(sum_j exp(scale * <q[i, h], k_j>))       (natural log)
 * over the key set J of query row i:
 *   - keys live in 64-row pages; logical key j of sequence b is row j % 64 of
 *     physical page block_table[b, j / 64]  (FlashMLA "Tensor Shapes
 *     Reference", section "Prefill to Cache Mapping"; the paged K/V blocks of
 *     section 1, flash_mla_with_kvcache, one 64 x D slab per page and head);
 *   - query head h reads KV head h / (Hq / Hk), contiguous groups (same page,
 *     "Grouped-Query Attention" diagram: q heads 0-1 -> kv head 0, ...);
 *   - only keys j < seq_len are used: "unused slots ignored via seq_lens"
 *     (section 1 notes);
 *   - with causal masking, query row i of a segment sees key j iff
 *     j <= qo_offset + i, where qo_offset defaults to kv_len - q_len (MATE
 *     msa_interface, _normalize_qo_offset and _resolve_seqused_k);
 *   - MLA (Modular flare_mla_prefill): the last rope_dim entries of each q row
 *     pair with k_rope[token, 0, :], one row shared by all heads; the first
 *     q_depth - rope_dim pair with the per-head k.
 *   - fp8 MLA (flare_mla_prefill's overload with q_nope, q_rope, q_scale and
 *     k_scales): the per-head parts of q and k are e4m3 codes times their
 *     head's scale; the rope parts and v stay 16-bit.
 *   - MLA with a quantised rope key (flare_mla_prefill's overload with
 *     k_rope and k_rope_scales): the shared rope key of token t is its e4m3
 *     codes times k_rope_scales[t]; q, the per-head k and v stay bf16.
 * New tokens are written into pages by oracle_append_kv ("prefill writes into
 * paged cache", section 4): token p of a sequence goes to row p % 64 of page
 * block_table[b, p / 64].
 * Every element is decoded exactly to double before use (bf16: the upper half
 * of an fp32 word; e4m3: sign, 4-bit exponent with bias 7, 3-bit mantissa,
 * subnormals, S.1111.111 = NaN, times the per-KV-head scale).  Scores, maximum,
 * sum and output are formed in double with a two-pass softmax: no online
 * rescaling, no splits, no tiles.  An empty key set gives out = 0 and
 * lse = -inf (the pages are silent on this case; this is the reading used).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_PAGE 64

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* bf16 -> double: the 16 bits are the high half of an IEEE binary32 word. */
double oracle_bf16_to_double(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* IEEE binary16 -> double: sign, 5-bit exponent with bias 15, 10-bit mantissa,
 * subnormals (exponent field 0: value = mantissa/1024 * 2^-14), inf, NaN. */
double oracle_f16_to_double(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 31;
    int m = bits & 1023;
    double mag;
    if (e == 31) mag = m ? NAN : INFINITY;
    else if (e == 0) mag = ldexp((double)m / 1024.0, -14);
    else mag = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return sign ? -mag : mag;
}

/* OCP FP8 E4M3 ("fn": no infinities) -> double. */
double oracle_e4m3_to_double(uint8_t bits) {
    int sign = (bits >> 7) & 1;
    int e = (bits >> 3) & 15;
    int m = bits & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);          /* subnormal: 2^-6 * m/8 */
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7); /* normal: 2^(e-7) * 1.m */
    return sign ? -mag : mag;
}

/* Element decoders over raw buffers: kind 0 = bf16 (uint16), 1 = e4m3 (uint8),
 * 2 = fp16 (uint16). */
static double load_elem(const void* base, int kind, int64_t idx) {
    if (kind == 0) return oracle_bf16_to_double(((const uint16_t*)base)[idx]);
    if (kind == 2) return oracle_f16_to_double(((const uint16_t*)base)[idx]);
    return oracle_e4m3_to_double(((const uint8_t*)base)[idx]);
}

/*
 * Attention for one query row over n keys whose rows are already decoded:
 *   q[dqk], kd[n][dqk], vd[n][dv]  ->  out[dv], *lse.
 * Two passes: scores and their maximum, then exp-weights, sum, weighted V.
 */
static void attend_row(const double* q, const double* kd, const double* vd, int64_t n,
                       int dqk, int dv, double scale, double* s, double* out, double* lse) {
    for (int d = 0; d < dv; ++d) out[d] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int d = 0; d < dqk; ++d) acc += q[d] * kd[j * dqk + d];
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double p = exp(s[j] - m);
        l += p;
        for (int d = 0; d < dv; ++d) out[d] += p * vd[j * dv + d];
    }
    for (int d = 0; d < dv; ++d) out[d] /= l;
    *lse = m + log(l);
}

/*
 * Single-token decode over a paged cache.
 *   q        bf16 [B, Hq, D] (fp16 when kv_kind is 2: q and the pools share the type)
 *   k_pool   [P, Hk, 64, D] of kind kv_kind (0 bf16, 1 e4m3, 2 fp16); v_pool the same
 *   k_scale, v_scale  double [Hk] dequantisation scales (NULL -> 1)
 *   block_table int32 [B, max_pages]; seq_lens int32 [B]
 *   out double [B, Hq, D]; lse double [B, Hq]
 * Returns 0, or -1 when a referenced page id is outside [0, P) or
 * seq_len > max_pages * 64 (the row is then left as zeros / NaN).
 */
int oracle_decode(int B, int Hq, int Hk, int D, int max_pages, int64_t num_pages, int kv_kind,
                  const uint16_t* q, const void* k_pool, const void* v_pool,
                  const double* k_scale, const double* v_scale,
                  const int32_t* block_table, const int32_t* seq_lens, double scale,
                  double* out, double* lse) {
    int bad = 0;
    int group = Hq / Hk;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t bh = 0; bh < (int64_t)B * Hq; ++bh) {
        int b = (int)(bh / Hq), h = (int)(bh % Hq);
        int kvh = h / group;
        int64_t n = seq_lens[b] > 0 ? seq_lens[b] : 0;
        double* o = out + bh * D;
        if (n > (int64_t)max_pages * ORACLE_PAGE) {
            for (int d = 0; d < D; ++d) o[d] = NAN;
            lse[bh] = NAN;
            bad |= 1;
            continue;
        }
        double* qd = (double*)malloc(sizeof(double) * D);
        double* kd = (double*)malloc(sizeof(double) * (size_t)(n ? n : 1) * D);
        double* vd = (double*)malloc(sizeof(double) * (size_t)(n ? n : 1) * D);
        double* s = (double*)malloc(sizeof(double) * (size_t)(n ? n : 1));
        double ks = k_scale ? k_scale[kvh] : 1.0, vs = v_scale ? v_scale[kvh] : 1.0;
        for (int d = 0; d < D; ++d) qd[d] = load_elem(q, kv_kind == 2 ? 2 : 0, bh * D + d);
        int ok = 1;
        for (int64_t j = 0; j < n && ok; ++j) {
            int64_t page = block_table[(int64_t)b * max_pages + j / ORACLE_PAGE];
            if (page < 0 || page >= num_pages) { ok = 0; break; }
            int64_t row = ((page * Hk + kvh) * ORACLE_PAGE + j % ORACLE_PAGE) * D;
            for (int d = 0; d < D; ++d) {
                kd[j * D + d] = load_elem(k_pool, kv_kind, row + d) * ks;
                vd[j * D + d] = load_elem(v_pool, kv_kind, row + d) * vs;
            }
        }
        if (ok) {
            attend_row(qd, kd, vd, n, D, D, scale, s, o, &lse[bh]);
        } else {
            for (int d = 0; d < D; ++d) o[d] = NAN;
            lse[bh] = NAN;
            bad |= 1;
        }
        free(qd); free(kd); free(vd); free(s);
    }
    return bad ? -1 : 0;
}

/*
 * Prefill / ragged attention (chunked causal against a paged cache, ragged
 * causal, and the MLA shape with a shared rope key).
 *   q      bf16 [total_q, Hq, Dqk]
 *   k      paged: bf16 [P, Hk, 64, Dk]   ragged: bf16 [total_k, Hk, Dk]
 *   v      paged: bf16 [P, Hk, 64, Dv]   ragged: bf16 [total_k, Hk, Dv]
 *          with Dk = Dqk - rope_dim
 *   k_rope bf16 [total_k, 1, rope_dim] (ragged only), or NULL with rope_dim 0
 *   cu_q, cu_k  int32 [B+1] running offsets of query rows / keys
 *   block_table int32 [B, max_pages] or NULL (ragged keys)
 *   qo_offset   int32 [B] or NULL (-> kv_len - q_len)
 *   rows   optional list of (token * Hq + h) rows to evaluate (NULL: all);
 *          out/lse are then [nrows, Dv] / [nrows]
 *   elem_kind  0: q, k, v, k_rope are bf16; 2: fp16
 * Returns 0, or -1 on an out-of-range page id or (paged keys) a kv_len above
 * max_pages * 64, which the block table cannot address (those rows are left
 * as NaN).
 */
int oracle_prefill(int B, int Hq, int Hk, int Dqk, int Dv, int rope_dim, int max_pages,
                   int64_t num_pages, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                   const uint16_t* k_rope, const int32_t* cu_q, const int32_t* cu_k,
                   const int32_t* block_table, const int32_t* qo_offset, int causal,
                   double scale, const int64_t* rows, int64_t nrows, double* out, double* lse,
                   int elem_kind) {
    int group = Hq / Hk;
    int Dk = Dqk - rope_dim;
    int64_t total_q = cu_q[B];
    if (!rows) nrows = total_q * Hq;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t flat = rows ? rows[r] : r;
        int64_t tok = flat / Hq;
        int h = (int)(flat % Hq);
        int kvh = h / group;
        /* the segment holding this query token */
        int b = 0;
        while (b < B - 1 && cu_q[b + 1] <= tok) ++b;
        int64_t i = tok - cu_q[b];
        int64_t q_len = cu_q[b + 1] - cu_q[b];
        int64_t kv_len = cu_k[b + 1] - cu_k[b];
        int64_t off = qo_offset ? qo_offset[b] : kv_len - q_len;
        int64_t n = kv_len;
        if (causal) {
            int64_t lim = off + i + 1; /* keys 0 .. off + i */
            if (lim < n) n = lim;
            if (n < 0) n = 0;
        }
        double* o = out + r * Dv;
        if (block_table && kv_len > (int64_t)max_pages * ORACLE_PAGE) {
            /* the segment's keys run past the block table's row */
            for (int d = 0; d < Dv; ++d) o[d] = NAN;
            lse[r] = NAN;
            bad |= 1;
            continue;
        }
        double* qd = (double*)malloc(sizeof(double) * Dqk);
        double* kd = (double*)malloc(sizeof(double) * (size_t)(n ? n : 1) * Dqk);
        double* vd = (double*)malloc(sizeof(double) * (size_t)(n ? n : 1) * Dv);
        double* s = (double*)malloc(sizeof(double) * (size_t)(n ? n : 1));
        for (int d = 0; d < Dqk; ++d) qd[d] = load_elem(q, elem_kind, (tok * Hq + h) * Dqk + d);
        int ok = 1;
        for (int64_t j = 0; j < n; ++j) {
            int64_t krow, vrow;
            if (block_table) {
                int64_t page = block_table[(int64_t)b * max_pages + j / ORACLE_PAGE];
                if (page < 0 || page >= num_pages) { ok = 0; break; }
                int64_t slab = (page * Hk + kvh) * ORACLE_PAGE + j % ORACLE_PAGE;
                krow = slab * Dk;
                vrow = slab * Dv;
            } else {
                int64_t t = cu_k[b] + j;
                krow = (t * Hk + kvh) * Dk;
                vrow = (t * Hk + kvh) * Dv;
            }
            for (int d = 0; d < Dk; ++d) kd[j * Dqk + d] = load_elem(k, elem_kind, krow + d);
            for (int d = 0; d < rope_dim; ++d)
                kd[j * Dqk + Dk + d] = load_elem(k_rope, elem_kind, (cu_k[b] + j) * rope_dim + d);
            for (int d = 0; d < Dv; ++d) vd[j * Dv + d] = load_elem(v, elem_kind, vrow + d);
        }
        if (ok) {
            attend_row(qd, kd, vd, n, Dqk, Dv, scale, s, o, &lse[r]);
        } else {
            for (int d = 0; d < Dv; ++d) o[d] = NAN;
            lse[r] = NAN;
            bad |= 1;
        }
        free(qd); free(kd); free(vd); free(s);
    }
    return bad ? -1 : 0;
}

/*
 * float -> OCP FP8 E4M3 ("fn"), rounding to nearest with ties to even and
 * saturating to +-448 (the largest finite value).  From the format's
 * definition: sign, 4-bit exponent with bias 7, 3-bit mantissa, subnormals
 * (exponent field 0: value = mantissa/8 * 2^-6).
 */
uint8_t oracle_e4m3_from_float(float x) {
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (isnan(x)) return 0x7F;
    if (a >= 448.0) return sign | 0x7E;
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);      /* a = f * 2^e, f in [0.5, 1): a in [2^(e-1), 2^e) */
    e -= 1;            /* a in [2^e, 2^(e+1)) */
    if (e < -6) {      /* subnormal range: multiples of 2^-9 */
        double m = nearbyint(ldexp(a, 9));  /* default rounding: ties to even */
        if (m >= 8.0) return sign | 0x08;    /* rounded up to the smallest normal */
        return sign | (uint8_t)m;
    }
    double m = nearbyint(ldexp(a, 3 - e));   /* in [8, 16] */
    if (m >= 16.0) { m = 8.0; e += 1; }
    int field = e + 7;
    int mant = (int)m - 8;
    if (field > 15 || (field == 15 && mant == 7)) return sign | 0x7E;
    return sign | (uint8_t)((field << 3) | mant);
}

/*
 * Append new tokens' keys and values to their pages: token i of sequence b
 * (new rows cu_new[b] .. cu_new[b+1]-1) sits at logical position
 * p = start_pos[b] + i, i.e. row p % 64 of page block_table[b, p / 64]
 * (FlashMLA "Tensor Shapes Reference", "Prefill to Cache Mapping").
 *   k_new, v_new  bf16 [total_new, Hk, D]
 *   pools         [P, Hk, 64, D]: kind 0 bf16 (bits copied), kind 1 e4m3:
 *                 code = e4m3(float(x) / scale[h]) (fp32 division)
 * Returns 0, or -1 if a position falls outside the block table or the pool.
 */
int oracle_append_kv(int B, int Hk, int D, int max_pages, int64_t num_pages, int kind,
                     const uint16_t* k_new, const uint16_t* v_new, const int32_t* cu_new,
                     const int32_t* start_pos, const int32_t* block_table, void* k_pool, void* v_pool,
                     const float* k_scale, const float* v_scale) {
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        for (int64_t t = cu_new[b]; t < cu_new[b + 1]; ++t) {
            int64_t p = (int64_t)start_pos[b] + (t - cu_new[b]);
            if (p < 0 || p / ORACLE_PAGE >= max_pages) { bad = 1; continue; }
            int64_t page = block_table[(int64_t)b * max_pages + p / ORACLE_PAGE];
            if (page < 0 || page >= num_pages) { bad = 1; continue; }
            for (int h = 0; h < Hk; ++h) {
                int64_t dst = ((page * Hk + h) * ORACLE_PAGE + p % ORACLE_PAGE) * D;
                int64_t src = (t * Hk + h) * D;
                for (int d = 0; d < D; ++d) {
                    if (kind == 0) {
                        ((uint16_t*)k_pool)[dst + d] = k_new[src + d];
                        ((uint16_t*)v_pool)[dst + d] = v_new[src + d];
                    } else {
                        float kf = (float)oracle_bf16_to_double(k_new[src + d]) / k_scale[h];
                        float vf = (float)oracle_bf16_to_double(v_new[src + d]) / v_scale[h];
                        ((uint8_t*)k_pool)[dst + d] = oracle_e4m3_from_float(kf);
                        ((uint8_t*)v_pool)[dst + d] = oracle_e4m3_from_float(vf);
                    }
                }
            }
        }
    }
    return bad ? -1 : 0;
}

/*
 * fp8 MLA prefill, ragged (Modular flare_mla_prefill, the overload taking
 * q_nope, q_rope, q_scale and k_scales).  The page lists those arguments
 * without their granularity; the reading here: one fp32 scale per head.
 *   q_nope  e4m3 [total_q, Hq, 128]    q_rope bf16 [total_q, Hq, 64]
 *   k_nope  e4m3 [total_k, Hk, 128]    k_rope bf16 [total_k, 1, 64]
 *   v       bf16 [total_k, Hk, 128]
 *   q_scale float [Hq], k_scale float [Hk]
 * Query row (i, h) is the vector (q_scale[h] * q_nope[i, h], q_rope[i, h]) and
 * key j of KV head g the vector (k_scale[g] * k_nope[j, g], k_rope[j, 0]);
 * then the attention of oracle_prefill (masking, offsets, row sampling, outputs
 * as there; out double [rows, 128]).
 */
int oracle_prefill_mla_e4m3(int B, int Hq, int Hk, const uint8_t* q_nope, const uint16_t* q_rope,
                            const float* q_scale, const uint8_t* k_nope, const float* k_scale,
                            const uint16_t* v, const uint16_t* k_rope, const int32_t* cu_q,
                            const int32_t* cu_k, const int32_t* qo_offset, int causal, double scale,
                            const int64_t* rows, int64_t nrows, double* out, double* lse) {
    enum { DN = 128, DR = 64, DQK = 192, DV = 128 };
    int group = Hq / Hk;
    int64_t total_q = cu_q[B];
    if (!rows) nrows = total_q * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t flat = rows ? rows[r] : r;
        int64_t tok = flat / Hq;
        int h = (int)(flat % Hq);
        int g = h / group;
        int b = 0;
        while (b < B - 1 && cu_q[b + 1] <= tok) ++b;
        int64_t i = tok - cu_q[b];
        int64_t q_len = cu_q[b + 1] - cu_q[b];
        int64_t kv_len = cu_k[b + 1] - cu_k[b];
        int64_t off = qo_offset ? qo_offset[b] : kv_len - q_len;
        int64_t n = kv_len;
        if (causal) {
            int64_t lim = off + i + 1;
            if (lim < n) n = lim;
            if (n < 0) n = 0;
        }
        double* qd = (double*)malloc(sizeof(double) * DQK);
        double* kd = (double*)malloc(sizeof(double) * (size_t)(n ? n : 1) * DQK);
        double* vd = (double*)malloc(sizeof(double) * (size_t)(n ? n : 1) * DV);
        double* sc = (double*)malloc(sizeof(double) * (size_t)(n ? n : 1));
        double qs = (double)q_scale[h], ks = (double)k_scale[g];
        for (int d = 0; d < DN; ++d) qd[d] = qs * oracle_e4m3_to_double(q_nope[(tok * Hq + h) * DN + d]);
        for (int d = 0; d < DR; ++d) qd[DN + d] = oracle_bf16_to_double(q_rope[(tok * Hq + h) * DR + d]);
        for (int64_t j = 0; j < n; ++j) {
            int64_t t = cu_k[b] + j;
            for (int d = 0; d < DN; ++d) kd[j * DQK + d] = ks * oracle_e4m3_to_double(k_nope[(t * Hk + g) * DN + d]);
            for (int d = 0; d < DR; ++d) kd[j * DQK + DN + d] = oracle_bf16_to_double(k_rope[t * DR + d]);
            for (int d = 0; d < DV; ++d) vd[j * DV + d] = oracle_bf16_to_double(v[(t * Hk + g) * DV + d]);
        }
        attend_row(qd, kd, vd, n, DQK, DV, scale, sc, out + r * DV, &lse[r]);
        free(qd); free(kd); free(vd); free(sc);
    }
    return 0;
}

/*
 * MLA prefill with the shared rope key in e4m3 (Modular flare_mla_prefill,
 * the overload taking k_rope and k_rope_scales).  The page gives the argument
 * without its granularity; the reading here: one fp32 scale per key token.
 *   q             bf16 [total_q, Hq, 192]  (128 per-head entries, then 64 rope)
 *   k_nope        bf16 [total_k, Hk, 128]
 *   v             bf16 [total_k, Hk, 128]
 *   k_rope        e4m3 [total_k, 64]       (one row per token, all heads)
 *   k_rope_scales float [total_k]
 * Key j (token t = cu_k[b] + j) of KV head g is the vector
 * (k_nope[t, g], k_rope_scales[t] * k_rope[t]); then the attention of
 * oracle_prefill (masking, offsets, row sampling, outputs as there; out
 * double [rows, 128]).
 */
int oracle_prefill_mla_rope_e4m3(int B, int Hq, int Hk, const uint16_t* q, const uint16_t* k_nope,
                                 const uint16_t* v, const uint8_t* k_rope, const float* k_rope_scales,
                                 const int32_t* cu_q, const int32_t* cu_k, const int32_t* qo_offset, int causal,
                                 double scale, const int64_t* rows, int64_t nrows, double* out, double* lse) {
    enum { DN = 128, DR = 64, DQK = 192, DV = 128 };
    int group = Hq / Hk;
    int64_t total_q = cu_q[B];
    if (!rows) nrows = total_q * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t flat = rows ? rows[r] : r;
        int64_t tok = flat / Hq;
        int h = (int)(flat % Hq);
        int g = h / group;
        int b = 0;
        while (b < B - 1 && cu_q[b + 1] <= tok) ++b;
        int64_t i = tok - cu_q[b];
        int64_t q_len = cu_q[b + 1] - cu_q[b];
        int64_t kv_len = cu_k[b + 1] - cu_k[b];
        int64_t off = qo_offset ? qo_offset[b] : kv_len - q_len;
        int64_t n = kv_len;
        if (causal) {
            int64_t lim = off + i + 1;
            if (lim < n) n = lim;
            if (n < 0) n = 0;
        }
        double* qd = (double*)malloc(sizeof(double) * DQK);
        double* kd = (double*)malloc(sizeof(double) * (size_t)(n ? n : 1) * DQK);
        double* vd = (double*)malloc(sizeof(double) * (size_t)(n ? n : 1) * DV);
        double* sc = (double*)malloc(sizeof(double) * (size_t)(n ? n : 1));
        for (int d = 0; d < DQK; ++d) qd[d] = oracle_bf16_to_double(q[(tok * Hq + h) * DQK + d]);
        for (int64_t j = 0; j < n; ++j) {
            int64_t t = cu_k[b] + j;
            double rs = (double)k_rope_scales[t];
            for (int d = 0; d < DN; ++d) kd[j * DQK + d] = oracle_bf16_to_double(k_nope[(t * Hk + g) * DN + d]);
            for (int d = 0; d < DR; ++d) kd[j * DQK + DN + d] = rs * oracle_e4m3_to_double(k_rope[t * DR + d]);
            for (int d = 0; d < DV; ++d) vd[j * DV + d] = oracle_bf16_to_double(v[(t * Hk + g) * DV + d]);
        }
        attend_row(qd, kd, vd, n, DQK, DV, scale, sc, out + r * DV, &lse[r]);
        free(qd); free(kd); free(vd); free(sc);
    }
    return 0;
}
