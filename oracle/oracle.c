/*
 * CPU oracle for Prefill Context Parallel (PCP) attention — TEST INFRASTRUCTURE.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * use this file. It is a plain, slow, fp64 restatement of what the method
 * computes, kept apart from the CUDA library (no shared headers, helpers or
 * tables). Nothing in the product path may call it.
 *
 * Sources (three pull-request pages on PCP for vLLM):
 *  - "Feat/pcp qwen36 hybrid", section "Changes": each PCP rank holds a
 *    contiguous local token slice; full-attention layers run end-aligned causal
 *    attention over the all-gathered K/V.
 *  - "[MRv2] FlashAttention PCP support for GQA on MRv2", "Pull request
 *    overview": optional sharded cached-prefix (context) attention merged with
 *    the new-token pass; mixed prefill+decode batches; PCP-aware KV-cache update.
 *  - "[MRv2][PCP] Carry the row plan in attention metadata; fix mixed
 *    prefill+decode crash", section 2: up to two rows per prefilling request;
 *    commit "drop pcp_has_prefill": PAD-masked slot mapping, negative slots are
 *    skipped, decode rows are written by rank 0 only; section "What made it
 *    removable": a row's seq_len is its end position, seq_len - query_len is the
 *    row start.
 *  - "[MRv2] FlashAttention PCP support ...", the context-pass call: FP8 KV
 *    cache descales of shape (num_seqs, num_kv_heads) built from the layer's
 *    k/v scales; the e4m3 format itself is the OCP 8-bit floating point one.
 *
 * Every function here is pinned by CPU tests against brute force (a dense
 * numpy softmax), closed forms and the invariants the pages fix.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_RANGE (-2)

/* Row record: eight int32 fields, in this order. */
enum { F_REQ = 0, F_SHARD, F_QSTART, F_QLEN, F_CTX, F_KVEND, F_CAUSAL, F_DECODE, F_NFIELDS };

/* bf16 bit pattern -> double (exact). */
static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Row plan of one step ("Carry the row plan ...", sections 1-2; "Feat/pcp
 * qwen36 hybrid", "Changes").
 *
 * Request r has P = num_computed[r] cached tokens and N = query_len[r] new
 * tokens, packed request-major. Its new tokens are cut into chunks:
 *   mode 0 (contiguous): shard i takes [floor(i N / S), floor((i+1) N / S));
 *   mode 1 (dual chunk): 2S chunks c_k = [floor(k N / 2S), floor((k+1) N / 2S));
 *                        shard i takes chunk i, then chunk 2S-1-i.
 * A request with N == 1 is one row on shard 0. Empty chunks give no row.
 * Rows are emitted shard-major: for shard i, for request r, its chunks in the
 * order above. For a chunk [c0, c1):
 *   q_start = packed offset of r + c0, q_len = c1 - c0, ctx_len = P,
 *   kv_end = P + c1 (the row's end position), causal_off = kv_end - ctx_len - q_len,
 *   is_decode = (N == 1 && P > 0).
 * cu_q is the running sum of q_len over rows. For every new token t of r at
 * absolute position pos = P + j: slot[t] = block_table[r][pos / bs] * bs + pos % bs,
 * owner[t] = the shard of the row holding t.
 * Returns ORC_ERR_RANGE when a needed page is missing or negative, or when
 * rows do not fit into rows_cap.
 */
int oracle_row_plan(int num_reqs, const int32_t* query_len, const int32_t* num_computed,
                    const int32_t* block_table, int max_blocks, int bs, int num_shards, int mode,
                    int32_t* rows, int rows_cap, int32_t* num_rows, int32_t* cu_q,
                    int64_t* slot, int8_t* owner) {
    if (num_reqs < 0 || bs <= 0 || num_shards <= 0 || (mode != 0 && mode != 1)) return ORC_ERR_ARG;
    int64_t* offs = (int64_t*)malloc(sizeof(int64_t) * (size_t)(num_reqs + 1));
    if (!offs) return ORC_ERR_ARG;
    offs[0] = 0;
    for (int r = 0; r < num_reqs; ++r) {
        if (query_len[r] < 0 || num_computed[r] < 0) { free(offs); return ORC_ERR_ARG; }
        offs[r + 1] = offs[r] + query_len[r];
    }
    int n = 0;
    cu_q[0] = 0;
    for (int s = 0; s < num_shards; ++s) {
        for (int r = 0; r < num_reqs; ++r) {
            int64_t N = query_len[r], P = num_computed[r];
            int64_t c0[2], c1[2];
            int nchunk = 0;
            if (N == 0) continue;
            if (N == 1) {
                if (s == 0) { c0[0] = 0; c1[0] = 1; nchunk = 1; }
            } else if (mode == 0) {
                c0[0] = (int64_t)s * N / num_shards;
                c1[0] = (int64_t)(s + 1) * N / num_shards;
                nchunk = 1;
            } else {
                int64_t twoS = 2 * (int64_t)num_shards;
                int64_t head = s, tail = twoS - 1 - s;
                c0[0] = head * N / twoS;  c1[0] = (head + 1) * N / twoS;
                c0[1] = tail * N / twoS;  c1[1] = (tail + 1) * N / twoS;
                nchunk = 2;
            }
            for (int c = 0; c < nchunk; ++c) {
                if (c1[c] <= c0[c]) continue;
                if (n >= rows_cap) { free(offs); return ORC_ERR_RANGE; }
                int32_t* row = rows + (size_t)n * F_NFIELDS;
                row[F_REQ] = r;
                row[F_SHARD] = s;
                row[F_QSTART] = (int32_t)(offs[r] + c0[c]);
                row[F_QLEN] = (int32_t)(c1[c] - c0[c]);
                row[F_CTX] = (int32_t)P;
                row[F_KVEND] = (int32_t)(P + c1[c]);
                row[F_CAUSAL] = row[F_KVEND] - row[F_CTX] - row[F_QLEN];
                row[F_DECODE] = (N == 1 && P > 0) ? 1 : 0;
                cu_q[n + 1] = cu_q[n] + row[F_QLEN];
                for (int64_t j = c0[c]; j < c1[c]; ++j) {
                    int64_t pos = P + j;
                    int64_t page = pos / bs;
                    if (page >= max_blocks) { free(offs); return ORC_ERR_RANGE; }
                    int64_t blk = block_table[(size_t)r * max_blocks + page];
                    if (blk < 0) { free(offs); return ORC_ERR_RANGE; }
                    slot[offs[r] + j] = blk * bs + pos % bs;
                    if (owner) owner[offs[r] + j] = (int8_t)s;
                }
                ++n;
            }
        }
    }
    *num_rows = n;
    free(offs);
    return ORC_OK;
}

/*
 * KV-cache write ("drop pcp_has_prefill": the cache writer skips negative
 * slots). cache is [num_blocks * bs][Hkv][D] in 16-bit words; for each token t
 * with slot[t] >= 0 the row src[t][.][.] is copied to cache[slot[t]][.][.].
 * Returns ORC_ERR_RANGE (after copying nothing for that token) for a slot past
 * the end of the cache.
 */
int oracle_cache_write(const uint16_t* src, const int64_t* slot, int64_t num_tokens,
                       uint16_t* cache, int64_t num_slots, int row_elems) {
    int rc = ORC_OK;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot[t];
        if (s < 0) continue;
        if (s >= num_slots) { rc = ORC_ERR_RANGE; continue; }
        memcpy(cache + (size_t)s * row_elems, src + (size_t)t * row_elems, sizeof(uint16_t) * (size_t)row_elems);
    }
    return rc;
}

/*
 * Attention of one query token against keys [k_lo, min(k_hi, pos + 1)) of its
 * request, for every q head ("Feat/pcp qwen36 hybrid", "Changes": end-aligned
 * causal attention over the reconstructed K/V; "[MRv2] FlashAttention PCP
 * support ...": context pass returning (out, lse)).
 *
 * q_tok: [Hq][D]; k, v: the request's contiguous keys [L][Hkv][D]; pos is the
 * token's absolute position. Head h reads kv head h / (Hq / Hkv).
 *   s_k = scale * sum_d q[h][d] * k[k][h_kv][d]
 *   lse = m + log(sum_k exp(s_k - m)),  m = max_k s_k
 *   out[h][d] = sum_k exp(s_k - lse) * v[k][h_kv][d]
 * With no visible key, lse = -inf and out = 0.
 */
static void attend_token(const uint16_t* q_tok, const uint16_t* k, const uint16_t* v,
                         int64_t pos, int64_t k_lo, int64_t k_hi, int Hq, int Hkv, int D,
                         double scale, double* out, double* lse, double* s_buf) {
    int G = Hq / Hkv;
    int64_t hi = k_hi < pos + 1 ? k_hi : pos + 1;
    int64_t lo = k_lo > 0 ? k_lo : 0;
    for (int h = 0; h < Hq; ++h) {
        int hk = h / G;
        double* o = out + (size_t)h * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (hi <= lo) { lse[h] = -INFINITY; continue; }
        double m = -INFINITY;
        for (int64_t kk = lo; kk < hi; ++kk) {
            const uint16_t* kr = k + ((size_t)kk * Hkv + hk) * D;
            const uint16_t* qr = q_tok + (size_t)h * D;
            double s = 0.0;
            for (int d = 0; d < D; ++d) s += bf16_to_double(qr[d]) * bf16_to_double(kr[d]);
            s *= scale;
            s_buf[kk - lo] = s;
            if (s > m) m = s;
        }
        double sum = 0.0;
        for (int64_t kk = lo; kk < hi; ++kk) sum += exp(s_buf[kk - lo] - m);
        double l = m + log(sum);
        lse[h] = l;
        for (int64_t kk = lo; kk < hi; ++kk) {
            double w = exp(s_buf[kk - lo] - l);
            const uint16_t* vr = v + ((size_t)kk * Hkv + hk) * D;
            for (int d = 0; d < D; ++d) o[d] += w * bf16_to_double(vr[d]);
        }
    }
}

/*
 * Attention for a list of packed query tokens.
 *
 * rows: [num_rows][8] row records (see oracle_row_plan); key_lo/key_hi: the key
 * range each row attends (the whole [0, kv_end) for the fused result;
 * [0, ctx_len) and [ctx_len, kv_end) for the two partials).
 * q: [T][Hq][D]; kv_k/kv_v: every request's contiguous keys back to back,
 * request r starting at token kv_off[r]. tokens: the packed indices to compute
 * (n_tok of them); each must lie in exactly one row.
 * out: [n_tok][Hq][D], lse: [n_tok][Hq]. A token at row-relative index j has
 * absolute position pos = kv_end - q_len + j.
 * Returns ORC_ERR_ARG when a token is in no row.
 */
int oracle_attention(int num_rows, const int32_t* rows, const int64_t* key_lo, const int64_t* key_hi,
                     const uint16_t* q, const uint16_t* kv_k, const uint16_t* kv_v,
                     const int64_t* kv_off, int Hq, int Hkv, int D, double scale,
                     const int64_t* tokens, int64_t n_tok, double* out, double* lse) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0) return ORC_ERR_ARG;
    int64_t max_len = 1;
    for (int i = 0; i < num_rows; ++i) {
        int64_t e = rows[(size_t)i * F_NFIELDS + F_KVEND];
        if (e > max_len) max_len = e;
    }
    int bad = 0;
#pragma omp parallel
    {
        double* s_buf = (double*)malloc(sizeof(double) * (size_t)max_len);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_tok; ++i) {
            int64_t t = tokens[i];
            int found = -1;
            for (int r = 0; r < num_rows; ++r) {
                const int32_t* row = rows + (size_t)r * F_NFIELDS;
                if (t >= row[F_QSTART] && t < (int64_t)row[F_QSTART] + row[F_QLEN]) { found = r; break; }
            }
            if (found < 0 || !s_buf) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            const int32_t* row = rows + (size_t)found * F_NFIELDS;
            int64_t j = t - row[F_QSTART];
            int64_t pos = (int64_t)row[F_KVEND] - row[F_QLEN] + j;
            int64_t base = kv_off[row[F_REQ]];
            attend_token(q + (size_t)t * Hq * D, kv_k + (size_t)base * Hkv * D,
                         kv_v + (size_t)base * Hkv * D, pos, key_lo[found], key_hi[found],
                         Hq, Hkv, D, scale, out + (size_t)i * Hq * D, lse + (size_t)i * Hq, s_buf);
        }
        free(s_buf);
    }
    return bad ? ORC_ERR_ARG : ORC_OK;
}

/*
 * Log-sum-exp merge of two partial results of the same queries ("[MRv2]
 * FlashAttention PCP support ...": the context pass returns (ctx_out, ctx_lse)
 * that is combined with the new-token pass; the DCP "LSE-combine").
 *   m = max(lse_a, lse_b), w_x = exp(lse_x - m),
 *   out = (w_a out_a + w_b out_b) / (w_a + w_b), lse = m + log(w_a + w_b).
 * A part with lse = -inf has weight 0; if both are -inf, out = 0 and lse = -inf.
 * out_*: [n][D], lse_*: [n].
 */
void oracle_lse_merge(const double* out_a, const double* lse_a, const double* out_b,
                      const double* lse_b, int64_t n, int D, double* out, double* lse) {
    for (int64_t i = 0; i < n; ++i) {
        double la = lse_a[i], lb = lse_b[i];
        double* o = out + (size_t)i * D;
        if (la == -INFINITY && lb == -INFINITY) {
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            lse[i] = -INFINITY;
            continue;
        }
        double m = la > lb ? la : lb;
        double wa = exp(la - m), wb = exp(lb - m);
        for (int d = 0; d < D; ++d)
            o[d] = (wa * out_a[(size_t)i * D + d] + wb * out_b[(size_t)i * D + d]) / (wa + wb);
        lse[i] = m + log(wa + wb);
    }
}

/*
 * FP8 (e4m3) KV cache ("[MRv2] FlashAttention PCP support for GQA on MRv2": the
 * context-pass call carries FP8 descales of shape (num_seqs, num_kv_heads)
 * and the layer's k/v scales).
 *
 * e4m3 as defined by the OCP 8-bit floating point format (the "fn" variant):
 * 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
 * encodes subnormals m * 2^-9; there is no infinity, S.1111.111 is NaN, and the
 * largest finite magnitude is 1.75 * 2^8 = 448.
 */
double oracle_e4m3_decode(uint8_t c) {
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Round a float to the nearest e4m3 value, ties to even, magnitudes above 448
 * saturating to 448 (NaN stays NaN). The non-negative finite values, codes 0
 * to 126, increase with the code (val[c] = value of code c), so the nearest
 * one is found by bisection: lo = the last code whose value is <= |x|, then
 * |x| is compared with the values of lo and lo + 1; an exact tie takes the even
 * code (mantissa lsb 0). */
static uint8_t encode_with(float x, const double* val) {
    if (x != x) return 0x7F;
    const uint8_t sign = (x < 0.0f || (x == 0.0f && signbit(x))) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    int lo = 0, hi = 0x7E;  /* val[lo] <= a < val[hi] */
    while (hi - lo > 1) {
        const int mid = (lo + hi) / 2;
        if (val[mid] <= a) lo = mid; else hi = mid;
    }
    const double dlo = a - val[lo], dhi = val[hi] - a;
    int c;
    if (dlo < dhi) c = lo;
    else if (dhi < dlo) c = hi;
    else c = (lo & 1) == 0 ? lo : hi;
    return sign | (uint8_t)c;
}

static void value_table(double* val) {
    for (int c = 0; c <= 0x7E; ++c) val[c] = oracle_e4m3_decode((uint8_t)c);
}

uint8_t oracle_e4m3_encode(float x) {
    double val[0x7F];
    value_table(val);
    return encode_with(x, val);
}

/*
 * FP8 cache write: code = e4m3(x / scale) with x the bf16 value and the
 * division done in fp32 (correctly rounded), scale = k_scale for keys and
 * v_scale for values; negative slots skipped; cache is [num_slots][row_elems]
 * bytes. Returns ORC_ERR_RANGE for a slot past the end.
 */
int oracle_cache_write_fp8(const uint16_t* src, const int64_t* slot, int64_t num_tokens, uint8_t* cache,
                           int64_t num_slots, int row_elems, float scale) {
    int rc = ORC_OK;
    double val[0x7F];
    value_table(val);
#pragma omp parallel for schedule(static) reduction(min : rc)
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot[t];
        if (s < 0) continue;
        if (s >= num_slots) { rc = ORC_ERR_RANGE; continue; }
        for (int e = 0; e < row_elems; ++e) {
            const float x = (float)bf16_to_double(src[(size_t)t * row_elems + e]);
            const float q = x / scale;
            cache[(size_t)s * row_elems + e] = encode_with(q, val);
        }
    }
    return rc;
}

/* out[i] = the e4m3 value of codes[i] (exact in double). */
void oracle_e4m3_decode_array(const uint8_t* codes, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(codes[i]);
}

/* attend_token for an FP8 cache: key k of the request, kv head g, dim d is
 * value(code_k[k][g][d]) * k_descale[g] (same for V); dec[c] is value(c). */
static void attend_token_fp8(const uint16_t* q_tok, const uint8_t* k, const uint8_t* v, const float* kd,
                             const float* vd, const double* dec, int64_t pos, int64_t k_lo, int64_t k_hi,
                             int Hq, int Hkv, int D, double scale, double* out, double* lse, double* s_buf) {
    int G = Hq / Hkv;
    int64_t hi = k_hi < pos + 1 ? k_hi : pos + 1;
    int64_t lo = k_lo > 0 ? k_lo : 0;
    for (int h = 0; h < Hq; ++h) {
        int hk = h / G;
        double* o = out + (size_t)h * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (hi <= lo) { lse[h] = -INFINITY; continue; }
        double m = -INFINITY;
        for (int64_t kk = lo; kk < hi; ++kk) {
            const uint8_t* kr = k + ((size_t)kk * Hkv + hk) * D;
            const uint16_t* qr = q_tok + (size_t)h * D;
            double s = 0.0;
            for (int d = 0; d < D; ++d) s += bf16_to_double(qr[d]) * (dec[kr[d]] * (double)kd[hk]);
            s *= scale;
            s_buf[kk - lo] = s;
            if (s > m) m = s;
        }
        double sum = 0.0;
        for (int64_t kk = lo; kk < hi; ++kk) sum += exp(s_buf[kk - lo] - m);
        double l = m + log(sum);
        lse[h] = l;
        for (int64_t kk = lo; kk < hi; ++kk) {
            double w = exp(s_buf[kk - lo] - l);
            const uint8_t* vr = v + ((size_t)kk * Hkv + hk) * D;
            for (int d = 0; d < D; ++d) o[d] += w * (dec[vr[d]] * (double)vd[hk]);
        }
    }
}

/* oracle_attention over an FP8 cache: every request's key and value codes
 * back to back ([L][Hkv][D] bytes, request r from token kv_off[r]) and the
 * descales k_descale, v_descale [num_reqs][Hkv]. Same arguments otherwise. */
int oracle_attention_fp8kv(int num_rows, const int32_t* rows, const int64_t* key_lo, const int64_t* key_hi,
                           const uint16_t* q, const uint8_t* kv_k, const uint8_t* kv_v, const int64_t* kv_off,
                           const float* k_descale, const float* v_descale, int Hq, int Hkv, int D,
                           double scale, const int64_t* tokens, int64_t n_tok, double* out, double* lse) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0) return ORC_ERR_ARG;
    double dec[256];
    for (int c = 0; c < 256; ++c) dec[c] = oracle_e4m3_decode((uint8_t)c);
    int64_t max_len = 1;
    for (int i = 0; i < num_rows; ++i) {
        int64_t e = rows[(size_t)i * F_NFIELDS + F_KVEND];
        if (e > max_len) max_len = e;
    }
    int bad = 0;
#pragma omp parallel
    {
        double* s_buf = (double*)malloc(sizeof(double) * (size_t)max_len);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_tok; ++i) {
            int64_t t = tokens[i];
            int found = -1;
            for (int r = 0; r < num_rows; ++r) {
                const int32_t* row = rows + (size_t)r * F_NFIELDS;
                if (t >= row[F_QSTART] && t < (int64_t)row[F_QSTART] + row[F_QLEN]) { found = r; break; }
            }
            if (found < 0 || !s_buf) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            const int32_t* row = rows + (size_t)found * F_NFIELDS;
            int64_t j = t - row[F_QSTART];
            int64_t pos = (int64_t)row[F_KVEND] - row[F_QLEN] + j;
            int32_t req = row[F_REQ];
            int64_t base = kv_off[req];
            attend_token_fp8(q + (size_t)t * Hq * D, kv_k + (size_t)base * Hkv * D, kv_v + (size_t)base * Hkv * D,
                             k_descale + (size_t)req * Hkv, v_descale + (size_t)req * Hkv, dec, pos,
                             key_lo[found], key_hi[found], Hq, Hkv, D, scale, out + (size_t)i * Hq * D,
                             lse + (size_t)i * Hq, s_buf);
        }
        free(s_buf);
    }
    return bad ? ORC_ERR_ARG : ORC_OK;
}
