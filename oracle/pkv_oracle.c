/*
 * pkv_oracle.c -- CPU float64 oracle for one batched paged-KV decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously-correct
 * statement of what the decode step computes.  Only the tests, the smoke check
 * and the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or helper with the CUDA library (paged_kv_decode_table_gb300/csrc), and
 * the CUDA library never calls it.
 *
 * Sources (web pages; cited by title and section):
 *  [LAB]  "Bai Lab tong hop -- Inference Engineering" (openarchlab.com,
 *         inference-lab), block [6] KV state manager (KVPool: block pool of
 *         shape [num_blocks, n_heads, block_size, d_head], write/gather through
 *         a per-sequence block table), block [5] forward (scores q.K/sqrt(d),
 *         max-subtracted softmax over positions, weights times V), block [8]
 *         sample (temperature softmax, top-k, renormalise, top-p, draw over
 *         vocabulary order).
 *  [CH5]  "Suy luan & Toi uu hoa (Inference)" (foundations-of-llms-vi, chapter
 *         5), section 1.2 (temperature p_i(T), top-k, the nucleus set V^(p) =
 *         smallest sorted prefix whose cumulative probability reaches p, and the
 *         renormalised distribution), section 3.1 (GQA: n_q query heads in equal
 *         groups sharing one K/V head), section 3.2 (PagedAttention block table),
 *         section 4.1 (online softmax running max / sum / output).
 *  [SERVE] "LLM inference serving tutorial" (wanshuiyin.github.io, ARIS-in-AI-
 *         Offer), section 3.1 (sampler table: T=0 is a separate greedy branch
 *         with lowest-index tie-break; top-k ties broken by (-z, token_id);
 *         top-p keeps the boundary token), section 1.6 (one RNG stream per
 *         request), appendix A invariants [D01]/[D02].
 *  [PHILOX] J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel Random Numbers:
 *         As Easy as 1, 2, 3", SC'11: the Philox4x64-10 counter-based generator.
 *
 * Readings where the pages leave a step open (each also listed in the design
 * notes): seq_lens counts the new token (the decode row attends to its own
 * position); query head qh reads KV head qh / (Hq/Hkv); scale defaults to
 * 1/sqrt(D); top-p acts on the renormalised top-k distribution; the draw walks
 * the kept set in token-id order; the uniform is the first Philox4x64-10 output
 * word of counter (offset,0,0,0) under key (seed,0), top 53 bits times 2^-53.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fopenmp -shared -fPIC (no fast-math).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Status codes returned by the oracle (same meanings as the library's, but
 * defined here independently). */
#define OR_OK 0
#define OR_INVALID_ARG 1
#define OR_DEVICE_BOUNDS 4
#define OR_NONFINITE 6

/* Element types of KV / q inputs. */
#define OR_F32 0
#define OR_BF16 1

/* ------------------------------------------------------------------------ */
/* Philox4x64-10 [PHILOX]: 10 rounds of the Philox S-box on a 4x64-bit counter,
 * with a Weyl-sequence key schedule.  Multipliers and Weyl constants are the
 * published ones. */
static const uint64_t PHILOX_M0 = 0xD2E7470EE14C6C93ULL;
static const uint64_t PHILOX_M1 = 0xCA5A826395121157ULL;
static const uint64_t PHILOX_W0 = 0x9E3779B97F4A7C15ULL; /* golden ratio */
static const uint64_t PHILOX_W1 = 0xBB67AE8584CAA73BULL; /* sqrt(3) - 1 */

void oracle_philox4x64_10(const uint64_t counter[4], const uint64_t key[2], uint64_t out[4]) {
    uint64_t x0 = counter[0], x1 = counter[1], x2 = counter[2], x3 = counter[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        unsigned __int128 prod0 = (unsigned __int128)PHILOX_M0 * x0;
        unsigned __int128 prod1 = (unsigned __int128)PHILOX_M1 * x2;
        uint64_t hi0 = (uint64_t)(prod0 >> 64), lo0 = (uint64_t)prod0;
        uint64_t hi1 = (uint64_t)(prod1 >> 64), lo1 = (uint64_t)prod1;
        uint64_t y0 = hi1 ^ x1 ^ k0;
        uint64_t y1 = lo1;
        uint64_t y2 = hi0 ^ x3 ^ k1;
        uint64_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += PHILOX_W0;
        k1 += PHILOX_W1;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* Per-request uniform in [0,1): the request's own stream ([SERVE] 1.6) is the
 * Philox key (seed, 0); the decode step picks the counter (offset, 0, 0, 0). */
double oracle_uniform(uint64_t seed, uint64_t offset) {
    uint64_t ctr[4] = {offset, 0, 0, 0};
    uint64_t key[2] = {seed, 0};
    uint64_t out[4];
    oracle_philox4x64_10(ctr, key, out);
    return (double)(out[0] >> 11) * (1.0 / 9007199254740992.0); /* 2^-53 */
}

/* Uniform number j of a request's stream: counter (offset, j, 0, 0) under key
 * (seed, 0); j = 0 is oracle_uniform. */
double oracle_uniform_at(uint64_t seed, uint64_t offset, uint64_t j) {
    uint64_t ctr[4] = {offset, j, 0, 0};
    uint64_t key[2] = {seed, 0};
    uint64_t out[4];
    oracle_philox4x64_10(ctr, key, out);
    return (double)(out[0] >> 11) * (1.0 / 9007199254740992.0); /* 2^-53 */
}

/* ------------------------------------------------------------------------ */
/* Element access: bf16 is the top half of an IEEE float32. */
static double load_elem(const void* base, size_t idx, int dtype) {
    if (dtype == OR_F32) return (double)((const float*)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static size_t elem_size(int dtype) { return dtype == OR_F32 ? 4 : 2; }

/* Offset (in elements) of token `pos` of sequence b, KV head h, in a pool laid
 * out [num_blocks, Hkv, BS, D] ([LAB] block [6]: the token at position pos lives
 * in physical block blocks[pos // BS], slot pos % BS).  Returns -1 when the
 * block-table entry is out of range. */
static long long pool_offset(const int32_t* block_tables, int max_blocks, int b, int pos,
                             int h, int Hkv, int BS, int D, int NB) {
    int logical = pos / BS;
    int slot = pos % BS;
    int32_t blk = block_tables[(size_t)b * max_blocks + logical];
    if (blk < 0 || blk >= NB) return -1;
    return (((long long)blk * Hkv + h) * BS + slot) * (long long)D;
}

/* ------------------------------------------------------------------------ */
/* KV append ([LAB] block [6] KVPool.write, one new token per sequence):
 * seq_lens[b] is the length AFTER the append, so the new token sits at
 * position L-1.  Copies element bits (no arithmetic).  Sequences whose length
 * is outside [1, max_blocks*BS] or whose block id is out of range are skipped
 * and reported. */
int oracle_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                     const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                     int B, int Hkv, int D, int BS, int NB, int dtype) {
    size_t es = elem_size(dtype);
    int status = OR_OK;
    for (int b = 0; b < B; ++b) {
        int L = seq_lens[b];
        if (L < 1 || (long long)L > (long long)max_blocks * BS) { status = OR_DEVICE_BOUNDS; continue; }
        int pos = L - 1;
        for (int h = 0; h < Hkv; ++h) {
            long long off = pool_offset(block_tables, max_blocks, b, pos, h, Hkv, BS, D, NB);
            if (off < 0) { status = OR_DEVICE_BOUNDS; continue; }
            size_t src = ((size_t)b * Hkv + h) * D;
            memcpy((char*)k_cache + (size_t)off * es, (const char*)k_new + src * es, D * es);
            memcpy((char*)v_cache + (size_t)off * es, (const char*)v_new + src * es, D * es);
        }
    }
    return status;
}

/* Gather ([LAB] block [6] KVPool.gather): the first L cached tokens of sequence
 * b, head h, in position order, as float64 [L, D].  Returns non-zero on a bad
 * block id. */
int oracle_gather(const void* cache, const int32_t* block_tables, int max_blocks, int b, int L,
                  int h, int Hkv, int D, int BS, int NB, int dtype, double* out) {
    for (int pos = 0; pos < L; ++pos) {
        long long off = pool_offset(block_tables, max_blocks, b, pos, h, Hkv, BS, D, NB);
        if (off < 0) return OR_DEVICE_BOUNDS;
        for (int d = 0; d < D; ++d) out[(size_t)pos * D + d] = load_elem(cache, (size_t)off + d, dtype);
    }
    return OR_OK;
}

/* Copy-on-write block copies ("LLM inference serving tutorial" 4.2: a shared
 * block that must diverge is copied and the writer's table points at the
 * copy).  For each pair in order, physical block dst[i] of both pools becomes
 * a byte copy of block src[i]: Hkv * BS * D elements per pool.  Pairs with an
 * id outside [0, NB) are skipped and reported. */
int oracle_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int n_pairs,
                       int Hkv, int D, int BS, int NB, int dtype) {
    size_t block_bytes = (size_t)Hkv * BS * D * elem_size(dtype);
    int status = OR_OK;
    for (int i = 0; i < n_pairs; ++i) {
        if (src[i] < 0 || src[i] >= NB || dst[i] < 0 || dst[i] >= NB) { status = OR_DEVICE_BOUNDS; continue; }
        memcpy((char*)k_cache + (size_t)dst[i] * block_bytes, (const char*)k_cache + (size_t)src[i] * block_bytes,
               block_bytes);
        memcpy((char*)v_cache + (size_t)dst[i] * block_bytes, (const char*)v_cache + (size_t)src[i] * block_bytes,
               block_bytes);
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Decode attention for one (sequence, query head), two-pass definition ([LAB]
 * block [5] forward: scores = q.K / sqrt(d), causal row covering every cached
 * position including the new one, softmax with the max subtracted, weights times
 * V; [CH5] 3.1: query head qh uses KV head qh / G).  out[D] in float64.
 * Writes sum(weights) - 1 to *wsum_err.  L = 0 gives zeros. */
static int attention_row(const void* q, size_t qrow, const void* k_cache, const void* v_cache, int dtype,
                         const int32_t* block_tables, int max_blocks, int b, int qh, int L,
                         int Hq, int Hkv, int D, int BS, int NB, double scale, double* out,
                         double* wsum_err) {
    int G = Hq / Hkv;
    int h = qh / G;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    *wsum_err = 0.0;
    if (L == 0) return OR_OK;
    double* K = (double*)malloc(sizeof(double) * (size_t)L * D);
    double* V = (double*)malloc(sizeof(double) * (size_t)L * D);
    double* s = (double*)malloc(sizeof(double) * (size_t)L);
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    int st = oracle_gather(k_cache, block_tables, max_blocks, b, L, h, Hkv, D, BS, NB, dtype, K);
    if (st == OR_OK) st = oracle_gather(v_cache, block_tables, max_blocks, b, L, h, Hkv, D, BS, NB, dtype, V);
    if (st == OR_OK) {
        for (int d = 0; d < D; ++d) qv[d] = load_elem(q, (qrow * Hq + qh) * D + d, dtype);
        double mx = -INFINITY;
        for (int j = 0; j < L; ++j) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qv[d] * K[(size_t)j * D + d];
            s[j] = acc * scale;
            if (s[j] > mx) mx = s[j];
        }
        double z = 0.0;
        for (int j = 0; j < L; ++j) { s[j] = exp(s[j] - mx); z += s[j]; }
        double wsum = 0.0;
        for (int j = 0; j < L; ++j) {
            double w = s[j] / z;
            wsum += w;
            for (int d = 0; d < D; ++d) out[d] += w * V[(size_t)j * D + d];
        }
        *wsum_err = wsum - 1.0;
    } else {
        for (int d = 0; d < D; ++d) out[d] = 0.0;
    }
    free(K); free(V); free(s); free(qv);
    return st;
}

/* Batched decode attention.  rows == NULL: every (b, qh) pair, out is
 * [B, Hq, D].  Otherwise rows holds nrows flat indices b*Hq+qh and out is
 * [nrows, D].  scale <= 0 selects 1/sqrt(D).  Sequences with L outside
 * [0, max_blocks*BS] or a bad block id give zeros and a status.  max_wsum_err
 * receives max |sum(weights) - 1|. */
int oracle_paged_attention(double* out, const void* q, const void* k_cache, const void* v_cache,
                           int dtype, const int32_t* block_tables, int max_blocks,
                           const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int BS, int NB,
                           double scale, const int64_t* rows, long long nrows,
                           double* max_wsum_err) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || BS <= 0) return OR_INVALID_ARG;
    if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
    long long n = rows ? nrows : (long long)B * Hq;
    int status = OR_OK;
    double werr = 0.0;
#pragma omp parallel for schedule(dynamic, 1) reduction(max : werr)
    for (long long i = 0; i < n; ++i) {
        long long flat = rows ? rows[i] : i;
        int b = (int)(flat / Hq), qh = (int)(flat % Hq);
        int L = seq_lens[b];
        double e = 0.0;
        int st;
        if (L < 0 || (long long)L > (long long)max_blocks * BS) {
            for (int d = 0; d < D; ++d) out[i * D + d] = 0.0;
            st = OR_DEVICE_BOUNDS;
        } else {
            st = attention_row(q, (size_t)b, k_cache, v_cache, dtype, block_tables, max_blocks, b, qh, L, Hq,
                               Hkv, D, BS, NB, scale, out + i * D, &e);
        }
        if (st != OR_OK) {
#pragma omp atomic write
            status = st;
        }
        if (fabs(e) > werr) werr = fabs(e);
    }
    if (max_wsum_err) *max_wsum_err = werr;
    return status;
}

/* Split-KV statement of the same row ([CH5] 4.1 online softmax): the L
 * positions are cut at multiples of chunk_tokens; chunk c yields its own max m_c,
 * sum l_c = sum exp(s - m_c) and unnormalised o_c = sum exp(s - m_c) V; the
 * chunks merge as M = max m_c, Lsum = sum l_c e^(m_c - M),
 * out = sum o_c e^(m_c - M) / Lsum.  Used to pin the split algebra against the
 * two-pass definition. */
int oracle_attention_split_row(double* out, const void* q, const void* k_cache,
                               const void* v_cache, int dtype, const int32_t* block_tables,
                               int max_blocks, int b, int qh, int L, int Hq, int Hkv, int D,
                               int BS, int NB, double scale, int chunk_tokens) {
    int G = Hq / Hkv, h = qh / G;
    if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (L == 0) return OR_OK;
    if (chunk_tokens <= 0) return OR_INVALID_ARG;
    double* K = (double*)malloc(sizeof(double) * (size_t)L * D);
    double* V = (double*)malloc(sizeof(double) * (size_t)L * D);
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    double* oc = (double*)malloc(sizeof(double) * (size_t)D);
    int nchunks = (L + chunk_tokens - 1) / chunk_tokens;
    double* mc = (double*)malloc(sizeof(double) * nchunks);
    double* lc = (double*)malloc(sizeof(double) * nchunks);
    double* occ = (double*)malloc(sizeof(double) * (size_t)nchunks * D);
    int st = oracle_gather(k_cache, block_tables, max_blocks, b, L, h, Hkv, D, BS, NB, dtype, K);
    if (st == OR_OK) st = oracle_gather(v_cache, block_tables, max_blocks, b, L, h, Hkv, D, BS, NB, dtype, V);
    if (st == OR_OK) {
        for (int d = 0; d < D; ++d) qv[d] = load_elem(q, ((size_t)b * Hq + qh) * D + d, dtype);
        for (int c = 0; c < nchunks; ++c) {
            int j0 = c * chunk_tokens, j1 = j0 + chunk_tokens < L ? j0 + chunk_tokens : L;
            double m = -INFINITY;
            for (int j = j0; j < j1; ++j) {
                double acc = 0.0;
                for (int d = 0; d < D; ++d) acc += qv[d] * K[(size_t)j * D + d];
                acc *= scale;
                if (acc > m) m = acc;
            }
            double l = 0.0;
            for (int d = 0; d < D; ++d) oc[d] = 0.0;
            for (int j = j0; j < j1; ++j) {
                double acc = 0.0;
                for (int d = 0; d < D; ++d) acc += qv[d] * K[(size_t)j * D + d];
                double e = exp(acc * scale - m);
                l += e;
                for (int d = 0; d < D; ++d) oc[d] += e * V[(size_t)j * D + d];
            }
            mc[c] = m; lc[c] = l;
            for (int d = 0; d < D; ++d) occ[(size_t)c * D + d] = oc[d];
        }
        double M = -INFINITY;
        for (int c = 0; c < nchunks; ++c) if (mc[c] > M) M = mc[c];
        double Ls = 0.0;
        for (int c = 0; c < nchunks; ++c) Ls += lc[c] * exp(mc[c] - M);
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int c = 0; c < nchunks; ++c) acc += occ[(size_t)c * D + d] * exp(mc[c] - M);
            out[d] = acc / Ls;
        }
    }
    free(K); free(V); free(qv); free(oc); free(mc); free(lc); free(occ);
    return st;
}

/* ------------------------------------------------------------------------ */
/* Sampler. */

typedef struct {
    float z;
    int32_t id;
} zid_t;

/* Sort key ([SERVE] 3.1 top-k row): descending logit, then ascending token id.
 * Compared as doubles, so -0.0 and +0.0 are equal and fall back to the id. */
static int cmp_zid(const void* a, const void* b) {
    const zid_t* x = (const zid_t*)a;
    const zid_t* y = (const zid_t*)b;
    double zx = (double)x->z, zy = (double)y->z;
    if (zx > zy) return -1;
    if (zx < zy) return 1;
    return (x->id < y->id) ? -1 : (x->id > y->id ? 1 : 0);
}

/* One row of the logits -> token step.
 *   T == 0      greedy branch: argmax, lowest index among ties ([SERVE] 3.1).
 *   T > 0       p_i = exp((z_i - z_max)/T) over finite logits ([CH5] 1.2 eq.
 *               for p_i(T), max subtracted as in [LAB] block [8] softmax);
 *               top-k keeps the first k of the (-z, id) order when 0 < k < |E|
 *               (E = finite logits; -inf entries are banned tokens, [SERVE] 3.3);
 *               renormalise over the top-k set ([LAB] block [8]);
 *               top-p (p < 1) keeps the smallest sorted prefix whose cumulative
 *               renormalised probability is >= p, boundary token included
 *               ([CH5] 1.2 set V^(p); [SERVE] 3.1 top-p row);
 *               renormalise over the nucleus ([CH5] 1.2 p~);
 *               draw: walk the kept tokens in token-id order and return the
 *               first whose running CDF exceeds u ([LAB] block [8] draws over
 *               VOCAB order; u from the request's own Philox stream).
 * Errors: a NaN or +inf logit, or no finite logit -> OR_NONFINITE;
 * T < 0 / NaN or p <= 0 / NaN -> OR_INVALID_ARG; token = -1 then.
 * Diagnostics: draw_margin = distance from u to the nearer CDF edge of the
 * chosen token; cut_margin = distance from p to the nearer of the two
 * cumulative sums that bracket the top-p cut (1.0 when top-p is off);
 * n_kept = size of the final support; probs (optional, length V) = final
 * renormalised distribution in token-id order. */
int oracle_sample_row_ex(const float* z, int V, float temperature, int top_k, float top_p, float min_p,
                         uint64_t seed, uint64_t offset, int32_t* token, double* draw_margin,
                         double* cut_margin, int32_t* n_kept, double* probs) {
    *token = -1;
    *draw_margin = 0.0;
    *cut_margin = 1.0;
    *n_kept = 0;
    if (probs) for (int i = 0; i < V; ++i) probs[i] = 0.0;
    int n_fin = 0;
    for (int i = 0; i < V; ++i) {
        if (isnan(z[i]) || (isinf(z[i]) && z[i] > 0)) return OR_NONFINITE;
        if (isfinite(z[i])) ++n_fin;
    }
    if (n_fin == 0) return OR_NONFINITE;
    if (!(temperature >= 0.0f)) return OR_INVALID_ARG; /* negative or NaN */
    if (temperature == 0.0f) {
        int best = -1;
        for (int i = 0; i < V; ++i)
            if (isfinite(z[i]) && (best < 0 || z[i] > z[best])) best = i;
        *token = best;
        *n_kept = 1;
        *draw_margin = 1.0;
        if (probs) probs[best] = 1.0;
        return OR_OK;
    }
    if (!(top_p > 0.0f)) return OR_INVALID_ARG; /* p <= 0 or NaN */
    if (isnan(min_p) || min_p > 1.0f) return OR_INVALID_ARG;

    zid_t* ord = (zid_t*)malloc(sizeof(zid_t) * (size_t)n_fin);
    int n = 0;
    for (int i = 0; i < V; ++i)
        if (isfinite(z[i])) { ord[n].z = z[i]; ord[n].id = i; ++n; }
    qsort(ord, (size_t)n, sizeof(zid_t), cmp_zid);

    /* top-k */
    if (top_k > 0 && top_k < n) n = top_k;

    /* temperature softmax over the top-k set, renormalised */
    double T = (double)temperature;
    double zmax = (double)ord[0].z;
    double* q = (double*)malloc(sizeof(double) * (size_t)n);
    double S = 0.0;
    for (int j = 0; j < n; ++j) { q[j] = exp(((double)ord[j].z - zmax) / T); S += q[j]; }
    for (int j = 0; j < n; ++j) q[j] /= S;

    /* top-p: smallest prefix with cumulative >= p */
    int m = n;
    if (top_p < 1.0f) {
        double p = (double)top_p;
        double cum = 0.0, prev = 0.0;
        for (int j = 0; j < n; ++j) {
            prev = cum;
            cum += q[j];
            if (cum >= p) { m = j + 1; break; }
        }
        double d1 = fabs(cum - p), d0 = fabs(prev - p);
        *cut_margin = d1 < d0 ? d1 : d0;
    }

    /* min-p ("LLM inference serving tutorial" 3.1, Q4): keep the tokens whose
     * probability is at least min_p times the largest, i.e. whose weight
     * exp((z - zmax) / T) relative to the maximum is >= min_p; the maximum is
     * always kept.  Applied after top-p (a prefix of the same order).  The
     * margin to that threshold joins cut_margin. */
    if (min_p > 0.0f) {
        double a = (double)min_p;
        int keep = 0;
        for (int j = 0; j < m; ++j) {
            double w = exp(((double)ord[j].z - zmax) / T);
            double d = fabs(w - a);
            if (d < *cut_margin) *cut_margin = d;
            if (w >= a) keep = j + 1;
        }
        m = keep;
    }

    /* renormalise over the nucleus; draw in token-id order */
    double Sp = 0.0;
    for (int j = 0; j < m; ++j) Sp += q[j];
    double* pi = (double*)calloc((size_t)V, sizeof(double));
    unsigned char* kept = (unsigned char*)calloc((size_t)V, 1);
    for (int j = 0; j < m; ++j) { pi[ord[j].id] = q[j] / Sp; kept[ord[j].id] = 1; }
    double u = oracle_uniform(seed, offset);
    double c = 0.0, cprev = 0.0;
    int tok = -1, last = -1;
    for (int i = 0; i < V; ++i) {
        if (!kept[i]) continue;
        last = i;
        cprev = c;
        c += pi[i];
        if (c > u) { tok = i; break; }
    }
    if (tok < 0) { tok = last; *draw_margin = 0.0; }
    else {
        double a = u - cprev, bnd = c - u;
        *draw_margin = a < bnd ? a : bnd;
    }
    *token = tok;
    *n_kept = m;
    if (probs) for (int i = 0; i < V; ++i) probs[i] = pi[i];
    free(ord); free(q); free(pi); free(kept);
    return OR_OK;
}

int oracle_sample_row(const float* z, int V, float temperature, int top_k, float top_p,
                      uint64_t seed, uint64_t offset, int32_t* token, double* draw_margin,
                      double* cut_margin, int32_t* n_kept, double* probs) {
    return oracle_sample_row_ex(z, V, temperature, top_k, top_p, 0.0f, seed, offset, token, draw_margin,
                                cut_margin, n_kept, probs);
}

/* Typical sampling ("LLM inference serving tutorial" 3.1, other samplers;
 * appendix A [D01]; Meister et al., "Locally Typical Sampling"), for one row,
 * literally in float64:
 *   a_i = (z_i - z_max) / T and p_i = exp(a_i) / S over the finite logits,
 *     S = sum_i exp(a_i) (T > 0);
 *   ln p_i = a_i - ln S (the logarithm of that same p_i, taken without the
 *     exp round trip so that it stays finite where exp(a_i) underflows);
 *   H(p) = -sum_i p_i ln p_i (a term with p_i = 0 contributes 0);
 *   d_i = |-ln p_i - H(p)|;
 *   the tokens in ascending d; equal d_i go to the larger logit (the more
 *   probable token) first, then to the smaller id;
 *   the kept set is the smallest prefix of that order whose cumulative
 *   probability reaches typical_p (boundary token kept), renormalised; the
 *   draw walks it in token-id order with the request's Philox uniform, as in
 *   oracle_sample_row_ex.
 * T == 0 is the greedy branch; typical_p >= 1 keeps every finite logit.
 * Errors: as oracle_sample_row_ex, and typical_p <= 0 or NaN -> OR_INVALID_ARG.
 * Diagnostics: entropy = H(p) in nats; order_margin = the gap in d (nats)
 * between the boundary token and its nearest neighbours in the order whose
 * logit differs from its own, below and above (1 when there is none): where
 * it is tiny, rounding in another implementation could exchange the two and
 * move the cut; cut_margin and draw_margin as in the top-p sampler; probs
 * (optional) = the final renormalised distribution. */
typedef struct {
    double d, p;
    float z;
    int32_t id;
} typ_t;

static int cmp_typ(const void* a, const void* b) {
    const typ_t* x = (const typ_t*)a;
    const typ_t* y = (const typ_t*)b;
    if (x->d < y->d) return -1;
    if (x->d > y->d) return 1;
    if (x->z > y->z) return -1;
    if (x->z < y->z) return 1;
    return (x->id < y->id) ? -1 : (x->id > y->id ? 1 : 0);
}

int oracle_sample_row_typical(const float* z, int V, float temperature, float typical_p, uint64_t seed,
                              uint64_t offset, int32_t* token, double* draw_margin, double* cut_margin,
                              double* order_margin, double* entropy, int32_t* n_kept, double* probs) {
    *order_margin = 1.0;
    *entropy = 0.0;
    if (temperature == 0.0f || typical_p >= 1.0f) /* greedy, or no truncation (NaN p goes on) */
        return oracle_sample_row_ex(z, V, temperature, 0, 1.0f, 0.0f, seed, offset, token, draw_margin,
                                    cut_margin, n_kept, probs);
    *token = -1;
    *draw_margin = 0.0;
    *cut_margin = 1.0;
    *n_kept = 0;
    if (probs) for (int i = 0; i < V; ++i) probs[i] = 0.0;
    int n = 0;
    float zmaxf = -INFINITY;
    for (int i = 0; i < V; ++i) {
        if (isnan(z[i]) || (isinf(z[i]) && z[i] > 0)) return OR_NONFINITE;
        if (isfinite(z[i])) {
            ++n;
            if (z[i] > zmaxf) zmaxf = z[i];
        }
    }
    if (n == 0) return OR_NONFINITE;
    if (!(temperature >= 0.0f)) return OR_INVALID_ARG;
    if (!(typical_p > 0.0f)) return OR_INVALID_ARG; /* <= 0 or NaN */

    /* the distribution p, ln p, the entropy H and d */
    const double T = (double)temperature, zmax = (double)zmaxf;
    typ_t* t = (typ_t*)malloc(sizeof(typ_t) * (size_t)n);
    double* a = (double*)malloc(sizeof(double) * (size_t)n);
    double S = 0.0;
    int k = 0;
    for (int i = 0; i < V; ++i)
        if (isfinite(z[i])) {
            t[k].id = i;
            t[k].z = z[i];
            a[k] = ((double)z[i] - zmax) / T;
            t[k].p = exp(a[k]);
            S += t[k].p;
            ++k;
        }
    const double lnS = log(S);
    double H = 0.0;
    for (int j = 0; j < n; ++j) {
        t[j].p /= S;
        if (t[j].p > 0.0) H -= t[j].p * (a[j] - lnS);
    }
    *entropy = H;
    for (int j = 0; j < n; ++j) t[j].d = fabs(-(a[j] - lnS) - H);
    free(a);
    qsort(t, (size_t)n, sizeof(typ_t), cmp_typ);

    /* smallest prefix reaching typical_p */
    const double tp = (double)typical_p;
    double cum = 0.0, prev = 0.0;
    int m = n;
    for (int j = 0; j < n; ++j) {
        prev = cum;
        cum += t[j].p;
        if (cum >= tp) { m = j + 1; break; }
    }
    {
        double d1 = fabs(cum - tp), d0 = fabs(prev - tp);
        *cut_margin = d1 < d0 ? d1 : d0;
    }
    {   /* gaps in d around the boundary token c = m - 1 */
        const int c = m - 1;
        double gap = 1.0;
        for (int j = c - 1; j >= 0; --j)
            if (t[j].z != t[c].z) {
                if (t[c].d - t[j].d < gap) gap = t[c].d - t[j].d;
                break;
            }
        for (int j = c + 1; j < n; ++j)
            if (t[j].z != t[c].z) {
                if (t[j].d - t[c].d < gap) gap = t[j].d - t[c].d;
                break;
            }
        *order_margin = gap;
    }

    /* renormalise; draw in token-id order */
    double Sp = 0.0;
    for (int j = 0; j < m; ++j) Sp += t[j].p;
    double* pi = (double*)calloc((size_t)V, sizeof(double));
    unsigned char* kept = (unsigned char*)calloc((size_t)V, 1);
    for (int j = 0; j < m; ++j) { pi[t[j].id] = t[j].p / Sp; kept[t[j].id] = 1; }
    const double u = oracle_uniform(seed, offset);
    double c = 0.0, cprev = 0.0;
    int tok = -1, last = -1;
    for (int i = 0; i < V; ++i) {
        if (!kept[i]) continue;
        last = i;
        cprev = c;
        c += pi[i];
        if (c > u) { tok = i; break; }
    }
    if (tok < 0) { tok = last; *draw_margin = 0.0; }
    else {
        double a = u - cprev, bnd = c - u;
        *draw_margin = a < bnd ? a : bnd;
    }
    *token = tok;
    *n_kept = m;
    if (probs) for (int i = 0; i < V; ++i) probs[i] = pi[i];
    free(t); free(pi); free(kept);
    return OR_OK;
}

/* Logits processors before the sampler ("LLM inference serving tutorial" 3.1
 * pipeline: hard constraints, then penalties, then temperature and filters;
 * 3.2 penalty definitions; 3.3 constraint masks), in place on logits [B, V]:
 *  1. mask (optional, uint32 [B, ceil(V/32)]): token i of row b is allowed iff
 *     bit (i % 32) of word i / 32 is set; a disallowed logit becomes -inf;
 *  2. for each (token, count c >= 1) listed for row b (CSR: row_ptr [B+1],
 *     tokens / counts [nnz]; each token at most once per row) whose logit is
 *     finite: the sign-aware repetition penalty r = rep[b] (z / r for z > 0,
 *     z * r for z < 0, z = 0 unchanged; r == 1 is a no-op), then
 *     z - freq[b] * c - pres[b], in double, rounded once to float.
 * rep, freq, pres may be NULL (off).  Errors: a listed token outside [0, V) or
 * r <= 0 / NaN -> OR_INVALID_ARG (that entry, or the row's penalties, skipped). */
int oracle_process_logits(float* logits, int B, int V, const uint32_t* mask, const int32_t* row_ptr,
                          const int32_t* tokens, const int32_t* counts, const float* rep, const float* freq,
                          const float* pres) {
    int status = OR_OK;
    int words = (V + 31) / 32;
    for (int b = 0; b < B; ++b) {
        float* z = logits + (size_t)b * V;
        if (mask) {
            const uint32_t* mrow = mask + (size_t)b * words;
            for (int i = 0; i < V; ++i)
                if (!((mrow[i / 32] >> (i % 32)) & 1u)) z[i] = -INFINITY;
        }
        if (!row_ptr) continue;
        double r = rep ? (double)rep[b] : 1.0;
        double f = freq ? (double)freq[b] : 0.0;
        double pr = pres ? (double)pres[b] : 0.0;
        if (!(r > 0.0)) { status = OR_INVALID_ARG; continue; }
        for (int e = row_ptr[b]; e < row_ptr[b + 1]; ++e) {
            int t = tokens[e], c = counts[e];
            if (t < 0 || t >= V) { status = OR_INVALID_ARG; continue; }
            if (c < 1 || !isfinite(z[t])) continue;
            double zd = (double)z[t];
            if (r != 1.0) zd = zd > 0.0 ? zd / r : (zd < 0.0 ? zd * r : zd);
            zd = zd - f * (double)c;
            zd = zd - pr;
            z[t] = (float)zd;
        }
    }
    return status;
}

/* Batched sampler over B rows of logits [B, V] (rows independent).  Per-row
 * status goes to status_out (may be NULL); returns the first non-zero status. */
int oracle_sample_batch(const float* logits, int B, int V, const float* temperature,
                        const int32_t* top_k, const float* top_p, const uint64_t* seeds,
                        const uint64_t* offsets, int32_t* tokens, double* draw_margin,
                        double* cut_margin, int32_t* n_kept, int32_t* status_out) {
    int status = OR_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        int st = oracle_sample_row(logits + (size_t)b * V, V, temperature[b], top_k[b], top_p[b],
                                   seeds[b], offsets[b], tokens + b, draw_margin + b,
                                   cut_margin + b, n_kept + b, NULL);
        if (status_out) status_out[b] = st;
        if (st != OR_OK) {
#pragma omp atomic write
            status = st;
        }
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Chunked prefill ("Bai Lab tong hop -- Inference Engineering" prefill of a
 * prompt through the same block table; "Suy luan & Toi uu hoa (Inference)"
 * 2.1: a chunk's queries attend causally to the whole cached prefix and to the
 * chunk itself; "LLM inference serving tutorial" 5.4 chunked prefill).  Sequence
 * b appends n_b = q_start[b+1] - q_start[b] new tokens (rows q_start[b] ..
 * q_start[b+1]-1 of the packed [T, Hkv, D] / [T, Hq, D] arrays); seq_lens[b]
 * is the length after the append, so new token i sits at position
 * L_b - n_b + i. */
static int seq_of_row(const int32_t* q_start, int B, int t) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {  /* last b with q_start[b] <= t */
        int mid = (lo + hi + 1) / 2;
        if (q_start[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

int oracle_kv_append_chunk(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                           const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                           const int32_t* q_start, int B, int Hkv, int D, int BS, int NB, int dtype) {
    size_t es = elem_size(dtype);
    int status = OR_OK;
    for (int b = 0; b < B; ++b) {
        int n = q_start[b + 1] - q_start[b], L = seq_lens[b];
        if (n < 0 || L < n || (long long)L > (long long)max_blocks * BS) { status = OR_DEVICE_BOUNDS; continue; }
        for (int i = 0; i < n; ++i) {
            int pos = L - n + i;
            size_t t = (size_t)q_start[b] + i;
            for (int h = 0; h < Hkv; ++h) {
                long long off = pool_offset(block_tables, max_blocks, b, pos, h, Hkv, BS, D, NB);
                if (off < 0) { status = OR_DEVICE_BOUNDS; continue; }
                size_t src = (t * Hkv + h) * D;
                memcpy((char*)k_cache + (size_t)off * es, (const char*)k_new + src * es, D * es);
                memcpy((char*)v_cache + (size_t)off * es, (const char*)v_new + src * es, D * es);
            }
        }
    }
    return status;
}

/* Causal attention of the chunk's queries: row (t, qh) of the packed q [T, Hq,
 * D] attends to positions 0 .. pos_t of its sequence through the table.  rows
 * (length nrows, values t * Hq + qh) selects the rows computed (NULL: all T *
 * Hq); out is [nrows, D] float64. */
int oracle_prefill_attention(double* out, const void* q, const void* k_cache, const void* v_cache, int dtype,
                             const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                             const int32_t* q_start, int B, int Hq, int Hkv, int D, int BS, int NB, double scale,
                             const int64_t* rows, int64_t nrows, double* max_wsum_err) {
    if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
    int T = q_start[B];
    if (!rows) nrows = (int64_t)T * Hq;
    int status = OR_OK;
    double werr = 0.0;
#pragma omp parallel for schedule(dynamic, 4) reduction(max : werr)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t flat = rows ? rows[i] : i;
        int t = (int)(flat / Hq), qh = (int)(flat % Hq);
        int b = seq_of_row(q_start, B, t);
        int n = q_start[b + 1] - q_start[b], L = seq_lens[b];
        double e = 0.0;
        int st;
        if (n < 1 || L < n || (long long)L > (long long)max_blocks * BS) {
            for (int d = 0; d < D; ++d) out[i * D + d] = 0.0;
            st = OR_DEVICE_BOUNDS;
        } else {
            int pos = L - n + (t - q_start[b]);
            st = attention_row(q, (size_t)t, k_cache, v_cache, dtype, block_tables, max_blocks, b, qh, pos + 1,
                               Hq, Hkv, D, BS, NB, scale, out + i * D, &e);
        }
        if (st != OR_OK) {
#pragma omp atomic write
            status = st;
        }
        if (fabs(e) > werr) werr = fabs(e);
    }
    if (max_wsum_err) *max_wsum_err = werr;
    return status;
}

/* ------------------------------------------------------------------------ */
/* Speculative-decoding verification ("Suy luan & Toi uu hoa (Inference)" 5.2,
 * speculative rejection sampling after Leviathan & Matias; "LLM inference
 * serving tutorial" section 7 and Q16: a variable number of accepted tokens,
 * and the KV of rejected candidates rolled back).  One request:
 *   target logits zt[gamma+1][V] (the target model's distributions p_1..p_{g+1}
 *   at the g draft positions and the one after), draft logits zd[gamma][V]
 *   (q_1..q_g), draft tokens x[gamma], temperature T, stream (seed, offset).
 *   p_i = softmax(zt[i] / T), q_i = softmax(zd[i] / T) over finite logits.
 *   T == 0: accept while x[i] is the target argmax of row i (lowest id among
 *     ties); the token after the accepted ones is the argmax of the first
 *     rejected row, or of row gamma when all are accepted.
 *   T > 0: for i = 0.. in order, u_i = uniform number i + 1 of the stream;
 *     accept x[i] iff u_i * q_i(x[i]) < p_i(x[i]) (probability min(1, p/q));
 *     stop at the first rejection.  Rejected at n: draw from the residual
 *     max(0, p_n - q_n) normalised (p_n when the residual is all zero); all
 *     accepted: draw from p_{gamma+1}.  The draw uses uniform number 0 and walks
 *     token ids in ascending order (first id whose running CDF exceeds u).
 * Outputs: tokens[0..n_acc) = accepted drafts, tokens[n_acc] = the drawn
 * token, tokens past it = -1; *n_acc; *seq_len_out = seq_len - gamma + n_acc
 * (seq_len counts the gamma draft positions whose KV the target pass wrote;
 * the rejected ones are rolled back).
 * Diagnostics: *test_margin = min over the tests made of |u_i - p/q| (1 when
 * none or T == 0); *draw_margin = distance from u to the nearer CDF edge of
 * the drawn token (1 for T == 0).
 * Errors: NaN / +inf logit or a row with no finite logit -> OR_NONFINITE;
 * T < 0 or NaN, a draft token outside [0, V), seq_len < gamma ->
 * OR_INVALID_ARG; then tokens are -1, n_acc = 0 and seq_len_out = seq_len. */
static int row_check(const float* z, int V) {
    int fin = 0;
    for (int i = 0; i < V; ++i) {
        if (isnan(z[i]) || (isinf(z[i]) && z[i] > 0)) return OR_NONFINITE;
        if (isfinite(z[i])) ++fin;
    }
    return fin ? OR_OK : OR_NONFINITE;
}

static int row_argmax(const float* z, int V) {
    int best = -1;
    for (int i = 0; i < V; ++i)
        if (isfinite(z[i]) && (best < 0 || z[i] > z[best])) best = i;
    return best;
}

/* probabilities softmax(z / T) over finite logits into pr[V] */
static void row_softmax(const float* z, int V, double T, double* pr) {
    double zmax = -INFINITY;
    for (int i = 0; i < V; ++i) if (isfinite(z[i]) && z[i] > zmax) zmax = z[i];
    double S = 0.0;
    for (int i = 0; i < V; ++i) { pr[i] = isfinite(z[i]) ? exp(((double)z[i] - zmax) / T) : 0.0; S += pr[i]; }
    for (int i = 0; i < V; ++i) pr[i] /= S;
}

/* inverse CDF in token-id order of the (unnormalised) weights w[V] */
static int draw_id_order(const double* w, int V, double u, double* margin) {
    double S = 0.0;
    for (int i = 0; i < V; ++i) S += w[i];
    double c = 0.0, cprev = 0.0;
    int last = -1;
    for (int i = 0; i < V; ++i) {
        if (w[i] <= 0.0) continue;
        last = i;
        cprev = c;
        c += w[i] / S;
        if (c > u) {
            double a = u - cprev, b = c - u;
            *margin = a < b ? a : b;
            return i;
        }
    }
    *margin = 0.0;
    return last;
}

int oracle_spec_verify_row(const float* zt, const float* zd, const int32_t* x, int gamma, int V,
                           float temperature, uint64_t seed, uint64_t offset, int32_t seq_len,
                           int32_t* tokens, int32_t* n_acc, int32_t* seq_len_out,
                           double* test_margin, double* draw_margin) {
    for (int i = 0; i <= gamma; ++i) tokens[i] = -1;
    *n_acc = 0;
    *seq_len_out = seq_len;
    *test_margin = 1.0;
    *draw_margin = 1.0;
    for (int i = 0; i <= gamma; ++i) { int st = row_check(zt + (size_t)i * V, V); if (st) return st; }
    for (int i = 0; i < gamma; ++i) { int st = row_check(zd + (size_t)i * V, V); if (st) return st; }
    if (!(temperature >= 0.0f) || seq_len < gamma) return OR_INVALID_ARG;
    for (int i = 0; i < gamma; ++i) if (x[i] < 0 || x[i] >= V) return OR_INVALID_ARG;
    int n = 0;
    if (temperature == 0.0f) {
        while (n < gamma && x[n] == row_argmax(zt + (size_t)n * V, V)) ++n;
        for (int i = 0; i < n; ++i) tokens[i] = x[i];
        tokens[n] = row_argmax(zt + (size_t)n * V, V);
    } else {
        double T = (double)temperature;
        double* p = (double*)malloc(sizeof(double) * (size_t)V);
        double* q = (double*)malloc(sizeof(double) * (size_t)V);
        int rejected = 0;
        while (n < gamma) {
            row_softmax(zt + (size_t)n * V, V, T, p);
            row_softmax(zd + (size_t)n * V, V, T, q);
            double u = oracle_uniform_at(seed, offset, (uint64_t)n + 1);
            double px = p[x[n]], qx = q[x[n]];
            if (qx > 0.0) {
                double mg = fabs(u - px / qx);
                if (mg < *test_margin) *test_margin = mg;
            }
            if (u * qx < px) { ++n; continue; }
            rejected = 1;
            break;
        }
        double u = oracle_uniform_at(seed, offset, 0);
        if (rejected) {
            /* p, q hold row n */
            double R = 0.0;
            for (int i = 0; i < V; ++i) { double d = p[i] - q[i]; q[i] = d > 0.0 ? d : 0.0; R += q[i]; }
            tokens[n] = draw_id_order(R > 0.0 ? q : p, V, u, draw_margin);
        } else {
            row_softmax(zt + (size_t)gamma * V, V, T, p);
            tokens[n] = draw_id_order(p, V, u, draw_margin);
        }
        for (int i = 0; i < n; ++i) tokens[i] = x[i];
        free(p);
        free(q);
    }
    *n_acc = n;
    *seq_len_out = seq_len - gamma + n;
    return OR_OK;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
