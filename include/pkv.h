/*
 * pkv.h -- C ABI of the paged-KV decode step for GB300 (sm_103a).
 *
 * One batched decode iteration over a paged KV cache, in three calls:
 *   pkv_kv_append               write each sequence's new K/V token into its
 *                               physical block through the block table;
 *   pkv_paged_decode_attention  GQA decode attention for one query token per
 *                               sequence over all cached K/V (split-KV inside);
 *                               pkv_paged_decode_attention_append does the
 *                               append and the attention in one call;
 *   pkv_sample_tokens           temperature -> top-k -> renormalise -> top-p ->
 *                               renormalise -> seeded per-request draw.
 * Shared prefixes: a host-side reference-counted block pool (pkv_block_pool_*,
 * pkv_seq_*) hands out block ids and reports the copy-on-write pairs that
 * pkv_copy_blocks copies on the GPU before the step's append.
 * Chunked prefill: pkv_kv_append_chunk and pkv_paged_prefill_attention.
 * Speculative decoding: pkv_spec_verify accepts or rejects draft tokens,
 * draws the correction or bonus token and returns the rolled-back lengths.
 *
 * Conventions shared by every call
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise.  The
 *    caller allocates and owns every buffer; the library allocates nothing,
 *    keeps no per-call state and never synchronises the stream.  All work is
 *    enqueued on `stream` (a cudaStream_t passed as void*; NULL = legacy
 *    default stream) in call order.
 *  - Host-detectable errors (null pointers, unsupported shapes, undersized
 *    workspace, misaligned pointers) return before anything is launched.
 *    B == 0 is a no-op returning PKV_OK.
 *  - Data-dependent problems found on the device (a block id outside
 *    [0, num_blocks), a sequence length outside the table, a NaN/+inf logit, an
 *    all -inf row, T < 0, top_p <= 0) never trap: the kernel records the first
 *    such code into *dev_status with an atomic compare-and-swap from 0, writes
 *    a defined value for the affected unit (zeros for attention rows, token -1
 *    for sampler rows) and carries on.  dev_status may be NULL to skip the
 *    report.  Read it after the stream has synchronised.
 *  - Layouts are row-major and dense:
 *      KV pools   k_cache, v_cache : [num_blocks, Hkv, block_size, D]
 *      new K/V    k_new, v_new     : [B, Hkv, D]
 *      queries    q                : [B, Hq, D]      output out: [B, Hq, D]
 *      tables     block_tables     : int32 [B, max_blocks_per_seq]
 *      lengths    seq_lens         : int32 [B], length AFTER this step's append
 *      logits                      : float32 [B, V]
 *
 * Sources (web pages, cited by title and section):
 *  [LAB]   "Bai Lab tong hop -- Inference Engineering", block [6] KV state
 *          manager (KVPool.write / gather), block [5] forward, block [8] sample.
 *  [CH5]   "Suy luan & Toi uu hoa (Inference)", chapter 5: 1.2 temperature /
 *          top-k / nucleus set and renormalisation; 3.1 GQA; 3.2 PagedAttention
 *          block table; 4.1 online softmax.
 *  [SERVE] "LLM inference serving tutorial": 3.1 sampler definitions and tie
 *          rules; 1.6 per-request RNG streams; appendix A [D01]/[D02].
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* host: bad pointer/shape/size; device: T < 0 or top_p <= 0 */
    PKV_ERR_UNSUPPORTED = 2,   /* host: a shape the library has no kernel for */
    PKV_ERR_CUDA = 3,          /* host: a CUDA runtime call or launch failed */
    PKV_ERR_DEVICE_BOUNDS = 4, /* device: block id or sequence length out of range */
    PKV_ERR_TIMEOUT = 5,       /* device: a bounded wait ran out (kernel returned early) */
    PKV_ERR_NONFINITE = 6,     /* device: NaN / +inf logit, or no finite logit in a row */
    PKV_ERR_CAPACITY = 7       /* host: the block pool has too few free blocks */
} pkv_status;

typedef enum { PKV_F32 = 0, PKV_BF16 = 1 } pkv_dtype;

/* Human-readable name of a status code (static string; never NULL). */
const char* pkv_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int pkv_version(void);

/*
 * KV append ([LAB] block [6] KVPool.write; [CH5] 3.2).
 * For every sequence b and KV head h: pos = seq_lens[b] - 1,
 * blk = block_tables[b][pos / block_size], slot = pos % block_size, and
 *   k_cache[blk][h][slot][:] = k_new[b][h][:],  v_cache[...] = v_new[b][h][:].
 * Bit copy (no arithmetic).  A sequence needs 1 <= seq_lens[b] <=
 * max_blocks_per_seq * block_size and a block id in [0, num_blocks); otherwise
 * it is skipped and PKV_ERR_DEVICE_BOUNDS is recorded.  Two sequences that map
 * the same slot race (the caller's tables must not alias a written slot).
 * dtype: element type of k_new/v_new/k_cache/v_cache.
 */
pkv_status pkv_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* seq_lens, int B, int Hkv, int D, int block_size,
                         int num_blocks, pkv_dtype dtype, int32_t* dev_status, void* stream);

/*
 * Workspace bytes pkv_paged_decode_attention needs for batch B, Hq query heads
 * and head dim D on a device with num_sms SMs (num_sms <= 0: the current
 * device): 16 bytes per sequence (where its blocks fall in the split) plus two
 * partial-result slots per SM of (max, sum, output[D]) float32 for every query
 * head, merged by the combine kernel; about 5 MiB for Hq = 32, D = 128 on 152
 * SMs.  Returns 0 on error.  Pure host arithmetic when num_sms > 0.
 */
size_t pkv_decode_workspace_bytes(int B, int Hq, int D, int num_sms);

/*
 * GQA paged decode attention, one query token per sequence ([LAB] block [5];
 * [CH5] 3.1, 3.2, 4.1).  For query head qh of sequence b, with KV head
 * h = qh / (Hq / Hkv) and L = seq_lens[b]:
 *   s_j = scale * <q[b][qh], K_j>  for j < L, K_j/V_j read through the table;
 *   out[b][qh] = sum_j softmax(s)_j V_j        (L == 0 gives zeros).
 * scale <= 0 selects 1/sqrt(D).  Accumulation is float32; the result is written
 * in `dtype`.  Long sequences are cut into balanced chunks across all SMs and
 * merged with the online-softmax rule; `workspace` (device, >=
 * pkv_decode_workspace_bytes(B, Hq, D, 0) bytes, 16-byte aligned, contents
 * ignored on entry) holds the partials.  Requires Hq % Hkv == 0 and
 * 1 <= D <= 256; the fast path (bf16, D = 128, block_size a multiple of 16,
 * 1 <= Hkv <= 8, Hq/Hkv <= 16, Hkv * block_size <= 256 with at least two
 * 512*Hkv*block_size-byte stages fitting in shared memory, 16-byte aligned q,
 * out and pools) uses TMA and tensor-core MMA in two kernels (split-KV, then the
 * combine) chained by programmatic dependent launch; other shapes use a generic CUDA-core kernel.  Sequences with a length outside [0, max_blocks_per_seq*block_size]
 * or a block id outside [0, num_blocks) get zero output and
 * PKV_ERR_DEVICE_BOUNDS.  The KV slots past L in a sequence's last block are
 * never used (their contents may be anything, NaN included).
 */
pkv_status pkv_paged_decode_attention(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* seq_lens, int B,
                                      int Hq, int Hkv, int D, int block_size, int num_blocks,
                                      float scale, pkv_dtype dtype, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * KV append and decode attention in one call: the same result (caches, out,
 * dev_status) as pkv_kv_append(k_new, v_new, k_cache, v_cache, ...) followed by
 * pkv_paged_decode_attention(out, q, k_cache, v_cache, ...) on the same stream,
 * with the arguments of both.  On the fast path (as for
 * pkv_paged_decode_attention, plus 16-byte aligned k_new and v_new) the
 * attention kernel writes each sequence's new token into its last block just
 * before loading that block, which saves the separate append launch and its
 * pass over the batch; elsewhere the two kernels run back to back.
 * Precondition (which copy-on-write guarantees): the block that receives a
 * sequence's new token is not read by another sequence of the same batch.
 * Lengths outside [1, max_blocks_per_seq*block_size] record
 * PKV_ERR_DEVICE_BOUNDS, as the append does.  k_cache and v_cache are written.
 */
pkv_status pkv_paged_decode_attention_append(void* out, const void* q, const void* k_new,
                                             const void* v_new, void* k_cache, void* v_cache,
                                             const int32_t* block_tables, int max_blocks_per_seq,
                                             const int32_t* seq_lens, int B, int Hq, int Hkv, int D,
                                             int block_size, int num_blocks, float scale,
                                             pkv_dtype dtype, void* workspace,
                                             size_t workspace_bytes, int32_t* dev_status,
                                             void* stream);

/*
 * pkv_paged_decode_attention without a caller-supplied workspace.  The pages
 * have no counterpart to this call: it exists for callers that cannot allocate
 * device memory at attention time (a serving loop that handed all free HBM to
 * its KV pool at start-up, code that must not risk the implicit device
 * synchronisation of an allocation, or a C host program with no allocator).
 * Same arguments, semantics and results as pkv_paged_decode_attention; the
 * split-KV workspace is instead a fixed 16 MiB device array inside the library,
 * present on every GPU that loads it until the process exits.  Every call looks
 * up that array's device address on the current device (cudaGetSymbolAddress;
 * the first lookup on a device loads the library's module there), so make the
 * first call on each device before any stream capture.  Requests that
 * would need more than 16 MiB of workspace (pkv_decode_workspace_bytes(B, Hq, D,
 * 0) > 16 MiB; Hq = 32, D = 128 needs about 5 MiB on 152 SMs) return
 * PKV_ERR_UNSUPPORTED and launch nothing.  Nothing is allocated or freed.  All
 * calls share the one array: calls that can overlap on the GPU (different
 * streams without ordering, or different host threads) race and corrupt each
 * other's partial results; serialise them on one stream.  The array keeps the
 * last call's contents; every call rewrites what it reads before reading it.
 */
pkv_status pkv_paged_decode_attention_noalloc(void* out, const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* block_tables,
                                              int max_blocks_per_seq, const int32_t* seq_lens, int B,
                                              int Hq, int Hkv, int D, int block_size, int num_blocks,
                                              float scale, pkv_dtype dtype, int32_t* dev_status,
                                              void* stream);

/*
 * Test hook for the failure path of the attention kernels; off by default and
 * not part of the decode step (the pages have no counterpart).  The fast
 * attention kernel waits on its stage barriers with a bounded number of polls
 * (about a second or more by default), after which it records PKV_ERR_TIMEOUT
 * in dev_status and returns instead of hanging.  This call sets, for every
 * later attention call of the process (all threads, all devices):
 *   polls       the poll budget of those waits; 0 restores the default;
 *   silent_cta  one CTA of the split-KV kernel whose loader issues no copy at
 *               all (-1: none), so that its consumers wait on stages nothing
 *               will fill and give up after `polls` polls, with no copy in
 *               flight.
 * With silent_cta >= 0 the output of the sequences that CTA covers is
 * undefined and dev_status reads PKV_ERR_TIMEOUT; the next call after the
 * hook is reset computes normally.  Returns PKV_ERR_INVALID_ARG for
 * silent_cta < -1.  Not synchronised with attention calls on other threads.
 */
pkv_status pkv_test_set_wait_limit(uint32_t polls, int silent_cta);

/*
 * Workspace bytes pkv_sample_tokens needs (B rows of V logits).  The current
 * sampler keeps each row on chip and needs none: returns 0.
 */
size_t pkv_sample_workspace_bytes(int B, int V);

/*
 * Logits -> token, one row per request ([CH5] 1.2; [LAB] block [8];
 * [SERVE] 3.1, 1.6).  Per row b with z = logits[b]:
 *   temperature[b] == 0 : greedy, argmax of z, lowest id among ties.
 *   temperature[b] >  0 : p_i = exp((z_i - max z) / T) over finite z_i (a -inf
 *     logit is a banned token); if 0 < top_k[b] < #finite keep the top_k
 *     largest under the order (z descending, token id ascending); renormalise;
 *     if top_p[b] < 1 keep the smallest prefix of that order whose cumulative
 *     probability is >= top_p[b] (boundary token kept); renormalise; draw
 *     u = Philox4x64-10(key = (seeds[b], 0), counter = (offsets[b], 0, 0, 0))
 *     word 0, top 53 bits * 2^-53, and return the first kept token, walking
 *     token ids in ascending order, whose running probability exceeds u.
 * temperature, top_p: float32 [B]; top_k: int32 [B] (<= 0 or >= V: off);
 * seeds, offsets: uint64 [B]; tokens: int32 [B] output.  Errors per row (token
 * -1): NaN or +inf logit / no finite logit -> PKV_ERR_NONFINITE; T < 0 (or NaN)
 * or top_p <= 0 (or NaN) -> PKV_ERR_INVALID_ARG.  Exponentials are float32 and
 * the probability masses are accumulated exactly in 64-bit fixed point, so a
 * draw can differ from a float64 evaluation only when u falls within ~1e-6 of a
 * CDF edge (or the top-p cut is within ~1e-6 of p).  Deterministic: the same
 * inputs give the same tokens on every run.  Requires 1 <= V <= 2^23.
 */
pkv_status pkv_sample_tokens(int32_t* tokens, const float* logits, int B, int V,
                             const float* temperature, const int32_t* top_k, const float* top_p,
                             const uint64_t* seeds, const uint64_t* offsets, void* workspace,
                             size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * Copy-on-write block copies ("LLM inference serving tutorial" 4.2; "Suy luan
 * & Toi uu hoa (Inference)" 3.2).  For i in [0, n_pairs): physical block
 * dst[i] of k_cache and of v_cache becomes a bit copy of block src[i] (every KV
 * head, every slot: Hkv * block_size * D elements per pool).  src, dst: device
 * int32 [n_pairs].  The dst ids must be distinct and none may appear among the
 * src ids of the same call (the copies run in parallel); a block id outside
 * [0, num_blocks) skips its pair and records PKV_ERR_DEVICE_BOUNDS.
 * n_pairs == 0 is a no-op.  Bit copy, no arithmetic.
 */
pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int n_pairs,
                           int Hkv, int D, int block_size, int num_blocks, pkv_dtype dtype, int32_t* dev_status,
                           void* stream);

/*
 * Chunked prefill, append half ("Bai Lab tong hop -- Inference Engineering"
 * prefill chunks written with KVPool.write; "LLM inference serving tutorial"
 * 5.4).  Sequence b appends n_b = q_start[b+1] - q_start[b] tokens: rows
 * q_start[b] .. q_start[b+1] - 1 of the packed k_new / v_new [T_new, Hkv, D]
 * (T_new = q_start[B]); seq_lens[b] is the length after the append, so row
 * q_start[b] + i goes to position seq_lens[b] - n_b + i through the table.
 * q_start: device int32 [B + 1], non-decreasing, q_start[0] = 0.  A sequence
 * with seq_lens[b] < n_b or beyond the table, or a block id outside [0,
 * num_blocks), is skipped and PKV_ERR_DEVICE_BOUNDS recorded.  Bit copy.
 */
pkv_status pkv_kv_append_chunk(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                               const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                               const int32_t* q_start, int B, int T_new, int Hkv, int D, int block_size,
                               int num_blocks, pkv_dtype dtype, int32_t* dev_status, void* stream);

/*
 * Chunked prefill, attention half ("Suy luan & Toi uu hoa (Inference)" 2.1;
 * the lab's forward over a prompt chunk; "LLM inference serving tutorial"
 * 5.4): for packed query row t of sequence b (q [T_new, Hq, D], rows laid out
 * as in pkv_kv_append_chunk), at position pos = seq_lens[b] - n_b + (t -
 * q_start[b]), query head qh attends to K/V head qh / (Hq / Hkv) at positions
 * 0 .. pos (causal), read through the table:
 *   out[t][qh] = sum_{j <= pos} softmax_j(scale * <q[t][qh], K_j>) V_j.
 * The chunk's own K/V must already be in the cache (pkv_kv_append_chunk first).
 * scale <= 0 selects 1/sqrt(D).  bf16 only, D = 128, block_size a multiple of
 * 16, Hq / Hkv <= 8, 16-byte aligned pools and 4-byte aligned q / out (else
 * PKV_ERR_UNSUPPORTED).  fp32 accumulation.  With 16-byte aligned q / out:
 * one CTA per (two tiles of up to 128 rows of chunk tokens x query heads, KV
 * head), the longest key ranges first, with tcgen05 MMAs and TMEM
 * accumulators; otherwise one CTA per (16 chunk tokens, KV head) with
 * mma.sync.  A sequence with an invalid length or block id gets zero output
 * and PKV_ERR_DEVICE_BOUNDS.
 */
pkv_status pkv_paged_prefill_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                       const int32_t* q_start, int B, int T_new, int Hq, int Hkv, int D,
                                       int block_size, int num_blocks, float scale, pkv_dtype dtype,
                                       int32_t* dev_status, void* stream);

/*
 * pkv_sample_tokens with min-p ("LLM inference serving tutorial" 3.1, Q4):
 * after top-p, a token stays in the support only if its probability is at
 * least min_p[b] times the largest one, i.e. its weight 2^((z - zmax) log2(e) /
 * T) is >= min_p[b] (taken in 2^-40 fixed point: mass >= ceil(min_p * 2^40));
 * the most probable token always stays.  min_p: float32 [B], or NULL (off);
 * min_p[b] <= 0 turns it off for row b; NaN or > 1 is PKV_ERR_INVALID_ARG
 * (token -1).  Everything else as pkv_sample_tokens (no workspace).
 */
pkv_status pkv_sample_tokens_ex(int32_t* tokens, const float* logits, int B, int V, const float* temperature,
                                const int32_t* top_k, const float* top_p, const float* min_p, const uint64_t* seeds,
                                const uint64_t* offsets, int32_t* dev_status, void* stream);

/*
 * Typical sampling ("LLM inference serving tutorial" 3.1, other samplers;
 * Meister et al., locally typical sampling): for row b with T = temperature[b]
 * > 0 and tau = typical_p[b] < 1, p = softmax(z / T) over the finite logits,
 * H(p) = -sum p_i ln p_i, and the kept set is the smallest prefix of the tokens
 * in ascending d_i = |-ln p_i - H(p)| whose probability reaches tau (boundary
 * token kept), renormalised and drawn in token-id order with the same Philox
 * uniform as pkv_sample_tokens (key (seeds[b], 0), counter (offsets[b], 0, 0,
 * 0)).  Since -ln p_i - H = ln 2 (ubar - u_i) with u_i = (z_i - zmax) log2(e) / T
 * and ubar the p-weighted mean of u, the order is taken as |u_i - ubar| in
 * float32 (u_i = (z_i - zmax) * min(log2(e) / T, 1e30), each operation rounded
 * on its own) with ubar rounded to a multiple of 2^-8; ties go to the larger
 * u_i, then to the smaller id.  T == 0 is greedy (lowest id among equal
 * maxima); tau >= 1 keeps every finite logit.  tokens: device int32 [B];
 * logits: device float32 [B, V] row-major (-inf = banned); temperature,
 * typical_p: device float32 [B]; seeds, offsets: device uint64 [B].  Errors
 * (token -1 for the row, status recorded): NaN / +inf / no finite logit ->
 * PKV_ERR_NONFINITE; T < 0 or NaN, or T > 0 with tau <= 0 or NaN ->
 * PKV_ERR_INVALID_ARG.  Host: B < 0, V < 1 or V > 2^23, NULL pointers ->
 * PKV_ERR_INVALID_ARG.  One thread-block cluster of 1-8 CTAs per row (as many
 * as fill the device with one CTA per SM); no workspace, nothing allocated.
 */
pkv_status pkv_sample_tokens_typical(int32_t* tokens, const float* logits, int B, int V, const float* temperature,
                                     const float* typical_p, const uint64_t* seeds, const uint64_t* offsets,
                                     int32_t* dev_status, void* stream);

/*
 * Logits processors, in place on logits float32 [B, V], in the order of the
 * "LLM inference serving tutorial" 3.1 pipeline (before temperature and the
 * filters of pkv_sample_tokens):
 *  1. constraint mask (3.3): allow_mask uint32 [B, ceil(V/32)] or NULL; token
 *     i of row b is allowed iff bit i % 32 of word i / 32 is set, else its
 *     logit becomes -inf;
 *  2. penalties (3.2) on the tokens listed for row b in CSR form (row_ptr int32
 *     [B + 1] or NULL, tokens / counts int32 [row_ptr[B]], each token at most
 *     once per row) with count c >= 1, an allowed mask bit and a finite logit:
 *     the sign-aware repetition penalty r = repetition[b] (z / r for z > 0,
 *     r * z for z < 0, 0 unchanged; r == 1 is a no-op), then
 *     z - frequency[b] * c - presence[b]; computed in double, each operation
 *     rounded on its own, then rounded once to float.
 * repetition / frequency / presence: float32 [B] or NULL (off).  Errors: a
 * listed token outside [0, V) (that entry skipped) or repetition <= 0 / NaN
 * (that row's penalties skipped) -> PKV_ERR_INVALID_ARG in dev_status.
 */
pkv_status pkv_apply_logits_processors(float* logits, int B, int V, const uint32_t* allow_mask,
                                       const int32_t* row_ptr, const int32_t* tokens, const int32_t* counts,
                                       const float* repetition, const float* frequency, const float* presence,
                                       int32_t* dev_status, void* stream);

/*
 * Workspace bytes pkv_spec_verify needs: 32 bytes per logits row,
 * B * (2 * gamma + 1) rows.  Pure host arithmetic.
 */
size_t pkv_spec_verify_workspace_bytes(int B, int gamma);

/*
 * Speculative-decoding verification ("Suy luan & Toi uu hoa (Inference)" 5.2;
 * "LLM inference serving tutorial" section 7 and Q16).  Per request b with
 * gamma draft tokens x_i (draft_tokens int32 [B, gamma]), the target model's
 * logits at the gamma draft positions and the next one (target_logits fp32
 * [B, gamma + 1, V]) and the draft model's logits at the draft positions
 * (draft_logits fp32 [B, gamma, V]):
 *   p_i = softmax(target_logits[b][i] / T), q_i = softmax(draft_logits[b][i] / T)
 *   over finite logits, T = temperature[b].
 *   T == 0: x_i is accepted while it is the target argmax of row i (lowest id
 *     among ties); the next token is the argmax of the first rejected row (row
 *     gamma when every draft is accepted).
 *   T > 0: u_i = Philox4x64-10(key (seeds[b], 0), counter (offsets[b], i + 1,
 *     0, 0)) word 0, top 53 bits * 2^-53; x_i is accepted iff u_i * q_i(x_i) <
 *     p_i(x_i), in order, up to the first rejection n.  The next token is drawn
 *     with u = the same generator at counter (offsets[b], 0, 0, 0), walking ids
 *     in ascending order: from max(0, p_n - q_n) normalised (p_n if that is all
 *     zero) when n < gamma, else from p_{gamma+1}.
 * Outputs (device): tokens_out int32 [B, gamma + 1] = the accepted drafts, the
 * drawn token, then -1; n_accepted int32 [B]; seq_lens_out int32 [B] =
 * seq_lens[b] - gamma + n_accepted[b], where seq_lens counts the gamma draft
 * positions whose KV the target pass appended (the rejected ones are rolled
 * back).  Probabilities are float32 exponentials with exact 2^-40 fixed-point
 * row sums; a decision can differ from a float64 evaluation only when u lies
 * within ~1e-6 of p/q or of a CDF edge.  Errors per request (tokens -1,
 * n_accepted 0, seq_lens_out = seq_lens): NaN / +inf logit or a row without a
 * finite logit -> PKV_ERR_NONFINITE; T < 0 or NaN, a draft token outside
 * [0, V), seq_lens < gamma -> PKV_ERR_INVALID_ARG.  0 <= gamma <= 32,
 * 1 <= V <= 2^23; workspace >= pkv_spec_verify_workspace_bytes(B, gamma).
 */
pkv_status pkv_spec_verify(int32_t* tokens_out, int32_t* n_accepted, int32_t* seq_lens_out,
                           const float* target_logits, const float* draft_logits, const int32_t* draft_tokens,
                           const int32_t* seq_lens, int B, int gamma, int V, const float* temperature,
                           const uint64_t* seeds, const uint64_t* offsets, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, void* stream);

/*
 * Reference-counted block pool (host only; "LLM inference serving tutorial"
 * 4.2, 1.7, appendix A [D07]-[D08]; "Bai Lab tong hop -- Inference
 * Engineering" block [6]).  Owns the ids 0..num_blocks-1 of a KV pool laid out
 * as above; never touches device memory.  Sequences are named by caller-chosen
 * int64 ids.  Every mutating call either succeeds or changes nothing; errors:
 * PKV_ERR_INVALID_ARG (unknown or duplicate sequence, length beyond
 * max_blocks_per_seq * block_size, null pointer), PKV_ERR_CAPACITY (no free
 * block).  Not thread-safe.
 *   create       all blocks free, reference counts 0; NULL on bad sizes.
 *   seq_add      a new sequence of `length` tokens gets ceil(length /
 *                block_size) fresh blocks (count 1 each).
 *   seq_fork     `child` shares every block of `parent` (each count + 1) and
 *                has its length: a common prefix or a beam branch.
 *   seq_append   reserves the slot of one new token at position length: a
 *                fresh block when the position opens a block; when the tail
 *                block is shared (count > 1), a fresh block replaces it in this
 *                sequence's table, the shared block's count drops by one, and
 *                the pair (shared -> fresh) is written to cow_src[0] /
 *                cow_dst[0] with *n_cow = 1 (else *n_cow = 0).  The caller
 *                copies the pairs with pkv_copy_blocks before pkv_kv_append.
 *   seq_free     every block's count drops by one; a block whose count reaches
 *                0 returns to the free list.  Freeing an unknown (or already
 *                freed) sequence is a no-op returning PKV_OK.
 *   block_tables rows of max_blocks_per_seq block ids for seqs[0..n) (host
 *                int32 [n, max_blocks_per_seq], unused entries -1) and their
 *                lengths (host int32 [n]), ready to upload.
 *   num_free / refcount / seq_length report state (-1 on a bad argument).
 */
typedef struct pkv_block_pool pkv_block_pool;
pkv_block_pool* pkv_block_pool_create(int num_blocks, int block_size, int max_blocks_per_seq);
void pkv_block_pool_destroy(pkv_block_pool* pool);
int pkv_block_pool_num_free(const pkv_block_pool* pool);
int pkv_block_pool_refcount(const pkv_block_pool* pool, int block);
pkv_status pkv_seq_add(pkv_block_pool* pool, int64_t seq, int length);
pkv_status pkv_seq_fork(pkv_block_pool* pool, int64_t parent, int64_t child);
pkv_status pkv_seq_append(pkv_block_pool* pool, int64_t seq, int32_t* cow_src, int32_t* cow_dst, int* n_cow);
pkv_status pkv_seq_free(pkv_block_pool* pool, int64_t seq);
int pkv_seq_length(const pkv_block_pool* pool, int64_t seq);
pkv_status pkv_block_tables(const pkv_block_pool* pool, const int64_t* seqs, int n, int32_t* block_tables,
                            int32_t* seq_lens);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
