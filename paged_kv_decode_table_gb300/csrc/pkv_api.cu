// pkv_api.cu -- the extern "C" entry points declared in include/pkv.h.
//
// Host-side argument validation, then one or more kernel launches on the
// caller's stream.  Nothing here allocates device memory or synchronises.
#include <cuda_runtime.h>
#include <math.h>

#include "pkv_common.cuh"

namespace pkv {
cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int32_t* block_tables, int max_blocks, const int32_t* seq_lens, int B, int Hkv,
                             int D, int BS, int NB, pkv_dtype dtype, int32_t* status, cudaStream_t stream);
cudaError_t launch_decode_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, int max_blocks, const int32_t* seq_lens, int B,
                                    int Hq, int Hkv, int D, int BS, int NB, float scale, pkv_dtype dtype,
                                    void* workspace, int P, int32_t* status, cudaStream_t stream, bool* used_fast,
                                    const void* k_new, const void* v_new);
size_t decode_workspace_bytes(int B, int Hq, int D, int P);
int device_sm_count();
cudaError_t launch_sampler(int32_t* tokens, const float* logits, int B, int V, const float* temperature,
                           const int32_t* top_k, const float* top_p, const float* min_p, const uint64_t* seeds,
                           const uint64_t* offsets, int32_t* status, cudaStream_t stream);
bool prefill_tc_supported(int Hq, int Hkv, int D, int BS, const void* q, const void* out, const void* k,
                          const void* v);
cudaError_t launch_prefill_tc(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                              const int32_t* q_start, int B, int T_new, int Hq, int Hkv, int BS, int NB, float scale,
                              int32_t* status, cudaStream_t stream);
cudaError_t launch_typical_sampler(int32_t* tokens, const float* logits, int B, int V, const float* temperature,
                                   const float* typical_p, const uint64_t* seeds, const uint64_t* offsets,
                                   int32_t* status, cudaStream_t stream);
cudaError_t launch_logits_processors(float* logits, int B, int V, const uint32_t* mask, const int32_t* row_ptr,
                                     const int32_t* tokens, const int32_t* counts, const float* rep,
                                     const float* freq, const float* pres, int32_t* status, cudaStream_t stream);
size_t spec_verify_workspace_bytes(int B, int gamma);
cudaError_t launch_spec_verify(int32_t* tokens_out, int32_t* n_accepted, int32_t* seq_lens_out, const float* target,
                               const float* draft, const int32_t* draft_tokens, const int32_t* seq_lens, int B,
                               int gamma, int V, const float* temperature, const uint64_t* seeds,
                               const uint64_t* offsets, void* workspace, int32_t* status, cudaStream_t stream);
cudaError_t launch_kv_append_chunk(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                   const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                                   const int32_t* q_start, int B, int T_new, int Hkv, int D, int BS, int NB,
                                   pkv_dtype dtype, int32_t* status, cudaStream_t stream);
cudaError_t launch_prefill_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                                     const int32_t* q_start, int B, int T_new, int Hq, int Hkv, int BS, int NB,
                                     float scale, int32_t* status, cudaStream_t stream);
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int n_pairs,
                               long long block_bytes, int NB, int32_t* status, cudaStream_t stream);
}  // namespace pkv

namespace {
bool dtype_ok(pkv_dtype d) { return d == PKV_F32 || d == PKV_BF16; }
pkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }
}  // namespace

extern "C" {

const char* pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
        case PKV_ERR_DEVICE_BOUNDS: return "PKV_ERR_DEVICE_BOUNDS";
        case PKV_ERR_TIMEOUT: return "PKV_ERR_TIMEOUT";
        case PKV_ERR_NONFINITE: return "PKV_ERR_NONFINITE";
        case PKV_ERR_CAPACITY: return "PKV_ERR_CAPACITY";
        default: return "PKV_ERR_UNKNOWN";
    }
}

int pkv_version(void) { return 100; }

pkv_status pkv_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens, int B, int Hkv,
                         int D, int block_size, int num_blocks, pkv_dtype dtype, int32_t* dev_status, void* stream) {
    if (B < 0 || Hkv < 1 || D < 1 || block_size < 1 || num_blocks < 1 || max_blocks_per_seq < 1 || !dtype_ok(dtype))
        return PKV_ERR_INVALID_ARG;
    if (B == 0) return PKV_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !block_tables || !seq_lens) return PKV_ERR_INVALID_ARG;
    return cuda_status(pkv::launch_kv_append(k_new, v_new, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                             seq_lens, B, Hkv, D, block_size, num_blocks, dtype, dev_status,
                                             static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int n_pairs,
                           int Hkv, int D, int block_size, int num_blocks, pkv_dtype dtype, int32_t* dev_status,
                           void* stream) {
    if (n_pairs < 0 || Hkv < 1 || D < 1 || block_size < 1 || num_blocks < 1 || !dtype_ok(dtype))
        return PKV_ERR_INVALID_ARG;
    if (n_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !src || !dst) return PKV_ERR_INVALID_ARG;
    const long long es = dtype == PKV_F32 ? 4 : 2;
    const long long block_bytes = static_cast<long long>(Hkv) * block_size * D * es;
    return cuda_status(pkv::launch_copy_blocks(k_cache, v_cache, src, dst, n_pairs, block_bytes, num_blocks,
                                               dev_status, static_cast<cudaStream_t>(stream)));
}

size_t pkv_spec_verify_workspace_bytes(int B, int gamma) {
    if (B < 0 || gamma < 0 || gamma > 32) return 0;
    return pkv::spec_verify_workspace_bytes(B, gamma);
}

pkv_status pkv_spec_verify(int32_t* tokens_out, int32_t* n_accepted, int32_t* seq_lens_out, const float* target_logits,
                           const float* draft_logits, const int32_t* draft_tokens, const int32_t* seq_lens, int B,
                           int gamma, int V, const float* temperature, const uint64_t* seeds, const uint64_t* offsets,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
    if (B < 0 || gamma < 0 || gamma > 32 || V < 1 || V > (1 << 23)) return PKV_ERR_INVALID_ARG;
    if (B == 0) return PKV_OK;
    if (!tokens_out || !n_accepted || !seq_lens_out || !target_logits || !seq_lens || !temperature || !seeds ||
        !offsets || !workspace)
        return PKV_ERR_INVALID_ARG;
    if (gamma > 0 && (!draft_logits || !draft_tokens)) return PKV_ERR_INVALID_ARG;
    if (workspace_bytes < pkv::spec_verify_workspace_bytes(B, gamma)) return PKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return PKV_ERR_INVALID_ARG;
    return cuda_status(pkv::launch_spec_verify(tokens_out, n_accepted, seq_lens_out, target_logits, draft_logits,
                                               draft_tokens, seq_lens, B, gamma, V, temperature, seeds, offsets,
                                               workspace, dev_status, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_kv_append_chunk(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                               const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                               const int32_t* q_start, int B, int T_new, int Hkv, int D, int block_size,
                               int num_blocks, pkv_dtype dtype, int32_t* dev_status, void* stream) {
    if (B < 0 || T_new < 0 || Hkv < 1 || D < 1 || block_size < 1 || num_blocks < 1 || max_blocks_per_seq < 1 ||
        !dtype_ok(dtype))
        return PKV_ERR_INVALID_ARG;
    if (B == 0 || T_new == 0) return PKV_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !block_tables || !seq_lens || !q_start) return PKV_ERR_INVALID_ARG;
    return cuda_status(pkv::launch_kv_append_chunk(k_new, v_new, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                                   seq_lens, q_start, B, T_new, Hkv, D, block_size, num_blocks, dtype,
                                                   dev_status, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_paged_prefill_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                       const int32_t* q_start, int B, int T_new, int Hq, int Hkv, int D,
                                       int block_size, int num_blocks, float scale, pkv_dtype dtype,
                                       int32_t* dev_status, void* stream) {
    if (B < 0 || T_new < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || block_size < 1 || num_blocks < 1 ||
        max_blocks_per_seq < 1 || !dtype_ok(dtype))
        return PKV_ERR_INVALID_ARG;
    if (B == 0 || T_new == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !q_start) return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_BF16 || D != 128 || block_size % 16 != 0 || Hq / Hkv > 8) return PKV_ERR_UNSUPPORTED;
    auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!aligned16(k_cache) || !aligned16(v_cache) || (reinterpret_cast<uintptr_t>(q) & 3u) ||
        (reinterpret_cast<uintptr_t>(out) & 3u))
        return PKV_ERR_UNSUPPORTED;
    if (scale <= 0.f) scale = 1.0f / sqrtf(static_cast<float>(D));
    if (pkv::prefill_tc_supported(Hq, Hkv, D, block_size, q, out, k_cache, v_cache))
        return cuda_status(pkv::launch_prefill_tc(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                                  seq_lens, q_start, B, T_new, Hq, Hkv, block_size, num_blocks,
                                                  scale, dev_status, static_cast<cudaStream_t>(stream)));
    return cuda_status(pkv::launch_prefill_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                                     seq_lens, q_start, B, T_new, Hq, Hkv, block_size, num_blocks,
                                                     scale, dev_status, static_cast<cudaStream_t>(stream)));
}

size_t pkv_decode_workspace_bytes(int B, int Hq, int D, int num_sms) {
    if (B < 0 || Hq < 1 || D < 1) return 0;
    const int P = num_sms > 0 ? num_sms : pkv::device_sm_count();
    if (P <= 0) return 0;
    return pkv::decode_workspace_bytes(B, Hq, D, P);
}

pkv_status pkv_paged_decode_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
                                      int B, int Hq, int Hkv, int D, int block_size, int num_blocks, float scale,
                                      pkv_dtype dtype, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                      void* stream) {
    if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 1 || D > 256 || block_size < 1 || num_blocks < 1 ||
        max_blocks_per_seq < 1 || !dtype_ok(dtype))
        return PKV_ERR_INVALID_ARG;
    if (B == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !workspace) return PKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return PKV_ERR_INVALID_ARG;
    const int P = pkv::device_sm_count();
    if (P <= 0) return PKV_ERR_CUDA;
    if (workspace_bytes < pkv::decode_workspace_bytes(B, Hq, D, P)) return PKV_ERR_INVALID_ARG;
    return cuda_status(pkv::launch_decode_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                                    seq_lens, B, Hq, Hkv, D, block_size, num_blocks, scale, dtype,
                                                    workspace, P, dev_status, static_cast<cudaStream_t>(stream),
                                                    nullptr, nullptr, nullptr));
}

pkv_status pkv_paged_decode_attention_append(void* out, const void* q, const void* k_new, const void* v_new,
                                             void* k_cache, void* v_cache, const int32_t* block_tables,
                                             int max_blocks_per_seq, const int32_t* seq_lens, int B, int Hq, int Hkv,
                                             int D, int block_size, int num_blocks, float scale, pkv_dtype dtype,
                                             void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                             void* stream) {
    if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 1 || D > 256 || block_size < 1 || num_blocks < 1 ||
        max_blocks_per_seq < 1 || !dtype_ok(dtype))
        return PKV_ERR_INVALID_ARG;
    if (B == 0) return PKV_OK;
    if (!out || !q || !k_new || !v_new || !k_cache || !v_cache || !block_tables || !seq_lens || !workspace)
        return PKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return PKV_ERR_INVALID_ARG;
    const int P = pkv::device_sm_count();
    if (P <= 0) return PKV_ERR_CUDA;
    if (workspace_bytes < pkv::decode_workspace_bytes(B, Hq, D, P)) return PKV_ERR_INVALID_ARG;
    return cuda_status(pkv::launch_decode_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                                    seq_lens, B, Hq, Hkv, D, block_size, num_blocks, scale, dtype,
                                                    workspace, P, dev_status, static_cast<cudaStream_t>(stream),
                                                    nullptr, k_new, v_new));
}

size_t pkv_sample_workspace_bytes(int B, int V) {
    (void)B;
    (void)V;
    return 0;
}

pkv_status pkv_sample_tokens(int32_t* tokens, const float* logits, int B, int V, const float* temperature,
                             const int32_t* top_k, const float* top_p, const uint64_t* seeds, const uint64_t* offsets,
                             void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
    (void)workspace;
    (void)workspace_bytes;
    if (B < 0 || V < 1 || V > (1 << 23)) return PKV_ERR_INVALID_ARG;
    if (B == 0) return PKV_OK;
    if (!tokens || !logits || !temperature || !top_k || !top_p || !seeds || !offsets) return PKV_ERR_INVALID_ARG;
    return cuda_status(pkv::launch_sampler(tokens, logits, B, V, temperature, top_k, top_p, nullptr, seeds, offsets,
                                           dev_status, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_sample_tokens_ex(int32_t* tokens, const float* logits, int B, int V, const float* temperature,
                                const int32_t* top_k, const float* top_p, const float* min_p, const uint64_t* seeds,
                                const uint64_t* offsets, int32_t* dev_status, void* stream) {
    if (B < 0 || V < 1 || V > (1 << 23)) return PKV_ERR_INVALID_ARG;
    if (B == 0) return PKV_OK;
    if (!tokens || !logits || !temperature || !top_k || !top_p || !seeds || !offsets) return PKV_ERR_INVALID_ARG;
    return cuda_status(pkv::launch_sampler(tokens, logits, B, V, temperature, top_k, top_p, min_p, seeds, offsets,
                                           dev_status, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_sample_tokens_typical(int32_t* tokens, const float* logits, int B, int V, const float* temperature,
                                     const float* typical_p, const uint64_t* seeds, const uint64_t* offsets,
                                     int32_t* dev_status, void* stream) {
    if (B < 0 || V < 1 || V > (1 << 23)) return PKV_ERR_INVALID_ARG;
    if (B == 0) return PKV_OK;
    if (!tokens || !logits || !temperature || !typical_p || !seeds || !offsets) return PKV_ERR_INVALID_ARG;
    return cuda_status(pkv::launch_typical_sampler(tokens, logits, B, V, temperature, typical_p, seeds, offsets,
                                                   dev_status, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_apply_logits_processors(float* logits, int B, int V, const uint32_t* allow_mask,
                                       const int32_t* row_ptr, const int32_t* tokens, const int32_t* counts,
                                       const float* repetition, const float* frequency, const float* presence,
                                       int32_t* dev_status, void* stream) {
    if (B < 0 || V < 1 || V > (1 << 23)) return PKV_ERR_INVALID_ARG;
    if (B == 0 || (!allow_mask && !row_ptr)) return PKV_OK;
    if (!logits || (row_ptr && (!tokens || !counts))) return PKV_ERR_INVALID_ARG;
    return cuda_status(pkv::launch_logits_processors(logits, B, V, allow_mask, row_ptr, tokens, counts, repetition,
                                                     frequency, presence, dev_status,
                                                     static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
