// kv_append.cu -- write each running sequence's new K/V token into its paged block.
//
// Follows the lab's KV state manager ("Bai Lab tong hop -- Inference
// Engineering", block [6], KVPool.write): the token at position pos lives in
// physical block blocks[pos // block_size], slot pos % block_size, for every head;
// pools are [num_blocks, Hkv, block_size, D].  seq_lens is the length after the
// append, so the new token goes to position L - 1.
//
// One warp per (sequence, KV head) row; lanes move 16-byte vectors when the row
// is 16-byte aligned, else elements.  The kernel is a pure bit copy and is
// latency-bound (a few MB per step); HBM bytes are 2 x (read + write) per row.
// Launched with programmatic stream serialisation, so it can start while its
// predecessor drains and the attention kernel after it can start its prologue
// while it runs; each waits (griddepcontrol.wait) before touching data.
#include "pkv_common.cuh"

namespace pkv {

constexpr int kAppendWarps = 8;

template <typename T>
__global__ void __launch_bounds__(kAppendWarps * 32)
    kv_append_kernel(const T* __restrict__ k_new, const T* __restrict__ v_new, T* __restrict__ k_cache,
                     T* __restrict__ v_cache, const int32_t* __restrict__ block_tables, int max_blocks,
                     const int32_t* __restrict__ seq_lens, int B, int Hkv, int D, int BS, int NB,
                     int vec_ok, int32_t* status) {
    // launched as a programmatic dependent: wait for the predecessor's writes
    // (new K/V, lengths, tables), then let the next kernel start its prologue
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = static_cast<int>(blockIdx.x) * kAppendWarps + warp;  // b * Hkv + h
    if (row >= B * Hkv) return;
    const int b = row / Hkv, h = row - b * Hkv;
    const int L = seq_lens[b];
    if (L < 1 || static_cast<long long>(L) > static_cast<long long>(max_blocks) * BS) {
        if (lane == 0) report(status, PKV_ERR_DEVICE_BOUNDS);
        return;
    }
    const int pos = L - 1;
    const int blk = block_tables[static_cast<long long>(b) * max_blocks + pos / BS];
    if (blk < 0 || blk >= NB) {
        if (lane == 0) report(status, PKV_ERR_DEVICE_BOUNDS);
        return;
    }
    const long long dst = ((static_cast<long long>(blk) * Hkv + h) * BS + pos % BS) * D;
    const long long src = static_cast<long long>(row) * D;
    if (vec_ok) {
        constexpr int kPerVec = 16 / sizeof(T);
        const int nvec = D / kPerVec;
        const int4* ks = reinterpret_cast<const int4*>(k_new + src);
        const int4* vs = reinterpret_cast<const int4*>(v_new + src);
        int4* kd = reinterpret_cast<int4*>(k_cache + dst);
        int4* vd = reinterpret_cast<int4*>(v_cache + dst);
        for (int i = lane; i < nvec; i += 32) {
            kd[i] = __ldg(ks + i);
            vd[i] = __ldg(vs + i);
        }
    } else {
        for (int i = lane; i < D; i += 32) {
            k_cache[dst + i] = k_new[src + i];
            v_cache[dst + i] = v_new[src + i];
        }
    }
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int32_t* block_tables, int max_blocks, const int32_t* seq_lens, int B,
                             int Hkv, int D, int BS, int NB, pkv_dtype dtype, int32_t* status,
                             cudaStream_t stream) {
    const size_t es = dtype == PKV_F32 ? 4 : 2;
    auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const int vec_ok = ((D * es) % 16 == 0) && aligned16(k_new) && aligned16(v_new) && aligned16(k_cache) &&
                       aligned16(v_cache);
    const long long rows = static_cast<long long>(B) * Hkv;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + kAppendWarps - 1) / kAppendWarps), 1, 1);
    cfg.blockDim = dim3(kAppendWarps * 32, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err;
    if (dtype == PKV_F32) {
        err = cudaLaunchKernelEx(&cfg, kv_append_kernel<float>, static_cast<const float*>(k_new),
                                 static_cast<const float*>(v_new), static_cast<float*>(k_cache),
                                 static_cast<float*>(v_cache), block_tables, max_blocks, seq_lens, B, Hkv, D, BS, NB,
                                 vec_ok, status);
    } else {
        err = cudaLaunchKernelEx(&cfg, kv_append_kernel<__nv_bfloat16>, static_cast<const __nv_bfloat16*>(k_new),
                                 static_cast<const __nv_bfloat16*>(v_new), static_cast<__nv_bfloat16*>(k_cache),
                                 static_cast<__nv_bfloat16*>(v_cache), block_tables, max_blocks, seq_lens, B, Hkv, D,
                                 BS, NB, vec_ok, status);
    }
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace pkv
