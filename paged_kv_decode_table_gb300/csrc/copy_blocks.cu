// copy_blocks.cu -- copy whole physical KV blocks (the copy half of copy-on-write).
//
// "LLM inference serving tutorial", section 4.2: physical blocks are shared by
// reference count between sequences with a common prefix or between beam
// branches; when a shared, still-writable tail block has to diverge, the block
// is copied and the writer's table is pointed at the copy instead of writing
// into the shared block.  "Suy luan & Toi uu hoa (Inference)" 3.2 describes the
// same sharing of prefix pages.  This kernel performs the copies a step needs:
// for each pair i, block dst[i] of both pools becomes a bit copy of block
// src[i] (all KV heads, all slots).
//
// In the [NB, Hkv, BS, D] layout a block is one contiguous run of
// Hkv * BS * D elements per pool, so a pair is two contiguous memcpys.  The
// grid has one CTA per (pair, pool, chunk of kChunk bytes); each thread moves
// 16-byte vectors, four in flight.  HBM-bound: bytes = 2 x (read + write) per
// pool and pair.
#include "pkv_common.cuh"

namespace pkv {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
constexpr long long kChunk = static_cast<long long>(kCopyThreads) * kCopyUnroll * 16;  // 16 KB per CTA

__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                       const int32_t* __restrict__ src, const int32_t* __restrict__ dst, int n_pairs,
                       long long block_bytes, int chunks, int NB, int vec_ok, int32_t* status) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long unit = blockIdx.x;  // (pair, pool, chunk)
    const int chunk = static_cast<int>(unit % chunks);
    const long long pp = unit / chunks;
    const int pool = static_cast<int>(pp & 1);
    const int i = static_cast<int>(pp >> 1);
    if (i >= n_pairs) return;
    const int s = src[i], d = dst[i];
    if (s < 0 || s >= NB || d < 0 || d >= NB) {
        if (threadIdx.x == 0 && chunk == 0 && pool == 0) report(status, PKV_ERR_DEVICE_BOUNDS);
        return;
    }
    uint8_t* base = pool ? v_cache : k_cache;
    const uint8_t* from = base + static_cast<long long>(s) * block_bytes;
    uint8_t* to = base + static_cast<long long>(d) * block_bytes;
    const long long c0 = chunk * kChunk;
    const long long c1 = min(block_bytes, c0 + kChunk);
    if (vec_ok) {
        const int4* f4 = reinterpret_cast<const int4*>(from);
        int4* t4 = reinterpret_cast<int4*>(to);
        const long long v0 = c0 / 16, v1 = c1 / 16;
        int4 r[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const long long v = v0 + threadIdx.x + static_cast<long long>(u) * kCopyThreads;
            if (v < v1) r[u] = __ldg(f4 + v);
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const long long v = v0 + threadIdx.x + static_cast<long long>(u) * kCopyThreads;
            if (v < v1) t4[v] = r[u];
        }
    } else {
        for (long long b = c0 + threadIdx.x; b < c1; b += kCopyThreads) to[b] = from[b];
    }
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int n_pairs,
                               long long block_bytes, int NB, int32_t* status, cudaStream_t stream) {
    auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const int vec_ok = (block_bytes % 16 == 0) && aligned16(k_cache) && aligned16(v_cache);
    const long long chunks = (block_bytes + kChunk - 1) / kChunk;
    const long long grid = static_cast<long long>(n_pairs) * 2 * chunks;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kCopyThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err = cudaLaunchKernelEx(&cfg, copy_blocks_kernel, static_cast<uint8_t*>(k_cache),
                                         static_cast<uint8_t*>(v_cache), src, dst, n_pairs, block_bytes,
                                         static_cast<int>(chunks), NB, vec_ok, status);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace pkv
