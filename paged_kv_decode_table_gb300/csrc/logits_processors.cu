// logits_processors.cu -- constraint masks and repetition / frequency /
// presence penalties, applied in place to a logits batch before the sampler.
//
// "LLM inference serving tutorial" section 3.1 fixes the pipeline order (hard
// constraints, then penalties, then temperature and the truncation filters),
// 3.2 the penalties (z - a_f c - a_p [c > 0]; the sign-aware repetition
// penalty z / r for z > 0 and r z for z < 0, only on tokens that appeared) and
// 3.3 constrained decoding (an illegal token's logit becomes -inf, then the row
// is sampled as usual).
//
// One kernel, two kinds of CTA per row: mask CTAs each take 256 words of the
// row's bitmask (8192 logits) and write -inf where a bit is clear (the logits
// are not read; each warp reads 32 words, then per word its 32 lanes store the
// word's 32 logits as one coalesced 128-byte masked store); one penalty CTA
// walks the row's (token, count) list.  A
// penalised token is skipped when its mask bit is clear or its logit is not
// finite, so the two kinds write disjoint elements and need no ordering.  The
// penalty arithmetic is double precision, each operation rounded on its own (no
// fused multiply-add), with one rounding to float at the end (a handful of
// tokens per row).
#include <math.h>

#include "pkv_common.cuh"

namespace pkv {

constexpr int kProcThreads = 256;
constexpr int kMaskWordsPerCta = kProcThreads;  // one 32-bit word per thread

__global__ void __launch_bounds__(kProcThreads)
    logits_processors_kernel(float* __restrict__ logits, int V, int mask_ctas, const uint32_t* __restrict__ mask,
                             const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ tokens,
                             const int32_t* __restrict__ counts, const float* __restrict__ rep,
                             const float* __restrict__ freq, const float* __restrict__ pres, int32_t* status) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int per_row = mask_ctas + 1;
    const int b = blockIdx.x / per_row, part = blockIdx.x - (blockIdx.x / per_row) * per_row;
    float* z = logits + static_cast<size_t>(b) * V;
    const int words = (V + 31) / 32;
    const uint32_t* mrow = mask ? mask + static_cast<size_t>(b) * words : nullptr;
    if (part < mask_ctas) {
        if (!mrow) return;
        const int lane = threadIdx.x & 31;
        const int w0 = part * kMaskWordsPerCta + (threadIdx.x & ~31);  // the warp's first word
        if (w0 >= words) return;                                        // warp-uniform
        const int w = w0 + lane;
        const uint32_t mine = w < words ? mrow[w] : 0xffffffffu;
        uint32_t todo = __ballot_sync(0xffffffffu, mine != 0xffffffffu);  // words with a clear bit
        while (todo) {
            const int j = __ffs(todo) - 1;
            todo &= todo - 1u;
            const uint32_t bits = __shfl_sync(0xffffffffu, mine, j);
            const int i = 32 * (w0 + j) + lane;
            if (!((bits >> lane) & 1u) && i < V) z[i] = -INFINITY;
        }
        return;
    }
    if (!row_ptr) return;
    const double r = rep ? static_cast<double>(rep[b]) : 1.0;
    const double f = freq ? static_cast<double>(freq[b]) : 0.0;
    const double pr = pres ? static_cast<double>(pres[b]) : 0.0;
    if (!(r > 0.0)) {
        if (threadIdx.x == 0) report(status, PKV_ERR_INVALID_ARG);
        return;
    }
    for (int e = row_ptr[b] + threadIdx.x; e < row_ptr[b + 1]; e += kProcThreads) {
        const int t = tokens[e], c = counts[e];
        if (t < 0 || t >= V) {
            report(status, PKV_ERR_INVALID_ARG);
            continue;
        }
        if (c < 1) continue;
        if (mrow && !((mrow[t >> 5] >> (t & 31)) & 1u)) continue;  // banned: the mask CTA writes -inf
        const float z0 = z[t];
        if (!isfinite(z0)) continue;
        double zd = static_cast<double>(z0);
        if (r != 1.0) zd = zd > 0.0 ? zd / r : (zd < 0.0 ? zd * r : zd);
        zd = __dsub_rn(zd, __dmul_rn(f, static_cast<double>(c)));  // no fused multiply-add
        zd = __dsub_rn(zd, pr);
        z[t] = static_cast<float>(zd);
    }
}

cudaError_t launch_logits_processors(float* logits, int B, int V, const uint32_t* mask, const int32_t* row_ptr,
                                     const int32_t* tokens, const int32_t* counts, const float* rep,
                                     const float* freq, const float* pres, int32_t* status, cudaStream_t stream) {
    const int words = (V + 31) / 32;
    const int mask_ctas = mask ? (words + kMaskWordsPerCta - 1) / kMaskWordsPerCta : 0;
    const long long grid = static_cast<long long>(B) * (mask_ctas + 1);
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kProcThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err = cudaLaunchKernelEx(&cfg, logits_processors_kernel, logits, V, mask_ctas, mask, row_ptr, tokens,
                                         counts, rep, freq, pres, status);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace pkv
