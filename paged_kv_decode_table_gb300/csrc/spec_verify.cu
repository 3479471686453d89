// spec_verify.cu -- speculative-decoding verification (accept / reject the draft
// tokens of every request, draw the correction or bonus token, roll back KV).
//
// "Suy luan & Toi uu hoa (Inference)" 5.2 (speculative rejection sampling after
// Leviathan & Matias): at draft position i the draft token x_i ~ q_i is kept
// with probability min(1, p_i(x_i) / q_i(x_i)); the first rejection ends the
// cycle with a token drawn from the residual max(0, p_i - q_i) normalised; when
// every draft is kept, one more token comes from p_{gamma+1}.  Greedy decoding
// (T = 0) keeps drafts while they equal the target argmax.  "LLM inference
// serving tutorial" section 7 / Q16: the number of accepted tokens varies per
// request, and the KV written for rejected drafts is rolled back, here by
// returning the committed length seq_len - gamma + n_accepted.
//
// p_i = softmax(z_target[i] / T) and q_i = softmax(z_draft[i] / T) over finite
// logits, represented as in the sampler: fixed-point masses floor(w * 2^40) of
// w = 2^((z - zmax) log2(e) / T).  The row sums for the tests come from one
// pass (a compensated fp32 sum of the weights, relative error ~1e-7); the
// final draw sums its own fixed-point masses exactly.  Uniform
// number j of a request is Philox4x64-10 word 0 at counter (offset, j, 0, 0)
// under key (seed, 0), top 53 bits: j = i + 1 for the test at draft position i,
// j = 0 for the final draw, which walks token ids in ascending order.
//
// Two kernels: row statistics (max, lowest argmax, mass sum in one pass over
// the row, the sum kept relative to a running maximum) with one CTA per logits
// row; then one thread-block cluster per request (1-8 CTAs) for the tests (one
// thread per draft position, in every CTA) and the final draw (chunked inverse
// CDF over the vocabulary, spread over the CTAs' slices).
#include <cooperative_groups.h>
#include <limits.h>
#include <math.h>

#include "pkv_common.cuh"
#include "sampling_math.cuh"

namespace cg = cooperative_groups;

namespace pkv {

constexpr int kVT = 512;             // threads per CTA
constexpr int kVW = kVT / 32;
constexpr int kDrawChunks = 2048;    // chunk sums kept in shared memory
constexpr int kSS = 256;             // threads per CTA of the row statistics (four CTAs per SM)
constexpr int kSSW = kSS / 32;

struct RowStat {   // 32 bytes per logits row
    float zmax;
    int argmax;    // lowest id holding zmax (-1: no finite logit)
    int bad;       // NaN or +inf present
    int pad;
    unsigned long long S;  // ~ 2^40 * sum of 2^((z - zmax) c2) (T > 0), relative error ~1e-7
    unsigned long long pad2;
};

__device__ __forceinline__ float4 load4_row(const float* row, int e, int n, bool al) {
    if (al && e + 4 <= n) return __ldg(reinterpret_cast<const float4*>(row + e));
    float4 q;
    q.x = e < n ? row[e] : -INFINITY;
    q.y = e + 1 < n ? row[e + 1] : -INFINITY;
    q.z = e + 2 < n ? row[e + 2] : -INFINITY;
    q.w = e + 3 < n ? row[e + 3] : -INFINITY;
    return q;
}

// ------------------------------------------------------------------ row statistics
// Row r of request b: r < gamma + 1 is target row r, else draft row r - gamma - 1.
// One 256-thread CTA per row, four per SM, so that a batch of up to 4 x #SM rows
// (64 requests with 4 drafts: 576) streams in one wave.
__global__ void __launch_bounds__(kSS, 4)
    spec_stats_kernel(const float* __restrict__ target, const float* __restrict__ draft, int gamma, int V,
                      const float* __restrict__ temperature, RowStat* __restrict__ stats) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ float smax[kSSW];
    __shared__ int sid[kSSW], sbad[kSSW];
    __shared__ unsigned long long ured[kSSW];
    const int rows = 2 * gamma + 1;
    const int b = blockIdx.x / rows, r = blockIdx.x - (blockIdx.x / rows) * rows;
    const float* row = r <= gamma ? target + (static_cast<size_t>(b) * (gamma + 1) + r) * V
                                  : draft + (static_cast<size_t>(b) * gamma + (r - gamma - 1)) * V;
    const bool al = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(row) & 15u) == 0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float T = temperature[b];
    const bool sum = T > 0.f;
    const float c2 = sum ? fminf(1.4426950408889634f / T, 1.0e30f) : 0.f;
    // one pass: running maximum (lowest id among equals) and the sum of the
    // weights 2^((z - m) c2) relative to it, compensated (Kahan) in fp32.  The
    // thread takes its logits in batches of 32; a batch's maximum is found
    // first, the sum so far is rescaled to it if it is larger (at most once per
    // batch), then the batch's weights are added.
    constexpr int kU = 8;  // float4 slots per batch
    float m = -INFINITY;
    int id = INT_MAX;
    int bad = 0;
    float ks = 0.f, kc = 0.f;  // the sum and its running compensation
    for (int e0 = 4 * tid; e0 < V; e0 += 4 * kSS * kU) {
        float4 q[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) q[u] = load4_row(row, e0 + 4 * kSS * u, V, al);
        float bm = -INFINITY;
        int bid = INT_MAX;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const float zz[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                bad |= (zz[j] < INFINITY) ? 0 : 1;  // NaN or +inf (slots past V read -inf)
                if (zz[j] > bm) {                   // ids grow within a batch: first max wins
                    bm = zz[j];
                    bid = e0 + 4 * kSS * u + j;
                }
            }
        }
        if (bm > m) {  // earlier batches hold lower ids, so an equal maximum keeps id
            if (sum && ks != 0.f) {
                const float sc = hw_exp2((m - bm) * c2);
                ks *= sc;
                kc *= sc;
            }
            m = bm;
            id = bid;
        }
        if (sum && m > -INFINITY) {
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const float zz[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float y = weight(zz[j], m, c2) - kc;
                    const float t = ks + y;
                    kc = (t - ks) - y;
                    ks = t;
                }
            }
        }
    }
    const float mt = m;  // this thread's maximum, the reference of acc
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const int id2 = __shfl_xor_sync(0xffffffffu, id, o);
        if (m2 > m || (m2 == m && id2 < id)) {
            m = m2;
            id = id2;
        }
        bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    if (lane == 0) {
        smax[warp] = m;
        sid[warp] = id;
        sbad[warp] = bad;
    }
    __syncthreads();
    m = smax[0];
    id = sid[0];
    bad = sbad[0];
    for (int w = 1; w < kSSW; ++w) {
        if (smax[w] > m || (smax[w] == m && sid[w] < id)) {
            m = smax[w];
            id = sid[w];
        }
        bad |= sbad[w];
    }
    uint64_t S = 0;
    if (!bad && m > -INFINITY && sum) {
        // each thread's sum moved to the row maximum, in units of 2^-40 (float
        // products, one rounding each; below 2^50 units), rounded to an integer
        // and summed exactly over the CTA (relative error ~1e-7; no double
        // arithmetic, whose rate on this GPU is a small fraction of float's)
        const float part =
            ks != 0.f ? __fmul_rn(__fmul_rn(__fsub_rn(ks, kc), hw_exp2((mt - m) * c2)), 1099511627776.0f) : 0.f;
        uint64_t v = __float2ull_rn(part);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) ured[warp] = v;
        __syncthreads();
        for (int w = 0; w < kSSW; ++w) S += ured[w];
    }
    if (tid == 0) {
        RowStat st;
        st.zmax = m;
        st.argmax = m > -INFINITY ? id : -1;
        st.bad = bad;
        st.pad = 0;
        st.S = S;
        st.pad2 = 0;
        stats[blockIdx.x] = st;
    }
}

// ------------------------------------------------------------------ inverse-CDF draw over a slice
// This CTA's part of a draw over the slices of a cluster: the first element e
// (ascending) of its slice [0, n) at which the running mass, counted from the
// masses of the earlier slices, exceeds the draw position.  Masses come four
// at a time from m4(e, out[4]).  Chunks of 128 * cpw elements: warp w sums
// chunks w, w + 16, ... (lane l takes elements 4l..4l+3 of each 128), the chunk
// sums are scanned in shared memory; xf(total, X) turns this slice's total into
// the draw position relative to the slice (~0 when it lies in another slice)
// and returns false when the cluster's total is 0; then warp 0 walks the chunk
// that holds the draw.  Returns the element, -1 when the draw lies in another
// slice, -2 when the cluster's total is 0.
template <typename M4, typename XF>
__device__ int cta_draw(int n, M4 m4, XF xf, unsigned long long* ctot, unsigned long long* red, int* sel) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nv = (n + 3) & ~3;
    const int cpw = max(1, (nv + 128 * kDrawChunks - 1) / (128 * kDrawChunks));
    const int csz = 128 * cpw;
    const int nch = (nv + csz - 1) / csz;
    for (int ch = warp; ch < nch; ch += kVW) {
        uint64_t w = 0;
        for (int k = 0; k < cpw; ++k) {
            const int e = ch * csz + 128 * k + 4 * lane;
            if (e < nv) {
                uint64_t m[4];
                m4(e, m);
                w += m[0] + m[1] + m[2] + m[3];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
        if (lane == 0) ctot[ch] = w;
    }
    __syncthreads();
    uint64_t t4[4], ts = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int ch = 4 * tid + q;
        t4[q] = ch < nch ? ctot[ch] : 0ull;
        ts += t4[q];
    }
    // exclusive scan over the CTA
    uint64_t x = ts;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) red[warp] = x;
    if (tid == 0) *sel = -1;
    __syncthreads();
    uint64_t before = 0, total = 0;
    for (int w = 0; w < kVW; ++w) {
        if (w < warp) before += red[w];
        total += red[w];
    }
    uint64_t run = before + x - ts;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int ch = 4 * tid + q;
        if (ch < nch) ctot[ch] = run;
        run += t4[q];
    }
    __syncthreads();
    uint64_t X = ~0ull;
    if (!xf(total, X)) return -2;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int ch = 4 * tid + q;
        if (ch < nch) {
            const uint64_t lo = ctot[ch], hi = ch + 1 < nch ? ctot[ch + 1] : total;
            if (lo <= X && X < hi) *sel = ch;
        }
    }
    __syncthreads();
    const int cs = *sel;
    __shared__ int found;
    if (tid == 0) found = -1;
    __syncthreads();
    if (warp == 0 && cs >= 0) {
        uint64_t base = ctot[cs];
        for (int k = 0; k < cpw; ++k) {
            const int e = cs * csz + 128 * k + 4 * lane;
            uint64_t m[4] = {0ull, 0ull, 0ull, 0ull};
            if (e < nv) m4(e, m);
            const uint64_t mine = m[0] + m[1] + m[2] + m[3];
            uint64_t inc = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint64_t y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            const uint64_t bl = base + inc - mine;
            if (bl <= X && X < bl + mine) {
                uint64_t cum = bl;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    cum += m[j];
                    if (cum > X) {
                        found = e + j;
                        break;
                    }
                }
            }
            base += __shfl_sync(0xffffffffu, inc, 31);
            if (base > X) break;
        }
    }
    __syncthreads();
    return found;
}

// ------------------------------------------------------------------ verification
// One cluster of nc CTAs per request: every CTA takes the (cheap) tests; the
// final draw is spread over the vocabulary slices [rank * slice, ...) of the
// cluster, the slices' totals exchanged through distributed shared memory,
// and the CTA whose slice holds the draw writes the token.  Rank 0 writes the
// other outputs.
__global__ void __launch_bounds__(kVT)
    spec_verify_kernel(int32_t* __restrict__ tokens_out, int32_t* __restrict__ n_accepted,
                       int32_t* __restrict__ seq_lens_out, const float* __restrict__ target,
                       const float* __restrict__ draft, const int32_t* __restrict__ draft_tokens,
                       const int32_t* __restrict__ seq_lens, int gamma, int V, int slice,
                       const float* __restrict__ temperature, const uint64_t* __restrict__ seeds,
                       const uint64_t* __restrict__ offsets, const RowStat* __restrict__ stats, int32_t* status) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the row statistics are complete
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ unsigned long long ctot[kDrawChunks];
    __shared__ unsigned long long red[kVW];
    __shared__ unsigned long long xslot[2];  // this slice's total, alternating per draw
    __shared__ int sel, nrej, err;
    __shared__ float sat, saq;  // 2^40 / S of the target and draft rows at the first rejection
    cg::cluster_group cl = cg::this_cluster();
    const int nc = static_cast<int>(cl.num_blocks()), rank = static_cast<int>(cl.block_rank());
    const int b = blockIdx.x / nc, tid = threadIdx.x;
    const int lo = min(V, rank * slice), ns = min(V, lo + slice) - lo;  // this CTA's slice of the vocabulary
    const int rows = 2 * gamma + 1;
    const RowStat* st = stats + static_cast<size_t>(b) * rows;
    const float T = temperature[b];
    const uint64_t seed = seeds[b], offset = offsets[b];
    const int L = seq_lens[b];
    int32_t* tok = tokens_out + static_cast<size_t>(b) * (gamma + 1);
    if (tid == 0) {
        int e = 0;
        for (int r = 0; r < rows; ++r)
            if (st[r].bad || st[r].argmax < 0) e = PKV_ERR_NONFINITE;
        if (!e) {
            if (!(T >= 0.f) || L < gamma) e = PKV_ERR_INVALID_ARG;
            for (int i = 0; i < gamma; ++i) {
                const int x = draft_tokens[static_cast<size_t>(b) * gamma + i];
                if (x < 0 || x >= V) e = PKV_ERR_INVALID_ARG;
            }
        }
        err = e;
        nrej = gamma;
    }
    __syncthreads();
    if (err) {  // the same in every CTA of the cluster, before any exchange
        if (rank == 0) {
            for (int i = tid; i <= gamma; i += kVT) tok[i] = -1;
            if (tid == 0) {
                n_accepted[b] = 0;
                seq_lens_out[b] = L;
                report(status, err);
            }
        }
        return;
    }
    const float c2 = fminf(1.4426950408889634f / T, 1.0e30f);
    // the tests: thread i decides draft position i; the first rejection ends the cycle
    if (tid < gamma) {
        const int x = draft_tokens[static_cast<size_t>(b) * gamma + tid];
        const float* zt = target + (static_cast<size_t>(b) * (gamma + 1) + tid) * V;
        const float* zd = draft + (static_cast<size_t>(b) * gamma + tid) * V;
        bool accept;
        if (T == 0.f) {
            accept = x == st[tid].argmax;
        } else {
            const RowStat& sp = st[tid];
            const RowStat& sq = st[gamma + 1 + tid];
            const double p = static_cast<double>(mass(zt[x], sp.zmax, c2)) / static_cast<double>(sp.S);
            const double q = static_cast<double>(mass(zd[x], sq.zmax, c2)) / static_cast<double>(sq.S);
            const double u = static_cast<double>(philox_word0(seed, offset, static_cast<uint64_t>(tid) + 1) >> 11) *
                             (1.0 / 9007199254740992.0);
            accept = u * q < p;
        }
        if (!accept) atomicMin(&nrej, tid);
    }
    __syncthreads();
    const int n = nrej;
    // the residual's scales, in double by one thread (this GPU's FP64 rate makes
    // a double division repeated by every thread cost microseconds)
    if (tid == 0 && T != 0.f && n < gamma) {
        sat = static_cast<float>(1099511627776.0 / static_cast<double>(st[n].S));
        saq = static_cast<float>(1099511627776.0 / static_cast<double>(st[gamma + 1 + n].S));
    }
    __syncthreads();
    // rank 0 writes every output but the drawn token (before the draw's cluster
    // barrier, so that the CTA holding the draw writes that one after it)
    if (rank == 0) {
        for (int i = tid; i <= gamma; i += kVT)
            tok[i] = i < n ? draft_tokens[static_cast<size_t>(b) * gamma + i] : (i == n && T == 0.f ? st[n].argmax : -1);
        if (tid == 0) {
            n_accepted[b] = n;
            seq_lens_out[b] = L - gamma + n;
        }
    }
    if (T != 0.f) {
        const uint64_t u53 = philox_word0(seed, offset, 0) >> 11;
        const float* zt = target + (static_cast<size_t>(b) * (gamma + 1) + n) * V;
        const bool alt = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(zt) & 15u) == 0);
        const float mt = st[n].zmax;
        auto target_mass = [&](int e, uint64_t* m) {
            const float4 q = load4_row(zt, e, V, alt);
            m[0] = mass(q.x, mt, c2);
            m[1] = mass(q.y, mt, c2);
            m[2] = mass(q.z, mt, c2);
            m[3] = mass(q.w, mt, c2);
        };
        int xk = 0;
        auto xf = [&](uint64_t tot, uint64_t& X) -> bool {  // the draw position relative to this slice
            if (tid == 0) xslot[xk & 1] = tot;
            cl.sync();
            uint64_t excl = 0, grand = 0;
            for (int r = 0; r < nc; ++r) {
                const uint64_t t = *cl.map_shared_rank(&xslot[xk & 1], r);
                excl += r < rank ? t : 0ull;
                grand += t;
            }
            ++xk;
            if (grand == 0) return false;
            const uint64_t Xg = static_cast<uint64_t>((static_cast<unsigned __int128>(u53) * grand) >> 53);
            X = (Xg >= excl && Xg - excl < tot) ? Xg - excl : ~0ull;
            return true;
        };
        int f = -2;
        if (n < gamma) {
            // residual max(0, p - q) in 2^-40 fixed point of probability
            const float* zd = draft + (static_cast<size_t>(b) * gamma + n) * V;
            const bool ald = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(zd) & 15u) == 0);
            const float mq = st[gamma + 1 + n].zmax;
            const float at = sat, aq = saq;
            auto resid_mass = [&](int e, uint64_t* m) {
                const float4 a = load4_row(zt, e, V, alt);
                const float4 d = load4_row(zd, e, V, ald);
                const float pa[4] = {a.x, a.y, a.z, a.w}, pd[4] = {d.x, d.y, d.z, d.w};
                // each operation rounded on its own: the chunk sums and the walk
                // of the drawn chunk evaluate this in separate inlined copies,
                // and a contraction into a fused multiply-add in one of them
                // only would give the two different masses
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float r = __fsub_rn(__fmul_rn(weight(pa[j], mt, c2), at), __fmul_rn(weight(pd[j], mq, c2), aq));
                    m[j] = fx40(fminf(fmaxf(r, 0.f), 1.f));
                }
            };
            f = cta_draw(ns, [&](int e, uint64_t* m) { resid_mass(lo + e, m); }, xf, ctot, red, &sel);
        }
        if (f == -2)  // no residual mass (or every draft kept): draw from p
            f = cta_draw(ns, [&](int e, uint64_t* m) { target_mass(lo + e, m); }, xf, ctot, red, &sel);
        if (f >= 0 && tid == 0) tok[n] = lo + f;
        cl.sync();  // no CTA leaves while a peer may still read its slot
    }
}

size_t spec_verify_workspace_bytes(int B, int gamma) {
    return static_cast<size_t>(B) * (2 * static_cast<size_t>(gamma) + 1) * sizeof(RowStat);
}

int device_sm_count();

cudaError_t launch_spec_verify(int32_t* tokens_out, int32_t* n_accepted, int32_t* seq_lens_out, const float* target,
                               const float* draft, const int32_t* draft_tokens, const int32_t* seq_lens, int B,
                               int gamma, int V, const float* temperature, const uint64_t* seeds,
                               const uint64_t* offsets, void* workspace, int32_t* status, cudaStream_t stream) {
    RowStat* stats = static_cast<RowStat*>(workspace);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B) * (2 * gamma + 1), 1, 1);
    cfg.blockDim = dim3(kSS, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err = cudaLaunchKernelEx(&cfg, spec_stats_kernel, target, draft, gamma, V, temperature, stats);
    if (err != cudaSuccess) return err;
    // CTAs per request: as many as fit two 512-thread CTAs per SM (1, 2, 4 or 8),
    // slices of at least 4096 logits
    const int sms = device_sm_count();
    int nc = 1;
    while (nc < 8 && static_cast<long long>(B) * nc * 2 <= 2LL * sms && V / (nc * 2) >= 4096) nc *= 2;
    int slice = (V + nc - 1) / nc;
    slice = (slice + 3) & ~3;  // slices start on 16-byte boundaries of a 16-byte aligned row
    cudaLaunchAttribute attr2[2];
    attr2[0] = attr[0];
    attr2[1].id = cudaLaunchAttributeClusterDimension;
    attr2[1].val.clusterDim.x = nc;
    attr2[1].val.clusterDim.y = 1;
    attr2[1].val.clusterDim.z = 1;
    cfg.attrs = attr2;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(static_cast<unsigned>(B) * nc, 1, 1);
    cfg.blockDim = dim3(kVT, 1, 1);  // the verification kernel's CTAs are 512 threads
    err = cudaLaunchKernelEx(&cfg, spec_verify_kernel, tokens_out, n_accepted, seq_lens_out, target, draft,
                             draft_tokens, seq_lens, gamma, V, slice, temperature, seeds, offsets,
                             static_cast<const RowStat*>(stats), status);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace pkv
