// sampler_rows.cu -- the sampler for many rows of a moderate vocabulary: one
// CTA of 256 threads per row, every row resident at once.
//
// Same definition as sampler.cu ("Suy luan & Toi uu hoa (Inference)" 1.2;
// "Bai Lab tong hop -- Inference Engineering" block [8]; "LLM inference
// serving tutorial" 3.1, 1.6): T == 0 -> the lowest id holding the maximum;
// otherwise masses floor(2^((z - zmax) log2(e) / T) * 2^40) over the finite
// logits, top-k on the order (z desc, id asc), top-p as the smallest prefix of
// that order whose mass reaches ceil(top_p * S_k), min-p, and the draw in
// token-id order with the request's Philox uniform.  The masses and every
// comparison are those of sampler.cu, so both kernels return the same token.
//
// Why a second kernel: with B rows of V <= 65536 logits and B larger than the
// resident CTAs of the cluster kernel (512-thread CTAs, two per SM), that
// kernel runs its rows in waves of long dependent phase chains.  Here a CTA of
// 256 threads holds a row (four per SM), so a batch of up to 4 x #SM rows is
// resident in one wave and the rows' chains overlap.
//
// Passes over the row (the first reads HBM, the others hit L2):
//  A: maximum, minimum, NaN/+inf flag, finite count, first index of the
//     maximum (thread t takes the 16-byte slots 4 (t + 256 m));
//  B: 2048 bins linear in (zmax - z): the count and the exact mass of every
//     bin as 32-bit shared sums (count, mass >> 20, mass mod 2^20).  The
//     cumulative counts give the top-k boundary bin bk, the cumulative masses
//     the bins [wlo, whi] that can hold the top-p cut;
//  C: in chunks of 512 consecutive ids (one warp, four float4 loads per lane):
//     the kept mass of every chunk's logits in bins < wlo, the masses of bins
//     < wlo and of the bins between the window and bk summed, and the logits of
//     bins wlo..whi (and of bin bk) gathered as sort keys.
// The gathered window is sorted (z desc, id asc); it gives the exact top-k
// part of bin bk, S_k, the top-p cut (checked to lie in the window), and the
// kept window entries, whose masses join their chunks.  An exclusive scan of
// the chunk sums locates the draw, and one warp walks that chunk.  A window
// larger than kRwCap logits, a bin of 4096 logits or more, or a cut outside
// the window takes an exact radix selection over the row instead.  Rows with
// 0 < top_k <= kRSmallK take the thread-maxima path after pass A.
#include <math.h>

#include "pkv_common.cuh"
#include "sampling_math.cuh"

namespace pkv {

constexpr int kRT = 256;             // threads per CTA
constexpr int kRW = kRT / 32;        // warps
constexpr int kRBins = 2048;         // linear bins
constexpr int kRwCap = 2048;         // gathered window capacity
constexpr int kRChunk = 512;         // ids per draw chunk (one warp's four loads of a chunk sweep)
constexpr int kRowMaxV = 65536;      // largest vocabulary this kernel serves
constexpr int kRChunks = kRowMaxV / kRChunk;
constexpr int kRSmallK = 64;         // top_k served by the thread-maxima path
static_assert(kRChunks >= 2 * kRSmallK, "the thread-maxima path keeps its keys and masses in csum");

struct RowSmem {
    unsigned int cnt[kRBins];            // count per bin
    unsigned int mhi[kRBins];            // sum of mass >> 20 per bin
    unsigned int mlo[kRBins];            // sum of mass & (2^20 - 1) per bin
    unsigned long long win[kRwCap];      // the gathered window (sort keys); radix histograms
    unsigned long long csum[kRChunks];   // kept mass per chunk of kRChunk ids
    unsigned long long wsum[kRW];
    unsigned long long bc[8];
    float fv[kRW];
    int iv[kRW];
    unsigned int nwin;
    unsigned int nq;                     // threads whose maximum is a candidate (small top-k)
    unsigned long long u53;
    float edge[4];                       // pass C's bin bounds as logit thresholds
    unsigned long long wsum2[kRW];
    unsigned long long wtot;             // logits in the window's bins
};
template <bool B>
struct RwFlag {
    static constexpr bool value = B;
};

// ------------------------------------------------------------------ CTA helpers
__device__ __forceinline__ uint64_t rw_sum(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// Exclusive prefix over the threads in index order; total = the sum.  Starts
// and ends with a barrier.
__device__ uint64_t rw_excl_scan(uint64_t v, RowSmem* sm, uint64_t& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    __syncthreads();
    if (lane == 31) sm->wsum[warp] = inc;
    __syncthreads();
    uint64_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kRW; ++w) {
        const uint64_t s = sm->wsum[w];
        before += w < warp ? s : 0ull;
        tot += s;
    }
    total = tot;
    __syncthreads();
    return before + inc - v;
}

// Two exclusive prefixes at once (one set of barriers); returns v0's, with
// e1 = v1's and the two totals.
__device__ uint64_t rw_excl_scan2(uint64_t v0, uint64_t v1, RowSmem* sm, uint64_t& t0, uint64_t& e1,
                                  uint64_t& t1) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t i0 = v0, i1 = v1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y0 = __shfl_up_sync(0xffffffffu, i0, o);
        const uint64_t y1 = __shfl_up_sync(0xffffffffu, i1, o);
        if (lane >= o) {
            i0 += y0;
            i1 += y1;
        }
    }
    __syncthreads();
    if (lane == 31) {
        sm->wsum[warp] = i0;
        sm->wsum2[warp] = i1;
    }
    __syncthreads();
    uint64_t b0 = 0, b1 = 0, s0 = 0, s1 = 0;
#pragma unroll
    for (int w = 0; w < kRW; ++w) {
        const uint64_t a = sm->wsum[w], c = sm->wsum2[w];
        b0 += w < warp ? a : 0ull;
        b1 += w < warp ? c : 0ull;
        s0 += a;
        s1 += c;
    }
    t0 = s0;
    t1 = s1;
    e1 = b1 + i1 - v1;
    __syncthreads();
    return b0 + i0 - v0;
}

// Four consecutive logits from slot e (entries past n read as -inf).
__device__ __forceinline__ float4 rw_load4(const float* __restrict__ z, int n, int e, bool a16) {
    if (a16 && e + 4 <= n) return __ldg(reinterpret_cast<const float4*>(z + e));
    float4 q;
    q.x = e < n ? z[e] : -INFINITY;
    q.y = e + 1 < n ? z[e + 1] : -INFINITY;
    q.z = e + 2 < n ? z[e + 2] : -INFINITY;
    q.w = e + 3 < n ? z[e + 3] : -INFINITY;
    return q;
}

// Every slot of the thread (4 (t + kRT m)), four loads in flight; f(e, q).
// The trip count is warp-uniform (lanes past the end see -inf), so f may use
// warp-collective operations, and one iteration of a warp covers the 128
// consecutive ids starting at 4 (32 w + kRT m).
template <typename F>
__device__ __forceinline__ void rw_sweep(const float* __restrict__ z, int n, bool a16, F&& f) {
    const int lane = threadIdx.x & 31;
    const int nvec = (n + 3) & ~3;
    for (int e0 = 4 * (static_cast<int>(threadIdx.x) - lane); e0 < nvec; e0 += 4 * kRT * 4) {
        float4 q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + 4 * lane + 4 * kRT * u;
            q[u] = e < nvec ? rw_load4(z, n, e, a16) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) f(e0 + 4 * lane + 4 * kRT * u, q[u]);
    }
}
// The row in chunks of kRChunk ids: warp w takes the chunks w, w + kRW, ...,
// lane l the float4s at 4 l + 128 u (u = 0..3) of each, four loads in flight;
// f(c0, q) with c0 the chunk's first id, element (u, j) being id
// c0 + 128 u + 4 l + j.  The trip count is warp-uniform.
template <typename F>
__device__ __forceinline__ void rw_sweep_chunks(const float* __restrict__ z, int n, bool a16, F&& f) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nvec = (n + 3) & ~3;
    for (int c0 = kRChunk * warp; c0 < nvec; c0 += kRChunk * kRW) {
        float4 q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = c0 + 4 * lane + 128 * u;
            q[u] = e < nvec ? rw_load4(z, n, e, a16) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
        f(c0, q);
    }
}
static_assert(kRChunk == 4 * 128, "a chunk is one warp's four float4 loads");
__device__ __forceinline__ float rw_at(const float4& q, int j) {
    return j == 0 ? q.x : (j == 1 ? q.y : (j == 2 ? q.z : q.w));
}

// Bitonic sort of a[0..n) (n a power of two) in descending order.
__device__ void rw_sort_desc(unsigned long long* a, int n) {
    for (int k = 2; k <= n; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += kRT) {
                const int l = i ^ j;
                if (l > i) {
                    const bool desc = (i & k) == 0;
                    const unsigned long long x = a[i], y = a[l];
                    if ((x < y) == desc) {
                        a[i] = y;
                        a[l] = x;
                    }
                }
            }
            __syncthreads();
        }
}

// ------------------------------------------------------------------ exact fallback
// Radix selection over the order-preserving keys of the row's finite logits
// (11/11/10-bit digits, from the largest key down): the key tau at which the
// cumulative weight (count, or mass when kMass) of the logits passing `in`
// first reaches target, with `above` the weight of the larger keys.
template <bool kMass, typename In>
__device__ uint32_t rw_radix(RowSmem* sm, const float* __restrict__ z, int n, bool a16, In in, float zmax, float c2,
                             uint64_t target, uint64_t& above) {
    const int tid = threadIdx.x;
    unsigned long long* h = sm->win;
    uint32_t prefix = 0u;
    int pbits = 0;
    const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
    for (int ps = 0; ps < 3; ++ps) {
        const int shift = shifts[ps], nb = 1 << widths[ps];
        for (int i = tid; i < nb; i += kRT) h[i] = 0ull;
        __syncthreads();
        rw_sweep(z, n, a16, [&](int e, const float4& q) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float x = rw_at(q, j);
                if (!(x > -INFINITY) || !in(x, e + j)) continue;
                const uint32_t key = okey(x);
                if (pbits && (key >> (32 - pbits)) != prefix) continue;
                const uint64_t w = kMass ? mass(x, zmax, c2) : 1ull;
                if (w) atomicAdd(&h[(key >> shift) & static_cast<uint32_t>(nb - 1)], static_cast<unsigned long long>(w));
            }
        });
        __syncthreads();
        // digits from the largest down, nb / kRT per thread
        const int bpt = nb / kRT;
        uint64_t ts = 0;
        for (int q = 0; q < bpt; ++q) ts += h[nb - 1 - (tid * bpt + q)];
        if (tid == 0) {
            sm->bc[0] = 0ull;
            sm->bc[1] = above;
        }
        uint64_t tot;
        const uint64_t ex = rw_excl_scan(ts, sm, tot);
        const uint64_t c0 = above + ex;
        if (c0 < target && c0 + ts >= target) {
            uint64_t cc = c0;
            for (int q = 0; q < bpt; ++q) {
                const uint64_t hv = h[nb - 1 - (tid * bpt + q)];
                if (cc + hv >= target) {
                    sm->bc[0] = static_cast<unsigned long long>(nb - 1 - (tid * bpt + q));
                    sm->bc[1] = cc;
                    break;
                }
                cc += hv;
            }
        }
        __syncthreads();
        prefix = (prefix << widths[ps]) | static_cast<uint32_t>(sm->bc[0]);
        pbits += widths[ps];
        above = sm->bc[1];
        __syncthreads();
    }
    return prefix;
}

// Id of the r-th (1-based) logit in id order whose key is tau and that passes
// `in` (contiguous runs of ids per thread, then a scan).
template <typename In>
__device__ int rw_tie(RowSmem* sm, const float* __restrict__ z, int n, In in, uint32_t tau, uint64_t r) {
    const int tid = threadIdx.x;
    int E = (n + kRT - 1) / kRT;
    if (E < 1) E = 1;
    const int b0 = min(n, tid * E), b1 = min(n, b0 + E);
    auto match = [&](int i) {
        const float x = z[i];
        return x > -INFINITY && okey(x) == tau && in(x, i);
    };
    uint64_t c = 0;
    for (int i = b0; i < b1; ++i) c += match(i) ? 1u : 0u;
    if (tid == 0) sm->bc[2] = 0xffffffffull;
    uint64_t tot;
    const uint64_t ex = rw_excl_scan(c, sm, tot);
    if (ex < r && r <= ex + c) {
        uint64_t need = r - ex;
        for (int i = b0; i < b1; ++i)
            if (match(i) && --need == 0) {
                sm->bc[2] = static_cast<unsigned long long>(i);
                break;
            }
    }
    __syncthreads();
    const int id = static_cast<int>(sm->bc[2]);
    __syncthreads();
    return id;
}

// ------------------------------------------------------------------ row order
// The row CTA blockIdx.x takes: the rows with the most work get the lowest CTA
// indices, so that they start first and spread over the SMs
// (longest-processing-time-first order; the tokens do not depend on it).
// Classes: 2 = top-p alone, 1 = top-k above kRSmallK or no truncation,
// 0 = greedy, small top-k or invalid parameters; order: class descending, row
// index ascending: the CTA counts the rows per class, then (unless every row
// is in one class, where it returns -1 for the natural order) finds the row of
// its rank within its class with warp ballots.
__device__ int rw_lpt_row(int B, int V, const float* __restrict__ temperature, const int32_t* __restrict__ top_k,
                          const float* __restrict__ top_p, RowSmem* sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    auto cls = [&](int r) -> int {  // loads all three parameters, so that no load waits on another
        const float t = temperature[r];
        const int k = top_k[r];
        const float p = top_p[r];
        const bool k_on = k > 0 && k < V;
        if (!(t > 0.f) || (k_on && k <= kRSmallK)) return 0;
        return !k_on && p < 1.f ? 2 : 1;
    };
    // scratch, cleared by pass A afterwards: the bin counts ([0..2] rows per
    // class, [3] the answer, [8..8+kRW) rows of the sought class per warp) and
    // the class of every row, one byte each, while they fit in the mass bins
    unsigned int* cc = sm->cnt;
    unsigned char* c8 = reinterpret_cast<unsigned char*>(sm->mhi);
    const bool keep = B <= static_cast<int>(sizeof(sm->mhi));
    if (tid < 4) cc[tid] = 0u;
    unsigned long long own = 0ull;  // this thread's rows per class, 21 bits each
#pragma unroll 4
    for (int r = tid; r < B; r += kRT) {
        const int c = cls(r);
        own += 1ull << (21 * c);
        if (keep) c8[r] = static_cast<unsigned char>(c);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) own += __shfl_xor_sync(0xffffffffu, own, o);
    __syncthreads();  // cc[0..3] cleared
    if (lane < 3) atomicAdd(&cc[lane], static_cast<unsigned int>((own >> (21 * lane)) & 0x1fffffull));
    __syncthreads();
    const int n2 = static_cast<int>(cc[2]), n1 = static_cast<int>(cc[1]);
    const int u = static_cast<int>(blockIdx.x);
    if (n2 == B || n1 == B || n2 + n1 == 0) {  // one class: the natural order
        __syncthreads();
        return -1;
    }
    const int cs = u < n2 ? 2 : (u < n2 + n1 ? 1 : 0);        // this CTA's class
    const int jj = u - (cs == 2 ? 0 : (cs == 1 ? n2 : n2 + n1));  // its rank within the class
    int before = 0;  // rows of class cs in earlier chunks (the same in every thread)
    for (int r0 = 0; r0 < B && before <= jj; r0 += kRT) {
        const int r = r0 + tid;
        const bool f = r < B && (keep ? static_cast<int>(c8[r]) : cls(r)) == cs;
        const unsigned int m = __ballot_sync(0xffffffffu, f);
        if (lane == 0) cc[8 + warp] = static_cast<unsigned int>(__popc(m));
        __syncthreads();
        int wb = before, tot = 0;
#pragma unroll
        for (int w = 0; w < kRW; ++w) {
            const int cw = static_cast<int>(cc[8 + w]);
            wb += w < warp ? cw : 0;
            tot += cw;
        }
        if (f && wb + __popc(m & ((1u << lane) - 1u)) == jj) cc[3] = static_cast<unsigned int>(r);
        before += tot;
        __syncthreads();
    }
    const int row = static_cast<int>(cc[3]);
    __syncthreads();
    return row;
}

// ------------------------------------------------------------------ kernel
// One row: the passes below, in a function so that the kernel can compile it
// twice, once for the natural order (row = blockIdx.x, which the compiler
// re-reads rather than keeping it live in the passes at the 64-register cap)
// and once for the row the ordering picked.
__device__ __forceinline__ void rw_sample_row(int row, int32_t* __restrict__ tokens,
                                              const float* __restrict__ logits, int V,
                                              const float* __restrict__ temperature,
                                              const int32_t* __restrict__ top_k, const float* __restrict__ top_p,
                                              const float* __restrict__ min_p, const uint64_t* __restrict__ seeds,
                                              const uint64_t* __restrict__ offsets, int32_t* status, RowSmem* sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* z = logits + static_cast<size_t>(row) * V;
    const bool a16 = (reinterpret_cast<uintptr_t>(z) & 15u) == 0;
    int32_t* tok_out = tokens + row;
    const float T = temperature[row];
    const float pp = top_p[row];
    const float mp = min_p ? min_p[row] : 0.f;
    const int kin = top_k[row];
    if (tid == 0) sm->u53 = philox_word0(seeds[row], offsets[row]) >> 11;

    // ---- A: maximum (first index), minimum over finite logits, NaN/+inf flag, finite count
    float mx = -INFINITY, mn = INFINITY;
    int am = 0x7fffffff;
    unsigned int bad = 0u, nf = 0u;
    rw_sweep(z, V, a16, [&](int e, const float4& q) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float x = rw_at(q, j);
            bad |= (x < INFINITY) ? 0u : 1u;
            const bool fin = x > -INFINITY && x < INFINITY;
            nf += fin ? 1u : 0u;
            if (fin && x > mx) {  // visited in ascending index order: the first one is kept
                mx = x;
                am = e + j;
            }
            mn = fminf(mn, fin ? x : INFINITY);
        }
    });
    float wm = mx, wn = mn;
    unsigned int wb = bad, wf = nf;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
        wn = fminf(wn, __shfl_xor_sync(0xffffffffu, wn, o));
        wb |= __shfl_xor_sync(0xffffffffu, wb, o);
        wf += __shfl_xor_sync(0xffffffffu, wf, o);
    }
    if (lane == 0) {
        sm->fv[warp] = wm;
        sm->wsum[warp] = (static_cast<unsigned long long>(wb) << 32) | wf;
        sm->iv[warp] = __float_as_int(wn);
    }
    for (int i = tid; i < kRBins; i += kRT) {
        sm->cnt[i] = 0u;
        sm->mhi[i] = 0u;
        sm->mlo[i] = 0u;
    }
    for (int i = tid; i < kRChunks; i += kRT) sm->csum[i] = 0ull;
    if (tid == 0) {
        sm->nwin = 0u;
        sm->nq = 0u;
    }
    __syncthreads();
    float zmax = -INFINITY, zmin = INFINITY;
    unsigned int gbad = 0u, nfin = 0u;
#pragma unroll
    for (int w = 0; w < kRW; ++w) {
        zmax = fmaxf(zmax, sm->fv[w]);
        zmin = fminf(zmin, __int_as_float(sm->iv[w]));
        gbad |= static_cast<unsigned int>(sm->wsum[w] >> 32);
        nfin += static_cast<unsigned int>(sm->wsum[w] & 0xffffffffull);
    }
    int err = 0;
    if (gbad || nfin == 0u) err = PKV_ERR_NONFINITE;
    else if (!(T >= 0.f)) err = PKV_ERR_INVALID_ARG;
    else if (T != 0.f && !(pp > 0.f)) err = PKV_ERR_INVALID_ARG;
    else if (T != 0.f && (mp != mp || mp > 1.f)) err = PKV_ERR_INVALID_ARG;  // min_p NaN or > 1
    if (err) {
        if (tid == 0) {
            *tok_out = -1;
            report(status, err);
        }
        return;
    }
    if (T == 0.f) {  // greedy: the lowest index holding the maximum
        int a = mx == zmax ? am : 0x7fffffff;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
        __syncthreads();  // fv / iv are reused
        if (lane == 0) sm->iv[warp] = a;
        __syncthreads();
        if (tid == 0) {
            int b = 0x7fffffff;
            for (int w = 0; w < kRW; ++w) b = min(b, sm->iv[w]);
            *tok_out = b;
        }
        return;
    }
    const float c2 = fminf(1.4426950408889634f / T, 1.0e30f);
    const int kk = (kin > 0 && static_cast<unsigned int>(kin) < nfin) ? kin : 0;  // 0: top-k off
    const uint64_t mth = mp > 0.f ? ceil_mul_p(mp, 1ull << 40) : 0ull;         // min-p threshold
    const float range = zmax - zmin;
    const float bsc = (range > 0.f && range < INFINITY) ? static_cast<float>(kRBins) / range : 0.f;
    // bin b holds the logits with b <= (zmax - x) * bsc < b + 1; floor by an
    // add in round-down mode (the integer lands in the significand)
    auto bin = [&](float x) {  // monotone non-increasing in x; bin 0 holds the largest logits
        const float t = (zmax - x) * bsc;
        return t < static_cast<float>(kRBins - 1) ? __float_as_int(__fadd_rd(t, 8388608.0f)) - 0x4B000000
                                                  : kRBins - 1;
    };

    // ---- small top-k (0 < kk <= kRSmallK): only the kk largest logits
    // matter.  Bin b* is the first where the count of thread maxima (pass A)
    // from the top reaches kk: at least kk logits lie in bins <= b*, and the
    // binning is monotone, so the top kk all lie there.  Only threads whose
    // maximum lies there can hold such a logit; their slots are read again
    // (L2), spread over the CTA, and every logit in bins <= b* is kept as a
    // sort key.  Each key's rank is the number of larger keys; the first kk in
    // rank order get their masses, top-p keeps the prefix whose mass before
    // the entry is below ceil(top_p * S_k), min-p drops masses below its
    // threshold, and the token whose interval in id order holds
    // X = floor(u * S_p) is drawn.  More than kRT candidates (a block of equal
    // logits) take the general path below.
    if (kk && kk <= kRSmallK) {
        constexpr int kPerS = kRBins / kRT;
        if (mx > -INFINITY) atomicAdd(&sm->cnt[bin(mx)], 1u);
        if (tid == 0) sm->bc[0] = kRBins - 1;  // fewer than kk finite maxima: every finite logit
        __syncthreads();
        uint64_t tc = 0;
        for (int q = 0; q < kPerS; ++q) tc += sm->cnt[kPerS * tid + q];
        uint64_t ctot;
        const uint64_t cex = rw_excl_scan(tc, sm, ctot);
        const uint64_t kq = static_cast<uint64_t>(kk);
        if (cex < kq && cex + tc >= kq) {
            uint64_t cc = cex;
            for (int q = 0; q < kPerS; ++q) {
                const uint64_t c1 = sm->cnt[kPerS * tid + q];
                if (cc < kq && cc + c1 >= kq) sm->bc[0] = static_cast<unsigned long long>(kPerS * tid + q);
                cc += c1;
            }
        }
        __syncthreads();
        const int bstar = static_cast<int>(sm->bc[0]);
        auto cand = [&](float x) { return x > -INFINITY && bin(x) <= bstar; };
        unsigned int* qlist = sm->mhi;
        if (cand(mx)) qlist[atomicAdd(&sm->nq, 1u)] = static_cast<unsigned int>(tid);
        __syncthreads();
        const int nq = static_cast<int>(sm->nq);
        const int nvec = (V + 3) & ~3;
        const int spt = (nvec + 4 * kRT - 1) / (4 * kRT);  // slots per thread
        const int nwork = nq * spt;
        for (int i0 = 0; i0 < nwork; i0 += 4 * kRT) {
            float4 qv[4];
            int ev[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {  // every load issued (slot 0 for idle lanes) before any is used
                const int i = i0 + u * kRT + tid;
                const int ic = i < nwork ? i : 0;
                const int qi = ic / spt;
                const int e = 4 * (static_cast<int>(qlist[qi]) + kRT * (ic - qi * spt));
                ev[u] = (i < nwork && e < nvec) ? e : -1;
                qv[u] = rw_load4(z, V, ev[u] >= 0 ? ev[u] : 0, a16);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float x = rw_at(qv[u], j);
                    if (ev[u] >= 0 && cand(x)) {
                        const unsigned int pos = atomicAdd(&sm->nwin, 1u);
                        if (pos < static_cast<unsigned int>(kRwCap)) sm->win[pos] = sort_key(x, ev[u] + j);
                    }
                }
        }
        __syncthreads();
        const int nl = static_cast<int>(sm->nwin);
        if (nl <= kRT) {
            unsigned long long* buf = sm->csum;        // the top kk keys in rank order
            unsigned long long* kwm = sm->csum + kRSmallK;  // their kept masses
            if (tid < nl) {
                const unsigned long long key = sm->win[tid];
                int rr = 0;
                for (int jj = 0; jj < nl; ++jj) rr += sm->win[jj] > key ? 1 : 0;
                if (rr < kk) buf[rr] = key;
            }
            __syncthreads();
            // four threads per entry i = tid / 4 (strided sums, reduced over the four lanes)
            const int i = tid >> 2, part = tid & 3;
            auto wof = [&](int jj) { return mass(key_float(static_cast<uint32_t>(buf[jj] >> 32)), zmax, c2); };
            uint64_t before = 0, sk = 0;
            for (int jj = part; jj < kk; jj += 4) {
                const uint64_t w = wof(jj);
                sk += w;
                before += jj < i ? w : 0ull;
            }
            sk += __shfl_xor_sync(0xffffffffu, sk, 1);
            sk += __shfl_xor_sync(0xffffffffu, sk, 2);
            before += __shfl_xor_sync(0xffffffffu, before, 1);
            before += __shfl_xor_sync(0xffffffffu, before, 2);
            const uint64_t Wi = i < kk ? wof(i) : 0ull;
            const bool kept = i < kk && (!(pp < 1.f) || before < ceil_mul_p(pp, sk)) && Wi >= mth;
            const uint64_t kw = kept ? Wi : 0ull;
            if (part == 0 && i < kk) kwm[i] = kw;
            __syncthreads();
            const uint32_t idi = i < kk ? static_cast<uint32_t>(sort_key_id(buf[i])) : 0xffffffffu;
            uint64_t bl = 0, sp = 0;  // kept mass at smaller ids; the kept total
            for (int jj = part; jj < kk; jj += 4) {
                const uint64_t w = kwm[jj];
                sp += w;
                bl += static_cast<uint32_t>(sort_key_id(buf[jj])) < idi ? w : 0ull;
            }
            sp += __shfl_xor_sync(0xffffffffu, sp, 1);
            sp += __shfl_xor_sync(0xffffffffu, sp, 2);
            bl += __shfl_xor_sync(0xffffffffu, bl, 1);
            bl += __shfl_xor_sync(0xffffffffu, bl, 2);
            const uint64_t X = static_cast<uint64_t>((static_cast<unsigned __int128>(sm->u53) * sp) >> 53);
            if (part == 0 && kw > 0 && bl <= X && X < bl + kw) *tok_out = static_cast<int32_t>(idi);
            return;
        }
        // a block of equal logits: back to the general path with clean bins
        for (int i = tid; i < kRBins; i += kRT) {
            sm->cnt[i] = 0u;
            sm->mhi[i] = 0u;
        }
        if (tid == 0) sm->nwin = 0u;
        __syncthreads();
    }

    // ---- B: count and exact mass per bin, as 32-bit sums of the mass's high
    // (>> 20) and low 20 bits: both stay below 2^32 while a bin holds fewer
    // than 4096 logits (masses are at most 2^40); a fuller bin sends the row
    // to the radix selection
    rw_sweep(z, V, a16, [&](int, const float4& q) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float x = rw_at(q, j);
            if (!(x > -INFINITY)) continue;
            const int b = bin(x);
            const uint64_t m = mass(x, zmax, c2);
            atomicAdd(&sm->cnt[b], 1u);
            atomicAdd(&sm->mhi[b], static_cast<unsigned int>(m >> 20));
            atomicAdd(&sm->mlo[b], static_cast<unsigned int>(m & 0xfffffu));
        }
    });
    __syncthreads();
    // thread t holds bins kPer t .. kPer t + kPer - 1
    constexpr int kPer = kRBins / kRT;
    auto cb = [&](int q) { return static_cast<uint64_t>(sm->cnt[kPer * tid + q]); };
    auto mb = [&](int q) {
        const int b = kPer * tid + q;
        return (static_cast<uint64_t>(sm->mhi[b]) << 20) + sm->mlo[b];
    };
    uint64_t tc = 0, tm = 0;
    unsigned int wide = 0u;
    for (int q = 0; q < kPer; ++q) {
        tc += cb(q);
        tm += mb(q);
        wide |= cb(q) >= 4096u ? 1u : 0u;
    }
    const bool exact = __syncthreads_or(wide) == 0;
    uint64_t ctot, S, mex;
    const uint64_t cex = rw_excl_scan2(tc, tm, sm, ctot, mex, S);
    if (tid == 0) {
        sm->bc[0] = kRBins;  // bk (kRBins: top-k off)
        sm->bc[1] = 0ull;    // logits before bk
        sm->bc[4] = 0ull;    // mass before bk
        sm->bc[6] = 0ull;    // mass of bin bk
    }
    __syncthreads();
    if (kk) {
        uint64_t cc = cex, mm = mex;
        for (int q = 0; q < kPer; ++q) {
            const uint64_t c1 = cb(q);
            if (cc < static_cast<uint64_t>(kk) && cc + c1 >= static_cast<uint64_t>(kk)) {
                sm->bc[0] = static_cast<unsigned long long>(kPer * tid + q);
                sm->bc[1] = cc;
                sm->bc[4] = mm;
                sm->bc[6] = mb(q);
            }
            cc += c1;
            mm += mb(q);
        }
    }
    __syncthreads();
    const int bk = static_cast<int>(sm->bc[0]);
    const uint64_t cnt_bk = sm->bc[1];
    const uint64_t rk = kk ? static_cast<uint64_t>(kk) - cnt_bk : 0ull;  // top-k entries of bin bk
    const bool p_on = pp < 1.f;
    // The cut bin: the first whose cumulative mass reaches ceil(top_p * S_k).
    // S_k = S with top-k off; with top-k on it lies in [mass before bk, that
    // + mass of bk], so the cut bin lies between the bins where the
    // cumulative reaches the two targets (capped at bk).
    const uint64_t sk_lo = kk ? sm->bc[4] : S, sk_hi = kk ? sm->bc[4] + sm->bc[6] : S;
    if (tid == 0) {
        sm->bc[2] = static_cast<unsigned long long>(p_on ? 0 : (kk ? bk : kRBins));  // wlo
        sm->bc[3] = static_cast<unsigned long long>(p_on ? (kk ? bk : kRBins - 1) : (kk ? bk : -1));  // whi
    }
    __syncthreads();
    if (p_on) {
        const uint64_t tg_lo = ceil_mul_p(pp, sk_lo), tg_hi = ceil_mul_p(pp, sk_hi);
        uint64_t mm = mex;
        for (int q = 0; q < kPer; ++q) {
            const int b = kPer * tid + q;
            if (kk && b > bk) break;
            const uint64_t nx = mm + mb(q);
            if (mm < tg_lo && nx >= tg_lo) sm->bc[2] = static_cast<unsigned long long>(b);
            if (mm < tg_hi && nx >= tg_hi) sm->bc[3] = static_cast<unsigned long long>(b);
            mm = nx;
        }
    }
    __syncthreads();
    const int wlo = static_cast<int>(sm->bc[2]);
    const int whi = max(static_cast<int>(static_cast<long long>(sm->bc[3])), wlo - 1);
    const bool gather_bk = kk && bk > whi;  // bin bk is gathered on its own for the exact S_k
    if (warp == 1) {  // the window's size from its bins' counts
        uint64_t wc = 0;
        for (int b = wlo + lane; b <= whi; b += 32) wc += sm->cnt[b];
        wc = rw_sum(wc);
        if (lane == 0) sm->wtot = wc + (gather_bk ? sm->cnt[bk] : 0u);
    }

    // Pass C's bin tests as comparisons: bin(x) is monotone non-increasing in
    // x, so bin(x) < c exactly when x >= edge(c), the smallest finite float
    // whose bin is below c (+inf for c = 0), found by bisection on the
    // order-preserving keys; -inf lies below every edge.
    if (tid < 4) {
        const int c = tid == 0 ? wlo : (tid == 1 ? whi + 1 : (tid == 2 ? bk : bk + 1));
        float ed = INFINITY;
        if (c > 0) {
            uint32_t lo = okey(-3.40282347e38f), hi = okey(zmax);  // bin(hi) = 0 < c
            if (bin(key_float(lo)) < c) {
                hi = lo;
            } else {
                while (hi - lo > 1u) {  // bin(lo) >= c > bin(hi)
                    const uint32_t mid = lo + (hi - lo) / 2u;
                    if (bin(key_float(mid)) < c)
                        hi = mid;
                    else
                        lo = mid;
                }
            }
            ed = key_float(hi);
        }
        sm->edge[tid] = ed;
    }
    __syncthreads();
    const float e_lo = sm->edge[0], e_win = sm->edge[1], e_bk = sm->edge[2], e_bk1 = sm->edge[3];
    const uint64_t wtot = sm->wtot;
    const bool fits = exact && wtot <= static_cast<uint64_t>(kRwCap);

    unsigned long long* win = sm->win;
    // the kept set: (key, id) at or before (cut_key, cut_id) in the order
    // (z desc, id asc) when kept_fn_cut, else every finite logit; min-p on top
    bool kept_fn_cut = false;
    uint32_t cut_key = 0u;
    int cut_id = -1;
    bool done = false;
    if (fits) {
        // ---- C: exact masses; chunk sums of bins < wlo; window gather
        uint64_t asum = 0, msum = 0;  // bins < wlo; top-k bins between the window and bk (top-k on)
        // compiled once with min-p and once without (then a chunk's sum is its
        // whole mass above the window, and the chunk sums give asum)
        auto pass_c = [&](auto minp_flag) {
          constexpr bool kMinP = decltype(minp_flag)::value;
          rw_sweep_chunks(z, V, a16, [&](int c0, const float4 (&q)[4]) {
            uint64_t s = 0;
            unsigned int inm = 0u;  // bit 4 u + j: element (u, j) lies in the window
#pragma unroll
            for (int u = 0; u < 4; ++u) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float x = rw_at(q[u], j);
                    if (x >= e_lo) {  // bin < wlo
                        const uint64_t m = mass(x, zmax, c2);
                        if constexpr (kMinP) {
                            asum += m;
                            s += m >= mth ? m : 0ull;
                        } else {
                            s += m;
                        }
                    } else if (x >= e_win || (gather_bk && x >= e_bk1 && x < e_bk)) {  // wlo..whi, or bk
                        inm |= 1u << (4 * u + j);
                    } else if (kk && x >= e_bk) {  // between the window and bk
                        msum += mass(x, zmax, c2);
                    }
                }
            }
            // the window's logits: a warp scan of the counts, one shared atomic per warp
            if (__any_sync(0xffffffffu, inm != 0u)) {
                const unsigned int cnt = __popc(inm);
                unsigned int inc = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned int y = __shfl_up_sync(0xffffffffu, inc, o);
                    if (lane >= o) inc += y;
                }
                unsigned int base = 0u;
                if (lane == 31) base = atomicAdd(&sm->nwin, inc);
                base = __shfl_sync(0xffffffffu, base, 31) + inc - cnt;
                if (inm) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (inm & (1u << (4 * u + j)))
                                win[base++] = sort_key(rw_at(q[u], j), c0 + 128 * u + 4 * lane + j);
                        }
                    }
                }
            }
            s = rw_sum(s);
            if (lane == 0 && c0 < V) {
                sm->csum[c0 / kRChunk] = s;
                if constexpr (!kMinP) asum += s;
            }
          });
        };
        if (mth)
            pass_c(RwFlag<true>{});
        else
            pass_c(RwFlag<false>{});
        uint64_t A, M = 0;  // (the scans begin with a barrier: the gather is complete after it)
        if (kk) {
            uint64_t mex_unused;
            rw_excl_scan2(asum, msum, sm, A, mex_unused, M);
        } else {
            rw_excl_scan(asum, sm, A);
        }
        const int nw = static_cast<int>(wtot);
        int np2 = 1;
        while (np2 < nw) np2 <<= 1;
        for (int i = nw + tid; i < np2; i += kRT) win[i] = 0ull;
        __syncthreads();
        rw_sort_desc(win, np2);
        // Window entries in order (z desc, id asc), thread t taking entries
        // [E t, E t + E).  The top-k part: the entries of bins < bk, then the
        // first rk entries of bin bk.  S_k = A + M + the top-k entries'
        // masses.  The last kept entry: the first whose cumulative mass from A
        // reaches ceil(top_p * S_k) (it must lie in the window proper), or with
        // top-p off the last top-k entry.
        const int E = (nw + kRT - 1) / kRT;
        const int e0 = min(nw, tid * E), e1 = min(nw, e0 + E);
        auto zof = [&](int i) { return key_float(static_cast<uint32_t>(win[i] >> 32)); };
        uint64_t nbk = 0;
        for (int i = e0; i < e1; ++i) nbk += bin(zof(i)) == bk ? 1u : 0u;
        uint64_t nbk_tot = 0, nbk_ex = 0;  // (no entry lies in bin bk with top-k off)
        if (kk) nbk_ex = rw_excl_scan(nbk, sm, nbk_tot);
        uint64_t wk = 0, ww = 0;  // top-k entries' mass; mass of the entries of the window proper
        {
            uint64_t bb = nbk_ex;  // bin-bk entries before i
            for (int i = e0; i < e1; ++i) {
                const float x = zof(i);
                const int b = bin(x);
                const bool is_bk = b == bk;
                const uint64_t m = mass(x, zmax, c2);
                if (!kk || !is_bk || bb < rk) wk += m;
                if (b <= whi && (!kk || !is_bk || bb < rk)) ww += m;
                bb += is_bk ? 1u : 0u;
            }
        }
        // with top-k off every entry is a top-k entry of the window proper: ww = wk
        uint64_t wk_tot, ww_tot, wk_ex;
        if (kk) {
            uint64_t ww_ex_unused;
            wk_ex = rw_excl_scan2(wk, ww, sm, wk_tot, ww_ex_unused, ww_tot);
        } else {
            wk_ex = rw_excl_scan(wk, sm, wk_tot);
            ww_tot = wk_tot;
        }
        const uint64_t Sk = kk ? A + M + wk_tot : S;
        const uint64_t target = p_on ? ceil_mul_p(pp, Sk) : 0ull;
        // the cut must lie in the window proper: A < target <= A + its mass
        const bool ok = !p_on || (A < target && target <= A + ww_tot);
        if (tid == 0) sm->bc[5] = ~0ull;
        __syncthreads();
        if (ok) {
            uint64_t cum = A + wk_ex, bb = nbk_ex;
            for (int i = e0; i < e1; ++i) {
                const float x = zof(i);
                const bool is_bk = bin(x) == bk;
                const bool ink = !kk || !is_bk || bb < rk;
                if (!ink) break;  // entries past the top-k part follow it
                if (p_on) {
                    const uint64_t m = mass(x, zmax, c2);
                    if (cum < target && cum + m >= target) sm->bc[5] = static_cast<unsigned long long>(i);
                    cum += m;
                } else if (is_bk && bb + 1 == rk) {
                    sm->bc[5] = static_cast<unsigned long long>(i);
                }
                bb += is_bk ? 1u : 0u;
            }
        }
        __syncthreads();
        const unsigned long long last = sm->bc[5];  // ~0: no cut (both filters off, empty window)
        if (ok) {
            if (last != ~0ull) {
                // the kept window entries join their chunks (min-p on each)
                for (int i = e0; i < e1 && static_cast<unsigned long long>(i) <= last; ++i) {
                    const uint64_t m = mass(zof(i), zmax, c2);
                    if (m && m >= mth)
                        atomicAdd(&sm->csum[sort_key_id(win[i]) / kRChunk], static_cast<unsigned long long>(m));
                }
                kept_fn_cut = true;
                cut_key = static_cast<uint32_t>(win[last] >> 32);
                cut_id = sort_key_id(win[last]);
            }
            done = true;
        }
        __syncthreads();
    }
    if (!done) {
        // ---- the window is too large, or (not expected) the cut lies outside
        // it: exact radix selection over the row
        for (int i = tid; i < kRChunks; i += kRT) sm->csum[i] = 0ull;
        __syncthreads();
        auto all = [&](float, int) { return true; };
        uint32_t k_key = 0u;
        int k_id = 0x7fffffff;
        if (kk) {
            uint64_t above = 0;
            k_key = rw_radix<false>(sm, z, V, a16, all, zmax, c2, static_cast<uint64_t>(kk), above);
            k_id = rw_tie(sm, z, V, all, k_key, static_cast<uint64_t>(kk) - above);
        }
        auto ink = [&](float x, int i) {
            if (!kk) return true;
            const uint32_t key = okey(x);
            return key > k_key || (key == k_key && i <= k_id);
        };
        if (p_on) {
            // S_k: the mass of the top-k set, then the top-p cut within it
            uint64_t sk = 0;
            rw_sweep(z, V, a16, [&](int e, const float4& q) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float x = rw_at(q, j);
                    if (x > -INFINITY && ink(x, e + j)) sk += mass(x, zmax, c2);
                }
            });
            uint64_t Sk;
            rw_excl_scan(sk, sm, Sk);
            const uint64_t target = ceil_mul_p(pp, Sk);
            uint64_t above = 0;
            const uint32_t pk = rw_radix<true>(sm, z, V, a16, ink, zmax, c2, target, above);
            const uint64_t mt = mass(key_float(pk), zmax, c2);
            const uint64_t need = (mt > 0 && target > above) ? (target - above + mt - 1) / mt : 1ull;
            cut_key = pk;
            cut_id = rw_tie(sm, z, V, ink, pk, need);
            kept_fn_cut = true;
        } else if (kk) {
            cut_key = k_key;
            cut_id = k_id;
            kept_fn_cut = true;
        }
        // chunk sums of the kept masses
        rw_sweep_chunks(z, V, a16, [&](int c0, const float4 (&q)[4]) {
            uint64_t s = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float x = rw_at(q[u], j);
                    if (!(x > -INFINITY)) continue;
                    const uint32_t key = okey(x);
                    const int id = c0 + 128 * u + 4 * lane + j;
                    if (kept_fn_cut && !(key > cut_key || (key == cut_key && id <= cut_id))) continue;
                    const uint64_t m = mass(x, zmax, c2);
                    s += m >= mth ? m : 0ull;
                }
            }
            s = rw_sum(s);
            if (lane == 0 && c0 < V) sm->csum[c0 / kRChunk] = s;
        });
    }
    __syncthreads();

    // ---- the draw: chunk holding X = floor(u * S_p), then one warp walks it
    static_assert(kRChunks <= kRT, "one chunk per thread");
    const int nch = (V + kRChunk - 1) / kRChunk;
    const uint64_t cs = tid < nch ? sm->csum[tid] : 0ull;
    uint64_t Sp;
    const uint64_t run = rw_excl_scan(cs, sm, Sp);
    const uint64_t X = static_cast<uint64_t>((static_cast<unsigned __int128>(sm->u53) * Sp) >> 53);
    if (tid == 0) sm->bc[7] = ~0ull;
    __syncthreads();
    if (cs && run <= X && X < run + cs) sm->bc[7] = static_cast<unsigned long long>(tid);
    __syncthreads();
    const unsigned long long cw = sm->bc[7];
    if (warp != 0 || cw == ~0ull) return;
    const int ch = static_cast<int>(cw);
    uint64_t base;  // the kept mass of the chunks before ch
    {
        uint64_t p = 0;
        for (int c = lane; c < ch; c += 32) p += sm->csum[c];
        base = rw_sum(p);
    }
    // lane l: the 16 ids from ch * kRChunk + 16 l, in order
    const int e = ch * kRChunk + 16 * lane;
    uint64_t m16[16];
    uint64_t mine = 0;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const float4 q = rw_load4(z, V, e + 4 * v, a16);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float x = rw_at(q, j);
            uint64_t m = 0;
            if (x > -INFINITY) {
                const uint32_t key = okey(x);
                const bool keep = !kept_fn_cut || key > cut_key || (key == cut_key && e + 4 * v + j <= cut_id);
                if (keep) {
                    m = mass(x, zmax, c2);
                    m = m >= mth ? m : 0ull;
                }
            }
            m16[4 * v + j] = m;
            mine += m;
        }
    }
    uint64_t inc = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    const uint64_t before = base + inc - mine;
    if (before <= X && X < before + mine) {
        uint64_t cum = before;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            cum += m16[j];
            if (cum > X) {
                *tok_out = e + j;
                break;
            }
        }
    }
}


__global__ void __launch_bounds__(kRT, 4)
    sampler_rows_kernel(int32_t* __restrict__ tokens, const float* __restrict__ logits, int V,
                        const float* __restrict__ temperature, const int32_t* __restrict__ top_k,
                        const float* __restrict__ top_p, const float* __restrict__ min_p,
                        const uint64_t* __restrict__ seeds, const uint64_t* __restrict__ offsets, int32_t* status,
                        int B) {
    __shared__ RowSmem smem;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int row = rw_lpt_row(B, V, temperature, top_k, top_p, &smem);
    if (row < 0)
        rw_sample_row(static_cast<int>(blockIdx.x), tokens, logits, V, temperature, top_k, top_p, min_p, seeds,
                      offsets, status, &smem);
    else
        rw_sample_row(row, tokens, logits, V, temperature, top_k, top_p, min_p, seeds, offsets, status, &smem);
}

bool sampler_rows_fits(int B, int V, int sms) { return V >= 1 && V <= kRowMaxV && B > 2 * sms && B < (1 << 21); }

cudaError_t launch_sampler_rows(int32_t* tokens, const float* logits, int B, int V, const float* temperature,
                                const int32_t* top_k, const float* top_p, const float* min_p,
                                const uint64_t* seeds, const uint64_t* offsets, int32_t* status,
                                cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B), 1, 1);
    cfg.blockDim = dim3(kRT, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sampler_rows_kernel, tokens, logits, V, temperature, top_k, top_p, min_p, seeds,
                              offsets, status, B);
}

}  // namespace pkv
