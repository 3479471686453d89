// sampler.cu -- logits -> token: temperature, top-k, top-p, renormalise, seeded draw.
//
// Definitions ("Suy luan & Toi uu hoa (Inference)" 1.2; "Bai Lab tong hop --
// Inference Engineering" block [8]; "LLM inference serving tutorial" 3.1, 1.6):
//   T == 0 -> argmax (lowest id among ties).  Otherwise p_i = exp((z_i - zmax)/T)
//   over finite logits; top-k keeps the k first under (z desc, id asc); top-p keeps
//   the smallest prefix of that order whose renormalised cumulative mass reaches
//   top_p (boundary kept); the draw walks kept ids in ascending order and returns
//   the first whose running mass exceeds u * (kept mass), u from Philox4x64-10
//   (key = (seed, 0), counter = (offset, 0, 0, 0), word 0 >> 11, times 2^-53).
//
// GB300 design: one thread-block cluster (up to 8 CTAs) per row; each CTA pulls
// its slice of the row from HBM once (1-D TMA bulk copy) into shared memory, and
// every later pass runs on chip; CTAs exchange small summaries through
// distributed shared memory.  A token's mass is exp2((z - zmax) * log2(e)/T) in
// fp32 turned into 64-bit fixed point (floor(w * 2^40)), so every sum, cut and
// CDF comparison is exact integer arithmetic and run-to-run deterministic.
//  * top-k rows: a histogram of 2048 bins linear in (zmax - z) finds the bin of
//    the k-th largest logit; the candidates above it (a superset of the top-k set,
//    typically k plus a few) are gathered into rank 0, which sorts them by
//    (z desc, id asc) and finishes top-k, top-p and the draw alone;
//  * top-p-only rows: the same bins carry fp32 masses that locate the cut
//    approximately; the bins around it are gathered into rank 0 and the exact
//    cut is found there, verified against exact fixed-point masses; every CTA
//    then walks its slice for the draw;
//  * rows that fail either fast path (too many candidates, or a cut outside the
//    window) take an exact radix search over 11/11/10-bit key digits with
//    64-bit shared-memory histograms.
#include <cooperative_groups.h>
#include <limits.h>
#include <math.h>

#include <map>
#include <mutex>
#include <tuple>

#include "pkv_common.cuh"
#include "sampling_math.cuh"

namespace cg = cooperative_groups;

namespace pkv {

constexpr int kST = 512;           // threads per CTA
constexpr int kSW = kST / 32;      // warps per CTA
constexpr int kHistBins = 2048;    // widest radix digit (11 bits) and linear bins
constexpr int kListCap = 2048;     // candidate list capacity (rank 0, gathered)
constexpr int kTopkBins = 512;     // bins of the bounded top-k histogram
constexpr int kLocBase = 1024;     // hist[kLocBase..kHistBins): this CTA's top-k candidates
constexpr int kLocCap = kHistBins - kLocBase;
constexpr int kRegTopk = 256;      // largest top-k taken from the first pass's thread maxima
constexpr int kMaxCluster = 8;
constexpr int kSliceSmemMax = 24576;  // floats of a row slice kept in shared memory

struct __align__(16) SampSmem {
    unsigned long long hist[kHistBins];  // u64 radix histogram, or u32 counts + f32 masses
    unsigned long long list[kListCap];   // rank 0: gathered candidates (sort keys)
    unsigned long long xch[2][8];
    unsigned long long gath[kMaxCluster][8];
    unsigned long long wsum[kSW];
    unsigned long long bc[8];
    unsigned long long aslot[kMaxCluster];
    unsigned long long bslot[kMaxCluster];
    uint64_t bar[4];        // one per chunk of the slice load
    unsigned int gcount;    // rank 0: candidates gathered so far
    int imin;
    unsigned int lcount;    // this CTA's top-k candidates (sort keys in hist[kLocBase..]), or its rescanning threads
    int pad_;
    unsigned long long u53;  // the row's uniform draw, top 53 bits of Philox word 0
    unsigned long long pad2_;
};
// The row slice follows the struct in shared memory; TMA bulk copies and the
// 16-byte vector loads need it 16-byte aligned.
static_assert(sizeof(SampSmem) % 16 == 0, "slice after SampSmem must stay 16-byte aligned");

// ------------------------------------------------------------------ block primitives
__device__ __forceinline__ uint64_t block_excl_scan_u64(uint64_t v, unsigned long long* wsum, uint64_t& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint64_t t = lane < kSW ? wsum[lane] : 0ull;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < kSW) wsum[lane] = t;
    }
    __syncthreads();
    const uint64_t before = warp ? wsum[warp - 1] : 0ull;
    total = wsum[kSW - 1];
    __syncthreads();
    return before + x - v;
}

// Odd per-thread run length, so that thread-contiguous runs hit distinct banks.
__device__ __forceinline__ int run_len(int n) {
    int e = (n + kST - 1) / kST;
    if (e < 1) e = 1;
    return (e & 1) ? e : e + 1;
}

// ------------------------------------------------------------------ context
struct View {
    const float* z;
    const int* id;  // nullptr: ids are idbase + i
    int n;
    int idbase;
    bool g16;  // z is a 16-byte aligned global pointer (4-wide loads allowed inside [0, n))
    __device__ __forceinline__ int idat(int i) const { return id ? id[i] : idbase + i; }
};

struct Keep {
    bool k_on, p_on;
    uint64_t mth;  // min-p: a kept token's mass must be >= mth (0: off)
    uint32_t tauk, taup;
    int idk, idp;
    float zk, zp;  // key_float(tauk), key_float(taup)
    // Same predicates on floats (-0.0 == +0.0 as with the keys); -inf never passes.
    __device__ __forceinline__ bool keep_f(float z, int id) const {
        const bool ok_k = !k_on || z > zk || (z == zk && id <= idk);
        const bool ok_p = !p_on || z > zp || (z == zp && id <= idp);
        return ok_k && ok_p && z > -INFINITY;
    }
    __device__ __forceinline__ bool topk(uint32_t key, int id) const {
        return !k_on || key > tauk || (key == tauk && id <= idk);
    }
    __device__ __forceinline__ bool topp(uint32_t key, int id) const {
        return !p_on || key > taup || (key == taup && id <= idp);
    }
};

struct Ctx {
    SampSmem* sm;
    int nc, rank, xb;
    __device__ __forceinline__ int nce() const { return nc; }
    __device__ __forceinline__ int rke() const { return rank; }
    __device__ __forceinline__ void csync() const { cg::this_cluster().sync(); }
    template <typename T>
    __device__ __forceinline__ T* remote(T* p, int r) const {
        return cg::this_cluster().map_shared_rank(p, r);
    }
};

// Split cluster barrier: arrive (release) as soon as this CTA's remote reads are
// done, wait (acquire) only before leaving.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Bitonic sort of a[0..n) (n a power of two) in shared memory by one CTA.
__device__ void bitonic_sort(unsigned long long* a, int n, bool descending) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += kST) {
                const int l = i ^ j;
                if (l > i) {
                    const bool up = ((i & k) == 0) != descending;
                    const unsigned long long x = a[i], y = a[l];
                    if ((x > y) == up) {
                        a[i] = y;
                        a[l] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
}

__device__ __forceinline__ int pow2_ceil(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

// Publish xch[xb][0..k) (written by thread 0 before the call) to every CTA of
// the cluster; afterwards gath[j][s] holds rank j's value s.
__device__ void exch(Ctx& c, int k) {
    SampSmem* sm = c.sm;
    c.csync();
    const int nce = c.nce();
    if (static_cast<int>(threadIdx.x) < nce * k) {
        const int j = threadIdx.x / k, s = threadIdx.x % k;
        sm->gath[j][s] = c.remote(&sm->xch[c.xb][0], j)[s];
    }
    __syncthreads();
    c.xb ^= 1;
}

// One radix pass: histogram (count or fixed-point mass) of the next digit of
// the keys that match `prefix` and pass the top-k filter, summed over the
// cluster; then the digit at which the cumulative weight (from the largest key
// down, starting at `above`) first reaches `target`.  With p_first the target is
// ceil(top_p * total) where total is this pass's whole weight (returned in S).
template <bool kMass>
__device__ void radix_pass(Ctx& c, const View& v, const Keep& kp, bool use_topk, uint32_t prefix, int pbits,
                           int shift, int nbits, uint64_t& target, uint64_t& above, uint32_t& digit, uint64_t& binw,
                           float zmax, float c2, bool p_first, float top_p, uint64_t* S_out) {
    SampSmem* sm = c.sm;
    const int tid = threadIdx.x;
    const int nb = 1 << nbits;
    for (int i = tid; i < nb; i += kST) sm->hist[i] = 0ull;
    if (tid == 0) {
        sm->bc[0] = 0ull;
        sm->bc[1] = above;
        sm->bc[2] = 0ull;
    }
    __syncthreads();
    for (int i = tid; i < v.n; i += kST) {
        const float z = v.z[i];
        if (!isfinite(z)) continue;
        const uint32_t key = okey(z);
        if (pbits && (key >> (32 - pbits)) != prefix) continue;
        if (use_topk && !kp.topk(key, v.idat(i))) continue;
        const uint32_t d = (key >> shift) & static_cast<uint32_t>(nb - 1);
        const uint64_t w = kMass ? mass(z, zmax, c2) : 1ull;
        if (w) atomicAdd(&sm->hist[d], static_cast<unsigned long long>(w));
    }
    c.csync();
    const int bpt = nb / kST;  // bins per thread (4 or 2), descending order
    uint64_t vals[4];
    uint64_t tsum = 0;
    const int nce = c.nce();
    for (int q = 0; q < bpt; ++q) {
        const int bin = nb - 1 - (tid * bpt + q);
        uint64_t s = 0;
        for (int j = 0; j < nce; ++j) s += c.remote(&sm->hist[0], j)[bin];
        vals[q] = s;
        tsum += s;
    }
    uint64_t tot;
    const uint64_t ex = block_excl_scan_u64(tsum, sm->wsum, tot);
    if (p_first) {
        target = ceil_mul_p(top_p, tot);
        if (S_out) *S_out = tot;
    }
    const uint64_t c0 = above + ex;
    if (c0 < target && c0 + tsum >= target) {
        uint64_t cc = c0;
        for (int q = 0; q < bpt; ++q) {
            if (cc + vals[q] >= target) {
                sm->bc[0] = static_cast<unsigned long long>(nb - 1 - (tid * bpt + q));
                sm->bc[1] = cc;
                sm->bc[2] = vals[q];
                break;
            }
            cc += vals[q];
        }
    }
    __syncthreads();
    digit = static_cast<uint32_t>(sm->bc[0]);
    above = sm->bc[1];
    binw = sm->bc[2];
    c.csync();  // every remote reader of hist is done before it is reused
}

// Id of the r-th (1-based) element, in id order over the cluster, whose key is
// `tau` and that passes the top-k filter (when use_topk).
__device__ int tie_select(Ctx& c, const View& v, const Keep& kp, bool use_topk, uint32_t tau, uint64_t r) {
    SampSmem* sm = c.sm;
    const int tid = threadIdx.x;
    const int E = run_len(v.n);
    const int b0 = min(v.n, tid * E), b1 = min(v.n, b0 + E);
    auto match = [&](int i) {
        const float z = v.z[i];
        if (!isfinite(z)) return false;
        const uint32_t key = okey(z);
        return key == tau && (!use_topk || kp.topk(key, v.idat(i)));
    };
    uint64_t cnt = 0;
    for (int i = b0; i < b1; ++i) cnt += match(i) ? 1u : 0u;
    if (tid == 0) sm->imin = INT_MAX;
    uint64_t tot;
    const uint64_t ex = block_excl_scan_u64(cnt, sm->wsum, tot);
    if (tid == 0) sm->xch[c.xb][0] = tot;
    exch(c, 1);
    uint64_t pre = 0;
    for (int j = 0; j < c.rke(); ++j) pre += sm->gath[j][0];
    if (pre < r && r <= pre + tot) {
        const uint64_t rl = r - pre;
        if (ex < rl && rl <= ex + cnt) {
            uint64_t need = rl - ex;
            for (int i = b0; i < b1; ++i)
                if (match(i) && --need == 0) {
                    atomicMin(&sm->imin, v.idat(i));
                    break;
                }
        }
    }
    __syncthreads();
    if (tid == 0) sm->xch[c.xb][0] = static_cast<unsigned long long>(static_cast<uint32_t>(sm->imin));
    exch(c, 1);
    int best = INT_MAX;
    for (int j = 0; j < c.nce(); ++j) best = min(best, static_cast<int>(static_cast<uint32_t>(sm->gath[j][0])));
    return best;
}

// ------------------------------------------------------------------ linear bins
// Bin of a finite logit on 2048 bins linear in (zmax - z): bin 0 holds the
// largest logits.  Monotone non-increasing in z, so "bin < b" implies a larger
// logit than any element of bin b.
struct Bins {
    float zmax, scale;
    int nb;  // number of bins (<= kHistBins)
    __device__ __forceinline__ int operator()(float z) const {
        if (scale == 0.f) return 0;
        const float t = (zmax - z) * scale;
        return t >= static_cast<float>(nb - 1) ? nb - 1 : static_cast<int>(t);
    }
};

// The smallest finite logit whose bin is below c (+inf for c <= 0): the bins
// are monotone non-increasing in z, so bins(z) < c exactly when z >= this
// edge; found by bisection on the order-preserving keys (bins(zmax) = 0).
__device__ float bin_edge(const Bins& bins, int c) {
    if (c <= 0) return INFINITY;
    uint32_t lo = okey(-3.40282347e38f), hi = okey(bins.zmax);
    if (bins(key_float(lo)) < c) return key_float(lo);
    while (hi - lo > 1u) {  // bins(lo) >= c > bins(hi)
        const uint32_t mid = lo + (hi - lo) / 2u;
        if (bins(key_float(mid)) < c)
            hi = mid;
        else
            lo = mid;
    }
    return key_float(hi);
}

// Four consecutive logits of the slice starting at e (a multiple of 4); entries
// at or past n read as -inf.  vec: the slice is the shared-memory copy, padded
// with -inf up to a multiple of 4 slots.  Otherwise the slice is read from
// global memory, 16 bytes at a time where aligned and wholly inside the row.
__device__ __forceinline__ float4 load4(const View& v, int e, bool vec) {
    if (vec) return *reinterpret_cast<const float4*>(v.z + e);
    if (v.g16 && e + 4 <= v.n) return __ldg(reinterpret_cast<const float4*>(v.z + e));
    float4 q;
    {
        q.x = e < v.n ? v.z[e] : 0.f;
        q.y = e + 1 < v.n ? v.z[e + 1] : 0.f;
        q.z = e + 2 < v.n ? v.z[e + 2] : 0.f;
        q.w = e + 3 < v.n ? v.z[e + 3] : 0.f;
    }
    if (e >= v.n) q.x = -INFINITY;
    if (e + 1 >= v.n) q.y = -INFINITY;
    if (e + 2 >= v.n) q.z = -INFINITY;
    if (e + 3 >= v.n) q.w = -INFINITY;
    return q;
}
__device__ __forceinline__ float f4at(const float4& q, int j) {
    return j == 0 ? q.x : (j == 1 ? q.y : (j == 2 ? q.z : q.w));
}

// Strided sweep over the 4-wide slots of the slice: slot e = 4 * (tid + kST * i).
// kU slots are loaded before any is processed, so that a thread keeps kU loads
// in flight when the slice is read from global memory.  The trip count is the
// same for every lane of a warp (lanes past the end see -inf), so f may use
// warp-collective operations.  f(e, q) gets the slot and its four logits.
template <int kU, typename F>
__device__ __forceinline__ void sweep4(const View& v, int nvec, bool vec, F&& f) {
    const int lane = threadIdx.x & 31;
    for (int e0 = 4 * (static_cast<int>(threadIdx.x) - lane); e0 < nvec; e0 += 4 * kST * kU) {
        float4 q[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int el = e0 + 4 * lane + 4 * kST * u;
            q[u] = el < nvec ? load4(v, el, vec) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) f(e0 + 4 * lane + 4 * kST * u, q[u]);
    }
}

// Per-thread run length for thread-contiguous passes: a multiple of 4 with an
// odd quotient, so that 16-byte loads of a quarter-warp hit distinct banks.
__device__ __forceinline__ int run_len4(int n) {
    int q = (n + 4 * kST - 1) / (4 * kST);
    if (q < 1) q = 1;
    if (!(q & 1)) ++q;
    return 4 * q;
}

// Append the lane's candidate (when pred) to rank 0's gathered list; one remote
// atomic per warp and element slot.  Every lane of the warp must call this.
__device__ __forceinline__ void gather_push(bool pred, unsigned long long key, unsigned int* gcount0,
                                            unsigned long long* list0, int cap = kListCap) {
    const unsigned int mask = __ballot_sync(0xffffffffu, pred);
    if (mask == 0u) return;
    const int lane = threadIdx.x & 31;
    unsigned int base = 0;
    if (lane == __ffs(mask) - 1) base = atomicAdd(gcount0, static_cast<unsigned int>(__popc(mask)));
    base = __shfl_sync(0xffffffffu, base, __ffs(mask) - 1);
    if (pred) {
        const unsigned int pos = base + static_cast<unsigned int>(__popc(mask & ((1u << lane) - 1u)));
        if (pos < static_cast<unsigned int>(cap)) list0[pos] = key;
    }
}

// Sum over the cluster of this thread's 4 consecutive histogram bins (16-byte
// remote loads, issued four ranks at a time).
__device__ __forceinline__ void sum_remote_u4(cg::cluster_group& cl, unsigned int* h, int nc, uint32_t (&g)[4]) {
#pragma unroll
    for (int r0 = 0; r0 < kMaxCluster; r0 += 4) {
        uint4 t[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (r0 + j < nc) t[j] = reinterpret_cast<const uint4*>(cl.map_shared_rank(h, r0 + j))[threadIdx.x];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (r0 + j < nc) {
                g[0] += t[j].x;
                g[1] += t[j].y;
                g[2] += t[j].z;
                g[3] += t[j].w;
            }
    }
}
__device__ __forceinline__ void sum_remote_f4(cg::cluster_group& cl, float* h, int nc, float (&g)[4]) {
#pragma unroll
    for (int r0 = 0; r0 < kMaxCluster; r0 += 4) {
        float4 t[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (r0 + j < nc) t[j] = reinterpret_cast<const float4*>(cl.map_shared_rank(h, r0 + j))[threadIdx.x];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (r0 + j < nc) {
                g[0] += t[j].x;
                g[1] += t[j].y;
                g[2] += t[j].z;
                g[3] += t[j].w;
            }
    }
}

// ------------------------------------------------------------------ draw (whole cluster)
// First kept id (ascending) whose running fixed-point mass exceeds
// floor(u * S_p), S_p = total kept mass.  The CTA that holds it writes the token.
// The slice is cut into chunks of 128 * cpw consecutive logits (cpw chosen so
// that there are at most kHistBins chunks); warp w sums the kept masses of
// chunks w, w + 16, ..., four chunks at a time, with coalesced 16-byte loads
// (lane l takes logits 4l..4l+3 of each 128), the chunk sums are scanned in
// shared memory (hist is free here), the CTA totals are exchanged, and in the
// CTA that holds the draw one warp walks the single chunk that holds it.
// Ends with this CTA's arrival on the cluster barrier; the caller waits on it.
__device__ void draw_pass(Ctx& c, const View& v, const Keep& kp, bool vec, float zmax, float c2,
                          int32_t* tok_out) {
    SampSmem* sm = c.sm;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nvec = (v.n + 3) & ~3;
    const int cpw = max(1, (nvec + 128 * kHistBins - 1) / (128 * kHistBins));
    const int csz = 128 * cpw;
    const int nch = (nvec + csz - 1) / csz;
    const bool filt = kp.k_on || kp.p_on;
    // -inf logits weigh 0, so without a filter every slot is simply summed
    auto kmass = [&](float z, int e) -> uint64_t {
        const uint64_t m = (!filt || kp.keep_f(z, v.idbase + e)) ? mass(z, zmax, c2) : 0ull;
        return m >= kp.mth ? m : 0ull;
    };
    // warp w takes chunks w, w + 16, w + 32, w + 48 together (four loads in
    // flight per lane), then w + 64, ...; slots past the end read as -inf (mass 0)
    constexpr int kDU = 4;
    unsigned long long* ctot = sm->hist;
    for (int cb = warp; cb < nch; cb += kDU * kSW) {
        uint64_t w[kDU];
#pragma unroll
        for (int u = 0; u < kDU; ++u) w[u] = 0;
        for (int k = 0; k < cpw; ++k) {
            float4 q[kDU];
#pragma unroll
            for (int u = 0; u < kDU; ++u) {
                const int e = (cb + u * kSW) * csz + 128 * k + 4 * lane;
                q[u] = e < nvec ? load4(v, e, vec) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
#pragma unroll
            for (int u = 0; u < kDU; ++u) {
                const int e = (cb + u * kSW) * csz + 128 * k + 4 * lane;
                w[u] += kmass(q[u].x, e) + kmass(q[u].y, e + 1) + kmass(q[u].z, e + 2) + kmass(q[u].w, e + 3);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int u = 0; u < kDU; ++u) w[u] += __shfl_xor_sync(0xffffffffu, w[u], o);
        if (lane == 0)
#pragma unroll
            for (int u = 0; u < kDU; ++u)
                if (cb + u * kSW < nch) ctot[cb + u * kSW] = w[u];
    }
    __syncthreads();
    // exclusive scan of the chunk sums, four consecutive chunks per thread
    uint64_t t4[4], ts = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int ch = 4 * tid + q;
        t4[q] = ch < nch ? ctot[ch] : 0ull;
        ts += t4[q];
    }
    uint64_t tot;
    uint64_t run = block_excl_scan_u64(ts, sm->wsum, tot);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int ch = 4 * tid + q;
        if (ch < nch) ctot[ch] = run;
        run += t4[q];
    }
    if (tid == 0) sm->xch[c.xb][0] = tot;
    exch(c, 1);  // its barriers also publish the scanned chunk sums
    uint64_t Sp = 0, pre = 0;
    for (int j = 0; j < c.nc; ++j) {
        Sp += sm->gath[j][0];
        if (j < c.rank) pre += sm->gath[j][0];
    }
    cluster_arrive();  // all remote reads of this CTA are done
    const uint64_t u53 = sm->u53;
    const uint64_t X = static_cast<uint64_t>((static_cast<unsigned __int128>(u53) * Sp) >> 53);  // floor(u*Sp) < Sp
    if (!(pre <= X && X < pre + tot)) return;  // the draw lies in another CTA
    const uint64_t Xr = X - pre;
    // the chunk holding Xr: the last chunk whose exclusive prefix is <= Xr and that
    // has mass (found by the thread that owns it; a unique match)
    if (tid == 0) sm->imin = -1;
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int ch = 4 * tid + q;
        if (ch < nch) {
            const uint64_t lo = ctot[ch], hi = ch + 1 < nch ? ctot[ch + 1] : tot;
            if (lo <= Xr && Xr < hi) sm->imin = ch;
        }
    }
    __syncthreads();
    const int cs = sm->imin;
    if (warp != 0 || cs < 0) return;
    uint64_t base = ctot[cs];
    for (int k = 0; k < cpw; ++k) {
        const int e = cs * csz + 128 * k + 4 * lane;
        float4 q = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (e < nvec) q = load4(v, e, vec);
        const uint64_t m0 = kmass(q.x, e), m1 = kmass(q.y, e + 1), m2 = kmass(q.z, e + 2), m3 = kmass(q.w, e + 3);
        const uint64_t mine = m0 + m1 + m2 + m3;
        uint64_t inc = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        const uint64_t before = base + inc - mine;
        if (before <= Xr && Xr < before + mine) {
            // the 4 logits of this lane: first whose running mass passes Xr
            uint64_t cum = before;
            const uint64_t ms[4] = {m0, m1, m2, m3};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                cum += ms[j];
                if (cum > Xr) {
                    *tok_out = v.idbase + e + j;
                    break;
                }
            }
        }
        base += __shfl_sync(0xffffffffu, inc, 31);
        if (base > Xr) break;  // found (warp-uniform)
    }
}

// ------------------------------------------------------------------ rank-0 finish on a gathered list
// The list holds n distinct candidate sort keys, a superset of the top-kk set.
// Small lists (n <= 128): G threads per candidate (G = 8 for n <= 64, else 4;
// candidate i = tid / G), each taking every G-th candidate j.  One loop gives
// the candidate's rank (larger keys) and the mass of the larger keys, its
// prefix in the order (z desc, id asc); S_k is that prefix plus the own mass
// of the candidate of rank kk - 1.  A second loop, over the kept masses, gives
// the kept mass at smaller ids and the kept total S_p; the candidate whose
// interval holds X = floor(u * S_p) is the token.  Two barriers, no atomics.
constexpr int kSmallList = 128;

__device__ __noinline__ void solo_finish_small(SampSmem* sm, int n, int kk, float pp, uint64_t mth, float zmax, float c2,
                                  int32_t* tok_out) {
    const int tid = threadIdx.x;
    const unsigned long long* a = sm->list;
    unsigned long long* wk = sm->hist;                                   // [128] kept masses (0: not kept)
    unsigned int* ids = reinterpret_cast<unsigned int*>(sm->hist + 128);  // [128] token ids
    unsigned long long* skp = sm->hist + 192;                             // S_k
    const int lg = n <= 64 ? 3 : 2;
    const int G = 1 << lg;
    const int i = tid >> lg, p = tid & (G - 1);
    const bool lead = i < n && p == 0;
    const unsigned long long key = i < n ? a[i] : ~0ull;  // (an invalid slot counts no larger key)
    const int ke = min(kk, n);
    uint32_t cnt = 0u;
    uint64_t P = 0;
    for (int j = p; j < n; j += G) {
        const unsigned long long kj = a[j];
        if (kj > key) {
            ++cnt;
            P += mass(key_float(static_cast<uint32_t>(kj >> 32)), zmax, c2);
        }
    }
    for (int o = 1; o < G; o <<= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        P += __shfl_xor_sync(0xffffffffu, P, o);
    }
    const uint64_t Wi = i < n ? mass(key_float(static_cast<uint32_t>(key >> 32)), zmax, c2) : 0ull;
    if (lead && cnt == static_cast<uint32_t>(ke - 1)) *skp = P + Wi;
    __syncthreads();
    // top-k, then top-p on the top-k set in rank order, then min-p
    bool kept = i < n && cnt < static_cast<uint32_t>(ke);
    if (pp < 1.f) kept = kept && P < ceil_mul_p(pp, *skp);
    const uint64_t wi = (kept && Wi >= mth) ? Wi : 0ull;
    const unsigned int idi = static_cast<unsigned int>(sort_key_id(key));
    if (lead) {
        wk[i] = wi;
        ids[i] = idi;
    }
    __syncthreads();
    // the draw: kept tokens in id order
    uint64_t Q = 0, Sp = 0;
    for (int j = p; j < n; j += G) {
        const uint64_t wj = wk[j];
        Sp += wj;
        Q += ids[j] < idi ? wj : 0ull;
    }
    for (int o = 1; o < G; o <<= 1) {
        Q += __shfl_xor_sync(0xffffffffu, Q, o);
        Sp += __shfl_xor_sync(0xffffffffu, Sp, o);
    }
    const uint64_t X = static_cast<uint64_t>((static_cast<unsigned __int128>(sm->u53) * Sp) >> 53);
    if (lead && wi > 0 && Q <= X && X < Q + wi) *tok_out = static_cast<int>(idi);
}

// Larger lists: bitonic sort by (z desc, id asc), keep the first kk, apply
// top-p exactly, re-sort the kept tokens by id and draw.
__device__ void solo_finish(SampSmem* sm, int n, int kk, float pp, uint64_t mth, float zmax, float c2,
                            int32_t* tok_out) {
    if (n <= kSmallList) {
        solo_finish_small(sm, n, kk, pp, mth, zmax, c2, tok_out);
        return;
    }
    const int tid = threadIdx.x;
    unsigned long long* a = sm->list;
    const int np2 = pow2_ceil(n);
    for (int i = n + tid; i < np2; i += kST) a[i] = 0ull;
    if (tid == 0) sm->bc[1] = static_cast<unsigned long long>(min(kk, n));
    __syncthreads();
    bitonic_sort(a, np2, true);
    const int m0 = min(kk, n);
    int m = m0;
    {
        const int E = run_len(m0);
        const int b0 = min(m0, tid * E), b1 = min(m0, b0 + E);
        uint64_t w = 0;
        for (int j = b0; j < b1; ++j) w += mass(key_float(static_cast<uint32_t>(a[j] >> 32)), zmax, c2);
        uint64_t tot;
        const uint64_t ex = block_excl_scan_u64(w, sm->wsum, tot);
        if (pp < 1.f) {
            const uint64_t target = ceil_mul_p(pp, tot);
            if (ex < target && ex + w >= target) {
                uint64_t cum = ex;
                for (int j = b0; j < b1; ++j) {
                    cum += mass(key_float(static_cast<uint32_t>(a[j] >> 32)), zmax, c2);
                    if (cum >= target) {
                        sm->bc[1] = static_cast<unsigned long long>(j + 1);
                        break;
                    }
                }
            }
            __syncthreads();
            m = static_cast<int>(sm->bc[1]);
        }
    }
    __syncthreads();
    // kept tokens re-keyed as (id << 41 | mass) and sorted by id
    for (int j = tid; j < m; j += kST) {
        const unsigned long long k = a[j];
        uint64_t W = mass(key_float(static_cast<uint32_t>(k >> 32)), zmax, c2);
        W = W >= mth ? W : 0ull;  // min-p, after top-p: weighs nothing in the draw
        a[j] = (static_cast<unsigned long long>(sort_key_id(k)) << 41) | W;
    }
    const int mp2 = pow2_ceil(m);
    for (int i = m + tid; i < mp2; i += kST) a[i] = ~0ull;
    __syncthreads();
    bitonic_sort(a, mp2, false);
    const unsigned long long wmask = (1ull << 41) - 1;
    const int E = run_len(m);
    const int b0 = min(m, tid * E), b1 = min(m, b0 + E);
    uint64_t w = 0;
    for (int j = b0; j < b1; ++j) w += a[j] & wmask;
    uint64_t Sp;
    const uint64_t ex = block_excl_scan_u64(w, sm->wsum, Sp);
    const uint64_t u53 = sm->u53;
    const uint64_t X = static_cast<uint64_t>((static_cast<unsigned __int128>(u53) * Sp) >> 53);
    if (ex <= X && X < ex + w) {
        uint64_t cum = ex;
        for (int j = b0; j < b1; ++j) {
            cum += a[j] & wmask;
            if (cum > X) {
                *tok_out = static_cast<int>(a[j] >> 41);
                break;
            }
        }
    }
}

// ------------------------------------------------------------------ exact fallback (whole cluster)
__device__ void fallback_select_and_draw(Ctx& c, const View& v, Keep& kp, bool vec, int kk, float pp, float zmax,
                                         float c2, int32_t* tok_out) {
    if (kk > 0) {
        kp.k_on = true;
        uint64_t target = static_cast<uint64_t>(kk), above = 0, binw = 0;
        uint32_t d0, d1, d2;
        radix_pass<false>(c, v, kp, false, 0u, 0, 21, 11, target, above, d0, binw, zmax, c2, false, 0.f, nullptr);
        radix_pass<false>(c, v, kp, false, d0, 11, 10, 11, target, above, d1, binw, zmax, c2, false, 0.f, nullptr);
        radix_pass<false>(c, v, kp, false, (d0 << 11) | d1, 22, 0, 10, target, above, d2, binw, zmax, c2, false, 0.f,
                          nullptr);
        kp.tauk = (d0 << 21) | (d1 << 10) | d2;
        kp.zk = key_float(kp.tauk);
        kp.idk = tie_select(c, v, kp, false, kp.tauk, target - above);
    }
    if (pp < 1.f) {
        kp.p_on = true;
        uint64_t target = 0, above = 0, binw = 0, Sk = 0;
        uint32_t d0, d1, d2;
        radix_pass<true>(c, v, kp, true, 0u, 0, 21, 11, target, above, d0, binw, zmax, c2, true, pp, &Sk);
        radix_pass<true>(c, v, kp, true, d0, 11, 10, 11, target, above, d1, binw, zmax, c2, false, 0.f, nullptr);
        radix_pass<true>(c, v, kp, true, (d0 << 11) | d1, 22, 0, 10, target, above, d2, binw, zmax, c2, false, 0.f,
                         nullptr);
        kp.taup = (d0 << 21) | (d1 << 10) | d2;
        const uint64_t wt = mass(key_float(kp.taup), zmax, c2);
        uint64_t need = 1;
        if (wt > 0 && target > above) need = (target - above + wt - 1) / wt;
        kp.zp = key_float(kp.taup);
        kp.idp = tie_select(c, v, kp, true, kp.taup, need);
    }
    draw_pass(c, v, kp, vec, zmax, c2, tok_out);
}

// ------------------------------------------------------------------ row order
// The row a cluster takes when the batch has more rows than SMs: the rows with
// the most work get the lowest cluster indices, so they start first and, with
// one CTA per row, rarely share an SM (longest-processing-time-first order; the
// tokens do not depend on it).  Classes: 2 = top-p alone (the cut and a draw
// over a long kept prefix), 1 = top-k above kRegTopk or no truncation,
// 0 = greedy, small top-k or invalid parameters; order: class descending, row
// index ascending.  Counts per class travel packed in 21-bit fields of one
// block-wide scan (B < 2^21).
__device__ int lpt_row(int B, int V, const float* __restrict__ temperature, const int32_t* __restrict__ top_k,
                       const float* __restrict__ top_p, int unit, SampSmem* sm) {
    const int tid = threadIdx.x;
    constexpr uint64_t kF = (1ull << 21) - 1ull;
    auto cls = [&](int r) -> int {
        const float t = temperature[r];
        const int k = top_k[r];
        if (!(t > 0.f)) return 0;
        const bool k_on = k > 0 && k < V;
        if (k_on && k <= kRegTopk) return 0;
        if (!k_on && top_p[r] < 1.f) return 2;
        return 1;
    };
    uint64_t tot = 0;
    for (int r0 = 0; r0 < B; r0 += kST) {
        const int r = r0 + tid;
        uint64_t t;
        block_excl_scan_u64(r < B ? (1ull << (21 * cls(r))) : 0ull, sm->wsum, t);
        tot += t;
    }
    const uint64_t n2 = (tot >> 42) & kF, n1 = (tot >> 21) & kF;
    if (tid == 0) sm->bc[7] = 0ull;
    __syncthreads();
    uint64_t run = 0;
    for (int r0 = 0; r0 < B; r0 += kST) {
        const int r = r0 + tid;
        const int c = r < B ? cls(r) : 0;
        uint64_t t;
        const uint64_t ex = block_excl_scan_u64(r < B ? (1ull << (21 * c)) : 0ull, sm->wsum, t);
        if (r < B) {
            const uint64_t base = c == 2 ? 0ull : (c == 1 ? n2 : n2 + n1);
            const uint64_t pos = base + (((run + ex) >> (21 * c)) & kF);
            if (pos == static_cast<uint64_t>(unit)) sm->bc[7] = static_cast<unsigned long long>(r);
        }
        run += t;
    }
    __syncthreads();
    const int row = static_cast<int>(sm->bc[7]);
    __syncthreads();
    return row;
}

// ------------------------------------------------------------------ kernel
constexpr int kLoadChunks = 4;

__global__ void __launch_bounds__(kST, 2)
    sampler_kernel(int32_t* __restrict__ tokens, const float* __restrict__ logits, int V, int S, int smem_slice,
                   const float* __restrict__ temperature, const int32_t* __restrict__ top_k,
                   const float* __restrict__ top_p, const float* __restrict__ min_p,
                   const uint64_t* __restrict__ seeds, const uint64_t* __restrict__ offsets, int32_t* status,
                   int lpt_B) {
    extern __shared__ __align__(16) uint8_t samp_smem_raw[];
    SampSmem* sm = reinterpret_cast<SampSmem*>(samp_smem_raw);
    float* zslice = reinterpret_cast<float*>(samp_smem_raw + sizeof(SampSmem));
    cg::cluster_group cluster = cg::this_cluster();
    Ctx c;
    c.sm = sm;
    c.nc = static_cast<int>(cluster.num_blocks());
    c.rank = static_cast<int>(cluster.block_rank());
    c.xb = 0;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // launched as a programmatic dependent: the row parameters and the logits
    // are read only after the predecessor grid has finished
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int unit = static_cast<int>(blockIdx.x) / c.nc;  // this CTA's cluster
    const int row = lpt_B ? lpt_row(lpt_B, V, temperature, top_k, top_p, unit, sm) : unit;
    const int lo = c.rank * S;
    const int n = max(0, min(S, V - lo));
    const float* grow = logits + static_cast<size_t>(row) * V + lo;
    int32_t* tok_out = tokens + row;

    View v;
    v.id = nullptr;
    v.n = n;
    v.idbase = lo;
    v.z = smem_slice ? zslice : grow;
    v.g16 = (reinterpret_cast<uintptr_t>(grow) & 15u) == 0;
    const bool vec = smem_slice != 0;

    // row parameters first: they decide what the passes must track
    const float T = temperature[row];
    const float pp = top_p[row];
    const float mp = min_p ? min_p[row] : 0.f;
    const int kk_in = top_k[row];
    const uint64_t seed = seeds[row], offset = offsets[row];
    const int nvec = (n + 3) & ~3;  // element slots visited by the 4-wide loops

    // ---- load (chunked bulk copies) overlapped with the first pass: max and min
    // over finite logits, NaN/+inf flag
    float zmx = -INFINITY, zmn = INFINITY;
    unsigned int bad = 0;
    auto stat1 = [&](float z) {
        zmx = fmaxf(zmx, z);
        zmn = fminf(zmn, z > -INFINITY ? z : INFINITY);
        bad |= (z < INFINITY) ? 0u : 1u;  // NaN or +inf
    };
    if (tid == 0) {
        sm->gcount = 0u;
        sm->lcount = 0u;
    }
    // the draw's uniform depends on the row's seed and offset alone: computed
    // here, off the critical path of the finish
    if (tid == kST - 1) sm->u53 = philox_word0(seed, offset) >> 11;
    if (smem_slice) {
        const bool aligned = ((reinterpret_cast<uintptr_t>(grow) & 15u) == 0);
        const int nbulk = aligned ? (n & ~3) : 0;
        const int cs = ((nbulk + 4 * kLoadChunks - 1) / (4 * kLoadChunks)) * 4;  // chunk length, multiple of 4
        if (tid == 0) {
            for (int k = 0; k < kLoadChunks; ++k) mbar_init(&sm->bar[k], 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (tid == 0) {
            for (int k = 0; k < kLoadChunks; ++k) {
                const int c0 = min(nbulk, k * cs), c1 = min(nbulk, c0 + cs);
                if (c1 > c0) {
                    mbar_arrive_expect_tx(&sm->bar[k], static_cast<uint32_t>(c1 - c0) * 4u);
                    tma_load_1d(zslice + c0, grow + c0, static_cast<uint32_t>(c1 - c0) * 4u, &sm->bar[k]);
                } else {
                    mbar_arrive(&sm->bar[k]);
                }
            }
        }
        for (int i = nbulk + tid; i < S; i += kST) zslice[i] = i < n ? grow[i] : -INFINITY;  // tail and padding
        for (int k = 0; k < kLoadChunks; ++k) {
            const int c0 = min(nbulk, k * cs), c1 = min(nbulk, c0 + cs);
            if (!mbar_wait(&sm->bar[k], 0)) report(status, PKV_ERR_TIMEOUT);
            for (int e = c0 + 4 * tid; e < c1; e += 4 * kST) {
                const float4 q = *reinterpret_cast<const float4*>(zslice + e);
                stat1(q.x);
                stat1(q.y);
                stat1(q.z);
                stat1(q.w);
            }
        }
        __syncthreads();  // tail written by every thread is visible
        for (int i = nbulk + tid; i < n; i += kST) stat1(zslice[i]);
    } else {
        sweep4<4>(v, nvec, false, [&](int, const float4& q) {
            stat1(q.x);
            stat1(q.y);
            stat1(q.z);
            stat1(q.w);
        });
    }
    const float tmax = zmx;  // this thread's own maximum
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        zmx = fmaxf(zmx, __shfl_xor_sync(0xffffffffu, zmx, o));
        zmn = fminf(zmn, __shfl_xor_sync(0xffffffffu, zmn, o));
        bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    {
        __shared__ float wz[kSW], wn[kSW];
        __shared__ unsigned int wb[kSW];
        __shared__ float lmax_sh, lmin_sh, xr_sh;
        __shared__ unsigned int h64[64];
        if (lane == 0) {
            wz[warp] = zmx;
            wn[warp] = zmn;
            wb[warp] = bad;
        }
        if (tid < 64) h64[tid] = 0u;
        __syncthreads();
        if (tid == 0) {
            float z = -INFINITY, zn = INFINITY;
            unsigned int b = 0;
            for (int w = 0; w < kSW; ++w) {
                z = fmaxf(z, wz[w]);
                zn = fminf(zn, wn[w]);
                b |= wb[w];
            }
            lmax_sh = z;
            lmin_sh = zn;
            xr_sh = -INFINITY;
            sm->xch[c.xb][0] = __float_as_uint(z);
            sm->xch[c.xb][1] = __float_as_uint(zn);
            sm->xch[c.xb][2] = b;
        }
        __syncthreads();
        // Local top-k bound: x_r such that at least top_k of this CTA's thread
        // maxima (hence top_k distinct logits) are >= x_r; then no member of the
        // row's top-k set lies below x_r.  Found on 64 bins over [min, max].
        if (kk_in > 0 && kk_in <= kST && T > 0.f) {
            const float lmax = lmax_sh, range = lmax_sh - lmin_sh;
            if (range > 0.f && range < INFINITY && tmax > -INFINITY) {
                const float t = (lmax - tmax) * (64.0f / range);
                atomicAdd(&h64[t >= 63.f ? 63 : static_cast<int>(t)], 1u);
            }
            __syncthreads();
            if (warp == 0 && range > 0.f && range < INFINITY) {
                const unsigned int two = h64[2 * lane] + h64[2 * lane + 1];
                unsigned int inc = two;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned int y = __shfl_up_sync(0xffffffffu, inc, o);
                    if (lane >= o) inc += y;
                }
                const unsigned int exl = inc - two;
                const unsigned int kq = static_cast<unsigned int>(kk_in);
                if (exl < kq && inc >= kq) {
                    const int b = exl + h64[2 * lane] >= kq ? 2 * lane : 2 * lane + 1;
                    xr_sh = lmax - (static_cast<float>(b) + 2.0f) * (range / 64.0f);  // one bin of margin
                }
            }
            __syncthreads();
            if (tid == 0) sm->xch[c.xb][3] = __float_as_uint(xr_sh);
        } else if (tid == 0) {
            sm->xch[c.xb][3] = __float_as_uint(-INFINITY);
        }
    }
    exch(c, 4);
    float zmax = -INFINITY, zmin = INFINITY, kbound = -INFINITY;
    unsigned int gbad = 0;
    for (int j = 0; j < c.nc; ++j) {
        zmax = fmaxf(zmax, __uint_as_float(static_cast<uint32_t>(sm->gath[j][0])));
        zmin = fminf(zmin, __uint_as_float(static_cast<uint32_t>(sm->gath[j][1])));
        gbad |= static_cast<unsigned int>(sm->gath[j][2]);
        kbound = fmaxf(kbound, __uint_as_float(static_cast<uint32_t>(sm->gath[j][3])));
    }
    int err = 0;
    if (gbad || !(zmax > -INFINITY)) err = PKV_ERR_NONFINITE;  // NaN / +inf, or no finite logit
    else if (!(T >= 0.f)) err = PKV_ERR_INVALID_ARG;
    else if (T != 0.f && !(pp > 0.f)) err = PKV_ERR_INVALID_ARG;
    else if (T != 0.f && (mp != mp || mp > 1.f)) err = PKV_ERR_INVALID_ARG;  // min_p NaN or > 1
    if (err) {
        if (c.rank == 0 && tid == 0) {
            *tok_out = -1;
            report(status, err);
        }
        cluster.sync();  // no CTA leaves while a peer may still read its shared memory
        return;
    }
    if (T == 0.f) {
        // greedy: the lowest id holding the maximum
        int amin = INT_MAX;
        for (int e = 4 * tid; e < nvec; e += 4 * kST) {
            const float4 q = load4(v, e, vec);
            if (q.w == zmax) amin = lo + e + 3;
            if (q.z == zmax) amin = lo + e + 2;
            if (q.y == zmax) amin = lo + e + 1;
            if (q.x == zmax) amin = lo + e;
            if (amin != INT_MAX) break;  // later slots of this thread hold larger ids
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amin = min(amin, __shfl_xor_sync(0xffffffffu, amin, o));
        if (tid == 0) sm->imin = INT_MAX;
        __syncthreads();
        if (lane == 0 && amin != INT_MAX) atomicMin(&sm->imin, amin);
        __syncthreads();
        if (tid == 0) sm->xch[c.xb][0] = static_cast<uint32_t>(sm->imin);
        exch(c, 1);
        if (c.rank == 0 && tid == 0) {
            int a = INT_MAX;
            for (int j = 0; j < c.nc; ++j) a = min(a, static_cast<int>(static_cast<uint32_t>(sm->gath[j][0])));
            *tok_out = a;
        }
        cluster.sync();
        return;
    }

    const float c2 = fminf(1.4426950408889634f / T, 1.0e30f);  // log2(e) / T, kept finite
    Keep kp;
    kp.k_on = false;
    kp.p_on = false;
    kp.mth = mp > 0.f ? ceil_mul_p(mp, 1ull << 40) : 0ull;  // min-p: mass >= ceil(min_p * 2^40)
    kp.tauk = kp.taup = 0u;
    kp.idk = kp.idp = INT_MAX;
    kp.zk = kp.zp = 0.f;
    Bins bins;
    bins.zmax = zmax;
    bins.nb = kHistBins;
    {
        const float range = zmax - zmin;
        const float sc = static_cast<float>(kHistBins) / range;
        bins.scale = (range > 0.f && sc < INFINITY) ? sc : 0.f;
    }
    unsigned int* cnt = reinterpret_cast<unsigned int*>(sm->hist);
    unsigned int* gcount0 = cluster.map_shared_rank(&sm->gcount, 0);
    unsigned long long* list0 = cluster.map_shared_rank(&sm->list[0], 0);
    int kk = 0;  // effective top-k (0: off); set once the finite count is known

    if (kk_in > 0) {
        // ---------------- top-k: count histogram over [kbound, zmax] (every top-k
        // member is >= kbound), candidate bin, gather, finish on rank 0
        const bool bounded = kbound > -INFINITY;
        Bins kb = bins;
        if (bounded) {
            kb.nb = kTopkBins;
            const float range = zmax - kbound;
            const float sc = static_cast<float>(kTopkBins) / range;
            kb.scale = (range > 0.f && sc < INFINITY) ? sc : 0.f;
        }
        const float zfloor = bounded ? kbound : -INFINITY;
        if (!vec && bounded && kk_in <= kRegTopk) {
            // Slice in global memory and a small k: the histogram is taken over
            // the first pass's thread maxima (distinct logits, held in
            // registers), so the slice is not read a second time.  Bin bk is
            // where the maxima >= kbound first number k: the k-th largest
            // maximum lies in bins 0..bk, hence so does every top-k member (each
            // is >= it).  A member is its thread's maximum or belongs to a thread
            // whose maximum is larger, so only the threads whose maximum is in
            // bins 0..bk read their logits again and push those in bins 0..bk.
            for (int i = tid; i < kb.nb; i += kST) cnt[i] = 0u;
            if (tid == 0) {
                sm->bc[0] = kb.nb - 1;
                sm->bc[1] = 0;
            }
            __syncthreads();
            if (tmax >= zfloor) atomicAdd(&cnt[kb(tmax)], 1u);
            cluster.sync();
            uint32_t g[4] = {0u, 0u, 0u, 0u};
            if (tid * 4 < kb.nb) sum_remote_u4(cluster, cnt, c.nc, g);
            const uint64_t tsum = static_cast<uint64_t>(g[0]) + g[1] + g[2] + g[3];
            uint64_t counted;
            const uint64_t ex = block_excl_scan_u64(tsum, sm->wsum, counted);
            kk = kk_in;
            if (ex < static_cast<uint64_t>(kk) && ex + tsum >= static_cast<uint64_t>(kk)) {
                uint64_t cc = ex;
                for (int q = 0; q < 4; ++q) {
                    cc += g[q];
                    if (cc >= static_cast<uint64_t>(kk)) {
                        sm->bc[0] = static_cast<unsigned long long>(tid * 4 + q);
                        sm->bc[1] = cc;
                        break;
                    }
                }
            }
            __syncthreads();
            const int bk = static_cast<int>(sm->bc[0]);
            const bool reached = sm->bc[1] >= static_cast<unsigned long long>(kk);  // same in every CTA
            if (reached) {
                // the qualifying threads' slots 4 (t + kST m) are spread over the
                // whole CTA, one 16-byte load per thread, so the rescans cost one
                // round trip to L2 instead of one per qualifying lane of a warp
                int* qlist = reinterpret_cast<int*>(sm->hist + kLocBase);
                if (tmax >= zfloor && kb(tmax) <= bk) qlist[atomicAdd(&sm->lcount, 1u)] = tid;
                __syncthreads();
                const int nq = static_cast<int>(sm->lcount);
                const int spt = (nvec + 4 * kST - 1) / (4 * kST);  // slots per thread
                for (int i0 = tid - lane; i0 < nq * spt; i0 += kST) {  // warp-uniform trip count
                    const int i = i0 + lane;
                    int el = 0;
                    float4 q = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                    if (i < nq * spt) {
                        const int qi = i / spt;
                        el = 4 * (qlist[qi] + kST * (i - qi * spt));
                        if (el < nvec) q = load4(v, el, false);
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float z = f4at(q, j);
                        const bool pred = z > -INFINITY && z >= zfloor && kb(z) <= bk;
                        gather_push(pred, pred ? sort_key(z, lo + el + j) : 0ull, gcount0, list0);
                    }
                }
            }
            cluster.sync();  // candidates complete in rank 0; its bins are no longer read
            const unsigned int ng = *gcount0;
            cluster_arrive();  // rank 0 stays until every CTA has read its count
            if (reached && ng <= static_cast<unsigned int>(kListCap)) {
                if (c.rank == 0) solo_finish(sm, static_cast<int>(ng), kk, pp, kp.mth, zmax, c2, tok_out);
                cluster_wait();
                return;
            }
            cluster_wait();
            fallback_select_and_draw(c, v, kp, vec, kk, pp, zmax, c2, tok_out);
            cluster_wait();
            return;
        }
        for (int i = tid; i < kb.nb; i += kST) cnt[i] = 0u;
        if (tid == 0) {
            sm->bc[0] = kb.nb - 1;
            sm->bc[1] = 0;
        }
        __syncthreads();
        // bounded: the counted logits (usually a few hundred) are also kept as
        // sort keys in this CTA's candidate list, so the gather below need not
        // read the slice again
        unsigned long long* loc = sm->hist + kLocBase;
        sweep4<4>(v, nvec, vec, [&](int el, const float4& q) {
            const bool any = q.x >= zfloor || q.y >= zfloor || q.z >= zfloor || q.w >= zfloor;
            if (!__any_sync(0xffffffffu, any)) return;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float z = f4at(q, j);
                const bool pred = z > -INFINITY && z >= zfloor;
                if (pred) atomicAdd(&cnt[kb(z)], 1u);
                if (bounded) gather_push(pred, pred ? sort_key(z, lo + el + j) : 0ull, &sm->lcount, loc, kLocCap);
            }
        });
        cluster.sync();
        uint32_t g[4] = {0u, 0u, 0u, 0u};
        if (tid * 4 < kb.nb) sum_remote_u4(cluster, cnt, c.nc, g);
        const uint64_t tsum = static_cast<uint64_t>(g[0]) + g[1] + g[2] + g[3];
        uint64_t counted;  // unbounded: every finite logit; bounded: those >= kbound (>= top_k of them)
        const uint64_t ex = block_excl_scan_u64(tsum, sm->wsum, counted);
        if (bounded || static_cast<uint64_t>(kk_in) < counted) {
            kk = kk_in;
            if (ex < static_cast<uint64_t>(kk) && ex + tsum >= static_cast<uint64_t>(kk)) {
                uint64_t cc = ex;
                for (int q = 0; q < 4; ++q) {
                    cc += g[q];
                    if (cc >= static_cast<uint64_t>(kk)) {
                        sm->bc[0] = static_cast<unsigned long long>(tid * 4 + q);
                        sm->bc[1] = cc;  // candidates: every counted logit in bins 0..bk
                        break;
                    }
                }
            }
            __syncthreads();
            const int bk = static_cast<int>(sm->bc[0]);
            const uint64_t total = sm->bc[1];
            if (total >= static_cast<uint64_t>(kk) && total <= static_cast<uint64_t>(kListCap)) {
                // every candidate has z >= zlow (two bins of margin for rounding)
                const float zlow =
                    kb.scale > 0.f ? fmaxf(zfloor, zmax - (static_cast<float>(bk) + 3.0f) / kb.scale) : zfloor;
                const int lc = static_cast<int>(sm->lcount);  // read after the cluster barrier above
                if (bounded && lc <= kLocCap) {
                    const unsigned long long* loc = sm->hist + kLocBase;
                    for (int i = tid - lane; i < lc; i += kST) {  // warp-uniform trip count
                        const int j = i + lane;
                        const unsigned long long key = j < lc ? loc[j] : 0ull;
                        const float z = key_float(static_cast<uint32_t>(key >> 32));
                        const bool pred = j < lc && kb(z) <= bk;
                        gather_push(pred, key, gcount0, list0);
                    }
                } else {
                    sweep4<4>(v, nvec, vec, [&](int el, const float4& q) {
                        const bool any = q.x >= zlow || q.y >= zlow || q.z >= zlow || q.w >= zlow;
                        if (!__any_sync(0xffffffffu, any)) return;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float z = f4at(q, j);
                            const bool pred = z > -INFINITY && z >= zfloor && kb(z) <= bk;
                            gather_push(pred, pred ? sort_key(z, lo + el + j) : 0ull, gcount0, list0);
                        }
                    });
                }
                cluster.sync();  // candidates complete in rank 0; no remote access follows
                if (c.rank != 0) return;
                solo_finish(sm, static_cast<int>(total), kk, pp, kp.mth, zmax, c2, tok_out);
                return;
            }
            cluster.sync();  // remote histogram reads are done before the fallback reuses it
            fallback_select_and_draw(c, v, kp, vec, kk, pp, zmax, c2, tok_out);
            cluster_wait();
            return;
        }
        cluster.sync();  // top_k >= finite count: top-k is off; the histogram is reused below
    }

    if (pp < 1.f) {
        // ---------------- top-p only.  On the 2048 linear bins of (zmax - z), each
        // bin gets its count and the sums of the high (>> 16) and low (mod 2^16)
        // parts of its logits' masses floor(w * 2^40), with u32 shared atomics.
        // Where the sums cannot have wrapped (count * an upper bound of the high
        // part < 2^32, count < 2^16) they give the bin's exact mass; other bins
        // are bounded by count times the weights at the bin's edges (1/64 bin of
        // margin for the rounding of the bin index, 2^-20 relative for the
        // approximate exponential).  The bounds bracket S and every cumulative
        // from the top, so the cut lies in the bins [blo, bhi] where they
        // straddle ceil(p * S); when every bin is exact that is one bin, and the
        // exact mass above it is already known.  A second pass gathers the
        // window into rank 0 (summing exact masses above and below it when some
        // bin was inexact), which sorts it and finds the cut exactly.
        constexpr int kPer = kHistBins / kST;  // 4 bins per thread
        unsigned int* pc = reinterpret_cast<unsigned int*>(sm->hist);   // counts
        unsigned int* ph = pc + kHistBins;                                // sums of mass >> 16
        unsigned int* pl = reinterpret_cast<unsigned int*>(sm->list);   // sums of mass & 0xffff
        for (int i = tid; i < kHistBins; i += kST) {
            pc[i] = 0u;
            ph[i] = 0u;
            pl[i] = 0u;
        }
        if (tid == 0) {
            sm->bc[2] = 0;
            sm->bc[3] = kHistBins - 1;
            sm->bc[7] = 0;
        }
        __syncthreads();
        sweep4<4>(v, nvec, vec, [&](int, const float4& q) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float z = f4at(q, j);
                if (z > -INFINITY) {
                    const int b = bins(z);
                    const uint64_t m = mass(z, zmax, c2);
                    atomicAdd(&pc[b], 1u);
                    atomicAdd(&ph[b], static_cast<unsigned int>(m >> 16));
                    atomicAdd(&pl[b], static_cast<unsigned int>(m & 0xffffu));
                }
            }
        });
        cluster.sync();  // every CTA's bins are complete
        // this thread's bins [4*tid, 4*tid + 4), summed over the cluster
        uint32_t gc[kPer] = {0u, 0u, 0u, 0u}, gh[kPer] = {0u, 0u, 0u, 0u}, gl[kPer] = {0u, 0u, 0u, 0u};
        for (int r = 0; r < c.nc; ++r) {
            const uint4 cc = reinterpret_cast<const uint4*>(cluster.map_shared_rank(pc, r))[tid];
            const uint4 hh = reinterpret_cast<const uint4*>(cluster.map_shared_rank(ph, r))[tid];
            const uint4 ll = reinterpret_cast<const uint4*>(cluster.map_shared_rank(pl, r))[tid];
            gc[0] += cc.x; gc[1] += cc.y; gc[2] += cc.z; gc[3] += cc.w;
            gh[0] += hh.x; gh[1] += hh.y; gh[2] += hh.z; gh[3] += hh.w;
            gl[0] += ll.x; gl[1] += ll.y; gl[2] += ll.z; gl[3] += ll.w;
        }
        cluster_arrive();  // remote reads of the bins are done (waited on before reuse)
        auto bin_bounds = [&](int q, uint64_t& mh, uint64_t& ml) {
            const uint64_t n = gc[q];
            mh = ml = 0;
            if (n == 0) return;
            const int bq = kPer * tid + q;
            // weights at the bin's edges: bin b holds (zmax - (b+1)/s, zmax - b/s]
            const float dh = bins.scale > 0.f ? (static_cast<float>(bq) - 0.015625f) / bins.scale : 0.f;
            const float dl = bins.scale > 0.f ? (static_cast<float>(bq + 1) + 0.015625f) / bins.scale : zmax - zmin;
            uint64_t hi = fx40(hw_exp2(fminf(-dh * c2, 0.f)));
            hi += (hi >> 20) + 1;
            if (n < 65536u && n * ((hi >> 16) + 1) < (1ull << 32)) {
                ml = mh = (static_cast<uint64_t>(gh[q]) << 16) + gl[q];  // the sums did not wrap: exact
                return;
            }
            uint64_t lo = fx40(hw_exp2(-dl * c2));
            lo = lo > (lo >> 20) + 1 ? lo - (lo >> 20) - 1 : 0ull;
            mh = n * hi;
            ml = n * lo;
        };
        uint64_t tlo = 0, thi = 0;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            uint64_t mh, ml;
            bin_bounds(q, mh, ml);
            thi += mh;
            tlo += ml;
        }
        uint64_t Shi, Slo;
        const uint64_t exh = block_excl_scan_u64(thi, sm->wsum, Shi);
        const uint64_t exl = block_excl_scan_u64(tlo, sm->wsum, Slo);
        const uint64_t tgt_lo = ceil_mul_p(pp, Slo), tgt_hi = ceil_mul_p(pp, Shi);
        {
            uint64_t ch = exh, cl = exl;
#pragma unroll
            for (int q = 0; q < kPer; ++q) {
                const int bq = kPer * tid + q;
                uint64_t mh, ml;
                bin_bounds(q, mh, ml);
                const uint64_t nh = ch + mh, nl = cl + ml;
                if (nh >= tgt_lo && (bq == 0 || ch < tgt_lo)) {
                    sm->bc[2] = static_cast<unsigned long long>(bq);
                    sm->bc[7] = ch;  // mass above bin blo (exact when every bin is)
                }
                if (nl >= tgt_hi && (bq == 0 || cl < tgt_hi)) sm->bc[3] = static_cast<unsigned long long>(bq);
                ch = nh;
                cl = nl;
            }
        }
        __syncthreads();
        const int blo = static_cast<int>(sm->bc[2]);
        const int bhi = max(blo, static_cast<int>(sm->bc[3]));
        const bool exact = Shi == Slo;  // every bin's mass is known exactly
        const uint64_t A_known = sm->bc[7];
        uint64_t wc = 0;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int bq = kPer * tid + q;
            if (bq >= blo && bq <= bhi) wc += gc[q];
        }
        uint64_t total;
        block_excl_scan_u64(wc, sm->wsum, total);
        cluster_wait();  // no CTA still reads another's counts
        if (total >= 1 && total <= static_cast<uint64_t>(kListCap)) {
            uint64_t at = 0, bt = 0;  // exact masses above and below the window
            if (exact) {
                // blo <= bin <= bhi as comparisons with the bins' edges (-inf
                // lies below both)
                __shared__ float edge_sh[2];
                if (tid < 2) edge_sh[tid] = bin_edge(bins, tid == 0 ? blo : bhi + 1);
                __syncthreads();
                const float e_in = edge_sh[0], e_out = edge_sh[1];
                sweep4<4>(v, nvec, vec, [&](int el, const float4& q) {
                    bool in[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float z = f4at(q, j);
                        in[j] = z < e_in && z >= e_out;
                    }
                    if (!__any_sync(0xffffffffu, in[0] || in[1] || in[2] || in[3])) return;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        gather_push(in[j], in[j] ? sort_key(f4at(q, j), lo + el + j) : 0ull, gcount0, list0);
                });
            } else {
                sweep4<4>(v, nvec, vec, [&](int el, const float4& q) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float z = f4at(q, j);
                        const bool fin = z > -INFINITY;
                        const int b = fin ? bins(z) : kHistBins;
                        if (fin && (b < blo || b > bhi)) {
                            const uint64_t m = mass(z, zmax, c2);
                            if (b < blo) at += m; else bt += m;
                        }
                        const bool pred = fin && b >= blo && b <= bhi;
                        gather_push(pred, pred ? sort_key(z, lo + el + j) : 0ull, gcount0, list0);
                    }
                });
            }
            uint64_t acta, bcta;
            block_excl_scan_u64(at, sm->wsum, acta);
            block_excl_scan_u64(bt, sm->wsum, bcta);
            if (tid == 0) {
                *cluster.map_shared_rank(&sm->aslot[c.rank], 0) = acta;
                *cluster.map_shared_rank(&sm->bslot[c.rank], 0) = bcta;
            }
            cluster.sync();  // window gathered and exact masses around it posted in rank 0
            if (c.rank == 0) {
                uint64_t A = 0, Bm = 0;
                for (int r = 0; r < c.nc; ++r) {
                    A += sm->aslot[r];
                    Bm += sm->bslot[r];
                }
                if (exact) A = A_known;  // and Bm stays 0: S is known
                unsigned long long* a = sm->list;
                const int nw = static_cast<int>(total);
                const int np2 = pow2_ceil(nw);
                for (int i = nw + tid; i < np2; i += kST) a[i] = 0ull;
                if (tid == 0) {
                    sm->bc[4] = 0ull;  // ok flag
                    sm->bc[5] = 0ull;
                    sm->bc[6] = 0ull;
                }
                __syncthreads();
                bitonic_sort(a, np2, true);
                const int E = run_len(nw);
                const int b0 = min(nw, tid * E), b1 = min(nw, b0 + E);
                uint64_t w = 0;
                for (int j = b0; j < b1; ++j) w += mass(key_float(static_cast<uint32_t>(a[j] >> 32)), zmax, c2);
                uint64_t wtot;
                const uint64_t wex = block_excl_scan_u64(w, sm->wsum, wtot);
                const uint64_t target = ceil_mul_p(pp, exact ? Shi : A + wtot + Bm);  // exact S
                if (A < target && A + wtot >= target && A + wex < target && A + wex + w >= target) {
                    uint64_t cum = A + wex;
                    for (int j = b0; j < b1; ++j) {
                        cum += mass(key_float(static_cast<uint32_t>(a[j] >> 32)), zmax, c2);
                        if (cum >= target) {
                            sm->bc[4] = 1ull;
                            sm->bc[5] = a[j] >> 32;
                            sm->bc[6] = static_cast<unsigned long long>(static_cast<uint32_t>(sort_key_id(a[j])));
                            break;
                        }
                    }
                }
                __syncthreads();
                if (tid < c.nc) {
                    unsigned long long* rb = cluster.map_shared_rank(&sm->bc[0], tid);
                    rb[4] = sm->bc[4];
                    rb[5] = sm->bc[5];
                    rb[6] = sm->bc[6];
                }
            }
            cluster.sync();  // cut broadcast to every rank
            if (sm->bc[4]) {
                kp.p_on = true;
                kp.taup = static_cast<uint32_t>(sm->bc[5]);
                kp.zp = key_float(kp.taup);
                kp.idp = static_cast<int>(static_cast<uint32_t>(sm->bc[6]));
                draw_pass(c, v, kp, vec, zmax, c2, tok_out);
                cluster_wait();
                return;
            }
        }
        fallback_select_and_draw(c, v, kp, vec, 0, pp, zmax, c2, tok_out);
        cluster_wait();
        return;
    }

    // ---------------- no filter: draw over every finite logit
    draw_pass(c, v, kp, vec, zmax, c2, tok_out);
    cluster_wait();
}

// ------------------------------------------------------------------ host side
// Launch plan: nc CTAs (one cluster) per row, each over a slice of S logits
// (a multiple of 4), kept in shared memory when smem_slice.
//
// A row's work is a short chain of dependent phases (load, bounds, histogram,
// gather, finish), so the kernel is fastest when every row's cluster is
// resident at once.  With the slice in shared memory (at most 24576 logits per
// CTA, so nc = ceil(V / 20480)) a CTA holds up to ~130 KB; once B rows of such
// clusters no longer fit on the GPU together, the slice is read from global
// memory instead (the first read streams it from HBM, later passes hit L2),
// with as many CTAs per row as still lets all B clusters be resident.
struct SamplerPlan {
    int nc, S, smem_slice;
    size_t smem;
};

static SamplerPlan make_plan(int V, int nc, bool smem_slice) {
    SamplerPlan p;
    int S = (V + nc - 1) / nc;
    S = (S + 3) & ~3;
    p.nc = nc;
    p.S = S;
    p.smem_slice = smem_slice ? 1 : 0;
    p.smem = sizeof(SampSmem) + (smem_slice ? static_cast<size_t>(S) * 4 : 0);  // S is a multiple of 4
    return p;
}

// Clusters of plan p that can be resident at once on the current device (0 on error).
static int resident_clusters(const SamplerPlan& p) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, size_t>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const auto key = std::make_tuple(dev, p.nc, p.smem);
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    if (cudaFuncSetAttribute(sampler_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(p.smem)) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.nc) * 64u, 1, 1);
    cfg.blockDim = dim3(kST, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.nc;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sampler_kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = n;
    return n;
}

static SamplerPlan plan_sampler(int B, int V, int sms) {
    int nc_s = (V + 20479) / 20480;
    nc_s = nc_s < 1 ? 1 : (nc_s > kMaxCluster ? kMaxCluster : nc_s);
    const SamplerPlan ps = make_plan(V, nc_s, true);
    const bool smem_ok = ps.S <= kSliceSmemMax;
    if (smem_ok && B <= resident_clusters(ps)) return ps;
    for (int nc = kMaxCluster; nc >= 1; --nc) {
        if (nc > 1 && (V + nc - 1) / nc < 4096) continue;  // keep slices long enough to be worth a CTA
        const SamplerPlan pg = make_plan(V, nc, false);
        if (B <= resident_clusters(pg)) {
            // one CTA per row in one wave with more rows than SMs: clusters of
            // the largest size (2, 3 or 4) whose CTAs fit two waves, heaviest
            // rows first.  Mixed 152064-logit batches of 170 / 200 / 256 / 300
            // rows: 106 / 111 / 132 / 152 us against 174 / 180 / 186 / 200;
            // batches of one kind move by -12% to +17%.
            if (nc == 1 && B > sms) {
                int nc2 = min(4, (2 * resident_clusters(pg)) / B);
                while (nc2 > 1 && (V + nc2 - 1) / nc2 < 4096) --nc2;
                if (nc2 >= 2) return make_plan(V, nc2, false);
            }
            return pg;
        }
    }
    return make_plan(V, 1, false);  // more rows than resident CTAs: one CTA per row, in waves
}

int device_sm_count();
bool sampler_rows_fits(int B, int V, int sms);
cudaError_t launch_sampler_rows(int32_t* tokens, const float* logits, int B, int V, const float* temperature,
                                const int32_t* top_k, const float* top_p, const float* min_p,
                                const uint64_t* seeds, const uint64_t* offsets, int32_t* status,
                                cudaStream_t stream);

cudaError_t launch_sampler(int32_t* tokens, const float* logits, int B, int V, const float* temperature,
                           const int32_t* top_k, const float* top_p, const float* min_p, const uint64_t* seeds,
                           const uint64_t* offsets, int32_t* status, cudaStream_t stream) {
    // more rows of a moderate vocabulary than this kernel keeps resident: one
    // 256-thread CTA per row (sampler_rows.cu), every row at once
    const int sms = device_sm_count();
    if (sampler_rows_fits(B, V, sms))
        return launch_sampler_rows(tokens, logits, B, V, temperature, top_k, top_p, min_p, seeds, offsets, status,
                                   stream);
    const SamplerPlan sp = plan_sampler(B, V, sms);
    // more rows than SMs: heaviest rows first
    const int lpt_B = (B > sms && B < (1 << 21)) ? B : 0;
    cudaError_t err = cudaFuncSetAttribute(sampler_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(sp.smem));
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B) * sp.nc, 1, 1);
    cfg.blockDim = dim3(kST, 1, 1);
    cfg.dynamicSmemBytes = sp.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = sp.nc;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, sampler_kernel, tokens, logits, V, sp.S, sp.smem_slice, temperature, top_k,
                              top_p, min_p, seeds, offsets, status, lpt_B);
}

}  // namespace pkv
