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
// every later pass runs on chip.  Selections are radix searches over 32-bit
// order-preserving keys (digits of 11/11/10 bits) whose per-CTA histograms are
// summed through distributed shared memory.  Masses are exp() in fp32 turned
// into 64-bit fixed point (floor(w * 2^40)), so every sum, cut and CDF
// comparison afterwards is exact integer arithmetic and run-to-run deterministic.
// When top-k leaves few candidates, the cluster gathers them into rank 0, which
// finishes alone without further cluster barriers.
#include <cooperative_groups.h>
#include <limits.h>
#include <math.h>

#include "pkv_common.cuh"

namespace cg = cooperative_groups;

namespace pkv {

constexpr int kST = 512;           // threads per CTA
constexpr int kSW = kST / 32;      // warps per CTA
constexpr int kHistBins = 2048;    // widest radix digit (11 bits)
constexpr int kListCap = 2048;     // candidate list capacity (rank 0, gathered)
constexpr int kMaxCluster = 8;
constexpr int kSliceSmemMax = 24576;  // floats of a row slice kept in shared memory

struct SampSmem {
    unsigned long long hist[kHistBins];
    unsigned long long xch[2][4];
    unsigned long long gath[kMaxCluster][4];
    unsigned long long wsum[kSW];
    unsigned long long bc[4];
    float list_z[kListCap];
    int list_id[kListCap];
    uint64_t bar;
    int imin;
};

// ------------------------------------------------------------------ numeric helpers
// Order-preserving key of a float (larger float -> larger key); -0.0 is folded
// onto +0.0 so that equal logits have equal keys.
__device__ __forceinline__ uint32_t okey(float z) {
    uint32_t u = __float_as_uint(z);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
    const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}
// floor(w * 2^40) for w in [0, 1], exactly, from the float's bits.
__device__ __forceinline__ uint64_t fx40(float w) {
    const uint32_t u = __float_as_uint(w);
    const int e = static_cast<int>((u >> 23) & 0xffu);
    if (e == 0 || e > 127) return 0ull;  // zero / denormal (or outside [0, 1], which cannot occur)
    const uint64_t m = static_cast<uint64_t>((u & 0x7fffffu) | 0x800000u);
    const int sh = e - 110;  // w * 2^40 = m * 2^(e - 110)
    if (sh >= 0) return m << sh;
    if (sh <= -24) return 0ull;
    return m >> (-sh);
}
// Fixed-point mass of a finite logit; the maximum itself weighs exactly 2^40
// (also when 1/T overflows and 0 * inf would be NaN).
__device__ __forceinline__ uint64_t mass(float z, float zmax, float invT) {
    const float d = z - zmax;
    if (d == 0.f) return 1ull << 40;
    return fx40(expf(d * invT));
}
// ceil(p * S) for p a float in (0, 1) and S < 2^63, exactly.
__device__ __forceinline__ uint64_t ceil_mul_p(float p, uint64_t S) {
    const uint32_t u = __float_as_uint(p);
    const int e = static_cast<int>((u >> 23) & 0xffu);
    const uint64_t m = e ? static_cast<uint64_t>((u & 0x7fffffu) | 0x800000u) : static_cast<uint64_t>(u & 0x7fffffu);
    const int sh = e ? 150 - e : 149;  // p = m * 2^-sh
    const unsigned __int128 N = static_cast<unsigned __int128>(m) * S;
    if (N == 0) return 0ull;
    if (sh >= 127) return 1ull;
    const unsigned __int128 one = 1;
    return static_cast<uint64_t>((N + ((one << sh) - 1)) >> sh);
}

// Philox4x64-10 (Salmon et al., SC'11), word 0 only.
__device__ __forceinline__ uint64_t philox_word0(uint64_t seed, uint64_t offset) {
    uint64_t x0 = offset, x1 = 0, x2 = 0, x3 = 0;
    uint64_t k0 = seed, k1 = 0;
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        const uint64_t lo0 = 0xD2E7470EE14C6C93ull * x0, hi0 = __umul64hi(0xD2E7470EE14C6C93ull, x0);
        const uint64_t lo1 = 0xCA5A826395121157ull * x2, hi1 = __umul64hi(0xCA5A826395121157ull, x2);
        const uint64_t y0 = hi1 ^ x1 ^ k0, y2 = hi0 ^ x3 ^ k1;
        x0 = y0;
        x1 = lo1;
        x2 = y2;
        x3 = lo0;
        k0 += 0x9E3779B97F4A7C15ull;
        k1 += 0xBB67AE8584CAA73Bull;
    }
    return x0;
}

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
    __device__ __forceinline__ int idat(int i) const { return id ? id[i] : idbase + i; }
};

struct Keep {
    bool k_on, p_on;
    uint32_t tauk, taup;
    int idk, idp;
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
    bool solo;  // true once rank 0 owns every candidate and runs alone
    __device__ __forceinline__ int nce() const { return solo ? 1 : nc; }
    __device__ __forceinline__ int rke() const { return solo ? 0 : rank; }
    __device__ __forceinline__ void csync() const {
        if (solo) __syncthreads();
        else cg::this_cluster().sync();
    }
    template <typename T>
    __device__ __forceinline__ T* remote(T* p, int r) const {
        return solo ? p : cg::this_cluster().map_shared_rank(p, r);
    }
};

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
                           float zmax, float invT, bool p_first, float top_p, uint64_t* S_out) {
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
        const uint64_t w = kMass ? mass(z, zmax, invT) : 1ull;
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

// ------------------------------------------------------------------ kernel
__global__ void __launch_bounds__(kST, 2)
    sampler_kernel(int32_t* __restrict__ tokens, const float* __restrict__ logits, int V, int S, int smem_slice,
                   const float* __restrict__ temperature, const int32_t* __restrict__ top_k,
                   const float* __restrict__ top_p, const uint64_t* __restrict__ seeds,
                   const uint64_t* __restrict__ offsets, int32_t* status) {
    extern __shared__ __align__(16) uint8_t samp_smem_raw[];
    SampSmem* sm = reinterpret_cast<SampSmem*>(samp_smem_raw);
    float* zslice = reinterpret_cast<float*>(samp_smem_raw + sizeof(SampSmem));
    cg::cluster_group cluster = cg::this_cluster();
    Ctx c;
    c.sm = sm;
    c.nc = static_cast<int>(cluster.num_blocks());
    c.rank = static_cast<int>(cluster.block_rank());
    c.xb = 0;
    c.solo = false;
    const int tid = threadIdx.x;
    const int row = blockIdx.x / c.nc;
    const int lo = c.rank * S;
    const int n = max(0, min(S, V - lo));
    const float* grow = logits + static_cast<size_t>(row) * V + lo;

    // ---- load this CTA's slice (bulk copy when 16-byte aligned)
    View v;
    v.id = nullptr;
    v.n = n;
    v.idbase = lo;
    if (smem_slice) {
        const bool aligned = ((reinterpret_cast<uintptr_t>(grow) & 15u) == 0);
        const int nbulk = aligned ? (n & ~3) : 0;
        if (tid == 0) {
            mbar_init(&sm->bar, 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (tid == 0) {
            if (nbulk > 0) {
                mbar_arrive_expect_tx(&sm->bar, static_cast<uint32_t>(nbulk) * 4u);
                tma_load_1d(zslice, grow, static_cast<uint32_t>(nbulk) * 4u, &sm->bar);
            } else {
                mbar_arrive(&sm->bar);
            }
        }
        for (int i = nbulk + tid; i < n; i += kST) zslice[i] = grow[i];
        if (!mbar_wait(&sm->bar, 0)) report(status, PKV_ERR_TIMEOUT);
        __syncthreads();
        v.z = zslice;
    } else {
        v.z = grow;
    }

    // ---- pass 1: max / argmax / finite count / non-finite flag
    uint64_t best = 0ull, nfin = 0ull, bad = 0ull;
    for (int i = tid; i < n; i += kST) {
        const float z = v.z[i];
        if (isfinite(z)) {
            ++nfin;
            const uint64_t pk = (static_cast<uint64_t>(okey(z)) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(lo + i));
            best = pk > best ? pk : best;
        } else if (!(z < 0.f)) {
            bad = 1ull;  // NaN or +inf
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t b2 = __shfl_xor_sync(0xffffffffu, best, o);
        best = b2 > best ? b2 : best;
        nfin += __shfl_xor_sync(0xffffffffu, nfin, o);
        bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    {
        __shared__ unsigned long long wb[kSW][3];
        if ((tid & 31) == 0) {
            wb[tid >> 5][0] = best;
            wb[tid >> 5][1] = nfin;
            wb[tid >> 5][2] = bad;
        }
        __syncthreads();
        if (tid == 0) {
            uint64_t b = 0, f = 0, x = 0;
            for (int w = 0; w < kSW; ++w) {
                b = wb[w][0] > b ? wb[w][0] : b;
                f += wb[w][1];
                x |= wb[w][2];
            }
            sm->xch[c.xb][0] = b;
            sm->xch[c.xb][1] = f;
            sm->xch[c.xb][2] = x;
        }
    }
    exch(c, 3);
    uint64_t gbest = 0, gfin = 0, gbad = 0;
    for (int j = 0; j < c.nc; ++j) {
        gbest = sm->gath[j][0] > gbest ? sm->gath[j][0] : gbest;
        gfin += sm->gath[j][1];
        gbad |= sm->gath[j][2];
    }
    const float T = temperature[row];
    const float pp = top_p[row];
    const int kk_in = top_k[row];
    int token = -1;
    int err = 0;
    if (gbad || gfin == 0) err = PKV_ERR_NONFINITE;
    else if (!(T >= 0.f)) err = PKV_ERR_INVALID_ARG;
    else if (T == 0.f) token = static_cast<int>(~static_cast<uint32_t>(gbest & 0xffffffffull));
    else if (!(pp > 0.f)) err = PKV_ERR_INVALID_ARG;
    if (err || token >= 0) {
        if (c.rank == 0 && tid == 0) {
            tokens[row] = err ? -1 : token;
            if (err) report(status, err);
        }
        cluster.sync();  // no CTA leaves while a peer may still read its shared memory
        return;
    }

    const float zmax = key_float(static_cast<uint32_t>(gbest >> 32));
    const float invT = 1.0f / T;
    const int kk = (kk_in > 0 && static_cast<uint64_t>(kk_in) < gfin) ? kk_in : 0;
    Keep kp;
    kp.k_on = kk > 0;
    kp.p_on = pp < 1.0f;
    kp.tauk = kp.taup = 0u;
    kp.idk = kp.idp = INT_MAX;

    // ---- top-k: three count passes (11/11/10 bits), candidate gather after the first
    if (kp.k_on) {
        uint64_t target = static_cast<uint64_t>(kk), above = 0, binw = 0;
        uint32_t d0, d1, d2;
        radix_pass<false>(c, v, kp, false, 0u, 0, 21, 11, target, above, d0, binw, zmax, invT, false, 0.f, nullptr);
        // Candidates: finite keys whose top digit is >= d0 (a superset of the top-k set).
        {
            const int E = run_len(v.n);
            const int b0 = min(v.n, tid * E), b1 = min(v.n, b0 + E);
            uint64_t cnt = 0;
            for (int i = b0; i < b1; ++i) {
                const float z = v.z[i];
                cnt += (isfinite(z) && (okey(z) >> 21) >= d0) ? 1u : 0u;
            }
            uint64_t tot;
            const uint64_t ex = block_excl_scan_u64(cnt, sm->wsum, tot);
            if (tid == 0) sm->xch[c.xb][0] = tot;
            exch(c, 1);
            uint64_t all = 0, pre = 0;
            for (int j = 0; j < c.nc; ++j) {
                all += sm->gath[j][0];
                if (j < c.rank) pre += sm->gath[j][0];
            }
            if (all <= static_cast<uint64_t>(kListCap)) {
                // gather every rank's candidates, in id order, into rank 0
                float* lz = cluster.map_shared_rank(&sm->list_z[0], 0);
                int* li = cluster.map_shared_rank(&sm->list_id[0], 0);
                uint64_t pos = pre + ex;
                for (int i = b0; i < b1; ++i) {
                    const float z = v.z[i];
                    if (isfinite(z) && (okey(z) >> 21) >= d0) {
                        lz[pos] = z;
                        li[pos] = lo + i;
                        ++pos;
                    }
                }
                cluster.sync();
                if (c.rank != 0) return;  // rank 0 finishes the row alone
                c.solo = true;
                v.z = sm->list_z;
                v.id = sm->list_id;
                v.n = static_cast<int>(all);
                v.idbase = 0;
            }
        }
        const uint32_t p1 = d0;
        radix_pass<false>(c, v, kp, false, p1, 11, 10, 11, target, above, d1, binw, zmax, invT, false, 0.f, nullptr);
        const uint32_t p2 = (d0 << 11) | d1;
        radix_pass<false>(c, v, kp, false, p2, 22, 0, 10, target, above, d2, binw, zmax, invT, false, 0.f, nullptr);
        kp.tauk = (d0 << 21) | (d1 << 10) | d2;
        kp.idk = tie_select(c, v, kp, false, kp.tauk, target - above);
    }

    // ---- top-p: three mass passes over the top-k set; the first also yields S_k
    if (kp.p_on) {
        uint64_t target = 0, above = 0, binw = 0, Sk = 0;
        uint32_t d0, d1, d2;
        radix_pass<true>(c, v, kp, true, 0u, 0, 21, 11, target, above, d0, binw, zmax, invT, true, pp, &Sk);
        radix_pass<true>(c, v, kp, true, d0, 11, 10, 11, target, above, d1, binw, zmax, invT, false, 0.f, nullptr);
        radix_pass<true>(c, v, kp, true, (d0 << 11) | d1, 22, 0, 10, target, above, d2, binw, zmax, invT, false, 0.f,
                         nullptr);
        kp.taup = (d0 << 21) | (d1 << 10) | d2;
        const uint64_t wt = mass(key_float(kp.taup), zmax, invT);
        uint64_t need = 1;
        if (wt > 0 && target > above) need = (target - above + wt - 1) / wt;
        kp.idp = tie_select(c, v, kp, true, kp.taup, need);
    }

    // ---- draw: first kept id (ascending) whose running mass exceeds u * S_p
    {
        const int E = run_len(v.n);
        const int b0 = min(v.n, tid * E), b1 = min(v.n, b0 + E);
        uint64_t w = 0;
        for (int i = b0; i < b1; ++i) {
            const float z = v.z[i];
            if (!isfinite(z)) continue;
            const uint32_t key = okey(z);
            const int id = v.idat(i);
            if (kp.topk(key, id) && kp.topp(key, id)) w += mass(z, zmax, invT);
        }
        if (tid == 0) sm->imin = INT_MAX;
        uint64_t tot;
        const uint64_t ex = block_excl_scan_u64(w, sm->wsum, tot);
        if (tid == 0) sm->xch[c.xb][0] = tot;
        exch(c, 1);
        uint64_t Sp = 0, pre = 0;
        for (int j = 0; j < c.nce(); ++j) {
            Sp += sm->gath[j][0];
            if (j < c.rke()) pre += sm->gath[j][0];
        }
        const uint64_t u53 = philox_word0(seeds[row], offsets[row]) >> 11;
        const uint64_t X = static_cast<uint64_t>((static_cast<unsigned __int128>(u53) * Sp) >> 53);  // floor(u*Sp) < Sp
        if (pre <= X && X < pre + tot && pre + ex <= X && X < pre + ex + w) {
            uint64_t cum = pre + ex;
            for (int i = b0; i < b1; ++i) {
                const float z = v.z[i];
                if (!isfinite(z)) continue;
                const uint32_t key = okey(z);
                const int id = v.idat(i);
                if (!(kp.topk(key, id) && kp.topp(key, id))) continue;
                cum += mass(z, zmax, invT);
                if (cum > X) {
                    atomicMin(&sm->imin, id);
                    break;
                }
            }
        }
        __syncthreads();
        if (tid == 0) sm->xch[c.xb][0] = static_cast<unsigned long long>(static_cast<uint32_t>(sm->imin));
        exch(c, 1);
        int tok = INT_MAX;
        for (int j = 0; j < c.nce(); ++j) tok = min(tok, static_cast<int>(static_cast<uint32_t>(sm->gath[j][0])));
        if (c.rke() == 0 && tid == 0) tokens[row] = tok == INT_MAX ? -1 : tok;
    }
    if (!c.solo) cluster.sync();
}

// ------------------------------------------------------------------ host side
struct SamplerPlan {
    int nc, S, smem_slice;
    size_t smem;
};

static SamplerPlan plan_sampler(int V) {
    SamplerPlan p;
    int nc = (V + 20479) / 20480;
    if (nc < 1) nc = 1;
    if (nc > kMaxCluster) nc = kMaxCluster;
    int S = (V + nc - 1) / nc;
    S = (S + 3) & ~3;
    p.nc = nc;
    p.S = S;
    p.smem_slice = S <= kSliceSmemMax ? 1 : 0;
    p.smem = sizeof(SampSmem) + (p.smem_slice ? static_cast<size_t>(S) * 4 : 0);
    return p;
}

cudaError_t launch_sampler(int32_t* tokens, const float* logits, int B, int V, const float* temperature,
                           const int32_t* top_k, const float* top_p, const uint64_t* seeds, const uint64_t* offsets,
                           int32_t* status, cudaStream_t stream) {
    const SamplerPlan sp = plan_sampler(V);
    cudaError_t err = cudaFuncSetAttribute(sampler_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(sp.smem));
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B) * sp.nc, 1, 1);
    cfg.blockDim = dim3(kST, 1, 1);
    cfg.dynamicSmemBytes = sp.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = sp.nc;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sampler_kernel, tokens, logits, V, sp.S, sp.smem_slice, temperature, top_k,
                              top_p, seeds, offsets, status);
}

}  // namespace pkv
