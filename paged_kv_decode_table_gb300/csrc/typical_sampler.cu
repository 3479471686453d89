// typical_sampler.cu -- typical sampling, one thread-block cluster per row.
//
// "LLM inference serving tutorial" section 3.1 (other samplers: typical
// sampling; Meister et al., locally typical sampling): over the temperature
// distribution p of the finite logits, tokens are taken in ascending
// d_i = |-ln p_i - H(p)| until their probability first reaches typical_p
// (boundary token kept); the kept set is renormalised and drawn in token-id
// order with the request's Philox uniform, as in the sampler.
//
// With u_i = (z_i - zmax) log2(e) / T and ubar = sum_i p_i u_i one has
// -ln p_i - H = ln 2 (ubar - u_i): the order by d is the order by
// D_i = |u_i - ubar|, so the kept set is an interval of logits around the
// p-weighted mean.  The order is taken on D in double: ubar from Kahan float
// sums per thread (u with the scale log2(e) / T carried in two floats),
// combined exactly as 64-bit integers in 2^-40 units across threads and CTAs
// (about 1e-7 in log2 units on vocabulary rows); u_i = (z_i - zmax) * log2(e) / T
// in double.  A float
// estimate of D with a stated error bound places each logit, so only the
// logits within that bound of a threshold compute D in double.  Equal D go to
// the larger logit, then to the smaller id.  Masses are 2^-40 fixed-point
// weights floor(2^u * 2^40), so the cut and the draw are exact integer
// arithmetic (with typical_p >= 1 they are the sampler's masses, so the draw
// is the sampler's).
//
// A row is spread over a cluster of 1-8 CTAs (as many as fill the GPU with
// one CTA per SM), each sweeping one slice; per-CTA partials are combined in
// rank order through distributed shared memory, so every CTA holds the same
// results.  Passes over the slices (the first from HBM, the rest from L2):
// maximum and finiteness; the mass sum S and the weighted sums for ubar; 2048
// float bins linear in the estimate of D, summed over the cluster, which
// locate the cut approximately; the logits of a window of bins around it
// (window membership decided on D in double near its edges) pushed into
// rank 0 with the exact mass before and inside the window, where they are
// sorted by (D, larger logit, id) and the cut found exactly; the draw (chunk
// sums of the kept masses, a scan over the cluster, one chunk walked by the
// CTA holding the draw).  When the window overflows 2048 logits or misses
// the cut, rank 0 alone takes an exact radix select over the window (the
// whole row when it missed): the 64 bits of D, then the logit, then the rank
// in id order, and draws.
#include <cooperative_groups.h>
#include <math.h>

#include "pkv_common.cuh"
#include "sampling_math.cuh"

namespace cg = cooperative_groups;

namespace pkv {

constexpr int kTyT = 1024;          // threads per CTA
constexpr int kTyW = kTyT / 32;     // warps
constexpr int kTyBins = 2048;       // radix digits (11 bits), or draw chunks

struct TySmem {
    unsigned long long hist[kTyBins];  // mass histogram, the window's D keys, or chunk sums / prefixes
    unsigned int cnt[kTyBins];         // the window's token ids
    unsigned int zk[kTyBins];          // the window's logit keys ~okey(z) (ascending: larger logit first)
    unsigned int nwin;
    unsigned long long wsum[kTyW];
    double dsc[4];  // row scalars in double, computed by one thread: log2(e) / T, the centre, the window's edges
    float fv[kTyW];
    unsigned long long bc[4];
    unsigned long long u53;  // the row's uniform, top 53 bits of Philox word 0
    // cluster exchange: one CTA's partial of a cluster-wide reduction, in two
    // alternating slots (a slot is rewritten only after the barrier of the
    // next exchange, which every reader of it has passed)
    struct {
        unsigned long long u[2];
        double d[2];
        float f[2];
    } xch[2];
    unsigned long long res[4];  // rank 0: the cut (found, D bits, logit key, id) for the cluster
};

// An opaque copy of a value: the compiler cannot trace it back to the double
// arithmetic it came from, so under register pressure it keeps or spills the
// value instead of recomputing it inside the per-logit loops (float <-> double
// conversions run on this GPU's slow FP64 pipe).
__device__ __forceinline__ float ty_pin(float v) {
    float r;
    asm volatile("mov.b32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// Compensated (Kahan) float summation: the sum so far is s - c, c carrying the
// rounding error of each addition (explicit round-to-nearest operations, so
// that no contraction or reassociation undoes it).
__device__ __forceinline__ void kahan_add(float& s, float& c, float v) {
    const float y = __fsub_rn(v, c);
    const float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
}

// ------------------------------------------------------------------ CTA reductions
// Every thread returns the CTA-wide result.  Each starts with a barrier, so
// back-to-back calls do not race on the per-warp slots.
__device__ __forceinline__ uint64_t ty_warp_sum(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ uint64_t ty_sum_u64(uint64_t v, TySmem* sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = ty_warp_sum(v);
    __syncthreads();
    if (lane == 0) sm->wsum[warp] = v;
    __syncthreads();
    return ty_warp_sum(sm->wsum[lane]);
}
template <bool kMax>
__device__ float ty_ext_f(float v, TySmem* sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float y = __shfl_xor_sync(0xffffffffu, v, o);
        v = kMax ? fmaxf(v, y) : fminf(v, y);
    }
    __syncthreads();
    if (lane == 0) sm->fv[warp] = v;
    __syncthreads();
    float t = sm->fv[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float y = __shfl_xor_sync(0xffffffffu, t, o);
        t = kMax ? fmaxf(t, y) : fminf(t, y);
    }
    return t;
}
// Exclusive prefix of v over the threads in index order; total = the sum.
__device__ uint64_t ty_excl_scan(uint64_t v, TySmem* sm, uint64_t& total) {
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
    const uint64_t w = sm->wsum[lane];
    uint64_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
    }
    total = __shfl_sync(0xffffffffu, wi, 31);
    const uint64_t before = __shfl_sync(0xffffffffu, wi - w, warp);
    return before + inc - v;
}

// Strided sweep over the row, f(i, x) for every element: thread t takes the
// 4-element slots 4 (t + kTyT m), kU of them loaded before any is processed
// (16-byte loads when the row is 16-byte aligned), so that each thread keeps
// kU loads in flight.
constexpr int kTyU = 4;
template <typename F>
__device__ __forceinline__ void ty_sweep(const float* __restrict__ z, int n, F&& f) {
    const bool a16 = (reinterpret_cast<uintptr_t>(z) & 15u) == 0;
    for (int e0 = 4 * static_cast<int>(threadIdx.x); e0 < n; e0 += 4 * kTyT * kTyU) {
        float4 q[kTyU];
#pragma unroll
        for (int u = 0; u < kTyU; ++u) {
            const int e = e0 + 4 * kTyT * u;
            if (a16 && e + 4 <= n) {
                q[u] = __ldg(reinterpret_cast<const float4*>(z + e));
            } else {
                q[u].x = e < n ? z[e] : -INFINITY;
                q[u].y = e + 1 < n ? z[e + 1] : -INFINITY;
                q[u].z = e + 2 < n ? z[e + 2] : -INFINITY;
                q[u].w = e + 3 < n ? z[e + 3] : -INFINITY;
            }
        }
#pragma unroll
        for (int u = 0; u < kTyU; ++u) {
            const int e = e0 + 4 * kTyT * u;
            if (e < n) f(e, q[u].x);
            if (e + 1 < n) f(e + 1, q[u].y);
            if (e + 2 < n) f(e + 2, q[u].z);
            if (e + 3 < n) f(e + 3, q[u].w);
        }
    }
}

// ------------------------------------------------------------------ radix select
// Among the row's elements that keyf accepts (keyf(x, i, key, m) -> in scope,
// with its 32-bit key and mass) and whose key matches `prefix` in the top
// `pbits` bits: the digit d of key bits [shift, shift + nbits) at which the
// cumulative mass in ascending key order, starting from `above`, first
// reaches `target`.  `above` is advanced past the smaller digits.
template <typename KeyF>
__device__ uint32_t ty_radix(const float* __restrict__ z, int n, TySmem* sm, KeyF keyf, uint32_t prefix, int pbits,
                             int shift, int nbits, uint64_t target, uint64_t& above) {
    const int tid = threadIdx.x;
    const int nb = 1 << nbits;
    for (int i = tid; i < nb; i += kTyT) sm->hist[i] = 0ull;
    if (tid == 0) {
        sm->bc[0] = static_cast<unsigned long long>(nb - 1);
        sm->bc[1] = above;
    }
    __syncthreads();
    // a thread's run of equal digits is added once (the leading digits of a
    // row cluster in a few bins, where shared atomics would serialise)
    uint32_t cd = 0u;
    uint64_t cs = 0;
    ty_sweep(z, n, [&](int i, float x) {
        uint32_t key;
        uint64_t m;
        if (!keyf(x, i, key, m)) return;
        if (pbits && (key >> (32 - pbits)) != prefix) return;
        const uint32_t d = (key >> shift) & static_cast<uint32_t>(nb - 1);
        if (d != cd) {
            if (cs) atomicAdd(&sm->hist[cd], static_cast<unsigned long long>(cs));
            cd = d;
            cs = 0;
        }
        cs += m;
    });
    if (cs) atomicAdd(&sm->hist[cd], static_cast<unsigned long long>(cs));
    __syncthreads();
    const int b0 = 2 * tid;  // two digits per thread, ascending
    const uint64_t h0 = b0 < nb ? sm->hist[b0] : 0ull, h1 = b0 + 1 < nb ? sm->hist[b0 + 1] : 0ull;
    uint64_t tot;
    const uint64_t c0 = above + ty_excl_scan(h0 + h1, sm, tot);
    if (c0 < target && c0 + h0 + h1 >= target) {
        if (c0 + h0 >= target) {
            sm->bc[0] = static_cast<unsigned long long>(b0);
            sm->bc[1] = c0;
        } else {
            sm->bc[0] = static_cast<unsigned long long>(b0 + 1);
            sm->bc[1] = c0 + h0;
        }
    }
    __syncthreads();
    const uint32_t d = static_cast<uint32_t>(sm->bc[0]);
    above = sm->bc[1];
    __syncthreads();  // bc and hist are reused by the next call
    return d;
}

// ------------------------------------------------------------------ ordered find
// First element i (ascending) at which the running sum of valf(z[i], i) exceeds
// X = xf(total).  The row is cut into chunks of 128 * cpw consecutive elements
// (at most kTyBins chunks); warp w sums chunks w, w + 32, ... with coalesced
// loads, the chunk sums are scanned, and warp 0 walks the one chunk holding X.
// Returns -1 when X >= total (nothing to find).
template <typename ValF, typename XF>
__device__ int ty_ordered_find(const float* __restrict__ z, int n, TySmem* sm, ValF valf, XF xf) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nvec = (n + 3) & ~3;
    const int cpw = max(1, (nvec + 128 * kTyBins - 1) / (128 * kTyBins));
    const int csz = 128 * cpw;
    const int nch = (nvec + csz - 1) / csz;
    const bool a16 = (reinterpret_cast<uintptr_t>(z) & 15u) == 0;
    auto load4 = [&](int e) -> float4 {  // the lane's 4 elements starting at e (-inf past n)
        if (a16 && e + 4 <= n) return __ldg(reinterpret_cast<const float4*>(z + e));
        float4 q;
        q.x = e < n ? z[e] : -INFINITY;
        q.y = e + 1 < n ? z[e + 1] : -INFINITY;
        q.z = e + 2 < n ? z[e + 2] : -INFINITY;
        q.w = e + 3 < n ? z[e + 3] : -INFINITY;
        return q;
    };
    auto val4 = [&](const float4& q, int e) -> uint64_t {
        return (e < n ? valf(q.x, e) : 0ull) + (e + 1 < n ? valf(q.y, e + 1) : 0ull) +
               (e + 2 < n ? valf(q.z, e + 2) : 0ull) + (e + 3 < n ? valf(q.w, e + 3) : 0ull);
    };
    // warp w sums chunks w, w + 32, w + 64, w + 96 together (four loads in flight)
    for (int cb = warp; cb < nch; cb += 4 * kTyW) {
        uint64_t w[4] = {0ull, 0ull, 0ull, 0ull};
        for (int k = 0; k < cpw; ++k) {
            float4 q[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) q[u] = load4((cb + u * kTyW) * csz + 128 * k + 4 * lane);
#pragma unroll
            for (int u = 0; u < 4; ++u) w[u] += val4(q[u], (cb + u * kTyW) * csz + 128 * k + 4 * lane);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint64_t t = ty_warp_sum(w[u]);
            if (lane == 0 && cb + u * kTyW < nch) sm->hist[cb + u * kTyW] = t;
        }
    }
    __syncthreads();
    const int c0 = 2 * tid;
    const uint64_t a0 = c0 < nch ? sm->hist[c0] : 0ull, a1 = c0 + 1 < nch ? sm->hist[c0 + 1] : 0ull;
    uint64_t tot;
    const uint64_t ex = ty_excl_scan(a0 + a1, sm, tot);
    if (c0 < nch) sm->hist[c0] = ex;
    if (c0 + 1 < nch) sm->hist[c0 + 1] = ex + a0;
    const uint64_t X = xf(tot);
    if (tid == 0) {
        sm->bc[2] = ~0ull;  // chunk holding X
        sm->bc[3] = ~0ull;  // the element found
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int ch = c0 + q;
        if (ch < nch) {
            const uint64_t lo = sm->hist[ch], hi = ch + 1 < nch ? sm->hist[ch + 1] : tot;
            if (lo <= X && X < hi) sm->bc[2] = static_cast<unsigned long long>(ch);
        }
    }
    __syncthreads();
    const unsigned long long cs = sm->bc[2];
    if (warp == 0 && cs != ~0ull) {
        uint64_t base = sm->hist[cs];
        for (int k = 0; k < cpw; ++k) {
            const int e = static_cast<int>(cs) * csz + 128 * k + 4 * lane;
            const float4 q = load4(e);
            const uint64_t m[4] = {e < n ? valf(q.x, e) : 0ull, e + 1 < n ? valf(q.y, e + 1) : 0ull,
                                   e + 2 < n ? valf(q.z, e + 2) : 0ull, e + 3 < n ? valf(q.w, e + 3) : 0ull};
            const uint64_t mine = m[0] + m[1] + m[2] + m[3];
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
                for (int j = 0; j < 4; ++j) {
                    cum += m[j];
                    if (cum > X) {
                        sm->bc[3] = static_cast<unsigned long long>(e + j);
                        break;
                    }
                }
            }
            base += __shfl_sync(0xffffffffu, inc, 31);
            if (base > X) break;  // warp-uniform
        }
    }
    __syncthreads();
    const unsigned long long f = sm->bc[3];
    __syncthreads();  // bc and hist are reused by the next call
    return f == ~0ull ? -1 : static_cast<int>(f);
}

// ------------------------------------------------------------------ kernel
// One cluster of nc CTAs per row; CTA `rank` sweeps the slice [lo, lo + n) of
// the row.  Reductions combine the CTAs' partials in rank order, so every CTA
// holds the same, deterministic results.
__global__ void __launch_bounds__(kTyT, 1)
    typical_sampler_kernel(int32_t* __restrict__ tokens, const float* __restrict__ logits, int V, int slice,
                           const float* __restrict__ temperature, const float* __restrict__ typical_p,
                           const uint64_t* __restrict__ seeds, const uint64_t* __restrict__ offsets,
                           int32_t* status) {
    __shared__ TySmem smem;
    TySmem* sm = &smem;
    cg::cluster_group cl = cg::this_cluster();
    const int nc = static_cast<int>(cl.num_blocks()), rank = static_cast<int>(cl.block_rank());
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x, row = blockIdx.x / nc;
    const float* z = logits + static_cast<size_t>(row) * V;
    const int lo = min(V, rank * slice), n = min(V, lo + slice) - lo;
    const float* zs = z + lo;  // this CTA's slice
    const float T = temperature[row], tp = typical_p[row];
    if (tid == kTyT - 1) sm->u53 = philox_word0(seeds[row], offsets[row]) >> 11;
    // log2(e) / T in double, by one thread (read after the next barrier)
    if (tid == 0) sm->dsc[0] = 1.4426950408889634 / static_cast<double>(T);
    if (rank == 0 && tid == 0) tokens[row] = -1;  // overwritten (after a cluster barrier) by the draw

    // cluster exchange: thread 0 publishes the CTA's partial, the barrier makes
    // it visible, every thread then reads the nc partials with rd(r)
    int xk = 0;
    auto publish = [&](unsigned long long u0, unsigned long long u1, double d0, double d1, float f0, float f1) {
        if (tid == 0) {
            sm->xch[xk & 1].u[0] = u0;
            sm->xch[xk & 1].u[1] = u1;
            sm->xch[xk & 1].d[0] = d0;
            sm->xch[xk & 1].d[1] = d1;
            sm->xch[xk & 1].f[0] = f0;
            sm->xch[xk & 1].f[1] = f1;
        }
        cl.sync();
    };
    auto rd = [&](int r) { return cl.map_shared_rank(&sm->xch[xk & 1], r); };
    // X (a position in the cluster's total of per-CTA totals `tot`, from Xof of
    // that total) relative to this CTA, or ~0 when it lies in another CTA
    auto cluster_x = [&](uint64_t tot, auto Xof) -> uint64_t {
        publish(tot, 0ull, 0.0, 0.0, 0.f, 0.f);
        uint64_t excl = 0, grand = 0;
        for (int r = 0; r < nc; ++r) {
            const uint64_t t = rd(r)->u[0];
            excl += r < rank ? t : 0ull;
            grand += t;
        }
        ++xk;
        const uint64_t X = Xof(grand);
        return (X >= excl && X - excl < tot) ? X - excl : ~0ull;
    };

    // ---- maximum and finiteness
    float mx = -INFINITY, mn = INFINITY;
    unsigned int bad = 0u;
    ty_sweep(zs, n, [&](int, float x) {
        mx = fmaxf(mx, x);
        mn = fminf(mn, x > -INFINITY ? x : INFINITY);
        bad |= (x < INFINITY) ? 0u : 1u;  // NaN or +inf
    });
    mx = ty_ext_f<true>(mx, sm);
    mn = ty_ext_f<false>(mn, sm);
    bad = static_cast<unsigned int>(ty_sum_u64(bad, sm));
    publish(bad, 0ull, 0.0, 0.0, mx, mn);
    bad = 0u;
    mx = -INFINITY;
    mn = INFINITY;
    for (int r = 0; r < nc; ++r) {
        bad |= static_cast<unsigned int>(rd(r)->u[0]);
        mx = fmaxf(mx, rd(r)->f[0]);
        mn = fminf(mn, rd(r)->f[1]);
    }
    ++xk;
    int err = 0;
    if (bad || !(mx > -INFINITY)) err = PKV_ERR_NONFINITE;
    else if (!(T >= 0.f)) err = PKV_ERR_INVALID_ARG;
    else if (T != 0.f && !(tp > 0.f)) err = PKV_ERR_INVALID_ARG;  // typical_p <= 0 or NaN
    if (err) {
        if (rank == 0 && tid == 0) report(status, err);
        cl.sync();  // no CTA leaves while a peer may still read its slot
        return;
    }
    if (T == 0.f) {  // greedy: the lowest id holding the maximum
        float first = INFINITY;
        for (int i = tid; i < n; i += kTyT)
            if (zs[i] == mx) {
                first = static_cast<float>(lo + i);  // ids < 2^24 are exact in float
                break;
            }
        first = ty_ext_f<false>(first, sm);
        publish(0ull, 0ull, 0.0, 0.0, first, 0.f);
        for (int r = 0; r < nc; ++r) first = fminf(first, rd(r)->f[0]);
        ++xk;
        if (rank == 0 && tid == 0) tokens[row] = static_cast<int32_t>(first);
        cl.sync();
        return;
    }
    const float c2 = fminf(1.4426950408889634f / T, 1.0e30f);  // log2(e) / T, kept finite
    auto uof = [&](float x) { return __fmul_rn(__fsub_rn(x, mx), c2); };
    // the fixed-point mass of a logit, as the sampler's (the untruncated draw)
    auto massof = [&](float x) { return fx40(hw_exp2(uof(x))); };
    // u with the scale log2(e) / T carried in two floats (chi + clo), for the
    // centre and the order; exact_only when that scale is beyond 1e30 (then
    // every order decision is taken on D in double)
    const double mxd = static_cast<double>(mx);
    const double c2d = sm->dsc[0];
    const bool exact_only = ty_pin(c2d <= 1.0e30 ? 0.f : 1.f) != 0.f;
    const float chi = ty_pin(exact_only ? 1.0e30f : static_cast<float>(c2d));
    const float clo = ty_pin(exact_only ? 0.f : static_cast<float>(c2d - static_cast<double>(static_cast<float>(c2d))));
    auto ucof = [&](float x) {
        const float dz = __fsub_rn(x, mx);
        return __fmaf_rn(dz, chi, __fmul_rn(dz, clo));
    };
    // the fixed-point mass of the truncated path, from the same u as the order
    auto massc = [&](float x) { return fx40(hw_exp2(ucof(x))); };
    auto draw_x = [&](uint64_t tot) {  // floor(u * tot) < tot
        return static_cast<uint64_t>((static_cast<unsigned __int128>(sm->u53) * tot) >> 53);
    };
    if (!(tp < 1.f)) {  // no truncation: every finite logit
        const int f = ty_ordered_find(
            zs, n, sm, [&](float x, int) -> uint64_t { return x > -INFINITY ? massof(x) : 0ull; },
            [&](uint64_t tot) { return cluster_x(tot, draw_x); });
        if (f >= 0 && tid == 0) tokens[row] = lo + f;
        cl.sync();
        return;
    }

    // ---- S (exact fixed-point masses) and the p-weighted mean of u.  The
    // centre ubar = sum w u / sum w takes u from the compensated scale ucof and
    // Kahan sums per thread (error ~1e-7 in log2 units on vocabulary rows; a
    // plain float scale would bias it by the rounding of log2(e) / T times the
    // spread of u); each thread's sum and compensation are turned into 2^-40
    // units (exact at these magnitudes, the floats' ulps being multiples of
    // 2^-40; |w u| <= 1 / (e ln 2) per logit keeps the totals below 2^57) and
    // added exactly as 64-bit integers across threads and CTAs.
    uint64_t s = 0;
    float ws = 0.f, wc = 0.f, us = 0.f, uc = 0.f;
    ty_sweep(zs, n, [&](int, float x) {
        if (!(x > -INFINITY)) return;
        const float u = ucof(x);
        const float w = hw_exp2(u);
        s += fx40(w);
        if (w > 0.f) {
            kahan_add(ws, wc, w);
            kahan_add(us, uc, __fmul_rn(w, u));
        }
    });
    const uint64_t Sc = ty_sum_u64(s, sm);
    auto units = [](float v) { return static_cast<uint64_t>(__float2ll_rn(__fmul_rn(v, 0x1p40f))); };
    const uint64_t Wc = ty_sum_u64(units(ws) - units(wc), sm);   // two's complement sums
    const uint64_t WUc = ty_sum_u64(units(us) - units(uc), sm);
    // (the signed total of w u travels as the bit pattern of a double slot)
    publish(Sc, Wc, __longlong_as_double(static_cast<long long>(WUc)), 0.0, 0.f, 0.f);
    uint64_t S = 0;
    for (int r = 0; r < nc; ++r) S += rd(r)->u[0];
    if (tid == 0) {  // the centre, by one thread
        uint64_t W = 0, WU = 0;
        for (int r = 0; r < nc; ++r) {
            W += rd(r)->u[1];
            WU += static_cast<uint64_t>(__double_as_longlong(rd(r)->d[0]));
        }
        // W >= 2^40: the maximum weighs 1
        sm->dsc[1] = static_cast<double>(static_cast<long long>(WU)) / static_cast<double>(W);
    }
    __syncthreads();
    ++xk;
    const double ubar = sm->dsc[1];
    const float ubf = ty_pin(static_cast<float>(ubar));
    // The order key: D = |u - ubar| in double (log2 units; d = D ln 2), with a
    // float estimate dk = |ucof(x) - ubf| within errf(u) of it (4x the error
    // bound of the float operations), so that only logits whose dk lies within
    // errf of a threshold need D.
    auto dex = [&](float x) -> double {
        return fabs(__dsub_rn(__dmul_rn(__dsub_rn(static_cast<double>(x), mxd), c2d), ubar));
    };
    auto dkf = [&](float u) { return fabsf(__fsub_rn(u, ubf)); };
    auto errf = [&](float u) {
        return exact_only ? INFINITY : __fmaf_rn(__fadd_rn(fabsf(u), fabsf(ubf)), 0x1p-19f, 0x1p-126f);
    };
    const uint64_t target = ceil_mul_p(tp, S);  // >= 1, <= S

    // ---- 2048 bins linear in dk over [0, dkmax] (bin 0: closest to the mean):
    // the weight per bin (float, summed over the cluster in rank order); the
    // bin where the cumulative weight in ascending dk first reaches the target
    // holds the cut, approximately
    const float dkmax = fmaxf(dkf(ucof(mn)), fabsf(ubf));
    const float sc = static_cast<float>(kTyBins) / dkmax;
    const float scale = (dkmax > 0.f && sc < INFINITY) ? sc : 0.f;  // 0: one bin
    auto dbin = [&](float dk) {  // monotone non-decreasing in dk; inf * 0 (NaN) -> the last bin
        const float t = dk * scale;
        return t < static_cast<float>(kTyBins - 1) ? static_cast<int>(t) : kTyBins - 1;
    };
    float* hf = reinterpret_cast<float*>(sm->hist);  // approximate bin weights 2^u
    for (int i = tid; i < kTyBins; i += kTyT) hf[i] = 0.f;
    if (tid == 0) sm->nwin = 0u;
    __syncthreads();
    {
        int cb = 0;  // a thread's run of equal bins is added once
        float cw = 0.f;
        ty_sweep(zs, n, [&](int, float x) {
            if (!(x > -INFINITY)) return;
            const float u = ucof(x);
            const int bq = dbin(dkf(u));
            if (bq != cb) {
                if (cw > 0.f) atomicAdd(&hf[cb], cw);
                cb = bq;
                cw = 0.f;
            }
            cw += hw_exp2(u);
        });
        if (cw > 0.f) atomicAdd(&hf[cb], cw);
    }
    cl.sync();  // every CTA's bins are complete (and rank 0's window count is zero)
    // The float sums locate the cut only approximately: the window of bins
    // [blo, bhi] covers cumulative masses within S / 2^13 of the target on
    // either side; the gather pass checks it with exact masses.
    {
        const int b0 = 2 * tid;
        float f0 = 0.f, f1 = 0.f;
        for (int r = 0; r < nc; ++r) {
            const float* hr = cl.map_shared_rank(hf, r);
            f0 += hr[b0];
            f1 += hr[b0 + 1];
        }
        const uint64_t del = (S >> 13) ? (S >> 13) : 1ull;
        const uint64_t tlo = target > del ? target - del : 1ull, thi = target + del;
        const uint64_t h0 = __float2ull_rn(f0 * 0x1p40f), h1 = __float2ull_rn(f1 * 0x1p40f);
        if (tid == 0) {
            sm->bc[0] = 0ull;
            sm->bc[1] = kTyBins - 1;
        }
        uint64_t tot;
        const uint64_t c0 = ty_excl_scan(h0 + h1, sm, tot);  // (begins with a barrier)
        if (c0 < tlo && c0 + h0 + h1 >= tlo) sm->bc[0] = static_cast<unsigned long long>(c0 + h0 >= tlo ? b0 : b0 + 1);
        if (c0 < thi && c0 + h0 + h1 >= thi) sm->bc[1] = static_cast<unsigned long long>(c0 + h0 >= thi ? b0 : b0 + 1);
    }
    __syncthreads();
    const int blo = static_cast<int>(sm->bc[0]), bhi = max(blo, static_cast<int>(sm->bc[1]));
    // ---- the window: logits with Ed <= D < Fd (the bins' edges, in double,
    // by one thread); membership is decided on D itself wherever dk is within
    // errf of an edge
    const bool one_bin = !(scale > 0.f);
    if (tid == 0) {
        sm->dsc[2] = (one_bin || blo == 0) ? 0.0 : static_cast<double>(blo) / static_cast<double>(scale);
        sm->dsc[3] = (one_bin || bhi >= kTyBins - 1) ? static_cast<double>(INFINITY)
                                                     : static_cast<double>(bhi + 1) / static_cast<double>(scale);
    }
    cl.sync();  // no CTA reads another's bins any more; rank 0's bins become the window list
    const double Ed = sm->dsc[2], Fd = sm->dsc[3];
    // 0: before [lo, hi) in the order, 1: inside, 2: after
    // (lof, hif: the bounds rounded to float once, outside the sweeps)
    auto where = [&](float x, double lod, double hid, float lof, float hif) -> int {
        const float u = ucof(x);
        const float dk = dkf(u), e = errf(u);
        if (dk < lof - e) return 0;
        if (dk > lof + e && dk < hif - e) return 1;
        if (dk > hif + e) return 2;
        const double D = dex(x);
        return D < lod ? 0 : (D < hid ? 1 : 2);
    };

    // ---- the window's logits into rank 0's shared memory, keyed (D bits,
    // logit key, id) ascending; the exact masses before and inside the window
    unsigned long long* key = sm->hist;
    unsigned int* ids = sm->cnt;
    unsigned int* zkw = sm->zk;
    unsigned long long* key0 = cl.map_shared_rank(sm->hist, 0);
    unsigned int* ids0 = cl.map_shared_rank(sm->cnt, 0);
    unsigned int* zk0 = cl.map_shared_rank(sm->zk, 0);
    unsigned int* nwin0 = cl.map_shared_rank(&sm->nwin, 0);
    uint64_t at = 0, in = 0;
    const float Ef = ty_pin(static_cast<float>(Ed)), Ff = ty_pin(static_cast<float>(Fd));
    ty_sweep(zs, n, [&](int i, float x) {
        if (!(x > -INFINITY)) return;
        const int w = where(x, Ed, Fd, Ef, Ff);
        if (w == 0) {
            at += massc(x);
        } else if (w == 1) {
            in += massc(x);
            const unsigned int slot = atomicAdd(nwin0, 1u);
            if (slot < static_cast<unsigned int>(kTyBins)) {
                key0[slot] = static_cast<unsigned long long>(__double_as_longlong(dex(x)));
                zk0[slot] = ~okey(x);
                ids0[slot] = static_cast<unsigned int>(lo + i);
            }
        }
    });
    const uint64_t atc = ty_sum_u64(at, sm);
    const uint64_t inc = ty_sum_u64(in, sm);
    publish(atc, inc, 0.0, 0.0, 0.f, 0.f);  // its barrier also completes the pushes into rank 0
    uint64_t above = 0, inwin = 0;
    for (int r = 0; r < nc; ++r) {
        above += rd(r)->u[0];  // exact mass before the window
        inwin += rd(r)->u[1];  // exact mass of the window
    }
    ++xk;
    const bool cut_in_window = above < target && target <= above + inwin;

    // ---- rank 0 sorts the window and finds the cut; the cluster reads the result
    unsigned long long dstar = 0ull;
    uint32_t zstar = 0u;
    int idstar = -1;
    bool found = false;
    if (rank == 0) {
        const unsigned int nw = sm->nwin;
        if (cut_in_window && nw <= static_cast<unsigned int>(kTyBins)) {
            int np2 = 1;
            while (np2 < static_cast<int>(nw)) np2 <<= 1;
            for (int i = static_cast<int>(nw) + tid; i < np2; i += kTyT) {
                key[i] = ~0ull;
                zkw[i] = ~0u;
                ids[i] = ~0u;
            }
            __syncthreads();
            for (int k = 2; k <= np2; k <<= 1)
                for (int j = k >> 1; j > 0; j >>= 1) {
                    for (int i = tid; i < np2; i += kTyT) {
                        const int l = i ^ j;
                        if (l > i) {
                            const bool up = (i & k) == 0;
                            const unsigned long long ki = key[i], kl = key[l];
                            const unsigned int zi = zkw[i], zl = zkw[l];
                            const bool gt = ki > kl || (ki == kl && (zi > zl || (zi == zl && ids[i] > ids[l])));
                            if (gt == up) {
                                key[i] = kl;
                                key[l] = ki;
                                zkw[i] = zl;
                                zkw[l] = zi;
                                const unsigned int t = ids[i];
                                ids[i] = ids[l];
                                ids[l] = t;
                            }
                        }
                    }
                    __syncthreads();
                }
            // cumulative mass in sorted order: thread t takes entries [2t, 2t + 2)
            auto wmass = [&](int j) -> uint64_t {
                return j < static_cast<int>(nw) ? massc(key_float(~zkw[j])) : 0ull;
            };
            const int j0 = 2 * tid;
            const uint64_t w0 = wmass(j0), w1 = wmass(j0 + 1);
            if (tid == 0) sm->bc[2] = ~0ull;
            uint64_t wt;
            const uint64_t c0 = above + ty_excl_scan(w0 + w1, sm, wt);  // (begins with a barrier)
            if (c0 < target && c0 + w0 + w1 >= target) sm->bc[2] = static_cast<unsigned long long>(c0 + w0 >= target ? j0 : j0 + 1);
            __syncthreads();
            if (sm->bc[2] != ~0ull) {  // always, since the cut lies in the window
                const int jc = static_cast<int>(sm->bc[2]);
                dstar = key[jc];
                zstar = zkw[jc];
                idstar = static_cast<int>(ids[jc]);
                found = true;
            }
            __syncthreads();  // hist / cnt / zk are reused below
        }
        if (tid == 0) {
            sm->res[0] = found ? 1ull : 0ull;
            sm->res[1] = dstar;
            sm->res[2] = zstar;
            sm->res[3] = static_cast<uint32_t>(idstar);
        }
    }
    cl.sync();
    {
        const unsigned long long* r0 = cl.map_shared_rank(sm->res, 0);
        found = r0[0] != 0ull;
        dstar = r0[1];
        zstar = static_cast<uint32_t>(r0[2]);
        idstar = static_cast<int>(static_cast<uint32_t>(r0[3]));
    }
    if (!found && rank == 0) {
        // ---- the window overflowed (more than 2048 logits) or missed the cut:
        // rank 0 alone, over the whole row, takes an exact radix select over
        // the window's logits (the whole row when it missed): the 64 bits of D,
        // then the logit key, then the rank in id order
        const bool whole = !cut_in_window;
        const double lod = whole ? 0.0 : Ed, hid = whole ? static_cast<double>(INFINITY) : Fd;
        above = whole ? 0ull : above;
        const float lof = ty_pin(static_cast<float>(lod)), hif = ty_pin(static_cast<float>(hid));
        auto inw = [&](float x) { return x > -INFINITY && (whole || where(x, lod, hid, lof, hif) == 1); };
        auto kh = [&](float x, int, uint32_t& k, uint64_t& m) -> bool {
            if (!inw(x)) return false;
            k = static_cast<uint32_t>(static_cast<unsigned long long>(__double_as_longlong(dex(x))) >> 32);
            m = massc(x);
            return true;
        };
        const uint32_t a0 = ty_radix(z, V, sm, kh, 0u, 0, 21, 11, target, above);
        const uint32_t a1 = ty_radix(z, V, sm, kh, a0, 11, 10, 11, target, above);
        const uint32_t a2 = ty_radix(z, V, sm, kh, (a0 << 11) | a1, 22, 0, 10, target, above);
        const uint32_t dhi = (a0 << 21) | (a1 << 10) | a2;
        auto kl = [&](float x, int, uint32_t& k, uint64_t& m) -> bool {
            if (!inw(x)) return false;
            const unsigned long long db = static_cast<unsigned long long>(__double_as_longlong(dex(x)));
            if (static_cast<uint32_t>(db >> 32) != dhi) return false;
            k = static_cast<uint32_t>(db);
            m = massc(x);
            return true;
        };
        const uint32_t b0 = ty_radix(z, V, sm, kl, 0u, 0, 21, 11, target, above);
        const uint32_t b1 = ty_radix(z, V, sm, kl, b0, 11, 10, 11, target, above);
        const uint32_t b2 = ty_radix(z, V, sm, kl, (b0 << 11) | b1, 22, 0, 10, target, above);
        dstar = (static_cast<unsigned long long>(dhi) << 32) | ((b0 << 21) | (b1 << 10) | b2);
        const double ds = __longlong_as_double(static_cast<long long>(dstar));
        // among equal D: the larger logit first (ascending ~okey)
        float gmin = INFINITY, gmax = -INFINITY;
        ty_sweep(z, V, [&](int, float x) {
            if (!inw(x) || dex(x) != ds) return;
            gmin = fminf(gmin, x);
            gmax = fmaxf(gmax, x);
        });
        gmin = ty_ext_f<false>(gmin, sm);
        gmax = ty_ext_f<true>(gmax, sm);
        zstar = ~okey(gmax);
        if (!(gmin == gmax)) {
            auto kz = [&](float x, int, uint32_t& k, uint64_t& m) -> bool {
                if (!inw(x) || dex(x) != ds) return false;
                k = ~okey(x);
                m = massc(x);
                return true;
            };
            const uint32_t e0 = ty_radix(z, V, sm, kz, 0u, 0, 21, 11, target, above);
            const uint32_t e1 = ty_radix(z, V, sm, kz, e0, 11, 10, 11, target, above);
            const uint32_t e2 = ty_radix(z, V, sm, kz, (e0 << 11) | e1, 22, 0, 10, target, above);
            zstar = (e0 << 21) | (e1 << 10) | e2;
        }
        // the cut among equal (D, logit) (equal masses): the r-th in id order
        const uint64_t mstar = massc(key_float(~zstar));
        const uint64_t need = target - above;
        const uint64_t r = mstar ? (need + mstar - 1) / mstar : 1ull;
        const uint32_t zs_ = zstar;
        idstar = ty_ordered_find(
            z, V, sm,
            [&](float x, int) -> uint64_t { return (inw(x) && dex(x) == ds && ~okey(x) == zs_) ? 1ull : 0ull; },
            [&](uint64_t) { return r - 1; });
    }

    // ---- the draw over the kept set in id order: (D, logit key, id) up to the cut's
    const double ds = __longlong_as_double(static_cast<long long>(dstar));
    const float dsf = ty_pin(static_cast<float>(ds));
    auto kept = [&](float x, int i) -> uint64_t {  // i: the id
        if (!(x > -INFINITY)) return 0ull;
        const float u = ucof(x);
        const float dk = dkf(u), e = errf(u);
        auto mass_u = [&] { return fx40(hw_exp2(u)); };
        bool keep;
        if (dk < dsf - e) {
            keep = true;
        } else if (dk > dsf + e) {
            keep = false;
        } else {
            const double D = dex(x);
            const uint32_t k = ~okey(x);
            keep = D < ds || (D == ds && (k < zstar || (k == zstar && i <= idstar)));
        }
        return keep ? mass_u() : 0ull;
    };
    if (!found) {
        if (rank == 0) {
            const int tok = ty_ordered_find(z, V, sm, kept, draw_x);
            if (tid == 0) tokens[row] = tok;
        }
        cl.sync();
        return;
    }
    const int f = ty_ordered_find(
        zs, n, sm, [&](float x, int i) { return kept(x, lo + i); },
        [&](uint64_t tot) { return cluster_x(tot, draw_x); });
    if (f >= 0 && tid == 0) tokens[row] = lo + f;
    cl.sync();  // no CTA leaves while a peer may still read its slot
}

int device_sm_count();

// CTAs per row: as many as fill the GPU with one CTA per SM (1, 2, 4 or 8),
// keeping slices of at least 2048 logits.
static int typical_cluster_size(int B, int V) {
    const int sms = device_sm_count();
    int nc = 1;
    while (nc < 8 && static_cast<long long>(B) * nc * 2 <= sms && V / (nc * 2) >= 2048) nc *= 2;
    return nc;
}

cudaError_t launch_typical_sampler(int32_t* tokens, const float* logits, int B, int V, const float* temperature,
                                   const float* typical_p, const uint64_t* seeds, const uint64_t* offsets,
                                   int32_t* status, cudaStream_t stream) {
    const int nc = typical_cluster_size(B, V);
    int slice = (V + nc - 1) / nc;
    slice = (slice + 3) & ~3;  // slices start on 16-byte boundaries of a 16-byte aligned row
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B) * nc, 1, 1);
    cfg.blockDim = dim3(kTyT, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = nc;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t err = cudaLaunchKernelEx(&cfg, typical_sampler_kernel, tokens, logits, V, slice, temperature,
                                         typical_p, seeds, offsets, status);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace pkv
