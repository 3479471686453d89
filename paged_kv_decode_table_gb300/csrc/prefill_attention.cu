// prefill_attention.cu -- chunked prefill over the paged cache: append a chunk
// of several new tokens per sequence through the block table, and the chunk's
// causal GQA attention over the cached prefix and the chunk itself.
//
// "Bai Lab tong hop -- Inference Engineering": the prefill of a prompt chunk
// starting at position lo reads the cached K/V through the table, runs the
// chunk, and writes the chunk's K/V back (KVPool.write); "Suy luan & Toi uu hoa
// (Inference)" 2.1: a prefill processes all its tokens in parallel; "LLM
// inference serving tutorial" 5.4: chunked prefill.  Sequence b appends n_b =
// q_start[b+1] - q_start[b] tokens (rows of the packed [T, Hkv, D] / [T, Hq, D]
// arrays); seq_lens[b] is the length after the append, so new token i sits at
// position L_b - n_b + i and attends to positions 0 .. L_b - n_b + i.
//
// Attention (bf16, D = 128, block_size a multiple of 16): one CTA per (tile of
// 16 chunk tokens of one sequence, KV head h), one warp per query head of the
// group.  A warp keeps its 16 query rows (tokens on M) in its own
// 128-byte-swizzled shared-memory tile and reads them as mma.sync A fragments
// with ldmatrix; the CTA streams head h's K and V in 32-key steps through a
// two-slot cp.async ring in shared memory (one step in flight while the other
// is used; rows past the tile's last position are zero-filled) shared by the G
// warps; S = Q K^T and O += P V by m16n8k16 bf16 MMAs with fp32 accumulation,
// causal mask and online softmax in the log2 domain.  Each K/V sub-tile is used
// by 16 tokens x G heads.  Up to 4 heads per group: 128-thread CTAs, four per
// SM; up to 8: 256 threads, two per SM (128 registers a thread either way).
#include <math.h>

#include "pkv_common.cuh"

namespace pkv {

constexpr int kPDim = 128;
constexpr int kPAppendWarps = 8;

// Sequence holding packed row t: the last b with q_start[b] <= t.
__device__ __forceinline__ int seq_of(const int32_t* q_start, int B, int t) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (q_start[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ------------------------------------------------------------------ chunk append
template <typename T>
__global__ void __launch_bounds__(kPAppendWarps * 32)
    kv_append_chunk_kernel(const T* __restrict__ k_new, const T* __restrict__ v_new, T* __restrict__ k_cache,
                           T* __restrict__ v_cache, const int32_t* __restrict__ block_tables, int max_blocks,
                           const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ q_start, int B,
                           int Hkv, int D, int BS, int NB, int vec_ok, int32_t* status) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * kPAppendWarps + warp;  // t * Hkv + h
    const int Tn = q_start[B];
    if (row >= static_cast<long long>(Tn) * Hkv) return;
    const int t = static_cast<int>(row / Hkv), h = static_cast<int>(row - static_cast<long long>(t) * Hkv);
    const int b = seq_of(q_start, B, t);
    const int n = q_start[b + 1] - q_start[b], L = seq_lens[b];
    if (L < n || static_cast<long long>(L) > static_cast<long long>(max_blocks) * BS) {
        if (lane == 0) report(status, PKV_ERR_DEVICE_BOUNDS);
        return;
    }
    const int pos = L - n + (t - q_start[b]);
    const int blk = block_tables[static_cast<size_t>(b) * max_blocks + pos / BS];
    if (blk < 0 || blk >= NB) {
        if (lane == 0) report(status, PKV_ERR_DEVICE_BOUNDS);
        return;
    }
    const long long dst = ((static_cast<long long>(blk) * Hkv + h) * BS + pos % BS) * D;
    const long long src = row * D;
    if (vec_ok) {
        const int nvec = D / (16 / static_cast<int>(sizeof(T)));
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

// ------------------------------------------------------------------ chunk attention
constexpr int kPBox = 16 * 128;      // one 64-dim half of a 16-row sub-tile, 128 B per row
constexpr int kPTile = 2 * kPBox;    // a K (or V) sub-tile: 16 rows x 128 dims bf16
constexpr int kPStage = 2 * kPTile;  // K and V
constexpr int kPRing = 2;            // pair slots (2 sub-tiles each): one pair in flight while one is used
constexpr int kPRingBytes = kPRing * 2 * kPStage;  // 32 KB, then each warp's 4 KB query tile
constexpr int kPTableWin = 512;  // block-table entries kept in shared memory at a time

// 2^x by the hardware's approximate base-2 exponential (P and the rescale
// factors of the online softmax, which are rounded to bf16 or only scale fp32
// accumulators).
__device__ __forceinline__ float ex2a(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int kThreads, int kMinBlocks>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
    prefill_attn_kernel(const __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ out,
                        const __nv_bfloat16* __restrict__ k_cache, const __nv_bfloat16* __restrict__ v_cache,
                        const int32_t* __restrict__ block_tables, int max_blocks, const int32_t* __restrict__ seq_lens,
                        const int32_t* __restrict__ q_start, int B, int Hq, int Hkv, int BS, int NB,
                        float scale_log2, int32_t* status) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the chunk's K/V appended, lengths final
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ __align__(1024) uint8_t ring[];  // kPRingBytes + 4 KB per warp
    __shared__ int s_b, s_tile, s_bad;
    __shared__ int tblk[kPTableWin];  // block ids of logical blocks win0 .. win0 + kPTableWin - 1
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nthr = blockDim.x;
    const int G = Hq / Hkv, h = blockIdx.y;
    if (tid == 0) {
        s_b = -1;
        s_tile = 0;
        s_bad = 0;
    }
    __syncthreads();
    if (warp == 0) {  // this CTA's tile: tiles of 16 chunk tokens, sequence after sequence
        int acc = 0;
        for (int base = 0; base < B; base += 32) {
            const int bb = base + lane;
            const int n = bb < B ? q_start[bb + 1] - q_start[bb] : 0;
            const int tiles = n > 0 ? (n + 15) >> 4 : 0;
            int inc = tiles;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            const int ex = acc + inc - tiles;
            const int x = static_cast<int>(blockIdx.x);
            if (tiles > 0 && ex <= x && x < ex + tiles) {
                s_b = bb;
                s_tile = x - ex;
            }
            acc += __shfl_sync(0xffffffffu, inc, 31);
            if (acc > x) break;
        }
    }
    __syncthreads();
    const int b = s_b, tile = s_tile;
    if (b < 0) return;  // a spare CTA of the upper-bound grid
    const int n = q_start[b + 1] - q_start[b], L = seq_lens[b];
    const int t0 = q_start[b] + 16 * tile, nt = min(16, n - 16 * tile);
    const int qh = h * G + warp;
    const int g = lane >> 2, r = lane & 3, mi = lane >> 3, rr = lane & 7;
    auto write_rows = [&](const float (&O)[16][4], float inv0, float inv1) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const int d = c * 8 + 2 * r;
            if (g < nt)
                *reinterpret_cast<uint32_t*>(out + (static_cast<size_t>(t0 + g) * Hq + qh) * kPDim + d) =
                    pack_bf16x2(O[c][0] * inv0, O[c][1] * inv0);
            if (g + 8 < nt)
                *reinterpret_cast<uint32_t*>(out + (static_cast<size_t>(t0 + g + 8) * Hq + qh) * kPDim + d) =
                    pack_bf16x2(O[c][2] * inv1, O[c][3] * inv1);
        }
    };
    float O[16][4];
#pragma unroll
    for (int c = 0; c < 16; ++c) O[c][0] = O[c][1] = O[c][2] = O[c][3] = 0.f;
    if (L < n || static_cast<long long>(L) > static_cast<long long>(max_blocks) * BS) {
        if (tid == 0) report(status, PKV_ERR_DEVICE_BOUNDS);
        write_rows(O, 0.f, 0.f);
        return;
    }
    const int p0 = L - n + 16 * tile;  // position of the tile's first token
    const int plast = p0 + nt - 1;
    const int nsub = plast / 16 + 1;   // 16-key sub-tiles covering positions 0 .. plast
    const int rpos0 = g < nt ? p0 + g : plast, rpos1 = g + 8 < nt ? p0 + g + 8 : plast;

    // this warp's query tile (16 tokens x 128 dims of head qh) in shared memory,
    // 128-byte-swizzled like the K tiles; rows past the chunk are zero
    // (q rows sit 256-byte multiples after q, so q's own alignment decides
    // between 16-byte loads and four 4-byte ones)
    uint8_t* qtile = ring + kPRingBytes + warp * 4096;
    const bool q16 = (reinterpret_cast<uintptr_t>(q) & 15u) == 0;
    for (int c = lane; c < 256; c += 32) {
        const int row = c >> 4, ch = c & 15;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < nt) {
            const __nv_bfloat16* src = q + (static_cast<size_t>(t0 + row) * Hq + qh) * kPDim + 8 * ch;
            if (q16) {
                v = __ldg(reinterpret_cast<const uint4*>(src));
            } else {
                const uint32_t* s4 = reinterpret_cast<const uint32_t*>(src);
                v = make_uint4(__ldg(s4), __ldg(s4 + 1), __ldg(s4 + 2), __ldg(s4 + 3));
            }
        }
        *reinterpret_cast<uint4*>(qtile + (ch >> 3) * kPBox + row * 128 + (((ch & 7) ^ (row & 7)) << 4)) = v;
    }
    __syncwarp();
    const uint32_t qtile_u32 = smem_u32(qtile);
    const uint32_t ring_u32 = smem_u32(ring);
    const int32_t* trow = block_tables + static_cast<size_t>(b) * max_blocks;
    // The block ids come from a window of the table in shared memory, so that
    // issuing a step's copies waits on no global load.  A step never spans more
    // than 3 logical blocks (32 keys, blocks of >= 16), so the window is moved
    // when the step's blocks would run past it.
    const int nblk_used = plast / BS + 1;
    int win0 = -kPTableWin;
    auto ensure_window = [&](int pr) {  // called by every thread with the same pr
        const int first = pr * 32 / BS, last = min(nblk_used - 1, (pr * 32 + 31) / BS);
        if (first >= win0 && last < win0 + kPTableWin) return;
        __syncthreads();  // nobody still reads the old window
        win0 = first;
        for (int i = tid; i < kPTableWin; i += nthr) tblk[i] = win0 + i < nblk_used ? trow[win0 + i] : -1;
        __syncthreads();
    };
    // a pair of 16-key sub-tiles (keys 32 * pr .. 32 * pr + 31) into slot st:
    // [sub-tile 0: K | V][sub-tile 1: K | V], 16 rows x 16 chunks of 16 bytes each
    auto load_pair = [&](int pr, int st) {
        // thread: 16-byte column ch of rows rsel, rsel + nthr/16, ... of the 32
        // rows (keys) of the step; K and V of a row share its block lookup
        const int ch = tid & 15;
        for (int row32 = tid >> 4; row32 < 32; row32 += nthr >> 4) {
            const int half = row32 >> 4, row = row32 & 15;
            const int pos = pr * 32 + row32;
            bool ok = pos <= plast;  // later keys are masked for every row of the tile
            int blk = 0;
            if (ok) {
                blk = tblk[pos / BS - win0];
                if (blk < 0 || blk >= NB) {
                    s_bad = 1;
                    ok = false;
                }
            }
            const size_t eoff = ok ? ((static_cast<size_t>(blk) * Hkv + h) * BS + pos % BS) * kPDim + ch * 8 : 0;
            const uint32_t dst = ring_u32 + (2 * st + half) * kPStage + (ch >> 3) * kPBox + row * 128 +
                                 (((ch & 7) ^ (row & 7)) << 4);
            cp_async16(dst, k_cache + eoff, ok ? 16 : 0);  // rows past the end (and bad blocks) are zero-filled
            cp_async16(dst + kPTile, v_cache + eoff, ok ? 16 : 0);
        }
        cp_async_commit();
    };
    // ring of kPRing pair slots: pair p lives in slot p % kPRing; one commit
    // group per pair (empty past the end), so that waiting for all but the
    // kPRing - 2 newest groups means pair p has landed
    const int npair = (nsub + 1) >> 1;
    for (int s0 = 0; s0 < kPRing - 1; ++s0) {
        if (s0 < npair) {
            ensure_window(s0);
            load_pair(s0, s0);
        } else {
            cp_async_commit();
        }
    }
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    for (int pr = 0; pr < npair; ++pr) {
        cp_async_wait<kPRing - 2>();
        __syncthreads();  // pair pr is in shared memory for every warp, and every
                          // warp is done with pair pr - 1, whose slot is refilled next
        if (pr + kPRing - 1 < npair) {
            ensure_window(pr + kPRing - 1);
            load_pair(pr + kPRing - 1, (pr + kPRing - 1) % kPRing);
        } else {
            cp_async_commit();
        }
        if (warp < G) {
            const uint32_t k0 = ring_u32 + (2 * (pr % kPRing)) * kPStage, k1 = k0 + kPStage;
            // ---- S = Q K^T for 32 keys: four independent n-tiles of 8
            float s[4][4];
#pragma unroll
            for (int t = 0; t < 4; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int row = (mi >> 1) * 8 + rr;
                const int dc = kk * 2 + (mi & 1);
                const uint32_t off = static_cast<uint32_t>(dc >> 3) * kPBox + static_cast<uint32_t>(row) * 128u +
                                     (static_cast<uint32_t>((dc & 7) ^ (row & 7)) << 4);
                // A fragments of the query tile: lane l reads row l % 16, 16-byte column 2 kk + l / 16
                const int qrow = lane & 15, qdc = kk * 2 + (lane >> 4);
                uint32_t qa[4];
                ldmatrix_x4(qa[0], qa[1], qa[2], qa[3],
                            qtile_u32 + static_cast<uint32_t>(qdc >> 3) * kPBox + static_cast<uint32_t>(qrow) * 128u +
                                (static_cast<uint32_t>((qdc & 7) ^ (qrow & 7)) << 4));
                uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
                ldmatrix_x4(b0, b1, b2, b3, k0 + off);
                ldmatrix_x4(c0, c1, c2, c3, k1 + off);
                mma_bf16_16816(s[0], qa, b0, b1);
                mma_bf16_16816(s[1], qa, b2, b3);
                mma_bf16_16816(s[2], qa, c0, c1);
                mma_bf16_16816(s[3], qa, c2, c3);
            }
            // causal mask: key position <= the row's position (only steps that
            // reach past the tile's first position need it)
            if (pr * 32 + 31 > p0) {
#pragma unroll
                for (int t = 0; t < 4; ++t)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int kp = pr * 32 + t * 8 + 2 * r + (e & 1);
                        const int rp = e < 2 ? rpos0 : rpos1;
                        s[t][e] = kp <= rp ? s[t][e] * scale_log2 : -INFINITY;
                    }
            } else {
#pragma unroll
                for (int t = 0; t < 4; ++t)
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[t][e] *= scale_log2;
            }
            float mx0 = fmaxf(fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1])),
                              fmaxf(fmaxf(s[2][0], s[2][1]), fmaxf(s[3][0], s[3][1])));
            float mx1 = fmaxf(fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3])),
                              fmaxf(fmaxf(s[2][2], s[2][3]), fmaxf(s[3][2], s[3][3])));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
            const float a0 = ex2a(m0 - mu0), a1 = ex2a(m1 - mu1);
            m0 = mn0;
            m1 = mn1;
            uint32_t pa[2][4];  // P for keys 0..15 and 16..31, A-fragment layout
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                pa[hh][0] = pack_bf16x2(ex2a(s[2 * hh][0] - mu0), ex2a(s[2 * hh][1] - mu0));
                pa[hh][2] = pack_bf16x2(ex2a(s[2 * hh + 1][0] - mu0), ex2a(s[2 * hh + 1][1] - mu0));
                pa[hh][1] = pack_bf16x2(ex2a(s[2 * hh][2] - mu1), ex2a(s[2 * hh][3] - mu1));
                pa[hh][3] = pack_bf16x2(ex2a(s[2 * hh + 1][2] - mu1), ex2a(s[2 * hh + 1][3] - mu1));
            }
            l0 = l0 * a0 + (((bf16_lo(pa[0][0]) + bf16_hi(pa[0][0])) + (bf16_lo(pa[0][2]) + bf16_hi(pa[0][2]))) +
                            ((bf16_lo(pa[1][0]) + bf16_hi(pa[1][0])) + (bf16_lo(pa[1][2]) + bf16_hi(pa[1][2]))));
            l1 = l1 * a1 + (((bf16_lo(pa[0][1]) + bf16_hi(pa[0][1])) + (bf16_lo(pa[0][3]) + bf16_hi(pa[0][3]))) +
                            ((bf16_lo(pa[1][1]) + bf16_hi(pa[1][1])) + (bf16_lo(pa[1][3]) + bf16_hi(pa[1][3]))));
            if (a0 != 1.f || a1 != 1.f) {  // the running maximum moved: rescale
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    O[c][0] *= a0;
                    O[c][1] *= a0;
                    O[c][2] *= a1;
                    O[c][3] *= a1;
                }
            }
            // ---- O += P V over the 32 keys
#pragma unroll
            for (int dp = 0; dp < 8; ++dp) {
                const int row = (mi & 1) * 8 + rr;
                const int dc = dp * 2 + (mi >> 1);
                const uint32_t off = kPTile + static_cast<uint32_t>(dc >> 3) * kPBox + static_cast<uint32_t>(row) * 128u +
                                     (static_cast<uint32_t>((dc & 7) ^ (row & 7)) << 4);
                uint32_t v0, v1, v2, v3, w0, w1, w2, w3;
                ldmatrix_x4_trans(v0, v1, v2, v3, k0 + off);
                ldmatrix_x4_trans(w0, w1, w2, w3, k1 + off);
                mma_bf16_16816(O[2 * dp], pa[0], v0, v1);
                mma_bf16_16816(O[2 * dp + 1], pa[0], v2, v3);
                mma_bf16_16816(O[2 * dp], pa[1], w0, w1);
                mma_bf16_16816(O[2 * dp + 1], pa[1], w2, w3);
            }
        }
    }
    cp_async_wait<0>();
    if (warp >= G) return;
    float t0l = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
    t0l += __shfl_xor_sync(0xffffffffu, t0l, 2);
    float t1l = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
    t1l += __shfl_xor_sync(0xffffffffu, t1l, 2);
    if (s_bad) {
        if (lane == 0) report(status, PKV_ERR_DEVICE_BOUNDS);
        write_rows(O, 0.f, 0.f);
        return;
    }
    write_rows(O, t0l > 0.f ? 1.f / t0l : 0.f, t1l > 0.f ? 1.f / t1l : 0.f);
}

// ------------------------------------------------------------------ host side
cudaError_t launch_kv_append_chunk(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                   const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                                   const int32_t* q_start, int B, int T_new, int Hkv, int D, int BS, int NB,
                                   pkv_dtype dtype, int32_t* status, cudaStream_t stream) {
    const size_t es = dtype == PKV_F32 ? 4 : 2;
    auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const int vec_ok = ((D * es) % 16 == 0) && aligned16(k_new) && aligned16(v_new) && aligned16(k_cache) &&
                       aligned16(v_cache);
    const long long rows = static_cast<long long>(T_new) * Hkv;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + kPAppendWarps - 1) / kPAppendWarps), 1, 1);
    cfg.blockDim = dim3(kPAppendWarps * 32, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err;
    if (dtype == PKV_F32)
        err = cudaLaunchKernelEx(&cfg, kv_append_chunk_kernel<float>, static_cast<const float*>(k_new),
                                 static_cast<const float*>(v_new), static_cast<float*>(k_cache),
                                 static_cast<float*>(v_cache), block_tables, max_blocks, seq_lens, q_start, B, Hkv, D,
                                 BS, NB, vec_ok, status);
    else
        err = cudaLaunchKernelEx(&cfg, kv_append_chunk_kernel<__nv_bfloat16>,
                                 static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new),
                                 static_cast<__nv_bfloat16*>(k_cache), static_cast<__nv_bfloat16*>(v_cache),
                                 block_tables, max_blocks, seq_lens, q_start, B, Hkv, D, BS, NB, vec_ok, status);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

// Grid: an upper bound on the tiles (sum over b of ceil(n_b / 16) <= T_new / 16 + B)
// times the KV heads; spare CTAs exit at once.
cudaError_t launch_prefill_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                                     const int32_t* q_start, int B, int T_new, int Hq, int Hkv, int BS, int NB,
                                     float scale, int32_t* status, cudaStream_t stream) {
    const long long tiles = static_cast<long long>(T_new) / 16 + B;
    if (tiles > 0x7fffffffLL || Hkv > 65535) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles), static_cast<unsigned>(Hkv), 1);
    cfg.blockDim = dim3(static_cast<unsigned>(32 * (Hq / Hkv)), 1, 1);
    const int G = Hq / Hkv;
    const int smem = kPRingBytes + 4096 * G;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    // up to 4 query heads per KV head: 128-thread CTAs, four per SM; else 256 threads, two per SM
    auto kern = G <= 4 ? prefill_attn_kernel<128, 4> : prefill_attn_kernel<256, 2>;
    cudaError_t aerr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (aerr != cudaSuccess) return aerr;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float scale_log2 = scale * 1.4426950408889634f;
    cudaError_t err = cudaLaunchKernelEx(&cfg, kern, static_cast<const __nv_bfloat16*>(q),
                                         static_cast<__nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(k_cache),
                                         static_cast<const __nv_bfloat16*>(v_cache), block_tables, max_blocks,
                                         seq_lens, q_start, B, Hq, Hkv, BS, NB, scale_log2, status);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace pkv
