// prefill_tc.cu -- chunked-prefill attention on the fifth-generation tensor
// cores: tcgen05 MMAs with accumulators in tensor memory (TMEM), operands
// staged in shared memory by TMA.  Same results as prefill_attn_kernel (the
// chunk's causal GQA attention over the paged cache; "Suy luan & Toi uu hoa
// (Inference)" 2.1 and 4.1, the lab's prefill step, "LLM inference serving
// tutorial" 5.4) for bf16, D = 128, G = Hq / Hkv from 1 to 8, block_size a
// multiple of 16 and 16-byte aligned q / out / pools.
//
//  * One CTA per (two query tiles of 128 rows, KV head h).  Row r of query
//    tile t is (chunk token t TQ + r / G, query head h G + r % G), TQ =
//    floor(128 / G): 2 TQ consecutive tokens of one sequence times the G heads
//    that share K/V head h, so each K/V tile serves up to 256 rows (rows TQ G
//    .. 127 of a tile, when G does not divide 128, are padding: computed on
//    zero queries and not stored).  The CTAs take the chunk tiles
//    longest first (by the number of key tiles they read; the KV head is the
//    innermost grid index), so that the longest start in the first wave.
//  * K and V of head h stream in 64-key tiles through a five-stage ring.  The
//    paged layout allows TMA boxes of one block's 16 keys at most.  K comes in
//    one 4 KB box per 16 keys through a 4-D view of the pool that lands the
//    two 64-dimension halves interleaved at 1 KB, so that for either half the
//    8-row groups of the tile sit 2 KB apart (one N = 64 MMA per k-step); V in
//    one 4 KB box per 16 keys (a 3-D view, both halves, one box per PV k-step).
//    Three producer warps issue a tile's eight boxes, each on its own (its
//    own window of the block table in shared memory, its own arrival on the
//    stage's barrier).  Each CTA walks its key tiles starting at a different
//    tile, so that the CTAs sharing a sequence do not read the same blocks at
//    the same time.
//  * Tensor memory, per query tile t (256 columns): Q (bf16, two per column)
//    at 256 t, S at 256 t + 64, O at 256 t + 128.  One warp issues
//    S = Q K^T (M 128, N 64, K 128; A = Q from tensor memory, B = K from the
//    stage), another O += P V (M 128, N 128, K 64; A = P from a K-major,
//    128-byte-swizzled shared tile per query tile, B = V as stored, MN-major,
//    one 16-key group per k-step).  The softmax releases S as soon as it has
//    read it, so S of tile j + 1 runs during the softmax of tile j; P of tile
//    j + 1 is written once the PV of tile j is complete.  The two query tiles
//    interleave on the tensor pipe.  Completion is signalled through
//    mbarriers (tcgen05.commit).
//  * Eight softmax warps, four per query tile: thread r owns row r (TMEM lane
//    r).  It reads its 64 scores (tcgen05.ld), applies the causal mask and the
//    scale in the log2 domain, and exponentiates against a reference maximum
//    that is raised only when the row maximum exceeds it by more than 8, in
//    which case the row of O in TMEM and the running sum are rescaled first;
//    P (bf16, values at most 2^8) goes to shared memory for the PV MMA, and
//    the sum accumulates the fp32 values.  Rows past the chunk are
//    computed on zero queries and not stored.  The V rows of keys at or past
//    the sequence length (which may hold anything, NaN included) are cleared
//    before the last PV MMAs.
//  * Epilogue: O / sum from TMEM to the bf16 output rows.
// Every mbarrier wait is bounded; a CTA that gives up records PKV_ERR_TIMEOUT,
// waits (bounded) for its own TMA copies, and still frees its TMEM.
#include <cuda.h>
#include <math.h>

#include "pkv_common.cuh"

namespace pkv {

bool encode_pool_box_halves(CUtensorMap* map, const void* pool, int NB, int Hkv, int BS, int box_rows);

constexpr int kTcDim = 128;
constexpr int kTcRows = 128;                 // query rows per query tile (TMEM lanes)
constexpr int kTcQT = 2;                     // query tiles per CTA, sharing every K/V tile
constexpr int kTcKeys = 64;                  // keys per tile
constexpr int kTcStages = 5;                 // K/V ring depth
constexpr int kTcPBytes = kTcRows * kTcKeys * 2;          // 16 KB: P of one query tile, one atom of 128 rows
constexpr int kTcKBytes = kTcKeys * kTcDim * 2;           // 16 KB per operand tile
constexpr int kTcGroupBytes = 16 * kTcDim * 2;            // 4 KB: 16 keys x 128 dimensions
constexpr int kTcStageBytes = 2 * kTcKBytes;              // K then V
constexpr int kTcProd = 3;                   // producer warps
constexpr int kTcWin = 640;                  // block-table entries kept in shared memory, per producer warp
// warps 0-7: softmax (warp w: query tile w / 4, TMEM lanes 32 (w % 4) ..); warps 8,
// 11 and 12: producers; warp 9: S MMAs (and the TMEM allocation); warp 10: PV MMAs
constexpr int kTcWarpProd = 8, kTcWarpS = 9, kTcWarpPV = 10;
constexpr int kTcThreads = 13 * 32;
constexpr int kTcTmemCols = 512;             // query tile t: Q at 256 t, S at 256 t + 64, O at 256 t + 128

struct TcSmem {  // follows the 1024-aligned operand area
    uint64_t kv_full[kTcStages], kv_empty[kTcStages];
    uint64_t s_full[kTcQT], s_free[kTcQT], p_full[kTcQT], o_done[kTcQT];
    uint32_t tmem_base;
    int b, tile, bad;
    int tbl[kTcProd][kTcWin];
};
constexpr size_t kTcOperandBytes = kTcQT * static_cast<size_t>(kTcPBytes) + kTcStages * static_cast<size_t>(kTcStageBytes);
constexpr size_t kTcSmemBytes = 1024 + kTcOperandBytes + sizeof(TcSmem);
static_assert(kTcSmemBytes <= 227 * 1024, "shared memory of one CTA");

// ------------------------------------------------------------------ tcgen05 helpers
// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// byte offset (K-major: unused; MN-major: the stride between 64-element atoms
// along M / N), stride byte offset (the stride between groups of 8 rows), the
// descriptor version of this architecture.
__device__ __forceinline__ uint64_t tc_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: bf16 A and B, fp32 accumulator, M x N,
// B K-major or MN-major (A always K-major here).
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// The same with A (M x 16 bf16, row m in TMEM lane m, two elements per column) in tensor memory.
__device__ __forceinline__ void tc_mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// Arrive on bar once every tcgen05 operation this thread issued so far is complete.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 32 consecutive columns of this thread's TMEM lane (warp w reads lanes 32 (w % 4) ..).
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Byte offset of (row, 16-byte chunk) in a tile of 128-byte rows with the
// 128-byte swizzle (the chunk index XOR the row's low three bits).
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
    return static_cast<uint32_t>(row) * 128u + (static_cast<uint32_t>(chunk ^ (row & 7)) << 4);
}
// 4-D tiled copy (the K boxes); x, y, z, w are the box's start coordinates.
__device__ __forceinline__ void tma_load_4d(void* smem_dst, const void* tmap, int x, int y, int z, int w,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
        : "memory");
}
// max(a, b, c) in one instruction
__device__ __forceinline__ float tc_max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// (x0, x1) = (a0 b + c, a1 b + c) and (s0, s1) += (a0, a1) as paired fp32 operations
__device__ __forceinline__ void tc_fma2(float& x0, float& x1, float a0, float a1, float b, float c) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %4};\n\tmov.b64 rc, {%5, %5};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(x0), "=f"(x1)
        : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
__device__ __forceinline__ void tc_add2(float& s0, float& s1, float a0, float a1) {
    asm("{\n\t.reg .b64 ra, rs;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rs, {%0, %1};\n\t"
        "add.rn.f32x2 rs, rs, ra;\n\tmov.b64 {%0, %1}, rs;\n\t}"
        : "+f"(s0), "+f"(s1)
        : "f"(a0), "f"(a1));
}
__device__ __forceinline__ float tc_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ int warp_sum_i(int x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ int warp_max_i(int x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
// Chunk tiles of one sequence (n chunk tokens, length L after the chunk, TC
// tokens per tile) that read more than v key tiles.  Full tile c reads up to
// position L - n + TC (c + 1) - 1, the last tile up to L - 1; the count grows
// with c.  L below n (an invalid length, reported by the CTA that owns the
// tile) is taken as n, so that the order is defined for any input.
__device__ __forceinline__ int tc_tiles_longer(int n, int L, int TC, int v) {
    if (n <= 0) return 0;
    const int tiles = (n + TC - 1) / TC;
    const long long Lc = max(L, n), P = Lc - n;
    int cnt = (Lc - 1) / kTcKeys + 1 > v ? 1 : 0;
    const long long x = static_cast<long long>(kTcKeys) * v - P + 1;  // full tile c qualifies iff TC (c + 1) >= x
    const long long cmin = x <= 0 ? 0 : (x + TC - 1) / TC - 1;
    cnt += static_cast<int>(max(0LL, static_cast<long long>(tiles - 1) - cmin));
    return cnt;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ out,
                      const int32_t* __restrict__ block_tables, int max_blocks, const int32_t* __restrict__ seq_lens,
                      const int32_t* __restrict__ q_start, int B, int Hq, int Hkv, int BS, int NB, float scale_log2,
                      int32_t* status) {
    extern __shared__ uint8_t tc_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sP = base;                          // P of query tile t at t kTcPBytes
    uint8_t* sKV = base + kTcQT * kTcPBytes;
    TcSmem* sm = reinterpret_cast<TcSmem*>(base + kTcOperandBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = Hq / Hkv, h = static_cast<int>(blockIdx.x) % Hkv;
    const int TQ = kTcRows / G;    // chunk tokens per query tile (rows TQ G .. 127 are padding)
    const int TC = kTcQT * TQ;     // chunk tokens per CTA

    // ---- prologue, independent of the inputs
    if (tid == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&sm->kv_full[s], kTcProd);  // one arrival (with its bytes) per producer warp
            mbar_init(&sm->kv_empty[s], 1);
        }
        for (int t = 0; t < kTcQT; ++t) {
            mbar_init(&sm->s_full[t], 1);
            mbar_init(&sm->s_free[t], kTcRows);
            mbar_init(&sm->p_full[t], kTcRows);
            mbar_init(&sm->o_done[t], 1);
        }
        fence_mbar_init();
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        sm->b = -1;
        sm->tile = 0;
        sm->bad = 0;
    }
    if (warp == kTcWarpS) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&sm->tmem_base)),
                     "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the chunk's K/V are in the cache
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        // This CTA's chunk tile: the one of rank k when the chunk tiles of all
        // sequences are ordered by their number of key tiles, longest first (ties:
        // sequence order, then tile order), so that the longest start in the first
        // wave.  v = the rank's key-tile count, found by bisection on the counts.
        const int k = static_cast<int>(blockIdx.x) / Hkv;
        int total = 0, vmax = 0;
        for (int b0 = 0; b0 < B; b0 += 32) {
            const int bb = b0 + lane;
            if (bb < B) {
                const int n = q_start[bb + 1] - q_start[bb];
                if (n > 0) {
                    total += (n + TC - 1) / TC;
                    vmax = max(vmax, (max(seq_lens[bb], n) - 1) / kTcKeys + 1);
                }
            }
        }
        total = warp_sum_i(total);
        vmax = warp_max_i(vmax);
        if (k < total) {
            auto longer = [&](int v) {  // chunk tiles (all sequences) with more than v key tiles
                int c = 0;
                for (int bb = lane; bb < B; bb += 32) c += tc_tiles_longer(q_start[bb + 1] - q_start[bb], seq_lens[bb], TC, v);
                return warp_sum_i(c);
            };
            int lo = 1, hi = vmax;  // the smallest v with longer(v) <= k
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (longer(mid) <= k) hi = mid;
                else lo = mid + 1;
            }
            const int v = lo;
            int idx = k - longer(v);  // among the tiles with exactly v key tiles, in sequence order
            for (int b0 = 0; b0 < B; b0 += 32) {
                const int bb = b0 + lane;
                int e = 0, first = 0;
                if (bb < B) {
                    const int n = q_start[bb + 1] - q_start[bb], L = seq_lens[bb];
                    const int ge = tc_tiles_longer(n, L, TC, v - 1);
                    e = ge - tc_tiles_longer(n, L, TC, v);
                    first = (n > 0 ? (n + TC - 1) / TC : 0) - ge;  // the counts grow along the chunk
                }
                int inc = e;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, inc, o);
                    if (lane >= o) inc += y;
                }
                const int ex = inc - e;
                if (e > 0 && ex <= idx && idx < inc) {
                    sm->b = bb;
                    sm->tile = first + (idx - ex);
                }
                const int tot = __shfl_sync(0xffffffffu, inc, 31);
                if (idx < tot) break;
                idx -= tot;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm->tmem_base;
    const int b = sm->b, tile = sm->tile;
    bool active = b >= 0;  // a spare CTA of the upper-bound grid has no tile
    int n = 0, L = 0, t0 = 0, nt = 0, p0 = 0;
    if (active) {
        n = q_start[b + 1] - q_start[b];
        L = seq_lens[b];
        t0 = q_start[b] + TC * tile;
        nt = min(TC, n - TC * tile);
        p0 = L - n + TC * tile;  // position of the CTA's first token
    }
    const bool bad_len = active && (L < n || static_cast<long long>(L) > static_cast<long long>(max_blocks) * BS);
    // this thread's row (softmax warps): query tile qt, row r = token tl of the CTA, query head qh
    const bool softmax_warp = warp < 4 * kTcQT;
    const int qt = warp >> 2, r = tid & (kTcRows - 1);
    const int tl = qt * TQ + r / G, qh = h * G + r % G;
    const bool row_valid = active && softmax_warp && r < TQ * G && tl < nt;  // rows TQ G .. 127: padding
    if (bad_len) {
        if (tid == 0) report(status, PKV_ERR_DEVICE_BOUNDS);
        if (row_valid) {
            uint4* o = reinterpret_cast<uint4*>(out + (static_cast<size_t>(t0 + tl) * Hq + qh) * kTcDim);
            for (int c = 0; c < 16; ++c) o[c] = make_uint4(0u, 0u, 0u, 0u);
        }
        active = false;
    }
    const int plast = p0 + nt - 1;                    // the CTA's last position (keys 0 .. plast are read)
    const int ntiles = active ? plast / kTcKeys + 1 : 0;
    // iteration j handles key tile (j + rot) mod ntiles (any order gives the same softmax)
    const int rot = ntiles > 0 ? static_cast<int>((blockIdx.x * 13u) % static_cast<unsigned>(ntiles)) : 0;
    const int nblk_used = active ? plast / BS + 1 : 0;
    const int pos = row_valid ? p0 + tl : plast;      // the row's position (rows past the chunk: the last)

    // ---- the query tiles: row r of tile qt into TMEM lane r, columns 256 qt .. + 63 (two
    // bf16 per column; rows past the chunk: zeros), the A operand of S = Q K^T
    if (active && softmax_warp) {
        const uint4* src = reinterpret_cast<const uint4*>(q + (static_cast<size_t>(t0 + (row_valid ? tl : 0)) * Hq + qh) * kTcDim);
        const uint32_t lrow = static_cast<uint32_t>((warp & 3) * 32) << 16;
#pragma unroll
        for (int hv = 0; hv < 2; ++hv) {
            uint32_t w[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 v = row_valid ? __ldg(src + 8 * hv + c) : make_uint4(0u, 0u, 0u, 0u);
                w[4 * c] = v.x;
                w[4 * c + 1] = v.y;
                w[4 * c + 2] = v.z;
                w[4 * c + 3] = v.w;
            }
            tc_st32(tmem + 256 * qt + lrow + 32 * hv, w);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    bool fail = false;
    if ((warp == kTcWarpProd || warp > kTcWarpPV) && active) {
        // ------------------------------------------------ producer warps 8, 11, 12
        // The three warps work independently: warp pw issues boxes i = pw, pw + 3,
        // pw + 6 of every tile (box i: K of 16-key group i for i < 4, V of group
        // i - 4 otherwise), with block ids from its own window of the block table;
        // it waits for the stage itself and arms the stage's transaction count
        // with its own bytes (the stage's full barrier expects one arrival per
        // producer warp), so one warp's bookkeeping overlaps the others' copies.
        const int pw = warp == kTcWarpProd ? 0 : warp - kTcWarpPV;
        const int nbox = pw < 2 ? 3 : 2;  // boxes of this warp per tile
        int* tbl = sm->tbl[pw];
        const int32_t* trow = block_tables + static_cast<size_t>(b) * max_blocks;
        int win0 = -kTcWin;
        for (int j = 0; j < ntiles && !fail; ++j) {
            const int s = j % kTcStages;
            const int kt = j + rot < ntiles ? j + rot : j + rot - ntiles;
            const int kb0 = (kt * kTcKeys) / BS, kb1 = min(nblk_used - 1, (kt * kTcKeys + kTcKeys - 1) / BS);
            if (kb0 < win0 || kb1 >= win0 + kTcWin) {  // move this warp's window of the block table
                __syncwarp();
                win0 = kb0;
                for (int i = lane; i < kTcWin; i += 32) tbl[i] = win0 + i < nblk_used ? trow[win0 + i] : 0;
                __syncwarp();
            }
            if (lane == 0 && !mbar_wait(&sm->kv_empty[s], ((j / kTcStages) & 1) ^ 1)) {
                report(status, PKV_ERR_TIMEOUT);
                fail = true;
            }
            fail = __shfl_sync(0xffffffffu, fail, 0);
            if (fail) break;
            const int bi = pw + 3 * lane;
            int row = 0;
            if (lane < nbox) {  // the pool row of box bi's first key
                const int key0 = kt * kTcKeys + 16 * (bi & 3);
                const int kb = key0 / BS;
                int blk = 0, slot = 0;
                if (kb < nblk_used) {  // later keys: any valid rows (masked; their V rows are cleared)
                    blk = tbl[kb - win0];
                    slot = key0 - kb * BS;
                    if (blk < 0 || blk >= NB) {
                        sm->bad = 1;
                        report(status, PKV_ERR_DEVICE_BOUNDS);
                        blk = 0;
                    }
                }
                row = (blk * Hkv + h) * BS + slot;
            }
            if (lane == 0) mbar_arrive_expect_tx(&sm->kv_full[s], nbox * kTcGroupBytes);
            __syncwarp();  // the arrival precedes this warp's copies
            if (lane < nbox) {
                uint8_t* st = sKV + static_cast<size_t>(s) * kTcStageBytes;
                if (bi < 4)  // K of group bi: [8-row half][64-dimension half][8 rows][128 B]
                    tma_load_4d(st + kTcGroupBytes * bi, &tmK, 0, 0, 0, row >> 3, &sm->kv_full[s]);
                else  // V of group bi - 4: [64-dimension half][16 rows][128 B]
                    tma_load_3d(st + kTcKBytes + kTcGroupBytes * (bi - 4), &tmV, 0, row, 0, &sm->kv_full[s]);
            }
            __syncwarp();
        }
        // no copy of this CTA may still be in flight when it exits
        if (lane == 0)
            for (int j = max(0, ntiles - kTcStages); j < ntiles; ++j)
                mbar_wait(&sm->kv_full[j % kTcStages], (j / kTcStages) & 1);
    } else if (warp == kTcWarpS && active) {
        // ------------------------------------------------ S = Q K^T for both query tiles (lane 0 issues)
        // Q (A) from tensor memory, K (B) from the stage.  S_j of query tile t
        // overwrites S_{j-1} once the softmax has read it, so it runs while the
        // softmax works on tile j - 1.
        if (lane == 0) {
            constexpr uint32_t idS = tc_idesc(kTcRows, kTcKeys, false);
            const uint32_t kva = smem_u32(sKV);
            for (int j = 0; j < ntiles && !fail; ++j) {
                const int s = j % kTcStages;
                if (!mbar_wait(&sm->kv_full[s], (j / kTcStages) & 1)) {
                    fail = true;
                    break;
                }
                const uint32_t kb = kva + s * kTcStageBytes;
                for (int t = 0; t < kTcQT; ++t) {
                    if (j >= 1 && !mbar_wait(&sm->s_free[t], (j - 1) & 1)) {
                        fail = true;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kTcDim / 16; ++kk)
                        tc_mma_ta(tmem + 256 * t + 64, tmem + 256 * t + 8 * kk,
                                  tc_desc(kb + (kk >> 2) * 1024 + 32 * (kk & 3), 16, 2048), idS, kk > 0 ? 1u : 0u);
                    tc_commit(&sm->s_full[t]);
                }
            }
            if (fail) report(status, PKV_ERR_TIMEOUT);
        }
        __syncwarp();
    } else if (warp == kTcWarpPV && active) {
        // ------------------------------------------------ O += P V for both query tiles (lane 0 issues)
        // P of query tile t (bf16, a K-major 128-byte-swizzled shared tile) is
        // the A operand.  Both P tiles of key tile j were written after the
        // softmax read S_j, so once their PV MMAs are complete nothing reads the
        // stage any more.
        if (lane == 0) {
            constexpr uint32_t idO = tc_idesc(kTcRows, kTcDim, true);
            const uint32_t pa = smem_u32(sP), kva = smem_u32(sKV);
            for (int j = 0; j < ntiles && !fail; ++j) {
                const int s = j % kTcStages;
                const uint32_t vb = kva + s * kTcStageBytes + kTcKBytes;
                for (int t = 0; t < kTcQT; ++t) {  // query tile 0 first: its softmax warps clear V rows past L
                    if (!mbar_wait(&sm->p_full[t], j & 1)) {
                        fail = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t pb = pa + t * kTcPBytes;
#pragma unroll
                    for (int kk = 0; kk < kTcKeys / 16; ++kk)
                        tc_mma(tmem + 256 * t + 128, tc_desc(pb + 32 * kk, 16, 1024),
                               tc_desc(vb + kTcGroupBytes * kk, kTcGroupBytes / 2, 1024), idO,
                               (j > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(&sm->o_done[t]);
                }
                if (!fail) tc_commit(&sm->kv_empty[s]);
            }
            if (fail) report(status, PKV_ERR_TIMEOUT);
        }
        __syncwarp();
    } else if (softmax_warp && active) {
        // ------------------------------------------------ softmax warps: thread r of query tile qt owns row r
        const uint32_t lrow = static_cast<uint32_t>((warp & 3) * 32) << 16;  // this warp's TMEM lanes
        const uint32_t tq = tmem + 256 * qt;
        const int p0t = p0 + qt * TQ;  // the query tile's first position
        float m_ref = -INFINITY, lsum = 0.f;
        for (int j = 0; j < ntiles; ++j) {
            if (!__all_sync(0xffffffffu, mbar_wait(&sm->s_full[qt], j & 1))) {  // tcgen05.ld needs the whole warp
                fail = true;
                break;
            }
            tc_fence_after();
            uint32_t sr[2][32];
            tc_ld32(tq + lrow + 64, sr[0]);
            tc_ld32(tq + lrow + 96, sr[1]);
            tc_fence_before();
            mbar_arrive(&sm->s_free[qt]);  // S may take the next tile
            const int kt = j + rot < ntiles ? j + rot : j + rot - ntiles;
            const int kbase = kt * kTcKeys;
            // maximum of the raw scores (the scale is positive), eight chains;
            // the causal mask only on tiles that reach past the query tile's first position
            // (three-input maxima: two scores per instruction, four chains)
            float mxs[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) mxs[k] = -INFINITY;
            if (kbase + kTcKeys - 1 > p0t) {
#pragma unroll
                for (int c = 0; c < kTcKeys; ++c) {
                    const float v = kbase + c <= pos ? __uint_as_float(sr[c >> 5][c & 31]) : -INFINITY;
                    sr[c >> 5][c & 31] = __float_as_uint(v);
                }
            }
#pragma unroll
            for (int c = 0; c < kTcKeys; c += 2)
                mxs[(c >> 1) & 3] = tc_max3(mxs[(c >> 1) & 3], __uint_as_float(sr[c >> 5][c & 31]),
                                            __uint_as_float(sr[(c + 1) >> 5][(c + 1) & 31]));
            const float mx = fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])) * scale_log2;
            // the reference maximum moves only when the row maximum passes it by more than 8
            const float m_new = mx > m_ref + 8.f ? mx : m_ref;
            const bool resc = m_new != m_ref;
            const float a = resc ? tc_ex2(m_ref - m_new) : 1.f;
            m_ref = m_new;
            const float nmu = m_ref == -INFINITY ? 0.f : -m_ref;
            // P = 2^(s scale - m_ref) (masked scores give 0), the sum in four chains of
            // pairs (the scale, the offset and the sum as paired fp32 operations)
            uint32_t pk[kTcKeys / 2];
            float ls[4][2];
#pragma unroll
            for (int k = 0; k < 4; ++k) ls[k][0] = ls[k][1] = 0.f;
#pragma unroll
            for (int c = 0; c < kTcKeys / 2; ++c) {
                float t0, t1;
                tc_fma2(t0, t1, __uint_as_float(sr[(2 * c) >> 5][(2 * c) & 31]),
                        __uint_as_float(sr[(2 * c + 1) >> 5][(2 * c + 1) & 31]), scale_log2, nmu);
                const float e0 = tc_ex2(t0), e1 = tc_ex2(t1);
                pk[c] = pack_bf16x2(e0, e1);
                tc_add2(ls[c & 3][0], ls[c & 3][1], e0, e1);
            }
            lsum = lsum * a + (((ls[0][0] + ls[0][1]) + (ls[1][0] + ls[1][1])) +
                               ((ls[2][0] + ls[2][1]) + (ls[3][0] + ls[3][1])));
            // the PV of tile j - 1 is complete: O may be rescaled and the P tile rewritten
            if (j > 0) {
                if (!__all_sync(0xffffffffu, mbar_wait(&sm->o_done[qt], (j - 1) & 1))) {
                    fail = true;
                    break;
                }
                tc_fence_after();
            }
            if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
                for (int cc = 0; cc < kTcDim / 32; ++cc) {
                    uint32_t o[32];
                    tc_ld32(tq + lrow + 128 + 32 * cc, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
                    tc_st32(tq + lrow + 128 + 32 * cc, o);
                }
            }
            if (qt == 0 && kt == ntiles - 1) {  // the V rows of keys at or past L may hold anything: clear them
                const int rlo = max(0, min(kTcKeys, L - kbase));
                uint8_t* vb = sKV + static_cast<size_t>(j % kTcStages) * kTcStageBytes + kTcKBytes;
                for (int idx = r; idx < (kTcKeys - rlo) * 16; idx += kTcRows) {
                    const int rr = rlo + (idx >> 4), half = (idx >> 3) & 1, ch = idx & 7;
                    *reinterpret_cast<uint4*>(vb + kTcGroupBytes * (rr >> 4) + half * (kTcGroupBytes / 2) +
                                              (rr & 15) * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // P row r (64 bf16 = 8 chunks of 16 bytes) into the K-major P tile of query tile qt
            uint8_t* pbuf = sP + qt * kTcPBytes;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                *reinterpret_cast<uint4*>(pbuf + sw128(r, ch)) =
                    make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
            fence_proxy_async_smem();  // P and the cleared V rows, for the PV MMA
            tc_fence_before();
            mbar_arrive(&sm->p_full[qt]);
        }
        // ---- epilogue: O / sum of the last PV
        if (!fail && ntiles > 0 &&
            !__all_sync(0xffffffffu, mbar_wait(&sm->o_done[qt], (ntiles - 1) & 1)))
            fail = true;
        if (fail) {
            if (lane == 0) report(status, PKV_ERR_TIMEOUT);
        } else {
            tc_fence_after();
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            const bool store = row_valid && !sm->bad;
            uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(t0 + (row_valid ? tl : 0)) * Hq + qh) * kTcDim);
#pragma unroll 1
            for (int cc = 0; cc < kTcDim / 32; ++cc) {
                uint32_t o[32];
                tc_ld32(tq + lrow + 128 + 32 * cc, o);
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
                if (row_valid) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dst[4 * cc + k] = store ? make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3])
                                                : make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
    }
    // ---- every role is done with TMEM
    tc_fence_before();
    __syncthreads();
    if (warp == kTcWarpS) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols)
                     : "memory");
    }
}

// The K pool [NB, Hkv, BS, 128] bf16 in four dimensions: (64 elements, 8 rows,
// the two 64-element halves of a row, groups of 8 rows), with boxes of
// 64 x 8 x 2 x 2.  One box holds 16 consecutive rows and lands as
// [8-row group][half][8 rows][128 B]: for either half, successive 8-row groups
// sit 2048 bytes apart, so a 64-key tile of four boxes is one K-major,
// 128-byte-swizzled operand per half with a 2048-byte group stride.
static bool encode_pool_k16(CUtensorMap* map, const void* pool, int NB, int Hkv, int BS) {
    typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static EncodeFn enc = nullptr;
    static bool tried = false;
    if (!tried) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qres) ==
                cudaSuccess &&
            qres == cudaDriverEntryPointSuccess)
            enc = reinterpret_cast<EncodeFn>(p);
        tried = true;
    }
    const cuuint64_t rows = static_cast<cuuint64_t>(NB) * Hkv * BS;
    if (!enc || rows % 8 != 0) return false;
    cuuint64_t gdim[4] = {64, 8, 2, rows / 8};
    cuuint64_t gstride[3] = {kTcDim * 2, 128, 8 * kTcDim * 2};
    cuuint32_t box[4] = {64, 8, 2, 2};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool prefill_tc_supported(int Hq, int Hkv, int D, int BS, const void* q, const void* out, const void* k,
                          const void* v) {
    const int G = Hkv > 0 ? Hq / Hkv : 0;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    return D == kTcDim && BS % 16 == 0 && G >= 1 && G <= 8 && Hq == G * Hkv && a16(q) && a16(out) && a16(k) &&
           a16(v);
}

cudaError_t launch_prefill_tc(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                              const int32_t* q_start, int B, int T_new, int Hq, int Hkv, int BS, int NB, float scale,
                              int32_t* status, cudaStream_t stream) {
    const int G = Hq / Hkv, TC = kTcQT * (kTcRows / G);
    const long long tiles = static_cast<long long>(T_new) / TC + B;
    if (tiles * Hkv > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    CUtensorMap tmK, tmV;
    if (!encode_pool_k16(&tmK, k_cache, NB, Hkv, BS) || !encode_pool_box_halves(&tmV, v_cache, NB, Hkv, BS, 16))
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kTcSmemBytes));
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * Hkv), 1, 1);  // KV head innermost
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = kTcSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float scale_log2 = scale * 1.4426950408889634f;
    err = cudaLaunchKernelEx(&cfg, prefill_tc_kernel, tmK, tmV, static_cast<const __nv_bfloat16*>(q),
                             static_cast<__nv_bfloat16*>(out), block_tables, max_blocks, seq_lens, q_start, B, Hq, Hkv,
                             BS, NB, scale_log2, status);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace pkv
