// decode_attention.cu -- GQA paged decode attention (one query token per sequence).
//
// What it computes ("Bai Lab tong hop -- Inference Engineering", block [5]
// forward; "Suy luan & Toi uu hoa (Inference)" 3.1 GQA, 3.2 PagedAttention, 4.1
// online softmax): for query head qh of sequence b, KV head h = qh / G,
//   out[b][qh] = softmax_j(scale * <q, K_j>) . V_j   over the L = seq_lens[b]
// cached positions, K_j / V_j read from physical block block_tables[b][j / BS],
// slot j % BS of the pools [NB, Hkv, BS, D].
//
// Fast path (bf16, D = 128, BS % 16 == 0): a persistent, balanced split-KV kernel.
//  * Work unit = one logical block of one sequence, ALL KV heads: in the
//    [NB, Hkv, BS, D] layout the K (and V) rows of a block for every head are one
//    contiguous Hkv*BS*256-byte run, fetched by two 128B-swizzled 2-D TMA boxes.
//  * The sum over sequences of ceil(L/BS) blocks is cut into P = #SM equal
//    contiguous ranges; every CTA derives the cut itself from seq_lens (a sum
//    and a prefix scan over the batch), then streams its range c through an
//    nst-deep mbarrier ring fed by one producer lane, so each SM keeps
//    ~128 KB of KV in flight regardless of how lengths are distributed.
//  * One consumer warp per KV head computes S = Q K^T and O += P V with
//    mma.sync m16n8k16 (query heads of the group on the M axis, 16 tokens on N/K),
//    online softmax in the log2 domain, fp32 accumulation.
//  * A sequence cut by a range boundary leaves per-piece (max, sum, unnormalised
//    output) partials in the workspace, in one of two slots per range (the
//    range's first sequence when it began in an earlier range, else its last);
//    the combine kernel merges them with the online-softmax rule.  Sequences
//    wholly inside one range are written directly.
//  * main -> combine are chained with programmatic dependent launch: each kernel
//    launches while its predecessor runs and waits (griddepcontrol.wait) only
//    before reading the predecessor's results.
// Generic path (fp32, other shapes): one CTA per (sequence, query head),
// CUDA-core fp32, chunked online softmax.
#include <cuda.h>
#include <math.h>

#include <atomic>

#include "pkv_common.cuh"

namespace pkv {

// ------------------------------------------------------------------ workspace
struct SeqInfo {  // 16 bytes per sequence with at least one block
    int s;        // first global block index of the sequence in the split order
    int n;        // number of blocks
    int W;        // blocks per CTA range in this call
    int pad;
};

struct WsLayout {
    size_t info, ml, o, total;
};

static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// info[B]; then per range two partial slots (2P in all) of (m, l) and o[D] for
// every query head.
static WsLayout ws_layout(int B, int Hq, int D, int P) {
    WsLayout w;
    const size_t slots = 2 * static_cast<size_t>(P);
    w.info = 0;
    w.ml = align_up(sizeof(SeqInfo) * static_cast<size_t>(B), 256);
    w.o = align_up(w.ml + slots * Hq * 2 * sizeof(float), 256);
    w.total = align_up(w.o + slots * Hq * static_cast<size_t>(D) * sizeof(float), 256);
    return w;
}

size_t decode_workspace_bytes(int B, int Hq, int D, int P) { return ws_layout(B, Hq, D, P).total; }

// Blocks of sequence b (0 for a length outside [0, max_blocks * BS]).
__device__ __forceinline__ int seq_blocks(const int32_t* seq_lens, int b, int max_blocks, int BS) {
    const int L = seq_lens[b];
    return (L >= 0 && static_cast<long long>(L) <= static_cast<long long>(max_blocks) * BS) ? (L + BS - 1) / BS : 0;
}

// Exclusive prefix sum over the CTA (any blockDim up to 1024); red holds 33 ints.
__device__ __forceinline__ int cta_excl_scan(int v, int* red, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) red[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = lane < nw ? red[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        red[lane] = t;  // inclusive
    }
    __syncthreads();
    const int before = warp ? red[warp - 1] : 0;
    total = red[nw - 1];
    __syncthreads();
    return before + x - v;
}

// ------------------------------------------------------------------ fast kernel
// Orders this thread's earlier generic-proxy global writes before its later
// async-proxy (TMA) accesses of global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

constexpr int kMaxStages = 8;
constexpr int kDim = 128;

struct StageMeta {
    int b, j, ntok, flags;
};
// kHead: the sequence began in an earlier range (its partial goes to slot 2c,
// otherwise to slot 2c + 1 of range c).
enum : int { kValid = 1, kFirst = 2, kLast = 4, kWhole = 8, kHead = 16 };

// Layout of the dynamic shared memory (base rounded up to 1024 bytes for the
// 128-byte TMA swizzle): nst stages of [K lo | K hi | V lo | V hi] boxes, each
// box Hkv*BS rows x 128 bytes; a 2-slot ring of query rows [Hq][128] bf16; the
// mbarriers; the per-stage metadata; the schedule scratch (40 ints).
static inline size_t fast_smem_bytes(int nst, int stage_bytes, int q_bytes) {
    return 1024 + static_cast<size_t>(nst) * stage_bytes + 2 * static_cast<size_t>(q_bytes) +
           (2 * kMaxStages + 4) * sizeof(uint64_t) + kMaxStages * sizeof(StageMeta) + 40 * sizeof(int) + 16;
}

constexpr int kFastMaxKvHeads = 8;

template <bool kRows16>  // true when G > 8: query rows 8..15 of the MMA tile are live
__global__ void __launch_bounds__((kFastMaxKvHeads + 1) * 32, 1)
    decode_attn_fast_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                            const __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ out,
                            const int32_t* __restrict__ block_tables, int max_blocks, int B, int Hq, int Hkv,
                            int BS, int NB, float scale_log2, int nst, const int32_t* __restrict__ seq_lens,
                            SeqInfo* __restrict__ info, float* __restrict__ part_ml, float* __restrict__ part_o,
                            int32_t* status, const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                            uint4* kpool, uint4* vpool, uint32_t max_polls, int silent_cta) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int R = Hkv * BS;
    const uint32_t box_bytes = static_cast<uint32_t>(R) * 128u;
    const uint32_t stage_bytes = 4u * box_bytes;
    const uint32_t q_bytes = static_cast<uint32_t>(Hq) * (kDim * 2);
    uint8_t* stages = smem;
    uint8_t* qring = smem + static_cast<size_t>(nst) * stage_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(qring + 2 * static_cast<size_t>(q_bytes));
    uint64_t* empty = full + kMaxStages;
    uint64_t* qfull = empty + kMaxStages;
    uint64_t* qempty = qfull + 2;
    StageMeta* meta = reinterpret_cast<StageMeta*>(qempty + 2);
    int* sch = reinterpret_cast<int*>(meta + kMaxStages);  // [0, 33) scan scratch, 33: b0, 34: s0

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int CW = Hkv;  // consumer warps: one per KV head
    const int G = Hq / Hkv;

    // prologue independent of the inputs (overlaps the predecessor kernel)
    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&qfull[s], 1);
            mbar_init(&qempty[s], CW);
        }
        fence_mbar_init();
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the predecessor's writes (KV, lengths) are visible
    // The combine kernel may launch now.  It reads seq_lens before its own
    // griddepcontrol.wait, which is safe only because every CTA reaches this
    // trigger after the wait above (no return before it): keep the trigger
    // after the wait.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- schedule: the blocks of all sequences in order, cut into gridDim.x
    // ranges of W; this CTA takes range blockIdx.x and finds the sequence that
    // holds its first block with a prefix scan (stopping once past it)
    const int nthr = blockDim.x;
    const int n_first = static_cast<int>(threadIdx.x) < B ? seq_blocks(seq_lens, threadIdx.x, max_blocks, BS) : 0;
    int tsum = n_first;
    for (int b = threadIdx.x + nthr; b < B; b += nthr) tsum += seq_blocks(seq_lens, b, max_blocks, BS);
    if (k_new != nullptr && blockIdx.x == 0) {
        // with the append fused in, a length the append cannot place is an
        // error even where attention alone accepts it (L = 0)
        for (int b = threadIdx.x; b < B; b += nthr) {
            const int L = seq_lens[b];
            if (L < 1 || static_cast<long long>(L) > static_cast<long long>(max_blocks) * BS)
                report(status, PKV_ERR_DEVICE_BOUNDS);
        }
    }
    int total;
    cta_excl_scan(tsum, sch, total);
    const int W = total > 0 ? (total + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x) : 1;
    const int start = blockIdx.x * W;
    const int end = min(total, start + W);
    if (start >= end) return;  // uniform over the CTA
    {
        int carry = 0;
        for (int base = 0; base < B; base += nthr) {
            const int b = base + threadIdx.x;
            const int n = base == 0 ? n_first : (b < B ? seq_blocks(seq_lens, b, max_blocks, BS) : 0);
            int tot;
            const int sb = carry + cta_excl_scan(n, sch, tot);
            if (n > 0 && sb <= start && start < sb + n) {  // exactly one thread of the CTA
                sch[33] = b;
                sch[34] = sb;
            }
            carry += tot;
            if (carry > start) break;  // same decision in every thread
        }
        __syncthreads();
    }

    if (warp == CW) {
        // ------------------------------------------------ producer warp
        // Lane 0 waits on the ring and issues the copies.  With the append
        // fused in, the whole warp first writes a sequence's new token (every
        // KV head) into its last block, just before that block is loaded: the
        // one CTA that reads the block is the one that writes it.
        // walk the sequences from the one holding block `start`; empty and
        // invalid sequences have no blocks and are stepped over
        int b = sch[33], cs = sch[34];
        int cn = seq_blocks(seq_lens, b, max_blocks, BS), cL = seq_lens[b];
        // The combine kernel's view of every sequence whose first block lies
        // in this range, written before any wait, so that it is complete even
        // when a wait below gives up.
        if (lane == 0) {
            int bb = b, bs = cs, bn = cn;
            while (bs < end) {
                if (bs >= start && bn > 0) {
                    SeqInfo si;
                    si.s = bs;
                    si.n = bn;
                    si.W = W;
                    si.pad = 0;
                    info[bb] = si;
                }
                bs += bn;
                if (++bb >= B) break;
                bn = seq_blocks(seq_lens, bb, max_blocks, BS);
            }
        }
        // Test hook (off unless pkv_test_set_wait_limit named this CTA): issue
        // no copy at all, so that this CTA's consumers wait on stages nothing
        // will fill, give up after max_polls polls and report PKV_ERR_TIMEOUT
        // with no copy in flight.
        if (static_cast<int>(blockIdx.x) == silent_cta) return;
        int piece = 0;
        // On a timeout, wait (bounded) for the copies this lane issued that
        // no consumer has seen land, so that the CTA never exits with a bulk
        // copy still writing into its shared memory: the latest round of each
        // stage (iterations it - nst .. it - 1) and of each query slot.
        auto drain = [&](int it) {
            for (int k = max(0, it - nst); k < it; ++k)
                mbar_wait(&full[k % nst], static_cast<uint32_t>(k / nst) & 1u, max_polls);
            for (int pk = max(0, piece - 2); pk < piece; ++pk)
                mbar_wait(&qfull[pk & 1], static_cast<uint32_t>(pk >> 1) & 1u, max_polls);
        };
        for (int i = start, it = 0; i < end; ++i, ++it) {
            while (cs + cn <= i) {
                cs += cn;
                ++b;
                cn = seq_blocks(seq_lens, b, max_blocks, BS);
                cL = seq_lens[b];
            }
            const int j = i - cs;
            const int blk = block_tables[static_cast<size_t>(b) * max_blocks + j];
            const bool valid = blk >= 0 && blk < NB;
            if (k_new != nullptr && valid && j == cn - 1) {  // warp-uniform
                // the new token sits at position cL - 1, in this block
                constexpr int kRowVecs = kDim * 2 / 16;
                const int slot = cL - 1 - j * BS;
                for (int e = lane; e < Hkv * kRowVecs; e += 32) {
                    const int hh = e / kRowVecs, c = e - hh * kRowVecs;
                    const size_t src = static_cast<size_t>(b * Hkv + hh) * kRowVecs + c;
                    const size_t dst = ((static_cast<size_t>(blk) * Hkv + hh) * BS + slot) * kRowVecs + c;
                    kpool[dst] = __ldg(k_new + src);
                    vpool[dst] = __ldg(v_new + src);
                }
                // the rows are written through the generic proxy and read
                // back by this warp's TMA (the async proxy)
                fence_proxy_async_global();
                __syncwarp();
            }
            int ok = 1;
            if (lane == 0) {
                const bool first = (j == 0) || (i == start);
                const bool last = (j == cn - 1) || (i == end - 1);
                const bool whole = (cs >= start) && (cs + cn <= end);
                const bool head = cs < start;  // began in an earlier range (set on every stage of the piece)
                const int stage = it % nst;
                const uint32_t round = static_cast<uint32_t>(it / nst);
                if (!mbar_wait(&empty[stage], (round & 1u) ^ 1u, max_polls)) {
                    report(status, PKV_ERR_TIMEOUT);
                    ok = 0;
                }
                if (ok && first) {
                    const int qs = piece & 1;
                    const uint32_t qr = static_cast<uint32_t>(piece >> 1);
                    if (!mbar_wait(&qempty[qs], (qr & 1u) ^ 1u, max_polls)) {
                        report(status, PKV_ERR_TIMEOUT);
                        ok = 0;
                    } else {
                        mbar_arrive_expect_tx(&qfull[qs], q_bytes);
                        tma_load_1d(qring + static_cast<size_t>(qs) * q_bytes,
                                    q + static_cast<size_t>(b) * Hq * kDim, q_bytes, &qfull[qs]);
                        ++piece;
                    }
                }
                if (ok) {
                    StageMeta mt;
                    mt.b = b;
                    mt.j = j;
                    mt.ntok = min(BS, cL - j * BS);
                    mt.flags = (valid ? kValid : 0) | (first ? kFirst : 0) | (last ? kLast : 0) |
                               (whole ? kWhole : 0) | (head ? kHead : 0);
                    meta[stage] = mt;
                    uint64_t* fb = &full[stage];
                    if (valid) {
                        mbar_arrive_expect_tx(fb, stage_bytes);
                        uint8_t* st = stages + static_cast<size_t>(stage) * stage_bytes;
                        const int y = blk * R;
                        tma_load_2d(st, &tmK, 0, y, fb);
                        tma_load_2d(st + box_bytes, &tmK, 64, y, fb);
                        tma_load_2d(st + 2 * box_bytes, &tmV, 0, y, fb);
                        tma_load_2d(st + 3 * box_bytes, &tmV, 64, y, fb);
                    } else {
                        report(status, PKV_ERR_DEVICE_BOUNDS);
                        mbar_arrive(fb);
                    }
                }
                if (!ok) drain(it);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) return;  // a wait ran out: the whole warp leaves
        }
        return;
    }

    // ---------------------------------------------------- consumers: warp h
    const int h = warp;
    const int g = lane >> 2, r = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float O[16][4];
    uint32_t qa[8][4];
    bool poisoned = false;
    int piece = 0;
    const uint32_t stages_u32 = smem_u32(stages);

    for (int i = start, it = 0; i < end; ++i, ++it) {
        const int stage = it % nst;
        const uint32_t round = static_cast<uint32_t>(it / nst);
        if (!mbar_wait(&full[stage], round & 1u, max_polls)) {
            if (lane == 0) report(status, PKV_ERR_TIMEOUT);
            return;
        }
        const StageMeta mt = meta[stage];
        if (mt.flags & kFirst) {
            const int qs = piece & 1;
            const uint32_t qr = static_cast<uint32_t>(piece >> 1);
            if (!mbar_wait(&qfull[qs], qr & 1u, max_polls)) {
                if (lane == 0) report(status, PKV_ERR_TIMEOUT);
                return;
            }
            const __nv_bfloat16* qsm = reinterpret_cast<const __nv_bfloat16*>(qring + static_cast<size_t>(qs) * q_bytes);
            const int row0 = h * G + g, row1 = h * G + g + 8;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int c0 = kk * 16 + 2 * r;
                qa[kk][0] = g < G ? *reinterpret_cast<const uint32_t*>(qsm + row0 * kDim + c0) : 0u;
                qa[kk][2] = g < G ? *reinterpret_cast<const uint32_t*>(qsm + row0 * kDim + c0 + 8) : 0u;
                if (kRows16) {
                    qa[kk][1] = (g + 8) < G ? *reinterpret_cast<const uint32_t*>(qsm + row1 * kDim + c0) : 0u;
                    qa[kk][3] = (g + 8) < G ? *reinterpret_cast<const uint32_t*>(qsm + row1 * kDim + c0 + 8) : 0u;
                } else {
                    qa[kk][1] = 0u;
                    qa[kk][3] = 0u;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&qempty[qs]);
            ++piece;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) O[nt][0] = O[nt][1] = O[nt][2] = O[nt][3] = 0.f;
            poisoned = false;
        }
        if (mt.flags & kValid) {
            const uint32_t kb = stages_u32 + static_cast<uint32_t>(stage) * stage_bytes;
            const uint32_t vb = kb + 2 * box_bytes;
            if (mt.ntok < BS) {
                // Slots past the sequence end may hold anything (NaN included):
                // clear this head's V rows there so that 0 * V stays 0.
                uint8_t* vsm = stages + static_cast<size_t>(stage) * stage_bytes + 2 * box_bytes;
                const int nrows = BS - mt.ntok;
                for (int e = lane; e < nrows * 16; e += 32) {  // 2 boxes x 128 B = 16 x 16 B per row
                    const int row = h * BS + mt.ntok + (e >> 4);
                    const int part = e & 15;
                    uint4* dst = reinterpret_cast<uint4*>(vsm + (part >> 3) * box_bytes + row * 128 + (part & 7) * 16);
                    *dst = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            const int nchunk = (min(mt.ntok, BS) + 15) >> 4;
            for (int c = 0; c < nchunk; ++c) {
                const int rbase = h * BS + c * 16;
                // ---- S = Q K^T for 16 tokens (two n-tiles of 8)
                float s[2][4];
#pragma unroll
                for (int t = 0; t < 2; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int tok = (mi >> 1) * 8 + rr;
                    const int dc = kk * 2 + (mi & 1);
                    const int row = rbase + tok;
                    const uint32_t addr = kb + static_cast<uint32_t>(dc >> 3) * box_bytes +
                                          static_cast<uint32_t>(row) * 128u +
                                          (static_cast<uint32_t>((dc & 7) ^ (row & 7)) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(b0, b1, b2, b3, addr);
                    mma_bf16_16816(s[0], qa[kk], b0, b1);
                    mma_bf16_16816(s[1], qa[kk], b2, b3);
                }
                // ---- online softmax (log2 domain), masking tokens past the end
                const int tb = c * 16;
#pragma unroll
                for (int t = 0; t < 2; ++t)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int tk = tb + t * 8 + 2 * r + (e & 1);
                        const float v = s[t][e] * scale_log2;
                        s[t][e] = tk < mt.ntok ? v : -INFINITY;
                    }
                float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                const float mn0 = fmaxf(m0, mx0);
                const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
                const float a0 = exp2f(m0 - mu0);
                m0 = mn0;
                float a1 = 1.f, mu1 = 0.f;
                if (kRows16) {
                    float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                    const float mn1 = fmaxf(m1, mx1);
                    mu1 = mn1 == -INFINITY ? 0.f : mn1;
                    a1 = exp2f(m1 - mu1);
                    m1 = mn1;
                }
                uint32_t pa[4];
                pa[0] = pack_bf16x2(exp2f(s[0][0] - mu0), exp2f(s[0][1] - mu0));
                pa[2] = pack_bf16x2(exp2f(s[1][0] - mu0), exp2f(s[1][1] - mu0));
                l0 = l0 * a0 + ((bf16_lo(pa[0]) + bf16_hi(pa[0])) + (bf16_lo(pa[2]) + bf16_hi(pa[2])));
                if (kRows16) {
                    pa[1] = pack_bf16x2(exp2f(s[0][2] - mu1), exp2f(s[0][3] - mu1));
                    pa[3] = pack_bf16x2(exp2f(s[1][2] - mu1), exp2f(s[1][3] - mu1));
                    l1 = l1 * a1 + ((bf16_lo(pa[1]) + bf16_hi(pa[1])) + (bf16_lo(pa[3]) + bf16_hi(pa[3])));
                } else {
                    pa[1] = 0u;
                    pa[3] = 0u;
                }
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    O[nt][0] *= a0;
                    O[nt][1] *= a0;
                    if (kRows16) {
                        O[nt][2] *= a1;
                        O[nt][3] *= a1;
                    }
                }
                // ---- O += P V
#pragma unroll
                for (int dp = 0; dp < 8; ++dp) {
                    const int tok = (mi & 1) * 8 + rr;
                    const int dc = dp * 2 + (mi >> 1);
                    const int row = rbase + tok;
                    const uint32_t addr = vb + static_cast<uint32_t>(dc >> 3) * box_bytes +
                                          static_cast<uint32_t>(row) * 128u +
                                          (static_cast<uint32_t>((dc & 7) ^ (row & 7)) << 4);
                    uint32_t v0, v1, v2, v3;
                    ldmatrix_x4_trans(v0, v1, v2, v3, addr);
                    mma_bf16_16816(O[2 * dp], pa, v0, v1);
                    mma_bf16_16816(O[2 * dp + 1], pa, v2, v3);
                }
            }
        } else {
            poisoned = true;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);

        if (mt.flags & kLast) {
            float lt0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
            lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
            float lt1 = 0.f;
            if (kRows16) {
                lt1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
                lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
            }
            const int b = mt.b;
            const int qh0 = h * G + g, qh1 = h * G + g + 8;
            const bool live0 = g < G, live1 = kRows16 && (g + 8) < G;
            if (mt.flags & kWhole) {
                const float inv0 = (!poisoned && lt0 > 0.f) ? 1.f / lt0 : 0.f;
                const float inv1 = (!poisoned && lt1 > 0.f) ? 1.f / lt1 : 0.f;
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    const int d = nt * 8 + 2 * r;
                    if (live0)
                        *reinterpret_cast<uint32_t*>(out + (static_cast<size_t>(b) * Hq + qh0) * kDim + d) =
                            pack_bf16x2(O[nt][0] * inv0, O[nt][1] * inv0);
                    if (live1)
                        *reinterpret_cast<uint32_t*>(out + (static_cast<size_t>(b) * Hq + qh1) * kDim + d) =
                            pack_bf16x2(O[nt][2] * inv1, O[nt][3] * inv1);
                }
            } else {
                const size_t slot = 2 * static_cast<size_t>(blockIdx.x) + ((mt.flags & kHead) ? 0 : 1);
                if (r == 0) {
                    if (live0) {
                        part_ml[(slot * Hq + qh0) * 2 + 0] = m0;
                        part_ml[(slot * Hq + qh0) * 2 + 1] = poisoned ? -1.f : lt0;
                    }
                    if (live1) {
                        part_ml[(slot * Hq + qh1) * 2 + 0] = m1;
                        part_ml[(slot * Hq + qh1) * 2 + 1] = poisoned ? -1.f : lt1;
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    const int d = nt * 8 + 2 * r;
                    if (live0)
                        *reinterpret_cast<float2*>(part_o + (slot * Hq + qh0) * kDim + d) =
                            make_float2(O[nt][0], O[nt][1]);
                    if (live1)
                        *reinterpret_cast<float2*>(part_o + (slot * Hq + qh1) * kDim + d) =
                            make_float2(O[nt][2], O[nt][3]);
                }
            }
        }
    }
}

// ------------------------------------------------------------------ combine kernel
// Merges the per-range partials of sequences that span several CTA ranges:
// M = max m_c, out = sum o_c 2^(m_c - M) / sum l_c 2^(m_c - M) (log2 domain).
// A sequence spanning ranges f..t left its piece in range f in slot 2f + 1 and
// its pieces in ranges f+1..t in slots 2c.
// Two forms.  With many (sequence, query head) units, one warp per unit (four
// dimensions per lane).  With few units, which then have many pieces each, one
// CTA of kCombWarps warps per unit: thread p reads piece p's (m, l) and warp w
// sums the outputs of pieces w, w + kCombWarps, ..., whose loads are issued
// together with the (m, l) reads, so up to kCombWarps * kCombGroup pieces cost
// one round trip to memory; the warps' sums meet in shared memory.  Both write
// zeros for empty, invalid or poisoned sequences and skip single-range
// sequences, which the fast kernel wrote directly.
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}
__device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

constexpr int kCombWarps = 4;
constexpr int kCombThreads = kCombWarps * 32;
constexpr int kCombGroup = 8;
constexpr int kCombMaxPieces = 1024;  // per sequence (a range holds >= 1 block, so pieces <= P)

// Many (sequence, head) units: one warp each, four dimensions per lane; the
// first kCombGroup pieces' outputs are requested together with the (m, l) pairs.
template <typename T>
__global__ void __launch_bounds__(kCombThreads)
    combine_warp_kernel(const SeqInfo* __restrict__ info, const int32_t* __restrict__ seq_lens, int max_blocks,
                        int BS, const float* __restrict__ part_ml, const float* __restrict__ part_o,
                        T* __restrict__ out, int B, int Hq, int P, int32_t* status) {
    const int lane = threadIdx.x & 31;
    const long long u = static_cast<long long>(blockIdx.x) * kCombWarps + (threadIdx.x >> 5);
    if (u >= static_cast<long long>(B) * Hq) return;
    const int b = static_cast<int>(u / Hq), qh = static_cast<int>(u - static_cast<long long>(b) * Hq);
    // the lengths predate the main kernel (which launched this one only after
    // its own wait on its predecessors), so they are read before the wait
    const int L = seq_lens[b];
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the main kernel's partials are visible
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const bool valid = L >= 0 && static_cast<long long>(L) <= static_cast<long long>(max_blocks) * BS;
    if (!valid && qh == 0 && lane == 0) report(status, PKV_ERR_DEVICE_BOUNDS);
    const int n = valid ? (L + BS - 1) / BS : 0;
    int pieces = 0, f = 0;
    if (n > 0) {
        const SeqInfo si = info[b];
        if (si.W > 0 && si.s >= 0) {
            f = si.s / si.W;
            pieces = (si.s + n - 1) / si.W - f + 1;
        }
        // a record that names slots outside the workspace's 2P (possible only
        // when the main kernel gave up on a wait) merges nothing
        if (f + pieces > P) pieces = 0;
    }
    if (pieces == 1) return;
    T* o = out + static_cast<size_t>(u) * kDim + 4 * lane;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float inv = 0.f;
    if (pieces > 1 && pieces <= kCombMaxPieces) {
        const size_t base = 2 * static_cast<size_t>(f);  // piece p at slot offset 2p + (p == 0)
        const size_t ml_stride = static_cast<size_t>(Hq) * 2, o_stride = static_cast<size_t>(Hq) * kDim;
        const float* mlp = part_ml + (base * Hq + qh) * 2;
        const float* op = part_o + (base * Hq + qh) * kDim + 4 * lane;
        auto off = [](int p) { return static_cast<size_t>(2 * p + (p == 0 ? 1 : 0)); };
        float4 og[kCombGroup];
#pragma unroll
        for (int j = 0; j < kCombGroup; ++j)
            og[j] = j < pieces ? __ldg(reinterpret_cast<const float4*>(op + off(j) * o_stride))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        float M = -INFINITY;
        bool bad = false;
        for (int c = lane; c < pieces; c += 32) {
            const float2 ml = __ldg(reinterpret_cast<const float2*>(mlp + off(c) * ml_stride));
            M = fmaxf(M, ml.x);
            bad |= ml.y < 0.f;
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
        bad = __any_sync(0xffffffffu, bad) || M == -INFINITY;
        if (!bad) {
            float Lsum = 0.f;
            for (int c0 = 0; c0 < pieces; c0 += 32) {
                float wl = 0.f;  // lane c: weight of piece c0 + c
                if (c0 + lane < pieces) {
                    const float2 ml = __ldg(reinterpret_cast<const float2*>(mlp + off(c0 + lane) * ml_stride));
                    wl = exp2f(ml.x - M);
                    Lsum = fmaf(ml.y, wl, Lsum);
                }
                const int nj = min(32, pieces - c0);
                for (int j0 = 0; j0 < nj; j0 += kCombGroup) {
                    if (c0 + j0 >= kCombGroup) {  // later groups: fetch now
#pragma unroll
                        for (int j = 0; j < kCombGroup; ++j)
                            og[j] = j0 + j < nj
                                        ? __ldg(reinterpret_cast<const float4*>(op + off(c0 + j0 + j) * o_stride))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int j = 0; j < kCombGroup; ++j) {
                        const float wj = __shfl_sync(0xffffffffu, wl, (j0 + j) & 31);
                        if (j0 + j < nj) {
                            acc.x = fmaf(wj, og[j].x, acc.x);
                            acc.y = fmaf(wj, og[j].y, acc.y);
                            acc.z = fmaf(wj, og[j].z, acc.z);
                            acc.w = fmaf(wj, og[j].w, acc.w);
                        }
                    }
                }
            }
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o2);
            inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        }
    }
    store4(o, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
}

// Few units (long sequences, many pieces each): one CTA per unit.
template <typename T>
__global__ void __launch_bounds__(kCombThreads)
    combine_kernel(const SeqInfo* __restrict__ info, const int32_t* __restrict__ seq_lens, int max_blocks, int BS,
                   const float* __restrict__ part_ml, const float* __restrict__ part_o, T* __restrict__ out,
                   int Hq, int P, int32_t* status) {
    __shared__ float wsh[kCombMaxPieces];
    __shared__ float4 accsh[kCombWarps][32];
    __shared__ float red[2][kCombWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x / Hq, qh = blockIdx.x - (blockIdx.x / Hq) * Hq;
    const int L = seq_lens[b];  // predates the main kernel: read before the wait
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the main kernel's partials are visible
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const bool valid = L >= 0 && static_cast<long long>(L) <= static_cast<long long>(max_blocks) * BS;
    if (!valid && qh == 0 && tid == 0) report(status, PKV_ERR_DEVICE_BOUNDS);
    const int n = valid ? (L + BS - 1) / BS : 0;
    int pieces = 0, f = 0;
    if (n > 0) {
        const SeqInfo si = info[b];
        if (si.W > 0 && si.s >= 0) {
            f = si.s / si.W;
            pieces = (si.s + n - 1) / si.W - f + 1;
        }
        // a record that names slots outside the workspace's 2P (possible only
        // when the main kernel gave up on a wait) merges nothing
        if (f + pieces > P) pieces = 0;
    }
    if (pieces == 1) return;  // uniform over the CTA
    T* o = out + (static_cast<size_t>(b) * Hq + qh) * kDim;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float inv = 0.f;
    if (pieces > 1 && pieces <= kCombMaxPieces) {
        // piece p sits in slot 2f + 1 (p = 0) or 2(f + p) (p > 0); from slot 2f
        // that is an offset of 2p + (p == 0) slots
        const size_t base = 2 * static_cast<size_t>(f);
        const size_t ml_stride = static_cast<size_t>(Hq) * 2, o_stride = static_cast<size_t>(Hq) * kDim;
        const float* mlp = part_ml + (base * Hq + qh) * 2;
        const float* op = part_o + (base * Hq + qh) * kDim + 4 * lane;
        auto off = [](int p) { return static_cast<size_t>(2 * p + (p == 0 ? 1 : 0)); };
        float4 og[kCombGroup];
#pragma unroll
        for (int j = 0; j < kCombGroup; ++j) {
            const int p = warp + kCombWarps * j;
            og[j] = p < pieces ? __ldg(reinterpret_cast<const float4*>(op + off(p) * o_stride))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float M = -INFINITY, Lsum = 0.f;
        bool bad = false;
        for (int p = tid; p < pieces; p += kCombThreads) {
            const float2 ml = __ldg(reinterpret_cast<const float2*>(mlp + off(p) * ml_stride));
            M = fmaxf(M, ml.x);
            bad |= ml.y < 0.f;
            wsh[p] = ml.x;
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
        bad = __syncthreads_or(bad ? 1 : 0) != 0;  // also publishes wsh
        if (lane == 0) red[0][warp] = M;
        __syncthreads();
        M = red[0][0];
#pragma unroll
        for (int w = 1; w < kCombWarps; ++w) M = fmaxf(M, red[0][w]);
        if (!bad && M > -INFINITY) {
            for (int p = tid; p < pieces; p += kCombThreads) {
                const float wgt = exp2f(wsh[p] - M);
                Lsum = fmaf(__ldg(mlp + off(p) * ml_stride + 1), wgt, Lsum);
                wsh[p] = wgt;
            }
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o2);
            if (lane == 0) red[1][warp] = Lsum;
            __syncthreads();  // weights and partial sums published
            float Lt = 0.f;
#pragma unroll
            for (int w = 0; w < kCombWarps; ++w) Lt += red[1][w];
            inv = Lt > 0.f ? 1.f / Lt : 0.f;
            for (int p0 = 0; p0 < pieces; p0 += kCombWarps * kCombGroup) {
                if (p0 > 0) {  // later groups: fetch now
#pragma unroll
                    for (int j = 0; j < kCombGroup; ++j) {
                        const int p = p0 + warp + kCombWarps * j;
                        og[j] = p < pieces ? __ldg(reinterpret_cast<const float4*>(op + off(p) * o_stride))
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
#pragma unroll
                for (int j = 0; j < kCombGroup; ++j) {
                    const int p = p0 + warp + kCombWarps * j;
                    if (p < pieces) {
                        const float wj = wsh[p];
                        acc.x = fmaf(wj, og[j].x, acc.x);
                        acc.y = fmaf(wj, og[j].y, acc.y);
                        acc.z = fmaf(wj, og[j].z, acc.z);
                        acc.w = fmaf(wj, og[j].w, acc.w);
                    }
                }
            }
        }
    }
    // the warps' sums meet in warp 0
    if (warp > 0) accsh[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int w = 1; w < kCombWarps; ++w) {
            const float4 t = accsh[w][lane];
            acc.x += t.x;
            acc.y += t.y;
            acc.z += t.z;
            acc.w += t.w;
        }
        store4(o + 4 * lane, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
    }
}

// ------------------------------------------------------------------ generic kernel
// One CTA per (sequence, query head); 128 threads; chunks of 128 tokens; fp32
// online softmax across chunks.  Handles any D <= 256, any block size, fp32 or
// bf16 storage.
constexpr int kGenThreads = 128;

template <typename T>
__global__ void __launch_bounds__(kGenThreads)
    decode_attn_generic_kernel(T* __restrict__ out, const T* __restrict__ q, const T* __restrict__ k_cache,
                               const T* __restrict__ v_cache, const int32_t* __restrict__ block_tables,
                               int max_blocks, const int32_t* __restrict__ seq_lens, int Hq, int Hkv, int D,
                               int BS, int NB, float scale, int32_t* status) {
    __shared__ float qs[256];
    __shared__ float ps[kGenThreads];
    __shared__ int blks[kGenThreads];
    __shared__ float red[kGenThreads / 32];
    __shared__ int bad;
    const int b = blockIdx.x / Hq, qh = blockIdx.x % Hq;
    const int G = Hq / Hkv, h = qh / G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    T* o = out + (static_cast<size_t>(b) * Hq + qh) * D;
    const int L = seq_lens[b];
    if (L < 0 || static_cast<long long>(L) > static_cast<long long>(max_blocks) * BS) {
        if (tid == 0) report(status, PKV_ERR_DEVICE_BOUNDS);
        for (int d = tid; d < D; d += kGenThreads) o[d] = from_f32<T>(0.f);
        return;
    }
    for (int d = tid; d < D; d += kGenThreads) qs[d] = to_f32(q[(static_cast<size_t>(b) * Hq + qh) * D + d]);
    if (tid == 0) bad = 0;
    __syncthreads();
    float m = -INFINITY, l = 0.f;
    float acc[2] = {0.f, 0.f};
    for (int t0 = 0; t0 < L; t0 += kGenThreads) {
        const int n = min(kGenThreads, L - t0);
        float s = -INFINITY;
        if (tid < n) {
            const int pos = t0 + tid;
            const int blk = block_tables[static_cast<size_t>(b) * max_blocks + pos / BS];
            blks[tid] = blk;
            if (blk < 0 || blk >= NB) {
                bad = 1;
            } else {
                const T* kr = k_cache + ((static_cast<size_t>(blk) * Hkv + h) * BS + pos % BS) * D;
                float dot = 0.f;
                for (int d = 0; d < D; ++d) dot = fmaf(qs[d], to_f32(kr[d]), dot);
                s = dot * scale;
            }
        }
        // block max
        float mx = s;
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (lane == 0) red[warp] = mx;
        __syncthreads();
        mx = red[0];
        for (int w = 1; w < kGenThreads / 32; ++w) mx = fmaxf(mx, red[w]);
        __syncthreads();
        const float mn = fmaxf(m, mx);
        const float mu = mn == -INFINITY ? 0.f : mn;
        const float alpha = expf(m - mu);
        const float p = (tid < n && s != -INFINITY) ? expf(s - mu) : 0.f;
        ps[tid] = p;
        float sm = p;
        for (int off = 16; off > 0; off >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, off);
        if (lane == 0) red[warp] = sm;
        __syncthreads();
        float psum = 0.f;
        for (int w = 0; w < kGenThreads / 32; ++w) psum += red[w];
        l = l * alpha + psum;
        m = mn;
        for (int k = 0; k < 2; ++k) {
            const int d = tid + k * kGenThreads;
            if (d < D) {
                float a = acc[k] * alpha;
                for (int t = 0; t < n; ++t) {
                    const float pt = ps[t];
                    const int blk = blks[t];
                    if (pt != 0.f && blk >= 0 && blk < NB) {
                        const int pos = t0 + t;
                        a = fmaf(pt, to_f32(v_cache[((static_cast<size_t>(blk) * Hkv + h) * BS + pos % BS) * D + d]), a);
                    }
                }
                acc[k] = a;
            }
        }
        __syncthreads();
    }
    const bool poisoned = bad != 0;
    if (poisoned && tid == 0) report(status, PKV_ERR_DEVICE_BOUNDS);
    const float inv = (!poisoned && l > 0.f) ? 1.f / l : 0.f;
    for (int k = 0; k < 2; ++k) {
        const int d = tid + k * kGenThreads;
        if (d < D) o[d] = from_f32<T>(acc[k] * inv);
    }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qres) ==
                cudaSuccess &&
            qres == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        tried = true;
    }
    return fn;
}

// Tensor map over a pool [NB, Hkv, BS, 128] bf16 seen as rows of 128 elements,
// boxes of 64 elements x box_rows rows, 128-byte swizzle.
bool encode_pool_box(CUtensorMap* map, const void* pool, int NB, int Hkv, int BS, int box_rows) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc || box_rows < 1 || box_rows > 256) return false;
    const cuuint64_t rows = static_cast<cuuint64_t>(NB) * Hkv * BS;
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(kDim), rows};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(kDim) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult res = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), gdim, gstride, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

// The same pool seen in three dimensions (64 elements, rows, the two 64-element
// halves of a row), boxes of 64 x box_rows x 2: both halves of box_rows rows
// in one copy, landing as [half][row][64] (two 128-byte-swizzled atoms).
bool encode_pool_box_halves(CUtensorMap* map, const void* pool, int NB, int Hkv, int BS, int box_rows) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc || box_rows < 1 || box_rows > 256) return false;
    const cuuint64_t rows = static_cast<cuuint64_t>(NB) * Hkv * BS;
    cuuint64_t gdim[3] = {64, rows, 2};
    cuuint64_t gstride[2] = {static_cast<cuuint64_t>(kDim) * 2, 128};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult res = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), gdim, gstride, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

// The attention stage: all Hkv * BS rows of one block in one box.
static bool encode_pool_map(CUtensorMap* map, const void* pool, int NB, int Hkv, int BS) {
    return encode_pool_box(map, pool, NB, Hkv, BS, Hkv * BS);
}

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

static int max_optin_smem() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    return n;
}

struct FastPlan {
    bool ok;
    int nst, stage_bytes, q_bytes;
    size_t smem;
};

static FastPlan plan_fast(int Hq, int Hkv, int D, int BS, pkv_dtype dt, const void* k, const void* v,
                          const void* q, const void* out) {
    FastPlan fp{false, 0, 0, 0, 0};
    auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (dt != PKV_BF16 || D != kDim || BS % 16 != 0 || Hkv < 1 || Hkv > kFastMaxKvHeads) return fp;
    const int G = Hq / Hkv;
    if (G < 1 || G > 16) return fp;
    const int R = Hkv * BS;
    if (R > 256) return fp;
    if (!aligned16(k) || !aligned16(v) || !aligned16(q) || !aligned16(out)) return fp;
    fp.stage_bytes = 4 * R * 128;
    fp.q_bytes = Hq * kDim * 2;
    const long long budget = max_optin_smem();
    long long nst = (budget - static_cast<long long>(fast_smem_bytes(0, fp.stage_bytes, fp.q_bytes))) / fp.stage_bytes;
    if (nst > kMaxStages) nst = kMaxStages;
    if (nst < 2) return fp;
    fp.nst = static_cast<int>(nst);
    fp.smem = fast_smem_bytes(fp.nst, fp.stage_bytes, fp.q_bytes);
    fp.ok = true;
    return fp;
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int32_t* block_tables, int max_blocks, const int32_t* seq_lens, int B, int Hkv,
                             int D, int BS, int NB, pkv_dtype dtype, int32_t* status, cudaStream_t stream);

// State of the failure-path test hook (pkv_test_set_wait_limit): the poll
// budget of the fast kernel's waits and the CTA whose loader stays silent.
static std::atomic<uint32_t> g_wait_polls{kMaxWaitIters};
static std::atomic<int> g_silent_cta{-1};

// k_new / v_new non-null: append each sequence's new token first (same result
// as launch_kv_append followed by attention).  The fast kernel does the append
// itself; every other case launches the append kernel before attention.
cudaError_t launch_decode_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, int max_blocks, const int32_t* seq_lens, int B,
                                    int Hq, int Hkv, int D, int BS, int NB, float scale, pkv_dtype dtype,
                                    void* workspace, int P, int32_t* status, cudaStream_t stream,
                                    bool* used_fast, const void* k_new, const void* v_new) {
    if (scale <= 0.f) scale = 1.0f / sqrtf(static_cast<float>(D));
    const FastPlan fp = plan_fast(Hq, Hkv, D, BS, dtype, k_cache, v_cache, q, out);
    CUtensorMap tmK, tmV;
    bool fast = fp.ok && encode_pool_map(&tmK, k_cache, NB, Hkv, BS) && encode_pool_map(&tmV, v_cache, NB, Hkv, BS);
    if (used_fast) *used_fast = fast;
    const bool append = k_new != nullptr;
    const bool fused = fast && append && (reinterpret_cast<uintptr_t>(k_new) & 15u) == 0 &&
                       (reinterpret_cast<uintptr_t>(v_new) & 15u) == 0;
    if (append && !fused) {
        cudaError_t e = launch_kv_append(k_new, v_new, const_cast<void*>(k_cache), const_cast<void*>(v_cache),
                                         block_tables, max_blocks, seq_lens, B, Hkv, D, BS, NB, dtype, status,
                                         stream);
        if (e != cudaSuccess) return e;
    }
    if (!fast) {
        const unsigned grid = static_cast<unsigned>(B) * Hq;
        if (dtype == PKV_F32)
            decode_attn_generic_kernel<float><<<grid, kGenThreads, 0, stream>>>(
                static_cast<float*>(out), static_cast<const float*>(q), static_cast<const float*>(k_cache),
                static_cast<const float*>(v_cache), block_tables, max_blocks, seq_lens, Hq, Hkv, D, BS, NB, scale,
                status);
        else
            decode_attn_generic_kernel<__nv_bfloat16><<<grid, kGenThreads, 0, stream>>>(
                static_cast<__nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(q),
                static_cast<const __nv_bfloat16*>(k_cache), static_cast<const __nv_bfloat16*>(v_cache), block_tables,
                max_blocks, seq_lens, Hq, Hkv, D, BS, NB, scale, status);
        return cudaGetLastError();
    }
    const WsLayout wl = ws_layout(B, Hq, D, P);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    SeqInfo* info = reinterpret_cast<SeqInfo*>(ws + wl.info);
    float* part_ml = reinterpret_cast<float*>(ws + wl.ml);
    float* part_o = reinterpret_cast<float*>(ws + wl.o);
    const float scale_log2 = scale * 1.4426950408889634f;
    const int G = Hq / Hkv;
    const unsigned threads = static_cast<unsigned>((Hkv + 1) * 32);
    auto kern = G > 8 ? decode_attn_fast_kernel<true> : decode_attn_fast_kernel<false>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(fp.smem));
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(P), 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = fp.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, kern, tmK, tmV, static_cast<const __nv_bfloat16*>(q),
                             static_cast<__nv_bfloat16*>(out), block_tables, max_blocks, B, Hq, Hkv, BS, NB,
                             scale_log2, fp.nst, seq_lens, info, part_ml, part_o, status,
                             static_cast<const uint4*>(fused ? k_new : nullptr),
                             static_cast<const uint4*>(fused ? v_new : nullptr),
                             static_cast<uint4*>(const_cast<void*>(k_cache)),
                             static_cast<uint4*>(const_cast<void*>(v_cache)), g_wait_polls.load(),
                             g_silent_cta.load());
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t ccfg = {};
    ccfg.blockDim = dim3(kCombThreads, 1, 1);
    ccfg.dynamicSmemBytes = 0;
    ccfg.stream = stream;
    ccfg.attrs = attr;
    ccfg.numAttrs = 1;
    const long long units = static_cast<long long>(B) * Hq;
    if (units >= 8LL * P) {
        ccfg.gridDim = dim3(static_cast<unsigned>((units + kCombWarps - 1) / kCombWarps), 1, 1);
        err = cudaLaunchKernelEx(&ccfg, combine_warp_kernel<__nv_bfloat16>, static_cast<const SeqInfo*>(info),
                                 seq_lens, max_blocks, BS, static_cast<const float*>(part_ml),
                                 static_cast<const float*>(part_o), static_cast<__nv_bfloat16*>(out), B, Hq, P,
                                 status);
    } else {
        ccfg.gridDim = dim3(static_cast<unsigned>(units), 1, 1);
        err = cudaLaunchKernelEx(&ccfg, combine_kernel<__nv_bfloat16>, static_cast<const SeqInfo*>(info), seq_lens,
                                 max_blocks, BS, static_cast<const float*>(part_ml),
                                 static_cast<const float*>(part_o), static_cast<__nv_bfloat16*>(out), Hq, P, status);
    }
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace pkv

// ------------------------------------------------------------------ allocation-free variant
// Some callers cannot allocate device memory when they run attention: a serving
// loop that reserved all free HBM for its KV pool up front, code that must not
// risk the implicit synchronisation an allocation can cause, or a plain C host
// program with no device allocator of its own.  For them the split-KV
// workspace lives in this fixed, file-scope device array instead.  It is
// allocated when the library is loaded onto a GPU and stays until the process
// exits, on every GPU that loads the library.
namespace pkv {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(16) << 20;  // 16 MiB
static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

// Device address of g_decode_scratch on the current device.  Looked up on
// every call (cheap once the module is loaded on the device): a cached address
// would go stale when the device's context is reset or another context is
// current, and the host-side symbol is only a stand-in, never a device address.
static void* decode_scratch_address(cudaError_t* err) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_decode_scratch);
    return *err == cudaSuccess ? p : nullptr;
}

}  // namespace pkv

extern "C" pkv_status pkv_paged_decode_attention_noalloc(void* out, const void* q, const void* k_cache,
                                                         const void* v_cache, const int32_t* block_tables,
                                                         int max_blocks_per_seq, const int32_t* seq_lens, int B,
                                                         int Hq, int Hkv, int D, int block_size, int num_blocks,
                                                         float scale, pkv_dtype dtype, int32_t* dev_status,
                                                         void* stream) {
    if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 1 || D > 256 || block_size < 1 || num_blocks < 1 ||
        max_blocks_per_seq < 1 || (dtype != PKV_F32 && dtype != PKV_BF16))
        return PKV_ERR_INVALID_ARG;
    if (B == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PKV_ERR_INVALID_ARG;
    const int P = pkv::device_sm_count();
    if (P <= 0) return PKV_ERR_CUDA;
    if (pkv::decode_workspace_bytes(B, Hq, D, P) > pkv::kStaticScratchBytes) return PKV_ERR_UNSUPPORTED;
    cudaError_t err;
    void* ws = pkv::decode_scratch_address(&err);
    if (ws == nullptr) return PKV_ERR_CUDA;
    err = pkv::launch_decode_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, B, Hq,
                                       Hkv, D, block_size, num_blocks, scale, dtype, ws, P, dev_status,
                                       static_cast<cudaStream_t>(stream), nullptr, nullptr, nullptr);
    return err == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" pkv_status pkv_test_set_wait_limit(uint32_t polls, int silent_cta) {
    if (silent_cta < -1) return PKV_ERR_INVALID_ARG;
    pkv::g_wait_polls.store(polls == 0 ? pkv::kMaxWaitIters : polls);
    pkv::g_silent_cta.store(silent_cta);
    return PKV_OK;
}
