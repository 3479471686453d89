// block_pool.cu -- host-side, reference-counted allocator of physical KV blocks.
//
// "LLM inference serving tutorial": section 4.2 (a block table maps each
// sequence's logical blocks to non-contiguous physical blocks; physical blocks
// are shared by reference count between common prefixes and beam branches; a
// shared writable tail block is copied before it diverges -- copy-on-write),
// section 1.7 (reclaim decrements reference counts, a block returns to the
// allocator only when its last holder releases it, and reclaiming twice must
// be harmless), appendix A [D07]-[D08] (logical vs allocated slots; sharing a
// full block brings lengths 6 and 7 at block size 4 from 4 physical blocks to
// 3).  "Bai Lab tong hop -- Inference Engineering" block [6] (KVPool: a free
// list of blocks, a per-sequence block list, allocation when a sequence's
// length crosses a block boundary, release on finish).
//
// The pool never touches device memory: it decides block ids, keeps the
// reference counts, and reports the (src, dst) pairs that pkv_copy_blocks must
// copy on the GPU before the step's kv_append writes into the new tail block.
// Allocation takes the most recently freed block first (LIFO free list; ids in
// ascending order at creation).  Every mutating call either succeeds wholly or
// changes nothing.  Not thread-safe: one pool per scheduler thread.
#include <stdint.h>

#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"

struct pkv_block_pool {
    int num_blocks, block_size, max_blocks_per_seq;
    std::vector<int32_t> ref;        // reference count per physical block
    std::vector<int32_t> free_list;  // stack: back() is allocated next
    struct Seq {
        int len;
        std::vector<int32_t> blocks;
    };
    std::unordered_map<int64_t, Seq> seqs;

    int32_t take() {
        const int32_t b = free_list.back();
        free_list.pop_back();
        ref[b] = 1;
        return b;
    }
    void release(int32_t b) {
        if (--ref[b] == 0) free_list.push_back(b);
    }
    long long blocks_for(long long len) const { return (len + block_size - 1) / block_size; }
};

extern "C" {

pkv_block_pool* pkv_block_pool_create(int num_blocks, int block_size, int max_blocks_per_seq) {
    if (num_blocks < 1 || block_size < 1 || max_blocks_per_seq < 1) return nullptr;
    pkv_block_pool* p = new (std::nothrow) pkv_block_pool();
    if (!p) return nullptr;
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->max_blocks_per_seq = max_blocks_per_seq;
    p->ref.assign(static_cast<size_t>(num_blocks), 0);
    p->free_list.reserve(static_cast<size_t>(num_blocks));
    for (int b = num_blocks - 1; b >= 0; --b) p->free_list.push_back(b);
    return p;
}

void pkv_block_pool_destroy(pkv_block_pool* p) { delete p; }

int pkv_block_pool_num_free(const pkv_block_pool* p) { return p ? static_cast<int>(p->free_list.size()) : -1; }

int pkv_block_pool_refcount(const pkv_block_pool* p, int block) {
    if (!p || block < 0 || block >= p->num_blocks) return -1;
    return p->ref[block];
}

pkv_status pkv_seq_add(pkv_block_pool* p, int64_t seq, int length) {
    if (!p || length < 0) return PKV_ERR_INVALID_ARG;
    if (p->seqs.count(seq)) return PKV_ERR_INVALID_ARG;
    const long long nb = p->blocks_for(length);
    if (nb > p->max_blocks_per_seq) return PKV_ERR_INVALID_ARG;
    if (nb > static_cast<long long>(p->free_list.size())) return PKV_ERR_CAPACITY;
    pkv_block_pool::Seq s;
    s.len = length;
    s.blocks.reserve(static_cast<size_t>(nb));
    for (long long i = 0; i < nb; ++i) s.blocks.push_back(p->take());
    p->seqs.emplace(seq, std::move(s));
    return PKV_OK;
}

pkv_status pkv_seq_fork(pkv_block_pool* p, int64_t parent, int64_t child) {
    if (!p) return PKV_ERR_INVALID_ARG;
    auto it = p->seqs.find(parent);
    if (it == p->seqs.end() || p->seqs.count(child)) return PKV_ERR_INVALID_ARG;
    pkv_block_pool::Seq s = it->second;
    for (int32_t b : s.blocks) ++p->ref[b];
    p->seqs.emplace(child, std::move(s));
    return PKV_OK;
}

pkv_status pkv_seq_append(pkv_block_pool* p, int64_t seq, int32_t* cow_src, int32_t* cow_dst, int* n_cow) {
    if (!p || !n_cow) return PKV_ERR_INVALID_ARG;
    *n_cow = 0;
    auto it = p->seqs.find(seq);
    if (it == p->seqs.end()) return PKV_ERR_INVALID_ARG;
    pkv_block_pool::Seq& s = it->second;
    const long long pos = s.len;  // the new token's position
    if (pos % p->block_size == 0) {
        // the token opens a new block
        if (static_cast<long long>(s.blocks.size()) >= p->max_blocks_per_seq) return PKV_ERR_INVALID_ARG;
        if (p->free_list.empty()) return PKV_ERR_CAPACITY;
        s.blocks.push_back(p->take());
    } else {
        const int32_t tail = s.blocks.back();
        if (p->ref[tail] > 1) {
            // shared partial tail: copy before writing
            if (!cow_src || !cow_dst) return PKV_ERR_INVALID_ARG;
            if (p->free_list.empty()) return PKV_ERR_CAPACITY;
            const int32_t fresh = p->take();
            --p->ref[tail];  // still held by the other sharers (count stays >= 1)
            s.blocks.back() = fresh;
            cow_src[0] = tail;
            cow_dst[0] = fresh;
            *n_cow = 1;
        }
    }
    ++s.len;
    return PKV_OK;
}

pkv_status pkv_seq_free(pkv_block_pool* p, int64_t seq) {
    if (!p) return PKV_ERR_INVALID_ARG;
    auto it = p->seqs.find(seq);
    if (it == p->seqs.end()) return PKV_OK;  // already reclaimed: nothing to do
    for (int32_t b : it->second.blocks) p->release(b);
    p->seqs.erase(it);
    return PKV_OK;
}

int pkv_seq_length(const pkv_block_pool* p, int64_t seq) {
    if (!p) return -1;
    auto it = p->seqs.find(seq);
    return it == p->seqs.end() ? -1 : it->second.len;
}

pkv_status pkv_block_tables(const pkv_block_pool* p, const int64_t* seqs, int n, int32_t* block_tables,
                            int32_t* seq_lens) {
    if (!p || n < 0 || (n > 0 && (!seqs || !block_tables || !seq_lens))) return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
        if (!p->seqs.count(seqs[i])) return PKV_ERR_INVALID_ARG;
    const size_t W = static_cast<size_t>(p->max_blocks_per_seq);
    for (int i = 0; i < n; ++i) {
        const pkv_block_pool::Seq& s = p->seqs.find(seqs[i])->second;
        int32_t* row = block_tables + static_cast<size_t>(i) * W;
        for (size_t j = 0; j < W; ++j) row[j] = j < s.blocks.size() ? s.blocks[j] : -1;
        seq_lens[i] = s.len;
    }
    return PKV_OK;
}

}  // extern "C"
