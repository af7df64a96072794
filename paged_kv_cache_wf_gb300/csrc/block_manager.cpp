// block_manager.cpp -- host-side block manager of the paged KV cache (the C ABI in
// include/wf_blocks.h).
//
// ember, "The core idea, in one picture": position p of a sequence lives in block
// table[p / P] at offset p % P.  tiny-vllm-py, "Mental Model": a request grows
// block by block from a shared free list; "Prefix Sharing": requests with a common
// prefix share its blocks, and a shared block that is only partly filled is copied
// before a request appends to it.
//
// Plain C++ over vectors: a LIFO free list, one reference count per block, and a
// hash map from sequence id to (block list, length).  Every call validates first
// and mutates second, so a failing call leaves the manager unchanged.
#include <cstdint>
#include <new>
#include <unordered_map>
#include <utility>
#include <vector>

#include "wf_blocks.h"

struct wf_block_manager {
    struct Seq {
        std::vector<int32_t> blocks;
        int64_t len = 0;
    };
    int32_t N = 0, P = 0;
    std::vector<int32_t> free_list;   // top = back
    std::vector<int32_t> ref;         // per block; 0 = free
    std::unordered_map<int64_t, Seq> seqs;

    int32_t take() {
        const int32_t b = free_list.back();
        free_list.pop_back();
        ref[b] = 1;
        return b;
    }
    void drop(int32_t b) {
        if (--ref[b] == 0) free_list.push_back(b);
    }
};

namespace {

uint64_t splitmix64(uint64_t& state) {
    uint64_t z = (state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

int64_t blocks_for(int64_t len, int32_t P) { return (len + P - 1) / P; }

}  // namespace

extern "C" {

wf_status wf_bm_create(int32_t num_blocks, int32_t block_size, uint64_t shuffle_seed, wf_block_manager** out) {
    if (out == nullptr || num_blocks < 1 || block_size < 1 || block_size > 1024) return WF_ERR_INVALID_ARG;
    wf_block_manager* bm = new (std::nothrow) wf_block_manager();
    if (bm == nullptr) return WF_ERR_INVALID_ARG;
    bm->N = num_blocks;
    bm->P = block_size;
    bm->ref.assign((size_t)num_blocks, 0);
    // the free list is popped from the back: store ids so that the first pops
    // give 0, 1, 2, ... (or the shuffled order)
    std::vector<int32_t> order((size_t)num_blocks);
    for (int32_t i = 0; i < num_blocks; ++i) order[(size_t)i] = i;
    if (shuffle_seed != 0) {
        uint64_t st = shuffle_seed;
        for (int32_t i = num_blocks - 1; i > 0; --i) {   // Fisher-Yates
            const int32_t j = (int32_t)(splitmix64(st) % (uint64_t)(i + 1));
            std::swap(order[(size_t)i], order[(size_t)j]);
        }
    }
    bm->free_list.assign(order.rbegin(), order.rend());
    *out = bm;
    return WF_OK;
}

void wf_bm_destroy(wf_block_manager* bm) { delete bm; }

int32_t wf_bm_num_free(const wf_block_manager* bm) { return bm ? (int32_t)bm->free_list.size() : -1; }

int64_t wf_bm_seq_len(const wf_block_manager* bm, int64_t seq) {
    if (bm == nullptr) return -1;
    auto it = bm->seqs.find(seq);
    return it == bm->seqs.end() ? -1 : it->second.len;
}

int32_t wf_bm_ref_count(const wf_block_manager* bm, int32_t block) {
    if (bm == nullptr || block < 0 || block >= bm->N) return -1;
    return bm->ref[(size_t)block];
}

wf_status wf_bm_append(wf_block_manager* bm, int64_t seq, int32_t n, int64_t* slots, int32_t* cow_pair,
                       int32_t* n_cow) {
    if (bm == nullptr || n < 0 || cow_pair == nullptr || n_cow == nullptr || (n > 0 && slots == nullptr))
        return WF_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    const int64_t len = it == bm->seqs.end() ? 0 : it->second.len;
    const int32_t P = bm->P;
    // a partly filled last block shared with another sequence is copied first
    bool cow = false;
    if (n > 0 && it != bm->seqs.end() && len % P != 0) cow = bm->ref[(size_t)it->second.blocks.back()] > 1;
    const int64_t need = (cow ? 1 : 0) + blocks_for(len + n, P) - blocks_for(len, P);
    if (need > (int64_t)bm->free_list.size()) return WF_ERR_NO_BLOCKS;
    wf_block_manager::Seq& s = bm->seqs[seq];   // creates a new sequence
    *n_cow = 0;
    if (cow) {
        const int32_t src = s.blocks.back();
        const int32_t dst = bm->take();
        bm->drop(src);
        s.blocks.back() = dst;
        cow_pair[0] = src;
        cow_pair[1] = dst;
        *n_cow = 1;
    }
    for (int32_t i = 0; i < n; ++i) {
        const int64_t pos = len + i;
        if (pos % P == 0) s.blocks.push_back(bm->take());
        slots[i] = (int64_t)s.blocks[(size_t)(pos / P)] * P + pos % P;
    }
    s.len = len + n;
    return WF_OK;
}

wf_status wf_bm_fork(wf_block_manager* bm, int64_t parent, int64_t child) {
    if (bm == nullptr || parent == child) return WF_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end() || bm->seqs.count(child) != 0) return WF_ERR_INVALID_ARG;
    wf_block_manager::Seq copy = it->second;
    for (int32_t b : copy.blocks) ++bm->ref[(size_t)b];
    bm->seqs.emplace(child, std::move(copy));
    return WF_OK;
}

wf_status wf_bm_free(wf_block_manager* bm, int64_t seq) {
    if (bm == nullptr) return WF_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return WF_ERR_INVALID_ARG;
    // release in reverse so that the sequence's first block is handed out first again
    for (auto b = it->second.blocks.rbegin(); b != it->second.blocks.rend(); ++b) bm->drop(*b);
    bm->seqs.erase(it);
    return WF_OK;
}

wf_status wf_bm_tables(const wf_block_manager* bm, const int64_t* seqs, int32_t B, int32_t M, int32_t pad_block,
                       int32_t* block_tables, int32_t* seq_lens) {
    if (bm == nullptr || B < 0 || M < 1 || (B > 0 && (seqs == nullptr || block_tables == nullptr || seq_lens == nullptr)))
        return WF_ERR_INVALID_ARG;
    for (int32_t b = 0; b < B; ++b) {
        auto it = bm->seqs.find(seqs[b]);
        if (it == bm->seqs.end() || (int64_t)it->second.blocks.size() > M || it->second.len > INT32_MAX)
            return WF_ERR_INVALID_ARG;
    }
    for (int32_t b = 0; b < B; ++b) {
        const wf_block_manager::Seq& s = bm->seqs.at(seqs[b]);
        int32_t* row = block_tables + (int64_t)b * M;
        for (int32_t j = 0; j < M; ++j) row[j] = j < (int32_t)s.blocks.size() ? s.blocks[(size_t)j] : pad_block;
        seq_lens[b] = (int32_t)s.len;
    }
    return WF_OK;
}

}  // extern "C"
