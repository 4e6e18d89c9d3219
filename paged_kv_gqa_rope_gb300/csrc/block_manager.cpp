// Host block manager of the paged KV cache (see include/pa_block_manager.h):
// block ownership with reference counts, prefix-cache reuse of full blocks
// by a chained hash, decode appends and chunked-prefill progress.
#include "pa_block_manager.h"

#include <algorithm>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {

// FNV-1a (64-bit) over the previous block's hash and the block's tokens,
// fed byte by byte in a fixed (little-endian) order whatever the host.
uint64_t block_hash(uint64_t prev, const int32_t *tok, int n) {
    uint64_t h = 14695981039346656037ull;
    auto eat = [&h](uint64_t v, int bytes) {
        for (int i = 0; i < bytes; ++i) {
            h ^= (v >> (8 * i)) & 0xffu;
            h *= 1099511628211ull;
        }
    };
    eat(prev, 8);
    for (int i = 0; i < n; ++i) eat((uint64_t)(uint32_t)tok[i], 4);
    return h;
}

struct Block {
    int ref = 0;
    bool hashed = false;          // registered in by_hash
    uint64_t hash = 0;
    std::vector<int32_t> tokens;  // the full block's tokens, to confirm a hash hit
    bool in_free = false;
    std::list<int>::iterator free_it;
};

struct Seq {
    std::vector<int32_t> tokens;  // prompt, then appended tokens
    std::vector<int32_t> blocks;
    int prompt = 0;
    int computed = 0;             // tokens whose K/V are in the cache
    uint64_t last_full_hash = 0;  // chained hash of the last full block
};

}  // namespace

struct pa_block_manager {
    int nb = 0, bs = 0;
    std::vector<Block> blocks;
    std::list<int> free_list;  // oldest-freed first
    std::unordered_map<uint64_t, int> by_hash;
    std::unordered_map<int64_t, Seq> seqs;

    // A free block for new contents (forgetting any hash it still had).
    int take_free() {
        if (free_list.empty()) return -1;
        const int b = free_list.front();
        free_list.pop_front();
        Block &k = blocks[b];
        k.in_free = false;
        if (k.hashed) {
            auto it = by_hash.find(k.hash);
            if (it != by_hash.end() && it->second == b) by_hash.erase(it);
            k.hashed = false;
            k.tokens.clear();
        }
        k.ref = 1;
        return b;
    }
    void reuse(int b) {
        Block &k = blocks[b];
        if (k.ref == 0 && k.in_free) {
            free_list.erase(k.free_it);
            k.in_free = false;
        }
        ++k.ref;
    }
    void release(int b) {
        Block &k = blocks[b];
        if (--k.ref == 0) {
            free_list.push_back(b);
            k.in_free = true;
            k.free_it = std::prev(free_list.end());
        }
    }
    // Register full block b under hash h (a block with the same contents
    // already registered keeps the entry).
    void set_hash(int b, uint64_t h, const int32_t *tok) {
        if (by_hash.count(h)) return;
        Block &k = blocks[b];
        k.hashed = true;
        k.hash = h;
        k.tokens.assign(tok, tok + bs);
        by_hash[h] = b;
    }
    // The registered block holding exactly these tokens under hash h, or -1.
    int lookup(uint64_t h, const int32_t *tok) const {
        auto it = by_hash.find(h);
        if (it == by_hash.end()) return -1;
        const Block &k = blocks[it->second];
        return std::equal(tok, tok + bs, k.tokens.begin()) ? it->second : -1;
    }
    Seq *find(int64_t id) {
        auto it = seqs.find(id);
        return it == seqs.end() ? nullptr : &it->second;
    }
};

extern "C" {

pa_bm_t pa_bm_create(int num_blocks, int block_size) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    if ((int64_t)num_blocks * block_size > INT32_MAX) return nullptr;  // slots are int32
    pa_block_manager *bm = new (std::nothrow) pa_block_manager;
    if (!bm) return nullptr;
    bm->nb = num_blocks;
    bm->bs = block_size;
    bm->blocks.resize(num_blocks);
    for (int b = 0; b < num_blocks; ++b) {
        bm->free_list.push_back(b);
        bm->blocks[b].in_free = true;
        bm->blocks[b].free_it = std::prev(bm->free_list.end());
    }
    return bm;
}

void pa_bm_destroy(pa_bm_t bm) { delete bm; }

int pa_bm_num_free(pa_bm_t bm) { return bm ? (int)bm->free_list.size() : -1; }

int pa_bm_blocks_needed(pa_bm_t bm, int num_tokens) {
    if (!bm || num_tokens < 0) return -1;
    return (num_tokens + bm->bs - 1) / bm->bs;
}

int pa_bm_allocate(pa_bm_t bm, int64_t seq_id, const int32_t *tokens, int num_tokens,
                   int *num_cached) {
    if (!bm || !tokens || num_tokens <= 0 || !num_cached || bm->find(seq_id)) return PA_ERR_INVALID;
    const int bs = bm->bs;
    const int need = (num_tokens + bs - 1) / bs, full = num_tokens / bs;
    // Matching full blocks, up to the first miss.
    std::vector<int> hits;
    std::vector<uint64_t> h(full);
    uint64_t prev = 0;
    for (int i = 0; i < full; ++i) {
        h[i] = block_hash(prev, tokens + (size_t)i * bs, bs);
        prev = h[i];
        if ((int)hits.size() == i) {
            const int b = bm->lookup(h[i], tokens + (size_t)i * bs);
            if (b >= 0) hits.push_back(b);
        }
    }
    int from_free = need - (int)hits.size();
    for (int b : hits) from_free += bm->blocks[b].ref == 0 ? 1 : 0;
    if (from_free > (int)bm->free_list.size()) return PA_ERR_WORKSPACE;

    Seq s;
    s.tokens.assign(tokens, tokens + num_tokens);
    s.prompt = num_tokens;
    for (int b : hits) {
        bm->reuse(b);
        s.blocks.push_back(b);
    }
    for (int i = (int)hits.size(); i < need; ++i) {
        const int b = bm->take_free();
        s.blocks.push_back(b);
        if (i < full) bm->set_hash(b, h[i], tokens + (size_t)i * bs);
    }
    s.last_full_hash = full > 0 ? h[full - 1] : 0;
    s.computed = std::min((int)hits.size() * bs, num_tokens - 1);
    *num_cached = s.computed;
    bm->seqs.emplace(seq_id, std::move(s));
    return PA_OK;
}

int pa_bm_next_chunk(pa_bm_t bm, int64_t seq_id, int max_tokens, int *num_cached,
                     int *num_new) {
    Seq *s = bm ? bm->find(seq_id) : nullptr;
    if (!s || max_tokens <= 0 || !num_cached || !num_new) return PA_ERR_INVALID;
    *num_cached = s->computed;
    *num_new = std::max(0, std::min(max_tokens, s->prompt - s->computed));
    return PA_OK;
}

int pa_bm_mark_computed(pa_bm_t bm, int64_t seq_id, int num_tokens) {
    Seq *s = bm ? bm->find(seq_id) : nullptr;
    if (!s || num_tokens < 0 || num_tokens > (int)s->tokens.size() - s->computed)
        return PA_ERR_INVALID;
    s->computed += num_tokens;
    return PA_OK;
}

int pa_bm_can_append(pa_bm_t bm, int64_t seq_id) {
    Seq *s = bm ? bm->find(seq_id) : nullptr;
    if (!s) return -PA_ERR_INVALID;
    return (s->tokens.size() % bm->bs) != 0 || !bm->free_list.empty() ? 1 : 0;
}

int pa_bm_append(pa_bm_t bm, int64_t seq_id, int32_t token, int32_t *slot) {
    Seq *s = bm ? bm->find(seq_id) : nullptr;
    if (!s || !slot || s->computed < (int)s->tokens.size()) return PA_ERR_INVALID;
    const int bs = bm->bs;
    const int pos = (int)s->tokens.size();
    if (pos % bs == 0) {
        const int b = bm->take_free();
        if (b < 0) return PA_ERR_WORKSPACE;
        s->blocks.push_back(b);
    }
    s->tokens.push_back(token);
    s->computed = pos + 1;
    const int blk = s->blocks[pos / bs];
    *slot = blk * bs + pos % bs;
    if ((pos + 1) % bs == 0) {  // the block just filled: it can be matched from now on
        const uint64_t h = block_hash(s->last_full_hash, s->tokens.data() + (pos + 1 - bs), bs);
        bm->set_hash(blk, h, s->tokens.data() + (pos + 1 - bs));
        s->last_full_hash = h;
    }
    return PA_OK;
}

int pa_bm_num_tokens(pa_bm_t bm, int64_t seq_id) {
    Seq *s = bm ? bm->find(seq_id) : nullptr;
    return s ? (int)s->tokens.size() : -1;
}

int pa_bm_block_table(pa_bm_t bm, int64_t seq_id, int32_t *table, int max_blocks,
                      int *num_blocks) {
    Seq *s = bm ? bm->find(seq_id) : nullptr;
    if (!s || !num_blocks || max_blocks < 0) return PA_ERR_INVALID;
    const int n = (int)s->blocks.size();
    *num_blocks = n;
    if (n > max_blocks || (n > 0 && !table)) return PA_ERR_INVALID;
    std::copy(s->blocks.begin(), s->blocks.end(), table);
    return PA_OK;
}

int pa_bm_free(pa_bm_t bm, int64_t seq_id) {
    Seq *s = bm ? bm->find(seq_id) : nullptr;
    if (!s) return PA_ERR_INVALID;
    for (auto it = s->blocks.rbegin(); it != s->blocks.rend(); ++it) bm->release(*it);
    bm->seqs.erase(seq_id);
    return PA_OK;
}

}  // extern "C"
