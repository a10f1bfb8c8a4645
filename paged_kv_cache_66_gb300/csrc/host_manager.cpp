// Host-side block manager: free list with reference counts, per-sequence
// block tables, copy-on-write decisions and a prefix table.
//
// "25. Paged attention and prefix caching": sections "The allocator" (free
// list plus refcounts), "The paged cache" (create / reserve / set_batch /
// fork / free / truncate), "Sharing blocks: forks and copy-on-write" and
// "Prefix caching".  Readings (first-in first-out free list, over-release
// rejected before the decrement, all-or-nothing reserve, the byte layout of
// the hash-chain prefix keys) are stated in include/pagedkv_host.h.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <deque>
#include <list>
#include <new>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "../../include/pagedkv_host.h"
#include "sha256.h"

namespace {

struct Seq {
    std::vector<int32_t> table;
    int64_t length = 0;
};

struct VecHash {
    size_t operator()(const std::vector<int64_t>& v) const noexcept {
        uint64_t h = 1469598103934665603ull;  // FNV-1a over the 8-byte words
        for (int64_t x : v) {
            h ^= static_cast<uint64_t>(x);
            h *= 1099511628211ull;
        }
        return static_cast<size_t>(h);
    }
};

// A hash-chain prefix key (SHA-256 digest).
struct ChainKey {
    uint8_t b[32];
    bool operator==(const ChainKey& o) const noexcept { return std::memcmp(b, o.b, 32) == 0; }
};
struct ChainKeyHash {
    size_t operator()(const ChainKey& k) const noexcept {  // the key is already uniformly distributed
        uint64_t x;
        std::memcpy(&x, k.b, 8);
        return static_cast<size_t>(x);
    }
};

constexpr char kChainDomain[] = "pagedkv.prefix.v1";

ChainKey chain_root(const void* salt, int64_t salt_len) {
    pa_sha256::Hasher hs;
    hs.update(kChainDomain, sizeof(kChainDomain) - 1);
    uint8_t len[8];
    for (int i = 0; i < 8; ++i) len[i] = static_cast<uint8_t>(static_cast<uint64_t>(salt_len) >> (8 * i));
    hs.update(len, 8);
    if (salt_len > 0) hs.update(salt, static_cast<size_t>(salt_len));
    ChainKey k;
    hs.finish(k.b);
    return k;
}

// key of the next full block: the parent key, the block size (u32 LE) and
// each token id (i64 LE)
ChainKey chain_next(const ChainKey& parent, const int64_t* tokens, int block_size) {
    pa_sha256::Hasher hs;
    hs.update(parent.b, 32);
    uint8_t buf[8];
    for (int i = 0; i < 4; ++i) buf[i] = static_cast<uint8_t>(static_cast<uint32_t>(block_size) >> (8 * i));
    hs.update(buf, 4);
    for (int t = 0; t < block_size; ++t) {
        const uint64_t x = static_cast<uint64_t>(tokens[t]);
        for (int i = 0; i < 8; ++i) buf[i] = static_cast<uint8_t>(x >> (8 * i));
        hs.update(buf, 8);
    }
    ChainKey k;
    hs.finish(k.b);
    return k;
}

// A node of the block prefix tree: one cached full block, reached from its parent by an
// edge labelled with the block's token ids.  Node 0 is the root (the empty prefix).
struct TreeNode {
    int32_t parent = -1;
    int32_t block = -1;
    int64_t used = 0;               // recency stamp: larger = more recently used
    std::vector<int64_t> label;     // the block's block_size token ids
    std::unordered_map<std::vector<int64_t>, int32_t, VecHash> children;
};

}  // namespace

struct pa_host {
    int64_t num_blocks = 0;
    int block_size = 0;
    std::deque<int32_t> free_list;
    std::vector<int32_t> refs;
    std::unordered_map<int64_t, Seq> seqs;
    // prefix table: key -> (block, position in the LRU list)
    std::list<std::vector<int64_t>> lru;  // front = least recently used
    std::unordered_map<std::vector<int64_t>, std::pair<int32_t, std::list<std::vector<int64_t>>::iterator>,
                       VecHash>
        entries;
    // hash-chain prefix table: chain key -> (block, position in its own LRU list)
    std::list<ChainKey> hlru;
    std::unordered_map<ChainKey, std::pair<int32_t, std::list<ChainKey>::iterator>, ChainKeyHash> hentries;
    // block prefix tree: nodes (slot 0 the root, freed slots reused), every non-root leaf ordered
    // by (recency stamp, node), and the stamp clock
    std::vector<TreeNode> tnodes = std::vector<TreeNode>(1);
    std::vector<int32_t> tfree;
    std::set<std::pair<int64_t, int32_t>> tleaves;
    int64_t tclock = 0;
    int64_t tcount = 0;

    int64_t blocks_needed(int64_t tokens) const { return (tokens + block_size - 1) / block_size; }

    pa_status allocate(int32_t* out) {
        if (free_list.empty()) return PA_ERR_POOL_EXHAUSTED;
        int32_t b = free_list.front();
        free_list.pop_front();
        refs[b] = 1;
        *out = b;
        return PA_OK;
    }
    pa_status share(int32_t b) {
        if (b < 0 || b >= num_blocks || refs[b] <= 0) return PA_ERR_OVER_RELEASE;
        refs[b] += 1;
        return PA_OK;
    }
    pa_status release(int32_t b) {
        if (b < 0 || b >= num_blocks || refs[b] <= 0) return PA_ERR_OVER_RELEASE;
        refs[b] -= 1;
        if (refs[b] == 0) free_list.push_back(b);
        return PA_OK;
    }
    Seq* find(int64_t id) {
        auto it = seqs.find(id);
        return it == seqs.end() ? nullptr : &it->second;
    }
    const Seq* find(int64_t id) const {
        auto it = seqs.find(id);
        return it == seqs.end() ? nullptr : &it->second;
    }

    // Reserve positions [len, len + n): copy-on-write of shared entries in the
    // written range, then append fresh blocks.  All-or-nothing.
    pa_status reserve(Seq& s, int64_t n, int64_t* pairs, int64_t cap, int64_t* npairs) {
        const int64_t start = s.length, end = s.length + n;
        const int64_t need = blocks_needed(end);
        const int64_t first = start / block_size;
        const int64_t tlen = static_cast<int64_t>(s.table.size());
        const int64_t cow_hi = std::min(tlen, need);
        int64_t cow = 0;
        for (int64_t i = first; i < cow_hi; ++i)
            if (refs[s.table[i]] > 1) ++cow;
        const int64_t grow = std::max<int64_t>(0, need - tlen);
        if (cow + grow > static_cast<int64_t>(free_list.size())) return PA_ERR_POOL_EXHAUSTED;
        if (cow > 0 && (pairs == nullptr || cow > cap)) return PA_ERR_INVALID;
        int64_t k = 0;
        for (int64_t i = first; i < cow_hi; ++i) {
            const int32_t old = s.table[i];
            if (refs[old] > 1) {
                int32_t fresh = -1;
                allocate(&fresh);
                pairs[2 * k] = old;
                pairs[2 * k + 1] = fresh;
                ++k;
                release(old);
                s.table[i] = fresh;
            }
        }
        while (static_cast<int64_t>(s.table.size()) < need) {
            int32_t b = -1;
            allocate(&b);
            s.table.push_back(b);
        }
        if (npairs) *npairs = k;
        return PA_OK;
    }
};

extern "C" {

pa_host* pa_host_create(int64_t num_blocks, int block_size, const int32_t* initial_order) {
    if (num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0) return nullptr;
    pa_host* h = new (std::nothrow) pa_host();
    if (!h) return nullptr;
    h->num_blocks = num_blocks;
    h->block_size = block_size;
    h->refs.assign(static_cast<size_t>(num_blocks), 0);
    if (initial_order) {
        std::vector<char> seen(static_cast<size_t>(num_blocks), 0);
        for (int64_t i = 0; i < num_blocks; ++i) {
            const int32_t b = initial_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete h;
                return nullptr;
            }
            seen[b] = 1;
            h->free_list.push_back(b);
        }
    } else {
        for (int64_t i = 0; i < num_blocks; ++i) h->free_list.push_back(static_cast<int32_t>(i));
    }
    return h;
}

void pa_host_destroy(pa_host* h) { delete h; }

pa_status pa_host_seq_create(pa_host* h, int64_t seq) {
    if (!h) return PA_ERR_INVALID;
    if (h->seqs.count(seq)) return PA_ERR_EXISTS;
    h->seqs.emplace(seq, Seq());
    return PA_OK;
}

pa_status pa_host_reserve(pa_host* h, int64_t seq, int64_t new_tokens, int64_t* pairs_out,
                          int64_t pairs_cap, int64_t* num_pairs) {
    if (!h || new_tokens < 0) return PA_ERR_INVALID;
    Seq* s = h->find(seq);
    if (!s) return PA_ERR_NOT_FOUND;
    int64_t k = 0;
    pa_status st = h->reserve(*s, new_tokens, pairs_out, pairs_cap, &k);
    if (num_pairs) *num_pairs = (st == PA_OK) ? k : 0;
    return st;
}

pa_status pa_host_slots(pa_host* h, int64_t seq, int64_t start, int64_t n, int64_t* slots_out) {
    if (!h || start < 0 || n < 0 || (n > 0 && !slots_out)) return PA_ERR_INVALID;
    const Seq* s = h->find(seq);
    if (!s) return PA_ERR_NOT_FOUND;
    const int64_t b = h->block_size;
    if (n > 0 && (start + n - 1) / b >= static_cast<int64_t>(s->table.size())) return PA_ERR_INVALID;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t p = start + i;
        slots_out[i] = static_cast<int64_t>(s->table[p / b]) * b + p % b;
    }
    return PA_OK;
}

pa_status pa_host_advance(pa_host* h, int64_t seq, int64_t n) {
    if (!h || n < 0) return PA_ERR_INVALID;
    Seq* s = h->find(seq);
    if (!s) return PA_ERR_NOT_FOUND;
    if (h->blocks_needed(s->length + n) > static_cast<int64_t>(s->table.size())) return PA_ERR_INVALID;
    s->length += n;
    return PA_OK;
}

pa_status pa_host_fork(pa_host* h, int64_t parent, int64_t child) {
    if (!h) return PA_ERR_INVALID;
    const Seq* p = h->find(parent);
    if (!p) return PA_ERR_NOT_FOUND;
    if (h->seqs.count(child)) return PA_ERR_EXISTS;
    Seq c = *p;
    for (int32_t b : c.table) h->refs[b] += 1;  // blocks of a live table are live
    h->seqs.emplace(child, std::move(c));
    return PA_OK;
}

pa_status pa_host_free(pa_host* h, int64_t seq) {
    if (!h) return PA_ERR_INVALID;
    auto it = h->seqs.find(seq);
    if (it == h->seqs.end()) return PA_ERR_NOT_FOUND;
    for (int32_t b : it->second.table) h->release(b);
    h->seqs.erase(it);
    return PA_OK;
}

pa_status pa_host_truncate(pa_host* h, int64_t seq, int64_t length) {
    if (!h || length < 0) return PA_ERR_INVALID;
    Seq* s = h->find(seq);
    if (!s) return PA_ERR_NOT_FOUND;
    const int64_t keep = h->blocks_needed(length);
    if (keep > static_cast<int64_t>(s->table.size())) return PA_ERR_INVALID;
    for (size_t i = static_cast<size_t>(keep); i < s->table.size(); ++i) h->release(s->table[i]);
    s->table.resize(static_cast<size_t>(keep));
    s->length = length;
    return PA_OK;
}

pa_status pa_host_length(const pa_host* h, int64_t seq, int64_t* length) {
    if (!h || !length) return PA_ERR_INVALID;
    const Seq* s = h->find(seq);
    if (!s) return PA_ERR_NOT_FOUND;
    *length = s->length;
    return PA_OK;
}

pa_status pa_host_table(const pa_host* h, int64_t seq, int32_t* out, int64_t cap, int64_t* n) {
    if (!h || !n) return PA_ERR_INVALID;
    const Seq* s = h->find(seq);
    if (!s) return PA_ERR_NOT_FOUND;
    const int64_t len = static_cast<int64_t>(s->table.size());
    *n = len;
    if (len > 0 && (!out || cap < len)) return PA_ERR_INVALID;
    if (len > 0) std::memcpy(out, s->table.data(), static_cast<size_t>(len) * sizeof(int32_t));
    return PA_OK;
}

int64_t pa_host_num_free(const pa_host* h) { return h ? static_cast<int64_t>(h->free_list.size()) : -1; }
int64_t pa_host_num_blocks(const pa_host* h) { return h ? h->num_blocks : -1; }

int32_t pa_host_refcount(const pa_host* h, int64_t block) {
    if (!h || block < 0 || block >= h->num_blocks) return -1;
    return h->refs[static_cast<size_t>(block)];
}

pa_status pa_host_batch(const pa_host* h, const int64_t* seqs, int64_t batch, int32_t* tables_out,
                        int64_t stride, int32_t* lens_out, int64_t* width) {
    if (!h || batch < 0 || (batch > 0 && (!seqs || !tables_out || !lens_out))) return PA_ERR_INVALID;
    int64_t w = 1;
    for (int64_t i = 0; i < batch; ++i) {
        const Seq* s = h->find(seqs[i]);
        if (!s) return PA_ERR_NOT_FOUND;
        w = std::max<int64_t>(w, static_cast<int64_t>(s->table.size()));
    }
    if (width) *width = w;
    if (stride < w) return PA_ERR_INVALID;
    for (int64_t i = 0; i < batch; ++i) {
        const Seq* s = h->find(seqs[i]);
        int32_t* row = tables_out + i * stride;
        const size_t n = s->table.size();
        if (n) std::memcpy(row, s->table.data(), n * sizeof(int32_t));
        std::fill(row + n, row + stride, 0);
        lens_out[i] = static_cast<int32_t>(s->length);
    }
    return PA_OK;
}

pa_status pa_host_decode_step(pa_host* h, const int64_t* seqs, int64_t batch, int64_t* slots_out,
                              int64_t* pairs_out, int64_t pairs_cap, int64_t* num_pairs,
                              int32_t* tables_out, int64_t stride, int32_t* lens_out, int64_t* width) {
    if (!h || batch < 0 || (batch > 0 && (!seqs || !slots_out))) return PA_ERR_INVALID;
    std::vector<Seq*> ss(static_cast<size_t>(batch));
    for (int64_t i = 0; i < batch; ++i) {
        ss[i] = h->find(seqs[i]);
        if (!ss[i]) return PA_ERR_NOT_FOUND;
        for (int64_t j = 0; j < i; ++j)
            if (ss[j] == ss[i]) return PA_ERR_INVALID;  // a sequence appears once per step
    }
    int64_t total = 0;
    for (int64_t i = 0; i < batch; ++i) {
        int64_t k = 0;
        int64_t* dst = pairs_out ? pairs_out + 2 * total : nullptr;
        pa_status st = h->reserve(*ss[i], 1, dst, pairs_cap - total, &k);
        if (st != PA_OK) {
            if (num_pairs) *num_pairs = total;
            return st;
        }
        total += k;
    }
    if (num_pairs) *num_pairs = total;
    const int64_t b = h->block_size;
    for (int64_t i = 0; i < batch; ++i) {
        Seq& s = *ss[i];
        const int64_t p = s.length;
        slots_out[i] = static_cast<int64_t>(s.table[p / b]) * b + p % b;
        s.length += 1;
    }
    if (tables_out || lens_out) return pa_host_batch(h, seqs, batch, tables_out, stride, lens_out, width);
    return PA_OK;
}

pa_status pa_host_prefix_attach(pa_host* h, int64_t seq, const int64_t* prompt, int64_t n,
                                int64_t* reused) {
    if (!h || n < 0 || (n > 0 && !prompt)) return PA_ERR_INVALID;
    if (h->seqs.count(seq)) return PA_ERR_EXISTS;
    Seq s;
    const int64_t size = h->block_size;
    int64_t r = 0;
    std::vector<int64_t> key;
    while (r + size <= n - 1) {
        key.assign(prompt, prompt + r + size);
        auto it = h->entries.find(key);
        if (it == h->entries.end()) break;
        h->lru.splice(h->lru.end(), h->lru, it->second.second);  // most recently used
        h->refs[it->second.first] += 1;                         // cached blocks are live
        s.table.push_back(it->second.first);
        r += size;
    }
    s.length = r;
    h->seqs.emplace(seq, std::move(s));
    if (reused) *reused = r;
    return PA_OK;
}

pa_status pa_host_prefix_remember(pa_host* h, int64_t seq, const int64_t* tokens, int64_t n) {
    if (!h || n < 0 || (n > 0 && !tokens)) return PA_ERR_INVALID;
    const Seq* s = h->find(seq);
    if (!s) return PA_ERR_NOT_FOUND;
    const int64_t size = h->block_size;
    const int64_t full = n / size;
    if (full > static_cast<int64_t>(s->table.size())) return PA_ERR_INVALID;
    for (int64_t i = 0; i < full; ++i) {
        std::vector<int64_t> key(tokens, tokens + (i + 1) * size);
        if (h->entries.count(key)) continue;
        const int32_t b = s->table[static_cast<size_t>(i)];
        h->refs[b] += 1;
        h->lru.push_back(key);
        auto pos = std::prev(h->lru.end());
        h->entries.emplace(std::move(key), std::make_pair(b, pos));
    }
    return PA_OK;
}

pa_status pa_host_prefix_evict(pa_host* h, int64_t blocks_wanted) {
    if (!h) return PA_ERR_INVALID;
    for (auto it = h->lru.begin(); it != h->lru.end();) {
        if (static_cast<int64_t>(h->free_list.size()) >= blocks_wanted) break;
        auto e = h->entries.find(*it);
        const int32_t b = e->second.first;
        if (h->refs[b] == 1) {
            h->entries.erase(e);
            it = h->lru.erase(it);
            h->release(b);
        } else {
            ++it;
        }
    }
    return PA_OK;
}

int64_t pa_host_prefix_entries(const pa_host* h) { return h ? static_cast<int64_t>(h->entries.size()) : -1; }

pa_status pa_prefix_chain_keys(const int64_t* tokens, int64_t n, int block_size, const void* salt, int64_t salt_len,
                               uint8_t* keys_out) {
    if (n < 0 || block_size <= 0 || salt_len < 0 || (n > 0 && !tokens) || (salt_len > 0 && !salt))
        return PA_ERR_INVALID;
    const int64_t full = n / block_size;
    if (full > 0 && !keys_out) return PA_ERR_INVALID;
    ChainKey k = chain_root(salt, salt_len);
    for (int64_t i = 0; i < full; ++i) {
        k = chain_next(k, tokens + i * block_size, block_size);
        std::memcpy(keys_out + 32 * i, k.b, 32);
    }
    return PA_OK;
}

pa_status pa_host_hprefix_attach(pa_host* h, int64_t seq, const int64_t* prompt, int64_t n, const void* salt,
                                 int64_t salt_len, int64_t* reused) {
    if (!h || n < 0 || salt_len < 0 || (n > 0 && !prompt) || (salt_len > 0 && !salt)) return PA_ERR_INVALID;
    if (h->seqs.count(seq)) return PA_ERR_EXISTS;
    Seq s;
    const int64_t size = h->block_size;
    int64_t r = 0;
    ChainKey k = chain_root(salt, salt_len);
    while (r + size <= n - 1) {  // at least one prompt token is left to prefill
        k = chain_next(k, prompt + r, h->block_size);
        auto it = h->hentries.find(k);
        if (it == h->hentries.end()) break;
        h->hlru.splice(h->hlru.end(), h->hlru, it->second.second);  // most recently used
        h->refs[it->second.first] += 1;
        s.table.push_back(it->second.first);
        r += size;
    }
    s.length = r;
    h->seqs.emplace(seq, std::move(s));
    if (reused) *reused = r;
    return PA_OK;
}

pa_status pa_host_hprefix_remember(pa_host* h, int64_t seq, const int64_t* tokens, int64_t n, const void* salt,
                                   int64_t salt_len) {
    if (!h || n < 0 || salt_len < 0 || (n > 0 && !tokens) || (salt_len > 0 && !salt)) return PA_ERR_INVALID;
    const Seq* s = h->find(seq);
    if (!s) return PA_ERR_NOT_FOUND;
    const int64_t size = h->block_size;
    const int64_t full = n / size;
    if (full > static_cast<int64_t>(s->table.size())) return PA_ERR_INVALID;
    ChainKey k = chain_root(salt, salt_len);
    for (int64_t i = 0; i < full; ++i) {
        k = chain_next(k, tokens + i * size, h->block_size);
        if (h->hentries.count(k)) continue;
        const int32_t b = s->table[static_cast<size_t>(i)];
        h->refs[b] += 1;
        h->hlru.push_back(k);
        h->hentries.emplace(k, std::make_pair(b, std::prev(h->hlru.end())));
    }
    return PA_OK;
}

pa_status pa_host_hprefix_evict(pa_host* h, int64_t blocks_wanted) {
    if (!h) return PA_ERR_INVALID;
    for (auto it = h->hlru.begin(); it != h->hlru.end();) {
        if (static_cast<int64_t>(h->free_list.size()) >= blocks_wanted) break;
        auto e = h->hentries.find(*it);
        const int32_t b = e->second.first;
        if (h->refs[b] == 1) {
            h->hentries.erase(e);
            it = h->hlru.erase(it);
            h->release(b);
        } else {
            ++it;
        }
    }
    return PA_OK;
}

int64_t pa_host_hprefix_entries(const pa_host* h) { return h ? static_cast<int64_t>(h->hentries.size()) : -1; }

int64_t pa_host_hprefix_blocks(const pa_host* h, int32_t* blocks_out, int64_t capacity) {
    if (!h || capacity < 0 || (capacity > 0 && !blocks_out)) return -1;
    int64_t i = 0;
    for (const ChainKey& k : h->hlru) {
        if (i < capacity) blocks_out[i] = h->hentries.find(k)->second.first;
        ++i;
    }
    return i;
}

// ------------------------------------------------------------------ block prefix tree
// The radix-tree form of the prefix table: rules in include/pagedkv_host.h.

namespace {

bool tree_is_leaf(const pa_host* h, int32_t node) { return node != 0 && h->tnodes[node].children.empty(); }

// stamp `node` most recently used, keeping the leaf order in step
void tree_touch(pa_host* h, int32_t node) {
    TreeNode& t = h->tnodes[node];
    const bool leaf = tree_is_leaf(h, node);
    if (leaf) h->tleaves.erase({t.used, node});
    t.used = ++h->tclock;
    if (leaf) h->tleaves.insert({t.used, node});
}

}  // namespace

pa_status pa_host_tprefix_attach(pa_host* h, int64_t seq, const int64_t* prompt, int64_t n, int64_t* reused) {
    if (!h || n < 0 || (n > 0 && !prompt)) return PA_ERR_INVALID;
    if (h->seqs.count(seq)) return PA_ERR_EXISTS;
    const int64_t size = h->block_size;
    std::vector<int32_t> path;
    int32_t node = 0;
    std::vector<int64_t> label;
    for (int64_t r = 0; r + size <= n - 1; r += size) {  // at least one prompt token is left to prefill
        label.assign(prompt + r, prompt + r + size);
        auto it = h->tnodes[node].children.find(label);
        if (it == h->tnodes[node].children.end()) break;
        node = it->second;
        path.push_back(node);
    }
    Seq s;
    for (int32_t v : path) {
        tree_touch(h, v);
        h->refs[h->tnodes[v].block] += 1;  // cached blocks are live
        s.table.push_back(h->tnodes[v].block);
    }
    s.length = static_cast<int64_t>(path.size()) * size;
    if (reused) *reused = s.length;
    h->seqs.emplace(seq, std::move(s));
    return PA_OK;
}

pa_status pa_host_tprefix_remember(pa_host* h, int64_t seq, const int64_t* tokens, int64_t n) {
    if (!h || n < 0 || (n > 0 && !tokens)) return PA_ERR_INVALID;
    const Seq* s = h->find(seq);
    if (!s) return PA_ERR_NOT_FOUND;
    const int64_t size = h->block_size;
    const int64_t full = n / size;
    if (full > static_cast<int64_t>(s->table.size())) return PA_ERR_INVALID;
    int32_t node = 0;
    std::vector<int64_t> label;
    for (int64_t i = 0; i < full; ++i) {
        label.assign(tokens + i * size, tokens + (i + 1) * size);
        auto it = h->tnodes[node].children.find(label);
        if (it != h->tnodes[node].children.end()) {  // cached: descend, recency unchanged
            node = it->second;
            continue;
        }
        int32_t v;
        if (!h->tfree.empty()) {
            v = h->tfree.back();
            h->tfree.pop_back();
        } else {
            v = static_cast<int32_t>(h->tnodes.size());
            h->tnodes.emplace_back();
        }
        if (tree_is_leaf(h, node)) h->tleaves.erase({h->tnodes[node].used, node});  // gains a child
        TreeNode& t = h->tnodes[v];
        t.parent = node;
        t.block = s->table[static_cast<size_t>(i)];
        t.used = ++h->tclock;
        t.label = label;
        t.children.clear();
        h->tnodes[node].children.emplace(label, v);
        h->tleaves.insert({t.used, v});
        h->refs[t.block] += 1;  // the tree's own reference
        ++h->tcount;
        node = v;
    }
    return PA_OK;
}

pa_status pa_host_tprefix_evict(pa_host* h, int64_t blocks_wanted) {
    if (!h) return PA_ERR_INVALID;
    // Leaves ahead of the cursor are held by a sequence; evicting other leaves does not change
    // that, so the scan never has to look back -- except at a parent that just became a leaf
    // with an older stamp, where it resumes.
    auto it = h->tleaves.begin();
    while (static_cast<int64_t>(h->free_list.size()) < blocks_wanted && it != h->tleaves.end()) {
        const int32_t v = it->second;
        TreeNode& t = h->tnodes[v];
        if (h->refs[t.block] != 1) {
            ++it;
            continue;
        }
        const int32_t parent = t.parent;
        h->tnodes[parent].children.erase(t.label);
        it = h->tleaves.erase(it);
        h->release(t.block);
        t.label.clear();
        t.block = -1;
        h->tfree.push_back(v);
        --h->tcount;
        if (tree_is_leaf(h, parent)) {
            auto ins = h->tleaves.insert({h->tnodes[parent].used, parent}).first;
            if (it == h->tleaves.end() || *ins < *it) it = ins;
        }
    }
    return PA_OK;
}

int64_t pa_host_tprefix_nodes(const pa_host* h) { return h ? h->tcount : -1; }

int64_t pa_host_tprefix_blocks(const pa_host* h, int32_t* blocks_out, int64_t capacity) {
    if (!h || capacity < 0 || (capacity > 0 && !blocks_out)) return -1;
    std::vector<int32_t> blocks;
    for (size_t v = 1; v < h->tnodes.size(); ++v)
        if (h->tnodes[v].block >= 0) blocks.push_back(h->tnodes[v].block);
    std::sort(blocks.begin(), blocks.end());
    for (int64_t i = 0; i < static_cast<int64_t>(blocks.size()) && i < capacity; ++i) blocks_out[i] = blocks[i];
    return static_cast<int64_t>(blocks.size());
}

}  // extern "C"
