// pa_block_manager.cpp -- host-side block manager (include/pa_block_manager.h).
//
// The pool keeps, per block, its reference count, whether it carries a
// prefix hash, and its links in the free queue.  The free queue is an
// intrusive doubly linked list over the block ids (prev/next arrays), so
// taking from the head, appending to either end and removing a prefix-cache
// hit from the middle are all O(1) ("vLLM intro part 2", section 6.2: why the
// free queue is a doubly linked list).  Hashes map to the blocks registered
// under them, in registration order; a lookup takes the first.
#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pa_block_manager.h"

namespace {

struct Hash32 {
    uint8_t b[PA_BM_HASH_BYTES];
    bool operator==(const Hash32& o) const { return std::memcmp(b, o.b, sizeof b) == 0; }
};
struct Hash32Fn {
    size_t operator()(const Hash32& h) const {
        uint64_t x;
        std::memcpy(&x, h.b, sizeof x);     // a cryptographic digest: any 8 bytes spread well
        return static_cast<size_t>(x);
    }
};

struct Request {
    std::vector<int32_t> blocks;
    std::vector<Hash32> hashes;   // hashes of its full prompt blocks
    int64_t num_tokens = 0;
    int32_t need = 0;             // blocks its tokens take
    uint32_t epoch = 0;           // changes whenever an existing table entry changes
    bool swapped = false;         // swapped out: host[j] >= 0 names the host block of entry j,
    std::vector<int32_t> host;    // whose GPU entry blocks[j] is then -1
};

}  // namespace

struct pa_bm {
    int32_t nb = 0, bs = 0;
    std::vector<int32_t> ref, prev, next;
    std::vector<uint8_t> queued, hashed;
    std::vector<Hash32> hash;
    int32_t head = -1, tail = -1, nfree = 0;
    std::unordered_map<Hash32, std::vector<int32_t>, Hash32Fn> cached;
    std::unordered_map<int64_t, Request> reqs;
    uint32_t next_epoch = 0;      // fresh epochs for new requests and copy-on-write
    int32_t nh = 0;               // host blocks for swapping, 0 .. nh-1
    std::deque<int32_t> host_free;   // free host blocks, head = next to be handed out
    int32_t nswapped = 0;

    // ---- free queue ----
    void push_back(int32_t b) {
        prev[b] = tail; next[b] = -1;
        if (tail >= 0) next[tail] = b; else head = b;
        tail = b; queued[b] = 1; ++nfree;
    }
    void push_front(int32_t b) {
        next[b] = head; prev[b] = -1;
        if (head >= 0) prev[head] = b; else tail = b;
        head = b; queued[b] = 1; ++nfree;
    }
    void unlink(int32_t b) {
        if (prev[b] >= 0) next[prev[b]] = next[b]; else head = next[b];
        if (next[b] >= 0) prev[next[b]] = prev[b]; else tail = prev[b];
        prev[b] = next[b] = -1; queued[b] = 0; --nfree;
    }

    // ---- pool operations ----
    void evict(int32_t b) {
        if (!hashed[b]) return;
        auto it = cached.find(hash[b]);
        if (it != cached.end()) {
            auto& ids = it->second;
            for (size_t k = 0; k < ids.size(); ++k)
                if (ids[k] == b) { ids.erase(ids.begin() + static_cast<long>(k)); break; }
            if (ids.empty()) cached.erase(it);
        }
        hashed[b] = 0;
    }
    int32_t take() {                                   // caller checked nfree > 0
        const int32_t b = head;
        unlink(b);
        evict(b);
        ref[b] += 1;
        return b;
    }
    void release(int32_t b) {
        ref[b] -= 1;
        if (ref[b] == 0) {
            if (hashed[b]) push_back(b); else push_front(b);
        }
    }
    void touch(int32_t b) {
        if (ref[b] == 0) unlink(b);
        ref[b] += 1;
    }
    void cache_block(int32_t b, const Hash32& h) {
        if (hashed[b]) return;
        hash[b] = h;
        hashed[b] = 1;
        cached[h].push_back(b);
    }
    int32_t lookup(const Hash32& h) const {
        auto it = cached.find(h);
        return (it == cached.end() || it->second.empty()) ? -1 : it->second.front();
    }
    bool complete(Request& r) {
        const int32_t missing = r.need - static_cast<int32_t>(r.blocks.size());
        if (missing > nfree) return false;
        const size_t start = r.blocks.size();
        for (int32_t k = 0; k < missing; ++k) r.blocks.push_back(take());
        for (size_t j = start; j < r.hashes.size(); ++j) cache_block(r.blocks[j], r.hashes[j]);
        return true;
    }
};

extern "C" {

pa_bm* pa_bm_create(int32_t num_blocks, int32_t block_size, const int32_t* order) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    pa_bm* m = new (std::nothrow) pa_bm;
    if (!m) return nullptr;
    try {
        m->nb = num_blocks;
        m->bs = block_size;
        m->ref.assign(num_blocks, 0);
        m->prev.assign(num_blocks, -1);
        m->next.assign(num_blocks, -1);
        m->queued.assign(num_blocks, 0);
        m->hashed.assign(num_blocks, 0);
        m->hash.resize(num_blocks);
        for (int32_t k = 0; k < num_blocks; ++k) {
            const int32_t b = order ? order[k] : k;
            if (b < 0 || b >= num_blocks || m->queued[b]) { delete m; return nullptr; }   // not a permutation
            m->push_back(b);
        }
    } catch (...) {
        delete m;
        return nullptr;
    }
    return m;
}

void pa_bm_destroy(pa_bm* m) { delete m; }

int32_t pa_bm_num_free(const pa_bm* m) { return m ? m->nfree : -1; }

int32_t pa_bm_ref_cnt(const pa_bm* m, int32_t block) {
    return (m && block >= 0 && block < m->nb) ? m->ref[block] : -1;
}

int32_t pa_bm_free_queue(const pa_bm* m, int32_t* ids, uint8_t* has_hash, int32_t cap) {
    if (!m) return -1;
    int32_t k = 0;
    for (int32_t b = m->head; b >= 0; b = m->next[b], ++k) {
        if (k < cap) {
            if (ids) ids[k] = b;
            if (has_hash) has_hash[k] = m->hashed[b];
        }
    }
    return k;
}

pa_bm_status pa_bm_allocate(pa_bm* m, int64_t req, int32_t num_tokens, const uint8_t* hashes,
                            int32_t num_hashes, int32_t* num_cached_tokens) {
    if (!m || num_tokens < 0 || num_hashes < 0 || (num_hashes > 0 && !hashes)) return PA_BM_INVALID_ARG;
    if (m->reqs.count(req)) return PA_BM_BAD_REQUEST;
    try {
        Request r;
        r.epoch = m->next_epoch++;
        r.num_tokens = num_tokens;
        r.need = static_cast<int32_t>((static_cast<int64_t>(num_tokens) + m->bs - 1) / m->bs);
        const int32_t nh = num_hashes < r.need ? num_hashes : r.need;
        r.hashes.resize(nh);
        for (int32_t j = 0; j < nh; ++j) std::memcpy(r.hashes[j].b, hashes + static_cast<size_t>(j) * PA_BM_HASH_BYTES,
                                                     PA_BM_HASH_BYTES);
        // prefix hits, from block 0 up to the first miss
        for (int32_t j = 0; j < nh; ++j) {
            const int32_t b = m->lookup(r.hashes[j]);
            if (b < 0) break;
            m->touch(b);
            r.blocks.push_back(b);
        }
        if (num_cached_tokens) *num_cached_tokens = static_cast<int32_t>(r.blocks.size()) * m->bs;
        Request& stored = m->reqs.emplace(req, std::move(r)).first->second;
        return m->complete(stored) ? PA_BM_OK : PA_BM_WAIT;
    } catch (...) {
        return PA_BM_INVALID_ARG;
    }
}

pa_bm_status pa_bm_resume(pa_bm* m, int64_t req) {
    if (!m) return PA_BM_INVALID_ARG;
    auto it = m->reqs.find(req);
    if (it == m->reqs.end()) return PA_BM_BAD_REQUEST;
    return m->complete(it->second) ? PA_BM_OK : PA_BM_WAIT;
}

pa_bm_status pa_bm_fork(pa_bm* m, int64_t parent, int64_t child) {
    if (!m) return PA_BM_INVALID_ARG;
    auto it = m->reqs.find(parent);
    if (it == m->reqs.end() || m->reqs.count(child)) return PA_BM_BAD_REQUEST;
    const Request& p = it->second;
    if (p.swapped || static_cast<int32_t>(p.blocks.size()) != p.need) return PA_BM_BAD_REQUEST;
    try {
        Request c;
        c.epoch = m->next_epoch++;
        c.blocks = p.blocks;
        c.num_tokens = p.num_tokens;
        c.need = p.need;
        for (int32_t b : c.blocks) m->ref[b] += 1;
        m->reqs.emplace(child, std::move(c));
    } catch (...) {
        return PA_BM_INVALID_ARG;
    }
    return PA_BM_OK;
}

pa_bm_status pa_bm_append_slots(pa_bm* m, int32_t n, const int64_t* reqs, int64_t* slot_mapping,
                                int64_t* pairs, int32_t pair_cap, int32_t* num_pairs, int32_t* num_done) {
    if (!m || n < 0 || (n > 0 && (!reqs || !slot_mapping)) || pair_cap < 0 || (pair_cap > 0 && !pairs))
        return PA_BM_INVALID_ARG;
    int32_t np = 0, k = 0;
    pa_bm_status st = PA_BM_OK;
    for (; k < n; ++k) {
        auto it = m->reqs.find(reqs[k]);
        if (it == m->reqs.end()) { st = PA_BM_BAD_REQUEST; break; }
        Request& r = it->second;
        if (r.swapped || static_cast<int32_t>(r.blocks.size()) != r.need) { st = PA_BM_BAD_REQUEST; break; }
        const int64_t j = r.num_tokens / m->bs;
        const int32_t off = static_cast<int32_t>(r.num_tokens % m->bs);
        if (off == 0) {
            if (m->nfree < 1) { st = PA_BM_NO_SPACE; break; }
            r.blocks.push_back(m->take());
            r.need += 1;
        } else {
            const int32_t old = r.blocks[static_cast<size_t>(j)];
            if (m->ref[old] > 1) {                          // shared and partly filled: copy on write
                if (m->nfree < 1) { st = PA_BM_NO_SPACE; break; }
                if (np >= pair_cap) { st = PA_BM_INVALID_ARG; break; }
                const int32_t fresh = m->take();           // 1. a new block
                pairs[2 * np] = old;                       // 2. copy old -> new
                pairs[2 * np + 1] = fresh;
                ++np;
                r.blocks[static_cast<size_t>(j)] = fresh;  // 3. repoint the table
                m->ref[old] -= 1;                          // 4. one reference less
                r.epoch = m->next_epoch++;
            }
        }
        r.num_tokens += 1;
        slot_mapping[k] = static_cast<int64_t>(r.blocks[static_cast<size_t>(j)]) * m->bs + off;
    }
    if (num_pairs) *num_pairs = np;
    if (num_done) *num_done = k;
    return st;
}

pa_bm_status pa_bm_cache_block(pa_bm* m, int64_t req, int32_t j, const uint8_t* hash) {
    if (!m || !hash) return PA_BM_INVALID_ARG;
    auto it = m->reqs.find(req);
    if (it == m->reqs.end() || it->second.swapped) return PA_BM_BAD_REQUEST;
    if (j < 0 || j >= static_cast<int32_t>(it->second.blocks.size())) return PA_BM_INVALID_ARG;
    Hash32 h;
    std::memcpy(h.b, hash, PA_BM_HASH_BYTES);
    try {
        m->cache_block(it->second.blocks[static_cast<size_t>(j)], h);
    } catch (...) {
        return PA_BM_INVALID_ARG;
    }
    return PA_BM_OK;
}

pa_bm_status pa_bm_free(pa_bm* m, int64_t req) {
    if (!m) return PA_BM_INVALID_ARG;
    auto it = m->reqs.find(req);
    if (it == m->reqs.end()) return PA_BM_BAD_REQUEST;
    const std::vector<int32_t>& bl = it->second.blocks;
    for (size_t k = bl.size(); k-- > 0;)                        // last block first
        if (bl[k] >= 0) m->release(bl[k]);
    if (it->second.swapped) {                                    // its host blocks, in table order
        for (int32_t h : it->second.host)
            if (h >= 0) m->host_free.push_back(h);
        m->nswapped -= 1;
    }
    m->reqs.erase(it);
    return PA_BM_OK;
}

int64_t pa_bm_num_tokens(const pa_bm* m, int64_t req) {
    if (!m) return -1;
    auto it = m->reqs.find(req);
    return it == m->reqs.end() ? -1 : it->second.num_tokens;
}

int32_t pa_bm_block_table(const pa_bm* m, int64_t req, int32_t* out, int32_t cap) {
    if (!m) return -1;
    auto it = m->reqs.find(req);
    if (it == m->reqs.end() || it->second.swapped) return -1;
    const std::vector<int32_t>& bl = it->second.blocks;
    const int32_t n = static_cast<int32_t>(bl.size());
    if (!out) cap = 0;                                          // size query
    for (int32_t k = 0; k < n && k < cap; ++k) out[k] = bl[static_cast<size_t>(k)];
    return n;
}

pa_bm_status pa_bm_block_tables(const pa_bm* m, int32_t n, const int64_t* reqs, int32_t* out,
                                int32_t max_blocks, int32_t pad) {
    if (!m || n < 0 || max_blocks < 0 || (n > 0 && (!reqs || !out))) return PA_BM_INVALID_ARG;
    for (int32_t k = 0; k < n; ++k) {
        auto it = m->reqs.find(reqs[k]);
        if (it == m->reqs.end() || it->second.swapped) return PA_BM_BAD_REQUEST;
        const std::vector<int32_t>& bl = it->second.blocks;
        if (static_cast<int64_t>(bl.size()) > max_blocks) return PA_BM_INVALID_ARG;
        int32_t* row = out + static_cast<size_t>(k) * max_blocks;
        size_t j = 0;
        for (; j < bl.size(); ++j) row[j] = bl[j];
        for (; j < static_cast<size_t>(max_blocks); ++j) row[j] = pad;
    }
    return PA_BM_OK;
}

pa_bm_status pa_bm_block_tables_update(const pa_bm* m, int32_t n, const int64_t* reqs, int32_t* out,
                                       int32_t max_blocks, int32_t pad, pa_bm_row* rows) {
    if (!m || n < 0 || max_blocks < 0 || (n > 0 && (!reqs || !out || !rows))) return PA_BM_INVALID_ARG;
    for (int32_t k = 0; k < n; ++k) {
        auto it = m->reqs.find(reqs[k]);
        if (it == m->reqs.end() || it->second.swapped) return PA_BM_BAD_REQUEST;
        const Request& r = it->second;
        const int32_t len = static_cast<int32_t>(r.blocks.size());
        if (len > max_blocks) return PA_BM_INVALID_ARG;
        int32_t* row = out + static_cast<size_t>(k) * max_blocks;
        pa_bm_row& st = rows[k];
        int32_t from = 0;
        if (st.len >= 0 && st.len <= len && st.req == reqs[k] && st.epoch == r.epoch) {
            from = st.len;                                  // same table, grown by appends
        } else {
            for (int32_t j = len; j < max_blocks; ++j) row[j] = pad;
        }
        for (int32_t j = from; j < len; ++j) row[j] = r.blocks[static_cast<size_t>(j)];
        st.req = reqs[k];
        st.epoch = r.epoch;
        st.len = len;
    }
    return PA_BM_OK;
}

pa_bm_status pa_bm_set_host_pool(pa_bm* m, int32_t num_host_blocks, const int32_t* order) {
    if (!m || num_host_blocks < 0) return PA_BM_INVALID_ARG;
    if (m->nswapped > 0) return PA_BM_BAD_REQUEST;
    try {
        std::vector<uint8_t> seen(static_cast<size_t>(num_host_blocks), 0);
        std::deque<int32_t> q;
        for (int32_t k = 0; k < num_host_blocks; ++k) {
            const int32_t h = order ? order[k] : k;
            if (h < 0 || h >= num_host_blocks || seen[static_cast<size_t>(h)]) return PA_BM_INVALID_ARG;
            seen[static_cast<size_t>(h)] = 1;
            q.push_back(h);
        }
        m->host_free.swap(q);
        m->nh = num_host_blocks;
    } catch (...) {
        return PA_BM_INVALID_ARG;
    }
    return PA_BM_OK;
}

int32_t pa_bm_num_host_free(const pa_bm* m) { return m ? static_cast<int32_t>(m->host_free.size()) : -1; }

pa_bm_status pa_bm_swap_out(pa_bm* m, int64_t req, int64_t* pairs, int32_t pair_cap, int32_t* num_pairs) {
    if (!m || pair_cap < 0 || (pair_cap > 0 && !pairs)) return PA_BM_INVALID_ARG;
    auto it = m->reqs.find(req);
    if (it == m->reqs.end()) return PA_BM_BAD_REQUEST;
    Request& r = it->second;
    if (r.swapped || static_cast<int32_t>(r.blocks.size()) != r.need) return PA_BM_BAD_REQUEST;
    // blocks held by this request alone move; shared ones stay (moving one
    // holder would not free their memory)
    int32_t priv = 0;
    for (int32_t b : r.blocks) priv += (m->ref[b] == 1) ? 1 : 0;
    if (priv > static_cast<int32_t>(m->host_free.size())) return PA_BM_NO_SPACE;
    if (priv > pair_cap) return PA_BM_INVALID_ARG;
    try {
        r.host.assign(r.blocks.size(), -1);
    } catch (...) {
        return PA_BM_INVALID_ARG;
    }
    int32_t np = 0;
    for (size_t j = 0; j < r.blocks.size(); ++j) {
        if (m->ref[r.blocks[j]] != 1) continue;
        const int32_t h = m->host_free.front();
        m->host_free.pop_front();
        pairs[2 * np] = r.blocks[j];
        pairs[2 * np + 1] = h;
        ++np;
        r.host[j] = h;
    }
    for (size_t j = r.blocks.size(); j-- > 0;) {              // released last block first
        if (r.host[j] < 0) continue;
        m->release(r.blocks[j]);
        r.blocks[j] = -1;
    }
    r.swapped = true;
    r.epoch = m->next_epoch++;
    m->nswapped += 1;
    if (num_pairs) *num_pairs = np;
    return PA_BM_OK;
}

pa_bm_status pa_bm_swap_in(pa_bm* m, int64_t req, int64_t* pairs, int32_t pair_cap, int32_t* num_pairs) {
    if (!m || pair_cap < 0 || (pair_cap > 0 && !pairs)) return PA_BM_INVALID_ARG;
    auto it = m->reqs.find(req);
    if (it == m->reqs.end()) return PA_BM_BAD_REQUEST;
    Request& r = it->second;
    if (!r.swapped) return PA_BM_BAD_REQUEST;
    int32_t cnt = 0;
    for (int32_t h : r.host) cnt += (h >= 0) ? 1 : 0;
    if (cnt > m->nfree) return PA_BM_NO_SPACE;
    if (cnt > pair_cap) return PA_BM_INVALID_ARG;
    int32_t np = 0;
    for (size_t j = 0; j < r.host.size(); ++j) {
        if (r.host[j] < 0) continue;
        const int32_t b = m->take();
        pairs[2 * np] = r.host[j];
        pairs[2 * np + 1] = b;
        ++np;
        r.blocks[j] = b;
    }
    try {
        for (size_t j = 0; j < r.host.size(); ++j) {
            if (r.host[j] < 0) continue;
            m->host_free.push_back(r.host[j]);
            if (j < r.hashes.size()) m->cache_block(r.blocks[j], r.hashes[j]);   // prompt blocks stay findable
        }
    } catch (...) {
        return PA_BM_INVALID_ARG;
    }
    r.host.clear();
    r.swapped = false;
    r.epoch = m->next_epoch++;
    m->nswapped -= 1;
    if (num_pairs) *num_pairs = np;
    return PA_BM_OK;
}

}  // extern "C"
