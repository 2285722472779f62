// Host block pool: free list, reference counts, fork and copy-on-write append.
//
// Semantics follow the BlockPool simulation on the "vLLM 与 PagedAttention"
// page (section 最小分页与 COW 模拟): LIFO free list, a fresh block when the
// tail is absent or full, a private copy when the tail is shared and not full,
// in-place otherwise.  Release (absent there) drops one reference per block and
// returns blocks that reach zero to the end of the free list, in table order.
// Instead of the simulation's token lists the pool keeps a fill count per
// block, which is all the allocation decisions need.
//
// Swap (preemption, on the same page: a request's physical blocks are released
// or migrated while its logical tokens are kept) moves a sequence to another pool
// of the same block size, e.g. one that stands for pinned host memory: every
// block of its table gets a fresh private block there holding the same tokens,
// then the sequence is released in the source pool.  The caller copies the
// returned (source block, destination block) pairs with pa_swap_blocks.
//
// Table deltas (MiniPaged-Qwen's closing notes: richer block metadata at lower
// host overhead): pa_pool_table_deltas names only the (row, logical block,
// physical block) entries a device-resident copy of the tables lacks, given
// that copy received every earlier export in order.  The pool remembers per
// sequence the row and table of its last export and per row the sequence last
// exported into it: a sequence still in its row sends the entries that changed
// or were added; one in another row, or new, sends all of them.
//
// Every failing call leaves the pool exactly as it was: single appends check
// before mutating; batch appends keep an undo log.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"
#include "pa_internal.h"

struct pa_pool {
    struct Seq {
        std::vector<int32_t> table;
        int64_t length = 0;
        int synced_row = -1;                // row of its last delta export (-1: never)
        std::vector<int32_t> synced_table;  // its table as of that export
    };
    int num_blocks = 0;
    int block_size = 0;
    std::vector<int32_t> free_list;  // back() is the next block handed out
    std::vector<int32_t> refs;       // per block; 0 = free
    std::vector<int32_t> fill;       // tokens stored in the block
    std::unordered_map<int64_t, Seq> seqs;
    std::unordered_map<int, int64_t> row_owner;  // device table row -> sequence last exported into it
    int64_t next_id = 0;
};

namespace {

enum AppendKind { kInPlace = 0, kFreshBlock = 1, kCopyOnWrite = 2 };

struct AppendRecord {
    int64_t seq_id;
    int kind;
    int32_t block;      // fresh or private block (kinds 1, 2)
    int32_t shared;     // the shared tail that was copied (kind 2)
};

// Allocation decision for one append; checks only (no mutation).
int plan_append(const pa_pool* p, const pa_pool::Seq& s, int* kind) {
    if (s.table.empty() || p->fill[s.table.back()] == p->block_size) {
        *kind = kFreshBlock;
    } else if (p->refs[s.table.back()] > 1) {
        *kind = kCopyOnWrite;
    } else {
        *kind = kInPlace;
    }
    if (*kind != kInPlace && p->free_list.empty()) return PA_ERR_POOL_EXHAUSTED;
    return PA_OK;
}

int32_t take_block(pa_pool* p) {
    int32_t b = p->free_list.back();
    p->free_list.pop_back();
    p->refs[b] = 1;
    p->fill[b] = 0;
    return b;
}

void give_back(pa_pool* p, int32_t b) {
    p->refs[b] = 0;
    p->fill[b] = 0;
    p->free_list.push_back(b);
}

// Performs an append whose plan succeeded.  Returns the record.
AppendRecord do_append(pa_pool* p, int64_t seq_id, pa_pool::Seq& s, int kind, int64_t* slot) {
    AppendRecord rec{seq_id, kind, -1, -1};
    if (kind == kFreshBlock) {
        rec.block = take_block(p);
        s.table.push_back(rec.block);
    } else if (kind == kCopyOnWrite) {
        rec.shared = s.table.back();
        rec.block = take_block(p);
        p->fill[rec.block] = p->fill[rec.shared];  // the private copy holds the same tokens
        p->refs[rec.shared] -= 1;
        s.table.back() = rec.block;
    }
    const int32_t tail = s.table.back();
    *slot = static_cast<int64_t>(tail) * p->block_size + p->fill[tail];
    p->fill[tail] += 1;
    s.length += 1;
    return rec;
}

void undo_append(pa_pool* p, const AppendRecord& rec) {
    pa_pool::Seq& s = p->seqs[rec.seq_id];
    const int32_t tail = s.table.back();
    p->fill[tail] -= 1;
    s.length -= 1;
    if (rec.kind == kFreshBlock) {
        s.table.pop_back();
        give_back(p, rec.block);
    } else if (rec.kind == kCopyOnWrite) {
        s.table.back() = rec.shared;
        p->refs[rec.shared] += 1;
        give_back(p, rec.block);
    }
}

pa_pool::Seq* find_seq(pa_pool* p, int64_t id) {
    auto it = p->seqs.find(id);
    return it == p->seqs.end() ? nullptr : &it->second;
}

const pa_pool::Seq* find_seq(const pa_pool* p, int64_t id) {
    auto it = p->seqs.find(id);
    return it == p->seqs.end() ? nullptr : &it->second;
}

}  // namespace

extern "C" {

int pa_pool_create(int num_blocks, int block_size, const int32_t* free_order, pa_pool** out) {
    if (!out) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_create: out is NULL");
    *out = nullptr;
    if (num_blocks < 0 || block_size <= 0)
        return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_create: num_blocks=%d block_size=%d", num_blocks, block_size);
    pa_pool* p = new (std::nothrow) pa_pool();
    if (!p) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_create: out of host memory");
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->refs.assign(num_blocks, 0);
    p->fill.assign(num_blocks, 0);
    p->free_list.resize(num_blocks);
    if (free_order) {
        std::vector<char> seen(num_blocks, 0);
        for (int i = 0; i < num_blocks; ++i) {
            int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete p;
                return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_create: free_order is not a permutation (entry %d)", i);
            }
            seen[b] = 1;
            p->free_list[i] = b;
        }
    } else {
        for (int i = 0; i < num_blocks; ++i) p->free_list[i] = i;
    }
    *out = p;
    return PA_OK;
}

void pa_pool_destroy(pa_pool* pool) { delete pool; }

int pa_seq_create(pa_pool* pool, int64_t* seq_id) {
    if (!pool || !seq_id) return pa::fail(PA_ERR_INVALID_ARG, "pa_seq_create: NULL argument");
    const int64_t id = pool->next_id++;
    pool->seqs.emplace(id, pa_pool::Seq{});
    *seq_id = id;
    return PA_OK;
}

int pa_seq_append(pa_pool* pool, int64_t seq_id, int64_t* slot, int64_t* cow_src, int64_t* cow_dst) {
    if (!pool || !slot) return pa::fail(PA_ERR_INVALID_ARG, "pa_seq_append: NULL argument");
    pa_pool::Seq* s = find_seq(pool, seq_id);
    if (!s) return pa::fail(PA_ERR_NOT_FOUND, "pa_seq_append: unknown sequence %lld", (long long)seq_id);
    int kind = 0;
    if (plan_append(pool, *s, &kind) != PA_OK)
        return pa::fail(PA_ERR_POOL_EXHAUSTED, "KV pool exhausted (sequence %lld)", (long long)seq_id);
    AppendRecord rec = do_append(pool, seq_id, *s, kind, slot);
    if (cow_src) *cow_src = rec.kind == kCopyOnWrite ? rec.shared : -1;
    if (cow_dst) *cow_dst = rec.kind == kCopyOnWrite ? rec.block : -1;
    return PA_OK;
}

int pa_seq_append_batch(pa_pool* pool, const int64_t* seq_ids, int n, int64_t* slots, int64_t* cow_pairs,
                        int* num_cow) {
    if (!pool || n < 0 || (n > 0 && (!seq_ids || !slots || !cow_pairs)) || !num_cow)
        return pa::fail(PA_ERR_INVALID_ARG, "pa_seq_append_batch: bad arguments");
    std::vector<AppendRecord> log;
    log.reserve(n);
    int cows = 0;
    for (int i = 0; i < n; ++i) {
        pa_pool::Seq* s = find_seq(pool, seq_ids[i]);
        int kind = 0;
        int status = s ? plan_append(pool, *s, &kind) : PA_ERR_NOT_FOUND;
        if (status != PA_OK) {
            for (auto it = log.rbegin(); it != log.rend(); ++it) undo_append(pool, *it);
            if (status == PA_ERR_NOT_FOUND)
                return pa::fail(status, "pa_seq_append_batch: unknown sequence %lld", (long long)seq_ids[i]);
            return pa::fail(status, "KV pool exhausted at batch entry %d (nothing appended)", i);
        }
        log.push_back(do_append(pool, seq_ids[i], *s, kind, &slots[i]));
        if (log.back().kind == kCopyOnWrite) {
            cow_pairs[2 * cows] = log.back().shared;
            cow_pairs[2 * cows + 1] = log.back().block;
            ++cows;
        }
    }
    *num_cow = cows;
    return PA_OK;
}

int pa_seq_fork(pa_pool* pool, int64_t parent_id, int64_t* child_id) {
    if (!pool || !child_id) return pa::fail(PA_ERR_INVALID_ARG, "pa_seq_fork: NULL argument");
    const pa_pool::Seq* parent = find_seq(pool, parent_id);
    if (!parent) return pa::fail(PA_ERR_NOT_FOUND, "pa_seq_fork: unknown sequence %lld", (long long)parent_id);
    pa_pool::Seq child = *parent;  // copy before emplace may rehash
    child.synced_row = -1;         // the child has never been exported
    child.synced_table.clear();
    for (int32_t b : child.table) pool->refs[b] += 1;
    const int64_t id = pool->next_id++;
    pool->seqs.emplace(id, std::move(child));
    *child_id = id;
    return PA_OK;
}

int pa_seq_release(pa_pool* pool, int64_t seq_id) {
    if (!pool) return pa::fail(PA_ERR_INVALID_ARG, "pa_seq_release: NULL pool");
    auto it = pool->seqs.find(seq_id);
    if (it == pool->seqs.end())
        return pa::fail(PA_ERR_NOT_FOUND, "pa_seq_release: unknown sequence %lld", (long long)seq_id);
    for (int32_t b : it->second.table) {
        pool->refs[b] -= 1;
        if (pool->refs[b] == 0) give_back(pool, b);
    }
    pool->seqs.erase(it);
    return PA_OK;
}

int pa_seq_swap(pa_pool* src, pa_pool* dst, int64_t seq_id, int64_t* new_seq_id, int64_t* block_pairs,
                int capacity, int* num_pairs) {
    if (!src || !dst || !new_seq_id || !num_pairs || capacity < 0 || (capacity > 0 && !block_pairs))
        return pa::fail(PA_ERR_INVALID_ARG, "pa_seq_swap: bad arguments");
    if (src == dst) return pa::fail(PA_ERR_INVALID_ARG, "pa_seq_swap: source and destination are the same pool");
    if (src->block_size != dst->block_size)
        return pa::fail(PA_ERR_INVALID_ARG, "pa_seq_swap: block sizes differ (%d vs %d)", src->block_size,
                        dst->block_size);
    auto it = src->seqs.find(seq_id);
    if (it == src->seqs.end())
        return pa::fail(PA_ERR_NOT_FOUND, "pa_seq_swap: unknown sequence %lld", (long long)seq_id);
    const std::vector<int32_t>& table = it->second.table;
    const int n = static_cast<int>(table.size());
    if (n > capacity)
        return pa::fail(PA_ERR_INVALID_ARG, "pa_seq_swap: %d pairs do not fit in %d", n, capacity);
    if (static_cast<int>(dst->free_list.size()) < n)
        return pa::fail(PA_ERR_POOL_EXHAUSTED, "pa_seq_swap: destination has %zu free blocks, sequence needs %d",
                        dst->free_list.size(), n);
    pa_pool::Seq moved;
    moved.length = it->second.length;
    moved.table.reserve(n);
    for (int j = 0; j < n; ++j) {
        const int32_t b = take_block(dst);
        dst->fill[b] = src->fill[table[j]];
        moved.table.push_back(b);
        block_pairs[2 * j] = table[j];
        block_pairs[2 * j + 1] = b;
    }
    const int64_t id = dst->next_id++;
    dst->seqs.emplace(id, std::move(moved));
    for (int32_t b : it->second.table) {
        src->refs[b] -= 1;
        if (src->refs[b] == 0) give_back(src, b);
    }
    src->seqs.erase(it);
    *new_seq_id = id;
    *num_pairs = n;
    return PA_OK;
}

int pa_pool_blocks_needed(const pa_pool* pool, const int64_t* seq_ids, const int32_t* counts, int n,
                          int64_t* needed) {
    if (!pool || !needed || n < 0 || (n > 0 && (!seq_ids || !counts)))
        return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_blocks_needed: bad arguments");
    // Dry run of the appends, in order, on overlays of the touched state (nothing changes).
    struct Tail {
        int32_t block;  // the tail block (>= 0 real, < 0 a block taken in the dry run)
        int32_t fill;
    };
    std::unordered_map<int64_t, Tail> tails;       // sequence -> its tail after the dry-run appends so far
    std::unordered_map<int32_t, int32_t> refs_of;  // real block -> reference count after the dry run
    int64_t taken = 0;
    for (int i = 0; i < n; ++i) {
        if (counts[i] < 0) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_blocks_needed: negative count");
        auto it = pool->seqs.find(seq_ids[i]);
        if (it == pool->seqs.end())
            return pa::fail(PA_ERR_NOT_FOUND, "pa_pool_blocks_needed: unknown sequence %lld",
                            (long long)seq_ids[i]);
        auto t = tails.find(seq_ids[i]);
        if (t == tails.end()) {
            const auto& tab = it->second.table;
            Tail cur{-1, pool->block_size};  // an empty table behaves as a full tail
            if (!tab.empty()) cur = Tail{tab.back(), pool->fill[tab.back()]};
            t = tails.emplace(seq_ids[i], cur).first;
        }
        for (int32_t k = 0; k < counts[i]; ++k) {
            Tail& tl = t->second;
            if (tl.fill == pool->block_size) {
                tl = Tail{(int32_t)(-1 - taken), 0};  // a fresh block
                ++taken;
            } else if (tl.block >= 0) {
                auto r = refs_of.find(tl.block);
                int32_t& refs = r == refs_of.end() ? (refs_of[tl.block] = pool->refs[tl.block]) : r->second;
                if (refs > 1) {  // copy-on-write: this sequence leaves the shared tail
                    refs -= 1;
                    tl = Tail{(int32_t)(-1 - taken), tl.fill};
                    ++taken;
                }
            }
            tl.fill += 1;
        }
    }
    *needed = taken;
    return PA_OK;
}

int pa_seq_length(const pa_pool* pool, int64_t seq_id, int64_t* length) {
    if (!pool || !length) return pa::fail(PA_ERR_INVALID_ARG, "pa_seq_length: NULL argument");
    const pa_pool::Seq* s = find_seq(pool, seq_id);
    if (!s) return pa::fail(PA_ERR_NOT_FOUND, "pa_seq_length: unknown sequence %lld", (long long)seq_id);
    *length = s->length;
    return PA_OK;
}

int pa_pool_table_deltas(pa_pool* pool, const int64_t* seq_ids, int n, int32_t* deltas, int capacity,
                         int* num_deltas, int32_t* lens) {
    if (!pool || n < 0 || capacity < 0 || !num_deltas || (n > 0 && (!seq_ids || !lens)) ||
        (capacity > 0 && !deltas))
        return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_table_deltas: bad arguments");
    // count first, so that a failure changes nothing
    int64_t count = 0;
    for (int i = 0; i < n; ++i) {
        const pa_pool::Seq* s = find_seq(pool, seq_ids[i]);
        if (!s)
            return pa::fail(PA_ERR_NOT_FOUND, "pa_pool_table_deltas: unknown sequence %lld", (long long)seq_ids[i]);
        for (int j = i + 1; j < n; ++j)
            if (seq_ids[j] == seq_ids[i])
                return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_table_deltas: sequence %lld in two rows",
                                (long long)seq_ids[i]);
        if (s->length > INT32_MAX) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_table_deltas: length > int32");
        auto owner = pool->row_owner.find(i);
        const bool kept = s->synced_row == i && owner != pool->row_owner.end() && owner->second == seq_ids[i];
        for (size_t j = 0; j < s->table.size(); ++j)
            if (!kept || j >= s->synced_table.size() || s->synced_table[j] != s->table[j]) ++count;
    }
    if (count > capacity)
        return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_table_deltas: %lld deltas do not fit in %d", (long long)count,
                        capacity);
    int k = 0;
    for (int i = 0; i < n; ++i) {
        pa_pool::Seq* s = find_seq(pool, seq_ids[i]);
        auto owner = pool->row_owner.find(i);
        const bool kept = s->synced_row == i && owner != pool->row_owner.end() && owner->second == seq_ids[i];
        for (size_t j = 0; j < s->table.size(); ++j) {
            if (!kept || j >= s->synced_table.size() || s->synced_table[j] != s->table[j]) {
                deltas[3 * k] = i;
                deltas[3 * k + 1] = static_cast<int32_t>(j);
                deltas[3 * k + 2] = s->table[j];
                ++k;
            }
        }
        s->synced_row = i;
        s->synced_table = s->table;
        pool->row_owner[i] = seq_ids[i];
        lens[i] = static_cast<int32_t>(s->length);
    }
    *num_deltas = k;
    return PA_OK;
}

int pa_pool_block_tables(const pa_pool* pool, const int64_t* seq_ids, int n, int32_t* tables, int max_blocks,
                         int32_t* lens) {
    if (!pool || n < 0 || max_blocks < 0 || (n > 0 && (!seq_ids || !tables || !lens)))
        return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_block_tables: bad arguments");
    for (int i = 0; i < n; ++i) {
        const pa_pool::Seq* s = find_seq(pool, seq_ids[i]);
        if (!s) return pa::fail(PA_ERR_NOT_FOUND, "pa_pool_block_tables: unknown sequence %lld", (long long)seq_ids[i]);
        if (static_cast<int64_t>(s->table.size()) > max_blocks)
            return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_block_tables: sequence %lld needs %zu blocks > %d",
                            (long long)seq_ids[i], s->table.size(), max_blocks);
        if (s->length > INT32_MAX)
            return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_block_tables: length does not fit int32");
    }
    for (int i = 0; i < n; ++i) {
        const pa_pool::Seq* s = find_seq(pool, seq_ids[i]);
        int32_t* row = tables + static_cast<int64_t>(i) * max_blocks;
        std::copy(s->table.begin(), s->table.end(), row);
        std::fill(row + s->table.size(), row + max_blocks, -1);
        lens[i] = static_cast<int32_t>(s->length);
    }
    return PA_OK;
}

int pa_pool_num_free(const pa_pool* pool) { return pool ? static_cast<int>(pool->free_list.size()) : -1; }
int pa_pool_num_blocks(const pa_pool* pool) { return pool ? pool->num_blocks : -1; }
int pa_pool_block_size(const pa_pool* pool) { return pool ? pool->block_size : -1; }

int pa_pool_refcount(const pa_pool* pool, int32_t block) {
    if (!pool || block < 0 || block >= pool->num_blocks) return -1;
    return pool->refs[block];
}

int pa_pool_free_list(const pa_pool* pool, int32_t* out, int capacity) {
    if (!pool || (capacity > 0 && !out)) return -1;
    const int n = static_cast<int>(pool->free_list.size());
    if (n > capacity) return -1;
    std::copy(pool->free_list.begin(), pool->free_list.end(), out);
    return n;
}

// ---- checkpoint / resume: the whole pool state as a flat little-endian byte image ----
namespace {

constexpr uint64_t kPoolMagic = 0x314c4f4f50415055ull;  // "UPAPOOL1"

struct Writer {
    uint8_t* p;
    size_t cap, n = 0;
    void put(const void* v, size_t bytes) {
        if (p && n + bytes <= cap) std::memcpy(p + n, v, bytes);
        n += bytes;
    }
    void i64(int64_t v) { put(&v, 8); }
    void i32s(const std::vector<int32_t>& v) {
        i64(static_cast<int64_t>(v.size()));
        if (!v.empty()) put(v.data(), v.size() * 4);
    }
};

struct Reader {
    const uint8_t* p;
    size_t size, n = 0;
    bool ok = true;
    bool get(void* v, size_t bytes) {
        if (!ok || n + bytes > size) return ok = false;
        std::memcpy(v, p + n, bytes);
        n += bytes;
        return true;
    }
    int64_t i64() {
        int64_t v = 0;
        get(&v, 8);
        return v;
    }
    bool i32s(std::vector<int32_t>& v, int64_t max_len) {
        const int64_t len = i64();
        if (!ok || len < 0 || len > max_len) return ok = false;
        v.resize(static_cast<size_t>(len));
        return len == 0 || get(v.data(), static_cast<size_t>(len) * 4);
    }
};

size_t write_state(const pa_pool* pool, uint8_t* buf, size_t cap) {
    Writer w{buf, cap};
    w.i64(static_cast<int64_t>(kPoolMagic));
    w.i64(pool->num_blocks);
    w.i64(pool->block_size);
    w.i64(pool->next_id);
    w.i32s(pool->free_list);
    w.i32s(pool->refs);
    w.i32s(pool->fill);
    // sequences in id order, so that equal pools give equal images
    std::vector<int64_t> ids;
    ids.reserve(pool->seqs.size());
    for (const auto& kv : pool->seqs) ids.push_back(kv.first);
    std::sort(ids.begin(), ids.end());
    w.i64(static_cast<int64_t>(ids.size()));
    for (int64_t id : ids) {
        const pa_pool::Seq& s = pool->seqs.at(id);
        w.i64(id);
        w.i64(s.length);
        w.i64(s.synced_row);
        w.i32s(s.table);
        w.i32s(s.synced_table);
    }
    std::vector<std::pair<int, int64_t>> rows(pool->row_owner.begin(), pool->row_owner.end());
    std::sort(rows.begin(), rows.end());
    w.i64(static_cast<int64_t>(rows.size()));
    for (const auto& r : rows) {
        w.i64(r.first);
        w.i64(r.second);
    }
    return w.n;
}

}  // namespace

size_t pa_pool_state_size(const pa_pool* pool) { return pool ? write_state(pool, nullptr, 0) : 0; }

int pa_pool_save(const pa_pool* pool, void* buffer, size_t capacity, size_t* written) {
    if (!pool || !written || (capacity > 0 && !buffer))
        return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_save: bad arguments");
    const size_t need = write_state(pool, nullptr, 0);
    if (need > capacity) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_save: %zu bytes needed, %zu given", need, capacity);
    *written = write_state(pool, static_cast<uint8_t*>(buffer), capacity);
    return PA_OK;
}

int pa_pool_load(const void* buffer, size_t size, pa_pool** out) {
    if (!buffer || !out) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_load: NULL argument");
    *out = nullptr;
    Reader r{static_cast<const uint8_t*>(buffer), size};
    if (static_cast<uint64_t>(r.i64()) != kPoolMagic || !r.ok)
        return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_load: not a pool image");
    const int64_t nb = r.i64(), bs = r.i64(), next_id = r.i64();
    if (!r.ok || nb < 0 || nb > INT32_MAX || bs <= 0 || bs > INT32_MAX || next_id < 0)
        return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_load: bad header");
    pa_pool* p = new (std::nothrow) pa_pool();
    if (!p) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_load: out of host memory");
    p->num_blocks = static_cast<int>(nb);
    p->block_size = static_cast<int>(bs);
    p->next_id = next_id;
    bool ok = r.i32s(p->free_list, nb) && r.i32s(p->refs, nb) && r.i32s(p->fill, nb) &&
              static_cast<int64_t>(p->refs.size()) == nb && static_cast<int64_t>(p->fill.size()) == nb;
    const int64_t nseq = ok ? r.i64() : -1;
    ok = ok && r.ok && nseq >= 0 && nseq <= (int64_t)1 << 40;
    for (int64_t i = 0; ok && i < nseq; ++i) {
        const int64_t id = r.i64();
        pa_pool::Seq s;
        s.length = r.i64();
        const int64_t row = r.i64();
        ok = r.ok && id >= 0 && id < next_id && s.length >= 0 && row >= -1 && row <= INT32_MAX &&
             r.i32s(s.table, nb) && r.i32s(s.synced_table, (int64_t)1 << 31) && !p->seqs.count(id);
        if (ok) {
            s.synced_row = static_cast<int>(row);
            p->seqs.emplace(id, std::move(s));
        }
    }
    const int64_t nrows = ok ? r.i64() : -1;
    ok = ok && r.ok && nrows >= 0 && nrows <= (int64_t)1 << 31;
    for (int64_t i = 0; ok && i < nrows; ++i) {
        const int64_t row = r.i64(), id = r.i64();
        ok = r.ok && row >= 0 && row <= INT32_MAX;
        if (ok) p->row_owner[static_cast<int>(row)] = id;
    }
    ok = ok && r.n == size;
    if (ok) {
        // the image must describe a consistent pool
        for (int32_t b : p->free_list) ok = ok && b >= 0 && b < nb && p->refs[b] == 0;
        for (const auto& kv : p->seqs)
            for (int32_t b : kv.second.table) ok = ok && b >= 0 && b < nb;
        if (ok && pa_pool_check_invariants(p) != PA_OK) ok = false;
    }
    if (!ok) {
        delete p;
        return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_load: corrupt or inconsistent pool image");
    }
    *out = p;
    pa::clear_error();
    return PA_OK;
}

int pa_pool_check_invariants(const pa_pool* pool) {
    if (!pool) return pa::fail(PA_ERR_INVALID_ARG, "pa_pool_check_invariants: NULL pool");
    const int bs = pool->block_size;
    std::vector<int32_t> counted(pool->num_blocks, 0);
    for (const auto& kv : pool->seqs) {
        const pa_pool::Seq& s = kv.second;
        const int64_t need = (s.length + bs - 1) / bs;
        if (static_cast<int64_t>(s.table.size()) != need)
            return pa::fail(PA_ERR_INVALID_ARG, "sequence %lld holds %zu blocks for %lld tokens", (long long)kv.first,
                            s.table.size(), (long long)s.length);
        for (size_t j = 0; j < s.table.size(); ++j) {
            const int32_t b = s.table[j];
            if (b < 0 || b >= pool->num_blocks)
                return pa::fail(PA_ERR_INVALID_ARG, "sequence %lld lists block %d", (long long)kv.first, b);
            counted[b] += 1;
            const int64_t expect = (j + 1 < s.table.size()) ? bs : s.length - static_cast<int64_t>(j) * bs;
            if (pool->fill[b] != expect)
                return pa::fail(PA_ERR_INVALID_ARG, "block %d holds %d tokens, sequence %lld expects %lld", b,
                                pool->fill[b], (long long)kv.first, (long long)expect);
        }
    }
    std::vector<char> is_free(pool->num_blocks, 0);
    for (int32_t b : pool->free_list) {
        if (b < 0 || b >= pool->num_blocks || is_free[b])
            return pa::fail(PA_ERR_INVALID_ARG, "free list holds %d twice or out of range", b);
        is_free[b] = 1;
    }
    for (int b = 0; b < pool->num_blocks; ++b) {
        if (counted[b] != pool->refs[b])
            return pa::fail(PA_ERR_INVALID_ARG, "block %d: refcount %d but %d tables hold it", b, pool->refs[b],
                            counted[b]);
        if (is_free[b] == (counted[b] > 0))
            return pa::fail(PA_ERR_INVALID_ARG, "block %d is %s", b, is_free[b] ? "free and used" : "lost");
    }
    return PA_OK;
}

}  // extern "C"
