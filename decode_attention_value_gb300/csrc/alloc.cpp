// alloc.cpp -- host-side chunk allocator for the compressed-KV arena (include/kvz.h).
//
// GAAC ("Block-Wise Compression Scheduling"): compressed and raw blocks live in two
// fixed storage classes (768-byte and 1024-byte block slots) recorded in the block
// table, so the serving system never makes arbitrary variable-size allocations.
// ZipFusion ("How it works", memory manager paragraph): the manager tracks the space
// left as pages compress, hands chunks freed by one layer (here: one sequence, all
// its layers) to another, and reports capacity to the scheduler.
//
// A group of four blocks takes 12..16 granules of 256 bytes (3 per 768-byte slot, 4
// per 1024-byte slot); a (page, KV head) takes two groups.  The device appends groups
// at a per-sequence cursor inside the sequence's current chunk; this allocator only
// decides, ahead of each encode call, whether the worst case of the pages about to
// be encoded still fits that chunk, and moves the cursor to a fresh chunk otherwise.
#include <cstdint>
#include <new>
#include <vector>

#include "../../include/kvz.h"

struct kvz_alloc {
    struct Cursor {
        std::vector<uint32_t> chunks;  // chunk ids, oldest first; the last one is current
        uint64_t bound = 0;            // upper bound of the device position (granules)
        uint64_t start = 0, end = 0;   // current chunk [start, end)
        uint64_t last_ticket = 0;
    };
    uint64_t chunk = 0;  // granules per chunk
    int32_t hkv = 0;
    std::vector<uint32_t> free_list;  // LIFO: back() is handed out next
    std::vector<Cursor> cur;
    uint64_t ticket = 0;
};

extern "C" {

int kvz_alloc_create(uint64_t arena_bytes, uint32_t chunk_granules, int32_t num_cursors, int32_t num_kv_heads,
                     kvz_alloc **out)
{
    if (!out || chunk_granules == 0 || num_cursors < 0 || num_kv_heads < 1) return KVZ_ERR_INVALID_ARG;
    const uint64_t granules = arena_bytes / KVZ_GRANULE_BYTES;
    const uint64_t nchunks = granules / chunk_granules;
    if (nchunks > 0xFFFFFFFFull || granules > 0xFFFFFFFFull) return KVZ_ERR_UNSUPPORTED;
    kvz_alloc *a = new (std::nothrow) kvz_alloc;
    if (!a) return KVZ_ERR_INVALID_ARG;
    a->chunk = chunk_granules;
    a->hkv = num_kv_heads;
    a->cur.resize((size_t)num_cursors);
    a->free_list.reserve((size_t)nchunks);
    for (uint64_t k = nchunks; k-- > 0;) a->free_list.push_back((uint32_t)k);  // chunk 0 first
    *out = a;
    return KVZ_OK;
}

void kvz_alloc_destroy(kvz_alloc *a) { delete a; }

}  // extern "C"

// Shared by both reservation calls: need_of(k) = granules cursor_ids[k] must hold.
template <class Need>
static int reserve_impl(kvz_alloc *a, const int32_t *cursor_ids, int32_t count, Need need_of, int32_t *upd_idx,
                        uint32_t *upd_pos, uint32_t *upd_end, int32_t *n_upd, uint64_t *ticket)
{
    size_t need_chunks = 0;
    for (int32_t k = 0; k < count; ++k) {
        const int32_t c = cursor_ids[k];
        if (c < 0 || (size_t)c >= a->cur.size()) return KVZ_ERR_INVALID_ARG;
        for (int32_t m = 0; m < k; ++m)
            if (cursor_ids[m] == c) return KVZ_ERR_INVALID_ARG;
        const uint64_t need = need_of(k);
        if (need > a->chunk) return KVZ_ERR_UNSUPPORTED;  // one call's pages must fit one chunk
        const kvz_alloc::Cursor &cu = a->cur[(size_t)c];
        if (need > 0 && (cu.chunks.empty() || cu.bound + need > cu.end)) ++need_chunks;
    }
    if (need_chunks > a->free_list.size()) return KVZ_ERR_OUT_OF_SPACE;
    const uint64_t t = ++a->ticket;
    int32_t nu = 0;
    for (int32_t k = 0; k < count; ++k) {
        kvz_alloc::Cursor &cu = a->cur[(size_t)cursor_ids[k]];
        const uint64_t need = need_of(k);
        if (need == 0) continue;
        if (cu.chunks.empty() || cu.bound + need > cu.end) {
            const uint32_t id = a->free_list.back();
            a->free_list.pop_back();
            cu.chunks.push_back(id);
            cu.start = (uint64_t)id * a->chunk;
            cu.end = cu.start + a->chunk;
            cu.bound = cu.start;
            upd_idx[nu] = cursor_ids[k];
            upd_pos[nu] = (uint32_t)cu.start;
            upd_end[nu] = (uint32_t)cu.end;
            ++nu;
        }
        cu.bound += need;
        cu.last_ticket = t;
    }
    *n_upd = nu;
    *ticket = t;
    return KVZ_OK;
}

extern "C" {

int kvz_alloc_reserve(kvz_alloc *a, const int32_t *cursor_ids, const int32_t *pages, int32_t count, int32_t *upd_idx,
                      uint32_t *upd_pos, uint32_t *upd_end, int32_t *n_upd, uint64_t *ticket)
{
    if (!a || count < 0 || (count > 0 && (!cursor_ids || !pages || !upd_idx || !upd_pos || !upd_end)) || !n_upd ||
        !ticket)
        return KVZ_ERR_INVALID_ARG;
    for (int32_t k = 0; k < count; ++k)
        if (pages[k] < 0) return KVZ_ERR_INVALID_ARG;
    const uint64_t worst_page = 2ull * 16ull * (uint64_t)a->hkv;  // two groups of at most 16 granules per head
    return reserve_impl(a, cursor_ids, count, [&](int32_t k) { return worst_page * (uint64_t)pages[k]; }, upd_idx,
                        upd_pos, upd_end, n_upd, ticket);
}

int kvz_alloc_reserve_granules(kvz_alloc *a, const int32_t *cursor_ids, const uint64_t *granules, int32_t count,
                               int32_t *upd_idx, uint32_t *upd_pos, uint32_t *upd_end, int32_t *n_upd,
                               uint64_t *ticket)
{
    if (!a || count < 0 || (count > 0 && (!cursor_ids || !granules || !upd_idx || !upd_pos || !upd_end)) ||
        !n_upd || !ticket)
        return KVZ_ERR_INVALID_ARG;
    return reserve_impl(a, cursor_ids, count, [&](int32_t k) { return granules[k]; }, upd_idx, upd_pos, upd_end,
                        n_upd, ticket);
}

int kvz_alloc_room(const kvz_alloc *a, int32_t c, uint64_t *room)
{
    if (!a || !room || c < 0 || (size_t)c >= a->cur.size()) return KVZ_ERR_INVALID_ARG;
    const kvz_alloc::Cursor &cu = a->cur[(size_t)c];
    *room = cu.chunks.empty() ? 0 : cu.end - cu.bound;
    return KVZ_OK;
}

int kvz_alloc_observe(kvz_alloc *a, uint64_t ticket, const uint32_t *snap)
{
    if (!a || !snap) return KVZ_ERR_INVALID_ARG;
    for (size_t c = 0; c < a->cur.size(); ++c) {
        kvz_alloc::Cursor &cu = a->cur[c];
        if (cu.chunks.empty() || cu.last_ticket > ticket) continue;
        const uint64_t pos = snap[2 * c], end = snap[2 * c + 1];
        if (end != cu.end || pos < cu.start || pos > cu.bound) continue;  // not this chunk's state
        cu.bound = pos;
    }
    return KVZ_OK;
}

int kvz_alloc_release(kvz_alloc *a, int32_t c)
{
    if (!a || c < 0 || (size_t)c >= a->cur.size()) return KVZ_ERR_INVALID_ARG;
    kvz_alloc::Cursor &cu = a->cur[(size_t)c];
    for (size_t k = cu.chunks.size(); k-- > 0;) a->free_list.push_back(cu.chunks[k]);
    cu = kvz_alloc::Cursor();
    return KVZ_OK;
}

int kvz_alloc_stats(const kvz_alloc *a, uint64_t *held_bytes, uint64_t *free_bytes, uint64_t *used_bytes_bound,
                    int32_t *chunks_held, int32_t *chunks_free)
{
    if (!a) return KVZ_ERR_INVALID_ARG;
    uint64_t held = 0, used = 0;
    for (const auto &cu : a->cur) {
        held += cu.chunks.size();
        if (!cu.chunks.empty()) used += (cu.chunks.size() - 1) * a->chunk + (cu.bound - cu.start);
    }
    if (held_bytes) *held_bytes = held * a->chunk * KVZ_GRANULE_BYTES;
    if (free_bytes) *free_bytes = (uint64_t)a->free_list.size() * a->chunk * KVZ_GRANULE_BYTES;
    if (used_bytes_bound) *used_bytes_bound = used * KVZ_GRANULE_BYTES;
    if (chunks_held) *chunks_held = (int32_t)held;
    if (chunks_free) *chunks_free = (int32_t)a->free_list.size();
    return KVZ_OK;
}

}  // extern "C"
