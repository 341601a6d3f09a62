// kvz_internal.h -- parameter blocks and launchers shared by the host runtime
// (kvz_api.cu) and the kernels (codec.cu, attention.cu).  Not installed.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kvz_device.cuh"

namespace kvz {

struct EncodeParams {
    int hkv;
    int n;
    const uint16_t *raw_pool;
    int64_t num_raw_pages;
    const int32_t *src_page, *dst_page, *dst_seq;
    uint64_t *meta;
    int64_t num_meta_pages;
    uint8_t *arena;
    uint64_t arena_bytes;
    uint32_t *cursors;
    int num_cursors;
    uint32_t *status;
    // group-adaptive tiles: 4-byte entries instead of meta, bases [hkv][2][2][128]
    uint32_t *meta32;
    const uint8_t *ga_bases;
    // workspace
    uint32_t *ws_hdr;        // [4]: validation failure bits (stored by the prepare kernel each call)
    uint32_t *ws_page_size;  // [n] granules per page, summed over heads (zeroed each call)
    uint32_t *ws_page_base;  // [n] granule position of each page's first group
    uint32_t *ws_pair_size;  // [n*hkv] granules per (page, head) K+V pair
    uint64_t *ws_tags;       // [n*hkv] the size pass's findings per (page, head) for the pack pass:
                             // 12-bit: the K group's four tag bytes | the V group's << 32 (null:
                             // not kept); group-adaptive and FP8 tiles: K tile escape bytes |
                             // V tile's << 32
};

// grid of a warp-per-item encoder pass with 8-warp CTAs: one wave of `per_sm` CTAs per
// SM, fewer when there are fewer items than warps
inline unsigned enc_warp_grid(int64_t items, int sms, int per_sm)
{
    const int64_t want = (items + 7) / 8, wave = (int64_t)(sms > 0 ? sms : 1) * per_sm;
    return (unsigned)(want < wave ? (want > 0 ? want : 1) : wave);
}

inline size_t encode_ws_bytes(int n, int hkv)
{
    const size_t a = ((size_t)n * 4 + 15) / 16 * 16;
    return 16 + 2 * a + ((size_t)n * hkv * 4 + 15) / 16 * 16 + (size_t)n * hkv * 8;
}
// byte offset of ws_tags in the encoder workspace
inline size_t encode_ws_tags_offset(int n, int hkv)
{
    const size_t a = ((size_t)n * 4 + 15) / 16 * 16;
    return 16 + 2 * a + ((size_t)n * hkv * 4 + 15) / 16 * 16;
}

struct DecodeParams {
    int hkv;
    int n;
    const uint64_t *meta;
    int64_t num_meta_pages;
    const uint8_t *arena;
    uint64_t arena_bytes;
    const int32_t *page;
    uint16_t *out;
    uint32_t *status;
    const uint32_t *meta32;  // group-adaptive tiles
    const uint8_t *ga_bases;
};

// Attention work split: grid = C CTAs over the flattened (sequence, KV head, page)
// list; partial results live in U + C - 1 slots (U = batch * Hkv units).
constexpr int kCtasPerSm = 3;
constexpr int kMinPagesPerCta = 4;
constexpr int kMaxBatch = 1024;

struct AttnParams {
    int batch, hkv, G, max_pages;
    int grid;  // C
    const uint16_t *q;
    const int32_t *page_ids, *seq_lens, *tail_page;
    const uint64_t *meta;
    const uint32_t *meta32;   // group-adaptive tiles: entries
    const uint8_t *ga_bases;  // group-adaptive tiles: [hkv][2][2][128]
    int64_t num_meta_pages;
    const uint8_t *arena;
    uint64_t arena_bytes;
    int64_t num_raw_pages;
    float *out;
    float *part_o;     // [slots][4 or 8][128] (heads per slot: attn_slot_heads(G))
    float *part_ml;    // [slots][4 or 8][2]
    uint32_t *status;
    float scale_log2;  // log2(e) / sqrt(128)
    int overlap;       // 1: launched as programmatic dependents (KVZ_ATTN_OVERLAP_PREVIOUS)
};

inline size_t attn_slots(int batch, int hkv, int grid) { return (size_t)batch * hkv + grid - 1; }
// heads per partial slot: 4 for G <= 4, 8 for G = 5..8
inline int attn_slot_heads(int G) { return G > 4 ? 8 : 4; }

// workspace layout: part_o, part_ml
inline size_t attn_ws_bytes(int batch, int hkv, int grid, int G = 4)
{
    size_t slots = attn_slots(batch, hkv, grid);
    const size_t gs = (size_t)attn_slot_heads(G);
    return slots * gs * 128 * 4 + slots * gs * 2 * 4;
}

cudaError_t launch_encode(const EncodeParams &P, cudaStream_t stream);
cudaError_t launch_enc_prepare(const EncodeParams &P, cudaStream_t stream);
cudaError_t launch_encode_sizes(const EncodeParams &P, cudaStream_t stream);
cudaError_t launch_enc_scan(const EncodeParams &P, cudaStream_t stream);
cudaError_t launch_ga_encode(const EncodeParams &P, cudaStream_t stream);
cudaError_t launch_ga_decode(const DecodeParams &P, cudaStream_t stream);
cudaError_t launch_wait_selftest(uint64_t limit_ns, uint32_t *status, uint64_t *out, cudaStream_t stream);
cudaError_t launch_late_writer(const void *src, void *dst, uint64_t bytes, uint64_t delay_ns, cudaStream_t stream);
cudaError_t launch_f8_calibrate(int fmt, int hkv, const uint16_t *raw_pool, int64_t num_raw_pages,
                                const int32_t *pages, int n, uint8_t *bases, uint32_t *status, cudaStream_t stream);
cudaError_t launch_f8_encode(int fmt, const EncodeParams &P, cudaStream_t stream);
cudaError_t launch_f8_decode(int fmt, const DecodeParams &P, cudaStream_t stream);
cudaError_t launch_ga_calibrate(int hkv, const uint16_t *raw_pool, int64_t num_raw_pages, const int32_t *pages, int n,
                                uint8_t *bases, uint32_t *status, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams &P, cudaStream_t stream);
cudaError_t launch_apply_cursor_updates(const int32_t *idx, const uint32_t *pos, const uint32_t *end, int n,
                                        uint32_t *cursors, int num_cursors, cudaStream_t stream);
// tmap: a CUtensorMap (128-byte object) over the raw pool viewed as
// [num_raw_pages*Hkv*32 rows][128 BF16], box 64 x 32, 128-byte swizzle.
// format: 0 plain BF16 pages, 1 12-bit block groups, 2 group-adaptive tiles,
// 3 / 4 FP8 E4M3 / E5M2 tiles (completed pages; the tail stays BF16)
enum AttnFormat : int { kFmtRaw = 0, kFmtZf = 1, kFmtGa = 2, kFmtF8E4 = 3, kFmtF8E5 = 4 };
cudaError_t launch_attention(const AttnParams &P, int format, const void *tmap, cudaStream_t stream);
// CTAs per SM both attention kernels can hold at this batch size (the smaller of the two)
cudaError_t attn_ctas_per_sm(int batch, int *out);

}  // namespace kvz
