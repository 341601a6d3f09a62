/*
 * oga.c -- CPU oracle for the group-adaptive additive exponent codec of the page
 * "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference on Personal
 * Devices" (section "Lossless KV Compression": "Contiguous exponent concentration" and
 * "Group-adaptive additive coding"; Table 9 "Storage"), applied to the same 16-token
 * pages as the 12-bit format.
 *
 * TEST INFRASTRUCTURE ONLY, like oref.c: plain scalar C, shares nothing with the CUDA
 * library, loaded only by the tests, the smoke check and the benchmark's CPU legs.
 *
 * The page's width formula and its encode/reconstruct formulas were lost in extraction;
 * the readings below are the plainest ones the surrounding text supports:
 *   - tile: one (page, KV head, K|V) slice, 16 tokens x 128 dims = 2048 values (the
 *     page's tile is a 128-dim half-head of 16 tokens);
 *   - group: 8 values in attention-access order = one lane's fragment, storage element
 *     (lane L, fragment f, i = 0..7) of block j (the same storage order as oref.c);
 *     group index q = 8L + 2j + f (lane-major over the tile);
 *   - per (layer, KV head, K|V, channel) calibrated bases b3 and b4 (windows of 8 and 16
 *     exponents); element i uses its channel's bases;
 *   - width of a group: 3 if every d3 = e - b3 lies in [0, 8), else 4 if every
 *     d4 = e - b4 lies in [0, 16), else 8 (raw exponent, base 0); mode tag 0, 1, 2;
 *   - code c = e - b_w; the low 3 bits of every code go to a common 3-bit stream; a
 *     4-bit group adds one escape byte (bit 3 of each code, bit i for element i); a raw
 *     group adds five escape bytes (bits 3..7 of each code, 5 bits per element, element
 *     i at bits [5i, 5i+5) of a little-endian 40-bit field);
 *   - sign and 7 fraction bits are kept unchanged in one byte per value:
 *     SF = sign << 7 | fraction; the value is sign<<15 | e<<7 | fraction;
 *   - tile layout (3008 bytes, a multiple of 64):
 *       [0, 2048)     SF bytes: block j, lane L, fragment f, element i at 512j+16L+8f+i
 *       [2048, 2816)  3-bit codes: group q at 2048 + 3q, element i at bits [3i, 3i+3)
 *                     of the little-endian 24-bit field
 *       [2816, 2880)  mode tags: group q at bits [2(q%4), 2(q%4)+2) of byte 2816 + q/4
 *       [2880, 3008)  escape bytes of the groups in q order, zero-padded
 *     a tile whose groups need more than 128 escape bytes is stored raw instead: 2048
 *     BF16 words in storage order (block j's 512 words as in oref.c), 4096 bytes;
 *   - calibration: over a sample of values of one channel, the window start with the
 *     most exponents inside [b, b+W-1] (b in [0, 256-W]); ties go to the lowest start.
 */
#include "oref.h"

#include <stdlib.h>
#include <string.h>

static unsigned ga_exp(uint16_t w) { return (w >> 7) & 0xFFu; }

/* element (L, f, i) of block j -> (token, dim); same map as oref_block_position */
static void ga_pos(int is_v, int j, int L, int f, int i, int *tok, int *dim)
{
    oref_block_position(is_v, j, L, f, i, tok, dim);
}

/* ---------------------------------------------------------------------------------
 * calibration ("Contiguous exponent concentration": for each head-channel pair the
 * contiguous windows of lengths 8 and 16 that cover the most exponent values)
 * ------------------------------------------------------------------------------- */
static unsigned best_window(const uint64_t hist[256], int width)
{
    uint64_t best = 0;
    unsigned best_b = 0;
    for (int b = 0; b + width <= 256; b++) {
        uint64_t cov = 0;
        for (int e = b; e < b + width; e++) cov += hist[e];
        if (cov > best) {
            best = cov;
            best_b = (unsigned)b;
        }
    }
    return best_b;
}

/* pages: [n][16][128] BF16 of one (layer, head, K|V); bases out: b3[128], b4[128] */
void oga_calibrate(const uint16_t *pages, int64_t n, uint8_t *b3, uint8_t *b4)
{
    for (int ch = 0; ch < 128; ch++) {
        uint64_t hist[256];
        memset(hist, 0, sizeof hist);
        for (int64_t p = 0; p < n; p++)
            for (int t = 0; t < 16; t++) hist[ga_exp(pages[(p * 16 + t) * 128 + ch])]++;
        b3[ch] = (uint8_t)best_window(hist, 8);
        b4[ch] = (uint8_t)best_window(hist, 16);
    }
}

/* ---------------------------------------------------------------------------------
 * tile encode / decode ("Group-adaptive additive coding")
 * ------------------------------------------------------------------------------- */
int oga_group_mode(const unsigned e[8], const unsigned b3[8], const unsigned b4[8])
{
    int ok3 = 1, ok4 = 1;
    for (int i = 0; i < 8; i++) {
        if (!(e[i] >= b3[i] && e[i] - b3[i] < 8)) ok3 = 0;
        if (!(e[i] >= b4[i] && e[i] - b4[i] < 16)) ok4 = 0;
    }
    return ok3 ? 0 : (ok4 ? 1 : 2);
}

/* Encode the 16x128 page slice; returns 3008 (compressed) or 4096 (raw). */
int oga_encode_tile(const uint16_t *page, int is_v, const uint8_t *b3c, const uint8_t *b4c, uint8_t *out)
{
    uint8_t tile[3008];
    uint8_t esc[256 * 5];
    int nesc = 0;
    memset(tile, 0, sizeof tile);
    for (int L = 0; L < 32; L++)
        for (int j = 0; j < 4; j++)
            for (int f = 0; f < 2; f++) {
                const int q = 8 * L + 2 * j + f;
                unsigned e[8], b3[8], b4[8], sf[8];
                for (int i = 0; i < 8; i++) {
                    int tok, dim;
                    ga_pos(is_v, j, L, f, i, &tok, &dim);
                    const uint16_t w = page[tok * 128 + dim];
                    e[i] = ga_exp(w);
                    sf[i] = ((w >> 8) & 0x80u) | (w & 0x7Fu);
                    b3[i] = b3c[dim];
                    b4[i] = b4c[dim];
                }
                const int mode = oga_group_mode(e, b3, b4);
                unsigned c[8];
                for (int i = 0; i < 8; i++) c[i] = e[i] - (mode == 0 ? b3[i] : mode == 1 ? b4[i] : 0u);
                uint32_t low = 0;
                for (int i = 0; i < 8; i++) {
                    tile[512 * j + 16 * L + 8 * f + i] = (uint8_t)sf[i];
                    low |= (c[i] & 7u) << (3 * i);
                }
                tile[2048 + 3 * q] = (uint8_t)low;
                tile[2048 + 3 * q + 1] = (uint8_t)(low >> 8);
                tile[2048 + 3 * q + 2] = (uint8_t)(low >> 16);
                tile[2816 + q / 4] |= (uint8_t)(mode << (2 * (q % 4)));
                if (mode == 1) {
                    uint8_t hb = 0;
                    for (int i = 0; i < 8; i++) hb |= (uint8_t)(((c[i] >> 3) & 1u) << i);
                    esc[nesc++] = hb;
                } else if (mode == 2) {
                    uint64_t hb = 0;
                    for (int i = 0; i < 8; i++) hb |= (uint64_t)((c[i] >> 3) & 31u) << (5 * i);
                    for (int k = 0; k < 5; k++) esc[nesc++] = (uint8_t)(hb >> (8 * k));
                }
            }
    if (nesc > 128) {
        /* raw fallback: the 4 blocks' words in storage order, little-endian */
        for (int j = 0; j < 4; j++)
            for (int L = 0; L < 32; L++)
                for (int f = 0; f < 2; f++)
                    for (int i = 0; i < 8; i++) {
                        int tok, dim;
                        ga_pos(is_v, j, L, f, i, &tok, &dim);
                        const uint16_t w = page[tok * 128 + dim];
                        const int n = 512 * j + (L * 2 + f) * 8 + i;
                        out[2 * n] = (uint8_t)(w & 0xFF);
                        out[2 * n + 1] = (uint8_t)(w >> 8);
                    }
        return 4096;
    }
    memcpy(tile + 2880, esc, (size_t)nesc);
    memcpy(out, tile, sizeof tile);
    return 3008;
}

/* Decode a tile (raw = 0: 3008-byte compressed tile, raw = 1: 4096-byte raw tile). */
void oga_decode_tile(const uint8_t *in, int raw, int is_v, const uint8_t *b3c, const uint8_t *b4c, uint16_t *page)
{
    int at = 2880;
    for (int L = 0; L < 32; L++)
        for (int j = 0; j < 4; j++)
            for (int f = 0; f < 2; f++) {
                const int q = 8 * L + 2 * j + f;
                const int mode = raw ? 0 : (in[2816 + q / 4] >> (2 * (q % 4))) & 3;
                const uint32_t low = raw ? 0 : (uint32_t)in[2048 + 3 * q] | ((uint32_t)in[2048 + 3 * q + 1] << 8) |
                                                   ((uint32_t)in[2048 + 3 * q + 2] << 16);
                uint64_t hb = 0;
                if (!raw && mode == 1) hb = in[at++];
                if (!raw && mode == 2) {
                    for (int k = 0; k < 5; k++) hb |= (uint64_t)in[at + k] << (8 * k);
                    at += 5;
                }
                for (int i = 0; i < 8; i++) {
                    int tok, dim;
                    ga_pos(is_v, j, L, f, i, &tok, &dim);
                    uint16_t w;
                    if (raw) {
                        const int n = 512 * j + (L * 2 + f) * 8 + i;
                        w = (uint16_t)(in[2 * n] | (in[2 * n + 1] << 8));
                    } else {
                        unsigned c = (low >> (3 * i)) & 7u;
                        if (mode == 1) c |= (unsigned)((hb >> i) & 1u) << 3;
                        if (mode == 2) c |= (unsigned)((hb >> (5 * i)) & 31u) << 3;
                        const unsigned e = c + (mode == 0 ? b3c[dim] : mode == 1 ? b4c[dim] : 0u);
                        const unsigned sf = in[512 * j + 16 * L + 8 * f + i];
                        w = (uint16_t)(((sf & 0x80u) << 8) | ((e & 0xFFu) << 7) | (sf & 0x7Fu));
                    }
                    page[tok * 128 + dim] = w;
                }
            }
}

/* ---------------------------------------------------------------------------------
 * pages of one layer ("Block-Wise Compression Scheduling": two storage classes, the
 * block table records each tile's mode and place; Table 9: a 4-byte entry per tile).
 * Same call structure as oref_encode_pages, with 64-byte granules: a compressed tile
 * takes 47 granules, a raw one 64.  bases: [hkv][2][2][128] = (head, K|V, b3|b4,
 * channel).  Entry (uint32, one per (page, head, K|V)): bits 0..30 = offset in
 * granules, bit 31 = raw tile; 0xFFFFFFFF = no tile (the arena was full).
 * ------------------------------------------------------------------------------- */
int oga_encode_pages(int hkv, const uint16_t *raw_pool, int64_t num_raw_pages, const uint8_t *bases,
                     const int32_t *src_page, const int32_t *dst_page, const int32_t *dst_seq, int32_t n,
                     uint32_t *meta, int64_t num_meta_pages, uint8_t *arena, uint64_t arena_bytes,
                     uint32_t *cursors, int32_t num_cursors)
{
    int status = 0;
    for (int p = 0; p < n; p++) {
        if (src_page[p] < 0 || src_page[p] >= num_raw_pages || dst_page[p] < 0 ||
            dst_page[p] >= num_meta_pages || dst_seq[p] < 0 || dst_seq[p] >= num_cursors)
            status |= OREF_BAD_INDEX;
        if (p > 0 && dst_seq[p] < dst_seq[p - 1]) status |= OREF_BAD_ORDER;
    }
    if (status) return status;
    uint64_t arena_granules = arena_bytes / 64;
    if (arena_granules > 0x7FFFFFFFull) arena_granules = 0x7FFFFFFFull; /* 31-bit offsets */
    uint8_t buf[4096];
    for (int p = 0; p < n; p++) {
        uint32_t *cur = &cursors[2 * dst_seq[p]];
        for (int h = 0; h < hkv; h++)
            for (int kv = 0; kv < 2; kv++) {
                const uint16_t *page = raw_pool + (((int64_t)src_page[p] * hkv + h) * 2 + kv) * 16 * 128;
                const uint8_t *bb = bases + ((size_t)h * 2 + kv) * 256;
                const int size = oga_encode_tile(page, kv, bb, bb + 128, buf);
                const uint64_t gran = (uint64_t)size / 64, off = cur[0];
                uint32_t *m = &meta[((int64_t)dst_page[p] * hkv + h) * 2 + kv];
                if (off + gran > cur[1] || off + gran > arena_granules) {
                    status |= OREF_ARENA_FULL;
                    *m = 0xFFFFFFFFu;
                } else {
                    memcpy(arena + off * 64, buf, (size_t)size);
                    *m = (uint32_t)off | (size == 4096 ? 0x80000000u : 0u);
                }
                cur[0] = (uint32_t)(off + gran);
            }
    }
    return status;
}

/* One tile from its entry; a missing or out-of-arena tile decodes as zeros. */
int oga_decode_entry(uint32_t entry, const uint8_t *arena, uint64_t arena_bytes, int is_v, const uint8_t *bb,
                     uint16_t *half_page)
{
    const uint64_t off = entry & 0x7FFFFFFFu;
    const int raw = (entry >> 31) != 0;
    const uint64_t size = raw ? 4096 : 3008;
    if (entry == 0xFFFFFFFFu || off * 64 + size > arena_bytes) {
        memset(half_page, 0, 16 * 128 * sizeof(uint16_t));
        return OREF_BAD_META;
    }
    oga_decode_tile(arena + off * 64, raw, is_v, bb, bb + 128, half_page);
    return 0;
}

int oga_decode_pages(int hkv, const uint32_t *meta, int64_t num_meta_pages, const uint8_t *arena,
                     uint64_t arena_bytes, const uint8_t *bases, const int32_t *page, int32_t n, uint16_t *out)
{
    int status = 0;
    for (int p = 0; p < n; p++)
        for (int h = 0; h < hkv; h++)
            for (int kv = 0; kv < 2; kv++) {
                uint16_t *dst = out + (((int64_t)p * hkv + h) * 2 + kv) * 16 * 128;
                if (page[p] < 0 || page[p] >= num_meta_pages) {
                    memset(dst, 0, 16 * 128 * sizeof(uint16_t));
                    status |= OREF_BAD_INDEX;
                    continue;
                }
                const uint32_t entry = meta[((int64_t)page[p] * hkv + h) * 2 + kv];
                status |= oga_decode_entry(entry, arena, arena_bytes, kv, bases + ((size_t)h * 2 + kv) * 256, dst);
            }
    return status;
}
