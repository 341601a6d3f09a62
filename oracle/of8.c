/*
 * of8.c -- CPU oracle for FP8 KV pages with lossless group-adaptive exponent coding:
 * the page "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference on
 * Personal Devices" applies its codec to KV states converted to FP8 ("Relation to FP8 KV",
 * Table 7: 1.09-1.14x on E4M3, 1.25-1.30x on E5M2).  The page gives the results, not the
 * format; the readings below carry its BF16 codec over to FP8 fields.
 *
 * TEST INFRASTRUCTURE ONLY (like oref.c and oga.c): plain scalar C, shares nothing with
 * the CUDA library.
 *
 * Readings:
 *   - formats: OCP FP8 E4M3 (bias 7, no infinities, S.1111.111 is NaN, max 448) and E5M2
 *     (bias 15, IEEE-like: exponent 31 is inf/NaN, max 57344); byte = s << 7 | e << M | m;
 *   - conversion from BF16 (done once, when a page completes): round to nearest, ties to
 *     even; magnitudes beyond the largest finite value (infinities included) saturate to it;
 *     NaN becomes the NaN byte 0x7F with the input's sign (E4M3 S.1111.111, E5M2 S.11111.11);
 *   - tile: one (page, KV head, K|V) slice of 2048 FP8 values in the storage order of the
 *     12-bit format; group q = 8L + 2j + f = elements (L, f, i = 0..7) of block j;
 *   - group modes (as the BF16 codec, on the exponent field e): 0 if every e - b3 is in
 *     [0,8), else 1 if every e - b4 is in [0,16), else 2 (code = e).  For E4M3 the
 *     16-wide window is the whole 4-bit field: b4 = 0 whatever the table holds (its E4M3
 *     b4 entries are not read), so mode 1 takes every group that mode 0 does not and
 *     mode 2 never occurs;
 *   - layout (S = 1 + M sign/mantissa bits: 3 for E5M2, 4 for E4M3):
 *       [0, 256 S)           sign/mantissa fields: group q at S*q bytes, element i at bits
 *                            S*i .. S*i+S-1 (value s << M | m), little-endian
 *       [256 S, 256 S + 768) 3-bit codes: group q at 3q, element i at bits 3i..3i+2
 *       then 64 bytes        2-bit modes: group q at byte q/4, bits 2(q%4)
 *       then 64 bytes        escapes in q order: mode 1: one byte, bit i = bit 3 of code i;
 *                            mode 2 (E5M2): two bytes, bits 3..4 of code i at bits 2i..2i+1
 *                            of a little-endian 16-bit field; zero padded
 *     E5M2 tile 1664 bytes (26 granules of 64), E4M3 1920 bytes (30 granules); a tile whose
 *     escapes exceed 64 bytes stays raw: 2048 FP8 bytes, element (L,f,i) of block j at
 *     512j + 16L + 8f + i (32 granules);
 *   - calibration: as the BF16 codec, over FP8 exponent fields (E4M3: b4 = 0);
 *   - pages and entries: as oga.c (uint32 entry: 64-byte granule offset, bit 31 = raw).
 */
#include "oref.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int ebits, mbits, bias, sm_bits;
    double max_finite;
} f8fmt;

static f8fmt fmt_of(int fmt)
{
    f8fmt f;
    if (fmt == OF8_E4M3) {
        f.ebits = 4; f.mbits = 3; f.bias = 7; f.max_finite = 448.0;
    } else {
        f.ebits = 5; f.mbits = 2; f.bias = 15; f.max_finite = 57344.0;
    }
    f.sm_bits = 1 + f.mbits;
    return f;
}

/* value of an FP8 byte; NaN for NaN codes, +-inf for E5M2 infinities */
double of8_value(int fmt, uint8_t b)
{
    const f8fmt F = fmt_of(fmt);
    const int s = b >> 7, e = (b >> F.mbits) & ((1 << F.ebits) - 1), m = b & ((1 << F.mbits) - 1);
    const int emax = (1 << F.ebits) - 1;
    double v;
    if (fmt == OF8_E4M3 && e == emax && m == 7) return NAN;
    if (fmt == OF8_E5M2 && e == emax) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, 1 - F.bias - F.mbits);
    else v = ldexp(1.0 + (double)m / (1 << F.mbits), e - F.bias);
    return s ? -v : v;
}

static int is_finite_code(int fmt, int b)
{
    const double v = of8_value(fmt, (uint8_t)b);
    return !isnan(v) && !isinf(v);
}

/* BF16 word -> FP8 byte: nearest finite value (ties to the even mantissa), saturating */
uint8_t of8_from_bf16(int fmt, uint16_t w)
{
    const f8fmt F = fmt_of(fmt);
    const double x = oref_bf16_value(w);
    const int sign = (w >> 15) & 1;
    if (isnan(x)) return (uint8_t)(sign << 7 | 0x7F);
    const double a = fabs(x);
    if (a >= F.max_finite) {
        for (int b = 127; b >= 0; b--)
            if (is_finite_code(fmt, b)) return (uint8_t)(sign << 7 | b);
    }
    int best = 0;
    double best_d = INFINITY;
    for (int b = 0; b < 128; b++) {
        if (!is_finite_code(fmt, b)) continue;
        const double d = fabs(of8_value(fmt, (uint8_t)b) - a);
        if (d < best_d || (d == best_d && (b & 1) == 0)) {
            best_d = d;
            best = b;
        }
    }
    return (uint8_t)(sign << 7 | best);
}

static unsigned f8_exp(const f8fmt *F, uint8_t b) { return (b >> F->mbits) & ((1u << F->ebits) - 1); }

static int tile_bytes(const f8fmt *F) { return 256 * F->sm_bits + 768 + 64 + 64; }

int of8_tile_bytes(int fmt)
{
    const f8fmt F = fmt_of(fmt);
    return tile_bytes(&F);
}

/* ---------------------------------------------------------------------------------
 * calibration over FP8 exponent fields (pages: FP8 bytes [n][16][128])
 * ------------------------------------------------------------------------------- */
static unsigned best_window(const uint64_t *hist, int nvals, int width)
{
    uint64_t best = 0;
    unsigned best_b = 0;
    for (int b = 0; b + width <= nvals; b++) {
        uint64_t cov = 0;
        for (int e = b; e < b + width; e++) cov += hist[e];
        if (cov > best) {
            best = cov;
            best_b = (unsigned)b;
        }
    }
    return best_b;
}

void of8_calibrate(int fmt, const uint8_t *pages, int64_t n, uint8_t *b3, uint8_t *b4)
{
    const f8fmt F = fmt_of(fmt);
    const int nvals = 1 << F.ebits;
    for (int ch = 0; ch < 128; ch++) {
        uint64_t hist[32];
        memset(hist, 0, sizeof hist);
        for (int64_t p = 0; p < n; p++)
            for (int t = 0; t < 16; t++) hist[f8_exp(&F, pages[(p * 16 + t) * 128 + ch])]++;
        b3[ch] = (uint8_t)best_window(hist, nvals, 8);
        b4[ch] = fmt == OF8_E4M3 ? 0 : (uint8_t)best_window(hist, nvals, 16);
    }
}

/* ---------------------------------------------------------------------------------
 * tiles
 * ------------------------------------------------------------------------------- */
static void put_bits(uint8_t *base, int bitpos, int nbits, unsigned v)
{
    for (int k = 0; k < nbits; k++)
        if ((v >> k) & 1u) base[(bitpos + k) >> 3] |= (uint8_t)(1u << ((bitpos + k) & 7));
}

static unsigned get_bits(const uint8_t *base, int bitpos, int nbits)
{
    unsigned v = 0;
    for (int k = 0; k < nbits; k++) v |= (unsigned)((base[(bitpos + k) >> 3] >> ((bitpos + k) & 7)) & 1u) << k;
    return v;
}

/* page: FP8 bytes [16][128]; returns the tile size (compressed) or 2048 (raw) */
int of8_encode_tile(int fmt, const uint8_t *page, int is_v, const uint8_t *b3c, const uint8_t *b4c, uint8_t *out)
{
    const f8fmt F = fmt_of(fmt);
    const int sm_off = 0, code_off = 256 * F.sm_bits, tag_off = code_off + 768, esc_off = tag_off + 64;
    const int size = tile_bytes(&F);
    uint8_t tile[1920];
    uint8_t esc[256 * 2];
    int nesc = 0;
    memset(tile, 0, sizeof tile);
    for (int L = 0; L < 32; L++)
        for (int j = 0; j < 4; j++)
            for (int f = 0; f < 2; f++) {
                const int q = 8 * L + 2 * j + f;
                unsigned e[8], b3[8], b4[8], sm[8];
                for (int i = 0; i < 8; i++) {
                    int tok, dim;
                    oref_block_position(is_v, j, L, f, i, &tok, &dim);
                    const uint8_t b = page[tok * 128 + dim];
                    e[i] = f8_exp(&F, b);
                    sm[i] = ((unsigned)(b >> 7) << F.mbits) | (b & ((1u << F.mbits) - 1));
                    b3[i] = b3c[dim];
                    b4[i] = fmt == OF8_E4M3 ? 0u : b4c[dim];
                }
                const int mode = oga_group_mode(e, b3, b4);
                for (int i = 0; i < 8; i++) {
                    const unsigned c = e[i] - (mode == 0 ? b3[i] : mode == 1 ? b4[i] : 0u);
                    put_bits(tile + sm_off, (F.sm_bits * 8) * q + F.sm_bits * i, F.sm_bits, sm[i]);
                    put_bits(tile + code_off, 24 * q + 3 * i, 3, c & 7u);
                }
                tile[tag_off + q / 4] |= (uint8_t)(mode << (2 * (q % 4)));
                if (mode == 1) {
                    uint8_t hb = 0;
                    for (int i = 0; i < 8; i++)
                        hb |= (uint8_t)((((e[i] - b4[i]) >> 3) & 1u) << i);
                    esc[nesc++] = hb;
                } else if (mode == 2) {
                    unsigned hb = 0;
                    for (int i = 0; i < 8; i++) hb |= ((e[i] >> 3) & 3u) << (2 * i);
                    esc[nesc++] = (uint8_t)hb;
                    esc[nesc++] = (uint8_t)(hb >> 8);
                }
            }
    if (nesc > 64) {
        for (int j = 0; j < 4; j++)
            for (int L = 0; L < 32; L++)
                for (int f = 0; f < 2; f++)
                    for (int i = 0; i < 8; i++) {
                        int tok, dim;
                        oref_block_position(is_v, j, L, f, i, &tok, &dim);
                        out[512 * j + 16 * L + 8 * f + i] = page[tok * 128 + dim];
                    }
        return 2048;
    }
    memcpy(tile + esc_off, esc, (size_t)nesc);
    memcpy(out, tile, (size_t)size);
    return size;
}

void of8_decode_tile(int fmt, const uint8_t *in, int raw, int is_v, const uint8_t *b3c, const uint8_t *b4c,
                     uint8_t *page)
{
    const f8fmt F = fmt_of(fmt);
    const int code_off = 256 * F.sm_bits, tag_off = code_off + 768, esc_off = tag_off + 64;
    int at = esc_off;
    for (int L = 0; L < 32; L++)
        for (int j = 0; j < 4; j++)
            for (int f = 0; f < 2; f++) {
                const int q = 8 * L + 2 * j + f;
                const int mode = raw ? 0 : (in[tag_off + q / 4] >> (2 * (q % 4))) & 3;
                unsigned hb = 0;
                if (!raw && mode == 1) hb = in[at++];
                if (!raw && mode == 2) {
                    hb = (unsigned)in[at] | ((unsigned)in[at + 1] << 8);
                    at += 2;
                }
                for (int i = 0; i < 8; i++) {
                    int tok, dim;
                    oref_block_position(is_v, j, L, f, i, &tok, &dim);
                    uint8_t b;
                    if (raw) {
                        b = in[512 * j + 16 * L + 8 * f + i];
                    } else {
                        unsigned c = get_bits(in + code_off, 24 * q + 3 * i, 3);
                        if (mode == 1) c |= ((hb >> i) & 1u) << 3;
                        if (mode == 2) c |= ((hb >> (2 * i)) & 3u) << 3;
                        const unsigned b4 = fmt == OF8_E4M3 ? 0u : b4c[dim];
                        const unsigned e = c + (mode == 0 ? b3c[dim] : mode == 1 ? b4 : 0u);
                        const unsigned sm = get_bits(in, (F.sm_bits * 8) * q + F.sm_bits * i, F.sm_bits);
                        b = (uint8_t)(((sm >> F.mbits) << 7) | ((e & ((1u << F.ebits) - 1)) << F.mbits) |
                                      (sm & ((1u << F.mbits) - 1)));
                    }
                    page[tok * 128 + dim] = b;
                }
            }
}

/* ---------------------------------------------------------------------------------
 * pages of one layer: BF16 raw pool in, FP8 tiles out (conversion, then coding);
 * bases [hkv][2][2][128]; entries uint32 (64-byte granule offset | raw << 31)
 * ------------------------------------------------------------------------------- */
void of8_quantize(int fmt, const uint16_t *in, int64_t n, uint8_t *out)
{
    for (int64_t k = 0; k < n; k++) out[k] = of8_from_bf16(fmt, in[k]);
}

int of8_encode_pages(int fmt, int hkv, const uint16_t *raw_pool, int64_t num_raw_pages, const uint8_t *bases,
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
    if (arena_granules > 0x7FFFFFFFull) arena_granules = 0x7FFFFFFFull;
    uint8_t page[2048], buf[2048];
    for (int p = 0; p < n; p++) {
        uint32_t *cur = &cursors[2 * dst_seq[p]];
        for (int h = 0; h < hkv; h++)
            for (int kv = 0; kv < 2; kv++) {
                of8_quantize(fmt, raw_pool + (((int64_t)src_page[p] * hkv + h) * 2 + kv) * 2048, 2048, page);
                const uint8_t *bb = bases + ((size_t)h * 2 + kv) * 256;
                const int size = of8_encode_tile(fmt, page, kv, bb, bb + 128, buf);
                const uint64_t gran = (uint64_t)size / 64, off = cur[0];
                uint32_t *m = &meta[((int64_t)dst_page[p] * hkv + h) * 2 + kv];
                if (off + gran > cur[1] || off + gran > arena_granules) {
                    status |= OREF_ARENA_FULL;
                    *m = 0xFFFFFFFFu;
                } else {
                    memcpy(arena + off * 64, buf, (size_t)size);
                    *m = (uint32_t)off | (size == 2048 ? 0x80000000u : 0u);
                }
                cur[0] = (uint32_t)(off + gran);
            }
    }
    return status;
}

int of8_decode_entry(int fmt, uint32_t entry, const uint8_t *arena, uint64_t arena_bytes, int is_v,
                     const uint8_t *bb, uint8_t *half_page)
{
    const uint64_t off = entry & 0x7FFFFFFFu;
    const int raw = (entry >> 31) != 0;
    const uint64_t size = raw ? 2048 : (uint64_t)of8_tile_bytes(fmt);
    if (entry == 0xFFFFFFFFu || off * 64 + size > arena_bytes) {
        memset(half_page, 0, 2048);
        return OREF_BAD_META;
    }
    of8_decode_tile(fmt, arena + off * 64, raw, is_v, bb, bb + 128, half_page);
    return 0;
}

int of8_decode_pages(int fmt, int hkv, const uint32_t *meta, int64_t num_meta_pages, const uint8_t *arena,
                     uint64_t arena_bytes, const uint8_t *bases, const int32_t *page, int32_t n, uint8_t *out)
{
    int status = 0;
    for (int p = 0; p < n; p++)
        for (int h = 0; h < hkv; h++)
            for (int kv = 0; kv < 2; kv++) {
                uint8_t *dst = out + (((int64_t)p * hkv + h) * 2 + kv) * 2048;
                if (page[p] < 0 || page[p] >= num_meta_pages) {
                    memset(dst, 0, 2048);
                    status |= OREF_BAD_INDEX;
                    continue;
                }
                status |= of8_decode_entry(fmt, meta[((int64_t)page[p] * hkv + h) * 2 + kv], arena, arena_bytes, kv,
                                           bases + ((size_t)h * 2 + kv) * 256, dst);
            }
    return status;
}
