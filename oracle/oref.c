/*
 * oref.c -- the CPU oracle for the 12-bit lossless BF16 KV block format and for
 * paged GQA decode attention over it.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, scalar restatement of what
 * the GPU library computes, written to be checked by eye against the pages it
 * follows.  Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load it.  It shares no code, header, table or constant with the CUDA library
 * (decode_attention_value_gb300/csrc) and must never be called by it.
 *
 * Sources (page titles, sections):
 *   [ZF]   "ZipFusion: Fusing Lossless KV Decompression with Attention for Efficient
 *          LLM Decoding", section "How it works", steps 1-4, the operand-role layout
 *          paragraph and the metadata paragraph.
 *   [GA]   "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference on
 *          Personal Devices", sections "Attention with On-the-Fly Decompression" and
 *          "Block-Wise Compression Scheduling".
 *   [EX]   "ExANS: lossless GPU compression for BF16 KV cache", section "Under the
 *          hood" (the BF16 field boundary and value formula).
 *
 * Readings of points the pages leave open:
 *   - a 16-token page of one layer, one KV head and one of K/V is a 16 x 128 BF16
 *     matrix [token][dim]; block j (0..3) is dims [32j, 32j+32) x all 16 tokens;
 *   - inside a block the 512 values are stored in "storage order" n = (L*2+f)*8+i
 *     for lane L (0..31), fragment f (0..1), element i (0..7), where with g = L/4,
 *     t = L%4, r = g + 8*((i/2)%2), c = 2t + i%2 + 8*(i/4):
 *         K block: token r,        dim 32j + 16f + c
 *         V block: token c,        dim 32j + 16f + r
 *     (this is the per-thread element set of a 16x16 tensor-core A operand, with K
 *     rows = tokens and V rows = dims, i.e. K and V each laid out for its own role);
 *   - an eligible block is 768 bytes: bytes [0,512) hold the low byte of value n at
 *     16L + 8f + i, bytes [512,768) hold the code bytes, code byte 512 + 8L + 4f + k
 *     (k = 0..3) pairing elements i = k and i = k+4 as
 *         bit 7 = sign(k), bits 6..4 = d(k+4), bit 3 = sign(k+4), bits 2..0 = d(k);
 *   - a raw block is 1024 bytes: value n as a little-endian 16-bit word at byte 2n;
 *   - group metadata (one 64-bit word, little-endian): bits 0..31 the first block's
 *     offset in 256-byte granules from the arena base, bits 32..63 the four tag
 *     bytes, tag = b/2 for an eligible block, 0xFF for a raw block;
 *   - group order inside one encode call: page (call order) -> KV head -> K then V;
 *     each page's groups are appended at its destination cursor;
 *   - softmax scale 1/sqrt(128), output in double.
 */
#include "oref.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------------------
 * BF16 fields: sign 1 bit, exponent 8 bits, fraction 7 bits ([ZF] "How it works";
 * [EX] "Under the hood").
 * ------------------------------------------------------------------------------- */
static unsigned sign_of(uint16_t w) { return (w >> 15) & 1u; }
static unsigned exponent_of(uint16_t w) { return (w >> 7) & 0xFFu; }
static unsigned fraction_of(uint16_t w) { return w & 0x7Fu; }

unsigned oref_bf16_exponent(uint16_t w) { return exponent_of(w); }

/* Position inside the 16x128 page of value (L, f, i) of block j. */
void oref_block_position(int is_v, int j, int L, int f, int i, int *token, int *dim)
{
    int g = L / 4, t = L % 4;
    int r = g + 8 * ((i / 2) % 2);
    int c = 2 * t + (i % 2) + 8 * (i / 4);
    if (!is_v) {
        *token = r;
        *dim = 32 * j + 16 * f + c;
    } else {
        *token = c;
        *dim = 32 * j + 16 * f + r;
    }
}

/* Gather block j of a 16x128 page into storage order. */
static void gather_block(const uint16_t *page, int is_v, int j, uint16_t v[512])
{
    for (int L = 0; L < 32; L++)
        for (int f = 0; f < 2; f++)
            for (int i = 0; i < 8; i++) {
                int tok, dim;
                oref_block_position(is_v, j, L, f, i, &tok, &dim);
                v[(L * 2 + f) * 8 + i] = page[tok * 128 + dim];
            }
}

/* ---------------------------------------------------------------------------------
 * [ZF] steps 2-3: base, eligibility, 12-bit code.
 * Returns the number of bytes written to out (768 or 1024) and sets *tag.
 * ------------------------------------------------------------------------------- */
int oref_encode_block(const uint16_t *page, int is_v, int j, uint8_t *out, uint8_t *tag)
{
    uint16_t v[512];
    gather_block(page, is_v, j, v);

    unsigned mn = 255, mx = 0;
    for (int n = 0; n < 512; n++) {
        unsigned e = exponent_of(v[n]);
        if (e < mn) mn = e;
        if (e > mx) mx = e;
    }
    /* step 2: b is the minimum exponent rounded down to an even number */
    unsigned b = (mn / 2) * 2;
    /* step 2: compressed only if every exponent lies in [b, b+15] */
    int eligible = 1;
    for (int n = 0; n < 512; n++) {
        unsigned e = exponent_of(v[n]);
        if (e < b || e > b + 15) eligible = 0;
    }

    if (!eligible) {
        for (int n = 0; n < 512; n++) {
            out[2 * n] = (uint8_t)(v[n] & 0xFF);
            out[2 * n + 1] = (uint8_t)(v[n] >> 8);
        }
        *tag = 0xFF;
        return 1024;
    }

    /* step 3: keep the low byte (exponent LSB + 7 fraction bits); add sign and
     * d = floor((e - b) / 2) */
    for (int L = 0; L < 32; L++)
        for (int f = 0; f < 2; f++) {
            unsigned s[8], d[8];
            for (int i = 0; i < 8; i++) {
                uint16_t w = v[(L * 2 + f) * 8 + i];
                unsigned e = exponent_of(w);
                out[16 * L + 8 * f + i] = (uint8_t)(((e & 1u) << 7) | fraction_of(w));
                s[i] = sign_of(w);
                d[i] = (e - b) / 2;
            }
            for (int k = 0; k < 4; k++)
                out[512 + 8 * L + 4 * f + k] =
                    (uint8_t)((s[k] << 7) | (d[k + 4] << 4) | (s[k + 4] << 3) | d[k]);
        }
    *tag = (uint8_t)(b / 2);
    return 768;
}

/* ---------------------------------------------------------------------------------
 * [ZF] step 4: restore e = b + 2d + r, with r the exponent bit kept in the low byte.
 * Writes the block's 512 values back to their page positions.  A tag in 0x80..0xFE
 * is not a valid block; the function then returns -1 and writes nothing.
 * ------------------------------------------------------------------------------- */
int oref_decode_block(const uint8_t *in, uint8_t tag, int is_v, int j, uint16_t *page)
{
    uint16_t v[512];
    if (tag == 0xFF) {
        for (int n = 0; n < 512; n++) v[n] = (uint16_t)(in[2 * n] | (in[2 * n + 1] << 8));
    } else if (tag >= 0x80) {
        return -1;
    } else {
        unsigned b = 2u * tag;
        for (int L = 0; L < 32; L++)
            for (int f = 0; f < 2; f++)
                for (int i = 0; i < 8; i++) {
                    uint8_t lo = in[16 * L + 8 * f + i];
                    uint8_t code = in[512 + 8 * L + 4 * f + (i % 4)];
                    unsigned s, d;
                    if (i < 4) {
                        s = (code >> 7) & 1u;
                        d = code & 7u;
                    } else {
                        s = (code >> 3) & 1u;
                        d = (code >> 4) & 7u;
                    }
                    unsigned r = (lo >> 7) & 1u;
                    unsigned e = b + 2 * d + r;
                    unsigned frac = lo & 0x7Fu;
                    v[(L * 2 + f) * 8 + i] = (uint16_t)((s << 15) | ((e & 0xFFu) << 7) | frac);
                }
    }
    for (int L = 0; L < 32; L++)
        for (int f = 0; f < 2; f++)
            for (int i = 0; i < 8; i++) {
                int tok, dim;
                oref_block_position(is_v, j, L, f, i, &tok, &dim);
                page[tok * 128 + dim] = v[(L * 2 + f) * 8 + i];
            }
    return tag == 0xFF ? 1024 : 768;
}

/* Size of a block in 256-byte granules from its tag: 3 (768 B) or 4 (1024 B). */
static uint32_t granules_of_tag(uint8_t tag) { return tag == 0xFF ? 4u : 3u; }

static int tag_valid(uint8_t tag) { return tag < 0x80 || tag == 0xFF; }

/* ---------------------------------------------------------------------------------
 * Encode a list of completed pages of one layer ([GA] "Block-Wise Compression
 * Scheduling": a page is encoded once, when it completes).
 *
 * raw_pool:  [num_raw_pages][Hkv][2][16][128] BF16 words (2 = K, V)
 * src_page:  raw page to encode, per call entry
 * dst_page:  metadata page index it becomes
 * dst_seq:   cursor it is appended to; must be non-decreasing over the call
 * meta:      [num_meta_pages][Hkv][2] 64-bit words
 * cursors:   [num_cursors][2] = {next free granule, end granule (exclusive)}
 *
 * For every page in call order, every head, K then V, the group's four blocks are
 * placed contiguously at the cursor ([ZF] metadata paragraph: blocks are located by
 * summing prior sizes) and the cursor advances by the group size.  A group that would
 * end past the cursor's end or past the arena is not written: its offset is stored
 * as 0xFFFFFFFF and status gets OREF_ARENA_FULL (the cursor still advances).
 * An out-of-range index or a decreasing dst_seq makes the whole call a no-op.
 * ------------------------------------------------------------------------------- */
int oref_encode_pages(int hkv, const uint16_t *raw_pool, int64_t num_raw_pages,
                      const int32_t *src_page, const int32_t *dst_page, const int32_t *dst_seq,
                      int32_t n, uint64_t *meta, int64_t num_meta_pages, uint8_t *arena,
                      uint64_t arena_bytes, uint32_t *cursors, int32_t num_cursors)
{
    int status = 0;
    for (int p = 0; p < n; p++) {
        if (src_page[p] < 0 || src_page[p] >= num_raw_pages || dst_page[p] < 0 ||
            dst_page[p] >= num_meta_pages || dst_seq[p] < 0 || dst_seq[p] >= num_cursors)
            status |= OREF_BAD_INDEX;
        if (p > 0 && dst_seq[p] < dst_seq[p - 1]) status |= OREF_BAD_ORDER;
    }
    if (status) return status;

    uint64_t arena_granules = arena_bytes / 256;
    uint8_t buf[4][1024];
    for (int p = 0; p < n; p++) {
        uint32_t *cur = &cursors[2 * dst_seq[p]];
        for (int h = 0; h < hkv; h++)
            for (int kv = 0; kv < 2; kv++) {
                const uint16_t *page =
                    raw_pool + (((int64_t)src_page[p] * hkv + h) * 2 + kv) * 16 * 128;
                uint8_t tags[4];
                int sizes[4];
                uint32_t group_granules = 0;
                for (int j = 0; j < 4; j++) {
                    sizes[j] = oref_encode_block(page, kv, j, buf[j], &tags[j]);
                    group_granules += granules_of_tag(tags[j]);
                }
                uint64_t offset0 = cur[0];
                uint64_t word_tags = (uint64_t)tags[0] | ((uint64_t)tags[1] << 8) |
                                     ((uint64_t)tags[2] << 16) | ((uint64_t)tags[3] << 24);
                uint64_t *m = &meta[((int64_t)dst_page[p] * hkv + h) * 2 + kv];
                if (offset0 + group_granules > cur[1] ||
                    offset0 + group_granules > arena_granules) {
                    status |= OREF_ARENA_FULL;
                    *m = 0xFFFFFFFFull | (word_tags << 32);
                } else {
                    uint64_t at = offset0 * 256;
                    for (int j = 0; j < 4; j++) {
                        memcpy(arena + at, buf[j], (size_t)sizes[j]);
                        at += (uint64_t)sizes[j];
                    }
                    *m = offset0 | (word_tags << 32);
                }
                cur[0] = (uint32_t)(offset0 + group_granules);
            }
    }
    return status;
}

/* Locate block j of a group from its metadata word; returns 0 and the byte offset,
 * or a status bit when the word is unusable. */
static int locate_block(uint64_t word, int j, uint64_t arena_bytes, uint64_t *byte_offset,
                        uint8_t *tag)
{
    uint32_t offset0 = (uint32_t)(word & 0xFFFFFFFFull);
    uint8_t tags[4];
    uint64_t group_granules = 0;
    for (int k = 0; k < 4; k++) {
        tags[k] = (uint8_t)(word >> (32 + 8 * k));
        if (!tag_valid(tags[k])) return OREF_BAD_META;
        group_granules += granules_of_tag(tags[k]);
    }
    if (offset0 == 0xFFFFFFFFu) return OREF_BAD_META;
    if (((uint64_t)offset0 + group_granules) * 256 > arena_bytes) return OREF_BAD_META;
    uint64_t g = offset0;
    for (int k = 0; k < j; k++) g += granules_of_tag(tags[k]);
    *byte_offset = g * 256;
    *tag = tags[j];
    return 0;
}

/* Decode one (page, head, K|V) 16x128 half-page from its group; on a bad word the
 * half-page is zero-filled and the status bit returned. */
static int decode_group(uint64_t word, const uint8_t *arena, uint64_t arena_bytes, int is_v,
                        uint16_t *half_page)
{
    for (int j = 0; j < 4; j++) {
        uint64_t at;
        uint8_t tag;
        int st = locate_block(word, j, arena_bytes, &at, &tag);
        if (st) {
            memset(half_page, 0, 16 * 128 * sizeof(uint16_t));
            return st;
        }
        oref_decode_block(arena + at, tag, is_v, j, half_page);
    }
    return 0;
}

/* ---------------------------------------------------------------------------------
 * Standalone decompression: pages -> [n][Hkv][2][16][128] BF16 words.
 * ------------------------------------------------------------------------------- */
int oref_decode_pages(int hkv, const uint64_t *meta, int64_t num_meta_pages, const uint8_t *arena,
                      uint64_t arena_bytes, const int32_t *page, int32_t n, uint16_t *out)
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
                uint64_t word = meta[((int64_t)page[p] * hkv + h) * 2 + kv];
                status |= decode_group(word, arena, arena_bytes, kv, dst);
            }
    return status;
}

/* ---------------------------------------------------------------------------------
 * Decode attention ([GA] "Attention with On-the-Fly Decompression": compressed
 * blocks and the raw tail share one softmax), in double precision.
 *
 * For sequence b with seq_lens[b] = 16*n_full + tail tokens, the first n_full pages
 * come from compressed pages page_ids[b][0..n_full) and the last `tail` tokens from
 * raw page tail_page[b].  Query head h reads KV head h / G, G = Hq / Hkv.
 *   s_t = (q . k_t) / sqrt(128);  o = sum_t exp(s_t - max s) v_t / sum_t exp(s_t - max s)
 * A page whose metadata is unusable is left out of the softmax (status bit set).
 * An empty context gives a zero output.
 * ------------------------------------------------------------------------------- */

static double bf16_to_double(uint16_t w)
{
    /* ([EX] "Under the hood") the BF16 word is the top half of an IEEE-754 binary32 */
    uint32_t u = (uint32_t)w << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oref_bf16_value(uint16_t w) { return bf16_to_double(w); }

/* the BF16 word of a value that BF16 represents exactly (FP8 values) */
static uint16_t bf16_of_double(double v)
{
    const float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

typedef struct {
    int hkv, batch, hq, max_pages, compressed; /* compressed: 0 raw, 1 12-bit blocks, 2 GA tiles */
    const uint16_t *q;
    const int32_t *page_ids, *seq_lens, *tail_page;
    const uint64_t *meta;
    const uint32_t *meta32; /* GA / FP8 tile entries */
    const uint8_t *bases;   /* GA / FP8 bases [hkv][2][2][128] */
    int f8fmt;              /* compressed == 3: OF8_E4M3 or OF8_E5M2 */
    int64_t num_meta_pages;
    const uint8_t *arena;
    uint64_t arena_bytes;
    const uint16_t *raw_pool;
    int64_t num_raw_pages;
    double *out;
    int next_unit;
    int status;
    pthread_mutex_t lock;
} attn_job;

static int attend_unit(attn_job *J, int unit)
{
    int status = 0;
    int b = unit / J->hkv, kvh = unit % J->hkv;
    int G = J->hq / J->hkv;
    int len = J->seq_lens[b];
    int npages = (len + 15) / 16;
    int n_full = len / 16;
    uint16_t *K = (uint16_t *)malloc((size_t)npages * 16 * 128 * sizeof(uint16_t) + 1);
    uint16_t *V = (uint16_t *)malloc((size_t)npages * 16 * 128 * sizeof(uint16_t) + 1);
    int *tok_ok = (int *)calloc((size_t)npages * 16 + 1, sizeof(int));
    double *s = (double *)malloc(((size_t)npages * 16 + 1) * sizeof(double));

    for (int p = 0; p < npages; p++) {
        uint16_t *kp = K + (size_t)p * 16 * 128, *vp = V + (size_t)p * 16 * 128;
        int valid = (p < n_full) ? 16 : len - 16 * n_full;
        int ok = 1;
        if (J->compressed && p < n_full) {
            int pid = J->page_ids[(int64_t)b * J->max_pages + p];
            if (pid < 0 || pid >= J->num_meta_pages) {
                status |= OREF_BAD_INDEX;
                ok = 0;
            } else {
                int st;
                if (J->compressed == 3) {
                    /* FP8 tiles: decode to FP8 bytes, then to the BF16 word of the same value
                       (every FP8 value is a BF16 value) */
                    const uint32_t *m = J->meta32 + ((int64_t)pid * J->hkv + kvh) * 2;
                    const uint8_t *bb = J->bases + (size_t)kvh * 2 * 256;
                    uint8_t k8[2048], v8[2048];
                    st = of8_decode_entry(J->f8fmt, m[0], J->arena, J->arena_bytes, 0, bb, k8);
                    st |= of8_decode_entry(J->f8fmt, m[1], J->arena, J->arena_bytes, 1, bb + 256, v8);
                    for (int k = 0; k < 2048; k++) {
                        kp[k] = bf16_of_double(of8_value(J->f8fmt, k8[k]));
                        vp[k] = bf16_of_double(of8_value(J->f8fmt, v8[k]));
                    }
                } else if (J->compressed == 2) {
                    const uint32_t *m = J->meta32 + ((int64_t)pid * J->hkv + kvh) * 2;
                    const uint8_t *bb = J->bases + (size_t)kvh * 2 * 256;
                    st = oga_decode_entry(m[0], J->arena, J->arena_bytes, 0, bb, kp);
                    st |= oga_decode_entry(m[1], J->arena, J->arena_bytes, 1, bb + 256, vp);
                } else {
                    const uint64_t *m = J->meta + ((int64_t)pid * J->hkv + kvh) * 2;
                    st = decode_group(m[0], J->arena, J->arena_bytes, 0, kp);
                    st |= decode_group(m[1], J->arena, J->arena_bytes, 1, vp);
                }
                if (st) {
                    status |= st;
                    ok = 0;
                }
            }
        } else {
            int pid = J->compressed ? J->tail_page[b] : J->page_ids[(int64_t)b * J->max_pages + p];
            if (pid < 0 || pid >= J->num_raw_pages) {
                status |= J->compressed && pid < 0 ? OREF_BAD_TAIL : OREF_BAD_INDEX;
                ok = 0;
            } else {
                const uint16_t *src = J->raw_pool + ((int64_t)pid * J->hkv + kvh) * 2 * 16 * 128;
                memcpy(kp, src, 16 * 128 * sizeof(uint16_t));
                memcpy(vp, src + 16 * 128, 16 * 128 * sizeof(uint16_t));
            }
        }
        for (int t = 0; t < 16; t++) tok_ok[p * 16 + t] = ok && t < valid;
    }

    const double scale = 1.0 / sqrt(128.0);
    for (int g = 0; g < G; g++) {
        int h = kvh * G + g;
        const uint16_t *qh = J->q + ((int64_t)b * J->hq + h) * 128;
        double *o = J->out + ((int64_t)b * J->hq + h) * 128;
        double mx = -INFINITY;
        for (int t = 0; t < npages * 16; t++) {
            if (!tok_ok[t]) continue;
            double acc = 0.0;
            for (int d = 0; d < 128; d++)
                acc += bf16_to_double(qh[d]) * bf16_to_double(K[(size_t)t * 128 + d]);
            s[t] = acc * scale;
            if (s[t] > mx) mx = s[t];
        }
        double denom = 0.0;
        for (int d = 0; d < 128; d++) o[d] = 0.0;
        for (int t = 0; t < npages * 16; t++) {
            if (!tok_ok[t]) continue;
            double p = exp(s[t] - mx);
            denom += p;
            for (int d = 0; d < 128; d++) o[d] += p * bf16_to_double(V[(size_t)t * 128 + d]);
        }
        if (denom > 0.0)
            for (int d = 0; d < 128; d++) o[d] /= denom;
    }
    free(K);
    free(V);
    free(tok_ok);
    free(s);
    return status;
}

static void *attn_worker(void *arg)
{
    attn_job *J = (attn_job *)arg;
    int units = J->batch * J->hkv;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int u = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (u >= units) break;
        int st = attend_unit(J, u);
        pthread_mutex_lock(&J->lock);
        J->status |= st;
        pthread_mutex_unlock(&J->lock);
    }
    return NULL;
}

static int run_attention(attn_job *J, int nthreads)
{
    J->next_unit = 0;
    J->status = 0;
    pthread_mutex_init(&J->lock, NULL);
    for (int b = 0; b < J->batch; b++) {
        int len = J->seq_lens[b];
        if (J->compressed && len % 16 != 0 && J->tail_page[b] < 0) J->status |= OREF_BAD_TAIL;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads == 1) {
        attn_worker(J);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        for (int i = 0; i < nthreads; i++) pthread_create(&th[i], NULL, attn_worker, J);
        for (int i = 0; i < nthreads; i++) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&J->lock);
    return J->status;
}

int oref_decode_attention(int hkv, int batch, int hq, const uint16_t *q, const int32_t *page_ids,
                          int max_pages, const int32_t *seq_lens, const int32_t *tail_page,
                          const uint64_t *meta, int64_t num_meta_pages, const uint8_t *arena,
                          uint64_t arena_bytes, const uint16_t *raw_pool, int64_t num_raw_pages,
                          double *out, int nthreads)
{
    attn_job J;
    memset(&J, 0, sizeof J);
    J.hkv = hkv;
    J.batch = batch;
    J.hq = hq;
    J.max_pages = max_pages;
    J.compressed = 1;
    J.q = q;
    J.page_ids = page_ids;
    J.seq_lens = seq_lens;
    J.tail_page = tail_page;
    J.meta = meta;
    J.num_meta_pages = num_meta_pages;
    J.arena = arena;
    J.arena_bytes = arena_bytes;
    J.raw_pool = raw_pool;
    J.num_raw_pages = num_raw_pages;
    J.out = out;
    return run_attention(&J, nthreads);
}

int oref_attention_raw(int hkv, int batch, int hq, const uint16_t *q, const int32_t *page_ids,
                       int max_pages, const int32_t *seq_lens, const uint16_t *raw_pool,
                       int64_t num_raw_pages, double *out, int nthreads)
{
    attn_job J;
    memset(&J, 0, sizeof J);
    J.hkv = hkv;
    J.batch = batch;
    J.hq = hq;
    J.max_pages = max_pages;
    J.compressed = 0;
    J.q = q;
    J.page_ids = page_ids;
    J.seq_lens = seq_lens;
    J.raw_pool = raw_pool;
    J.num_raw_pages = num_raw_pages;
    J.out = out;
    return run_attention(&J, nthreads);
}

/* The same attention over group-adaptive tiles (GAAC, "Attention with On-the-Fly
 * Decompression"): finalized pages come from tiles, the partial last page from the
 * raw pool. */
int oref_ga_decode_attention(int hkv, int batch, int hq, const uint16_t *q, const int32_t *page_ids,
                             int max_pages, const int32_t *seq_lens, const int32_t *tail_page,
                             const uint32_t *meta, int64_t num_meta_pages, const uint8_t *arena,
                             uint64_t arena_bytes, const uint8_t *bases, const uint16_t *raw_pool,
                             int64_t num_raw_pages, double *out, int nthreads)
{
    attn_job J;
    memset(&J, 0, sizeof J);
    J.hkv = hkv;
    J.batch = batch;
    J.hq = hq;
    J.max_pages = max_pages;
    J.compressed = 2;
    J.q = q;
    J.page_ids = page_ids;
    J.seq_lens = seq_lens;
    J.tail_page = tail_page;
    J.meta32 = meta;
    J.bases = bases;
    J.num_meta_pages = num_meta_pages;
    J.arena = arena;
    J.arena_bytes = arena_bytes;
    J.raw_pool = raw_pool;
    J.num_raw_pages = num_raw_pages;
    J.out = out;
    return run_attention(&J, nthreads);
}

/* Attention over FP8 tiles (completed pages, converted to FP8 and coded) + BF16 tail. */
int oref_f8_decode_attention(int fmt, int hkv, int batch, int hq, const uint16_t *q, const int32_t *page_ids,
                             int max_pages, const int32_t *seq_lens, const int32_t *tail_page,
                             const uint32_t *meta, int64_t num_meta_pages, const uint8_t *arena,
                             uint64_t arena_bytes, const uint8_t *bases, const uint16_t *raw_pool,
                             int64_t num_raw_pages, double *out, int nthreads)
{
    attn_job J;
    memset(&J, 0, sizeof J);
    J.hkv = hkv;
    J.batch = batch;
    J.hq = hq;
    J.max_pages = max_pages;
    J.compressed = 3;
    J.f8fmt = fmt;
    J.q = q;
    J.page_ids = page_ids;
    J.seq_lens = seq_lens;
    J.tail_page = tail_page;
    J.meta32 = meta;
    J.bases = bases;
    J.num_meta_pages = num_meta_pages;
    J.arena = arena;
    J.arena_bytes = arena_bytes;
    J.raw_pool = raw_pool;
    J.num_raw_pages = num_raw_pages;
    J.out = out;
    return run_attention(&J, nthreads);
}
