/*
 * oref.h -- CPU oracle (test infrastructure only; see oref.c for the sources it
 * restates and the readings it takes).  Not part of the GPU library.
 */
#ifndef OREF_H
#define OREF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status bits reported by the oracle */
#define OREF_ARENA_FULL 1
#define OREF_BAD_INDEX 2
#define OREF_BAD_ORDER 4
#define OREF_BAD_META 8
#define OREF_BAD_TAIL 32

unsigned oref_bf16_exponent(uint16_t w);
double oref_bf16_value(uint16_t w);
void oref_block_position(int is_v, int j, int L, int f, int i, int *token, int *dim);

int oref_encode_block(const uint16_t *page, int is_v, int j, uint8_t *out, uint8_t *tag);
int oref_decode_block(const uint8_t *in, uint8_t tag, int is_v, int j, uint16_t *page);

int oref_encode_pages(int hkv, const uint16_t *raw_pool, int64_t num_raw_pages,
                      const int32_t *src_page, const int32_t *dst_page, const int32_t *dst_seq,
                      int32_t n, uint64_t *meta, int64_t num_meta_pages, uint8_t *arena,
                      uint64_t arena_bytes, uint32_t *cursors, int32_t num_cursors);

int oref_decode_pages(int hkv, const uint64_t *meta, int64_t num_meta_pages, const uint8_t *arena,
                      uint64_t arena_bytes, const int32_t *page, int32_t n, uint16_t *out);

int oref_decode_attention(int hkv, int batch, int hq, const uint16_t *q, const int32_t *page_ids,
                          int max_pages, const int32_t *seq_lens, const int32_t *tail_page,
                          const uint64_t *meta, int64_t num_meta_pages, const uint8_t *arena,
                          uint64_t arena_bytes, const uint16_t *raw_pool, int64_t num_raw_pages,
                          double *out, int nthreads);

int oref_attention_raw(int hkv, int batch, int hq, const uint16_t *q, const int32_t *page_ids,
                       int max_pages, const int32_t *seq_lens, const uint16_t *raw_pool,
                       int64_t num_raw_pages, double *out, int nthreads);

/* group-adaptive additive tiles (oga.c) */
void oga_calibrate(const uint16_t *pages, int64_t n, uint8_t *b3, uint8_t *b4);
int oga_group_mode(const unsigned e[8], const unsigned b3[8], const unsigned b4[8]);
int oga_encode_tile(const uint16_t *page, int is_v, const uint8_t *b3, const uint8_t *b4, uint8_t *out);
void oga_decode_tile(const uint8_t *in, int raw, int is_v, const uint8_t *b3, const uint8_t *b4, uint16_t *page);
int oga_encode_pages(int hkv, const uint16_t *raw_pool, int64_t num_raw_pages, const uint8_t *bases,
                     const int32_t *src_page, const int32_t *dst_page, const int32_t *dst_seq, int32_t n,
                     uint32_t *meta, int64_t num_meta_pages, uint8_t *arena, uint64_t arena_bytes,
                     uint32_t *cursors, int32_t num_cursors);
int oga_decode_entry(uint32_t entry, const uint8_t *arena, uint64_t arena_bytes, int is_v, const uint8_t *bb,
                     uint16_t *half_page);
int oga_decode_pages(int hkv, const uint32_t *meta, int64_t num_meta_pages, const uint8_t *arena,
                     uint64_t arena_bytes, const uint8_t *bases, const int32_t *page, int32_t n, uint16_t *out);
int oref_ga_decode_attention(int hkv, int batch, int hq, const uint16_t *q, const int32_t *page_ids,
                             int max_pages, const int32_t *seq_lens, const int32_t *tail_page,
                             const uint32_t *meta, int64_t num_meta_pages, const uint8_t *arena,
                             uint64_t arena_bytes, const uint8_t *bases, const uint16_t *raw_pool,
                             int64_t num_raw_pages, double *out, int nthreads);

/* FP8 tiles (of8.c) */
#define OF8_E4M3 1
#define OF8_E5M2 2
double of8_value(int fmt, uint8_t b);
uint8_t of8_from_bf16(int fmt, uint16_t w);
int of8_tile_bytes(int fmt);
void of8_calibrate(int fmt, const uint8_t *pages, int64_t n, uint8_t *b3, uint8_t *b4);
int of8_encode_tile(int fmt, const uint8_t *page, int is_v, const uint8_t *b3, const uint8_t *b4, uint8_t *out);
void of8_decode_tile(int fmt, const uint8_t *in, int raw, int is_v, const uint8_t *b3, const uint8_t *b4,
                     uint8_t *page);
void of8_quantize(int fmt, const uint16_t *in, int64_t n, uint8_t *out);
int of8_encode_pages(int fmt, int hkv, const uint16_t *raw_pool, int64_t num_raw_pages, const uint8_t *bases,
                     const int32_t *src_page, const int32_t *dst_page, const int32_t *dst_seq, int32_t n,
                     uint32_t *meta, int64_t num_meta_pages, uint8_t *arena, uint64_t arena_bytes,
                     uint32_t *cursors, int32_t num_cursors);
int of8_decode_entry(int fmt, uint32_t entry, const uint8_t *arena, uint64_t arena_bytes, int is_v,
                     const uint8_t *bb, uint8_t *half_page);
int of8_decode_pages(int fmt, int hkv, const uint32_t *meta, int64_t num_meta_pages, const uint8_t *arena,
                     uint64_t arena_bytes, const uint8_t *bases, const int32_t *page, int32_t n, uint8_t *out);
int oref_f8_decode_attention(int fmt, int hkv, int batch, int hq, const uint16_t *q, const int32_t *page_ids,
                             int max_pages, const int32_t *seq_lens, const int32_t *tail_page,
                             const uint32_t *meta, int64_t num_meta_pages, const uint8_t *arena,
                             uint64_t arena_bytes, const uint8_t *bases, const uint16_t *raw_pool,
                             int64_t num_raw_pages, double *out, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
