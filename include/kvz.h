/*
 * kvz.h -- C ABI of libkvz: lossless 12-bit BF16 KV-cache pages and paged GQA decode
 * attention that reads them, for one NVIDIA GB300 (sm_103a).
 *
 * The block format is the one fixed on the page "ZipFusion: Fusing Lossless KV
 * Decompression with Attention for Efficient LLM Decoding" (section "How it works",
 * steps 1-4, the operand-role layout paragraph and the metadata paragraph); the
 * page lifecycle (encode once on completion, raw BF16 tail until then) and the one
 * shared softmax over compressed pages and the raw tail follow "GAAC: Lossless KV
 * Compression for Bandwidth-Efficient LLM Inference on Personal Devices" (sections
 * "Attention with On-the-Fly Decompression" and "Block-Wise Compression Scheduling").
 *
 * ---------------------------------------------------------------------------------
 * Data layouts (all little-endian; every pointer is DEVICE memory owned by the
 * caller unless stated otherwise; the library never allocates device memory):
 *
 *  raw pool   BF16 [num_raw_pages][Hkv][2][16][128]; [2] = K, V; a page slice is
 *             [token][dim].  Base 16-byte aligned.
 *  block      One (page, KV head, K|V) slice splits into 4 blocks of 512 values;
 *             block j holds dims [32j, 32j+32) of all 16 tokens.  Inside a block the
 *             values are in "storage order": lane L (0..31), fragment f (0..1),
 *             element i (0..7); with g = L/4, t = L%4, r = g + 8*((i/2)%2),
 *             c = 2t + i%2 + 8*(i/4):  K value (token r, dim 32j+16f+c), V value
 *             (token c, dim 32j+16f+r).  This is the per-lane A operand of a 16x16
 *             tensor-core tile in each block's role: K for QK^T, V^T for PV.
 *  eligible   b = min exponent rounded down to even; every exponent in [b, b+15].
 *  block (768 B)  bytes [0,512): low byte of element (L,f,i) at 16L+8f+i (exponent
 *             LSB + 7 fraction bits); bytes [512,768): code byte 512+8L+4f+k pairs
 *             elements k and k+4:  sign_k<<7 | d_(k+4)<<4 | sign_(k+4)<<3 | d_k,
 *             d = (e-b)/2.  Restore: e = b + 2d + r (r = exponent LSB).
 *  raw block (1024 B)  512 BF16 words in storage order.
 *  meta       uint64 [num_meta_pages][Hkv][2]: per (page, head, K|V) group of 4
 *             blocks, bits 0..31 = offset of the group's first block in 256-byte
 *             granules from the arena base, bits 32..63 = one tag byte per block:
 *             b/2 (0..127) or 0xFF = raw.  Block j starts at offset0 + sum over
 *             k<j of (3 or 4) granules.  offset0 = 0xFFFFFFFF marks an unwritten group.
 *  arena      uint8 buffer, 256-byte aligned; groups are placed back to back at
 *             per-cursor positions.
 *  cursors    uint32 [num_cursors][2] = {next free granule, end granule (excl.)}.
 *
 * Error behaviour: every call validates its arguments on the host and returns 0 or
 * a negative KVZ_ERR_* code without launching anything.  Calls are asynchronous on
 * `stream` and never synchronise.  Conditions only the device can see (an index out
 * of range, unusable metadata, a full cursor region, a bounded wait that expired)
 * are OR-ed as KVZ_STATUS_* bits into *status (a device uint32 the caller zeroes and
 * reads when it wants); the offending page or group is skipped, never trapped on.
 */
#ifndef KVZ_H
#define KVZ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVZ_PAGE_TOKENS 16
#define KVZ_HEAD_DIM 128
#define KVZ_GRANULE_BYTES 256
#define KVZ_BLOCK_BYTES_ELIGIBLE 768
#define KVZ_BLOCK_BYTES_RAW 1024
#define KVZ_TAG_RAW 0xFF
#define KVZ_OFFSET_INVALID 0xFFFFFFFFu

/* host-side return codes */
#define KVZ_OK 0
#define KVZ_ERR_INVALID_ARG -1
#define KVZ_ERR_UNSUPPORTED -2
#define KVZ_ERR_ALIGNMENT -3
#define KVZ_ERR_WORKSPACE -4
#define KVZ_ERR_CUDA -5
#define KVZ_ERR_DEVICE -6
#define KVZ_ERR_OUT_OF_SPACE -7
#define KVZ_ERR_NOALLOC_LIMIT -8

/* device-side status bits */
#define KVZ_STATUS_ARENA_FULL 1u
#define KVZ_STATUS_BAD_INDEX 2u
#define KVZ_STATUS_BAD_ORDER 4u
#define KVZ_STATUS_BAD_META 8u
#define KVZ_STATUS_TIMEOUT 16u
#define KVZ_STATUS_BAD_TAIL 32u
#define KVZ_STATUS_Q_RANGE 64u /* FP8 attention: a query beyond the f16 range (|q| >= 65520) */

/* A CUDA stream (same object as cudaStream_t / CUstream); NULL = legacy stream. */
typedef struct CUstream_st *kvz_stream_t;

/* Shapes shared by every call.  head_dim must be 128 and page_size 16. */
typedef struct {
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t page_size;
} kvz_dims;

/* ---------------------------------------------------------------------------------
 * kvz_encode_pages -- compress completed pages of one layer (ZipFusion "How it
 * works" steps 1-3 and the metadata paragraph; GAAC "Block-Wise Compression
 * Scheduling": each page is encoded once, when it completes).
 *
 *  raw_pool         raw pool of this layer (see layouts), num_raw_pages pages
 *  src_page[n]      raw page to encode, per entry
 *  dst_page[n]      meta page index the result is recorded under
 *  dst_seq[n]       cursor the groups are appended at; must be non-decreasing
 *  meta             this layer's metadata table, num_meta_pages pages (16-B aligned)
 *  arena            compressed storage, arena_bytes long (256-B aligned)
 *  cursors          num_cursors cursor pairs, advanced in place
 *  workspace        >= kvz_encode_workspace_size(n) bytes of scratch (16-B aligned)
 * Placement: entries in call order, then KV head, then K before V; each group's four
 * blocks are contiguous at its cursor, which then advances by the group's size.  A
 * group that would pass its cursor's end or the arena is not written (offset0 set to
 * KVZ_OFFSET_INVALID, KVZ_STATUS_ARENA_FULL), the cursor still advances.  An index out
 * of range (KVZ_STATUS_BAD_INDEX) or a decreasing dst_seq (KVZ_STATUS_BAD_ORDER) makes
 * the whole call write nothing.
 * --------------------------------------------------------------------------------- */
size_t kvz_encode_workspace_size(kvz_dims dims, int32_t n);
int kvz_encode_pages(kvz_dims dims, const void *raw_pool, int64_t num_raw_pages,
                     const int32_t *src_page, const int32_t *dst_page, const int32_t *dst_seq,
                     int32_t n, uint64_t *meta, int64_t num_meta_pages, uint8_t *arena,
                     uint64_t arena_bytes, uint32_t *cursors, int32_t num_cursors,
                     void *workspace, size_t workspace_bytes, uint32_t *status,
                     kvz_stream_t stream);

/* kvz_encode_sizes -- the encoder's size pass alone: granules[i] (device uint32) = the
 * 256-byte granules page src_page[i] will take in the arena (all KV heads, K and V: each
 * group 12..16), exactly what kvz_encode_pages will place for it.  Lets the caller
 * reserve exact space (kvz_alloc_reserve_granules) instead of the worst case.  Same
 * validation as kvz_encode_pages for src_page (KVZ_STATUS_BAD_INDEX: no page is read
 * and every granules[i] is 0); workspace: kvz_encode_workspace_size(dims, n). */
int kvz_encode_sizes(kvz_dims dims, const void *raw_pool, int64_t num_raw_pages, const int32_t *src_page,
                     int32_t n, uint32_t *granules, void *workspace, size_t workspace_bytes, uint32_t *status,
                     kvz_stream_t stream);

/* ---------------------------------------------------------------------------------
 * kvz_decode_blocks -- standalone bit-exact decompression (ZipFusion "How it works"
 * step 4), used to check the format and to time decoding on its own.
 *  page[n]     meta page indices;  out_pages: BF16 [n][Hkv][2][16][128] (16-B aligned)
 * A group with unusable metadata is written as zeros (KVZ_STATUS_BAD_META); an out of
 * range page index zero-fills that page (KVZ_STATUS_BAD_INDEX).
 * --------------------------------------------------------------------------------- */
int kvz_decode_blocks(kvz_dims dims, const uint64_t *meta, int64_t num_meta_pages,
                      const uint8_t *arena, uint64_t arena_bytes, const int32_t *page, int32_t n,
                      void *out_pages, uint32_t *status, kvz_stream_t stream);

/* ---------------------------------------------------------------------------------
 * kvz_decode_attention -- GQA paged decode attention over compressed pages plus an
 * uncompressed tail page, one softmax over both (GAAC "Attention with On-the-Fly
 * Decompression"; ZipFusion "How it works": restore in registers, tensor-core QK^T
 * and PV, no decompressed copy in memory).
 *
 *  q            BF16 [batch][num_q_heads][128]; query head h reads KV head h/G,
 *               G = num_q_heads / num_kv_heads (an integer, 1 <= G <= 8)
 *  page_ids     int32 [batch][max_pages] meta page ids of each sequence's completed pages
 *  seq_lens     int32 [batch] tokens in context; the first seq_lens/16 pages come from
 *               page_ids, the last seq_lens%16 tokens from raw page tail_page[b]
 *  tail_page    int32 [batch] raw page id of the tail (-1 when seq_lens%16 == 0)
 *  out          float32 [batch][num_q_heads][128]:
 *               softmax(q.K^T / sqrt(128)) V over the sequence's tokens
 *  workspace    >= kvz_attention_workspace_size(dims, batch, num_q_heads, max_pages + 1)
 *               bytes (16-B aligned); the split-KV partial results
 * Output for an empty sequence is zero.  A page with unusable metadata or an index out
 * of range is left out of the softmax and flagged.
 * Determinism: the work split depends only on (batch, num_kv_heads, seq_lens, the
 * block-table width counted with its tail slot, and the device's SM count), so for
 * the same data this call and kvz_decode_attention_raw (given a table one column
 * wider that ends in the tail page) return bit-identical outputs.
 * --------------------------------------------------------------------------------- */
size_t kvz_attention_workspace_size(kvz_dims dims, int32_t batch, int32_t num_q_heads,
                                    int32_t table_pages);
int kvz_decode_attention(kvz_dims dims, int32_t batch, int32_t num_q_heads, const void *q,
                         const int32_t *page_ids, int32_t max_pages, const int32_t *seq_lens,
                         const int32_t *tail_page, const uint64_t *meta, int64_t num_meta_pages,
                         const uint8_t *arena, uint64_t arena_bytes, const void *raw_pool,
                         int64_t num_raw_pages, float *out, void *workspace,
                         size_t workspace_bytes, uint32_t *status, kvz_stream_t stream);

/* ---------------------------------------------------------------------------------
 * kvz_decode_attention_raw -- the same kernel over plain BF16 pages: the in-run
 * uncompressed baseline.  page_ids [batch][max_pages] are raw page ids covering all
 * ceil(seq_lens/16) pages (the last one possibly partial).  workspace >=
 * kvz_attention_workspace_size(dims, batch, num_q_heads, max_pages).
 * --------------------------------------------------------------------------------- */
int kvz_decode_attention_raw(kvz_dims dims, int32_t batch, int32_t num_q_heads, const void *q,
                             const int32_t *page_ids, int32_t max_pages, const int32_t *seq_lens,
                             const void *raw_pool, int64_t num_raw_pages, float *out,
                             void *workspace, size_t workspace_bytes, uint32_t *status,
                             kvz_stream_t stream);

/* ---------------------------------------------------------------------------------
 * kvz_decode_attention_ex / kvz_decode_attention_raw_ex -- the two attention calls with
 * launch flags.  flags = 0 is exactly kvz_decode_attention / kvz_decode_attention_raw.
 * The pages describe no launch mechanics; this is a GB300 launch option.
 *
 * KVZ_ATTN_OVERLAP_PREVIOUS: the call's kernels are launched as programmatic dependents
 * (CUDA programmatic dependent launch), so its attention kernel may begin while the
 * kernel before it on the stream is still running, and the call's merge kernel lets a
 * programmatic dependent launched after it begin early.  In a decode step this overlaps
 * each layer's start-up (lengths, page table, metadata, the first pages of the stream)
 * with the kernel that produces the layer's queries.  Contract:
 *  - Read before that kernel has finished: seq_lens, page_ids, tail_page, meta, arena,
 *    and every raw page except each sequence's last page (the tail page of the
 *    compressed call; the last page of each sequence in the raw call).  The kernel right
 *    before this call must not write any of these (in particular, a page-completion
 *    encode must not be the kernel right before an overlapped call).
 *  - Read or written only after that kernel has finished and its writes are visible: q,
 *    each sequence's last page, the workspace and out.  The preceding kernel may write q
 *    and the step's new token into the last page.
 *  - status may be OR-ed before that kernel has finished: do not clear it there.
 *  - A kernel launched after this call as a programmatic dependent must wait for this
 *    call to complete (griddepcontrol.wait / cudaGridDependencySynchronize) before it
 *    reads out or reuses the workspace; another overlapped call does so.
 * Results are bit-identical to flags = 0 (same split, same arithmetic).  Flags outside
 * KVZ_ATTN_FLAGS_ALL return KVZ_ERR_INVALID_ARG.
 * --------------------------------------------------------------------------------- */
#define KVZ_ATTN_OVERLAP_PREVIOUS 1u
#define KVZ_ATTN_FLAGS_ALL 1u
int kvz_decode_attention_ex(kvz_dims dims, int32_t batch, int32_t num_q_heads, const void *q,
                            const int32_t *page_ids, int32_t max_pages, const int32_t *seq_lens,
                            const int32_t *tail_page, const uint64_t *meta, int64_t num_meta_pages,
                            const uint8_t *arena, uint64_t arena_bytes, const void *raw_pool,
                            int64_t num_raw_pages, float *out, void *workspace, size_t workspace_bytes,
                            uint32_t *status, uint32_t flags, kvz_stream_t stream);
int kvz_decode_attention_raw_ex(kvz_dims dims, int32_t batch, int32_t num_q_heads, const void *q,
                                const int32_t *page_ids, int32_t max_pages, const int32_t *seq_lens,
                                const void *raw_pool, int64_t num_raw_pages, float *out, void *workspace,
                                size_t workspace_bytes, uint32_t *status, uint32_t flags, kvz_stream_t stream);

/* ---------------------------------------------------------------------------------
 * kvz_decode_attention_noalloc -- kvz_decode_attention for callers that cannot
 * allocate device memory.  The pages describe no such variant; it exists for callers
 * such as runtime plugins whose host framework owns every device allocation, code that
 * must not grow the device footprint while it runs, or work recorded into CUDA graphs
 * under an allocation-free policy.  Arguments and results are those of
 * kvz_decode_attention without the workspace: the split-KV partial results go to a
 * fixed array compiled into libkvz (KVZ_NOALLOC_SCRATCH_BYTES, on every device that
 * loads the library, held until the process exits).  The library allocates nothing.
 *  - A problem whose kvz_attention_workspace_size(dims, batch, num_q_heads,
 *    max_pages + 1) exceeds KVZ_NOALLOC_SCRATCH_BYTES returns KVZ_ERR_NOALLOC_LIMIT
 *    before anything is launched.
 *  - The first call on a device looks up that device's address of the array; make
 *    that first call before any stream capture on that device.
 *  - Every call on a device uses the same array and leaves its contents behind; each
 *    call rewrites all of it that it reads, nothing needs to start at zero.  Calls
 *    whose kernels overlap on the GPU (different streams, no ordering) race on the
 *    array: order them on one stream or use kvz_decode_attention with separate
 *    workspaces.
 * --------------------------------------------------------------------------------- */
#define KVZ_NOALLOC_SCRATCH_BYTES (4u << 20)
int kvz_decode_attention_noalloc(kvz_dims dims, int32_t batch, int32_t num_q_heads, const void *q,
                                 const int32_t *page_ids, int32_t max_pages, const int32_t *seq_lens,
                                 const int32_t *tail_page, const uint64_t *meta, int64_t num_meta_pages,
                                 const uint8_t *arena, uint64_t arena_bytes, const void *raw_pool,
                                 int64_t num_raw_pages, float *out, uint32_t *status, kvz_stream_t stream);

/* ---------------------------------------------------------------------------------
 * Group-adaptive additive tiles: a second compressed format, from the page "GAAC:
 * Lossless KV Compression for Bandwidth-Efficient LLM Inference on Personal Devices"
 * (section "Lossless KV Compression": "Contiguous exponent concentration" and
 * "Group-adaptive additive coding"; Table 9 "Storage"; "Block-Wise Compression
 * Scheduling" for the two storage classes and the 4-byte block-table entry).
 *
 *  bases      uint8 [Hkv][2][2][128] per layer: (head, K|V, b3|b4, channel); b3 is the
 *             start of the 8-exponent window, b4 of the 16-exponent window.
 *  tile       one (page, head, K|V) slice of 2048 values in the storage order above;
 *             group q = 8L + 2j + f is the 8 elements (L, f, i) of block j.  A group
 *             takes mode 0 if every e - b3[channel] is in [0,8), else mode 1 if every
 *             e - b4[channel] is in [0,16), else mode 2 (code = e).  Layout (3008 B):
 *               [0,2048)    sign<<7 | fraction of element (L,f,i) of block j at
 *                           512j + 16L + 8f + i
 *               [2048,2816) 3-bit codes, group q at 2048+3q, element i at bits 3i..3i+2
 *               [2816,2880) 2-bit modes, group q at byte 2816+q/4, bits 2(q%4)
 *               [2880,3008) escape bytes of the mode-1 (1 byte: bit i = bit 3 of code
 *                           i) and mode-2 (5 bytes: bits 3..7 of code i at 5i..5i+4)
 *                           groups in q order, then zeros
 *             A tile needing more than 128 escape bytes is kept raw: 4096 bytes, BF16
 *             words in storage order (the 4 blocks of a raw 12-bit group).
 *  meta32     uint32 [num_meta_pages][Hkv][2] entries: bits 0..30 = tile offset in
 *             64-byte granules from the arena base, bit 31 = raw tile;
 *             KVZ_GA_ENTRY_INVALID = not written.
 *  arena      64-byte aligned; cursors count 64-byte granules (47 per compressed tile,
 *             64 per raw tile).  Offsets above 2^31-1 granules are not representable:
 *             space beyond 128 GiB of one arena is never used.
 * --------------------------------------------------------------------------------- */
#define KVZ_GA_GRANULE_BYTES 64
#define KVZ_GA_TILE_BYTES 3008
#define KVZ_GA_RAW_TILE_BYTES 4096
#define KVZ_GA_ENTRY_RAW 0x80000000u
#define KVZ_GA_ENTRY_INVALID 0xFFFFFFFFu

/* kvz_ga_calibrate -- window bases of one layer ("Contiguous exponent concentration":
 * per head-channel pair and separately for K and V, the 8- and 16-wide exponent windows
 * that cover the most sample values; ties go to the lowest start).
 *  pages[n]   raw page ids of the sample (device int32); bases: uint8 [Hkv][2][2][128]
 * A sample page id out of range is skipped (KVZ_STATUS_BAD_INDEX).  n = 0 gives zeros. */
int kvz_ga_calibrate(kvz_dims dims, const void *raw_pool, int64_t num_raw_pages, const int32_t *pages,
                     int32_t n, uint8_t *bases, uint32_t *status, kvz_stream_t stream);

/* kvz_ga_encode_pages -- kvz_encode_pages for tiles: same arguments, placement and
 * error behaviour, with `bases` (16-B aligned) and uint32 entries (8-B aligned) in
 * 64-byte granules.  workspace: kvz_encode_workspace_size(dims, n). */
int kvz_ga_encode_pages(kvz_dims dims, const void *raw_pool, int64_t num_raw_pages, const uint8_t *bases,
                        const int32_t *src_page, const int32_t *dst_page, const int32_t *dst_seq, int32_t n,
                        uint32_t *meta, int64_t num_meta_pages, uint8_t *arena, uint64_t arena_bytes,
                        uint32_t *cursors, int32_t num_cursors, void *workspace, size_t workspace_bytes,
                        uint32_t *status, kvz_stream_t stream);

/* kvz_ga_decode_blocks -- kvz_decode_blocks for tiles (bit-exact BF16 pages). */
int kvz_ga_decode_blocks(kvz_dims dims, const uint32_t *meta, int64_t num_meta_pages, const uint8_t *arena,
                         uint64_t arena_bytes, const uint8_t *bases, const int32_t *page, int32_t n,
                         void *out_pages, uint32_t *status, kvz_stream_t stream);

/* kvz_ga_decode_attention -- kvz_decode_attention over tiles (GAAC "Attention with
 * On-the-Fly Decompression"): same arguments with uint32 entries and `bases`; same
 * workspace, work split and determinism (bit-identical to kvz_decode_attention_raw on
 * the same data). */
int kvz_ga_decode_attention(kvz_dims dims, int32_t batch, int32_t num_q_heads, const void *q,
                            const int32_t *page_ids, int32_t max_pages, const int32_t *seq_lens,
                            const int32_t *tail_page, const uint32_t *meta, int64_t num_meta_pages,
                            const uint8_t *arena, uint64_t arena_bytes, const uint8_t *bases,
                            const void *raw_pool, int64_t num_raw_pages, float *out, void *workspace,
                            size_t workspace_bytes, uint32_t *status, kvz_stream_t stream);

/* ---------------------------------------------------------------------------------
 * FP8 pages: completed pages converted to FP8 and coded losslessly with the
 * group-adaptive scheme above (GAAC, "Relation to FP8 KV": the codec on KV converted to
 * FP8, Table 7).  The page gives results only; the format carries the BF16 tile over:
 *  conversion  BF16 -> FP8 when a page completes: nearest value, ties to even, saturating
 *              to the largest finite value (infinities included); NaN -> sign | 0x7F.
 *              E4M3: bias 7, no infinities, max 448; E5M2: bias 15, max 57344.
 *  tile        2048 FP8 values in storage order, group q = 8L + 2j + f.  With M mantissa
 *              bits and S = 1 + M (E5M2 3, E4M3 4):
 *                [0, 256 S)      sign/mantissa fields s << M | m, group q at S*q, element i
 *                                at bits S*i (little-endian)
 *                [+0, +768)      3-bit exponent codes, group q at 3q
 *                [+768, +832)    2-bit modes, group q at byte q/4, bits 2(q%4)
 *                [+832, +896)    escapes: mode 1 one byte (bit 3 of code i at bit i);
 *                                mode 2 (E5M2 only) two bytes (bits 3..4 of code i at 2i)
 *              modes on the exponent field e: 0 if all e - b3 in [0,8), 1 if all e - b4 in
 *              [0,16), else 2 (code = e); E4M3 takes b4 = 0 (the table's E4M3 b4 entries
 *              are not read), so its groups use modes 0 and 1 only.  E5M2 tile 1664 B (26 granules
 *              of 64), E4M3 1920 B (30); more than 64 escape bytes: raw tile of 2048 FP8
 *              bytes, element (L, f, i) of block j at 512j + 16L + 8f + i.
 *  entries, bases, arena, cursors: as the group-adaptive tiles.  The tail page stays BF16.
 * --------------------------------------------------------------------------------- */
#define KVZ_F8_E4M3 1
#define KVZ_F8_E5M2 2

/* Bases [Hkv][2][2][128] over the FP8 exponent fields of the converted sample pages. */
int kvz_f8_calibrate(kvz_dims dims, int32_t format, const void *raw_pool, int64_t num_raw_pages,
                     const int32_t *pages, int32_t n, uint8_t *bases, uint32_t *status, kvz_stream_t stream);
/* kvz_ga_encode_pages for FP8: converts each completed BF16 page, then codes it. */
int kvz_f8_encode_pages(kvz_dims dims, int32_t format, const void *raw_pool, int64_t num_raw_pages,
                        const uint8_t *bases, const int32_t *src_page, const int32_t *dst_page,
                        const int32_t *dst_seq, int32_t n, uint32_t *meta, int64_t num_meta_pages,
                        uint8_t *arena, uint64_t arena_bytes, uint32_t *cursors, int32_t num_cursors,
                        void *workspace, size_t workspace_bytes, uint32_t *status, kvz_stream_t stream);
/* Decode to the stored FP8 bytes: out uint8 [n][Hkv][2][16][128] (16-B aligned). */
int kvz_f8_decode_blocks(kvz_dims dims, int32_t format, const uint32_t *meta, int64_t num_meta_pages,
                         const uint8_t *arena, uint64_t arena_bytes, const uint8_t *bases, const int32_t *page,
                         int32_t n, void *out_pages, uint32_t *status, kvz_stream_t stream);
/* kvz_decode_attention over FP8 tiles plus the BF16 tail; same workspace, split and
 * determinism.  FP8 pages are multiplied in f16 (every FP8 value is an f16 value): the
 * queries are rounded to f16 for them, which is exact for |q| in [2^-17, 65504]; larger
 * queries overflow (flagged as KVZ_STATUS_Q_RANGE; that output is not usable), so q must
 * stay below 65504 in magnitude.  The tail page is multiplied in BF16 with the BF16
 * queries. */
int kvz_f8_decode_attention(kvz_dims dims, int32_t format, int32_t batch, int32_t num_q_heads, const void *q,
                            const int32_t *page_ids, int32_t max_pages, const int32_t *seq_lens,
                            const int32_t *tail_page, const uint32_t *meta, int64_t num_meta_pages,
                            const uint8_t *arena, uint64_t arena_bytes, const uint8_t *bases,
                            const void *raw_pool, int64_t num_raw_pages, float *out, void *workspace,
                            size_t workspace_bytes, uint32_t *status, kvz_stream_t stream);

/* ---------------------------------------------------------------------------------
 * Host-side chunk allocator for the arena (GAAC "Block-Wise Compression Scheduling":
 * two fixed storage classes, 768-byte and 1024-byte block slots; ZipFusion: the memory
 * manager tracks the space left, hands chunks freed by one layer or sequence to
 * another, and reports capacity).  Pure host code, no device memory is touched.
 *
 * The arena is cut into fixed chunks of chunk_granules granules.  Each cursor (one per
 * sequence, shared by all its layers) owns a chain of chunks and a device cursor pair.
 * Before an encode call the caller asks kvz_alloc_reserve for room for `pages` pages
 * on each cursor: the allocator keeps an upper bound of every cursor's position
 * (pos + worst case of every reservation since the last observation), and when the
 * worst case of the new pages does not fit the current chunk it takes a fresh chunk.
 * The cursor pairs the device must hold before the encode are returned as updates
 * (cursor index, pos, end) for the caller to copy to the device.  kvz_alloc_observe
 * feeds back a device snapshot of the cursors taken after reservation `ticket`, which
 * tightens the bounds.  kvz_alloc_release returns a finished sequence's chunks.
 * --------------------------------------------------------------------------------- */
typedef struct kvz_alloc kvz_alloc;
int kvz_alloc_create(uint64_t arena_bytes, uint32_t chunk_granules, int32_t num_cursors,
                     int32_t num_kv_heads, kvz_alloc **out);
void kvz_alloc_destroy(kvz_alloc *a);
/* pages[k] pages for cursor cursor_ids[k] (host arrays, k < count, each cursor at most
 * once).  upd_idx/upd_pos/upd_end (host, capacity `count`) receive *n_upd updates;
 * *ticket identifies the reservation.  Returns KVZ_ERR_OUT_OF_SPACE (nothing changed)
 * when no free chunk is left for a cursor that needs one. */
int kvz_alloc_reserve(kvz_alloc *a, const int32_t *cursor_ids, const int32_t *pages, int32_t count,
                      int32_t *upd_idx, uint32_t *upd_pos, uint32_t *upd_end, int32_t *n_upd,
                      uint64_t *ticket);
/* Like kvz_alloc_reserve with exact sizes: granules[k] granules for cursor cursor_ids[k]
 * (e.g. the totals kvz_encode_sizes reports for the pages about to be encoded there).
 * With exact sizes the bound equals the device cursor after the encode, so no
 * observation is needed, and a chunk is left only when the next pages do not fit it. */
int kvz_alloc_reserve_granules(kvz_alloc *a, const int32_t *cursor_ids, const uint64_t *granules, int32_t count,
                               int32_t *upd_idx, uint32_t *upd_pos, uint32_t *upd_end, int32_t *n_upd,
                               uint64_t *ticket);
/* Granules left in cursor c's current chunk by the allocator's bound (0 without a chunk). */
int kvz_alloc_room(const kvz_alloc *a, int32_t cursor_id, uint64_t *room);
/* cursors_snapshot: host copy of the device cursors [num_cursors][2] taken after the
 * encode that used reservation `ticket` completed. */
int kvz_alloc_observe(kvz_alloc *a, uint64_t ticket, const uint32_t *cursors_snapshot);
int kvz_alloc_release(kvz_alloc *a, int32_t cursor_id);
/* bytes in chunks held by cursors, bytes in free chunks, bytes known used (observed
 * cursor positions), chunks held, chunks free */
int kvz_alloc_stats(const kvz_alloc *a, uint64_t *held_bytes, uint64_t *free_bytes,
                    uint64_t *used_bytes_bound, int32_t *chunks_held, int32_t *chunks_free);

/* Copy n cursor updates (device arrays idx[n], pos[n], end[n]) into cursors. */
int kvz_apply_cursor_updates(const int32_t *idx, const uint32_t *pos, const uint32_t *end,
                             int32_t n, uint32_t *cursors, int32_t num_cursors,
                             kvz_stream_t stream);

/* kvz_selftest_bounded_wait -- diagnostic with no counterpart on the pages: runs, on the
 * device, the bounded barrier wait that every kernel here uses for its pipeline.  One wait
 * targets an already complete phase (must return at once); one targets a phase no thread
 * ever completes (must give up after limit_ns, OR KVZ_STATUS_TIMEOUT into *status and
 * return).  out: device uint64[3] = {ns of the first wait, ns of the second,
 * bit 0 = first wait succeeded, bit 1 = second wait succeeded}.  limit_ns in (0, 10 s]. */
int kvz_selftest_bounded_wait(uint64_t limit_ns, uint32_t *status, uint64_t *out, kvz_stream_t stream);

/* kvz_selftest_late_writer -- test helper with no counterpart on the pages: a kernel that
 * lets a programmatic dependent launch begin at once, waits delay_ns (<= 1 s) on the
 * device, then copies `bytes` (a multiple of 16, <= 1 GiB; 16-byte aligned device
 * pointers) from src to dst.  Launched right before an overlapped attention call, it
 * checks that the call reads q and the last pages only after the wait. */
int kvz_selftest_late_writer(const void *src, void *dst, uint64_t bytes, uint64_t delay_ns, kvz_stream_t stream);

/* Text for a KVZ_ERR_* code. */
const char *kvz_strerror(int code);
/* The last CUDA error seen by a failed call on this thread (a cudaError_t value). */
int kvz_last_cuda_error(void);
/* SM count of the current device, as used for the attention work split. */
int kvz_device_sm_count(void);

#ifdef __cplusplus
}
#endif
#endif
