// codec.cu -- page encoder (validation, block sizes, segmented placement scan over
// pages, pack) and standalone decoder for the 12-bit BF16 block format.
//
// Format (ZipFusion, "How it works" steps 1-4, layout and metadata paragraphs): a
// 16-token page slice of one KV head, K or V, is four 512-value blocks (dims
// [32j, 32j+32) x 16 tokens).  A block whose exponents all lie in [b, b+15], b the
// even floor of the minimum, keeps every value's low byte and a 4-bit (sign, d)
// code, d = (e-b)/2: 768 bytes.  Any other block stays raw: 1024 bytes.  Values are
// stored in the tensor-core fragment order of the block's role (K rows = tokens for
// QK^T, V rows = dims for PV), so the attention kernel restores each lane's eight
// operand elements from one 8-byte low run and one 4-byte code word.
#include "kvz_internal.h"
#include "stage.cuh"

namespace kvz {

__device__ __forceinline__ void exponent_range(const uint32_t (&w)[8], uint32_t &mn, uint32_t &mx)
{
    mn = 255;
    mx = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        uint32_t e0 = (w[k] >> 7) & 0xFFu, e1 = (w[k] >> 23) & 0xFFu;
        mn = min(mn, min(e0, e1));
        mx = max(mx, max(e0, e1));
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
}

// ---------------------------------------------------------------------------------
// launch 1: group sizes
// ---------------------------------------------------------------------------------
// Warp-per-item size pass: each warp takes whole (entry, head) items in a grid-stride
// loop, issues all sixteen 16-byte loads of the item's 8 KB at once (lane = row pair of a
// 16 x 32 slab per block) and reduces the eight blocks itself: no shared memory, no
// block-wide barrier, many slices in flight per SM.
__global__ void __launch_bounds__(256, 3) k_enc_sizes_w(EncodeParams P)
{
    if (P.ws_hdr[0] != 0) return;
    const int lane = threadIdx.x & 31;
    const int64_t items = (int64_t)P.n * P.hkv;
    const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t it = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items; it += stride) {
        const int entry = (int)(it / P.hkv), head = (int)(it % P.hkv);
        const uint16_t *slice = P.raw_pool + ((int64_t)P.src_page[entry] * P.hkv + head) * 2 * kPage * kDim;
        uint4 v[16];
#pragma unroll
        for (int b = 0; b < 8; ++b) {  // block (kv = b/4, j = b%4)
            const uint4 *p = reinterpret_cast<const uint4 *>(slice + (b >> 2) * kPage * kDim + (lane >> 1) * kDim +
                                                             32 * (b & 3) + 16 * (lane & 1));
            v[2 * b] = p[0];
            v[2 * b + 1] = p[1];
        }
        uint32_t g = 0, tags[2] = {0, 0};
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            uint32_t w[8] = {v[2 * b].x, v[2 * b].y, v[2 * b].z, v[2 * b].w,
                             v[2 * b + 1].x, v[2 * b + 1].y, v[2 * b + 1].z, v[2 * b + 1].w};
            uint32_t mn, mx;
            exponent_range(w, mn, mx);
            const uint32_t base = mn & ~1u;
            const bool ok = mx <= base + 15;
            g += ok ? 3u : 4u;
            tags[b >> 2] |= (ok ? (base >> 1) : 0xFFu) << (8 * (b & 3));
        }
        if (lane == 0) {
            P.ws_pair_size[it] = g;
            atomicAdd(P.ws_page_size + entry, g);  // integer sum: the same whatever the order
            if (P.ws_tags) P.ws_tags[it] = tags[0] | ((uint64_t)tags[1] << 32);  // for the pack pass
        }
    }
}

// Validation before anything is written (an index out of range or a decreasing dst_seq
// makes the whole call a no-op), and the per-call reset of the page-size sums: one block
// walks the entries, so the header word is stored whole and nothing has to be zeroed
// before the call (a memset node costs several microseconds inside a CUDA graph).
constexpr int kPrepThreads = 1024;

__global__ void __launch_bounds__(kPrepThreads) k_enc_prepare(EncodeParams P)
{
    __shared__ uint32_t s_err[kPrepThreads / 32];
    uint32_t err = 0;
    for (int e = threadIdx.x; e < P.n; e += kPrepThreads) {
        P.ws_page_size[e] = 0;
        // a size-only call (kvz_encode_sizes) has no destination sequences
        const int s = P.src_page[e], d = P.dst_page[e], q = P.dst_seq ? P.dst_seq[e] : 0;
        if (s < 0 || s >= P.num_raw_pages || d < 0 || d >= P.num_meta_pages || q < 0 || q >= P.num_cursors)
            err |= KVZ_STATUS_BAD_INDEX;
        if (P.dst_seq && e > 0 && q < P.dst_seq[e - 1]) err |= KVZ_STATUS_BAD_ORDER;
    }
    err = __reduce_or_sync(0xffffffffu, err);
    if ((threadIdx.x & 31) == 0) s_err[threadIdx.x >> 5] = err;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t all = 0;
        for (int w = 0; w < kPrepThreads / 32; ++w) all |= s_err[w];
        P.ws_hdr[0] = all;
        if (all) atomicOr(P.status, all);
    }
}

// ---------------------------------------------------------------------------------
// Placement: one CTA scans the pages [e0, e1) in call order -- a segmented exclusive
// scan of page sizes (per page, summed over heads by the size pass), segments = runs
// of equal dst_seq.  A segment's first page reads its cursor, its last page writes it
// back.
// ---------------------------------------------------------------------------------
constexpr int kScanThreads = 1024;
constexpr int kScanItems = 4;  // pages per thread per tile

__global__ void __launch_bounds__(kScanThreads) k_enc_scan(EncodeParams P, int e0, int e1)
{
    __shared__ uint32_t s_flag[kScanThreads / 32];
    __shared__ uint64_t s_sum[kScanThreads / 32];
    __shared__ uint32_t s_carry_flag;
    __shared__ uint64_t s_carry;
    if (P.ws_hdr[0] != 0) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_carry = 0;
        s_carry_flag = 0;
    }
    __syncthreads();
    for (int t0 = e0; t0 < e1; t0 += kScanThreads * kScanItems) {
        const int i0 = t0 + tid * kScanItems;
        uint64_t val[kScanItems];
        uint32_t head[kScanItems];
        uint32_t any_head = 0;
        uint64_t run = 0;
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            const int e = i0 + k;
            val[k] = 0;
            head[k] = 0;
            if (e < e1) {
                const int seq = P.dst_seq[e];
                const bool is_head = e == e0 || P.dst_seq[e - 1] != seq;
                uint64_t v = P.ws_page_size[e];
                if (is_head) v += P.cursors[2 * seq];  // absolute granule position
                head[k] = is_head;
                val[k] = v;
            }
            run = head[k] ? val[k] : run + val[k];  // inclusive segmented scan within the run
            any_head |= head[k];
            val[k] = run;
        }
        // warp-level inclusive segmented scan of (flag, run total)
        uint32_t f = any_head;
        uint64_t sm = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint64_t so = __shfl_up_sync(0xffffffffu, sm, off);
            const uint32_t fo = __shfl_up_sync(0xffffffffu, f, off);
            if (lane >= off) {
                if (!f) sm += so;
                f |= fo;
            }
        }
        if (lane == 31) {
            s_flag[warp] = f;
            s_sum[warp] = sm;
        }
        __syncthreads();
        if (warp == 0) {
            uint32_t wf = s_flag[lane];
            uint64_t ws = s_sum[lane];
            if (lane == 0) {  // fold in the carry from the previous tile
                if (!wf) ws += s_carry;
                wf |= s_carry_flag;
            }
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint64_t so = __shfl_up_sync(0xffffffffu, ws, off);
                const uint32_t fo = __shfl_up_sync(0xffffffffu, wf, off);
                if (lane >= off) {
                    if (!wf) ws += so;
                    wf |= fo;
                }
            }
            s_flag[lane] = wf;
            s_sum[lane] = ws;
        }
        __syncthreads();
        // exclusive prefix of this thread's run: inclusive of the previous lane, combined
        // with the previous warps' inclusive total
        const uint64_t prev_s = __shfl_up_sync(0xffffffffu, sm, 1);
        const uint32_t prev_f = __shfl_up_sync(0xffffffffu, f, 1);
        const uint64_t wpre_s = warp > 0 ? s_sum[warp - 1] : s_carry;
        const uint64_t excl = lane == 0 ? wpre_s : (prev_f ? prev_s : prev_s + wpre_s);
        bool seen_head = false;
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            const int e = i0 + k;
            if (e >= e1) break;
            seen_head |= head[k] != 0;
            const uint64_t incl = seen_head ? val[k] : val[k] + excl;
            const uint64_t pos = incl - P.ws_page_size[e];
            P.ws_page_base[e] = (uint32_t)(pos < 0xFFFFFFFFull ? pos : 0xFFFFFFFFull);
            const bool last = e == e1 - 1 || P.dst_seq[e + 1] != P.dst_seq[e];
            if (last) P.cursors[2 * P.dst_seq[e]] = (uint32_t)(incl < 0xFFFFFFFFull ? incl : 0xFFFFFFFFull);
        }
        __syncthreads();
        if (tid == kScanThreads - 1) {
            s_carry = s_sum[31];  // inclusive total of the whole tile (previous carry folded in)
            s_carry_flag = s_flag[31];
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------------
// packing of one staged (entry, head) slice: its K group at pair_base, its V group right
// after, each block eligible (768 B: low bytes + codes) or raw (1024 B), in storage order,
// and the two 8-byte group words; a group past its cursor's end is not written (offset
// KVZ_OFFSET_INVALID, KVZ_STATUS_ARENA_FULL).  One warp.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void pack_groups(const EncodeParams &P, const uint8_t *stage, int lane, uint32_t tagsK,
                                            uint32_t tagsV, uint64_t pair_base, int seq, int dst, int head)
{
    const uint32_t gK = group_granules(tagsK), gV = group_granules(tagsV);
    const uint64_t end = min((uint64_t)P.cursors[2 * seq + 1], P.arena_bytes / kGranule);
#pragma unroll 1
    for (int kv = 0; kv < 2; ++kv) {
        const uint64_t offset0 = pair_base + (kv ? gK : 0);
        const uint32_t group_tags = kv ? tagsV : tagsK;
        const bool fits = offset0 + (kv ? gV : gK) <= end;
        uint32_t before = 0;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
            const uint32_t tag = (group_tags >> (8 * j)) & 0xFFu;
            if (fits) {
                uint32_t w[8];
                gather_block(stage, kv, j, lane, w);
                uint8_t *blk = P.arena + (offset0 + before) * kGranule;
                if (tag != 0xFFu) {
                    const uint32_t b = tag << 1;
                    uint32_t low[4], code[2];
#pragma unroll
                    for (int f = 0; f < 2; ++f) {
                        uint32_t lo03 = 0, lo47 = 0, cw = 0;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint32_t x = (w[f * 4 + i / 2] >> (16 * (i & 1))) & 0xFFFFu;
                            const uint32_t sg = x >> 15, e = (x >> 7) & 0xFFu, d = (e - b) >> 1;
                            if (i < 4) {
                                lo03 |= (x & 0xFFu) << (8 * i);
                                cw |= ((sg << 7) | d) << (8 * i);
                            } else {
                                lo47 |= (x & 0xFFu) << (8 * (i - 4));
                                cw |= ((sg << 3) | (d << 4)) << (8 * (i - 4));
                            }
                        }
                        low[2 * f] = lo03;
                        low[2 * f + 1] = lo47;
                        code[f] = cw;
                    }
                    *reinterpret_cast<uint4 *>(blk + 16 * lane) = make_uint4(low[0], low[1], low[2], low[3]);
                    *reinterpret_cast<uint2 *>(blk + 512 + 8 * lane) = make_uint2(code[0], code[1]);
                } else {
                    *reinterpret_cast<uint4 *>(blk + 32 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4 *>(blk + 32 * lane + 16) = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
            before += tag_granules(tag);
        }
        if (lane == 0) {
            const uint64_t off_word = fits ? offset0 : (uint64_t)KVZ_OFFSET_INVALID;
            P.meta[((int64_t)dst * P.hkv + head) * 2 + kv] = off_word | ((uint64_t)group_tags << 32);
            if (!fits) atomicOr(P.status, KVZ_STATUS_ARENA_FULL);
        }
    }
}

// ---------------------------------------------------------------------------------
// launch 3: pack
// ---------------------------------------------------------------------------------
// Warp-per-item pack: each warp stages one (entry, head) slice in its own shared-memory
// buffer, computes the eight tags, places the K and V groups and writes them; items come
// in a grid-stride loop, so an SM keeps many slices in flight without block-wide barriers.
constexpr int kPackWarps = 8;

__global__ void __launch_bounds__(kPackWarps * 32, 2) k_enc_pack_w(EncodeParams P)
{
    extern __shared__ __align__(16) uint8_t pack_smem[];
    if (P.ws_hdr[0] != 0) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *stage = pack_smem + warp * (32 * kStagePitch);
    const int64_t items = (int64_t)P.n * P.hkv;
    const int64_t stride = (int64_t)gridDim.x * kPackWarps;
    for (int64_t it = (int64_t)blockIdx.x * kPackWarps + warp; it < items; it += stride) {
        const int entry = (int)(it / P.hkv), head = (int)(it % P.hkv);
        const int src = P.src_page[entry], dst = P.dst_page[entry], seq = P.dst_seq[entry];
        // the heads before this one in the page: one load per lane, then a warp sum
        const uint32_t ps = lane < head ? P.ws_pair_size[(int64_t)entry * P.hkv + lane] : 0u;
        const uint4 *s4 = reinterpret_cast<const uint4 *>(P.raw_pool + ((int64_t)src * P.hkv + head) * 2 * kPage * kDim);
        uint4 v[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = s4[lane + 32 * k];
        uint32_t before_heads = __reduce_add_sync(0xffffffffu, ps);
        for (int h = 32; h < head; ++h) before_heads += P.ws_pair_size[(int64_t)entry * P.hkv + h];
        __syncwarp();  // the previous item's gathers are done with the buffer
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int q = lane + 32 * k;  // 16-byte chunk q -> row q/16, byte (q%16)*16
            *reinterpret_cast<uint4 *>(stage + (q >> 4) * kStagePitch + (q & 15) * 16) = v[k];
        }
        __syncwarp();
        // one tag byte per block, as the size pass found them
        const uint64_t tags = P.ws_tags[it];
        pack_groups(P, stage, lane, (uint32_t)tags, (uint32_t)(tags >> 32),
                    (uint64_t)P.ws_page_base[entry] + before_heads, seq, dst, head);
    }
}

// ---------------------------------------------------------------------------------
// standalone decode: warp per (entry, head) item in a grid-stride loop.  The warp issues
// the loads of all eight blocks of the item (K and V groups) together, restores each
// lane's fragments with the same register restore the attention kernel uses, scatters
// them into its own staged page slice, and writes the 8 KB slice back in the plain page
// layout with 16-byte stores.  The next item's page id and group words are loaded while
// this one is restored, so only the block loads wait on memory.  Many items per SM stay in
// flight (a CTA per item with a warp per block kept too few in flight to cover the three
// dependent loads of page id, group words and blocks).
// ---------------------------------------------------------------------------------
constexpr int kDecWarps = 8;
constexpr int kDecCtasPerSm = 2;  // registers for both groups' loads in flight at once

// Group words of (page, head); bad |= KVZ_STATUS_BAD_INDEX (words 0) for a page out of range.
__device__ __forceinline__ void dec_words(const DecodeParams &P, int page, int head, uint64_t (&w)[2], uint32_t &bad)
{
    w[0] = w[1] = 0;
    bad = 0;
    if (page < 0 || page >= P.num_meta_pages) {
        bad = KVZ_STATUS_BAD_INDEX;
    } else {
        const uint64_t *m = P.meta + ((int64_t)page * P.hkv + head) * 2;
        w[0] = m[0];
        w[1] = m[1];
    }
}

__global__ void __launch_bounds__(kDecWarps * 32, kDecCtasPerSm) k_decode_w(DecodeParams P)
{
    extern __shared__ __align__(16) uint8_t dec_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *stage = dec_smem + warp * (32 * kStagePitch);
    const int64_t items = (int64_t)P.n * P.hkv;
    const int64_t stride = (int64_t)gridDim.x * kDecWarps;
    int64_t it = (int64_t)blockIdx.x * kDecWarps + warp;
    // this item's group words, and the next item's page id, loaded an iteration ahead
    uint64_t words[2] = {0, 0};
    uint32_t bad_idx = 0;
    int page_next = 0;
    if (it < items) dec_words(P, P.page[it / P.hkv], (int)(it % P.hkv), words, bad_idx);
    if (it + stride < items) page_next = P.page[(it + stride) / P.hkv];
    for (; it < items; it += stride) {
        const int entry = (int)(it / P.hkv), head = (int)(it % P.hkv);
        // both groups' blocks: every load first (a bad K word leaves the V group usable)
        uint32_t bad = bad_idx, tags[2] = {0, 0}, use[2] = {0, 0};
        uint4 x[2][4], y[2][4];
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
            const uint32_t offset0 = (uint32_t)words[kv];
            tags[kv] = (uint32_t)(words[kv] >> 32);
            use[kv] = !(bad_idx & KVZ_STATUS_BAD_INDEX);
            if (use[kv] && (!tags_valid(tags[kv]) || offset0 == KVZ_OFFSET_INVALID ||
                            ((uint64_t)offset0 + group_granules(tags[kv])) * kGranule > P.arena_bytes)) {
                bad |= KVZ_STATUS_BAD_META;
                use[kv] = 0;
            }
            uint32_t before = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t tag = (tags[kv] >> (8 * j)) & 0xFFu;
                x[kv][j] = make_uint4(0, 0, 0, 0);
                y[kv][j] = make_uint4(0, 0, 0, 0);
                if (use[kv]) {
                    const uint8_t *blk = P.arena + ((uint64_t)offset0 + before) * kGranule;
                    if (tag == 0xFFu) {
                        x[kv][j] = __ldg(reinterpret_cast<const uint4 *>(blk + 32 * lane));
                        y[kv][j] = __ldg(reinterpret_cast<const uint4 *>(blk + 32 * lane + 16));
                    } else {
                        x[kv][j] = __ldg(reinterpret_cast<const uint4 *>(blk + 16 * lane));
                        const uint2 code = __ldg(reinterpret_cast<const uint2 *>(blk + 512 + 8 * lane));
                        y[kv][j].x = code.x;
                        y[kv][j].y = code.y;
                    }
                }
                before += tag_granules(tag);
            }
        }
        // the next item's group words and the page id of the one after it
        {
            const int64_t nx = it + stride;
            if (nx < items) dec_words(P, page_next, (int)(nx % P.hkv), words, bad_idx);
            if (nx + stride < items) page_next = P.page[(nx + stride) / P.hkv];
        }
        __syncwarp();  // the previous item's stores are done with the buffer
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t tag = (tags[kv] >> (8 * j)) & 0xFFu;
                uint32_t w[8];
                if (!use[kv] || tag == 0xFFu) {
                    w[0] = x[kv][j].x; w[1] = x[kv][j].y; w[2] = x[kv][j].z; w[3] = x[kv][j].w;
                    w[4] = y[kv][j].x; w[5] = y[kv][j].y; w[6] = y[kv][j].z; w[7] = y[kv][j].w;
                } else {
                    const uint32_t bb = tag * 0x01010101u;
                    uint32_t f0[4], f1[4];
                    restore_fragment(x[kv][j].x, x[kv][j].y, y[kv][j].x, bb, f0);
                    restore_fragment(x[kv][j].z, x[kv][j].w, y[kv][j].y, bb, f1);
                    w[0] = f0[0]; w[1] = f0[1]; w[2] = f0[2]; w[3] = f0[3];
                    w[4] = f1[0]; w[5] = f1[1]; w[6] = f1[2]; w[7] = f1[3];
                }
                // scatter to the staged slice (inverse of gather_block)
#pragma unroll
                for (int f = 0; f < 2; ++f)
#pragma unroll
                    for (int i = 0; i < 8; i += 2) {
                        const int r = frag_row(lane, i), c = frag_col(lane, i);
                        const int dim0 = 32 * j + 16 * f;
                        const uint32_t v = w[f * 4 + i / 2];
                        if (kv == 0) {
                            *reinterpret_cast<uint32_t *>(stage + r * kStagePitch + (dim0 + c) * 2) = v;
                        } else {
                            uint8_t *base = stage + (16 + c) * kStagePitch + (dim0 + r) * 2;
                            *reinterpret_cast<uint16_t *>(base) = (uint16_t)(v & 0xFFFFu);
                            *reinterpret_cast<uint16_t *>(base + kStagePitch) = (uint16_t)(v >> 16);
                        }
                    }
            }
        }
        if (bad && lane == 0) atomicOr(P.status, bad);
        __syncwarp();
        uint4 *out = reinterpret_cast<uint4 *>(P.out + ((int64_t)entry * P.hkv + head) * 2 * kPage * kDim);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int q = lane + 32 * k;  // 16-byte chunk q -> row q/16, byte (q%16)*16
            out[q] = *reinterpret_cast<const uint4 *>(stage + (q >> 4) * kStagePitch + (q & 15) * 16);
        }
    }
}

__global__ void k_apply_cursor_updates(const int32_t *idx, const uint32_t *pos, const uint32_t *end, int n,
                                       uint32_t *cursors, int num_cursors)
{
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k < n) {
        const int c = idx[k];
        if (c >= 0 && c < num_cursors) {
            cursors[2 * c] = pos[k];
            cursors[2 * c + 1] = end[k];
        }
    }
}

// ---------------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------------
constexpr int kPackSmem = kPackWarps * 32 * kStagePitch;  // 68 KB: one slice buffer per warp
constexpr int kDecSmem = kDecWarps * 32 * kStagePitch;    // the same for the decoder

// SM count of the current device, and the pack kernel's shared-memory opt-in (once per
// device and process)
static cudaError_t encode_grid(int *sms)
{
    static unsigned long long done = 0;  // bit per device ordinal < 64
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess && !(dev < 64 && ((__atomic_load_n(&done, __ATOMIC_ACQUIRE) >> dev) & 1ull))) {
        e = cudaFuncSetAttribute(k_enc_pack_w, cudaFuncAttributeMaxDynamicSharedMemorySize, kPackSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_decode_w, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmem);
        if (e == cudaSuccess && dev < 64) __atomic_fetch_or(&done, 1ull << dev, __ATOMIC_ACQ_REL);
    }
    return e;
}

// one wave of `per_sm` CTAs per SM, fewer when there are fewer items than warps
static unsigned grid_for(size_t items, int sms, int per_sm)
{
    const size_t want = (items + 7) / 8;
    const size_t wave = (size_t)(sms > 0 ? sms : 1) * per_sm;
    return (unsigned)(want < wave ? (want > 0 ? want : 1) : wave);
}

cudaError_t launch_encode(const EncodeParams &P, cudaStream_t stream)
{
    k_enc_prepare<<<1, kPrepThreads, 0, stream>>>(P);
    const size_t items = (size_t)P.n * P.hkv;
    int sms = 0;
    cudaError_t e = encode_grid(&sms);
    if (e != cudaSuccess) return e;
    k_enc_sizes_w<<<grid_for(items, sms, 3), 256, 0, stream>>>(P);
    k_enc_scan<<<1, kScanThreads, 0, stream>>>(P, 0, P.n);
    k_enc_pack_w<<<grid_for(items, sms, 2), kPackWarps * 32, kPackSmem, stream>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_encode_sizes(const EncodeParams &P, cudaStream_t stream)
{
    // validation, then the size pass alone: P.ws_page_size is the caller's output array
    k_enc_prepare<<<1, kPrepThreads, 0, stream>>>(P);
    int sms = 0;
    cudaError_t e = encode_grid(&sms);
    if (e != cudaSuccess) return e;
    k_enc_sizes_w<<<grid_for((size_t)P.n * P.hkv, sms, 3), 256, 0, stream>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_enc_prepare(const EncodeParams &P, cudaStream_t stream)
{
    k_enc_prepare<<<1, kPrepThreads, 0, stream>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_enc_scan(const EncodeParams &P, cudaStream_t stream)
{
    k_enc_scan<<<1, kScanThreads, 0, stream>>>(P, 0, P.n);
    return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams &P, cudaStream_t stream)
{
    int sms = 0;
    cudaError_t e = encode_grid(&sms);
    if (e != cudaSuccess) return e;
    k_decode_w<<<grid_for((size_t)P.n * P.hkv, sms, kDecCtasPerSm), kDecWarps * 32, kDecSmem, stream>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_apply_cursor_updates(const int32_t *idx, const uint32_t *pos, const uint32_t *end, int n,
                                        uint32_t *cursors, int num_cursors, cudaStream_t stream)
{
    if (n <= 0) return cudaSuccess;
    k_apply_cursor_updates<<<(n + 255) / 256, 256, 0, stream>>>(idx, pos, end, n, cursors, num_cursors);
    return cudaGetLastError();
}

}  // namespace kvz
