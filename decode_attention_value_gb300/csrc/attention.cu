// attention.cu -- split-KV GQA paged decode attention over compressed pages plus a raw
// BF16 tail (12-bit block groups, kFmt = kFmtZf; group-adaptive tiles, kFmt = kFmtGa;
// FP8 tiles, kFmt = kFmtF8E4 / kFmtF8E5), and the same kernel over plain BF16 pages
// (kFmt = kFmtRaw, the in-run uncompressed baseline).  kG8 selects the instantiation for
// 5..8 query heads per KV head.
//
// GAAC ("Attention with On-the-Fly Decompression"): the kernel reads compressed tiles
// and their metadata, rebuilds BF16 only in registers, and compressed blocks and the
// raw tail share one softmax.  ZipFusion ("How it works"): the restored values feed
// the tensor cores for QK^T and PV.
//
// GB300 design:
//  * one wave of C = SMs x k CTAs; the (sequence, KV head, page) list is flattened and
//    cut into C equal page ranges (the split depends only on shapes and seq_lens);
//  * per CTA one producer warp and four consumer warps; the producer resolves page
//    ids and metadata 32-64 pages ahead and streams each page into an 8-stage shared
//    memory ring with TMA: two 1-D bulk copies (the K and V groups, 3-4 KB each) for a
//    compressed page, two 2-D tensor copies with 128-byte swizzle for a raw page.
//    One lane per stage issues at once, each as soon as its stage is free, so no
//    serial per-page chain of one thread paces the stream;
//  * each consumer warp takes whole pages: per 512-value block one 16-byte and one
//    8-byte shared load per lane, an integer restore into bf16x2 fragments, and
//    mma.sync m16n8k16 with K (QK^T, tokens x dims) and V^T (PV, dims x tokens) as the
//    A operand and the G query heads in the N columns (Q read from global memory once
//    per segment, as the B fragments).  G <= 4 leaves four spare N
//    columns: Q is duplicated there for QK^T, and for PV they carry the low part of
//    P = hi + lo (both bf16), so the PV product keeps ~16 bits of P for free.  FP8 tiles
//    multiply in f16 (their values widen to f16 exactly) and the tile formats read their
//    per-channel exponent bases from a shared-memory table built once per segment;
//  * warps merge their online-softmax states per (sequence, KV head) segment, and a
//    small follow-up kernel merges the segments in a fixed order.
#include <cuda.h>

#include <cstring>

#include "f8.cuh"
#include "ga.cuh"
#include "kvz_internal.h"

namespace kvz {

constexpr int kStages = 8;
constexpr int kStageBytes = 8192;
constexpr int kConsumers = 4;
constexpr int kThreads = (kConsumers + 1) * 32;
static_assert(kStages % kConsumers == 0, "a stage's consecutive fills must go to the same consumer warp");

enum : uint32_t { kKindPair = 0, kKindRaw = 1, kKindSkip = 2 };

struct __align__(16) StageInfo {
    uint32_t kind, valid, tagsK, tagsV;
};

// dynamic shared memory layout (offsets from a 1024-aligned base)
struct Smem {
    static constexpr int stage = 0;
    static constexpr int full = stage + kStages * kStageBytes;
    static constexpr int empty = full + kStages * 8;
    static constexpr int info = empty + kStages * 8;
    static constexpr int mm = info + kStages * 16;
    static constexpr int ml = mm + kConsumers * 8 * 4;  // per warp: (max, sum) of up to 8 heads
    static constexpr int mo = ml + kConsumers * 8 * 4;
    static constexpr int pref = mo + kConsumers * 4 * 128 * 4;
    __host__ __device__ static int tail(int batch) { return pref + (batch + 1) * 4; }
    // tile formats: the segment's KV-head base table (256 words)
    __host__ __device__ static int bases(int batch) { return (tail(batch) + batch + 15) & ~15; }
    __host__ __device__ static int bytes(int batch, bool tiles) { return bases(batch) + (tiles ? 1024 : 0); }
};

__device__ __forceinline__ uint32_t swz128(int row, int col)
{
    // byte offset of element (row, col) of a [32][128] BF16 tile loaded as two
    // 64-column boxes with the 128-byte swizzle (16-byte chunk index ^= row % 8)
    return (uint32_t)((col >> 6) * 4096 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) + (col & 7) * 2);
}

struct PageLoc {
    int b, kvh, p;
};

// Largest b in [0, batch) with hkv * pref[b] <= x, then the KV head and page.
__device__ __forceinline__ PageLoc locate(const int32_t *pref, int batch, int hkv, int64_t x)
{
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)hkv * pref[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    const int n = pref[lo + 1] - pref[lo];
    const int64_t r = x - (int64_t)hkv * pref[lo];
    PageLoc L;
    L.b = lo;
    L.kvh = (int)(r / n);
    L.p = (int)(r - (int64_t)L.kvh * n);
    return L;
}

__device__ __forceinline__ int64_t unit_end(const int32_t *pref, int hkv, const PageLoc &L)
{
    const int n = pref[L.b + 1] - pref[L.b];
    return (int64_t)hkv * pref[L.b] + (int64_t)(L.kvh + 1) * n;
}

// ---------------------------------------------------------------------------------
// consumer-side fragment loads
// ---------------------------------------------------------------------------------
// One 512-value block of a compressed group in shared memory -> the two A fragments.
__device__ __forceinline__ void block_frags(const uint8_t *blk, uint32_t tag, int lane, uint32_t (&a0)[4],
                                            uint32_t (&a1)[4])
{
    if (tag == 0xFFu) {
        const uint4 x = *reinterpret_cast<const uint4 *>(blk + 32 * lane);
        const uint4 y = *reinterpret_cast<const uint4 *>(blk + 32 * lane + 16);
        a0[0] = x.x; a0[1] = x.y; a0[2] = x.z; a0[3] = x.w;
        a1[0] = y.x; a1[1] = y.y; a1[2] = y.z; a1[3] = y.w;
    } else {
        const uint4 low = *reinterpret_cast<const uint4 *>(blk + 16 * lane);
        const uint2 code = *reinterpret_cast<const uint2 *>(blk + 512 + 8 * lane);
        const uint32_t bb = tag * 0x01010101u;
        restore_fragment(low.x, low.y, code.x, bb, a0);
        restore_fragment(low.z, low.w, code.y, bb, a1);
    }
}

// K operand (tokens x 16 dims) of k-tile (j, f) from a swizzled raw page.
__device__ __forceinline__ void raw_k_frag(uint32_t st, int j, int f, int lane, uint32_t (&a)[4])
{
    const int mi = lane >> 3, rr = lane & 7;
    const int tok = rr + 8 * (mi & 1), col = 32 * j + 16 * f + 8 * (mi >> 1);
    ldmatrix_x4(st + swz128(tok, col), a);
}

// V^T operand (16 dims x tokens) of tile (j, f) from a swizzled raw page.
__device__ __forceinline__ void raw_v_frag(uint32_t st, int j, int f, int lane, uint32_t (&a)[4])
{
    const int mi = lane >> 3, rr = lane & 7;
    const int tok = rr + 8 * (mi >> 1), col = 32 * j + 16 * f + 8 * (mi & 1);
    ldmatrix_x4_trans(st + swz128(16 + tok, col), a);
}

// Zero the V^T operand halves of tokens >= valid (a partial tail page may hold stale
// values beyond its last token; P is 0 there but 0 * NaN is not 0).
__device__ __forceinline__ void mask_v_frag(uint32_t (&a)[4], int lane, int valid)
{
    const int t = lane & 3;
    const int t0 = 2 * t, t1 = 2 * t + 1, t8 = 2 * t + 8, t9 = 2 * t + 9;
    const uint32_t mlo = (t0 < valid ? 0x0000FFFFu : 0u) | (t1 < valid ? 0xFFFF0000u : 0u);
    const uint32_t mhi = (t8 < valid ? 0x0000FFFFu : 0u) | (t9 < valid ? 0xFFFF0000u : 0u);
    a[0] &= mlo;
    a[1] &= mlo;
    a[2] &= mhi;
    a[3] &= mhi;
}

// ---------------------------------------------------------------------------------
// FMA consumer: a build-time alternative (-DKVZ_CONSUMER_FMA=1) to the tensor-core
// QK^T and PV of the 12-bit and raw pages for G <= 4, kept to measure the choice.  It
// takes the same A fragments (the storage order of the blocks), so the compressed and
// raw kernels stay bit-identical to each other in that build.
// ---------------------------------------------------------------------------------
#ifndef KVZ_CONSUMER_FMA
#define KVZ_CONSUMER_FMA 0
#endif

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Scores of tile kt (16 dims): s[head][token g | g+8] += the lane's dims {2t, 2t+1, 2t+8,
// 2t+9} of the K fragment times the four heads' queries, read from the table
// qs[kt][t][slot][head] (fp32).
__device__ __forceinline__ void fma_qk_tile(float (&s)[4][2], const uint32_t (&a)[4], const float *qs, int kt, int t)
{
    const float4 *qv = reinterpret_cast<const float4 *>(qs + (kt * 4 + t) * 16);
    const float4 v0 = qv[0], v1 = qv[1], v2 = qv[2], v3 = qv[3];
    const float q[4][4] = {{v0.x, v0.y, v0.z, v0.w}, {v1.x, v1.y, v1.z, v1.w}, {v2.x, v2.y, v2.z, v2.w},
                           {v3.x, v3.y, v3.z, v3.w}};
    const float k0[4] = {bf_lo(a[0]), bf_hi(a[0]), bf_lo(a[2]), bf_hi(a[2])};  // token g, slots 0..3
    const float k1[4] = {bf_lo(a[1]), bf_hi(a[1]), bf_lo(a[3]), bf_hi(a[3])};  // token g + 8
#pragma unroll
    for (int h = 0; h < 4; ++h)
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
            s[h][0] = fmaf(k0[sl], q[sl][h], s[h][0]);
            s[h][1] = fmaf(k1[sl], q[sl][h], s[h][1]);
        }
}

// o[head][dim g | g+8] += the V^T fragment (dims g, g+8 x tokens 2t, 2t+1, 2t+8, 2t+9)
// times p[token slot][head].
__device__ __forceinline__ void fma_pv_tile(float (&o)[4][2], const uint32_t (&a)[4], const float (&p)[4][4])
{
    const float v0[4] = {bf_lo(a[0]), bf_hi(a[0]), bf_lo(a[2]), bf_hi(a[2])};  // dim g
    const float v1[4] = {bf_lo(a[1]), bf_hi(a[1]), bf_lo(a[3]), bf_hi(a[3])};  // dim g + 8
#pragma unroll
    for (int h = 0; h < 4; ++h)
#pragma unroll
        for (int ts = 0; ts < 4; ++ts) {
            o[h][0] = fmaf(v0[ts], p[ts][h], o[h][0]);
            o[h][1] = fmaf(v1[ts], p[ts][h], o[h][1]);
        }
}

// ---------------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------------
template <int kFmt, bool kG8>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) k_attn(const AttnParams P, const __grid_constant__ CUtensorMap tmap)
{
    constexpr bool kCompressed = kFmt != kFmtRaw;
    constexpr bool kGa = kFmt == kFmtGa;
    constexpr bool kF8 = kFmt == kFmtF8E4 || kFmt == kFmtF8E5;
    constexpr bool kE5 = kFmt == kFmtF8E5;
    constexpr bool kTiles = kGa || kF8;  // 4-byte tile entries (K, V) per (page, head)
    constexpr bool kFma = KVZ_CONSUMER_FMA != 0 && !kG8 && (kFmt == kFmtZf || kFmt == kFmtRaw);
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_addr(smem);
    if (sbase & 1023u) {  // the swizzled TMA destinations need 1024-byte alignment
        if (threadIdx.x == 0) atomicOr(P.status, KVZ_STATUS_BAD_INDEX);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int32_t *pref = reinterpret_cast<int32_t *>(smem + Smem::pref);
    uint8_t *tail_len = smem + Smem::tail(P.batch);  // tokens in each sequence's last page if partial, else 0
    StageInfo *info = reinterpret_cast<StageInfo *>(smem + Smem::info);
    const int B = P.batch, hkv = P.hkv, G = P.G;
    constexpr bool G8 = kG8;  // G = 5..8: every MMA column is a head (zero for heads >= G), no spare columns
    // overlapped launch: the merge kernel may be scheduled now (it waits for this grid)
    if (P.overlap) pdl_launch_dependents();

    // ---- barriers, and the per-sequence page-count prefix ----
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(sbase + Smem::full + 8 * s, 1);
            mbar_init(sbase + Smem::empty + 8 * s, 1);
        }
        fence_barrier_init();
    }
    if (warp == 0) {
        const int chunk = (B + 31) / 32;
        const int b0 = min(B, lane * chunk), b1 = min(B, b0 + chunk);
        int s = 0;
        uint32_t bad_len = 0;
        const uint64_t keep = l2_evict_last();
        for (int b = b0; b < b1; ++b) {
            const int L = ld_keep_s32(P.seq_lens + b, keep);
            bad_len |= L < 0;
            s += L > 0 ? (L + kPage - 1) / kPage : 0;
        }
        if (bad_len) atomicOr(P.status, KVZ_STATUS_BAD_INDEX);
        int incl = s;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        int run = incl - s;
        for (int b = b0; b < b1; ++b) {
            pref[b] = run;
            const int L = ld_keep_s32(P.seq_lens + b, keep);
            run += L > 0 ? (L + kPage - 1) / kPage : 0;
            tail_len[b] = (uint8_t)(L > 0 ? L % kPage : 0);
        }
        if (lane == 31) pref[B] = incl;
    }
    __syncthreads();

    const int64_t T = (int64_t)hkv * pref[B];
    const int64_t C = gridDim.x, c = blockIdx.x;
    const int64_t lo = (c * T + C - 1) / C, hi = ((c + 1) * T + C - 1) / C;

    if (warp == kConsumers) {
        // =============================== producer ===============================
        // Page ids and metadata are fetched for 32 pages at a time, one page per lane,
        // a batch ahead of use (warp-wide loads, so no lane waits on another's load).
        // Each lane derives its page's stage descriptor; then in four rounds eight lanes
        // (one per stage) wait for their stages and issue their pages' copies.
        prefetch_tensormap(&tmap);
        const int64_t npage = hi - lo;
        // the KV stream is read once per step; the tables each step starts from stay in L2
        const uint64_t keep = l2_evict_last(), stream_once = l2_evict_first();
        struct Pre {
            PageLoc L;
            int32_t pid, n, tl;  // page id, pages in the sequence, tail tokens (0 = none)
        };
        // locate + page id: the table entry and the tail id do not wait on each other
        auto prep = [&](int64_t x, Pre &r) {
            r.pid = INT32_MIN;
            r.n = 0;
            r.tl = 0;
            r.L = PageLoc{0, 0, 0};
            if (x >= hi) return;
            r.L = locate(pref, B, hkv, x);
            r.n = pref[r.L.b + 1] - pref[r.L.b];
            r.tl = tail_len[r.L.b];
            const bool last_partial = (r.L.p == r.n - 1) && r.tl != 0;
            const int32_t tab =
                r.L.p < P.max_pages ? ld_keep_s32(P.page_ids + (int64_t)r.L.b * P.max_pages + r.L.p, keep) : INT32_MIN;
            if (kCompressed && last_partial) r.pid = ld_keep_s32(P.tail_page + r.L.b, keep);
            else r.pid = tab;
        };
        auto is_compressed = [&](const Pre &r) { return kCompressed && !((r.L.p == r.n - 1) && r.tl != 0); };
        auto load_meta = [&](const Pre &r, uint64_t &m0, uint64_t &m1) {  // metadata (global load)
            m0 = m1 = 0;
            if (is_compressed(r) && r.pid >= 0 && r.pid < P.num_meta_pages) {
                if (kTiles)  // the K and V tile entries
                    m0 = ld_keep_u64(reinterpret_cast<const uint64_t *>(P.meta32 + ((int64_t)r.pid * hkv + r.L.kvh) * 2),
                                     keep);
                else
                    ld_keep_u64x2(P.meta + ((int64_t)r.pid * hkv + r.L.kvh) * 2, keep, m0, m1);
            }
        };
        Pre cur, nxt;
        uint64_t cm0 = 0, cm1 = 0;
        prep(lo + lane, cur);
        prep(lo + 32 + lane, nxt);
        load_meta(cur, cm0, cm1);

        bool ok = true;
        static_assert(kStages <= 32, "a round is kStages lanes, one per stage");
        for (int64_t base = 0; base < npage; base += 32) {
            // ---- this lane's page descriptor: kind | valid << 8 | status << 16, source, sizes, tags ----
            uint32_t d_kind = kKindSkip, d_valid = 0, d_bad = 0, d_tK = 0, d_tV = 0, d_bytes = 0;
            uint64_t d_srcK = 0, d_srcV = 0;
            bool d_last = false;  // a raw copy of the sequence's last page (the page the step's token went to)
            if (base + lane < npage) {
                if (kTiles && is_compressed(cur)) {
                    const uint32_t eK = (uint32_t)cm0, eV = (uint32_t)(cm0 >> 32);
                    const uint64_t oK = eK & kGaOffsetMask, oV = eV & kGaOffsetMask;
                    const uint32_t bK = kGa ? ga_entry_bytes(eK) : f8_entry_bytes(kE5 ? kF8E5M2 : kF8E4M3, eK);
                    const uint32_t bV = kGa ? ga_entry_bytes(eV) : f8_entry_bytes(kE5 ? kF8E5M2 : kF8E4M3, eV);
                    if (cur.pid < 0 || cur.pid >= P.num_meta_pages) {
                        d_bad = KVZ_STATUS_BAD_INDEX;
                    } else if (eK == kGaEntryInvalid || eV == kGaEntryInvalid ||
                               oK * kGaGranule + bK > P.arena_bytes || oV * kGaGranule + bV > P.arena_bytes) {
                        d_bad = KVZ_STATUS_BAD_META;
                    } else {
                        d_kind = kKindPair;
                        d_valid = kPage;
                        d_tK = eK >> 31;  // 1: raw tile
                        d_tV = eV >> 31;
                        d_srcK = oK * kGaGranule;
                        d_srcV = oV * kGaGranule;
                        d_bytes = bK | (bV << 16);
                    }
                } else if (is_compressed(cur)) {
                    const uint32_t offK = (uint32_t)cm0, offV = (uint32_t)cm1;
                    const uint32_t tK = (uint32_t)(cm0 >> 32), tV = (uint32_t)(cm1 >> 32);
                    if (cur.pid < 0 || cur.pid >= P.num_meta_pages) {
                        d_bad = KVZ_STATUS_BAD_INDEX;
                    } else if (!tags_valid(tK) || !tags_valid(tV) || offK == KVZ_OFFSET_INVALID ||
                               offV == KVZ_OFFSET_INVALID ||
                               ((uint64_t)offK + group_granules(tK)) * kGranule > P.arena_bytes ||
                               ((uint64_t)offV + group_granules(tV)) * kGranule > P.arena_bytes) {
                        d_bad = KVZ_STATUS_BAD_META;
                    } else {
                        d_kind = kKindPair;
                        d_valid = kPage;
                        d_tK = tK;
                        d_tV = tV;
                        d_srcK = (uint64_t)offK * kGranule;
                        d_srcV = (uint64_t)offV * kGranule;
                        d_bytes = (group_granules(tK) * kGranule) | ((group_granules(tV) * kGranule) << 16);
                    }
                } else {
                    if (cur.pid < 0 || cur.pid >= P.num_raw_pages) {
                        d_bad = (kCompressed && cur.pid == -1) ? KVZ_STATUS_BAD_TAIL : KVZ_STATUS_BAD_INDEX;
                    } else {
                        d_kind = kKindRaw;
                        d_last = cur.L.p == cur.n - 1;
                        d_valid = (cur.L.p == cur.n - 1 && cur.tl != 0) ? (uint32_t)cur.tl : (uint32_t)kPage;
                        d_srcK = (uint64_t)(((int64_t)cur.pid * hkv + cur.L.kvh) * 32);  // tensor row
                    }
                }
                if (d_bad) atomicOr(P.status, d_bad);
            }
            // ---- next batches: metadata of batch +1 (its page ids arrived a batch ago), ids of batch +2 ----
            uint64_t nm0 = 0, nm1 = 0;
            load_meta(nxt, nm0, nm1);
            Pre nn;
            prep(lo + base + 64 + lane, nn);

            // lane L's page base + L goes to stage (base + L) % kStages; round r is lanes
            // [r kStages, (r + 1) kStages): the previous fill of each of their stages was issued
            // by round r - 1 or by the previous batch (base is a multiple of 32)
            const int cnt = (int)(npage - base < 32 ? npage - base : 32);
            const int s = (int)((base + lane) % kStages);
            const uint32_t parity = (uint32_t)((((base + lane) / kStages) & 1) ^ 1);
            const uint32_t emptybar = sbase + Smem::empty + 8 * s, fullbar = sbase + Smem::full + 8 * s;
            for (int r = 0; kStages * r < cnt && ok; ++r) {
                bool pending = lane / kStages == r && lane < cnt, mine_ok = true;
                uint32_t it = 0;
                uint64_t t0 = 0;
                while (__any_sync(0xffffffffu, pending)) {
                    if (!pending) continue;
                    if (mbar_test_wait(emptybar, parity)) {
                        pending = false;
                        // overlapped launch: the kernel before this one may still be writing the
                        // sequence's last page; everything else was complete before it started
                        if (P.overlap && d_last) pdl_wait_primary();
                        info[s] = StageInfo{d_kind, d_valid, d_tK, d_tV};
                        const uint32_t dst = sbase + Smem::stage + s * kStageBytes;
                        if (d_kind == kKindPair) {
                            const uint32_t bK = d_bytes & 0xFFFFu, bV = d_bytes >> 16;
                            mbar_arrive_expect_tx(fullbar, bK + bV);
                            if (!kTiles && d_srcV == d_srcK + bK) {
                                // 12-bit groups: V right after K in the stage; one copy when the
                                // encoder placed them next to each other (pages encoded together)
                                bulk_copy_g2s_hint(dst, P.arena + d_srcK, bK + bV, fullbar, stream_once);
                            } else {
                                bulk_copy_g2s_hint(dst, P.arena + d_srcK, bK, fullbar, stream_once);
                                bulk_copy_g2s_hint(dst + (kTiles ? 4096u : bK), P.arena + d_srcV, bV, fullbar,
                                                   stream_once);
                            }
                        } else if (d_kind == kKindRaw) {
                            mbar_arrive_expect_tx(fullbar, kStageBytes);
                            tensor_copy_2d_g2s_hint(dst, &tmap, 0, (int32_t)d_srcK, fullbar, stream_once);
                            tensor_copy_2d_g2s_hint(dst + 4096, &tmap, 64, (int32_t)d_srcK, fullbar, stream_once);
                        } else {
                            mbar_arrive(fullbar);
                        }
                    } else if ((++it & 255u) == 0) {  // bounded: give up after kWaitLimitNs
                        const uint64_t now = globaltimer_ns();
                        if (t0 == 0) {
                            t0 = now;
                        } else if (now - t0 > kWaitLimitNs) {
                            atomicOr(P.status, KVZ_STATUS_TIMEOUT);
                            pending = mine_ok = false;
                        }
                    }
                }
                ok = __all_sync(0xffffffffu, mine_ok);
            }
            cur = nxt;
            cm0 = nm0;
            cm1 = nm1;
            nxt = nn;
        }
        // never leave with copies in flight: wait for the last fill of every stage
        if (lane == 0) {
            for (int s = 0; s < kStages && s < npage; ++s) {
                const int64_t last = (npage - 1 - s) / kStages;
                mbar_wait(sbase + Smem::full + 8 * s, (uint32_t)(last & 1), P.status);
            }
        }
        return;
    }

    // =============================== consumers ===============================
    const int g = lane >> 2, t = lane & 3;
    const float NEG_INF = -INFINITY;
    float *mm = reinterpret_cast<float *>(smem + Smem::mm);
    float *mlv = reinterpret_cast<float *>(smem + Smem::ml);
    float *mo = reinterpret_cast<float *>(smem + Smem::mo);
    bool ok = true;
    // overlapped launch: q, the workspace and the outputs belong to the kernel before this
    // one until it has finished
    if (P.overlap) pdl_wait_primary();
    int64_t x = lo, ibase = 0;
    while (x < hi) {
        const PageLoc L = locate(pref, B, hkv, x);
        const int64_t send = min(hi, unit_end(pref, hkv, L));
        const int64_t cnt = send - x;
        // tile formats: this KV head's base vectors as a shared-memory table (the previous
        // segment's readers have passed its closing barrier)
        uint32_t *btbl = reinterpret_cast<uint32_t *>(smem + Smem::bases(B));
        if constexpr (kTiles) {
            ga_fill_bases_table(P.ga_bases + (size_t)L.kvh * 512, btbl, tid, kFmt == kFmtF8E4);
            asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
        }

        // queries of this segment: B operand of QK^T, read from global memory.  G <= 4:
        // column n = head n % 4 (zero if >= G); G = 5..8: column n = head n (zero if >= G).
        // FP8 pages multiply in f16 (every FP8 value is an f16 value, so the K and V
        // operands need no further widening): Q is converted once per segment and reloaded
        // in BF16 for a raw BF16 tail page.
        uint32_t qf[8][2];
        const int qhead = G8 ? g : (g & 3);
        const bool qhas = qhead < G;
        const uint32_t *qg = reinterpret_cast<const uint32_t *>(
            P.q + ((int64_t)L.b * hkv * G + (int64_t)L.kvh * G + (qhas ? qhead : 0)) * kDim);
        uint32_t qbad = 0;  // FP8: a finite query that overflows f16
#pragma unroll
        for (int kt = 0; kt < 8; ++kt) {
            qf[kt][0] = qhas ? __ldg(qg + 8 * kt + t) : 0u;
            qf[kt][1] = qhas ? __ldg(qg + 8 * kt + t + 4) : 0u;
            if constexpr (kF8) {
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const uint32_t b = qf[kt][w], h = bf16x2_to_f16x2(b);
                    // per half: f16 exponent all ones while the BF16 exponent is not
                    const uint32_t hinf = ~h & 0x7C007C00u, binf = ~b & 0x7F807F80u;
                    qbad |= ((hinf & 0x7C00u) == 0 && (binf & 0x7F80u) != 0) ||
                            ((hinf & 0x7C000000u) == 0 && (binf & 0x7F800000u) != 0);
                    qf[kt][w] = h;
                }
            }
        }
        if (kF8 && __any_sync(0xffffffffu, qbad) && lane == 0) atomicOr(P.status, KVZ_STATUS_Q_RANGE);

        // FMA consumer: the segment's four heads' queries as an fp32 table [kt][t][slot][head]
        // in the warp-merge buffer, idle until the segment ends (the previous segment's
        // readers have passed its closing barrier)
        const float *qs = mo;
        float of[8][4][2];  // FMA consumer: O^T [dim tile][head][dim g | g+8], over the lane's tokens
        if constexpr (kFma) {
            for (int i = tid; i < 512; i += kConsumers * 32) {
                const int h = i & 3, sl = (i >> 2) & 3, tt = (i >> 4) & 3, kt = i >> 6;
                const int d = 16 * kt + 2 * tt + (sl & 1) + 8 * (sl >> 1);
                const uint32_t w =
                    h < G ? P.q[((int64_t)L.b * hkv * G + (int64_t)L.kvh * G + h) * kDim + d] : 0u;
                mo[i] = __uint_as_float(w << 16);
            }
            asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int h = 0; h < 4; ++h) of[a][h][0] = of[a][h][1] = 0.f;
        }

        float o[8][4];
#pragma unroll
        for (int a = 0; a < 8; ++a) o[a][0] = o[a][1] = o[a][2] = o[a][3] = 0.f;
        float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;

        for (int64_t k = warp; k < cnt; k += kConsumers) {
            const int64_t i = ibase + k;
            const int s = (int)(i % kStages);
            const int64_t fill = i / kStages;
            if (ok) ok = mbar_wait(sbase + Smem::full + 8 * s, (uint32_t)(fill & 1), P.status);
            ok = __all_sync(0xffffffffu, ok);  // warp-uniform: the page body uses warp collectives
            const StageInfo inf = info[s];
            if (ok && inf.kind != kKindSkip) {
                const uint8_t *st = smem + Smem::stage + s * kStageBytes;
                const uint32_t sta = sbase + Smem::stage + s * kStageBytes;
                // ---- S^T = K Q^T over the page's 16 tokens ----
                float sc[4] = {0.f, 0.f, 0.f, 0.f};
                float sf[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};  // FMA: [head][token g | g+8]
                // QK^T of block j (two 16-dim tiles) for the 12-bit and raw pages
                auto qk = [&](int j, const uint32_t (&a0)[4], const uint32_t (&a1)[4]) {
                    if constexpr (kFma) {
                        fma_qk_tile(sf, a0, qs, 2 * j, t);
                        fma_qk_tile(sf, a1, qs, 2 * j + 1, t);
                    } else {
                        mma_bf16_16816(sc, a0, qf[2 * j][0], qf[2 * j][1]);
                        mma_bf16_16816(sc, a1, qf[2 * j + 1][0], qf[2 * j + 1][1]);
                    }
                };
                if (kGa && inf.kind == kKindPair && !inf.tagsK) {
                    GaLane gs = ga_lane_load(st, lane);
                    const bool any2 = ga_tile_any_raw_groups(gs);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t a0[4], a1[4];
                        ga_block_frags<false>(st, btbl, gs, any2, lane, j, a0, a1);
                        mma_bf16_16816(sc, a0, qf[2 * j][0], qf[2 * j][1]);
                        mma_bf16_16816(sc, a1, qf[2 * j + 1][0], qf[2 * j + 1][1]);
                    }
                } else if (kF8 && inf.kind == kKindPair && !inf.tagsK) {
                    F8Lane<kE5> fs = f8_lane_load<kE5>(st, lane);
                    const bool any2 = kE5 && __any_sync(0xffffffffu, fs.modes & 0xAAAAu);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t fb[4], a0[4], a1[4];
                        f8_block_bytes<kE5, false>(st, btbl, fs, any2, lane, j, fb);
                        f8_frags_f16<kE5>(fb, a0, a1);
                        mma_f16_16816(sc, a0, qf[2 * j][0], qf[2 * j][1]);
                        mma_f16_16816(sc, a1, qf[2 * j + 1][0], qf[2 * j + 1][1]);
                    }
                } else if (kF8 && inf.kind == kKindPair) {  // raw FP8 tile
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(st + 512 * j + 16 * lane);
                        const uint32_t fb[4] = {v.x, v.y, v.z, v.w};
                        uint32_t a0[4], a1[4];
                        f8_frags_f16<kE5>(fb, a0, a1);
                        mma_f16_16816(sc, a0, qf[2 * j][0], qf[2 * j][1]);
                        mma_f16_16816(sc, a1, qf[2 * j + 1][0], qf[2 * j + 1][1]);
                    }
                } else if (kGa && inf.kind == kKindPair) {  // raw tile: 4 raw 1024-byte blocks
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t a0[4], a1[4];
                        block_frags(st + 1024 * j, 0xFFu, lane, a0, a1);
                        mma_bf16_16816(sc, a0, qf[2 * j][0], qf[2 * j][1]);
                        mma_bf16_16816(sc, a1, qf[2 * j + 1][0], qf[2 * j + 1][1]);
                    }
                } else if (!kTiles && kCompressed && inf.kind == kKindPair) {
                    uint32_t off = 0;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t tag = (inf.tagsK >> (8 * j)) & 0xFFu;
                        uint32_t a0[4], a1[4];
                        block_frags(st + off, tag, lane, a0, a1);
                        qk(j, a0, a1);
                        off += tag_granules(tag) * kGranule;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t a0[4], a1[4];
                        raw_k_frag(sta, j, 0, lane, a0);
                        raw_k_frag(sta, j, 1, lane, a1);
                        if constexpr (kF8) {  // BF16 page: BF16 queries again
                            const int k0 = 2 * j, k1 = 2 * j + 1;
                            const uint32_t q00 = qhas ? __ldg(qg + 8 * k0 + t) : 0u;
                            const uint32_t q01 = qhas ? __ldg(qg + 8 * k0 + t + 4) : 0u;
                            const uint32_t q10 = qhas ? __ldg(qg + 8 * k1 + t) : 0u;
                            const uint32_t q11 = qhas ? __ldg(qg + 8 * k1 + t + 4) : 0u;
                            mma_bf16_16816(sc, a0, q00, q01);
                            mma_bf16_16816(sc, a1, q10, q11);
                        } else {
                            qk(j, a0, a1);
                        }
                    }
                }
                if constexpr (kFma) {  // full dot products on all four t lanes, then this lane's columns
#pragma unroll
                    for (int h = 0; h < 4; ++h)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            sf[h][e] += __shfl_xor_sync(0xffffffffu, sf[h][e], 1);
                            sf[h][e] += __shfl_xor_sync(0xffffffffu, sf[h][e], 2);
                        }
                    const bool hp = t & 1;  // columns 2t, 2t+1 are heads 2t % 4, (2t+1) % 4
                    sc[0] = hp ? sf[2][0] : sf[0][0];
                    sc[1] = hp ? sf[3][0] : sf[1][0];
                    sc[2] = hp ? sf[2][1] : sf[0][1];
                    sc[3] = hp ? sf[3][1] : sf[1][1];
                }
                // sc: (token g, col 2t), (token g, col 2t+1), (token g+8, col 2t), (token g+8, col 2t+1)
                const int valid = (int)inf.valid;
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[e] *= P.scale_log2;
                if (valid < kPage) {
                    if (g >= valid) sc[0] = sc[1] = NEG_INF;
                    if (g + 8 >= valid) sc[2] = sc[3] = NEG_INF;
                }
                // ---- online softmax (column max over the 16 tokens: lanes with equal t) ----
                float x0 = fmaxf(sc[0], sc[2]), x1 = fmaxf(sc[1], sc[3]);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
                    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
                }
                const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
                if (__any_sync(0xffffffffu, (n0 > m0) || (n1 > m1))) {
                    const float a0 = (n0 == NEG_INF) ? 1.f : exp2f(m0 - n0);
                    const float a1 = (n1 == NEG_INF) ? 1.f : exp2f(m1 - n1);
                    if constexpr (kFma) {  // every head's factor: the other pair's from lane t ^ 1
                        const float b0 = __shfl_xor_sync(0xffffffffu, a0, 1), b1 = __shfl_xor_sync(0xffffffffu, a1, 1);
                        const bool hp = t & 1;
                        const float al[4] = {hp ? b0 : a0, hp ? b1 : a1, hp ? a0 : b0, hp ? a1 : b1};
#pragma unroll
                        for (int a = 0; a < 8; ++a)
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                of[a][h][0] *= al[h];
                                of[a][h][1] *= al[h];
                            }
                    } else {
#pragma unroll
                        for (int a = 0; a < 8; ++a) {
                            o[a][0] *= a0;
                            o[a][2] *= a0;
                            o[a][1] *= a1;
                            o[a][3] *= a1;
                        }
                    }
                    l0 *= a0;
                    l1 *= a1;
                    m0 = n0;
                    m1 = n1;
                }
                const float u0 = (m0 == NEG_INF) ? 0.f : m0, u1 = (m1 == NEG_INF) ? 0.f : m1;
                const float p0 = exp2f(sc[0] - u0), p1 = exp2f(sc[1] - u1);
                const float p2 = exp2f(sc[2] - u0), p3 = exp2f(sc[3] - u1);
                l0 += p0 + p2;
                l1 += p1 + p3;
                // P split.  G <= 4: columns 0..3 (t < 2) carry bf16(p), columns 4..7 carry
                // bf16(p - bf16(p)), one MMA per tile.  G > 4: bf16(p) and the remainder go
                // through two MMAs into the same accumulator.
                // (FP8 tiles: the same split in f16, for the f16 PV product)
                const bool pf16 = kF8 && inf.kind == kKindPair;
                auto rnd = [&](float x) { return pf16 ? f16_round(x) : bf16_round(x); };
                auto pack = [&](float a, float b) { return pf16 ? pack_f16x2(a, b) : pack_bf16x2(a, b); };
                float v0 = p0, v1 = p1, v2 = p2, v3 = p3;
                const float r0 = p0 - rnd(p0), r1 = p1 - rnd(p1);
                const float r2 = p2 - rnd(p2), r3 = p3 - rnd(p3);
                if (!G8 && t >= 2) {  // (the remainders are computed by these lanes only)
                    v0 = r0;
                    v1 = r1;
                    v2 = r2;
                    v3 = r3;
                }
                const uint32_t pb0 = movmatrix_trans(pack(v0, v1));  // tokens 0..7
                const uint32_t pb1 = movmatrix_trans(pack(v2, v3));  // tokens 8..15
                uint32_t pl0 = 0, pl1 = 0;
                if (G8) {
                    pl0 = movmatrix_trans(pack(r0, r1));
                    pl1 = movmatrix_trans(pack(r2, r3));
                }
                auto pv = [&](float (&acc)[4], const uint32_t (&a)[4]) {
                    mma_bf16_16816(acc, a, pb0, pb1);
                    if (G8) mma_bf16_16816(acc, a, pl0, pl1);
                };
                auto pv16 = [&](float (&acc)[4], const uint32_t (&a)[4]) {
                    mma_f16_16816(acc, a, pb0, pb1);
                    if (G8) mma_f16_16816(acc, a, pl0, pl1);
                };
                // FMA consumer: P through the warp's table [16 tokens][4 heads] (fp32): each lane
                // needs its tokens 2t, 2t+1, 2t+8, 2t+9 for every head
                float pp[4][4];
                if constexpr (kFma) {
                    float *ps = mo + 512 + warp * 64;
                    if (t < 2) {
                        *reinterpret_cast<float2 *>(ps + g * 4 + 2 * t) = make_float2(p0, p1);
                        *reinterpret_cast<float2 *>(ps + (g + 8) * 4 + 2 * t) = make_float2(p2, p3);
                    }
                    __syncwarp();
                    const int tok[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
                    for (int ts = 0; ts < 4; ++ts) {
                        const float4 v = *reinterpret_cast<const float4 *>(ps + tok[ts] * 4);
                        pp[ts][0] = v.x;
                        pp[ts][1] = v.y;
                        pp[ts][2] = v.z;
                        pp[ts][3] = v.w;
                    }
                }
                // PV of block j (two 16-dim tiles) for the 12-bit and raw pages
                auto pvt = [&](int j, const uint32_t (&a0)[4], const uint32_t (&a1)[4]) {
                    if constexpr (kFma) {
                        fma_pv_tile(of[2 * j], a0, pp);
                        fma_pv_tile(of[2 * j + 1], a1, pp);
                    } else {
                        pv(o[2 * j], a0);
                        pv(o[2 * j + 1], a1);
                    }
                };
                // ---- O^T += V^T P^T ----
                if (kGa && inf.kind == kKindPair && !inf.tagsV) {
                    const uint8_t *tv = st + 4096;
                    GaLane gs = ga_lane_load(tv, lane);
                    const bool any2 = ga_tile_any_raw_groups(gs);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t a0[4], a1[4];
                        ga_block_frags<true>(tv, btbl, gs, any2, lane, j, a0, a1);
                        pv(o[2 * j], a0);
                        pv(o[2 * j + 1], a1);
                    }
                } else if (kF8 && inf.kind == kKindPair && !inf.tagsV) {
                    const uint8_t *tv = st + 4096;
                    F8Lane<kE5> fs = f8_lane_load<kE5>(tv, lane);
                    const bool any2 = kE5 && __any_sync(0xffffffffu, fs.modes & 0xAAAAu);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t fb[4], a0[4], a1[4];
                        f8_block_bytes<kE5, true>(tv, btbl, fs, any2, lane, j, fb);
                        f8_frags_f16<kE5>(fb, a0, a1);
                        pv16(o[2 * j], a0);
                        pv16(o[2 * j + 1], a1);
                    }
                } else if (kF8 && inf.kind == kKindPair) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(st + 4096 + 512 * j + 16 * lane);
                        const uint32_t fb[4] = {v.x, v.y, v.z, v.w};
                        uint32_t a0[4], a1[4];
                        f8_frags_f16<kE5>(fb, a0, a1);
                        pv16(o[2 * j], a0);
                        pv16(o[2 * j + 1], a1);
                    }
                } else if (kGa && inf.kind == kKindPair) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t a0[4], a1[4];
                        block_frags(st + 4096 + 1024 * j, 0xFFu, lane, a0, a1);
                        pv(o[2 * j], a0);
                        pv(o[2 * j + 1], a1);
                    }
                } else if (!kTiles && kCompressed && inf.kind == kKindPair) {
                    uint32_t off = group_granules(inf.tagsK) * kGranule;  // V right after K
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t tag = (inf.tagsV >> (8 * j)) & 0xFFu;
                        uint32_t a0[4], a1[4];
                        block_frags(st + off, tag, lane, a0, a1);
                        pvt(j, a0, a1);
                        off += tag_granules(tag) * kGranule;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t a0[4], a1[4];
                        raw_v_frag(sta, j, 0, lane, a0);
                        raw_v_frag(sta, j, 1, lane, a1);
                        if (valid < kPage) {
                            mask_v_frag(a0, lane, valid);
                            mask_v_frag(a1, lane, valid);
                        }
                        pvt(j, a0, a1);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sbase + Smem::empty + 8 * s);
        }

        // ---- warp state -> shared memory, then the four warps merged (fixed order) into this
        // segment's partial.  G <= 4: columns h and h+4 summed (hi and lo parts of P), one
        // pass.  G > 4: heads 0..3 (lanes t < 2) then heads 4..7 (t >= 2), two passes through
        // the same buffer. ----
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        if constexpr (kFma) {  // sums over all 16 tokens of each page, then this lane's columns
            // the other warps may still read the query and P tables in the merge buffer
            asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int h = 0; h < 4; ++h)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        of[a][h][e] += __shfl_xor_sync(0xffffffffu, of[a][h][e], 1);
                        of[a][h][e] += __shfl_xor_sync(0xffffffffu, of[a][h][e], 2);
                    }
            const bool hp = t & 1;
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                o[a][0] = hp ? of[a][2][0] : of[a][0][0];
                o[a][1] = hp ? of[a][3][0] : of[a][1][0];
                o[a][2] = hp ? of[a][2][1] : of[a][0][1];
                o[a][3] = hp ? of[a][3][1] : of[a][1][1];
            }
        } else if (!G8) {  // columns h and h + 4: the hi and lo parts of P
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[a][e] += __shfl_xor_sync(0xffffffffu, o[a][e], 2);
        }
        const int64_t slot = (int64_t)(L.b * hkv + L.kvh) + c;
        const int gs = G8 ? 8 : 4;  // heads per partial slot
        for (int pass = 0; pass < (G8 ? 2 : 1); ++pass) {
            if ((t >> 1) == pass) {
                const int h0 = 2 * t, h1 = 2 * t + 1;  // heads; buffer rows h - 4 * pass
                if (g == 0) {
                    mm[warp * 8 + h0] = m0;
                    mm[warp * 8 + h1] = m1;
                    mlv[warp * 8 + h0] = l0;
                    mlv[warp * 8 + h1] = l1;
                }
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    const int d0 = 16 * a + g, d1 = 16 * a + g + 8;
                    const int r0 = warp * 4 + h0 - 4 * pass, r1 = warp * 4 + h1 - 4 * pass;
                    mo[r0 * 128 + d0] = o[a][0];
                    mo[r1 * 128 + d0] = o[a][1];
                    mo[r0 * 128 + d1] = o[a][2];
                    mo[r1 * 128 + d1] = o[a][3];
                }
            }
            asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
            {
                const int d = tid;  // 0..127
                const int hend = min(G, 4 * pass + 4);
                for (int h = 4 * pass; h < hend; ++h) {
                    float M = NEG_INF;
#pragma unroll
                    for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, mm[w * 8 + h]);
                    float Lsum = 0.f, Osum = 0.f;
                    if (M != NEG_INF) {
#pragma unroll
                        for (int w = 0; w < kConsumers; ++w) {
                            const float sw = exp2f(mm[w * 8 + h] - M);
                            Lsum += sw * mlv[w * 8 + h];
                            Osum += sw * mo[(w * 4 + h - 4 * pass) * 128 + d];
                        }
                    }
                    P.part_o[(slot * gs + h) * 128 + d] = Osum;
                    if (d == 0) {
                        P.part_ml[(slot * gs + h) * 2 + 0] = M;
                        P.part_ml[(slot * gs + h) * 2 + 1] = Lsum;
                    }
                }
            }
            asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
        }
        x = send;
        ibase += cnt;
    }
}

// ---------------------------------------------------------------------------------
// merge the per-segment partials of each (sequence, KV head): fixed order over CTAs
// ---------------------------------------------------------------------------------
constexpr int kMergeChunk = 8;   // slots whose partials one thread keeps in flight at once
constexpr int kMergeGroups = 4;  // slot ranges merged side by side, then combined in order,
                                 // when units span many CTAs

// Running merge of slots [c0, c1] of one unit (head block hb, dimension d) into M, Ls, Os.
__device__ __forceinline__ void merge_slots(const AttnParams &P, int64_t u, int64_t c0, int64_t c1, int64_t T,
                                            int64_t C, int gs, int hb, int d, float (&M)[4], float (&Ls)[4],
                                            float (&Os)[4])
{
    const int G = P.G;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        M[h] = -INFINITY;
        Ls[h] = 0.f;
        Os[h] = 0.f;
    }
    // within a chunk every load is independent
    for (int64_t cb = c0; cb <= c1; cb += kMergeChunk) {
        float mv[kMergeChunk][4], lv[kMergeChunk][4], ov[kMergeChunk][4];
#pragma unroll
        for (int k = 0; k < kMergeChunk; ++k) {
            const int64_t c = cb + k;
            // (64-bit divisions only when some CTA ranges are empty)
            const bool w = c <= c1 && (T >= C || (c * T + C - 1) / C < ((c + 1) * T + C - 1) / C);
            const int64_t slot = u + c;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                mv[k][h] = -INFINITY;
                lv[k][h] = 0.f;
                ov[k][h] = 0.f;
                if (w && hb + h < G) {
                    const float2 ml = *reinterpret_cast<const float2 *>(P.part_ml + (slot * gs + hb + h) * 2);
                    mv[k][h] = ml.x;
                    lv[k][h] = ml.y;
                    ov[k][h] = P.part_o[(slot * gs + hb + h) * 128 + d];
                }
            }
        }
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            float m = M[h];
#pragma unroll
            for (int k = 0; k < kMergeChunk; ++k) m = fmaxf(m, mv[k][h]);
            if (m == -INFINITY) continue;
            const float r = exp2f(M[h] - m);  // M[h] = -inf -> 0
            float l = Ls[h] * r, o = Os[h] * r;
#pragma unroll
            for (int k = 0; k < kMergeChunk; ++k) {
                const float wgt = exp2f(mv[k][h] - m);
                l += wgt * lv[k][h];
                o += wgt * ov[k][h];
            }
            M[h] = m;
            Ls[h] = l;
            Os[h] = o;
        }
    }
}

// One block per (sequence, KV head), kGroups x 128 threads.  The unit's slots are cut into
// kGroups ranges of at least kMergeChunk slots; each group of 128 threads merges its range,
// and group 0 combines the group results in group order.  A unit with at most kMergeChunk
// slots is merged by group 0 alone (the same arithmetic for every kGroups).
// The launch bounds ask for one block per SM: compiled to fit four blocks per SM (128
// registers instead of ~150), the overlapped launch chain ran 40% slower (8K layer: 106 vs
// 74 us), the plain launches the same.
template <int kGroups>
__global__ void __launch_bounds__(128 * kGroups, 1) k_attn_merge(const AttnParams P)
{
    __shared__ float gm[kGroups][4], gl[kGroups][4], go[kGroups][4][128];
    __shared__ int s_cnt[kGroups * 4][3];
    if (P.overlap) pdl_launch_dependents();  // the next overlapped call may place its CTAs
    const int u = blockIdx.x, hkv = P.hkv, G = P.G;
    const int b = u / hkv, kvh = u % hkv, d = threadIdx.x & 127, grp = threadIdx.x >> 7;
    // pages of the sequences before b, of b, and of all, from the lengths (the attention
    // kernel's count), before the wait: the lengths were complete before the call started
    int pb = 0, nb = 0, pB = 0;
    for (int i = threadIdx.x; i < P.batch; i += blockDim.x) {
        const int L = P.seq_lens[i];
        const int pages = L > 0 ? (L + kPage - 1) / kPage : 0;
        pB += pages;
        pb += i < b ? pages : 0;
        nb += i == b ? pages : 0;
    }
    pb = __reduce_add_sync(0xffffffffu, pb);
    nb = __reduce_add_sync(0xffffffffu, nb);
    pB = __reduce_add_sync(0xffffffffu, pB);
    if ((threadIdx.x & 31) == 0) {
        s_cnt[threadIdx.x >> 5][0] = pb;
        s_cnt[threadIdx.x >> 5][1] = nb;
        s_cnt[threadIdx.x >> 5][2] = pB;
    }
    __syncthreads();
    pb = nb = pB = 0;
#pragma unroll
    for (int w = 0; w < kGroups * 4; ++w) {
        pb += s_cnt[w][0];
        nb += s_cnt[w][1];
        pB += s_cnt[w][2];
    }
    if (P.overlap) pdl_wait_primary();  // the attention grid's partials are complete
    const int64_t n = nb;
    const int64_t T = (int64_t)hkv * pB;
    const int64_t C = P.grid;
    float *out = P.out + ((int64_t)b * hkv * G + (int64_t)kvh * G) * kDim;
    if (n == 0) {
        if (grp == 0)
            for (int h = 0; h < G; ++h) out[h * kDim + d] = 0.f;
        return;
    }
    // CTA c covers pages [ceil(cT/C), ceil((c+1)T/C)); page x belongs to CTA floor(xC/T).
    // CTAs between the first and last owner with an empty range (T < C) wrote nothing.
    const int64_t S = (int64_t)hkv * pb + (int64_t)kvh * n, E = S + n;
    const int64_t c0 = (S * C) / T, c1 = ((E - 1) * C) / T;
    const int64_t ns = c1 - c0 + 1, per = max((int64_t)kMergeChunk, (ns + kGroups - 1) / kGroups);
    const int64_t g0 = c0 + grp * per, g1 = min(c1, g0 + per - 1);  // empty when g0 > c1
    const int gs = G > 4 ? 8 : 4;  // heads per partial slot
    // heads in blocks of four (two blocks for G = 5..8)
    for (int hb = 0; hb < G; hb += 4) {
        float M[4], Ls[4], Os[4];
        merge_slots(P, u, g0, g1, T, C, gs, hb, d, M, Ls, Os);
        if (kGroups == 1 || ns <= kMergeChunk) {  // group 0 holds every slot
            if (grp == 0) {
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    if (hb + h < G) out[(hb + h) * kDim + d] = Ls[h] > 0.f ? Os[h] / Ls[h] : 0.f;
            }
            continue;
        }
        if constexpr (kGroups > 1) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                if (d == 0) {
                    gm[grp][h] = M[h];
                    gl[grp][h] = Ls[h];
                }
                go[grp][h][d] = Os[h];
            }
            __syncthreads();
            if (grp == 0) {
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    float m = -INFINITY;
#pragma unroll
                    for (int k = 0; k < kGroups; ++k) m = fmaxf(m, gm[k][h]);
                    float l = 0.f, o = 0.f;
                    if (m != -INFINITY) {
#pragma unroll
                        for (int k = 0; k < kGroups; ++k) {
                            const float wgt = exp2f(gm[k][h] - m);  // empty group: -inf -> 0
                            l += wgt * gl[k][h];
                            o += wgt * go[k][h][d];
                        }
                    }
                    if (hb + h < G) out[(hb + h) * kDim + d] = l > 0.f ? o / l : 0.f;
                }
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------------------------
// launcher
// ---------------------------------------------------------------------------------
template <int kFmt, bool kG8>
static cudaError_t configure(int dev)
{
    // per process and device: allow the full shared-memory carve-out (attributes are per function)
    static unsigned long long done = 0;  // bit per device ordinal < 64
    if (dev < 64 && (__atomic_load_n(&done, __ATOMIC_ACQUIRE) >> dev) & 1ull) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(k_attn<kFmt, kG8>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attn<kFmt, kG8>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    // the merge runs between attention launches: same carve-out, no reconfiguration
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_attn_merge<1>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attn_merge<kMergeGroups>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess && dev < 64) __atomic_fetch_or(&done, 1ull << dev, __ATOMIC_ACQ_REL);
    return e;
}

template <int kFmt, bool kG8>
static cudaError_t occupancy(int dev, int batch, int *n)
{
    cudaError_t e = configure<kFmt, kG8>(dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, k_attn<kFmt, kG8>, kThreads,
                                                                     Smem::bytes(batch, kFmt >= kFmtGa));
    return e;
}

cudaError_t attn_ctas_per_sm(int batch, int *out)
{
    // the same split for every format and group size: the smallest occupancy of the kernels
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    int n[10] = {0};
    if (e == cudaSuccess) e = occupancy<kFmtRaw, false>(dev, batch, &n[0]);
    if (e == cudaSuccess) e = occupancy<kFmtZf, false>(dev, batch, &n[1]);
    if (e == cudaSuccess) e = occupancy<kFmtGa, false>(dev, batch, &n[2]);
    if (e == cudaSuccess) e = occupancy<kFmtF8E4, false>(dev, batch, &n[3]);
    if (e == cudaSuccess) e = occupancy<kFmtF8E5, false>(dev, batch, &n[4]);
    if (e == cudaSuccess) e = occupancy<kFmtRaw, true>(dev, batch, &n[5]);
    if (e == cudaSuccess) e = occupancy<kFmtZf, true>(dev, batch, &n[6]);
    if (e == cudaSuccess) e = occupancy<kFmtGa, true>(dev, batch, &n[7]);
    if (e == cudaSuccess) e = occupancy<kFmtF8E4, true>(dev, batch, &n[8]);
    if (e == cudaSuccess) e = occupancy<kFmtF8E5, true>(dev, batch, &n[9]);
    int m = n[0];
    for (int k = 1; k < 10; ++k) m = min(m, n[k]);
    *out = e == cudaSuccess ? m : 0;
    return e;
}

template <int kFmt, bool kG8>
static cudaError_t launch_impl(const AttnParams &P, const void *tmap, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = configure<kFmt, kG8>(dev);
    if (e != cudaSuccess) return e;
    CUtensorMap map;
    memcpy(&map, tmap, sizeof(map));
    // slot groups only when the average unit spans more than a chunk of CTAs
    const int64_t units = (int64_t)P.batch * P.hkv;
    const bool groups = (int64_t)P.grid > (int64_t)kMergeChunk * units;
    if (!P.overlap) {
        k_attn<kFmt, kG8><<<P.grid, kThreads, Smem::bytes(P.batch, kFmt >= kFmtGa), stream>>>(P, map);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (groups)
            k_attn_merge<kMergeGroups><<<P.batch * P.hkv, 128 * kMergeGroups, 0, stream>>>(P);
        else
            k_attn_merge<1><<<P.batch * P.hkv, 128, 0, stream>>>(P);
        return cudaGetLastError();
    }
    // overlapped: both kernels are programmatic dependents of the work before them
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(P.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Smem::bytes(P.batch, kFmt >= kFmtGa);
    cfg.stream = stream;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_attn<kFmt, kG8>, P, map);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(P.batch * P.hkv);
    cfg.blockDim = dim3(groups ? 128 * kMergeGroups : 128);
    cfg.dynamicSmemBytes = 0;
    e = groups ? cudaLaunchKernelEx(&cfg, k_attn_merge<kMergeGroups>, P) : cudaLaunchKernelEx(&cfg, k_attn_merge<1>, P);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <bool kG8>
static cudaError_t launch_format(const AttnParams &P, int format, const void *tmap, cudaStream_t stream)
{
    switch (format) {
    case kFmtRaw: return launch_impl<kFmtRaw, kG8>(P, tmap, stream);
    case kFmtZf: return launch_impl<kFmtZf, kG8>(P, tmap, stream);
    case kFmtGa: return launch_impl<kFmtGa, kG8>(P, tmap, stream);
    case kFmtF8E4: return launch_impl<kFmtF8E4, kG8>(P, tmap, stream);
    case kFmtF8E5: return launch_impl<kFmtF8E5, kG8>(P, tmap, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_attention(const AttnParams &P, int format, const void *tmap, cudaStream_t stream)
{
    return P.G > 4 ? launch_format<true>(P, format, tmap, stream) : launch_format<false>(P, format, tmap, stream);
}

}  // namespace kvz
