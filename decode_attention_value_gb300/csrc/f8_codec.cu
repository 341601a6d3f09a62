// f8_codec.cu -- FP8 KV pages: conversion of completed BF16 pages to FP8 (E4M3 or E5M2)
// and their group-adaptive exponent coding (GAAC, "Relation to FP8 KV" applied to the
// codec of "Group-adaptive additive coding"): calibration, encoder (size pass, the shared
// placement scan, pack) and the standalone decoder to FP8 bytes.  Layout and restore:
// f8.cuh.
#include "f8.cuh"
#include "kvz_internal.h"
#include "stage.cuh"

namespace kvz {

// ---------------------------------------------------------------------------------
// calibration over the FP8 exponent fields of the converted sample pages; E4M3 has
// b4 = 0 (its 16-wide window is the whole field)
// ---------------------------------------------------------------------------------
template <bool kE5>
__global__ void __launch_bounds__(256) k_f8_calibrate(int hkv, const uint16_t *pool, int64_t num_raw_pages,
                                                      const int32_t *pages, int n, uint8_t *bases, uint32_t *status)
{
    constexpr int kVals = kE5 ? 32 : 16;
    constexpr int kM = F8Layout<kE5>::kM;
    __shared__ uint32_t hist[kVals][32];
    const int quarter = blockIdx.x & 3, kv = (blockIdx.x >> 2) & 1, head = blockIdx.x >> 3;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int k = threadIdx.x; k < kVals * 32; k += blockDim.x) (&hist[0][0])[k] = 0;
    __syncthreads();
    const int ch = 32 * quarter + lane;
    uint32_t bad = 0;
    for (int64_t item = warp; item < (int64_t)n * kPage; item += 8) {
        const int p = pages[item / kPage], tok = (int)(item % kPage);
        if (p < 0 || p >= num_raw_pages) {
            bad = 1;
            continue;
        }
        const uint32_t w = pool[(((int64_t)p * hkv + head) * 2 + kv) * kPage * kDim + tok * kDim + ch];
        const uint32_t b = f8_from_bf16x2<kE5>(w) & 0xFFu;
        atomicAdd(&hist[(b >> kM) & (kVals - 1)][lane], 1u);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(status, KVZ_STATUS_BAD_INDEX);
    __syncthreads();
    if (warp == 0) {
        uint8_t *out = bases + ((size_t)head * 2 + kv) * 256;
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            const int width = w ? 16 : 8;
            uint32_t cov = 0;
            for (int e = 0; e < width; ++e) cov += hist[e][lane];
            uint32_t best = cov, best_b = 0;
            for (int b = 1; b + width <= kVals; ++b) {
                cov += hist[b + width - 1][lane] - hist[b - 1][lane];
                if (cov > best) {
                    best = cov;
                    best_b = (uint32_t)b;
                }
            }
            out[w * 128 + ch] = (uint8_t)best_b;
        }
    }
}

// ---------------------------------------------------------------------------------
// a lane's two groups of block (kv, j): FP8 bytes and modes
// ---------------------------------------------------------------------------------
template <bool kE5>
struct F8Groups {
    uint32_t fb[4];    // FP8 bytes: fragment 0 elements 0..3, 4..7; fragment 1 likewise
    uint32_t mode[2];
    uint32_t esc[2];
};

template <bool kE5>
__device__ __forceinline__ void f8_modes(const uint8_t *stage, const uint8_t *sb, int kv, int j, int lane,
                                         F8Groups<kE5> &G)
{
    constexpr int kM = F8Layout<kE5>::kM;
    uint32_t w[8];
    gather_block(stage, kv, j, lane, w);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t lo = f8_from_bf16x2<kE5>(w[2 * k]), hi = f8_from_bf16x2<kE5>(w[2 * k + 1]);
        G.fb[k] = lo | (hi << 16);
    }
#pragma unroll
    for (int f = 0; f < 2; ++f) {
        bool ok3 = true, ok4 = true;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t b = (G.fb[2 * f + i / 4] >> (8 * (i & 3))) & 0xFFu;
            const uint32_t e = (b >> kM) & (kE5 ? 31u : 15u);
            const int dim = 32 * j + 16 * f + (kv == 0 ? frag_col(lane, i) : frag_row(lane, i));
            const uint32_t b3 = sb[(kv * 2 + 0) * 128 + dim], b4 = sb[(kv * 2 + 1) * 128 + dim];
            ok3 = ok3 && e >= b3 && e - b3 < 8u;
            ok4 = ok4 && e >= b4 && e - b4 < 16u;
        }
        G.mode[f] = ok3 ? 0u : (ok4 ? 1u : 2u);
        G.esc[f] = ok3 ? 0u : (ok4 ? 1u : F8Layout<kE5>::kEscRaw);
    }
}

__device__ __forceinline__ void f8_stage_page(const EncodeParams &P, int entry, int head, uint8_t *stage, uint8_t *sb)
{
    const int src = P.src_page[entry];
    const uint16_t *slice = P.raw_pool + ((int64_t)src * P.hkv + head) * 2 * kPage * kDim;
    load_slice_to_stage(slice, stage, threadIdx.x, blockDim.x);
    for (int k = threadIdx.x; k < 512 / 16; k += blockDim.x)
        reinterpret_cast<uint4 *>(sb)[k] = reinterpret_cast<const uint4 *>(P.ga_bases + (size_t)head * 512)[k];
}

template <bool kE5>
__host__ __device__ __forceinline__ uint32_t f8_granules(uint32_t escapes)
{
    return (escapes <= F8Layout<kE5>::kEscCap ? F8Layout<kE5>::kTileBytes : 2048u) / kGaGranule;
}

template <bool kE5>
__global__ void __launch_bounds__(256) k_f8_sizes(EncodeParams P)
{
    __shared__ __align__(16) uint8_t stage[32 * kStagePitch];
    __shared__ __align__(16) uint8_t sb[512];
    __shared__ uint32_t esc[8];
    if (P.ws_hdr[0] != 0) return;
    const int entry = (int)(blockIdx.x / P.hkv), head = (int)(blockIdx.x % P.hkv);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kv = warp >> 2, j = warp & 3;
    f8_stage_page(P, entry, head, stage, sb);
    __syncthreads();
    F8Groups<kE5> G;
    f8_modes<kE5>(stage, sb, kv, j, lane, G);
    const uint32_t n = __reduce_add_sync(0xffffffffu, G.esc[0] + G.esc[1]);
    if (lane == 0) esc[warp] = n;
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t g = f8_granules<kE5>(esc[0] + esc[1] + esc[2] + esc[3]) +
                           f8_granules<kE5>(esc[4] + esc[5] + esc[6] + esc[7]);
        P.ws_pair_size[(int64_t)entry * P.hkv + head] = g;
        atomicAdd(P.ws_page_size + entry, g);
    }
}

template <bool kE5>
__global__ void __launch_bounds__(256) k_f8_pack(EncodeParams P)
{
    using Lt = F8Layout<kE5>;
    constexpr int kM = Lt::kM, kS = Lt::kS;
    __shared__ __align__(16) uint8_t stage[32 * kStagePitch];
    __shared__ __align__(16) uint8_t sb[512];
    __shared__ __align__(16) uint8_t tile[2][Lt::kTileBytes];
    __shared__ uint8_t cnt[2][32][4];
    __shared__ uint32_t total[2];
    if (P.ws_hdr[0] != 0) return;
    const int entry = (int)(blockIdx.x / P.hkv), head = (int)(blockIdx.x % P.hkv);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kv = warp >> 2, j = warp & 3;
    const int dst = P.dst_page[entry], seq = P.dst_seq[entry];
    f8_stage_page(P, entry, head, stage, sb);
    // every tile byte is OR-ed or written below: start from zero
    for (int k = threadIdx.x; k < (int)(2 * Lt::kTileBytes / 16); k += blockDim.x)
        reinterpret_cast<uint4 *>(&tile[0][0])[k] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    F8Groups<kE5> G;
    f8_modes<kE5>(stage, sb, kv, j, lane, G);
    cnt[kv][lane][j] = (uint8_t)(G.esc[0] + G.esc[1]);
    __syncthreads();
    uint32_t tot = 0, before_j = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t c = cnt[kv][lane][k];
        tot += c;
        if (k < j) before_j += c;
    }
    uint32_t incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31 && j == 0) total[kv] = incl;
    const bool compressed = __shfl_sync(0xffffffffu, incl, 31) <= Lt::kEscCap;
    uint64_t pair_base = P.ws_page_base[entry];
    for (int h = 0; h < head; ++h) pair_base += P.ws_pair_size[(int64_t)entry * P.hkv + h];
    __syncthreads();
    const uint32_t gK = f8_granules<kE5>(total[0]), gV = f8_granules<kE5>(total[1]);
    const uint64_t off0 = pair_base + (kv ? gK : 0);
    uint64_t end = P.cursors[2 * seq + 1];
    end = min(end, P.arena_bytes / kGaGranule);
    end = min(end, (uint64_t)kGaOffsetMask);
    const bool fits = off0 + (kv ? gV : gK) <= end;

    if (compressed) {
        uint8_t *t = tile[kv];
        uint32_t off = (incl - tot) + before_j;
#pragma unroll
        for (int f = 0; f < 2; ++f) {
            const int q = 8 * lane + 2 * j + f;
            uint32_t smf = 0, codef = 0, hb = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t b = (G.fb[2 * f + i / 4] >> (8 * (i & 3))) & 0xFFu;
                const uint32_t e = (b >> kM) & (kE5 ? 31u : 15u);
                const int dim = 32 * j + 16 * f + (kv == 0 ? frag_col(lane, i) : frag_row(lane, i));
                const uint32_t base = G.mode[f] == 0 ? sb[kv * 256 + dim] : (G.mode[f] == 1 ? sb[kv * 256 + 128 + dim] : 0u);
                const uint32_t c = e - base;
                smf |= (((b >> 7) << kM) | (b & ((1u << kM) - 1))) << (kS * i);
                codef |= (c & 7u) << (3 * i);
                if (G.mode[f] == 1) hb |= ((c >> 3) & 1u) << i;
                if (G.mode[f] == 2) hb |= ((c >> 3) & 3u) << (2 * i);
            }
#pragma unroll
            for (int k = 0; k < kS; ++k) t[kS * q + k] = (uint8_t)(smf >> (8 * k));
#pragma unroll
            for (int k = 0; k < 3; ++k) t[Lt::kCodeOff + 3 * q + k] = (uint8_t)(codef >> (8 * k));
            atomicOr(reinterpret_cast<uint32_t *>(t + Lt::kTagOff + ((q >> 2) & ~3)), G.mode[f] << (2 * (q & 15)));
            if (G.mode[f] == 1) {
                t[Lt::kEscOff + off] = (uint8_t)hb;
                off += 1;
            } else if (G.mode[f] == 2) {
                t[Lt::kEscOff + off] = (uint8_t)hb;
                t[Lt::kEscOff + off + 1] = (uint8_t)(hb >> 8);
                off += 2;
            }
        }
    } else if (fits) {
        // raw: the FP8 bytes in storage order, 16 per lane per block
        uint8_t *blk = P.arena + off0 * kGaGranule + 512 * j + 16 * lane;
        *reinterpret_cast<uint4 *>(blk) = make_uint4(G.fb[0], G.fb[1], G.fb[2], G.fb[3]);
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const bool comp = total[t] <= Lt::kEscCap;
        const uint64_t o = pair_base + (t ? gK : 0);
        const bool fit = o + (t ? gV : gK) <= end;
        if (comp && fit) {
            uint4 *d = reinterpret_cast<uint4 *>(P.arena + o * kGaGranule);
            const uint4 *s = reinterpret_cast<const uint4 *>(tile[t]);
            for (int k = threadIdx.x; k < (int)(Lt::kTileBytes / 16); k += blockDim.x) d[k] = s[k];
        }
        if (threadIdx.x == 0) {
            const uint32_t word = fit ? ((uint32_t)o | (comp ? 0u : kGaEntryRaw)) : kGaEntryInvalid;
            P.meta32[((int64_t)dst * P.hkv + head) * 2 + t] = word;
            if (!fit) atomicOr(P.status, KVZ_STATUS_ARENA_FULL);
        }
    }
}

// ---------------------------------------------------------------------------------
// standalone decode to FP8 bytes: out uint8 [n][hkv][2][16][128].  Warp per (entry, head)
// item in a grid-stride loop: per tile the lane state is loaded once and the four blocks
// are restored with the attention kernel's register path into the warp's 4 KB page buffer.
// ---------------------------------------------------------------------------------
constexpr int kF8DecWarps = 8;
constexpr int kF8DecSmem = kF8DecWarps * 2 * kPage * kDim;  // 32 KB

template <bool kE5>
__global__ void __launch_bounds__(kF8DecWarps * 32) k_f8_decode_w(DecodeParams P)
{
    extern __shared__ __align__(16) uint8_t f8_dec_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *page = f8_dec_smem + warp * (2 * kPage * kDim);
    const int64_t items = (int64_t)P.n * P.hkv;
    const int64_t stride = (int64_t)gridDim.x * kF8DecWarps;
    for (int64_t it = (int64_t)blockIdx.x * kF8DecWarps + warp; it < items; it += stride) {
        const int entry = (int)(it / P.hkv), head = (int)(it % P.hkv);
        const int pid = P.page[entry];
        const bool page_ok = pid >= 0 && pid < P.num_meta_pages;
        uint32_t bad = page_ok ? 0u : KVZ_STATUS_BAD_INDEX;
        uint2 words = make_uint2(kGaEntryInvalid, kGaEntryInvalid);
        if (page_ok) words = *reinterpret_cast<const uint2 *>(P.meta32 + ((int64_t)pid * P.hkv + head) * 2);
        __syncwarp();  // the previous item's stores are done with the buffer
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
            const uint32_t word = kv ? words.y : words.x;
            const uint64_t off = word & kGaOffsetMask;
            bool use = page_ok;
            if (use && (word == kGaEntryInvalid ||
                        off * kGaGranule + f8_entry_bytes(kE5 ? kF8E5M2 : kF8E4M3, word) > P.arena_bytes)) {
                bad |= KVZ_STATUS_BAD_META;
                use = false;
            }
            const uint8_t *tile = P.arena + off * kGaGranule;
            const uint8_t *row = P.ga_bases + ((size_t)head * 2 + kv) * 256;
            const bool raw = use && (word & kGaEntryRaw);
            F8Lane<kE5> s;
            bool any2 = false;
            if (use && !raw) {  // warp-uniform
                s = f8_lane_load<kE5>(tile, lane);
                any2 = __any_sync(0xffffffffu, s.modes & 0xAAAAu);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t fb[4] = {0, 0, 0, 0};
                if (raw) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(tile + 512 * j + 16 * lane);
                    fb[0] = v.x; fb[1] = v.y; fb[2] = v.z; fb[3] = v.w;
                } else if (use) {
                    if (kv == 0) f8_block_bytes<kE5, false>(tile, row, s, any2, lane, j, fb);
                    else f8_block_bytes<kE5, true>(tile, row, s, any2, lane, j, fb);
                }
#pragma unroll
                for (int f = 0; f < 2; ++f)
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int r = frag_row(lane, i), c = frag_col(lane, i);
                        const int dim0 = 32 * j + 16 * f;
                        const uint8_t b = (uint8_t)(fb[2 * f + i / 4] >> (8 * (i & 3)));
                        if (kv == 0) page[r * kDim + dim0 + c] = b;                      // K: token r, dim c
                        else page[kPage * kDim + c * kDim + dim0 + r] = b;                // V: token c, dim r
                    }
            }
        }
        if (bad && lane == 0) atomicOr(P.status, bad);
        __syncwarp();
        uint4 *out = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(P.out) +
                                               ((int64_t)entry * P.hkv + head) * 2 * kPage * kDim);
#pragma unroll
        for (int k = 0; k < 8; ++k) out[lane + 32 * k] = reinterpret_cast<const uint4 *>(page)[lane + 32 * k];
    }
}

// ---------------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------------
cudaError_t launch_f8_calibrate(int fmt, int hkv, const uint16_t *raw_pool, int64_t num_raw_pages,
                                const int32_t *pages, int n, uint8_t *bases, uint32_t *status, cudaStream_t stream)
{
    if (fmt == kF8E5M2) k_f8_calibrate<true><<<hkv * 8, 256, 0, stream>>>(hkv, raw_pool, num_raw_pages, pages, n, bases, status);
    else k_f8_calibrate<false><<<hkv * 8, 256, 0, stream>>>(hkv, raw_pool, num_raw_pages, pages, n, bases, status);
    return cudaGetLastError();
}

cudaError_t launch_f8_encode(int fmt, const EncodeParams &P, cudaStream_t stream)
{
    cudaError_t e = launch_enc_prepare(P, stream);  // validation and page-size reset
    if (e != cudaSuccess) return e;
    const unsigned items = (unsigned)((size_t)P.n * P.hkv);
    if (fmt == kF8E5M2) k_f8_sizes<true><<<items, 256, 0, stream>>>(P);
    else k_f8_sizes<false><<<items, 256, 0, stream>>>(P);
    e = launch_enc_scan(P, stream);
    if (e != cudaSuccess) return e;
    if (fmt == kF8E5M2) k_f8_pack<true><<<items, 256, 0, stream>>>(P);
    else k_f8_pack<false><<<items, 256, 0, stream>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_f8_decode(int fmt, const DecodeParams &P, cudaStream_t stream)
{
    static unsigned long long done = 0;  // bit per device ordinal < 64: shared-memory opt-in
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess && !(dev < 64 && ((__atomic_load_n(&done, __ATOMIC_ACQUIRE) >> dev) & 1ull))) {
        e = cudaFuncSetAttribute(k_f8_decode_w<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kF8DecSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_f8_decode_w<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kF8DecSmem);
        if (e == cudaSuccess && dev < 64) __atomic_fetch_or(&done, 1ull << dev, __ATOMIC_ACQ_REL);
    }
    if (e != cudaSuccess) return e;
    const int64_t items = (int64_t)P.n * P.hkv, want = (items + kF8DecWarps - 1) / kF8DecWarps;
    const int64_t wave = (int64_t)(sms > 0 ? sms : 1) * 4;
    const unsigned grid = (unsigned)(want < wave ? (want > 0 ? want : 1) : wave);
    if (fmt == kF8E5M2) k_f8_decode_w<true><<<grid, kF8DecWarps * 32, kF8DecSmem, stream>>>(P);
    else k_f8_decode_w<false><<<grid, kF8DecWarps * 32, kF8DecSmem, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace kvz
