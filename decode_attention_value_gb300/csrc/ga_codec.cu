// ga_codec.cu -- calibration, page encoder and standalone decoder for the
// group-adaptive additive tile format (GAAC, "Lossless KV Compression":
// "Contiguous exponent concentration", "Group-adaptive additive coding"; Table 9;
// "Block-Wise Compression Scheduling": two storage classes recorded in the block
// table).  Tile layout and restore: ga.cuh.
//
// Encoding reuses the 12-bit encoder's validation and placement scan: a size pass
// (tile escape bytes -> 47 or 64 granules of 64 B per tile), the segmented scan over
// pages that advances each sequence's cursor, and a pack pass that builds each
// compressed tile in shared memory and writes it out with 16-byte stores.
#include "ga.cuh"
#include "kvz_internal.h"
#include "stage.cuh"

namespace kvz {

// ---------------------------------------------------------------------------------
// calibration: per (head, K|V, channel) exponent histogram over the sample pages, then
// the 8- and 16-wide windows covering the most values (lowest start on ties).
// Grid: (head, K|V, quarter of the channels); 8 warps stride over the sample tokens,
// lane = channel.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_ga_calibrate(int hkv, const uint16_t *pool, int64_t num_raw_pages,
                                                      const int32_t *pages, int n, uint8_t *bases, uint32_t *status)
{
    __shared__ uint32_t hist[256][32];
    const int quarter = blockIdx.x & 3, kv = (blockIdx.x >> 2) & 1, head = blockIdx.x >> 3;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int k = threadIdx.x; k < 256 * 32; k += blockDim.x) (&hist[0][0])[k] = 0;
    __syncthreads();
    const int ch = 32 * quarter + lane;
    uint32_t bad = 0;
    for (int64_t item = warp; item < (int64_t)n * kPage; item += 8) {
        const int p = pages[item / kPage], tok = (int)(item % kPage);
        if (p < 0 || p >= num_raw_pages) {
            bad = 1;
            continue;
        }
        const uint16_t w = pool[(((int64_t)p * hkv + head) * 2 + kv) * kPage * kDim + tok * kDim + ch];
        atomicAdd(&hist[(w >> 7) & 0xFFu][lane], 1u);
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
            for (int b = 1; b + width <= 256; ++b) {
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
// group modes of a lane's two groups of block (kv, j), from the staged slice
// ---------------------------------------------------------------------------------
struct GaGroups {
    uint32_t w[8];     // the 16 values in storage order (see gather_block)
    uint32_t mode[2];  // per fragment f
    uint32_t esc[2];   // escape bytes per fragment
};

// sb: this head's bases in shared memory, [2 kv][2 width][128]
__device__ __forceinline__ void ga_modes(const uint8_t *stage, const uint8_t *sb, int kv, int j, int lane, GaGroups &G)
{
    gather_block(stage, kv, j, lane, G.w);
#pragma unroll
    for (int f = 0; f < 2; ++f) {
        bool ok3 = true, ok4 = true;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t v = (G.w[f * 4 + i / 2] >> (16 * (i & 1))) & 0xFFFFu;
            const uint32_t e = (v >> 7) & 0xFFu;
            const int dim = 32 * j + 16 * f + (kv == 0 ? frag_col(lane, i) : frag_row(lane, i));
            const uint32_t b3 = sb[(kv * 2 + 0) * 128 + dim], b4 = sb[(kv * 2 + 1) * 128 + dim];
            ok3 = ok3 && e >= b3 && e - b3 < 8u;
            ok4 = ok4 && e >= b4 && e - b4 < 16u;
        }
        G.mode[f] = ok3 ? 0u : (ok4 ? 1u : 2u);
        G.esc[f] = ok3 ? 0u : (ok4 ? 1u : 5u);
    }
}

__device__ __forceinline__ void ga_stage_page(const EncodeParams &P, int entry, int head, uint8_t *stage, uint8_t *sb)
{
    const int src = P.src_page[entry];
    const uint16_t *slice = P.raw_pool + ((int64_t)src * P.hkv + head) * 2 * kPage * kDim;
    load_slice_to_stage(slice, stage, threadIdx.x, blockDim.x);
    for (int k = threadIdx.x; k < 512 / 16; k += blockDim.x)
        reinterpret_cast<uint4 *>(sb)[k] = reinterpret_cast<const uint4 *>(P.ga_bases + (size_t)head * 512)[k];
}

// ---------------------------------------------------------------------------------
// size pass: one CTA per (entry, head); warp w = block (kv = w/4, j = w%4)
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_ga_sizes(EncodeParams P)
{
    __shared__ __align__(16) uint8_t stage[32 * kStagePitch];
    __shared__ __align__(16) uint8_t sb[512];
    __shared__ uint32_t esc[8];
    if (P.ws_hdr[0] != 0) return;
    const int entry = (int)(blockIdx.x / P.hkv), head = (int)(blockIdx.x % P.hkv);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kv = warp >> 2, j = warp & 3;
    ga_stage_page(P, entry, head, stage, sb);
    __syncthreads();
    GaGroups G;
    ga_modes(stage, sb, kv, j, lane, G);
    const uint32_t n = __reduce_add_sync(0xffffffffu, G.esc[0] + G.esc[1]);
    if (lane == 0) esc[warp] = n;
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t eK = esc[0] + esc[1] + esc[2] + esc[3], eV = esc[4] + esc[5] + esc[6] + esc[7];
        const uint32_t g = (eK <= kGaEscCap ? kGaTileBytes : kGaRawBytes) / kGaGranule +
                           (eV <= kGaEscCap ? kGaTileBytes : kGaRawBytes) / kGaGranule;
        P.ws_pair_size[(int64_t)entry * P.hkv + head] = g;
        atomicAdd(P.ws_page_size + entry, g);
    }
}

// ---------------------------------------------------------------------------------
// pack pass: one CTA per (entry, head).  Each warp (kv, j) computes its lanes' two
// groups, the escape offsets (lane-major group order) come from per-lane counts in
// shared memory, compressed tiles are assembled in shared memory and copied out,
// raw tiles are written straight from the gathered words.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_ga_pack(EncodeParams P)
{
    __shared__ __align__(16) uint8_t stage[32 * kStagePitch];
    __shared__ __align__(16) uint8_t sb[512];
    __shared__ __align__(16) uint8_t tile[2][kGaTileBytes];
    __shared__ uint8_t cnt[2][32][4];  // escape bytes of lane L's two groups of block j
    __shared__ uint32_t total[2];
    if (P.ws_hdr[0] != 0) return;
    const int entry = (int)(blockIdx.x / P.hkv), head = (int)(blockIdx.x % P.hkv);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kv = warp >> 2, j = warp & 3;
    const int dst = P.dst_page[entry], seq = P.dst_seq[entry];
    ga_stage_page(P, entry, head, stage, sb);
    // modes and escape area start at zero; the other tile bytes are all written below
    for (int k = threadIdx.x; k < 2 * 12; k += blockDim.x)  // bytes [2816, 3008) = 12 uint4 per tile
        reinterpret_cast<uint4 *>(tile[k / 12] + kGaTagOff)[k % 12] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    GaGroups G;
    ga_modes(stage, sb, kv, j, lane, G);
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
    const uint32_t tile_esc = __shfl_sync(0xffffffffu, incl, 31);
    const bool compressed = tile_esc <= kGaEscCap;

    // placement: the page's position, then the heads before this one, then K before V
    uint64_t pair_base = P.ws_page_base[entry];
    for (int h = 0; h < head; ++h) pair_base += P.ws_pair_size[(int64_t)entry * P.hkv + h];
    __syncthreads();  // total[] visible
    const uint32_t gK = (total[0] <= kGaEscCap ? kGaTileBytes : kGaRawBytes) / kGaGranule;
    const uint32_t gV = (total[1] <= kGaEscCap ? kGaTileBytes : kGaRawBytes) / kGaGranule;
    const uint64_t gmine = kv ? gV : gK;
    const uint64_t off0 = pair_base + (kv ? gK : 0);
    uint64_t end = P.cursors[2 * seq + 1];
    end = min(end, P.arena_bytes / kGaGranule);
    end = min(end, (uint64_t)kGaOffsetMask);
    const bool fits = off0 + gmine <= end;

    if (compressed) {
        uint8_t *t = tile[kv];
        uint32_t sfw[4], codes[2];
#pragma unroll
        for (int f = 0; f < 2; ++f) {
            uint32_t sf0 = 0, sf1 = 0, field = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t v = (G.w[f * 4 + i / 2] >> (16 * (i & 1))) & 0xFFFFu;
                const uint32_t e = (v >> 7) & 0xFFu;
                const uint32_t sf = ((v >> 8) & 0x80u) | (v & 0x7Fu);
                const int dim = 32 * j + 16 * f + (kv == 0 ? frag_col(lane, i) : frag_row(lane, i));
                const uint32_t b = G.mode[f] == 0 ? sb[kv * 256 + dim] : (G.mode[f] == 1 ? sb[kv * 256 + 128 + dim] : 0u);
                const uint32_t c = e - b;
                if (i < 4) sf0 |= sf << (8 * i);
                else sf1 |= sf << (8 * (i - 4));
                field |= (c & 7u) << (3 * i);
            }
            sfw[2 * f] = sf0;
            sfw[2 * f + 1] = sf1;
            codes[f] = field;
        }
        *reinterpret_cast<uint4 *>(t + 512 * j + 16 * lane) = make_uint4(sfw[0], sfw[1], sfw[2], sfw[3]);
#pragma unroll
        for (int f = 0; f < 2; ++f) {
            const int q = 8 * lane + 2 * j + f;
            t[kGaCodeOff + 3 * q] = (uint8_t)codes[f];
            t[kGaCodeOff + 3 * q + 1] = (uint8_t)(codes[f] >> 8);
            t[kGaCodeOff + 3 * q + 2] = (uint8_t)(codes[f] >> 16);
        }
        // modes: this warp's two groups are bits [4(j%2), 4(j%2)+4) of byte 2L + j/2
        const uint32_t nib = G.mode[0] | (G.mode[1] << 2);
        const int tb = 2 * lane + (j >> 1);
        atomicOr(reinterpret_cast<uint32_t *>(t + kGaTagOff + (tb & ~3)), nib << (8 * (tb & 3) + 4 * (j & 1)));
        // escape bytes
        uint32_t off = (incl - tot) + before_j;
#pragma unroll
        for (int f = 0; f < 2; ++f) {
            if (G.mode[f] == 0) continue;
            uint32_t hb_lo = 0, hb_hi = 0;  // 40-bit field for raw groups, byte for 4-bit groups
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t v = (G.w[f * 4 + i / 2] >> (16 * (i & 1))) & 0xFFFFu;
                const uint32_t e = (v >> 7) & 0xFFu;
                const int dim = 32 * j + 16 * f + (kv == 0 ? frag_col(lane, i) : frag_row(lane, i));
                if (G.mode[f] == 1) {
                    hb_lo |= (((e - sb[kv * 256 + 128 + dim]) >> 3) & 1u) << i;
                } else {
                    const uint64_t h5 = (uint64_t)((e >> 3) & 31u) << (5 * i);
                    hb_lo |= (uint32_t)h5;
                    hb_hi |= (uint32_t)(h5 >> 32);
                }
            }
            uint8_t *e = t + kGaEscOff;
            if (G.mode[f] == 1) {
                e[off] = (uint8_t)hb_lo;
                off += 1;
            } else {
                e[off] = (uint8_t)hb_lo;
                e[off + 1] = (uint8_t)(hb_lo >> 8);
                e[off + 2] = (uint8_t)(hb_lo >> 16);
                e[off + 3] = (uint8_t)(hb_lo >> 24);
                e[off + 4] = (uint8_t)hb_hi;
                off += 5;
            }
        }
    } else if (fits) {
        uint8_t *blk = P.arena + off0 * kGaGranule + 1024 * j;
        *reinterpret_cast<uint4 *>(blk + 32 * lane) = make_uint4(G.w[0], G.w[1], G.w[2], G.w[3]);
        *reinterpret_cast<uint4 *>(blk + 32 * lane + 16) = make_uint4(G.w[4], G.w[5], G.w[6], G.w[7]);
    }
    __syncthreads();
    // copy the compressed tiles out (188 uint4 each)
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const bool comp = total[t] <= kGaEscCap;
        const uint64_t o = pair_base + (t ? gK : 0);
        const bool fit = o + (t ? gV : gK) <= end;
        if (comp && fit) {
            uint4 *d = reinterpret_cast<uint4 *>(P.arena + o * kGaGranule);
            const uint4 *s = reinterpret_cast<const uint4 *>(tile[t]);
            for (int k = threadIdx.x; k < (int)(kGaTileBytes / 16); k += blockDim.x) d[k] = s[k];
        }
        if (threadIdx.x == 0) {
            const uint32_t word = fit ? ((uint32_t)o | (comp ? 0u : kGaEntryRaw)) : kGaEntryInvalid;
            P.meta32[((int64_t)dst * P.hkv + head) * 2 + t] = word;
            if (!fit) atomicOr(P.status, KVZ_STATUS_ARENA_FULL);
        }
    }
}

// ---------------------------------------------------------------------------------
// standalone decode: warp per (entry, head) item in a grid-stride loop; per tile the
// lane state (modes, escape offset, codes) is loaded once and the four blocks are
// restored with the attention kernel's register path, scattered into the warp's staged
// page slice and written back in the plain page layout.
// ---------------------------------------------------------------------------------
constexpr int kGaDecWarps = 8;

__global__ void __launch_bounds__(kGaDecWarps * 32, 3) k_ga_decode_w(DecodeParams P)
{
    extern __shared__ __align__(16) uint8_t ga_dec_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *stage = ga_dec_smem + warp * (32 * kStagePitch);
    const int64_t items = (int64_t)P.n * P.hkv;
    const int64_t stride = (int64_t)gridDim.x * kGaDecWarps;
    for (int64_t it = (int64_t)blockIdx.x * kGaDecWarps + warp; it < items; it += stride) {
        const int entry = (int)(it / P.hkv), head = (int)(it % P.hkv);
        const int page = P.page[entry];
        const bool page_ok = page >= 0 && page < P.num_meta_pages;
        uint32_t bad = page_ok ? 0u : KVZ_STATUS_BAD_INDEX;
        uint2 words = make_uint2(kGaEntryInvalid, kGaEntryInvalid);
        if (page_ok) words = *reinterpret_cast<const uint2 *>(P.meta32 + ((int64_t)page * P.hkv + head) * 2);
        __syncwarp();  // the previous item's stores are done with the buffer
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
            const uint32_t ew = kv ? words.y : words.x;
            const uint64_t off = ew & kGaOffsetMask;
            bool use = page_ok;
            if (use && (ew == kGaEntryInvalid || off * kGaGranule + ga_entry_bytes(ew) > P.arena_bytes)) {
                bad |= KVZ_STATUS_BAD_META;
                use = false;
            }
            const uint8_t *tile = P.arena + off * kGaGranule;
            const uint8_t *row = P.ga_bases + ((size_t)head * 2 + kv) * 256;
            const bool raw = use && (ew & kGaEntryRaw);
            GaLane gs;
            bool any2 = false;
            if (use && !raw) {  // warp-uniform
                gs = ga_lane_load(tile, lane);
                any2 = ga_tile_any_raw_groups(gs);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                if (raw) {
                    const uint4 a = *reinterpret_cast<const uint4 *>(tile + 1024 * j + 32 * lane);
                    const uint4 c = *reinterpret_cast<const uint4 *>(tile + 1024 * j + 32 * lane + 16);
                    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
                    w[4] = c.x; w[5] = c.y; w[6] = c.z; w[7] = c.w;
                } else if (use) {
                    uint32_t a0[4], a1[4];
                    if (kv == 0) ga_block_frags<false>(tile, row, gs, any2, lane, j, a0, a1);
                    else ga_block_frags<true>(tile, row, gs, any2, lane, j, a0, a1);
                    w[0] = a0[0]; w[1] = a0[1]; w[2] = a0[2]; w[3] = a0[3];
                    w[4] = a1[0]; w[5] = a1[1]; w[6] = a1[2]; w[7] = a1[3];
                }
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
            const int q = lane + 32 * k;
            out[q] = *reinterpret_cast<const uint4 *>(stage + (q >> 4) * kStagePitch + (q & 15) * 16);
        }
    }
}

// ---------------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------------
cudaError_t launch_ga_calibrate(int hkv, const uint16_t *raw_pool, int64_t num_raw_pages, const int32_t *pages, int n,
                                uint8_t *bases, uint32_t *status, cudaStream_t stream)
{
    k_ga_calibrate<<<hkv * 8, 256, 0, stream>>>(hkv, raw_pool, num_raw_pages, pages, n, bases, status);
    return cudaGetLastError();
}

cudaError_t launch_ga_encode(const EncodeParams &P, cudaStream_t stream)
{
    cudaError_t e = launch_enc_prepare(P, stream);  // validation and page-size reset
    if (e != cudaSuccess) return e;
    const unsigned items = (unsigned)((size_t)P.n * P.hkv);
    k_ga_sizes<<<items, 256, 0, stream>>>(P);
    e = launch_enc_scan(P, stream);
    if (e != cudaSuccess) return e;
    k_ga_pack<<<items, 256, 0, stream>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_ga_decode(const DecodeParams &P, cudaStream_t stream)
{
    constexpr int smem = kGaDecWarps * 32 * kStagePitch;
    static unsigned long long done = 0;  // bit per device ordinal < 64: shared-memory opt-in
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess && !(dev < 64 && ((__atomic_load_n(&done, __ATOMIC_ACQUIRE) >> dev) & 1ull))) {
        e = cudaFuncSetAttribute(k_ga_decode_w, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess && dev < 64) __atomic_fetch_or(&done, 1ull << dev, __ATOMIC_ACQ_REL);
    }
    if (e != cudaSuccess) return e;
    const int64_t items = (int64_t)P.n * P.hkv, want = (items + kGaDecWarps - 1) / kGaDecWarps;
    const int64_t wave = (int64_t)(sms > 0 ? sms : 1) * 3;
    k_ga_decode_w<<<(unsigned)(want < wave ? (want > 0 ? want : 1) : wave), kGaDecWarps * 32, smem, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace kvz
