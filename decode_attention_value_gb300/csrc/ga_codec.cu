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
// Window tests, two values at a time.  With the exponents of a bf16x2 word spread to
// 16-bit halves, X = (w >> 7) & 0x00FF00FF, and the bases spread the same way, each half
// of D = X + 0x0100 - B is 256 + e - b in [1, 511] (no borrow between halves), and e lies
// in [b, b + 8) exactly when (D & 0x1F8) == 0x100 (0x1F0 for [b, b + 16)).
// ---------------------------------------------------------------------------------
constexpr uint32_t kGaHalfOne = 0x01000100u, kGaWin8 = 0x01F801F8u, kGaWin16 = 0x01F001F0u;

__device__ __forceinline__ uint32_t ga_exp2(uint32_t w) { return (w >> 7) & 0x00FF00FFu; }
// nonzero half: that value is outside the window
__device__ __forceinline__ uint32_t ga_viol(uint32_t d, uint32_t win) { return (d & win) ^ kGaHalfOne; }

// ---------------------------------------------------------------------------------
// size pass: warp per (entry, head) item in a grid-stride loop.  The page slice is read in
// its plain layout (lane = token lane/2, channels 16*(lane%2)..+16 of each block), the
// window tests run on bf16x2 words, and each storage-order group (lane', f) is gathered
// from the lanes that hold it with shuffles: a K group is channels {c, c+1, c+8, c+9} of
// tokens r and r+8 (words c/2 and c/2+4 of lanes 2r+f and 2r+f+16); a V group is channels
// r and r+8 (one half of words r/2 and r/2+4) of tokens c, c+1, c+8, c+9 (lanes 2c+f
// xor 0, 2, 16, 18).  It records the granules of the pair and the two tiles' escape
// byte counts for the pack pass.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ga_block_flags(const uint4 &lo, const uint4 &hi, const uint8_t *row)
{
    // row: the block's 16 channels of this lane in the b3 table; b4 is 128 bytes on
    const uint4 b3 = __ldg(reinterpret_cast<const uint4 *>(row));
    const uint4 b4 = __ldg(reinterpret_cast<const uint4 *>(row + 128));
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const uint32_t s3[4] = {b3.x, b3.y, b3.z, b3.w}, s4[4] = {b4.x, b4.y, b4.z, b4.w};
    uint32_t p3[4] = {0, 0, 0, 0}, p4[4] = {0, 0, 0, 0};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t x = ga_exp2(w[k]) + kGaHalfOne;
        p3[k & 3] |= ga_viol(x - enc_spread2(s3[k >> 1], k & 1), kGaWin8);
        p4[k & 3] |= ga_viol(x - enc_spread2(s4[k >> 1], k & 1), kGaWin16);
    }
    // per half: bit 2g (8-wide window missed) and 2g+1 (16-wide missed) for words g, g+4;
    // halves are <= 0x1F8, so adding 0x7FFF sets bit 15 exactly when one is nonzero
    uint32_t m = 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        m |= (((p3[g] + 0x7FFF7FFFu) & 0x80008000u) >> (15 - 2 * g));
        m |= (((p4[g] + 0x7FFF7FFFu) & 0x80008000u) >> (14 - 2 * g));
    }
    return m;  // bits 0..7: low halves; bits 16..23: high halves
}

// escape bytes of the groups in a flag word (bit 2g: 8-wide missed, 2g+1: 16-wide missed):
// 0 for the 3-bit mode, 1 for the 4-bit mode, 5 for raw groups
__device__ __forceinline__ uint32_t ga_flag_escapes(uint32_t m)
{
    const uint32_t n3 = m & 0x55555555u, n4 = (m >> 1) & 0x55555555u;
    return __popc(n3) + 4 * __popc(n3 & n4);
}

__global__ void __launch_bounds__(256, 3) k_ga_sizes_w(EncodeParams P)
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
        const uint8_t *rows = P.ga_bases + (size_t)head * 512 + 16 * (lane & 1);
        uint32_t fk = 0, fv01 = 0, fv23 = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t mk = ga_block_flags(v[2 * j], v[2 * j + 1], rows + 32 * j);
            fk |= ((mk | (mk >> 16)) & 0xFFu) << (8 * j);  // a K group spans both halves
            const uint32_t mv = ga_block_flags(v[8 + 2 * j], v[9 + 2 * j], rows + 256 + 32 * j);
            if (j < 2) fv01 |= mv << (8 * j);
            else fv23 |= mv << (8 * (j - 2));
        }
        fk |= __shfl_xor_sync(0xffffffffu, fk, 16);
        fv01 |= __shfl_xor_sync(0xffffffffu, fv01, 2);
        fv23 |= __shfl_xor_sync(0xffffffffu, fv23, 2);
        fv01 |= __shfl_xor_sync(0xffffffffu, fv01, 16);
        fv23 |= __shfl_xor_sync(0xffffffffu, fv23, 16);
        // each group counted once: K by the lanes of tokens 0..7, V by those of tokens 0, 2, 4, 6
        const uint32_t eK = __reduce_add_sync(0xffffffffu, lane < 16 ? ga_flag_escapes(fk) : 0u);
        const uint32_t eV =
            __reduce_add_sync(0xffffffffu, (lane & 18) == 0 ? ga_flag_escapes(fv01) + ga_flag_escapes(fv23) : 0u);
        if (lane == 0) {
            const uint32_t g = (eK <= kGaEscCap ? kGaTileBytes : kGaRawBytes) / kGaGranule +
                               (eV <= kGaEscCap ? kGaTileBytes : kGaRawBytes) / kGaGranule;
            P.ws_pair_size[it] = g;
            atomicAdd(P.ws_page_size + entry, g);  // integer sum: the same whatever the order
            P.ws_tags[it] = eK | ((uint64_t)eV << 32);
        }
    }
}

// ---------------------------------------------------------------------------------
// pack pass: warp per (entry, head) item.  The warp stages the slice in its own shared
// buffer, gathers each block in storage order, and per group (lane, f) picks the mode,
// writes the sign/mantissa bytes straight to the arena and keeps the 3-bit codes and the
// escape bits in registers; after a warp scan of the escape bytes (lane-major group
// order) the code, mode and escape areas are assembled in shared memory and copied out.
// Raw tiles are written from the gathered words.
// ---------------------------------------------------------------------------------
constexpr int kGaPackWarps = 8;
constexpr int kGaAuxBytes = (int)(kGaTileBytes - kGaCodeOff);  // 960: codes, modes, escapes
constexpr int kGaPackWarpSmem = 32 * kStagePitch + kGaAuxBytes;
constexpr int kGaPackSmem = kGaPackWarps * kGaPackWarpSmem;
static_assert(kGaPackWarpSmem % 16 == 0 && kGaAuxBytes % 16 == 0, "16-byte staging");

// In the pack pass the window tests run on the exponents in place: with Ex = w & 0x7F807F80
// and the bases shifted the same way (b << 7 in each half), D = Ex + 0x80008000 - B holds
// (256 + e - b) << 7 per half, so e - b is bits 7.. of each half and e is in [b, b + 8)
// exactly when (D & 0xFC00) == 0x8000 (0xF800 for [b, b + 16)).
constexpr uint32_t kGaExMask = 0x7F807F80u, kGaHalfOneS = 0x80008000u;
constexpr uint32_t kGaWin8S = 0xFC00FC00u, kGaWin16S = 0xF800F800u;

// nonzero: some half of the four words lies outside its window
__device__ __forceinline__ uint32_t ga_miss4(const uint32_t (&d)[4], uint32_t win)
{
    const uint32_t any = (d[0] | d[1] | d[2] | d[3]) & (win ^ kGaHalfOneS);  // a bit that must be clear
    const uint32_t all = d[0] & d[1] & d[2] & d[3];                            // the bit that must be set
    return any | (~all & kGaHalfOneS);
}

template <bool kV>
__device__ __forceinline__ void ga_pack_tile(const uint8_t *stage, uint8_t *aux, const uint8_t *row, int lane,
                                             uint8_t *tile)
{
    // codes: group q = 8 lane + 2 j + f at bytes 3q..3q+2, so this lane's eight 24-bit
    // fields fill six words; escape bits per group (the fifth byte of raw groups in ehi)
    uint32_t modes = 0, cnt = 0, cw[6] = {0, 0, 0, 0, 0, 0}, elo[8], ehi[2] = {0, 0};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t w[8];
        gather_block(stage, kV ? 1 : 0, j, lane, w);
        uint32_t sfw[4];
#pragma unroll
        for (int f = 0; f < 2; ++f) {
            const int q = 2 * j + f;
            // bases (shifted) of words 0..3: K [A, A, C, C] (channels c, c+1 | c+8, c+9);
            // V [A, C, A, C] (channel r | r+8, both halves)
            uint32_t A3, C3, A4, C4;
            if (!kV) {
                const uint8_t *p = row + 32 * j + 16 * f + 2 * (lane & 3);
                A3 = enc_spread2(__ldg(reinterpret_cast<const uint16_t *>(p)), 0) << 7;
                C3 = enc_spread2(__ldg(reinterpret_cast<const uint16_t *>(p + 8)), 0) << 7;
                A4 = enc_spread2(__ldg(reinterpret_cast<const uint16_t *>(p + 128)), 0) << 7;
                C4 = enc_spread2(__ldg(reinterpret_cast<const uint16_t *>(p + 136)), 0) << 7;
            } else {
                const uint8_t *p = row + 32 * j + 16 * f + (lane >> 2);
                A3 = __ldg(p) * 0x00800080u;
                C3 = __ldg(p + 8) * 0x00800080u;
                A4 = __ldg(p + 128) * 0x00800080u;
                C4 = __ldg(p + 136) * 0x00800080u;
            }
            uint32_t Ex[4], D3[4], D4[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const bool second = kV ? (k & 1) : (k >> 1);
                Ex[k] = w[4 * f + k] & kGaExMask;
                D3[k] = Ex[k] + kGaHalfOneS - (second ? C3 : A3);
                D4[k] = Ex[k] + kGaHalfOneS - (second ? C4 : A4);
            }
            const uint32_t mode = ga_miss4(D3, kGaWin8S) == 0 ? 0u : (ga_miss4(D4, kGaWin16S) == 0 ? 1u : 2u);
            modes |= mode << (2 * q);
            cnt += mode == 0 ? 0u : (mode == 1 ? 1u : 5u);
            // sign | 7 mantissa bits per value: the low bytes with bit 7 from the sign-replicated high bytes
            const uint32_t *wf = w + 4 * f;
            sfw[2 * f] = (prmt_b32(wf[0], wf[1], 0x6420) & 0x7F7F7F7Fu) | (prmt_b32(wf[0], wf[1], 0xFDB9) & 0x80808080u);
            sfw[2 * f + 1] = (prmt_b32(wf[2], wf[3], 0x6420) & 0x7F7F7F7Fu) | (prmt_b32(wf[2], wf[3], 0xFDB9) & 0x80808080u);
            // codes: the low three bits of e - base (bits 7..9 of each half of the mode's D;
            // base 0 for raw groups), value i at bits 3i of the 24-bit field
            const uint32_t As = mode == 0 ? A3 : (mode == 1 ? A4 : 0u), Cs = mode == 0 ? C3 : (mode == 1 ? C4 : 0u);
            uint32_t t[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const bool second = kV ? (k & 1) : (k >> 1);
                t[k] = (Ex[k] + kGaHalfOneS - (second ? Cs : As)) & 0x03800380u;
            }
            // pairs of words: values 2k, 2k+2 at bits 7, 13 and 2k+1, 2k+3 at 23, 29; then
            // the high half folded down next to the low one -> four values at bits 7..18
            const uint32_t p01 = t[0] + t[1] * 64u, p23 = t[2] + t[3] * 64u;
            const uint32_t u01 = (p01 | (p01 >> 13)) & 0x7FF80u, u23 = (p23 | (p23 >> 13)) & 0x7FF80u;
            const uint32_t field = (u01 >> 7) + (u23 << 5);
            uint32_t lo = 0, hi = 0;
            if (mode == 1) {  // bit 3 of e - b4 of each value (bits 10 and 26 of D4)
                const uint32_t s01 = (D4[0] & 0x04000400u) + (D4[1] & 0x04000400u) * 4u;
                const uint32_t s23 = (D4[2] & 0x04000400u) + (D4[3] & 0x04000400u) * 4u;
                const uint32_t v01 = (s01 | (s01 >> 15)) & 0x3C00u, v23 = (s23 | (s23 >> 15)) & 0x3C00u;
                lo = (v01 + (v23 << 4)) >> 10;
            } else if (mode == 2) {  // e >> 3 of each value, 5 bits each (bits 10..14 and 26..30 of Ex)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t u = ((Ex[k] >> 10) & 0x1Fu) | ((Ex[k] >> 21) & 0x3E0u);
                    lo |= u << (10 * k);
                    if (k == 3) hi = u >> 2;
                }
            }
            const int bit = 24 * q, wi = bit >> 5, sh = bit & 31;
            cw[wi] |= field << sh;
            if (sh > 8) cw[wi + 1] |= field >> (32 - sh);
            elo[q] = lo;
            ehi[q >> 2] |= hi << (8 * (q & 3));
        }
        *reinterpret_cast<uint4 *>(tile + 512 * j + 16 * lane) = make_uint4(sfw[0], sfw[1], sfw[2], sfw[3]);
    }
    // escape bytes in lane-major group order
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
    __syncwarp();  // the previous tile's copy-out is done with aux
    uint2 *c2 = reinterpret_cast<uint2 *>(aux + 24 * lane);
    c2[0] = make_uint2(cw[0], cw[1]);
    c2[1] = make_uint2(cw[2], cw[3]);
    c2[2] = make_uint2(cw[4], cw[5]);
    *reinterpret_cast<uint16_t *>(aux + (kGaTagOff - kGaCodeOff) + 2 * lane) = (uint16_t)modes;
    uint8_t *esc = aux + (kGaEscOff - kGaCodeOff);
    if (lane < (int)(kGaEscCap / 16)) reinterpret_cast<uint4 *>(esc)[lane] = make_uint4(0, 0, 0, 0);
    __syncwarp();
    if (total <= kGaEscCap) {  // the size pass found the same total; never past the area
        uint32_t off = incl - cnt;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint32_t m = (modes >> (2 * q)) & 3u;
            if (m == 1) {
                esc[off] = (uint8_t)elo[q];
                off += 1;
            } else if (m == 2) {
                esc[off] = (uint8_t)elo[q];
                esc[off + 1] = (uint8_t)(elo[q] >> 8);
                esc[off + 2] = (uint8_t)(elo[q] >> 16);
                esc[off + 3] = (uint8_t)(elo[q] >> 24);
                esc[off + 4] = (uint8_t)(ehi[q >> 2] >> (8 * (q & 3)));
                off += 5;
            }
        }
    }
    __syncwarp();
    uint4 *dst = reinterpret_cast<uint4 *>(tile + kGaCodeOff);
    const uint4 *src = reinterpret_cast<const uint4 *>(aux);
    for (int k = lane; k < kGaAuxBytes / 16; k += 32) dst[k] = src[k];
}

__global__ void __launch_bounds__(kGaPackWarps * 32, 2) k_ga_pack_w(EncodeParams P)
{
    extern __shared__ __align__(16) uint8_t ga_pack_smem[];
    if (P.ws_hdr[0] != 0) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *stage = ga_pack_smem + warp * kGaPackWarpSmem;
    uint8_t *aux = stage + 32 * kStagePitch;
    const int64_t items = (int64_t)P.n * P.hkv;
    const int64_t stride = (int64_t)gridDim.x * kGaPackWarps;
    for (int64_t it = (int64_t)blockIdx.x * kGaPackWarps + warp; it < items; it += stride) {
        const int entry = (int)(it / P.hkv), head = (int)(it % P.hkv);
        const int src = P.src_page[entry], dst = P.dst_page[entry], seq = P.dst_seq[entry];
        // the heads before this one in the page: one load per lane, then a warp sum
        const uint32_t ps = lane < head ? P.ws_pair_size[(int64_t)entry * P.hkv + lane] : 0u;
        const uint4 *s4 = reinterpret_cast<const uint4 *>(P.raw_pool + ((int64_t)src * P.hkv + head) * 2 * kPage * kDim);
        uint4 v[8];  // the slice in two halves (K rows, then V rows)
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = s4[lane + 32 * k];
        uint32_t before_heads = __reduce_add_sync(0xffffffffu, ps);
        for (int h = 32; h < head; ++h) before_heads += P.ws_pair_size[(int64_t)entry * P.hkv + h];
        __syncwarp();  // the previous item's gathers are done with the buffer
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            if (half) {
#pragma unroll
                for (int k = 0; k < 8; ++k) v[k] = s4[lane + 32 * (k + 8)];
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int q = lane + 32 * (k + 8 * half);  // 16-byte chunk q -> row q/16, byte (q%16)*16
                *reinterpret_cast<uint4 *>(stage + (q >> 4) * kStagePitch + (q & 15) * 16) = v[k];
            }
        }
        __syncwarp();
        const uint64_t esc = P.ws_tags[it];
        const bool compK = (uint32_t)esc <= kGaEscCap, compV = (uint32_t)(esc >> 32) <= kGaEscCap;
        const uint32_t gK = (compK ? kGaTileBytes : kGaRawBytes) / kGaGranule;
        const uint32_t gV = (compV ? kGaTileBytes : kGaRawBytes) / kGaGranule;
        const uint64_t pair_base = (uint64_t)P.ws_page_base[entry] + before_heads;
        uint64_t end = min((uint64_t)P.cursors[2 * seq + 1], P.arena_bytes / kGaGranule);
        end = min(end, (uint64_t)kGaOffsetMask);
        const uint8_t *row = P.ga_bases + (size_t)head * 512;
#pragma unroll 1
        for (int kv = 0; kv < 2; ++kv) {
            const uint64_t o = pair_base + (kv ? gK : 0);
            const bool comp = kv ? compV : compK;
            const bool fit = o + (kv ? gV : gK) <= end;
            uint8_t *tile = P.arena + o * kGaGranule;
            if (fit && comp) {
                if (kv == 0) ga_pack_tile<false>(stage, aux, row, lane, tile);
                else ga_pack_tile<true>(stage, aux, row + 256, lane, tile);
            } else if (fit) {
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {
                    uint32_t w[8];
                    gather_block(stage, kv, j, lane, w);
                    uint8_t *blk = tile + 1024 * j;
                    *reinterpret_cast<uint4 *>(blk + 32 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4 *>(blk + 32 * lane + 16) = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
            if (lane == 0) {
                P.meta32[((int64_t)dst * P.hkv + head) * 2 + kv] =
                    fit ? ((uint32_t)o | (comp ? 0u : kGaEntryRaw)) : kGaEntryInvalid;
                if (!fit) atomicOr(P.status, KVZ_STATUS_ARENA_FULL);
            }
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
    static unsigned long long done = 0;  // bit per device ordinal < 64: shared-memory opt-in
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess && !(dev < 64 && ((__atomic_load_n(&done, __ATOMIC_ACQUIRE) >> dev) & 1ull))) {
        e = cudaFuncSetAttribute(k_ga_pack_w, cudaFuncAttributeMaxDynamicSharedMemorySize, kGaPackSmem);
        if (e == cudaSuccess && dev < 64) __atomic_fetch_or(&done, 1ull << dev, __ATOMIC_ACQ_REL);
    }
    if (e != cudaSuccess) return e;
    e = launch_enc_prepare(P, stream);  // validation and page-size reset
    if (e != cudaSuccess) return e;
    const int64_t items = (int64_t)P.n * P.hkv;
    k_ga_sizes_w<<<enc_warp_grid(items, sms, 3), 256, 0, stream>>>(P);
    e = launch_enc_scan(P, stream);
    if (e != cudaSuccess) return e;
    k_ga_pack_w<<<enc_warp_grid(items, sms, 2), kGaPackWarps * 32, kGaPackSmem, stream>>>(P);
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
