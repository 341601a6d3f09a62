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

template <bool kE5>
__host__ __device__ __forceinline__ uint32_t f8_granules(uint32_t escapes)
{
    return (escapes <= F8Layout<kE5>::kEscCap ? F8Layout<kE5>::kTileBytes : 2048u) / kGaGranule;
}

// ---------------------------------------------------------------------------------
// Window tests on FP8 exponents, two values per word: an FP8 pair from the conversion is
// spread to 16-bit halves (X = byte 0 | byte 1 << 16), the exponent field Ex = X & emask
// sits at bits M.. of each half, and with the bases spread and shifted the same way each
// half of D = Ex + (256 << M) - (b << M) is (256 + e - b) << M (e <= 31, b <= 255: no
// borrow between halves), so e is in [b, b + 8) exactly when (D & (0x1F8 << M)) == 256 << M
// (0x1F0 << M for [b, b + 16)).  E4M3's 16-wide window is the whole 4-bit field: b4 = 0
// whatever the table holds, so its groups take modes 0 and 1 only.
// ---------------------------------------------------------------------------------
template <bool kE5>
struct F8Win {
    static constexpr int kM = F8Layout<kE5>::kM;
    static constexpr uint32_t kEx = ((kE5 ? 0x1Fu : 0x0Fu) << kM) * 0x00010001u;  // exponent fields
    static constexpr uint32_t kOne = 0x01000100u << kM;
    static constexpr uint32_t kWin8 = 0x01F801F8u << kM, kWin16 = 0x01F001F0u << kM;
};

// nonzero: some half of the four words lies outside its window
template <bool kE5>
__device__ __forceinline__ uint32_t f8_miss4(const uint32_t (&d)[4], uint32_t win)
{
    using W = F8Win<kE5>;
    const uint32_t any = (d[0] | d[1] | d[2] | d[3]) & (win ^ W::kOne);
    const uint32_t all = d[0] & d[1] & d[2] & d[3];
    return any | (~all & W::kOne);
}

// ---------------------------------------------------------------------------------
// size pass: warp per (entry, head) item, the page read in its plain layout as in the
// group-adaptive BF16 encoder (same lane-to-group shuffles); records the granules of the
// pair and the two tiles' escape byte counts for the pack pass.
// ---------------------------------------------------------------------------------
template <bool kE5>
__device__ __forceinline__ uint32_t f8_block_flags(const uint4 &lo, const uint4 &hi, const uint8_t *row)
{
    using W = F8Win<kE5>;
    const uint4 b3 = __ldg(reinterpret_cast<const uint4 *>(row));
    const uint4 b4 = kE5 ? __ldg(reinterpret_cast<const uint4 *>(row + 128)) : make_uint4(0, 0, 0, 0);
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const uint32_t s3[4] = {b3.x, b3.y, b3.z, b3.w}, s4[4] = {b4.x, b4.y, b4.z, b4.w};
    uint32_t p3[4] = {0, 0, 0, 0}, p4[4] = {0, 0, 0, 0};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t x = (enc_spread2(f8_from_bf16x2<kE5>(w[k]), 0) & W::kEx) + W::kOne;
        p3[k & 3] |= ((x - (enc_spread2(s3[k >> 1], k & 1) << W::kM)) & W::kWin8) ^ W::kOne;
        if (kE5) p4[k & 3] |= ((x - (enc_spread2(s4[k >> 1], k & 1) << W::kM)) & W::kWin16) ^ W::kOne;
    }
    // per half: bit 2g (8-wide window missed), 2g+1 (16-wide missed) for words g, g+4;
    // halves are below 0x8000, so adding 0x7FFF sets bit 15 exactly when one is nonzero
    uint32_t m = 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        m |= (((p3[g] + 0x7FFF7FFFu) & 0x80008000u) >> (15 - 2 * g));
        if (kE5) m |= (((p4[g] + 0x7FFF7FFFu) & 0x80008000u) >> (14 - 2 * g));
    }
    return m;  // bits 0..7: low halves; bits 16..23: high halves
}

// escape bytes of the groups in a flag word: mode 1 one byte, mode 2 (E5M2) two
__device__ __forceinline__ uint32_t f8_flag_escapes(uint32_t m)
{
    const uint32_t n3 = m & 0x55555555u, n4 = (m >> 1) & 0x55555555u;
    return __popc(n3) + __popc(n3 & n4);
}

template <bool kE5>
__global__ void __launch_bounds__(256, 3) k_f8_sizes_w(EncodeParams P)
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
            const uint32_t mk = f8_block_flags<kE5>(v[2 * j], v[2 * j + 1], rows + 32 * j);
            fk |= ((mk | (mk >> 16)) & 0xFFu) << (8 * j);  // a K group spans both halves
            const uint32_t mv = f8_block_flags<kE5>(v[8 + 2 * j], v[9 + 2 * j], rows + 256 + 32 * j);
            if (j < 2) fv01 |= mv << (8 * j);
            else fv23 |= mv << (8 * (j - 2));
        }
        fk |= __shfl_xor_sync(0xffffffffu, fk, 16);
        fv01 |= __shfl_xor_sync(0xffffffffu, fv01, 2);
        fv23 |= __shfl_xor_sync(0xffffffffu, fv23, 2);
        fv01 |= __shfl_xor_sync(0xffffffffu, fv01, 16);
        fv23 |= __shfl_xor_sync(0xffffffffu, fv23, 16);
        // each group counted once: K by the lanes of tokens 0..7, V by those of tokens 0, 2, 4, 6
        const uint32_t eK = __reduce_add_sync(0xffffffffu, lane < 16 ? f8_flag_escapes(fk) : 0u);
        const uint32_t eV =
            __reduce_add_sync(0xffffffffu, (lane & 18) == 0 ? f8_flag_escapes(fv01) + f8_flag_escapes(fv23) : 0u);
        if (lane == 0) {
            const uint32_t g = f8_granules<kE5>(eK) + f8_granules<kE5>(eV);
            P.ws_pair_size[it] = g;
            atomicAdd(P.ws_page_size + entry, g);  // integer sum: the same whatever the order
            P.ws_tags[it] = eK | ((uint64_t)eV << 32);
        }
    }
}

// ---------------------------------------------------------------------------------
// pack pass: warp per (entry, head) item; the warp stages the BF16 slice, gathers each
// block in storage order, converts it, picks each group's mode, writes the sign/mantissa
// fields straight to the arena and assembles codes, modes and escapes in shared memory.
// Raw tiles get the FP8 bytes in storage order.
// ---------------------------------------------------------------------------------
constexpr int kF8PackWarps = 8;
constexpr int kF8AuxBytes = 768 + 64 + 64;  // codes, modes, escapes
constexpr int kF8PackWarpSmem = 32 * kStagePitch + kF8AuxBytes;
constexpr int kF8PackSmem = kF8PackWarps * kF8PackWarpSmem;
static_assert(kF8PackWarpSmem % 16 == 0 && kF8AuxBytes % 16 == 0, "16-byte staging");

// the eight FP8 bytes of a gathered fragment (storage order) from its four bf16x2 words
template <bool kE5>
__device__ __forceinline__ void f8_convert_frag(const uint32_t *w, uint32_t (&r)[4], uint32_t &f0, uint32_t &f1)
{
#pragma unroll
    for (int k = 0; k < 4; ++k) r[k] = f8_from_bf16x2<kE5>(w[k]);
    f0 = __byte_perm(r[0], r[1], 0x5410);
    f1 = __byte_perm(r[2], r[3], 0x5410);
}

// sign | mantissa of four FP8 bytes: E4M3 4-bit fields (16 bits), E5M2 3-bit (12 bits)
template <bool kE5>
__device__ __forceinline__ uint32_t f8_sm4(uint32_t fb)
{
    if (kE5) {
        const uint32_t n = ((fb >> 5) & 0x04040404u) | (fb & 0x03030303u);
        const uint32_t t = (n | (n >> 5)) & 0x003F003Fu;
        return (t | (t >> 10)) & 0xFFFu;
    } else {
        const uint32_t n = ((fb >> 4) & 0x08080808u) | (fb & 0x07070707u);
        const uint32_t t = (n | (n >> 4)) & 0x00FF00FFu;
        return __byte_perm(t, 0, 0x4420);
    }
}

template <bool kE5, bool kV>
__device__ __forceinline__ void f8_pack_tile(const uint8_t *stage, uint8_t *aux, const uint8_t *row, int lane,
                                             uint8_t *tile)
{
    using Lt = F8Layout<kE5>;
    using W = F8Win<kE5>;
    constexpr int kM = W::kM;
    // this lane's eight groups q = 2 j + f: codes (24 bits each) fill six words; E5M2
    // sign/mantissa fields (24 bits each) likewise; escape fields 8 (mode 1) or 16 bits
    uint32_t modes = 0, cnt = 0, cw[6] = {0, 0, 0, 0, 0, 0}, smw[6] = {0, 0, 0, 0, 0, 0}, esc16[4] = {0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t w[8];
        gather_block(stage, kV ? 1 : 0, j, lane, w);
        uint32_t sm4[2];
#pragma unroll
        for (int f = 0; f < 2; ++f) {
            const int q = 2 * j + f;
            uint32_t r[4], fb0, fb1;
            f8_convert_frag<kE5>(w + 4 * f, r, fb0, fb1);
            // bases (shifted) of words 0..3: K [A, A, C, C], V [A, C, A, C]
            uint32_t A3, C3, A4 = 0, C4 = 0;
            if (!kV) {
                const uint8_t *p = row + 32 * j + 16 * f + 2 * (lane & 3);
                A3 = enc_spread2(__ldg(reinterpret_cast<const uint16_t *>(p)), 0) << kM;
                C3 = enc_spread2(__ldg(reinterpret_cast<const uint16_t *>(p + 8)), 0) << kM;
                if (kE5) {
                    A4 = enc_spread2(__ldg(reinterpret_cast<const uint16_t *>(p + 128)), 0) << kM;
                    C4 = enc_spread2(__ldg(reinterpret_cast<const uint16_t *>(p + 136)), 0) << kM;
                }
            } else {
                const uint8_t *p = row + 32 * j + 16 * f + (lane >> 2);
                A3 = __ldg(p) * (0x00010001u << kM);
                C3 = __ldg(p + 8) * (0x00010001u << kM);
                if (kE5) {
                    A4 = __ldg(p + 128) * (0x00010001u << kM);
                    C4 = __ldg(p + 136) * (0x00010001u << kM);
                }
            }
            uint32_t Ex[4], D3[4], D4[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const bool second = kV ? (k & 1) : (k >> 1);
                Ex[k] = enc_spread2(r[k], 0) & W::kEx;
                D3[k] = Ex[k] + W::kOne - (second ? C3 : A3);
                D4[k] = Ex[k] + W::kOne - (second ? C4 : A4);
            }
            uint32_t mode = f8_miss4<kE5>(D3, W::kWin8) == 0 ? 0u : 1u;
            if (kE5 && mode == 1 && f8_miss4<kE5>(D4, W::kWin16) != 0) mode = 2;
            modes |= mode << (2 * q);
            cnt += mode == 0 ? 0u : (mode == 1 ? 1u : 2u);
            // sign/mantissa fields
            const uint32_t smf = f8_sm4<kE5>(fb0) | (f8_sm4<kE5>(fb1) << (kE5 ? 12 : 16));
            if (kE5) {
                const int bit = 24 * q, wi = bit >> 5, sh = bit & 31;
                smw[wi] |= smf << sh;
                if (sh > 8) smw[wi + 1] |= smf >> (32 - sh);
            } else {
                sm4[f] = smf;
            }
            // codes: the low three bits of e - base (bits M..M+2 of each half of the mode's
            // D; base 0 for raw groups), value i at bits 3i of the 24-bit field
            const uint32_t As = mode == 0 ? A3 : (mode == 1 ? A4 : 0u), Cs = mode == 0 ? C3 : (mode == 1 ? C4 : 0u);
            uint32_t t[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const bool second = kV ? (k & 1) : (k >> 1);
                t[k] = (Ex[k] + W::kOne - (second ? Cs : As)) & (0x00070007u << kM);
            }
            const uint32_t p01 = t[0] + t[1] * 64u, p23 = t[2] + t[3] * 64u;
            const uint32_t u01 = (p01 | (p01 >> 13)) & (0xFFFu << kM), u23 = (p23 | (p23 >> 13)) & (0xFFFu << kM);
            const uint32_t field = (u01 >> kM) + (u23 << (12 - kM));
            const int bit = 24 * q, wi = bit >> 5, sh = bit & 31;
            cw[wi] |= field << sh;
            if (sh > 8) cw[wi + 1] |= field >> (32 - sh);
            uint32_t e = 0;
            if (mode == 1) {  // bit 3 of e - b4 of each value (bit M+3 of each half of D4)
                constexpr uint32_t m = 0x00080008u << kM;
                const uint32_t s01 = (D4[0] & m) + (D4[1] & m) * 4u, s23 = (D4[2] & m) + (D4[3] & m) * 4u;
                const uint32_t v01 = (s01 | (s01 >> 15)) & (0xFu << (kM + 3));
                const uint32_t v23 = (s23 | (s23 >> 15)) & (0xFu << (kM + 3));
                e = (v01 + (v23 << 4)) >> (kM + 3);
            } else if (kE5 && mode == 2) {  // bits 3..4 of e of each value at bits 2i..2i+1
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    e |= (((Ex[k] >> (kM + 3)) & 3u) | ((Ex[k] >> (kM + 17)) & 0xCu)) << (4 * k);
            }
            esc16[q >> 1] |= e << (16 * (q & 1));
        }
        if (!kE5) *reinterpret_cast<uint2 *>(tile + 32 * lane + 8 * j) = make_uint2(sm4[0], sm4[1]);
    }
    if (kE5) {
        uint2 *s2 = reinterpret_cast<uint2 *>(tile + 24 * lane);
        s2[0] = make_uint2(smw[0], smw[1]);
        s2[1] = make_uint2(smw[2], smw[3]);
        s2[2] = make_uint2(smw[4], smw[5]);
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
    *reinterpret_cast<uint16_t *>(aux + 768 + 2 * lane) = (uint16_t)modes;
    uint8_t *esc = aux + 768 + 64;
    if (lane < (int)(Lt::kEscCap / 16)) reinterpret_cast<uint4 *>(esc)[lane] = make_uint4(0, 0, 0, 0);
    __syncwarp();
    if (total <= Lt::kEscCap) {  // the size pass found the same total; never past the area
        uint32_t off = incl - cnt;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint32_t m = (modes >> (2 * q)) & 3u;
            const uint32_t e = (esc16[q >> 1] >> (16 * (q & 1))) & 0xFFFFu;
            if (m == 1) {
                esc[off] = (uint8_t)e;
                off += 1;
            } else if (kE5 && m == 2) {
                esc[off] = (uint8_t)e;
                esc[off + 1] = (uint8_t)(e >> 8);
                off += 2;
            }
        }
    }
    __syncwarp();
    uint4 *dst = reinterpret_cast<uint4 *>(tile + Lt::kCodeOff);
    const uint4 *src = reinterpret_cast<const uint4 *>(aux);
    for (int k = lane; k < kF8AuxBytes / 16; k += 32) dst[k] = src[k];
}

template <bool kE5>
__global__ void __launch_bounds__(kF8PackWarps * 32, 2) k_f8_pack_w(EncodeParams P)
{
    extern __shared__ __align__(16) uint8_t f8_pack_smem[];
    if (P.ws_hdr[0] != 0) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *stage = f8_pack_smem + warp * kF8PackWarpSmem;
    uint8_t *aux = stage + 32 * kStagePitch;
    const int64_t items = (int64_t)P.n * P.hkv;
    const int64_t stride = (int64_t)gridDim.x * kF8PackWarps;
    for (int64_t it = (int64_t)blockIdx.x * kF8PackWarps + warp; it < items; it += stride) {
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
        const uint64_t esc = P.ws_tags[it];
        const uint32_t gK = f8_granules<kE5>((uint32_t)esc), gV = f8_granules<kE5>((uint32_t)(esc >> 32));
        const bool compK = (uint32_t)esc <= F8Layout<kE5>::kEscCap;
        const bool compV = (uint32_t)(esc >> 32) <= F8Layout<kE5>::kEscCap;
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
                if (kv == 0) f8_pack_tile<kE5, false>(stage, aux, row, lane, tile);
                else f8_pack_tile<kE5, true>(stage, aux, row + 256, lane, tile);
            } else if (fit) {  // raw: the FP8 bytes in storage order, 16 per lane per block
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {
                    uint32_t w[8], r[4], fb[4];
                    gather_block(stage, kv, j, lane, w);
                    f8_convert_frag<kE5>(w, r, fb[0], fb[1]);
                    f8_convert_frag<kE5>(w + 4, r, fb[2], fb[3]);
                    *reinterpret_cast<uint4 *>(tile + 512 * j + 16 * lane) = make_uint4(fb[0], fb[1], fb[2], fb[3]);
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
    static unsigned long long done = 0;  // bit per device ordinal < 64: shared-memory opt-in
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess && !(dev < 64 && ((__atomic_load_n(&done, __ATOMIC_ACQUIRE) >> dev) & 1ull))) {
        e = cudaFuncSetAttribute(k_f8_pack_w<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kF8PackSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_f8_pack_w<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kF8PackSmem);
        if (e == cudaSuccess && dev < 64) __atomic_fetch_or(&done, 1ull << dev, __ATOMIC_ACQ_REL);
    }
    if (e != cudaSuccess) return e;
    e = launch_enc_prepare(P, stream);  // validation and page-size reset
    if (e != cudaSuccess) return e;
    const int64_t items = (int64_t)P.n * P.hkv;
    if (fmt == kF8E5M2) k_f8_sizes_w<true><<<enc_warp_grid(items, sms, 3), 256, 0, stream>>>(P);
    else k_f8_sizes_w<false><<<enc_warp_grid(items, sms, 3), 256, 0, stream>>>(P);
    e = launch_enc_scan(P, stream);
    if (e != cudaSuccess) return e;
    const unsigned grid = enc_warp_grid(items, sms, 2);
    if (fmt == kF8E5M2) k_f8_pack_w<true><<<grid, kF8PackWarps * 32, kF8PackSmem, stream>>>(P);
    else k_f8_pack_w<false><<<grid, kF8PackWarps * 32, kF8PackSmem, stream>>>(P);
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
