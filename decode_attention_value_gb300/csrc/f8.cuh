// f8.cuh -- FP8 KV tiles with group-adaptive exponent coding (GAAC, "Relation to FP8
// KV": the codec applied to KV converted to FP8; "Group-adaptive additive coding" for
// the modes): layout constants, BF16 -> FP8 conversion, and the register restore shared
// by the standalone decoder and the attention kernel.
//
// A tile is one 16-token K or V slice of one KV head (2048 values) in the storage order
// of the 12-bit format; group q = 8L + 2j + f is one lane's fragment.  With M mantissa
// bits (E5M2: 2, E4M3: 3) and S = 1 + M:
//   [0, 256 S)        sign/mantissa fields s << M | m, group q at S*q bytes, element i at
//                     bits S*i.. (E5M2: 3 bits, E4M3: 4 bits)
//   +768              3-bit exponent codes, group q at 3q, element i at bits 3i..3i+2
//   +64               2-bit modes, group q at byte q/4, bits 2(q%4)
//   +64               escapes in q order: mode 1 one byte (bit 3 of code i at bit i),
//                     mode 2 (E5M2) two bytes (bits 3..4 of code i at bits 2i..2i+1)
// Mode 0: e = code + b3[ch]; mode 1: e = code + b4[ch] (E4M3: b4 = 0, whatever the bases
// table holds); mode 2: e = code.
// E5M2 tile 1664 B, E4M3 1920 B; a tile needing more than 64 escape bytes stays raw:
// 2048 FP8 bytes, element (L, f, i) of block j at 512j + 16L + 8f + i.
#pragma once

#include "ga.cuh"

namespace kvz {

enum : int { kF8E4M3 = 1, kF8E5M2 = 2 };

template <bool kE5>
struct F8Layout {
    static constexpr int kM = kE5 ? 2 : 3;               // mantissa bits
    static constexpr int kS = kM + 1;                    // sign/mantissa bits
    static constexpr uint32_t kSmBytes = 256u * kS;      // 768 / 1024
    static constexpr uint32_t kCodeOff = kSmBytes;
    static constexpr uint32_t kTagOff = kCodeOff + 768u;
    static constexpr uint32_t kEscOff = kTagOff + 64u;
    static constexpr uint32_t kEscCap = 64u;
    static constexpr uint32_t kTileBytes = kEscOff + kEscCap;  // 1664 / 1920
    static constexpr uint32_t kRawBytes = 2048u;
    static constexpr uint32_t kEscRaw = kE5 ? 2u : 1u;   // escape bytes of a mode-2 group (unused for E4M3)
};

__host__ __device__ __forceinline__ uint32_t f8_tile_bytes(int fmt) { return fmt == kF8E5M2 ? 1664u : 1920u; }
__host__ __device__ __forceinline__ uint32_t f8_entry_bytes(int fmt, uint32_t entry)
{
    return (entry & kGaEntryRaw) ? 2048u : f8_tile_bytes(fmt);
}

// BF16 pair (low half = first value) -> two FP8 bytes (low byte = first value): nearest,
// ties to even, saturating to the largest finite value; NaN -> sign | 0x7F.
template <bool kE5>
__device__ __forceinline__ uint32_t f8_from_bf16x2(uint32_t w2)
{
    const float lo = __uint_as_float(w2 << 16), hi = __uint_as_float(w2 & 0xFFFF0000u);
    uint16_t r;
    if (kE5) asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    uint32_t out = r;
    if (lo != lo) out = (out & 0xFF00u) | ((w2 >> 8) & 0x80u) | 0x7Fu;
    if (hi != hi) out = (out & 0x00FFu) | (((w2 >> 24) & 0x80u) | 0x7Fu) << 8;
    return out;
}

// Sign/mantissa field of a group -> per-element values s << M | m in bytes (elements 0..3,
// 4..7).  E5M2: 24-bit field of 3-bit values; E4M3: 32-bit field of nibbles.
template <bool kE5>
__device__ __forceinline__ void f8_sm_bytes(uint32_t field, uint32_t &s0, uint32_t &s1)
{
    if (kE5) {
        s0 = ga_spread3(field & 0xFFFu);
        s1 = ga_spread3((field >> 12) & 0xFFFu);
    } else {
        uint32_t z = field & 0xFFFFu;
        z = (z | (z << 8)) & 0x00FF00FFu;
        s0 = (z | (z << 4)) & 0x0F0F0F0Fu;
        z = field >> 16;
        z = (z | (z << 8)) & 0x00FF00FFu;
        s1 = (z | (z << 4)) & 0x0F0F0F0Fu;
    }
}

// FP8 bytes from sign/mantissa bytes and exponent bytes.
template <bool kE5>
__device__ __forceinline__ uint32_t f8_assemble(uint32_t sm, uint32_t e)
{
    constexpr int M = F8Layout<kE5>::kM;
    constexpr uint32_t mmask = kE5 ? 0x03030303u : 0x07070707u;
    constexpr uint32_t smask = kE5 ? 0x04040404u : 0x08080808u;
    return ((sm & smask) << (7 - M)) | (e << M) | (sm & mmask);
}

template <typename Row>
struct RowIsBytes {
    static constexpr bool value = false;
};
template <>
struct RowIsBytes<uint8_t> {
    static constexpr bool value = true;
};

// One group of a compressed tile -> its 8 FP8 bytes (f0: elements 0..3, f1: 4..7).
// Modes 0 and 1 take no branch; raw-exponent groups (E5M2 mode 2) are handled in a
// branch that only tiles holding them enter (any2, warp-uniform).
template <bool kE5, bool kV, typename Row>
__device__ __forceinline__ void f8_restore_group(uint32_t smfield, uint32_t code, uint32_t mode, bool any2,
                                                 const uint8_t *esc, uint32_t &off, const Row *row, int lane,
                                                 int j, int f, uint32_t &f0, uint32_t &f1)
{
    using Lt = F8Layout<kE5>;
    const uint32_t m1 = mode & 1u;
    uint32_t h = 0;
    if (m1) h = esc[min(off, Lt::kEscCap - 1)];
    off += m1;
    uint32_t b0, b1;
    ga_bases<kV>(row, m1, lane, j, f, b0, b1);
    // E4M3: b4 = 0 (the 16-wide window is the whole field); a base table (uint32 words)
    // already holds 0 there, a byte row of the bases table is not read for it
    if (!kE5 && RowIsBytes<Row>::value && m1) b0 = b1 = 0;
    const uint32_t l0 = ga_spread3(code & 0xFFFu), l1 = ga_spread3((code >> 12) & 0xFFFu);
    uint32_t c0 = l0 | ga_spread1_hi(h), c1 = l1 | ga_spread1_hi(h >> 4);
    if (kE5 && any2) {
        if (mode >= 2) {
            const uint8_t *p = esc + min(off, Lt::kEscCap - 2);
            const uint32_t hb = (uint32_t)p[0] | ((uint32_t)p[1] << 8);
            // bits 3..4 of code i sit at bits 2i..2i+1: spread the 2-bit fields to bytes
            uint32_t z0 = hb & 0xFFu, z1 = hb >> 8;
            z0 = (z0 | (z0 << 12)) & 0x000F000Fu;
            z0 = (z0 | (z0 << 6)) & 0x03030303u;
            z1 = (z1 | (z1 << 12)) & 0x000F000Fu;
            z1 = (z1 | (z1 << 6)) & 0x03030303u;
            c0 = l0 | (z0 << 3);
            c1 = l1 | (z1 << 3);
            b0 = b1 = 0;
            off += 2;
        }
    }
    uint32_t s0, s1;
    f8_sm_bytes<kE5>(smfield, s0, s1);
    f0 = f8_assemble<kE5>(s0, c0 + b0);  // byte adds never carry (every e fits its field)
    f1 = f8_assemble<kE5>(s1, c1 + b1);
}

// One compressed tile's per-lane state.
template <bool kE5>
struct F8Lane {
    uint32_t modes, off;
    uint32_t code[6];
    uint32_t sm[8];  // E5M2: 6 words used (24 bytes), E4M3: 8 words (32 bytes)
};

template <bool kE5>
__device__ __forceinline__ uint32_t f8_escapes_of(uint32_t modes16)
{
    return __popc(modes16 & 0x5555u) + (kE5 ? 2u : 1u) * __popc(modes16 & 0xAAAAu);
}

template <bool kE5>
__device__ __forceinline__ F8Lane<kE5> f8_lane_load(const uint8_t *tile, int lane)
{
    using Lt = F8Layout<kE5>;
    F8Lane<kE5> s;
    s.modes = *reinterpret_cast<const uint16_t *>(tile + Lt::kTagOff + 2 * lane);
    const uint32_t cnt = f8_escapes_of<kE5>(s.modes);
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    s.off = incl - cnt;
    const uint2 *c = reinterpret_cast<const uint2 *>(tile + Lt::kCodeOff + 24 * lane);
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const uint2 v = c[k];
        s.code[2 * k] = v.x;
        s.code[2 * k + 1] = v.y;
    }
    if (kE5) {
        const uint2 *m = reinterpret_cast<const uint2 *>(tile + 24 * lane);
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const uint2 v = m[k];
            s.sm[2 * k] = v.x;
            s.sm[2 * k + 1] = v.y;
        }
        s.sm[6] = s.sm[7] = 0;
    } else {
        const uint4 *m = reinterpret_cast<const uint4 *>(tile + 32 * lane);
        const uint4 a = m[0], b = m[1];
        s.sm[0] = a.x; s.sm[1] = a.y; s.sm[2] = a.z; s.sm[3] = a.w;
        s.sm[4] = b.x; s.sm[5] = b.y; s.sm[6] = b.z; s.sm[7] = b.w;
    }
    return s;
}

template <bool kE5>
__device__ __forceinline__ uint32_t f8_sm_field(const F8Lane<kE5> &s, int k)
{
    if (kE5) {  // 24-bit fields packed in six words
        const int bit = 24 * k, wi = bit >> 5, sh = bit & 31;
        const uint32_t lo = s.sm[wi], hi = wi + 1 < 6 ? s.sm[wi + 1] : 0u;
        return __funnelshift_r(lo, hi, sh) & 0xFFFFFFu;
    }
    return s.sm[k];
}

// FP8 bytes of block j (both f) of a compressed tile: f[0..1] fragment 0, f[2..3] fragment 1.
template <bool kE5, bool kV, typename Row>
__device__ __forceinline__ void f8_block_bytes(const uint8_t *tile, const Row *row, F8Lane<kE5> &s, bool any2,
                                               int lane, int j, uint32_t (&fb)[4])
{
    const uint8_t *esc = tile + F8Layout<kE5>::kEscOff;
    const uint32_t m0 = (s.modes >> (4 * j)) & 3u, m1 = (s.modes >> (4 * j + 2)) & 3u;
    f8_restore_group<kE5, kV>(f8_sm_field<kE5>(s, 2 * j), ga_code_field(s.code, 2 * j), m0, any2, esc, s.off, row,
                              lane, j, 0, fb[0], fb[1]);
    f8_restore_group<kE5, kV>(f8_sm_field<kE5>(s, 2 * j + 1), ga_code_field(s.code, 2 * j + 1), m1, any2, esc, s.off,
                              row, lane, j, 1, fb[2], fb[3]);
}

// 16 FP8 bytes of a lane (fragment 0: fb[0..1], fragment 1: fb[2..3]) -> the two f16 A
// fragments (every FP8 value is an f16 value: E5M2 is the high byte of an f16, E4M3 widens
// exactly in hardware).
template <bool kE5>
__device__ __forceinline__ uint32_t f8x2_to_f16x2(uint32_t x)
{
    if (kE5) return __byte_perm(x, 0, 0x1404);
    uint32_t h2;
    const uint16_t a = (uint16_t)x;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(a));
    return h2;
}

template <bool kE5>
__device__ __forceinline__ void f8_frags_f16(const uint32_t (&fb)[4], uint32_t (&a0)[4], uint32_t (&a1)[4])
{
    a0[0] = f8x2_to_f16x2<kE5>(fb[0] & 0xFFFFu);
    a0[1] = f8x2_to_f16x2<kE5>(fb[0] >> 16);
    a0[2] = f8x2_to_f16x2<kE5>(fb[1] & 0xFFFFu);
    a0[3] = f8x2_to_f16x2<kE5>(fb[1] >> 16);
    a1[0] = f8x2_to_f16x2<kE5>(fb[2] & 0xFFFFu);
    a1[1] = f8x2_to_f16x2<kE5>(fb[2] >> 16);
    a1[2] = f8x2_to_f16x2<kE5>(fb[3] & 0xFFFFu);
    a1[3] = f8x2_to_f16x2<kE5>(fb[3] >> 16);
}

}  // namespace kvz
