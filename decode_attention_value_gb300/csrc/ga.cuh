// ga.cuh -- group-adaptive additive tiles (GAAC, "Lossless KV Compression":
// "Contiguous exponent concentration", "Group-adaptive additive coding"; Table 9
// "Storage"): layout constants and the register restore shared by the standalone
// decoder and the attention kernel.
//
// A tile is one 16-token K or V page slice of one KV head (2048 values) in the
// storage order of the 12-bit format: element (lane L, fragment f, i) of 512-value
// block j.  Group q = 8L + 2j + f is one lane's fragment, so each lane restores its
// own tensor-core operands from its own groups.
//   [0, 2048)     sign/fraction bytes (sign << 7 | 7 fraction bits) at 512j + 16L + 8f + i
//   [2048, 2816)  3-bit codes, group q at 2048 + 3q (element i at bits 3i..3i+2)
//   [2816, 2880)  2-bit modes, group q at byte 2816 + q/4, bits 2(q%4)
//   [2880, 3008)  escape bytes of the wide groups in q order (4-bit mode: one byte,
//                 bit i = bit 3 of code i; raw mode: five bytes, code bits 3..7 of
//                 element i at bits 5i..5i+4), zero padded
// Mode 0: e = code + b3[channel]; mode 1: e = code + b4[channel]; mode 2: e = code.
// A tile whose escape bytes exceed 128 is stored raw (4096 bytes of BF16 words in
// storage order, as a raw 12-bit block group).
#pragma once

#include "kvz_device.cuh"

namespace kvz {

constexpr uint32_t kGaGranule = 64;
constexpr uint32_t kGaTileBytes = 3008, kGaRawBytes = 4096;
constexpr uint32_t kGaCodeOff = 2048, kGaTagOff = 2816, kGaEscOff = 2880, kGaEscCap = 128;
constexpr uint32_t kGaEntryRaw = 0x80000000u, kGaEntryInvalid = 0xFFFFFFFFu, kGaOffsetMask = 0x7FFFFFFFu;

__host__ __device__ __forceinline__ uint32_t ga_entry_bytes(uint32_t entry)
{
    return (entry & kGaEntryRaw) ? kGaRawBytes : kGaTileBytes;
}

// Four 3-bit fields at bits 3k of v (v < 2^12) -> byte k.
__device__ __forceinline__ uint32_t ga_spread3(uint32_t v)
{
    const uint32_t z = (v | (v << 10)) & 0x003F003Fu;
    return (z | (z << 5)) & 0x07070707u;
}

// Four 5-bit fields at bits 5k of v (v < 2^20) -> bits 3..7 of byte k.
__device__ __forceinline__ uint32_t ga_spread5_hi(uint32_t v)
{
    uint32_t z = (v & 0x3FFu) | ((v << 6) & 0x03FF0000u);
    z = (z & 0x001F001Fu) | ((z << 3) & 0x1F001F00u);
    return z << 3;
}

// Four bits of h (bit k) -> bit 3 of byte k.
__device__ __forceinline__ uint32_t ga_spread1_hi(uint32_t h) { return ((h & 0xFu) * 0x01020408u) & 0x08080808u; }

// Offset (from the escape area) of this lane's first escape byte: an exclusive warp
// scan of the escape bytes of each lane's eight groups.  Warp-collective.
__device__ __forceinline__ uint32_t ga_lane_escape_base(uint32_t modes16, int lane)
{
    const uint32_t cnt = __popc(modes16 & 0x5555u) + 5u * __popc(modes16 & 0xAAAAu);
    uint32_t incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    return incl - cnt;
}

// Per-element bases of one group as two byte vectors (elements 0..3, 4..7).
// K: element i is channel 32j+16f + 2t + i%2 + 8(i/4); V: channel 32j+16f + g + 8((i/2)%2).
// row: this head's b3 row (b4 row = row + 128) for this K|V; w = 0 (b3) or 1 (b4).
template <bool kV>
__device__ __forceinline__ void ga_bases(const uint8_t *row, uint32_t w, int lane, int j, int f, uint32_t &b0,
                                         uint32_t &b1)
{
    const uint8_t *r = row + w * 128 + 32 * j + 16 * f;
    if (!kV) {
        const int c = 2 * (lane & 3);
        const uint32_t x = __ldg(reinterpret_cast<const uint16_t *>(r + c));
        const uint32_t y = __ldg(reinterpret_cast<const uint16_t *>(r + c + 8));
        b0 = x * 0x00010001u;  // [x0 x1 x0 x1]: multiplies run beside the byte ops
        b1 = y * 0x00010001u;
    } else {
        const int g = lane >> 2;
        const uint32_t x = __ldg(r + g), y = __ldg(r + g + 8);
        b0 = b1 = (x + y * 0x10000u) * 0x0101u;  // [x x y y]
    }
}

// The same base vectors from a per-KV-head table in shared memory, built once per
// attention segment by ga_fill_bases_table: K words [((2j + f) * 2 + w) * 4 + t] as
// (b0, b1) pairs at 2x, V words at 128 + ((2j + f) * 2 + w) * 8 + g (b0 = b1).
template <bool kV>
__device__ __forceinline__ void ga_bases(const uint32_t *tbl, uint32_t w, int lane, int j, int f, uint32_t &b0,
                                         uint32_t &b1)
{
    if (!kV) {
        const uint2 v = *reinterpret_cast<const uint2 *>(tbl + 2 * (((2 * j + f) * 2 + (int)w) * 4 + (lane & 3)));
        b0 = v.x;
        b1 = v.y;
    } else {
        b0 = b1 = tbl[128 + ((2 * j + f) * 2 + (int)w) * 8 + (lane >> 2)];
    }
}

// Build the table above for one KV head (row: its 512 bytes of bases, K b3 | K b4 | V b3 |
// V b4), 128 threads (tid 0..127): the same words ga_bases computes from the row.  zero_b4:
// the b4 words are 0 (FP8 E4M3, whose 16-wide window is the whole exponent field).
__device__ __forceinline__ void ga_fill_bases_table(const uint8_t *row, uint32_t *tbl, int tid, bool zero_b4)
{
    if (tid < 64) {  // K pair: (2j + f, w, t)
        const int t = tid & 3, w = (tid >> 2) & 1, jf = tid >> 3;
        uint32_t b0, b1;
        ga_bases<false>(row, (uint32_t)w, t, jf >> 1, jf & 1, b0, b1);
        tbl[2 * tid] = zero_b4 && w ? 0u : b0;
        tbl[2 * tid + 1] = zero_b4 && w ? 0u : b1;
    }
    {  // V word: (2j + f, w, g)
        const int g = tid & 7, w = (tid >> 3) & 1, jf = tid >> 4;
        uint32_t b0, b1;
        ga_bases<true>(row + 256, (uint32_t)w, g << 2, jf >> 1, jf & 1, b0, b1);
        tbl[128 + tid] = zero_b4 && w ? 0u : b0;
    }
}

// Exponent bytes + sign/fraction bytes -> the four bf16x2 fragment registers.
__device__ __forceinline__ void ga_assemble(uint32_t sf0, uint32_t sf1, uint32_t e0, uint32_t e1, uint32_t (&a)[4])
{
    const uint32_t h0 = ((e0 >> 1) & 0x7F7F7F7Fu) | (sf0 & 0x80808080u);
    const uint32_t l0 = ((e0 << 7) & 0x80808080u) | (sf0 & 0x7F7F7F7Fu);
    const uint32_t h1 = ((e1 >> 1) & 0x7F7F7F7Fu) | (sf1 & 0x80808080u);
    const uint32_t l1 = ((e1 << 7) & 0x80808080u) | (sf1 & 0x7F7F7F7Fu);
    a[0] = __byte_perm(l0, h0, 0x5140);
    a[1] = __byte_perm(l0, h0, 0x7362);
    a[2] = __byte_perm(l1, h1, 0x5140);
    a[3] = __byte_perm(l1, h1, 0x7362);
}

// Restore one group.  Modes 0 and 1 take no branch: a 3-bit group reads no escape
// byte and adds its b3 vector, a 4-bit group adds bit 3 from its escape byte and its b4
// vector.  Raw-exponent groups (mode 2, rare) are patched in a branch that only tiles
// holding such groups enter (any2, warp-uniform).  sf0/sf1: sign/fraction bytes of
// elements 0..3 / 4..7; code: 24-bit field; esc: the tile's escape area; off: running
// offset of this lane's next escape byte.
template <bool kV, typename Row>
__device__ __forceinline__ void ga_restore_group_fast(uint32_t sf0, uint32_t sf1, uint32_t code, uint32_t mode,
                                                      bool any2, const uint8_t *esc, uint32_t &off,
                                                      const Row *row, int lane, int j, int f, uint32_t (&a)[4])
{
    const uint32_t m1 = mode & 1u;
    uint32_t h = 0;
    if (m1) h = esc[min(off, kGaEscCap - 1)];
    off += m1;
    uint32_t b0, b1;
    ga_bases<kV>(row, m1, lane, j, f, b0, b1);
    const uint32_t l0 = ga_spread3(code & 0xFFFu), l1 = ga_spread3((code >> 12) & 0xFFFu);
    uint32_t c0 = l0 | ga_spread1_hi(h), c1 = l1 | ga_spread1_hi(h >> 4);
    if (any2) {
        if (mode >= 2) {
            const uint8_t *p = esc + min(off, kGaEscCap - 5);
            const uint32_t lo =
                (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
            c0 = l0 | ga_spread5_hi(lo & 0xFFFFFu);
            c1 = l1 | ga_spread5_hi((lo >> 20) | ((uint32_t)p[4] << 12));
            b0 = b1 = 0;
            off += 5;
        }
    }
    ga_assemble(sf0, sf1, c0 + b0, c1 + b1, a);  // byte adds never carry (every e <= 255)
}

// This lane's 24 code bytes (groups 8L..8L+7) as six words; group k's field.
__device__ __forceinline__ uint32_t ga_code_field(const uint32_t (&w)[6], int k)
{
    const int bit = 24 * k, wi = bit >> 5, sh = bit & 31;
    const uint32_t lo = w[wi], hi = wi + 1 < 6 ? w[wi + 1] : 0u;
    return __funnelshift_r(lo, hi, sh) & 0xFFFFFFu;
}

// One compressed tile's per-lane state: modes, escape offset, code words.
struct GaLane {
    uint32_t modes, off;
    uint32_t code[6];
};

__device__ __forceinline__ GaLane ga_lane_load(const uint8_t *tile, int lane)
{
    GaLane s;
    s.modes = *reinterpret_cast<const uint16_t *>(tile + kGaTagOff + 2 * lane);
    s.off = ga_lane_escape_base(s.modes, lane);
    const uint2 *c = reinterpret_cast<const uint2 *>(tile + kGaCodeOff + 24 * lane);
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const uint2 v = c[k];
        s.code[2 * k] = v.x;
        s.code[2 * k + 1] = v.y;
    }
    return s;
}

// Fragments of block j (both f) of a compressed tile; row = this head's b3 row;
// any2: some lane's group of this tile has mode 2 (warp-uniform).
template <bool kV, typename Row>
__device__ __forceinline__ void ga_block_frags(const uint8_t *tile, const Row *row, GaLane &s, bool any2, int lane,
                                               int j, uint32_t (&a0)[4], uint32_t (&a1)[4])
{
    const uint4 sf = *reinterpret_cast<const uint4 *>(tile + 512 * j + 16 * lane);
    const uint8_t *esc = tile + kGaEscOff;
    const uint32_t m0 = (s.modes >> (4 * j)) & 3u, m1 = (s.modes >> (4 * j + 2)) & 3u;
    ga_restore_group_fast<kV>(sf.x, sf.y, ga_code_field(s.code, 2 * j), m0, any2, esc, s.off, row, lane, j, 0, a0);
    ga_restore_group_fast<kV>(sf.z, sf.w, ga_code_field(s.code, 2 * j + 1), m1, any2, esc, s.off, row, lane, j, 1, a1);
}

// Whether any lane's groups of this tile use the raw-exponent mode.  Warp-collective.
__device__ __forceinline__ bool ga_tile_any_raw_groups(const GaLane &s) { return __any_sync(0xffffffffu, s.modes & 0xAAAAu); }

}  // namespace kvz
