// stage.cuh -- shared-memory staging of one (page, KV head) K+V slice and the gather
// of a lane's fragment elements in the storage order both compressed formats use.
#pragma once

#include "kvz_device.cuh"

namespace kvz {

// ---------------------------------------------------------------------------------
// storage order: element (lane, f, i) of block j  ->  (token, dim) of the page slice
// ---------------------------------------------------------------------------------
__device__ __forceinline__ int frag_row(int lane, int i) { return (lane >> 2) + 8 * ((i >> 1) & 1); }
__device__ __forceinline__ int frag_col(int lane, int i) { return 2 * (lane & 3) + (i & 1) + 8 * (i >> 2); }

// Page slice staging in shared memory: 32 rows (K tokens 0..15, V tokens 16..31) of
// 128 BF16 with a 272-byte pitch, so the fragment gathers below hit 32 distinct banks.
constexpr int kStagePitch = 272;

// Gather this lane's 16 values of block (kv, j) in storage order as 8 bf16x2 words
// (w[0..3] = fragment 0 elements (0,1),(2,3),(4,5),(6,7); w[4..7] = fragment 1).
__device__ __forceinline__ void gather_block(const uint8_t *stage, int kv, int j, int lane, uint32_t (&w)[8])
{
#pragma unroll
    for (int f = 0; f < 2; ++f)
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const int r = frag_row(lane, i), c = frag_col(lane, i);
            const int dim0 = 32 * j + 16 * f;
            uint32_t v;
            if (kv == 0) {  // K: token r, dims c and c+1 are adjacent
                v = *reinterpret_cast<const uint32_t *>(stage + r * kStagePitch + (dim0 + c) * 2);
            } else {  // V: tokens c and c+1 of dim r
                const uint8_t *base = stage + (16 + c) * kStagePitch + (dim0 + r) * 2;
                uint32_t lo = *reinterpret_cast<const uint16_t *>(base);
                uint32_t hi = *reinterpret_cast<const uint16_t *>(base + kStagePitch);
                v = lo | (hi << 16);
            }
            w[f * 4 + i / 2] = v;
        }
}

// bytes 2s and 2s+1 of x -> the low bytes of two 16-bit halves
__device__ __forceinline__ uint32_t enc_spread2(uint32_t x, int s) { return __byte_perm(x, 0, s ? 0x4342 : 0x4140); }

// prmt with the selector used as is: a selector nibble with bit 3 set gives the sign bit of
// the chosen byte replicated over the result byte
__device__ __forceinline__ uint32_t prmt_b32(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ void load_slice_to_stage(const uint16_t *src, uint8_t *stage, int tid, int nthreads)
{
    // 8 KB slice: 512 chunks of 16 B; chunk q -> row q/16, byte (q%16)*16
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
    for (int q = tid; q < 512; q += nthreads) {
        uint4 v = s4[q];
        *reinterpret_cast<uint4 *>(stage + (q >> 4) * kStagePitch + (q & 15) * 16) = v;
    }
}

}  // namespace kvz
