// kvz_device.cuh -- device-side building blocks of libkvz (sm_103a): inline-PTX
// wrappers for mbarriers, bulk and tensor TMA copies, ldmatrix/movmatrix, the
// m16n8k16 BF16 tensor-core MMA, and the 12-bit block restore.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/kvz.h"

namespace kvz {

constexpr int kPage = 16;
constexpr int kDim = 128;
constexpr uint32_t kGranule = 256;

// ---------------------------------------------------------------------------------
// bit helpers
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Granules of a block from its tag: 3 (768 B) eligible, 4 (1024 B) raw.
__host__ __device__ __forceinline__ uint32_t tag_granules(uint32_t tag) { return tag == 0xFFu ? 4u : 3u; }

// A tag byte is valid when it is b/2 (< 0x80) or the raw sentinel 0xFF.
__host__ __device__ __forceinline__ bool tags_valid(uint32_t tags)
{
    for (int k = 0; k < 4; ++k) {
        uint32_t t = (tags >> (8 * k)) & 0xFFu;
        if (t >= 0x80u && t != 0xFFu) return false;
    }
    return true;
}

__host__ __device__ __forceinline__ uint32_t group_granules(uint32_t tags)
{
    uint32_t g = 0;
    for (int k = 0; k < 4; ++k) g += tag_granules((tags >> (8 * k)) & 0xFFu);
    return g;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------------
// 12-bit restore: one masked branch and one nibble-swapped branch of the code word,
// each plus b/2 replicated per byte (never carries: b/2 + d <= 127), interleaved
// with the kept low bytes into four bf16x2 registers (elements 0..7 of a fragment).
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void restore_fragment(uint32_t low03, uint32_t low47, uint32_t code,
                                                 uint32_t bb, uint32_t (&a)[4])
{
    const uint32_t h03 = (code & 0x87878787u) + bb;
    const uint32_t h47 = (((code >> 4) & 0x07070707u) | ((code << 4) & 0x80808080u)) + bb;
    a[0] = __byte_perm(low03, h03, 0x5140);
    a[1] = __byte_perm(low03, h03, 0x7362);
    a[2] = __byte_perm(low47, h47, 0x5140);
    a[3] = __byte_perm(low47, h47, 0x7362);
}

// ---------------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test for the phase of `parity` (the thread is never suspended, so the
// lanes of a warp can poll different barriers together).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `parity` with a time limit.  Returns false (and sets the
// timeout status bit) when the limit passes; the caller then stops using the stage.
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s: kernels here run for micro- to milliseconds

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t *status,
                                          uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) {
            atomicOr(status, KVZ_STATUS_TIMEOUT);
            return false;
        }
    }
}

// ---------------------------------------------------------------------------------
// TMA: 1-D bulk copy and 2-D tiled tensor copy into this CTA's shared memory
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tensor_copy_2d_g2s(uint32_t dst, const void *tmap, int32_t c0, int32_t c1, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// L2 cache policies: the KV stream is read once per step (evict first), while the
// small tables every step starts from (lengths, page ids, metadata) should stay
// resident across steps (evict last).
__device__ __forceinline__ uint64_t l2_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void bulk_copy_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                                   uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tensor_copy_2d_g2s_hint(uint32_t dst, const void *tmap, int32_t c0, int32_t c1,
                                                        uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ int32_t ld_keep_s32(const int32_t *p, uint64_t policy)
{
    int32_t v;
    asm volatile("ld.global.L2::cache_hint.b32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(policy));
    return v;
}

__device__ __forceinline__ void ld_keep_u64x2(const uint64_t *p, uint64_t policy, uint64_t &a, uint64_t &b)
{
    asm volatile("ld.global.L2::cache_hint.v2.b64 {%0, %1}, [%2], %3;" : "=l"(a), "=l"(b) : "l"(p), "l"(policy));
}

__device__ __forceinline__ uint64_t ld_keep_u64(const uint64_t *p, uint64_t policy)
{
    uint64_t v;
    asm volatile("ld.global.L2::cache_hint.b64 %0, [%1], %2;" : "=l"(v) : "l"(p), "l"(policy));
    return v;
}

__device__ __forceinline__ void prefetch_tensormap(const void *tmap)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ---------------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------------
// warp-level matrix ops
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a)
{
    uint32_t d;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// D = A(16x16, bf16, row) * B(16x8, bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// bf16x2 pack, round to nearest even: low half = lo, high half = hi.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_round(float x)
{
    uint32_t r = pack_bf16x2(x, 0.0f);
    return __uint_as_float(r << 16);
}

// D = A(16x16, f16, row) * B(16x8, f16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// f16x2 pack, round to nearest even: low half = lo, high half = hi.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float f16_round(float x)
{
    float r;
    asm("{\n\t.reg .f16 h;\n\tcvt.rn.f16.f32 h, %1;\n\tcvt.f32.f16 %0, h;\n\t}" : "=f"(r) : "f"(x));
    return r;
}

// bf16x2 -> f16x2, round to nearest even (exact for values in the f16 normal range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w)
{
    return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

}  // namespace kvz
