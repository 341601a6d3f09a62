// kvz_api.cu -- the C ABI (include/kvz.h): host-side argument checks, launch
// configuration and the TMA tensor map for raw pages.  All compute runs in the
// kernels of codec.cu, ga_codec.cu and attention.cu; nothing here touches device data.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "kvz_internal.h"

using namespace kvz;

namespace {

thread_local int g_last_cuda = 0;

int fail_cuda(cudaError_t e)
{
    g_last_cuda = static_cast<int>(e);
    return KVZ_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool dims_ok(const kvz_dims &d) { return d.num_kv_heads >= 1 && d.head_dim == kDim && d.page_size == kPage; }

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// Number of attention CTAs: one wave of the CTAs the device holds, but at least
// kMinPagesPerCta pages each.  Depends only on shapes and the device.
int attention_grid(int batch, int hkv, int table_pages, int *grid)
{
    int per_sm = 0;
    cudaError_t e = attn_ctas_per_sm(batch, &per_sm);
    if (e != cudaSuccess) return fail_cuda(e);
    if (per_sm < 1) return KVZ_ERR_UNSUPPORTED;
    const int sms = sm_count();
    if (sms < 1) return KVZ_ERR_DEVICE;
    const int64_t wave = (int64_t)sms * per_sm;
    const int64_t pages = (int64_t)batch * hkv * (int64_t)(table_pages > 0 ? table_pages : 1);
    int64_t c = (pages + kMinPagesPerCta - 1) / kMinPagesPerCta;
    if (c > wave) c = wave;
    if (c < 1) c = 1;
    *grid = (int)c;
    return KVZ_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Raw pool as a 2-D tensor [num_raw_pages * hkv * 32 rows][128 BF16]; box = 64 columns
// x 32 rows (the K and V rows of one page and head), 128-byte swizzle.
int raw_tensor_map(const void *raw_pool, int64_t num_raw_pages, int hkv, CUtensorMap *map)
{
    thread_local const void *c_ptr = nullptr;
    thread_local int64_t c_rows = -1;
    thread_local CUtensorMap c_map;
    const int64_t rows = num_raw_pages * hkv * 32;
    if (c_ptr == raw_pool && c_rows == rows) {
        *map = c_map;
        return KVZ_OK;
    }
    auto enc = tensor_map_encoder();
    if (!enc) return KVZ_ERR_DEVICE;
    cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kDim * 2};
    cuuint32_t box[2] = {64, 32};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(raw_pool), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        g_last_cuda = (int)r;
        return KVZ_ERR_CUDA;
    }
    c_ptr = raw_pool;
    c_rows = rows;
    c_map = *map;
    return KVZ_OK;
}

int check_attention_common(const kvz_dims &d, int batch, int hq, const void *q, const int32_t *seq_lens,
                           const void *raw_pool, int64_t num_raw_pages, const float *out, const void *ws,
                           const uint32_t *status, int max_pages, const int32_t *page_ids)
{
    if (!dims_ok(d)) return d.num_kv_heads >= 1 ? KVZ_ERR_UNSUPPORTED : KVZ_ERR_INVALID_ARG;
    if (batch < 0 || hq < 1 || max_pages < 0 || num_raw_pages < 0) return KVZ_ERR_INVALID_ARG;
    if (hq % d.num_kv_heads != 0) return KVZ_ERR_INVALID_ARG;
    const int G = hq / d.num_kv_heads;
    if (G < 1 || G > 8) return KVZ_ERR_UNSUPPORTED;
    if (batch > kMaxBatch) return KVZ_ERR_UNSUPPORTED;
    if (batch == 0) return KVZ_OK;
    if (!q || !seq_lens || !out || !ws || !status || (max_pages > 0 && !page_ids)) return KVZ_ERR_INVALID_ARG;
    if (num_raw_pages > 0 && !raw_pool) return KVZ_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(ws, 16) || !aligned(out, 4) || !aligned(raw_pool, 16) || !aligned(seq_lens, 4) ||
        !aligned(status, 4))
        return KVZ_ERR_ALIGNMENT;
    if (num_raw_pages * d.num_kv_heads * 32 >= (int64_t)1 << 31) return KVZ_ERR_UNSUPPORTED;
    return KVZ_OK;
}

struct FormatArgs {
    int format;  // AttnFormat
    const uint64_t *meta;
    const uint32_t *meta32;
    const uint8_t *ga_bases;
};

int run_attention(const FormatArgs &F, const kvz_dims &d, int batch, int hq, const void *q, const int32_t *page_ids,
                  int max_pages, const int32_t *seq_lens, const int32_t *tail_page, int64_t num_meta_pages,
                  const uint8_t *arena, uint64_t arena_bytes, const void *raw_pool, int64_t num_raw_pages, float *out,
                  void *ws, size_t ws_bytes, uint32_t *status, cudaStream_t stream, uint32_t flags = 0)
{
    const int hkv = d.num_kv_heads;
    const int table_pages = F.format != kFmtRaw ? max_pages + 1 : max_pages;
    int grid = 0;
    int rc = attention_grid(batch, hkv, table_pages, &grid);
    if (rc) return rc;
    if (attn_ws_bytes(batch, hkv, grid, hq / hkv) > ws_bytes) return KVZ_ERR_WORKSPACE;
    CUtensorMap map;
    // a pool with no pages still needs a valid map object; it is never dereferenced
    rc = raw_tensor_map(raw_pool ? raw_pool : ws, num_raw_pages > 0 ? num_raw_pages : 1, hkv, &map);
    if (rc) return rc;
    AttnParams P;
    memset(&P, 0, sizeof P);
    P.batch = batch;
    P.hkv = hkv;
    P.G = hq / hkv;
    P.max_pages = max_pages;
    P.grid = grid;
    P.q = static_cast<const uint16_t *>(q);
    P.page_ids = page_ids;
    P.seq_lens = seq_lens;
    P.tail_page = tail_page;
    P.meta = F.meta;
    P.meta32 = F.meta32;
    P.ga_bases = F.ga_bases;
    P.num_meta_pages = num_meta_pages;
    P.arena = arena;
    P.arena_bytes = arena_bytes;
    P.num_raw_pages = num_raw_pages;
    P.out = out;
    uint8_t *w = static_cast<uint8_t *>(ws);
    const size_t slots = attn_slots(batch, hkv, grid);
    P.part_o = reinterpret_cast<float *>(w);
    w += slots * attn_slot_heads(hq / hkv) * 128 * 4;
    P.part_ml = reinterpret_cast<float *>(w);
    P.status = status;
    P.scale_log2 = (float)(1.4426950408889634 / 11.313708498984761);  // log2(e) / sqrt(128)
    P.overlap = (flags & KVZ_ATTN_OVERLAP_PREVIOUS) ? 1 : 0;
    cudaError_t e = launch_attention(P, F.format, &map, stream);
    return e == cudaSuccess ? KVZ_OK : fail_cuda(e);
}

// ---------------------------------------------------------------------------------
// Fixed scratch for kvz_decode_attention_noalloc.  In host code the array's name is
// only a host-side stand-in; its device address comes from cudaGetSymbolAddress, looked
// up once per device (with that device current) and cached.
// ---------------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_noalloc_scratch[KVZ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDevices] = {};

int noalloc_scratch(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return KVZ_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return fail_cuda(e);
        if (!p) return KVZ_ERR_DEVICE;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return KVZ_OK;
}

}  // namespace

extern "C" {

const char *kvz_strerror(int code)
{
    switch (code) {
    case KVZ_OK: return "ok";
    case KVZ_ERR_INVALID_ARG: return "invalid argument";
    case KVZ_ERR_UNSUPPORTED: return "unsupported shape";
    case KVZ_ERR_ALIGNMENT: return "pointer misaligned";
    case KVZ_ERR_WORKSPACE: return "workspace too small";
    case KVZ_ERR_CUDA: return "CUDA error (see kvz_last_cuda_error)";
    case KVZ_ERR_DEVICE: return "no usable CUDA device";
    case KVZ_ERR_OUT_OF_SPACE: return "no free arena chunk";
    case KVZ_ERR_NOALLOC_LIMIT: return "problem needs more split-KV scratch than the fixed no-alloc array holds";
    default: return "unknown error";
    }
}

int kvz_last_cuda_error(void) { return g_last_cuda; }

int kvz_device_sm_count(void) { return sm_count(); }

size_t kvz_encode_workspace_size(kvz_dims dims, int32_t n)
{
    if (!dims_ok(dims) || n < 0) return 0;
    return encode_ws_bytes(n, dims.num_kv_heads);
}

int kvz_encode_pages(kvz_dims dims, const void *raw_pool, int64_t num_raw_pages, const int32_t *src_page,
                     const int32_t *dst_page, const int32_t *dst_seq, int32_t n, uint64_t *meta,
                     int64_t num_meta_pages, uint8_t *arena, uint64_t arena_bytes, uint32_t *cursors,
                     int32_t num_cursors, void *workspace, size_t workspace_bytes, uint32_t *status,
                     kvz_stream_t stream)
{
    if (!dims_ok(dims)) return dims.num_kv_heads >= 1 ? KVZ_ERR_UNSUPPORTED : KVZ_ERR_INVALID_ARG;
    if (n < 0 || num_raw_pages < 0 || num_meta_pages < 0 || num_cursors < 0) return KVZ_ERR_INVALID_ARG;
    if (n == 0) return KVZ_OK;
    if (!raw_pool || !src_page || !dst_page || !dst_seq || !meta || !arena || !cursors || !workspace || !status)
        return KVZ_ERR_INVALID_ARG;
    if (!aligned(raw_pool, 16) || !aligned(meta, 16) || !aligned(arena, 256) || !aligned(cursors, 8) ||
        !aligned(workspace, 16) || !aligned(status, 4))
        return KVZ_ERR_ALIGNMENT;
    if ((int64_t)n * dims.num_kv_heads > (int64_t)1 << 30) return KVZ_ERR_UNSUPPORTED;
    if (workspace_bytes < kvz_encode_workspace_size(dims, n)) return KVZ_ERR_WORKSPACE;
    EncodeParams P;
    memset(&P, 0, sizeof P);
    P.hkv = dims.num_kv_heads;
    P.n = n;
    P.raw_pool = static_cast<const uint16_t *>(raw_pool);
    P.num_raw_pages = num_raw_pages;
    P.src_page = src_page;
    P.dst_page = dst_page;
    P.dst_seq = dst_seq;
    P.meta = meta;
    P.num_meta_pages = num_meta_pages;
    P.arena = arena;
    P.arena_bytes = arena_bytes;
    P.cursors = cursors;
    P.num_cursors = num_cursors;
    P.status = status;
    uint8_t *w = static_cast<uint8_t *>(workspace);
    const size_t a = ((size_t)n * 4 + 15) / 16 * 16;
    P.ws_hdr = reinterpret_cast<uint32_t *>(w);
    P.ws_page_size = reinterpret_cast<uint32_t *>(w + 16);  // page-size sums after the header
    P.ws_page_base = reinterpret_cast<uint32_t *>(w + 16 + a);
    P.ws_pair_size = reinterpret_cast<uint32_t *>(w + 16 + 2 * a);
    P.ws_tags = reinterpret_cast<uint64_t *>(w + encode_ws_tags_offset(n, dims.num_kv_heads));
    cudaError_t e = launch_encode(P, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVZ_OK : fail_cuda(e);
}

int kvz_encode_sizes(kvz_dims dims, const void *raw_pool, int64_t num_raw_pages, const int32_t *src_page, int32_t n,
                     uint32_t *granules, void *workspace, size_t workspace_bytes, uint32_t *status,
                     kvz_stream_t stream)
{
    if (!dims_ok(dims)) return dims.num_kv_heads >= 1 ? KVZ_ERR_UNSUPPORTED : KVZ_ERR_INVALID_ARG;
    if (n < 0 || num_raw_pages < 0) return KVZ_ERR_INVALID_ARG;
    if (n == 0) return KVZ_OK;
    if (!raw_pool || !src_page || !granules || !workspace || !status) return KVZ_ERR_INVALID_ARG;
    if (!aligned(raw_pool, 16) || !aligned(granules, 4) || !aligned(workspace, 16) || !aligned(status, 4))
        return KVZ_ERR_ALIGNMENT;
    if ((int64_t)n * dims.num_kv_heads > (int64_t)1 << 30) return KVZ_ERR_UNSUPPORTED;
    if (workspace_bytes < kvz_encode_workspace_size(dims, n)) return KVZ_ERR_WORKSPACE;
    EncodeParams P;
    memset(&P, 0, sizeof P);
    P.hkv = dims.num_kv_heads;
    P.n = n;
    P.raw_pool = static_cast<const uint16_t *>(raw_pool);
    P.num_raw_pages = num_raw_pages;
    P.src_page = src_page;
    P.dst_page = src_page;  // only validated: no metadata is written
    P.dst_seq = nullptr;
    P.num_meta_pages = num_raw_pages;
    P.num_cursors = 1;
    P.status = status;
    uint8_t *w = static_cast<uint8_t *>(workspace);
    const size_t a = ((size_t)n * 4 + 15) / 16 * 16;
    P.ws_hdr = reinterpret_cast<uint32_t *>(w);
    P.ws_page_size = granules;
    P.ws_pair_size = reinterpret_cast<uint32_t *>(w + 16 + 2 * a);
    cudaError_t e = launch_encode_sizes(P, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVZ_OK : fail_cuda(e);
}

int kvz_decode_blocks(kvz_dims dims, const uint64_t *meta, int64_t num_meta_pages, const uint8_t *arena,
                      uint64_t arena_bytes, const int32_t *page, int32_t n, void *out_pages, uint32_t *status,
                      kvz_stream_t stream)
{
    if (!dims_ok(dims)) return dims.num_kv_heads >= 1 ? KVZ_ERR_UNSUPPORTED : KVZ_ERR_INVALID_ARG;
    if (n < 0 || num_meta_pages < 0) return KVZ_ERR_INVALID_ARG;
    if (n == 0) return KVZ_OK;
    if (!meta || !arena || !page || !out_pages || !status) return KVZ_ERR_INVALID_ARG;
    if (!aligned(meta, 8) || !aligned(arena, 256) || !aligned(out_pages, 16) || !aligned(status, 4))
        return KVZ_ERR_ALIGNMENT;
    if ((int64_t)n * dims.num_kv_heads > (int64_t)1 << 30) return KVZ_ERR_UNSUPPORTED;
    DecodeParams P;
    memset(&P, 0, sizeof P);
    P.hkv = dims.num_kv_heads;
    P.n = n;
    P.meta = meta;
    P.num_meta_pages = num_meta_pages;
    P.arena = arena;
    P.arena_bytes = arena_bytes;
    P.page = page;
    P.out = static_cast<uint16_t *>(out_pages);
    P.status = status;
    cudaError_t e = launch_decode(P, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVZ_OK : fail_cuda(e);
}

size_t kvz_attention_workspace_size(kvz_dims dims, int32_t batch, int32_t num_q_heads, int32_t table_pages)
{
    if (!dims_ok(dims) || batch < 0 || num_q_heads < 1 || table_pages < 0) return 0;
    if (batch == 0) return 16;
    int grid = 0;
    if (attention_grid(batch, dims.num_kv_heads, table_pages, &grid) != KVZ_OK) return 0;
    return attn_ws_bytes(batch, dims.num_kv_heads, grid, num_q_heads / dims.num_kv_heads);
}

int kvz_decode_attention(kvz_dims dims, int32_t batch, int32_t num_q_heads, const void *q, const int32_t *page_ids,
                         int32_t max_pages, const int32_t *seq_lens, const int32_t *tail_page, const uint64_t *meta,
                         int64_t num_meta_pages, const uint8_t *arena, uint64_t arena_bytes, const void *raw_pool,
                         int64_t num_raw_pages, float *out, void *workspace, size_t workspace_bytes,
                         uint32_t *status, kvz_stream_t stream)
{
    int rc = check_attention_common(dims, batch, num_q_heads, q, seq_lens, raw_pool, num_raw_pages, out, workspace,
                                    status, max_pages, page_ids);
    if (rc || batch == 0) return rc;
    if (!tail_page || !meta || !arena || num_meta_pages < 0) return KVZ_ERR_INVALID_ARG;
    if (!aligned(meta, 16) || !aligned(arena, 256) || !aligned(tail_page, 4)) return KVZ_ERR_ALIGNMENT;
    return run_attention(FormatArgs{kFmtZf, meta, nullptr, nullptr}, dims, batch, num_q_heads, q, page_ids,
                         max_pages, seq_lens, tail_page, num_meta_pages, arena, arena_bytes, raw_pool, num_raw_pages,
                         out, workspace, workspace_bytes, status, reinterpret_cast<cudaStream_t>(stream));
}

int kvz_decode_attention_raw(kvz_dims dims, int32_t batch, int32_t num_q_heads, const void *q,
                             const int32_t *page_ids, int32_t max_pages, const int32_t *seq_lens,
                             const void *raw_pool, int64_t num_raw_pages, float *out, void *workspace,
                             size_t workspace_bytes, uint32_t *status, kvz_stream_t stream)
{
    int rc = check_attention_common(dims, batch, num_q_heads, q, seq_lens, raw_pool, num_raw_pages, out, workspace,
                                    status, max_pages, page_ids);
    if (rc || batch == 0) return rc;
    return run_attention(FormatArgs{kFmtRaw, nullptr, nullptr, nullptr}, dims, batch, num_q_heads, q, page_ids,
                         max_pages, seq_lens, nullptr, 0, nullptr, 0, raw_pool, num_raw_pages, out, workspace,
                         workspace_bytes, status, reinterpret_cast<cudaStream_t>(stream));
}

int kvz_decode_attention_ex(kvz_dims dims, int32_t batch, int32_t num_q_heads, const void *q, const int32_t *page_ids,
                            int32_t max_pages, const int32_t *seq_lens, const int32_t *tail_page,
                            const uint64_t *meta, int64_t num_meta_pages, const uint8_t *arena, uint64_t arena_bytes,
                            const void *raw_pool, int64_t num_raw_pages, float *out, void *workspace,
                            size_t workspace_bytes, uint32_t *status, uint32_t flags, kvz_stream_t stream)
{
    if (flags & ~KVZ_ATTN_FLAGS_ALL) return KVZ_ERR_INVALID_ARG;
    int rc = check_attention_common(dims, batch, num_q_heads, q, seq_lens, raw_pool, num_raw_pages, out, workspace,
                                    status, max_pages, page_ids);
    if (rc || batch == 0) return rc;
    if (!tail_page || !meta || !arena || num_meta_pages < 0) return KVZ_ERR_INVALID_ARG;
    if (!aligned(meta, 16) || !aligned(arena, 256) || !aligned(tail_page, 4)) return KVZ_ERR_ALIGNMENT;
    return run_attention(FormatArgs{kFmtZf, meta, nullptr, nullptr}, dims, batch, num_q_heads, q, page_ids,
                         max_pages, seq_lens, tail_page, num_meta_pages, arena, arena_bytes, raw_pool, num_raw_pages,
                         out, workspace, workspace_bytes, status, reinterpret_cast<cudaStream_t>(stream), flags);
}

int kvz_decode_attention_raw_ex(kvz_dims dims, int32_t batch, int32_t num_q_heads, const void *q,
                                const int32_t *page_ids, int32_t max_pages, const int32_t *seq_lens,
                                const void *raw_pool, int64_t num_raw_pages, float *out, void *workspace,
                                size_t workspace_bytes, uint32_t *status, uint32_t flags, kvz_stream_t stream)
{
    if (flags & ~KVZ_ATTN_FLAGS_ALL) return KVZ_ERR_INVALID_ARG;
    int rc = check_attention_common(dims, batch, num_q_heads, q, seq_lens, raw_pool, num_raw_pages, out, workspace,
                                    status, max_pages, page_ids);
    if (rc || batch == 0) return rc;
    return run_attention(FormatArgs{kFmtRaw, nullptr, nullptr, nullptr}, dims, batch, num_q_heads, q, page_ids,
                         max_pages, seq_lens, nullptr, 0, nullptr, 0, raw_pool, num_raw_pages, out, workspace,
                         workspace_bytes, status, reinterpret_cast<cudaStream_t>(stream), flags);
}

int kvz_decode_attention_noalloc(kvz_dims dims, int32_t batch, int32_t num_q_heads, const void *q,
                                 const int32_t *page_ids, int32_t max_pages, const int32_t *seq_lens,
                                 const int32_t *tail_page, const uint64_t *meta, int64_t num_meta_pages,
                                 const uint8_t *arena, uint64_t arena_bytes, const void *raw_pool,
                                 int64_t num_raw_pages, float *out, uint32_t *status, kvz_stream_t stream)
{
    void *scratch = nullptr;
    if (batch > 0) {
        int src = noalloc_scratch(&scratch);  // device address of the fixed array
        if (src) return src;
    }
    int rc = check_attention_common(dims, batch, num_q_heads, q, seq_lens, raw_pool, num_raw_pages, out, scratch,
                                    status, max_pages, page_ids);
    if (rc || batch == 0) return rc;
    if (!tail_page || !meta || !arena || num_meta_pages < 0) return KVZ_ERR_INVALID_ARG;
    if (!aligned(meta, 16) || !aligned(arena, 256) || !aligned(tail_page, 4)) return KVZ_ERR_ALIGNMENT;
    int grid = 0;
    rc = attention_grid(batch, dims.num_kv_heads, max_pages + 1, &grid);
    if (rc) return rc;
    if (attn_ws_bytes(batch, dims.num_kv_heads, grid, num_q_heads / dims.num_kv_heads) > (size_t)KVZ_NOALLOC_SCRATCH_BYTES)
        return KVZ_ERR_NOALLOC_LIMIT;
    return run_attention(FormatArgs{kFmtZf, meta, nullptr, nullptr}, dims, batch, num_q_heads, q, page_ids,
                         max_pages, seq_lens, tail_page, num_meta_pages, arena, arena_bytes, raw_pool, num_raw_pages,
                         out, scratch, KVZ_NOALLOC_SCRATCH_BYTES, status, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------------
// group-adaptive additive tiles
// ---------------------------------------------------------------------------------
int kvz_ga_calibrate(kvz_dims dims, const void *raw_pool, int64_t num_raw_pages, const int32_t *pages, int32_t n,
                     uint8_t *bases, uint32_t *status, kvz_stream_t stream)
{
    if (!dims_ok(dims)) return dims.num_kv_heads >= 1 ? KVZ_ERR_UNSUPPORTED : KVZ_ERR_INVALID_ARG;
    if (n < 0 || num_raw_pages < 0) return KVZ_ERR_INVALID_ARG;
    if (!bases || !status || (n > 0 && (!raw_pool || !pages))) return KVZ_ERR_INVALID_ARG;
    if (!aligned(raw_pool, 16) || !aligned(pages, 4) || !aligned(status, 4)) return KVZ_ERR_ALIGNMENT;
    if ((int64_t)n * kPage >= (int64_t)1 << 40 || dims.num_kv_heads > (1 << 20)) return KVZ_ERR_UNSUPPORTED;
    cudaError_t e = launch_ga_calibrate(dims.num_kv_heads, static_cast<const uint16_t *>(raw_pool), num_raw_pages,
                                        pages, n, bases, status, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVZ_OK : fail_cuda(e);
}

int kvz_ga_encode_pages(kvz_dims dims, const void *raw_pool, int64_t num_raw_pages, const uint8_t *bases,
                        const int32_t *src_page, const int32_t *dst_page, const int32_t *dst_seq, int32_t n,
                        uint32_t *meta, int64_t num_meta_pages, uint8_t *arena, uint64_t arena_bytes,
                        uint32_t *cursors, int32_t num_cursors, void *workspace, size_t workspace_bytes,
                        uint32_t *status, kvz_stream_t stream)
{
    if (!dims_ok(dims)) return dims.num_kv_heads >= 1 ? KVZ_ERR_UNSUPPORTED : KVZ_ERR_INVALID_ARG;
    if (n < 0 || num_raw_pages < 0 || num_meta_pages < 0 || num_cursors < 0) return KVZ_ERR_INVALID_ARG;
    if (n == 0) return KVZ_OK;
    if (!raw_pool || !bases || !src_page || !dst_page || !dst_seq || !meta || !arena || !cursors || !workspace ||
        !status)
        return KVZ_ERR_INVALID_ARG;
    if (!aligned(raw_pool, 16) || !aligned(bases, 16) || !aligned(meta, 8) || !aligned(arena, 64) ||
        !aligned(cursors, 8) || !aligned(workspace, 16) || !aligned(status, 4))
        return KVZ_ERR_ALIGNMENT;
    if ((int64_t)n * dims.num_kv_heads > (int64_t)1 << 30) return KVZ_ERR_UNSUPPORTED;
    if (workspace_bytes < kvz_encode_workspace_size(dims, n)) return KVZ_ERR_WORKSPACE;
    EncodeParams P;
    memset(&P, 0, sizeof P);
    P.hkv = dims.num_kv_heads;
    P.n = n;
    P.raw_pool = static_cast<const uint16_t *>(raw_pool);
    P.num_raw_pages = num_raw_pages;
    P.src_page = src_page;
    P.dst_page = dst_page;
    P.dst_seq = dst_seq;
    P.meta32 = meta;
    P.ga_bases = bases;
    P.num_meta_pages = num_meta_pages;
    P.arena = arena;
    P.arena_bytes = arena_bytes;
    P.cursors = cursors;
    P.num_cursors = num_cursors;
    P.status = status;
    uint8_t *w = static_cast<uint8_t *>(workspace);
    const size_t a = ((size_t)n * 4 + 15) / 16 * 16;
    P.ws_hdr = reinterpret_cast<uint32_t *>(w);
    P.ws_page_size = reinterpret_cast<uint32_t *>(w + 16);
    P.ws_page_base = reinterpret_cast<uint32_t *>(w + 16 + a);
    P.ws_pair_size = reinterpret_cast<uint32_t *>(w + 16 + 2 * a);
    P.ws_tags = reinterpret_cast<uint64_t *>(w + encode_ws_tags_offset(n, dims.num_kv_heads));
    cudaError_t e = launch_ga_encode(P, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVZ_OK : fail_cuda(e);
}

int kvz_ga_decode_blocks(kvz_dims dims, const uint32_t *meta, int64_t num_meta_pages, const uint8_t *arena,
                         uint64_t arena_bytes, const uint8_t *bases, const int32_t *page, int32_t n, void *out_pages,
                         uint32_t *status, kvz_stream_t stream)
{
    if (!dims_ok(dims)) return dims.num_kv_heads >= 1 ? KVZ_ERR_UNSUPPORTED : KVZ_ERR_INVALID_ARG;
    if (n < 0 || num_meta_pages < 0) return KVZ_ERR_INVALID_ARG;
    if (n == 0) return KVZ_OK;
    if (!meta || !arena || !bases || !page || !out_pages || !status) return KVZ_ERR_INVALID_ARG;
    if (!aligned(meta, 4) || !aligned(arena, 64) || !aligned(out_pages, 16) || !aligned(status, 4))
        return KVZ_ERR_ALIGNMENT;
    if ((int64_t)n * dims.num_kv_heads > (int64_t)1 << 30) return KVZ_ERR_UNSUPPORTED;
    DecodeParams P;
    memset(&P, 0, sizeof P);
    P.hkv = dims.num_kv_heads;
    P.n = n;
    P.meta32 = meta;
    P.ga_bases = bases;
    P.num_meta_pages = num_meta_pages;
    P.arena = arena;
    P.arena_bytes = arena_bytes;
    P.page = page;
    P.out = static_cast<uint16_t *>(out_pages);
    P.status = status;
    cudaError_t e = launch_ga_decode(P, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVZ_OK : fail_cuda(e);
}

int kvz_ga_decode_attention(kvz_dims dims, int32_t batch, int32_t num_q_heads, const void *q,
                            const int32_t *page_ids, int32_t max_pages, const int32_t *seq_lens,
                            const int32_t *tail_page, const uint32_t *meta, int64_t num_meta_pages,
                            const uint8_t *arena, uint64_t arena_bytes, const uint8_t *bases, const void *raw_pool,
                            int64_t num_raw_pages, float *out, void *workspace, size_t workspace_bytes,
                            uint32_t *status, kvz_stream_t stream)
{
    int rc = check_attention_common(dims, batch, num_q_heads, q, seq_lens, raw_pool, num_raw_pages, out, workspace,
                                    status, max_pages, page_ids);
    if (rc || batch == 0) return rc;
    if (!tail_page || !meta || !arena || !bases || num_meta_pages < 0) return KVZ_ERR_INVALID_ARG;
    if (!aligned(meta, 8) || !aligned(arena, 64) || !aligned(tail_page, 4) || !aligned(bases, 2))
        return KVZ_ERR_ALIGNMENT;
    return run_attention(FormatArgs{kFmtGa, nullptr, meta, bases}, dims, batch, num_q_heads, q, page_ids, max_pages,
                         seq_lens, tail_page, num_meta_pages, arena, arena_bytes, raw_pool, num_raw_pages, out,
                         workspace, workspace_bytes, status, reinterpret_cast<cudaStream_t>(stream));
}

int kvz_selftest_late_writer(const void *src, void *dst, uint64_t bytes, uint64_t delay_ns, kvz_stream_t stream)
{
    if (bytes == 0) return KVZ_OK;
    if (!src || !dst) return KVZ_ERR_INVALID_ARG;
    if (!aligned(src, 16) || !aligned(dst, 16) || bytes % 16 != 0) return KVZ_ERR_ALIGNMENT;
    if (delay_ns > 1000000000ull || bytes > ((uint64_t)1 << 30)) return KVZ_ERR_INVALID_ARG;  // <= 1 s, <= 1 GiB
    cudaError_t e = launch_late_writer(src, dst, bytes, delay_ns, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVZ_OK : fail_cuda(e);
}

int kvz_selftest_bounded_wait(uint64_t limit_ns, uint32_t *status, uint64_t *out, kvz_stream_t stream)
{
    if (!status || !out) return KVZ_ERR_INVALID_ARG;
    if (!aligned(status, 4) || !aligned(out, 8)) return KVZ_ERR_ALIGNMENT;
    if (limit_ns == 0 || limit_ns > 10000000000ull) return KVZ_ERR_INVALID_ARG;  // (0, 10 s]
    cudaError_t e = launch_wait_selftest(limit_ns, status, out, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVZ_OK : fail_cuda(e);
}

// ---------------------------------------------------------------------------------
// FP8 tiles
// ---------------------------------------------------------------------------------
static bool f8_format_ok(int32_t f) { return f == KVZ_F8_E4M3 || f == KVZ_F8_E5M2; }

int kvz_f8_calibrate(kvz_dims dims, int32_t format, const void *raw_pool, int64_t num_raw_pages, const int32_t *pages,
                     int32_t n, uint8_t *bases, uint32_t *status, kvz_stream_t stream)
{
    if (!f8_format_ok(format)) return KVZ_ERR_INVALID_ARG;
    if (!dims_ok(dims)) return dims.num_kv_heads >= 1 ? KVZ_ERR_UNSUPPORTED : KVZ_ERR_INVALID_ARG;
    if (n < 0 || num_raw_pages < 0) return KVZ_ERR_INVALID_ARG;
    if (!bases || !status || (n > 0 && (!raw_pool || !pages))) return KVZ_ERR_INVALID_ARG;
    if (!aligned(raw_pool, 16) || !aligned(pages, 4) || !aligned(status, 4)) return KVZ_ERR_ALIGNMENT;
    if (dims.num_kv_heads > (1 << 20)) return KVZ_ERR_UNSUPPORTED;
    cudaError_t e = launch_f8_calibrate(format, dims.num_kv_heads, static_cast<const uint16_t *>(raw_pool),
                                        num_raw_pages, pages, n, bases, status, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVZ_OK : fail_cuda(e);
}

int kvz_f8_encode_pages(kvz_dims dims, int32_t format, const void *raw_pool, int64_t num_raw_pages,
                        const uint8_t *bases, const int32_t *src_page, const int32_t *dst_page, const int32_t *dst_seq,
                        int32_t n, uint32_t *meta, int64_t num_meta_pages, uint8_t *arena, uint64_t arena_bytes,
                        uint32_t *cursors, int32_t num_cursors, void *workspace, size_t workspace_bytes,
                        uint32_t *status, kvz_stream_t stream)
{
    if (!f8_format_ok(format)) return KVZ_ERR_INVALID_ARG;
    if (!dims_ok(dims)) return dims.num_kv_heads >= 1 ? KVZ_ERR_UNSUPPORTED : KVZ_ERR_INVALID_ARG;
    if (n < 0 || num_raw_pages < 0 || num_meta_pages < 0 || num_cursors < 0) return KVZ_ERR_INVALID_ARG;
    if (n == 0) return KVZ_OK;
    if (!raw_pool || !bases || !src_page || !dst_page || !dst_seq || !meta || !arena || !cursors || !workspace ||
        !status)
        return KVZ_ERR_INVALID_ARG;
    if (!aligned(raw_pool, 16) || !aligned(bases, 16) || !aligned(meta, 8) || !aligned(arena, 64) ||
        !aligned(cursors, 8) || !aligned(workspace, 16) || !aligned(status, 4))
        return KVZ_ERR_ALIGNMENT;
    if ((int64_t)n * dims.num_kv_heads > (int64_t)1 << 30) return KVZ_ERR_UNSUPPORTED;
    if (workspace_bytes < kvz_encode_workspace_size(dims, n)) return KVZ_ERR_WORKSPACE;
    EncodeParams P;
    memset(&P, 0, sizeof P);
    P.hkv = dims.num_kv_heads;
    P.n = n;
    P.raw_pool = static_cast<const uint16_t *>(raw_pool);
    P.num_raw_pages = num_raw_pages;
    P.src_page = src_page;
    P.dst_page = dst_page;
    P.dst_seq = dst_seq;
    P.meta32 = meta;
    P.ga_bases = bases;
    P.num_meta_pages = num_meta_pages;
    P.arena = arena;
    P.arena_bytes = arena_bytes;
    P.cursors = cursors;
    P.num_cursors = num_cursors;
    P.status = status;
    uint8_t *w = static_cast<uint8_t *>(workspace);
    const size_t a = ((size_t)n * 4 + 15) / 16 * 16;
    P.ws_hdr = reinterpret_cast<uint32_t *>(w);
    P.ws_page_size = reinterpret_cast<uint32_t *>(w + 16);
    P.ws_page_base = reinterpret_cast<uint32_t *>(w + 16 + a);
    P.ws_pair_size = reinterpret_cast<uint32_t *>(w + 16 + 2 * a);
    P.ws_tags = reinterpret_cast<uint64_t *>(w + encode_ws_tags_offset(n, dims.num_kv_heads));
    cudaError_t e = launch_f8_encode(format, P, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVZ_OK : fail_cuda(e);
}

int kvz_f8_decode_blocks(kvz_dims dims, int32_t format, const uint32_t *meta, int64_t num_meta_pages,
                         const uint8_t *arena, uint64_t arena_bytes, const uint8_t *bases, const int32_t *page,
                         int32_t n, void *out_pages, uint32_t *status, kvz_stream_t stream)
{
    if (!f8_format_ok(format)) return KVZ_ERR_INVALID_ARG;
    if (!dims_ok(dims)) return dims.num_kv_heads >= 1 ? KVZ_ERR_UNSUPPORTED : KVZ_ERR_INVALID_ARG;
    if (n < 0 || num_meta_pages < 0) return KVZ_ERR_INVALID_ARG;
    if (n == 0) return KVZ_OK;
    if (!meta || !arena || !bases || !page || !out_pages || !status) return KVZ_ERR_INVALID_ARG;
    if (!aligned(meta, 4) || !aligned(arena, 64) || !aligned(out_pages, 16) || !aligned(status, 4) ||
        !aligned(bases, 2))
        return KVZ_ERR_ALIGNMENT;
    if ((int64_t)n * dims.num_kv_heads > (int64_t)1 << 30) return KVZ_ERR_UNSUPPORTED;
    DecodeParams P;
    memset(&P, 0, sizeof P);
    P.hkv = dims.num_kv_heads;
    P.n = n;
    P.meta32 = meta;
    P.ga_bases = bases;
    P.num_meta_pages = num_meta_pages;
    P.arena = arena;
    P.arena_bytes = arena_bytes;
    P.page = page;
    P.out = static_cast<uint16_t *>(out_pages);
    P.status = status;
    cudaError_t e = launch_f8_decode(format, P, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVZ_OK : fail_cuda(e);
}

int kvz_f8_decode_attention(kvz_dims dims, int32_t format, int32_t batch, int32_t num_q_heads, const void *q,
                            const int32_t *page_ids, int32_t max_pages, const int32_t *seq_lens,
                            const int32_t *tail_page, const uint32_t *meta, int64_t num_meta_pages,
                            const uint8_t *arena, uint64_t arena_bytes, const uint8_t *bases, const void *raw_pool,
                            int64_t num_raw_pages, float *out, void *workspace, size_t workspace_bytes,
                            uint32_t *status, kvz_stream_t stream)
{
    if (!f8_format_ok(format)) return KVZ_ERR_INVALID_ARG;
    int rc = check_attention_common(dims, batch, num_q_heads, q, seq_lens, raw_pool, num_raw_pages, out, workspace,
                                    status, max_pages, page_ids);
    if (rc || batch == 0) return rc;
    if (!tail_page || !meta || !arena || !bases || num_meta_pages < 0) return KVZ_ERR_INVALID_ARG;
    if (!aligned(meta, 8) || !aligned(arena, 64) || !aligned(tail_page, 4) || !aligned(bases, 2))
        return KVZ_ERR_ALIGNMENT;
    const int fmt = format == KVZ_F8_E4M3 ? kFmtF8E4 : kFmtF8E5;
    return run_attention(FormatArgs{fmt, nullptr, meta, bases}, dims, batch, num_q_heads, q, page_ids, max_pages,
                         seq_lens, tail_page, num_meta_pages, arena, arena_bytes, raw_pool, num_raw_pages, out,
                         workspace, workspace_bytes, status, reinterpret_cast<cudaStream_t>(stream));
}

int kvz_apply_cursor_updates(const int32_t *idx, const uint32_t *pos, const uint32_t *end, int32_t n,
                             uint32_t *cursors, int32_t num_cursors, kvz_stream_t stream)
{
    if (n < 0 || num_cursors < 0) return KVZ_ERR_INVALID_ARG;
    if (n == 0) return KVZ_OK;
    if (!idx || !pos || !end || !cursors) return KVZ_ERR_INVALID_ARG;
    cudaError_t e = launch_apply_cursor_updates(idx, pos, end, n, cursors, num_cursors,
                                                reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KVZ_OK : fail_cuda(e);
}

}  // extern "C"
