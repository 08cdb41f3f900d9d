// Cold-page codec for sm_103a: offload (quantize a batch of hot 16-bit pages and write their
// cold blocks in the same pass) and onboard (read cold blocks and write the dequantized hot
// pages in the same pass) ("KV Cache Compression in TensorRT LLM", NVIDIA: "NVFP4 Cold-Page
// Compression", "How It Works", Figure 6 and Figure 7: encode is fused into the offload copy,
// decode into the onboard copy, one fixed-size block per page).
//
// The cold pool is usually pinned host memory reached over the host link, so the kernels are
// shaped for that link: every store to (and load from) the cold block is a whole-warp run of
// contiguous bytes, and the block scales, one byte per 16 values, are gathered in shared memory
// and moved as 16-byte vectors instead of single bytes. Numerics are those of the page codec:
// the same block encode (codec_core.cuh) and the same exact FP16 decode products.
//
// Work items: (page, tensor, chunk of kChunk blocks) for K and V, then (page, chunk of
// kExtraChunk bytes) for the lossless part. A CTA takes items in a grid-stride loop.
#include <cstdint>
#include <cuda_runtime.h>

#include "codec_core.cuh"
#include "common.cuh"
#include "host_util.h"

namespace nvfp4kv {
namespace {

constexpr int kColdThreads = 256;
constexpr int kColdUnits = 8;                          // blocks per thread per item
constexpr int kChunk = kColdThreads * kColdUnits;      // blocks per item (2048)
constexpr int kExtraVecs = 4;                          // 16-byte vectors per thread per item
constexpr int kExtraChunk = kColdThreads * 16 * kExtraVecs;

struct ColdParams {
    const uint8_t* hot[2];      // K and V hot pools (bytes); onboard writes through them
    int64_t hot_stride;         // bytes between consecutive hot pages
    int32_t hot_pool;
    const int32_t* hot_ids;
    const float* g[2];          // NULL: 1
    uint8_t* extra;             // lossless bytes of each hot page
    int64_t extra_stride;
    int32_t extra_bytes;
    uint8_t* cold;
    int64_t block_bytes;        // one cold block
    int64_t off_data[2];        // offsets of the K / V parts in a block
    int64_t off_scales[2];
    int64_t off_extra;
    int32_t cold_slots;
    const int32_t* cold_ids;
    int32_t bpp;                // 16-value blocks per page per tensor
    int32_t chunks;             // ceil(bpp / kChunk)
    int32_t extra_items;        // ceil(extra_bytes / kExtraChunk)
    int32_t num_pages;
    int32_t* status;
};

struct ItemPos {
    int32_t page;     // index into the batch
    int32_t tensor;   // 0 K, 1 V, 2 extra
    int32_t chunk;
};

__device__ __forceinline__ ItemPos item_pos(const ColdParams& p, int64_t item) {
    const int32_t per_page = 2 * p.chunks + p.extra_items;
    ItemPos r;
    r.page = static_cast<int32_t>(item / per_page);
    const int32_t q = static_cast<int32_t>(item - static_cast<int64_t>(r.page) * per_page);
    if (q < 2 * p.chunks) {
        r.tensor = q >= p.chunks ? 1 : 0;
        r.chunk = q - r.tensor * p.chunks;
    } else {
        r.tensor = 2;
        r.chunk = q - 2 * p.chunks;
    }
    return r;
}

// Bounds of the item's page ids; false (and the status bit) when either is outside its pool.
__device__ __forceinline__ bool item_pages(const ColdParams& p, int32_t i, int32_t& hp,
                                           int32_t& cs) {
    hp = p.hot_ids ? __ldg(p.hot_ids + i) : i;
    cs = p.cold_ids ? __ldg(p.cold_ids + i) : i;
    if (hp < 0 || hp >= p.hot_pool || cs < 0 || cs >= p.cold_slots) {
        if (threadIdx.x == 0) flag_status(p.status, NVFP4KV_STATUS_PAGE_OOB);
        return false;
    }
    return true;
}

// Copy n bytes (n a multiple of 16, both ends 16-byte aligned) of one extra chunk.
__device__ __forceinline__ void copy_extra(const uint8_t* src, uint8_t* dst, int32_t n) {
    uint4 v[kExtraVecs];
#pragma unroll
    for (int u = 0; u < kExtraVecs; ++u) {
        const int32_t o = (u * kColdThreads + static_cast<int32_t>(threadIdx.x)) * 16;
        if (o < n) v[u] = *reinterpret_cast<const uint4*>(src + o);
    }
#pragma unroll
    for (int u = 0; u < kExtraVecs; ++u) {
        const int32_t o = (u * kColdThreads + static_cast<int32_t>(threadIdx.x)) * 16;
        if (o < n) *reinterpret_cast<uint4*>(dst + o) = v[u];
    }
}

// Offload. SRC: NVFP4KV_BF16 or NVFP4KV_FP16.
template <int SRC>
__global__ void __launch_bounds__(kColdThreads) cold_offload_kernel(const ColdParams p) {
    __shared__ __align__(16) uint8_t s_sc[kChunk];
    const float gk = p.g[0] ? __ldg(p.g[0]) : 1.0f;
    const float gv = p.g[1] ? __ldg(p.g[1]) : 1.0f;
    const int64_t total = static_cast<int64_t>(p.num_pages) * (2 * p.chunks + p.extra_items);
    for (int64_t item = blockIdx.x; item < total; item += gridDim.x) {
        const ItemPos ip = item_pos(p, item);
        int32_t hp, cs;
        if (!item_pages(p, ip.page, hp, cs)) continue;
        uint8_t* const blk_base = p.cold + static_cast<int64_t>(cs) * p.block_bytes;
        if (ip.tensor == 2) {
            const int32_t o = ip.chunk * kExtraChunk;
            copy_extra(p.extra + static_cast<int64_t>(hp) * p.extra_stride + o,
                       blk_base + p.off_extra + o, min(kExtraChunk, p.extra_bytes - o));
            continue;
        }
        const int t = ip.tensor;
        const float g = t ? gv : gk;
        const float d = __fmul_rn(6.0f, g);
        const uint8_t* src = p.hot[t] + static_cast<int64_t>(hp) * p.hot_stride;
        const int32_t b0 = ip.chunk * kChunk;
        const int32_t n = min(kChunk, p.bpp - b0);
        U8x32 raw[kColdUnits];
#pragma unroll
        for (int u = 0; u < kColdUnits; ++u) {
            const int32_t b = u * kColdThreads + static_cast<int32_t>(threadIdx.x);
            if (b < n) raw[u] = load_raw<SRC, false>(src, b0 + b);
        }
        uint8_t* const data = blk_base + p.off_data[t] + static_cast<int64_t>(b0) * 8;
#pragma unroll
        for (int u = 0; u < kColdUnits; ++u) {
            const int32_t b = u * kColdThreads + static_cast<int32_t>(threadIdx.x);
            if (b >= n) continue;
            float x[16];
            widen<SRC>(raw[u], 1.0f, x);
            uint32_t sb;
            float r;
            pick_scale(x, g, d, sb, r);
            uint32_t w0 = 0u, w1 = 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                w0 |= f32x2_to_e2m1x2(__fmul_rn(x[2 * j], r), __fmul_rn(x[2 * j + 1], r)) << (8 * j);
                w1 |= f32x2_to_e2m1x2(__fmul_rn(x[8 + 2 * j], r), __fmul_rn(x[9 + 2 * j], r))
                      << (8 * j);
            }
            *reinterpret_cast<uint2*>(data + static_cast<int64_t>(b) * 8) = make_uint2(w0, w1);
            s_sc[b] = static_cast<uint8_t>(sb);
        }
        __syncthreads();
        // the chunk's scales are n contiguous bytes of the block: 16-byte stores, then the tail
        uint8_t* const sdst = blk_base + p.off_scales[t] + b0;
        const int32_t nv = n >> 4;
        for (int32_t v = threadIdx.x; v < nv; v += kColdThreads)
            *reinterpret_cast<uint4*>(sdst + v * 16) = *reinterpret_cast<const uint4*>(s_sc + v * 16);
        for (int32_t j = nv * 16 + static_cast<int32_t>(threadIdx.x); j < n; j += kColdThreads)
            sdst[j] = s_sc[j];
        __syncthreads();
    }
}

// Onboard. DST: NVFP4KV_BF16 or NVFP4KV_FP16. v = e2m1 * e4m3 is exact in FP16; the output is
// the 16-bit rounding of fp32(v * g).
template <int DST>
__global__ void __launch_bounds__(kColdThreads) cold_onboard_kernel(const ColdParams p) {
    __shared__ __align__(16) uint8_t s_sc[kChunk];
    const float gk = p.g[0] ? __ldg(p.g[0]) : 1.0f;
    const float gv = p.g[1] ? __ldg(p.g[1]) : 1.0f;
    const int64_t total = static_cast<int64_t>(p.num_pages) * (2 * p.chunks + p.extra_items);
    for (int64_t item = blockIdx.x; item < total; item += gridDim.x) {
        const ItemPos ip = item_pos(p, item);
        int32_t hp, cs;
        if (!item_pages(p, ip.page, hp, cs)) continue;
        const uint8_t* const blk_base = p.cold + static_cast<int64_t>(cs) * p.block_bytes;
        if (ip.tensor == 2) {
            const int32_t o = ip.chunk * kExtraChunk;
            copy_extra(blk_base + p.off_extra + o,
                       p.extra + static_cast<int64_t>(hp) * p.extra_stride + o,
                       min(kExtraChunk, p.extra_bytes - o));
            continue;
        }
        const int t = ip.tensor;
        const float g = t ? gv : gk;
        const int32_t b0 = ip.chunk * kChunk;
        const int32_t n = min(kChunk, p.bpp - b0);
        const uint8_t* const data = blk_base + p.off_data[t] + static_cast<int64_t>(b0) * 8;
        uint2 code[kColdUnits];
#pragma unroll
        for (int u = 0; u < kColdUnits; ++u) {
            const int32_t b = u * kColdThreads + static_cast<int32_t>(threadIdx.x);
            if (b < n) code[u] = *reinterpret_cast<const uint2*>(data + static_cast<int64_t>(b) * 8);
        }
        const uint8_t* const ssrc = blk_base + p.off_scales[t] + b0;
        const int32_t nv = n >> 4;
        for (int32_t v = threadIdx.x; v < nv; v += kColdThreads)
            *reinterpret_cast<uint4*>(s_sc + v * 16) = *reinterpret_cast<const uint4*>(ssrc + v * 16);
        for (int32_t j = nv * 16 + static_cast<int32_t>(threadIdx.x); j < n; j += kColdThreads)
            s_sc[j] = ssrc[j];
        __syncthreads();
        uint8_t* const dst = const_cast<uint8_t*>(p.hot[t]) + static_cast<int64_t>(hp) * p.hot_stride;
#pragma unroll
        for (int u = 0; u < kColdUnits; ++u) {
            const int32_t b = u * kColdThreads + static_cast<int32_t>(threadIdx.x);
            if (b >= n) continue;
            const uint32_t s2 = e4m3x2_to_f16x2(static_cast<uint32_t>(s_sc[b]) * 0x0101u);
            uint32_t v[8];
            e2m1x8_to_f16x2x4(code[u].x, *reinterpret_cast<uint32_t(*)[4]>(v));
            e2m1x8_to_f16x2x4(code[u].y, *reinterpret_cast<uint32_t(*)[4]>(v + 4));
            uint32_t o[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t e = hmul2_u32(v[j], s2);
                const float lo = __fmul_rn(f16_lo(e), g), hi = __fmul_rn(f16_hi(e), g);
                o[j] = (DST == NVFP4KV_BF16) ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
            }
            uint8_t* q = dst + static_cast<int64_t>(b0 + b) * 32;
            *reinterpret_cast<uint4*>(q) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(q + 16) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        __syncthreads();
    }
}

inline int64_t round16(int64_t x) { return (x + 15) & ~int64_t{15}; }

bool cold_layout(const nvfp4kv_layout* l, int32_t extra_bytes, nvfp4kv_cold_block_layout* o) {
    if (!layout_ok(l) || extra_bytes < 0 || (extra_bytes & 15)) return false;
    const int64_t vals = static_cast<int64_t>(l->num_kv_heads) * l->page_size * l->head_dim;
    const int64_t db = vals / 2, sb = vals / 16;
    o->k_data = 0;
    o->k_scales = round16(db);
    o->v_data = o->k_scales + round16(sb);
    o->v_scales = o->v_data + round16(db);
    o->extra = o->v_scales + round16(sb);
    o->bytes = o->extra + extra_bytes;
    return true;
}

// Shared validation and parameter setup of both directions; returns OK or the error.
nvfp4kv_status setup(ColdParams& p, const nvfp4kv_layout* layout, nvfp4kv_dtype hot_dtype,
                     const void* hot_k, const void* hot_v, int64_t hot_page_stride,
                     int32_t hot_pool_pages, const int32_t* hot_page_ids, const float* gk,
                     const float* gv, const uint8_t* extra, int64_t extra_page_stride,
                     int32_t extra_bytes, const uint8_t* cold, int32_t cold_slots,
                     const int32_t* cold_slot_ids, int32_t num_pages, int32_t* status) {
    nvfp4kv_cold_block_layout bl;
    if (!cold_layout(layout, extra_bytes, &bl) || num_pages < 0 || hot_pool_pages < 0 ||
        cold_slots < 0)
        return NVFP4KV_ERR_INVALID_ARG;
    if (hot_dtype != NVFP4KV_BF16 && hot_dtype != NVFP4KV_FP16) return NVFP4KV_ERR_UNSUPPORTED;
    const int64_t vals = static_cast<int64_t>(layout->num_kv_heads) * layout->page_size *
                         layout->head_dim;
    if (vals / 16 > (int64_t{1} << 30)) return NVFP4KV_ERR_UNSUPPORTED;
    if (num_pages == 0) return NVFP4KV_OK;
    if (!hot_k || !hot_v || !cold || !aligned16(hot_k) || !aligned16(hot_v) || !aligned16(cold) ||
        hot_page_stride < vals || (hot_page_stride & 7))
        return NVFP4KV_ERR_INVALID_ARG;
    if (extra_bytes > 0 &&
        (!extra || !aligned16(extra) || extra_page_stride < extra_bytes || (extra_page_stride & 15)))
        return NVFP4KV_ERR_INVALID_ARG;
    if ((!hot_page_ids && hot_pool_pages < num_pages) || (!cold_slot_ids && cold_slots < num_pages))
        return NVFP4KV_ERR_INVALID_ARG;
    p = ColdParams{};
    p.hot[0] = static_cast<const uint8_t*>(hot_k);
    p.hot[1] = static_cast<const uint8_t*>(hot_v);
    p.hot_stride = hot_page_stride * 2;
    p.hot_pool = hot_pool_pages;
    p.hot_ids = hot_page_ids;
    p.g[0] = gk;
    p.g[1] = gv;
    p.extra = const_cast<uint8_t*>(extra);
    p.extra_stride = extra_page_stride;
    p.extra_bytes = extra_bytes;
    p.cold = const_cast<uint8_t*>(cold);
    p.block_bytes = bl.bytes;
    p.off_data[0] = bl.k_data;
    p.off_data[1] = bl.v_data;
    p.off_scales[0] = bl.k_scales;
    p.off_scales[1] = bl.v_scales;
    p.off_extra = bl.extra;
    p.cold_slots = cold_slots;
    p.cold_ids = cold_slot_ids;
    p.bpp = static_cast<int32_t>(vals / 16);
    p.chunks = (p.bpp + kChunk - 1) / kChunk;
    p.extra_items = (extra_bytes + kExtraChunk - 1) / kExtraChunk;
    p.num_pages = num_pages;
    p.status = status;
    return NVFP4KV_OK;
}

int cold_grid(const ColdParams& p) {
    const int64_t items = static_cast<int64_t>(p.num_pages) * (2 * p.chunks + p.extra_items);
    const int64_t cap = static_cast<int64_t>(num_sms()) * 4;
    return static_cast<int>(items < cap ? (items < 1 ? 1 : items) : cap);
}

}  // namespace
}  // namespace nvfp4kv

using namespace nvfp4kv;

extern "C" nvfp4kv_status nvfp4_kv_cold_block_layout(const nvfp4kv_layout* layout,
                                                     int32_t extra_bytes,
                                                     nvfp4kv_cold_block_layout* out) {
    if (!out) return NVFP4KV_ERR_INVALID_ARG;
    return cold_layout(layout, extra_bytes, out) ? NVFP4KV_OK : NVFP4KV_ERR_INVALID_ARG;
}

extern "C" nvfp4kv_status nvfp4_kv_offload_pages(
    const nvfp4kv_layout* layout, nvfp4kv_dtype hot_dtype, const void* hot_k, const void* hot_v,
    int64_t hot_page_stride, int32_t hot_pool_pages, const int32_t* hot_page_ids,
    const float* k_global_scale, const float* v_global_scale, const uint8_t* extra,
    int64_t extra_page_stride, int32_t extra_bytes, uint8_t* cold, int32_t cold_slots,
    const int32_t* cold_slot_ids, int32_t num_pages, int32_t* status, nvfp4kv_stream_t stream) {
    ColdParams p;
    const nvfp4kv_status st =
        setup(p, layout, hot_dtype, hot_k, hot_v, hot_page_stride, hot_pool_pages, hot_page_ids,
              k_global_scale, v_global_scale, extra, extra_page_stride, extra_bytes, cold,
              cold_slots, cold_slot_ids, num_pages, status);
    if (st != NVFP4KV_OK || num_pages == 0) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (hot_dtype == NVFP4KV_BF16)
        cold_offload_kernel<NVFP4KV_BF16><<<cold_grid(p), kColdThreads, 0, s>>>(p);
    else
        cold_offload_kernel<NVFP4KV_FP16><<<cold_grid(p), kColdThreads, 0, s>>>(p);
    return launch_status();
}

extern "C" nvfp4kv_status nvfp4_kv_onboard_pages(
    const nvfp4kv_layout* layout, const uint8_t* cold, int32_t cold_slots,
    const int32_t* cold_slot_ids, const float* k_global_scale, const float* v_global_scale,
    nvfp4kv_dtype hot_dtype, void* hot_k, void* hot_v, int64_t hot_page_stride,
    int32_t hot_pool_pages, const int32_t* hot_page_ids, uint8_t* extra,
    int64_t extra_page_stride, int32_t extra_bytes, int32_t num_pages, int32_t* status,
    nvfp4kv_stream_t stream) {
    ColdParams p;
    const nvfp4kv_status st =
        setup(p, layout, hot_dtype, hot_k, hot_v, hot_page_stride, hot_pool_pages, hot_page_ids,
              k_global_scale, v_global_scale, extra, extra_page_stride, extra_bytes, cold,
              cold_slots, cold_slot_ids, num_pages, status);
    if (st != NVFP4KV_OK || num_pages == 0) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (hot_dtype == NVFP4KV_BF16)
        cold_onboard_kernel<NVFP4KV_BF16><<<cold_grid(p), kColdThreads, 0, s>>>(p);
    else
        cold_onboard_kernel<NVFP4KV_FP16><<<cold_grid(p), kColdThreads, 0, s>>>(p);
    return launch_status();
}

extern "C" nvfp4kv_status nvfp4_kv_host_device_pointer(void* host_ptr, void** device_ptr) {
    if (!host_ptr || !device_ptr) return NVFP4KV_ERR_INVALID_ARG;
    *device_ptr = nullptr;
    if (cudaHostGetDevicePointer(device_ptr, host_ptr, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        return NVFP4KV_ERR_INVALID_ARG;
    }
    return NVFP4KV_OK;
}
