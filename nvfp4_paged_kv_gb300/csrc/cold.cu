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
// kExtraChunk bytes) for the lossless part. A CTA takes items in a grid-stride loop. When the
// RoPE part of K is kept apart (the same page, "The RoPE part of K": kept at 16 bits, or two
// NVFP4 components of which the second encodes the first one's rounding error), K is cut into
// items of whole token rows instead, a multiple of 16 rows, so that each of K's split scale
// regions starts on a 16-byte boundary in every item.
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
    // RoPE part of K (rope_mode != 0): blocks [rb, rb + nbr) of each row of nb blocks
    int32_t rope_mode, nb, rb, nbr, nbn, rows, rows_per_item, k_items;
    uint64_t nb_magic;
    int64_t off_rope, off_rope_s, off_rope2, off_rope2_s;
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

// Items of a page: K (k_items), V (chunks), extra (extra_items).
__device__ __forceinline__ ItemPos item_pos(const ColdParams& p, int64_t item) {
    const int32_t per_page = p.k_items + p.chunks + p.extra_items;
    ItemPos r;
    r.page = static_cast<int32_t>(item / per_page);
    const int32_t q = static_cast<int32_t>(item - static_cast<int64_t>(r.page) * per_page);
    if (q < p.k_items) {
        r.tensor = 0;
        r.chunk = q;
    } else if (q < p.k_items + p.chunks) {
        r.tensor = 1;
        r.chunk = q - p.k_items;
    } else {
        r.tensor = 2;
        r.chunk = q - p.k_items - p.chunks;
    }
    return r;
}

// Copy n bytes of shared memory to dst (dst 16-byte aligned): 16-byte stores, then the tail.
__device__ __forceinline__ void smem_to_global(uint8_t* dst, const uint8_t* s, int32_t n) {
    const int32_t nv = n >> 4;
    for (int32_t v = threadIdx.x; v < nv; v += kColdThreads)
        *reinterpret_cast<uint4*>(dst + v * 16) = *reinterpret_cast<const uint4*>(s + v * 16);
    for (int32_t j = nv * 16 + static_cast<int32_t>(threadIdx.x); j < n; j += kColdThreads)
        dst[j] = s[j];
}
// The reverse (src 16-byte aligned).
__device__ __forceinline__ void global_to_smem(uint8_t* s, const uint8_t* src, int32_t n) {
    const int32_t nv = n >> 4;
    for (int32_t v = threadIdx.x; v < nv; v += kColdThreads)
        *reinterpret_cast<uint4*>(s + v * 16) = *reinterpret_cast<const uint4*>(src + v * 16);
    for (int32_t j = nv * 16 + static_cast<int32_t>(threadIdx.x); j < n; j += kColdThreads)
        s[j] = src[j];
}

// Where block col of a row goes: the other dims (index within the row's N/16 blocks) or the
// RoPE dims (index within the row's R/16 blocks).
__device__ __forceinline__ bool rope_col(const ColdParams& p, int32_t col, int32_t& idx) {
    if (col >= p.rb && col < p.rb + p.nbr) {
        idx = col - p.rb;
        return true;
    }
    idx = col < p.rb ? col : col - p.nbr;
    return false;
}

// Offload of one K item of whole rows when the RoPE part is kept apart (MODE 1: 16-bit copy,
// MODE 2: two NVFP4 components).
template <int SRC, int MODE>
__device__ __forceinline__ void offload_k_rows(const ColdParams& p, uint8_t* blk_base,
                                               const uint8_t* src, float g, int32_t chunk,
                                               uint8_t* s_n, uint8_t* s_r1, uint8_t* s_r2) {
    const float d = __fmul_rn(6.0f, g);
    const int32_t row0 = chunk * p.rows_per_item;
    const int32_t nrows = min(p.rows_per_item, p.rows - row0);
    const int32_t nblk = nrows * p.nb;
    uint8_t* const kd = blk_base + p.off_data[0] + static_cast<int64_t>(row0) * p.nbn * 8;
    uint8_t* const kr = blk_base + p.off_rope +
                        static_cast<int64_t>(row0) * p.nbr * (MODE == NVFP4KV_ROPE_SKIP ? 32 : 8);
    uint8_t* const kr2 = blk_base + p.off_rope2 + static_cast<int64_t>(row0) * p.nbr * 8;
    for (int32_t b = threadIdx.x; b < nblk; b += kColdThreads) {
        const int32_t r = static_cast<int32_t>(fast_div(static_cast<uint32_t>(b), p.nb_magic));
        const int32_t col = b - r * p.nb;
        const int64_t sblk = static_cast<int64_t>(row0) * p.nb + b;
        int32_t idx;
        const bool rope = rope_col(p, col, idx);
        if (rope && MODE == NVFP4KV_ROPE_SKIP) {
            const uint8_t* a = src + sblk * 32;
            const uint4 lo = ld_stream_16B(a), hi = ld_stream_16B(a + 16);
            uint8_t* q = kr + static_cast<int64_t>(r * p.nbr + idx) * 32;
            *reinterpret_cast<uint4*>(q) = lo;
            *reinterpret_cast<uint4*>(q + 16) = hi;
            continue;
        }
        float x[16];
        widen<SRC>(load_raw<SRC, false>(src, sblk), 1.0f, x);
        uint32_t sb;
        float rcp;
        pick_scale(x, g, d, sb, rcp);
        const uint2 c1 = pack_e2m1_block(x, rcp);
        if (!rope) {
            const int32_t ni = r * p.nbn + idx;
            *reinterpret_cast<uint2*>(kd + static_cast<int64_t>(ni) * 8) = c1;
            s_n[ni] = static_cast<uint8_t>(sb);
            continue;
        }
        if constexpr (MODE == NVFP4KV_ROPE_2FP4) {
            // second component: the first one's rounding error r = fp32(x - fp32(v1 g))
            float v1[16], res[16];
            block_values(c1, sb, v1);
#pragma unroll
            for (int k = 0; k < 16; ++k) res[k] = __fsub_rn(x[k], __fmul_rn(v1[k], g));
            uint32_t sb2;
            float rcp2;
            pick_scale(res, g, d, sb2, rcp2);
            const uint2 c2 = pack_e2m1_block(res, rcp2);
            const int32_t ri = r * p.nbr + idx;
            *reinterpret_cast<uint2*>(kr + static_cast<int64_t>(ri) * 8) = c1;
            *reinterpret_cast<uint2*>(kr2 + static_cast<int64_t>(ri) * 8) = c2;
            s_r1[ri] = static_cast<uint8_t>(sb);
            s_r2[ri] = static_cast<uint8_t>(sb2);
        }
    }
    __syncthreads();
    smem_to_global(blk_base + p.off_scales[0] + static_cast<int64_t>(row0) * p.nbn, s_n,
                   nrows * p.nbn);
    if constexpr (MODE == NVFP4KV_ROPE_2FP4) {
        smem_to_global(blk_base + p.off_rope_s + static_cast<int64_t>(row0) * p.nbr, s_r1,
                       nrows * p.nbr);
        smem_to_global(blk_base + p.off_rope2_s + static_cast<int64_t>(row0) * p.nbr, s_r2,
                       nrows * p.nbr);
    }
    __syncthreads();
}

// Onboard of one K item of whole rows when the RoPE part is kept apart.
template <int DST, int MODE>
__device__ __forceinline__ void onboard_k_rows(const ColdParams& p, const uint8_t* blk_base,
                                               uint8_t* dst, float g, int32_t chunk,
                                               uint8_t* s_n, uint8_t* s_r1, uint8_t* s_r2) {
    const int32_t row0 = chunk * p.rows_per_item;
    const int32_t nrows = min(p.rows_per_item, p.rows - row0);
    const int32_t nblk = nrows * p.nb;
    global_to_smem(s_n, blk_base + p.off_scales[0] + static_cast<int64_t>(row0) * p.nbn,
                   nrows * p.nbn);
    if constexpr (MODE == NVFP4KV_ROPE_2FP4) {
        global_to_smem(s_r1, blk_base + p.off_rope_s + static_cast<int64_t>(row0) * p.nbr,
                       nrows * p.nbr);
        global_to_smem(s_r2, blk_base + p.off_rope2_s + static_cast<int64_t>(row0) * p.nbr,
                       nrows * p.nbr);
    }
    __syncthreads();
    const uint8_t* const kd = blk_base + p.off_data[0] + static_cast<int64_t>(row0) * p.nbn * 8;
    const uint8_t* const kr = blk_base + p.off_rope +
                              static_cast<int64_t>(row0) * p.nbr * (MODE == NVFP4KV_ROPE_SKIP ? 32 : 8);
    const uint8_t* const kr2 = blk_base + p.off_rope2 + static_cast<int64_t>(row0) * p.nbr * 8;
    for (int32_t b = threadIdx.x; b < nblk; b += kColdThreads) {
        const int32_t r = static_cast<int32_t>(fast_div(static_cast<uint32_t>(b), p.nb_magic));
        const int32_t col = b - r * p.nb;
        uint8_t* const q = dst + (static_cast<int64_t>(row0) * p.nb + b) * 32;
        int32_t idx;
        const bool rope = rope_col(p, col, idx);
        float y[16];
        if (!rope) {
            const int32_t ni = r * p.nbn + idx;
            block_values(*reinterpret_cast<const uint2*>(kd + static_cast<int64_t>(ni) * 8), s_n[ni], y);
#pragma unroll
            for (int k = 0; k < 16; ++k) y[k] = __fmul_rn(y[k], g);
        } else if constexpr (MODE == NVFP4KV_ROPE_SKIP) {
            const uint8_t* a = kr + static_cast<int64_t>(r * p.nbr + idx) * 32;
            *reinterpret_cast<uint4*>(q) = *reinterpret_cast<const uint4*>(a);
            *reinterpret_cast<uint4*>(q + 16) = *reinterpret_cast<const uint4*>(a + 16);
            continue;
        } else {
            const int32_t ri = r * p.nbr + idx;
            float v2[16];
            block_values(*reinterpret_cast<const uint2*>(kr + static_cast<int64_t>(ri) * 8), s_r1[ri], y);
            block_values(*reinterpret_cast<const uint2*>(kr2 + static_cast<int64_t>(ri) * 8), s_r2[ri], v2);
#pragma unroll
            for (int k = 0; k < 16; ++k) y[k] = __fadd_rn(__fmul_rn(y[k], g), __fmul_rn(v2[k], g));
        }
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            o[j] = (DST == NVFP4KV_BF16) ? pack_bf16x2(y[2 * j], y[2 * j + 1])
                                         : pack_f16x2(y[2 * j], y[2 * j + 1]);
        st_global_32B(q, o);
    }
    __syncthreads();
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

// Offload. SRC: NVFP4KV_BF16 or NVFP4KV_FP16; MODE: how the RoPE part of K is kept.
template <int SRC, int MODE>
__global__ void __launch_bounds__(kColdThreads) cold_offload_kernel(const ColdParams p) {
    pdl_enter();
    __shared__ __align__(16) uint8_t s_sc[kChunk];
    __shared__ __align__(16) uint8_t s_r1[MODE == NVFP4KV_ROPE_2FP4 ? kChunk : 16];
    __shared__ __align__(16) uint8_t s_r2[MODE == NVFP4KV_ROPE_2FP4 ? kChunk : 16];
    const float gk = p.g[0] ? __ldg(p.g[0]) : 1.0f;
    const float gv = p.g[1] ? __ldg(p.g[1]) : 1.0f;
    const int64_t total =
        static_cast<int64_t>(p.num_pages) * (p.k_items + p.chunks + p.extra_items);
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
        if constexpr (MODE != NVFP4KV_ROPE_QUANTIZE) {
            if (t == 0) {
                offload_k_rows<SRC, MODE>(p, blk_base, src, g, ip.chunk, s_sc, s_r1, s_r2);
                continue;
            }
        }
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
template <int DST, int MODE>
__global__ void __launch_bounds__(kColdThreads) cold_onboard_kernel(const ColdParams p) {
    pdl_enter();
    __shared__ __align__(16) uint8_t s_sc[kChunk];
    __shared__ __align__(16) uint8_t s_r1[MODE == NVFP4KV_ROPE_2FP4 ? kChunk : 16];
    __shared__ __align__(16) uint8_t s_r2[MODE == NVFP4KV_ROPE_2FP4 ? kChunk : 16];
    const float gk = p.g[0] ? __ldg(p.g[0]) : 1.0f;
    const float gv = p.g[1] ? __ldg(p.g[1]) : 1.0f;
    const int64_t total =
        static_cast<int64_t>(p.num_pages) * (p.k_items + p.chunks + p.extra_items);
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
        if constexpr (MODE != NVFP4KV_ROPE_QUANTIZE) {
            if (t == 0) {
                onboard_k_rows<DST, MODE>(
                    p, blk_base, const_cast<uint8_t*>(p.hot[0]) + static_cast<int64_t>(hp) * p.hot_stride,
                    g, ip.chunk, s_sc, s_r1, s_r2);
                continue;
            }
        }
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
            st_global_32B(dst + static_cast<int64_t>(b0 + b) * 32, o);
        }
        __syncthreads();
    }
}

inline int64_t round16(int64_t x) { return (x + 15) & ~int64_t{15}; }

// RoPE option: mode, first dim, dims; false if malformed.
bool rope_ok(const nvfp4kv_layout* l, const nvfp4kv_cold_rope* r) {
    if (!r || r->mode == NVFP4KV_ROPE_QUANTIZE) return true;
    if (r->mode != NVFP4KV_ROPE_SKIP && r->mode != NVFP4KV_ROPE_2FP4) return false;
    return r->first_dim >= 0 && r->dims > 0 && (r->first_dim % 16) == 0 && (r->dims % 16) == 0 &&
           r->first_dim + r->dims <= l->head_dim && l->head_dim <= 2048;
}

bool cold_layout(const nvfp4kv_layout* l, const nvfp4kv_cold_rope* rope, int32_t extra_bytes,
                 nvfp4kv_cold_block_layout* o) {
    if (!layout_ok(l) || extra_bytes < 0 || (extra_bytes & 15) || !rope_ok(l, rope)) return false;
    const int mode = rope ? rope->mode : NVFP4KV_ROPE_QUANTIZE;
    const int64_t rows = static_cast<int64_t>(l->num_kv_heads) * l->page_size;
    const int64_t vals = rows * l->head_dim;
    const int64_t R = (mode == NVFP4KV_ROPE_QUANTIZE) ? 0 : rope->dims;
    const int64_t kvals = rows * (l->head_dim - R), rvals = rows * R;
    int64_t at = 0;
    auto part = [&](int64_t bytes) {
        const int64_t off = at;
        at = round16(at + bytes);
        return off;
    };
    o->k_data = part(kvals / 2);
    o->k_scales = part(kvals / 16);
    o->k_rope = o->k_rope_scales = o->k_rope2 = o->k_rope2_scales = -1;
    if (mode == NVFP4KV_ROPE_SKIP) {
        o->k_rope = part(rvals * 2);
    } else if (mode == NVFP4KV_ROPE_2FP4) {
        o->k_rope = part(rvals / 2);
        o->k_rope_scales = part(rvals / 16);
        o->k_rope2 = part(rvals / 2);
        o->k_rope2_scales = part(rvals / 16);
    }
    o->v_data = part(vals / 2);
    o->v_scales = part(vals / 16);
    o->extra = at;
    o->bytes = at + extra_bytes;
    return true;
}

// Shared validation and parameter setup of both directions; returns OK or the error.
nvfp4kv_status setup(ColdParams& p, const nvfp4kv_layout* layout, nvfp4kv_dtype hot_dtype,
                     const void* hot_k, const void* hot_v, int64_t hot_page_stride,
                     int32_t hot_pool_pages, const int32_t* hot_page_ids, const float* gk,
                     const float* gv, const nvfp4kv_cold_rope* rope, const uint8_t* extra,
                     int64_t extra_page_stride,
                     int32_t extra_bytes, const uint8_t* cold, int32_t cold_slots,
                     const int32_t* cold_slot_ids, int32_t num_pages, int32_t* status) {
    nvfp4kv_cold_block_layout bl;
    if (!cold_layout(layout, rope, extra_bytes, &bl) || num_pages < 0 || hot_pool_pages < 0 ||
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
    p.rope_mode = rope ? rope->mode : NVFP4KV_ROPE_QUANTIZE;
    p.nb = layout->head_dim / 16;
    p.nb_magic = div_magic(static_cast<uint32_t>(p.nb));
    p.rows = layout->num_kv_heads * layout->page_size;
    p.k_items = p.chunks;
    if (p.rope_mode != NVFP4KV_ROPE_QUANTIZE) {
        p.rb = rope->first_dim / 16;
        p.nbr = rope->dims / 16;
        p.nbn = p.nb - p.nbr;
        p.rows_per_item = max(16, (kChunk / p.nb) / 16 * 16);
        p.k_items = (p.rows + p.rows_per_item - 1) / p.rows_per_item;
        p.off_rope = bl.k_rope;
        p.off_rope_s = bl.k_rope_scales;
        p.off_rope2 = bl.k_rope2;
        p.off_rope2_s = bl.k_rope2_scales;
    }
    p.extra_items = (extra_bytes + kExtraChunk - 1) / kExtraChunk;
    p.num_pages = num_pages;
    p.status = status;
    return NVFP4KV_OK;
}

int cold_grid(const ColdParams& p) {
    const int64_t items =
        static_cast<int64_t>(p.num_pages) * (p.k_items + p.chunks + p.extra_items);
    const int64_t cap = static_cast<int64_t>(num_sms()) * 4;
    return static_cast<int>(items < cap ? (items < 1 ? 1 : items) : cap);
}

}  // namespace
}  // namespace nvfp4kv

using namespace nvfp4kv;

extern "C" nvfp4kv_status nvfp4_kv_cold_block_layout(const nvfp4kv_layout* layout,
                                                     const nvfp4kv_cold_rope* rope,
                                                     int32_t extra_bytes,
                                                     nvfp4kv_cold_block_layout* out) {
    if (!out) return NVFP4KV_ERR_INVALID_ARG;
    return cold_layout(layout, rope, extra_bytes, out) ? NVFP4KV_OK : NVFP4KV_ERR_INVALID_ARG;
}

extern "C" nvfp4kv_status nvfp4_kv_offload_pages(
    const nvfp4kv_layout* layout, nvfp4kv_dtype hot_dtype, const void* hot_k, const void* hot_v,
    int64_t hot_page_stride, int32_t hot_pool_pages, const int32_t* hot_page_ids,
    const float* k_global_scale, const float* v_global_scale, const nvfp4kv_cold_rope* rope,
    const uint8_t* extra, int64_t extra_page_stride, int32_t extra_bytes, uint8_t* cold,
    int32_t cold_slots, const int32_t* cold_slot_ids, int32_t num_pages, int32_t* status,
    nvfp4kv_stream_t stream) {
    ColdParams p;
    const nvfp4kv_status st =
        setup(p, layout, hot_dtype, hot_k, hot_v, hot_page_stride, hot_pool_pages, hot_page_ids,
              k_global_scale, v_global_scale, rope, extra, extra_page_stride, extra_bytes, cold,
              cold_slots, cold_slot_ids, num_pages, status);
    if (st != NVFP4KV_OK || num_pages == 0) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int grid = cold_grid(p);
#define NVFP4KV_OFF(SRC)                                                                      \
    do {                                                                                      \
        if (p.rope_mode == NVFP4KV_ROPE_SKIP)                                                 \
            launch_pdl(cold_offload_kernel<SRC, NVFP4KV_ROPE_SKIP>, grid, kColdThreads, 0, s, p);     \
        else if (p.rope_mode == NVFP4KV_ROPE_2FP4)                                            \
            launch_pdl(cold_offload_kernel<SRC, NVFP4KV_ROPE_2FP4>, grid, kColdThreads, 0, s, p);     \
        else                                                                                  \
            launch_pdl(cold_offload_kernel<SRC, NVFP4KV_ROPE_QUANTIZE>, grid, kColdThreads, 0, s, p); \
    } while (0)
    if (hot_dtype == NVFP4KV_BF16)
        NVFP4KV_OFF(NVFP4KV_BF16);
    else
        NVFP4KV_OFF(NVFP4KV_FP16);
#undef NVFP4KV_OFF
    return launch_status();
}

extern "C" nvfp4kv_status nvfp4_kv_onboard_pages(
    const nvfp4kv_layout* layout, const uint8_t* cold, int32_t cold_slots,
    const int32_t* cold_slot_ids, const float* k_global_scale, const float* v_global_scale,
    const nvfp4kv_cold_rope* rope, nvfp4kv_dtype hot_dtype, void* hot_k, void* hot_v,
    int64_t hot_page_stride, int32_t hot_pool_pages, const int32_t* hot_page_ids, uint8_t* extra,
    int64_t extra_page_stride, int32_t extra_bytes, int32_t num_pages, int32_t* status,
    nvfp4kv_stream_t stream) {
    ColdParams p;
    const nvfp4kv_status st =
        setup(p, layout, hot_dtype, hot_k, hot_v, hot_page_stride, hot_pool_pages, hot_page_ids,
              k_global_scale, v_global_scale, rope, extra, extra_page_stride, extra_bytes, cold,
              cold_slots, cold_slot_ids, num_pages, status);
    if (st != NVFP4KV_OK || num_pages == 0) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int grid = cold_grid(p);
#define NVFP4KV_ON(DST)                                                                      \
    do {                                                                                     \
        if (p.rope_mode == NVFP4KV_ROPE_SKIP)                                                \
            launch_pdl(cold_onboard_kernel<DST, NVFP4KV_ROPE_SKIP>, grid, kColdThreads, 0, s, p);    \
        else if (p.rope_mode == NVFP4KV_ROPE_2FP4)                                           \
            launch_pdl(cold_onboard_kernel<DST, NVFP4KV_ROPE_2FP4>, grid, kColdThreads, 0, s, p);    \
        else                                                                                 \
            launch_pdl(cold_onboard_kernel<DST, NVFP4KV_ROPE_QUANTIZE>, grid, kColdThreads, 0, s, p); \
    } while (0)
    if (hot_dtype == NVFP4KV_BF16)
        NVFP4KV_ON(NVFP4KV_BF16);
    else
        NVFP4KV_ON(NVFP4KV_FP16);
#undef NVFP4KV_ON
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
