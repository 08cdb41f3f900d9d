// NVFP4 page codec for sm_103a: encode (quantize), decode (dequantize to BF16 / FP16 / FP8) and
// the tensor amax -> global scale reduction.
//
// Format: 4-bit E2M1 values, one E4M3 scale per 16-value block, one FP32 scale per tensor
// ("Accelerating Long-Context and Agentic Inference with NVFP4 KV Cache", LMSYS: introduction,
// Figure 1; "KV Cache Compression in TensorRT LLM", NVIDIA: "NVFP4 Cold-Page Compression",
// Figure 6). Encode and decode run on a batch of pages per call on the caller's stream, as the
// TensorRT LLM codec does ("How It Works": the cache manager hands the codec a batch of pages
// at a time, on a stream of the manager's); the extend path's FP8 workspace fill is the FP8-output decode
// (LMSYS, "Path 2: Chunked prefill / Extend").
//
// All three kernels stream HBM once: every byte of input is loaded with one coalesced vector
// load (256-bit for 16-bit pages), every byte of output is written once, nothing is staged
// through shared memory because no value is reused. Work is cut into (page, chunk-of-blocks)
// items so that small batches still fill all SMs; the page id is read once per item.
#include <cstdint>
#include <cuda_runtime.h>

#include "codec_core.cuh"
#include "common.cuh"
#include "host_util.h"

namespace nvfp4kv {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerThread = 4;                      // 16-value blocks per thread per item
constexpr int kItemBlocks = kThreads * kBlocksPerThread; // blocks per work item

struct QuantParams {
    const void* src;
    const int32_t* src_ids;
    const float* src_scale;
    const float* g;
    uint8_t* dst_data;
    uint8_t* dst_scales;
    const int32_t* dst_ids;
    int32_t src_pool;
    int32_t dst_pool;
    int32_t num_pages;
    int32_t bpp;            // 16-value blocks per page = H * T * D / 16
    int32_t nb;             // blocks per token row = D / 16
    uint64_t nb_magic;      // div_magic(nb)
    int32_t units;          // work units per page (blocks, or block pairs for token pairs)
    int32_t items_per_page; // ceil(units / kItemUnits)
    int32_t* status;
    // extend write only: the FP8 E4M3 workspace copy of the source pages
    uint8_t* ws;
    const int32_t* ws_ids;
    const float* ws_scale;  // y = E4M3(fp32(x * fp32(1 / ws_scale))); NULL: 1
    int32_t ws_pool;
};

// FP8 E4M3 bytes (round to nearest even, saturating) of fp32(x[k] * m), k = 0 .. 15
__device__ __forceinline__ uint4 fp8_block(const float (&x)[16], float m) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        w[q] = f32x2_to_e4m3x2(__fmul_rn(x[4 * q], m), __fmul_rn(x[4 * q + 1], m)) |
               (f32x2_to_e4m3x2(__fmul_rn(x[4 * q + 2], m), __fmul_rn(x[4 * q + 3], m)) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// SRC: NVFP4KV_BF16, NVFP4KV_FP16 or NVFP4KV_FP8_E4M3. A32: a 16-bit source is 32-byte aligned
// (one 256-bit load per block). PACK: NVFP4KV_PACK_DIM_PAIRS (a unit is one block of one token)
// or NVFP4KV_PACK_TOKEN_PAIRS (a unit is the same block of tokens 2p and 2p+1; the E2M1 pair
// conversion of (token 2p, token 2p+1) at one head dim is directly the interleaved byte).
// WS: also write the FP8 workspace copy of every source block (the extend path's fused write).
// CTAs per SM the register budget must allow: 4 for the plain encode (64 registers; the
// dim-pair variant would take 70 and fit only 3, and 4 means a third more loads in flight:
// 56.0 -> 53.3 us on 268 MB of BF16), 3 for the FP16 token-pair encode (held at 64 it spills
// heavily), none (0) for the extend write, whose variants keep the compiler's own choice.
template <int SRC, int PACK, bool WS>
constexpr int quantize_min_ctas() {
    return WS ? 0 : ((SRC == NVFP4KV_FP16 && PACK == NVFP4KV_PACK_TOKEN_PAIRS) ? 3 : 4);
}

// One work item of the encode: item = (page i, chunk k of its units). g, d = fp32(6 g), the FP8
// source scale and the workspace multiplier are the call's scalars.
template <int SRC, bool A32, int PACK, bool WS>
__device__ __forceinline__ void quant_item(const QuantParams& p, int64_t item, float g, float d,
                                           float sscale, float wm) {
    constexpr int kUnitsPerThread = (PACK == NVFP4KV_PACK_TOKEN_PAIRS) ? kBlocksPerThread / 2
                                                                        : kBlocksPerThread;
    constexpr int kItemUnits = kThreads * kUnitsPerThread;
    const int32_t i = static_cast<int32_t>(item / p.items_per_page);
    const int32_t k = static_cast<int32_t>(item - static_cast<int64_t>(i) * p.items_per_page);
    const int32_t sp = p.src_ids ? __ldg(p.src_ids + i) : i;
    const int32_t dp = p.dst_ids ? __ldg(p.dst_ids + i) : i;
    int32_t wp = 0;
    if constexpr (WS) wp = p.ws_ids ? __ldg(p.ws_ids + i) : i;
    if (sp < 0 || sp >= p.src_pool || dp < 0 || dp >= p.dst_pool ||
        (WS && (wp < 0 || wp >= p.ws_pool))) {
        if (threadIdx.x == 0) flag_status(p.status, NVFP4KV_STATUS_PAGE_OOB);
        return;
    }
    const int64_t src_blk0 = static_cast<int64_t>(sp) * p.bpp;
    const int64_t dst_blk0 = static_cast<int64_t>(dp) * p.bpp;
    uint8_t* const ws_page = WS ? p.ws + static_cast<int64_t>(wp) * p.bpp * 16 : nullptr;
    const int32_t u_begin = k * kItemUnits + threadIdx.x;
    if constexpr (PACK == NVFP4KV_PACK_DIM_PAIRS) {
        U8x32 raw[kUnitsPerThread];
#pragma unroll
        for (int u = 0; u < kUnitsPerThread; ++u) {
            const int32_t blk = u_begin + u * kThreads;
            if (blk < p.units) raw[u] = load_raw<SRC, A32>(p.src, src_blk0 + blk);
        }
#pragma unroll
        for (int u = 0; u < kUnitsPerThread; ++u) {
            const int32_t blk = u_begin + u * kThreads;
            if (blk >= p.units) continue;
            float x[16];
            widen<SRC>(raw[u], sscale, x);
            uint32_t sb;
            float r;
            pick_scale(x, g, d, sb, r);
            uint32_t w0 = 0u, w1 = 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                w0 |= f32x2_to_e2m1x2(__fmul_rn(x[2 * j], r), __fmul_rn(x[2 * j + 1], r))
                      << (8 * j);
                w1 |= f32x2_to_e2m1x2(__fmul_rn(x[8 + 2 * j], r), __fmul_rn(x[9 + 2 * j], r))
                      << (8 * j);
            }
            st_cs(p.dst_data + (dst_blk0 + blk) * 8, make_uint2(w0, w1));
            st_cs_u8(p.dst_scales + dst_blk0 + blk, sb);
            if constexpr (WS)
                st_cs(ws_page + static_cast<int64_t>(blk) * 16, fp8_block(x, wm));
        }
    } else {
        U8x32 raw0[kUnitsPerThread], raw1[kUnitsPerThread];
#pragma unroll
        for (int u = 0; u < kUnitsPerThread; ++u) {
            const int32_t unit = u_begin + u * kThreads;
            if (unit < p.units) {
                const uint32_t row_pair = fast_div(unit, p.nb_magic);
                const int32_t b = unit - static_cast<int32_t>(row_pair) * p.nb;
                const int64_t blk = src_blk0 + static_cast<int64_t>(2 * row_pair) * p.nb + b;
                raw0[u] = load_raw<SRC, A32>(p.src, blk);
                raw1[u] = load_raw<SRC, A32>(p.src, blk + p.nb);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnitsPerThread; ++u) {
            const int32_t unit = u_begin + u * kThreads;
            if (unit >= p.units) continue;
            float x0[16], x1[16];
            widen<SRC>(raw0[u], sscale, x0);
            widen<SRC>(raw1[u], sscale, x1);
            uint32_t s0, s1;
            float r0, r1;
            pick_scale(x0, g, d, s0, r0);
            pick_scale(x1, g, d, s1, r1);
            uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int e = 0; e < 16; ++e)
                w[e >> 2] |= f32x2_to_e2m1x2(__fmul_rn(x0[e], r0), __fmul_rn(x1[e], r1))
                             << (8 * (e & 3));
            // unit index = (row pair, block): data at unit * 16, scales at unit * 2
            const int64_t o = dst_blk0 / 2 + unit;
            st_cs(p.dst_data + o * 16, make_uint4(w[0], w[1], w[2], w[3]));
            st_cs_u16(p.dst_scales + o * 2, s0 | (s1 << 8));
            if constexpr (WS) {
                // the same block of tokens 2p and 2p+1 in the plain [token][dim] workspace
                const uint32_t row_pair = fast_div(unit, p.nb_magic);
                const int32_t b = unit - static_cast<int32_t>(row_pair) * p.nb;
                const int64_t wb = static_cast<int64_t>(2 * row_pair) * p.nb + b;
                st_cs(ws_page + wb * 16, fp8_block(x0, wm));
                st_cs(ws_page + (wb + p.nb) * 16, fp8_block(x1, wm));
            }
        }
    }
}

template <int SRC, bool A32, int PACK, bool WS = false>
__global__ void __launch_bounds__(kThreads, quantize_min_ctas<SRC, PACK, WS>())
    quantize_pages_kernel(const QuantParams p) {
    pdl_enter();
    const float g = __ldg(p.g);
    const float d = __fmul_rn(6.0f, g);
    const float sscale = (SRC == NVFP4KV_FP8_E4M3 && p.src_scale) ? __ldg(p.src_scale) : 1.0f;
    const float wm = (WS && p.ws_scale) ? __frcp_rn(__ldg(p.ws_scale)) : 1.0f;
    const int64_t total_items = static_cast<int64_t>(p.num_pages) * p.items_per_page;
    for (int64_t item = blockIdx.x; item < total_items; item += gridDim.x)
        quant_item<SRC, A32, PACK, WS>(p, item, g, d, sscale, wm);
}

// ------------------------------------------------------------------------------------------
// Decode. v = e2m1(c) * e4m3(s) is formed exactly in FP16 (cvt.rn.f16x2.e2m1x2 and
// cvt.rn.f16x2.e4m3x2 are exact, and the product has at most 6 significant bits), widened to
// fp32 exactly, multiplied by g (BF16 / FP16 out) or m = fp32(g / dst_scale) (FP8 out) with
// one IEEE fp32 multiply, and rounded to the output type to nearest even (FP8 saturating).
// A unit is one block of one token (dim pairs: 8 code bytes + the block's scale, 16 outputs,
// one 32-byte store) or 8 head dims of a token pair (token pairs: 8 code bytes + the pair's 2
// scales, 8 outputs for each of the two tokens). FP8 outputs are half as wide: a dim-pair unit
// stores 16 bytes, a token-pair unit covers 16 dims of the pair.
// ------------------------------------------------------------------------------------------
struct DequantParams {
    const uint8_t* src_data;
    const uint8_t* src_scales;
    const int32_t* src_ids;
    const float* g;
    const float* dst_scale;
    void* dst;
    const int32_t* dst_ids;
    int32_t src_pool;
    int32_t dst_pool;
    int32_t num_pages;
    int32_t bpp;            // blocks per page
    int32_t nb;             // blocks per token row
    uint64_t nb2_magic;     // div_magic(2 * nb)
    uint64_t nb_magic;      // div_magic(nb)
    int32_t units;          // units per page
    int32_t items_per_page; // ceil(units / units per item)
    int32_t* status;
};

template <int DST>
__device__ __forceinline__ void store8(void* dst, int64_t elem, const float (&y)[8]) {
    if constexpr (DST == NVFP4KV_FP8_E4M3) {
        uint2 o;
        o.x = f32x2_to_e4m3x2(y[0], y[1]) | (f32x2_to_e4m3x2(y[2], y[3]) << 16);
        o.y = f32x2_to_e4m3x2(y[4], y[5]) | (f32x2_to_e4m3x2(y[6], y[7]) << 16);
        st_cs(static_cast<uint8_t*>(dst) + elem, o);
    } else {
        uint4 o;
        if constexpr (DST == NVFP4KV_BF16) {
            o = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                           pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
        } else {
            o = make_uint4(pack_f16x2(y[0], y[1]), pack_f16x2(y[2], y[3]),
                           pack_f16x2(y[4], y[5]), pack_f16x2(y[6], y[7]));
        }
        st_cs(static_cast<uint8_t*>(dst) + elem * 2, o);
    }
}

// One work item of the decode: item = (page i, chunk k of its units); mult is g, or
// fp32(g / dst_scale) for FP8 output.
template <int DST, int PACK>
__device__ __forceinline__ void dequant_item(const DequantParams& p, int64_t item, float mult) {
    constexpr int kU = kBlocksPerThread;  // units per thread per item
    const int32_t i = static_cast<int32_t>(item / p.items_per_page);
    const int32_t k = static_cast<int32_t>(item - static_cast<int64_t>(i) * p.items_per_page);
    const int32_t sp = p.src_ids ? __ldg(p.src_ids + i) : i;
    const int32_t dp = p.dst_ids ? __ldg(p.dst_ids + i) : i;
    if (sp < 0 || sp >= p.src_pool || dp < 0 || dp >= p.dst_pool) {
        if (threadIdx.x == 0) flag_status(p.status, NVFP4KV_STATUS_PAGE_OOB);
        return;
    }
    const int64_t src_blk0 = static_cast<int64_t>(sp) * p.bpp;
    const int64_t dst_elem0 = static_cast<int64_t>(dp) * p.bpp * 16;
    const int32_t u_begin = k * kThreads * kU + threadIdx.x;
    if constexpr (DST == NVFP4KV_FP8_E4M3) {
        // one 16-byte load of codes (dim pairs: 8 bytes) per unit, 16-byte FP8 stores
        uint4 code[kU];
        uint32_t sc[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int32_t unit = u_begin + u * kThreads;
            if (unit < p.units) {
                if constexpr (PACK == NVFP4KV_PACK_DIM_PAIRS) {
                    const uint2 c2 = ld_stream_8B(p.src_data + (src_blk0 + unit) * 8);
                    code[u] = make_uint4(c2.x, c2.y, 0u, 0u);
                    sc[u] = ld_stream_1B(p.src_scales + src_blk0 + unit) * 0x0101u;
                } else {
                    code[u] = ld_stream_16B(p.src_data + src_blk0 * 8 + static_cast<int64_t>(unit) * 16);
                    sc[u] = *reinterpret_cast<const uint16_t*>(p.src_scales + src_blk0 +
                                                               static_cast<int64_t>(unit) * 2);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int32_t unit = u_begin + u * kThreads;
            if (unit >= p.units) continue;
            if constexpr (PACK == NVFP4KV_PACK_DIM_PAIRS) {
                // 16 values of one token: (s, s) times each code pair
                const uint32_t s2 = e4m3x2_to_f16x2(sc[u]);
                uint32_t v[8];
                e2m1x8_to_f16x2x4(code[u].x, *reinterpret_cast<uint32_t(*)[4]>(v));
                e2m1x8_to_f16x2x4(code[u].y, *reinterpret_cast<uint32_t(*)[4]>(v + 4));
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t a = hmul2_u32(v[2 * j], s2), b = hmul2_u32(v[2 * j + 1], s2);
                    o[j] = f32x2_to_e4m3x2(__fmul_rn(f16_lo(a), mult), __fmul_rn(f16_hi(a), mult)) |
                           (f32x2_to_e4m3x2(__fmul_rn(f16_lo(b), mult), __fmul_rn(f16_hi(b), mult))
                            << 16);
                }
                st_cs(static_cast<uint8_t*>(p.dst) + dst_elem0 + static_cast<int64_t>(unit) * 16,
                      make_uint4(o[0], o[1], o[2], o[3]));
            } else {
                const uint32_t s2 = e4m3x2_to_f16x2(sc[u]);
                // 16 head dims of tokens 2rp (low nibbles) and 2rp+1 (high nibbles)
                const uint32_t rp = fast_div(unit, p.nb_magic);
                const int32_t blk = unit - static_cast<int32_t>(rp) * p.nb;
                const uint32_t words[4] = {code[u].x, code[u].y, code[u].z, code[u].w};
                uint32_t o0[4], o1[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t v[4];
                    e2m1x8_to_f16x2x4(words[q], v);  // v[j]: dim 4q + j of (token 2rp, 2rp+1)
                    const uint32_t a0 = hmul2_u32(v[0], s2), a1 = hmul2_u32(v[1], s2);
                    const uint32_t a2 = hmul2_u32(v[2], s2), a3 = hmul2_u32(v[3], s2);
                    o0[q] = f32x2_to_e4m3x2(__fmul_rn(f16_lo(a0), mult), __fmul_rn(f16_lo(a1), mult)) |
                            (f32x2_to_e4m3x2(__fmul_rn(f16_lo(a2), mult), __fmul_rn(f16_lo(a3), mult))
                             << 16);
                    o1[q] = f32x2_to_e4m3x2(__fmul_rn(f16_hi(a0), mult), __fmul_rn(f16_hi(a1), mult)) |
                            (f32x2_to_e4m3x2(__fmul_rn(f16_hi(a2), mult), __fmul_rn(f16_hi(a3), mult))
                             << 16);
                }
                const int64_t e0 = dst_elem0 + static_cast<int64_t>(2 * rp) * p.nb * 16 + blk * 16;
                uint8_t* d8 = static_cast<uint8_t*>(p.dst);
                st_cs(d8 + e0, make_uint4(o0[0], o0[1], o0[2], o0[3]));
                st_cs(d8 + e0 + p.nb * 16, make_uint4(o1[0], o1[1], o1[2], o1[3]));
            }
        }
    } else if constexpr (PACK == NVFP4KV_PACK_DIM_PAIRS) {
        // a unit is one block: 8 code bytes and its scale in, 16 outputs (32 bytes) out
        uint2 code[kBlocksPerThread];
        uint32_t sbyte[kBlocksPerThread];
#pragma unroll
        for (int u = 0; u < kBlocksPerThread; ++u) {
            const int32_t unit = u_begin + u * kThreads;
            if (unit < p.units) {
                code[u] = ld_stream_8B(p.src_data + (src_blk0 + unit) * 8);
                sbyte[u] = ld_stream_1B(p.src_scales + src_blk0 + unit);
            }
        }
#pragma unroll
        for (int u = 0; u < kBlocksPerThread; ++u) {
            const int32_t unit = u_begin + u * kThreads;
            if (unit >= p.units) continue;
            const uint32_t s2 = e4m3x2_to_f16x2(sbyte[u] * 0x0101u);  // (s, s)
            uint32_t v[8];
            e2m1x8_to_f16x2x4(code[u].x, *reinterpret_cast<uint32_t(*)[4]>(v));
            e2m1x8_to_f16x2x4(code[u].y, *reinterpret_cast<uint32_t(*)[4]>(v + 4));
            uint32_t o[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t v2 = hmul2_u32(v[j], s2);
                const float lo = __fmul_rn(f16_lo(v2), mult), hi = __fmul_rn(f16_hi(v2), mult);
                o[j] = (DST == NVFP4KV_BF16) ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
            }
            st_global_32B(static_cast<uint8_t*>(p.dst) + (dst_elem0 + static_cast<int64_t>(unit) * 16) * 2, o);
        }
    } else {
        uint2 code[kBlocksPerThread];
        uint32_t spair[kBlocksPerThread];
#pragma unroll
        for (int u = 0; u < kBlocksPerThread; ++u) {
            const int32_t unit = u_begin + u * kThreads;
            if (unit < p.units) {
                code[u] = *reinterpret_cast<const uint2*>(p.src_data + src_blk0 * 8 +
                                                          static_cast<int64_t>(unit) * 8);
                // the unit's block: (row pair, block) = unit / 2; its two scales side by side
                spair[u] = *reinterpret_cast<const uint16_t*>(p.src_scales + src_blk0 +
                                                              (unit >> 1) * 2);
            }
        }
#pragma unroll
        for (int u = 0; u < kBlocksPerThread; ++u) {
            const int32_t unit = u_begin + u * kThreads;
            if (unit >= p.units) continue;
            const uint32_t s2 = e4m3x2_to_f16x2(spair[u]);  // (s token 2p, s token 2p+1)
            const uint32_t row_pair = fast_div(unit, p.nb2_magic);
            const int32_t rem = unit - static_cast<int32_t>(row_pair) * 2 * p.nb;  // 8-dim slot
            float y0[8], y1[8];
            const uint32_t words[2] = {code[u].x, code[u].y};
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t v[4];
                e2m1x8_to_f16x2x4(words[q], v);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t v2 = hmul2_u32(v[j], s2);  // (token 2p, token 2p+1)
                    y0[4 * q + j] = __fmul_rn(f16_lo(v2), mult);
                    y1[4 * q + j] = __fmul_rn(f16_hi(v2), mult);
                }
            }
            const int64_t e0 = dst_elem0 + static_cast<int64_t>(2 * row_pair) * p.nb * 16 +
                               rem * 8;
            store8<DST>(p.dst, e0, y0);
            store8<DST>(p.dst, e0 + p.nb * 16, y1);
        }
    }
}

template <int DST, int PACK>
__global__ void __launch_bounds__(kThreads) dequantize_pages_kernel(const DequantParams p) {
    pdl_enter();
    const float g = __ldg(p.g);
    const float mult = (DST == NVFP4KV_FP8_E4M3)
                           ? (p.dst_scale ? __fdiv_rn(g, __ldg(p.dst_scale)) : g)
                           : g;
    const int64_t total_items = static_cast<int64_t>(p.num_pages) * p.items_per_page;
    for (int64_t item = blockIdx.x; item < total_items; item += gridDim.x)
        dequant_item<DST, PACK>(p, item, mult);
}

// ------------------------------------------------------------------------------------------
// Tensor amax and global scale. Non-negative IEEE values order like their bit patterns, so the
// maximum of |x| is taken on the sign-cleared 16-bit (BF16 / FP16) or 8-bit (FP8) patterns with
// SIMD unsigned maxima; each CTA raises a tagged maximum word in the workspace and bumps a
// tagged count, and the CTA that completes the count writes g = fp32(amax / 2688), or 1 when
// that is 0: one launch, and the workspace never needs clearing. For FP8 sources the maximum
// of fp32(e4m3 * src_scale) is fp32(max|e4m3| * |src_scale|) because rounding is monotone.
// ------------------------------------------------------------------------------------------
constexpr int kAmaxThreads = 256;
constexpr int kAmaxLoads = 8;   // 16-byte loads per thread per item (128 bytes in flight)

struct AmaxParams {
    const void* src;
    const int32_t* src_ids;
    int32_t src_pool;
    int32_t num_pages;
    int64_t page_bytes;   // bytes of one page (a multiple of 16)
    int32_t items_per_page;
    int32_t item_bytes;   // kAmaxThreads * 16 * kAmaxLoads
    unsigned long long* word;  // [0] tagged maximum pattern, [1] tagged count of finished CTAs
    uint32_t nonce;       // tag of this call
    const float* src_scale;
    float* out;
    int32_t* status;
};

// g of the maximum magnitude pattern r: fp32(amax / 2688), 1 when that is 0. FP8 sources:
// amax = fp32(max|e4m3| * |src_scale|) (rounding is monotone).
template <int SRC>
__device__ __forceinline__ float global_scale_of(uint32_t r, const float* src_scale) {
    float amax;
    if constexpr (SRC == NVFP4KV_FP8_E4M3) {
        amax = __fmul_rn(e4m3_to_f32(r), fabsf(src_scale ? *src_scale : 1.0f));
    } else if constexpr (SRC == NVFP4KV_BF16) {
        amax = __uint_as_float(r << 16);
    } else {
        amax = __half2float(__ushort_as_half(static_cast<uint16_t>(r)));
    }
    const float g = __fdiv_rn(amax, 2688.0f);
    return (g == 0.0f) ? 1.0f : g;
}

// Raise the tagged maximum (tag in the high 32 bits) to r. Tags grow from call to call, so a
// word of an earlier call is replaced by the first atomicMax; a word holding a larger tag
// (garbage) is installed over with a bounded compare-and-swap loop. Returns false when that
// loop ran out without installing r.
__device__ __forceinline__ bool tagged_max(unsigned long long* w, uint32_t nonce, uint32_t r) {
    const unsigned long long v = (static_cast<unsigned long long>(nonce) << 32) | r;
    unsigned long long old = atomicMax(w, v);
    if (static_cast<uint32_t>(old >> 32) <= nonce) return true;
    for (int it = 0; it < 256; ++it) {
        const unsigned long long seen = atomicCAS(w, old, v);
        if (seen == old) return true;
        old = seen;
        if (static_cast<uint32_t>(old >> 32) <= nonce) {
            atomicMax(w, v);
            return true;
        }
    }
    return false;
}

template <int SRC>
__global__ void __launch_bounds__(kAmaxThreads) amax_kernel(const AmaxParams p) {
    pdl_enter();
    const uint32_t mask = (SRC == NVFP4KV_FP8_E4M3) ? 0x7F7F7F7Fu : 0x7FFF7FFFu;
    uint32_t m = 0u;
    const int64_t total_items = static_cast<int64_t>(p.num_pages) * p.items_per_page;
    for (int64_t item = blockIdx.x; item < total_items; item += gridDim.x) {
        const int32_t i = static_cast<int32_t>(item / p.items_per_page);
        const int32_t k = static_cast<int32_t>(item - static_cast<int64_t>(i) * p.items_per_page);
        const int32_t sp = p.src_ids ? __ldg(p.src_ids + i) : i;
        if (sp < 0 || sp >= p.src_pool) {
            if (threadIdx.x == 0) flag_status(p.status, NVFP4KV_STATUS_PAGE_OOB);
            continue;
        }
        const uint8_t* base = static_cast<const uint8_t*>(p.src) + sp * p.page_bytes;
        const int64_t off0 = static_cast<int64_t>(k) * p.item_bytes + threadIdx.x * 16;
        uint4 raw[kAmaxLoads];
        bool ok[kAmaxLoads];
#pragma unroll
        for (int u = 0; u < kAmaxLoads; ++u) {
            const int64_t off = off0 + static_cast<int64_t>(u) * kAmaxThreads * 16;
            ok[u] = off < p.page_bytes;
            if (ok[u]) raw[u] = ld_stream_16B(base + off);
        }
#pragma unroll
        for (int u = 0; u < kAmaxLoads; ++u) {
            if (!ok[u]) continue;
            const uint32_t wv[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if constexpr (SRC == NVFP4KV_FP8_E4M3)
                    m = __vmaxu4(m, wv[j] & mask);
                else
                    m = __vmaxu2(m, wv[j] & mask);
            }
        }
    }
    // combine the lanes of the packed maximum, then reduce over the CTA
    if constexpr (SRC == NVFP4KV_FP8_E4M3) {
        m = max(max(m & 0xFFu, (m >> 8) & 0xFFu), max((m >> 16) & 0xFFu, m >> 24));
    } else {
        m = max(m & 0xFFFFu, m >> 16);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    __shared__ uint32_t red[kAmaxThreads / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t r = 0u;
        for (int w = 0; w < kAmaxThreads / 32; ++w) r = max(r, red[w]);
        // the CTA's maximum into the call's tagged maximum, then the count; the CTA that
        // completes the count writes g
        if (!tagged_max(p.word, p.nonce, r)) flag_status(p.status, NVFP4KV_STATUS_TIMEOUT);
        fence_acq_rel_gpu();  // release: the maximum is in before the count says so
        const uint32_t k = tagged_finish(p.word + 1, atomicAdd(p.word + 1, 1ull), p.nonce, 1);
        if (k == kTagGiveUp) flag_status(p.status, NVFP4KV_STATUS_TIMEOUT);
        if (k == gridDim.x - 1) {
            fence_acq_rel_gpu();  // acquire: every CTA's maximum is read after the count
            const unsigned long long w = atomicAdd(p.word, 0ull);
            const uint32_t best = (static_cast<uint32_t>(w >> 32) == p.nonce)
                                      ? static_cast<uint32_t>(w)
                                      : 0u;
            *p.out = global_scale_of<SRC>(best, p.src_scale);
            // every CTA has counted: both words go back to 0, so a replay of the same launch
            // (a captured CUDA graph, same tag) starts clean
            atomicExch(p.word, 0ull);
            atomicExch(p.word + 1, 0ull);
        }
    }
}

__global__ void write_one_kernel(float* out) {
    pdl_enter();
    *out = 1.0f;
}

// ------------------------------------------------------------------------------------------
// The encoder's two roundings on their own (exhaustive verification over fp32 inputs).
// ------------------------------------------------------------------------------------------
__global__ void round_f32_kernel(const float* x, size_t n, int32_t target, uint8_t* out) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const float v = x[i];
        out[i] = static_cast<uint8_t>(target == 0 ? (f32x2_to_e2m1x2(v, 0.0f) & 0xFu)
                                                  : (f32x2_to_e4m3x2(v, 0.0f) & 0xFFu));
    }
}

// ------------------------------------------------------------------------------------------
// Extend step: the cached prefix of K and V gathered into the FP8 workspace and the current chunk
// of K and V written as NVFP4 pages and as its FP8 workspace copy, all in one grid. The grid is
// cut into four consecutive CTA ranges, one per job (gather K, gather V, write K, write V), sized
// in proportion to the job's work items; a CTA takes the items of its own job with the job's
// CTA count as stride, as in the separate calls. One launch, one ramp and one tail instead of
// four; a CTA holds only its own job's parameters.
// ------------------------------------------------------------------------------------------
struct ExtendStepParams {
    DequantParams gather[2];   // per tensor: NVFP4 prefix pages -> FP8 workspace slots
    QuantParams write[2];      // per tensor: chunk pages -> NVFP4 pages + FP8 workspace slots
    int32_t packing[2];        // per tensor: NVFP4 pool packing
    int32_t cta_end[4];        // cumulative CTA counts of the jobs
};

template <int SRC, bool A32, int PACK>
__device__ __forceinline__ void extend_write_job(const QuantParams& q, int c0, int nc) {
    const float g = __ldg(q.g);
    const float d = __fmul_rn(6.0f, g);
    const float sscale = (SRC == NVFP4KV_FP8_E4M3 && q.src_scale) ? __ldg(q.src_scale) : 1.0f;
    const float wm = q.ws_scale ? __frcp_rn(__ldg(q.ws_scale)) : 1.0f;
    const int64_t total = static_cast<int64_t>(q.num_pages) * q.items_per_page;
    for (int64_t item = blockIdx.x - c0; item < total; item += nc)
        quant_item<SRC, A32, PACK, true>(q, item, g, d, sscale, wm);
}

template <int PACK>
__device__ __forceinline__ void gather_job(const DequantParams& q, int c0, int nc) {
    const float g = __ldg(q.g);
    const float mult = q.dst_scale ? __fdiv_rn(g, __ldg(q.dst_scale)) : g;
    const int64_t total = static_cast<int64_t>(q.num_pages) * q.items_per_page;
    for (int64_t item = blockIdx.x - c0; item < total; item += nc)
        dequant_item<NVFP4KV_FP8_E4M3, PACK>(q, item, mult);
}

// Register budget of 4 CTAs per SM (64 registers): the gather items stream best with many warps,
// and the encode items spill only a few bytes at that budget. Measured on the extend workload
// (16 x 4096-token prefix + 16 x 512-token chunk, K and V, 269 MB): 2 CTAs per SM (the
// compiler's 108 registers) 62.5 us, 3 per SM 50.4 us, 4 per SM 45.1 us; 5 and 6 spill
// 650-1250 bytes per thread.
template <int SRC, bool A32>
__global__ void __launch_bounds__(kThreads, 4) extend_step_kernel(const ExtendStepParams p) {
    pdl_enter();
    const int c = blockIdx.x;
    if (c < p.cta_end[0]) {
        if (p.packing[0] == NVFP4KV_PACK_TOKEN_PAIRS)
            gather_job<NVFP4KV_PACK_TOKEN_PAIRS>(p.gather[0], 0, p.cta_end[0]);
        else
            gather_job<NVFP4KV_PACK_DIM_PAIRS>(p.gather[0], 0, p.cta_end[0]);
    } else if (c < p.cta_end[1]) {
        const int c0 = p.cta_end[0], nc = p.cta_end[1] - c0;
        if (p.packing[1] == NVFP4KV_PACK_TOKEN_PAIRS)
            gather_job<NVFP4KV_PACK_TOKEN_PAIRS>(p.gather[1], c0, nc);
        else
            gather_job<NVFP4KV_PACK_DIM_PAIRS>(p.gather[1], c0, nc);
    } else if (c < p.cta_end[2]) {
        const int c0 = p.cta_end[1], nc = p.cta_end[2] - c0;
        if (p.packing[0] == NVFP4KV_PACK_TOKEN_PAIRS)
            extend_write_job<SRC, A32, NVFP4KV_PACK_TOKEN_PAIRS>(p.write[0], c0, nc);
        else
            extend_write_job<SRC, A32, NVFP4KV_PACK_DIM_PAIRS>(p.write[0], c0, nc);
    } else {
        const int c0 = p.cta_end[2], nc = p.cta_end[3] - c0;
        if (p.packing[1] == NVFP4KV_PACK_TOKEN_PAIRS)
            extend_write_job<SRC, A32, NVFP4KV_PACK_TOKEN_PAIRS>(p.write[1], c0, nc);
        else
            extend_write_job<SRC, A32, NVFP4KV_PACK_DIM_PAIRS>(p.write[1], c0, nc);
    }
}

int grid_for(int64_t items, int ctas_per_sm) {
    const int64_t cap = static_cast<int64_t>(num_sms()) * ctas_per_sm;
    return static_cast<int>(items < cap ? (items < 1 ? 1 : items) : cap);
}

// Launch the extend step: one wave of resident CTAs, split over the jobs in proportion to the
// bytes each moves (an encode item moves 2 + 9/16 + 1 bytes per value, a decode item 9/16 + 1),
// at least one CTA for a job with items and no more CTAs than items.
template <int SRC, bool A32>
cudaError_t launch_extend_step(ExtendStepParams& p, const int64_t (&items)[4],
                               const double (&bytes)[4], cudaStream_t s) {
    const int64_t budget = static_cast<int64_t>(num_sms()) *
                           resident_ctas<extend_step_kernel<SRC, A32>>(kThreads, 0);
    double total = 0.0;
    for (int j = 0; j < 4; ++j) total += bytes[j];
    int acc = 0;
    for (int j = 0; j < 4; ++j) {
        int64_t cj = 0;
        if (items[j] > 0) {
            cj = static_cast<int64_t>(bytes[j] / total * static_cast<double>(budget) + 0.5);
            cj = cj < 1 ? 1 : (cj > items[j] ? items[j] : cj);
        }
        acc += static_cast<int>(cj);
        p.cta_end[j] = acc;
    }
    const cudaError_t e = launch_pdl(extend_step_kernel<SRC, A32>, acc, kThreads, 0, s, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Host-side validation and parameters of an encode job (quantize, or the NVFP4 half of an
// extend write). Returns NVFP4KV_OK with p filled, or the error the entry point reports;
// num_pages == 0 is OK with nothing to launch. The source dtype is checked by the caller.
nvfp4kv_status encode_job(const nvfp4kv_layout* layout, const void* src, int32_t src_pool_pages,
                          const int32_t* src_page_ids, const float* src_scale,
                          const float* global_scale, uint8_t* dst_data, uint8_t* dst_scales,
                          int32_t dst_pool_pages, const int32_t* dst_page_ids, int32_t num_pages,
                          int32_t* status, QuantParams& p) {
    p = QuantParams{};
    if (num_pages == 0) return NVFP4KV_OK;
    if (!src || !global_scale || !dst_data || !dst_scales || !aligned16(src) ||
        !aligned16(dst_data) || !aligned16(dst_scales))
        return NVFP4KV_ERR_INVALID_ARG;
    // without id lists the pages are 0..num_pages-1 and the pools must hold them
    if ((!src_page_ids && src_pool_pages < num_pages) ||
        (!dst_page_ids && dst_pool_pages < num_pages))
        return NVFP4KV_ERR_INVALID_ARG;
    const int pack = layout->packing;
    if (pack != NVFP4KV_PACK_DIM_PAIRS && pack != NVFP4KV_PACK_TOKEN_PAIRS)
        return NVFP4KV_ERR_INVALID_ARG;
    if (pack == NVFP4KV_PACK_TOKEN_PAIRS && (layout->page_size & 1)) return NVFP4KV_ERR_INVALID_ARG;
    const int64_t bpp64 = static_cast<int64_t>(layout->num_kv_heads) * layout->page_size *
                          (layout->head_dim / 16);
    if (bpp64 > (int64_t{1} << 29) || layout->head_dim > 16 * 1024) return NVFP4KV_ERR_UNSUPPORTED;
    p.src = src;
    p.src_ids = src_page_ids;
    p.src_scale = src_scale;
    p.g = global_scale;
    p.dst_data = dst_data;
    p.dst_scales = dst_scales;
    p.dst_ids = dst_page_ids;
    p.src_pool = src_pool_pages;
    p.dst_pool = dst_pool_pages;
    p.num_pages = num_pages;
    p.bpp = static_cast<int32_t>(bpp64);
    p.nb = layout->head_dim / 16;
    p.nb_magic = div_magic(static_cast<uint32_t>(p.nb));
    p.units = (pack == NVFP4KV_PACK_TOKEN_PAIRS) ? p.bpp / 2 : p.bpp;
    const int item_units = (pack == NVFP4KV_PACK_TOKEN_PAIRS) ? kItemBlocks / 2 : kItemBlocks;
    p.items_per_page = (p.units + item_units - 1) / item_units;
    p.status = status;
    return NVFP4KV_OK;
}

// Host-side validation and parameters of a decode job (to BF16 / FP16, or to FP8 E4M3).
nvfp4kv_status decode_job(const nvfp4kv_layout* layout, const uint8_t* src_data,
                          const uint8_t* src_scales, int32_t src_pool_pages,
                          const int32_t* src_page_ids, const float* global_scale,
                          nvfp4kv_dtype dst_dtype, void* dst, int32_t dst_pool_pages,
                          const int32_t* dst_page_ids, const float* dst_scale, int32_t num_pages,
                          int32_t* status, DequantParams& p) {
    p = DequantParams{};
    if (num_pages == 0) return NVFP4KV_OK;
    if (!src_data || !src_scales || !global_scale || !dst || !aligned16(src_data) ||
        !aligned16(src_scales) || !aligned16(dst))
        return NVFP4KV_ERR_INVALID_ARG;
    if ((!src_page_ids && src_pool_pages < num_pages) ||
        (!dst_page_ids && dst_pool_pages < num_pages))
        return NVFP4KV_ERR_INVALID_ARG;
    const int pack = layout->packing;
    if (pack != NVFP4KV_PACK_DIM_PAIRS && pack != NVFP4KV_PACK_TOKEN_PAIRS)
        return NVFP4KV_ERR_INVALID_ARG;
    if (pack == NVFP4KV_PACK_TOKEN_PAIRS && (layout->page_size & 1)) return NVFP4KV_ERR_INVALID_ARG;
    const int64_t bpp64 = static_cast<int64_t>(layout->num_kv_heads) * layout->page_size *
                          (layout->head_dim / 16);
    if (bpp64 > (int64_t{1} << 29) || layout->head_dim > 16 * 1024) return NVFP4KV_ERR_UNSUPPORTED;
    p.src_data = src_data;
    p.src_scales = src_scales;
    p.src_ids = src_page_ids;
    p.g = global_scale;
    p.dst_scale = dst_scale;
    p.dst = dst;
    p.dst_ids = dst_page_ids;
    p.src_pool = src_pool_pages;
    p.dst_pool = dst_pool_pages;
    p.num_pages = num_pages;
    p.bpp = static_cast<int32_t>(bpp64);
    p.nb = layout->head_dim / 16;
    p.nb2_magic = div_magic(static_cast<uint32_t>(2 * p.nb));
    p.nb_magic = div_magic(static_cast<uint32_t>(p.nb));
    // BF16 / FP16 out: a block per dim-pair unit, 16 codes per token-pair unit (2 per block
    // pair); FP8 out: a block per dim-pair unit, 32 codes per token-pair unit
    if (dst_dtype == NVFP4KV_FP8_E4M3)
        p.units = (pack == NVFP4KV_PACK_TOKEN_PAIRS) ? p.bpp / 2 : p.bpp;
    else
        p.units = p.bpp;
    p.items_per_page = (p.units + kItemBlocks - 1) / kItemBlocks;
    p.status = status;
    return NVFP4KV_OK;
}

}  // namespace
}  // namespace nvfp4kv

using namespace nvfp4kv;

extern "C" size_t nvfp4_kv_global_scale_workspace_size(void) {
    return 2 * sizeof(unsigned long long);
}

extern "C" nvfp4kv_status nvfp4_kv_compute_global_scale(
    const nvfp4kv_layout* layout, nvfp4kv_dtype src_dtype, const void* src,
    int32_t src_pool_pages, const int32_t* src_page_ids, int32_t num_pages,
    const float* src_scale, float* global_scale_out, void* workspace, size_t workspace_bytes,
    int32_t* status, nvfp4kv_stream_t stream) {
    if (!layout_ok(layout) || !dtype_ok(src_dtype) || !global_scale_out || num_pages < 0 ||
        src_pool_pages < 0)
        return NVFP4KV_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (num_pages == 0) {
        launch_pdl(write_one_kernel, 1, 1, 0, s, global_scale_out);
        return launch_status();
    }
    if (!src || !aligned16(src)) return NVFP4KV_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < nvfp4_kv_global_scale_workspace_size() ||
        !aligned16(workspace))
        return NVFP4KV_ERR_WORKSPACE;
    const int64_t elems = static_cast<int64_t>(layout->num_kv_heads) * layout->page_size *
                          layout->head_dim;
    AmaxParams p{};
    p.src = src;
    p.src_ids = src_page_ids;
    if (!src_page_ids && src_pool_pages < num_pages) return NVFP4KV_ERR_INVALID_ARG;
    p.src_pool = src_pool_pages;
    p.num_pages = num_pages;
    p.page_bytes = elems * static_cast<int64_t>(dtype_bytes(src_dtype));
    p.item_bytes = kAmaxThreads * 16 * kAmaxLoads;
    p.items_per_page = static_cast<int32_t>((p.page_bytes + p.item_bytes - 1) / p.item_bytes);
    p.word = static_cast<unsigned long long*>(workspace);
    p.nonce = next_nonce();
    p.src_scale = src_scale;
    p.out = global_scale_out;
    p.status = status;
    // one wave of resident CTAs: each CTA reads its items and raises the maximum once (a CTA
    // that waited for a slot would read its whole share after the others have finished)
    const int64_t items = static_cast<int64_t>(num_pages) * p.items_per_page;
#define NVFP4KV_ALAUNCH(SRC) \
    launch_pdl(amax_kernel<SRC>, wave_grid<amax_kernel<SRC>>(items, kAmaxThreads), kAmaxThreads, 0, s, p)
    switch (src_dtype) {
    case NVFP4KV_BF16: NVFP4KV_ALAUNCH(NVFP4KV_BF16); break;
    case NVFP4KV_FP16: NVFP4KV_ALAUNCH(NVFP4KV_FP16); break;
    default: NVFP4KV_ALAUNCH(NVFP4KV_FP8_E4M3); break;
    }
#undef NVFP4KV_ALAUNCH
    return launch_status();
}

extern "C" nvfp4kv_status nvfp4_kv_quantize_pages(
    const nvfp4kv_layout* layout, nvfp4kv_dtype src_dtype, const void* src,
    int32_t src_pool_pages, const int32_t* src_page_ids, const float* src_scale,
    const float* global_scale, uint8_t* dst_data, uint8_t* dst_scales, int32_t dst_pool_pages,
    const int32_t* dst_page_ids, int32_t num_pages, int32_t* status, nvfp4kv_stream_t stream) {
    if (!layout_ok(layout) || !dtype_ok(src_dtype) || num_pages < 0 || src_pool_pages < 0 ||
        dst_pool_pages < 0)
        return NVFP4KV_ERR_INVALID_ARG;
    QuantParams p;
    const nvfp4kv_status st = encode_job(layout, src, src_pool_pages, src_page_ids, src_scale,
                                         global_scale, dst_data, dst_scales, dst_pool_pages,
                                         dst_page_ids, num_pages, status, p);
    if (st != NVFP4KV_OK || num_pages == 0) return st;
    const int pack = layout->packing;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int grid = grid_for(static_cast<int64_t>(num_pages) * p.items_per_page, 8);
    const bool a32 = (reinterpret_cast<uintptr_t>(src) & 31u) == 0;
#define NVFP4KV_QLAUNCH(SRC, A32, PK) \
    launch_pdl(quantize_pages_kernel<SRC, A32, PK>, grid, kThreads, 0, s, p)
#define NVFP4KV_QPACK(SRC, A32)                                          \
    do {                                                                  \
        if (pack == NVFP4KV_PACK_TOKEN_PAIRS)                             \
            NVFP4KV_QLAUNCH(SRC, A32, NVFP4KV_PACK_TOKEN_PAIRS);          \
        else                                                              \
            NVFP4KV_QLAUNCH(SRC, A32, NVFP4KV_PACK_DIM_PAIRS);            \
    } while (0)
    switch (src_dtype) {
    case NVFP4KV_BF16:
        if (a32) NVFP4KV_QPACK(NVFP4KV_BF16, true);
        else NVFP4KV_QPACK(NVFP4KV_BF16, false);
        break;
    case NVFP4KV_FP16:
        if (a32) NVFP4KV_QPACK(NVFP4KV_FP16, true);
        else NVFP4KV_QPACK(NVFP4KV_FP16, false);
        break;
    default: NVFP4KV_QPACK(NVFP4KV_FP8_E4M3, false); break;
    }
#undef NVFP4KV_QPACK
#undef NVFP4KV_QLAUNCH
    return launch_status();
}

extern "C" nvfp4kv_status nvfp4_kv_extend_write(
    const nvfp4kv_layout* layout, nvfp4kv_dtype src_dtype, const void* src,
    int32_t src_pool_pages, const int32_t* src_page_ids, const float* src_scale,
    const float* global_scale, uint8_t* dst_data, uint8_t* dst_scales, int32_t dst_pool_pages,
    const int32_t* dst_page_ids, uint8_t* ws_fp8, int32_t ws_pool_pages, const int32_t* ws_page_ids, const float* ws_scale,
    int32_t num_pages, int32_t* status, nvfp4kv_stream_t stream) {
    if (!layout_ok(layout) || num_pages < 0 || src_pool_pages < 0 || dst_pool_pages < 0 ||
        ws_pool_pages < 0)
        return NVFP4KV_ERR_INVALID_ARG;
    if (src_dtype != NVFP4KV_BF16 && src_dtype != NVFP4KV_FP16 && src_dtype != NVFP4KV_FP8_E4M3)
        return NVFP4KV_ERR_UNSUPPORTED;
    if (num_pages == 0) return NVFP4KV_OK;
    if (!ws_fp8 || !aligned16(ws_fp8) || (!ws_page_ids && ws_pool_pages < num_pages))
        return NVFP4KV_ERR_INVALID_ARG;
    QuantParams p;
    const nvfp4kv_status st = encode_job(layout, src, src_pool_pages, src_page_ids, src_scale,
                                         global_scale, dst_data, dst_scales, dst_pool_pages,
                                         dst_page_ids, num_pages, status, p);
    if (st != NVFP4KV_OK) return st;
    const int pack = layout->packing;
    p.ws = ws_fp8;
    p.ws_ids = ws_page_ids;
    p.ws_scale = ws_scale;
    p.ws_pool = ws_pool_pages;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int grid = grid_for(static_cast<int64_t>(num_pages) * p.items_per_page, 8);
    const bool a32 = (reinterpret_cast<uintptr_t>(src) & 31u) == 0;
#define NVFP4KV_XLAUNCH(SRC, A32)                                                             \
    do {                                                                                     \
        if (pack == NVFP4KV_PACK_TOKEN_PAIRS)                                                \
            launch_pdl(quantize_pages_kernel<SRC, A32, NVFP4KV_PACK_TOKEN_PAIRS, true>, grid, kThreads, 0, s, p); \
        else                                                                                 \
            launch_pdl(quantize_pages_kernel<SRC, A32, NVFP4KV_PACK_DIM_PAIRS, true>, grid, kThreads, 0, s, p);   \
    } while (0)
    if (src_dtype == NVFP4KV_BF16) {
        if (a32) NVFP4KV_XLAUNCH(NVFP4KV_BF16, true);
        else NVFP4KV_XLAUNCH(NVFP4KV_BF16, false);
    } else if (src_dtype == NVFP4KV_FP16) {
        if (a32) NVFP4KV_XLAUNCH(NVFP4KV_FP16, true);
        else NVFP4KV_XLAUNCH(NVFP4KV_FP16, false);
    } else {
        NVFP4KV_XLAUNCH(NVFP4KV_FP8_E4M3, false);
    }
#undef NVFP4KV_XLAUNCH
    return launch_status();
}

extern "C" nvfp4kv_status nvfp4_kv_dequantize_pages(
    const nvfp4kv_layout* layout, const uint8_t* src_data, const uint8_t* src_scales,
    int32_t src_pool_pages, const int32_t* src_page_ids, const float* global_scale,
    nvfp4kv_dtype dst_dtype, void* dst, int32_t dst_pool_pages, const int32_t* dst_page_ids,
    const float* dst_scale, int32_t num_pages, int32_t* status, nvfp4kv_stream_t stream) {
    if (!layout_ok(layout) || !dtype_ok(dst_dtype) || num_pages < 0 || src_pool_pages < 0 ||
        dst_pool_pages < 0)
        return NVFP4KV_ERR_INVALID_ARG;
    DequantParams p;
    const nvfp4kv_status st = decode_job(layout, src_data, src_scales, src_pool_pages,
                                         src_page_ids, global_scale, dst_dtype, dst,
                                         dst_pool_pages, dst_page_ids, dst_scale, num_pages,
                                         status, p);
    if (st != NVFP4KV_OK || num_pages == 0) return st;
    const int pack = layout->packing;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // up to 32 CTAs per SM, several waves of short-lived CTAs (one or two 32 KB items each): the
    // block scheduler then hands the remaining items to whichever SM frees a slot first, which
    // evens out the SMs' different streaming rates (BF16 out 57.3 -> 53.2 us, FP8 out 34.8 ->
    // 32.8 us on 4096 pages against 8 CTAs per SM)
    const int grid = grid_for(static_cast<int64_t>(num_pages) * p.items_per_page, 32);
#define NVFP4KV_DQLAUNCH(DST)                                                                \
    do {                                                                                      \
        if (pack == NVFP4KV_PACK_TOKEN_PAIRS)                                                 \
            launch_pdl(dequantize_pages_kernel<DST, NVFP4KV_PACK_TOKEN_PAIRS>, grid, kThreads, 0, s, p); \
        else                                                                                  \
            launch_pdl(dequantize_pages_kernel<DST, NVFP4KV_PACK_DIM_PAIRS>, grid, kThreads, 0, s, p);   \
    } while (0)
    switch (dst_dtype) {
    case NVFP4KV_BF16: NVFP4KV_DQLAUNCH(NVFP4KV_BF16); break;
    case NVFP4KV_FP16: NVFP4KV_DQLAUNCH(NVFP4KV_FP16); break;
    default: NVFP4KV_DQLAUNCH(NVFP4KV_FP8_E4M3); break;
    }
#undef NVFP4KV_DQLAUNCH
    return launch_status();
}

extern "C" nvfp4kv_status nvfp4_kv_extend_step(const nvfp4kv_extend_tensor* tensors,
                                               int32_t num_tensors, int32_t* status,
                                               nvfp4kv_stream_t stream) {
    if (!tensors || num_tensors < 1 || num_tensors > 2) return NVFP4KV_ERR_INVALID_ARG;
    ExtendStepParams p{};
    int src_dtype = -1;
    bool a32 = true;
    for (int t = 0; t < num_tensors; ++t) {
        const nvfp4kv_extend_tensor& x = tensors[t];
        const nvfp4kv_layout* layout = &x.layout;
        if (!layout_ok(layout) || x.pool_pages < 0 || x.prefix_pages < 0 || x.ws_pages < 0 ||
            x.chunk_pool_pages < 0 || x.chunk_pages < 0)
            return NVFP4KV_ERR_INVALID_ARG;
        if (x.chunk_pages > 0) {
            if (x.chunk_dtype != NVFP4KV_BF16 && x.chunk_dtype != NVFP4KV_FP16 &&
                x.chunk_dtype != NVFP4KV_FP8_E4M3)
                return NVFP4KV_ERR_UNSUPPORTED;
            if (src_dtype >= 0 && src_dtype != x.chunk_dtype) return NVFP4KV_ERR_UNSUPPORTED;
            src_dtype = x.chunk_dtype;
            a32 = a32 && (reinterpret_cast<uintptr_t>(x.chunk) & 31u) == 0;
        }
        // the prefix: FP8 decode into the workspace slots, with the workspace scale
        nvfp4kv_status st = decode_job(layout, x.data, x.scales, x.pool_pages, x.prefix_page_ids,
                                       x.global_scale, NVFP4KV_FP8_E4M3, x.ws, x.ws_pages,
                                       x.ws_prefix_ids, x.ws_scale, x.prefix_pages, status,
                                       p.gather[t]);
        if (st != NVFP4KV_OK) return st;
        // the chunk: NVFP4 pages of the pool plus the FP8 copy in the workspace slots
        if (x.chunk_pages > 0 && (!x.ws || !aligned16(x.ws) ||
                                  (!x.ws_chunk_ids && x.ws_pages < x.chunk_pages)))
            return NVFP4KV_ERR_INVALID_ARG;
        st = encode_job(layout, x.chunk, x.chunk_pool_pages, x.chunk_page_ids,
                        x.chunk_src_scale, x.global_scale, x.data, x.scales, x.pool_pages,
                        x.chunk_dst_ids, x.chunk_pages, status, p.write[t]);
        if (st != NVFP4KV_OK) return st;
        p.write[t].ws = x.ws;
        p.write[t].ws_ids = x.ws_chunk_ids;
        p.write[t].ws_scale = x.ws_scale;
        p.write[t].ws_pool = x.ws_pages;
        p.packing[t] = layout->packing;
    }
    // the jobs: gather 0, gather 1, write 0, write 1 (absent jobs have no items)
    const int64_t items[4] = {
        static_cast<int64_t>(p.gather[0].num_pages) * p.gather[0].items_per_page,
        static_cast<int64_t>(p.gather[1].num_pages) * p.gather[1].items_per_page,
        static_cast<int64_t>(p.write[0].num_pages) * p.write[0].items_per_page,
        static_cast<int64_t>(p.write[1].num_pages) * p.write[1].items_per_page};
    const double bytes[4] = {
        static_cast<double>(p.gather[0].num_pages) * p.gather[0].bpp * 25.0,
        static_cast<double>(p.gather[1].num_pages) * p.gather[1].bpp * 25.0,
        static_cast<double>(p.write[0].num_pages) * p.write[0].bpp * 57.0,
        static_cast<double>(p.write[1].num_pages) * p.write[1].bpp * 57.0};
    if (items[0] + items[1] + items[2] + items[3] == 0) return NVFP4KV_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (src_dtype == NVFP4KV_FP16) {
        e = a32 ? launch_extend_step<NVFP4KV_FP16, true>(p, items, bytes, s)
                : launch_extend_step<NVFP4KV_FP16, false>(p, items, bytes, s);
    } else if (src_dtype == NVFP4KV_FP8_E4M3) {
        e = launch_extend_step<NVFP4KV_FP8_E4M3, false>(p, items, bytes, s);
    } else {  // BF16 chunks, or no chunk at all
        e = a32 ? launch_extend_step<NVFP4KV_BF16, true>(p, items, bytes, s)
                : launch_extend_step<NVFP4KV_BF16, false>(p, items, bytes, s);
    }
    if (e != cudaSuccess) return NVFP4KV_ERR_CUDA;
    return launch_status();
}

extern "C" nvfp4kv_status nvfp4_kv_round_f32(const float* x, size_t n, int32_t target,
                                             uint8_t* out, nvfp4kv_stream_t stream) {
    if ((target != 0 && target != 1) || (n > 0 && (!x || !out))) return NVFP4KV_ERR_INVALID_ARG;
    if (n == 0) return NVFP4KV_OK;
    const int64_t blocks = static_cast<int64_t>((n + 255) / 256);
    round_f32_kernel<<<grid_for(blocks, 8), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        x, n, target, out);
    return launch_status();
}
