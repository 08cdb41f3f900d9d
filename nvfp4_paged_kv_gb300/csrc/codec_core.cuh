// Encode building blocks shared by the page codec and the cold-page codec: streaming vector
// loads, the fixed-point division by a per-call constant, the load and exact widening of one
// 16-value block, and the block scale pick of the NVFP4 encoder (LMSYS, "Accelerating
// Long-Context and Agentic Inference with NVFP4 KV Cache": introduction, Figure 1).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace nvfp4kv {

// ------------------------------------------------------------------------------------------
// Streaming loads / stores
// ------------------------------------------------------------------------------------------
struct U8x32 {
    uint32_t w[8];
};

__device__ __forceinline__ U8x32 ld_stream_32B(const void* p) {
    U8x32 r;
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]),
                   "=r"(r.w[5]), "=r"(r.w[6]), "=r"(r.w[7])
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ld_stream_16B(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ld_stream_8B(const void* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.b32 {%0,%1}, [%2];"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_stream_4B(const void* p) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_stream_1B(const void* p) {
    uint16_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

// n / d for n * d < 2^40 with a 64-bit multiply: magic = ceil(2^40 / d).
__device__ __forceinline__ uint32_t fast_div(uint32_t n, uint64_t magic) {
    return static_cast<uint32_t>((static_cast<uint64_t>(n) * magic) >> 40);
}
inline uint64_t div_magic(uint32_t d) { return ((uint64_t{1} << 40) + d - 1) / d; }

// One block of 16 source values as loaded: 32 bytes (16-bit sources) or 16 bytes (FP8).
template <int SRC, bool A32>
__device__ __forceinline__ U8x32 load_raw(const void* src, int64_t blk) {
    U8x32 raw;
    if constexpr (SRC == NVFP4KV_FP8_E4M3) {
        const uint4 v = ld_stream_16B(static_cast<const uint8_t*>(src) + blk * 16);
        raw.w[0] = v.x;
        raw.w[1] = v.y;
        raw.w[2] = v.z;
        raw.w[3] = v.w;
    } else {
        const uint8_t* a = static_cast<const uint8_t*>(src) + blk * 32;
        if constexpr (A32) {
            raw = ld_stream_32B(a);
        } else {
            const uint4 lo = ld_stream_16B(a), hi = ld_stream_16B(a + 16);
            raw = U8x32{{lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w}};
        }
    }
    return raw;
}

// The 16 values as exact fp32 (BF16 / FP16 widening is exact; FP8 sources are
// x = fp32(e4m3 * src_scale)).
template <int SRC>
__device__ __forceinline__ void widen(const U8x32& raw, float sscale, float (&x)[16]) {
    if constexpr (SRC == NVFP4KV_FP8_E4M3) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t h[2];
            e4m3x4_to_f16x2x2(raw.w[j], h);
            x[4 * j + 0] = __fmul_rn(f16_lo(h[0]), sscale);
            x[4 * j + 1] = __fmul_rn(f16_hi(h[0]), sscale);
            x[4 * j + 2] = __fmul_rn(f16_lo(h[1]), sscale);
            x[4 * j + 3] = __fmul_rn(f16_hi(h[1]), sscale);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if constexpr (SRC == NVFP4KV_BF16) {
                x[2 * j] = bf16_lo(raw.w[j]);
                x[2 * j + 1] = bf16_hi(raw.w[j]);
            } else {
                x[2 * j] = f16_lo(raw.w[j]);
                x[2 * j + 1] = f16_hi(raw.w[j]);
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
// Encode one block of 16 exact fp32 values x:
//   a  = max |x_i|                                          (exact)
//   s  = E4M3_rne_satfinite(fp32(a / d)), d = fp32(6 g)      one IEEE division
//   r  = fp32(1 / fp32(s g)), or 0 when s g == 0             one IEEE reciprocal
//   c_i = E2M1_rne_satfinite(fp32(x_i * r)), sign kept
// ------------------------------------------------------------------------------------------
// Block scale pick of one block: s, and r = fp32(1 / fp32(s g)) (0 when s g == 0).
__device__ __forceinline__ void pick_scale(const float (&x)[16], float g, float d,
                                           uint32_t& sbyte, float& r) {
    float a = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) a = fmaxf(a, fabsf(x[k]));
    sbyte = f32x2_to_e4m3x2(__fdiv_rn(a, d), 0.0f) & 0xFFu;
    const float sg = __fmul_rn(e4m3_to_f32(sbyte), g);
    r = (sg == 0.0f) ? 0.0f : __frcp_rn(sg);
}

// E2M1 codes of fp32(x_i * r), round to nearest even, saturating, sign kept, packed two per byte
// (value 2j in the low nibble of byte j).
__device__ __forceinline__ uint2 pack_e2m1_block(const float (&x)[16], float r) {
    uint32_t w0 = 0u, w1 = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        w0 |= f32x2_to_e2m1x2(__fmul_rn(x[2 * j], r), __fmul_rn(x[2 * j + 1], r)) << (8 * j);
        w1 |= f32x2_to_e2m1x2(__fmul_rn(x[8 + 2 * j], r), __fmul_rn(x[9 + 2 * j], r)) << (8 * j);
    }
    return make_uint2(w0, w1);
}

// The 16 values e2m1(c_i) * e4m3(s) of one block (8 code bytes, scale byte), exact: the FP16
// conversions are exact and the products have at most 6 significant bits.
__device__ __forceinline__ void block_values(uint2 code, uint32_t sbyte, float (&v)[16]) {
    const uint32_t s2 = e4m3x2_to_f16x2(sbyte * 0x0101u);
    uint32_t h[8];
    e2m1x8_to_f16x2x4(code.x, *reinterpret_cast<uint32_t(*)[4]>(h));
    e2m1x8_to_f16x2x4(code.y, *reinterpret_cast<uint32_t(*)[4]>(h + 4));
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t e = hmul2_u32(h[j], s2);
        v[2 * j] = f16_lo(e);
        v[2 * j + 1] = f16_hi(e);
    }
}

// 32 bytes to global memory with one 256-bit store when p is 32-byte aligned (a warp then
// writes whole 32-byte sectors with each instruction), else as two 16-byte stores.
__device__ __forceinline__ void st_global_32B(void* p, const uint32_t (&w)[8]) {
    if ((reinterpret_cast<uintptr_t>(p) & 31u) == 0) {
        asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]),
                     "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
    } else {
        asm volatile("st.global.cs.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3])
                     : "memory");
        asm volatile("st.global.cs.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(static_cast<uint8_t*>(p) + 16),
                     "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
    }
}

// Streaming stores (.cs: the lines are evicted first from L2, as outputs of this pass are not
// read again by it).
__device__ __forceinline__ void st_cs(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_cs(void* p, uint2 v) {
    asm volatile("st.global.cs.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ void st_cs_u16(void* p, uint32_t v) {
    asm volatile("st.global.cs.u16 [%0], %1;" ::"l"(p), "h"(static_cast<uint16_t>(v)) : "memory");
}
__device__ __forceinline__ void st_cs_u8(void* p, uint32_t v) {
    asm volatile("st.global.cs.u8 [%0], %1;" ::"l"(p), "h"(static_cast<uint16_t>(v)) : "memory");
}

}  // namespace nvfp4kv
