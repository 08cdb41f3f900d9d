// Device helpers shared by the NVFP4 kernels (sm_103a): the tagged counters and status word of a
// call, programmatic dependent launch, FP4/FP8/FP16 conversions, warp-level MMA and the L2
// eviction policy of streamed loads. Every conversion here is the hardware instruction named in
// its comment; the exact numerics of each kernel are stated next to the kernel.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "../../include/nvfp4_kv.h"

namespace nvfp4kv {

// ------------------------------------------------------------------------------------------
// Status word
// ------------------------------------------------------------------------------------------
// Returned by tagged_finish when its bounded compare-and-swap loop could not install the call's
// tag (the word held a larger tag and kept changing): the unit that counted is then never
// completed, and the kernel ORs NVFP4KV_STATUS_TIMEOUT into the caller's status word.
constexpr uint32_t kTagGiveUp = 0xFFFFFFFFu;

// Tagged counter (tag in the high 32 bits, count in the low 32): add inc and return the count
// before the add, treating a word whose tag is not this call's as a count of 0. `old` is the
// value returned by a first atomicAdd. Tags grow from call to call, so a stale word is replaced
// by one atomicMax (which never lowers an installed count); a word holding a larger tag
// (garbage) falls back to a compare-and-swap loop. Only values returned by atomics are used:
// a plain re-read could be served stale from L1.
__device__ __forceinline__ uint32_t tagged_finish(unsigned long long* w, unsigned long long old,
                                                  uint32_t nonce, uint32_t inc) {
    if (static_cast<uint32_t>(old >> 32) == nonce) return static_cast<uint32_t>(old);
    const unsigned long long base = static_cast<unsigned long long>(nonce) << 32;
    atomicMax(w, base);
    unsigned long long cur = atomicAdd(w, static_cast<unsigned long long>(inc));
    if (static_cast<uint32_t>(cur >> 32) == nonce) return static_cast<uint32_t>(cur);
    cur += inc;
    for (int it = 0; it < 256; ++it) {
        if (static_cast<uint32_t>(cur >> 32) == nonce) {
            const unsigned long long o2 = atomicAdd(w, static_cast<unsigned long long>(inc));
            if (static_cast<uint32_t>(o2 >> 32) == nonce) return static_cast<uint32_t>(o2);
            cur = o2 + inc;
            continue;
        }
        const unsigned long long seen = atomicCAS(w, cur, base | inc);
        if (seen == cur) return 0;
        cur = seen;
    }
    return kTagGiveUp;  // could not install the tag: the caller reports NVFP4KV_STATUS_TIMEOUT
}

// Acquire-release fence at GPU scope: with a relaxed atomic after it, the writes before it are
// visible to whoever reads the atomic's result (release); after a relaxed atomic whose result
// was read, the reads after it see what was released (acquire). Lighter than __threadfence(),
// which is a sequentially consistent fence.
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// Programmatic dependent launch: wait until the previous grid on the stream has completed and
// its memory is visible (a no-op when the launch did not allow overlap), then let the next grid
// be scheduled.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void flag_status(int32_t* status, int32_t bit) {
    if (status) atomicOr(status, bit);
}

// ------------------------------------------------------------------------------------------
// Conversions
// ------------------------------------------------------------------------------------------

// The four bytes of w, each as two E2M1 codes -> FP16 pair (o[k] from byte k). The bytes are
// split with a vector move into 8-bit registers, which the conversions read directly (no shifts).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&o)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}

// The two 16-bit halves of w, each as two E4M3 bytes -> FP16 pair (o[0] from the low half).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t (&o)[2]) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(o[0]), "=r"(o[1])
        : "r"(w));
}

// Two E4M3 bytes (low byte -> low half) to two exact FP16 values: cvt.rn.f16x2.e4m3x2.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes_in_low_bits) {
    uint32_t out;
    const uint16_t h = static_cast<uint16_t>(two_bytes_in_low_bits);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(h));
    return out;
}

// E2M1 codes of (lo, hi), round-to-nearest-even with saturation at +-6, packed lo | hi << 4:
// cvt.rn.satfinite.e2m1x2.f32 (first source -> upper nibble).
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
    uint32_t out;
    asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\tcvt.u32.u8 %0, b;\n\t}"
        : "=r"(out) : "f"(hi), "f"(lo));
    return out;
}

// E4M3 bytes of (lo, hi), round-to-nearest-even with saturation at +-448, packed lo | hi << 8:
// cvt.rn.satfinite.e4m3x2.f32 (first source -> upper byte).
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t out;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(hi), "f"(lo));
    return out;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
    const uint32_t h2 = e4m3x2_to_f16x2(byte & 0xFFu);
    return __half2float(__ushort_as_half(static_cast<uint16_t>(h2 & 0xFFFFu)));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float f16_lo(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<uint16_t>(w & 0xFFFFu)));
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<uint16_t>(w >> 16)));
}

// (lo, hi) -> packed bf16x2 / f16x2, round to nearest even: cvt.rn.bf16x2.f32 / cvt.rn.f16x2.f32
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t out;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
    return out;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t out;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
    return out;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    uint32_t out;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out) : "r"(a), "r"(b));
    return out;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------------------------------------
// Warp-level tensor-core MMA and fragment moves
// ------------------------------------------------------------------------------------------

// D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col)
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// L2 eviction policy for data that is read once per call: its lines are the first to go.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

}  // namespace nvfp4kv
