// Host-side helpers shared by the C-ABI entry points: validation, device properties, launch
// error mapping. No device code here.
#pragma once

#include <atomic>
#include <chrono>
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <utility>
#include <cuda_runtime.h>

#include "../../include/nvfp4_kv.h"

namespace nvfp4kv {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool layout_ok(const nvfp4kv_layout* l) {
    return l && l->num_kv_heads > 0 && l->head_dim > 0 && l->page_size > 0 &&
           (l->head_dim % 16) == 0;
}

inline bool dtype_ok(int32_t d) {
    return d == NVFP4KV_BF16 || d == NVFP4KV_FP16 || d == NVFP4KV_FP8_E4M3;
}

inline size_t dtype_bytes(int32_t d) { return d == NVFP4KV_FP8_E4M3 ? 1 : 2; }

// Streaming multiprocessor count of the current device (cached per device id).
inline int num_sms() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0)
            n = 152;
        cache[dev] = n;
    }
    return cache[dev];
}

// One tag per call (all devices): counters of earlier calls never carry it. Tags grow from call
// to call, which lets a stale counter be replaced by one atomicMax.
inline uint32_t next_nonce() {
    static std::atomic<uint32_t> counter{static_cast<uint32_t>(
        std::chrono::steady_clock::now().time_since_epoch().count() & 0x3FFFFFFF) + 1u};
    uint32_t n = counter.fetch_add(1) + 1;
    if (n == 0) n = counter.fetch_add(1) + 1;
    return n;
}

// CTAs of `Kernel` (with `threads` threads and `smem` bytes of dynamic shared memory) that fit on
// one SM at once, asked of the runtime once per kernel (at least 1).
template <auto Kernel>
inline int resident_ctas(int threads, size_t smem) {
    static const int n = [&] {
        int v = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, Kernel, threads, smem) != cudaSuccess ||
            v < 1)
            v = 1;
        return v;
    }();
    return n;
}

// Grid of a grid-strided kernel over `items` work items: one full wave of resident CTAs (no CTA
// waits for a slot and then runs its share of items after the others have finished), or fewer
// CTAs when there are fewer items.
template <auto Kernel>
inline int wave_grid(int64_t items, int threads, size_t smem = 0) {
    const int64_t cap = static_cast<int64_t>(num_sms()) * resident_ctas<Kernel>(threads, smem);
    return static_cast<int>(items < cap ? (items < 1 ? 1 : items) : cap);
}

// Launch with programmatic dependent launch allowed: the grid may be scheduled while the
// previous kernel on the stream drains; every kernel of this library waits for the previous
// grid (griddepcontrol.wait) before its first global memory access, so data dependencies on the
// stream are kept.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

inline nvfp4kv_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? NVFP4KV_OK : NVFP4KV_ERR_CUDA;
}

}  // namespace nvfp4kv
