// Paged decode attention for callers that cannot allocate device memory.
//
// nvfp4_paged_decode_attention needs a caller-provided workspace for its split-KV partial
// results. Some callers have no way to get one: a plugin running inside another framework
// that owns every device allocation, a serving process that has already handed all free HBM to
// its KV-cache pool, or code that must not call cudaMalloc on its hot path because the call
// synchronises the device. This file gives them a variant whose scratch lives in a fixed-size
// array in the library's own device memory, allocated once when the library's module is loaded
// on a GPU and held until the process exits.
#include <cstdint>
#include <mutex>
#include <vector>
#include <cuda_runtime.h>

#include "../../include/nvfp4_kv.h"

namespace {

// The scratch: one array per GPU that loads the library, shared by every call on that GPU.
static __device__ __align__(256) uint8_t g_decode_scratch[NVFP4KV_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
std::vector<void*> g_scratch_addr;  // device address of g_decode_scratch, per device id

// Device address of the scratch on the current device. In host code the array's name is only a
// host-side stand-in, so the address comes from cudaGetSymbolAddress, once per device, with
// that device current. The address is kept until the process exits; cudaDeviceReset ends the
// context that owns the array, after which this entry point must not be used on that device.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_mu);
    if (dev >= static_cast<int>(g_scratch_addr.size())) g_scratch_addr.resize(dev + 1, nullptr);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" nvfp4kv_status nvfp4_paged_decode_attention_noalloc(
    const nvfp4kv_layout* layout, int32_t batch, int32_t num_q_heads, const void* q,
    const uint8_t* k_data, const uint8_t* k_scales, const float* k_global_scale,
    const uint8_t* v_data, const uint8_t* v_scales, const float* v_global_scale,
    int32_t pool_pages, const int32_t* page_table, int32_t max_pages_per_seq,
    const int32_t* seq_lens, float sm_scale, int32_t max_num_splits, void* out, float* lse,
    int32_t* status, nvfp4kv_stream_t stream) {
    const size_t need = nvfp4_paged_decode_workspace_size(layout, batch, num_q_heads,
                                                          max_pages_per_seq, max_num_splits);
    if (need > NVFP4KV_NOALLOC_SCRATCH_BYTES) return NVFP4KV_ERR_WORKSPACE;
    // The scratch address is that of the current device's copy of the array: a stream of another
    // device would run the kernel against memory of the wrong GPU.
    if (stream != nullptr) {
        int cur = 0, sdev = 0;
        if (cudaGetDevice(&cur) != cudaSuccess ||
            cudaStreamGetDevice(reinterpret_cast<cudaStream_t>(stream), &sdev) != cudaSuccess)
            return NVFP4KV_ERR_CUDA;
        if (sdev != cur) return NVFP4KV_ERR_INVALID_ARG;
    }
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return NVFP4KV_ERR_CUDA;
    // Same kernel and split plan as the workspace entry point; every record the split merge
    // reads is written by the same call first, and the finished-piece counts are tagged with
    // the call, so the scratch needs no clearing between calls.
    return nvfp4_paged_decode_attention(layout, batch, num_q_heads, q, k_data, k_scales,
                                        k_global_scale, v_data, v_scales, v_global_scale,
                                        pool_pages, page_table, max_pages_per_seq, seq_lens,
                                        sm_scale, max_num_splits, scratch,
                                        NVFP4KV_NOALLOC_SCRATCH_BYTES, out, lse, status, stream);
}
