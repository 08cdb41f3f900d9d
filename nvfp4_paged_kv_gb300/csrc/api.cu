// Library-wide C entry points of libnvfp4kv.so that belong to no kernel.
#include "../../include/nvfp4_kv.h"

extern "C" const char* nvfp4kv_status_string(nvfp4kv_status s) {
    switch (s) {
    case NVFP4KV_OK: return "NVFP4KV_OK";
    case NVFP4KV_ERR_INVALID_ARG: return "NVFP4KV_ERR_INVALID_ARG: null/misaligned pointer or bad size";
    case NVFP4KV_ERR_UNSUPPORTED: return "NVFP4KV_ERR_UNSUPPORTED: shape not implemented";
    case NVFP4KV_ERR_WORKSPACE: return "NVFP4KV_ERR_WORKSPACE: workspace missing or too small";
    case NVFP4KV_ERR_CUDA: return "NVFP4KV_ERR_CUDA: CUDA launch or runtime error";
    }
    return "unknown nvfp4kv_status";
}

extern "C" int32_t nvfp4kv_version(void) { return 100; /* 0.1.0 */ }
