/* A plain C99 caller of the NVFP4 KV library.
 *
 * Compiled with gcc -std=c99 -pedantic -Wall -Wextra -Werror against include/nvfp4_kv.h and
 * linked to libnvfp4kv.so, it shows that the header is valid C (no C++ in the declarations,
 * no missing includes, no implicit conversions a C compiler warns about) and that a C program
 * resolves and calls the exported symbols. It calls only what runs on the host: the version
 * and status strings, the size and layout queries, and argument checks that fail before any
 * CUDA call. Pointers passed to the failing checks are never dereferenced by the library.
 * Exit status 0 means every check held; each failed check prints one line. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "nvfp4_kv.h"

static int failures = 0;

static void check(int ok, const char* what) {
    if (!ok) {
        printf("FAILED: %s\n", what);
        ++failures;
    }
}

static int aligned16(int64_t off) { return off == -1 || (off >= 0 && off % 16 == 0); }

int main(void) {
    nvfp4kv_layout lay;
    nvfp4kv_layout bad;
    nvfp4kv_layout d96;
    nvfp4kv_cold_block_layout cold;
    nvfp4kv_cold_rope rope;
    nvfp4kv_extend_tensor parts[3];
    void* fake = (void*)(uintptr_t)4096;     /* never dereferenced: validation fails first */
    int s;

    lay.num_kv_heads = 8;
    lay.head_dim = 128;
    lay.page_size = 64;
    lay.packing = NVFP4KV_PACK_DIM_PAIRS;
    bad = lay;
    bad.head_dim = 120;                       /* not a multiple of 16 */
    d96 = lay;
    d96.head_dim = 96;                        /* valid geometry, no decode kernel */

    check(nvfp4kv_version() >= 100, "version");
    for (s = NVFP4KV_OK; s <= NVFP4KV_ERR_CUDA; ++s) {
        const char* name = nvfp4kv_status_string((nvfp4kv_status)s);
        check(name != NULL && strncmp(name, "NVFP4KV_", 8) == 0, "status string");
    }

    check(nvfp4_kv_global_scale_workspace_size() == 16, "global scale workspace size");
    {
        size_t w1 = nvfp4_paged_decode_workspace_size(&lay, 2, 32, 16, 4);
        size_t w2 = nvfp4_paged_decode_workspace_size(&lay, 4, 32, 16, 4);
        check(w1 > 0 && w2 > w1, "decode workspace grows with the batch");
        check(nvfp4_paged_decode_workspace_size(&bad, 2, 32, 16, 4) == 0,
              "decode workspace of an invalid layout");
        check(nvfp4_paged_decode_workspace_size(&lay, 2, 36, 16, 4) == 0,
              "decode workspace with num_q_heads not a multiple of num_kv_heads");
        check(nvfp4_paged_decode_workspace_size(&lay, 2, 32, 16, 65) == 0,
              "decode workspace with too many splits");
    }

    /* Cold block: two NVFP4 tensors of 9/16 byte per element plus the extra bytes. */
    check(nvfp4_kv_cold_block_layout(&lay, NULL, 32, &cold) == NVFP4KV_OK, "cold layout");
    check(cold.bytes == 2 * 9 * 8 * 64 * 128 / 16 + 32, "cold block bytes");
    check(cold.k_data == 0 && cold.k_rope == -1 && cold.k_rope2 == -1, "cold K parts");
    check(aligned16(cold.k_scales) && aligned16(cold.v_data) && aligned16(cold.v_scales) &&
              aligned16(cold.extra), "cold parts start on 16 bytes");
    check(cold.k_data < cold.k_scales && cold.k_scales < cold.v_data &&
              cold.v_data < cold.v_scales && cold.v_scales < cold.extra &&
              cold.extra + 32 == cold.bytes, "cold parts in order");
    rope.mode = NVFP4KV_ROPE_SKIP;
    rope.first_dim = 64;
    rope.dims = 64;
    check(nvfp4_kv_cold_block_layout(&lay, &rope, 0, &cold) == NVFP4KV_OK && cold.k_rope >= 0 &&
              aligned16(cold.k_rope), "cold layout with the RoPE part kept");
    check(nvfp4_kv_cold_block_layout(&lay, NULL, 8, &cold) == NVFP4KV_ERR_INVALID_ARG,
          "cold extra bytes not a multiple of 16");
    rope.dims = 8;
    check(nvfp4_kv_cold_block_layout(&lay, &rope, 0, &cold) == NVFP4KV_ERR_INVALID_ARG,
          "cold RoPE dims not a multiple of 16");

    /* Argument checks that fail before any CUDA call. */
    check(nvfp4_kv_quantize_pages(&bad, NVFP4KV_BF16, fake, 1, NULL, NULL, (const float*)fake,
                                  (uint8_t*)fake, (uint8_t*)fake, 1, NULL, 1, NULL,
                                  NULL) == NVFP4KV_ERR_INVALID_ARG,
          "quantize with head_dim 120");
    check(nvfp4_kv_quantize_pages(&lay, (nvfp4kv_dtype)7, fake, 1, NULL, NULL,
                                  (const float*)fake, (uint8_t*)fake, (uint8_t*)fake, 1, NULL, 1,
                                  NULL, NULL) == NVFP4KV_ERR_INVALID_ARG,
          "quantize with an unknown dtype");
    check(nvfp4_paged_decode_attention(&d96, 1, 16, fake, (const uint8_t*)fake,
                                       (const uint8_t*)fake, (const float*)fake,
                                       (const uint8_t*)fake, (const uint8_t*)fake,
                                       (const float*)fake, 1, (const int32_t*)fake, 1,
                                       (const int32_t*)fake, 0.1f, 0, fake, 1 << 20, fake, NULL,
                                       NULL, NULL) == NVFP4KV_ERR_UNSUPPORTED,
          "decode with head_dim 96");
    check(nvfp4_paged_decode_attention(&lay, 0, 32, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1,
                                       NULL, 1, NULL, 0.1f, 0, NULL, 0, NULL, NULL, NULL,
                                       NULL) == NVFP4KV_OK,
          "decode of an empty batch is a no-op");
    check(nvfp4_paged_decode_attention_noalloc(&lay, 256, 64, fake, (const uint8_t*)fake,
                                               (const uint8_t*)fake, (const float*)fake,
                                               (const uint8_t*)fake, (const uint8_t*)fake,
                                               (const float*)fake, 1, (const int32_t*)fake, 2048,
                                               (const int32_t*)fake, 0.1f, 64, fake, NULL, NULL,
                                               NULL) == NVFP4KV_ERR_WORKSPACE,
          "no-allocation decode beyond its fixed scratch");
    check(nvfp4_kv_round_f32(NULL, 0, 0, NULL, NULL) == NVFP4KV_OK, "round of no values");
    check(nvfp4_kv_round_f32((const float*)fake, 4, 2, (uint8_t*)fake, NULL) ==
              NVFP4KV_ERR_INVALID_ARG, "round to an unknown target");
    memset(parts, 0, sizeof parts);
    check(nvfp4_kv_extend_step(NULL, 1, NULL, NULL) == NVFP4KV_ERR_INVALID_ARG,
          "extend step without tensors");
    check(nvfp4_kv_extend_step(parts, 3, NULL, NULL) == NVFP4KV_ERR_INVALID_ARG,
          "extend step with three tensors");
    parts[0].layout = bad;
    check(nvfp4_kv_extend_step(parts, 1, NULL, NULL) == NVFP4KV_ERR_INVALID_ARG,
          "extend step with head_dim 120");
    parts[0].layout = lay;
    parts[0].chunk_pages = 1;
    parts[0].chunk_dtype = 7;
    check(nvfp4_kv_extend_step(parts, 1, NULL, NULL) == NVFP4KV_ERR_UNSUPPORTED,
          "extend step with an unknown chunk dtype");
    /* a first tensor that passes every check, then a second whose chunk dtype differs */
    parts[0].chunk_dtype = NVFP4KV_BF16;
    parts[0].global_scale = (const float*)fake;
    parts[0].data = (uint8_t*)fake;
    parts[0].scales = (uint8_t*)fake;
    parts[0].pool_pages = 1;
    parts[0].prefix_pages = 1;
    parts[0].ws = (uint8_t*)fake;
    parts[0].ws_pages = 2;
    parts[0].chunk = fake;
    parts[0].chunk_pool_pages = 1;
    parts[1] = parts[0];
    parts[1].chunk_dtype = NVFP4KV_FP16;
    check(nvfp4_kv_extend_step(parts, 2, NULL, NULL) == NVFP4KV_ERR_UNSUPPORTED,
          "extend step with two chunk dtypes");
    parts[1].chunk_dtype = NVFP4KV_BF16;
    parts[1].ws = NULL;
    check(nvfp4_kv_extend_step(parts, 2, NULL, NULL) == NVFP4KV_ERR_INVALID_ARG,
          "extend step whose second tensor has no workspace");

    check(nvfp4_kv_dequantize_pages(&lay, (const uint8_t*)fake, (const uint8_t*)fake, 1, NULL,
                                    (const float*)fake, (nvfp4kv_dtype)9, fake, 1, NULL, NULL, 1,
                                    NULL, NULL) == NVFP4KV_ERR_INVALID_ARG,
          "dequantize to an unknown dtype");
    check(nvfp4_kv_dequantize_pages(&lay, (const uint8_t*)fake, (const uint8_t*)fake, 1, NULL,
                                    (const float*)fake, NVFP4KV_BF16,
                                    (void*)((uintptr_t)4096 + 4), 1, NULL, NULL, 1, NULL,
                                    NULL) == NVFP4KV_ERR_INVALID_ARG,
          "dequantize to a misaligned destination");
    check(nvfp4_kv_compute_global_scale(&lay, NVFP4KV_BF16, fake, 1, NULL, 1, NULL, NULL, fake,
                                        16, NULL, NULL) == NVFP4KV_ERR_INVALID_ARG,
          "global scale without an output");
    check(nvfp4_kv_extend_write(&lay, NVFP4KV_BF16, fake, 1, NULL, NULL, (const float*)fake,
                                (uint8_t*)fake, (uint8_t*)fake, 1, NULL, NULL, 1, NULL, NULL, 1,
                                NULL, NULL) == NVFP4KV_ERR_INVALID_ARG,
          "extend write without a workspace");
    {
        /* forced splits: the workspace need is known on the host, no device query */
        size_t need = nvfp4_paged_decode_workspace_size(&lay, 2, 32, 4, 2);
        check(need > 0, "decode workspace with forced splits");
        check(nvfp4_paged_decode_attention(&lay, 2, 32, fake, (const uint8_t*)fake,
                                           (const uint8_t*)fake, (const float*)fake,
                                           (const uint8_t*)fake, (const uint8_t*)fake,
                                           (const float*)fake, 8, (const int32_t*)fake, 4,
                                           (const int32_t*)fake, 0.1f, 2, fake, need - 1, fake,
                                           NULL, NULL, NULL) == NVFP4KV_ERR_WORKSPACE,
              "decode with a workspace one byte short");
        check(nvfp4_paged_decode_attention(&lay, 2, 72, fake, (const uint8_t*)fake,
                                           (const uint8_t*)fake, (const float*)fake,
                                           (const uint8_t*)fake, (const uint8_t*)fake,
                                           (const float*)fake, 8, (const int32_t*)fake, 4,
                                           (const int32_t*)fake, 0.1f, 2, fake, need, fake, NULL,
                                           NULL, NULL) == NVFP4KV_ERR_UNSUPPORTED,
              "decode with a query group of 9");
        check(nvfp4_paged_decode_attention(&lay, 2, 32, (const void*)((uintptr_t)4096 + 2),
                                           (const uint8_t*)fake, (const uint8_t*)fake,
                                           (const float*)fake, (const uint8_t*)fake,
                                           (const uint8_t*)fake, (const float*)fake, 8,
                                           (const int32_t*)fake, 4, (const int32_t*)fake, 0.1f,
                                           2, fake, need, fake, NULL, NULL,
                                           NULL) == NVFP4KV_ERR_INVALID_ARG,
              "decode with misaligned queries");
    }
    rope.mode = NVFP4KV_ROPE_2FP4;
    rope.first_dim = 120;
    rope.dims = 16;
    check(nvfp4_kv_offload_pages(&lay, NVFP4KV_BF16, fake, fake, 8 * 64 * 128, 1, NULL, NULL,
                                 NULL, &rope, NULL, 0, 0, (uint8_t*)fake, 1, NULL, 1, NULL,
                                 NULL) == NVFP4KV_ERR_INVALID_ARG,
          "offload with a RoPE part past head_dim");

    if (failures == 0) printf("all checks passed\n");
    return failures == 0 ? 0 : 1;
}
