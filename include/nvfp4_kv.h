/*
 * nvfp4_kv.h -- C ABI of libnvfp4kv.so: NVFP4 paged KV cache codec and paged decode attention
 * for NVIDIA GB300 (sm_103a).
 *
 * NVFP4 stores each K/V value as a 4-bit E2M1 code, with one E4M3 scale per block of 16 values
 * and one FP32 scale per tensor ("Accelerating Long-Context and Agentic Inference with NVFP4 KV
 * Cache", LMSYS blog: introduction and Figure 1; "KV Cache Compression in TensorRT LLM", NVIDIA:
 * "NVFP4 Cold-Page Compression", Figure 6). A block of 16 values takes 8 bytes of packed codes
 * plus 1 byte of scale (LMSYS, "NVFP4 KV Decode Attention Kernel Implementation").
 *
 * ------------------------------------------------------------------------------------------
 * Page layout (one K or V tensor of one layer; all buffers caller-owned device memory)
 *   H = layout.num_kv_heads, T = layout.page_size (tokens), D = layout.head_dim (D % 16 == 0).
 *   Block b of a token covers head dims 16b .. 16b+15 and has one E4M3 scale byte. Each
 *   (page, head) owns one contiguous run of T tokens in both pools. Two byte packings:
 *   NVFP4KV_PACK_DIM_PAIRS (layout.packing = 0; the K cache of the decode call)
 *     packed data  : uint8 [pool_pages][H][T][D/2]        byte j of a token: head dim 2j in the
 *                                                         low nibble, 2j+1 in the high nibble
 *     block scales : uint8 [pool_pages][H][T][D/16]
 *   NVFP4KV_PACK_TOKEN_PAIRS (layout.packing = 1; the V cache of the decode call; T even)
 *     packed data  : uint8 [pool_pages][H][T/2][D]        byte d of token pair p: head dim d of
 *                                                         token 2p (low) and 2p+1 (high nibble)
 *     block scales : uint8 [pool_pages][H][T/2][D/16][2]  block scales of tokens 2p, 2p+1
 *   Both packings hold the same codes and scales and have the same size; the decode kernel
 *   reduces over head dims for Q.K (dim pairs feed its matmul directly) and over tokens for P.V
 *   (token pairs feed it directly).
 *   16/8-bit pages (BF16 / FP16 / FP8 E4M3 sources and outputs): [pool_pages][H][T][D]
 *   The two NVFP4 pools are read together by attention (TensorRT LLM page, Figure 6: the codes
 *   and the scales sit in separate pools).
 *
 * Numerics (all bit-exact and reproducible; g is the FP32 tensor scale):
 *   encode  a = max |x| over the block; s = E4M3_rne_satfinite(fp32(a / fp32(6 g)));
 *           r = fp32(1 / fp32(s g)) (0 if s g == 0); code_i = E2M1_rne_satfinite(fp32(x_i r)),
 *           sign kept (a negative value rounding to zero is code 0x8). FP8 sources are first
 *           widened to x = fp32(e4m3 * src_scale).
 *   decode  v = e2m1(code) * e4m3(s) (exact); BF16/FP16 out = round_rne(fp32(v g));
 *           FP8 out = E4M3_rne_satfinite(fp32(v fp32(g / dst_scale))).
 *   global scale  g = fp32(amax / 2688) (2688 = 448 * 6 maps the tensor maximum to the top of
 *           both grids); g = 1 when that is zero. A caller may pass any positive g (the LMSYS
 *           page's experiments use 1.0, "Limitations and Ongoing Items").
 *
 * Conventions shared by every call:
 *   - Every pointer except `layout` is device memory owned by the caller; the library never
 *     allocates, frees or synchronises. Work is enqueued on `stream` (may be 0) and returns
 *     without waiting; scalars that come from earlier GPU work (global scales) are passed by
 *     device pointer so a sequence of calls needs no host round trip, and such a sequence can be
 *     captured into a CUDA graph and replayed. Kernels are launched with programmatic dependent
 *     launch: each waits for the earlier work on the stream to complete before it touches
 *     memory (stream order is kept), while its launch overlaps the end of the previous kernel.
 *   - The return value reports host-side validation (NVFP4KV_ERR_INVALID_ARG /
 *     NVFP4KV_ERR_UNSUPPORTED / NVFP4KV_ERR_WORKSPACE) and launch failures (NVFP4KV_ERR_CUDA).
 *     On an error nothing is enqueued.
 *   - Data-dependent faults found on the device are OR-ed into the caller's `status` word
 *     (optional, int32 device memory, NVFP4KV_STATUS_* bits) and nothing traps; the caller
 *     clears the word. A page id outside [0, pool_pages) (PAGE_OOB) or a sequence length outside
 *     [0, max_pages_per_seq * T] (BAD_SEQ_LEN) skips the offending page / sequence. TIMEOUT: the
 *     tagged words of a workspace (a per-call tag in the high 32 bits) are installed over a word
 *     holding a larger tag (garbage) by a compare-and-swap loop bounded at 256 rounds; if that
 *     loop runs out (other CTAs kept changing the word), the count it served never completes,
 *     so the affected (sequence, KV head) pair of a decode call keeps its previous output and
 *     LSE, and a global-scale call may leave g unwritten or too small. No kernel spins on a flag
 *     or a barrier; the decode's asynchronous copies complete without polling.
 *   - `stream` must belong to the current device (or be 0), and every pointer must be memory
 *     that device can address: grids are sized for the current device.
 *   - Buffers must be 16-byte aligned; sources and destinations must not overlap.
 *   - Inputs must be finite. Unused slots of a page (past the end of a sequence) are never read
 *     by attention; the codec encodes every slot of every listed page.
 */
#ifndef NVFP4_KV_H_
#define NVFP4_KV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* nvfp4kv_stream_t;

typedef enum nvfp4kv_status {
    NVFP4KV_OK = 0,
    NVFP4KV_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, bad size or enum value        */
    NVFP4KV_ERR_UNSUPPORTED = 2,  /* valid but not implemented shape (e.g. head_dim 96 decode) */
    NVFP4KV_ERR_WORKSPACE = 3,    /* workspace pointer null or smaller than required          */
    NVFP4KV_ERR_CUDA = 4          /* a CUDA launch or runtime call failed                     */
} nvfp4kv_status;

/* Bits OR-ed into the optional device status word. */
#define NVFP4KV_STATUS_PAGE_OOB 0x1      /* a page id was outside [0, pool_pages): skipped        */
#define NVFP4KV_STATUS_BAD_SEQ_LEN 0x2   /* seq_len < 0 or > max_pages_per_seq * T: seq skipped   */
#define NVFP4KV_STATUS_TIMEOUT 0x4       /* a bounded retry loop on a workspace word gave up       */

typedef enum nvfp4kv_packing {
    NVFP4KV_PACK_DIM_PAIRS = 0,   /* a byte holds two head dims of one token (K cache)          */
    NVFP4KV_PACK_TOKEN_PAIRS = 1  /* a byte holds one head dim of two tokens (V cache)          */
} nvfp4kv_packing;

typedef enum nvfp4kv_dtype {
    NVFP4KV_BF16 = 0,
    NVFP4KV_FP16 = 1,
    NVFP4KV_FP8_E4M3 = 2
} nvfp4kv_dtype;

/* Geometry of one paged K or V tensor. head_dim % 16 == 0; the first three fields > 0. */
typedef struct nvfp4kv_layout {
    int32_t num_kv_heads; /* H */
    int32_t head_dim;     /* D */
    int32_t page_size;    /* T, tokens per page (even for NVFP4KV_PACK_TOKEN_PAIRS) */
    int32_t packing;      /* nvfp4kv_packing of the NVFP4 pool; read by the codec calls */
} nvfp4kv_layout;

/* Human-readable name of a status value (static storage). */
const char* nvfp4kv_status_string(nvfp4kv_status s);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t nvfp4kv_version(void);

/* ------------------------------------------------------------------------------------------
 * Tensor scale. g = fp32(amax / 2688) over every slot of the listed pages, 1.0 when that is 0.
 * The calibrated per-tensor FP32 scale of NVFP4's two-level scaling (LMSYS page, introduction;
 * "Limitations and Ongoing Items": calibration of the FP32 global scale may reduce overflow and
 * underflow).
 *   src            pages of src_dtype, [src_pool_pages][H][T][D]
 *   src_page_ids   [num_pages] page ids into src (NULL = 0 .. num_pages-1)
 *   src_scale      FP8 sources only: device scalar, x = fp32(e4m3 * src_scale) (NULL = 1)
 *   global_scale_out  device float written with g
 *   workspace      device scratch of nvfp4_kv_global_scale_workspace_size() bytes (16): a
 *                  tagged maximum and a tagged count; never needs clearing (a word left by
 *                  another call or holding garbage is replaced through its tag), and the CTA
 *                  that finishes last sets both words back to 0, so a replayed CUDA graph that
 *                  repeats a captured call (same tag) starts clean; calls that can overlap on
 *                  the GPU must not share it
 * One launch: the CTA that finishes last writes g. num_pages == 0 writes g = 1.
 * ------------------------------------------------------------------------------------------ */
size_t nvfp4_kv_global_scale_workspace_size(void);

nvfp4kv_status nvfp4_kv_compute_global_scale(const nvfp4kv_layout* layout,
                                             nvfp4kv_dtype src_dtype, const void* src,
                                             int32_t src_pool_pages,
                                             const int32_t* src_page_ids, int32_t num_pages,
                                             const float* src_scale, float* global_scale_out,
                                             void* workspace, size_t workspace_bytes,
                                             int32_t* status, nvfp4kv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Encode pages to NVFP4 (block amax -> E4M3 scale pick -> E2M1 round-to-nearest-even -> pack).
 * LMSYS page, "Path 1: Initial prefill" and "Path 2: Chunked prefill / Extend" (the current
 * K/V is quantized and written into the NVFP4 cache); TensorRT LLM page, "How It Works"
 * (the paragraph on the fused encode and decode: a batch of pages per call, on the caller's
 * stream).
 *   src / src_page_ids / src_pool_pages   as above (BF16, FP16 or FP8 E4M3 pages)
 *   src_scale      FP8 sources: device scalar (NULL = 1); ignored for 16-bit sources
 *   global_scale   device scalar g (> 0)
 *   dst_data, dst_scales  NVFP4 pools [dst_pool_pages][H][T][D/2] and [..][D/16]
 *   dst_page_ids   [num_pages] destination page ids (NULL = 0 .. num_pages-1)
 * Listed page i goes from src page src_page_ids[i] to dst page dst_page_ids[i]. Two entries
 * naming the same destination page race.
 * ------------------------------------------------------------------------------------------ */
nvfp4kv_status nvfp4_kv_quantize_pages(const nvfp4kv_layout* layout, nvfp4kv_dtype src_dtype,
                                       const void* src, int32_t src_pool_pages,
                                       const int32_t* src_page_ids, const float* src_scale,
                                       const float* global_scale, uint8_t* dst_data,
                                       uint8_t* dst_scales, int32_t dst_pool_pages,
                                       const int32_t* dst_page_ids, int32_t num_pages,
                                       int32_t* status, nvfp4kv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Decode NVFP4 pages to BF16 / FP16 pages, or to FP8 E4M3 pages (the FP8 workspace the
 * extend path gathers the cached prefix into: LMSYS page, "Path 2: Chunked prefill / Extend";
 * the onboard decode of the TensorRT LLM page, "How It Works").
 *   src_data, src_scales, src_pool_pages, src_page_ids   NVFP4 pools and the pages to read
 *   global_scale   device scalar g of the tensor
 *   dst_dtype      NVFP4KV_BF16, NVFP4KV_FP16 or NVFP4KV_FP8_E4M3
 *   dst            [dst_pool_pages][H][T][D] of dst_dtype
 *   dst_page_ids   destination pages (NULL = 0 .. num_pages-1: a gather into consecutive slots)
 *   dst_scale      FP8 output only: device scalar, y = value / dst_scale (NULL = 1)
 * ------------------------------------------------------------------------------------------ */
nvfp4kv_status nvfp4_kv_dequantize_pages(const nvfp4kv_layout* layout, const uint8_t* src_data,
                                         const uint8_t* src_scales, int32_t src_pool_pages,
                                         const int32_t* src_page_ids, const float* global_scale,
                                         nvfp4kv_dtype dst_dtype, void* dst,
                                         int32_t dst_pool_pages, const int32_t* dst_page_ids,
                                         const float* dst_scale, int32_t num_pages,
                                         int32_t* status, nvfp4kv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Extend-path write of the current chunk (LMSYS page, "Path 2: Chunked prefill / Extend": the
 * chunk's K/V are copied into the FP8 workspace that attention reads, and the cache keeps them
 * as NVFP4). One pass over the chunk's pages writes both, reading the chunk once:
 *   NVFP4 pages: exactly as nvfp4_kv_quantize_pages (same codes and scales, same packing)
 *   FP8 pages:   y = E4M3_rne_satfinite(fp32(x * fp32(1 / ws_scale))), layout [page][H][T][D]
 * with x the source value (BF16 / FP16 exactly; FP8 as x = fp32(e4m3 * src_scale), so an FP8
 * chunk written with ws_scale == src_scale gets its own bytes back).
 *   src_dtype      NVFP4KV_BF16, NVFP4KV_FP16 or NVFP4KV_FP8_E4M3 (else NVFP4KV_ERR_UNSUPPORTED)
 *   src, src_pool_pages, src_page_ids, src_scale, global_scale, dst_data, dst_scales,
 *   dst_pool_pages, dst_page_ids   as in nvfp4_kv_quantize_pages
 *   ws_fp8         FP8 E4M3 workspace pool [ws_pool_pages][H][T][D], 16-byte aligned
 *   ws_page_ids    workspace page of each source page (NULL = 0 .. num_pages-1)
 *   ws_scale       device scalar (NULL = 1)
 * A page id outside its pool sets NVFP4KV_STATUS_PAGE_OOB and that page is skipped in all three
 * pools. Source and outputs must not overlap.
 * ------------------------------------------------------------------------------------------ */
nvfp4kv_status nvfp4_kv_extend_write(const nvfp4kv_layout* layout, nvfp4kv_dtype src_dtype,
                                     const void* src, int32_t src_pool_pages,
                                     const int32_t* src_page_ids, const float* src_scale,
                                     const float* global_scale,
                                     uint8_t* dst_data, uint8_t* dst_scales,
                                     int32_t dst_pool_pages, const int32_t* dst_page_ids,
                                     uint8_t* ws_fp8, int32_t ws_pool_pages,
                                     const int32_t* ws_page_ids, const float* ws_scale,
                                     int32_t num_pages, int32_t* status, nvfp4kv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * The extend step in one launch (LMSYS page, "Path 2: Chunked prefill / Extend": the cached
 * prefix of the sequences is dequantized into the FP8 workspace that the extend attention reads,
 * and the current chunk's K/V go into the NVFP4 cache and into that workspace). For each of
 * num_tensors (1 or 2: K and V) tensors this does exactly what these two calls do, byte for byte:
 *   nvfp4_kv_dequantize_pages(prefix pages -> FP8 workspace slots, dst_scale = ws_scale)
 *   nvfp4_kv_extend_write(chunk pages -> NVFP4 pool pages + FP8 workspace slots, ws_scale)
 * but the work items of every tensor's gather and chunk write form one grid: one launch, one
 * ramp and one tail instead of four. Validation and errors are those of the two calls (a pool,
 * id list or pointer the calls would reject gives the same status; nothing is launched); every
 * tensor's chunk has the same dtype (else NVFP4KV_ERR_UNSUPPORTED). The chunk's NVFP4 destination
 * pages must not be among the prefix pages the same call reads, and the workspace slots of the
 * prefix and of the chunk must be distinct (the work items run in no fixed order).
 * ------------------------------------------------------------------------------------------ */
typedef struct nvfp4kv_extend_tensor {
    nvfp4kv_layout layout;           /* geometry and packing of this tensor's NVFP4 pool */
    const float* global_scale;       /* device scalar g of the tensor */
    uint8_t* data;                   /* NVFP4 pool codes  [pool_pages][H][T][D/2] (packing) */
    uint8_t* scales;                 /* NVFP4 pool scales [pool_pages][H][T][D/16] */
    int32_t pool_pages;
    const int32_t* prefix_page_ids;  /* [prefix_pages] pool pages of the cached prefix
                                        (NULL = 0 .. prefix_pages-1) */
    int32_t prefix_pages;
    uint8_t* ws;                     /* FP8 E4M3 workspace [ws_pages][H][T][D], 16-byte aligned */
    int32_t ws_pages;
    const int32_t* ws_prefix_ids;    /* [prefix_pages] workspace slot of each prefix page */
    const int32_t* ws_chunk_ids;     /* [chunk_pages] workspace slot of each chunk page */
    const float* ws_scale;           /* device scalar: FP8 value = x / ws_scale (NULL = 1) */
    int32_t chunk_dtype;             /* nvfp4kv_dtype of the chunk: BF16, FP16 or FP8 E4M3 */
    const void* chunk;               /* chunk pages [chunk_pool_pages][H][T][D] */
    int32_t chunk_pool_pages;
    const int32_t* chunk_page_ids;   /* [chunk_pages] chunk pages to write (NULL = 0 .. n-1) */
    const float* chunk_src_scale;    /* FP8 chunk: x = fp32(e4m3 * chunk_src_scale) (NULL = 1) */
    const int32_t* chunk_dst_ids;    /* [chunk_pages] pool page of each chunk page */
    int32_t chunk_pages;
} nvfp4kv_extend_tensor;

nvfp4kv_status nvfp4_kv_extend_step(const nvfp4kv_extend_tensor* tensors, int32_t num_tensors,
                                    int32_t* status, nvfp4kv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Paged GQA decode attention reading NVFP4 K/V directly from the cache (LMSYS page, "Path 3:
 * Decode" and "NVFP4 KV Decode Attention Kernel Implementation", Figure 3: BF16 queries, packed
 * K/V tiles and their E4M3 block scales staged in shared memory, e2m1x2 conversion in
 * registers, scales applied with packed multiplies, tensor-core matmuls, the global K/V scales
 * folded into the attention scaling).
 *
 * For query head qh of sequence b, with KV head h = qh / (num_q_heads / num_kv_heads), token t
 * at page page_table[b][t / T], slot t % T, and k_t, v_t the decoded values times g_K, g_V:
 *   out[b][qh] = sum_t softmax_t(sm_scale * q . k_t) v_t        (BF16, round to nearest even)
 *   lse[b][qh] = log(sum_t exp(sm_scale * q . k_t))              (natural log; optional)
 * A sequence of length 0 gives out = 0 and lse = -inf.
 *
 * Split-KV: the (sequence, KV head) pairs are cut into 64-token stages (32 at head_dim 256), the
 * stages of all pairs form one list, and the list is cut into equal runs, one per warp (one CTA
 * per SM). Each (run, pair) piece of a pair split over several runs leaves a partial (max, sum,
 * unnormalised output) in the workspace and bumps the pair's counter; the CTA whose warp
 * completes the count merges the pair's partials after its own runs and writes the outputs (one
 * kernel launch). The workspace needs no initialisation: its counters carry a per-call tag, and
 * the CTA that merges a pair sets that pair's counter back to 0, so a replayed CUDA graph that
 * repeats a captured call (same tag) starts clean.
 *   q              BF16 [batch][num_q_heads][D]
 *   k_data, k_scales   NVFP4 K pool in NVFP4KV_PACK_DIM_PAIRS (layout.packing is not read)
 *   v_data, v_scales   NVFP4 V pool in NVFP4KV_PACK_TOKEN_PAIRS
 *   k_global_scale, v_global_scale       device scalars g_K, g_V
 *   page_table     int32 [batch][max_pages_per_seq] device
 *   seq_lens       int32 [batch] device; 0 <= seq_len <= max_pages_per_seq * T
 *   sm_scale       softmax scale (e.g. 1/sqrt(D))
 *   max_num_splits 0 = automatic: one run per warp of one CTA per SM;
 *                  n in 1..64: n * batch * num_kv_heads runs (n runs per pair when all
 *                  sequences have the same length)
 *   workspace      device scratch of nvfp4_paged_decode_workspace_size(...) bytes
 *   out            BF16 [batch][num_q_heads][D]
 *   lse            float [batch][num_q_heads] or NULL
 * Supported: head_dim 64, 128 or 256; 1 <= num_q_heads / num_kv_heads <= 8 (and
 * num_q_heads % num_kv_heads == 0); page_size % 16 == 0.
 * ------------------------------------------------------------------------------------------ */
size_t nvfp4_paged_decode_workspace_size(const nvfp4kv_layout* layout, int32_t batch,
                                         int32_t num_q_heads, int32_t max_pages_per_seq,
                                         int32_t max_num_splits);

nvfp4kv_status nvfp4_paged_decode_attention(
    const nvfp4kv_layout* layout, int32_t batch, int32_t num_q_heads, const void* q,
    const uint8_t* k_data, const uint8_t* k_scales, const float* k_global_scale,
    const uint8_t* v_data, const uint8_t* v_scales, const float* v_global_scale,
    int32_t pool_pages, const int32_t* page_table, int32_t max_pages_per_seq,
    const int32_t* seq_lens, float sm_scale, int32_t max_num_splits, void* workspace,
    size_t workspace_bytes, void* out, float* lse, int32_t* status, nvfp4kv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * nvfp4_paged_decode_attention for callers that cannot allocate device memory. The source
 * pages have no counterpart to this call; it exists for library users who cannot provide a
 * workspace: a plugin inside a framework that owns every device allocation, a serving process
 * that has given all free HBM to its KV-cache pool, or a hot path that must not call cudaMalloc
 * because that synchronises the device.
 *
 * Same arguments, numerics, kernels and split plan as nvfp4_paged_decode_attention, minus the
 * workspace: the split partials live in a fixed array of NVFP4KV_NOALLOC_SCRATCH_BYTES inside
 * the library, which every GPU that loads the library holds until the process exits. The call
 * allocates nothing. The caller still provides inputs and outputs.
 *   - A call whose workspace need (nvfp4_paged_decode_workspace_size with the same arguments)
 *     exceeds NVFP4KV_NOALLOC_SCRATCH_BYTES returns NVFP4KV_ERR_WORKSPACE and enqueues nothing.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 *     with that device current); make that first call before any stream capture. The address
 *     is kept for the life of the process: after cudaDeviceReset (which ends the context that
 *     owns the array) the call must not be used on that device again.
 *   - `stream` must be 0 or a stream of the current device, else NVFP4KV_ERR_INVALID_ARG.
 *   - Every call on a device shares the one array and leaves its contents behind. Calls that
 *     can overlap on the GPU (different streams without ordering between them) race on it.
 * ------------------------------------------------------------------------------------------ */
#define NVFP4KV_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20) /* 32 MiB */

nvfp4kv_status nvfp4_paged_decode_attention_noalloc(
    const nvfp4kv_layout* layout, int32_t batch, int32_t num_q_heads, const void* q,
    const uint8_t* k_data, const uint8_t* k_scales, const float* k_global_scale,
    const uint8_t* v_data, const uint8_t* v_scales, const float* v_global_scale,
    int32_t pool_pages, const int32_t* page_table, int32_t max_pages_per_seq,
    const int32_t* seq_lens, float sm_scale, int32_t max_num_splits, void* out, float* lse,
    int32_t* status, nvfp4kv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Cold-page codec ("KV Cache Compression in TensorRT LLM", NVIDIA: "NVFP4 Cold-Page
 * Compression", "How It Works", Figure 6 and Figure 7). A hot page lives on the GPU in 16 bits
 * per value; a cold page is one fixed-size block per page, holding the NVFP4 data and block
 * scales of K and V and, optionally, lossless bytes copied unchanged. Offload quantizes a batch
 * of hot pages and writes their cold blocks in the same pass; onboard reads cold blocks and
 * writes the dequantized hot pages in the same pass. The cold pool may be pinned host memory
 * (cudaHostAlloc / cudaHostRegister, addressed through unified virtual addressing; the kernels
 * then read or write it over the host link directly, with no separate copy) or device memory.
 *
 * The position-encoded (RoPE) part of K (the same page, "The RoPE part of K"): head dims
 * [first_dim, first_dim + dims) of every K vector, both multiples of 16. Three modes:
 *   NVFP4KV_ROPE_QUANTIZE  quantized like the rest (the default; also rope == NULL)
 *   NVFP4KV_ROPE_SKIP      kept at the hot page's 16-bit precision
 *   NVFP4KV_ROPE_2FP4      two NVFP4 components: c1 encodes x as usual; with v1 = e2m1(c1) *
 *                          e4m3(s1), the residual r = fp32(x - fp32(v1 g)) is encoded the same
 *                          way (same g) into c2; decode is fp32(fp32(v1 g) + fp32(v2 g)),
 *                          then the 16-bit rounding
 *
 * Cold block of one page, byte offsets from its base (every offset a multiple of 16); K's
 * blocks split into the N = D - dims other head dims and the R = dims RoPE dims of each row:
 *   k_data        K codes of the other dims, dim-pair packing [H][T][N/2] (byte j = dims 2j
 *                 low, 2j+1 high nibble, counted within the other dims in order)
 *   k_scales      their block scales [H][T][N/16], E4M3
 *   k_rope        SKIP: the RoPE values [H][T][R] (16-bit); 2FP4: codes of c1 [H][T][R/2]
 *   k_rope_scales 2FP4: block scales of c1 [H][T][R/16]
 *   k_rope2       2FP4: codes of c2 [H][T][R/2]
 *   k_rope2_scales 2FP4: block scales of c2 [H][T][R/16]
 *   v_data        V codes, dim-pair packing [H][T][D/2]
 *   v_scales      V block scales [H][T][D/16]
 *   extra         extra_bytes copied unchanged (e.g. state that must not be quantized)
 * each part starting at the previous part's end rounded up to 16 (parts a mode does not use are
 * -1 and take no room; with QUANTIZE, N = D); `bytes` is the end of the extra part. When
 * H*T*D/16 is a multiple of 16 and QUANTIZE is used there is no padding and
 * bytes = 2 * (9/16) * H*T*D + extra_bytes. Slot s of the cold pool starts at cold + s * bytes.
 * The layout's `packing` field is ignored here (cold blocks always use dim pairs).
 * ------------------------------------------------------------------------------------------ */
typedef enum nvfp4kv_rope_mode {
    NVFP4KV_ROPE_QUANTIZE = 0,
    NVFP4KV_ROPE_SKIP = 1,
    NVFP4KV_ROPE_2FP4 = 2
} nvfp4kv_rope_mode;

typedef struct nvfp4kv_cold_rope {
    int32_t mode;       /* nvfp4kv_rope_mode */
    int32_t first_dim;  /* multiple of 16 */
    int32_t dims;       /* multiple of 16, > 0, first_dim + dims <= head_dim (<= 2048) */
} nvfp4kv_cold_rope;

typedef struct nvfp4kv_cold_block_layout {
    int64_t k_data, k_scales, k_rope, k_rope_scales, k_rope2, k_rope2_scales;
    int64_t v_data, v_scales, extra, bytes;
} nvfp4kv_cold_block_layout;

/* Fills *out for `layout`, the RoPE option (NULL = QUANTIZE) and extra_bytes (>= 0, a multiple
 * of 16). Host only. */
nvfp4kv_status nvfp4_kv_cold_block_layout(const nvfp4kv_layout* layout,
                                          const nvfp4kv_cold_rope* rope, int32_t extra_bytes,
                                          nvfp4kv_cold_block_layout* out);

/* Offload: hot page hot_page_ids[i] -> cold slot cold_slot_ids[i], for i < num_pages.
 *   hot_dtype          NVFP4KV_BF16 or NVFP4KV_FP16 (else NVFP4KV_ERR_UNSUPPORTED)
 *   hot_k, hot_v       hot pools, page p of K at hot_k + p * hot_page_stride elements, laid out
 *                      [H][T][D] (K and V may be two pools, or one pool holding both:
 *                      hot_v = hot_k + H*T*D and hot_page_stride = 2*H*T*D); 16-byte aligned
 *   hot_page_stride    elements between consecutive pages, >= H*T*D, a multiple of 8
 *   hot_pool_pages, hot_page_ids   pages in each hot pool; ids (NULL = 0 .. num_pages-1)
 *   k_global_scale, v_global_scale device scalars g of K and V (NULL = 1); codes and scales
 *                      are exactly those of nvfp4_kv_quantize_pages with the same g
 *   rope               host pointer, the RoPE part of K and its mode (NULL = QUANTIZE)
 *   extra, extra_page_stride, extra_bytes   lossless bytes of hot page p at
 *                      extra + p * extra_page_stride (16-byte aligned; stride a multiple of 16);
 *                      extra_bytes = 0 (extra may be NULL) copies none
 *   cold, cold_slots, cold_slot_ids  cold pool of cold_slots blocks (16-byte aligned); slots
 *                      (NULL = 0 .. num_pages-1)
 * A page id or slot outside its pool sets NVFP4KV_STATUS_PAGE_OOB and that page is skipped. */
nvfp4kv_status nvfp4_kv_offload_pages(
    const nvfp4kv_layout* layout, nvfp4kv_dtype hot_dtype, const void* hot_k, const void* hot_v,
    int64_t hot_page_stride, int32_t hot_pool_pages, const int32_t* hot_page_ids,
    const float* k_global_scale, const float* v_global_scale, const nvfp4kv_cold_rope* rope,
    const uint8_t* extra, int64_t extra_page_stride, int32_t extra_bytes, uint8_t* cold,
    int32_t cold_slots, const int32_t* cold_slot_ids, int32_t num_pages, int32_t* status,
    nvfp4kv_stream_t stream);

/* Onboard: cold slot cold_slot_ids[i] -> hot page hot_page_ids[i], for i < num_pages. Values
 * are exactly those of nvfp4_kv_dequantize_pages (BF16 / FP16 output) with the same g (RoPE
 * part: SKIP copies it back, 2FP4 decodes as above); the extra bytes are copied back
 * unchanged. Arguments as in nvfp4_kv_offload_pages, with the same `rope`. */
nvfp4kv_status nvfp4_kv_onboard_pages(
    const nvfp4kv_layout* layout, const uint8_t* cold, int32_t cold_slots,
    const int32_t* cold_slot_ids, const float* k_global_scale, const float* v_global_scale,
    const nvfp4kv_cold_rope* rope, nvfp4kv_dtype hot_dtype, void* hot_k, void* hot_v, int64_t hot_page_stride,
    int32_t hot_pool_pages, const int32_t* hot_page_ids, uint8_t* extra,
    int64_t extra_page_stride, int32_t extra_bytes, int32_t num_pages, int32_t* status,
    nvfp4kv_stream_t stream);

/* Device address of pinned host memory (cudaHostGetDevicePointer): the address to pass as
 * `cold` when the cold pool is pinned host memory. NVFP4KV_ERR_INVALID_ARG if host_ptr is not
 * pinned memory known to CUDA. Host only; enqueues nothing. */
nvfp4kv_status nvfp4_kv_host_device_pointer(void* host_ptr, void** device_ptr);

/* ------------------------------------------------------------------------------------------
 * The two roundings of the encoder on their own, for exhaustive verification over fp32 inputs:
 * target 0 writes E2M1 codes (RNE, satfinite at 6, sign kept, one code per byte), target 1
 * writes E4M3 bytes (RNE, satfinite at 448, sign kept). x: n finite floats; out: n bytes.
 * ------------------------------------------------------------------------------------------ */
nvfp4kv_status nvfp4_kv_round_f32(const float* x, size_t n, int32_t target, uint8_t* out,
                                  nvfp4kv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_KV_H_ */
