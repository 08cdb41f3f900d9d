// Split-KV paged GQA decode attention over NVFP4 K/V for sm_103a, with its split merge.
//
// What it computes ("Accelerating Long-Context and Agentic Inference with NVFP4 KV Cache",
// LMSYS: "Path 3: Decode", "NVFP4 KV Decode Attention Kernel Implementation", Figure 3): for
// each sequence and query head, softmax(sm_scale q.K^T) V over the sequence's tokens, with K
// and V read in their packed NVFP4 form straight from the paged cache and dequantized in
// registers. The global K/V scales are folded into the score scale and the final output (the
// page applies them through the attention matmuls' scaling parameters).
//
// Design for GB300 (the SM120 kernel of the LMSYS page is prior art, not the blueprint):
//  * Work is a flat list of stages: stage j of pair (sequence b, KV head h) covers tokens
//    [TOK j, TOK j + TOK) of b (TOK = 64 tokens, 32 at head_dim 256), pairs in (b, h) order.
//    One persistent CTA per SM runs (12 warps at head_dim 128, 16 at 64, 8 at 256: all warps
//    of an SM are equally old, so none is favoured by the schedulers), and the list is cut into
//    equal runs, one per warp, so every warp streams the same number of bytes whatever the mix
//    of sequence lengths. A run may cross pairs; each (warp, pair) piece of a pair that is
//    split over several warps leaves one partial record gw + bh (gw the warp's run, bh the
//    pair), so records never collide and their number is bounded by runs + pairs before any
//    length is known.
//  * Every warp is an independent pipeline: after the stage prefix and the query cache fill at
//    the start, no barrier ties the warps of a CTA together. A warp streams its run through its
//    own ring of two shared-memory slots with asynchronous copies (cp.async, 16 bytes per lane,
//    completion per warp by wait_group), straight across pair boundaries: the packed K rows,
//    the token-pair packed V rows and both scale pools of a stage are four contiguous runs of
//    its page. The page ids come from a 32-entry register window of the page table (one id per
//    lane) whose successor is loaded a window ahead; the queries of the pairs the CTA touches
//    (consecutive pairs, so one contiguous slice of q) are staged in shared memory at the
//    start. A small header in each slot tells the consumer which sub-tiles are real, where the
//    piece starts and ends and which pair it belongs to, so a pair boundary costs no wait for
//    global memory.
//  * S^T = K^ Q^T runs on the tensor cores with tokens as M = 16 and the GQA query group as
//    N = 8 (mma.sync m16n8k16, FP16 in, FP32 accumulate). K is stored dim-pair packed, so every
//    converted byte (cvt.rn.f16x2.e2m1x2) is one A-register: two adjacent head dims of one
//    token, exact in FP16, times its E4M3 block scale (exact). Q is brought into FP16 exactly by
//    a per-head power of two; head dims inside a k-step are permuted identically in K and Q.
//  * online softmax per stage in the log2 domain, column maxima by warp shuffles on packed
//    FP16 pairs; the running maximum moves only when it grows by more than 2^8, so accumulator
//    rescaling is rare. P^T moves to the B-operand layout with movmatrix.
//  * O^T += V^^T P^T with head dims as M: V is stored token-pair packed, so every converted byte
//    is one A-register (one head dim of two adjacent tokens) times the pair's two block scales.
//  * at the end of a piece the warp writes the BF16 output and the natural-log LSE directly
//    when the piece is the whole pair, otherwise its record (from registers), then bumps the
//    pair's finished-piece count (a word tagged with the call, release/acquire fences around
//    the atomic). The warp whose count completes the pair queues it in its CTA; after every
//    run of the CTA is done, the CTA merges its queued pairs by log-sum-exp: the records of as
//    many pairs as fit are staged in shared memory in one round trip, and every thread then
//    takes float4 output columns and forms its head's weights from the staged maxima itself.
//    A pair with more records than fit at once is merged by chunks.
// Bytes per (token, KV head) at head_dim 128: 64 + 8 (K) + 64 + 8 (V) = 144.
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_util.h"

namespace nvfp4kv {
namespace {

constexpr int kMaxGroup = 8;
constexpr int kMaxSplits = 64;     // bound of the caller-forced split count
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kFirst = 1u, kLast = 2u;  // slot header flags: first / last stage of a piece
constexpr int kSmemPerSm = 233472;           // shared memory of an SM (228 KiB)

template <int D>
struct Geo {
    static constexpr int TOK = (D == 256) ? 32 : 64;  // tokens of a stage
    static constexpr int SUB = TOK / 16;              // 16-token MMA tiles of a stage
    static constexpr int NB = D / 16;                 // blocks (= scales) per token row
    static constexpr int SK = TOK * D / 2;            // packed K rows of a stage
    static constexpr int SV = TOK * D / 2;            // token-pair V rows (TOK / 2 rows of D)
    static constexpr int SS = TOK * NB;               // one scale pool of a stage
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = SK;
    static constexpr int KS_OFF = SK + SV;
    static constexpr int VS_OFF = KS_OFF + SS;
    static constexpr int HDR_OFF = VS_OFF + SS;  // slot header (8 words)
    static constexpr int SLOT = HDR_OFF + 32;
    static constexpr int SLOTS = 2;              // ring slots per warp: one in flight, one computed
    // warps of the one CTA per SM (register budget: 16 x 32 x 128, 12 x 32 x 170, 8 x 32 x 255)
    static constexpr int WARPS = (D == 64) ? 16 : (D == 128 ? 12 : 8);
    static constexpr int THREADS = WARPS * 32;
    static constexpr int RING = SLOTS * SLOT;     // per warp
    static constexpr int QCACHE = (D == 128) ? 8192 : 16384;  // queries of the CTA's pairs
    static constexpr int Q_OFF = WARPS * RING;
    static constexpr int SMEM = Q_OFF + QCACHE;
    static constexpr int KSTEPS = D / 16;       // k-steps of S^T = K Q^T
    static constexpr int CHUNK = D / 8;         // bytes of a row one quad lane owns
    static constexpr int CW = CHUNK / 4;        // ... as 32-bit words
    static constexpr int VCH = D / 16;          // 16-byte chunks per V pair row
    static constexpr int SWZ = (VCH < 8 ? VCH : 8) - 1;  // chunk XOR mask
    static constexpr int DCH = SK / (16 * 32);  // 16-byte chunks per lane of one data pool
    static constexpr int SUB_DIV = D / 64;      // data chunk i of a lane lies in sub-tile i / SUB_DIV
    static constexpr int SCH = SS / 16;         // 16-byte chunks of one scale pool
    static constexpr int SC_PER_LANE = 2 * SCH / 32;
    static_assert(DCH * 32 * 16 == SK && DCH == SUB * SUB_DIV, "copy split");
    static_assert(SC_PER_LANE * 32 == 2 * SCH, "scale copy split");
    static_assert(SLOT % 16 == 0 && RING % 16 == 0, "16-byte aligned slots");
    static_assert(SMEM + 1024 + 512 <= kSmemPerSm, "shared memory budget");
};

struct DecodeParams {
    const uint16_t* q;  // BF16 bit patterns [B][Hq][D]
    const uint8_t* kd;
    const uint8_t* ks;
    const uint8_t* vd;
    const uint8_t* vs;
    const float* gk;
    const int32_t* page_table;
    const int32_t* seq_lens;
    const float* gv;
    uint16_t* out;      // BF16 bits [B][Hq][D]
    float* lse;         // [B][Hq] or null
    unsigned long long* done;  // [B * H] tagged counts of finished pieces of each pair
    float* rec_o;       // [records][G][D] unnormalised output
    float* rec_ml;      // [records][G][2] running max (log2 domain), sum of exp2(x - max)
    int32_t* status;
    uint64_t t_magic;   // ceil(2^64 / T)
    uint32_t nonce;     // tag of this call
    int32_t B, Hq, H, G, T, pool_pages, max_pages, num_runs;
    float sm_scale;
};

__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b) {
    const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a),
                              *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
}

template <int N>
__device__ __forceinline__ void lds_words(uint32_t (&w)[N], uint32_t addr) {
    if constexpr (N == 1) {
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w[0]) : "r"(addr));
    } else if constexpr (N == 2) {
        asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "r"(addr));
    } else {
#pragma unroll
        for (int i = 0; i < N; i += 4)
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(w[i]), "=r"(w[i + 1]), "=r"(w[i + 2]), "=r"(w[i + 3])
                         : "r"(addr + 4 * i));
    }
}

__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// Shared-memory offset of byte x of token-pair row pr of a stage's V rows: 16-byte chunks are
// XOR-swizzled by the row so that the 4 lanes of a quad (rows c and c+4) hit distinct banks.
template <int D>
__device__ __forceinline__ uint32_t v_swz(int pr, int x) {
    return static_cast<uint32_t>(pr * D + ((((x >> 4) ^ (pr & Geo<D>::SWZ))) << 4) + (x & 15));
}

// 16-byte asynchronous copy global -> shared, with compile-time offsets on both addresses, under
// the L2 policy `pol` (evict-first for the K/V stream: each byte is read once per call, so its
// lines are the first to go and other lines, such as outputs still waiting to be written back,
// are not pushed out by it).
template <int OFF_S, int OFF_G>
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0+%2], [%1+%3], 16, %4;" ::"r"(dst),
                 "l"(src), "n"(OFF_S), "n"(OFF_G), "l"(pol)
                 : "memory");
}
// The same with a source size of 16 or 0 bytes (0: the 16 bytes are zero-filled, nothing read).
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, uint32_t bytes,
                                                 uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst),
                 "l"(src), "r"(bytes), "l"(pol)
                 : "memory");
}
// 16-byte asynchronous copy with the default L2 policy (the queries: read once per piece).
__device__ __forceinline__ void cp_async16_plain(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename F, int... I>
__device__ __forceinline__ void static_for_impl(F&& f, std::integer_sequence<int, I...>) {
    (f(std::integral_constant<int, I>{}), ...);
}
// f(std::integral_constant<int, i>) for i = 0 .. N-1, each i a compile-time constant.
template <int N, typename F>
__device__ __forceinline__ void static_for(F&& f) {
    static_for_impl(f, std::make_integer_sequence<int, N>{});
}

// Stages (of tok tokens) of a sequence of length L; 0 for an invalid length.
__device__ __forceinline__ int seq_stages(int L, int max_tokens, int tok) {
    return (L > 0 && L <= max_tokens) ? (L + tok - 1) / tok : 0;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Merge the records of pair (b, h) (pieces of runs gf .. gl, records gf + bh .. gl + bh, one
// contiguous block) by log-sum-exp and write its outputs; the whole CTA, after its runs. The
// block is staged in shared memory by asynchronous copies (one round trip), the (max, sum) of
// each query head reduced by one warp per head, and the weighted sum of the records' outputs
// split over the threads: thread t takes one float4 column of the G x D outputs and every R-th
// record of the chunk, R = threads / columns.
template <int D>
__device__ __forceinline__ void merge_pair(const DecodeParams& p, int b, int h, int64_t rec0,
                                           int n, uint8_t* smem) {
    using G_ = Geo<D>;
    constexpr int NT = G_::THREADS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = p.G;
    const int64_t bh = static_cast<int64_t>(b) * p.H + h;
    // no fence here: the thread that saw the count complete fenced after it, and the CTA
    // barrier between that and this merge orders every thread's reads after the fence
    if (tid == 0) atomicExch(p.done + bh, 0ull);  // a replay with the same tag starts from 0
    const int rec_bytes = G * D * 4;
    // shared memory: records' outputs [KC][G][D], (max, sum) [KC][G], weights [KC][G],
    // per-head running max / sum / rescale [8] x 3, partial sums [NT] float4
    constexpr int kStage = G_::Q_OFF - (NT * 16 + 3 * kMaxGroup * 4) - 2048;
    const int KC = min(n, min(64, kStage / (rec_bytes + G * 12)));
    float* o_s = reinterpret_cast<float*>(smem);
    float2* ml_s = reinterpret_cast<float2*>(smem + KC * rec_bytes);
    float* w_s = reinterpret_cast<float*>(smem + KC * (rec_bytes + G * 8));
    float* hd_s = reinterpret_cast<float*>(smem + kStage);  // M, L, rescale per head
    float4* part_s = reinterpret_cast<float4*>(smem + kStage + 3 * kMaxGroup * 4);
    const int C4 = G * D / 4;                    // float4 columns of the outputs
    // columns per thread when there are more columns than threads (head_dim 256, 8 heads), else
    // R = threads / columns groups of records per column
    constexpr int CPT = (kMaxGroup * D / 4 + NT - 1) / NT;
    const int R = max(1, NT / C4);
    const int grp = (R > 1) ? tid / C4 : 0;
    const int col0 = (R > 1) ? tid % C4 : tid;
    if (tid < G) {
        hd_s[tid] = -INFINITY;
        hd_s[kMaxGroup + tid] = 0.0f;
    }
    float4 acc[CPT];
#pragma unroll
    for (int j = 0; j < CPT; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    const uint32_t s_base = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    for (int k0 = 0; k0 < n; k0 += KC) {
        const int nk = min(KC, n - k0);
        // stage the chunk's records: outputs and (max, sum), both contiguous in global memory
        {
            const uint8_t* src = reinterpret_cast<const uint8_t*>(p.rec_o + (rec0 + k0) * G * D);
            const int nc = nk * rec_bytes / 16;
            for (int i = tid; i < nc; i += NT) cp_async16_plain(s_base + 16 * i, src + 16 * i);
            const float* msrc = p.rec_ml + (rec0 + k0) * G * 2;
            for (int i = tid; i < nk * G; i += NT) ml_s[i] = __ldcg(reinterpret_cast<const float2*>(msrc) + i);
            cp_async_commit();
            cp_async_wait<0>();
        }
        __syncthreads();
        // per head: the chunk's maximum, the running maximum, weights and sum
        if (warp < G) {
            const int g = warp;
            float mx = -INFINITY;
            for (int k = lane; k < nk; k += 32) mx = fmaxf(mx, ml_s[k * G + g].x);
            mx = warp_max(mx);
            const float Mo = hd_s[g];
            const float Mn = fmaxf(Mo, mx);
            float s = 0.0f;
            for (int k = lane; k < nk; k += 32) {
                const float2 ml = ml_s[k * G + g];
                const float w = (ml.x == -INFINITY) ? 0.0f : exp2f(ml.x - Mn);
                w_s[k * G + g] = w;
                s += w * ml.y;
            }
            s = warp_sum(s);
            __syncwarp();
            if (lane == 0) {
                const float a = (Mo == -INFINITY) ? 0.0f : exp2f(Mo - Mn);
                hd_s[g] = Mn;
                hd_s[kMaxGroup + g] = hd_s[kMaxGroup + g] * a + s;
                hd_s[2 * kMaxGroup + g] = a;
            }
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const int col = col0 + NT * j;
            if (grp >= R || col >= C4) continue;
            const int g_col = col * 4 / D;
            const float a = hd_s[2 * kMaxGroup + g_col];
            float4 v4 = acc[j];
            v4.x *= a;
            v4.y *= a;
            v4.z *= a;
            v4.w *= a;
            for (int k = grp; k < nk; k += R) {
                const float w = w_s[k * G + g_col];
                const float4 v = reinterpret_cast<const float4*>(o_s + k * G * D)[col];
                v4.x += w * v.x;
                v4.y += w * v.y;
                v4.z += w * v.z;
                v4.w += w * v.w;
            }
            acc[j] = v4;
        }
        __syncthreads();  // the chunk's buffers are free
    }
    // sum the record groups (R > 1 only when every column has one thread per group), normalise
    if (R > 1) {
        if (grp < R) part_s[tid] = acc[0];
        __syncthreads();
        if (grp == 0) {
            for (int r = 1; r < R; ++r) {
                const float4 v = part_s[col0 + r * C4];
                acc[0].x += v.x;
                acc[0].y += v.y;
                acc[0].z += v.z;
                acc[0].w += v.w;
            }
        }
    }
    const float gvs = __ldg(p.gv);
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
        const int col = col0 + NT * j;
        if (grp != 0 || col >= C4) continue;
        const int g_col = col * 4 / D;
        const float L = hd_s[kMaxGroup + g_col];
        const float f = L > 0.0f ? gvs / L : 0.0f;
        uint2 o;
        o.x = pack_bf16x2(acc[j].x * f, acc[j].y * f);
        o.y = pack_bf16x2(acc[j].z * f, acc[j].w * f);
        *reinterpret_cast<uint2*>(p.out + (static_cast<int64_t>(b) * p.Hq + h * G) * D + 4 * col) = o;
    }
    if (tid < G && p.lse) {
        const float L = hd_s[kMaxGroup + tid];
        p.lse[static_cast<int64_t>(b) * p.Hq + h * G + tid] =
            L > 0.0f ? (hd_s[tid] + log2f(L)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();  // shared memory is reused by the next pair
}

__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ int align16i(int x) { return (x + 15) & ~15; }

// Merge pending pairs pend[first], pend[first + 1], ... (b, h, first record, records) together,
// as many as fit in shared memory at once (whole CTA, after its runs). The records' outputs and
// (max, sum) pairs of all of them are staged by asynchronous copies in one round trip; then every
// thread takes float4 columns of the outputs and forms the weights of its column's query head
// from the staged maxima itself, so no reduction across threads and no second barrier is needed.
// Returns how many pairs were merged (0 when the first pair alone does not fit: the caller merges
// it by chunks).
template <int D>
__device__ __forceinline__ int merge_batch(const DecodeParams& p, const int (*pend)[4], int first,
                                           int n_pend, uint8_t* smem) {
    using G_ = Geo<D>;
    constexpr int NT = G_::THREADS;
    const int tid = threadIdx.x;
    const int G = p.G;
    const int rec_bytes = G * D * 4;
    // per pair: outputs n x rec_bytes, then (max, sum) n x G x 8
    auto bytes_of = [&](int n) { return n * rec_bytes + align16i(n * G * 8); };
    int cnt = 0, used = 0;
    for (int i = first; i < n_pend; ++i) {
        const int need = bytes_of(pend[i][3]);
        if (used + need > G_::SMEM) break;
        used += need;
        ++cnt;
    }
    if (cnt == 0) return 0;
    // no fence here: the threads that saw the counts complete fenced after them, and the CTA
    // barrier since then orders every thread's reads after those fences
    const uint32_t s_base = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    {
        int off = 0;
        for (int i = first; i < first + cnt; ++i) {
            const int n = pend[i][3];
            const int64_t rec0 = pend[i][2];
            const int64_t bh = static_cast<int64_t>(pend[i][0]) * p.H + pend[i][1];
            if (tid == 0) atomicExch(p.done + bh, 0ull);  // a replay with the same tag starts from 0
            const uint8_t* src = reinterpret_cast<const uint8_t*>(p.rec_o + rec0 * G * D);
            const int nc = n * rec_bytes / 16;
            for (int c = tid; c < nc; c += NT) cp_async16_plain(s_base + off + 16 * c, src + 16 * c);
            off += n * rec_bytes;
            const float* msrc = p.rec_ml + rec0 * G * 2;
            for (int c = tid; c < n * G; c += NT) cp_async8(s_base + off + 8 * c, msrc + 2 * c);
            off += align16i(n * G * 8);
        }
        cp_async_commit();
        cp_async_wait<0>();
    }
    __syncthreads();
    const float gvs = __ldg(p.gv);
    const int C4 = G * D / 4;
    int i = first, off = 0, base = 0;  // columns [base, base + C4) belong to pair i, staged at off
    for (int cc = tid; cc < cnt * C4; cc += NT) {
        while (cc >= base + C4) {
            off += bytes_of(pend[i][3]);
            base += C4;
            ++i;
        }
        const int n = pend[i][3], col = cc - base, g = col * 4 / D;
        const float4* o_s = reinterpret_cast<const float4*>(smem + off);
        const float2* ml_s = reinterpret_cast<const float2*>(smem + off + n * rec_bytes);
        float M = -INFINITY;
        for (int k = 0; k < n; ++k) M = fmaxf(M, ml_s[k * G + g].x);
        float L = 0.0f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < n; ++k) {
            const float2 ml = ml_s[k * G + g];
            const float w = (ml.x == -INFINITY) ? 0.0f : exp2f(ml.x - M);
            L += w * ml.y;
            const float4 v = o_s[k * C4 + col];
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
        const float f = L > 0.0f ? gvs / L : 0.0f;
        uint2 o;
        o.x = pack_bf16x2(acc.x * f, acc.y * f);
        o.y = pack_bf16x2(acc.z * f, acc.w * f);
        const int64_t row = static_cast<int64_t>(pend[i][0]) * p.Hq + pend[i][1] * G;
        *reinterpret_cast<uint2*>(p.out + row * D + 4 * col) = o;
        if (p.lse && col * 4 == g * D)  // the head's first column also writes its LSE
            p.lse[row + g] = L > 0.0f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();  // shared memory is reused by the next batch
    return cnt;
}

template <int D>
__global__ void __launch_bounds__(Geo<D>::THREADS, 1) decode_split_kernel(const DecodeParams p) {
    pdl_enter();
    using G_ = Geo<D>;
    constexpr int TOK = G_::TOK;
    constexpr int NW = G_::WARPS;
    constexpr int NT = G_::THREADS;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int scan_warp[NW];
    __shared__ int start_bp[NW][3];  // run start of each warp: sequence, its first stage, length
    __shared__ int span_pair[2];     // first and last pair (b H + h) the CTA's runs touch
    __shared__ int pend_n;           // pairs whose last piece finished in this CTA ...
    __shared__ int pend[2 * NW][4];  // ... (b, h, first record, records): merged at the end

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int r = lane >> 2;  // row group of the MMA fragments
    const int c = lane & 3;   // column pair of the MMA fragments
    const int H = p.H, G = p.G, T = p.T;
    const int max_tokens = p.max_pages * T;

    // ------------------------------------------------ stage prefix over the sequences
    // Thread t owns sequences [t C, t C + C); PS_b = H * sum_{b' < b} stages(b').
    // The first two lengths stay in registers for the walk below (a second load of the same
    // words would cost another round trip at the start).
    const int C = (p.B + NT - 1) / NT;
    const int b_lo = min(p.B, tid * C), b_hi = min(p.B, b_lo + C);
    const int kept0 = (b_lo < b_hi) ? __ldg(p.seq_lens + b_lo) : 0;
    const int kept1 = (b_lo + 1 < b_hi) ? __ldg(p.seq_lens + b_lo + 1) : 0;
    auto len_of = [&](int b) {
        return b == b_lo ? kept0 : (b == b_lo + 1 ? kept1 : __ldg(p.seq_lens + b));
    };
    int local = 0;
    for (int b = b_lo; b < b_hi; ++b) {
        const int L = len_of(b);
        if (blockIdx.x == 0 && (L < 0 || L > max_tokens))
            flag_status(p.status, NVFP4KV_STATUS_BAD_SEQ_LEN);
        local += H * seq_stages(L, max_tokens, TOK);
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) scan_warp[warp] = incl;
    if (tid < 2) span_pair[tid] = 0;
    if (tid == 0) pend_n = 0;
    __syncthreads();
    int excl = incl - local, total = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        if (w < warp) excl += scan_warp[w];
        total += scan_warp[w];
    }
    // warp run gw takes [gw W, gw W + W) of the stage list
    const int num_runs = p.num_runs;
    const int W = max(1, (total + num_runs - 1) / num_runs);
    if (blockIdx.x == 0) {
        // sequences without stages (length 0 or invalid): output 0, LSE -inf
        for (int b = b_lo; b < b_hi; ++b) {
            if (seq_stages(__ldg(p.seq_lens + b), max_tokens, TOK) != 0) continue;
            uint16_t* ob = p.out + static_cast<int64_t>(b) * p.Hq * D;
            for (int i = 0; i < p.Hq * D; ++i) ob[i] = 0;
            if (p.lse)
                for (int i = 0; i < p.Hq; ++i) p.lse[static_cast<int64_t>(b) * p.Hq + i] = -INFINITY;
        }
    }
    // One walk over this thread's sequences finds the sequence holding each of the CTA's run
    // starts and its two span ends (32-bit arithmetic: the host bounds stages + runs below 2^31).
    const int gw0 = blockIdx.x * NW;
    const int n_runs_cta = max(0, min(num_runs - gw0, NW));
    const int span_lo = (n_runs_cta > 0 && gw0 < (total + W - 1) / W) ? gw0 * W : total;
    const int span_hi = min(total, (gw0 + n_runs_cta) * W);
    if (local > 0 && span_lo < span_hi && span_lo < excl + local && span_hi > excl) {
        int acc = excl;
        for (int b = b_lo; b < b_hi && acc < span_hi; ++b) {
            const int L = len_of(b);
            const int S = seq_stages(L, max_tokens, TOK);
            const int n = H * S;
            if (n > 0 && acc + n > span_lo) {
                // runs of this CTA starting in [acc, acc + n): w in [w_a, w_b)
                const int w_a = max(0, (acc - gw0 * W + W - 1) / W);
                const int w_b = min(n_runs_cta, (acc + n - gw0 * W + W - 1) / W);
                for (int w = w_a; w < w_b; ++w) {
                    start_bp[w][0] = b;
                    start_bp[w][1] = acc;
                    start_bp[w][2] = L;
                }
                if (span_lo >= acc && span_lo < acc + n) span_pair[0] = b * H + (span_lo - acc) / S;
                if (span_hi - 1 >= acc && span_hi - 1 < acc + n)
                    span_pair[1] = b * H + (span_hi - 1 - acc) / S;
            }
            acc += n;
        }
    }
    __syncthreads();

    // ------------------------------------------------ queries of the CTA's pairs
    const uint32_t smem_base = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    const uint32_t qcache = smem_base + G_::Q_OFF;
    const int q_first = span_pair[0];
    const int q_cached = (span_lo < span_hi)
                             ? min(span_pair[1] - span_pair[0] + 1, G_::QCACHE / (G * D * 2))
                             : 0;
    {
        const uint8_t* qsrc = reinterpret_cast<const uint8_t*>(p.q + static_cast<int64_t>(q_first) * G * D);
        const int nq = q_cached * G * D * 2 / 16;
        for (int ci = tid; ci < nq; ci += NT) cp_async16_plain(qcache + 16 * ci, qsrc + 16 * ci);
        cp_async_commit();
    }

    const int gw = gw0 + warp;
    const int64_t s_begin64 = static_cast<int64_t>(gw) * W;
    const bool has_run = gw < num_runs && s_begin64 < total;
    const int s_begin = has_run ? static_cast<int>(s_begin64) : 0;
    const int n_st = has_run ? min(total - s_begin, W) : 0;

    // ------------------------------------------------ per-lane constants
    const uint32_t ring = smem_base + warp * G_::RING;
    // V chunk j = lane + 32 i of a stage lands XOR-swizzled by its pair row
    uint32_t v_dst[G_::DCH];
#pragma unroll
    for (int i = 0; i < G_::DCH; ++i) {
        const int j = lane + 32 * i;
        const int pr = j / G_::VCH, cj = j - pr * G_::VCH;
        v_dst[i] = G_::V_OFF + pr * D + 16 * (cj ^ (pr & G_::SWZ));
    }
    const int rho = (r >> 1) | ((r & 1) << 2);  // V rows of this lane: chunk rho of a pair row

    // ------------------------------------------------ issue side: the walk over the run
    int ib = has_run ? start_bp[warp][0] : 0;
    int ilen = has_run ? start_bp[warp][2] : 0;
    int iS = has_run ? seq_stages(ilen, max_tokens, TOK) : 1;
    int ih = has_run ? (s_begin - start_bp[warp][1]) / iS : 0;
    int ij = has_run ? (s_begin - start_bp[warp][1]) - ih * iS : 0;
    int ips = has_run ? start_bp[warp][1] + ih * iS : 0;  // flat index of stage 0 of (ib, ih)
    bool ifirst = true;                     // the next stage to issue starts a piece
    int issued = 0;
    int nlen = (has_run && ib + 1 < p.B) ? __ldg(p.seq_lens + ib + 1) : 0;  // next sequence
    // page-id windows: lane l holds the id of page base + l of a sequence's page-table row; the
    // window after the current one (in issue order) is loaded when the current one is taken
    int wrow = -1, wbase = 0, win = 0;
    int prow = -1, pbase = 0, pwin = 0;
    auto load_window = [&](int b_, int base) -> int {
        const int i = base + lane;
        return (i < p.max_pages) ? __ldg(p.page_table + static_cast<int64_t>(b_) * p.max_pages + i)
                                 : -1;
    };
    // make the window holding page pidx of sequence ib current (its loads are only issued) and
    // start loading the one after it
    auto set_window = [&](int pidx) {
        const int nbase = pidx & ~31;
        win = (ib == prow && nbase == pbase) ? pwin : load_window(ib, nbase);
        wrow = ib;
        wbase = nbase;
        const int npg = (ilen + T - 1) / T;
        if (nbase + 32 < npg) {
            prow = ib;
            pbase = nbase + 32;
        } else {
            prow = (ih + 1 < H) ? ib : ib + 1;  // a zero-length next sequence makes this a miss
            pbase = 0;
        }
        if (prow < p.B && !(prow == wrow && pbase == wbase))
            pwin = load_window(prow, pbase);
        else
            prow = -1;
    };
    auto page_of = [&](int pidx) -> int {  // warp-uniform pidx of sequence ib; every lane calls
        if (ib != wrow || pidx < wbase || pidx >= wbase + 32) set_window(pidx);
        const int pg = __shfl_sync(0xFFFFFFFFu, win, pidx - wbase);
        return (pg >= 0 && pg < p.pool_pages) ? pg : -1;
    };

    const int64_t page_rows = static_cast<int64_t>(H) * T;
    const bool page_aligned = (T % TOK) == 0;
    // issue the next stage of the walk into `slot`, then advance the walk
    auto issue_next = [&](uint32_t slot) {
        const uint64_t kv_pol = l2_policy_evict_first();
        const int t0 = ij * TOK;
        const int nval = min(TOK, ilen - t0);
        const int64_t head_rows = static_cast<int64_t>(ih) * T;
        int64_t row0[G_::SUB];  // token row of each sub-tile in its pool, -1: not real
        if (page_aligned) {
            const int pidx = static_cast<int>(__umul64hi(static_cast<uint64_t>(t0), p.t_magic));
            const int pg = page_of(pidx);
            const int64_t r0 = pg * page_rows + head_rows + (t0 - pidx * T);
#pragma unroll
            for (int u = 0; u < G_::SUB; ++u)
                row0[u] = (pg >= 0 && 16 * u < nval) ? r0 + 16 * u : -1;
        } else {
#pragma unroll
            for (int u = 0; u < G_::SUB; ++u) {
                const int t = t0 + 16 * u;
                const int pidx = static_cast<int>(__umul64hi(static_cast<uint64_t>(t), p.t_magic));
                const int pg = page_of(min(pidx, max(0, (ilen - 1) / T)));
                row0[u] = (pg >= 0 && 16 * u < nval) ? pg * page_rows + head_rows + (t - pidx * T)
                                                      : -1;
            }
        }
        uint32_t okbits = 0;
#pragma unroll
        for (int u = 0; u < G_::SUB; ++u) okbits |= (row0[u] >= 0 ? 1u : 0u) << u;
        const uint32_t want = (1u << ((nval + 15) / 16)) - 1u;
        if (okbits != want && lane == 0) flag_status(p.status, NVFP4KV_STATUS_PAGE_OOB);
        if (page_aligned && okbits == (1u << G_::SUB) - 1) {
            // the whole stage is one run of each pool: offsets are compile-time constants
            const int64_t doff = row0[0] * (D / 2) + 16 * lane;
            const uint8_t* ksrc = p.kd + doff;
            const uint8_t* vsrc = p.vd + doff;
            static_for<G_::DCH>([&](auto I) {
                constexpr int i = decltype(I)::value;
                cp_async16<G_::K_OFF + 512 * i, 512 * i>(slot + 16 * lane, ksrc, kv_pol);
                cp_async16<0, 512 * i>(slot + v_dst[i], vsrc, kv_pol);
            });
            const int64_t soff = row0[0] * G_::NB;
#pragma unroll
            for (int k = 0; k < G_::SC_PER_LANE; ++k) {
                const int jc = lane + 32 * k;
                const bool kpool = jc < G_::SCH;
                const int jj = kpool ? jc : jc - G_::SCH;
                cp_async16<0, 0>(slot + (kpool ? G_::KS_OFF : G_::VS_OFF) + 16 * jj,
                                 (kpool ? p.ks : p.vs) + soff + 16 * jj, kv_pol);
            }
        } else {
#pragma unroll
            for (int i = 0; i < G_::DCH; ++i) {
                const int u = i / G_::SUB_DIV;
                const int jj = lane + 32 * i - u * (D / 2);  // chunk within the sub-tile
                const bool ok = row0[u] >= 0;
                const int64_t off = ok ? row0[u] * (D / 2) + 16 * jj : 0;
                cp_async16_zfill(slot + G_::K_OFF + 16 * (lane + 32 * i), p.kd + off,
                                 ok ? 16u : 0u, kv_pol);
                cp_async16_zfill(slot + v_dst[i], p.vd + off, ok ? 16u : 0u, kv_pol);
            }
#pragma unroll
            for (int k = 0; k < G_::SC_PER_LANE; ++k) {
                const int jc = lane + 32 * k;
                const bool kpool = jc < G_::SCH;
                const int jj = kpool ? jc : jc - G_::SCH;
                const int u = jj / (D / 16);
                int64_t ru = row0[0];  // row0[u] without a dynamically indexed array
#pragma unroll
                for (int uu = 1; uu < G_::SUB; ++uu)
                    if (u == uu) ru = row0[uu];
                const bool ok = ru >= 0;
                const int64_t off = ok ? ru * G_::NB + 16 * (jj - u * (D / 16)) : 0;
                cp_async16_zfill(slot + (kpool ? G_::KS_OFF : G_::VS_OFF) + 16 * jj,
                                 (kpool ? p.ks : p.vs) + off, ok ? 16u : 0u, kv_pol);
            }
        }
        const bool last = (ij == iS - 1) || (issued == n_st - 1);
        const uint32_t flags = (ifirst ? kFirst : 0u) | (last ? kLast : 0u);
        if (lane == 0) {
            sts_v4(slot + G_::HDR_OFF, okbits | (static_cast<uint32_t>(nval) << 8), flags,
                   static_cast<uint32_t>(ib), static_cast<uint32_t>(ih));
            sts_v4(slot + G_::HDR_OFF + 16, static_cast<uint32_t>(ips), static_cast<uint32_t>(iS),
                   0u, 0u);
        }
        // advance the walk
        ++issued;
        ifirst = false;
        if (last) {
            ij = 0;
            ips += iS;
            ifirst = true;
            if (issued < n_st && ++ih == H) {
                ih = 0;
                ++ib;
                ilen = nlen;
                iS = seq_stages(ilen, max_tokens, TOK);
                while (iS == 0) {  // sequences without stages are not in the list
                    ++ib;
                    ilen = __ldg(p.seq_lens + ib);
                    iS = seq_stages(ilen, max_tokens, TOK);
                }
                nlen = (ib + 1 < p.B) ? __ldg(p.seq_lens + ib + 1) : 0;
            }
        } else {
            ++ij;
        }
    };

    // ------------------------------------------------ start: stage 0, then the query cache
    // The first page-id window is loaded while the query cache fills; the first copies go out
    // as soon as the page ids are in, and the queries are waited for behind them.
    if (n_st > 0) issue_next(ring);
    cp_async_commit();
    cp_async_wait<1>();  // this thread's query chunks have landed ...
    __syncthreads();     // ... and every thread's: from here on warps run alone until the merge

    // ------------------------------------------------ compute side
    uint32_t qf[G_::KSTEPS][2];
    float cs0 = 0.0f, cs1 = 0.0f;
    float o[G_::KSTEPS][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    const float gvs = __ldg(p.gv);

#pragma unroll 1
    for (int i = 0; i < n_st; ++i) {
        // the next stage goes into the slot computed at iteration i - 1
        if (i + 1 < n_st) issue_next(ring + ((i + 1) % G_::SLOTS) * G_::SLOT);
        cp_async_commit();
        cp_async_wait<1>();  // this lane's copies of stage i are done ...
        __syncwarp();        // ... and so are the other lanes'
        const uint32_t st = ring + (i % G_::SLOTS) * G_::SLOT;
        uint32_t hdr[4];
        lds_words(hdr, st + G_::HDR_OFF);
        const uint32_t okbits = hdr[0] & 0xFFu;
        const int nval = static_cast<int>(hdr[0] >> 8);
        const uint32_t flags = hdr[1];
        if (flags & kFirst) {
            // ---- Q fragments of the piece: lane (r, c) holds head r of the group; k-step kk
            // covers head dims c*D/4 + 4kk + {0..3} (the same permutation is used for K), as
            // FP16 q * 2^kq. From the query cache, or from global memory for a pair beyond it.
            const int qpair = static_cast<int>(hdr[2]) * H + static_cast<int>(hdr[3]);
            float qv[D / 4];
            float qmax = 0.0f;
            if (r < G) {
                uint32_t qw[D / 8];
                const int qi = qpair - q_first;
                if (qi >= 0 && qi < q_cached) {
                    lds_words(qw, qcache + ((qi * G + r) * D + c * (D / 4)) * 2);
                } else {
                    const uint4* qsrc = reinterpret_cast<const uint4*>(
                        p.q + (static_cast<int64_t>(qpair) * G + r) * D + c * (D / 4));
#pragma unroll
                    for (int k = 0; k < D / 32; ++k) {
                        const uint4 v = __ldg(qsrc + k);
                        qw[4 * k] = v.x;
                        qw[4 * k + 1] = v.y;
                        qw[4 * k + 2] = v.z;
                        qw[4 * k + 3] = v.w;
                    }
                }
#pragma unroll
                for (int k = 0; k < D / 8; ++k) {
                    qv[2 * k] = bf16_lo(qw[k]);
                    qv[2 * k + 1] = bf16_hi(qw[k]);
                }
#pragma unroll
                for (int k = 0; k < D / 4; ++k) qmax = fmaxf(qmax, fabsf(qv[k]));
            } else {
#pragma unroll
                for (int k = 0; k < D / 4; ++k) qv[k] = 0.0f;
            }
            qmax = fmaxf(qmax, __shfl_xor_sync(0xFFFFFFFFu, qmax, 1));
            qmax = fmaxf(qmax, __shfl_xor_sync(0xFFFFFFFFu, qmax, 2));
            // qmax * 2^kq in [2^14, 2^15): every BF16 value of the head is exact in FP16 down
            // to 2^-18 of the head maximum.
            int kq = (qmax > 0.0f) ? (14 - ilogbf(qmax)) : 0;
            kq = max(-120, min(kq, 120));
            const float up = ldexpf(1.0f, kq);
#pragma unroll
            for (int kk = 0; kk < G_::KSTEPS; ++kk) {
                qf[kk][0] = pack_f16x2(qv[4 * kk] * up, qv[4 * kk + 1] * up);
                qf[kk][1] = pack_f16x2(qv[4 * kk + 2] * up, qv[4 * kk + 3] * up);
            }
            const float cs_row = (r < G) ? p.sm_scale * __ldg(p.gk) * kLog2e * ldexpf(1.0f, -kq)
                                         : 0.0f;
            // score scale of this lane's two S^T columns (query heads 2c, 2c+1)
            cs0 = __shfl_sync(0xFFFFFFFFu, cs_row, 8 * c);
            cs1 = __shfl_sync(0xFFFFFFFFu, cs_row, 8 * c + 4);
#pragma unroll
            for (int m = 0; m < G_::KSTEPS; ++m)
#pragma unroll
                for (int k = 0; k < 4; ++k) o[m][k] = 0.0f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.0f;
        }

        if (okbits != 0u) {
            const bool full = (okbits == (1u << G_::SUB) - 1) && nval >= TOK;
            // valid-token bits of each sub-tile (only read when !full)
            uint32_t tmask[G_::SUB];
#pragma unroll
            for (int u = 0; u < G_::SUB; ++u) {
                const int nv = min(16, max(0, nval - 16 * u));
                tmask[u] = ((okbits >> u) & 1u) ? ((nv >= 16) ? 0xFFFFu : ((1u << nv) - 1u)) : 0u;
            }

            // ---- S^T = K^ Q^T for the SUB sub-tiles
            float x[G_::SUB][4];
#pragma unroll
            for (int u = 0; u < G_::SUB; ++u) {
                const int row0 = 16 * u + r;
                const int row1 = row0 + 8;
                uint32_t kw0[G_::CW], kw1[G_::CW];
                lds_words(kw0, st + G_::K_OFF + row0 * (D / 2) + c * G_::CHUNK);
                lds_words(kw1, st + G_::K_OFF + row1 * (D / 2) + c * G_::CHUNK);
                // FP16 (s, s) of the lane's D/64 blocks in rows row0 / row1: the scale byte
                // is duplicated by an integer multiply, then converted as an E4M3 pair
                uint32_t ks0[D / 64], ks1[D / 64];
#pragma unroll
                for (int q = 0; q < D / 64; ++q) {
                    ks0[q] = e4m3x2_to_f16x2(
                        lds_u8(st + G_::KS_OFF + row0 * G_::NB + c * (D / 64) + q) * 0x0101u);
                    ks1[q] = e4m3x2_to_f16x2(
                        lds_u8(st + G_::KS_OFF + row1 * G_::NB + c * (D / 64) + q) * 0x0101u);
                }
                float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int q = 0; q < G_::CW; ++q) {
                    uint32_t c0[4], c1[4];
                    e2m1x8_to_f16x2x4(kw0[q], c0);
                    e2m1x8_to_f16x2x4(kw1[q], c1);
#pragma unroll
                    for (int hk = 0; hk < 2; ++hk) {
                        const int kk = 2 * q + hk;  // k-step: bytes 2kk, 2kk+1 of the chunk
                        const int blk = kk / 4;     // block of the lane's chunk
                        uint32_t a[4];
                        a[0] = h2_mul(c0[2 * hk], ks0[blk]);
                        a[1] = h2_mul(c1[2 * hk], ks1[blk]);
                        a[2] = h2_mul(c0[2 * hk + 1], ks0[blk]);
                        a[3] = h2_mul(c1[2 * hk + 1], ks1[blk]);
                        mma_f16_16816(acc, a, qf[kk][0], qf[kk][1]);
                    }
                }
                x[u][0] = acc[0] * cs0;
                x[u][1] = acc[1] * cs1;
                x[u][2] = acc[2] * cs0;
                x[u][3] = acc[3] * cs1;
            }

            // ---- online softmax over the stage, columns = query heads 2c, 2c+1
            if (!full) {
#pragma unroll
                for (int u = 0; u < G_::SUB; ++u) {
                    if (!((tmask[u] >> r) & 1u)) x[u][0] = x[u][1] = -INFINITY;
                    if (!((tmask[u] >> (r + 8)) & 1u)) x[u][2] = x[u][3] = -INFINITY;
                }
            }
            float lm0 = fmaxf(x[0][0], x[0][2]), lm1 = fmaxf(x[0][1], x[0][3]);
#pragma unroll
            for (int u = 1; u < G_::SUB; ++u) {
                lm0 = fmaxf(lm0, fmaxf(x[u][0], x[u][2]));
                lm1 = fmaxf(lm1, fmaxf(x[u][1], x[u][3]));
            }
            // column maxima over the stage, both columns in one FP16 pair (the running
            // maximum only has to be close to the true one: p = 2^(x - m) stays below 2^8)
            __half2 hm = __floats2half2_rn(lm0, lm1);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                const uint32_t uu =
                    __shfl_xor_sync(0xFFFFFFFFu, *reinterpret_cast<const uint32_t*>(&hm), off);
                hm = __hmax2(hm, *reinterpret_cast<const __half2*>(&uu));
            }
            float mx0 = __low2float(hm), mx1 = __high2float(hm);
            if (__any_sync(0xFFFFFFFFu, fmaxf(mx0, mx1) > 65000.0f)) {
                // scores beyond the FP16 range: reduce in fp32 instead
                mx0 = lm0;
                mx1 = lm1;
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, off));
                }
            }
            const bool grow = (mx0 > m0 + kRescaleThreshold) || (mx1 > m1 + kRescaleThreshold);
            if (__any_sync(0xFFFFFFFFu, grow)) {
                const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
                const float a0 = ex2_approx(m0 - n0), a1 = ex2_approx(m1 - n1);
                m0 = n0;
                m1 = n1;
                l0 *= a0;
                l1 *= a1;
#pragma unroll
                for (int m = 0; m < G_::KSTEPS; ++m) {
                    o[m][0] *= a0;
                    o[m][1] *= a1;
                    o[m][2] *= a0;
                    o[m][3] *= a1;
                }
            }
            uint32_t pb[G_::SUB][2];
#pragma unroll
            for (int u = 0; u < G_::SUB; ++u) {
                const float p0 = ex2_approx(x[u][0] - m0), p1 = ex2_approx(x[u][1] - m1);
                const float p2 = ex2_approx(x[u][2] - m0), p3 = ex2_approx(x[u][3] - m1);
                l0 += p0 + p2;
                l1 += p1 + p3;
                // P^T (tokens x heads) -> B operand (k = tokens, n = heads)
                pb[u][0] = movmatrix_trans(pack_f16x2(p0, p1));
                pb[u][1] = movmatrix_trans(pack_f16x2(p2, p3));
            }

            // ---- O^T += V^^T P^T. Lane pairs: pr0 (tokens 2c, 2c+1), pr1 (tokens 2c+8, 2c+9)
#pragma unroll
            for (int u = 0; u < G_::SUB; ++u) {
                const int pr0 = 8 * u + c, pr1 = pr0 + 4;
                // the lane's chunk covers head dims rho*D/8 .. +D/8-1: blocks (rho*D/8)/16 ...
                constexpr int kBlkPerChunk = (D / 8 + 15) / 16;
                uint32_t vsc0[kBlkPerChunk], vsc1[kBlkPerChunk];
#pragma unroll
                for (int q = 0; q < kBlkPerChunk; ++q) {
                    const int blk = (rho * (D / 8)) / 16 + q;
                    vsc0[q] = e4m3x2_to_f16x2(lds_u16(st + G_::VS_OFF + pr0 * 2 * G_::NB + 2 * blk));
                    vsc1[q] = e4m3x2_to_f16x2(lds_u16(st + G_::VS_OFF + pr1 * 2 * G_::NB + 2 * blk));
                }
                if (!full && tmask[u] != 0xFFFFu) {
                    // tokens past the sequence end in a real page: their V scales may be
                    // anything, so they are zeroed (P is 0 there already)
                    const uint32_t tm = tmask[u];
                    const uint32_t keep0 = (((tm >> (2 * c)) & 1u) ? 0x0000FFFFu : 0u) |
                                           (((tm >> (2 * c + 1)) & 1u) ? 0xFFFF0000u : 0u);
                    const uint32_t keep1 = (((tm >> (2 * c + 8)) & 1u) ? 0x0000FFFFu : 0u) |
                                           (((tm >> (2 * c + 9)) & 1u) ? 0xFFFF0000u : 0u);
#pragma unroll
                    for (int q = 0; q < kBlkPerChunk; ++q) {
                        vsc0[q] &= keep0;
                        vsc1[q] &= keep1;
                    }
                }
                uint32_t vw0[G_::CW], vw1[G_::CW];
#pragma unroll
                for (int q = 0; q < G_::CW; q += (G_::CW >= 4 ? 4 : G_::CW)) {
                    const int xb = rho * G_::CHUNK + 4 * q;  // logical byte of the chunk piece
                    uint32_t t0w[G_::CW >= 4 ? 4 : G_::CW], t1w[G_::CW >= 4 ? 4 : G_::CW];
                    lds_words(t0w, st + G_::V_OFF + v_swz<D>(pr0, xb));
                    lds_words(t1w, st + G_::V_OFF + v_swz<D>(pr1, xb));
#pragma unroll
                    for (int e = 0; e < (G_::CW >= 4 ? 4 : G_::CW); ++e) {
                        vw0[q + e] = t0w[e];
                        vw1[q + e] = t1w[e];
                    }
                }
#pragma unroll
                for (int q = 0; q < G_::CW; ++q) {
                    uint32_t c0[4], c1[4];
                    e2m1x8_to_f16x2x4(vw0[q], c0);
                    e2m1x8_to_f16x2x4(vw1[q], c1);
#pragma unroll
                    for (int hm2 = 0; hm2 < 2; ++hm2) {
                        const int m = 2 * q + hm2;   // M-tile: bytes 2m, 2m+1 of the chunk
                        const int sq = (2 * m) / 16; // block of that byte within the chunk
                        uint32_t a[4];
                        a[0] = h2_mul(c0[2 * hm2], vsc0[sq]);
                        a[1] = h2_mul(c0[2 * hm2 + 1], vsc0[sq]);
                        a[2] = h2_mul(c1[2 * hm2], vsc1[sq]);
                        a[3] = h2_mul(c1[2 * hm2 + 1], vsc1[sq]);
                        mma_f16_16816(o[m], a, pb[u][0], pb[u][1]);
                    }
                }
            }
        }

        if (flags & kLast) {
            // ---- end of a piece: the whole pair (outputs) or a record
            uint32_t h2[4];
            lds_words(h2, st + G_::HDR_OFF + 16);
            const int pb_ = static_cast<int>(hdr[2]), ph = static_cast<int>(hdr[3]);
            const int pps = static_cast<int>(h2[0]), pS = static_cast<int>(h2[1]);
            float ls0 = l0, ls1 = l1;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                ls0 += __shfl_xor_sync(0xFFFFFFFFu, ls0, off);
                ls1 += __shfl_xor_sync(0xFFFFFFFFu, ls1, off);
            }
            const int g0 = 2 * c, g1 = 2 * c + 1;
            const int gf = pps / W, gl = (pps + pS - 1) / W;
            const int64_t bh = static_cast<int64_t>(pb_) * H + ph;
            if (gf == gl) {
                // the whole pair is this piece: normalise and write the output directly
                uint16_t* ob = p.out + (static_cast<int64_t>(pb_) * p.Hq + ph * G) * D;
                const float f0 = ls0 > 0.0f ? gvs / ls0 : 0.0f;
                const float f1 = ls1 > 0.0f ? gvs / ls1 : 0.0f;
#pragma unroll
                for (int m = 0; m < G_::KSTEPS; ++m) {
                    const int d0 = rho * (D / 8) + 2 * m;
                    if (g0 < G)
                        *reinterpret_cast<uint32_t*>(ob + g0 * D + d0) =
                            pack_bf16x2(o[m][0] * f0, o[m][2] * f0);
                    if (g1 < G)
                        *reinterpret_cast<uint32_t*>(ob + g1 * D + d0) =
                            pack_bf16x2(o[m][1] * f1, o[m][3] * f1);
                }
                if (r == 0 && p.lse) {
                    float* lb = p.lse + static_cast<int64_t>(pb_) * p.Hq + ph * G;
                    if (g0 < G) lb[g0] = ls0 > 0.0f ? (m0 + log2f(ls0)) * 0.6931471805599453f : -INFINITY;
                    if (g1 < G) lb[g1] = ls1 > 0.0f ? (m1 + log2f(ls1)) * 0.6931471805599453f : -INFINITY;
                }
            } else {
                const int64_t rec = gw + bh;
                float* ro = p.rec_o + rec * G * D;
#pragma unroll
                for (int m = 0; m < G_::KSTEPS; ++m) {
                    const int d0 = rho * (D / 8) + 2 * m;
                    if (g0 < G) *reinterpret_cast<float2*>(ro + g0 * D + d0) = make_float2(o[m][0], o[m][2]);
                    if (g1 < G) *reinterpret_cast<float2*>(ro + g1 * D + d0) = make_float2(o[m][1], o[m][3]);
                }
                if (r == 0) {
                    if (g0 < G) *reinterpret_cast<float2*>(p.rec_ml + (rec * G + g0) * 2) = make_float2(m0, ls0);
                    if (g1 < G) *reinterpret_cast<float2*>(p.rec_ml + (rec * G + g1) * 2) = make_float2(m1, ls1);
                }
                __syncwarp();
                if (lane == 0) {
                    fence_acq_rel_gpu();  // release: the record is visible before the count says so
                    unsigned long long* cnt = p.done + bh;
                    const uint32_t k = tagged_finish(cnt, atomicAdd(cnt, 1ull), p.nonce, 1);
                    if (k == kTagGiveUp) flag_status(p.status, NVFP4KV_STATUS_TIMEOUT);
                    if (k == static_cast<uint32_t>(gl - gf)) {  // every piece is in: merge here
                        // acquire: the other pieces' records are read after their counts (the
                        // CTA barrier before the merge carries this to every thread)
                        fence_acq_rel_gpu();
                        const int slot = atomicAdd(&pend_n, 1);
                        pend[slot][0] = pb_;
                        pend[slot][1] = ph;
                        pend[slot][2] = static_cast<int>(gf + bh);
                        pend[slot][3] = gl - gf + 1;
                    }
                }
            }
        }
        __syncwarp();  // every lane is done reading the slot before it refills
    }
    cp_async_wait<0>();
    __syncthreads();  // every warp's run is done: the rings are free for the merge
    const int n_pend = pend_n;
    for (int k = 0; k < n_pend;) {
        const int m = merge_batch<D>(p, pend, k, n_pend, smem);
        if (m == 0) {  // a pair whose records do not fit at once: by chunks
            merge_pair<D>(p, pend[k][0], pend[k][1], pend[k][2], pend[k][3], smem);
            ++k;
        }
        k += m;
    }
}

// ------------------------------------------------------------------------------------------
// Host side: grid, workspace carving
// ------------------------------------------------------------------------------------------
size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int stage_tokens(int D) { return D == 256 ? 32 : 64; }
int warps_per_cta(int D) { return D == 64 ? 16 : (D == 128 ? 12 : 8); }

// Warp runs of the split kernel: one per warp of one CTA per SM (automatic), or n runs per
// (sequence, KV head) pair.
int64_t decode_runs(int batch, int H, int D, int max_num_splits) {
    if (max_num_splits > 0) return static_cast<int64_t>(max_num_splits) * batch * H;
    return static_cast<int64_t>(num_sms()) * warps_per_cta(D);
}

struct WsLayout {
    size_t done, ml, o, total;
};

// Records: one per (warp run, pair) piece; bounded by runs + pairs because runs are consecutive.
WsLayout ws_layout(int batch, int H, int Hq, int D, int64_t runs) {
    const size_t pairs = static_cast<size_t>(batch) * H;
    const size_t records = static_cast<size_t>(runs) + pairs;
    const size_t G = static_cast<size_t>(Hq / H);
    WsLayout w;
    w.done = 0;
    w.ml = align256(pairs * sizeof(unsigned long long));
    w.o = w.ml + align256(records * G * 2 * sizeof(float));
    w.total = w.o + align256(records * G * D * sizeof(float));
    return w;
}

bool decode_shape_ok(const nvfp4kv_layout* l, int Hq) {
    if (!layout_ok(l)) return false;
    const int D = l->head_dim;
    if (D != 64 && D != 128 && D != 256) return false;
    if (l->page_size % 16 != 0) return false;
    if (Hq <= 0 || Hq % l->num_kv_heads != 0) return false;
    const int G = Hq / l->num_kv_heads;
    return G >= 1 && G <= kMaxGroup;
}

// The flat stage list, the token positions and the records index with 32-bit integers.
bool decode_size_ok(int batch, int H, int D, int max_pages, int T, int64_t runs) {
    const int64_t max_tokens = static_cast<int64_t>(max_pages) * T;
    const int64_t tok = stage_tokens(D);
    const int64_t stages = (max_tokens + tok - 1) / tok * batch * H;
    const int64_t lim = (int64_t{1} << 31) - 1;
    return max_tokens < lim - tok && stages + runs < lim &&
           runs + static_cast<int64_t>(batch) * H < lim;
}

template <int D>
cudaError_t launch_decode(const DecodeParams& p, int64_t runs, cudaStream_t s) {
    using G_ = Geo<D>;
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, G_::SMEM);
    if (e != cudaSuccess) return e;
    const int64_t ctas = (runs + G_::WARPS - 1) / G_::WARPS;
    e = launch_pdl(decode_split_kernel<D>, static_cast<unsigned>(ctas), G_::THREADS,
                   static_cast<size_t>(G_::SMEM), s, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace
}  // namespace nvfp4kv

using namespace nvfp4kv;

extern "C" size_t nvfp4_paged_decode_workspace_size(const nvfp4kv_layout* layout, int32_t batch,
                                                    int32_t num_q_heads,
                                                    int32_t max_pages_per_seq,
                                                    int32_t max_num_splits) {
    if (!layout_ok(layout) || batch < 0 || num_q_heads <= 0 || max_pages_per_seq <= 0 ||
        max_num_splits < 0 || max_num_splits > kMaxSplits)
        return 0;
    if (num_q_heads % layout->num_kv_heads != 0) return 0;
    const int H = layout->num_kv_heads;
    const int64_t runs = decode_runs(batch, H, layout->head_dim, max_num_splits);
    return ws_layout(batch, H, num_q_heads, layout->head_dim, runs).total;
}

extern "C" nvfp4kv_status nvfp4_paged_decode_attention(
    const nvfp4kv_layout* layout, int32_t batch, int32_t num_q_heads, const void* q,
    const uint8_t* k_data, const uint8_t* k_scales, const float* k_global_scale,
    const uint8_t* v_data, const uint8_t* v_scales, const float* v_global_scale,
    int32_t pool_pages, const int32_t* page_table, int32_t max_pages_per_seq,
    const int32_t* seq_lens, float sm_scale, int32_t max_num_splits, void* workspace,
    size_t workspace_bytes, void* out, float* lse, int32_t* status, nvfp4kv_stream_t stream) {
    if (!layout_ok(layout) || batch < 0 || num_q_heads <= 0 || max_pages_per_seq <= 0 ||
        pool_pages <= 0 || max_num_splits < 0 || max_num_splits > kMaxSplits)
        return NVFP4KV_ERR_INVALID_ARG;
    if (!decode_shape_ok(layout, num_q_heads)) return NVFP4KV_ERR_UNSUPPORTED;
    if (batch == 0) return NVFP4KV_OK;
    if (!q || !k_data || !k_scales || !k_global_scale || !v_data || !v_scales ||
        !v_global_scale || !page_table || !seq_lens || !out)
        return NVFP4KV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_data) || !aligned16(k_scales) || !aligned16(v_data) ||
        !aligned16(v_scales) || !aligned16(out))
        return NVFP4KV_ERR_INVALID_ARG;
    if (batch > 65535 || num_q_heads > 65535) return NVFP4KV_ERR_UNSUPPORTED;
    const int D = layout->head_dim;
    const int H = layout->num_kv_heads;
    const int T = layout->page_size;
    const int64_t runs = decode_runs(batch, H, D, max_num_splits);
    if (!decode_size_ok(batch, H, D, max_pages_per_seq, T, runs)) return NVFP4KV_ERR_UNSUPPORTED;
    const WsLayout wl = ws_layout(batch, H, num_q_heads, D, runs);
    if (!workspace || workspace_bytes < wl.total || !aligned16(workspace))
        return NVFP4KV_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);

    DecodeParams p{};
    p.q = static_cast<const uint16_t*>(q);
    p.kd = k_data;
    p.ks = k_scales;
    p.vd = v_data;
    p.vs = v_scales;
    p.gk = k_global_scale;
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.gv = v_global_scale;
    p.out = static_cast<uint16_t*>(out);
    p.lse = lse;
    p.done = reinterpret_cast<unsigned long long*>(ws + wl.done);
    p.nonce = next_nonce();
    p.rec_ml = reinterpret_cast<float*>(ws + wl.ml);
    p.rec_o = reinterpret_cast<float*>(ws + wl.o);
    p.status = status;
    p.t_magic = UINT64_MAX / static_cast<uint64_t>(T) + 1;
    p.B = batch;
    p.Hq = num_q_heads;
    p.H = H;
    p.G = num_q_heads / H;
    p.T = T;
    p.pool_pages = pool_pages;
    p.max_pages = max_pages_per_seq;
    p.num_runs = static_cast<int32_t>(runs);
    p.sm_scale = sm_scale;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (D) {
    case 64: e = launch_decode<64>(p, runs, s); break;
    case 128: e = launch_decode<128>(p, runs, s); break;
    default: e = launch_decode<256>(p, runs, s); break;
    }
    if (e != cudaSuccess) return NVFP4KV_ERR_CUDA;

    return NVFP4KV_OK;
}
