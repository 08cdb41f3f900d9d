// Split-KV paged GQA decode attention over NVFP4 K/V for sm_103a, its merge in the same launch.
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
//    One persistent wave of CTAs cuts the list into equal runs, so every SM streams about the
//    same number of bytes whatever the mix of sequence lengths. A run may cross pairs; each
//    (CTA, pair) piece leaves one partial record c + bh, so records never collide and their
//    number is bounded by (CTAs + pairs) before any length is known. The last CTA to finish a
//    pair (counted with a per-pair counter that carries a per-call tag, so the workspace never
//    needs clearing) merges the pair's records and writes the outputs: no second kernel.
//  * A CTA has 4 warps; warp w takes stages w, w+4, ... of the piece. A stage is SUB MMA tiles
//    of 16 tokens, streamed through a per-warp 2-slot shared-memory ring by asynchronous copies
//    (cp.async, 16 bytes per lane, completion per warp by wait_group): the packed K rows,
//    token-pair packed V rows and both scale pools of a stage are four contiguous runs of its
//    page. Sub-tiles whose page id is out of range or that lie past the sequence end are
//    zero-filled, and a small slot header tells the consumer which sub-tiles are real.
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
//  * at the end of a piece the 4 warps merge (max, sum, output) in shared memory; a piece that
//    is a whole pair writes the BF16 output and the natural-log LSE directly, otherwise the CTA
//    writes its record and the pair's last CTA merges the records by log-sum-exp.
//  * a piece boundary inside a run holds up the CTA as little as possible: the next piece's
//    page ids are loaded into registers while the current piece streams, and the record's count
//    is bumped by one lane while the CTA already streams the next piece; the outcome is read at
//    that piece's end, where the CTA merges the pair if its count completed it.
// Bytes per (token, KV head) at head_dim 128: 64 + 8 (K) + 64 + 8 (V) = 144.
#include <atomic>
#include <chrono>
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_util.h"

namespace nvfp4kv {
namespace {

constexpr int kWarps = 4;
constexpr int kDecThreads = kWarps * 32;
constexpr int kSlots = 2;          // stages per warp ring
constexpr int kMaxGroup = 8;
constexpr int kMaxSplits = 64;     // bound of the caller-forced split count
constexpr int kPageBuf = 256;      // page ids of a piece kept in shared memory
constexpr int kMaxRecW = 64;      // merge: weights of up to this many records kept in shared memory
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

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
    static constexpr int HDR_OFF = VS_OFF + SS;  // slot header: real sub-tiles, tokens
    static constexpr int SLOT = HDR_OFF + 16;
    static constexpr int RING = kSlots * SLOT;  // per warp
    static constexpr int SMEM = kWarps * RING;
    static constexpr int KSTEPS = D / 16;       // k-steps of S^T = K Q^T
    static constexpr int CHUNK = D / 8;         // bytes of a row one quad lane owns
    static constexpr int CW = CHUNK / 4;        // ... as 32-bit words
    static constexpr int VCH = D / 16;          // 16-byte chunks per V pair row
    static constexpr int SWZ = (VCH < 8 ? VCH : 8) - 1;  // chunk XOR mask
    static constexpr int DCH = SK / (16 * 32);  // 16-byte chunks per lane of one data pool
    static constexpr int SUB_DIV = D / 64;      // data chunk i of a lane lies in sub-tile i / SUB_DIV
    static constexpr int SCH = SS / 16;         // 16-byte chunks of one scale pool
    static constexpr int SC_PER_LANE = 2 * SCH / 32;
    // CTAs per SM: head_dim 64 at 4 (the register budget of 5 held it at 96 registers, and 4 at
    // 121 registers decodes a 32 x 8192 batch 18 % faster), 256 at 2 (232 registers, no spills;
    // 2-3 % faster than 3 with spills), 128 at 3
    static constexpr int BLOCKS_PER_SM = (D == 64) ? 4 : (D == 256 ? 2 : 3);
    static_assert(DCH * 32 * 16 == SK && DCH == SUB * SUB_DIV, "copy split");
    static_assert(SC_PER_LANE * 32 == 2 * SCH, "scale copy split");
    static_assert((kWarps * kMaxGroup * D + 2 * kMaxRecW * kMaxGroup + 2 * kMaxGroup) * 4 <= SMEM,
                  "merge buffers must fit in the rings");
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
    int32_t B, Hq, H, G, T, pool_pages, max_pages, min_w;
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

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
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

template <int D>
__global__ void __launch_bounds__(kDecThreads, Geo<D>::BLOCKS_PER_SM)
    decode_split_kernel(const DecodeParams p) {
    pdl_enter();
    using G_ = Geo<D>;
    constexpr int TOK = G_::TOK;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ float red_m[kWarps][kMaxGroup];
    __shared__ float red_l[kWarps][kMaxGroup];
    __shared__ int page_ids[kPageBuf];
    __shared__ int scan_warp[kWarps];
    __shared__ int start_bp[2];  // pair walk start: sequence, its first stage
    __shared__ int last_s;
    __shared__ int pend_s[5];  // a pair whose count was bumped at the previous boundary: last?, b, h, start, stages

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int r = lane >> 2;  // row group of the MMA fragments
    const int c = lane & 3;   // column pair of the MMA fragments
    const int H = p.H, G = p.G, T = p.T;
    const int max_tokens = p.max_pages * T;

    // ------------------------------------------------ stage prefix over the sequences
    // Thread t owns sequences [t C, t C + C); PS_b = H * sum_{b' < b} stages(b').
    const int C = (p.B + kDecThreads - 1) / kDecThreads;
    const int b_lo = min(p.B, tid * C), b_hi = min(p.B, b_lo + C);
    int local = 0;
    for (int b = b_lo; b < b_hi; ++b) {
        const int L = __ldg(p.seq_lens + b);
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
    __syncthreads();
    int excl = incl - local, total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        if (w < warp) excl += scan_warp[w];
        total += scan_warp[w];
    }
    // CTA c takes the run [c W, c W + W) of the stage list
    const int n_ctas = gridDim.x;
    const int W = max(p.min_w, max(1, (total + n_ctas - 1) / n_ctas));
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
    const int s_begin = blockIdx.x * W;
    const int s_end = min(total, s_begin + W);
    if (s_begin >= s_end) return;
    if (s_begin >= excl && s_begin < excl + local) {
        int acc = excl;
        for (int b = b_lo; b < b_hi; ++b) {
            const int n = H * seq_stages(__ldg(p.seq_lens + b), max_tokens, TOK);
            if (s_begin < acc + n) {
                start_bp[0] = b;
                start_bp[1] = acc;
                break;
            }
            acc += n;
        }
    }
    if (tid == 0) pend_s[0] = 0;
    __syncthreads();

    // ------------------------------------------------ per-lane constants
    const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(smem)) + warp * G_::RING;
    // V chunk j = lane + 32 i of a stage lands XOR-swizzled by its pair row
    uint32_t v_dst[G_::DCH];
#pragma unroll
    for (int i = 0; i < G_::DCH; ++i) {
        const int j = lane + 32 * i;
        const int pr = j / G_::VCH, cj = j - pr * G_::VCH;
        v_dst[i] = G_::V_OFF + pr * D + 16 * (cj ^ (pr & G_::SWZ));
    }
    const int rho = (r >> 1) | ((r & 1) << 2);  // V rows of this lane: chunk rho of a pair row

    // ------------------------------------------------ walk the pieces of this CTA's run
    int b = start_bp[0];
    int S_b = seq_stages(__ldg(p.seq_lens + b), max_tokens, TOK);
    int h = (s_begin - start_bp[1]) / S_b;
    int j = (s_begin - start_bp[1]) - h * S_b;
    int pair_start = start_bp[1] + h * S_b;  // flat index of stage 0 of pair (b, h)
    int s = s_begin;
    bool first_piece = true;
    while (s < s_end) {
        const int j0 = j, j1 = min(S_b, j + (s_end - s));
        const int L = __ldg(p.seq_lens + b);
        const int tok_end = min(j1 * TOK, L);
        const int first_page = (j0 * TOK) / T;
        const int n_pages = (tok_end + T - 1) / T - first_page;
        const int32_t* pt_row = p.page_table + static_cast<int64_t>(b) * p.max_pages;
        if (first_piece) {
            for (int i = tid; i < n_pages && i < kPageBuf; i += kDecThreads)
                page_ids[i] = __ldg(pt_row + first_page + i);
            __syncthreads();
        }
        // (later pieces: their page ids were put in place before the previous piece's last barrier)
        first_piece = false;
        // the next piece of the run (the pair after (b, h), from its stage 0) and its page ids,
        // loaded now so that they are in registers when this piece ends
        const bool has_next = s + (j1 - j0) < s_end;
        int nid[2] = {0, 0};
        int nn_pages = 0;
        if (has_next) {
            int nb = b, nh = h + 1, nS = S_b;
            if (nh == H) {
                nh = 0;
                do {
                    ++nb;
                    nS = seq_stages(__ldg(p.seq_lens + nb), max_tokens, TOK);
                } while (nS == 0);
            }
            const int nj1 = min(nS, s_end - (pair_start + S_b));
            nn_pages = (min(nj1 * TOK, __ldg(p.seq_lens + nb)) + T - 1) / T;
            const int32_t* npt = p.page_table + static_cast<int64_t>(nb) * p.max_pages;
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                const int i = tid + q2 * kDecThreads;
                if (i < nn_pages && i < kPageBuf) nid[q2] = __ldg(npt + i);
            }
        }
        auto page_of = [&](int pidx) {
            const int k = pidx - first_page;
            const int pg = (k < kPageBuf) ? page_ids[k] : __ldg(pt_row + pidx);
            return (pg >= 0 && pg < p.pool_pages) ? pg : -1;
        };

        // ---- issue of one stage (index js within the pair) into a ring slot
        const int64_t head_rows = static_cast<int64_t>(h) * T;
        const int64_t page_rows = static_cast<int64_t>(H) * T;
        const bool page_aligned = (T % TOK) == 0;
        auto issue_stage = [&](int js, uint32_t slot) {
            const uint64_t kv_pol = l2_policy_evict_first();
            const int t0 = js * TOK;
            const int nval = min(TOK, L - t0);
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
                    row0[u] = -1;
                    if (16 * u < nval) {
                        const int t = t0 + 16 * u;
                        const int pidx =
                            static_cast<int>(__umul64hi(static_cast<uint64_t>(t), p.t_magic));
                        const int pg = page_of(pidx);
                        if (pg >= 0) row0[u] = pg * page_rows + head_rows + (t - pidx * T);
                    }
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
            if (lane == 0) sts_u32(slot + G_::HDR_OFF, okbits | (static_cast<uint32_t>(nval) << 8));
        };

        // this warp's stages of the piece: j0 + warp, j0 + warp + 4, ...
        const int n_st = max(0, (j1 - j0 - warp + kWarps - 1) / kWarps);
#pragma unroll
        for (int k = 0; k < kSlots - 1; ++k) {
            if (k < n_st) issue_stage(j0 + warp + kWarps * k, ring + k * G_::SLOT);
            cp_async_commit();
        }

        // ---- Q fragments of (b, h): lane (r, c) holds head r of the group; k-step kk covers
        // head dims c*D/4 + 4kk + {0..3} (the same permutation is used for K), as FP16 q * 2^kq.
        uint32_t qf[G_::KSTEPS][2];
        float cs_row = 0.0f;
        {
            float qv[D / 4];
            float qmax = 0.0f;
            if (r < G) {
                const uint16_t* qp =
                    p.q + (static_cast<int64_t>(b) * p.Hq + h * G + r) * D + c * (D / 4);
#pragma unroll
                for (int i = 0; i < D / 4; i += 8) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4*>(qp + i));
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        qv[i + 2 * k] = bf16_lo(wv[k]);
                        qv[i + 2 * k + 1] = bf16_hi(wv[k]);
                    }
                }
#pragma unroll
                for (int i = 0; i < D / 4; ++i) qmax = fmaxf(qmax, fabsf(qv[i]));
            } else {
#pragma unroll
                for (int i = 0; i < D / 4; ++i) qv[i] = 0.0f;
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
            if (r < G) cs_row = p.sm_scale * __ldg(p.gk) * kLog2e * ldexpf(1.0f, -kq);
        }
        // score scale of this lane's two S^T columns (query heads 2c, 2c+1)
        const float cs0 = __shfl_sync(0xFFFFFFFFu, cs_row, 8 * c);
        const float cs1 = __shfl_sync(0xFFFFFFFFu, cs_row, 8 * c + 4);

        float o[G_::KSTEPS][4];
#pragma unroll
        for (int m = 0; m < G_::KSTEPS; ++m)
#pragma unroll
            for (int k = 0; k < 4; ++k) o[m][k] = 0.0f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;

        // ---- main loop over this warp's stages
        for (int i = 0; i < n_st; ++i) {
            if (i + kSlots - 1 < n_st)
                issue_stage(j0 + warp + kWarps * (i + kSlots - 1),
                            ring + ((i + kSlots - 1) % kSlots) * G_::SLOT);
            cp_async_commit();
            cp_async_wait<kSlots - 1>();  // this lane's copies of stage i are done ...
            __syncwarp();                 // ... and so are the other lanes'
            const uint32_t st = ring + (i % kSlots) * G_::SLOT;
            const uint32_t hdr = lds_u32(st + G_::HDR_OFF);
            const uint32_t okbits = hdr & 0xFFu;
            const int nval = static_cast<int>(hdr >> 8);
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
            __syncwarp();  // every lane is done reading the slot before it refills
        }
        cp_async_wait<0>();

        // ---- merge the 4 warps and write the piece's record
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, off);
            l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, off);
        }
        if (r == 0) {
            red_m[warp][2 * c] = m0;
            red_m[warp][2 * c + 1] = m1;
            red_l[warp][2 * c] = l0;
            red_l[warp][2 * c + 1] = l1;
        }
        __syncthreads();  // every warp is done with its ring: the rings hold the merge buffer
        // the outcome of the count bumped at the previous boundary (written before this barrier)
        const int pend_last = pend_s[0];
        const int pend_b = pend_s[1], pend_h = pend_s[2], pend_ps = pend_s[3], pend_S = pend_s[4];
        float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            M0 = fmaxf(M0, red_m[w][2 * c]);
            M1 = fmaxf(M1, red_m[w][2 * c + 1]);
        }
        const float f0 = (m0 == -INFINITY) ? 0.0f : ex2_approx(m0 - M0);
        const float f1 = (m1 == -INFINITY) ? 0.0f : ex2_approx(m1 - M1);
        // over the drained rings: the warps' partial outputs [kWarps][kMaxGroup][D], then the
        // merge weights of a pair's records [kMaxRecW][kMaxGroup], merged (max, sum) per head, and the
        // records' sums [kMaxRecW][kMaxGroup]
        float* so = reinterpret_cast<float*>(smem);
        float (*mw_s)[kMaxGroup] = reinterpret_cast<float (*)[kMaxGroup]>(so + kWarps * kMaxGroup * D);
        float (*ml_s)[2] = reinterpret_cast<float (*)[2]>(so + kWarps * kMaxGroup * D + kMaxRecW * kMaxGroup);
        float (*lw_s)[kMaxGroup] = reinterpret_cast<float (*)[kMaxGroup]>(
            so + kWarps * kMaxGroup * D + kMaxRecW * kMaxGroup + 2 * kMaxGroup);
#pragma unroll
        for (int m = 0; m < G_::KSTEPS; ++m) {
            const int d0 = rho * (D / 8) + 2 * m;
            float* base = so + (warp * kMaxGroup + 2 * c) * D;
            base[d0] = o[m][0] * f0;
            base[D + d0] = o[m][1] * f1;
            base[d0 + 1] = o[m][2] * f0;
            base[D + d0 + 1] = o[m][3] * f1;
        }
        __syncthreads();
        // CTAs c_first .. c_last cover the pair, each leaving record c + (b H + h); the last of
        // them to finish merges the records
        const int c_first = pair_start / W, c_last = (pair_start + S_b - 1) / W;
        const int n_rec = c_last - c_first + 1;
        const int64_t bh64 = static_cast<int64_t>(b) * H + h;
        auto rec_index = [&](int k) -> int64_t { return c_first + k + bh64; };
        const float gvs = __ldg(p.gv);
        // merge the records of pair (mb, mh) once all of them are written (by the CTA whose
        // count completed them), writing its output and LSE
        auto merge_records = [&](int mb, int mh, int mps, int mS) {
            const int c_first_m = mps / W, c_last_m = (mps + mS - 1) / W;
            const int n_rec_m = c_last_m - c_first_m + 1;
            const int64_t bh_m = static_cast<int64_t>(mb) * H + mh;
            auto rec_index_m = [&](int k) -> int64_t { return c_first_m + k + bh_m; };
            // every record of the pair is written: merge them (L2 reads, not L1). The (max,
            // sum) pairs of up to kMaxRecW records are staged in shared memory by one round
            // of loads while the first records' outputs are already in flight.
            __threadfence();
            // every CTA of the pair has counted, so the count can go back to 0: a replay of the
            // same launch (a captured CUDA graph, same tag) starts from a clean word
            if (tid == 0) atomicExch(p.done + bh_m, 0ull);
            constexpr int NQ = kMaxGroup * D / kDecThreads;
            constexpr int kRecUnroll = NQ >= 16 ? 2 : 8;  // record values in flight: 32 or 64
            const int n_fast = min(n_rec_m, kMaxRecW);
            for (int idx = tid; idx < n_fast * G; idx += kDecThreads) {
                const int k = idx / G, col = idx - (idx / G) * G;
                const float2 ml = __ldcg(reinterpret_cast<const float2*>(
                    p.rec_ml + (rec_index_m(k) * G + col) * 2));
                mw_s[k][col] = ml.x;
                lw_s[k][col] = ml.y;
            }
            float v[kRecUnroll][NQ];
            auto load_recs = [&](int k0) {
#pragma unroll
                for (int u = 0; u < kRecUnroll; ++u) {
                    const int k = min(k0 + u, n_rec_m - 1);
                    const float* rk = p.rec_o + rec_index_m(k) * G * D;
#pragma unroll
                    for (int q = 0; q < NQ; ++q) {
                        const int i = tid + kDecThreads * q;
                        v[u][q] = (i < G * D) ? __ldcg(rk + i) : 0.0f;
                    }
                }
            };
            load_recs(0);
            __syncthreads();
            if (warp < G) {  // warp w: query heads w, w + 4
                for (int col = warp; col < G; col += kWarps) {
                    auto m_of = [&](int k) {
                        return k < n_fast ? mw_s[k][col]
                                          : __ldcg(p.rec_ml + (rec_index_m(k) * G + col) * 2);
                    };
                    float M = -INFINITY;
                    for (int k = lane; k < n_rec_m; k += 32) M = fmaxf(M, m_of(k));
#pragma unroll
                    for (int o2 = 16; o2 > 0; o2 >>= 1)
                        M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o2));
                    float lsum = 0.0f;
                    for (int k = lane; k < n_rec_m; k += 32) {
                        const float mk = m_of(k);
                        const float lk = k < n_fast
                                             ? lw_s[k][col]
                                             : __ldcg(p.rec_ml + (rec_index_m(k) * G + col) * 2 + 1);
                        const float wk = (mk == -INFINITY) ? 0.0f : exp2f(mk - M);
                        if (k < n_fast) mw_s[k][col] = wk;  // this lane alone reads entry k
                        lsum += wk * lk;
                    }
#pragma unroll
                    for (int o2 = 16; o2 > 0; o2 >>= 1)
                        lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, o2);
                    if (lane == 0) {
                        ml_s[col][0] = M;
                        ml_s[col][1] = lsum;
                        if (p.lse)
                            p.lse[static_cast<int64_t>(mb) * p.Hq + mh * G + col] =
                                (lsum > 0.0f) ? (M + log2f(lsum)) * 0.6931471805599453f
                                              : -INFINITY;
                    }
                }
            }
            __syncthreads();
            // thread tid owns outputs i = tid + kDecThreads q; kRecUnroll records at a time
            float acc[NQ];
#pragma unroll
            for (int q = 0; q < NQ; ++q) acc[q] = 0.0f;
            for (int k0 = 0; k0 < n_rec_m; k0 += kRecUnroll) {
                if (k0 > 0) load_recs(k0);
#pragma unroll
                for (int u = 0; u < kRecUnroll; ++u) {
                    const int k = k0 + u;
                    if (k >= n_rec_m) break;
#pragma unroll
                    for (int q = 0; q < NQ; ++q) {
                        const int i = tid + kDecThreads * q;
                        if (i >= G * D) continue;
                        const int col = i / D;
                        float wk;
                        if (k < n_fast) {
                            wk = mw_s[k][col];
                        } else {
                            const float mk = __ldcg(p.rec_ml + (rec_index_m(k) * G + col) * 2);
                            wk = (mk == -INFINITY) ? 0.0f : exp2f(mk - ml_s[col][0]);
                        }
                        acc[q] += wk * v[u][q];
                    }
                }
            }
            uint16_t* ob = p.out + (static_cast<int64_t>(mb) * p.Hq + mh * G) * D;
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const int i = tid + kDecThreads * q;
                if (i >= G * D) continue;
                const float ls = ml_s[i / D][1];
                const __nv_bfloat16 yb = __float2bfloat16_rn(ls > 0.0f ? acc[q] * (gvs / ls) : 0.0f);
                ob[i] = *reinterpret_cast<const uint16_t*>(&yb);
            }
        };
        if (n_rec == 1) {
            // the whole pair is this piece: normalise and write the output directly
            if (tid < G) {
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w][tid]);
                float lsum = 0.0f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float mw = red_m[w][tid];
                    if (mw != -INFINITY) lsum += red_l[w][tid] * ex2_approx(mw - M);
                }
                ml_s[tid][0] = M;
                ml_s[tid][1] = lsum;
                if (p.lse)
                    p.lse[static_cast<int64_t>(b) * p.Hq + h * G + tid] =
                        (lsum > 0.0f) ? (M + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
            }
            __syncthreads();
            uint16_t* ob = p.out + (static_cast<int64_t>(b) * p.Hq + h * G) * D;
            for (int i = tid; i < G * D; i += kDecThreads) {
                const int col = i / D, d = i - (i / D) * D;
                float acc = 0.0f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) acc += so[(w * kMaxGroup + col) * D + d];
                const float ls = ml_s[col][1];
                const __nv_bfloat16 yb = __float2bfloat16_rn(ls > 0.0f ? acc * (gvs / ls) : 0.0f);
                ob[i] = *reinterpret_cast<const uint16_t*>(&yb);
            }
        } else {
            const int64_t rec = blockIdx.x + bh64;
            float* ro = p.rec_o + rec * G * D;
            for (int i = tid; i < G * D; i += kDecThreads) {
                const int col = i / D, d = i - (i / D) * D;
                float acc = 0.0f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) acc += so[(w * kMaxGroup + col) * D + d];
                ro[i] = acc;
            }
            if (tid < G) {
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w][tid]);
                float lsum = 0.0f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float mw = red_m[w][tid];
                    if (mw != -INFINITY) lsum += red_l[w][tid] * ex2_approx(mw - M);
                }
                p.rec_ml[(rec * G + tid) * 2] = M;
                p.rec_ml[(rec * G + tid) * 2 + 1] = lsum;
            }
        }
        if (has_next) {
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                const int i = tid + q2 * kDecThreads;
                if (i < nn_pages && i < kPageBuf) page_ids[i] = nid[q2];
            }
        }
        __syncthreads();  // outputs / record written, merge buffer read, next page ids in place
        if (pend_last) {
            merge_records(pend_b, pend_h, pend_ps, pend_S);
            __syncthreads();  // the merge is done with the rings
        }
        if (n_rec > 1) {
            if (has_next) {
                // publish the record without holding up the next piece: one lane of the last
                // warp makes it visible and bumps the count; the outcome is read at the next
                // piece's end, where a completed pair is merged
                if (warp == kWarps - 1 && lane == 0) {
                    __threadfence();
                    unsigned long long* cnt = p.done + bh64;
                    const uint32_t k = tagged_finish(cnt, atomicAdd(cnt, 1ull), p.nonce, 1);
                    pend_s[0] = (k == static_cast<uint32_t>(n_rec - 1)) ? 1 : 0;
                    pend_s[1] = b;
                    pend_s[2] = h;
                    pend_s[3] = pair_start;
                    pend_s[4] = S_b;
                }
            } else {
                if (tid == 0) {
                    __threadfence();  // the record is visible before the count says so
                    unsigned long long* cnt = p.done + bh64;
                    const uint32_t k = tagged_finish(cnt, atomicAdd(cnt, 1ull), p.nonce, 1);
                    last_s = (k == static_cast<uint32_t>(n_rec - 1)) ? 1 : 0;
                }
                __syncthreads();
                if (last_s) merge_records(b, h, pair_start, S_b);
            }
        } else if (has_next && warp == kWarps - 1 && lane == 0) {
            pend_s[0] = 0;
        }

        // ---- next piece: the next pair with at least one stage
        s += j1 - j0;
        j = 0;
        pair_start += S_b;
        if (s < s_end) {
            if (++h == H) {
                h = 0;
                do {
                    ++b;
                    S_b = seq_stages(__ldg(p.seq_lens + b), max_tokens, TOK);
                } while (S_b == 0);
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
// Host side: grid, workspace carving
// ------------------------------------------------------------------------------------------
size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int stage_tokens(int D) { return D == 256 ? 32 : 64; }
int blocks_per_sm(int D) { return D == 64 ? 4 : (D == 256 ? 2 : 3); }

// CTAs of the split kernel: one wave (automatic), or n runs per (sequence, KV head) pair.
int64_t decode_ctas(int batch, int H, int D, int max_num_splits) {
    if (max_num_splits > 0) return static_cast<int64_t>(max_num_splits) * batch * H;
    return static_cast<int64_t>(num_sms()) * blocks_per_sm(D);
}

struct WsLayout {
    size_t done, ml, o, total;
};

// Records: one per (CTA, pair) it covers; bounded by CTAs + pairs because runs are consecutive
WsLayout ws_layout(int batch, int H, int Hq, int D, int64_t ctas) {
    const size_t pairs = static_cast<size_t>(batch) * H;
    const size_t records = static_cast<size_t>(ctas) + pairs;
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
bool decode_size_ok(int batch, int H, int D, int max_pages, int T, int64_t ctas) {
    const int64_t max_tokens = static_cast<int64_t>(max_pages) * T;
    const int64_t tok = stage_tokens(D);
    const int64_t stages = (max_tokens + tok - 1) / tok * batch * H;
    const int64_t lim = (int64_t{1} << 31) - 1;
    return max_tokens < lim - tok && stages + ctas * kWarps < lim &&
           ctas + static_cast<int64_t>(batch) * H < lim;
}

template <int D>
cudaError_t launch_decode(const DecodeParams& p, int64_t ctas, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Geo<D>::SMEM);
    if (e != cudaSuccess) return e;
    e = launch_pdl(decode_split_kernel<D>, static_cast<unsigned>(ctas), kDecThreads,
                   static_cast<size_t>(Geo<D>::SMEM), s, p);
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
    const int64_t ctas = decode_ctas(batch, H, layout->head_dim, max_num_splits);
    return ws_layout(batch, H, num_q_heads, layout->head_dim, ctas).total;
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
    const int64_t ctas = decode_ctas(batch, H, D, max_num_splits);
    if (!decode_size_ok(batch, H, D, max_pages_per_seq, T, ctas)) return NVFP4KV_ERR_UNSUPPORTED;
    const WsLayout wl = ws_layout(batch, H, num_q_heads, D, ctas);
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
    p.min_w = (max_num_splits > 0) ? 1 : kWarps;
    p.sm_scale = sm_scale;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (D) {
    case 64: e = launch_decode<64>(p, ctas, s); break;
    case 128: e = launch_decode<128>(p, ctas, s); break;
    default: e = launch_decode<256>(p, ctas, s); break;
    }
    if (e != cudaSuccess) return NVFP4KV_ERR_CUDA;

    return NVFP4KV_OK;
}
