// Split-KV paged GQA decode attention over NVFP4 K/V for sm_103a, plus the combine pass.
//
// What it computes ("Accelerating Long-Context and Agentic Inference with NVFP4 KV Cache",
// LMSYS: "Path 3: Decode", "NVFP4 KV Decode Attention Kernel Implementation", Figure 3): for
// each sequence and query head, softmax(sm_scale q.K^T) V over the sequence's tokens, with K
// and V read in their packed NVFP4 form straight from the paged cache and dequantized in
// registers. The global K/V scales are folded into the score scale and the final output
// ("supplied through the attention BMM scaling parameters").
//
// Design for GB300 (the SM120 kernel of the LMSYS page is prior art, not the blueprint):
//  * one CTA per (sequence, KV head, split) of 4 warps; a split is a run of 64-token stages.
//    Each stage is staged into shared memory by 1-D bulk async copies (TMA engine, one issuing
//    thread, L2 evict-first) of the packed K/V rows and their E4M3 scales, page by page through
//    the page table, into a 4-deep ring tracked by mbarriers with transaction counts.
//  * each warp owns 16 tokens of a stage. S^T = K^ Q^T on the tensor cores with tokens as the
//    M = 16 dimension and the GQA query group as N = 8 (mma.sync m16n8k16, FP16 in, FP32
//    accumulate): the decoded K values e2m1 * e4m3 are exact in FP16 (cvt.rn.f16x2.e2m1x2,
//    cvt.rn.f16x2.e4m3x2, one packed multiply), and Q is brought into FP16 exactly by a
//    per-head power of two. The head dimension inside a k-step is permuted identically in K and
//    Q so that every K fragment register is one converted byte.
//  * online softmax in the log2 domain with warp shuffles for the column maxima; the running
//    maximum is only moved when it grows by more than 2^8, so rescaling of the accumulators is
//    rare. P^T goes from the score accumulator layout to the B-operand layout with movmatrix.
//  * O^T += V^^T P^T with head_dim as M: V tiles are read transposed with ldmatrix.trans, each
//    register is split into four e2m1x2 conversions and re-paired by token with byte permutes,
//    and the V block scales are applied per element pair (exact in FP16).
//  * the 4 warps merge their (max, sum, output) in shared memory and the CTA writes one
//    partial per (sequence, query head, split); a second kernel merges the splits by their
//    log-sum-exp and writes BF16 output and the natural-log LSE.
// Everything is HBM-bound: 144 bytes of K+V per (token, KV head) at head_dim 128.
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_util.h"

namespace nvfp4kv {
namespace {

constexpr int kWarps = 4;
constexpr int kDecThreads = kWarps * 32;
constexpr int kStageTokens = 64;
constexpr int kStages = 4;
constexpr int kMaxGroup = 8;
constexpr int kMaxSplits = 64;
constexpr uint64_t kWaitLimitNs = 500ull * 1000ull * 1000ull;  // 0.5 s per copy-completion wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Geo {
    static constexpr int KD = kStageTokens * D / 2;   // packed bytes of one stage of K (or V)
    static constexpr int KS = kStageTokens * D / 16;  // scale bytes of one stage of K (or V)
    static constexpr int STAGE = 2 * (KD + KS);
    static constexpr int NB = D / 16;                 // blocks (= scales) per token row
    static constexpr int KSTEPS = D / 16;             // k-steps of S^T = K Q^T
    static constexpr int SEGS = D / 32;               // 16-byte segments of a packed token row
    static constexpr int CHUNK = D / 8;               // bytes of a K row owned by one quad lane
    static constexpr int SMEM = kStages * STAGE;
};

struct DecodeParams {
    const uint16_t* q;  // BF16 bit patterns [B][Hq][D]
    const uint8_t* kd;
    const uint8_t* ks;
    const uint8_t* vd;
    const uint8_t* vs;
    const float* gk;
    const float* gv;
    const int32_t* page_table;
    const int32_t* seq_lens;
    float* part_o;  // [B][Hq][S][D]
    float* part_m;  // [B][Hq][S]   running max (log2 domain)
    float* part_l;  // [B][Hq][S]   sum of exp2(x - m)
    int32_t* status;
    int32_t B, Hq, H, G, T, pool_pages, max_pages, num_splits, stages_per_split;
    float sm_scale;
};

__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b) {
    const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a),
                              *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// E4M3 byte `k` of word w, as an FP16 pair (s, s).
__device__ __forceinline__ uint32_t scale_bcast(uint32_t w, int k) {
    const uint32_t b = (w >> (8 * k)) & 0xFFu;
    return e4m3x2_to_f16x2(b * 0x0101u);
}

template <int N>
__device__ __forceinline__ void lds_words(uint32_t (&w)[N], const uint8_t* p) {
    if constexpr (N == 1) {
        w[0] = *reinterpret_cast<const uint32_t*>(p);
    } else if constexpr (N == 2) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        w[0] = v.x;
        w[1] = v.y;
    } else {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(p + 4 * i);
            w[i] = v.x;
            w[i + 1] = v.y;
            w[i + 2] = v.z;
            w[i + 3] = v.w;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kDecThreads, 4) decode_split_kernel(const DecodeParams p) {
    using G_ = Geo<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ uint64_t stage_mask[kStages];
    __shared__ float red_m[kWarps][kMaxGroup];
    __shared__ float red_l[kWarps][kMaxGroup];

    const int split = blockIdx.x;
    const int h = blockIdx.y;
    const int b = blockIdx.z;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int r = lane >> 2;  // row group of the MMA fragments
    const int c = lane & 3;   // column pair of the MMA fragments

    const int L = __ldg(p.seq_lens + b);
    if (L < 0 || L > p.max_pages * p.T) {
        if (tid == 0 && split == 0 && h == 0) flag_status(p.status, NVFP4KV_STATUS_BAD_SEQ_LEN);
        return;  // the combine pass applies the same rule and writes zeros
    }
    const int total_stages = (L + kStageTokens - 1) / kStageTokens;
    const int st_begin = split * p.stages_per_split;
    const int st_end = min(st_begin + p.stages_per_split, total_stages);
    if (st_begin >= st_end) return;  // beyond this sequence: no partial (combine skips it)
    const int nst = st_end - st_begin;
    const int G = p.G;
    const int64_t part_row = (static_cast<int64_t>(b) * p.Hq + h * G) * p.num_splits + split;

    // ---------------------------------------------------------------- producer (thread 0)
    const uint64_t policy = l2_policy_evict_first();
    auto issue_stage = [&](int gs, int slot) {
        const int tok0 = gs * kStageTokens;
        uint8_t* st = smem + slot * G_::STAGE;
        int piece_tok[kStageTokens / 16], piece_n[kStageTokens / 16], piece_pg[kStageTokens / 16];
        int np = 0;
        uint64_t mask = 0;
        uint32_t bytes = 0;
        for (int t = tok0; t < tok0 + kStageTokens && t < L;) {
            const int pidx = t / p.T;
            const int off = t - pidx * p.T;
            const int n = min(p.T - off, tok0 + kStageTokens - t);
            const int page = __ldg(p.page_table + static_cast<int64_t>(b) * p.max_pages + pidx);
            if (page >= 0 && page < p.pool_pages) {
                piece_tok[np] = t;
                piece_n[np] = n;
                piece_pg[np] = page;
                ++np;
                bytes += 2u * n * (D / 2 + G_::NB);
                const int valid = min(n, L - t);
                const uint64_t bits = (valid >= 64) ? ~0ull : ((1ull << valid) - 1ull);
                mask |= bits << (t - tok0);
            } else {
                flag_status(p.status, NVFP4KV_STATUS_PAGE_OOB);
            }
            t += n;
        }
        stage_mask[slot] = mask;
        mbar_arrive_expect_tx(&full_bar[slot], bytes);
        for (int i = 0; i < np; ++i) {
            const int off = piece_tok[i] - (piece_tok[i] / p.T) * p.T;
            const int64_t row = (static_cast<int64_t>(piece_pg[i]) * p.H + h) * p.T + off;
            const int lt = piece_tok[i] - tok0;
            const uint32_t nd = piece_n[i] * (D / 2), ns = piece_n[i] * G_::NB;
            bulk_g2s(st + lt * (D / 2), p.kd + row * (D / 2), nd, &full_bar[slot], policy);
            bulk_g2s(st + G_::KD + lt * (D / 2), p.vd + row * (D / 2), nd, &full_bar[slot],
                     policy);
            bulk_g2s(st + 2 * G_::KD + lt * G_::NB, p.ks + row * G_::NB, ns, &full_bar[slot],
                     policy);
            bulk_g2s(st + 2 * G_::KD + G_::KS + lt * G_::NB, p.vs + row * G_::NB, ns,
                     &full_bar[slot], policy);
        }
    };

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s) mbar_init(&full_bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        for (int s = 0; s < kStages && s < nst; ++s) issue_stage(st_begin + s, s);
    }

    // ---------------------------------------------------------------- Q fragments
    // Lane (r, c) holds head r of the group; k-step j covers head dims c*D/4 + 4j + {0..3}
    // (the same permutation is used for K), as FP16 q * 2^kq.
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
        // qmax * 2^kq in [2^14, 2^15): every BF16 value of the head is exact in FP16 down to
        // 2^-18 of the head maximum.
        int kq = (qmax > 0.0f) ? (14 - ilogbf(qmax)) : 0;
        kq = max(-120, min(kq, 120));
        const float up = ldexpf(1.0f, kq);
#pragma unroll
        for (int j = 0; j < G_::KSTEPS; ++j) {
            qf[j][0] = pack_f16x2(qv[4 * j] * up, qv[4 * j + 1] * up);
            qf[j][1] = pack_f16x2(qv[4 * j + 2] * up, qv[4 * j + 3] * up);
        }
        if (r < G) cs_row = p.sm_scale * __ldg(p.gk) * kLog2e * ldexpf(1.0f, -kq);
    }
    // score scale of this lane's two S^T columns (query heads 2c, 2c+1)
    const float cs0 = __shfl_sync(0xFFFFFFFFu, cs_row, 8 * c);
    const float cs1 = __shfl_sync(0xFFFFFFFFu, cs_row, 8 * c + 4);

    float o[G_::SEGS][2][4];
#pragma unroll
    for (int s = 0; s < G_::SEGS; ++s)
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int k = 0; k < 4; ++k) o[s][x][k] = 0.0f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    const uint32_t vsel = 0x6240u + (r >> 2) * 0x1111u;  // V scale byte pairing (see below)

    // ---------------------------------------------------------------- main loop
    bool timed_out = false;
    int failed_at = 0;
    for (int j = 0; j < nst; ++j) {
        const int slot = j % kStages;
        const uint32_t parity = (j / kStages) & 1;
        const bool ok = mbar_wait_bounded(&full_bar[slot], parity, kWaitLimitNs);
        const uint32_t tmask =
            ok ? static_cast<uint32_t>(stage_mask[slot] >> (16 * warp)) & 0xFFFFu : 0u;
        if (tmask != 0u) {
            const uint8_t* st = smem + slot * G_::STAGE;
            const uint8_t* kd_s = st;
            const uint8_t* vd_s = st + G_::KD;
            const uint8_t* ks_s = st + 2 * G_::KD;
            const uint8_t* vs_s = ks_s + G_::KS;
            const int row0 = 16 * warp + r;
            const int row1 = row0 + 8;

            // ---- S^T = K^ Q^T (tokens x query heads)
            uint32_t kw0[G_::CHUNK / 4], kw1[G_::CHUNK / 4];
            lds_words(kw0, kd_s + row0 * (D / 2) + c * G_::CHUNK);
            lds_words(kw1, kd_s + row1 * (D / 2) + c * G_::CHUNK);
            uint32_t ksw0, ksw1;  // this lane's D/64 scale bytes of rows row0 / row1
            if constexpr (D == 64) {
                ksw0 = ks_s[row0 * G_::NB + c];
                ksw1 = ks_s[row1 * G_::NB + c];
            } else if constexpr (D == 128) {
                ksw0 = *reinterpret_cast<const uint16_t*>(ks_s + row0 * G_::NB + 2 * c);
                ksw1 = *reinterpret_cast<const uint16_t*>(ks_s + row1 * G_::NB + 2 * c);
            } else {
                ksw0 = *reinterpret_cast<const uint32_t*>(ks_s + row0 * G_::NB + 4 * c);
                ksw1 = *reinterpret_cast<const uint32_t*>(ks_s + row1 * G_::NB + 4 * c);
            }
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int k = 0; k < G_::KSTEPS; ++k) {
                const uint32_t w0 = kw0[k / 2], w1 = kw1[k / 2];
                const int sh = (k & 1) * 16;
                const uint32_t s0 = scale_bcast(ksw0, k / 4);
                const uint32_t s1 = scale_bcast(ksw1, k / 4);
                uint32_t a[4];
                a[0] = h2_mul(e2m1x2_to_f16x2(w0 >> sh), s0);
                a[1] = h2_mul(e2m1x2_to_f16x2(w1 >> sh), s1);
                a[2] = h2_mul(e2m1x2_to_f16x2(w0 >> (sh + 8)), s0);
                a[3] = h2_mul(e2m1x2_to_f16x2(w1 >> (sh + 8)), s1);
                mma_f16_16816(acc, a, qf[k][0], qf[k][1]);
            }

            // ---- online softmax (log2 domain), columns = query heads 2c, 2c+1
            float x0 = acc[0] * cs0, x1 = acc[1] * cs1, x2 = acc[2] * cs0, x3 = acc[3] * cs1;
            if (tmask != 0xFFFFu) {
                if (!((tmask >> r) & 1u)) x0 = x1 = -INFINITY;
                if (!((tmask >> (r + 8)) & 1u)) x2 = x3 = -INFINITY;
            }
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, off));
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
                for (int s = 0; s < G_::SEGS; ++s)
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        o[s][x][0] *= a0;
                        o[s][x][1] *= a1;
                        o[s][x][2] *= a0;
                        o[s][x][3] *= a1;
                    }
            }
            const float p0 = ex2_approx(x0 - m0), p1 = ex2_approx(x1 - m1);
            const float p2 = ex2_approx(x2 - m0), p3 = ex2_approx(x3 - m1);
            l0 += p0 + p2;
            l1 += p1 + p3;
            // P^T (tokens x heads) -> B operand (k = tokens, n = heads)
            const uint32_t pb0 = movmatrix_trans(pack_f16x2(p0, p1));
            const uint32_t pb1 = movmatrix_trans(pack_f16x2(p2, p3));

            // ---- V block scales: pair (token a = 2c + 8hf, token b = a + 1) of block
            // 2*seg + (r >> 2), for every segment seg; zero for tokens outside the sequence.
            uint32_t vsp[G_::SEGS][2];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int ta = 16 * warp + 2 * c + 8 * hf;
                uint32_t wa[G_::NB / 4], wb[G_::NB / 4];
                lds_words(wa, vs_s + ta * G_::NB);
                lds_words(wb, vs_s + (ta + 1) * G_::NB);
                uint32_t keep = 0xFFFFFFFFu;
                if (tmask != 0xFFFFu) {
                    keep = (((tmask >> (2 * c + 8 * hf)) & 1u) ? 0x0000FFFFu : 0u) |
                           (((tmask >> (2 * c + 1 + 8 * hf)) & 1u) ? 0xFFFF0000u : 0u);
                }
#pragma unroll
                for (int u = 0; u < G_::NB / 4; ++u) {
                    const uint32_t pr = prmt(wa[u], wb[u], vsel);
                    vsp[2 * u][hf] = e4m3x2_to_f16x2(pr & 0xFFFFu) & keep;
                    vsp[2 * u + 1][hf] = e4m3x2_to_f16x2(pr >> 16) & keep;
                }
            }

            // ---- O^T += V^^T P^T, head dims as M: M-tile (seg, x) row r <-> dim
            // 32 seg + 4 r + 2 x, row r + 8 <-> that dim + 1.
#pragma unroll
            for (int g4 = 0; g4 < D / 64; ++g4) {
                const int mi = lane >> 3;  // which of the 4 matrices this lane addresses
                const int seg_l = 2 * g4 + (mi >> 1);
                const int tok_l = 16 * warp + 8 * (mi & 1) + (lane & 7);
                uint32_t R[4];
                ldmatrix_x4_trans(R, smem_u32(vd_s + tok_l * (D / 2) + seg_l * 16));
#pragma unroll
                for (int sx = 0; sx < 2; ++sx) {
                    const int seg = 2 * g4 + sx;
                    uint32_t va[2][4];
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const uint32_t w = R[2 * sx + hf];
                        const uint32_t X0 = e2m1x2_to_f16x2(w);
                        const uint32_t X1 = e2m1x2_to_f16x2(w >> 8);
                        const uint32_t Y0 = e2m1x2_to_f16x2(w >> 16);
                        const uint32_t Y1 = e2m1x2_to_f16x2(w >> 24);
                        const uint32_t sc = vsp[seg][hf];
                        va[0][2 * hf + 0] = h2_mul(prmt(X0, Y0, 0x5410u), sc);
                        va[0][2 * hf + 1] = h2_mul(prmt(X0, Y0, 0x7632u), sc);
                        va[1][2 * hf + 0] = h2_mul(prmt(X1, Y1, 0x5410u), sc);
                        va[1][2 * hf + 1] = h2_mul(prmt(X1, Y1, 0x7632u), sc);
                    }
                    mma_f16_16816(o[seg][0], va[0], pb0, pb1);
                    mma_f16_16816(o[seg][1], va[1], pb0, pb1);
                }
            }
        }
        timed_out = !ok;
        if (__syncthreads_or(timed_out ? 1 : 0)) {
            timed_out = true;
            failed_at = j;
            break;
        }
        if (tid == 0 && j + kStages < nst) issue_stage(st_begin + j + kStages, slot);
    }

    if (timed_out) {
        // Some copy never completed: wait (bounded) for every stage still in flight, then
        // leave an empty partial so the combine pass ignores this unit.
        if (tid == 0) {
            flag_status(p.status, NVFP4KV_STATUS_TIMEOUT);
            // stages failed_at .. failed_at + kStages - 1 may have been issued
            for (int jj = failed_at; jj < nst && jj < failed_at + kStages; ++jj)
                (void)mbar_wait_bounded(&full_bar[jj % kStages], (jj / kStages) & 1, kWaitLimitNs);
        }
        __syncthreads();
        for (int i = tid; i < G * D; i += kDecThreads)
            p.part_o[(part_row + static_cast<int64_t>(i / D) * p.num_splits) * D + i % D] = 0.0f;
        if (tid < G) {
            p.part_m[part_row + static_cast<int64_t>(tid) * p.num_splits] = -INFINITY;
            p.part_l[part_row + static_cast<int64_t>(tid) * p.num_splits] = 0.0f;
        }
        return;
    }

    // ---------------------------------------------------------------- merge the 4 warps
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
    __syncthreads();  // all stages consumed: the stage ring is free for the merge buffer
    float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        M0 = fmaxf(M0, red_m[w][2 * c]);
        M1 = fmaxf(M1, red_m[w][2 * c + 1]);
    }
    const float f0 = (m0 == -INFINITY) ? 0.0f : ex2_approx(m0 - M0);
    const float f1 = (m1 == -INFINITY) ? 0.0f : ex2_approx(m1 - M1);
    float* so = reinterpret_cast<float*>(smem);  // [kWarps][kMaxGroup][D]
#pragma unroll
    for (int s = 0; s < G_::SEGS; ++s)
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const int d0 = 32 * s + 4 * r + 2 * x;
            float* base = so + (warp * kMaxGroup + 2 * c) * D;
            base[d0] = o[s][x][0] * f0;
            base[D + d0] = o[s][x][1] * f1;
            base[d0 + 1] = o[s][x][2] * f0;
            base[D + d0 + 1] = o[s][x][3] * f1;
        }
    __syncthreads();
    for (int i = tid; i < G * D; i += kDecThreads) {
        const int col = i / D, d = i - (i / D) * D;
        float acc = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) acc += so[(w * kMaxGroup + col) * D + d];
        p.part_o[(part_row + static_cast<int64_t>(col) * p.num_splits) * D + d] = acc;
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
        p.part_m[part_row + static_cast<int64_t>(tid) * p.num_splits] = M;
        p.part_l[part_row + static_cast<int64_t>(tid) * p.num_splits] = lsum;
    }
}

// ------------------------------------------------------------------------------------------
// Combine: out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s; lse = ln 2 (M + log2 L).
// The global V scale multiplies the result once here.
// ------------------------------------------------------------------------------------------
struct CombineParams {
    const float* part_o;
    const float* part_m;
    const float* part_l;
    const int32_t* seq_lens;
    const float* gv;
    uint16_t* out;  // BF16 bits [B][Hq][D]
    float* lse;     // [B][Hq] or null
    int32_t Hq, D, T, max_pages, num_splits, stages_per_split;
};

__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
    const int qh = blockIdx.x, b = blockIdx.y;
    const int L = __ldg(p.seq_lens + b);
    int n_act = 0;
    if (L > 0 && L <= p.max_pages * p.T) {
        const int total_stages = (L + kStageTokens - 1) / kStageTokens;
        n_act = (total_stages + p.stages_per_split - 1) / p.stages_per_split;
    }
    const int64_t row = (static_cast<int64_t>(b) * p.Hq + qh) * p.num_splits;
    __shared__ float w_s[kMaxSplits];
    __shared__ float inv_l;
    if (threadIdx.x == 0) {
        float M = -INFINITY;
        for (int s = 0; s < n_act; ++s) M = fmaxf(M, p.part_m[row + s]);
        float lsum = 0.0f;
        for (int s = 0; s < n_act; ++s) {
            const float ms = p.part_m[row + s];
            const float w = (ms == -INFINITY) ? 0.0f : exp2f(ms - M);
            w_s[s] = w;
            lsum += w * p.part_l[row + s];
        }
        inv_l = (lsum > 0.0f) ? __ldg(p.gv) / lsum : 0.0f;
        if (p.lse)
            p.lse[static_cast<int64_t>(b) * p.Hq + qh] =
                (lsum > 0.0f) ? (M + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    for (int d = threadIdx.x; d < p.D; d += blockDim.x) {
        float acc = 0.0f;
        for (int s = 0; s < n_act; ++s)
            if (w_s[s] != 0.0f) acc += w_s[s] * p.part_o[(row + s) * p.D + d];
        const float y = acc * inv_l;
        const __nv_bfloat16 yb = __float2bfloat16_rn(y);
        p.out[(static_cast<int64_t>(b) * p.Hq + qh) * p.D + d] =
            *reinterpret_cast<const uint16_t*>(&yb);
    }
}

// ------------------------------------------------------------------------------------------
// Host side: split heuristic and workspace carving
// ------------------------------------------------------------------------------------------
struct SplitPlan {
    int num_splits;
    int stages_per_split;
};

SplitPlan plan_splits(int batch, int H, int max_pages, int T, int max_num_splits) {
    const int64_t max_tokens = static_cast<int64_t>(max_pages) * T;
    const int max_stages =
        static_cast<int>(std::max<int64_t>(1, (max_tokens + kStageTokens - 1) / kStageTokens));
    int cap = max_num_splits > 0 ? max_num_splits : kMaxSplits;
    cap = std::min(cap, max_stages);
    int n;
    if (max_num_splits > 0) {
        n = cap;
    } else {
        // about four waves of four resident CTAs per SM
        const int64_t target = static_cast<int64_t>(num_sms()) * 16;
        const int64_t pairs = std::max<int64_t>(1, static_cast<int64_t>(batch) * H);
        n = static_cast<int>(std::min<int64_t>(cap, (target + pairs - 1) / pairs));
        n = std::max(n, 1);
    }
    const int sps = (max_stages + n - 1) / n;
    return SplitPlan{(max_stages + sps - 1) / sps, sps};
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
    size_t o, m, l, total;
};

WsLayout ws_layout(int batch, int Hq, int D, int S) {
    const size_t rows = static_cast<size_t>(batch) * Hq * S;
    WsLayout w;
    w.o = 0;
    w.m = align256(rows * D * sizeof(float));
    w.l = w.m + align256(rows * sizeof(float));
    w.total = w.l + align256(rows * sizeof(float));
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

template <int D>
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Geo<D>::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(p.num_splits, p.H, p.B);
    decode_split_kernel<D><<<grid, kDecThreads, Geo<D>::SMEM, s>>>(p);
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
    const SplitPlan plan = plan_splits(batch, layout->num_kv_heads, max_pages_per_seq,
                                       layout->page_size, max_num_splits);
    return ws_layout(batch, num_q_heads, layout->head_dim, plan.num_splits).total;
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
    if (batch > 65535 || layout->num_kv_heads > 65535 || num_q_heads > 65535)
        return NVFP4KV_ERR_UNSUPPORTED;
    const int D = layout->head_dim;
    const SplitPlan plan = plan_splits(batch, layout->num_kv_heads, max_pages_per_seq,
                                       layout->page_size, max_num_splits);
    const WsLayout wl = ws_layout(batch, num_q_heads, D, plan.num_splits);
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
    p.gv = v_global_scale;
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.part_o = reinterpret_cast<float*>(ws + wl.o);
    p.part_m = reinterpret_cast<float*>(ws + wl.m);
    p.part_l = reinterpret_cast<float*>(ws + wl.l);
    p.status = status;
    p.B = batch;
    p.Hq = num_q_heads;
    p.H = layout->num_kv_heads;
    p.G = num_q_heads / layout->num_kv_heads;
    p.T = layout->page_size;
    p.pool_pages = pool_pages;
    p.max_pages = max_pages_per_seq;
    p.num_splits = plan.num_splits;
    p.stages_per_split = plan.stages_per_split;
    p.sm_scale = sm_scale;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (D) {
    case 64: e = launch_decode<64>(p, s); break;
    case 128: e = launch_decode<128>(p, s); break;
    default: e = launch_decode<256>(p, s); break;
    }
    if (e != cudaSuccess) return NVFP4KV_ERR_CUDA;

    CombineParams cp{};
    cp.part_o = p.part_o;
    cp.part_m = p.part_m;
    cp.part_l = p.part_l;
    cp.seq_lens = seq_lens;
    cp.gv = v_global_scale;
    cp.out = static_cast<uint16_t*>(out);
    cp.lse = lse;
    cp.Hq = num_q_heads;
    cp.D = D;
    cp.T = layout->page_size;
    cp.max_pages = max_pages_per_seq;
    cp.num_splits = plan.num_splits;
    cp.stages_per_split = plan.stages_per_split;
    combine_kernel<<<dim3(num_q_heads, batch), 128, 0, s>>>(cp);
    return launch_status();
}
