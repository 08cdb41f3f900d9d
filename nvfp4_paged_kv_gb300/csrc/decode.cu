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
//  * one CTA per (sequence, KV head, split) of 4 warps; a split is a run of 64-token stages and
//    warp w owns the 16-token tiles w, w+4, w+8, ... of it. Each warp streams its own tiles
//    through a private 4-slot shared-memory ring with asynchronous copies (cp.async, 16 bytes
//    per lane, completion per warp by wait_group): packed K rows, token-pair packed V rows and
//    both scale pools of a tile are four contiguous runs of its page. The warps never wait for
//    one another until the final merge, so each keeps three tiles in flight behind the one it
//    computes. V rows land XOR-swizzled by 16-byte chunk so the fragment reads hit distinct banks.
//  * S^T = K^ Q^T runs on the tensor cores with tokens as M = 16 and the GQA query group as
//    N = 8 (mma.sync m16n8k16, FP16 in, FP32 accumulate). K is stored dim-pair packed, so every
//    converted byte (cvt.rn.f16x2.e2m1x2) is one A-register: two adjacent head dims of one
//    token, exact in FP16, times its E4M3 block scale (exact). Q is brought into FP16 exactly by
//    a per-head power of two; head dims inside a k-step are permuted identically in K and Q.
//  * online softmax in the log2 domain, column maxima by warp shuffles; the running maximum
//    moves only when it grows by more than 2^8, so accumulator rescaling is rare. P^T moves from
//    the score layout to the B-operand layout with movmatrix.
//  * O^T += V^^T P^T with head dims as M: V is stored token-pair packed, so every converted byte
//    is one A-register (one head dim of two adjacent tokens) times the pair's two block scales.
//  * the 4 warps merge (max, sum, output) in shared memory and the CTA writes one partial per
//    (sequence, query head, split); a second kernel merges the splits by log-sum-exp and writes
//    the BF16 output and the natural-log LSE.
// Bytes per (token, KV head) at head_dim 128: 64 + 8 (K) + 64 + 8 (V) = 144.
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_util.h"

namespace nvfp4kv {
namespace {

constexpr int kWarps = 4;
constexpr int kDecThreads = kWarps * 32;
constexpr int kStageTokens = 64;  // split granularity (4 warps x 16-token tiles)
constexpr int kSlots = 4;         // tiles per warp ring
constexpr int kMaxGroup = 8;
constexpr int kMaxSplits = 64;
constexpr int kPageBuf = 256; // page ids of a split kept in shared memory
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Geo {
    static constexpr int NB = D / 16;            // blocks (= scales) per token row
    static constexpr int TK = 16 * D / 2;         // packed K rows of a 16-token tile
    static constexpr int TV = 8 * D;              // token-pair V rows of a tile (8 pairs)
    static constexpr int TS = 16 * NB;            // one scale pool of a tile
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = TK;
    static constexpr int KS_OFF = TK + TV;
    static constexpr int VS_OFF = TK + TV + TS;
    static constexpr int SLOT = TK + TV + 2 * TS;  // 18 D bytes
    static constexpr int RING = kSlots * SLOT;     // per warp
    static constexpr int SMEM = kWarps * RING;
    static constexpr int KSTEPS = D / 16;          // k-steps of S^T = K Q^T
    static constexpr int CHUNK = D / 8;            // bytes of a row one quad lane owns
    static constexpr int CW = CHUNK / 4;           // ... as 32-bit words
    static constexpr int VCH = D / 16;             // 16-byte chunks per V pair row
    static constexpr int SWZ = (VCH < 8 ? VCH : 8) - 1;  // chunk XOR mask
    static_assert(kWarps * kMaxGroup * D * 4 <= SMEM, "merge buffer must fit in the rings");
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

// Shared-memory offset of byte x of token-pair row pr of a tile's V rows: 16-byte chunks are
// XOR-swizzled by the row so that the 4 lanes of a quad (rows c and c+4) hit distinct banks.
template <int D>
__device__ __forceinline__ uint32_t v_swz(int pr, int x) {
    return static_cast<uint32_t>(pr * D + ((((x >> 4) ^ (pr & Geo<D>::SWZ))) << 4) + (x & 15));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kDecThreads, D == 256 ? 3 : 5)
    decode_split_kernel(const DecodeParams p) {
    using G_ = Geo<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ float red_m[kWarps][kMaxGroup];
    __shared__ float red_l[kWarps][kMaxGroup];
    __shared__ int page_ids[kPageBuf];

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
    const int tok_begin = st_begin * kStageTokens;
    const int tok_end = min(st_end * kStageTokens, L);
    const int G = p.G;
    const int64_t part_row = (static_cast<int64_t>(b) * p.Hq + h * G) * p.num_splits + split;

    // The split's page ids, read once here instead of on each tile's critical path.
    const int first_page = tok_begin / p.T;
    const int end_page = (tok_end + p.T - 1) / p.T;
    const int32_t* pt_row = p.page_table + static_cast<int64_t>(b) * p.max_pages;
    for (int i = tid; i < end_page - first_page && i < kPageBuf; i += kDecThreads)
        page_ids[i] = __ldg(pt_row + first_page + i);
    __syncthreads();
    auto page_of = [&](int pidx) {
        const int k = pidx - first_page;
        const int pg = (k < kPageBuf) ? page_ids[k] : __ldg(pt_row + pidx);
        return (pg >= 0 && pg < p.pool_pages) ? pg : -1;
    };

    // ---------------------------------------------------------------- this warp's tiles
    // tile k of this warp covers tokens tok_begin + 16 (4k + warp) .. +15 (one page: T % 16 == 0)
    const int n_tiles = max(0, (tok_end - tok_begin - 16 * warp + 16 * kWarps - 1) / (16 * kWarps));
    const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(smem)) + warp * G_::RING;
    // Loop-invariant per-lane chunk offsets: this lane copies 16-byte chunks j = lane + 32 i of
    // the tile's K rows and V rows (V chunks land XOR-swizzled) and, for lanes < 2 NB, one chunk
    // of a scale pool. K rows, V rows and the two scale pools of a tile share one base offset
    // each: row0 * D/2 bytes for the data, row0 * NB for the scales.
    uint32_t v_dst[D / 64];
#pragma unroll
    for (int i = 0; i < D / 64; ++i) {
        const int j = lane + 32 * i;
        const int pr = j / G_::VCH, cj = j - pr * G_::VCH;
        v_dst[i] = G_::V_OFF + pr * D + 16 * (cj ^ (pr & G_::SWZ));
    }
    const bool sc_lane = lane < 2 * G_::NB;
    const uint8_t* sc_pool = (lane < G_::NB) ? p.ks : p.vs;
    const uint32_t sc_dst = (lane < G_::NB) ? G_::KS_OFF + 16 * lane : G_::VS_OFF + 16 * (lane - G_::NB);
    const uint32_t sc_src = 16 * ((lane < G_::NB) ? lane : lane - G_::NB);
    // Page index / slot of this warp's next tile to issue, advanced by 64 tokens per tile
    // without divisions (T >= 16, so at most 4 page steps per tile).
    struct TilePos {
        int pidx, off;
        __device__ __forceinline__ void advance(int T) {
            off += 16 * kWarps;
            while (off >= T) {
                off -= T;
                ++pidx;
            }
        }
    };
    const int t_first = tok_begin + 16 * warp;
    TilePos ipos{t_first / p.T, t_first - (t_first / p.T) * p.T};  // next tile to issue
    TilePos cpos = ipos;                                              // next tile to consume
    const int64_t head_rows = static_cast<int64_t>(h) * p.T;          // row offset of head h
    const int64_t page_rows = static_cast<int64_t>(p.H) * p.T;        // rows per page
    auto issue_tile = [&](int k) {
        if (k < n_tiles) {
            const int page = page_of(ipos.pidx);
            if (page >= 0) {
                const int64_t row0 = page * page_rows + head_rows + ipos.off;
                const uint32_t slot = ring + (k % kSlots) * G_::SLOT;
                const int64_t doff = row0 * (D / 2);
                const uint8_t* ksrc = p.kd + doff + 16 * lane;
                const uint8_t* vsrc = p.vd + doff + 16 * lane;
#pragma unroll
                for (int i = 0; i < D / 64; ++i) {
                    cp_async16(slot + G_::K_OFF + 16 * lane + 512 * i, ksrc + 512 * i);
                    cp_async16(slot + v_dst[i], vsrc + 512 * i);
                }
                if (sc_lane) cp_async16(slot + sc_dst, sc_pool + row0 * G_::NB + sc_src);
            } else if (lane == 0) {
                flag_status(p.status, NVFP4KV_STATUS_PAGE_OOB);
            }
            ipos.advance(p.T);
        }
        cp_async_commit();
    };
#pragma unroll
    for (int k = 0; k < kSlots - 1; ++k) issue_tile(k);

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

    // V rows of this lane: chunk rho of every token pair; M-tile m row r <-> head dim
    // rho*D/8 + 2m, row r+8 <-> that dim + 1 (rho spreads the quad lanes over the banks).
    const int rho = (r >> 1) | ((r & 1) << 2);
    float o[G_::KSTEPS][4];
#pragma unroll
    for (int m = 0; m < G_::KSTEPS; ++m)
#pragma unroll
        for (int k = 0; k < 4; ++k) o[m][k] = 0.0f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;

    // ---------------------------------------------------------------- main loop
    for (int kt = 0; kt < n_tiles; ++kt) {
        issue_tile(kt + kSlots - 1);    // into the slot tile kt-1 used (released below)
        cp_async_wait<kSlots - 1>();    // this lane's copies of tile kt are done ...
        __syncwarp();                   // ... and so are the other lanes'
        const int t0 = tok_begin + 16 * (kWarps * kt + warp);
        uint32_t tmask = 0u;
        if (page_of(cpos.pidx) >= 0) {
            const int valid = min(16, L - t0);
            tmask = (valid >= 16) ? 0xFFFFu : ((1u << valid) - 1u);
        }
        cpos.advance(p.T);
        if (tmask != 0u) {
            const uint32_t st = ring + (kt % kSlots) * G_::SLOT;
            const int row0 = r;
            const int row1 = r + 8;
            // ---- S^T = K^ Q^T (tokens x query heads)
            uint32_t kw0[G_::CW], kw1[G_::CW];
            lds_words(kw0, st + G_::K_OFF + row0 * (D / 2) + c * G_::CHUNK);
            lds_words(kw1, st + G_::K_OFF + row1 * (D / 2) + c * G_::CHUNK);
            // FP16 (s, s) of the lane's D/64 blocks in rows row0 / row1: the scale byte is
            // duplicated by an integer multiply, then converted as an E4M3 pair
            uint32_t ks0[D / 64], ks1[D / 64];
#pragma unroll
            for (int q = 0; q < D / 64; ++q) {
                ks0[q] = e4m3x2_to_f16x2(lds_u8(st + G_::KS_OFF + row0 * G_::NB + c * (D / 64) + q) *
                                         0x0101u);
                ks1[q] = e4m3x2_to_f16x2(lds_u8(st + G_::KS_OFF + row1 * G_::NB + c * (D / 64) + q) *
                                         0x0101u);
            }
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int q = 0; q < G_::CW; ++q) {
                uint32_t c0[4], c1[4];
                e2m1x8_to_f16x2x4(kw0[q], c0);
                e2m1x8_to_f16x2x4(kw1[q], c1);
#pragma unroll
                for (int hk = 0; hk < 2; ++hk) {
                    const int k = 2 * q + hk;  // k-step: bytes 2k, 2k+1 of the lane's chunk
                    const int blk = k / 4;     // block of the lane's chunk
                    uint32_t a[4];
                    a[0] = h2_mul(c0[2 * hk], ks0[blk]);
                    a[1] = h2_mul(c1[2 * hk], ks1[blk]);
                    a[2] = h2_mul(c0[2 * hk + 1], ks0[blk]);
                    a[3] = h2_mul(c1[2 * hk + 1], ks1[blk]);
                    mma_f16_16816(acc, a, qf[k][0], qf[k][1]);
                }
            }

            // ---- online softmax (log2 domain), columns = query heads 2c, 2c+1
            float x0 = acc[0] * cs0, x1 = acc[1] * cs1, x2 = acc[2] * cs0, x3 = acc[3] * cs1;
            if (tmask != 0xFFFFu) {
                if (!((tmask >> r) & 1u)) x0 = x1 = -INFINITY;
                if (!((tmask >> (r + 8)) & 1u)) x2 = x3 = -INFINITY;
            }
            // column maxima over the 16 tokens, both columns in one FP16 pair (the running
            // maximum only has to be close to the true one: p = 2^(x - m) stays below 2^8)
            __half2 hm = __floats2half2_rn(fmaxf(x0, x2), fmaxf(x1, x3));
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                const uint32_t u =
                    __shfl_xor_sync(0xFFFFFFFFu, *reinterpret_cast<const uint32_t*>(&hm), off);
                hm = __hmax2(hm, *reinterpret_cast<const __half2*>(&u));
            }
            float mx0 = __low2float(hm), mx1 = __high2float(hm);
            if (__any_sync(0xFFFFFFFFu, fmaxf(mx0, mx1) > 65000.0f)) {
                // scores beyond the FP16 range: reduce in fp32 instead
                mx0 = fmaxf(x0, x2);
                mx1 = fmaxf(x1, x3);
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
            const float p0 = ex2_approx(x0 - m0), p1 = ex2_approx(x1 - m1);
            const float p2 = ex2_approx(x2 - m0), p3 = ex2_approx(x3 - m1);
            l0 += p0 + p2;
            l1 += p1 + p3;
            // P^T (tokens x heads) -> B operand (k = tokens, n = heads)
            const uint32_t pb0 = movmatrix_trans(pack_f16x2(p0, p1));
            const uint32_t pb1 = movmatrix_trans(pack_f16x2(p2, p3));

            // ---- O^T += V^^T P^T. Lane pairs: pr0 (tokens 2c, 2c+1), pr1 (tokens 2c+8, 2c+9)
            const int pr0 = c, pr1 = c + 4;
            uint32_t keep0 = 0xFFFFFFFFu, keep1 = 0xFFFFFFFFu;
            if (tmask != 0xFFFFu) {
                keep0 = (((tmask >> (2 * c)) & 1u) ? 0x0000FFFFu : 0u) |
                        (((tmask >> (2 * c + 1)) & 1u) ? 0xFFFF0000u : 0u);
                keep1 = (((tmask >> (2 * c + 8)) & 1u) ? 0x0000FFFFu : 0u) |
                        (((tmask >> (2 * c + 9)) & 1u) ? 0xFFFF0000u : 0u);
            }
            // the lane's chunk covers head dims rho*D/8 .. +D/8-1: blocks (rho*D/8)/16 ...
            constexpr int kBlkPerChunk = (D / 8 + 15) / 16;
            uint32_t vsc0[kBlkPerChunk], vsc1[kBlkPerChunk];
#pragma unroll
            for (int q = 0; q < kBlkPerChunk; ++q) {
                const int blk = (rho * (D / 8)) / 16 + q;
                vsc0[q] = e4m3x2_to_f16x2(lds_u16(st + G_::VS_OFF + pr0 * 2 * G_::NB + 2 * blk));
                vsc1[q] = e4m3x2_to_f16x2(lds_u16(st + G_::VS_OFF + pr1 * 2 * G_::NB + 2 * blk));
                if (tmask != 0xFFFFu) {
                    vsc0[q] &= keep0;
                    vsc1[q] &= keep1;
                }
            }
            uint32_t vw0[G_::CW], vw1[G_::CW];
#pragma unroll
            for (int q = 0; q < G_::CW; q += (G_::CW >= 4 ? 4 : G_::CW)) {
                const int x = rho * G_::CHUNK + 4 * q;  // logical byte of the chunk piece
                uint32_t t0[G_::CW >= 4 ? 4 : G_::CW], t1[G_::CW >= 4 ? 4 : G_::CW];
                lds_words(t0, st + G_::V_OFF + v_swz<D>(pr0, x));
                lds_words(t1, st + G_::V_OFF + v_swz<D>(pr1, x));
#pragma unroll
                for (int i = 0; i < (G_::CW >= 4 ? 4 : G_::CW); ++i) {
                    vw0[q + i] = t0[i];
                    vw1[q + i] = t1[i];
                }
            }
#pragma unroll
            for (int q = 0; q < G_::CW; ++q) {
                uint32_t c0[4], c1[4];
                e2m1x8_to_f16x2x4(vw0[q], c0);
                e2m1x8_to_f16x2x4(vw1[q], c1);
#pragma unroll
                for (int hm = 0; hm < 2; ++hm) {
                    const int m = 2 * q + hm;            // M-tile: bytes 2m, 2m+1 of the chunk
                    const int sq = (2 * m) / 16;         // block of that byte within the chunk
                    uint32_t a[4];
                    a[0] = h2_mul(c0[2 * hm], vsc0[sq]);
                    a[1] = h2_mul(c0[2 * hm + 1], vsc0[sq]);
                    a[2] = h2_mul(c1[2 * hm], vsc1[sq]);
                    a[3] = h2_mul(c1[2 * hm + 1], vsc1[sq]);
                    mma_f16_16816(o[m], a, pb0, pb1);
                }
            }
        }
        __syncwarp();                   // every lane is done reading the slot before it refills
    }
    cp_async_wait<0>();

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
    __syncthreads();  // every warp is done with its ring: the rings hold the merge buffer
    float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        M0 = fmaxf(M0, red_m[w][2 * c]);
        M1 = fmaxf(M1, red_m[w][2 * c + 1]);
    }
    const float f0 = (m0 == -INFINITY) ? 0.0f : ex2_approx(m0 - M0);
    const float f1 = (m1 == -INFINITY) ? 0.0f : ex2_approx(m1 - M1);
    float* so = reinterpret_cast<float*>(smem);  // [kWarps][kMaxGroup][D], over the rings
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
    __shared__ float red[2][4];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // one split per thread (n_act <= 64): maximum, then weights and weighted sum of l
    const float ms = (tid < n_act) ? p.part_m[row + tid] : -INFINITY;
    const float ls = (tid < n_act) ? p.part_l[row + tid] : 0.0f;
    float M = ms;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    if (lane == 0) red[0][warp] = M;
    __syncthreads();
    M = fmaxf(fmaxf(red[0][0], red[0][1]), fmaxf(red[0][2], red[0][3]));
    const float w = (ms == -INFINITY) ? 0.0f : exp2f(ms - M);
    if (tid < kMaxSplits) w_s[tid] = w;
    float lsum = w * ls;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, o);
    if (lane == 0) red[1][warp] = lsum;
    __syncthreads();
    lsum = red[1][0] + red[1][1] + red[1][2] + red[1][3];
    const float inv_l = (lsum > 0.0f) ? __ldg(p.gv) / lsum : 0.0f;
    if (tid == 0 && p.lse)
        p.lse[static_cast<int64_t>(b) * p.Hq + qh] =
            (lsum > 0.0f) ? (M + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
    for (int d = tid; d < p.D; d += blockDim.x) {
        float acc = 0.0f;
        for (int s = 0; s < n_act; ++s) {
            const float ws = w_s[s];
            if (ws != 0.0f) acc += ws * p.part_o[(row + s) * p.D + d];
        }
        const __nv_bfloat16 yb = __float2bfloat16_rn(acc * inv_l);
        p.out[(static_cast<int64_t>(b) * p.Hq + qh) * p.D + d] =
            *reinterpret_cast<const uint16_t*>(&yb);
    }
}

// ------------------------------------------------------------------------------------------
// Host side: split heuristic, workspace carving, V tensor map
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
