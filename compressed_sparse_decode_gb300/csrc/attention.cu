// attention.cu -- sink-merged split-precision attention on the tensor cores
// over [top-k entries] ++ [SWA window] (CSA) or [all visible entries] ++
// [SWA window] (HCA) ("DSV4 Inference Kernel" README, Architecture: one
// 512-d latent per entry serves as key and value of all 128 heads, sink
// weights merge the sparse and SWA terms; "DSV4 Audit", sections A3 and B1:
// the FP8 nope dims are fed to attention without a BF16 copy in memory).
//
// For head h over candidates j (x_j the dequantised latent):
//   z_j = scale * q_h . x_j,  o_h = sum_j e^{z_j-M} x_j / (e^{sink_h-M} + sum_j e^{z_j-M}),
//   lse_h = M + ln(den),  M = max(sink_h, max_j z_j).
//
// Work unit = (query token, candidate split, output half): two CTAs share a
// (query, split); CTA r writes latent dims [256 r, 256 r + 256) of the output.
// O (128 heads x 256 fp32) fills half of the tensor memory, so one CTA cannot
// hold all 512 output dims; instead of exchanging partial scores between the
// two halves (the SM-to-SM network moves only a few bytes per cycle), both
// CTAs compute the full scores -- QK with K = 512 -- and run the softmax on
// them, then each accumulates its own half of PV. Per CTA:
//   * Q dims 0..383 live in TMEM (BF16 pairs) and dims 384..511 in shared
//     memory; QK(j) = Q X_j^T (tcgen05.mma kind::f16, M = 128 heads, N = 64
//     candidates, K = 512) lands in the TMEM score buffer. (A second score
//     buffer would push Q operands into shared memory, whose bandwidth the
//     QK reads already share with the dequantised stores.)
//   * P (BF16, K-major rows in the 128-byte swizzle) is the A operand of
//     PV: O += P X_j[:, half] (M = 128, N = 256, K = 64); O stays in TMEM.
//   * Candidate records are copied straight from the FP8/BF16 caches into
//     shared staging (16-byte cp.async, one chunk ahead, block-table
//     resolved) and dequantised there to BF16 (code x block multiplier);
//     there is no dequantised copy in HBM. X is kept as two halves, dims
//     0..255 ("lo") and 256..511 ("hi"), each double-buffered: the half this
//     CTA does not output is released as soon as QK has read it, its own half
//     after PV.
// Warps: a record-pointer producer, the MMA issuer (and TMEM owner), 8
// load + dequantise warps and 4 softmax / epilogue warps (thread = head); see
// warp_role for the placement on the four schedulers. The running max
// is rescaled lazily (only when it grows by more than 2^8), in the log2
// domain. With one split per query the CTAs write the BF16 output and LSE;
// with several, each split writes a normalised BF16 partial and (max, sum),
// and a combine kernel folds the splits and the sink. Every wait is bounded.
#include <cuda.h>

#include <mutex>
#include <type_traits>

#include <cmath>

#include "common.cuh"
#include "ptx.cuh"

namespace csa {

namespace {

constexpr int kChunk = 64;                  // candidates per chunk
constexpr int kHalf = 256;                  // output latent dims per CTA
constexpr int kRopePairs = 32;              // rope dims 448..511 as (x, y) pairs
constexpr int kFp4RowBytes = kDim / 2;      // E2M1 output bytes per head
constexpr int kQTmemDims = 384;             // Q dims held in TMEM; the rest in shared memory
constexpr int kPtrRing = 8;                 // chunks of resolved record pointers
constexpr int kIdxAhead = 4;                // chunks ahead whose candidate indices the producer has loaded
constexpr int kThreads = 480;               // 15 warps (roles: see warp_role)
constexpr int kAtom = kChunk * 128;         // one 64-dim column block of X: 64 rows x 128 B
constexpr int kXHalfBytes = 4 * kAtom;      // 256 dims, 32 KB
constexpr int kOwnBufs = 2;                 // buffers of the X half a CTA outputs (held until PV)
constexpr int kOthBufs = 2;                 // buffers of the other half (held until QK)
constexpr int kQAtom = kHeads * 128;        // one 64-dim column block of Q: 128 rows x 128 B
constexpr int kConvWarps = 8;               // load + dequantise warps
constexpr int kLoPieces = 4;                // per thread: codes 0..255 of a record in 16-byte pieces, 4 threads a row
constexpr int kHiPieces = 5;                // per thread: codes 256..447 and the rope dims (3 + 2 pieces)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazy = 8.f;                // rescale only when the max grows by > 2^8

constexpr uint32_t kColQ = 0;    // 192 columns: Q dims 0..383, BF16 pairs
constexpr uint32_t kColS = 192;  // 64 columns: scores
constexpr uint32_t kColO = 256;  // 256 columns: O half, fp32
constexpr uint32_t kTmemCols = 512;

// Raw bytes of one half of a chunk's records. Thread t (row t / 4, quarter
// c = t % 4) copies the half's 16-byte pieces c, c + 4, c + 8, ... into
// piece[i][t] (consecutive threads touch consecutive words, in global and in
// shared memory) and, for c = 0, the row's four block multipliers into
// scale[row]. Lo: codes 0..255 (16 pieces a row); hi: codes 256..447 then
// the 64 BF16 rope dims (20 pieces a row).
template <int kPieces>
struct HalfStage {
    uint4 piece[kPieces][4 * kChunk];
    float4 scale[kChunk];
};

// x_own / x_oth hold 64 candidates x 256 dims of a chunk (BF16, K-major rows
// of 128 B in the 128-byte swizzle, 4 column blocks of 64 dims): the half of
// the latent this CTA outputs, and the other half; qs holds Q dims 384..511
// (2 column blocks); p holds P (128 heads x 64 candidates, BF16, swizzled
// 128-byte rows), the A operand of PV.
struct AttSmem {
    alignas(1024) uint8_t x_own[kOwnBufs][kXHalfBytes];
    alignas(1024) uint8_t x_oth[kOthBufs][kXHalfBytes];
    alignas(1024) uint8_t qs[2 * kQAtom];
    alignas(1024) uint8_t p[kHeads * 128];
    alignas(16) HalfStage<kLoPieces> stage_lo;
    alignas(16) HalfStage<kHiPieces> stage_hi;
    const uint8_t *rec[kPtrRing][kChunk];       // record of each candidate (nullptr: skipped)
    uint64_t vmask[kPtrRing];
    uint64_t ptr_full[kPtrRing], ptr_empty[kPtrRing];
    uint64_t own_full[kOwnBufs], own_empty[kOwnBufs], oth_full[kOthBufs], oth_empty[kOthBufs];
    uint64_t s_full, s_free, p_full;
    uint64_t o_done[2], o_final, q_ready, mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

static_assert(sizeof(AttSmem) + 1024 <= 232448, "shared memory plan exceeds the per-CTA limit");

// Output epilogue: inverse RoPE of the rope dims at the query position and/or
// E2M1 output with one multiplier per 128 dims. Applied where the final
// output is formed: the attention kernel with one split, else the combine.
struct EpiParams {
    uint8_t *out_fp4;      // null: BF16 output
    float *out_fp4_scale;  // [rows, 128, 4]
    int inv_rope;
    double rope_freq[kRopePairs];  // radians per position of rope pair i
};

struct AttParams {
    const __nv_bfloat16 *q;
    const float *sink;
    float scale_log2;  // softmax scale * log2(e)
    CacheView comp;
    const uint8_t *ring;
    int R, W;
    const int32_t *topk_idx, *topk_cnt, *n_comp, *q_pos;
    int m_hca, hca, T, k, n_split;
    __nv_bfloat16 *out;
    float *lse;
    __nv_bfloat16 *part_o;  // [rows, n_split, 128, 512] BF16 (n_split > 1)
    float2 *part_ml;        // [rows, n_split, 128] (max, sum) in log2 units
    int *err;
    uint64_t wait_ns;  // limit of each bounded wait (drains keep kDrainWaitNs)
    EpiParams epi;
};

struct Unit {
    int r, b, split, p, n_sel, j0, cb, ce, n_chunks;
};

__device__ __forceinline__ Unit make_unit(const AttParams &P) {
    Unit u;
    const int pair = blockIdx.x >> 1;
    u.r = pair / P.n_split;
    u.split = pair % P.n_split;
    u.b = u.r / P.T;
    u.p = __ldg(P.q_pos + u.r);
    if (P.hca) {
        u.n_sel = visible_entries(u.p, P.m_hca, __ldg(P.n_comp + u.b), P.comp.seq_capacity);
    } else {
        const int c = __ldg(P.topk_cnt + u.r);
        u.n_sel = c < 0 ? 0 : (c > P.k ? P.k : c);
    }
    u.j0 = max(0, u.p - P.W + 1);
    const int nswa = u.p >= 0 ? u.p - u.j0 + 1 : 0;
    const int n = u.n_sel + nswa;
    const int per = ((n + P.n_split - 1) / P.n_split + kChunk - 1) / kChunk * kChunk;
    u.cb = min(n, u.split * per);
    u.ce = min(n, u.cb + per);
    u.n_chunks = (u.ce - u.cb + kChunk - 1) / kChunk;
    return u;
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// 8 E4M3 codes (two 32-bit words) times a multiplier -> 8 BF16 values (uint4).
__device__ __forceinline__ uint4 dequant8(uint32_t w0, uint32_t w1, float s) {
    uint32_t out[4];
    const uint32_t w[2] = {w0, w1};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float2 a = e4m3x2_to_float2(static_cast<uint16_t>(w[i] & 0xFFFFu));
        const float2 c = e4m3x2_to_float2(static_cast<uint16_t>(w[i] >> 16));
        out[2 * i] = bf16x2_bits(a.x * s, a.y * s);
        out[2 * i + 1] = bf16x2_bits(c.x * s, c.y * s);
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// 16-byte chunk cc of row `row` of a swizzled block of 128-byte rows.
__device__ __forceinline__ uint4 *sw128(uint8_t *block, int row, int cc) {
    return reinterpret_cast<uint4 *>(block + row * 128 + ((cc ^ (row & 7)) << 4));
}

// Pipeline per chunk j (64 candidates), per CTA (b = j % 2; "oth" is the half
// of X this CTA does not output, "own" the one it does):
//   producer:  record pointers and validity mask of chunk j -> rec[j % 8]
//   dequant:   oth(j) from the staging into x_oth[j % 2] (after QK(j-2)
//              freed it), then copies oth(j+1) into the staging; the same for
//              own(j) into x_own[j % 2] (after PV(j-2) freed it)
//   MMA:       QK(j+1) -> S once the softmax has read S(j) (oth K-steps, then
//              own), then PV(j) = P X(j)[:, own] -> O once P(j) is ready
//   softmax:   reads S(j) and the mask, releases S, writes P(j) once PV(j-1)
//              is done
// QK(j) completion frees x_oth[j % 2]; PV(j) completion frees x_own[j % 2] and P.
// Warp roles. A warp's scheduler is warp % 4, and the softmax warps must
// cover the four TMEM lane quarters (warp % 4 = 0..3). The MMA issuer shares
// its scheduler only with the light pointer producer and one softmax warp:
// tcgen05.mma issue slows down markedly next to two dequantise warps.
//   scheduler 0: dequantise 0, 4, 8   softmax 12
//   scheduler 1: MMA 1, producer 5     softmax 13   (warp 9 idle)
//   scheduler 2: dequantise 2, 6, 10  softmax 14
//   scheduler 3: dequantise 3, 7      softmax 11
enum WarpRole { kRoleProducer, kRoleMma, kRoleConvert, kRoleSoftmax, kRoleIdle };
__device__ __forceinline__ int warp_role(int w) {
    if (w == 5) return kRoleProducer;
    if (w == 1) return kRoleMma;
    if (w == 9) return kRoleIdle;
    return w >= 11 ? kRoleSoftmax : kRoleConvert;
}
// index 0..7 of a dequantise warp
__device__ __forceinline__ int convert_index(int w) { return w == 0 ? 0 : (w < 5 ? w - 1 : (w < 9 ? w - 2 : 7)); }

__global__ void __launch_bounds__(kThreads, 1)
attention_tc_kernel(const AttParams P) {
    extern __shared__ uint8_t smem_raw[];
    AttSmem &s = *reinterpret_cast<AttSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int role = warp_role(warp);
    const int rank = blockIdx.x & 1;  // output half: 0 = lo, 1 = hi
    volatile int *abort = &s.abort_flag;

    // The query rows are an input, not produced by the kernels before this one:
    // their prefetch into L2 starts at once, before the wait for the top-k
    // (the prefetch is a hint; the loads themselves follow the wait).
    if (threadIdx.x == 32 * 9) {  // the otherwise idle warp
        const uint8_t *qrow = reinterpret_cast<const uint8_t *>(P.q) +
                              (size_t)((blockIdx.x >> 1) / P.n_split) * kHeads * kDim * sizeof(__nv_bfloat16);
#pragma unroll
        for (int i = 0; i < 8; ++i) ptx::prefetch_l2_bulk(qrow + i * 16384, 16384u);
        static_assert(kHeads * kDim * sizeof(__nv_bfloat16) == 8 * 16384, "one query's rows are 8 x 16 KB");
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kPtrRing; ++i) {
            ptx::mbar_init(&s.ptr_full[i], 32);  // every producer lane has written its pointers
            ptx::mbar_init(&s.ptr_empty[i], kConvWarps + 4);  // every dequantise and softmax warp has read them
        }
        for (int i = 0; i < kOwnBufs; ++i) {
            ptx::mbar_init(&s.own_full[i], kConvWarps);
            ptx::mbar_init(&s.own_empty[i], 1);
        }
        for (int i = 0; i < kOthBufs; ++i) {
            ptx::mbar_init(&s.oth_full[i], kConvWarps);
            ptx::mbar_init(&s.oth_empty[i], 1);
        }
        ptx::mbar_init(&s.s_full, 1);
        ptx::mbar_init(&s.s_free, 4);
        ptx::mbar_init(&s.p_full, 4);
        for (int i = 0; i < 2; ++i) ptx::mbar_init(&s.o_done[i], 1);  // PV of a chunk of this parity is done
        ptx::mbar_init(&s.o_final, 1);
        ptx::mbar_init(&s.q_ready, 4);
        ptx::mbar_init(&s.mma_done, 1);
        s.abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(&s.tmem_base, kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = s.tmem_base;
    ptx::griddep_wait();               // the top-k output (previous kernel in the stream) is complete
    const Unit u = make_unit(P);

    auto fail = [&]() {
        report_error(P.err, CSA_ERR_TIMEOUT);
        *abort = 1;
    };
    auto wait = [&](uint64_t *bar, uint32_t parity) {
        return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, abort, P.wait_ns)) != 0;
    };

    if (role == kRoleProducer) {
        // ------------------------------------------------------------ record-pointer producer
        // Candidate indices are loaded kIdxAhead chunks ahead; lane L holds
        // candidates L and L + 32 of a chunk. A rolled loop keeps this warp's
        // code small: it shares an instruction cache with the MMA issuer.
        auto load_raw = [&](int jj, int &r0, int &r1) {
            const int i0 = u.cb + jj * kChunk + lane, i1 = i0 + 32;
            const int32_t *src = P.topk_idx + (size_t)u.r * P.k;
            r0 = (!P.hca && i0 < u.ce && i0 < u.n_sel) ? __ldg(src + i0) : i0;
            r1 = (!P.hca && i1 < u.ce && i1 < u.n_sel) ? __ldg(src + i1) : i1;
        };
        int ahead[kIdxAhead][2];
#pragma unroll
        for (int q = 0; q < kIdxAhead; ++q)
            if (q < u.n_chunks) load_raw(q, ahead[q][0], ahead[q][1]);
        bool ok = true;
#pragma unroll 1
        for (int j = 0; j < u.n_chunks && ok; ++j) {
            const int raw[2] = {ahead[0][0], ahead[0][1]};
#pragma unroll
            for (int q = 0; q + 1 < kIdxAhead; ++q) {
                ahead[q][0] = ahead[q + 1][0];
                ahead[q][1] = ahead[q + 1][1];
            }
            if (j + kIdxAhead < u.n_chunks) load_raw(j + kIdxAhead, ahead[kIdxAhead - 1][0], ahead[kIdxAhead - 1][1]);
            const int pr = j % kPtrRing;
            if (!wait(&s.ptr_empty[pr], ((j / kPtrRing) & 1) ^ 1)) { fail(); ok = false; break; }
            bool valid[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int i = u.cb + j * kChunk + e * 32 + lane;
                const uint8_t *rec = nullptr;
                if (i < u.ce) {
                    if (i < u.n_sel) {
                        const int64_t ri = record_index(P.comp, u.b, raw[e]);
                        if (ri >= 0) rec = P.comp.base + ri * kRecBytes;
                        else if (rank == 0) report_error(P.err, CSA_ERR_BAD_INDEX);
                    } else {
                        const int pos = u.j0 + (i - u.n_sel);
                        rec = P.ring + ((int64_t)u.b * P.R + pos % P.R) * kRecBytes;
                    }
                }
                valid[e] = rec != nullptr;
                s.rec[pr][e * 32 + lane] = rec;
            }
            const uint32_t m0 = __ballot_sync(0xffffffffu, valid[0]);
            const uint32_t m1 = __ballot_sync(0xffffffffu, valid[1]);
            if (lane == 0) s.vmask[pr] = (uint64_t)m0 | ((uint64_t)m1 << 32);
            __syncwarp();
            ptx::mbar_arrive(&s.ptr_full[pr]);
        }
    } else if (role == kRoleMma) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t kIdescQK = ptx::idesc_f32acc(1, 1, 128, kChunk);
        constexpr uint32_t kIdescPV = ptx::idesc_f32acc(1, 1, 128, kHalf, 1);
        bool ok = u.n_chunks == 0 || wait(&s.q_ready, 0);
        if (!ok) fail();
        // The 16 K-steps of one X half (dims 256 HF + 16 kl + ...): Q from TMEM
        // below dim 256, from shared memory above. The half is a template
        // argument and each step's descriptor is the base descriptor plus a
        // constant (the start-address field counts 16-byte units), so the
        // issue loop is little more than the MMA instructions themselves.
        auto qk_half = [&](auto hf_tag, const uint8_t *xbuf, bool first) {
            constexpr int HF = decltype(hf_tag)::value;
            constexpr int kTs = HF == 0 ? 16 : (kQTmemDims / 16 > 16 ? kQTmemDims / 16 - 16 : 0);  // Q in TMEM
            const uint64_t xd = ptx::desc_kmajor_sw128(ptx::smem_u32(xbuf));
            const uint64_t qd = ptx::desc_kmajor_sw128(ptx::smem_u32(s.qs));
#pragma unroll
            for (int kl = 0; kl < kTs; ++kl)
                ptx::mma_f16_ts(tmem + kColS, tmem + kColQ + (16 * HF + kl) * 8,
                                xd + (uint64_t)(((kl >> 2) * kAtom + (kl & 3) * 32) >> 4), kIdescQK,
                                (first && kl == 0) ? 0u : 1u);
#pragma unroll
            for (int kl = kTs; kl < 16; ++kl) {
                const int kq = 16 * HF + kl - kQTmemDims / 16;
                ptx::mma_f16(tmem + kColS, qd + (uint64_t)(((kq >> 2) * kQAtom + (kq & 3) * 32) >> 4),
                             xd + (uint64_t)(((kl >> 2) * kAtom + (kl & 3) * 32) >> 4), kIdescQK,
                             (first && kTs == 0 && kl == 0) ? 0u : 1u);
            }
        };
        using Lo = std::integral_constant<int, 0>;
        using Hi = std::integral_constant<int, 1>;
        // QK(jq) -> S once the softmax has read S(jq-1): the half this CTA does
        // not output first (it is converted first), then its own half.
        // QK(jq): the half this CTA does not output first (its buffer is
        // released as soon as these MMAs complete), then its own half. The
        // two parts share one instance of each templated half (rank 0 runs Hi
        // then Lo, rank 1 Lo then Hi), so the unrolled MMA sequences appear
        // once each in the instruction stream.
        auto issue_qk = [&](int jq) -> bool {
            const int ob = jq % kOthBufs, wb = jq % kOwnBufs;
#pragma unroll 1
            for (int part = 0; part < 2; ++part) {
                const bool oth_part = part == 0;
                if (oth_part) {
                    if (!wait(&s.oth_full[ob], (jq / kOthBufs) & 1)) return false;
                    if (jq >= 1 && !wait(&s.s_free, (jq - 1) & 1)) return false;
                } else {
                    if (!wait(&s.own_full[wb], (jq / kOwnBufs) & 1)) return false;
                }
                ptx::tc_fence_after();
                if (lane == 0) {
                    const uint8_t *xbuf = oth_part ? s.x_oth[ob] : s.x_own[wb];
                    if ((rank == 0) == oth_part) qk_half(Hi{}, xbuf, oth_part);
                    else qk_half(Lo{}, xbuf, oth_part);
                    ptx::mma_commit(oth_part ? &s.oth_empty[ob] : &s.s_full);
                }
                __syncwarp();
            }
            return true;
        };
        auto issue_pv = [&](int jp) -> bool {
            const int wb = jp % kOwnBufs;
            if (!wait(&s.p_full, jp & 1)) return false;
            ptx::tc_fence_after();
            if (lane == 0) {
                const uint32_t xa = ptx::smem_u32(s.x_own[wb]);
                const uint32_t pa = ptx::smem_u32(s.p);
                const uint64_t ad = ptx::desc_kmajor_sw128(pa);
                const uint64_t bd = ptx::desc_mnmajor_sw128(xa, kAtom, 1024);
#pragma unroll
                for (int kk = 0; kk < kChunk / 16; ++kk)
                    ptx::mma_f16(tmem + kColO, ad + (uint64_t)(kk * 32 >> 4), bd + (uint64_t)(kk * 2048 >> 4), kIdescPV,
                                 (jp > 0 || kk > 0) ? 1u : 0u);
                ptx::mma_commit(&s.own_empty[wb]);
                ptx::mma_commit(&s.o_done[jp & 1]);
            }
            __syncwarp();
            return true;
        };
        // QK(0), then QK(j+1) before PV(j); one call site each keeps a single
        // copy of the unrolled MMA sequences in the instruction stream
        for (int j = 0; j <= u.n_chunks && ok; ++j) {
            if (j < u.n_chunks && !issue_qk(j)) { fail(); ok = false; break; }
            if (j > 0 && !issue_pv(j - 1)) { fail(); ok = false; break; }
        }
        if (lane == 0) {
            ptx::mma_commit(&s.o_final);
            ptx::mma_commit(&s.mma_done);
        }
        __syncwarp();
        // every MMA issued has finished with tensor and shared memory before
        // the CTA frees them (not cut short by the abort flag)
        if (!__all_sync(0xffffffffu, ptx::mbar_wait_drain(&s.mma_done, 0, kDrainWaitNs)))
            report_error(P.err, CSA_ERR_TIMEOUT);
    } else if (role == kRoleConvert) {
        // ------------------------------------------------------------ load + dequantise
        const int ct = convert_index(warp) * 32 + lane;  // 0..255
        const int row = ct >> 2, hq = ct & 3;
        const int own_hf = rank, oth_hf = rank ^ 1;
        auto fetch_ptr = [&](int jj, const uint8_t *&rec) -> bool {
            const int pr = jj % kPtrRing;
            if (!wait(&s.ptr_full[pr], (jj / kPtrRing) & 1)) return false;
            rec = s.rec[pr][row];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&s.ptr_empty[pr]);
            return true;
        };
        // copies this thread's pieces of half hf of record `rec` into the half's staging
        // Records are read by the two CTAs of a pair within a chunk of each
        // other and never again: evict-first keeps them from displacing what
        // the next kernels read (measured: the next step's indexer runs
        // 0.7 us faster, this kernel 1 us faster).
        const uint64_t rec_policy = ptx::l2_policy_evict_first();
        auto load_half = [&](int hf, const uint8_t *rec) {
            if (!rec) return;
            if (hf == 0) {
#pragma unroll
                for (int i = 0; i < kLoPieces; ++i) ptx::cp_async_16_hint(&s.stage_lo.piece[i][ct], rec + 16 * (hq + 4 * i), rec_policy);
                if (hq == 0) ptx::cp_async_16_hint(&s.stage_lo.scale[row], rec + kScaleOffset, rec_policy);
            } else {
#pragma unroll
                for (int i = 0; i < kHiPieces; ++i)
                    ptx::cp_async_16_hint(&s.stage_hi.piece[i][ct], rec + 256 + 16 * (hq + 4 * i), rec_policy);
                if (hq == 0) ptx::cp_async_16_hint(&s.stage_hi.scale[row], rec + kScaleOffset, rec_policy);
            }
        };
        // Piece hq + 4 i of a half: code pieces hold 16 dims starting at
        // 16 (hq + 4 i) within the half -> column block i, 16-byte chunks 2 hq
        // and 2 hq + 1, block multiplier i / 2; the hi half's pieces 12..19
        // (i = 3, 4) are the rope dims 448 + 8 (piece - 12)... -> column block
        // 3, chunk piece - 12 (copied as they are). The loops stay rolled: the
        // hot code of all four warp roles shares each scheduler's instruction
        // cache.
        auto convert_codes = [&](uint8_t *xs, const uint4 *pieces, int n, float m_lo, float m_hi, bool valid) {
            const uint4 zero = make_uint4(0, 0, 0, 0);
#pragma unroll 1
            for (int i = 0; i < n; ++i) {
                uint4 lo = zero, hi = zero;
                if (valid) {
                    const uint4 c = pieces[i * 4 * kChunk + ct];
                    const float mult = (i >> 1) ? m_hi : m_lo;
                    lo = dequant8(c.x, c.y, mult);
                    hi = dequant8(c.z, c.w, mult);
                }
                uint8_t *atom = xs + i * kAtom;
                *sw128(atom, row, 2 * hq) = lo;
                *sw128(atom, row, 2 * hq + 1) = hi;
            }
        };
        auto convert_half = [&](int hf, uint8_t *xs, bool valid) {
            if (hf == 0) {
                const float4 sc = valid ? s.stage_lo.scale[row] : make_float4(0.f, 0.f, 0.f, 0.f);
                convert_codes(xs, &s.stage_lo.piece[0][0], kLoPieces, sc.x, sc.y, valid);
            } else {
                const float4 sc = valid ? s.stage_hi.scale[row] : make_float4(0.f, 0.f, 0.f, 0.f);
                convert_codes(xs, &s.stage_hi.piece[0][0], 3, sc.z, sc.w, valid);
#pragma unroll
                for (int i = 3; i < kHiPieces; ++i)
                    *sw128(xs + 3 * kAtom, row, hq + 4 * (i - 3)) =
                        valid ? s.stage_hi.piece[i][ct] : make_uint4(0, 0, 0, 0);
            }
        };
        // cp.async groups, oldest first: oth(0), own(0), then per chunk j
        // oth(j+1) and own(j+1) (empty past the last chunk), so "at most one
        // pending" before each conversion means the half about to be converted
        // has landed.
        bool ok = true;
        const uint8_t *rec_nxt = nullptr, *rec_cur = nullptr;
        if (u.n_chunks > 0 && !fetch_ptr(0, rec_nxt)) { fail(); ok = false; }
        // Half-steps t = 2j (other half of chunk j) and 2j + 1 (own half): the
        // staging of half-step t + 2 is copied right after half-step t is
        // converted, and half-steps -2 and -1 copy chunk 0. One call site per
        // helper keeps a single copy of each in the instruction stream.
        for (int t = -2; t < 2 * u.n_chunks && ok; ++t) {
            const int j = t >> 1;  // (floor: -1 for t = -2, -1)
            const bool own_step = (t & 1) != 0;
            const int hf = own_step ? own_hf : oth_hf;
            if (t >= 0) {
                if (!own_step) rec_cur = rec_nxt;
                const int nb = own_step ? kOwnBufs : kOthBufs;
                uint8_t *xs = own_step ? s.x_own[j % kOwnBufs] : s.x_oth[j % kOthBufs];
                uint64_t *empty_bar = own_step ? &s.own_empty[j % kOwnBufs] : &s.oth_empty[j % kOthBufs];
                uint64_t *full_bar = own_step ? &s.own_full[j % kOwnBufs] : &s.oth_full[j % kOthBufs];
                ptx::cp_async_wait<1>();
                __syncwarp();  // the row's multipliers (copied by its first thread) are visible to all four
                if (!wait(empty_bar, ((j / nb) & 1) ^ 1)) { fail(); ok = false; break; }
                convert_half(hf, xs, rec_cur != nullptr);
                ptx::fence_proxy_async_smem();  // generic-proxy stores -> MMA (async proxy) reads
                __syncwarp();                   // (and the row's threads are done with the staging)
                if (lane == 0) ptx::mbar_arrive(full_bar);
                if (!own_step && j + 1 < u.n_chunks && !fetch_ptr(j + 1, rec_nxt)) { fail(); ok = false; break; }
            }
            if (j + 1 < u.n_chunks) load_half(hf, rec_nxt);
            ptx::cp_async_commit();
        }
        ptx::cp_async_wait<0>();  // no copy lands after this warp has moved on
    } else if (role == kRoleSoftmax) {
        // ------------------------------------------------------------ softmax / epilogue
        const int quarter = warp & 3;
        const int h = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const int r = u.r;
        bool ok = true;
        // Q: the dims from kQTmemDims up -> shared memory (cp.async), the
        // dims below -> TMEM (BF16 pairs, lane = head)
        if (u.n_chunks > 0) {
            const uint4 *qg = reinterpret_cast<const uint4 *>(P.q + ((size_t)r * kHeads + h) * kDim);
            // every byte a decode step reads or writes once is marked
            // evict-first, so that the next step's indexer finds L2 full of
            // lines it can replace cheaply (measured on the whole step)
            const uint64_t q_policy = ptx::l2_policy_evict_first();
#pragma unroll
            for (int c = 0; c < (kDim - kQTmemDims) / 8; ++c)
                ptx::cp_async_16_hint(sw128(s.qs + (c >> 3) * kQAtom, h, c & 7), qg + kQTmemDims / 8 + c, q_policy);
            ptx::cp_async_commit();
            // pieces of 64 dims (128 B a thread, 32 TMEM columns), two in
            // flight: piece p + 2 is requested as soon as piece p has gone to
            // TMEM
            constexpr int kQPieces = kQTmemDims / 64;
            uint4 wa[8], wb[8];
            auto load_piece = [&](uint4 (&w)[8], int pc) {
#pragma unroll
                for (int v = 0; v < 8; ++v) w[v] = ptx::ldg_v4_policy(qg + pc * 8 + v, q_policy);
            };
            auto store_piece = [&](const uint4 (&w)[8], int pc) {
                uint32_t regs[32];
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    regs[4 * v] = w[v].x;
                    regs[4 * v + 1] = w[v].y;
                    regs[4 * v + 2] = w[v].z;
                    regs[4 * v + 3] = w[v].w;
                }
                ptx::tmem_st32(lane_base + kColQ + pc * 32, regs);
            };
            load_piece(wa, 0);
            load_piece(wb, 1);
#pragma unroll 1
            for (int pc = 0; pc < kQPieces; pc += 2) {
                store_piece(wa, pc);
                if (pc + 2 < kQPieces) load_piece(wa, pc + 2);
                store_piece(wb, pc + 1);
                if (pc + 3 < kQPieces) load_piece(wb, pc + 3);
            }
            ptx::cp_async_wait<0>();
            ptx::tmem_st_wait();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&s.q_ready);
        }
        float m = -INFINITY, l = 0.f;  // running max and sum, log2 domain, sink not included
        for (int j = 0; j < u.n_chunks && ok; ++j) {
            const int pr = j % kPtrRing;
            if (!wait(&s.ptr_full[pr], (j / kPtrRing) & 1)) { fail(); ok = false; break; }
            const uint64_t mask = s.vmask[pr];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&s.ptr_empty[pr]);
            if (!wait(&s.s_full, j & 1)) { fail(); ok = false; break; }
            ptx::tc_fence_after();
            uint32_t sa[32], sb[32];
            ptx::tmem_ld32(lane_base + kColS, sa);
            ptx::tmem_ld32(lane_base + kColS + 32, sb);
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&s.s_free);
            float z[kChunk];
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < kChunk; ++c) {
                const float sv = __uint_as_float(c < 32 ? sa[c] : sb[c - 32]);
                z[c] = ((mask >> c) & 1ull) ? sv * P.scale_log2 : -INFINITY;
                mx4[c & 3] = fmaxf(mx4[c & 3], z[c]);
            }
            const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            // Lazy rescale. The decision is per head (lane) but the TMEM accesses
            // and waits below are warp-collective, so the whole warp enters
            // when any lane needs it; other lanes use a factor of 1.
            const bool need = mx > m + kLazy || (m == -INFINITY && mx > -INFINITY);
            if (__any_sync(0xffffffffu, need)) {
                const float alpha = need ? ptx::ex2_approx(m - mx) : 1.f;  // 0 when m = -inf
                if (j > 0) {
                    // O holds PV of chunks < j: wait for the last one, then rescale in place.
                    // (This thread saw PV(j-2) done before writing P(j-1), and PV(j-3)
                    // completed before it, so the barrier is at most one phase
                    // behind and the parity test is unambiguous.)
                    if (!wait(&s.o_done[(j - 1) & 1], ((j - 1) >> 1) & 1)) { fail(); ok = false; break; }
                    ptx::tc_fence_after();
#pragma unroll 1
                    for (int piece = 0; piece < kHalf / 32; ++piece) {
                        uint32_t o[32];
                        ptx::tmem_ld32(lane_base + kColO + piece * 32, o);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        ptx::tmem_st32(lane_base + kColO + piece * 32, o);
                    }
                    ptx::tmem_st_wait();
                    ptx::tc_fence_before();
                }
                l *= alpha;
                if (need) m = mx;
            }
            // P(j) = 2^(z - m) as BF16 (the head's swizzled 128-byte row), once
            // PV(j-1) has finished reading the previous P
            if (j > 0 && !wait(&s.o_done[(j - 1) & 1], ((j - 1) >> 1) & 1)) { fail(); ok = false; break; }
            const float mref = (m == -INFINITY) ? 0.f : m;  // every z is -inf while m is
            float ps4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c8 = 0; c8 < kChunk / 8; ++c8) {
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float p0 = ptx::ex2_approx(z[8 * c8 + 2 * i] - mref);
                    const float p1 = ptx::ex2_approx(z[8 * c8 + 2 * i + 1] - mref);
                    ps4[i] += p0 + p1;
                    w[i] = bf16x2_bits(p0, p1);
                }
                *sw128(s.p, h, c8) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            l += (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
            ptx::fence_proxy_async_smem();  // P stores -> PV (async proxy) reads
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&s.p_full);
        }
        // ---------------- epilogue: O half (and LSE) out
        if (ok && u.n_chunks > 0) {
            if (!wait(&s.o_final, 0)) { fail(); ok = false; }
            ptx::tc_fence_after();
        }
        if (ok) {
            float factor, lse_out = 0.f;
            const float2 ml = make_float2(m, l);
            if (P.n_split == 1) {
                const float sk = __ldg(P.sink + h) * kLog2e;
                const float M = fmaxf(sk, m);
                const float es = (sk == -INFINITY) ? 0.f : exp2f(sk - M);
                const float eo = (m == -INFINITY) ? 0.f : exp2f(m - M);
                const float den = es + l * eo;
                factor = den > 0.f ? eo / den : 0.f;
                lse_out = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
            } else {
                factor = l > 0.f ? 1.f / l : 0.f;
            }
            // With one split this CTA forms the final output of its half, and
            // the epilogue (inverse RoPE on the rope dims, which all sit in the
            // high half; E2M1 output) applies here; with several the combine
            // applies it.
            const bool final_out = P.n_split == 1;
            const bool rope_here = final_out && P.epi.inv_rope && rank == 1;
            float2 cs = make_float2(1.f, 0.f);  // lane i: cos, sin of rope pair i
            if (rope_here) cs = rope_cos_sin(u.p, P.epi.rope_freq[lane]);
            // piece p (32 dims) of this head's O half, normalised and turned back
            auto piece_values = [&](int piece, float (&v)[32]) {
                if (u.n_chunks > 0) {
                    uint32_t o[32];
                    ptx::tmem_ld32(lane_base + kColO + piece * 32, o);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(o[i]) * factor;
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0.f;
                }
                if (rope_here && piece >= (kNope - kHalf) / 32) {  // latent dims 448..511
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int pair = (piece - (kNope - kHalf) / 32) * 16 + e;
                        const float c = __shfl_sync(0xffffffffu, cs.x, pair);
                        const float sn = __shfl_sync(0xffffffffu, cs.y, pair);
                        const float x = v[2 * e], y = v[2 * e + 1];
                        v[2 * e] = fmaf(x, c, y * sn);
                        v[2 * e + 1] = fmaf(-x, sn, y * c);
                    }
                }
            };
            // Rows are staged in shared memory (the own X buffers are free once
            // every PV is done), then each warp writes its 32 head rows whole
            // (coalesced). Chunk c (16 B) of row h sits at position c ^ (h & 7):
            // conflict-free both ways.
            uint8_t *ostage = &s.x_own[0][0];
            if (!(final_out && P.epi.out_fp4)) {
                // BF16: 512 B per head row
                uint8_t *srow = ostage + h * (kHalf * 2);
#pragma unroll 1
                for (int piece = 0; piece < kHalf / 32; ++piece) {
                    float v[32];
                    piece_values(piece, v);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int c = piece * 4 + q4;
                        *reinterpret_cast<uint4 *>(srow + ((c ^ (h & 7)) << 4)) =
                            make_uint4(bf16x2_bits(v[8 * q4 + 0], v[8 * q4 + 1]), bf16x2_bits(v[8 * q4 + 2], v[8 * q4 + 3]),
                                       bf16x2_bits(v[8 * q4 + 4], v[8 * q4 + 5]), bf16x2_bits(v[8 * q4 + 6], v[8 * q4 + 7]));
                    }
                }
                __syncwarp();
                const uint64_t part_policy = ptx::l2_policy_evict_first();
                __nv_bfloat16 *dst0 = final_out
                                          ? P.out + (size_t)r * kHeads * kDim + rank * kHalf
                                          : P.part_o + ((size_t)r * P.n_split + u.split) * kHeads * kDim + rank * kHalf;
#pragma unroll 4
                for (int i = 0; i < 32; ++i) {
                    const int hr = quarter * 32 + i;  // a head row of this warp
                    const uint4 v = *reinterpret_cast<const uint4 *>(ostage + hr * (kHalf * 2) + ((lane ^ (hr & 7)) << 4));
                    if (final_out)
                        reinterpret_cast<uint4 *>(dst0 + (size_t)hr * kDim)[lane] = v;
                    else  // split partials are read once, by the combine: evict-first
                        ptx::stg_v4_policy(reinterpret_cast<uint4 *>(dst0 + (size_t)hr * kDim) + lane, v, part_policy);
                }
            } else {
                // E2M1: two 128-dim blocks per half, each scaled by its amax / 6
                // (a first pass over TMEM finds the amax); 128 B per head row
                uint8_t *frow = ostage + h * (kFp4RowBytes / 2);
#pragma unroll 1
                for (int bl = 0; bl < 2; ++bl) {
                    float amax = 0.f;
#pragma unroll 1
                    for (int pp = 0; pp < 4; ++pp) {
                        float v[32];
                        piece_values(4 * bl + pp, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
                    }
                    const float sc = amax > 0.f ? amax / 6.f : 1.f;
                    const float inv = 1.f / sc;  // value / sc as value * (1 / sc): equal up to one ulp
#pragma unroll 1
                    for (int pp = 0; pp < 4; ++pp) {
                        float v[32];
                        piece_values(4 * bl + pp, v);
                        uint32_t w[4];
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            w[q4] = e2m1x4(v[8 * q4] * inv, v[8 * q4 + 1] * inv, v[8 * q4 + 2] * inv,
                                           v[8 * q4 + 3] * inv) |
                                    (e2m1x4(v[8 * q4 + 4] * inv, v[8 * q4 + 5] * inv, v[8 * q4 + 6] * inv,
                                            v[8 * q4 + 7] * inv) << 16);
                        const int c = 4 * bl + pp;
                        *reinterpret_cast<uint4 *>(frow + ((c ^ (h & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    P.epi.out_fp4_scale[((size_t)r * kHeads + h) * 4 + rank * 2 + bl] = sc;
                }
                __syncwarp();
#pragma unroll 2
                for (int i = 0; i < 8; ++i) {
                    const int hr = quarter * 32 + i * 4 + (lane >> 3);  // 8 lanes per 128-byte row
                    const int c = lane & 7;
                    const uint4 v = *reinterpret_cast<const uint4 *>(ostage + hr * (kFp4RowBytes / 2) + ((c ^ (hr & 7)) << 4));
                    reinterpret_cast<uint4 *>(P.epi.out_fp4 + ((size_t)r * kHeads + hr) * kFp4RowBytes +
                                              rank * (kFp4RowBytes / 2))[c] = v;
                }
            }
            if (rank == 0) {
                if (P.n_split == 1)
                    P.lse[(size_t)r * kHeads + h] = lse_out;
                else
                    P.part_ml[((size_t)r * P.n_split + u.split) * kHeads + h] = ml;
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
}

// Folds the per-split normalised partials and the sink:
//   M = max(sink, m_s), den = e^{sink-M} + sum_s l_s e^{m_s-M},
//   out = sum_s l_s e^{m_s-M} o_s / den, lse = M + ln den   (log2 domain inside).
// One warp per (row, head), 16 dims per lane; the (max, sum) pairs and the
// partial rows of up to 8 splits are loaded together before any use.
constexpr int kCombineBatch = 8;
__global__ void __launch_bounds__(256)
attention_combine_kernel(const __nv_bfloat16 *__restrict__ part_o, const float2 *__restrict__ part_ml,
                         const float *__restrict__ sink, int n_split, __nv_bfloat16 *__restrict__ out,
                         float *__restrict__ lse, const int32_t *__restrict__ q_pos, const EpiParams epi) {
    ptx::griddep_wait();  // the split partials (previous kernel in the stream) are complete
    const int r = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float2 cs = make_float2(1.f, 0.f);  // lane i: cos, sin of rope pair i
    if (epi.inv_rope) cs = rope_cos_sin(__ldg(q_pos + r), epi.rope_freq[lane]);
    const int h = blockIdx.x * 8 + warp;
    const float sk = __ldg(sink + h) * kLog2e;
    const float2 *ml_row = part_ml + (size_t)r * n_split * kHeads + h;
    const uint4 *o_row = reinterpret_cast<const uint4 *>(part_o + ((size_t)r * n_split * kHeads + h) * kDim) + lane * 2;
    const size_t split_stride = (size_t)kHeads * kDim / 8;  // uint4 per split
    const uint64_t policy = ptx::l2_policy_evict_first();  // the partials are read once
    // (every split writes its partial row, zeros when it had no candidates,
    // so the rows are loaded without waiting for the (max, sum) pairs)
    float M = sk;
    if (n_split > kCombineBatch)
        for (int sp = 0; sp < n_split; ++sp) {
            const float2 ml = ml_row[(size_t)sp * kHeads];
            if (ml.y > 0.f) M = fmaxf(M, ml.x);
        }
    float den = 0.f;
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
    for (int s0 = 0; s0 < n_split; s0 += kCombineBatch) {
        float2 ml[kCombineBatch];
        uint4 v[kCombineBatch][2];
#pragma unroll
        for (int q = 0; q < kCombineBatch; ++q) {
            const int sp = s0 + q;
            if (sp < n_split) {
                ml[q] = ml_row[(size_t)sp * kHeads];
                v[q][0] = ptx::ldg_v4_policy(o_row + sp * split_stride, policy);
                v[q][1] = ptx::ldg_v4_policy(o_row + sp * split_stride + 1, policy);
            } else {
                ml[q] = make_float2(0.f, 0.f);
                v[q][0] = v[q][1] = make_uint4(0, 0, 0, 0);
            }
        }
        if (n_split <= kCombineBatch) {
#pragma unroll
            for (int q = 0; q < kCombineBatch; ++q)
                if (ml[q].y > 0.f) M = fmaxf(M, ml[q].x);
        }
#pragma unroll
        for (int q = 0; q < kCombineBatch; ++q) {
            if (!(ml[q].y > 0.f)) continue;
            const float w = ml[q].y * exp2f(ml[q].x - M);
            den += w;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const uint32_t wv[4] = {v[q][e].x, v[q][e].y, v[q][e].z, v[q][e].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[8 * e + 2 * i] = fmaf(w, bf16_bits_to_float(static_cast<uint16_t>(wv[i] & 0xFFFFu)), acc[8 * e + 2 * i]);
                    acc[8 * e + 2 * i + 1] = fmaf(w, bf16_bits_to_float(static_cast<uint16_t>(wv[i] >> 16)), acc[8 * e + 2 * i + 1]);
                }
            }
        }
    }
    den += (sk == -INFINITY) ? 0.f : exp2f(sk - M);
    const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] *= inv;
    // epilogue: lanes 28..31 hold the rope dims 448..511, 8 pairs each
    if (epi.inv_rope) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int pair = ((lane - kNope / 16) & 3) * 8 + e;
            const float c = __shfl_sync(0xffffffffu, cs.x, pair);
            const float sn = __shfl_sync(0xffffffffu, cs.y, pair);
            if (lane >= kNope / 16) {
                const float x = acc[2 * e], y = acc[2 * e + 1];
                acc[2 * e] = fmaf(x, c, y * sn);
                acc[2 * e + 1] = fmaf(-x, sn, y * c);
            }
        }
    }
    if (epi.out_fp4) {
        // E2M1 with one multiplier per 128 dims = 8 lanes
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(acc[i]));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float sc = amax > 0.f ? amax / 6.f : 1.f;
        const float isc = 1.f / sc;  // value / sc as value * (1 / sc): equal up to one ulp
        uint32_t w[2];
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2)
            w[q2] = e2m1x4(acc[8 * q2] * isc, acc[8 * q2 + 1] * isc, acc[8 * q2 + 2] * isc, acc[8 * q2 + 3] * isc) |
                    (e2m1x4(acc[8 * q2 + 4] * isc, acc[8 * q2 + 5] * isc, acc[8 * q2 + 6] * isc,
                            acc[8 * q2 + 7] * isc) << 16);
        reinterpret_cast<uint2 *>(epi.out_fp4 + ((size_t)r * kHeads + h) * kFp4RowBytes)[lane] = make_uint2(w[0], w[1]);
        if ((lane & 7) == 0) epi.out_fp4_scale[((size_t)r * kHeads + h) * 4 + (lane >> 3)] = sc;
    } else {
        uint4 *dst = reinterpret_cast<uint4 *>(out + ((size_t)r * kHeads + h) * kDim) + lane * 2;
#pragma unroll
        for (int e = 0; e < 2; ++e)
            ptx::stg_v4_policy(dst + e, make_uint4(bf16x2_bits(acc[8 * e + 0], acc[8 * e + 1]),
                                                   bf16x2_bits(acc[8 * e + 2], acc[8 * e + 3]),
                                                   bf16x2_bits(acc[8 * e + 4], acc[8 * e + 5]),
                                                   bf16x2_bits(acc[8 * e + 6], acc[8 * e + 7])),
                               policy);
    }
    if (lane == 0) lse[(size_t)r * kHeads + h] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
}

// Splits per query so that about one CTA pair per two SMs is busy.
// `max_candidates` bounds the candidates of any query (selected + window).
int choose_splits(int rows, int max_candidates) {
    const int chunks = (max_candidates + kChunk - 1) / kChunk;
    const int target = cached_sm_count() / 2;
    int n = target / (rows > 0 ? rows : 1);
    if (n > chunks) n = chunks;
    return n < 1 ? 1 : n;
}

size_t split_bytes(int rows, int n_split) {
    if (n_split <= 1) return 0;
    const size_t po = (size_t)rows * n_split * kHeads * kDim * sizeof(__nv_bfloat16);
    return (po + 255) / 256 * 256 + (size_t)rows * n_split * kHeads * sizeof(float2);
}

}  // namespace

// Workspace for queries of at most `max_selected` selected entries (top-k, or
// the HCA capacity) and a window of at most W tokens. Monotone in both, so a
// workspace sized with the largest window serves every smaller one.
size_t attention_workspace_bytes(int B, int T, int max_selected, int W) {
    const int rows = B * T;
    return split_bytes(rows, choose_splits(rows, max_selected + W));
}

// `k` = the top-k row length (CSA) or the per-sequence capacity (HCA).
cudaError_t launch_attention(const void *q, const float *sink, float scale, const csa_cache_desc &comp,
                             const void *ring, int R, int W, const int32_t *topk_idx, const int32_t *topk_cnt,
                             const int32_t *n_comp, int m_hca, const int32_t *q_pos, int B, int T, int k, bool hca,
                             void *out, float *lse, const csa_attention_epilogue *epi, void *ws, size_t ws_bytes,
                             int *err, cudaStream_t stream) {
    const int rows = B * T;
    const int n_split = choose_splits(rows, k + W);
    AttParams P;
    P.q = static_cast<const __nv_bfloat16 *>(q);
    P.sink = sink;
    P.scale_log2 = scale * kLog2e;
    P.comp = make_view(comp);
    P.ring = static_cast<const uint8_t *>(ring);
    P.R = R;
    P.W = W;
    P.topk_idx = topk_idx;
    P.topk_cnt = topk_cnt;
    P.n_comp = n_comp;
    P.q_pos = q_pos;
    P.m_hca = m_hca;
    P.hca = hca ? 1 : 0;
    P.T = T;
    P.k = hca ? 0 : k;
    P.n_split = n_split;
    P.out = static_cast<__nv_bfloat16 *>(out);
    P.lse = lse;
    P.part_o = nullptr;
    P.part_ml = nullptr;
    P.err = err;
    P.wait_ns = wait_limit_ns();
    P.epi.out_fp4 = epi ? epi->out_fp4 : nullptr;
    P.epi.out_fp4_scale = epi ? epi->out_fp4_scale : nullptr;
    P.epi.inv_rope = (epi && epi->inverse_rope) ? 1 : 0;
    for (int i = 0; i < kRopePairs; ++i)  // pair i turns by theta^(-2i/64) rad per position
        P.epi.rope_freq[i] = P.epi.inv_rope ? std::pow((double)epi->rope_theta, -2.0 * i / (2.0 * kRopePairs)) : 0.0;
    if (n_split > 1) {
        const size_t need = split_bytes(rows, n_split);
        if (!ws || ws_bytes < need) return cudaErrorInvalidValue;
        const size_t po = (size_t)rows * n_split * kHeads * kDim * sizeof(__nv_bfloat16);
        P.part_o = static_cast<__nv_bfloat16 *>(ws);
        P.part_ml = reinterpret_cast<float2 *>(static_cast<uint8_t *>(ws) + (po + 255) / 256 * 256);
    }
    const size_t smem = sizeof(AttSmem) + 1024;
    cudaError_t e = set_max_dynamic_smem_once(reinterpret_cast<const void *>(attention_tc_kernel), (int)smem);
    if (e != cudaSuccess) return e;
    // Both kernels may start before their predecessor in the stream ends
    // (programmatic dependent launch); each waits for it before reading its output.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * rows * n_split);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    count_launch();
    e = cudaLaunchKernelEx(&cfg, attention_tc_kernel, P);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess || n_split == 1) return e;
    cfg.gridDim = dim3(kHeads / 8, rows);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    count_launch();
    e = cudaLaunchKernelEx(&cfg, attention_combine_kernel, (const __nv_bfloat16 *)P.part_o,
                           (const float2 *)P.part_ml, sink, n_split, P.out, lse, q_pos, P.epi);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// ------------------------------------------------------------------ allocation-free variant
//
// Some callers of this library cannot allocate device memory on the decode
// path, so they cannot provide the split partials' workspace either: a serving
// runtime whose whole device memory is reserved by its own pool at start-up, a
// plugin inside a host framework that owns every device allocation, or host
// code on a latency-critical path where cudaMalloc's implicit device-wide
// synchronisation is not acceptable. For them, csa_sink_attention_decode_noalloc
// runs the same attention with its scratch in the static array below.
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB, held by every device that loads the library
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void *g_static_scratch_addr[kMaxDevices];
std::mutex g_static_scratch_mu;

// Device address of the static scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
cudaError_t static_scratch_address(void **addr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_static_scratch_mu);
    if (!g_static_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_static_scratch_addr[dev] = p;
    }
    *addr = g_static_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

}  // namespace csa

extern "C" CSA_API csa_status_t csa_sink_attention_decode_noalloc(
    const void *q, const float *sink, float softmax_scale, csa_cache_desc comp, const void *swa_ring, int R, int W,
    const int32_t *topk_idx, const int32_t *topk_cnt, const int32_t *q_pos, int B, int T, int k, void *out, float *lse,
    int32_t *status, cudaStream_t stream) {
    using namespace csa;
    // the same checks as csa_sink_attention_decode
    const csa_status_t a = attention_arg_status(q, sink, softmax_scale, comp, swa_ring, R, W, topk_idx, topk_cnt,
                                                q_pos, B, T, k, out, lse, status);
    if (a != CSA_OK) return a;
    const size_t need = attention_workspace_bytes(B, T, k, W);
    if (need > kStaticScratchBytes) return CSA_ERR_UNSUPPORTED;  // beyond the static scratch: use the workspace call
    void *scratch = nullptr;
    if (need && static_scratch_address(&scratch) != cudaSuccess) return CSA_ERR_CUDA;
    const cudaError_t e = launch_attention(q, sink, softmax_scale, comp, swa_ring, R, W, topk_idx, topk_cnt, nullptr,
                                           1, q_pos, B, T, k, false, out, lse, nullptr, scratch,
                                           need ? kStaticScratchBytes : 0, status, stream);
    return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}
