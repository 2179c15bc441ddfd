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
// Work unit = (query token, candidate split), run by a cluster of two CTAs;
// CTA rank r owns latent dims [256 r, 256 r + 256):
//   * Q[:, half] (128 heads x 256 BF16) lives in TMEM and is the A operand of
//     QK; each CTA computes the partial scores of its half for a chunk of 64
//     candidates (tcgen05.mma kind::f16, M=128 heads, N=64, K=256) and the two
//     partials are exchanged through distributed shared memory, so both CTAs
//     hold identical full scores and run an identical softmax.
//   * P (BF16) is written back into the score columns of TMEM and is the A
//     operand of PV: O[:, half] += P X[:, half] (M=128, N=256, K=64); O stays
//     in TMEM (256 fp32 columns) across chunks.
//   * Candidate bytes are gathered straight from the FP8/BF16 caches (TMA bulk
//     copies, block-table strided) and dequantised in shared memory to BF16
//     (code x block multiplier); there is no dequantised copy in HBM.
// Warps: 0 gather producer, 1 MMA issuer (and TMEM owner), 2-5 dequantise,
// 6-9 softmax / exchange / epilogue (thread = head). The running max is
// rescaled lazily (only when it grows by more than 2^8), in the log2 domain.
// With one split per query the CTA pair writes the BF16 output and LSE; with
// several, each split writes a normalised BF16 partial and (max, sum), and a
// combine kernel folds the splits and the sink. Every wait is bounded.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace csa {

namespace {

constexpr int kChunk = 64;                  // candidates per chunk
constexpr int kHalf = 256;                  // latent dims per CTA
constexpr int kSlot = 336;                  // staged bytes per candidate
constexpr int kStages = 2;                  // staging ring depth (chunks)
constexpr int kXBuf = 3;                    // dequantised chunk buffers
constexpr int kBatch = 4;                   // chunks whose indices the producer loads at once
constexpr int kThreads = 320;               // 10 warps
constexpr int kAtom = kChunk * 128;         // one 64-dim column block of X: 64 rows x 128 B
constexpr int kXBytes = 4 * kAtom;          // 32 KB
constexpr uint64_t kWaitNs = 1000000000ull; // 1 s per wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazy = 8.f;                // rescale only when the max grows by > 2^8

constexpr uint32_t kColQ = 0;    // 128 columns: Q half, BF16 pairs
constexpr uint32_t kColO = 128;  // 256 columns: O half, fp32
constexpr uint32_t kColS = 384;  // 2 x 64 columns: partial scores
constexpr uint32_t kTmemCols = 512;

// recv[b] receives the peer's partial scores of a chunk ([16 float4][128
// heads], fp32); p holds the chunk's P (128 heads x 64 candidates, BF16,
// K-major rows of 128 B in the 128-byte swizzle), the A operand of PV.
struct AttSmem {
    alignas(1024) uint8_t x[kXBuf][kXBytes];    // dequantised candidates, 128-byte swizzle
    alignas(1024) float4 recv[2][16 * kHeads];
    alignas(1024) uint8_t p[kHeads * 128];
    alignas(128) uint8_t stage[kStages][kChunk * kSlot];
    uint64_t vmask[kStages], smask[kXBuf];
    uint64_t stg_full[kStages], stg_empty[kStages];
    uint64_t x_full[kXBuf], x_empty[kXBuf];
    uint64_t s_full[2], s_free[2], p_full[2], rd_done[2];
    uint64_t xchg_full[2], xchg_free[2];
    uint64_t o_done[2], o_final, q_ready, mma_done;
    uint32_t tmem_base;
    int abort_flag;
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
};

struct Unit {
    int r, b, split, p, n_sel, j0, cb, ce, n_chunks;
};

__device__ __forceinline__ Unit make_unit(const AttParams &P) {
    Unit u;
    const int cluster = blockIdx.x >> 1;
    u.r = cluster / P.n_split;
    u.split = cluster % P.n_split;
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

// 16 E4M3 codes times a multiplier -> 16 BF16 values (two uint4).
__device__ __forceinline__ void dequant16(uint4 c, float s, uint4 &lo, uint4 &hi) {
    lo = dequant8(c.x, c.y, s);
    hi = dequant8(c.z, c.w, s);
}

// One 64-dim block of a row in the 128-byte swizzle: 16-byte chunk cc of the
// 128-byte row lands at position cc ^ (row & 7).
__device__ __forceinline__ void store_atom_row(uint8_t *xa, int row, const uint4 (&v)[8]) {
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) *reinterpret_cast<uint4 *>(xa + ((cc ^ (row & 7)) << 4)) = v[cc];
}

// Pipeline per chunk j (64 candidates), per CTA of the pair:
//   producer:  gather raw bytes of chunk j            -> stage[j % 2]
//   dequant:   stage -> X[j % 3] (BF16)               (after PV(j-3) freed it)
//   MMA:       QK(j) -> S[j & 1] (after the softmax released S(j-2));
//              PV(j) = P(j) X(j) -> O (after P(j) is ready); QK(j+2) is
//              issued before PV(j), so scores run two chunks ahead
//   softmax:   sends S(j+1) to the peer, combines S(j) with the peer's
//              partial, releases S[j & 1] and (to the peer) recv[j & 1],
//              writes P(j) into the P buffer once PV(j-1) is done
//   PV(j) completion frees X[j % 3] and the P buffer.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
attention_tc_kernel(const AttParams P) {
    extern __shared__ uint8_t smem_raw[];
    AttSmem &s = *reinterpret_cast<AttSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    volatile int *abort = &s.abort_flag;
    const Unit u = make_unit(P);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(&s.stg_full[i], 64);  // 32 copy-completion arrivals + 32 lane arrivals
            ptx::mbar_init(&s.stg_empty[i], 4);
        }
        for (int i = 0; i < kXBuf; ++i) {
            ptx::mbar_init(&s.x_full[i], 4);
            ptx::mbar_init(&s.x_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&s.s_full[i], 1);
            ptx::mbar_init(&s.s_free[i], 4);
            ptx::mbar_init(&s.p_full[i], 4);
            ptx::mbar_init(&s.rd_done[i], 4);  // every softmax warp has read recv[i]
            ptx::mbar_init(&s.xchg_full[i], 1);  // local expect_tx + the peer's st.async bytes
            ptx::mbar_init(&s.xchg_free[i], 1);  // the peer has read its recv[i]
            ptx::mbar_init(&s.o_done[i], 1);     // PV of a chunk of this parity is done
        }
        ptx::mbar_init(&s.o_final, 1);
        ptx::mbar_init(&s.q_ready, 4);
        ptx::mbar_init(&s.mma_done, 1);
        s.abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(&s.tmem_base, kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();  // the peer's barriers exist before anyone signals them
    ptx::tc_fence_after();
    const uint32_t tmem = s.tmem_base;

    auto fail = [&]() {
        report_error(P.err, CSA_ERR_TIMEOUT);
        *abort = 1;
    };
    auto wait = [&](uint64_t *bar, uint32_t parity) {
        return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, abort, kWaitNs)) != 0;
    };
    auto wait_cluster = [&](uint64_t *bar, uint32_t parity) {
        return __all_sync(0xffffffffu, ptx::mbar_wait_cluster(bar, parity, abort, kWaitNs)) != 0;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ gather producer
        // Candidate indices are loaded one batch (4 chunks) ahead; lane L holds
        // candidates L + 32 q (q = 0..7) of the batch, i.e. candidates L and
        // L + 32 of each of its 4 chunks.
        auto load_raw = [&](int g, int (&raw)[2 * kBatch]) {
#pragma unroll
            for (int q = 0; q < 2 * kBatch; ++q) {
                const int i = u.cb + g * kBatch * kChunk + q * 32 + lane;
                raw[q] = (!P.hca && i < u.ce && i < u.n_sel) ? __ldg(P.topk_idx + (size_t)u.r * P.k + i) : i;
            }
        };
        const int n_batches = (u.n_chunks + kBatch - 1) / kBatch;
        int cur[2 * kBatch], nxt[2 * kBatch];
        if (n_batches > 0) load_raw(0, nxt);
        int j = 0;
        bool ok = true;
        for (int g = 0; g < n_batches && ok; ++g) {
#pragma unroll
            for (int q = 0; q < 2 * kBatch; ++q) cur[q] = nxt[q];
            if (g + 1 < n_batches) load_raw(g + 1, nxt);
#pragma unroll
            for (int cc = 0; cc < kBatch; ++cc) {
                if (j >= u.n_chunks || !ok) break;
                const int st = j % kStages;
                if (!wait(&s.stg_empty[st], ((j / kStages) & 1) ^ 1)) { fail(); ok = false; break; }
                bool valid[2];
                const uint8_t *rec[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int i = u.cb + j * kChunk + e * 32 + lane;
                    rec[e] = nullptr;
                    if (i < u.ce) {
                        if (i < u.n_sel) {
                            const int64_t ri = record_index(P.comp, u.b, cur[2 * cc + e]);
                            if (ri >= 0) rec[e] = P.comp.base + ri * kRecBytes;
                            else if (rank == 0) report_error(P.err, CSA_ERR_BAD_INDEX);
                        } else {
                            const int pos = u.j0 + (i - u.n_sel);
                            rec[e] = P.ring + ((int64_t)u.b * P.R + pos % P.R) * kRecBytes;
                        }
                    }
                    valid[e] = rec[e] != nullptr;
                }
                // each lane copies its two candidates' bytes in 16-byte pieces:
                // rank 0 bytes [0,256) + [576,592), rank 1 bytes [256,592)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    if (!valid[e]) continue;
                    uint8_t *dst = s.stage[st] + (e * 32 + lane) * kSlot;
                    if (rank == 0) {
#pragma unroll
                        for (int pc = 0; pc < 16; ++pc) ptx::cp_async_16(dst + pc * 16, rec[e] + pc * 16);
                        ptx::cp_async_16(dst + 256, rec[e] + kScaleOffset);
                    } else {
#pragma unroll
                        for (int pc = 0; pc < 21; ++pc) ptx::cp_async_16(dst + pc * 16, rec[e] + 256 + pc * 16);
                    }
                }
                ptx::cp_async_arrive_noinc(&s.stg_full[st]);
                const uint32_t m0 = __ballot_sync(0xffffffffu, valid[0]);
                const uint32_t m1 = __ballot_sync(0xffffffffu, valid[1]);
                if (lane == 0) s.vmask[st] = (uint64_t)m0 | ((uint64_t)m1 << 32);
                __syncwarp();
                ptx::mbar_arrive(&s.stg_full[st]);
                ++j;
            }
        }
        // drain: every issued copy has landed before the CTA may exit
        for (int q = (j > kStages ? j - kStages : 0); q < j; ++q) wait(&s.stg_full[q % kStages], (q / kStages) & 1);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t kIdescQK = ptx::idesc_f32acc(1, 1, 128, kChunk);
        constexpr uint32_t kIdescPV = ptx::idesc_f32acc(1, 1, 128, kHalf, 1);
        bool ok = u.n_chunks == 0 || wait(&s.q_ready, 0);
        if (!ok) fail();
        auto issue_qk = [&](int jq) -> bool {
            const int xb = jq % kXBuf, sb = jq & 1;
            if (!wait(&s.x_full[xb], (jq / kXBuf) & 1)) return false;
            if (jq >= 2 && !wait(&s.s_free[sb], ((jq - 2) >> 1) & 1)) return false;
            ptx::tc_fence_after();
            if (lane == 0) {
                const uint32_t xa = ptx::smem_u32(s.x[xb]);
#pragma unroll
                for (int kk = 0; kk < kHalf / 16; ++kk)
                    ptx::mma_f16_ts(tmem + kColS + sb * kChunk, tmem + kColQ + kk * 8,
                                    ptx::desc_kmajor_sw128(xa + (kk >> 2) * kAtom + (kk & 3) * 32), kIdescQK,
                                    kk > 0 ? 1u : 0u);
                ptx::mma_commit(&s.s_full[sb]);
            }
            __syncwarp();
            return true;
        };
        auto issue_pv = [&](int jp) -> bool {
            const int xb = jp % kXBuf, pb = jp & 1;
            if (!wait(&s.p_full[pb], (jp >> 1) & 1)) return false;
            ptx::tc_fence_after();
            if (lane == 0) {
                const uint32_t xa = ptx::smem_u32(s.x[xb]);
                const uint32_t pa = ptx::smem_u32(s.p);
#pragma unroll
                for (int kk = 0; kk < kChunk / 16; ++kk)
                    ptx::mma_f16(tmem + kColO, ptx::desc_kmajor_sw128(pa + kk * 32),
                                 ptx::desc_mnmajor_sw128(xa + kk * 2048, kAtom, 1024), kIdescPV,
                                 (jp > 0 || kk > 0) ? 1u : 0u);
                ptx::mma_commit(&s.x_empty[xb]);
                ptx::mma_commit(&s.o_done[pb]);
            }
            __syncwarp();
            return true;
        };
        if (ok && u.n_chunks > 0 && !issue_qk(0)) { fail(); ok = false; }
        if (ok && u.n_chunks > 1 && !issue_qk(1)) { fail(); ok = false; }
        for (int j = 0; j < u.n_chunks && ok; ++j) {
            if (j + 2 < u.n_chunks && !issue_qk(j + 2)) { fail(); ok = false; break; }
            if (!issue_pv(j)) { fail(); ok = false; break; }
        }
        if (lane == 0) {
            ptx::mma_commit(&s.o_final);
            ptx::mma_commit(&s.mma_done);
        }
        __syncwarp();
        wait(&s.mma_done, 0);
    } else if (warp < 6) {
        // ------------------------------------------------------------ dequantise
        const int ct = threadIdx.x - 64;  // 0..127
        const int ci = ct >> 1;           // candidate row of the chunk
        const int half = ct & 1;          // local dims [128 half, 128 half + 128)
        bool ok = true;
        for (int j = 0; j < u.n_chunks && ok; ++j) {
            const int st = j % kStages, xb = j % kXBuf;
            if (!wait(&s.stg_full[st], (j / kStages) & 1)) { fail(); ok = false; break; }
            if (!wait(&s.x_empty[xb], ((j / kXBuf) & 1) ^ 1)) { fail(); ok = false; break; }
            const uint64_t mask = s.vmask[st];
            const bool valid = (mask >> ci) & 1ull;
            const uint8_t *slot = s.stage[st] + ci * kSlot;
            uint8_t *xrow = s.x[xb] + ci * 128;
            // this thread's two 64-dim blocks of the row: local dims [128 half, 128 half + 128)
            // rank 0: latent dims 128 half + ..., one multiplier (block `half`)
            // rank 1: half 0 -> latent 256..383 (block 2); half 1 -> latent 384..447
            //         (block 3) then the 64 rope dims (BF16, copied)
            uint4 v[2][8];
            if (valid) {
                const uint4 *codes = reinterpret_cast<const uint4 *>(slot + 128 * half);
                if (rank == 0 || half == 0) {
                    const float sc = *reinterpret_cast<const float *>(slot + (rank == 0 ? 256 + 4 * half : 320 + 8));
                    uint4 cv[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) cv[q] = codes[q];
#pragma unroll
                    for (int q = 0; q < 8; ++q) dequant16(cv[q], sc, v[q >> 2][(q & 3) * 2], v[q >> 2][(q & 3) * 2 + 1]);
                } else {
                    const float sc = *reinterpret_cast<const float *>(slot + 320 + 12);
                    uint4 cv[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) cv[q] = codes[q];
                    const uint4 *rope = reinterpret_cast<const uint4 *>(slot + 192);
#pragma unroll
                    for (int q = 0; q < 8; ++q) v[1][q] = rope[q];
#pragma unroll
                    for (int q = 0; q < 4; ++q) dequant16(cv[q], sc, v[0][2 * q], v[0][2 * q + 1]);
                }
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) v[0][q] = v[1][q] = make_uint4(0, 0, 0, 0);
            }
            store_atom_row(xrow + (2 * half) * kAtom, ci, v[0]);
            store_atom_row(xrow + (2 * half + 1) * kAtom, ci, v[1]);
            ptx::fence_proxy_async_smem();  // generic-proxy stores -> MMA (async proxy) reads
            if (ct == 0) s.smask[xb] = mask;
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(&s.stg_empty[st]);
                ptx::mbar_arrive(&s.x_full[xb]);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax / exchange / epilogue
        const int quarter = warp & 3;
        const int h = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const int r = u.r;
        bool ok = true;
        // Q half -> TMEM (BF16 pairs, lane = head)
        if (u.n_chunks > 0) {
            const uint4 *qg = reinterpret_cast<const uint4 *>(P.q + ((size_t)r * kHeads + h) * kDim + rank * kHalf);
#pragma unroll
            for (int piece = 0; piece < 4; ++piece) {
                uint32_t regs[32];
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const uint4 w4 = __ldg(qg + piece * 8 + v);
                    regs[4 * v] = w4.x;
                    regs[4 * v + 1] = w4.y;
                    regs[4 * v + 2] = w4.z;
                    regs[4 * v + 3] = w4.w;
                }
                ptx::tmem_st32(lane_base + kColQ + piece * 32, regs);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&s.q_ready);
        }
        const uint32_t recv_peer[2] = {ptx::mapa(ptx::smem_u32(s.recv[0]), peer),
                                       ptx::mapa(ptx::smem_u32(s.recv[1]), peer)};
        const uint32_t full_peer[2] = {ptx::mapa(ptx::smem_u32(&s.xchg_full[0]), peer),
                                       ptx::mapa(ptx::smem_u32(&s.xchg_full[1]), peer)};
        const uint32_t free_peer[2] = {ptx::mapa(ptx::smem_u32(&s.xchg_free[0]), peer),
                                       ptx::mapa(ptx::smem_u32(&s.xchg_free[1]), peer)};
        float m = -INFINITY, l = 0.f;  // running max and sum, log2 domain, sink not included
        // Sends this CTA's partial scores of chunk jj into the peer's recv
        // (st.async, completing bytes on the peer's xchg_full barrier) once the
        // peer has read chunk jj-2 out of that buffer, and arms the local
        // receive barrier of chunk jj.
        auto send = [&](int jj) -> bool {
            const int b2 = jj & 1;
            if (!wait(&s.s_full[b2], (jj >> 1) & 1)) return false;
            ptx::tc_fence_after();
            uint32_t sa[32], sb[32];
            ptx::tmem_ld32(lane_base + kColS + b2 * kChunk, sa);
            ptx::tmem_ld32(lane_base + kColS + b2 * kChunk + 32, sb);
            ptx::tmem_ld_wait();
            if (threadIdx.x == 192) ptx::mbar_arrive_expect_tx(&s.xchg_full[b2], 16 * kHeads * 16);
            if (jj >= 2 && !wait_cluster(&s.xchg_free[b2], ((jj - 2) >> 1) & 1)) return false;
#pragma unroll
            for (int cq = 0; cq < 8; ++cq) {
                ptx::st_async_v4(recv_peer[b2] + (uint32_t)((cq * kHeads + h) * 16),
                                 make_float4(__uint_as_float(sa[4 * cq]), __uint_as_float(sa[4 * cq + 1]),
                                             __uint_as_float(sa[4 * cq + 2]), __uint_as_float(sa[4 * cq + 3])),
                                 full_peer[b2]);
                ptx::st_async_v4(recv_peer[b2] + (uint32_t)(((8 + cq) * kHeads + h) * 16),
                                 make_float4(__uint_as_float(sb[4 * cq]), __uint_as_float(sb[4 * cq + 1]),
                                             __uint_as_float(sb[4 * cq + 2]), __uint_as_float(sb[4 * cq + 3])),
                                 full_peer[b2]);
            }
            return true;
        };
        if (u.n_chunks > 0 && !send(0)) { fail(); ok = false; }
        for (int j = 0; j < u.n_chunks && ok; ++j) {
            const int jb = j & 1, xb = j % kXBuf;
            if (j + 1 < u.n_chunks && !send(j + 1)) { fail(); ok = false; break; }
            if (!wait_cluster(&s.xchg_full[jb], (j >> 1) & 1)) { fail(); ok = false; break; }
            // own partial of chunk j from TMEM, then release the score buffer
            uint32_t sa[32], sb[32];
            ptx::tmem_ld32(lane_base + kColS + jb * kChunk, sa);
            ptx::tmem_ld32(lane_base + kColS + jb * kChunk + 32, sb);
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&s.s_free[jb]);
            float z[kChunk];
#pragma unroll
            for (int cq = 0; cq < 16; ++cq) {
                const float4 pv = s.recv[jb][cq * kHeads + h];
                const uint32_t *own = cq < 8 ? &sa[4 * cq] : &sb[4 * (cq - 8)];
                z[4 * cq + 0] = __uint_as_float(own[0]) + pv.x;
                z[4 * cq + 1] = __uint_as_float(own[1]) + pv.y;
                z[4 * cq + 2] = __uint_as_float(own[2]) + pv.z;
                z[4 * cq + 3] = __uint_as_float(own[3]) + pv.w;
            }
            // once every softmax thread has read recv[jb], the peer may refill it
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&s.rd_done[jb]);
            if (!wait(&s.rd_done[jb], (j >> 1) & 1)) { fail(); ok = false; break; }
            if (threadIdx.x == 192) ptx::mbar_arrive_remote(free_peer[jb]);
            if (!wait(&s.x_full[xb], (j / kXBuf) & 1)) { fail(); ok = false; break; }
            const uint64_t mask = s.smask[xb];
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < kChunk; ++c) {
                z[c] = ((mask >> c) & 1ull) ? z[c] * P.scale_log2 : -INFINITY;
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
                    // (PV(j-3) is done -- it freed X for chunk j -- so this barrier is at
                    // most one phase behind and the parity test is unambiguous.)
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
            // P(j) = 2^(z - m) as BF16 rows (K-major, 128-byte swizzle), once PV(j-1)
            // has finished reading the previous P
            if (j > 0 && !wait(&s.o_done[(j - 1) & 1], ((j - 1) >> 1) & 1)) { fail(); ok = false; break; }
            const float mref = (m == -INFINITY) ? 0.f : m;  // every z is -inf while m is
            float ps4[4] = {0.f, 0.f, 0.f, 0.f};
            uint8_t *prow = s.p + h * 128;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float p0 = ptx::ex2_approx(z[8 * c8 + 2 * i] - mref);
                    const float p1 = ptx::ex2_approx(z[8 * c8 + 2 * i + 1] - mref);
                    ps4[i] += p0 + p1;
                    w[i] = bf16x2_bits(p0, p1);
                }
                *reinterpret_cast<uint4 *>(prow + ((c8 ^ (h & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            l += (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
            ptx::fence_proxy_async_smem();  // P stores -> PV (async proxy) reads
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&s.p_full[jb]);
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
            __nv_bfloat16 *dst = (P.n_split == 1)
                                     ? P.out + ((size_t)r * kHeads + h) * kDim + rank * kHalf
                                     : P.part_o + (((size_t)r * P.n_split + u.split) * kHeads + h) * kDim + rank * kHalf;
#pragma unroll 1
            for (int piece = 0; piece < kHalf / 32; ++piece) {
                uint32_t o[32];
                if (u.n_chunks > 0) {
                    ptx::tmem_ld32(lane_base + kColO + piece * 32, o);
                    ptx::tmem_ld_wait();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                uint4 *d4 = reinterpret_cast<uint4 *>(dst + piece * 32);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    d4[v] = make_uint4(bf16x2_bits(__uint_as_float(o[8 * v + 0]) * factor, __uint_as_float(o[8 * v + 1]) * factor),
                                       bf16x2_bits(__uint_as_float(o[8 * v + 2]) * factor, __uint_as_float(o[8 * v + 3]) * factor),
                                       bf16x2_bits(__uint_as_float(o[8 * v + 4]) * factor, __uint_as_float(o[8 * v + 5]) * factor),
                                       bf16x2_bits(__uint_as_float(o[8 * v + 6]) * factor, __uint_as_float(o[8 * v + 7]) * factor));
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
    ptx::cluster_sync();  // no remote access to this CTA's shared memory after this point
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
}

// Folds the per-split normalised partials and the sink:
//   M = max(sink, m_s), den = e^{sink-M} + sum_s l_s e^{m_s-M},
//   out = sum_s l_s e^{m_s-M} o_s / den, lse = M + ln den   (log2 domain inside).
__global__ void __launch_bounds__(256)
attention_combine_kernel(const __nv_bfloat16 *__restrict__ part_o, const float2 *__restrict__ part_ml,
                         const float *__restrict__ sink, int n_split, __nv_bfloat16 *__restrict__ out,
                         float *__restrict__ lse) {
    const int r = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x * 8 + warp;
    const float sk = __ldg(sink + h) * kLog2e;
    float M = sk;
    for (int sp = 0; sp < n_split; ++sp) {
        const float2 ml = part_ml[((size_t)r * n_split + sp) * kHeads + h];
        if (ml.y > 0.f) M = fmaxf(M, ml.x);
    }
    float den = (sk == -INFINITY) ? 0.f : exp2f(sk - M);
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
    for (int sp = 0; sp < n_split; ++sp) {
        const float2 ml = part_ml[((size_t)r * n_split + sp) * kHeads + h];
        if (!(ml.y > 0.f)) continue;
        const float w = ml.y * exp2f(ml.x - M);
        den += w;
        const uint4 *src = reinterpret_cast<const uint4 *>(part_o + (((size_t)r * n_split + sp) * kHeads + h) * kDim) + lane * 2;
#pragma unroll
        for (int v = 0; v < 2; ++v) {
            const uint4 x = src[v];
            const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[8 * v + 2 * i] = fmaf(w, bf16_bits_to_float(static_cast<uint16_t>(wv[i] & 0xFFFFu)), acc[8 * v + 2 * i]);
                acc[8 * v + 2 * i + 1] = fmaf(w, bf16_bits_to_float(static_cast<uint16_t>(wv[i] >> 16)), acc[8 * v + 2 * i + 1]);
            }
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    uint4 *dst = reinterpret_cast<uint4 *>(out + ((size_t)r * kHeads + h) * kDim) + lane * 2;
#pragma unroll
    for (int v = 0; v < 2; ++v)
        dst[v] = make_uint4(bf16x2_bits(acc[8 * v + 0] * inv, acc[8 * v + 1] * inv),
                            bf16x2_bits(acc[8 * v + 2] * inv, acc[8 * v + 3] * inv),
                            bf16x2_bits(acc[8 * v + 4] * inv, acc[8 * v + 5] * inv),
                            bf16x2_bits(acc[8 * v + 6] * inv, acc[8 * v + 7] * inv));
    if (lane == 0) lse[(size_t)r * kHeads + h] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

// Splits per query so that about one CTA pair per two SMs is busy.
int choose_splits(int rows, int max_candidates) {
    const int chunks = (max_candidates + kChunk - 1) / kChunk;
    const int target = sm_count() / 2;
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

size_t attention_workspace_bytes(int B, int T, int max_candidates) {
    const int rows = B * T;
    return split_bytes(rows, choose_splits(rows, max_candidates));
}

cudaError_t launch_attention(const void *q, const float *sink, float scale, const csa_cache_desc &comp,
                             const void *ring, int R, int W, const int32_t *topk_idx, const int32_t *topk_cnt,
                             const int32_t *n_comp, int m_hca, const int32_t *q_pos, int B, int T, int k, bool hca,
                             int max_candidates, void *out, float *lse, void *ws, size_t ws_bytes, int *err,
                             cudaStream_t stream) {
    const int rows = B * T;
    const int n_split = choose_splits(rows, max_candidates);
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
    P.k = k;
    P.n_split = n_split;
    P.out = static_cast<__nv_bfloat16 *>(out);
    P.lse = lse;
    P.part_o = nullptr;
    P.part_ml = nullptr;
    P.err = err;
    if (n_split > 1) {
        const size_t need = split_bytes(rows, n_split);
        if (!ws || ws_bytes < need) return cudaErrorInvalidValue;
        const size_t po = (size_t)rows * n_split * kHeads * kDim * sizeof(__nv_bfloat16);
        P.part_o = static_cast<__nv_bfloat16 *>(ws);
        P.part_ml = reinterpret_cast<float2 *>(static_cast<uint8_t *>(ws) + (po + 255) / 256 * 256);
    }
    const size_t smem = sizeof(AttSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    count_launch();
    attention_tc_kernel<<<2 * rows * n_split, kThreads, smem, stream>>>(P);
    e = cudaGetLastError();
    if (e != cudaSuccess || n_split == 1) return e;
    count_launch();
    attention_combine_kernel<<<dim3(kHeads / 8, rows), 256, 0, stream>>>(P.part_o, P.part_ml, sink, n_split,
                                                                         P.out, lse);
    return cudaGetLastError();
}

int *error_word_for_current_device();

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
    cudaStream_t stream) {
    using namespace csa;
    const auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!q || !sink || !swa_ring || !topk_idx || !topk_cnt || !q_pos || !out || !lse) return CSA_ERR_INVALID_ARG;
    if (!a16(q) || !a16(swa_ring) || !a16(out) || !comp.base || !a16(comp.base) || comp.n_records <= 0 ||
        comp.seq_capacity <= 0)
        return CSA_ERR_INVALID_ARG;
    if (comp.block_table ? (!a16(comp.block_table) || comp.page_records <= 0 || comp.max_pages <= 0)
                         : (comp.seq_stride < 0 || (B > 1 && comp.seq_stride < comp.seq_capacity)))
        return CSA_ERR_INVALID_ARG;
    if (B < 1 || T < 1 || T > CSA_MAX_TOKENS_PER_SEQ || (int64_t)B * T > 65535 || k < 1 || W < 1 ||
        W > CSA_MAX_SWA_WINDOW || R < W || !(softmax_scale > 0.f))
        return CSA_ERR_INVALID_ARG;
    if (k > CSA_MAX_TOPK) return CSA_ERR_UNSUPPORTED;
    const size_t need = attention_workspace_bytes(B, T, k + CSA_MAX_SWA_WINDOW);
    if (need > kStaticScratchBytes) return CSA_ERR_UNSUPPORTED;  // beyond the static scratch: use the workspace call
    void *scratch = nullptr;
    if (need && static_scratch_address(&scratch) != cudaSuccess) return CSA_ERR_CUDA;
    const cudaError_t e = launch_attention(q, sink, softmax_scale, comp, swa_ring, R, W, topk_idx, topk_cnt, nullptr,
                                           1, q_pos, B, T, k, false, k + CSA_MAX_SWA_WINDOW, out, lse, scratch,
                                           need ? kStaticScratchBytes : 0, error_word_for_current_device(), stream);
    return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}
