// topk.cu -- top-k of the indexer logits over the visible entries
// ("DSV4 Audit", section B2; "ROADMAP -- Stage E", section E7: top-k with
// warp-level reductions and no global lock).
//
// Three kernels. Rows of up to 32768 entries take one CTA each with the keys
// in registers (topk_row_kernel, at the end); longer rows whose keys fit in
// the shared memory of one cluster (up to 360448 entries) take the 8-bit
// radix select over a cluster (topk_radix8_kernel); the 11-bit cluster kernel
// described next serves longer rows still, its keys read from global memory
// in every pass when they do not fit.
//
// Cluster kernel: one row (query token) per cluster of 8 CTAs of 512 threads
// (1024 for rows above 64K entries); CTA rank c owns the slice
// [c * slice, (c + 1) * slice) of the row, and thread t of a CTA owns the
// contiguous run of E = slice / threads entries starting at t * E (kept in
// shared memory transposed, keys[j][t], so every access is conflict-free). The
// CTA loads its slice once as order-preserving 32-bit keys; a radix select
// then finds the k-th largest key K* in three digit passes (bits 31..21,
// 20..10, 9..0): per pass every CTA builds a histogram of its matching keys in
// its own shared memory, and after a cluster barrier each thread sums 4 bins
// over the 8 CTAs through distributed shared memory; a block-wide scan over
// the bins (largest digit first) picks the digit, identically in every CTA.
// Finally each CTA keeps its keys > K* and, in index order, the lowest-index
// keys == K* still needed: per-thread counts are scanned, the per-CTA totals
// are exchanged through rank 0, and every thread writes its run at its global
// offset, so the output is in ascending index order. No lock and no global
// atomic is used.
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace csa {

namespace {

constexpr int kCtas = 8;                 // CTAs per row (a portable cluster)
// Threads per CTA: 512, or 1024 for rows long enough that 512 threads would
// hold more than kRunSplit entries each (the per-thread loops of the three
// passes and the compaction are the kernel's serial work).
constexpr int kMaxThreads = 1024;
constexpr int kRunSplit = 16;
constexpr int kBins = 2048;              // 11-bit digits (the last pass uses 10)
constexpr int kMaxRun = 64;             // entries per thread held in shared memory

struct TopkShared {
    alignas(16) uint32_t local[3][kBins];  // this CTA's histogram, one buffer per pass (read by every CTA)
    alignas(16) int counts[kCtas][2];      // rank 0's copy: (keys > K*, keys == K*) per CTA
    alignas(16) int peer_counts[kCtas][2];
    alignas(16) uint32_t reduced[3][kBins / kCtas];  // this CTA's range of the cluster-wide histogram
    int range_total[3][kCtas];                       // written by every CTA: its range's total
    int wsum[kMaxThreads / 32];
    uint32_t digit;
    int remaining;
};

// Block-wide exclusive prefix sum of a uint32 (modular); every thread must call it.
template <int kThreads>
__device__ __forceinline__ uint32_t block_exclusive_sum_u32(uint32_t v, int *wsum, uint32_t &total) {
    constexpr int kWarps = kThreads / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) wsum[warp] = (int)incl;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t x = (uint32_t)wsum[w];
        before += w < warp ? x : 0u;
        all += x;
    }
    __syncthreads();
    total = all;
    return before + incl - v;
}

__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int v) {
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

template <int kThreads>
__global__ void __launch_bounds__(kThreads)
topk_cluster_kernel(const float *__restrict__ logits, const int32_t *__restrict__ q_pos,
                    const int32_t *__restrict__ n_comp, int T, int Ncap, int m, int k, int run, int resident,
                    int32_t *__restrict__ idx_out, int32_t *__restrict__ cnt_out) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    TopkShared &s = *reinterpret_cast<TopkShared *>(smem_raw);
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem_raw + sizeof(TopkShared));  // [run][kThreads]
    const int tid = threadIdx.x;
    const uint32_t crank = ptx::cluster_ctarank();
    ptx::griddep_wait();               // the logits (previous kernel in the stream) are complete and visible
    const int r = blockIdx.x / kCtas;
    const int b = r / T;
    const float *row = logits + (size_t)r * Ncap;
    int32_t *out = idx_out + (size_t)r * k;
    const int nv = visible_entries(__ldg(q_pos + r), m, __ldg(n_comp + b), Ncap);

    if (nv <= k) {
        // every visible entry is selected; CTAs split the k output slots
        const int per = (k + kCtas - 1) / kCtas;
        for (int i = crank * per + tid; i < min(k, (int)(crank + 1) * per); i += kThreads) out[i] = i < nv ? i : -1;
        if (crank == 0 && tid == 0) cnt_out[r] = nv;
        return;  // uniform over the cluster: no shared memory of another CTA is touched
    }

    const int slice = run * kThreads;
    const int mine = crank * slice + tid * run;  // first entry of this thread's run
    const int n_my = max(0, min(run, nv - mine));
    auto key_j = [&](int j) -> uint32_t {
        return resident ? keys[j * kThreads + tid] : order_key(__ldg(row + mine + j));
    };
    if (resident) {
        // 16-byte loads where the run is whole and aligned (rows of a multiple
        // of 4 entries, runs of a multiple of 4), scalar loads otherwise
        int j = 0;
        if ((Ncap & 3) == 0 && (run & 3) == 0) {
            const float4 *r4 = reinterpret_cast<const float4 *>(row + mine);
            const uint64_t policy = ptx::l2_policy_evict_first();  // the logits are read once
            for (; j + 3 < n_my; j += 4) {
                const uint4 w = ptx::ldg_v4_policy(r4 + (j >> 2), policy);
                const float4 v = make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                                             __uint_as_float(w.w));
                keys[(j + 0) * kThreads + tid] = order_key(v.x);
                keys[(j + 1) * kThreads + tid] = order_key(v.y);
                keys[(j + 2) * kThreads + tid] = order_key(v.z);
                keys[(j + 3) * kThreads + tid] = order_key(v.w);
            }
        }
        for (; j < n_my; ++j) keys[j * kThreads + tid] = order_key(__ldg(row + mine + j));
    }
    for (int i = tid; i < 3 * kBins; i += kThreads) (&s.local[0][0])[i] = 0u;
    __syncthreads();

    uint32_t prefix = 0, mask = 0;
    int remaining = k;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);  // digits: bits 31..21, 20..10, 9..0
        const uint32_t dmask = pass == 2 ? 0x3FFu : 0x7FFu;
        for (int j = 0; j < n_my; ++j) {
            const uint32_t key = key_j(j);
            if ((key & mask) == prefix) atomicAdd(&s.local[pass][(key >> shift) & dmask], 1u);
        }
        ptx::cluster_sync();  // every CTA's histogram of this pass is complete
        // Reduce-scatter: CTA c sums bins [c * per, (c + 1) * per) over the 8
        // CTAs (one vector load of distributed shared memory per CTA and 4
        // bins) and publishes its range total to every CTA.
        const int nb = (int)dmask + 1, per = nb / kCtas;
        int part = 0;
        if (tid < per / 4) {
            const uint32_t off = ptx::smem_u32(&s.local[pass][crank * per + 4 * tid]);
            uint4 v[kCtas];
#pragma unroll
            for (int c = 0; c < kCtas; ++c) v[c] = ld_cluster_v4(ptx::mapa(off, c));
            uint4 acc = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int c = 0; c < kCtas; ++c) {
                acc.x += v[c].x;
                acc.y += v[c].y;
                acc.z += v[c].z;
                acc.w += v[c].w;
            }
            reinterpret_cast<uint4 *>(s.reduced[pass])[tid] = acc;
            part = (int)(acc.x + acc.y + acc.z + acc.w);
        }
        // this CTA's range total: the partial sums sit in the first per/4 <= 64 threads
        if (tid < 64) {
            const int w = (int)__reduce_add_sync(0xffffffffu, (unsigned)part);
            if ((tid & 31) == 0) s.wsum[tid >> 5] = w;
        }
        __syncthreads();
        if (tid < kCtas)
            st_cluster_s32(ptx::mapa(ptx::smem_u32(&s.range_total[pass][crank]), tid), s.wsum[0] + s.wsum[1]);
        ptx::cluster_sync();  // every range total has arrived
        // The range holding the `remaining`-th largest matching key (ranges of
        // larger digits first); every CTA reads that range's bins and picks the
        // same digit.
        int owner = 0, above = 0;
        for (int c = kCtas - 1; c >= 0; --c) {
            const int t = s.range_total[pass][c];
            if (above + t >= remaining) {
                owner = c;
                break;
            }
            above += t;
        }
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            const int bpl = per / 32;  // 8 or 4 bins per lane, lane 0 takes the largest
            int cnt[8];
            const uint32_t roff = ptx::mapa(ptx::smem_u32(&s.reduced[pass][per - bpl * (lane + 1)]), owner);
            const uint4 hi4 = ld_cluster_v4(roff + (bpl == 8 ? 16u : 0u));
            const uint4 lo4 = bpl == 8 ? ld_cluster_v4(roff) : make_uint4(0, 0, 0, 0);
            cnt[0] = (int)hi4.w; cnt[1] = (int)hi4.z; cnt[2] = (int)hi4.y; cnt[3] = (int)hi4.x;
            cnt[4] = (int)lo4.w; cnt[5] = (int)lo4.z; cnt[6] = (int)lo4.y; cnt[7] = (int)lo4.x;
            int sum = 0;
            for (int q = 0; q < bpl; ++q) sum += cnt[q];
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            const int need = remaining - above;
            const int excl = incl - sum;
            if (sum > 0 && excl < need && need <= incl) {
                int cum = excl;
                for (int q = 0; q < bpl; ++q) {
                    if (cum + cnt[q] >= need) {
                        s.digit = (uint32_t)(owner * per + per - 1 - (bpl * lane + q));
                        s.remaining = need - cum;
                        break;
                    }
                    cum += cnt[q];
                }
            }
        }
        __syncthreads();
        prefix |= s.digit << shift;
        mask |= dmask << shift;
        remaining = s.remaining;
    }

    // prefix = K*: keep every key > K* and the first `remaining` keys == K* in index order
    int gt = 0, eq = 0;
    for (int j = 0; j < n_my; ++j) {
        const uint32_t key = key_j(j);
        gt += key > prefix;
        eq += key == prefix;
    }
    int gt_excl, eq_excl, tot_gt, tot_eq;
    if (slice < 65536) {
        // one scan of (gt << 16 | eq): a CTA holds fewer than 65536 entries,
        // so the low half never carries into the high half
        uint32_t tot_packed;
        const uint32_t excl = block_exclusive_sum_u32<kThreads>(((uint32_t)gt << 16) | (uint32_t)eq, s.wsum, tot_packed);
        gt_excl = (int)(excl >> 16);
        eq_excl = (int)(excl & 0xFFFFu);
        tot_gt = (int)(tot_packed >> 16);
        tot_eq = (int)(tot_packed & 0xFFFFu);
    } else {
        uint32_t t0, t1;
        gt_excl = (int)block_exclusive_sum_u32<kThreads>((uint32_t)gt, s.wsum, t0);
        eq_excl = (int)block_exclusive_sum_u32<kThreads>((uint32_t)eq, s.wsum, t1);
        tot_gt = (int)t0;
        tot_eq = (int)t1;
    }
    const uint32_t counts0 = ptx::mapa(ptx::smem_u32(&s.counts[0][0]), 0);
    if (tid == 0) {
        st_cluster_s32(counts0 + crank * 8, tot_gt);
        st_cluster_s32(counts0 + crank * 8 + 4, tot_eq);
    }
    ptx::cluster_sync();
    if (tid < kCtas * 2 / 4) reinterpret_cast<uint4 *>(&s.peer_counts[0][0])[tid] = ld_cluster_v4(counts0 + tid * 16);
    __syncthreads();
    int base = 0, eq_before = 0;
    for (int c = 0; c < (int)crank; ++c) {
        const int ce = s.peer_counts[c][1];
        base += s.peer_counts[c][0] + min(max(remaining - eq_before, 0), ce);
        eq_before += ce;
    }
    // keys == K* are taken in index order while the budget lasts, so the
    // threads before this one took min(budget, eq_excl) of them
    const int budget = max(remaining - eq_before, 0);
    int pos = base + gt_excl + min(budget, eq_excl);
    int eq_seen = eq_before + eq_excl;
    for (int j = 0; j < n_my; ++j) {
        const uint32_t key = key_j(j);
        bool keep = key > prefix;
        if (key == prefix) {
            keep = eq_seen < remaining;
            ++eq_seen;
        }
        if (keep && pos < k) out[pos++] = mine + j;
    }
    if (crank == 0 && tid == 0) cnt_out[r] = k;
    ptx::cluster_sync();  // no CTA leaves while another may still read rank 0's counts
}

// ------------------------------------------------------------------ 8-bit radix select
//
// One row per cluster of C CTAs (256 threads each up to 65536 entries, 1024
// above): C is the smallest power of two up to 8 that holds the row at <= 8
// keys a thread, lowered (C = 7, 6, ...) while the rows' clusters would not
// all be resident at once and the keys still fit (<= 44 a thread). The radix
// select takes four 8-bit digit passes
// (bits 31..24, 23..16, 15..8, 7..0 of the order-preserving key). The top
// digit of float keys is the sign and the high exponent bits, so nearly all
// keys share two or three values of it and a histogram of it serialises on a
// few counters; but the k-th largest key lies near the largest: pass 0 first
// takes the row's largest key and counts, in registers, the keys whose top
// digit is within 4 of its, and only if the k-th key lies below that window
// does it build the histogram. Each warp counts into its own 256-bin
// histogram, which keeps collisions within a warp. Per pass the warp histograms are summed
// into the CTA's, the C CTA histograms are summed through distributed shared
// memory after one cluster barrier (double-buffered by pass parity, so one
// barrier per pass suffices; each thread issues its C remote loads together,
// one round trip), and one warp picks the digit, identically in every CTA. The compaction is the one above: keys > K*, then the
// lowest-index keys == K* while the budget lasts, in ascending index order.
constexpr int kR8MaxRun = 44;  // keys per thread held in shared memory (212 KB at 1024 threads)
constexpr int kR8MaxCtas = 8;
constexpr int kR8TargetRun = 8;  // keys per thread the cluster width aims at (up to 8 CTAs)

template <int kThreads>
struct alignas(16) Radix8Shared {  // the keys follow it as 16-byte groups
    static constexpr int kWarps = kThreads / 32;
    uint32_t whist[kWarps][256];       // per-warp histograms of the current pass
    // Every CTA's partial results, each written into every CTA of the cluster
    // by its owner before a cluster barrier, so that after the barrier every
    // CTA reads them from its own shared memory (no remote loads on the
    // critical path, and no remote access at all after the last barrier).
    uint16_t peer_hist[2][kR8MaxCtas][256];  // per-CTA histogram of a pass (<= 45056 keys a CTA), by pass parity
    uint32_t peer_top[kR8MaxCtas];           // per-CTA largest key
    uint32_t peer_win[kR8MaxCtas][4];        // per-CTA counts of the top-digit window
    int peer_counts[kR8MaxCtas][2];          // per-CTA (keys > K*, keys == K*)
    uint32_t hist[256];                // the row's histogram of the current pass
    int wsum[kWarps];
    uint32_t wmax[kWarps];             // per-warp largest key
    int wwin[kWarps][4];               // per-warp counts of the keys in the top-digit window
    uint32_t digit;
    int remaining;
    int fallback;                      // pass 0 needs the histogram
};

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared::cluster.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}


template <int kThreads>
__global__ void __launch_bounds__(kThreads)
topk_radix8_kernel(const float *__restrict__ logits, const int32_t *__restrict__ q_pos,
                   const int32_t *__restrict__ n_comp, int T, int Ncap, int m, int k, int run,
                   int32_t *__restrict__ idx_out, int32_t *__restrict__ cnt_out) {
    using S = Radix8Shared<kThreads>;
    static_assert(sizeof(S) % 16 == 0, "the keys after the shared struct must be 16-byte aligned");
    extern __shared__ __align__(16) uint8_t smem_raw[];
    S &s = *reinterpret_cast<S *>(smem_raw);
    // keys4[g][t]: the g-th group of 4 consecutive entries of thread t's run
    uint4 *keys4 = reinterpret_cast<uint4 *>(smem_raw + sizeof(S));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t crank = ptx::cluster_ctarank(), nctas = cluster_nctarank();
    const bool clustered = nctas > 1;
    auto sync_all = [&]() {
        if (clustered) ptx::cluster_sync();
        else __syncthreads();
    };
    ptx::griddep_wait();  // the logits (previous kernel in the stream) are complete and visible
    const int r = blockIdx.x / (int)nctas;
    const int b = r / T;
    const float *row = logits + (size_t)r * Ncap;
    int32_t *out = idx_out + (size_t)r * k;
    const int nv = visible_entries(__ldg(q_pos + r), m, __ldg(n_comp + b), Ncap);

    if (nv <= k) {
        // every visible entry is selected; the CTAs split the k output slots
        const int per = (k + (int)nctas - 1) / (int)nctas;
        for (int i = (int)crank * per + tid; i < min(k, (int)(crank + 1) * per); i += kThreads) out[i] = i < nv ? i : -1;
        if (crank == 0 && tid == 0) cnt_out[r] = nv;
        return;  // uniform over the cluster: no shared memory of another CTA is touched
    }

    const int slice = run * kThreads;
    const int mine = (int)crank * slice + tid * run;  // first entry of this thread's run
    const int n_my = max(0, min(run, nv - mine));
    const int groups = (n_my + 3) >> 2;               // groups of 4 holding this thread's visible entries
    {
        // 16-byte cp.async (no L1 staging) when the row allows it, else scalar loads
        if ((Ncap & 3) == 0) {
            const uint64_t policy = ptx::l2_policy_evict_first();  // the logits are read once
            for (int g = 0; g < groups; ++g)
                ptx::cp_async_16_hint(&keys4[g * kThreads + tid], row + mine + 4 * g, policy);
            ptx::cp_async_commit();
            ptx::cp_async_wait<0>();
        } else {
            uint32_t *k1 = reinterpret_cast<uint32_t *>(keys4);
            for (int j = 0; j < n_my; ++j) k1[((j >> 2) * kThreads + tid) * 4 + (j & 3)] = __float_as_uint(__ldg(row + mine + j));
        }
        // float bits -> order-preserving keys, in place; entries past the
        // visible range of a partial group become 0 (below every real key)
        for (int g = 0; g < groups; ++g) {
            uint4 v = keys4[g * kThreads + tid];
            const int j0 = 4 * g;
            v.x = j0 + 0 < n_my ? order_key(__uint_as_float(v.x)) : 0u;
            v.y = j0 + 1 < n_my ? order_key(__uint_as_float(v.y)) : 0u;
            v.z = j0 + 2 < n_my ? order_key(__uint_as_float(v.z)) : 0u;
            v.w = j0 + 3 < n_my ? order_key(__uint_as_float(v.w)) : 0u;
            keys4[g * kThreads + tid] = v;
        }
    }
    // (a key of 0 belongs to no float: the padding never matches a digit
    // below, since the window and the passes only count keys whose top digit
    // is at least the selected one, and 0 is counted nowhere else)

    uint32_t prefix = 0, mask = 0;
    int remaining = k;
    // `field` of this CTA's shared memory, in CTA c of the cluster
    auto in_cta = [&](const void *field, int c) { return ptx::mapa(ptx::smem_u32(field), (uint32_t)c); };
    // ---- pass 0 through the window below the largest key's top digit
    {
        uint32_t mx = 0u;
        for (int g = 0; g < groups; ++g) {
            const uint4 v = keys4[g * kThreads + tid];
            mx = max(max(mx, max(v.x, v.y)), max(v.z, v.w));
        }
        mx = __reduce_max_sync(0xffffffffu, mx);
        if (lane == 0) s.wmax[warp] = mx;
        __syncthreads();
        if (tid < (int)nctas) {  // thread c gives CTA c this CTA's largest key
            uint32_t m2 = 0u;
            for (int w = 0; w < S::kWarps; ++w) m2 = max(m2, s.wmax[w]);
            st_cluster_u32(in_cta(&s.peer_top[crank], tid), m2);
        }
        sync_all();
        uint32_t top = 0u;
        for (int c = 0; c < (int)nctas; ++c) top = max(top, s.peer_top[c]);
        const uint32_t tdig = top >> 24;
        // four 8-bit counters in one register (a thread holds <= 44 keys)
        uint32_t packed = 0u;
        auto win = [&](uint32_t key) {
            const uint32_t d = tdig - (key >> 24);
            if (key != 0u && d < 4u) packed += 1u << (8u * d);
        };
        for (int g = 0; g < groups; ++g) {
            const uint4 v = keys4[g * kThreads + tid];
            win(v.x);
            win(v.y);
            win(v.z);
            win(v.w);
        }
#pragma unroll
        for (int d = 0; d < 4; ++d) {
            const int c = (int)__reduce_add_sync(0xffffffffu, (packed >> (8 * d)) & 0xFFu);
            if (lane == 0) s.wwin[warp][d] = c;
        }
        __syncthreads();
        if (tid < 4 * (int)nctas) {  // thread 4 c + d gives CTA c this CTA's count of digit tdig - d
            const int d = tid & 3;
            int c = 0;
            for (int w = 0; w < S::kWarps; ++w) c += s.wwin[w][d];
            st_cluster_u32(in_cta(&s.peer_win[crank][d], tid >> 2), (uint32_t)c);
        }
        sync_all();
        if (tid == 0) {
            int cum = 0, found = 0;
            for (int d = 0; d < 4 && !found; ++d) {
                int cd = 0;
                for (int c = 0; c < (int)nctas; ++c) cd += (int)s.peer_win[c][d];
                if ((int)tdig - d >= 0 && cum + cd >= remaining) {
                    s.digit = tdig - (uint32_t)d;
                    s.remaining = remaining - cum;
                    found = 1;
                }
                cum += cd;
            }
            s.fallback = !found;
        }
        __syncthreads();
        if (!s.fallback) {
            prefix = s.digit << 24;
            mask = 0xFF000000u;
            remaining = s.remaining;
        }
    }
    const int first_pass = s.fallback ? 0 : 1;  // uniform over the cluster
#pragma unroll 1
    for (int pass = first_pass; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        uint32_t *wh = s.whist[warp];
#pragma unroll
        for (int i = 0; i < 8; ++i) wh[lane * 8 + i] = 0u;
        __syncwarp();
        auto count = [&](uint32_t key) {
            if (key != 0u && (key & mask) == prefix) atomicAdd(&wh[(key >> shift) & 0xFFu], 1u);
        };
        for (int g = 0; g < groups; ++g) {
            const uint4 v = keys4[g * kThreads + tid];
            count(v.x);
            count(v.y);
            count(v.z);
            count(v.w);
        }
        __syncthreads();  // every warp histogram of this pass is complete
        if (tid < 256) {
            // this CTA's count of bin `tid`, given to every CTA (buffer by
            // pass parity: a CTA reads buffer p & 1 before it arrives at the
            // barrier of pass p + 1, and nobody writes it again before then)
            uint32_t sum = 0;
#pragma unroll 8
            for (int w = 0; w < S::kWarps; ++w) sum += s.whist[w][tid];
            for (int c = 0; c < (int)nctas; ++c)
                st_cluster_u16(in_cta(&s.peer_hist[pass & 1][crank][tid], c), (uint16_t)sum);
        }
        sync_all();  // every CTA's histogram of this pass has arrived
        if (tid < 256) {
            uint32_t total = 0;
            for (int c = 0; c < (int)nctas; ++c) total += s.peer_hist[pass & 1][c][tid];
            s.hist[tid] = total;
        }
        __syncthreads();
        // the digit of the `remaining`-th largest matching key: lane L holds
        // bins 255 - 8 L .. 248 - 8 L (largest first)
        if (warp == 0) {
            int cnt[8], sum = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                cnt[q] = (int)s.hist[255 - 8 * lane - q];
                sum += cnt[q];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            const int excl = incl - sum;
            if (sum > 0 && excl < remaining && remaining <= incl) {
                int cum = excl;
                for (int q = 0; q < 8; ++q) {
                    if (cum + cnt[q] >= remaining) {
                        s.digit = (uint32_t)(255 - 8 * lane - q);
                        s.remaining = remaining - cum;
                        break;
                    }
                    cum += cnt[q];
                }
            }
        }
        __syncthreads();
        prefix |= s.digit << shift;
        mask |= 0xFFu << shift;
        remaining = s.remaining;
    }

    // prefix = K*: keep every key > K* and the first `remaining` keys == K* in index order
    int gt = 0, eq = 0;
    for (int g = 0; g < groups; ++g) {
        const uint4 v = keys4[g * kThreads + tid];
        gt += (v.x > prefix) + (v.y > prefix) + (v.z > prefix) + (v.w > prefix);
        eq += (v.x == prefix) + (v.y == prefix) + (v.z == prefix) + (v.w == prefix);
    }
    // one scan of (gt << 16 | eq): a CTA holds fewer than 65536 entries, so
    // the low half never carries into the high half
    uint32_t tot_packed;
    const uint32_t excl = block_exclusive_sum_u32<kThreads>(((uint32_t)gt << 16) | (uint32_t)eq, s.wsum, tot_packed);
    const int gt_excl = (int)(excl >> 16), eq_excl = (int)(excl & 0xFFFFu);
    int base = 0, eq_before = 0;
    if (clustered) {
        if (tid < (int)nctas) {  // thread c gives CTA c this CTA's totals
            st_cluster_u32(in_cta(&s.peer_counts[crank][0], tid), tot_packed >> 16);
            st_cluster_u32(in_cta(&s.peer_counts[crank][1], tid), tot_packed & 0xFFFFu);
        }
        // the last barrier: no CTA touches another's shared memory after it,
        // so each may leave as soon as it is done
        ptx::cluster_sync();
        for (int c = 0; c < (int)crank; ++c) {
            const int ce = s.peer_counts[c][1];
            base += s.peer_counts[c][0] + min(max(remaining - eq_before, 0), ce);
            eq_before += ce;
        }
    }
    // keys == K* are taken in index order while the budget lasts, so the
    // threads before this one took min(budget, eq_excl) of them
    const int budget = max(remaining - eq_before, 0);
    int pos = base + gt_excl + min(budget, eq_excl);
    int eq_seen = eq_before + eq_excl;
    auto emit = [&](uint32_t key, int j) {
        bool keep = key > prefix;
        if (key == prefix) {
            keep = eq_seen < remaining;
            ++eq_seen;
        }
        if (keep && pos < k) out[pos++] = mine + j;
    };
    for (int g = 0; g < groups; ++g) {
        const uint4 v = keys4[g * kThreads + tid];
        emit(v.x, 4 * g);
        emit(v.y, 4 * g + 1);
        emit(v.z, 4 * g + 2);
        emit(v.w, 4 * g + 3);
    }
    if (crank == 0 && tid == 0) cnt_out[r] = k;
}

// ------------------------------------------------------------------ one CTA per row
//
// Rows of up to 32768 entries: one CTA of 1024 threads per row, the row's keys
// in registers (KPT a thread), so that no step needs a cluster barrier: at
// these sizes the barriers and remote round trips of the cluster kernels above
// cost more than their passes' work. Warp w holds the contiguous chunk
// [w * 32 * KPT, (w + 1) * 32 * KPT) of the row, loaded as coalesced 16-byte
// groups: lane L holds the chunk's groups j * 32 + L (j < KPT / 4).
//
// The radix select takes two 16-bit digits. The first is counted into a
// 65536-bin shared-memory histogram (two 16-bit counters a word: a row has at
// most 32768 keys) with one predicated shared-memory add per key, no per-key
// branch; a descending scan over it (thread t owns 64 bins, thread order =
// descending bin order; one block scan of the per-thread totals, then the
// owner's warp walks its 64 bins) finds the bin of the k-th largest key. The
// keys of that bin, usually a few dozen, are listed and ranked against each
// other by their low 16 bits (up to kRowMaxList of them; more are counted
// into a second histogram the same way). The compaction builds a keep mask a
// thread and gives every kept key its slot in closed form, in index order
// (warp, group j, lane, element): per group a warp scan of byte-packed kept
// counts, on top of the kept counts of the warps before, walking only the
// set bits. Keys equal to K* are kept up to the budget, lowest index first:
// when the budget cuts them (ties), the index of the last one kept is found
// first, in the same index order.
struct RowShared {
    int wsum[32];
    int wtot[32];
    uint32_t sel;  // the selected bin of the current pass
    int rem;       // keys still needed from that bin
    int cnt;       // keys in that bin
    int ithr;      // index of the last key == K* kept
    int nlist;     // keys listed for the second digit (short-list path)
};
constexpr int kRowMaxList = 256;  // second digit by ranking a list of at most this many keys
constexpr int kRowThreads = 1024;
constexpr size_t kRowHistBytes = 65536 * 2;  // 65536 16-bit counters

__device__ __forceinline__ void red_shared_add_if(uint32_t saddr, uint32_t v, bool c) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q red.shared.add.u32 [%0], %1;\n\t}" ::"r"(saddr), "r"(v),
        "r"((uint32_t)c)
        : "memory");
}
__device__ __forceinline__ uint32_t byte_sum(uint32_t x) { return (x & 0xFFu) + ((x >> 8) & 0xFFu) + ((x >> 16) & 0xFFu) + (x >> 24); }

// Inclusive warp scan of four byte counters packed in a word (each column's
// sum stays below 256).
__device__ __forceinline__ uint32_t warp_scan_bytes(uint32_t v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

// (Not inlined: called twice with the 32 keys a thread live in registers, it
// kept the kernel from spilling.)
// The bin of the `need`-th largest counted key (1 <= need <= counted keys):
// s.sel, s.rem (keys still needed from it), s.cnt (keys in it). Every thread
// calls it; the histogram is complete and visible on entry, s.* on return.
__device__ __noinline__ void select_bin(const uint32_t *h32, int need, RowShared &s, int tid, int lane, int warp) {
    const int u = kRowThreads - 1 - tid;  // thread order = descending bins
    const uint4 *w4 = reinterpret_cast<const uint4 *>(h32 + 32 * u);
    uint32_t acc = 0u;  // per half: at most 32768 counts, so the low half never carries
#pragma unroll 2
    for (int i = 0; i < 8; ++i) {
        const uint4 v = w4[(i + lane) & 7];  // rotated: lanes of a quarter warp read distinct banks
        acc += v.x + v.y + v.z + v.w;
    }
    const int total = (int)((acc & 0xFFFFu) + (acc >> 16));
    int incl = total;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s.wsum[warp] = incl;
    __syncthreads();
    const int base = (int)__reduce_add_sync(0xffffffffu, lane < warp ? (unsigned)s.wsum[lane] : 0u);
    const int cum = base + incl - total;
    // the warp whose thread holds it walks that thread's 64 bins, two a lane
    // (lane L: bins 64 u' + 63 - 2 L, 64 u' + 62 - 2 L, largest first)
    const unsigned own = __ballot_sync(0xffffffffu, total > 0 && cum < need && need <= cum + total);
    if (own) {  // uniform over the warp
        const int src = __ffs(own) - 1;
        const int uo = kRowThreads - 1 - (warp * 32 + src);
        const int c0 = __shfl_sync(0xffffffffu, cum, src);
        const uint32_t x = h32[32 * uo + 31 - lane];
        const int hi = (int)(x >> 16), lo = (int)(x & 0xFFFFu);
        int in = hi + lo;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, in, o);
            if (lane >= o) in += t;
        }
        const int before = c0 + in - hi - lo;
        if (before < need && need <= before + hi + lo) {
            const bool top = need <= before + hi;
            s.sel = (uint32_t)(64 * uo + 63 - 2 * lane - (top ? 0 : 1));
            s.rem = need - (top ? before : before + hi);
            s.cnt = top ? hi : lo;
        }
    }
    __syncthreads();
}

// What one CTA of topk_row_kernel selects from: a whole row; one slice of
// kRowThreads * KPT entries of a longer row (first stage: the slice's top k,
// indices into the row with their order-preserving keys, unused slots -1 and
// key 0, and the slice's k-th key); or the candidates of all S slices of a
// row, S * k of them (second stage: the row's top k among them).
enum RowMode { kModeWhole = 0, kModeSlice = 1, kModeMerge = 2 };

// The two-stage scratch of `slots` = rows * S candidate lists of k: indices
// int32 [slots][k], then (16-byte aligned) keys uint32 [slots][k], then the
// slices' k-th keys uint32 [slots].
__host__ __device__ __forceinline__ size_t cand_keys_offset(size_t slots, int k) {
    return (slots * (size_t)k + 3) & ~(size_t)3;
}

template <int KPT, int kMode>
__global__ void __launch_bounds__(kRowThreads, 1)
topk_row_kernel(const float *__restrict__ logits, const int32_t *__restrict__ q_pos,
                const int32_t *__restrict__ n_comp, int T, int Ncap, int m, int k, int S, int32_t *__restrict__ cand,
                int32_t *__restrict__ idx_out, int32_t *__restrict__ cnt_out) {
    static_assert(KPT % 4 == 0 && KPT <= 32, "keys a thread: groups of 4, one bit each in a 32-bit mask");
    constexpr int G = KPT / 4;
    extern __shared__ __align__(16) uint32_t h32[];  // the histogram, kRowHistBytes
    __shared__ RowShared s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint4 *h4 = reinterpret_cast<uint4 *>(h32);
    const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 0; i < (int)(kRowHistBytes / 16 / kRowThreads); ++i) h4[i * kRowThreads + tid] = zero4;
    if (tid == 0) s.nlist = 0;
    ptx::griddep_wait();  // the logits (and candidates) of the previous kernel in the stream are complete and visible
    const int r = kMode == kModeSlice ? (int)blockIdx.x / S : (int)blockIdx.x;
    const int b = r / T;
    const float *lrow = logits + (size_t)r * Ncap;
    const int nv = visible_entries(__ldg(q_pos + r), m, __ldg(n_comp + b), Ncap);
    // this CTA's entries [0, n): row entry base + i (whole row, slice) or the
    // row entry named by candidate i (merge)
    int n = nv, base = 0;
    int32_t *out = idx_out + (size_t)r * k;
    const size_t slots = kMode == kModeSlice ? gridDim.x : (size_t)gridDim.x * S;  // rows * S
    uint32_t *const ckeys = reinterpret_cast<uint32_t *>(cand + cand_keys_offset(slots, k));
    uint32_t *const cthr = ckeys + slots * k;
    const int32_t *crow = cand + (size_t)r * S * k;
    uint32_t *kout = nullptr;  // slice: the candidates' keys
    if (kMode == kModeSlice) {
        base = ((int)blockIdx.x - r * S) * kRowThreads * KPT;
        n = min(max(nv - base, 0), kRowThreads * KPT);
        out = cand + (size_t)blockIdx.x * k;
        kout = ckeys + (size_t)blockIdx.x * k;
    } else if (kMode == kModeMerge) {
        n = S * k;
    }

    if ((kMode == kModeSlice ? n : nv) <= k) {
        // every visible entry (of the slice) is selected
        const int all = kMode == kModeSlice ? n : nv;
        for (int i = tid; i < k; i += kRowThreads) {
            out[i] = i < all ? base + i : -1;
            if (kMode == kModeSlice) kout[i] = i < all ? order_key(__ldg(lrow + base + i)) : 0u;
        }
        if (kMode != kModeSlice && tid == 0) cnt_out[r] = nv;
        if (kMode == kModeSlice && tid == 0) cthr[blockIdx.x] = 0u;  // no k-th key: no bound on the row's
        return;
    }

    const int chunk = warp * 32 * KPT;
    auto first = [&](int j) { return chunk + 4 * (j * 32 + lane); };  // first entry of group j
    uint32_t key[KPT];
    // Merge: the candidates' indices, copied into shared memory behind the
    // histogram while the selection runs (read back for the kept keys only).
    int32_t *const sidx = reinterpret_cast<int32_t *>(h32 + kRowHistBytes / 4);
    const bool idx_in_smem = kMode == kModeMerge && KPT <= 16 && (n & 3) == 0;
    if (idx_in_smem) {
        const uint64_t policy = ptx::l2_policy_evict_first();
        for (int c = tid; c < n / 4; c += kRowThreads) ptx::cp_async_16_hint(sidx + 4 * c, crow + 4 * c, policy);
        ptx::cp_async_commit();
    }
    if (kMode == kModeMerge) {
        // the candidates' keys (unused slots hold key 0)
        const uint32_t *krow = ckeys + (size_t)r * S * k;
        if ((n & 3) == 0) {  // with k % 4 == 0 every row of keys is 16-byte aligned
#pragma unroll
            for (int j = 0; j < G; ++j) {
                uint4 v = zero4;
                if (first(j) < n) v = __ldg(reinterpret_cast<const uint4 *>(krow + first(j)));
                key[4 * j] = v.x;
                key[4 * j + 1] = v.y;
                key[4 * j + 2] = v.z;
                key[4 * j + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < KPT; ++i) {
                const int e = first(i >> 2) + (i & 3);
                key[i] = e < n ? __ldg(krow + e) : 0u;
            }
        }
    } else {
        const float *row = lrow + base;
        if ((Ncap & 3) == 0) {
            // rows of a multiple of 4 entries: every group inside the row is a whole, aligned float4
            const uint64_t policy = ptx::l2_policy_evict_first();  // the logits are read once
            uint4 w[G];
#pragma unroll
            for (int j = 0; j < G; ++j) {
                w[j] = zero4;
                if (first(j) < n) w[j] = ptx::ldg_v4_policy(row + first(j), policy);
            }
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const uint32_t v[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) key[4 * j + e] = order_key(__uint_as_float(v[e]));
            }
        } else {
#pragma unroll
            for (int j = 0; j < G; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = first(j) + e;
                    key[4 * j + e] = i < n ? order_key(__ldg(row + i)) : 0u;
                }
        }
        if (first(G - 1) + 3 >= n) {
            // the visible end falls in this thread's groups: entries past it become key 0
#pragma unroll
            for (int j = 0; j < G; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) key[4 * j + e] = first(j) + e < n ? key[4 * j + e] : 0u;
        }
    }
    // (entries past the visible range hold key 0, below every real key and
    // counted in neither pass; K* is a real key)
    __syncthreads();  // the zeroed histogram

    // Keys below `floor` are counted nowhere (and so never selected). Merge:
    // the largest of the slices' k-th keys, which the row's k-th key is not
    // below (that slice alone holds k keys at or above it); it drops most of
    // the candidates, which crowd into few bins of the first digit.
    uint32_t floor = 1u;
    if (kMode == kModeMerge)
        floor = max(1u, __reduce_max_sync(0xffffffffu, lane < S ? __ldg(cthr + (size_t)r * S + lane) : 0u));
    const uint32_t hbase = ptx::smem_u32(h32);
    // ---- pass 1: the top 16 bits (bin = key >> 16: word key >> 17, half bit 16)
#pragma unroll
    for (int i = 0; i < KPT; ++i)
        red_shared_add_if(hbase + ((key[i] >> 17) << 2), 1u << ((key[i] >> 12) & 16u), key[i] >= floor);
    __syncthreads();
    select_bin(h32, k, s, tid, lane, warp);
    const uint32_t hi16 = s.sel;
    const int need = s.rem;
    if (s.cnt <= kRowMaxList) {  // uniform
        // ---- pass 2, short list: the few keys of that bin, ranked by their low
        // 16 bits (the histogram's memory is free from here on)
        const int n = s.cnt;
#pragma unroll
        for (int i = 0; i < KPT; ++i)
            if (key[i] >= floor && (key[i] >> 16) == hi16) h32[atomicAdd(&s.nlist, 1)] = key[i] & 0xFFFFu;
        __syncthreads();
        if (tid < n) {
            const uint32_t v = h32[tid];
            int gt = 0, ge = 0;
            for (int i = 0; i < n; ++i) {
                const uint32_t x = h32[i];
                gt += x > v ? 1 : 0;
                ge += x >= v ? 1 : 0;
            }
            if (gt < need && need <= ge) {  // every thread holding the selected value writes the same
                s.sel = v;
                s.rem = need - gt;
                s.cnt = ge - gt;
            }
        }
        __syncthreads();
    } else {
#pragma unroll
        for (int i = 0; i < (int)(kRowHistBytes / 16 / kRowThreads); ++i) h4[i * kRowThreads + tid] = zero4;
        __syncthreads();
        // ---- pass 2: the low 16 bits of the keys in that bin
#pragma unroll
        for (int i = 0; i < KPT; ++i)
            red_shared_add_if(hbase + ((key[i] & 0xFFFFu) >> 1 << 2), 1u << ((key[i] & 1u) << 4),
                              key[i] >= floor && (key[i] >> 16) == hi16);
        __syncthreads();
        select_bin(h32, need, s, tid, lane, warp);
    }
    const uint32_t kstar = (hi16 << 16) | s.sel;
    const int budget = s.rem;  // keys == K* kept, of s.cnt
    if (kMode == kModeSlice && tid == 0) cthr[blockIdx.x] = kstar;  // the slice's k-th key
    if (kMode == kModeSlice) {
        // the keys into the (now unused) histogram memory, by entry, for the
        // kept ones' candidate keys (each thread reads back only its own)
#pragma unroll
        for (int j = 0; j < G; ++j)
            *reinterpret_cast<uint4 *>(h32 + first(j)) = make_uint4(key[4 * j], key[4 * j + 1], key[4 * j + 2], key[4 * j + 3]);
    }
    // keep: bit 4 j + e for the key of group j, element e
    uint32_t keep = 0u;
    if (budget == s.cnt) {  // uniform: every key == K* is kept
#pragma unroll
        for (int i = 0; i < KPT; ++i) keep |= (key[i] >= kstar ? 1u : 0u) << i;
    } else {
        // ---- the budget cuts the keys == K* (ties): find the index of the last one kept
        uint32_t gtm = 0u, eqm = 0u;
#pragma unroll
        for (int i = 0; i < KPT; ++i) {
            gtm |= (key[i] > kstar ? 1u : 0u) << i;
            eqm |= (key[i] == kstar ? 1u : 0u) << i;
        }
        uint32_t pk[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < G; ++j) pk[j >> 2] |= (uint32_t)__popc((eqm >> (4 * j)) & 0xFu) << (8 * (j & 3));
        const uint32_t in0 = warp_scan_bytes(pk[0], lane), in1 = warp_scan_bytes(pk[1], lane);
        const uint32_t t0 = __shfl_sync(0xffffffffu, in0, 31), t1 = __shfl_sync(0xffffffffu, in1, 31);
        if (lane == 0) s.wtot[warp] = (int)(byte_sum(t0) + byte_sum(t1));
        __syncthreads();
        const int before = (int)__reduce_add_sync(0xffffffffu, lane < warp ? (unsigned)s.wtot[lane] : 0u);
        if (before < budget && budget <= before + s.wtot[warp]) {  // uniform over the warp
            int left = budget - before;  // the left-th key == K* of this warp, in index order
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const uint32_t tj = ((j < 4 ? t0 : t1) >> (8 * (j & 3))) & 0xFFu;
                const uint32_t ij = ((j < 4 ? in0 : in1) >> (8 * (j & 3))) & 0xFFu;
                const uint32_t nib = (eqm >> (4 * j)) & 0xFu;
                const int ex = (int)ij - __popc(nib);
                if (left > 0 && left <= (int)tj && ex < left && left <= (int)ij) {
                    // this lane holds it: the (left - ex)-th set bit of its group
                    int c = left - ex;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if ((nib >> e) & 1u) {
                            if (--c == 0) s.ithr = first(j) + e;
                        }
                    }
                }
                left -= left > 0 ? (int)tj : 0;
            }
        }
        __syncthreads();
        const int ithr = s.ithr;
        keep = gtm;
#pragma unroll
        for (int i = 0; i < KPT; ++i) keep |= ((eqm >> i) & 1u) && first(i >> 2) + (i & 3) <= ithr ? 1u << i : 0u;
    }

    if (idx_in_smem) ptx::cp_async_wait<0>();  // made visible to the block by the barrier below

    // ---- compaction: keys > K*, and keys == K* up to the budget
    uint32_t pk[2] = {0u, 0u};  // kept keys per group, bytes (groups 0-3, 4-7)
#pragma unroll
    for (int j = 0; j < G; ++j) pk[j >> 2] |= (uint32_t)__popc((keep >> (4 * j)) & 0xFu) << (8 * (j & 3));
    const uint32_t in0 = warp_scan_bytes(pk[0], lane), in1 = G > 4 ? warp_scan_bytes(pk[1], lane) : 0u;
    const uint32_t t0 = __shfl_sync(0xffffffffu, in0, 31), t1 = __shfl_sync(0xffffffffu, in1, 31);
    if (lane == 0) s.wtot[warp] = (int)(byte_sum(t0) + byte_sum(t1));
    __syncthreads();
    const int wbase = (int)__reduce_add_sync(0xffffffffu, lane < warp ? (unsigned)s.wtot[lane] : 0u);
    const uint32_t ex0 = in0 - pk[0], ex1 = in1 - pk[1];  // kept keys of the lanes before, per group (bytes)
    // every kept key (about k / 1024 a thread): its slot = the warps before + the
    // groups before + the lanes before in its group + its group's keys before it
    for (uint32_t mk = keep; mk != 0u; mk &= mk - 1u) {
        const int bit = __ffs(mk) - 1, j = bit >> 2;
        const uint32_t sh = 8u * (uint32_t)(j & 3), below = (1u << sh) - 1u;
        const int groups_before = j < 4 ? (int)__dp4a(t0 & below, 0x01010101u, 0u)
                                        : (int)(__dp4a(t0, 0x01010101u, 0u) + __dp4a(t1 & below, 0x01010101u, 0u));
        const int lanes_before = (int)(((j < 4 ? ex0 : ex1) >> sh) & 0xFFu);
        const int pos = wbase + groups_before + lanes_before + __popc(keep & (0xFu << (4 * j)) & ((1u << bit) - 1u));
        const int i = first(j) + (bit & 3);
        if (pos < k) {
            out[pos] = kMode == kModeMerge ? (idx_in_smem ? sidx[i] : __ldg(crow + i)) : base + i;
            if (kMode == kModeSlice) kout[pos] = h32[i];
        }
    }
    if (kMode != kModeSlice && tid == 0) cnt_out[r] = k;
}


template <int kThreads>
cudaError_t launch_t(const float *logits, const int32_t *q_pos, const int32_t *n_comp, int B, int T, int Ncap, int m,
                     int k, int32_t *idx_out, int32_t *cnt_out, cudaStream_t stream) {
    const int per_cta = (Ncap + kCtas - 1) / kCtas;
    const int run = (per_cta + kThreads - 1) / kThreads;
    const int resident = run <= kMaxRun ? 1 : 0;
    const size_t smem = sizeof(TopkShared) + (resident ? (size_t)run * kThreads * sizeof(uint32_t) : 0);
    cudaError_t e =
        set_max_dynamic_smem_once(reinterpret_cast<const void *>(topk_cluster_kernel<kThreads>), (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B * T * kCtas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start before the indexer ends
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    count_launch();
    e = cudaLaunchKernelEx(&cfg, topk_cluster_kernel<kThreads>, logits, q_pos, n_comp, T, Ncap, m, k, run, resident,
                           idx_out, cnt_out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

// Clusters of `kernel` (launched as `cfg`, one cluster's worth of CTAs) that
// the device holds at once, looked up once per device, kernel and size.
int max_active_clusters(const void *kernel, cudaLaunchConfig_t cfg, int ctas) {
    struct Entry {
        const void *kernel;
        int dev, ctas;
        size_t smem;
        int n;
    };
    static Entry cache[32];
    static int used = 0;
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].kernel == kernel && cache[i].dev == dev && cache[i].ctas == ctas &&
            cache[i].smem == cfg.dynamicSmemBytes)
            return cache[i].n;
    int n = 0;
    cfg.gridDim = dim3(ctas);
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();  // a failed query reads as "does not fit"
        n = 0;
    }
    if (used < 32) cache[used++] = {kernel, dev, ctas, cfg.dynamicSmemBytes, n};
    return n;
}

template <int kThreads>
cudaError_t launch_r8(const float *logits, const int32_t *q_pos, const int32_t *n_comp, int B, int T, int Ncap, int m,
                      int k, int32_t *idx_out, int32_t *cnt_out, cudaStream_t stream) {
    const void *kernel = reinterpret_cast<const void *>(topk_radix8_kernel<kThreads>);
    auto run_for = [&](int c) {
        const int r = ((Ncap + c - 1) / c + kThreads - 1) / kThreads;
        return (r + 3) & ~3;  // whole groups of 4 (16-byte copies)
    };
    int ctas = 1;
    while ((Ncap + ctas - 1) / ctas > kThreads * kR8TargetRun && ctas < kR8MaxCtas) ctas *= 2;
    if (run_for(ctas) > kR8MaxRun) return cudaErrorInvalidValue;  // rows longer than the kernel holds
    const size_t smem_max = sizeof(Radix8Shared<kThreads>) + (size_t)kR8MaxRun * kThreads * sizeof(uint32_t);
    cudaError_t e = set_max_dynamic_smem_once(kernel, (int)smem_max);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start before the indexer ends
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    auto configure = [&](int c) {
        attr[1].val.clusterDim.x = c;
        cfg.dynamicSmemBytes = sizeof(Radix8Shared<kThreads>) + (size_t)run_for(c) * kThreads * sizeof(uint32_t);
    };
    // All rows' clusters should be resident at once: a second wave doubles
    // the time (measured for 16 rows of 262144 entries in 8-CTA clusters of
    // one SM each: 15 clusters resident, 28 -> 55 us). Fewer, fuller CTAs per
    // row fit more clusters beside each other.
    configure(ctas);
    if (ctas > 1 && max_active_clusters(kernel, cfg, ctas) < B * T) {
        for (int c = ctas - 1; c >= 2 && run_for(c) <= kR8MaxRun; --c) {
            configure(c);
            if (max_active_clusters(kernel, cfg, c) >= B * T) {
                ctas = c;
                break;
            }
        }
        configure(ctas);
    }
    const int run = run_for(ctas);
    cfg.gridDim = dim3(B * T * ctas);
    count_launch();
    e = cudaLaunchKernelEx(&cfg, topk_radix8_kernel<kThreads>, logits, q_pos, n_comp, T, Ncap, m, k, run, idx_out,
                           cnt_out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

namespace {

template <int KPT, int kMode>
cudaError_t launch_row(const float *logits, const int32_t *q_pos, const int32_t *n_comp, int rows, int ctas, int T,
                       int Ncap, int m, int k, int S, int32_t *cand, int32_t *idx_out, int32_t *cnt_out,
                       cudaStream_t stream) {
    const void *kernel = reinterpret_cast<const void *>(topk_row_kernel<KPT, kMode>);
    // merge with up to 16384 candidates: their indices after the histogram
    const size_t smem = kRowHistBytes + (kMode == kModeMerge && KPT <= 16 ? sizeof(int32_t) * kRowThreads * KPT : 0);
    cudaError_t e = set_max_dynamic_smem_once(kernel, (int)smem);
    if (e != cudaSuccess) return e;
    (void)rows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kRowThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start before its predecessor ends
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launch();
    e = cudaLaunchKernelEx(&cfg, topk_row_kernel<KPT, kMode>, logits, q_pos, n_comp, T, Ncap, m, k, S, cand, idx_out,
                           cnt_out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Rows longer than one CTA holds, cut into S slices of kRowSlice entries:
// the slices' candidates (S * k of them) must fit one CTA too.
constexpr int kRowSlice = kRowThreads * 32;
int row_slices(int Ncap, int k) {
    if (Ncap <= kRowSlice) return 0;
    const int S = (Ncap + kRowSlice - 1) / kRowSlice;
    return (int64_t)S * k <= kRowSlice ? S : 0;
}

}  // namespace

size_t topk_workspace_bytes(int B, int T, int Ncap, int k) {
    // two-stage rows: the slices' candidates (indices, keys) and k-th keys
    if (B < 1 || T < 1 || k < 1) return 0;
    const int S = row_slices(Ncap, k);
    if (!S) return 0;
    const size_t slots = (size_t)B * T * S;
    return sizeof(uint32_t) * (cand_keys_offset(slots, k) + slots * k + slots);
}

cudaError_t launch_topk(const float *logits, const int32_t *q_pos, const int32_t *n_comp, int B, int T, int Ncap,
                        int m, int k, int32_t *idx_out, int32_t *cnt_out, void *workspace, size_t,
                        cudaStream_t stream) {
    // Rows of up to 32768 entries: one CTA a row, keys in registers (8, 16 or
    // 32 a thread).
    const int rows = B * T;
    if (Ncap <= kRowThreads * 8)
        return launch_row<8, kModeWhole>(logits, q_pos, n_comp, rows, rows, T, Ncap, m, k, 0, nullptr, idx_out, cnt_out,
                                        stream);
    if (Ncap <= kRowThreads * 16)
        return launch_row<16, kModeWhole>(logits, q_pos, n_comp, rows, rows, T, Ncap, m, k, 0, nullptr, idx_out,
                                         cnt_out, stream);
    if (Ncap <= kRowThreads * 32)
        return launch_row<32, kModeWhole>(logits, q_pos, n_comp, rows, rows, T, Ncap, m, k, 0, nullptr, idx_out,
                                         cnt_out, stream);
    // Longer rows whose slices' candidates fit one CTA: two stages, the top k
    // of every 32768-entry slice (one CTA a slice), then the top k of those
    // candidates (one CTA a row). Exact: a key that its slice drops has k keys
    // of the slice before it in (logit, lower index) order, so the row's top k
    // does not hold it either.
    if (const int S = row_slices(Ncap, k)) {
        int32_t *cand = static_cast<int32_t *>(workspace);
        cudaError_t e = launch_row<32, kModeSlice>(logits, q_pos, n_comp, rows, rows * S, T, Ncap, m, k, S, cand,
                                                  nullptr, nullptr, stream);
        if (e != cudaSuccess) return e;
        if (S * k <= kRowThreads * 16)
            return launch_row<16, kModeMerge>(logits, q_pos, n_comp, rows, rows, T, Ncap, m, k, S, cand, idx_out,
                                             cnt_out, stream);
        return launch_row<32, kModeMerge>(logits, q_pos, n_comp, rows, rows, T, Ncap, m, k, S, cand, idx_out, cnt_out,
                                         stream);
    }
    // Longer rows whose keys fit in the shared memory of a cluster (up to 8 x
    // 1024 threads x 44 keys): the 8-bit radix select, 256 threads a CTA up to
    // 65536 entries, 1024 above. Measured against the 11-bit cluster kernel
    // (events around 20 calls on rotating inputs): 8.1 against 14.2 us for
    // 256-entry rows, 13.6 against 14.3 us for 8192, 18.8 against 19.9 us for
    // 32768, 37.4 against 58.7 us for 262144 (where 8-CTA clusters of one SM
    // each left one of the 16 rows for a second wave). Longer rows: the
    // cluster kernel, whose keys may stay in global memory.
    if (Ncap <= kR8MaxCtas * 1024 * kR8MaxRun) {
        if (Ncap <= kR8MaxCtas * 256 * 32)
            return launch_r8<256>(logits, q_pos, n_comp, B, T, Ncap, m, k, idx_out, cnt_out, stream);
        return launch_r8<1024>(logits, q_pos, n_comp, B, T, Ncap, m, k, idx_out, cnt_out, stream);
    }
    const int per_cta = (Ncap + kCtas - 1) / kCtas;
    if ((per_cta + 511) / 512 > kRunSplit)
        return launch_t<1024>(logits, q_pos, n_comp, B, T, Ncap, m, k, idx_out, cnt_out, stream);
    return launch_t<512>(logits, q_pos, n_comp, B, T, Ncap, m, k, idx_out, cnt_out, stream);
}

}  // namespace csa
