// topk.cu -- top-k of the indexer logits over the visible entries
// ("DSV4 Audit", section B2; "ROADMAP -- Stage E", section E7: top-k with
// warp-level reductions and no global lock).
//
// Two kernels. The 8-bit radix select below (topk_radix8_kernel) serves every
// row whose keys fit in the shared memory of one cluster (up to 360448
// entries); the 11-bit cluster kernel that follows serves longer rows, its
// keys read from global memory in every pass when they do not fit.
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

}  // namespace

size_t topk_workspace_bytes(int, int, int, int) { return 0; }

namespace {

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

cudaError_t launch_topk(const float *logits, const int32_t *q_pos, const int32_t *n_comp, int B, int T, int Ncap,
                        int m, int k, int32_t *idx_out, int32_t *cnt_out, void *, size_t, cudaStream_t stream) {
    // Rows whose keys fit in the shared memory of a cluster (up to 8 x 1024
    // threads x 44 keys): the 8-bit radix select, 256 threads a CTA up to
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
