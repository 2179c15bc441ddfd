// topk.cu -- top-k of the indexer logits over the visible entries
// ("DSV4 Audit", section B2; "ROADMAP -- Stage E", section E7: top-k with
// warp-level reductions and no global lock).
//
// One row (query token) per cluster of 8 CTAs; CTA rank c owns the slice
// [c * slice, (c + 1) * slice) of the row. Each CTA loads its slice once into
// shared memory as order-preserving 32-bit keys, then a radix select finds the
// k-th largest key K* in three digit passes (bits 31..21, 20..10, 9..0):
// per pass, every CTA builds a histogram of its matching keys in its own
// shared memory (warp-aggregated with __match_any_sync); after a cluster
// barrier each thread sums its bins over the 8 CTAs through distributed shared
// memory, and every CTA picks the same digit. Finally each CTA keeps its keys
// > K* and, in index order, the lowest-index keys == K* still needed; the
// per-CTA counts are exchanged through rank 0 so every CTA writes at its
// global offset and the output is in ascending index order. No lock and no
// global atomic is used.
#include "common.cuh"
#include "ptx.cuh"

namespace csa {

namespace {

constexpr int kCtas = 8;                 // CTAs per row (a portable cluster)
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;              // 11-bit digits (the last pass uses 10)
constexpr int kMaxResident = 32768;      // keys per CTA held in shared memory

struct TopkShared {
    alignas(16) uint32_t local[3][kBins];  // this CTA's histogram, one buffer per pass (read by every CTA)
    alignas(16) uint32_t view[kBins];      // the cluster-wide histogram of the current pass
    alignas(16) int counts[kCtas][2];  // rank 0's copy: (keys > K*, keys == K*) per CTA
    int scan[kWarps + 1];
    int wsum[2][kWarps];
    uint32_t digit;
    int remaining;
};

// Block-wide exclusive prefix sum of a 0/1 flag; every thread must call it.
__device__ __forceinline__ int block_exclusive_scan(int flag, int *s_warp, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned bal = __ballot_sync(0xffffffffu, flag);
    const int rank = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) s_warp[warp] = __popc(bal);
    __syncthreads();
    if (warp == 0) {
        const int v = lane < kWarps ? s_warp[lane] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        if (lane < kWarps) s_warp[lane] = incl - v;
        if (lane == 31) s_warp[kWarps] = incl;
    }
    __syncthreads();
    const int res = s_warp[warp] + rank;
    total = s_warp[kWarps];
    __syncthreads();
    return res;
}

__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int v) {
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__global__ void __launch_bounds__(kThreads)
topk_cluster_kernel(const float *__restrict__ logits, const int32_t *__restrict__ q_pos,
                    const int32_t *__restrict__ n_comp, int T, int Ncap, int m, int k, int slice, int resident,
                    int32_t *__restrict__ idx_out, int32_t *__restrict__ cnt_out) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    TopkShared &s = *reinterpret_cast<TopkShared *>(smem_raw);
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem_raw + sizeof(TopkShared));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t crank = ptx::cluster_ctarank();
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

    const int lo = crank * slice;
    const int hi = min(nv, lo + slice);
    auto key_at = [&](int i) -> uint32_t {  // i in [lo, hi)
        return resident ? keys[i - lo] : order_key(__ldg(row + i));
    };
    if (resident)
        for (int i = lo + tid; i < hi; i += kThreads) keys[i - lo] = order_key(__ldg(row + i));
    for (int i = tid; i < 3 * kBins; i += kThreads) (&s.local[0][0])[i] = 0u;
    __syncthreads();

    uint32_t prefix = 0, mask = 0;
    int remaining = k;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);  // digits: bits 31..21, 20..10, 9..0
        const uint32_t dmask = pass == 2 ? 0x3FFu : 0x7FFu;
        // local histogram of keys matching the digits chosen so far
        for (int base = lo; base < hi; base += kThreads) {
            const int i = base + tid;
            const bool in = i < hi;
            const uint32_t key = in ? key_at(i) : 0u;
            const bool match = in && (key & mask) == prefix;
            const unsigned act = __ballot_sync(0xffffffffu, match);
            if (match) {
                const uint32_t d = (key >> shift) & dmask;
                const unsigned peers = __match_any_sync(act, d);
                if (lane == __ffs(peers) - 1) atomicAdd(&s.local[pass][d], (uint32_t)__popc(peers));
            }
        }
        ptx::cluster_sync();  // every CTA's histogram of this pass is complete
        // the cluster-wide histogram: each thread sums 4 bins over the 8 CTAs
        // (one vector load of distributed shared memory per CTA)
        if (tid < (int)(dmask + 1) / 4) {
            const uint32_t off = ptx::smem_u32(&s.local[pass][4 * tid]);
            uint4 acc = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int c = 0; c < kCtas; ++c) {
                const uint4 v = ld_cluster_v4(ptx::mapa(off, c));
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            reinterpret_cast<uint4 *>(s.view)[tid] = acc;
        }
        __syncthreads();
        if (warp == 0) {
            const int nb = (int)dmask + 1, per = nb / 32;  // bins per lane, descending digits
            int sum = 0;
            for (int j = 0; j < per; ++j) sum += (int)s.view[nb - 1 - (lane * per + j)];
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            const int excl = incl - sum;
            const unsigned here = __ballot_sync(0xffffffffu, excl < remaining && remaining <= incl);
            if (lane == __ffs(here) - 1) {
                int cum = excl;
                for (int j = 0; j < per; ++j) {
                    const int d = nb - 1 - (lane * per + j);
                    const int c = (int)s.view[d];
                    if (cum + c >= remaining) {
                        s.digit = (uint32_t)d;
                        s.remaining = remaining - cum;
                        break;
                    }
                    cum += c;
                }
            }
        }
        __syncthreads();
        prefix |= s.digit << shift;
        mask |= dmask << shift;
        remaining = s.remaining;
        __syncthreads();
    }

    // prefix = K*; keep every key > K* and the first `remaining` keys == K* (index order)
    int gt = 0, eq = 0;
    for (int i = lo + tid; i < hi; i += kThreads) {
        const uint32_t key = key_at(i);
        gt += key > prefix;
        eq += key == prefix;
    }
    // block totals of both counts
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        gt += __shfl_xor_sync(0xffffffffu, gt, o);
        eq += __shfl_xor_sync(0xffffffffu, eq, o);
    }
    if (lane == 0) {
        s.wsum[0][warp] = gt;
        s.wsum[1][warp] = eq;
    }
    __syncthreads();
    int tot_gt = 0, tot_eq = 0;
    for (int w = 0; w < kWarps; ++w) {
        tot_gt += s.wsum[0][w];
        tot_eq += s.wsum[1][w];
    }
    const uint32_t counts0 = ptx::mapa(ptx::smem_u32(&s.counts[0][0]), 0);
    if (tid == 0) {
        st_cluster_s32(counts0 + crank * 8, tot_gt);
        st_cluster_s32(counts0 + crank * 8 + 4, tot_eq);
    }
    ptx::cluster_sync();
    if (tid < kCtas * 2 / 4) reinterpret_cast<uint4 *>(s.view)[tid] = ld_cluster_v4(counts0 + tid * 16);
    __syncthreads();
    int base = 0, eq_before = 0;
    for (int c = 0; c < (int)crank; ++c) {
        const int cg = (int)s.view[2 * c];
        const int ce = (int)s.view[2 * c + 1];
        const int take_eq = min(max(remaining - eq_before, 0), ce);
        base += cg + take_eq;
        eq_before += ce;
    }
    int out_pos = base, eq_seen = eq_before;
    for (int start = lo; start < hi; start += kThreads) {
        const int i = start + tid;
        const uint32_t key = i < hi ? key_at(i) : 0u;
        const int g = (i < hi) && key > prefix;
        const int e = (i < hi) && key == prefix;
        int e_total, t_total;
        const int e_rank = block_exclusive_scan(e, s.scan, e_total);
        const int take = g || (e && eq_seen + e_rank < remaining);
        const int pos = block_exclusive_scan(take, s.scan, t_total);
        if (take && out_pos + pos < k) out[out_pos + pos] = i;
        out_pos += t_total;
        eq_seen += e_total;
    }
    if (crank == 0 && tid == 0) cnt_out[r] = k;
    ptx::cluster_sync();  // no CTA leaves while another may still read rank 0's counts
}

}  // namespace

size_t topk_workspace_bytes(int, int, int, int) { return 0; }

cudaError_t launch_topk(const float *logits, const int32_t *q_pos, const int32_t *n_comp, int B, int T, int Ncap,
                        int m, int k, int32_t *idx_out, int32_t *cnt_out, void *, size_t, cudaStream_t stream) {
    const int slice = (Ncap + kCtas - 1) / kCtas;
    const int resident = slice <= kMaxResident ? 1 : 0;
    const size_t smem = sizeof(TopkShared) + (resident ? (size_t)slice * sizeof(uint32_t) : 0);
    cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B * T * kCtas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launch();
    e = cudaLaunchKernelEx(&cfg, topk_cluster_kernel, logits, q_pos, n_comp, T, Ncap, m, k, slice, resident, idx_out,
                           cnt_out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace csa
