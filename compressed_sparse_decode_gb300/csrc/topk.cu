// topk.cu -- top-k of the indexer logits over the visible entries
// ("DSV4 Audit", section B2; "ROADMAP -- Stage E", section E7: warp-level
// selection, no global lock).
//
// Radix select on order-preserving 32-bit keys: four 8-bit digit passes find
// the k-th largest key K* and how many entries equal to K* must be kept; a
// final pass in index order keeps every key > K* and the lowest-index entries
// equal to K*. Prefix sums are warp ballots plus one shared-memory scan, so no
// lock and no global atomic is involved. Output is in ascending index order.
#include "common.cuh"

namespace csa {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

// Block-wide exclusive prefix sum of a 0/1 flag; every thread must call it.
__device__ __forceinline__ int block_exclusive_scan(int flag, int *s_warp, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned bal = __ballot_sync(0xffffffffu, flag);
    const int rank = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) s_warp[warp] = __popc(bal);
    __syncthreads();
    if (warp == 0) {
        int v = s_warp[lane];
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        s_warp[lane] = incl - v;
        if (lane == 31) s_warp[32] = incl;
    }
    __syncthreads();
    const int res = s_warp[warp] + rank;
    total = s_warp[32];
    __syncthreads();
    return res;
}

__global__ void __launch_bounds__(kThreads)
topk_radix_kernel(const float *__restrict__ logits, const int32_t *__restrict__ q_pos,
                  const int32_t *__restrict__ n_comp, int T, int Ncap, int m, int k,
                  int32_t *__restrict__ idx_out, int32_t *__restrict__ cnt_out) {
    __shared__ uint32_t hist[256];
    __shared__ int s_warp[kWarps + 1];
    __shared__ uint32_t s_digit;
    __shared__ int s_remaining;

    const int r = blockIdx.x;
    const int b = r / T;
    const int tid = threadIdx.x;
    const float *row = logits + (size_t)r * Ncap;
    int32_t *out = idx_out + (size_t)r * k;
    const int nv = visible_entries(q_pos[r], m, n_comp[b], Ncap);

    if (nv <= k) {
        for (int i = tid; i < k; i += kThreads) out[i] = i < nv ? i : -1;
        if (tid == 0) cnt_out[r] = nv;
        return;
    }

    uint32_t prefix = 0, mask = 0;
    int remaining = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
        __syncthreads();
        for (int i = tid; i < nv; i += kThreads) {
            const uint32_t key = order_key(row[i]);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 0xFFu], 1u);
        }
        __syncthreads();
        if (tid < 32) {
            // lane l owns digits 255-8l .. 248-8l (descending order)
            int c[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = (int)hist[255 - (tid * 8 + j)];
                sum += c[j];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += u;
            }
            const int excl = incl - sum;
            const unsigned here = __ballot_sync(0xffffffffu, excl < remaining && remaining <= incl);
            if (tid == __ffs(here) - 1) {
                int cum = excl;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (cum + c[j] >= remaining) {
                        s_digit = 255u - (uint32_t)(tid * 8 + j);
                        s_remaining = remaining - cum;
                        break;
                    }
                    cum += c[j];
                }
            }
        }
        __syncthreads();
        prefix |= s_digit << shift;
        mask |= 0xFFu << shift;
        remaining = s_remaining;
        __syncthreads();
    }

    // prefix = K*; keep every key > K* and the first `remaining` keys == K*.
    int out_base = 0, eq_seen = 0;
    for (int start = 0; start < nv && out_base < k; start += kThreads) {
        const int i = start + tid;
        const uint32_t key = i < nv ? order_key(row[i]) : 0u;
        const int gt = (i < nv) && key > prefix;
        const int eq = (i < nv) && key == prefix;
        int eq_total, take_total;
        const int eq_rank = block_exclusive_scan(eq, s_warp, eq_total);
        const int take = gt || (eq && eq_seen + eq_rank < remaining);
        const int pos = block_exclusive_scan(take, s_warp, take_total);
        if (take && out_base + pos < k) out[out_base + pos] = i;
        out_base += take_total;
        eq_seen += eq_total;
    }
    if (tid == 0) cnt_out[r] = k;
}

}  // namespace

size_t topk_workspace_bytes(int, int, int, int) { return 0; }

cudaError_t launch_topk(const float *logits, const int32_t *q_pos, const int32_t *n_comp, int B, int T,
                        int Ncap, int m, int k, int32_t *idx_out, int32_t *cnt_out, void *, size_t,
                        cudaStream_t stream) {
    count_launch();
    topk_radix_kernel<<<B * T, kThreads, 0, stream>>>(logits, q_pos, n_comp, T, Ncap, m, k, idx_out, cnt_out);
    return cudaGetLastError();
}

}  // namespace csa
