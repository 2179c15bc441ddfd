// gather.cu -- packed candidate records [top-k entries] ++ [SWA window]
// ("DSV4 Audit", section A3; "ROADMAP -- Stage E", section E1: one fused
// gather straight from the FP8 cache, block-table strided, no dequantisation).
#include "common.cuh"

namespace csa {

namespace {

constexpr int kWarpsPerCta = 8;
constexpr int kChunks = kRecBytes / 16;  // 37 x 16 B per record

// One warp per output slot; lanes move the record as 16-byte vectors.
__global__ void __launch_bounds__(kWarpsPerCta * 32)
gather_kernel(CacheView comp, const uint8_t *__restrict__ ring, int R, int W,
              const int32_t *__restrict__ topk_idx, const int32_t *__restrict__ topk_cnt,
              const int32_t *__restrict__ q_pos, int T, int k, uint8_t *__restrict__ kv_out,
              int32_t *__restrict__ kv_cnt, int *err) {
    const int r = blockIdx.y;
    const int b = r / T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = blockIdx.x * kWarpsPerCta + warp;
    int cnt = topk_cnt[r];
    const int p = q_pos[r];
    if (cnt < 0 || cnt > k) {
        if (threadIdx.x == 0 && blockIdx.x == 0) report_error(err, CSA_ERR_BAD_INDEX);
        cnt = cnt < 0 ? 0 : k;
    }
    if (p < 0 && threadIdx.x == 0 && blockIdx.x == 0) report_error(err, CSA_ERR_BAD_INDEX);
    const int j0 = max(0, p - W + 1);
    const int nswa = p >= 0 ? p - j0 + 1 : 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) kv_cnt[r] = cnt + nswa;
    if (slot >= cnt + nswa) return;
    const uint8_t *src;
    if (slot < cnt) {
        const int64_t rec = record_index(comp, b, topk_idx[(size_t)r * k + slot]);
        if (rec < 0) {
            if (lane == 0) report_error(err, CSA_ERR_BAD_INDEX);
            return;
        }
        src = comp.base + rec * kRecBytes;
    } else {
        const int j = j0 + (slot - cnt);
        src = ring + ((int64_t)b * R + j % R) * kRecBytes;
    }
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
    uint4 *d4 = reinterpret_cast<uint4 *>(kv_out + ((size_t)r * (k + W) + slot) * kRecBytes);
    for (int c = lane; c < kChunks; c += 32) d4[c] = __ldg(s4 + c);
}

}  // namespace

cudaError_t launch_gather(const csa_cache_desc &comp, const void *ring, int R, int W, const int32_t *topk_idx,
                          const int32_t *topk_cnt, const int32_t *q_pos, int B, int T, int k, void *kv_out,
                          int32_t *kv_cnt, int *err, cudaStream_t stream) {
    dim3 grid((k + W + kWarpsPerCta - 1) / kWarpsPerCta, B * T);
    count_launch();
    gather_kernel<<<grid, kWarpsPerCta * 32, 0, stream>>>(make_view(comp), static_cast<const uint8_t *>(ring), R, W,
                                                          topk_idx, topk_cnt, q_pos, T, k,
                                                          static_cast<uint8_t *>(kv_out), kv_cnt, err);
    return cudaGetLastError();
}

}  // namespace csa
