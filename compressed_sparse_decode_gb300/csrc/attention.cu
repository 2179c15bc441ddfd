// attention.cu -- sink-merged split-precision attention over the candidates
// [top-k entries] ++ [SWA window] (CSA) or [all visible entries] ++ [SWA
// window] (HCA) ("DSV4 Inference Kernel" README, Architecture; "DSV4 Audit",
// sections A3 and B1).
//
// The sink logit enters the running max and the denominator from the start
// (m = sink, l = 1, o = 0), so the online softmax over the candidates ends at
//   o = sum_j e^{z_j - M} x_j / (e^{sink - M} + sum_j e^{z_j - M}),
//   lse = M + ln(den).
// Candidates are read straight from the FP8/BF16 records, dequantised in
// registers (nope code times its block multiplier; rope as BF16).
#include "common.cuh"

namespace csa {

namespace {

constexpr int kHeadsPerCta = 8;  // one warp per head

struct Lane16 {
    float v[16];
};

// Latent dims owned by `lane`: lanes 0..27 hold nope dims [16 lane, 16 lane + 16),
// lanes 28..31 hold rope dims [448 + 16 (lane-28), +16).
__device__ __forceinline__ void load_latent(const uint8_t *rec, int lane, Lane16 &x) {
    if (lane < 28) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(rec + lane * 16));
        const float s = __ldg(reinterpret_cast<const float *>(rec + kScaleOffset) + (lane >> 3));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float2 lo = e4m3x2_to_float2(static_cast<uint16_t>(w[j] & 0xFFFF));
            float2 hi = e4m3x2_to_float2(static_cast<uint16_t>(w[j] >> 16));
            x.v[4 * j + 0] = lo.x * s;
            x.v[4 * j + 1] = lo.y * s;
            x.v[4 * j + 2] = hi.x * s;
            x.v[4 * j + 3] = hi.y * s;
        }
    } else {
        const uint4 *p = reinterpret_cast<const uint4 *>(rec + kRopeOffset + (lane - 28) * 32);
        const uint4 a = __ldg(p), c = __ldg(p + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            x.v[2 * j + 0] = bf16_bits_to_float(static_cast<uint16_t>(w[j] & 0xFFFF));
            x.v[2 * j + 1] = bf16_bits_to_float(static_cast<uint16_t>(w[j] >> 16));
        }
    }
}

__device__ __forceinline__ int lane_dim0(int lane) { return lane < 28 ? lane * 16 : kNope + (lane - 28) * 16; }

__global__ void __launch_bounds__(kHeadsPerCta * 32)
attention_simt_kernel(const __nv_bfloat16 *__restrict__ q, const float *__restrict__ sink, float scale,
                      CacheView comp, const uint8_t *__restrict__ ring, int R, int W,
                      const int32_t *__restrict__ topk_idx, const int32_t *__restrict__ topk_cnt,
                      const int32_t *__restrict__ n_comp, int m_hca, const int32_t *__restrict__ q_pos,
                      int T, int k, int hca, __nv_bfloat16 *__restrict__ out, float *__restrict__ lse,
                      int *err) {
    const int r = blockIdx.y;
    const int b = r / T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x * kHeadsPerCta + warp;
    const int d0 = lane_dim0(lane);
    const int p = q_pos[r];

    int n_sel;
    if (hca) {
        n_sel = visible_entries(p, m_hca, n_comp[b], comp.seq_capacity);
    } else {
        n_sel = topk_cnt[r];
        if (n_sel < 0 || n_sel > k) {
            if (lane == 0) report_error(err, CSA_ERR_BAD_INDEX);
            n_sel = n_sel < 0 ? 0 : k;
        }
    }
    if (p < 0 && lane == 0) report_error(err, CSA_ERR_BAD_INDEX);
    const int j0 = max(0, p - W + 1);
    const int nswa = p >= 0 ? p - j0 + 1 : 0;

    float qv[16];
    {
        const uint4 *qp = reinterpret_cast<const uint4 *>(q + ((size_t)r * kHeads + h) * kDim + d0);
        const uint4 a = __ldg(qp), c = __ldg(qp + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            qv[2 * j + 0] = bf16_bits_to_float(static_cast<uint16_t>(w[j] & 0xFFFF));
            qv[2 * j + 1] = bf16_bits_to_float(static_cast<uint16_t>(w[j] >> 16));
        }
    }

    const float sk = sink[h];
    float mrun = sk;                          // running max, starts at the sink logit
    float l = (sk == -INFINITY) ? 0.f : 1.f;  // e^{sink - m}
    float o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i] = 0.f;

    const int n = n_sel + nswa;
    for (int j = 0; j < n; ++j) {
        const uint8_t *rec;
        if (j < n_sel) {
            const int c = hca ? j : __ldg(topk_idx + (size_t)r * k + j);
            const int64_t ri = record_index(comp, b, c);
            if (ri < 0) {
                if (lane == 0) report_error(err, CSA_ERR_BAD_INDEX);
                continue;
            }
            rec = comp.base + ri * kRecBytes;
        } else {
            const int pos = j0 + (j - n_sel);
            rec = ring + ((int64_t)b * R + pos % R) * kRecBytes;
        }
        Lane16 x;
        load_latent(rec, lane, x);
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) dot = fmaf(qv[i], x.v[i], dot);
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o2);
        const float z = dot * scale;
        const float mnew = fmaxf(mrun, z);
        const float corr = __expf(mrun - mnew);
        const float pj = __expf(z - mnew);
        l = l * corr + pj;
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = fmaf(o[i], corr, pj * x.v[i]);
        mrun = mnew;
    }

    const float inv = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16 ob[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) ob[i] = __float2bfloat16_rn(o[i] * inv);
    uint4 *op = reinterpret_cast<uint4 *>(out + ((size_t)r * kHeads + h) * kDim + d0);
    op[0] = *reinterpret_cast<const uint4 *>(&ob[0]);
    op[1] = *reinterpret_cast<const uint4 *>(&ob[8]);
    if (lane == 0) lse[(size_t)r * kHeads + h] = l > 0.f ? mrun + logf(l) : sk;
}

}  // namespace

size_t attention_workspace_bytes(int, int, int) { return 0; }

cudaError_t launch_attention(const void *q, const float *sink, float scale, const csa_cache_desc &comp,
                             const void *ring, int R, int W, const int32_t *topk_idx, const int32_t *topk_cnt,
                             const int32_t *n_comp, int m_hca, const int32_t *q_pos, int B, int T, int k, bool hca,
                             void *out, float *lse, void *, size_t, int *err, cudaStream_t stream) {
    dim3 grid(kHeads / kHeadsPerCta, B * T);
    count_launch();
    attention_simt_kernel<<<grid, kHeadsPerCta * 32, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(q), sink, scale, make_view(comp), static_cast<const uint8_t *>(ring), R, W,
        topk_idx, topk_cnt, n_comp, m_hca, q_pos, T, k, hca ? 1 : 0, static_cast<__nv_bfloat16 *>(out), lse, err);
    return cudaGetLastError();
}

}  // namespace csa
