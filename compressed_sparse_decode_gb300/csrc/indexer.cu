// indexer.cu -- lightning-indexer logits ("DSV4 Audit", section B2).
//
// logits[b,t,c] = sk[b,c] * sum_h (w[b,t,h] * sq[b,t,h]) * relu(sum_d q8[b,t,h,d] k8[b,c,d])
// which equals the weighted-ReLU form because the scales are positive.
// Entries c >= n_vis(b,t) get -inf ("DSV4 Audit", section A3, item 1).
#include "common.cuh"

namespace csa {

namespace {

constexpr int kKeysPerCta = 128;

// One thread per key. Query codes (exact as floats) and the per-head weights
// w*sq for every token of the sequence sit in shared memory; each key's 128
// codes sit in registers.
__global__ void __launch_bounds__(kKeysPerCta)
indexer_simt_kernel(const uint8_t *__restrict__ q_idx, const float *__restrict__ q_scale,
                    const float *__restrict__ w_idx, const uint8_t *__restrict__ k_idx,
                    const float *__restrict__ k_scale, const int32_t *__restrict__ q_pos,
                    const int32_t *__restrict__ n_comp, int T, int Ncap, int m,
                    float *__restrict__ logits) {
    extern __shared__ float4 smem4[];
    float *qf = reinterpret_cast<float *>(smem4);          // [T][64][128]
    float *ws = qf + T * kIdxHeads * kIdxDim;              // [T][64]
    __shared__ int nvis[CSA_MAX_TOKENS_PER_SEQ];

    const int b = blockIdx.y;
    const int tid = threadIdx.x;
    const uint8_t *qb = q_idx + (size_t)b * T * kIdxHeads * kIdxDim;
    for (int i = tid * 2; i < T * kIdxHeads * kIdxDim; i += blockDim.x * 2) {
        float2 v = e4m3x2_to_float2(*reinterpret_cast<const uint16_t *>(qb + i));
        qf[i] = v.x;
        qf[i + 1] = v.y;
    }
    for (int i = tid; i < T * kIdxHeads; i += blockDim.x)
        ws[i] = w_idx[(size_t)b * T * kIdxHeads + i] * q_scale[(size_t)b * T * kIdxHeads + i];
    if (tid < T) nvis[tid] = visible_entries(q_pos[b * T + tid], m, n_comp[b], Ncap);
    __syncthreads();

    const int c = blockIdx.x * kKeysPerCta + tid;
    if (c >= Ncap) return;
    int nv_max = 0;
    for (int t = 0; t < T; ++t) nv_max = max(nv_max, nvis[t]);
    if (c >= nv_max) {
        for (int t = 0; t < T; ++t) logits[((size_t)b * T + t) * Ncap + c] = -INFINITY;
        return;
    }
    float kf[kIdxDim];
    const uint4 *kp = reinterpret_cast<const uint4 *>(k_idx + ((size_t)b * Ncap + c) * kIdxDim);
#pragma unroll
    for (int v = 0; v < kIdxDim / 16; ++v) {
        uint4 u = __ldg(kp + v);
        uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float2 lo = e4m3x2_to_float2(static_cast<uint16_t>(w4[j] & 0xFFFF));
            float2 hi = e4m3x2_to_float2(static_cast<uint16_t>(w4[j] >> 16));
            kf[v * 16 + j * 4 + 0] = lo.x;
            kf[v * 16 + j * 4 + 1] = lo.y;
            kf[v * 16 + j * 4 + 2] = hi.x;
            kf[v * 16 + j * 4 + 3] = hi.y;
        }
    }
    const float sk = __ldg(k_scale + (size_t)b * Ncap + c);
    for (int t = 0; t < T; ++t) {
        float acc = 0.f;
        for (int h = 0; h < kIdxHeads; ++h) {
            const float4 *qrow = reinterpret_cast<const float4 *>(qf + (t * kIdxHeads + h) * kIdxDim);
            float dot = 0.f;
#pragma unroll
            for (int d4 = 0; d4 < kIdxDim / 4; ++d4) {
                float4 qv = qrow[d4];
                dot = fmaf(qv.x, kf[d4 * 4 + 0], dot);
                dot = fmaf(qv.y, kf[d4 * 4 + 1], dot);
                dot = fmaf(qv.z, kf[d4 * 4 + 2], dot);
                dot = fmaf(qv.w, kf[d4 * 4 + 3], dot);
            }
            acc = fmaf(ws[t * kIdxHeads + h], fmaxf(dot, 0.f), acc);
        }
        logits[((size_t)b * T + t) * Ncap + c] = c < nvis[t] ? acc * sk : -INFINITY;
    }
}

}  // namespace

cudaError_t launch_indexer(const uint8_t *q_idx, const float *q_scale, const float *w_idx,
                           const uint8_t *k_idx, const float *k_scale, const int32_t *q_pos,
                           const int32_t *n_comp, int B, int T, int Ncap, int m, float *logits,
                           cudaStream_t stream) {
    size_t smem = sizeof(float) * (size_t)T * kIdxHeads * (kIdxDim + 1);
    cudaError_t e = cudaFuncSetAttribute(indexer_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((Ncap + kKeysPerCta - 1) / kKeysPerCta, B);
    count_launch();
    indexer_simt_kernel<<<grid, kKeysPerCta, smem, stream>>>(q_idx, q_scale, w_idx, k_idx, k_scale, q_pos,
                                                              n_comp, T, Ncap, m, logits);
    return cudaGetLastError();
}

}  // namespace csa
