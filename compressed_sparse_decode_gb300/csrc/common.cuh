// common.cuh -- shared device helpers of libcsa (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>

#include "../../include/csa.h"

namespace csa {

constexpr int kHeads = CSA_HEADS;
constexpr int kDim = CSA_LATENT_DIM;
constexpr int kNope = CSA_NOPE_DIM;
constexpr int kRope = CSA_ROPE_DIM;
constexpr int kScaleBlock = CSA_SCALE_BLOCK;
constexpr int kRecBytes = CSA_RECORD_BYTES;
constexpr int kRopeOffset = kNope;                 // 448
constexpr int kScaleOffset = kNope + 2 * kRope;    // 576
constexpr int kIdxHeads = CSA_INDEXER_HEADS;
constexpr int kIdxDim = CSA_INDEXER_DIM;

// Host-side count of kernel launches issued by the library.
void count_launch(int n = 1);
// Time limit of the bounded waits in the tensor-core kernels (GPU global
// time): one second unless a diagnostic call shortened it.
constexpr uint64_t kDefaultWaitNs = 1000000000ull;
// Drain waits (copies and MMAs already issued) always keep the default.
constexpr uint64_t kDrainWaitNs = kDefaultWaitNs;
void set_wait_limit_ns(uint64_t ns);
uint64_t wait_limit_ns();
// Shared host-side argument checks.
bool valid_cache(const csa_cache_desc &c, int B);
bool valid_dims(int B, int T);
bool valid_status_word(const int32_t *status);
csa_status_t attention_arg_status(const void *q, const float *sink, float softmax_scale, const csa_cache_desc &comp,
                                  const void *swa_ring, int R, int W, const int32_t *topk_idx,
                                  const int32_t *topk_cnt, const int32_t *q_pos, int B, int T, int k,
                                  const void *out, const float *lse, const int32_t *status);
// Host-side per-device caches (thread-safe): SM count of the current device,
// and the dynamic shared-memory opt-in of a kernel, set once per device.
int cached_sm_count();
cudaError_t set_max_dynamic_smem_once(const void *kernel, int bytes);
// Every host-side check csa_decode_step makes, before any launch.
csa_status_t decode_step_arg_status(const uint8_t *q_idx, const float *q_idx_scale, const float *w_idx,
                                    const uint8_t *k_idx, const float *k_idx_scale, const void *q, const float *sink,
                                    float softmax_scale, const csa_cache_desc &comp, const void *swa_ring, int R,
                                    int W, const int32_t *q_pos, const int32_t *n_comp, int B, int T, int Ncap,
                                    int m, int k, const void *out, const float *lse, const int32_t *topk_idx,
                                    const void *workspace, size_t workspace_bytes, const int32_t *status);

// Records a code in the caller's status word (device memory); the first
// error since the word was last cleared wins. No word: nothing is recorded.
__device__ __forceinline__ void report_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// Visible compressed entries of a query at 0-based position p: blocks strictly
// before its own block floor(p/m), bounded by the stored entries and capacity
// ("DSV4 Audit", section A3, item 1).
__device__ __forceinline__ int visible_entries(int p, int m, int n_comp, int cap) {
    if (p < 0) return 0;
    int nv = p / m;
    nv = nv < n_comp ? nv : n_comp;
    nv = nv < cap ? nv : cap;
    return nv < 0 ? 0 : nv;
}

// Device view of csa_cache_desc.
struct CacheView {
    const uint8_t *base;
    int64_t n_records;
    int64_t seq_stride;
    const int32_t *block_table;
    int32_t page_records;
    int32_t max_pages;
    int32_t seq_capacity;
};

inline CacheView make_view(const csa_cache_desc &d) {
    CacheView v;
    v.base = static_cast<const uint8_t *>(d.base);
    v.n_records = d.n_records;
    v.seq_stride = d.seq_stride;
    v.block_table = d.block_table;
    v.page_records = d.page_records;
    v.max_pages = d.max_pages;
    v.seq_capacity = d.seq_capacity;
    return v;
}

// Physical record index of logical entry c of sequence b, or -1 outside the
// cache (block-table strided, "ROADMAP -- Stage E", section E1).
__device__ __forceinline__ int64_t record_index(const CacheView &v, int b, int c) {
    if (c < 0 || c >= v.seq_capacity) return -1;
    int64_t rec;
    if (v.block_table) {
        int page = c / v.page_records;
        if (page >= v.max_pages) return -1;
        int32_t phys = __ldg(v.block_table + (int64_t)b * v.max_pages + page);
        if (phys < 0) return -1;
        rec = (int64_t)phys * v.page_records + c % v.page_records;
    } else {
        rec = (int64_t)b * v.seq_stride + c;
    }
    return (rec >= 0 && rec < v.n_records) ? rec : -1;
}

// Two E4M3 codes (low byte first) -> two floats through the hardware
// conversion (cvt e4m3x2 -> f16x2), exact.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
    return __half22float2(*reinterpret_cast<__half2 *>(&h));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Four floats -> four E2M1 codes in 16 bits (value i in bits 4i..4i+3): the
// hardware conversion, round to nearest with ties to even, saturating at +-6.
// (The instruction puts its first source in the high nibble of the byte.)
__device__ __forceinline__ uint32_t e2m1x4(float v0, float v1, float v2, float v3) {
    uint16_t r;
    asm("{\n\t.reg .b8 b0, b1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "mov.b16 %0, {b0, b1};\n\t}"
        : "=h"(r)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
    return r;
}

// cos and sin of the angle t * freq (freq in radians per position): the
// angle is formed and reduced to [-pi, pi] in double precision (t * freq
// reaches 10^6 rad at a 1M-token context, where a float angle would be off
// by up to 0.03 rad), then the special-function unit's sine and cosine run on
// the reduced angle (absolute error about 4e-7 on [-pi, pi]; no local-memory
// slow path for large arguments).
__device__ __forceinline__ float2 rope_cos_sin(int t, double freq) {
    const double a = (double)t * freq;
    const double turns = rint(a * 0.15915494309189535);  // a / (2 pi)
    const double r = fma(-turns, 6.283185307179586, a);
    float sn, cs;
    __sincosf(static_cast<float>(r), &sn, &cs);
    return make_float2(cs, sn);
}

// Order-preserving map of fp32 to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace csa
