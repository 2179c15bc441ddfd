// api.cu -- the extern "C" entry points of libcsa: host-side argument checks,
// workspace carving and kernel launches. No call allocates device memory or
// synchronises the device (except csa_read_device_error, a diagnostic).
// In-kernel problems go to the caller's status word (an int32 in device
// memory passed to every compute call).
#include <cmath>
#include <cstdint>
#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace csa {
cudaError_t launch_indexer(const uint8_t *, const float *, const float *, const uint8_t *, const float *,
                           const int32_t *, const int32_t *, int, int, int, int, float *, int *, cudaStream_t);
size_t topk_workspace_bytes(int, int, int, int);
cudaError_t launch_topk(const float *, const int32_t *, const int32_t *, int, int, int, int, int, int32_t *,
                        int32_t *, void *, size_t, cudaStream_t);
cudaError_t launch_gather(const csa_cache_desc &, const void *, int, int, const int32_t *, const int32_t *,
                          const int32_t *, int, int, int, void *, int32_t *, int *, cudaStream_t);
size_t attention_workspace_bytes(int B, int T, int max_selected, int W);
cudaError_t launch_attention(const void *, const float *, float, const csa_cache_desc &, const void *, int, int,
                             const int32_t *, const int32_t *, const int32_t *, int, const int32_t *, int, int, int,
                             bool, void *, float *, const csa_attention_epilogue *, void *, size_t, int *,
                             cudaStream_t);
}  // namespace csa

namespace csa {
static std::atomic<uint64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {
constexpr int kMaxDevs = 64;
int g_sm_count[kMaxDevs];
struct SmemOptIn {
    const void *kernel;
    int dev, bytes;
};
SmemOptIn g_smem_opt_in[64];
int g_n_smem_opt_in;
std::mutex g_host_cache_mu;
}  // namespace

namespace {
std::atomic<uint64_t> g_wait_limit_ns{0};
}
void set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns, std::memory_order_relaxed); }
uint64_t wait_limit_ns() {
    const uint64_t v = g_wait_limit_ns.load(std::memory_order_relaxed);
    return v ? v : kDefaultWaitNs;
}

int cached_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevs) return 1;
    std::lock_guard<std::mutex> g(g_host_cache_mu);
    if (g_sm_count[dev] <= 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sm_count[dev] = n > 0 ? n : 1;
    }
    return g_sm_count[dev];
}

cudaError_t set_max_dynamic_smem_once(const void *kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> g(g_host_cache_mu);
    for (int i = 0; i < g_n_smem_opt_in; ++i)
        if (g_smem_opt_in[i].kernel == kernel && g_smem_opt_in[i].dev == dev && g_smem_opt_in[i].bytes >= bytes)
            return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && g_n_smem_opt_in < 64) g_smem_opt_in[g_n_smem_opt_in++] = {kernel, dev, bytes};
    return e;
}
}  // namespace csa

using namespace csa;

namespace {

constexpr size_t kWsAlign = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

csa_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

namespace csa {
bool valid_cache(const csa_cache_desc &c, int B) {
    if (!c.base || !aligned16(c.base) || c.n_records <= 0 || c.seq_capacity <= 0) return false;
    if (c.block_table) {
        if (!aligned16(c.block_table) || c.page_records <= 0 || c.max_pages <= 0) return false;
    } else {
        if (c.seq_stride < 0) return false;
        if (B > 1 && c.seq_stride < c.seq_capacity) return false;
    }
    return true;
}

bool valid_dims(int B, int T) { return B >= 1 && T >= 1 && T <= CSA_MAX_TOKENS_PER_SEQ && (int64_t)B * T <= 65535; }

bool valid_status_word(const int32_t *status) { return aligned4(status); }

csa_status_t attention_arg_status(const void *q, const float *sink, float softmax_scale, const csa_cache_desc &comp,
                                  const void *swa_ring, int R, int W, const int32_t *topk_idx,
                                  const int32_t *topk_cnt, const int32_t *q_pos, int B, int T, int k,
                                  const void *out, const float *lse, const int32_t *status) {
    if (!q || !sink || !swa_ring || !topk_idx || !topk_cnt || !q_pos || !out || !lse) return CSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(swa_ring) || !aligned16(out) || !valid_cache(comp, B) ||
        !valid_status_word(status))
        return CSA_ERR_INVALID_ARG;
    if (!valid_dims(B, T) || k < 1 || W < 1 || W > CSA_MAX_SWA_WINDOW || R < W || !(softmax_scale > 0.f))
        return CSA_ERR_INVALID_ARG;
    if (k > CSA_MAX_TOPK) return CSA_ERR_UNSUPPORTED;
    return CSA_OK;
}

// The host-side checks of csa_indexer_logits, csa_topk and
// csa_sink_attention_decode for the arguments csa_decode_step passes them, so
// that a bad argument is reported before any of the three launches.
csa_status_t decode_step_arg_status(const uint8_t *q_idx, const float *q_idx_scale, const float *w_idx,
                                    const uint8_t *k_idx, const float *k_idx_scale, const void *q, const float *sink,
                                    float softmax_scale, const csa_cache_desc &comp, const void *swa_ring, int R,
                                    int W, const int32_t *q_pos, const int32_t *n_comp, int B, int T, int Ncap,
                                    int m, int k, const void *out, const float *lse, const int32_t *topk_idx,
                                    const void *workspace, size_t workspace_bytes, const int32_t *status) {
    if (!valid_dims(B, T) || Ncap < 1 || k < 1 || m < 1) return CSA_ERR_INVALID_ARG;
    if (!valid_status_word(status)) return CSA_ERR_INVALID_ARG;
    if (!q_idx || !q_idx_scale || !w_idx || !k_idx || !k_idx_scale || !q || !sink || !swa_ring || !q_pos ||
        !n_comp || !out || !lse)
        return CSA_ERR_INVALID_ARG;
    if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(q_idx_scale) || !aligned16(w_idx) ||
        !aligned16(k_idx_scale) || !aligned16(q) || !aligned16(swa_ring) || !aligned16(out) ||
        (topk_idx && !aligned16(topk_idx)) || !valid_cache(comp, B))
        return CSA_ERR_INVALID_ARG;
    if (W < 1 || W > CSA_MAX_SWA_WINDOW || R < W || !(softmax_scale > 0.f)) return CSA_ERR_INVALID_ARG;
    if (k > Ncap || k > CSA_MAX_TOPK) return CSA_ERR_UNSUPPORTED;
    if ((int64_t)B * Ncap >= ((int64_t)1 << 31)) return CSA_ERR_UNSUPPORTED;
    const size_t need = csa_workspace_bytes(CSA_OP_DECODE_STEP, B, T, Ncap, k);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign))
        return CSA_ERR_WORKSPACE;
    return CSA_OK;
}
}  // namespace csa

extern "C" {

int csa_version(void) { return 100; }

uint64_t csa_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char *csa_status_string(csa_status_t s) {
    switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID_ARG: return "invalid argument";
    case CSA_ERR_UNSUPPORTED: return "unsupported shape";
    case CSA_ERR_WORKSPACE: return "workspace missing or too small";
    case CSA_ERR_CUDA: return "CUDA error";
    case CSA_ERR_TIMEOUT: return "bounded wait expired in a kernel";
    case CSA_ERR_BAD_INDEX: return "index or position outside a cache";
    }
    return "unknown status";
}

size_t csa_workspace_bytes(csa_op_t op, int B, int T, int Ncap, int k) {
    if (B < 1 || T < 1 || Ncap < 1) return 0;
    switch (op) {
    case CSA_OP_INDEXER: return 0;
    case CSA_OP_TOPK: return topk_workspace_bytes(B, T, Ncap, k);
    case CSA_OP_ATTENTION: return attention_workspace_bytes(B, T, k, CSA_MAX_SWA_WINDOW);
    case CSA_OP_HCA_ATTENTION: return attention_workspace_bytes(B, T, Ncap, CSA_MAX_SWA_WINDOW);
    case CSA_OP_DECODE_STEP:
        return align_up(sizeof(float) * (size_t)B * T * Ncap, kWsAlign) +
               2 * align_up(sizeof(int32_t) * (size_t)B * T * k, kWsAlign) +
               align_up(topk_workspace_bytes(B, T, Ncap, k), kWsAlign) +
               align_up(attention_workspace_bytes(B, T, k, CSA_MAX_SWA_WINDOW), kWsAlign);
    }
    return 0;
}

csa_status_t csa_indexer_logits(const uint8_t *q_idx, const float *q_idx_scale, const float *w_idx,
                                const uint8_t *k_idx, const float *k_idx_scale, const int32_t *q_pos,
                                const int32_t *n_comp, int B, int T, int Ncap, int m, float *logits,
                                int32_t *status, cudaStream_t stream) {
    if (!q_idx || !q_idx_scale || !w_idx || !k_idx || !k_idx_scale || !q_pos || !n_comp || !logits)
        return CSA_ERR_INVALID_ARG;
    if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(logits) || !aligned16(q_idx_scale) ||
        !aligned16(w_idx) || !aligned16(k_idx_scale) || !valid_status_word(status))
        return CSA_ERR_INVALID_ARG;
    if (!valid_dims(B, T) || Ncap < 1 || m < 1) return CSA_ERR_INVALID_ARG;
    if ((int64_t)B * Ncap >= ((int64_t)1 << 31)) return CSA_ERR_UNSUPPORTED;
    return cuda_status(launch_indexer(q_idx, q_idx_scale, w_idx, k_idx, k_idx_scale, q_pos, n_comp, B, T, Ncap, m,
                                      logits, status, stream));
}

csa_status_t csa_topk(const float *logits, const int32_t *q_pos, const int32_t *n_comp, int B, int T, int Ncap,
                      int m, int k, int32_t *topk_idx, int32_t *topk_cnt, void *workspace, size_t workspace_bytes,
                      int32_t *status, cudaStream_t stream) {
    if (!logits || !q_pos || !n_comp || !topk_idx || !topk_cnt) return CSA_ERR_INVALID_ARG;
    if (!aligned16(logits) || !aligned16(topk_idx) || !valid_status_word(status)) return CSA_ERR_INVALID_ARG;
    if (!valid_dims(B, T) || Ncap < 1 || m < 1 || k < 1) return CSA_ERR_INVALID_ARG;
    if (k > Ncap || k > CSA_MAX_TOPK) return CSA_ERR_UNSUPPORTED;
    const size_t need = topk_workspace_bytes(B, T, Ncap, k);
    if (need && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign)))
        return CSA_ERR_WORKSPACE;
    return cuda_status(launch_topk(logits, q_pos, n_comp, B, T, Ncap, m, k, topk_idx, topk_cnt, workspace,
                                   workspace_bytes, stream));
}

csa_status_t csa_gather_swa(csa_cache_desc comp, const void *swa_ring, int R, int W, const int32_t *topk_idx,
                            const int32_t *topk_cnt, const int32_t *q_pos, int B, int T, int k, void *kv_out,
                            int32_t *kv_cnt, int32_t *status, cudaStream_t stream) {
    if (!swa_ring || !topk_idx || !topk_cnt || !q_pos || !kv_out || !kv_cnt) return CSA_ERR_INVALID_ARG;
    if (!aligned16(swa_ring) || !aligned16(kv_out) || !valid_cache(comp, B) || !valid_status_word(status))
        return CSA_ERR_INVALID_ARG;
    if (!valid_dims(B, T) || k < 1 || W < 1 || W > CSA_MAX_SWA_WINDOW || R < W) return CSA_ERR_INVALID_ARG;
    return cuda_status(launch_gather(comp, swa_ring, R, W, topk_idx, topk_cnt, q_pos, B, T, k, kv_out, kv_cnt,
                                     status, stream));
}

namespace {
// An epilogue the kernels can apply; `out` is required unless the output is E2M1.
csa_status_t epilogue_status(const csa_attention_epilogue *epi, const void *out) {
    const bool fp4 = epi && epi->out_fp4;
    if (!fp4 && (!out || !aligned16(out))) return CSA_ERR_INVALID_ARG;
    if (!epi) return CSA_OK;
    if (epi->inverse_rope && !(epi->rope_theta > 1.f && std::isfinite(epi->rope_theta))) return CSA_ERR_INVALID_ARG;
    if (fp4 && (!epi->out_fp4_scale || !aligned16(epi->out_fp4) || !aligned16(epi->out_fp4_scale)))
        return CSA_ERR_INVALID_ARG;
    return CSA_OK;
}
// The output pointer the shared checks look at: E2M1 output stands in for `out`.
const void *checked_out(const csa_attention_epilogue *epi, const void *out) {
    return (epi && epi->out_fp4) ? static_cast<const void *>(epi->out_fp4) : out;
}
}  // namespace

csa_status_t csa_sink_attention_decode_ex(const void *q, const float *sink, float softmax_scale, csa_cache_desc comp,
                                          const void *swa_ring, int R, int W, const int32_t *topk_idx,
                                          const int32_t *topk_cnt, const int32_t *q_pos, int B, int T, int k,
                                          void *out, float *lse, const csa_attention_epilogue *epilogue,
                                          void *workspace, size_t workspace_bytes, int32_t *status,
                                          cudaStream_t stream) {
    csa_status_t a = epilogue_status(epilogue, out);
    if (a != CSA_OK) return a;
    a = attention_arg_status(q, sink, softmax_scale, comp, swa_ring, R, W, topk_idx, topk_cnt, q_pos, B, T, k,
                             checked_out(epilogue, out), lse, status);
    if (a != CSA_OK) return a;
    const size_t need = attention_workspace_bytes(B, T, k, W);
    if (need && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign)))
        return CSA_ERR_WORKSPACE;
    return cuda_status(launch_attention(q, sink, softmax_scale, comp, swa_ring, R, W, topk_idx, topk_cnt, nullptr, 1,
                                        q_pos, B, T, k, false, out, lse, epilogue, workspace, workspace_bytes, status,
                                        stream));
}

csa_status_t csa_sink_attention_decode(const void *q, const float *sink, float softmax_scale, csa_cache_desc comp,
                                       const void *swa_ring, int R, int W, const int32_t *topk_idx,
                                       const int32_t *topk_cnt, const int32_t *q_pos, int B, int T, int k, void *out,
                                       float *lse, void *workspace, size_t workspace_bytes, int32_t *status,
                                       cudaStream_t stream) {
    return csa_sink_attention_decode_ex(q, sink, softmax_scale, comp, swa_ring, R, W, topk_idx, topk_cnt, q_pos, B, T,
                                        k, out, lse, nullptr, workspace, workspace_bytes, status, stream);
}

csa_status_t hca_sink_attention_decode_ex(const void *q, const float *sink, float softmax_scale, csa_cache_desc comp,
                                          const int32_t *n_comp, const void *swa_ring, int R, int W,
                                          const int32_t *q_pos, int B, int T, int m_hca, void *out, float *lse,
                                          const csa_attention_epilogue *epilogue, void *workspace,
                                          size_t workspace_bytes, int32_t *status, cudaStream_t stream) {
    const csa_status_t a = epilogue_status(epilogue, out);
    if (a != CSA_OK) return a;
    if (!q || !sink || !n_comp || !swa_ring || !q_pos || !lse) return CSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(swa_ring) || !valid_cache(comp, B) || !valid_status_word(status))
        return CSA_ERR_INVALID_ARG;
    if (!valid_dims(B, T) || W < 1 || W > CSA_MAX_SWA_WINDOW || R < W || m_hca < 1 || !(softmax_scale > 0.f))
        return CSA_ERR_INVALID_ARG;
    const size_t need = attention_workspace_bytes(B, T, comp.seq_capacity, W);
    if (need && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign)))
        return CSA_ERR_WORKSPACE;
    return cuda_status(launch_attention(q, sink, softmax_scale, comp, swa_ring, R, W, nullptr, nullptr, n_comp, m_hca,
                                        q_pos, B, T, comp.seq_capacity, true, out, lse, epilogue, workspace,
                                        workspace_bytes, status, stream));
}

csa_status_t hca_sink_attention_decode(const void *q, const float *sink, float softmax_scale, csa_cache_desc comp,
                                       const int32_t *n_comp, const void *swa_ring, int R, int W,
                                       const int32_t *q_pos, int B, int T, int m_hca, void *out, float *lse,
                                       void *workspace, size_t workspace_bytes, int32_t *status,
                                       cudaStream_t stream) {
    return hca_sink_attention_decode_ex(q, sink, softmax_scale, comp, n_comp, swa_ring, R, W, q_pos, B, T, m_hca, out,
                                        lse, nullptr, workspace, workspace_bytes, status, stream);
}

csa_status_t csa_decode_step_ex(const uint8_t *q_idx, const float *q_idx_scale, const float *w_idx,
                                const uint8_t *k_idx, const float *k_idx_scale, const void *q, const float *sink,
                                float softmax_scale, csa_cache_desc comp, const void *swa_ring, int R, int W,
                                const int32_t *q_pos, const int32_t *n_comp, int B, int T, int Ncap, int m, int k,
                                void *out, float *lse, int32_t *topk_idx, int32_t *topk_cnt,
                                const csa_attention_epilogue *epilogue, void *workspace, size_t workspace_bytes,
                                int32_t *status, cudaStream_t stream) {
    // every argument of the three calls is checked before the first launch
    csa_status_t a = epilogue_status(epilogue, out);
    if (a != CSA_OK) return a;
    a = csa::decode_step_arg_status(q_idx, q_idx_scale, w_idx, k_idx, k_idx_scale, q, sink, softmax_scale, comp,
                                    swa_ring, R, W, q_pos, n_comp, B, T, Ncap, m, k, checked_out(epilogue, out), lse,
                                    topk_idx, workspace, workspace_bytes, status);
    if (a != CSA_OK) return a;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *logits = reinterpret_cast<float *>(ws);
    ws += align_up(sizeof(float) * (size_t)B * T * Ncap, kWsAlign);
    int32_t *idx = topk_idx ? topk_idx : reinterpret_cast<int32_t *>(ws);
    ws += align_up(sizeof(int32_t) * (size_t)B * T * k, kWsAlign);
    int32_t *cnt = topk_cnt ? topk_cnt : reinterpret_cast<int32_t *>(ws);
    ws += align_up(sizeof(int32_t) * (size_t)B * T * k, kWsAlign);
    const size_t tk_bytes = align_up(topk_workspace_bytes(B, T, Ncap, k), kWsAlign);
    void *tk_ws = tk_bytes ? ws : nullptr;
    ws += tk_bytes;
    const size_t at_bytes = align_up(attention_workspace_bytes(B, T, k, CSA_MAX_SWA_WINDOW), kWsAlign);
    csa_status_t s = csa_indexer_logits(q_idx, q_idx_scale, w_idx, k_idx, k_idx_scale, q_pos, n_comp, B, T, Ncap, m,
                                        logits, status, stream);
    if (s != CSA_OK) return s;
    s = csa_topk(logits, q_pos, n_comp, B, T, Ncap, m, k, idx, cnt, tk_ws, tk_bytes, status, stream);
    if (s != CSA_OK) return s;
    return csa_sink_attention_decode_ex(q, sink, softmax_scale, comp, swa_ring, R, W, idx, cnt, q_pos, B, T, k, out,
                                        lse, epilogue, at_bytes ? ws : nullptr, at_bytes, status, stream);
}

csa_status_t csa_decode_step(const uint8_t *q_idx, const float *q_idx_scale, const float *w_idx,
                             const uint8_t *k_idx, const float *k_idx_scale, const void *q, const float *sink,
                             float softmax_scale, csa_cache_desc comp, const void *swa_ring, int R, int W,
                             const int32_t *q_pos, const int32_t *n_comp, int B, int T, int Ncap, int m, int k,
                             void *out, float *lse, int32_t *topk_idx, int32_t *topk_cnt, void *workspace,
                             size_t workspace_bytes, int32_t *status, cudaStream_t stream) {
    return csa_decode_step_ex(q_idx, q_idx_scale, w_idx, k_idx, k_idx_scale, q, sink, softmax_scale, comp, swa_ring,
                              R, W, q_pos, n_comp, B, T, Ncap, m, k, out, lse, topk_idx, topk_cnt, nullptr, workspace,
                              workspace_bytes, status, stream);
}

csa_status_t csa_check_device_status(int32_t *status, int32_t *host_status, cudaStream_t stream) {
    if (!status || !host_status || !aligned4(status) || !aligned4(host_status)) return CSA_ERR_INVALID_ARG;
    if (cudaMemcpyAsync(host_status, status, sizeof(int32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return CSA_ERR_CUDA;
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), stream) != cudaSuccess) return CSA_ERR_CUDA;
    return CSA_OK;
}

csa_status_t csa_read_device_error(int32_t *status, int32_t *host_code, cudaStream_t stream) {
    if (!host_code) return CSA_ERR_INVALID_ARG;
    int32_t v = 0;
    const csa_status_t s = csa_check_device_status(status, &v, stream);
    if (s != CSA_OK) return s;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return CSA_ERR_CUDA;
    *host_code = v;
    return CSA_OK;
}

void csa_debug_set_wait_limit_ns(uint64_t ns) { csa::set_wait_limit_ns(ns); }

}  // extern "C"
