// pipeline.cu -- the host-I/O decode pipeline: csa_decode_step on per-step
// copies of the query-side inputs taken from host memory, with the results
// copied back to host memory. Host code only (no kernels of its own).
//
// Step i uses staging slot s = i mod depth and three streams:
//   copy-in   waits computed[s] (step i-depth no longer reads slot s's inputs),
//             copies the five inputs host->device, records in_ready[s]
//   compute   waits in_ready[s] and out_done[s] (step i-depth's results have
//             left slot s), runs csa_decode_step, records computed[s]
//   copy-out  waits computed[s], copies out and lse device->host, records
//             out_done[s]
// so the copies of steps i-1 and i+1 overlap step i's kernels. Every wait is
// on the latest record of an event, made by step i-depth: calls are issued in
// step order from the host, so no record of a later step can exist yet.
#include <new>

#include "common.cuh"

struct csa_pipeline_s {
    int dev = 0;
    int B = 0, T = 0, depth = 0;
    cudaStream_t compute = nullptr, copy_in = nullptr, copy_out = nullptr;
    cudaEvent_t in_ready[CSA_PIPELINE_MAX_DEPTH] = {};
    cudaEvent_t computed[CSA_PIPELINE_MAX_DEPTH] = {};
    cudaEvent_t out_done[CSA_PIPELINE_MAX_DEPTH] = {};
    uint8_t *staging = nullptr;
    size_t slot_bytes = 0;
    int64_t steps = 0;
};

namespace {

constexpr size_t kAlign = 256;

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Byte sizes of the per-slot tensors, in slot order.
struct SlotLayout {
    size_t q_idx, q_idx_scale, w_idx, q, q_pos, out, lse;
    size_t off_q_idx, off_q_idx_scale, off_w_idx, off_q, off_q_pos, off_out, off_lse, total;
    SlotLayout(int B, int T) {
        const size_t bt = (size_t)B * T;
        q_idx = bt * CSA_INDEXER_HEADS * CSA_INDEXER_DIM;
        q_idx_scale = bt * CSA_INDEXER_HEADS * sizeof(float);
        w_idx = bt * CSA_INDEXER_HEADS * sizeof(float);
        q = bt * CSA_HEADS * CSA_LATENT_DIM * 2;
        q_pos = bt * sizeof(int32_t);
        out = bt * CSA_HEADS * CSA_LATENT_DIM * 2;
        lse = bt * CSA_HEADS * sizeof(float);
        off_q_idx = 0;
        off_q_idx_scale = off_q_idx + up(q_idx);
        off_w_idx = off_q_idx_scale + up(q_idx_scale);
        off_q = off_w_idx + up(w_idx);
        off_q_pos = off_q + up(q);
        off_out = off_q_pos + up(q_pos);
        off_lse = off_out + up(out);
        total = off_lse + up(lse);
    }
};

bool sizes_ok(int B, int T, int depth) {
    return B >= 1 && T >= 1 && T <= CSA_MAX_TOKENS_PER_SEQ && (int64_t)B * T <= 65535 && depth >= 2 &&
           depth <= CSA_PIPELINE_MAX_DEPTH;
}

void release(csa_pipeline_s *p) {
    for (int i = 0; i < CSA_PIPELINE_MAX_DEPTH; ++i) {
        if (p->in_ready[i]) cudaEventDestroy(p->in_ready[i]);
        if (p->computed[i]) cudaEventDestroy(p->computed[i]);
        if (p->out_done[i]) cudaEventDestroy(p->out_done[i]);
    }
    if (p->copy_in) cudaStreamDestroy(p->copy_in);
    if (p->copy_out) cudaStreamDestroy(p->copy_out);
    delete p;
}

bool on_pipeline_device(const csa_pipeline_s *p) {
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess && dev == p->dev;
}

}  // namespace

extern "C" {

size_t csa_pipeline_staging_bytes(int B, int T, int depth) {
    if (!sizes_ok(B, T, depth)) return 0;
    return (size_t)depth * SlotLayout(B, T).total;
}

csa_status_t csa_pipeline_create(csa_pipeline_t *pipeline, int B, int T, int depth, void *staging,
                                 size_t staging_bytes, cudaStream_t compute) {
    if (!pipeline) return CSA_ERR_INVALID_ARG;
    *pipeline = nullptr;
    if (!sizes_ok(B, T, depth) || !staging || (reinterpret_cast<uintptr_t>(staging) % kAlign) ||
        staging_bytes < csa_pipeline_staging_bytes(B, T, depth))
        return CSA_ERR_INVALID_ARG;
    csa_pipeline_s *p = new (std::nothrow) csa_pipeline_s;
    if (!p) return CSA_ERR_CUDA;
    p->B = B;
    p->T = T;
    p->depth = depth;
    p->compute = compute;
    p->staging = static_cast<uint8_t *>(staging);
    p->slot_bytes = SlotLayout(B, T).total;
    bool ok = cudaGetDevice(&p->dev) == cudaSuccess;
    ok = ok && cudaStreamCreateWithFlags(&p->copy_in, cudaStreamNonBlocking) == cudaSuccess;
    ok = ok && cudaStreamCreateWithFlags(&p->copy_out, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; i < depth && ok; ++i) {
        ok = ok && cudaEventCreateWithFlags(&p->in_ready[i], cudaEventDisableTiming) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&p->computed[i], cudaEventDisableTiming) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&p->out_done[i], cudaEventDisableTiming) == cudaSuccess;
    }
    if (!ok) {
        release(p);
        return CSA_ERR_CUDA;
    }
    *pipeline = p;
    return CSA_OK;
}

csa_status_t csa_decode_step_host(csa_pipeline_t p, const uint8_t *h_q_idx, const float *h_q_idx_scale,
                                  const float *h_w_idx, const void *h_q, const int32_t *h_q_pos,
                                  const uint8_t *k_idx, const float *k_idx_scale, const float *sink,
                                  float softmax_scale, csa_cache_desc comp, const void *swa_ring, int R, int W,
                                  const int32_t *n_comp, int Ncap, int m, int k, void *h_out, float *h_lse,
                                  void *workspace, size_t workspace_bytes, int32_t *status, int64_t *step_out) {
    if (!p || !h_q_idx || !h_q_idx_scale || !h_w_idx || !h_q || !h_q_pos || !h_out || !h_lse)
        return CSA_ERR_INVALID_ARG;
    if (!on_pipeline_device(p)) return CSA_ERR_INVALID_ARG;
    const int B = p->B, T = p->T;
    const SlotLayout L(B, T);
    const int s = (int)(p->steps % p->depth);
    uint8_t *slot = p->staging + (size_t)s * p->slot_bytes;
    uint8_t *q_idx = slot + L.off_q_idx;
    float *q_idx_scale = reinterpret_cast<float *>(slot + L.off_q_idx_scale);
    float *w_idx = reinterpret_cast<float *>(slot + L.off_w_idx);
    void *q = slot + L.off_q;
    int32_t *q_pos = reinterpret_cast<int32_t *>(slot + L.off_q_pos);
    void *out = slot + L.off_out;
    float *lse = reinterpret_cast<float *>(slot + L.off_lse);
    const csa_status_t a =
        csa::decode_step_arg_status(q_idx, q_idx_scale, w_idx, k_idx, k_idx_scale, q, sink, softmax_scale, comp,
                                    swa_ring, R, W, q_pos, n_comp, B, T, Ncap, m, k, out, lse, nullptr, workspace,
                                    workspace_bytes, status);
    if (a != CSA_OK) return a;

    // host -> device, once step (i - depth) has finished reading this slot
    cudaError_t e = cudaStreamWaitEvent(p->copy_in, p->computed[s], 0);
    const struct {
        void *dst;
        const void *src;
        size_t n;
    } in[5] = {{q_idx, h_q_idx, L.q_idx},
               {q_idx_scale, h_q_idx_scale, L.q_idx_scale},
               {w_idx, h_w_idx, L.w_idx},
               {q, h_q, L.q},
               {q_pos, h_q_pos, L.q_pos}};
    for (int i = 0; i < 5 && e == cudaSuccess; ++i)
        e = cudaMemcpyAsync(in[i].dst, in[i].src, in[i].n, cudaMemcpyHostToDevice, p->copy_in);
    if (e == cudaSuccess) e = cudaEventRecord(p->in_ready[s], p->copy_in);
    // kernels, once the inputs have landed and step (i - depth)'s results have left
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->compute, p->in_ready[s], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->compute, p->out_done[s], 0);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
    const csa_status_t st = csa_decode_step(q_idx, q_idx_scale, w_idx, k_idx, k_idx_scale, q, sink, softmax_scale,
                                            comp, swa_ring, R, W, q_pos, n_comp, B, T, Ncap, m, k, out, lse, nullptr,
                                            nullptr, workspace, workspace_bytes, status, p->compute);
    // computed[s] is recorded even after a failed launch, so that the slot's
    // later users do not wait on a stale record
    e = cudaEventRecord(p->computed[s], p->compute);
    if (st != CSA_OK) return st;
    // device -> host
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->copy_out, p->computed[s], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h_out, out, L.out, cudaMemcpyDeviceToHost, p->copy_out);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h_lse, lse, L.lse, cudaMemcpyDeviceToHost, p->copy_out);
    if (e == cudaSuccess) e = cudaEventRecord(p->out_done[s], p->copy_out);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
    if (step_out) *step_out = p->steps;
    ++p->steps;
    return CSA_OK;
}

csa_status_t csa_pipeline_wait(csa_pipeline_t p, int64_t step) {
    if (!p || step < 0 || step >= p->steps) return CSA_ERR_INVALID_ARG;
    // The copy-out stream runs the steps' device->host copies in order, so the
    // latest record of the slot's event (this step's or a later one's)
    // completing implies this step's copies have completed; its host->device
    // copies completed before its kernels started.
    return cudaEventSynchronize(p->out_done[step % p->depth]) == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

csa_status_t csa_pipeline_sync(csa_pipeline_t p) {
    if (!p) return CSA_ERR_INVALID_ARG;
    bool ok = cudaStreamSynchronize(p->copy_in) == cudaSuccess;
    ok = cudaStreamSynchronize(p->compute) == cudaSuccess && ok;
    ok = cudaStreamSynchronize(p->copy_out) == cudaSuccess && ok;
    return ok ? CSA_OK : CSA_ERR_CUDA;
}

csa_status_t csa_pipeline_destroy(csa_pipeline_t p) {
    if (!p) return CSA_OK;
    const csa_status_t s = csa_pipeline_sync(p);
    release(p);
    return s;
}

}  // extern "C"
