/*
 * csa.h -- C ABI of the GB300 (sm_103a) compressed sparse attention decode
 * library, libcsa.so.
 *
 * One decode step of DSV4-style Compressed Sparse Attention (CSA), as the
 * project's pages describe it:
 *   1. lightning-indexer logits of each query token against every compressed
 *      KV entry            -> csa_indexer_logits
 *   2. top-k over the causally visible entries  -> csa_topk
 *   3. gather of the selected FP8/BF16 latents together with the SWA window
 *                          -> fused into step 4 (csa_gather_swa is the
 *                             standalone packed gather)
 *   4. one sink-merged attention pass  -> csa_sink_attention_decode
 * and the heavily-compressed (HCA) variant that attends to every visible entry
 * with no indexer -> hca_sink_attention_decode. csa_decode_step runs 1, 2, 4.
 *
 * Conventions for every call
 *  - Pointers are DEVICE pointers unless stated; the caller owns all memory.
 *    The library allocates no device memory (csa_pipeline_create makes a
 *    small host object, two streams and events) and keeps no state beyond
 *    per-process caches of kernel attributes, device properties and TMA
 *    descriptors.
 *  - Calls are asynchronous on `stream`; none synchronises the device (the
 *    diagnostics and csa_pipeline_wait/sync/destroy block the host).
 *    Argument errors are detected on the host before any launch and returned
 *    as codes; launch failures return CSA_ERR_CUDA (cudaGetLastError).
 *  - Status word: every compute call takes `status`, a caller-owned int32 in
 *    device memory (4-byte aligned; NULL = do not record). Problems found
 *    inside a kernel are recorded there, the first one winning (atomic
 *    compare-and-swap from CSA_OK): an index or position that would address
 *    memory outside a cache (the access is skipped: CSA_ERR_BAD_INDEX) and a
 *    bounded wait that expired (the kernel winds down: CSA_ERR_TIMEOUT).
 *    Kernels never trap. The word is read without stalling the stream by
 *    csa_check_device_status ("ROADMAP -- Stage E", section E4: no
 *    synchronisation on the decode path; return codes instead). Calls that
 *    share a word share its first-error-wins slot; give concurrent streams
 *    their own words.
 *  - Shapes fixed by the method: H = 128 query heads, latent D = 512 = 448
 *    FP8 E4M3 "nope" dims + 64 BF16 rope dims, indexer Hi = 64 heads x Di = 128
 *    FP8 dims. Tensors are dense row-major in the order of their index lists.
 *  - Every pointer must be 16-byte aligned.
 *
 * Latent record (one compressed entry or one SWA token), CSA_RECORD_BYTES:
 *   bytes [0,448)   nope dims, FP8 E4M3
 *   bytes [448,576) rope dims, BF16
 *   bytes [576,592) 4 fp32 dequantisation multipliers; multiplier i covers
 *                   nope dims [128i, min(128i+128, 448))
 * (pages: "DSV4 Audit", section B1 -- FP8 nope + BF16 rope, fed to attention
 * without a BF16 dequantised copy; "ROADMAP -- Stage E", section E1 -- FP8
 * entries with the inverse scale stored alongside.)
 */
#ifndef CSA_H_
#define CSA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define CSA_API __attribute__((visibility("default")))
#else
#define CSA_API
#endif

#define CSA_HEADS 128
#define CSA_LATENT_DIM 512
#define CSA_NOPE_DIM 448
#define CSA_ROPE_DIM 64
#define CSA_SCALE_BLOCK 128
#define CSA_RECORD_BYTES 592
#define CSA_INDEXER_HEADS 64
#define CSA_INDEXER_DIM 128
#define CSA_MAX_TOKENS_PER_SEQ 128 /* T: query tokens per sequence and step */
#define CSA_MAX_TOPK 2048
#define CSA_MAX_SWA_WINDOW 512 /* W */

typedef enum {
    CSA_OK = 0,
    CSA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, size out of range */
    CSA_ERR_UNSUPPORTED = 2, /* a shape outside what the kernels implement */
    CSA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
    CSA_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
    CSA_ERR_TIMEOUT = 5,     /* (device word) a bounded wait in a kernel expired */
    CSA_ERR_BAD_INDEX = 6    /* (device word) an index/position outside a cache */
} csa_status_t;

/* A cache of latent records (compressed entries). Logical entry c of sequence
 * b (0 <= c < seq_capacity) is record
 *     b * seq_stride + c                                     if block_table == NULL
 *     block_table[b*max_pages + c/page_records]*page_records + c%page_records
 * ("DSV4 Inference Kernel" README, Architecture: classical paged cache of
 * 128-token pages, i.e. 32 CSA entries or 1 HCA entry per page).
 * Records outside [0, n_records) are never read. */
typedef struct {
    const void *base;           /* device, n_records * CSA_RECORD_BYTES bytes */
    int64_t n_records;          /* records addressable from base */
    int64_t seq_stride;         /* contiguous mode: records between sequences */
    const int32_t *block_table; /* device [B, max_pages] or NULL */
    int32_t page_records;       /* paged mode: records per page (> 0) */
    int32_t max_pages;          /* paged mode: block-table row length */
    int32_t seq_capacity;       /* logical entries per sequence (Ncap) */
} csa_cache_desc;

typedef enum {
    CSA_OP_INDEXER = 0,
    CSA_OP_TOPK = 1,
    CSA_OP_ATTENTION = 2,     /* csa_sink_attention_decode, `k` = top-k */
    CSA_OP_HCA_ATTENTION = 3, /* hca_sink_attention_decode, `k` ignored */
    CSA_OP_DECODE_STEP = 4    /* csa_decode_step */
} csa_op_t;

/* Workspace bytes that `op` needs for these sizes (0 if none). A workspace
 * passed to a call must be at least this large and 256-byte aligned; its
 * contents need no initialisation and are scratch between calls. */
CSA_API size_t csa_workspace_bytes(csa_op_t op, int B, int T, int Ncap, int k);

/* Step 1 -- lightning-indexer logits ("DSV4 Audit", section B2: weighted-ReLU
 * MQA logits of every query token against every compressed entry, FP8 keys).
 *   logits[b,t,c] = sum_h w_idx[b,t,h] *
 *                   max(0, q_idx_scale[b,t,h] * k_idx_scale[b,c] *
 *                          sum_d e4m3(q_idx[b,t,h,d]) * e4m3(k_idx[b,c,d]))
 * for c < n_vis(b,t), and -inf for n_vis(b,t) <= c < Ncap, where
 *   n_vis(b,t) = min(floor(q_pos[b,t] / m), n_comp[b], Ncap)
 * ("DSV4 Audit", section A3 item 1: a query sees only the compressed blocks
 * strictly before its own incomplete block; q_pos is the 0-based position).
 *   q_idx       [B,T,64,128] e4m3 codes     q_idx_scale [B,T,64] fp32 (> 0)
 *   w_idx       [B,T,64] fp32               k_idx [B,Ncap,128] e4m3 codes
 *   k_idx_scale [B,Ncap] fp32 (> 0)          q_pos [B,T] int32, n_comp [B] int32
 *   logits      [B,T,Ncap] fp32 (written in full)
 * Requires 1 <= T <= CSA_MAX_TOKENS_PER_SEQ, Ncap >= 1, m >= 1. Accumulation
 * is fp32. Up to 4 tokens of a sequence share one read of its keys; larger T
 * (a prefill-style step, "ROADMAP -- Stage E" section E8) runs as groups of
 * up to 4 tokens (the largest of 4, 3, 2, 1 dividing T), each reading the
 * keys again. */
CSA_API csa_status_t csa_indexer_logits(const uint8_t *q_idx, const float *q_idx_scale, const float *w_idx,
                                const uint8_t *k_idx, const float *k_idx_scale,
                                const int32_t *q_pos, const int32_t *n_comp,
                                int B, int T, int Ncap, int m, float *logits, int32_t *status,
                                cudaStream_t stream);

/* Step 2 -- top-k of the indexer logits over the visible entries ("DSV4
 * Audit", section B2 and "ROADMAP -- Stage E", section E7: top-k per query
 * token with warp-level reductions and no global lock).
 * For each (b,t): the min(k, n_vis) entries c < n_vis with the largest
 * logits, ties going to the lower index, written to topk_idx[b,t,0..cnt) in
 * ascending index order, the rest of the row set to -1; topk_cnt[b,t] = cnt.
 *   logits [B,T,Ncap] fp32 (entries >= n_vis are not read), topk_idx [B,T,k]
 *   int32, topk_cnt [B,T] int32. Requires 1 <= k <= min(Ncap, CSA_MAX_TOPK).
 * The workspace may be NULL when csa_workspace_bytes(CSA_OP_TOPK, ...) is 0;
 * rows of more than 32768 entries with ceil(Ncap / 32768) * k <= 32768 are
 * selected in two stages and keep the slices' candidate indices there
 * (4 * B * T * ceil(Ncap / 32768) * (k + 1) bytes). */
CSA_API csa_status_t csa_topk(const float *logits, const int32_t *q_pos, const int32_t *n_comp,
                      int B, int T, int Ncap, int m, int k, int32_t *topk_idx, int32_t *topk_cnt,
                      void *workspace, size_t workspace_bytes, int32_t *status, cudaStream_t stream);

/* Step 3, standalone -- packed candidate records ("DSV4 Audit", section A3:
 * the query attends to [top-k compressed entries] ++ [SWA window]; a token in
 * both is kept twice; "ROADMAP -- Stage E", section E1: gathers straight from
 * the FP8 cache, block-table strided).
 * For each (b,t) with p = q_pos[b,t]: kv_out[b,t,i] = comp entry
 * topk_idx[b,t,i] for i < topk_cnt[b,t], followed by the SWA records of
 * positions max(0,p-W+1) .. p (oldest first), position j read from
 * swa_ring[b, j mod R]; kv_cnt[b,t] = number written. Slots past kv_cnt are
 * not written. Byte-exact copies, no dequantisation.
 *   swa_ring [B,R,592] bytes, kv_out [B,T,k+W,592] bytes, kv_cnt [B,T] int32.
 * Requires 1 <= W <= R and q_pos >= 0. The caller keeps the ring holding the
 * window of every query token (R >= W + T - 1 for consecutive tokens). */
CSA_API csa_status_t csa_gather_swa(csa_cache_desc comp, const void *swa_ring, int R, int W,
                            const int32_t *topk_idx, const int32_t *topk_cnt, const int32_t *q_pos,
                            int B, int T, int k, void *kv_out, int32_t *kv_cnt, int32_t *status,
                            cudaStream_t stream);

/* Step 4 -- sink-merged attention over [top-k entries] ++ [SWA window]
 * ("DSV4 Inference Kernel" README, Architecture: one 512-d latent per entry
 * shared by all 128 heads as key and value; sink weights merge the sparse and
 * SWA terms). With x_j the dequantised candidate latents (nope code times
 * its block multiplier, rope as BF16), for every head h:
 *   z_j   = softmax_scale * sum_d q[b,t,h,d] * x_j[d]
 *   M     = max(sink[h], max_j z_j)
 *   den   = exp(sink[h] - M) + sum_j exp(z_j - M)
 *   out   = sum_j exp(z_j - M) x_j / den       (BF16)
 *   lse   = M + ln(den)                         (fp32)
 * No candidates: out = 0 and lse = sink[h].
 *   q [B,T,128,512] bf16, sink [128] fp32, out [B,T,128,512] bf16,
 *   lse [B,T,128] fp32; other arguments as in csa_gather_swa.
 * The candidates are read straight from the caches (no packed copy). */
CSA_API csa_status_t csa_sink_attention_decode(const void *q, const float *sink, float softmax_scale,
                                       csa_cache_desc comp, const void *swa_ring, int R, int W,
                                       const int32_t *topk_idx, const int32_t *topk_cnt,
                                       const int32_t *q_pos, int B, int T, int k,
                                       void *out, float *lse, void *workspace, size_t workspace_bytes,
                                       int32_t *status, cudaStream_t stream);

/* HCA variant ("DSV4 Inference Kernel" README, Architecture, m' = 128;
 * "ROADMAP -- Stage E", section E1, gather of all compressed entries):
 * step 4 with the candidates = every visible entry c < n_vis(b,t) (computed
 * with m = m_hca as in csa_indexer_logits) ++ the SWA window. No indexer. */
CSA_API csa_status_t hca_sink_attention_decode(const void *q, const float *sink, float softmax_scale,
                                       csa_cache_desc comp, const int32_t *n_comp,
                                       const void *swa_ring, int R, int W, const int32_t *q_pos,
                                       int B, int T, int m_hca, void *out, float *lse,
                                       void *workspace, size_t workspace_bytes, int32_t *status,
                                       cudaStream_t stream);

/* Output epilogue of the attention ("DSV4 Audit" section A4: the attention
 * output is turned back by RoPE(-t) at the query position t, which makes the
 * absolute positions carried by the summed latents relative; "ROADMAP --
 * Stage E" section E6: the output may leave the attention as FP4 E2M1 with a
 * per-128-element block amax, packed inside the same launch). Used by the
 * _ex entry points; NULL there means plain BF16 output.
 *   inverse_rope   nonzero: the rope dims of every head's output, pair i =
 *                  dims (448 + 2i, 449 + 2i), i < 32, are turned back by
 *                  a = t * rope_theta^(-2i/64) radians, t = q_pos[b,t]:
 *                    x' = x cos a + y sin a,   y' = -x sin a + y cos a
 *                  (the pages fix no RoPE convention; this pairing and
 *                  frequency schedule are this library's reading)
 *   rope_theta     RoPE base, > 1 (e.g. 10000); read only with inverse_rope
 *   out_fp4        NULL: BF16 output in `out`. Otherwise device
 *                  [B,T,128,256] bytes, 16-byte aligned: the E2M1 codes of
 *                  the 512 output dims (after the rotation), dim 2i in the
 *                  low nibble of byte i; `out` is not written and may be NULL
 *   out_fp4_scale  with out_fp4: device [B,T,128,4] fp32, 16-byte aligned:
 *                  s = amax / 6 of output dims [128 j, 128 j + 128) (1 when
 *                  they are all zero); code = the E2M1 value nearest to
 *                  value / s (ties to even, saturating at 6), so that
 *                  value ~ e2m1(code) * s */
typedef struct {
    int32_t inverse_rope;
    float rope_theta;
    uint8_t *out_fp4;
    float *out_fp4_scale;
} csa_attention_epilogue;

/* csa_sink_attention_decode / hca_sink_attention_decode with an output
 * epilogue (see csa_attention_epilogue); identical to them when `epilogue`
 * is NULL or asks for neither step. Same workspace sizes. A bad epilogue
 * (theta <= 1 with inverse_rope, out_fp4 without out_fp4_scale, misaligned
 * pointers) returns CSA_ERR_INVALID_ARG before any launch. */
CSA_API csa_status_t csa_sink_attention_decode_ex(const void *q, const float *sink, float softmax_scale,
                                                  csa_cache_desc comp, const void *swa_ring, int R, int W,
                                                  const int32_t *topk_idx, const int32_t *topk_cnt,
                                                  const int32_t *q_pos, int B, int T, int k, void *out, float *lse,
                                                  const csa_attention_epilogue *epilogue, void *workspace,
                                                  size_t workspace_bytes, int32_t *status, cudaStream_t stream);
CSA_API csa_status_t hca_sink_attention_decode_ex(const void *q, const float *sink, float softmax_scale,
                                                  csa_cache_desc comp, const int32_t *n_comp, const void *swa_ring,
                                                  int R, int W, const int32_t *q_pos, int B, int T, int m_hca,
                                                  void *out, float *lse, const csa_attention_epilogue *epilogue,
                                                  void *workspace, size_t workspace_bytes, int32_t *status,
                                                  cudaStream_t stream);

/* Allocation-free variant of csa_sink_attention_decode (the pages have no
 * counterpart; it exists for callers of this library that cannot allocate
 * device memory on the decode path -- e.g. a serving runtime whose device
 * memory is all reserved by its own pool at start-up, a plugin whose host
 * framework owns every device allocation, or latency-critical host code that
 * cannot afford cudaMalloc's implicit synchronisation -- and so cannot pass a
 * workspace). Same arguments and results as csa_sink_attention_decode minus
 * the workspace: the split partials live in a static 16 MiB device array that
 * every device which loads the library holds until the process exits.
 *  - No cudaMalloc, cudaFree or allocating library call is made.
 *  - The first call on a device (with that device current) looks up the
 *    array's device address once (cudaGetSymbolAddress) and caches it; make
 *    that first call before any stream capture.
 *  - Sizes whose partials exceed the array return CSA_ERR_UNSUPPORTED (use
 *    csa_sink_attention_decode with a workspace instead); every size with
 *    csa_workspace_bytes(CSA_OP_ATTENTION, B, T, Ncap, k) <= 16 MiB fits.
 *  - Argument checks and their status codes are those of
 *    csa_sink_attention_decode; `status` is the caller's status word.
 *  - Every call shares the array and leaves its contents behind; nothing in it
 *    needs to start at zero. Calls that overlap on the GPU (concurrent streams)
 *    race on the array: serialise them. */
CSA_API csa_status_t csa_sink_attention_decode_noalloc(const void *q, const float *sink, float softmax_scale,
                                                       csa_cache_desc comp, const void *swa_ring, int R, int W,
                                                       const int32_t *topk_idx, const int32_t *topk_cnt,
                                                       const int32_t *q_pos, int B, int T, int k, void *out,
                                                       float *lse, int32_t *status, cudaStream_t stream);

/* One CSA decode step: csa_indexer_logits -> csa_topk ->
 * csa_sink_attention_decode on one stream. Logits, indices and attention
 * scratch live in the workspace (csa_workspace_bytes(CSA_OP_DECODE_STEP,...)).
 * The indexer keys are contiguous per sequence ([B,Ncap,...]); comp may be
 * paged. Arguments keep the meaning given above. topk_idx/topk_cnt may be
 * NULL; if given ([B,T,k] / [B,T]) they receive the selection. */
CSA_API csa_status_t csa_decode_step(const uint8_t *q_idx, const float *q_idx_scale, const float *w_idx,
                             const uint8_t *k_idx, const float *k_idx_scale,
                             const void *q, const float *sink, float softmax_scale,
                             csa_cache_desc comp, const void *swa_ring, int R, int W,
                             const int32_t *q_pos, const int32_t *n_comp,
                             int B, int T, int Ncap, int m, int k,
                             void *out, float *lse, int32_t *topk_idx, int32_t *topk_cnt,
                             void *workspace, size_t workspace_bytes, int32_t *status, cudaStream_t stream);

/* csa_decode_step with the attention's output epilogue
 * (csa_attention_epilogue; NULL = csa_decode_step): the step's last kernel
 * writes the inverse-RoPE'd and/or E2M1 output ("ROADMAP -- Stage E",
 * section E6: the quantised output leaves the attention in the same launch).
 * With E2M1 output `out` may be NULL. Checks as csa_decode_step plus those of
 * csa_sink_attention_decode_ex, all before the first launch. */
CSA_API csa_status_t csa_decode_step_ex(const uint8_t *q_idx, const float *q_idx_scale, const float *w_idx,
                                        const uint8_t *k_idx, const float *k_idx_scale, const void *q,
                                        const float *sink, float softmax_scale, csa_cache_desc comp,
                                        const void *swa_ring, int R, int W, const int32_t *q_pos,
                                        const int32_t *n_comp, int B, int T, int Ncap, int m, int k, void *out,
                                        float *lse, int32_t *topk_idx, int32_t *topk_cnt,
                                        const csa_attention_epilogue *epilogue, void *workspace,
                                        size_t workspace_bytes, int32_t *status, cudaStream_t stream);

/* Host-I/O decode pipeline (the pages have no counterpart; it serves callers
 * whose query-side inputs arrive in, and whose results go back to, host
 * memory). csa_decode_step_host runs csa_decode_step on per-step copies of
 * the query-side inputs taken from host memory and copies out/lse back to
 * host memory. Each step uses one of `depth` staging slots in device memory,
 * so the host->device copy of step i+1 and the device->host copy of step i-1
 * run on two copy streams while step i's kernels run on the compute stream;
 * nothing blocks the host until csa_pipeline_wait / csa_pipeline_sync
 * ("ROADMAP -- Stage E", section E4: no synchronisation on the decode path).
 * Results are identical to csa_decode_step on the same inputs.
 *
 * csa_pipeline_staging_bytes: device bytes of the staging area for these
 * sizes (depth slots of q_idx, q_idx_scale, w_idx, q, q_pos, out, lse, each
 * 256-byte aligned); 0 if an argument is out of range. */
typedef struct csa_pipeline_s *csa_pipeline_t;
#define CSA_PIPELINE_MAX_DEPTH 4

CSA_API size_t csa_pipeline_staging_bytes(int B, int T, int depth);

/* Creates a pipeline for B sequences x T tokens on the current device.
 *   staging   device memory of >= csa_pipeline_staging_bytes(B, T, depth)
 *             bytes, 256-byte aligned, owned by the caller and untouched by
 *             anything else while the pipeline lives
 *   depth     2..CSA_PIPELINE_MAX_DEPTH staging slots
 *   compute   the caller's stream for the kernels (0 = legacy default)
 * Allocates the host-side object and creates two non-blocking copy streams
 * and 3 x depth events on the current device (no device memory). Returns
 * CSA_ERR_INVALID_ARG for a null handle or staging, a misaligned or short
 * staging area, or sizes out of range; CSA_ERR_CUDA if a stream or event
 * cannot be created (nothing is left behind). */
CSA_API csa_status_t csa_pipeline_create(csa_pipeline_t *pipeline, int B, int T, int depth, void *staging,
                                         size_t staging_bytes, cudaStream_t compute);

/* Enqueues one decode step. Pointers prefixed h_ are HOST memory with the
 * layouts of csa_decode_step (q_idx [B,T,64,128] e4m3 codes, q_idx_scale and
 * w_idx [B,T,64] fp32, q [B,T,128,512] bf16, q_pos [B,T] int32; out
 * [B,T,128,512] bf16, lse [B,T,128] fp32); page-locked host memory lets the
 * copies run asynchronously and overlap (pageable memory works, serialised).
 * The other arguments are the device-resident layer state and sizes of
 * csa_decode_step (B and T are the pipeline's). The host inputs must stay
 * unchanged and the host outputs unread until csa_pipeline_wait(step) (or
 * csa_pipeline_sync) returns. *step_out (may be NULL) receives the step's
 * ordinal, 0 for the first step of the pipeline. Arguments are checked before
 * anything is enqueued; CSA_ERR_INVALID_ARG also when the current device is
 * not the pipeline's. */
CSA_API csa_status_t csa_decode_step_host(csa_pipeline_t pipeline, const uint8_t *h_q_idx,
                                          const float *h_q_idx_scale, const float *h_w_idx, const void *h_q,
                                          const int32_t *h_q_pos, const uint8_t *k_idx, const float *k_idx_scale,
                                          const float *sink, float softmax_scale, csa_cache_desc comp,
                                          const void *swa_ring, int R, int W, const int32_t *n_comp, int Ncap,
                                          int m, int k, void *h_out, float *h_lse, void *workspace,
                                          size_t workspace_bytes, int32_t *status, int64_t *step_out);

/* Blocks the host until step `step` (an ordinal returned by
 * csa_decode_step_host) has its results in host memory and its host inputs
 * are no longer read. CSA_ERR_INVALID_ARG for a step not yet enqueued;
 * CSA_ERR_CUDA if a copy or kernel failed. */
CSA_API csa_status_t csa_pipeline_wait(csa_pipeline_t pipeline, int64_t step);

/* Blocks the host until every enqueued step has completed. */
CSA_API csa_status_t csa_pipeline_sync(csa_pipeline_t pipeline);

/* Waits for every enqueued step, then releases the streams, events and host
 * object (not the staging memory, which the caller owns). NULL is a no-op. */
CSA_API csa_status_t csa_pipeline_destroy(csa_pipeline_t pipeline);

/* Reads and clears a status word without synchronising ("ROADMAP -- Stage
 * E", section E4: no synchronisation on the decode path; errors come back as
 * codes). Enqueues on `stream` a copy of *status (device) into *host_status
 * (host memory; page-locked memory keeps the copy asynchronous, pageable
 * memory makes the runtime stage it) followed by a reset of *status to
 * CSA_OK. The value in *host_status is valid once the stream has passed this
 * point (an event recorded after the call, or a synchronisation chosen by
 * the caller): CSA_OK, or the first CSA_ERR_TIMEOUT / CSA_ERR_BAD_INDEX that
 * a kernel recorded in the word since the previous reset. Work enqueued on
 * the stream after this call records into a clean word. Legal inside CUDA
 * graph capture. CSA_ERR_INVALID_ARG for a null or misaligned pointer,
 * CSA_ERR_CUDA if the copy or the reset cannot be enqueued. */
CSA_API csa_status_t csa_check_device_status(int32_t *status, int32_t *host_status, cudaStream_t stream);

/* Blocking convenience for tests and diagnostics: csa_check_device_status
 * into a local, then cudaStreamSynchronize(stream), then *host_code = the
 * value read. Not for the decode path. */
CSA_API csa_status_t csa_read_device_error(int32_t *status, int32_t *host_code, cudaStream_t stream);

/* Diagnostic: sets the time limit of the bounded waits inside the tensor-core
 * kernels (indexer and attention) for launches made after this call, in
 * nanoseconds of GPU global time; 0 restores the default of one second. A
 * wait that reaches the limit records CSA_ERR_TIMEOUT in the status word and
 * the kernel winds down: it drains its own copies and MMAs already in flight
 * (those waits keep the one-second limit), frees its tensor memory and exits.
 * Exists so that tests can drive the timeout path without hanging or faulting
 * anything; process-wide, not for the decode path. */
CSA_API void csa_debug_set_wait_limit_ns(uint64_t ns);

/* Static description of a status code. */
CSA_API const char *csa_status_string(csa_status_t status);

/* Number of kernels this process has launched through the library (all
 * devices, all streams; a host-side counter incremented at every launch). */
CSA_API uint64_t csa_kernel_launches(void);

/* Library ABI version (major * 100 + minor). */
CSA_API int csa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CSA_H_ */
