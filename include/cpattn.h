/*
 * cpattn.h -- C ABI of libcpattn.so: context-parallel (CP) ring attention for
 * long-context prefill, single GB300 GPU (sm_103a).
 *
 * Source of the operations: "Scaling LLM Inference: Innovations in Tensor
 * Parallelism, Context Parallelism, and Expert Parallelism" (Meta engineering
 * article, techreport.ngo rewrite), section "Context Parallelism for
 * Million-Token Contexts": the sequence is split across CP ranks; in Pass-KV
 * each rank keeps its Q and exchanges K and V so that it computes attention
 * over the full context; in Pass-Q the query tensors travel instead.  The
 * soumitrasaha.com reading notes of the same article (section "The
 * communication bottleneck across all three axes", CP paragraph) describe the
 * ring that passes K/V so each rank accumulates the full attention result.
 * The pages give no formula, interface or kernel; the conventions below are
 * this library's:
 *
 *   - Layout BSHD: q/o are [b, s, hq, d], k/v are [b, s, hkv, d], innermost
 *     dimension contiguous, other strides given in elements.
 *   - LSE is fp32, natural log of sum_j exp(scale * q.k_j), laid out
 *     [b, hq, s] contiguous.  A row with no visible key has LSE = -inf, O = 0.
 *   - Causal mask: key at absolute position pk is visible to a query at
 *     absolute position pq iff pk <= pq (inclusive diagonal).
 *   - GQA: query head h reads kv head h / (hq / hkv).
 *   - scale <= 0 selects 1/sqrt(d).
 *
 * Ownership and concurrency: the caller owns every buffer (inputs, outputs
 * and workspace are device memory unless stated).  The library never
 * allocates device memory, never frees, never synchronises the stream it is
 * given: every device-buffer compute call only enqueues kernels (and, for a
 * single-launch Pass-KV ring, one device memset of its progress counters) on
 * `stream` (a cudaStream_t; NULL = legacy default stream) and returns.  No
 * such call copies from host memory, so none waits on the host, and each can
 * be captured into a CUDA graph.  cpattn_prefill_host is the exception: its
 * contract is to copy host buffers and return finished results.
 *
 * Errors: argument errors are detected on the host before anything is
 * enqueued and return CPATTN_ERR_INVALID_ARG / CPATTN_ERR_UNSUPPORTED /
 * CPATTN_ERR_WORKSPACE with no side effect.  A failed launch returns
 * CPATTN_ERR_CUDA.  Faults during execution surface at the caller's next
 * synchronisation.  Kernel-side waits are bounded; one that gives up records
 * CPATTN_ERR_TIMEOUT in a device status word read by cpattn_device_status().
 * No C++ exception crosses this interface.
 */
#ifndef CPATTN_H_
#define CPATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CPATTN_OK = 0,
  CPATTN_ERR_INVALID_ARG = 1,  /* null pointer, bad shape/stride/alignment, bad enum */
  CPATTN_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. head_dim not 64/128) */
  CPATTN_ERR_WORKSPACE = 3,    /* workspace missing, misaligned or too small */
  CPATTN_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  CPATTN_ERR_TIMEOUT = 5,      /* a kernel-side bounded wait gave up (device status) */
  CPATTN_ERR_DEVICE_CHECK = 6  /* debug builds: a kernel bounds check failed (device status) */
} cpattn_status;

typedef enum { CPATTN_BF16 = 0, CPATTN_FP32 = 1 } cpattn_dtype;

/* The two ring schedules of the article's CP section. */
typedef enum { CPATTN_PASS_KV = 1, CPATTN_PASS_Q = 2 } cpattn_mode;

/*
 * A strided 4-D tensor view [b, s, h, d].  `data` is a device pointer (host
 * pointer for cpattn_prefill_host), 16-byte aligned.  Strides are in
 * elements, the d dimension is contiguous, and stride_b/stride_s/stride_h
 * times the element size must be multiples of 16 bytes.
 */
typedef struct {
  void *data;
  int32_t dtype; /* cpattn_dtype */
  int32_t reserved;
  int64_t b, s, h, d;
  int64_t stride_b, stride_s, stride_h;
} cpattn_tensor;

/*
 * cpattn_partial -- attention of one (Q-chunk, KV-chunk) pair with its LSE.
 * The per-pair step that both CP schedules run on every rank (article's CP
 * section, Pass-KV and Pass-Q bullets).
 *
 *   q      [b, sq, hq, d]    bf16 or fp32; row i is at absolute position q_off + i
 *   k, v   [b, skv, hkv, d]  same dtype as q; row j at absolute position kv_off + j
 *   causal nonzero: mask keys after each query's absolute position
 *   scale  logit scale; <= 0 selects 1/sqrt(d)
 *   o      [b, sq, hq, d]    output, bf16 or fp32 (fp32 keeps an unrounded partial)
 *   lse    [b, hq, sq]       fp32 output, contiguous
 * d must be 64 or 128; hq % hkv == 0.  sq or skv may be 0 (skv = 0 gives
 * empty rows: O = 0, LSE = -inf).
 */
cpattn_status cpattn_partial(const cpattn_tensor *q, const cpattn_tensor *k,
                             const cpattn_tensor *v, int64_t q_off, int64_t kv_off,
                             int causal, float scale, cpattn_tensor *o, float *lse,
                             void *stream);

/*
 * cpattn_merge -- in place, (o_a, lse_a) <- merge((o_a, lse_a), (o_b, lse_b)),
 * the LSE-weighted combination of two partial results over disjoint key sets:
 *   LSE = log(exp(LSE_a) + exp(LSE_b)),
 *   O   = exp(LSE_a - LSE) O_a + exp(LSE_b - LSE) O_b.
 * This is how a rank folds another rank's contribution into its own so that
 * it "accumulates the full attention result" (reading notes, CP paragraph).
 * o_a and o_b: same shape [b, s, h, d], same dtype (bf16 or fp32); lse_a and
 * lse_b: [b, h, s] fp32 contiguous.  Both sides -inf gives (0, -inf).
 */
cpattn_status cpattn_merge(cpattn_tensor *o_a, float *lse_a, const cpattn_tensor *o_b,
                           const float *lse_b, void *stream);

/*
 * cpattn_prefill_workspace_size -- device bytes cpattn_prefill needs for the
 * given shapes, schedule and mask.  Pass-KV: an fp32 running accumulator
 * [b, sq, hq, d] plus its LSE.  Pass-Q: one fp32 partial (O and LSE) per
 * non-empty (Q-chunk, KV-chunk) pair of every Q chunk that more than one KV
 * chunk reaches.  Writes the size to *bytes (0 is possible).
 */
cpattn_status cpattn_prefill_workspace_size(const cpattn_tensor *q, const cpattn_tensor *k,
                                            int64_t q_base, int n_chunks, int mode,
                                            int causal, size_t *bytes);

/*
 * cpattn_prefill -- CP prefill of one attention layer, emulating n_chunks CP
 * ranks on one GPU (article's CP section).  Q rows [c*sq/N, (c+1)*sq/N) and
 * K/V rows [c*skv/N, (c+1)*skv/N) form chunk c; query row i is at absolute
 * position q_base + i and key row j at position j.  Ring step t pairs rank r
 * with chunk (r - t) mod N of the travelling tensor: K/V for CPATTN_PASS_KV
 * (Q resident, online LSE accumulation fused into the attention kernel's
 * epilogue), Q for CPATTN_PASS_Q (K/V resident, per-pair partials merged by
 * LSE in ascending KV-chunk order after the ring).  Pairs with no visible key
 * are skipped.  Steps are launched back to back on `stream`.
 *
 *   n_chunks  1..64, dividing both sq and skv
 *   o         [b, sq, hq, d] bf16 or fp32;  lse [b, hq, sq] fp32 contiguous
 *   workspace device buffer of at least cpattn_prefill_workspace_size bytes,
 *             256-byte aligned (may be NULL when that size is 0)
 * Result: full causal attention of every query row over keys 0..skv-1.
 */
cpattn_status cpattn_prefill(const cpattn_tensor *q, const cpattn_tensor *k,
                             const cpattn_tensor *v, int64_t q_base, int n_chunks,
                             int mode, int causal, float scale, cpattn_tensor *o,
                             float *lse, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * cpattn_decode -- Pass-Q for decode-shaped queries: a few new tokens attend
 * to a long KV cache sharded over n_chunks emulated CP ranks (article's CP
 * section, Pass-Q bullet: query tensors are passed among the ranks while K/V
 * stay; the reading notes' framing that decode is memory-bound and prefill
 * compute-bound, section "The communication bottleneck across all three
 * axes").  Each rank's chunk is split further into pieces of whole 128-key
 * tiles so that every SM streams K/V; each piece yields an fp32 partial and
 * all partials are merged by LSE in ascending (chunk, piece) order.
 *
 *   q      [b, n_tok, hq, d]   token i at absolute position q_base + i
 *   k, v   [b, skv, hkv, d]    the cache; key row j at position j
 *   o, lse as for cpattn_prefill ([b, n_tok, hq, d], [b, hq, n_tok])
 *   n_chunks 1..64 dividing skv; workspace >= cpattn_decode_workspace_size
 * bf16 with d = 128 and n_tok * (hq / hkv) <= 128 (hq / hkv dividing 128)
 * packs all query heads of a kv head into one tensor-core tile; other shapes
 * run one tile per head (or the fp32/d=64 kernel) with one piece per chunk.
 */
cpattn_status cpattn_decode_workspace_size(const cpattn_tensor *q, const cpattn_tensor *k,
                                           int64_t q_base, int n_chunks, int causal,
                                           size_t *bytes);
cpattn_status cpattn_decode(const cpattn_tensor *q, const cpattn_tensor *k, const cpattn_tensor *v,
                            int64_t q_base, int n_chunks, int causal, float scale,
                            cpattn_tensor *o, float *lse, void *workspace, size_t workspace_bytes,
                            void *stream);

/*
 * One entry of the host-side ring plan (no GPU needed): at ring `step`, the
 * pair (q_chunk, kv_chunk) is computed and its result routed by `role`.
 */
typedef enum {
  CPATTN_ROLE_STORE = 0,      /* only contribution: write O/LSE to the output */
  CPATTN_ROLE_ACC_INIT = 1,   /* Pass-KV: first contribution, start the accumulator */
  CPATTN_ROLE_ACC_MERGE = 2,  /* Pass-KV: merge into the accumulator */
  CPATTN_ROLE_ACC_FINAL = 3,  /* Pass-KV: last contribution, merge and write the output */
  CPATTN_ROLE_PARTIAL = 4     /* Pass-Q: write an fp32 partial to workspace slot `slot` */
} cpattn_role;

typedef struct {
  int32_t step;      /* ring step t */
  int32_t q_chunk;   /* Q piece (= chunk for the contiguous assignment) */
  int32_t kv_chunk;  /* K/V piece */
  int32_t role;      /* cpattn_role */
  int32_t slot;      /* CPATTN_ROLE_PARTIAL: workspace slot, else -1 */
  int32_t launch;    /* index of the kernel launch that computes this pair */
  int32_t rank;      /* emulated CP rank that computes this pair */
} cpattn_plan_entry;

/*
 * cpattn_prefill_plan -- the pair list cpattn_prefill launches, in launch
 * order (host computation only).  Writes up to `capacity` entries and the
 * total count to *n_entries; returns CPATTN_ERR_INVALID_ARG for bad sizes.
 */
cpattn_status cpattn_prefill_plan(int64_t sq, int64_t skv, int64_t q_base, int n_chunks,
                                  int mode, int causal, cpattn_plan_entry *entries,
                                  int capacity, int *n_entries);

/*
 * Chunk-to-rank assignment (options of the *_ex calls).  With contiguous
 * chunks the causal work of rank r grows with r, so a real ring waits for
 * rank N-1 at every step.  CPATTN_ASSIGN_ZIGZAG cuts the sequence into 2N
 * pieces and gives rank r pieces r and 2N-1-r (the same for Q and K/V), which
 * evens the causal work out.  The result is the same attention either way.
 * Zigzag needs sq and skv divisible by 2N and N <= 32 (Pass-KV) or N <= 16
 * (Pass-Q); Pass-KV then launches once per visiting K/V piece.
 */
typedef enum { CPATTN_ASSIGN_CONTIGUOUS = 0, CPATTN_ASSIGN_ZIGZAG = 1 } cpattn_assignment;

/*
 * How the ring steps are launched (bf16, d = 128 tensor-core path; other
 * shapes always launch per step):
 *   PER_STEP             one launch per ring step, one CTA per work item;
 *   PERSISTENT_STEP      one launch per ring step, one CTA per SM looping over
 *                        the step's work items;
 *   SINGLE               one persistent launch for all ring steps (the
 *                        single-GPU form of a device-driven ring): work items
 *                        keep the ring order, and a Pass-KV accumulator update
 *                        waits -- bounded, CPATTN_ERR_TIMEOUT if it gives up --
 *                        until the previous step's update of the same rows has
 *                        finished.  Launched cooperatively (all CTAs resident).
 *   SINGLE_ONCHIP        one persistent launch for all ring steps; Pass-KV
 *                        keeps each query tile's accumulator on chip (TMEM)
 *                        while the visiting K/V pieces stream through it in
 *                        ring order, and writes O and LSE once (no fp32
 *                        accumulator in the workspace, no ordered waits).
 *                        Pass-Q runs as SINGLE.  Tensor-core kernel only
 *                        (bf16, head_dim 128); otherwise PER_STEP.
 *   AUTO                 when the tensor-core kernel applies (bf16, head_dim
 *                        128): for Pass-KV, SINGLE_ONCHIP when the ring's
 *                        work items are short -- fewer than 48 visible
 *                        128-key tiles per 128-row query tile on average,
 *                        where a CTA's fixed start-up and write-out cost is a
 *                        large share of its work -- or when K and V take at
 *                        most 96 MiB (they then stay in L2 while on-chip
 *                        items stream different pieces), else PER_STEP; for
 *                        Pass-Q, SINGLE when items are short, else PER_STEP.
 *                        Without the tensor-core kernel: PER_STEP.
 * CPATTN_LAUNCH_DEFAULT (options NULL or launch = DEFAULT) is AUTO.
 */
typedef enum {
  CPATTN_LAUNCH_PER_STEP = 0,
  CPATTN_LAUNCH_PERSISTENT_STEP = 1,
  CPATTN_LAUNCH_SINGLE = 2,
  CPATTN_LAUNCH_AUTO = 3,
  CPATTN_LAUNCH_DEFAULT = 3,
  CPATTN_LAUNCH_SINGLE_ONCHIP = 4
} cpattn_launch_mode;

/*
 * hold_ordered_waits -- failure-detection test only (zero in normal use).
 * Nonzero makes every ordered Pass-KV accumulator update of a SINGLE launch
 * wait for a progress count that is never reached: the wait gives up after
 * its bound (2 s), cpattn_device_status() then reports CPATTN_ERR_TIMEOUT, O
 * and LSE are undefined, and the CUDA context stays usable.  Ignored by the
 * other launch modes and by Pass-Q, which have no ordered updates.
 */
typedef struct {
  int32_t assignment;          /* cpattn_assignment */
  int32_t launch;              /* cpattn_launch_mode */
  int32_t hold_ordered_waits;  /* see above; 0 */
  int32_t reserved[5];         /* zero */
} cpattn_prefill_options;

/*
 * cpattn_prefill_launch_mode -- the launch mode cpattn_prefill_ex would use
 * for these shapes and options (CPATTN_LAUNCH_AUTO resolved to PER_STEP,
 * SINGLE or SINGLE_ONCHIP; an explicit mode is returned as given).  Host
 * only, no CUDA call.
 */
cpattn_status cpattn_prefill_launch_mode(const cpattn_tensor *q, const cpattn_tensor *k,
                                         int64_t q_base, int n_chunks, int mode, int causal,
                                         const cpattn_prefill_options *opts, int *launch);

/* cpattn_prefill / _workspace_size / _plan with options (NULL = defaults). */
cpattn_status cpattn_prefill_ex(const cpattn_tensor *q, const cpattn_tensor *k,
                                const cpattn_tensor *v, int64_t q_base, int n_chunks, int mode,
                                int causal, float scale, cpattn_tensor *o, float *lse,
                                void *workspace, size_t workspace_bytes,
                                const cpattn_prefill_options *opts, void *stream);
cpattn_status cpattn_prefill_workspace_size_ex(const cpattn_tensor *q, const cpattn_tensor *k,
                                               int64_t q_base, int n_chunks, int mode, int causal,
                                               const cpattn_prefill_options *opts, size_t *bytes);
cpattn_status cpattn_prefill_plan_ex(int64_t sq, int64_t skv, int64_t q_base, int n_chunks,
                                     int mode, int causal, const cpattn_prefill_options *opts,
                                     cpattn_plan_entry *entries, int capacity, int *n_entries);

/*
 * cpattn_prefill_critical_path -- the ring's critical path on N GPUs, from
 * the plan (host only): each step lasts as long as its busiest rank, so
 * *critical = sum over steps of max over ranks of the rank's work, *total =
 * all work, both in visible (query, key) pairs per (batch, head) (multiply by
 * 4 * d * hq * b for FLOPs).  step_max (may be NULL) receives the per-step
 * maxima [n_chunks].  total / (N * critical) is the ring's load balance.
 */
cpattn_status cpattn_prefill_critical_path(int64_t sq, int64_t skv, int64_t q_base, int n_chunks,
                                           int mode, int causal,
                                           const cpattn_prefill_options *opts,
                                           double *step_max, double *critical, double *total);

/*
 * cpattn_prefill_choose_mode -- pick the ring schedule that moves fewer bytes
 * between CP ranks (host only; the article's CP section offers both Pass-KV
 * and Pass-Q without a rule, this is the plainest traffic model).  Over the
 * N - 1 ring hops every rank forwards one chunk:
 *   Pass-KV bytes = N (N-1) * 2 * C_kv * hkv * d * es           (K and V travel)
 *   Pass-Q  bytes = N (N-1) * C_q * hq * (d * es                (Q travels)
 *                                          + d * es + 4)        (O and LSE return)
 * with C_kv = skv / N, C_q = sq / N and es the element size.  *mode receives
 * the cheaper one (ties go to Pass-KV); either byte count pointer may be NULL.
 */
cpattn_status cpattn_prefill_choose_mode(const cpattn_tensor *q, const cpattn_tensor *k,
                                         int n_chunks, int *mode, double *pass_kv_bytes,
                                         double *pass_q_bytes);

/*
 * cpattn_prefill_choose_mode_ex -- the same choice for the ring that
 * cpattn_prefill_ex actually runs (q_base, causal mask, chunk-to-rank
 * assignment of `opts`; host only).  A chunk travels only as far as the
 * ring needs it: at step t rank r holds the travelling chunk of rank
 * (r - t) mod N, so the chunk of rank s makes max (r - s) mod N hops over the
 * ranks r whose pairs with it have a visible key (0 if none).  With a causal
 * mask and contiguous chunks K/V therefore travel N (N-1) / 2 hops in all,
 * Q (N-1)^2 (a Q chunk sees the ranks before it, which the ring reaches
 * last).  Bytes:
 *   Pass-KV = sum over ranks of hops * 2 * (pieces per rank) * C_kv * hkv * d * es * b
 *   Pass-Q  = sum over ranks of hops * (pieces per rank) * C_q * hq * d * es * b
 *             + (visible piece pairs on different ranks) * C_q * hq * (d * es + 4) * b
 *             (each remote partial O and its LSE return to the Q owner once)
 * with C_kv, C_q the piece lengths.  *mode receives the cheaper schedule (ties
 * go to Pass-KV); either byte count pointer may be NULL.
 */
cpattn_status cpattn_prefill_choose_mode_ex(const cpattn_tensor *q, const cpattn_tensor *k,
                                            int64_t q_base, int n_chunks, int causal,
                                            const cpattn_prefill_options *opts, int *mode,
                                            double *pass_kv_bytes, double *pass_q_bytes);

/*
 * cpattn_prefill_host -- end-to-end convenience: q, k, v, o are HOST tensors
 * (pageable or pinned); lse is a host array [b, hq, sq].  Copies inputs to
 * device staging buffers the caller provides (`dev_scratch`, at least
 * cpattn_prefill_host_scratch_size bytes, 256-byte aligned), runs
 * cpattn_prefill there, copies O and LSE back, and synchronises `stream`.
 * The copies overlap the ring: Q goes up one piece at a time after K and V,
 * work starts on each piece once it has landed, and output pieces go back as
 * soon as they are final.  The launch mode is AUTO's.  One launch per ring
 * step: the first step runs one launch per pair, each as its Q piece lands.
 * Where work items are long the call works through consecutive groups of Q
 * pieces in arrival order (a small first group, up to three of about equal
 * size, then the last piece alone), each started once its pieces are in and
 * each group's rows copied back while the later groups run: the on-chip
 * Pass-KV launch becomes one launch per group, and Pass-Q runs the ring's
 * pairs grouped by Q piece, each group merged right after its pairs.  Every
 * pair and merge is computed as in cpattn_prefill, so results equal its bit
 * for bit.
 */
cpattn_status cpattn_prefill_host_scratch_size(const cpattn_tensor *q, const cpattn_tensor *k,
                                               int64_t q_base, int n_chunks, int mode,
                                               int causal, int out_dtype, size_t *bytes);
cpattn_status cpattn_prefill_host(const cpattn_tensor *q, const cpattn_tensor *k,
                                  const cpattn_tensor *v, int64_t q_base, int n_chunks,
                                  int mode, int causal, float scale, cpattn_tensor *o,
                                  float *lse, void *dev_scratch, size_t scratch_bytes,
                                  void *stream);

/*
 * cpattn_prefill_noalloc -- cpattn_prefill without a caller-provided
 * workspace; this call allocates nothing.  The paper has no counterpart: it
 * is an interface convenience of this library.
 *
 * For callers that cannot call cudaMalloc: code embedded in a framework whose
 * own pool owns all device memory and forbids raw allocations, or a
 * latency-critical loop that cannot afford cudaMalloc's implicit device
 * synchronisation.  The caller still provides q, k, v, o and lse; the Pass-KV
 * accumulator or the Pass-Q partial stack lives in one static device buffer
 * of CPATTN_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that
 * loads this code holds until the process exits.
 *
 *   - Problems whose cpattn_prefill_workspace_size exceeds
 *     CPATTN_NOALLOC_SCRATCH_BYTES return CPATTN_ERR_UNSUPPORTED before
 *     anything is enqueued (e.g. Pass-KV fits sq * hq * b <= ~130K rows at d = 128).
 *   - The first call in each CUDA context of a device (the first call on
 *     the device, and again after a cudaDeviceReset) looks up the buffer's
 *     device address (cudaGetSymbolAddress) with that device current; make
 *     that first call before any stream capture.
 *   - All calls share the one buffer and it keeps the previous call's
 *     contents; nothing in it has to start at zero.  Calls that overlap on
 *     the GPU (different streams, or different host threads without ordering)
 *     race on the buffer: serialise them.
 * Other arguments and errors as for cpattn_prefill.
 */
#define CPATTN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
cpattn_status cpattn_prefill_noalloc(const cpattn_tensor *q, const cpattn_tensor *k,
                                     const cpattn_tensor *v, int64_t q_base, int n_chunks,
                                     int mode, int causal, float scale, cpattn_tensor *o,
                                     float *lse, void *stream);

/* Human-readable name of a status code (static string). */
const char *cpattn_status_string(cpattn_status s);

/*
 * cpattn_device_status -- read (and if `clear`, reset) the device status words
 * that kernels set when a bounded wait gives up, or -- in a library built with
 * -DCPATTN_DEBUG -- when a bounds check on a destination row, workspace slot
 * or progress counter fails (the write is skipped; nothing traps).
 * Synchronises the device.  Returns CPATTN_OK, CPATTN_ERR_TIMEOUT (takes
 * precedence), CPATTN_ERR_DEVICE_CHECK or CPATTN_ERR_CUDA.
 */
cpattn_status cpattn_device_status(int clear);

/*
 * Launch profiling for benchmarks.  cpattn_profile_begin(capacity) arms
 * recording: each later kernel launch by this library records a pair of CUDA
 * events around it on its stream (host-side resources only, up to
 * `capacity` launches).  cpattn_profile_end() synchronises those events,
 * fills up to `capacity` records and disarms.  `work` is the launch's
 * algorithmic work: causal-effective FLOPs for attention kernels, bytes
 * moved for merge kernels.  Not thread safe.
 */
typedef enum {
  CPATTN_KERNEL_ATTN_TC = 1,    /* tcgen05 partial-attention kernel */
  CPATTN_KERNEL_ATTN_SIMT = 2,  /* fp32 / head_dim 64 partial-attention kernel */
  CPATTN_KERNEL_MERGE2 = 3,     /* pairwise LSE merge */
  CPATTN_KERNEL_MERGEN = 4,     /* N-way LSE merge of Pass-Q partials */
  CPATTN_KERNEL_TABLE = 5,      /* pair-table upload of a single-launch ring (work = bytes) */
  CPATTN_KERNEL_ATTN_TC_ONCHIP = 6  /* tcgen05 kernel, Pass-KV with the accumulator on chip */
} cpattn_kernel_kind;

typedef struct {
  int32_t kind; /* cpattn_kernel_kind */
  float ms;
  double work;
} cpattn_profile_record;

cpattn_status cpattn_profile_begin(int capacity);
cpattn_status cpattn_profile_end(cpattn_profile_record *records, int capacity, int *n_records);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H_ */
