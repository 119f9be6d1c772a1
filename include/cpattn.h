/*
 * cpattn -- context-parallel ring attention for one GB300 (sm_103a).
 *
 * The C ABI of the hot path behind context parallelism (CP): blockwise causal
 * ring attention over a packed variable-length (THD) batch, with the
 * online-softmax merge that folds each KV chunk's partial result into the
 * running (O, m, l), and the dynamic-CP planner that picks each sample's CP
 * size.  CP is emulated on one GPU: a sample split over c ranks becomes c
 * chunks resident in device memory, and the ring's KV hand-off becomes a loop
 * over those chunks in ring order.
 *
 * Sources (cited by title and section):
 *   [6D-CP] "Megatron 架构与 6D 并行完整指南", section 六 (context parallelism in
 *           depth): the ring_attention listing and its online-softmax merge.
 *   [DCP]   "Dynamic Context Parallelism (DCP)", verl 0.9.0 docs,
 *           docs/advance/dynamic_context_parallel.
 *   [MCore] "20-Megatron-MCore-TP-PP-EP如何支撑MoE", sections 1 and 4.
 *
 * Conventions shared by every call:
 *   - Packed THD layout.  Q, K, V and O are [T, H, D] row-major (D fastest);
 *     LSE, m and l are [T, H]; per-step partials are [S, T, H, D] and
 *     [S, T, H].  cu_seqlens is the [B + 1] prefix sum of sample lengths,
 *     cu_seqlens[0] = 0 and cu_seqlens[B] = T.
 *   - Positions are 0-based within a sample.  A sample of length L with CP
 *     size c is split into contiguous chunks of ceil(L / c) tokens; chunk r is
 *     [r * ceil(L/c), min((r+1) * ceil(L/c), L)) and the last chunks may be
 *     short or empty.  Rank r holds Q chunk r and, at ring step s, the KV chunk
 *     of rank (r - s) mod c.
 *   - Causal attention lets position p see key positions 0..p of its own
 *     sample.  Scores are softmax_scale * <q, k>; LSE is the natural-log
 *     log-sum-exp of the scaled scores.
 *   - The library allocates no device memory.  Every buffer is owned by the
 *     caller; the library never frees or retains one past the call (except
 *     through work already enqueued on `stream`).
 *   - Device calls enqueue on `stream` (a cudaStream_t, NULL = legacy default
 *     stream) and return without synchronising.  Argument errors are detected
 *     on the host and return before anything is enqueued.  Errors found by the
 *     kernels (bad cu_seqlens, a CP size above max_cp, a bounded wait that ran
 *     out) are written to the workspace's error word and read back with
 *     cpattn_poll_error.
 *   - Device pointers must be 16-byte aligned; float arrays 4-byte aligned.
 *   - Thread safety: calls may be made from several host threads; internal
 *     state is a mutex-guarded cache of device properties.
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
  CPATTN_ERR_INVALID_ARG = 1,        /* bad pointer, size, alignment or layout   */
  CPATTN_ERR_UNSUPPORTED = 2,        /* e.g. head_dim other than 64 or 128       */
  CPATTN_ERR_WORKSPACE_TOO_SMALL = 3,
  CPATTN_ERR_PLAN_INFEASIBLE = 4,    /* a sample does not fit at max_cp          */
  CPATTN_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed        */
  CPATTN_ERR_DEVICE_TIMEOUT = 6,     /* a kernel's bounded wait ran out          */
  CPATTN_ERR_DEVICE_BOUNDS = 7       /* debug build only: a kernel's bounds check
                                        failed (the access was skipped)          */
} cpattn_status;

/* Kernel modes of cpattn_fwd. */
#define CPATTN_MODE_FUSED 0    /* merge folded into the attention kernel        */
#define CPATTN_MODE_UNFUSED 1  /* per-step partials in the workspace, then merge */

/*
 * cpattn_plan -- dynamic-CP planning of one mini-batch (host only).
 *
 * [DCP]: the CP size is chosen per sample from its length by a
 * sequence-length-aware scheduler; every DPxCP rank sees the same samples;
 * the DPxCP world size is even and at least 2; CP groups are power-of-two
 * subgroups plus, when needed, the full DPxCP group; the per-rank packing
 * limit is max_seqlen_per_dp_cp_rank (the static budget divided by the static
 * CP size, e.g. 16384 / 4 = 4096).  [MCore] section 4: a micro-batch holds
 * world * limit tokens.  The pages do not give the scheduler's algorithm;
 * this call implements the following deterministic rules:
 *   1. cp_size[b] = smallest c in {1, 2, 4, ... < max_cp} U {max_cp} with
 *      ceil(seqlens[b] / c) <= max_seqlen_per_dp_cp_rank;
 *   2. samples are placed longest first, equal lengths by ascending index;
 *   3. a sample with CP c occupies an aligned rank group [g*c, (g+1)*c),
 *      g = 0 .. world/c - 1, adding ceil(L / c) tokens to each rank's load;
 *   4. first fit: the first micro-batch (in creation order) and within it the
 *      first group where every rank stays within the limit; otherwise a new
 *      micro-batch is opened and the sample takes its group 0.
 *
 * Arguments (all host memory, owned by the caller):
 *   seqlens            [n] sample lengths, each >= 0.
 *   n                  number of samples, >= 0.
 *   dpxcp_world_size   W, even, 2 <= W <= 4096.
 *   max_seqlen_per_dp_cp_rank   per-rank token limit, >= 1.
 *   max_cp             largest CP size: a power of two <= W, or W itself.
 *   cp_size, micro_batch, first_rank   [n] outputs per original sample index.
 *   order              [n] output: sample indices in placement order.
 *   num_micro_batches  [1] output.
 *   rank_load          [n * W] output or NULL: rank_load[mb * W + r] is the
 *                      token load of rank r in micro-batch mb, for
 *                      mb < *num_micro_batches; the rest is left untouched.
 * Returns CPATTN_OK, CPATTN_ERR_INVALID_ARG (argument rule broken; outputs
 * untouched) or CPATTN_ERR_PLAN_INFEASIBLE (some ceil(L / max_cp) exceeds the
 * limit; outputs untouched).
 */
int cpattn_plan(const int32_t* seqlens, int32_t n, int32_t dpxcp_world_size,
                int32_t max_seqlen_per_dp_cp_rank, int32_t max_cp,
                int32_t* cp_size, int32_t* micro_batch, int32_t* first_rank,
                int32_t* order, int32_t* num_micro_batches, int32_t* rank_load);

/*
 * cpattn_fwd_workspace_size -- bytes of device workspace cpattn_fwd needs.
 *
 * total_tokens T, num_seqs B, num_heads H, head_dim D, max_cp (the bound on
 * every cp_size[b]) and mode as passed to cpattn_fwd.  In CPATTN_MODE_UNFUSED
 * the workspace also holds the per-step partials (max_cp * T * H * (D + 2)
 * floats).  Returns 0 for invalid arguments.
 */
size_t cpattn_fwd_workspace_size(int64_t total_tokens, int32_t num_seqs,
                                 int32_t num_heads, int32_t head_dim,
                                 int32_t max_cp, int32_t mode);

/*
 * cpattn_fwd -- ring attention forward over a packed THD batch.
 *
 * [6D-CP] ring_attention: for every sample b split into c = cp_size[b]
 * chunks and every rank i, start from O = 0, m = -inf, l = 0; for
 * step = 0 .. c-1 attend Q chunk i to KV chunk (i - step) mod c (block
 * attention giving O_step, m_step, l_step) and fold it in with
 *   m_new = max(m, m_step), alpha = exp(m - m_new), beta = exp(m_step - m_new),
 *   l = alpha * l + beta * l_step, O = alpha * O + beta * O_step, m = m_new;
 * return O / l.  The result equals full softmax attention of each sample up
 * to rounding.  CPATTN_MODE_FUSED keeps (O, m, l) on chip for all steps;
 * CPATTN_MODE_UNFUSED writes every step's (O_step, m_step, l_step) to the
 * workspace and folds them with the merge kernel.
 *
 * Arguments:
 *   q, k, v        device, bf16 [T, H, D], 16-byte aligned.
 *   cu_seqlens     device int32 [B + 1].
 *   cp_size        device int32 [B] with 1 <= cp_size[b] <= max_cp, or NULL
 *                  (every sample at CP 1).
 *   num_seqs       B >= 0.   total_tokens  T >= 0 (= cu_seqlens[B]).
 *   max_seqlen     upper bound on every sample length (> 0 when T > 0).
 *   max_cp         upper bound on cp_size[b], 1 .. 64.
 *   num_heads      H >= 1.   head_dim  D in {64, 128} (else UNSUPPORTED).
 *   softmax_scale  multiplies <q, k>; finite and > 0.
 *   causal         1 causal, 0 full attention within each sample.
 *   mode           CPATTN_MODE_FUSED or CPATTN_MODE_UNFUSED.
 *   out            device bf16 [T, H, D]: O / l.
 *   lse            device float [T, H]: m + ln l (natural log).  May be NULL.
 *   workspace      device, >= cpattn_fwd_workspace_size(...) bytes, 256-byte
 *                  aligned; its first bytes hold the error word.
 *   stream         cudaStream_t.
 * The kernels check cu_seqlens (non-decreasing, cu[0] = 0, cu[B] = T, every
 * length <= max_seqlen) and cp_size (1 .. max_cp); a violation sets
 * CPATTN_ERR_INVALID_ARG in the error word and writes no output.
 */
int cpattn_fwd(const void* q, const void* k, const void* v,
               const int32_t* cu_seqlens, const int32_t* cp_size,
               int32_t num_seqs, int64_t total_tokens, int32_t max_seqlen,
               int32_t max_cp, int32_t num_heads, int32_t head_dim,
               float softmax_scale, int32_t causal, int32_t mode,
               void* out, float* lse, void* workspace, size_t workspace_bytes,
               void* stream);

/*
 * cpattn_fwd_partials -- the per-step block attentions of the ring, stored.
 *
 * [6D-CP]: the result of each ring step's block attention before it is
 * merged: for token t (rank i of its sample) and step s < c,
 *   m_steps[s, t, h] = max of the visible scaled scores against KV chunk
 *                      (i - s) mod c (-inf when none is visible),
 *   l_steps[s, t, h] = sum of exp(score - m_steps),
 *   o_steps[s, t, h, :] = sum of exp(score - m_steps) * v  (not normalised).
 * Steps s >= c, and steps that see no key, hold (0, -inf, 0).  The kernel may
 * use any reference value in place of the exact step maximum, as long as
 * o_steps and l_steps are scaled by the same exp(-reference): every quantity
 * the merge uses (O_step / l_step and m_step + ln l_step) is unchanged.
 *
 * Arguments as cpattn_fwd, plus:
 *   num_steps  S >= max_cp.
 *   o_steps    device float [S, T, H, D];  m_steps, l_steps device float
 *              [S, T, H].  Caller-owned; every element is written.
 *   workspace  >= cpattn_fwd_workspace_size(T, B, H, D, max_cp,
 *              CPATTN_MODE_FUSED) bytes.
 */
int cpattn_fwd_partials(const void* q, const void* k, const void* v,
                        const int32_t* cu_seqlens, const int32_t* cp_size,
                        int32_t num_seqs, int64_t total_tokens,
                        int32_t max_seqlen, int32_t max_cp, int32_t num_heads,
                        int32_t head_dim, float softmax_scale, int32_t causal,
                        int32_t num_steps, float* o_steps, float* m_steps,
                        float* l_steps, void* workspace, size_t workspace_bytes,
                        void* stream);

/*
 * cpattn_merge -- fold S stored partials with the [6D-CP] merge.
 *
 * For every row (t, h): starting from (O, m, l) = (0, -inf, 0), fold steps
 * s = 0 .. S-1 with the formulas above; exp(-inf - x) counts as 0.  Writes
 *   out_o[t, h, :] = O / l (0 when l = 0), out_m[t, h] = m, out_l[t, h] = l.
 * The kernel evaluates the fold in closed form (m* = max_s m_s first, then
 * sums weighted by exp(m_s - m*)), which is the same value up to rounding.
 *
 * Arguments (device float, caller-owned, 16-byte aligned):
 *   o_steps [S, T, H, D], m_steps [S, T, H], l_steps [S, T, H];
 *   num_steps S in 1 .. 64; T >= 0; H >= 1; D in {64, 128};
 *   out_o [T, H, D]; out_m, out_l [T, H] (either may be NULL).
 */
int cpattn_merge(const float* o_steps, const float* m_steps,
                 const float* l_steps, int32_t num_steps, int64_t total_tokens,
                 int32_t num_heads, int32_t head_dim, float* out_o,
                 float* out_m, float* out_l, void* stream);

/*
 * cpattn_bwd_workspace_size -- bytes of device workspace cpattn_bwd needs for
 * a problem of this size (0 on invalid arguments).  The workspace holds the
 * error word, the schedule, one 16-byte work entry per backward CTA (two
 * tables) and D = rowsum(dO * O) as float32 [T, H].
 */
size_t cpattn_bwd_workspace_size(int64_t total_tokens, int32_t num_seqs,
                                 int32_t num_heads, int32_t head_dim,
                                 int32_t max_cp);

/*
 * cpattn_bwd -- gradients dQ, dK, dV of cpattn_fwd's output O with respect to
 * Q, K and V, for an upstream gradient dO.
 *
 * The pages run a backward pass after the forward in every training step
 * ("20-Megatron-MCore-TP-PP-EP如何支撑MoE", section 4, forward_backward_batch;
 * "VeRL Backend Parallelism", MindSpeed-MM recipe, loss.backward()) but give no
 * formula; this is the exact derivative of the forward's definition ("Megatron
 * 架构与 6D 并行完整指南", section 六).  With P = exp(scale * Q K^T - LSE) over
 * the visible pairs of each sample:
 *   dV = P^T dO,  D = rowsum(dO * O),  dS = P * (dO V^T - D),
 *   dQ = scale * dS K,  dK = scale * dS^T Q.
 * The work follows the ring's chunks of each sample (cp_size): dQ of a query
 * block walks the KV chunks in the forward's ring order; dK, dV of a key block
 * walk the query chunks that see it in the order they visit it.
 *
 * Arguments (device pointers unless stated; everything enqueued on `stream`):
 *   q, k, v, cu_seqlens, cp_size, num_seqs, total_tokens, max_seqlen, max_cp,
 *   num_heads, head_dim, softmax_scale, causal
 *          exactly as passed to the cpattn_fwd call being differentiated.
 *   out    bf16 [T, H, D]: that call's O (16-byte aligned).
 *   dout   bf16 [T, H, D]: dO (16-byte aligned).
 *   lse    float32 [T, H]: that call's LSE (natural log).
 *   dq, dk, dv  bf16 [T, H, D] outputs (16-byte aligned; every row of every
 *          sample is written).
 *   workspace, workspace_bytes  at least cpattn_bwd_workspace_size(...) bytes,
 *          256-byte aligned, caller-owned.
 * Precision: fp32 accumulation on the tensor cores; P and dS are rounded to
 * bf16 before their products; outputs are rounded to bf16.
 * Errors: argument problems return CPATTN_ERR_INVALID_ARG /
 * CPATTN_ERR_UNSUPPORTED / CPATTN_ERR_WORKSPACE_TOO_SMALL before anything is
 * enqueued; device-side problems are reported by cpattn_poll_error.
 */
int cpattn_bwd(const void* q, const void* k, const void* v, const void* out,
               const void* dout, const float* lse, const int32_t* cu_seqlens,
               const int32_t* cp_size, int32_t num_seqs, int64_t total_tokens,
               int32_t max_seqlen, int32_t max_cp, int32_t num_heads,
               int32_t head_dim, float softmax_scale, int32_t causal, void* dq,
               void* dk, void* dv, void* workspace, size_t workspace_bytes,
               void* stream);

/*
 * Dynamic-CP data movement ("Dynamic Context Parallelism (DCP)", verl
 * documentation: each DPxCP rank selects its assigned samples from the shared
 * mini-batch; each CP group's output is gathered; verl restores the original
 * sample order afterwards).  On one device both are permutations of whole
 * samples between the original packed THD array (samples 0..num_seqs-1 in
 * original order, cu_seqlens `orig_cu`) and a packed array holding samples
 * ids[0..n-1] in that order (cu_seqlens `pack_cu`).
 *
 * cpattn_select_cu -- pack_cu of a selection: dst_cu[0] = 0,
 *   dst_cu[i+1] = dst_cu[i] + length of sample ids[i].
 *   src_cu   device int32 [num_seqs + 1] (original cu_seqlens)
 *   ids      device int32 [n]; dst_cu device int32 [n + 1] (written)
 *   status   device int32 [1]: set to 0, or to 1 if an id is outside
 *            [0, num_seqs) (such a sample counts as empty; the permutation
 *            below then copies nothing).
 * cpattn_permute_samples -- copies rows of row_bytes bytes (a multiple of 4;
 *   16-byte vector copies when it and both buffers allow): gather = 1 copies
 *   sample ids[i] of the original array `src` to slot i of the packed array
 *   `dst`; gather = 0 copies slot i of the packed array `src` back to sample
 *   ids[i] of the original array `dst`.  `status` is the word
 *   cpattn_select_cu wrote for these ids (nothing is copied when it is
 *   nonzero).  The packed array holds pack_cu[n] rows; rows of a slot
 *   beyond its original sample's length are not copied.  Samples not in ids
 *   are untouched.
 * Both enqueue on `stream` and return CPATTN_ERR_INVALID_ARG for null or
 * misaligned pointers and negative sizes before launching.
 */
int cpattn_select_cu(const int32_t* src_cu, int32_t num_seqs, const int32_t* ids,
                     int32_t n, int32_t* dst_cu, int32_t* status, void* stream);
int cpattn_permute_samples(const void* src, const int32_t* orig_cu,
                           int32_t num_seqs, const int32_t* pack_cu,
                           const int32_t* ids, int32_t n, int64_t row_bytes,
                           int32_t gather, void* dst, const int32_t* status,
                           void* stream);

/*
 * Decode-time context parallelism ("VeRL Backend Parallelism", backend matrix
 * and vLLM inference section: for the vLLM engines CP means decode context
 * parallelism, the KV cache of a sequence split over ranks).  One new query
 * token per sequence attends to every cached key of its sequence; with decode
 * CP size `cp` the cache of a sequence of length L is cut into cp contiguous
 * shards of ceil(L / cp) keys, shard s gives the normalised partial
 * O_s = softmax(scale q K_s^T) V_s with lse_s = ln sum exp(scale q K_s^T)
 * (an empty shard: O_s = 0, lse_s = -inf), and the partials merge in the LSE
 * form: LSE = ln sum_s exp(lse_s), O = sum_s exp(lse_s - LSE) O_s.
 *
 *   q      bf16 [num_seqs, H, D] (16-byte aligned): the new tokens
 *   k, v   bf16 [total_tokens, H, D]: the KV cache, packed by cu_seqlens
 *   cu_seqlens  device int32 [num_seqs + 1]
 *   head_dim 64 or 128; 1 <= cp <= 64.
 *
 * cpattn_decode_partials -- the shard partials: o_steps float32
 *   [cp, num_seqs, H, D] (16-byte aligned), lse_steps float32 [cp, num_seqs, H].
 * cpattn_merge_lse -- the LSE-form merge of `num_steps` normalised partials
 *   over `rows` rows: out_o float32 [rows, D], out_lse float32 [rows] or NULL.
 * cpattn_decode -- both: out bf16 [num_seqs, H, D], lse float32 [num_seqs, H]
 *   or NULL; workspace >= cpattn_decode_workspace_size(...) bytes, 256-byte
 *   aligned (holds the partials).
 * All enqueue on `stream`; argument errors return before any launch.
 */
size_t cpattn_decode_workspace_size(int32_t num_seqs, int32_t num_heads,
                                    int32_t head_dim, int32_t cp);
int cpattn_decode_partials(const void* q, const void* k, const void* v,
                           const int32_t* cu_seqlens, int32_t num_seqs,
                           int64_t total_tokens, int32_t num_heads,
                           int32_t head_dim, float softmax_scale, int32_t cp,
                           float* o_steps, float* lse_steps, void* stream);
int cpattn_merge_lse(const float* o_steps, const float* lse_steps,
                     int32_t num_steps, int64_t rows, int32_t head_dim,
                     float* out_o, float* out_lse, void* stream);
int cpattn_decode(const void* q, const void* k, const void* v,
                  const int32_t* cu_seqlens, int32_t num_seqs,
                  int64_t total_tokens, int32_t num_heads, int32_t head_dim,
                  float softmax_scale, int32_t cp, void* out, float* lse,
                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Ulysses sequence parallelism ("VeRL Backend Parallelism", the USP section:
 * verl's ulysses_sequence_parallel_size splits the sequence over the SP group
 * of a [dp, sp] mesh; an all-to-all before attention gives every rank the
 * whole sequence for H / P of the heads, and the inverse follows attention).
 * The sequence shards of the P ranks, concatenated, are the packed [T, H, E]
 * array, so on one device each all-to-all is a layout transform between
 *   sequence layout    [T, H, E]
 *   head-group layout  [P, T, H / P, E]  (group p = heads [p H/P, (p+1) H/P))
 * where E = head_bytes (2 D for bf16 Q/K/V/O rows, 4 for an fp32 LSE).
 *
 * cpattn_ulysses_layout -- to_head_groups = 1: sequence -> head-group layout;
 *   0: head-group -> sequence layout.  src and dst are device buffers of
 *   num_tokens * num_heads * head_bytes bytes that must not overlap, 4-byte
 *   aligned (16-byte aligned buffers with 16-byte multiples of (H / P) E use
 *   16-byte vector copies).  Requirements: num_heads % sp_size == 0,
 *   (H / P) * head_bytes a multiple of 4, num_tokens * sp_size < 2^31.
 *   Bit-exact copy; num_tokens = 0 does nothing.
 * cpattn_ulysses_seqlens -- the cu_seqlens / cp_size of the head-group layout
 *   seen as one packed batch of P * num_seqs samples with H / P heads, so that
 *   a single cpattn_fwd (total tokens P T) runs the attention of every group:
 *   cu_out[p B + b] = cu_seqlens[b] + p T, cu_out[P B] = cu_seqlens[B] +
 *   (P - 1) T; cp_out[p B + b] = cp_size[b] (1 when cp_size is NULL; cp_out
 *   may be NULL).  cu_out holds P B + 1 int32, cp_out P B; all device memory.
 * Both enqueue on `stream` and return CPATTN_ERR_INVALID_ARG for null,
 * misaligned or overlapping-by-identity pointers and out-of-range sizes before
 * launching.
 */
int cpattn_ulysses_layout(const void* src, void* dst, int64_t num_tokens,
                          int32_t num_heads, int64_t head_bytes, int32_t sp_size,
                          int32_t to_head_groups, void* stream);
int cpattn_ulysses_seqlens(const int32_t* cu_seqlens, const int32_t* cp_size,
                           int32_t num_seqs, int64_t num_tokens, int32_t sp_size,
                           int32_t* cu_out, int32_t* cp_out, void* stream);

/*
 * cpattn_fwd_noalloc -- cpattn_fwd (CPATTN_MODE_FUSED) for callers that cannot
 * allocate device memory.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot hand the library a workspace: code running inside a host program
 * whose memory pool owns the whole device budget and forbids further
 * allocations, or latency-critical code that must avoid cudaMalloc/cudaFree
 * because they can synchronise the device.  It computes exactly what
 * cpattn_fwd computes in the fused mode, but keeps its scratch (error word
 * and work list) in a fixed 1 MiB array inside the library's device image,
 * which every GPU that loads the library holds until the process exits.  It
 * allocates nothing.
 *
 * Arguments as cpattn_fwd, without mode / workspace / workspace_bytes, plus:
 *   status  device int32 [1] or NULL: receives the call's device status (the
 *           error word cpattn_poll_error would report) once the kernels have
 *           finished, in stream order.
 * Limits and behaviour:
 *   - Problems whose fused workspace (cpattn_fwd_workspace_size(T, B, H, D,
 *     max_cp, CPATTN_MODE_FUSED)) exceeds 1 MiB are rejected with
 *     CPATTN_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.  That size
 *     is about 256 + 4 (B + 1) + (8 + 16 H) (T / 256 + B max_cp + 1) bytes
 *     (each of the three parts rounded up to 256): at H = 32 some 2,000 work
 *     items, e.g. a 16,384-token batch of 7 samples at max_cp 4 uses 49 KB,
 *     while one call over more than about 510K tokens is refused.
 *   - The first call in each CUDA context (normally the device's primary
 *     context; with that device current) looks up the array's device address
 *     and caches it for that context; make that first call before any stream
 *     capture.  A context created later (e.g. after cudaDeviceReset) gets its
 *     own lookup on its first call.
 *   - Every call shares the one array and leaves its contents behind; each
 *     call clears the parts that must start at zero itself.  Calls whose
 *     kernels overlap on the GPU (for example on two streams at once) race on
 *     the array: serialise them.
 */
int cpattn_fwd_noalloc(const void* q, const void* k, const void* v,
                       const int32_t* cu_seqlens, const int32_t* cp_size,
                       int32_t num_seqs, int64_t total_tokens, int32_t max_seqlen,
                       int32_t max_cp, int32_t num_heads, int32_t head_dim,
                       float softmax_scale, int32_t causal, void* out, float* lse,
                       int32_t* status, void* stream);

/*
 * cpattn_poll_error -- synchronise `stream` and return the workspace's error
 * word (CPATTN_OK when every kernel since the last cpattn_fwd on this
 * workspace finished normally), or CPATTN_ERR_CUDA if the stream reports a
 * CUDA error.  The word is cleared by the next cpattn_fwd on the workspace.
 */
int cpattn_poll_error(const void* workspace, void* stream);

/* Human-readable name of a status code (static string). */
const char* cpattn_status_string(int status);

/* Library version, (major << 16) | (minor << 8) | patch. */
int cpattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H_ */
