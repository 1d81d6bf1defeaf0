/*
 * slimspec.h -- C ABI of the GB300 (sm_103a) drafter-head and verifier library.
 *
 * Sources named below (article title, section):
 *   [SlimSpec]  荷兰Nebius团队：给AI“起草员“瘦身，大模型推理速度提升5倍 (mhpn.cn)
 *   [SpecVocab] 动态词汇推测加速大语言模型推理 (2kiu.com)
 *   [Explainer] 大模型批改 5 个词，和自己写 1 个词一样快：投机解码讲人话 (liuchunshan.com)
 *   [SpecTr-GBV] SpecTr-GBV: Multi-Draft Block Verification (hypresin.com)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  * Every tensor pointer is DEVICE memory owned by the caller; row-major,
 *    contiguous, 16-byte aligned.  The library never allocates or frees
 *    memory and never synchronises the stream inside a forward call.
 *  * Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *    A call returns SS_OK once its kernels are enqueued.  Argument errors are
 *    detected on the host before anything is launched and nothing is written.
 *    A failed launch returns SS_ERR_CUDA.
 *  * `workspace` is caller-owned device scratch of at least the size the
 *    matching *_workspace_size() reports (256-byte aligned).  Its contents on
 *    entry do not matter; two calls in flight at once need two workspaces.
 *  * Sampling draws take one uniform in [0, 1) each.  A call that samples
 *    (temperature > 0) takes `seed`, `offset` and a nullable `uniforms`:
 *    with `uniforms` NULL, draw (row, slot) uses the Philox4x32-10 stream
 *    (Salmon, Moraes, Dror & Shaw, "Parallel Random Numbers: As Easy as 1, 2,
 *    3", SC'11) at key = (seed mod 2^32, seed >> 32) and counter = (row, slot,
 *    offset mod 2^32, offset >> 32), u = (first output word >> 8) * 2^-24;
 *    with `uniforms` given, it uses uniforms[row * slots + slot] instead (a
 *    hook for exact tests).  Each call names its rows and slots.  Advance
 *    `offset` between calls so that no two calls share a counter.
 *    Temperature 0 means greedy: nothing is drawn.
 *  * Ties in every argmax, top-k and inverse-CDF go to the lowest vocabulary
 *    index.  Results are deterministic: the same inputs give the same bits.
 *  * Device-side anomalies (a draft token outside [0, V), a bounded wait that
 *    ran out) are recorded in a per-device error word; ss_get_device_error()
 *    reads and clears it.
 */
#ifndef SLIMSPEC_H_
#define SLIMSPEC_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SS_OK = 0,
  SS_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad size or value   */
  SS_ERR_UNSUPPORTED = 2,   /* valid request the library has no kernel for   */
  SS_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or too small     */
  SS_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed    */
  SS_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out             */
  SS_ERR_DEVICE_INDEX = 6   /* a device-side index input was out of range     */
} ss_status;

typedef enum { SS_F32 = 0, SS_BF16 = 1 } ss_dtype;

/* Human-readable name of a status code; never NULL. */
const char* ss_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int ss_version(void);

/* ------------------------------------------------------------------------ *
 * The Philox4x32-10 stream on the device (the paper above, section 4).
 *
 * ss_philox_uniforms: out[row * slots + slot] = the uniform the sampling
 *   calls draw at (seed, offset, row, slot) when given no uniforms; rows,
 *   slots >= 0 with rows * slots < 2^31 (else SS_ERR_UNSUPPORTED); out is
 *   rows x slots float32.
 * ss_philox4x32_10: raw blocks; blocks is n x 6 uint32 (counter words c0..c3,
 *   key words k0, k1), out is n x 4 uint32 (the ten-round output words).
 * Both asynchronous on `stream`; SS_ERR_INVALID_ARG on a null or unaligned
 * pointer or a negative size.
 * ------------------------------------------------------------------------ */
int ss_philox_uniforms(uint64_t seed, uint64_t offset, int rows, int slots, float* out,
                       cudaStream_t stream);
int ss_philox4x32_10(const uint32_t* blocks, int n, uint32_t* out, cudaStream_t stream);

/* Reads and clears the device error word of the current device after
 * synchronising `stream`.  Returns SS_OK, SS_ERR_TIMEOUT, SS_ERR_DEVICE_INDEX
 * or SS_ERR_CUDA. */
int ss_get_device_error(cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Failure detection (the articles have no counterpart).  Every wait of a
 * kernel on its own pipeline (a TMA stage, an MMA accumulator, a tile id) is
 * bounded; when one runs out the kernel records SS_ERR_TIMEOUT in the error
 * word, lets what it already issued land (drain waits, always bounded at
 * 1 s), frees its tensor memory and returns, leaving the context usable.
 * ss_set_wait_limit_ns: the limit of the pipeline waits on the current
 *   device, 0 .. 10^10 ns (default 10^9).  A short limit can make a slow but
 *   healthy call fail.
 * ss_set_stall_test: with `on` non-zero, the MMA issuer of the tensor-core
 *   up-projection first waits on a barrier that nothing arrives on, so every
 *   call on the current device that runs it (bf16 low-rank heads, the trimmed
 *   head, the SpecVocab router, the low-rank verifier's recompute) times out
 *   and its outputs are undefined -- a way to test the timeout path without
 *   a fault.
 * Both synchronise the device first and apply to kernels launched after they
 * return.
 * ------------------------------------------------------------------------ */
int ss_set_wait_limit_ns(uint64_t limit_ns);
int ss_set_stall_test(int on);

/* ------------------------------------------------------------------------ *
 * SlimSpec low-rank drafter head, fused with its per-row reduction.
 *
 * [SlimSpec] section 三: W_down maps the d-wide hidden state to an r-wide
 * summary, W_up maps the summary to scores over all V vocabulary entries;
 * cost O(r*d + V*r) instead of O(V*d).  Computes, per row m:
 *   z[m]      = h[m] . W_down^T                 (fp32 accumulate; rounded to
 *                                                nearest-even bf16 when dtype
 *                                                is SS_BF16)
 *   l[m, v]   = z[m] . W_up[v]^T   for v < V    (fp32 accumulate)
 *   greedy (temperature == 0): token = lowest v attaining max_v l[m, v]
 *   sampling (temperature > 0): w_v = exp((l[m,v] - max)/T); token = smallest
 *     v whose ascending-order partial sum of w exceeds u_m * sum_v w_v, u_m
 *     the uniform of draw (row m, slot 0)
 * The M x V logits are reduced on chip and never written unless out_logits
 * is given (debug).
 *
 *  hidden      M x d      dtype         w_down  r x d   dtype
 *  w_up        V x r      dtype
 *  M >= 0 (0 is a no-op), d % 8 == 0, V >= 1, and
 *    bf16: r % 8 == 0, 8 <= r <= 1024 at any M; 1024 < r <= 4096 while the
 *          M x r rows of z fit in shared memory beside the W_up stages of
 *          the tensor-core head (M <= 40 at r = 2048, M <= 16 at r = 4096);
 *    f32:  r % 4 == 0, 4 <= r <= 256.
 *  Other shapes return SS_ERR_UNSUPPORTED (their workspace size is 0).
 *  temperature >= 0 and finite.  uniforms, when given, are M floats in
 *  [0, 1).
 *  out_tokens  M int32 (required)
 *  out_logprob M float   log softmax(l/T)[token]; 0 when greedy   (nullable)
 *  out_row_max M float   max_v l[m, v]                           (nullable)
 *  out_row_lse M float   log sum_v exp(l[m,v]/T); the max when greedy (nullable)
 *  out_z       M x r dtype, the rounded intermediate              (nullable)
 *  out_logits  M x V float32 (debug; slows the call)              (nullable)
 * ------------------------------------------------------------------------ */
size_t slimspec_head_workspace_size(int M, int d, int r, int V, int dtype);

int slimspec_head_forward(const void* hidden, const void* w_down, const void* w_up,
                          int M, int d, int r, int V, int dtype, float temperature,
                          uint64_t seed, uint64_t offset, const float* uniforms,
                          int32_t* out_tokens, float* out_logprob, float* out_row_max,
                          float* out_row_lse, void* out_z, float* out_logits, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * slimspec_head_forward without a workspace.  The articles have no
 * counterpart: this serves callers that cannot allocate device memory (a
 * runtime that fixes its device-memory budget at start-up, plugin code with
 * no device allocator, a loop that cannot afford cudaMalloc's possible
 * device-wide synchronisation).
 *
 * Same arguments, results and errors as slimspec_head_forward, minus the
 * workspace.  The scratch is a fixed array of SS_NOALLOC_SCRATCH_BYTES inside
 * the library, present on every GPU that loads it until the process exits.
 * A request whose slimspec_head_workspace_size() exceeds that returns
 * SS_ERR_WORKSPACE before anything is launched: bf16 heads fit up to M = 109
 * rows at the GPT-OSS shape (r = 360, V = 201088), 167 at the Llama shape
 * (r = 512, V = 128256) and 144 at the Qwen shape (r = 256, V = 151936);
 * slimspec_head_workspace_size() gives the bytes of any other shape.  The
 * first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it with the id of the device's current
 * context; a call that finds another context current (after a
 * cudaDeviceReset, say) looks it up again.  Make those calls outside stream
 * capture.  All calls share the array and each leaves its contents behind:
 * calls that overlap on the GPU race.  It allocates nothing.
 * ------------------------------------------------------------------------ */
#define SS_NOALLOC_SCRATCH_BYTES (4u << 20) /* 4 MiB */

int slimspec_head_forward_noalloc(const void* hidden, const void* w_down, const void* w_up,
                                  int M, int d, int r, int V, int dtype, float temperature,
                                  uint64_t seed, uint64_t offset, const float* uniforms,
                                  int32_t* out_tokens, float* out_logprob, float* out_row_max,
                                  float* out_row_lse, void* out_z, float* out_logits,
                                  cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Static trimmed head: the dense head over a fixed subset of the vocabulary.
 *
 * [SlimSpec] section 二 (FR-Spec, VocabTrim: the drafter scores only a kept
 * subset of the vocabulary).  logits = h W_kept^T over the V_kept kept rows,
 * then the per-row reduction of slimspec_head_forward over those scores; the
 * chosen kept row i is reported as the vocabulary id kept_ids[i].  Ties and
 * the inverse-CDF order follow the kept rows' order (ascending kept_ids make
 * that ascending vocabulary id); ids outside the kept set are never drafted.
 *  hidden    M x d bf16;  w_kept  V_kept x d bf16 (the kept rows of the head)
 *  kept_ids  V_kept int32 vocabulary ids (not checked)
 *  d % 8 == 0; d <= 4096; h must fit in shared memory beside the W stages
 *  (M <= 16 at d = 4096), else SS_ERR_UNSUPPORTED
 *  outputs, seed, offset and uniforms as for slimspec_head_forward (logprob
 *  and lse over the kept set).
 * ------------------------------------------------------------------------ */
size_t trimmed_head_workspace_size(int M, int d, int V_kept);

int trimmed_head_forward(const void* hidden, const void* w_kept, const int32_t* kept_ids, int M,
                         int d, int V_kept, float temperature, uint64_t seed, uint64_t offset,
                         const float* uniforms,
                         int32_t* out_tokens, float* out_logprob, float* out_row_max,
                         float* out_row_lse, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * SpecVocab-style dynamic-vocabulary drafter head (bf16 only).
 *
 * [SpecVocab] sections 2.2.1-2.2.3:
 *   h'[m] = bf16( h[m] . W_down^T )       d' = d/16 in the write-up
 *   s[m]  = h'[m] . W_vocab^T             approximate scores over all V
 *   K[m]  = the k largest s[m, v] (ties to the lowest v), ascending id order
 *   z'[m, j] = U[K[m, j]] . h[m]          exact logits of the candidates
 *   q[m]  = softmax(z'[m] / T); token = K[m, j*] with j* the greedy argmax
 *           (T == 0) or the inverse-CDF draw of row m (draw (row m, slot 0))
 *           over the candidates in ascending id order.
 *  hidden M x d, w_down d' x d, w_vocab V x d', u_full V x d (all bf16)
 *  d % 8 == 0, d' % 8 == 0, d' <= 1024, d <= 4096, 1 <= k <= min(V, 4096)
 *  out_tokens      M int32 (required)
 *  out_topk_idx    M x k int32 candidate ids, ascending            (nullable)
 *  out_topk_prob   M x k float q over the candidates (T > 0; one-hot
 *                  at the argmax when greedy)                      (nullable)
 *  out_topk_logits M x k float z', the candidates' exact logits   (nullable)
 *  out_scores      M x V float approximate scores (debug)          (nullable)
 * ------------------------------------------------------------------------ */
size_t specvocab_head_workspace_size(int M, int d, int d_prime, int V, int k);

int specvocab_head_forward(const void* hidden, const void* w_down, const void* w_vocab,
                           const void* u_full, int M, int d, int d_prime, int V, int k,
                           float temperature, uint64_t seed, uint64_t offset,
                           const float* uniforms, int32_t* out_tokens, int32_t* out_topk_idx,
                           float* out_topk_prob, float* out_topk_logits, float* out_scores,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* The top-k stage of the SpecVocab head on its own ([SpecVocab] section
 * 2.2.2): for each of M rows of V float32 scores, the k largest, ties to the
 * lowest index, written in ascending index order to out_idx (M x k int32).
 * -0.0 and +0.0 compare equal; scores must not be NaN. */
size_t ss_topk_workspace_size(int M, int V, int k);

int ss_topk_rows(const float* scores, int M, int V, int k, int32_t* out_idx,
                 void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Speculative verification of B sequences with gamma drafted tokens each.
 *
 * [Explainer] sections "小模型起草，大模型批改" and "为什么答案不会变";
 * [SpecTr-GBV] 第三步.  With p_j = softmax(target[b, j] / T) and
 * q_j = softmax(draft[b, j] / T):
 *   greedy (T == 0): a_j = lowest-index argmax of target[b, j]; n = first j
 *     with x_j != a_j (else gamma); emit x_0..x_{n-1}, a_n.
 *   sampling (T > 0): position j keeps x_j iff u[b,j] * q_j(x_j) < p_j(x_j);
 *     at the first rejection n the token is the inverse-CDF draw with
 *     u[b, gamma] from max(0, p_n - q_n) (from p_n if that is all zero); if all
 *     gamma are kept, the bonus token is drawn from p_gamma with u[b, gamma].
 *     u[b, j] is draw (row b, slot j) of gamma + 1 slots.
 *  target_logits B x (gamma+1) x V float32
 *  draft_logits  B x gamma x V float32 (may be NULL when T == 0)
 *  draft_tokens  B x gamma int32, each in [0, V) (checked on the device)
 *  uniforms      NULL (Philox at seed, offset), or B x (gamma+1) floats in
 *                [0, 1)
 *  1 <= gamma <= 32, 1 <= V <= 524288, B >= 0; SS_ERR_UNSUPPORTED when
 *    B*(gamma+1)*V >= 2^40 or B*(2*gamma+1)*ceil(V/2048) >= 2^31
 *  out_tokens    B x (gamma+1) int32: the n+1 emitted tokens, then -1
 *  out_num_accepted B int32: n
 * A position's decision needs only its own rows, so rows of positions after
 * a sequence's first rejection are not read once that rejection is known
 * (rows already in flight are still reduced; the results do not depend on
 * it).  The workspace's contents need no initialisation.
 * ------------------------------------------------------------------------ */
size_t spec_verify_workspace_size(int B, int gamma, int V, float temperature);

int spec_verify(const float* target_logits, const float* draft_logits,
                const int32_t* draft_tokens, int B, int gamma, int V,
                float temperature, uint64_t seed, uint64_t offset,
                const float* uniforms, int32_t* out_tokens,
                int32_t* out_num_accepted, void* workspace, size_t workspace_bytes,
                cudaStream_t stream);

/* The same verification on the lazy schedule of [Explainer] "小模型起草，大模型
 * 批改" (stop at the first mismatch): the rows of position j are read only for
 * the sequences that kept positions 0 .. j-1, and position j is decided before
 * position j+1 is read, so exactly the rows the accept chain needs are read
 * (one row pass and one decision launch per position).  spec_verify instead
 * decides position 0 alone first and then reads every later row of the
 * sequences that kept it, which is faster on the shapes measured here.
 * Arguments, workspace (spec_verify_workspace_size), errors and results are
 * those of spec_verify; the results are identical. */
int spec_verify_lazy(const float* target_logits, const float* draft_logits,
                     const int32_t* draft_tokens, int B, int gamma, int V,
                     float temperature, uint64_t seed, uint64_t offset,
                     const float* uniforms, int32_t* out_tokens,
                     int32_t* out_num_accepted, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Sampling verification with the draft side taken from the low-rank head.
 *
 * [SlimSpec] section 三 (the drafter's scores are z W_up^T over the whole
 * vocabulary) with [Explainer] "为什么答案不会变" (the accept test needs q(x),
 * the residual draw needs the whole q row at the first rejection).  The
 * same outcome as spec_verify with draft_logits = z W_up^T, but no draft row
 * is read or needed: position j uses log q_j(x_j) and the row's log-sum-exp
 * as the head reported them (slimspec_head_forward's out_logprob and
 * out_row_lse, same T), and the one draft row a rejection needs is
 * recomputed from its z row on the tensor cores.
 *  target_logits B x (gamma+1) x V float32
 *  z             the drafter's z rows, bf16, r wide (slimspec_head_forward's
 *                out_z): the row of sequence b, position j starts at row
 *                b * seq_stride + j * pos_stride (gamma x B head outputs:
 *                seq_stride 1, pos_stride B; B x gamma: gamma, 1)
 *  w_up          V x r bf16, the head's up-projection
 *  draft_logprob, draft_lse   float32, indexed like the rows of z
 *  draft_tokens  int32, indexed like the rows of z (checked on the device)
 *  seed, offset, uniforms as for spec_verify
 *  temperature > 0; 1 <= gamma <= 32; r % 8 == 0, r <= 512; B <= 256;
 *  V <= 524288; z, w_up and target_logits 16-byte aligned
 *  out_tokens, out_num_accepted as for spec_verify.
 * Returns SS_ERR_INVALID_ARG / SS_ERR_UNSUPPORTED / SS_ERR_WORKSPACE as
 * spec_verify does; nothing is launched then.
 * ------------------------------------------------------------------------ */
size_t spec_verify_lowrank_workspace_size(int B, int gamma, int V, int r);

int spec_verify_lowrank(const float* target_logits, const void* z, const void* w_up,
                        const float* draft_logprob, const float* draft_lse, int seq_stride,
                        int pos_stride, int r, const int32_t* draft_tokens, int B, int gamma,
                        int V, float temperature, uint64_t seed, uint64_t offset,
                        const float* uniforms, int32_t* out_tokens, int32_t* out_num_accepted,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ *
 * Instrumentation (no counterpart in the articles; used by the benchmark).
 *
 * ss_launch_count: kernels this library has launched in this process.
 * ss_profile_start / ss_profile_stop: while on, each launch is bracketed by
 *   two CUDA events recorded on its stream (host cost: two event records).
 * ss_profile_read: synchronises on the recorded events and writes, for kernel
 *   kind 0 .. n_kinds-1, the number of timed launches and their summed device
 *   time in ms; then forgets the records unless `keep` is non-zero (events
 *   captured into a CUDA graph are re-recorded by every replay, so a caller
 *   can read after each replay).  ss_profile_kind_name names a kind.
 * ------------------------------------------------------------------------ */
long long ss_launch_count(void);
int ss_profile_start(void);
int ss_profile_stop(void);
int ss_profile_read(int* launches, double* total_ms, int n_kinds, int keep);
const char* ss_profile_kind_name(int kind);

#ifdef __cplusplus
}
#endif
#endif /* SLIMSPEC_H_ */
