// api.cu -- the extern "C" boundary of libslimspec (declared in include/slimspec.h).
//
// Every entry point validates its arguments on the host before anything is
// launched (nothing is written on an argument error), carves its workspace
// and enqueues the kernels of head.cu / verify.cu / specvocab.cu on the
// caller's stream.  No entry point allocates, frees or synchronises.
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/slimspec.h"
#include "ss_common.cuh"
#include "ss_internal.h"

namespace ss {

// Per-device control block (one instance per device the library is loaded
// on): the error word, the stall test switch, the pipeline wait limit.
__device__ DeviceControl g_control = {0u, 0u, kWaitLimitNs};

unsigned* error_word() {
  static unsigned* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (cached[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_control) != cudaSuccess) return nullptr;
    cached[dev] = &static_cast<DeviceControl*>(p)->err;
  }
  return cached[dev];
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
static bool temp_ok(float t) { return isfinite(t) && t >= 0.f; }
static int cuda_status(cudaError_t e) { return e == cudaSuccess ? SS_OK : SS_ERR_CUDA; }

// bf16 heads run the up-projection on the tensor cores whenever the shape
// fits the tcgen05 kernel (r a multiple of 8 up to 4096, M up to 256), even for
// a single row of z: the MMA takes the multiply-adds off the issue slots, so
// the kernel only moves W_up.  fp32 heads, and bf16 shapes outside that range,
// stream W_up through the CUDA cores.
// From this many rows of h the down-projection runs on the tensor cores.
constexpr int kDownMmaMinM = 64;

static bool use_mma(bool bf16, int M, int r, int V) {
  return bf16 && M >= 1 && mma_plan(r, M, V).ok;
}

static size_t head_ws_bytes(int M, int r, int V, bool bf16) {
  if (use_mma(bf16, M, r, V)) {
    const MmaPlan p = mma_plan(r, M, V);
    size_t s = align256((size_t)M * r * 2);
    s += 3 * align256((size_t)M * p.n_sub * sizeof(float));
    // tile counters of the two launches, then the rows' best keys (greedy);
    // the down-projection zeroes them all
    s += align256((2 * kMmaCtrs + 2 * (size_t)M) * sizeof(unsigned));
    return s;
  }
  const HeadPlan plan = head_plan(bf16, r, M, V);
  if (!plan.ok) return 0;
  size_t s = 0;
  s += align256((size_t)M * r * (bf16 ? 2 : 4));
  s += 3 * align256((size_t)M * plan.n_sub * sizeof(float));
  s += 3 * align256((size_t)M * plan.grid * sizeof(float));
  s += align256((size_t)plan.n_launch * sizeof(unsigned));
  return s;
}

}  // namespace ss

using namespace ss;

extern "C" {

const char* ss_status_string(int status) {
  switch (status) {
    case SS_OK: return "SS_OK";
    case SS_ERR_INVALID_ARG: return "SS_ERR_INVALID_ARG: invalid argument";
    case SS_ERR_UNSUPPORTED: return "SS_ERR_UNSUPPORTED: no kernel for this shape";
    case SS_ERR_WORKSPACE: return "SS_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case SS_ERR_CUDA: return "SS_ERR_CUDA: CUDA runtime error";
    case SS_ERR_TIMEOUT: return "SS_ERR_TIMEOUT: a bounded device wait ran out";
    case SS_ERR_DEVICE_INDEX: return "SS_ERR_DEVICE_INDEX: device-side index out of range";
    default: return "unknown status";
  }
}

int ss_version(void) { return 200; }

int ss_get_device_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SS_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_control, sizeof(v), offsetof(DeviceControl, err)) != cudaSuccess)
    return SS_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_control, &zero, sizeof(zero), offsetof(DeviceControl, err)) !=
        cudaSuccess)
      return SS_ERR_CUDA;
  }
  if (v & kErrTimeout) return SS_ERR_TIMEOUT;
  if (v & kErrIndex) return SS_ERR_DEVICE_INDEX;
  return SS_OK;
}

int ss_set_wait_limit_ns(uint64_t limit_ns) {
  if (limit_ns > 10 * kWaitLimitNs) return SS_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return SS_ERR_CUDA;
  const unsigned long long v = limit_ns;
  return cuda_status(
      cudaMemcpyToSymbol(g_control, &v, sizeof(v), offsetof(DeviceControl, wait_limit_ns)));
}

int ss_set_stall_test(int on) {
  if (cudaDeviceSynchronize() != cudaSuccess) return SS_ERR_CUDA;
  const unsigned v = on ? 1u : 0u;
  return cuda_status(
      cudaMemcpyToSymbol(g_control, &v, sizeof(v), offsetof(DeviceControl, stall_head)));
}

// ------------------------------------------------------------------- head --
static int head_check(int M, int d, int r, int V, int dtype) {
  if (M < 0 || d <= 0 || r <= 0 || V <= 0) return SS_ERR_INVALID_ARG;
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_INVALID_ARG;
  const bool bf16 = dtype == SS_BF16;
  if (d % 8 != 0 || r % (bf16 ? 8 : 4) != 0) return SS_ERR_INVALID_ARG;
  if ((long long)V * r * (bf16 ? 2 : 4) >= (1LL << 40)) return SS_ERR_UNSUPPORTED;
  if (!use_mma(bf16, M, r, V) && !head_plan(bf16, r, M, V).ok) return SS_ERR_UNSUPPORTED;
  return SS_OK;
}

// ----------------------------------------------------- static trimmed head --
static size_t trimmed_ws_bytes(int M, int d, int Vk) {
  const MmaPlan p = mma_plan(d, M, Vk);
  if (!p.ok) return 0;
  size_t s = 3 * align256((size_t)M * p.n_sub * sizeof(float));  // sub-tile partials
  s += align256((kMmaCtrs + 2 * (size_t)M) * sizeof(unsigned));  // tile counters, best keys
  return s;
}

size_t trimmed_head_workspace_size(int M, int d, int V_kept) {
  if (M <= 0 || d <= 0 || d % 8 != 0 || V_kept <= 0) return 0;
  return trimmed_ws_bytes(M, d, V_kept);
}

int trimmed_head_forward(const void* hidden, const void* w_kept, const int32_t* kept_ids, int M,
                         int d, int V_kept, float temperature, uint64_t seed, uint64_t offset,
                         const float* uniforms, int32_t* out_tokens, float* out_logprob,
                         float* out_row_max, float* out_row_lse, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
  if (M < 0 || d <= 0 || d % 8 != 0 || V_kept <= 0 || !temp_ok(temperature))
    return SS_ERR_INVALID_ARG;
  if ((long long)V_kept * d * 2 >= (1LL << 40)) return SS_ERR_UNSUPPORTED;
  if (M == 0) return SS_OK;
  if (!hidden || !w_kept || !kept_ids || !out_tokens) return SS_ERR_INVALID_ARG;
  if (uniforms && !aligned(uniforms, 4)) return SS_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(w_kept, 16) || !aligned(kept_ids, 4) ||
      !aligned(out_tokens, 4) || (out_logprob && !aligned(out_logprob, 4)) ||
      (out_row_max && !aligned(out_row_max, 4)) || (out_row_lse && !aligned(out_row_lse, 4)))
    return SS_ERR_INVALID_ARG;
  const MmaPlan mp = mma_plan(d, M, V_kept);
  if (!mp.ok) return SS_ERR_UNSUPPORTED;  // h must fit in shared memory beside the W stages
  const size_t need = trimmed_ws_bytes(M, d, V_kept);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return SS_ERR_WORKSPACE;
  Carver cv(workspace);
  MmaWork wk;
  wk.pmax = cv.take<float>((size_t)M * mp.n_sub);
  wk.psum = cv.take<float>((size_t)M * mp.n_sub);
  wk.parg = cv.take<int>((size_t)M * mp.n_sub);
  const size_t n_ctr = kMmaCtrs + 2 * (size_t)M;  // counters, then M 64-bit best keys
  unsigned* ctr = cv.take<unsigned>(n_ctr);
  wk.best = reinterpret_cast<unsigned long long*>(ctr + kMmaCtrs);
  // the rows of h are the tensor-core kernel's z; its tile counters and keys start at 0
  cudaError_t e = cudaMemsetAsync(ctr, 0, n_ctr * sizeof(unsigned), stream);
  if (e != cudaSuccess) return cuda_status(e);
  const HeadOutputs outs{Draws{uniforms, seed, offset}, out_tokens, out_logprob, out_row_max,
                         out_row_lse, kept_ids};
  e = launch_head_mma(mp, hidden, w_kept, M, d, V_kept, temperature, wk, outs, nullptr, ctr,
                      stream);
  return cuda_status(e);
}

size_t slimspec_head_workspace_size(int M, int d, int r, int V, int dtype) {
  if (head_check(M, d, r, V, dtype) != SS_OK) return 0;
  return head_ws_bytes(M, r, V, dtype == SS_BF16);
}

int slimspec_head_forward(const void* hidden, const void* w_down, const void* w_up, int M, int d,
                          int r, int V, int dtype, float temperature, uint64_t seed,
                          uint64_t offset, const float* uniforms, int32_t* out_tokens,
                          float* out_logprob, float* out_row_max, float* out_row_lse, void* out_z,
                          float* out_logits, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
  int st = head_check(M, d, r, V, dtype);
  if (st != SS_OK) return st;
  if (!temp_ok(temperature)) return SS_ERR_INVALID_ARG;
  if (M == 0) return SS_OK;
  if (!hidden || !w_down || !w_up || !out_tokens) return SS_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(w_down, 16) || !aligned(w_up, 16)) return SS_ERR_INVALID_ARG;
  if (!aligned(out_tokens, 4) || (out_logprob && !aligned(out_logprob, 4)) ||
      (out_row_max && !aligned(out_row_max, 4)) || (out_row_lse && !aligned(out_row_lse, 4)) ||
      (out_z && !aligned(out_z, 4)) || (out_logits && !aligned(out_logits, 4)))
    return SS_ERR_INVALID_ARG;
  if (uniforms && !aligned(uniforms, 4)) return SS_ERR_INVALID_ARG;
  const bool bf16 = dtype == SS_BF16;
  const size_t need = head_ws_bytes(M, r, V, bf16);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return SS_ERR_WORKSPACE;

  if (use_mma(bf16, M, r, V)) {
    const MmaPlan mp = mma_plan(r, M, V);
    Carver cv(workspace);
    void* z_ws = cv.take<uint8_t>((size_t)M * r * 2);
    MmaWork wk;
    wk.pmax = cv.take<float>((size_t)M * mp.n_sub);
    wk.psum = cv.take<float>((size_t)M * mp.n_sub);
    wk.parg = cv.take<int>((size_t)M * mp.n_sub);
    const int n_ctr = 2 * kMmaCtrs + 2 * M;  // counters, then M 64-bit best keys
    unsigned* ctr = cv.take<unsigned>((size_t)n_ctr);
    wk.best = reinterpret_cast<unsigned long long*>(ctr + 2 * kMmaCtrs);
    const HeadOutputs outs{Draws{uniforms, seed, offset}, out_tokens, out_logprob, out_row_max,
                           out_row_lse};
    // many rows of h: the down-projection as a split-K tensor-core GEMM, its
    // fp32 slices in the (not yet used) partial arrays, contiguous from pmax
    const size_t part_cap = 3 * align256((size_t)M * mp.n_sub * sizeof(float));
    const DownMmaPlan dp = M >= kDownMmaMinM ? down_mma_plan(M, d, r, part_cap) : DownMmaPlan{};
    cudaError_t e =
        dp.ok ? launch_down_mma(dp, hidden, w_down, M, d, r, wk.pmax, z_ws, out_z, ctr, n_ctr,
                                stream)
              : launch_down_proj(bf16, hidden, w_down, M, d, r, true, z_ws, out_z, ctr, n_ctr,
                                 stream);
    if (e == cudaSuccess && out_logits != nullptr)
      e = launch_head_mma(mp, z_ws, w_up, M, r, V, 0.f, wk, outs, out_logits, ctr, stream);
    if (e == cudaSuccess)
      e = launch_head_mma(mp, z_ws, w_up, M, r, V, temperature, wk, outs, nullptr,
                          ctr + kMmaCtrs, stream);
    return cuda_status(e);
  }
  const HeadPlan plan = head_plan(bf16, r, M, V);
  Carver cv(workspace);
  void* z_ws = cv.take<uint8_t>((size_t)M * r * (bf16 ? 2 : 4));
  HeadPartials part;
  part.pmax = cv.take<float>((size_t)M * plan.n_sub);
  part.psum = cv.take<float>((size_t)M * plan.n_sub);
  part.parg = cv.take<int>((size_t)M * plan.n_sub);
  part.cmax = cv.take<float>((size_t)M * plan.grid);
  part.csum = cv.take<float>((size_t)M * plan.grid);
  part.carg = cv.take<int>((size_t)M * plan.grid);
  part.ctr = cv.take<unsigned>((size_t)plan.n_launch);
  const HeadOutputs outs{Draws{uniforms, seed, offset}, out_tokens, out_logprob, out_row_max,
                           out_row_lse};

  cudaError_t e = launch_down_proj(bf16, hidden, w_down, M, d, r, bf16, z_ws, out_z, part.ctr,
                                   plan.n_launch, stream);
  if (e == cudaSuccess)
    e = launch_head_stream(plan, bf16, w_up, z_ws, M, r, V, temperature, part, out_logits, outs,
                           stream);
  return cuda_status(e);
}

// -------------------------------------------------------------- specvocab --
static int sv_check(int M, int d, int d_prime, int V, int k) {
  if (M < 0 || d <= 0 || d_prime <= 0 || V <= 0) return SS_ERR_INVALID_ARG;
  if (d % 8 != 0 || d_prime % 8 != 0) return SS_ERR_INVALID_ARG;
  if (k < 1 || k > V) return SS_ERR_INVALID_ARG;
  if (d > 4096 || d_prime > 1024 || k > 4096) return SS_ERR_UNSUPPORTED;
  if ((long long)V * d * 2 >= (1LL << 40)) return SS_ERR_UNSUPPORTED;
  if (!mma_plan(d_prime, M, V).ok && !head_plan(true, d_prime, M, V).ok) return SS_ERR_UNSUPPORTED;
  return SS_OK;
}

size_t specvocab_head_workspace_size(int M, int d, int d_prime, int V, int k) {
  if (sv_check(M, d, d_prime, V, k) != SS_OK) return 0;
  return specvocab_ws_bytes(M, d, d_prime, V, k);
}

int specvocab_head_forward(const void* hidden, const void* w_down, const void* w_vocab,
                           const void* u_full, int M, int d, int d_prime, int V, int k,
                           float temperature, uint64_t seed, uint64_t offset,
                           const float* uniforms, int32_t* out_tokens, int32_t* out_topk_idx,
                           float* out_topk_prob, float* out_topk_logits, float* out_scores,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  int st = sv_check(M, d, d_prime, V, k);
  if (st != SS_OK) return st;
  if (!temp_ok(temperature)) return SS_ERR_INVALID_ARG;
  if (M == 0) return SS_OK;
  if (!hidden || !w_down || !w_vocab || !u_full || !out_tokens) return SS_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(w_down, 16) || !aligned(w_vocab, 16) || !aligned(u_full, 16))
    return SS_ERR_INVALID_ARG;
  if (!aligned(out_tokens, 4) || (out_topk_idx && !aligned(out_topk_idx, 4)) ||
      (out_topk_prob && !aligned(out_topk_prob, 4)) ||
      (out_topk_logits && !aligned(out_topk_logits, 4)) || (out_scores && !aligned(out_scores, 4)))
    return SS_ERR_INVALID_ARG;
  if (uniforms && !aligned(uniforms, 4)) return SS_ERR_INVALID_ARG;
  const size_t need = specvocab_ws_bytes(M, d, d_prime, V, k);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return SS_ERR_WORKSPACE;
  return cuda_status(launch_specvocab(hidden, w_down, w_vocab, u_full, M, d, d_prime, V, k,
                                      temperature, Draws{uniforms, seed, offset}, out_tokens,
                                      out_topk_idx, out_topk_prob, out_topk_logits, out_scores,
                                      workspace, stream));
}

size_t ss_topk_workspace_size(int M, int V, int k) {
  if (M < 0 || V <= 0 || k < 1 || k > V) return 0;
  return topk_ws_bytes(M, V, k);
}

int ss_topk_rows(const float* scores, int M, int V, int k, int32_t* out_idx, void* workspace,
                 size_t workspace_bytes, cudaStream_t stream) {
  if (M < 0 || V <= 0 || k < 1 || k > V) return SS_ERR_INVALID_ARG;
  if (M == 0) return SS_OK;
  if (!scores || !out_idx || !aligned(scores, 4) || !aligned(out_idx, 4)) return SS_ERR_INVALID_ARG;
  if (workspace_bytes < topk_ws_bytes(M, V, k)) return SS_ERR_WORKSPACE;
  return cuda_status(launch_topk(scores, M, V, k, out_idx, workspace, stream));
}

// ----------------------------------------------------------------- verify --
size_t spec_verify_workspace_size(int B, int gamma, int V, float temperature) {
  if (B < 0 || gamma < 1 || gamma > 32 || V <= 0 || !temp_ok(temperature)) return 0;
  return verify_ws_bytes(B, gamma, V, temperature > 0.f);
}

size_t spec_verify_lowrank_workspace_size(int B, int gamma, int V, int r) {
  if (B < 0 || gamma < 1 || gamma > 32 || V <= 0 || r <= 0) return 0;
  return verify_lowrank_ws_bytes(B, gamma, V, r);
}

int spec_verify_lowrank(const float* target_logits, const void* z, const void* w_up,
                        const float* draft_logprob, const float* draft_lse, int seq_stride,
                        int pos_stride, int r, const int32_t* draft_tokens, int B, int gamma,
                        int V, float temperature, uint64_t seed, uint64_t offset,
                        const float* uniforms, int32_t* out_tokens, int32_t* out_num_accepted,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (B < 0 || gamma < 1 || gamma > 32 || V <= 0 || r <= 0 || seq_stride < 0 || pos_stride < 0 ||
      !(temperature > 0.f) || !temp_ok(temperature))
    return SS_ERR_INVALID_ARG;
  if ((long long)B * (gamma + 1) * V >= (1LL << 40)) return SS_ERR_UNSUPPORTED;
  if (V > 524288) return SS_ERR_UNSUPPORTED;  // the final draw scans at most 256 chunks
  if ((long long)B * (gamma + 1) * ((V + 2047) / 2048) >= (1LL << 31)) return SS_ERR_UNSUPPORTED;
  if (B == 0) return SS_OK;
  // the recompute: B <= 256 rows; its finish holds a z row in two chunks per lane
  if (r > 512 || !mma_plan(r, B, V).ok) return SS_ERR_UNSUPPORTED;
  if (!target_logits || !z || !w_up || !draft_logprob || !draft_lse || !draft_tokens ||
      !out_tokens || !out_num_accepted)
    return SS_ERR_INVALID_ARG;
  if (!aligned(target_logits, 16) || !aligned(z, 16) || !aligned(w_up, 16) ||
      !aligned(draft_logprob, 4) || !aligned(draft_lse, 4) || !aligned(draft_tokens, 4) ||
      (uniforms && !aligned(uniforms, 4)) || !aligned(out_tokens, 4) ||
      !aligned(out_num_accepted, 4))
    return SS_ERR_INVALID_ARG;
  const size_t need = verify_lowrank_ws_bytes(B, gamma, V, r);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return SS_ERR_WORKSPACE;
  return cuda_status(launch_verify_lowrank(target_logits, z, w_up, draft_logprob, draft_lse,
                                           seq_stride, pos_stride, r, draft_tokens, B, gamma, V,
                                           temperature, Draws{uniforms, seed, offset}, out_tokens,
                                           out_num_accepted, workspace, stream));
}

// Both schedules: the split one (spec_verify) and, lazy, position by position.
static int verify_entry(const float* target_logits, const float* draft_logits,
                        const int32_t* draft_tokens, int B, int gamma, int V, float temperature,
                        uint64_t seed, uint64_t offset, const float* uniforms, int32_t* out_tokens,
                        int32_t* out_num_accepted, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream, bool lazy) {
  if (B < 0 || gamma < 1 || gamma > 32 || V <= 0 || !temp_ok(temperature))
    return SS_ERR_INVALID_ARG;
  if ((long long)B * (gamma + 1) * V >= (1LL << 40)) return SS_ERR_UNSUPPORTED;
  if (V > 524288) return SS_ERR_UNSUPPORTED;  // the final draw scans at most 256 chunks
  // the row pass numbers its (row, 2048-float chunk) units in 32 bits
  if ((long long)B * (2 * gamma + 1) * ((V + 2047) / 2048) >= (1LL << 31))
    return SS_ERR_UNSUPPORTED;
  if (B == 0) return SS_OK;
  const bool sample = temperature > 0.f;
  if (!target_logits || !draft_tokens || !out_tokens || !out_num_accepted) return SS_ERR_INVALID_ARG;
  if (sample && !draft_logits) return SS_ERR_INVALID_ARG;
  if (!aligned(target_logits, 16) || (draft_logits && !aligned(draft_logits, 16)) ||
      !aligned(draft_tokens, 4) || !aligned(out_tokens, 4) || !aligned(out_num_accepted, 4) ||
      (uniforms && !aligned(uniforms, 4)))
    return SS_ERR_INVALID_ARG;
  const size_t need = verify_ws_bytes(B, gamma, V, sample);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return SS_ERR_WORKSPACE;
  return cuda_status(launch_verify(target_logits, draft_logits, draft_tokens, B, gamma, V,
                                   temperature, Draws{uniforms, seed, offset}, out_tokens,
                                   out_num_accepted, workspace, stream, lazy));
}

int spec_verify(const float* target_logits, const float* draft_logits, const int32_t* draft_tokens,
                int B, int gamma, int V, float temperature, uint64_t seed, uint64_t offset,
                const float* uniforms, int32_t* out_tokens, int32_t* out_num_accepted,
                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return verify_entry(target_logits, draft_logits, draft_tokens, B, gamma, V, temperature, seed,
                      offset, uniforms, out_tokens, out_num_accepted, workspace, workspace_bytes,
                      stream, false);
}

int spec_verify_lazy(const float* target_logits, const float* draft_logits,
                     const int32_t* draft_tokens, int B, int gamma, int V, float temperature,
                     uint64_t seed, uint64_t offset, const float* uniforms, int32_t* out_tokens,
                     int32_t* out_num_accepted, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream) {
  return verify_entry(target_logits, draft_logits, draft_tokens, B, gamma, V, temperature, seed,
                      offset, uniforms, out_tokens, out_num_accepted, workspace, workspace_bytes,
                      stream, true);
}

// ------------------------------------------------------- Philox uniforms --
int ss_philox_uniforms(uint64_t seed, uint64_t offset, int rows, int slots, float* out,
                       cudaStream_t stream) {
  if (rows < 0 || slots < 0) return SS_ERR_INVALID_ARG;
  if ((long long)rows * slots == 0) return SS_OK;
  if ((long long)rows * slots >= (1LL << 31)) return SS_ERR_UNSUPPORTED;
  if (!out || !aligned(out, 4)) return SS_ERR_INVALID_ARG;
  return cuda_status(launch_philox_uniforms(seed, offset, rows, slots, out, stream));
}

int ss_philox4x32_10(const uint32_t* blocks, int n, uint32_t* out, cudaStream_t stream) {
  if (n < 0) return SS_ERR_INVALID_ARG;
  if (n == 0) return SS_OK;
  if (!blocks || !out || !aligned(blocks, 4) || !aligned(out, 4)) return SS_ERR_INVALID_ARG;
  return cuda_status(launch_philox_blocks(blocks, n, out, stream));
}

}  // extern "C"
