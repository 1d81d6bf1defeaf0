// ss_internal.h -- host-side launchers shared between the translation units of
// libslimspec.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ss {

// Number of SMs of the current device (cached per device).
int sm_count();

// Device address of the current device's error word (cached per device).
unsigned* error_word();

// Rounds a byte count up to the 256-byte workspace granule.
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Carves consecutive 256-byte aligned regions out of a workspace.
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* p) : base(static_cast<char*>(p)) {}
  template <class T>
  T* take(size_t count) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += align256(count * sizeof(T));
    return p;
  }
};

// ------------------------------------------------------------------- head --
// Geometry of the streaming up-projection for one (dtype, r, M) request.
struct HeadPlan {
  int lpr, cpl, mt;     // lanes per row, 16-byte chunks per lane, rows of z per pass
  int sub_rows;         // vocabulary rows per partial (the recompute unit)
  int n_sub;            // ceil(V / sub_rows)
  bool ok;
};
HeadPlan head_plan(bool bf16, int r, int M, int V);

// Down-projection z = h W^T (M x r), written as fp32 to z_ws (rounded to bf16
// values when `round_bf16`), and in the input dtype to out_z when non-null.
cudaError_t launch_down_proj(bool bf16, const void* h, const void* w, int M, int d, int r,
                             bool round_bf16, float* z_ws, void* out_z, cudaStream_t st);

// Up-projection over all V rows with per-(row, sub-tile) softmax partials,
// then the per-row merge and draw.
struct HeadPartials {
  float* pmax;
  float* psum;
  int* parg;
};
cudaError_t launch_head_stream(const HeadPlan& plan, bool bf16, const void* w_up,
                               const float* z_ws, int M, int r, int V, float temperature,
                               HeadPartials part, float* out_logits, cudaStream_t st);
cudaError_t launch_head_finish(const HeadPlan& plan, bool bf16, const void* w_up,
                               const float* z_ws, int M, int r, int V, float temperature,
                               HeadPartials part, const float* uniforms, int32_t* out_tokens,
                               float* out_logprob, float* out_row_max, float* out_row_lse,
                               cudaStream_t st);

// ---------------------------------------------------------------- verify --
size_t verify_ws_bytes(int B, int gamma, int V, bool sample);
cudaError_t launch_verify(const float* target, const float* draft, const int32_t* tokens, int B,
                          int gamma, int V, float temperature, const float* uniforms,
                          int32_t* out_tokens, int32_t* out_nacc, void* ws, cudaStream_t st);

// ------------------------------------------------------------- specvocab --
size_t topk_ws_bytes(int M, int V, int k);
cudaError_t launch_topk(const float* scores, int M, int V, int k, int32_t* out_idx, void* ws,
                        cudaStream_t st);
size_t specvocab_ws_bytes(int M, int d, int d_prime, int V, int k);
cudaError_t launch_specvocab(const void* h, const void* w_down, const void* w_vocab,
                             const void* u_full, int M, int d, int d_prime, int V, int k,
                             float temperature, const float* uniforms, int32_t* out_tokens,
                             int32_t* out_idx, float* out_prob, float* out_scores, void* ws,
                             cudaStream_t st);

}  // namespace ss
