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

// Kernel kinds known to the optional profiler (profile.cu).
enum KernelKind {
  kKDownProj = 0, kKHeadStream, kKHeadFinish, kKVerifyRows, kKVerifyDecide, kKVerifyResid,
  kKVerifyFinish, kKTopk, kKGather, kKCandFinish, kKHeadMma, kKVerifyFirst, kKVerifyQRow,
  kKDownReduce, kKindCount
};

// Counts one launch and, while profiling is on, brackets it with two events
// recorded on `st`.  Construct immediately before the launch, destroy after.
struct ProfScope {
  int slot;
  cudaStream_t stream;
  ProfScope(int kind, cudaStream_t st);
  ~ProfScope();
};

// CTAs of `kernel` (threads per CTA, dynamic shared memory) resident per SM,
// from the occupancy calculator, cached per (kernel, device).
int resident_blocks(const void* kernel, int threads, size_t smem);

// Sets a kernel's dynamic shared memory limit and the largest shared-memory
// carveout once per (kernel, device), so that no attribute call happens while
// a stream is being captured later.
cudaError_t set_smem_once(const void* kernel, int bytes);

// Where a call's sampling draws come from: the caller's uniforms (rows x
// slots, row-major), or, when that is null, Philox4x32-10 at counter (row,
// slot, offset) under key seed (see draw_uniform in ss_common.cuh).
struct Draws {
  const float* uniforms;
  uint64_t seed, offset;
};

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
  int lpr, cpl;         // lanes per row, 16-byte chunks per lane
  int mtw, split, mt;   // rows of z per warp, warps per ring, rows of z per launch
  int sub_rows;         // vocabulary rows per partial (the recompute unit)
  int units;            // row ranges (one ring each) per CTA
  int grid;             // CTAs of the stream kernel (at most one per SM)
  int n_sub;            // partials per row of z: 8 * grid warp ranges x sub-tiles each
  int n_launch;         // ceil(M / mt) launches of the stream kernel
  bool ok;
};
HeadPlan head_plan(bool bf16, int r, int M, int V);

// Down-projection z = h W^T (M x r), written in the input dtype (rounded to
// nearest-even bf16 when `round_bf16`) to z_ws, and to out_z when non-null.
// Also zeroes the n_ctr completion counters the stream kernel uses.
cudaError_t launch_down_proj(bool bf16, const void* h, const void* w, int M, int d, int r,
                             bool round_bf16, void* z_ws, void* out_z, unsigned* ctr, int n_ctr,
                             cudaStream_t st);

// Up-projection over all V rows with per-(row, sub-tile) softmax partials;
// the last CTA of each launch merges them and draws the tokens.
struct HeadPartials {
  float* pmax;    // [M][n_sub] per vocabulary sub-tile
  float* psum;
  int* parg;
  float* cmax;    // [M][grid] per CTA
  float* csum;
  int* carg;
  unsigned* ctr;  // one completion counter per launch (zeroed by the down-projection)
};
struct HeadOutputs {
  Draws draws;    // one per row of z: (row m, slot 0)
  int32_t* tokens;
  float* logprob;
  float* row_max;
  float* row_lse;
  const int32_t* id_map;  // nullable: tokens are id_map[row of W_up] (a trimmed head)
};
cudaError_t launch_head_stream(const HeadPlan& plan, bool bf16, const void* w_up,
                               const void* z_ws, int M, int r, int V, float temperature,
                               HeadPartials part, float* out_logits, const HeadOutputs& out,
                               cudaStream_t st);

// Tensor-core up-projection (head_mma.cu) for bf16 heads.
struct MmaPlan {
  int mt;       // 128-row tiles of z (1 or 2), each taken by its own CTAs
  int kb;       // 64-wide K blocks of r
  int kps;      // K blocks per W_up stage (1 for 2-D boxes; more for wide stages)
  int wb;       // of those, full K blocks loaded by one 4-D box (wide stages)
  int nst;      // W_up stages in shared memory
  int smem;     // dynamic shared memory bytes
  int n_tiles;  // 128-row vocabulary tiles
  int grid;     // CTAs (one per SM; a multiple of mt)
  int n_sub;    // 64-row partials per row of z (2 per tile)
  bool dual;    // every CTA holds both M tiles of z (see mma_plan_dual)
  bool ok;
};
MmaPlan mma_plan(int r, int M, int V);
// The down-projection as a split-K tcgen05 GEMM (head_mma.cu), for many rows
// of h: S K slices of kbs 64-wide blocks per 128 x 128 block of z, their fp32
// partials (S x M x r, at most part_cap bytes) summed in order by a second
// kernel, which also clears n_ctr up-projection tile counters.
struct DownMmaPlan {
  int n_mt, n_nt, S, kbs, smem;
  bool ok;
};
DownMmaPlan down_mma_plan(int M, int d, int r, size_t part_cap);
cudaError_t launch_down_mma(const DownMmaPlan& plan, const void* h, const void* w_down, int M,
                            int d, int r, float* part, void* z_ws, void* out_z, unsigned* ctr,
                            int n_ctr, cudaStream_t st);

// A row of the tcgen05 up-projection's residual mode: the final draw of a
// verified sequence whose draft row is z W_up^T.  For vocabulary row v with
// target logit t_v and recomputed draft logit l_v: p(v) = 2^((t_v - pmx) c)
// * pinv and q(v) = 2^((l_v - qoff) c); the row's weights are max(0, p - q)
// (mode 0) or p (mode 1).
struct ResidRow {
  const float* trow;  // the target row of the final-draw position (V floats)
  float pmx, pinv, qoff;
  int mode;
};
// The residual mode's launch: per (row, 64-row sub-tile) the residual mass
// (rmass) and the p mass (pmass), B x n_sub each.
cudaError_t launch_head_mma_resid(const MmaPlan& plan, const void* z, const void* w_up, int B,
                                  int r, int V, float temperature, const ResidRow* rows,
                                  float* rmass, float* pmass, unsigned* ctr, cudaStream_t st);
struct MmaWork {
  float* pmax;  // [M][n_sub] sub-tile partials (sampling)
  float* psum;
  int* parg;    // [M][n_sub], unused by the head: with pmax and psum, contiguous
                // room for the down-projection's split-K slices
  // greedy (required then): per row, the largest (value key, inverted index)
  // over every CTA, zeroed with the tile counters (see k_head_mma)
  unsigned long long* best = nullptr;
};
// z_ws: M x r bf16.  With `scores` non-null the fp32 products z W_up^T are
// written there (M x V) instead of being reduced.  ctr: the launch's kMmaCtrs
// tile counters (one per M tile), zeroed by the down-projection that precedes
// it in the stream.
constexpr int kMmaCtrs = 2;
cudaError_t launch_head_mma(const MmaPlan& plan, const void* z_ws, const void* w_up, int M, int r,
                            int V, float temperature, const MmaWork& work,
                            const HeadOutputs& out, float* scores, unsigned* ctr,
                            cudaStream_t st, KernelKind kind = kKHeadMma);

// ---------------------------------------------------------------- verify --
size_t verify_ws_bytes(int B, int gamma, int V, bool sample);
// Sampling verification with the low-rank draft side (see spec_verify_lowrank).
size_t verify_lowrank_ws_bytes(int B, int gamma, int V, int r);
cudaError_t launch_verify_lowrank(const float* target, const void* z, const void* w_up,
                                  const float* logprob, const float* lse, int seq_stride,
                                  int pos_stride, int r, const int32_t* tokens, int B, int gamma,
                                  int V, float temperature, const Draws& draws,
                                  int32_t* out_tokens, int32_t* out_nacc, void* ws,
                                  cudaStream_t st);
cudaError_t launch_verify(const float* target, const float* draft, const int32_t* tokens, int B,
                          int gamma, int V, float temperature, const Draws& draws,
                          int32_t* out_tokens, int32_t* out_nacc, void* ws, cudaStream_t st,
                          bool lazy = false);

// ------------------------------------------------------------- specvocab --
size_t topk_ws_bytes(int M, int V, int k);
cudaError_t launch_topk(const float* scores, int M, int V, int k, int32_t* out_idx, void* ws,
                        cudaStream_t st);
size_t specvocab_ws_bytes(int M, int d, int d_prime, int V, int k);
cudaError_t launch_specvocab(const void* h, const void* w_down, const void* w_vocab,
                             const void* u_full, int M, int d, int d_prime, int V, int k,
                             float temperature, const Draws& draws, int32_t* out_tokens,
                             int32_t* out_idx, float* out_prob, float* out_logits,
                             float* out_scores, void* ws, cudaStream_t st);
// Philox4x32-10 on the device (the generator behind Draws with no uniforms):
// n blocks of (counter[4], key[2]) words -> out (n x 4 words); the (rows x
// slots) uniforms of one call.
cudaError_t launch_philox_blocks(const uint32_t* in, int n, uint32_t* out, cudaStream_t st);
cudaError_t launch_philox_uniforms(uint64_t seed, uint64_t offset, int rows, int slots, float* out,
                                   cudaStream_t st);

}  // namespace ss
