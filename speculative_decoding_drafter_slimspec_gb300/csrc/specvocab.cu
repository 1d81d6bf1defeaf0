// specvocab.cu -- SpecVocab-style dynamic-vocabulary head on sm_103a.
//
// SpecVocab write-up (动态词汇推测加速大语言模型推理), sections 2.2.1-2.2.3:
//   h' = bf16(W_down h)        (k_down_proj, shared with the low-rank head)
//   s  = W_vocab h'            (the head's streaming GEMV, scores written out)
//   K  = topk(s, k)            k_topk: radix select on order-preserving keys,
//                              ties to the lowest id, ordered compaction
//   z' = U[K] h                k_gather_logits: a warp per candidate row of U
//                              (8 KB at d = 4096) with h held in registers;
//                              CTAs of one candidate range across all rows of
//                              h run together so rows picked by several
//                              sequences are served from L2
//   q  = softmax(z'/T), draw   k_cand_finish: per row, fixed-order scan
// The write-up's own kernel (one thread block per candidate, section 2.3) is
// prior art; here a warp handles a candidate and 64 candidates share a CTA.
#include <algorithm>

#include "ss_common.cuh"
#include "ss_internal.h"

namespace ss {

// ------------------------------------------------------------- block scan --
// Inclusive scan of one int per thread over a 1024-thread block (fixed order).
__device__ __forceinline__ int block_scan_incl_1024(int x, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const int add = warp > 0 ? s_warp[warp - 1] : 0;
  __syncthreads();
  return x + add;
}

// ------------------------------------------------------------------- top-k --
// One CTA of 1024 threads per row.  Three histogram passes over the keys
// (digits of 11, 11 and 10 bits, most significant first) find the key T* of
// the k-th largest score and how many of the keys equal to T* are kept; an
// ordered compaction then writes the kept ids in ascending order.
__global__ void __launch_bounds__(1024) k_topk(const float* __restrict__ scores, int V, int k,
                                               int32_t* __restrict__ out_idx) {
  const int row = blockIdx.x, tid = threadIdx.x;
  const float* s = scores + (size_t)row * V;
  __shared__ int hist[2048];
  __shared__ int s_warp[32];
  __shared__ int s_bin, s_above;
  uint32_t prefix = 0, pmask = 0;
  int need = k;
  if (tid == 0) { s_bin = 0; s_above = 0; }
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int nb = pass < 2 ? 2048 : 1024;
    const int shift = pass == 0 ? 21 : pass == 1 ? 10 : 0;
    for (int i = tid; i < 2048; i += 1024) hist[i] = 0;
    __syncthreads();
    for (int v = tid; v < V; v += 1024) {
      const uint32_t key = float_key(s[v]);
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1);
    }
    __syncthreads();
    // thread t owns bins nb-1-t*bpt-i (i < bpt): descending bin order
    const int bpt = nb / 1024;
    int local = 0;
    for (int i = 0; i < bpt; ++i) local += hist[nb - 1 - tid * bpt - i];
    const int incl = block_scan_incl_1024(local, s_warp);
    const int excl = incl - local;
    if (excl < need && incl >= need) {
      int cum = excl;
      for (int i = 0; i < bpt; ++i) {
        const int bin = nb - 1 - tid * bpt - i;
        if (cum + hist[bin] >= need) {
          s_bin = bin;
          s_above = cum;
          break;
        }
        cum += hist[bin];
      }
    }
    __syncthreads();
    need -= s_above;
    prefix |= (uint32_t)s_bin << shift;
    pmask |= (uint32_t)(nb - 1) << shift;
    __syncthreads();
  }
  const uint32_t thr = prefix;  // key of the k-th largest score
  // ordered compaction over contiguous segments
  const int seg = (V + 1023) / 1024;
  const int lo = min(V, tid * seg), hi = min(V, lo + seg);
  int gt = 0, eq = 0;
  for (int v = lo; v < hi; ++v) {
    const uint32_t key = float_key(s[v]);
    gt += key > thr;
    eq += key == thr;
  }
  const int gt_incl = block_scan_incl_1024(gt, s_warp);
  const int eq_incl = block_scan_incl_1024(eq, s_warp);
  int pos = (gt_incl - gt) + min(eq_incl - eq, need);
  int eq_seen = eq_incl - eq;
  int32_t* out = out_idx + (size_t)row * k;
  for (int v = lo; v < hi; ++v) {
    const uint32_t key = float_key(s[v]);
    if (key > thr) {
      if (pos < k) out[pos] = v;
      ++pos;
    } else if (key == thr) {
      if (eq_seen < need) {
        if (pos < k) out[pos] = v;
        ++pos;
      }
      ++eq_seen;
    }
  }
}

// ----------------------------------------------------------------- gather --
// blockIdx.x = row m of h, blockIdx.y = block of 64 candidates; warp w takes
// candidates 8w .. 8w+7 of the block.  h[m] lives in registers (CPL 16-byte
// chunks per lane, d <= 256 * CPL).
template <int CPL>
__global__ void __launch_bounds__(256)
    k_gather_logits(const uint8_t* __restrict__ h, const uint8_t* __restrict__ U,
                    const int32_t* __restrict__ idx, int M, int d, int k, int V,
                    float* __restrict__ cand_logits) {
  const int m = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nch = d / 8;
  const size_t rowb = (size_t)d * 2;
  float hr[CPL][8];
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    const int ch = lane + 32 * c;
    if (ch < nch) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(h + (size_t)m * rowb + ch * 16));
      hr[c][0] = bf16lo(w.x); hr[c][1] = bf16hi(w.x); hr[c][2] = bf16lo(w.y); hr[c][3] = bf16hi(w.y);
      hr[c][4] = bf16lo(w.z); hr[c][5] = bf16hi(w.z); hr[c][6] = bf16lo(w.w); hr[c][7] = bf16hi(w.w);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) hr[c][e] = 0.f;
    }
  }
  const int j0 = blockIdx.y * 64 + warp * 8;
  for (int jj = 0; jj < 8; ++jj) {
    const int j = j0 + jj;
    if (j >= k) break;
    const int v = idx[(size_t)m * k + j];
    if (v < 0 || v >= V) {  // cannot happen for a valid top-k; never read out of range
      if (lane == 0) cand_logits[(size_t)m * k + j] = kNegInf;
      continue;
    }
    const uint8_t* urow = U + (size_t)v * rowb;
    uint4 wv[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int ch = lane + 32 * c;
      wv[c] = ch < nch ? __ldg(reinterpret_cast<const uint4*>(urow + ch * 16)) : make_uint4(0, 0, 0, 0);
    }
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const uint4 w = wv[c];
      acc = __fmaf_rn(bf16lo(w.x), hr[c][0], acc);
      acc = __fmaf_rn(bf16hi(w.x), hr[c][1], acc);
      acc = __fmaf_rn(bf16lo(w.y), hr[c][2], acc);
      acc = __fmaf_rn(bf16hi(w.y), hr[c][3], acc);
      acc = __fmaf_rn(bf16lo(w.z), hr[c][4], acc);
      acc = __fmaf_rn(bf16hi(w.z), hr[c][5], acc);
      acc = __fmaf_rn(bf16lo(w.w), hr[c][6], acc);
      acc = __fmaf_rn(bf16hi(w.w), hr[c][7], acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, o));
    if (lane == 0) cand_logits[(size_t)m * k + j] = acc;
  }
}

// ----------------------------------------------------------- candidate draw --
// One CTA of 256 threads per row; candidate j in ascending id order, thread t
// owns the contiguous range [t*seg, (t+1)*seg).
__global__ void __launch_bounds__(256)
    k_cand_finish(const float* __restrict__ zc, const int32_t* __restrict__ idx, int k, float c,
                  const float* __restrict__ uniforms, int32_t* __restrict__ out_tokens,
                  int32_t* __restrict__ out_idx, float* __restrict__ out_prob) {
  constexpr int NT = 256;
  const int m = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* z = zc + (size_t)m * k;
  const int32_t* id = idx + (size_t)m * k;
  const int seg = (k + NT - 1) / NT;
  const int lo = min(k, tid * seg), hi = min(k, lo + seg);
  __shared__ float s_f[8];
  __shared__ int s_i[8];
  __shared__ float s_mx, s_W, s_resid;
  __shared__ int s_arg, s_first, s_last;

  RowState st = row_state_empty();
  for (int j = lo; j < hi; ++j) row_state_push<false>(st, z[j], j, c);
#pragma unroll
  for (int b = 0; b < 5; ++b) st = shfl_merge<false>(st, 1 << b, c);
  if (lane == 0) { s_f[warp] = st.mx; s_i[warp] = st.arg; }
  __syncthreads();
  if (tid == 0) {
    RowState a{s_f[0], 0.f, s_i[0]};
    for (int q = 1; q < 8; ++q) a = row_state_merge<false>(a, RowState{s_f[q], 0.f, s_i[q]}, c);
    s_mx = a.mx;
    s_arg = a.arg;
  }
  __syncthreads();
  const float mx = s_mx;
  if (out_idx)
    for (int j = tid; j < k; j += NT) out_idx[(size_t)m * k + j] = id[j];
  if (c == 0.f) {  // greedy
    if (tid == 0) out_tokens[m] = id[s_arg];
    if (out_prob)
      for (int j = tid; j < k; j += NT) out_prob[(size_t)m * k + j] = (j == s_arg) ? 1.f : 0.f;
    return;
  }
  float my = 0.f;
  for (int j = lo; j < hi; ++j) my = __fadd_rn(my, fast_exp2((z[j] - mx) * c));
  float incl = my;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl = __fadd_rn(y, incl);
  }
  float ex_w = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
  if (lane == 0) ex_w = 0.f;
  if (lane == 31) s_f[warp] = incl;
  if (tid == 0) { s_first = NT; s_last = -1; }
  __syncthreads();
  if (tid == 0) {
    float run = 0.f;
    for (int q = 0; q < 8; ++q) { const float x = s_f[q]; s_f[q] = run; run = __fadd_rn(run, x); }
    s_W = run;
    s_resid = uniforms[m] * run;
  }
  __syncthreads();
  const float W = s_W, target = s_resid;
  const float excl = __fadd_rn(s_f[warp], ex_w);
  const float incl_blk = __fadd_rn(s_f[warp], incl);
  if (my > 0.f) {
    atomicMax(&s_last, tid);
    if (incl_blk > target) atomicMin(&s_first, tid);
  }
  __syncthreads();
  const int owner = s_first < NT ? s_first : s_last;
  if (owner < 0 && tid == 0) out_tokens[m] = id[s_arg];
  if (tid == owner) {
    float cum = excl;
    int tok = -1, lastp = -1;
    for (int j = lo; j < hi; ++j) {
      const float wj = fast_exp2((z[j] - mx) * c);
      if (wj > 0.f) {
        lastp = j;
        cum = __fadd_rn(cum, wj);
        if (cum > target) { tok = j; break; }
      }
    }
    if (tok < 0) tok = lastp;
    out_tokens[m] = id[tok];
  }
  if (out_prob) {
    const float inv = 1.f / W;
    for (int j = tid; j < k; j += NT)
      out_prob[(size_t)m * k + j] = fast_exp2((z[j] - mx) * c) * inv;
  }
}

// -------------------------------------------------------------- host side --
size_t topk_ws_bytes(int M, int V, int k) { return 0; }

cudaError_t launch_topk(const float* scores, int M, int V, int k, int32_t* out_idx, void* ws,
                        cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  ProfScope ps(kKTopk, st);
  k_topk<<<M, 1024, 0, st>>>(scores, V, k, out_idx);
  return cudaGetLastError();
}

size_t specvocab_ws_bytes(int M, int d, int d_prime, int V, int k) {
  const HeadPlan plan = head_plan(true, d_prime, M, V);
  if (!plan.ok) return 0;
  size_t s = 0;
  s += align256((size_t)M * d_prime * 2);                  // h' (bf16)
  s += 3 * align256((size_t)M * plan.grid * sizeof(float));   // router CTA partials
  s += align256((size_t)M * V * sizeof(float));            // scores
  s += 3 * align256((size_t)M * plan.n_sub * sizeof(float));  // router partials (unused values)
  s += align256((size_t)plan.n_launch * sizeof(unsigned));    // router completion counters
  s += align256((size_t)M * sizeof(int32_t));                 // router argmax (unused)
  s += align256((size_t)M * k * sizeof(int32_t));          // candidates
  s += align256((size_t)M * k * sizeof(float));            // candidate logits
  return s;
}

cudaError_t launch_specvocab(const void* h, const void* w_down, const void* w_vocab,
                             const void* u_full, int M, int d, int d_prime, int V, int k,
                             float temperature, const float* uniforms, int32_t* out_tokens,
                             int32_t* out_idx, float* out_prob, float* out_scores, void* ws,
                             cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  const HeadPlan plan = head_plan(true, d_prime, M, V);
  Carver cv(ws);
  void* hp = cv.take<uint8_t>((size_t)M * d_prime * 2);
  float* scores = cv.take<float>((size_t)M * V);
  HeadPartials part;
  part.pmax = cv.take<float>((size_t)M * plan.n_sub);
  part.psum = cv.take<float>((size_t)M * plan.n_sub);
  part.parg = cv.take<int>((size_t)M * plan.n_sub);
  part.cmax = cv.take<float>((size_t)M * plan.grid);
  part.csum = cv.take<float>((size_t)M * plan.grid);
  part.carg = cv.take<int>((size_t)M * plan.grid);
  part.ctr = cv.take<unsigned>((size_t)plan.n_launch);
  int32_t* router_arg = cv.take<int32_t>((size_t)M);
  int32_t* cand = cv.take<int32_t>((size_t)M * k);
  float* zc = cv.take<float>((size_t)M * k);
  if (out_scores) scores = out_scores;
  const HeadOutputs router_out{nullptr, router_arg, nullptr, nullptr, nullptr};

  cudaError_t e = launch_down_proj(true, h, w_down, M, d, d_prime, true, hp, nullptr, part.ctr,
                                   plan.n_launch, st);
  if (e != cudaSuccess) return e;
  e = launch_head_stream(plan, true, w_vocab, hp, M, d_prime, V, 0.f, part, scores, router_out,
                         st);
  if (e != cudaSuccess) return e;
  e = launch_topk(scores, M, V, k, cand, nullptr, st);
  if (e != cudaSuccess) return e;
  const dim3 grid(M, (k + 63) / 64);
  const int cpl = (d + 255) / 256;
  {
  ProfScope ps(kKGather, st);
  if (cpl <= 4)
    k_gather_logits<4><<<grid, 256, 0, st>>>((const uint8_t*)h, (const uint8_t*)u_full, cand, M,
                                              d, k, V, zc);
  else if (cpl <= 8)
    k_gather_logits<8><<<grid, 256, 0, st>>>((const uint8_t*)h, (const uint8_t*)u_full, cand, M,
                                              d, k, V, zc);
  else
    k_gather_logits<16><<<grid, 256, 0, st>>>((const uint8_t*)h, (const uint8_t*)u_full, cand,
                                               M, d, k, V, zc);
  }
  const float c = temperature > 0.f ? (float)(1.4426950408889634 / (double)temperature) : 0.f;
  ProfScope ps(kKCandFinish, st);
  k_cand_finish<<<M, 256, 0, st>>>(zc, cand, k, c, uniforms, out_tokens, out_idx, out_prob);
  return cudaGetLastError();
}

}  // namespace ss
