// head.cu -- SlimSpec low-rank drafter head on sm_103a CUDA cores.
//
// SlimSpec article (荷兰Nebius团队：给AI“起草员“瘦身…), section 三: the V x d head is
// replaced by W_down (d -> r) and W_up (r -> V).  The up-projection reads W_up
// (V x r, 78-145 MB at the article's model shapes) once per call and is bound
// by HBM bandwidth for a handful of rows, so it is written as a streaming
// GEMV whose per-row softmax reduction is fused into the stream:
//
//   k_down_proj    z = bf16(h W_down^T)                       (small, L2-bound)
//   k_head_stream  W_up tiles -> shared memory by cp.async.bulk (a 3-deep ring
//                  per warp), dot products on the FMA pipe with z held in
//                  registers, reduce-scatter across lanes, and an online
//                  (max, sum of exp, argmax) state per row of z.  One partial
//                  per (row of z, 32-row vocabulary tile) is written; logits
//                  never leave the chip.
//   k_head_finish  per row: merge of the tile partials in a fixed order; greedy
//                  takes the argmax, sampling locates the tile where the
//                  inverse CDF crosses u * W, recomputes that tile's logits
//                  bit-identically and walks it.
#include <algorithm>

#include "ss_common.cuh"
#include "ss_internal.h"

namespace ss {

// ----------------------------------------------------------- geometry -------
// kBF16: element type of W_up / z storage; LPR lanes share one row; each lane
// holds CPL 16-byte chunks of the row; MT rows of z are processed per launch.
template <bool kBF16, int LPR_, int CPL_, int MT_>
struct Gemv {
  static constexpr bool BF16 = kBF16;
  static constexpr int LPR = LPR_, CPL = CPL_, MT = MT_;
  static constexpr int E = kBF16 ? 8 : 4;           // elements per 16-byte chunk
  static constexpr int EB = kBF16 ? 2 : 4;          // bytes per element
  static constexpr int R = (MT == 8 || CPL >= 3) ? 4 : 8;  // rows per lane group per pass
  static constexpr int GROUPS = 32 / LPR;           // lane groups per warp
  static constexpr int PASS_ROWS = R * GROUPS;
  static constexpr int MAX_ROW_BYTES = LPR * CPL * 16;
  static constexpr int STAGE_RAW = 8192 / MAX_ROW_BYTES;
  static constexpr int STAGE_ROWS =
      STAGE_RAW < PASS_ROWS ? PASS_ROWS : (STAGE_RAW / PASS_ROWS) * PASS_ROWS;
  static constexpr int SUB_ROWS =
      STAGE_ROWS >= 32 ? STAGE_ROWS : ((32 + STAGE_ROWS - 1) / STAGE_ROWS) * STAGE_ROWS;
  static constexpr int SPS = SUB_ROWS / STAGE_ROWS;  // stages per sub-tile
  static constexpr int STAGE_BYTES = STAGE_ROWS * MAX_ROW_BYTES;
  static constexpr int N = R * MT;                  // values per lane before the reduction
  static constexpr int NF = N >= LPR ? N / LPR : 1; // values per lane after it
  static constexpr int S = ilog2(N / NF);           // scatter steps
  static constexpr int LG = ilog2(LPR);
  static constexpr int DUP_BITS = LG - S;           // lanes differing only here hold equal sums
  static constexpr int LMT = ilog2(MT), LNF = ilog2(NF);
  static constexpr int MERGE_LO = DUP_BITS + (LMT > LNF ? LMT - LNF : 0);
  static constexpr int WARPS = 8;
  static constexpr int NST = 3;                     // ring depth per warp
  static constexpr int SMEM = WARPS * NST * STAGE_BYTES + WARPS * NST * 8;
  static_assert(LNF <= LMT, "reduced values of one lane must belong to distinct rows of z");
  static_assert(SUB_ROWS % PASS_ROWS == 0 && STAGE_ROWS % PASS_ROWS == 0, "pass alignment");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// ------------------------------------------------------------- loads --------
__device__ __forceinline__ uint4 lds16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 ldg16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

template <bool kBF16>
__device__ __forceinline__ void unpack16(const uint4 w, float* f) {
  if constexpr (kBF16) {
    f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
    f[4] = bf16lo(w.z); f[5] = bf16hi(w.z); f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
  } else {
    f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y);
    f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
  }
}

// z rows m0 .. m0+MT-1, the lane's chunks, as fp32 registers (0 outside).
template <class G>
__device__ __forceinline__ void load_z(float (&zr)[G::MT][G::CPL][G::E], const float* z, int M,
                                       int m0, int r, int li) {
  const int nch = r / G::E;
#pragma unroll
  for (int m = 0; m < G::MT; ++m)
#pragma unroll
    for (int c = 0; c < G::CPL; ++c) {
      const int ch = li + c * G::LPR;
      const bool ok = (m0 + m < M) && (ch < nch);
#pragma unroll
      for (int e = 0; e < G::E; ++e)
        zr[m][c][e] = ok ? z[(size_t)(m0 + m) * r + ch * G::E + e] : 0.f;
    }
}

// Dot products of the PASS_ROWS rows of one pass with the MT rows of z,
// reduced across each lane group.  Row i of the pass starts at byte offset
// i * row_bytes from `base`; rows at or beyond `nvalid` contribute zeros.
// The arithmetic (explicit fmaf / fadd in a fixed order) is the same wherever
// it is inlined, so the stream and the recompute produce identical bits.
template <class G, bool kShared>
__device__ __forceinline__ void pass_dots(const uint8_t* gbase, uint32_t sbase, int row_bytes,
                                          int nvalid, int nch,
                                          const float (&zr)[G::MT][G::CPL][G::E],
                                          float (&v)[G::N], int lane) {
  const int g = lane / G::LPR, li = lane % G::LPR;
  float acc[G::R][G::MT];
#pragma unroll
  for (int rho = 0; rho < G::R; ++rho)
#pragma unroll
    for (int m = 0; m < G::MT; ++m) acc[rho][m] = 0.f;
#pragma unroll
  for (int rho = 0; rho < G::R; ++rho) {
    const int row = rho * G::GROUPS + g;
    if (row < nvalid) {
#pragma unroll
      for (int c = 0; c < G::CPL; ++c) {
        const int ch = li + c * G::LPR;
        if (ch < nch) {
          const int off = row * row_bytes + ch * 16;
          const uint4 w = kShared ? lds16(sbase + off) : ldg16(gbase + off);
          float wf[G::E];
          unpack16<G::BF16>(w, wf);
#pragma unroll
          for (int e = 0; e < G::E; ++e)
#pragma unroll
            for (int m = 0; m < G::MT; ++m)
              acc[rho][m] = __fmaf_rn(wf[e], zr[m][c][e], acc[rho][m]);
        }
      }
    }
  }
#pragma unroll
  for (int rho = 0; rho < G::R; ++rho)
#pragma unroll
    for (int m = 0; m < G::MT; ++m) v[rho * G::MT + m] = acc[rho][m];
  ReduceScatter<G::N, G::LPR / 2>::run(v, lane);
}

// Index (row of the pass, row of z) held in reduced slot j of a lane.
template <class G>
__device__ __forceinline__ void slot_of(int lane, int j, int& row_in_pass, int& m) {
  const int li = lane % G::LPR, g = lane / G::LPR;
  const int idx = ((li >> G::DUP_BITS) << G::LNF) + j;
  m = idx % G::MT;
  row_in_pass = (idx / G::MT) * G::GROUPS + g;
}

// --------------------------------------------------------- down-projection --
// CTA: JT=4 output columns x MT=8 rows of h; its 8 warps split the d axis.
template <bool kBF16>
__global__ void __launch_bounds__(256) k_down_proj(const uint8_t* __restrict__ h,
                                                   const uint8_t* __restrict__ w, int M, int d,
                                                   int r, int round, float* __restrict__ z_ws,
                                                   uint8_t* __restrict__ out_z) {
  constexpr int E = kBF16 ? 8 : 4, EB = kBF16 ? 2 : 4, JT = 4, MT = 8;
  const int j0 = blockIdx.x * JT, m0 = blockIdx.y * MT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch = d / E;
  const size_t rowb = (size_t)d * EB;
  float acc[JT][MT];
#pragma unroll
  for (int a = 0; a < JT; ++a)
#pragma unroll
    for (int b = 0; b < MT; ++b) acc[a][b] = 0.f;
  for (int q = lane + 32 * warp; q < nch; q += 256) {
    float wf[JT][E];
#pragma unroll
    for (int a = 0; a < JT; ++a) {
      if (j0 + a < r) {
        unpack16<kBF16>(ldg16(w + (size_t)(j0 + a) * rowb + q * 16), wf[a]);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) wf[a][e] = 0.f;
      }
    }
#pragma unroll
    for (int b = 0; b < MT; ++b) {
      if (m0 + b < M) {
        float hf[E];
        unpack16<kBF16>(ldg16(h + (size_t)(m0 + b) * rowb + q * 16), hf);
#pragma unroll
        for (int a = 0; a < JT; ++a)
#pragma unroll
          for (int e = 0; e < E; ++e) acc[a][b] = __fmaf_rn(wf[a][e], hf[e], acc[a][b]);
      }
    }
  }
  float v[32];
#pragma unroll
  for (int a = 0; a < JT; ++a)
#pragma unroll
    for (int b = 0; b < MT; ++b) v[a * MT + b] = acc[a][b];
  ReduceScatter<32, 16>::run(v, lane);  // lane l now holds entry l = (a, b) = (l/8, l%8)
  __shared__ float red[8][32];
  red[warp][lane] = v[0];
  __syncthreads();
  if (warp == 0) {
    float s = red[0][lane];
#pragma unroll
    for (int k = 1; k < 8; ++k) s = __fadd_rn(s, red[k][lane]);
    const int j = j0 + lane / MT, m = m0 + lane % MT;
    if (j < r && m < M) {
      const float zv = round ? round_bf16(s) : s;
      z_ws[(size_t)m * r + j] = zv;
      if (out_z) {
        if (kBF16)
          reinterpret_cast<uint16_t*>(out_z)[(size_t)m * r + j] = f32_to_bf16_bits(zv);
        else
          reinterpret_cast<float*>(out_z)[(size_t)m * r + j] = zv;
      }
    }
  }
}

// ----------------------------------------------------------- stream (K2) ----
// Grid: G CTAs (at most one per SM).  Vocabulary sub-tiles t = 0 .. n_sub-1
// of SUB_ROWS rows go round-robin to CTAs (t = cta + j*G) and the CTA's j-th
// tile to warp j % WARPS.  Each warp runs its own cp.async.bulk ring and never
// synchronises with other warps.
template <class G, bool kSample>
__global__ void __launch_bounds__(256, 1)
    k_head_stream(const uint8_t* __restrict__ w, const float* __restrict__ z, int M, int m0,
                  int r, int V, float c, int n_sub, float* __restrict__ pmax,
                  float* __restrict__ psum, int* __restrict__ parg,
                  float* __restrict__ out_logits, unsigned* err) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grid = gridDim.x, cta = blockIdx.x;
  const int first = cta + warp * grid;
  if (first >= n_sub) return;
  const int stride = G::WARPS * grid;
  const int n_tiles = (n_sub - 1 - first) / stride + 1;
  const int n_stages = n_tiles * G::SPS;
  uint8_t* ring = smem + warp * G::NST * G::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G::WARPS * G::NST * G::STAGE_BYTES) +
                   warp * G::NST;
  const int row_bytes = r * G::EB;
  const int nch = r / G::E;

  auto stage_rows = [&](int s, int& row0) -> int {
    const int t = first + (s / G::SPS) * stride;
    row0 = t * G::SUB_ROWS + (s % G::SPS) * G::STAGE_ROWS;
    const int n = V - row0;
    return n <= 0 ? 0 : (n < G::STAGE_ROWS ? n : G::STAGE_ROWS);
  };
  auto issue = [&](int s) {
    int row0;
    const int n = stage_rows(s, row0);
    if (n > 0) {
      const uint32_t bytes = (uint32_t)(n * row_bytes);
      uint64_t* b = &bars[s % G::NST];
      mbar_arrive_expect_tx(b, bytes);
      bulk_g2s(ring + (s % G::NST) * G::STAGE_BYTES, w + (size_t)row0 * row_bytes, bytes, b);
    }
  };

  if (lane == 0) {
    for (int s = 0; s < G::NST; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (lane == 0)
    for (int s = 0; s < G::NST && s < n_stages; ++s) issue(s);

  float zr[G::MT][G::CPL][G::E];
  load_z<G>(zr, z, M, m0, r, lane % G::LPR);
  RowState st[G::NF];
#pragma unroll
  for (int j = 0; j < G::NF; ++j) st[j] = row_state_empty();
  const bool dup_leader = (lane & ((1 << G::DUP_BITS) - 1)) == 0;

  int s = 0;
  for (; s < n_stages; ++s) {
    int row0;
    const int n = stage_rows(s, row0);
    if (n > 0) {
      const bool ok = mbar_wait_bounded(&bars[s % G::NST], (s / G::NST) & 1, err);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      const uint32_t sb = smem_u32(ring + (s % G::NST) * G::STAGE_BYTES);
      for (int p = 0; p < n; p += G::PASS_ROWS) {
        float v[G::N];
        pass_dots<G, true>(nullptr, sb + p * row_bytes, row_bytes, n - p, nch, zr, v, lane);
#pragma unroll
        for (int j = 0; j < G::NF; ++j) {
          int rip, m;
          slot_of<G>(lane, j, rip, m);
          const int row = p + rip;
          if (row < n) {
            row_state_push<kSample>(st[j], v[j], row0 + row, c);
            if (out_logits != nullptr && dup_leader && m0 + m < M)
              out_logits[(size_t)(m0 + m) * V + row0 + row] = v[j];
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0 && s + G::NST < n_stages) {
      fence_proxy_async_smem();
      issue(s + G::NST);
    }
    if (s % G::SPS == G::SPS - 1) {
      const int t = first + (s / G::SPS) * stride;
#pragma unroll
      for (int j = 0; j < G::NF; ++j) {
#pragma unroll
        for (int b = G::MERGE_LO; b < 5; ++b) st[j] = shfl_merge<kSample>(st[j], 1 << b, c);
      }
      if ((lane >> G::MERGE_LO) == 0 && dup_leader) {
#pragma unroll
        for (int j = 0; j < G::NF; ++j) {
          int rip, m;
          slot_of<G>(lane, j, rip, m);
          if (m0 + m < M) {
            const size_t o = (size_t)(m0 + m) * n_sub + t;
            pmax[o] = st[j].mx;
            parg[o] = st[j].arg;
            if (kSample) psum[o] = st[j].sum;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < G::NF; ++j) st[j] = row_state_empty();
    }
  }
  if (s < n_stages && lane == 0) {
    // A wait ran out: drain (bounded) the copies still in flight into this
    // warp's ring before the CTA's shared memory is released.
    for (int k = s; k < n_stages && k < s + G::NST; ++k) {
      int row0;
      if (stage_rows(k, row0) > 0) mbar_wait_bounded(&bars[k % G::NST], (k / G::NST) & 1, err);
    }
  }
}

// ----------------------------------------------------------- finish (K4) ----
template <class G, bool kSample>
__global__ void __launch_bounds__(256)
    k_head_finish(const uint8_t* __restrict__ w, const float* __restrict__ z, int M, int r, int V,
                  float c, float inv_t, int n_sub, const float* __restrict__ pmax,
                  const float* __restrict__ psum, const int* __restrict__ parg,
                  const float* __restrict__ uniforms, int32_t* __restrict__ out_tokens,
                  float* __restrict__ out_logprob, float* __restrict__ out_row_max,
                  float* __restrict__ out_row_lse) {
  constexpr int NT = 256;
  const int m = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* pm = pmax + (size_t)m * n_sub;
  const int* pa = parg + (size_t)m * n_sub;
  __shared__ float s_f[8];
  __shared__ int s_i[8];
  __shared__ float s_bcast[4];
  __shared__ int s_ibcast[4];
  __shared__ float s_logit[G::SUB_ROWS];

  // 1. maximum and its lowest index
  RowState st = row_state_empty();
  for (int t = tid; t < n_sub; t += NT) {
    RowState o{pm[t], 0.f, pa[t]};
    st = row_state_merge<false>(st, o, c);
  }
#pragma unroll
  for (int b = 0; b < 5; ++b) st = shfl_merge<false>(st, 1 << b, c);
  if (lane == 0) { s_f[warp] = st.mx; s_i[warp] = st.arg; }
  __syncthreads();
  if (tid == 0) {
    RowState a{s_f[0], 0.f, s_i[0]};
    for (int k = 1; k < 8; ++k) a = row_state_merge<false>(a, RowState{s_f[k], 0.f, s_i[k]}, c);
    s_bcast[0] = a.mx;
    s_ibcast[0] = a.arg;
  }
  __syncthreads();
  const float gmax = s_bcast[0];
  const int garg = s_ibcast[0];
  if (!kSample) {
    if (tid == 0) {
      out_tokens[m] = garg;
      if (out_logprob) out_logprob[m] = 0.f;
      if (out_row_max) out_row_max[m] = gmax;
      if (out_row_lse) out_row_lse[m] = gmax;
    }
    return;
  }

  // 2. tile masses relative to the row maximum, contiguous segments per thread
  const float* ps = psum + (size_t)m * n_sub;
  const int seg = (n_sub + NT - 1) / NT;
  const int t0 = min(n_sub, tid * seg), t1 = min(n_sub, t0 + seg);
  float my = 0.f;
  for (int t = t0; t < t1; ++t) my = __fadd_rn(my, ps[t] * fast_exp2((pm[t] - gmax) * c));
  // exclusive scan over threads (fixed order)
  float incl = my;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl = __fadd_rn(y, incl);
  }
  __shared__ float s_wsum[8];
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    float run = 0.f;
    for (int k = 0; k < 8; ++k) {
      const float x = s_wsum[k];
      s_wsum[k] = run;
      run = __fadd_rn(run, x);
    }
    s_bcast[1] = run;  // W
  }
  __syncthreads();
  float ex_w = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
  if (lane == 0) ex_w = 0.f;
  const float incl_blk = __fadd_rn(s_wsum[warp], incl);
  const float excl = __fadd_rn(s_wsum[warp], ex_w);  // prefix before this thread
  const float W = s_bcast[1];
  const float target = uniforms[m] * W;

  // 3. first thread whose running total passes the target
  if (tid == 0) { s_ibcast[1] = NT; s_ibcast[3] = 0; s_bcast[2] = 0.f; }
  __syncthreads();
  if (incl_blk > target && my > 0.f) atomicMin(&s_ibcast[1], tid);
  __syncthreads();
  int owner = s_ibcast[1];
  if (owner == NT) {  // rounding: take the last thread with positive mass
    if (tid == 0) s_ibcast[2] = -1;
    __syncthreads();
    if (my > 0.f) atomicMax(&s_ibcast[2], tid);
    __syncthreads();
    owner = s_ibcast[2];
  }
  if (tid == owner) {
    float cum = excl, before_last = excl;
    int tstar = -1, last = -1;
    for (int t = t0; t < t1; ++t) {
      const float mt = ps[t] * fast_exp2((pm[t] - gmax) * c);
      if (mt > 0.f) { last = t; before_last = cum; }
      const float nc = __fadd_rn(cum, mt);
      if (mt > 0.f && nc > target) { tstar = t; before_last = cum; break; }
      cum = nc;
    }
    if (tstar < 0) tstar = last;
    s_ibcast[3] = tstar;
    s_bcast[2] = target - before_last;  // mass still to cover inside the tile
  }
  __syncthreads();
  const int tstar = s_ibcast[3];
  const float resid = s_bcast[2];

  // 4. recompute tile tstar with the stream's arithmetic (warp 0)
  if (warp == 0) {
    const int m0 = (m / G::MT) * G::MT;
    float zr[G::MT][G::CPL][G::E];
    load_z<G>(zr, z, M, m0, r, lane % G::LPR);
    const int row_bytes = r * G::EB, nch = r / G::E;
    const int trow0 = tstar * G::SUB_ROWS;
    const int n = min(G::SUB_ROWS, V - trow0);
    const uint8_t* base = w + (size_t)trow0 * row_bytes;
    const bool dup_leader = (lane & ((1 << G::DUP_BITS) - 1)) == 0;
    for (int p = 0; p < n; p += G::PASS_ROWS) {
      float v[G::N];
      pass_dots<G, false>(base + (size_t)p * row_bytes, 0u, row_bytes, n - p, nch, zr, v, lane);
#pragma unroll
      for (int j = 0; j < G::NF; ++j) {
        int rip, mm;
        slot_of<G>(lane, j, rip, mm);
        if (dup_leader && m0 + mm == m && p + rip < n) s_logit[p + rip] = v[j];
      }
    }
    __syncwarp();
    if (lane == 0) {
      float cum = 0.f;
      int tok = -1, last = -1;
      for (int i = 0; i < n; ++i) {
        const float wv = fast_exp2((s_logit[i] - gmax) * c);
        if (wv > 0.f) last = i;
        cum = __fadd_rn(cum, wv);
        if (wv > 0.f && cum > resid) { tok = i; break; }
      }
      if (tok < 0) tok = last < 0 ? 0 : last;
      const float lW = logf(W);
      out_tokens[m] = trow0 + tok;
      if (out_logprob) out_logprob[m] = (s_logit[tok] - gmax) * inv_t - lW;
      if (out_row_max) out_row_max[m] = gmax;
      if (out_row_lse) out_row_lse[m] = gmax * inv_t + lW;
    }
  }
}

// ------------------------------------------------------------- host side ----
int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

cudaError_t launch_down_proj(bool bf16, const void* h, const void* w, int M, int d, int r,
                             bool round_bf16_z, float* z_ws, void* out_z, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  dim3 grid((r + 3) / 4, (M + 7) / 8);
  if (bf16)
    k_down_proj<true><<<grid, 256, 0, st>>>((const uint8_t*)h, (const uint8_t*)w, M, d, r,
                                            round_bf16_z ? 1 : 0, z_ws, (uint8_t*)out_z);
  else
    k_down_proj<false><<<grid, 256, 0, st>>>((const uint8_t*)h, (const uint8_t*)w, M, d, r, 0,
                                             z_ws, (uint8_t*)out_z);
  return cudaGetLastError();
}

// The geometries this build instantiates.
#define SS_HEAD_GEOMS(X)         \
  X(true, 32, 1, 1)              \
  X(true, 32, 1, 4)              \
  X(true, 32, 1, 8)              \
  X(true, 32, 2, 1)              \
  X(true, 32, 2, 4)              \
  X(true, 32, 2, 8)              \
  X(true, 32, 4, 1)              \
  X(true, 32, 4, 4)              \
  X(false, 8, 1, 1)              \
  X(false, 8, 1, 8)              \
  X(false, 32, 1, 1)             \
  X(false, 32, 1, 8)             \
  X(false, 32, 2, 1)             \
  X(false, 32, 2, 8)

HeadPlan head_plan(bool bf16, int r, int M, int V) {
  HeadPlan p{};
  p.ok = false;
  if (bf16) {
    const int nch = r / 8;
    if (nch <= 32) p.cpl = 1;
    else if (nch <= 64) p.cpl = 2;
    else if (nch <= 128) p.cpl = 4;
    else return p;
    p.lpr = 32;
    p.mt = (M <= 1) ? 1 : (M <= 4 || p.cpl == 4) ? 4 : 8;
  } else {
    const int nch = r / 4;
    if (nch <= 8) { p.lpr = 8; p.cpl = 1; }
    else if (nch <= 32) { p.lpr = 32; p.cpl = 1; }
    else if (nch <= 64) { p.lpr = 32; p.cpl = 2; }
    else return p;
    p.mt = (M <= 1) ? 1 : 8;
  }
#define SS_SUBROWS(B, L, C, T)                                     \
  if (bf16 == B && p.lpr == L && p.cpl == C && p.mt == T) {        \
    p.sub_rows = Gemv<B, L, C, T>::SUB_ROWS;                       \
    p.ok = true;                                                   \
  }
  SS_HEAD_GEOMS(SS_SUBROWS)
#undef SS_SUBROWS
  p.n_sub = p.ok ? (V + p.sub_rows - 1) / p.sub_rows : 0;
  return p;
}

template <class G, bool kSample>
static cudaError_t stream_one(const void* w_up, const float* z_ws, int M, int r, int V, float c,
                              const HeadPlan& plan, HeadPartials part, float* out_logits,
                              cudaStream_t st) {
  auto kern = k_head_stream<G, kSample>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
  if (e != cudaSuccess) return e;
  const int grid = std::min(plan.n_sub, sm_count());
  for (int m0 = 0; m0 < M; m0 += G::MT) {
    kern<<<grid, 32 * G::WARPS, G::SMEM, st>>>((const uint8_t*)w_up, z_ws, M, m0, r, V, c,
                                               plan.n_sub, part.pmax, part.psum, part.parg,
                                               out_logits, error_word());
  }
  return cudaGetLastError();
}

template <class G, bool kSample>
static cudaError_t finish_one(const void* w_up, const float* z_ws, int M, int r, int V, float c,
                              float inv_t, const HeadPlan& plan, HeadPartials part,
                              const float* uniforms, int32_t* out_tokens, float* out_logprob,
                              float* out_row_max, float* out_row_lse, cudaStream_t st) {
  k_head_finish<G, kSample><<<M, 256, 0, st>>>((const uint8_t*)w_up, z_ws, M, r, V, c, inv_t,
                                               plan.n_sub, part.pmax, part.psum, part.parg,
                                               uniforms, out_tokens, out_logprob, out_row_max,
                                               out_row_lse);
  return cudaGetLastError();
}

cudaError_t launch_head_stream(const HeadPlan& plan, bool bf16, const void* w_up,
                               const float* z_ws, int M, int r, int V, float temperature,
                               HeadPartials part, float* out_logits, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  const bool sample = temperature > 0.f;
  const float c = sample ? (float)(1.4426950408889634 / (double)temperature) : 0.f;
#define SS_STREAM(B, L, C, T)                                                                \
  if (bf16 == B && plan.lpr == L && plan.cpl == C && plan.mt == T)                           \
    return sample ? stream_one<Gemv<B, L, C, T>, true>(w_up, z_ws, M, r, V, c, plan, part,   \
                                                       out_logits, st)                       \
                  : stream_one<Gemv<B, L, C, T>, false>(w_up, z_ws, M, r, V, c, plan, part,  \
                                                        out_logits, st);
  SS_HEAD_GEOMS(SS_STREAM)
#undef SS_STREAM
  return cudaErrorInvalidConfiguration;
}

cudaError_t launch_head_finish(const HeadPlan& plan, bool bf16, const void* w_up,
                               const float* z_ws, int M, int r, int V, float temperature,
                               HeadPartials part, const float* uniforms, int32_t* out_tokens,
                               float* out_logprob, float* out_row_max, float* out_row_lse,
                               cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  const bool sample = temperature > 0.f;
  const double inv = sample ? 1.0 / (double)temperature : 0.0;
  const float c = (float)(1.4426950408889634 * inv), inv_t = (float)inv;
#define SS_FINISH(B, L, C, T)                                                                 \
  if (bf16 == B && plan.lpr == L && plan.cpl == C && plan.mt == T)                            \
    return sample ? finish_one<Gemv<B, L, C, T>, true>(w_up, z_ws, M, r, V, c, inv_t, plan,   \
                                                       part, uniforms, out_tokens,            \
                                                       out_logprob, out_row_max, out_row_lse, \
                                                       st)                                    \
                  : finish_one<Gemv<B, L, C, T>, false>(w_up, z_ws, M, r, V, c, inv_t, plan,  \
                                                        part, uniforms, out_tokens,           \
                                                        out_logprob, out_row_max,             \
                                                        out_row_lse, st);
  SS_HEAD_GEOMS(SS_FINISH)
#undef SS_FINISH
  return cudaErrorInvalidConfiguration;
}

}  // namespace ss
