// verify.cu -- speculative verification on sm_103a.
//
// Explainer (大模型批改 5 个词…), sections "小模型起草，大模型批改" and "为什么答案不会变",
// and SpecTr-GBV article, 第三步.  The verifier reads target rows (fp32, V
// wide) and, when sampling, draft rows: an HBM streaming reduction.  A
// position's decision needs only its own rows, and no row after a sequence's
// first rejection is used, so for large inputs position 0 is decided first
// and the other positions are read only for sequences that kept it.
//
//   k_verify_rows    one warp per (row, 2048-float chunk) of the rows of a
//                    range of positions: 16-byte streaming loads, online
//                    (max, sum of exp at T, argmax) -> partials
//   k_verify_first   one CTA per sequence: position 0's accept test, between
//                    a pass over the position-0 rows and one over the rest
//   k_verify_decide  one CTA per sequence: merges the partials of its rows,
//                    greedy prefix match or the min(1, p/q) accept tests
//   k_verify_resid   one warp per (sequence, chunk) of the final draw's row:
//                    chunk masses of max(0, p_n - q_n) (bonus: of p_gamma,
//                    straight from the partials)
//   k_verify_finish  one CTA per sequence: inverse CDF over the chunk masses,
//                    then an ordered scan of the one chunk that holds the draw
//
// The low-rank draft side (SlimSpec article, section 三: q is the drafter
// head's softmax(z W_up^T / T)) reads no draft rows: the accept tests take
// log q(x) from the head, the decide kernel gathers the z row of each
// sequence's final draw, and the draw's draft row is recomputed by the
// tcgen05 up-projection (head_mma.cu) -- written out for k_verify_resid /
// k_verify_finish, or, from kFusedResidMinB sequences on, reduced in its
// epilogue to sub-tile masses of max(0, p - q) and p for
//   k_verify_lr_finish  one CTA per sequence: ordered scan of the sub-tile
//                    masses, one 64-row sub-tile recomputed on CUDA cores,
//                    an ordered walk
#include <algorithm>

#include "ss_common.cuh"
#include "ss_internal.h"

namespace ss {

constexpr int kVChunk = 2048;  // floats per partial (8 KB: one round trip of 16 B x 16 per lane)

struct VerifyInfo {
  int n;        // accepted drafted tokens
  int mode;     // 0: residual of row n, 1: target row n alone (bonus / fallback)
  float pmx, pinv, qmx, qinv;  // row maxima and reciprocal normalisers
  float pad0, pad1;
};

template <bool kSample>
__device__ __forceinline__ void push4(RowState& s, const float4 a, int v0, float c) {
  const float m01 = fmaxf(a.x, a.y), m23 = fmaxf(a.z, a.w), m4 = fmaxf(m01, m23);
  const int off = (a.x == m4) ? 0 : (a.y == m4) ? 1 : (a.z == m4) ? 2 : 3;
  if (m4 > s.mx) {
    if (kSample) s.sum = s.sum * fast_exp2((s.mx - m4) * c);
    s.mx = m4;
    s.arg = v0 + off;
  }
  if (kSample) {
    const float mx = s.mx;
    float t = fast_exp2((a.x - mx) * c);
    t = __fadd_rn(t, fast_exp2((a.y - mx) * c));
    t = __fadd_rn(t, fast_exp2((a.z - mx) * c));
    t = __fadd_rn(t, fast_exp2((a.w - mx) * c));
    s.sum = __fadd_rn(s.sum, t);
  }
}

// ------------------------------------------------------------------- K8 ----
// One warp per (row, kVChunk-float chunk) unit over the rows of positions
// j0..j1 of every sequence: its target rows, then (sampling) its draft rows
// of drafted positions.  With seq_ok given, the units of sequences whose
// seq_ok entry is 0 are skipped (their first rejection is before j0).
template <bool kSample>
__global__ void __launch_bounds__(256)
    k_verify_rows(const float* __restrict__ target, const float* __restrict__ draft, int B,
                  int gamma, int V, float c, int n_chunks, int j0, int j1,
                  const int* __restrict__ seq_ok, float* __restrict__ vmax,
                  float* __restrict__ vsum, int* __restrict__ varg) {
  pdl_launch_dependents();
  // the logit rows are inputs: read and reduced while a preceding kernel may
  // still run; the flags and the partials wait for it (below)
  if (seq_ok != nullptr) pdl_wait_producer();
  const int lane = threadIdx.x & 31;
  const unsigned gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const unsigned nw = gridDim.x * (blockDim.x >> 5);
  const bool vec = (V & 3) == 0;
  const int g1 = gamma + 1;
  const int nt = j1 - j0 + 1;                                    // target rows per sequence
  const int nd = (kSample && draft != nullptr) ? max(0, min(j1, gamma - 1) - j0 + 1) : 0;
  const unsigned seq_units = (unsigned)(nt + nd) * (unsigned)n_chunks;
  const unsigned units = (unsigned)B * seq_units;  // < 2^31: checked by the host
  for (unsigned u = gw; u < units; u += nw) {
    const int b = (int)(u / seq_units);
    if (seq_ok != nullptr && __ldg(seq_ok + b) == 0) continue;  // warp-uniform
    const unsigned rem = u - (unsigned)b * seq_units;
    const int ri = (int)(rem / (unsigned)n_chunks);
    const int ch = (int)(rem - (unsigned)ri * (unsigned)n_chunks);
    const int row = ri < nt ? b * g1 + j0 + ri : B * g1 + b * gamma + j0 + (ri - nt);
    const float* src = ri < nt ? target + (size_t)row * V
                               : draft + ((size_t)b * gamma + j0 + (ri - nt)) * V;
    const int lo = ch * kVChunk, hi = min(V, lo + kVChunk);
    RowState s = row_state_empty();
    if (vec) {
      const float4* p4 = reinterpret_cast<const float4*>(src);
      const int q0 = lo >> 2, q1 = hi >> 2;
      float4 a[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int q = q0 + lane + 32 * k;
        if (q < q1) a[k] = __ldcs(p4 + q);
      }
      if (!kSample) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int q = q0 + lane + 32 * k;
          if (q < q1) push4<false>(s, a[k], q * 4, c);
        }
      } else {
        // sampling needs no argmax: the lane's maximum, then one pass of
        // 2^(x c - max c) in four fixed-order partial sums
        float m = kNegInf;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int q = q0 + lane + 32 * k;
          if (q < q1) m = fmaxf(m, fmaxf(fmaxf(a[k].x, a[k].y), fmaxf(a[k].z, a[k].w)));
        }
        if (m != kNegInf) {
          const float off = -m * c;
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int q = q0 + lane + 32 * k;
            if (q < q1) {
              s0 = __fadd_rn(s0, fast_exp2(__fmaf_rn(a[k].x, c, off)));
              s1 = __fadd_rn(s1, fast_exp2(__fmaf_rn(a[k].y, c, off)));
              s2 = __fadd_rn(s2, fast_exp2(__fmaf_rn(a[k].z, c, off)));
              s3 = __fadd_rn(s3, fast_exp2(__fmaf_rn(a[k].w, c, off)));
            }
          }
          s.mx = m;
          s.sum = __fadd_rn(__fadd_rn(s0, s1), __fadd_rn(s2, s3));
        }
      }
    } else {
      for (int i = lo + lane; i < hi; i += 32) row_state_push<kSample>(s, __ldcs(src + i), i, c);
    }
#pragma unroll
    for (int bit = 0; bit < 5; ++bit) s = shfl_merge<kSample>(s, 1 << bit, c);
    pdl_wait_producer();  // (returns at once after the first time)
    if (lane == 0) {
      const size_t o = (size_t)row * n_chunks + ch;
      vmax[o] = s.mx;
      varg[o] = s.arg;
      if (kSample) vsum[o] = s.sum;
    }
  }
}

// Merged state of one row from its chunk partials (result in every lane);
// all loads of a lane are issued before the merges.
template <bool kSample>
__device__ __forceinline__ RowState warp_row_state(int row, int n_chunks, const float* vmax,
                                                   const float* vsum, const int* varg, float c,
                                                   int lane) {
  constexpr int NC = 8;
  float mx[NC], sm[NC];
  int ag[NC];
  RowState s = row_state_empty();
  for (int c0 = 0; c0 < n_chunks; c0 += 32 * NC) {
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      const int ch = c0 + lane + 32 * k;
      const size_t o = (size_t)row * n_chunks + ch;
      const bool ok = ch < n_chunks;
      mx[k] = ok ? vmax[o] : kNegInf;
      sm[k] = (ok && kSample) ? vsum[o] : 0.f;
      ag[k] = ok ? varg[o] : 0x7FFFFFFF;
    }
#pragma unroll
    for (int k = 0; k < NC; ++k) s = row_state_merge<kSample>(s, RowState{mx[k], sm[k], ag[k]}, c);
  }
#pragma unroll
  for (int b = 0; b < 5; ++b) s = shfl_merge<kSample>(s, 1 << b, c);
  return s;
}

// What the accept test of drafted position j of sequence b reads besides
// the row states: the drafted token, its target and draft logits and the
// uniform (loaded apart from, and in parallel with, the partial merges).
struct PosInputs {
  int x;
  float lp, lq, u;  // lq: the draft logit at x, or (low-rank form) log q(x)
};

// Where the draft distribution of a drafted position comes from: its logits
// (B x gamma x V rows), or -- the low-rank form -- the drafter head's own
// outputs: log q(x), the row's log-sum-exp at T and its z row, with the
// final draw's draft row recomputed as z W_up^T.
struct DraftSide {
  const float* rows;       // B x gamma x V draft logits, or nullptr (low-rank form)
  int ts, tp;              // drafted token of (b, j) at tokens[b * ts + j * tp]
  const float* logprob;    // low-rank: log q_j(x_j) at T, entry b * ss + j * sp
  const float* lse;        // low-rank: log sum_v exp(l_v / T), same indexing
  const uint16_t* z;       // low-rank: z rows (bf16, r wide), same indexing
  int ss, sp, r;           // low-rank: strides in rows (sequence, position) and rank
  uint16_t* z_sel;         // low-rank workspace: the z row of each sequence's draw
  unsigned* mma_ctr;       // low-rank workspace: tile counters of the recompute
  ResidRow* rrows;         // low-rank workspace: each sequence's final draw for it
};
template <bool kSample>
__device__ __forceinline__ PosInputs load_position(const float* __restrict__ target,
                                                   const DraftSide& ds,
                                                   const int32_t* __restrict__ tokens,
                                                   const Draws& dr, int b, int j, int gamma,
                                                   int V) {
  const int g1 = gamma + 1;
  PosInputs in{tokens[(size_t)b * ds.ts + (size_t)j * ds.tp], 0.f, 0.f, 0.f};
  if (kSample) {
    in.u = draw_uniform(dr.uniforms, dr.seed, dr.offset, b, j, g1);
    if (ds.rows == nullptr) in.lq = ds.logprob[(size_t)b * ds.ss + (size_t)j * ds.sp];
    if (in.x >= 0 && in.x < V) {
      in.lp = target[((size_t)b * g1 + j) * V + in.x];
      if (ds.rows != nullptr) in.lq = ds.rows[((size_t)b * gamma + j) * V + in.x];
    }
  }
  return in;
}

// Accept test of a drafted position from its merged target row state
// (pmx, psum, parg) and, when sampling, draft row state (qmx, qsum): greedy
// keeps the token iff it is the target argmax; sampling keeps it iff
// u * q(x) < p(x).  An out-of-range token rejects.
// (low-rank form: q(x) = exp(log q(x)) directly.)
template <bool kSample>
__device__ __forceinline__ bool position_accepts(const PosInputs& in, int V, float c, float pmx,
                                                 float psum, int parg, float qmx, float qsum,
                                                 bool lowrank) {
  if (in.x < 0 || in.x >= V) return false;
  if (!kSample) return in.x == parg;
  const float px = __fdiv_rn(fast_exp2((in.lp - pmx) * c), psum);
  const float qx = lowrank ? fast_exp2(in.lq * 1.4426950408889634f)
                           : __fdiv_rn(fast_exp2((in.lq - qmx) * c), qsum);
  return in.u * qx < px;
}

// ---------------------------------------------------------------- K8b ----
// Position j of every sequence, decided between row passes: one CTA per
// sequence, warp 0 merging the partials of the target row, warp 1 those of
// the draft row (sampling) and warp 2 loading the token-side inputs.  j = 0
// sets seq_ok[b] = 1 iff the drafted token is kept; j > 0 (the lazy
// schedule) clears it when position j rejects, for the sequences still kept
// (the later positions are read only for those).
template <bool kSample>
__global__ void __launch_bounds__(96)
    k_verify_first(const float* __restrict__ target, DraftSide ds,
                   const int32_t* __restrict__ tokens, int B, int gamma, int V, float c,
                   int n_chunks, const float* __restrict__ vmax, const float* __restrict__ vsum,
                   const int* __restrict__ varg, Draws dr, int j, int* __restrict__ seq_ok) {
  __shared__ RowState s_st[2];
  __shared__ PosInputs s_in;
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.x;
  if (warp == 2) {  // inputs that do not depend on the row pass
    if (lane == 0) s_in = load_position<kSample>(target, ds, tokens, dr, b, j, gamma, V);
  }
  pdl_wait_producer();
  if (j > 0 && seq_ok[b] == 0) return;  // rejected earlier: position j was not read
  if (warp == 0 || (kSample && warp == 1 && ds.rows != nullptr)) {
    const int row = warp == 0 ? b * (gamma + 1) + j : B * (gamma + 1) + b * gamma + j;
    const RowState st = warp_row_state<kSample>(row, n_chunks, vmax, vsum, varg, c, lane);
    if (lane == 0) s_st[warp] = st;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const RowState pt = s_st[0];
    const RowState pq = (kSample && ds.rows != nullptr) ? s_st[1] : row_state_empty();
    seq_ok[b] = position_accepts<kSample>(s_in, V, c, pt.mx, pt.sum, pt.arg, pq.mx, pq.sum,
                                          ds.rows == nullptr) ? 1 : 0;
  }
}

// ------------------------------------------------------------------- K9 ----
// One CTA per sequence.  All warps but the last merge the chunk partials of
// the sequence's gamma+1 target rows (and gamma draft rows) in parallel; the
// last warp loads each position's token-side inputs meanwhile.  Lane j of
// warp 0 then takes position j's decision, and the first failing position is
// found with a ballot.  With seq_ok given, position 0 was decided between
// the row passes (the same test on the same partials) and rows after a
// rejection there were not read.
constexpr int kMaxGamma = 32;
template <bool kSample>
__global__ void __launch_bounds__(544)
    k_verify_decide(const float* __restrict__ target, DraftSide ds,
                    const int32_t* __restrict__ tokens, int B, int gamma, int V, float c,
                    int n_chunks, const float* __restrict__ vmax, const float* __restrict__ vsum,
                    const int* __restrict__ varg, Draws dr,
                    const int* __restrict__ seq_ok, int32_t* __restrict__ out_tokens,
                    int32_t* __restrict__ out_nacc, VerifyInfo* __restrict__ info,
                    unsigned* err) {
  __shared__ float s_mx[2 * kMaxGamma + 1], s_sum[2 * kMaxGamma + 1];
  __shared__ int s_arg[2 * kMaxGamma + 1];
  __shared__ PosInputs s_in[kMaxGamma];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n_merge = (blockDim.x >> 5) - 1;  // merging warps; the last one loads
  const int b = blockIdx.x;
  const int g1 = gamma + 1;
  const int n_target_rows = B * g1;
  const bool lowrank = kSample && ds.rows == nullptr;
  const int rows = (kSample && !lowrank) ? g1 + gamma : g1;
  if (lowrank && b == 0 && threadIdx.x < kMmaCtrs) ds.mma_ctr[threadIdx.x] = 0u;  // recompute's
  if (warp == n_merge) {
    if (lane < gamma) {
      const PosInputs in = load_position<kSample>(target, ds, tokens, dr, b, lane, gamma, V);
      if (in.x < 0 || in.x >= V) raise_error(err, kErrIndex);
      s_in[lane] = in;
    }
  }
  pdl_wait_producer();
  for (int i = warp; i < rows && warp < n_merge; i += n_merge) {
    const int row = i < g1 ? b * g1 + i : n_target_rows + b * gamma + (i - g1);
    const RowState st = warp_row_state<kSample>(row, n_chunks, vmax, vsum, varg, c, lane);
    if (lane == 0) { s_mx[i] = st.mx; s_sum[i] = st.sum; s_arg[i] = st.arg; }
  }
  __syncthreads();
  if (warp != 0) return;
  // lane j < gamma: the decision at drafted position j
  bool ok = true;
  if (lane < gamma) {
    if (lane == 0 && seq_ok != nullptr)
      ok = seq_ok[b] != 0;
    else
      ok = position_accepts<kSample>(s_in[lane], V, c, s_mx[lane], s_sum[lane], s_arg[lane],
                                     (kSample && !lowrank) ? s_mx[g1 + lane] : 0.f,
                                     (kSample && !lowrank) ? s_sum[g1 + lane] : 1.f, lowrank);
  }
  const unsigned fail = __ballot_sync(0xFFFFFFFFu, lane < gamma && !ok);
  const int n = fail ? __ffs(fail) - 1 : gamma;
  for (int i = lane; i < g1; i += 32) {
    int32_t t = -1;
    if (i < n) t = tokens[(size_t)b * ds.ts + (size_t)i * ds.tp];
    else if (i == n) t = kSample ? -1 : s_arg[n];
    out_tokens[(size_t)b * g1 + i] = t;
  }
  if (lowrank) {
    // the z row of the final draw's draft row (position n; any row when the
    // draw is the bonus, whose weights do not use q), for the recompute
    const size_t src = (size_t)b * ds.ss + (size_t)min(n, gamma - 1) * ds.sp;
    const uint4* zs = reinterpret_cast<const uint4*>(ds.z + src * ds.r);
    uint4* zd = reinterpret_cast<uint4*>(ds.z_sel + (size_t)b * ds.r);
    for (int i = lane; i < ds.r / 8; i += 32) zd[i] = zs[i];
  }
  if (lane == 0) {
    out_nacc[b] = n;
    if (kSample) {
      VerifyInfo in{};
      in.n = n;
      in.mode = (n == gamma) ? 1 : 0;
      in.pmx = s_mx[n];
      in.pinv = __frcp_rn(s_sum[n]);
      if (n == gamma) {
        in.qmx = 0.f;
        in.qinv = 0.f;
      } else if (lowrank) {
        // q(v) = exp(l_v / T - lse) = 2^((l_v - lse T) c)
        in.qmx = ds.lse[(size_t)b * ds.ss + (size_t)n * ds.sp] * (1.4426950408889634f / c);
        in.qinv = 1.f;
      } else {
        in.qmx = s_mx[g1 + n];
        in.qinv = __frcp_rn(s_sum[g1 + n]);
      }
      info[b] = in;
      if (lowrank)
        ds.rrows[b] = ResidRow{target + ((size_t)b * g1 + n) * V, in.pmx, in.pinv, in.qmx,
                               in.mode};
    }
  }
}

// Weight of token v in the final draw of a sequence.
__device__ __forceinline__ float final_weight(const VerifyInfo& in, int mode, float lt, float lq,
                                              float c) {
  const float pv = fast_exp2((lt - in.pmx) * c) * in.pinv;
  if (mode == 1) return pv;
  const float qv = fast_exp2((lq - in.qmx) * c) * in.qinv;
  return fmaxf(pv - qv, 0.f);
}

// ------------------------------------------------------------------ K10 ----
// One warp per (sequence, chunk): mass of the final draw's distribution over
// the chunk.  Residual rows are read in two steps of 8 x 16-byte loads of
// each of the two rows in flight per lane (all 16 at once took 170 registers,
// one CTA per SM, and measured 5% slower over the whole verification); bonus
// rows come straight from the partials.
__global__ void __launch_bounds__(256)
    k_verify_resid(const float* __restrict__ target, const float* __restrict__ draft, int qs,
                   int qp, int B, int gamma, int V, float c, int n_chunks,
                   const float* __restrict__ vmax,
                   const float* __restrict__ vsum, const VerifyInfo* __restrict__ info,
                   float* __restrict__ rmass) {
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nw = gridDim.x * (blockDim.x >> 5);
  const int g1 = gamma + 1;
  const bool vec = (V & 3) == 0;
  const long long units = (long long)B * n_chunks;
  for (long long u = gw; u < units; u += nw) {
    const int b = (int)(u / n_chunks), ch = (int)(u % n_chunks);
    const VerifyInfo in = info[b];
    const int trow = b * g1 + in.n;
    float s = 0.f;
    if (in.mode == 1) {
      if (lane == 0) {
        const size_t o = (size_t)trow * n_chunks + ch;
        s = vsum[o] * fast_exp2((vmax[o] - in.pmx) * c) * in.pinv;
      }
    } else {
      const float* t = target + (size_t)trow * V;
      const float* q = draft + ((size_t)b * qs + (size_t)in.n * qp) * V;
      const int lo = ch * kVChunk, hi = min(V, lo + kVChunk);
      if (vec) {
        const float4* t4 = reinterpret_cast<const float4*>(t);
        const float4* q4 = reinterpret_cast<const float4*>(q);
        const int q1 = hi >> 2;
#pragma unroll 1
        for (int q0 = lo >> 2; q0 < q1; q0 += 32 * 8) {
          float4 a[8], bq[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int i = q0 + lane + 32 * k;
            if (i < q1) { a[k] = __ldg(t4 + i); bq[k] = __ldg(q4 + i); }
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int i = q0 + lane + 32 * k;
            if (i < q1) {
              s = __fadd_rn(s, final_weight(in, 0, a[k].x, bq[k].x, c));
              s = __fadd_rn(s, final_weight(in, 0, a[k].y, bq[k].y, c));
              s = __fadd_rn(s, final_weight(in, 0, a[k].z, bq[k].z, c));
              s = __fadd_rn(s, final_weight(in, 0, a[k].w, bq[k].w, c));
            }
          }
        }
      } else {
        for (int i = lo + lane; i < hi; i += 32)
          s = __fadd_rn(s, final_weight(in, 0, __ldg(t + i), __ldg(q + i), c));
      }
    }
    s = warp_sum_fixed(s);
    if (lane == 0) rmass[(size_t)b * n_chunks + ch] = s;
  }
}

// ------------------------------------------------------------------ K11 ----
constexpr int kMaxChunkRegs = 8;  // up to 256 chunks of 2048 floats: V <= 524288

__global__ void __launch_bounds__(256)
    k_verify_finish(const float* __restrict__ target, const float* __restrict__ draft, int qs,
                    int qp, int B, int gamma, int V, float c, int n_chunks,
                    const float* __restrict__ vmax,
                    const float* __restrict__ vsum, const VerifyInfo* __restrict__ info,
                    const float* __restrict__ rmass, Draws dr,
                    int32_t* __restrict__ out_tokens) {
  constexpr int NT = 256, PER = kVChunk / NT;  // contiguous elements per thread
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g1 = gamma + 1;
  const VerifyInfo in = info[b];
  const int trow = b * g1 + in.n;
  __shared__ int s_ch, s_mode;
  __shared__ float s_resid;
  if (warp == 0) {
    // chunk masses (up to 32 * kMaxChunkRegs chunks) in registers, one round trip
    constexpr int NC = kMaxChunkRegs;
    float rm[NC], pmass[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      const int ch = lane + 32 * k;
      const bool ok = ch < n_chunks;
      rm[k] = ok ? __ldcg(rmass + (size_t)b * n_chunks + ch) : 0.f;
      const size_t o = (size_t)trow * n_chunks + ch;
      pmass[k] = ok ? __ldcg(vsum + o) * fast_exp2((__ldcg(vmax + o) - in.pmx) * c) * in.pinv : 0.f;
    }
    int mode = in.mode;
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < NC; ++k) acc = __fadd_rn(acc, mode == 0 ? rm[k] : pmass[k]);
    float R = warp_sum_fixed(acc);
    if (!(R > 0.f) && mode == 0) {  // residual vanished: draw from p_n
      mode = 1;
      acc = 0.f;
#pragma unroll
      for (int k = 0; k < NC; ++k) acc = __fadd_rn(acc, pmass[k]);
      R = warp_sum_fixed(acc);
    }
    float mass[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) mass[k] = mode == 0 ? rm[k] : pmass[k];
    const float target_mass = draw_uniform(dr.uniforms, dr.seed, dr.offset, b, gamma, g1) * R;
    float before = 0.f;
    const int sel = ordered_crossing_regs<NC>(n_chunks, target_mass, mass, before, lane);
    if (lane == 0) {
      s_ch = sel;
      s_mode = mode;
      s_resid = target_mass - before;
    }
  }
  __syncthreads();
  const int ch = s_ch, mode = s_mode;
  const float resid = s_resid;
  const float* t = target + (size_t)trow * V;
  const float* q = draft + ((size_t)b * qs + (size_t)in.n * qp) * V;
  const int lo = ch * kVChunk + tid * PER, hi = min(V, ch * kVChunk + kVChunk);
  float wv[PER];
  float my = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int v = lo + i;
    wv[i] = (v < hi) ? final_weight(in, mode, t[v], mode == 0 ? q[v] : 0.f, c) : 0.f;
    my = __fadd_rn(my, wv[i]);
  }
  // exclusive scan of the per-thread sums (fixed order)
  float incl = my;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl = __fadd_rn(y, incl);
  }
  float ex_w = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
  if (lane == 0) ex_w = 0.f;
  __shared__ float s_w[8];
  __shared__ int s_first, s_last;
  if (lane == 31) s_w[warp] = incl;
  if (tid == 0) { s_first = NT; s_last = -1; }
  __syncthreads();
  if (tid == 0) {
    float run = 0.f;
    for (int k = 0; k < 8; ++k) { const float x = s_w[k]; s_w[k] = run; run = __fadd_rn(run, x); }
  }
  __syncthreads();
  const float excl = __fadd_rn(s_w[warp], ex_w);
  const float incl_blk = __fadd_rn(s_w[warp], incl);
  if (my > 0.f) {
    atomicMax(&s_last, tid);
    if (incl_blk > resid) atomicMin(&s_first, tid);
  }
  __syncthreads();
  const int owner = s_first < NT ? s_first : s_last;
  if (tid == owner) {
    float cum = excl;
    int tok = -1, lastp = -1;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      if (wv[i] > 0.f) {
        lastp = i;
        cum = __fadd_rn(cum, wv[i]);
        if (tok < 0 && cum > resid) tok = i;
      }
    }
    if (tok < 0) tok = lastp;
    out_tokens[(size_t)b * g1 + in.n] = lo + tok;
  } else if (owner < 0 && tid == 0) {
    out_tokens[(size_t)b * g1 + in.n] = ch * kVChunk;  // unreachable for finite inputs
  }
}

// ------------------------------------------------------------------ K12 ----
// The final draw of the low-rank draft side: one CTA of 256 threads per
// sequence.  The tcgen05 residual mode left, per 64-row sub-tile, the mass of
// max(0, p - q) and of p.  Thread j owns a contiguous run of sub-tiles; the
// draw uses the residual masses (p's when the draw is the bonus or the
// residual vanished), an ordered block scan finds the thread and then the
// sub-tile holding u * W, whose 64 draft logits are recomputed on CUDA cores
// from the sequence's z row (fp32 sums of the bf16 products) and walked in
// order with its target values.
constexpr int kLrPer = 24;  // sub-tile masses per thread: n_sub <= 6144
__global__ void __launch_bounds__(256)
    k_verify_lr_finish(const ResidRow* __restrict__ rows, const VerifyInfo* __restrict__ info,
                       const uint8_t* __restrict__ w_up, const uint16_t* __restrict__ z_sel, int r,
                       int V, float c, int n_sub, const float* __restrict__ rmass,
                       const float* __restrict__ pmass, Draws dr, int gamma,
                       int32_t* __restrict__ out_tokens) {
  constexpr int NT = 256, kW = 64;
  __shared__ float s_wsum[NT / 32], s_rsum[NT / 32];
  __shared__ float s_w[kW];
  __shared__ int s_first, s_last, s_sid;
  __shared__ float s_resid;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g1 = gamma + 1;
  const ResidRow rr = rows[b];
  const int n = info[b].n;
  const float u = draw_uniform(dr.uniforms, dr.seed, dr.offset, b, gamma, g1);
  const int per = (n_sub + NT - 1) / NT;
  const int j0 = min(n_sub, tid * per), nj = min(n_sub, j0 + per) - j0;
  float rm[kLrPer], pm[kLrPer];
#pragma unroll
  for (int k = 0; k < kLrPer; ++k) {
    rm[k] = k < nj ? __ldcg(rmass + (size_t)b * n_sub + j0 + k) : 0.f;
    pm[k] = k < nj ? __ldcg(pmass + (size_t)b * n_sub + j0 + k) : 0.f;
  }
  float mr = 0.f, mp = 0.f;
#pragma unroll
  for (int k = 0; k < kLrPer; ++k) {
    mr = __fadd_rn(mr, rm[k]);
    mp = __fadd_rn(mp, pm[k]);
  }
  // the residual's total decides which masses the draw uses
  const float wr = warp_incl_scan(mr, lane);
  if (lane == 31) s_rsum[warp] = wr;
  if (tid == 0) { s_first = NT; s_last = -1; }
  __syncthreads();
  float R = 0.f;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) R = __fadd_rn(R, s_rsum[w]);
  const bool use_p = rr.mode == 1 || !(R > 0.f);
  const float mass = use_p ? mp : mr;
  // ordered block scan of the thread masses
  const float wincl = warp_incl_scan(mass, lane);
  if (lane == 31) s_wsum[warp] = wincl;
  __syncthreads();
  float woff = 0.f, W = 0.f;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    if (w < warp) woff = __fadd_rn(woff, s_wsum[w]);
    W = __fadd_rn(W, s_wsum[w]);
  }
  const float incl = __fadd_rn(woff, wincl);
  const float prev = __shfl_up_sync(0xFFFFFFFFu, wincl, 1);
  const float excl = lane > 0 ? __fadd_rn(woff, prev) : woff;
  const float target = u * W;
  // the first thread whose inclusive mass passes the target, else (rounding)
  // the last thread with any mass
  if (mass > 0.f) {
    atomicMax(&s_last, tid);
    if (incl > target) atomicMin(&s_first, tid);
  }
  __syncthreads();
  const int sel = s_first < NT ? s_first : max(0, s_last);
  if (tid == sel) {
    float cum = excl, before_sid = excl, before_last = excl;
    int sid = -1, lastpos = -1;
#pragma unroll
    for (int k = 0; k < kLrPer; ++k) {
      const float mk = use_p ? pm[k] : rm[k];
      if (k < nj && sid < 0) {
        const float nxt = __fadd_rn(cum, mk);
        if (mk > 0.f) {
          if (nxt > target) {
            sid = j0 + k;
            before_sid = cum;
          } else {
            lastpos = j0 + k;
            before_last = cum;
          }
        }
        cum = nxt;
      }
    }
    if (sid < 0) {
      sid = lastpos >= 0 ? lastpos : j0;
      before_sid = before_last;
    }
    s_sid = sid;
    s_resid = target - before_sid;
  }
  __syncthreads();
  const int v0 = s_sid * kW;
  const int nv = max(0, min(kW, V - v0));
  // recompute: warp w takes rows 8w .. 8w+7 of the sub-tile, lanes over K
  const int nch = r / 8;  // <= 64: two 16-byte chunks per lane
  uint4 zc[2], wv[8][2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int ch = lane + 32 * q;
    zc[q] = ch < nch ? __ldg(reinterpret_cast<const uint4*>(z_sel + (size_t)b * r) + ch)
                     : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int ii = 0; ii < 8; ++ii) {
    const int i = warp * 8 + ii;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int ch = lane + 32 * q;
      wv[ii][q] = (i < nv && ch < nch)
                      ? __ldg(reinterpret_cast<const uint4*>(w_up + ((size_t)(v0 + i) * r) * 2) + ch)
                      : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  const float tv = (lane < 8 && warp * 8 + lane < nv) ? rr.trow[v0 + warp * 8 + lane] : 0.f;
#pragma unroll
  for (int ii = 0; ii < 8; ++ii) {
    float a = 0.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t ww[4] = {wv[ii][q].x, wv[ii][q].y, wv[ii][q].z, wv[ii][q].w};
      const uint32_t zz[4] = {zc[q].x, zc[q].y, zc[q].z, zc[q].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        a = fma_bf16_lo(ww[e], zz[e], a);
        a = fma_bf16_hi(ww[e], zz[e], a);
      }
    }
    a = warp_sum_fixed(a);
    const float t = __shfl_sync(0xFFFFFFFFu, tv, ii);
    if (lane == 0) {
      const int i = warp * 8 + ii;
      float w = 0.f;
      if (i < nv) {
        const float pv = fast_exp2((t - rr.pmx) * c) * rr.pinv;
        w = use_p ? pv : fmaxf(pv - fast_exp2((a - rr.qoff) * c), 0.f);
      }
      s_w[i] = w;
    }
  }
  __syncthreads();
  if (warp != 0) return;
  const float resid = s_resid;
  float cum = 0.f;
  int tok = -1, lastp = -1;
#pragma unroll
  for (int h = 0; h < kW; h += 32) {
    const float w1 = s_w[h + lane];
    const float csum = __fadd_rn(cum, warp_incl_scan(w1, lane));
    const unsigned pos = __ballot_sync(0xFFFFFFFFu, w1 > 0.f);
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, w1 > 0.f && csum > resid);
    if (tok < 0 && hit) tok = h + __ffs(hit) - 1;
    if (pos) lastp = h + 31 - __clz(pos);
    cum = __shfl_sync(0xFFFFFFFFu, csum, 31);
  }
  if (tok < 0) tok = lastp < 0 ? 0 : lastp;
  if (lane == 0) out_tokens[(size_t)b * g1 + n] = v0 + tok;
}

// -------------------------------------------------------------- host side --
// The low-rank draft side recomputes the final draws' draft rows either
// reduced on the fly to sub-tile masses against the target rows (the
// residual mode, from this many sequences on: with fewer rows per tile the
// epilogue's target loads are not hidden), or written out for the residual
// and finish kernels.
constexpr int kFusedResidMinB = 32;

// Workspace of the verifier; `lowrank` adds the draws' z rows, the
// recompute's outputs and tile counters, and drops the draft rows' partials.
static size_t ws_bytes(int B, int gamma, int V, bool sample, bool lowrank, int r) {
  const int n_chunks = (V + kVChunk - 1) / kVChunk;
  const size_t rows = (size_t)B * (gamma + 1) + ((sample && !lowrank) ? (size_t)B * gamma : 0);
  size_t s = 0;
  s += align256(rows * n_chunks * sizeof(float));       // vmax
  s += align256(rows * n_chunks * sizeof(float));       // vsum
  s += align256(rows * n_chunks * sizeof(int));         // varg
  s += align256((size_t)B * sizeof(VerifyInfo));        // info
  s += align256((size_t)B * n_chunks * sizeof(float));  // rmass
  s += align256((size_t)B * sizeof(int));               // seq_ok
  if (lowrank) {
    const size_t n_sub = 2 * (size_t)((V + 127) / 128);  // 64-row sub-tiles of the recompute
    s += align256((size_t)B * r * 2);                    // z rows of the draws
    s += align256((size_t)B * sizeof(ResidRow));         // the draws
    if (B >= kFusedResidMinB)
      s += 2 * align256((size_t)B * n_sub * sizeof(float));  // residual and p masses
    else
      s += align256((size_t)B * V * sizeof(float));          // the recomputed draft rows
    s += align256(kMmaCtrs * sizeof(unsigned));          // recompute tile counters
  }
  return s;
}
size_t verify_ws_bytes(int B, int gamma, int V, bool sample) {
  return ws_bytes(B, gamma, V, sample, false, 0);
}
size_t verify_lowrank_ws_bytes(int B, int gamma, int V, int r) {
  return ws_bytes(B, gamma, V, true, true, r);
}

namespace {
// Rows of fp32 logits above which position 0 is decided before the other
// positions are read (below it the extra launch costs more than the rows of
// sequences rejected at position 0).
constexpr double kSplitBytes = 64.0 * 1024 * 1024;

template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, int grid, int block, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Both forms: `ds.rows` (draft logits) or the low-rank draft side (with
// `w_up`, the drafter's V x r up-projection, for the recompute).
cudaError_t verify_impl(const float* target, DraftSide ds, const void* w_up,
                        const int32_t* tokens, int B, int gamma, int V, float temperature,
                        const Draws& dr, int32_t* out_tokens, int32_t* out_nacc, void* ws,
                        cudaStream_t st, bool lazy = false) {
  if (B <= 0) return cudaSuccess;
  const bool sample = temperature > 0.f;
  const bool lowrank = sample && ds.rows == nullptr;
  const float c = sample ? (float)(1.4426950408889634 / (double)temperature) : 0.f;
  const int n_chunks = (V + kVChunk - 1) / kVChunk;
  const int g1 = gamma + 1;
  const int n_target_rows = B * g1;
  const int n_rows = n_target_rows + ((sample && !lowrank) ? B * gamma : 0);
  Carver cv(ws);
  float* vmax = cv.take<float>((size_t)n_rows * n_chunks);
  float* vsum = cv.take<float>((size_t)n_rows * n_chunks);
  int* varg = cv.take<int>((size_t)n_rows * n_chunks);
  VerifyInfo* info = cv.take<VerifyInfo>(B);
  float* rmass = cv.take<float>((size_t)B * n_chunks);
  int* seq_ok = cv.take<int>(B);
  const int n_sub = 2 * ((V + 127) / 128);
  const bool fused = lowrank && B >= kFusedResidMinB;
  float* rm = nullptr;
  float* pm = nullptr;
  float* q_rows = nullptr;
  if (lowrank) {
    ds.z_sel = cv.take<uint16_t>((size_t)B * ds.r);
    ds.rrows = cv.take<ResidRow>(B);
    if (fused) {
      rm = cv.take<float>((size_t)B * n_sub);
      pm = cv.take<float>((size_t)B * n_sub);
    } else {
      q_rows = cv.take<float>((size_t)B * V);
    }
    ds.mma_ctr = cv.take<unsigned>(kMmaCtrs);
  }
  const bool split = (double)n_rows * V * 4.0 >= kSplitBytes;

  // one warp per unit; the grid is what fits on the GPU at once (one wave)
  constexpr int kThr = 256;
  const void* rows_kern = sample ? reinterpret_cast<const void*>(k_verify_rows<true>)
                                 : reinterpret_cast<const void*>(k_verify_rows<false>);
  const long long cap = (long long)resident_blocks(rows_kern, kThr, 0) * sm_count();
  const float* draft = ds.rows;
  auto rows_pass = [&](int j0, int j1, const int* ok, bool pdl) -> cudaError_t {
    const int nt = j1 - j0 + 1;
    const int nd = (sample && draft) ? std::max(0, std::min(j1, gamma - 1) - j0 + 1) : 0;
    const long long units = (long long)B * (nt + nd) * n_chunks;
    const int grid = (int)std::max<long long>(1, std::min<long long>((units + 7) / 8, cap));
    ProfScope ps(kKVerifyRows, st);
    if (pdl)
      return sample ? launch_pdl(k_verify_rows<true>, grid, kThr, st, target, draft, B, gamma, V,
                                 c, n_chunks, j0, j1, ok, vmax, vsum, varg)
                    : launch_pdl(k_verify_rows<false>, grid, kThr, st, target, draft, B, gamma,
                                 V, c, n_chunks, j0, j1, ok, vmax, vsum, varg);
    if (sample)
      k_verify_rows<true><<<grid, kThr, 0, st>>>(target, draft, B, gamma, V, c, n_chunks, j0, j1,
                                                 ok, vmax, vsum, varg);
    else
      k_verify_rows<false><<<grid, kThr, 0, st>>>(target, draft, B, gamma, V, c, n_chunks, j0,
                                                  j1, ok, vmax, vsum, varg);
    return cudaGetLastError();
  };
  cudaError_t e;
  auto decide_at = [&](int j) -> cudaError_t {
    ProfScope ps(kKVerifyFirst, st);
    return sample ? launch_pdl(k_verify_first<true>, B, 96, st, target, ds, tokens, B, gamma, V,
                               c, n_chunks, (const float*)vmax, (const float*)vsum,
                               (const int*)varg, dr, j, seq_ok)
                  : launch_pdl(k_verify_first<false>, B, 96, st, target, ds, tokens, B, gamma,
                               V, c, n_chunks, (const float*)vmax, (const float*)vsum,
                               (const int*)varg, dr, j, seq_ok);
  };
  if (lazy) {
    // position by position: each position's rows only for the sequences that
    // kept every earlier drafted token, then that position's tests; the
    // bonus row only for the sequences that kept all gamma
    for (int j = 0; j <= gamma; ++j) {
      if ((e = rows_pass(j, j, j == 0 ? nullptr : seq_ok, j > 0)) != cudaSuccess) return e;
      if (j < gamma && (e = decide_at(j)) != cudaSuccess) return e;
    }
  } else if (split) {
    // position 0 of every sequence, its decision, then the rest of the
    // sequences that kept their position-0 token
    if ((e = rows_pass(0, 0, nullptr, false)) != cudaSuccess) return e;
    if ((e = decide_at(0)) != cudaSuccess) return e;
    if ((e = rows_pass(1, gamma, seq_ok, true)) != cudaSuccess) return e;
  } else {
    // greedy: a dependent launch, streaming the rows while the preceding
    // kernel finishes
    if ((e = rows_pass(0, gamma, nullptr, !sample)) != cudaSuccess) return e;
  }
  {
    const int rows = (sample && !lowrank) ? 2 * gamma + 1 : gamma + 1;
    const int dthreads = 32 * (std::min(16, rows) + 1);  // merging warps + a loading warp
    // (lazy: every position up to a sequence's first rejection has its
    // partials, and the decide recomputes them all)
    const int* ok = split && !lazy ? seq_ok : nullptr;
    ProfScope ps(kKVerifyDecide, st);
    e = sample ? launch_pdl(k_verify_decide<true>, B, dthreads, st, target, ds, tokens, B,
                            gamma, V, c, n_chunks, (const float*)vmax, (const float*)vsum,
                            (const int*)varg, dr, ok, out_tokens, out_nacc, info,
                            error_word())
               : launch_pdl(k_verify_decide<false>, B, dthreads, st, target, ds, tokens, B,
                            gamma, V, c, n_chunks, (const float*)vmax, (const float*)vsum,
                            (const int*)varg, dr, ok, out_tokens, out_nacc, info,
                            error_word());
    if (e != cudaSuccess) return e;
  }
  if (fused) {
    // the final draws' draft rows z W_up^T on the tensor cores, reduced on the
    // fly to per-sub-tile residual and p masses against the target rows
    const MmaPlan mp = mma_plan(ds.r, B, V);
    e = launch_head_mma_resid(mp, ds.z_sel, w_up, B, ds.r, V, temperature, ds.rrows, rm, pm,
                              ds.mma_ctr, st);
    if (e != cudaSuccess) return e;
    ProfScope ps(kKVerifyFinish, st);
    k_verify_lr_finish<<<B, 256, 0, st>>>(ds.rrows, info, (const uint8_t*)w_up, ds.z_sel, ds.r,
                                          V, c, n_sub, rm, pm, dr, gamma, out_tokens);
    return cudaGetLastError();
  }
  if (sample) {
    int qs = gamma, qp = 1;
    const float* qbase = draft;
    if (lowrank) {
      // the final draws' draft rows z W_up^T on the tensor cores, written out
      const MmaPlan mp = mma_plan(ds.r, B, V);
      const MmaWork none{nullptr, nullptr, nullptr};
      const HeadOutputs no_out{Draws{nullptr, 0, 0}, nullptr, nullptr, nullptr, nullptr};
      e = launch_head_mma(mp, ds.z_sel, w_up, B, ds.r, V, 0.f, none, no_out, q_rows, ds.mma_ctr,
                          st, kKVerifyQRow);
      if (e != cudaSuccess) return e;
      qbase = q_rows;
      qs = 1;
      qp = 0;
    }
    const long long ru = (long long)B * n_chunks;
    const long long rcap = (long long)resident_blocks(reinterpret_cast<const void*>(k_verify_resid),
                                                      256, 0) * sm_count();
    const int rgrid = (int)std::max<long long>(1, std::min<long long>((ru + 7) / 8, rcap));
    {
      ProfScope ps(kKVerifyResid, st);
      k_verify_resid<<<rgrid, 256, 0, st>>>(target, qbase, qs, qp, B, gamma, V, c, n_chunks,
                                            vmax, vsum, info, rmass);
    }
    ProfScope ps(kKVerifyFinish, st);
    k_verify_finish<<<B, 256, 0, st>>>(target, qbase, qs, qp, B, gamma, V, c, n_chunks, vmax,
                                       vsum, info, rmass, dr, out_tokens);
  }
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_verify(const float* target, const float* draft, const int32_t* tokens, int B,
                          int gamma, int V, float temperature, const Draws& draws,
                          int32_t* out_tokens, int32_t* out_nacc, void* ws, cudaStream_t st,
                          bool lazy) {
  DraftSide ds{};
  ds.rows = draft;
  ds.ts = gamma;
  ds.tp = 1;
  return verify_impl(target, ds, nullptr, tokens, B, gamma, V, temperature, draws, out_tokens,
                     out_nacc, ws, st, lazy);
}

cudaError_t launch_verify_lowrank(const float* target, const void* z, const void* w_up,
                                  const float* logprob, const float* lse, int seq_stride,
                                  int pos_stride, int r, const int32_t* tokens, int B, int gamma,
                                  int V, float temperature, const Draws& draws,
                                  int32_t* out_tokens, int32_t* out_nacc, void* ws,
                                  cudaStream_t st) {
  DraftSide ds{};
  ds.rows = nullptr;
  ds.logprob = logprob;
  ds.lse = lse;
  ds.z = reinterpret_cast<const uint16_t*>(z);
  ds.ss = seq_stride;
  ds.sp = pos_stride;
  ds.ts = seq_stride;
  ds.tp = pos_stride;
  ds.r = r;
  return verify_impl(target, ds, w_up, tokens, B, gamma, V, temperature, draws, out_tokens,
                     out_nacc, ws, st);
}

}  // namespace ss
