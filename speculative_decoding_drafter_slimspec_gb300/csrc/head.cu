// head.cu -- SlimSpec low-rank drafter head on sm_103a CUDA cores.
//
// SlimSpec article (荷兰Nebius团队：给AI“起草员“瘦身…), section 三: the V x d head is
// replaced by W_down (d -> r) and W_up (r -> V).  The up-projection reads W_up
// (V x r, 78-145 MB at the article's model shapes) once per call and, for a
// handful of rows, is bound by HBM bandwidth; it is written as a streaming
// GEMV with the per-row softmax reduction fused into the stream:
//
//   k_down_proj    z = bf16(h W_down^T); all loads of a thread issued before
//                  any use (one round trip); also clears the CTA counters.
//                  Launched as a dependent of the previous library kernel: it
//                  reads and multiplies while that kernel finishes and waits
//                  for it only before writing.
//   k_head_stream  W_up tiles -> shared memory by cp.async.bulk (a 3-deep ring
//                  per warp, no cross-warp synchronisation in the stream), dot
//                  products with mixed-precision FMAs (bf16 x bf16 + fp32, no
//                  widening instructions) and z held in registers as bf16
//                  pairs, a select-free reduce-scatter across lanes, and
//                  an online (max, sum of exp, argmax) state per row of z.  One
//                  partial per (row of z, vocabulary tile) goes to workspace;
//                  logits never leave the chip.  The last CTA to finish (an
//                  atomic counter) merges the partials, one warp per row of z:
//                  greedy takes the argmax; sampling finds the tile where the
//                  inverse CDF crosses u * W, recomputes that tile's logits
//                  bit-identically and walks it.
#include <algorithm>

#include "ss_common.cuh"
#include "ss_internal.h"

namespace ss {

// ----------------------------------------------------------- geometry -------
// kBF16: element type of W_up; LPR lanes share one row; each lane holds CPL
// 16-byte chunks of the row; MT rows of z are handled per launch.
template <bool kBF16, int LPR_, int CPL_, int MT_, int SPLIT_, int UNITS_>
struct Gemv {
  static constexpr bool BF16 = kBF16;
  static constexpr int LPR = LPR_, CPL = CPL_, MT = MT_;  // MT rows of z per warp
  static constexpr int SPLIT = SPLIT_;              // warps sharing one ring (and row range)
  static constexpr int MTL = MT * SPLIT;            // rows of z per launch
  static constexpr int E = kBF16 ? 8 : 4;           // elements per 16-byte chunk
  static constexpr int EB = kBF16 ? 2 : 4;          // bytes per element
  static constexpr int GROUPS = 32 / LPR;           // lane groups per warp
  static constexpr int UNITS = UNITS_;              // rings (row ranges) per CTA
  static constexpr int NST = 3;                     // ring depth
  static constexpr int STAGE_TARGET = 196608 / (UNITS * NST);  // 192 KB of rings per CTA
  static constexpr int MAX_ROW_BYTES = LPR * CPL * 16;
  static constexpr int R_CAP = STAGE_TARGET / (MAX_ROW_BYTES * GROUPS);  // a pass fits a stage
  static constexpr int R_WANT = (SPLIT > 1 ? 8 : (UNITS > 8 ? 16 : 32)) / MT;
  static constexpr int R_RAW = R_WANT < R_CAP ? R_WANT : R_CAP;
  static constexpr int R = R_RAW < 1 ? 1 : (R_RAW > 8 ? 8 : R_RAW);  // rows per group per pass
  static constexpr int PASS_ROWS = R * GROUPS;
  static constexpr int STAGE_RAW = STAGE_TARGET / MAX_ROW_BYTES;
  static constexpr int STAGE_ROWS =
      STAGE_RAW < PASS_ROWS ? PASS_ROWS : (STAGE_RAW / PASS_ROWS) * PASS_ROWS;
  static constexpr int PPS = STAGE_ROWS / PASS_ROWS;  // passes per stage
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
  static constexpr int WARPS = UNITS * SPLIT;
  static constexpr int SMEM = UNITS * NST * STAGE_BYTES + UNITS * NST * 8;
  static_assert(LNF <= LMT, "reduced values of one lane must belong to distinct rows of z");
  static_assert(SUB_ROWS % PASS_ROWS == 0 && STAGE_ROWS % PASS_ROWS == 0, "pass alignment");
  static_assert(SUB_ROWS <= 64, "finish walks at most two rows per lane");
  static_assert(MTL <= WARPS, "one finishing warp per row of z");
  static_assert(SPLIT == 1 || SPLIT == 2, "one or two warps per ring");
  static_assert(WARPS <= 32, "at most 1024 threads");
  static_assert(SMEM <= 220 * 1024, "shared memory");
  static_assert(SMEM >= MTL * 24576, "the finish reuses the rings: 24 KB per finishing warp");
  static_assert(12288 / MAX_ROW_BYTES >= PASS_ROWS, "a finish chunk holds at least one pass");
};

// Lane-dependent slot permutation of the select-free reduce-scatter.
template <class G>
__device__ __forceinline__ int slot_mask(int lane) {
  return ((lane % G::LPR) >> G::DUP_BITS) << G::LNF;
}

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

// z rows of the warp's slice starting at m0, in this lane's slot order
// (register j holds z row m0 + (j ^ zmask)), this lane's chunks as four 32-bit
// words per chunk (bf16 pairs or fp32 values, as the workspace holds them);
// zero outside the matrix.
template <class G>
__device__ __forceinline__ void load_z(uint32_t (&zr)[G::MT][G::CPL][4], const uint8_t* z, int M,
                                       int m0, int r, int lane) {
  const int nch = r / G::E;
  const int li = lane % G::LPR;
  const int zmask = slot_mask<G>(lane) & (G::MT - 1);
#pragma unroll
  for (int j = 0; j < G::MT; ++j) {
    const int m = m0 + (j ^ zmask);
#pragma unroll
    for (int c = 0; c < G::CPL; ++c) {
      const int ch = li + c * G::LPR;
      const bool ok = (m < M) && (ch < nch);
      const uint4 a = ok ? ldg16(z + ((size_t)m * r + (size_t)ch * G::E) * G::EB)
                         : make_uint4(0u, 0u, 0u, 0u);
      zr[j][c][0] = a.x;
      zr[j][c][1] = a.y;
      zr[j][c][2] = a.z;
      zr[j][c][3] = a.w;
    }
  }
}

// Dot products of the PASS_ROWS rows of one pass with the MT rows of z,
// reduced across each lane group.  Row i of the pass starts at byte offset
// i * row_bytes from the base; rows at or beyond `nvalid` contribute zeros.
// The arithmetic (explicit packed fma / add in a fixed order, per lane) is the
// same wherever it is inlined, so the stream and the recompute produce
// identical bits.
template <class G, bool kShared>
__device__ __forceinline__ void pass_dots(const uint8_t* gbase, uint32_t sbase, int row_bytes,
                                          int nvalid, int nch,
                                          const uint32_t (&zr)[G::MT][G::CPL][4],
                                          float (&v)[G::N], int lane) {
  const int g = lane / G::LPR, li = lane % G::LPR;
  const int rmask = slot_mask<G>(lane) >> G::LMT;
  uint4 wv[G::R][G::CPL];
#pragma unroll
  for (int q = 0; q < G::R; ++q) {
    const int row = (q ^ rmask) * G::GROUPS + g;
#pragma unroll
    for (int c = 0; c < G::CPL; ++c) {
      const int ch = li + c * G::LPR;
      if (row < nvalid && ch < nch) {
        const int off = row * row_bytes + ch * 16;
        wv[q][c] = kShared ? lds16(sbase + off) : ldg16(gbase + off);
      } else {
        wv[q][c] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  float acc[G::R][G::MT];
#pragma unroll
  for (int q = 0; q < G::R; ++q)
#pragma unroll
    for (int j = 0; j < G::MT; ++j) acc[q][j] = 0.f;
  // element order within a lane: chunk c, word i, low then high half; the
  // R * MT accumulators are independent between two updates of the same one
#pragma unroll
  for (int c = 0; c < G::CPL; ++c) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int q = 0; q < G::R; ++q) {
        const uint32_t wq = i == 0 ? wv[q][c].x : i == 1 ? wv[q][c].y : i == 2 ? wv[q][c].z
                                                                                : wv[q][c].w;
#pragma unroll
        for (int j = 0; j < G::MT; ++j) {
          if constexpr (G::BF16) {
            acc[q][j] = fma_bf16_lo(wq, zr[j][c][i], acc[q][j]);
            acc[q][j] = fma_bf16_hi(wq, zr[j][c][i], acc[q][j]);
          } else {
            acc[q][j] = __fmaf_rn(__uint_as_float(wq), __uint_as_float(zr[j][c][i]), acc[q][j]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int q = 0; q < G::R; ++q)
#pragma unroll
    for (int j = 0; j < G::MT; ++j) v[q * G::MT + j] = acc[q][j];
  ReduceScatterP<G::N, G::LPR / 2>::run(v);
}

// Contiguous vocabulary rows of stream warp g out of TW: equal shares, the
// first V % TW warps one row more.
__device__ __forceinline__ void warp_rows(int g, int TW, int V, int& start, int& count) {
  const int base = V / TW, extra = V % TW;
  start = g * base + min(g, extra);
  count = base + (g < extra ? 1 : 0);
}

// Index (row of the pass, row of z within the tile) held in reduced slot j.
template <class G>
__device__ __forceinline__ void slot_of(int lane, int j, int& row_in_pass, int& m) {
  const int g = lane / G::LPR;
  const int idx = slot_mask<G>(lane) + j;
  m = idx % G::MT;
  row_in_pass = (idx / G::MT) * G::GROUPS + g;
}

// --------------------------------------------------------- down-projection --
// CTA: JT=4 output columns x MT=8 rows of h; its 8 warps split the d axis; each
// thread issues all of its loads (Q chunks of 4 W rows and 8 h rows) first.
template <bool kBF16, int Q>
__global__ void __launch_bounds__(256) k_down_proj(const uint8_t* __restrict__ h,
                                                   const uint8_t* __restrict__ w, int M, int d,
                                                   int r, int round, uint8_t* __restrict__ z_ws,
                                                   uint8_t* __restrict__ out_z,
                                                   unsigned* __restrict__ ctr, int n_ctr) {
  constexpr int E = kBF16 ? 8 : 4, EB = kBF16 ? 2 : 4, JT = 4, MT = 8;
  const int j0 = blockIdx.x * JT, m0 = blockIdx.y * MT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();  // the up-projection may start its W_up prologue now
  const int nch = d / E;
  const size_t rowb = (size_t)d * EB;
  uint4 wr[Q][JT], hr[Q][MT];
#pragma unroll
  for (int k = 0; k < Q; ++k) {
    const int q = lane + 32 * warp + 256 * k;
#pragma unroll
    for (int a = 0; a < JT; ++a)
      wr[k][a] = (q < nch && j0 + a < r) ? ldg16(w + (size_t)(j0 + a) * rowb + q * 16)
                                         : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int b = 0; b < MT; ++b)
      hr[k][b] = (q < nch && m0 + b < M) ? ldg16(h + (size_t)(m0 + b) * rowb + q * 16)
                                         : make_uint4(0u, 0u, 0u, 0u);
  }
  float acc[JT][MT];
#pragma unroll
  for (int a = 0; a < JT; ++a)
#pragma unroll
    for (int b = 0; b < MT; ++b) acc[a][b] = 0.f;
#pragma unroll
  for (int k = 0; k < Q; ++k) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int a = 0; a < JT; ++a) {
        const uint4 wa = wr[k][a];
        const uint32_t wq = i == 0 ? wa.x : i == 1 ? wa.y : i == 2 ? wa.z : wa.w;
#pragma unroll
        for (int b = 0; b < MT; ++b) {
          const uint4 hb = hr[k][b];
          const uint32_t hq = i == 0 ? hb.x : i == 1 ? hb.y : i == 2 ? hb.z : hb.w;
          if constexpr (kBF16) {
            acc[a][b] = fma_bf16_lo(wq, hq, acc[a][b]);
            acc[a][b] = fma_bf16_hi(wq, hq, acc[a][b]);
          } else {
            acc[a][b] = __fmaf_rn(__uint_as_float(wq), __uint_as_float(hq), acc[a][b]);
          }
        }
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
  // Launched as a dependent of the previous library kernel: h and W are
  // inputs (never library outputs), read above while it may still run; z and
  // the counters may still be in use by it, so they wait for its completion.
  pdl_wait_producer();
  if (ctr != nullptr && blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < n_ctr; i += blockDim.x) ctr[i] = 0u;
  __syncthreads();
  if (warp == 0) {
    float s = red[0][lane];
#pragma unroll
    for (int k = 1; k < 8; ++k) s = __fadd_rn(s, red[k][lane]);
    const int j = j0 + lane / MT, m = m0 + lane % MT;
    if (j < r && m < M) {
      const float zv = round ? round_bf16(s) : s;
      if (kBF16) {
        const uint16_t bits = f32_to_bf16_bits(zv);
        reinterpret_cast<uint16_t*>(z_ws)[(size_t)m * r + j] = bits;
        if (out_z) reinterpret_cast<uint16_t*>(out_z)[(size_t)m * r + j] = bits;
      } else {
        reinterpret_cast<float*>(z_ws)[(size_t)m * r + j] = zv;
        if (out_z) reinterpret_cast<float*>(out_z)[(size_t)m * r + j] = zv;
      }
    }
  }
}

// -------------------------------------------------------- per-row finish ----
struct HeadOut {
  Draws draws;  // row m draws (row m, slot 0)
  int32_t* tokens;
  float* logprob;
  float* row_max;
  float* row_lse;
};

struct HeadPart {
  float* pmax;  // [M][n_sub] sub-tile partials
  float* psum;
  int* parg;
  float* cmax;  // [M][grid] CTA partials
  float* csum;
  int* carg;
};

constexpr int kFinChunks = 8;       // per-CTA partials scanned by the finish: up to 256 CTAs
constexpr int kFinBytes = 24576;    // shared memory per finishing warp for the recompute

// One warp reduces the partials of row m and draws its token: the maximum
// and W from the per-CTA partials, then (sampling) the CTA and, inside it, the
// sub-tile where the inverse CDF crosses u * W, whose logits are recomputed
// from a copy of its rows in shared memory (fsmem, kFinBytes, two halves each
// tracked by one of the mbarriers fbar[0..1]).
template <class G, bool kSample>
__device__ __forceinline__ void finish_row(int m, const uint8_t* __restrict__ w,
                                           const uint8_t* __restrict__ z, int M, int r, int V,
                                           float c, float inv_t, int n_sub, int grid,
                                           const HeadPart& part, const HeadOut& out,
                                           float* s_logit, uint8_t* fsmem, uint64_t* fbar,
                                           unsigned* err, int lane) {
  const float* cm = part.cmax + (size_t)m * grid;
  const int* ca = part.carg + (size_t)m * grid;
  const float* cs = part.csum + (size_t)m * grid;
  // 1. all CTA partials of the row in registers (one round trip)
  float pmx[kFinChunks], psm[kFinChunks];
  int pag[kFinChunks];
#pragma unroll
  for (int k = 0; k < kFinChunks; ++k) {
    const int t = lane + 32 * k;
    const bool ok = t < grid;
    pmx[k] = ok ? __ldcg(cm + t) : kNegInf;
    pag[k] = ok ? __ldcg(ca + t) : 0x7FFFFFFF;
    psm[k] = (ok && kSample) ? __ldcg(cs + t) : 0.f;
  }
  RowState st = row_state_empty();
#pragma unroll
  for (int k = 0; k < kFinChunks; ++k) st = row_state_merge<false>(st, RowState{pmx[k], 0.f, pag[k]}, c);
#pragma unroll
  for (int b = 0; b < 5; ++b) st = shfl_merge<false>(st, 1 << b, c);
  const float gmax = st.mx;
  if (!kSample) {
    if (lane == 0) {
      out.tokens[m] = st.arg;
      if (out.logprob) out.logprob[m] = 0.f;
      if (out.row_max) out.row_max[m] = gmax;
      if (out.row_lse) out.row_lse[m] = gmax;
    }
    return;
  }
  // 2. CTA masses relative to the row maximum and their total W (fixed order)
  float cmass[kFinChunks];
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < kFinChunks; ++k) {
    cmass[k] = psm[k] * fast_exp2((pmx[k] - gmax) * c);
    acc = __fadd_rn(acc, cmass[k]);
  }
  const float W = warp_sum_fixed(acc);
  const float target =
      draw_uniform(out.draws.uniforms, out.draws.seed, out.draws.offset, m, 0, 1) * W;
  // 3. the CTA, then the sub-tile inside it, where the running mass passes u * W
  float before1 = 0.f, before2 = 0.f;
  const int cta = ordered_crossing_regs<kFinChunks>(grid, target, cmass, before1, lane);
  const int per_cta = n_sub / grid;  // UNITS * spw sub-tiles, contiguous per CTA
  const float* pm = part.pmax + (size_t)m * n_sub + (size_t)cta * per_cta;
  const float* ps = part.psum + (size_t)m * n_sub + (size_t)cta * per_cta;
  float smass[kFinChunks];
#pragma unroll
  for (int k = 0; k < kFinChunks; ++k) {
    const int t = lane + 32 * k;
    smass[k] = t < per_cta ? __ldcg(ps + t) * fast_exp2((__ldcg(pm + t) - gmax) * c) : 0.f;
  }
  const float resid1 = target - before1;
  const int tstar = cta * per_cta + ordered_crossing_regs<kFinChunks>(per_cta, resid1, smass, before2, lane);
  const float resid = resid1 - before2;
  // 4. recompute the logits of sub-tile tstar with the stream's arithmetic,
  //    its rows copied to shared memory in chunks (two in flight)
  const int m0 = (m / G::MT) * G::MT;   // the warp slice of the stream that held row m
  uint32_t zr[G::MT][G::CPL][4];
  load_z<G>(zr, z, M, m0, r, lane);
  const int row_bytes = r * G::EB, nch = r / G::E;
  const int tw = G::UNITS * grid;
  const int spw = n_sub / tw;
  int wstart, wcount;
  warp_rows(tstar / spw, tw, V, wstart, wcount);
  const int trow0 = wstart + (tstar % spw) * G::SUB_ROWS;
  const int n = max(0, min(G::SUB_ROWS, wstart + wcount - trow0));
  const uint8_t* base = w + (size_t)trow0 * row_bytes;
  const bool dup_leader = (lane & ((1 << G::DUP_BITS) - 1)) == 0;
  const int crows = ((kFinBytes / 2) / row_bytes) / G::PASS_ROWS * G::PASS_ROWS;  // >= PASS_ROWS
  if (lane == 0) {
    mbar_init(&fbar[0], 1);
    mbar_init(&fbar[1], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const int n_chunks = (n + crows - 1) / crows;
  auto issue_chunk = [&](int k) {
    const int r0 = k * crows, nr = min(crows, n - r0);
    const uint32_t bytes = (uint32_t)(nr * row_bytes);
    mbar_arrive_expect_tx(&fbar[k & 1], bytes);
    bulk_g2s(fsmem + (k & 1) * (kFinBytes / 2), base + (size_t)r0 * row_bytes, bytes, &fbar[k & 1]);
  };
  if (lane == 0) {
    if (n_chunks > 0) issue_chunk(0);
    if (n_chunks > 1) issue_chunk(1);
  }
  bool ok = true;
  int kfail = n_chunks;
  for (int k = 0; k < n_chunks; ++k) {
    ok = ok && __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&fbar[k & 1], (k >> 1) & 1, err));
    if (!ok) {
      kfail = k;
      break;
    }
    const int r0 = k * crows, nr = min(crows, n - r0);
    const uint32_t sb = smem_u32(fsmem + (k & 1) * (kFinBytes / 2));
#pragma unroll 1
    for (int p = 0; p < nr; p += G::PASS_ROWS) {
      float v[G::N];
      pass_dots<G, true>(nullptr, sb + p * row_bytes, row_bytes, nr - p, nch, zr, v, lane);
#pragma unroll
      for (int j = 0; j < G::NF; ++j) {
        int rip, mm;
        slot_of<G>(lane, j, rip, mm);
        if (dup_leader && m0 + mm == m && p + rip < nr) s_logit[r0 + p + rip] = v[j];
      }
    }
    __syncwarp();
    if (lane == 0 && k + 2 < n_chunks) {
      fence_proxy_async_smem();
      issue_chunk(k + 2);
    }
  }
  if (!ok) {
    // a copy did not arrive in time: leave the row's token invalid, after
    // the copies still in flight into this warp's buffers have landed
    // (chunks kfail and kfail + 1: each later one is issued only after the
    // one two before it was consumed)
    if (lane == 0) {
      out.tokens[m] = -1;
      for (int k = kfail; k < n_chunks && k < kfail + 2; ++k)
        mbar_wait_drain(&fbar[k & 1], (k >> 1) & 1, err);
    }
    __syncwarp();
    return;
  }
  __syncwarp();
  // 5. walk the sub-tile in row order: lane i holds rows i and i + 32
  float cum = 0.f;
  int tok = -1, lastp = -1;
#pragma unroll
  for (int h = 0; h < G::SUB_ROWS; h += 32) {
    const int i = h + lane;
    const float wv = i < n ? fast_exp2((s_logit[i] - gmax) * c) : 0.f;
    const float csum = __fadd_rn(cum, warp_incl_scan(wv, lane));
    const unsigned pos = __ballot_sync(0xFFFFFFFFu, wv > 0.f);
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, wv > 0.f && csum > resid);
    if (tok < 0 && hit) tok = h + __ffs(hit) - 1;
    if (pos) lastp = h + 31 - __clz(pos);
    cum = __shfl_sync(0xFFFFFFFFu, csum, 31);
  }
  if (tok < 0) tok = lastp < 0 ? 0 : lastp;
  if (lane == 0) {
    const float lW = logf(W);
    out.tokens[m] = trow0 + tok;
    if (out.logprob) out.logprob[m] = (s_logit[tok] - gmax) * inv_t - lW;
    if (out.row_max) out.row_max[m] = gmax;
    if (out.row_lse) out.row_lse[m] = gmax * inv_t + lW;
  }
}

// ----------------------------------------------------------- stream (K2) ----
// Grid: at most one CTA per SM, WARPS warps each.  The vocabulary is cut into
// one contiguous range of rows per warp (equal shares), each range into
// sub-tiles of SUB_ROWS rows (partial t = warp * spw + sub-tile).  Each warp
// runs its own cp.async.bulk ring over its range.
template <class G, bool kSample>
__global__ void __launch_bounds__(32 * G::WARPS, 1)
    k_head_stream(const uint8_t* __restrict__ w, const uint8_t* __restrict__ z, int M, int m0,
                  int r, int V, float c, float inv_t, int n_sub, HeadPart part,
                  float* __restrict__ out_logits, unsigned* __restrict__ ctr, HeadOut out,
                  unsigned* err) {
  float* __restrict__ pmax = part.pmax;
  float* __restrict__ psum = part.psum;
  int* __restrict__ parg = part.parg;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_fin[G::WARPS][G::SUB_ROWS];
  __shared__ int s_last;
  __shared__ int s_abort[G::UNITS];
  __shared__ RowState s_tot[G::UNITS][G::MTL];
  __shared__ uint64_t s_fbar[G::MTL][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = warp / G::SPLIT;               // ring / row range of this warp
  const int half = warp % G::SPLIT;               // its slice of the launch's rows of z
  const bool leader = half == 0;                  // the warp that refills the ring
  const int mw = m0 + half * G::MT;               // first row of z of this warp
  const int grid = gridDim.x;
  const int TW = G::UNITS * grid;                 // row ranges in the grid
  const int gw = blockIdx.x * G::UNITS + unit;    // this warp's range
  const int spw = n_sub / TW;                     // sub-tiles per range
  int wstart, wcount;
  warp_rows(gw, TW, V, wstart, wcount);
  const int n_stages = spw * G::SPS;
  uint8_t* ring = smem + unit * G::NST * G::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G::UNITS * G::NST * G::STAGE_BYTES) +
                   unit * G::NST;
  if (lane == 0 && leader) s_abort[unit] = 0;
  const int row_bytes = r * G::EB;
  const int nch = r / G::E;

  // stage s = sub-tile s / SPS of the range, its (s % SPS)-th STAGE_ROWS rows;
  // empty stages (past the range end) only occur at the end
  auto stage_rows = [&](int s, int& row0) -> int {
    row0 = wstart + (s / G::SPS) * G::SUB_ROWS + (s % G::SPS) * G::STAGE_ROWS;
    const int n = wstart + wcount - row0;
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

  // both warps of a unit meet at a named barrier (id 1 + unit) once per stage
  auto unit_sync = [&]() {
    if constexpr (G::SPLIT > 1)
      asm volatile("bar.sync %0, %1;" ::"r"(1 + unit), "r"(32 * G::SPLIT) : "memory");
    else
      __syncwarp();
  };
  if (n_stages > 0) {
    if (lane == 0 && leader) {
      for (int s = 0; s < G::NST; ++s) mbar_init(&bars[s], 1);
      fence_mbar_init();
    }
    unit_sync();
    if (lane == 0 && leader)
      for (int s = 0; s < G::NST && s < n_stages; ++s) issue(s);
    // z and the completion counter come from the down-projection
    pdl_wait_producer();

    uint32_t zr[G::MT][G::CPL][4];
    load_z<G>(zr, z, M, mw, r, lane);
    RowState st[G::NF], tot[G::NF];
#pragma unroll
    for (int j = 0; j < G::NF; ++j) st[j] = tot[j] = row_state_empty();
    const bool dup_leader = (lane & ((1 << G::DUP_BITS) - 1)) == 0;

    int s = 0;
    for (; s < n_stages; ++s) {
      int row0;
      const int n = stage_rows(s, row0);
      bool stage_ok = true;
      if (n > 0) {
        const bool ok = mbar_wait_bounded(&bars[s % G::NST], (s / G::NST) & 1, err);
        stage_ok = __all_sync(0xFFFFFFFFu, ok);
        if (!stage_ok && lane == 0) s_abort[unit] = 1;
      }
      if (n > 0 && stage_ok) {
        const uint32_t sb = smem_u32(ring + (s % G::NST) * G::STAGE_BYTES);
#pragma unroll
        for (int pp = 0; pp < G::PPS; ++pp) {
          const int p = pp * G::PASS_ROWS;
          if (p < n) {
            float v[G::N];
            pass_dots<G, true>(nullptr, sb + p * row_bytes, row_bytes, n - p, nch, zr, v, lane);
#pragma unroll
            for (int j = 0; j < G::NF; ++j) {
              int rip, m;
              slot_of<G>(lane, j, rip, m);
              const int row = p + rip;
              if (row < n) {
                row_state_push<kSample>(st[j], v[j], row0 + row, c);
                if (out_logits != nullptr && dup_leader && mw + m < M)
                  out_logits[(size_t)(mw + m) * V + row0 + row] = v[j];
              }
            }
          }
        }
      }
      unit_sync();
      if (s_abort[unit]) break;  // a wait of this unit ran out (both warps see it)
      if (lane == 0 && leader && s + G::NST < n_stages) {
        fence_proxy_async_smem();
        issue(s + G::NST);
      }
      if (s % G::SPS == G::SPS - 1) {
        const int t = gw * spw + s / G::SPS;
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
            if (mw + m < M) {
              const size_t o = (size_t)(mw + m) * n_sub + t;
              pmax[o] = st[j].mx;
              parg[o] = st[j].arg;
              if (kSample) psum[o] = st[j].sum;
            }
            tot[j] = row_state_merge<kSample>(tot[j], st[j], c);
          }
        }
#pragma unroll
        for (int j = 0; j < G::NF; ++j) st[j] = row_state_empty();
      }
    }
    // the unit's totals (held by the writer lanes) go to shared memory
    if ((lane >> G::MERGE_LO) == 0 && dup_leader) {
#pragma unroll
      for (int j = 0; j < G::NF; ++j) {
        int rip, m;
        slot_of<G>(lane, j, rip, m);
        s_tot[unit][half * G::MT + m] = tot[j];
      }
    }
    if (s < n_stages && lane == 0 && leader) {
      // A wait ran out: drain (bounded) the copies still in flight into this
      // warp's ring before the CTA's shared memory is released.
      for (int k = s; k < n_stages && k < s + G::NST; ++k) {
        int row0;
        if (stage_rows(k, row0) > 0) mbar_wait_drain(&bars[k % G::NST], (k / G::NST) & 1, err);
      }
    }
  }

  // one partial per (row of z, CTA): the units' totals merged in unit order
  if (n_stages <= 0) pdl_wait_producer();
  __syncthreads();
  if (lane == 0 && warp < G::MTL && m0 + warp < M) {
    RowState a = s_tot[0][warp];
    for (int u = 1; u < G::UNITS; ++u) a = row_state_merge<kSample>(a, s_tot[u][warp], c);
    const size_t o = (size_t)(m0 + warp) * grid + blockIdx.x;
    part.cmax[o] = a.mx;
    part.carg[o] = a.arg;
    if (kSample) part.csum[o] = a.sum;
  }
  // the last CTA to finish merges the partials of this launch's rows of z
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(ctr, 1u);
    s_last = (prev == (unsigned)grid - 1u) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int m = m0 + warp;
  if (warp < G::MTL && m < M)
    finish_row<G, kSample>(m, w, z, M, r, V, c, inv_t, n_sub, grid, part, out, s_fin[warp],
                           smem + warp * kFinBytes, s_fbar[warp], err, lane);
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
                             bool round_bf16_z, void* z_ws, void* out_z, unsigned* ctr,
                             int n_ctr, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  dim3 grid((r + 3) / 4, (M + 7) / 8);
  const int nch = d / (bf16 ? 8 : 4);
  const int q = (nch + 255) / 256;
  const uint8_t* hp = (const uint8_t*)h;
  const uint8_t* wp = (const uint8_t*)w;
  uint8_t* oz = (uint8_t*)out_z;
  const int rnd = round_bf16_z ? 1 : 0;
  ProfScope ps(kKDownProj, st);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
#define SS_DOWN(B, Q)                                                                     \
  do {                                                                                      \
    cudaError_t e0 = set_smem_once(reinterpret_cast<const void*>(k_down_proj<B, Q>), 0);    \
    if (e0 != cudaSuccess) return e0;                                                       \
    e0 = cudaLaunchKernelEx(&cfg, k_down_proj<B, Q>, hp, wp, M, d, r, rnd, (uint8_t*)z_ws,  \
                            oz, ctr, n_ctr);                                                \
    if (e0 != cudaSuccess) return e0;                                                       \
  } while (0)
  if (bf16) {
    if (q <= 1) SS_DOWN(true, 1);
    else if (q <= 2) SS_DOWN(true, 2);
    else if (q <= 4) SS_DOWN(true, 4);
    else return cudaErrorInvalidConfiguration;
  } else {
    if (q <= 1) SS_DOWN(false, 1);
    else if (q <= 2) SS_DOWN(false, 2);
    else if (q <= 4) SS_DOWN(false, 4);
    else return cudaErrorInvalidConfiguration;
  }
#undef SS_DOWN
  return cudaGetLastError();
}

// The geometries the library instantiates: (bf16, lanes per row, chunks per
// lane, rows of z per warp, warps per ring).
#define SS_HEAD_GEOMS(X)  \
  X(true, 32, 1, 1, 1, 16)  \
  X(true, 32, 1, 4, 1, 16)  \
  X(true, 32, 1, 8, 1, 16)  \
  X(true, 32, 2, 1, 1, 16)  \
  X(true, 32, 2, 4, 1, 16)  \
  X(true, 32, 2, 8, 1, 16)  \
  X(true, 32, 4, 1, 1, 16)  \
  X(true, 32, 4, 4, 1, 16)  \
  X(false, 8, 1, 1, 1, 8)   \
  X(false, 8, 1, 8, 1, 8)   \
  X(false, 32, 1, 1, 1, 8)  \
  X(false, 32, 1, 8, 1, 8)  \
  X(false, 32, 2, 1, 1, 8)  \
  X(false, 32, 2, 8, 1, 8)

HeadPlan head_plan(bool bf16, int r, int M, int V) {
  HeadPlan p{};
  p.ok = false;
  int mtw = 1, split = 1;
  if (bf16) {
    const int nch = r / 8;
    if (nch <= 32) p.cpl = 1;
    else if (nch <= 64) p.cpl = 2;
    else if (nch <= 128) p.cpl = 4;
    else return p;
    p.lpr = 32;
    mtw = (M <= 1) ? 1 : (M <= 4 || p.cpl == 4) ? 4 : 8;
  } else {
    const int nch = r / 4;
    if (nch <= 8) { p.lpr = 8; p.cpl = 1; }
    else if (nch <= 32) { p.lpr = 32; p.cpl = 1; }
    else if (nch <= 64) { p.lpr = 32; p.cpl = 2; }
    else return p;
    mtw = (M <= 1) ? 1 : 8;
  }
  p.mtw = mtw;
  p.split = split;
  p.mt = mtw * split;
#define SS_SUBROWS(B, L, C, T, SP, U)                                    \
  if (bf16 == B && p.lpr == L && p.cpl == C && mtw == T && split == SP) { \
    p.sub_rows = Gemv<B, L, C, T, SP, U>::SUB_ROWS;                       \
    p.units = U;                                                          \
    p.ok = true;                                                          \
  }
  SS_HEAD_GEOMS(SS_SUBROWS)
#undef SS_SUBROWS
  if (p.ok) {
    const int want = (V + p.units * 32 - 1) / (p.units * 32);  // >= ~32 rows per range
    p.grid = std::max(1, std::min(sm_count(), want));
    const int tw = p.units * p.grid;
    const int max_rows = (V + tw - 1) / tw;
    const int spw = std::max(1, (max_rows + p.sub_rows - 1) / p.sub_rows);
    p.n_sub = tw * spw;
    p.n_launch = (M + p.mt - 1) / p.mt;
  }
  return p;
}

template <class G, bool kSample>
static cudaError_t stream_one(const void* w_up, const void* z_ws, int M, int r, int V, float c,
                              float inv_t, const HeadPlan& plan, HeadPartials part,
                              float* out_logits, const HeadOutputs& o, cudaStream_t st) {
  auto kern = k_head_stream<G, kSample>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), G::SMEM);
  if (e != cudaSuccess) return e;
  const int grid = plan.grid;
  HeadOut out{o.draws, o.tokens, o.logprob, o.row_max, o.row_lse};
  for (int m0 = 0, k = 0; m0 < M; m0 += G::MTL, ++k) {
    ProfScope ps(kKHeadStream, st);
    const HeadPart hp{part.pmax, part.psum, part.parg, part.cmax, part.csum, part.carg};
    // programmatic dependent launch: overlaps this grid's prologue (barrier
    // set-up, first W_up copies) with the tail of the kernel before it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32 * G::WARPS);
    cfg.dynamicSmemBytes = G::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, (const uint8_t*)w_up, (const uint8_t*)z_ws, M, m0, r, V, c,
                           inv_t, plan.n_sub, hp, out_logits, part.ctr + k, out, error_word());
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_head_stream(const HeadPlan& plan, bool bf16, const void* w_up,
                               const void* z_ws, int M, int r, int V, float temperature,
                               HeadPartials part, float* out_logits, const HeadOutputs& o,
                               cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  const bool sample = temperature > 0.f;
  const double inv = sample ? 1.0 / (double)temperature : 0.0;
  const float c = (float)(1.4426950408889634 * inv), inv_t = (float)inv;
#define SS_STREAM(B, L, C, T, SP, U)                                                          \
  if (bf16 == B && plan.lpr == L && plan.cpl == C && plan.mtw == T && plan.split == SP)       \
    return sample ? stream_one<Gemv<B, L, C, T, SP, U>, true>(w_up, z_ws, M, r, V, c, inv_t,  \
                                                              plan, part, out_logits, o, st)  \
                  : stream_one<Gemv<B, L, C, T, SP, U>, false>(w_up, z_ws, M, r, V, c, inv_t, \
                                                               plan, part, out_logits, o, st);
  SS_HEAD_GEOMS(SS_STREAM)
#undef SS_STREAM
  return cudaErrorInvalidConfiguration;
}

}  // namespace ss
