// head_mma.cu -- the low-rank head's up-projection on the 5th-generation tensor
// cores (tcgen05), for blocks of more than 8 rows of z.
//
// SlimSpec article (荷兰Nebius团队：给AI“起草员“瘦身…), section 三: logits = z W_up^T
// over the full vocabulary.  With tens to hundreds of rows of z this is a real
// dense contraction (M x r times r x V), so it runs as a warp-specialised,
// persistent tcgen05 GEMM whose epilogue is the per-row softmax reduction:
//
//   warp 0      TMA producer: z (A, 128-row tiles, once) and W_up (B, 128-row
//               vocabulary tiles, one 64-wide K block per stage) into
//               128B-swizzled shared memory
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma kind::f16 (bf16 x bf16
//               -> fp32) into a double-buffered TMEM accumulator
//               D[m, v] (lanes = rows of z, columns = vocabulary rows)
//   warps 2-9   epilogue: tcgen05.ld of 32 columns at a time; every thread owns
//               one row of z and keeps its online (max, sum of exp, argmax)
//               state; one partial per (row, 64-row sub-tile) and per (row,
//               CTA) go to workspace (or, in the scores mode, the fp32 values
//               are written out)
//
// k_head_mma_finish then reduces the partials, one CTA per row of z: greedy
// argmax, or the inverse-CDF draw with the one sub-tile it lands in recomputed
// on CUDA cores.
#include <cuda.h>  // CUtensorMap and its enums; the encoder is fetched at run time

#include <algorithm>

#include "ss_common.cuh"
#include "ss_internal.h"

namespace ss {
namespace {

constexpr int kTileN = 128;               // vocabulary rows per tile (MMA N)
constexpr int kTileM = 128;               // rows of z per M tile (MMA M)
constexpr int kBlockBytes = 128 * 128;    // one [128 rows x 64 K] bf16 block
constexpr int kSubW = 64;                 // vocabulary rows per partial
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kMaxStages = 8;
constexpr int kSmemCap = 223 * 1024;   // dynamic; static barriers and merge buffers use the rest

// ------------------------------------------------------------- PTX wrappers --
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D (+)= A * B^T with A, B K-major bf16 tiles described by smem descriptors.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The mbarrier tracks completion of every tcgen05 operation this thread issued.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
        "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
        "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled tile whose
// 8-row groups are 1024 bytes apart (the layout TMA writes for a box of 64
// bf16 x rows with SWIZZLE_128B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4)  // start address
         | ((uint64_t)1 << 16)                // leading byte offset (unused here)
         | ((uint64_t)(1024 >> 4) << 32)      // stride byte offset: 8 rows x 128 B
         | ((uint64_t)1 << 46)                // descriptor version
         | ((uint64_t)2 << 61);               // 128-byte swizzle
}

// Instruction descriptor: bf16 A and B (K-major), fp32 accumulator, M x N.
constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4)                     // D format fp32
         | (1u << 7) | (1u << 10)      // A, B format bf16
         | ((uint32_t)(n >> 3) << 17)  // N / 8
         | ((uint32_t)(m >> 4) << 24); // M / 16
}

__device__ __forceinline__ void cta_tiles(int n_tiles, int grid, int cta, int& t0, int& nt) {
  const int base = n_tiles / grid, extra = n_tiles % grid;
  t0 = cta * base + min(cta, extra);
  nt = base + (cta < extra ? 1 : 0);
}

}  // namespace

struct MmaPart {
  float* pmax;  // [M][n_sub]  per 64-row vocabulary sub-tile
  float* psum;
  int* parg;
  float* cmax;  // [M][grid]   per CTA
  float* csum;
  int* carg;
};

// One chunk of 32 logits of a thread's row pushed into its running state.
// Out-of-range columns (only in the last vocabulary tile) are masked to -inf.
// Greedy: a max tree, and the lowest index of the maximum is looked up only
// when it beats the running maximum.  Sampling: the maximum (no index: the
// draw does not need it), then sum of 2^(x*c - max*c) in four fixed-order
// partial sums.
template <bool kSample>
__device__ __forceinline__ void epi_chunk(const uint32_t (&v)[32], int vid0, int V, RowState& st,
                                          float c) {
  float x[32];
  const bool full = vid0 + 32 <= V;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    x[j] = __uint_as_float(v[j]);
    if (!full && vid0 + j >= V) x[j] = kNegInf;
  }
  float t16[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) t16[j] = fmaxf(x[j], x[j + 16]);
#pragma unroll
  for (int w = 8; w > 0; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) t16[j] = fmaxf(t16[j], t16[j + w]);
  const float cm = t16[0];
  if (!kSample) {
    if (cm > st.mx) {
      int idx = 31;
#pragma unroll
      for (int j = 31; j >= 0; --j)
        if (x[j] == cm) idx = j;
      st.mx = cm;
      st.arg = vid0 + idx;
    }
    return;
  }
  if (cm > st.mx) {
    st.sum = st.mx == kNegInf ? 0.f : st.sum * fast_exp2((st.mx - cm) * c);
    st.mx = cm;
  }
  if (st.mx == kNegInf) return;  // nothing in range yet: -max*c would be +inf
  const float off = -st.mx * c;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    a0 = __fadd_rn(a0, fast_exp2(__fmaf_rn(x[j], c, off)));
    a1 = __fadd_rn(a1, fast_exp2(__fmaf_rn(x[j + 1], c, off)));
    a2 = __fadd_rn(a2, fast_exp2(__fmaf_rn(x[j + 2], c, off)));
    a3 = __fadd_rn(a3, fast_exp2(__fmaf_rn(x[j + 3], c, off)));
  }
  st.sum = __fadd_rn(st.sum, __fadd_rn(__fadd_rn(a0, a1), __fadd_rn(a2, a3)));
}

// ------------------------------------------------------------------ kernel --
// MT: M tiles of 128 rows of z (1 or 2).  kMode 0: softmax partials; kMode 1:
// the fp32 scores D[m, v] are written to out_scores (M x V).
template <bool kSample, int MT, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    k_head_mma(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_w,
               int M, int V, int KB, int NST, float c, int n_tiles, MmaPart part,
               float* __restrict__ out_scores, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;                                 // MT * KB blocks of z
  uint8_t* sB = smem + (size_t)MT * KB * kBlockBytes; // NST stages of W_up
  __shared__ uint64_t full[kMaxStages], empty[kMaxStages], a_full, acc_full[2], acc_empty[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ RowState s_half[kTileM];
  constexpr uint32_t kCols = 2 * MT * kTileN;  // double-buffered accumulators
  constexpr uint32_t kIdesc = idesc_bf16(kTileM, kTileN);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int t0, nt;
  cta_tiles(n_tiles, gridDim.x, blockIdx.x, t0, nt);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&a_full, 1);
    mbar_init(&acc_full[0], 1);
    mbar_init(&acc_full[1], 1);
    mbar_init(&acc_empty[0], kEpiWarps);
    mbar_init(&acc_empty[1], kEpiWarps);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&s_tmem, kCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_launch_dependents();  // the finish may be scheduled; it waits for this grid

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      tma_prefetch_desc(&tm_w);
      tma_prefetch_desc(&tm_z);
      int it = 0;
      bool a_issued = false;
      const int total = nt * KB;
      for (; it < total; ++it) {
        const int s = it % NST;
        if (it >= NST && !a_issued) {
          // z is written by the down-projection that precedes this grid
          pdl_wait_producer();
          mbar_arrive_expect_tx(&a_full, (uint32_t)(MT * KB * kBlockBytes));
          for (int mt = 0; mt < MT; ++mt)
            for (int kb = 0; kb < KB; ++kb)
              tma_load_2d(sA + (size_t)(mt * KB + kb) * kBlockBytes, &tm_z, kb * 64,
                          mt * kTileM, &a_full);
          a_issued = true;
        }
        if (!mbar_wait_bounded(&empty[s], ((it / NST) & 1) ^ 1, err)) {
          s_abort = 1;
          break;
        }
        const int t = t0 + it / KB, kb = it % KB;
        mbar_arrive_expect_tx(&full[s], (uint32_t)kBlockBytes);
        tma_load_2d(sB + (size_t)s * kBlockBytes, &tm_w, kb * 64, t * kTileN, &full[s]);
      }
      if (!a_issued && it >= total) {
        pdl_wait_producer();
        mbar_arrive_expect_tx(&a_full, (uint32_t)(MT * KB * kBlockBytes));
        for (int mt = 0; mt < MT; ++mt)
          for (int kb = 0; kb < KB; ++kb)
            tma_load_2d(sA + (size_t)(mt * KB + kb) * kBlockBytes, &tm_z, kb * 64, mt * kTileM,
                        &a_full);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      bool ok = mbar_wait_bounded(&a_full, 0, err);
      tc_fence_after();
      int it = 0;
      for (int i = 0; i < nt && ok; ++i) {
        const int buf = i & 1;
        if (!mbar_wait_bounded(&acc_empty[buf], ((i >> 1) & 1) ^ 1, err)) { ok = false; break; }
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % NST;
          if (!mbar_wait_bounded(&full[s], (it / NST) & 1, err)) { ok = false; break; }
          tc_fence_after();
          const uint64_t bdesc = sw128_desc(smem_u32(sB + (size_t)s * kBlockBytes));
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              const uint64_t adesc =
                  sw128_desc(smem_u32(sA + (size_t)(mt * KB + kb) * kBlockBytes));
              mma_bf16(tmem + (uint32_t)((buf * MT + mt) * kTileN), adesc + 2 * k4,
                       bdesc + 2 * k4, kIdesc, (kb | k4) != 0 ? 1u : 0u);
            }
          }
          mma_commit(&empty[s]);  // the stage is free once these MMAs complete
        }
        if (!ok) break;
        mma_commit(&acc_full[buf]);
      }
      if (!ok) s_abort = 1;
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int ew = warp - 2;             // 0 .. 7
    const int quad = warp & 3;           // the TMEM lane quadrant this warp may read
    const int mt = MT == 2 ? ew / 4 : 0;
    const int half = MT == 2 ? 0 : ew / 4;
    const int row = mt * kTileM + quad * 32 + lane;  // row of z owned by this thread
    const bool live = row < M;
    const bool warp_live = mt * kTileM + quad * 32 < M;  // any live row in this warp
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    RowState tot = row_state_empty();
    for (int i = 0; i < nt; ++i) {
      const int buf = i & 1;
      const bool ok = mbar_wait_bounded(&acc_full[buf], (i >> 1) & 1, err);
      if (!__all_sync(0xFFFFFFFFu, ok) || *(volatile int*)&s_abort) break;
      tc_fence_after();
      const int t = t0 + i;
#pragma unroll
      for (int hh = 0; hh < (MT == 2 ? 2 : 1); ++hh) {
        const int h = MT == 2 ? hh : half;
        RowState st = row_state_empty();
        if (warp_live) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int col = h * kSubW + cc * 32;
            uint32_t v[32];
            tmem_ld32(tmem + lane_addr + (uint32_t)((buf * MT + mt) * kTileN + col), v);
            const int vid0 = t * kTileN + col;
            if (kMode == 1) {
              if (live) {
                float* dst = out_scores + (size_t)row * V + vid0;
                if (vid0 + 32 <= V && (V & 3) == 0) {
#pragma unroll
                  for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4*>(dst + j) =
                        make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                    __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
                } else {
                  for (int j = 0; j < 32; ++j)
                    if (vid0 + j < V) dst[j] = __uint_as_float(v[j]);
                }
              }
            } else {
              epi_chunk<kSample>(v, vid0, V, st, c);
            }
          }
        }
        if (kMode == 0) {
          if (live) {
            const size_t o = (size_t)row * (2 * n_tiles) + 2 * t + h;
            part.pmax[o] = st.mx;
            part.parg[o] = st.arg;
            if (kSample) part.psum[o] = st.sum;
          }
          tot = row_state_merge<kSample>(tot, st, c);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
    if (kMode == 0) {
      // one partial per (row, CTA); with MT == 1 two warps hold the two
      // column halves of each row and are merged in a fixed order
      if (MT == 1) {
        if (half == 1) s_half[quad * 32 + lane] = tot;
        asm volatile("bar.sync 1, %0;" ::"r"(32 * kEpiWarps) : "memory");
        if (half == 0) tot = row_state_merge<kSample>(tot, s_half[quad * 32 + lane], c);
      }
      if (live && (MT == 2 || half == 0)) {
        const size_t o = (size_t)row * gridDim.x + blockIdx.x;
        part.cmax[o] = tot.mx;
        part.carg[o] = tot.arg;
        if (kSample) part.csum[o] = tot.sum;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kCols);
}

// ------------------------------------------------------------------ finish --
// One CTA of 8 warps per row of z.  Warp 0 merges the partials: the maximum,
// W and (sampling) the CTA and the 64-row sub-tile where the inverse CDF
// crosses u * W.  The 8 warps then recompute that sub-tile's logits (8 rows
// each, every load issued up front; CUDA-core fp32 accumulation of the same
// bf16 products) and warp 0 walks them in row order.
template <bool kSample>
__global__ void __launch_bounds__(256)
    k_head_mma_finish(const uint8_t* __restrict__ w_up, const uint8_t* __restrict__ z, int M,
                      int r, int V, float c, float inv_t, int n_tiles, int grid, MmaPart part,
                      HeadOutputs out) {
  __shared__ float s_logit[kSubW];
  __shared__ float s_f[4];  // gmax, W, resid
  __shared__ int s_i[2];    // sub-tile, token (greedy)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x;
  pdl_wait_producer();
  if (m >= M) return;
  const int n_sub = 2 * n_tiles;
  if (warp == 0) {
    const float* cm = part.cmax + (size_t)m * grid;
    const int* ca = part.carg + (size_t)m * grid;
    const float* cs = part.csum + (size_t)m * grid;
    constexpr int NC = 8;  // up to 256 CTAs
    float pmx[NC], psm[NC];
    int pag[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      const int t = lane + 32 * k;
      const bool ok = t < grid;
      pmx[k] = ok ? __ldcg(cm + t) : kNegInf;
      pag[k] = ok ? __ldcg(ca + t) : 0x7FFFFFFF;
      psm[k] = (ok && kSample) ? __ldcg(cs + t) : 0.f;
    }
    RowState st = row_state_empty();
#pragma unroll
    for (int k = 0; k < NC; ++k)
      st = row_state_merge<false>(st, RowState{pmx[k], 0.f, pag[k]}, c);
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
    } else {
      float cmass[NC];
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < NC; ++k) {
        cmass[k] = psm[k] * fast_exp2((pmx[k] - gmax) * c);
        acc = __fadd_rn(acc, cmass[k]);
      }
      const float W = warp_sum_fixed(acc);
      const float target = __ldg(out.uniforms + m) * W;
      float before1 = 0.f, before2 = 0.f;
      const int cta = ordered_crossing_regs<NC>(grid, target, cmass, before1, lane);
      int ct0, cnt;
      cta_tiles(n_tiles, grid, cta, ct0, cnt);
      const int s0 = 2 * ct0, ns = 2 * cnt;  // this CTA's sub-tiles, contiguous
      const float* pm = part.pmax + (size_t)m * n_sub + s0;
      const float* ps = part.psum + (size_t)m * n_sub + s0;
      float smass[NC];
#pragma unroll
      for (int k = 0; k < NC; ++k) {
        const int t = lane + 32 * k;
        smass[k] = t < ns ? __ldcg(ps + t) * fast_exp2((__ldcg(pm + t) - gmax) * c) : 0.f;
      }
      const float resid1 = target - before1;
      const int sid = s0 + ordered_crossing_regs<NC>(ns, resid1, smass, before2, lane);
      if (lane == 0) {
        s_f[0] = gmax;
        s_f[1] = W;
        s_f[2] = resid1 - before2;
        s_i[0] = sid;
      }
    }
  }
  if (!kSample) return;
  __syncthreads();
  const float gmax = s_f[0], W = s_f[1], resid = s_f[2];
  const int v0 = s_i[0] * kSubW;
  const int n = max(0, min(kSubW, V - v0));
  // recompute: warp w takes rows 8w .. 8w+7 of the sub-tile, lanes over K
  const int nch = r / 8;
  uint4 zc[2], wv[8][2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int ch = lane + 32 * q;
    zc[q] = ch < nch ? __ldg(reinterpret_cast<const uint4*>(z + ((size_t)m * r + ch * 8) * 2))
                     : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int ii = 0; ii < 8; ++ii) {
    const int i = warp * 8 + ii;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int ch = lane + 32 * q;
      wv[ii][q] = (i < n && ch < nch) ? __ldg(reinterpret_cast<const uint4*>(
                                            w_up + ((size_t)(v0 + i) * r + ch * 8) * 2))
                                      : make_uint4(0u, 0u, 0u, 0u);
    }
  }
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
    if (lane == 0) s_logit[warp * 8 + ii] = a;
  }
  __syncthreads();
  if (warp != 0) return;
  float cum = 0.f;
  int tok = -1, lastp = -1;
#pragma unroll
  for (int h = 0; h < kSubW; h += 32) {
    const int i = h + lane;
    const float wv1 = i < n ? fast_exp2((s_logit[i] - gmax) * c) : 0.f;
    const float csum = __fadd_rn(cum, warp_incl_scan(wv1, lane));
    const unsigned pos = __ballot_sync(0xFFFFFFFFu, wv1 > 0.f);
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, wv1 > 0.f && csum > resid);
    if (tok < 0 && hit) tok = h + __ffs(hit) - 1;
    if (pos) lastp = h + 31 - __clz(pos);
    cum = __shfl_sync(0xFFFFFFFFu, csum, 31);
  }
  if (tok < 0) tok = lastp < 0 ? 0 : lastp;
  if (lane == 0) {
    const float lW = logf(W);
    out.tokens[m] = v0 + tok;
    if (out.logprob) out.logprob[m] = (s_logit[tok] - gmax) * inv_t - lW;
    if (out.row_max) out.row_max[m] = gmax;
    if (out.row_lse) out.row_lse[m] = gmax * inv_t + lW;
  }
}

// -------------------------------------------------------------- host side --
namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D bf16 tensor [rows x cols] (row-major), boxes of 64 columns x 128 rows,
// 128-byte swizzle, out-of-range elements read as zero.
bool make_map(CUtensorMap* map, const void* base, int rows, int cols) {
  EncodeTiledFn enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

MmaPlan mma_plan(int r, int M, int V) {
  MmaPlan p{};
  p.ok = false;
  if (M <= 0 || M > 2 * kTileM || r % 8 != 0 || r > 512) return p;  // finish: <= 2 chunks per lane
  p.mt = M <= kTileM ? 1 : 2;
  p.kb = (r + 63) / 64;
  const int a_bytes = p.mt * p.kb * kBlockBytes;
  const int room = kSmemCap - 1024 - a_bytes;
  p.nst = std::min(kMaxStages, room / kBlockBytes);
  if (p.nst < 3) return p;
  p.smem = 1024 + a_bytes + p.nst * kBlockBytes;
  p.n_tiles = (V + kTileN - 1) / kTileN;
  p.grid = std::max(1, std::min(sm_count(), p.n_tiles));
  p.n_sub = 2 * p.n_tiles;
  p.ok = true;
  return p;
}

template <bool kSample, int MT, int kMode>
static cudaError_t launch_mma_one(const MmaPlan& p, const CUtensorMap& tz, const CUtensorMap& tw,
                                  int M, int V, float c, const MmaPart& part, float* scores,
                                  cudaStream_t st) {
  auto kern = k_head_mma<kSample, MT, kMode>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), p.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ProfScope ps(kKHeadMma, st);
  return cudaLaunchKernelEx(&cfg, kern, tz, tw, M, V, p.kb, p.nst, c, p.n_tiles, part, scores,
                            error_word());
}

cudaError_t launch_head_mma(const MmaPlan& p, const void* z_ws, const void* w_up, int M, int r,
                            int V, float temperature, const MmaWork& w, const HeadOutputs& out,
                            float* scores, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  CUtensorMap tz, tw;
  if (!make_map(&tz, z_ws, M, r) || !make_map(&tw, w_up, V, r)) return cudaErrorInvalidValue;
  const bool sample = temperature > 0.f && scores == nullptr;
  const double inv = sample ? 1.0 / (double)temperature : 0.0;
  const float c = (float)(1.4426950408889634 * inv), inv_t = (float)inv;
  const MmaPart part{w.pmax, w.psum, w.parg, w.cmax, w.csum, w.carg};
  cudaError_t e;
  if (scores != nullptr) {
    e = p.mt == 1 ? launch_mma_one<false, 1, 1>(p, tz, tw, M, V, c, part, scores, st)
                  : launch_mma_one<false, 2, 1>(p, tz, tw, M, V, c, part, scores, st);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  if (sample)
    e = p.mt == 1 ? launch_mma_one<true, 1, 0>(p, tz, tw, M, V, c, part, nullptr, st)
                  : launch_mma_one<true, 2, 0>(p, tz, tw, M, V, c, part, nullptr, st);
  else
    e = p.mt == 1 ? launch_mma_one<false, 1, 0>(p, tz, tw, M, V, c, part, nullptr, st)
                  : launch_mma_one<false, 2, 0>(p, tz, tw, M, V, c, part, nullptr, st);
  if (e != cudaSuccess) return e;
  // the per-row finish, launched to overlap the tail of the MMA grid
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ProfScope ps(kKHeadFinish, st);
  if (sample)
    e = cudaLaunchKernelEx(&cfg, k_head_mma_finish<true>, (const uint8_t*)w_up,
                           (const uint8_t*)z_ws, M, r, V, c, inv_t, p.n_tiles, p.grid, part, out);
  else
    e = cudaLaunchKernelEx(&cfg, k_head_mma_finish<false>, (const uint8_t*)w_up,
                           (const uint8_t*)z_ws, M, r, V, c, inv_t, p.n_tiles, p.grid, part, out);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace ss
