// head_mma.cu -- the low-rank head's up-projection on the 5th-generation tensor
// cores (tcgen05), for bf16 heads with up to 256 rows of z.
//
// SlimSpec article (荷兰Nebius团队：给AI“起草员“瘦身…), section 三: logits = z W_up^T
// over the full vocabulary.  The product is a skinny dense contraction
// (M x r times r x V).  Even for a single row of z it runs on the tensor
// cores: they take the multiply-adds off the issue slots, and the kernel is
// left to move W_up at the speed of HBM.  One persistent CTA per SM,
// warp-specialised, with the per-row softmax reduction as the GEMM epilogue:
//
//   warp 0      producer.  It takes 128-row vocabulary tiles (fixed ones,
//               then the next free tile from a global counter, so that SMs
//               that stream faster take more tiles; under a full HBM queue an
//               atomic takes microseconds, so each draw is made a tile ahead),
//               hands their ids to the other warps through a small ring in
//               shared memory,
//               and loads W_up (B, one 64-wide K block of a tile per 16 KB
//               stage, or several as one 4-D box, 128B-swizzled) with TMA,
//               L2 evict-first.  One issuing thread keeps only
//               about one box per 800 cycles under way, short of this SM's
//               share of HBM bandwidth, so lane 0 waits for a group of up to
//               four free stages and that many lanes issue together.
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma kind::f16 (bf16 x bf16
//               -> fp32) into a double-buffered TMEM accumulator
//               D[m, v] (lanes = rows of z, columns = vocabulary rows)
//   warps 2-9   epilogue.  First, once the down-projection is complete, they
//               copy z (A, 128-row tiles) into shared memory with ordinary
//               loads, in the 128B-swizzled layout, so that it does not queue
//               behind the W_up boxes already in flight.  Then, per tile,
//               tcgen05.ld of 32 columns at a time; every thread owns one row
//               of z.  Sampling: each 64-row sub-tile reduced to one partial
//               (max, sum of exp) in workspace.  Greedy: one running key of
//               the row's maximum and its lowest index, added with a 64-bit
//               atomicMax at the end.  (The scores mode writes the fp32
//               values out.)
//
// z is stored compactly: a 128-row tile of z with only M' live rows keeps
// ceil(M'/8) swizzle atoms (8 rows x 128 bytes) per K block.  The MMA still
// reads 128 rows; rows past the live ones come from whatever follows in shared
// memory and only reach rows of D that nothing reads.  For a few rows of z
// this frees almost all of shared memory for W_up stages.
//
// k_head_mma_finish then writes the outputs: greedy, one thread per row of z
// from its key; sampling, one CTA per row reduces the partials in vocabulary
// order to the inverse-CDF draw, the one sub-tile it lands in recomputed on
// CUDA cores.
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
constexpr int kProdGroup = 4;             // stages the producer issues together
constexpr int kMmaWarp = 1;               // TMEM owner and MMA issuer
constexpr int kEpiWarp0 = 2;              // first epilogue warp
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kMaxStages = 16;
constexpr int kTileRing = 8;              // tile ids in flight between the warps
constexpr int kStaticTiles = 2;           // tiles b, b + grid of CTA b; the rest are claimed
constexpr int kSmemCap = 223 * 1024;      // dynamic; static barriers use the rest
constexpr int kSmemCapDual = 226 * 1024;  // the dual plan: all but 1 KB of the 227 KB a CTA may use
constexpr int kFinThreads = 256;
constexpr int kFinPer = 24;               // partials per finish thread: n_sub <= 6144

// ------------------------------------------------------------- PTX wrappers --
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// The same load with an L2 cache policy (createpolicy) for the lines read.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
// One box of a 4-D map (x, y, z, w) -- the wide stages' {64, 8, 4, 16} boxes --
// with an L2 cache policy.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            int w, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)),
      "l"(pol)
      : "memory");
}
// L2 policies: lines read once are evicted first, so that a stream larger
// than L2 does not push out what was written beside it and is read next
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// A box of a tensor map brought into L2 only (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* map, int x, int y, int z, int w) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(w)
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
// 16-byte asynchronous global -> shared copy; src_bytes < 16 zero-fills the rest.
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane; the registers are
// valid after tmem_ld_wait().
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&v)[32]) {
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
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled tile: 8-row
// groups (swizzle atoms of 8 x 128 bytes) `sbo` bytes apart -- 1024 for a box
// of 64 bf16 x rows written by TMA with SWIZZLE_128B, 4096 inside a wide
// stage where the four K blocks of each 8-row group sit side by side.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t sbo = 1024) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4)  // start address
         | ((uint64_t)1 << 16)                // leading byte offset (unused here)
         | ((uint64_t)(sbo >> 4) << 32)       // stride byte offset between 8-row groups
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

// Swizzle atoms (8 rows of z) kept per K block for a CTA's Ml <= 128 rows of
// z, the byte offset of K block kb of them in shared memory, and their size.
__host__ __device__ __forceinline__ int z_atoms(int Ml) {
  return Ml >= kTileM ? kTileM / 8 : (Ml + 7) / 8;
}
__host__ __device__ __forceinline__ int z_block_off(int Ml, int kb) {
  return kb * z_atoms(Ml) * 1024;
}
__host__ __device__ __forceinline__ int z_bytes(int Ml, int KB) { return KB * z_atoms(Ml) * 1024; }

}  // namespace

struct MmaPart {
  float* pmax;  // [M][n_sub]  per 64-row vocabulary sub-tile (sampling, residual)
  float* psum;
  // greedy: per row of z, atomicMax of (float_key(max) << 32 | ~index) over
  // every thread's tiles -- the row's maximum with the lowest index among ties
  unsigned long long* best;
};

__device__ __forceinline__ unsigned long long best_key(float v, int idx) {
  return ((unsigned long long)float_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}
// the float a float_key came from (the key maps -0 to +0)
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// The greedy outputs of row m from its best key: the token (through the id
// map of a trimmed head), log-probability 0, and the maximum as both the row's
// maximum and its log-sum-exp (the temperature-0 limit).  No key, or an index
// outside the vocabulary, only follows an aborted up-projection: no token then,
// and no id-map read.
__device__ __forceinline__ void write_greedy(const HeadOutputs& out, int V, int m,
                                             unsigned long long kk) {
  const float gmax = kk != 0ull ? key_float((uint32_t)(kk >> 32)) : kNegInf;
  const int idx = (int)(0xFFFFFFFFu - (uint32_t)kk);
  const bool in = kk != 0ull && idx >= 0 && idx < V;
  out.tokens[m] = !in ? -1 : out.id_map != nullptr ? out.id_map[idx] : idx;
  if (out.logprob) out.logprob[m] = 0.f;
  if (out.row_max) out.row_max[m] = gmax;
  if (out.row_lse) out.row_lse[m] = gmax;
}

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
// Every CTA holds one M tile of up to 128 rows of z: CTA b takes M tile
// b % m_tiles and streams the vocabulary tiles of that M tile with the other
// gridDim.x / m_tiles CTAs of it (their own tile counter).  With two M tiles
// each W_up tile is then read by two CTAs (the second read mostly from L2);
// the dual plan below instead keeps both tiles of z in every CTA, when three
// W_up stages still fit beside them, so that each SM takes W_up in once.  kMode 0: softmax
// partials (sampling) or best keys (greedy); kMode 1: the fp32 scores
// D[m, v] are written to out_scores (M x V); kMode 2: the residual masses of
// a verified sequence's final draw (ResidRow), the target values of each
// tile loaded ahead of its accumulator, into part.pmax (residual) and
// part.psum (p).  kWide false: a
// W_up stage is one K block, a 2-D box of 128 rows x 128 bytes.  kWide true:
// a stage is KPS K blocks -- WB full ones as one 4-D box of 128 rows x WB*128
// contiguous bytes (every row's bytes of the stage in one request run: fewer
// DRAM page openings per byte), then, when r is not a multiple of 64, the
// ragged last block as a 2-D box.  kDual (softmax partials, 2-D stages,
// 128 < M <= 256): every CTA holds both M tiles of z and issues both MMA
// chains on each W_up stage, into four TMEM accumulators (two tiles x double
// buffering), so each SM takes in W_up once instead of once per M tile;
// m_tiles is then 1 and all CTAs share one tile counter.  tile_ctr is zeroed
// by the down-projection that precedes this grid.
template <bool kSample, int kMode, bool kWide, bool kDual = false>
__global__ void __launch_bounds__(kThreads, 1)
    k_head_mma(const uint16_t* __restrict__ z, const __grid_constant__ CUtensorMap tm_w,
               const __grid_constant__ CUtensorMap tm_w2, int M, int m_tiles, int R, int V, int KB,
               int KPS, int WB, int NST, float c, int n_tiles, MmaPart part,
               float* __restrict__ out_scores, const ResidRow* __restrict__ rrows,
               unsigned* __restrict__ tile_ctr, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int mtc = (int)blockIdx.x % m_tiles;   // this CTA's M tile
  const int cb = (int)blockIdx.x / m_tiles;    // its index among that tile's CTAs
  const int gm = (int)gridDim.x / m_tiles;     // CTAs per M tile
  const int m0 = mtc * kTileM;                 // first row of z of this CTA
  const int Ml = min(kTileM, M - m0);          // rows of z of this CTA (its first M tile)
  const int Ml1 = kDual ? M - kTileM : 0;      // rows of its second M tile (dual)
  uint8_t* sA = smem;                          // KB compact blocks of z
  uint8_t* sA1 = smem + z_bytes(Ml, KB);       // the second M tile's blocks (dual)
  uint8_t* sB = sA1 + (kDual ? z_bytes(Ml1, KB) : 0);  // NST stages of W_up
  const int kStageBytes = (kWide ? KPS : 1) * kBlockBytes;
  const int SPT = kWide ? KB / KPS : KB;       // stages per vocabulary tile
  __shared__ uint64_t full[kMaxStages], empty[kMaxStages], a_full, acc_full[2], acc_empty[2];
  __shared__ uint64_t tile_full[kTileRing], tile_empty[kTileRing], mma_done, never;
  __shared__ int s_tile[kTileRing];    // vocabulary tile ids, -1 = no more
  __shared__ int s_fills[kMaxStages];  // TMA fills issued per stage (drained before exit)
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  constexpr int kMT = kDual ? 2 : 1;                  // M tiles per CTA
  constexpr uint32_t kCols = 2 * kMT * kTileN;        // double-buffered accumulators
  constexpr uint32_t kIdesc = idesc_bf16(kTileM, kTileN);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      s_fills[s] = 0;
    }
    for (int s = 0; s < kTileRing; ++s) {
      mbar_init(&tile_full[s], 1);
      mbar_init(&tile_empty[s], 1 + kEpiWarps);  // the MMA thread and each epilogue warp
    }
    mbar_init(&a_full, kEpiWarps);
    mbar_init(&acc_full[0], 1);
    mbar_init(&acc_full[1], 1);
    mbar_init(&acc_empty[0], kEpiWarps);
    mbar_init(&acc_empty[1], kEpiWarps);
    mbar_init(&mma_done, 1);
    mbar_init(&never, 1);  // nothing arrives on it: the stall test's wait
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&s_tmem, kCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_launch_dependents();  // the finish may be scheduled; it waits for this grid

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    // Stage `it` (counted over all tiles in order) lives in slot it % NST.
    // Lane 0 waits until the last stage of a group of G is free: the MMA
    // frees stages in order, so the earlier ones are free too, and with
    // G <= NST the parity of that slot's barrier names the round waited for.
    if (lane == 0) {
      tma_prefetch_desc(&tm_w);
      if (kWide && WB < KPS) tma_prefetch_desc(&tm_w2);
      // the static tiles' stages beyond the ring, into L2 while z is still
      // being computed: they are read as soon as the MMAs free the ring (at
      // most one more ring's worth: a tile of many K blocks would otherwise
      // bring megabytes per CTA into L2 long before they are used)
      for (int q = NST; q < kStaticTiles * SPT && q < 2 * NST; ++q) {
        const int t = cb + (q / SPT) * gm;
        if (t >= n_tiles) break;
        const int kb0 = (q % SPT) * (kWide ? KPS : 1);
        if (!kWide) {
          tma_prefetch_2d(&tm_w, kb0 * 64, t * kTileN);
        } else {
          if (WB > 0) tma_prefetch_4d(&tm_w, 0, 0, kb0, t * (kTileN / 8));
          if (WB < KPS) tma_prefetch_2d(&tm_w2, (kb0 + WB) * 64, t * kTileN);
        }
      }
    }
    // Waiting for the last of G stages leaves NST - G + 1 in flight when a
    // group goes out: a short ring (a large z) issues in pairs, a ring of wide
    // stages one at a time (one 64 KB box keeps ~80 B/clk under way).
    const int G = kWide ? 1 : (NST >= 2 * kProdGroup ? kProdGroup : 2);
    // W_up is read once when one M tile (or every CTA both) covers z: its
    // lines go first, and the partials, keys and z stay in L2 for the finish.
    // With the M tiles split over CTAs the second read is meant to hit L2.
    const uint64_t pol = m_tiles == 1 ? l2_evict_first() : l2_evict_normal();
    int it = 0;
    bool ok = true;
    // Tiles cb + k * gm (k < kStaticTiles) are this CTA's own (the first is
    // loaded while the down-projection runs); tile kStaticTiles * gm + k goes
    // to whichever CTA of this M tile draws k from its counter.  Lane 0 draws one tile ahead:
    // the draw gets a tile's worth of loads to come back, and a CTA holds at
    // most one tile it has not started when the counter runs out.
    unsigned q0 = 0;
    for (int i = 0; ok; ++i) {
      int t;
      if (i < kStaticTiles) {
        t = cb + i * gm;
      } else {
        t = kStaticTiles * gm + (int)__shfl_sync(0xFFFFFFFFu, q0, 0);
        if (lane == 0 && t < n_tiles) q0 = atomicAdd(tile_ctr + mtc, 1u);  // none past the end
      }
      if (t >= n_tiles) t = -1;
      const int slot = i % kTileRing;
      if (lane == 0) {
        ok = mbar_wait_bounded(&tile_empty[slot], ((i / kTileRing) & 1) ^ 1, err);
        if (ok) {
          s_tile[slot] = t;
          mbar_arrive(&tile_full[slot]);
        } else {
          s_abort = 1;
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (t < 0) break;
      for (int st0 = 0; st0 < SPT && ok; st0 += G) {
        const int g = SPT - st0 < G ? SPT - st0 : G;
        const int last = it + g - 1;
        if (lane == 0 && !mbar_wait_bounded(&empty[last % NST], ((last / NST) & 1) ^ 1, err)) {
          ok = false;
          s_abort = 1;
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
        if (lane < g) {
          const int s = (it + lane) % NST;
          mbar_arrive_expect_tx(&full[s], (uint32_t)kStageBytes);
          uint8_t* dst = sB + (size_t)s * kStageBytes;
          if (!kWide) {
            tma_load_2d(dst, &tm_w, (st0 + lane) * 64, t * kTileN, &full[s], pol);
          } else {
            const int kb0 = (st0 + lane) * KPS;
            if (WB > 0) tma_load_4d(dst, &tm_w, 0, 0, kb0, t * (kTileN / 8), &full[s], pol);
            if (WB < KPS)  // the ragged last K block (columns past r read as zero)
              tma_load_2d(dst + (size_t)WB * kBlockBytes, &tm_w2, (kb0 + WB) * 64, t * kTileN,
                          &full[s], pol);
          }
          atomicAdd(&s_fills[s], 1);
        }
        __syncwarp();
        it += g;
      }
      if (i == kStaticTiles - 1 && lane == 0) {
        pdl_wait_producer();  // the counter is zeroed by the down-projection
        q0 = atomicAdd(tile_ctr + mtc, 1u);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      // the failure-detection test: with the control block's switch on, the
      // issuer first waits on a barrier that nothing arrives on, runs out of
      // time, and the whole CTA takes its abort path
      bool ok = !(err != nullptr && control(err)->stall_head != 0u) ||
                mbar_wait_bounded(&never, 0, err);
      ok = ok && mbar_wait_bounded(&a_full, 0, err);
      tc_fence_after();
      int it = 0;
      for (int i = 0; ok; ++i) {
        const int slot = i % kTileRing;
        if (!mbar_wait_bounded(&tile_full[slot], (i / kTileRing) & 1, err)) { ok = false; break; }
        const int t = *(volatile int*)&s_tile[slot];
        mbar_arrive(&tile_empty[slot]);
        if (t < 0) break;
        const int buf = i & 1;
        if (!mbar_wait_bounded(&acc_empty[buf], ((i >> 1) & 1) ^ 1, err)) { ok = false; break; }
        tc_fence_after();
        for (int sj = 0; sj < SPT; ++sj, ++it) {
          const int s = it % NST;
          if (!mbar_wait_bounded(&full[s], (it / NST) & 1, err)) { ok = false; break; }
          tc_fence_after();
          const int kps = kWide ? KPS : 1;
          for (int kbi = 0; kbi < kps; ++kbi) {
            const int kb = sj * kps + kbi;
            uint8_t* stg = sB + (size_t)s * kStageBytes;
            const uint64_t bdesc =
                !kWide ? sw128_desc(smem_u32(stg))
                : kbi < WB ? sw128_desc(smem_u32(stg + kbi * 1024), (uint32_t)WB * 1024u)
                           : sw128_desc(smem_u32(stg + (size_t)WB * kBlockBytes));
            const uint64_t adesc = sw128_desc(smem_u32(sA + z_block_off(Ml, kb)));
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
              mma_bf16(tmem + (uint32_t)(buf * kMT * kTileN), adesc + 2 * k4, bdesc + 2 * k4,
                       kIdesc, (kb | k4) != 0 ? 1u : 0u);
            if (kDual) {  // the second M tile, on the same stage
              const uint64_t adesc1 = sw128_desc(smem_u32(sA1 + z_block_off(Ml1, kb)));
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4)
                mma_bf16(tmem + (uint32_t)((buf * kMT + 1) * kTileN), adesc1 + 2 * k4,
                         bdesc + 2 * k4, kIdesc, (kb | k4) != 0 ? 1u : 0u);
            }
          }
          mma_commit(&empty[s]);  // the stage is free once these MMAs complete
        }
        if (!ok) break;
        mma_commit(&acc_full[buf]);
      }
      if (!ok) s_abort = 1;
      // every MMA this thread issued has completed before TMEM is freed
      mma_commit(&mma_done);
      mbar_wait_drain(&mma_done, 0, err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue --
    const int ew = warp - kEpiWarp0;     // 0 .. 7
    const int quad = warp & 3;           // the TMEM lane quadrant this warp may read
    {
      // z is written by the down-projection that precedes this grid.  Block
      // kb holds this CTA's rows m0 .. m0+Ml-1 and columns kb*64 .. +63 of z;
      // row i of a block is 128 bytes at i*128, its 16-byte chunk c stored at
      // chunk c ^ (i % 8) (the 128-byte swizzle).  Columns past r are zero.
      // Every 16-byte piece is an asynchronous copy, all of a thread's in
      // flight at once (under a full memory queue each round trip takes
      // microseconds); pieces past r are zero-filled by the copy itself.
      pdl_wait_producer();
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        const int mrows = mt == 0 ? Ml : Ml1, mbase = m0 + mt * kTileM;
        uint8_t* dstA = mt == 0 ? sA : sA1;
        const int n_items = mrows * KB * 8;  // (row i, K block, 16-byte chunk), chunk fastest
        for (int it = ew * 32 + lane; it < n_items; it += 32 * kEpiWarps) {
          const int c8 = it & 7, q = it >> 3;
          const int i = q / KB, kb = q - i * KB;
          const int k0 = kb * 64 + c8 * 8;
          const bool in = k0 < R;
          cp_async16_zfill(dstA + z_block_off(mrows, kb) + i * 128 + ((c8 ^ (i & 7)) * 16),
                           z + (size_t)(mbase + i) * R + (in ? k0 : 0), in ? 16u : 0u);
        }
      }
      cp_async_wait_all();
      fence_proxy_async_smem();  // visible to the tensor cores (async proxy)
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full);
    }
    const int half = ew / 4;                 // the 64-column half of each tile
    const int row = m0 + quad * 32 + lane;   // row of z owned by this thread (first M tile)
    const bool live = quad * 32 + lane < Ml;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const int n_sub = 2 * n_tiles;
    ResidRow rr{nullptr, 0.f, 0.f, 0.f, 1};
    if (kMode == 2 && live) rr = rrows[row];
    // greedy: each row's running best key over this thread's tiles
    constexpr bool keys = kMode == 0 && !kSample;
    unsigned long long run_key[kMT];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) run_key[mt] = 0ull;
    for (int i = 0;; ++i) {
      const int slot = i % kTileRing;
      bool ok = mbar_wait_bounded(&tile_full[slot], (i / kTileRing) & 1, err);
      const int t = ok ? *(volatile int*)&s_tile[slot] : -1;
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive(&tile_empty[slot]);
      if (!__all_sync(0xFFFFFFFFu, ok) || t < 0) break;
      const int buf = i & 1;
      // residual mode: this row's 64 target values of the tile, in flight
      // while the accumulator is computed
      float tv[kMode == 2 ? kSubW : 1];
      if (kMode == 2 && live) {
        const int v0 = t * kTileN + half * kSubW;
        if ((V & 3) == 0 && v0 + kSubW <= V) {
          const float4* tp = reinterpret_cast<const float4*>(rr.trow + v0);
#pragma unroll
          for (int j = 0; j < kSubW / 4; ++j) {
            const float4 a = __ldcs(tp + j);
            tv[4 * j] = a.x; tv[4 * j + 1] = a.y; tv[4 * j + 2] = a.z; tv[4 * j + 3] = a.w;
          }
        } else {
#pragma unroll
          for (int j = 0; j < kSubW; ++j) tv[j] = v0 + j < V ? __ldcs(rr.trow + v0 + j) : 0.f;
        }
      }
      ok = mbar_wait_bounded(&acc_full[buf], (i >> 1) & 1, err);
      if (!__all_sync(0xFFFFFFFFu, ok) || *(volatile int*)&s_abort) break;
      tc_fence_after();
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        // (dual) the second M tile's rows and accumulator
        const int row = m0 + mt * kTileM + quad * 32 + lane;
        const int mrows = mt == 0 ? Ml : Ml1;
        const bool live = quad * 32 + lane < mrows;
        const bool warp_live = quad * 32 < mrows;
        const uint32_t acc_col = (uint32_t)((buf * kMT + mt) * kTileN);
        const int h = half;
        RowState st = row_state_empty();
        if (warp_live) {
          // both 32-column loads of the sub-tile in flight, one wait
          uint32_t v2[2][32];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
            tmem_ld32_issue(tmem + lane_addr + acc_col + (uint32_t)(h * kSubW + cc * 32),
                            v2[cc]);
          tmem_ld_wait();
          if (kMode == 2) {
            // weights max(0, p - q) (mode 0) or p, and p alone, in four
            // fixed-order partial sums each
            const int vb = t * kTileN + h * kSubW;
            float r4[4] = {0.f, 0.f, 0.f, 0.f}, p4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < kSubW; ++j) {
              const float l = __uint_as_float(v2[j >> 5][j & 31]);
              const float pv = fast_exp2((tv[j] - rr.pmx) * c) * rr.pinv;
              const float w = rr.mode == 0 ? fmaxf(pv - fast_exp2((l - rr.qoff) * c), 0.f) : pv;
              const bool in = vb + j < V;
              r4[j & 3] = __fadd_rn(r4[j & 3], in ? w : 0.f);
              p4[j & 3] = __fadd_rn(p4[j & 3], in ? pv : 0.f);
            }
            st.mx = __fadd_rn(__fadd_rn(r4[0], r4[1]), __fadd_rn(r4[2], r4[3]));
            st.sum = __fadd_rn(__fadd_rn(p4[0], p4[1]), __fadd_rn(p4[2], p4[3]));
          }
#pragma unroll
          for (int cc = 0; cc < (kMode == 2 ? 0 : 2); ++cc) {
            const int col = h * kSubW + cc * 32;
            const uint32_t (&v)[32] = v2[cc];
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
        if (keys && live) {
          if (st.mx != kNegInf) {
            const unsigned long long kk = best_key(st.mx, st.arg);
            run_key[mt] = kk > run_key[mt] ? kk : run_key[mt];
          }
        } else if (kMode == 0 && live) {
          const size_t o = (size_t)row * n_sub + 2 * t + h;
          part.pmax[o] = st.mx;
          part.psum[o] = st.sum;
        }
        if (kMode == 2 && live) {
          const size_t o = (size_t)row * n_sub + 2 * t + h;
          part.pmax[o] = st.mx;   // residual mass of the sub-tile
          part.psum[o] = st.sum;  // p mass of the sub-tile
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
    if (keys) {  // this thread's rows, once: the finish reads one key per row
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        const int rw = m0 + mt * kTileM + quad * 32 + lane;
        const int mrows = mt == 0 ? Ml : Ml1;
        if (quad * 32 + lane < mrows && run_key[mt] != 0ull) atomicMax(part.best + rw, run_key[mt]);
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    // No copy may still be landing in shared memory when the CTA exits.  On
    // the normal path the MMA thread waited for every fill; after an abort it
    // stopped early, so wait for each stage's last fill (every fill has been
    // issued by now).  Not the producer's lane 0: a claim it no longer needs
    // may still be in flight there.
    if (lane == 0 && *(volatile int*)&s_abort)
      for (int s = 0; s < NST; ++s)
        if (s_fills[s] > 0) mbar_wait_drain(&full[s], (s_fills[s] - 1) & 1, err);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// ------------------------------------------------------- down-projection --
// z = bf16(h W_down^T) for many rows of h, as a split-K tcgen05 GEMM: CTA
// (tile, s) computes the 128 x 128 block of z at rows mt*128 of h and rows
// nt*128 of W_down over K slice s (KBs 64-wide K blocks, loaded whole by TMA;
// out-of-range rows and columns read as zero) into TMEM, and writes it in
// fp32 to part[s] (M x r).  k_down_reduce then sums the slices in order and
// rounds.  h and W_down are inputs, loaded while the previous library kernel
// may still run; the partials are written only after it completes (their
// workspace region may still be read by it).
constexpr int kDownThreads = 128;
constexpr int kDownMaxSlices = 32;  // K slices per block of z
__global__ void __launch_bounds__(kDownThreads, 1)
    k_down_mma(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
               int M, int r, int KBs, int n_nt, float* __restrict__ part, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;                              // KBs blocks of h
  uint8_t* sB = smem + (size_t)KBs * kBlockBytes;  // KBs blocks of W_down
  __shared__ uint64_t full, done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_ok;
  constexpr uint32_t kIdesc = idesc_bf16(kTileM, kTileN);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.y;                        // K slice
  const int mt = blockIdx.x / n_nt, nt = blockIdx.x - mt * n_nt;
  if (threadIdx.x == 0) {
    mbar_init(&full, 1);
    mbar_init(&done, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&s_tmem, kTileN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_launch_dependents();
  bool ok = true;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&full, (uint32_t)(2 * KBs * kBlockBytes));
    for (int kb = 0; kb < KBs; ++kb) {
      const int x = (s * KBs + kb) * 64;
      tma_load_2d(sA + (size_t)kb * kBlockBytes, &tm_h, x, mt * kTileM, &full);
      tma_load_2d(sB + (size_t)kb * kBlockBytes, &tm_w, x, nt * kTileN, &full);
    }
    ok = mbar_wait_bounded(&full, 0, err);
    if (ok) {
      tc_fence_after();
      for (int kb = 0; kb < KBs; ++kb) {
        const uint64_t ad = sw128_desc(smem_u32(sA + (size_t)kb * kBlockBytes));
        const uint64_t bd = sw128_desc(smem_u32(sB + (size_t)kb * kBlockBytes));
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          mma_bf16(tmem, ad + 2 * k4, bd + 2 * k4, kIdesc, (kb | k4) != 0 ? 1u : 0u);
      }
    }
    s_ok = ok ? 1 : 0;
    mma_commit(&done);  // also after an abort: every issued MMA completes first
  }
  const bool done_ok = mbar_wait_drain(&done, 0, err);
  __syncthreads();
  tc_fence_after();
  const bool all_ok = s_ok != 0 && __syncthreads_and(done_ok ? 1 : 0) != 0;
  pdl_wait_producer();
  if (all_ok) {
    // thread t holds row mt*128 + t of the block: 128 fp32 columns
    const int row = mt * kTileM + warp * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
    float* dst = part + ((size_t)s * M + row) * r + nt * kTileN;
#pragma unroll
    for (int c4 = 0; c4 < kTileN / 64; ++c4) {
      uint32_t v[2][32];
      tmem_ld32_issue(tmem + lane_addr + (uint32_t)(c4 * 64), v[0]);
      tmem_ld32_issue(tmem + lane_addr + (uint32_t)(c4 * 64 + 32), v[1]);
      tmem_ld_wait();
      if (row < M) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c0 = nt * kTileN + c4 * 64 + h * 32;
          if (c0 + 32 <= r) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(dst + c4 * 64 + h * 32 + j) =
                  make_float4(__uint_as_float(v[h][j]), __uint_as_float(v[h][j + 1]),
                              __uint_as_float(v[h][j + 2]), __uint_as_float(v[h][j + 3]));
          } else {
            for (int j = 0; j < 32; ++j)
              if (c0 + j < r) dst[c4 * 64 + h * 32 + j] = __uint_as_float(v[h][j]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    // no copy may still land in shared memory after an abort: wait (bounded)
    // for the loads once more
    if (lane == 0 && !all_ok) mbar_wait_drain(&full, 0, err);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTileN);
  }
}

// z[m, j] = RNE_bf16(sum_s part[s][m][j]), the slices added in order; also
// clears the up-projection's tile counters (as the CUDA-core down-projection
// does).  A dependent launch: it waits for the slices.
__global__ void __launch_bounds__(256)
    k_down_reduce(const float* __restrict__ part, int M, int r, int S,
                  uint16_t* __restrict__ z_ws, uint16_t* __restrict__ out_z,
                  unsigned* __restrict__ ctr, int n_ctr) {
  pdl_launch_dependents();
  pdl_wait_producer();
  if (ctr != nullptr && blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_ctr; i += blockDim.x) ctr[i] = 0u;
  const size_t n = (size_t)M * r;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    float v[kDownMaxSlices];  // every slice's load in flight, then the ordered sum
#pragma unroll
    for (int k = 0; k < kDownMaxSlices; ++k) v[k] = k < S ? __ldcg(part + (size_t)k * n + i) : 0.f;
    float a = 0.f;
#pragma unroll
    for (int k = 0; k < kDownMaxSlices; ++k)
      if (k < S) a = __fadd_rn(a, v[k]);
    const uint16_t bits = f32_to_bf16_bits(a);
    z_ws[i] = bits;
    if (out_z) out_z[i] = bits;
  }
}

// ------------------------------------------------------------------ finish --
// Fixed-order block reductions over the 256 threads of the finish.
// Maximum over the block; every thread gets it (sh: one float per warp).
__device__ __forceinline__ float block_max(float x, float* sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
  if (lane == 0) sh[warp] = x;
  __syncthreads();
  float r = sh[0];
#pragma unroll
  for (int w = 1; w < kFinThreads / 32; ++w) r = fmaxf(r, sh[w]);
  return r;
}

// One group of 64 16-byte chunks of K for rows 8w .. 8w+7 of a 64-row
// sub-tile starting at v0 (n live rows): every load issued up front, then the
// bf16 products accumulated in chunk order into acc.
__device__ __forceinline__ void recompute_group(const uint8_t* __restrict__ w_up,
                                                const uint8_t* __restrict__ z, int m, int r,
                                                int v0, int n, int nch, int c0, int warp,
                                                int lane, float (&acc)[8]) {
  uint4 zc[2], wv[8][2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int ch = c0 + lane + 32 * q;
    zc[q] = ch < nch ? __ldg(reinterpret_cast<const uint4*>(z + ((size_t)m * r + ch * 8) * 2))
                     : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int ii = 0; ii < 8; ++ii) {
    const int i = warp * 8 + ii;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int ch = c0 + lane + 32 * q;
      wv[ii][q] = (i < n && ch < nch) ? __ldg(reinterpret_cast<const uint4*>(
                                            w_up + ((size_t)(v0 + i) * r + ch * 8) * 2))
                                      : make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int ii = 0; ii < 8; ++ii) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t ww[4] = {wv[ii][q].x, wv[ii][q].y, wv[ii][q].z, wv[ii][q].w};
      const uint32_t zz[4] = {zc[q].x, zc[q].y, zc[q].z, zc[q].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[ii] = fma_bf16_lo(ww[e], zz[e], acc[ii]);
        acc[ii] = fma_bf16_hi(ww[e], zz[e], acc[ii]);
      }
    }
  }
}

// Greedy: one thread per row of z reads the row's best key (the maximum and
// its lowest vocabulary id, reduced by the up-projection) and writes the
// outputs.  Sampling: one CTA of 8 warps per row.  Warp w owns a contiguous
// run of 32 * per sub-tile partials (per <= kPer, the register arrays' size:
// 8, 16 or kFinPer, the smallest that holds per), lane-interleaved and
// loaded once into registers (all loads of the CTA in flight together): the
// maximum g, the masses psum_s 2^((pmax_s - g)c), each warp's total over its
// chunks of 32 in vocabulary order, the warp totals in order, and the warp
// whose run holds the crossing of u * W walks its chunks to the sub-tile; the
// 8 warps then recompute that sub-tile's logits (8 rows each, every load
// issued up front, CUDA-core fp32 accumulation of the same bf16 products) and
// warp 0 walks them in row order.
// (88 registers: the default allocation for 256 threads spilled a value;
// 88 x 256 still leaves room beside an up-projection CTA on the same SM)
template <bool kSample, int kPer>
__global__ void __maxnreg__(88)
    k_head_mma_finish(const uint8_t* __restrict__ w_up, const uint8_t* __restrict__ z, int M,
                      int r, int V, float c, float inv_t, int n_sub, MmaPart part,
                      HeadOutputs out) {
  __shared__ float s_logit[kSubW];
  __shared__ float s_max[kFinThreads / 32];
  __shared__ float s_wsum[kFinThreads / 32];
  __shared__ float s_f[2];  // W, residual mass inside the chosen sub-tile
  __shared__ int s_sid;     // chosen sub-tile
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = kSample ? (int)blockIdx.x : (int)(blockIdx.x * blockDim.x + threadIdx.x);
  pdl_launch_dependents();  // the next call's down-projection may start reading
  // an input (or the counter-based stream): read before the wait
  const float u = (kSample && m < M) ? draw_uniform(out.draws.uniforms, out.draws.seed,
                                                    out.draws.offset, m, 0, 1)
                                     : 0.f;
  pdl_wait_producer();
  if (m >= M) return;
  if (!kSample) {
    write_greedy(out, V, m, __ldcg(part.best + m));
    return;
  }
  // Warp w owns the run of sub-tiles [w*32*per, (w+1)*32*per), lane l its
  // elements l + 32k (k < per): each load of a warp is 128 contiguous bytes,
  // and the run is scanned chunk by chunk of 32 in vocabulary order.
  const int per = (n_sub + kFinThreads - 1) / kFinThreads;
  const int wbase = warp * 32 * per;
  const float* pm = part.pmax + (size_t)m * n_sub;
  const float* ps = part.psum + (size_t)m * n_sub;
  float vmx[kPer], vsm[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int e = wbase + 32 * k + lane;
    const bool in = k < per && e < n_sub;
    vmx[k] = in ? __ldcg(pm + e) : kNegInf;
    vsm[k] = in ? __ldcg(ps + e) : 0.f;
  }
  float lmax = kNegInf;
#pragma unroll
  for (int k = 0; k < kPer; ++k) lmax = fmaxf(lmax, vmx[k]);
  const float gmax = block_max(lmax, s_max);
  // the masses, and each chunk's total as a butterfly sum (every lane gets
  // the same value; the chunks' sums are independent and overlap)
  float tk[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    vsm[k] = vsm[k] * fast_exp2((vmx[k] - gmax) * c);  // 0 past the run (0 * 2^-inf)
    tk[k] = vsm[k];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int k = 0; k < kPer; ++k) tk[k] = __fadd_rn(tk[k], __shfl_xor_sync(0xFFFFFFFFu, tk[k], o));
  float wtot = 0.f;  // the chunk totals in order (those past the run are 0)
#pragma unroll
  for (int k = 0; k < kPer; ++k) wtot = __fadd_rn(wtot, tk[k]);
  if (lane == 0) s_wsum[warp] = wtot;
  __syncthreads();
  // every thread: W, this warp's offset, and the crossing warp -- the first
  // whose inclusive total passes u * W, else (the target at the very top
  // after rounding) the last one with mass
  float W = 0.f, woff = 0.f;
#pragma unroll
  for (int w = 0; w < kFinThreads / 32; ++w) W = __fadd_rn(W, s_wsum[w]);
  const float target = u * W;
  int cw = -1, lastw = 0;
  {
    float run = 0.f;
#pragma unroll
    for (int w = 0; w < kFinThreads / 32; ++w) {
      const float t = s_wsum[w], nxt = __fadd_rn(run, t);
      if (w == warp) woff = run;
      if (t > 0.f && cw < 0) {
        if (nxt > target) cw = w;
        else lastw = w;
      }
      run = nxt;
    }
  }
  if (cw < 0) cw = lastw;
  if (warp == cw) {
    // the chunk whose running total passes the target, else (rounding) the
    // last chunk with mass; then, in it, the first element whose running
    // total passes, else the last element with mass
    float cum = woff, before_c = woff, last_c = woff;
    int kc = -1, klast = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const float nxt = __fadd_rn(cum, tk[k]);
      if (tk[k] > 0.f && kc < 0) {
        if (nxt > target) {
          kc = k;
          before_c = cum;
        } else {
          klast = k;
          last_c = cum;
        }
      }
      cum = nxt;
    }
    const bool top = kc < 0;
    if (top) {
      kc = klast;
      before_c = last_c;
    }
    float mk = 0.f;
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if (k == kc) mk = vsm[k];
    const float incl = warp_incl_scan(mk, lane);
    const float up = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
    const float ce = lane > 0 ? __fadd_rn(before_c, up) : before_c;
    const unsigned pos = __ballot_sync(0xFFFFFFFFu, mk > 0.f);
    const unsigned hit =
        __ballot_sync(0xFFFFFFFFu, mk > 0.f && __fadd_rn(before_c, incl) > target) & (top ? 0u : ~0u);
    const int l = hit ? __ffs(hit) - 1 : pos ? 31 - __clz(pos) : 0;
    const float before = __shfl_sync(0xFFFFFFFFu, ce, l);
    if (lane == 0) {
      s_f[0] = W;
      s_f[1] = target - before;
      s_sid = min(wbase + 32 * kc + l, n_sub - 1);
    }
  }
  __syncthreads();
  const float resid = s_f[1];
  const int v0 = s_sid * kSubW;
  const int n = max(0, min(kSubW, V - v0));
  // recompute: warp w takes rows 8w .. 8w+7 of the sub-tile, lanes over K in
  // groups of 64 16-byte chunks (every load of a group issued up front); one
  // group (r <= 512) as straight-line code
  const int nch = r / 8;
  float acc[8];
#pragma unroll
  for (int ii = 0; ii < 8; ++ii) acc[ii] = 0.f;
  if (nch <= 64) {
    recompute_group(w_up, z, m, r, v0, n, nch, 0, warp, lane, acc);
  } else {
    for (int c0 = 0; c0 < nch; c0 += 64)
      recompute_group(w_up, z, m, r, v0, n, nch, c0, warp, lane, acc);
  }
#pragma unroll
  for (int ii = 0; ii < 8; ++ii) {
    const float a = warp_sum_fixed(acc[ii]);
    if (lane == 0) s_logit[warp * 8 + ii] = a;
  }
  __syncthreads();
  if (warp != 0) return;
  float cum = 0.f;
  int tok = -1, lastp2 = -1;
#pragma unroll
  for (int h = 0; h < kSubW; h += 32) {
    const int i = h + lane;
    const float wv1 = i < n ? fast_exp2((s_logit[i] - gmax) * c) : 0.f;
    const float csum = __fadd_rn(cum, warp_incl_scan(wv1, lane));
    const unsigned pos = __ballot_sync(0xFFFFFFFFu, wv1 > 0.f);
    const unsigned hitm = __ballot_sync(0xFFFFFFFFu, wv1 > 0.f && csum > resid);
    if (tok < 0 && hitm) tok = h + __ffs(hitm) - 1;
    if (pos) lastp2 = h + 31 - __clz(pos);
    cum = __shfl_sync(0xFFFFFFFFu, csum, 31);
  }
  if (tok < 0) tok = lastp2 < 0 ? 0 : lastp2;
  if (lane == 0) {
    const float lW = logf(s_f[0]);
    out.tokens[m] = out.id_map != nullptr ? out.id_map[v0 + tok] : v0 + tok;
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

// The same bf16 tensor [rows x cols] seen as 4-D (64 columns, 8 rows, the
// cols/64 full K blocks, rows/8 row groups) for the wide stages: a box
// {64, 8, wb, 16} is 128 rows x wb K blocks, landing as 16 groups x wb K blocks
// x 8 rows x 128 B.  Needs rows % 8 == 0 (every element of an in-range group
// exists); groups past the end read as zero.
bool make_map_wide(CUtensorMap* map, const void* base, int rows, int cols, int wb) {
  EncodeTiledFn enc = encoder();
  if (!enc || rows % 8 != 0 || wb < 1 || wb > cols / 64) return false;
  const cuuint64_t dims[4] = {64, 8, (cuuint64_t)(cols / 64), (cuuint64_t)(rows / 8)};
  const cuuint64_t strides[3] = {(cuuint64_t)cols * 2, 128, (cuuint64_t)cols * 16};
  const cuuint32_t box[4] = {64, 8, (cuuint32_t)wb, (cuuint32_t)(kTileN / 8)};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

MmaPlan mma_plan(int r, int M, int V) {
  MmaPlan p{};
  p.ok = false;
  if (M <= 0 || M > 2 * kTileM || r % 8 != 0 || r > 4096) return p;
  p.mt = M <= kTileM ? 1 : 2;  // M tiles, one per CTA
  p.kb = (r + 63) / 64;
  const int a_bytes = z_bytes(std::min(M, kTileM), p.kb);  // the largest CTA's z
  const int room = kSmemCap - 1024 - a_bytes;
  // wide stages (several K blocks per request run of each row) when the 4-D
  // view is exact (V % 8 == 0) and z leaves room for two of them: 4 K blocks
  // when r is a multiple of 256; else a whole tile of up to 6 K blocks (the
  // full ones by 4-D box, a ragged last one by 2-D box); else, when r is a
  // multiple of 64, the largest count of 5 .. 2 full K blocks that divides
  // the tile
  p.kps = 1;
  p.wb = 0;
  if (V % 8 == 0) {
    if (r % 256 == 0 && room / (4 * kBlockBytes) >= 2) {
      p.kps = 4;
      p.wb = 4;
    } else if (p.kb <= 6 && r >= 64 && room / (p.kb * kBlockBytes) >= 2) {
      p.kps = p.kb;
      p.wb = r / 64;
    } else if (r % 64 == 0) {
      for (int k = 5; k >= 2; --k)
        if (p.kb % k == 0 && room / (k * kBlockBytes) >= 2) {
          p.kps = k;
          p.wb = k;
          break;
        }
    }
  }
  const int stage = p.kps * kBlockBytes;
  p.nst = std::min(p.kps > 1 ? 4 : kMaxStages, room / stage);
  if (p.nst < (p.kps > 1 ? 2 : 3)) return p;
  p.smem = 1024 + a_bytes + p.nst * stage;
  p.n_tiles = (V + kTileN - 1) / kTileN;
  p.grid = p.mt * std::max(1, std::min(sm_count() / p.mt, p.n_tiles));
  p.n_sub = 2 * p.n_tiles;
  if (p.n_sub > kFinThreads * kFinPer) return p;  // V > 786432: beyond the finish's registers
  p.ok = true;
  return p;
}

// Both M tiles of z in every CTA (softmax partials, 128 < M <= 256), with 2-D
// W_up stages in the room left: chosen when at least four stages fit.
MmaPlan mma_plan_dual(int r, int M, int V) {
  MmaPlan p{};
  p.ok = false;
  if (M <= kTileM || M > 2 * kTileM || r % 8 != 0 || r > 4096) return p;
  p.mt = 1;  // one tile counter; each CTA takes both M tiles of every tile it draws
  p.dual = true;
  p.kb = (r + 63) / 64;
  const int a_bytes = z_bytes(kTileM, p.kb) + z_bytes(M - kTileM, p.kb);
  const int room = kSmemCapDual - 1024 - a_bytes;
  p.kps = 1;
  p.wb = 0;
  if (V % 8 == 0 && r % 128 == 0 && room >= 2 * 2 * kBlockBytes) {
    p.kps = 2;  // stages of two K blocks: 256 contiguous bytes of each row per request run
    p.wb = 2;
  }
  const int stage = p.kps * kBlockBytes;
  p.nst = room > 0 ? std::min(p.kps > 1 ? 4 : kMaxStages, room / stage) : 0;
  if (p.nst < (p.kps > 1 ? 2 : 4)) return p;
  p.smem = 1024 + a_bytes + p.nst * stage;
  p.n_tiles = (V + kTileN - 1) / kTileN;
  p.grid = std::max(1, std::min(sm_count(), p.n_tiles));
  p.n_sub = 2 * p.n_tiles;
  if (p.n_sub > kFinThreads * kFinPer) return p;
  p.ok = true;
  return p;
}

template <bool kSample, int kMode, bool kWide, bool kDual = false>
static cudaError_t launch_mma_kps(const MmaPlan& p, const void* z, const CUtensorMap& tw,
                                  const CUtensorMap& tw2, int M, int r, int V, float c,
                                  const MmaPart& part, float* scores, unsigned* ctr,
                                  cudaStream_t st, KernelKind kind,
                                  const ResidRow* rrows = nullptr) {
  auto kern = k_head_mma<kSample, kMode, kWide, kDual>;
  // the limit is set once per kernel: make it the largest size any plan asks for
  cudaError_t e =
      set_smem_once(reinterpret_cast<const void*>(kern), kDual ? kSmemCapDual : kSmemCap);
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
  ProfScope ps(kind, st);
  return cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const uint16_t*>(z), tw, tw2, M, p.mt, r,
                            V, p.kb, p.kps, p.wb, p.nst, c, p.n_tiles, part, scores, rrows, ctr,
                            error_word());
}
template <bool kSample, int kMode>
static cudaError_t launch_mma_one(const MmaPlan& p, const void* z, const CUtensorMap& tw,
                                  const CUtensorMap& tw2, int M, int r, int V, float c,
                                  const MmaPart& part, float* scores, unsigned* ctr,
                                  cudaStream_t st, KernelKind kind,
                                  const ResidRow* rrows = nullptr) {
  if (p.kps > 1)
    return launch_mma_kps<kSample, kMode, true>(p, z, tw, tw2, M, r, V, c, part, scores, ctr, st,
                                                 kind, rrows);
  return launch_mma_kps<kSample, kMode, false>(p, z, tw, tw2, M, r, V, c, part, scores, ctr, st,
                                                kind, rrows);
}

// The two tensor maps of W_up a plan needs: tw for the stages (2-D, or 4-D for
// wide stages), tw2 the 2-D map for a wide stage's ragged last K block.
static bool make_maps(const MmaPlan& p, const void* w_up, int V, int r, CUtensorMap* tw,
                      CUtensorMap* tw2) {
  if (!make_map(tw2, w_up, V, r)) return false;
  if (p.kps > 1 && p.wb > 0) return make_map_wide(tw, w_up, V, r, p.wb);
  *tw = *tw2;
  return true;
}

DownMmaPlan down_mma_plan(int M, int d, int r, size_t part_cap) {
  DownMmaPlan p{};
  p.ok = false;
  if (M <= 0 || r <= 0 || d % 8 != 0 || r % 8 != 0) return p;
  p.n_mt = (M + kTileM - 1) / kTileM;
  p.n_nt = (r + kTileN - 1) / kTileN;
  const int tiles = p.n_mt * p.n_nt;
  const int KB = (d + 63) / 64;
  for (int S = std::max(1, std::min(std::min(KB, kDownMaxSlices), 128 / tiles)); S >= 1; --S) {
    const int kbs = (KB + S - 1) / S;
    const int s2 = (KB + kbs - 1) / kbs;  // no empty slices
    if (kbs <= 6 && (size_t)s2 * M * r * sizeof(float) <= part_cap) {
      p.S = s2;
      p.kbs = kbs;
      p.smem = 1024 + 2 * kbs * kBlockBytes;
      p.ok = true;
      return p;
    }
  }
  return p;
}

cudaError_t launch_down_mma(const DownMmaPlan& p, const void* h, const void* w_down, int M, int d,
                            int r, float* part, void* z_ws, void* out_z, unsigned* ctr, int n_ctr,
                            cudaStream_t st) {
  CUtensorMap th, tw;
  if (!make_map(&th, h, M, d) || !make_map(&tw, w_down, r, d)) return cudaErrorInvalidValue;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(k_down_mma), kSmemCap);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.n_mt * p.n_nt), (unsigned)p.S);
  cfg.blockDim = dim3(kDownThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  {
    ProfScope ps(kKDownProj, st);
    e = cudaLaunchKernelEx(&cfg, k_down_mma, th, tw, M, r, p.kbs, p.n_nt, part, error_word());
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cr = {};
  const long long n = (long long)M * r;
  cr.gridDim = dim3((unsigned)std::max<long long>(1, std::min<long long>((n + 255) / 256,
                                                                        4LL * sm_count())));
  cr.blockDim = dim3(256);
  cr.stream = st;
  cr.attrs = attr;
  cr.numAttrs = 1;
  ProfScope ps(kKDownReduce, st);
  e = cudaLaunchKernelEx(&cr, k_down_reduce, (const float*)part, M, r, p.S, (uint16_t*)z_ws,
                         (uint16_t*)out_z, ctr, n_ctr);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_head_mma_resid(const MmaPlan& p, const void* z, const void* w_up, int B,
                                  int r, int V, float temperature, const ResidRow* rows,
                                  float* rmass, float* pmass, unsigned* ctr, cudaStream_t st) {
  if (B <= 0) return cudaSuccess;
  CUtensorMap tw, tw2;
  if (!make_maps(p, w_up, V, r, &tw, &tw2)) return cudaErrorInvalidValue;
  const float c = (float)(1.4426950408889634 / (double)temperature);
  const MmaPart part{rmass, pmass, nullptr};
  const cudaError_t e = launch_mma_one<false, 2>(p, z, tw, tw2, B, r, V, c, part, nullptr, ctr,
                                                 st, kKVerifyQRow, rows);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_head_mma(const MmaPlan& p, const void* z_ws, const void* w_up, int M, int r,
                            int V, float temperature, const MmaWork& w, const HeadOutputs& out,
                            float* scores, unsigned* ctr, cudaStream_t st, KernelKind kind) {
  if (M <= 0) return cudaSuccess;
  // tw: the stages' map (2-D, or 4-D for wide stages); tw2: the 2-D map, for
  // a wide stage's ragged last K block
  CUtensorMap tw, tw2;
  if (!make_map(&tw2, w_up, V, r)) return cudaErrorInvalidValue;
  if (p.kps > 1 && p.wb > 0) {
    if (!make_map_wide(&tw, w_up, V, r, p.wb)) return cudaErrorInvalidValue;
  } else {
    tw = tw2;
  }
  const bool sample = temperature > 0.f && scores == nullptr;
  const double inv = sample ? 1.0 / (double)temperature : 0.0;
  const float c = (float)(1.4426950408889634 * inv), inv_t = (float)inv;
  // a greedy head reduces into the rows' best keys
  if (!sample && scores == nullptr && w.best == nullptr) return cudaErrorInvalidValue;
  const MmaPart part{w.pmax, w.psum, w.best};
  cudaError_t e;
  if (scores != nullptr) {
    e = launch_mma_one<false, 1>(p, z_ws, tw, tw2, M, r, V, c, part, scores, ctr, st, kind);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  // both M tiles in every CTA when they and four stages fit (128 < M <= 256)
  const MmaPlan pd = M > kTileM ? mma_plan_dual(r, M, V) : MmaPlan{};
  if (pd.ok) {
    CUtensorMap dw, dw2;
    if (!make_maps(pd, w_up, V, r, &dw, &dw2)) return cudaErrorInvalidValue;
    if (pd.kps > 1)
      e = sample ? launch_mma_kps<true, 0, true, true>(pd, z_ws, dw, dw2, M, r, V, c, part,
                                                       nullptr, ctr, st, kind)
                 : launch_mma_kps<false, 0, true, true>(pd, z_ws, dw, dw2, M, r, V, c, part,
                                                        nullptr, ctr, st, kind);
    else
      e = sample ? launch_mma_kps<true, 0, false, true>(pd, z_ws, dw, dw2, M, r, V, c, part,
                                                        nullptr, ctr, st, kind)
                 : launch_mma_kps<false, 0, false, true>(pd, z_ws, dw, dw2, M, r, V, c, part,
                                                         nullptr, ctr, st, kind);
  } else if (sample) {
    e = launch_mma_one<true, 0>(p, z_ws, tw, tw2, M, r, V, c, part, nullptr, ctr, st, kind);
  } else {
    e = launch_mma_one<false, 0>(p, z_ws, tw, tw2, M, r, V, c, part, nullptr, ctr, st, kind);
  }
  if (e != cudaSuccess) return e;
  // the per-row finish, launched to overlap the tail of the MMA grid: a CTA
  // per row when sampling, a thread per row when greedy
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sample ? M : (M + 31) / 32);
  cfg.blockDim = dim3(sample ? kFinThreads : 32);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ProfScope ps(kKHeadFinish, st);
  const int per = (p.n_sub + kFinThreads - 1) / kFinThreads;  // <= kFinPer (the plan checks)
  if (!sample)
    e = cudaLaunchKernelEx(&cfg, k_head_mma_finish<false, 8>, (const uint8_t*)w_up,
                           (const uint8_t*)z_ws, M, r, V, c, inv_t, p.n_sub, part, out);
  else if (per <= 8)
    e = cudaLaunchKernelEx(&cfg, k_head_mma_finish<true, 8>, (const uint8_t*)w_up,
                           (const uint8_t*)z_ws, M, r, V, c, inv_t, p.n_sub, part, out);
  else if (per <= 16)
    e = cudaLaunchKernelEx(&cfg, k_head_mma_finish<true, 16>, (const uint8_t*)w_up,
                           (const uint8_t*)z_ws, M, r, V, c, inv_t, p.n_sub, part, out);
  else
    e = cudaLaunchKernelEx(&cfg, k_head_mma_finish<true, kFinPer>, (const uint8_t*)w_up,
                           (const uint8_t*)z_ws, M, r, V, c, inv_t, p.n_sub, part, out);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace ss
