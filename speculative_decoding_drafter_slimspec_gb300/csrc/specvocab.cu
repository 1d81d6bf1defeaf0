// specvocab.cu -- SpecVocab-style dynamic-vocabulary head on sm_103a.
//
// SpecVocab write-up (动态词汇推测加速大语言模型推理), sections 2.2.1-2.2.3:
//   h' = bf16(W_down h)        (k_down_proj, shared with the low-rank head)
//   s  = W_vocab h'            (the head's tcgen05 up-projection in its scores
//                              mode, or the CUDA-core stream when it does not fit)
//   K  = topk(s, k)            k_topk: a cluster of CTAs per row filters the
//                              row against a sampled threshold; radix select
//                              on order-preserving keys, ties to the lowest
//                              id, ordered compaction
//   z' = U[K] h                k_gather_logits: a warp per candidate row of U
//                              (8 KB at d = 4096), h in shared memory; CTAs
//                              of 8 candidates dispatched in candidate order,
//                              so rows picked by several sequences are read
//                              from DRAM about once
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
// Keys are order-preserving uint32 images of the fp32 scores (float_key), so
// "largest scores" = "largest keys", and ties are broken by the lowest id.
constexpr int kTopkThreads = 1024;
constexpr int kTopkCap = 8192;     // candidate buffer (keys + ids) in shared memory
constexpr int kTopkSample = 8192;  // sampled scores that estimate the threshold

struct KeysFromScores {  // the row's scores, read from global memory
  const float* s;
  __device__ bool live(int) const { return true; }
  __device__ uint32_t operator()(int i) const { return float_key(s[i]); }
};
struct KeysInShared {
  const uint32_t* k;
  __device__ bool live(int) const { return true; }
  __device__ uint32_t operator()(int i) const { return k[i]; }
};

// Key T of the q-th largest of n keys (1 <= q <= n) and `need`, how many of
// the keys equal to T are among the q largest.  Three histogram passes over
// digits of 11, 11 and 10 bits, most significant first; every thread of the
// block calls it.  With passes = 2 it stops after 22 bits: T is then the
// lowest key sharing the q-th largest key's top 22 bits (a lower bound of
// it; `need` is not meaningful).
template <class Keys>
__device__ void block_select_desc(const Keys& key_at, int n, int q, int* hist, int* s_warp,
                                  int* s_sel, uint32_t& thr, int& need, int passes = 3) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0, pmask = 0;
  need = q;
#pragma unroll 1
  for (int pass = 0; pass < passes; ++pass) {
    const int nb = pass < 2 ? 2048 : 1024;
    const int shift = pass == 0 ? 21 : pass == 1 ? 10 : 0;
    for (int i = tid; i < 2048; i += kTopkThreads) hist[i] = 0;
    if (tid == 0) { s_sel[0] = 0; s_sel[1] = 0; }
    __syncthreads();
    for (int i = tid; i < n; i += kTopkThreads) {
      if (!key_at.live(i)) continue;
      const uint32_t key = key_at(i);
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1);
    }
    __syncthreads();
    // thread t owns bins nb-1-t*bpt-i (i < bpt): descending bin order
    const int bpt = nb / kTopkThreads;
    int local = 0;
    for (int i = 0; i < bpt; ++i) local += hist[nb - 1 - tid * bpt - i];
    const int incl = block_scan_incl_1024(local, s_warp);
    const int excl = incl - local;
    if (excl < need && incl >= need) {
      int cum = excl;
      for (int i = 0; i < bpt; ++i) {
        const int bin = nb - 1 - tid * bpt - i;
        if (cum + hist[bin] >= need) {
          s_sel[0] = bin;
          s_sel[1] = cum;
          break;
        }
        cum += hist[bin];
      }
    }
    __syncthreads();
    need -= s_sel[1];
    prefix |= (uint32_t)s_sel[0] << shift;
    pmask |= (uint32_t)(nb - 1) << shift;
    __syncthreads();
  }
  thr = prefix;
}

// Ordered compaction of n keys against (thr, need): every key above thr and
// the first `need` keys equal to it, in index order.  Warp w owns a
// contiguous segment of entries and walks it 32 at a time (coalesced reads);
// ballots rank the kept entries of a step, so the output is in index order.
template <class Keys, class Ids>
__device__ void block_compact(const Keys& key_at, const Ids& id_at, int n, uint32_t thr, int need,
                              int k, int* s_cnt, int32_t* out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int segw = ((n + 1023) / 1024) * 32;  // entries per warp, a multiple of 32
  const int lo = min(n, warp * segw), hi = min(n, lo + segw);
  const unsigned lt = (1u << lane) - 1u;
  int gt = 0, eq = 0;
  for (int v0 = lo; v0 < hi; v0 += 32) {
    const int v = v0 + lane;
    const uint32_t key = v < hi ? key_at(v) : 0u;
    gt += __popc(__ballot_sync(0xFFFFFFFFu, v < hi && key > thr));
    eq += __popc(__ballot_sync(0xFFFFFFFFu, v < hi && key == thr));
  }
  if (lane == 0) { s_cnt[warp] = gt; s_cnt[32 + warp] = eq; }
  __syncthreads();
  int gt_pre = 0, eq_pre = 0;
  for (int w = 0; w < warp; ++w) { gt_pre += s_cnt[w]; eq_pre += s_cnt[32 + w]; }
  __syncthreads();
  int pos = gt_pre + min(eq_pre, need), eq_seen = eq_pre;
  for (int v0 = lo; v0 < hi; v0 += 32) {
    const int v = v0 + lane;
    const uint32_t key = v < hi ? key_at(v) : 0u;
    const bool is_gt = v < hi && key > thr, is_eq = v < hi && key == thr;
    const unsigned eqb = __ballot_sync(0xFFFFFFFFu, is_eq);
    const bool keep = is_gt || (is_eq && eq_seen + __popc(eqb & lt) < need);
    const unsigned kb = __ballot_sync(0xFFFFFFFFu, keep);
    const int my = pos + __popc(kb & lt);
    if (keep && my < k) out[my] = id_at(v);
    pos += __popc(kb);
    eq_seen += __popc(eqb);
  }
}
// The region buffer: 32 per-warp regions of kTopkRegion entries each.
constexpr int kTopkRegion = kTopkCap / 32;

struct IdSelf {
  __device__ int32_t operator()(int i) const { return i; }
};
struct IdInShared {
  const int32_t* id;
  __device__ int32_t operator()(int i) const { return id[i]; }
};

// Clusters: rank and size of this CTA in its cluster, the cluster-wide
// barrier (release / acquire: shared-memory writes before it, local or
// remote, are visible after it), and loads / stores to another CTA's shared
// memory at the address of a local object.
__device__ __forceinline__ int cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return (int)r;
}
__device__ __forceinline__ int cluster_size() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return (int)r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_addr(const void* local, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_cluster(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// One cluster of C CTAs (1024 threads each) per row; CTA rank j takes the
// j-th of C equal id ranges of the row.
//   1. A threshold t: the key of rank ~1.25 k V / S in a strided sample of S
//      scores (exact rank k when the sample is the whole row); every CTA of
//      the cluster computes the same one.
//   2. One ordered pass over the CTA's range keeps every score with key >= t,
//      in id order, in per-warp regions of a shared buffer.
//   3. After a cluster barrier every CTA writes its candidates, in id order,
//      into the first CTA's compact buffer (CTAs in rank order, warps in
//      order), through distributed shared memory.
//   4. The first CTA selects exactly among them: they hold the k largest
//      whenever there are at least k of them, so the result is the full
//      row's; otherwise (or when a region or the compact buffer would
//      overflow) it selects over the whole row instead.
__global__ void __launch_bounds__(kTopkThreads) k_topk(const float* __restrict__ scores, int V,
                                                       int k, int32_t* __restrict__ out_idx) {
  extern __shared__ uint32_t s_dyn[];
  uint32_t* c_key = s_dyn;                                         // kTopkCap keys (regions)
  int32_t* c_id = reinterpret_cast<int32_t*>(s_dyn + kTopkCap);    // kTopkCap ids (regions)
  uint32_t* a_key = s_dyn + 2 * kTopkCap;                          // compact keys (first CTA)
  int32_t* a_id = reinterpret_cast<int32_t*>(s_dyn + 3 * kTopkCap);  // compact ids
  __shared__ int hist[2048];
  __shared__ int s_warp[32];
  __shared__ int s_sel[2];
  __shared__ int s_reg[32];     // candidates kept per warp region
  __shared__ int s_over;        // a region of this CTA overflowed
  __shared__ int s_all[8 * 32]; // every CTA's region counts, CTAs in rank order
  __shared__ int s_any;         // an overflow anywhere in the cluster
  const int C = cluster_size(), rank = cluster_rank();
  const int row = blockIdx.x / C, tid = threadIdx.x;
  const float* s = scores + (size_t)row * V;
  int32_t* out = out_idx + (size_t)row * k;
  const KeysFromScores row_keys{s};

  // 1. the threshold from the sample (held in the region buffer for now):
  //    S scores in blocks of 32 consecutive ones spread evenly over the row
  const int S = min(V, kTopkSample);
  const int lane = tid & 31, warp = tid >> 5;
  if (S == V) {
    for (int i = tid; i < S; i += kTopkThreads) c_key[i] = float_key(s[i]);
  } else {
    // kTopkSample / 32 = 256 blocks, 8 per warp, all loads in flight together
    constexpr int kNblk = kTopkSample / 32, kPerWarp = kNblk / (kTopkThreads / 32);
    float sv[kPerWarp];
#pragma unroll
    for (int j = 0; j < kPerWarp; ++j) {
      const int b = warp + j * (kTopkThreads / 32);
      sv[j] = s[(int)(((long long)b * (V - 32)) / (kNblk - 1)) + lane];
    }
#pragma unroll
    for (int j = 0; j < kPerWarp; ++j)
      c_key[(warp + j * (kTopkThreads / 32)) * 32 + lane] = float_key(sv[j]);
  }
  __syncthreads();
  int q = k;
  if (S < V) q = min(S, (int)((5LL * k * S + 4LL * V - 1) / (4LL * V)) + 8);
  uint32_t t_low;
  int unused;
  // (two passes: a threshold at or below the sampled rank is all step 2 needs)
  block_select_desc(KeysInShared{c_key}, S, q, hist, s_warp, s_sel, t_low, unused, 2);

  // 2. (the sample's keys are no longer read: block_select_desc ended on a
  //    barrier) one pass over this CTA's ids: warp w walks a contiguous
  //    segment, 16 loads in flight per lane, and appends the scores with
  //    key >= t, in id order, to region w of the buffer
  if (tid == 0) s_over = 0;
  const int part = (V + C - 1) / C;
  const int p_lo = min(V, rank * part), p_hi = min(V, p_lo + part);
  const int segw = ((p_hi - p_lo + 1023) / 1024) * 32;
  const int lo = min(p_hi, p_lo + warp * segw), hi = min(p_hi, lo + segw);
  const unsigned lt = (1u << lane) - 1u;
  int cnt = 0;
  constexpr int kDepth = 16;
  for (int b0 = lo; b0 < hi; b0 += 32 * kDepth) {
    float x[kDepth];
#pragma unroll
    for (int j = 0; j < kDepth; ++j) {
      const int v = b0 + 32 * j + lane;
      x[j] = v < hi ? s[v] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kDepth; ++j) {
      const int v = b0 + 32 * j + lane;
      const uint32_t key = float_key(x[j]);
      const bool keep = v < hi && key >= t_low;
      const unsigned kb = __ballot_sync(0xFFFFFFFFu, keep);
      const int my = cnt + __popc(kb & lt);
      if (keep && my < kTopkRegion) {
        c_key[warp * kTopkRegion + my] = key;
        c_id[warp * kTopkRegion + my] = v;
      }
      cnt += __popc(kb);
    }
  }
  __syncthreads();
  if (lane == 0) {
    s_reg[warp] = min(cnt, kTopkRegion);
    if (cnt > kTopkRegion) s_over = 1;
  }
  cluster_barrier();  // every CTA's regions and counts are final

  // 3. every CTA's counts (CTAs in rank order), then this CTA's candidates into
  //    the first CTA's compact buffer
  if (tid == 0) s_any = 0;
  __syncthreads();
  if (tid < C * 32) s_all[tid] = (int)ld_cluster(cluster_addr(&s_reg[tid & 31], tid >> 5));
  if (tid < C && ld_cluster(cluster_addr(&s_over, tid)) != 0u) atomicOr(&s_any, 1);
  __syncthreads();
  int base = 0, n_c = 0;
  for (int i = 0; i < C * 32; ++i) {
    if (i < rank * 32 + warp) base += s_all[i];
    n_c += s_all[i];
  }
  const bool ok = s_any == 0 && n_c >= k && n_c <= kTopkCap;
  if (ok) {
    const uint32_t dk = cluster_addr(a_key, 0), di = cluster_addr(a_id, 0);
    for (int i = lane; i < s_reg[warp]; i += 32) {
      st_cluster(dk + 4u * (uint32_t)(base + i), c_key[warp * kTopkRegion + i]);
      st_cluster(di + 4u * (uint32_t)(base + i), (uint32_t)c_id[warp * kTopkRegion + i]);
    }
  }
  cluster_barrier();  // the first CTA's compact buffer is complete
  if (rank != 0) return;

  // 4. exact selection
  uint32_t thr;
  int need;
  if (ok) {
    block_select_desc(KeysInShared{a_key}, n_c, k, hist, s_warp, s_sel, thr, need);
    block_compact(KeysInShared{a_key}, IdInShared{a_id}, n_c, thr, need, k, hist, out);
  } else {
    block_select_desc(row_keys, V, k, hist, s_warp, s_sel, thr, need);
    block_compact(row_keys, IdSelf{}, V, thr, need, k, hist, out);
  }
}

// ----------------------------------------------------------------- gather --
// blockIdx.x = row m of h, blockIdx.y = block of 8 candidates; warp w takes
// candidate 8y + w of row m's ascending list.  CTAs are short (one U row per
// warp) and dispatched in block order, so every row of h sweeps its sorted
// candidates at the same pace: a U row that several rows of h picked is
// requested by them at about the same time and DRAM delivers it about once
// (the union of the top-k sets), in roughly ascending address order.  (64
// candidates per CTA, 8 per warp in turn, kept all CTAs resident at once, so
// every candidate position was requested together: 90.8 us against 64.3 us
// at the Qwen3-8B shape, M = 32, k = 2048.)  h[m] (bf16, d <= 256 * CPL)
// sits in shared memory, so a thread holds only its CPL 16-byte chunks of
// the U row in flight.  Products are the bf16 x bf16 products (exact in
// fp32), accumulated in chunk order, element order.
template <int CPL, int CPW>
__global__ void __launch_bounds__(256)
    k_gather_logits(const uint8_t* __restrict__ h, const uint8_t* __restrict__ U,
                    const int32_t* __restrict__ idx, int M, int d, int k, int V,
                    float* __restrict__ cand_logits) {
  __shared__ uint4 s_h[32 * CPL];
  const int m = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nch = d / 8;
  const size_t rowb = (size_t)d * 2;
  for (int ch = threadIdx.x; ch < 32 * CPL; ch += blockDim.x)
    s_h[ch] = ch < nch ? __ldg(reinterpret_cast<const uint4*>(h + (size_t)m * rowb + ch * 16))
                       : make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  const int j0 = blockIdx.y * (8 * CPW) + warp * CPW;
  for (int jj = 0; jj < CPW; ++jj) {
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
      wv[c] = ch < nch ? ldg16_inflight(urow + ch * 16) : make_uint4(0, 0, 0, 0);
    }
    // the h reads below may not move above this point: every load of the
    // row is issued before the first product waits for one
    asm volatile("" ::: "memory");
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const uint4 w = wv[c], x = s_h[lane + 32 * c];
      acc = fma_bf16_lo(w.x, x.x, acc);
      acc = fma_bf16_hi(w.x, x.x, acc);
      acc = fma_bf16_lo(w.y, x.y, acc);
      acc = fma_bf16_hi(w.y, x.y, acc);
      acc = fma_bf16_lo(w.z, x.z, acc);
      acc = fma_bf16_hi(w.z, x.z, acc);
      acc = fma_bf16_lo(w.w, x.w, acc);
      acc = fma_bf16_hi(w.w, x.w, acc);
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
                  Draws dr, int32_t* __restrict__ out_tokens,
                  int32_t* __restrict__ out_idx, float* __restrict__ out_prob) {
  constexpr int NT = 256;
  pdl_launch_dependents();  // the next call's down-projection may start reading
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
    s_resid = draw_uniform(dr.uniforms, dr.seed, dr.offset, m, 0, 1) * run;
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

namespace {
// CTAs per row: the largest power of two <= 8 with M * C <= the SM count that
// the occupancy calculator accepts as a cluster (C >= 1).
int topk_cluster(int M) {
  static int fits[4] = {-1, -1, -1, -1};  // C = 1, 2, 4, 8
  int C = 1;
  while (C < 8 && (long long)M * C * 2 <= sm_count()) C *= 2;
  for (; C > 1; C >>= 1) {
    int& f = fits[C == 2 ? 1 : C == 4 ? 2 : 3];
    if (f < 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)C);
      cfg.blockDim = dim3(kTopkThreads);
      cfg.dynamicSmemBytes = kTopkCap * 16;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)C;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, k_topk, &cfg);
      if (e != cudaSuccess) (void)cudaGetLastError();
      f = (e == cudaSuccess && n > 0) ? 1 : 0;
    }
    if (f == 1) break;
  }
  return C;
}
}  // namespace

cudaError_t launch_topk(const float* scores, int M, int V, int k, int32_t* out_idx, void* ws,
                        cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  const int smem = kTopkCap * 16;  // region keys and ids, compact keys and ids
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(k_topk), smem);
  if (e != cudaSuccess) return e;
  const int C = topk_cluster(M);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(M * C));
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ProfScope ps(kKTopk, st);
  e = cudaLaunchKernelEx(&cfg, k_topk, scores, V, k, out_idx);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The router runs on the tensor cores when the shape fits the tcgen05 kernel.
static bool router_mma(int M, int d_prime, int V) { return mma_plan(d_prime, M, V).ok; }

size_t specvocab_ws_bytes(int M, int d, int d_prime, int V, int k) {
  if (router_mma(M, d_prime, V)) {
    size_t s = 0;
    s += align256((size_t)M * d_prime * 2);          // h' (bf16)
    s += align256((size_t)M * V * sizeof(float));    // scores
    s += align256(kMmaCtrs * sizeof(unsigned));      // the router's tile counters
    s += align256((size_t)M * k * sizeof(int32_t));  // candidates
    s += align256((size_t)M * k * sizeof(float));    // candidate logits
    return s;
  }
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
                             float temperature, const Draws& draws, int32_t* out_tokens,
                             int32_t* out_idx, float* out_prob, float* out_logits,
                             float* out_scores, void* ws, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  Carver cv(ws);
  void* hp = cv.take<uint8_t>((size_t)M * d_prime * 2);
  float* scores = cv.take<float>((size_t)M * V);
  int32_t* cand = nullptr;
  float* zc = nullptr;
  cudaError_t e;
  if (router_mma(M, d_prime, V)) {
    // s = W_vocab h' as the tcgen05 kernel's fp32 scores
    unsigned* ctr = cv.take<unsigned>(kMmaCtrs);
    cand = cv.take<int32_t>((size_t)M * k);
    zc = cv.take<float>((size_t)M * k);
    if (out_scores) scores = out_scores;
    // h' = bf16(W_down h): for many rows a split-K tensor-core GEMM whose fp32
    // slices live in the scores buffer until the router overwrites it
    const DownMmaPlan dp = M >= 32 ? down_mma_plan(M, d, d_prime, (size_t)M * V * sizeof(float))
                                   : DownMmaPlan{};
    e = dp.ok ? launch_down_mma(dp, h, w_down, M, d, d_prime, scores, hp, nullptr, ctr, kMmaCtrs,
                                st)
              : launch_down_proj(true, h, w_down, M, d, d_prime, true, hp, nullptr, ctr, kMmaCtrs,
                                 st);
    if (e != cudaSuccess) return e;
    const MmaPlan mp = mma_plan(d_prime, M, V);
    const MmaWork none{nullptr, nullptr, nullptr};
    const HeadOutputs no_out{Draws{nullptr, 0, 0}, nullptr, nullptr, nullptr, nullptr};
    e = launch_head_mma(mp, hp, w_vocab, M, d_prime, V, 0.f, none, no_out, scores, ctr, st);
    if (e != cudaSuccess) return e;
  } else {
  const HeadPlan plan = head_plan(true, d_prime, M, V);
  HeadPartials part;
  part.pmax = cv.take<float>((size_t)M * plan.n_sub);
  part.psum = cv.take<float>((size_t)M * plan.n_sub);
  part.parg = cv.take<int>((size_t)M * plan.n_sub);
  part.cmax = cv.take<float>((size_t)M * plan.grid);
  part.csum = cv.take<float>((size_t)M * plan.grid);
  part.carg = cv.take<int>((size_t)M * plan.grid);
  part.ctr = cv.take<unsigned>((size_t)plan.n_launch);
  int32_t* router_arg = cv.take<int32_t>((size_t)M);
  cand = cv.take<int32_t>((size_t)M * k);
  zc = cv.take<float>((size_t)M * k);
  if (out_scores) scores = out_scores;
  const HeadOutputs router_out{Draws{nullptr, 0, 0}, router_arg, nullptr, nullptr, nullptr};

  e = launch_down_proj(true, h, w_down, M, d, d_prime, true, hp, nullptr, part.ctr,
                       plan.n_launch, st);
  if (e != cudaSuccess) return e;
  e = launch_head_stream(plan, true, w_vocab, hp, M, d_prime, V, 0.f, part, scores, router_out,
                         st);
  if (e != cudaSuccess) return e;
  }
  e = launch_topk(scores, M, V, k, cand, nullptr, st);
  if (e != cudaSuccess) return e;
  if (out_logits) zc = out_logits;  // the candidates' exact logits, requested as an output
  constexpr int kCpw = 1;  // candidates per warp
  const dim3 grid(M, (k + 8 * kCpw - 1) / (8 * kCpw));
  const int cpl = (d + 255) / 256;
  {
  ProfScope ps(kKGather, st);
  if (cpl <= 4)
    k_gather_logits<4, kCpw><<<grid, 256, 0, st>>>((const uint8_t*)h, (const uint8_t*)u_full, cand,
                                                   M, d, k, V, zc);
  else if (cpl <= 8)
    k_gather_logits<8, kCpw><<<grid, 256, 0, st>>>((const uint8_t*)h, (const uint8_t*)u_full, cand,
                                                   M, d, k, V, zc);
  else
    k_gather_logits<16, kCpw><<<grid, 256, 0, st>>>((const uint8_t*)h, (const uint8_t*)u_full,
                                                    cand, M, d, k, V, zc);
  }
  const float c = temperature > 0.f ? (float)(1.4426950408889634 / (double)temperature) : 0.f;
  ProfScope ps(kKCandFinish, st);
  k_cand_finish<<<M, 256, 0, st>>>(zc, cand, k, c, draws, out_tokens, out_idx, out_prob);
  return cudaGetLastError();
}

}  // namespace ss
