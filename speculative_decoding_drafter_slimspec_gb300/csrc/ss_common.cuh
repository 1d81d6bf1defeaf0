// ss_common.cuh -- device helpers shared by the sm_103a kernels of libslimspec.
//
// Holds: the per-device error word, bounded mbarrier waits, 1-D bulk copies
// (cp.async.bulk) into shared memory, bf16 unpacking, lane reductions, the
// (max, sum, argmax) running state of an online softmax and the Philox4x32-10
// uniforms of the sampling draws.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/slimspec.h"

namespace ss {

// ------------------------------------------------------------------ errors --
enum : unsigned { kErrTimeout = 1u, kErrIndex = 2u };

// A bounded wait gives up after this many nanoseconds and reports kErrTimeout.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

// The per-device control block of the library.  Kernels receive the device
// address of its first word, the error word, as `err` and record anomalies
// there with atomicOr (see ss_get_device_error); the other words are read
// only by the bounded waits: the limit of the pipeline waits (host-settable,
// kWaitLimitNs by default) and a test switch that makes the tensor-core
// head's MMA issuer wait on a barrier nothing arrives on.
struct DeviceControl {
  unsigned err;
  unsigned stall_head;
  unsigned long long wait_limit_ns;
};

__device__ __forceinline__ void raise_error(unsigned* err, unsigned bits) {
  if (err) atomicOr(err, bits);
}

__device__ __forceinline__ const volatile DeviceControl* control(const unsigned* err) {
  return reinterpret_cast<const volatile DeviceControl*>(err);
}

// ------------------------------------------------------------ time / waits --
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false (and
// records kErrTimeout) if it has not completed within `limit_ns`.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, unsigned* err,
                                              uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) {
      raise_error(err, kErrTimeout);
      return false;
    }
  }
}

// A wait of the pipeline (a stage to fill or free, an accumulator, a tile
// id): bounded by the control block's host-settable limit.  After one of
// these runs out, the caller abandons the pipeline and drains.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned* err) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_for(bar, parity, err, err ? control(err)->wait_limit_ns : kWaitLimitNs);
}

// A drain wait (copies or MMAs already issued, before their shared memory or
// TMEM is released): always the fixed kWaitLimitNs, whatever the pipeline
// limit, so that nothing in flight outlives the CTA.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, unsigned* err) {
  return mbar_wait_for(bar, parity, err, kWaitLimitNs);
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// 1-D bulk copy global -> shared, completing `bytes` transactions on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ----------------------------------------------- programmatic dependent launch --
// The producer lets its dependent grid start early; the dependent waits for
// the producer's memory operations before its first read of them.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_producer() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// --------------------------------------------------------------- numerics --
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// d = a * b + c with a, b the low (or high) bf16 halves of two 32-bit words and
// c, d fp32, rounded once (fma.rn.f32.bf16, sm_100+).  A bf16 x bf16 product
// is exact in fp32, so this equals fmaf on the widened operands; it saves the
// widening instructions and issues at the scalar FFMA rate.
// 16-byte read-only load that stays in program order with the other ones
// (volatile): a run of them is issued back to back, all in flight together.
__device__ __forceinline__ uint4 ldg16_inflight(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float fma_bf16_lo(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %3;\n\t}"
      : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_bf16_hi(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, ah, bh, %3;\n\t}"
      : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}

// Round-to-nearest-even of an fp32 value to bf16, returned as fp32 and as bits.
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  uint32_t b = __float_as_uint(x);
  b += 0x7FFFu + ((b >> 16) & 1u);
  return static_cast<uint16_t>(b >> 16);
}
__device__ __forceinline__ float round_bf16(float x) {
  return __uint_as_float(static_cast<uint32_t>(f32_to_bf16_bits(x)) << 16);
}

constexpr float kLog2e = 1.4426950408889634f;

// 2**x on the SFU (ex2.approx; relative error about 2**-22); 2**-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kNegInf = -__builtin_huge_valf();

// Running state of an online softmax over a stream of logits:
//   mx  = largest logit seen, arg = lowest index attaining it,
//   sum = sum_v exp2((l_v - mx) * c)  with c = log2(e) / T  (sampling only).
struct RowState {
  float mx;
  float sum;
  int arg;
};

__device__ __forceinline__ RowState row_state_empty() { return {kNegInf, 0.f, 0x7FFFFFFF}; }

template <bool kSample>
__device__ __forceinline__ void row_state_push(RowState& s, float x, int v, float c) {
  if (x > s.mx) {
    if (kSample) s.sum = __fmaf_rn(s.sum, fast_exp2((s.mx - x) * c), 1.0f);
    s.mx = x;
    s.arg = v;
  } else if (kSample) {
    s.sum = __fadd_rn(s.sum, fast_exp2((x - s.mx) * c));
  }
}

// Combines two states; the argmax tie goes to the lower index.
template <bool kSample>
__device__ __forceinline__ RowState row_state_merge(RowState a, RowState b, float c) {
  RowState o;
  const bool take_b = (b.mx > a.mx) || (b.mx == a.mx && b.arg < a.arg);
  o.mx = take_b ? b.mx : a.mx;
  o.arg = take_b ? b.arg : a.arg;
  if (kSample) {
    const float sa = (a.mx == o.mx) ? a.sum : a.sum * fast_exp2((a.mx - o.mx) * c);
    const float sb = (b.mx == o.mx) ? b.sum : b.sum * fast_exp2((b.mx - o.mx) * c);
    o.sum = __fadd_rn(sa, sb);
  } else {
    o.sum = 0.f;
  }
  return o;
}

template <bool kSample>
__device__ __forceinline__ RowState shfl_merge(RowState s, int offset, float c) {
  RowState o;
  o.mx = __shfl_xor_sync(0xFFFFFFFFu, s.mx, offset);
  o.sum = __shfl_xor_sync(0xFFFFFFFFu, s.sum, offset);
  o.arg = __shfl_xor_sync(0xFFFFFFFFu, s.arg, offset);
  return row_state_merge<kSample>(s, o, c);
}

// Reduce-scatter of N per-lane values over aligned groups of G lanes
// (N, G powers of two).  After the call lane l holds, in v[0 .. max(N/G,1)-1],
// the group-wide sums of the entries with indices
//   ((l % G) >> (log2 G - s)) << log2(max(N/G,1)) + i,   s = log2(N / max(N/G,1)),
// and lanes that differ only in their low (log2 G - s) bits hold equal values.
template <int N, int O>
struct ReduceScatter {
  static __device__ __forceinline__ void run(float* v, int lane) {
    if constexpr (O == 0) {
      return;
    } else if constexpr (N > 1) {
      const bool hi = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        const float send = hi ? v[i] : v[i + N / 2];
        const float keep = hi ? v[i + N / 2] : v[i];
        v[i] = __fadd_rn(keep, __shfl_xor_sync(0xFFFFFFFFu, send, O));
      }
      ReduceScatter<N / 2, O / 2>::run(v, lane);
    } else {
      v[0] = __fadd_rn(v[0], __shfl_xor_sync(0xFFFFFFFFu, v[0], O));
      ReduceScatter<1, O / 2>::run(v, lane);
    }
  }
};

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// Select-free reduce-scatter.  Each lane must hold its N values in the
// lane-permuted slot order slot s <-> index s ^ mask, with
//   mask = ((l % G) >> (log2 G - s)) << log2(max(N/G, 1))
// (s, G as for ReduceScatter): at every step the half a lane keeps is then
// its first half, and the partner's second half holds the same indices.
// Afterwards v[i], i < max(N/G,1), holds the group-wide sum of index mask + i.
template <int N, int O>
struct ReduceScatterP {
  static __device__ __forceinline__ void run(float* v) {
    if constexpr (O == 0) {
      return;
    } else if constexpr (N > 1) {
#pragma unroll
      for (int i = 0; i < N / 2; ++i)
        v[i] = __fadd_rn(v[i], __shfl_xor_sync(0xFFFFFFFFu, v[i + N / 2], O));
      ReduceScatterP<N / 2, O / 2>::run(v);
    } else {
      v[0] = __fadd_rn(v[0], __shfl_xor_sync(0xFFFFFFFFu, v[0], O));
      ReduceScatterP<1, O / 2>::run(v);
    }
  }
};

// Fixed-order warp sum: tree toward lane 0, result broadcast from lane 0, so
// every lane holds the same bits.
__device__ __forceinline__ float warp_sum_fixed(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = __fadd_rn(x, __shfl_down_sync(0xFFFFFFFFu, x, o));
  return __shfl_sync(0xFFFFFFFFu, x, 0);
}

// Inclusive prefix sum across the 32 lanes in lane order (fixed order).
__device__ __forceinline__ float warp_incl_scan(float x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x = __fadd_rn(y, x);
  }
  return x;
}

// First index in [0, n) (ascending) whose running total passes `target`, with
// the running total before it; the last index with a positive value if
// rounding leaves none.  Lane l holds the value of index l + 32 k in mass[k];
// chunks of 32 are scanned in order with the fixed-order warp scan.
template <int NC>
__device__ __forceinline__ int ordered_crossing_regs(int n, float target, const float (&mass)[NC],
                                                     float& before, int lane) {
  float run = 0.f, before_last = 0.f;
  int sel = -1, last = -1;
#pragma unroll
  for (int k = 0; k < NC; ++k) {
    const int i0 = 32 * k;
    if (i0 < n && sel < 0) {
      const float mt = mass[k];
      const float cum = __fadd_rn(run, warp_incl_scan(mt, lane));
      const unsigned pos = __ballot_sync(0xFFFFFFFFu, mt > 0.f);
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, mt > 0.f && cum > target);
      if (hit) {
        const int l = __ffs(hit) - 1;
        sel = i0 + l;
        before = __shfl_sync(0xFFFFFFFFu, __fsub_rn(cum, mt), l);
      } else if (pos) {
        const int l = 31 - __clz(pos);
        last = i0 + l;
        before_last = __shfl_sync(0xFFFFFFFFu, __fsub_rn(cum, mt), l);
      }
      run = __shfl_sync(0xFFFFFFFFu, cum, 31);
    }
  }
  if (sel < 0) {
    sel = last < 0 ? 0 : last;
    before = before_last;
  }
  return sel;
}

// ------------------------------------------------------ Philox uniforms --
// Philox4x32-10: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel
// Random Numbers: As Easy as 1, 2, 3" (SC'11), section 4.  A round multiplies
// counter words 0 and 2 by the paper's two 32-bit multipliers (full 64-bit
// products), then permutes: word 0 = hi(M1 c2) ^ c1 ^ k0, word 1 = lo(M1 c2),
// word 2 = hi(M0 c0) ^ c3 ^ k1, word 3 = lo(M0 c0).  The key advances by the
// Weyl constants between rounds; ten rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    if (i > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// Uniform in [0, 1) of draw (row, slot) of the call (seed, offset): key =
// (seed mod 2^32, seed >> 32), counter = (row, slot, offset mod 2^32,
// offset >> 32), u = (first output word >> 8) * 2^-24 (exact in fp32).
__device__ __forceinline__ float philox_uniform(uint64_t seed, uint64_t offset, uint32_t row,
                                                uint32_t slot) {
  const uint4 x = philox4x32_10(
      make_uint4(row, slot, (uint32_t)offset, (uint32_t)(offset >> 32)), (uint32_t)seed,
      (uint32_t)(seed >> 32));
  return (float)(x.x >> 8) * 5.9604644775390625e-8f;  // 2^-24
}

// The uniform of draw (row, slot): the caller's uniforms[row * n_slots +
// slot] when given, else the Philox stream at (seed, offset).
__device__ __forceinline__ float draw_uniform(const float* uniforms, uint64_t seed,
                                              uint64_t offset, uint32_t row, uint32_t slot,
                                              uint32_t n_slots) {
  if (uniforms != nullptr) return __ldg(uniforms + (size_t)row * n_slots + slot);
  return philox_uniform(seed, offset, row, slot);
}

// Orderable 32-bit key of a float: larger float <=> larger key; -0 == +0.
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

}  // namespace ss
