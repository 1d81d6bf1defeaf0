// philox.cu -- the Philox4x32-10 stream behind the sampling calls, exposed on
// its own: raw blocks (counter and key words in, four output words out) and
// the (rows x slots) uniforms one call draws when the caller passes no
// uniforms of its own.  The generator itself (philox4x32_10, philox_uniform)
// lives in ss_common.cuh beside the kernels that call it.
#include "ss_common.cuh"
#include "ss_internal.h"

namespace ss {

// One thread per block of six input words (c0..c3, k0, k1).
__global__ void __launch_bounds__(256)
    k_philox_blocks(const uint32_t* __restrict__ in, int n, uint32_t* __restrict__ out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t* w = in + (size_t)i * 6;
  const uint4 x = philox4x32_10(make_uint4(w[0], w[1], w[2], w[3]), w[4], w[5]);
  uint32_t* o = out + (size_t)i * 4;
  o[0] = x.x;
  o[1] = x.y;
  o[2] = x.z;
  o[3] = x.w;
}

// One thread per draw (row, slot), row-major.
__global__ void __launch_bounds__(256)
    k_philox_uniforms(uint64_t seed, uint64_t offset, int rows, int slots,
                      float* __restrict__ out) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)rows * slots) return;
  const int row = (int)(i / slots), slot = (int)(i - (long long)row * slots);
  out[i] = philox_uniform(seed, offset, (uint32_t)row, (uint32_t)slot);
}

cudaError_t launch_philox_blocks(const uint32_t* in, int n, uint32_t* out, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  k_philox_blocks<<<(n + 255) / 256, 256, 0, st>>>(in, n, out);
  return cudaGetLastError();
}

cudaError_t launch_philox_uniforms(uint64_t seed, uint64_t offset, int rows, int slots, float* out,
                                   cudaStream_t st) {
  const long long n = (long long)rows * slots;
  if (n <= 0) return cudaSuccess;
  k_philox_uniforms<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(seed, offset, rows, slots, out);
  return cudaGetLastError();
}

}  // namespace ss
