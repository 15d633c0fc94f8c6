// Test helper, compiled by tests/test_gpu_philox.py: Philox4x32-10 on the
// device for a list of (counter, key) tuples, once with the library's own
// generator (common.cuh) and once with cuRAND's Philox4_32_10 device API.
//
// cuRAND's mapping (curand_kernel.h, curand_philox4x32_x.h): curand_init sets
// the key to the seed's low and high words and the counter to zero, skips
// `subsequence` into counter words (z, w) and `offset / 4` into words (x, y);
// the first curand4 then returns the block of that counter. So counter
// (c0, c1, c2, c3) is reached with subsequence (c3 << 32 | c2) and offset
// 4 * (c1 << 32 | c0), which needs c1 < 2^30.
#include <curand_kernel.h>

#include "common.cuh"

__global__ void philox_probe_kernel(const uint32_t* in, uint32_t* lib_out, uint32_t* curand_out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t* c = in + 6 * i;
  const specv::Philox4 a = specv::philox4x32_10(c[0], c[1], c[2], c[3], c[4], c[5]);
  for (int j = 0; j < 4; ++j) lib_out[4 * i + j] = a.v[j];
  if (c[1] >= (1u << 30)) return;  // the offset would not fit in 64 bits
  curandStatePhilox4_32_10_t st;
  const unsigned long long seed = (unsigned long long)c[4] | ((unsigned long long)c[5] << 32);
  const unsigned long long subsequence = (unsigned long long)c[2] | ((unsigned long long)c[3] << 32);
  const unsigned long long offset = 4ull * ((unsigned long long)c[0] | ((unsigned long long)c[1] << 32));
  curand_init(seed, subsequence, offset, &st);
  const uint4 r = curand4(&st);
  curand_out[4 * i + 0] = r.x;
  curand_out[4 * i + 1] = r.y;
  curand_out[4 * i + 2] = r.z;
  curand_out[4 * i + 3] = r.w;
}

// Device pointers; in: n x 6 words (c0 c1 c2 c3 k0 k1), outputs n x 4 words.
extern "C" int philox_probe(const uint32_t* in, uint32_t* lib_out, uint32_t* curand_out, int n) {
  if (n <= 0) return 0;
  philox_probe_kernel<<<(n + 127) / 128, 128>>>(in, lib_out, curand_out, n);
  return (int)cudaDeviceSynchronize();
}
