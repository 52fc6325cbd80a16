// Test helper: words of cuRAND's device Philox4_32_10 generator, used to pin the
// oracle's own Philox4x32-10 implementation to an independent library.
// For thread t: curand_init(seed, subsequence, 4 * (g0 + t)) then curand4().
#include <cstdint>
#include <curand_kernel.h>

__global__ void philox_words(unsigned long long seed, unsigned long long subsequence, unsigned long long g0, int n,
                             uint4* out) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n) return;
  curandStatePhilox4_32_10_t st;
  curand_init(seed, subsequence, 4ull * (g0 + (unsigned long long)t), &st);
  out[t] = curand4(&st);
}

extern "C" int curand_philox_words(unsigned long long seed, unsigned long long subsequence, unsigned long long g0,
                                   int n, unsigned int* host_out) {
  uint4* d = nullptr;
  if (cudaMalloc(&d, sizeof(uint4) * n) != cudaSuccess) return 1;
  philox_words<<<(n + 127) / 128, 128>>>(seed, subsequence, g0, n, d);
  int rc = cudaDeviceSynchronize() == cudaSuccess ? 0 : 2;
  if (!rc && cudaMemcpy(host_out, d, sizeof(uint4) * n, cudaMemcpyDeviceToHost) != cudaSuccess) rc = 3;
  cudaFree(d);
  return rc;
}
