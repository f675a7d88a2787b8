// Seeded synthetic tensors on the device: the same counter-based generator as
// the package's inputs.py (SplitMix64 -- Steele, Lea and Flood, OOPSLA 2014 --
// then the cosine branch of Box-Muller, in double, rounded to fp32 and, for
// bf16 tensors, again to bf16, both round-to-nearest-even).  Holds none of the
// MoE layer's arithmetic; it only fills buffers with test data.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void normal_kernel(void* out, int64_t n, int is_bf16, uint64_t key, double stdev,
                              int64_t start) {
  const double two_pi = 6.283185307179586;  // nearest double to 2 pi
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t u = mix64(key + (uint64_t)(start + i + 1) * kGamma);
    const double u1 = __dmul_rn((double)(u >> 32) + 1.0, 2.3283064365386963e-10);
    const double u2 = __dmul_rn((double)(u & 0xffffffffull), 2.3283064365386963e-10);
    const double z = __dmul_rn(sqrt(__dmul_rn(-2.0, log(u1))), cos(__dmul_rn(two_pi, u2)));
    const float f = __double2float_rn(__dmul_rn(stdev, z));
    if (is_bf16)
      static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(f);
    else
      static_cast<float*>(out)[i] = f;
  }
}

}  // namespace

extern "C" {

// Fills out[0..n) with elements [start, start+n) of the stream (seed, tag):
// value = stdev * z rounded to fp32 (dtype 0) or to bf16 via fp32 (dtype 1).
// Returns a cudaError_t value (0 on success).
int moe_synth_normal(void* out, int64_t n, int dtype, uint64_t seed, uint64_t tag, double stdev,
                     int64_t start, void* stream) {
  if (n <= 0) return 0;
  const uint64_t key = mix64(seed * kGamma + tag);
  int sms = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks_needed = (n + 255) / 256;
  const int blocks = (int)(blocks_needed < (int64_t)sms * 16 ? blocks_needed : (int64_t)sms * 16);
  normal_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(out, n, dtype == 1, key,
                                                                       stdev, start);
  return (int)cudaGetLastError();
}

}  // extern "C"
