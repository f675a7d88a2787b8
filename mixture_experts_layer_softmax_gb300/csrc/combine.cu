// Combine: probability-weighted unpermute back to token order.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (review),
// §2.1 "Combine" (the expert outputs are un-permuted to the original token
// order) with §1.1's MoE(x) = sum_i p_i E_i(x); the skill page
// "emerging-techniques-moe-training" accumulates with index_add_.  Here the
// sum is a gather: token t reads its K rows y_perm[dst_row[t,k]], accumulates
// w[t,k] * row in fp32 in fixed k order (then + shared_y[t]) and rounds once,
// so the result is bitwise deterministic -- no atomics.
#include "common.cuh"

namespace moe {

template <typename T>
__global__ void __launch_bounds__(256) combine_kernel(const T* __restrict__ y_perm,
                                                      const int32_t* __restrict__ dst_row,
                                                      const float* __restrict__ w,
                                                      const T* __restrict__ shared_y, int ntok,
                                                      int K, int h, T* __restrict__ y,
                                                      int* status) {
  constexpr int V = Vec<T>::N;
  constexpr int kMaxVec = 4;
  const int lane = threadIdx.x & 31;
  const int nvec = h / V;
  const int64_t P = (int64_t)ntok * K;
  for (int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); t < ntok;
       t += (int64_t)gridDim.x * 8) {
    int src[16];
    float wk[16];
    for (int k = 0; k < K; ++k) {
      int r = __ldg(dst_row + t * K + k);
      if (r < 0 || r >= P) {
        report(status, MOE_ERR_DEVICE_BOUNDS);
        r = -1;
      }
      src[k] = r;
      wk[k] = w ? __ldg(w + t * K + k) : 1.f;
    }
    for (int v0 = 0; v0 < nvec; v0 += 32 * kMaxVec) {
      float acc[kMaxVec][V];
#pragma unroll
      for (int i = 0; i < kMaxVec; ++i)
#pragma unroll
        for (int q = 0; q < V; ++q) acc[i][q] = 0.f;
      for (int k = 0; k < K; ++k) {
        if (src[k] < 0) continue;
        const T* row = y_perm + (int64_t)src[k] * h;
#pragma unroll
        for (int i = 0; i < kMaxVec; ++i) {
          const int v = v0 + i * 32 + lane;
          if (v < nvec) {
            const Vec<T> u = ld16_stream(row + (int64_t)v * V);
#pragma unroll
            for (int q = 0; q < V; ++q) acc[i][q] = fmaf(wk[k], to_f32(u.v[q]), acc[i][q]);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kMaxVec; ++i) {
        const int v = v0 + i * 32 + lane;
        if (v >= nvec) continue;
        if (shared_y) {
          const Vec<T> u = ld16_stream(shared_y + t * h + (int64_t)v * V);
#pragma unroll
          for (int q = 0; q < V; ++q) acc[i][q] += to_f32(u.v[q]);
        }
        Vec<T> o;
#pragma unroll
        for (int q = 0; q < V; ++q) o.v[q] = from_f32<T>(acc[i][q]);
        st16(y + t * h + (int64_t)v * V, o);
      }
    }
  }
}

int scatter_grid(int ntok, int sms);

cudaError_t launch_combine(const moe_config_t& c, const void* y_perm, const int32_t* dst_row,
                           const float* w, const void* shared_y, void* y, int sms, int* status,
                           cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const int grid = scatter_grid(c.T, sms);
  if (c.dtype == MOE_BF16)
    combine_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(y_perm), dst_row, w,
        static_cast<const __nv_bfloat16*>(shared_y), c.T, c.K, c.h,
        static_cast<__nv_bfloat16*>(y), status);
  else
    combine_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(y_perm), dst_row, w,
                                               static_cast<const float*>(shared_y), c.T, c.K, c.h,
                                               static_cast<float*>(y), status);
  return cudaGetLastError();
}

}  // namespace moe
