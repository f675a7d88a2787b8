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

// One 128-thread block per token (the grid covers every token, so the block
// scheduler balances the load); each thread owns 16-byte column vectors and
// issues the loads of all K rows before it accumulates them.
template <typename T, int KMAX>
__global__ void __launch_bounds__(128) combine_kernel(const T* __restrict__ y_perm,
                                                      const int32_t* __restrict__ dst_row,
                                                      const float* __restrict__ w,
                                                      const T* __restrict__ shared_y, int ntok,
                                                      int K, int h, T* __restrict__ y,
                                                      int* status) {
  constexpr int V = Vec<T>::N;
  __shared__ int64_t s_off[KMAX];
  __shared__ float s_w[KMAX];
  const int64_t t = blockIdx.x;
  const int64_t P = (int64_t)ntok * K;
  if (threadIdx.x < KMAX) {
    const int k = threadIdx.x;
    int64_t off = -1;
    float wk = 0.f;
    if (k < K) {
      const int r = __ldg(dst_row + t * K + k);
      if (r >= 0 && r < P) {
        off = (int64_t)r * h;
        wk = w ? __ldg(w + t * K + k) : 1.f;
      } else if (r != -1) {  // -1: a dropped slot (capacity) or an id reported by dispatch
        report(status, MOE_ERR_DEVICE_BOUNDS);
      }
    }
    s_off[k] = off;
    s_w[k] = wk;
  }
  __syncthreads();
  const int nvec = h / V;
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    Vec<T> u[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      if (s_off[k] >= 0) u[k] = ld16_stream(y_perm + s_off[k] + (int64_t)v * V);
    float acc[V];
#pragma unroll
    for (int q = 0; q < V; ++q) acc[q] = 0.f;
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      if (s_off[k] >= 0) {
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] = fmaf(s_w[k], to_f32(u[k].v[q]), acc[q]);
      }
    if (shared_y) {
      const Vec<T> sv = ld16_stream(shared_y + t * h + (int64_t)v * V);
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] += to_f32(sv.v[q]);
    }
    Vec<T> o;
#pragma unroll
    for (int q = 0; q < V; ++q) o.v[q] = from_f32<T>(acc[q]);
    st16(y + t * h + (int64_t)v * V, o);
  }
}

template <typename T>
static cudaError_t combine_t(const moe_config_t& c, const void* y_perm, const int32_t* dst_row,
                             const float* w, const void* shared_y, void* y, int* status,
                             cudaStream_t s) {
  const unsigned grid = (unsigned)c.T;
  const T* yp = static_cast<const T*>(y_perm);
  const T* sy = static_cast<const T*>(shared_y);
  T* out = static_cast<T*>(y);
  if (c.K <= 2)
    combine_kernel<T, 2><<<grid, 128, 0, s>>>(yp, dst_row, w, sy, c.T, c.K, c.h, out, status);
  else if (c.K <= 4)
    combine_kernel<T, 4><<<grid, 128, 0, s>>>(yp, dst_row, w, sy, c.T, c.K, c.h, out, status);
  else if (c.K <= 8)
    combine_kernel<T, 8><<<grid, 128, 0, s>>>(yp, dst_row, w, sy, c.T, c.K, c.h, out, status);
  else
    combine_kernel<T, 16><<<grid, 128, 0, s>>>(yp, dst_row, w, sy, c.T, c.K, c.h, out, status);
  return cudaGetLastError();
}

cudaError_t launch_combine(const moe_config_t& c, const void* y_perm, const int32_t* dst_row,
                           const float* w, const void* shared_y, void* y, int sms, int* status,
                           cudaStream_t s) {
  (void)sms;
  if (c.T == 0) return cudaSuccess;
  if (c.dtype == MOE_BF16)
    return combine_t<__nv_bfloat16>(c, y_perm, dst_row, w, shared_y, y, status, s);
  return combine_t<float>(c, y_perm, dst_row, w, shared_y, y, status, s);
}

}  // namespace moe
