// Backward of Route and Combine (the training configuration).
//
// The pages give no backward formulas; these are the reverse-mode derivatives
// of the forward with the selection held fixed (the selection bias gets no
// gradient: it only selects, "Scalable Training of Mixture-of-Experts Models
// with Megatron Core", review §2.2, aux-loss-free balancing):
//   dprob[t,k] = <dy_t, E_k(x_t)>                       (from the FC2 dgrad epilogue)
//   softmax, renormalised:  dl_k = p_k (dprob_k - sum_j p_j dprob_j)
//   sigmoid, renormalised:  dl_k = s_k (1 - s_k) (dprob_k - sum_j p_j dprob_j) / sum_sel s
//   dW_r[e] = sum over e's rows r of dl_r x_r,  db_r[e] = sum dl_r  (dl is zero off the selection)
//   dx[t]   = sum_k dx_perm[dst_row[t,k]] + dx_shared[t] + sum_k dl[t,k] W_r[e_k]
// Every sum runs in a fixed order: the results are bitwise reproducible.
#include "common.cuh"

namespace moe {

// dprob_perm[r] = sum of the FC2 dgrad epilogue's per-N-tile partials.
__global__ void dprob_reduce_kernel(const float* __restrict__ part, int rows, int nt,
                                    float* __restrict__ dprob_perm) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= rows) return;
  float s = 0.f;
  for (int j = 0; j < nt; ++j) s += __ldg(part + r * nt + j);
  dprob_perm[r] = s;
}

// Warp per token: dl for the K selected experts.
__global__ void __launch_bounds__(256) router_bwd_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ idx,
    const float* __restrict__ prob, const int32_t* __restrict__ dst_row,
    const float* __restrict__ dprob_perm, int T, int E, int K, int P, int score,
    float* __restrict__ dl_topk, float* __restrict__ dl_perm, int* status) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const bool act = lane < K;
  int r = -1, e = 0;
  float dp = 0.f, p = 0.f, s = 0.f;
  if (act) {
    r = __ldg(dst_row + t * K + lane);
    e = __ldg(idx + t * K + lane);
    if (r < 0 || r >= P || e < 0 || e >= E) {
      report(status, MOE_ERR_DEVICE_BOUNDS);
      r = -1;
    } else {
      dp = __ldg(dprob_perm + r);
      p = __ldg(prob + t * K + lane);
      s = sigmoid_f(__ldg(logits + t * E + e));
    }
  }
  float pdp = p * dp, ssum = s;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    pdp += __shfl_xor_sync(0xffffffffu, pdp, off);
    ssum += __shfl_xor_sync(0xffffffffu, ssum, off);
  }
  if (!act || r < 0) return;
  const float dl = score == MOE_SCORE_SOFTMAX ? p * (dp - pdp) : s * (1.f - s) * (dp - pdp) / ssum;
  dl_topk[t * K + lane] = dl;
  dl_perm[r] = dl;
}

// dW_r[e, c..c+8) = sum over expert e's rows of dl_perm[r] * x[src_token[r], c..c+8)
// (fp32, rows in order); db_r[e] = sum of dl_perm over the rows.
template <typename T>
__global__ void __launch_bounds__(256) router_wgrad_kernel(
    const T* __restrict__ x, const int32_t* __restrict__ src_token,
    const int32_t* __restrict__ offsets, const float* __restrict__ dl_perm, int h,
    float* __restrict__ dw_r, float* __restrict__ db_r) {
  constexpr int V = 8;
  const int e = blockIdx.x;
  const int c = (blockIdx.y * blockDim.x + threadIdx.x) * V;
  const int r0 = __ldg(offsets + e), r1 = __ldg(offsets + e + 1);
  if (c < h) {
    float acc[V] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int r = r0; r < r1; ++r) {
      const float d = __ldg(dl_perm + r);
      const T* row = x + (int64_t)__ldg(src_token + r) * h + c;
      float v[V];
      if constexpr (sizeof(T) == 2) {
        const Vec<__nv_bfloat16> u = ldg16(reinterpret_cast<const __nv_bfloat16*>(row));
#pragma unroll
        for (int i = 0; i < V; ++i) v[i] = __bfloat162float(u.v[i]);
      } else {
        const float4 a = __ldg(reinterpret_cast<const float4*>(row));
        const float4 b = __ldg(reinterpret_cast<const float4*>(row + 4));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
      }
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(d, v[i], acc[i]);
    }
    float* o = dw_r + (int64_t)e * h + c;
    *reinterpret_cast<float4*>(o) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(o + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  if (db_r && blockIdx.y == 0 && threadIdx.x == 0) {
    float s = 0.f;
    for (int r = r0; r < r1; ++r) s += __ldg(dl_perm + r);
    db_r[e] = s;
  }
}

// Warp per token: dx[t] = sum_k dx_perm[dst_row[t,k]] (+ dx_shared[t])
//                        + sum_k dl_topk[t,k] * W_r[idx[t,k]]   (when dl_topk given)
// fp32 accumulation in a fixed order, one rounding to the output type.
template <typename T>
__global__ void __launch_bounds__(256) bwd_combine_kernel(
    const T* __restrict__ dx_perm, const int32_t* __restrict__ dst_row,
    const T* __restrict__ dx_shared, const float* __restrict__ dl_topk,
    const int32_t* __restrict__ idx, const float* __restrict__ w_r, int ntok, int K, int E, int h,
    T* __restrict__ dx, float* __restrict__ dx_f32, int* status) {
  constexpr int V = 8;  // columns per lane per pass (one 16-B bf16 vector)
  const int lane = threadIdx.x & 31;
  const int64_t P = (int64_t)ntok * K;
  for (int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); t < ntok;
       t += (int64_t)gridDim.x * 8) {
    int src[16], ex[16];
    float dl[16];
    for (int k = 0; k < K; ++k) {
      int r = dx_perm ? __ldg(dst_row + t * K + k) : 0;
      if (dx_perm && (r < 0 || r >= P)) {
        report(status, MOE_ERR_DEVICE_BOUNDS);
        r = -1;
      }
      src[k] = r;
      int e = dl_topk ? __ldg(idx + t * K + k) : 0;
      if (e < 0 || e >= E) {
        report(status, MOE_ERR_DEVICE_BOUNDS);
        e = -1;
      }
      ex[k] = e;
      dl[k] = dl_topk ? __ldg(dl_topk + t * K + k) : 0.f;
    }
    for (int c = lane * V; c < h; c += 32 * V) {
      float acc[V] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (dx_perm) {
        for (int k = 0; k < K; ++k) {
          if (src[k] < 0) continue;
          const T* row = dx_perm + (int64_t)src[k] * h + c;
#pragma unroll
          for (int i = 0; i < V; ++i) acc[i] += to_f32(row[i]);
        }
      }
      if (dx_shared) {
        const T* row = dx_shared + t * h + c;
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] += to_f32(row[i]);
      }
      if (dl_topk) {
        for (int k = 0; k < K; ++k) {
          if (ex[k] < 0) continue;
          const float* wr = w_r + (int64_t)ex[k] * h + c;
#pragma unroll
          for (int i = 0; i < V; ++i) acc[i] = fmaf(dl[k], __ldg(wr + i), acc[i]);
        }
      }
      if (dx) {
#pragma unroll
        for (int i = 0; i < V; ++i) dx[t * h + c + i] = from_f32<T>(acc[i]);
      }
      if (dx_f32) {
#pragma unroll
        for (int i = 0; i < V; ++i) dx_f32[t * h + c + i] = acc[i];
      }
    }
  }
}

int scatter_grid(int ntok, int sms);

cudaError_t launch_dprob_reduce(const float* part, int rows, int nt, float* dprob_perm,
                                cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  dprob_reduce_kernel<<<(unsigned)ceil_div(rows, 256), 256, 0, s>>>(part, rows, nt, dprob_perm);
  return cudaGetLastError();
}

cudaError_t launch_router_bwd(const moe_config_t& c, const float* logits, const int32_t* idx,
                              const float* prob, const int32_t* dst_row, const float* dprob_perm,
                              float* dl_topk, float* dl_perm, int* status, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  router_bwd_kernel<<<(unsigned)ceil_div(c.T, 8), 256, 0, s>>>(
      logits, idx, prob, dst_row, dprob_perm, c.T, c.E, c.K, c.T * c.K, c.score, dl_topk, dl_perm,
      status);
  return cudaGetLastError();
}

cudaError_t launch_router_wgrad(const moe_config_t& c, const void* x, const int32_t* src_token,
                                const int32_t* offsets, const float* dl_perm, float* dw_r,
                                float* db_r, cudaStream_t s) {
  dim3 grid((unsigned)c.E, (unsigned)ceil_div(c.h, 256 * 8));
  if (c.dtype == MOE_BF16)
    router_wgrad_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(x), src_token, offsets, dl_perm, c.h, dw_r, db_r);
  else
    router_wgrad_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(x), src_token,
                                                    offsets, dl_perm, c.h, dw_r, db_r);
  return cudaGetLastError();
}

cudaError_t launch_bwd_combine(const moe_config_t& c, const void* dx_perm, const int32_t* dst_row,
                               const void* dx_shared, const float* dl_topk, const int32_t* idx,
                               const float* w_r, void* dx, float* dx_f32, int sms, int* status,
                               cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const int grid = scatter_grid(c.T, sms);
  if (c.dtype == MOE_BF16)
    bwd_combine_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(dx_perm), dst_row,
        static_cast<const __nv_bfloat16*>(dx_shared), dl_topk, idx, w_r, c.T, c.K, c.E, c.h,
        static_cast<__nv_bfloat16*>(dx), dx_f32, status);
  else
    bwd_combine_kernel<float><<<grid, 256, 0, s>>>(
        static_cast<const float*>(dx_perm), dst_row, static_cast<const float*>(dx_shared), dl_topk,
        idx, w_r, c.T, c.K, c.E, c.h, static_cast<float*>(dx), dx_f32, status);
  return cudaGetLastError();
}

}  // namespace moe
