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
//             (+ dx_add[t]: the dense router term of the load-balancing losses)
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
  // a slot dropped by the expert capacity (dst_row -1) has no expert output,
  // so dprob = 0, but its weight still enters the normalisation of the kept
  // ones and gets a gradient through them
  bool act = lane < K;
  int r = -1, e = 0;
  float dp = 0.f, p = 0.f, s = 0.f;
  if (act) {
    r = __ldg(dst_row + t * K + lane);
    e = __ldg(idx + t * K + lane);
    if (r < -1 || r >= P || e < 0 || e >= E) {
      report(status, MOE_ERR_DEVICE_BOUNDS);
      act = false;
      r = -1;
    } else {
      dp = r >= 0 ? __ldg(dprob_perm + r) : 0.f;
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
  if (lane >= K) return;
  if (!act) {  // an invalid slot: no gradient
    dl_topk[t * K + lane] = 0.f;
    return;
  }
  const float dl = score == MOE_SCORE_SOFTMAX ? p * (dp - pdp) : s * (1.f - s) * (dp - pdp) / ssum;
  dl_topk[t * K + lane] = dl;
  if (r >= 0) dl_perm[r] = dl;
}

// dW_r[e, c0..c0+256) = sum over expert e's rows r of dl_perm[r] * x[src_token[r], ...]
// (fp32); db_r[e] = sum of dl_perm over the rows.  One block per (expert,
// 256 columns): the expert's token ids and dl values are staged in shared
// memory (1024 rows at a time), 8 row groups of 32 lanes each sum the rows
// r = r0 + g, r0 + g + 8, ... in order (lane = 8 columns, several row loads in
// flight), and the 8 group sums are added in group order: a fixed summation
// order, so reruns are bitwise identical.
template <typename T>
__global__ void __launch_bounds__(256) router_wgrad_kernel(
    const T* __restrict__ x, const int32_t* __restrict__ src_token,
    const int32_t* __restrict__ offsets, const float* __restrict__ dl_perm, int h,
    float* __restrict__ dw_r, float* __restrict__ db_r) {
  constexpr int V = 8, G = 8, CHUNK = 1024;
  __shared__ int32_t s_tok[CHUNK];
  __shared__ float s_dl[CHUNK];
  __shared__ float s_acc[G][32 * V];
  const int e = blockIdx.x;
  const int g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.y * (32 * V) + lane * V;
  const int r0 = __ldg(offsets + e), r1 = __ldg(offsets + e + 1);
  float acc[V] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float dsum = 0.f;  // db_r: thread 0 adds the dl values in row order
  for (int q0 = r0; q0 < r1; q0 += CHUNK) {
    const int n = min(CHUNK, r1 - q0);
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      s_tok[i] = __ldg(src_token + q0 + i);
      s_dl[i] = __ldg(dl_perm + q0 + i);
    }
    __syncthreads();
    if (db_r && blockIdx.y == 0 && threadIdx.x == 0)
      for (int i = 0; i < n; ++i) dsum += s_dl[i];
    if (c < h) {
#pragma unroll 4
      for (int i = g; i < n; i += G) {
        const float d = s_dl[i];
        const T* row = x + (int64_t)s_tok[i] * h + c;
        float v[V];
        if constexpr (sizeof(T) == 2) {
          const Vec<__nv_bfloat16> u = ldg16(reinterpret_cast<const __nv_bfloat16*>(row));
#pragma unroll
          for (int j = 0; j < V; ++j) v[j] = __bfloat162float(u.v[j]);
        } else {
          const float4 a = __ldg(reinterpret_cast<const float4*>(row));
          const float4 b = __ldg(reinterpret_cast<const float4*>(row + 4));
          v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        }
#pragma unroll
        for (int j = 0; j < V; ++j) acc[j] = fmaf(d, v[j], acc[j]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < V; ++j) s_acc[g][lane * V + j] = acc[j];
  __syncthreads();
  const int col = blockIdx.y * (32 * V) + threadIdx.x;
  if (col < h) {
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < G; ++k) sum += s_acc[k][threadIdx.x];
    dw_r[(int64_t)e * h + col] = sum;
  }
  if (db_r && blockIdx.y == 0 && threadIdx.x == 0) db_r[e] = dsum;
}

// One 128-thread block per token:
//   dx[t] = sum_k dx_perm[dst_row[t,k]] (+ dx_shared[t]) + sum_k dl_topk[t,k] * W_r[idx[t,k]]
// each thread owns 8-column vectors and issues the K row loads before adding;
// fp32 accumulation in a fixed order, one rounding to the output type.
template <typename T, int KMAX>
__global__ void __launch_bounds__(128) bwd_combine_kernel(
    const T* __restrict__ dx_perm, const int32_t* __restrict__ dst_row,
    const T* __restrict__ dx_shared, const float* __restrict__ dl_topk,
    const int32_t* __restrict__ idx, const float* __restrict__ w_r,
    const float* __restrict__ dx_add, int ntok, int K, int E, int h, T* __restrict__ dx,
    float* __restrict__ dx_f32, int* status) {
  constexpr int V = 8;
  __shared__ int64_t s_src[KMAX];
  __shared__ int64_t s_w[KMAX];
  __shared__ float s_dl[KMAX];
  const int64_t t = blockIdx.x;
  const int64_t P = (int64_t)ntok * K;
  if (threadIdx.x < KMAX) {
    const int k = threadIdx.x;
    int64_t src = -1, wo = -1;
    float d = 0.f;
    if (k < K) {
      if (dx_perm) {
        const int r = __ldg(dst_row + t * K + k);
        if (r >= 0 && r < P)
          src = (int64_t)r * h;
        else if (r != -1)  // -1: a dropped slot, no expert output to differentiate
          report(status, MOE_ERR_DEVICE_BOUNDS);
      }
      if (dl_topk) {
        const int e = __ldg(idx + t * K + k);
        if (e >= 0 && e < E) {
          wo = (int64_t)e * h;
          d = __ldg(dl_topk + t * K + k);
        } else {
          report(status, MOE_ERR_DEVICE_BOUNDS);
        }
      }
    }
    s_src[k] = src;
    s_w[k] = wo;
    s_dl[k] = d;
  }
  __syncthreads();
  for (int c = threadIdx.x * V; c < h; c += blockDim.x * V) {
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    if (dx_perm) {
      Vec<T> u[KMAX];
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (s_src[k] >= 0) {
          if constexpr (sizeof(T) == 2) {
            u[k] = ld16_stream(dx_perm + s_src[k] + c);
          }
        }
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (s_src[k] >= 0) {
          if constexpr (sizeof(T) == 2) {
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] += to_f32(u[k].v[i]);
          } else {
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] += to_f32(dx_perm[s_src[k] + c + i]);
          }
        }
    }
    if (dx_shared) {
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += to_f32(dx_shared[t * h + c + i]);
    }
    if (dl_topk) {
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (s_w[k] >= 0) {
          const float4 a = __ldg(reinterpret_cast<const float4*>(w_r + s_w[k] + c));
          const float4 b = __ldg(reinterpret_cast<const float4*>(w_r + s_w[k] + c + 4));
          const float d = s_dl[k];
          acc[0] = fmaf(d, a.x, acc[0]); acc[1] = fmaf(d, a.y, acc[1]);
          acc[2] = fmaf(d, a.z, acc[2]); acc[3] = fmaf(d, a.w, acc[3]);
          acc[4] = fmaf(d, b.x, acc[4]); acc[5] = fmaf(d, b.y, acc[5]);
          acc[6] = fmaf(d, b.z, acc[6]); acc[7] = fmaf(d, b.w, acc[7]);
        }
    }
    if (dx_add) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(dx_add + t * h + c));
      const float4 b = __ldg(reinterpret_cast<const float4*>(dx_add + t * h + c + 4));
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    if (dx) {
      if constexpr (sizeof(T) == 2) {
        Vec<T> o;
#pragma unroll
        for (int i = 0; i < V; ++i) o.v[i] = from_f32<T>(acc[i]);
        st16(dx + t * h + c, o);
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) dx[t * h + c + i] = from_f32<T>(acc[i]);
      }
    }
    if (dx_f32) {
      *reinterpret_cast<float4*>(dx_f32 + t * h + c) = make_float4(acc[0], acc[1], acc[2], acc[3]);
      *reinterpret_cast<float4*>(dx_f32 + t * h + c + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
  }
}

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
  dim3 grid((unsigned)c.E, (unsigned)ceil_div(c.h, 256));
  if (c.dtype == MOE_BF16)
    router_wgrad_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(x), src_token, offsets, dl_perm, c.h, dw_r, db_r);
  else
    router_wgrad_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(x), src_token,
                                                    offsets, dl_perm, c.h, dw_r, db_r);
  return cudaGetLastError();
}

template <typename T>
static cudaError_t bwd_combine_t(const moe_config_t& c, const void* dx_perm,
                                 const int32_t* dst_row, const void* dx_shared,
                                 const float* dl_topk, const int32_t* idx, const float* w_r,
                                 const float* dx_add, void* dx, float* dx_f32, int* status,
                                 cudaStream_t s) {
  const unsigned grid = (unsigned)c.T;
  const T* dp = static_cast<const T*>(dx_perm);
  const T* ds = static_cast<const T*>(dx_shared);
  T* o = static_cast<T*>(dx);
#define MOE_BWD_COMBINE(KM)                                                                    \
  bwd_combine_kernel<T, KM><<<grid, 128, 0, s>>>(dp, dst_row, ds, dl_topk, idx, w_r, dx_add,    \
                                                 c.T, c.K, c.E, c.h, o, dx_f32, status)
  if (c.K <= 2) MOE_BWD_COMBINE(2);
  else if (c.K <= 4) MOE_BWD_COMBINE(4);
  else if (c.K <= 8) MOE_BWD_COMBINE(8);
  else MOE_BWD_COMBINE(16);
#undef MOE_BWD_COMBINE
  return cudaGetLastError();
}

cudaError_t launch_bwd_combine(const moe_config_t& c, const void* dx_perm, const int32_t* dst_row,
                               const void* dx_shared, const float* dl_topk, const int32_t* idx,
                               const float* w_r, const float* dx_add, void* dx, float* dx_f32,
                               int sms, int* status, cudaStream_t s) {
  (void)sms;
  if (c.T == 0) return cudaSuccess;
  if (c.dtype == MOE_BF16)
    return bwd_combine_t<__nv_bfloat16>(c, dx_perm, dst_row, dx_shared, dl_topk, idx, w_r, dx_add,
                                        dx, dx_f32, status, s);
  return bwd_combine_t<float>(c, dx_perm, dst_row, dx_shared, dl_topk, idx, w_r, dx_add, dx,
                              dx_f32, status, s);
}

}  // namespace moe
