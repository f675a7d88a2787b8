// Load-balancing losses of the router and their logit gradients.
//
// Skill page "emerging-techniques-moe-training", "Load Balancing":
//   "Auxiliary Loss": f_e = fraction of the routed (token, slot) pairs that go
//   to expert e, P_e = mean over tokens of softmax(l_t)_e, aux = E sum_e f_e P_e;
//   "Router Z-Loss": z = mean over tokens of logsumexp(l_t)^2.
// The review page's training configuration weights the auxiliary loss by 1e-3.
// The fractions count a discrete selection and carry no gradient, so
//   d aux / d l_tj = (E / T) s_tj (f_j - sum_e f_e s_te),
//   d z / d l_tj   = (2 / T) lse_t s_tj,                 s_t = softmax(l_t).
//
// Three launches, every sum in a fixed order (bitwise reproducible):
//   1. aux_partials: block b takes a contiguous range of tokens, one warp per
//      token (lane l holds experts l, l + 32, ...); each warp accumulates, in
//      token order and in fp64, sum_t s_te and sum_t lse_t^2, and counts the
//      slots per expert; the block adds its 8 warps in warp order and writes
//      one partial row.
//   2. aux_finalize: one block adds the partial rows in block order, forms
//      f, P, aux and z, writes the two losses and f (for the gradient).
//   3. aux_grad (optional): one warp per token adds the weighted gradient of
//      both losses to the caller's dlogits.
#include "common.cuh"

namespace moe {

constexpr int kAuxWarps = 8;
constexpr int kAuxMaxJ = 8;  // E <= 256

// Numerically safe softmax pieces of one token spread over a warp: the row
// maximum, the sum of exp(l - max) and the log-sum-exp.
template <int J>
MOE_D void row_softmax_stats(const float (&l)[J], int E, int lane, float& m, float& sum,
                             float& lse) {
  m = -INFINITY;
#pragma unroll
  for (int j = 0; j < J; ++j)
    if (lane + 32 * j < E) m = fmaxf(m, l[j]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  sum = 0.f;
#pragma unroll
  for (int j = 0; j < J; ++j)
    if (lane + 32 * j < E) sum += expf(l[j] - m);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  lse = m + logf(sum);
}

template <int J>
__global__ void __launch_bounds__(256) aux_partials_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ idx, int T, int E, int K,
    int tokens_per_block, double* __restrict__ part_p, double* __restrict__ part_z,
    int32_t* __restrict__ part_cnt, int* status) {
  __shared__ double s_p[kAuxWarps][32 * kAuxMaxJ];
  __shared__ double s_z[kAuxWarps];
  __shared__ int32_t s_cnt[kAuxWarps][32 * kAuxMaxJ];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double accp[J], accz = 0.0;
  int cnt[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    accp[j] = 0.0;
    cnt[j] = 0;
  }
  const int64_t t0 = (int64_t)blockIdx.x * tokens_per_block;
  const int64_t t1 = min((int64_t)T, t0 + tokens_per_block);
  for (int64_t t = t0 + warp; t < t1; t += kAuxWarps) {
    float l[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int e = lane + 32 * j;
      l[j] = e < E ? __ldg(logits + t * E + e) : 0.f;
    }
    float m, sum, lse;
    row_softmax_stats<J>(l, E, lane, m, sum, lse);
    const float inv = 1.f / sum;
#pragma unroll
    for (int j = 0; j < J; ++j)
      if (lane + 32 * j < E) accp[j] += (double)(expf(l[j] - m) * inv);
    accz += (double)lse * (double)lse;  // the same on every lane
    // slots of this token routed to each expert: lane k reads slot k
    const int e_slot = lane < K ? __ldg(idx + t * K + lane) : -1;
    if (lane < K && (e_slot < 0 || e_slot >= E)) report(status, MOE_ERR_DEVICE_BOUNDS);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      if (k >= K) break;
      const int e = __shfl_sync(0xffffffffu, e_slot, k);
      if (e >= 0 && e < E && (e & 31) == lane) {
#pragma unroll
        for (int j = 0; j < J; ++j)
          if ((e >> 5) == j) ++cnt[j];
      }
    }
  }
#pragma unroll
  for (int j = 0; j < J; ++j) {
    s_p[warp][lane + 32 * j] = accp[j];
    s_cnt[warp][lane + 32 * j] = cnt[j];
  }
  if (lane == 0) s_z[warp] = accz;
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    double p = 0.0;
    int c = 0;
    for (int w = 0; w < kAuxWarps; ++w) {  // warp order
      p += s_p[w][e];
      c += s_cnt[w][e];
    }
    part_p[(int64_t)blockIdx.x * E + e] = p;
    part_cnt[(int64_t)blockIdx.x * E + e] = c;
  }
  if (threadIdx.x == 0) {
    double z = 0.0;
    for (int w = 0; w < kAuxWarps; ++w) z += s_z[w];
    part_z[blockIdx.x] = z;
  }
}

// One block of 256 threads: thread e sums expert e's partials over the blocks
// in block order; aux = E sum_e f_e P_e by a fixed shared-memory tree.
__global__ void __launch_bounds__(256) aux_finalize_kernel(
    const double* __restrict__ part_p, const double* __restrict__ part_z,
    const int32_t* __restrict__ part_cnt, int nblk, int T, int E, int K, float* __restrict__ f_out,
    float* __restrict__ losses) {
  __shared__ double s_fp[256];
  const int e = threadIdx.x;
  double fp = 0.0;
  if (e < E) {
    double p = 0.0;
    int64_t c = 0;
    for (int b = 0; b < nblk; ++b) {
      p += part_p[(int64_t)b * E + e];
      c += part_cnt[(int64_t)b * E + e];
    }
    const double f = (double)c / ((double)T * K);
    f_out[e] = (float)f;
    fp = f * (p / T);
  }
  s_fp[threadIdx.x] = fp;
  __syncthreads();
  for (int half = 128; half >= 1; half >>= 1) {
    if (threadIdx.x < half) s_fp[threadIdx.x] += s_fp[threadIdx.x + half];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    double z = 0.0;
    for (int b = 0; b < nblk; ++b) z += part_z[b];
    losses[0] = (float)(E * s_fp[0]);
    losses[1] = (float)(z / T);
  }
}

// One warp per token: dl[t, j] += ca (E / T) s_tj (f_j - sum_e f_e s_te)
//                                 + cz (2 / T) lse_t s_tj.
template <int J>
__global__ void __launch_bounds__(256) aux_grad_kernel(const float* __restrict__ logits,
                                                       const float* __restrict__ f, int T, int E,
                                                       float ca, float cz,
                                                       float* __restrict__ dlogits) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * kAuxWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  float l[J], s[J], fv[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int e = lane + 32 * j;
    l[j] = e < E ? __ldg(logits + t * E + e) : 0.f;
    fv[j] = e < E ? __ldg(f + e) : 0.f;
  }
  float m, sum, lse;
  row_softmax_stats<J>(l, E, lane, m, sum, lse);
  const float inv = 1.f / sum;
  float g = 0.f;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    s[j] = lane + 32 * j < E ? expf(l[j] - m) * inv : 0.f;
    g = fmaf(fv[j], s[j], g);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) g += __shfl_xor_sync(0xffffffffu, g, off);
  const float a = ca * (float)E / (float)T, zc = cz * 2.f * lse / (float)T;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int e = lane + 32 * j;
    if (e < E) dlogits[t * E + e] += a * s[j] * (fv[j] - g) + zc * s[j];
  }
}

cudaError_t launch_aux_loss(const moe_config_t& c, const float* logits, const int32_t* idx,
                            float ca, float cz, float* losses, float* dlogits, double* part_p,
                            double* part_z, int32_t* part_cnt, float* f, int* status,
                            cudaStream_t s) {
  if (c.T == 0) {
    return cudaMemsetAsync(losses, 0, 2 * sizeof(float), s);
  }
  const int nblk = aux_loss_blocks(c.T);
  const int tpb = (int)ceil_div(c.T, nblk);
  const int J = (int)ceil_div(c.E, 32);
  const int gblocks = (int)ceil_div(c.T, kAuxWarps);
#define MOE_AUX(JJ)                                                                            \
  do {                                                                                         \
    aux_partials_kernel<JJ><<<nblk, 256, 0, s>>>(logits, idx, c.T, c.E, c.K, tpb, part_p,      \
                                                 part_z, part_cnt, status);                    \
    aux_finalize_kernel<<<1, 256, 0, s>>>(part_p, part_z, part_cnt, nblk, c.T, c.E, c.K, f,     \
                                          losses);                                             \
    if (dlogits && (ca != 0.f || cz != 0.f))                                                   \
      aux_grad_kernel<JJ><<<gblocks, 256, 0, s>>>(logits, f, c.T, c.E, ca, cz, dlogits);       \
  } while (0)
  switch (J) {
    case 1: MOE_AUX(1); break;
    case 2: MOE_AUX(2); break;
    case 3: case 4: MOE_AUX(4); break;
    default: MOE_AUX(8); break;
  }
#undef MOE_AUX
  return cudaGetLastError();
}

}  // namespace moe

namespace moe {

// ---- dense router backward (for a logit gradient that is nonzero everywhere,
// like the two losses' gradients): C[m, n] (+)= sum_k A(k, m) B(k, n) in fp32,
// with A(k, m) = a[k * sak + m * sam] (fp32) and B(k, n) = b[k * ldb + n]
// (bf16 or fp32 rows).  64 x 128 tiles, 16-deep k chunks staged in shared
// memory, 256 threads with 4 x 8 outputs each, each output summed in k order
// by one thread (reproducible).  Used for dW_r = dl^T x (a = dl [T, E]:
// sak = E, sam = 1; colsum = db_r, the sums over k of A(k, m)) and
// dx_add = dl W_r (a = dl: sak = 1, sam = E).
template <typename TB>
__global__ void __launch_bounds__(256) dense_tn_gemm_kernel(
    const float* __restrict__ a, int64_t sak, int64_t sam, const TB* __restrict__ b, int64_t ldb,
    int M, int N, int Kd, float* __restrict__ c, int64_t ldc, bool accumulate,
    float* __restrict__ colsum) {
  constexpr int BM = 64, BN = 128, BK = 16;
  __shared__ float As[BK][BM];
  __shared__ float Bs[BK][BN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 x 16 threads
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  float acc[4][8] = {};
  float csum = 0.f;  // block column 0 only: sum over k of A(k, m) for m = m0 + threadIdx.x
  for (int k0 = 0; k0 < Kd; k0 += BK) {
    // A tile: 16 x 64 (4 per thread)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int li = threadIdx.x + i * 256;
      const int kk = li / BM, mm = li % BM;
      const int k = k0 + kk, m = m0 + mm;
      As[kk][mm] = (k < Kd && m < M) ? __ldg(a + (int64_t)k * sak + (int64_t)m * sam) : 0.f;
    }
    // B tile: 16 x 128 (8 per thread)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int li = threadIdx.x + i * 256;
      const int kk = li / BN, nn = li % BN;
      const int k = k0 + kk, n = n0 + nn;
      float v = 0.f;
      if (k < Kd && n < N) v = to_f32(b[(int64_t)k * ldb + n]);
      Bs[kk][nn] = v;
    }
    __syncthreads();
    if (colsum && blockIdx.x == 0 && threadIdx.x < BM) {
#pragma unroll
      for (int kk = 0; kk < BK; ++kk) csum += As[kk][threadIdx.x];
    }
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[4], bv[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 8; ++j) bv[j] = Bs[kk][tx * 8 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int n = n0 + tx * 8 + j;
      if (n >= N) continue;
      float* o = c + (int64_t)m * ldc + n;
      *o = accumulate ? *o + acc[i][j] : acc[i][j];
    }
  }
  if (colsum && blockIdx.x == 0 && threadIdx.x < BM && m0 + threadIdx.x < M) {
    float* o = colsum + m0 + threadIdx.x;
    *o = accumulate ? *o + csum : csum;
  }
}

// Adds the routed slots' logit gradient dl_topk [T, K] into the dense [T, E]
// one (the K experts of a token are distinct: one thread per element).
__global__ void scatter_topk_grad_kernel(const float* __restrict__ dl_topk,
                                         const int32_t* __restrict__ idx, int T, int K, int E,
                                         float* __restrict__ dl) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)T * K) return;
  const int e = __ldg(idx + i);
  if (e >= 0 && e < E) dl[(i / K) * E + e] += __ldg(dl_topk + i);
}

cudaError_t launch_scatter_topk_grad(const moe_config_t& c, const float* dl_topk,
                                     const int32_t* idx, float* dl, cudaStream_t s) {
  const int64_t n = (int64_t)c.T * c.K;
  if (n == 0) return cudaSuccess;
  scatter_topk_grad_kernel<<<(unsigned)ceil_div(n, 256), 256, 0, s>>>(dl_topk, idx, c.T, c.K, c.E,
                                                                      dl);
  return cudaGetLastError();
}

// dW_r [E,h] = dl^T x and db_r [E] = sum_t dl (when given) for a dense logit
// gradient dl [T, E] (fp32); both written, not accumulated.
cudaError_t launch_dense_router_wgrad(const moe_config_t& c, const float* dl, const void* x,
                                      float* dw_r, float* db_r, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const dim3 gw((unsigned)ceil_div(c.h, 128), (unsigned)ceil_div(c.E, 64));
  if (c.dtype == MOE_BF16)
    dense_tn_gemm_kernel<__nv_bfloat16><<<gw, 256, 0, s>>>(
        dl, c.E, 1, static_cast<const __nv_bfloat16*>(x), c.h, c.E, c.h, c.T, dw_r, c.h, false,
        db_r);
  else
    dense_tn_gemm_kernel<float><<<gw, 256, 0, s>>>(dl, c.E, 1, static_cast<const float*>(x), c.h,
                                                   c.E, c.h, c.T, dw_r, c.h, false, db_r);
  return cudaGetLastError();
}

// dx_add [T,h] = dl W_r (written).
cudaError_t launch_dense_router_dx(const moe_config_t& c, const float* dl, const float* w_r,
                                   float* dx_add, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const dim3 gx((unsigned)ceil_div(c.h, 128), (unsigned)ceil_div(c.T, 64));
  dense_tn_gemm_kernel<float><<<gx, 256, 0, s>>>(dl, 1, c.E, w_r, c.h, c.T, c.h, c.E, dx_add, c.h,
                                                 false, nullptr);
  return cudaGetLastError();
}

}  // namespace moe
