// Grouped expert GEMMs on the SIMT FMA units (fp32 configurations, and a
// cross-check path for bf16).
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (review),
// §2.1 "Expert computation" (all local experts in one grouped GEMM call) and
// §4.1.1 memory-efficient permutation (p applied before the second linear
// layer when the expert has no bias).  Expert FFNs follow the skill page
// "emerging-techniques-moe-training" (Linear -> GELU -> Linear with biases)
// and the SwiGLU expert (silu(gate) * up, bias-free).
//
// Grid: x = m-blocks over all experts (an upper bound, P/64 + E, computed on
// the host without reading the device offsets; blocks past the real count
// exit), y = n-blocks.  Each block scans the offsets to find its expert.
#include "common.cuh"

namespace moe {

enum GemmMode { kFc1SwiGLU = 0, kFc1Gelu = 1, kFc2 = 2 };

struct SimtArgs {
  const void* A;       // [P, Kd] rows in expert order
  const void* B;       // [E][Nb][Kd]
  const void* bias;    // FC1: b1 [E][F]; FC2: b2 [E][h]; or null
  const float* prob;   // [P] or null
  const int32_t* offsets;
  void* out;           // FC1: a [P, F]; FC2: y_perm [P, h]
  void* act_save;      // FC1: H [P, Nb] or null
  int E, Kd, N, Nb;    // N output columns; Nb rows of B per expert (2F for SwiGLU)
  int prob_here;       // apply p in this GEMM's epilogue
};

template <int BM>
MOE_D int find_group(const int32_t* offsets, int E, int b, int* s_mb, int& row0, int& row_end) {
  // s_mb[e] = first m-block of expert e; computed by the 256-thread block.
  __shared__ int s_warp[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int total = 0;
  for (int e0 = 0; e0 < E; e0 += 256) {
    const int e = e0 + threadIdx.x;
    const int m = e < E ? __ldg(offsets + e + 1) - __ldg(offsets + e) : 0;
    const int v = (m + BM - 1) / BM;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int wbase = 0, bsum = 0;
    for (int w = 0; w < 8; ++w) {
      if (w < warp) wbase += s_warp[w];
      bsum += s_warp[w];
    }
    if (e < E) s_mb[e] = total + wbase + incl - v;
    total += bsum;
    __syncthreads();
  }
  if (threadIdx.x == 0) s_mb[E] = total;
  __syncthreads();
  if (b >= total) return -1;
  int lo = 0, hi = E - 1;  // largest e with s_mb[e] <= b
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_mb[mid] <= b) lo = mid; else hi = mid - 1;
  }
  // skip empty experts that share the same start
  int e = lo;
  while (e + 1 < E && s_mb[e + 1] <= b) ++e;
  row0 = __ldg(offsets + e) + (b - s_mb[e]) * BM;
  row_end = __ldg(offsets + e + 1);
  return e;
}

template <typename T>
MOE_D void load4(const T* p, float* v) {
  if constexpr (sizeof(T) == 2) {
    const uint2 r = __ldg(reinterpret_cast<const uint2*>(p));
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
    v[0] = __low2float(a); v[1] = __high2float(a); v[2] = __low2float(b); v[3] = __high2float(b);
  } else {
    const float4 r = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w;
  }
}

template <typename T, int MODE>
__global__ void __launch_bounds__(256) grouped_gemm_simt_kernel(SimtArgs g) {
  constexpr int BM = 64, BN = 64, BK = 16;
  constexpr int NB = MODE == kFc1SwiGLU ? 2 * BN : BN;  // B rows per tile
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][NB + 4];
  __shared__ int s_mb[257];
  int row0 = 0, row_end = 0;
  const int e = find_group<BM>(g.offsets, g.E, blockIdx.x, s_mb, row0, row_end);
  if (e < 0) return;
  const int n0 = blockIdx.y * BN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const T* A = static_cast<const T*>(g.A);
  const T* B = static_cast<const T*>(g.B) + (int64_t)e * g.Nb * g.Kd;
  float acc[4][4] = {}, acc2[4][4] = {};
  for (int k0 = 0; k0 < g.Kd; k0 += BK) {
    {  // A: 64 x 16, 4 per thread
      const int r = threadIdx.x >> 2, c = (threadIdx.x & 3) * 4;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      const int64_t row = (int64_t)row0 + r;
      if (row < row_end && k0 + c + 4 <= g.Kd) load4(A + row * g.Kd + k0 + c, v);
#pragma unroll
      for (int q = 0; q < 4; ++q) As[c + q][r] = v[q];
    }
#pragma unroll
    for (int part = 0; part < NB / 64; ++part) {  // B: NB x 16
      const int r = threadIdx.x >> 2, c = (threadIdx.x & 3) * 4;
      const int n = n0 + r;
      // SwiGLU: rows [0,64) of the tile are gate rows n, [64,128) up rows F + n
      const int brow = part == 0 ? n : g.N + n;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (n < g.N && k0 + c + 4 <= g.Kd) load4(B + (int64_t)brow * g.Kd + k0 + c, v);
#pragma unroll
      for (int q = 0; q < 4; ++q) Bs[c + q][part * 64 + r] = v[q];
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 av = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 bv = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float a4[4] = {av.x, av.y, av.z, av.w}, b4[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a4[i], b4[j], acc[i][j]);
      if constexpr (MODE == kFc1SwiGLU) {
        const float4 uv = *reinterpret_cast<const float4*>(&Bs[kk][64 + tx * 4]);
        const float u4[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc2[i][j] = fmaf(a4[i], u4[j], acc2[i][j]);
      }
    }
    __syncthreads();
  }
  // epilogue
  T* out = static_cast<T*>(g.out);
  T* save = static_cast<T*>(g.act_save);
  const T* bias = static_cast<const T*>(g.bias);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t row = (int64_t)row0 + ty * 4 + i;
    if (row >= row_end) continue;
    const float p = (g.prob && g.prob_here) ? __ldg(g.prob + row) : 1.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= g.N) continue;
      float o;
      if constexpr (MODE == kFc1SwiGLU) {
        const float gt = acc[i][j], up = acc2[i][j];
        if (save) {
          save[row * g.Nb + n] = from_f32<T>(gt);
          save[row * g.Nb + g.N + n] = from_f32<T>(up);
        }
        o = p * (silu_f(gt) * up);
      } else if constexpr (MODE == kFc1Gelu) {
        float hv = acc[i][j];
        if (bias) hv += to_f32(bias[(int64_t)e * g.N + n]);
        if (save) save[row * g.Nb + n] = from_f32<T>(hv);
        o = p * gelu_f(hv);
      } else {
        float yv = acc[i][j];
        if (bias) yv += to_f32(bias[(int64_t)e * g.N + n]);
        o = p * yv;
      }
      out[row * g.N + n] = from_f32<T>(o);
    }
  }
}

template <typename T>
static cudaError_t launch_simt_t(const SimtArgs& g, int mode, int P, cudaStream_t s) {
  const int64_t mblocks = ceil_div(P, 64) + g.E;
  dim3 grid((unsigned)mblocks, (unsigned)ceil_div(g.N, 64));
  if (mode == kFc1SwiGLU) grouped_gemm_simt_kernel<T, kFc1SwiGLU><<<grid, 256, 0, s>>>(g);
  else if (mode == kFc1Gelu) grouped_gemm_simt_kernel<T, kFc1Gelu><<<grid, 256, 0, s>>>(g);
  else grouped_gemm_simt_kernel<T, kFc2><<<grid, 256, 0, s>>>(g);
  return cudaGetLastError();
}

// One of the two expert GEMMs (fc = 1: x_perm -> a, fc = 2: a -> y_perm).
cudaError_t launch_expert_gemm_simt(const moe_config_t& c, int fc, int P, const void* A,
                                    const int32_t* offsets, const float* prob, const void* w,
                                    const void* bias, void* act_save, void* out, cudaStream_t s) {
  if (P == 0) return cudaSuccess;
  const bool swiglu = c.act == MOE_ACT_SWIGLU;
  const bool prob_after = c.has_bias != 0;  // with b2, p multiplies the FC2 output
  SimtArgs g{};
  g.A = A; g.B = w; g.bias = bias; g.prob = prob; g.offsets = offsets; g.out = out; g.E = c.E;
  int mode;
  if (fc == 1) {
    g.act_save = act_save; g.Kd = c.h; g.N = c.F; g.Nb = swiglu ? 2 * c.F : c.F;
    g.prob_here = !prob_after;
    mode = swiglu ? kFc1SwiGLU : kFc1Gelu;
  } else {
    g.act_save = nullptr; g.Kd = c.F; g.N = c.h; g.Nb = c.h;
    g.prob_here = prob_after;
    mode = kFc2;
  }
  return c.dtype == MOE_BF16 ? launch_simt_t<__nv_bfloat16>(g, mode, P, s)
                             : launch_simt_t<float>(g, mode, P, s);
}

}  // namespace moe
