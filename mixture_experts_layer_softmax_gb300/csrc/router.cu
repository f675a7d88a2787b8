// Route: gating projection, scoring, top-k selection and normalisation.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (review),
// §2.2 "Router architecture": gating l = W_r^T x, softmax or sigmoid scoring,
// top-k selection; balancing by a selection-only bias (aux-loss-free) or by
// force-balanced routing; §5.1 keeps the router in FP32.  The skill page
// "emerging-techniques-moe-training" ("Top-2 Routing (Mixtral)") divides the
// selected scores by their sum (MOE_FLAG_RENORM).
//
// Kernels:
//  * bf16 tokens, E <= 8: router_tc_small (router_tc.cu), the whole route in
//    one launch on the tensor cores.
//  * other bf16 tokens: the gating GEMM runs on the tensor cores.  W_r
//    (fp32) is split exactly into three bf16 parts, w = hi + mid + lo (24
//    mantissa bits = 3 x 8), tiled so that each GEMM tile holds the three
//    parts of a group of experts; x (bf16, exact) times each part is exact in
//    fp32 and accumulates in fp32 in TMEM, and the tile's epilogue adds the
//    three sums.  Small batches cut the h reduction into slices whose partial
//    logits router_select adds in slice order (+ b_r) before selecting.
//  * fp32 tokens:
//  * router_fused_small: E <= 32.  One block stages W_r chunks in shared
//    memory; each warp accumulates the gating dot products of a few tokens,
//    reduces them across the warp (31 shuffles for 32 sums), then selects
//    top-k with warp shuffles.  One pass over x, no logits round trip.
//  * router_gemm: E > 32.  SIMT fp32 tiled GEMM logits = x W_r^T (+ b_r).
//  * router_select: warp per token top-k + probabilities on fp32 logits.
#include <float.h>

#include <algorithm>

#include "router_select.cuh"

namespace moe {

// ---- top-k on given logits: one warp per token --------------------------
// logits: [T, E] fp32; or, when parts is given, the tensor-core router's
// partial logits: slab s (s < nsplit, split_stride floats apart) holds [T, ldp];
// l = the slabs added in slab order (+ gate_bias), written to logits_out when
// that is given.
template <int J>
__global__ void __launch_bounds__(256) router_select_kernel(const float* __restrict__ logits,
                                                             const float* __restrict__ parts,
                                                             int ldp, int nsplit,
                                                             int64_t split_stride,
                                                             const float* __restrict__ gate_bias,
                                                             float* __restrict__ logits_out,
                                                             RouterArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= a.T) return;
  float l[J];
  if (parts) {
    // slab 0 for every slot, then one batch of loads per further slab
    const float* pr = parts + t * ldp;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int e = lane + 32 * j;
      l[j] = e < a.E ? __ldg(pr + e) : 0.f;
    }
    for (int sl = 1; sl < nsplit; ++sl) {
      const float* ps = pr + sl * split_stride;
      float v[J];
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        v[j] = e < a.E ? __ldg(ps + e) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < J; ++j) l[j] = __fadd_rn(l[j], v[j]);
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int e = lane + 32 * j;
      if (e < a.E) {
        if (gate_bias) l[j] = __fadd_rn(l[j], __ldg(gate_bias + e));
        if (logits_out) logits_out[t * a.E + e] = l[j];
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int e = lane + 32 * j;
      l[j] = e < a.E ? __ldg(logits + t * a.E + e) : 0.f;
    }
  }
  select_and_write<J>(l, (int)t, a, lane);
}

// The router weight split exactly into three bf16 parts, w = hi + mid + lo
// (hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid); each difference
// is exact in fp32), laid out for the gating GEMM's tiles: tile n has rows
// [hi of experts n*ept .. n*ept + ept - 1 | mid of the same | lo of the same |
// zeros up to bn].  Grid: x over groups of 4 weights of a row (h is a
// multiple of 8), y over expert slots (ntiles * ept: the slots past E get
// zero rows) and then the ntiles * (bn - 3 ept) padding rows.  Block (0, 0)
// also writes the one-group row offsets {0, T}.
__global__ void split_router_weight_kernel(const float* __restrict__ w_r, int E, int h, int ept,
                                           int bn, int ntiles, __nv_bfloat16* __restrict__ w3,
                                           int32_t* offs, int T) {
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    offs[0] = 0;
    offs[1] = T;
  }
  const int k = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (k >= h) return;
  const int y = blockIdx.y;
  const int slots = ntiles * ept;
  if (y < slots) {  // expert slot y: its hi, mid and lo rows
    const int64_t row0 = (int64_t)(y / ept) * bn + (y % ept);
    uint2 hv = make_uint2(0u, 0u), mv = hv, lv = hv;
    if (y < E) {
      const float4 w = __ldg(reinterpret_cast<const float4*>(w_r + (int64_t)y * h + k));
      const float wv[4] = {w.x, w.y, w.z, w.w};
      __nv_bfloat16 hi[4], mid[4], lo[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) split3_bf16(wv[j], hi[j], mid[j], lo[j]);
      hv = *reinterpret_cast<const uint2*>(hi);
      mv = *reinterpret_cast<const uint2*>(mid);
      lv = *reinterpret_cast<const uint2*>(lo);
    }
    *reinterpret_cast<uint2*>(w3 + row0 * h + k) = hv;
    *reinterpret_cast<uint2*>(w3 + (row0 + ept) * h + k) = mv;
    *reinterpret_cast<uint2*>(w3 + (row0 + 2 * ept) * h + k) = lv;
  } else {  // padding row r of tile n
    const int zrows = bn - 3 * ept;
    const int z = y - slots;
    const int64_t row = (int64_t)(z / zrows) * bn + 3 * ept + z % zrows;
    *reinterpret_cast<uint2*>(w3 + row * h + k) = make_uint2(0u, 0u);
  }
}

// ---- fused gating + top-k for E <= 32 ------------------------------------
// EP: padded expert count (8, 16 or 32); TPW = 32 / EP tokens per warp, so a
// warp reduces exactly 32 partial sums.
template <typename Tin, int EP>
__global__ void __launch_bounds__(256) router_fused_small_kernel(
    const Tin* __restrict__ x, const float* __restrict__ w_r, const float* __restrict__ gate_bias,
    float* __restrict__ logits_out, RouterArgs a, int hc) {
  constexpr int TPW = 32 / EP;
  constexpr int kWarps = 8;
  extern __shared__ float sw[];  // [EP][hc] chunk of W_r
  __shared__ float s_logit[kWarps][TPW][EP];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t t0 = ((int64_t)blockIdx.x * kWarps + warp) * TPW;
  float acc[TPW * EP];
#pragma unroll
  for (int i = 0; i < TPW * EP; ++i) acc[i] = 0.f;

  for (int c0 = 0; c0 < a.h; c0 += hc) {
    const int cw = min(hc, a.h - c0);
    __syncthreads();
    for (int i = threadIdx.x * 4; i < EP * hc; i += blockDim.x * 4) {
      const int e = i / hc, c = i % hc;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < a.E && c < cw) v = __ldg(reinterpret_cast<const float4*>(w_r + (int64_t)e * a.h + c0 + c));
      *reinterpret_cast<float4*>(sw + e * hc + c) = v;
    }
    __syncthreads();
    // each lane takes 4 consecutive columns, the warp strides by 128
    for (int c = lane * 4; c < cw; c += 128) {
      float wv[EP][4];
#pragma unroll
      for (int e = 0; e < EP; ++e) {
        const float4 q = *reinterpret_cast<const float4*>(sw + e * hc + c);
        wv[e][0] = q.x; wv[e][1] = q.y; wv[e][2] = q.z; wv[e][3] = q.w;
      }
#pragma unroll
      for (int u = 0; u < TPW; ++u) {
        const int64_t t = t0 + u;
        if (t >= a.T) continue;
        float xv[4];
        const Tin* px = x + t * a.h + c0 + c;
        if constexpr (sizeof(Tin) == 2) {
          const uint2 r = __ldg(reinterpret_cast<const uint2*>(px));
          const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
          const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
          xv[0] = __low2float(p0); xv[1] = __high2float(p0);
          xv[2] = __low2float(p1); xv[3] = __high2float(p1);
        } else {
          const float4 r = __ldg(reinterpret_cast<const float4*>(px));
          xv[0] = r.x; xv[1] = r.y; xv[2] = r.z; xv[3] = r.w;
        }
#pragma unroll
        for (int e = 0; e < EP; ++e)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[u * EP + e] = fmaf(xv[q], wv[e][q], acc[u * EP + e]);
      }
    }
  }
  // 32 sums across 32 lanes in 31 shuffles: lane l ends with sum #l.
  const unsigned FULL = 0xffffffffu;
#pragma unroll
  for (int off = 16, n = 32; off >= 1; off >>= 1, n >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? acc[i] : acc[i + n / 2];
      const float keep = upper ? acc[i + n / 2] : acc[i];
      acc[i] = keep + __shfl_xor_sync(FULL, send, off);
    }
  }
  {
    const int u = lane / EP, e = lane % EP;
    float v = acc[0];
    if (gate_bias && e < a.E) v += __ldg(gate_bias + e);
    s_logit[warp][u][e] = v;
    const int64_t t = t0 + u;
    if (logits_out && t < a.T && e < a.E) logits_out[t * a.E + e] = v;
  }
  __syncwarp();
#pragma unroll 1
  for (int u = 0; u < TPW; ++u) {
    const int64_t t = t0 + u;
    if (t >= a.T) break;
    float l[1] = {lane < EP ? s_logit[warp][u][lane] : 0.f};
    select_and_write<1>(l, (int)t, a, lane);
  }
}

// ---- SIMT fp32 gating GEMM for E > 32 -----------------------------------
// logits[T,E] = x[T,h] W_r[E,h]^T + b_r.  64x64 tile, BK = 32, 256 threads,
// 4x4 outputs per thread, operands transposed into shared memory.
template <typename Tin>
__global__ void __launch_bounds__(256) router_gemm_kernel(const Tin* __restrict__ x,
                                                          const float* __restrict__ w_r,
                                                          const float* __restrict__ gate_bias,
                                                          float* __restrict__ logits, int T, int E,
                                                          int h) {
  constexpr int BT = 64, BE = 64, BK = 32;
  __shared__ float xs[BK][BT + 4];
  __shared__ float ws[BK][BE + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t tb = (int64_t)blockIdx.y * BT;
  const int eb = blockIdx.x * BE;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < h; k0 += BK) {
    // x tile: 64 rows x 32 cols, 8 consecutive elements per thread
    {
      const int r = threadIdx.x >> 2, c = (threadIdx.x & 3) * 8;
      const int64_t t = tb + r;
      float v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = 0.f;
      if (t < T) {
        const Tin* p = x + t * h + k0 + c;
        if constexpr (sizeof(Tin) == 2) {
          if (k0 + c + 8 <= h) {
            const Vec<__nv_bfloat16> u = ldg16(reinterpret_cast<const __nv_bfloat16*>(p));
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = __bfloat162float(u.v[q]);
          }
        } else {
#pragma unroll
          for (int hq = 0; hq < 2; ++hq)
            if (k0 + c + 4 * hq + 4 <= h) {
              const float4 u = __ldg(reinterpret_cast<const float4*>(p + 4 * hq));
              v[4 * hq] = u.x; v[4 * hq + 1] = u.y; v[4 * hq + 2] = u.z; v[4 * hq + 3] = u.w;
            }
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) xs[c + q][r] = v[q];
    }
    // W tile: 64 experts x 32 cols
    {
      const int r = threadIdx.x >> 2, c = (threadIdx.x & 3) * 8;
      const int e = eb + r;
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {
        float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < E && k0 + c + 4 * hq + 4 <= h)
          u = __ldg(reinterpret_cast<const float4*>(w_r + (int64_t)e * h + k0 + c + 4 * hq));
        ws[c + 4 * hq][r] = u.x; ws[c + 4 * hq + 1][r] = u.y;
        ws[c + 4 * hq + 2][r] = u.z; ws[c + 4 * hq + 3][r] = u.w;
      }
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      const float4 av = *reinterpret_cast<const float4*>(&xs[kk][ty * 4]);
      const float4 bv = *reinterpret_cast<const float4*>(&ws[kk][tx * 4]);
      const float a4[4] = {av.x, av.y, av.z, av.w}, b4[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a4[i], b4[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t t = tb + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = eb + tx * 4 + j;
      if (e < E) logits[t * E + e] = acc[i][j] + (gate_bias ? __ldg(gate_bias + e) : 0.f);
    }
  }
}

// ---- host launchers -------------------------------------------------------
static RouterArgs make_args(const moe_config_t& c, const float* sel_bias, int32_t* idx,
                            float* prob, uint8_t* map) {
  RouterArgs a;
  a.T = c.T; a.E = c.E; a.K = c.K; a.h = c.h; a.score = c.score;
  a.renorm = (c.flags & MOE_FLAG_RENORM) != 0;
  a.force_balance = (c.flags & MOE_FLAG_FORCE_BALANCE) != 0;
  a.sel_bias = sel_bias; a.topk_idx = idx; a.topk_prob = prob; a.routing_map = map;
  return a;
}

static cudaError_t select_launch(const moe_config_t& c, const float* logits, const float* parts,
                                 int ldp, int nsplit, int64_t split_stride,
                                 const float* gate_bias, float* logits_out, RouterArgs a,
                                 cudaStream_t s) {
  const int blocks = (int)ceil_div(c.T, 8);
  const int J = (int)ceil_div(c.E, 32);
#define MOE_SELECT(JJ)                                                                  \
  router_select_kernel<JJ><<<blocks, 256, 0, s>>>(logits, parts, ldp, nsplit, split_stride, \
                                                   gate_bias, logits_out, a)
  switch (J) {
    case 1: MOE_SELECT(1); break;
    case 2: MOE_SELECT(2); break;
    case 3: case 4: MOE_SELECT(4); break;
    default: MOE_SELECT(8); break;
  }
#undef MOE_SELECT
  return cudaGetLastError();
}

cudaError_t launch_router_select(const moe_config_t& c, const float* logits, const float* sel_bias,
                                 int32_t* idx, float* prob, uint8_t* map, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  return select_launch(c, logits, nullptr, 0, 1, 0, nullptr, nullptr,
                       make_args(c, sel_bias, idx, prob, map), s);
}

template <typename Tin, int EP>
static cudaError_t launch_fused(const moe_config_t& c, const Tin* x, const float* w_r,
                                const float* gate_bias, float* logits, RouterArgs a,
                                cudaStream_t s) {
  constexpr int TPW = 32 / EP;
  const int hc = (8192 / EP) / 128 * 128;  // 32 KB of W_r per chunk
  const size_t smem = (size_t)EP * hc * sizeof(float);
  const int blocks = (int)ceil_div(c.T, 8 * TPW);
  router_fused_small_kernel<Tin, EP><<<blocks, 256, smem, s>>>(x, w_r, gate_bias, logits, a, hc);
  return cudaGetLastError();
}

cudaError_t launch_router_gemm_tc(int T, const void* x, int h, const void* w3, int E, int ept,
                                  int bn, float* logit_parts, int ldo, const int32_t* offsets,
                                  int ksplit, int64_t split_stride, int sms, int* status,
                                  cudaStream_t s);
bool router_tc_small_ok(const moe_config_t& c);
cudaError_t launch_router_tc_small(const moe_config_t& c, const void* x, const float* w_r,
                                   const float* gate_bias, float* logits, const RouterArgs& a,
                                   int32_t* hist, int sms, int* status, cudaStream_t s);

cudaError_t launch_chunk_hist(const moe_config_t& c, const int32_t* idx, int32_t* hist,
                              int* status, cudaStream_t s);

static cudaError_t launch_router_body(const moe_config_t& c, const void* x, const float* w_r,
                                      const float* gate_bias, const float* sel_bias,
                                      float* logits, int32_t* idx, float* prob, uint8_t* map,
                                      const RouterScratch& rs, int sms, int* status,
                                      cudaStream_t s);

// hist (or null): also leave the dispatch's per-chunk expert histograms of
// idx there -- from the one-launch router's epilogue when it runs, else by
// the dispatch's own histogram step right after the route.
cudaError_t launch_router(const moe_config_t& c, const void* x, const float* w_r,
                          const float* gate_bias, const float* sel_bias, float* logits,
                          int32_t* idx, float* prob, uint8_t* map, const RouterScratch& rs,
                          int sms, int* status, cudaStream_t s, int32_t* hist) {
  if (c.T == 0) return cudaSuccess;
  if (router_tc_small_ok(c)) {  // one launch: gating, slice sum, selection (and histograms)
    RouterArgs a = make_args(c, sel_bias, idx, prob, map);
    return launch_router_tc_small(c, x, w_r, gate_bias, logits, a, hist, sms, status, s);
  }
  cudaError_t e = launch_router_body(c, x, w_r, gate_bias, sel_bias, logits, idx, prob, map, rs,
                                     sms, status, s);
  if (e == cudaSuccess && hist) e = launch_chunk_hist(c, idx, hist, status, s);
  return e;
}

static cudaError_t launch_router_body(const moe_config_t& c, const void* x, const float* w_r,
                                      const float* gate_bias, const float* sel_bias,
                                      float* logits, int32_t* idx, float* prob, uint8_t* map,
                                      const RouterScratch& rs, int sms, int* status,
                                      cudaStream_t s) {
  RouterArgs a = make_args(c, sel_bias, idx, prob, map);
  if (c.dtype == MOE_BF16) {
    const int ept = router_ept(c.E), bn = router_bn(c.E);
    const int ntiles = router_ntiles(c.E);
    const dim3 grid((unsigned)ceil_div(c.h / 4, 256), (unsigned)(ntiles * (ept + bn - 3 * ept)));
    split_router_weight_kernel<<<grid, 256, 0, s>>>(w_r, c.E, c.h, ept, bn, ntiles, rs.w3, rs.offs,
                                                    c.T);
    const int64_t stride = (int64_t)c.T * rs.ldp;
    const int nsplit = router_ksplit(c, rs.ksplit, sms);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
      e = launch_router_gemm_tc(c.T, x, c.h, rs.w3, c.E, ept, bn, rs.parts, rs.ldp, rs.offs,
                                nsplit, stride, sms, status, s);
    if (e != cudaSuccess) return e;
    return select_launch(c, nullptr, rs.parts, rs.ldp, nsplit, stride, gate_bias, logits, a, s);
  }
  const float* xf = static_cast<const float*>(x);
  if (c.E <= 32) {
    const int EP = c.E <= 8 ? 8 : (c.E <= 16 ? 16 : 32);
    if (EP == 8) return launch_fused<float, 8>(c, xf, w_r, gate_bias, logits, a, s);
    if (EP == 16) return launch_fused<float, 16>(c, xf, w_r, gate_bias, logits, a, s);
    return launch_fused<float, 32>(c, xf, w_r, gate_bias, logits, a, s);
  }
  dim3 grid((unsigned)ceil_div(c.E, 64), (unsigned)ceil_div(c.T, 64));
  router_gemm_kernel<float><<<grid, 256, 0, s>>>(xf, w_r, gate_bias, logits, c.T, c.E, c.h);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_router_select(c, logits, sel_bias, idx, prob, map, s);
}

}  // namespace moe
