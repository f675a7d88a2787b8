// Internal helpers shared by the library's translation units (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

#define MOE_HD __host__ __device__ __forceinline__
#define MOE_D __device__ __forceinline__

namespace moe {

constexpr int kWarp = 32;

// Status word codes written on the device (same values as moe_status_t).
MOE_D void report(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---- element conversions ------------------------------------------------
MOE_D float to_f32(float v) { return v; }
MOE_D float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> MOE_D T from_f32(float v);
template <> MOE_D float from_f32<float>(float v) { return v; }
template <> MOE_D __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// 16-byte vector of elements: 4 fp32 or 8 bf16.
template <typename T> struct Vec;
template <> struct Vec<float> {
  static constexpr int N = 4;
  float v[4];
};
template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __nv_bfloat16 v[8];
};

template <typename T> MOE_D Vec<T> ldg16(const T* p) {
  Vec<T> r;
  *reinterpret_cast<uint4*>(&r) = __ldg(reinterpret_cast<const uint4*>(p));
  return r;
}
// Streaming load that does not allocate in L1 (data read once).
template <typename T> MOE_D Vec<T> ld16_stream(const T* p) {
  Vec<T> r;
  uint4 u;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
               : "l"(p));
  *reinterpret_cast<uint4*>(&r) = u;
  return r;
}
template <typename T> MOE_D void st16(T* p, const Vec<T>& v) {
  *reinterpret_cast<uint4*>(p) = *reinterpret_cast<const uint4*>(&v);
}

MOE_HD int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
MOE_HD size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Exact GELU (erf form) and SiLU in fp32.  erff/expf are CUDA's own.
MOE_D float gelu_f(float z) { return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f)); }
MOE_D float sigmoid_f(float z) { return 1.0f / (1.0f + expf(-z)); }
MOE_D float silu_f(float z) { return z * sigmoid_f(z); }

// Scratch of the tensor-core router (in the workspace): w3 [3E, h] bf16 (the
// exactly split router weight), parts [T, ldp] fp32 partial logits, offs [2].
struct RouterScratch {
  __nv_bfloat16* w3;
  float* parts;
  int ldp;
  int32_t* offs;
};

// ---- workspace layout ----------------------------------------------------
// One layout per config, shared by every entry point, so the backward can find
// what a SAVE_FOR_BWD forward left behind.
struct Workspace {
  size_t router_w3, router_parts, router_off, logits, topk_idx, topk_prob, hist, chunk_base, counts, offsets, dst_row, src_token,
      perm_prob, x_perm, act_save, a, y_perm, shared_off, shared_h, shared_a, shared_y,
      // backward (MOE_FLAG_SAVE_FOR_BWD only)
      dy_perm, dh, dx_perm, dprob_part, dprob_perm, dl_topk, dl_perm, shared_dh, shared_dx,
      total;
};

inline size_t elem_bytes(int dtype) { return dtype == MOE_BF16 ? 2 : 4; }

inline Workspace workspace_layout(const moe_config_t& c) {
  Workspace w{};
  const size_t T = (size_t)c.T, h = (size_t)c.h, E = (size_t)c.E, K = (size_t)c.K,
               F = (size_t)c.F;
  const size_t P = T * K, eb = elem_bytes(c.dtype);
  const size_t R1 = c.act == MOE_ACT_SWIGLU ? 2 * F : F;
  const size_t NC = (T + 31) / 32;
  const bool save = (c.flags & MOE_FLAG_SAVE_FOR_BWD) != 0;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t ldp = (3 * E + 7) / 8 * 8;
  const bool tc_router = c.dtype == MOE_BF16;
  w.router_w3 = take(tc_router ? 3 * E * h * 2 : 0);
  w.router_parts = take(tc_router ? T * ldp * 4 : 0);
  w.router_off = take(2 * 4);
  w.logits = take(T * E * 4);
  w.topk_idx = take(P * 4);
  w.topk_prob = take(P * 4);
  w.hist = take(NC * E * 4);
  w.chunk_base = take(NC * E * 4);
  w.counts = take(E * 4);
  w.offsets = take((E + 1) * 4);
  w.dst_row = take(P * 4);
  w.src_token = take(P * 4);
  w.perm_prob = take(P * 4);
  w.x_perm = take(P * h * eb);
  w.act_save = take(save ? P * R1 * eb : 0);
  w.a = take(P * F * eb);
  w.y_perm = take(P * h * eb);
  w.shared_off = take(2 * 4);
  w.shared_h = take(c.n_shared && save ? T * R1 * eb : 0);
  w.shared_a = take(c.n_shared ? T * F * eb : 0);
  w.shared_y = take(c.n_shared ? T * h * eb : 0);
  const size_t NT = (F + 255) / 256;  // N tiles of the FC2 data-gradient GEMM
  w.dy_perm = take(save ? P * h * eb : 0);
  w.dh = take(save ? P * R1 * eb : 0);
  w.dx_perm = take(save ? P * h * eb : 0);
  w.dprob_part = take(save ? P * NT * 4 : 0);
  w.dprob_perm = take(save ? P * 4 : 0);
  w.dl_topk = take(save ? P * 4 : 0);
  w.dl_perm = take(save ? P * 4 : 0);
  w.shared_dh = take(save && c.n_shared ? T * R1 * eb : 0);
  w.shared_dx = take(save && c.n_shared ? T * h * eb : 0);
  w.total = off;
  return w;
}

}  // namespace moe
