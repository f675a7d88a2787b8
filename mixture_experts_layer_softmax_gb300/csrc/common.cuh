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
// The exact three-way bf16 split of an fp32 value: hi = bf16(w),
// mid = bf16(w - hi), lo = bf16(w - hi - mid); each difference is exact in
// fp32 and w = hi + mid + lo (8 + 8 + 8 mantissa bits).
MOE_D void split3_bf16(float w, __nv_bfloat16& hi, __nv_bfloat16& mid, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(w);
  const float r1 = w - __bfloat162float(hi);
  mid = __float2bfloat16_rn(r1);
  lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
}

MOE_D float gelu_f(float z) { return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f)); }
MOE_D float sigmoid_f(float z) { return 1.0f / (1.0f + expf(-z)); }
MOE_D float silu_f(float z) { return z * sigmoid_f(z); }

// Scratch of the tensor-core router (in the workspace): w3 [ntiles * bn, h]
// bf16 (the exactly split router weight, tiled as router_ept describes),
// parts [ksplit][T, ldp] fp32 partial logits (one slab per slice of the h
// reduction; ksplit = room for at most that many slices), offs [2].
struct RouterScratch {
  __nv_bfloat16* w3;
  float* parts;
  int ldp;
  int ksplit;
  int32_t* offs;
};

// Tiles of the tensor-core gating GEMM: each N tile covers `ept` experts as
// three column groups (the hi, mid and lo parts of the exactly split fp32
// router weight), so its epilogue can add them; bn = 3 ept rounded up to a
// tcgen05 N (a multiple of 16).
inline int router_ept(int E) { return E <= 8 ? 8 : (E <= 16 ? 16 : (E <= 32 ? 32 : 64)); }
inline int router_bn(int E) {
  const int ept = router_ept(E);
  return ept == 8 ? 32 : (ept == 16 ? 48 : (ept == 32 ? 96 : 192));
}
inline int router_ntiles(int E) { return (E + router_ept(E) - 1) / router_ept(E); }
inline int router_parts_ld(int E) { return (E + 7) / 8 * 8; }

// The gating GEMM's h reduction may be cut into slices (split-K), each
// writing its own fp32 partial logits (E per token) that the selection kernel
// adds in slice order.  router_ksplit_max bounds the slices by the config
// alone (it sizes the workspace): at most 8, at most one per 64-wide K block,
// and only while the partial logits stay small next to the token row they
// come from (at most half its bytes).
inline int router_ksplit_max(const moe_config_t& c) {
  const int64_t kb = ((int64_t)c.h + 63) / 64;
  const int64_t row_bytes = (int64_t)c.h * (c.dtype == MOE_BF16 ? 2 : 4);
  int64_t s = row_bytes / (2 * 4 * (int64_t)router_parts_ld(c.E));
  if (s > 8) s = 8;
  if (s > kb) s = kb;
  return s < 1 ? 1 : (int)s;
}
// The slice count used on a GPU with `sms` SMs: the fewest slices that
// minimise (waves of tiles) x (K blocks per slice) + 2 per extra slice (the
// selection kernel reads one more slab of partial logits per slice).
inline int router_ksplit(const moe_config_t& c, int smax, int sms) {
  if (c.T <= 0 || sms <= 0) return 1;
  const int64_t tiles = ((int64_t)c.T + 127) / 128 * router_ntiles(c.E);
  const int64_t kb = ((int64_t)c.h + 63) / 64;
  int best = 1;
  int64_t best_cost = -1;
  for (int s = 1; s <= smax; ++s) {
    const int64_t per = (kb + s - 1) / s;
    if ((kb + per - 1) / per != s) continue;  // some slice would be empty
    const int64_t waves = (tiles * s + sms - 1) / sms;
    const int64_t cost = waves * per + 2 * (s - 1);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// Blocks of the load-balancing-loss partial sums: about 64 tokens each, at
// most 512 (their partial rows live in the workspace).
inline int aux_loss_blocks(int T) {
  const int64_t nb = ((int64_t)T + 63) / 64;
  return (int)(nb < 512 ? (nb > 0 ? nb : 1) : 512);
}

// ---- workspace layout ----------------------------------------------------
// One layout per config, shared by every entry point, so the backward can find
// what a SAVE_FOR_BWD forward left behind.
struct Workspace {
  size_t router_w3, router_parts, router_off, logits, topk_idx, topk_prob, hist, chunk_base,
      counts, offsets, dst_row, src_token, perm_prob, aux_part_p, aux_part_z, aux_part_cnt, aux_f,
      aux_losses, aux_dl, aux_dx, x_perm, act_save, a, y_perm, shared_off, shared_h, shared_a, shared_y,
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
  const size_t ldp = (size_t)router_parts_ld(c.E);
  const bool tc_router = c.dtype == MOE_BF16;
  w.router_w3 = take(tc_router ? (size_t)router_ntiles(c.E) * router_bn(c.E) * h * 2 : 0);
  w.router_parts = take(tc_router ? (size_t)router_ksplit_max(c) * T * ldp * 4 : 0);
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
  const size_t NB = (size_t)aux_loss_blocks(c.T);
  w.aux_part_p = take(NB * E * 8);
  w.aux_part_z = take(NB * 8);
  w.aux_part_cnt = take(NB * E * 4);
  w.aux_f = take(E * 4);
  const bool lb = c.aux_loss_coeff != 0.f || c.z_loss_coeff != 0.f;
  w.aux_losses = take(2 * 4);
  w.aux_dl = take((lb || c.capacity > 0) && save ? T * E * 4 : 0);  // dense router gradient
  w.aux_dx = take(lb && save ? T * h * 4 : 0);
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
