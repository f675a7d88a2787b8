// Route for bf16 tokens and E <= 8 experts in one launch on the tensor cores:
// gating GEMM, slice sum, top-k selection and probabilities.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (review),
// §2.2 "Router architecture" (l = W_r^T x, scores, top-k) and §5.1 (the router
// stays in FP32): W_r (fp32) is split exactly into three bf16 parts
// w = hi + mid + lo (24 mantissa bits = 3 x 8); x (bf16) times each part is
// exact in fp32 and accumulates in fp32 in TMEM, and each logit is formed as
// (lo + mid) + hi.
//
// The product is computed transposed, D = W3 x^T: the 24 split weight rows
// (hi of experts 0-7, mid, lo) are the MMA's A operand (M = 128; rows 24-127
// are whatever shared memory follows, their outputs are never read) and 256
// tokens are its N, so one M128 N256 K16 MMA consumes 8 KB of x (a tcgen05
// MMA costs about the same time at N = 32 as at N = 256).
//
// A cluster of four CTAs owns one tile of 256 tokens (the grid has one cluster
// per tile) and splits the h reduction: CTA r takes the r-th quarter of the K
// blocks of 64.  Per stage the TMA brings the tile's 256 x 64 bf16 slab of x
// (128-byte swizzle) and the 8 x 64 fp32 slab of W_r; the four epilogue warps
// split the W_r slab into the A operand (128-byte swizzled K-major, the layout
// the TMA would write) and the MMA warp issues four MMAs.  At the end the warp
// that may read TMEM lanes 0-31 copies rows 0-23 into the (now idle) x ring;
// every epilogue thread forms the slice's logits (lo + mid) + hi of two tokens
// and sends them to the CTA that finalises them (CTA q takes tokens
// 64 q .. 64 q + 63) through distributed shared memory; each CTA adds the four
// slices in slice order, adds b_r, writes the logits and selects top-k, one
// thread per token.
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 TMEM owner and MMA
// issuer, warps 2-5 W_r split during the main loop, then the epilogue.  Every
// wait is bounded; a wait that gives up records MOE_ERR_TIMEOUT, every role
// leaves its loop, copies and MMAs in flight are waited for, TMEM is freed.
#include <algorithm>

#include "router_select.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int kRCl = 4;                 // CTAs per cluster (slices of h)
constexpr int kRBN = 256, kRBK = 64;    // tokens per tile, K per stage
constexpr int kRFin = kRBN / kRCl;      // tokens each CTA finalises
constexpr int kRStages = 5;
constexpr int kRThreads = 192;
constexpr int kRX = kRBN * kRBK * 2;    // 32 KB of x per stage
constexpr int kRA = 24 * kRBK * 2;      // 3 KB: the split W_r rows of a stage
constexpr int kRW = 8 * kRBK * 4;       // 2 KB: the fp32 W_r slab
constexpr int kRDumpLd = kRBN + 4;      // floats per dumped TMEM row (16-B aligned, banks spread)

struct RCtl {
  uint64_t full[kRStages], aready[kRStages], empty[kRStages];
  uint64_t tmem_full, drain, dumped, xch_full;
  uint32_t tmem_base;
  int abort;
};

// Shared memory: [A parts: stages x 3 KB][x: stages x 32 KB][W_r: stages x
// 2 KB][slices of the tokens this CTA finalises: 4 x 64 x 8 fp32][control].
// The A operand of stage s spans 16 KB from its parts (M = 128 rows of 128 B),
// so it reads into the x ring: valid memory, unused rows.  After the main loop
// the x ring holds TMEM rows 0-23 (24 x kRDumpLd fp32).
constexpr int kROffX = kRStages * kRA;
constexpr int kROffW = kROffX + kRStages * kRX;
constexpr int kROffXch = kROffW + kRStages * kRW;
constexpr int kROffCtl = kROffXch + kRCl * kRFin * 8 * 4;
constexpr size_t kRSmem = 1024 + (size_t)kROffCtl + sizeof(RCtl);
static_assert(kROffX % 1024 == 0 && kROffW % 1024 == 0, "operand tiles must be 1024-B aligned");
static_assert((kRStages - 1) * kRA + 128 * 128 <= kROffW, "the A tile must stay in the ring");
static_assert(24 * kRDumpLd * 4 <= kRStages * kRX, "the TMEM rows fit in the x ring");

struct RouterTcParams {
  int T, h, E;
  const float* gate_bias;
  float* logits;
  int32_t* hist;  // [ceil(T/32)][E] per-chunk expert histograms of the selection, or null
  RouterArgs a;
  int* status;
};

// The 128-byte swizzle of a K-major tile with 128-byte rows: 16-byte chunk c of
// row r sits at chunk c ^ (r mod 8) (tile base 1024-byte aligned).
MOE_D uint32_t sw128_offset(int row, int byte_in_row) {
  return (uint32_t)(row * 128 + ((((byte_in_row >> 4) ^ (row & 7)) << 4) | (byte_in_row & 15)));
}

__global__ void __cluster_dims__(kRCl, 1, 1) __launch_bounds__(kRThreads, 1)
    router_tc_small_kernel(const __grid_constant__ CUtensorMap tmX,
                           const __grid_constant__ CUtensorMap tmW, const RouterTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sX = smem + kROffX;
  uint8_t* sW = smem + kROffW;
  float* dump = reinterpret_cast<float*>(sX);               // [24][kRDumpLd], after the main loop
  float* xch = reinterpret_cast<float*>(smem + kROffXch);   // [4 slices][64 tokens][8]
  RCtl& ctl = *reinterpret_cast<RCtl*>(smem + kROffCtl);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_ctarank();
  const int KB = (p.h + kRBK - 1) / kRBK;
  const int kb_lo = (int)(((int64_t)KB * rank) / kRCl);
  const int nkb = (int)(((int64_t)KB * (rank + 1)) / kRCl) - kb_lo;
  const int tile = blockIdx.x / kRCl;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      tc::mbar_init(tc::smem_u32(&ctl.full[s]), 1);
      tc::mbar_init(tc::smem_u32(&ctl.aready[s]), 4);
      tc::mbar_init(tc::smem_u32(&ctl.empty[s]), 1);
    }
    tc::mbar_init(tc::smem_u32(&ctl.tmem_full), 1);
    tc::mbar_init(tc::smem_u32(&ctl.drain), 1);
    tc::mbar_init(tc::smem_u32(&ctl.dumped), 32);
    // one arrival per sending warp (after __syncwarp, which orders the warp's
    // stores before its lane's release): three remote warps and this CTA's own
    tc::mbar_init(tc::smem_u32(&ctl.xch_full), kRCl);
    ctl.abort = 0;
    tc::fence_barrier_init();
    tc::fence_proxy_async_smem();
    tc::prefetch_tensormap(&tmX);
    tc::prefetch_tensormap(&tmW);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(&ctl.tmem_base), kRBN);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  tc::cluster_sync();  // every CTA's barriers exist before any remote arrive
  tc::fence_after_sync();
  const uint32_t tmem_base = ctl.tmem_base;
  tc::WaitCtl wc{p.status, &ctl.abort, 2000000000ull, 0};
  tc::WaitCtl wdrain{p.status, nullptr, 1000000000ull, 0};
  const unsigned FULL = 0xffffffffu;

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_par = 0;
      for (int kb = kb_lo; kb < kb_lo + nkb; ++kb) {
        if (!tc::mbar_wait(tc::smem_u32(&ctl.empty[stage]), phase ^ 1, wc)) break;
        const uint32_t fb = tc::smem_u32(&ctl.full[stage]);
        tc::mbar_arrive_expect_tx(fb, kRX + kRW);
        tc::tma_load_2d(tc::smem_u32(sX + stage * kRX), &tmX, kb * kRBK, tile * kRBN, fb);
        tc::tma_load_2d(tc::smem_u32(sW + stage * kRW), &tmW, kb * kRBK, 0, fb);
        issued |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        if (++stage == kRStages) { stage = 0; phase ^= 1; }
      }
      for (int s = 0; s < kRStages; ++s)  // copies in flight land before the block exits
        if ((issued >> s) & 1u)
          tc::mbar_wait(tc::smem_u32(&ctl.full[s]), (issued_par >> s) & 1u, wdrain);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(128, kRBN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kbl = 0; kbl < nkb; ++kbl) {
        if (!tc::mbar_wait(tc::smem_u32(&ctl.aready[stage]), phase, wc) ||
            !tc::mbar_wait(tc::smem_u32(&ctl.full[stage]), phase, wc)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t a0 = tc::smem_u32(sA + stage * kRA);
        const uint32_t b0 = tc::smem_u32(sX + stage * kRX);
#pragma unroll
        for (int k = 0; k < kRBK / 16; ++k)
          tc::mma_bf16(tmem_base, tc::desc_kmajor_sw128(a0 + k * 32),
                       tc::desc_kmajor_sw128(b0 + k * 32), idesc, (kbl | k) != 0);
        tc::mma_commit(tc::smem_u32(&ctl.empty[stage]));
        if (++stage == kRStages) { stage = 0; phase ^= 1; }
      }
      if (ok) tc::mma_commit(tc::smem_u32(&ctl.tmem_full));  // no MMAs (nkb = 0): arrives at once
      if (ctl.abort) {  // every issued MMA finishes before TMEM is freed
        tc::mma_commit(tc::smem_u32(&ctl.drain));
        tc::mbar_wait(tc::smem_u32(&ctl.drain), 0, wdrain);
      }
    }
    __syncwarp();
  } else {
    // ================= W_r split, then the epilogue (warps 2-5) =================
    const int ct = threadIdx.x - 64;              // 0 .. 127
    const int we = ct >> 4, wc4 = (ct & 15) * 4;  // this thread's W_r row and 4 columns
    const uint32_t xch_full = tc::smem_u32(&ctl.xch_full);
    const RouterArgs ra = p.a;  // a register copy (a reference to the parameter would go to local memory)
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int kbl = 0; kbl < nkb; ++kbl) {
      if (!__all_sync(FULL, tc::mbar_wait(tc::smem_u32(&ctl.full[stage]), phase, wc))) {
        ok = false;
        break;
      }
      const float4 wv = *reinterpret_cast<const float4*>(sW + stage * kRW + we * 256 + wc4 * 4);
      const float w4[4] = {wv.x, wv.y, wv.z, wv.w};
      __nv_bfloat16 hi[4], mid[4], lo[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) split3_bf16(w4[j], hi[j], mid[j], lo[j]);
      uint8_t* ast = sA + stage * kRA;
      const int byte = wc4 * 2;  // 8 bytes of each part row
      *reinterpret_cast<uint2*>(ast + sw128_offset(we, byte)) = *reinterpret_cast<const uint2*>(hi);
      *reinterpret_cast<uint2*>(ast + sw128_offset(8 + we, byte)) =
          *reinterpret_cast<const uint2*>(mid);
      *reinterpret_cast<uint2*>(ast + sw128_offset(16 + we, byte)) =
          *reinterpret_cast<const uint2*>(lo);
      tc::fence_proxy_async_smem();  // generic writes -> the MMA's async reads
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&ctl.aready[stage]));
      if (++stage == kRStages) { stage = 0; phase ^= 1; }
    }
    // ---- epilogue ----
    // TMEM lane m holds row m of W3 x^T: lanes e, 8 + e, 16 + e are the hi,
    // mid and lo sums of expert e, one column per token.  Only the warp with
    // warp % 4 == 0 may read lanes 0-31: it copies rows 0-23 to `dump` (the x
    // ring: every stage has been consumed once the accumulator is complete).
    if (ok && warp == 4) {
      if (__all_sync(FULL, tc::mbar_wait(tc::smem_u32(&ctl.tmem_full), 0, wc))) {
        tc::fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < kRBN / 32; ++c) {
          uint32_t r[32];
          if (nkb > 0) {
            tc::tmem_ld_32x32b_x32(tmem_base + c * 32, r);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = 0u;
          }
          if (lane < 24) {
            float4* d = reinterpret_cast<float4*>(dump + lane * kRDumpLd + c * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              d[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                 __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
          }
        }
        tc::fence_before_sync();
        tc::mbar_arrive(tc::smem_u32(&ctl.dumped));
      } else {
        ok = false;
      }
    }
    if (ok && __all_sync(FULL, tc::mbar_wait(tc::smem_u32(&ctl.dumped), 0, wc))) {
      // tokens 2 ct and 2 ct + 1 of the tile: this slice's logits (lo + mid) + hi,
      // sent to the CTA that finalises them (warp w's tokens belong to CTA w)
      float pl[2][8];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int tl = 2 * ct + u;
          pl[u][e] = __fadd_rn(
              __fadd_rn(dump[(16 + e) * kRDumpLd + tl], dump[(8 + e) * kRDumpLd + tl]),
              dump[e * kRDumpLd + tl]);
        }
      const int owner = ct >> 5;                 // 0 .. 3
      const int fl = 2 * ct - owner * kRFin;     // first of the two tokens, local to the owner
      float* slot = xch + (rank * kRFin + fl) * 8;  // slice `rank` of the owner's buffer
      if ((uint32_t)owner == rank) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          reinterpret_cast<float4*>(slot + 8 * u)[0] = make_float4(pl[u][0], pl[u][1], pl[u][2], pl[u][3]);
          reinterpret_cast<float4*>(slot + 8 * u)[1] = make_float4(pl[u][4], pl[u][5], pl[u][6], pl[u][7]);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(xch_full);
      } else {
        const uint32_t dst = tc::mapa(tc::smem_u32(slot), (uint32_t)owner);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          tc::st_cluster_f32x4(dst + 32 * u, pl[u][0], pl[u][1], pl[u][2], pl[u][3]);
          tc::st_cluster_f32x4(dst + 32 * u + 16, pl[u][4], pl[u][5], pl[u][6], pl[u][7]);
        }
        __syncwarp();
        if (lane == 0) tc::arrive_cluster(tc::mapa(xch_full, (uint32_t)owner));
      }
      // finalise this CTA's 64 tokens: thread ct < 64 takes token ct
      if (__all_sync(FULL, tc::mbar_wait_cluster(xch_full, 0, wc)) && ct < kRFin) {
        float l[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) l[e] = xch[ct * 8 + e];
#pragma unroll
        for (int r = 1; r < kRCl; ++r)  // slices in order
#pragma unroll
          for (int e = 0; e < 8; ++e) l[e] = __fadd_rn(l[e], xch[(r * kRFin + ct) * 8 + e]);
        if (p.gate_bias)
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (e < p.E) l[e] = __fadd_rn(l[e], __ldg(p.gate_bias + e));
        const int64_t t = (int64_t)tile * kRBN + rank * kRFin + ct;
        uint32_t taken = 0u;
        if (t < p.T) {
          if (p.logits) {
            float* lrow = p.logits + t * p.E;
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (e < p.E) lrow[e] = l[e];
          }
          taken = select_row8(l, (int)t, ra);
        }
        // the dispatch's chunk histogram: this warp's 32 tokens are exactly
        // one chunk of 32 (tiles and the 64-token quarters are chunk-aligned)
        if (p.hist) {
          const int64_t t0 = t - lane;
          int cnt = 0;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int ce = (int)__reduce_add_sync(FULL, (taken >> e) & 1u);
            if (lane == e) cnt = ce;
          }
          if (t0 < p.T && lane < p.E) p.hist[(t0 / 32) * p.E + lane] = cnt;
        }
      }
    }
  }
  tc::fence_before_sync();
  tc::cluster_sync();  // other CTAs may still touch this CTA's shared memory until here
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, kRBN);
  }
}

}  // namespace

// bf16 tokens, E <= 8, h a multiple of 8 (TMA row strides are multiples of 16 bytes).
bool router_tc_small_ok(const moe_config_t& c) {
  return c.dtype == MOE_BF16 && c.E >= 1 && c.E <= 8 && c.h % 8 == 0 && c.h > 0;
}

cudaError_t launch_router_tc_small(const moe_config_t& c, const void* x, const float* w_r,
                                   const float* gate_bias, float* logits, const RouterArgs& a,
                                   int32_t* hist, int sms, int* status, cudaStream_t s) {
  (void)sms;  // one cluster per tile, whatever the SM count
  if (c.T == 0) return cudaSuccess;
  if (!router_tc_small_ok(c)) return cudaErrorInvalidValue;
  tc::EncodeTiledFn fn = tc::encode_tiled_fn();
  if (!fn) return cudaErrorInvalidValue;
  CUtensorMap mx, mw;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)c.h, (cuuint64_t)c.T};
    const cuuint64_t strides[1] = {(cuuint64_t)c.h * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kRBK, (cuuint32_t)kRBN};
    const cuuint32_t estr[2] = {1, 1};
    if (fn(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)c.h, (cuuint64_t)c.E};
    const cuuint64_t strides[1] = {(cuuint64_t)c.h * 4};
    const cuuint32_t box[2] = {(cuuint32_t)kRBK, 8u};  // rows past E read as zero
    const cuuint32_t estr[2] = {1, 1};
    if (fn(&mw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(w_r), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  RouterTcParams p;
  p.T = c.T; p.h = c.h; p.E = c.E;
  p.gate_bias = gate_bias; p.logits = logits; p.hist = hist; p.a = a; p.status = status;
  cudaError_t e = cudaFuncSetAttribute(router_tc_small_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRSmem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = ceil_div(c.T, kRBN);  // one cluster per tile
  if (tiles * kRCl > 0x7fffffff) return cudaErrorInvalidValue;
  router_tc_small_kernel<<<(unsigned)(tiles * kRCl), kRThreads, kRSmem, s>>>(mx, mw, p);
  return cudaGetLastError();
}

}  // namespace moe
