// MXFP8 expert GEMMs: E4M3 operands with one E8M0 scale per 1 x 32 block
// along K, block-scaled MMAs on the 5th-generation tensor cores
// (tcgen05.mma kind::mxf8f6f4, scales in TMEM), fp32 accumulate.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (review),
// §5.3.3 "MXFP8 (Blackwell)": activations and weights both quantised in 1 x 32
// blocks with E8M0 scale factors, native to the Blackwell tensor cores; §5.4
// "Dynamic shape alignment" (MXFP8 GEMM dimensions aligned to 32).  Element
// and scale rules are the OCP Microscaling v1.0 ones that MXFP8 names: shared
// exponent X = floor(log2 max|x|) - 8, element = x / 2^X rounded to nearest
// even and saturated to +-448.
//
// Operand format (written by mxfp8_quantize_kernel or by the FC1 epilogue):
//   codes  [rows, K] uint8 (E4M3), row-major like the bf16 tensor;
//   scales in "scale atoms": the rows of each group (expert) are cut into
//     128-row tiles, numbered group after group (tile t of group g is
//     rtile[g] + t, rtile = exclusive scan of ceil(rows_g / 128)); atom
//     (tile, kb) = 512 bytes holding the scales of the tile's 128 rows for
//     K columns kb*128 .. kb*128+127 (4 blocks of 32): row i, block j at
//     byte 16 (i % 32) + 4 (i / 32) + j; atoms ordered (tile, kb), kb fastest.
//   One atom is what one tcgen05.cp 32x128b.warpx4 moves into TMEM (lane
//   quarter w, column c + i / 32 of lane 32 w + i % 32 holding row i's 4
//   block scales), the layout the block-scaled MMA reads with scale id j.
//
// GEMM kernel (persistent, 1 CTA per SM, 320 threads):
//   warp 0     TMA producer: 4 stages of {A 128 x 128 B, B 256 x 128 B}
//              (128-byte swizzle) plus the stage's three scale atoms (bulk
//              copies), one mbarrier per stage.
//   warp 1     TMEM owner and MMA issuer: per stage, tcgen05.cp of the
//              scale atoms into TMEM columns of the stage, then 4 MMAs
//              M128 N256 K32 with scale ids 0..3; one 256-column fp32
//              accumulator (TMEM also holds 4 stages x 16 scale columns).
//   warps 2-9  epilogue, two warps per TMEM lane quarter, each taking half
//              of the tile's columns: TMEM -> registers 32 columns at a
//              time; a warp releases the accumulator right after its last
//              read, so the next tile's MMAs overlap the math and stores.
//   FC1 (SwiGLU): B holds 128 gate rows and the matching 128 up rows;
//   a = p * silu(gate) * up is stored as bf16 and/or re-quantised in place
//   (each 32-column chunk of a thread's row is one MXFP8 block of FC2's A
//   operand; the tile's 128 columns fill exactly one scale atom).
//   FC2: plain output, bf16.
// Every wait is bounded; a wait that gives up records MOE_ERR_TIMEOUT and
// every role leaves its loop as in the bf16 kernels.
#include <cuda_fp8.h>

#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int BM = 128, BN = 256, BK = 128;  // BK: K elements (= bytes) per stage
constexpr int A_BYTES = BM * BK;             // 16 KB
constexpr int B_BYTES = BN * BK;             // 32 KB
constexpr int ATOM = 512;                    // one scale atom
constexpr int SF_BYTES = 3 * ATOM;           // A atom + two B atoms
constexpr int STAGES = 4;
constexpr int kThreads = 320;  // producer, MMA, 8 epilogue warps
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_COL0 = 256, SF_STRIDE = 16;  // per stage: A scales +0..3, B +8..15

enum MxMode { kMxSwiGLU = 0, kMxPlain = 1 };

struct MxParams {
  const int32_t* offsets;  // [E+1]
  const float* prob;       // FC1: [P] or null
  const uint8_t* a_sf;     // A scale atoms
  const uint8_t* b_sf;     // B scale atoms (uniform groups of Nb rows)
  __nv_bfloat16* out;      // [P, N] bf16 or null
  uint8_t* out_q;          // FC1: codes of a [P, N] or null
  uint8_t* out_sf;         // FC1: scale atoms of a
  int E, Kd, N, Nb;
  int* status;
  uint64_t wait_limit_ns;
};

struct MxCtl {
  uint64_t full[STAGES], empty[STAGES], tmem_full, tmem_empty, drain;
  uint32_t tmem_base;
  int abort;
  int tile_start[257];  // GEMM tiles before expert e
  int rtile[257];       // 128-row tiles before expert e (scale atom numbering)
  int off[257];
};

constexpr size_t kSmem = 1024 + (size_t)STAGES * (A_BYTES + B_BYTES + SF_BYTES) + sizeof(MxCtl);

// ---- E8M0 / E4M3 helpers ------------------------------------------------------
// E8M0 code of a block with maximum magnitude amax (finite fp32):
// X + 127 with X = floor(log2 amax) - 8 clamped at -127; amax's biased
// exponent field e gives floor(log2 amax) = e - 127 for normal amax, and a zero
// or subnormal amax (field 0) lands on the clamp.
MOE_D uint32_t e8m0_code(float amax) {
  const uint32_t e = (__float_as_uint(amax) >> 23) & 0xFFu;
  return e > 8u ? e - 8u : 0u;
}
// 2^-X for scale code c (X = c - 127): the fp32 with exponent field 254 - c.
MOE_D float e8m0_inverse(uint32_t c) { return __uint_as_float((254u - c) << 23); }

// 8 values (already divided by the scale) -> 8 E4M3 codes, round to nearest
// even with saturation (cvt.rn.satfinite through cuda_fp8.h).
MOE_D uint2 e4m3x8(const float* v) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = __nv_cvt_float2_to_fp8x2(make_float2(v[2 * i], v[2 * i + 1]), __NV_SATFINITE, __NV_E4M3);
  return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

MOE_D uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Byte offset of row i's scale word (blocks j = 0..3) in atom (tile, kb).
MOE_HD int64_t atom_word(int64_t tile, int KB, int kb, int i) {
  return (tile * KB + kb) * ATOM + 16 * (i & 31) + 4 * (i >> 5);
}

// ---- quantiser ------------------------------------------------------------------
// One 16-thread group per (row, 128-column chunk): each thread converts 8
// consecutive values, 4 threads share a 32-value block (amax by shuffles),
// and the group's first thread writes the chunk's 4 scale codes as one word.
// Groups: offsets [G+1] on the device, or uniform groups of `urows` rows.
__global__ void __launch_bounds__(256)
    mxfp8_quantize_kernel(const __nv_bfloat16* __restrict__ x, int rows, int K, int G,
                          const int32_t* __restrict__ offsets, int urows,
                          uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  __shared__ int s_off[257], s_rt[257];
  if (offsets) {
    for (int g = threadIdx.x; g <= G; g += blockDim.x) s_off[g] = __ldg(offsets + g);
    __syncthreads();
    if (threadIdx.x < 32) {  // rtile = exclusive scan of ceil(rows_g / 128)
      const int lane = threadIdx.x;
      int running = 0;
      for (int g0 = 0; g0 < G; g0 += 32) {
        const int g = g0 + lane;
        const int v = g < G ? (s_off[g + 1] - s_off[g] + 127) / 128 : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        if (g < G) s_rt[g] = running + incl - v;
        running += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    __syncthreads();
  }
  const int KB = K / BK;
  const int lane = threadIdx.x & 31;
  const int sub = lane & 15;  // thread within the 16-thread group
  const int64_t chunks = (int64_t)rows * KB;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
  // every lane of a warp runs the same iterations (two chunks per warp), so
  // the shuffles below always see the whole warp
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); 2 * w < chunks;
       w += nwarps) {
    const int64_t ch = 2 * w + (lane >> 4);
    const bool valid = ch < chunks;
    const int r = valid ? (int)(ch / KB) : 0;
    const int kb = valid ? (int)(ch - (int64_t)r * KB) : 0;
    const int64_t base = (int64_t)r * K + kb * BK + sub * 8;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (valid) raw = __ldg(reinterpret_cast<const uint4*>(x + base));
    const __nv_bfloat16* xv = reinterpret_cast<const __nv_bfloat16*>(&raw);
    float v[8], amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] = __bfloat162float(xv[i]);
      amax = fmaxf(amax, fabsf(v[i]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const uint32_t code = e8m0_code(amax);
    const float inv = e8m0_inverse(code);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] *= inv;  // exact: a power of two
    // the chunk's 4 block codes (threads 0, 4, 8, 12 of the group) -> one word
    const uint32_t c1 = __shfl_down_sync(0xffffffffu, code, 4);
    const uint32_t c2 = __shfl_down_sync(0xffffffffu, code, 8);
    const uint32_t c3 = __shfl_down_sync(0xffffffffu, code, 12);
    if (!valid) continue;
    *reinterpret_cast<uint2*>(q + base) = e4m3x8(v);
    if (sub == 0) {
      int i;
      int64_t tile;
      if (offsets) {
        if (r < s_off[0] || r >= s_off[G]) continue;  // a row of no group: no scale atom
        int lo = 0, hi = G - 1;  // the group holding row r: last g with off[g] <= r
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (s_off[mid] <= r) lo = mid; else hi = mid - 1;
        }
        const int lr = r - s_off[lo];
        tile = s_rt[lo] + lr / 128;
        i = lr & 127;
      } else {
        const int g = r / urows;
        const int lr = r - g * urows;
        tile = (int64_t)g * ((urows + 127) / 128) + lr / 128;
        i = lr & 127;
      }
      *reinterpret_cast<uint32_t*>(sf + atom_word(tile, KB, kb, i)) =
          code | (c1 << 8) | (c2 << 16) | (c3 << 24);
    }
  }
}

// ---- dispatch with the quantisation fused in ------------------------------------
// One warp per token (grid-stride): the token row x[t] (bf16, h columns) is
// read once, quantised to MXFP8 (lanes 4j..4j+3 share a 32-value block, lanes
// 16c..16c+15 a 128-column chunk), and its codes and scale words are written
// to each of its K destination rows dst_row[t, k] of the permuted operand
// (the scale atom of row r of expert e: tile rtile[e] + (r - off[e]) / 128).
// Dropped slots (dst_row -1) are skipped; other out-of-range rows or expert
// ids are reported (MOE_ERR_DEVICE_BOUNDS) and skipped.
template <int KMAX>
__global__ void __launch_bounds__(256)
    scatter_quantize_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ idx,
                            const int32_t* __restrict__ dst_row,
                            const int32_t* __restrict__ offsets, int T, int K, int E, int h,
                            uint8_t* __restrict__ q, uint8_t* __restrict__ sf, int* status) {
  __shared__ int s_off[257], s_rt[257];
  for (int g = threadIdx.x; g <= E; g += blockDim.x) s_off[g] = __ldg(offsets + g);
  __syncthreads();
  if (threadIdx.x < 32) {  // rtile = exclusive scan of ceil(rows_e / 128)
    const int lane = threadIdx.x;
    int running = 0;
    for (int g0 = 0; g0 < E; g0 += 32) {
      const int g = g0 + lane;
      const int v = g < E ? (s_off[g + 1] - s_off[g] + 127) / 128 : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (g < E) s_rt[g] = running + incl - v;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int KB = h / BK;
  const int nvec = h / 8;  // 16-byte vectors per row
  const int64_t P = (int64_t)T * K;
  constexpr int kMaxVec = 4;
  for (int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); t < T; t += (int64_t)gridDim.x * 8) {
    int64_t row[KMAX], atom0[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      row[k] = -1;
      if (k < K) {
        const int r = __ldg(dst_row + t * K + k);
        const int e = __ldg(idx + t * K + k);
        if (r >= 0 && r < P && e >= 0 && e < E && r >= s_off[e] && r < s_off[e + 1]) {
          const int lr = r - s_off[e];
          row[k] = r;
          atom0[k] = atom_word(s_rt[e] + lr / 128, KB, 0, lr & 127);
        } else if (r != -1) {
          report(status, MOE_ERR_DEVICE_BOUNDS);
        }
      }
    }
    const __nv_bfloat16* src = x + t * h;
    for (int v0 = 0; v0 < nvec; v0 += 32 * kMaxVec) {
      uint4 raw[kMaxVec];
#pragma unroll
      for (int i = 0; i < kMaxVec; ++i) {
        const int v = v0 + i * 32 + lane;
        raw[i] = make_uint4(0, 0, 0, 0);
        if (v < nvec) raw[i] = __ldg(reinterpret_cast<const uint4*>(src) + v);
      }
#pragma unroll
      for (int i = 0; i < kMaxVec; ++i) {
        const int v = v0 + i * 32 + lane;
        const __nv_bfloat16* xv = reinterpret_cast<const __nv_bfloat16*>(&raw[i]);
        float f[8], amax = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          f[j] = __bfloat162float(xv[j]);
          amax = fmaxf(amax, fabsf(f[j]));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const uint32_t code = e8m0_code(amax);
        const float inv = e8m0_inverse(code);
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] *= inv;
        const uint2 c8 = e4m3x8(f);
        const uint32_t c1 = __shfl_down_sync(0xffffffffu, code, 4);
        const uint32_t c2 = __shfl_down_sync(0xffffffffu, code, 8);
        const uint32_t c3 = __shfl_down_sync(0xffffffffu, code, 12);
        const uint32_t word = code | (c1 << 8) | (c2 << 16) | (c3 << 24);
        if (v < nvec) {
#pragma unroll
          for (int k = 0; k < KMAX; ++k) {
            if (row[k] < 0) continue;
            *reinterpret_cast<uint2*>(q + row[k] * h + (int64_t)v * 8) = c8;
            if ((lane & 15) == 0)
              *reinterpret_cast<uint32_t*>(sf + atom0[k] + (int64_t)(v >> 4) * ATOM) = word;
          }
        }
      }
    }
  }
}

// ---- GEMM -------------------------------------------------------------------------
MOE_D void decode_tile(const MxCtl& c, int E, int nblk, int tile, int& e, int& mb, int& nb) {
  int lo = 0, hi = E - 1;  // largest e with tile_start[e] <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (c.tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  e = lo;
  const int local = tile - c.tile_start[e];
  const int mblk = (c.off[e + 1] - c.off[e] + BM - 1) / BM;
  nb = local / mblk;
  mb = local - nb * mblk;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_mxfp8_kernel(const __grid_constant__ CUtensorMap tmA,
                              const __grid_constant__ CUtensorMap tmB, const MxParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + STAGES * A_BYTES;
  uint8_t* sSF = sB + STAGES * B_BYTES;
  MxCtl& ctl = *reinterpret_cast<MxCtl*>(sSF + STAGES * SF_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const int nblk = MODE == kMxSwiGLU ? (p.N + 127) / 128 : (p.N + BN - 1) / BN;
  const int KB = p.Kd / BK;
  const int nbt = p.Nb / 128;  // B row tiles per expert

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(tc::smem_u32(&ctl.full[s]), 1);
      tc::mbar_init(tc::smem_u32(&ctl.empty[s]), 1);
    }
    tc::mbar_init(tc::smem_u32(&ctl.tmem_full), 1);
    tc::mbar_init(tc::smem_u32(&ctl.tmem_empty), 8);
    tc::mbar_init(tc::smem_u32(&ctl.drain), 1);
    ctl.abort = 0;
    tc::fence_barrier_init();
    tc::fence_proxy_async_smem();
    tc::prefetch_tensormap(&tmA);
    tc::prefetch_tensormap(&tmB);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(&ctl.tmem_base), TMEM_COLS);
    tc::tmem_relinquish();
  }
  for (int e = threadIdx.x; e <= E; e += kThreads) ctl.off[e] = __ldg(p.offsets + e);
  __syncthreads();
  if (warp == 2) {  // tile_start and rtile: exclusive scans over the experts
    int run_t = 0, run_r = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int mblk = e < E ? (ctl.off[e + 1] - ctl.off[e] + BM - 1) / BM : 0;
      int it = mblk * nblk, ir = mblk;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, it, o);
        const int r = __shfl_up_sync(0xffffffffu, ir, o);
        if (lane >= o) { it += t; ir += r; }
      }
      if (e < E) {
        ctl.tile_start[e] = run_t + it - mblk * nblk;
        ctl.rtile[e] = run_r + ir - mblk;
      }
      run_t += __shfl_sync(0xffffffffu, it, 31);
      run_r += __shfl_sync(0xffffffffu, ir, 31);
    }
    if (lane == 0) ctl.tile_start[E] = run_t;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = ctl.tmem_base;
  const int total = ctl.tile_start[E];
  tc::WaitCtl wc{p.status, &ctl.abort, p.wait_limit_ns, 0};
  tc::WaitCtl wdrain{p.status, nullptr, 1000000000ull, 0};

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_par = 0;
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        int e, mb, nb;
        decode_tile(ctl, E, nblk, tile, e, mb, nb);
        const int a_row = ctl.off[e] + mb * BM;
        const int64_t a_atom = (int64_t)(ctl.rtile[e] + mb) * KB;
        int b_row0, b_row1;
        int64_t b_atom0, b_atom1;
        bool two_b = true;
        if (MODE == kMxSwiGLU) {  // gate rows nb*128.., up rows N + nb*128..
          b_row0 = e * p.Nb + nb * 128;
          b_row1 = e * p.Nb + p.N + nb * 128;
          b_atom0 = ((int64_t)e * nbt + nb) * KB;
          b_atom1 = ((int64_t)e * nbt + p.N / 128 + nb) * KB;
        } else {
          b_row0 = e * p.Nb + nb * BN;
          b_row1 = b_row0 + 128;
          b_atom0 = ((int64_t)e * nbt + 2 * nb) * KB;
          b_atom1 = b_atom0 + KB;
          two_b = nb * BN + 128 < p.N;  // a half past N has no scale atom to read
        }
        const uint32_t tx = A_BYTES + B_BYTES + (two_b ? 3 : 2) * ATOM;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc::mbar_wait(tc::smem_u32(&ctl.empty[stage]), phase ^ 1, wc)) { ok = false; break; }
          const uint32_t fb = tc::smem_u32(&ctl.full[stage]);
          tc::mbar_arrive_expect_tx(fb, tx);
          const uint32_t a_dst = tc::smem_u32(sA + stage * A_BYTES);
          const uint32_t b_dst = tc::smem_u32(sB + stage * B_BYTES);
          const uint32_t sf_dst = tc::smem_u32(sSF + stage * SF_BYTES);
          tc::tma_load_2d(a_dst, &tmA, kb * BK, a_row, fb);
          tc::tma_load_2d(b_dst, &tmB, kb * BK, b_row0, fb);
          tc::tma_load_2d(b_dst + B_BYTES / 2, &tmB, kb * BK, b_row1, fb);
          tc::bulk_load(sf_dst, p.a_sf + (a_atom + kb) * ATOM, ATOM, fb);
          tc::bulk_load(sf_dst + ATOM, p.b_sf + (b_atom0 + kb) * ATOM, ATOM, fb);
          if (two_b) tc::bulk_load(sf_dst + 2 * ATOM, p.b_sf + (b_atom1 + kb) * ATOM, ATOM, fb);
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u)
          tc::mbar_wait(tc::smem_u32(&ctl.full[s]), (issued_par >> s) & 1u, wdrain);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        if (!tc::mbar_wait(tc::smem_u32(&ctl.tmem_empty), acc_phase ^ 1, wc)) break;
        tc::fence_after_sync();
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc::mbar_wait(tc::smem_u32(&ctl.full[stage]), phase, wc)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t a0 = tc::smem_u32(sA + stage * A_BYTES);
          const uint32_t b0 = tc::smem_u32(sB + stage * B_BYTES);
          const uint32_t sf0 = tc::smem_u32(sSF + stage * SF_BYTES);
          const uint32_t sfa = tmem_base + SF_COL0 + stage * SF_STRIDE;
          const uint32_t sfb = sfa + 8;
          tc::tmem_cp_32x128b_warpx4(sfa, tc::desc_sf_atom(sf0));
          tc::tmem_cp_32x128b_warpx4(sfb, tc::desc_sf_atom(sf0 + ATOM));
          tc::tmem_cp_32x128b_warpx4(sfb + 4, tc::desc_sf_atom(sf0 + 2 * ATOM));
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            tc::mma_mxf8(tmem_base, tc::desc_kmajor_sw128(a0 + k * 32),
                         tc::desc_kmajor_sw128(b0 + k * 32), tc::idesc_mxf8_e4m3(BM, BN, k, k), sfa,
                         sfb, (kb | k) != 0);
          tc::mma_commit(tc::smem_u32(&ctl.empty[stage]));
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc::mma_commit(tc::smem_u32(&ctl.tmem_full));
        acc_phase ^= 1;
      }
      if (ctl.abort) {  // let every issued MMA finish before TMEM is freed
        tc::mma_commit(tc::smem_u32(&ctl.drain));
        tc::mbar_wait(tc::smem_u32(&ctl.drain), 0, wdrain);
      }
    }
    __syncwarp();
  } else {
    // ================= epilogue (warps 2..9) =================
    // two warps per TMEM lane quarter, each taking half of the tile's columns;
    // each releases the accumulator as soon as its TMEM reads are done
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int hf = (warp - 2) >> 2;  // which half of the columns
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int e, mb, nb;
      decode_tile(ctl, E, nblk, tile, e, mb, nb);
      if (!tc::mbar_wait(tc::smem_u32(&ctl.tmem_full), acc_phase, wc)) break;
      tc::fence_after_sync();
      const int m_e = ctl.off[e + 1] - ctl.off[e];
      const int i = q * 32 + lane;  // row within the tile
      const bool valid = mb * BM + i < m_e;
      const int64_t row = (int64_t)ctl.off[e] + mb * BM + i;
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16);
      if (MODE == kMxSwiGLU) {
        // columns: gate hf*64 .. +63 and the matching up columns (two 32-wide chunks)
        const float pr = (p.prob && valid) ? __ldg(p.prob + row) : 1.f;
        // all of this warp's TMEM reads first (gate and up, two 32-column
        // chunks each), then the release, then the math: the next tile's MMAs
        // need not wait for the SiLU evaluations
        uint32_t g[2][32], u[2][32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col = hf * 64 + c * 32;
          tc::tmem_ld_32x32b_x32(tbase + col, g[c]);
          tc::tmem_ld_32x32b_x32(tbase + 128 + col, u[c]);
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&ctl.tmem_empty));
        float a[2][32];
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j)
            a[c][j] = pr * (silu_f(__uint_as_float(g[c][j])) * __uint_as_float(u[c][j]));
        uint32_t codes = 0;  // this warp's 2 of the row's 4 block scales
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int n = nb * 128 + hf * 64 + c * 32;
          if (valid && p.out) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint4 w;
              w.x = pack_bf16x2(a[c][j], a[c][j + 1]);
              w.y = pack_bf16x2(a[c][j + 2], a[c][j + 3]);
              w.z = pack_bf16x2(a[c][j + 4], a[c][j + 5]);
              w.w = pack_bf16x2(a[c][j + 6], a[c][j + 7]);
              *reinterpret_cast<uint4*>(p.out + row * p.N + n + j) = w;
            }
          }
          if (p.out_q) {
            float amax = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(a[c][j]));
            const uint32_t code = e8m0_code(amax);
            const float inv = e8m0_inverse(code);
#pragma unroll
            for (int j = 0; j < 32; ++j) a[c][j] *= inv;
            codes |= code << (8 * c);
            if (valid) {
              const uint2 c0 = e4m3x8(a[c]), c1 = e4m3x8(a[c] + 8), c2 = e4m3x8(a[c] + 16),
                          c3 = e4m3x8(a[c] + 24);
              uint8_t* dst = p.out_q + row * p.N + n;
              *reinterpret_cast<uint4*>(dst) = make_uint4(c0.x, c0.y, c1.x, c1.y);
              *reinterpret_cast<uint4*>(dst + 16) = make_uint4(c2.x, c2.y, c3.x, c3.y);
            }
          }
        }
        if (p.out_q)  // FC2's A operand: atom (rtile[e] + mb, kb = nb), row i, blocks 2 hf, 2 hf + 1
          *reinterpret_cast<uint16_t*>(
              p.out_sf + atom_word(ctl.rtile[e] + mb, p.N / 128, nb, i) + 2 * hf) =
              (uint16_t)(valid ? codes : 0u);
      } else {
        // columns hf*128 .. +127: all four 32-column loads first, then release
        uint32_t r[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tmem_ld_32x32b_x32(tbase + hf * 128 + c * 32, r[c]);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&ctl.tmem_empty));
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int n = nb * BN + hf * 128 + c * 32;
          if (valid && n < p.N) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(r[c][j]), __uint_as_float(r[c][j + 1]));
              w.y = pack_bf16x2(__uint_as_float(r[c][j + 2]), __uint_as_float(r[c][j + 3]));
              w.z = pack_bf16x2(__uint_as_float(r[c][j + 4]), __uint_as_float(r[c][j + 5]));
              w.w = pack_bf16x2(__uint_as_float(r[c][j + 6]), __uint_as_float(r[c][j + 7]));
              *reinterpret_cast<uint4*>(p.out + row * p.N + n + j) = w;
            }
          }
        }
      }
      acc_phase ^= 1;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---- host side ----------------------------------------------------------------------
// 2-D uint8 [rows, cols] map with a {128, 128} box, 128-byte swizzle, zero fill.
bool encode_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  tc::EncodeTiledFn fn = tc::encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {(cuuint32_t)BK, 128};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t mxfp8_scale_bytes(int64_t rows, int K, int groups) {
  return (size_t)(ceil_div(rows, 128) + groups) * (K / BK) * ATOM;
}

cudaError_t launch_mxfp8_quantize(int rows, int K, int groups, const int32_t* offsets,
                                  const void* x, uint8_t* q, uint8_t* sf, int sms,
                                  cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int64_t chunks = (int64_t)rows * (K / BK);
  const int64_t blocks = ceil_div(chunks, 2 * (256 / 32));
  const int grid = (int)(blocks < 8LL * sms ? blocks : 8LL * sms);
  mxfp8_quantize_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), rows, K, groups,
                                             offsets, offsets ? 0 : rows / groups, q, sf);
  return cudaGetLastError();
}

cudaError_t launch_scatter_quantize(const moe_config_t& c, const void* x, const int32_t* idx,
                                    const int32_t* dst_row, const int32_t* offsets, uint8_t* q,
                                    uint8_t* sf, int sms, int* status, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const int64_t need = ceil_div(c.T, 8);
  const int grid = (int)(need < 8LL * sms ? need : 8LL * sms);
  const __nv_bfloat16* xs = static_cast<const __nv_bfloat16*>(x);
#define MOE_SQ(KM) \
  scatter_quantize_kernel<KM><<<grid, 256, 0, s>>>(xs, idx, dst_row, offsets, c.T, c.K, c.E, c.h, q, sf, status)
  if (c.K <= 2) MOE_SQ(2);
  else if (c.K <= 4) MOE_SQ(4);
  else if (c.K <= 8) MOE_SQ(8);
  else MOE_SQ(16);
#undef MOE_SQ
  return cudaGetLastError();
}

// One MXFP8 grouped GEMM.  swiglu (FC1): A = x_perm codes [P, Kd], B = W1
// codes [E * 2N, Kd] (gate rows then up rows per expert), out = a [P, N]
// bf16 (or null) and/or out_q / out_sf = a re-quantised for FC2; p scales a.
// Plain (FC2): B = W2 codes [E * N, Kd], out [P, N] bf16.
cudaError_t launch_grouped_gemm_mxfp8(bool swiglu, int P, const uint8_t* A, const uint8_t* A_sf,
                                      int Kd, const uint8_t* B, const uint8_t* B_sf, int Nb,
                                      int E, int N, const int32_t* offsets, const float* prob,
                                      void* out, uint8_t* out_q, uint8_t* out_sf, int sms,
                                      int* status, cudaStream_t s) {
  if (P == 0) return cudaSuccess;
  CUtensorMap ma, mb;
  if (!encode_u8(&ma, A, (uint64_t)P, (uint64_t)Kd)) return cudaErrorInvalidValue;
  if (!encode_u8(&mb, B, (uint64_t)E * Nb, (uint64_t)Kd)) return cudaErrorInvalidValue;
  MxParams p{};
  p.offsets = offsets; p.prob = prob; p.a_sf = A_sf; p.b_sf = B_sf;
  p.out = static_cast<__nv_bfloat16*>(out); p.out_q = out_q; p.out_sf = out_sf;
  p.E = E; p.Kd = Kd; p.N = N; p.Nb = Nb;
  p.status = status;
  p.wait_limit_ns = 2000000000ull;
  const int nblk = swiglu ? (N + 127) / 128 : (N + BN - 1) / BN;
  const int64_t tiles_max = (ceil_div(P, BM) + E) * (int64_t)nblk;
  const int grid = (int)(tiles_max < sms ? tiles_max : sms);
  auto kern = swiglu ? grouped_gemm_mxfp8_kernel<kMxSwiGLU> : grouped_gemm_mxfp8_kernel<kMxPlain>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, kSmem, s>>>(ma, mb, p);
  return cudaGetLastError();
}

}  // namespace moe
