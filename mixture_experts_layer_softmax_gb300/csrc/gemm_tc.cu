// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// operands staged by TMA.  bf16 in, fp32 accumulate, bf16 out.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (review),
// §2.1 "Expert computation" (every local expert in one grouped GEMM call) and
// §4.3.1 (grouped GEMM); §4.1.1 memory-efficient permutation: for bias-free
// experts the routing weight p scales the activation in the FC1 epilogue, so
// FC2 is a plain GEMM; with expert biases p scales the FC2 output instead.
//
// One persistent CTA per SM walks a device-side tile list (no host sync: the
// per-expert row offsets are read on the device, review §4.3.3).  Tiles are
// 128 rows x 256 accumulator columns; an expert's rows start a new tile, so a
// tile never mixes experts (rows past the expert's end are computed and
// dropped).  Tiles are ordered expert by expert, m fastest, so the CTAs that
// run at the same time share one weight panel and one activation panel in L2.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: 4-stage ring of {A 128x64, B 256x64} bf16 tiles
//               (128-byte swizzle), completion on mbarriers (expect_tx).
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma M128 N256 K16, fp32
//               accumulators in TMEM, double buffered (2 x 256 columns), so the
//               epilogue of tile i overlaps the main loop of tile i+1.
//   warps 2-5   epilogue: tcgen05.ld 32 lanes x 32 columns, activation / bias /
//               probability, bf16 stores.
// SwiGLU FC1 tiles load 128 gate rows and the matching 128 up rows of W1, so
// silu(gate) * up is formed from two columns of the same thread's TMEM lane.
//
// Every wait is bounded (time limit); a wait that gives up records
// MOE_ERR_TIMEOUT, every role leaves its loop, the producer waits (bounded) for
// its copies in flight, the MMA issuer for its MMAs, and TMEM is freed.

#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int BM = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB

// Tile width BN (accumulator columns; 256 for the expert GEMMs, narrower for
// the router's few output columns) fixes the B stage size, the ring depth
// that fits in ~200 KB of shared memory, and the TMEM double buffer (2 x BN).
constexpr uint32_t pow2_at_least(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}
template <int BNT>
struct Tile {
  static constexpr int BN = BNT;
  static constexpr int B_BYTES = BNT * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (200 * 1024 / STAGE_BYTES) < 8 ? (200 * 1024 / STAGE_BYTES) : 8;
  static constexpr uint32_t TMEM_COLS = pow2_at_least(2 * BNT);  // allocations are powers of 2
};

enum TcMode { kTcSwiGLU = 0, kTcGelu = 1, kTcFc2 = 2, kTcF32 = 3 };

// Epilogue warps per CTA: FC1's SwiGLU/GELU epilogue writes more per tile
// than the others and gets two warps per TMEM lane quarter (each storing half
// of the quarter's columns), so that it keeps up with tiles of short K; the
// CTA is the producer, the MMA issuer and the epilogue warps.
MOE_HD constexpr int epi_warps(int mode) { return mode == kTcSwiGLU || mode == kTcGelu ? 8 : 4; }
MOE_HD constexpr int cta_threads(int mode) { return 32 * (2 + epi_warps(mode)); }

struct TcParams {
  const int32_t* offsets;        // [E+1]
  const __nv_bfloat16* xg;       // gather mode: token rows [*, Kd]
  const int32_t* src_token;      // gather mode: token of each permuted row
  const float* prob;             // [P] or null
  const __nv_bfloat16* bias;     // GELU FC1: b1 [E][N]; FC2: b2 [E][N]; or null
  __nv_bfloat16* out;            // [P, N]
  __nv_bfloat16* act_save;       // [P, Nb] or null (FC1 only)
  float* out_f32;                // kTcF32: [ksplit][P, ldo] fp32
  int ldo;
  int ept;                       // kTcF32: experts per N tile (hi, mid, lo column groups)
  int ksplit, kb_per;            // kTcF32: the K blocks are cut into ksplit slices of kb_per
  int64_t split_stride;          // kTcF32: floats between the slices' outputs
  int E, Kd, N, Nb;              // output columns N; B rows per expert Nb
  int prob_here;                 // apply p in this epilogue
  int* status;
  uint64_t wait_limit_ns;
};

template <int STAGES>
struct SmemCtl {
  uint64_t full[STAGES], empty[STAGES], tmem_full[2], tmem_empty[2], drain;
  uint32_t tmem_base;
  int abort;
  int tile_start[257];
  int off[257];
};

template <int BNT>
constexpr size_t smem_bytes() {
  return 1024 + (size_t)Tile<BNT>::STAGES * Tile<BNT>::STAGE_BYTES +
         sizeof(SmemCtl<Tile<BNT>::STAGES>);
}

// Tile -> (group e, m block, n block).  Within a group the m blocks run
// fastest, so the CTAs that run together share one weight panel; with
// n_fastest (the router's gating GEMM: one group, a weight of a few MB, a
// token matrix that may exceed L2) the n blocks of one m block run together
// and share its token rows instead.
template <typename Ctl>
MOE_D void decode_tile(const Ctl& c, int E, int nblk, int tile, int& e, int& mb, int& nb,
                       bool n_fastest = false) {
  int lo = 0, hi = E - 1;  // largest e with tile_start[e] <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (c.tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  e = lo;
  const int local = tile - c.tile_start[e];
  if (n_fastest) {
    mb = local / nblk;
    nb = local - mb * nblk;
    return;
  }
  const int mblk = (c.off[e + 1] - c.off[e] + BM - 1) / BM;
  nb = local / mblk;
  mb = local - nb * mblk;
}

MOE_D uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

MOE_D void store8(__nv_bfloat16* dst, const float* v) {
  uint4 u;
  u.x = pack_bf16x2(v[0], v[1]);
  u.y = pack_bf16x2(v[2], v[3]);
  u.z = pack_bf16x2(v[4], v[5]);
  u.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(dst) = u;
}

// GATHER (FC1 only): the A rows are the token rows x[src_token[r]], fetched
// by the TMA engine with tile::gather4 loads (four token rows each; the x map's
// box is one row high): the producer warp's 32 lanes each fetch 4 of the
// tile's 128 rows per stage into the same 128-byte-swizzled layout, completing
// on the stage barrier like the tiled loads.  Rows past the expert's end load
// token row 0 (their outputs are never stored).
template <int MODE, int BNT, bool GATHER = false>
__global__ void __launch_bounds__(cta_threads(MODE), 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB, const TcParams p) {
  constexpr int BN = Tile<BNT>::BN;
  constexpr int B_BYTES = Tile<BNT>::B_BYTES;
  constexpr int STAGE_BYTES = Tile<BNT>::STAGE_BYTES;
  constexpr int STAGES = Tile<BNT>::STAGES;
  constexpr uint32_t TMEM_COLS = Tile<BNT>::TMEM_COLS;
  constexpr uint32_t ACC_STRIDE = TMEM_COLS / 2;  // the two accumulators, power-of-2 aligned
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  SmemCtl<STAGES>& ctl = *reinterpret_cast<SmemCtl<STAGES>*>(smem + STAGES * STAGE_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const int nblk = MODE == kTcSwiGLU ? (p.N + BN / 2 - 1) / (BN / 2)
                   : MODE == kTcF32  ? (p.N + p.ept - 1) / p.ept
                                     : (p.N + BN - 1) / BN;
  const int KB = (p.Kd + BK - 1) / BK;

  // ---- prologue: barriers, TMEM, tile list ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(tc::smem_u32(&ctl.full[s]), 1);
      tc::mbar_init(tc::smem_u32(&ctl.empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(tc::smem_u32(&ctl.tmem_full[a]), 1);
      tc::mbar_init(tc::smem_u32(&ctl.tmem_empty[a]), epi_warps(MODE));
    }
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
  for (int e = threadIdx.x; e <= E; e += cta_threads(MODE)) ctl.off[e] = __ldg(p.offsets + e);
  __syncthreads();
  if (warp == 2) {  // tile_start = exclusive scan of m-blocks x n-blocks
    int running = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? ((ctl.off[e + 1] - ctl.off[e] + BM - 1) / BM) * nblk : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (e < E) ctl.tile_start[e] = running + incl - v;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) ctl.tile_start[E] = running;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = ctl.tmem_base;
  // kTcF32 (the router's gating GEMM) may cut the K loop into slices: tile =
  // base_tile * ksplit + slice, each slice writing its own partial sums.
  const int S = MODE == kTcF32 ? p.ksplit : 1;
  const int total = ctl.tile_start[E] * S;
  tc::WaitCtl wc{p.status, &ctl.abort, p.wait_limit_ns, 0};
  tc::WaitCtl wdrain{p.status, nullptr, 1000000000ull, 0};

  if (warp == 0 && GATHER) {
    // ================= gathering TMA producer (whole warp) =================
    int stage = 0;
    uint32_t phase = 0, issued = 0, issued_par = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      int e, mb, nb;
      decode_tile(ctl, E, nblk, tile / S, e, mb, nb, MODE == kTcF32);
      const int m_e = ctl.off[e + 1] - ctl.off[e];
      int b_row0, b_row1 = 0;
      if (MODE == kTcSwiGLU) {
        b_row0 = e * p.Nb + nb * (BN / 2);
        b_row1 = e * p.Nb + p.N + nb * (BN / 2);
      } else {
        b_row0 = e * p.Nb + nb * BN;
      }
      int rr[4];  // this lane's 4 rows (4 lane .. 4 lane + 3) of the tile's 128
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int lr = mb * BM + 4 * lane + j;
        rr[j] = lr < m_e ? __ldg(p.src_token + ctl.off[e] + lr) : 0;
      }
      for (int kb = 0; kb < KB; ++kb) {
        int w_ok = lane == 0 ? (int)tc::mbar_wait(tc::smem_u32(&ctl.empty[stage]), phase ^ 1, wc) : 0;
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) { ok = false; break; }
        const uint32_t fb = tc::smem_u32(&ctl.full[stage]);
        if (lane == 0) {
          tc::mbar_arrive_expect_tx(fb, STAGE_BYTES);
          const uint32_t b_dst = tc::smem_u32(sB + stage * B_BYTES);
          if (MODE == kTcSwiGLU) {
            tc::tma_load_2d(b_dst, &tmB, kb * BK, b_row0, fb);
            tc::tma_load_2d(b_dst + B_BYTES / 2, &tmB, kb * BK, b_row1, fb);
          } else {
            tc::tma_load_2d(b_dst, &tmB, kb * BK, b_row0, fb);
          }
        }
        tc::tma_gather4(tc::smem_u32(sA + stage * A_BYTES) + lane * 512, &tmA, kb * BK, rr[0], rr[1],
                        rr[2], rr[3], fb);
        issued |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
    // copies still in flight must land before the block exits
    if (lane == 0)
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u)
          tc::mbar_wait(tc::smem_u32(&ctl.full[s]), (issued_par >> s) & 1u, wdrain);
    __syncwarp();
  } else if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_par = 0;
      for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        int e, mb, nb;
        decode_tile(ctl, E, nblk, tile / S, e, mb, nb, MODE == kTcF32);
        const int kb0 = MODE == kTcF32 ? (tile % S) * p.kb_per : 0;
        const int kb1 = MODE == kTcF32 ? min(KB, kb0 + p.kb_per) : KB;
        const int a_row = ctl.off[e] + mb * BM;
        int b_row0, b_row1 = 0;
        if (MODE == kTcSwiGLU) {
          b_row0 = e * p.Nb + nb * (BN / 2);
          b_row1 = e * p.Nb + p.N + nb * (BN / 2);
        } else {
          b_row0 = e * p.Nb + nb * BN;
        }
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!tc::mbar_wait(tc::smem_u32(&ctl.empty[stage]), phase ^ 1, wc)) { ok = false; break; }
          const uint32_t fb = tc::smem_u32(&ctl.full[stage]);
          tc::mbar_arrive_expect_tx(fb, STAGE_BYTES);
          const uint32_t a_dst = tc::smem_u32(sA + stage * A_BYTES);
          const uint32_t b_dst = tc::smem_u32(sB + stage * B_BYTES);
          tc::tma_load_2d(a_dst, &tmA, kb * BK, a_row, fb);
          if (MODE == kTcSwiGLU) {
            tc::tma_load_2d(b_dst, &tmB, kb * BK, b_row0, fb);
            tc::tma_load_2d(b_dst + B_BYTES / 2, &tmB, kb * BK, b_row1, fb);
          } else {
            tc::tma_load_2d(b_dst, &tmB, kb * BK, b_row0, fb);
          }
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
      // copies still in flight must land before the block exits
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u)
          tc::mbar_wait(tc::smem_u32(&ctl.full[s]), (issued_par >> s) & 1u, wdrain);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, BN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        if (!tc::mbar_wait(tc::smem_u32(&ctl.tmem_empty[acc]), acc_phase ^ 1, wc)) break;
        tc::fence_after_sync();
        const uint32_t d = tmem_base + (uint32_t)(acc * ACC_STRIDE);
        const int kb0 = MODE == kTcF32 ? (tile % S) * p.kb_per : 0;
        const int nkb = MODE == kTcF32 ? min(KB, kb0 + p.kb_per) - kb0 : KB;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!tc::mbar_wait(tc::smem_u32(&ctl.full[stage]), phase, wc)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t a0 = tc::smem_u32(sA + stage * A_BYTES);
          const uint32_t b0 = tc::smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc::mma_bf16(d, tc::desc_kmajor_sw128(a0 + k * 32), tc::desc_kmajor_sw128(b0 + k * 32),
                         idesc, (kb | k) != 0);
          tc::mma_commit(tc::smem_u32(&ctl.empty[stage]));
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc::mma_commit(tc::smem_u32(&ctl.tmem_full[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (ctl.abort) {  // let every issued MMA finish before TMEM is freed
        tc::mma_commit(tc::smem_u32(&ctl.drain));
        tc::mbar_wait(tc::smem_u32(&ctl.drain), 0, wdrain);
      }
    }
    __syncwarp();
  } else {
    // ================= epilogue (warps 2 ..) =================
    // epi_warps / 4 warps per TMEM lane quarter q (the quarter this warp may
    // access); warp hf of them takes that share of the quarter's columns
    constexpr int NW = epi_warps(MODE) / 4;
    const int q = warp & 3;
    const int hf = (warp - 2) >> 2;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int e, mb, nb;
      decode_tile(ctl, E, nblk, tile / S, e, mb, nb, MODE == kTcF32);
      if (!tc::mbar_wait(tc::smem_u32(&ctl.tmem_full[acc]), acc_phase, wc)) break;
      tc::fence_after_sync();
      const int m_e = ctl.off[e + 1] - ctl.off[e];
      const int local_row = mb * BM + q * 32 + lane;
      const bool valid = local_row < m_e;
      const int64_t row = (int64_t)ctl.off[e] + local_row;
      const float pr = (p.prob && p.prob_here && valid) ? __ldg(p.prob + row) : 1.f;
      const uint32_t tbase = tmem_base + (uint32_t)(acc * ACC_STRIDE) + ((uint32_t)(q * 32) << 16);
      if (MODE == kTcSwiGLU) {
#pragma unroll 1
        for (int c = hf * (BN / 2 / 32 / NW); c < (hf + 1) * (BN / 2 / 32 / NW); ++c) {
          uint32_t g[32], u[32];
          tc::tmem_ld_32x32b_x32(tbase + c * 32, g);
          tc::tmem_ld_32x32b_x32(tbase + BN / 2 + c * 32, u);
          const int n = nb * (BN / 2) + c * 32;
          if (valid) {
#pragma unroll
            for (int gq = 0; gq < 4; ++gq) {
              if (n + gq * 8 >= p.N) break;
              float o[8], gv[8], uv[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                gv[i] = __uint_as_float(g[gq * 8 + i]);
                uv[i] = __uint_as_float(u[gq * 8 + i]);
                o[i] = pr * (silu_f(gv[i]) * uv[i]);
              }
              store8(p.out + row * p.N + n + gq * 8, o);
              if (p.act_save) {
                store8(p.act_save + row * p.Nb + n + gq * 8, gv);
                store8(p.act_save + row * p.Nb + p.N + n + gq * 8, uv);
              }
            }
          }
        }
      } else if (MODE == kTcF32) {
        // the router's gating GEMM: this tile holds, per token, the partial
        // sums of ept experts against the hi, mid and lo parts of the split
        // weight (column groups [0, ept), [ept, 2 ept), [2 ept, 3 ept)); each
        // logit is (lo + mid) + hi, stored 8 experts at a time
        const int ept = p.ept;
        float* dst = p.out_f32 + (tile % S) * p.split_stride + row * p.ldo + nb * ept;
#pragma unroll 1
        for (int c0 = 0; c0 < ept; c0 += 8) {
          uint32_t hi[8], mid[8], lo[8];
          tc::tmem_ld_32x32b_x8x3(tbase + c0, tbase + ept + c0, tbase + 2 * ept + c0, hi, mid, lo);
          if (valid && nb * ept + c0 < p.N) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              v[i] = __fadd_rn(__fadd_rn(__uint_as_float(lo[i]), __uint_as_float(mid[i])),
                               __uint_as_float(hi[i]));
            *reinterpret_cast<float4*>(dst + c0) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4*>(dst + c0 + 4) = make_float4(v[4], v[5], v[6], v[7]);
          }
        }
      } else {
#pragma unroll 1
        for (int c = hf * (BN / 32 / NW); c < (hf + 1) * (BN / 32 / NW); ++c) {
          uint32_t r[32];
          tc::tmem_ld_32x32b_x32(tbase + c * 32, r);
          const int n = nb * BN + c * 32;
          if (valid) {
#pragma unroll
            for (int gq = 0; gq < 4; ++gq) {
              const int n8 = n + gq * 8;
              if (n8 >= p.N) break;
              float v[8], o[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                v[i] = __uint_as_float(r[gq * 8 + i]);
                if (p.bias) v[i] += __bfloat162float(p.bias[(int64_t)e * p.N + n8 + i]);
              }
              if (MODE == kTcGelu) {
                if (p.act_save) store8(p.act_save + row * p.Nb + n8, v);
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = pr * gelu_f(v[i]);
              } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = pr * v[i];
              }
              store8(p.out + row * p.N + n8, o);
            }
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&ctl.tmem_empty[acc]));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---- host side ----------------------------------------------------------------
// 2-D bf16 row-major [rows, cols] map with a {64, box_rows} box, 128-B swizzle.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  tc::EncodeTiledFn fn = tc::encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int BNT = 256, bool GATHER = false>
cudaError_t launch_mode(const CUtensorMap& a, const CUtensorMap& b, const TcParams& p, int grid,
                        cudaStream_t s) {
  constexpr size_t bytes = smem_bytes<BNT>();
  auto kern = grouped_gemm_tc_kernel<MODE, BNT, GATHER>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, cta_threads(MODE), bytes, s>>>(a, b, p);
  return cudaGetLastError();
}

}  // namespace

// One grouped GEMM: out[r, :] = epilogue(A[r, :] B_e^T) for the rows r of each
// expert e.  A [P, Kd]; B [E * Nb, Kd] (bf16, row-major).  With src_token (FC1
// only), row r of the GEMM is token row A[src_token[r]] (A = x, [T, Kd]).
cudaError_t launch_grouped_gemm_tc(int mode, int P, const void* A, int Kd, const void* B, int Nb,
                                   int E, int N, const int32_t* offsets, const float* prob,
                                   int prob_here, const void* bias, void* out, void* act_save,
                                   int sms, int* status, cudaStream_t s,
                                   const int32_t* src_token, int T) {
  if (P == 0) return cudaSuccess;
  const bool gather = src_token != nullptr;
  if (gather && mode != kTcSwiGLU && mode != kTcGelu) return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  constexpr int BN = 256;
  const uint32_t brows = mode == kTcSwiGLU ? BN / 2 : BN;
  if (!encode_2d(&mb, B, (uint64_t)E * Nb, (uint64_t)Kd, brows)) return cudaErrorInvalidValue;
  // gather: the token rows x [T, Kd], fetched four rows at a time (box one row high)
  if (!encode_2d(&ma, A, (uint64_t)(gather ? T : P), (uint64_t)Kd, gather ? 1 : BM))
    return cudaErrorInvalidValue;
  TcParams p;
  p.offsets = offsets; p.prob = prob;
  p.xg = static_cast<const __nv_bfloat16*>(A);
  p.src_token = src_token;
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.act_save = static_cast<__nv_bfloat16*>(act_save);
  p.E = E; p.Kd = Kd; p.N = N; p.Nb = Nb; p.prob_here = prob_here;
  p.out_f32 = nullptr; p.ldo = 0; p.ept = 0;
  p.ksplit = 1; p.kb_per = (Kd + BK - 1) / BK; p.split_stride = 0;
  p.status = status;
  p.wait_limit_ns = 2000000000ull;  // 2 s: far above any real wait
  const int nblk = mode == kTcSwiGLU ? (N + BN / 2 - 1) / (BN / 2) : (N + BN - 1) / BN;
  const int64_t tiles_max = (ceil_div(P, BM) + E) * (int64_t)nblk;
  const int grid = (int)(tiles_max < sms ? tiles_max : sms);
  switch (mode) {
    case kTcSwiGLU:
      return gather ? launch_mode<kTcSwiGLU, 256, true>(ma, mb, p, grid, s)
                    : launch_mode<kTcSwiGLU>(ma, mb, p, grid, s);
    case kTcGelu:
      return gather ? launch_mode<kTcGelu, 256, true>(ma, mb, p, grid, s)
                    : launch_mode<kTcGelu>(ma, mb, p, grid, s);
    case kTcF32: return launch_mode<kTcF32>(ma, mb, p, grid, s);
    default: return launch_mode<kTcFc2>(ma, mb, p, grid, s);
  }
}

cudaError_t launch_grouped_gemm_tc2(int mode, int P, const void* A, int Kd, const void* B, int Nb,
                                    int E, int N, const int32_t* offsets, const float* prob,
                                    int prob_here, const void* bias, void* out, void* act_save,
                                    int sms, int* status, cudaStream_t s,
                                    const int32_t* src_token, int T);

// One of the two expert GEMMs (fc = 1: x_perm -> a, fc = 2: a -> y_perm), on
// CTA pairs when the experts are large enough to fill 256-row tiles.  With
// src_token, FC1 gathers its rows from the token rows A = x instead.
cudaError_t launch_expert_gemm_tc(const moe_config_t& c, int fc, int P, const void* A,
                                  const int32_t* offsets, const float* prob, const void* w,
                                  const void* bias, void* act_save, void* out, int sms,
                                  int* status, cudaStream_t s, const int32_t* src_token) {
  const bool swiglu = c.act == MOE_ACT_SWIGLU;
  const bool prob_after = c.has_bias != 0;
  const bool pair = (c.flags & MOE_FLAG_GEMM_2CTA) ||
                    (!(c.flags & MOE_FLAG_GEMM_1CTA) && (int64_t)P >= 512LL * c.E);
  auto run = pair ? launch_grouped_gemm_tc2 : launch_grouped_gemm_tc;
  if (fc == 1)
    return run(swiglu ? kTcSwiGLU : kTcGelu, P, A, c.h, w, swiglu ? 2 * c.F : c.F, c.E, c.F,
               offsets, prob, !prob_after, bias, out, act_save, sms, status, s, src_token, c.T);
  return run(kTcFc2, P, A, c.F, w, c.h, c.E, c.h, offsets, prob, prob_after, bias, out, nullptr,
             sms, status, s, nullptr, c.T);
}

// Router gating on the tensor cores.  w3 holds the exactly split router
// weight in tiles of bn rows: tile n = [hi | mid | lo] rows of experts
// n*ept .. n*ept + ept - 1 (then zero rows up to bn).  logit_parts[s][t, e] =
// the sum over the s-th slice of h of x[t] * (w_hi + w_mid + w_lo)[e], summed
// as (lo + mid) + hi (fp32, row stride ldo, slices split_stride floats apart);
// offsets = {0, T} (one group).
cudaError_t launch_router_gemm_tc(int T, const void* x, int h, const void* w3, int E, int ept,
                                  int bn, float* logit_parts, int ldo, const int32_t* offsets,
                                  int ksplit, int64_t split_stride, int sms, int* status,
                                  cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (bn != 32 && bn != 48 && bn != 96 && bn != 192) return cudaErrorInvalidValue;
  if (3 * ept > bn || ept % 8) return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  const int ntiles = (E + ept - 1) / ept;
  if (!encode_2d(&ma, x, (uint64_t)T, (uint64_t)h, BM)) return cudaErrorInvalidValue;
  if (!encode_2d(&mb, w3, (uint64_t)ntiles * bn, (uint64_t)h, (uint32_t)bn))
    return cudaErrorInvalidValue;
  const int KB = (h + BK - 1) / BK;
  if (ksplit < 1 || ksplit > KB) return cudaErrorInvalidValue;
  TcParams p{};
  p.offsets = offsets;
  p.E = 1; p.Kd = h; p.N = E; p.Nb = ntiles * bn; p.prob_here = 0;
  p.out_f32 = logit_parts; p.ldo = ldo; p.ept = ept;
  p.kb_per = (KB + ksplit - 1) / ksplit;
  p.ksplit = (KB + p.kb_per - 1) / p.kb_per;  // every slice non-empty
  p.split_stride = split_stride;
  p.status = status;
  p.wait_limit_ns = 2000000000ull;
  const int64_t tiles = ceil_div(T, BM) * ntiles * p.ksplit;
  const int grid = (int)(tiles < sms ? tiles : sms);
  switch (bn) {
    case 32: return launch_mode<kTcF32, 32>(ma, mb, p, grid, s);
    case 48: return launch_mode<kTcF32, 48>(ma, mb, p, grid, s);
    case 96: return launch_mode<kTcF32, 96>(ma, mb, p, grid, s);
    default: return launch_mode<kTcF32, 192>(ma, mb, p, grid, s);
  }
}

// ---- test hook: a wait nothing will complete ---------------------------------
__global__ void bounded_wait_probe_kernel(int* status, int64_t max_polls) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(tc::smem_u32(&bar), 1);
    abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    tc::WaitCtl w{status, &abort_flag, 1000000000ull, max_polls};
    tc::mbar_wait(tc::smem_u32(&bar), 0, w);  // phase 0 never completes
  }
}

cudaError_t launch_bounded_wait_probe(int64_t max_polls, int* status, cudaStream_t s) {
  bounded_wait_probe_kernel<<<1, 32, 0, s>>>(status, max_polls);
  return cudaGetLastError();
}

}  // namespace moe
