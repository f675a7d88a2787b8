// Forward expert GEMMs on CTA pairs (tcgen05.mma.cta_group::2): the same
// computation as grouped_gemm_tc_kernel (gemm_tc.cu), for experts with many
// rows.  "Scalable Training of Mixture-of-Experts Models with Megatron Core"
// (review), §2.1 / §4.3.1: every expert in one grouped GEMM call.
//
// A cluster of two CTAs computes a 256 x 256 tile: CTA r holds rows
// [128r, 128r+128) of A and B rows [128r, 128r+128) of the tile's 256 B rows
// (for SwiGLU: CTA 0 the 128 gate rows, CTA 1 the matching up rows), the even
// CTA issues one M256 N256 K16 MMA over both CTAs' shared memory, and each
// CTA's TMEM receives its own 128 rows x 256 fp32 columns.  Against the 1-CTA
// kernel this halves the B bytes each SM pulls from L2 and its shared-memory
// stage.
//
// A ring stage is 128 deep in K (two 64-column TMA boxes per operand, 64 KB
// per CTA, 3 stages): 8 MMAs per stage wait, fence and commit once.  The MMA
// thread spends about 190 cycles observing a stage barrier (even one whose
// phase completed long before) and 45-75 issuing each tcgen05 instruction;
// with 64-deep stages its wait, 4 MMAs, commit and bookkeeping took about as
// long as the 512 cycles the 4 MMAs run, and the tensor pipe idled between
// stages.
//
// Half tiles: an expert's last row block with at most 128 rows is computed
// as a 128 x 256 tile (M128 N256 K16 pair MMAs, which take half the cycles
// of M256 ones) instead of a padded 256-row one.  CTA r then loads 64 A rows
// [64r, 64r+64) and still 128 B rows; its TMEM lanes 0-63 receive its 64 rows
// x output columns 0-127 (products with CTA 0's B rows) in accumulator
// columns 0-127, and lanes 64-127 the same 64 rows x output columns 128-255
// (CTA 1's B rows).  For SwiGLU each CTA loads 64 gate rows and the matching
// 64 up rows, so that a lane's gate and up values of one hidden column share
// the lane: gate in accumulator columns 0-63, up in 64-127.
//
// Protocol (all waits bounded):
//   full[s]       even CTA, count 1: its producer posts expect_tx for both CTAs'
//                 bytes; both CTAs' TMA loads complete on it (.cta_group::2).
//   empty[s]      both CTAs: the even CTA's MMA commit arrives on both (multicast).
//   tmem_full[a]  both CTAs: multicast commit after a tile's last MMA.
//   tmem_empty[a] even CTA: one arrival per epilogue warp of each CTA.  FC1
//                 has 8 epilogue warps (two per TMEM lane quarter, each storing
//                 half of the quarter's columns; its SwiGLU/GELU epilogue writes
//                 more per tile than FC2's), FC2 has 4.
//   drain         both CTAs: a final multicast commit, so no MMA completion can
//                 still be in flight towards a CTA that is leaving.
// TMEM is allocated and freed with cta_group::2 by one warp of each CTA.
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;  // rows per CTA; the cluster tile is 256 rows
constexpr int BMC = 256;
constexpr int BN = 256;  // accumulator columns
constexpr int BNL = 128; // B rows each CTA loads
constexpr int BK = 64;                  // K columns per TMA box (one 128-byte swizzle row)
constexpr int KSUB = 2;                 // boxes per operand per stage: stages are 128 deep in K
constexpr int SUB_A = BM * BK * 2;      // 16 KB
constexpr int SUB_B = BNL * BK * 2;     // 16 KB
constexpr int A_BYTES = KSUB * SUB_A;   // 32 KB
constexpr int B_BYTES = KSUB * SUB_B;   // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int STAGES = 3;
constexpr uint32_t TMEM_COLS = 512;
enum Tc2Mode { kSwiGLU = 0, kGelu = 1, kFc2 = 2 };

// epilogue warps per CTA, and the CTA size: producer, MMA issuer, epilogue
MOE_HD constexpr int epi_warps(int mode) { return mode == kFc2 ? 4 : 8; }
MOE_HD constexpr int cta_threads(int mode) { return 32 * (2 + epi_warps(mode)); }

struct Tc2Params {
  const int32_t* offsets;
  const __nv_bfloat16* xg;     // gather mode: token rows [*, Kd]
  const int32_t* src_token;    // gather mode: token of each permuted row
  const float* prob;
  const __nv_bfloat16* bias;
  __nv_bfloat16* out;
  __nv_bfloat16* act_save;
  int E, Kd, N, Nb;
  int prob_here;
  int* status;
  uint64_t wait_limit_ns;
};

struct SmemCtl {
  uint64_t full[STAGES], empty[STAGES], tmem_full[2], tmem_empty[2], drain;
  uint32_t tmem_base;
  int abort;
  int tile_start[257];
  int off[257];
};

constexpr size_t kSmemBytes = 1024 + (size_t)STAGES * STAGE_BYTES + sizeof(SmemCtl);

// ---- cluster / pair PTX ------------------------------------------------------
using tc::arrive_cluster;
using tc::cluster_ctarank;
using tc::cluster_sync;
using tc::mapa;
using tc::commit_pair_multicast;
using tc::mma_pair;
using tc::tma_load_2d_pair;
using tc::tmem_alloc_pair;
using tc::tmem_dealloc_pair;
using tc::tmem_relinquish_pair;
MOE_D void decode_tile(const SmemCtl& c, int E, int nblk, int tile, int& e, int& mb, int& nb,
                       bool& half) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (c.tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  e = lo;
  const int local = tile - c.tile_start[e];
  const int mblk = (c.off[e + 1] - c.off[e] + BMC - 1) / BMC;
  nb = local / mblk;
  mb = local - nb * mblk;
  half = c.off[e + 1] - c.off[e] - mb * BMC <= BM;  // at most 128 rows left
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

// GATHER: the A rows are not a permuted buffer's consecutive rows but the
// token rows x[src_token[r]], fetched by the TMA engine with tile::gather4
// loads (four token rows per load, the x map's box one row high): per
// 64-column box the producer warp's 32 lanes each fetch 4 of the CTA's 128
// rows (a half tile's 64 rows: lanes 0-15) into the same 128-byte-swizzled
// layout, completing on the same stage barrier as the tiled loads.  Rows past
// the expert's end load token row 0 (their outputs are never stored).
MOE_D void tma_gather4_pair(uint32_t dst, const CUtensorMap* map, int32_t c0, int4 rows,
                            uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile::gather4"
      ".mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(rows.x), "r"(rows.y), "r"(rows.z),
      "r"(rows.w), "r"(bar_cluster)
      : "memory");
}

// Bytes both CTAs' loads of one stage deliver (the even CTA's expect_tx); a
// half tile loads 64 A rows per CTA.
MOE_D uint32_t stage_tx(bool half) {
  return 2u * KSUB * ((half ? SUB_A / 2 : SUB_A) + SUB_B);
}

// First weight row this CTA loads for N block nb of expert e.  SwiGLU (B =
// [gate; up] per expert): a full tile's CTA r loads 128 gate (r = 0) or up
// (r = 1) rows; a half tile's CTA r loads gate rows [64r, 64r + 64) of the
// block and the matching up rows (returned: the first gate row).  Otherwise
// CTA r loads B rows [128r, 128r + 128) of the block's 256.
template <int MODE>
MOE_D int b_first_row_t(const Tc2Params& p, int e, int nb, uint32_t rank, bool half) {
  if (MODE == kSwiGLU)
    return half ? e * p.Nb + nb * BNL + (int)rank * (BNL / 2)
                : e * p.Nb + (int)rank * p.N + nb * BNL;
  return e * p.Nb + nb * BN + (int)rank * BNL;
}

template <int MODE, bool GATHER>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(cta_threads(MODE), 1)
    grouped_gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmA64,
                            const __grid_constant__ CUtensorMap tmB64, const Tc2Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  SmemCtl& ctl = *reinterpret_cast<SmemCtl*>(smem + STAGES * STAGE_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool even = rank == 0;
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  const int E = p.E;
  const int nblk = MODE == kSwiGLU ? (p.N + BNL - 1) / BNL : (p.N + BN - 1) / BN;
  const int KB = (p.Kd + KSUB * BK - 1) / (KSUB * BK);  // 128-deep stages (a box past Kd reads zeros)
  auto b_first_row = [](const Tc2Params& pp, int e, int nb, uint32_t r, bool half) {
    return b_first_row_t<MODE>(pp, e, nb, r, half);
  };
  // The B rows of one 64-column box: one 128-row box, or for a SwiGLU half
  // tile a 64-row box of gate rows and one of the matching up rows (p.N rows
  // further).
  auto load_b = [](uint32_t dst, const CUtensorMap* m128, const CUtensorMap* m64, int k, int row,
                   int n_rows, bool half, uint32_t bar) {
    if (MODE == kSwiGLU && half) {
      tma_load_2d_pair(dst, m64, k, row, bar);
      tma_load_2d_pair(dst + SUB_B / 2, m64, k, row + n_rows, bar);
    } else {
      tma_load_2d_pair(dst, m128, k, row, bar);
    }
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(tc::smem_u32(&ctl.full[s]), 1);
      tc::mbar_init(tc::smem_u32(&ctl.empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(tc::smem_u32(&ctl.tmem_full[a]), 1);
      tc::mbar_init(tc::smem_u32(&ctl.tmem_empty[a]), 2 * epi_warps(MODE));
    }
    tc::mbar_init(tc::smem_u32(&ctl.drain), 1);
    ctl.abort = 0;
    tc::fence_barrier_init();
    tc::prefetch_tensormap(&tmA);
    tc::prefetch_tensormap(&tmB);
    if (!GATHER) tc::prefetch_tensormap(&tmA64);
    if (MODE == kSwiGLU) tc::prefetch_tensormap(&tmB64);
  }
  if (warp == 1) {
    tmem_alloc_pair(tc::smem_u32(&ctl.tmem_base), TMEM_COLS);
    tmem_relinquish_pair();
  }
  for (int e = threadIdx.x; e <= E; e += cta_threads(MODE)) ctl.off[e] = __ldg(p.offsets + e);
  __syncthreads();
  if (warp == 2) {
    int running = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? ((ctl.off[e + 1] - ctl.off[e] + BMC - 1) / BMC) * nblk : 0;
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
  cluster_sync();  // both CTAs' barriers exist before any remote arrive or TMA signal
  tc::fence_after_sync();
  const uint32_t tmem_base = ctl.tmem_base;
  const int total = ctl.tile_start[E];
  tc::WaitCtl wc{p.status, &ctl.abort, p.wait_limit_ns, 0};
  tc::WaitCtl wdrain{p.status, nullptr, 1000000000ull, 0};

  if (warp == 0 && GATHER) {
    // ================= gathering TMA producer (whole warp, both CTAs) =======
    int stage = 0;
    uint32_t phase = 0, issued = 0, issued_par = 0;
    bool ok = true;
    for (int tile = cid; tile < total && ok; tile += ncl) {
      int e, mb, nb;
      bool half;
      decode_tile(ctl, E, nblk, tile, e, mb, nb, half);
      const int rows_cta = half ? BM / 2 : BM;
      const int lrow0 = mb * BMC + (int)rank * rows_cta;  // first A row of this CTA, inside the expert
      const int m_e = ctl.off[e + 1] - ctl.off[e];
      const int b_row = b_first_row(p, e, nb, rank, half);
      // this lane's 4 rows (4 lane .. 4 lane + 3) of the CTA's 128 (64 in a
      // half tile: lanes 16..31 then load nothing)
      const bool gl = 4 * lane < rows_cta;
      int rr[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int lr = lrow0 + 4 * lane + j;
        rr[j] = lr < m_e ? __ldg(p.src_token + ctl.off[e] + lr) : 0;
      }
      const int4 rows = make_int4(rr[0], rr[1], rr[2], rr[3]);
      for (int kb = 0; kb < KB; ++kb) {
        int w_ok = lane == 0 ? (int)tc::mbar_wait(tc::smem_u32(&ctl.empty[stage]), phase ^ 1, wc) : 0;
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) { ok = false; break; }
        const uint32_t full_local = tc::smem_u32(&ctl.full[stage]);
        const uint32_t full_even = mapa(full_local, 0);
        if (lane == 0) {
          if (even) tc::mbar_arrive_expect_tx(full_local, stage_tx(half));
#pragma unroll
          for (int j = 0; j < KSUB; ++j)
            load_b(tc::smem_u32(sB + stage * B_BYTES + j * SUB_B), &tmB, &tmB64, (kb * KSUB + j) * BK,
                   b_row, p.N, half, full_even);
        }
        if (gl) {
#pragma unroll
          for (int j = 0; j < KSUB; ++j)
            tma_gather4_pair(tc::smem_u32(sA + stage * A_BYTES + j * SUB_A) + lane * 512, &tmA,
                             (kb * KSUB + j) * BK, rows, full_even);
        }
        issued |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
    if (lane == 0)
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u)
          tc::mbar_wait(tc::smem_u32(&ctl.empty[s]), (issued_par >> s) & 1u, wdrain);
    __syncwarp();
  } else if (warp == 0) {
    // ================= TMA producer (both CTAs) =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_par = 0;
      bool ok = true;
      for (int tile = cid; tile < total && ok; tile += ncl) {
        int e, mb, nb;
        bool half;
        decode_tile(ctl, E, nblk, tile, e, mb, nb, half);
        const int a_row = ctl.off[e] + mb * BMC + (int)rank * (half ? BM / 2 : BM);
        const int b_row = b_first_row(p, e, nb, rank, half);
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc::mbar_wait(tc::smem_u32(&ctl.empty[stage]), phase ^ 1, wc)) { ok = false; break; }
          const uint32_t full_local = tc::smem_u32(&ctl.full[stage]);
          if (even) tc::mbar_arrive_expect_tx(full_local, stage_tx(half));
          const uint32_t full_even = mapa(full_local, 0);
#pragma unroll
          for (int j = 0; j < KSUB; ++j) {
            tma_load_2d_pair(tc::smem_u32(sA + stage * A_BYTES + j * SUB_A), half ? &tmA64 : &tmA,
                             (kb * KSUB + j) * BK, a_row, full_even);
            load_b(tc::smem_u32(sB + stage * B_BYTES + j * SUB_B), &tmB, &tmB64, (kb * KSUB + j) * BK,
                   b_row, p.N, half, full_even);
          }
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      // Every issued stage must have been consumed (the even CTA's MMA commit
      // arrives on both CTAs' empty barriers only after the bytes landed and
      // the MMAs reading them finished) before the CTA may leave.
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u)
          tc::mbar_wait(tc::smem_u32(&ctl.empty[s]), (issued_par >> s) & 1u, wdrain);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer (even CTA) =================
    if (even && lane == 0) {
      constexpr uint32_t idesc_full = tc::idesc_bf16_f32(BMC, BN);
      constexpr uint32_t idesc_half = tc::idesc_bf16_f32(BM, BN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = cid; tile < total && ok; tile += ncl) {
        int e, mb, nb;
        bool half;
        decode_tile(ctl, E, nblk, tile, e, mb, nb, half);
        const uint32_t idesc = half ? idesc_half : idesc_full;
        if (!tc::mbar_wait(tc::smem_u32(&ctl.tmem_empty[acc]), acc_phase ^ 1, wc)) break;
        tc::fence_after_sync();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc::mbar_wait(tc::smem_u32(&ctl.full[stage]), phase, wc)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t a0 = tc::smem_u32(sA + stage * A_BYTES);
          const uint32_t b0 = tc::smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int j = 0; j < KSUB; ++j)
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              mma_pair(d, tc::desc_kmajor_sw128(a0 + j * SUB_A + k * 32),
                       tc::desc_kmajor_sw128(b0 + j * SUB_B + k * 32), idesc, (kb | j | k) != 0);
          commit_pair_multicast(tc::smem_u32(&ctl.empty[stage]), 0x3);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        commit_pair_multicast(tc::smem_u32(&ctl.tmem_full[acc]), 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      commit_pair_multicast(tc::smem_u32(&ctl.drain), 0x3);
    }
    __syncwarp();
  } else {
    // ================= epilogue (warps 2..9, both CTAs) =================
    // epi_warps / 4 warps per TMEM lane quarter q; warp hf of them takes that
    // share of the quarter's accumulator columns
    constexpr int NW = epi_warps(MODE) / 4;
    const int q = warp & 3;
    const int hf = (warp - 2) >> 2;
    int acc = 0;
    uint32_t acc_phase = 0;
    const uint32_t tmem_empty_even0 = mapa(tc::smem_u32(&ctl.tmem_empty[0]), 0);
    const uint32_t tmem_empty_even1 = mapa(tc::smem_u32(&ctl.tmem_empty[1]), 0);
    for (int tile = cid; tile < total; tile += ncl) {
      int e, mb, nb;
      bool half;
      decode_tile(ctl, E, nblk, tile, e, mb, nb, half);
      if (!tc::mbar_wait(tc::smem_u32(&ctl.tmem_full[acc]), acc_phase, wc)) break;
      tc::fence_after_sync();
      const int m_e = ctl.off[e + 1] - ctl.off[e];
      // Full tile: lane quarter q holds rows 32q.. of the CTA's 128, every
      // column.  Half tile: quarters 0-1 and 2-3 hold the same 64 rows (lanes
      // 0-63 and 64-127), quarters 2-3 the second half of the output columns.
      const int local_row = half ? mb * BMC + (int)rank * (BM / 2) + (q & 1) * 32 + lane
                                 : mb * BMC + (int)rank * BM + q * 32 + lane;
      const int col_half = half ? (q >> 1) : 0;
      const bool valid = local_row < m_e;
      const int64_t row = (int64_t)ctl.off[e] + local_row;
      const float pr = (p.prob && p.prob_here && valid) ? __ldg(p.prob + row) : 1.f;
      const uint32_t tbase = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      if (MODE == kSwiGLU) {
        // gate at accumulator column c, up at c + ncol (ncol = 128 or 64)
        const int ncol = half ? BNL / 2 : BNL;
        const int n0 = nb * BNL + col_half * (BNL / 2);
#pragma unroll 1
        for (int c = hf * (ncol / 32 / NW); c < (hf + 1) * (ncol / 32 / NW); ++c) {
          uint32_t g[32], u[32];
          tc::tmem_ld_32x32b_x32(tbase + c * 32, g);
          tc::tmem_ld_32x32b_x32(tbase + ncol + c * 32, u);
          const int n = n0 + c * 32;
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
      } else {
        const int ncol = half ? BN / 2 : BN;
        const int n0 = nb * BN + col_half * (BN / 2);
#pragma unroll 1
        for (int c = hf * (ncol / 32 / NW); c < (hf + 1) * (ncol / 32 / NW); ++c) {
          uint32_t r[32];
          tc::tmem_ld_32x32b_x32(tbase + c * 32, r);
          const int n = n0 + c * 32;
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
              if (MODE == kGelu) {
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
      if (lane == 0) arrive_cluster(acc == 0 ? tmem_empty_even0 : tmem_empty_even1);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }
  // the even CTA's final multicast commit lands after every MMA and every
  // earlier commit: once it is seen, nothing is in flight towards this CTA
  if (threadIdx.x == 0) tc::mbar_wait(tc::smem_u32(&ctl.drain), 0, wdrain);
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc::fence_after_sync();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

bool encode(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  tc::EncodeTiledFn fn = tc::encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, bool GATHER>
cudaError_t launch_mode2(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& a64,
                         const CUtensorMap& b64, const Tc2Params& p, int64_t tiles, int sms,
                         cudaStream_t s) {
  auto kern = grouped_gemm_tc2_kernel<MODE, GATHER>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  // as many pairs as can be resident at once (a pair needs two SMs of one
  // cluster-capable group), capped by the tile count
  int max_clusters = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (unsigned)((sms + 1) / 2));
  cfg.blockDim = dim3(cta_threads(MODE));
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg) != cudaSuccess ||
      max_clusters < 1)
    max_clusters = sms / 2;
  const int64_t pairs = tiles < max_clusters ? tiles : max_clusters;
  kern<<<(unsigned)(2 * pairs), cta_threads(MODE), kSmemBytes, s>>>(a, b, a64, b64, p);
  return cudaGetLastError();
}

}  // namespace

// Pair-tile version of launch_grouped_gemm_tc (same modes: 0 SwiGLU FC1,
// 1 GELU FC1, 2 FC2; same arguments).  With src_token (FC1 only), A is not a
// permuted buffer: row r of the GEMM is token row A[src_token[r]] (A = x, [T, Kd]).
cudaError_t launch_grouped_gemm_tc2(int mode, int P, const void* A, int Kd, const void* B, int Nb,
                                    int E, int N, const int32_t* offsets, const float* prob,
                                    int prob_here, const void* bias, void* out, void* act_save,
                                    int sms, int* status, cudaStream_t s,
                                    const int32_t* src_token, int T) {
  if (P == 0) return cudaSuccess;
  const bool gather = src_token != nullptr;
  if (gather && mode == kFc2) return cudaErrorInvalidValue;
  CUtensorMap ma, mb, ma64, mb64;
  if (!encode(&mb, B, (uint64_t)E * Nb, (uint64_t)Kd, BNL)) return cudaErrorInvalidValue;
  // gather: the token rows x [T, Kd], fetched four rows at a time (box one row high)
  if (!encode(&ma, A, (uint64_t)(gather ? T : P), (uint64_t)Kd, gather ? 1 : BM))
    return cudaErrorInvalidValue;
  // half tiles: 64 A rows per CTA, and for SwiGLU 64 gate + 64 up weight rows
  if (gather) ma64 = ma;
  else if (!encode(&ma64, A, (uint64_t)P, (uint64_t)Kd, BM / 2)) return cudaErrorInvalidValue;
  if (mode != kSwiGLU) mb64 = mb;
  else if (!encode(&mb64, B, (uint64_t)E * Nb, (uint64_t)Kd, BNL / 2)) return cudaErrorInvalidValue;
  Tc2Params p;
  p.offsets = offsets; p.prob = prob;
  p.xg = static_cast<const __nv_bfloat16*>(A);
  p.src_token = src_token;
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.act_save = static_cast<__nv_bfloat16*>(act_save);
  p.E = E; p.Kd = Kd; p.N = N; p.Nb = Nb; p.prob_here = prob_here;
  p.status = status;
  p.wait_limit_ns = 2000000000ull;
  const int nblk = mode == kSwiGLU ? (N + BNL - 1) / BNL : (N + BN - 1) / BN;
  const int64_t tiles = (ceil_div(P, BMC) + E) * (int64_t)nblk;
  switch (mode) {
    case kSwiGLU:
      return gather ? launch_mode2<kSwiGLU, true>(ma, mb, ma64, mb64, p, tiles, sms, s)
                    : launch_mode2<kSwiGLU, false>(ma, mb, ma64, mb64, p, tiles, sms, s);
    case kGelu:
      return gather ? launch_mode2<kGelu, true>(ma, mb, ma64, mb64, p, tiles, sms, s)
                    : launch_mode2<kGelu, false>(ma, mb, ma64, mb64, p, tiles, sms, s);
    default: return launch_mode2<kFc2, false>(ma, mb, ma64, mb64, p, tiles, sms, s);
  }
}

}  // namespace moe
