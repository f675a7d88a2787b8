// Backward grouped GEMMs of the expert FFNs on the tensor cores (tcgen05 +
// TMEM, TMA-fed), bf16 operands, fp32 accumulation.
//
// The pages give no backward formulas ("Scalable Training of Mixture-of-
// Experts Models with Megatron Core", review, §4.1.2 only says which
// activations are recomputed for it); these are the plain reverse-mode
// derivatives of the forward expert FFN with the routing held fixed:
//   G      = dy_perm W2_e                       (FC2 dgrad, [rows, F])
//   dprob  = <G, silu(g) * u>  per row          (fused, partial sums per N tile)
//   dH     = [p G u silu'(g), p G silu(g)]      (fused dSwiGLU, [rows, 2F])
//   dW2_e  = dy_perm_e^T a_e                    (FC2 wgrad, [h, F])
//   dx_perm= dH W1_e                            (FC1 dgrad, [rows, h])
//   dW1_e  = dH_e^T x_perm_e                    (FC1 wgrad, [2F, h])
//
// Operand layouts come straight from the forward buffers and the weights, no
// transposes: the dgrad B operand (W2_e read as [F x h], W1_e as [h x 2F]) is
// MN-major, fetched by a 3-D TMA map [E][K][N] so K never runs into the next
// expert; the wgrad operands are MN-major slices of the permuted activations,
// and the reduction runs over the expert's own rows: in the last 64-row block
// only ceil(v/16) MMA K-steps are issued and the < 16 rows past the expert's
// end are zeroed in shared memory first.
//
// Kernel structure as the forward kernel: persistent, 1 CTA per SM, TMA warp,
// MMA warp, 4 epilogue warps, TMEM 2 x 256 columns, bounded waits.  The data
// gradients use a 4-stage ring of 48 KB; the weight gradient 2 stages of
// 96 KB (one 128-row block of the expert per stage) and streams its output
// through 32 KB of staging with TMA stores.  The weight gradient of an expert
// without rows is zero: its tiles never reach the producer or the MMA warp;
// the epilogue warps write them with plain 16-byte stores, interleaved with
// the computed tiles (each CTA spreads its share of zero tiles evenly between
// its computed ones), so that those stores overlap the computed tiles' operand
// loads instead of idling the loads and MMAs for rounds of empty experts.  MN-major tiles are {64 elements,
// BK K-rows} TMA boxes with 128-byte swizzle: LBO = 64 x BK x 2 bytes between
// 64-element atoms, SBO = 1 KB between 8-row groups.
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BN = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr int kThreads = 192;

enum BwdKind { kDgradSwiGLU = 0, kDgradPlain = 1, kWgrad = 2 };

// Per-kind pipeline.  The data-gradient kernels reduce over thousands of K
// values in 4 stages of 64.  The weight-gradient kernel reduces over one
// expert's rows (about a hundred in a fine-grained layer) with its operands in
// L2, where a stage's load rate grows with the size of its TMA boxes: it uses
// 2 stages of 128 rows (96 KB, six {64 column, 128 row} boxes), one stage per
// tile at that size.
template <int KIND>
struct BwdCfg {
  static constexpr int BK = KIND == kWgrad ? 128 : 64;
  static constexpr int STAGES = KIND == kWgrad ? 2 : 4;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int ATOM = 64 * BK * 2;  // one MN-major {64 columns, BK rows} box
  static constexpr int NTS = KIND == kWgrad ? 1 : 257;  // tile_start entries needed
};

struct BwdParams {
  const int32_t* offsets;      // [E+1]
  const float* prob;           // dSwiGLU: [rows] or null (weight 1)
  const __nv_bfloat16* H;      // dSwiGLU: pre-activation [rows, 2N] (gate | up)
  __nv_bfloat16* out;          // dSwiGLU: dH [rows, 2N]; plain: [rows, N]; wgrad: [E][M][N]
  float* dprob_part;           // dSwiGLU: [rows, nblk] or null
  int E, Kd, M, N;
  int* status;
  uint64_t wait_limit_ns;
};

template <int STAGES, int NTS>
struct SmemCtl {
  uint8_t with_rows[256];  // wgrad: experts with rows, in order (E <= 256)
  uint8_t no_rows[256];    // wgrad: experts without rows
  int n_with_rows, n_no_rows;
  uint64_t full[STAGES], empty[STAGES], tmem_full[2], tmem_empty[2], drain;
  uint32_t tmem_base;
  int abort;
  int total;
  int tile_start[NTS];
  int off[257];
};

// The weight-gradient kernel writes its 128 x 256 output tile through shared
// memory with TMA stores, 64 columns at a time: each epilogue warp has two
// 4 KB slots ({64 column, 32 row} boxes) and refills one while the other's
// store is still reading it (32 KB of staging).
constexpr int STAGING_BYTES = 4 * 2 * 4096;
template <int KIND>
constexpr size_t smem_bytes() {
  return 1024 + (size_t)BwdCfg<KIND>::STAGES * BwdCfg<KIND>::STAGE_BYTES +
         (KIND == kWgrad ? STAGING_BYTES : 0) +
         sizeof(SmemCtl<BwdCfg<KIND>::STAGES, BwdCfg<KIND>::NTS>);
}

MOE_D void tma_store_3d(const CUtensorMap* map, int32_t c0, int32_t c1, int32_t c2, uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(src)
      : "memory");
}
MOE_D void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
MOE_D void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
MOE_D void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

MOE_D void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1, int32_t c2,
                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

MOE_D uint32_t pack2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}
MOE_D void store8(__nv_bfloat16* dst, const float* v) {
  uint4 u;
  u.x = pack2(v[0], v[1]); u.y = pack2(v[2], v[3]); u.z = pack2(v[4], v[5]); u.w = pack2(v[6], v[7]);
  *reinterpret_cast<uint4*>(dst) = u;
}
MOE_D void load8(const __nv_bfloat16* src, float* v) {
  const uint4 u = *reinterpret_cast<const uint4*>(src);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __low2float(h[i]);
    v[2 * i + 1] = __high2float(h[i]);
  }
}

// Epilogue of one weight-gradient tile for one epilogue warp (TMEM lane
// quarter q): its 32 rows x 256 columns, 64 columns at a time: TMEM -> bf16 ->
// a swizzled {64 col, 32 row} box in one of the warp's two 4 KB shared-memory
// slots (row `lane`, 16-B chunk c at c ^ (lane & 7)) -> one TMA store (rows
// past M are clipped).  A slot is refilled once the store issued from it two
// boxes earlier has read it, so the other slot's store stays in flight.  The
// TMEM load of the next 64 columns is issued before this box is converted and
// stored (two register buffers), so its latency overlaps the store path
// instead of adding to it.  The accumulator is released (tmem_empty) once its
// last load has completed.  have_rows false: the expert has no rows and the
// tile is zeros.
MOE_D void wgrad_box(const uint32_t (&r)[64], bool have_rows, uint8_t* box, int lane) {
  if (lane == 0) bulk_wait_read1();  // the store from this slot (two boxes back) has read it
  __syncwarp();
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (have_rows) {
      u.x = pack2(__uint_as_float(r[g * 8 + 0]), __uint_as_float(r[g * 8 + 1]));
      u.y = pack2(__uint_as_float(r[g * 8 + 2]), __uint_as_float(r[g * 8 + 3]));
      u.z = pack2(__uint_as_float(r[g * 8 + 4]), __uint_as_float(r[g * 8 + 5]));
      u.w = pack2(__uint_as_float(r[g * 8 + 6]), __uint_as_float(r[g * 8 + 7]));
    }
    *reinterpret_cast<uint4*>(box + lane * 128 + ((g ^ (lane & 7)) << 4)) = u;
  }
  tc::fence_proxy_async_smem();
  __syncwarp();
}

MOE_D void wgrad_store_tile(uint32_t tbase, bool have_rows, int e, int mb, int nb, int q,
                            int lane, uint8_t* staging, const CUtensorMap* tmC,
                            uint32_t tmem_empty_bar) {
  static_assert(BN == 256, "four 64-column boxes per tile");
  uint8_t* slots = staging + q * 2 * 4096;
  uint32_t ra[64], rb[64];
  if (have_rows) {
    tc::tmem_ld_32x32b_x64_nowait(tbase, ra);
    tc::tmem_ld_wait_x64(ra);
  }
  auto store = [&](int j) {
    if (lane == 0) {
      tma_store_3d(tmC, nb * BN + j * 64, mb * BM + q * 32, e, tc::smem_u32(slots + (j & 1) * 4096));
      bulk_commit();
    }
  };
  auto release = [&]() {  // every TMEM load of this tile has completed
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(tmem_empty_bar);
  };
  // box 0 from ra while box 1 loads into rb; box 1 from rb while box 2 loads
  // into ra; box 2 from ra while box 3 loads into rb; box 3 from rb
  if (have_rows) tc::tmem_ld_32x32b_x64_nowait(tbase + 64, rb);
  wgrad_box(ra, have_rows, slots, lane);
  store(0);
  if (have_rows) {
    tc::tmem_ld_wait_x64(rb);
    tc::tmem_ld_32x32b_x64_nowait(tbase + 128, ra);
  }
  wgrad_box(rb, have_rows, slots + 4096, lane);
  store(1);
  if (have_rows) {
    tc::tmem_ld_wait_x64(ra);
    tc::tmem_ld_32x32b_x64_nowait(tbase + 192, rb);
  }
  wgrad_box(ra, have_rows, slots, lane);
  store(2);
  if (have_rows) tc::tmem_ld_wait_x64(rb);
  release();
  wgrad_box(rb, have_rows, slots + 4096, lane);
  store(3);
}

// One epilogue warp's share of a zero weight-gradient tile (an expert without
// rows): its 32 rows of the 128 x 256 tile, one row per instruction, 32 lanes
// x 16 bytes = 256 bf16 columns, coalesced; rows past M and columns past N are
// skipped (N is a multiple of 8).
MOE_D void wgrad_zero_tile(__nv_bfloat16* out, int M, int N, int e, int mb, int nb, int q,
                           int lane) {
  const int col = nb * BN + lane * 8;
  if (col >= N) return;
  for (int r = 0; r < 32; ++r) {
    const int row = mb * BM + q * 32 + r;
    if (row >= M) break;
    *reinterpret_cast<uint4*>(out + ((int64_t)e * M + row) * N + col) = make_uint4(0, 0, 0, 0);
  }
}

template <int KIND>
struct Tiles {
  // dgrad: row tiles of each expert x N tiles; wgrad: M tiles x N tiles per expert
  template <typename Ctl>
  MOE_D static void decode(const Ctl& c, int E, int mt, int nt, int tile, int& e, int& mb,
                           int& nb) {
    if (KIND == kWgrad) {  // tile indexes the computed tiles: those of experts with rows
      const int tpe = mt * nt;
      const int k = tile / tpe;
      e = c.with_rows[k];
      const int local = tile - k * tpe;
      nb = local / mt;
      mb = local - nb * mt;
      return;
    }
    int lo = 0, hi = E - 1;
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
};

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_tc_bwd_kernel(const __grid_constant__ CUtensorMap tmA,
                               const __grid_constant__ CUtensorMap tmB,
                               const __grid_constant__ CUtensorMap tmC, const BwdParams p) {
  constexpr int STAGES = BwdCfg<KIND>::STAGES;
  constexpr int BK = BwdCfg<KIND>::BK;
  constexpr int A_BYTES = BwdCfg<KIND>::A_BYTES;
  constexpr int B_BYTES = BwdCfg<KIND>::B_BYTES;
  constexpr int STAGE_BYTES = BwdCfg<KIND>::STAGE_BYTES;
  constexpr int ATOM = BwdCfg<KIND>::ATOM;
  using Ctl = SmemCtl<STAGES, BwdCfg<KIND>::NTS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint8_t* sC = smem + STAGES * STAGE_BYTES;  // wgrad output staging (32 KB)
  Ctl& ctl = *reinterpret_cast<Ctl*>(sC + (KIND == kWgrad ? STAGING_BYTES : 0));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const int nt = (p.N + BN - 1) / BN;
  const int mt = (p.M + BM - 1) / BM;  // wgrad only
  const int KBfix = (p.Kd + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(tc::smem_u32(&ctl.full[s]), 1);
      tc::mbar_init(tc::smem_u32(&ctl.empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(tc::smem_u32(&ctl.tmem_full[a]), 1);
      tc::mbar_init(tc::smem_u32(&ctl.tmem_empty[a]), 4);
    }
    tc::mbar_init(tc::smem_u32(&ctl.drain), 1);
    ctl.abort = 0;
    tc::fence_barrier_init();
    tc::fence_proxy_async_smem();
    tc::prefetch_tensormap(&tmA);
    tc::prefetch_tensormap(&tmB);
    if (KIND == kWgrad) tc::prefetch_tensormap(&tmC);
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(&ctl.tmem_base), TMEM_COLS);
    tc::tmem_relinquish();
  }
  for (int e = threadIdx.x; e <= E; e += kThreads) ctl.off[e] = __ldg(p.offsets + e);
  __syncthreads();
  if (warp == 2) {
    if (KIND == kWgrad) {
      // the experts with rows and those without, each in expert order
      int n_ne = 0, n_z = 0;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const bool in = e < E;
        const bool has = in && ctl.off[e + 1] > ctl.off[e];
        const uint32_t m_has = __ballot_sync(0xffffffffu, has);
        const uint32_t m_none = __ballot_sync(0xffffffffu, in && !has);
        const uint32_t below = (1u << lane) - 1u;
        if (has) ctl.with_rows[n_ne + __popc(m_has & below)] = (uint8_t)e;
        if (in && !has) ctl.no_rows[n_z + __popc(m_none & below)] = (uint8_t)e;
        n_ne += __popc(m_has);
        n_z += __popc(m_none);
      }
      if (lane == 0) {
        ctl.n_with_rows = n_ne;
        ctl.n_no_rows = n_z;
        ctl.total = n_ne * mt * nt;  // computed tiles
      }
    } else {
      int running = 0;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const int v = e < E ? ((ctl.off[e + 1] - ctl.off[e] + BM - 1) / BM) * nt : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        if (e < E) ctl.tile_start[e] = running + incl - v;
        running += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) ctl.total = running;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem_base = ctl.tmem_base;
  const int total = ctl.total;
  tc::WaitCtl wc{p.status, &ctl.abort, p.wait_limit_ns, 0};
  tc::WaitCtl wdrain{p.status, nullptr, 1000000000ull, 0};

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        int e, mb, nb;
        Tiles<KIND>::decode(ctl, E, mt, nt, tile, e, mb, nb);
        const int rows0 = ctl.off[e];
        const int m_e = ctl.off[e + 1] - rows0;
        const int KB = KIND == kWgrad ? (m_e + BK - 1) / BK : KBfix;
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc::mbar_wait(tc::smem_u32(&ctl.empty[stage]), phase ^ 1, wc)) { ok = false; break; }
          const uint32_t fb = tc::smem_u32(&ctl.full[stage]);
          tc::mbar_arrive_expect_tx(fb, STAGE_BYTES);
          const uint32_t a_dst = tc::smem_u32(sA + stage * A_BYTES);
          const uint32_t b_dst = tc::smem_u32(sB + stage * B_BYTES);
          if (KIND == kWgrad) {
            const int krow = rows0 + kb * BK;
#pragma unroll
            for (int j = 0; j < 2; ++j) tc::tma_load_2d(a_dst + j * ATOM, &tmA, mb * BM + j * 64, krow, fb);
#pragma unroll
            for (int j = 0; j < 4; ++j) tc::tma_load_2d(b_dst + j * ATOM, &tmB, nb * BN + j * 64, krow, fb);
          } else {
            tc::tma_load_2d(a_dst, &tmA, kb * BK, rows0 + mb * BM, fb);
#pragma unroll
            for (int j = 0; j < 4; ++j) tma_load_3d(b_dst + j * ATOM, &tmB, nb * BN + j * 64, kb * BK, e, fb);
          }
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u)
          tc::mbar_wait(tc::smem_u32(&ctl.full[s]), (issued_par >> s) & 1u, wdrain);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer (whole warp: the wgrad tail is zeroed by all lanes) =====
    constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, BN, KIND == kWgrad, true);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      int e, mb, nb;
      Tiles<KIND>::decode(ctl, E, mt, nt, tile, e, mb, nb);
      const int m_e = ctl.off[e + 1] - ctl.off[e];
      const int KB = KIND == kWgrad ? (m_e + BK - 1) / BK : KBfix;
      int w_ok = lane == 0 ? (int)tc::mbar_wait(tc::smem_u32(&ctl.tmem_empty[acc]), acc_phase ^ 1, wc) : 0;
      if (!__shfl_sync(0xffffffffu, w_ok, 0)) break;
      tc::fence_after_sync();
      const uint32_t d = tmem_base + (uint32_t)(acc * BN);
      for (int kb = 0; kb < KB; ++kb) {
        w_ok = lane == 0 ? (int)tc::mbar_wait(tc::smem_u32(&ctl.full[stage]), phase, wc) : 0;
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) { ok = false; break; }
        tc::fence_after_sync();
        int nk = BK / 16;
        if (KIND == kWgrad) {
          const int v = m_e - kb * BK;  // valid K rows in this block
          if (v < BK) {
            // every writing lane acquires the completed TMA phase itself (it
            // completed already: this returns at the first poll)
            if (!tc::mbar_wait(tc::smem_u32(&ctl.full[stage]), phase, wc)) ok = false;
            if (!__all_sync(0xffffffffu, ok)) {
              ok = false;
              break;
            }
            nk = (v + 15) / 16;
            const int v16 = nk * 16;
            // zero rows [v, v16) of the 2 A atoms and 4 B atoms (whole 128-B
            // rows: the swizzle only permutes 16-B chunks inside a row)
            const int nrows = v16 - v;
            for (int i = lane; i < nrows * 8 * 6; i += 32) {
              const int atom = i / (nrows * 8);
              const int rem = i - atom * nrows * 8;
              const int row = v + rem / 8, chunk = rem % 8;
              uint8_t* base = atom < 2 ? sA + stage * A_BYTES + atom * ATOM
                                       : sB + stage * B_BYTES + (atom - 2) * ATOM;
              *reinterpret_cast<uint4*>(base + row * 128 + chunk * 16) = make_uint4(0, 0, 0, 0);
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
          }
        }
        if (lane == 0) {
          const uint32_t a0 = tc::smem_u32(sA + stage * A_BYTES);
          const uint32_t b0 = tc::smem_u32(sB + stage * B_BYTES);
          for (int k = 0; k < nk; ++k) {
            const uint64_t ad = KIND == kWgrad ? tc::desc_mnmajor_sw128(a0 + k * 2048, ATOM)
                                               : tc::desc_kmajor_sw128(a0 + k * 32);
            const uint64_t bd = tc::desc_mnmajor_sw128(b0 + k * 2048, ATOM);
            tc::mma_bf16(d, ad, bd, idesc, (kb | k) != 0);
          }
          tc::mma_commit(tc::smem_u32(&ctl.empty[stage]));
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      if (lane == 0) tc::mma_commit(tc::smem_u32(&ctl.tmem_full[acc]));
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (lane == 0 && ctl.abort) {
      tc::mma_commit(tc::smem_u32(&ctl.drain));
      tc::mbar_wait(tc::smem_u32(&ctl.drain), 0, wdrain);
    }
    __syncwarp();
  } else {
    // ================= epilogue (warps 2..5) =================
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    // wgrad: this CTA's zero tiles (index zi = blockIdx.x + j * gridDim.x over
    // the tiles of experts without rows), spread evenly between its computed
    // tiles: after its k-th computed tile the first k * nz / nc of them
    const int tpe = mt * nt;
    const int G = (int)gridDim.x, b = (int)blockIdx.x;
    const int nzt = KIND == kWgrad ? ctl.n_no_rows * tpe : 0;
    const int nc = total > b ? (total - b + G - 1) / G : 0;
    const int nz = nzt > b ? (nzt - b + G - 1) / G : 0;
    int zdone = 0, kc = 0;
    bool aborted = false;
    auto zero_upto = [&](int target) {
      for (; zdone < target; ++zdone) {
        const int zi = b + zdone * G;
        const int k = zi / tpe, local = zi - k * tpe;
        const int nbz = local / mt, mbz = local - nbz * mt;
        wgrad_zero_tile(p.out, p.M, p.N, ctl.no_rows[k], mbz, nbz, q, lane);
      }
    };
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int e, mb, nb;
      Tiles<KIND>::decode(ctl, E, mt, nt, tile, e, mb, nb);
      const int m_e = ctl.off[e + 1] - ctl.off[e];
      if (!tc::mbar_wait(tc::smem_u32(&ctl.tmem_full[acc]), acc_phase, wc)) {
        aborted = true;
        break;
      }
      tc::fence_after_sync();
      const uint32_t tbase = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      if (KIND == kWgrad) {
        wgrad_store_tile(tbase, m_e > 0, e, mb, nb, q, lane, sC, &tmC,
                         tc::smem_u32(&ctl.tmem_empty[acc]));
        ++kc;
        zero_upto((int)((int64_t)kc * nz / nc));
      } else {
        const int local_row = mb * BM + q * 32 + lane;
        const bool valid = local_row < m_e;
        const int64_t row = (int64_t)ctl.off[e] + local_row;
        float pr = 1.f, dpr = 0.f;
        if (KIND == kDgradSwiGLU && valid && p.prob) pr = __ldg(p.prob + row);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tc::tmem_ld_32x32b_x32(tbase + c * 32, r);
          const int n = nb * BN + c * 32;
          if (!valid) continue;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int n8 = n + g * 8;
            if (n8 >= p.N) break;
            float G[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) G[i] = __uint_as_float(r[g * 8 + i]);
            if (KIND == kDgradPlain) {
              store8(p.out + row * p.N + n8, G);
            } else {
              float gt[8], up[8], dg[8], du[8];
              load8(p.H + row * 2 * p.N + n8, gt);
              load8(p.H + row * 2 * p.N + p.N + n8, up);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float s = sigmoid_f(gt[i]);
                const float sl = gt[i] * s;
                dpr = fmaf(G[i], sl * up[i], dpr);
                const float dz = pr * G[i];
                du[i] = dz * sl;
                dg[i] = dz * up[i] * (s * (1.f + gt[i] * (1.f - s)));
              }
              store8(p.out + row * 2 * p.N + n8, dg);
              store8(p.out + row * 2 * p.N + p.N + n8, du);
            }
          }
        }
        if (KIND == kDgradSwiGLU && valid && p.dprob_part) p.dprob_part[row * nt + nb] = dpr;
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tc::smem_u32(&ctl.tmem_empty[acc]));
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (KIND == kWgrad && !aborted) zero_upto(nz);  // the rest (all of them when nc = 0)
    if (KIND == kWgrad && lane == 0) bulk_wait0();  // every TMA store has completed
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// bf16 map with a {64, rows} box: 2-D [rows, cols] when depth == 0, else
// 3-D [depth][rows][cols].  128-byte swizzle, zero fill out of bounds.
bool encode_map(CUtensorMap* m, const void* base, uint64_t depth, uint64_t rows, uint64_t cols,
                uint32_t box_rows) {
  tc::EncodeTiledFn fn = tc::encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {cols, rows, depth ? depth : 1};
  const cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, depth ? 3 : 2, const_cast<void*>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KIND>
cudaError_t launch_kind(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                        const BwdParams& p, int grid, cudaStream_t s) {
  constexpr size_t bytes = smem_bytes<KIND>();
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_tc_bwd_kernel<KIND>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  grouped_gemm_tc_bwd_kernel<KIND><<<grid, kThreads, bytes, s>>>(a, b, c, p);
  return cudaGetLastError();
}

}  // namespace

// Data gradient through one expert weight: out = A W_e with A [rows, Kd]
// (K-major) and W [E][Kd][N].  swiglu: also the fused dSwiGLU epilogue, with H
// [rows, 2N], p [rows] (null: 1), out = dH [rows, 2N], dprob_part [rows, ceil(N/256)].
cudaError_t launch_tc_dgrad(bool swiglu, int rows, const void* A, int Kd, const void* W, int E,
                            int N, const int32_t* offsets, const float* prob, const void* H,
                            void* out, float* dprob_part, int sms, int* status, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  CUtensorMap ma, mb;
  if (!encode_map(&ma, A, 0, (uint64_t)rows, (uint64_t)Kd, BM)) return cudaErrorInvalidValue;
  if (!encode_map(&mb, W, (uint64_t)E, (uint64_t)Kd, (uint64_t)N, 64)) return cudaErrorInvalidValue;
  BwdParams p{};
  p.offsets = offsets; p.prob = prob; p.H = static_cast<const __nv_bfloat16*>(H);
  p.out = static_cast<__nv_bfloat16*>(out); p.dprob_part = dprob_part;
  p.E = E; p.Kd = Kd; p.M = 0; p.N = N; p.status = status; p.wait_limit_ns = 2000000000ull;
  const int64_t tiles_max = (ceil_div(rows, BM) + E) * ceil_div(N, BN);
  const int grid = (int)(tiles_max < sms ? tiles_max : sms);
  return swiglu ? launch_kind<kDgradSwiGLU>(ma, mb, mb, p, grid, s)
                : launch_kind<kDgradPlain>(ma, mb, mb, p, grid, s);
}

// Weight gradient of every expert: dW_e = A_e^T B_e with A [rows, M] and
// B [rows, N] (the expert's rows offsets[e]..offsets[e+1]), out [E][M][N];
// experts without rows get zeros.
cudaError_t launch_tc_wgrad(int rows, const void* A, int M, const void* B, int N, int E,
                            const int32_t* offsets, void* out, int sms, int* status,
                            cudaStream_t s) {
  CUtensorMap ma, mb;
  const uint64_t r = rows > 0 ? (uint64_t)rows : 1;  // a map needs a non-empty extent
  constexpr uint32_t kbox = BwdCfg<kWgrad>::BK;
  if (!encode_map(&ma, A, 0, r, (uint64_t)M, kbox)) return cudaErrorInvalidValue;
  if (!encode_map(&mb, B, 0, r, (uint64_t)N, kbox)) return cudaErrorInvalidValue;
  BwdParams p{};
  p.offsets = offsets; p.out = static_cast<__nv_bfloat16*>(out);
  p.E = E; p.Kd = 0; p.M = M; p.N = N; p.status = status; p.wait_limit_ns = 2000000000ull;
  CUtensorMap mc;  // the output dW [E][M][N], stored in {64, 32, 1} boxes
  if (!encode_map(&mc, out, (uint64_t)E, (uint64_t)M, (uint64_t)N, 32)) return cudaErrorInvalidValue;
  const int64_t tiles = (int64_t)E * ceil_div(M, BM) * ceil_div(N, BN);
  const int grid = (int)(tiles < sms ? tiles : sms);
  return launch_kind<kWgrad>(ma, mb, mc, p, grid, s);
}

}  // namespace moe
