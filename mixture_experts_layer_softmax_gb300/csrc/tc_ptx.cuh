// Blackwell (sm_100 family, built for sm_103a) building blocks written as
// inline PTX: mbarriers with bounded waits, TMA tensor loads, and the
// tcgen05 tensor-core path (TMEM allocation, shared-memory matrix
// descriptors, instruction descriptors, MMA, commit, TMEM loads).
//
// Encodings follow the PTX ISA's tcgen05 chapter: the shared memory
// descriptor (start address >> 4 in bits 0-13, leading-byte offset >> 4 in
// 16-29, stride-byte offset >> 4 in 32-45, version 1 in 46-47, swizzle mode in
// 61-63) and the kind::f16 instruction descriptor (D format in bits 4-5, A/B
// formats in 7-9 / 10-12, A/B major-ness in 15 / 16, N >> 3 in 17-22,
// M >> 4 in 24-28).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {
namespace tc {

MOE_D uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

MOE_D uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier -------------------------------------------------------------
MOE_D void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
MOE_D void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
MOE_D void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
MOE_D void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
MOE_D void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
MOE_D bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P1;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P1;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with `parity` to complete.  Gives up after
// `limit_ns` of wall time or `max_polls` polls (whichever first), or as soon as
// another role of the block raised *abort.  On giving up it records
// MOE_ERR_TIMEOUT (unless another role already aborted) and returns false.
struct WaitCtl {
  int* status;
  volatile int* abort;
  uint64_t limit_ns;
  int64_t max_polls;
};

MOE_D bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (int64_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (w.abort && *w.abort) return false;
      if ((w.max_polls > 0 && i >= w.max_polls) || globaltimer_ns() - t0 > w.limit_ns) {
        report(w.status, MOE_ERR_TIMEOUT);
        if (w.abort) *w.abort = 1;
        return false;
      }
    }
  }
}

// The same bounded wait with cluster-scope acquire: for a barrier that CTAs
// of the cluster arrive on remotely (release.cluster) after writing this
// CTA's shared memory.
MOE_D bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P1;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 P1, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P1;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
MOE_D bool mbar_wait_cluster(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (int64_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (w.abort && *w.abort) return false;
      if ((w.max_polls > 0 && i >= w.max_polls) || globaltimer_ns() - t0 > w.limit_ns) {
        report(w.status, MOE_ERR_TIMEOUT);
        if (w.abort) *w.abort = 1;
        return false;
      }
    }
  }
}

// ---- clusters -----------------------------------------------------------------
MOE_D uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address of this CTA's shared-memory location `addr` in CTA `rank`.
MOE_D uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
  return out;
}
MOE_D void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Arrive on an mbarrier of any CTA of the cluster (address from mapa).
MOE_D void arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}
MOE_D void st_cluster_f32x4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// ---- TMA --------------------------------------------------------------------
MOE_D void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
// Four rows of a 2-D tensor (box one row high): rows r0..r3 at column c0,
// written to shared memory one after the other (the map's swizzle applies by
// shared-memory address, as for a 4-row box).
MOE_D void tma_gather4(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t r0, int32_t r1,
                       int32_t r2, int32_t r3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
      "r"(bar)
      : "memory");
}
// Untiled bulk copy of `bytes` (a multiple of 16) from global to shared
// memory, both addresses 16-byte aligned; completes as transaction bytes on
// the mbarrier `bar`.
MOE_D void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
MOE_D void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- tcgen05 ------------------------------------------------------------------
MOE_D void tmem_alloc(uint32_t holder_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   holder_smem),
               "r"(ncols)
               : "memory");
}
MOE_D void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MOE_D void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
MOE_D void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_D void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major operand tile in the 128-byte swizzle layout written by TMA with
// CU_TENSOR_MAP_SWIZZLE_128B and a 64-element (bf16) inner box: rows of 128 B,
// 8-row groups 1024 B apart.  `addr` must lie in a 1024-byte-aligned tile.
MOE_D uint64_t desc_kmajor_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;               // leading-byte offset (unused when swizzled K-major)
  d |= (uint64_t)(1024u >> 4) << 32;    // stride-byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;               // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;               // 128-byte swizzle
  return d;
}

// MN-major operand tile in the 128-byte swizzle layout: TMA box {64 (MN, inner),
// rows (K)} gives K-rows of 128 B holding 64 consecutive MN elements; atoms of
// 64 MN elements are `lbo` bytes apart, 8-row K groups 1024 B apart.
MOE_D uint64_t desc_mnmajor_sw128(uint32_t addr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// kind::f16 instruction descriptor: bf16 x bf16 -> fp32, dense.
// a_mn / b_mn: operand is MN-major (transposed) instead of K-major.
MOE_HD constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn = false, bool b_mn = false) {
  return (1u << 4)                      // D: f32
         | (1u << 7)                    // A: bf16
         | (1u << 10)                   // B: bf16
         | ((a_mn ? 1u : 0u) << 15)     // A major
         | ((b_mn ? 1u : 0u) << 16)     // B major
         | ((uint32_t)(N >> 3) << 17)   // N >> 3
         | ((uint32_t)(M >> 4) << 24);  // M >> 4
}

MOE_D void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// ---- block-scaled MMA (kind::mxf8f6f4) ------------------------------------------
// Instruction descriptor for E4M3 x E4M3 -> fp32 with E8M0 scales, both
// operands K-major: B scale id in bits 4-5, A/B formats (E4M3 = 0) in 7-9 /
// 10-12, N >> 3 in 17-22, scale format UE8M0 (1) in bit 23, M >> 4 in 24-28,
// A scale id in 29-30.  The scale id picks the byte of each 32-bit TMEM scale
// word (one 32-element K block per MMA of K = 32).
MOE_HD constexpr uint32_t idesc_mxf8_e4m3(int M, int N, int sfa_id, int sfb_id) {
  return ((uint32_t)sfb_id << 4) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
         ((uint32_t)(M >> 4) << 24) | ((uint32_t)sfa_id << 29);
}

MOE_D void mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                    uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Shared-memory descriptor of one 512-byte scale atom as the source of a
// tcgen05.cp 32x128b: 32 rows of 16 bytes, no swizzle, 8-row core-matrix
// groups 128 bytes apart.
MOE_D uint64_t desc_sf_atom(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Copy 32 rows x 128 bits from shared memory into TMEM columns taddr ..
// taddr + 3 of all four lane quarters (row r to lane r of each quarter).
// Ordered before later tcgen05.mma of the same thread.
MOE_D void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread is done.
MOE_D void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i gets lane (base + i).
// The load and its completion wait are one asm statement, so no use of the
// destination registers can be scheduled before the data has arrived.
MOE_D void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// Three 32 lanes x 8 column loads (three column groups of the same lanes)
// and one wait, in one asm statement.
MOE_D void tmem_ld_32x32b_x8x3(uint32_t ta, uint32_t tb, uint32_t tcol, uint32_t (&a)[8],
                               uint32_t (&b)[8], uint32_t (&c)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%24];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%25];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%26];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]),
        "=r"(a[7]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]),
        "=r"(b[6]), "=r"(b[7]), "=r"(c[0]), "=r"(c[1]), "=r"(c[2]), "=r"(c[3]), "=r"(c[4]),
        "=r"(c[5]), "=r"(c[6]), "=r"(c[7])
      : "r"(ta), "r"(tb), "r"(tcol)
      : "memory");
}
// 32 lanes x 64 consecutive columns: two 32-column loads and one wait in a
// single asm statement.
MOE_D void tmem_ld_32x32b_x64(uint32_t taddr, uint32_t (&r)[64]) {
#define MOE_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), \
                  "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : MOE_R8(0), MOE_R8(8), MOE_R8(16), MOE_R8(24), MOE_R8(32), MOE_R8(40), MOE_R8(48),
        MOE_R8(56)
      : "r"(taddr), "r"(taddr + 32)
      : "memory");
#undef MOE_R8
}
MOE_D void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// The same 32 lanes x 64 columns without the wait, so the load overlaps other
// work; the registers may only be read after tmem_ld_wait_x64 on them.
MOE_D void tmem_ld_32x32b_x64_nowait(uint32_t taddr, uint32_t (&r)[64]) {
#define MOE_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), \
                  "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];"
      : MOE_R8(0), MOE_R8(8), MOE_R8(16), MOE_R8(24), MOE_R8(32), MOE_R8(40), MOE_R8(48),
        MOE_R8(56)
      : "r"(taddr), "r"(taddr + 32)
      : "memory");
#undef MOE_R8
}
// Waits for this thread's TMEM loads.  The 64 destination registers are
// operands (read and written), so no use of them can be scheduled before the
// wait.
MOE_D void tmem_ld_wait_x64(uint32_t (&r)[64]) {
#define MOE_W8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), \
                  "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : MOE_W8(0), MOE_W8(8), MOE_W8(16), MOE_W8(24), MOE_W8(32), MOE_W8(40),
                 MOE_W8(48), MOE_W8(56)
               :
               : "memory");
#undef MOE_W8
}

// ---- CTA pairs (cta_group::2, cluster of two CTAs) -------------------------------
// A 2-D tile load into this CTA's shared memory whose completion is counted
// on the mbarrier `bar_cluster` (a shared::cluster address, e.g. the even
// CTA's barrier through mapa).
MOE_D void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                            uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster)
      : "memory");
}
MOE_D void tmem_alloc_pair(uint32_t holder, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(holder),
               "r"(ncols)
               : "memory");
}
MOE_D void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
MOE_D void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// bf16 MMA over both CTAs' shared memory (issued by the even CTA).
MOE_D void mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once) on the barrier at this shared offset in every CTA of `mask`
// when all MMAs issued so far by this thread are complete.
MOE_D void commit_pair_multicast(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// ---- host: the driver's tensor-map encoder ------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled, looked up once through the runtime (the library
// does not link against the driver library); null if the driver lacks it.
inline EncodeTiledFn encode_tiled_fn() {
  static const EncodeTiledFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

}  // namespace tc
}  // namespace moe
