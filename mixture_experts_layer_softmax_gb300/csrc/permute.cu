// Dispatch: expert-contiguous permutation of the T*K (token, slot) pairs.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (review),
// §2.1 "Dispatch" (tokens are permuted so each expert's rows are contiguous,
// with per-expert counts and offsets) and §4.3.1 (permutation fusion);
// §4.3.3 asks for sync-free kernels: counts and offsets never leave the device.
//
// Positions are decided without atomics, so the permutation is unique and
// bit-reproducible: inside an expert's segment rows are in ascending token
// order.  Tokens are cut into chunks of 32 (one warp each):
//   1. chunk_hist:   hist[c][e] = pairs of chunk c routed to e
//   2. chunk_scan:   base[c][e] = sum_{c' < c} hist[c'][e]; counts[e] (warp per expert);
//                    for small batches (ceil(T/32) * E <= 8192) every block of
//                    step 3 redoes this scan in shared memory instead (one
//                    launch fewer)
//   3. chunk_ranks:  offsets = exclusive scan of counts; for every pair
//                    dst_row = offsets[e] + base[c][e] + rank inside the chunk
//                    (ranks from ballots over the lanes' expert ids);
//                    src_token, perm_prob are the inverse maps.
//   With an expert capacity C (skill page "emerging-techniques-moe-training",
//   "Capacity Factor Tuning"), counts[e] = min(slots, C) and a pair whose
//   position base + rank inside its expert is >= C is dropped (dst_row = -1):
//   every expert keeps its first C slots in ascending token order.
//   4. scatter_rows: each token's row is read once and written to its K
//                    destinations with 16-byte vectors.
#include "common.cuh"

namespace moe {

constexpr int kChunk = 32;

// Programmatic dependent launch: a kernel launched with pdl_launch may be
// scheduled while the previous kernel on the stream is still finishing; it
// waits here, before its first memory access, until that kernel has
// completed and its writes are visible (a no-op without a dependency).  The
// previous kernel lets it be scheduled early with pdl_trigger.
MOE_D void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_D void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
static cudaError_t launch_maybe_pdl(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block,
                                   size_t smem, cudaStream_t s, Args... args);

template <typename... KArgs, typename... Args>
static cudaError_t pdl_launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// With pdl false a plain launch: the kernel's pdl_wait returns at once and
// it starts only after everything before it on the stream has completed.
template <typename... KArgs, typename... Args>
static cudaError_t launch_maybe_pdl(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block,
                                   size_t smem, cudaStream_t s, Args... args) {
  if (pdl) return pdl_launch(kern, grid, block, smem, s, args...);
  kern<<<grid, block, smem, s>>>(args...);
  return cudaGetLastError();
}

// ---- per-warp steps ----------------------------------------------------------

// hist[c][e] for chunk c; `my` is this warp's [E] shared-memory counter row.
MOE_D void hist_chunk(int c, int lane, int32_t* my, const int32_t* __restrict__ idx, int T, int K,
                      int E, int32_t* __restrict__ hist, int* status) {
  for (int e = lane; e < E; e += 32) my[e] = 0;
  __syncwarp();
  const int64_t t = (int64_t)c * kChunk + lane;
  if (t < T)
    for (int k = 0; k < K; ++k) {
      const int e = __ldg(idx + t * K + k);
      if (e >= 0 && e < E)
        atomicAdd(&my[e], 1);
      else
        report(status, MOE_ERR_DEVICE_BOUNDS);
    }
  __syncwarp();
  for (int e = lane; e < E; e += 32) hist[(int64_t)c * E + e] = my[e];
  __syncwarp();
}

// Exclusive scan of hist[:, e] over the chunks into base[:, e]; counts[e] =
// the slots expert e keeps (all of them, or at most `cap` when cap > 0).
MOE_D void scan_expert(int e, int lane, const int32_t* hist, int NC, int E, int cap,
                       int32_t* base, int32_t* counts) {
  int running = 0;
  for (int c0 = 0; c0 < NC; c0 += 32) {
    const int c = c0 + lane;
    const int v = c < NC ? hist[(int64_t)c * E + e] : 0;  // global or shared memory
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (c < NC) base[(int64_t)c * E + e] = running + incl - v;
    running += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) counts[e] = (cap > 0 && running > cap) ? cap : running;
}

// Whole block (256 threads): s_off[0..E] = exclusive scan of counts[0..E)
// (zero past E, s_off[256] the total); block 0 also writes offsets_out.
MOE_D void block_offsets(const int32_t* __restrict__ counts, int E, int32_t* s_off,
                         int32_t* s_warp, int32_t* offsets_out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = threadIdx.x;
  const int v = e < E ? __ldg(counts + e) : 0;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += s_warp[w];
  s_off[e] = wbase + incl - v;
  if (e == 255) s_off[256] = wbase + incl;
  __syncthreads();
  if (blockIdx.x == 0 && offsets_out && e <= E) offsets_out[e] = s_off[e];
  if (blockIdx.x == 0 && offsets_out && E == 256 && e == 0) offsets_out[256] = s_off[256];
}

// Destination rows of chunk c's pairs: the pair's position among expert e's
// slots is base[c][e] + its rank among the chunk's earlier tokens routed to e
// (from ballots over the lanes' expert-id bits, E <= 256); dst_row =
// offsets[e] + position, or -1 when cap > 0 and position >= cap (dropped:
// beyond the expert's capacity).  src_token and perm_prob are the inverse
// maps of the kept pairs.  Expert ids outside [0, E) get dst_row = -1
// (reported by the histogram step).
MOE_D void ranks_chunk(int c, int lane, const int32_t* __restrict__ idx,
                       const float* __restrict__ prob, int T, int K, int E, int cap,
                       const int32_t* base, const int32_t* s_off, int32_t* __restrict__ dst_row,
                       int32_t* __restrict__ src_token, float* __restrict__ perm_prob,
                       int* status) {
  const int64_t t = (int64_t)c * kChunk + lane;
  const bool valid = t < T;
  const unsigned lt_mask = (1u << lane) - 1u;
  int my_e[16], rank[16];
  for (int k = 0; k < K; ++k) {
    const int e = valid ? __ldg(idx + t * K + k) : -1;
    my_e[k] = (e >= 0 && e < E) ? e : -1;
    rank[k] = 0;
  }
  for (int k2 = 0; k2 < K; ++k2) {
    const int v = my_e[k2];
    const unsigned present = __ballot_sync(0xffffffffu, v >= 0);
    unsigned bits[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) bits[b] = __ballot_sync(0xffffffffu, (v >> b) & 1);
    for (int k = 0; k < K; ++k) {
      const int e = my_e[k];
      unsigned m = present & lt_mask;
#pragma unroll
      for (int b = 0; b < 8; ++b) m &= ((e >> b) & 1) ? bits[b] : ~bits[b];
      rank[k] += __popc(m);
    }
  }
  if (valid) {
    for (int k = 0; k < K; ++k) {
      const int e = my_e[k];
      if (e < 0) {
        dst_row[t * K + k] = -1;
        continue;
      }
      const int pos = base[(int64_t)c * E + e] + rank[k];  // global or shared memory
      if (cap > 0 && pos >= cap) {
        dst_row[t * K + k] = -1;
        continue;
      }
      const int r = s_off[e] + pos;
      if (r < 0 || (int64_t)r >= (int64_t)T * K) {  // histograms that do not match idx
        report(status, MOE_ERR_DEVICE_BOUNDS);
        dst_row[t * K + k] = -1;
        continue;
      }
      dst_row[t * K + k] = r;
      src_token[r] = (int32_t)t;
      if (perm_prob) perm_prob[r] = prob ? __ldg(prob + t * K + k) : 1.f;
    }
  }
}

// Token t's row, read once (16-byte vectors, up to 8 per lane in flight) and
// written to its K destination rows.  The first batch of the row's vectors is
// loaded before pdl_wait: x is never written by the map steps this kernel
// follows (and was final before they started), so under programmatic
// dependent launch that read overlaps the previous kernel's tail; the
// destination rows are read only after the wait.
template <typename T, int KMAX>
MOE_D void scatter_token(int64_t t, int lane, const T* __restrict__ x,
                         const int32_t* __restrict__ dst_row,
                         int ntok, int K, int h, T* __restrict__ x_perm, int* status) {
  constexpr int V = Vec<T>::N;
  constexpr int kMaxVec = 8;
  const int nvec = h / V;
  const int64_t P = (int64_t)ntok * K;
  const T* src = x + t * h;
  Vec<T> buf[kMaxVec];
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    const int v = i * 32 + lane;
    if (v < nvec) buf[i] = ld16_stream(src + (int64_t)v * V);
  }
  pdl_wait();
  T* dst[KMAX];
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    dst[k] = nullptr;
    if (k < K) {
      const int r = __ldg(dst_row + t * K + k);
      if (r >= 0 && r < P)
        dst[k] = x_perm + (int64_t)r * h;
      else if (r >= P)
        report(status, MOE_ERR_DEVICE_BOUNDS);
    }
  }
  for (int v0 = 0; v0 < nvec; v0 += 32 * kMaxVec) {
    if (v0 > 0) {
#pragma unroll
      for (int i = 0; i < kMaxVec; ++i) {
        const int v = v0 + i * 32 + lane;
        if (v < nvec) buf[i] = ld16_stream(src + (int64_t)v * V);
      }
    }
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (!dst[k]) continue;
#pragma unroll
      for (int i = 0; i < kMaxVec; ++i) {
        const int v = v0 + i * 32 + lane;
        if (v < nvec) st16(dst[k] + (int64_t)v * V, buf[i]);
      }
    }
  }
}

// ---- separate kernels -------------------------------------------------------

// One warp per chunk of 32 tokens; 8 warps per block.
__global__ void __launch_bounds__(256) chunk_hist_kernel(const int32_t* __restrict__ idx, int T,
                                                         int K, int E, int NC,
                                                         int32_t* __restrict__ hist, int* status) {
  extern __shared__ int32_t sh[];  // [8][E]
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x * 8 + warp;
  if (c < NC) hist_chunk(c, lane, sh + warp * E, idx, T, K, E, hist, status);
}

// Warp per expert: exclusive scan of hist[:, e] over the chunks.
__global__ void __launch_bounds__(256) chunk_scan_kernel(const int32_t* __restrict__ hist, int NC,
                                                         int E, int cap,
                                                         int32_t* __restrict__ base,
                                                         int32_t* __restrict__ counts) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (e < E) scan_expert(e, lane, hist, NC, E, cap, base, counts);
}

// Block: exclusive scan of counts into shared offsets, then one warp per chunk
// computes every pair's destination row.
__global__ void __launch_bounds__(256) chunk_ranks_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ prob, int T, int K, int E, int cap,
    int NC, const int32_t* __restrict__ base, const int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets_out, int32_t* __restrict__ dst_row,
    int32_t* __restrict__ src_token, float* __restrict__ perm_prob, int* status) {
  __shared__ int32_t s_off[257];
  __shared__ int32_t s_warp[8];
  block_offsets(counts, E, s_off, s_warp, offsets_out);
  const int c = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (c < NC)
    ranks_chunk(c, threadIdx.x & 31, idx, prob, T, K, E, cap, base, s_off, dst_row, src_token,
                perm_prob, status);
}

// Steps 2 and 3 in one kernel for small batches (NC * E <= kScanInBlock):
// every block copies the chunk histograms into shared memory and scans them
// per expert itself (a few thousand integers, L2-resident), so the separate
// scan launch goes away; block 0 writes counts and offsets.  Same per-warp
// steps, same maps.
constexpr int64_t kScanInBlock = 8192;

__global__ void __launch_bounds__(256) chunk_scan_ranks_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ prob, int T, int K, int E, int cap,
    int NC, const int32_t* __restrict__ hist, int32_t* __restrict__ counts_out,
    int32_t* __restrict__ offsets_out, int32_t* __restrict__ dst_row,
    int32_t* __restrict__ src_token, float* __restrict__ perm_prob, int* status) {
  extern __shared__ int32_t sh[];
  pdl_wait();
  pdl_trigger();
  int32_t* s_base = sh;                        // [NC][E]: hist, then base in place
  int32_t* s_cnt = s_base + (int64_t)NC * E;   // [E]
  int32_t* s_off = s_cnt + E;                  // [E + 1]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t i = threadIdx.x; i < (int64_t)NC * E; i += blockDim.x) s_base[i] = __ldg(hist + i);
  __syncthreads();
  for (int e = warp; e < E; e += 8) scan_expert(e, lane, s_base, NC, E, cap, s_base, s_cnt);
  __syncthreads();
  if (warp == 0) {  // s_off = exclusive scan of the counts
    int running = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? s_cnt[e] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (e < E) {
        s_off[e] = running + incl - v;
        if (blockIdx.x == 0) {
          offsets_out[e] = running + incl - v;
          counts_out[e] = v;
        }
      }
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      s_off[E] = running;
      if (blockIdx.x == 0) offsets_out[E] = running;
    }
  }
  __syncthreads();
  const int c = blockIdx.x * 8 + warp;
  if (c < NC)
    ranks_chunk(c, lane, idx, prob, T, K, E, cap, s_base, s_off, dst_row, src_token, perm_prob,
                status);
}

// One warp per token (the grid covers every token, so the block scheduler
// balances the load).
template <typename T, int KMAX>
__global__ void __launch_bounds__(256) scatter_rows_kernel(const T* __restrict__ x,
                                                           const int32_t* __restrict__ dst_row,
                                                           int ntok, int K, int h,
                                                           T* __restrict__ x_perm, int* status) {
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t < ntok)
    scatter_token<T, KMAX>(t, threadIdx.x & 31, x, dst_row, ntok, K, h, x_perm, status);
  else
    pdl_wait();
}

int num_chunks(int T) { return (int)ceil_div(T, kChunk); }

// Step 1 alone: the per-chunk histograms of idx (the router's hand-off to
// the dispatch when its own epilogue does not produce them).
cudaError_t launch_chunk_hist(const moe_config_t& c, const int32_t* idx, int32_t* hist,
                              int* status, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const int NC = num_chunks(c.T);
  chunk_hist_kernel<<<(unsigned)ceil_div(NC, 8), 256, 8 * c.E * sizeof(int32_t), s>>>(
      idx, c.T, c.K, c.E, NC, hist, status);
  return cudaGetLastError();
}

// hist_ready: hist already holds idx's chunk histograms (written by the
// router), so step 1 is skipped.
cudaError_t launch_permute_maps(const moe_config_t& c, const int32_t* idx, const float* prob,
                                int32_t* hist, int32_t* base, int32_t* counts, int32_t* offsets,
                                int32_t* dst_row, int32_t* src_token, float* perm_prob,
                                int* status, cudaStream_t s, bool hist_ready) {
  const int NC = num_chunks(c.T);
  if (c.T == 0) {
    // no rows: counts and offsets are all zero
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.E, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (c.E + 1), s);
    return e;
  }
  const int blocks = (int)ceil_div(NC, 8);
  if (!hist_ready)
    chunk_hist_kernel<<<blocks, 256, 8 * c.E * sizeof(int32_t), s>>>(idx, c.T, c.K, c.E, NC, hist,
                                                                    status);
  if ((int64_t)NC * c.E <= kScanInBlock) {
    const size_t bytes = sizeof(int32_t) * ((size_t)NC * c.E + 2 * c.E + 1);
    return pdl_launch(chunk_scan_ranks_kernel, dim3(blocks), dim3(256), bytes, s, idx, prob, c.T,
                      c.K, c.E, c.capacity, NC, (const int32_t*)hist, counts, offsets, dst_row,
                      src_token, perm_prob, status);
  }
  chunk_scan_kernel<<<(unsigned)ceil_div(c.E, 8), 256, 0, s>>>(hist, NC, c.E, c.capacity, base,
                                                                counts);
  chunk_ranks_kernel<<<blocks, 256, 0, s>>>(idx, prob, c.T, c.K, c.E, c.capacity, NC, base, counts,
                                            offsets, dst_row, src_token, perm_prob, status);
  return cudaGetLastError();
}

int scatter_grid(int ntok, int sms) {
  const int64_t need = ceil_div(ntok, 8);
  const int64_t cap = (int64_t)sms * 8;
  return (int)(need < cap ? (need > 0 ? need : 1) : cap);
}

template <typename T>
static cudaError_t scatter_t(const moe_config_t& c, const void* x, const int32_t* dst_row,
                             void* x_perm, int* status, cudaStream_t s, bool pdl) {
  const unsigned grid = (unsigned)ceil_div(c.T, 8);
  const T* xs = static_cast<const T*>(x);
  T* xp = static_cast<T*>(x_perm);
  if (c.K <= 2)
    return launch_maybe_pdl(pdl, scatter_rows_kernel<T, 2>, dim3(grid), dim3(256), 0, s, xs, dst_row,
                            c.T, c.K, c.h, xp, status);
  else if (c.K <= 4)
    return launch_maybe_pdl(pdl, scatter_rows_kernel<T, 4>, dim3(grid), dim3(256), 0, s, xs, dst_row,
                            c.T, c.K, c.h, xp, status);
  else if (c.K <= 8)
    return launch_maybe_pdl(pdl, scatter_rows_kernel<T, 8>, dim3(grid), dim3(256), 0, s, xs, dst_row,
                            c.T, c.K, c.h, xp, status);
  else
    return launch_maybe_pdl(pdl, scatter_rows_kernel<T, 16>, dim3(grid), dim3(256), 0, s, xs, dst_row,
                            c.T, c.K, c.h, xp, status);
  return cudaGetLastError();
}

// after_maps: the launch directly follows this library's map steps on the
// stream, so it may overlap their tail (programmatic dependent launch); any
// other caller gets a plain launch.
cudaError_t launch_scatter_rows(const moe_config_t& c, const void* x, const int32_t* dst_row,
                                void* x_perm, int sms, int* status, cudaStream_t s,
                                bool after_maps) {
  (void)sms;
  if (c.T == 0) return cudaSuccess;
  if (c.dtype == MOE_BF16)
    return scatter_t<__nv_bfloat16>(c, x, dst_row, x_perm, status, s, after_maps);
  return scatter_t<float>(c, x, dst_row, x_perm, status, s, after_maps);
}

}  // namespace moe
