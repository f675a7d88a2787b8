// moe_permute_noalloc: the dispatch step (moe_permute) without a workspace
// argument, for callers that cannot allocate device memory.
//
// Who needs it: code that runs inside a host framework which owns every byte
// of device memory and exposes no allocator to its plugins, and serving loops
// that must never allocate after start-up (a cudaMalloc can stall the whole
// device).  Such a caller still provides its inputs and outputs, but has no
// way to provide the per-chunk scratch tables moe_permute keeps in the
// workspace.  Here those tables live in a fixed array compiled into the
// library instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (kScratchInts * 2 int32 = 2 MiB) until the process exits.
// Host code cannot use the array's name as a device address (on the host it
// names a stand-in object), so the first call on each device looks up the
// real address with cudaGetSymbolAddress while that device is current, and
// passes it to the kernels.
#include <mutex>

#include "common.cuh"

namespace moe {
cudaError_t launch_permute_maps(const moe_config_t&, const int32_t*, const float*, int32_t*,
                                int32_t*, int32_t*, int32_t*, int32_t*, int32_t*, float*, int*,
                                cudaStream_t, bool hist_ready = false);
cudaError_t launch_scatter_rows(const moe_config_t&, const void*, const int32_t*, void*, int,
                                int*, cudaStream_t, bool after_maps = false);
int num_chunks(int T);
moe_status_t validate_config(const moe_config_t* c);
int* device_status_word();
}  // namespace moe

namespace {

// Two tables of ceil(T/32) x E int32: per-chunk expert histograms and their
// prefix sums over the chunks.
constexpr int64_t kScratchInts = 262144;

static __device__ __align__(256) int32_t g_permute_scratch[2 * kScratchInts];

constexpr int kMaxDevices = 64;
struct NoAllocDevice {
  int32_t* scratch = nullptr;
  int sms = 0;
  bool ready = false;
};
NoAllocDevice g_noalloc[kMaxDevices];
std::mutex g_noalloc_mu;

// Once per device, with that device current: the device address of the
// scratch array and the SM count.
moe_status_t noalloc_setup(NoAllocDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc[dev];
  if (!d.ready) {
    int32_t* ptr = nullptr;
    if (cudaGetSymbolAddress((void**)&ptr, g_permute_scratch) != cudaSuccess || !ptr)
      return MOE_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    d.scratch = ptr;
    d.sms = sms;
    d.ready = true;
  }
  *out = &d;
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status_t moe_permute_noalloc(const moe_config_t* cfg, const void* x,
                                            const int32_t* topk_idx, const float* topk_prob,
                                            void* x_perm, int32_t* counts, int32_t* offsets,
                                            int32_t* dst_row, int32_t* src_token,
                                            float* perm_prob, moe_stream_t stream) {
  // The same argument rules as moe_permute, minus the workspace.
  moe_status_t st = moe::validate_config(cfg);
  if (st != MOE_OK) return st;
  if ((int64_t)moe::num_chunks(cfg->T) * cfg->E > kScratchInts)
    return MOE_ERR_UNSUPPORTED;  // the fixed scratch holds ceil(T/32) * E <= 262144 entries
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!topk_idx || !dst_row || !src_token)) return MOE_ERR_INVALID_ARG;
  if ((x == nullptr) != (x_perm == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  // The status word first: a failed lookup (or an injected failure) returns
  // MOE_ERR_CUDA before anything is queued, as every other entry point does.
  int* status = moe::device_status_word();
  if (!status) return MOE_ERR_CUDA;
  NoAllocDevice* d = nullptr;
  if ((st = noalloc_setup(&d)) != MOE_OK) return st;
  // Both tables are fully rewritten by every call before they are read, so
  // nothing needs clearing between calls.
  int32_t* hist = d->scratch;
  int32_t* base = d->scratch + kScratchInts;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = moe::launch_permute_maps(*cfg, topk_idx, topk_prob, hist, base, counts, offsets,
                                           dst_row, src_token, perm_prob, status, s);
  if (e == cudaSuccess && x)
    e = moe::launch_scatter_rows(*cfg, x, dst_row, x_perm, d->sms, status, s, true);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
