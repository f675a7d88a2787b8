// The C ABI (include/moe.h): argument validation, workspace carving and the
// order of the layer's steps.  Host code here only validates and enqueues; it
// never reads device memory or synchronises (except moe_get_error).
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "common.cuh"

namespace moe {
cudaError_t launch_router(const moe_config_t&, const void*, const float*, const float*,
                          const float*, float*, int32_t*, float*, uint8_t*, const RouterScratch&,
                          int, int*, cudaStream_t, int32_t* hist = nullptr);
cudaError_t launch_router_select(const moe_config_t&, const float*, const float*, int32_t*,
                                 float*, uint8_t*, cudaStream_t);
cudaError_t launch_permute_maps(const moe_config_t&, const int32_t*, const float*, int32_t*,
                                int32_t*, int32_t*, int32_t*, int32_t*, int32_t*, float*, int*,
                                cudaStream_t, bool hist_ready = false);
cudaError_t launch_scatter_rows(const moe_config_t&, const void*, const int32_t*, void*, int,
                                int*, cudaStream_t, bool after_maps = false);
cudaError_t launch_combine(const moe_config_t&, const void*, const int32_t*, const float*,
                           const void*, void*, int, int*, cudaStream_t);
cudaError_t launch_expert_gemm_simt(const moe_config_t&, int, int, const void*, const int32_t*,
                                    const float*, const void*, const void*, void*, void*,
                                    cudaStream_t);
cudaError_t launch_expert_gemm_tc(const moe_config_t&, int, int, const void*, const int32_t*,
                                  const float*, const void*, const void*, void*, void*, int, int*,
                                  cudaStream_t, const int32_t*);
cudaError_t launch_bounded_wait_probe(int64_t, int*, cudaStream_t);
cudaError_t launch_aux_loss(const moe_config_t&, const float*, const int32_t*, float, float, float*,
                            float*, double*, double*, int32_t*, float*, int*, cudaStream_t);
cudaError_t launch_tc_dgrad(bool, int, const void*, int, const void*, int, int, const int32_t*,
                            const float*, const void*, void*, float*, int, int*, cudaStream_t);
cudaError_t launch_tc_wgrad(int, const void*, int, const void*, int, int, const int32_t*, void*,
                            int, int*, cudaStream_t);
cudaError_t launch_dprob_reduce(const float*, int, int, float*, cudaStream_t);
cudaError_t launch_router_bwd(const moe_config_t&, const float*, const int32_t*, const float*,
                              const int32_t*, const float*, float*, float*, int*, cudaStream_t);
cudaError_t launch_router_wgrad(const moe_config_t&, const void*, const int32_t*, const int32_t*,
                                const float*, float*, float*, cudaStream_t);
cudaError_t launch_bwd_combine(const moe_config_t&, const void*, const int32_t*, const void*,
                               const float*, const int32_t*, const float*, const float*, void*,
                               float*, int, int*, cudaStream_t);
cudaError_t launch_scatter_topk_grad(const moe_config_t&, const float*, const int32_t*, float*,
                                     cudaStream_t);
cudaError_t launch_dense_router_wgrad(const moe_config_t&, const float*, const void*, float*,
                                      float*, cudaStream_t);
cudaError_t launch_dense_router_dx(const moe_config_t&, const float*, const float*, float*,
                                   cudaStream_t);
size_t mxfp8_scale_bytes(int64_t rows, int K, int groups);
cudaError_t launch_mxfp8_quantize(int, int, int, const int32_t*, const void*, uint8_t*, uint8_t*,
                                  int, cudaStream_t);
cudaError_t launch_scatter_quantize(const moe_config_t&, const void*, const int32_t*,
                                    const int32_t*, const int32_t*, uint8_t*, uint8_t*, int, int*,
                                    cudaStream_t);
cudaError_t launch_grouped_gemm_mxfp8(bool, int, const uint8_t*, const uint8_t*, int,
                                      const uint8_t*, const uint8_t*, int, int, int,
                                      const int32_t*, const float*, void*, uint8_t*, uint8_t*,
                                      int, int*, cudaStream_t);
}  // namespace moe

using namespace moe;

// Per-device status word: device-side checks record the first error here.
__device__ int g_moe_status = 0;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int* status = nullptr;
  int sms = 0;
  bool ready = false;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Test hook (moe_test_inject_cuda_failure): calls left that must fail as if
// their first CUDA runtime call had failed.
std::atomic<int> g_inject_failures{0};

// Stage timing (moe_set_stage_events): per host thread and pass, the caller's
// CUDA events that the layer calls record at their stage boundaries.
constexpr int kMaxStageEvents = 16;
struct StageEvents {
  cudaEvent_t ev[kMaxStageEvents] = {};
  int n = 0;
};
thread_local StageEvents g_stage_events[2];

// Records boundary i of pass p (MOE_PASS_FWD / MOE_PASS_BWD) on stream s when
// the calling thread registered an event for it; otherwise does nothing.
cudaError_t mark_stage(int pass, int i, cudaStream_t s) {
  const StageEvents& se = g_stage_events[pass];
  if (i >= se.n || !se.ev[i]) return cudaSuccess;
  return cudaEventRecord(se.ev[i], s);
}

// NVTX ranges around the steps of a layer pass (host-side annotations: a
// profiler attributes each step's launches to its range; no cost otherwise).
class NvtxStage {
 public:
  explicit NvtxStage(const char* name) { nvtxRangePushA(name); }
  void next(const char* name) {
    nvtxRangePop();
    nvtxRangePushA(name);
  }
  ~NvtxStage() { nvtxRangePop(); }
  NvtxStage(const NvtxStage&) = delete;
  NvtxStage& operator=(const NvtxStage&) = delete;
};

// Status-word address and SM count of the current device (looked up once per
// device, with that device current).
// (inject: a pending injected failure makes this call fail; moe_get_error
// looks the device up without consuming one.)
const DeviceInfo* device_info(bool inject = true) {
  if (inject)
    for (int n = g_inject_failures.load(); n > 0; n = g_inject_failures.load())
      if (g_inject_failures.compare_exchange_weak(n, n - 1)) return nullptr;  // injected failure
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_moe_status) != cudaSuccess) return nullptr;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return nullptr;
    d.status = static_cast<int*>(p);
    d.sms = sms;
    d.ready = true;
  }
  return &d;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t check_config(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->h < 1 || c->E < 1 || c->K < 1 || c->F < 1) return MOE_ERR_INVALID_ARG;
  if (c->K > c->E) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->score != MOE_SCORE_SOFTMAX && c->score != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (c->act != MOE_ACT_GELU && c->act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  if ((c->has_bias != 0 && c->has_bias != 1) || (c->n_shared != 0 && c->n_shared != 1))
    return MOE_ERR_INVALID_ARG;
  const uint32_t known = MOE_FLAG_RENORM | MOE_FLAG_FORCE_BALANCE | MOE_FLAG_VALIDATE_ONLY |
                         MOE_FLAG_SAVE_FOR_BWD | MOE_FLAG_GEMM_SIMT | MOE_FLAG_GEMM_1CTA |
                         MOE_FLAG_GEMM_2CTA | MOE_FLAG_HIST_FROM_ROUTER;
  if (c->flags & ~known) return MOE_ERR_INVALID_ARG;
  if ((c->flags & MOE_FLAG_GEMM_1CTA) && (c->flags & MOE_FLAG_GEMM_2CTA)) return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(c->aux_loss_coeff) || !std::isfinite(c->z_loss_coeff))
    return MOE_ERR_INVALID_ARG;
  if (c->capacity < 0) return MOE_ERR_INVALID_ARG;
  if (c->E > 256 || c->K > 16) return MOE_ERR_UNSUPPORTED;
  if (c->act == MOE_ACT_SWIGLU && c->has_bias) return MOE_ERR_UNSUPPORTED;
  const int vec = c->dtype == MOE_BF16 ? 8 : 4;
  if (c->h % vec || c->F % vec) return MOE_ERR_UNSUPPORTED;
  const int64_t R1 = c->act == MOE_ACT_SWIGLU ? 2LL * c->F : c->F;
  if ((int64_t)c->T * c->K >= (1LL << 31) || (int64_t)c->E * R1 >= (1LL << 31) ||
      (int64_t)c->E * c->h >= (1LL << 31))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t check_ws(const moe_config_t* c, const void* ws, size_t ws_bytes) {
  const size_t need = workspace_layout(*c).total;
  if (need == 0) return MOE_OK;
  if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

template <typename T> T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

RouterScratch router_scratch(const moe_config_t& c, void* ws) {
  const Workspace w = workspace_layout(c);
  RouterScratch rs;
  rs.w3 = at<__nv_bfloat16>(ws, w.router_w3);
  rs.parts = at<float>(ws, w.router_parts);
  rs.ldp = router_parts_ld(c.E);
  rs.ksplit = router_ksplit_max(c);
  rs.offs = at<int32_t>(ws, w.router_off);
  return rs;
}

__global__ void fill_shared_offsets(int32_t* off, int T) {
  off[0] = 0;
  off[1] = T;
}

bool use_tensor_cores(const moe_config_t& c) {
  return c.dtype == MOE_BF16 && !(c.flags & MOE_FLAG_GEMM_SIMT);
}

// src_token (tensor cores, FC1 only): A is the token rows x and GEMM row r
// reads x[src_token[r]] (the gather-fused FC1) instead of a permuted buffer.
cudaError_t run_expert_gemm(const moe_config_t& c, int fc, int rows, const void* A,
                            const int32_t* offsets, const float* prob, const void* w,
                            const void* bias, void* act_save, void* out, const DeviceInfo* d,
                            cudaStream_t s, const int32_t* src_token = nullptr) {
  if (use_tensor_cores(c))
    return launch_expert_gemm_tc(c, fc, rows, A, offsets, prob, w, bias, act_save, out, d->sms,
                                 d->status, s, src_token);
  if (src_token) return cudaErrorInvalidValue;
  return launch_expert_gemm_simt(c, fc, rows, A, offsets, prob, w, bias, act_save, out, s);
}

cudaError_t run_grouped_mlp(const moe_config_t& c, int rows, const void* x_perm,
                            const int32_t* offsets, const float* prob, const void* w1,
                            const void* b1, const void* w2, const void* b2, void* act_save,
                            void* a, void* y_perm, const DeviceInfo* d, cudaStream_t s,
                            const int32_t* src_token = nullptr) {
  cudaError_t e =
      run_expert_gemm(c, 1, rows, x_perm, offsets, prob, w1, b1, act_save, a, d, s, src_token);
  if (e != cudaSuccess) return e;
  return run_expert_gemm(c, 2, rows, a, offsets, prob, w2, b2, nullptr, y_perm, d, s);
}

// The backward covers the training configuration: bf16 SwiGLU experts with a
// renormalised router (softmax or sigmoid).
moe_status_t check_bwd_support(const moe_config_t& c) {
  if (c.dtype != MOE_BF16 || c.act != MOE_ACT_SWIGLU || !(c.flags & MOE_FLAG_RENORM))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Expert-FFN backward over permuted rows: dH and dprob partials (FC2 dgrad with
// the dSwiGLU epilogue), dW2, dx_perm (FC1 dgrad), dW1.
cudaError_t run_mlp_bwd(const moe_config_t& c, int rows, int E, const void* dy_rows,
                        const void* x_rows, const void* H, const void* a, const int32_t* offsets,
                        const float* prob, const void* w1, const void* w2, void* dH,
                        float* dprob_part, void* dx_rows, void* dw1, void* dw2,
                        const DeviceInfo* d, cudaStream_t s, int mark = -1) {
  const int F = c.F, h = c.h;
  if (rows == 0) {  // no rows: every weight gradient is zero
    cudaError_t e = cudaMemsetAsync(dw1, 0, (size_t)E * 2 * F * h * 2, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dw2, 0, (size_t)E * h * F * 2, s);
    return e;
  }
  // mark: the first of four stage boundaries to record after the four GEMMs
  // (FC2 dgrad, FC2 wgrad, FC1 dgrad, FC1 wgrad), or -1 for none
  auto after = [&](cudaError_t e, int k) {
    return (e == cudaSuccess && mark >= 0) ? mark_stage(MOE_PASS_BWD, mark + k, s) : e;
  };
  cudaError_t e = launch_tc_dgrad(true, rows, dy_rows, h, w2, E, F, offsets, prob, H, dH,
                                  dprob_part, d->sms, d->status, s);
  e = after(e, 0);
  if (e == cudaSuccess)
    e = launch_tc_wgrad(rows, dy_rows, h, a, F, E, offsets, dw2, d->sms, d->status, s);
  e = after(e, 1);
  if (e == cudaSuccess)
    e = launch_tc_dgrad(false, rows, dH, 2 * F, w1, E, h, offsets, nullptr, nullptr, dx_rows,
                        nullptr, d->sms, d->status, s);
  e = after(e, 2);
  if (e == cudaSuccess)
    e = launch_tc_wgrad(rows, dH, 2 * F, x_rows, h, E, offsets, dw1, d->sms, d->status, s);
  return after(e, 3);
}

}  // namespace

namespace moe {
// Internal accessors for other translation units of the library.
moe_status_t validate_config(const moe_config_t* c) { return check_config(c); }
int* device_status_word() {
  const DeviceInfo* d = device_info();
  return d ? d->status : nullptr;
}
}  // namespace moe

extern "C" {

int32_t moe_expert_capacity(int32_t T, int32_t K, int32_t E, float capacity_factor,
                            int32_t min_capacity) {
  if (T < 0 || K < 1 || E < 1 || !std::isfinite(capacity_factor) || capacity_factor <= 0.f)
    return -1;
  const double c = std::floor((double)capacity_factor * (double)T * (double)K / (double)E);
  const double m = c > (double)min_capacity ? c : (double)min_capacity;
  if (m > 2147483647.0) return -1;
  return (int32_t)m;
}

size_t moe_workspace_size(const moe_config_t* cfg) {
  if (check_config(cfg) != MOE_OK) return 0;
  return workspace_layout(*cfg).total;
}

moe_status_t moe_router_topk(const moe_config_t* cfg, const void* x, const float* w_r,
                             const float* gate_bias, const float* sel_bias, float* logits,
                             int32_t* topk_idx, float* topk_prob, uint8_t* routing_map, void* ws,
                             size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T > 0 && (!x || !w_r || !topk_idx || !topk_prob)) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(w_r)) return MOE_ERR_INVALID_ARG;
  // bf16 tokens: the tensor-core router keeps its split weight and partial
  // sums in the workspace; fp32 tokens need it only for E > 32 without logits
  const bool want_hist = (cfg->flags & MOE_FLAG_HIST_FROM_ROUTER) != 0;
  const bool need_ws = cfg->dtype == MOE_BF16 || (!logits && cfg->E > 32) || want_hist;
  if (need_ws && (st = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return st;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  if (cfg->T == 0) return MOE_OK;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  float* lg = logits;
  if (!lg && cfg->E > 32 && cfg->dtype != MOE_BF16) lg = at<float>(ws, workspace_layout(*cfg).logits);
  RouterScratch rs{};
  if (need_ws) rs = router_scratch(*cfg, ws);
  int32_t* hist = want_hist ? at<int32_t>(ws, workspace_layout(*cfg).hist) : nullptr;
  return cuda_status(launch_router(*cfg, x, w_r, gate_bias, sel_bias, lg, topk_idx, topk_prob,
                                   routing_map, rs, d->sms, d->status,
                                   static_cast<cudaStream_t>(stream), hist));
}

moe_status_t moe_router_topk_from_logits(const moe_config_t* cfg, const float* logits,
                                         const float* sel_bias, int32_t* topk_idx,
                                         float* topk_prob, uint8_t* routing_map,
                                         moe_stream_t stream) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T > 0 && (!logits || !topk_idx || !topk_prob)) return MOE_ERR_INVALID_ARG;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  if (cfg->T == 0) return MOE_OK;
  return cuda_status(launch_router_select(*cfg, logits, sel_bias, topk_idx, topk_prob,
                                          routing_map, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_permute(const moe_config_t* cfg, const void* x, const int32_t* topk_idx,
                         const float* topk_prob, void* x_perm, int32_t* counts, int32_t* offsets,
                         int32_t* dst_row, int32_t* src_token, float* perm_prob, void* ws,
                         size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!topk_idx || !dst_row || !src_token)) return MOE_ERR_INVALID_ARG;
  if ((x == nullptr) != (x_perm == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(x_perm)) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return st;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Workspace w = workspace_layout(*cfg);
  cudaError_t e = launch_permute_maps(*cfg, topk_idx, topk_prob, at<int32_t>(ws, w.hist),
                                      at<int32_t>(ws, w.chunk_base), counts, offsets, dst_row,
                                      src_token, perm_prob, d->status, s,
                                      (cfg->flags & MOE_FLAG_HIST_FROM_ROUTER) != 0);
  if (e == cudaSuccess && x)
    e = launch_scatter_rows(*cfg, x, dst_row, x_perm, d->sms, d->status, s, true);
  return cuda_status(e);
}

moe_status_t moe_grouped_mlp_fwd(const moe_config_t* cfg, const void* x_perm,
                                 const int32_t* offsets, const float* perm_prob, const void* w1,
                                 const void* b1, const void* w2, const void* b2, void* act_save,
                                 void* y_perm, void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (!x_perm || !offsets || !w1 || !w2 || !y_perm) return MOE_ERR_INVALID_ARG;
  if (cfg->has_bias && (!b1 || !b2)) return MOE_ERR_INVALID_ARG;
  if (!al16(x_perm) || !al16(w1) || !al16(w2) || !al16(y_perm) || !al16(act_save))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return st;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  const Workspace w = workspace_layout(*cfg);
  const int P = cfg->T * cfg->K;
  return cuda_status(run_grouped_mlp(*cfg, P, x_perm, offsets, perm_prob, w1,
                                     cfg->has_bias ? b1 : nullptr, w2,
                                     cfg->has_bias ? b2 : nullptr, act_save,
                                     at<void>(ws, w.a), y_perm, d,
                                     static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_expert_fc1(const moe_config_t* cfg, const void* x_perm, const int32_t* offsets,
                            const float* perm_prob, const void* w1, const void* b1,
                            void* act_save, void* a, moe_stream_t stream) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (!x_perm || !offsets || !w1 || !a) return MOE_ERR_INVALID_ARG;
  if (cfg->has_bias && !b1) return MOE_ERR_INVALID_ARG;
  if (!al16(x_perm) || !al16(w1) || !al16(a) || !al16(act_save)) return MOE_ERR_INVALID_ARG;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  return cuda_status(run_expert_gemm(*cfg, 1, cfg->T * cfg->K, x_perm, offsets, perm_prob, w1,
                                     cfg->has_bias ? b1 : nullptr, act_save, a, d,
                                     static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_expert_fc1_gather(const moe_config_t* cfg, const void* x,
                                   const int32_t* src_token, const int32_t* offsets,
                                   const float* perm_prob, const void* w1, const void* b1,
                                   void* act_save, void* a, moe_stream_t stream) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (!use_tensor_cores(*cfg)) return MOE_ERR_UNSUPPORTED;
  if (!x || !src_token || !offsets || !w1 || !a) return MOE_ERR_INVALID_ARG;
  if (cfg->has_bias && !b1) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(w1) || !al16(a) || !al16(act_save)) return MOE_ERR_INVALID_ARG;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  return cuda_status(run_expert_gemm(*cfg, 1, cfg->T * cfg->K, x, offsets, perm_prob, w1,
                                     cfg->has_bias ? b1 : nullptr, act_save, a, d,
                                     static_cast<cudaStream_t>(stream), src_token));
}

moe_status_t moe_expert_fc2(const moe_config_t* cfg, const void* a, const int32_t* offsets,
                            const float* perm_prob, const void* w2, const void* b2,
                            void* y_perm, moe_stream_t stream) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (!a || !offsets || !w2 || !y_perm) return MOE_ERR_INVALID_ARG;
  if (cfg->has_bias && !b2) return MOE_ERR_INVALID_ARG;
  if (!al16(a) || !al16(w2) || !al16(y_perm)) return MOE_ERR_INVALID_ARG;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  return cuda_status(run_expert_gemm(*cfg, 2, cfg->T * cfg->K, a, offsets, perm_prob, w2,
                                     cfg->has_bias ? b2 : nullptr, nullptr, y_perm, d,
                                     static_cast<cudaStream_t>(stream)));
}

size_t moe_mxfp8_scale_bytes(int64_t rows, int32_t K, int32_t groups) {
  if (rows < 0 || K <= 0 || K % 128 || groups < 1) return 0;
  return mxfp8_scale_bytes(rows, K, groups);
}

moe_status_t moe_mxfp8_quantize(int64_t rows, int32_t K, int32_t groups, const int32_t* offsets,
                                const void* x, uint8_t* q, uint8_t* sf, moe_stream_t stream) {
  if (rows < 0 || rows > INT32_MAX || K <= 0 || groups < 1 || groups > 256)
    return MOE_ERR_INVALID_ARG;
  if (K % 128) return MOE_ERR_UNSUPPORTED;
  if (!offsets && rows % groups) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x || !q || !sf || !al16(x) || !al16(q) || !al16(sf)) return MOE_ERR_INVALID_ARG;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  return cuda_status(launch_mxfp8_quantize((int)rows, K, groups, offsets, x, q, sf, d->sms,
                                           static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_permute_mxfp8(const moe_config_t* cfg, const void* x, const int32_t* topk_idx,
                               const float* topk_prob, uint8_t* x_q, uint8_t* x_sf,
                               int32_t* counts, int32_t* offsets, int32_t* dst_row,
                               int32_t* src_token, float* perm_prob, void* ws, size_t ws_bytes,
                               moe_stream_t stream) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (cfg->dtype != MOE_BF16 || cfg->h % 128) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!x || !topk_idx || !dst_row || !src_token || !x_q || !x_sf))
    return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(x_q) || !al16(x_sf)) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return st;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Workspace w = workspace_layout(*cfg);
  cudaError_t e = launch_permute_maps(*cfg, topk_idx, topk_prob, at<int32_t>(ws, w.hist),
                                      at<int32_t>(ws, w.chunk_base), counts, offsets, dst_row,
                                      src_token, perm_prob, d->status, s,
                                      (cfg->flags & MOE_FLAG_HIST_FROM_ROUTER) != 0);
  if (e == cudaSuccess)
    e = launch_scatter_quantize(*cfg, x, topk_idx, dst_row, offsets, x_q, x_sf, d->sms,
                                d->status, s);
  return cuda_status(e);
}

namespace {
moe_status_t check_mxfp8(const moe_config_t* cfg) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (cfg->dtype != MOE_BF16 || cfg->act != MOE_ACT_SWIGLU || cfg->has_bias || cfg->h % 128 ||
      cfg->F % 128)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}
}  // namespace

moe_status_t moe_expert_fc1_mxfp8(const moe_config_t* cfg, const uint8_t* x_q,
                                  const uint8_t* x_sf, const int32_t* offsets,
                                  const float* perm_prob, const uint8_t* w1_q,
                                  const uint8_t* w1_sf, void* a, uint8_t* a_q, uint8_t* a_sf,
                                  moe_stream_t stream) {
  moe_status_t st = check_mxfp8(cfg);
  if (st != MOE_OK) return st;
  if (!x_q || !x_sf || !offsets || !w1_q || !w1_sf) return MOE_ERR_INVALID_ARG;
  if (!a && !a_q) return MOE_ERR_INVALID_ARG;
  if (!a_q != !a_sf) return MOE_ERR_INVALID_ARG;
  if (!al16(x_q) || !al16(x_sf) || !al16(w1_q) || !al16(w1_sf) || !al16(a) || !al16(a_q) ||
      !al16(a_sf))
    return MOE_ERR_INVALID_ARG;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  const moe_config_t& c = *cfg;
  return cuda_status(launch_grouped_gemm_mxfp8(true, c.T * c.K, x_q, x_sf, c.h, w1_q, w1_sf,
                                               2 * c.F, c.E, c.F, offsets, perm_prob, a, a_q, a_sf,
                                               d->sms, d->status,
                                               static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_expert_fc2_mxfp8(const moe_config_t* cfg, const uint8_t* a_q,
                                  const uint8_t* a_sf, const int32_t* offsets,
                                  const uint8_t* w2_q, const uint8_t* w2_sf, void* y_perm,
                                  moe_stream_t stream) {
  moe_status_t st = check_mxfp8(cfg);
  if (st != MOE_OK) return st;
  if (!a_q || !a_sf || !offsets || !w2_q || !w2_sf || !y_perm) return MOE_ERR_INVALID_ARG;
  if (!al16(a_q) || !al16(a_sf) || !al16(w2_q) || !al16(w2_sf) || !al16(y_perm))
    return MOE_ERR_INVALID_ARG;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  const moe_config_t& c = *cfg;
  return cuda_status(launch_grouped_gemm_mxfp8(false, c.T * c.K, a_q, a_sf, c.F, w2_q, w2_sf, c.h,
                                               c.E, c.h, offsets, nullptr, y_perm, nullptr,
                                               nullptr, d->sms, d->status,
                                               static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_unpermute_combine(const moe_config_t* cfg, const void* y_perm,
                                   const int32_t* dst_row, const float* topk_prob,
                                   const void* shared_y, void* y, moe_stream_t stream) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T > 0 && (!y_perm || !dst_row || !y)) return MOE_ERR_INVALID_ARG;
  if (!al16(y_perm) || !al16(shared_y) || !al16(y)) return MOE_ERR_INVALID_ARG;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  return cuda_status(launch_combine(*cfg, y_perm, dst_row, topk_prob, shared_y, y, d->sms,
                                    d->status, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_layer_fwd(const moe_config_t* cfg, const void* x, const float* w_r,
                           const float* gate_bias, const float* sel_bias, const void* w1,
                           const void* b1, const void* w2, const void* b2,
                           const void* w1_shared, const void* w2_shared, void* y,
                           int32_t* topk_idx_out, float* topk_prob_out, void* ws,
                           size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  const moe_config_t& c = *cfg;
  if (c.T > 0 && (!x || !w_r || !w1 || !w2 || !y)) return MOE_ERR_INVALID_ARG;
  if (c.has_bias && (!b1 || !b2)) return MOE_ERR_INVALID_ARG;
  if (c.n_shared && (!w1_shared || !w2_shared)) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(w_r) || !al16(w1) || !al16(w2) || !al16(y) || !al16(w1_shared) ||
      !al16(w2_shared))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return st;
  if (c.flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  if (c.T == 0) return MOE_OK;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Workspace w = workspace_layout(c);
  const bool save = (c.flags & MOE_FLAG_SAVE_FOR_BWD) != 0;
  int32_t* idx = at<int32_t>(ws, w.topk_idx);
  float* prob = at<float>(ws, w.topk_prob);
  int32_t* offsets = at<int32_t>(ws, w.offsets);
  int32_t* dst_row = at<int32_t>(ws, w.dst_row);
  float* perm_prob = at<float>(ws, w.perm_prob);
  // Route
  NvtxStage stage("moe_layer_fwd/route");
  cudaError_t e = mark_stage(MOE_PASS_FWD, 0, s);
  if (e == cudaSuccess)
    e = launch_router(c, x, w_r, gate_bias, sel_bias, at<float>(ws, w.logits), idx,
                      prob, nullptr, router_scratch(c, ws), d->sms, d->status, s,
                      at<int32_t>(ws, w.hist));  // the dispatch's chunk histograms too
  if (e == cudaSuccess && (c.aux_loss_coeff != 0.f || c.z_loss_coeff != 0.f))
    e = launch_aux_loss(c, at<float>(ws, w.logits), idx, 0.f, 0.f, at<float>(ws, w.aux_losses),
                        nullptr, at<double>(ws, w.aux_part_p), at<double>(ws, w.aux_part_z),
                        at<int32_t>(ws, w.aux_part_cnt), at<float>(ws, w.aux_f), d->status, s);
  // Dispatch: the maps, then the rows scattered once into x_perm.  (FC1 could
  // gather its rows from x instead -- moe_expert_fc1_gather -- but it re-reads
  // each row block once per N tile, and a gathered re-read costs the TMA
  // engine far more than a tiled one: the one-pass scatter is faster.)
  stage.next("moe_layer_fwd/dispatch");
  if (e == cudaSuccess) e = mark_stage(MOE_PASS_FWD, 1, s);
  if (e == cudaSuccess)
    e = launch_permute_maps(c, idx, prob, at<int32_t>(ws, w.hist), at<int32_t>(ws, w.chunk_base),
                            at<int32_t>(ws, w.counts), offsets, dst_row,
                            at<int32_t>(ws, w.src_token), perm_prob, d->status, s,
                            /*hist_ready=*/true);
  if (e == cudaSuccess)
    e = launch_scatter_rows(c, x, dst_row, at<void>(ws, w.x_perm), d->sms, d->status, s, true);
  // Expert computation
  stage.next("moe_layer_fwd/experts");
  if (e == cudaSuccess) e = mark_stage(MOE_PASS_FWD, 2, s);
  if (e == cudaSuccess)
    e = run_expert_gemm(c, 1, c.T * c.K, at<void>(ws, w.x_perm), offsets, perm_prob, w1, b1,
                        save ? at<void>(ws, w.act_save) : nullptr, at<void>(ws, w.a), d, s);
  if (e == cudaSuccess) e = mark_stage(MOE_PASS_FWD, 3, s);
  if (e == cudaSuccess)
    e = run_expert_gemm(c, 2, c.T * c.K, at<void>(ws, w.a), offsets, perm_prob, w2, b2, nullptr,
                        at<void>(ws, w.y_perm), d, s);
  if (e == cudaSuccess) e = mark_stage(MOE_PASS_FWD, 4, s);
  const void* shared_y = nullptr;
  if (e == cudaSuccess && c.n_shared) {
    moe_config_t cs = c;  // one always-on expert over all T tokens, weight 1
    cs.E = 1;
    cs.K = 1;
    cs.has_bias = 0;
    int32_t* soff = at<int32_t>(ws, w.shared_off);
    fill_shared_offsets<<<1, 1, 0, s>>>(soff, c.T);
    e = cudaGetLastError();
    if (e == cudaSuccess)
      e = run_grouped_mlp(cs, c.T, x, soff, nullptr, w1_shared, nullptr, w2_shared, nullptr,
                          save ? at<void>(ws, w.shared_h) : nullptr, at<void>(ws, w.shared_a),
                          at<void>(ws, w.shared_y), d, s);
    shared_y = at<void>(ws, w.shared_y);
  }
  // Combine (probabilities were applied inside the expert GEMMs)
  stage.next("moe_layer_fwd/combine");
  if (e == cudaSuccess) e = mark_stage(MOE_PASS_FWD, 5, s);
  if (e == cudaSuccess)
    e = launch_combine(c, at<void>(ws, w.y_perm), dst_row, nullptr, shared_y, y, d->sms,
                       d->status, s);
  if (e == cudaSuccess) e = mark_stage(MOE_PASS_FWD, 6, s);
  if (e == cudaSuccess && topk_idx_out)
    e = cudaMemcpyAsync(topk_idx_out, idx, sizeof(int32_t) * c.T * c.K, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && topk_prob_out)
    e = cudaMemcpyAsync(topk_prob_out, prob, sizeof(float) * c.T * c.K, cudaMemcpyDeviceToDevice, s);
  return cuda_status(e);
}

moe_status_t moe_grouped_mlp_bwd(const moe_config_t* cfg, const void* dy_perm, const void* x_perm,
                                 const void* act_save, const void* a, const int32_t* offsets,
                                 const float* perm_prob, const void* w1, const void* w2,
                                 void* dx_perm, void* dw1, void* dw2, float* dprob_perm, void* ws,
                                 size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if ((st = check_bwd_support(*cfg)) != MOE_OK) return st;
  if (!dy_perm || !x_perm || !act_save || !a || !offsets || !w1 || !w2 || !dx_perm || !dw1 || !dw2)
    return MOE_ERR_INVALID_ARG;
  if (!al16(dy_perm) || !al16(x_perm) || !al16(act_save) || !al16(a) || !al16(w1) || !al16(w2) ||
      !al16(dx_perm) || !al16(dw1) || !al16(dw2))
    return MOE_ERR_INVALID_ARG;
  moe_config_t cs = *cfg;
  cs.flags |= MOE_FLAG_SAVE_FOR_BWD;
  if ((st = check_ws(&cs, ws, ws_bytes)) != MOE_OK) return st;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Workspace w = workspace_layout(cs);
  const int P = cfg->T * cfg->K;
  float* part = at<float>(ws, w.dprob_part);
  cudaError_t e = run_mlp_bwd(*cfg, P, cfg->E, dy_perm, x_perm, act_save, a, offsets, perm_prob,
                              w1, w2, at<void>(ws, w.dh), part, dx_perm, dw1, dw2, d, s);
  if (e == cudaSuccess && dprob_perm)
    e = launch_dprob_reduce(part, P, (cfg->F + 255) / 256, dprob_perm, s);
  return cuda_status(e);
}

moe_status_t moe_router_bwd(const moe_config_t* cfg, const void* x, const float* logits,
                            const int32_t* topk_idx, const float* topk_prob,
                            const int32_t* offsets, const int32_t* dst_row,
                            const int32_t* src_token, const float* dprob_perm, const float* w_r,
                            float* dl_topk, float* dw_r, float* db_r, float* dx_router, void* ws,
                            size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  // with an expert capacity, dropped slots get a router gradient but have no
  // permuted row for the segmented dW_r sum: moe_layer_bwd handles them
  if (cfg->capacity > 0) return MOE_ERR_UNSUPPORTED;
  if ((st = check_bwd_support(*cfg)) != MOE_OK) return st;
  if (cfg->T > 0 && (!x || !logits || !topk_idx || !topk_prob || !offsets || !dst_row ||
                     !src_token || !dprob_perm || !dl_topk || !dw_r))
    return MOE_ERR_INVALID_ARG;
  if (dx_router && !w_r) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(dw_r) || !al16(w_r) || !al16(dx_router)) return MOE_ERR_INVALID_ARG;
  moe_config_t cs = *cfg;
  cs.flags |= MOE_FLAG_SAVE_FOR_BWD;
  if ((st = check_ws(&cs, ws, ws_bytes)) != MOE_OK) return st;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Workspace w = workspace_layout(cs);
  float* dl_perm = at<float>(ws, w.dl_perm);
  cudaError_t e = launch_router_bwd(*cfg, logits, topk_idx, topk_prob, dst_row, dprob_perm,
                                    dl_topk, dl_perm, d->status, s);
  if (e == cudaSuccess)
    e = launch_router_wgrad(*cfg, x, src_token, offsets, dl_perm, dw_r, db_r, s);
  if (e == cudaSuccess && dx_router)
    e = launch_bwd_combine(*cfg, nullptr, nullptr, nullptr, dl_topk, topk_idx, w_r, nullptr,
                           nullptr, dx_router, d->sms, d->status, s);
  return cuda_status(e);
}

moe_status_t moe_router_aux_loss(const moe_config_t* cfg, const float* logits,
                                 const int32_t* topk_idx, float aux_coeff, float z_coeff,
                                 float* losses, float* dlogits, void* ws, size_t ws_bytes,
                                 moe_stream_t stream) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (!losses || (cfg->T > 0 && (!logits || !topk_idx))) return MOE_ERR_INVALID_ARG;
  if (!(aux_coeff == aux_coeff) || !(z_coeff == z_coeff)) return MOE_ERR_INVALID_ARG;  // NaN
  if ((st = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return st;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  const Workspace w = workspace_layout(*cfg);
  return cuda_status(launch_aux_loss(*cfg, logits, topk_idx, aux_coeff, z_coeff, losses, dlogits,
                                     at<double>(ws, w.aux_part_p), at<double>(ws, w.aux_part_z),
                                     at<int32_t>(ws, w.aux_part_cnt), at<float>(ws, w.aux_f),
                                     d->status, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_layer_losses(const moe_config_t* cfg, float* losses, void* ws, size_t ws_bytes,
                              moe_stream_t stream) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  if (!losses || (cfg->aux_loss_coeff == 0.f && cfg->z_loss_coeff == 0.f))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return st;
  if (cfg->flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  if (cfg->T == 0)
    return cuda_status(cudaMemsetAsync(losses, 0, 2 * sizeof(float),
                                       static_cast<cudaStream_t>(stream)));
  return cuda_status(cudaMemcpyAsync(losses, at<float>(ws, workspace_layout(*cfg).aux_losses),
                                     2 * sizeof(float), cudaMemcpyDeviceToDevice,
                                     static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_layer_bwd(const moe_config_t* cfg, const void* x, const float* w_r,
                           const void* w1, const void* w2, const void* w1_shared,
                           const void* w2_shared, const void* dy, void* dx, float* dw_r,
                           float* db_r, void* dw1, void* dw2, void* dw1_shared, void* dw2_shared,
                           void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = check_config(cfg);
  if (st != MOE_OK) return st;
  const moe_config_t& c = *cfg;
  if ((st = check_bwd_support(c)) != MOE_OK) return st;
  if (!(c.flags & MOE_FLAG_SAVE_FOR_BWD)) return MOE_ERR_INVALID_ARG;
  if (!x || !w_r || !w1 || !w2 || !dy || !dx || !dw_r || !dw1 || !dw2) return MOE_ERR_INVALID_ARG;
  if (c.n_shared && (!w1_shared || !w2_shared || !dw1_shared || !dw2_shared))
    return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(w_r) || !al16(w1) || !al16(w2) || !al16(dy) || !al16(dx) ||
      !al16(dw_r) || !al16(dw1) || !al16(dw2) || !al16(w1_shared) || !al16(w2_shared) ||
      !al16(dw1_shared) || !al16(dw2_shared))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, ws, ws_bytes)) != MOE_OK) return st;
  if (c.flags & MOE_FLAG_VALIDATE_ONLY) return MOE_OK;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Workspace w = workspace_layout(c);
  const int P = c.T * c.K;
  if (c.T == 0) {
    cudaError_t e = cudaMemsetAsync(dw_r, 0, (size_t)c.E * c.h * 4, s);
    if (e == cudaSuccess && db_r) e = cudaMemsetAsync(db_r, 0, (size_t)c.E * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dw1, 0, (size_t)c.E * 2 * c.F * c.h * 2, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dw2, 0, (size_t)c.E * c.h * c.F * 2, s);
    if (e == cudaSuccess && c.n_shared) e = cudaMemsetAsync(dw1_shared, 0, (size_t)2 * c.F * c.h * 2, s);
    if (e == cudaSuccess && c.n_shared) e = cudaMemsetAsync(dw2_shared, 0, (size_t)c.h * c.F * 2, s);
    return cuda_status(e);
  }
  const int32_t* offsets = at<int32_t>(ws, w.offsets);
  const int32_t* dst_row = at<int32_t>(ws, w.dst_row);
  const int32_t* idx = at<int32_t>(ws, w.topk_idx);
  float* dl_topk = at<float>(ws, w.dl_topk);
  // dy in expert order, then the routed experts' backward
  NvtxStage stage("moe_layer_bwd/experts");
  cudaError_t e = mark_stage(MOE_PASS_BWD, 0, s);
  if (e == cudaSuccess)
    e = launch_scatter_rows(c, dy, dst_row, at<void>(ws, w.dy_perm), d->sms, d->status, s);
  if (e == cudaSuccess) e = mark_stage(MOE_PASS_BWD, 1, s);
  if (e == cudaSuccess)
    e = run_mlp_bwd(c, P, c.E, at<void>(ws, w.dy_perm), at<void>(ws, w.x_perm),
                    at<void>(ws, w.act_save), at<void>(ws, w.a), offsets,
                    at<float>(ws, w.perm_prob), w1, w2, at<void>(ws, w.dh),
                    at<float>(ws, w.dprob_part), at<void>(ws, w.dx_perm), dw1, dw2, d, s, 2);
  // the shared expert: one group of all T tokens, weight 1
  if (e == cudaSuccess && c.n_shared)
    e = run_mlp_bwd(c, c.T, 1, dy, x, at<void>(ws, w.shared_h), at<void>(ws, w.shared_a),
                    at<int32_t>(ws, w.shared_off), nullptr, w1_shared, w2_shared,
                    at<void>(ws, w.shared_dh), nullptr, at<void>(ws, w.shared_dx), dw1_shared,
                    dw2_shared, d, s);
  // Route backward: dprob -> dl -> dW_r, db_r
  stage.next("moe_layer_bwd/router");
  if (e == cudaSuccess) e = mark_stage(MOE_PASS_BWD, 6, s);
  if (e == cudaSuccess)
    e = launch_dprob_reduce(at<float>(ws, w.dprob_part), P, (c.F + 255) / 256,
                            at<float>(ws, w.dprob_perm), s);
  if (e == cudaSuccess)
    e = launch_router_bwd(c, at<float>(ws, w.logits), idx, at<float>(ws, w.topk_prob), dst_row,
                          at<float>(ws, w.dprob_perm), dl_topk, at<float>(ws, w.dl_perm),
                          d->status, s);
  // Router weight gradient.  Dropless without load-balancing losses: a
  // segmented sum over each expert's permuted rows.  Otherwise the logit
  // gradient is dense or reaches dropped slots that have no permuted row, so
  // it is gathered into a dense [T, E] matrix and pushed through the gating
  // layer by dense products: the losses' part first goes to dx (dx_add = dl
  // W_r; the routed part reaches dx through the combine below), then the
  // routed slots are added and dW_r = dl^T x, db_r = sum_t dl.
  const bool lb = c.aux_loss_coeff != 0.f || c.z_loss_coeff != 0.f;
  const float* dx_add = nullptr;
  if (!lb && c.capacity == 0) {
    if (e == cudaSuccess)
      e = launch_router_wgrad(c, x, at<int32_t>(ws, w.src_token), offsets,
                              at<float>(ws, w.dl_perm), dw_r, db_r, s);
  } else {
    float* dl_dense = at<float>(ws, w.aux_dl);
    if (e == cudaSuccess) e = cudaMemsetAsync(dl_dense, 0, sizeof(float) * c.T * c.E, s);
    if (lb) {
      if (e == cudaSuccess)
        e = launch_aux_loss(c, at<float>(ws, w.logits), idx, c.aux_loss_coeff, c.z_loss_coeff,
                            at<float>(ws, w.aux_losses), dl_dense, at<double>(ws, w.aux_part_p),
                            at<double>(ws, w.aux_part_z), at<int32_t>(ws, w.aux_part_cnt),
                            at<float>(ws, w.aux_f), d->status, s);
      if (e == cudaSuccess) e = launch_dense_router_dx(c, dl_dense, w_r, at<float>(ws, w.aux_dx), s);
      dx_add = at<float>(ws, w.aux_dx);
    }
    if (e == cudaSuccess) e = launch_scatter_topk_grad(c, dl_topk, idx, dl_dense, s);
    if (e == cudaSuccess) e = launch_dense_router_wgrad(c, dl_dense, x, dw_r, db_r, s);
  }
  // dx = routed + shared + router contributions
  stage.next("moe_layer_bwd/combine");
  if (e == cudaSuccess) e = mark_stage(MOE_PASS_BWD, 7, s);
  if (e == cudaSuccess)
    e = launch_bwd_combine(c, at<void>(ws, w.dx_perm), dst_row,
                           c.n_shared ? at<void>(ws, w.shared_dx) : nullptr, dl_topk, idx, w_r,
                           dx_add, dx, nullptr, d->sms, d->status, s);
  if (e == cudaSuccess) e = mark_stage(MOE_PASS_BWD, 8, s);
  return cuda_status(e);
}

moe_status_t moe_get_error(moe_stream_t stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  const DeviceInfo* d = device_info(false);
  if (!d) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return static_cast<moe_status_t>(v);
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_BOUNDS: return "device-side index out of range";
  }
  return "unknown status";
}

const char* moe_version(void) { return "0.1.0"; }

moe_status_t moe_set_stage_events(int32_t pass, void* const* events, int32_t n) {
  if (pass != MOE_PASS_FWD && pass != MOE_PASS_BWD) return MOE_ERR_INVALID_ARG;
  if (n < 0 || n > kMaxStageEvents || (n > 0 && !events)) return MOE_ERR_INVALID_ARG;
  StageEvents& se = g_stage_events[pass];
  for (int i = 0; i < kMaxStageEvents; ++i)
    se.ev[i] = i < n ? static_cast<cudaEvent_t>(events[i]) : nullptr;
  se.n = n;
  return MOE_OK;
}

int32_t moe_test_inject_cuda_failure(int32_t n) {
  if (n < 0) return -1;
  return g_inject_failures.exchange(n);
}

moe_status_t moe_test_bounded_wait(int64_t max_polls, moe_stream_t stream) {
  if (max_polls < 1) return MOE_ERR_INVALID_ARG;
  const DeviceInfo* d = device_info();
  if (!d) return MOE_ERR_CUDA;
  return cuda_status(
      launch_bounded_wait_probe(max_polls, d->status, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
