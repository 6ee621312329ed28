// C ABI of libmoe (declared in include/moe.h): argument checks, the
// workspace layout, and the order of launches. All compute is in the
// kernels of router.cu, dispatch.cu, ffn_tc.cu, ffn_simt.cu and combine.cu.
#include "moe_common.cuh"

#include <math.h>

#include <algorithm>

#include <mutex>

namespace moe {

namespace {
constexpr int64_t kMaxT = int64_t(1) << 24;

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int dtype_size(const moe_config* c) { return c->dtype == MOE_BF16 ? 2 : 4; }
}  // namespace

bool config_valid(const moe_config* c, moe_status* why) {
  auto bad = [&](moe_status s) {
    if (why) *why = s;
    return false;
  };
  if (!c) return bad(MOE_ERR_INVALID);
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return bad(MOE_ERR_INVALID);
  if (c->activation != MOE_SWIGLU && c->activation != MOE_GELU) return bad(MOE_ERR_INVALID);
  if ((c->has_bias != 0 && c->has_bias != 1) || (c->add_residual != 0 && c->add_residual != 1))
    return bad(MOE_ERR_INVALID);
  if (c->gate_mode != MOE_GATE_RENORM && c->gate_mode != MOE_GATE_SOFTMAX)
    return bad(MOE_ERR_INVALID);
  if (c->n_shared < 0) return bad(MOE_ERR_INVALID);
  if (c->save_for_backward != 0 && c->save_for_backward != 1) return bad(MOE_ERR_INVALID);
  if (c->n_shared > 8) return bad(MOE_ERR_UNSUPPORTED);
  if (c->T < 0 || c->d_model <= 0 || c->d_ff <= 0 || c->n_experts <= 0 || c->top_k <= 0)
    return bad(MOE_ERR_INVALID);
  if (c->top_k > c->n_experts) return bad(MOE_ERR_INVALID);
  if (isnan(c->capacity_factor) || !isfinite(c->alpha)) return bad(MOE_ERR_INVALID);
  if (c->T > kMaxT || c->n_experts > 256 || c->top_k > 8) return bad(MOE_ERR_UNSUPPORTED);
  if (c->d_model % (c->dtype == MOE_BF16 ? 8 : 4) != 0 || c->d_ff % 4 != 0)
    return bad(MOE_ERR_UNSUPPORTED);
  if (c->has_bias && c->activation != MOE_GELU) return bad(MOE_ERR_UNSUPPORTED);
  return true;
}

// floor(K * CF * T / N) on the exact value of the float CF. K*CF*T is exact
// in double (a 24-bit significand times an integer below 2^27); the quotient
// is then corrected against exact integer products.
int32_t capacity_of(const moe_config* c) {
  const double cf = static_cast<double>(c->capacity_factor);
  if (!(cf > 0.0) || isinf(cf)) return INT32_MAX;
  const double q = static_cast<double>(c->top_k) * cf * static_cast<double>(c->T);
  const double n = static_cast<double>(c->n_experts);
  double f = floor(q / n);
  while ((f + 1.0) * n <= q) f += 1.0;
  while (f > 0.0 && f * n > q) f -= 1.0;
  return f >= static_cast<double>(INT32_MAX) ? INT32_MAX : static_cast<int32_t>(f);
}

int64_t a_max_of(const moe_config* c) {
  const int64_t tk = static_cast<int64_t>(c->T) * c->top_k;
  const int64_t nc = static_cast<int64_t>(c->n_experts) * capacity_of(c);
  return tk < nc ? tk : nc;
}

int64_t rows_max_of(const moe_config* c) {
  return a_max_of(c) + static_cast<int64_t>(c->n_shared) * c->T;
}

WsLayout ws_layout(const moe_config* c) {
  WsLayout L{};
  size_t total = 0;
  auto take = [&](size_t bytes) {
    const size_t off = total;
    total += align256(bytes);
    return off;
  };
  const size_t T = static_cast<size_t>(c->T), K = c->top_k, N = c->n_experts;
  const size_t d = c->d_model, F = c->d_ff, es = dtype_size(c);
  L.a_max = a_max_of(c);
  L.nblk_r = router_small(*c) ? static_cast<int>(T)
                              : static_cast<int>((T + kTopkTokensPerBlock - 1) / kTopkTokensPerBlock);
  L.nblk_d = static_cast<int>((T + kDispatchTokensPerBlock - 1) / kDispatchTokensPerBlock);
  const size_t nr = L.nblk_r > 0 ? L.nblk_r : 1, nd = L.nblk_d > 0 ? L.nblk_d : 1;
  const size_t A = static_cast<size_t>(rows_max_of(c));  // routed + shared rows
  const size_t S = static_cast<size_t>(c->n_shared);
  L.idx = take(T * K * 4);
  L.gate = take(T * K * 4);
  L.psum = take(nr * (N + 2) * 4);  // rows N, N+1: z-loss and entropy partials
  L.pcnt = take(nr * N * 4);
  const RouterTcPlan rp = router_tc_plan(*c);
  L.w3 = take(rp.use ? static_cast<size_t>(3) * rp.NP * d * 2 : 0);
  L.part = take(rp.use && !rp.fused ? static_cast<size_t>(rp.S) * T * rp.NP * 4 : 0);
  L.ghist = take(K * nd * N * 4);
  L.gbase = take(K * nd * N * 4);
  L.offsets = take((N + S + 1) * 4);
  L.slot_of = take(T * (K + S) * 4);
  L.token_of_slot = take((A > 0 ? A : 1) * 4);
  L.x_perm = take(A * d * es);
  L.h = take(A * F * es);
  L.o = take(A * d * 4);
  const int ks = ffn_tc_supported(*c) ? gate_up_ksplit(*c, static_cast<int64_t>(A)) : 1;
  L.gu_part = take(ks > 1 ? static_cast<size_t>(ks) * A * 2 * F * 4 : 0);
  L.sched = take(2 * 4);
  const bool bw = c->save_for_backward != 0;
  // router-gradient K splits: about 1024 tokens each, at most 32
  L.rsplits = bw ? static_cast<int>(std::min<size_t>(32, std::max<size_t>(1, T / 1024))) : 0;
  L.logits = take(bw ? T * N * 4 : 0);
  const bool ftc = bw && ffn_bwd_tc_supported(*c);
  const size_t Apad = ftc ? static_cast<size_t>(ffn_bwd_pad_rows(*c)) : A;
  L.pre = take(bw ? Apad * 2 * F * es : 0);
  L.count = take(bw ? N * 4 : 0);
  L.dout = take(bw ? Apad * d * es : 0);
  L.poff = take(bw ? (N + S + 1) * 4 : 0);
  L.dg = take(bw ? T * K * 4 : 0);
  L.dl = take(bw ? T * N * 4 : 0);
  L.rpart = take(bw ? static_cast<size_t>(L.rsplits) * N * (d + 1) * 4 : 0);
  L.bpart = take(bw ? ((T + 255) / 256 > 0 ? (T + 255) / 256 : 1) * N * 4 : 0);
  const bool rtc = bw && router_bwd_tc_supported(*c);
  const RouterBwdPlan rb = rtc ? router_bwd_tc_plan(*c) : RouterBwdPlan{0, 0};
  L.r_ar = take(rtc ? (T + 63) / 64 * 64 * 3 * rb.NP * 2 : 0);
  L.r_br = take(rtc ? static_cast<size_t>(3) * rb.NP * d * 2 : 0);
  L.r_goff = take(rtc ? static_cast<size_t>(2 * rb.G + 6) * 4 : 0);
  L.r_part = take(rtc ? static_cast<size_t>(rb.G) * 2 * rb.NP * d * 4 : 0);
  L.total = total;
  return L;
}

namespace {
// Per-thread trace registration (moe_trace_events).
constexpr int kMaxTrace = 8;
thread_local cudaEvent_t g_trace[kMaxTrace] = {};
thread_local int g_ntrace = 0;
}  // namespace

void trace_record(int i, cudaStream_t s) {
  if (i >= g_ntrace || g_trace[i] == nullptr) return;
  // inside a stream capture a plain record only orders the graph; the
  // external form records the event each time the graph is replayed
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(g_trace[i], s, cudaEventRecordExternal);
  else
    cudaEventRecord(g_trace[i], s);
}

int sm_count() {
  static int counts[64] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && counts[dev] > 0) return counts[dev];
  int n = 148;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < 64) counts[dev] = n;
  return n;
}

namespace {

moe_status check_ws(const moe_config* c, const void* ws) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
  (void)c;
  return MOE_OK;
}

uint8_t* at(void* ws, size_t off) {
  return static_cast<uint8_t*>(ws) + off;
}

RouterScratch router_scratch(void* ws, const WsLayout& L, bool keep_logits) {
  return RouterScratch{reinterpret_cast<float*>(at(ws, L.psum)),
                       reinterpret_cast<int32_t*>(at(ws, L.pcnt)),
                       reinterpret_cast<__nv_bfloat16*>(at(ws, L.w3)),
                       reinterpret_cast<float*>(at(ws, L.part)),
                       keep_logits ? reinterpret_cast<float*>(at(ws, L.logits)) : nullptr};
}

moe_status check_weights(const moe_config* c, const moe_expert_weights* w) {
  if (!w) return MOE_ERR_INVALID;
  if (c->activation == MOE_SWIGLU) {
    if (!w->w_gate || !w->w_up || !w->w_down) return MOE_ERR_INVALID;
    if (!aligned16(w->w_gate) || !aligned16(w->w_up) || !aligned16(w->w_down))
      return MOE_ERR_INVALID;
  } else {
    if (!w->w1 || !w->w2) return MOE_ERR_INVALID;
    if (c->has_bias && (!w->b1 || !w->b2)) return MOE_ERR_INVALID;
    if (!aligned16(w->w1) || !aligned16(w->w2)) return MOE_ERR_INVALID;
  }
  return MOE_OK;
}

// Per-thread trace: events recorded on the launch stream at the stage
// boundaries of moe_forward and moe_backward (see moe_trace_events).

void trace(int i, cudaStream_t s) { trace_record(i, s); }

moe_status ffn_impl(const moe_config* c, const void* x_perm, const int32_t* offsets,
                    const moe_expert_weights* w, float* o, moe_stats* stats, void* ws,
                    cudaStream_t s, bool traced, bool keep_pre, bool sched_zeroed,
                    const FusedCombine* fc = nullptr) {
  const WsLayout L = ws_layout(c);
  void* h = at(ws, L.h);
  void* pre = keep_pre ? at(ws, L.pre) : nullptr;
  int32_t* poff = reinterpret_cast<int32_t*>(at(ws, L.poff));
  if (keep_pre && ffn_tc_supported(*c)) {  // the tensor-core path keeps them in padded rows
    const moe_status r = launch_pad_offsets(offsets, c->n_experts + c->n_shared, poff, s);
    if (r != MOE_OK) return r;
  }
  const bool tc = ffn_tc_supported(*c);
  uint32_t* status = stats ? stats->status : nullptr;
  for (int part = 1; part <= 2; ++part) {
    const int64_t rows = rows_max_of(c);
    const moe_status r =
        tc ? launch_ffn_tc(*c, rows, x_perm, offsets, *w, h, o, pre, poff,
                           reinterpret_cast<float*>(at(ws, L.gu_part)),
                           reinterpret_cast<int32_t*>(at(ws, L.sched)), sched_zeroed, status,
                           s, part, fc)
           : launch_ffn_simt(*c, rows, x_perm, offsets, *w, h, o, pre, s, part);
    if (r != MOE_OK) return r;
    if (traced) trace(2 + part, s);
  }
  return MOE_OK;
}

// moe_forward writes y from the down projection's epilogue (no fp32 o, no
// combine pass) when each token has at most one expert output (K = 1 and no
// shared experts) on the tensor-core path, and the backward pass does not
// need o.
bool combine_fused(const moe_config& c) {
  return c.top_k == 1 && c.n_shared == 0 && c.save_for_backward == 0 && ffn_tc_supported(c);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_size(const moe_config* cfg) {
  if (!config_valid(cfg, nullptr)) return 0;
  return ws_layout(cfg).total;
}

int32_t moe_capacity(const moe_config* cfg) {
  if (!config_valid(cfg, nullptr)) return -1;
  return capacity_of(cfg);
}

int32_t moe_forward_launch_count(const moe_config* cfg) {
  if (!config_valid(cfg, nullptr)) return -1;
  if (cfg->T == 0) return 1;  // the dispatch scan still writes offsets and counts
  const RouterTcPlan rp = router_tc_plan(*cfg);
  // decode-sized batches or no tensor cores: one CUDA-core kernel; else the
  // weight split and the GEMM (+ top-K unless fused)
  const int router = router_small(*cfg) || !rp.use ? 1 : (rp.fused ? 2 : 3);
  const int stats = route_stats_launches(*cfg);         // per-expert reduction (+ L_aux)
  // histogram, scan, permute, gather; at most 256 tokens: the one-block
  // dispatch and the gather
  const int dispatch = cfg->T <= kDispatchTokensPerBlock ? 2 : 4;
  // gate/up (+ the SwiGLU of a split reduction), down
  const int ffn = 2 + (ffn_tc_supported(*cfg) && gate_up_ksplit(*cfg, rows_max_of(cfg)) > 1 ? 1 : 0);
  const int combine = 1;  // or, fused into the down projection, the dropped-token pass
  // keeping the pre-activations for the tensor-core backward: their padded offsets
  const int keep = cfg->save_for_backward && ffn_tc_supported(*cfg) ? 1 : 0;
  return router + stats + dispatch + ffn + combine + keep;
}

int32_t moe_backward_launch_count(const moe_config* cfg) {
  if (!config_valid(cfg, nullptr) || cfg->save_for_backward == 0) return -1;
  return backward_launch_count(*cfg);
}

int32_t moe_ffn_uses_tensor_cores(const moe_config* cfg) {
  if (!config_valid(cfg, nullptr)) return -1;
  return ffn_tc_supported(*cfg) ? 1 : 0;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_NONFINITE: return "non-finite router logit";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_INDEX: return "expert index out of range";
  }
  return "unknown status";
}

moe_status moe_trace_events(void* const* events, int32_t n) {
  if (n < 0 || n > kMaxTrace || (n > 0 && events == nullptr)) return MOE_ERR_INVALID;
  for (int i = 0; i < kMaxTrace; ++i)
    g_trace[i] = i < n ? static_cast<cudaEvent_t>(events[i]) : nullptr;
  g_ntrace = n;
  return MOE_OK;
}

moe_status moe_route(const moe_config* cfg, const void* x, const float* w_r, const float* b_r,
                     int32_t* idx, float* gate, moe_stats* stats, void* ws, moe_stream_t stream) {
  try {
    moe_status why = MOE_OK;
    if (!config_valid(cfg, &why)) return why;
    if (!x || !w_r || !idx || !gate) return MOE_ERR_INVALID;
    if (!aligned16(x) || !aligned16(w_r) || !aligned16(idx) || !aligned16(gate) ||
        (b_r && !aligned16(b_r)))
      return MOE_ERR_INVALID;
    if (moe_status s = check_ws(cfg, ws)) return s;
    const WsLayout L = ws_layout(cfg);
    return launch_router(*cfg, x, w_r, b_r, idx, gate, router_scratch(ws, L, false), stats,
                         static_cast<cudaStream_t>(stream));
  } catch (...) {
    return MOE_ERR_CUDA;
  }
}

moe_status moe_dispatch(const moe_config* cfg, const void* x, const int32_t* idx, int32_t* offsets,
                        int32_t* slot_of, int32_t* token_of_slot, void* x_perm, moe_stats* stats,
                        void* ws, moe_stream_t stream) {
  try {
    moe_status why = MOE_OK;
    if (!config_valid(cfg, &why)) return why;
    if (!x || !idx || !offsets || !slot_of || !token_of_slot || !x_perm) return MOE_ERR_INVALID;
    if (!aligned16(x) || !aligned16(idx) || !aligned16(offsets) || !aligned16(slot_of) ||
        !aligned16(token_of_slot) || !aligned16(x_perm))
      return MOE_ERR_INVALID;
    if (moe_status s = check_ws(cfg, ws)) return s;
    const WsLayout L = ws_layout(cfg);
    return launch_dispatch(*cfg, x, idx, offsets, slot_of, token_of_slot, x_perm,
                           reinterpret_cast<int32_t*>(at(ws, L.ghist)),
                           reinterpret_cast<int32_t*>(at(ws, L.gbase)), stats,
                           static_cast<cudaStream_t>(stream));
  } catch (...) {
    return MOE_ERR_CUDA;
  }
}

moe_status moe_expert_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                          const moe_expert_weights* weights, float* o, moe_stats* stats, void* ws,
                          moe_stream_t stream) {
  try {
    moe_status why = MOE_OK;
    if (!config_valid(cfg, &why)) return why;
    if (!x_perm || !offsets || !o) return MOE_ERR_INVALID;
    if (!aligned16(x_perm) || !aligned16(offsets) || !aligned16(o)) return MOE_ERR_INVALID;
    if (moe_status s = check_weights(cfg, weights)) return s;
    if (moe_status s = check_ws(cfg, ws)) return s;
    return ffn_impl(cfg, x_perm, offsets, weights, o, stats, ws,
                    static_cast<cudaStream_t>(stream), false, false, false);
  } catch (...) {
    return MOE_ERR_CUDA;
  }
}

moe_status moe_combine(const moe_config* cfg, const float* o, const int32_t* slot_of,
                       const float* gate, const void* x, void* y, moe_stream_t stream) {
  try {
    moe_status why = MOE_OK;
    if (!config_valid(cfg, &why)) return why;
    if (!o || !slot_of || !gate || !y || (cfg->add_residual && !x)) return MOE_ERR_INVALID;
    if (!aligned16(o) || !aligned16(slot_of) || !aligned16(gate) || !aligned16(y) ||
        (x && !aligned16(x)))
      return MOE_ERR_INVALID;
    return launch_combine(*cfg, o, slot_of, gate, x, y, static_cast<cudaStream_t>(stream));
  } catch (...) {
    return MOE_ERR_CUDA;
  }
}

moe_status moe_forward(const moe_config* cfg, const void* x, const float* w_r, const float* b_r,
                       const moe_expert_weights* weights, void* y, moe_stats* stats, void* ws,
                       moe_stream_t stream) {
  try {
    moe_status why = MOE_OK;
    if (!config_valid(cfg, &why)) return why;
    // no token: x and y may be NULL (an empty tensor has no storage)
    if (!w_r || (cfg->T > 0 && (!x || !y))) return MOE_ERR_INVALID;
    if (!aligned16(x) || !aligned16(w_r) || !aligned16(y) || (b_r && !aligned16(b_r)))
      return MOE_ERR_INVALID;
    if (moe_status s = check_weights(cfg, weights)) return s;
    if (moe_status s = check_ws(cfg, ws)) return s;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const WsLayout L = ws_layout(cfg);
    int32_t* idx = reinterpret_cast<int32_t*>(at(ws, L.idx));
    float* gate = reinterpret_cast<float*>(at(ws, L.gate));
    int32_t* offsets = reinterpret_cast<int32_t*>(at(ws, L.offsets));
    int32_t* slot_of = reinterpret_cast<int32_t*>(at(ws, L.slot_of));
    int32_t* tos = reinterpret_cast<int32_t*>(at(ws, L.token_of_slot));
    void* x_perm = at(ws, L.x_perm);
    float* o = reinterpret_cast<float*>(at(ws, L.o));
    const bool keep = cfg->save_for_backward != 0;
    trace(0, s);
    moe_status r =
        launch_router(*cfg, x, w_r, b_r, idx, gate, router_scratch(ws, L, keep), stats, s);
    if (r != MOE_OK) return r;
    trace(1, s);
    // the backward pass reads the counts from the workspace (the router's
    // statistics kernel still writes the caller's copy)
    moe_stats dst = stats ? *stats : moe_stats{};
    if (keep) dst.count = reinterpret_cast<int32_t*>(at(ws, L.count));
    const bool any = dst.count || dst.kept || dst.n_dropped || dst.status;
    r = launch_dispatch(*cfg, x, idx, offsets, slot_of, tos, x_perm,
                        reinterpret_cast<int32_t*>(at(ws, L.ghist)),
                        reinterpret_cast<int32_t*>(at(ws, L.gbase)), any ? &dst : nullptr, s,
                        reinterpret_cast<int32_t*>(at(ws, L.sched)));
    if (r != MOE_OK) return r;
    trace(2, s);
    if (combine_fused(*cfg)) {
      const FusedCombine fc{tos, gate, cfg->add_residual ? x : nullptr, y};
      r = ffn_impl(cfg, x_perm, offsets, weights, o, stats, ws, s, true, keep, true, &fc);
      if (r != MOE_OK) return r;
      r = launch_dropped_residual(*cfg, slot_of, x, y, s);
    } else {
      r = ffn_impl(cfg, x_perm, offsets, weights, o, stats, ws, s, true, keep, true);
      if (r != MOE_OK) return r;
      r = launch_combine(*cfg, o, slot_of, gate, x, y, s);
    }
    trace(5, s);
    return r;
  } catch (...) {
    return MOE_ERR_CUDA;
  }
}

moe_status moe_backward(const moe_config* cfg, const void* x, const float* w_r,
                        const moe_expert_weights* weights, const void* dy, float z_coef,
                        moe_grads* grads, moe_stats* stats, void* ws, moe_stream_t stream) {
  try {
    moe_status why = MOE_OK;
    if (!config_valid(cfg, &why)) return why;
    if (cfg->save_for_backward == 0) return MOE_ERR_INVALID;
    const bool none = cfg->T == 0;  // no token: x, dy and dx may be NULL
    if (!w_r || !grads || !grads->dw_r || (!none && (!x || !dy || !grads->dx)))
      return MOE_ERR_INVALID;
    if (!isfinite(z_coef) || z_coef < 0.f) return MOE_ERR_INVALID;
    if (!aligned16(x) || !aligned16(w_r) || !aligned16(dy) || !aligned16(grads->dx) ||
        !aligned16(grads->dw_r) || (grads->db_r && !aligned16(grads->db_r)))
      return MOE_ERR_INVALID;
    if (moe_status s = check_weights(cfg, weights)) return s;
    if (cfg->activation == MOE_SWIGLU) {
      if (!grads->dw_gate || !grads->dw_up || !grads->dw_down) return MOE_ERR_INVALID;
      if (!aligned16(grads->dw_gate) || !aligned16(grads->dw_up) || !aligned16(grads->dw_down))
        return MOE_ERR_INVALID;
    } else {
      if (!grads->dw1 || !grads->dw2) return MOE_ERR_INVALID;
      if (cfg->has_bias && (!grads->db1 || !grads->db2)) return MOE_ERR_INVALID;
      if (!aligned16(grads->dw1) || !aligned16(grads->dw2)) return MOE_ERR_INVALID;
    }
    if (moe_status s = check_ws(cfg, ws)) return s;
    const WsLayout L = ws_layout(cfg);
    return launch_backward(*cfg, L, ws, x, w_r, *weights, dy, z_coef, *grads,
                           stats ? stats->status : nullptr, static_cast<cudaStream_t>(stream));
  } catch (...) {
    return MOE_ERR_CUDA;
  }
}

}  // extern "C"
