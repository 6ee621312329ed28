// Internal declarations shared by the translation units of libmoe.
// Not part of the public ABI (that is include/moe.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ---- device helpers --------------------------------------------------------
__device__ __forceinline__ void set_status(uint32_t* status, moe_status code) {
  if (status) atomicOr(status, 1u << static_cast<uint32_t>(code));
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Load 4 consecutive elements (16-byte aligned for fp32, 8-byte for bf16).
__device__ __forceinline__ float4 load4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&u.x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&u.y);
  float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}
__device__ __forceinline__ void store4(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// ---- workspace layout ------------------------------------------------------
// Every region is 256-byte aligned. The same layout serves every entry point;
// moe_workspace_size() returns its total.
constexpr int kRouterTokensPerBlock = 32;   // tokens per CUDA-core router block
constexpr int kTopkTokensPerBlock = 8;      // tokens per top-K block (one per warp)
constexpr int kDispatchTokensPerBlock = 256; // tokens per dispatch block

struct WsLayout {
  size_t idx, gate;           // [T][K] int32 / fp32 (moe_forward only)
  size_t psum, pcnt;          // router partials [N+2][nblk_r], [N][nblk_r] (expert-major);
                              // nblk_r = ceil(T / kTopkTokensPerBlock), or T for the
                              // small-batch router, covers every router
  size_t w3, part;            // tensor-core router: W_r split [3][NP][d] bf16,
                              // partial logits [S][T][NP] fp32
  size_t ghist, gbase;        // dispatch histograms [K][nblk_d][N]
  size_t offsets;             // [N+1] (moe_forward only)
  size_t slot_of;             // [T][K] (moe_forward only)
  size_t token_of_slot;       // [A_max] (moe_forward only)
  size_t x_perm;              // [A_max][d] dtype (moe_forward only)
  size_t h;                   // [A_max][F] dtype
  size_t o;                   // [A_max][d] fp32 (moe_forward only); the backward
                              // pass reuses it for the expert input gradients
  size_t gu_part;             // [ksplit][R_max][2F] fp32 split gate/up partials (decode)
  size_t sched;               // [2] int32 tile counters of the CTA-pair GEMMs (gate/up, down)
  // save_for_backward only (size 0 otherwise):
  size_t logits;              // [T][N] fp32 router logits
  size_t pre;                 // [R_max][2F] dtype: SwiGLU gate | up pre-activations
                              // (GELU: z in the first F columns); the backward pass
                              // overwrites them in place with their gradients. The
                              // tensor-core path: [R_pad][2F], padded rows
  size_t count;               // [N] int32 assignments per expert
  size_t dout;                // [R_pad][d] dtype: expert output gradients (tensor-core path:
                              // padded rows, each expert's rows rounded up to 64)
  size_t poff;                // [N+S+1] int32 padded row offsets
  size_t dg;                  // [T][K] fp32 gate gradients
  size_t dl;                  // [T][N] fp32 logit gradients
  size_t rpart;               // [rsplits][N][d + 1] fp32 router-gradient partials
  size_t bpart;               // [ceil(T/256)][N] fp32 partial column sums of dl (db_r)
  // tensor-core router gradients (bf16 layers with d % 256 == 0):
  size_t r_ar;                // [Tp][3 NP] bf16: dl_hi | dl_lo | dl_hi (Tp = T rounded up to 64)
  size_t r_br;                // [3 NP][d] bf16: W_hi ; W_hi ; W_mid
  size_t r_goff;              // [2G + 6] int32 token-group offsets (A rows, x rows), then dx's
  size_t r_part;              // [G][2 NP][d] fp32 partial dW_r
  size_t total;
  int64_t a_max;
  int nblk_r, nblk_d, rsplits;
};

// Host-side helpers implemented in moe_api.cu.
bool config_valid(const moe_config* c, moe_status* why);
int32_t capacity_of(const moe_config* c);
int64_t a_max_of(const moe_config* c);
int64_t rows_max_of(const moe_config* c);  // routed A_max + n_shared * T
WsLayout ws_layout(const moe_config* c);
int sm_count();
// Records the i-th event registered by moe_trace_events for this host thread
// on stream s (nothing if fewer are registered).
void trace_record(int i, cudaStream_t s);

// ---- launchers (each returns MOE_OK or MOE_ERR_CUDA) -----------------------
// Tensor-core router plan: NP = experts padded to 32/64/128/256, NPT = experts
// per tile, S = K splits of kb_per_split 64-wide steps each. fused: one split
// and one expert tile, so selection runs in the GEMM epilogue (no partial
// logits, no top-K kernel). stat_blocks: the per-block statistics partials the
// router leaves (one per 128-token tile when fused, else one per 32 tokens).
struct RouterTcPlan {
  bool use, fused;
  int NP, NPT, S, kb_per_split, stat_blocks;
};
RouterTcPlan router_tc_plan(const moe_config& c);

// Router scratch: per-block partial statistics (always), plus the weight
// split and partial logits of the tensor-core router (NULL: CUDA-core router)
// and the [T][N] logits kept for the backward pass (NULL: not kept).
struct RouterScratch {
  float* psum;
  int32_t* pcnt;
  __nv_bfloat16* w3;
  float* part;
  float* logits;
};
// Decode-sized batches take the one-launch CUDA-core router (one block per
// token; statistics partials per token, nblk = T).
bool router_small(const moe_config& c);
moe_status launch_router(const moe_config& c, const void* x, const float* w_r,
                         const float* b_r, int32_t* idx, float* gate, const RouterScratch& sc,
                         const moe_stats* st, cudaStream_t s);
// Kernels launch_router uses to reduce the statistics partials (all of them
// requested, the tensor-core router when the plan uses it): 1 or 2.
int route_stats_launches(const moe_config& c);
moe_status launch_router_tc(const moe_config& c, const RouterTcPlan& p, const void* x,
                            const float* w_r, const float* b_r, int32_t* idx, float* gate,
                            __nv_bfloat16* w3, float* part, float* psum, int32_t* pcnt,
                            uint32_t* status, float* logits, cudaStream_t s);

moe_status launch_dispatch(const moe_config& c, const void* x, const int32_t* idx,
                           int32_t* offsets, int32_t* slot_of, int32_t* token_of_slot,
                           void* x_perm, int32_t* ghist, int32_t* gbase,
                           const moe_stats* st, cudaStream_t s,
                           int32_t* sched_zero = nullptr);  // [2] zeroed by the scan, or NULL

moe_status launch_combine(const moe_config& c, const float* o, const int32_t* slot_of,
                          const float* gate, const void* x, void* y, cudaStream_t s);
// With the combine fused into the down projection (K = 1, S = 0): y[t] = x[t]
// (residual) or 0 for every token whose one assignment was dropped.
moe_status launch_dropped_residual(const moe_config& c, const int32_t* slot_of, const void* x,
                                   void* y, cudaStream_t s);

// Expert FFN on CUDA cores (any dtype/shape) over the N + n_shared experts;
// rows = rows of x_perm / h / o. part: 1 = gate/up (or the first Linear +
// GELU) into h, 2 = down projection into o, 3 = both. pre (NULL or
// [rows][2F] dtype): the pre-activations kept for the backward pass.
moe_status launch_ffn_simt(const moe_config& c, int64_t rows, const void* x_perm,
                           const int32_t* offsets, const moe_expert_weights& w,
                           void* h, float* o, void* pre, cudaStream_t s, int part);

// Expert FFN on tcgen05 tensor cores (bf16, d % 256 == 0, F % 128 == 0).
bool ffn_tc_supported(const moe_config& c);
// The down projection writes y directly instead of o when every token has at
// most one expert output (K = 1, no shared experts): y[token_of_slot[s]] =
// bf16(gate[t] * o[s] (+ x[t])), the combine's arithmetic; the tokens the
// capacity dropped are written by launch_dropped_residual.
struct FusedCombine {
  const int32_t* token_of_slot;
  const float* gate;
  const void* x;  // residual rows or NULL
  void* y;
};
// pre (NULL or [padded rows][2F]) at rows poff[e] + r (the backward's padded
// row space, each expert's rows rounded up to 64). gu_part: fp32 partials
// [gate_up_ksplit][rows][2F] of a split gate/up reduction (decode-sized
// batches; NULL when gate_up_ksplit(c, rows) == 1). sched: two int32 tile
// counters that the CTA-pair GEMMs claim tiles from (gate/up, down); they
// must be 0 when each such GEMM starts: sched_zeroed says an earlier kernel
// on the stream (the dispatch scan) zeroed both, otherwise each part zeroes
// its counter before its launch.
int gate_up_ksplit(const moe_config& c, int64_t rows);
moe_status launch_ffn_tc(const moe_config& c, int64_t rows, const void* x_perm,
                         const int32_t* offsets, const moe_expert_weights& w,
                         void* h, float* o, void* pre, const int32_t* poff, float* gu_part,
                         int32_t* sched, bool sched_zeroed, uint32_t* status, cudaStream_t s,
                         int part, const FusedCombine* fc = nullptr);
// poff[e] = sum over e' < e of the rows of e' rounded up to 64 (one warp).
moe_status launch_pad_offsets(const int32_t* offsets, int G, int32_t* poff, cudaStream_t s);

// Backward pass (backward.cu): every gradient, from the state moe_forward
// kept in the workspace.
// Tensor-core router gradients (ffn_bwd_tc.cu): NP = N rounded up to 64, G
// token groups for the weight gradient's reduction.
struct RouterBwdPlan {
  int NP, G;
};
bool router_bwd_tc_supported(const moe_config& c);
RouterBwdPlan router_bwd_tc_plan(const moe_config& c);
moe_status launch_router_bwd_tc(const moe_config& c, const RouterBwdPlan& p, const float* dl,
                                const float* w_r, const void* x, float* dx, float* dw_r,
                                __nv_bfloat16* ar, __nv_bfloat16* br, int32_t* goff,
                                float* part, uint32_t* status, cudaStream_t s);

moe_status launch_backward(const moe_config& c, const WsLayout& L, void* ws, const void* x,
                           const float* w_r, const moe_expert_weights& w, const void* dy,
                           float z_coef, const moe_grads& g, uint32_t* status, cudaStream_t s);
int backward_launch_count(const moe_config& c);
bool ffn_bwd_tc_supported(const moe_config& c);
int64_t ffn_bwd_pad_rows(const moe_config& c);

}  // namespace moe
