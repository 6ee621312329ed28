// Gate-weighted combine: y[t] = sum_k gate[t][k] * o[slot_of[t][k]]
// + sum_s o[slot_of[t][K+s]] (shared experts, gate 1) (+ x[t]).
//
// Sources: "混合专家模型（Mixture of Experts, MoE）" 结构 3 (y = Σ_{i∈TopK}
// G(x)_i·E_i(x)); "MoE 如何替代 FFN？…" §2 (MoE(x) = Σ g(x)_i·Expert_i(x));
// "MoE 混合专家模型稀疏激活的架构原理与负载均衡挑战" §2.3 (dropped tokens pass
// on the residual).
//
// Each thread owns 4 consecutive columns (16-byte loads of the fp32 expert
// outputs) of a few tokens, accumulates the ranks in ascending order in fp32
// and rounds once. Each output element is written by exactly one thread: no
// atomics, deterministic.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

// Four consecutive residual elements kept in their storage form until used
// (two registers for bf16 instead of four floats).
template <typename Tx>
struct Residual4;
template <>
struct Residual4<float> {
  using Raw = float4;
  static __device__ __forceinline__ Raw load(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
  }
  static __device__ __forceinline__ Raw zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
  static __device__ __forceinline__ float4 value(Raw r) { return r; }
};
template <>
struct Residual4<__nv_bfloat16> {
  using Raw = uint2;
  static __device__ __forceinline__ Raw load(const __nv_bfloat16* p) {
    return __ldg(reinterpret_cast<const uint2*>(p));
  }
  static __device__ __forceinline__ Raw zero() { return make_uint2(0u, 0u); }
  static __device__ __forceinline__ float4 value(Raw r) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
};

// TPB tokens per block: each thread owns 4 consecutive columns of all TPB
// tokens, so its TPB * (K + S) 16-byte loads are independent and in flight
// together. With one or two expert outputs per token, one token per block
// leaves too few bytes in flight per SM to reach HBM rate (TPB = 4 measured
// 10% faster on the Switch-shaped layer); with eight, one token per block is
// faster (measured 0.16 ms against 0.28 ms on the DeepSeek-shaped layer).
template <typename Tx, int TPB>
__global__ void __launch_bounds__(kThreads, TPB == 4 ? 4 : 1)
combine_kernel(const float* __restrict__ o, const int32_t* __restrict__ slot_of,
               const float* __restrict__ gate, const Tx* __restrict__ x, Tx* __restrict__ y,
               int T, int K, int S, int d, int add_residual) {
  __shared__ int32_t s_slot[TPB][16];
  __shared__ float s_gate[TPB][16];
  const int t0 = blockIdx.x * TPB;
  const int KS = K + S;  // routed ranks, then shared experts with gate 1
  for (int i = threadIdx.x; i < TPB * KS; i += kThreads) {
    const int tt = i / KS, k = i % KS, t = t0 + tt;
    s_slot[tt][k] = t < T ? slot_of[static_cast<size_t>(t) * KS + k] : -1;
    s_gate[tt][k] = (t < T && k < K) ? gate[static_cast<size_t>(t) * K + k] : 1.f;
  }
  // The residual rows do not depend on the routing: the first columns' loads
  // go out before the barrier, overlapping the slot lookups.
  using R = Residual4<Tx>;
  typename R::Raw xr[TPB];
  auto load_residual = [&](int c) {
#pragma unroll
    for (int tt = 0; tt < TPB; ++tt) {
      const int t = t0 + tt;
      xr[tt] = (add_residual && t < T) ? R::load(x + static_cast<size_t>(t) * d + c) : R::zero();
    }
  };
  // block column slice y of gridDim.y (one slice unless the batch is small)
  const int c0 = (static_cast<int>(blockIdx.y) * kThreads + threadIdx.x) * 4;
  const int cstride = kThreads * 4 * static_cast<int>(gridDim.y);
  if (c0 < d) load_residual(c0);
  __syncthreads();
  for (int c = c0; c < d; c += cstride) {
    if (c != c0) load_residual(c);
    float4 acc[TPB];
#pragma unroll
    for (int tt = 0; tt < TPB; ++tt) acc[tt] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < KS; ++k) {
#pragma unroll
      for (int tt = 0; tt < TPB; ++tt) {
        const int s = s_slot[tt][k];
        if (s < 0) continue;
        const float g = s_gate[tt][k];
        const float4 v =
            __ldg(reinterpret_cast<const float4*>(o + static_cast<size_t>(s) * d + c));
        acc[tt].x = fmaf(g, v.x, acc[tt].x);
        acc[tt].y = fmaf(g, v.y, acc[tt].y);
        acc[tt].z = fmaf(g, v.z, acc[tt].z);
        acc[tt].w = fmaf(g, v.w, acc[tt].w);
      }
    }
#pragma unroll
    for (int tt = 0; tt < TPB; ++tt) {
      const int t = t0 + tt;
      if (t >= T) break;
      if (add_residual) {
        const float4 xv = R::value(xr[tt]);
        acc[tt].x += xv.x;
        acc[tt].y += xv.y;
        acc[tt].z += xv.z;
        acc[tt].w += xv.w;
      }
      store4(y + static_cast<size_t>(t) * d + c, acc[tt]);
    }
  }
}

// One warp per token: a token whose one assignment was dropped (slot -1)
// gets y = x (residual) or 0; kept tokens are left to the fused down
// projection.
template <typename Tx>
__global__ void __launch_bounds__(256)
dropped_residual_kernel(const int32_t* __restrict__ slot_of, const Tx* __restrict__ x,
                        Tx* __restrict__ y, int T, int d, int add_residual) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T || slot_of[t] >= 0) return;
  const int lane = threadIdx.x & 31;
  const int chunks = d * static_cast<int>(sizeof(Tx)) / 16;
  uint4* dst = reinterpret_cast<uint4*>(y + static_cast<size_t>(t) * d);
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d);
  for (int c = lane; c < chunks; c += 32)
    dst[c] = add_residual ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace

moe_status launch_dropped_residual(const moe_config& c, const int32_t* slot_of, const void* x,
                                   void* y, cudaStream_t s) {
  if (c.T == 0) return MOE_OK;
  const unsigned blocks = static_cast<unsigned>((c.T + 7) / 8);
  if (c.dtype == MOE_BF16)
    dropped_residual_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
        slot_of, static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), c.T,
        c.d_model, c.add_residual);
  else
    dropped_residual_kernel<float><<<blocks, 256, 0, s>>>(
        slot_of, static_cast<const float*>(x), static_cast<float*>(y), c.T, c.d_model,
        c.add_residual);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_combine(const moe_config& c, const float* o, const int32_t* slot_of,
                          const float* gate, const void* x, void* y, cudaStream_t s) {
  if (c.T == 0) return MOE_OK;
  // A small batch (fewer token blocks than twice the SMs) takes one token per
  // block and splits the columns over blockIdx.y, so its few rows still
  // spread over many SMs (decode: 16 tokens in 64 blocks instead of 4).
  const int cols_per_block = kThreads * 4;
  const bool small = c.T < 2 * sm_count();
  const bool wide = c.top_k + c.n_shared <= 2 && !small;
  const int tpb = wide ? 4 : 1;
  const int slices = small ? (c.d_model + cols_per_block - 1) / cols_per_block : 1;
  const dim3 blocks(static_cast<unsigned>((c.T + tpb - 1) / tpb), static_cast<unsigned>(slices));
#define MOE_COMBINE(TX, TPBV)                                                                  \
  combine_kernel<TX, TPBV><<<blocks, kThreads, 0, s>>>(o, slot_of, gate,                       \
                                                       static_cast<const TX*>(x),              \
                                                       static_cast<TX*>(y), c.T, c.top_k,      \
                                                       c.n_shared, c.d_model, c.add_residual)
  if (c.dtype == MOE_BF16) {
    if (wide) MOE_COMBINE(__nv_bfloat16, 4);
    else MOE_COMBINE(__nv_bfloat16, 1);
  } else {
    if (wide) MOE_COMBINE(float, 4);
    else MOE_COMBINE(float, 1);
  }
#undef MOE_COMBINE
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
