// Gate-weighted combine: y[t] = sum_k gate[t][k] * o[slot_of[t][k]]
// + sum_s o[slot_of[t][K+s]] (shared experts, gate 1) (+ x[t]).
//
// Sources: "混合专家模型（Mixture of Experts, MoE）" 结构 3 (y = Σ_{i∈TopK}
// G(x)_i·E_i(x)); "MoE 如何替代 FFN？…" §2 (MoE(x) = Σ g(x)_i·Expert_i(x));
// "MoE 混合专家模型稀疏激活的架构原理与负载均衡挑战" §2.3 (dropped tokens pass
// on the residual).
//
// One block per token; each thread owns 4 consecutive columns (16-byte
// loads of the fp32 expert outputs), accumulates the K ranks in ascending
// order in fp32 and rounds once. Each output element is written by exactly
// one thread: no atomics, deterministic.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

template <typename Tx>
__global__ void __launch_bounds__(kThreads)
combine_kernel(const float* __restrict__ o, const int32_t* __restrict__ slot_of,
               const float* __restrict__ gate, const Tx* __restrict__ x, Tx* __restrict__ y,
               int K, int S, int d, int add_residual) {
  __shared__ int32_t s_slot[16];
  __shared__ float s_gate[16];
  const int t = blockIdx.x;
  const int KS = K + S;  // routed ranks, then shared experts with gate 1
  if (threadIdx.x < KS) {
    s_slot[threadIdx.x] = slot_of[static_cast<size_t>(t) * KS + threadIdx.x];
    s_gate[threadIdx.x] =
        threadIdx.x < K ? gate[static_cast<size_t>(t) * K + threadIdx.x] : 1.f;
  }
  __syncthreads();
  for (int c = threadIdx.x * 4; c < d; c += kThreads * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < KS; ++k) {
      const int s = s_slot[k];
      if (s < 0) continue;
      const float g = s_gate[k];
      const float4 v = __ldg(reinterpret_cast<const float4*>(o + static_cast<size_t>(s) * d + c));
      acc.x = fmaf(g, v.x, acc.x);
      acc.y = fmaf(g, v.y, acc.y);
      acc.z = fmaf(g, v.z, acc.z);
      acc.w = fmaf(g, v.w, acc.w);
    }
    if (add_residual) {
      const float4 xv = load4(x + static_cast<size_t>(t) * d + c);
      acc.x += xv.x;
      acc.y += xv.y;
      acc.z += xv.z;
      acc.w += xv.w;
    }
    store4(y + static_cast<size_t>(t) * d + c, acc);
  }
}

}  // namespace

moe_status launch_combine(const moe_config& c, const float* o, const int32_t* slot_of,
                          const float* gate, const void* x, void* y, cudaStream_t s) {
  if (c.T == 0) return MOE_OK;
  if (c.dtype == MOE_BF16)
    combine_kernel<__nv_bfloat16><<<c.T, kThreads, 0, s>>>(
        o, slot_of, gate, static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y),
        c.top_k, c.n_shared, c.d_model, c.add_residual);
  else
    combine_kernel<float><<<c.T, kThreads, 0, s>>>(o, slot_of, gate, static_cast<const float*>(x),
                                                   static_cast<float*>(y), c.top_k, c.n_shared,
                                                   c.d_model, c.add_residual);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
