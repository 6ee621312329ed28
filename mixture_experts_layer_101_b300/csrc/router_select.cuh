// Per-token expert selection shared by the router kernels: softmax over the
// N experts, top-K by logit (ties go to the lower expert index), gates =
// softmax of the K selected logits, and the per-block partial sums of the
// load-balance statistics.
//
// Sources: "MoE 混合专家模型稀疏激活的架构原理与负载均衡挑战" §三
// MoERouter.forward (torch.topk on the logits, softmax of the top-k logits,
// softmax(logits).mean(0) and the counts of the top-k indices for the
// load-balance loss); "混合专家模型（Mixture of Experts, MoE）" 运行示例
// (softmax, top-k, renormalised weights); "MoE 的核心思想" 具体数值示例.
#pragma once

#include "moe_common.cuh"

namespace moe {

constexpr int kSelectWarps = 8;  // warps per router block (256 threads)

// One warp holds one token's logits: lane owns experts lane + 32*j, j < NJ
// (entries of experts >= N are ignored). Writes idx/gate of token t, adds the
// token's softmax to pacc, counts the chosen experts in scnt (shared), and in
// lane 0 adds the token's squared log-sum-exp to zacc and its routing entropy
// to hacc. sel_bias (NULL or [N]) shifts the logits for the top-K choice
// only ("混合专家模型（Mixture of Experts, MoE）" 结构 4); gate_mode picks the
// renormalised or the full-softmax gate. logits_out (NULL or [T][N]) keeps
// the token's logits for the backward pass.
template <int NJ>
__device__ __forceinline__ void route_one_token(const float (&v)[NJ], int N, int K, size_t t,
                                                int lane, const float* __restrict__ sel_bias,
                                                int gate_mode, int32_t* __restrict__ idx_out,
                                                float* __restrict__ gate_out, float (&pacc)[NJ],
                                                float& zacc, float& hacc, int32_t* scnt,
                                                uint32_t* status, float* logits_out = nullptr) {
  if (logits_out != nullptr) {
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      if (lane + 32 * j < N) logits_out[t * N + lane + 32 * j] = v[j];
  }
  bool bad = false;
#pragma unroll
  for (int j = 0; j < NJ; ++j)
    if (lane + 32 * j < N && !isfinite(v[j])) bad = true;
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, MOE_ERR_NONFINITE);
  // softmax over the N experts
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < NJ; ++j)
    if (lane + 32 * j < N) m = fmaxf(m, v[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float p[NJ], s = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    p[j] = (lane + 32 * j < N) ? expf(v[j] - m) : 0.f;
    s += p[j];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float inv = 1.f / s;
  float pv = 0.f;  // sum_e p_e * l_e, for the entropy lse - sum p l
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    pacc[j] += p[j] * inv;
    if (p[j] > 0.f) pv += p[j] * inv * v[j];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) pv += __shfl_xor_sync(0xffffffffu, pv, o);
  const float lse = m + logf(s);
  if (lane == 0) {
    zacc += lse * lse;
    hacc += lse - pv;
  }

  // top-K: K rounds of a warp arg-max of the (biased) selection key; ties go
  // to the lower index; every lane records the unbiased logits selected
  float key[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    const float vv = isnan(v[j]) ? -INFINITY : v[j];
    key[j] = (sel_bias != nullptr && e < N) ? vv + sel_bias[e] : vv;
  }
  uint32_t taken = 0;
  float sel_u[8];
  int sel_e = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) sel_u[k] = -INFINITY;
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY, bu = -INFINITY;
    int be = INT32_MAX;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      if (e < N && !(taken & (1u << j)) && (key[j] > bv || (key[j] == bv && e < be))) {
        bv = key[j];
        be = e;
        bu = v[j];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      const float ou = __shfl_xor_sync(0xffffffffu, bu, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
        bu = ou;
      }
    }
    if (be < 0 || be >= N) be = 0;  // unreachable while K <= N; keeps indices in range
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      if (kk == k) sel_u[kk] = bu;
    if (lane == k) sel_e = be;
  }
  if (lane < K) {
    float my_u = sel_u[0];
#pragma unroll
    for (int kk = 1; kk < 8; ++kk)
      if (kk == lane) my_u = sel_u[kk];
    float g;
    if (gate_mode == MOE_GATE_SOFTMAX) {
      g = expf(my_u - m) * inv;
    } else {  // softmax over the K selected unbiased logits, summed in rank order
      float msel = sel_u[0];
#pragma unroll
      for (int kk = 1; kk < 8; ++kk)
        if (kk < K) msel = fmaxf(msel, sel_u[kk]);
      float gsum = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        if (kk < K) gsum += expf(sel_u[kk] - msel);
      g = expf(my_u - msel) / gsum;
    }
    idx_out[t * K + lane] = sel_e;
    gate_out[t * K + lane] = g;
    atomicAdd(&scnt[sel_e], 1);
  }
}

// Block-level partial statistics, summed over the block's warps in order,
// stored expert-major so that one expert's partials are contiguous:
// psum[e][blk] = softmax mass of the block's tokens on e, pcnt[e][blk] =
// their assignments to e, psum[N][blk] / psum[N+1][blk] = their summed
// squared log-sum-exp / entropy (nblk = gridDim.x). zh is a shared float[16].
// Every thread of the block calls this.
template <int NJ>
__device__ __forceinline__ void write_block_stats(const float (&pacc)[NJ], float zacc, float hacc,
                                                  float (*pw)[256], float* zh,
                                                  const int32_t* scnt, int N, size_t blk,
                                                  float* __restrict__ psum,
                                                  int32_t* __restrict__ pcnt) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#pragma unroll
  for (int j = 0; j < NJ; ++j)
    if (lane + 32 * j < 256) pw[warp][lane + 32 * j] = pacc[j];
  if (lane == 0) {
    zh[warp] = zacc;
    zh[kSelectWarps + warp] = hacc;
  }
  __syncthreads();
  const size_t nblk = gridDim.x;
  for (int e = tid; e < N; e += blockDim.x) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kSelectWarps; ++w) s += pw[w][e];
    psum[static_cast<size_t>(e) * nblk + blk] = s;
    pcnt[static_cast<size_t>(e) * nblk + blk] = scnt[e];
  }
  if (tid < 2) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kSelectWarps; ++w) s += zh[tid * kSelectWarps + w];
    psum[static_cast<size_t>(N + tid) * nblk + blk] = s;
  }
}

}  // namespace moe
