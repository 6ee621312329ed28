// Backward pass of the sparse MoE layer: the gradients of
//   L = <dy, y> + L_aux + z_coef * z_loss
// with respect to x, the router weight and bias, and every expert weight.
//
// Sources: "MoE 混合专家模型稀疏激活的架构原理与负载均衡挑战" §四 训练不稳定性
// (the top-K choice has zero gradient, the gate softmax is differentiable)
// and §2.2 (f_i is a discrete count, P_i the continuous mean probability);
// "混合专家模型（Mixture of Experts, MoE）" 结构 2 (the router is trained end
// to end, its gradient flows back from the layer) and 结构 4 (the selection
// bias is not trained by gradient); "MoE 的核心思想" 辅助损失公式 and Router
// Z-Loss (both added to the training objective).
//
// Launch order (one stream; the forward's state is in the workspace):
//   1 combine_bwd   per token: dg[t][k] = <dy[t], o[slot]>, dout[slot] =
//                   g * dy[t] (shared experts: dy[t]), rounded to the dtype
//   2 router_bwd    per token: dl[t][:] from dg, P's share of L_aux and the
//                   z-loss, through the softmax and the gates
//   3 expert dgrad  dh = dout W_down^T-part, fused with the activation's
//                   derivative: pre <- (d gate-pre, d up-pre) in place
//   4 expert wgrad  dW_down[e] = dout_e^T h_e
//   5 expert dgrad  dx_perm = dpre_gate W_gate + dpre_up W_up (into o's buffer)
//   6 expert wgrad  dW_gate[e] = dpre_gate_e^T x_perm_e, dW_up likewise
//   7 dx            dx[t] = [residual] dy[t] + sum over t's slots of dx_perm
//   8 dx           += dl W_r
//   9 router wgrad  dW_r = dl^T x, db_r = sum_t dl (K-split partials, then a
//                   fixed-order reduction)
// Every reduction runs in a fixed order: the gradients are bitwise
// reproducible run to run.
#include "moe_common.cuh"

#include <algorithm>

namespace moe {

// Tensor-core expert gradients (ffn_bwd_tc.cu). dout and the pre-activations
// (then their gradients, in place) live in the padded row space poff (each
// expert's rows rounded up to 64, pad rows zero).
bool ffn_bwd_tc_supported(const moe_config& c);
int64_t ffn_bwd_pad_rows(const moe_config& c);
moe_status launch_ffn_bwd_tc(const moe_config& c, int64_t rows, int64_t rows_pad,
                             const int32_t* offsets, const int32_t* poff,
                             const moe_expert_weights& w, const void* x_perm, const void* h,
                             void* pre, const void* dout, float* dx_perm, const moe_grads& g,
                             uint32_t* status, cudaStream_t s);
int ffn_bwd_tc_launches(const moe_config& c);

namespace {

constexpr int kThreads = 256;

// ---- padded row space --------------------------------------------------------
// poff[e] = sum over e' < e of (offsets[e'+1] - offsets[e']) rounded up to 64
// (one warp; G <= 288).
__global__ void pad_offsets_kernel(const int32_t* __restrict__ offsets, int G,
                                   int32_t* __restrict__ poff) {
  const int lane = threadIdx.x;
  constexpr int PER = 9;
  int loc[PER], sum = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = lane * PER + j;
    loc[j] = e < G ? (offsets[e + 1] - offsets[e] + 63) / 64 * 64 : 0;
    sum += loc[j];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int run = incl - sum;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = lane * PER + j;
    if (e < G) poff[e] = run;
    run += loc[j];
  }
  if (lane == 31) poff[G] = incl;
}

}  // namespace

moe_status launch_pad_offsets(const int32_t* offsets, int G, int32_t* poff, cudaStream_t s) {
  pad_offsets_kernel<<<1, 32, 0, s>>>(offsets, G, poff);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

namespace {

// Zero the pad rows [poff[e] + count, poff[e+1]) of a [rows][ld] bf16 buffer;
// block e, at most 63 rows.
__global__ void __launch_bounds__(kThreads)
zero_pad_rows_kernel(__nv_bfloat16* __restrict__ buf, int ld, const int32_t* __restrict__ offsets,
                     const int32_t* __restrict__ poff) {
  const int e = blockIdx.x;
  const int r0 = poff[e] + (offsets[e + 1] - offsets[e]), r1 = poff[e + 1];
  const int per_row = ld / 8;  // 16-byte pieces
  for (int i = threadIdx.x; i < (r1 - r0) * per_row; i += kThreads) {
    const int r = r0 + i / per_row, c = i % per_row;
    reinterpret_cast<uint4*>(buf + static_cast<size_t>(r) * ld)[c] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// The weight-gradient products reduce over whole 64-row steps of the padded
// rows, so the last expert's step reads up to 63 forward rows past its end
// (multiplied by zero rows of A). Those rows [offsets[G], offsets[G] + 63) of
// x_perm and h are unused workspace: zero them (within rows_max) so that no
// stale bit pattern (NaN, infinity) meets the zeros.
__global__ void __launch_bounds__(kThreads)
zero_tail_rows_kernel(__nv_bfloat16* __restrict__ x_perm, int d, __nv_bfloat16* __restrict__ h,
                      int F, const int32_t* __restrict__ end, int64_t rows_max) {
  const int64_t r0 = *end;
  const int64_t r1 = min(rows_max, r0 + 63);
  const int pd = d / 8, pf = F / 8;  // 16-byte pieces per row
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x;
       i < (r1 - r0) * (pd + pf); i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t r = r0 + i / (pd + pf);
    const int c = static_cast<int>(i % (pd + pf));
    if (c < pd)
      reinterpret_cast<uint4*>(x_perm + r * d)[c] = make_uint4(0u, 0u, 0u, 0u);
    else
      reinterpret_cast<uint4*>(h + r * F)[c - pd] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// ---- 1. combine backward -----------------------------------------------------
// dout rows: slot s of expert e goes to row s - offsets[e] + poff[e] (poff ==
// offsets: the dispatch's own rows). TPB tokens per block, kThreads / TPB
// threads (whole warps) per token: dg[t][k] = <dy[t], o[slot]> is summed per
// thread over its columns, across each warp by a fixed butterfly and over the
// token's warps in order. A token with no kept slot (dropped everywhere)
// reads nothing and gets dg = 0.
template <typename Tx, int TPB>
__global__ void __launch_bounds__(kThreads)
combine_bwd_kernel(const Tx* __restrict__ dy, const float* __restrict__ o,
                   const int32_t* __restrict__ slot_of, const float* __restrict__ gate,
                   const int32_t* __restrict__ idx, const int32_t* __restrict__ offsets,
                   const int32_t* __restrict__ poff, int T, int N, int K, int S, int d,
                   Tx* __restrict__ dout, float* __restrict__ dg) {
  constexpr int TPT = kThreads / TPB;  // threads per token
  constexpr int WPT = TPT / 32;        // warps per token
  static_assert(TPT % 32 == 0, "whole warps per token");
  __shared__ int32_t s_slot[TPB][16], s_prow[TPB][16];
  __shared__ float s_gate[TPB][16];
  __shared__ float s_red[kThreads / 32][8];
  const int KS = K + S;
  const int tt = threadIdx.x / TPT, tid = threadIdx.x - tt * TPT;
  const int t = blockIdx.x * TPB + tt;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < TPB * KS; i += kThreads) {
    const int ti = i / KS, k = i - ti * KS, tok = blockIdx.x * TPB + ti;
    int slot = -1, prow = -1;
    float g = 1.f;
    if (tok < T) {
      slot = slot_of[static_cast<size_t>(tok) * KS + k];
      const int e = k < K ? idx[static_cast<size_t>(tok) * K + k] : N + (k - K);
      prow = slot >= 0 ? slot - offsets[e] + poff[e] : -1;
      if (k < K) g = gate[static_cast<size_t>(tok) * K + k];
    }
    s_slot[ti][k] = slot;
    s_prow[ti][k] = prow;
    s_gate[ti][k] = g;
  }
  __syncthreads();
  bool any = false;  // the same for the token's whole warps
  for (int k = 0; k < KS; ++k) any |= s_slot[tt][k] >= 0;
  float part[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) part[k] = 0.f;
  if (any) {
    for (int c = tid * 4; c < d; c += TPT * 4) {
      const float4 g4 = load4(dy + static_cast<size_t>(t) * d + c);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k >= K) break;
        const int sl = s_slot[tt][k];
        if (sl < 0) continue;
        const float4 ov =
            __ldg(reinterpret_cast<const float4*>(o + static_cast<size_t>(sl) * d + c));
        float p = part[k];
        p = fmaf(g4.x, ov.x, p);
        p = fmaf(g4.y, ov.y, p);
        p = fmaf(g4.z, ov.z, p);
        p = fmaf(g4.w, ov.w, p);
        part[k] = p;
        const float g = s_gate[tt][k];
        store4(dout + static_cast<size_t>(s_prow[tt][k]) * d + c,
               make_float4(g * g4.x, g * g4.y, g * g4.z, g * g4.w));
      }
      for (int k = K; k < KS; ++k)  // shared experts: gate 1
        store4(dout + static_cast<size_t>(s_prow[tt][k]) * d + c, g4);
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (k >= K) break;
    float v = part[k];
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o2);
    if (lane == 0) s_red[warp][k] = v;
  }
  __syncthreads();
  if (tid < K && t < T) {
    const int k = tid;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < WPT; ++w) v += s_red[tt * WPT + w][k];
    dg[static_cast<size_t>(t) * K + k] = s_slot[tt][k] >= 0 ? v : 0.f;
  }
}

// ---- 2. router backward: warp per token, lane owns experts lane + 32 j -------
template <int NJ>
__global__ void __launch_bounds__(kThreads)
router_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                  const float* __restrict__ gate, const float* __restrict__ dg,
                  const int32_t* __restrict__ count, int T, int N, int K, float alpha,
                  float z_coef, int gate_mode, float* __restrict__ dl) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kThreads / 32) + warp;
  if (t >= T) return;
  const float* lt = logits + static_cast<size_t>(t) * N;
  float v[NJ], p[NJ], dp[NJ], dsel[NJ];
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    v[j] = e < N ? lt[e] : -INFINITY;
    m = fmaxf(m, v[j]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    p[j] = lane + 32 * j < N ? expf(v[j] - m) : 0.f;
    s += p[j];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float inv = 1.f / s;
  const float lse = m + logf(s);
  // L_aux = alpha N sum_e f_e P_e, P_e = (1/T) sum_t p_te: dL/dp_te = alpha N f_e / T
  const float tk = static_cast<float>(T) * static_cast<float>(K);
  const float aux = alpha * static_cast<float>(N) / static_cast<float>(T);
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    p[j] *= inv;
    dp[j] = e < N ? aux * (static_cast<float>(count[e]) / tk) : 0.f;
    dsel[j] = 0.f;
  }
  const size_t tk0 = static_cast<size_t>(t) * K;
  if (gate_mode == MOE_GATE_SOFTMAX) {  // g_k = p[i_k]
    for (int k = 0; k < K; ++k) {
      const int e = idx[tk0 + k];
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        if (e == lane + 32 * j) dp[j] += dg[tk0 + k];
    }
  } else {  // g_k = softmax of the selected logits: dl_{i_k} += g_k (dg_k - sum g dg)
    float sg = 0.f;
    for (int k = 0; k < K; ++k) sg = fmaf(gate[tk0 + k], dg[tk0 + k], sg);
    for (int k = 0; k < K; ++k) {
      const int e = idx[tk0 + k];
      const float add = gate[tk0 + k] * (dg[tk0 + k] - sg);
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        if (e == lane + 32 * j) dsel[j] += add;
    }
  }
  float pd = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) pd = fmaf(p[j], dp[j], pd);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) pd += __shfl_xor_sync(0xffffffffu, pd, o);
  const float zc = z_coef * 2.f * lse / static_cast<float>(T);
  float* dlt = dl + static_cast<size_t>(t) * N;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    if (e < N) dlt[e] = dsel[j] + zc * p[j] + p[j] * (dp[j] - pd);
  }
}

// ---- 7. dx[t] = [residual] dy[t] + sum of dx_perm over t's slots --------------
// accumulate: dx already holds the router term dl W_r, which is added first.
template <typename Tx>
__global__ void __launch_bounds__(kThreads)
dx_gather_kernel(const Tx* __restrict__ dy, const float* __restrict__ dxp,
                 const int32_t* __restrict__ slot_of, int KS, int d, int add_residual,
                 int accumulate, float* __restrict__ dx) {
  __shared__ int32_t s_slot[16];
  const int t = blockIdx.x;
  if (threadIdx.x < KS) s_slot[threadIdx.x] = slot_of[static_cast<size_t>(t) * KS + threadIdx.x];
  __syncthreads();
  for (int c = threadIdx.x * 4; c < d; c += kThreads * 4) {
    float4 acc = accumulate ? *reinterpret_cast<const float4*>(dx + static_cast<size_t>(t) * d + c)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    if (add_residual) {
      const float4 r = load4(dy + static_cast<size_t>(t) * d + c);
      acc.x += r.x;
      acc.y += r.y;
      acc.z += r.z;
      acc.w += r.w;
    }
    for (int k = 0; k < KS; ++k) {
      const int s = s_slot[k];
      if (s < 0) continue;
      const float4 v = __ldg(reinterpret_cast<const float4*>(dxp + static_cast<size_t>(s) * d + c));
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    store4(dx + static_cast<size_t>(t) * d + c, acc);
  }
}

// ---- CUDA-core GEMMs ---------------------------------------------------------
constexpr int BM = 64, BN = 64, BK = 16;

enum { EPI_STORE = 0, EPI_ACCUM = 1, EPI_SWIGLU_BWD = 2, EPI_GELU_BWD = 3 };

// Row-grouped product: for the rows r of group g ([off[g], off[g+1]), or one
// group of n_rows rows when off is NULL),
//   acc[r][n] = sum_k A[r][k] * B_g(k, n),
//   B_g(k, n) = B0[g*bgs + k*ldb + n] (k < ksplit), B1[g*bgs + (k-ksplit)*ldb + n].
// Epilogue: STORE C = acc; ACCUM C += acc; SWIGLU_BWD: acc is dh, with
// (a, b) = (pre[r][n], pre[r][n_out + n]) -> pre = (dh b silu'(a), dh silu(a));
// GELU_BWD: acc is dh, z = pre[r][n] -> pre = dh gelu'(z).
// Grid: x = (group, 64-row tile) pairs (upper bound; extra blocks exit), y =
// 64-column tiles.
template <typename TA, typename TB, int EPI, typename TP>
__global__ void __launch_bounds__(kThreads)
gemm_rows_simt(const TA* __restrict__ A, int lda, const TB* __restrict__ B0,
               const TB* __restrict__ B1, int ksplit, size_t bgs, int ldb,
               const int32_t* __restrict__ off, int groups, int n_rows, int n_out, int kdim,
               float* __restrict__ C, int ldc, TP* __restrict__ pre, int ldp) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  __shared__ int s_g, s_m;
  if (threadIdx.x == 0) {
    int rem = blockIdx.x, gf = -1, mf = 0;
    for (int g = 0; g < groups; ++g) {
      const int cnt = off ? off[g + 1] - off[g] : n_rows;
      const int mt = (cnt + BM - 1) / BM;
      if (rem < mt) {
        gf = g;
        mf = rem;
        break;
      }
      rem -= mt;
    }
    s_g = gf;
    s_m = mf;
  }
  __syncthreads();
  const int g = s_g;
  if (g < 0) return;
  const int gbeg = off ? off[g] : 0, gend = off ? off[g + 1] : n_rows;
  const int row0 = gbeg + s_m * BM;
  const int rows = min(BM, gend - row0);
  const int n0 = blockIdx.y * BN;
  const TB* Bg0 = B0 + static_cast<size_t>(g) * bgs;
  const TB* Bg1 = B1 ? B1 + static_cast<size_t>(g) * bgs : nullptr;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < kdim; k0 += BK) {
    for (int i = threadIdx.x; i < BM * BK; i += kThreads) {
      const int r = i / BK, kk = i % BK, k = k0 + kk;
      As[kk][r] = (r < rows && k < kdim) ? to_f32(A[static_cast<size_t>(row0 + r) * lda + k]) : 0.f;
      const int kb = i / BN, n = i % BN, kg = k0 + kb;
      float bv = 0.f;
      if (n0 + n < n_out && kg < kdim)
        bv = kg < ksplit ? to_f32(Bg0[static_cast<size_t>(kg) * ldb + n0 + n])
                         : to_f32(Bg1[static_cast<size_t>(kg - ksplit) * ldb + n0 + n]);
      Bs[kb][n] = bv;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty * 4 + i;
    if (r >= rows) continue;
    const size_t grow = static_cast<size_t>(row0 + r);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= n_out) continue;
      const float v = acc[i][j];
      if (EPI == EPI_STORE) {
        C[grow * ldc + n] = v;
      } else if (EPI == EPI_ACCUM) {
        C[grow * ldc + n] += v;
      } else if (EPI == EPI_SWIGLU_BWD) {
        TP* pr = pre + grow * ldp;
        const float a = to_f32(pr[n]), b = to_f32(pr[n_out + n]);
        const float sg = 1.f / (1.f + expf(-a));
        pr[n] = from_f32<TP>(v * b * sg * (1.f + a * (1.f - sg)));
        pr[n_out + n] = from_f32<TP>(v * a * sg);
      } else {
        TP* pr = pre + grow * ldp;
        const float z = to_f32(pr[n]);
        const float cdf = 0.5f * (1.f + erff(z * 0.70710678118654752f));
        const float pdf = expf(-0.5f * z * z) * 0.39894228040143268f;
        pr[n] = from_f32<TP>(v * (cdf + z * pdf));
      }
    }
  }
}

// Weight-gradient product (reduction over the rows of a group):
//   out[sp][g][m][n] = sum over rows r of split sp of group g of
//                      A[r*lda + acol + m] * B[r*ldb + bcol + n]
// Group g has rows [off[g], off[g+1]) (off NULL: one group of n_rows); split
// sp takes the sp-th of `splits` equal row ranges. Grid: (M/64, Nn/64,
// groups * splits). An empty range writes zeros.
template <typename TA, typename TB>
__global__ void __launch_bounds__(kThreads)
gemm_wgrad_simt(const TA* __restrict__ A, int lda, int acol, const TB* __restrict__ B, int ldb,
                int bcol, const int32_t* __restrict__ off, int n_rows, int groups, int splits,
                int M, int Nn, float* __restrict__ out) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int g = blockIdx.z % groups, sp = blockIdx.z / groups;
  const int rb = off ? off[g] : 0, re = off ? off[g + 1] : n_rows;
  const int chunk = (re - rb + splits - 1) / splits;
  const int r0 = min(re, rb + sp * chunk), r1 = min(re, r0 + chunk);
  const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int k0 = r0; k0 < r1; k0 += BK) {
    for (int i = threadIdx.x; i < BM * BK; i += kThreads) {
      const int kk = i / BM, c = i % BM, r = k0 + kk;
      As[kk][c] = (r < r1 && m0 + c < M)
                      ? to_f32(A[static_cast<size_t>(r) * lda + acol + m0 + c]) : 0.f;
      Bs[kk][c] = (r < r1 && n0 + c < Nn)
                      ? to_f32(B[static_cast<size_t>(r) * ldb + bcol + n0 + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* o = out + (static_cast<size_t>(sp) * groups + g) * M * Nn;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < Nn) o[static_cast<size_t>(m) * Nn + n] = acc[i][j];
    }
  }
}

// Column sums per group and split: out[sp][g][c] = sum over the split's rows
// of A[r*lda + c], rows ascending. Grid: (ceil(ncols/256), groups * splits).
template <typename TA>
__global__ void __launch_bounds__(kThreads)
colsum_kernel(const TA* __restrict__ A, int lda, const int32_t* __restrict__ off, int n_rows,
              int groups, int splits, int ncols, float* __restrict__ out) {
  const int g = blockIdx.y % groups, sp = blockIdx.y / groups;
  const int c = blockIdx.x * kThreads + threadIdx.x;
  if (c >= ncols) return;
  const int rb = off ? off[g] : 0, re = off ? off[g + 1] : n_rows;
  const int chunk = (re - rb + splits - 1) / splits;
  const int r0 = min(re, rb + sp * chunk), r1 = min(re, r0 + chunk);
  float s = 0.f;
  for (int r = r0; r < r1; ++r) s += to_f32(A[static_cast<size_t>(r) * lda + c]);
  out[(static_cast<size_t>(sp) * groups + g) * ncols + c] = s;
}

// part[b][e] = sum of dl[t][e] over the 256 tokens of block b, ascending
// (thread e per column; N <= 256).
__global__ void __launch_bounds__(kThreads)
logit_colsum_kernel(const float* __restrict__ dl, int T, int N, float* __restrict__ part) {
  const int e = threadIdx.x;
  if (e >= N) return;
  const int t0 = blockIdx.x * 256, t1 = min(T, t0 + 256);
  float s = 0.f;
#pragma unroll 8
  for (int t = t0; t < t1; ++t) s += dl[static_cast<size_t>(t) * N + e];
  part[static_cast<size_t>(blockIdx.x) * N + e] = s;
}

// out[i] = sum_{sp ascending} part[sp * n + i]
__global__ void __launch_bounds__(kThreads)
reduce_splits_kernel(const float* __restrict__ part, int splits, size_t n,
                     float* __restrict__ out) {
  for (size_t i = blockIdx.x * static_cast<size_t>(kThreads) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * kThreads) {
    float s = 0.f;
    for (int sp = 0; sp < splits; ++sp) s += part[sp * n + i];
    out[i] = s;
  }
}

inline bool ok() { return cudaGetLastError() == cudaSuccess; }

unsigned row_tiles(int64_t rows, int groups) {
  return static_cast<unsigned>(groups + (rows + BM - 1) / BM);
}

// The expert part (steps 3-6) on CUDA cores, any dtype and activation.
template <typename Tx>
moe_status expert_bwd_simt(const moe_config& c, int64_t rows, const int32_t* offsets,
                           const moe_expert_weights& w, const Tx* x_perm, const Tx* h, Tx* pre,
                           const Tx* dout, float* dxp, const moe_grads& gr, cudaStream_t s) {
  const int E = c.n_experts + c.n_shared, d = c.d_model, F = c.d_ff;
  const bool swiglu = c.activation == MOE_SWIGLU;
  const Tx* wd = static_cast<const Tx*>(swiglu ? w.w_down : w.w2);       // [E][d][F]
  const Tx* w1 = static_cast<const Tx*>(swiglu ? w.w_gate : w.w1);       // [E][F][d]
  const Tx* wu = swiglu ? static_cast<const Tx*>(w.w_up) : nullptr;      // [E][F][d]
  float* dwd = swiglu ? gr.dw_down : gr.dw2;
  float* dw1 = swiglu ? gr.dw_gate : gr.dw1;
  const dim3 gF(row_tiles(rows, E), (F + BN - 1) / BN), gD(row_tiles(rows, E), (d + BN - 1) / BN);
  // 3: dh = dout . W_down (B_g(k = j, n = f) = W_down[e][j][f]) + activation derivative
  if (swiglu)
    gemm_rows_simt<Tx, Tx, EPI_SWIGLU_BWD, Tx><<<gF, kThreads, 0, s>>>(
        dout, d, wd, nullptr, d, static_cast<size_t>(d) * F, F, offsets, E, 0, F, d, nullptr, 0,
        pre, 2 * F);
  else
    gemm_rows_simt<Tx, Tx, EPI_GELU_BWD, Tx><<<gF, kThreads, 0, s>>>(
        dout, d, wd, nullptr, d, static_cast<size_t>(d) * F, F, offsets, E, 0, F, d, nullptr, 0,
        pre, 2 * F);
  if (!ok()) return MOE_ERR_CUDA;
  trace_record(2, s);
  // 4: dW_down[e] = dout_e^T h_e  ([d][F] per expert)
  gemm_wgrad_simt<Tx, Tx><<<dim3((d + BM - 1) / BM, (F + BN - 1) / BN, E), kThreads, 0, s>>>(
      dout, d, 0, h, F, 0, offsets, 0, E, 1, d, F, dwd);
  if (!ok()) return MOE_ERR_CUDA;
  if (!swiglu && c.has_bias) {  // db2[e] = sum of the expert's output gradients
    colsum_kernel<Tx><<<dim3((d + kThreads - 1) / kThreads, E), kThreads, 0, s>>>(
        dout, d, offsets, 0, E, 1, d, gr.db2);
    if (!ok()) return MOE_ERR_CUDA;
  }
  trace_record(3, s);
  // 5: dx_perm = dpre_gate . W_gate + dpre_up . W_up (B_g(k = f, n = j) = W[e][f][j])
  gemm_rows_simt<Tx, Tx, EPI_STORE, Tx><<<gD, kThreads, 0, s>>>(
      pre, 2 * F, w1, wu, F, static_cast<size_t>(F) * d, d, offsets, E, 0, d,
      swiglu ? 2 * F : F, dxp, d, nullptr, 0);
  if (!ok()) return MOE_ERR_CUDA;
  trace_record(4, s);
  // 6: dW_gate[e] = dpre_gate_e^T x_perm_e ([F][d]); dW_up from columns F..2F
  const dim3 gw((F + BM - 1) / BM, (d + BN - 1) / BN, E);
  gemm_wgrad_simt<Tx, Tx><<<gw, kThreads, 0, s>>>(pre, 2 * F, 0, x_perm, d, 0, offsets, 0, E, 1,
                                                   F, d, dw1);
  if (!ok()) return MOE_ERR_CUDA;
  if (swiglu) {
    gemm_wgrad_simt<Tx, Tx><<<gw, kThreads, 0, s>>>(pre, 2 * F, F, x_perm, d, 0, offsets, 0, E,
                                                     1, F, d, gr.dw_up);
    if (!ok()) return MOE_ERR_CUDA;
  } else if (c.has_bias) {  // db1[e] = sum of the expert's dz rows
    colsum_kernel<Tx><<<dim3((F + kThreads - 1) / kThreads, E), kThreads, 0, s>>>(
        pre, 2 * F, offsets, 0, E, 1, F, gr.db1);
    if (!ok()) return MOE_ERR_CUDA;
  }
  trace_record(5, s);
  return MOE_OK;
}

template <typename Tx>
moe_status backward_t(const moe_config& c, const WsLayout& L, void* ws, const Tx* x,
                      const float* w_r, const moe_expert_weights& w, const Tx* dy, float z_coef,
                      const moe_grads& gr, uint32_t* status, cudaStream_t s) {
  auto at = [&](size_t o) { return static_cast<uint8_t*>(ws) + o; };
  const int T = c.T, N = c.n_experts, K = c.top_k, S = c.n_shared, d = c.d_model;
  const int E = N + S, F = c.d_ff;
  const int32_t* idx = reinterpret_cast<const int32_t*>(at(L.idx));
  const float* gate = reinterpret_cast<const float*>(at(L.gate));
  const int32_t* offsets = reinterpret_cast<const int32_t*>(at(L.offsets));
  const int32_t* slot_of = reinterpret_cast<const int32_t*>(at(L.slot_of));
  const Tx* x_perm = reinterpret_cast<const Tx*>(at(L.x_perm));
  const Tx* h = reinterpret_cast<const Tx*>(at(L.h));
  float* o = reinterpret_cast<float*>(at(L.o));  // expert outputs, then dx_perm
  const float* logits = reinterpret_cast<const float*>(at(L.logits));
  Tx* pre = reinterpret_cast<Tx*>(at(L.pre));
  const int32_t* count = reinterpret_cast<const int32_t*>(at(L.count));
  Tx* dout = reinterpret_cast<Tx*>(at(L.dout));
  float* dg = reinterpret_cast<float*>(at(L.dg));
  float* dl = reinterpret_cast<float*>(at(L.dl));
  float* rpart = reinterpret_cast<float*>(at(L.rpart));
  const int64_t rows = rows_max_of(&c);

  if (T == 0) {  // no tokens: every gradient is zero
    const size_t es = sizeof(float);
    if (cudaMemsetAsync(gr.dw_r, 0, static_cast<size_t>(N) * d * es, s) != cudaSuccess ||
        (gr.db_r && cudaMemsetAsync(gr.db_r, 0, N * es, s) != cudaSuccess))
      return MOE_ERR_CUDA;
    const size_t wsz = static_cast<size_t>(E) * F * d * es;
    float* mats[3] = {c.activation == MOE_SWIGLU ? gr.dw_gate : gr.dw1,
                      c.activation == MOE_SWIGLU ? gr.dw_up : nullptr,
                      c.activation == MOE_SWIGLU ? gr.dw_down : gr.dw2};
    for (float* m : mats)
      if (m && cudaMemsetAsync(m, 0, wsz, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (c.activation == MOE_GELU && c.has_bias &&
        (cudaMemsetAsync(gr.db1, 0, static_cast<size_t>(E) * F * es, s) != cudaSuccess ||
         cudaMemsetAsync(gr.db2, 0, static_cast<size_t>(E) * d * es, s) != cudaSuccess))
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  trace_record(0, s);
  const bool tc = ffn_bwd_tc_supported(c);
  // the tensor-core path keeps dout and the pre-activation gradients in the
  // padded row space; the CUDA-core path in the dispatch's rows
  int32_t* poff = reinterpret_cast<int32_t*>(at(L.poff));
  if (tc) {  // poff: written by the forward (with the pre-activations)
    zero_pad_rows_kernel<<<E, kThreads, 0, s>>>(reinterpret_cast<__nv_bfloat16*>(dout), d,
                                                offsets, poff);
    if (!ok()) return MOE_ERR_CUDA;
    zero_tail_rows_kernel<<<16, kThreads, 0, s>>>(
        reinterpret_cast<__nv_bfloat16*>(const_cast<Tx*>(x_perm)), d,
        reinterpret_cast<__nv_bfloat16*>(const_cast<Tx*>(h)), F, offsets + E, rows);
    if (!ok()) return MOE_ERR_CUDA;
  }
  // 1
  // narrow rows (d <= 1024): four tokens per block, so each thread has several
  // columns in flight (measured on the Switch-shaped layer: 115 -> 82 us for
  // this stage); wider rows keep a whole block per token (four tokens per
  // block measured slower there: 0.34 -> 0.44 ms on the DeepSeek-shaped layer)
  if (d <= 1024)
    combine_bwd_kernel<Tx, 4><<<(T + 3) / 4, kThreads, 0, s>>>(
        dy, o, slot_of, gate, idx, offsets, tc ? poff : offsets, T, N, K, S, d, dout, dg);
  else
    combine_bwd_kernel<Tx, 1><<<T, kThreads, 0, s>>>(
        dy, o, slot_of, gate, idx, offsets, tc ? poff : offsets, T, N, K, S, d, dout, dg);
  if (!ok()) return MOE_ERR_CUDA;
  // 2
  const unsigned rb = static_cast<unsigned>((T + kThreads / 32 - 1) / (kThreads / 32));
#define MOE_RBWD(NJ)                                                                           \
  router_bwd_kernel<NJ><<<rb, kThreads, 0, s>>>(logits, idx, gate, dg, count, T, N, K, c.alpha, \
                                                z_coef, c.gate_mode, dl)
  if (N <= 32) MOE_RBWD(1);
  else if (N <= 64) MOE_RBWD(2);
  else if (N <= 128) MOE_RBWD(4);
  else MOE_RBWD(8);
#undef MOE_RBWD
  if (!ok()) return MOE_ERR_CUDA;
  trace_record(1, s);
  // 3-6 (trace events 2-5 after each of the four products)
  moe_status r = tc ? launch_ffn_bwd_tc(c, rows, ffn_bwd_pad_rows(c), offsets, poff, w, x_perm,
                                        h, pre, dout, o, gr, status, s)
                    : expert_bwd_simt<Tx>(c, rows, offsets, w, x_perm, h, pre, dout, o, gr, s);
  if (r != MOE_OK) return r;
  const int sp = L.rsplits;
  if (router_bwd_tc_supported(c)) {
    // 8 then 7: dx = dl W_r on the tensor cores, then the gather adds the
    // residual and the expert input gradients; 9: dW_r on the tensor cores
    r = launch_router_bwd_tc(c, router_bwd_tc_plan(c), dl, w_r, x, gr.dx, gr.dw_r,
                             reinterpret_cast<__nv_bfloat16*>(at(L.r_ar)),
                             reinterpret_cast<__nv_bfloat16*>(at(L.r_br)),
                             reinterpret_cast<int32_t*>(at(L.r_goff)),
                             reinterpret_cast<float*>(at(L.r_part)), status, s);
    if (r != MOE_OK) return r;
    dx_gather_kernel<Tx><<<T, kThreads, 0, s>>>(dy, o, slot_of, K + S, d, c.add_residual, 1,
                                                gr.dx);
    if (!ok()) return MOE_ERR_CUDA;
    trace_record(6, s);
  } else {
    // 7
    dx_gather_kernel<Tx><<<T, kThreads, 0, s>>>(dy, o, slot_of, K + S, d, c.add_residual, 0,
                                                gr.dx);
    if (!ok()) return MOE_ERR_CUDA;
    // 8: dx += dl . W_r  (B(k = e, n = j) = W_r[e][j])
    gemm_rows_simt<float, float, EPI_ACCUM, float>
        <<<dim3(row_tiles(T, 1), (d + BN - 1) / BN), kThreads, 0, s>>>(
            dl, N, w_r, nullptr, N, 0, d, nullptr, 1, T, d, N, gr.dx, d, nullptr, 0);
    if (!ok()) return MOE_ERR_CUDA;
    trace_record(6, s);
    // 9: dW_r = dl^T x (split over tokens, then reduced)
    gemm_wgrad_simt<float, Tx>
        <<<dim3((N + BM - 1) / BM, (d + BN - 1) / BN, sp), kThreads, 0, s>>>(
            dl, N, 0, x, d, 0, nullptr, T, 1, sp, N, d, rpart);
    if (!ok()) return MOE_ERR_CUDA;
    const size_t nd = static_cast<size_t>(N) * d;
    const unsigned redb = static_cast<unsigned>(std::min<size_t>(
        (nd + kThreads - 1) / kThreads, static_cast<size_t>(sm_count()) * 8));
    reduce_splits_kernel<<<redb, kThreads, 0, s>>>(rpart, sp, nd, gr.dw_r);
    if (!ok()) return MOE_ERR_CUDA;
  }
  if (gr.db_r) {  // db_r = column sums of dl: 256-token blocks, then a fixed-order reduction
    float* bpart = reinterpret_cast<float*>(at(L.bpart));
    const int nb = (T + 255) / 256;
    logit_colsum_kernel<<<nb, kThreads, 0, s>>>(dl, T, N, bpart);
    if (!ok()) return MOE_ERR_CUDA;
    reduce_splits_kernel<<<1, kThreads, 0, s>>>(bpart, nb, N, gr.db_r);
    if (!ok()) return MOE_ERR_CUDA;
  }
  trace_record(7, s);
  return MOE_OK;
}

}  // namespace

int backward_launch_count(const moe_config& c) {
  if (c.T == 0) return 0;
  const bool swiglu = c.activation == MOE_SWIGLU;
  int n = 2;  // combine_bwd, router_bwd
  // + pad rows of dout, tail rows of x_perm and h
  if (ffn_bwd_tc_supported(c)) n += 2 + ffn_bwd_tc_launches(c);
  else n += swiglu ? 5 : (c.has_bias ? 6 : 4);
  if (router_bwd_tc_supported(c)) n += 5;  // split, dl W_r, gather, dW_r partials, reduction
  else n += 4;                              // gather, dl W_r, dW_r partials, reduction
  n += 2;                                   // db_r partials, reduction
  return n;
}

moe_status launch_backward(const moe_config& c, const WsLayout& L, void* ws, const void* x,
                           const float* w_r, const moe_expert_weights& w, const void* dy,
                           float z_coef, const moe_grads& g, uint32_t* status, cudaStream_t s) {
  if (c.dtype == MOE_BF16)
    return backward_t<__nv_bfloat16>(c, L, ws, static_cast<const __nv_bfloat16*>(x), w_r, w,
                                     static_cast<const __nv_bfloat16*>(dy), z_coef, g, status, s);
  return backward_t<float>(c, L, ws, static_cast<const float*>(x), w_r, w,
                           static_cast<const float*>(dy), z_coef, g, status, s);
}

}  // namespace moe
