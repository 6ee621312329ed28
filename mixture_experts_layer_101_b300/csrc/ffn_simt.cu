// Grouped expert FFN on CUDA cores (fp32 FFMA): the path for fp32 layers
// (fp32 results within 1e-4 of the float64 definition rule out tf32 tensor
// cores) and for bf16 shapes the tensor-core kernel does not tile
// (d % 256 != 0 or F % 128 != 0).
//
// Sources: "MoE 混合专家模型稀疏激活的架构原理与负载均衡挑战" §三 class Expert
// (down(silu(gate(x)) * up(x))); "混合专家模型（Mixture of Experts, MoE）"
// 运行示例 (Linear(h, 2h) -> GELU -> Linear(2h, h), with bias).
//
// C[s][n] = sum_k A[s][k] * B[e][n][k] for the rows s of expert e, 64x64
// output tiles, 16-wide K steps staged in shared memory, 4x4 per thread.
// Block x indexes the (expert, 64-row tile) pairs in expert order (found
// from the device offsets), block y the 64-column tiles.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, kThreads = 256;

enum { EPI_SWIGLU = 0, EPI_GELU = 1, EPI_LINEAR = 2 };

template <typename T, int EPI, typename TOut>
__global__ void __launch_bounds__(kThreads)
grouped_gemm_simt(const T* __restrict__ A, const T* __restrict__ B0, const T* __restrict__ B1,
                  const T* __restrict__ bias, const int32_t* __restrict__ offsets, int n_experts,
                  int n_out, int kdim, TOut* __restrict__ C, T* __restrict__ pre) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs0[BK][BN + 4];
  __shared__ float Bs1[(EPI == EPI_SWIGLU) ? BK : 1][BN + 4];
  __shared__ int s_e, s_m;

  if (threadIdx.x == 0) {
    int rem = blockIdx.x, e_found = -1, m_found = 0;
    for (int e = 0; e < n_experts; ++e) {
      const int cnt = offsets[e + 1] - offsets[e];
      const int mt = (cnt + BM - 1) / BM;
      if (rem < mt) {
        e_found = e;
        m_found = rem;
        break;
      }
      rem -= mt;
    }
    s_e = e_found;
    s_m = m_found;
  }
  __syncthreads();
  const int e = s_e;
  if (e < 0) return;
  const int row0 = offsets[e] + s_m * BM;
  const int rows = min(BM, offsets[e + 1] - row0);
  const int n0 = blockIdx.y * BN;

  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc0[4][4] = {}, acc1[4][4] = {};
  const T* Bb0 = B0 + static_cast<size_t>(e) * n_out * kdim;
  const T* Bb1 = (EPI == EPI_SWIGLU) ? B1 + static_cast<size_t>(e) * n_out * kdim : nullptr;

  // A (64 x 16) and B (64 x 16) per K step: 1024 elements each, 4 per thread
  // (element i = threadIdx.x + j * kThreads). The next step's elements are
  // loaded into registers before this step's products, so their latency
  // overlaps the arithmetic (small layers are latency-bound).
  constexpr int PER = BM * BK / kThreads;
  float ra[PER], rb0[PER], rb1[PER];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = threadIdx.x + j * kThreads;
      const int r = i / BK, kk = i % BK;
      const int k = k0 + kk;
      ra[j] = (r < rows && k < kdim) ? to_f32(A[static_cast<size_t>(row0 + r) * kdim + k]) : 0.f;
      const int n = n0 + r;
      rb0[j] = (n < n_out && k < kdim) ? to_f32(Bb0[static_cast<size_t>(n) * kdim + k]) : 0.f;
      if (EPI == EPI_SWIGLU)
        rb1[j] = (n < n_out && k < kdim) ? to_f32(Bb1[static_cast<size_t>(n) * kdim + k]) : 0.f;
    }
  };
  fetch(0);
  for (int k0 = 0; k0 < kdim; k0 += BK) {
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = threadIdx.x + j * kThreads;
      const int r = i / BK, kk = i % BK;
      As[kk][r] = ra[j];
      Bs0[kk][r] = rb0[j];
      if (EPI == EPI_SWIGLU) Bs1[kk][r] = rb1[j];
    }
    __syncthreads();
    if (k0 + BK < kdim) fetch(k0 + BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b0[4], b1[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        b0[j] = Bs0[kk][tx * 4 + j];
        if (EPI == EPI_SWIGLU) b1[j] = Bs1[kk][tx * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc0[i][j] = fmaf(a[i], b0[j], acc0[i][j]);
          if (EPI == EPI_SWIGLU) acc1[i][j] = fmaf(a[i], b1[j], acc1[i][j]);
        }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty * 4 + i;
    if (r >= rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= n_out) continue;
      float v;
      // pre (backward pass): [row][2 * n_out], gate | up pre-activations (GELU: z)
      T* pre_row = pre ? pre + static_cast<size_t>(row0 + r) * 2 * n_out : nullptr;
      if (EPI == EPI_SWIGLU) {
        const float g = acc0[i][j];
        v = g / (1.f + expf(-g)) * acc1[i][j];
        if (pre_row) {
          pre_row[n] = from_f32<T>(g);
          pre_row[n_out + n] = from_f32<T>(acc1[i][j]);
        }
      } else if (EPI == EPI_GELU) {
        float z = acc0[i][j];
        if (bias) z += to_f32(bias[static_cast<size_t>(e) * n_out + n]);
        v = 0.5f * z * (1.f + erff(z * 0.70710678118654752f));
        if (pre_row) pre_row[n] = from_f32<T>(z);
      } else {
        v = acc0[i][j];
        if (bias) v += to_f32(bias[static_cast<size_t>(e) * n_out + n]);
      }
      C[static_cast<size_t>(row0 + r) * n_out + n] = from_f32<TOut>(v);
    }
  }
}

template <typename T>
moe_status run(const moe_config& c, int64_t a_max, const T* x_perm, const int32_t* offsets,
               const moe_expert_weights& w, T* h, float* o, T* pre, cudaStream_t s, int part) {
  const int N = c.n_experts + c.n_shared, d = c.d_model, F = c.d_ff;  // routed + shared
  const int64_t mtiles = N + (a_max + BM - 1) / BM;  // upper bound on (expert, m-tile) pairs
  if (mtiles > 0x7fffffff) return MOE_ERR_UNSUPPORTED;
  dim3 g1(static_cast<unsigned>(mtiles), (F + BN - 1) / BN), g2(static_cast<unsigned>(mtiles),
                                                                 (d + BN - 1) / BN);
  const bool swiglu = c.activation == MOE_SWIGLU;
  if (part & 1) {
    if (swiglu)
      grouped_gemm_simt<T, EPI_SWIGLU, T><<<g1, kThreads, 0, s>>>(
          x_perm, static_cast<const T*>(w.w_gate), static_cast<const T*>(w.w_up), nullptr,
          offsets, N, F, d, h, pre);
    else
      grouped_gemm_simt<T, EPI_GELU, T><<<g1, kThreads, 0, s>>>(
          x_perm, static_cast<const T*>(w.w1), nullptr, static_cast<const T*>(w.b1), offsets, N,
          F, d, h, pre);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (part & 2) {
    grouped_gemm_simt<T, EPI_LINEAR, float><<<g2, kThreads, 0, s>>>(
        h, static_cast<const T*>(swiglu ? w.w_down : w.w2), nullptr,
        swiglu ? nullptr : static_cast<const T*>(w.b2), offsets, N, d, F, o, nullptr);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace

moe_status launch_ffn_simt(const moe_config& c, int64_t a_max, const void* x_perm,
                           const int32_t* offsets, const moe_expert_weights& w, void* h, float* o,
                           void* pre, cudaStream_t s, int part) {
  if (a_max == 0) return MOE_OK;
  if (c.dtype == MOE_BF16)
    return run<__nv_bfloat16>(c, a_max, static_cast<const __nv_bfloat16*>(x_perm), offsets, w,
                              static_cast<__nv_bfloat16*>(h), o,
                              static_cast<__nv_bfloat16*>(pre), s, part);
  return run<float>(c, a_max, static_cast<const float*>(x_perm), offsets, w,
                    static_cast<float*>(h), o, static_cast<float*>(pre), s, part);
}

}  // namespace moe
