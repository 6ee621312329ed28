// Fused router: logits = x W_r^T (+ b_r), softmax, top-K, renormalised gates,
// and per-block partial sums of the load-balance statistics; then a one-block
// kernel reduces the partials in a fixed order into count, f, P and L_aux.
//
// Sources: "MoE 混合专家模型稀疏激活的架构原理与负载均衡挑战" §2.1 (logits =
// x·W_r, Top-K, softmax over the selected logits) and §2.2 (L_aux =
// alpha·N·Σ f_i·P_i, f from the top-k indices, P the mean router probability);
// "混合专家模型（Mixture of Experts, MoE）" 结构 2 (G(x) = Softmax(W_r·x)) and
// 运行示例 (router = nn.Linear with bias; renormalised top-K weights).
//
// Design: one block of 256 threads owns 32 tokens and all N experts. The 8
// warps split the work (experts x d-slices) so that every N in [1, 256] keeps
// all warps busy; the d-slices are summed in shared memory in a fixed order
// (deterministic), the logits of the block's 32 tokens then sit in shared
// memory and each warp runs softmax / top-K / gates for 4 tokens with warp
// shuffles. The contraction runs in fp32 FFMA (tf32 tensor cores would not
// keep the logits accurate enough for bit-exact routing against float64).
#include "moe_common.cuh"
#include "router_select.cuh"

#include <float.h>

#include <cuda.h>

#include <mutex>

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
static_assert(kWarps == kSelectWarps, "router block shape");
constexpr int BM = kRouterTokensPerBlock;  // 32 tokens per block

// NPW: experts per warp (8: N <= 8, one token per lane; 32: 4 tokens x 8
// experts per lane). WS_N: warps across experts; the other 8/WS_N warps split d.
template <typename Tx, int NPW, int WS_N>
__global__ void __launch_bounds__(kThreads)
router_kernel(const Tx* __restrict__ x, const float* __restrict__ w_r,
              const float* __restrict__ b_r, const float* __restrict__ sel_bias, int gate_mode,
              int T, int d, int N, int K,
              int32_t* __restrict__ idx_out, float* __restrict__ gate_out,
              float* __restrict__ psum, int32_t* __restrict__ pcnt,
              uint32_t* __restrict__ status, float* __restrict__ logits_out) {
  constexpr int WS_K = kWarps / WS_N;
  constexpr int NP = NPW * WS_N;                  // padded expert count
  constexpr int LT = (NPW == 8) ? 32 : 8;         // lanes across tokens
  constexpr int LE = 32 / LT;                     // lanes across experts
  constexpr int TT = BM / LT;                     // tokens per lane
  constexpr int TE = NPW / LE;                    // experts per lane (8)
  static_assert(TT * LT == BM && TE * LE == NPW, "tile shape");

  __shared__ float red[WS_K * BM * NP];           // partial logits per d-slice
  __shared__ float pw[kWarps][256];               // per-warp probability sums
  __shared__ float zh[2 * kWarps];                // per-warp z-loss / entropy sums
  __shared__ int32_t scnt[256];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * BM;
  const int wn = warp % WS_N, wk = warp / WS_N;
  const int lt = lane / LE, le = lane % LE;

  for (int i = tid; i < 256; i += kThreads) scnt[i] = 0;

  // ---- phase A: partial logits over this warp's d-slice ----
  float acc[TT][TE];
#pragma unroll
  for (int i = 0; i < TT; ++i)
#pragma unroll
    for (int j = 0; j < TE; ++j) acc[i][j] = 0.f;

  const int slice = ((d / 4 + WS_K - 1) / WS_K) * 4;
  const int kb = min(d, wk * slice), ke = min(d, kb + slice);
  const Tx* xrow[TT];
  bool tok_ok[TT];
#pragma unroll
  for (int i = 0; i < TT; ++i) {
    const int t = t0 + lt * TT + i;
    tok_ok[i] = t < T;
    xrow[i] = x + static_cast<size_t>(tok_ok[i] ? t : 0) * d;
  }
  const float* wrow[TE];
  bool exp_ok[TE];
#pragma unroll
  for (int j = 0; j < TE; ++j) {
    const int e = wn * NPW + le * TE + j;
    exp_ok[j] = e < N;
    wrow[j] = w_r + static_cast<size_t>(exp_ok[j] ? e : 0) * d;
  }
  for (int k = kb; k < ke; k += 4) {
    float4 xv[TT], wv[TE];
#pragma unroll
    for (int i = 0; i < TT; ++i) xv[i] = load4(xrow[i] + k);
#pragma unroll
    for (int j = 0; j < TE; ++j) wv[j] = load4(wrow[j] + k);
#pragma unroll
    for (int i = 0; i < TT; ++i)
#pragma unroll
      for (int j = 0; j < TE; ++j) {
        float a = acc[i][j];
        a = fmaf(xv[i].x, wv[j].x, a);
        a = fmaf(xv[i].y, wv[j].y, a);
        a = fmaf(xv[i].z, wv[j].z, a);
        a = fmaf(xv[i].w, wv[j].w, a);
        acc[i][j] = a;
      }
  }
#pragma unroll
  for (int i = 0; i < TT; ++i)
#pragma unroll
    for (int j = 0; j < TE; ++j)
      red[(wk * BM + lt * TT + i) * NP + wn * NPW + le * TE + j] = acc[i][j];
  __syncthreads();

  // ---- phase B: sum the d-slices in a fixed order, add the bias ----
  for (int i = tid; i < BM * NP; i += kThreads) {
    float s = red[i];
#pragma unroll
    for (int q = 1; q < WS_K; ++q) s += red[q * BM * NP + i];
    const int e = i % NP;
    if (b_r != nullptr && e < N) s += b_r[e];
    red[i] = s;
  }
  __syncthreads();

  // ---- phase C: softmax, top-K and gates; warp per token ----
  constexpr int NJ = (NP + 31) / 32;  // experts per lane in this phase
  float pacc[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) pacc[j] = 0.f;
  float zacc = 0.f, hacc = 0.f;

  for (int tl = warp; tl < BM; tl += kWarps) {
    const int t = t0 + tl;
    if (t >= T) break;
    float v[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      v[j] = (e < N) ? red[tl * NP + e] : -INFINITY;
    }
    route_one_token<NJ>(v, N, K, static_cast<size_t>(t), lane, sel_bias, gate_mode, idx_out,
                        gate_out, pacc, zacc, hacc, scnt, status, logits_out);
  }

  // ---- phase D: per-block partials in a fixed order ----
  write_block_stats<NJ>(pacc, zacc, hacc, pw, zh, scnt, N, blockIdx.x, psum, pcnt);
}

// One block per expert e reduces the router blocks' partials psum[e][*] and
// pcnt[e][*] (contiguous, coalesced): thread i sums blocks i, i+256, ... in
// order, then fixed shuffle and shared-memory trees; every run adds in the
// same order. Writes count[e], P[e] = sum / T, f[e] = count / (T*K), and
// leaves the totals in psum[e][0], pcnt[e][0] for route_laux_kernel.
__global__ void __launch_bounds__(256)
route_stats_kernel(float* __restrict__ psum, int32_t* __restrict__ pcnt, int nblk, int T, int N,
                   int K, int32_t* count, float* f, float* P, float* z_loss, float* entropy) {
  __shared__ float ws_s[8];
  __shared__ int32_t ws_c[8];
  const int e = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool expert = e < N;  // rows N, N+1: z-loss and entropy sums
  const float* ps = psum + static_cast<size_t>(e) * nblk;
  const int32_t* pc = pcnt + static_cast<size_t>(expert ? e : 0) * nblk;
  float s = 0.f;
  int32_t c = 0;
  for (int b = threadIdx.x; b < nblk; b += blockDim.x) {
    s += ps[b];
    if (expert) c += pc[b];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    c += __shfl_xor_sync(0xffffffffu, c, o);
  }
  if (lane == 0) {
    ws_s[warp] = s;
    ws_c[warp] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float st = 0.f;
    int32_t ct = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
      st += ws_s[w];
      ct += ws_c[w];
    }
    const float mean = T > 0 ? st / static_cast<float>(T) : 0.f;
    if (!expert) {
      float* dst = e == N ? z_loss : entropy;
      if (dst) *dst = mean;
      return;
    }
    if (count) count[e] = ct;
    if (f) f[e] = T > 0 ? static_cast<float>(ct) / (static_cast<float>(T) * K) : 0.f;
    if (P) P[e] = mean;
    psum[static_cast<size_t>(e) * nblk] = st;  // only this block reads row e
    pcnt[static_cast<size_t>(e) * nblk] = ct;
  }
}

// L_aux = alpha * N * sum_e f[e] * P[e] from the per-expert totals that
// route_stats_kernel left in psum[e][0], pcnt[e][0]. One thread per expert
// loads its two totals (all loads in flight at once); warp w then adds the
// products of experts 32w .. 32w+31 with a fixed butterfly and thread 0 adds
// the warps in order.
__global__ void __launch_bounds__(256)
route_laux_kernel(const float* __restrict__ psum, const int32_t* __restrict__ pcnt, int nblk,
                  int T, int N, int K, float alpha, float* l_aux) {
  __shared__ float wsum[8];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  float s = 0.f;
  if (e < N && T > 0) {
    const float Pe = psum[static_cast<size_t>(e) * nblk] / static_cast<float>(T);
    const float fe = static_cast<float>(pcnt[static_cast<size_t>(e) * nblk]) /
                     (static_cast<float>(T) * K);
    s = fe * Pe;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) wsum[warp] = s;
  __syncthreads();
  if (e == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += wsum[w];
    *l_aux = alpha * static_cast<float>(N) * t;
  }
}

// With at most 64 partial blocks per row (small batches) one block of 1024
// threads reduces every row and then L_aux: one launch instead of two. Warp w
// sums rows w, w + 32, ...: lane l takes partial blocks l and l + 32, then a fixed butterfly adds the lanes; L_aux adds f * P over the
// experts in a fixed order. With many more partial blocks a warp would walk
// them serially (measured: 15 us for 256 per row, 78 us for 512 rows of 258,
// latency-bound), so the per-row blocks of route_stats_kernel take them
// instead.
constexpr int kStatsOneBlockMaxBlocks = 64;

__global__ void __launch_bounds__(1024)
route_stats_one_block_kernel(const float* __restrict__ psum, const int32_t* __restrict__ pcnt,
                             int nblk, int T, int N, int K, float alpha, int32_t* count,
                             float* f, float* P, float* z_loss, float* entropy, float* l_aux) {
  __shared__ float tot[258];
  __shared__ int32_t totc[256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = static_cast<int>(blockDim.x >> 5);
  for (int r = warp; r < N + 2; r += nwarps) {
    const bool expert = r < N;  // rows N, N+1: z-loss and entropy sums
    const float* ps = psum + static_cast<size_t>(r) * nblk;
    const int32_t* pc = pcnt + static_cast<size_t>(expert ? r : 0) * nblk;
    float sum = 0.f;
    int32_t c = 0;
#pragma unroll 4
    for (int b = lane; b < nblk; b += 32) {
      sum += ps[b];
      if (expert) c += pc[b];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sum += __shfl_xor_sync(0xffffffffu, sum, o);
      c += __shfl_xor_sync(0xffffffffu, c, o);
    }
    if (lane == 0) {
      tot[r] = sum;
      if (expert) totc[r] = c;
    }
  }
  __syncthreads();
  for (int r = threadIdx.x; r < N + 2; r += blockDim.x) {
    const float mean = T > 0 ? tot[r] / static_cast<float>(T) : 0.f;
    if (r < N) {
      if (count) count[r] = totc[r];
      if (f) f[r] = T > 0 ? static_cast<float>(totc[r]) / (static_cast<float>(T) * K) : 0.f;
      if (P) P[r] = mean;
    } else {
      float* dst = r == N ? z_loss : entropy;
      if (dst) *dst = mean;
    }
  }
  if (warp == 0 && l_aux != nullptr) {
    float sum = 0.f;
    for (int e = lane; e < N; e += 32) {
      const float Pe = T > 0 ? tot[e] / static_cast<float>(T) : 0.f;
      const float fe =
          T > 0 ? static_cast<float>(totc[e]) / (static_cast<float>(T) * K) : 0.f;
      sum += fe * Pe;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) *l_aux = alpha * static_cast<float>(N) * sum;
  }
}

// Decode-sized batches (router_small: T <= 128, N <= 32): one block of 8
// warps per token. Warp w takes the w-th eighth of d (whole groups of four);
// each lane keeps one fp32 partial per expert over its share, a
// reduce-scatter across the warp (full butterfly steps over the offsets >= NE,
// then halving steps in which the lanes with bit o set keep the upper half)
// leaves lane l with the warp's partial for expert l % NE, and warp 0 adds the
// eight warps' partials in order, adds b_r and runs the shared selection. One
// launch replaces the tensor-core router's weight split, split-K GEMM and
// top-K kernel, whose fixed costs exceed the work at this size. The
// statistics partials are per token (nblk = T).
template <typename Tx, int NE>
__global__ void __launch_bounds__(kThreads)
router_small_kernel(const Tx* __restrict__ x, const float* __restrict__ w_r,
                    const float* __restrict__ b_r, const float* __restrict__ sel_bias,
                    int gate_mode, int T, int d, int N, int K, int32_t* __restrict__ idx_out,
                    float* __restrict__ gate_out, float* __restrict__ psum,
                    int32_t* __restrict__ pcnt, uint32_t* __restrict__ status,
                    float* __restrict__ logits_out) {
  __shared__ float red[kWarps][32];
  __shared__ float pw[kWarps][256];
  __shared__ float zh[2 * kWarps];
  __shared__ int32_t scnt[256];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.x;
  for (int i = tid; i < 256; i += kThreads) scnt[i] = 0;

  float acc[NE];
#pragma unroll
  for (int e = 0; e < NE; ++e) acc[e] = 0.f;
  const int slice = ((d / 4 + kWarps - 1) / kWarps) * 4;
  const int kb = min(d, warp * slice), ke = min(d, kb + slice);
  const Tx* xr = x + static_cast<size_t>(t) * d;
  // two groups of four per lane in flight (four, fully unrolled, measured
  // slower on the decode-shaped router: 14.1 -> 16.4 us)
#pragma unroll 2
  for (int k = kb + lane * 4; k < ke; k += 128) {
    const float4 xv = load4(xr + k);
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      if (e < N) {
        const float4 wv = load4(w_r + static_cast<size_t>(e) * d + k);
        float a = acc[e];
        a = fmaf(xv.x, wv.x, a);
        a = fmaf(xv.y, wv.y, a);
        a = fmaf(xv.z, wv.z, a);
        a = fmaf(xv.w, wv.w, a);
        acc[e] = a;
      }
    }
  }
#pragma unroll
  for (int o = 16; o >= NE; o >>= 1)
#pragma unroll
    for (int e = 0; e < NE; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
#pragma unroll
  for (int o = NE / 2; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? acc[i] : acc[i + o];
      const float keep = upper ? acc[i + o] : acc[i];
      acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  if (lane < NE) red[warp][lane] = acc[0];
  __syncthreads();

  float pacc[1] = {0.f};
  float zacc = 0.f, hacc = 0.f;
  if (warp == 0) {
    float v[1] = {-INFINITY};
    if (lane < N) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += red[w][lane];
      if (b_r != nullptr) s += b_r[lane];
      v[0] = s;
    }
    route_one_token<1>(v, N, K, static_cast<size_t>(t), lane, sel_bias, gate_mode, idx_out,
                       gate_out, pacc, zacc, hacc, scnt, status, logits_out);
  }
  write_block_stats<1>(pacc, zacc, hacc, pw, zh, scnt, N, blockIdx.x, psum, pcnt);
}

template <typename Tx>
cudaError_t launch_router_small(const moe_config& c, const Tx* x, const float* w_r,
                                const float* b_r, int32_t* idx, float* gate, float* psum,
                                int32_t* pcnt, uint32_t* status, float* logits, cudaStream_t s) {
  const int N = c.n_experts;
#define MOE_SMALL(NE)                                                                         \
  router_small_kernel<Tx, NE><<<c.T, kThreads, 0, s>>>(x, w_r, b_r, c.select_bias,            \
                                                       c.gate_mode, c.T, c.d_model, N,        \
                                                       c.top_k, idx, gate, psum, pcnt,        \
                                                       status, logits)
  if (N <= 8) MOE_SMALL(8);
  else if (N <= 16) MOE_SMALL(16);
  else MOE_SMALL(32);
#undef MOE_SMALL
  return cudaGetLastError();
}

template <typename Tx>
cudaError_t launch_router_t(const moe_config& c, const Tx* x, const float* w_r, const float* b_r,
                            int32_t* idx, float* gate, float* psum, int32_t* pcnt,
                            uint32_t* status, float* logits, cudaStream_t s) {
  const int nblk = (c.T + BM - 1) / BM;
  const int N = c.n_experts;
  dim3 grid(nblk), block(kThreads);
#define MOE_ROUTER(NPW, WSN)                                                                  \
  router_kernel<Tx, NPW, WSN><<<grid, block, 0, s>>>(x, w_r, b_r, c.select_bias, c.gate_mode, \
                                                     c.T, c.d_model, N, c.top_k, idx, gate,    \
                                                     psum, pcnt, status, logits)
  if (N <= 8) MOE_ROUTER(8, 1);
  else if (N <= 32) MOE_ROUTER(32, 1);
  else if (N <= 64) MOE_ROUTER(32, 2);
  else if (N <= 128) MOE_ROUTER(32, 4);
  else MOE_ROUTER(32, 8);
#undef MOE_ROUTER
  return cudaGetLastError();
}

}  // namespace

moe_status launch_router(const moe_config& c, const void* x, const float* w_r, const float* b_r,
                         int32_t* idx, float* gate, const RouterScratch& sc, const moe_stats* st,
                         cudaStream_t s) {
  if (c.T == 0) return MOE_OK;
  uint32_t* status = st ? st->status : nullptr;
  float* psum = sc.psum;
  int32_t* pcnt = sc.pcnt;
  const RouterTcPlan plan = router_tc_plan(c);
  int nblk = (c.T + BM - 1) / BM;  // statistics partials left by the router
  if (router_small(c)) {
    nblk = c.T;
    const cudaError_t err =
        c.dtype == MOE_BF16
            ? launch_router_small(c, static_cast<const __nv_bfloat16*>(x), w_r, b_r, idx, gate,
                                  psum, pcnt, status, sc.logits, s)
            : launch_router_small(c, static_cast<const float*>(x), w_r, b_r, idx, gate, psum,
                                  pcnt, status, sc.logits, s);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
  } else if (plan.use && sc.w3 != nullptr && (plan.fused || sc.part != nullptr)) {
    nblk = plan.stat_blocks;
    const moe_status r = launch_router_tc(c, plan, x, w_r, b_r, idx, gate, sc.w3, sc.part, psum,
                                          pcnt, status, sc.logits, s);
    if (r != MOE_OK) return r;
  } else {
    cudaError_t err;
    if (c.dtype == MOE_BF16)
      err = launch_router_t(c, static_cast<const __nv_bfloat16*>(x), w_r, b_r, idx, gate, psum,
                            pcnt, status, sc.logits, s);
    else
      err = launch_router_t(c, static_cast<const float*>(x), w_r, b_r, idx, gate, psum, pcnt,
                            status, sc.logits, s);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (st && (st->count || st->f || st->P || st->l_aux || st->z_loss || st->entropy)) {
    if (nblk <= kStatsOneBlockMaxBlocks) {
      route_stats_one_block_kernel<<<1, 1024, 0, s>>>(psum, pcnt, nblk, c.T, c.n_experts,
                                                      c.top_k, c.alpha, st->count, st->f,
                                                      st->P, st->z_loss, st->entropy, st->l_aux);
      return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    route_stats_kernel<<<c.n_experts + 2, 256, 0, s>>>(psum, pcnt, nblk, c.T, c.n_experts,
                                                       c.top_k, st->count, st->f, st->P,
                                                       st->z_loss, st->entropy);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    if (st->l_aux) {
      route_laux_kernel<<<1, 256, 0, s>>>(psum, pcnt, nblk, c.T, c.n_experts, c.top_k, c.alpha,
                                          st->l_aux);
      if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    }
  }
  return MOE_OK;
}

bool router_small(const moe_config& c) {
  return c.T > 0 && c.T <= 128 && c.n_experts <= 32 && c.d_model % 4 == 0;
}

int route_stats_launches(const moe_config& c) {
  const RouterTcPlan plan = router_tc_plan(c);
  const int64_t nblk =
      router_small(c) ? c.T : (plan.use ? plan.stat_blocks : (c.T + BM - 1) / BM);
  return nblk <= kStatsOneBlockMaxBlocks ? 1 : 2;
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Router without a caller workspace.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: a
// serving process whose device memory is all owned by its own pool and that
// forbids any other allocation after start-up, or a plug-in interface whose
// signature has no workspace argument. For them moe_route_no_workspace runs
// the CUDA-core (FFMA) router and the statistics kernels of moe_route, with
// the per-block partial sums held in the fixed array below instead of the
// workspace. moe_route takes the tensor-core router for bf16 layers whose d
// is a multiple of 64; the two sum the logits in different orders, so their
// choices can differ on near-tie tokens (an adjacent gap among the K+1
// largest logits below 1e-5) and this entry point can be slower there. The
// array lives in every GPU that loads this library, until the process exits.
//
// Limit: ceil(T / 32) * (N + 2) <= kRouteScratchElems (131072; 1 MiB of
// scratch: one fp32 per (token block, expert or z-loss/entropy row) and one
// int32 per (token block, expert)); larger requests return MOE_ERR_WORKSPACE
// before anything is launched.
//
// Sharing: every call uses the same array. The router kernel writes every
// partial it later reads, so nothing needs clearing between calls, but calls
// whose kernels overlap on the GPU (different streams, or different host
// threads) race on the array; serialise them.
// ---------------------------------------------------------------------------
namespace moe {
namespace {

constexpr size_t kRouteScratchElems = 131072;
static __device__ __align__(256) unsigned char g_route_scratch[kRouteScratchElems * 8];

// Device address of g_route_scratch, looked up once per CUDA context with
// that context current (in host code the symbol's name is only a host-side
// stand-in, never a device address). A context belongs to one device, and
// its ID (cuCtxGetId) is never reused within the process, so an address
// cached under a context that was destroyed (cudaDeviceReset) or belongs to
// another context on the same device is never handed out again. When the
// driver's context calls are unavailable the address is looked up on every
// call instead.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name, int version) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}

constexpr int kScratchCache = 64;
struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
ScratchEntry g_scratch_cache[kScratchCache] = {};
int g_scratch_next = 0;
std::mutex g_scratch_mu;

moe_status route_scratch_address(void** out) {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 4000);
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
  auto context_id = [](unsigned long long* id) {
    CUcontext ctx = nullptr;
    return get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
           get_id(ctx, id) == CUDA_SUCCESS && *id != 0;
  };
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long id = 0;
  if (context_id(&id))
    for (const ScratchEntry& e : g_scratch_cache)
      if (e.ctx_id == id) {
        *out = e.addr;
        return MOE_OK;
      }
  // the lookup also makes the device's primary context current when this
  // thread has none yet; the key is read again after it
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr)
    return MOE_ERR_CUDA;
  if (context_id(&id)) {
    g_scratch_cache[g_scratch_next] = ScratchEntry{id, p};
    g_scratch_next = (g_scratch_next + 1) % kScratchCache;
  }
  *out = p;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_no_workspace(const moe_config* cfg, const void* x,
                                             const float* w_r, const float* b_r, int32_t* idx,
                                             float* gate, moe_stats* stats,
                                             moe_stream_t stream) {
  using namespace moe;
  try {
    moe_status why = MOE_OK;
    if (!config_valid(cfg, &why)) return why;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!x || !w_r || !idx || !gate) return MOE_ERR_INVALID;
    if (!a16(x) || !a16(w_r) || !a16(idx) || !a16(gate) || (b_r && !a16(b_r)))
      return MOE_ERR_INVALID;
    const size_t nblk = (static_cast<size_t>(cfg->T) + BM - 1) / BM;
    if (nblk * static_cast<size_t>(cfg->n_experts + 2) > kRouteScratchElems)
      return MOE_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (moe_status s = route_scratch_address(&scratch)) return s;
    float* psum = static_cast<float*>(scratch);
    int32_t* pcnt = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(scratch) +
                                               kRouteScratchElems * sizeof(float));
    const RouterScratch sc{psum, pcnt, nullptr, nullptr, nullptr};  // CUDA-core router
    return launch_router(*cfg, x, w_r, b_r, idx, gate, sc, stats,
                         static_cast<cudaStream_t>(stream));
  } catch (...) {
    return MOE_ERR_CUDA;
  }
}
