// Router logits on the tcgen05 tensor cores, exact to fp32 accuracy.
//
// Sources: "MoE 混合专家模型稀疏激活的架构原理与负载均衡挑战" §2.1 (logits =
// x·W_r with W_r in R^{d x N}) and §三 MoERouter (weight stored (N, d),
// logits = x @ W^T); "混合专家模型（Mixture of Experts, MoE）" 结构 2.
//
// The router weight is fp32; bf16 tensor cores multiply bf16 operands. Each
// fp32 weight w is split exactly into three bf16 numbers, w = hi + mid + lo
// (hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid); each residual
// is exact in fp32 and the last one has at most 8 significant bits). x is
// bf16, so every product x*hi, x*mid, x*lo is exact in the fp32 accumulator,
// and x . W = x . hi + x . mid + x . lo is computed with fp32 accumulation
// only: the same accuracy class as an fp32 FFMA dot product, which routing
// that must match float64 needs (a 10-bit tf32 product would not do).
//
// Kernels:
//   router_split_kernel  W_r [N][d] fp32 -> W3 [3][NP][d] bf16 (rows >= N zero)
//   router_gemm_tc<NPT>  per (128-token tile, NPT-expert tile, K split):
//                        part[s][t][e] = sum over the split's K of x[t] . W3[*][e]
//                        (TMA ring of x and the three planes, tcgen05.mma
//                        M=128 N=NPT K=16 into two alternating TMEM
//                        accumulators, summed in fp32 registers)
//   router_topk_kernel   per token: logits = sum_s part[s][t] (s ascending)
//                        + b_r, then softmax / top-K / gates / statistics.
// Accumulation length: the tensor core adds each product into the fp32
// accumulator with less than round-to-nearest accuracy, so a long chain of
// MMAs into one TMEM accumulator drifts (measured on the DeepSeek-shaped
// router: gate error 2.3e-5 with 112 64-wide K steps per chain, 9e-7 with 2).
// The MMA warp therefore restarts the accumulator every kChunkKb K steps,
// alternating between two TMEM buffers, and the epilogue adds each finished
// chunk into fp32 registers (round-to-nearest), overlapped with the next
// chunk's MMAs. The K split gives enough CTAs for small T; chunk and split
// sums are added in a fixed order, so results are deterministic.
#include "moe_common.cuh"
#include "ptx_sm100.cuh"
#include "router_select.cuh"

#include <cudaTypedefs.h>

#include <mutex>

namespace moe {
namespace {

constexpr int kThreads = 192;
constexpr int BM = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kTargetCtas = 148;  // split K until the grid roughly fills a B300
constexpr int kMaxSplits = 16;
constexpr int kChunkKb = 2;  // 64-wide K steps per TMEM accumulation chain

// FUSED kernels keep two stages, so that two CTAs share an SM (NPT <= 64) and
// one CTA's selection epilogue overlaps the other's main loop.
template <int NPT, bool FUSED>
struct Shape {
  static constexpr int B_PLANE = NPT * BK * 2;           // one plane's tile
  static constexpr int STAGE = A_BYTES + 3 * B_PLANE;     // x tile + 3 planes
  static constexpr int STAGES = FUSED ? 2 : ((NPT == 128) ? 3 : (NPT == 64 ? 5 : 6));
  static constexpr int TMEM_COLS = 2 * NPT;  // two chunk accumulators
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  static constexpr int SMEM = 1024 + STAGES * STAGE + NUM_BARS * 8 + 16;
  static constexpr uint32_t IDESC = ptx::idesc_bf16_f32(128, NPT);
};

// Four consecutive weights per thread (d % 64 == 0 on this path): one
// 16-byte load, one 8-byte store per plane.
__global__ void __launch_bounds__(256)
router_split_kernel(const float* __restrict__ w_r, int N, int NP, int d,
                    __nv_bfloat16* __restrict__ w3) {
  const size_t total = static_cast<size_t>(NP) * d;
  for (size_t i = (blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x) * 4; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x * 4) {
    const size_t e = i / d;  // the four weights share a row: d % 4 == 0
    const float4 w4 = e < static_cast<size_t>(N) ? __ldg(reinterpret_cast<const float4*>(w_r + i))
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
    const float w[4] = {w4.x, w4.y, w4.z, w4.w};
    uint32_t bits[3][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(w[j]);
      const float r1 = w[j] - __bfloat162float(hi);
      const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
      const float r2 = r1 - __bfloat162float(mid);
      bits[0][j] = __bfloat16_as_ushort(hi);
      bits[1][j] = __bfloat16_as_ushort(mid);
      bits[2][j] = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
    }
#pragma unroll
    for (int q = 0; q < 3; ++q)
      *reinterpret_cast<uint2*>(w3 + q * total + i) =
          make_uint2(bits[q][0] | (bits[q][1] << 16), bits[q][2] | (bits[q][3] << 16));
  }
}

struct GemmArgs {
  int T, NP, KB, kb_per_split;
  float* part;  // [S][T][NP] (unfused)
  uint32_t* status;
  // fused selection (one K split, all experts in one tile)
  int N, K, gate_mode;
  const float* b_r;
  const float* sel_bias;
  int32_t* idx;
  float* gate;
  float* psum;   // [N+2][nblk], nblk = ceil(T/128)
  int32_t* pcnt; // [N][nblk]
  float* logits; // [T][N] kept for the backward pass, or NULL
};

// ---- fused selection in the GEMM epilogue ----------------------------------
// Scratch in the drained stage buffers: p[128][NPT + 1] (the block's softmax
// rows; the odd row pitch keeps both the row writes and the column reads free
// of bank conflicts), zh[2][128] (per-token squared log-sum-exp and entropy),
// cnt[NPT] (assignment counts), bias[NPT] and sbias[NPT] (router and
// selection biases).
template <int NPT>
struct FusedScratch {
  float* p;
  float* zh;
  int32_t* cnt;
  float* bias;   // b_r (0 where absent), read by every token's selection
  float* sbias;  // selection bias (0 where absent)
  __device__ explicit FusedScratch(uint8_t* base)
      : p(reinterpret_cast<float*>(base)),
        zh(p + 128 * (NPT + 1)),
        cnt(reinterpret_cast<int32_t*>(zh + 256)),
        bias(reinterpret_cast<float*>(cnt + NPT)),
        sbias(bias + NPT) {}
  static constexpr int BYTES = (128 * (NPT + 1) + 256 + 3 * NPT) * 4;
};

// One token per thread: v holds the token's NPT accumulated logits (entries
// >= N unused). Top-K first, on the biased selection keys (ties to the lower
// index), then the softmax, whose exponentials overwrite v. Same arithmetic
// as route_one_token, serial instead of across a warp.
__device__ __forceinline__ void epilogue_bar() {  // the 128 epilogue threads
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

template <int NPT>
__device__ __forceinline__ void fused_select(float (&v)[NPT], const GemmArgs& a, int t, int row,
                                             const FusedScratch<NPT>& sc) {
  const int N = a.N, K = a.K;
  float* prow = sc.p + row * (NPT + 1);
  if (t >= a.T) {  // past the last token: contributes nothing
#pragma unroll
    for (int e = 0; e < NPT; ++e) prow[e] = 0.f;
    sc.zh[row] = 0.f;
    sc.zh[128 + row] = 0.f;
    return;
  }
  float mx = -INFINITY;
  bool bad = false;
#pragma unroll
  for (int e = 0; e < NPT; ++e) {
    if (e < N) {
      if (a.b_r != nullptr) v[e] += sc.bias[e];
      if (!isfinite(v[e])) bad = true;
      mx = fmaxf(mx, v[e]);
    }
  }
  if (bad) set_status(a.status, MOE_ERR_NONFINITE);
  if (a.logits != nullptr) {
    float* lrow = a.logits + static_cast<size_t>(t) * N;
#pragma unroll
    for (int e = 0; e < NPT; ++e)
      if (e < N) lrow[e] = v[e];
  }
  // top-K
  uint32_t taken[(NPT + 31) / 32];
#pragma unroll
  for (int i = 0; i < (NPT + 31) / 32; ++i) taken[i] = 0u;
  int sel_e[8];
  float sel_u[8];
  // The rank loop stays rolled (sel_* then live in local memory): unrolled
  // eight times over NPT experts, the epilogue's code outgrows the
  // instruction cache.
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    sel_e[k] = 0;
    sel_u[k] = -INFINITY;
  }
#pragma unroll 1
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY, bu = -INFINITY;
    int be = -1;
#pragma unroll
    for (int e = 0; e < NPT; ++e) {
      if (e >= N || ((taken[e >> 5] >> (e & 31)) & 1u)) continue;
      const float u = isnan(v[e]) ? -INFINITY : v[e];
      const float key = a.sel_bias != nullptr ? u + sc.sbias[e] : u;
      if (be < 0 || key > bv) {
        bv = key;
        be = e;
        bu = v[e];
      }
    }
    if (be < 0) be = 0;  // unreachable while K <= N; keeps indices in range
#pragma unroll
    for (int i = 0; i < (NPT + 31) / 32; ++i)
      if (i == (be >> 5)) taken[i] |= 1u << (be & 31);
    sel_e[k] = be;
    sel_u[k] = bu;
  }
  // softmax over the N experts
  float sum = 0.f, pv = 0.f;
#pragma unroll
  for (int e = 0; e < NPT; ++e) {
    if (e < N) {
      const float ex = expf(v[e] - mx);
      sum += ex;
      if (ex > 0.f) pv += ex * v[e];
      v[e] = ex;
    }
  }
  const float inv = 1.f / sum;
#pragma unroll
  for (int e = 0; e < NPT; ++e) prow[e] = e < N ? v[e] * inv : 0.f;
  const float lse = mx + logf(sum);
  sc.zh[row] = lse * lse;
  sc.zh[128 + row] = lse - pv * inv;
  // gates
  float msel = sel_u[0];
#pragma unroll
  for (int k = 1; k < 8; ++k)
    if (k < K) msel = fmaxf(msel, sel_u[k]);
  float gsum = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if (k < K) gsum += expf(sel_u[k] - msel);
  const size_t t0 = static_cast<size_t>(t) * K;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (k >= K) break;
    a.idx[t0 + k] = sel_e[k];
    a.gate[t0 + k] = a.gate_mode == MOE_GATE_SOFTMAX ? expf(sel_u[k] - mx) * inv
                                                     : expf(sel_u[k] - msel) / gsum;
    atomicAdd(&sc.cnt[sel_e[k]], 1);
  }
}

// The block's partial statistics, in the layout write_block_stats uses
// (psum[e][blk], pcnt[e][blk], psum[N][blk] and psum[N+1][blk]), rows summed
// in ascending order; one column per thread.
template <int NPT>
__device__ __forceinline__ void fused_block_stats(const GemmArgs& a, int m, int row,
                                                  const FusedScratch<NPT>& sc) {
  const size_t nblk = gridDim.x;
  for (int j = row; j < a.N + 2; j += 128) {
    float s = 0.f;
    if (j < a.N) {
      for (int r = 0; r < 128; ++r) s += sc.p[r * (NPT + 1) + j];
      a.pcnt[static_cast<size_t>(j) * nblk + m] = sc.cnt[j];
    } else {
      for (int r = 0; r < 128; ++r) s += sc.zh[(j - a.N) * 128 + r];
    }
    a.psum[static_cast<size_t>(j) * nblk + m] = s;
  }
}

// FUSED: one K split and all experts in one tile, so the thread that owns a
// token's TMEM row holds all of its logits; it then runs softmax, top-K,
// gates and the block's statistics partials itself (the whole router in one
// kernel), using the drained stage buffers as scratch.
template <int NPT, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1)
router_gemm_tc(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
               const GemmArgs args) {
  using namespace ptx;
  using S = Shape<NPT, FUSED>;
  static_assert(!FUSED || FusedScratch<NPT>::BYTES <= S::STAGES * S::STAGE, "scratch");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + S::STAGES * S::STAGE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + S::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x, ntile = blockIdx.y, split = blockIdx.z;
  const int kb0 = split * args.kb_per_split;
  const int kb1 = min(args.KB, kb0 + args.kb_per_split);
  const int nchunks = (kb1 - kb0 + kChunkKb - 1) / kChunkKb;
  auto bar_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return smem_u32(bars + S::STAGES + s); };
  auto bar_tfull = [&](int a) { return smem_u32(bars + 2 * S::STAGES + a); };
  auto bar_tempty = [&](int a) { return smem_u32(bars + 2 * S::STAGES + 2 + a); };
  const uint32_t bar_drain = smem_u32(bars + 2 * S::STAGES + 4);
  auto stage_a = [&](int s) { return base + static_cast<uint32_t>(s * S::STAGE); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::STAGES; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull(a), 1);
      mbar_init(bar_tempty(a), 4);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    tmem_slot[2] = 0;  // epilogue failure flag (FUSED)
    fence_mbar_init();
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), S::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  auto fail = [&]() {
    set_status(args.status, MOE_ERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0 && lane == 0) {
    // ---- TMA producer: x tile + the three weight planes per stage ----
    int stage = 0;
    uint32_t phase = 0, issued = 0, issued_parity = 0;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait(bar_empty(stage), phase ^ 1u, kWaitLimitNs, abort_flag)) {
        fail();
        for (int s = 0; s < S::STAGES; ++s)
          if (issued & (1u << s))
            mbar_wait(bar_full(s), (issued_parity >> s) & 1u, kWaitLimitNs, nullptr);
        break;
      }
      mbar_arrive_expect_tx(bar_full(stage), S::STAGE);
      const uint32_t a = stage_a(stage);
      tma_load_2d(a, &tmX, bar_full(stage), kb * BK, m * BM);
#pragma unroll
      for (int p = 0; p < 3; ++p)
        tma_load_2d(a + A_BYTES + p * S::B_PLANE, &tmW, bar_full(stage), kb * BK,
                    p * args.NP + ntile * NPT);
      issued |= 1u << stage;
      issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == S::STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer: chunks of kChunkKb K steps, alternating accumulators ----
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true, issued_any = false;
    for (int c = 0; c < nchunks && ok; ++c) {
      if (!mbar_wait(bar_tempty(acc), acc_phase ^ 1u, kWaitLimitNs, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * NPT);
      const int cb = kb0 + c * kChunkKb, ce = min(kb1, cb + kChunkKb);
      for (int kb = cb; kb < ce; ++kb) {
        if (!mbar_wait(bar_full(stage), phase, kWaitLimitNs, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a = stage_a(stage);
#pragma unroll
        for (int p = 0; p < 3; ++p)
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16(d_tmem, sdesc_kmajor_sw128(a + kk * 32),
                     sdesc_kmajor_sw128(a + A_BYTES + p * S::B_PLANE + kk * 32), S::IDESC,
                     (kb != cb || p != 0 || kk != 0) ? 1u : 0u);
        issued_any = true;
        mma_commit(bar_empty(stage));
        if (++stage == S::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      mma_commit(bar_tfull(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) {
      fail();
      if (issued_any) {
        mma_commit(bar_drain);
        mbar_wait(bar_drain, 0, kWaitLimitNs, nullptr);
      }
    }
  } else if (warp >= 2) {
    // ---- epilogue: add each finished chunk into fp32 registers ----
    const int q = warp & 3;
    float run[NPT];
#pragma unroll
    for (int j = 0; j < NPT; ++j) run[j] = 0.f;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      ok = mbar_wait(bar_tfull(acc), acc_phase, kWaitLimitNs, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + static_cast<uint32_t>(acc * NPT) +
                             (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll
      for (int cc = 0; cc < NPT / 32; ++cc) {
        uint32_t v[32];
        tmem_ld32(taddr + cc * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) run[cc * 32 + j] += __uint_as_float(v[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) {
      if (lane == 0) fail();
    } else if (!FUSED) {
      const int t = m * BM + q * 32 + lane;
      if (t < args.T) {
        float4* dst = reinterpret_cast<float4*>(
            args.part + (static_cast<size_t>(split) * args.T + static_cast<size_t>(t)) * args.NP +
            ntile * NPT);
#pragma unroll
        for (int j = 0; j < NPT / 4; ++j)
          dst[j] = make_float4(run[4 * j], run[4 * j + 1], run[4 * j + 2], run[4 * j + 3]);
      }
    }
    if (FUSED) {
      // Every epilogue thread passes the same three named barriers whatever
      // happened, so a timeout in one warp leaves no other warp waiting; the
      // selection runs only if all four warps saw every chunk, which also
      // means every MMA has finished reading the stage buffers.
      volatile int* epi_fail = reinterpret_cast<volatile int*>(tmem_slot + 2);
      const FusedScratch<NPT> sc(gbase);
      const int row = q * 32 + lane;
      if (!ok && lane == 0) *epi_fail = 1;
      epilogue_bar();
      const bool all_ok = *epi_fail == 0;
      if (all_ok && row < NPT) {  // staged once here instead of NPT global loads per token
        sc.cnt[row] = 0;
        sc.bias[row] = (args.b_r != nullptr && row < args.N) ? args.b_r[row] : 0.f;
        sc.sbias[row] = (args.sel_bias != nullptr && row < args.N) ? args.sel_bias[row] : 0.f;
      }
      epilogue_bar();
      if (all_ok) fused_select<NPT>(run, args, m * BM + row, row, sc);
      epilogue_bar();
      if (all_ok) fused_block_stats<NPT>(args, m, row, sc);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

// Warp per token: logits = sum over the K splits in order + bias; then the
// shared selection code. One token per warp, 8 per 256-thread block (enough
// blocks to fill the GPU at a few thousand tokens).
template <int NJ>
__global__ void __launch_bounds__(256)
router_topk_kernel(const float* __restrict__ part, int S, int NP, const float* __restrict__ b_r,
                   const float* __restrict__ sel_bias, int gate_mode, int T, int N, int K,
                   int32_t* __restrict__ idx_out, float* __restrict__ gate_out,
                   float* __restrict__ psum, int32_t* __restrict__ pcnt,
                   uint32_t* __restrict__ status, float* __restrict__ logits_out) {
  __shared__ float pw[kSelectWarps][256];
  __shared__ float zh[2 * kSelectWarps];
  __shared__ int32_t scnt[256];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 256; i += blockDim.x) scnt[i] = 0;
  __syncthreads();
  float pacc[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) pacc[j] = 0.f;
  float zacc = 0.f, hacc = 0.f;
  const int t0 = blockIdx.x * kTopkTokensPerBlock;
  for (int tl = warp; tl < kTopkTokensPerBlock; tl += kSelectWarps) {
    const int t = t0 + tl;
    if (t >= T) break;
    float v[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      float acc = -INFINITY;
      if (e < N) {
        acc = 0.f;
        for (int s = 0; s < S; ++s)
          acc += part[(static_cast<size_t>(s) * T + t) * NP + e];
        if (b_r != nullptr) acc += b_r[e];
      }
      v[j] = acc;
    }
    route_one_token<NJ>(v, N, K, static_cast<size_t>(t), lane, sel_bias, gate_mode, idx_out,
                        gate_out, pacc, zacc, hacc, scnt, status, logits_out);
  }
  write_block_stats<NJ>(pacc, zacc, hacc, pw, zh, scnt, N, blockIdx.x, psum, pcnt);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NPT, bool FUSED>
cudaError_t launch_gemm(const CUtensorMap& mx, const CUtensorMap& mw, const GemmArgs& a,
                        dim3 grid, cudaStream_t s) {
  static std::mutex mu;
  static int done_mask = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!(dev < 31 && (done_mask >> dev) & 1)) {
      const cudaError_t e = cudaFuncSetAttribute(
          router_gemm_tc<NPT, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
          Shape<NPT, FUSED>::SMEM);
      if (e != cudaSuccess) return e;
      if (dev < 31) done_mask |= 1 << dev;
    }
  }
  router_gemm_tc<NPT, FUSED><<<grid, kThreads, Shape<NPT, FUSED>::SMEM, s>>>(mx, mw, a);
  return cudaGetLastError();
}

}  // namespace

RouterTcPlan router_tc_plan(const moe_config& c) {
  RouterTcPlan p{};
  p.use = c.dtype == MOE_BF16 && c.d_model % BK == 0 && c.T > 0;
  if (!p.use) return p;
  const int N = c.n_experts;
  p.NP = N <= 32 ? 32 : (N <= 64 ? 64 : (N <= 128 ? 128 : 256));
  p.NPT = p.NP > 128 ? 128 : p.NP;
  const int KB = c.d_model / BK;
  const int tiles = ((c.T + BM - 1) / BM) * (p.NP / p.NPT);
  int S = kTargetCtas / tiles;
  S = S < 1 ? 1 : (S > kMaxSplits ? kMaxSplits : S);
  S = S > KB ? KB : S;
  p.kb_per_split = (KB + S - 1) / S;
  p.S = (KB + p.kb_per_split - 1) / p.kb_per_split;  // no empty split
  // one split and one expert tile: the GEMM epilogue holds whole tokens
  p.fused = p.S == 1 && p.NP == p.NPT;
  p.stat_blocks = p.fused ? (c.T + BM - 1) / BM
                          : (c.T + kTopkTokensPerBlock - 1) / kTopkTokensPerBlock;
  return p;
}

moe_status launch_router_tc(const moe_config& c, const RouterTcPlan& p, const void* x,
                            const float* w_r, const float* b_r, int32_t* idx, float* gate,
                            __nv_bfloat16* w3, float* part, float* psum, int32_t* pcnt,
                            uint32_t* status, float* logits, cudaStream_t s) {
  const int N = c.n_experts, d = c.d_model, T = c.T;
  router_split_kernel<<<sm_count() * 4, 256, 0, s>>>(w_r, N, p.NP, d, w3);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  CUtensorMap mx, mw;
  if (!make_map(&mx, x, static_cast<uint64_t>(T), d, BM) ||
      !make_map(&mw, w3, static_cast<uint64_t>(3) * p.NP, d, p.NPT))
    return MOE_ERR_CUDA;
  GemmArgs a{T, p.NP, d / BK, p.kb_per_split, part, status, N, c.top_k, c.gate_mode, b_r,
             c.select_bias, idx, gate, psum, pcnt, logits};
  const dim3 grid((T + BM - 1) / BM, p.NP / p.NPT, p.S);
  cudaError_t e;
  if (p.fused) {
    if (p.NPT == 128) e = launch_gemm<128, true>(mx, mw, a, grid, s);
    else if (p.NPT == 64) e = launch_gemm<64, true>(mx, mw, a, grid, s);
    else e = launch_gemm<32, true>(mx, mw, a, grid, s);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  if (p.NPT == 128) e = launch_gemm<128, false>(mx, mw, a, grid, s);
  else if (p.NPT == 64) e = launch_gemm<64, false>(mx, mw, a, grid, s);
  else e = launch_gemm<32, false>(mx, mw, a, grid, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  const int nblk = (T + kTopkTokensPerBlock - 1) / kTopkTokensPerBlock;
#define MOE_TOPK(NJ)                                                                           \
  router_topk_kernel<NJ><<<nblk, 256, 0, s>>>(part, p.S, p.NP, b_r, c.select_bias, c.gate_mode, \
                                              T, N, c.top_k, idx, gate, psum, pcnt, status,    \
                                              logits)
  if (N <= 32) MOE_TOPK(1);
  else if (N <= 64) MOE_TOPK(2);
  else if (N <= 128) MOE_TOPK(4);
  else MOE_TOPK(8);
#undef MOE_TOPK
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
