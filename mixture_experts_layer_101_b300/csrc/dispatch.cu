// Capacity-limited dispatch: histogram -> prefix scan -> stable permute and
// gather of the token rows into expert-contiguous order.
//
// Source: "MoE 混合专家模型稀疏激活的架构原理与负载均衡挑战" §2.3 (capacity
// floor(K/N·CF·S); tokens beyond it are dropped and pass on the residual) and
// §三 MoELayer.forward (outer loop over the top-k rank, tokens in ascending
// order within it, truncation of each expert's list at the capacity).
//
// Visiting order q = k*T + t (rank-major). The grid is (token blocks of 256) x
// (K ranks); block (b, k) owns the assignments (t in block b, rank k), which
// are contiguous in q. Rank of an assignment within its expert =
//   base[k][b][e]  (assignments to e in all earlier (k', b') blocks)
// + assignments to e in earlier warps of this block
// + earlier lanes of this warp with the same expert (warp match).
// Every step is integer and order-defined, so slots are bit-exact.
// Shared experts (indices N .. N+S-1) follow the routed slots: shared expert
// s takes every token in order, slots offsets[N] + s*T + t, recorded in
// slot_of[t][K+s].
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kThreads = kDispatchTokensPerBlock;  // 256 = one token per thread

__global__ void __launch_bounds__(kThreads)
dispatch_hist_kernel(const int32_t* __restrict__ idx, int T, int K, int N,
                     int32_t* __restrict__ ghist, uint32_t* status) {
  __shared__ int32_t hist[256];
  const int b = blockIdx.x, k = blockIdx.y, nb = gridDim.x;
  for (int i = threadIdx.x; i < 256; i += kThreads) hist[i] = 0;
  __syncthreads();
  const int t = b * kThreads + threadIdx.x;
  if (t < T) {
    const int e = idx[static_cast<size_t>(t) * K + k];
    if (e >= 0 && e < N) atomicAdd(&hist[e], 1);
    else set_status(status, MOE_ERR_INDEX);
  }
  __syncthreads();
  int32_t* out = ghist + (static_cast<size_t>(k) * nb + b) * N;
  for (int e = threadIdx.x; e < N; e += kThreads) out[e] = hist[e];
}

// One block. Thread (g, e) = (tid / N, tid % N) owns the g-th of
// G = kScanThreads / N runs of consecutive (k, b) blocks in expert e's
// column: it sums its run, then writes the column's exclusive prefix over
// its run starting from the totals of the runs before it (all integer, so
// the result does not depend on the split). Warp 0 then scans the kept
// counts over the experts.
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads)
dispatch_scan_kernel(const int32_t* __restrict__ ghist, int nq, int N, int32_t C, int S, int T,
                     int32_t* __restrict__ gbase, int32_t* __restrict__ offsets,
                     int32_t* count, int32_t* kept_out, int32_t* n_dropped,
                     int32_t* sched_zero) {
  __shared__ int32_t run_sum[kScanThreads];
  __shared__ int32_t kept[256], cnt[256];
  const int tid = threadIdx.x;
  const int G = kScanThreads / N;  // N <= 256, so G >= 4
  const int g = tid / N, e = tid - g * N;
  const bool active = g < G;
  const int per = (nq + G - 1) / G;
  const int q0 = min(nq, g * per), q1 = min(nq, q0 + per);
  int32_t sum = 0;
  if (active)
    for (int q = q0; q < q1; ++q) sum += ghist[static_cast<size_t>(q) * N + e];
  run_sum[tid] = sum;
  __syncthreads();
  if (active) {
    int32_t run = 0;
    for (int h = 0; h < g; ++h) run += run_sum[h * N + e];
    for (int q = q0; q < q1; ++q) {
      gbase[static_cast<size_t>(q) * N + e] = run;
      run += ghist[static_cast<size_t>(q) * N + e];
    }
    if (g == G - 1) {  // the last run ends the column: run is the expert's total
      cnt[e] = run;
      kept[e] = run < C ? run : C;
      if (count) count[e] = run;
      if (kept_out) kept_out[e] = kept[e];
    }
  }
  __syncthreads();
  if (tid < 32) {
    const int per_lane = (N + 31) / 32;
    const int e0 = min(N, tid * per_lane), e1 = min(N, e0 + per_lane);
    int32_t ks = 0, ds = 0;
    for (int i = e0; i < e1; ++i) {
      ks += kept[i];
      ds += cnt[i] - kept[i];
    }
    int32_t inc = ks;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, inc, o);
      if (tid >= o) inc += v;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ds += __shfl_xor_sync(0xffffffffu, ds, o);
    int32_t off = inc - ks;
    for (int i = e0; i < e1; ++i) {
      offsets[i] = off;
      off += kept[i];
    }
    const int32_t total = __shfl_sync(0xffffffffu, inc, 31);
    if (tid == 0) {
      if (sched_zero) sched_zero[0] = sched_zero[1] = 0;  // the expert GEMMs' tile counters
      offsets[N] = total;
      for (int s2 = 0; s2 < S; ++s2) offsets[N + s2 + 1] = total + (s2 + 1) * T;  // shared experts
      if (n_dropped) *n_dropped = ds;
    }
  }
}

__global__ void __launch_bounds__(kThreads)
dispatch_permute_kernel(const int32_t* __restrict__ idx, int T, int K, int N, int S, int32_t C,
                        const int32_t* __restrict__ gbase, const int32_t* __restrict__ offsets,
                        int32_t* __restrict__ slot_of, int32_t* __restrict__ token_of_slot) {
  __shared__ int32_t wcnt[kThreads / 32][256];
  const int b = blockIdx.x, k = blockIdx.y, nb = gridDim.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < (kThreads / 32) * 256; i += kThreads) (&wcnt[0][0])[i] = 0;

  const int t = b * kThreads + tid;
  int e = -1;
  if (t < T) e = idx[static_cast<size_t>(t) * K + k];
  const bool valid = (t < T) && e >= 0 && e < N;
  // peers: lanes of this warp routed to the same expert (unique keys otherwise)
  const int key = valid ? e : N + lane;
  const uint32_t peers = __match_any_sync(0xffffffffu, key);
  const uint32_t lower = peers & ((1u << lane) - 1u);
  const int rank_w = __popc(lower);
  __syncthreads();
  if (valid && rank_w == 0) wcnt[warp][e] = __popc(peers);
  __syncthreads();

  const int KS = K + S;  // slot_of row: K routed ranks, then the shared experts
  int32_t slot = -1;
  if (valid) {
    int32_t rank = gbase[(static_cast<size_t>(k) * nb + b) * N + e] + rank_w;
    for (int w = 0; w < warp; ++w) rank += wcnt[w][e];
    if (rank < C) {
      slot = offsets[e] + rank;
      token_of_slot[slot] = t;
    }
  }
  if (t < T) {
    slot_of[static_cast<size_t>(t) * KS + k] = slot;
    if (k == 0)
      for (int s2 = 0; s2 < S; ++s2)
        slot_of[static_cast<size_t>(t) * KS + K + s2] = offsets[N] + s2 * T + t;
  }
}

// Batches of at most 256 tokens (one token block): histogram, capacity scan
// and permute in one block of 256 threads, one token per thread, with the
// multi-block kernels' arithmetic: pass 1 counts each expert's assignments
// over all ranks; warp 0 scans the kept counts into the offsets; pass 2 walks
// the ranks k = 0 .. K-1 in order, where an assignment's rank within its
// expert is the expert's count over the earlier ranks, plus the earlier warps'
// counts at this rank, plus the earlier lanes of its warp with the same expert
// (warp match). Same slots, bit for bit, in one launch instead of three.
__global__ void __launch_bounds__(kThreads)
dispatch_small_kernel(const int32_t* __restrict__ idx, int T, int K, int N, int S, int32_t C,
                      int32_t* __restrict__ offsets, int32_t* __restrict__ slot_of,
                      int32_t* __restrict__ token_of_slot, int32_t* count, int32_t* kept_out,
                      int32_t* n_dropped, int32_t* sched_zero, uint32_t* status) {
  __shared__ int32_t tot[256], kept[256], off[256], base[256];
  __shared__ int32_t wcnt[kThreads / 32][256];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = tid;
  tot[tid] = 0;
  base[tid] = 0;
  __syncthreads();
  for (int k = 0; k < K; ++k) {
    if (t < T) {
      const int e = idx[static_cast<size_t>(t) * K + k];
      if (e >= 0 && e < N) atomicAdd(&tot[e], 1);
      else set_status(status, MOE_ERR_INDEX);
    }
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the kept counts over the experts
    const int per_lane = (N + 31) / 32;
    const int e0 = min(N, lane * per_lane), e1 = min(N, e0 + per_lane);
    int32_t ks = 0, ds = 0;
    for (int e = e0; e < e1; ++e) {
      const int32_t kp = tot[e] < C ? tot[e] : C;
      kept[e] = kp;
      ks += kp;
      ds += tot[e] - kp;
    }
    int32_t inc = ks;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ds += __shfl_xor_sync(0xffffffffu, ds, o);
    int32_t run = inc - ks;
    for (int e = e0; e < e1; ++e) {
      off[e] = run;
      offsets[e] = run;
      run += kept[e];
    }
    const int32_t total = __shfl_sync(0xffffffffu, inc, 31);
    if (lane == 0) {
      if (sched_zero) sched_zero[0] = sched_zero[1] = 0;  // the expert GEMMs' tile counters
      offsets[N] = total;
      for (int s2 = 0; s2 < S; ++s2) offsets[N + s2 + 1] = total + (s2 + 1) * T;
      if (n_dropped) *n_dropped = ds;
    }
  }
  for (int e = tid; e < N; e += kThreads) {
    if (count) count[e] = tot[e];
    if (kept_out) kept_out[e] = tot[e] < C ? tot[e] : C;
  }
  __syncthreads();
  const int KS = K + S;
  for (int k = 0; k < K; ++k) {
    for (int i = tid; i < (kThreads / 32) * 256; i += kThreads) (&wcnt[0][0])[i] = 0;
    int e = -1;
    if (t < T) e = idx[static_cast<size_t>(t) * K + k];
    const bool valid = (t < T) && e >= 0 && e < N;
    const int key = valid ? e : N + lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    const int rank_w = __popc(peers & ((1u << lane) - 1u));
    __syncthreads();
    if (valid && rank_w == 0) wcnt[warp][e] = __popc(peers);
    __syncthreads();
    int32_t slot = -1;
    if (valid) {
      int32_t rank = base[e] + rank_w;
      for (int w = 0; w < warp; ++w) rank += wcnt[w][e];
      if (rank < C) {
        slot = off[e] + rank;
        token_of_slot[slot] = t;
      }
    }
    if (t < T) slot_of[static_cast<size_t>(t) * KS + k] = slot;
    __syncthreads();
    for (int e2 = tid; e2 < N; e2 += kThreads) {
      int32_t add = 0;
      for (int w = 0; w < kThreads / 32; ++w) add += wcnt[w][e2];
      base[e2] += add;
    }
    __syncthreads();
  }
  if (t < T) {
    const int32_t routed = offsets[N];
    for (int s2 = 0; s2 < S; ++s2)
      slot_of[static_cast<size_t>(t) * KS + K + s2] = routed + s2 * T + t;
  }
}

// x_perm[s] = x[token_of_slot[s]] for s < offsets[N]: one warp per slot and
// column slice (blockIdx.y of gridDim.y: one slice unless the batch is small),
// 16 bytes per lane per step, four steps in flight.
template <typename Tx>
__global__ void __launch_bounds__(256)
dispatch_gather_kernel(const Tx* __restrict__ x, const int32_t* __restrict__ token_of_slot,
                       const int32_t* __restrict__ offsets, int N, int S, int T, int d,
                       Tx* __restrict__ x_perm) {
  const int routed = offsets[N];
  const int slot = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (slot >= routed + S * T) return;
  const int lane = threadIdx.x & 31;
  // routed slots come from the permutation; shared slots hold the tokens in order
  const int t = slot < routed ? token_of_slot[slot] : (slot - routed) % T;
  const int all = d * static_cast<int>(sizeof(Tx)) / 16;
  const int per = (all + gridDim.y - 1) / gridDim.y;
  const int c0 = min(all, static_cast<int>(blockIdx.y) * per);
  const int chunks = min(all, c0 + per) - c0;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d) + c0;
  uint4* dst = reinterpret_cast<uint4*>(x_perm + static_cast<size_t>(slot) * d) + c0;
  int c = lane;
  for (; c + 96 < chunks; c += 128) {
    const uint4 a = __ldg(src + c), b = __ldg(src + c + 32), e = __ldg(src + c + 64),
                f = __ldg(src + c + 96);
    dst[c] = a;
    dst[c + 32] = b;
    dst[c + 64] = e;
    dst[c + 96] = f;
  }
  for (; c < chunks; c += 32) dst[c] = __ldg(src + c);
}

}  // namespace

moe_status launch_dispatch(const moe_config& c, const void* x, const int32_t* idx,
                           int32_t* offsets, int32_t* slot_of, int32_t* token_of_slot,
                           void* x_perm, int32_t* ghist, int32_t* gbase, const moe_stats* st,
                           cudaStream_t s, int32_t* sched_zero) {
  const int N = c.n_experts, K = c.top_k;
  const int32_t C = capacity_of(&c);
  uint32_t* status = st ? st->status : nullptr;
  const int nb = (c.T + kThreads - 1) / kThreads;
  if (nb == 1) {
    dispatch_small_kernel<<<1, kThreads, 0, s>>>(
        idx, c.T, K, N, c.n_shared, C, offsets, slot_of, token_of_slot, st ? st->count : nullptr,
        st ? st->kept : nullptr, st ? st->n_dropped : nullptr, sched_zero, status);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  } else {
    if (c.T > 0) {
      dispatch_hist_kernel<<<dim3(nb, K), kThreads, 0, s>>>(idx, c.T, K, N, ghist, status);
      if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    }
    dispatch_scan_kernel<<<1, kScanThreads, 0, s>>>(
        ghist, c.T > 0 ? K * nb : 0, N, C, c.n_shared, c.T, gbase, offsets,
        st ? st->count : nullptr, st ? st->kept : nullptr, st ? st->n_dropped : nullptr,
        sched_zero);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    if (c.T > 0) {
      dispatch_permute_kernel<<<dim3(nb, K), kThreads, 0, s>>>(
          idx, c.T, K, N, c.n_shared, C, gbase, offsets, slot_of, token_of_slot);
      if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    }
  }
  if (c.T > 0) {
    const int64_t rows = rows_max_of(&c);
    // few rows (decode): split each row's columns over blockIdx.y, 4 KB a slice
    const int row_bytes = c.d_model * (c.dtype == MOE_BF16 ? 2 : 4);
    const unsigned slices =
        rows < 2 * sm_count() ? static_cast<unsigned>((row_bytes + 4095) / 4096) : 1u;
    const dim3 gblocks(static_cast<unsigned>((rows + 7) / 8), slices);
    if (rows > 0) {
      if (c.dtype == MOE_BF16)
        dispatch_gather_kernel<__nv_bfloat16><<<gblocks, 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(x), token_of_slot, offsets, N, c.n_shared, c.T,
            c.d_model, static_cast<__nv_bfloat16*>(x_perm));
      else
        dispatch_gather_kernel<float><<<gblocks, 256, 0, s>>>(
            static_cast<const float*>(x), token_of_slot, offsets, N, c.n_shared, c.T, c.d_model,
            static_cast<float*>(x_perm));
      if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    }
  }
  return MOE_OK;
}

}  // namespace moe
