// Expert-parallel (EP) staging: the local data movement around the two
// all-to-alls of an expert-parallel MoE layer. No exchange happens here; the
// caller moves the packed buffers between devices with its own collective.
//
// Source: "MoE 的核心思想", Expert Parallelism (专家并行) and 前向传播中的
// All-to-All 通信: the experts are spread over devices; in the dispatch step
// each device sends its tokens to the devices holding their experts, each
// device runs its own experts on what it received, and in the combine step
// the outputs go back to the source devices for the gate-weighted sum.
//
// Layouts (rows of d elements; every permutation is integer and exact):
//   source device, after moe_dispatch: x_perm, expert e at rows
//     [offsets[e], offsets[e+1]).
//   send buffer (moe_ep_pack): destination r ascending, then r's experts
//     ascending, then each expert's rows in slot order; send_counts[r] rows
//     go to r. The slot s of expert e sits at base[e] + (s - offsets[e]).
//   receive buffer of device r (the all-to-all's order): source s ascending,
//     each source's rows of r's experts in the order s sent them.
//   local rows of device r (moe_ep_regroup): r's experts ascending (local
//     index j), then sources ascending; local_offsets[j] is expert j's first
//     row. Local row p of (j, s) comes from receive row
//     rstart[j][s] + (p - lstart[j][s]).
// moe_ep_unpack and moe_ep_regroup_back are the inverse permutations, on the
// fp32 expert outputs.
//
// Each call is two launches: a one-block plan kernel (position tables in the
// caller's workspace, argument checks that need device data) and a row
// kernel, one warp per row, 16-byte vectors, that does nothing when the plan
// found an error.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kPlanThreads = 256;   // >= N (N <= 256) and >= R (R <= 256)
constexpr int kMaxRanks = 256;

struct EpWs {
  size_t ok, base, loff, lstart, rstart, total;
};

EpWs ep_ws_layout(int N, int R) {
  auto a256 = [](size_t b) { return (b + 255) & ~size_t(255); };
  EpWs L{};
  size_t t = 0;
  L.ok = t;      t += a256(4);
  L.base = t;    t += a256(static_cast<size_t>(N) * 4);
  L.loff = t;    t += a256(static_cast<size_t>(N + 1) * 4);
  L.lstart = t;  t += a256(static_cast<size_t>(N) * R * 4);
  L.rstart = t;  t += a256(static_cast<size_t>(N) * R * 4);
  L.total = t;
  return L;
}

// Source plan: send_counts[r] = rows of r's experts; base[e] = send position
// of expert e's first slot. ok = 0 (and MOE_ERR_INDEX) if an owner is out of
// range or the offsets are not those of a dispatch (offsets[0] = 0,
// non-decreasing, offsets[N] <= a_max): then no row is moved.
__global__ void __launch_bounds__(kPlanThreads)
ep_source_plan_kernel(const int32_t* __restrict__ owner, const int32_t* __restrict__ offsets,
                      int N, int R, int64_t a_max, int32_t* __restrict__ base,
                      int32_t* __restrict__ send_counts, int32_t* __restrict__ ok,
                      uint32_t* status) {
  __shared__ int32_t own[256], kept[256], cnt[kMaxRanks], displ[kMaxRanks];
  __shared__ int bad;
  const int tid = threadIdx.x;
  if (tid == 0) bad = (offsets[0] != 0 || offsets[N] > a_max) ? 1 : 0;
  __syncthreads();
  if (tid < N) {
    own[tid] = owner[tid];
    const int64_t k = static_cast<int64_t>(offsets[tid + 1]) - offsets[tid];
    kept[tid] = static_cast<int32_t>(k);
    if (own[tid] < 0 || own[tid] >= R || k < 0) bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      *ok = 0;
      set_status(status, MOE_ERR_INDEX);
    }
    return;
  }
  if (tid < R) {  // rows for destination tid
    int32_t c = 0;
    for (int e = 0; e < N; ++e) c += own[e] == tid ? kept[e] : 0;
    cnt[tid] = c;
  }
  __syncthreads();
  if (tid == 0) {
    int32_t run = 0;
    for (int r = 0; r < R; ++r) {
      displ[r] = run;
      run += cnt[r];
    }
    *ok = 1;
  }
  __syncthreads();
  if (tid < R && send_counts) send_counts[tid] = cnt[tid];
  if (tid < N) {  // earlier experts of the same destination come first
    const int r = own[tid];
    int32_t b = displ[r];
    for (int e = 0; e < tid; ++e) b += own[e] == r ? kept[e] : 0;
    base[tid] = b;
  }
}

// Destination plan of device `rank`. kept_all [R][N]: kept rows of expert e
// on source s. Local experts j (owner == rank, ascending) get loff[j] (and
// loff[E_r..N] = the total rows), lstart[j][s] and rstart[j][s] as described
// above. ok = 0 with MOE_ERR_INDEX (owner out of range or a negative count)
// or MOE_ERR_WORKSPACE (more rows than rows_cap).
__global__ void __launch_bounds__(kPlanThreads)
ep_dest_plan_kernel(const int32_t* __restrict__ owner, const int32_t* __restrict__ kept_all,
                    int N, int R, int rank, int64_t rows_cap, int32_t* __restrict__ loff,
                    int32_t* __restrict__ lstart, int32_t* __restrict__ rstart,
                    int32_t* __restrict__ ok, uint32_t* status) {
  __shared__ int32_t own[256], local_e[256], lofs[257], rdispl[kMaxRanks];
  __shared__ int64_t lcnt[256];
  __shared__ int bad, n_local, fits_s;
  const int tid = threadIdx.x;
  if (tid == 0) bad = 0;
  __syncthreads();
  if (tid < N) {
    own[tid] = owner[tid];
    if (own[tid] < 0 || own[tid] >= R) bad = 1;
  }
  for (int i = tid; i < R * N; i += blockDim.x)
    if (kept_all[i] < 0) bad = 1;
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      *ok = 0;
      set_status(status, MOE_ERR_INDEX);
    }
    return;
  }
  if (tid < N && own[tid] == rank) {  // local index of expert tid
    int j = 0;
    for (int e = 0; e < tid; ++e) j += own[e] == rank;
    local_e[j] = tid;
  }
  if (tid == 0) {
    int c = 0;
    for (int e = 0; e < N; ++e) c += own[e] == rank;
    n_local = c;
  }
  __syncthreads();
  const int E = n_local;
  if (tid < E) {  // rows of local expert tid over all sources; its starts per source
    const int e = local_e[tid];
    int64_t c = 0;
    for (int s = 0; s < R; ++s) c += kept_all[static_cast<size_t>(s) * N + e];
    lcnt[tid] = c;
  }
  __syncthreads();
  if (tid == 0) {
    int64_t run = 0;
    for (int j = 0; j < E; ++j) {
      lofs[j] = static_cast<int32_t>(run);
      run += lcnt[j];
    }
    const bool fits = run <= rows_cap;
    if (!fits)
      for (int j = 0; j < E; ++j) lofs[j] = 0;
    lofs[E] = fits ? static_cast<int32_t>(run) : 0;
    fits_s = fits ? 1 : 0;
    *ok = fits ? 1 : 0;
    if (!fits) set_status(status, MOE_ERR_WORKSPACE);
  }
  __syncthreads();
  for (int j = tid; j <= N; j += blockDim.x) loff[j] = lofs[j < E ? j : E];
  if (!fits_s) return;  // too many rows: the tables are not needed
  // the total fits in int32 from here on, and every partial sum below is
  // bounded by it
  if (tid < E) {
    const int e = local_e[tid];
    int32_t run = lofs[tid];
    for (int s = 0; s < R; ++s) {
      lstart[static_cast<size_t>(tid) * R + s] = run;
      run += kept_all[static_cast<size_t>(s) * N + e];
    }
  }
  if (tid < R) {  // rows source tid sends to this device
    int32_t c = 0;
    for (int j = 0; j < E; ++j) c += kept_all[static_cast<size_t>(tid) * N + local_e[j]];
    rdispl[tid] = c;
  }
  __syncthreads();
  if (tid == 0) {
    int32_t run = 0;
    for (int s = 0; s < R; ++s) {
      const int32_t c = rdispl[s];
      rdispl[s] = run;
      run += c;
    }
  }
  __syncthreads();
  if (tid < R) {
    int32_t run = rdispl[tid];
    for (int j = 0; j < E; ++j) {
      rstart[static_cast<size_t>(j) * R + tid] = run;
      run += kept_all[static_cast<size_t>(tid) * N + local_e[j]];
    }
  }
}

// One row of `chunks` 16-byte vectors, warp-wide, four loads in flight.
__device__ __forceinline__ void copy_row(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                         int chunks, int lane) {
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

// Slot s of the source device <-> its send position. INVERSE = 0 (pack):
// dst[pos] = src[s]; 1 (unpack): dst[s] = src[pos]. Warp per slot.
template <int INVERSE>
__global__ void __launch_bounds__(256)
ep_source_rows_kernel(const int32_t* __restrict__ offsets, const int32_t* __restrict__ base,
                      const int32_t* __restrict__ ok, int N, int chunks,
                      const uint4* __restrict__ src, uint4* __restrict__ dst) {
  __shared__ int32_t offs[257], bs[256];
  for (int i = threadIdx.x; i <= N; i += blockDim.x) {
    offs[i] = offsets[i];
    if (i < N) bs[i] = base[i];
  }
  __syncthreads();
  if (*ok == 0) return;
  const int s = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (s >= offs[N]) return;
  int lo = 0, hi = N - 1;  // the last expert whose first slot is <= s
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (offs[mid] <= s) lo = mid;
    else hi = mid - 1;
  }
  const int64_t pos = bs[lo] + (s - offs[lo]);
  const int64_t from = INVERSE ? pos : s, to = INVERSE ? s : pos;
  copy_row(src + from * chunks, dst + to * chunks, chunks, threadIdx.x & 31);
}

// Local row p of the destination device <-> its receive row. INVERSE = 0
// (regroup): dst[p] = src[q]; 1 (regroup back): dst[q] = src[p].
template <int INVERSE>
__global__ void __launch_bounds__(256)
ep_dest_rows_kernel(const int32_t* __restrict__ loff, const int32_t* __restrict__ lstart,
                    const int32_t* __restrict__ rstart, const int32_t* __restrict__ ok, int N,
                    int R, int chunks, const uint4* __restrict__ src, uint4* __restrict__ dst) {
  __shared__ int32_t lo_s[257];
  for (int i = threadIdx.x; i <= N; i += blockDim.x) lo_s[i] = loff[i];
  __syncthreads();
  if (*ok == 0) return;
  const int p = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (p >= lo_s[N]) return;
  int lo = 0, hi = N - 1;  // local expert: the last j with loff[j] <= p (and rows)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (lo_s[mid] <= p) lo = mid;
    else hi = mid - 1;
  }
  const int j = lo;
  const int32_t* ls = lstart + static_cast<size_t>(j) * R;
  int a = 0, b = R - 1;  // source: the last s with lstart[j][s] <= p
  while (a < b) {
    const int mid = (a + b + 1) >> 1;
    if (__ldg(ls + mid) <= p) a = mid;
    else b = mid - 1;
  }
  const int64_t q = __ldg(rstart + static_cast<size_t>(j) * R + a) + (p - __ldg(ls + a));
  const int64_t from = INVERSE ? p : q, to = INVERSE ? q : p;
  copy_row(src + from * chunks, dst + to * chunks, chunks, threadIdx.x & 31);
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status ep_check(const moe_config* c, int R, const void* ws) {
  moe_status why = MOE_OK;
  if (!config_valid(c, &why)) return why;
  if (R < 1) return MOE_ERR_INVALID;
  if (R > kMaxRanks || c->n_shared != 0) return MOE_ERR_UNSUPPORTED;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

uint8_t* at(void* ws, size_t off) { return static_cast<uint8_t*>(ws) + off; }

moe_status source_rows(const moe_config* c, int R, const int32_t* owner, const int32_t* offsets,
                       const void* src, void* dst, int row_bytes, int32_t* send_counts,
                       moe_stats* st, void* ws, cudaStream_t s, bool inverse) {
  const int N = c->n_experts;
  const EpWs L = ep_ws_layout(N, R);
  int32_t* ok = reinterpret_cast<int32_t*>(at(ws, L.ok));
  int32_t* base = reinterpret_cast<int32_t*>(at(ws, L.base));
  const int64_t rows = a_max_of(c);  // the plan checks offsets[N] <= A_max
  ep_source_plan_kernel<<<1, kPlanThreads, 0, s>>>(owner, offsets, N, R, rows, base, send_counts,
                                                   ok, st ? st->status : nullptr);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  if (rows == 0) return MOE_OK;
  const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
  const int chunks = row_bytes / 16;
  if (inverse)
    ep_source_rows_kernel<1><<<blocks, 256, 0, s>>>(offsets, base, ok, N, chunks,
                                                    static_cast<const uint4*>(src),
                                                    static_cast<uint4*>(dst));
  else
    ep_source_rows_kernel<0><<<blocks, 256, 0, s>>>(offsets, base, ok, N, chunks,
                                                    static_cast<const uint4*>(src),
                                                    static_cast<uint4*>(dst));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status dest_rows(const moe_config* c, int R, int rank, const int32_t* owner,
                     const int32_t* kept_all, int64_t rows_cap, const void* src, void* dst,
                     int row_bytes, int32_t* local_offsets, moe_stats* st, void* ws,
                     cudaStream_t s, bool inverse) {
  const int N = c->n_experts;
  const EpWs L = ep_ws_layout(N, R);
  int32_t* ok = reinterpret_cast<int32_t*>(at(ws, L.ok));
  int32_t* loff = local_offsets ? local_offsets : reinterpret_cast<int32_t*>(at(ws, L.loff));
  int32_t* lstart = reinterpret_cast<int32_t*>(at(ws, L.lstart));
  int32_t* rstart = reinterpret_cast<int32_t*>(at(ws, L.rstart));
  ep_dest_plan_kernel<<<1, kPlanThreads, 0, s>>>(owner, kept_all, N, R, rank, rows_cap, loff,
                                                 lstart, rstart, ok, st ? st->status : nullptr);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  if (rows_cap == 0) return MOE_OK;
  const unsigned blocks = static_cast<unsigned>((rows_cap + 7) / 8);
  const int chunks = row_bytes / 16;
  if (inverse)
    ep_dest_rows_kernel<1><<<blocks, 256, 0, s>>>(loff, lstart, rstart, ok, N, R, chunks,
                                                  static_cast<const uint4*>(src),
                                                  static_cast<uint4*>(dst));
  else
    ep_dest_rows_kernel<0><<<blocks, 256, 0, s>>>(loff, lstart, rstart, ok, N, R, chunks,
                                                  static_cast<const uint4*>(src),
                                                  static_cast<uint4*>(dst));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int dtype_bytes(const moe_config* c) { return c->dtype == MOE_BF16 ? 2 : 4; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_ep_workspace_size(const moe_config* cfg, int32_t n_ranks) {
  if (!config_valid(cfg, nullptr) || n_ranks < 1 || n_ranks > kMaxRanks) return 0;
  return ep_ws_layout(cfg->n_experts, n_ranks).total;
}

moe_status moe_ep_pack(const moe_config* cfg, int32_t n_ranks, const int32_t* owner,
                       const int32_t* offsets, const void* x_perm, void* send,
                       int32_t* send_counts, moe_stats* stats, void* ws, moe_stream_t stream) {
  try {
    if (moe_status r = ep_check(cfg, n_ranks, ws)) return r;
    if (!owner || !offsets || !send_counts || (cfg->T > 0 && (!x_perm || !send)))
      return MOE_ERR_INVALID;
    if (!a16(owner) || !a16(offsets) || !a16(send_counts) || !a16(x_perm) || !a16(send))
      return MOE_ERR_INVALID;
    return source_rows(cfg, n_ranks, owner, offsets, x_perm, send,
                       cfg->d_model * dtype_bytes(cfg), send_counts, stats, ws,
                       static_cast<cudaStream_t>(stream), false);
  } catch (...) {
    return MOE_ERR_CUDA;
  }
}

moe_status moe_ep_unpack(const moe_config* cfg, int32_t n_ranks, const int32_t* owner,
                         const int32_t* offsets, const float* back, float* o, moe_stats* stats,
                         void* ws, moe_stream_t stream) {
  try {
    if (moe_status r = ep_check(cfg, n_ranks, ws)) return r;
    if (!owner || !offsets || (cfg->T > 0 && (!back || !o))) return MOE_ERR_INVALID;
    if (!a16(owner) || !a16(offsets) || !a16(back) || !a16(o)) return MOE_ERR_INVALID;
    return source_rows(cfg, n_ranks, owner, offsets, back, o, cfg->d_model * 4, nullptr, stats,
                       ws, static_cast<cudaStream_t>(stream), true);
  } catch (...) {
    return MOE_ERR_CUDA;
  }
}

moe_status moe_ep_regroup(const moe_config* cfg, int32_t n_ranks, int32_t rank,
                          const int32_t* owner, const int32_t* kept_all, int64_t rows_cap,
                          const void* recv, void* x_local, int32_t* local_offsets,
                          moe_stats* stats, void* ws, moe_stream_t stream) {
  try {
    if (moe_status r = ep_check(cfg, n_ranks, ws)) return r;
    if (rank < 0 || rank >= n_ranks || rows_cap < 0 || rows_cap > INT32_MAX)
      return MOE_ERR_INVALID;
    if (!owner || !kept_all || !local_offsets || (rows_cap > 0 && (!recv || !x_local)))
      return MOE_ERR_INVALID;
    if (!a16(owner) || !a16(kept_all) || !a16(local_offsets) || !a16(recv) || !a16(x_local))
      return MOE_ERR_INVALID;
    return dest_rows(cfg, n_ranks, rank, owner, kept_all, rows_cap, recv, x_local,
                     cfg->d_model * dtype_bytes(cfg), local_offsets, stats, ws,
                     static_cast<cudaStream_t>(stream), false);
  } catch (...) {
    return MOE_ERR_CUDA;
  }
}

moe_status moe_ep_regroup_back(const moe_config* cfg, int32_t n_ranks, int32_t rank,
                               const int32_t* owner, const int32_t* kept_all, int64_t rows_cap,
                               const float* o_local, float* back, moe_stats* stats, void* ws,
                               moe_stream_t stream) {
  try {
    if (moe_status r = ep_check(cfg, n_ranks, ws)) return r;
    if (rank < 0 || rank >= n_ranks || rows_cap < 0 || rows_cap > INT32_MAX)
      return MOE_ERR_INVALID;
    if (!owner || !kept_all || (rows_cap > 0 && (!o_local || !back))) return MOE_ERR_INVALID;
    if (!a16(owner) || !a16(kept_all) || !a16(o_local) || !a16(back)) return MOE_ERR_INVALID;
    return dest_rows(cfg, n_ranks, rank, owner, kept_all, rows_cap, o_local, back,
                     cfg->d_model * 4, nullptr, stats, ws, static_cast<cudaStream_t>(stream),
                     true);
  } catch (...) {
    return MOE_ERR_CUDA;
  }
}

}  // extern "C"
