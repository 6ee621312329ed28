// Grouped expert FFN on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// Sources: "MoE 混合专家模型稀疏激活的架构原理与负载均衡挑战" §三 class Expert
// (down(silu(gate(x)) * up(x))) and its note in MoELayer.forward that the
// per-expert loop should become a grouped matrix multiply in production.
//
// Two launches of one persistent, warp-specialised kernel:
//   gate/up:  h[s, n] = silu(x_perm[s] . W_gate[e, n]) * (x_perm[s] . W_up[e, n])
//             output tile 128 rows x 128 columns of h; the MMA's B operand is
//             128 rows of W_gate followed by the same 128 rows of W_up, so one
//             M=128, N=256 MMA produces both halves side by side in TMEM and
//             the SwiGLU is applied in the epilogue (h rounded to bf16 once).
//   down:     o[s, n] = h[s] . W_down[e, n], tile 128 x 256, fp32 output.
// The rows s of expert e are the contiguous slots [offsets[e], offsets[e+1])
// written by the dispatch; a 128-row tile may run past its expert's last
// slot: those rows are computed from whatever follows and never stored (rows
// of D depend only on the same rows of A).
//
// Per CTA (one per SM, 192 threads):
//   warp 0      TMA producer: A and B tiles (128-byte swizzle, 64 bf16 of K
//               per row) into a 4-stage shared-memory ring;
//   warp 1      allocates 512 TMEM columns and issues tcgen05.mma (M=128,
//               N=256, K=16; four per 64-wide stage) into one of two fp32
//               accumulators (256 columns each), committing each stage back
//               to the producer and each finished tile to the epilogue;
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter, activation,
//               stores; the second accumulator lets tile i's epilogue overlap
//               tile i+1's main loop.
// Tiles are (expert, n-tile, m-tile) with m fastest, dealt round-robin over
// the CTAs, so CTAs running at the same time share weight tiles through L2.
// Every wait is bounded (1 s of wall time); on expiry the block records
// MOE_ERR_TIMEOUT in the status word, lets its copies and MMAs drain,
// frees its TMEM and returns.
#include "moe_common.cuh"
#include "ptx_sm100.cuh"

#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

namespace moe {
namespace {

constexpr int BM = 128, BK = 64, kThreads = 192;
constexpr int A_BYTES = BM * BK * 2;    // 16 KB
constexpr int ACC_COLS = 256;           // fp32 accumulator 128 x 256 (CTA-pair kernel)
constexpr int MAX_EXPERTS = 264;  // 256 routed + 8 shared

// Tile shape of the one-CTA kernel. MODE 0 (gate/up): BNH output columns of
// h per tile, i.e. BNH gate rows + BNH up rows of weights, MMA N = 2*BNH.
// MODE 1 (down): BNH = 128, MMA N = 256 output columns. (Narrower gate/up
// tiles, tried for small batches to even out the last wave, measured slower:
// with 8 KB of weights per stage the single producer thread cannot keep the
// loads in flight.)
template <int MODE, int BNH>
struct TcShape {
  static constexpr int BN = 2 * BNH;                    // MMA N
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (196608 / STAGE_BYTES) > 8 ? 8 : (196608 / STAGE_BYTES);
  static constexpr int ACC = BN;                        // TMEM columns per accumulator
  static constexpr int TMEM_COLS = 2 * BN;              // two accumulators
  static constexpr int NUM_BARS = 2 * STAGES + 5;       // full, empty, tfull[2], tempty[2], drain
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + NUM_BARS * 8 + 16 +
                              2 * (MAX_EXPERTS + 1) * 4;
  static constexpr uint32_t IDESC = ptx::idesc_bf16_f32(128, BN);
  static constexpr int OUT_COLS = MODE == 0 ? BNH : BN;  // output columns per tile
};
constexpr uint64_t kWaitLimitNs = 1000000000ull;

struct TcArgs {
  const int32_t* offsets;  // [N+1] slot offsets of the experts
  int n_experts;
  int kdim;                // reduction length: d (gate/up) or F (down)
  int n_tiles;             // output tiles per expert: F/128 (gate/up) or d/256 (down)
  int b_rows;              // rows of B per expert: F (gate/up) or d (down)
  void* out;               // h (bf16, row length F) or o (fp32, row length d)
  int ldo;
  uint32_t* status;
  void* pre;               // gate/up: NULL, or [padded rows][2F] bf16 pre-activations
                           // (gate | up) kept for the backward pass, row poff[e] + r for
                           // row r of expert e
  const int32_t* poff;     // [N+1] padded row offsets (with pre)
  int ksplit;              // gate/up: reduction split in ksplit parts (1: none); with
  float* part;             // ksplit > 1 the epilogue writes fp32 gate | up partials
  int64_t rows_part;       // part[ks][row][2F] (rows_part rows per part) and
                           // swiglu_combine_kernel applies SwiGLU
  // down with the combine fused (one routed expert per token, no shared
  // experts): y != NULL makes the epilogue write y[token] = g * o (+ x[token])
  // in bf16 instead of o
  const int32_t* token_of_slot;
  const float* gate;       // [T] the token's gate
  const __nv_bfloat16* xres;  // [T][d] residual rows or NULL
  __nv_bfloat16* y;        // [T][d]
  int32_t* sched;          // CTA-pair kernel: tile counter, 0 at launch
};

// silu(g) * u. The division is the fast reciprocal-multiply form (about two
// ulp in fp32, far below the bf16 rounding of h); where 1 + e^-g exceeds
// 2^126 it returns 0, the limit of silu there. The IEEE division it replaces
// made the gate/up epilogue the slowest stage of short-reduction tiles.
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fdividef(g, 1.f + __expf(-g)) * u;
}

// The 32 gate and 32 up pre-activations of one row chunk, rounded to bf16, at
// dst[0..32) and dst[F..F+32) (the backward pass's copy).
__device__ __forceinline__ void store_pre(__nv_bfloat16* dst, int F, const uint32_t (&g)[32],
                                          const uint32_t (&u)[32]) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint32_t(&src)[32] = half == 0 ? g : u;
    uint32_t p[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(src[2 * j]),
                                               __uint_as_float(src[2 * j + 1]));
      p[j] = *reinterpret_cast<uint32_t*>(&b);
    }
    uint4* d4 = reinterpret_cast<uint4*>(dst + half * F);
#pragma unroll
    for (int v = 0; v < 4; ++v) d4[v] = make_uint4(p[4 * v], p[4 * v + 1], p[4 * v + 2], p[4 * v + 3]);
  }
}

// Fused combine of one row chunk: y[t][col .. col+32) = bf16(g * o (+ x)),
// with the rounding steps of the combine kernel (the gate product rounded to
// fp32, then the residual added in fp32, then one rounding to bf16), so the
// result is the same bit for bit.
__device__ __forceinline__ void store_y_chunk(const TcArgs& a, int t, float g, int col,
                                              const uint32_t (&v)[32]) {
  const size_t base = static_cast<size_t>(t) * a.ldo + col;
  uint4 xr[4] = {};
  if (a.xres != nullptr) {
    const uint4* src = reinterpret_cast<const uint4*>(a.xres + base);
#pragma unroll
    for (int q = 0; q < 4; ++q) xr[q] = __ldg(src + q);
  }
  const __nv_bfloat162* xh = reinterpret_cast<const __nv_bfloat162*>(xr);
  uint32_t packed[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float a0 = __fmaf_rn(g, __uint_as_float(v[2 * j]), 0.f);
    float a1 = __fmaf_rn(g, __uint_as_float(v[2 * j + 1]), 0.f);
    if (a.xres != nullptr) {
      const float2 xv = __bfloat1622float2(xh[j]);
      a0 = __fadd_rn(a0, xv.x);
      a1 = __fadd_rn(a1, xv.y);
    }
    __nv_bfloat162 b = __floats2bfloat162_rn(a0, a1);
    packed[j] = *reinterpret_cast<uint32_t*>(&b);
  }
  uint4* dst = reinterpret_cast<uint4*>(a.y + base);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
}

// MODE 0: gate/up + SwiGLU -> h (bf16). MODE 1: down -> o (fp32), or y with
// the combine fused.
template <int MODE, int BNH>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmA64,
                const __grid_constant__ CUtensorMap tmA32,
                const __grid_constant__ CUtensorMap tmA16, const TcArgs args) {
  using namespace ptx;
  using Sh = TcShape<MODE, BNH>;
  constexpr int STAGES = Sh::STAGES, B_BYTES = Sh::B_BYTES, STAGE_BYTES = Sh::STAGE_BYTES;
  constexpr int NUM_BARS = Sh::NUM_BARS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base, sB = base + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + STAGES * STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* tile_start = reinterpret_cast<int*>(tmem_slot + 4);
  int* seg_off = tile_start + (MAX_EXPERTS + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = args.n_experts;
  const int KB = args.kdim / BK;
  auto bar_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto bar_tfull = [&](int a) { return smem_u32(bars + 2 * STAGES + a); };
  auto bar_tempty = [&](int a) { return smem_u32(bars + 2 * STAGES + 2 + a); };
  const uint32_t bar_drain = smem_u32(bars + 2 * STAGES + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull(a), 1);
      mbar_init(bar_tempty(a), 4);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB0);
    if (MODE == 0) prefetch_tmap(&tmB1);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Sh::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) {
    // tile_start[e] = tiles of experts < e; lane owns experts [PER*lane, PER*lane+PER)
    constexpr int PER = (MAX_EXPERTS + 31) / 32;
    int local[PER], sum = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int e = lane * PER + j;
      int tiles = 0;
      if (e < N) {
        const int o0 = args.offsets[e], o1 = args.offsets[e + 1];
        seg_off[e] = o0;
        tiles = ((o1 - o0 + BM - 1) / BM) * args.n_tiles * args.ksplit;
      }
      local[j] = tiles;
      sum += tiles;
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
      if (e < N) tile_start[e] = run;
      run += local[j];
    }
    if (lane == 31) tile_start[N] = incl;
    if (lane == 0) seg_off[N] = args.offsets[N];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = tile_start[N];

  // tile -> expert e, row tile m, column tile n, reduction part ks (m fastest,
  // then ks, then n: CTAs running together share the weight tile's rows)
  auto decode = [&](int tile, int& e, int& m, int& n, int& ks) {
    int lo = 0, hi = N - 1;  // last expert whose first tile is <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_start[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    e = lo;
    const int mt = (seg_off[e + 1] - seg_off[e] + BM - 1) / BM;
    const int local = tile - tile_start[e];
    n = local / (mt * args.ksplit);
    const int rem = local - n * mt * args.ksplit;
    ks = rem / mt;
    m = rem - ks * mt;
  };
  // the 64-wide K steps of reduction part ks
  auto kb_begin = [&](int ks) { return ks * KB / args.ksplit; };
  auto kb_end = [&](int ks) { return (ks + 1) * KB / args.ksplit; };
  auto fail = [&]() {
    set_status(args.status, MOE_ERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer ----
    int stage = 0;
    uint32_t phase = 0, issued = 0, issued_parity = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      int e, m, n, ks;
      decode(tile, e, m, n, ks);
      const int row_a = seg_off[e] + m * BM;
      const int row_b = e * args.b_rows + n * Sh::OUT_COLS;
      // Only the expert's rows of this tile are fetched (smallest box that
      // covers them); the rest of the 128-row A tile keeps stale data, which
      // only reaches accumulator rows that are never stored.
      const int rows = min(BM, seg_off[e + 1] - row_a);
      const CUtensorMap* mapA = rows > 64 ? &tmA : (rows > 32 ? &tmA64 : (rows > 16 ? &tmA32 : &tmA16));
      const uint32_t a_bytes = static_cast<uint32_t>(rows > 64 ? 128 : (rows > 32 ? 64 : (rows > 16 ? 32 : 16))) * BK * 2;
      for (int kb = kb_begin(ks); kb < kb_end(ks); ++kb) {
        if (!mbar_wait(bar_empty(stage), phase ^ 1u, kWaitLimitNs, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar_full(stage), a_bytes + B_BYTES);
        const uint32_t a_dst = sA + stage * A_BYTES, b_dst = sB + stage * B_BYTES;
        tma_load_2d(a_dst, mapA, bar_full(stage), kb * BK, row_a);
        if (MODE == 0) {
          tma_load_2d(b_dst, &tmB0, bar_full(stage), kb * BK, row_b);
          tma_load_2d(b_dst + B_BYTES / 2, &tmB1, bar_full(stage), kb * BK, row_b);
        } else {
          tma_load_2d(b_dst, &tmB0, bar_full(stage), kb * BK, row_b);
        }
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok) {
      fail();
      // let the copies already in flight land before the block exits
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s)) mbar_wait(bar_full(s), (issued_parity >> s) & 1u, kWaitLimitNs, nullptr);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ MMA issuer ----
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true, issued_any = false;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      int e, m, n, ks;
      decode(tile, e, m, n, ks);
      const int kb0 = kb_begin(ks), kb1 = kb_end(ks);
      if (!mbar_wait(bar_tempty(acc), acc_phase ^ 1u, kWaitLimitNs, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Sh::ACC);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(bar_full(stage), phase, kWaitLimitNs, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = sA + stage * A_BYTES, b0 = sB + stage * B_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_bf16(d_tmem, sdesc_kmajor_sw128(a0 + kk * 32), sdesc_kmajor_sw128(b0 + kk * 32),
                   Sh::IDESC, (kb != kb0 || kk != 0) ? 1u : 0u);
        issued_any = true;
        mma_commit(bar_empty(stage));
        if (++stage == STAGES) {
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
      if (issued_any) {  // wait for the MMAs in flight before TMEM is freed
        mma_commit(bar_drain);
        mbar_wait(bar_drain, 0, kWaitLimitNs, nullptr);
      }
    }
  } else if (warp >= 2) {
    // ------------------------------------------------ epilogue ----
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int e, m, n, ks;
      decode(tile, e, m, n, ks);
      const int cnt = seg_off[e + 1] - seg_off[e];
      bool ok = mbar_wait(bar_tfull(acc), acc_phase, kWaitLimitNs, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const int r = m * BM + q * 32 + lane;
      const bool valid = r < cnt;
      const size_t grow = static_cast<size_t>(seg_off[e]) + static_cast<size_t>(r);
      const uint32_t taddr = tmem_base + static_cast<uint32_t>(acc * Sh::ACC) +
                             (static_cast<uint32_t>(q * 32) << 16);
      if (MODE == 0 && args.ksplit > 1) {
        // reduction part ks: fp32 gate | up partials of this row
        float* pg = args.part + (static_cast<size_t>(ks) * args.rows_part + grow) * 2 * args.ldo +
                    n * Sh::OUT_COLS;
#pragma unroll 1
        for (int c = 0; c < BNH / 32; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c * 32, g);
          tmem_ld32(taddr + BNH + c * 32, u);
          tmem_ld_wait();
          if (valid) {
            float4* dg = reinterpret_cast<float4*>(pg + c * 32);
            float4* du = reinterpret_cast<float4*>(pg + args.ldo + c * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              dg[j] = make_float4(__uint_as_float(g[4 * j]), __uint_as_float(g[4 * j + 1]),
                                  __uint_as_float(g[4 * j + 2]), __uint_as_float(g[4 * j + 3]));
              du[j] = make_float4(__uint_as_float(u[4 * j]), __uint_as_float(u[4 * j + 1]),
                                  __uint_as_float(u[4 * j + 2]), __uint_as_float(u[4 * j + 3]));
            }
          }
        }
      } else if (MODE == 0) {
        __nv_bfloat16* out =
            static_cast<__nv_bfloat16*>(args.out) + grow * args.ldo + n * Sh::OUT_COLS;
#pragma unroll 1
        for (int c = 0; c < BNH / 32; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c * 32, g);
          tmem_ld32(taddr + BNH + c * 32, u);
          tmem_ld_wait();
          uint32_t packed[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float g0 = __uint_as_float(g[2 * j]), g1 = __uint_as_float(g[2 * j + 1]);
            const float u0 = __uint_as_float(u[2 * j]), u1 = __uint_as_float(u[2 * j + 1]);
            const float h0 = silu_mul(g0, u0);
            const float h1 = silu_mul(g1, u1);
            __nv_bfloat162 hb = __floats2bfloat162_rn(h0, h1);
            packed[j] = *reinterpret_cast<uint32_t*>(&hb);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                                  packed[4 * v + 3]);
            if (args.pre != nullptr)
              store_pre(static_cast<__nv_bfloat16*>(args.pre) +
                            (static_cast<size_t>(args.poff[e]) + r) * 2 * args.ldo +
                            n * Sh::OUT_COLS + c * 32,
                        args.ldo, g, u);
          }
        }
      } else if (args.y != nullptr) {
        const int t = valid ? args.token_of_slot[grow] : 0;
        const float g = valid ? args.gate[t] : 0.f;
#pragma unroll 1
        for (int c = 0; c < Sh::BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(taddr + c * 32, v);
          tmem_ld_wait();
          if (valid) store_y_chunk(args, t, g, n * Sh::OUT_COLS + c * 32, v);
        }
      } else {
        float* out = static_cast<float*>(args.out) + grow * args.ldo + n * Sh::OUT_COLS;
#pragma unroll 1
        for (int c = 0; c < Sh::BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(taddr + c * 32, v);
          tmem_ld_wait();
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(out + c * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                   __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Sh::TMEM_COLS);
  }
}

// ---- CTA-pair variant (cta_group::2) -------------------------------------------
// Two CTAs of a cluster compute a 256-row tile together: the even CTA takes
// m-tile 2p, the odd CTA m-tile 2p+1 of the same (expert, n-tile). Each CTA
// loads its own 128 rows of A and one half of the weight tile (MODE 0: the
// gate rows in the even CTA, the up rows in the odd one; MODE 1: rows
// [0,128) and [128,256) of the down tile), so each SM fetches 32 KB per 64-wide
// K step instead of 48 KB for the same MMA work, and the ring gets 6 stages.
// The even CTA issues every MMA (M=256, N=256) for the pair; both CTAs'
// loads report to its full barrier, and its commits release the stages and
// announce finished accumulators in both CTAs. Each CTA drains its own TMEM
// rows; the odd CTA reports a drained accumulator to the even CTA remotely.
// Tiles are claimed, not dealt: the even CTA's producer takes the next tile
// index from a global counter (atomicAdd) and hands it through a small queue
// to its MMA and epilogue warps and to the odd CTA. The clusters then work on
// consecutive tiles at any moment, so the row tiles that share one weight tile
// read it while it is still in L2. Dealt with a fixed stride, clusters drifted
// apart by whole tiles over a long launch and fetched weight tiles from HBM
// again (measured on the Mixtral-shaped prefill gate/up GEMM: 1.24-1.52x its
// algorithmic DRAM bytes dealt, 1.00x claimed; that launch 6 % faster).
constexpr int P_STAGES = 6;
constexpr int P_A_BYTES = 128 * BK * 2;
constexpr int P_B_BYTES = 128 * BK * 2;
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
constexpr int P_ACC_BUFS = 2;
constexpr int P_TMEM_COLS = ACC_COLS * P_ACC_BUFS;
constexpr int P_TQ = 4;  // depth of the claimed-tile queue
// consumers of a queue entry: the MMA warp and 4 epilogue warps of the even
// CTA, the producer and 4 epilogue warps of the odd CTA
constexpr int P_TQ_CONSUMERS = 10;
constexpr int P_NUM_BARS = 2 * P_STAGES + 5 + 2 * P_TQ;
constexpr int P_SMEM_BYTES = 1024 + P_STAGES * P_STAGE_BYTES + P_NUM_BARS * 8 + 16 +
                             2 * (MAX_EXPERTS + 1) * 4 + P_TQ * 4;
constexpr uint32_t P_IDESC = ptx::idesc_bf16_f32(256, 256);

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_pair(const __grid_constant__ CUtensorMap tmA,
                  const __grid_constant__ CUtensorMap tmB0,
                  const __grid_constant__ CUtensorMap tmB1, const TcArgs args) {
  using namespace ptx;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base, sB = base + P_STAGES * P_A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + P_STAGES * P_STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + P_NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* tile_start = reinterpret_cast<int*>(tmem_slot + 4);
  int* seg_off = tile_start + (MAX_EXPERTS + 1);
  volatile int* tq = seg_off + (MAX_EXPERTS + 1);  // claimed tiles, -1 ends

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = args.n_experts;
  const int KB = args.kdim / BK;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  constexpr uint16_t kBoth = 0x3;
  auto bar_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return smem_u32(bars + P_STAGES + s); };
  auto bar_tfull = [&](int a) { return smem_u32(bars + 2 * P_STAGES + a); };
  auto bar_tempty = [&](int a) { return smem_u32(bars + 2 * P_STAGES + 2 + a); };
  const uint32_t bar_drain = smem_u32(bars + 2 * P_STAGES + 4);
  auto bar_qfull = [&](int q) { return smem_u32(bars + 2 * P_STAGES + 5 + q); };
  auto bar_qempty = [&](int q) { return smem_u32(bars + 2 * P_STAGES + 5 + P_TQ + q); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(bar_full(s), 1);   // even CTA: its producer's expect_tx arrive
      mbar_init(bar_empty(s), 1);  // the even CTA's commit, multicast to both
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull(a), 1);
      mbar_init(bar_tempty(a), 8);  // even CTA: 4 local + 4 remote epilogue warps
    }
    mbar_init(bar_drain, 1);
    for (int q = 0; q < P_TQ; ++q) {
      mbar_init(bar_qfull(q), 1);  // this CTA's producer (odd CTA: with the st.async's 4 bytes)
      mbar_init(bar_qempty(q), P_TQ_CONSUMERS);  // used in the even CTA only
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB0);
    if (MODE == 0) prefetch_tmap(&tmB1);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), P_TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 2) {
    constexpr int PER = (MAX_EXPERTS + 31) / 32;
    int local[PER], sum = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int e = lane * PER + j;
      int tiles = 0;
      if (e < N) {
        const int o0 = args.offsets[e], o1 = args.offsets[e + 1];
        seg_off[e] = o0;
        tiles = ((o1 - o0 + 2 * BM - 1) / (2 * BM)) * args.n_tiles;
      }
      local[j] = tiles;
      sum += tiles;
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
      if (e < N) tile_start[e] = run;
      run += local[j];
    }
    if (lane == 31) tile_start[N] = incl;
    if (lane == 0) seg_off[N] = args.offsets[N];
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  cluster_sync();  // both CTAs' barriers and TMEM exist before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = tile_start[N];

  auto decode = [&](int tile, int& e, int& m, int& n) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_start[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    e = lo;
    const int mtp = (seg_off[e + 1] - seg_off[e] + 2 * BM - 1) / (2 * BM);
    const int local = tile - tile_start[e];
    n = local / mtp;
    m = (local - n * mtp) * 2 + static_cast<int>(rank);
  };
  auto fail = [&]() {
    set_status(args.status, MOE_ERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer (both CTAs) ----
    // The even CTA's producer claims the tiles and publishes each (then -1)
    // in the queue of both CTAs; the odd CTA's producer reads them from it.
    // A tile is claimed when the previous one starts and published halfway
    // through its loads, so the atomic's round trip (long behind a saturated
    // memory system) does not hold up the loads. The odd CTA gets each entry
    // by st.async, which completes on its full barrier, and its consumers free
    // a slot with relaxed remote arrives made after (control-dependent on)
    // their read of it. Measured: with a remote store and remote arrives of
    // release semantics instead, the handoff cost 0.4-1.9 us per tile on the
    // memory-bound layers; in this form it costs nothing measurable.
    int stage = 0, qs = 0;
    uint32_t phase = 0, qphase = 0, issued = 0, issued_parity = 0;
    bool ok = true;
    auto publish = [&](int t) -> bool {
      if (!mbar_wait_cluster(bar_qempty(qs), qphase ^ 1u, kWaitLimitNs, abort_flag))
        return false;
      tq[qs] = t;
      mbar_arrive(bar_qfull(qs));
      st_async_remote_u32(map_to_rank(smem_u32(const_cast<int*>(tq + qs)), 1),
                          static_cast<uint32_t>(t), map_to_rank(bar_qfull(qs), 1));
      if (++qs == P_TQ) {
        qs = 0;
        qphase ^= 1u;
      }
      return true;
    };
    int tile = -1;
    if (leader) {
      const int c = atomicAdd(args.sched, 1);
      tile = c < total ? c : -1;
      ok = publish(tile);
    }
    const int pub_kb = KB / 2;
    while (ok) {
      if (!leader) {
        mbar_arrive_expect_tx(bar_qfull(qs), 4);  // the entry's st.async
        if (!mbar_wait(bar_qfull(qs), qphase, kWaitLimitNs, abort_flag)) {
          ok = false;
          break;
        }
        tile = tq[qs];
        if (tile >= -1) mbar_arrive_remote_relaxed(map_to_rank(bar_qempty(qs), 0));
        if (++qs == P_TQ) {
          qs = 0;
          qphase ^= 1u;
        }
      }
      if (tile < 0) break;
      const int following = leader ? atomicAdd(args.sched, 1) : 0;
      int e, m, n;
      decode(tile, e, m, n);
      // A CTA whose 128 rows all lie past the expert's last row loads its A
      // tile from beyond the activation rows: TMA fills it with zeros without
      // reading memory, and zeros cost the tensor cores less energy than the
      // next expert's rows would (measured: the step runs faster under the
      // power cap when rows are zero)
      const int row_a = m * BM >= seg_off[e + 1] - seg_off[e]
                            ? static_cast<int>(args.rows_part)
                            : seg_off[e] + m * BM;
      const int row_b = e * args.b_rows + n * (MODE == 0 ? 128 : 256) +
                        (MODE == 1 ? 128 * static_cast<int>(rank) : 0);
      for (int kb = 0; kb < KB; ++kb) {
        if (leader && kb == pub_kb && !publish(following < total ? following : -1)) {
          ok = false;
          break;
        }
        if (!mbar_wait(bar_empty(stage), phase ^ 1u, kWaitLimitNs, abort_flag)) {
          ok = false;
          break;
        }
        if (leader) mbar_arrive_expect_tx(bar_full(stage), 2 * P_STAGE_BYTES);
        const uint32_t full_leader = map_to_rank(bar_full(stage), 0);
        tma_load_2d_pair(sA + stage * P_A_BYTES, &tmA, full_leader, kb * BK, row_a);
        tma_load_2d_pair(sB + stage * P_B_BYTES, (MODE == 0 && !leader) ? &tmB1 : &tmB0,
                         full_leader, kb * BK, row_b);
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == P_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (leader) tile = following < total ? following : -1;
    }
    if (!ok) {
      fail();
      if (leader)  // the even CTA's full barriers count both CTAs' copies
        for (int s = 0; s < P_STAGES; ++s)
          if (issued & (1u << s))
            mbar_wait_cluster(bar_full(s), (issued_parity >> s) & 1u, kWaitLimitNs, nullptr);
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------ MMA issuer (even CTA) ----
    int stage = 0, acc = 0, qs = 0;
    uint32_t phase = 0, acc_phase = 0, qphase = 0;
    bool ok = true, issued_any = false;
    while (ok) {
      if (!mbar_wait(bar_qfull(qs), qphase, kWaitLimitNs, abort_flag)) {
        ok = false;
        break;
      }
      const int tile = tq[qs];
      mbar_arrive(bar_qempty(qs));
      if (++qs == P_TQ) {
        qs = 0;
        qphase ^= 1u;
      }
      if (tile < 0) break;
      if (!mbar_wait_cluster(bar_tempty(acc), acc_phase ^ 1u, kWaitLimitNs, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ACC_COLS);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_cluster(bar_full(stage), phase, kWaitLimitNs, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = sA + stage * P_A_BYTES, b0 = sB + stage * P_B_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_bf16_pair(d_tmem, sdesc_kmajor_sw128(a0 + kk * 32),
                        sdesc_kmajor_sw128(b0 + kk * 32), P_IDESC, (kb | kk) != 0 ? 1u : 0u);
        issued_any = true;
        mma_commit_pair(bar_empty(stage), kBoth);
        if (++stage == P_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      mma_commit_pair(bar_tfull(acc), kBoth);
      if (++acc == P_ACC_BUFS) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok) {
      fail();
      if (issued_any) {
        mma_commit_pair(bar_drain, 0x1);
        mbar_wait(bar_drain, 0, kWaitLimitNs, nullptr);
      }
    }
  } else if (warp >= 2) {
    // ------------------------------------------------ epilogue (both CTAs) ----
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    const uint32_t tempty_leader0 = map_to_rank(bar_tempty(0), 0);
    const uint32_t tempty_leader1 = map_to_rank(bar_tempty(1), 0);
    int qs = 0;
    uint32_t qphase = 0;
    for (;;) {
      bool got = mbar_wait(bar_qfull(qs), qphase, kWaitLimitNs, abort_flag);
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        if (lane == 0) fail();
        break;
      }
      const int tile = tq[qs];
      __syncwarp();
      if (lane == 0 && tile >= -1) {
        if (leader) mbar_arrive(bar_qempty(qs));
        else mbar_arrive_remote_relaxed(map_to_rank(bar_qempty(qs), 0));
      }
      if (++qs == P_TQ) {
        qs = 0;
        qphase ^= 1u;
      }
      if (tile < 0) break;
      int e, m, n;
      decode(tile, e, m, n);
      const int cnt = seg_off[e + 1] - seg_off[e];
      bool ok = mbar_wait_cluster(bar_tfull(acc), acc_phase, kWaitLimitNs, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const int r = m * BM + q * 32 + lane;
      const bool valid = r < cnt;
      const size_t grow = static_cast<size_t>(seg_off[e]) + static_cast<size_t>(r);
      const uint32_t taddr = tmem_base + static_cast<uint32_t>(acc * ACC_COLS) +
                             (static_cast<uint32_t>(q * 32) << 16);
      if (MODE == 0) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out) + grow * args.ldo + n * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c * 32, g);
          tmem_ld32(taddr + 128 + c * 32, u);
          tmem_ld_wait();
          uint32_t packed[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float g0 = __uint_as_float(g[2 * j]), g1 = __uint_as_float(g[2 * j + 1]);
            const float u0 = __uint_as_float(u[2 * j]), u1 = __uint_as_float(u[2 * j + 1]);
            const float h0 = silu_mul(g0, u0);
            const float h1 = silu_mul(g1, u1);
            __nv_bfloat162 hb = __floats2bfloat162_rn(h0, h1);
            packed[j] = *reinterpret_cast<uint32_t*>(&hb);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                                  packed[4 * v + 3]);
            if (args.pre != nullptr)
              store_pre(static_cast<__nv_bfloat16*>(args.pre) +
                            (static_cast<size_t>(args.poff[e]) + r) * 2 * args.ldo + n * 128 +
                            c * 32,
                        args.ldo, g, u);
          }
        }
      } else if (args.y != nullptr) {
        const int t = valid ? args.token_of_slot[grow] : 0;
        const float g = valid ? args.gate[t] : 0.f;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[32];
          tmem_ld32(taddr + c * 32, v);
          tmem_ld_wait();
          if (valid) store_y_chunk(args, t, g, n * 256 + c * 32, v);
        }
      } else {
        float* out = static_cast<float*>(args.out) + grow * args.ldo + n * 256;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[32];
          tmem_ld32(taddr + c * 32, v);
          tmem_ld_wait();
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(out + c * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                   __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(bar_tempty(acc));
        else mbar_arrive_remote(acc == 0 ? tempty_leader0 : tempty_leader1);
      }
      if (++acc == P_ACC_BUFS) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  __syncwarp();
  cluster_sync();  // no CTA of the pair leaves while the other may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, P_TMEM_COLS);
  }
}

// Gate/up with a split reduction: h[r][f] = silu(g) * u with g, u the sums of
// the parts' fp32 partials in ascending part order (the same SwiGLU as the
// GEMM epilogue); with pre, (g, u) rounded to bf16 are kept at padded row
// poff[e] + (r - offsets[e]). Block (r, c) handles columns [512 c, 512 c + 512)
// of row r, two per thread (rows past offsets[E] have no data and return), so
// a decode-sized batch of a few dozen rows still fills the GPU.
constexpr int kSwigluCols = 512;

__global__ void __launch_bounds__(256)
swiglu_combine_kernel(const float* __restrict__ part, int ksplit, int64_t rows_part,
                      const int32_t* __restrict__ offsets, int E, int F,
                      __nv_bfloat16* __restrict__ h, __nv_bfloat16* __restrict__ pre,
                      const int32_t* __restrict__ poff) {
  const int r = blockIdx.x;
  if (r >= offsets[E]) return;
  int prow = 0;
  if (pre != nullptr) {
    int lo = 0, hi = E - 1;  // the expert whose rows hold r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (offsets[mid] <= r) lo = mid;
      else hi = mid - 1;
    }
    prow = poff[lo] + (r - offsets[lo]);
  }
  const int f_end = min(F, static_cast<int>(blockIdx.y + 1) * kSwigluCols);
  for (int f = static_cast<int>(blockIdx.y) * kSwigluCols + threadIdx.x * 2; f < f_end;
       f += blockDim.x * 2) {
    float2 g = make_float2(0.f, 0.f), u = make_float2(0.f, 0.f);
    for (int ks = 0; ks < ksplit; ++ks) {
      const float* row = part + (static_cast<size_t>(ks) * rows_part + r) * 2 * F;
      const float2 pg = *reinterpret_cast<const float2*>(row + f);
      const float2 pu = *reinterpret_cast<const float2*>(row + F + f);
      g.x += pg.x;
      g.y += pg.y;
      u.x += pu.x;
      u.y += pu.y;
    }
    const float h0 = silu_mul(g.x, u.x);
    const float h1 = silu_mul(g.y, u.y);
    *reinterpret_cast<__nv_bfloat162*>(h + static_cast<size_t>(r) * F + f) =
        __floats2bfloat162_rn(h0, h1);
    if (pre != nullptr) {
      __nv_bfloat16* pr = pre + static_cast<size_t>(prow) * 2 * F;
      *reinterpret_cast<__nv_bfloat162*>(pr + f) = __floats2bfloat162_rn(g.x, g.y);
      *reinterpret_cast<__nv_bfloat162*>(pr + F + f) = __floats2bfloat162_rn(u.x, u.y);
    }
  }
}

// ---- host side ---------------------------------------------------------------
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

// Row-major bf16 matrix [rows][cols] as a 2-D tensor map with a box of
// box_rows x 64 columns and the 128-byte swizzle; out-of-range rows read 0.
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

bool set_smem_attr() {
  // Per device; the attribute is cheap to set, so set it on every device once.
  static int done_mask = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 31 && (done_mask >> dev) & 1) return true;
  if (cudaFuncSetAttribute(grouped_gemm_tc<0, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           TcShape<0, 128>::SMEM) != cudaSuccess ||
      cudaFuncSetAttribute(grouped_gemm_tc<1, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           TcShape<1, 128>::SMEM) != cudaSuccess)
    return false;
  if (cudaFuncSetAttribute(grouped_gemm_pair<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           P_SMEM_BYTES) != cudaSuccess ||
      cudaFuncSetAttribute(grouped_gemm_pair<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           P_SMEM_BYTES) != cudaSuccess)
    return false;
  if (dev < 31) done_mask |= 1 << dev;
  return true;
}

// CTA pairs pay off when experts have several 128-row tiles (then both CTAs
// of a pair compute stored rows; with about one tile per expert the odd CTA
// would mostly compute discarded rows) and the reduction is long enough to
// amortise the pair's coupling per tile (measured on the Switch-shaped gate/up
// GEMM, 16 K-steps per tile: pairs 4 % faster than one CTA per tile; shorter
// reductions were not measured and stay on one CTA per tile).
bool use_pairs(const moe_config& c, int64_t rows, int kdim) {
  return rows >= static_cast<int64_t>(c.n_experts + c.n_shared) * BM * 4 && kdim >= 1024;
}

// The down projection also takes CTA pairs when experts have about one row
// tile each, as long as its pair tiles fill the clusters at least twice:
// measured on the DeepSeek-shaped layer (128 rows per expert, F = 2048) the
// down GEMM went 1.90 -> 1.55 ms on pairs (a pair's odd CTA reads no
// activation rows there and stores nothing; each SM streams half a weight
// tile per K step), while its gate/up GEMM got slower on pairs (2.57 -> 2.86
// ms). Decode-sized batches (too few pair tiles) stay on one CTA per tile.
bool down_uses_pairs(const moe_config& c, int64_t rows) {
  if (use_pairs(c, rows, c.d_ff)) return true;
  if (c.d_ff < 1024) return false;
  const int64_t E = c.n_experts + c.n_shared;
  const int64_t pair_tiles = (E + (rows + 2 * BM - 1) / (2 * BM)) * (c.d_model / 256);
  return pair_tiles >= sm_count();  // two per cluster of two SMs
}

template <int MODE>
cudaError_t launch_pair(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                        const TcArgs& args, int64_t pair_tiles, cudaStream_t s) {
  const int sms = sm_count();
  int64_t clusters = pair_tiles < sms / 2 ? pair_tiles : sms / 2;
  if (clusters < 1) clusters = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = P_SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_pair<MODE>, a, b0, b1, args);
}

}  // namespace

// Reduction split of the one-CTA gate/up GEMM for batches with about one row
// tile per expert (decode): the persistent grid then deals E_active x F/128
// weight-streaming tiles to the SMs, and the last partial wave can cost a
// whole tile time (8 x 112 tiles on 148 SMs: 6.05 waves take 7). Splitting
// each tile's reduction in s parts makes the units s times smaller; s is the
// smallest in 1..8 whose last wave wastes at most 4 % (experts assumed all
// active, each with one row tile). Returns 1 otherwise.
int gate_up_ksplit(const moe_config& c, int64_t rows) {
  const int E = c.n_experts + c.n_shared;
  const int KB = c.d_model / BK;
  if (c.dtype != MOE_BF16 || rows > static_cast<int64_t>(E) * BM || KB < 16) return 1;
  const int64_t active = rows < E ? rows : E;
  const int64_t tiles = active * (c.d_ff / 128);
  const int sms = sm_count();
  int best = 1;
  double best_waste = 1e9;
  for (int sp = 1; sp <= 8 && KB / sp >= 4; ++sp) {
    const double units = static_cast<double>(tiles) * sp;
    const double waves = units / sms;
    const double waste = std::ceil(waves) / waves - 1.0;
    if (waste < best_waste - 1e-9) {
      best_waste = waste;
      best = sp;
    }
    if (waste <= 0.04) break;
  }
  return best;
}

bool ffn_tc_supported(const moe_config& c) {
  return c.dtype == MOE_BF16 && c.activation == MOE_SWIGLU && c.d_model % 256 == 0 &&
         c.d_ff % 128 == 0 && c.n_experts + c.n_shared <= MAX_EXPERTS;
}

moe_status launch_ffn_tc(const moe_config& c, int64_t rows, const void* x_perm,
                         const int32_t* offsets, const moe_expert_weights& w, void* h, float* o,
                         void* pre, const int32_t* poff, float* gu_part, int32_t* sched,
                         bool sched_zeroed, uint32_t* status, cudaStream_t s, int part,
                         const FusedCombine* fc) {
  if (rows == 0) return MOE_OK;
  const int E = c.n_experts + c.n_shared, d = c.d_model, F = c.d_ff;  // routed + shared
  const bool pairs1 = use_pairs(c, rows, d);  // gate/up: reduction over d
  const bool pairs2 = down_uses_pairs(c, rows);  // down: reduction over F
  if (!set_smem_attr()) return MOE_ERR_CUDA;
  const int64_t mtiles = E + (rows + BM - 1) / BM;       // upper bound on (expert, m-tile)
  const int64_t ptiles = E + (rows + 2 * BM - 1) / (2 * BM);
  const int sms = sm_count();
  if (part & 1) {
    CUtensorMap mx, mg, mu;
    if (!make_map(&mx, x_perm, rows, d, 128) ||
        !make_map(&mg, w.w_gate, static_cast<uint64_t>(E) * F, d, 128) ||
        !make_map(&mu, w.w_up, static_cast<uint64_t>(E) * F, d, 128))
      return MOE_ERR_CUDA;
    const int ksplit = pairs1 ? 1 : gate_up_ksplit(c, rows);
    TcArgs a1{offsets, E, d, F / 128, F, h, F, status, pre, poff, ksplit, gu_part, rows,
              nullptr, nullptr, nullptr, nullptr, sched};
    if (pairs1) {
      if ((!sched_zeroed && cudaMemsetAsync(sched, 0, sizeof(int32_t), s) != cudaSuccess) ||
          launch_pair<0>(mx, mg, mu, a1, ptiles * (F / 128), s) != cudaSuccess)
        return MOE_ERR_CUDA;
    } else {
      CUtensorMap mx64, mx32, mx16;  // activation boxes for partly filled tiles
      if (!make_map(&mx64, x_perm, rows, d, 64) || !make_map(&mx32, x_perm, rows, d, 32) ||
          !make_map(&mx16, x_perm, rows, d, 16))
        return MOE_ERR_CUDA;
      const int64_t t1 = mtiles * (F / 128) * ksplit;
      grouped_gemm_tc<0, 128><<<static_cast<unsigned>(t1 < sms ? t1 : sms), kThreads,
                                TcShape<0, 128>::SMEM, s>>>(mx, mg, mu, mx64, mx32, mx16, a1);
      if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
      if (ksplit > 1) {
        const dim3 grid(static_cast<unsigned>(rows), (F + kSwigluCols - 1) / kSwigluCols);
        swiglu_combine_kernel<<<grid, 256, 0, s>>>(
            gu_part, ksplit, rows, offsets, E, F, static_cast<__nv_bfloat16*>(h),
            static_cast<__nv_bfloat16*>(pre), poff);
        if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
      }
    }
  }
  if (part & 2) {
    CUtensorMap mh, md;
    if (!make_map(&mh, h, rows, F, 128) ||
        !make_map(&md, w.w_down, static_cast<uint64_t>(E) * d, F, pairs2 ? 128 : 256))
      return MOE_ERR_CUDA;
    TcArgs a2{offsets, E, F, d / 256, d, o, d, status, nullptr, nullptr, 1, nullptr, rows,
              fc ? fc->token_of_slot : nullptr, fc ? fc->gate : nullptr,
              fc ? static_cast<const __nv_bfloat16*>(fc->x) : nullptr,
              fc ? static_cast<__nv_bfloat16*>(fc->y) : nullptr, sched + 1};
    if (pairs2) {
      if ((!sched_zeroed && cudaMemsetAsync(sched + 1, 0, sizeof(int32_t), s) != cudaSuccess) ||
          launch_pair<1>(mh, md, md, a2, ptiles * (d / 256), s) != cudaSuccess)
        return MOE_ERR_CUDA;
    } else {
      CUtensorMap mh64, mh32, mh16;
      if (!make_map(&mh64, h, rows, F, 64) || !make_map(&mh32, h, rows, F, 32) ||
          !make_map(&mh16, h, rows, F, 16))
        return MOE_ERR_CUDA;
      const int64_t t2 = mtiles * (d / 256);
      grouped_gemm_tc<1, 128><<<static_cast<unsigned>(t2 < sms ? t2 : sms), kThreads,
                                TcShape<1, 128>::SMEM, s>>>(mh, md, md, mh64, mh32, mh16, a2);
      if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    }
  }
  return MOE_OK;
}
}  // namespace moe

// ---------------------------------------------------------------------------
// Self-test of the bounded wait used by every mbarrier wait of the tensor-core
// kernels: one thread waits on an mbarrier that nothing will ever arrive at,
// gives up after limit_ns, records MOE_ERR_TIMEOUT in the status word and the
// kernel returns normally (the GPU context stays usable).
// ---------------------------------------------------------------------------
namespace moe {
namespace {

__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns, uint32_t* status) {
  using namespace ptx;
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&bar), 1);
  abort_flag = 0;
  fence_mbar_init();
  if (!mbar_wait(smem_u32(&bar), 0, limit_ns, &abort_flag)) set_status(status, MOE_ERR_TIMEOUT);
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_selftest_bounded_wait(uint32_t limit_us, uint32_t* status,
                                                moe_stream_t stream) {
  if (status == nullptr || limit_us == 0 || limit_us > 10000000u) return MOE_ERR_INVALID;
  moe::bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint64_t>(limit_us) * 1000u, status);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
