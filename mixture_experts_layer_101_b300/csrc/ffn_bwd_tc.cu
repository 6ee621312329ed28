// Expert gradients of the backward pass on the tcgen05 tensor cores (bf16
// SwiGLU layers whose forward runs on the tensor cores).
//
// Sources: the derivatives of "MoE 混合专家模型稀疏激活的架构原理与负载均衡挑战"
// §三 class Expert (down(silu(gate(x)) * up(x))), trained end to end with the
// router ("混合专家模型（Mixture of Experts, MoE）" 结构 2).
//
// For the rows r of expert e ([offsets[e], offsets[e+1]), routed experts
// then shared ones), with a | b the kept gate | up pre-activations, h the
// forward's hidden activation and dout the output gradient g * dy:
//   DGRAD_SWIGLU  dh[r][f] = sum_j dout[r][j] W_down[e][j][f], and in the
//                 epilogue (da, db) = (dh b silu'(a), dh silu(a)) written
//                 over (a, b) in place (bf16)
//   WGRAD         dW_down[e][j][f] = sum_r dout[r][j] h[r][f]
//   DGRAD_STORE   dx_perm[r][j] = sum_f da[r][f] W_gate[e][f][j]
//                                + sum_f db[r][f] W_up[e][f][j]   (fp32)
//   WGRAD         dW_gate[e][f][j] = sum_r da[r][f] x_perm[r][j] and
//                 dW_up[e][f][j] = sum_r db[r][f] x_perm[r][j]: one launch
//                 over M = 2F rows of (da | db)
// The weights enter the dgrad products with their output dimension
// contiguous, and both operands of the weight-gradient products have their
// M / N dimension contiguous along the token rows, so those operands are
// loaded as MN-major tiles (the TMA box is 64 columns x 64 rows; the MMA
// reads 64-column slices 8 KB apart); only the dgrad A operand is K-major.
//
// Row spaces: the forward's activations (x_perm, h, the kept pre-activations,
// and dx_perm) use the dispatch's slots, boff[e] .. boff[e+1]. The backward's
// own activations (dout and the pre-activation gradients) use a padded
// space, aoff[e] = sum over earlier experts of their row counts rounded up
// to 64, whose pad rows are zero: a weight-gradient reduction can then run
// over whole 64-row steps of A, since the zero pad rows cancel whatever the
// B operand (forward rows of the next expert) holds there.
//
// Kernel: persistent and warp-specialised like the forward's grouped GEMM
// (warp 0 TMA producer, warp 1 MMA issuer, warps 2-5 epilogue, two TMEM
// accumulators of BN fp32 columns), in two forms: one CTA per tile (M = 128)
// or a CTA pair of one cluster (cta_group::2, M = 256 = 128 rows per CTA,
// each CTA loading its own A rows and its half of the B columns, the even
// CTA issuing the MMAs), which halves the bytes each SM pulls per MMA cycle.
// DGRAD tiles are (expert, 128-row tile, BN-column tile); a row tile may run
// past its expert's rows, whose accumulator rows are never stored. WGRAD
// tiles are (expert, 128-row block of M, BN-column block), reduced over the
// expert's padded rows. An expert with no rows gets zeros. Every wait is
// bounded.
#include "moe_common.cuh"
#include "ptx_sm100.cuh"

#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

namespace moe {
namespace {

constexpr int BM = 128, BK = 64;
constexpr int MAX_GROUPS = 264;
constexpr int CHUNK = 64 * 128;  // one 64-column x 64-row MN-major box: 8 KB
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;

enum { DGRAD_STORE = 0, DGRAD_SWIGLU = 1, WGRAD = 2 };

// PAIR: BN columns per pair tile, BN / 2 of B held by each CTA. The staging
// buffers of the fp32 transposes are 32 x 32 floats per epilogue warp,
// 16-byte chunks XOR-swizzled by row (no padding, no bank conflicts).
template <int KIND, int BN, bool PAIR>
struct BwShape {
  static constexpr int BNL = PAIR ? BN / 2 : BN;  // B columns in this CTA's shared memory
  static constexpr int A_BYTES = BM * BK * 2;     // 16 KB
  static constexpr int B_BYTES = BNL * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = (196608 / STAGE) > 6 ? 6 : (196608 / STAGE);
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  static constexpr bool STAGED = KIND != DGRAD_SWIGLU;
  static constexpr int STG_FLOATS = 32 * 32;
  static constexpr int SMEM = 1024 + STAGES * STAGE + NUM_BARS * 8 + 16 +
                              3 * (MAX_GROUPS + 1) * 4 + 16 +
                              (STAGED ? kEpiWarps * STG_FLOATS * 4 : 0);
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(!PAIR || BN == 256, "pair tiles are 256 columns wide");
  static constexpr uint32_t IDESC =
      ptx::idesc_bf16_f32_major(PAIR ? 2 * BM : BM, BN, KIND == WGRAD, true);
};

struct BwArgs {
  const int32_t* aoff;     // [G+1] rows of the A operand (padded space; DGRAD_SWIGLU: also dpre)
  const int32_t* boff;     // [G+1] forward rows (WGRAD B, pre, DGRAD_STORE output); counts
  int groups;
  int kb_total;            // DGRAD: 64-wide K steps
  int kb_split;            // DGRAD: K steps read from the first B map (rest: second)
  int b_rows;              // DGRAD: rows of a B map per expert (its K extent)
  int n_tiles;             // BN-column tiles per output row block
  int m_blocks;            // WGRAD: 128-row blocks of M per expert
  int m_split;             // WGRAD: output rows >= m_split go to out2 (row - m_split)
  int acol;                // WGRAD: first column of A used
  float* out;              // DGRAD_STORE: [rows][ldo]; WGRAD: [G][m_split or M][ldo]
  float* out2;             // WGRAD: second output (dW_up) or NULL
  int ldo;
  __nv_bfloat16* pre;        // DGRAD_SWIGLU: [padded rows][2F] a | b in, da | db out (in
                             // place), pad rows zeroed
  int F;
  uint32_t* status;
};

template <int KIND, int BN, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
grouped_bwd_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
               const __grid_constant__ CUtensorMap tmB1, const BwArgs args) {
  using namespace ptx;
  using Sh = BwShape<KIND, BN, PAIR>;
  constexpr int STAGES = Sh::STAGES;
  constexpr bool W = KIND == WGRAD;
  constexpr int MU = PAIR ? 2 : 1;  // 128-row units of M per tile
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base, sB = base + STAGES * Sh::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + STAGES * Sh::STAGE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Sh::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* tile_start = reinterpret_cast<int*>(tmem_slot + 4);
  int* seg_a = tile_start + (MAX_GROUPS + 1);
  int* seg_b = seg_a + (MAX_GROUPS + 1);
  float* staging = reinterpret_cast<float*>(
      (reinterpret_cast<uintptr_t>(seg_b + MAX_GROUPS + 1) + 15) &
      ~static_cast<uintptr_t>(15));  // STAGED kinds only

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = args.groups;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int first = PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int stride = PAIR ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
  auto bar_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto bar_tfull = [&](int a) { return smem_u32(bars + 2 * STAGES + a); };
  auto bar_tempty = [&](int a) { return smem_u32(bars + 2 * STAGES + 2 + a); };
  const uint32_t bar_drain = smem_u32(bars + 2 * STAGES + 4);
  auto wait = [&](uint32_t bar, uint32_t parity, const volatile int* ab) {
    return PAIR ? mbar_wait_cluster(bar, parity, kWaitLimitNs, ab)
                : mbar_wait(bar, parity, kWaitLimitNs, ab);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full(s), 1);   // pair: the even CTA's expect_tx arrive (both CTAs' bytes)
      mbar_init(bar_empty(s), 1);  // the (even CTA's) commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull(a), 1);
      mbar_init(bar_tempty(a), MU * kEpiWarps);  // pair: local + remote epilogue warps
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB0);
    if (!W) prefetch_tmap(&tmB1);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), Sh::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), Sh::TMEM_COLS);
      tmem_relinquish();
    }
  }
  if (warp == 2) {
    // tile_start[e]: tiles of experts < e. DGRAD: row tiles of MU*128 rows x
    // column tiles; WGRAD: a fixed m_blocks / MU x n_tiles per expert.
    constexpr int PER = (MAX_GROUPS + 31) / 32;
    int local[PER], sum = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int e = lane * PER + j;
      int tiles = 0;
      if (e < G) {
        const int b0 = args.boff[e], b1 = args.boff[e + 1];
        seg_a[e] = args.aoff[e];
        seg_b[e] = b0;
        tiles = W ? (args.m_blocks / MU) * args.n_tiles
                  : ((b1 - b0 + MU * BM - 1) / (MU * BM)) * args.n_tiles;
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
      if (e < G) tile_start[e] = run;
      run += local[j];
    }
    if (lane == 31) tile_start[G] = incl;
    if (lane == 0) {
      seg_a[G] = args.aoff[G];
      seg_b[G] = args.boff[G];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) {
    __syncwarp();
    cluster_sync();  // both CTAs' barriers and TMEM exist before any remote use
  }
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = tile_start[G];

  // tile -> expert e, this CTA's 128-row tile / M block m, column tile n
  auto decode = [&](int tile, int& e, int& m, int& n) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_start[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    e = lo;
    const int local = tile - tile_start[e];
    int p;
    if (W) {
      p = local / args.n_tiles;
      n = local - p * args.n_tiles;
    } else {
      const int mt = (seg_b[e + 1] - seg_b[e] + MU * BM - 1) / (MU * BM);
      n = local / mt;
      p = local - n * mt;
    }
    m = p * MU + static_cast<int>(rank);
  };
  auto ksteps = [&](int e) { return W ? (seg_a[e + 1] - seg_a[e]) / BK : args.kb_total; };
  auto fail = [&]() {
    set_status(args.status, MOE_ERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer (every CTA) ----
    int stage = 0;
    uint32_t phase = 0, issued = 0, issued_parity = 0;
    bool ok = true;
    for (int tile = first; tile < total && ok; tile += stride) {
      int e, m, n;
      decode(tile, e, m, n);
      const int nkb = ksteps(e);
      const int bcol = n * BN + static_cast<int>(rank) * Sh::BNL;  // this CTA's B columns
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(bar_empty(stage), phase ^ 1u, kWaitLimitNs, abort_flag)) {
          ok = false;
          break;
        }
        if (leader) mbar_arrive_expect_tx(bar_full(stage), MU * Sh::STAGE);
        const uint32_t fb = PAIR ? map_to_rank(bar_full(stage), 0) : bar_full(stage);
        auto load = [&](uint32_t dst, const CUtensorMap* map, int x, int y) {
          if (PAIR) tma_load_2d_pair(dst, map, fb, x, y);
          else tma_load_2d(dst, map, fb, x, y);
        };
        const uint32_t a_dst = sA + stage * Sh::A_BYTES, b_dst = sB + stage * Sh::B_BYTES;
        if (W) {
          const int ra = seg_a[e] + kb * BK, rb = seg_b[e] + kb * BK;
#pragma unroll
          for (int c = 0; c < BM / 64; ++c) load(a_dst + c * CHUNK, &tmA, args.acol + m * BM + c * 64, ra);
#pragma unroll
          for (int c = 0; c < Sh::BNL / 64; ++c) load(b_dst + c * CHUNK, &tmB0, bcol + c * 64, rb);
        } else {
          load(a_dst, &tmA, kb * BK, seg_a[e] + m * BM);
          const bool first_map = kb < args.kb_split;
          const int krow = e * args.b_rows + (first_map ? kb : kb - args.kb_split) * BK;
#pragma unroll
          for (int c = 0; c < Sh::BNL / 64; ++c)
            load(b_dst + c * CHUNK, first_map ? &tmB0 : &tmB1, bcol + c * 64, krow);
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
      if (leader)  // (pair: the even CTA's full barriers count both CTAs' copies)
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s))
            wait(bar_full(s), (issued_parity >> s) & 1u, nullptr);
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------ MMA issuer (even CTA) ----
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true, issued_any = false;
    for (int tile = first; tile < total && ok; tile += stride) {
      int e, m, n;
      decode(tile, e, m, n);
      const int nkb = ksteps(e);
      if (!wait(bar_tempty(acc), acc_phase ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
      for (int kb = 0; kb < nkb; ++kb) {
        if (!wait(bar_full(stage), phase, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = sA + stage * Sh::A_BYTES, b0 = sB + stage * Sh::B_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = W ? sdesc_mnmajor_sw128(a0 + kk * 2048, CHUNK)
                                : sdesc_kmajor_sw128(a0 + kk * 32);
          const uint64_t bd = sdesc_mnmajor_sw128(b0 + kk * 2048, CHUNK);
          const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
          if (PAIR) mma_bf16_pair(d_tmem, ad, bd, Sh::IDESC, accum);
          else mma_bf16(d_tmem, ad, bd, Sh::IDESC, accum);
        }
        issued_any = true;
        if (PAIR) mma_commit_pair(bar_empty(stage), 0x3);
        else mma_commit(bar_empty(stage));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      // with no K step (an expert without rows) this arrives at once
      if (PAIR) mma_commit_pair(bar_tfull(acc), 0x3);
      else mma_commit(bar_tfull(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) {
      fail();
      if (issued_any) {
        if (PAIR) mma_commit_pair(bar_drain, 0x1);
        else mma_commit(bar_drain);
        mbar_wait(bar_drain, 0, kWaitLimitNs, nullptr);
      }
    }
  } else if (warp >= 2) {
    // ------------------------------------------------ epilogue (every CTA) ----
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    const uint32_t tempty_l0 = PAIR ? map_to_rank(bar_tempty(0), 0) : 0u;
    const uint32_t tempty_l1 = PAIR ? map_to_rank(bar_tempty(1), 0) : 0u;
    for (int tile = first; tile < total; tile += stride) {
      int e, m, n;
      decode(tile, e, m, n);
      const int cnt = seg_b[e + 1] - seg_b[e];
      bool ok = wait(bar_tfull(acc), acc_phase, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const int r = m * BM + q * 32 + lane;  // row of the tile this thread drains
      const uint32_t taddr = tmem_base + static_cast<uint32_t>(acc * BN) +
                             (static_cast<uint32_t>(q * 32) << 16);
      if (W || KIND == DGRAD_STORE) {
        // fp32 rows through a shared-memory transpose: the thread that owns
        // TMEM lane `lane` writes its 32 values as one staging row, then
        // each group of 8 lanes stores one 128-byte row segment (4 rows per
        // instruction, whole sectors) instead of 32 scattered 16-byte pieces.
        float* stg = staging + (warp - 2) * Sh::STG_FLOATS;
        const int r0 = m * BM + q * 32;  // first tile row of this warp
        float* rowbase;                   // row r0 of the output, at this tile's columns
        int nvalid;                       // rows of the warp's 32 that are stored
        if (W) {
          const bool second = args.out2 != nullptr && m * BM >= args.m_split;
          const int mrows = args.out2 ? args.m_split : args.m_blocks * BM;
          rowbase = (second ? args.out2 + (static_cast<size_t>(e) * args.m_split +
                                           (r0 - args.m_split)) * args.ldo
                            : args.out + (static_cast<size_t>(e) * mrows + r0) * args.ldo) +
                    n * BN;
          nvalid = 32;
        } else {
          rowbase = args.out + (static_cast<size_t>(seg_b[e]) + r0) * args.ldo + n * BN;
          nvalid = min(32, max(0, cnt - r0));
        }
        const int sub = lane >> 3, q4 = lane & 7, col4 = q4 * 4;
        if (W && cnt == 0) {
          const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int c = 0; c < BN / 32; ++c)
#pragma unroll
            for (int it = 0; it < 8; ++it)
              *reinterpret_cast<float4*>(rowbase + static_cast<size_t>(it * 4 + sub) * args.ldo +
                                         c * 32 + col4) = z;
        } else if (nvalid > 0) {
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(taddr + c * 32, v);
            tmem_ld_wait();
            // row `lane`, 16-byte chunk j stored at chunk j ^ (lane & 7)
            float4* my = reinterpret_cast<float4*>(stg + lane * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              my[j ^ (lane & 7)] =
                  make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                              __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
            __syncwarp();
#pragma unroll
            for (int it = 0; it < 8; ++it) {
              const int row = it * 4 + sub;
              if (row < nvalid)
                *reinterpret_cast<float4*>(rowbase + static_cast<size_t>(row) * args.ldo +
                                           c * 32 + col4) =
                    *reinterpret_cast<const float4*>(stg + row * 32 + 4 * (q4 ^ (row & 7)));
            }
            __syncwarp();
          }
        }
      } else {
        // (a, b) -> (dh b silu'(a), dh silu(a)), bf16, in place in the padded
        // rows; the pad rows after the expert's last row are written as zeros.
        // The next chunk's (a, b) are loaded while this chunk's accumulator is
        // read and processed, so the global latency overlaps the TMEM read.
        const bool valid = r < cnt;
        const bool pad = !valid && r < ((cnt + BK - 1) / BK) * BK;
        __nv_bfloat16* qa_base =
            args.pre + (static_cast<size_t>(seg_a[e]) + r) * 2 * args.F + n * BN;
        __nv_bfloat16* qb_base = qa_base + args.F;
        const __nv_bfloat16* pa = qa_base;
        const __nv_bfloat16* pb = qb_base;
        if (pad) {
          for (int c = 0; c < BN / 32; ++c)
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
              reinterpret_cast<uint4*>(qa_base + c * 32)[w4] = make_uint4(0u, 0u, 0u, 0u);
              reinterpret_cast<uint4*>(qb_base + c * 32)[w4] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        uint4 ua[4], ub[4];
        if (valid) {
#pragma unroll
          for (int w4 = 0; w4 < 4; ++w4) {
            ua[w4] = reinterpret_cast<const uint4*>(pa)[w4];
            ub[w4] = reinterpret_cast<const uint4*>(pb)[w4];
          }
        }
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint4 na[4], nb[4];
          if (valid && c + 1 < BN / 32) {
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
              na[w4] = reinterpret_cast<const uint4*>(pa + (c + 1) * 32)[w4];
              nb[w4] = reinterpret_cast<const uint4*>(pb + (c + 1) * 32)[w4];
            }
          }
          uint32_t v[32];
          tmem_ld32(taddr + c * 32, v);
          tmem_ld_wait();
          if (valid) {
            uint4* qa = reinterpret_cast<uint4*>(qa_base + c * 32);
            uint4* qb = reinterpret_cast<uint4*>(qb_base + c * 32);
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
              uint32_t* ea = reinterpret_cast<uint32_t*>(&ua[w4]);
              uint32_t* eb = reinterpret_cast<uint32_t*>(&ub[w4]);
#pragma unroll
              for (int p2 = 0; p2 < 4; ++p2) {
                const float2 a2 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&ea[p2]));
                const float2 b2 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&eb[p2]));
                const float dh0 = __uint_as_float(v[w4 * 8 + p2 * 2]);
                const float dh1 = __uint_as_float(v[w4 * 8 + p2 * 2 + 1]);
                // sigmoid with the fast intrinsics: their fp32 error is far
                // below the bf16 rounding of the results
                const float s0 = __fdividef(1.f, 1.f + __expf(-a2.x));
                const float s1 = __fdividef(1.f, 1.f + __expf(-a2.y));
                const __nv_bfloat162 da = __floats2bfloat162_rn(
                    dh0 * b2.x * s0 * (1.f + a2.x * (1.f - s0)),
                    dh1 * b2.y * s1 * (1.f + a2.y * (1.f - s1)));
                const __nv_bfloat162 db =
                    __floats2bfloat162_rn(dh0 * a2.x * s0, dh1 * a2.y * s1);
                ea[p2] = *reinterpret_cast<const uint32_t*>(&da);
                eb[p2] = *reinterpret_cast<const uint32_t*>(&db);
              }
              qa[w4] = ua[w4];
              qb[w4] = ub[w4];
            }
          }
#pragma unroll
          for (int w4 = 0; w4 < 4; ++w4) {
            ua[w4] = na[w4];
            ub[w4] = nb[w4];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(bar_tempty(acc));
        else mbar_arrive_remote(acc == 0 ? tempty_l0 : tempty_l1);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) {
    __syncwarp();
    cluster_sync();  // no CTA of the pair leaves while the other may still signal it
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem_base, Sh::TMEM_COLS);
    else tmem_dealloc(tmem_base, Sh::TMEM_COLS);
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

// Row-major bf16 [rows][cols] as a 2-D tensor map, box box_rows x 64 columns,
// 128-byte swizzle; rows past the end read as zeros.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KIND, int BN, bool PAIR>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                   const BwArgs& args, int64_t tiles_bound, cudaStream_t s) {
  using Sh = BwShape<KIND, BN, PAIR>;
  static std::mutex mu;
  static int done_mask = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!(dev < 31 && (done_mask >> dev) & 1)) {
      const cudaError_t e = cudaFuncSetAttribute(
          grouped_bwd_tc<KIND, BN, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM);
      if (e != cudaSuccess) return e;
      if (dev < 31) done_mask |= 1 << dev;
    }
  }
  const int64_t sms = sm_count();
  if constexpr (!PAIR) {
    const unsigned grid = static_cast<unsigned>(tiles_bound < sms ? tiles_bound : sms);
    if (grid == 0) return cudaSuccess;
    grouped_bwd_tc<KIND, BN, false><<<grid, kThreads, Sh::SMEM, s>>>(a, b0, b1, args);
    return cudaGetLastError();
  } else {
  const int64_t clusters = tiles_bound < sms / 2 ? tiles_bound : sms / 2;
  if (clusters == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Sh::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_bwd_tc<KIND, BN, true>, a, b0, b1, args);
  }
}

// CTA pairs for the weight-gradient products when the experts' rows (an
// upper bound: rows of the workspace, before capacity) average at least 1024,
// i.e. reductions of 16 or more 64-row steps per tile: there they are limited
// by the bytes each SM loads per MMA cycle (measured on the Mixtral-shaped
// layer: 1.08 -> 0.87 ms and 2.12 -> 1.70 ms); with ~200 rows per expert (the
// Switch-shaped layer) pairs lose. The input-gradient products take pairs
// from 512 rows per expert (256-row pair tiles): the SwiGLU-derivative one
// when its reduction over d is >= 1024 (measured: Switch-shaped 0.277 ->
// 0.258 ms, Mixtral-shaped 0.96-0.99 -> 0.92-0.94 ms), the gate/up one
// (reduction over 2F) always (0.252 -> 0.231 ms and 1.49-1.52 -> 1.36 ms).
bool use_pairs(int E, int64_t rows) { return rows >= static_cast<int64_t>(E) * 1024; }

}  // namespace

bool ffn_bwd_tc_supported(const moe_config& c) {
  return ffn_tc_supported(c) && c.n_experts + c.n_shared <= MAX_GROUPS;
}

int ffn_bwd_tc_launches(const moe_config&) { return 4; }

int64_t ffn_bwd_pad_rows(const moe_config& c) {
  return rows_max_of(&c) + static_cast<int64_t>(BK - 1) * (c.n_experts + c.n_shared);
}

moe_status launch_ffn_bwd_tc(const moe_config& c, int64_t rows, int64_t rows_pad,
                             const int32_t* offsets, const int32_t* poff,
                             const moe_expert_weights& w, const void* x_perm, const void* h,
                             void* pre, const void* dout, float* dx_perm, const moe_grads& g,
                             uint32_t* status, cudaStream_t s) {
  if (!ffn_bwd_tc_supported(c)) return MOE_ERR_UNSUPPORTED;
  const int E = c.n_experts + c.n_shared, d = c.d_model, F = c.d_ff;
  const bool f256 = F % 256 == 0;  // column tile along F
  if (rows == 0) {
    // no row at all: the weight gradients are zero
    const size_t wsz = static_cast<size_t>(E) * F * d * sizeof(float);
    for (float* m : {g.dw_gate, g.dw_up, g.dw_down})
      if (cudaMemsetAsync(m, 0, wsz, s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  const bool pairs = use_pairs(E, rows);
  const int64_t mt_bound = E + (rows + BM - 1) / BM;           // (expert, 128-row tile) bound
  CUtensorMap m_dout128, m_dout64, m_h, m_dpre128, m_dpre64, m_x, m_wd, m_wg, m_wu;
  if (!make_map(&m_dout128, dout, rows_pad, d, 128) ||
      !make_map(&m_dout64, dout, rows_pad, d, 64) || !make_map(&m_h, h, rows, F, 64) ||
      !make_map(&m_dpre128, pre, rows_pad, 2 * F, 128) ||
      !make_map(&m_dpre64, pre, rows_pad, 2 * F, 64) || !make_map(&m_x, x_perm, rows, d, 64) ||
      !make_map(&m_wd, w.w_down, static_cast<uint64_t>(E) * d, F, 64) ||
      !make_map(&m_wg, w.w_gate, static_cast<uint64_t>(E) * F, d, 64) ||
      !make_map(&m_wu, w.w_up, static_cast<uint64_t>(E) * F, d, 64))
    return MOE_ERR_CUDA;
  __nv_bfloat16* pre_b = static_cast<__nv_bfloat16*>(pre);
  cudaError_t err;
  // 1. dh = dout . W_down, activation derivative over (a | b) in place
  {
    BwArgs a{poff, offsets, E, d / BK, d / BK, d, F / (f256 ? 256 : 128), 0, 0, 0, nullptr,
             nullptr, 0, pre_b, F, status};
    const bool dpairs = rows >= static_cast<int64_t>(E) * 512 && d >= 1024;  // 256-row pair tiles
    if (f256 && dpairs)
      err = launch<DGRAD_SWIGLU, 256, true>(m_dout128, m_wd, m_wd, a,
                                            (E + (rows + 2 * BM - 1) / (2 * BM)) * a.n_tiles, s);
    else if (f256)
      err = launch<DGRAD_SWIGLU, 256, false>(m_dout128, m_wd, m_wd, a, mt_bound * a.n_tiles, s);
    else
      err = launch<DGRAD_SWIGLU, 128, false>(m_dout128, m_wd, m_wd, a, mt_bound * a.n_tiles, s);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    trace_record(2, s);
  }
  // 2. dW_down[e] = dout_e^T h_e: M = d, N = F
  {
    BwArgs a{poff, offsets, E, 0, 0, 0, F / (f256 ? 256 : 128), d / BM, d, 0, g.dw_down,
             nullptr, F, nullptr, F, status};
    const int64_t tiles = static_cast<int64_t>(E) * a.m_blocks * a.n_tiles;
    if (pairs && f256) err = launch<WGRAD, 256, true>(m_dout64, m_h, m_h, a, tiles / 2, s);
    else if (f256) err = launch<WGRAD, 256, false>(m_dout64, m_h, m_h, a, tiles, s);
    else err = launch<WGRAD, 128, false>(m_dout64, m_h, m_h, a, tiles, s);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    trace_record(3, s);
  }
  // 3. dx_perm = da . W_gate + db . W_up: K = 2F (first F from W_gate), N = d
  {
    BwArgs a{poff, offsets, E, 2 * F / BK, F / BK, F, d / 256, 0, 0, 0, dx_perm, nullptr, d,
             nullptr, F, status};
    const bool spairs = rows >= static_cast<int64_t>(E) * 512;  // 256-row pair tiles
    err = spairs ? launch<DGRAD_STORE, 256, true>(m_dpre128, m_wg, m_wu, a,
                                                 (E + (rows + 2 * BM - 1) / (2 * BM)) * a.n_tiles, s)
                 : launch<DGRAD_STORE, 256, false>(m_dpre128, m_wg, m_wu, a, mt_bound * a.n_tiles, s);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    trace_record(4, s);
  }
  // 4. dW_gate | dW_up [e] = (da | db)_e^T x_perm_e: M = 2F rows split at F, N = d
  {
    BwArgs a{poff, offsets, E, 0, 0, 0, d / 256, 2 * F / BM, F, 0, g.dw_gate, g.dw_up, d,
             nullptr, F, status};
    const int64_t tiles = static_cast<int64_t>(E) * a.m_blocks * a.n_tiles;
    err = pairs ? launch<WGRAD, 256, true>(m_dpre64, m_x, m_x, a, tiles / 2, s)
                : launch<WGRAD, 256, false>(m_dpre64, m_x, m_x, a, tiles, s);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    trace_record(5, s);
  }
  return MOE_OK;
}


// ---- router gradients on the tensor cores ------------------------------------
// dx += dl W_r and dW_r = dl^T x for bf16 layers. dl (fp32) and W_r (fp32)
// are split into bf16 pairs, dl = dl_hi + dl_lo and W_r = W_hi + W_mid, each
// exact to 2^-16 relative; the products keep the three terms above that
// level, dl_hi W_hi + dl_lo W_hi + dl_hi W_mid, as one reduction over
// K = 3 NP (NP = N rounded up to 64): A_r = [dl_hi | dl_lo | dl_hi],
// B_r = [W_hi ; W_hi ; W_mid]. dW_r takes A_r's first 2 NP columns as
// 2 NP output rows (hi then lo parts of dl) against x, over token groups of
// T / G rows each, and a fixed-order reduction adds groups and parts.
namespace {

// A_r has Tp = T rounded up to 64 rows, rows T..Tp zero. goff: G+1 A-row
// group offsets (multiples of 64, the last Tp), G+1 token offsets (the same,
// the last T), then {0, Tp} and {0, T} for the single group of dx.
__global__ void __launch_bounds__(256)
router_bwd_prep_kernel(const float* __restrict__ dl, const float* __restrict__ w_r, int T, int N,
                       int NP, int d, int G, __nv_bfloat16* __restrict__ ar,
                       __nv_bfloat16* __restrict__ br, int32_t* __restrict__ goff) {
  const int Tp = (T + 63) / 64 * 64;
  const size_t na = static_cast<size_t>(Tp) * NP, nb = static_cast<size_t>(NP) * d;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < na + nb;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    if (i < na) {
      const size_t t = i / NP;
      const int e = static_cast<int>(i % NP);
      const float v = (e < N && t < static_cast<size_t>(T)) ? dl[t * N + e] : 0.f;
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
      __nv_bfloat16* row = ar + t * 3 * NP;
      row[e] = hi;
      row[NP + e] = lo;
      row[2 * NP + e] = hi;
    } else {
      const size_t k = i - na;
      const int e = static_cast<int>(k / d), j = static_cast<int>(k % d);
      const float w = e < N ? w_r[static_cast<size_t>(e) * d + j] : 0.f;
      const __nv_bfloat16 hi = __float2bfloat16_rn(w);
      const __nv_bfloat16 mid = __float2bfloat16_rn(w - __bfloat162float(hi));
      br[static_cast<size_t>(e) * d + j] = hi;
      br[(static_cast<size_t>(NP) + e) * d + j] = hi;
      br[(static_cast<size_t>(2 * NP) + e) * d + j] = mid;
    }
  }
  if (blockIdx.x == 0) {
    for (int g = threadIdx.x; g <= G; g += blockDim.x) {
      const int32_t o = g == G ? Tp
                               : static_cast<int32_t>(static_cast<int64_t>(T) * g / G / 64 * 64);
      goff[g] = o;
      goff[G + 1 + g] = g == G ? T : o;
    }
    if (threadIdx.x == 0) {
      goff[2 * G + 2] = 0;
      goff[2 * G + 3] = Tp;
      goff[2 * G + 4] = 0;
      goff[2 * G + 5] = T;
    }
  }
}

// dW_r[e][j] = sum_g (P[g][e][j] + P[g][NP + e][j]), groups ascending.
__global__ void __launch_bounds__(256)
router_wgrad_reduce_kernel(const float* __restrict__ part, int G, int N, int NP, int d,
                           float* __restrict__ dw_r) {
  const size_t n = static_cast<size_t>(N) * d;
  const size_t gs = static_cast<size_t>(2 * NP) * d;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t lo = static_cast<size_t>(NP) * d;
    float s = 0.f;
    for (int g = 0; g < G; ++g) s += part[g * gs + i] + part[g * gs + lo + i];
    dw_r[i] = s;
  }
}

}  // namespace

bool router_bwd_tc_supported(const moe_config& c) {
  return c.dtype == MOE_BF16 && c.d_model % 256 == 0 && c.T > 0;
}

RouterBwdPlan router_bwd_tc_plan(const moe_config& c) {
  RouterBwdPlan p{};
  p.NP = (c.n_experts + 63) / 64 * 64;
  const int tiles_per_group = (2 * p.NP / BM) * (c.d_model / 256);
  int G = (2 * 148 + tiles_per_group - 1) / tiles_per_group;  // about two waves of CTAs
  G = G < 1 ? 1 : (G > 64 ? 64 : G);
  if (G > c.T) G = c.T > 0 ? c.T : 1;
  p.G = G;
  return p;
}

moe_status launch_router_bwd_tc(const moe_config& c, const RouterBwdPlan& p, const float* dl,
                                const float* w_r, const void* x, float* dx, float* dw_r,
                                __nv_bfloat16* ar, __nv_bfloat16* br, int32_t* goff,
                                float* part, uint32_t* status, cudaStream_t s) {
  const int T = c.T, N = c.n_experts, d = c.d_model, NP = p.NP, G = p.G;
  const size_t work = static_cast<size_t>(T) * NP + static_cast<size_t>(NP) * d;
  const unsigned pb = static_cast<unsigned>(
      std::min<size_t>((work + 255) / 256, static_cast<size_t>(sm_count()) * 16));
  router_bwd_prep_kernel<<<pb, 256, 0, s>>>(dl, w_r, T, N, NP, d, G, ar, br, goff);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  const uint64_t Tp = (static_cast<uint64_t>(T) + 63) / 64 * 64;
  CUtensorMap m_ar128, m_ar64, m_br, m_x;
  if (!make_map(&m_ar128, ar, Tp, 3 * NP, 128) || !make_map(&m_ar64, ar, Tp, 3 * NP, 64) ||
      !make_map(&m_br, br, 3 * NP, d, 64) || !make_map(&m_x, x, T, d, 64))
    return MOE_ERR_CUDA;
  // dx = dl W_r: one group of T rows, K = 3 NP, N = d (written; the gather adds the rest)
  {
    BwArgs a{goff + 2 * G + 2, goff + 2 * G + 4, 1, 3 * NP / BK, 3 * NP / BK, 0, d / 256, 0, 0,
             0, dx, nullptr, d, nullptr, 0, status};
    const int64_t tiles = (static_cast<int64_t>(T) + BM - 1) / BM * (d / 256);
    if (launch<DGRAD_STORE, 256, false>(m_ar128, m_br, m_br, a, tiles, s) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  // partial dW_r per token group: M = 2 NP rows (dl_hi | dl_lo), N = d
  {
    BwArgs a{goff, goff + G + 1, G, 0, 0, 0, d / 256, 2 * NP / BM, 2 * NP, 0, part, nullptr, d,
             nullptr, 0, status};
    const int64_t tiles = static_cast<int64_t>(G) * a.m_blocks * a.n_tiles;
    if (launch<WGRAD, 256, false>(m_ar64, m_x, m_x, a, tiles, s) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  const size_t nd = static_cast<size_t>(N) * d;
  const unsigned rb = static_cast<unsigned>(
      std::min<size_t>((nd + 255) / 256, static_cast<size_t>(sm_count()) * 8));
  router_wgrad_reduce_kernel<<<rb, 256, 0, s>>>(part, G, N, NP, d, dw_r);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
