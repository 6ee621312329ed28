/*
 * moe.h — C ABI of libmoe: the forward and backward passes of a sparse
 * Mixture-of-Experts FFN layer on one NVIDIA B300 (sm_103a).
 *
 * Sources (web pages on Mixture-of-Experts layers; cited by title + section):
 *   [MoE核心思想]  "MoE 的核心思想" (wmrh.cn/news/98181): 公式表达重点,
 *                  具体数值示例, 专家容量, 辅助损失公式.
 *   [稀疏激活原理] "MoE 混合专家模型稀疏激活的架构原理与负载均衡挑战"
 *                  (mzlw.cn/news/6844): §2.1 Top-K 路由的决策流程,
 *                  §2.2 负载均衡损失, §2.3 容量因子与 Token 丢弃,
 *                  §三 MoE 层的生产级 PyTorch 实现 (classes Expert,
 *                  MoERouter, MoELayer).
 *   [概念卡]       "混合专家模型（Mixture of Experts, MoE）"
 *                  (learnagent.wiki): 结构 2 路由器, 结构 3 Top-K 选择与输出融合,
 *                  运行示例 (minimal MoELayer).
 *   [替代FFN]      "MoE 如何替代 FFN？它解决了什么问题？带来哪些新挑战？"
 *                  (mstx.cn/posts/467.html): §1 标准 FFN, §2 MoE 如何替代 FFN,
 *                  §4 (3) 路由与梯度.
 *
 * Notation: T tokens, d = d_model, N routed experts, S shared experts,
 * K = top-K, F = d_ff, C = per-expert capacity, A = number of kept
 * (token, rank) assignments, R_max = A_max + S*T rows of permuted tokens.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Memory: the caller owns every buffer. The library never allocates or
 *    frees device memory. All tensor pointers are DEVICE pointers, 16-byte
 *    aligned, row-major and dense (no strides). Scratch space is the caller's
 *    workspace `ws` of at least moe_workspace_size(cfg) bytes, 256-byte
 *    aligned; its contents on entry are ignored.
 *  - Asynchrony: every call only enqueues kernels on `stream` (0 = legacy
 *    default stream) and returns. Results are valid after the stream is
 *    synchronised. No call synchronises or allocates, so after one call on
 *    a device (which sets kernel attributes and looks up the CUDA driver's
 *    tensor-map encoder) the calls can be captured into a CUDA graph and
 *    replayed with the same buffers.
 *  - Errors: every argument error that the host can see (NULL pointer,
 *    misalignment, bad sizes, unsupported combination) is returned before
 *    anything is launched. Errors found on the device (a bounded wait that
 *    timed out, a non-finite router logit, an expert index out of range in
 *    moe_dispatch's input) are OR-ed as (1u << code) into *stats->status
 *    when stats and stats->status are non-NULL; read it after a sync.
 *    The caller zeroes *status before the call if it wants a fresh word.
 *    No C++ exception crosses this ABI.
 *  - Limits: 1 <= K <= min(N, 8); N <= 256; 0 <= S <= 8; 1 <= T <= 2^24
 *    (T = 0 is accepted and does nothing); d % 8 == 0 for bf16, d % 4 == 0
 *    for fp32; F % 4 == 0.
 *  - Determinism: every result is bitwise reproducible run to run (fixed
 *    reduction orders, no floating-point atomics).
 */
#ifndef MOE_B300_H_
#define MOE_B300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (cudaStream_t / CUstream); kept opaque so that this
 * header does not need the CUDA headers. */
typedef void* moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = 1,     /* bad argument (NULL, alignment, size)          */
  MOE_ERR_UNSUPPORTED = 2, /* valid, but outside the limits above           */
  MOE_ERR_CUDA = 3,        /* a CUDA runtime call failed (e.g. launch)      */
  MOE_ERR_TIMEOUT = 4,     /* device: a bounded wait gave up (status word)  */
  MOE_ERR_NONFINITE = 5,   /* device: a router logit was NaN or infinite    */
  MOE_ERR_WORKSPACE = 6,   /* workspace NULL, misaligned or too small       */
  MOE_ERR_INDEX = 7        /* device: an expert index outside [0, N)        */
} moe_status;

enum { MOE_F32 = 0, MOE_BF16 = 1 };      /* dtype of x, expert weights, y   */
enum { MOE_SWIGLU = 0, MOE_GELU = 1 };   /* expert activation               */
/* Gate of a selected expert:
 *   MOE_GATE_RENORM   softmax over the K selected logits (default; [稀疏激活原理]
 *                     §三 MoERouter, [概念卡] 运行示例, [MoE核心思想] 公式表达重点)
 *   MOE_GATE_SOFTMAX  its probability under the softmax over all N experts,
 *                     not renormalised ([稀疏激活原理] §2.1 formula; the Switch
 *                     gate for K = 1)                                        */
enum { MOE_GATE_RENORM = 0, MOE_GATE_SOFTMAX = 1 };

/* Layer configuration (plain old data). */
typedef struct {
  int32_t T;          /* tokens (batch * sequence, flattened)               */
  int32_t d_model;    /* d                                                  */
  int32_t d_ff;       /* F, expert hidden width                             */
  int32_t n_experts;  /* N                                                  */
  int32_t top_k;      /* K                                                  */
  int32_t dtype;      /* MOE_F32 | MOE_BF16                                 */
  int32_t activation; /* MOE_SWIGLU | MOE_GELU                              */
  int32_t has_bias;   /* expert biases present (GELU experts only)          */
  float capacity_factor; /* CF; <= 0 or +inf means no capacity limit       */
  float alpha;        /* coefficient of the load-balance loss               */
  int32_t add_residual; /* 1: y = x + sum_k g*E(x); a fully dropped token's
                           output is then x itself                          */
  int32_t gate_mode;  /* MOE_GATE_RENORM | MOE_GATE_SOFTMAX                 */
  const float* select_bias; /* DEVICE [N] fp32 or NULL: added to the logits for
                           the top-K choice only; gates and statistics use the
                           unbiased logits (auxiliary-loss-free balancing,
                           [概念卡] 结构 4)                                    */
  int32_t n_shared;   /* S in [0, 8]: shared experts, stacked after the N
                           routed ones in every weight array; each takes every
                           token with gate 1, outside the router, the capacity
                           and the statistics ([替代FFN] §5, DeepSeek-MoE)     */
  int32_t save_for_backward; /* 1: moe_forward also keeps in the workspace
                           what moe_backward needs (router logits [T][N] fp32,
                           the expert pre-activations [R_max][2F] in cfg->dtype,
                           the counts) and moe_workspace_size grows by those
                           and by moe_backward's scratch; 0: inference only  */
} moe_config;

/* Device-side statistics; every member is a caller-owned DEVICE pointer and
 * may be NULL (that output is skipped). The whole struct pointer may be NULL.
 *   count[N]   assignments routed to each expert before capacity (int32)
 *   kept[N]    assignments each expert keeps after capacity (int32)
 *   n_dropped  assignments dropped by capacity (one int32)
 *   f[N]       count / (T*K)                            (fp32)
 *   P[N]       mean over tokens of the router softmax   (fp32)
 *   l_aux      alpha * N * sum_e f[e]*P[e]               (one fp32)
 *   status     device error bits, (1u << moe_status)     (one uint32)
 *   z_loss     mean over tokens of (log sum_e exp l[t,e])^2 (one fp32):
 *              the router z-loss ([MoE核心思想] Router Z-Loss, which gives no
 *              formula; read as the squared log-sum-exp)
 *   entropy    mean over tokens of -sum_e p log p        (one fp32):
 *              the routing entropy ([替代FFN] §4 (6))                     */
typedef struct {
  int32_t* count;
  int32_t* kept;
  int32_t* n_dropped;
  float* f;
  float* P;
  float* l_aux;
  uint32_t* status;
  float* z_loss;
  float* entropy;
} moe_stats;

/* Expert weights, stacked over experts, in the nn.Linear (out, in) layout of
 * each expert ([稀疏激活原理] §三 class Expert; [概念卡] 运行示例): the N
 * routed experts, then the S shared ones (E = N + S).
 * Element type is cfg->dtype. Unused members are NULL.
 *   SwiGLU: w_gate [E][F][d], w_up [E][F][d], w_down [E][d][F]
 *   GELU:   w1 [E][F][d], w2 [E][d][F]; biases b1 [E][F], b2 [E][d]
 *           (same dtype), required iff cfg->has_bias.                      */
typedef struct {
  const void* w_gate;
  const void* w_up;
  const void* w_down;
  const void* w1;
  const void* b1;
  const void* w2;
  const void* b2;
} moe_expert_weights;

/* Bytes of workspace that moe_forward needs for cfg (an upper bound for the
 * other entry points too). Pure host function; returns 0 if cfg is invalid.
 * It covers x_perm [R_max][d], h [R_max][F] and o [R_max][d] fp32, where
 * A_max = min(T*K, N*C) and R_max = A_max + S*T; with
 * cfg->save_for_backward also the saved state and the scratch of
 * moe_backward (pre-activations and output gradients [R_max][2F] and
 * [R_max][d] in cfg->dtype, logits and their gradient [T][N] fp32). */
size_t moe_workspace_size(const moe_config* cfg);

/* Capacity C per expert: floor(K * CF * T / N), computed exactly on the
 * rational value of the float CF; INT32_MAX when CF <= 0 or CF = +inf.
 * [稀疏激活原理] §2.3 (capacity_i formula) and §三 MoELayer.forward
 * (capacity = int(top_k / num_experts * capacity_factor * num_tokens), with
 * num_tokens = batch * seq_len). Returns -1 if cfg is invalid. */
int32_t moe_capacity(const moe_config* cfg);

/* Router: logits = x W_r^T (+ b_r), softmax over the N experts, top-K of the
 * logits (ties -> lower expert index; ranked by descending logit), gates =
 * softmax over the K selected logits (the renormalised gate weights), and
 * the load-balance statistics count, f, P, l_aux.
 * [稀疏激活原理] §2.1 (logits = x·W_r, Top-K, then softmax) and §2.2
 * (L_aux = alpha·N·Σ f_i·P_i); [概念卡] 结构 2 (G(x) = Softmax(W_r·x)) and
 * 运行示例 (softmax -> topk -> renormalise); [MoE核心思想] 公式表达重点 and
 * 具体数值示例 (8 experts, top-2, gates 0.67 / 0.33).
 *   x    [T][d]  cfg->dtype        w_r [N][d] fp32      b_r [N] fp32 or NULL
 *   idx  [T][K]  int32 (out)       gate [T][K] fp32 (out)
 *   stats: count, f, P, l_aux, z_loss, entropy, status are written
 *   (kept/n_dropped are not).
 * Errors: MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE,
 * MOE_ERR_CUDA; device: MOE_ERR_NONFINITE. */
moe_status moe_route(const moe_config* cfg, const void* x, const float* w_r,
                     const float* b_r, int32_t* idx, float* gate,
                     moe_stats* stats, void* ws, moe_stream_t stream);

/* moe_route for callers that cannot allocate device memory (the pages have
 * no counterpart: this is an interface variant, not a different method).
 * A serving process whose device memory is all owned by its own pool, or a
 * plug-in interface that passes no workspace, can call this instead of
 * moe_route. It always runs a CUDA-core (FFMA) router and the statistics
 * kernels of moe_route, with the per-block partial sums of the statistics in
 * a fixed array inside the library (1 MiB, held on every GPU that loads the
 * library until the process exits) instead of a caller workspace. Nothing is
 * allocated: no cudaMalloc, no cudaFree.
 *   Results: those of moe_route (for at most 128 tokens and 32 experts both
 *   run the same small-batch router), except that for larger bf16 layers
 *   with d % 64 == 0 moe_route takes the tensor-core router, which sums the
 *   logits in another order: the choice can then differ on near-tie tokens (some
 *   adjacent gap among the K+1 largest logits below 1e-5), and this call can
 *   be slower on those layers.
 *   Limit: ceil(T / 32) * (N + 2) <= 131072 (e.g. T <= 16256 with N = 256,
 *   T <= 419424 with N = 8); beyond it returns MOE_ERR_WORKSPACE before
 *   launching anything.
 *   Set-up: the first call in each CUDA context (normally once per device:
 *   the runtime's primary context) looks up the array's device address
 *   (cudaGetSymbolAddress) with that context current; make that first call
 *   before any stream capture on that device.
 *   Sharing: all calls share the array and it keeps the last call's
 *   contents; each call rewrites every element it reads, so nothing needs
 *   clearing, but calls whose kernels overlap on the GPU (other streams or
 *   host threads) race on it: serialise them.
 * Arguments, outputs and errors are those of moe_route, without ws. */
moe_status moe_route_no_workspace(const moe_config* cfg, const void* x,
                                  const float* w_r, const float* b_r,
                                  int32_t* idx, float* gate, moe_stats* stats,
                                  moe_stream_t stream);

/* Capacity-limited dispatch. Assignments are visited rank-major (k = 0..K-1,
 * then t = 0..T-1); an assignment (t, k) to expert e is kept iff fewer than C
 * earlier assignments went to e. Kept assignments of expert e occupy the
 * contiguous slots [offsets[e], offsets[e+1]) in that visiting order, and
 * x_perm[slot] = x[t]. Dropped assignments get slot_of = -1 and contribute
 * nothing to y (the residual carries the token, [稀疏激活原理] §2.3).
 * Shared expert s (index N + s) takes every token in order: its slots are
 * offsets[N+s] + t with offsets[N+s] = offsets[N] + s*T, recorded as
 * slot_of[t][K+s].
 * [稀疏激活原理] §2.3 and §三 MoELayer.forward (outer loop over top-k rank,
 * tokens in ascending order, truncation at capacity).
 *   x [T][d] cfg->dtype, idx [T][K] int32 (values in [0, N))
 *   offsets [N+S+1] int32 (out), slot_of [T][K+S] int32 (out),
 *   token_of_slot [R_max] int32 (out, first offsets[N] valid),
 *   x_perm [R_max][d] cfg->dtype (out).
 *   stats: count, kept, n_dropped, status are written.
 * Errors: as moe_route; device: MOE_ERR_INDEX (bad idx value; that
 * assignment is treated as dropped). */
moe_status moe_dispatch(const moe_config* cfg, const void* x,
                        const int32_t* idx, int32_t* offsets, int32_t* slot_of,
                        int32_t* token_of_slot, void* x_perm, moe_stats* stats,
                        void* ws, moe_stream_t stream);

/* Grouped expert FFN over the permuted tokens: for every expert e < N + S
 * and every slot s in [offsets[e], offsets[e+1]),
 *   SwiGLU: o[s] = W_down,e (silu(W_gate,e x) * (W_up,e x))
 *   GELU:   o[s] = W2,e gelu_erf(W1,e x + b1,e) + b2,e
 * with x = x_perm[s]; silu(a) = a / (1 + e^-a); gelu_erf(z) =
 * z/2 (1 + erf(z / sqrt 2)). The hidden activation h is rounded to cfg->dtype
 * (bf16 or fp32) before the down projection; o is fp32.
 * [稀疏激活原理] §三 class Expert (SwiGLU); [概念卡] 运行示例
 * (Linear -> GELU -> Linear); [替代FFN] §1 (FFN(x) = W_2 act(W_1 x)).
 *   x_perm [R_max][d] cfg->dtype, offsets [N+S+1] int32 (device, as written
 *   by moe_dispatch), o [R_max][d] fp32 (out). Rows past offsets[N+S]
 *   untouched.
 * Errors: as moe_route; device: MOE_ERR_TIMEOUT. */
moe_status moe_expert_ffn(const moe_config* cfg, const void* x_perm,
                          const int32_t* offsets,
                          const moe_expert_weights* weights, float* o,
                          moe_stats* stats, void* ws, moe_stream_t stream);

/* Gate-weighted combine: y[t] = sum over k ascending with slot_of[t][k] >= 0
 * of gate[t][k] * o[slot_of[t][k]], then + o[slot_of[t][K+s]] for the
 * shared experts s ascending (gate 1), accumulated in fp32 and rounded once
 * to cfg->dtype; plus x[t] when cfg->add_residual. No atomics.
 * [概念卡] 结构 3 (y = Σ_{i∈TopK} G(x)_i E_i(x)); [替代FFN] §2 (MoE(x) formula);
 * [稀疏激活原理] §2.1.
 *   o [R_max][d] fp32, slot_of [T][K+S] int32, gate [T][K] fp32,
 *   x [T][d] (read only if add_residual; may be NULL otherwise),
 *   y [T][d] cfg->dtype (out).
 * Errors: MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
moe_status moe_combine(const moe_config* cfg, const float* o,
                       const int32_t* slot_of, const float* gate,
                       const void* x, void* y, moe_stream_t stream);

/* The whole layer: moe_route -> moe_dispatch -> moe_expert_ffn ->
 * moe_combine on one stream, with every intermediate in the workspace.
 * [稀疏激活原理] §三 MoELayer.forward; [概念卡] 核心原理 (four steps).
 *   x [T][d], w_r [N][d] fp32, b_r [N] fp32 or NULL, weights as above,
 *   y [T][d] (out), stats (all members optional), ws >= moe_workspace_size.
 *   With T = 0, x and y may be NULL.
 * Errors: the union of the above. */
moe_status moe_forward(const moe_config* cfg, const void* x, const float* w_r,
                       const float* b_r, const moe_expert_weights* weights,
                       void* y, moe_stats* stats, void* ws,
                       moe_stream_t stream);

/* Gradients written by moe_backward: caller-owned DEVICE fp32 buffers, each
 * overwritten (not accumulated). E = N + S; shapes follow the weights.
 *   dx [T][d] and dw_r [N][d] are required; db_r [N] may be NULL.
 *   SwiGLU: dw_gate [E][F][d], dw_up [E][F][d], dw_down [E][d][F].
 *   GELU:   dw1 [E][F][d], dw2 [E][d][F]; db1 [E][F], db2 [E][d] iff
 *           cfg->has_bias. Members of the other activation are ignored.   */
typedef struct {
  float* dx;
  float* dw_r;
  float* db_r;
  float* dw_gate;
  float* dw_up;
  float* dw_down;
  float* dw1;
  float* db1;
  float* dw2;
  float* db2;
} moe_grads;

/* Backward pass: the gradients of the training objective
 *   L = sum_{t,j} dy[t][j] * y[t][j] + L_aux + z_coef * z_loss
 * (dy = dLoss/dy of whatever follows the layer; L_aux = alpha*N*sum f*P and
 * z_loss as reported in moe_stats) with respect to x, W_r, b_r and every
 * expert weight. The top-K choice, the capacity truncation and the selection
 * bias are piecewise constant and pass no gradient ([稀疏激活原理] §四
 * 训练不稳定性: the expert choice itself has zero gradient, the gate softmax
 * is differentiable; [替代FFN] §4 (3)); f is a count and passes none, P
 * carries L_aux's gradient ([稀疏激活原理] §2.2); the router receives
 * gradient through the gates, P and the z-loss ([概念卡] 结构 2: trained end
 * to end); a dropped assignment passes none; shared experts receive dy.
 * Steps (all on the GPU): gate and output gradients of the combine; logit
 * gradient; per expert, the down projection's input and weight gradients
 * (with the activation's derivative), the first projection's input and
 * weight gradients; dx = residual + sum of the expert input gradients +
 * dlogits W_r; dW_r = dlogits^T x.
 * Precondition: ws holds the state of the latest moe_forward with the same
 * cfg (save_for_backward = 1), x, w_r, b_r and weights, unchanged since.
 *   x [T][d] cfg->dtype, w_r [N][d] fp32, weights as in moe_forward,
 *   dy [T][d] cfg->dtype, z_coef >= 0 (finite), grads as above (x, dy and
 *   grads->dx may be NULL when T = 0; every weight gradient is then zero).
 * Intermediate gradients are rounded to cfg->dtype where they feed a
 * tensor-core product (the expert output gradient g*dy and the
 * pre-activation gradients), as the forward rounds h.
 * Errors: MOE_ERR_INVALID (NULL or misaligned pointers, z_coef not finite or
 * negative, cfg->save_for_backward == 0), MOE_ERR_UNSUPPORTED,
 * MOE_ERR_WORKSPACE, MOE_ERR_CUDA; device: MOE_ERR_TIMEOUT. */
moe_status moe_backward(const moe_config* cfg, const void* x, const float* w_r,
                        const moe_expert_weights* weights, const void* dy,
                        float z_coef, moe_grads* grads, moe_stats* stats,
                        void* ws, moe_stream_t stream);

/* ---- Expert-parallel staging ------------------------------------------
 * The local data movement around the two all-to-alls of an expert-parallel
 * layer ("MoE 的核心思想", Expert Parallelism and 前向传播中的 All-to-All 通信:
 * the experts are spread over R devices; in the dispatch step every device
 * sends its tokens to the devices that hold their experts, each device runs
 * its own experts on what it received, and in the combine step the outputs
 * return to their source devices for the gate-weighted sum). These calls
 * only lay rows out on one device; the caller exchanges the buffers with its
 * own collective (e.g. an all-to-all with the split sizes below).
 * Placement: owner[e] in [0, R) is the device that holds expert e (DEVICE
 * [N] int32); the pages name no placement. Capacity and dispatch stay per
 * source device (moe_dispatch on its own tokens). Shared experts are not
 * exchanged: these calls need cfg->n_shared == 0 (MOE_ERR_UNSUPPORTED).
 * Every call is two launches on `stream`: a one-block plan kernel that writes
 * position tables into ws (>= moe_ep_workspace_size bytes, 256-byte aligned;
 * contents on entry ignored) and a row-copy kernel. Rows move bit for bit.
 * Device-detected errors go to stats->status (stats may be NULL) and then
 * no row is written: MOE_ERR_INDEX for an owner outside [0, R), a negative
 * count or offsets that no dispatch writes; MOE_ERR_WORKSPACE when a
 * device would receive more than rows_cap rows. Limits: 1 <= R <= 256. */

/* Bytes of workspace the four calls below need for cfg and R devices
 * (about 8 * N * R bytes); 0 if cfg or n_ranks is invalid. */
size_t moe_ep_workspace_size(const moe_config* cfg, int32_t n_ranks);

/* Dispatch step, source device: x_perm [A_max][d] (cfg->dtype, expert e at
 * rows [offsets[e], offsets[e+1]) as moe_dispatch writes them) laid out by
 * destination into send [A_max][d]: destination r ascending, then r's
 * experts ascending, then each expert's rows in slot order.
 * send_counts [R] int32 (DEVICE, out): rows for each destination (their
 * exclusive prefix sums are the send offsets). The rows sent to r hold
 * kept[e] rows for each of r's experts e ascending, so a receiver knows its
 * layout from every source's kept[N] (gathered into kept_all below). */
moe_status moe_ep_pack(const moe_config* cfg, int32_t n_ranks, const int32_t* owner,
                       const int32_t* offsets, const void* x_perm, void* send,
                       int32_t* send_counts, moe_stats* stats, void* ws,
                       moe_stream_t stream);

/* Local-compute set-up on device `rank`: recv (rows from every source s
 * ascending, each source's rows for this device in the order it sent them)
 * rearranged into x_local, expert-major: this device's experts ascending
 * (local index j), then sources ascending. kept_all [R][N] int32 (DEVICE):
 * kept[e] of every source s. local_offsets [N+1] int32 (DEVICE, out):
 * local expert j's rows are [local_offsets[j], local_offsets[j+1]) for j <
 * E_r (the number of experts with owner == rank); entries E_r..N hold the
 * total. recv and x_local hold rows_cap rows of d elements (cfg->dtype).
 * The experts then run with moe_expert_ffn on a config with n_experts = E_r,
 * top_k = 1, no capacity and T >= the total rows, the offsets
 * local_offsets and the weights of this device's experts stacked in
 * ascending expert order. */
moe_status moe_ep_regroup(const moe_config* cfg, int32_t n_ranks, int32_t rank,
                          const int32_t* owner, const int32_t* kept_all, int64_t rows_cap,
                          const void* recv, void* x_local, int32_t* local_offsets,
                          moe_stats* stats, void* ws, moe_stream_t stream);

/* The inverse of moe_ep_regroup on the expert outputs: o_local [rows_cap][d]
 * fp32 in expert-major order put back into receive order in back
 * [rows_cap][d] fp32, ready for the combine all-to-all (which returns to
 * each source the rows it sent, in the order it sent them). */
moe_status moe_ep_regroup_back(const moe_config* cfg, int32_t n_ranks, int32_t rank,
                               const int32_t* owner, const int32_t* kept_all,
                               int64_t rows_cap, const float* o_local, float* back,
                               moe_stats* stats, void* ws, moe_stream_t stream);

/* Combine step, source device: the inverse of moe_ep_pack on the returned
 * expert outputs: back [A_max][d] fp32 in send order put at their slots in
 * o [A_max][d] fp32, so that moe_combine forms y exactly as on one device. */
moe_status moe_ep_unpack(const moe_config* cfg, int32_t n_ranks, const int32_t* owner,
                         const int32_t* offsets, const float* back, float* o,
                         moe_stats* stats, void* ws, moe_stream_t stream);

/* Tracing (instrumentation; the pages have no counterpart). Registers up to
 * 8 caller-created CUDA events (cudaEvent_t, passed as void*) for the
 * calling host thread; n = 0 clears them. While registered, moe_forward and
 * moe_backward record them on their stream at their stage boundaries:
 *   moe_forward:  [0] before the router, [1] after the router and
 *     statistics, [2] after the dispatch, [3] after the gate/up (or first
 *     Linear) grouped GEMM, [4] after the down grouped GEMM, [5] after the
 *     combine;
 *   moe_backward: [0] at the start, [1] after the combine and router
 *     backward, [2] after the down projection's input gradient, [3] after
 *     its weight gradient, [4] after the first projection's input gradient,
 *     [5] after its weight gradient, [6] after dx, [7] after the router
 *     weight gradient.
 * Events beyond n are not recorded. The library does not own, create or
 * destroy the events. On a stream that is being captured into a CUDA graph
 * they are recorded as external event-record nodes, so every replay of the
 * graph records them again.
 * Errors: MOE_ERR_INVALID (n outside [0, 8], or events NULL with n > 0). */
moe_status moe_trace_events(void* const* events, int32_t n);

/* Self-test of failure detection (the pages have no counterpart). Launches
 * one thread that waits, with the same bounded wait every mbarrier wait of
 * the tensor-core kernels uses, on an mbarrier that nothing arrives at; after
 * limit_us microseconds of wall time it gives up, ORs (1u << MOE_ERR_TIMEOUT)
 * into *status (device pointer) and returns normally. Nothing faults, traps
 * or hangs. limit_us in [1, 10^7].
 * Errors: MOE_ERR_INVALID (status NULL, limit out of range), MOE_ERR_CUDA. */
moe_status moe_selftest_bounded_wait(uint32_t limit_us, uint32_t* status,
                                     moe_stream_t stream);

/* Static, NUL-terminated description of a status code. Never NULL. */
const char* moe_status_string(moe_status s);

/* Number of kernels one moe_forward call on cfg launches (with every member
 * of stats non-NULL; one more with save_for_backward on the tensor-core
 * path), for accounting by benchmarks and tracers; -1 if cfg is invalid.
 * Instrumentation; the pages have no counterpart. */
int32_t moe_forward_launch_count(const moe_config* cfg);

/* Number of kernels one moe_backward call on cfg launches (with db_r
 * non-NULL; two fewer without it, none for T = 0); -1 if cfg is invalid or
 * has save_for_backward == 0. Instrumentation. */
int32_t moe_backward_launch_count(const moe_config* cfg);

/* 1 if the expert FFN of cfg runs on the tcgen05 tensor-core path, 0 if it
 * runs on the CUDA-core path (fp32 configurations, or shapes whose d is not a
 * multiple of 64 or F not a multiple of 128), -1 if cfg is invalid. */
int32_t moe_ffn_uses_tensor_cores(const moe_config* cfg);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H_ */
