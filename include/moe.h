/*
 * moe.h - C ABI of a B300-native (sm_103a) forward pass of a Mixture-of-Experts
 * FFN layer on one GPU: router logits -> top-K routing -> dispatch layout ->
 * permute -> grouped SwiGLU FFN -> weighted combine.
 *
 * Sources (cited by page title and section):
 *  [overview] "专家并行 / 总览" (t6page.pages.dev): glossary table
 *             tbl-ep-overview-glossary (Router, top-K, Dispatch, Combine, EP 组,
 *             Expert group, Balancedness); "MoE 路由机制是什么" (the flow Router ->
 *             Dispatch -> Expert Compute -> Combine); "Dispatch 通信矩阵" (eq.
 *             par-ep-dispatch-matrix, expert_id / experts_per_chip = chip_id);
 *             "通信量公式" (eqs. par-ep-comm-total / per-chip / pair).
 *  [notes]    "专家并行与 MoE" (note.yj-dis.top): "MoE 结构回顾" (router, capacity
 *             factor, token drop); "负载均衡" (aux-loss-free per-expert bias;
 *             drop/pad).
 *  [compass]  "專家並行（Expert Parallelism, EP）" (compassingai.com): "技術原理"
 *             (route, dispatch, expert compute, weighted combine); "關鍵引數與考量"
 *             (capacity factor).
 *  [serving]  "MoE 服務的專家並行性" (aiunderstanding.org): "技術洞察" (capacity,
 *             drop or pad so every expert GEMM has a predictable shape).
 *  [lqhl]     "Expert-Parallelism" (papers.lqhl.me): design routes (fused
 *             operators, index lists instead of routing buffers).
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller, except the
 *    two host buffers of moe_layer_forward_host and moe_block_forward_host.
 *    The library never allocates or frees memory.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and does not synchronise the host, except moe_check.
 *    Kernels are launched with programmatic stream serialisation: a kernel
 *    may be scheduled while the stream's previous kernel finishes, but it
 *    waits for that kernel's completion before touching memory, so results
 *    follow plain stream order (also under stream capture).
 *  - Arguments are validated on the host before any launch; a bad argument
 *    returns an error status and launches nothing.  There is no CPU fallback.
 *  - Row-major layouts, the last index contiguous.  "dtype" tensors hold
 *    float32 (MOE_F32) or bfloat16 (MOE_BF16) elements.
 *  - Tensor pointers of dtype must be 16-byte aligned; int32/float32 index and
 *    weight arrays 4-byte aligned; int64 arrays 8-byte aligned.
 *  - Device-side failures (a bounded wait that ran out, an out-of-range expert
 *    id) set a sticky per-device error word; moe_check reports and clears it.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,          /* NULL config/pointer, size out of range */
  MOE_ERR_UNSUPPORTED = 2,          /* valid but not implemented combination */
  MOE_ERR_ALIGNMENT = 3,            /* pointer misaligned (see conventions) */
  MOE_ERR_WORKSPACE_TOO_SMALL = 4,  /* workspace_bytes below moe_workspace_size */
  MOE_ERR_CUDA = 5,                 /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE_TIMEOUT = 6,       /* a bounded device-side wait ran out */
  MOE_ERR_DEVICE_BAD_INDEX = 7      /* an expert id outside [0, E) reached the device */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;
typedef enum { MOE_SOFTMAX = 0, MOE_SIGMOID = 1 } moe_score;
typedef enum {
  MOE_OP_LAYOUT = 0,      /* moe_dispatch_layout */
  MOE_OP_FFN = 1,         /* moe_grouped_ffn */
  MOE_OP_LAYER = 2,       /* moe_layer_forward */
  MOE_OP_LAYER_HOST = 3,  /* moe_layer_forward_host */
  MOE_OP_SHARED = 4,      /* moe_shared_ffn */
  MOE_OP_BLOCK = 5,       /* moe_block_forward */
  MOE_OP_BLOCK_HOST = 6,  /* moe_block_forward_host */
  MOE_OP_FFN_FP8 = 7,     /* moe_grouped_ffn_fp8 */
  MOE_OP_LAYER_FP8 = 8,   /* moe_layer_forward_fp8 */
  MOE_OP_LOGITS = 9,      /* moe_router_logits */
  MOE_OP_FFN_COMBINE = 10 /* moe_grouped_ffn_combine */
} moe_op;

/* Layer description.  Limits: T >= 0; h % 64 == 0; I % 64 == 0; 1 <= E <= 1024;
 * 1 <= K <= min(E, 16); T*K and the permuted row count below 2^31.  "Experts"
 * below means the P = E + n_redundant physical experts wherever the call works
 * after routing (counts, kept, offsets, capacity, n_ij, the FFN's segments). */
typedef struct moe_config {
  int32_t T;            /* tokens (the pages' B) */
  int32_t h;            /* hidden size */
  int32_t E;            /* routed experts */
  int32_t K;            /* experts per token (top-K) */
  int32_t I;            /* expert intermediate size (SwiGLU) */
  int32_t dtype;        /* moe_dtype of activations, weights and outputs */
  int32_t score;        /* moe_score: softmax over experts or elementwise sigmoid */
  int32_t renormalize;  /* 1: chosen weights are divided by their sum */
  float scale;          /* routed scaling factor applied to the weights */
  int32_t n_groups;     /* 0: no group limit; else E % n_groups == 0, n_groups <= 32 */
  int32_t topk_groups;  /* groups kept per token (group-limited routing) */
  int32_t group_topn;   /* a group's score = sum of its group_topn largest keys */
  int32_t capacity;     /* 0: dropless; > 0: per-expert cap, overflow dropped in token order */
  int32_t pad;          /* 1 (needs capacity > 0): expert e owns rows [e*cap, (e+1)*cap) */
  int32_t ep_size;      /* virtual expert-parallel group size N_EP; E % ep_size == 0 */
  int32_t shared_I;     /* intermediate size of the shared expert (0: none); % 64 == 0 */
  int32_t n_redundant;  /* replicas beyond the E logical experts (load balancing, 0: none);
                         * E + n_redundant <= 1024 physical experts, a multiple of ep_size.
                         * Routing chooses among the E logical experts; layout, permute,
                         * FFN and combine work on the E + n_redundant physical ones. */
} moe_config;

/* Scalar results of moe_dispatch_layout (device memory, 32 bytes). */
typedef struct moe_layout_stats {
  int64_t kept_total;       /* assignments kept (permuted rows that carry a token) */
  int64_t dropped;          /* T*K - kept_total */
  int64_t offdiag_rows;     /* sum of n_ij over i != j: rows that would cross chips */
  int32_t experts_touched;  /* experts with at least one kept row */
  float balancedness;       /* sum_j recv_j / (N_EP * max_j recv_j); 1 if nothing received */
} moe_layout_stats;

/* Stages of the layer calls, in execution order.  A stage a configuration does
 * not have (the replica map without replicas, the shared expert outside the
 * block) takes no time. */
enum moe_layer_stage {
  MOE_STAGE_LOGITS = 0,
  MOE_STAGE_ROUTE = 1,
  MOE_STAGE_EPLB_MAP = 2,
  MOE_STAGE_LAYOUT = 3,
  MOE_STAGE_PERMUTE = 4,
  MOE_STAGE_FFN = 5,
  MOE_STAGE_SHARED = 6,
  MOE_STAGE_COMBINE = 7,
  MOE_LAYER_STAGES = 8
};

/* Optional device outputs of moe_layer_forward.  Any NULL member is kept in the
 * workspace instead.  Shapes as in the individual calls below.
 *
 * stage_events: NULL, or MOE_LAYER_STAGES + 1 cudaEvent_t handles (created by
 * the caller, owned by the caller).  The layer records stage_events[0] on its
 * stream before its first kernel and stage_events[s + 1] after stage s
 * (moe_layer_stage), so cudaEventElapsedTime(stage_events[s],
 * stage_events[s + 1]) is the device time of stage s inside the one call.
 * An entry may be NULL: that event is not recorded (an event between two
 * kernels keeps the second from being scheduled while the first drains, so a
 * caller timing one stage passes only that stage's two events).
 * Ignored by the host-buffer calls. */
typedef struct moe_layer_out {
  float* logits;            /* [T, E] */
  int32_t* topk_ids;        /* [T, K] */
  float* topk_w;            /* [T, K] */
  int32_t* counts;          /* [E] */
  int32_t* kept;            /* [E] */
  int32_t* offsets;         /* [E + 1] */
  int32_t* slot;            /* [T, K] */
  int32_t* row_src;         /* [R] */
  int64_t* n_ij;            /* [N_EP, N_EP] */
  int64_t* rank_bytes;      /* [2, N_EP]: sent then received bytes per chip */
  moe_layout_stats* stats;  /* [1] */
  void* const* stage_events; /* [MOE_LAYER_STAGES + 1] cudaEvent_t, or NULL */
} moe_layer_out;

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status s);

/* Checks a configuration against the limits above (host only, no CUDA call). */
moe_status moe_validate_config(const moe_config* cfg);

/* Rows R of the permuted buffers: T*K, or E*capacity when pad is set. */
moe_status moe_rows(const moe_config* cfg, int64_t* rows);

/* Workspace bytes needed by `op`, one of moe_op (the call named beside each;
 * host only). */
moe_status moe_workspace_size(const moe_config* cfg, int32_t op, size_t* bytes);

/* Kernels this library has launched in the process so far (every successful
 * launch, any stream or device).  Reading it before and after a region counts
 * the region's launches; it is never reset.  Host only, thread-safe. */
uint64_t moe_launch_count(void);

/* Zero-fills a workspace.  Must run once after allocation, and again after a call
 * on it returned MOE_ERR_DEVICE_TIMEOUT; calls that succeed leave it reusable. */
moe_status moe_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Router logits ([overview] glossary "Router"): logits[t,e] = sum_j x[t,j] w_r[e,j]
 * (+ logit_offset[e]), float32 accumulation.  x [T,h] dtype; w_r [E,h] dtype;
 * logit_offset [E] float32 or NULL; logits [T,E] float32.  bf16 layers cut the
 * sum over j into up to 8 slices (chosen from T, E, h and the SM count) whose
 * float32 partial sums are added in slice order, so a result never depends on
 * timing.  workspace: workspace_bytes >= moe_workspace_size(MOE_OP_LOGITS),
 * 256-byte aligned (else MOE_ERR_WORKSPACE_TOO_SMALL / MOE_ERR_ALIGNMENT before
 * any launch); float32 layers ignore it (NULL allowed).  One call at a time per
 * workspace. */
moe_status moe_router_logits(const moe_config* cfg, const void* x, const void* w_r,
                             const float* logit_offset, float* logits, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Top-K routing ([overview] glossary "top-K"; [notes] "负载均衡": the aux-loss-free
 * per-expert bias steers selection only; [overview] glossary "Expert group").
 * Scores s = softmax(logits) or sigmoid(logits) in float64.  Selection key
 * fl32(s + sel_bias) (logits themselves for softmax without bias or groups).
 * Group limit: keep the topk_groups groups with the largest float32 sum of their
 * group_topn best keys (ties to the lower group).  Top-K by key descending,
 * ties to the lower id, written in that order.  Weights: unbiased scores of the
 * chosen experts, divided by their sum if renormalize, times scale, float32.
 * logits [T,E] float32; sel_bias [E] float32 or NULL; topk_ids [T,K] int32;
 * topk_w [T,K] float32. */
moe_status moe_route(const moe_config* cfg, const float* logits, const float* sel_bias,
                     int32_t* topk_ids, float* topk_w, void* stream);

/* Dispatch layout ([overview] "Dispatch 通信矩阵", eq. par-ep-dispatch-matrix;
 * [compass] "關鍵引數與考量"; [notes] "负载均衡" drop/pad).  Histogram and a stable
 * rank of every assignment (t,k) inside its expert in token order (one pass,
 * decoupled look-back); capacity drop in token order; offsets = exclusive scan of
 * kept (pad: e*capacity); slot[t,k] = offsets[e] + rank or -1 if dropped;
 * row_src[r] = token of permuted row r or -1; n_ij[i][j] = kept assignments from
 * chip i = t*N_EP/T to chip j = e/(E/N_EP); rank_bytes = n_ij row/column sums times
 * h*dtype_size; stats as in moe_layout_stats.
 * topk_ids [T,K] int32; counts, kept [E] int32; offsets [E+1] int32; slot [T,K]
 * int32; row_src [R] int32; n_ij [N_EP,N_EP] int64; rank_bytes [2,N_EP] int64;
 * stats [1]; workspace >= moe_workspace_size(MOE_OP_LAYOUT), initialised once. */
moe_status moe_dispatch_layout(const moe_config* cfg, const int32_t* topk_ids, int32_t* counts,
                               int32_t* kept, int32_t* offsets, int32_t* slot, int32_t* row_src,
                               int64_t* n_ij, int64_t* rank_bytes, moe_layout_stats* stats,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Largest scratch moe_dispatch_layout_static can use (bytes of device memory
 * held by every GPU that loads the library, until the process exits). */
#define MOE_LAYOUT_STATIC_SCRATCH_BYTES ((size_t)1 << 20)

/* moe_dispatch_layout without a workspace, for callers that cannot allocate
 * device memory and have none to lend: for example code running inside a host
 * framework that owns all device memory through its own allocator and forbids
 * direct allocations, or a latency-critical loop that cannot afford the implicit
 * device synchronisation of cudaMalloc.  The pages have no counterpart of this
 * call; it exists for such callers only.
 *
 * Same arguments, outputs and checks as moe_dispatch_layout, minus the
 * workspace.  The look-back scratch lives in a fixed device array of
 * MOE_LAYOUT_STATIC_SCRATCH_BYTES inside the library; a configuration whose
 * layout needs more (moe_workspace_size(cfg, MOE_OP_LAYOUT) above that limit)
 * is refused with MOE_ERR_WORKSPACE_TOO_SMALL before any launch.  The call
 * allocates nothing: no cudaMalloc, no cudaFree.  Its first call on a device
 * looks up the array's device address for that device (cudaGetSymbolAddress),
 * so make that first call before any stream capture; the address is kept for
 * the life of the process, so after cudaDeviceReset on a device this call must
 * not be used on that device again.  Every call clears the
 * part of the array that must start at zero.  All calls on a device share the
 * one array: two calls that overlap on the GPU (different streams, no ordering
 * between them) race and give wrong results; serialise them. */
moe_status moe_dispatch_layout_static(const moe_config* cfg, const int32_t* topk_ids, int32_t* counts,
                                      int32_t* kept, int32_t* offsets, int32_t* slot, int32_t* row_src,
                                      int64_t* n_ij, int64_t* rank_bytes, moe_layout_stats* stats, void* stream);

/* Permute: the on-device stand-in for the dispatch All-to-All ([overview] glossary
 * "Dispatch"; [compass] "技術原理" step 2).  xp[slot[t,k]] = x[t] for every kept
 * (t,k); with pad, rows whose row_src is -1 are zero-filled; other rows are not
 * written.  x [T,h] dtype; slot [T,K]; row_src [R] (read only with pad; may be
 * NULL otherwise); xp [R,h] dtype. */
moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* slot,
                       const int32_t* row_src, void* xp, void* stream);

/* Grouped SwiGLU FFN over ragged expert segments ([compass] "技術原理" step 3;
 * [serving] "技術洞察": grouped GEMM).  For every expert e and row r in
 * [offsets[e], offsets[e] + kept[e]): a = silu(xp[r] Wg_e^T) * (xp[r] Wu_e^T),
 * stored in dtype; yp[r] = a Wd_e^T, stored in dtype.  float32 accumulation.
 * xp [R,h] dtype; offsets [E+1]; kept [E]; w13 [E,2I,h] dtype (gate rows 0..I-1
 * then up rows I..2I-1); w2 [E,h,I] dtype; yp [R,h] dtype (rows outside the
 * segments are not written); workspace >= moe_workspace_size(MOE_OP_FFN). */
moe_status moe_grouped_ffn(const moe_config* cfg, const void* xp, const int32_t* offsets,
                           const int32_t* kept, const void* w13, const void* w2, void* yp,
                           void* workspace, size_t workspace_bytes, void* stream);

/* moe_permute and moe_grouped_ffn in one: the gate/up GEMM reads every row of
 * an expert's segment straight from x through row_src (16-byte copies into the
 * tensor cores' shared-memory layout), so no permuted copy of x is written or
 * read ("index lists instead of routing buffers": [lqhl] "Expert-Parallelism",
 * design routes, route 5).  x [T,h] bf16; row_src [R] from
 * moe_dispatch_layout; other arguments as in moe_grouped_ffn; bf16 layers
 * whose experts are expected to see at most 160 rows (else
 * MOE_ERR_UNSUPPORTED).  It saves the R x h permuted copy of x (470 MB at the
 * DeepSeek-V3 shape); the rows are gathered once per feature tile, and on B300
 * that costs a few percent more than moe_permute + moe_grouped_ffn, so the
 * layer calls permute explicitly. */
moe_status moe_grouped_ffn_gather(const moe_config* cfg, const void* x, const int32_t* row_src,
                                  const int32_t* offsets, const int32_t* kept, const void* w13, const void* w2,
                                  void* yp, void* workspace, size_t workspace_bytes, void* stream);

/* moe_grouped_ffn and moe_combine in one: the weighted combine is fused into
 * the down projection's epilogue ([serving] "MoE 服務專家並行的未來": fused
 * dispatch-compute-combine kernels; [lqhl] "Expert-Parallelism", design
 * routes, route 5).  Every expert output row is still staged in yp; each
 * stored 32-feature piece of a row counts one arrival for its (token, feature
 * group), and the K-th arrival computes y[t, group] = sum_k topk_w[t,k] *
 * yp[slot[t,k], group] with float32 fused multiply-adds in k order and stores
 * it in bf16: bit-identical to moe_combine on the same yp.  Arguments as in
 * moe_grouped_ffn, plus row_src [R], slot [T,K] and topk_w [T,K] from
 * moe_dispatch_layout / moe_route, and y [T,h] bf16.  bf16, dropless
 * (capacity 0), no replicas, experts expected to see at most 160 rows (else
 * MOE_ERR_UNSUPPORTED).  workspace >= moe_workspace_size(MOE_OP_FFN_COMBINE),
 * zero-filled once by moe_workspace_init: its arrival counters are left at
 * zero by every call that completes (re-initialise it after
 * MOE_ERR_DEVICE_TIMEOUT).  Calls that overlap on the GPU must not share a
 * workspace. */
moe_status moe_grouped_ffn_combine(const moe_config* cfg, const void* xp, const int32_t* offsets,
                                   const int32_t* kept, const void* w13, const void* w2, const int32_t* row_src,
                                   const int32_t* slot, const float* topk_w, void* yp, void* y, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* Weighted combine ([compass] "技術原理" step 4; [overview] glossary "Combine"):
 * y[t] = sum_{k: slot[t,k] >= 0} topk_w[t,k] * yp[slot[t,k]], float32 sum in k order,
 * stored in dtype; dropped assignments contribute nothing (no renormalisation).
 * yp [R,h] dtype; slot [T,K]; topk_w [T,K] float32; y [T,h] dtype. */
moe_status moe_combine(const moe_config* cfg, const void* yp, const int32_t* slot,
                       const float* topk_w, void* y, void* stream);

/* The whole layer ([overview] "MoE 路由机制是什么"): router_logits -> route ->
 * dispatch_layout -> permute -> grouped_ffn -> combine on one stream.
 * x [T,h]; w_r [E,h]; logit_offset, sel_bias [E] float32 or NULL; w13, w2 as in
 * moe_grouped_ffn; y [T,h]; out: optional extra outputs (NULL = none);
 * workspace >= moe_workspace_size(MOE_OP_LAYER), initialised once. */
moe_status moe_layer_forward(const moe_config* cfg, const void* x, const void* w_r,
                             const float* logit_offset, const float* sel_bias, const void* w13,
                             const void* w2, void* y, const moe_layer_out* out, void* workspace,
                             size_t workspace_bytes, void* stream);

/* moe_layer_forward with HOST activations: copies x_host [T,h] (pinned host
 * memory recommended) to the device, runs the layer, and copies y back to
 * y_host [T,h], all asynchronously on `stream`; weights stay on the device.
 * workspace >= moe_workspace_size(MOE_OP_LAYER_HOST). */
moe_status moe_layer_forward_host(const moe_config* cfg, const void* x_host, const void* w_r,
                                  const float* logit_offset, const float* sel_bias,
                                  const void* w13, const void* w2, void* y_host,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* Shared expert ([overview] glossary "Expert": DeepSeek-V3 has 256 routed
 * experts plus 1 shared expert per layer, "MoE 路由机制是什么"): a SwiGLU FFN that
 * every token passes through, outside the routing.  For every token t:
 * a = silu(x[t] Wg^T) * (x[t] Wu^T), stored in dtype; ys[t] = a Wd^T, stored in
 * dtype; float32 accumulation.  Needs cfg->shared_I > 0.
 * x [T,h] dtype; w13s [2*shared_I, h] dtype (gate rows then up rows); w2s
 * [h, shared_I] dtype; ys [T,h] dtype; workspace >= moe_workspace_size(MOE_OP_SHARED). */
moe_status moe_shared_ffn(const moe_config* cfg, const void* x, const void* w13s, const void* w2s, void* ys,
                          void* workspace, size_t workspace_bytes, void* stream);

/* moe_combine plus a per-token term: y[t] = ys[t] + sum_{k: slot[t,k] >= 0}
 * topk_w[t,k] * yp[slot[t,k]], float32 sum (ys first, then k order), stored in
 * dtype.  ys [T,h] dtype (the shared expert's output); other arguments as in
 * moe_combine. */
moe_status moe_combine_add(const moe_config* cfg, const void* yp, const int32_t* slot, const float* topk_w,
                           const void* ys, void* y, void* stream);

/* The DeepSeek-V3 MoE block: moe_layer_forward's routed experts plus the shared
 * expert, y = ys + routed combine (moe_shared_ffn, then moe_combine_add in place
 * of moe_combine).  Needs cfg->shared_I > 0.  Arguments as in moe_layer_forward
 * plus w13s, w2s as in moe_shared_ffn; workspace >= moe_workspace_size(MOE_OP_BLOCK). */
moe_status moe_block_forward(const moe_config* cfg, const void* x, const void* w_r, const float* logit_offset,
                             const float* sel_bias, const void* w13, const void* w2, const void* w13s,
                             const void* w2s, void* y, const moe_layer_out* out, void* workspace,
                             size_t workspace_bytes, void* stream);

/* moe_block_forward with HOST activations, as moe_layer_forward_host:
 * x_host [T,h] in, y_host [T,h] out, copies on `stream`;
 * workspace >= moe_workspace_size(MOE_OP_BLOCK_HOST). */
moe_status moe_block_forward_host(const moe_config* cfg, const void* x_host, const void* w_r,
                                  const float* logit_offset, const float* sel_bias, const void* w13,
                                  const void* w2, const void* w13s, const void* w2s, void* y_host,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* Replica plan for expert-parallel load balancing ([overview] glossary "Logical
 * expert", "Physical expert / Replica", "Redundant expert": hot logical experts
 * are copied so that E + n_redundant physical experts, a multiple of the GPU
 * count, flatten the load).  Host only, integer arithmetic:
 *  - each of the n_redundant replicas goes, one at a time, to the logical expert
 *    with the largest counts[e] / n_rep[e] (ties to the lower id);
 *  - a logical expert's count is split over its replicas as evenly as possible
 *    (replica r gets counts/n + (r < counts % n));
 *  - replicas, heaviest first (ties: lower expert, lower replica), go to the
 *    rank with the least load among ranks with a free slot (ties to the lower
 *    rank); each of the ep_size ranks has (E + n_redundant) / ep_size slots and
 *    physical ids are rank-major in placement order.
 * counts [E] int64 (tokens per logical expert, e.g. from a previous batch);
 * outputs, host memory: rep_offsets [E+1] and rep_phys [E+n_redundant] (the
 * physical ids of e's replicas are rep_phys[rep_offsets[e] .. rep_offsets[e+1])),
 * phys_to_log [E+n_redundant], rank_load [ep_size] (may be NULL). */
moe_status moe_eplb_plan(int32_t E, int32_t ep_size, int32_t n_redundant, const int64_t* counts,
                         int32_t* rep_offsets, int32_t* rep_phys, int32_t* phys_to_log, int64_t* rank_load);

/* Physical expert of every routed (t, k): replica t mod n_rep(e) of its logical
 * expert e = topk_ids[t,k] (a function of (t, e) only).  topk_ids, phys_ids
 * [T,K] int32 device; rep_offsets, rep_phys device copies of moe_eplb_plan's. */
moe_status moe_eplb_map(const moe_config* cfg, const int32_t* topk_ids, const int32_t* rep_offsets,
                        const int32_t* rep_phys, int32_t* phys_ids, void* stream);

/* moe_grouped_ffn over physical experts whose weights are their logical
 * experts': segment p uses w13[phys_to_log[p]], w2[phys_to_log[p]], so
 * replicas share one copy.  w13 [E,2I,h], w2 [E,h,I]; phys_to_log
 * [E+n_redundant] int32 device; other arguments as in moe_grouped_ffn. */
moe_status moe_grouped_ffn_mapped(const moe_config* cfg, const void* xp, const int32_t* offsets, const int32_t* kept,
                                  const int32_t* phys_to_log, const void* w13, const void* w2, void* yp,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* moe_layer_forward with replicas: route over the E logical experts,
 * moe_eplb_map, then layout / permute / mapped FFN / combine over the physical
 * experts (n_ij, rank bytes and Balancedness per physical placement).  The plan
 * arrays are device copies of moe_eplb_plan's; out->topk_ids receives logical
 * ids, out->counts/kept/offsets physical ones.  moe_layer_forward and the
 * block calls refuse n_redundant > 0.  workspace >= moe_workspace_size(MOE_OP_LAYER). */
moe_status moe_layer_forward_eplb(const moe_config* cfg, const void* x, const void* w_r, const float* logit_offset,
                                  const float* sel_bias, const void* w13, const void* w2, const int32_t* rep_offsets,
                                  const int32_t* rep_phys, const int32_t* phys_to_log, void* y,
                                  const moe_layer_out* out, void* workspace, size_t workspace_bytes, void* stream);

/* FP8 experts.  The pages name FP8 MoE (expert weights and activations in 8
 * bits) without a format; this library uses OCP E4M3 codes (round to nearest
 * even, saturating at 448) with one float32 scale per row: scale = amax/448
 * (1 for an all-zero row), code = E4M3(v / scale), both divisions in IEEE
 * float32.  Weights are quantised per output row (w13 rows = gate/up units, w2
 * rows = output features), expert inputs per token, and the bf16 SwiGLU
 * intermediate per row before the down projection.  FP8 calls need a bf16
 * layer with h % 128 == 0, I % 128 == 0, no shared expert and no replicas, and
 * experts expected to see at most 160 rows (else MOE_ERR_UNSUPPORTED). */

/* Row quantisation: codes[r, c] and scales[r] of src [rows, cols] (dtype
 * MOE_BF16 or MOE_F32; cols % 16 == 0; src and codes 16-byte aligned), e.g.
 * w13 viewed as [E*2I, h] and w2 as [E*h, I], once, before the layer runs. */
moe_status moe_quantize_fp8(int64_t rows, int32_t cols, int32_t dtype, const void* src, uint8_t* codes,
                            float* scales, void* stream);

/* moe_permute with the expert inputs quantised: each token's row x[t] is
 * quantised once and its codes and scale written to every kept permuted row
 * slot[t,k]: xq [R,h] uint8, sx [R] float32 (pad rows are not written). */
moe_status moe_permute_fp8(const moe_config* cfg, const void* x, const int32_t* slot, uint8_t* xq, float* sx,
                           void* stream);

/* moe_grouped_ffn on FP8 operands: g = (xq . w13q_gate) * sx[r] * s13[unit], u
 * likewise, a = silu(g) * u stored in bf16 and re-quantised per row; yp[r] =
 * (aq . w2q) * sa[r] * s2[feature], bf16; float32 accumulation.  xq [R,h],
 * sx [R]; w13q [E,2I,h] uint8, s13 [E,2I] float32; w2q [E,h,I] uint8, s2 [E,h];
 * yp [R,h] bf16; workspace >= moe_workspace_size(MOE_OP_FFN_FP8). */
moe_status moe_grouped_ffn_fp8(const moe_config* cfg, const uint8_t* xq, const float* sx, const int32_t* offsets,
                               const int32_t* kept, const uint8_t* w13q, const float* s13, const uint8_t* w2q,
                               const float* s2, void* yp, void* workspace, size_t workspace_bytes, void* stream);

/* moe_layer_forward with FP8 experts: bf16 router and routing, moe_permute_fp8,
 * moe_grouped_ffn_fp8, combine.  workspace >= moe_workspace_size(MOE_OP_LAYER_FP8). */
moe_status moe_layer_forward_fp8(const moe_config* cfg, const void* x, const void* w_r, const float* logit_offset,
                                 const float* sel_bias, const uint8_t* w13q, const float* s13, const uint8_t* w2q,
                                 const float* s2, void* y, const moe_layer_out* out, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* Synchronises `stream`, then reports and clears the sticky device error word of
 * the current device: MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_DEVICE_BAD_INDEX,
 * MOE_ERR_CUDA for a pending CUDA error, else MOE_OK. */
moe_status moe_check(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
