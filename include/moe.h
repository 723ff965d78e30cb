/*
 * moe.h — C ABI of the B300 (sm_103a) MoE expert layer.
 *
 * The layer is the single-GPU expert block behind the "grouped_mm" expert
 * backend: a router picks k experts per token, the token-slots are sorted by
 * expert, each expert's SwiGLU MLP runs as one grouped GEMM over its rows
 * without copying any expert parameters, and the expert outputs are combined
 * back per token with the router weights; forward and backward.
 *
 * Source: NeMo AutoModel blog (zh-CN / ja translations of "Accelerating
 * Transformers fine-tuning with NVIDIA NeMo AutoModel"), table
 * "专家后端 / エキスパートバックエンド" (expert backends), grouped_mm row:
 * sort the tokens by assigned expert and run a single grouped GEMM, memory
 * efficient, no parameter copies; "v4 死锁原因" (why v4 deadlocks): experts
 * are fused 3-D parameter tensors; "关于路由门的说明" (note on the routing
 * gate): the balanced gate forces tokens evenly across experts.  Readings of
 * what the pages leave open (router formula, activation, gate rule) are given
 * at each call.
 *
 * Conventions for every call
 *   - All tensor arguments are DEVICE pointers to row-major, densely packed
 *     arrays owned by the caller.  bf16 tensors are raw bfloat16 bits
 *     (moe_bf16) and must be 16-byte aligned.  The library never allocates,
 *     frees or copies expert weights; weights are read-only.
 *   - Every compute call is asynchronous on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and never synchronises, except
 *     moe_read_device_status.
 *   - Host-side validation happens before anything is launched; a rejected
 *     call launches nothing and returns MOE_ERR_INVALID_ARG,
 *     MOE_ERR_UNSUPPORTED_SHAPE or MOE_ERR_WORKSPACE_TOO_SMALL.  A failed
 *     launch returns MOE_ERR_CUDA.  Problems found on the device (an expert
 *     id outside [0, E), a wait that ran out of time) are written to the
 *     status word in the workspace; read it with moe_read_device_status.
 *     There is no CPU fallback.
 *   - Deterministic: identical inputs give bit-identical outputs.
 *
 * Shapes: T tokens, H hidden, E experts, k experts per token, I expert
 * intermediate size, I_shared intermediate size of the optional always-on
 * shared expert (0 = none), S = T*k token-slots, slot s = t*k + j.
 * Supported: 1 <= E <= 256, 1 <= k <= min(E, 32), H and I (and I_shared when
 * non-zero) positive multiples of 64, T >= 1, T*k < 2^31.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16; /* raw bfloat16 bits */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,         /* null pointer, misalignment, bad enum */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,   /* dims outside the supported set above */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < moe_workspace_size() */
  MOE_ERR_CUDA = 4,                /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE_INDEX = 5,        /* device saw an expert id outside [0, E) */
  MOE_ERR_TIMEOUT = 6              /* a device-side wait ran out of time */
} moe_status;

typedef enum {
  MOE_GATE_SOFTMAX_TOPK = 0, /* learned router: softmax, top-k, renormalise */
  MOE_GATE_BALANCED = 1      /* balanced gate: slot (t,j) -> expert (t*k+j) mod E */
} moe_gate_mode;

/*
 * capacity: expert capacity, the most token-slots one expert processes
 * (0 = no limit, < 0 rejected).  The pages name expert overflow as a risk of
 * uneven routing ("NVIDIA NeMo AutoModel MoE 微調的 3.7 倍加速突破", closing
 * paragraph on load balancing) but give no rule; the reading here: an expert
 * keeps its first `capacity` slots in slot order s = t*k + j (the stable
 * sort's order), the rest are dropped.  A dropped slot adds nothing to out
 * (its weight is not redistributed), its expert never sees it, its dL/dw is
 * 0, and the router gradient keeps its formula.  For a capacity factor f use
 * capacity = ceil(f * T * k / E).
 */
typedef struct {
  int32_t T, H, E, k, I, I_shared;
  int32_t capacity;
} moe_dims;

/* Version of this ABI (bumped on any signature or enum change). */
int32_t moe_abi_version(void);

/* Static text for a moe_status value. */
const char* moe_status_string(int32_t status);

/*
 * Bytes of device workspace the calls below need for these dims.  One
 * workspace can serve moe_route, moe_route_permute, moe_permute,
 * moe_grouped_mlp_fwd and, with
 * with_backward = 1, moe_layer_bwd given the saved pre-activations; with
 * with_backward = 2, also moe_layer_bwd recomputing them (gu_saved and/or
 * sh_gu_saved NULL: room for [S,2I] and [T,2*I_shared] bf16 more).
 * with_backward = 0: forward calls only.  The first 256 bytes hold the device
 * status word; callers zero them once (cudaMemset) before first use.
 * Errors: MOE_ERR_INVALID_ARG (null, with_backward outside 0..2),
 * MOE_ERR_UNSUPPORTED_SHAPE.
 */
moe_status moe_workspace_size(const moe_dims* d, int32_t with_backward, size_t* bytes);

/*
 * Router (note on the routing gate; the pages name the native router but not
 * its formula — reading used here):
 *   logits[t,e] = sum_h x[t,h] W_r[e,h] + bias[e]     (fp32 accumulate)
 *   p[t,:] = softmax(logits[t,:]) over all E experts
 *   SOFTMAX_TOPK: topk_idx[t,0..k-1] = the k largest logits, largest first,
 *                 equal logits -> lower expert id first
 *   BALANCED:     topk_idx[t,j] = (t*k + j) mod E  (exactly T*k/E slots per
 *                 expert when E divides T*k; distinct experts when k <= E)
 *   topk_w[t,j] = p[t,topk_idx[t,j]] / sum_j' p[t,topk_idx[t,j']]
 *   prob_sum[e] = sum_t p[t,e]   (optional; for moe_aux_loss)
 * x: bf16 [T,H]; w_router: bf16 [E,H]; router_bias: fp32 [E] or NULL;
 * logits_out: fp32 [T,E] or NULL; topk_idx: int32 [T,k]; topk_w: fp32 [T,k];
 * prob_sum: fp32 [E] or NULL (a fixed-order sum: bit-identical run to run).
 * One kernel computes the logits on the tensor cores (K split over a cluster
 * of CTAs whose partial sums are added on chip, in a fixed order) and the
 * softmax, selection and weights; a second one sums prob_sum when asked for.
 * Errors: MOE_ERR_INVALID_ARG (null, misaligned x / w_router / workspace, bad
 * gate_mode), MOE_ERR_UNSUPPORTED_SHAPE, MOE_ERR_WORKSPACE_TOO_SMALL,
 * MOE_ERR_CUDA.
 */
moe_status moe_route(const moe_dims* d, int32_t gate_mode, const moe_bf16* x,
                     const moe_bf16* w_router, const float* router_bias, float* logits_out,
                     int32_t* topk_idx, float* topk_w, float* prob_sum, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * moe_route followed by moe_permute, in two kernels instead of four: the
 * router kernel also counts, per CTA, the chosen slots of each expert, and
 * one sort pass places every slot from those counts (the grouped_mm row's
 * "sort the tokens by their assigned expert", fused with the router).
 * Outputs are bit-identical to moe_route then moe_permute on the same
 * inputs: logits_out, topk_idx, topk_w, prob_sum as moe_route;
 * expert_offsets [E+1], perm_slot [S], slot_perm [S] (with d->capacity) as
 * moe_permute.  All pointers are caller-owned device memory; logits_out and
 * prob_sum may be NULL.  Errors: as moe_route.
 */
moe_status moe_route_permute(const moe_dims* d, int32_t gate_mode, const moe_bf16* x,
                             const moe_bf16* w_router, const float* router_bias,
                             float* logits_out, int32_t* topk_idx, float* topk_w,
                             float* prob_sum, int32_t* expert_offsets, int32_t* perm_slot,
                             int32_t* slot_perm, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * Auxiliary load-balancing loss ("NVIDIA NeMo AutoModel MoE 微調的 3.7 倍加速突破",
 * closing paragraph on load balancing: an auxiliary loss keeps token routing
 * even; the routing-gate note: a load-balancing loss drives expert utilisation
 * towards uniform).  The pages give no formula; the Switch Transformer form
 * is used:
 *   f_e = (expert_offsets[e+1] - expert_offsets[e]) / (T*k)   slots routed to e
 *   P_e = prob_sum[e] / T                                      mean router probability
 *   *loss = alpha * E * sum_e f_e P_e     (alpha when routing is uniform)
 *   coef[e] = alpha * E * f_e / T          (= dloss/dp[t,e]; counts pass no gradient)
 * prob_sum: fp32 [E] from moe_route; expert_offsets: int32 [E+1] from
 * moe_permute; loss: fp32 [1] or NULL; coef: fp32 [E] or NULL (not both NULL).
 * Pass coef and the forward's logits_out to moe_layer_bwd to add the loss's
 * gradient.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_SHAPE.
 */
moe_status moe_aux_loss(const moe_dims* d, const float* prob_sum, const int32_t* expert_offsets,
                        float alpha, float* loss, float* coef, void* stream);

/*
 * Sort the token-slots by expert (grouped_mm row: "sort the tokens by their
 * assigned expert"): a stable counting sort of s = 0..S-1 by topk_idx[s].
 *   expert_offsets: int32 [E+1], expert e owns sorted rows
 *                   expert_offsets[e] .. expert_offsets[e+1]-1; offsets[E] = S
 *   perm_slot:      int32 [S], slot id at sorted row r (ascending within an expert)
 *   slot_perm:      int32 [S], sorted row of slot s (inverse of perm_slot)
 * With d->capacity > 0, expert e's first min(count_e, capacity) rows are its
 * kept slots; the rest are dropped, and slot_perm is -1 for a dropped slot
 * (perm_slot and expert_offsets stay the full sort).
 * Only ids move; no expert weight is touched.  Expert ids outside [0, E) are
 * skipped and reported as MOE_ERR_DEVICE_INDEX in the status word.
 */
moe_status moe_permute(const moe_dims* d, const int32_t* topk_idx, int32_t* expert_offsets,
                       int32_t* perm_slot, int32_t* slot_perm, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * Grouped expert MLP on the sorted rows (grouped_mm row: one grouped GEMM per
 * projection over the expert-sorted tokens, no parameter copies).  For sorted
 * row r of expert e, with token t = perm_slot[r] / k:
 *   [g | u] = x[t] W_gu[e]^T        (W_gu[e] rows 0..I-1 = gate, I..2I-1 = up)
 *   h = silu(g) * u                  (SwiGLU; the pages do not name the activation)
 *   y_perm[r] = h W_down[e]^T
 * w_gate_up: bf16 [E,2I,H]; w_down: bf16 [E,H,I] (fused 3-D expert tensors,
 * "v4 死锁原因"); gu_saved: bf16 [S,2I] pre-activations for the backward, or
 * NULL; y_perm: bf16 [S,H].  g, u and h are rounded to bf16 once.
 * Shared expert (d->I_shared > 0): y_shared[t] = SwiGLU-MLP(x[t]) with
 * w_sh_gate_up bf16 [2*I_shared,H], w_sh_down bf16 [H,I_shared]; sh_gu_saved
 * bf16 [T,2*I_shared] or NULL; y_shared bf16 [T,H].  Pass NULLs when
 * I_shared == 0.
 * With d->capacity > 0 each expert runs only its first min(count_e, capacity)
 * rows; the rows of dropped slots in y_perm and gu_saved are not written.
 */
moe_status moe_grouped_mlp_fwd(const moe_dims* d, const moe_bf16* x,
                               const int32_t* expert_offsets, const int32_t* perm_slot,
                               const moe_bf16* w_gate_up, const moe_bf16* w_down,
                               moe_bf16* gu_saved, moe_bf16* y_perm,
                               const moe_bf16* w_sh_gate_up, const moe_bf16* w_sh_down,
                               moe_bf16* sh_gu_saved, moe_bf16* y_shared, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * Weighted un-permute / combine (the "combine" half of dispatch-and-combine,
 * DeepEP paragraphs):
 *   out[t] = sum_{j=0..k-1} topk_w[t,j] * y_perm[slot_perm[t*k+j]]  (+ y_shared[t])
 * summed in fp32 in j order, rounded to bf16 once.  y_perm bf16 [S,H];
 * slot_perm int32 [S] (-1: slot dropped by the expert capacity, skipped);
 * topk_w fp32 [T,k]; y_shared bf16 [T,H] or NULL; out bf16 [T,H].  Needs no
 * workspace.
 */
moe_status moe_unpermute_combine(const moe_dims* d, const moe_bf16* y_perm,
                                 const int32_t* slot_perm, const float* topk_w,
                                 const moe_bf16* y_shared, moe_bf16* out, void* stream);

/*
 * Backward of the whole layer (the pages time forward+loss and backward
 * separately, single-node 30B benchmark table; full-parameter fine-tuning
 * updates every parameter).  Given grad_out = dL/d(out) bf16 [T,H], the
 * forward's inputs and saved routing (topk_idx, topk_w, expert_offsets,
 * perm_slot, slot_perm) and saved pre-activations (gu_saved, sh_gu_saved),
 * writes bf16 gradients:
 *   grad_x [T,H], grad_w_router [E,H], grad_w_gate_up [E,2I,H],
 *   grad_w_down [E,H,I], and when I_shared > 0 grad_w_sh_gate_up
 *   [2*I_shared,H], grad_w_sh_down [H,I_shared]; grad_router_bias fp32 [E]
 *   or NULL.
 * Activation recompute (the activation checkpointing listed among the run's
 * features, NeMo AutoModel blog, "性能对比", Nemotron 3 Ultra 550B method
 * table): gu_saved = NULL (and/or sh_gu_saved = NULL) makes
 * this call recompute those pre-activations with the forward's gate/up GEMM
 * into the workspace (size it with moe_workspace_size(d, 2, ...)) instead of
 * reading a copy kept since the forward; the gradients are bit-identical.
 * SwiGLU is recomputed from the saved (g, u).  Router: the renormalised
 * top-k weights are a softmax over the chosen logits, so
 * dlogit[t,e_j] = w_j (dw_j - sum_i w_i dw_i) with dw_j = <dout[t], y_j>,
 * and top-k selection itself passes no gradient.  With the auxiliary loss
 * (aux_coef = moe_aux_loss's coef, fp32 [E]; router_logits = the forward's
 * logits_out, fp32 [T,E]), its gradient p[t,e] (c_e - sum_e' c_e' p[t,e']) is
 * added for every expert of every token; NULL aux_coef: no auxiliary loss
 * (router_logits may then be NULL).  Experts that received no
 * token get exact-zero weight gradients.  With d->capacity > 0 (the same
 * value as in the forward), dropped slots (slot_perm -1) send no gradient to
 * their expert and have dw_j = 0; their dlogit still follows the formula.
 */
moe_status moe_layer_bwd(const moe_dims* d, const moe_bf16* grad_out, const moe_bf16* x,
                         const moe_bf16* w_router, const int32_t* topk_idx, const float* topk_w,
                         const int32_t* expert_offsets, const int32_t* perm_slot,
                         const int32_t* slot_perm, const moe_bf16* w_gate_up,
                         const moe_bf16* w_down, const moe_bf16* gu_saved,
                         const moe_bf16* w_sh_gate_up, const moe_bf16* w_sh_down,
                         const moe_bf16* sh_gu_saved, moe_bf16* grad_x, moe_bf16* grad_w_router,
                         float* grad_router_bias, moe_bf16* grad_w_gate_up,
                         moe_bf16* grad_w_down, moe_bf16* grad_w_sh_gate_up,
                         moe_bf16* grad_w_sh_down, const float* router_logits,
                         const float* aux_coef, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * Synchronise `stream`, then copy the workspace's device status word to
 * *device_status (a moe_status value; MOE_OK if nothing was recorded).  When
 * clear != 0 the word is reset to MOE_OK afterwards.  For tests and
 * debugging; this is the only call that synchronises.
 */
moe_status moe_read_device_status(void* workspace, size_t workspace_bytes, void* stream,
                                  int32_t clear, int32_t* device_status);

/*
 * Allocation-free variant of moe_permute (no counterpart on the pages).
 *
 * For callers that cannot allocate device memory, so cannot pass the
 * workspace moe_permute needs: code running where cudaMalloc is not allowed
 * or not wanted (inside a pre-sized memory pool, a plugin whose host owns all
 * device allocations, a program that must not allocate after start-up).
 * Results are identical to moe_permute's: same expert_offsets [E+1],
 * perm_slot [S] and slot_perm [S] (device pointers, caller-owned).
 *
 * Its scratch (the per-block expert histograms, ceil(T*k / 1024) * E int32)
 * lives in a fixed 256 KiB device array built into the library, which every
 * GPU that loads the library holds until the process exits.  Limit:
 * ceil(T*k / 1024) * E <= 65536 (e.g. T*k <= 524288 slots with E = 128);
 * larger shapes return MOE_ERR_UNSUPPORTED_SHAPE before anything is launched.
 * The call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine).  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) for that device; make that first call before any
 * stream capture.  The address is kept per device together with the id of
 * the context it was taken in; after a device reset (or any re-created
 * context) the next call sees a different context and looks the address up
 * again, so make that call, too, outside a stream capture.  Both launches
 * are counted by the kernel accounting below (sort_histogram, sort_scatter).
 * Every call on a device shares the one array and it keeps
 * the last call's contents (nothing in it needs clearing: each call writes
 * every entry it reads); calls whose work overlaps on the GPU (different
 * streams, no ordering between them) race on it.
 * device_status: optional device int32 (NULL to skip); expert ids outside
 * [0, E) are skipped and MOE_ERR_DEVICE_INDEX is recorded there if it holds
 * MOE_OK (the caller zeroes it).
 * Errors: MOE_ERR_INVALID_ARG (null pointer), MOE_ERR_UNSUPPORTED_SHAPE,
 * MOE_ERR_CUDA (symbol lookup or launch failed).
 */
moe_status moe_permute_static_scratch(const moe_dims* d, const int32_t* topk_idx,
                                      int32_t* expert_offsets, int32_t* perm_slot,
                                      int32_t* slot_perm, int32_t* device_status, void* stream);

/*
 * Expert parallelism (NeMo AutoModel blog, "专家并行与 DeepEP": every rank holds
 * 1/ep of the experts, split along the expert dimension as Shard(0) splits it,
 * and trains on its own tokens; DeepEP dispatches the tokens to their experts'
 * ranks and combines the outputs back with all-to-all exchanges).  The
 * exchange is the caller's collective; these two calls lay the rows out
 * around it.  A source sorts its slots with moe_route_permute (expert order is
 * rank order, because every rank's experts are contiguous) and gathers its
 * token rows in that order; a receiver groups what it got by expert with
 * moe_ep_receive_layout, runs moe_grouped_mlp_fwd over its local experts
 * (dims T = rows received, k = 1, E = local experts; perm_slot = recv_perm),
 * puts the outputs back in receive order with moe_gather_rows (idx =
 * recv_inv), and exchanges them back; the source then holds y_perm in its
 * own sorted order and calls moe_unpermute_combine.
 */

/*
 * dst[i] = src[idx[i] / div] for i < n: rows of H bf16 (H a multiple of 8),
 * src [src_rows, H], dst [n, H], idx int32 [n]; all device memory, caller-owned.
 * A row index outside [0, src_rows) gives a zero row and MOE_ERR_DEVICE_INDEX
 * in *device_status (optional, device int32; recorded only over MOE_OK).
 * Errors: MOE_ERR_INVALID_ARG (null, misaligned src/dst, n < 0, div < 1),
 * MOE_ERR_UNSUPPORTED_SHAPE (H), MOE_ERR_CUDA.
 */
moe_status moe_gather_rows(const moe_bf16* src, int64_t src_rows, int32_t H, const int32_t* idx,
                           int32_t n, int32_t div, moe_bf16* dst, int32_t* device_status,
                           void* stream);

/*
 * A receiving rank's layout.  counts: int32 [n_src, E_local] (device), the
 * rows source s sent for local expert e; the receive buffer holds source 0's
 * rows, then source 1's, ..., each source's in expert order; R = their total.
 * Writes local_offsets [E_local+1] (local expert e owns grouped rows
 * local_offsets[e] .. local_offsets[e+1]-1), recv_perm [R] (grouped row g is
 * receive row recv_perm[g]; grouped order: expert, then source, then the
 * source's order) and recv_inv [R] (its inverse).  A total that is not R is
 * recorded as MOE_ERR_DEVICE_INDEX in *device_status (optional).  Limits:
 * E_local <= 256, n_src * E_local <= 4096.  Errors: MOE_ERR_INVALID_ARG,
 * MOE_ERR_UNSUPPORTED_SHAPE, MOE_ERR_CUDA.
 */
moe_status moe_ep_receive_layout(int32_t n_src, int32_t E_local, const int32_t* counts, int32_t R,
                                 int32_t* local_offsets, int32_t* recv_perm, int32_t* recv_inv,
                                 int32_t* device_status, void* stream);

/*
 * dst[i] = src[idx[i] / div] for i < n, 4-byte elements (a source's routing
 * weights topk_w, read as [T*k], in its sorted order: idx = perm_slot, div =
 * 1).  src [src_n], dst [n], idx int32 [n], 4-byte aligned device memory.  An
 * index outside [0, src_n) gives 0 and MOE_ERR_DEVICE_INDEX in
 * *device_status (optional).  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA.
 */
moe_status moe_gather_scalars(const void* src, int64_t src_n, const int32_t* idx, int32_t n,
                              int32_t div, void* dst, int32_t* device_status, void* stream);

/*
 * The expert-parallel backward, in two calls around the exchanges (same
 * pages; the backward of dispatch is a combine of the slots' gradients and the
 * backward of combine a dispatch of grad_out).  A source gathers its
 * grad_out rows (moe_gather_rows, idx = perm_slot, div = k) and its routing
 * weights (moe_gather_scalars) in its sorted order and sends them like the
 * forward's token rows.  The experts' rank runs moe_experts_bwd on what it
 * received and sends dx_rows and dw_rows back; the source, now holding its
 * slots' dx and dw in its sorted order, runs moe_router_bwd.  The results
 * equal moe_layer_bwd's on the same rows bit for bit, except the router's
 * weight and bias gradients, which each rank forms over its own tokens (the
 * caller sums them over the ranks, as data parallelism sums any replicated
 * parameter's gradient).
 *
 * moe_experts_bwd: the experts part.  d: T = rows received, k = 1, E = local
 * experts, I, I_shared = 0, capacity = 0 (MOE_ERR_UNSUPPORTED_SHAPE
 * otherwise).  grad_out_rows, x_rows bf16 [T,H]: the received rows' grad_out
 * and token rows, receive order; row_w fp32 [T]: each row's routing weight;
 * expert_offsets [E+1], perm_slot [T] (= recv_perm), slot_perm [T] (=
 * recv_inv): moe_ep_receive_layout's grouping; gu_saved bf16 [T, 2I] from
 * the experts' moe_grouped_mlp_fwd on the same grouping (or NULL: recomputed
 * into the workspace).  Writes dx_rows bf16 [T,H] (each row's input
 * gradient), dw_rows fp32 [T] (each row's d loss / d routing weight),
 * grad_w_gate_up [E,2I,H], grad_w_down [E,H,I].  Workspace:
 * moe_workspace_size(d, 1 or 2, ...).
 *
 * moe_router_bwd: the router part on the tokens' rank.  d: the rank's own
 * dims (T tokens, E = all experts, k), I_shared = 0; x, w_router and the
 * forward's routing (topk_idx, topk_w, expert_offsets, perm_slot, slot_perm);
 * dx_sorted bf16 [T*k, H] and dw_sorted fp32 [T*k]: the slots' dx and dw in
 * the rank's sorted order (slot s at row slot_perm[s]).  Writes grad_x
 * [T,H], grad_w_router [E,H] (this rank's tokens' part), grad_router_bias fp32
 * [E] or NULL.  No auxiliary loss in this form.  Workspace as moe_layer_bwd.
 *
 * Errors: MOE_ERR_INVALID_ARG (null, misaligned), MOE_ERR_UNSUPPORTED_SHAPE,
 * MOE_ERR_WORKSPACE_TOO_SMALL, MOE_ERR_CUDA; device-detected bad indices in the
 * workspace's status word.
 */
moe_status moe_experts_bwd(const moe_dims* d, const moe_bf16* grad_out_rows,
                           const moe_bf16* x_rows, const float* row_w,
                           const int32_t* expert_offsets, const int32_t* perm_slot,
                           const int32_t* slot_perm, const moe_bf16* w_gate_up,
                           const moe_bf16* w_down, const moe_bf16* gu_saved, moe_bf16* dx_rows,
                           float* dw_rows, moe_bf16* grad_w_gate_up, moe_bf16* grad_w_down,
                           void* workspace, size_t workspace_bytes, void* stream);
moe_status moe_router_bwd(const moe_dims* d, const moe_bf16* x, const moe_bf16* w_router,
                          const int32_t* topk_idx, const float* topk_w,
                          const int32_t* expert_offsets, const int32_t* perm_slot,
                          const int32_t* slot_perm, const moe_bf16* dx_sorted,
                          const float* dw_sorted, moe_bf16* grad_x, moe_bf16* grad_w_router,
                          float* grad_router_bias, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * Kernel accounting, for benchmarks and tests (no counterpart on the pages).
 * Every kernel the calls above launch is counted under one of the ids below.
 * While timing is enabled, each launch is also bracketed by a pair of CUDA
 * events recorded on the launch stream.
 */
typedef enum {
  MOE_K_ROUTER = 0,          /* moe_route(_permute): router GEMM + softmax + top-k (+ expert counts) */
  MOE_K_ROUTE_SORT,          /* moe_route_permute: sort pass from the router's expert counts */
  MOE_K_SORT_HISTOGRAM,      /* moe_permute, pass 1: per-block expert histograms */
  MOE_K_SORT_SCATTER,        /* moe_permute, pass 2: scan + stable scatter */
  MOE_K_GATE_UP,             /* grouped gate/up GEMM + SwiGLU (token rows gathered in-kernel) */
  MOE_K_DOWN,                /* grouped down GEMM */
  MOE_K_SHARED_GATE_UP,      /* shared expert gate/up GEMM + SwiGLU */
  MOE_K_SHARED_DOWN,         /* shared expert down GEMM */
  MOE_K_COMBINE,             /* weighted un-permute / combine */
  MOE_K_DGRAD_DOWN,          /* backward: down data-gradient + SwiGLU backward (+ padded offsets) */
  MOE_K_DGRAD_GATE_UP,       /* backward: gate/up data-gradient (per slot) */
  MOE_K_SHARED_DGRAD_DOWN,
  MOE_K_SHARED_DGRAD_GATE_UP,
  MOE_K_DX_GATHER,           /* backward: router logit gradient + per-token sum of slot gradients */
  MOE_K_ROUTER_WGRAD,        /* backward: router weight gradient GEMM (split-K over tokens) */
  MOE_K_WGRAD_DOWN,          /* backward: grouped down weight-gradient GEMM */
  MOE_K_WGRAD_GATE_UP,       /* backward: grouped gate/up weight-gradient GEMM */
  MOE_K_SHARED_WGRAD_DOWN,
  MOE_K_SHARED_WGRAD_GATE_UP,
  MOE_K_ROUTER_WGRAD_REDUCE, /* backward: sum of the router weight-gradient splits, bias gradient */
  MOE_K_AUX,                 /* auxiliary loss: probability sums, loss, dense logit gradient */
  MOE_K_ROUTER_DX,           /* backward with the auxiliary loss: grad_x = DL W_r (GEMM), before
                                the per-token gather adds the slot gradients into it */
  MOE_K_GATHER_ROWS,         /* moe_gather_rows */
  MOE_K_EP_LAYOUT,           /* moe_ep_receive_layout */
  MOE_K_EP_ROWS_OUT,         /* moe_experts_bwd: the slots' dx and dw back in receive order */
  MOE_K_GATHER_SCALARS,      /* moe_gather_scalars */
  MOE_K_COUNT
} moe_kernel_id;

/* Number of kernel ids (MOE_K_COUNT) and a static name for each. */
int32_t moe_kernel_count(void);
const char* moe_kernel_name(int32_t id);

/* Turn per-launch event timing on or off (host-side state shared by all
 * streams of the process).  Events are created lazily and reused. */
moe_status moe_timing_enable(int32_t on);

/*
 * launches[i]: kernels of id i launched since the last reset (always
 * counted).  event_ms[i]: summed event-timed duration of the launches of id i
 * recorded while timing was enabled (waits for those events to complete).
 * Either array (length moe_kernel_count()) may be NULL.  reset != 0 clears
 * both afterwards.  Errors: MOE_ERR_CUDA if an event query fails.
 */
moe_status moe_kernel_stats(int32_t reset, int64_t* launches, double* event_ms);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
