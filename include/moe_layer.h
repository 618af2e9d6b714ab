/*
 * moe_layer.h -- C ABI of the GB300 (sm_103a) quantised MoE layer forward.
 *
 * The layer (per token t with hidden state x[t], fp16 [H]):
 *   1. router logits  l[t][e] = x[t] . Wr[e] (+ bias[e]) for every expert e
 *      (the router scores every expert from the token's hidden state:
 *      "12GB显卡跑68GB大模型：Betelgeuse引擎实测22 tok/s", MoE background);
 *   2. top-k experts with softmax renormalised weights w[t][j]
 *      (top-2 of 64: "Strata" article, section 1.1; top-4 of 512:
 *      "Flash-MoE" article, section 1);
 *   3. grouping of the (token, slot) pairs by expert, so that one read of an
 *      expert's weights serves every token routed to it
 *      ("为什么12G显存笔记本能跑MoE-16B", section 2.3; "Strata" section 2.3);
 *   4. per routed pair, the expert FFN with group-wise dequantised weights
 *      W = (q - zero) * scale, one fp16 scale and one zero point per 128
 *      consecutive K elements ("Strata" section 2.2; "为什么12G显存笔记本能跑
 *      MoE-16B" section 4.2: dequantised inside the kernel, never written
 *      back), gate/up projection, SwiGLU h = silu(g) * u, down projection
 *      ("Flash-MoE" section 3: dequant matvec and fused SwiGLU);
 *   5. out[t] = x[t] + sum_j w[t][j] y[t][j] + sigmoid(x[t] . wg) y_shared[t]
 *      ("Flash-MoE" section 3: fused combine + residual + sigmoid gate).
 *
 * Numerics (the library's contract):
 *   - a logit is the EXACT sum of the exact fp16 x fp16 products, rounded
 *     once to fp32 (nearest even), then one fp32 add of the bias; top-k is by
 *     logit descending, ties to the lower expert id.  Routing is therefore
 *     independent of summation order and reproducible bit for bit;
 *   - grouping is a stable sort of pair ids p = t*k + j by expert;
 *   - expert arithmetic accumulates in fp32; the SwiGLU activation h is
 *     kept in fp16 between the two projections; the output is fp16 (nearest
 *     even).
 *
 * Conventions: every tensor argument of the compute calls is a DEVICE pointer
 * (row-major, contiguous, caller-owned) on the current CUDA device; `stream`
 * is a cudaStream_t (NULL = the legacy default stream).  fp16 tensors are
 * IEEE binary16.  Calls are asynchronous on `stream`, allocate nothing and do
 * not synchronise the host, except moe_layer_create, moe_check_status and
 * moe_layer_destroy.  A layer holds one workspace: use it from one stream at a
 * time.  Every call returns MOE_OK (0) or a negative status; the message of
 * the last failure on the calling thread is in moe_last_error().  No call
 * throws, traps or aborts; argument checks happen before any CUDA call.
 */
#ifndef MOE_LAYER_H
#define MOE_LAYER_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,   /* null pointer, bad size or shape, aliasing */
    MOE_ERR_UNSUPPORTED = -2,   /* wbits, group size or dtype not supported */
    MOE_ERR_OOM = -3,           /* device allocation failed in create */
    MOE_ERR_CUDA = -4,          /* a CUDA call or launch failed */
    MOE_ERR_DEVICE_STATUS = -5  /* a kernel guard fired (see moe_check_status) */
};

enum { MOE_FP16 = 0 };

/* Device status bits reported by moe_check_status (or'ed together). */
enum {
    MOE_STATUS_BAD_EXPERT = 1,  /* a routing index outside [0, E): pair skipped */
    MOE_STATUS_NONFINITE = 2,   /* an inf/nan fp16 input reached the router */
    MOE_STATUS_TIMEOUT = 4,     /* a pipeline wait gave up after its time limit:
                                   the outputs of that call are incomplete */
    MOE_STATUS_TIER_OVERFLOW = 8 /* a call touched more host-resident experts than
                                   free device slots (see moe_layer_set_residency):
                                   the surplus experts contributed 0 */
};

typedef struct moe_layer moe_layer_t;

typedef struct {
    int hidden;        /* H: multiple of 128, <= 16384 */
    int inter;         /* I: routed expert intermediate size, multiple of 128 */
    int n_experts;     /* E: 1 .. 1024 */
    int top_k;         /* k: 1 .. min(E, 32) */
    int group_size;    /* quantisation group along K: must be 128 */
    int wbits;         /* 4 or 2 */
    int has_shared;    /* 1: a shared expert behind a sigmoid gate */
    int shared_inter;  /* its intermediate size (multiple of 128) */
    int residual;      /* 1: add x to the output (0: omit) */
    int io_dtype;      /* MOE_FP16 */
    int max_tokens;    /* largest n_tokens of any later call: 1 .. 65536 */
} moe_cfg_t;

/*
 * Canonical packed weights, all DEVICE pointers, read only during
 * moe_layer_create (the caller may free them when it returns).
 *   codes[m]  : uint8 [E][rows][K*wbits/8]; 4-bit: element k in byte k/2, low
 *               nibble = even k; 2-bit: element k in byte k/4, bits 2(k%4)..+1
 *   scales[m] : fp16 [E][rows][K/128]
 *   zeros[m]  : uint8 [E][rows][K/128], values 0 .. 2^wbits-1
 *   m = 0 gate (rows I, K H), 1 up (rows I, K H), 2 down (rows H, K I)
 *   router_w  : fp16 [E][H]; router_bias: fp32 [E] or NULL
 *   sh_*      : the shared expert, same layout with E = 1 and I = shared_inter
 *   sh_gate_w : fp16 [H] (sigmoid gate of the shared expert)
 */
typedef struct {
    const uint8_t *codes[3];
    const uint16_t *scales[3];
    const uint8_t *zeros[3];
    const uint16_t *router_w;
    const float *router_bias;
    const uint8_t *sh_codes[3];
    const uint16_t *sh_scales[3];
    const uint8_t *sh_zeros[3];
    const uint16_t *sh_gate_w;
} moe_packed_weights_t;

/* Read-only facts about a created layer (for accounting and benchmarks). */
typedef struct {
    int64_t weight_bytes;      /* device bytes of the repacked expert weights */
    int64_t workspace_bytes;   /* device bytes of the per-layer workspace */
    int64_t expert_bytes;      /* streamed bytes of one routed expert */
    int64_t shared_bytes;      /* streamed bytes of the shared expert */
    int num_sms;
    int grid_ffn;              /* CTAs of the expert-FFN kernels */
    int n_phases;              /* phases timed by moe_profile_read */
    int gemm_min_tokens;       /* see moe_layer_set_gemm_min_tokens */
} moe_layer_info_t;

/*
 * Creates a layer on the current CUDA device: validates cfg, copies and
 * repacks the weights into library-owned device memory (a tile layout for
 * 128-bit coalesced loads), allocates the workspace for cfg->max_tokens and
 * synchronises the device before returning.  *out receives the handle (NULL
 * on failure; nothing stays allocated then).
 * Errors: INVALID_ARG (null pointer, non-device weight pointer, bad shape),
 * UNSUPPORTED (wbits, group_size, io_dtype), OOM, CUDA.
 */
int moe_layer_create(const moe_cfg_t *cfg, const moe_packed_weights_t *w, moe_layer_t **out);

/* Frees everything the layer owns (synchronises the device first).  NULL-safe. */
void moe_layer_destroy(moe_layer_t *layer);

/*
 * Routing only (steps 1-3) for x fp16 [n_tokens][H].  Outputs (any may be
 * NULL): topk_idx int32 [n][k], topk_w fp32 [n][k], counts int32 [E],
 * offsets int32 [E+1] (exclusive prefix of counts), perm int32 [n*k] (pair
 * ids p = t*k + j sorted stably by expert).
 * Errors: INVALID_ARG (null layer or x, n_tokens outside 1..max_tokens), CUDA.
 */
int moe_route_topk(moe_layer_t *layer, const void *x, int n_tokens, int32_t *topk_idx,
                   float *topk_w, int32_t *counts, int32_t *offsets, int32_t *perm,
                   void *stream);

/* Router logits only (step 1): logits fp32 [n_tokens][E], bias included. */
int moe_router_logits(moe_layer_t *layer, const void *x, int n_tokens, float *logits,
                      void *stream);

/*
 * Routing without a layer and without any device allocation: router logits,
 * top-k and softmax weights (steps 1-2) of x fp16 [n_tokens][hidden] against
 * router_w fp16 [n_experts][hidden] and router_bias fp32 [n_experts] (or
 * NULL).  Outputs topk_idx int32 [n_tokens][top_k] and topk_w fp32
 * [n_tokens][top_k].  All pointers are DEVICE pointers owned by the caller.
 * The numerics are those of moe_route_topk: exact logits rounded once to
 * fp32, ties to the lower expert id, so both calls give identical results.
 *
 * The pages have no counterpart for this call: they route only inside a
 * loaded model.  It serves callers that cannot allocate device memory where
 * they route, e.g. a scheduler choosing which experts to stage before any
 * layer object exists, on a device whose memory its own pool has already
 * reserved (a cudaMalloc there fails, or synchronises the device and stalls
 * every other stream).
 *
 * Scratch: one fixed buffer per device inside the library, sized for
 * n_tokens * n_experts <= MOE_NOALLOC_MAX_SCORES; larger calls are rejected
 * (INVALID_ARG) before any CUDA work.  The call clears the buffer's
 * must-be-zero part on `stream` before its kernel.  The first call on each
 * device does the setup: it looks up the buffer's address and sets the
 * kernel's shared-memory attribute; make that first call before any stream
 * capture.  Calls whose executions overlap (different streams, or threads
 * without ordering between them) share the buffer and race: their results are
 * wrong.  Order them on one stream.  Non-finite inputs count as zero and are
 * not reported by this call.
 * Alignment: x 16 bytes; router_w 8 bytes; router_bias, topk_idx, topk_w 4
 * bytes.
 * Errors: INVALID_ARG (null, misaligned or non-device pointer, hidden not a
 * multiple of 128 or above 16384, n_experts outside 1..1024, top_k outside
 * 1..min(32, n_experts), n_tokens < 1, n_tokens * n_experts too large), CUDA.
 */
enum { MOE_NOALLOC_MAX_SCORES = 16384 };
int moe_route_topk_noalloc(const void *x, const void *router_w, const float *router_bias,
                           int n_tokens, int hidden, int n_experts, int top_k, int32_t *topk_idx,
                           float *topk_w, void *stream);

/*
 * The whole layer (steps 1-5): x fp16 [n_tokens][H] -> out fp16 [n_tokens][H].
 * out must not overlap x.  out is device memory, or pinned host memory that
 * the device maps (the last kernel writes the rows there in place, so no
 * separate copy back is needed); the same holds for the out arguments of
 * moe_forward_routed and moe_forward_prenorm.
 * Errors: INVALID_ARG (null pointer, n_tokens outside 1..max_tokens, overlap,
 * out neither device nor pinned host memory), CUDA.
 */
int moe_forward(moe_layer_t *layer, const void *x, void *out, int n_tokens, void *stream);

/*
 * Steps 3-5 with caller-given routing: topk_idx int32 [n][k] (expert ids),
 * topk_w fp32 [n][k].  A pair whose expert id lies outside [0, E) is skipped
 * and sets MOE_STATUS_BAD_EXPERT in the device status word.
 */
int moe_forward_routed(moe_layer_t *layer, const void *x, const int32_t *topk_idx,
                       const float *topk_w, void *out, int n_tokens, void *stream);

/*
 * Two-pass RMSNorm ("Flash-MoE" article, section 3: the two-pass RMSNorm
 * among a layer's kernels, the step in front of the router):
 *   xn[t][h] = fp16( (resid[t][h] * rs_t) * gamma[h] ),
 *   rs_t = 1 / sqrt( (sum_h resid[t][h]^2) / H + eps ).
 * The pages give no precision.  Each value is within one fp16 ulp of the
 * correctly rounded real value r*g/sqrt(mean(r^2)+eps), and equal to it
 * almost always.  The library computes in fp32 in one fixed order, so a
 * given input always gives the same bits (reproducible routing): the sum of
 * squares per 128-element group (32 partials of 4 consecutive squares,
 * combined pairwise by lane distance 16, 8, 4, 2, 1), the group sums added
 * in order, each step rounded to nearest even.
 * resid fp16 [n_tokens][hidden], gamma fp16 [hidden], xn fp16
 * [n_tokens][hidden]: DEVICE pointers owned by the caller, 16-byte aligned;
 * xn may equal resid (in place).  No layer, no allocation; asynchronous on
 * `stream`.
 * Errors: INVALID_ARG (null or misaligned pointer, n_tokens < 1, hidden not a
 * multiple of 128 or above 16384, eps negative, NaN or infinite), CUDA.
 */
int moe_rmsnorm(const void *resid, const void *gamma, float eps, int n_tokens, int hidden,
                void *xn, void *stream);

/*
 * The layer with the RMSNorm in front (steps 0-5): the layer runs on
 * xn = moe_rmsnorm(resid, gamma, eps), and its residual term is resid:
 *   out[t] = resid[t] + sum_j w_j y_j(xn[t]) + sigmoid(xn[t] . wg) y_sh(xn[t])
 * (the residual term is left out when the layer was created with residual
 * = 0).  resid, out fp16 [n_tokens][H], gamma fp16 [H]: DEVICE pointers owned
 * by the caller (out may also be pinned host memory, as for moe_forward);
 * out must not overlap resid.  xn lives in the layer's
 * workspace (one stream at a time, like every call on the layer).
 * Errors: those of moe_forward and moe_rmsnorm.
 */
int moe_forward_prenorm(moe_layer_t *layer, const void *resid, const void *gamma, float eps,
                        void *out, int n_tokens, void *stream);

/*
 * Copy of `bytes` from src to dst by a kernel on `stream`, launched like the
 * layer's own kernels, so that it chains with them.  Each pointer may be
 * device memory, managed memory or pinned host memory that the device maps
 * (cudaHostAlloc, cudaHostRegister with mapping; on GB300 the SMs reach it
 * over NVLink-C2C).  The pages have no counterpart: this is the host <->
 * device step of an end-to-end call (pinned input rows in, output rows back)
 * without copy-engine round trips between it and the layer's kernels.
 * dst, src and bytes must be multiples of 16 bytes, the ranges must lie
 * inside their buffers and must not overlap.  Asynchronous; bytes = 0 does
 * nothing.
 * Errors: INVALID_ARG (null, misaligned, overlapping, or a pointer the
 * device cannot reach, e.g. pageable host memory), CUDA.
 */
int moe_copy(void *dst, const void *src, size_t bytes, void *stream);

/*
 * Synchronises the device, returns MOE_OK when no kernel guard fired since
 * the last check, else MOE_ERR_DEVICE_STATUS with the MOE_STATUS_* bits in
 * *bits (may be NULL).  Clears the status word.
 */
int moe_check_status(moe_layer_t *layer, int *bits);

/*
 * Expert FFN kernel choice.  Within one call, an expert that receives at
 * least min_tokens tokens (and the shared expert when n_tokens >= min_tokens)
 * runs on the tensor-core GEMM kernels (tcgen05, accumulators in tensor
 * memory, weights dequantised once per 64 tokens); every other expert runs on
 * the decode kernels, which stream its weights once per 8 tokens.  0 puts
 * every expert on the decode kernels.  Default for 4-bit layers: 9 when one
 * routed expert's gate/up has at least one 128-row tile per SM (2 * inter /
 * 128 >= SM count) and hidden, inter and shared_inter are all at least 512;
 * otherwise 0 (the GEMM kernels would leave most SMs idle).  2-bit layers
 * always use the decode kernels (UNSUPPORTED for min_tokens > 0).
 * Host-only: takes effect from the next call on the layer's stream.
 * The GEMM kernels round each dequantised weight (q - z) * s once to fp16
 * before the multiply; the decode kernels apply the scale in fp32.
 */
int moe_layer_set_gemm_min_tokens(moe_layer_t *layer, int min_tokens);

/*
 * Expert residency tiers ("Luce Spark", sections 1-2: the most frequently
 * routed experts pinned on the GPU, the rest in host RAM and brought in on
 * demand; "12GB显卡跑68GB大模型：Betelgeuse引擎实测22 tok/s": a pool of VRAM
 * slots for the experts in use, resolved inside the stream without host
 * round trips).
 *
 * After this call the layer's routed experts live in two tiers:
 *   - the n_resident experts listed in `resident` (host array of distinct
 *     ids, any order) stay in device memory for good;
 *   - every other expert lives in pinned host memory (allocated here; the
 *     GB300 SMs read it over NVLink-C2C), and n_slots device slots cache the
 *     ones in use.
 * Each later forward, after grouping, finds on the device which touched
 * experts are cold: those already in a slot are hits; each miss takes a slot
 * that the call does not otherwise use, least recently used first (ties to
 * the lower slot; misses in expert order), and its records are copied into
 * it from host memory by the SMs.  No host synchronisation, so the forward
 * stays graph-capturable.  Results are bit-identical to the untiered layer.
 * n_slots must lie in min(E - n_resident, max_tokens * top_k) .. E -
 * n_resident, so that one call's cold experts always fit (it is ignored when
 * n_resident = E).  The shared expert is always resident.  May be called
 * again to change the tiers (the slots start empty).  Synchronises the
 * device.  Device memory afterwards: the resident experts, the slots and one
 * expert-sized zero block (moe_layer_info's weight_bytes).
 * Errors: INVALID_ARG (bad ids, duplicates, n_slots out of range), OOM,
 * CUDA; after a failure other than INVALID_ARG destroy the layer.
 */
int moe_layer_set_residency(moe_layer_t *layer, const int32_t *resident, int n_resident,
                            int n_slots);

/*
 * Placement policy ("Luce Spark", section 1: per-(layer, expert) routing
 * frequencies pick the experts pinned on the GPU): the n_resident experts
 * with the largest counts (host array int64 [n_experts], e.g. sums of
 * moe_route_topk's counts over calibration batches), ties to the lower id,
 * written to resident[0 .. n_resident-1] in that order.  Host only.
 * Errors: INVALID_ARG (null pointer, n_experts outside 1..1024, n_resident
 * outside 0..n_experts, a negative count).
 */
int moe_residency_plan(const int64_t *counts, int n_experts, int n_resident, int32_t *resident);

/*
 * Tier counters of a tiered layer since moe_layer_set_residency (synchronises
 * the device): slot hits and misses over all forwards (a touched cold expert
 * counts once per call), and the slots holding an expert.  Any output may be
 * NULL.  moe_layer_tier_slots copies the expert held by each slot (-1: none)
 * into slot_expert[0 .. n_slots-1] (n >= n_slots).
 * Errors: INVALID_ARG (null layer, untiered layer), CUDA.
 */
int moe_layer_tier_stats(moe_layer_t *layer, uint64_t *hits, uint64_t *misses,
                         int *slots_filled);
int moe_layer_tier_slots(moe_layer_t *layer, int32_t *slot_expert, int n);

/*
 * Expert-parallel layer across GPUs ("Strata" article, section 5.2: with two
 * cards the expert cache is sharded per card).  The routed experts are
 * partitioned by id over `world` ranks: rank r owns experts
 * [r*E/world, (r+1)*E/world) (integer division).  A forward on each rank:
 *   1. route its tokens (moe_route_topk_noalloc, or moe_route_topk);
 *   2. moe_ep_dispatch: pack one activation row per (token, slot) pair into
 *      send_x, grouped by destination rank (pair order kept inside a rank),
 *      with the owner's local expert id of each row;
 *   3. all-to-all of the rows and ids (the caller's collective, e.g. NCCL);
 *   4. each owner runs its experts on the rows it received: a layer created
 *      with its E_local experts, top_k = 1, residual = 0 and no shared
 *      expert, called with moe_forward_routed (local ids, weight 1): fp16
 *      rows back;
 *   5. all-to-all of the result rows back, in the order they came;
 *   6. moe_ep_combine: out[t] = x[t] + sum_j w[t][j] y[pos(t, j)]
 *      + sigmoid(x[t] . wg) y_shared[t], fp32 in slot order, rounded once
 *      to fp16; y_shared from the rank's own copy of the shared expert (a
 *      one-expert layer, top_k = 1, residual = 0, moe_forward_routed).
 * The result rows travel as fp16 (half the bytes of fp32); that adds one
 * fp16 rounding of each expert output before the weighted sum.
 *
 * moe_ep_dispatch: x fp16 [n_tokens][hidden], topk_idx int32
 * [n_tokens][top_k] (global expert ids); outputs send_x fp16 [n*k][hidden]
 * (rows 0 .. sum(dest_counts)-1 written), send_expert int32 [n*k] (local id
 * at the owner), pos_of_pair int32 [n*k] (send row of pair p = t*k + j, -1
 * for an id outside [0, E)), dest_counts int32 [world] (rows per destination,
 * in rank order), status int32 [1] (set to 1 when an id was outside [0, E);
 * never cleared here).  All DEVICE pointers owned by the caller; x and
 * send_x 16-byte aligned.  No allocation; asynchronous on `stream`.
 * Errors: INVALID_ARG (null, misaligned or non-device pointer, sizes, world
 * outside 1..min(32, n_experts)), CUDA.
 *
 * moe_ep_combine: x fp16 [n][hidden] (the tokens, and the residual when
 * residual = 1), topk_w fp32 [n][top_k], pos_of_pair int32 [n*k] (from
 * moe_ep_dispatch), y_rows fp16 [rows][hidden] (the returned rows in send
 * order), sh_gate_w fp16 [hidden] and y_shared fp16 [n][hidden] (both NULL
 * without a shared expert), out fp16 [n][hidden] (must not overlap x).
 * DEVICE pointers, 16-byte aligned rows.  Asynchronous on `stream`.
 * Errors: INVALID_ARG (null, misaligned or non-device pointer, overlap,
 * sizes, only one of sh_gate_w / y_shared), CUDA.
 */
int moe_ep_dispatch(const void *x, int n_tokens, int hidden, const int32_t *topk_idx,
                    int top_k, int n_experts, int world, void *send_x, int32_t *send_expert,
                    int32_t *pos_of_pair, int32_t *dest_counts, int *status, void *stream);
int moe_ep_combine(const void *x, int n_tokens, int hidden, int top_k, const float *topk_w,
                   const int32_t *pos_of_pair, const void *y_rows, const void *sh_gate_w,
                   const void *y_shared, int residual, void *out, void *stream);

/* Facts about the layer (no device work). */
int moe_layer_info(const moe_layer_t *layer, moe_layer_info_t *info);

/*
 * Per-phase timing: with on = 1 every later moe_forward records CUDA events
 * between its kernels on its stream; moe_profile_read synchronises and
 * returns the accumulated milliseconds per phase in ms[0 .. n_phases-1]
 * (routing, grouping, gate/up, down, combine) and the number of
 * forwards timed, then resets the sums.  Do not enable while capturing a
 * CUDA graph.
 */
int moe_profile_enable(moe_layer_t *layer, int on);
int moe_profile_read(moe_layer_t *layer, float *ms, int n, int *calls);

/* Message of the last failed call on this thread ("" if none). */
const char *moe_last_error(void);

#ifdef __cplusplus
}
#endif
#endif
