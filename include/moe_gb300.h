/*
 * moe_gb300.h - C ABI of a GB300 (sm_103a) forward pass of one
 * Mixture-of-Experts layer on one GPU.
 *
 * The layer (MoE comm bottleneck page, section 1.1; MoE module notes page,
 * sections 3.1-3.3 and the MoELayer listing of 4.2):
 *   logits  = x . gate (+ bias)                       router, a Linear H -> E
 *   p       = softmax(logits) over the E experts
 *   idx, w  = top-k of the logits, weights p renormalised over the k chosen
 *   stats   = routed counts, P_e = mean_t p[t,e], aux = E * sum_e f_e P_e
 *   dispatch: capacity C = max(1, ceil(cf * T*k / E)); each expert serves
 *             its assignments in token order and drops those at position
 *             >= C; kept rows are gathered expert-major into x_perm
 *   FFN     : act = bf16(gelu_tanh(x_perm . W1[e])); y_perm = bf16(act . W2[e])
 *   combine : y[t] = bf16(sum over kept slots j, ascending, of w[t,j] y_perm[row])
 *
 * Conventions for every entry point
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise; the
 *     shape struct is a host pointer. The caller owns all memory. The library
 *     never allocates; scratch comes from the caller's workspace `ws`
 *     (size from moe_workspace_size). Pointers must be 16-byte aligned.
 *   - Arrays are dense and row-major: x [T,H], gate [H,E], W1 [E,H,h],
 *     W2 [E,h,H], topk_idx/topk_w/dest_row [T,k], x_perm/y_perm [T*k,H],
 *     act [T*k,h], y [T,H]. bf16 arrays hold raw bf16 bit patterns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronise with the host. The number of
 *     kept rows N is only known on the device, so row buffers hold T*k rows;
 *     rows at index >= offsets[E] are left unspecified.
 *   - Host-side checks return a status before anything is launched. A
 *     launch failure returns MOE_ERR_CUDA. Problems found in device data
 *     (bad expert index, non-finite logits, a wait that ran out) are OR-ed
 *     as MOE_DEV_* bits into *dev_status; the kernels then finish normally.
 *     The caller clears *dev_status; a NULL dev_status uses a workspace word.
 *   - Workspace contents do not survive between calls, and two calls that
 *     share a workspace must be ordered on one stream.
 *   - Supported: 0 <= T, T*k < 2^31; 1 <= E <= 256; 1 <= k <= min(E, 8);
 *     H and h multiples of 64, >= 64; capacity_factor finite and > 0.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols of the shared library (everything else is hidden). */
#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#define MOE_GB300_ABI_VERSION 1

typedef uint16_t moe_bf16; /* a bf16 value as its 16 bits */

typedef struct {
  int64_t T;               /* tokens */
  int64_t H;               /* hidden size */
  int64_t E;               /* number of experts */
  int64_t top_k;           /* experts per token, k */
  int64_t h;               /* expert FFN width */
  double capacity_factor;  /* cf, binary64 (see moe_capacity) */
} moe_shape;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_NULL = 1,        /* a required pointer is NULL */
  MOE_ERR_SHAPE = 2,       /* a size is negative, zero where it may not be, or overflows */
  MOE_ERR_UNSUPPORTED = 3, /* valid but outside the supported ranges above */
  MOE_ERR_WORKSPACE = 4,   /* ws_bytes < moe_workspace_size */
  MOE_ERR_ALIGN = 5,       /* a pointer is not 16-byte aligned */
  MOE_ERR_CUDA = 6         /* a CUDA call or launch failed */
} moe_status;

/* Bits OR-ed into *dev_status by the kernels. */
#define MOE_DEV_BAD_INDEX 1u  /* an expert index outside [0,E): slot dropped */
#define MOE_DEV_DUP_INDEX 2u  /* a token names one expert twice: later slot dropped */
#define MOE_DEV_NONFINITE 4u  /* a router logit is NaN or infinite */
#define MOE_DEV_TIMEOUT 8u    /* a pipeline wait gave up; outputs are incomplete */

/* Number of CUDA events moe_layer_fwd records when given an event array. */
#define MOE_LAYER_NUM_EVENTS 7

/* Capacity per expert, C = max(1, ceil(cf * (T*k) / E)), evaluated in
 * binary64 in exactly that order (MoE comm bottleneck, section 3.1, gives
 * capacity = ceil(capacity_factor * tokens / num_experts); the MoE module
 * notes' listing, section 4.2, counts tokens as T*k and floors C at 1).
 * Returns -1 for E < 1, k < 1, T < 0 or a non-finite/non-positive cf.
 * Host only; needs no GPU. */
MOE_API int64_t moe_capacity(int64_t T, int64_t E, int64_t top_k, double capacity_factor);

/* Bytes of device workspace any entry point needs for this shape (one size
 * serves all of them). Host only. Returns MOE_ERR_NULL / _SHAPE /
 * _UNSUPPORTED for bad arguments. */
MOE_API moe_status moe_workspace_size(const moe_shape* s, size_t* bytes);

/* Static text for a status code. Host only. */
MOE_API const char* moe_status_str(moe_status st);

/* MOE_GB300_ABI_VERSION of the built library. Host only. */
MOE_API int moe_abi_version(void);

/* Router: logits GEMM on the tensor cores, softmax, top-k, renormalised
 * weights and the load-balancing statistics (MoE module notes, section 3.1
 * router listing; MoE comm bottleneck, section 3.2 auxiliary loss).
 *   in : x [T,H] bf16, gate [H,E] bf16, gate_bias [E] fp32 or NULL
 *   out: topk_idx [T,k] int32 (largest logit first; equal logits by lower
 *        expert index), topk_w [T,k] fp32 (sum to 1 per token),
 *        routed_counts [E] int32 (assignments per expert before drops),
 *        P [E] fp32 (mean softmax probability), aux [1] fp32
 *        (E * sum_e routed_e/(T*k) * P_e; the loss weight alpha is the
 *        caller's), logits_out [T,E] fp32 or NULL (bias included).
 * routed_counts, P, aux may be NULL. */
MOE_API moe_status moe_route(const moe_shape* s, const moe_bf16* x, const moe_bf16* gate,
                     const float* gate_bias, int32_t* topk_idx, float* topk_w,
                     int32_t* routed_counts, float* P, float* aux, float* logits_out,
                     uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream);

/* The router's steps after the GEMM, on caller-given fp32 logits [T,E]
 * (the MoE module notes, section 5.2, take top-k directly on the logits at
 * inference). Same outputs and rules as moe_route; with equal logits the
 * two give identical indices, weights and statistics. */
MOE_API moe_status moe_route_logits(const moe_shape* s, const float* logits, int32_t* topk_idx,
                            float* topk_w, int32_t* routed_counts, float* P, float* aux,
                            uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream);

/* The training router of the MoE module notes page, section 3.1: Gumbel
 * noise is added to the logits and the sum is divided by a temperature,
 *   scores = (x . gate + bias + g) / temperature,
 *   g = -log(-log(u + 1e-9) + 1e-9),
 * with u the caller's uniform draws in [0,1) (noise_u [T,E] fp32, device;
 * the library draws no random numbers). Top-k is taken on the scores, the
 * weights are softmax(scores) renormalised over the k chosen, and the
 * balance statistics use softmax(scores) (the module notes feed these
 * probabilities to their balance loss). scores_out [T,E] fp32 or NULL
 * receives the scores. temperature must be finite and > 0. Other arguments
 * as moe_route. */
MOE_API moe_status moe_route_gumbel(const moe_shape* s, const moe_bf16* x, const moe_bf16* gate,
                            const float* gate_bias, const float* noise_u, float temperature,
                            int32_t* topk_idx, float* topk_w, int32_t* routed_counts, float* P,
                            float* aux, float* scores_out, uint32_t* dev_status, void* ws,
                            size_t ws_bytes, void* stream);

/* Dispatch: capacity-bounded, token-ordered permutation of token rows into
 * expert-major order - the single-GPU form of the dispatch all-to-all (MoE
 * comm bottleneck, sections 1.1 and 3.1: tokens beyond an expert's
 * capacity are dropped, later tokens first).
 *   in : x [T,H] bf16, topk_idx [T,k] int32
 *   out: kept_counts [E] = min(routed_e, C); offsets [E+1] exclusive scan;
 *        dest_row [T,k] = offsets[e] + position, or -1 if dropped;
 *        src_token [T*k] (row -> token, rows < offsets[E]);
 *        x_perm [T*k,H] bf16 (row dest_row[t,j] = x[t]).
 * kept_counts, src_token may be NULL; x_perm may be NULL when src_token is
 * given (the permutation only, for moe_expert_ffn_gathered). Bad or repeated
 * indices set MOE_DEV_BAD_INDEX / MOE_DEV_DUP_INDEX and that slot is dropped. */
MOE_API moe_status moe_permute(const moe_shape* s, const moe_bf16* x, const int32_t* topk_idx,
                       int32_t* kept_counts, int32_t* offsets, int32_t* dest_row,
                       int32_t* src_token, moe_bf16* x_perm, uint32_t* dev_status,
                       void* ws, size_t ws_bytes, void* stream);

/* Expert FFN over the ragged expert-major rows as two grouped GEMMs on the
 * tensor cores (MoE comm bottleneck, section 5.1 grouped GEMM; expert =
 * Linear -> GELU -> Linear, MoE module notes section 3.3, bias-free weights
 * as in the 4.2 listing). Rows [offsets[e], offsets[e+1]) use expert e.
 *   in : x_perm [T*k,H] bf16, offsets [E+1] int32, W1 [E,H,h], W2 [E,h,H]
 *   out: act [T*k,h] bf16 = bf16(gelu_tanh(x_perm . W1[e])) (fp32 accumulate),
 *        y_perm [T*k,H] bf16 = bf16(act . W2[e]). */
MOE_API moe_status moe_expert_ffn(const moe_shape* s, const moe_bf16* x_perm, const int32_t* offsets,
                          const moe_bf16* W1, const moe_bf16* W2, moe_bf16* act,
                          moe_bf16* y_perm, uint32_t* dev_status, void* ws, size_t ws_bytes,
                          void* stream);

/* moe_expert_ffn with the dispatch's row copy fused into GEMM1's operand
 * load: row r of GEMM1's A is x[src_token[r]], fetched by TMA row gathers,
 * so the permuted copy x_perm is neither written nor read. The pages print
 * no such step: it removes, on one GPU, the round trip of the dispatch bytes
 * (MoE comm bottleneck section 2.1). Same act / y_perm as moe_expert_ffn on
 * x_perm = x[src_token]. src_token [T*k] from moe_permute (rows <
 * offsets[E]); entries outside [0, T) read row 0 or T-1. It saves the
 * T*k*H*2-byte x_perm buffer and its traffic but runs GEMM1 about 3x slower
 * on GB300 (the TMA moves the A operand as 32 four-row gathers per stage
 * instead of one tile), so moe_layer_fwd keeps the permuted copy. */
MOE_API moe_status moe_expert_ffn_gathered(const moe_shape* s, const moe_bf16* x,
                                   const int32_t* src_token, const int32_t* offsets,
                                   const moe_bf16* W1, const moe_bf16* W2, moe_bf16* act,
                                   moe_bf16* y_perm, uint32_t* dev_status, void* ws,
                                   size_t ws_bytes, void* stream);

/* Combine: weighted sum of each token's kept expert rows, back at the
 * token's position (MoE comm bottleneck, section 1.1, the combine step).
 * y[t] = bf16(sum_{j: dest_row[t,j] >= 0, ascending j} topk_w[t,j] *
 * y_perm[dest_row[t,j]]), fp32 accumulation; a token with no kept slot gets
 * zeros. Needs no workspace. */
MOE_API moe_status moe_combine(const moe_shape* s, const moe_bf16* y_perm, const int32_t* dest_row,
                       const float* topk_w, moe_bf16* y, void* stream);

/* The whole layer forward: route, dispatch, expert FFN and combine on one
 * stream, with no host synchronisation.
 *   in : x, gate, gate_bias (or NULL), W1, W2 as above
 *   out: y [T,H] bf16 (required); aux, topk_idx, topk_w, routed_counts, P,
 *        kept_counts, offsets, dest_row may each be NULL (then kept in ws).
 *   events: NULL, or MOE_LAYER_NUM_EVENTS cudaEvent_t handles (host
 *        pointer to an array); events[0] is recorded before the first
 *        kernel and events[1..6] after the route, scan, permute, FFN GEMM1,
 *        FFN GEMM2 and combine stages, for per-stage timing. */
MOE_API moe_status moe_layer_fwd(const moe_shape* s, const moe_bf16* x, const moe_bf16* gate,
                         const float* gate_bias, const moe_bf16* W1, const moe_bf16* W2,
                         moe_bf16* y, float* aux, int32_t* topk_idx, float* topk_w,
                         int32_t* routed_counts, float* P, int32_t* kept_counts,
                         int32_t* offsets, int32_t* dest_row, uint32_t* dev_status,
                         void* ws, size_t ws_bytes, void* stream, void* const* events);

/* moe_layer_fwd with the training router of moe_route_gumbel (Gumbel noise
 * from the caller's uniforms noise_u [T,E], temperature > 0); events as in
 * moe_layer_fwd. */
MOE_API moe_status moe_layer_fwd_gumbel(const moe_shape* s, const moe_bf16* x, const moe_bf16* gate,
                                const float* gate_bias, const float* noise_u, float temperature,
                                const moe_bf16* W1, const moe_bf16* W2, moe_bf16* y, float* aux,
                                int32_t* topk_idx, float* topk_w, int32_t* routed_counts, float* P,
                                int32_t* kept_counts, int32_t* offsets, int32_t* dest_row,
                                uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream,
                                void* const* events);

/* Bytes of device workspace moe_layer_fwd_host needs for micro-batches of
 * this shape: the layer workspace plus two token and two output buffers.
 * Host only. */
MOE_API moe_status moe_host_workspace_size(const moe_shape* s, size_t* bytes);

/* Host-to-host layer forward over n_micro micro-batches of s->T tokens each,
 * pipelined over three caller streams - the dual-stream, micro-batch overlap
 * of the MoE comm bottleneck page, section 5.2, with the host<->device copies
 * in the role of the dispatch/combine traffic: while micro-batch i runs the
 * layer on streams[0], micro-batch i+1's tokens are copied in on streams[1]
 * and micro-batch i-1's outputs are copied out on streams[2].
 *   x_host[i], y_host[i] (i < n_micro): HOST pointers to [T,H] bf16 tokens
 *        and outputs; page-locked memory (cudaHostAlloc / cudaHostRegister)
 *        is needed for the copies to overlap. The same pointer may repeat.
 *   aux_host: HOST array of n_micro floats, or NULL.
 *   gate, gate_bias (nullable), W1, W2: device, as in moe_layer_fwd.
 *   dev_status: device word or NULL.
 *   ws: device, >= moe_host_workspace_size bytes.
 *   streams: host array of 3 cudaStream_t (compute, copy-in, copy-out),
 *        owned by the caller; they must be distinct streams (not the legacy
 *        default stream, which would serialise them).
 *   events: host array of 6 cudaEvent_t created by the caller (timing may be
 *        disabled); they order the buffers between the streams.
 * Everything is enqueued and the call returns; y_host and aux_host are valid
 * once streams[2] has completed. */
MOE_API moe_status moe_layer_fwd_host(const moe_shape* s, int64_t n_micro, const moe_bf16* const* x_host,
                              moe_bf16* const* y_host, float* aux_host, const moe_bf16* gate,
                              const float* gate_bias, const moe_bf16* W1, const moe_bf16* W2,
                              uint32_t* dev_status, void* ws, size_t ws_bytes,
                              void* const* streams, void* const* events);

/* Bytes of device workspace moe_layer_fwd_pipelined needs: two layer
 * workspaces, used by alternate micro-batches. Host only. */
MOE_API moe_status moe_pipelined_workspace_size(const moe_shape* s, size_t* bytes);

/* The layer forward over n_micro micro-batches of s->T tokens each, on the
 * device, pipelined over two caller streams - the dual-stream, micro-batch
 * overlap of the MoE comm bottleneck page, section 5.2, with the on-device
 * dispatch and combine in the role of the all-to-alls: while micro-batch i
 * runs its two expert GEMMs on streams[1], streams[0] routes and permutes
 * micro-batch i+1 and combines micro-batch i-1, so those memory-bound
 * kernels run beside the GEMMs on the SM resources the GEMM leaves free.
 *   x [n_micro*T, H], y [n_micro*T, H] bf16 (device): micro-batch i is rows
 *        i*T .. i*T+T-1; each micro-batch is a layer forward of its own
 *        (its own routing, capacity and statistics), with the outputs of
 *        moe_layer_fwd on those rows.
 *   aux [n_micro] fp32 (device) or NULL: each micro-batch's aux.
 *   gate, gate_bias (nullable), W1, W2, dev_status (nullable): as moe_layer_fwd.
 *   ws: >= moe_pipelined_workspace_size bytes.
 *   streams: host array of 2 cudaStream_t (dispatch, expert), distinct and
 *        not the legacy default stream; give the dispatch stream the higher
 *        priority (cudaStreamCreateWithPriority) so that its kernels are
 *        scheduled as soon as resources free up.
 *   events: host array of 4 cudaEvent_t created by the caller (timing may be
 *        disabled); they order the two streams.
 * Everything is enqueued and the call returns; y and aux are complete once
 * streams[0] has completed (its last kernel is the last combine). */
MOE_API moe_status moe_layer_fwd_pipelined(const moe_shape* s, int64_t n_micro, const moe_bf16* x,
                                           const moe_bf16* gate, const float* gate_bias,
                                           const moe_bf16* W1, const moe_bf16* W2, moe_bf16* y,
                                           float* aux, uint32_t* dev_status, void* ws,
                                           size_t ws_bytes, void* const* streams,
                                           void* const* events);

/* ------------------------------------------------------------- FP8 ----
 * FP8 (e4m3) dispatch and expert FFN: the MoE comm bottleneck page, section
 * 5.3, sends FP8 hidden states to halve the dispatch bytes; here the
 * dispatched rows are e4m3 and both expert GEMMs run on the FP8 tensor-core
 * path. Scaling (one reading; the page fixes none): one fp32 scale per row
 * of activations and per output column of weights. For a row with largest
 * magnitude amax: inv = 448 / amax, q = e4m3(v * inv) (round to nearest
 * even, saturating at +-448), scale = amax / 448, all in fp32; a zero row
 * has q = 0 and scale = 0. A GEMM of quantised operands is the fp32 sum of
 * q products times the row scale times the column scale. e4m3 arrays hold
 * raw bytes. */

/* Bytes of device workspace the FP8 entry points need (more than
 * moe_workspace_size: row scales and the quantised activations). Host only. */
MOE_API moe_status moe_workspace_size_fp8(const moe_shape* s, size_t* bytes);

/* Weight quantisation, done once per weight tensor: W [E,K,N] bf16 (K the
 * input dimension) -> Wq [E,N,K] e4m3, each output column a contiguous row,
 * and w_scale [E,N] fp32 column scales. For the layer: W1 gives W1q [E,h,H]
 * and w1_scale [E,h]; W2 gives W2q [E,H,h] and w2_scale [E,H].
 * 1 <= E <= 256; K, N multiples of 64, at most 65536. Needs no workspace
 * (w_scale doubles as scratch). */
MOE_API moe_status moe_quantize_weights_fp8(int64_t E, int64_t K, int64_t N, const moe_bf16* W,
                                    uint8_t* Wq, float* w_scale, void* stream);

/* moe_permute with an FP8 payload: each token row is quantised once with
 * its own scale, and the e4m3 row and scale go to every kept destination:
 * x_q [T*k,H] e4m3 and x_scale [T*k] fp32 instead of x_perm. Other
 * arguments, results and the workspace as moe_permute. */
MOE_API moe_status moe_permute_fp8(const moe_shape* s, const moe_bf16* x, const int32_t* topk_idx,
                           int32_t* kept_counts, int32_t* offsets, int32_t* dest_row,
                           int32_t* src_token, uint8_t* x_q, float* x_scale,
                           uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream);

/* moe_expert_ffn on e4m3 rows: u = x_scale[r] * w1_scale[e,:] * (x_q[r] .
 * W1q[e]^T) in fp32; act [T*k,h] bf16 = bf16(gelu_tanh(u)); act is
 * quantised per row (scale from the largest |act| of the row) and the
 * expert outputs are v = bf16(act_scale[r] * w2_scale[e,:] * (act_q[r] .
 * W2q[e]^T)), written either
 *   - as y_perm [T*k,H] bf16 (y_q, y_scale NULL), or
 *   - as y_q [T*k,H] e4m3 with y_scale [T*k, ceil(H/128)] fp32, one scale per
 *     128-column block of a row formed from the bf16 values v like a row
 *     scale (y_perm NULL): the FP8 payload of the combine.
 * Both y_perm and y_q given returns MOE_ERR_UNSUPPORTED. ws must hold
 * moe_workspace_size_fp8 bytes. */
MOE_API moe_status moe_expert_ffn_fp8(const moe_shape* s, const uint8_t* x_q, const float* x_scale,
                              const int32_t* offsets, const uint8_t* W1q, const float* w1_scale,
                              const uint8_t* W2q, const float* w2_scale, moe_bf16* act,
                              moe_bf16* y_perm, uint8_t* y_q, float* y_scale,
                              uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream);

/* moe_combine on the e4m3 expert outputs of moe_expert_ffn_fp8:
 * y[t] = bf16(sum over kept slots j, ascending, of topk_w[t,j] *
 * y_q[r,c] * y_scale[r, c/128]), r = dest_row[t,j], fp32 accumulation. The
 * combine's FP8 half of the comm bottleneck page, section 5.3. Needs no
 * workspace. */
MOE_API moe_status moe_combine_fp8(const moe_shape* s, const uint8_t* y_q, const float* y_scale,
                           const int32_t* dest_row, const float* topk_w, moe_bf16* y,
                           void* stream);

/* moe_layer_fwd with the FP8 dispatch, the FP8 expert FFN (weights from
 * moe_quantize_weights_fp8) and the FP8 combine (expert outputs as e4m3
 * with 128-column block scales); the router is that of moe_layer_fwd. ws
 * must hold moe_workspace_size_fp8 bytes. events as in moe_layer_fwd,
 * events[4] recorded after GEMM1 and the act quantisation. */
MOE_API moe_status moe_layer_fwd_fp8(const moe_shape* s, const moe_bf16* x, const moe_bf16* gate,
                             const float* gate_bias, const uint8_t* W1q, const float* w1_scale,
                             const uint8_t* W2q, const float* w2_scale, moe_bf16* y, float* aux,
                             int32_t* topk_idx, float* topk_w, int32_t* routed_counts, float* P,
                             int32_t* kept_counts, int32_t* offsets, int32_t* dest_row,
                             uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream,
                             void* const* events);

/* moe_layer_fwd_host with the FP8 layer of moe_layer_fwd_fp8: the same
 * three-stream micro-batch pipeline (bf16 tokens in, bf16 outputs out), with
 * the quantised weights of moe_quantize_weights_fp8. ws must hold
 * moe_host_workspace_size_fp8 bytes. Other arguments as moe_layer_fwd_host. */
MOE_API moe_status moe_host_workspace_size_fp8(const moe_shape* s, size_t* bytes);
MOE_API moe_status moe_layer_fwd_host_fp8(const moe_shape* s, int64_t n_micro,
                                  const moe_bf16* const* x_host, moe_bf16* const* y_host,
                                  float* aux_host, const moe_bf16* gate, const float* gate_bias,
                                  const uint8_t* W1q, const float* w1_scale, const uint8_t* W2q,
                                  const float* w2_scale, uint32_t* dev_status, void* ws,
                                  size_t ws_bytes, void* const* streams, void* const* events);

/* ---------------------------------------------- expert parallelism ----
 * Experts spread over `world` ranks, rank g holding the E/world consecutive
 * experts g*E/world .. (g+1)*E/world - 1, and each token's rows sent to the
 * rank of its expert and back: the dispatch and combine all-to-alls of the
 * MoE comm bottleneck page, section 1.1 (byte counts in section 2.1), and
 * the MoE module notes' MoELayer listing, section 4.2 (_all_to_all_routed).
 * The library provides the per-rank steps; the exchanges themselves are the
 * caller's collectives (e.g. NCCL all-to-all): rank r sends rows
 * [offsets[g*E/world], offsets[(g+1)*E/world]) of its x_perm to rank g
 * (send_counts[g] of them) and kept_counts[g*E/world ..] to rank g as its
 * counts row r; rank g regroups what it received (moe_ep_regroup), runs
 * moe_expert_ffn on its experts, regroups back and returns the rows in the
 * same order; rank r then runs moe_combine on them as usual. */

/* moe_permute for one rank of an expert-parallel group (s->T = this rank's
 * tokens, s->E = all experts; world must divide E; 0 <= rank < world).
 *   routed_all [world][E] int32 (device): every rank's routed counts (the
 *        moe_route output, gathered from all ranks, this rank's row
 *        included). Given, each expert serves the group's tokens in global
 *        order - rank 0's tokens first, then rank 1's, ... - against the
 *        capacity of the group's batch, C = max(1, ceil(cf * T_global*k / E)):
 *        this rank keeps its assignment at local position pos iff the earlier
 *        ranks' assignments to that expert plus pos are below C, which makes
 *        the sharded layer equal to the single-device layer over all tokens.
 *        NULL: the rank applies the capacity of its own batch (s->T) to its
 *        own tokens alone, as the module notes' listing computes capacity
 *        from the local batch; T_global is then ignored.
 *   T_global: the group's tokens (>= s->T) when routed_all is given.
 *   send_counts [world] int32 (device, out): rows for each rank's experts.
 * Other arguments, results (expert-major x_perm, whose rows for rank g's
 * experts are contiguous) and the workspace as moe_permute. */
MOE_API moe_status moe_ep_permute(const moe_shape* s, int64_t world, int64_t rank,
                                  const int32_t* routed_all, int64_t T_global,
                                  const moe_bf16* x, const int32_t* topk_idx,
                                  int32_t* kept_counts, int32_t* offsets, int32_t* dest_row,
                                  int32_t* src_token, moe_bf16* x_perm, int32_t* send_counts,
                                  uint32_t* dev_status, void* ws, size_t ws_bytes, void* stream);

/* Moves rows of width H between the two orders of the rows a rank receives
 * in an expert-parallel exchange:
 *   source-major: from each source rank r in order, its rows of this rank's
 *        E_local experts, expert by expert (what an all-to-all delivers);
 *   expert-major: expert by expert, and within an expert source by source,
 *        i.e. in global token order (what moe_expert_ffn takes).
 *   counts [world][E_local] int32 (device): rows source r sent for local
 *        expert e (row r is source r's kept_counts for these experts);
 *        negative counts are read as 0.
 *   to_expert_major 1: src source-major -> dst expert-major, and
 *        local_offsets [E_local+1] (device, may be NULL) receives the
 *        expert-major segment offsets for moe_expert_ffn; 0: the inverse
 *        (src expert-major -> dst source-major; local_offsets unused).
 *   rows: rows src and dst can hold; rows at or past it are not touched
 *        (counts summing to more are cut there).
 * world * E_local <= 256; H a multiple of 64. Needs no workspace. */
MOE_API moe_status moe_ep_regroup(int64_t world, int64_t E_local, int64_t H, int64_t rows,
                                  int to_expert_major, const int32_t* counts, const moe_bf16* src,
                                  moe_bf16* dst, int32_t* local_offsets, void* stream);

/* moe_permute for callers that cannot allocate device memory. The pages
 * have no counterpart to this entry point; it serves code that may not call
 * cudaMalloc or hold a workspace: a plugin inside a runtime that owns all
 * device memory, or code issuing work while a stream is being captured.
 * Same arguments and results as moe_permute, minus ws/ws_bytes (x_perm may
 * be NULL when src_token is given): the scratch is one static 1 MiB device
 * array per GPU, held until the process exits.
 *   - Shapes whose scratch exceeds 1 MiB return MOE_ERR_UNSUPPORTED before
 *     any launch. The scratch is 2*r(4*E*ceil(T/128)) + r(T*k) + 2*r(4*E)
 *     + 512 bytes, r() rounding up to a multiple of 256 (tile counts and
 *     bases, in-tile ranks, per-expert counts and sums, ticket and status).
 *   - The first call in a CUDA context looks the array's address up (again
 *     after the context is torn down and made anew, e.g. by
 *     cudaDeviceReset); make it before any stream capture.
 *   - All calls on a device share the array; calls that overlap on the GPU
 *     race and must be serialised by the caller. Allocates nothing. */
MOE_API moe_status moe_permute_noalloc(const moe_shape* s, const moe_bf16* x, const int32_t* topk_idx,
                               int32_t* kept_counts, int32_t* offsets, int32_t* dest_row,
                               int32_t* src_token, moe_bf16* x_perm, uint32_t* dev_status,
                               void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
