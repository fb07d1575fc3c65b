/*
 * moe.h -- C ABI of the GB300 (sm_103a) Mixture-of-Experts layer forward.
 *
 * One MoE layer on one GPU, in three stream-ordered calls:
 *
 *   moe_route    gate GEMM (fp32), softmax over all experts, top-k by logit
 *                with ties to the lower expert id, optional renormalisation;
 *   moe_permute  expert -> expert-slot map (identity or replica table),
 *                optional expert-parallel local-range mask/remap, per-slot
 *                histogram, exclusive scan, stable token scatter;
 *   moe_forward  grouped GEMM FC1 with a fused SwiGLU epilogue, grouped GEMM
 *                FC2, then the routing-weighted combine of each token's k
 *                expert outputs plus an optional shared expert.
 *
 * moe_forward is also exposed as its three stages (moe_grouped_fc1,
 * moe_grouped_fc2, moe_finalize) so each can be checked on its own.
 *
 * Conventions (all calls):
 *  - Every data pointer is a DEVICE pointer owned by the caller.  Shapes are
 *    row-major with the last index contiguous.  bf16 data is passed as its
 *    16-bit patterns (moe_bf16_t).  Pointers must be 16-byte aligned and row
 *    strides multiples of 16 bytes (true when H and I are multiples of 64).
 *  - The library allocates no memory and never synchronises the host: every
 *    call enqueues kernels on `stream` and returns.  Scratch space is the
 *    caller's workspace `ws` (size from moe_workspace_size, zeroed once with
 *    moe_workspace_init).  Calls that share a workspace must be ordered on one
 *    stream; calls that overlap on the GPU with one workspace race.
 *  - The return value reports host-side argument checks and launch errors.
 *    Errors found by kernels (an expert id or slot id out of range, a wait
 *    that timed out) are OR-ed into a status word inside `ws`; read and clear
 *    it with moe_get_device_status.  Kernels never trap: a bad pair is dropped
 *    and flagged, a timed-out wait abandons its tile and flags.
 *  - T = 0 is valid and enqueues nothing.
 *  - Supported sizes: H and I multiples of 64, 1 <= k <= 32, k <= E <= 512,
 *    S (slots) <= 1024, T * k < 2^31; anything else -> MOE_ERR_UNSUPPORTED.
 *
 * Source pages of the method (cited by title and section):
 *  [TRT-4495]  TensorRT-LLM PR #4495, "large-scale EP (part 3): refactor
 *              FusedMoe for redundant expert", Description (experts vs expert
 *              slots; weights live in slots; the fused op computes on slots).
 *  [TRT-10985] TensorRT-LLM PR #10985, "MoE all-to-all paradigm" (fused MoE op
 *              trtllm_moe_fused(tokens, experts, weights[, mapping_config]),
 *              gated-MLP experts, workspace sized by max_num_tokens).
 *  [VLLM-EP]   vLLM EP-aware FusedMoE override (ep_fused_moe_patch.py): module
 *              docstring "EP expert dispatch" (global top-k ids on every rank,
 *              mask non-local experts, per-expert loop that skips count 0),
 *              ep_mask_and_remap, ep_reduce_output, the patched __init__.
 *  [DS-6964]   DeepSpeed PR #6964, AutoTP for MoE models (one reduction after
 *              the weighted sum of the selected experts' outputs per layer).
 */
#ifndef SERVING_ROUTER_GATE_GB300_MOE_H
#define SERVING_ROUTER_GATE_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16_t;            /* bf16 bit pattern */
typedef struct CUstream_st *moe_stream_t; /* same handle as cudaStream_t; NULL = legacy default stream */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,    /* a NULL pointer, a negative size, k > E, a range outside [0, S) ... */
    MOE_ERR_UNSUPPORTED = 2,    /* sizes outside the supported envelope above */
    MOE_ERR_WORKSPACE = 3,      /* ws is NULL or smaller than the call needs */
    MOE_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed (launch, tensor map, attribute) */
    MOE_ERR_DEVICE_BOUNDS = 8,  /* device status bit: an expert or slot id was out of range (pair dropped) */
    MOE_ERR_TIMEOUT = 16        /* device status bit: a bounded wait inside a kernel gave up */
} moe_status_t;

typedef enum {
    MOE_NONLOCAL_SKIP = 0,      /* non-local pairs get slot -1 and are not computed */
    MOE_NONLOCAL_MOD = 1        /* non-local pairs get slot (slot mod local_count) with weight 0 */
} moe_nonlocal_mode_t;

/* Human-readable name of a status value (static string). */
MOE_API const char *moe_status_string(int status);

/* Bytes of workspace that moe_route, moe_permute and moe_forward need for up
 * to max_T tokens (the same buffer serves all three calls).  S = number of
 * expert slots the forward computes (the local count when a local range is
 * used), I_shared_total = summed intermediate size of the shared experts (0:
 * none).  Returns 0 for invalid sizes.  Sized by the largest token count the
 * caller will pass, as [TRT-10985] sizes its workspace by max_num_tokens. */
MOE_API size_t moe_workspace_size(int64_t max_T, int H, int I, int E, int S, int k, int I_shared_total);

/* The first MOE_WS_HEADER_BYTES bytes of every workspace are its header: the
 * device status word and counters.  Kernels leave the small-batch router's
 * counter at zero when they finish, so the header is zeroed only once, by
 * moe_workspace_init; a caller never writes it. */
#define MOE_WS_HEADER_BYTES 256

/* Zero the workspace's header (status word and counters).  Call once after
 * allocating ws, before the first call that uses it. */
MOE_API moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, moe_stream_t stream);

/* Read the device status word (an OR of MOE_ERR_DEVICE_BOUNDS /
 * MOE_ERR_TIMEOUT bits, 0 when clean) into *device_status and clear it.  This
 * call synchronises `stream` (it copies 4 bytes to the host). */
MOE_API moe_status_t moe_get_device_status(void *ws, moe_stream_t stream, int32_t *device_status);

/* Number of tokens whose top-k decision needed a recheck of a near-tied
 * cluster (compensated fp32, and fp64 where that still leaves a gap inside its
 * bound) in the moe_route calls since moe_workspace_init (diagnostic;
 * synchronises). */
MOE_API moe_status_t moe_get_route_stats(void *ws, moe_stream_t stream, int64_t *refined_tokens);

/* ------------------------------------------------------------------------ */
/* moe_route -- router: gate GEMM, softmax, top-k, renormalisation.          */
/* ------------------------------------------------------------------------ */
/* [VLLM-EP] docstring "EP expert dispatch": top-k routing produces global
 * expert ids, identical on every rank; patched __init__: renormalize defaults
 * to true and routing runs over the global expert count.
 *
 *   x          [T, H] bf16         token activations
 *   gate_w     [E, H] fp32         router weight
 *   logit_bias [E] fp32 or NULL    added to the logits before the softmax
 *   renorm     0/1                 divide the k probabilities by their sum
 *   topk_ids   [T, k] int32 out    experts by descending logit, ties -> lower id
 *   topk_w     [T, k] fp32 out     softmax probability over all E experts of
 *                                  each selected expert (renormalised if asked)
 *
 * Logits are computed in fp32 on CUDA cores with a certified error bound per
 * token; whenever two logits that decide the selection or its order lie within
 * that bound, those logits are recomputed in fp64, so the ids equal those of an
 * exact (fp64) evaluation up to fp64 rounding. */
MOE_API moe_status_t moe_route(const moe_bf16_t *x, const float *gate_w, const float *logit_bias,
                       int64_t T, int H, int E, int k, int renorm,
                       int32_t *topk_ids, float *topk_w,
                       void *ws, size_t ws_bytes, moe_stream_t stream);

/* moe_route_noalloc -- moe_route without a workspace.  The source pages have
 * no counterpart of this call; it exists for callers that cannot allocate
 * device memory at all: a plugin that its host framework hands only input and
 * output buffers, a runtime whose device memory belongs to a pool this library
 * cannot reach, or a service that forbids device allocation once it is
 * running.  Same arguments, kernels and results as moe_route (the same ids;
 * weights within the same certified fp32 bound), minus the workspace.
 *
 * Its scratch is a 16 MiB array in this library's own device memory
 * (file-scope __device__ storage, held by every GPU that loads the library
 * until the process exits).  Limit: nsplit*T*E + nsplit*T + nsplit*E fp32
 * values (each part rounded up to 256 bytes) must fit in 16 MiB for the
 * smallest split nsplit = 1, i.e. roughly T*(E+1) <= 4.19 million; larger
 * calls return MOE_ERR_UNSUPPORTED before any launch.  The call allocates
 * nothing (no cudaMalloc, no allocating library routine).  The first call on
 * each device looks up the array's device address (cudaGetSymbolAddress), so
 * make that first call before any stream capture.  Every call reuses the same
 * array: calls that overlap on the GPU (on two streams) race; calls ordered on
 * one stream do not.  The refined-token counter of moe_get_route_stats is not
 * kept by this call. */
MOE_API moe_status_t moe_route_noalloc(const moe_bf16_t *x, const float *gate_w, const float *logit_bias,
                               int64_t T, int H, int E, int k, int renorm,
                               int32_t *topk_ids, float *topk_w, moe_stream_t stream);

/* moe_route_grouped -- moe_route with group-limited top-k ([VLLM-EP] _ep_init
 * arguments use_grouped_topk, num_expert_group, topk_group; the pages name them
 * only, and this is the plainest reading, DeepSeek-V2's group-limited routing):
 * the E experts form n_group groups of E / n_group consecutive ids; a group's
 * score is its largest logit; the topk_group best groups are kept (ties to the
 * lower group index) and the top-k runs over their experts only.  The softmax
 * still covers all E experts.  The group choice is certified like the top-k:
 * group scores within the fp32 bound of each other are recomputed
 * (compensated fp32, then fp64 if needed).
 * Requires 1 <= n_group <= 32, E % n_group == 0, 1 <= topk_group <= n_group and
 * k <= topk_group * E / n_group; otherwise MOE_ERR_INVALID_ARG.  Other
 * arguments, outputs and errors as moe_route. */
MOE_API moe_status_t moe_route_grouped(const moe_bf16_t *x, const float *gate_w, const float *logit_bias,
                               int64_t T, int H, int E, int k, int renorm, int n_group, int topk_group,
                               int32_t *topk_ids, float *topk_w, void *ws, size_t ws_bytes,
                               moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* moe_permute -- slot map, local mask/remap, histogram, scan, scatter.     */
/* ------------------------------------------------------------------------ */
/* Slot map [TRT-4495]: slot = expert id when rep_offset is NULL (then S must
 * equal E); otherwise expert e owns rep_offset[e+1] - rep_offset[e] >= 1 slots
 * listed at rep_slots[rep_offset[e] ...] and token t uses replica (t mod that
 * count).  Local range [VLLM-EP] ep_mask_and_remap, applied to slot ids when
 * local_count >= 0: a pair is local iff local_start <= slot < local_start +
 * local_count; topk_w is multiplied by that 0/1 mask IN PLACE; local slots
 * become slot - local_start, non-local ones -1 (MOE_NONLOCAL_SKIP) or slot mod
 * local_count (MOE_NONLOCAL_MOD, computed with weight 0).  local_count = -1:
 * no mask, S_local = S.  Otherwise S_local = local_count.
 *
 *   topk_ids  [T, k] int32 in      expert ids (out-of-range ids are dropped and flagged)
 *   topk_w    [T, k] fp32 in/out   routing weights, zeroed for non-local pairs
 *   rep_offset [E+1] int32 or NULL, rep_slots [S] int32
 *   x         [T, H] bf16 in
 *   slot_ids  [T, k] int32 out     local slot of each pair, or -1 (dropped)
 *   counts    [S_local] int32 out  pairs per local slot
 *   offsets   [S_local+1] int32 out exclusive scan of counts (offsets[S_local] = rows)
 *   perm_src  [T*k] int32 out      row r (< offsets[S_local]) holds pair perm_src[r]
 *                                  (pair index t*k + j); entries past the row count
 *                                  are left unspecified
 *   pair_row  [T*k] int32 out      row of pair p, or -1
 *   x_perm    [T*k, H] bf16 out    x_perm[r] = x[perm_src[r] / k]; rows past the
 *                                  row count are left unspecified.  May be NULL (then
 *                                  x may be NULL too): only the routing tables are
 *                                  written, for a consumer that reads the token rows
 *                                  through pair_row (moe_forward_nvfp4,
 *                                  moe_forward_w8a8)
 * Rows of one slot hold its pairs in ascending pair index (a stable grouping). */
MOE_API moe_status_t moe_permute(const int32_t *topk_ids, float *topk_w, int64_t T, int k, int E,
                         const int32_t *rep_offset, const int32_t *rep_slots, int S,
                         int local_start, int local_count, int nonlocal_mode,
                         const moe_bf16_t *x, int H,
                         int32_t *slot_ids, int32_t *counts, int32_t *offsets,
                         int32_t *perm_src, int32_t *pair_row, moe_bf16_t *x_perm,
                         void *ws, size_t ws_bytes, moe_stream_t stream);

/* moe_permute_on_input -- moe_permute with the routing applied on the input
 * ([TRT-10985] review of torch_moe.py: apply_routing_on_input, "BMM-style
 * routing"): every kept pair's row is its token's row scaled by the pair's
 * routing weight after the mask, rounded once to bf16 (nearest, ties to even):
 *     x_perm[r] = bf16(topk_w[p] * x[p / k]),  p = perm_src[r].
 * The expert outputs are then summed unweighted: pass topk_w = NULL to
 * moe_forward / moe_finalize.  Arguments, outputs and errors as moe_permute
 * (x and x_perm are required here). */
MOE_API moe_status_t moe_permute_on_input(const int32_t *topk_ids, float *topk_w, int64_t T, int k, int E,
                                  const int32_t *rep_offset, const int32_t *rep_slots, int S, int local_start,
                                  int local_count, int nonlocal_mode, const moe_bf16_t *x, int H,
                                  int32_t *slot_ids, int32_t *counts, int32_t *offsets, int32_t *perm_src,
                                  int32_t *pair_row, moe_bf16_t *x_perm, void *ws, size_t ws_bytes,
                                  moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* moe_forward -- FC1 + SwiGLU, FC2, weighted combine (+ shared expert).    */
/* ------------------------------------------------------------------------ */
/* Per slot s (rows offsets[s] .. offsets[s+1]-1 of x_perm), the gated MLP of
 * [TRT-10985] (is_gated_mlp, act_fn per expert):
 *     h = bf16( silu(x_perm W1[s]_gate^T) * (x_perm W1[s]_up^T) ),  y = bf16(h W2[s]^T)
 * slots with no rows are skipped ([VLLM-EP] docstring: the per-expert loop
 * skips experts with count 0).  Then per token, the weighted sum of its
 * selected experts' outputs in fixed j order ([DS-6964]; [VLLM-EP]
 * ep_reduce_output adds the shared expert: out = routed + shared):
 *     out[t] = bf16( sum_j topk_w[t,j] * y[pair_row[t,j]]  (pairs with row -1 skipped)
 *                    + g_t * shared(x[t]) )
 * where shared() is the gated MLP with W1s/W2s and g_t = sigmoid(x[t] . shared_gate_w)
 * (fp32 dot) when shared_gate_w is given, else 1.
 *
 *   x_perm    [P_cap, H] bf16       permuted activations (moe_permute)
 *   offsets   [S_local+1] int32     row offsets per slot (device; read by the kernels)
 *   P_cap     rows of x_perm's allocation (>= offsets[S_local]; normally T*k)
 *   W1        [S_local, 2I, H] bf16  per slot: I gate rows, then I up rows
 *   W2        [S_local, H, I] bf16
 *   pair_row  [T, k] int32, topk_w [T, k] fp32 (after the mask), or NULL: every
 *             kept pair weighs 1 (routing applied on the input, moe_permute_on_input)
 *   x         [T, H] bf16           input of the shared expert (may be NULL if none)
 *   W1s       [2*I_shared_total, H] bf16 (gate rows then up rows) or NULL
 *   W2s       [H, I_shared_total] bf16 or NULL
 *   shared_gate_w [H] bf16 or NULL
 *   out       [T, H] bf16 out
 * Several shared experts are passed as one gated MLP whose gate rows, up rows
 * and W2 columns are the experts' concatenated (the sum of their outputs). */
MOE_API moe_status_t moe_forward(const moe_bf16_t *x_perm, const int32_t *offsets, int S_local, int64_t P_cap,
                         const moe_bf16_t *W1, const moe_bf16_t *W2, int H, int I,
                         const int32_t *pair_row, const float *topk_w, int64_t T, int k,
                         const moe_bf16_t *x, const moe_bf16_t *W1s, const moe_bf16_t *W2s,
                         int I_shared_total, const moe_bf16_t *shared_gate_w,
                         moe_bf16_t *out, void *ws, size_t ws_bytes, moe_stream_t stream);

/* moe_forward_fp8 -- moe_forward with E4M3 expert weights ([TRT-10985] review
 * of torch_moe.py: the MoE ops have FP8 and NVFP4 paths; the pages fix no
 * format).  Each weight matrix is E4M3 bytes (OCP "fn" encoding) with one fp32
 * scale per row, W[r][c] = scale[r] * e4m3(q[r][c]) -- see
 * moe_quantize_fp8_rows.  The tensor cores still compute in bf16: the weights
 * are widened to bf16 in shared memory (exactly: every E4M3 value is a bf16
 * value), and each accumulator column is multiplied by its row's scale before
 * SwiGLU (FC1) or the store (FC2).  Halves the weight bytes each step reads.
 *
 *   W1q [S_local, 2I, H] uint8, W1_scale [S_local, 2I] fp32
 *   W2q [S_local, H, I] uint8,  W2_scale [S_local, H] fp32
 *   W1sq [2*I_shared_total, H] uint8, W1s_scale [2*I_shared_total] fp32 (or NULL)
 *   W2sq [H, I_shared_total] uint8,   W2s_scale [H] fp32 (or NULL)
 * Everything else as moe_forward. */
MOE_API moe_status_t moe_forward_fp8(const moe_bf16_t *x_perm, const int32_t *offsets, int S_local, int64_t P_cap,
                             const uint8_t *W1q, const float *W1_scale, const uint8_t *W2q,
                             const float *W2_scale, int H, int I, const int32_t *pair_row,
                             const float *topk_w, int64_t T, int k, const moe_bf16_t *x,
                             const uint8_t *W1sq, const float *W1s_scale, const uint8_t *W2sq,
                             const float *W2s_scale, int I_shared_total, const moe_bf16_t *shared_gate_w,
                             moe_bf16_t *out, void *ws, size_t ws_bytes, moe_stream_t stream);

/* Row-wise E4M3 quantisation of a bf16 matrix w [rows, K] (K a multiple of
 * 64), for moe_forward_fp8: scale[r] = amax_c |w[r][c]| / 448 and
 * q[r][c] = e4m3(w[r][c] / scale[r]), both divisions in IEEE binary32 and the
 * conversion to nearest, ties to even (the row's largest |w| becomes +-448
 * exactly); an all-zero row gets scale 0 and q = 0.  Expert weights laid out
 * as [S, R, K] are quantised as one [S*R, K] matrix.  w must be 16-byte and q
 * 8-byte aligned (MOE_ERR_INVALID_ARG otherwise).  Asynchronous on `stream`;
 * allocates nothing. */
MOE_API moe_status_t moe_quantize_fp8_rows(const moe_bf16_t *w, int64_t rows, int K, uint8_t *q, float *scale,
                                   moe_stream_t stream);

/* moe_forward_w8a8 -- moe_forward_fp8 with E4M3 activations as well (the same
 * source, the same silence on the format).  Each expert input row (a row of
 * x_perm) and each bf16 intermediate row h is quantised on its own with a
 * power-of-two scale (moe_quantize_act_rows); the shared experts' input is x,
 * quantised the same way per token.  FC1 and FC2 then run on E4M3 operands
 * (tcgen05.mma kind::f8f6f4, fp32 accumulation), and each accumulator is
 * multiplied by its A row's and its B row's scale.  With topk_w given (weights
 * applied at the output) the rows of x_perm must be the copies of token rows
 * that moe_permute writes: for batches of more than 64 tokens, or when x_perm
 * is NULL, the call then quantises each row of x once and places its codes at
 * the token's pair rows (pair_row) without reading x_perm (moe_permute with
 * x_perm = NULL then skips the row copies); otherwise, and with topk_w = NULL
 * (moe_permute_on_input) or x = NULL, it quantises the rows of x_perm, which
 * must then be given.  Launches two quantisation kernels besides moe_forward's three.  The workspace regions for the
 * quantised rows are part of moe_workspace_size.  Arguments, layouts,
 * ownership and errors as moe_forward_fp8. */
MOE_API moe_status_t moe_forward_w8a8(const moe_bf16_t *x_perm, const int32_t *offsets, int S_local, int64_t P_cap,
                              const uint8_t *W1q, const float *W1_scale, const uint8_t *W2q,
                              const float *W2_scale, int H, int I, const int32_t *pair_row,
                              const float *topk_w, int64_t T, int k, const moe_bf16_t *x,
                              const uint8_t *W1sq, const float *W1s_scale, const uint8_t *W2sq,
                              const float *W2s_scale, int I_shared_total, const moe_bf16_t *shared_gate_w,
                              moe_bf16_t *out, void *ws, size_t ws_bytes, moe_stream_t stream);

/* Row-wise E4M3 quantisation of activations v [rows, K] bf16 (K a multiple of
 * 64), as moe_forward_w8a8 does: per row, scale = 2^e with e the smallest
 * integer >= -126 such that amax_c |v[r][c]| <= 448 * 2^e, and
 * q[r][c] = e4m3(v[r][c] / 2^e) to nearest, ties to even (the division is
 * exact).  An all-zero row gets scale 2^-126 and q = 0.  v must be 16-byte
 * and q 8-byte aligned (MOE_ERR_INVALID_ARG otherwise).  Asynchronous on
 * `stream`; allocates nothing. */
MOE_API moe_status_t moe_quantize_act_rows(const moe_bf16_t *v, int64_t rows, int K, uint8_t *q, float *scale,
                                   moe_stream_t stream);

/* moe_forward_nvfp4 -- moe_forward with NVFP4 experts: E2M1 weights and
 * activations with E4M3 block scales ([TRT-10985] review of torch_moe.py: the
 * MoE ops have FP8 and NVFP4 paths; the pages fix no encoding).  Every expert
 * matrix and every activation row is stored as moe_quantize_nvfp4_rows writes
 * it: the weights with row scales amax / 2688 (pow2 = 0); the expert input rows
 * (of x_perm), the shared experts' input x and the bf16 intermediates h are
 * quantised inside the call with power-of-two row scales (pow2 = 1).  FC1 and
 * FC2 run on tcgen05.mma kind::mxf4nvf4 (one E4M3 scale per 16 elements of
 * both operands, fp32 accumulation); each accumulator is then multiplied by
 * its A row's and its B row's fp32 scale.
 *
 *   W1q [S_local, 2I, H/2] uint8, W1_sf [S_local, 2I, MOE_NVFP4_SF_ROW_BYTES(H)],
 *       W1_scale [S_local, 2I] fp32
 *   W2q [S_local, H, I/2] uint8,  W2_sf [S_local, H, MOE_NVFP4_SF_ROW_BYTES(I)],
 *       W2_scale [S_local, H] fp32
 *   W1sq [2*I_shared_total, H/2], W1s_sf, W1s_scale; W2sq [H, I_shared_total/2],
 *       W2s_sf, W2s_scale (the shared experts as one concatenated MLP; NULL if none)
 * H, I and I_shared_total at most 16384 (MOE_ERR_UNSUPPORTED otherwise).
 * With topk_w and x given (weights applied at the output) the rows of x_perm
 * must be the copies of token rows that moe_permute writes; the call then
 * quantises each token row of x once and places its codes at the rows of its
 * pairs (pair_row) and at the shared experts' row, without reading x_perm, which
 * may be NULL (moe_permute with x_perm = NULL then skips the row copies).  With
 * topk_w = NULL (moe_permute_on_input) or x = NULL it quantises the rows of
 * x_perm, which must be given.  x_perm (when read) and x must be 16-byte
 * aligned.  Launches two quantisation kernels besides moe_forward's three; their
 * scratch is part of moe_workspace_size.  Everything else as moe_forward. */
MOE_API moe_status_t moe_forward_nvfp4(const moe_bf16_t *x_perm, const int32_t *offsets, int S_local, int64_t P_cap,
                               const uint8_t *W1q, const uint8_t *W1_sf, const float *W1_scale,
                               const uint8_t *W2q, const uint8_t *W2_sf, const float *W2_scale, int H, int I,
                               const int32_t *pair_row, const float *topk_w, int64_t T, int k,
                               const moe_bf16_t *x, const uint8_t *W1sq, const uint8_t *W1s_sf,
                               const float *W1s_scale, const uint8_t *W2sq, const uint8_t *W2s_sf,
                               const float *W2s_scale, int I_shared_total, const moe_bf16_t *shared_gate_w,
                               moe_bf16_t *out, void *ws, size_t ws_bytes, moe_stream_t stream);

/* Bytes of one row of NVFP4 block scales of K elements: one E4M3 byte per 16
 * elements, padded with zero bytes to a multiple of 16 bytes (one 16-byte piece
 * per 256 elements). */
#define MOE_NVFP4_SF_ROW_BYTES(K) (16 * (((K) + 255) / 256))

/* NVFP4 quantisation of a bf16 matrix v [rows, K] (K a multiple of 64, at most
 * 16384; MOE_ERR_UNSUPPORTED otherwise), as
 * moe_forward_nvfp4 reads it.  Per row: the row scale s = amax / 2688 (one
 * binary32 division; pow2 = 0, for weights) or the smallest power of two 2^e,
 * e >= -126, with amax <= 2688 * 2^e (pow2 = 1, for activations); per block of
 * 16 elements sb = e4m3(bmax / (6 s)) and per element q = e2m1(v / (sb * s)),
 * every product and division in binary32 and every conversion to nearest with
 * ties to even, saturating (E4M3 at 448, E2M1 at 6).  An all-zero row gets zero
 * codes and block scales (and s = 0 for weights).
 *   q     [rows, K/2] uint8 out    codes, element 2i in the low nibble of byte i
 *   sb    [rows, MOE_NVFP4_SF_ROW_BYTES(K)] uint8 out  E4M3 block scales, then zeros
 *   scale [rows] fp32 out          row scales
 * Expert weights [S, R, K] are quantised as one [S*R, K] matrix.  v must be
 * 16-byte and q 8-byte aligned (MOE_ERR_INVALID_ARG otherwise).  Asynchronous on
 * `stream`; allocates nothing. */
MOE_API moe_status_t moe_quantize_nvfp4_rows(const moe_bf16_t *v, int64_t rows, int K, int pow2, uint8_t *q,
                                     uint8_t *sb, float *scale, moe_stream_t stream);

/* ---- the three stages of moe_forward ------------------------------------ */

/* FC1 + SwiGLU on the tcgen05 tensor cores.  Routed problem: for each of the G
 * groups, rows offsets[g] .. offsets[g+1]-1 of a ([rows_cap, K=H] bf16) times
 * W1[g] ([2I, H]) -> h ([rows_cap, I] bf16).  Shared problem (skipped when
 * I_shared_total = 0): a_shared ([T, H]) times W1s ([2*I_shared_total, H]) ->
 * h_shared ([T, I_shared_total] bf16).  ws: only its status word is used. */
MOE_API moe_status_t moe_grouped_fc1(const moe_bf16_t *a, int64_t rows_cap, const int32_t *offsets, int G,
                             const moe_bf16_t *W1, int H, int I,
                             const moe_bf16_t *a_shared, int64_t T, const moe_bf16_t *W1s,
                             int I_shared_total, moe_bf16_t *h, moe_bf16_t *h_shared,
                             void *ws, size_t ws_bytes, moe_stream_t stream);

/* FC2 on the tcgen05 tensor cores: h ([rows_cap, I]) times W2[g] ([H, I]) ->
 * y ([rows_cap, H] bf16) per group; h_shared ([T, I_shared_total]) times W2s
 * ([H, I_shared_total]) -> y_shared ([T, H] bf16). */
MOE_API moe_status_t moe_grouped_fc2(const moe_bf16_t *h, int64_t rows_cap, const int32_t *offsets, int G,
                             const moe_bf16_t *W2, int H, int I,
                             const moe_bf16_t *h_shared, int64_t T, const moe_bf16_t *W2s,
                             int I_shared_total, moe_bf16_t *y, moe_bf16_t *y_shared,
                             void *ws, size_t ws_bytes, moe_stream_t stream);

/* moe_grouped_fc2 whose routed output row r is stored at y row y_row[r]
 * (y_row [rows_cap] int32, device; its first offsets[G] entries must be
 * distinct rows of y, e.g. the row map moe_a2a_regroup writes); the shared
 * problem's rows are stored as they are.  An entry outside [0, rows_cap) is
 * undefined behaviour (the bounds-checked build flags it and skips the row). */
MOE_API moe_status_t moe_grouped_fc2_scatter(const moe_bf16_t *h, int64_t rows_cap, const int32_t *offsets, int G,
                                     const moe_bf16_t *W2, int H, int I, const moe_bf16_t *h_shared, int64_t T,
                                     const moe_bf16_t *W2s, int I_shared_total, const int32_t *y_row,
                                     moe_bf16_t *y, moe_bf16_t *y_shared, void *ws, size_t ws_bytes,
                                     moe_stream_t stream);

/* moe_grouped_fc1 / moe_grouped_fc2 with E4M3 weights and fp32 row scales
 * (the stages of moe_forward_fp8; layouts as there). */
MOE_API moe_status_t moe_grouped_fc1_fp8(const moe_bf16_t *a, int64_t rows_cap, const int32_t *offsets, int G,
                                 const uint8_t *W1q, const float *W1_scale, int H, int I,
                                 const moe_bf16_t *a_shared, int64_t T, const uint8_t *W1sq,
                                 const float *W1s_scale, int I_shared_total, moe_bf16_t *h,
                                 moe_bf16_t *h_shared, void *ws, size_t ws_bytes, moe_stream_t stream);
MOE_API moe_status_t moe_grouped_fc2_fp8(const moe_bf16_t *h, int64_t rows_cap, const int32_t *offsets, int G,
                                 const uint8_t *W2q, const float *W2_scale, int H, int I,
                                 const moe_bf16_t *h_shared, int64_t T, const uint8_t *W2sq,
                                 const float *W2s_scale, int I_shared_total, moe_bf16_t *y,
                                 moe_bf16_t *y_shared, void *ws, size_t ws_bytes, moe_stream_t stream);

/* The GEMM stages of moe_forward_w8a8: A operands are E4M3 rows with one fp32
 * scale per row (aq [rows_cap, H] + a_scale [rows_cap], a_shared_q [T, H] +
 * a_shared_scale [T]; for FC2 hq [rows_cap, I] + h_scale, h_shared_q
 * [T, I_shared_total] + h_shared_scale), weights as moe_forward_fp8. */
MOE_API moe_status_t moe_grouped_fc1_w8a8(const uint8_t *aq, const float *a_scale, int64_t rows_cap,
                                  const int32_t *offsets, int G, const uint8_t *W1q, const float *W1_scale,
                                  int H, int I, const uint8_t *a_shared_q, const float *a_shared_scale,
                                  int64_t T, const uint8_t *W1sq, const float *W1s_scale, int I_shared_total,
                                  moe_bf16_t *h, moe_bf16_t *h_shared, void *ws, size_t ws_bytes,
                                  moe_stream_t stream);
MOE_API moe_status_t moe_grouped_fc2_w8a8(const uint8_t *hq, const float *h_scale, int64_t rows_cap,
                                  const int32_t *offsets, int G, const uint8_t *W2q, const float *W2_scale,
                                  int H, int I, const uint8_t *h_shared_q, const float *h_shared_scale,
                                  int64_t T, const uint8_t *W2sq, const float *W2s_scale, int I_shared_total,
                                  moe_bf16_t *y, moe_bf16_t *y_shared, void *ws, size_t ws_bytes,
                                  moe_stream_t stream);

/* Unpermute + weighted combine: out[t] = bf16(sum_j topk_w[t,j] * y[pair_row[t,j]]
 * + g_t * y_shared[t]), fp32 accumulation in fixed j order (topk_w NULL: weight
 * 1 for every kept pair).  y_shared may be
 * NULL (no shared expert); g_t as in moe_forward (x and shared_gate_w NULL ->
 * g_t = 1).  pair_row entries outside [0, rows_cap) other than -1 are
 * dropped and flagged. */
MOE_API moe_status_t moe_finalize(const moe_bf16_t *y, int64_t rows_cap, const int32_t *pair_row,
                          const float *topk_w, int64_t T, int k, int H,
                          const moe_bf16_t *y_shared, const moe_bf16_t *x,
                          const moe_bf16_t *shared_gate_w, moe_bf16_t *out,
                          void *ws, size_t ws_bytes, moe_stream_t stream);

/* ---- all-to-all expert parallelism --------------------------------------- */

/* moe_a2a_regroup -- the row reorder of one rank of the all-to-all
 * expert-parallel layer ([TRT-10985] sequence diagram, all-to-all path: the
 * tokens are dispatched to the ranks responsible for their experts, each rank
 * computes the MoE on its local experts, the results go back to the tokens'
 * ranks).  Each rank sends its moe_permute rows (grouped by slot; the slots of
 * one destination rank are a contiguous range), so a rank receives them in
 * EXCHANGE order: source rank 0's rows, then rank 1's, ...; inside a source's
 * block, its rows of local slot 0, then slot 1, ...  The grouped GEMMs take
 * GEMM order: slot 0's rows, then slot 1's, ...; inside a slot, the rows of
 * source 0, then source 1, ... (each source's rows in the order it sent them).
 * The call copies whole rows from one order to the other:
 *
 *   recv_counts [N, S_local] int32   rows source rank n sent for local slot c
 *                                    (the counts exchanged before the rows)
 *   N, S_local   ranks and local slots, N * S_local <= 4096 (MOE_ERR_UNSUPPORTED)
 *   src, dst     [rows_cap, H] bf16, distinct buffers; rows past the total
 *                sum(recv_counts) are neither read nor written
 *   direction    MOE_A2A_TO_GEMM: src in exchange order, dst in GEMM order;
 *                MOE_A2A_TO_EXCHANGE: src in GEMM order, dst in exchange order
 *   offsets      [S_local + 1] int32 out, or NULL: the GEMM-order row offsets of
 *                the local slots (offsets[S_local] = total), for moe_grouped_fc1/fc2
 *   row_map      [rows_cap] int32 out, or NULL: for each of the first `total` rows
 *                of dst, the src row it was copied from (after MOE_A2A_TO_GEMM: the
 *                exchange-order row of each GEMM row, the y_row that lets
 *                moe_grouped_fc2_scatter store FC2's rows straight in exchange order)
 *   ws           workspace: only its status word is used
 *
 * A negative count, or a total above rows_cap, sets MOE_ERR_DEVICE_BOUNDS in the
 * status word and moves no row (offsets and row_map are then not written). */
enum { MOE_A2A_TO_GEMM = 0, MOE_A2A_TO_EXCHANGE = 1 };
MOE_API moe_status_t moe_a2a_regroup(const int32_t *recv_counts, int N, int S_local, const moe_bf16_t *src,
                                     moe_bf16_t *dst, int64_t rows_cap, int H, int direction, int32_t *offsets,
                                     int32_t *row_map, void *ws, size_t ws_bytes, moe_stream_t stream);

/* ---- the expert-parallel reduction by peer loads -------------------------- */

/* The one SUM over the ranks of expert parallelism ([VLLM-EP] ep_reduce_output:
 * each rank's routed plus shared partial output, summed over the ranks;
 * ep_reduce_scatter_output: the same sum, each rank keeping a slice of the rows;
 * [DS-6964]: one reduction per layer), done by plain loads of the ranks'
 * partials instead of a collective library.  Each rank's bf16 partial [T, H]
 * lives in memory every rank can read (its own GPU's, mapped into the others'
 * address spaces with moe_ipc_export / moe_ipc_import); each rank holds an int32
 * flag per rank.  Per step with epoch e (e grows by one per step; flags start
 * at 0, so e starts at 1):
 *   1. a rank writes its partial into slot e % 2 of its two partial buffers,
 *   2. moe_ep_signal raises its flag to e in every rank's flag array,
 *   3. moe_ep_reduce waits until every flag of its own array has reached e and
 *      forms its rows of the sum from slot e % 2 of every rank.
 * Two slots suffice: a rank writes slot e % 2 again at step e + 2 only after its
 * step e + 1 reduce saw every rank's flag e + 1, which each rank raises after
 * its own step e reduce (the last read of that slot) on its stream. */

/* Raise this rank's flag to `epoch` in every rank's flag array: peer_flags is a
 * HOST array of N device pointers, peer_flags[n] = rank n's int32 flags[N] (as
 * mapped on this GPU); flag `rank` of each is written.  Enqueued on `stream`
 * after the work that writes this rank's partial: the kernel waits for it,
 * fences at system scope and stores with release semantics.  N <= 16. */
MOE_API moe_status_t moe_ep_signal(int32_t *const *peer_flags, int N, int rank, int32_t epoch, moe_stream_t stream);

/* out rows [row0, row1) of [T, H] = bf16( sum over n = 0 .. N-1, in that order,
 * of the fp32 values of partials[n] rows ) (row1 = T on every rank: the
 * all-reduce; a slice per rank: the reduce-scatter).  partials is a HOST array
 * of N device pointers to the [T, H] bf16 partials (16-byte aligned; as mapped
 * on this GPU).  The kernel first waits until flags[n] - epoch >= 0 (int32
 * wrap-around) for every n, at most the library's wait limit
 * (moe_set_wait_timeout_ns); on timeout it sets MOE_ERR_TIMEOUT in the status
 * word and writes nothing.  ws: only its status word is used.  N <= 16. */
MOE_API moe_status_t moe_ep_reduce(const moe_bf16_t *const *partials, int N, const int32_t *flags, int32_t epoch,
                                   int64_t row0, int64_t row1, int H, moe_bf16_t *out, void *ws, size_t ws_bytes,
                                   moe_stream_t stream);

/* Host-side mapping of device buffers between processes (CUDA IPC), for the
 * partial buffers and flags above.  moe_ipc_export writes the
 * MOE_IPC_HANDLE_BYTES-byte handle of the allocation holding `ptr` and ptr's
 * offset inside it; moe_ipc_import, in another process, maps that allocation
 * (with peer access enabled) and returns the address of the same byte;
 * moe_ipc_close unmaps it (pass the imported pointer and its offset).  The
 * exporting process must keep the allocation alive while it is mapped. */
#define MOE_IPC_HANDLE_BYTES 64
MOE_API moe_status_t moe_ipc_export(const void *ptr, uint8_t *handle, int64_t *offset);
MOE_API moe_status_t moe_ipc_import(const uint8_t *handle, int64_t offset, void **ptr);
MOE_API moe_status_t moe_ipc_close(void *ptr, int64_t offset);

/* ---- diagnostics ---------------------------------------------------------- */

/* Launch one block whose single thread waits on an mbarrier that nothing ever
 * completes, with the same bounded wait the GEMM kernels use, limited to
 * timeout_ns.  The kernel returns normally and sets MOE_ERR_TIMEOUT in the
 * device status word.  Lets a test check the timeout path without a hang. */
MOE_API moe_status_t moe_debug_wait_timeout(void *ws, size_t ws_bytes, uint64_t timeout_ns, moe_stream_t stream);

/* Set the limit (ns) after which a wait inside a kernel gives up (default 4 s).
 * Process-wide; applies to launches made after the call. */
MOE_API void moe_set_wait_timeout_ns(uint64_t timeout_ns);

/* How the grouped GEMMs map tiles to CTAs (process-wide, for launches made
 * after the call): 0 = (default) one CTA per 128-row tile (tcgen05.mma
 * cta_group::1); 1 = CTA pairs (thread-block clusters of 2) running 2-SM MMAs
 * (cta_group::2, M = 256: each SM stages its A rows and half of the weight
 * tile) when the launch has at least 4 tiles per SM; 2 = CTA pairs whenever a
 * launch has two or more tiles.  All modes give bitwise the same results.
 * Pairs lose on ragged groups with an odd number of 128-row tiles (half a pair
 * idles) and, on a power-capped GB300, on total energy, so 0 is the default.
 * MOE_ERR_INVALID_ARG for other values. */
MOE_API moe_status_t moe_set_gemm_pair_mode(int mode);

/* 1 (default): launch the layer's kernels with programmatic dependent launch,
 * so each kernel's launch and set-up overlap the end of the previous one (each
 * still waits for its predecessor before touching memory); 0: plain stream
 * order.  Process-wide; results are identical.  MOE_ERR_INVALID_ARG otherwise. */
MOE_API moe_status_t moe_set_pdl(int enable);

/* Number of kernel launches the library has issued in this process (all
 * threads, all devices), counted on the host as each launch is made.  A CUDA
 * graph captured from library calls holds the launches counted during its
 * capture; replaying it issues them again without counting. */
MOE_API uint64_t moe_get_launch_count(void);

/* Per-kernel timing of the library's own launches (diagnostics).
 *
 * moe_launch_events_arm(events, n): `events` holds n CUDA event handles
 * (cudaEvent_t, created by the caller with timing enabled; they stay the
 * caller's and must outlive their use).  While armed, each kernel launch the
 * library issues first records the next unused event on the launch's stream,
 * and moe_launch_events_mark records the next one on `stream` with no launch
 * (to close the last kernel's interval).  Under stream capture the record is
 * captured as an external event node, so every replay of the graph records the
 * event again.  While armed, kernels go without programmatic dependent launch,
 * so the time between consecutive events is one kernel (plus the record).
 * Once the n events are used, further launches and marks record nothing.
 * n = 0 (events may be NULL) disarms and forgets the events; arming again
 * starts from the first event.  Process-wide: arm it only while one host thread
 * issues library calls.  MOE_ERR_INVALID_ARG for n < 0 or a NULL array with
 * n > 0; MOE_ERR_CUDA if a record failed (the launch is then not made).
 *
 * moe_launch_events_used(names, cap): how many events have been recorded since
 * arming; when `names` is not NULL, copies the first min(count, cap) labels into
 * it, MOE_LAUNCH_LABEL_BYTES (48) bytes each, zero-terminated: the kernel's name for a launch (grouped
 * GEMMs carry their tile variant, e.g. "grouped_gemm_fc1_n256_short"), "mark"
 * for a mark. */
#define MOE_LAUNCH_LABEL_BYTES 48
MOE_API moe_status_t moe_launch_events_arm(void *const *events, int n);
MOE_API moe_status_t moe_launch_events_mark(moe_stream_t stream);
MOE_API int moe_launch_events_used(char *names, int cap);

#ifdef __cplusplus
}
#endif

#endif /* SERVING_ROUTER_GATE_GB300_MOE_H */
