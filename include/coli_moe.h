/*
 * coli_moe.h -- C ABI of libcolimoe, the routed Mixture-of-Experts layer of a
 * GLM-5.2-style decoder on one sm_103a GPU.
 *
 * The layer (colibrì v1.0 README, "What's implemented"; "Colibri (colibrì):
 * GLM-5.2 local inference on 25 GB of RAM", "How it works (validated core
 * mechanics)"):
 *   1. sigmoid noaux_tc router: s = sigmoid(x . Wr^T); experts ranked by
 *      s + correction_bias inside the topk_group best groups; gate weights are
 *      the unbiased s of the selection renormalised, times
 *      routed_scaling_factor;
 *   2. batch-union dispatch: each distinct expert of a call is streamed from
 *      HBM once and applied to every position routed to it;
 *   3. Q8_0-style int8 activations (blocks of 32, one fp32 scale each);
 *   4. packed-int4 (or int8) x int8 SwiGLU expert products with per-row fp32
 *      weight scales; h = silu(g) * u is re-quantised to Q8_0 before the down
 *      product;
 *   5. y = sum_j w_j * expert_j(x) + sum_s shared_s(x).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers, row-major, owned by the caller;
 *     the library allocates nothing and keeps no state between calls.
 *   - Every pointer must be 16-byte aligned (TMA bulk copies read them).
 *   - Work is enqueued on `stream`; no call synchronises except
 *     coli_moe_status().  A call whose return value is not COLI_OK enqueued
 *     nothing.
 *   - Data-dependent failures (non-finite input, an out-of-range expert id,
 *     an expired bounded wait) cannot be returned synchronously: they are OR-ed
 *     into a sticky status word at the start of the workspace and read (and
 *     cleared) with coli_moe_status().
 *   - Calls that share a workspace must be ordered on one stream.
 *   - Kernels of this library may start while the kernel before them on the
 *     stream is finishing (programmatic dependent launch).  Before that
 *     kernel has completed they read only weights (router_w, corr_bias,
 *     expert records and scales), never x, routing or the workspace, so one
 *     call's outputs may be the next call's inputs directly.
 */
#ifndef COLI_MOE_H
#define COLI_MOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes (synchronous). */
#define COLI_OK            0
#define COLI_EINVAL       -1   /* bad shape, config or null pointer            */
#define COLI_EALIGN       -2   /* a pointer is not 16-byte aligned             */
#define COLI_EWORKSPACE   -3   /* workspace smaller than coli_moe_workspace_size */
#define COLI_ECUDA        -4   /* a CUDA launch or query failed                */
#define COLI_EUNSUPPORTED -5   /* shape outside the kernels' limits            */

/* Device status bits (asynchronous, sticky until read by coli_moe_status). */
#define COLI_STATUS_NONFINITE 1u  /* non-finite router logit, bias or activation */
#define COLI_STATUS_BADIDX    2u  /* forward saw an expert id outside [-1, E)    */
#define COLI_STATUS_TIMEOUT   4u  /* a bounded device wait expired               */

/* Layer shape.  Limits (COLI_EINVAL / COLI_EUNSUPPORTED otherwise):
 * hidden % 128 == 0, inter % 128 == 0, shared_inter % 128 == 0 when
 * n_shared > 0, n_experts <= 1024, n_experts % n_groups == 0,
 * n_groups <= 32, 1 <= topk_group <= n_groups,
 * 1 <= top_k <= topk_group * n_experts / n_groups, top_k <= 32,
 * 0 <= n_shared <= 8, weight_bits in {2, 4, 8}; a gate+up row pair of
 * hidden and four down rows of max(inter, shared_inter) must each fit in
 * 32 KiB (int4: hidden <= 32768, intermediate sizes <= 16384; int8: half;
 * int2: double).  Packed int2 (colibrì v1.0 README, "What's implemented":
 * int8 / packed int4 / packed int2 weights with per-row scales) takes
 * per-row scales only; it runs on the fused single-position kernel for one
 * position per call, on the few-position kernels for 2 to 4 and on the
 * general expert kernel beyond. */
typedef struct coli_moe_cfg {
    int32_t hidden;                 /* H                                    */
    int32_t n_experts;              /* E routed experts                     */
    int32_t n_groups;               /* G expert groups (E/G experts each)   */
    int32_t topk_group;             /* groups kept per token                */
    int32_t top_k;                  /* experts selected per token (k)       */
    int32_t inter;                  /* I, intermediate size of routed experts */
    int32_t n_shared;               /* always-on shared experts             */
    int32_t shared_inter;           /* intermediate size of shared experts  */
    int32_t weight_bits;            /* 4: packed int4, 2: packed int2, 8: int8 */
    float   routed_scaling_factor;  /* multiplies the renormalised weights  */
    int32_t group_size;             /* 0: one scale per output row;
                                       64: one per 64 weights of a row ("gs64",
                                       int4 only: COLI_EUNSUPPORTED with int8
                                       or int2) */
    int32_t ep_rank;                /* expert-parallel shard of this call   */
    int32_t ep_size;                /* shards (0 or 1: no sharding)         */
} coli_moe_cfg;

/* Expert-parallel sharding (colibrì v1.0 README, "Experimental resident CUDA
 * backend": each expert lives whole on one device; JustVugg/colibri README,
 * "Local cluster mode": one batch-union request per layer to each worker).
 * With ep_size = P > 1 a call computes only its shard's part of the layer:
 *   - routed expert e belongs to shard e mod P.  `weights.experts` and
 *     `expert_scales` then hold only this shard's experts, in ascending id
 *     order: expert e (e mod P == ep_rank) is local record e / P;
 *   - the shared experts belong to shard 0 (the other shards pass no shared
 *     weights and compute none);
 *   - the router is not sharded: every shard runs it on the same x and gets
 *     the same topk_idx / topk_w;
 *   - routed slots whose expert belongs to another shard are skipped like
 *     id -1 (no status bit), so the union tables list this shard's experts
 *     only, and y is the shard's partial output
 *         y_r[t] = sum_{j: idx[t][j] mod P == r} w_j o_j + [r == 0] sum_s o_s[t];
 *   - the sum of y_r over the P shards is the layer's output; the caller
 *     forms it (e.g. one all-reduce of y per layer call).
 * Requires 0 <= ep_rank < ep_size <= n_experts (COLI_EINVAL otherwise);
 * ep_size 0 or 1 needs ep_rank 0.  The workspace size depends on the shard
 * (shard 0 holds the shared experts' pairs), so size it with the shard's own
 * cfg. */

/* Expert weights.  One expert "record" is its three matrices stored adjacent
 * (colibrì "JustVugg/colibri" README, "Never wait for the disk twice": an
 * expert's three matrices are read in one go):
 *     gate [Ie][H], up [Ie][H], down [H][Ie]     (Ie = inter or shared_inter)
 * each row-major with K (the reduction dimension) contiguous.
 *   weight_bits 8: one int8 code per weight.
 *   weight_bits 4: two codes per byte; byte j of a row holds element 2j in the
 *                  low nibble and 2j+1 in the high nibble, each stored as
 *                  code + 8 (codes in [-8, 7]).
 *   weight_bits 2: four codes per byte; byte j of a row holds elements
 *                  4j .. 4j+3, element 4j+m in bits 2m and 2m+1, each stored
 *                  as code + 2 (codes in [-2, 1]).
 * Records are consecutive: expert e starts at experts + e * record_bytes,
 * record_bytes = (2*Ie*H + H*Ie) * weight_bits / 8 (with expert-parallel
 * sharding, e is the local record index e / ep_size; see below).
 * Scales are fp32 per output row, consecutive per expert:
 *     expert_scales[e * (2*I + H) + {0..I-1: gate, I..2I-1: up, 2I..: down}]
 * and likewise shared_scales with shared_inter.
 * With group_size 64 (the group-scaled container the colibri GLM-5.2 quick
 * start recommends, "2. Get the model") every run of 64 weights of a row has
 * its own fp32 scale: per expert 3*I*H/64 scales,
 *     gate [I][H/64] | up [I][H/64] | down [H][I/64], each row-major,
 * and an output is sum over Q8_0 blocks b of s[row][b/2] * d_b * (block dot). */
typedef struct coli_moe_weights {
    const void*  experts;        /* [n_experts] records                 */
    const float* expert_scales;  /* [n_experts][2*inter + hidden]       */
    const void*  shared;         /* [n_shared] records (shared_inter)   */
    const float* shared_scales;  /* [n_shared][2*shared_inter + hidden] */
} coli_moe_weights;

/* Bytes of workspace needed for calls with up to max_T positions.  The
 * workspace is caller-owned device memory; it must be prepared once with
 * coli_moe_workspace_init() and may then be reused by any number of calls on
 * one stream.  Returns 0 on an invalid config. */
size_t coli_moe_workspace_size(const coli_moe_cfg* cfg, int32_t max_T);

/* Clears the header of a workspace (enqueued on `stream`): the status word,
 * the device counters and the router's tagged exchange words, i.e. the first
 * min(ws_bytes, 8704) bytes. */
int coli_moe_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream);

/* Router: "How it works (validated core mechanics)" of the GLM-5.2 write-up
 * ("Colibri (colibrì): GLM-5.2 local inference on 25 GB of RAM")
 * (sigmoid affinities, bias for ranking only, lower id wins ties, unbiased
 * renormalised weights, non-finite input rejected) with DeepSeek-V3 group
 * limiting: group score = sum of the two best biased scores of the group,
 * the topk_group best groups kept (ties to the lower group id), dropped
 * groups never selectable.
 *   x          [T][H]  fp32 activations
 *   router_w   [E][H]  fp32 router weight
 *   corr_bias  [E]     fp32 correction bias (ranking only)
 *   topk_idx   [T][k]  int32 out: expert ids by descending biased score
 *   topk_w     [T][k]  fp32  out: s_sel / sum(s_sel) * routed_scaling_factor
 * Logits are fp32.  A position with a non-finite logit or bias gets ids -1
 * and weights 0, and sets COLI_STATUS_NONFINITE.  T == 0 is a no-op. */
int coli_moe_route(const coli_moe_cfg* cfg, const float* x, int32_t T,
                   const float* router_w, const float* corr_bias,
                   int32_t* topk_idx, float* topk_w,
                   void* ws, size_t ws_bytes, cudaStream_t stream);

/* Q8_0-style activation quantisation (colibrì v1.0 README, "What's
 * implemented", integer-dot kernels): per block of 32 consecutive values,
 * d = amax/127 (IEEE fp32), inv = d > 0 ? 1/d : 0,
 * q = clamp(roundf(x * inv), -127, 127) (half away from zero).
 *   x [T][K] fp32 in, K % 32 == 0;  q [T][K] int8 out;  d [T][K/32] fp32 out.
 * A non-finite value gives code 0 for its element (no status word: this
 * entry point takes no workspace). */
int coli_moe_quantize_act(const float* x, int32_t T, int32_t K,
                          int8_t* q, float* d, cudaStream_t stream);

/* The expert layer for given routing (colibrì v1.0 README, "What's
 * implemented": Q8_0-style int8 activations against packed int4 / int8
 * weights, batch-union MoE, the always-on shared expert; "Experimental Metal
 * backend": the routed-expert SwiGLU; the combine weights are the router's, as
 * "How it works (validated core mechanics)" of the GLM-5.2 write-up gives
 * them): quantise x, build the batch-union
 * tables, run each distinct expert once over its positions (gate/up, SwiGLU,
 * re-quantise h, down) and combine
 *     y[t] = sum_j topk_w[t][j] * o[t,j] + sum_s o_shared_s[t]
 * in fixed j order (deterministic, no floating-point atomics).
 *   x        [T][H] fp32;   topk_idx [T][k] int32 (id -1: slot skipped);
 *   topk_w   [T][k] fp32;   y [T][H] fp32 out.
 * Ids outside [-1, E) are skipped and set COLI_STATUS_BADIDX; non-finite
 * activations set COLI_STATUS_NONFINITE.  T == 0 is a no-op. */
int coli_moe_forward(const coli_moe_cfg* cfg, const coli_moe_weights* weights,
                     const float* x, int32_t T,
                     const int32_t* topk_idx, const float* topk_w, float* y,
                     void* ws, size_t ws_bytes, cudaStream_t stream);

/* The whole layer (the router and the expert layer above, with the passages
 * they cite): coli_moe_route followed by coli_moe_forward, with the
 * same arguments, results and status rules as the two calls (topk_idx and
 * topk_w are outputs here, and the forward part reads them).  For a single
 * position (T == 1, packed int4 or int2) that fits the fused kernel's shared memory,
 * the router runs inside the expert-layer kernel: one launch per call, the
 * shared expert's gate/up rows requested before the routing is known.  The
 * results are bit-identical to the two separate calls. */
int coli_moe_layer(const coli_moe_cfg* cfg, const coli_moe_weights* weights,
                   const float* x, int32_t T,
                   const float* router_w, const float* corr_bias,
                   int32_t* topk_idx, float* topk_w, float* y,
                   void* ws, size_t ws_bytes, cudaStream_t stream);

/* The two launches coli_moe_forward makes, callable separately (e.g. to time
 * the expert kernel alone; the operations and passages of coli_moe_forward).  coli_moe_dispatch quantises x and builds the
 * union tables in ws; coli_moe_experts runs the expert products and the
 * combine from those tables.  Same arguments and rules as coli_moe_forward;
 * coli_moe_experts must follow a coli_moe_dispatch with the same T on the
 * same workspace. */
int coli_moe_dispatch(const coli_moe_cfg* cfg, const float* x, int32_t T,
                      const int32_t* topk_idx, void* ws, size_t ws_bytes,
                      cudaStream_t stream);
int coli_moe_experts(const coli_moe_cfg* cfg, const coli_moe_weights* weights,
                     int32_t T, const float* topk_w, float* y,
                     void* ws, size_t ws_bytes, cudaStream_t stream);

/* Synchronises `stream`, returns the workspace's status bits in *status and
 * clears them. */
int coli_moe_status(void* ws, cudaStream_t stream, uint32_t* status);

/* Static text for a return code. */
const char* coli_moe_strerror(int code);

/* ---- a stack of layers ---------------------------------------------------
 * One decode step through a stack of MoE layers with the hidden state kept
 * on the device between layers (JustVugg/colibri README, "Never wait for the
 * disk twice": the residual stream stays resident on the GPU across layers,
 * COLI_CUDA_PIPE=2).  Layer l runs coli_moe_layer on xs[l]; then a small
 * kernel writes the next layer's input
 *     xs[l+1] = xs[l] + residual[l]            (add_output == 0)
 *     xs[l+1] = (xs[l] + y[l]) + residual[l]   (add_output == 1)
 * in fp32.  Nothing returns to the host between layers; the whole step can
 * be captured once in a CUDA graph and replayed.
 *   layers    [n_layers] per-layer config, weights, router weight and bias;
 *             every layer has the same hidden and top_k (COLI_EINVAL
 *             otherwise); weight formats and the other shapes may differ
 *   xs        [n_layers + 1][T][H] fp32: xs[0] is read, xs[1..] written
 *   residual  [n_layers][T][H] fp32 (NULL: zero)
 *   topk_idx  [n_layers][T][k] int32 out, topk_w [n_layers][T][k] fp32 out
 *   y         [n_layers][T][H] fp32 out: each layer's output
 *   ws        one workspace of at least the largest
 *             coli_moe_workspace_size(layers[l].cfg, T) (COLI_EWORKSPACE
 *             otherwise), prepared with coli_moe_workspace_init
 * Arguments are checked for every layer before anything is enqueued; status
 * bits of all layers accumulate in the workspace's status word. */
typedef struct coli_moe_stack_layer {
    coli_moe_cfg     cfg;
    coli_moe_weights weights;
    const float*     router_w;   /* [E][H] */
    const float*     corr_bias;  /* [E]    */
} coli_moe_stack_layer;

int coli_moe_stack_forward(const coli_moe_stack_layer* layers, int32_t n_layers, int32_t T,
                           float* xs, const float* residual, int32_t add_output,
                           int32_t* topk_idx, float* topk_w, float* y,
                           void* ws, size_t ws_bytes, cudaStream_t stream);

/* ---- inspection (tests) -------------------------------------------------
 * Byte offsets, inside the workspace of coli_moe_workspace_size(cfg, max_T),
 * of the tables and intermediates coli_moe_dispatch / coli_moe_experts leave
 * behind, so that a test can compare them with a reference.  Layouts:
 *   n_entries   int32: routed distinct experts U + n_shared
 *   entry_expert[U+n_shared] int32: ascending routed ids, then E + s
 *   entry_count [U+n_shared] int32: positions per entry
 *   entry_offset[U+n_shared+1] int32: first pair slot of each entry
 *   pair_token  [P] int32, pair_slot_of[T][k] int32 (-1 = skipped)
 *   qx [T][H] int8, dx [T][H/32] fp32  (Q8_0 of x)
 *   qh [P][Imax] int8, dh [P][Imax/32] fp32 (Q8_0 of h per pair slot)
 *   o  [P][H] fp32 (expert output per pair slot)
 * with P = T*k + n_shared*T and Imax = max(inter, shared_inter).  For
 * weight_bits 4, qx and qh hold each group of 8 consecutive codes in the
 * order 0,2,4,6,1,3,5,7 (the order of the low then high nibbles of 4 packed
 * bytes); for weight_bits 2 each group of 16 in the order 0,4,8,12, 1,5,9,13,
 * 2,6,10,14, 3,7,11,15 (the order of the four 2-bit fields of 4 packed bytes);
 * for weight_bits 8 the order is natural. */
typedef struct coli_moe_ws_layout {
    size_t status, n_entries, entry_expert, entry_count, entry_offset,
           pair_token, pair_slot_of, qx, dx, qh, dh, o, total;
} coli_moe_ws_layout;
int coli_moe_workspace_layout(const coli_moe_cfg* cfg, int32_t max_T,
                              coli_moe_ws_layout* out);

/* Test entry point: coli_moe_forward run through the same kernels compiled
 * with a dump of the exact int32 per-32-block dot products:
 *   acc_gu [P][2][Imax][H/32] int32   (gate then up, per pair slot)
 *   acc_d  [P][H][Imax/32]    int32   (down, per pair slot)
 * Either pointer may be NULL.  Slower than coli_moe_forward. */
int coli_moe_forward_dump(const coli_moe_cfg* cfg, const coli_moe_weights* weights,
                          const float* x, int32_t T,
                          const int32_t* topk_idx, const float* topk_w, float* y,
                          void* ws, size_t ws_bytes,
                          int32_t* acc_gu, int32_t* acc_d, cudaStream_t stream);

/* ---- no-allocation variant ----------------------------------------------
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory to pass a workspace -- a plain C or FFI
 * host that links only this library and owns no allocator, or a runtime that
 * keeps the whole device-memory budget and forbids stray cudaMalloc calls.
 *
 * coli_moe_forward_static computes exactly what coli_moe_forward computes,
 * with its workspace taken from one static device array of
 * COLI_STATIC_WS_BYTES inside the library (held on every GPU that loads the
 * library until the process exits).  It calls no cudaMalloc, cudaFree or
 * other allocating routine.  The caller still passes x, routing and y.
 *   - Limit: the layer's workspace for T positions must fit in
 *     COLI_STATIC_WS_BYTES (24 MiB: the GLM-5.2-shaped layer up to T = 76);
 *     larger T returns COLI_EWORKSPACE and enqueues nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it per
 *     device ordinal for the life of the process; make that first call before
 *     any stream capture.  The cache assumes the runtime's primary context:
 *     after cudaDeviceReset, or from another driver-API context on the same
 *     device, the cached address is stale and must not be used (this entry
 *     point then gives undefined results).
 *   - Every call on a device shares the one array: calls that overlap on the
 *     GPU (different streams, or host threads without ordering) race and give
 *     wrong results.  Calls ordered on one stream are safe; each call rewrites
 *     every table and counter it reads.
 *   - Device status bits (non-finite input, expert ids outside [-1, E), an
 *     expired bounded wait) are recorded in the array but cannot be read or
 *     cleared by the caller.  In those cases y is undefined: rows of
 *     positions with non-finite x, or with an out-of-range id, and every row
 *     after an expired wait may hold anything.  Callers that need to detect
 *     them use coli_moe_forward with a workspace and coli_moe_status. */
#define COLI_STATIC_WS_BYTES (24u << 20)
int coli_moe_forward_static(const coli_moe_cfg* cfg, const coli_moe_weights* weights,
                            const float* x, int32_t T,
                            const int32_t* topk_idx, const float* topk_w, float* y,
                            cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* COLI_MOE_H */
