/*
 * moe_q8k.h — C ABI of the block-quantized routed MoE layer for GB300 (sm_103a).
 *
 * The operation is the per-token Mixture-of-Experts layer of the SSD/RAM-tiered
 * MoE engines described on the Pulsar README and the Strata pages: a router
 * chooses top-k experts per token (softmax or sigmoid gates renormalised over
 * the k), tokens are bucketed by expert, every selected expert and the shared
 * expert run gate/up matrix-vector products on q8_K-quantized activations
 * against block-quantized weights (integer sub-block dot products), a SwiGLU,
 * and the down projection on the re-quantized intermediate, and the outputs
 * are combined with the gates into the residual.
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers owned by the caller unless stated otherwise.
 *    Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream) and allocates no memory.
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns a negative status and launches nothing.  Errors found
 *    on the device (an out-of-range expert id, a bounded wait that ran out)
 *    are recorded in the workspace status word and read with moe_get_status.
 *  - Calls are reentrant for distinct workspaces; calls sharing a workspace
 *    must be ordered on one stream.
 *  - Results are deterministic: no floating-point atomics; every sum is taken
 *    in a fixed order.
 *
 * Matrix byte format (every format): W[N, K] with N, K multiples of 256 is a
 * sequence of "slabs", one per (row group of 32 rows, 256-column super-block),
 * row-group-major.  A slab holds the super-blocks of its 32 rows field by
 * field: 32 headers ({fp16 d, fp16 dmin} words, or fp16 d alone), then the
 * 32 scale/min records, then the code lines (16 bytes per row per line).
 * Full bit-level description: synth/layout.py.
 *   Q4_K-style: 144 bytes per super-block, 4-bit codes, eight 32-weight
 *     sub-blocks with 6-bit scale and min; weight = d*scale_j*q - dmin*min_j.
 *   Q2_K-style: 84 bytes, 2-bit codes, sixteen 16-weight sub-blocks with
 *     4-bit scale and min; weight = d*scale_j*q - dmin*min_j.
 *   Q5_K-style: 176 bytes, as Q4_K-style with 5-bit codes.
 *   Q3_K-style: 110 bytes, 3-bit codes, sixteen sub-blocks with 6-bit scales
 *     u_j; weight = d*(u_j - 32)*(q - 4).
 *   Q6_K-style: 210 bytes, 6-bit codes, sixteen sub-blocks with int8 scales;
 *     weight = d*scale_j*(q - 32).
 *   IQ2-style grid format: 70 bytes (2.19 bits per weight); per group of 8
 *     weights a grid index u and 7 sign bits (the 8th sign makes the minus
 *     signs even), per 32 weights a 4-bit scale t; weight = d*(2t+1)*sign*
 *     C[u][i], C the 256 vectors of {1,3,5}^8 with the smallest sums of
 *     squares (equal sums in increasing base-3 order, element 0 first).
 * (Pulsar README, "What it does today": Q4_K/Q6_K matmuls on q8_K
 * activations, IQ2_XXS builds; "Get a model": q3_K/q5_K/q6_K tensors;
 * Strata engine article, finding 7: i-quant codebook lookups cost decode
 * compute.  The "-style" layouts and the grid are this library's own.)
 * Every matrix pointer must be 16-byte aligned.
 */
#ifndef MOE_Q8K_H
#define MOE_Q8K_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)    /* NULL or misaligned pointer, bad size  */
#define MOE_ERR_UNSUPPORTED (-2)    /* shape outside the supported range     */
#define MOE_ERR_WORKSPACE (-3)      /* workspace too small                   */
#define MOE_ERR_CUDA (-4)           /* a CUDA launch or API call failed      */
#define MOE_ERR_DEVICE_BOUNDS (-5)  /* device saw an out-of-range index      */
#define MOE_ERR_DEVICE_TIMEOUT (-6) /* a bounded device wait ran out         */

/* ---- limits ------------------------------------------------------------ */
#define MOE_MAX_EXPERTS 1024 /* E                                          */
#define MOE_MAX_SHARED 2     /* n_shared                                   */
#define MOE_MAX_TOPK 16      /* top_k                                      */
#define MOE_MAX_DIM 16384    /* H and I                                    */

typedef enum {
  MOE_FMT_Q4K = 0, /* Q4_K-style: 144 B per super-block                            */
  MOE_FMT_Q2K = 1, /* Q2_K-style: 84 B                                             */
  MOE_FMT_Q5K = 2, /* Q5_K-style: 176 B (Q4_K-style with 5-bit codes)             */
  MOE_FMT_Q3K = 3, /* Q3_K-style: 110 B, 3-bit codes, signed 6-bit scales, no min  */
  MOE_FMT_Q6K = 4, /* Q6_K-style: 210 B, 6-bit codes, int8 scales, no min          */
  MOE_FMT_IQ2G = 5 /* IQ2-style grid format: 70 B, grid indices and signs          */
} moe_wfmt;
typedef enum { MOE_ROUTE_SOFTMAX = 0, MOE_ROUTE_SIGMOID = 1 } moe_route_kind;

/* Shape of one MoE layer. */
typedef struct {
  int32_t H;        /* hidden size, multiple of 256, <= MOE_MAX_DIM            */
  int32_t I;        /* expert intermediate size, multiple of 256               */
  int32_t E;        /* routed experts, 1..MOE_MAX_EXPERTS                      */
  int32_t top_k;    /* experts per token, 1..min(E, MOE_MAX_TOPK)              */
  int32_t n_shared; /* always-on shared experts, 0..MOE_MAX_SHARED             */
  int32_t route;    /* moe_route_kind                                          */
  int32_t fmt;      /* moe_wfmt of every expert matrix                         */
  int32_t T_max;    /* largest token count of a call (sizes the workspace)     */
} moe_layer_desc;

/* One expert's matrices: gate [I, H], up [I, H], down [H, I].  In a pointer
 * table a NULL gate means "not mine": the expert is not present and
 * contributes nothing (Pulsar README, "How the streaming works": explicit
 * per-(token, slot) gate/up/down pointers, NULL = not mine). */
typedef struct {
  const void* gate;
  const void* up;
  const void* down;
} moe_expert_ptrs;

/* Byte offsets of the intermediate results inside a moe_layer_forward
 * workspace (for inspection after the call; all 256-byte aligned).
 * P = T_max * (top_k + n_shared) is the number of (token, slot) rows. */
typedef struct {
  size_t status;   /* int32[4]: [0] = device status word                       */
  size_t xq;       /* int8  [T_max, H]      q8_K codes of x                    */
  size_t xd;       /* float [T_max, H/256]  q8_K scales of x                   */
  size_t xbs;      /* int16 [T_max, H/16]   sums of 16 codes                   */
  size_t logits;   /* float [T_max, E]                                         */
  size_t ids;      /* int32 [T_max, top_k]                                     */
  size_t gates;    /* float [T_max, top_k]                                     */
  size_t gap;      /* float [T_max]  l_(k) - l_(k+1)                           */
  size_t counts;   /* int32 [E + n_shared]                                     */
  size_t offsets;  /* int32 [E + n_shared + 1]                                 */
  size_t perm;     /* int32 [P]  bucket position -> slot index                 */
  size_t inv;      /* int32 [P]  slot index -> bucket position                 */
  size_t h;        /* float [P, I]     silu(G) * U, rows in bucket order       */
  size_t hq;       /* int8  [P, I]     q8_K codes of h                         */
  size_t hd;       /* float [P, I/256]                                         */
  size_t hbs;      /* int16 [P, I/16]                                          */
  size_t y;        /* float [P, H]     expert outputs, indexed by slot index   */
  size_t phase_ns; /* uint64 [16] SM clock-cycle stamps (clock64) taken by CTA 0
                      of the single-launch decode kernel at its phase
                      boundaries: [0] start, [1] router done, [2] after
                      barrier 1, [9] top-k done, [10] counts and scan,
                      [11] bucket positions, [3] tile plan done, [4] gate/up
                      done, [5] after barrier 2, [6] down done, [7] after
                      barrier 3, [8] combine done; [15] = 1 after the
                      sequential schedule, 2 after the pipelined one (see
                      moe_stack_forward); a pipelined run stamps, for the stage
                      holding the gate/up of layer L-2: [0] stage start, [3]
                      x staged, [4] gate/up, [6] down of the layer before,
                      [1] router of layer+2, [8] combine, [12] next layer's
                      routing taken and its experts prefetched; [14] the
                      grid size (CTAs) of the single-launch kernel         */
  size_t total;    /* bytes required                                           */
} moe_ws_layout;

/* Workspace bytes moe_layer_forward needs for `desc` (0 if desc is invalid). */
size_t moe_layer_workspace_size(const moe_layer_desc* desc);

/* Offsets of the intermediates in that workspace.  Returns MOE_OK or
 * MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED. */
int moe_workspace_layout(const moe_layer_desc* desc, moe_ws_layout* out);

/* q8_K quantization of x[T, K] (fp32, row-major, K a multiple of 256):
 * per 256-element block d = max|x| / 127 (IEEE fp32 division) and
 * q = round-half-away-from-zero(x / d) (IEEE fp32 division), q = 0 when
 * d = 0; bsum16 = sums of each 16 consecutive codes.
 * Outputs q int8 [T, K], d float [T, K/256], bsum16 int16 [T, K/16]
 * (bsum16 may be NULL).  Source: Pulsar README, "Fidelity notes" (all
 * matmuls run on q8_0/q8_K activations with integer dp4a dots). */
int moe_q8k_quantize(const float* x, int64_t T, int64_t K, int8_t* q, float* d, int16_t* bsum16,
                     void* stream);

/* Router and top-k.  logits[t, e] = sum_h w_router[e, h] * x[t, h] + bias[e]
 * in fp32 from the unquantized fp32 x [T, H]; w_router fp32 [E, H]; bias fp32
 * [E] or NULL.  The k largest logits are selected (equal logits: lower expert
 * index first) into ids int32 [T, k] in descending order; gates float [T, k]:
 * route 0 softmax over the k selected logits, route 1 sigmoid of each
 * selected logit divided by their sum.  gap float [T] (nullable) =
 * l_(k) - l_(k+1), +inf when k == E.  logits float [T, E] is an output the
 * caller provides.  Sources: Pulsar README, "What it does today" (softmax
 * router, qwen3moe); Pulsar digest note, section 1 (512-way sigmoid-gated
 * router + shared expert); Strata summary (~10 experts per token). */
int moe_route_topk(const float* x, const float* w_router, const float* bias, int32_t T, int32_t H,
                   int32_t E, int32_t k, int32_t route, float* logits, int32_t* ids, float* gates,
                   float* gap, void* stream);

/* Workspace bytes moe_bucket needs for T tokens, k slots, E experts. */
size_t moe_bucket_workspace_size(int32_t T, int32_t k, int32_t E, int32_t n_shared);

/* Bucketing of the T*k (token, slot) pairs by expert (a counting sort, stable
 * by token) plus one bucket per shared expert holding every token.
 *   counts  int32 [E + n_shared]
 *   offsets int32 [E + n_shared + 1] (exclusive prefix sum of counts)
 *   perm    int32 [T*(k + n_shared)]: perm[offsets[e] + i] is the slot index of
 *           the i-th pair of bucket e; slot index = t*k + s for routed pairs and
 *           T*k + sh*T + t for shared expert sh.
 *   inv     int32 [T*(k + n_shared)] (nullable): inv[perm[j]] = j.
 * ids outside [0, E) are recorded as MOE_ERR_DEVICE_BOUNDS in the status word
 * of ws and skipped.  Source: Pulsar README, "How the streaming works" (per
 * prefill chunk, one expert union across the whole batch). */
int moe_bucket(const int32_t* ids, int32_t T, int32_t k, int32_t E, int32_t n_shared,
               int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv, void* ws,
               size_t ws_bytes, void* stream);

/* Workspace bytes moe_expert_ffn needs for `desc` with T tokens. */
size_t moe_expert_ffn_workspace_size(const moe_layer_desc* desc, int32_t T);

/* Expert FFNs over the buckets.  For every expert e with a non-NULL gate in
 * `table` (device array of E + n_shared entries) and every slot row j of its
 * bucket (token t of slot perm[j]):
 *   G = gate_e . q8_K(x_t),  U = up_e . q8_K(x_t)   (integer sub-block dots)
 *   h = silu(G) * U  (fp32),  y_slots[perm[j]] = down_e . q8_K(h)
 * Rows of experts whose gate is NULL are written as zeros.  Each expert's
 * weights are read once for all the tokens of its bucket (per group of up to
 * 16 tokens).  q/d/bsum16: q8_K of x as moe_q8k_quantize writes them (T rows
 * of H).  counts/offsets/perm: as moe_bucket writes them.  y_slots float
 * [T*(k + n_shared), H] indexed by slot index.  Sources: Pulsar README, "What
 * it does today" (warp-cooperative Q4_K/Q6_K matmuls on q8_K activations,
 * FFN triple gate/up/down) and "How the streaming works". */
int moe_expert_ffn(const moe_layer_desc* desc, const moe_expert_ptrs* table, const int8_t* q,
                   const float* d, const int16_t* bsum16, const int32_t* counts,
                   const int32_t* offsets, const int32_t* perm, int32_t T, float* y_slots,
                   void* ws, size_t ws_bytes, void* stream);

/* Gate-weighted combine into the residual, in a fixed order:
 *   out[t] = (sum_{s<k} gates[t, s] * y_slots[t*k + s] + sum_sh y_slots[T*k + sh*T + t])
 *            + residual[t]
 * residual float [T, H] may be NULL (treated as 0) and may alias out.
 * Source: Pulsar README, "Fidelity notes" (the per-slot sum). */
int moe_combine(const float* y_slots, const float* gates, int32_t T, int32_t H, int32_t k,
                int32_t n_shared, const float* residual, float* out, void* stream);

/* The whole layer: q8_K(x), router top-k, bucketing, expert FFNs and the
 * combine, on T <= desc->T_max tokens.  x float [T, H]; w_router float [E, H];
 * router_bias float [E] or NULL; residual float [T, H] or NULL (may alias
 * out); out float [T, H]; table: device array of E + n_shared expert pointer
 * records.  ids_out int32 [T, k] and gates_out float [T, k] are optional
 * copies of the routing (NULL to skip).  ws: at least
 * moe_layer_workspace_size(desc) bytes, 256-byte aligned; the intermediates
 * stay in it after the call at the offsets moe_workspace_layout gives.
 * Sources: Pulsar README, "How the streaming works" (per token the router
 * picks the experts first; the expert kernels receive explicit per-(token,
 * slot) gate/up/down pointers, NULL = not mine; one expert union per batch)
 * and "Fidelity notes" (every matmul on q8_K activations with integer dp4a
 * dots; the layer output is the per-slot sum of the expert outputs). */
int moe_layer_forward(const moe_layer_desc* desc, const moe_expert_ptrs* table,
                      const float* w_router, const float* router_bias, const float* x,
                      const float* residual, float* out, int32_t T, int32_t* ids_out,
                      float* gates_out, void* ws, size_t ws_bytes, void* stream);

/* The pointers of one layer of a stack (see moe_stack_forward); the same
 * meaning and rules as the arguments of moe_layer_forward. */
typedef struct {
  const moe_expert_ptrs* table; /* device array of E + n_shared records      */
  const float* w_router;        /* [E, H]                                     */
  const float* router_bias;     /* [E] or NULL                                */
  const float* x;               /* [T, H]; may be a previous layer's out      */
  const float* residual;        /* [T, H] or NULL; may alias out              */
  float* out;                   /* [T, H]                                     */
  int32_t* ids_out;             /* [T, k] or NULL                             */
  float* gates_out;             /* [T, k] or NULL                             */
} moe_layer_ptrs;

/* Workspace bytes moe_stack_forward needs for n_layers layers of `desc`
 * (0 if desc is invalid or n_layers < 1): a moe_layer_forward workspace
 * followed by per-layer buffers (logits, q8_K(x), routing, h, y) and the
 * stack's dependency counters.  Grows linearly with n_layers and T_max. */
size_t moe_stack_workspace_size(const moe_layer_desc* desc, int32_t n_layers);

/* A stack of n_layers MoE layers of the same shape in ONE cooperative
 * launch, with the results of running them one after the other: a layer's x
 * may point at the previous layer's out (a decode step through the stack).
 * The stack runs as a sequence of small work items (router rows, routing,
 * gate/up row groups, down row groups, combine chunks) handed out
 * round-robin, ordered by per-layer dependency counters instead of grid
 * barriers.  When no layer's out overlaps another layer's x, residual or
 * out (independent inputs), neighbouring layers overlap; otherwise each
 * layer starts after the previous one has finished.  Both orders give the
 * same results.  `layers` is a DEVICE array of n_layers records.  Only the
 * single-launch decode shapes are accepted: T <= 16, T*top_k <= 256, and the
 * layer's staging fits in shared memory; otherwise MOE_ERR_UNSUPPORTED (run
 * moe_layer_forward per layer instead).  ws: moe_stack_workspace_size(desc,
 * n_layers) bytes, 256-byte aligned, its 16-byte status block zero before
 * the first call (e.g. a zero-filled allocation); ids/gates/counts/offsets/
 * perm in it hold the last layer's routing.  Stacks of fewer than 4
 * layers with many expert items per SM (a wide layer on its own) run
 * instead on the barrier-pipelined single-launch kernel, which prefetches
 * all of a CTA's items of a layer at once.  phase_ns[15] reports what ran: 3 dataflow,
 * layers overlapped; 4 dataflow, one layer after the other; 2 pipelined
 * kernel, neighbouring layers overlapped; 1 pipelined kernel, sequential.  Sources: Pulsar
 * README, "How the streaming works" (the next layer's experts are fetched
 * while the current one computes); Strata summary (the per-token layer loop
 * run as captured, replayed work with no allocation on the token path). */
int moe_stack_forward(const moe_layer_desc* desc, int32_t n_layers, const moe_layer_ptrs* layers, int32_t T,
                      void* ws, size_t ws_bytes, void* stream);

/* Byte offsets, from the start of a moe_stack_forward workspace, of the
 * buffers that layer `layer` of the dataflow stack kernel (MOE_STACK_DATAFLOW)
 * fills, for inspection after a call with the same desc, n_layers and T.
 * P = T * (top_k + n_shared) bucket positions; bucket positions are ordered
 * by expert (routed experts ascending, then the shared experts), and within
 * an expert by token. */
typedef struct {
  size_t logits; /* float [T, E]      router logits                             */
  size_t xq;     /* int8  [T, H]      q8_K codes of x                           */
  size_t xd;     /* float [T, H/256]                                            */
  size_t xbs;    /* int16 [T, H/16]                                             */
  size_t ids;    /* int32 [T, top_k]  selected experts                          */
  size_t gates;  /* float [T, top_k]  renormalised gates                        */
  size_t tok;    /* int32 [P]         token of each bucket position             */
  size_t slot;   /* int32 [P]         slot index of each bucket position (the
                                      perm of moe_bucket)                       */
  size_t h;      /* float [P, I]      silu(G) * U, rows in bucket order         */
  size_t y;      /* float [P, H]      expert outputs, by slot index             */
} moe_stack_ws_layout;

/* Fills `out` for layer 0 <= layer < n_layers.  Host-side only.  Returns
 * MOE_OK, MOE_ERR_INVALID_ARG, or MOE_ERR_UNSUPPORTED for shapes that
 * moe_stack_forward rejects.  No counterpart on the pages. */
int moe_stack_layer_layout(const moe_layer_desc* desc, int32_t n_layers, int32_t T, int32_t layer,
                           moe_stack_ws_layout* out);

/* Largest workspace, in bytes, that moe_layer_forward_noalloc can serve. */
#define MOE_NOALLOC_MAX_WORKSPACE ((size_t)16 << 20)

/* moe_layer_forward without a workspace argument and without any memory
 * allocation.  (No counterpart on the pages: this is a convenience of this
 * library.)  It is meant for callers that cannot call cudaMalloc where they
 * run the layer: an engine whose memory planner gives the whole device to
 * its own pool, a plugin that only receives the tensors it reads and writes,
 * or a token loop that must not allocate because allocating can synchronise
 * the device mid-step.  The caller still passes every input and output; the
 * intermediates live in a 16 MiB array that is part of the library (every
 * GPU that loads the library holds it until the process exits).
 *   - Arguments and results are those of moe_layer_forward.
 *   - Descriptors whose moe_layer_workspace_size exceeds
 *     MOE_NOALLOC_MAX_WORKSPACE are rejected with MOE_ERR_WORKSPACE (decode
 *     shapes fit: e.g. H=6144, I=2048, 192 experts, top-8, 16 tokens needs
 *     about 5 MB).
 *   - Each call looks up the array's device address in the context current
 *     on the calling thread (a host-side lookup; the runtime's primary
 *     context or a context the caller made current both work).  The first
 *     call on a device may also load the library's device code there: make
 *     that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents;
 *     each call clears the parts that must start at zero.  Calls that
 *     overlap on the GPU (other streams, other host threads) race on it:
 *     order them.
 *   - Device-side errors are not reported (there is no workspace to read
 *     with moe_get_status); use moe_layer_forward for that. */
int moe_layer_forward_noalloc(const moe_layer_desc* desc, const moe_expert_ptrs* table,
                              const float* w_router, const float* router_bias, const float* x,
                              const float* residual, float* out, int32_t T, int32_t* ids_out,
                              float* gates_out, void* stream);

/* Synchronizes `stream`, then reads and clears the status word of a
 * workspace written by moe_layer_forward, moe_bucket or moe_expert_ffn.
 * Returns MOE_OK, a device-recorded error, or MOE_ERR_CUDA. */
int moe_get_status(void* ws, void* stream);

/* The cudaError_t code of the last failed CUDA call made by this library on
 * the calling host thread (0 if none).  Explains an MOE_ERR_CUDA status. */
int moe_last_cuda_error(void);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(int status);

/* Profiling hook.  While set, the expert kernels launched by this host
 * thread record the next unused entries of `events` (cudaEvent_t handles
 * created by the caller with timing enabled) on their stream, immediately
 * before and after each launch: two entries per single-launch decode layer
 * (moe_layer_forward with T <= 16 and T*top_k <= 256), four per expert-FFN
 * sequence otherwise (gate/up kernel, then down kernel).  Under stream
 * capture a record is made with cudaEventRecordExternal (an event-record
 * node of the graph), outside capture with a plain cudaEventRecord.  When
 * the array is used up, or a record fails (the error is consumed), recording
 * stops.  events = NULL or n_events = 0
 * turns the hook off.  Returns MOE_OK or MOE_ERR_INVALID_ARG. */
int moe_trace_events(void* const* events, int32_t n_events);

/* Number of entries recorded since the last moe_trace_events call. */
int32_t moe_trace_used(void);

/* Total number of kernel launches this library has issued in the process
 * (all host threads, all devices), including launches recorded into a CUDA
 * graph during stream capture.  The difference across one call counts that
 * call's kernels.  This library has no other side effect to observe. */
unsigned long long moe_kernel_launch_count(void);

/* Which implementation moe_layer_forward uses for T tokens of `desc`
 * (no device work):
 *   MOE_PATH_DECODE_FUSED   one cooperative launch (T <= 16, T*top_k <= 256
 *                           and the routing state fits the kernel's shared
 *                           memory; if the device cannot make the grid
 *                           co-resident the call falls back to the GEMV path)
 *   MOE_PATH_GEMV           separate routing / bucketing / dp4a GEMV kernels
 *   MOE_PATH_TENSOR_PREFILL tcgen05 grouped GEMMs over the expert buckets
 *                           (T*top_k > 256 and T*top_k >= 16 * E: experts
 *                           average at least 16 routed tokens)
 * Returns one of them, or a negative status for an invalid descriptor or T. */
#define MOE_PATH_DECODE_FUSED 0
#define MOE_PATH_GEMV 1
#define MOE_PATH_TENSOR_PREFILL 2
int moe_layer_path(const moe_layer_desc* desc, int32_t T);

/* Token tile of the tensor-core prefill path (MOE_PATH_TENSOR_PREFILL): an
 * expert with c routed tokens gets t = ceil(c / n) token tiles of
 * ceil(c / t) bucket rows each (the last one shorter), n the value
 * returned.  Host-side only; launches nothing.  No counterpart on the pages
 * (their prefill GEMM tiles are not specified). */
int moe_prefill_tile_tokens(void);

/* Which single-launch kernel moe_stack_forward runs for a stack of n_layers
 * layers of `desc` at T tokens on a device with n_sms SMs (n_sms <= 0: the
 * current device's).  Host-side only; launches nothing:
 *   MOE_STACK_DATAFLOW   the layers as a dataflow of small items ordered by
 *                        per-layer counters (phase_ns[15] = 3 or 4)
 *   MOE_STACK_PIPELINED  the barrier-pipelined kernel (phase_ns[15] = 1 or 2):
 *                        layers with more than 2 gate/up + down items per SM
 *                        in stacks of fewer than 4 layers
 * Returns one of them, MOE_ERR_UNSUPPORTED for shapes moe_stack_forward
 * rejects, or MOE_ERR_INVALID_ARG.  No counterpart on the pages. */
#define MOE_STACK_PIPELINED 1
#define MOE_STACK_DATAFLOW 2
int moe_stack_kernel(const moe_layer_desc* desc, int32_t n_layers, int32_t T, int32_t n_sms);

/* Test hook for failure detection: one kernel waits on a word of the
 * workspace's status block for a value nothing ever writes, with the same
 * kind of bound as every wait in the library's kernels; after limit_us
 * microseconds (1 .. 1,000,000) it records MOE_ERR_DEVICE_TIMEOUT in the
 * status word and returns, leaving the context usable.  moe_get_status then
 * reports it.  No counterpart on the pages.  Returns MOE_OK, or
 * MOE_ERR_INVALID_ARG / MOE_ERR_CUDA. */
int moe_debug_wait_timeout(void* ws, int32_t limit_us, void* stream);

/* Test hook: the integer sub-block sums of the device dot routine that the
 * expert kernels use, for matrix w [N, K] against q8_K codes q [T, K]:
 *   isum int32 [T, N, K/256, n_sub] = sum over sub-block j of q_w * q_a,
 *   bsum int32 [T, K/256, n_sub]    = sum over sub-block j of q_a,
 * n_sub = 8 (Q4_K-style) or 16 (Q2_K-style).  T <= 16. */
int moe_debug_subblock_dots(int32_t fmt, const void* w, int32_t N, int32_t K, const int8_t* q,
                            int32_t T, int32_t* isum, int32_t* bsum, void* stream);

/* Workspace bytes moe_debug_prefill_sums needs (0 for invalid sizes). */
size_t moe_debug_prefill_sums_workspace_size(int32_t N, int32_t K, int32_t T);

/* Test hook: the integer super-block sums that the tensor-core (prefill)
 * path forms, for matrix w [N, K] (N a multiple of 128, K of 256) against
 * the q8_K rows q [T, K], d [T, K/256], bsum16 [T, K/16] (as
 * moe_q8k_quantize writes them):
 *   S int32 [T, N, K/256] = sum_j scale_j * (sum over sub-block j of q_w * q_a)
 *   M int32 [T, N, K/256] = sum_j min_j * (sum over sub-block j of q_a)
 * computed by the same tcgen05 GEMM kernel and TMEM accumulators as the
 * prefill expert FFNs (token tiles of up to 128 rows), with an epilogue that
 * writes S and M instead of the rescaled sum.  ws: at least
 * moe_debug_prefill_sums_workspace_size(N, K, T) bytes, 256-byte aligned.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG / UNSUPPORTED / WORKSPACE or
 * MOE_ERR_CUDA.  Source: Pulsar README, "What it does today" (int8
 * tensor-core expert GEMMs that keep the weights block-quantized and
 * rescale per quant block). */
int moe_debug_prefill_sums(int32_t fmt, const void* w, int32_t N, int32_t K, const int8_t* q, const float* d,
                           const int16_t* bsum16, int32_t T, int32_t* S, int32_t* M, void* ws, size_t ws_bytes,
                           void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_Q8K_H */
