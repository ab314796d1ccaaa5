/*
 * moe.h -- C ABI of the GB300 small-M routed-MoE decode/verify layer.
 *
 * One call runs a whole routed-MoE layer for M = 1..64 tokens on one GPU:
 *   router gate matvec -> softmax top-k with renormalisation -> on-device
 *   token->expert compaction -> fused gate/up GEMV + SwiGLU -> down GEMV with
 *   the routing-weighted combine in its epilogue.
 * One persistent kernel (one CTA per SM by default, grid-wide waits
 * inside), chained to the previous work on the stream with Programmatic
 * Dependent Launch and capturable in a CUDA graph.  No host
 * synchronisation, no allocation and no device->host copy happens inside the
 * forward call.  Every CTA of the kernel must be resident at once: they are
 * when no other work holds an SM for the kernel's whole duration.  A caller
 * that runs other kernels beside the layer (a collective on a second
 * stream, say) gives the layer fewer CTAs with moe_set_grid and leaves the
 * other SMs to that work; a kernel whose CTAs cannot all become resident
 * reports MOE_ERR_DEVICE_TIMEOUT through moe_get_status (its waits are
 * bounded), it never hangs.
 *
 * Source of the method (page title and section):
 *   "How Ling-3.0-flash reduces batch 1 decoding latency by 54% on 4
 *   Blackwell GPUs" (mirror of the LMSYS post "Chasing the batch-1 floor:
 *   Ling-3.0-flash speculative decode on Blackwell"):
 *     - "Two kinds of idle": a batch-1 step is bounded by the cold read of
 *       the activated expert weights plus the launch floor of small kernels;
 *     - "PDL: the latency floor of stacked small kernels": the router chain
 *       (gate matvec -> top-k) and the MoE chain (align -> up-GEMM ->
 *       activation -> down-GEMM -> combine), producer-independent loads
 *       issued before the dependency wait, the combine as an fp32 sum with
 *       a single final cast;
 *     - "Two fusions and a retune": the pair-axis token->expert bucketing
 *       (stable in pair index, tail beyond the published total unwritten),
 *       SwiGLU in the up-GEMM epilogue with a per-expert gate/up row
 *       interleave applied at weight load;
 *     - "bf16 router gate and lm_head": the router weight is bf16;
 *     - "Economics of speculation at batch 1": verifying M tokens reads the
 *       same weights as verifying one, so one weight pass serves all M.
 *
 * Conventions for every entry point:
 *   - bf16 means IEEE bfloat16 (1-8-7), 2 bytes, little endian.
 *   - "device" pointers are CUDA device (or managed) memory of the current
 *     device; "host" pointers are ordinary host memory.
 *   - Integer status returns are moe_status_t values; 0 is success.
 *   - After any non-zero return, moe_last_error() gives a thread-local
 *     description of the failure.
 *   - A handle is not thread-safe: use one handle from one host thread and
 *     one stream at a time.
 *   - The target is sm_103a (GB300).  Other devices are refused at create.
 */
#ifndef WSE_MOE_H
#define WSE_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same representation as cudaStream_t / cudaEvent_t (opaque pointers), so
 * callers need no CUDA header to use this ABI. */
typedef struct CUstream_st* moe_stream_t;
typedef struct CUevent_st* moe_event_t;

typedef struct moe_layer moe_layer_t; /* opaque; owned by the library */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* bad pointer, size, alignment or handle     */
  MOE_ERR_UNSUPPORTED = 2,    /* valid request outside what the library supports */
  MOE_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed       */
  MOE_ERR_OOM = 4,            /* device allocation failed at create         */
  MOE_ERR_DEVICE_TIMEOUT = 5  /* a bounded in-kernel wait gave up           */
} moe_status_t;

/* Largest M accepted by one forward call (the workspace is sized for it). */
#define MOE_MAX_TOKENS 64

/* Flags for moe_forward_ex. */
#define MOE_FWD_NO_PDL 0x1u /* launch without PDL                            */
#define MOE_FWD_GRAPH 0x2u  /* replay a per-(handle, M) CUDA graph instead of
                               a launch; the graph is captured on first use
                               and updated when the pointers change           */
#define MOE_FWD_TRACE 0x4u  /* record per-CTA phase timestamps of this call
                               (read with moe_read_trace); same results       */
#define MOE_FWD_OUT_F32 0x8u /* `out` is fp32 [M][H] and receives the combine's
                                fp32 sums unrounded: the partial output of one
                                slice of a tensor-parallel split (see
                                moe_combine_partials)                          */
#define MOE_FWD_TEST_SKIP_ARRIVAL 0x40000000u
                            /* test aid: one CTA leaves out one grid-wide
                               arrival, so the call's dependent waits run out
                               after the handle's wait limit and
                               moe_get_status reports MOE_ERR_DEVICE_TIMEOUT;
                               the outputs of such a call are undefined        */

/*
 * moe_create -- build a layer handle from bf16 weights.
 *
 * Defines the layer of the "PDL: ..." section's router and MoE chains.
 *   hidden     H: model width.  Must be a multiple of 256 with H/256 in
 *              {1,2,4,5,8,10,12,16}; (2560 = Ling-3.0-flash width).
 *   n_experts  E: routed experts, topk <= E <= 1024.
 *   topk       k: experts per token, 1 <= k <= 32.
 *   inter      I: expert intermediate width, one of {128, 256, 512},
 *              dividing hidden.
 *   w_router   device bf16 [E][H], row e = router row of expert e
 *              (the hidden -> n_experts mapping, stored one row per expert).
 *              All three weight pointers must be 16-byte aligned.
 *   w_gate_up  device bf16 [E][2I][H]; rows [0,I) are the gate projection,
 *              rows [I,2I) the up projection of each expert.
 *   w_down     device bf16 [E][H][I]; the down projection of each expert.
 * Ownership: the library COPIES the weights into its own device memory
 *   (re-laid out for streaming: gate/up rows interleaved per expert as in
 *   "Two fusions and a retune", fragment order for the tensor-core loads);
 *   the caller may free its buffers when this returns.  The call is
 *   synchronous on the current device: it first waits for all work already
 *   queued on the device (on any stream: the weights may still be being
 *   written by it), then allocates that device's memory (weights ~= the
 *   input size, plus a few MB of workspace) and copies.
 * Returns NULL on error (moe_last_error() says why): invalid sizes or
 *   pointers, a device other than sm_103, or allocation failure.
 */
moe_layer_t* moe_create(int hidden, int n_experts, int topk, int inter,
                        const void* w_router, const void* w_gate_up,
                        const void* w_down);

/*
 * Layer variants of the post's model (zero-initialise, then set fields):
 *   - a shared expert every token passes with weight 1, fused as one more
 *     bucket next to the routed experts ("a 513-expert decode", section "Two
 *     kinds of idle"), with the routed experts' inter size;
 *   - a routed scaling factor: the combine is an fp32 sum times a scale
 *     ("PDL: ..."), here a factor on every routed weight;
 *   - a router bias that chooses the experts without weighing them (the
 *     router top-k "prefetches its bias").
 * Combine per token: out = bf16( sum over slots j < k, in order, of
 * (routed_scale * w_j) * y_j, then + y_shared ), one rounding.
 */
typedef struct {
  const void* w_shared_gate_up; /* device bf16 [2I][H] (gate rows first), 16-byte
                                   aligned, or NULL: no shared expert */
  const void* w_shared_down;    /* device bf16 [H][I], or NULL (both or neither) */
  float routed_scale;           /* factor on every routed weight; <= 0 means 1 */
  int bias_selection_only;      /* 1: moe_set_router_bias's bias picks the
                                   experts only; the weights are the softmax of
                                   the unbiased logits renormalised over the k.
                                   0: the bias shifts the logits for both. */
} moe_layer_opts_t;

/*
 * moe_create_ex -- moe_create with the layer variants (opts NULL: none).
 * The shared expert's weights are copied and re-laid out like the routed
 * ones.  topk_idx / topk_w of the forward calls hold the routed experts
 * only (topk_w unscaled); moe_read_routing also lists the shared expert's
 * pairs (pair M*k + m of token m, expert id n_experts, weight 1) and its
 * pair_w values include the scale.  Errors as moe_create.
 */
moe_layer_t* moe_create_ex(int hidden, int n_experts, int topk, int inter,
                           const void* w_router, const void* w_gate_up,
                           const void* w_down, const moe_layer_opts_t* opts);

/*
 * moe_create_fp8 -- a layer whose expert weights are fp8 (the post: "once
 * fp8 weights shrink the fixed base"): OCP E4M3 codes with one fp32 scale
 * per output row, so the dequantized matrix is diag(scale) * decode(codes);
 * each expert GEMV sums x * code in fp32 and applies the row scale after
 * the sum.  The router stays bf16.  The forward call and its outputs are
 * those of moe_create's layers; the activations and h are taken to f16 on
 * the chip (exact for |values| within f16's normal range, 6.1e-5 .. 65504).
 *   w_router   device bf16 [E][H] (16-byte aligned).
 *   q_gate_up  device uint8 [E][2I][H] E4M3 codes (gate rows first), 16-byte
 *              aligned;      s_gate_up device fp32 [E][2I], 4-byte aligned.
 *              Codes must be finite (not S.1111.111, E4M3's NaN).
 *   q_down     device uint8 [E][H][I] E4M3 codes, 16-byte aligned;
 *              s_down     device fp32 [E][H], 4-byte aligned.
 * hidden, n_experts, topk, inter as moe_create.  The codes and scales are
 * copied (codes re-laid out into 16-row tiles); the caller may free them.
 * Streams half the bytes of a bf16 layer per activated expert (3*H*I bytes
 * + (2I + H) * 4 bytes of scales).  Errors as moe_create.
 */
moe_layer_t* moe_create_fp8(int hidden, int n_experts, int topk, int inter,
                            const void* w_router, const void* q_gate_up,
                            const float* s_gate_up, const void* q_down,
                            const float* s_down);

/*
 * moe_forward -- run the layer on M tokens, asynchronously on `stream`.
 *   x         device bf16 [M][H], 16-byte aligned, read only.
 *   out       device bf16 [M][H]: out[m] = bf16( sum_j w[m][j] * y_j ),
 *             y_j = W_d[e_j] (silu(W_g[e_j] x[m]) * (W_u[e_j] x[m])),
 *             fp32 accumulation, one final rounding ("PDL: ..." section,
 *             single-cast combine).  Must not overlap x.
 *   topk_idx  device int32 [M][k]: the chosen experts of each token in
 *             descending router-logit order, ties to the lower expert id.
 *   M         0 <= M <= MOE_MAX_TOKENS; M = 0 is a no-op returning MOE_OK.
 *   stream    CUDA stream (NULL = legacy default stream).
 * The routing weights are the softmax over all E logits renormalised over
 * the chosen k.  No host sync, allocation or device->host copy: the call can
 * be captured into a caller's CUDA graph.  Errors: MOE_ERR_INVALID_ARG for a
 * NULL handle/pointer or misalignment, MOE_ERR_UNSUPPORTED for M > 64,
 * MOE_ERR_CUDA if a launch fails.  Device-side wait timeouts are reported
 * later by moe_get_status().
 */
int moe_forward(moe_layer_t* h, const void* x, void* out, int32_t* topk_idx,
                int M, moe_stream_t stream);

/*
 * moe_forward_ex -- moe_forward with options.
 *   topk_w  NULL, or device fp32 [M][k] receiving the routing weights.
 *   flags   MOE_FWD_NO_PDL, MOE_FWD_GRAPH, MOE_FWD_TRACE, MOE_FWD_OUT_F32
 *           (then `out` is fp32 [M][H], 4-byte aligned: out[m] = the fp32
 *           sum over slots before the final rounding).
 * Results are bitwise identical for every flag combination (PDL and graph
 * replay change scheduling only).  MOE_FWD_GRAPH on a stream that is being
 * captured by the caller falls back to plain launches (they join the
 * caller's graph).
 */
int moe_forward_ex(moe_layer_t* h, const void* x, void* out, int32_t* topk_idx,
                   float* topk_w, int M, moe_stream_t stream, unsigned flags);

/*
 * moe_forward_timed -- profiling variant: a plain launch without PDL, with
 * ev[0] recorded before the layer kernel and ev[1] after it, on `stream`.
 * ev must point to 2 valid events.  Same results as moe_forward.  Under
 * stream capture the records become event nodes of the graph, so a replay
 * times the kernel with no host gap around it.
 */
int moe_forward_timed(moe_layer_t* h, const void* x, void* out,
                      int32_t* topk_idx, int M, moe_stream_t stream,
                      moe_event_t* ev);

/*
 * moe_set_router_bias -- optional per-expert router bias.
 *   bias  device fp32 [E] added to every logit before selection and softmax
 *         (the "router top-k prefetches its bias" of the "PDL: ..."
 *         section), or NULL to remove it.  The values are copied
 *         (synchronously); the caller keeps ownership of `bias`.
 */
int moe_set_router_bias(moe_layer_t* h, const float* bias);

/*
 * moe_set_grid -- the number of CTAs a forward call of this handle launches.
 *   ctas  1 .. SMs of the device, or 0 for one per SM (the default).
 * The layer kernel's CTAs wait on one another, so all of them must be
 * resident at once; a caller that runs other kernels concurrently with the
 * layer (for example a collective on another stream) leaves SMs to them by
 * giving the layer fewer CTAs.  The work is split over gridDim, so results
 * are the same for every grid (bit for bit).  Synchronises the device and
 * restarts the handle's arrival counts (no forward call of the handle may be
 * in flight); drops the handle's cached graphs.  MOE_ERR_UNSUPPORTED if the
 * grid cannot be resident on an idle device, MOE_ERR_INVALID_ARG outside
 * the range.  Graphs captured by the caller keep the grid they captured.
 */
int moe_set_grid(moe_layer_t* h, int ctas);

/*
 * moe_set_wait_limit -- limit (ns) of every bounded wait inside the layer
 * kernel (0: the default, 2 s).  A forward call whose waits run out leaves
 * its outputs undefined and is reported by moe_get_status.  Tests set a
 * short limit to make a wait run out quickly; graphs cached by the handle
 * are dropped (they hold the old limit).
 */
int moe_set_wait_limit(moe_layer_t* h, unsigned long long ns);

/*
 * moe_combine_partials -- the exchange step of a tensor-parallel split of
 * the layer ("PDL: ..." section: the MoE chain ends in an all-reduce of the
 * GPUs' partial outputs; the post splits the layer four ways).  Each GPU
 * holds 1/G of every expert's intermediate rows (gate and up rows
 * [r*I/G, (r+1)*I/G) and the matching down columns) and runs the full
 * routing; its moe_forward_ex(..., MOE_FWD_OUT_F32) output is the fp32
 * partial sum over its slice.  This call sums G such partials in order and
 * rounds once to bf16, so the split layer rounds exactly once, like the
 * unsplit one:
 *   out[i] = bf16( ((parts[0][i] + parts[1][i]) + ...) + parts[G-1][i] ).
 *   parts  device fp32 [n_parts][n] (contiguous, as an all-gather leaves
 *          them), 16-byte aligned.
 *   n      elements per part (M * hidden), a multiple of 4.
 *   out    device bf16 [n], 8-byte aligned; must not overlap parts.
 * Asynchronous on `stream`; allocates nothing.  MOE_ERR_INVALID_ARG for bad
 * pointers, sizes or alignment; MOE_ERR_CUDA if the launch fails.
 */
int moe_combine_partials(const float* parts, int n_parts, size_t n, void* out, moe_stream_t stream);

/*
 * moe_get_status -- synchronises the device, then returns and clears the
 * handle's sticky device error word: MOE_OK, or MOE_ERR_DEVICE_TIMEOUT if a
 * bounded wait inside the kernel gave up (a staging wait, or a grid-wide
 * wait when not every CTA could be resident), after which the outputs of
 * that call are undefined; moe_last_error() then names the first wait that
 * gave up.  Not for the hot path.
 */
int moe_get_status(moe_layer_t* h);

/* Layer facts for tests and benchmarks (all host values). */
typedef struct {
  int hidden, n_experts, topk, inter;
  int max_tokens;          /* MOE_MAX_TOKENS */
  int n_sms;               /* SMs of the device the handle lives on */
  int gateup_stages;       /* shared-memory ring depth of the gate/up phase
                              (the ring of a call at M = 64: calls with
                              M <= 8 run a second instance, with one token
                              set per expert group; an fp8 layer's has a
                              smaller reduction area and deeper rings) */
  int down_stages;         /* shared-memory stages of the down phase (M = 64) */
  int gateup_tile_bytes;   /* bytes of one gate/up weight tile (8 bf16 or
                              16 fp8 rows x H) */
  int down_tile_bytes;     /* bytes of one down super tile at M = 64: 8
                              cells, one per consumer warp, of one slab (8
                              bf16 or 16 fp8 rows x I) each; a bf16 layer's
                              calls with M <= 8 use cells of up to 512 / I
                              slabs (64 KB super tiles) */
  size_t weight_bytes;     /* device bytes held for the weights */
  size_t workspace_bytes;  /* device bytes held for the workspace */
  int kernels_per_forward; /* kernel launches per forward call (1) */
  int router_split;        /* hidden-dim split of the router matvec units */
  size_t smem_bytes;       /* dynamic shared memory per CTA at M = 64 */
  int shared_expert;       /* 1 if the layer has a shared expert */
  float routed_scale;      /* factor on every routed weight */
  int bias_selection_only; /* 1 if the router bias only picks the experts */
  int fp8_experts;         /* 1 if the expert weights are E4M3 codes */
  int grid_ctas;           /* CTAs a forward call launches (moe_set_grid) */
  unsigned long long wait_limit_ns; /* limit of the kernel's bounded waits */
} moe_info_t;

int moe_get_info(const moe_layer_t* h, moe_info_t* out);

/*
 * moe_read_routing -- copy the last forward call's on-device compaction to
 * host memory (synchronises the device; test aid, not the hot path).
 * The compaction is the pair-axis bucketing of "Two fusions and a retune":
 * the NP = M*k (token, slot) pairs sorted by expert id, stable in pair index
 * p = token*k + slot, split into groups of at most 16 pairs per expert.
 *   n_groups, n_active   host int*: groups written, distinct experts.
 *   grp_expert, grp_start, grp_cnt   host int32 [cap]: per group its expert,
 *                        first sorted position and pair count (<= 16).
 *   pair_list            host int32 [NP]: pair id at each sorted position.
 *   pair_w               host fp32 [NP]: routing weight of each pair id.
 *   cap                  capacity of the grp_* arrays (>= NP suffices).
 * With a shared expert NP = M*(k+1): pairs M*k .. M*k+M-1 are the shared
 * expert's (expert id n_experts).
 */
int moe_read_routing(moe_layer_t* h, int M, int* n_groups, int* n_active,
                     int32_t* grp_expert, int32_t* grp_start, int32_t* grp_cnt,
                     int32_t* pair_list, float* pair_w, int cap);

/*
 * moe_read_trace -- copy the phase timestamps of the last call made with
 * MOE_FWD_TRACE (synchronises the device; profiling aid).
 *   out   host uint64 [cap]: for CTA c, slots [32c, 32c + 32) hold
 *         %globaltimer values in ns: 0 dependency wait passed, 1 router
 *         matvec done, 2 (unused), 3 groups counted by the producer warp
 *         (its first gate/up copies follow at once),
 *         4 first gate/up tile consumed, 5 gate/up loop left, 6 every CTA's
 *         statically split gate/up tiles reduced (publisher), 7 down loop
 *         left, 8 combine done (the CTAs that combine), 9 producer issued
 *         its last gate/up tile, 10 producer issued its last down tile,
 *         12 top-k done, 13 compaction done (the other warps), 14 first down
 *         tile consumed,
 *         15 combine starts (combining CTAs; calls of more than 8 tokens:
 *         after every CTA's weighted rows are written, fewer: at once, the
 *         rows carry their call's index and are polled), 17 every
 *         CTA's gate/up tiles reduced (publisher), 18 this CTA's static
 *         gate/up tiles counted in, 19 CTA started, 20 prologue done (before
 *         the dependency wait).  Slot 11 holds the CTA's gate/up tile COUNT
 *         and slot 16 its down super-tile COUNT.  Slots of phases a CTA did
 *         not reach keep older values.
 * Returns the number of values written (min(cap, 32 x SMs)), or on error
 * the negated moe_status_t (a positive status could not be told apart from a
 * count).
 */
int moe_read_trace(moe_layer_t* h, uint64_t* out, int cap);

/*
 * moe_route_static -- the router alone (gate matvec + softmax top-k with
 * renormalisation) for callers that cannot allocate device memory.
 *
 * The source post has no counterpart: this is a library service.  Callers
 * that cannot call cudaMalloc (code running while someone else captures a
 * CUDA graph, allocators that forbid outside allocations, paths that must not
 * risk an allocation failure or the synchronisation an allocation can imply)
 * get the same routing as moe_forward without a handle: the call allocates
 * nothing.  Its scratch (partial logits, an arrival counter, a status word)
 * is one fixed array inside the library image, 78,080 bytes, which every GPU
 * that loads the library holds until the process exits.  Its arithmetic is
 * moe_forward's own router (same matvec split and summation order, same
 * top-k), so both give the same routing for the same x -- for a layer whose
 * router bias shifts the logits for both the choice and the weights (the
 * default; a layer made with bias_selection_only weighs its experts with the
 * unbiased logits, this call with the biased ones).
 *   hidden, n_experts, topk   as for moe_create.
 *   x          device bf16 [M][hidden], 16-byte aligned.
 *   w_router   device bf16 [n_experts][hidden], 16-byte aligned; read in
 *              place (not copied), caller-owned.
 *   bias       device fp32 [n_experts] added to the logits, or NULL.
 *   M          0 <= M <= 16 (the scratch is sized for 16 tokens).
 *   topk_idx   device int32 [M][topk]: experts by descending logit, ties to
 *              the lower id (same values as moe_forward's topk_idx).
 *   topk_w     NULL or device fp32 [M][topk]: the renormalised weights.
 *   stream     CUDA stream.
 * The first call on a device resolves the array's device address (a one-time
 * set-up); make that first call before any stream capture.  Every call on a
 * device uses the same array and it keeps
 * the last call's contents (the counter that must start at zero is cleared by
 * each call on its stream), so calls whose work can overlap on the GPU --
 * different streams without ordering -- race.  Returns MOE_ERR_UNSUPPORTED
 * (with a moe_last_error() message) for M > 16, sizes outside the limits, or
 * a device whose SM count gives moe_forward's matvec split more partial
 * logits than the array holds (never on a 152-SM GB300: the split would
 * differ, and with it the summation order); MOE_ERR_INVALID_ARG for bad
 * pointers, MOE_ERR_CUDA if set-up or the launch fails.  Errors found on the
 * device (a top-k without a candidate, which cannot happen while
 * topk <= n_experts) are not returned here: read them with
 * moe_route_static_read_status before the next call on the device.
 */
int moe_route_static(int hidden, int n_experts, int topk, const void* x,
                     const void* w_router, const float* bias, int M,
                     int32_t* topk_idx, float* topk_w, moe_stream_t stream);

/*
 * moe_route_static_read_status -- copy the device status word of the last
 * moe_route_static call on the current device to `status` (device or host
 * int, 4-byte aligned) with one asynchronous copy on `stream`; allocates
 * nothing.  The value is 0, or 8 if a top-k found no candidate.  Enqueue it
 * on the stream of the call it reads, before the next moe_route_static call
 * (which clears the word); read `status` after the stream reaches the copy.
 * MOE_ERR_INVALID_ARG for a NULL pointer, MOE_ERR_CUDA if set-up or the copy
 * fails.
 */
int moe_route_static_read_status(int* status, moe_stream_t stream);

/* moe_destroy -- synchronises the handle's device, frees everything.
 * NULL is a no-op. */
void moe_destroy(moe_layer_t* h);

/* Thread-local text of the last error set on this thread ("" if none). */
const char* moe_last_error(void);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* WSE_MOE_H */
