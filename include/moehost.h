/*
 * moehost.h -- C ABI of the GB300 (sm_103a) library for the mixture-of-experts
 * layer of a decode step whose experts do not all fit in HBM.
 *
 * Method (from "DeepSeek-V4.1-Flash on One GB300 Without the Second GPU: What the
 * Sidecar Is Worth", section 1, The idea): the router picks the top-k experts per
 * token; cold experts live in pinned host memory; one kernel per layer copies only
 * the routed cold experts into a shared HBM slot scratch and remaps their ids; one
 * grouped SwiGLU expert call then runs over all experts as if they were resident;
 * outputs are combined with the router weights; between steps a residency manager
 * promotes often-picked cold experts and demotes quiet hot ones.
 *
 * Conventions
 *  - Every call returns an int status: MOE_OK (0) or a negative MOE_ERR_* code.
 *    A call that returns MOE_ERR_INVALID_ARG has launched nothing; after
 *    MOE_ERR_CUDA part of its work may already be enqueued.  Where a call lists no
 *    errors, a null handle or pointer gives MOE_ERR_INVALID_ARG and a failed CUDA
 *    call MOE_ERR_CUDA.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    All device work is enqueued on it; nothing synchronises the stream except
 *    residency_update on an acting step in the synchronous residency mode (it
 *    reads the pick counters on the host), moe_get_status, moe_layer_get_loc and
 *    moe_layer_get_counts.  In the default deferred mode residency_update waits
 *    (host side) only for the previous acting call's counter copy.
 *  - Errors found by a kernel after launch (non-finite logits, an expert id out of
 *    range) are written to the layer's device status word (first error wins);
 *    moe_get_status reads it.
 *  - Ownership: the caller owns every buffer it passes (device memory, and host
 *    blobs that are pinned and mapped, e.g. cudaHostAlloc or torch pin_memory).
 *    The library borrows raw pointers for the life of the layer and owns only its
 *    handles and small internal tables (placement map, phys-id pointer table, pick
 *    counters, status word), freed by the destroy calls.
 *  - Shapes: H and I multiples of 128; 1 <= k <= 32; k <= E <= 1024.
 *  - Host threads: a layer (and the scratch it shares) keeps host-side state
 *    (placement map, pending-copy flag, step count), so calls on one layer, or on
 *    layers sharing a scratch, must not run concurrently from several host
 *    threads; distinct layers with distinct scratches may.  moe_combine,
 *    moe_quant_mxfp4 and moe_residency_plan hold no state.
 *
 * Expert blob format (one contiguous blob per expert, every plane 16-byte aligned):
 *   w13 nibbles [2I][H/2] | w13 scales [2I][H/32] | w2 nibbles [H][I/2] | w2 scales [H][I/32]
 *   MXFP4: E2M1 elements, E8M0 scale per 32-element block along the reduction
 *   dimension ("A 475 GB Model Across Two Workstations, With the Table on Disk",
 *   Abstract: routed experts ship in MXFP4).  w13 rows 0..I-1 are the gate
 *   projection, rows I..2I-1 the up projection (the fused w13/w2 planes of "Milo
 *   and James Try Inference Engineering", offload flag table).  Rows are K-major:
 *   element k of a row is in byte k/2, low nibble when k is even.  Scale byte b
 *   of a row is the exponent of elements 32b..32b+31.
 *
 * Placement: loc[e] in [0, n_hot) is an HBM slot; loc[e] = n_hot + c is cold slot
 * c, whose bytes live in host blob c and are copied to scratch slot c when routed.
 * The physical id of a pick is loc of its expert.
 */
#ifndef MOEHOST_H
#define MOEHOST_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)
#define MOE_ERR_CUDA (-2)
#define MOE_ERR_NONFINITE (-3)
#define MOE_ERR_BAD_EXPERT (-4)
#define MOE_ERR_TIMEOUT (-5)
#define MOE_ERR_NOMEM (-6)
#define MOE_ERR_INJECTED (-7)
#define MOE_ERR_SCRATCH_TOO_SMALL (-8)

/* Layer parameters.
 *  E, k        experts and picks per token ("Milo and James Try Inference
 *              Engineering", the mixture-of-experts paragraph: 384 experts, 6 per
 *              token).
 *  H, I        hidden and expert intermediate sizes.
 *  n_hot       experts resident in HBM; n_cold = E - n_hot in pinned host memory
 *              ("DeepSeek-V4.1-Flash on One GB300 ...", section 1: 255 / 129).
 *  renorm      0: pick weight = softmax probability; 1: divided by the sum over
 *              the k picks.
 *  swap_every  residency_update acts on every swap_every-th call (0 = never).
 *  max_swaps   at most this many swaps per acting update (<= 64).
 *  hysteresis  a cold expert is promoted over a hot one only when its window
 *              count exceeds hysteresis times the hot one's (same page, section 3:
 *              3.0 is the published default).
 *  host_mirror 0: cold_blobs_host holds the n_cold cold slots' blobs and a swap
 *              exchanges bytes between an HBM slot and a host blob.  1:
 *              cold_blobs_host holds a pinned copy of every expert, indexed by
 *              expert id (E blobs); a demotion moves no bytes and a promotion
 *              copies the expert into its HBM slot from its scratch slot when that
 *              slot still holds this layer's copy of it, else from its host copy.
 *              The host copies must equal the HBM-resident experts' bytes.
 *  zero_copy   0: cold_gather copies the picked cold experts into their scratch
 *              slots and moe_grouped_ffn reads them there.  1 (calls of at most 64
 *              tokens): cold_gather only remaps, and moe_grouped_ffn reads the
 *              picked cold experts' weights in place from their pinned host blobs,
 *              on the layer's copy stream alongside the experts in HBM ("Milo and
 *              James Try Inference Engineering": reading expert rows from pinned
 *              host memory over the link; "Running High-Quality DeepSeek V4 Flash
 *              on One 96 GB GPU": mapped host planes read in place).  Larger calls
 *              copy as with 0. */
typedef struct moe_params {
    int E, k, H, I, n_hot, n_cold;
    int renorm;
    int swap_every;
    int max_swaps;
    float hysteresis;
    int host_mirror;
    int zero_copy;
} moe_params;

typedef struct moe_scratch moe_scratch;
typedef struct moe_layer moe_layer;

/* Bytes of one expert blob for (H, I): 3*H*I/2 nibble bytes + 3*H*I/32 scale
 * bytes.  Returns 0 if H or I is not a positive multiple of 128. */
size_t moe_expert_bytes(int H, int I);

/* Shared cold-slot scratch ("DeepSeek-V4.1-Flash on One GB300 ...", section 1:
 * one scratch area with a slot per cold expert, shared by all layers because they
 * run one after another).  slot_dev: caller-owned device memory of
 * n_slots * expert_bytes bytes, 256-byte aligned; slot c starts at
 * slot_dev + c * expert_bytes.  All layers that share it must run their
 * cold_gather and moe_grouped_ffn calls in stream order.  The library keeps a
 * small device table of which layer last copied into each slot.
 * Errors: MOE_ERR_INVALID_ARG (null, n_slots < 0, misaligned, not device memory),
 * MOE_ERR_CUDA, MOE_ERR_NOMEM. */
int moe_scratch_create(int n_slots, size_t expert_bytes, void* slot_dev, moe_scratch** out);
int moe_scratch_destroy(moe_scratch* s);

/* One MoE layer.  hot_blobs_dev[h] (h < n_hot): device pointer of HBM slot h's
 * blob.  cold_blobs_host[c] (c < n_cold): host pointer of cold slot c's blob,
 * pinned and mapped; with host_mirror = 1 instead cold_blobs_host[e] (e < E) is
 * the host copy of expert e.  init_loc: host array [E], a bijection onto [0, E).
 * The scratch must have at least n_cold slots of moe_expert_bytes(H, I) bytes.
 * Validates shapes, 16-byte alignment, memory kinds (cudaPointerGetAttributes)
 * and the map.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA, MOE_ERR_NOMEM. */
int moe_layer_create(const moe_params* p, moe_scratch* scratch, void* const* hot_blobs_dev,
                     void* const* cold_blobs_host, const int32_t* init_loc, moe_layer** out);
int moe_layer_destroy(moe_layer* L);

/* Router: top-k, softmax weights and token-to-expert bucketing for T tokens
 * ("Milo and James Try Inference Engineering", the mixture-of-experts paragraph;
 * "DeepSeek-V4.1-Flash on One GB300 ...", section 1: the copy kernel looks at
 * which experts the router picked).
 *  logits   device fp32 [T][E] row-major.
 *  topk_ids device int32 [T][k]: expert e is picked iff fewer than k experts have
 *           a larger logit or an equal logit and a lower index; listed by that
 *           rank (descending logit, ties to the lower index).
 *  topk_w   device fp32 [T][k]: softmax probability of each pick over all E
 *           (renorm: divided by the sum over the picks).
 *  counts   device int32 [E]; offsets device int32 [E+1] (exclusive prefix);
 *  entries  device int32 [T*k]: pick ids t*k+j grouped by expert, ascending.
 * Also adds the picks to the layer's window counters used by residency_update.
 * A token with a non-finite logit gets ids 0..k-1 and weights 0, and the status
 * word becomes MOE_ERR_NONFINITE.  T = 0 is valid (offsets become all zero).
 * Errors: MOE_ERR_INVALID_ARG (null pointer with T > 0, T < 0), MOE_ERR_CUDA. */
int moe_route(moe_layer* L, const float* logits, int T, int32_t* topk_ids, float* topk_w, int32_t* counts,
              int32_t* offsets, int32_t* entries, void* stream);

/* Cold dedupe, id remap and gather ("DeepSeek-V4.1-Flash on One GB300 ...",
 * section 1: one small kernel copies just the routed cold experts into their
 * slots; section 3: that copy was 2.60 ms of a 10.49 ms step).
 *  topk_ids      device int32 [T][k].
 *  phys_ids      device int32 [T][k] out: loc of each pick's expert (-1 for an id
 *                outside [0, E), which also sets MOE_ERR_BAD_EXPERT in the status).
 *  cold_list     device int32 [min(n_cold, T*k)] out: distinct cold slots picked,
 *                ascending.
 *  n_cold_picked device int32 [1] out.
 * Every listed slot of the scratch is overwritten with the bytes of its host blob,
 * read zero-copy with 16-byte loads; unlisted slots are left as they were.  With
 * moe_params.zero_copy set and T <= 64 nothing is copied (moe_grouped_ffn reads the
 * cold experts in place) and only the outputs above are produced.
 * phys_ids, cold_list and n_cold_picked are ready in `stream` order.  The byte
 * copy itself runs on the layer's own copy stream, forked from `stream` at this
 * call, so that moe_grouped_ffn can work on the experts in HBM while the link
 * streams the cold ones; it moves every picked blob's gate/up planes (w13 nibbles
 * and scales) first and its down planes second, so that moe_grouped_ffn can run
 * the cold experts' gate/up phase while the down planes stream.
 * moe_grouped_ffn and residency_update on this layer join it, and so does
 * moe_gather_join.  A layer sharing the scratch must not call
 * cold_gather before this layer's copy has been joined into `stream`.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA. */
int cold_gather(moe_layer* L, const int32_t* topk_ids, int T, int32_t* phys_ids, int32_t* cold_list,
                int32_t* n_cold_picked, void* stream);

/* Makes `stream` wait for the layer's work in flight on its copy stream: the cold
 * copy, and a deferred residency move with its map upload (no-op when none).
 * Needed only to read the scratch slots, the expert bytes or the placement
 * without calling cold_gather or moe_grouped_ffn. */
int moe_gather_join(moe_layer* L, void* stream);

/* Device workspace bytes moe_grouped_ffn needs for T tokens. */
int moe_ffn_workspace_bytes(const moe_layer* L, int T, size_t* bytes);

/* Grouped SwiGLU expert FFN over all picks ("DeepSeek-V4.1-Flash on One GB300
 * ...", section 1: the layer runs all experts in a single call).  For pick
 * i = t*k + j with expert blob B = blob of physical id phys_ids[i]:
 *   g = W_gate x_t, u = W_up x_t, h = SiLU(g) * u, y_i = W2 h.
 *  x        device bf16 [T][H].
 *  phys_ids device int32 [T][k] (from cold_gather); counts/offsets/entries from
 *           moe_route.
 *  y        device fp32 [T*k][H] out, row i = pick i.
 *  workspace device memory of at least moe_ffn_workspace_bytes(L, T) bytes,
 *           256-byte aligned; its contents are overwritten.
 * Each distinct expert's weights are streamed once per call (with
 * moe_params.zero_copy set and T <= 64, the picked cold experts' straight from their
 * pinned host blobs, on the layer's copy stream, joined into `stream` before the
 * call returns).  Errors:
 * MOE_ERR_INVALID_ARG (null, T < 0, workspace too small), MOE_ERR_CUDA. */
int moe_grouped_ffn(moe_layer* L, const void* x, int T, const int32_t* phys_ids, const int32_t* counts,
                    const int32_t* offsets, const int32_t* entries, float* y, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Arithmetic of calls with more than 64 tokens (prefill-sized buckets).
 *  kind 0 (default): weights expanded exactly from MXFP4 to f16 and multiplied with
 *         f16 activations on tcgen05 kind::f16 tensor cores (buckets above 64
 *         tokens; smaller ones on the decode kernel), fp32 accumulation: the result
 *         of the unquantised layer within rounding.
 *  kind 1 (all-FP4): x and h are converted to MXFP4 as well (each 32-element block
 *         of a row gets the exponent floor(log2(max |v|)) - 2 clamped to
 *         [-127, 127], each element the nearest E2M1 value, ties to the even code,
 *         saturating at 6), and every bucket of the call runs on block-scaled
 *         tcgen05 kind::mxf4 tensor cores with fp32 accumulation ("A 475 GB Model
 *         Across Two Workstations, With the Table on Disk", Abstract: the experts
 *         ship in MXFP4).  The result is the layer with both activations
 *         quantised, which differs from the unquantised layer by the quantisation
 *         of x and h.
 * Calls of at most 64 tokens follow moe_layer_set_decode_kind.
 * moe_ffn_workspace_bytes follows the kinds; set them before sizing the workspace.
 * Errors: MOE_ERR_INVALID_ARG (null, kind not 0 or 1). */
int moe_layer_set_prefill_kind(moe_layer* L, int kind);

/* Arithmetic of calls with at most 64 tokens (decode-sized).
 *  kind 1: the dequant-GEMV kernel (E2M1 weights expanded to f16 in registers, f16
 *         activations, mma.sync).
 *  kind 2: every bucket on block-scaled tcgen05 kind::mxf4 tensor cores, which
 *         decode the MXFP4 weights themselves; each activation (x, then h) is
 *         written as a sum of four MXFP4 terms, the first the activation rounded to
 *         MXFP4 and each further one the remainder of those before, with block
 *         exponents chosen so that no element saturates (each remainder is exact in
 *         fp32), so the result is the unquantised layer's to about 2e-4 relative.
 *  kind 0 (default): kind 2 (on a GB300 the block-scaled kernels are the faster at
 *         every decode size of H = 4096, I = 3072, k = 6, from one token up).
 * Layers that read cold experts in place (moe_params.zero_copy) run kind 1 for
 * calls with cold experts.  Errors: MOE_ERR_INVALID_ARG (null, kind not 0, 1 or 2). */
int moe_layer_set_decode_kind(moe_layer* L, int kind);

/* moe_grouped_ffn for callers that cannot allocate device memory (an engine that
 * has given all free HBM to its own pools and forbids later allocations, code
 * running during a global-mode stream capture, embedders with their own
 * allocator).  No counterpart in the published method: same arguments and results as
 * moe_grouped_ffn minus the workspace, which here is a fixed array of
 * MOE_NOALLOC_SCRATCH_BYTES inside the library's device image (every GPU that
 * loads the library holds one copy until the process exits).  The call
 * allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  All calls on
 * a device share the array and it keeps the previous call's contents (the FFN
 * clears what must start at zero itself), so calls that overlap on the GPU race:
 * order them on one stream or otherwise serialise them.
 * Errors: MOE_ERR_SCRATCH_TOO_SMALL when T needs more than the array holds
 * (moe_ffn_workspace_bytes(L, T) > MOE_NOALLOC_SCRATCH_BYTES; each of the T*k picks
 * takes 2*max(H, I) + 4*I + 4 bytes, each section rounded up to 256 bytes, so
 * T <= 68 at H=4096, I=3072, k=6), MOE_ERR_INVALID_ARG, MOE_ERR_CUDA. */
#define MOE_NOALLOC_SCRATCH_BYTES (8u << 20)
int moe_grouped_ffn_noalloc(moe_layer* L, const void* x, int T, const int32_t* phys_ids, const int32_t* counts,
                            const int32_t* offsets, const int32_t* entries, float* y, void* stream);

/* Combine ("DeepSeek-V4.1-Flash on One GB300 ...", section 4: contributions are
 * summed; the order only moves the last decimal places).  out[t] = sum over
 * j = 0..k-1, in that order, of topk_w[t][j] * y[t*k+j], in fp32.
 *  y device fp32 [T*k][H]; topk_w device fp32 [T][k];
 *  out device [T][H]: bf16 (round to nearest even) when out_fp32 = 0, else fp32.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA. */
int moe_combine(const float* y, const float* topk_w, int T, int k, int H, void* out, int out_fp32, void* stream);

/* Adaptive residency ("DeepSeek-V4.1-Flash on One GB300 ...", section 1: between
 * steps a manager swaps often-picked experts into the hot set and quiet ones out;
 * section 3: hysteresis 3.0 as the published default).  Call once per step, after
 * the layer's moe_grouped_ffn (and moe_combine) on the same stream.  Every
 * swap_every-th call closes a window of pick counts; the plan pairs cold experts
 * picked at least once (count desc, id asc) with hot experts (count asc, id asc)
 * and swaps pair i while count(cold) > hysteresis * count(hot) (at most
 * max_swaps, stopping at the first pair that fails); applying a pair moves the
 * bytes (host_mirror 0: exchanges the two experts' bytes in place between the
 * HBM slot and the host blob; host_mirror 1: copies the promoted expert into the
 * HBM slot, see moe_params) and rewrites the placement map.  Each expert is in at
 * most one pair, so any prefix of a plan is a valid placement.
 *  Deferred mode (default, moe_layer_set_residency_defer 1): the closing call
 *  enqueues a copy of the window's counters to the host and starts the next
 *  window in a second counter buffer, without synchronising; the layer's next
 *  call (one step later) makes the plan from those counts and the current
 *  placement.  The plan's n pairs land in plan order, paced over the calls
 *  before the next window closes: pair i at the plan's call floor(i * span / n)
 *  (call 0 being the one that made it, span = max(1, swap_every - 1)); pairs
 *  still unapplied when the next plan is made land first.  Each landing moves
 *  its bytes on the layer's copy stream, after the work already on `stream`,
 *  while later layers run; the layer's next cold_gather or moe_grouped_ffn waits
 *  for the move.  The promoted expert is read from its host blob (host copy),
 *  never from the shared scratch.  The counts and plans are those of the
 *  synchronous mode; only the times at which the pairs land differ.
 *  Synchronous mode (0): the closing call synchronises `stream`, reads the
 *  counters, and moves the bytes on `stream` at once; with host copies it
 *  promotes from the scratch slot while that slot still holds this layer's copy.
 *  Layers sharing a scratch must make this call before a later layer's
 *  cold_gather on the same stream order (it may read a slot).
 *  n_swaps_out host int32 [1] out: the swaps applied by this call (deferred: by
 *  the plan of the previous closing call).
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA, MOE_ERR_INJECTED (test hook: on a
 * closing call, before anything is enqueued or applied). */
int residency_update(moe_layer* L, int32_t* n_swaps_out, void* stream);

/* Selects the residency mode of residency_update: 1 deferred (default), 0
 * synchronous.  A plan already pending is applied at the next call either way.
 * Errors: MOE_ERR_INVALID_ARG (null, defer not 0 or 1). */
int moe_layer_set_residency_defer(moe_layer* L, int defer);

/* The plan one acting residency_update applies, computed on the host with no
 * device work (callable without a GPU): the same ranking, pairing and stopping
 * rule, from a window's pick counts and a placement.
 *  counts    host int32 [E], each >= 0.
 *  loc       host int32 [E]: a placement (a permutation of 0..E-1; values below
 *            n_hot are HBM slots).
 *  loc_out   host int32 [E] out: the placement after the swaps (may equal loc).
 *  promoted, demoted  host int32 [max_swaps] out (may be NULL when max_swaps is
 *            0): pair i moved promoted[i] into demoted[i]'s HBM slot and
 *            demoted[i] into promoted[i]'s cold slot.
 *  1 <= E <= 1024, 0 <= n_hot <= E, 0 <= max_swaps <= 64, hysteresis finite >= 0.
 * Returns the number of swaps (>= 0), or MOE_ERR_INVALID_ARG (bad sizes, a
 * negative count, or loc not a permutation). */
int moe_residency_plan(const int32_t* counts, const int32_t* loc, int E, int n_hot, int max_swaps, float hysteresis,
                       int32_t* loc_out, int32_t* promoted, int32_t* demoted);

/* MXFP4 quantisation of bf16 activation rows, the first step of the all-FP4
 * prefill mode (a block-scaled FP4 x FP4 tensor-core product takes both operands
 * in MXFP4).  Each 32-element block of a row gets the shared exponent
 * floor(log2(max |v|)) - 2 clamped to [-127, 127] (an all-zero block: -127),
 * stored as scale byte exponent + 127; each element gets |v| / 2^exponent rounded
 * to the nearest E2M1 magnitude {0, 0.5, 1, 1.5, 2, 3, 4, 6}, ties to the even
 * code, above 6 saturating to 6, with v's sign bit (the OCP Microscaling
 * conversion for E2M1).  Output in the weights' row layout.
 *  x_bf16  device bf16 [rows][K], finite values; K a positive multiple of 32.
 *  nib     device uint8 [rows][K/2] out: element k of a row in byte k/2, low
 *          nibble when k is even.
 *  scales  device uint8 [rows][K/32] out.
 * rows = 0 is valid.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA. */
int moe_quant_mxfp4(const void* x_bf16, int rows, int K, uint8_t* nib, uint8_t* scales, void* stream);

/* Copies the placement map to host int32 [E] (synchronous). */
int moe_layer_get_loc(moe_layer* L, int32_t* loc_host);

/* Copies the window pick counters to host int32 [E] (synchronous). */
int moe_layer_get_counts(moe_layer* L, int32_t* counts_host);

/* Reads the layer's device status word (synchronous); 0 = no error so far. */
int moe_get_status(moe_layer* L, int* status);

/* Clears the device status word and the diagnostic record (synchronous). */
int moe_clear_status(moe_layer* L);

/* Copies the diagnostic record of the first device-side wait that ran out of
 * time (set together with MOE_ERR_TIMEOUT) to host int32 [16]: [0] 1 when set,
 * [1] block, [2] warp, [3] wait kind (1 stage full, 2 stage empty), [4] ring slot,
 * [5] parity waited for, [6] stage index, [7] task << 8 | token columns,
 * [8] 1 if the other parity had completed.  All zero when nothing timed out. */
int moe_get_diag(moe_layer* L, int32_t* diag_host);

/* Text for a status code. */
const char* moe_strerror(int code);

/* Number of CTAs the cold copy kernel runs on (0 = the default, 3/16 of the SMs:
 * enough to keep the host link busy on GB300).  A zero-copy layer's cold FFN chain
 * runs on the same number of CTAs, or a quarter of the SMs if that is more.
 * The copy shares the GPU with the FFN over HBM-resident experts. */
int moe_layer_set_copy_ctas(moe_layer* L, int ctas);

/* Timing: after moe_layer_profile(L, n) (which first waits for the device to go
 * idle) the next n cold_gather calls record CUDA events around their byte copy on
 * the layer's copy stream, and the next n moe_grouped_ffn calls record events
 * around their kernels on the caller's stream; n = 0 stops and frees them.
 * moe_layer_profile_read waits for the copy records and writes up to `max`
 * durations in ms to host float copy_ms[] and their number to *n_out.
 * moe_layer_profile_read_ffn does the same for the FFN calls: each duration is the
 * call's kernel time without the waits for the cold copy (the work before the join
 * of the cold gate/up planes, between that join and the join of the rest, and
 * after it).  0 <= n <= 2^20, else MOE_ERR_INVALID_ARG. */
int moe_layer_profile(moe_layer* L, int max_records);
int moe_layer_profile_read(moe_layer* L, float* copy_ms, int max, int* n_out);
int moe_layer_profile_read_ffn(moe_layer* L, float* ffn_ms, int max, int* n_out);

/* Test hook for host-side fault injection: what = 1 makes the next acting
 * residency_update fail with MOE_ERR_INJECTED before any copy or map change (as a
 * failed host copy would); what = 0 clears it.  Never set in normal use. */
int moe_layer_inject_fault(moe_layer* L, int what);

/* Host-link probe: copies `bytes` (a multiple of 16) from mapped pinned host
 * memory `src_host` to device memory `dst_dev` with the same zero-copy 16-byte
 * load loop as cold_gather, on `ctas` CTAs (0 = one per SM).  Used to measure
 * the link peak the cold gather is reported against. */
int moe_link_probe(const void* src_host, void* dst_dev, size_t bytes, int ctas, void* stream);

/* Dense block-scaled FP4 tensor-core rate probe (the denominator the all-FP4
 * prefill path is reported against): `ctas` CTAs (0 = one per SM) each issue
 * `iters` back-to-back tcgen05 kind::mxf4 MMAs of M = 128, N = 256, K = 64
 * (2 * 128 * 256 * 64 flops each) on operands resident in shared memory; the
 * caller times the launch on `stream`.  status_dev: device int, set to
 * MOE_ERR_TIMEOUT if the kernel's bounded wait for its MMAs ran out (zero it
 * first).  1 <= iters <= 2^20.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA. */
int moe_mxf4_peak_probe(int iters, int ctas, int* status_dev, void* stream);

/* Test hook for the bounded device waits of the pipelined kernels: launches one
 * thread that waits on an mbarrier phase that nothing completes.  The wait gives
 * up at its deadline (2 s), writes its record to diag_dev (device int32 [16], the
 * layout moe_get_diag describes; zero it first) and MOE_ERR_TIMEOUT to
 * *status_dev (device int; the first error written wins, so zero it first), and
 * the kernel returns, leaving the context usable: how a lost producer is reported
 * without faulting or hanging the GPU. */
int moe_debug_wait_timeout(int* status_dev, int32_t* diag_dev, void* stream);

/* Lane-layout check of the E2M1 pair conversion used by the FFN kernels: writes
 * for every byte b (0..255) the two f16 values it decodes to (low nibble first)
 * as uint32 [256] to out_dev (device). */
int moe_debug_e2m1_pairs(uint32_t* out_dev, void* stream);

/* Test hook: both E2M1 roundings of n fp32 values |v| < 8 (already divided by their
 * block scale).  out_dev uint32 [2n]: out[2i] from the hardware pair conversion the
 * block-scaled kernels use (round to nearest, ties to the even code, saturating at
 * 6), out[2i + 1] from the comparison rule of the stand-alone quantiser; both with
 * the sign in bit 3.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_CUDA. */
int moe_debug_e2m1_round(const float* v_dev, int n, uint32_t* out_dev, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOEHOST_H */
