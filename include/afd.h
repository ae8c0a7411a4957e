/*
 * afd.h -- C ABI of the GB300 (sm_103a) library for the FFN side of
 * Attention-FFN Disaggregation (AFD): fan-in of per-peer slots, softmax top-k
 * router, stable per-expert token permutation, grouped SwiGLU experts on the
 * tensor cores (plus an optional shared expert), top-k weighted combine, and
 * the split back into per-peer return slots.
 *
 * Sources (page title, section):
 *  - "[RFC]: Async GPU Connector" (vllm-project/afd-plugin #233):
 *    "Window and slot layout", "Capacity and ring depth", "Data flow",
 *    "Attention gate and FFN expert compute", "FFN main loop",
 *    "Risks and alternatives".
 *  - "Data on the wire: tensors per layer and stage": steps 1-4 and
 *    "What can go wrong".
 *  - "[RFC]: Async AFD for Prefill on Ascend NPU": "Architecture",
 *    "Asynchronous work-item contract", "Risks".
 *
 * One process, one GPU.  The attention peers are regions of a device
 * "window" owned by the library (two windows: the FFN inbox that peers pack
 * into, and the return inbox the FFN step writes).  All pointers passed in
 * are plain device pointers unless a comment says host; no call allocates
 * device memory except afd_create / afd_set_layer.
 *
 * Conventions
 *  - Every call returns an int status: AFD_OK (0) or an AFD_ERR_* code.
 *  - Calls that launch work are asynchronous and ordered on the context's
 *    stream.  Errors that only the device can see (header checks, bounded
 *    waits) are recorded in a device status word; afd_poll_status reads it.
 *    After a device error, later steps on the same context do no work until
 *    the status is polled (sticky first error).
 *  - Activation element type: AFD_DTYPE_BF16 or AFD_DTYPE_F32.  Weights use
 *    the activation type; the router weight and bias are fp32.
 */
#ifndef AFD_H
#define AFD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define AFD_OK 0
#define AFD_ERR_ARG 1          /* invalid argument (range, duplicate peer, NULL) */
#define AFD_ERR_SHAPE 2        /* token counts disagree (header vs seq_lens,
                                  Data on the wire, "What can go wrong") */
#define AFD_ERR_CAPACITY 3     /* over token_cap / max_total_tokens: raise,
                                  never truncate (Async GPU Connector,
                                  "Capacity and ring depth") */
#define AFD_ERR_HEADER 4       /* magic / version / length self-check failed */
#define AFD_ERR_SEQ 5          /* header seq or echo_seq mismatch (Async GPU
                                  Connector, "Risks and alternatives") */
#define AFD_ERR_LAYER 6        /* header layer != requested layer, or no
                                  weights registered for it */
#define AFD_ERR_STAGE 7        /* header stage != requested stage */
#define AFD_ERR_TIMEOUT 8      /* a bounded device wait gave up */
#define AFD_ERR_SHUTDOWN 9     /* the peer set the shutdown bit */
#define AFD_ERR_SPLIT_UNEVEN 10 /* even-split fallback does not divide */
#define AFD_ERR_NOT_DEVICE 11  /* a host pointer where device memory is required
                                  (Data on the wire: CPU tensors are rejected) */
#define AFD_ERR_CUDA 12        /* a CUDA runtime/driver call failed */
#define AFD_ERR_UNSUPPORTED 13 /* configuration outside what the kernels cover */
#define AFD_ERR_CANARY 14      /* a guard word after a slot field was overwritten */
#define AFD_ERR_BOUNDS 15      /* debug build: an index a kernel derived was out of range */

#define AFD_DTYPE_F32 0
#define AFD_DTYPE_BF16 1

/* GEMM engine of the expert projections.  TENSOR (default for bf16) is the
 * tcgen05/TMEM grouped GEMM on SM pairs (cta_group::2, 256 weight rows per
 * unit); TENSOR_1CTA the same GEMM with one SM per 128-row tile; SIMT a
 * plain fp32-FMA CUDA kernel that serves fp32 activations and cross-checks
 * the tensor-core engines. */
#define AFD_GEMM_TENSOR 0
#define AFD_GEMM_SIMT 1
#define AFD_GEMM_TENSOR_1CTA 2

#define AFD_MAX_PEERS 64
#define AFD_MAX_RING 64    /* most stages in flight per peer (ring_depth) */

/* ---- configuration -------------------------------------------------------
 * num_peers        attention peers = window regions (with one FFN rank the
 *                  region count max(attn, ffn) is the peer count)
 * ring_depth       slots per peer, one per stage in flight (1 without
 *                  micro-batching; Async GPU Connector, "Capacity and ring
 *                  depth": an invariant, not a knob); 1..AFD_MAX_RING
 * token_cap        max tokens per slot (max_num_batched_tokens)
 * max_total_tokens max fan-in total per forward; 0 = num_peers * token_cap
 * hidden, num_experts, topk, inter (routed SwiGLU intermediate),
 * shared_inter     shared SwiGLU intermediate, 0 = no shared expert
 * act_dtype        AFD_DTYPE_*; renorm: top-k weights renormalised to sum 1
 * routed_scaling   routed_scaling_factor applied to the gate weights
 * routed_cap_multiplier  sizes the routed rows of a rank's slot under
 *                  token-level dispatch (>= 1; see ffn_size)
 * wait_timeout_ns  bound on every device-side wait (flag polls); 0 = 1 s
 * gemm             AFD_GEMM_*; max_layers: size of the layer weight table
 * flags            AFD_CFG_* bits, 0 for the defaults
 * ffn_rank, ffn_size  0 (default): this context routes itself (token form)
 *                  or receives grouped rows of at most token_cap per slot.
 *                  ffn_size >= 1: the context is FFN rank ffn_rank of
 *                  ffn_size (<= AFD_MAX_FFN_RANKS) receiving token-level
 *                  dispatch (Async GPU Connector, "Data flow" and "Capacity
 *                  and ring depth"): num_experts is the rank's own expert
 *                  count (afd_expert_range), only the grouped calls apply,
 *                  a peer's shared rows are its tokens ffn_rank, ffn_rank +
 *                  ffn_size, ... and a slot holds
 *                  routed_cap = ceil(ceil(token_cap * topk / ffn_size)
 *                  * routed_cap_multiplier) routed rows (AFD_ERR_CAPACITY
 *                  above it, never truncation).
 */
#define AFD_MAX_FFN_RANKS 16
/* Launch every kernel after the previous one has fully finished, instead of
 * letting its CTAs be scheduled (and wait on the device) while the previous
 * kernel drains (programmatic dependent launch, the default). */
#define AFD_CFG_NO_PDL 1
/* Guard words after the flag array and after every slot field, filled with
 * a position-dependent pattern when the windows are created and checked by
 * afd_check_canaries: a write past the end of a field changes them.  Each
 * guard is one alignment unit (afd_layout.align bytes), so every field
 * stays aligned; the offsets afd_slot_layout gives include the guards.  A
 * substitute for a memory checker, for tests. */
#define AFD_CFG_CANARY 2
/* With the SM-pair engine the SwiGLU and down projections run as one
 * persistent launch: a pair that has no SwiGLU unit left starts down units
 * whose token tile's h rows are all stored (per-tile counters in the
 * workspace), so the down weights stream while the last SwiGLU units finish
 * and no launch boundary separates the two.  This flag launches them as two
 * kernels instead (the stage times then split them). */
#define AFD_CFG_SPLIT_GEMMS 4
typedef struct afd_config {
  int32_t num_peers;
  int32_t ring_depth;
  int32_t token_cap;
  int32_t max_total_tokens;
  int32_t hidden;
  int32_t num_experts;
  int32_t topk;
  int32_t inter;
  int32_t shared_inter;
  int32_t act_dtype;
  int32_t renorm;
  int32_t max_layers;
  int32_t gemm;
  int32_t flags;
  float routed_scaling;
  float routed_cap_multiplier;
  int64_t wait_timeout_ns;
  int32_t ffn_rank;
  int32_t ffn_size;
} afd_config;

/* Byte offsets of the slot fields and window sizes.  Async GPU Connector,
 * "Window and slot layout":
 *   window = [ flag[num_regions * ring_depth] | slot(0,0) | slot(0,1) | ... ]
 *   slot   = [ header | route_table | routed_x | shared_idx | shared_x ]
 * Every field is aligned to align = lcm(256, hidden * element size), so each
 * field is 256-byte aligned and every activation row is a whole row of the
 * window viewed as a [rows, hidden] matrix.  Sizes: header (12 + E) int32;
 * route_table [token_cap, topk] int32; routed_x and shared_x
 * [token_cap, hidden]; shared_idx [token_cap] int32; the shared fields are
 * empty without a shared expert.  Under token-level dispatch (ffn_size >= 1)
 * routed_x holds max(token_cap, routed_cap) rows and route_table
 * max(token_cap * topk, routed_cap) int32 (the sender's partial index
 * t * topk + j of each routed row).  Flags are uint64 sequence numbers; slot
 * (peer p, stage s) is slot number p * ring_depth + s, as is its flag. */
typedef struct afd_layout {
  int64_t header, route_table, routed_x, shared_idx, shared_x;
  int64_t slot_bytes, flags_bytes, window_bytes, align;
  /* AFD_CFG_CANARY: bytes of each guard (align), else 0.  A field's guard is
   * the `guard` bytes before the next field's offset (before slot_bytes for
   * the slot's last field); the flag array's, the `guard` bytes before
   * flags_bytes. */
  int64_t guard;
} afd_layout;

/* Header words (int32), Async GPU Connector, "Window and slot layout": a
 * fixed 12 words then expert_counts[num_experts]; the page names the fields
 * but not their order, which is this library's:
 *   0 magic (bytes 'A','F','D','G'), 1 version (1), 2 flags (bit 1, value
 *   2, = shutdown), 3 seq (low 32 bits of the flag), 4 echo_seq, 5 layer,
 *   6 stage, 7 num_tokens, 8 routed_tokens, 9 shared_tokens, 10 num_experts,
 *   11 header length in words (12 + num_experts).
 * Dispatch: routed_x = the peer's tokens in order, routed_tokens = 0 (no
 * partials routed by the sender: the FFN routes), shared_tokens = 0 or
 * num_tokens with shared_idx = 0..n-1 and shared_x = the same rows.
 * Return: routed_x = output rows, route_table = chosen expert ids [n, topk],
 * routed_tokens = n * topk, expert_counts = this peer's per-expert partial
 * counts, seq = echo_seq = the dispatch seq; the return flag = that seq. */
#define AFD_HEADER_FIXED_WORDS 12
#define AFD_HEADER_MAGIC 0x47444641
#define AFD_HEADER_VERSION 1
#define AFD_FLAG_SHUTDOWN 2

#define AFD_DIR_DISPATCH 0  /* FFN inbox: peers pack into it */
#define AFD_DIR_RETURN 1    /* return inbox: the FFN step writes it */

/* workspace buffers exposed for inspection (afd_get_workspace) */
#define AFD_WS_IDS 0        /* int32 [T, topk] chosen expert ids */
#define AFD_WS_WEIGHTS 1    /* fp32 [T, topk] gate weights */
#define AFD_WS_COUNTS 2     /* int32 [E] partials per expert */
#define AFD_WS_OFFSETS 3    /* int32 [E + 1] exclusive prefix of counts */
#define AFD_WS_PERM 4       /* int32 [T*topk] position -> flattened index t*k+j */
#define AFD_WS_INV 5        /* int32 [T*topk] flattened index -> position */
#define AFD_WS_XP 6         /* act [T*topk, hidden] permuted routed rows (shared rows stay in the slots) */
#define AFD_WS_H 7          /* act [T*topk, inter] routed SwiGLU output */
#define AFD_WS_Y 8          /* routed down projection [T*topk, hidden]: token form with bf16
                               activations 24-bit (u16 high plane, then the u8 low plane; value =
                               bits (hi << 16 | lo << 8) as fp32), fp32 activations fp32;
                               grouped form: act */
#define AFD_WS_HS 9         /* act [T, shared_inter] shared SwiGLU output */
#define AFD_WS_S 10         /* fp32 [T, hidden] shared expert output */
#define AFD_WS_STATUS 11    /* int32 device status word */

typedef struct afd_ctx afd_ctx;

typedef struct afd_stats {
  int64_t window_bytes;      /* one window */
  int64_t workspace_bytes;
  int32_t last_total_tokens; /* T of the last forward */
  int32_t num_sms;
  int64_t forwards;
} afd_stats;

/* Create a context on the current CUDA device: validates cfg, allocates the
 * two windows (zeroed: every flag 0), the workspace sized for
 * max_total_tokens, and the layer table.  cuda_stream is a cudaStream_t (NULL
 * = the legacy default stream).  *out is owned by the caller; release it
 * with afd_destroy.  Errors: AFD_ERR_ARG / AFD_ERR_UNSUPPORTED for bad cfg,
 * AFD_ERR_CUDA when a device call fails (e.g. no GPU). */
int afd_create(const afd_config* cfg, void* cuda_stream, afd_ctx** out);

/* Synchronise the context's stream and free everything it owns. NULL is a
 * no-op. */
void afd_destroy(afd_ctx* ctx);

/* Change the stream later calls are ordered on. */
int afd_set_stream(afd_ctx* ctx, void* cuda_stream);

/* Host only (no GPU needed): the slot layout for cfg. */
int afd_slot_layout(const afd_config* cfg, afd_layout* out);

/* Host only.  Data on the wire, step 4 and "What can go wrong": split
 * `total` tokens over n_peers by the recorded lengths (seq_lens, host array
 * of n_lens ints) in peer order; when n_lens != n_peers the split is even
 * and AFD_ERR_SPLIT_UNEVEN is returned if it does not divide.  Lengths that
 * do not sum to total give AFD_ERR_SHAPE.  sizes: host array [n_peers]. */
int afd_split_sizes(int total, int n_peers, const int* seq_lens, int n_lens, int* sizes);

/* Register the weights of one layer (layer-select table, Async AFD for
 * Prefill on Ascend NPU, "Architecture": an address table for every layer).
 *   Wg   fp32 [hidden, E] row-major (router); NULL on an FFN rank under
 *        token-level dispatch (ffn_size >= 1), which never routes
 *   bias fp32 [E] or NULL (added to the logits)
 *   W13  act [E, 2*inter, hidden]: rows 0..inter-1 gate, inter..2*inter-1 up
 *   Wd   act [E, hidden, inter]
 *   W13_s act [2*shared_inter, hidden], Wd_s act [hidden, shared_inter]
 *        (both NULL when shared_inter == 0)
 * All device pointers, caller-owned, 16-byte aligned.  The library keeps an
 * fp32 copy of Wg rearranged as [ceil(E / 4)][hidden][4 experts] and, for
 * the tensor engines (cfg.gemm != AFD_GEMM_SIMT), copies of W13, Wd, W13_s
 * and Wd_s re-laid as [E][128-row tiles][64-column k-blocks] blocks of
 * 128 x 64 (16 contiguous KB, the unit one TMA load reads; zero past the
 * weight's edges; within a W13 tile, 16 gate rows then the 16 matching up
 * rows, four times).  The call returns once the copies are complete, so
 * with a tensor engine the caller's expert weights may then be freed;
 * with AFD_GEMM_SIMT they are read in place and must stay valid while the
 * layer is used (Wg need not: it is copied in both cases).  Registering a
 * layer again replaces its copies in place, ordered after the forwards
 * already enqueued.  Errors: AFD_ERR_ARG, AFD_ERR_NOT_DEVICE, AFD_ERR_CUDA. */
int afd_set_layer(afd_ctx* ctx, int layer, const float* Wg, const float* bias,
                  const void* W13, const void* Wd, const void* W13_s, const void* Wd_s);

/* The attention side's send, simulated (Async GPU Connector, "Window and
 * slot layout" and "Data flow"): copy x (device, act [n_tokens, hidden],
 * row-major) into slot (peer, stage) of the dispatch window -- routed_x, and
 * shared_idx/shared_x when with_shared -- then write the header (layer,
 * stage, num_tokens, seq) and, after the payload, the flag = seq.  seq must
 * exceed the previous seq packed into that slot (monotonic, host-checked:
 * AFD_ERR_SEQ).  n_tokens may be 0 (x may then be NULL).  Errors:
 * AFD_ERR_ARG, AFD_ERR_CAPACITY (n_tokens > token_cap), AFD_ERR_NOT_DEVICE,
 * AFD_ERR_SEQ. */
int afd_pack_slot(afd_ctx* ctx, int peer, int stage, int layer, const void* x, int n_tokens,
                  int with_shared, uint64_t seq);

/* Publish an empty slot whose header carries the shutdown bit (Async GPU
 * Connector, "FFN main loop": announce_shutdown); a forward that reads it
 * records AFD_ERR_SHUTDOWN. */
int afd_announce_shutdown(afd_ctx* ctx, int peer, int stage, uint64_t seq);

/* The FFN step over one fan-in (the timed hot path).  seq_lens and slots
 * are host arrays of n_peers ints: slots[i] is the peer whose slot (peer,
 * stage) is the i-th part of the concatenation and seq_lens[i] its token
 * count (Data on the wire, steps 2-4).  On the device, in stream order:
 *   a0 bounded wait for each listed flag to pass the last value consumed,
 *      then header checks (magic, version, length, seq/echo, shutdown,
 *      layer, stage, num_tokens == seq_lens[i], shared fields);
 *   a1 router over the virtual concatenation (fp32 logits, top-k with
 *      lowest-index ties, softmax gate weights);
 *   a2/a3 per-expert counts and offsets, stable permutation, gather of the
 *      rows straight from the peer slots;
 *   a4-a6 grouped SwiGLU GEMMs for the routed experts and the shared expert;
 *   a7 weighted combine, split into each peer's return slot (routed_x,
 *      route_table, header), then each return flag = the dispatch seq.
 * Host-checked errors (returned): AFD_ERR_ARG (peer range/duplicates, stage
 * range, n_peers), AFD_ERR_CAPACITY, AFD_ERR_LAYER (no weights).  Device
 * errors (afd_poll_status): AFD_ERR_TIMEOUT, AFD_ERR_HEADER, AFD_ERR_SEQ,
 * AFD_ERR_SHUTDOWN, AFD_ERR_LAYER, AFD_ERR_STAGE, AFD_ERR_SHAPE. */
int afd_ffn_forward(afd_ctx* ctx, int layer, int stage, const int* seq_lens, const int* slots,
                    int n_peers);

/* The attention side's receive, simulated (Data on the wire, step 4: each
 * peer receives its slice): bounded wait until the return flag of (peer,
 * stage) equals expect_seq, check magic / version / echo_seq / num_tokens
 * == n_tokens, then copy the n_tokens output rows into out (device, act
 * [n_tokens, hidden]).  Device errors: AFD_ERR_TIMEOUT, AFD_ERR_SEQ (flag
 * past expect_seq or echo mismatch), AFD_ERR_HEADER, AFD_ERR_SHAPE. */
int afd_unpack_split(afd_ctx* ctx, int peer, int stage, void* out, int n_tokens,
                     uint64_t expect_seq);

/* afd_pack_slot for n peers of one stage in one call: peers[i] (distinct),
 * x[i] (host array of device pointers, 16-byte aligned; NULL for 0 tokens),
 * n_tokens[i] and seq[i] (host arrays), with_shared for all.  Two launches
 * whatever n: every payload, then every header with its flag released after
 * that peer's payload.  Every argument is checked before anything is
 * launched; the errors are afd_pack_slot's.  A process that hosts several
 * attention peers (or the peers' emulation) packs a step in one call. */
int afd_pack_slots(afd_ctx* ctx, int n, const int32_t* peers, int stage, int layer,
                   const void* const* x, const int32_t* n_tokens, int with_shared,
                   const uint64_t* seq);

/* afd_unpack_split for n peers of one stage in one call (host arrays of
 * peers, device output pointers, token counts and expected seqs); one
 * launch, each peer's rows copied after its own flag and header check.
 * Errors as afd_unpack_split. */
int afd_unpack_splits(afd_ctx* ctx, int n, const int32_t* peers, int stage, void* const* out,
                      const int32_t* n_tokens, const uint64_t* expect_seq);

/* ---- grouped form: the Attention side routes ------------------------------
 * [RFC]: Async GPU Connector, "Data flow" steps 1-4 and "Attention gate and
 * FFN expert compute": the Attention side computes the gate, sorts the
 * flattened top-k ids stably and sends each FFN rank its routed rows grouped
 * by expert, with the rows per expert (group_list) in the header; the FFN
 * must not route again and runs every row through its expert with a unit
 * weight (a top-1 problem), the shared rows through the shared expert as
 * their own batch; the gate weights never travel, and the Attention side
 * weights and combines what comes back.
 *
 * afd_pack_grouped -- the Attention side's send of this form, simulated:
 *   rows        device act [n_rows, hidden], grouped by expert (ascending e)
 *   group_list  host int32 [num_experts], rows per expert, summing to n_rows
 *   x           device act [n_tokens, hidden], the peer's tokens: the shared
 *               rows (shared_idx = 0..n_tokens-1) when with_shared
 * Writes routed_x, shared rows, then the header (routed_tokens = n_rows,
 * num_tokens = n_tokens, expert_counts = group_list) and the flag = seq.
 * Errors: AFD_ERR_ARG, AFD_ERR_CAPACITY (n_rows or n_tokens > token_cap),
 * AFD_ERR_SHAPE (group_list does not sum to n_rows), AFD_ERR_SEQ,
 * AFD_ERR_NOT_DEVICE. */
int afd_pack_grouped(afd_ctx* ctx, int peer, int stage, int layer, const void* rows, int n_rows,
                     const int* group_list, const void* x, int n_tokens, int with_shared,
                     uint64_t seq);

/* afd_ffn_forward_grouped -- the FFN-side step of the grouped form over the
 * listed slots: n_rows[i] / seq_lens[i] (host) are the routed rows and the
 * tokens of list entry i.  Header checks as afd_ffn_forward plus
 * routed_tokens == n_rows[i] and the group list summing to it; the rows of
 * all entries grouped by expert (entry order within an expert); the routed
 * and shared SwiGLU GEMMs; then each entry's return slot gets routed_x = the
 * expert output of each of its rows in arrival order, shared_x = its shared
 * outputs, the header (routed_tokens, shared_tokens and expert_counts as
 * received) and the flag = the dispatch seq.  Capacity: n_rows[i] <=
 * token_cap, sum n_rows <= max_total_tokens * topk.  Errors as
 * afd_ffn_forward. */
int afd_ffn_forward_grouped(afd_ctx* ctx, int layer, int stage, const int* n_rows,
                            const int* seq_lens, const int* slots, int n_peers);

/* afd_unpack_grouped -- the Attention side's receive of the grouped form,
 * simulated: bounded wait for the return flag == expect_seq, header checks
 * (num_tokens == n_tokens, routed_tokens == n_rows), then the n_rows expert
 * outputs into y_out (device act [n_rows, hidden]) and, when s_out is not
 * NULL, the n_tokens shared outputs into s_out.  Errors as afd_unpack_split. */
int afd_unpack_grouped(afd_ctx* ctx, int peer, int stage, void* y_out, int n_rows, void* s_out,
                       int n_tokens, uint64_t expect_seq);
/* (On an FFN rank among several, s_out receives the peer's round-robin
 * share of shared outputs, tokens ffn_rank, ffn_rank + ffn_size, ...; n_rows
 * may be up to routed_cap.) */

/* ---- device-resident work-item loop ---------------------------------------
 * [RFC]: Async AFD for Prefill on Ascend NPU, "Asynchronous work-item
 * contract" and "FFN execution modes"; [RFC]: Async GPU Connector, "FFN main
 * loop" and the device-side wait_any named under "Risks and alternatives".
 * A work item is one stage of the ring over the listed peers (one Attention
 * replica).  It is ready once every listed peer has published a flag newer
 * than the one last consumed from its (peer, stage) slot.  Each step of the
 * loop, on the device and in stream order:
 *   - waits (bounded by wait_timeout_ns) for any ready stage; the scan
 *     starts after the stage served last, so a ready stage waits for at most
 *     ring_depth - 1 others;
 *   - takes the layer (header word layer_idx, which must agree across the
 *     listed peers) and the token / routed-row counts from the headers;
 *   - runs the same FFN step as afd_ffn_forward (form AFD_FORM_TOKENS) or
 *     afd_ffn_forward_grouped (AFD_FORM_GROUPED) with that layer's weights,
 *     which come from a device copy of the table afd_set_layer fills.
 * The host reads nothing back to drive a step, and every launch has a fixed
 * shape: the most tokens a step may carry (min(max_total_tokens, n_peers *
 * token_cap); grouped rows: min(max_total_tokens * topk, n_peers *
 * token_cap)), with the kernels bounded by the counts on the device.
 * Device errors (afd_poll_status) as afd_ffn_forward, plus AFD_ERR_TIMEOUT
 * when no stage gets ready, AFD_ERR_LAYER for a layer outside the table or
 * without weights, AFD_ERR_CAPACITY for a step over the shape above.  The
 * first error ends the loop: later steps do no work until it is polled. */
#define AFD_FORM_TOKENS 0
#define AFD_FORM_GROUPED 1

/* Enqueue n_items steps of the loop over the peers slots[0..n_peers-1]
 * (host ints) on the context's stream (eager mode).  Host-checked errors:
 * AFD_ERR_ARG (form, peer range or duplicates, n_peers, n_items < 0). */
int afd_ffn_serve(afd_ctx* ctx, const int* slots, int n_peers, int n_items, int form);

/* The same n_items steps captured once into a CUDA graph (graph mode: the
 * loop runs a fixed number of items and is replayed without host
 * orchestration).  Captured on a stream of the library's own; *kernels (may
 * be NULL) receives the kernel launches the graph holds.  The graph refers to
 * the context's window, workspace and layer table, not to the weights: a
 * later afd_set_layer takes effect in the next replay.  Errors: as
 * afd_ffn_serve, n_items == 0 is AFD_ERR_ARG, AFD_ERR_CUDA if the capture or
 * the instantiation fails. */
typedef struct afd_serve_graph afd_serve_graph;
int afd_serve_graph_create(afd_ctx* ctx, const int* slots, int n_peers, int n_items, int form,
                           afd_serve_graph** out, int64_t* kernels);
/* Replay on the context's current stream. */
int afd_serve_graph_launch(afd_serve_graph* g);
void afd_serve_graph_destroy(afd_serve_graph* g);

/* Synchronise the stream and copy out the loop's record of the items it
 * served, oldest first: records (host int32 [max_records][4]) gets (stage,
 * layer, tokens, routed rows) of the last min(max_records, served, 64)
 * items and *n_records how many that is; *n_served (may be NULL) the items
 * served since creation.  Errors: AFD_ERR_ARG, AFD_ERR_CUDA. */
int afd_serve_log(afd_ctx* ctx, int32_t* records, int max_records, int* n_records,
                  int64_t* n_served);

/* Synchronise the stream, return the first device-recorded error since the
 * last poll (AFD_OK if none) and clear it; AFD_ERR_CUDA if the stream itself
 * failed. */
int afd_poll_status(afd_ctx* ctx);

/* The context's configuration (host copy). */
int afd_get_config(afd_ctx* ctx, afd_config* out);

/* ---- token-level dispatch to several FFN ranks ------------------------------
 * [RFC]: Async GPU Connector, "Data flow" steps 1-4 and "Capacity and ring
 * depth".  The experts are split over ffn_size FFN ranks, each an afd_ctx
 * created with ffn_rank / ffn_size and num_experts = its own count; an
 * Attention peer sends every rank the routed rows of its experts (grouped
 * by local expert, with the group list in the header) and its round-robin
 * share of the shared rows, and combines what the ranks return.  On one GPU
 * every rank's window is local memory.
 *
 * afd_expert_range -- experts of rank ffn_rank among ffn_size for
 * num_experts experts in all: a contiguous block, the first
 * num_experts % ffn_size ranks one expert more (the pages fix no placement;
 * balanced contiguous blocks are this library's reading).  AFD_ERR_ARG for
 * ffn_size < 1, num_experts < ffn_size or a rank out of range. */
int afd_expert_range(int num_experts, int ffn_size, int ffn_rank, int* first, int* count);

/* afd_attn_create -- one Attention peer's side over the FFN ranks
 * ranks[0..ffn_size-1] (ranks[r] must be rank r, all with the same peers,
 * stages, token_cap, hidden, topk, activation type, shared expert and
 * routed_cap_multiplier, and num_experts = afd_expert_range's count of
 * num_experts in all, at most 256).  Allocates its per-stage plan buffers
 * (2 * token_cap * topk int32 per stage).  Work is ordered on cuda_stream;
 * it must be ordered before the ranks' steps that consume it (the same
 * stream, or events).  Errors: AFD_ERR_ARG, AFD_ERR_CUDA. */
typedef struct afd_attn afd_attn;
int afd_attn_create(afd_ctx* const* ranks, int ffn_size, int peer, int num_experts,
                    void* cuda_stream, afd_attn** out);
void afd_attn_destroy(afd_attn* a);

/* afd_attn_dispatch -- the peer's send of one stage (steps 1-3):
 *   x          device act [n_tokens, hidden], 16-byte aligned
 *   topk_ids   device int32 [n_tokens, topk], expert ids 0..num_experts-1
 * On the device: a stable sort of the flattened ids (one pass gives the
 * segments by rank and the local-expert groups within them), then every
 * rank's slot (peer, stage) gets routed_x = the rows x[f / topk] of its
 * segment, route_table = their partial indices f, shared rows = tokens
 * ffn_rank, ffn_rank + ffn_size, ... (shared_idx = those indices) when
 * with_shared, the header (num_tokens, routed_tokens, shared_tokens,
 * num_experts = the rank's count, expert_counts = its group list) and the
 * flag = seq.  Every rank gets its message, empty ones included.  A segment
 * over routed_cap is a device error AFD_ERR_CAPACITY (nothing is written to
 * any rank); an id out of range AFD_ERR_ARG (afd_attn_poll_status).  Host
 * errors: AFD_ERR_ARG, AFD_ERR_CAPACITY (n_tokens > token_cap),
 * AFD_ERR_NOT_DEVICE. */
int afd_attn_dispatch(afd_attn* a, int stage, int layer, const void* x, int n_tokens,
                      const int32_t* topk_ids, int with_shared, uint64_t seq);

/* afd_attn_combine -- the peer's receive of that stage (step 4): a bounded
 * wait for the return flag == expect_seq of every rank that got rows (a
 * rank sent no rows is not waited for), header checks (magic, version, echoed
 * seq, num_tokens, routed and shared rows as sent), then out[t] = sum over
 * j ascending of topk_weights[t, j] * (rank output of partial t * topk + j)
 * + (shared output of token t, from rank t mod ffn_size), in fp32, rounded
 * once to the activation type.
 *   topk_weights  device fp32 [n_tokens, topk]   out  device act [n_tokens, hidden]
 * n_tokens must be that of the stage's last dispatch (else AFD_ERR_SHAPE).
 * Device errors: AFD_ERR_TIMEOUT, AFD_ERR_SEQ, AFD_ERR_HEADER, AFD_ERR_SHAPE. */
int afd_attn_combine(afd_attn* a, int stage, const float* topk_weights, void* out, int n_tokens,
                     uint64_t expect_seq);

/* Synchronise the peer's stream and copy out the routed rows its last
 * dispatch of the stage sent to each rank (host int [ffn_size]). */
int afd_attn_rows(afd_attn* a, int stage, int* rows);
/* Synchronise the peer's stream; return and clear its first device error. */
int afd_attn_poll_status(afd_attn* a);
/* Kernel launches issued by this peer's calls. */
int64_t afd_attn_launch_count(afd_attn* a);

/* Device base pointer and size of a window (AFD_DIR_*). */
int afd_get_window(afd_ctx* ctx, int direction, void** dev_ptr, int64_t* bytes);

/* Device pointer and capacity in bytes of a workspace buffer (AFD_WS_*);
 * contents describe the last forward. */
int afd_get_workspace(afd_ctx* ctx, int which, void** dev_ptr, int64_t* bytes);

int afd_get_stats(afd_ctx* ctx, afd_stats* out);

/* Synchronise the stream and copy the per-expert counts of the last step
 * that ran (token form: routed partials per expert; grouped form: received
 * rows per expert) into counts (host int32 [n]); the first min(n,
 * num_experts) experts are copied and *n_experts (may be NULL) receives
 * num_experts.  These are the counts the return headers carry per peer
 * (Async GPU Connector, "Window and slot layout": expert_counts travel in
 * band), summed over the step's peers.  Zeros before the first step.
 * Errors: AFD_ERR_ARG, AFD_ERR_CUDA. */
int afd_last_expert_counts(afd_ctx* ctx, int32_t* counts, int n, int* n_experts);

/* Kernel launches the library issued on this context since creation. */
int64_t afd_launch_count(afd_ctx* ctx);

/* Synchronise the stream and check every guard word of both windows of a
 * context created with AFD_CFG_CANARY.  AFD_OK when all are intact, else
 * AFD_ERR_CANARY with *window (AFD_DIR_*) and *offset (byte offset within
 * that window of the first changed word; both may be NULL).  AFD_ERR_ARG for
 * a context without guards, AFD_ERR_CUDA if the check itself fails. */
int afd_check_canaries(afd_ctx* ctx, int* window, int64_t* offset);

/* Bounds checks of the debug build.  The library compiled with
 * -DAFD_DEBUG_BOUNDS (combine_peer_slot_gb300/build.py, debug=True:
 * libafd_gb300_dbg.so) checks, before each use, the indices its kernels take
 * from arrays that earlier kernels of the step wrote: the partial positions
 * the gather and the combine read through inv / perm (and the grouped form's
 * row positions), and every output row range of the grouped GEMMs' units
 * (AFD_DBG_* sites below).  A failed check skips the access (a position is
 * replaced by 0), sets the step's status to AFD_ERR_BOUNDS and records the
 * first failure: site, index and the bound it broke.  The release build
 * compiles the checks out.  (Expert ids and the slot header's counts and
 * shared indices are checked in both builds.)
 * afd_debug_bounds synchronises the stream and returns AFD_OK when nothing
 * failed since the context was created or last planted, else AFD_ERR_BOUNDS
 * with *site, *index and *limit (each may be NULL).  afd_debug_plant clears
 * the record and makes every later check at `site` fail (its bound is taken
 * as 0, so the valid access is skipped; no index out of range is ever
 * used), site 0 none: a test of the reporting path.  Both return
 * AFD_ERR_UNSUPPORTED in the release build, AFD_ERR_ARG / AFD_ERR_CUDA on
 * failure. */
#define AFD_DBG_GATHER_INV 1     /* k_rank_gather (token order): inv[t, j] < T * k */
#define AFD_DBG_GATHER_PERM 2    /* k_gather, position order: perm[r] < T * k */
#define AFD_DBG_GATHER_GROUPED 3 /* k_gather, grouped form: row position < routed rows */
#define AFD_DBG_COMBINE_INV 4    /* k_combine: inv[t, j] < T * k */
#define AFD_DBG_SCATTER_INV 5    /* k_scatter_grouped: inv[r] < routed rows */
#define AFD_DBG_GEMM_OUT 6       /* grouped GEMMs: a unit's last output row < output rows */
#define AFD_DBG_NUM_SITES 7
int afd_debug_bounds(afd_ctx* ctx, int32_t* site, int64_t* index, int64_t* limit);
int afd_debug_plant(afd_ctx* ctx, int32_t site);

/* Stage timing.  With enable != 0, every afd_ffn_forward records a CUDA
 * event on the context's stream before and after each stage:
 *   0 header check, 1 router, 2 plan, 3 gather, 4 SwiGLU GEMM (routed +
 *   shared), 5 down GEMM (routed + shared), 6 combine + split, 7 return
 *   headers and flags.
 * The events of up to 64 forwards are kept; a forward that would overwrite
 * unread ones first waits for the oldest and folds it into a running sum.
 * afd_stage_times waits for every recorded forward, writes the summed
 * elapsed milliseconds of the first n (<= AFD_NUM_STAGES) stages over the
 * forwards since the previous call into ms (host array), their number into
 * *forwards (host, may be NULL), and clears the sum.  A forward that fails
 * part-way contributes nothing.  Events cost no device work; timing is off
 * by default. */
#define AFD_NUM_STAGES 8
int afd_profile(afd_ctx* ctx, int enable);
int afd_stage_times(afd_ctx* ctx, float* ms, int n, int64_t* forwards);

/* Router without device allocation.  The pages have no counterpart: this
 * entry point exists for callers that cannot call cudaMalloc -- a serving
 * process whose memory pool already holds the device's free memory, or a
 * plugin that must not cause the device-wide synchronisation an allocation
 * or free can bring.  It computes exactly the router step of
 * afd_ffn_forward (same kernel, same fp32 logit order, same top-k and gate
 * weights) for a plain activation block:
 *   x        device, act [n_tokens, hidden] row-major, 16-byte aligned
 *   Wg       device fp32 [hidden, num_experts]; bias device fp32 [E] or NULL
 *   ids      device int32 [n_tokens, topk] out; weights device fp32
 *            [n_tokens, topk] out
 *   cuda_stream  cudaStream_t the work is ordered on (NULL = legacy stream)
 * Its scratch (the router weight rearranged as [ceil(E / 4)][hidden][4],
 * the router logits and a status word) is a file-scope device array of
 * AFD_NOALLOC_MAX_ROUTER_WEIGHTS + AFD_NOALLOC_MAX_LOGITS + 64 floats
 * (about 5 MiB) that every GPU loading this library holds until exit; the
 * first call on a device looks up that array's device address (once per
 * device, safe from several host threads).  All calls share the array: each
 * call rewrites it and clears the status word first, and calls that overlap
 * on the GPU race on it.
 * 4 * ceil(num_experts / 4) * hidden above
 * AFD_NOALLOC_MAX_ROUTER_WEIGHTS or n_tokens * num_experts above
 * AFD_NOALLOC_MAX_LOGITS returns AFD_ERR_CAPACITY; bad arguments
 * AFD_ERR_ARG; a failing CUDA call AFD_ERR_CUDA.  Asynchronous; allocates
 * nothing.  Device-side failures (a bounded wait inside the router that
 * gives up) cannot be returned by an asynchronous call and nothing polls
 * the status word: instead every ids entry of the call is then -1 and every
 * weight NaN. */
#define AFD_NOALLOC_MAX_ROUTER_WEIGHTS 262144
#define AFD_NOALLOC_MAX_LOGITS 1048576
int afd_route_noalloc(const void* x, int n_tokens, int hidden, int act_dtype, const float* Wg,
                      const float* bias, int num_experts, int topk, int renorm,
                      float routed_scaling, int32_t* ids, float* weights, void* cuda_stream);

/* Static string for a status code. */
const char* afd_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* AFD_H */
