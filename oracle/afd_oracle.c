/*
 * afd_oracle.c -- plain, slow CPU oracle for the FFN side of Attention-FFN
 * Disaggregation (AFD): fan-in of peer slots, softmax top-k router, stable
 * per-expert permutation, routed + shared SwiGLU experts, top-k weighted
 * combine and the per-peer split back into return slots; and the grouped
 * form, where the Attention side has routed and the FFN runs each received
 * row through its expert (top-1, unit weight).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file.  Only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library: every rule below is restated here from the pages.
 *
 * Sources (page title, section):
 *  [RFC-GPU]  "[RFC]: Async GPU Connector" (vllm-project/afd-plugin #233):
 *             "Window and slot layout", "Capacity and ring depth",
 *             "Data flow", "Attention gate and FFN expert compute",
 *             "Risks and alternatives".
 *  [WIRE]     "Data on the wire: tensors per layer and stage":
 *             Steps 2-4 and "What can go wrong".
 *  [NPU]      "[RFC]: Async AFD for Prefill on Ascend NPU": "Architecture".
 *
 * Arithmetic: fp64 accumulation everywhere except the router logits, whose
 * fp32 reduction order is fixed (see orc_router_logits) so that expert ids
 * are reproducible bit for bit.  Compile with -ffp-contract=off so that no
 * multiply-add is fused behind the code's back.
 *
 * Parity status of each function is stated at the function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ORC_PLANT selects one deliberately wrong variant of the oracle, used only
 * by the test that shows the pins catch plausible mistakes (0 = correct):
 *  1 gate and up swapped        2 shared branch dropped
 *  3 ties to the higher index   4 sign of the SiLU exponent flipped
 *  5 gate weights paired with the wrong j   6 unstable bucket order
 *  7 rows read from the wrong peer's slot    8 logits as one sequential chain */
#ifndef ORC_PLANT
#define ORC_PLANT 0
#endif

/* ------------------------------------------------------------------------ */
/* status codes (the library's error codes, restated)                        */
/* ------------------------------------------------------------------------ */
enum {
  ORC_OK = 0,
  ORC_ERR_ARG = 1,
  ORC_ERR_SHAPE = 2,
  ORC_ERR_CAPACITY = 3,
  ORC_ERR_HEADER = 4,
  ORC_ERR_SEQ = 5,
  ORC_ERR_LAYER = 6,
  ORC_ERR_STAGE = 7,
  ORC_ERR_TIMEOUT = 8,
  ORC_ERR_SHUTDOWN = 9,
  ORC_ERR_SPLIT_UNEVEN = 10
};

/* Header words.  [RFC-GPU] "Window and slot layout": a fixed 12 int32 words
 * followed by expert_counts[expert_per_rank]; magic "AFDG", a version, and
 * bit 1 of the flags word is the shutdown sentinel.  The page names the
 * fields but not their positions; the order below is this implementation's reading. */
enum {
  H_MAGIC = 0, H_VERSION, H_FLAGS, H_SEQ, H_ECHO_SEQ, H_LAYER, H_STAGE,
  H_NUM_TOKENS, H_ROUTED_TOKENS, H_SHARED_TOKENS, H_NUM_EXPERTS, H_LEN,
  H_FIXED_WORDS
};
/* the four bytes 'A','F','D','G' read as a little-endian 32-bit word */
static const uint32_t ORC_MAGIC = (uint32_t)'A' | ((uint32_t)'F' << 8) |
                                  ((uint32_t)'D' << 16) | ((uint32_t)'G' << 24);
static const int32_t ORC_VERSION = 1;
static const int32_t ORC_FLAG_SHUTDOWN = 1 << 1;

/* ------------------------------------------------------------------------ */
/* bf16 <-> binary64                                                          */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of a binary32; widening is exact.  Pinned against
 * torch's dtype conversion in the tests. */
double orc_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a binary64 value once, to nearest with ties to even, onto the bf16
 * grid (8 significant bits, binary32 exponent range, gradual underflow).
 * Written from the definition of the format: scale by the quantum of the
 * binade, round to an integer with rint (default mode: ties to even), scale
 * back.  Pinned against torch's float32 -> bfloat16 conversion and against
 * hand-derived double-rounding cases in the tests. */
uint16_t orc_f64_to_bf16(double v) {
  uint32_t u;
  float f;
  if (isnan(v)) return 0x7FC0;
  if (v == 0.0 || isinf(v)) {
    f = (float)v;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
  }
  int e = ilogb(v);              /* |v| in [2^e, 2^(e+1)) */
  if (e < -126) e = -126;        /* subnormal binade: fixed quantum 2^-133 */
  double quantum = ldexp(1.0, e - 7);
  double r = rint(v / quantum) * quantum;
  /* largest finite bf16 is (2 - 2^-7) * 2^127 */
  if (fabs(r) > ldexp(255.0, 120)) r = copysign(INFINITY, v);
  f = (float)r;                  /* exact: r has <= 8 significant bits */
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------ */
/* window and slot layout                                                     */
/* ------------------------------------------------------------------------ */

typedef struct orc_layout {
  int64_t header, route_table, routed_x, shared_idx, shared_x; /* offsets in slot */
  int64_t slot_bytes;      /* stride between consecutive slots */
  int64_t flags_bytes;     /* size of the flag area at the start of the window */
  int64_t window_bytes;    /* flags + num_regions * ring_depth slots */
  int64_t align;           /* alignment unit every field is padded to */
} orc_layout;

static int64_t orc_gcd(int64_t a, int64_t b) {
  while (b) { int64_t t = a % b; a = b; b = t; }
  return a;
}
static int64_t orc_round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

/* [RFC-GPU] "Window and slot layout":
 *   window = [ flag[num_regions * ring_depth] | slot(0,0) | slot(0,1) | ... ]
 *   slot   = [ header | route_table | routed_x | shared_idx | shared_x ]
 * with every field 256-byte aligned; one layout serves both directions.
 * This implementation also aligns every field to the activation row pitch (hidden *
 * element size), so the unit is lcm(256, row pitch): any payload row is then
 * a whole row of the window read as a [rows, hidden] matrix.  Field sizes:
 * header (12 + E) int32, route_table [token_cap, topk] int32, routed_x and
 * shared_x [token_cap, hidden] activations, shared_idx [token_cap] int32; the
 * two shared fields are empty when the layer has no shared expert.  Flags are
 * 64-bit sequence numbers.  Slot (region r, ring s) is slot number
 * r * ring_depth + s.  Parity: pinned by the disjoint / in-bounds / aligned
 * checks the page lists under "Existing verification". */
/* Slot of an FFN rank among several ([RFC-GPU] "Capacity and ring depth":
 * the routed fields hold routed_cap partial rows, the token fields
 * token_cap tokens): routed_x holds max(token_cap, routed_cap) rows and
 * route_table max(token_cap * topk, routed_cap) int32 (a token's k chosen
 * ids in the return direction of the token form; the sender's partial
 * index of each routed row in the dispatch direction of the multi-rank
 * form).  routed_cap = 0: one FFN rank, the plain layout above. */
int orc_slot_layout_ranks(int num_regions, int ring_depth, int token_cap, int topk,
                          int hidden, int act_bytes, int num_experts, int has_shared,
                          int64_t routed_cap, orc_layout* L) {
  if (num_regions <= 0 || ring_depth <= 0 || token_cap <= 0 || topk <= 0 ||
      hidden <= 0 || (act_bytes != 2 && act_bytes != 4) || num_experts <= 0 || routed_cap < 0)
    return ORC_ERR_ARG;
  int64_t row = (int64_t)hidden * act_bytes;
  int64_t a = 256 / orc_gcd(256, row) * row;
  int64_t rows = routed_cap > token_cap ? routed_cap : token_cap;
  int64_t table = (int64_t)token_cap * topk;
  if (routed_cap > table) table = routed_cap;
  int64_t off = 0;
  L->align = a;
  L->header = off;
  off += orc_round_up((int64_t)(H_FIXED_WORDS + num_experts) * 4, a);
  L->route_table = off;
  off += orc_round_up(table * 4, a);
  L->routed_x = off;
  off += orc_round_up(rows * row, a);
  L->shared_idx = off;
  if (has_shared) off += orc_round_up((int64_t)token_cap * 4, a);
  L->shared_x = off;
  if (has_shared) off += orc_round_up((int64_t)token_cap * row, a);
  L->slot_bytes = off;
  L->flags_bytes = orc_round_up((int64_t)num_regions * ring_depth * 8, a);
  L->window_bytes = L->flags_bytes + (int64_t)num_regions * ring_depth * off;
  return ORC_OK;
}

int orc_slot_layout(int num_regions, int ring_depth, int token_cap, int topk,
                    int hidden, int act_bytes, int num_experts, int has_shared,
                    orc_layout* L) {
  return orc_slot_layout_ranks(num_regions, ring_depth, token_cap, topk, hidden, act_bytes,
                               num_experts, has_shared, 0, L);
}

/* ------------------------------------------------------------------------ */
/* several FFN ranks ([RFC-GPU] "Capacity and ring depth", "Data flow")       */
/* ------------------------------------------------------------------------ */

/* Experts of FFN rank r among F: a contiguous block; the pages fix no
 * placement, and this implementation reads it as the balanced linear one -- the
 * first E mod F ranks hold one expert more than the others. */
void orc_expert_range(int E, int F, int r, int* first, int* count) {
  int base = E / F, rem = E % F;
  *count = base + (r < rem ? 1 : 0);
  *first = r * base + (r < rem ? r : rem);
}

/* routed_cap = ceil(max_num_batched_tokens * topk / ffn_size) *
 * routed_cap_multiplier, read as ceil(ceil(token_cap * topk / F) * mult). */
int64_t orc_routed_cap(int token_cap, int topk, int F, double multiplier) {
  int64_t even = ((int64_t)token_cap * topk + F - 1) / F;
  return (int64_t)ceil((double)even * multiplier);
}

/* Shared rows of FFN rank r: tokens arange(r, n, F) ([RFC-GPU] "Data flow"
 * step 3), i.e. how many of r, r + F, r + 2F, ... are below n. */
int orc_rr_rows(int n, int r, int F) { return n > r ? (n - r + F - 1) / F : 0; }

static uint8_t* orc_slot(uint8_t* win, const orc_layout* L, int region, int ring,
                         int ring_depth) {
  return win + L->flags_bytes + ((int64_t)region * ring_depth + ring) * L->slot_bytes;
}
static uint64_t* orc_flag(uint8_t* win, int region, int ring, int ring_depth) {
  return (uint64_t*)win + (int64_t)region * ring_depth + ring;
}

/* ------------------------------------------------------------------------ */
/* pack / unpack (the Attention side, simulated)                              */
/* ------------------------------------------------------------------------ */

/* Write one dispatch slot: payload (routed_x = the peer's tokens in order;
 * with a shared expert, shared_idx = 0..n-1 and shared_x = the same rows,
 * since with one FFN rank every token is a shared token -- [RFC-GPU]
 * "Data flow" step 3, arange(ffn_rank, num_tokens, ffn_size)), then the
 * header, then the flag = seq ([RFC-GPU] "Window and slot layout": the flag
 * is the sender's monotonically increasing seq and is written after the
 * payload).  The dispatch route_table is left untouched: routing happens on
 * the FFN side in this implementation.  Parity: pinned by the round-trip test. */
int orc_pack_slot(uint8_t* win, const orc_layout* L, int ring_depth, int region,
                  int stage, int layer, const void* x, int n_tokens, int hidden,
                  int act_bytes, int token_cap, int num_experts, int with_shared,
                  int has_shared, uint64_t seq, int shutdown) {
  if (n_tokens < 0 || n_tokens > token_cap) return ORC_ERR_CAPACITY;
  if (with_shared && !has_shared) return ORC_ERR_ARG;
  uint8_t* s = orc_slot(win, L, region, stage, ring_depth);
  int64_t row = (int64_t)hidden * act_bytes;
  if (n_tokens) memcpy(s + L->routed_x, x, (size_t)(n_tokens * row));
  if (with_shared) {
    int32_t* sidx = (int32_t*)(s + L->shared_idx);
    for (int i = 0; i < n_tokens; i++) sidx[i] = i;
    if (n_tokens) memcpy(s + L->shared_x, x, (size_t)(n_tokens * row));
  }
  int32_t* h = (int32_t*)(s + L->header);
  memset(h, 0, (size_t)(H_FIXED_WORDS + num_experts) * 4);
  h[H_MAGIC] = (int32_t)ORC_MAGIC;
  h[H_VERSION] = ORC_VERSION;
  h[H_FLAGS] = shutdown ? ORC_FLAG_SHUTDOWN : 0;
  h[H_SEQ] = (int32_t)(uint32_t)seq;
  h[H_ECHO_SEQ] = (int32_t)(uint32_t)seq;
  h[H_LAYER] = layer;
  h[H_STAGE] = stage;
  h[H_NUM_TOKENS] = n_tokens;
  h[H_ROUTED_TOKENS] = 0;   /* no pre-routed partials: the FFN routes */
  h[H_SHARED_TOKENS] = with_shared ? n_tokens : 0;
  h[H_NUM_EXPERTS] = num_experts;
  h[H_LEN] = H_FIXED_WORDS + num_experts;
  *orc_flag(win, region, stage, ring_depth) = seq;
  return ORC_OK;
}

/* Read one return slot back ([WIRE] step 4: each peer receives its slice).
 * The flag must equal expect_seq (lower: not yet written, i.e. a wait that
 * never ends; higher: a stale request), the header must carry the magic and
 * echo the sequence number ([RFC-GPU] "Risks and alternatives": the echo_seq
 * check), and the token count must match.  Parity: round-trip test. */
int orc_unpack_split(uint8_t* win, const orc_layout* L, int ring_depth, int region,
                     int stage, void* out, int n_tokens, int hidden, int act_bytes,
                     int num_experts, uint64_t expect_seq) {
  uint64_t f = *orc_flag(win, region, stage, ring_depth);
  if (f < expect_seq) return ORC_ERR_TIMEOUT;
  if (f > expect_seq) return ORC_ERR_SEQ;
  uint8_t* s = orc_slot(win, L, region, stage, ring_depth);
  const int32_t* h = (const int32_t*)(s + L->header);
  if ((uint32_t)h[H_MAGIC] != ORC_MAGIC || h[H_VERSION] != ORC_VERSION ||
      h[H_NUM_EXPERTS] != num_experts || h[H_LEN] != H_FIXED_WORDS + num_experts)
    return ORC_ERR_HEADER;
  if ((uint32_t)h[H_ECHO_SEQ] != (uint32_t)expect_seq) return ORC_ERR_SEQ;
  if (h[H_NUM_TOKENS] != n_tokens) return ORC_ERR_SHAPE;
  if (n_tokens) memcpy(out, s + L->routed_x, (size_t)n_tokens * hidden * act_bytes);
  return ORC_OK;
}

/* [WIRE] step 4 and "What can go wrong": split sizes follow the recorded
 * per-peer lengths in peer order; when they do not cover every peer the
 * split is even, and an uneven division raises.  Pinned by hand-derived
 * fixtures. */
int orc_split_sizes(int total, int n_peers, const int* seq_lens, int n_lens,
                    int* sizes) {
  if (n_peers <= 0 || total < 0) return ORC_ERR_ARG;
  if (n_lens == n_peers) {
    int64_t s = 0;
    for (int i = 0; i < n_peers; i++) {
      if (seq_lens[i] < 0) return ORC_ERR_ARG;
      s += seq_lens[i];
      sizes[i] = seq_lens[i];
    }
    return s == total ? ORC_OK : ORC_ERR_SHAPE;
  }
  if (total % n_peers) return ORC_ERR_SPLIT_UNEVEN;
  for (int i = 0; i < n_peers; i++) sizes[i] = total / n_peers;
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* router                                                                     */
/* ------------------------------------------------------------------------ */

/* Router logits for one token, l_e = sum_h x_h * Wg[h, e] (+ b_e), in fp32
 * in this implementation's canonical reduction order (the pages fix none):
 *   partial_l = fp32 fused multiply-add chain over h = l, l+32, l+64, ...
 *               ascending, starting from +0 (l = 0..31);
 *   then a butterfly: for off = 16, 8, 4, 2, 1: v_l <- v_l + v_(l xor off);
 *   the result (equal for every l) plus b_e in fp32.
 * Wg is [hidden, E] row-major fp32; x is the token row widened exactly to
 * fp32.  Parity: pinned against an fp64 recomputation within the fp32 error
 * bound, and through the ids against a full sort of the fp64 logits. */
static void orc_router_logits(const float* x, int hidden, const float* Wg,
                              const float* bias, int E, float* logits) {
  float part[32], nxt[32];
  for (int e = 0; e < E; e++) {
    for (int l = 0; l < 32; l++) {
      float acc = 0.0f;
      for (int h = l; h < hidden; h += 32) acc = fmaf(x[h], Wg[(int64_t)h * E + e], acc);
      part[l] = acc;
    }
    for (int off = 16; off >= 1; off >>= 1) {
      for (int l = 0; l < 32; l++) nxt[l] = part[l] + part[l ^ off];
      memcpy(part, nxt, sizeof part);
    }
#if ORC_PLANT == 8
    part[0] = 0.0f;
    for (int h = 0; h < hidden; h++) part[0] = fmaf(x[h], Wg[(int64_t)h * E + e], part[0]);
#endif
    logits[e] = bias ? part[0] + bias[e] : part[0];
  }
}

/* Selection key of a logit: a NaN ranks below every number (as -inf). */
static float rank_key(float v) { return isnan(v) ? -INFINITY : v; }

/* Top-k on the logits with ties broken toward the lower expert index, then
 * gate weights from a softmax over all E experts ([RFC-GPU] "Attention gate
 * and FFN expert compute": softmax router; the k chosen experts carry their
 * probabilities, optionally renormalised to sum 1, times
 * routed_scaling_factor).  The softmax runs in fp64 from the fp32 logits and
 * is rounded once to fp32.  gap = (k-th chosen) - (best unchosen) of the
 * fp64 logits, so a near-tie is visible.  Parity: pinned by brute force. */
static void orc_router_token(const float* x, int hidden, const float* Wg,
                             const float* bias, int E, int k, int renorm,
                             float scale, int* ids, float* w, double* gap,
                             float* logits_out) {
  float* lg = (float*)malloc(sizeof(float) * E);
  char* taken = (char*)calloc(E, 1);
  orc_router_logits(x, hidden, Wg, bias, E, lg);
  for (int j = 0; j < k; j++) {
    int best = -1;
    for (int e = 0; e < E; e++)
#if ORC_PLANT == 3
      if (!taken[e] && (best < 0 || rank_key(lg[e]) >= rank_key(lg[best]))) best = e;
#else
      if (!taken[e] && (best < 0 || rank_key(lg[e]) > rank_key(lg[best]))) best = e;
#endif
    taken[best] = 1;
    ids[j] = best;
  }
  double mx = lg[0];
  for (int e = 1; e < E; e++) if (lg[e] > mx) mx = lg[e];
  double den = 0.0;
  for (int e = 0; e < E; e++) den += exp((double)lg[e] - mx);
  double* p = (double*)malloc(sizeof(double) * k);
  double psum = 0.0;
  for (int j = 0; j < k; j++) {
    p[j] = exp((double)lg[ids[j]] - mx) / den;
    psum += p[j];
  }
  for (int j = 0; j < k; j++) {
    double v = renorm ? p[j] / psum : p[j];
    w[j] = (float)(v * (double)scale);
  }
  if (gap) {
    /* fp64 logits, summed in index order */
    double kth = 0.0, best_out = -INFINITY;
    for (int e = 0; e < E; e++) {
      double s = 0.0;
      for (int h = 0; h < hidden; h++) s += (double)x[h] * (double)Wg[(int64_t)h * E + e];
      if (bias) s += bias[e];
      if (e == ids[k - 1]) kth = s;
      if (!taken[e] && s > best_out) best_out = s;
    }
    *gap = (k < E) ? kth - best_out : INFINITY;
  }
  if (logits_out) memcpy(logits_out, lg, sizeof(float) * E);
  free(p);
  free(lg);
  free(taken);
}

/* Route a [T, hidden] activation matrix (act_bytes 2 = bf16, 4 = fp32).
 * logits may be NULL. */
void orc_route(const void* x, int act_bytes, int T, int hidden, const float* Wg,
               const float* bias, int E, int k, int renorm, float scale, int* ids,
               float* w, double* gap, float* logits, int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
#endif
  for (int t = 0; t < T; t++) {
    float* xr = (float*)malloc(sizeof(float) * hidden);
    for (int h = 0; h < hidden; h++)
      xr[h] = act_bytes == 2 ? (float)orc_bf16_to_f64(((const uint16_t*)x)[(int64_t)t * hidden + h])
                             : ((const float*)x)[(int64_t)t * hidden + h];
    orc_router_token(xr, hidden, Wg, bias, E, k, renorm, scale, ids + (int64_t)t * k,
                     w + (int64_t)t * k, gap ? gap + t : NULL,
                     logits ? logits + (int64_t)t * E : NULL);
    free(xr);
  }
}

/* ------------------------------------------------------------------------ */
/* dispatch plan                                                              */
/* ------------------------------------------------------------------------ */

/* [RFC-GPU] "Data flow" step 1: flatten topk_ids (index f = t*k + j), sort
 * stably by expert id (argsort(stable=True)); bincount gives the per-expert
 * counts (the group list) and their exclusive prefix sum the segment
 * offsets.  Written as a counting sort: a stable sort by key.
 *   counts[e]   = #{f : ids[f] = e}
 *   offsets[e]  = sum_{e' < e} counts[e'], offsets[E] = T*k
 *   perm[pos]   = f, the f-th partial's position pos = inv[f]
 * Parity: pinned against numpy's stable argsort and bincount. */
int orc_plan(const int* ids, int n, int E, int* counts, int* offsets, int* perm,
             int* inv) {
  for (int e = 0; e < E; e++) counts[e] = 0;
  for (int f = 0; f < n; f++) {
    if (ids[f] < 0 || ids[f] >= E) return ORC_ERR_ARG;
    counts[ids[f]]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; e++) offsets[e + 1] = offsets[e] + counts[e];
  int* cur = (int*)malloc(sizeof(int) * (E > 0 ? E : 1));
  for (int e = 0; e < E; e++) cur[e] = offsets[e];
#if ORC_PLANT == 6
  for (int f = n - 1; f >= 0; f--) {
#else
  for (int f = 0; f < n; f++) {
#endif
    int pos = cur[ids[f]]++;
    perm[pos] = f;
    inv[f] = pos;
  }
  free(cur);
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* experts and combine                                                        */
/* ------------------------------------------------------------------------ */

static double orc_ld(const void* p, int act_bytes, int64_t i) {
  return act_bytes == 2 ? orc_bf16_to_f64(((const uint16_t*)p)[i]) : (double)((const float*)p)[i];
}
/* round a value to the activation type and widen it back */
static double orc_round_act(double v, int act_bytes) {
  return act_bytes == 2 ? orc_bf16_to_f64(orc_f64_to_bf16(v)) : (double)(float)v;
}

/* One SwiGLU expert applied to one row, accumulating alpha * y into acc:
 *   g_i = sum_h x_h W13[i, h],  u_i = sum_h x_h W13[I + i, h]     (fp64)
 *   h_i = act(silu(g_i) * u_i),  silu(g) = g / (1 + e^-g)
 *   y_f = sum_i h_i Wd[f, i]                                      (fp64)
 * W13 is [2I, hidden] (rows 0..I-1 gate, I..2I-1 up), Wd is [hidden, I],
 * both row-major in the activation type.  h is rounded to the activation
 * type because it is the operand of the down projection.  [RFC-GPU]
 * "Attention gate and FFN expert compute" (fused_experts: gate/up GEMM,
 * SiLU-and-multiply, down GEMM); [NPU] "Architecture" (W1 with SwiGLU, then
 * W2).  Parity: pinned by the dense-SwiGLU (E = 1, k = 1) and dense-mixture
 * identities against numpy matmuls.  h_out (optional) receives h. */
static void orc_swiglu_row(const double* x, int hidden, int inter, const void* W13,
                           const void* Wd, int act_bytes, double alpha, double* acc,
                           double* h_out) {
  double* h = (double*)malloc(sizeof(double) * inter);
  for (int i = 0; i < inter; i++) {
    double g = 0.0, u = 0.0;
    int64_t rg = (int64_t)i * hidden, ru = (int64_t)(inter + i) * hidden;
    for (int c = 0; c < hidden; c++) {
      g += x[c] * orc_ld(W13, act_bytes, rg + c);
      u += x[c] * orc_ld(W13, act_bytes, ru + c);
    }
#if ORC_PLANT == 1
    { double tmp = g; g = u; u = tmp; }
#endif
#if ORC_PLANT == 4
    double silu = g / (1.0 + exp(g));
#else
    double silu = g / (1.0 + exp(-g));
#endif
    h[i] = orc_round_act(silu * u, act_bytes);
    if (h_out) h_out[i] = h[i];
  }
  for (int f = 0; f < hidden; f++) {
    double y = 0.0;
    int64_t r = (int64_t)f * inter;
    for (int i = 0; i < inter; i++) y += h[i] * orc_ld(Wd, act_bytes, r + i);
    acc[f] += alpha * y;
  }
  free(h);
}

typedef struct orc_weights {
  const float* Wg;     /* [hidden, E] fp32 */
  const float* bias;   /* [E] fp32 or NULL */
  const void* W13;     /* [E, 2I, hidden] act */
  const void* Wd;      /* [E, hidden, I] act */
  const void* W13s;    /* [2Is, hidden] act or NULL */
  const void* Wds;     /* [hidden, Is] act or NULL */
} orc_weights;

/* Combine for one token ([RFC-GPU] "Data flow", combine_scatter: a weighted
 * sum of the token's top-k expert outputs, plus the shared branch by
 * shared_idx):  out = sum_{j ascending} w_j * y_j + s, in fp64, rounded once
 * to the activation type.  x_routed and x_shared are the token's rows from
 * routed_x and shared_x.  h_out, if given, receives the k routed h rows
 * ([k, I], in j order). */
static void orc_token_forward(const double* x_routed, const double* x_shared, int hidden,
                              int E, int k, int inter, int shared_inter,
                              const orc_weights* W, int act_bytes, const int* ids,
                              const float* w, double* out, double* h_out) {
  (void)E;
  for (int f = 0; f < hidden; f++) out[f] = 0.0;
  int64_t e13 = (int64_t)2 * inter * hidden, ed = (int64_t)hidden * inter;
  for (int j = 0; j < k; j++) {
    int e = ids[j];
    const char* w13 = (const char*)W->W13 + (int64_t)e * e13 * act_bytes;
    const char* wd = (const char*)W->Wd + (int64_t)e * ed * act_bytes;
#if ORC_PLANT == 5
    double wj = (double)w[k - 1 - j];
#else
    double wj = (double)w[j];
#endif
    orc_swiglu_row(x_routed, hidden, inter, w13, wd, act_bytes, wj, out,
                   h_out ? h_out + (int64_t)j * inter : NULL);
  }
#if ORC_PLANT != 2
  if (x_shared && shared_inter > 0 && W->W13s)
    orc_swiglu_row(x_shared, hidden, shared_inter, W->W13s, W->Wds, act_bytes, 1.0, out,
                   NULL);
#endif
}

/* Dense-mixture form used by the pins: apply the token rows to every expert
 * e with weight wdense[t, e] (zero for unselected experts) plus the shared
 * expert; out is fp64 [T, hidden], no rounding of the sum. */
void orc_dense_mixture(const void* x, int act_bytes, int T, int hidden, int E,
                       int inter, int shared_inter, const orc_weights* W,
                       const double* wdense, double* out) {
  double* xr = (double*)malloc(sizeof(double) * hidden);
  int64_t e13 = (int64_t)2 * inter * hidden, ed = (int64_t)hidden * inter;
  for (int t = 0; t < T; t++) {
    for (int c = 0; c < hidden; c++) xr[c] = orc_ld(x, act_bytes, (int64_t)t * hidden + c);
    double* o = out + (int64_t)t * hidden;
    for (int f = 0; f < hidden; f++) o[f] = 0.0;
    for (int e = 0; e < E; e++) {
      double a = wdense[(int64_t)t * E + e];
      if (a == 0.0) continue;
      orc_swiglu_row(xr, hidden, inter, (const char*)W->W13 + (int64_t)e * e13 * act_bytes,
                     (const char*)W->Wd + (int64_t)e * ed * act_bytes, act_bytes, a, o, NULL);
    }
    if (shared_inter > 0 && W->W13s)
      orc_swiglu_row(xr, hidden, shared_inter, W->W13s, W->Wds, act_bytes, 1.0, o, NULL);
  }
  free(xr);
}

/* ------------------------------------------------------------------------ */
/* the FFN-side forward over slots                                            */
/* ------------------------------------------------------------------------ */

typedef struct orc_cfg {
  int num_regions, ring_depth, token_cap, hidden, act_bytes, num_experts, topk;
  int inter, shared_inter, renorm, max_total_tokens;
  float routed_scaling;
  /* this FFN rank among ffn_size (num_experts is then the rank's own count;
   * ffn_size 0 or 1: one rank); routed_cap > 0: the rank receives token-level
   * dispatch and its slots hold routed_cap routed rows (0: token_cap) */
  int ffn_rank, ffn_size;
  int64_t routed_cap;
} orc_cfg;

/* Header check of one dispatch slot ([RFC-GPU] "Window and slot layout":
 * the flag advancing past what was last seen means a new payload; magic and
 * version self-check; layer and token counts travel in band; the shutdown
 * bit; [RFC-GPU] "Risks and alternatives": the header's echoed seq;
 * [WIRE] step 2: the token count must equal the recorded length).  The
 * first failing check, in this order, is reported. */
static int orc_check_slot(const orc_cfg* c, uint8_t* win, const orc_layout* L,
                          int region, int stage, int layer, int seq_len,
                          uint64_t seen) {
  uint64_t f = *orc_flag(win, region, stage, c->ring_depth);
  if (f <= seen) return ORC_ERR_TIMEOUT;
  const uint8_t* s = orc_slot(win, L, region, stage, c->ring_depth);
  const int32_t* h = (const int32_t*)(s + L->header);
  if ((uint32_t)h[H_MAGIC] != ORC_MAGIC || h[H_VERSION] != ORC_VERSION ||
      h[H_NUM_EXPERTS] != c->num_experts || h[H_LEN] != H_FIXED_WORDS + c->num_experts)
    return ORC_ERR_HEADER;
  if ((uint32_t)h[H_SEQ] != (uint32_t)f || h[H_ECHO_SEQ] != h[H_SEQ]) return ORC_ERR_SEQ;
  if (h[H_FLAGS] & ORC_FLAG_SHUTDOWN) return ORC_ERR_SHUTDOWN;
  if (h[H_LAYER] != layer) return ORC_ERR_LAYER;
  if (h[H_STAGE] != stage) return ORC_ERR_STAGE;
  if (h[H_NUM_TOKENS] != seq_len) return ORC_ERR_SHAPE;
  if (h[H_NUM_TOKENS] > c->token_cap) return ORC_ERR_CAPACITY;
  if (h[H_ROUTED_TOKENS] != 0) return ORC_ERR_SHAPE;
  int st = h[H_SHARED_TOKENS];
  if (st != 0 && (st != seq_len || c->shared_inter <= 0)) return ORC_ERR_SHAPE;
  if (st) {
    const int32_t* sidx = (const int32_t*)(s + L->shared_idx);
    for (int i = 0; i < st; i++) if (sidx[i] != i) return ORC_ERR_SHAPE;
  }
  return ORC_OK;
}

/* Host-side argument rules of the forward call: peers listed once each and
 * in range, non-negative lengths, total within the configured capacity
 * ([RFC-GPU] "Capacity and ring depth": overflow raises, never truncates). */
static int orc_check_args(const orc_cfg* c, int stage, const int* seq_lens,
                          const int* slots, int n_peers) {
  if (n_peers <= 0 || n_peers > c->num_regions) return ORC_ERR_ARG;
  if (stage < 0 || stage >= c->ring_depth) return ORC_ERR_ARG;
  int64_t T = 0;
  for (int i = 0; i < n_peers; i++) {
    if (slots[i] < 0 || slots[i] >= c->num_regions) return ORC_ERR_ARG;
    for (int j = 0; j < i; j++) if (slots[j] == slots[i]) return ORC_ERR_ARG;
    if (seq_lens[i] < 0) return ORC_ERR_ARG;
    if (seq_lens[i] > c->token_cap) return ORC_ERR_CAPACITY;
    T += seq_lens[i];
  }
  int cap = c->max_total_tokens > 0 ? c->max_total_tokens : c->num_regions * c->token_cap;
  if (T > cap) return ORC_ERR_CAPACITY;
  return ORC_OK;
}

/* The whole FFN-side step over one fan-in.
 *  1. [WIRE] step 3: the input is the concatenation of the listed peers'
 *     rows, in list order; token t belongs to the peer whose prefix range
 *     holds it.
 *  2. router, 3. plan, 4. experts + combine (above).
 *  5. [WIRE] step 4: rows [prefix_i, prefix_i + n_i) go back to peer i:
 *     the return slot (same layout, [RFC-GPU]) gets routed_x = the output
 *     rows, route_table = the chosen expert ids, the header (echoing the
 *     dispatch seq; routed_tokens = n*k, shared_tokens as received,
 *     expert_counts = this peer's own per-expert partial counts), then the
 *     return flag = the dispatch seq.
 * seen[] holds, per slot number, the last flag value consumed; it is
 * updated on success.  Optional outputs (NULL to skip): ids/w [T,k],
 * counts [E], offsets [E+1], perm/inv [T*k], gap [T], out64 [T, hidden]
 * unrounded, h_out [T, k, I]. */
int orc_ffn_forward(const orc_cfg* c, uint8_t* in_win, uint8_t* ret_win,
                    const orc_weights* W, int layer, int stage, const int* seq_lens,
                    const int* slots, int n_peers, uint64_t* seen, int* ids_out,
                    float* w_out, int* counts_out, int* offsets_out, int* perm_out,
                    int* inv_out, double* gap_out, double* out64, double* h_out,
                    int nthreads) {
  orc_layout L;
  int rc = orc_slot_layout(c->num_regions, c->ring_depth, c->token_cap, c->topk,
                           c->hidden, c->act_bytes, c->num_experts, c->shared_inter > 0, &L);
  if (rc) return rc;
  rc = orc_check_args(c, stage, seq_lens, slots, n_peers);
  if (rc) return rc;
  for (int i = 0; i < n_peers; i++) {
    rc = orc_check_slot(c, in_win, &L, slots[i], stage, layer, seq_lens[i],
                        seen[(int64_t)slots[i] * c->ring_depth + stage]);
    if (rc) return rc;
  }
  const int H = c->hidden, E = c->num_experts, k = c->topk, ab = c->act_bytes;
  int* prefix = (int*)malloc(sizeof(int) * (n_peers + 1));
  prefix[0] = 0;
  for (int i = 0; i < n_peers; i++) prefix[i + 1] = prefix[i] + seq_lens[i];
  const int T = prefix[n_peers];
  int* ids = (int*)malloc(sizeof(int) * ((int64_t)T * k + 1));
  float* w = (float*)malloc(sizeof(float) * ((int64_t)T * k + 1));
  double* out = (double*)malloc(sizeof(double) * ((int64_t)T * H + 1));

#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int t = 0; t < T; t++) {
    int i = 0;
    while (t >= prefix[i + 1]) i++;
    int local = t - prefix[i];
#if ORC_PLANT == 7
    const uint8_t* s = orc_slot(in_win, &L, slots[n_peers - 1 - i], stage, c->ring_depth);
#else
    const uint8_t* s = orc_slot(in_win, &L, slots[i], stage, c->ring_depth);
#endif
    const int32_t* hd = (const int32_t*)(s + L.header);
    double* xr = (double*)malloc(sizeof(double) * H);
    double* xs = NULL;
    float* xf = (float*)malloc(sizeof(float) * H);
    for (int h = 0; h < H; h++) {
      xr[h] = orc_ld(s + L.routed_x, ab, (int64_t)local * H + h);
      xf[h] = (float)xr[h];
    }
    if (hd[H_SHARED_TOKENS] > 0) {
      xs = (double*)malloc(sizeof(double) * H);
      for (int h = 0; h < H; h++) xs[h] = orc_ld(s + L.shared_x, ab, (int64_t)local * H + h);
    }
    orc_router_token(xf, H, W->Wg, W->bias, E, k, c->renorm, c->routed_scaling,
                     ids + (int64_t)t * k, w + (int64_t)t * k, gap_out ? gap_out + t : NULL,
                     NULL);
    orc_token_forward(xr, xs, H, E, k, c->inter, c->shared_inter, W, ab,
                      ids + (int64_t)t * k, w + (int64_t)t * k, out + (int64_t)t * H,
                      h_out ? h_out + (int64_t)t * k * c->inter : NULL);
    free(xr);
    free(xf);
    free(xs);
  }

  int* counts = (int*)malloc(sizeof(int) * E);
  int* offsets = (int*)malloc(sizeof(int) * (E + 1));
  int* perm = (int*)malloc(sizeof(int) * ((int64_t)T * k + 1));
  int* inv = (int*)malloc(sizeof(int) * ((int64_t)T * k + 1));
  orc_plan(ids, T * k, E, counts, offsets, perm, inv);

  /* split back into the return slots */
  for (int i = 0; i < n_peers; i++) {
    int p = slots[i], n = seq_lens[i];
    uint64_t seq = *orc_flag(in_win, p, stage, c->ring_depth);
    const int32_t* hin = (const int32_t*)(orc_slot(in_win, &L, p, stage, c->ring_depth) + L.header);
    uint8_t* s = orc_slot(ret_win, &L, p, stage, c->ring_depth);
    for (int r = 0; r < n; r++) {
      int t = prefix[i] + r;
      for (int h = 0; h < H; h++) {
        double v = out[(int64_t)t * H + h];
        if (ab == 2)
          ((uint16_t*)(s + L.routed_x))[(int64_t)r * H + h] = orc_f64_to_bf16(v);
        else
          ((float*)(s + L.routed_x))[(int64_t)r * H + h] = (float)v;
      }
      for (int j = 0; j < k; j++)
        ((int32_t*)(s + L.route_table))[(int64_t)r * k + j] = ids[(int64_t)t * k + j];
    }
    int32_t* h = (int32_t*)(s + L.header);
    memset(h, 0, (size_t)(H_FIXED_WORDS + E) * 4);
    h[H_MAGIC] = (int32_t)ORC_MAGIC;
    h[H_VERSION] = ORC_VERSION;
    h[H_FLAGS] = 0;
    h[H_SEQ] = (int32_t)(uint32_t)seq;
    h[H_ECHO_SEQ] = (int32_t)(uint32_t)seq;
    h[H_LAYER] = layer;
    h[H_STAGE] = stage;
    h[H_NUM_TOKENS] = n;
    h[H_ROUTED_TOKENS] = n * k;
    h[H_SHARED_TOKENS] = hin[H_SHARED_TOKENS];
    h[H_NUM_EXPERTS] = E;
    h[H_LEN] = H_FIXED_WORDS + E;
    for (int r = 0; r < n; r++)
      for (int j = 0; j < k; j++) h[H_FIXED_WORDS + ids[(int64_t)(prefix[i] + r) * k + j]]++;
    *orc_flag(ret_win, p, stage, c->ring_depth) = seq;
    seen[(int64_t)p * c->ring_depth + stage] = seq;
  }

  if (ids_out) memcpy(ids_out, ids, sizeof(int) * (size_t)T * k);
  if (w_out) memcpy(w_out, w, sizeof(float) * (size_t)T * k);
  if (counts_out) memcpy(counts_out, counts, sizeof(int) * E);
  if (offsets_out) memcpy(offsets_out, offsets, sizeof(int) * (E + 1));
  if (perm_out) memcpy(perm_out, perm, sizeof(int) * (size_t)T * k);
  if (inv_out) memcpy(inv_out, inv, sizeof(int) * (size_t)T * k);
  if (out64) memcpy(out64, out, sizeof(double) * (size_t)T * H);
  free(prefix); free(ids); free(w); free(out);
  free(counts); free(offsets); free(perm); free(inv);
  return ORC_OK;
}

/* Per-token outputs for a sample of global token indices of a fan-in
 * (used where the whole fan-in is too large for the oracle): the same steps
 * as orc_ffn_forward restricted to the listed tokens; no slot is written.
 * out64 is [n_sample, hidden]; ids/w are [n_sample, k]. */
int orc_forward_tokens(const orc_cfg* c, uint8_t* in_win, const orc_weights* W,
                       int stage, const int* seq_lens, const int* slots, int n_peers,
                       const int* tokens, int n_sample, int* ids_out, float* w_out,
                       double* out64, int nthreads) {
  orc_layout L;
  int rc = orc_slot_layout(c->num_regions, c->ring_depth, c->token_cap, c->topk,
                           c->hidden, c->act_bytes, c->num_experts, c->shared_inter > 0, &L);
  if (rc) return rc;
  const int H = c->hidden, k = c->topk, ab = c->act_bytes;
  int* prefix = (int*)malloc(sizeof(int) * (n_peers + 1));
  prefix[0] = 0;
  for (int i = 0; i < n_peers; i++) prefix[i + 1] = prefix[i] + seq_lens[i];
  for (int q = 0; q < n_sample; q++)
    if (tokens[q] < 0 || tokens[q] >= prefix[n_peers]) { free(prefix); return ORC_ERR_ARG; }
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int q = 0; q < n_sample; q++) {
    int t = tokens[q], i = 0;
    while (t >= prefix[i + 1]) i++;
    int local = t - prefix[i];
    const uint8_t* s = orc_slot(in_win, &L, slots[i], stage, c->ring_depth);
    const int32_t* hd = (const int32_t*)(s + L.header);
    double* xr = (double*)malloc(sizeof(double) * H);
    double* xs = NULL;
    float* xf = (float*)malloc(sizeof(float) * H);
    for (int h = 0; h < H; h++) {
      xr[h] = orc_ld(s + L.routed_x, ab, (int64_t)local * H + h);
      xf[h] = (float)xr[h];
    }
    if (hd[H_SHARED_TOKENS] > 0) {
      xs = (double*)malloc(sizeof(double) * H);
      for (int h = 0; h < H; h++) xs[h] = orc_ld(s + L.shared_x, ab, (int64_t)local * H + h);
    }
    orc_router_token(xf, H, W->Wg, W->bias, c->num_experts, k, c->renorm,
                     c->routed_scaling, ids_out + (int64_t)q * k, w_out + (int64_t)q * k,
                     NULL, NULL);
    orc_token_forward(xr, xs, H, c->num_experts, k, c->inter, c->shared_inter, W, ab,
                      ids_out + (int64_t)q * k, w_out + (int64_t)q * k,
                      out64 + (int64_t)q * H, NULL);
    free(xr); free(xf); free(xs);
  }
  free(prefix);
  return ORC_OK;
}

/* Combine alone, for the identity-expert check of [RFC-GPU] "Existing
 * verification": out[t] = sum_j w[t,j] * y[t,j,:] (+ s[t]) in fp64. */
void orc_combine(const double* y, const float* w, const double* s, int T, int k,
                 int hidden, double* out) {
  for (int t = 0; t < T; t++)
    for (int f = 0; f < hidden; f++) {
      double a = 0.0;
      for (int j = 0; j < k; j++) a += (double)w[(int64_t)t * k + j] * y[((int64_t)t * k + j) * hidden + f];
      if (s) a += s[(int64_t)t * hidden + f];
      out[(int64_t)t * hidden + f] = a;
    }
}

/* ------------------------------------------------------------------------ */
/* the Attention-side gate: routed rows arrive already grouped by expert      */
/* ------------------------------------------------------------------------ */

/* Dispatch slot of the grouped form ([RFC-GPU] "Data flow" steps 1-3: the
 * Attention side routes, sorts the flattened top-k ids stably and sends the
 * routed rows grouped by expert, with the per-expert row counts (group_list)
 * in the header; the shared rows travel as in the token form).  routed_x =
 * the R rows in group order, expert_counts = group_list (sum R),
 * routed_tokens = R, num_tokens = the peer's n tokens, shared_x = the n token
 * rows with shared_idx = 0..n-1 when with_shared.  Payload, then header, then
 * the flag.  Parity: the round trip and the combine identity below. */
int orc_pack_grouped(uint8_t* win, const orc_layout* L, int ring_depth, int region,
                     int stage, int layer, const void* rows, int R, const int* group_list,
                     const void* x, int n_tokens, int hidden, int act_bytes, int token_cap,
                     int num_experts, int with_shared, int has_shared, uint64_t seq) {
  if (n_tokens < 0 || n_tokens > token_cap || R < 0 || R > token_cap) return ORC_ERR_CAPACITY;
  if (with_shared && !has_shared) return ORC_ERR_ARG;
  int64_t sum = 0;
  for (int e = 0; e < num_experts; e++) {
    if (group_list[e] < 0) return ORC_ERR_ARG;
    sum += group_list[e];
  }
  if (sum != R) return ORC_ERR_SHAPE;
  uint8_t* s = orc_slot(win, L, region, stage, ring_depth);
  int64_t row = (int64_t)hidden * act_bytes;
  if (R) memcpy(s + L->routed_x, rows, (size_t)(R * row));
  if (with_shared) {
    int32_t* sidx = (int32_t*)(s + L->shared_idx);
    for (int i = 0; i < n_tokens; i++) sidx[i] = i;
    if (n_tokens) memcpy(s + L->shared_x, x, (size_t)(n_tokens * row));
  }
  int32_t* h = (int32_t*)(s + L->header);
  memset(h, 0, (size_t)(H_FIXED_WORDS + num_experts) * 4);
  h[H_MAGIC] = (int32_t)ORC_MAGIC;
  h[H_VERSION] = ORC_VERSION;
  h[H_SEQ] = (int32_t)(uint32_t)seq;
  h[H_ECHO_SEQ] = (int32_t)(uint32_t)seq;
  h[H_LAYER] = layer;
  h[H_STAGE] = stage;
  h[H_NUM_TOKENS] = n_tokens;
  h[H_ROUTED_TOKENS] = R;
  h[H_SHARED_TOKENS] = with_shared ? n_tokens : 0;
  h[H_NUM_EXPERTS] = num_experts;
  h[H_LEN] = H_FIXED_WORDS + num_experts;
  for (int e = 0; e < num_experts; e++) h[H_FIXED_WORDS + e] = group_list[e];
  *orc_flag(win, region, stage, ring_depth) = seq;
  return ORC_OK;
}

/* Routed rows a grouped slot may carry: routed_cap when the rank receives
 * token-level dispatch ([RFC-GPU] "Capacity and ring depth"; routed_cap > 0
 * in the configuration, with any number of ranks), else token_cap. */
static int64_t orc_rows_cap(const orc_cfg* c) {
  return c->routed_cap > 0 ? c->routed_cap : c->token_cap;
}

/* Header check of a grouped dispatch slot: the common fields in the order of
 * orc_check_slot, then num_tokens == n (within token_cap), routed_tokens ==
 * R (within the routed-row capacity), expert_counts summing to R, shared
 * rows 0 or the rank's round-robin share of the n tokens with shared_idx =
 * r, r + F, ... ([RFC-GPU] "Data flow" step 3; with one rank 0..n-1). */
static int orc_check_grouped(const orc_cfg* c, uint8_t* win, const orc_layout* L, int region,
                             int stage, int layer, int R, int n, uint64_t seen) {
  uint64_t f = *orc_flag(win, region, stage, c->ring_depth);
  if (f <= seen) return ORC_ERR_TIMEOUT;
  const uint8_t* s = orc_slot(win, L, region, stage, c->ring_depth);
  const int32_t* h = (const int32_t*)(s + L->header);
  if ((uint32_t)h[H_MAGIC] != ORC_MAGIC || h[H_VERSION] != ORC_VERSION ||
      h[H_NUM_EXPERTS] != c->num_experts || h[H_LEN] != H_FIXED_WORDS + c->num_experts)
    return ORC_ERR_HEADER;
  if ((uint32_t)h[H_SEQ] != (uint32_t)f || h[H_ECHO_SEQ] != h[H_SEQ]) return ORC_ERR_SEQ;
  if (h[H_FLAGS] & ORC_FLAG_SHUTDOWN) return ORC_ERR_SHUTDOWN;
  if (h[H_LAYER] != layer) return ORC_ERR_LAYER;
  if (h[H_STAGE] != stage) return ORC_ERR_STAGE;
  if (h[H_NUM_TOKENS] != n) return ORC_ERR_SHAPE;
  if (h[H_NUM_TOKENS] > c->token_cap) return ORC_ERR_CAPACITY;
  if (h[H_ROUTED_TOKENS] != R) return ORC_ERR_SHAPE;
  if (h[H_ROUTED_TOKENS] > orc_rows_cap(c)) return ORC_ERR_CAPACITY;
  int64_t sum = 0;
  for (int e = 0; e < c->num_experts; e++) {
    if (h[H_FIXED_WORDS + e] < 0) return ORC_ERR_SHAPE;
    sum += h[H_FIXED_WORDS + e];
  }
  if (sum != R) return ORC_ERR_SHAPE;
  const int F = c->ffn_size > 1 ? c->ffn_size : 1, rank = F > 1 ? c->ffn_rank : 0;
  int st = h[H_SHARED_TOKENS];
  if (st != 0 && (st != orc_rr_rows(n, rank, F) || c->shared_inter <= 0)) return ORC_ERR_SHAPE;
  if (st) {
    const int32_t* sidx = (const int32_t*)(s + L->shared_idx);
    for (int i = 0; i < st; i++) if (sidx[i] != rank + i * F) return ORC_ERR_SHAPE;
  }
  return ORC_OK;
}

/* The FFN step of the grouped form ([RFC-GPU] "Attention gate and FFN expert
 * compute": what arrives is already routed and grouped, so the FFN must not
 * route again; every row gets the expert id expanded from group_list and a
 * unit weight, i.e. a top-1 problem; the shared rows go through the shared
 * expert as their own batch; [RFC-GPU] "Data flow" step 4: the gate weights
 * stay on the Attention side, which weights and combines).  For each listed
 * peer i: y_r = expert(e_r)(row r) for its R_i rows and s_t = shared(x_t) for
 * its shared rows, in fp64, rounded once into the return slot (routed_x = the
 * y rows in arrival order, shared_x = the s rows); header echoing seq, with
 * routed_tokens = R_i, shared_tokens and expert_counts as received; then the
 * return flag = seq.  The argument rules follow orc_check_args with rows
 * (at most the routed-row capacity per peer) in place of tokens; the totals are bounded by
 * max_total_tokens * topk rows and max_total_tokens tokens.  Optional
 * outputs: y64 [sum R, hidden], s64 [sum of each peer's shared-row count
 * (n with one FFN rank, its round-robin share with several), hidden] (rows of the shared
 * branch of peers without shared rows are zero).  Parity: pinned by the
 * dense identity (E = 1) and by the combine identity with orc_ffn_forward. */
int orc_grouped_forward(const orc_cfg* c, uint8_t* in_win, uint8_t* ret_win,
                        const orc_weights* W, int layer, int stage, const int* rows,
                        const int* seq_lens, const int* slots, int n_peers, uint64_t* seen,
                        double* y64, double* s64, int nthreads) {
  orc_layout L;
  int rc = orc_slot_layout_ranks(c->num_regions, c->ring_depth, c->token_cap, c->topk,
                                 c->hidden, c->act_bytes, c->num_experts, c->shared_inter > 0,
                                 c->routed_cap, &L);
  if (rc) return rc;
  rc = orc_check_args(c, stage, seq_lens, slots, n_peers);
  if (rc) return rc;
  const int F = c->ffn_size > 1 ? c->ffn_size : 1, rank = F > 1 ? c->ffn_rank : 0;
  int64_t Rtot = 0;
  for (int i = 0; i < n_peers; i++) {
    if (rows[i] < 0) return ORC_ERR_ARG;
    if (rows[i] > orc_rows_cap(c)) return ORC_ERR_CAPACITY;
    Rtot += rows[i];
  }
  int cap = c->max_total_tokens > 0 ? c->max_total_tokens : c->num_regions * c->token_cap;
  if (Rtot > (int64_t)cap * c->topk) return ORC_ERR_CAPACITY;
  for (int i = 0; i < n_peers; i++) {
    rc = orc_check_grouped(c, in_win, &L, slots[i], stage, layer, rows[i], seq_lens[i],
                           seen[(int64_t)slots[i] * c->ring_depth + stage]);
    if (rc) return rc;
  }
  const int H = c->hidden, E = c->num_experts, ab = c->act_bytes;
  int64_t e13 = (int64_t)2 * c->inter * H, ed = (int64_t)H * c->inter;
  int64_t rbase = 0, tbase = 0;
  for (int i = 0; i < n_peers; i++) {
    int p = slots[i], R = rows[i], n = seq_lens[i];
    const uint8_t* sin = orc_slot(in_win, &L, p, stage, c->ring_depth);
    const int32_t* hin = (const int32_t*)(sin + L.header);
    uint8_t* sout = orc_slot(ret_win, &L, p, stage, c->ring_depth);
    const int shared = hin[H_SHARED_TOKENS] > 0;
    const int ns = orc_rr_rows(n, rank, F);   /* this rank's shared rows of the peer */
    /* expert of row r: the group of group_list holding it */
    int* expert = (int*)malloc(sizeof(int) * (R + 1));
    for (int e = 0, r = 0; e < E; e++)
      for (int q = 0; q < hin[H_FIXED_WORDS + e]; q++) expert[r++] = e;
    int nrows = R + (shared ? ns : 0);
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int q = 0; q < nrows; q++) {
      const int routed = q < R;
      const int r = routed ? q : q - R;
      const uint8_t* src = sin + (routed ? L.routed_x : L.shared_x);
      double* x = (double*)malloc(sizeof(double) * H);
      double* y = (double*)calloc((size_t)H, sizeof(double));
      for (int h = 0; h < H; h++) x[h] = orc_ld(src, ab, (int64_t)r * H + h);
      if (routed) {
        int e = expert[r];
        orc_swiglu_row(x, H, c->inter, (const char*)W->W13 + (int64_t)e * e13 * ab,
                       (const char*)W->Wd + (int64_t)e * ed * ab, ab, 1.0, y, NULL);
      } else {
        orc_swiglu_row(x, H, c->shared_inter, W->W13s, W->Wds, ab, 1.0, y, NULL);
      }
      uint8_t* dst = sout + (routed ? L.routed_x : L.shared_x);
      for (int h = 0; h < H; h++) {
        if (ab == 2) ((uint16_t*)dst)[(int64_t)r * H + h] = orc_f64_to_bf16(y[h]);
        else ((float*)dst)[(int64_t)r * H + h] = (float)y[h];
      }
      if (routed && y64) memcpy(y64 + (rbase + r) * H, y, sizeof(double) * H);
      if (!routed && s64) memcpy(s64 + (tbase + r) * H, y, sizeof(double) * H);
      free(x);
      free(y);
    }
    if (s64 && !shared) memset(s64 + tbase * H, 0, sizeof(double) * (size_t)ns * H);
    free(expert);
    uint64_t seq = *orc_flag(in_win, p, stage, c->ring_depth);
    int32_t* h = (int32_t*)(sout + L.header);
    memset(h, 0, (size_t)(H_FIXED_WORDS + E) * 4);
    h[H_MAGIC] = (int32_t)ORC_MAGIC;
    h[H_VERSION] = ORC_VERSION;
    h[H_SEQ] = (int32_t)(uint32_t)seq;
    h[H_ECHO_SEQ] = (int32_t)(uint32_t)seq;
    h[H_LAYER] = layer;
    h[H_STAGE] = stage;
    h[H_NUM_TOKENS] = n;
    h[H_ROUTED_TOKENS] = R;
    h[H_SHARED_TOKENS] = hin[H_SHARED_TOKENS];
    h[H_NUM_EXPERTS] = E;
    h[H_LEN] = H_FIXED_WORDS + E;
    for (int e = 0; e < E; e++) h[H_FIXED_WORDS + e] = hin[H_FIXED_WORDS + e];
    *orc_flag(ret_win, p, stage, c->ring_depth) = seq;
    seen[(int64_t)p * c->ring_depth + stage] = seq;
    rbase += R;
    tbase += ns;
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* token-level dispatch to several FFN ranks and the Attention-side combine   */
/* ------------------------------------------------------------------------ */

/* One Attention peer's send to F FFN ranks ([RFC-GPU] "Data flow" steps 1-3
 * and "Capacity and ring depth").  ids: the peer's top-k expert ids [n, k]
 * (global, 0..E-1).  Step 1: the flattened ids are sorted stably; since every
 * rank owns a contiguous block of experts (orc_expert_range), the sorted
 * order is segmented by destination rank and grouped by local expert within
 * each segment; the bincount gives each rank's group list.  A segment longer
 * than routed_cap raises (AFD_ERR_CAPACITY) before anything is written.
 * Step 3: rank r's slot (region = this peer, ring = stage) gets routed_x =
 * the rows x[f / k] of its segment in order, route_table = their flattened
 * indices f, shared rows = the tokens arange(r, n, F) with shared_idx = those
 * token indices (when with_shared), and the header (num_tokens = n,
 * routed_tokens = the segment's length, shared_tokens, num_experts = the
 * rank's count, expert_counts = its group list), then the flag = seq.  Every
 * rank gets its message, empty ones included.  Outputs for the combine:
 * dst[f] = rank of partial f, pos[f] = its row in that rank's segment,
 * rows_out[r] = segment lengths.  wins[r] / Ls[r]: rank r's dispatch window
 * and slot layout.  Parity: pinned by the page's unit-test list (every
 * partial routed exactly once, segments grouped by local expert, E not
 * divisible by F, an empty destination) and by the round trip below. */
int orc_dispatch_ranks(uint8_t** wins, const orc_layout* Ls, int F, int ring_depth, int region,
                       int stage, int layer, const void* x, int n, const int* ids, int k, int E,
                       int hidden, int act_bytes, int token_cap, int64_t routed_cap,
                       int with_shared, int has_shared, uint64_t seq, int* dst, int* pos,
                       int* rows_out) {
  if (F < 1 || n < 0 || k < 1 || E < F) return ORC_ERR_ARG;
  if (n > token_cap) return ORC_ERR_CAPACITY;
  if (with_shared && !has_shared) return ORC_ERR_ARG;
  const int N = n * k;
  for (int f = 0; f < N; f++) if (ids[f] < 0 || ids[f] >= E) return ORC_ERR_ARG;
  /* stable sort of the flattened ids (insertion sort: plain and stable) */
  int* order = (int*)malloc(sizeof(int) * (N + 1));
  for (int f = 0; f < N; f++) {
    int q = f;
    while (q > 0 && ids[order[q - 1]] > ids[f]) { order[q] = order[q - 1]; q--; }
    order[q] = f;
  }
  int* counts = (int*)calloc((size_t)E, sizeof(int));
  for (int f = 0; f < N; f++) counts[ids[f]]++;
  int64_t seg = 0;
  int rc = ORC_OK;
  for (int r = 0; r < F && !rc; r++) {
    int first, cnt;
    orc_expert_range(E, F, r, &first, &cnt);
    int R = 0;
    for (int e = first; e < first + cnt; e++) R += counts[e];
    rows_out[r] = R;
    if (R > routed_cap) rc = ORC_ERR_CAPACITY;
  }
  if (rc) { free(order); free(counts); return rc; }
  const int64_t row = (int64_t)hidden * act_bytes;
  for (int r = 0; r < F; r++) {
    int first, cnt;
    orc_expert_range(E, F, r, &first, &cnt);
    const int R = rows_out[r];
    uint8_t* s = orc_slot(wins[r], &Ls[r], region, stage, ring_depth);
    int32_t* table = (int32_t*)(s + Ls[r].route_table);
    for (int q = 0; q < R; q++) {
      const int f = order[seg + q];
      memcpy(s + Ls[r].routed_x + (int64_t)q * row, (const char*)x + (int64_t)(f / k) * row,
             (size_t)row);
      table[q] = f;
      dst[f] = r;
      pos[f] = q;
    }
    seg += R;
    const int ns = with_shared ? orc_rr_rows(n, r, F) : 0;
    int32_t* sidx = (int32_t*)(s + Ls[r].shared_idx);
    for (int i = 0; i < ns; i++) {
      const int t = r + i * F;
      sidx[i] = t;
      memcpy(s + Ls[r].shared_x + (int64_t)i * row, (const char*)x + (int64_t)t * row, (size_t)row);
    }
    int32_t* h = (int32_t*)(s + Ls[r].header);
    memset(h, 0, (size_t)(H_FIXED_WORDS + cnt) * 4);
    h[H_MAGIC] = (int32_t)ORC_MAGIC;
    h[H_VERSION] = ORC_VERSION;
    h[H_SEQ] = (int32_t)(uint32_t)seq;
    h[H_ECHO_SEQ] = (int32_t)(uint32_t)seq;
    h[H_LAYER] = layer;
    h[H_STAGE] = stage;
    h[H_NUM_TOKENS] = n;
    h[H_ROUTED_TOKENS] = R;
    h[H_SHARED_TOKENS] = ns;
    h[H_NUM_EXPERTS] = cnt;
    h[H_LEN] = H_FIXED_WORDS + cnt;
    for (int e = 0; e < cnt; e++) h[H_FIXED_WORDS + e] = counts[first + e];
    *orc_flag(wins[r], region, stage, ring_depth) = seq;
  }
  free(order);
  free(counts);
  return ORC_OK;
}

/* The Attention side's receive of a multi-rank step ([RFC-GPU] "Data flow":
 * recv_ffn_output waits only on the ranks that received data at dispatch --
 * a rank that was sent no rows is not waited for -- and accumulates each arrival in
 * fp32 with the weighted scatter; the shared branch is added by shared_idx).
 * For every rank r with rows_out[r] routed rows or shared rows: its return
 * flag must equal expect_seq and its header echo it, with routed_tokens =
 * rows_out[r] and shared_tokens = its round-robin share (or 0 without
 * shared rows).  Then, in fp64, out[t] = sum over j ascending of w[t, j] *
 * y(dst[t k + j], pos[t k + j]) + s(t mod F, t div F) -- y and s as the ranks
 * returned them -- rounded once to the activation type into out_act (when
 * not NULL); out64 keeps the unrounded sums.  Parity: the round trip with F
 * ranks equals the one with a single rank exactly (pinned in the tests). */
int orc_attn_combine(uint8_t** rets, const orc_layout* Ls, int F, int ring_depth, int region,
                     int stage, int n, int k, const int* dst, const int* pos, const float* w,
                     const int* rows_out, int with_shared, int hidden, int act_bytes,
                     uint64_t expect_seq, double* out64, void* out_act) {
  for (int r = 0; r < F; r++) {
    const int ns = with_shared ? orc_rr_rows(n, r, F) : 0;
    if (rows_out[r] == 0 && ns == 0) continue;  /* nothing sent there: no wait */
    uint64_t fl = *orc_flag(rets[r], region, stage, ring_depth);
    if (fl < expect_seq) return ORC_ERR_TIMEOUT;
    if (fl > expect_seq) return ORC_ERR_SEQ;
    const int32_t* h = (const int32_t*)(orc_slot(rets[r], &Ls[r], region, stage, ring_depth) +
                                        Ls[r].header);
    if ((uint32_t)h[H_MAGIC] != ORC_MAGIC || h[H_VERSION] != ORC_VERSION) return ORC_ERR_HEADER;
    if ((uint32_t)h[H_ECHO_SEQ] != (uint32_t)expect_seq) return ORC_ERR_SEQ;
    if (h[H_NUM_TOKENS] != n || h[H_ROUTED_TOKENS] != rows_out[r] || h[H_SHARED_TOKENS] != ns)
      return ORC_ERR_SHAPE;
  }
  for (int t = 0; t < n; t++)
    for (int c = 0; c < hidden; c++) {
      double a = 0.0;
      for (int j = 0; j < k; j++) {
        const int f = t * k + j, r = dst[f];
        const uint8_t* s = orc_slot(rets[r], &Ls[r], region, stage, ring_depth);
        a += (double)w[f] * orc_ld(s + Ls[r].routed_x, act_bytes, (int64_t)pos[f] * hidden + c);
      }
      if (with_shared) {
        const int r = t % F;
        const uint8_t* s = orc_slot(rets[r], &Ls[r], region, stage, ring_depth);
        a += orc_ld(s + Ls[r].shared_x, act_bytes, (int64_t)(t / F) * hidden + c);
      }
      if (out64) out64[(int64_t)t * hidden + c] = a;
      if (out_act) {
        if (act_bytes == 2) ((uint16_t*)out_act)[(int64_t)t * hidden + c] = orc_f64_to_bf16(a);
        else ((float*)out_act)[(int64_t)t * hidden + c] = (float)a;
      }
    }
  return ORC_OK;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
