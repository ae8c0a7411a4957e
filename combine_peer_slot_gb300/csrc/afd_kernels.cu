// afd_kernels.cu -- the memory-bound and control kernels of the AFD FFN-side
// step on sm_103a: slot pack / header / flag, header check with a bounded
// flag wait, router, dispatch plan, permute-gather, combine + split, return
// header + flag, unpack, and the SIMT GEMM used for fp32 activations.
#include "afd_internal.cuh"

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint8_t* slot_ptr(uint8_t* win, const WinGeom& g, int region,
                                             int stage) {
  return win + g.flags_bytes + ((int64_t)region * g.ring_depth + stage) * g.slot_bytes;
}
__device__ __forceinline__ const uint8_t* slot_ptr(const uint8_t* win, const WinGeom& g,
                                                   int region, int stage) {
  return win + g.flags_bytes + ((int64_t)region * g.ring_depth + stage) * g.slot_bytes;
}

// list entry i holding global token t of the concatenation
__device__ __forceinline__ int entry_of(const FanIn& f, int t) {
  int lo = 0, hi = f.n_peers - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (f.prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}

// ---------------------------------------------------------------------------
// pack: payload, then header + flag (Async GPU Connector, "Window and slot
// layout": the flag is written after the payload, on the same stream)
// ---------------------------------------------------------------------------
__global__ void k_pack_payload(uint8_t* win, WinGeom g, int region, int stage,
                               const uint4* __restrict__ x, int n, int row_bytes,
                               int with_shared) {
  uint8_t* slot = slot_ptr(win, g, region, stage);
  uint4* rx = reinterpret_cast<uint4*>(slot + g.routed_x);
  uint4* sx = reinterpret_cast<uint4*>(slot + g.shared_x);
  int32_t* sidx = reinterpret_cast<int32_t*>(slot + g.shared_idx);
  const int64_t nvec = (int64_t)n * row_bytes / 16;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    uint4 v = x[i];
    rx[i] = v;
    if (with_shared) sx[i] = v;
  }
  if (with_shared)
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
      sidx[i] = (int32_t)i;
}

__global__ void k_pack_header(uint8_t* win, WinGeom g, int region, int stage, int layer, int n,
                              int with_shared, int num_experts, uint64_t seq, int shutdown) {
  uint8_t* slot = slot_ptr(win, g, region, stage);
  int32_t* h = reinterpret_cast<int32_t*>(slot + g.header);
  for (int i = threadIdx.x; i < AFD_HEADER_FIXED_WORDS + num_experts; i += blockDim.x) {
    int32_t v = 0;
    switch (i) {
      case 0: v = (int32_t)AFD_HEADER_MAGIC; break;
      case 1: v = AFD_HEADER_VERSION; break;
      case 2: v = shutdown ? AFD_FLAG_SHUTDOWN : 0; break;
      case 3: v = (int32_t)(uint32_t)seq; break;
      case 4: v = (int32_t)(uint32_t)seq; break;
      case 5: v = layer; break;
      case 6: v = stage; break;
      case 7: v = n; break;
      case 8: v = 0; break;
      case 9: v = with_shared ? n : 0; break;
      case 10: v = num_experts; break;
      case 11: v = AFD_HEADER_FIXED_WORDS + num_experts; break;
      default: v = 0;
    }
    h[i] = v;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence_system();
    uint64_t* flag = reinterpret_cast<uint64_t*>(win) + (int64_t)region * g.ring_depth + stage;
    st_release_u64(flag, seq);
  }
}

// ---------------------------------------------------------------------------
// a0: bounded wait for each listed flag, then header checks.  The order of
// the checks fixes which error is reported: the first failing check of the
// first failing list entry.
// ---------------------------------------------------------------------------
__global__ void k_header_check(const uint8_t* win, WinGeom g, FanIn f, DevWS ws, int E,
                               int token_cap, int has_shared_expert, int64_t timeout_ns) {
  __shared__ int err[AFD_MAX_PEERS];
  __shared__ int bad_sidx[AFD_MAX_PEERS];
  __shared__ int shared_n[AFD_MAX_PEERS];
  __shared__ int skip;
  const int tid = threadIdx.x;
  if (tid == 0) skip = read_status(ws.status);
  if (tid < AFD_MAX_PEERS) { err[tid] = 0; bad_sidx[tid] = 0; shared_n[tid] = 0; }
  __syncthreads();
  if (skip) return;
  if (tid < f.n_peers) {
    const int i = tid;
    const int slotno = f.region[i] * g.ring_depth + f.stage;
    const uint64_t* flagp = reinterpret_cast<const uint64_t*>(win) + slotno;
    const uint64_t seen = ws.seen[slotno];
    const uint64_t t0 = globaltimer_ns();
    uint64_t fl = ld_acquire_u64(flagp);
    unsigned backoff = 32;
    int e = 0;
    while (fl <= seen) {
      if (globaltimer_ns() - t0 > (uint64_t)timeout_ns) { e = AFD_ERR_TIMEOUT; break; }
      __nanosleep(backoff);
      if (backoff < 1024) backoff <<= 1;
      fl = ld_acquire_u64(flagp);
    }
    if (!e) {
      const volatile int32_t* h =
          reinterpret_cast<const volatile int32_t*>(slot_ptr(win, g, f.region[i], f.stage) + g.header);
      const int n = f.prefix[i + 1] - f.prefix[i];
      if ((uint32_t)h[0] != (uint32_t)AFD_HEADER_MAGIC || h[1] != AFD_HEADER_VERSION ||
          h[10] != E || h[11] != AFD_HEADER_FIXED_WORDS + E)
        e = AFD_ERR_HEADER;
      else if ((uint32_t)h[3] != (uint32_t)fl || h[4] != h[3])
        e = AFD_ERR_SEQ;
      else if (h[2] & AFD_FLAG_SHUTDOWN)
        e = AFD_ERR_SHUTDOWN;
      else if (h[5] != f.layer)
        e = AFD_ERR_LAYER;
      else if (h[6] != f.stage)
        e = AFD_ERR_STAGE;
      else if (h[7] != n)
        e = AFD_ERR_SHAPE;
      else if (h[7] > token_cap)
        e = AFD_ERR_CAPACITY;
      else if (h[8] != 0)
        e = AFD_ERR_SHAPE;
      else if (h[9] != 0 && (h[9] != n || !has_shared_expert))
        e = AFD_ERR_SHAPE;
      if (!e) shared_n[i] = h[9];
    }
    err[i] = e;
    ws.cur_seq[i] = fl;
  }
  __syncthreads();
  // shared_idx must be 0..n-1: with one FFN rank every token is a shared
  // token (Async GPU Connector, "Data flow" step 3).
  for (int i = 0; i < f.n_peers; i++) {
    if (err[i] || shared_n[i] == 0) continue;
    const int32_t* sidx = reinterpret_cast<const int32_t*>(slot_ptr(win, g, f.region[i], f.stage) +
                                                           g.shared_idx);
    for (int r = tid; r < shared_n[i]; r += blockDim.x)
      if (sidx[r] != r) bad_sidx[i] = 1;
  }
  __syncthreads();
  if (tid == 0) {
    int first = 0;
    for (int i = 0; i < f.n_peers && !first; i++) {
      int e = err[i];
      if (!e && bad_sidx[i]) e = AFD_ERR_SHAPE;
      first = e;
    }
    if (first) {
      set_error(ws.status, first);
    } else {
      for (int i = 0; i < f.n_peers; i++) {
        ws.seen[f.region[i] * g.ring_depth + f.stage] = ws.cur_seq[i];
        ws.peer_shared[i] = shared_n[i] > 0;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// a1: router.  logits in the canonical fp32 order: lane l of a warp owns the
// fused multiply-add chain over h = l, l+32, ... ascending (from +0), then a
// butterfly with xor offsets 16, 8, 4, 2, 1, then + bias.  Top-k on the
// logits (ties -> lower expert index), softmax over all E for the weights.
// Block: 16 warps x 16 tokens; warp w owns experts [4w', 4w'+4) for
// w' = w, w+16, ...  Wg is read transposed ([E, hidden]) so each expert's
// column is coalesced.
// ---------------------------------------------------------------------------
// exp(a - b) for fp32 a >= ... b: the difference is split exactly into
// s + err (two-sum), so exp(a - b) = expf(s) * (1 + err) to first order.
__device__ __forceinline__ double exp_of_diff(float a, float b) {
  const float s = __fsub_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(-b, bb));
  return (double)expf(s) * (1.0 + (double)err);
}

constexpr int kRtTok = 16;
constexpr int kRtWarps = 16;
constexpr int kRtEpw = 4;

template <bool ACT_F32>
__global__ void __launch_bounds__(kRtWarps * 32)
k_router(const uint8_t* win, WinGeom g, FanIn f, DevWS ws, int hidden,
         const float* __restrict__ WgT, const float* __restrict__ bias, int E, int k,
         int renorm, float scale) {
  extern __shared__ __align__(16) uint8_t rt_smem[];
  using act_t = typename std::conditional<ACT_F32, float, uint16_t>::type;
  act_t* xs = reinterpret_cast<act_t*>(rt_smem);                       // [kRtTok][hidden]
  float* lg = reinterpret_cast<float*>(rt_smem + (size_t)kRtTok * hidden * sizeof(act_t));  // [kRtTok][E]
  if (read_status(ws.status)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRtTok;
  const int row_bytes = hidden * (int)sizeof(act_t);
  // stage the token rows straight from the peer slots (16-byte vectors)
  for (int tt = warp; tt < kRtTok; tt += kRtWarps) {
    const int t = t0 + tt;
    uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)tt * hidden);
    if (t < f.total) {
      const int i = entry_of(f, t);
      const uint4* src = reinterpret_cast<const uint4*>(
          slot_ptr(win, g, f.region[i], f.stage) + g.routed_x + (int64_t)(t - f.prefix[i]) * row_bytes);
      for (int v = lane; v < row_bytes / 16; v += 32) dst[v] = src[v];
    } else {
      for (int v = lane; v < row_bytes / 16; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
    }
  }
  __syncthreads();
  for (int eg = warp; eg * kRtEpw < E; eg += kRtWarps) {
    const int e0 = eg * kRtEpw;
    float acc[kRtTok][kRtEpw];
#pragma unroll
    for (int a = 0; a < kRtTok; a++)
#pragma unroll
      for (int b = 0; b < kRtEpw; b++) acc[a][b] = 0.0f;
    for (int h = lane; h < hidden; h += 32) {
      float wv[kRtEpw];
#pragma unroll
      for (int b = 0; b < kRtEpw; b++)
        wv[b] = (e0 + b < E) ? __ldg(WgT + (int64_t)(e0 + b) * hidden + h) : 0.0f;
#pragma unroll
      for (int a = 0; a < kRtTok; a++) {
        float xv;
        if constexpr (ACT_F32) xv = xs[(size_t)a * hidden + h];
        else xv = bf16_bits_to_f32(xs[(size_t)a * hidden + h]);
#pragma unroll
        for (int b = 0; b < kRtEpw; b++) acc[a][b] = __fmaf_rn(xv, wv[b], acc[a][b]);
      }
    }
#pragma unroll
    for (int a = 0; a < kRtTok; a++)
#pragma unroll
      for (int b = 0; b < kRtEpw; b++) {
        float v = acc[a][b];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
        acc[a][b] = v;
      }
    // lane a (< kRtTok) writes token a's logits
#pragma unroll
    for (int a = 0; a < kRtTok; a++)
      if (lane == a)
#pragma unroll
        for (int b = 0; b < kRtEpw; b++)
          if (e0 + b < E)
            lg[a * E + e0 + b] = bias ? __fadd_rn(acc[a][b], bias[e0 + b]) : acc[a][b];
  }
  __syncthreads();
  // top-k and gate weights: one warp per token
  for (int tt = warp; tt < kRtTok; tt += kRtWarps) {
    const int t = t0 + tt;
    if (t >= f.total) continue;
    const float* l = lg + tt * E;
    uint32_t taken = 0;  // bit m: expert lane + 32m chosen (E <= 256)
    float top_logit = 0.0f;
    int my_id = 0;       // lane j keeps the j-th choice
    float my_logit = 0.0f;
    for (int j = 0; j < k; j++) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      for (int m = 0; m * 32 + lane < E; m++) {
        const int e = m * 32 + lane;
        if (taken & (1u << m)) continue;
        float v = l[e];
        if (v != v) v = -INFINITY;  // a NaN logit ranks below every number
        if (v > bv || (v == bv && e < bi)) { bv = v; bi = e; }
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (j == 0) top_logit = bv;
      if (lane == j) { my_id = bi; my_logit = bv; }
    }
    // softmax over all E relative to the maximum; the denominator and the
    // renormalisation sum are accumulated in fp64
    double den = 0.0;
    for (int m = 0; m * 32 + lane < E; m++) den += exp_of_diff(l[m * 32 + lane], top_logit);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    const double p = (lane < k) ? exp_of_diff(my_logit, top_logit) / den : 0.0;
    double psum = p;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
    if (lane < k) {
      const double v = renorm ? p / psum : p;
      ws.ids[(int64_t)t * k + lane] = my_id;
      ws.w[(int64_t)t * k + lane] = (float)(v * (double)scale);
    }
  }
}

// ---------------------------------------------------------------------------
// a2/a3 plan: per-expert counts, exclusive offsets, the stable permutation
// of the flattened partial index f = t*k + j (a stable counting sort by
// expert, equal to argsort(stable=True) of the flattened ids, Async GPU
// Connector, "Data flow" step 1), per-peer counts for the return headers,
// and the tile tables of both grouped GEMMs.  One CTA of 32 warps: warp w
// owns a contiguous chunk of f; per-warp histograms give each warp's base
// per expert; within a warp, 32-element groups are ranked with match_any.
// ---------------------------------------------------------------------------
constexpr int kPlanWarps = 32;

__global__ void __launch_bounds__(kPlanWarps * 32)
k_plan(FanIn f, DevWS ws, int E, int k, int inter, int shared_inter, int hidden, int has_shared,
       int bn, GemmPlan* plan1, GemmPlan* plan2) {
  extern __shared__ __align__(16) int pl_smem[];
  int* hist = pl_smem;                          // [kPlanWarps][E]
  int* pcnt = hist + kPlanWarps * E;            // [n_peers][E]
  int* offs = pcnt + f.n_peers * E;             // [E + 1]
  __shared__ int skip;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) skip = read_status(ws.status);
  for (int i = tid; i < kPlanWarps * E + f.n_peers * E; i += blockDim.x) pl_smem[i] = 0;
  __syncthreads();
  if (skip) return;
  const int N = f.total * k;
  const int chunk = (N + kPlanWarps - 1) / kPlanWarps;
  const int c0 = min(N, warp * chunk), c1 = min(N, c0 + chunk);
  for (int fi = c0 + lane; fi < c1; fi += 32) {
    int e = ws.ids[fi];
    if (e < 0 || e >= E) {  // cannot come from the router; keep every index in range
      set_error(ws.status, AFD_ERR_SHAPE);
      e = 0;
      ws.ids[fi] = 0;
    }
    atomicAdd(&hist[warp * E + e], 1);
    atomicAdd(&pcnt[entry_of(f, fi / k) * E + e], 1);
  }
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < E; e++) {
      offs[e] = run;
      int c = 0;
      for (int w = 0; w < kPlanWarps; w++) c += hist[w * E + e];
      run += c;
    }
    offs[E] = run;
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int base = offs[e];
    for (int w = 0; w < kPlanWarps; w++) {
      const int c = hist[w * E + e];
      hist[w * E + e] = base;  // becomes warp w's cursor for expert e
      base += c;
    }
    ws.counts[e] = offs[e + 1] - offs[e];
    ws.offsets[e] = offs[e];
  }
  if (tid == 0) ws.offsets[E] = offs[E];
  for (int i = tid; i < f.n_peers * E; i += blockDim.x) ws.peer_counts[i] = pcnt[i];
  __syncthreads();
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int g0 = c0; g0 < c1; g0 += 32) {
    const int fi = g0 + lane;
    const bool ok = fi < c1;
    const int e = ok ? ws.ids[fi] : -1 - lane;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    int pos = 0;
    if (ok) pos = hist[warp * E + e] + rank;
    __syncwarp();
    if (ok && rank == 0) hist[warp * E + e] += __popc(peers);
    __syncwarp();
    if (ok) {
      ws.perm[pos] = fi;
      ws.inv[fi] = pos;
    }
  }
  // tile tables
  if (tid == 0) {
    int tiles1 = 0, tiles2 = 0, ng = 0;
    const int mt1 = (inter + 63) / 64, mt2 = (hidden + 127) / 128;
    for (int e = 0; e < E; e++, ng++) {
      const int rows = offs[e + 1] - offs[e];
      const int nt = (rows + bn - 1) / bn;
      GemmGroup a{rows, offs[e], offs[e], e, 0, mt1, nt, tiles1};
      GemmGroup b{rows, offs[e], offs[e], e, 0, mt2, nt, tiles2};
      plan1->g[ng] = a;
      plan2->g[ng] = b;
      tiles1 += mt1 * nt;
      tiles2 += mt2 * nt;
    }
    if (has_shared) {
      const int rows = f.total;
      const int nt = (rows + bn - 1) / bn;
      const int mts = (shared_inter + 63) / 64;
      GemmGroup a{rows, N, 0, 0, 1, mts, nt, tiles1};
      GemmGroup b{rows, 0, 0, 0, 1, mt2, nt, tiles2};
      plan1->g[ng] = a;
      plan2->g[ng] = b;
      tiles1 += mts * nt;
      tiles2 += mt2 * nt;
      ng++;
    }
    plan1->ngroups = ng;
    plan2->ngroups = ng;
    plan1->total_tiles = tiles1;
    plan2->total_tiles = tiles2;
    plan1->bn = bn;
    plan2->bn = bn;
  }
}

// ---------------------------------------------------------------------------
// a3 gather: Xp[pos] = the row of token perm[pos] / k, read straight from its
// peer slot (the fan-in concatenation is never materialised), then the
// shared rows in concatenation order.  One warp per row, 16-byte vectors.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
k_gather(const uint8_t* win, WinGeom g, FanIn f, DevWS ws, int k, int row_bytes,
         int has_shared) {
  if (read_status(ws.status)) return;
  const int N = f.total * k;
  const int rows = N + (has_shared ? f.total : 0);
  const int nvec = row_bytes / 16;
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(ws.xp) + (int64_t)r * row_bytes);
    int t;
    int64_t field;
    if (r < N) {
      t = ws.perm[r] / k;
      field = g.routed_x;
    } else {
      t = r - N;
      field = g.shared_x;
    }
    const int i = entry_of(f, t);
    const int lane = threadIdx.x & 31;
    if (r >= N && !ws.peer_shared[i]) {
      for (int v = lane; v < nvec; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(slot_ptr(win, g, f.region[i], f.stage) + field +
                                                      (int64_t)(t - f.prefix[i]) * row_bytes);
    for (int v = lane; v < nvec; v += 32) dst[v] = __ldg(src + v);
  }
}

// ---------------------------------------------------------------------------
// SIMT grouped GEMM (fp32 FMA; fp32 activations and cross-checks):
//   SwiGLU: h[r, c] = silu(g) * u, g = A[c] . B[r], u = A[M/2 + c] . B[r]
//   plain:  y[r, c] = A[c] . B[r]
// one thread per output element; blockIdx.y = group.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ld_act(const void* p, int64_t i, int act_f32) {
  return act_f32 ? reinterpret_cast<const float*>(p)[i]
                 : bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(p)[i]);
}

__global__ void __launch_bounds__(kThreads) k_gemm_simt(SimtArgs a) {
  if (read_status(a.status)) return;
  const GemmPlan* plan = a.plan;
  const int gi = blockIdx.y;
  if (gi >= plan->ngroups) return;
  const GemmGroup G = plan->g[gi];
  const int kind = G.kind;
  const int K = a.K[kind];
  const int cols = a.swiglu ? a.M[kind] / 2 : a.M[kind];
  const int64_t total = (int64_t)G.rows * cols;
  const void* A = a.A[kind];
  const int64_t a_off = (int64_t)G.a_idx * a.M[kind] * K;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(idx / cols), c = (int)(idx % cols);
    const int64_t brow = (int64_t)(G.b_row0 + r) * a.ldb[kind];
    float v;
    if (a.swiglu) {
      float gs = 0.0f, us = 0.0f;
      const int64_t ga = a_off + (int64_t)c * K, ua = a_off + (int64_t)(cols + c) * K;
      for (int q = 0; q < K; q++) {
        const float b = ld_act(a.B[kind], brow + q, a.act_f32);
        gs = fmaf(ld_act(A, ga + q, a.act_f32), b, gs);
        us = fmaf(ld_act(A, ua + q, a.act_f32), b, us);
      }
      v = gs / (1.0f + expf(-gs)) * us;
    } else {
      float s = 0.0f;
      const int64_t ra = a_off + (int64_t)c * K;
      for (int q = 0; q < K; q++) s = fmaf(ld_act(A, ra + q, a.act_f32), ld_act(a.B[kind], brow + q, a.act_f32), s);
      v = s;
    }
    const int64_t o = (int64_t)(G.out_row0 + r) * a.ldo[kind] + c;
    if (a.out_f32[kind]) reinterpret_cast<float*>(a.out[kind])[o] = v;
    else reinterpret_cast<__nv_bfloat16*>(a.out[kind])[o] = __float2bfloat16_rn(v);
  }
}

// ---------------------------------------------------------------------------
// a7 combine + split: out[t] = sum_{j ascending} w[t,j] * y[inv[t,j]] + s[t]
// in fp32 (fused multiply-add in j order, then + s), rounded to the
// activation type and written straight into the return slot of t's peer at
// its local row; the route_table row gets the chosen ids.  Deterministic:
// each output element is reduced by one thread in a fixed order.
// ---------------------------------------------------------------------------
template <bool ACT_F32, bool Y_F32>
__global__ void __launch_bounds__(kThreads)
k_combine(uint8_t* ret, WinGeom g, FanIn f, DevWS ws, int hidden, int k, int has_shared) {
  if (read_status(ws.status)) return;
  constexpr int kVec = 4;  // elements per thread step
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < f.total; t += warps) {
    const int i = entry_of(f, t);
    const int local = t - f.prefix[i];
    uint8_t* slot = slot_ptr(ret, g, f.region[i], f.stage);
    int my_pos = 0;
    float my_w = 0.0f;
    if (lane < k) {
      my_pos = ws.inv[(int64_t)t * k + lane];
      my_w = ws.w[(int64_t)t * k + lane];
      reinterpret_cast<int32_t*>(slot + g.route_table)[(int64_t)local * k + lane] =
          ws.ids[(int64_t)t * k + lane];
    }
    for (int c = lane * kVec; c < hidden; c += 32 * kVec) {
      float acc[kVec] = {0.f, 0.f, 0.f, 0.f};
      for (int j = 0; j < k; j++) {
        const int pos = __shfl_sync(0xffffffffu, my_pos, j);
        const float wj = __shfl_sync(0xffffffffu, my_w, j);
        float yv[kVec];
        if constexpr (Y_F32) {
          const float4 v = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(ws.y) +
                                                            (int64_t)pos * hidden + c);
          yv[0] = v.x; yv[1] = v.y; yv[2] = v.z; yv[3] = v.w;
        } else {
          const uint2 v = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(ws.y) +
                                                          (int64_t)pos * hidden + c);
          yv[0] = __uint_as_float(v.x << 16); yv[1] = __uint_as_float(v.x & 0xffff0000u);
          yv[2] = __uint_as_float(v.y << 16); yv[3] = __uint_as_float(v.y & 0xffff0000u);
        }
#pragma unroll
        for (int q = 0; q < kVec; q++) acc[q] = __fmaf_rn(wj, yv[q], acc[q]);
      }
      if (has_shared) {
        const float4 sv = *reinterpret_cast<const float4*>(ws.s + (int64_t)t * hidden + c);
        acc[0] = __fadd_rn(acc[0], sv.x); acc[1] = __fadd_rn(acc[1], sv.y);
        acc[2] = __fadd_rn(acc[2], sv.z); acc[3] = __fadd_rn(acc[3], sv.w);
      }
      if constexpr (ACT_F32) {
        *reinterpret_cast<float4*>(slot + g.routed_x + ((int64_t)local * hidden + c) * 4) =
            make_float4(acc[0], acc[1], acc[2], acc[3]);
      } else {
        __nv_bfloat162 p0 = __floats2bfloat162_rn(acc[0], acc[1]);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(acc[2], acc[3]);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t*>(&p0);
        o.y = *reinterpret_cast<uint32_t*>(&p1);
        *reinterpret_cast<uint2*>(slot + g.routed_x + ((int64_t)local * hidden + c) * 2) = o;
      }
    }
  }
}

// return headers, then the return flags (release) = the dispatch seq
__global__ void k_return_header(uint8_t* ret, WinGeom g, FanIn f, DevWS ws, int E, int k) {
  if (read_status(ws.status)) return;
  const int i = blockIdx.x;
  if (i >= f.n_peers) return;
  const int n = f.prefix[i + 1] - f.prefix[i];
  const uint64_t seq = ws.cur_seq[i];
  int32_t* h = reinterpret_cast<int32_t*>(slot_ptr(ret, g, f.region[i], f.stage) + g.header);
  for (int w = threadIdx.x; w < AFD_HEADER_FIXED_WORDS + E; w += blockDim.x) {
    int32_t v;
    switch (w) {
      case 0: v = (int32_t)AFD_HEADER_MAGIC; break;
      case 1: v = AFD_HEADER_VERSION; break;
      case 2: v = 0; break;
      case 3: v = (int32_t)(uint32_t)seq; break;
      case 4: v = (int32_t)(uint32_t)seq; break;
      case 5: v = f.layer; break;
      case 6: v = f.stage; break;
      case 7: v = n; break;
      case 8: v = n * k; break;
      case 9: v = ws.peer_shared[i] ? n : 0; break;
      case 10: v = E; break;
      case 11: v = AFD_HEADER_FIXED_WORDS + E; break;
      default: v = ws.peer_counts[i * E + (w - AFD_HEADER_FIXED_WORDS)];
    }
    h[w] = v;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence_system();
    st_release_u64(reinterpret_cast<uint64_t*>(ret) + f.region[i] * g.ring_depth + f.stage, seq);
  }
}

// Unpack: block-local bounded wait on the return flag and header check by
// thread 0, then the block copies its share of the rows.
__global__ void __launch_bounds__(kThreads)
k_unpack(const uint8_t* ret, WinGeom g, int region, int stage, uint4* out, int n, int row_bytes,
         int E, uint64_t expect_seq, int32_t* status, int64_t timeout_ns) {
  __shared__ int ok;
  if (threadIdx.x == 0) {
    int e = read_status(status) ? -1 : 0;
    if (!e) {
      const uint64_t* flagp = reinterpret_cast<const uint64_t*>(ret) + (int64_t)region * g.ring_depth + stage;
      const uint64_t t0 = globaltimer_ns();
      uint64_t fl = ld_acquire_u64(flagp);
      unsigned backoff = 32;
      while (fl < expect_seq) {
        if (globaltimer_ns() - t0 > (uint64_t)timeout_ns) { e = AFD_ERR_TIMEOUT; break; }
        __nanosleep(backoff);
        if (backoff < 1024) backoff <<= 1;
        fl = ld_acquire_u64(flagp);
      }
      if (!e && fl > expect_seq) e = AFD_ERR_SEQ;
      if (!e) {
        const volatile int32_t* h = reinterpret_cast<const volatile int32_t*>(
            slot_ptr(ret, g, region, stage) + g.header);
        if ((uint32_t)h[0] != (uint32_t)AFD_HEADER_MAGIC || h[1] != AFD_HEADER_VERSION ||
            h[10] != E || h[11] != AFD_HEADER_FIXED_WORDS + E)
          e = AFD_ERR_HEADER;
        else if ((uint32_t)h[4] != (uint32_t)expect_seq)
          e = AFD_ERR_SEQ;
        else if (h[7] != n)
          e = AFD_ERR_SHAPE;
      }
      if (e > 0) set_error(status, e);
    }
    ok = (e == 0);
  }
  __syncthreads();
  if (!ok) return;
  const uint4* src = reinterpret_cast<const uint4*>(slot_ptr(ret, g, region, stage) + g.routed_x);
  const int64_t nvec = (int64_t)n * row_bytes / 16;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec;
       v += (int64_t)gridDim.x * blockDim.x)
    out[v] = src[v];
}

__global__ void k_transpose_wg(const float* Wg, float* WgT, int hidden, int E) {
  const int64_t n = (int64_t)hidden * E;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(i / hidden), h = (int)(i % hidden);
    WgT[i] = Wg[(int64_t)h * E + e];
  }
}

inline int grid_for(int64_t work, int per_block, int cap) {
  int64_t b = (work + per_block - 1) / per_block;
  if (b < 1) b = 1;
  if (b > cap) b = cap;
  return (int)b;
}

}  // namespace

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_pack_payload(const LaunchCtx& lc, const WinGeom& g, uint8_t* win, int region,
                                int stage, const void* x, int n, int row_bytes, int with_shared,
                                const int32_t*) {
  if (n == 0) return cudaSuccess;
  const int64_t nvec = (int64_t)n * row_bytes / 16;
  k_pack_payload<<<grid_for(nvec, kThreads * 4, lc.num_sms * 8), kThreads, 0, lc.stream>>>(
      win, g, region, stage, reinterpret_cast<const uint4*>(x), n, row_bytes, with_shared);
  ++*lc.launches;
  return cudaGetLastError();
}

cudaError_t launch_pack_header(const LaunchCtx& lc, const WinGeom& g, uint8_t* win, int region,
                               int stage, int layer, int n, int with_shared, int num_experts,
                               uint64_t seq, int shutdown) {
  k_pack_header<<<1, 128, 0, lc.stream>>>(win, g, region, stage, layer, n, with_shared,
                                          num_experts, seq, shutdown);
  ++*lc.launches;
  return cudaGetLastError();
}

cudaError_t launch_header_check(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                                const FanIn& f, const DevWS& ws, int num_experts, int token_cap,
                                int has_shared_expert, int64_t timeout_ns) {
  k_header_check<<<1, kThreads, 0, lc.stream>>>(win, g, f, ws, num_experts, token_cap,
                                                has_shared_expert, timeout_ns);
  ++*lc.launches;
  return cudaGetLastError();
}

cudaError_t launch_router(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                          const FanIn& f, const DevWS& ws, int hidden, int act_f32,
                          const float* WgT, const float* bias, int E, int k, int renorm,
                          float scale) {
  if (f.total == 0) return cudaSuccess;
  const size_t smem = (size_t)kRtTok * hidden * (act_f32 ? 4 : 2) + (size_t)kRtTok * E * 4;
  const int grid = (f.total + kRtTok - 1) / kRtTok;
  cudaError_t err;
  if (act_f32) {
    err = cudaFuncSetAttribute(k_router<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    k_router<true><<<grid, kRtWarps * 32, smem, lc.stream>>>(win, g, f, ws, hidden, WgT, bias, E, k,
                                                             renorm, scale);
  } else {
    err = cudaFuncSetAttribute(k_router<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    k_router<false><<<grid, kRtWarps * 32, smem, lc.stream>>>(win, g, f, ws, hidden, WgT, bias, E,
                                                              k, renorm, scale);
  }
  ++*lc.launches;
  return cudaGetLastError();
}

cudaError_t launch_plan(const LaunchCtx& lc, const FanIn& f, const DevWS& ws, int E, int k,
                        int inter, int shared_inter, int hidden, int has_shared, int bn,
                        GemmPlan* plan1, GemmPlan* plan2) {
  const size_t smem = (size_t)(kPlanWarps * E + f.n_peers * E + E + 1) * 4;
  cudaError_t err = cudaFuncSetAttribute(k_plan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  k_plan<<<1, kPlanWarps * 32, smem, lc.stream>>>(f, ws, E, k, inter, shared_inter, hidden,
                                                  has_shared, bn, plan1, plan2);
  ++*lc.launches;
  return cudaGetLastError();
}

cudaError_t launch_gather(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                          const FanIn& f, const DevWS& ws, int k, int row_bytes, int has_shared) {
  const int64_t rows = (int64_t)f.total * k + (has_shared ? f.total : 0);
  if (rows == 0) return cudaSuccess;
  k_gather<<<grid_for(rows, kThreads / 32, lc.num_sms * 8), kThreads, 0, lc.stream>>>(
      win, g, f, ws, k, row_bytes, has_shared);
  ++*lc.launches;
  return cudaGetLastError();
}

cudaError_t launch_gemm_simt(const LaunchCtx& lc, const SimtArgs& a, int max_groups) {
  dim3 grid(lc.num_sms * 2, max_groups);
  k_gemm_simt<<<grid, kThreads, 0, lc.stream>>>(a);
  ++*lc.launches;
  return cudaGetLastError();
}

cudaError_t launch_combine(const LaunchCtx& lc, const WinGeom& g, uint8_t* ret, const FanIn& f,
                           const DevWS& ws, int hidden, int k, int act_f32, int has_shared,
                           int y_f32) {
  if (f.total == 0) return cudaSuccess;
  const int grid = grid_for(f.total, kThreads / 32, lc.num_sms * 8);
  if (act_f32 && y_f32)
    k_combine<true, true><<<grid, kThreads, 0, lc.stream>>>(ret, g, f, ws, hidden, k, has_shared);
  else if (!act_f32 && y_f32)
    k_combine<false, true><<<grid, kThreads, 0, lc.stream>>>(ret, g, f, ws, hidden, k, has_shared);
  else if (!act_f32 && !y_f32)
    k_combine<false, false><<<grid, kThreads, 0, lc.stream>>>(ret, g, f, ws, hidden, k, has_shared);
  else
    return cudaErrorInvalidValue;
  ++*lc.launches;
  return cudaGetLastError();
}

cudaError_t launch_return_header(const LaunchCtx& lc, const WinGeom& g, uint8_t* ret,
                                 const uint8_t*, const FanIn& f, const DevWS& ws, int E, int k) {
  k_return_header<<<f.n_peers, 128, 0, lc.stream>>>(ret, g, f, ws, E, k);
  ++*lc.launches;
  return cudaGetLastError();
}

cudaError_t launch_unpack(const LaunchCtx& lc, const WinGeom& g, const uint8_t* ret, int region,
                          int stage, void* out, int n, int row_bytes, int num_experts,
                          uint64_t expect_seq, int32_t* status, int64_t timeout_ns) {
  const int64_t nvec = (int64_t)n * row_bytes / 16;
  k_unpack<<<grid_for(nvec, kThreads * 4, lc.num_sms * 4), kThreads, 0, lc.stream>>>(
      ret, g, region, stage, reinterpret_cast<uint4*>(out), n, row_bytes, num_experts, expect_seq,
      status, timeout_ns);
  ++*lc.launches;
  return cudaGetLastError();
}

cudaError_t launch_transpose_wg(const LaunchCtx& lc, const float* Wg, float* WgT, int hidden,
                                int E) {
  k_transpose_wg<<<grid_for((int64_t)hidden * E, kThreads, 1024), kThreads, 0, lc.stream>>>(
      Wg, WgT, hidden, E);
  ++*lc.launches;
  return cudaGetLastError();
}
