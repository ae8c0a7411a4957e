// afd_attn.cu -- one Attention peer's side of token-level dispatch to several
// FFN ranks ([RFC]: Async GPU Connector, "Data flow" steps 1-4 and "Capacity
// and ring depth"), on the device:
//   send  -- the plan that segments the peer's top-k partials by destination
//            rank and groups them by local expert (one stable sort), the copy
//            of every routed row and every round-robin shared row into the
//            destination ranks' dispatch slots, then each rank's header and
//            flag (every rank gets its message, empty ones included);
//   recv  -- a bounded wait on the ranks that received rows (a rank sent
//            nothing is not waited for), then the weighted combine of the routed
//            outputs they returned plus the shared outputs, straight from
//            their return slots.
// The gate weights never leave the peer: the combine takes them from the
// caller.  The FFN ranks are afd_ctx contexts created with ffn_rank /
// ffn_size; they serve the rows with the grouped calls or the work-item loop.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <vector>

#include "afd_internal.cuh"

namespace {

constexpr int kThreads = 256;

struct AttnDst {        // one destination FFN rank
  uint8_t* win;         // its dispatch window
  const uint8_t* ret;   // its return window
  WinGeom g;            // their slot geometry (header length follows the rank's expert count)
  int first, count;     // its experts
};

struct AttnDsts {
  AttnDst d[AFD_MAX_FFN_RANKS];
  int F;
};

// per-stage plan of the last send, kept for the combine (the page's
// Attention-side pending FIFO)
struct AttnPlan {
  int32_t* dst;     // [token_cap * k] destination rank of partial t * k + j
  int32_t* pos;     // [token_cap * k] its row in the rank's segment
  int32_t* rows;    // [F] segment lengths
  int32_t* counts;  // [E] partials per (global) expert
  int32_t* seg;     // [F] first position of each rank's segment in the sorted order
};

__device__ __forceinline__ uint8_t* slot_of(uint8_t* win, const WinGeom& g, int region, int stage) {
  return win + g.flags_bytes + ((int64_t)region * g.ring_depth + stage) * g.slot_bytes;
}
__device__ __forceinline__ const uint8_t* slot_of(const uint8_t* win, const WinGeom& g, int region,
                                                  int stage) {
  return win + g.flags_bytes + ((int64_t)region * g.ring_depth + stage) * g.slot_bytes;
}

// ---------------------------------------------------------------------------
// send, step 1: one stable sort of the flattened ids, in three kernels over
// blocks of 16 tokens (16 * k consecutive partials).  k_attn_hist: a warp
// per block counts its partials per expert (hist[b][e]) and checks the ids.
// k_attn_scan (one CTA): per-expert totals and exclusive offsets (global
// expert order = destination order, then local expert order), each block's
// first position within each expert's run (base[b][e]), each rank's segment
// length; a segment over routed_cap raises AFD_ERR_CAPACITY, an id outside
// 0..E-1 AFD_ERR_ARG, and the later kernels write nothing.  k_attn_rank: a
// warp per block ranks its partials among the earlier ones of their expert
// (match_any over 32-element rounds, cursors from base) and records each
// partial's rank and row within that rank's segment.
// ---------------------------------------------------------------------------
constexpr int kBlkTok = 16;
constexpr int kPlanWarps = 8;

__global__ void __launch_bounds__(kPlanWarps * 32)
k_attn_hist(const int32_t* __restrict__ ids, int n, int k, int E, int32_t* __restrict__ hist,
            int32_t* status) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int hw[kPlanWarps][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kPlanWarps + warp;
  const int nb = (n + kBlkTok - 1) / kBlkTok;
  for (int e = lane; e < E; e += 32) hw[warp][e] = 0;
  __syncwarp();
  if (b >= nb || read_status(status)) return;
  const int f0 = b * kBlkTok * k, f1 = min(n * k, f0 + kBlkTok * k);
  bool bad = false;
  for (int fi = f0 + lane; fi < f1; fi += 32) {
    const int e = ids[fi];
    if (e < 0 || e >= E) {
      bad = true;
      continue;
    }
    atomicAdd(&hw[warp][e], 1);
  }
  if (bad) set_error(status, AFD_ERR_ARG);
  __syncwarp();
  for (int e = lane; e < E; e += 32) hist[(int64_t)b * E + e] = hw[warp][e];
}

constexpr int kScanSegs = 16;  // 16 segments of blocks x 64 experts per pass of 1024 threads

__global__ void __launch_bounds__(1024)
k_attn_scan(int n, int E, AttnDsts ds, AttnPlan pl, const int32_t* __restrict__ hist,
            int32_t* __restrict__ base, int64_t routed_cap, int32_t* status) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int cnt[256];
  __shared__ int offs[257];
  __shared__ int seg_sum[kScanSegs][64];
  __shared__ int skip;
  const int tid = threadIdx.x;
  if (tid == 0) skip = read_status(status);
  __syncthreads();
  if (skip) return;
  const int nb = (n + kBlkTok - 1) / kBlkTok;
  const int sg = tid / 64, el = tid % 64;
  const int L = (nb + kScanSegs - 1) / kScanSegs;
  const int b_lo = min(nb, sg * L), b_hi = min(nb, b_lo + L);
  for (int e0 = 0; e0 < E; e0 += 64) {
    const int e = e0 + el;
    int sum = 0;
    if (e < E)
      for (int b = b_lo; b < b_hi; b++) sum += hist[(int64_t)b * E + e];
    seg_sum[sg][el] = sum;
    __syncthreads();
    if (sg == 0 && e < E) {
      int tot = 0;
      for (int q = 0; q < kScanSegs; q++) tot += seg_sum[q][el];
      cnt[e] = tot;
    }
    __syncthreads();
  }
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < E; e++) { offs[e] = run; run += cnt[e]; }
    offs[E] = run;
    int over = 0;
    for (int r = 0; r < ds.F; r++) {
      const int R = offs[ds.d[r].first + ds.d[r].count] - offs[ds.d[r].first];
      pl.rows[r] = R;
      pl.seg[r] = offs[ds.d[r].first];
      over |= R > routed_cap;
    }
    if (over) set_error(status, AFD_ERR_CAPACITY);
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) pl.counts[e] = cnt[e];
  // each block's first position within each expert's run
  for (int e0 = 0; e0 < E; e0 += 64) {
    const int e = e0 + el;
    int sum = 0;
    if (e < E)
      for (int b = b_lo; b < b_hi; b++) sum += hist[(int64_t)b * E + e];
    seg_sum[sg][el] = sum;
    __syncthreads();
    if (e < E) {
      int run = offs[e];
      for (int q = 0; q < sg; q++) run += seg_sum[q][el];
      for (int b = b_lo; b < b_hi; b++) {
        base[(int64_t)b * E + e] = run;
        run += hist[(int64_t)b * E + e];
      }
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kPlanWarps * 32)
k_attn_rank(const int32_t* __restrict__ ids, int n, int k, int E, AttnDsts ds, AttnPlan pl,
            const int32_t* __restrict__ base, const int32_t* status) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int run_s[kPlanWarps][256];
  __shared__ int rank_of[256], seg_s[AFD_MAX_FFN_RANKS];
  for (int r = 0; r < ds.F; r++)
    for (int e = ds.d[r].first + threadIdx.x; e < ds.d[r].first + ds.d[r].count; e += blockDim.x)
      rank_of[e] = r;
  if (threadIdx.x < ds.F) seg_s[threadIdx.x] = pl.seg[threadIdx.x];
  __syncthreads();
  if (read_status(status)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kPlanWarps + warp;
  if (b >= (n + kBlkTok - 1) / kBlkTok) return;
  int* run = run_s[warp];
  for (int e = lane; e < E; e += 32) run[e] = base[(int64_t)b * E + e];
  __syncwarp();
  const int f0 = b * kBlkTok * k, f1 = min(n * k, f0 + kBlkTok * k);
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int g0 = f0; g0 < f1; g0 += 32) {
    const int fi = g0 + lane;
    const bool ok = fi < f1;
    const int e = ok ? ids[fi] : -1 - lane;
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & lt_mask);
    int p = 0;
    if (ok) p = run[e] + rank;
    __syncwarp();
    if (ok && rank == 0) run[e] += __popc(same);
    __syncwarp();
    if (ok) {
      const int r = rank_of[e];
      pl.dst[fi] = r;
      pl.pos[fi] = p - seg_s[r];
    }
  }
}

// ---------------------------------------------------------------------------
// send, step 3: a warp per row.  Routed row f (partial t * k + j) -> row
// pos[f] of its rank's routed_x, route_table entry = f; shared token t ->
// row t / F of rank t mod F's shared_x, shared_idx = t.  16-byte vectors.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
k_attn_copy(const uint4* __restrict__ x, int n, int k, int row_bytes, AttnDsts ds, AttnPlan pl,
            int region, int stage, int with_shared, const int32_t* status) {
  grid_dep_wait();
  grid_dep_launch();
  if (read_status(status)) return;
  const int N = n * k;
  const int rows = N + (with_shared ? n : 0);
  const int nvec = row_bytes / 16;
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    int d, q, t;
    int64_t field, table_field;
    if (r < N) {
      d = pl.dst[r];
      q = pl.pos[r];
      t = r / k;
      field = ds.d[d].g.routed_x;
      table_field = ds.d[d].g.route_table;
    } else {
      t = r - N;
      d = t % ds.F;
      q = t / ds.F;
      field = ds.d[d].g.shared_x;
      table_field = ds.d[d].g.shared_idx;
    }
    uint8_t* slot = slot_of(ds.d[d].win, ds.d[d].g, region, stage);
    uint4* dst = reinterpret_cast<uint4*>(slot + field + (int64_t)q * row_bytes);
    const uint4* src = x + (int64_t)t * nvec;
    for (int v = lane; v < nvec; v += 32) dst[v] = __ldg(src + v);
    if (lane == 0) reinterpret_cast<int32_t*>(slot + table_field)[q] = r < N ? r : t;
  }
}

// send, headers: CTA per rank; header then the flag = seq (release)
__global__ void k_attn_headers(AttnDsts ds, AttnPlan pl, int region, int stage, int layer, int n,
                               int with_shared, uint64_t seq, const int32_t* status) {
  grid_dep_wait();
  grid_dep_launch();
  if (read_status(status)) return;
  const int d = blockIdx.x;
  if (d >= ds.F) return;
  const AttnDst& D = ds.d[d];
  uint8_t* slot = slot_of(D.win, D.g, region, stage);
  int32_t* h = reinterpret_cast<int32_t*>(slot + D.g.header);
  const int ns = with_shared ? rr_rows(n, d, ds.F) : 0;
  for (int w = threadIdx.x; w < AFD_HEADER_FIXED_WORDS + D.count; w += blockDim.x) {
    int32_t v;
    switch (w) {
      case 0: v = (int32_t)AFD_HEADER_MAGIC; break;
      case 1: v = AFD_HEADER_VERSION; break;
      case 2: v = 0; break;
      case 3: v = (int32_t)(uint32_t)seq; break;
      case 4: v = (int32_t)(uint32_t)seq; break;
      case 5: v = layer; break;
      case 6: v = stage; break;
      case 7: v = n; break;
      case 8: v = pl.rows[d]; break;
      case 9: v = ns; break;
      case 10: v = D.count; break;
      case 11: v = AFD_HEADER_FIXED_WORDS + D.count; break;
      default: v = pl.counts[D.first + (w - AFD_HEADER_FIXED_WORDS)];
    }
    h[w] = v;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    st_release_u64(reinterpret_cast<uint64_t*>(D.win) + (int64_t)region * D.g.ring_depth + stage, seq);
  }
}

// ---------------------------------------------------------------------------
// recv: thread d waits (bounded) for rank d's return flag to reach
// expect_seq when the rank got rows, then checks magic, version, the echoed
// seq and the row counts.  First failing rank's code wins.
// ---------------------------------------------------------------------------
__global__ void k_attn_wait(AttnDsts ds, AttnPlan pl, int region, int stage, int n,
                            int with_shared, uint64_t expect_seq, int32_t* status,
                            int64_t timeout_ns) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int err[AFD_MAX_FFN_RANKS];
  const int d = threadIdx.x;
  if (d < AFD_MAX_FFN_RANKS) err[d] = 0;
  __syncthreads();
  if (read_status(status)) return;
  if (d < ds.F) {
    const AttnDst& D = ds.d[d];
    const int R = pl.rows[d];
    const int ns = with_shared ? rr_rows(n, d, ds.F) : 0;
    int e = 0;
    if (R || ns) {
      const uint64_t* flagp = reinterpret_cast<const uint64_t*>(D.ret) +
                              (int64_t)region * D.g.ring_depth + stage;
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
        const int32_t* h = reinterpret_cast<const int32_t*>(slot_of(D.ret, D.g, region, stage) + D.g.header);
        int32_t w[10];
#pragma unroll
        for (int q = 0; q < 10; q++)
          asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(w[q]) : "l"(h + q) : "memory");
        if ((uint32_t)w[0] != (uint32_t)AFD_HEADER_MAGIC || w[1] != AFD_HEADER_VERSION)
          e = AFD_ERR_HEADER;
        else if ((uint32_t)w[4] != (uint32_t)expect_seq)
          e = AFD_ERR_SEQ;
        else if (w[7] != n || w[8] != R || w[9] != ns)
          e = AFD_ERR_SHAPE;
      }
    }
    err[d] = e;
  }
  __syncthreads();
  if (threadIdx.x == 0)
    for (int q = 0; q < ds.F; q++)
      if (err[q]) {
        set_error(status, err[q]);
        break;
      }
}

// recv, combine: work item = (token, block of 256 features), a warp per item;
// out[t] = sum over j ascending of w[t, j] * y(rank dst, row pos) + s(row
// t / F of rank t mod F), fp32, rounded once to the activation type.  Lane
// j < k finds its partial's row once per item; the rows are then read in
// rounds of kBatch (all loads of a round before its multiply-adds, which
// stay in ascending j): 1 keeps the registers low and the SM full for
// large fan-ins, 8 keeps loads in flight when few warps have work.
template <bool ACT_F32, int kBatch>
__global__ void __launch_bounds__(kThreads)
k_attn_combine(AttnDsts ds, AttnPlan pl, int region, int stage, int n, int k, int hidden,
               const float* __restrict__ wts, uint8_t* out, int with_shared, const int32_t* status) {
  grid_dep_wait();
  grid_dep_launch();
  if (read_status(status)) return;
  constexpr int kVec = 8;  // features per lane step
  constexpr int kEl = ACT_F32 ? 4 : 2;
  constexpr int kWords = ACT_F32 ? 2 : 1;  // 16-byte loads per lane and row
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int nfb = (hidden + 32 * kVec - 1) / (32 * kVec);
  const int64_t items = (int64_t)n * nfb;
  const int64_t row_bytes = (int64_t)hidden * kEl;
  for (int64_t it = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items; it += warps) {
    const int t = (int)(it / nfb), fb = (int)(it % nfb);
    const int c0 = fb * 32 * kVec + lane * kVec;
    const bool valid = c0 < hidden;
    const int64_t cb = (int64_t)(valid ? c0 : 0) * kEl;
    const uint8_t* my_row = nullptr;
    float my_w = 0.0f;
    if (lane < k) {
      const int d = pl.dst[(int64_t)t * k + lane];
      my_row = slot_of(ds.d[d].ret, ds.d[d].g, region, stage) + ds.d[d].g.routed_x +
               (int64_t)pl.pos[(int64_t)t * k + lane] * row_bytes;
      my_w = wts[(int64_t)t * k + lane];
    }
    float acc[kVec];
#pragma unroll
    for (int v = 0; v < kVec; v++) acc[v] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += kBatch) {
      uint4 raw[kBatch][kWords];
      float wj[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; u++) {
        const int j = (j0 + u) & 31;
        const uint8_t* row = reinterpret_cast<const uint8_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(my_row), j));
        wj[u] = __shfl_sync(0xffffffffu, my_w, j);
        const bool ld = valid && j0 + u < k;
#pragma unroll
        for (int q = 0; q < kWords; q++)
          raw[u][q] = ld ? reinterpret_cast<const uint4*>(row + cb)[q] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kBatch; u++) {
        if (j0 + u >= k) break;
        float y[kVec];
        if constexpr (ACT_F32) {
          y[0] = __uint_as_float(raw[u][0].x); y[1] = __uint_as_float(raw[u][0].y);
          y[2] = __uint_as_float(raw[u][0].z); y[3] = __uint_as_float(raw[u][0].w);
          y[4] = __uint_as_float(raw[u][kWords - 1].x); y[5] = __uint_as_float(raw[u][kWords - 1].y);
          y[6] = __uint_as_float(raw[u][kWords - 1].z); y[7] = __uint_as_float(raw[u][kWords - 1].w);
        } else {
          const uint32_t p[4] = {raw[u][0].x, raw[u][0].y, raw[u][0].z, raw[u][0].w};
#pragma unroll
          for (int v = 0; v < 4; v++) {
            y[2 * v] = __uint_as_float(p[v] << 16);
            y[2 * v + 1] = __uint_as_float(p[v] & 0xffff0000u);
          }
        }
#pragma unroll
        for (int v = 0; v < kVec; v++) acc[v] = __fmaf_rn(wj[u], y[v], acc[v]);
      }
    }
    if (!valid) continue;
    if (with_shared) {
      const int d = t % ds.F;
      const uint8_t* row = slot_of(ds.d[d].ret, ds.d[d].g, region, stage) + ds.d[d].g.shared_x +
                           (int64_t)(t / ds.F) * row_bytes + cb;
      float y[kVec];
      if constexpr (ACT_F32) {
        const float4 a = *reinterpret_cast<const float4*>(row);
        const float4 b = *reinterpret_cast<const float4*>(row + 16);
        y[0] = a.x; y[1] = a.y; y[2] = a.z; y[3] = a.w;
        y[4] = b.x; y[5] = b.y; y[6] = b.z; y[7] = b.w;
      } else {
        const uint4 u = *reinterpret_cast<const uint4*>(row);
        const uint32_t p[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int v = 0; v < 4; v++) {
          y[2 * v] = __uint_as_float(p[v] << 16);
          y[2 * v + 1] = __uint_as_float(p[v] & 0xffff0000u);
        }
      }
#pragma unroll
      for (int v = 0; v < kVec; v++) acc[v] = __fadd_rn(acc[v], y[v]);
    }
    uint8_t* o = out + (int64_t)t * row_bytes + cb;
    if constexpr (ACT_F32) {
      reinterpret_cast<float4*>(o)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      reinterpret_cast<float4*>(o)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      uint32_t p[4];
#pragma unroll
      for (int v = 0; v < 4; v++) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * v], acc[2 * v + 1]);
        p[v] = *reinterpret_cast<uint32_t*>(&b2);
      }
      *reinterpret_cast<uint4*>(o) = make_uint4(p[0], p[1], p[2], p[3]);
    }
  }
}

int grid_rows(int64_t work, int per_block, int cap) {
  int64_t g = (work + per_block - 1) / per_block;
  return (int)std::max<int64_t>(1, std::min<int64_t>(g, cap));
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
struct afd_attn {
  int F = 0, peer = 0, E = 0, k = 0, token_cap = 0, ring = 0, hidden = 0, act_f32 = 0;
  int has_shared = 0;
  int64_t routed_cap = 0, timeout_ns = 0;
  int num_sms = 0, pdl = 1;
  cudaStream_t stream = nullptr;
  AttnDsts ds;
  uint8_t* mem = nullptr;
  int32_t* status = nullptr;
  int32_t* hist = nullptr;   // [token_cap / 16][E] per-block expert counts of a send
  int32_t* base = nullptr;   // [token_cap / 16][E] their first positions
  std::vector<AttnPlan> plans;   // one per stage
  std::vector<int> last_n;       // tokens of each stage's last send
  std::vector<int> last_shared;  // whether it carried shared rows
  int64_t launches = 0;
  LaunchCtx lc() { return LaunchCtx{stream, num_sms, &launches, pdl}; }
};

static int attn_fail(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return AFD_OK;
  fprintf(stderr, "afd: %s: %s\n", what, cudaGetErrorString(e));
  cudaGetLastError();
  return AFD_ERR_CUDA;
}

static bool is_device_ptr(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

int afd_expert_range(int num_experts, int ffn_size, int ffn_rank, int* first, int* count) {
  if (!first || !count || ffn_size < 1 || num_experts < ffn_size || ffn_rank < 0 ||
      ffn_rank >= ffn_size)
    return AFD_ERR_ARG;
  const int base = num_experts / ffn_size, rem = num_experts % ffn_size;
  *count = base + (ffn_rank < rem ? 1 : 0);
  *first = ffn_rank * base + std::min(ffn_rank, rem);
  return AFD_OK;
}

int afd_attn_create(afd_ctx* const* ranks, int ffn_size, int peer, int num_experts,
                    void* cuda_stream, afd_attn** out) {
  if (!out) return AFD_ERR_ARG;
  *out = nullptr;
  if (!ranks || ffn_size < 1 || ffn_size > AFD_MAX_FFN_RANKS || num_experts < ffn_size ||
      num_experts > 256)
    return AFD_ERR_ARG;
  afd_config c0;
  if (!ranks[0] || afd_get_config(ranks[0], &c0)) return AFD_ERR_ARG;
  if (peer < 0 || peer >= c0.num_peers) return AFD_ERR_ARG;
  afd_attn* a = new afd_attn();
  a->F = ffn_size;
  a->peer = peer;
  a->E = num_experts;
  a->k = c0.topk;
  a->token_cap = c0.token_cap;
  a->ring = c0.ring_depth;
  a->hidden = c0.hidden;
  a->act_f32 = c0.act_dtype == AFD_DTYPE_F32;
  a->has_shared = c0.shared_inter > 0;
  a->timeout_ns = c0.wait_timeout_ns ? c0.wait_timeout_ns : 1000000000ll;
  a->pdl = (c0.flags & AFD_CFG_NO_PDL) ? 0 : 1;
  a->stream = reinterpret_cast<cudaStream_t>(cuda_stream);
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&a->num_sms, cudaDevAttrMultiProcessorCount, dev);
  memset(&a->ds, 0, sizeof a->ds);
  a->ds.F = ffn_size;
  for (int r = 0; r < ffn_size; r++) {
    afd_config c;
    int first = 0, count = 0;
    afd_expert_range(num_experts, ffn_size, r, &first, &count);
    // every rank: the same peers, stages and shapes, its own rank and experts
    if (!ranks[r] || afd_get_config(ranks[r], &c) || c.ffn_size != ffn_size || c.ffn_rank != r ||
        c.num_experts != count || c.num_peers != c0.num_peers || c.ring_depth != c0.ring_depth ||
        c.token_cap != c0.token_cap || c.hidden != c0.hidden || c.topk != c0.topk ||
        c.act_dtype != c0.act_dtype || c.shared_inter != c0.shared_inter ||
        c.routed_cap_multiplier != c0.routed_cap_multiplier) {
      delete a;
      return AFD_ERR_ARG;
    }
    afd_layout L;
    void* win = nullptr;
    void* ret = nullptr;
    int64_t bytes = 0;
    if (afd_slot_layout(&c, &L) || afd_get_window(ranks[r], AFD_DIR_DISPATCH, &win, &bytes) ||
        afd_get_window(ranks[r], AFD_DIR_RETURN, &ret, &bytes)) {
      delete a;
      return AFD_ERR_ARG;
    }
    AttnDst& D = a->ds.d[r];
    D.win = static_cast<uint8_t*>(win);
    D.ret = static_cast<const uint8_t*>(ret);
    D.g = WinGeom{L.flags_bytes, L.slot_bytes, L.header, L.route_table, L.routed_x, L.shared_idx,
                  L.shared_x, c.ring_depth, c.num_peers};
    D.first = first;
    D.count = count;
  }
  {
    const int64_t even = ((int64_t)c0.token_cap * c0.topk + ffn_size - 1) / ffn_size;
    a->routed_cap = (int64_t)std::ceil((double)even * (double)c0.routed_cap_multiplier);
  }
  // scratch: status, the sort's per-block histograms and bases, then per
  // stage dst / pos [token_cap * k], rows [F], counts [E], segment starts [F]
  const int64_t nk = (int64_t)a->token_cap * a->k;
  const int64_t nb = (a->token_cap + kBlkTok - 1) / kBlkTok;
  const int64_t hist_bytes = ((nb * num_experts * 4 + 255) / 256) * 256;
  const int64_t per_stage = (2 * nk + 2 * AFD_MAX_FFN_RANKS + 256) * 4;
  const int64_t total = 256 + 2 * hist_bytes + per_stage * a->ring;
  if (attn_fail(cudaMalloc(&a->mem, total), "attention-side scratch") ||
      attn_fail(cudaMemset(a->mem, 0, total), "attention-side scratch")) {
    cudaFree(a->mem);
    delete a;
    return AFD_ERR_CUDA;
  }
  a->status = reinterpret_cast<int32_t*>(a->mem);
  a->hist = reinterpret_cast<int32_t*>(a->mem + 256);
  a->base = reinterpret_cast<int32_t*>(a->mem + 256 + hist_bytes);
  for (int s = 0; s < a->ring; s++) {
    int32_t* b = reinterpret_cast<int32_t*>(a->mem + 256 + 2 * hist_bytes + per_stage * s);
    a->plans.push_back(AttnPlan{b, b + nk, b + 2 * nk, b + 2 * nk + AFD_MAX_FFN_RANKS,
                                b + 2 * nk + AFD_MAX_FFN_RANKS + 256});
  }
  a->last_n.assign(a->ring, -1);
  a->last_shared.assign(a->ring, 0);
  *out = a;
  return AFD_OK;
}

void afd_attn_destroy(afd_attn* a) {
  if (!a) return;
  if (a->stream) cudaStreamSynchronize(a->stream);
  cudaFree(a->mem);
  delete a;
}

int afd_attn_dispatch(afd_attn* a, int stage, int layer, const void* x, int n_tokens,
                      const int32_t* topk_ids, int with_shared, uint64_t seq) {
  if (!a || stage < 0 || stage >= a->ring || n_tokens < 0) return AFD_ERR_ARG;
  if (with_shared && !a->has_shared) return AFD_ERR_ARG;
  if (n_tokens > a->token_cap) return AFD_ERR_CAPACITY;
  if (n_tokens > 0) {
    if (!x || !topk_ids || !is_device_ptr(x) || !is_device_ptr(topk_ids)) return AFD_ERR_NOT_DEVICE;
    if (reinterpret_cast<uintptr_t>(x) & 15) return AFD_ERR_ARG;
  }
  const AttnPlan& pl = a->plans[stage];
  LaunchCtx lc = a->lc();
  const int row_bytes = a->hidden * (a->act_f32 ? 4 : 2);
  const int nb = (n_tokens + kBlkTok - 1) / kBlkTok;
  const int plan_grid = (nb + kPlanWarps - 1) / kPlanWarps;
  int rc = AFD_OK;
  if (nb)
    rc = attn_fail(launch_k(lc, k_attn_hist, plan_grid, kPlanWarps * 32, 0, topk_ids, n_tokens,
                            a->k, a->E, a->hist, a->status),
                   "dispatch histograms");
  if (!rc)
    rc = attn_fail(launch_k(lc, k_attn_scan, 1, 1024, 0, n_tokens, a->E, a->ds, pl,
                            (const int32_t*)a->hist, a->base, a->routed_cap, a->status),
                   "dispatch scan");
  if (!rc && nb)
    rc = attn_fail(launch_k(lc, k_attn_rank, plan_grid, kPlanWarps * 32, 0, topk_ids, n_tokens,
                            a->k, a->E, a->ds, pl, (const int32_t*)a->base,
                            (const int32_t*)a->status),
                   "dispatch rank");
  const int64_t rows = (int64_t)n_tokens * a->k + (with_shared ? n_tokens : 0);
  if (!rc && rows > 0)
    rc = attn_fail(launch_k(lc, k_attn_copy, grid_rows(rows, kThreads / 32, a->num_sms * 8), kThreads,
                            0, reinterpret_cast<const uint4*>(x), n_tokens, a->k, row_bytes, a->ds,
                            pl, a->peer, stage, with_shared, (const int32_t*)a->status),
                   "dispatch copy");
  if (!rc)
    rc = attn_fail(launch_k(lc, k_attn_headers, a->F, 128, 0, a->ds, pl, a->peer, stage, layer,
                            n_tokens, with_shared, seq, (const int32_t*)a->status),
                   "dispatch headers");
  if (!rc) {
    a->last_n[stage] = n_tokens;
    a->last_shared[stage] = with_shared ? 1 : 0;
  }
  return rc;
}

int afd_attn_combine(afd_attn* a, int stage, const float* topk_weights, void* out, int n_tokens,
                     uint64_t expect_seq) {
  if (!a || stage < 0 || stage >= a->ring || n_tokens < 0) return AFD_ERR_ARG;
  if (n_tokens != a->last_n[stage]) return AFD_ERR_SHAPE;
  if (n_tokens > 0) {
    if (!out || !topk_weights || !is_device_ptr(out) || !is_device_ptr(topk_weights))
      return AFD_ERR_NOT_DEVICE;
    if (reinterpret_cast<uintptr_t>(out) & 15) return AFD_ERR_ARG;
  }
  const AttnPlan& pl = a->plans[stage];
  LaunchCtx lc = a->lc();
  const int ws = a->last_shared[stage];
  int rc = attn_fail(launch_k(lc, k_attn_wait, 1, 32, 0, a->ds, pl, a->peer, stage, n_tokens, ws,
                              expect_seq, a->status, a->timeout_ns),
                     "combine wait");
  if (rc || n_tokens == 0) return rc;
  const int64_t items = (int64_t)n_tokens * ((a->hidden + 255) / 256);
  const int grid = grid_rows(items, kThreads / 32, a->num_sms * 8);
  const bool small = items < (int64_t)a->num_sms * 64;
  auto kern = a->act_f32 ? (small ? k_attn_combine<true, 8> : k_attn_combine<true, 1>)
                         : (small ? k_attn_combine<false, 8> : k_attn_combine<false, 1>);
  return attn_fail(launch_k(lc, kern, grid, kThreads, 0, a->ds, pl, a->peer, stage, n_tokens, a->k,
                            a->hidden, topk_weights, static_cast<uint8_t*>(out), ws,
                            (const int32_t*)a->status),
                   "combine");
}

int afd_attn_rows(afd_attn* a, int stage, int* rows) {
  if (!a || !rows || stage < 0 || stage >= a->ring) return AFD_ERR_ARG;
  if (attn_fail(cudaStreamSynchronize(a->stream), "stream sync")) return AFD_ERR_CUDA;
  int32_t r[AFD_MAX_FFN_RANKS];
  if (attn_fail(cudaMemcpy(r, a->plans[stage].rows, sizeof(int32_t) * a->F, cudaMemcpyDeviceToHost),
                "rows read"))
    return AFD_ERR_CUDA;
  for (int q = 0; q < a->F; q++) rows[q] = r[q];
  return AFD_OK;
}

int afd_attn_poll_status(afd_attn* a) {
  if (!a) return AFD_ERR_ARG;
  if (attn_fail(cudaStreamSynchronize(a->stream), "stream sync")) return AFD_ERR_CUDA;
  int32_t st = 0;
  if (attn_fail(cudaMemcpy(&st, a->status, 4, cudaMemcpyDeviceToHost), "status read"))
    return AFD_ERR_CUDA;
  if (st && attn_fail(cudaMemset(a->status, 0, 4), "status clear")) return AFD_ERR_CUDA;
  return st;
}

int64_t afd_attn_launch_count(afd_attn* a) { return a ? a->launches : 0; }
