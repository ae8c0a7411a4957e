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
constexpr int kPlanThreads = 1024;

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
};

__device__ __forceinline__ uint8_t* slot_of(uint8_t* win, const WinGeom& g, int region, int stage) {
  return win + g.flags_bytes + ((int64_t)region * g.ring_depth + stage) * g.slot_bytes;
}
__device__ __forceinline__ const uint8_t* slot_of(const uint8_t* win, const WinGeom& g, int region,
                                                  int stage) {
  return win + g.flags_bytes + ((int64_t)region * g.ring_depth + stage) * g.slot_bytes;
}

// ---------------------------------------------------------------------------
// send, step 1 (one CTA): bincount of the flattened ids, exclusive offsets
// (global expert order = destination order, then local expert order), the
// stable rank of every partial among the earlier partials of its expert
// (warp w owns a contiguous chunk of the partials; per-warp histograms give
// its cursors; 32-element rounds ranked with match_any), each rank's
// segment length.  A segment over routed_cap raises AFD_ERR_CAPACITY, an id
// outside 0..E-1 AFD_ERR_ARG; the later kernels then write nothing.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPlanThreads)
k_attn_plan(const int32_t* __restrict__ ids, int n, int k, int E, AttnDsts ds, AttnPlan pl,
            int64_t routed_cap, int32_t* status) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int hist_w[32][256];
  __shared__ int cnt[256];
  __shared__ int offs[257];
  __shared__ int rank_of[256];
  __shared__ int bad;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 32 * 256; i += blockDim.x) (&hist_w[0][0])[i] = 0;
  if (tid == 0) bad = read_status(status);
  for (int r = 0; r < ds.F; r++)
    for (int e = ds.d[r].first + tid; e < ds.d[r].first + ds.d[r].count; e += blockDim.x)
      rank_of[e] = r;
  __syncthreads();
  if (bad) return;
  const int N = n * k;
  const int chunk = (N + 31) / 32;
  const int c0 = min(N, warp * chunk), c1 = min(N, c0 + chunk);
  for (int fi = c0 + lane; fi < c1; fi += 32) {
    const int e = ids[fi];
    if (e < 0 || e >= E) {
      bad = 1;
      continue;
    }
    atomicAdd(&hist_w[warp][e], 1);
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) set_error(status, AFD_ERR_ARG);
    return;
  }
  for (int e = tid; e < E; e += blockDim.x) {
    int c = 0;
    for (int w = 0; w < 32; w++) c += hist_w[w][e];
    cnt[e] = c;
  }
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < E; e++) { offs[e] = run; run += cnt[e]; }
    offs[E] = run;
    for (int r = 0; r < ds.F; r++) {
      const int R = offs[ds.d[r].first + ds.d[r].count] - offs[ds.d[r].first];
      pl.rows[r] = R;
      if (R > routed_cap) bad = 1;
    }
    if (bad) set_error(status, AFD_ERR_CAPACITY);
  }
  __syncthreads();
  if (bad) return;
  for (int e = tid; e < E; e += blockDim.x) {
    pl.counts[e] = cnt[e];
    int base = offs[e];
    for (int w = 0; w < 32; w++) {
      const int c = hist_w[w][e];
      hist_w[w][e] = base;  // warp w's cursor for expert e
      base += c;
    }
  }
  __syncthreads();
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int g0 = c0; g0 < c1; g0 += 32) {
    const int fi = g0 + lane;
    const bool ok = fi < c1;
    const int e = ok ? ids[fi] : -1 - lane;
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & lt_mask);
    int p = 0;
    if (ok) p = hist_w[warp][e] + rank;
    __syncwarp();
    if (ok && rank == 0) hist_w[warp][e] += __popc(same);
    __syncwarp();
    if (ok) {
      const int r = rank_of[e];
      pl.dst[fi] = r;
      pl.pos[fi] = p - offs[ds.d[r].first];
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
// t / F of rank t mod F), fp32, rounded once to the activation type.
template <bool ACT_F32>
__global__ void __launch_bounds__(kThreads)
k_attn_combine(AttnDsts ds, AttnPlan pl, int region, int stage, int n, int k, int hidden,
               const float* __restrict__ wts, uint8_t* out, int with_shared, const int32_t* status) {
  grid_dep_wait();
  grid_dep_launch();
  if (read_status(status)) return;
  constexpr int kVec = 8;  // features per lane step
  constexpr int kEl = ACT_F32 ? 4 : 2;
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int nfb = (hidden + 32 * kVec - 1) / (32 * kVec);
  const int64_t items = (int64_t)n * nfb;
  const int64_t row_bytes = (int64_t)hidden * kEl;
  for (int64_t it = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items; it += warps) {
    const int t = (int)(it / nfb), fb = (int)(it % nfb);
    const int c = fb * 32 * kVec + lane * kVec;
    int my_d = 0, my_q = 0;
    float my_w = 0.0f;
    if (lane < k) {
      my_d = pl.dst[(int64_t)t * k + lane];
      my_q = pl.pos[(int64_t)t * k + lane];
      my_w = wts[(int64_t)t * k + lane];
    }
    float acc[kVec];
#pragma unroll
    for (int v = 0; v < kVec; v++) acc[v] = 0.0f;
    for (int j = 0; j < k; j++) {
      const int d = __shfl_sync(0xffffffffu, my_d, j);
      const int q = __shfl_sync(0xffffffffu, my_q, j);
      const float wj = __shfl_sync(0xffffffffu, my_w, j);
      if (c >= hidden) continue;
      const uint8_t* row = slot_of(ds.d[d].ret, ds.d[d].g, region, stage) + ds.d[d].g.routed_x +
                           (int64_t)q * row_bytes + (int64_t)c * kEl;
      if constexpr (ACT_F32) {
        const float4 a = *reinterpret_cast<const float4*>(row);
        const float4 b = *reinterpret_cast<const float4*>(row + 16);
        const float y[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int v = 0; v < kVec; v++) acc[v] = __fmaf_rn(wj, y[v], acc[v]);
      } else {
        const uint4 u = *reinterpret_cast<const uint4*>(row);
        const uint32_t p[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int v = 0; v < 4; v++) {
          acc[2 * v] = __fmaf_rn(wj, __uint_as_float(p[v] << 16), acc[2 * v]);
          acc[2 * v + 1] = __fmaf_rn(wj, __uint_as_float(p[v] & 0xffff0000u), acc[2 * v + 1]);
        }
      }
    }
    if (c >= hidden) continue;
    if (with_shared) {
      const int d = t % ds.F;
      const uint8_t* row = slot_of(ds.d[d].ret, ds.d[d].g, region, stage) + ds.d[d].g.shared_x +
                           (int64_t)(t / ds.F) * row_bytes + (int64_t)c * kEl;
      if constexpr (ACT_F32) {
        const float4 a = *reinterpret_cast<const float4*>(row);
        const float4 b = *reinterpret_cast<const float4*>(row + 16);
        const float y[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int v = 0; v < kVec; v++) acc[v] = __fadd_rn(acc[v], y[v]);
      } else {
        const uint4 u = *reinterpret_cast<const uint4*>(row);
        const uint32_t p[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int v = 0; v < 4; v++) {
          acc[2 * v] = __fadd_rn(acc[2 * v], __uint_as_float(p[v] << 16));
          acc[2 * v + 1] = __fadd_rn(acc[2 * v + 1], __uint_as_float(p[v] & 0xffff0000u));
        }
      }
    }
    uint8_t* o = out + (int64_t)t * row_bytes + (int64_t)c * kEl;
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
  // scratch: status, then per stage dst / pos [token_cap * k], rows [F], counts [E]
  const int64_t nk = (int64_t)a->token_cap * a->k;
  const int64_t per_stage = (2 * nk + AFD_MAX_FFN_RANKS + 256) * 4;
  const int64_t total = 256 + per_stage * a->ring;
  if (attn_fail(cudaMalloc(&a->mem, total), "attention-side scratch") ||
      attn_fail(cudaMemset(a->mem, 0, total), "attention-side scratch")) {
    cudaFree(a->mem);
    delete a;
    return AFD_ERR_CUDA;
  }
  a->status = reinterpret_cast<int32_t*>(a->mem);
  for (int s = 0; s < a->ring; s++) {
    int32_t* b = reinterpret_cast<int32_t*>(a->mem + 256 + per_stage * s);
    a->plans.push_back(AttnPlan{b, b + nk, b + 2 * nk, b + 2 * nk + AFD_MAX_FFN_RANKS});
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
  int rc = attn_fail(launch_k(lc, k_attn_plan, 1, kPlanThreads, 0, topk_ids, n_tokens, a->k, a->E,
                              a->ds, pl, a->routed_cap, a->status),
                     "dispatch plan");
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
  auto kern = a->act_f32 ? k_attn_combine<true> : k_attn_combine<false>;
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
