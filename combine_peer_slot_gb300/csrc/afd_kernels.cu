// afd_kernels.cu -- the memory-bound and control kernels of the AFD FFN-side
// step on sm_103a: slot pack / header / flag, header check with a bounded
// flag wait, router, dispatch plan, permute-gather, combine + split, return
// header + flag, unpack, and the SIMT GEMM used for fp32 activations.
#include <algorithm>

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

// row r of a slot field as a row of the window seen as a [rows, hidden]
// matrix (every field starts on a whole row)
__device__ __forceinline__ int32_t window_row(const WinGeom& g, int region, int stage, int64_t field,
                                              int r, int row_bytes) {
  return (int32_t)((g.flags_bytes + ((int64_t)region * g.ring_depth + stage) * g.slot_bytes + field) /
                   row_bytes) + r;
}

// list entry i holding shared row r of the concatenation of the entries'
// shared rows
__device__ __forceinline__ int entry_of_shared(const FanIn& f, int r) {
  int lo = 0, hi = f.n_peers - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (f.sprefix[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// grouped form: list entry i holding routed row r of the concatenation
__device__ __forceinline__ int entry_of_rows(const FanIn& f, int r) {
  int lo = 0, hi = f.n_peers - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (f.rprefix[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The fan-in of the step: the kernel argument for a host-described step
// (kDev false), else the one the work-item head built in the workspace,
// copied into shared memory by the whole CTA (every thread must call this,
// before any early return) so that the per-row peer lookups stay on chip.
template <bool kDev>
__device__ __forceinline__ const FanIn& step_item(const FanIn& fp, const FanIn* g) {
  if constexpr (kDev) {
    __shared__ FanIn s;
    constexpr int kWords = (int)(sizeof(FanIn) / 4);
    for (int i = threadIdx.x; i < kWords; i += blockDim.x)
      reinterpret_cast<int32_t*>(&s)[i] = reinterpret_cast<const int32_t*>(g)[i];
    __syncthreads();
    return s;
  } else {
    return fp;
  }
}

// The return header of list entry i (every word but the flag): magic,
// version, the dispatch seq echoed, layer, stage, counts and the entry's
// per-expert partial counts; the threads of a CTA share the words.
__device__ void write_return_header(uint8_t* ret, const WinGeom& g, const FanIn& f, const DevWS& ws,
                                    int E, int k, int i) {
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
      case 8: v = f.grouped ? f.rprefix[i + 1] - f.rprefix[i] : n * k; break;
      case 9: v = ws.peer_shared[i] ? f.sprefix[i + 1] - f.sprefix[i] : 0; break;
      case 10: v = E; break;
      case 11: v = AFD_HEADER_FIXED_WORDS + E; break;
      default: v = ws.peer_counts[i * E + (w - AFD_HEADER_FIXED_WORDS)];
    }
    h[w] = v;
  }
}

__device__ __forceinline__ uint64_t* return_flag(uint8_t* ret, const WinGeom& g, const FanIn& f, int i) {
  return reinterpret_cast<uint64_t*>(ret) + f.region[i] * g.ring_depth + f.stage;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}

// ---------------------------------------------------------------------------
// pack: payload, then header + flag (Async GPU Connector, "Window and slot
// layout": the flag is written after the payload, on the same stream)
// ---------------------------------------------------------------------------
__global__ void k_pack_payload(uint8_t* win, WinGeom g, int region, int stage,
                               const uint4* __restrict__ rows, int n_rows,
                               const uint4* __restrict__ xs, int n_shared, int row_bytes) {
  grid_dep_wait();
  grid_dep_launch();
  uint8_t* slot = slot_ptr(win, g, region, stage);
  uint4* rx = reinterpret_cast<uint4*>(slot + g.routed_x);
  uint4* sx = reinterpret_cast<uint4*>(slot + g.shared_x);
  int32_t* sidx = reinterpret_cast<int32_t*>(slot + g.shared_idx);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nvec = (int64_t)n_rows * row_bytes / 16;
  for (int64_t i = i0; i < nvec; i += stride) rx[i] = rows[i];
  if (xs) {
    const int64_t svec = (int64_t)n_shared * row_bytes / 16;
    for (int64_t i = i0; i < svec; i += stride) sx[i] = xs[i];
    for (int64_t i = i0; i < n_shared; i += stride) sidx[i] = (int32_t)i;
  }
}

// the header of slot (region, stage), then (after the CTA's stores) its
// flag = seq; one CTA
__device__ void write_dispatch_header(uint8_t* win, const WinGeom& g, int region, int stage, int layer, int n,
                                      int with_shared, int num_experts, uint64_t seq, int shutdown,
                                      int routed_tokens, const GroupList* gl) {
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
      case 8: v = routed_tokens; break;
      case 9: v = with_shared ? n : 0; break;
      case 10: v = num_experts; break;
      case 11: v = AFD_HEADER_FIXED_WORDS + num_experts; break;
      default: v = gl ? gl->n[i - AFD_HEADER_FIXED_WORDS] : 0;
    }
    h[i] = v;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    uint64_t* flag = reinterpret_cast<uint64_t*>(win) + (int64_t)region * g.ring_depth + stage;
    st_release_u64(flag, seq);
  }
}

__global__ void k_pack_header(uint8_t* win, WinGeom g, int region, int stage, int layer, int n,
                              int with_shared, int num_experts, uint64_t seq, int shutdown,
                              int routed_tokens, const __grid_constant__ GroupList gl) {
  grid_dep_wait();
  grid_dep_launch();
  write_dispatch_header(win, g, region, stage, layer, n, with_shared, num_experts, seq, shutdown,
                        routed_tokens, &gl);
}

// Several peers' packs (afd_pack_slots): CTA row y = entry y of the list,
// its CTAs striding over that peer's vectors; then a CTA per entry writes
// its header and releases its flag.
__global__ void k_pack_payload_multi(uint8_t* win, WinGeom g, int stage, const __grid_constant__ PackList pl,
                                     int with_shared, int row_bytes) {
  grid_dep_wait();
  grid_dep_launch();
  const int e = blockIdx.y;
  if (e >= pl.n) return;
  uint8_t* slot = slot_ptr(win, g, pl.region[e], stage);
  uint4* rx = reinterpret_cast<uint4*>(slot + g.routed_x);
  uint4* sx = reinterpret_cast<uint4*>(slot + g.shared_x);
  int32_t* sidx = reinterpret_cast<int32_t*>(slot + g.shared_idx);
  const uint4* __restrict__ rows = pl.rows[e];
  const int n = pl.n_rows[e];
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nvec = (int64_t)n * row_bytes / 16;
  for (int64_t i = i0; i < nvec; i += stride) {
    const uint4 v = rows[i];
    rx[i] = v;
    if (with_shared) sx[i] = v;
  }
  if (with_shared)
    for (int64_t i = i0; i < n; i += stride) sidx[i] = (int32_t)i;
}

__global__ void k_pack_header_multi(uint8_t* win, WinGeom g, int stage, int layer,
                                    const __grid_constant__ PackList pl, int with_shared, int num_experts) {
  grid_dep_wait();
  grid_dep_launch();
  const int e = blockIdx.x;
  if (e >= pl.n) return;
  write_dispatch_header(win, g, pl.region[e], stage, layer, pl.n_rows[e], with_shared, num_experts,
                        pl.seq[e], 0, 0, nullptr);
}

// ---------------------------------------------------------------------------
// a0: bounded wait for each listed flag, then header checks.  The order of
// the checks fixes which error is reported: the first failing check of the
// first failing list entry, then item_err (a fault of the step as a whole).
// kFromHeaders: f was built from these headers (work-item loop), so the
// token and row counts are checked against the slot capacity instead of a
// count the host gave.  Returns true (block-uniform) when every check passed;
// the consumed flags are then recorded in ws.seen.
// ---------------------------------------------------------------------------
template <bool kFromHeaders>
__device__ bool check_entries(const uint8_t* win, const WinGeom& g, const FanIn& f, const DevWS& ws,
                              int E, int token_cap, int rows_cap, int has_shared_expert,
                              int64_t timeout_ns, int item_err, bool check_status,
                              uint32_t go_token) {
  __shared__ int err[AFD_MAX_PEERS];
  __shared__ int bad_sidx[AFD_MAX_PEERS];
  __shared__ int shared_n[AFD_MAX_PEERS];
  __shared__ int skip;
  const int tid = threadIdx.x;
  // each entry's first flag poll is issued with the status word's load
  const int slotno = tid < f.n_peers ? f.region[tid] * g.ring_depth + f.stage : 0;
  const uint64_t* flagp = reinterpret_cast<const uint64_t*>(win) + slotno;
  uint64_t seen = 0, fl = 0;
  if (tid < f.n_peers) {
    seen = ws.seen[slotno];
    fl = ld_acquire_u64(flagp);
  }
  if (tid == 0) skip = check_status ? read_status(ws.status) : 0;
  if (tid < AFD_MAX_PEERS) { err[tid] = 0; bad_sidx[tid] = 0; shared_n[tid] = 0; }
  __syncthreads();
  if (skip) {
    if (tid == 0 && go_token) st_release_u32(ws.go, go_token | AFD_GO_ABORT);
    return false;
  }
  int e = 0;
  if (tid < f.n_peers) {
    const uint64_t t0 = globaltimer_ns();
    unsigned backoff = 32;
    while (fl <= seen) {
      if (globaltimer_ns() - t0 > (uint64_t)timeout_ns) { e = AFD_ERR_TIMEOUT; break; }
      __nanosleep(backoff);
      if (backoff < 1024) backoff <<= 1;
      fl = ld_acquire_u64(flagp);
    }
  }
  // every listed flag acquired (or given up on): the router may read the
  // rows, and this block reads the headers and shared_idx fields at once
  const bool late = __syncthreads_or(e != 0);
  if (go_token && tid == 0) st_release_u32(ws.go, late ? (go_token | AFD_GO_ABORT) : go_token);
  // shared_idx must list the entry's shared tokens: row j is token
  // ffn_rank + j * ffn_size (0..n-1 with one FFN rank: every token is a
  // shared token; Async GPU Connector, "Data flow" step 3, arange(ffn_rank,
  // n, ffn_size)).  The rows the fan-in expects of every entry (sprefix)
  // form one index space, 8 independent loads in flight per thread, read
  // with the headers; a mismatch counts only for an entry whose header
  // announces its shared rows (shared_n below).
  {
    const int total = f.sprefix[f.n_peers];
    for (int r0 = tid; r0 < total; r0 += 8 * blockDim.x) {
      int v[8], want[8], who[8];
#pragma unroll
      for (int u = 0; u < 8; u++) {
        const int r = r0 + u * blockDim.x;
        who[u] = -1;
        v[u] = want[u] = 0;
        if (r < total) {
          const int lo = entry_of_shared(f, r);
          const int32_t* sidx = reinterpret_cast<const int32_t*>(
              slot_ptr(win, g, f.region[lo], f.stage) + g.shared_idx);
          const int j = r - f.sprefix[lo];
          want[u] = f.ffn_rank + j * f.ffn_size;
          who[u] = lo;
          v[u] = sidx[j];
        }
      }
#pragma unroll
      for (int u = 0; u < 8; u++)
        if (who[u] >= 0 && v[u] != want[u]) bad_sidx[who[u]] = 1;
    }
  }
  if (tid < f.n_peers) {
    const int i = tid;
    if (!e) {
      // the 12 fixed words in three 16-byte loads, ordered after the acquire
      int32_t h[12];
      const int4* hp = reinterpret_cast<const int4*>(slot_ptr(win, g, f.region[i], f.stage) + g.header);
#pragma unroll
      for (int q = 0; q < 3; q++) {
        int4 v;
        asm volatile("ld.relaxed.gpu.global.v4.s32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "l"(hp + q)
                     : "memory");
        h[4 * q] = v.x; h[4 * q + 1] = v.y; h[4 * q + 2] = v.z; h[4 * q + 3] = v.w;
      }
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
      else if (kFromHeaders ? h[7] < 0 : h[7] != n)
        e = AFD_ERR_SHAPE;
      else if (h[7] > token_cap)
        e = AFD_ERR_CAPACITY;
      else if (kFromHeaders ? (h[8] < 0 || (!f.grouped && h[8] != 0))
                            : h[8] != (f.grouped ? f.rprefix[i + 1] - f.rprefix[i] : 0))
        e = AFD_ERR_SHAPE;
      else if (h[8] > rows_cap)
        e = AFD_ERR_CAPACITY;
      if (!e && f.grouped) {
        // the group list: rows per expert, each >= 0, summing to the rows;
        // kept for the plan and the return header
        // (ordered after the flag's acquire by the asm memory clobbers above)
        const int32_t* gl = reinterpret_cast<const int32_t*>(hp) + AFD_HEADER_FIXED_WORDS;
        int64_t sum = 0;
        int neg = 0;
        for (int x = 0; x < E; x++) {
          const int32_t v = gl[x];
          neg |= v < 0;
          sum += v;
          ws.peer_counts[i * E + x] = v;
        }
        if (neg || sum != h[8]) e = AFD_ERR_SHAPE;
      }
      // shared rows: none, or the entry's share (all n tokens with one FFN
      // rank, tokens ffn_rank, ffn_rank + ffn_size, ... with several)
      if (!e && h[9] != 0 && (h[9] != f.sprefix[i + 1] - f.sprefix[i] || !has_shared_expert))
        e = AFD_ERR_SHAPE;
      if (!e) shared_n[i] = h[9];
    }
    err[i] = e;
    ws.cur_seq[i] = fl;
  }
  __syncthreads();
  __shared__ int ok_s;
  if (tid == 0) {
    int first = 0;
    for (int i = 0; i < f.n_peers && !first; i++) {
      int e = err[i];
      if (!e && shared_n[i] > 0 && bad_sidx[i]) e = AFD_ERR_SHAPE;
      first = e;
    }
    if (!first) first = item_err;
    if (first) {
      set_error(ws.status, first);
    } else {
      for (int i = 0; i < f.n_peers; i++) {
        ws.seen[f.region[i] * g.ring_depth + f.stage] = ws.cur_seq[i];
        ws.peer_shared[i] = shared_n[i] > 0;
      }
    }
    ok_s = !first;
  }
  __syncthreads();
  return ok_s != 0;
}

// host-described step: f comes from the host, and so it does for the
// kernels after this one
__global__ void __launch_bounds__(1024)
k_header_check(const uint8_t* win, WinGeom g, const __grid_constant__ FanIn f, DevWS ws, int E,
               int token_cap, int rows_cap, int has_shared_expert, int64_t timeout_ns,
               uint32_t go_token) {
  grid_dep_wait();
  grid_dep_launch();
  check_entries<false>(win, g, f, ws, E, token_cap, rows_cap, has_shared_expert, timeout_ns, 0, true,
                       go_token);
}

// ---------------------------------------------------------------------------
// Head of a step of the device-resident work-item loop ([RFC]: Async AFD
// for Prefill on Ascend NPU, "Asynchronous work-item contract" and "FFN
// execution modes"; [RFC]: Async GPU Connector, the wait_any kernel named
// under "Risks and alternatives").  A stage of the ring is a work item; it
// is ready once every listed peer has published a flag newer than the one
// last consumed from its slot.  The scan starts after the stage served
// last, so a ready stage waits for at most ring_depth - 1 others.  The wait
// is bounded (AFD_ERR_TIMEOUT).  The layer and the token / row counts are
// then taken from the headers, never read back by the host: the fan-in is
// built here, checked like a host-described one, written to ws.item, and
// the item is appended to the loop's log.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
k_item_head(const uint8_t* win, WinGeom g, PeerList pl, DevWS ws, int E, int token_cap,
            int rows_cap, int ffn_rank, int ffn_size, int has_shared_expert, int grouped, int tmax,
            int rmax, int max_layers, int64_t timeout_ns) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ FanIn fs;
  __shared__ int hl[AFD_MAX_PEERS], hn[AFD_MAX_PEERS], hr[AFD_MAX_PEERS];
  __shared__ int skip, rot, item_err;
  const int tid = threadIdx.x;
  const int R = g.ring_depth;
  const uint64_t* flags = reinterpret_cast<const uint64_t*>(win);
  if (tid == 0) {
    skip = read_status(ws.status);
    rot = ws.loop[AFD_LOOP_ROT];
  }
  __syncthreads();
  if (skip) return;
  // wait_any: block-uniform scan of the stages from rot
  const uint64_t t0 = globaltimer_ns();
  unsigned backoff = 32;
  int chosen = -1;
  for (;;) {
    for (int s = 0; s < R && chosen < 0; s++) {
      const int r = (rot + s) % R;
      bool ready = true;
      if (tid < pl.n) {
        const int slotno = pl.slot[tid] * R + r;
        ready = ld_acquire_u64(flags + slotno) > ws.seen[slotno];
      }
      if (__syncthreads_and(ready)) chosen = r;
    }
    if (chosen >= 0) break;
    if (__syncthreads_or(tid == 0 && globaltimer_ns() - t0 > (uint64_t)timeout_ns)) break;
    __nanosleep(backoff);
    if (backoff < 1024) backoff <<= 1;
  }
  if (chosen < 0) {
    if (tid == 0) set_error(ws.status, AFD_ERR_TIMEOUT);
    return;
  }
  // layer and counts of every entry, ordered after its flag
  if (tid < pl.n) {
    (void)ld_acquire_u64(flags + pl.slot[tid] * R + chosen);
    const int32_t* hp = reinterpret_cast<const int32_t*>(slot_ptr(win, g, pl.slot[tid], chosen) + g.header);
    int32_t w5, w7, w8;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(w5) : "l"(hp + 5) : "memory");
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(w7) : "l"(hp + 7) : "memory");
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(w8) : "l"(hp + 8) : "memory");
    hl[tid] = w5;
    hn[tid] = w7;
    hr[tid] = w8;
  }
  __syncthreads();
  if (tid == 0) {
    fs.n_peers = pl.n;
    fs.stage = chosen;
    fs.layer = hl[0];
    fs.grouped = grouped;
    fs.num_experts = E;
    fs.ffn_rank = ffn_rank;
    fs.ffn_size = ffn_size;
    int64_t T = 0, Rr = 0, S = 0;
    for (int i = 0; i < pl.n; i++) {
      fs.region[i] = pl.slot[i];
      fs.prefix[i] = (int)T;
      fs.rprefix[i] = (int)Rr;
      fs.sprefix[i] = (int)S;
      // out-of-range counts count as 0 here; the checks report them
      const int n = (hn[i] >= 0 && hn[i] <= token_cap) ? hn[i] : 0;
      T += n;
      S += rr_rows(n, ffn_rank, ffn_size);
      Rr += (grouped && hr[i] >= 0 && hr[i] <= rows_cap) ? hr[i] : 0;
    }
    fs.prefix[pl.n] = fs.total = (int)T;
    fs.rprefix[pl.n] = fs.rtotal = (int)Rr;
    fs.sprefix[pl.n] = fs.stotal = (int)S;
    const int L = fs.layer;
    item_err = (L < 0 || L >= max_layers || !ws.layers[L].set) ? AFD_ERR_LAYER
               : (T > tmax || Rr > rmax)                        ? AFD_ERR_CAPACITY
                                                                : 0;
  }
  __syncthreads();
  if (!check_entries<true>(win, g, fs, ws, E, token_cap, rows_cap, has_shared_expert, timeout_ns,
                           item_err, false, 0))
    return;
  {
    const int32_t* src = reinterpret_cast<const int32_t*>(&fs);
    int32_t* dst = reinterpret_cast<int32_t*>(ws.item);
    for (int i = tid; i < (int)(sizeof(FanIn) / 4); i += blockDim.x) dst[i] = src[i];
  }
  if (tid == 0) {
    ws.loop[AFD_LOOP_ROT] = (chosen + 1) % R;
    const int c = ws.loop[AFD_LOOP_COUNT];
    int32_t* rec = ws.loop + AFD_LOOP_LOG + 4 * (c % AFD_LOOP_LOG_N);
    rec[0] = chosen;
    rec[1] = fs.layer;
    rec[2] = fs.total;
    rec[3] = fs.rtotal;
    ws.loop[AFD_LOOP_COUNT] = c + 1;
  }
}

// ---------------------------------------------------------------------------
// a1: router (DeepSeek-V2 MoE gate: softmax over the expert affinities,
// top-k of them).  Two kernels: k_router_logits writes the fp32 logits in
// one fixed summation order, k_router_topk selects and weights.
// ---------------------------------------------------------------------------
// Float-float helpers for the softmax: a value carried as hi + lo with the
// rounding error of every addition kept (two-sum), so sums of E terms carry
// no accumulated rounding and no fp64 arithmetic is needed.
struct ffloat {
  float hi, lo;
};
__device__ __forceinline__ ffloat ff_add(ffloat a, float b) {
  const float s = __fadd_rn(a.hi, b);
  const float bb = __fsub_rn(s, a.hi);
  const float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, __fadd_rn(a.lo, e)};
}
__device__ __forceinline__ ffloat ff_add(ffloat a, ffloat b) {
  ffloat r = ff_add(a, b.hi);
  r.lo = __fadd_rn(r.lo, b.lo);
  return r;
}
__device__ __forceinline__ ffloat ff_shfl_xor(ffloat a, int off) {
  return {__shfl_xor_sync(0xffffffffu, a.hi, off), __shfl_xor_sync(0xffffffffu, a.lo, off)};
}
// a / (d.hi + d.lo) to about one ulp
__device__ __forceinline__ float ff_div(float a, ffloat d) {
  const float q = __fdiv_rn(a, d.hi);
  return __fmaf_rn(-q, __fdiv_rn(d.lo, d.hi), q);
}
// exp(a - b): the difference is split exactly into s + err (two-sum), so
// exp(a - b) = expf(s) * (1 + err) to first order.
__device__ __forceinline__ float exp_of_diff(float a, float b) {
  const float s = __fsub_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(-b, bb));
  const float e = expf(s);
  return __fmaf_rn(e, err, e);
}

constexpr int kRtTok = 16;        // tokens per top-k CTA (and per plan histogram)
constexpr int kPlanSmallMax = 8192;  // partials up to which one CTA plans (no histograms)
constexpr int kLgTok = 8;         // tokens per logits warp
constexpr int kLgEpw = 4;         // experts per logits warp
constexpr int kLgWarps = 4;
constexpr int kLgEblk = kLgWarps * kLgEpw;   // experts per logits CTA

// Token tile of a logits CTA in smem (bf16 bits, or fp32 for fp32
// activations), in 16-byte groups of tokens, group-major
// ([group][h][tokens of the group]): the lane owning h reads a group with
// one 16-byte load, contiguous across the warp's lanes (no bank conflicts).
template <typename XS>
__device__ __forceinline__ int lg_index(int h, int tt, int hidden) {
  constexpr int per = 16 / sizeof(XS);
  return ((tt / per) * hidden + h) * per + (tt % per);
}

// a1 router, part 1: logits in the canonical fp32 order.  Lane l of a warp
// owns the fused multiply-add chain over h = l, l+32, ... ascending (from
// +0); a butterfly with xor offsets 16, 8, 4, 2, 1 sums the 32 chains, then
// + bias.  CTA (8 tokens, 16 experts): warp w takes experts 4w..4w+3 for all
// 8 tokens; the token rows are staged from the peer slots into smem, the
// transposed router weight [E][hidden] is read from L2 with the next step's
// values loaded ahead of the current step's multiply-adds.
template <typename XS, bool kDev>
__global__ void __launch_bounds__(kLgWarps * 32)
k_router_logits(const uint8_t* win, WinGeom g, const __grid_constant__ FanIn fp, DevWS ws, int hidden,
                const float* __restrict__ WgQ, const float* __restrict__ bias, int E,
                float* __restrict__ logits) {
  grid_dep_wait();
  grid_dep_launch();
  const FanIn& f = step_item<kDev>(fp, ws.item);
  if (!WgQ) {  // the layer of the step was chosen on the device
    WgQ = ws.layers[f.layer].WgQ;
    bias = ws.layers[f.layer].bias;
  }
  extern __shared__ __align__(16) uint8_t lg_smem[];
  XS* xT = reinterpret_cast<XS*>(lg_smem);       // [hidden][8 tokens]
  if (read_status(ws.status)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kLgTok;
  constexpr bool kF32 = sizeof(XS) == 4;
  const int row_bytes = hidden * (int)sizeof(XS);
  constexpr int kVecElems = 16 / sizeof(XS);
  {
    // thread -> (token tt, vectors v = tid / 8, + 16, ...); 4 loads in flight
    const int tt = threadIdx.x % kLgTok;
    const int t = t0 + tt;
    const int nvec = row_bytes / 16;
    const int step = blockDim.x / kLgTok;
    const uint4* src = nullptr;
    if (t < f.total) {
      const int i = entry_of(f, t);
      src = reinterpret_cast<const uint4*>(slot_ptr(win, g, f.region[i], f.stage) + g.routed_x +
                                           (int64_t)(t - f.prefix[i]) * row_bytes);
    }
    for (int v0 = threadIdx.x / kLgTok; v0 < nvec; v0 += 4 * step) {
      uint4 val[4];
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int v = v0 + u * step;
        val[u] = (src && v < nvec) ? src[v] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int v = v0 + u * step;
        if (v >= nvec) break;
        const XS* e8 = reinterpret_cast<const XS*>(&val[u]);
#pragma unroll
        for (int m = 0; m < kVecElems; m++) xT[lg_index<XS>(v * kVecElems + m, tt, hidden)] = e8[m];
      }
    }
  }
  __syncthreads();
  const int e0 = blockIdx.y * kLgEblk + warp * kLgEpw;
  if (e0 >= E) return;
  const float* wrow[kLgEpw];  // expert e, h at wrow[b][4 h]
#pragma unroll
  for (int b = 0; b < kLgEpw; b++) {
    const int e = min(e0 + b, E - 1);
    wrow[b] = WgQ + (int64_t)(e >> 2) * hidden * 4 + (e & 3);
  }
  float acc[kLgTok][kLgEpw];
#pragma unroll
  for (int a = 0; a < kLgTok; a++)
#pragma unroll
    for (int b = 0; b < kLgEpw; b++) acc[a][b] = 0.0f;
  // 4 h-steps per batch: their 16 weight values are loaded together
  const int nsteps = (hidden + 31) / 32;
  for (int i0 = 0; i0 < nsteps; i0 += 4) {
    float wv[4][kLgEpw];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int h = lane + 32 * (i0 + u);
#pragma unroll
      for (int b = 0; b < kLgEpw; b++) wv[u][b] = h < hidden ? __ldg(wrow[b] + 4 * h) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int h = lane + 32 * (i0 + u);
      if (h < hidden) {
        float xv[kLgTok];
        if constexpr (kF32) {
#pragma unroll
          for (int q = 0; q < kLgTok / 4; q++) {
            const float4 v4 = *reinterpret_cast<const float4*>(xT + lg_index<XS>(h, 4 * q, hidden));
            xv[4 * q] = v4.x; xv[4 * q + 1] = v4.y; xv[4 * q + 2] = v4.z; xv[4 * q + 3] = v4.w;
          }
        } else {
          const uint4 v4 = *reinterpret_cast<const uint4*>(xT + lg_index<XS>(h, 0, hidden));
          const uint32_t w4[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
          for (int m = 0; m < 4; m++) {
            xv[2 * m] = __uint_as_float(w4[m] << 16);
            xv[2 * m + 1] = __uint_as_float(w4[m] & 0xffff0000u);
          }
        }
#pragma unroll
        for (int a = 0; a < kLgTok; a++)
#pragma unroll
          for (int b = 0; b < kLgEpw; b++) acc[a][b] = __fmaf_rn(xv[a], wv[u][b], acc[a][b]);
      }
    }
  }
#pragma unroll
  for (int a = 0; a < kLgTok; a++)
#pragma unroll
    for (int b = 0; b < kLgEpw; b++) {
      float v = acc[a][b];
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
      acc[a][b] = v;
    }
#pragma unroll
  for (int a = 0; a < kLgTok; a++)
    if (lane == a && t0 + a < f.total)
#pragma unroll
      for (int b = 0; b < kLgEpw; b++)
        if (e0 + b < E)
          logits[(int64_t)(t0 + a) * E + e0 + b] = bias ? __fadd_rn(acc[a][b], bias[e0 + b]) : acc[a][b];
}

// a1 router, part 1, weight-stationary form (same canonical order as
// k_router_logits).  A CTA owns a block of 4 * EPW experts, whose rows of the
// transposed router weight stay in shared memory for its whole life, and
// walks the token tiles blockIdx.x, + gridDim.x, ...: each tile of 8 token
// rows is copied from the peer slots with one bulk copy per row into a ring
// of `ns` buffers, the copies of later tiles in flight while the four warps
// compute (warp w: experts 4w..4w+3 of the block x the 8 tokens).
constexpr int kWsTok = 8;
constexpr int kWsWarps = 4;
constexpr uint64_t kWsTimeoutNs = 1000000000ull;

struct WsGeom {
  int ns;          // x ring buffers
  size_t w_bytes;  // weight block, 128-byte rounded
  size_t tile_bytes;
  size_t smem;
};

template <typename XS, int EPW, bool kDev>
__global__ void __launch_bounds__(kWsWarps * 32, 1)
k_router_logits_ws(const uint8_t* win, WinGeom g, const __grid_constant__ FanIn fp, DevWS ws, int hidden,
                   const float* __restrict__ WgQ, const float* __restrict__ bias, int E,
                   float* __restrict__ logits, WsGeom geo) {
  grid_dep_wait();
  grid_dep_launch();
  const FanIn& f = step_item<kDev>(fp, ws.item);
  if (!WgQ) {  // the layer of the step was chosen on the device
    WgQ = ws.layers[f.layer].WgQ;
    bias = ws.layers[f.layer].bias;
  }
  extern __shared__ __align__(128) uint8_t ws_smem[];
  constexpr int EB = EPW * kWsWarps;
  const float* Ws = reinterpret_cast<const float*>(ws_smem);  // [EB / 4][hidden][4]
  const uint8_t* xring = ws_smem + geo.w_bytes;                                  // [ns][8][hidden]
  uint64_t* bars = reinterpret_cast<uint64_t*>(ws_smem + geo.w_bytes + geo.ns * geo.tile_bytes);
  __shared__ int abort_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (read_status(ws.status)) return;
  const int e_base = blockIdx.y * EB;
  const int ne = min(EB, E - e_base);
  const int ntiles = (f.total + kWsTok - 1) / kWsTok;
  if ((int)blockIdx.x >= ntiles || ne <= 0) return;
  const int my_tiles = (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1;
  const int row_bytes = hidden * (int)sizeof(XS);
  const uint32_t wbar = smem_u32(&bars[geo.ns]);
  auto issue = [&](int i) {  // tile i of this CTA into buffer i % ns (thread 0)
    const int buf = i % geo.ns;
    const int t0 = ((int)blockIdx.x + i * (int)gridDim.x) * kWsTok;
    const int nt = min(kWsTok, f.total - t0);
    const uint32_t bar = smem_u32(&bars[buf]);
    mbar_expect_tx(bar, (uint32_t)(nt * row_bytes));
    for (int r = 0; r < nt; r++) {
      const int t = t0 + r;
      const int e = entry_of(f, t);
      const uint8_t* src = slot_ptr(win, g, f.region[e], f.stage) + g.routed_x +
                           (int64_t)(t - f.prefix[e]) * row_bytes;
      bulk_load(smem_u32(xring + buf * geo.tile_bytes + (size_t)r * row_bytes), src,
                (uint32_t)row_bytes, bar);
    }
  };
  if (tid == 0) {
    abort_s = 0;
    for (int b = 0; b <= geo.ns; b++) mbar_init(smem_u32(&bars[b]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const uint32_t wbytes = (uint32_t)(((ne + 3) / 4) * hidden * 16);
    mbar_expect_tx(wbar, wbytes);
    bulk_load(smem_u32(ws_smem), WgQ + (int64_t)e_base * hidden, wbytes, wbar);
    for (int i = 0; i < min(geo.ns, my_tiles); i++) issue(i);
  }
  __syncthreads();
  const uint64_t deadline = globaltimer_ns() + kWsTimeoutNs;
  auto wait = [&](uint32_t bar, uint32_t parity) {
    uint32_t spins = 0;
    while (!mbar_try_wait(bar, parity)) {
      if ((++spins & 255u) == 0 && (*(volatile int*)&abort_s || globaltimer_ns() > deadline)) {
        abort_s = 1;
        return false;
      }
    }
    return true;
  };
  int done = 0;  // tiles consumed
  // every wait is followed by a block-wide vote, so all threads leave together
  if (!__syncthreads_or(!wait(wbar, 0))) {
    const int el = warp * EPW;  // first local expert of this warp
    const float* wrow[EPW];  // local expert e, h at wrow[b][4 h]
#pragma unroll
    for (int b = 0; b < EPW; b++) {
      const int e = min(el + b, ne - 1);
      wrow[b] = Ws + (size_t)(e >> 2) * hidden * 4 + (e & 3);
    }
    const int nfull = hidden / 32;
    for (int i = 0; i < my_tiles; i++) {
      const int buf = i % geo.ns;
      if (__syncthreads_or(!wait(smem_u32(&bars[buf]), (uint32_t)((i / geo.ns) & 1)))) break;
      const XS* xt = reinterpret_cast<const XS*>(xring + buf * geo.tile_bytes);
      float acc[kWsTok][EPW];
#pragma unroll
      for (int a = 0; a < kWsTok; a++)
#pragma unroll
        for (int b = 0; b < EPW; b++) acc[a][b] = 0.0f;
      auto step = [&](int h) {
        float wv[EPW];
#pragma unroll
        for (int b = 0; b < EPW; b++) wv[b] = wrow[b][4 * h];
#pragma unroll
        for (int a = 0; a < kWsTok; a++) {
          float xv;
          if constexpr (sizeof(XS) == 4) xv = reinterpret_cast<const float*>(xt)[(size_t)a * hidden + h];
          else xv = bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(xt)[(size_t)a * hidden + h]);
#pragma unroll
          for (int b = 0; b < EPW; b++) acc[a][b] = __fmaf_rn(xv, wv[b], acc[a][b]);
        }
      };
#pragma unroll 4
      for (int j = 0; j < nfull; j++) step(32 * j + lane);
      if (32 * nfull + lane < hidden) step(32 * nfull + lane);
#pragma unroll
      for (int a = 0; a < kWsTok; a++)
#pragma unroll
        for (int b = 0; b < EPW; b++) {
          float v = acc[a][b];
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
          acc[a][b] = v;
        }
      const int t0 = ((int)blockIdx.x + i * (int)gridDim.x) * kWsTok;
#pragma unroll
      for (int a = 0; a < kWsTok; a++)
        if (lane == a && t0 + a < f.total)
#pragma unroll
          for (int b = 0; b < EPW; b++)
            if (el + b < ne) {
              const int e = e_base + el + b;
              logits[(int64_t)(t0 + a) * E + e] = bias ? __fadd_rn(acc[a][b], bias[e]) : acc[a][b];
            }
      __syncthreads();  // every warp is done with this buffer
      done = i + 1;
      if (tid == 0 && i + geo.ns < my_tiles && !abort_s) issue(i + geo.ns);
    }
  }
  __syncthreads();
  if (abort_s && tid == 0) {
    set_error(ws.status, AFD_ERR_TIMEOUT);
    // copies still in flight land in this CTA's shared memory: wait (bounded)
    const uint64_t dl = globaltimer_ns() + 100000000ull;
    while (!mbar_try_wait(wbar, 0) && globaltimer_ns() < dl) {}
    const int issued = min(my_tiles, done + geo.ns);
    for (int i = done; i < issued; i++)
      while (!mbar_try_wait(smem_u32(&bars[i % geo.ns]), (uint32_t)((i / geo.ns) & 1)) &&
             globaltimer_ns() < dl) {}
  }
}

// a1 router, part 1, for bf16 activations: weight-stationary with the token
// tile transposed in shared memory (same canonical order).  A CTA owns 16
// experts (4 groups of the rearranged weight, 4 per warp) for its whole life
// and walks the token tiles blockIdx.x, + gridDim.x, ...  A tile of 8 token
// rows lands by bulk copies in a row-major staging buffer (the next tile's
// copies overlap the current tile's arithmetic); the CTA then transposes it
// to one 16-byte record per h holding the 8 tokens' values (a 16-byte pad
// after every 8 records keeps both the transposing stores and the reads free
// of bank conflicts).  Per h a lane then needs one 16-byte load of tokens
// and one of weights for 32 multiply-adds, issued as pairs over two tokens.
// Butterfly over the 32 lanes for 32 values at once, scattered: at offset o
// a lane keeps the half of its values selected by its lane bit o and adds
// the partner's copy, so lane l ends with value l summed over all lanes.
// Each value sees exactly the additions of the all-lane butterfly with
// offsets 16, 8, 4, 2, 1 (addition commutes), in 31 shuffles instead of 160.
__device__ __forceinline__ float butterfly_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; i++) {
      const float send = up ? v[i] : v[i + o];
      const float keep = up ? v[i + o] : v[i];
      v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, o));
    }
  }
  return v[0];
}

constexpr int kTwTok = 8;
constexpr int kTwWarps = 4;
constexpr int kTwExperts = 4 * kTwWarps;

__host__ __device__ inline size_t tw_rec_offset(int h) { return 16 * (size_t)h + 16 * (size_t)(h >> 3); }

struct TwGeom {
  size_t w_bytes;      // weight block, 128-byte rounded
  size_t stage_bytes;  // 8 rows, row-major
  size_t xt_bytes;     // transposed records
  size_t smem;
};

template <bool kDev>
__global__ void __launch_bounds__(kTwWarps * 32, 1)
k_router_logits_tw(const uint8_t* win, WinGeom g, const __grid_constant__ FanIn fp, DevWS ws, int hidden,
                   const float* __restrict__ WgQ, const float* __restrict__ bias, int E,
                   float* __restrict__ logits, TwGeom geo) {
  grid_dep_wait();
  grid_dep_launch();
  const FanIn& f = step_item<kDev>(fp, ws.item);
  if (!WgQ) {  // the layer of the step was chosen on the device
    WgQ = ws.layers[f.layer].WgQ;
    bias = ws.layers[f.layer].bias;
  }
  extern __shared__ __align__(128) uint8_t tw_smem[];
  const float4* Wq = reinterpret_cast<const float4*>(tw_smem);  // [4 groups][hidden]
  uint8_t* stage = tw_smem + geo.w_bytes;                         // [8][hidden] bf16
  uint8_t* xt = stage + geo.stage_bytes;                          // records
  uint64_t* bars = reinterpret_cast<uint64_t*>(xt + geo.xt_bytes);  // [0] weights, [1] stage
  __shared__ int abort_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (read_status(ws.status)) return;
  const int e_base = blockIdx.y * kTwExperts;
  const int ne = min(kTwExperts, E - e_base);
  const int ntiles = (f.total + kTwTok - 1) / kTwTok;
  if ((int)blockIdx.x >= ntiles || ne <= 0) return;
  const int my_tiles = (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1;
  const int row_bytes = hidden * 2;
  const uint32_t wbar = smem_u32(&bars[0]), sbar = smem_u32(&bars[1]);
  auto issue = [&](int i) {  // tile i of this CTA into the staging buffer (thread 0)
    const int t0 = ((int)blockIdx.x + i * (int)gridDim.x) * kTwTok;
    const int nt = min(kTwTok, f.total - t0);
    mbar_expect_tx(sbar, (uint32_t)(nt * row_bytes));
    for (int r = 0; r < nt; r++) {
      const int t = t0 + r;
      const int e = entry_of(f, t);
      const uint8_t* src = slot_ptr(win, g, f.region[e], f.stage) + g.routed_x +
                           (int64_t)(t - f.prefix[e]) * row_bytes;
      bulk_load(smem_u32(stage + (size_t)r * row_bytes), src, (uint32_t)row_bytes, sbar);
    }
  };
  if (tid == 0) {
    abort_s = 0;
    mbar_init(wbar, 1);
    mbar_init(sbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const uint32_t wbytes = (uint32_t)(((ne + 3) / 4) * hidden * 16);
    mbar_expect_tx(wbar, wbytes);
    bulk_load(smem_u32(tw_smem), WgQ + (int64_t)e_base * hidden, wbytes, wbar);
    issue(0);
  }
  __syncthreads();
  const uint64_t deadline = globaltimer_ns() + kWsTimeoutNs;
  auto wait = [&](uint32_t bar, uint32_t parity) {
    uint32_t spins = 0;
    while (!mbar_try_wait(bar, parity)) {
      if ((++spins & 255u) == 0 && (*(volatile int*)&abort_s || globaltimer_ns() > deadline)) {
        abort_s = 1;
        return false;
      }
    }
    return true;
  };
  int done = 0;  // tiles consumed
  // every wait is followed by a block-wide vote, so all threads leave together
  if (!__syncthreads_or(!wait(wbar, 0))) {
    const int grp = min(warp, (ne - 1) / 4);  // a warp past the block's experts computes a copy
    const float4* wq = Wq + (size_t)grp * hidden;
    const int nchunks = hidden / 8;
    for (int i = 0; i < my_tiles; i++) {
      if (__syncthreads_or(!wait(sbar, (uint32_t)(i & 1)))) break;
      // stage [t][h] -> records [h][t]: thread takes 8-wide h chunks; rows
      // past the fan-in total hold stale bytes whose results are not stored
      for (int c = tid; c < nchunks; c += blockDim.x) {
        uint4 in[kTwTok];
#pragma unroll
        for (int t = 0; t < kTwTok; t++)
          in[t] = *reinterpret_cast<const uint4*>(stage + (size_t)t * row_bytes + 16 * c);
        const uint32_t* iw[kTwTok];
#pragma unroll
        for (int t = 0; t < kTwTok; t++) iw[t] = reinterpret_cast<const uint32_t*>(&in[t]);
#pragma unroll
        for (int j = 0; j < 8; j++) {
          const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
          uint4 o;
          o.x = __byte_perm(iw[0][j >> 1], iw[1][j >> 1], sel);
          o.y = __byte_perm(iw[2][j >> 1], iw[3][j >> 1], sel);
          o.z = __byte_perm(iw[4][j >> 1], iw[5][j >> 1], sel);
          o.w = __byte_perm(iw[6][j >> 1], iw[7][j >> 1], sel);
          *reinterpret_cast<uint4*>(xt + tw_rec_offset(8 * c + j)) = o;
        }
      }
      __syncthreads();  // records written, staging buffer free
      done = i + 1;
      if (tid == 0 && i + 1 < my_tiles) issue(i + 1);
      float2 acc[kTwTok / 2][4];  // {token 2p, token 2p + 1} x expert b of the group
#pragma unroll
      for (int p = 0; p < kTwTok / 2; p++)
#pragma unroll
        for (int b = 0; b < 4; b++) acc[p][b] = make_float2(0.0f, 0.0f);
      auto step = [&](int h) {
        const uint4 xr = *reinterpret_cast<const uint4*>(xt + tw_rec_offset(h));
        const float4 w4 = wq[h];
        const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w};
        const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int p = 0; p < kTwTok / 2; p++) {
          const float2 xp = make_float2(__uint_as_float(xw[p] << 16), __uint_as_float(xw[p] & 0xffff0000u));
#pragma unroll
          for (int b = 0; b < 4; b++) acc[p][b] = __ffma2_rn(xp, make_float2(wv[b], wv[b]), acc[p][b]);
        }
      };
      const int nfull = hidden / 32;
#pragma unroll 4
      for (int j = 0; j < nfull; j++) step(32 * j + lane);
      if (32 * nfull + lane < hidden) step(32 * nfull + lane);
      float v[32];  // index 4 t + b
#pragma unroll
      for (int p = 0; p < kTwTok / 2; p++)
#pragma unroll
        for (int b = 0; b < 4; b++) {
          v[8 * p + b] = acc[p][b].x;
          v[8 * p + 4 + b] = acc[p][b].y;
        }
      const float sum = butterfly_scatter32(v, lane);  // token lane / 4, expert lane % 4
      const int t = ((int)blockIdx.x + i * (int)gridDim.x) * kTwTok + (lane >> 2);
      const int el = 4 * warp + (lane & 3);
      if (t < f.total && el < ne) {
        const int e = e_base + el;
        logits[(int64_t)t * E + e] = bias ? __fadd_rn(sum, bias[e]) : sum;
      }
      __syncthreads();  // every warp is done with the records
    }
  }
  __syncthreads();
  if (abort_s && tid == 0) {
    set_error(ws.status, AFD_ERR_TIMEOUT);
    // copies still in flight land in this CTA's shared memory: wait (bounded)
    const uint64_t dl = globaltimer_ns() + 100000000ull;
    while (!mbar_try_wait(wbar, 0) && globaltimer_ns() < dl) {}
    if (done < my_tiles)
      while (!mbar_try_wait(sbar, (uint32_t)(done & 1)) && globaltimer_ns() < dl) {}
  }
}

// The same computation with two independent tile streams per CTA (for
// hidden <= 2048): warps 0-3 and warps 4-7 each own a transposed-record
// buffer and take alternate token tiles, synchronising only among
// themselves (named barriers), so one stream's transposition and barrier
// waits overlap the other's arithmetic.  A stream's next tile is loaded from
// the peer slots into registers while it computes the current one.
constexpr int kTw2Chunks = 2;  // 8-element h chunks per thread and token: hidden <= 2048

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <bool kDev>
__global__ void __launch_bounds__(2 * kTwWarps * 32, 1)
k_router_logits_tw2(const uint8_t* win, WinGeom g, const __grid_constant__ FanIn fp, DevWS ws, int hidden,
                    const float* __restrict__ WgQ, const float* __restrict__ bias, int E,
                    float* __restrict__ logits, TwGeom geo, uint32_t go_token, int64_t go_timeout_ns) {
  // go_token != 0 (host-described steps): started before the header check
  // ends; the gate weights load at once, the fan-in's rows once ws.go holds
  // the token, and the wait on the check moves to every exit, so the end of
  // this grid still implies the check's
  struct ExitWait {
    bool on;
    __device__ ~ExitWait() {
      if (on) grid_dep_wait();
    }
  } exit_wait{go_token != 0};
  if (!go_token) grid_dep_wait();
  grid_dep_launch();
  const FanIn& f = step_item<kDev>(fp, ws.item);
  if (!WgQ) {  // the layer of the step was chosen on the device
    WgQ = ws.layers[f.layer].WgQ;
    bias = ws.layers[f.layer].bias;
  }
  extern __shared__ __align__(128) uint8_t tw_smem[];
  const float4* Wq = reinterpret_cast<const float4*>(tw_smem);  // [4 groups][hidden]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int set = warp / kTwWarps, wis = warp % kTwWarps, tis = tid % (kTwWarps * 32);
  uint8_t* xt = tw_smem + geo.w_bytes + set * geo.xt_bytes;      // this stream's records
  uint64_t* wbar_p = reinterpret_cast<uint64_t*>(tw_smem + geo.w_bytes + 2 * geo.xt_bytes);
  if (!go_token && read_status(ws.status)) return;
  const int e_base = blockIdx.y * kTwExperts;
  const int ne = min(kTwExperts, E - e_base);
  const int ntiles = (f.total + kTwTok - 1) / kTwTok;
  if ((int)blockIdx.x >= ntiles || ne <= 0) return;
  const int my_tiles = (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1;
  const int row_bytes = hidden * 2;
  const int nchunks = hidden / 8;
  const uint32_t wbar = smem_u32(wbar_p);
  if (tid == 0) {
    mbar_init(wbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const uint32_t wbytes = (uint32_t)(((ne + 3) / 4) * hidden * 16);
    mbar_expect_tx(wbar, wbytes);
    bulk_load(smem_u32(tw_smem), WgQ + (int64_t)e_base * hidden, wbytes, wbar);
  }
  if (go_token) {
    __shared__ int go_ok;
    if (tid == 0) {
      const uint64_t t0 = globaltimer_ns();
      int r = 0;
      for (;;) {
        const uint32_t v = ld_acquire_u32(ws.go);
        if (v == go_token) { r = 1; break; }
        if (v == (go_token | AFD_GO_ABORT)) break;  // the check reports the error
        if (globaltimer_ns() - t0 > (uint64_t)go_timeout_ns) {
          set_error(ws.status, AFD_ERR_TIMEOUT);
          break;
        }
        __nanosleep(64);
      }
      go_ok = r && !read_status(ws.status);
    }
    __syncthreads();
    if (!go_ok) {
      if (tid == 0) {  // the weight copy lands in this CTA's shared memory: wait (bounded)
        const uint64_t dl = globaltimer_ns() + 100000000ull;
        while (!mbar_try_wait(wbar, 0) && globaltimer_ns() < dl) {}
      }
      return;
    }
  }
  // tiles of this stream: local index i = set, set + 2, ...
  uint4 pre[kTw2Chunks][kTwTok];
  auto fetch = [&](int i) {  // tile i's chunks of this thread into pre (zeros past the fan-in)
    const int t0 = ((int)blockIdx.x + i * (int)gridDim.x) * kTwTok;
#pragma unroll
    for (int r = 0; r < kTwTok; r++) {
      const int t = t0 + r;
      const uint4* src = nullptr;
      if (t < f.total) {
        const int e = entry_of(f, t);
        src = reinterpret_cast<const uint4*>(slot_ptr(win, g, f.region[e], f.stage) + g.routed_x +
                                             (int64_t)(t - f.prefix[e]) * row_bytes);
      }
#pragma unroll
      for (int cc = 0; cc < kTw2Chunks; cc++) {
        const int c = tis + cc * kTwWarps * 32;
        pre[cc][r] = (src && c < nchunks) ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      }
    }
  };
  if (set < my_tiles) fetch(set);
  __syncthreads();
  const uint64_t deadline = globaltimer_ns() + kWsTimeoutNs;
  bool ok = true;
  {
    uint32_t spins = 0;
    while (!mbar_try_wait(wbar, 0)) {
      if ((++spins & 255u) == 0 && globaltimer_ns() > deadline) { ok = false; break; }
    }
  }
  if (__syncthreads_or(!ok)) {
    if (tid == 0) {
      set_error(ws.status, AFD_ERR_TIMEOUT);
      const uint64_t dl = globaltimer_ns() + 100000000ull;
      while (!mbar_try_wait(wbar, 0) && globaltimer_ns() < dl) {}
    }
    return;
  }
  const int grp = min(wis, (ne - 1) / 4);  // a warp past the block's experts computes a copy
  const float4* wq = Wq + (size_t)grp * hidden;
  const int bar_id = 1 + set;
  for (int i = set; i < my_tiles; i += 2) {
    named_bar_sync(bar_id, kTwWarps * 32);  // this stream is done reading its records
#pragma unroll
    for (int cc = 0; cc < kTw2Chunks; cc++) {
      const int c = tis + cc * kTwWarps * 32;
      if (c < nchunks) {
        const uint32_t* iw[kTwTok];
#pragma unroll
        for (int t = 0; t < kTwTok; t++) iw[t] = reinterpret_cast<const uint32_t*>(&pre[cc][t]);
#pragma unroll
        for (int j = 0; j < 8; j++) {
          const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
          uint4 o;
          o.x = __byte_perm(iw[0][j >> 1], iw[1][j >> 1], sel);
          o.y = __byte_perm(iw[2][j >> 1], iw[3][j >> 1], sel);
          o.z = __byte_perm(iw[4][j >> 1], iw[5][j >> 1], sel);
          o.w = __byte_perm(iw[6][j >> 1], iw[7][j >> 1], sel);
          *reinterpret_cast<uint4*>(xt + tw_rec_offset(8 * c + j)) = o;
        }
      }
    }
    named_bar_sync(bar_id, kTwWarps * 32);  // records complete
    if (i + 2 < my_tiles) fetch(i + 2);
    float2 acc[kTwTok / 2][4];  // {token 2p, token 2p + 1} x expert b of the group
#pragma unroll
    for (int p = 0; p < kTwTok / 2; p++)
#pragma unroll
      for (int b = 0; b < 4; b++) acc[p][b] = make_float2(0.0f, 0.0f);
    auto step = [&](int h) {
      const uint4 xr = *reinterpret_cast<const uint4*>(xt + tw_rec_offset(h));
      const float4 w4 = wq[h];
      const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w};
      const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int p = 0; p < kTwTok / 2; p++) {
        const float2 xp = make_float2(__uint_as_float(xw[p] << 16), __uint_as_float(xw[p] & 0xffff0000u));
#pragma unroll
        for (int b = 0; b < 4; b++) acc[p][b] = __ffma2_rn(xp, make_float2(wv[b], wv[b]), acc[p][b]);
      }
    };
    const int nfull = hidden / 32;
#pragma unroll 8
    for (int j = 0; j < nfull; j++) step(32 * j + lane);
    if (32 * nfull + lane < hidden) step(32 * nfull + lane);
    float v[32];  // index 4 t + b
#pragma unroll
    for (int p = 0; p < kTwTok / 2; p++)
#pragma unroll
      for (int b = 0; b < 4; b++) {
        v[8 * p + b] = acc[p][b].x;
        v[8 * p + 4 + b] = acc[p][b].y;
      }
    const float sum = butterfly_scatter32(v, lane);  // token lane / 4, expert lane % 4
    const int t = ((int)blockIdx.x + i * (int)gridDim.x) * kTwTok + (lane >> 2);
    const int el = 4 * wis + (lane & 3);
    if (t < f.total && el < ne) {
      const int e = e_base + el;
      logits[(int64_t)t * E + e] = bias ? __fadd_rn(sum, bias[e]) : sum;
    }
  }
}

// Top-k and gate weights of one token, by one warp.  lv[m] is the logit of
// expert lane + 32 m (-inf past E).  Selection on the logits, ties to the
// lower expert index, a NaN logit below every number; p_e = softmax over all
// E relative to the top logit (sums as float-float); the k chosen experts'
// p (renormalised to sum 1 if asked) times the scale.  Lane j < k returns
// the j-th choice and its weight.  The same steps for every NL: entries past
// E are skipped, so NL = 4 and NL = 8 give identical results for E <= 128.
template <int NL>
__device__ __forceinline__ void route_token(const float (&lv)[NL], int E, int k, int renorm, float scale,
                                            int lane, int& my_id, float& my_w) {
  uint32_t taken = 0;  // bit m: expert lane + 32m chosen
  float top_logit = 0.0f;
  my_id = 0;           // lane j keeps the j-th choice
  float my_logit = 0.0f;
  for (int j = 0; j < k; j++) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int m = 0; m < NL; m++) {
      const int e = m * 32 + lane;
      if (e >= E || (taken & (1u << m))) continue;
      float v = lv[m];
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
  ffloat den = {0.0f, 0.0f};
#pragma unroll
  for (int m = 0; m < NL; m++)
    if (m * 32 + lane < E) den = ff_add(den, exp_of_diff(lv[m], top_logit));
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) den = ff_add(den, ff_shfl_xor(den, off));
  const float p = (lane < k) ? ff_div(exp_of_diff(my_logit, top_logit), den) : 0.0f;
  ffloat psum = {p, 0.0f};
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) psum = ff_add(psum, ff_shfl_xor(psum, off));
  const float v = renorm ? ff_div(p, psum) : p;
  my_w = __fmul_rn(v, scale);
}

// a1 router, part 2: top-k on the logits (ties -> lower expert index, NaN
// below every number) and the gate weights from a softmax over all E
// (sums carried as float-float); one warp per token, 16 tokens per CTA,
// whose per-expert histogram (hist[cta][e]) feeds the plan.  With no hist
// (the allocation-free router, whose caller cannot poll a status word) a
// recorded error leaves id -1 and a NaN weight in every output instead.
template <bool kDev>
__global__ void __launch_bounds__(kRtTok * 32)
k_router_topk(const __grid_constant__ FanIn fp, DevWS ws, const float* __restrict__ logits, int E, int k, int renorm,
              float scale, int32_t* __restrict__ hist, int nblocks) {
  grid_dep_wait();
  grid_dep_launch();
  const FanIn& f = step_item<kDev>(fp, ws.item);
  __shared__ int hs[256];
  __shared__ int skip;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRtTok + warp;
  // the token's logits are loaded with the status word (in bounds either way)
  float lv[8];  // logit of expert lane + 32m
  {
    const float* l = logits + (int64_t)min(t, f.total - 1) * E;
#pragma unroll
    for (int m = 0; m < 8; m++) lv[m] = (t < f.total && m * 32 + lane < E) ? l[m * 32 + lane] : -INFINITY;
  }
  if (threadIdx.x == 0) skip = read_status(ws.status);
  for (int e = threadIdx.x; e < E; e += blockDim.x) hs[e] = 0;
  __syncthreads();
  if (skip) {
    if (!hist && t < f.total && lane < k) {
      ws.ids[(int64_t)t * k + lane] = -1;
      ws.w[(int64_t)t * k + lane] = __int_as_float(0x7fc00000);
    }
    return;
  }
  if (t < f.total) {
    int my_id;
    float my_w;
    route_token<8>(lv, E, k, renorm, scale, lane, my_id, my_w);
    if (lane < k) {
      ws.ids[(int64_t)t * k + lane] = my_id;
      ws.w[(int64_t)t * k + lane] = my_w;
      atomicAdd(&hs[my_id], 1);
    }
  }
  __syncthreads();
  if (hist)  // block-major: hist[cta][e]
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(int64_t)blockIdx.x * E + e] = hs[e];
}

// ---------------------------------------------------------------------------
// a1 router, fused (bf16 activations, hidden <= 2048, E <= 128): logits and
// top-k in one kernel on a thread-block cluster of C = ceil(E / 16) CTAs.
// CTA rank r holds the fp32 gate weights of experts [16 r, 16 r + 16) in
// shared memory for its whole life; all CTAs of a cluster walk the same
// 16-token blocks (two 8-token tiles each), so together they produce every
// logit of a block.  Eight compute warps form teams of 16 / EPW warps; a
// team takes one tile, warp w of it experts [EPW w, EPW w + EPW) of the
// CTA's 16 for the tile's 8 tokens, in the canonical fp32 order of
// k_router_logits (lane l's fused multiply-add chain over h = l, l + 32, ...
// ascending, a butterfly with xor offsets 16 .. 1, then + bias).  The tile's
// rows are staged in h-chunks of 256 * (16 / EPW) as transposed 16-byte
// records (8 tokens of one h), double-buffered, the next chunk loaded into
// registers while the current one is used.  Each finished logit goes by
// st.async straight into the shared memory of the block's owner, one CTA of
// the cluster in rotation, whose mbarrier counts the bytes; the owner's four
// top-k warps then select, weight and count the block's 16 tokens (ids,
// gate weights, the block's expert histogram for the plan) and give the
// buffer back through an mbarrier in every CTA.  The logits never reach
// global memory and no second kernel runs.  Every wait is bounded; an
// error stops the arithmetic but not the exchange, so every byte sent is
// awaited before the cluster's CTAs leave.
// ---------------------------------------------------------------------------
constexpr int kFrWarps = 8;                       // compute warps per CTA
constexpr int kFrSlots = 2;                       // logit buffers per CTA
constexpr int kFrMaxC = 8;                        // CTAs per cluster (E <= 128)
constexpr int kFrBlk = 16;                        // tokens per block: two 8-token tiles
static_assert(kFrBlk == kRtTok, "the plan's histogram rows are router blocks of kRtTok tokens");

struct FrGeom {
  uint32_t rec_off, rec_bytes;  // record buffers: [teams][2][rec_bytes]
  uint32_t lb_off;              // logit buffers: [kFrSlots][16][ep] fp32
  uint32_t hist_off;            // block histograms: [kFrSlots][ep] int
  uint32_t bar_off;             // weights, full[kFrSlots], empty[kFrMaxC][kFrSlots]
  uint32_t smem;
  int C, ep;                    // CTAs per cluster; experts rounded up to 16
};

__device__ __forceinline__ uint32_t fr_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// this CTA's shared address as seen in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t fr_mapa(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void fr_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 4 bytes into a peer's shared memory, counted on the peer's mbarrier
__device__ __forceinline__ void fr_st_async(uint32_t raddr, float v, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
               ::"r"(raddr), "r"(__float_as_uint(v)), "r"(rbar) : "memory");
}
__device__ __forceinline__ void fr_arrive_remote(uint32_t raddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(raddr) : "memory");
}
__device__ __forceinline__ bool fr_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// TK top-k warps.  Each SM sub-partition holds three of the CTA's twelve
// warps, so a thread gets at most 168 registers (16384 per sub-partition);
// fewer top-k warps would not give the compute warps more.
template <int EPW, bool kSpread, bool kDev, int TK = 4>
__global__ void __launch_bounds__((kFrWarps + TK) * 32, 1)
k_router_fused(const uint8_t* win, WinGeom g, const __grid_constant__ FanIn fp, DevWS ws, int hidden,
               const float* __restrict__ WgQ, const float* __restrict__ bias, int E, int k, int renorm,
               float scale, int32_t* __restrict__ hist, FrGeom geo, uint32_t go_token,
               int64_t go_timeout_ns) {
  constexpr int WPT = 16 / EPW;          // warps per team (one tile)
  // kSpread: row r of every block is routed by CTA r mod C (small fan-ins,
  // whose plan needs no histograms: every top-k warp takes about one
  // token); else each block has one owner CTA in rotation, which also
  // writes the block's expert histogram
  constexpr int TEAMS = kFrWarps / WPT;  // tiles in flight per CTA
  constexpr int BPI = TEAMS / 2;         // blocks per cluster iteration
  constexpr int CHUNK = WPT * 32 * 8;    // h per staged chunk: one 8-h group per team thread
  static_assert(EPW == 4 || EPW == 8, "4 or 8 experts per warp");
  // go_token != 0 (host-described steps): started before the header check
  // ends (see k_router_logits_tw2); the wait on the check moves to the exit
  struct ExitWait {
    bool on;
    __device__ ~ExitWait() {
      if (on) grid_dep_wait();
    }
  } exit_wait{go_token != 0};
  if (!go_token) grid_dep_wait();
  // the plan kernel after this one is let in only as this grid's warps
  // finish: its CTA resident from the start (waiting on this grid)
  // measured 7 us per decode layer slower, as did starting without the go
  // token
  const FanIn& f = step_item<kDev>(fp, ws.item);
  if (!WgQ) {  // the layer of the step was chosen on the device
    WgQ = ws.layers[f.layer].WgQ;
    bias = ws.layers[f.layer].bias;
  }
  extern __shared__ __align__(128) uint8_t fr_smem[];
  __shared__ int skipv[kFrMaxC];
  __shared__ int skip_s;
  __shared__ int abort_s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = geo.C, ep = geo.ep;
  const uint32_t rank = fr_ctarank();
  const int cid = (int)blockIdx.x / C, ncl = (int)gridDim.x / C;
  const int e_base = (int)rank * 16;
  const int ne = min(16, E - e_base);
  const int T = f.total;
  const int nblocks = (T + kFrBlk - 1) / kFrBlk;
  const uint32_t bar0 = smem_u32(fr_smem + geo.bar_off);
  const uint32_t wbar = bar0;
  auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)(1 + s); };
  auto empty_bar = [&](int q, int s) { return bar0 + 8u * (uint32_t)(1 + kFrSlots + q * kFrSlots + s); };
  float* lb = reinterpret_cast<float*>(fr_smem + geo.lb_off);  // [kFrSlots][16][ep]
  // rows of a block this CTA routes, and the bytes its buffer receives per block
  const int my_rows = kSpread ? (kFrBlk - (int)rank + C - 1) / C : kFrBlk;
  const uint32_t block_bytes = (uint32_t)(my_rows * E * 4);
  int* hs = reinterpret_cast<int*>(fr_smem + geo.hist_off);    // [kFrSlots][ep]
  if (tid == 0) {
    abort_s = 0;
    mbar_init(wbar, 1);
    for (int s = 0; s < kFrSlots; s++) mbar_init(full_bar(s), 1);
    for (int q = 0; q < C; q++)
      for (int s = 0; s < kFrSlots; s++) mbar_init(empty_bar(q, s), 1);
    // each logit buffer is armed (its one arrival and the block's bytes:
    // 16 tokens x E logits) before any peer may send into it, here for its
    // first use and by the top-k warps before each later one
    for (int s = 0; s < kFrSlots; s++) mbar_expect_tx(full_bar(s), block_bytes);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const uint32_t wbytes = (uint32_t)(((ne + 3) / 4) * hidden * 16);
    mbar_expect_tx(wbar, wbytes);
    bulk_load(smem_u32(fr_smem), WgQ + (int64_t)e_base * hidden, wbytes, wbar);
  }
  for (int i = tid; i < kFrSlots * ep; i += blockDim.x) hs[i] = 0;
  __syncthreads();
  // this CTA has started and its barriers are initialised
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  if (tid == 0) {
    int ok = 1;
    if (go_token) {  // the header check hands over the fan-in (bounded)
      const uint64_t t0 = globaltimer_ns();
      ok = 0;
      for (;;) {
        const uint32_t v = ld_acquire_u32(ws.go);
        if (v == go_token) { ok = 1; break; }
        if (v == (go_token | AFD_GO_ABORT)) break;  // the check reports the error
        if (globaltimer_ns() - t0 > (uint64_t)go_timeout_ns) {
          set_error(ws.status, AFD_ERR_TIMEOUT);
          break;
        }
        __nanosleep(64);
      }
    }
    skip_s = !ok || read_status(ws.status);
  }
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every peer has started
  // the skip decision is the cluster's: each CTA's into every CTA
  if (tid < C)
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(fr_mapa(smem_u32(&skipv[rank]), (uint32_t)tid)),
                 "r"(skip_s)
                 : "memory");
  fr_cluster_sync();
  int skip = 0;
  for (int q = 0; q < C; q++) skip |= skipv[q];
  if (skip) {  // the whole cluster leaves; nothing was exchanged
    if (tid == 0) {  // the weight copy lands in this CTA's shared memory: wait (bounded)
      const uint64_t dl = globaltimer_ns() + 100000000ull;
      while (!mbar_try_wait(wbar, 0) && globaltimer_ns() < dl) {}
    }
    return;
  }
  // a wait that runs out records the error once; later waits give up fast
  auto waitb = [&](uint32_t bar, uint32_t parity, uint64_t start) {
    uint32_t spins = 0;
    while (!fr_try_wait(bar, parity)) {
      if ((++spins & 63u) == 0) {
        const uint64_t lim = *(volatile int*)&abort_s ? 1000000ull : 1000000000ull;
        if (globaltimer_ns() - start > lim) {
          if (atomicExch(&abort_s, 1) == 0) set_error(ws.status, AFD_ERR_TIMEOUT);
          return false;
        }
      }
    }
    return true;
  };
  if (warp < kFrWarps) {
    // ------------------------------------------------------------ compute
    const int m = warp / WPT, wt = warp % WPT;
    const int team_tid = tid - m * WPT * 32;
    const int bar_id = 2 + m;
    uint8_t* rec = fr_smem + geo.rec_off + (size_t)m * 2 * geo.rec_bytes;
    const float4* Wq = reinterpret_cast<const float4*>(fr_smem);  // [4 groups][hidden]
    const int grp0 = EPW == 8 ? 2 * wt : wt;
    const int row_bytes = hidden * 2;
    const int nch = (hidden + CHUNK - 1) / CHUNK;
    auto block_of = [&](int it) { return (cid + ncl * it) * BPI + m / 2; };
    const uint8_t* rows[8];
    uint4 pre[8];
    auto set_rows = [&](int it) {  // the tile's token rows, straight from the peer slots
      const int t0 = (2 * block_of(it) + (m & 1)) * 8;
#pragma unroll
      for (int r = 0; r < 8; r++) {
        const int t = t0 + r;
        rows[r] = nullptr;
        if (t < T) {
          const int e = entry_of(f, t);
          rows[r] = slot_ptr(win, g, f.region[e], f.stage) + g.routed_x + (int64_t)(t - f.prefix[e]) * row_bytes;
        }
      }
    };
    auto fetch = [&](int c) {  // this thread's 8-h group of chunk c, 8 tokens (zeros past the fan-in)
      const int h = c * CHUNK + team_tid * 8;
#pragma unroll
      for (int r = 0; r < 8; r++)
        pre[r] = (rows[r] && h < hidden) ? __ldg(reinterpret_cast<const uint4*>(rows[r] + (int64_t)h * 2))
                                         : make_uint4(0, 0, 0, 0);
    };
    if (block_of(0) < nblocks) {  // the first chunk's loads fly while the weights land
      set_rows(0);
      fetch(0);
    }
    waitb(wbar, 0, globaltimer_ns());
    int cc = 0;  // chunks consumed by this team
    for (int it = 0; block_of(it) < nblocks; it++) {
      float2 acc[4][EPW];  // {token 2p, token 2p + 1} x expert
#pragma unroll
      for (int p = 0; p < 4; p++)
#pragma unroll
        for (int b = 0; b < EPW; b++) acc[p][b] = make_float2(0.0f, 0.0f);
      for (int c = 0; c < nch; c++, cc++) {
        uint8_t* xt = rec + (size_t)(cc & 1) * geo.rec_bytes;
        if (c * CHUNK + team_tid * 8 < hidden) {  // [t][8 h] -> records [h][8 t]
          const uint32_t* iw[8];
#pragma unroll
          for (int t = 0; t < 8; t++) iw[t] = reinterpret_cast<const uint32_t*>(&pre[t]);
#pragma unroll
          for (int j = 0; j < 8; j++) {
            const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
            uint4 o;
            o.x = __byte_perm(iw[0][j >> 1], iw[1][j >> 1], sel);
            o.y = __byte_perm(iw[2][j >> 1], iw[3][j >> 1], sel);
            o.z = __byte_perm(iw[4][j >> 1], iw[5][j >> 1], sel);
            o.w = __byte_perm(iw[6][j >> 1], iw[7][j >> 1], sel);
            *reinterpret_cast<uint4*>(xt + tw_rec_offset(8 * team_tid + j)) = o;
          }
        }
        // records complete; every warp of the team is past the chunk that
        // used the other buffer
        named_bar_sync(bar_id, WPT * 32);
        if (c + 1 < nch) {
          fetch(c + 1);
        } else if (block_of(it + 1) < nblocks) {
          set_rows(it + 1);
          fetch(0);
        }
        if (!*(volatile int*)&abort_s) {
          const int h0 = c * CHUNK, len = min(CHUNK, hidden - h0);
          auto step = [&](int hh) {
            const uint4 xr = *reinterpret_cast<const uint4*>(xt + tw_rec_offset(hh));
            float wv[EPW];
            {
              const float4 w0 = Wq[(size_t)grp0 * hidden + h0 + hh];
              wv[0] = w0.x; wv[1] = w0.y; wv[2] = w0.z; wv[3] = w0.w;
              if constexpr (EPW == 8) {
                const float4 w1 = Wq[(size_t)(grp0 + 1) * hidden + h0 + hh];
                wv[4] = w1.x; wv[5] = w1.y; wv[6] = w1.z; wv[7] = w1.w;
              }
            }
            const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w};
#pragma unroll
            for (int p = 0; p < 4; p++) {
              const float2 xp = make_float2(__uint_as_float(xw[p] << 16), __uint_as_float(xw[p] & 0xffff0000u));
#pragma unroll
              for (int b = 0; b < EPW; b++) acc[p][b] = __ffma2_rn(xp, make_float2(wv[b], wv[b]), acc[p][b]);
            }
          };
          const int nfull = len / 32;
#pragma unroll 4
          for (int j = 0; j < nfull; j++) step(32 * j + lane);
          if (32 * nfull + lane < len) step(32 * nfull + lane);
        }
      }
      // the tile's 8 x EPW logits: lane l ends with one (two) of them
      float va[32];
#pragma unroll
      for (int p = 0; p < 4; p++)
#pragma unroll
        for (int b = 0; b < EPW; b++) {
          if (EPW * 2 * p + b < 32) va[EPW * 2 * p + b] = acc[p][b].x;
          if (EPW * (2 * p + 1) + b < 32) va[EPW * (2 * p + 1) + b] = acc[p][b].y;
        }
      const float sum_a = butterfly_scatter32(va, lane);  // token lane / EPW, expert lane % EPW
      float sum_b = 0.0f;                                 // EPW 8: token 4 + lane / 8
      if constexpr (EPW == 8) {
        float vb[32];
#pragma unroll
        for (int p = 2; p < 4; p++)
#pragma unroll
          for (int b = 0; b < 8; b++) {
            vb[8 * (2 * p) + b - 32] = acc[p][b].x;
            vb[8 * (2 * p + 1) + b - 32] = acc[p][b].y;
          }
        sum_b = butterfly_scatter32(vb, lane);
      }
      // to the CTA that routes each row: the block's owner, or row mod C
      const int lblk = it * BPI + m / 2;
      const int owner = lblk % C;
      const int s = kSpread ? lblk % kFrSlots : (lblk / C) % kFrSlots;
      const uint32_t use = (uint32_t)(kSpread ? lblk / kFrSlots : (lblk / C) / kFrSlots);
      bool ok = true;
      if (lane == 0) {  // every receiving CTA has given this buffer back
        if (kSpread) {
          for (int q = 0; q < C && ok; q++) ok = waitb(empty_bar(q, s), (use & 1u) ^ 1u, globaltimer_ns());
        } else {
          ok = waitb(empty_bar(owner, s), (use & 1u) ^ 1u, globaltimer_ns());
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (ok) {
        const int el = EPW * wt + (lane % EPW);
        const int e = e_base + el;
        if (el < ne) {
          const float bv = bias ? bias[e] : 0.0f;
          auto send = [&](int row, float sum) {
            const int q = kSpread ? row % C : owner;
            const float v = bias ? __fadd_rn(sum, bv) : sum;
            fr_st_async(fr_mapa(smem_u32(lb + ((size_t)s * 16 + row) * ep + e), (uint32_t)q), v,
                        fr_mapa(full_bar(s), (uint32_t)q));
          };
          const int row_a = (m & 1) * 8 + lane / EPW;
          send(row_a, sum_a);
          if constexpr (EPW == 8) send(row_a + 4, sum_b);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ top-k
    const int tw = warp - kFrWarps;
    const int ttid = tid - kFrWarps * 32;
    for (int lblk = kSpread ? 0 : (int)rank;; lblk += kSpread ? 1 : C) {
      const int it = lblk / BPI, j = lblk % BPI;
      const int b = (cid + ncl * it) * BPI + j;
      if (b >= nblocks) break;
      const int s = kSpread ? lblk % kFrSlots : (lblk / C) % kFrSlots;
      const uint32_t use = (uint32_t)(kSpread ? lblk / kFrSlots : (lblk / C) / kFrSlots);
      const bool ok = waitb(full_bar(s), use & 1u, globaltimer_ns()) && !*(volatile int*)&abort_s;
      if (ok) {
#pragma unroll 1
        for (int i = tw; i < my_rows; i += TK) {
          const int r = kSpread ? (int)rank + C * i : i;
          const int t = b * kFrBlk + r;
          if (t >= T) break;
          float lv[4];
#pragma unroll
          for (int mm = 0; mm < 4; mm++) {
            const int e = lane + 32 * mm;
            lv[mm] = e < E ? lb[((size_t)s * 16 + r) * ep + e] : -INFINITY;
          }
          int my_id;
          float my_w;
          route_token<4>(lv, E, k, renorm, scale, lane, my_id, my_w);
          if (lane < k) {
            ws.ids[(int64_t)t * k + lane] = my_id;
            ws.w[(int64_t)t * k + lane] = my_w;
            atomicAdd(&hs[s * ep + my_id], 1);
          }
        }
      }
      named_bar_sync(1, TK * 32);  // the buffer is read, the histogram complete
      for (int e = ttid; e < E; e += TK * 32) {
        if (!kSpread && hist && !*(volatile int*)&abort_s) hist[(int64_t)b * E + e] = hs[s * ep + e];
        hs[s * ep + e] = 0;
      }
      // armed for its next use, then back to the producers of every CTA
      if (ttid == 0) mbar_expect_tx(full_bar(s), block_bytes);
      named_bar_sync(1, TK * 32);
      if (ttid < C) fr_arrive_remote(fr_mapa(empty_bar((int)rank, s), (uint32_t)ttid));
    }
  }
  // each warp lets the next kernel in once its part is done (the compute
  // warps before the top-k warps); after the CTA barrier instead measured
  // 7 us per decode layer slower
  grid_dep_launch();
  __syncthreads();
  fr_cluster_sync();  // no peer sends to or signals this CTA past this point
}

// ---------------------------------------------------------------------------
// a2 plan for larger fan-ins (one CTA): per-expert counts and exclusive
// offsets from the router blocks' histograms (bincount + cumsum, Async GPU
// Connector, "Data flow" step 1), each router block's base position within
// each expert's segment (base[b][e] = sum of hist[b'][e] for b' < b), the
// zeroed per-peer counts, and the tile tables of both grouped GEMMs; the
// stable ranks follow in k_rank_gather.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Tile tables of both grouped GEMMs from the per-expert counts and offsets:
// the shared expert's group(s) over its rows, then one group per expert
// (rows = its partials, in permuted order); tile0 / unit0 are prefixes of
// the one-CTA tiles and of the SM-pair units.
// Called by one whole warp: lane l takes a contiguous run of at most
// ceil(E / 32) experts (<= 8), and every group's first tile and unit are
// warp prefix sums, so the tables equal those of a walk in group order.
// The shared expert's groups come first: their units are the heaviest of
// the down GEMM (K = shared_inter), so the units go out largest first and
// the light routed units fill the end (shared groups last measured slower:
// prefill 1.479 -> 1.483 ms, decode 6.46 -> 6.58 ms per 26 layers).
__device__ void write_tile_tables(const FanIn& f, const DevWS& ws, const WinGeom& g, int row_bytes,
                                  int k, int E, int inter, int shared_inter, int hidden,
                                  int has_shared, int sh_in_place, int bn, const int* cnt,
                                  const int* offs, GemmPlan* plan1, GemmPlan* plan2) {
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int N = f.grouped ? f.rtotal : f.total * k;  // routed rows (Xp rows 0..N-1)
  const int mt1 = (inter + 63) / 64, mt2 = (hidden + 127) / 128;
  const int u1_per = (mt1 + 1) / 2, u2_per = (mt2 + 1) / 2;
  int tiles1 = 0, tiles2 = 0, units1 = 0, units2 = 0, ng = 0;
  int ntiles = 0;  // token tiles of the groups so far (dependency counters of the one-launch GEMMs)
  // the shared expert: one group over the gathered shared rows (Xp rows
  // N..), or one group per entry that sent shared rows, read in place from
  // its slot's shared_x (window rows); outputs at the shared-row offsets
  const int mts = (shared_inter + 63) / 64;
  const int us_per = (mts + 1) / 2;
  if (has_shared && !sh_in_place) {
    const int rows = f.stotal;
    const int nt = (rows + bn - 1) / bn;
    if (lane == 0) {
      plan1->g[0] = GemmGroup{rows, N, 0, 0, 1, mts, nt, 0, 0, 0};
      plan2->g[0] = GemmGroup{rows, 0, 0, 0, 1, mt2, nt, 0, 0, 0};
    }
    tiles1 = mts * nt;
    tiles2 = mt2 * nt;
    units1 = us_per * nt;
    units2 = u2_per * nt;
    ntiles = nt;
    ng = 1;
  }
  if (has_shared && sh_in_place) {
    for (int r0 = 0; r0 < f.n_peers; r0 += 32) {  // entries in rounds of 32, in list order
      const int i = r0 + lane;
      const int rows = (i < f.n_peers && ws.peer_shared[i]) ? f.sprefix[i + 1] - f.sprefix[i] : 0;
      const unsigned has = __ballot_sync(0xffffffffu, rows > 0);
      const int nt = (rows + bn - 1) / bn;
      const int nt_incl = warp_incl_scan(nt, lane);
      const int nt_before = nt_incl - nt;
      if (rows > 0) {
        const int gi = ng + __popc(has & lt_mask);
        const int wr = window_row(g, f.region[i], f.stage, g.shared_x, 0, row_bytes);
        plan1->g[gi] = GemmGroup{rows, wr, f.sprefix[i], 0, 1, mts, nt, tiles1 + mts * nt_before,
                                 units1 + us_per * nt_before, ntiles + nt_before};
        plan2->g[gi] = GemmGroup{rows, f.sprefix[i], f.sprefix[i], 0, 1, mt2, nt,
                                 tiles2 + mt2 * nt_before, units2 + u2_per * nt_before, ntiles + nt_before};
      }
      const int nt_round = __shfl_sync(0xffffffffu, nt_incl, 31);
      tiles1 += mts * nt_round;
      tiles2 += mt2 * nt_round;
      units1 += us_per * nt_round;
      units2 += u2_per * nt_round;
      ntiles += nt_round;
      ng += __popc(has);
    }
  }
  // one group per expert, after the shared groups
  const int epl = (E + 31) / 32;
  const int e0 = min(E, lane * epl), e1 = min(E, e0 + epl);
  int nts = 0;  // token tiles of this lane's experts
  for (int e = e0; e < e1; e++) nts += (cnt[e] + bn - 1) / bn;
  const int nts_incl = warp_incl_scan(nts, lane);
  int nt_run = nts_incl - nts;  // token tiles of the experts before this lane's
  for (int e = e0; e < e1; e++) {
    const int rows = cnt[e];
    const int nt = (rows + bn - 1) / bn;
    plan1->g[ng + e] = GemmGroup{rows, offs[e], offs[e], e, 0, mt1, nt, tiles1 + mt1 * nt_run,
                                 units1 + u1_per * nt_run, ntiles + nt_run};
    plan2->g[ng + e] = GemmGroup{rows, offs[e], offs[e], e, 0, mt2, nt, tiles2 + mt2 * nt_run,
                                 units2 + u2_per * nt_run, ntiles + nt_run};
    nt_run += nt;
  }
  const int nt_all = __shfl_sync(0xffffffffu, nts_incl, 31);
  if (lane == 0) {
    plan1->ngroups = ng + E;
    plan2->ngroups = ng + E;
    plan1->total_tiles = tiles1 + mt1 * nt_all;
    plan2->total_tiles = tiles2 + mt2 * nt_all;
    plan1->total_units = units1 + u1_per * nt_all;
    plan2->total_units = units2 + u2_per * nt_all;
    plan1->total_ntiles = plan2->total_ntiles = ntiles + nt_all;
    plan1->bn = bn;
    plan2->bn = bn;
  }
  // the one-launch GEMMs count each token tile's finished SwiGLU units here
  for (int i = lane; i < ntiles + nt_all; i += 32) ws.dep[i] = 0;
}

constexpr int kScanWarps = 32;
constexpr int kScanSegs = kScanWarps * 32 / 64;  // 16 segments x 64 experts per pass

template <bool kDev>
__global__ void __launch_bounds__(kScanWarps * 32)
k_plan_scan(const __grid_constant__ FanIn fp, DevWS ws, int E, int k, int inter, int shared_inter, int hidden,
            int has_shared, int bn, const int32_t* __restrict__ hist, int32_t* __restrict__ base,
            GemmPlan* plan1, GemmPlan* plan2, WinGeom g, int row_bytes, int sh_in_place) {
  grid_dep_wait();
  grid_dep_launch();
  const FanIn& f = step_item<kDev>(fp, ws.item);
  __shared__ int cnt[256];
  __shared__ int offs[257];
  __shared__ int skip;
  const int tid = threadIdx.x;
  if (tid == 0) skip = read_status(ws.status);
  __syncthreads();
  if (skip) return;
  // 64 experts per pass; thread = (segment sg of the router CTAs, expert),
  // so a warp's loads of one CTA's histogram row are contiguous
  __shared__ int seg_sum[kScanSegs][64];
  const int sg = tid / 64, el = tid % 64;
  const int nblocks = (f.total + kRtTok - 1) / kRtTok;  // router CTAs of this step
  const int L = (nblocks + kScanSegs - 1) / kScanSegs;
  const int b_lo = min(nblocks, sg * L), b_hi = min(nblocks, b_lo + L);
  for (int e0 = 0; e0 < E; e0 += 64) {
    const int e = e0 + el;
    int sum = 0;
    if (e < E) {
      int b = b_lo;
      for (; b + 8 <= b_hi; b += 8) {  // 8 loads in flight
        int v[8];
#pragma unroll
        for (int u = 0; u < 8; u++) v[u] = hist[(int64_t)(b + u) * E + e];
#pragma unroll
        for (int u = 0; u < 8; u++) sum += v[u];
      }
      for (; b < b_hi; b++) sum += hist[(int64_t)b * E + e];
    }
    seg_sum[sg][el] = sum;
    __syncthreads();
    int run = 0;
    for (int q = 0; q < sg; q++) run += seg_sum[q][el];
    if (e < E) {
      for (int b = b_lo; b < b_hi; b++) {
        const int v = hist[(int64_t)b * E + e];
        base[(int64_t)b * E + e] = run;
        run += v;
      }
      if (sg == kScanSegs - 1) cnt[e] = run;
    }
    __syncthreads();
  }
  for (int i = tid; i < f.n_peers * E; i += blockDim.x) ws.peer_counts[i] = 0;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < E; e++) {
      offs[e] = run;
      run += cnt[e];
    }
    offs[E] = run;
  }
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) {
    ws.offsets[e] = offs[e];
    if (e < E) ws.counts[e] = cnt[e];
  }
  if (tid < 32)
    write_tile_tables(f, ws, g, row_bytes, k, E, inter, shared_inter, hidden, has_shared,
                      sh_in_place, bn, cnt, offs, plan1, plan2);
}

// ---------------------------------------------------------------------------
// a2/a3 plan for small fan-ins (T*k <= kPlanSmallMax, e.g. decode): one CTA
// does the counts, offsets, per-peer counts, the stable permutation (warp w
// owns a contiguous chunk of f; per-warp histograms give its cursor per
// expert; 32-element rounds are ranked with match_any) and the tile tables.
// ---------------------------------------------------------------------------
constexpr int kPlanPerLane = kPlanSmallMax / 1024;  // ids per lane: a warp's chunk is <= 256

template <bool kDev>
__global__ void __launch_bounds__(1024)
k_plan_small(const __grid_constant__ FanIn fp, DevWS ws, int E, int k, int inter, int shared_inter, int hidden,
             int has_shared, int bn, GemmPlan* plan1, GemmPlan* plan2, WinGeom g, int row_bytes,
             int sh_in_place) {
  grid_dep_wait();
  grid_dep_launch();
  const FanIn& f = step_item<kDev>(fp, ws.item);
  __shared__ int hist_w[32][256];
  __shared__ int cnt[256];
  __shared__ int offs[257];
  __shared__ int skip;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = f.total * k;
  const int chunk = (N + 31) / 32;
  const int c0 = min(N, warp * chunk), c1 = min(N, c0 + chunk);
  const int nr = (c1 - c0 + 31) / 32;  // 32-entry rounds of this warp (<= kPlanPerLane)
  // the warp's expert ids, loaded once (one round trip, the status word's
  // load alongside) and kept in registers for both passes
  int ev[kPlanPerLane];
#pragma unroll
  for (int j = 0; j < kPlanPerLane; j++) {
    const int fi = c0 + 32 * j + lane;
    ev[j] = fi < c1 ? ws.ids[fi] : 0;
  }
  if (tid == 0) skip = read_status(ws.status);
  for (int i = tid; i < 32 * 256; i += blockDim.x) (&hist_w[0][0])[i] = 0;
  for (int i = tid; i < f.n_peers * E; i += blockDim.x) ws.peer_counts[i] = 0;
  __syncthreads();
  if (skip) return;
#pragma unroll
  for (int j = 0; j < kPlanPerLane; j++) {
    const int fi = c0 + 32 * j + lane;
    if (fi < c1) {
      if (ev[j] < 0 || ev[j] >= E) {  // cannot come from the router; keep every index in range
        set_error(ws.status, AFD_ERR_SHAPE);
        ev[j] = 0;
        ws.ids[fi] = 0;
      }
      atomicAdd(&hist_w[warp][ev[j]], 1);
      atomicAdd(&ws.peer_counts[entry_of(f, fi / k) * E + ev[j]], 1);
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int c = 0;
    for (int w = 0; w < 32; w++) c += hist_w[w][e];
    cnt[e] = c;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive offsets: lane l scans a run of <= 8 experts
    const int epl = (E + 31) / 32;
    const int e0 = min(E, lane * epl), e1 = min(E, e0 + epl);
    int sum = 0;
    for (int e = e0; e < e1; e++) sum += cnt[e];
    const int incl = warp_incl_scan(sum, lane);
    int run = incl - sum;
    for (int e = e0; e < e1; e++) { offs[e] = run; run += cnt[e]; }
    if (lane == 31) offs[E] = incl;
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int base = offs[e];
    for (int w = 0; w < 32; w++) {
      const int c = hist_w[w][e];
      hist_w[w][e] = base;  // warp w's cursor for expert e
      base += c;
    }
  }
  for (int e = tid; e <= E; e += blockDim.x) {
    ws.offsets[e] = offs[e];
    if (e < E) ws.counts[e] = cnt[e];
  }
  __syncthreads();
  // stable ranks: rounds of 32 entries in order, ties within a round ranked
  // by lane (match_any)
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < kPlanPerLane; j++) {
    if (j < nr) {
      const int fi = c0 + 32 * j + lane;
      const bool ok = fi < c1;
      const int e = ok ? ev[j] : -1 - lane;
      const unsigned same = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(same & lt_mask);
      int pos = 0;
      if (ok) pos = hist_w[warp][e] + rank;
      __syncwarp();
      if (ok && rank == 0) hist_w[warp][e] += __popc(same);
      __syncwarp();
      if (ok) {
        ws.perm[pos] = fi;
        ws.inv[fi] = pos;
      }
    }
  }
  if (tid < 32)
    write_tile_tables(f, ws, g, row_bytes, k, E, inter, shared_inter, hidden, has_shared,
                      sh_in_place, bn, cnt, offs, plan1, plan2);
}

// ---------------------------------------------------------------------------
// Plan of the grouped form (the Attention side routed; [RFC]: Async GPU
// Connector, "Data flow" steps 1-3): the entries' group lists (from their
// headers) give the per-expert counts and offsets; entry i's rows of expert e
// go, in arrival order, after the same expert's rows of the entries before
// it (stable in list order).  One CTA.
// ---------------------------------------------------------------------------
template <bool kDev>
__global__ void __launch_bounds__(1024)
k_plan_grouped(const __grid_constant__ FanIn fp, DevWS ws, int E, int inter, int shared_inter, int hidden, int has_shared,
               int bn, GemmPlan* plan1, GemmPlan* plan2, WinGeom g, int row_bytes, int in_place,
               int sh_in_place) {
  grid_dep_wait();
  grid_dep_launch();
  const FanIn& f = step_item<kDev>(fp, ws.item);
  __shared__ int cnt[256];
  __shared__ int offs[257];
  __shared__ int skip;
  const int tid = threadIdx.x;
  if (tid == 0) skip = read_status(ws.status);
  __syncthreads();
  if (skip) return;
  const int P = f.n_peers;
  int* base = ws.gbase;                       // [P][E] first position of entry i's expert-e rows
  int* gpre = ws.gbase + AFD_MAX_PEERS * E;   // [P][E] first row of expert e within entry i
  for (int e = tid; e < E; e += blockDim.x) {
    int c = 0;
    for (int i = 0; i < P; i++) c += ws.peer_counts[i * E + e];
    cnt[e] = c;
  }
  for (int i = tid; i < P; i += blockDim.x) {
    int r = 0;
    for (int e = 0; e < E; e++) {
      gpre[i * E + e] = r;
      r += ws.peer_counts[i * E + e];
    }
  }
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < E; e++) { offs[e] = run; run += cnt[e]; }
    offs[E] = run;
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int b = offs[e];
    for (int i = 0; i < P; i++) {
      base[i * E + e] = b;
      b += ws.peer_counts[i * E + e];
    }
  }
  for (int e = tid; e <= E; e += blockDim.x) {
    ws.offsets[e] = offs[e];
    if (e < E) ws.counts[e] = cnt[e];
  }
  __syncthreads();
  if (!in_place) {  // the gather places each row (and records perm / inv)
    if (tid < 32)
      write_tile_tables(f, ws, g, row_bytes, 1, E, inter, shared_inter, hidden, has_shared,
                        sh_in_place, bn, cnt, offs, plan1, plan2);
    return;
  }
  // the entries' group lists in shared memory for the one-thread table walk
  // (in place: n_peers * E <= AFD_MAX_GROUPS)
  __shared__ int gl_s[AFD_MAX_GROUPS];
  for (int x = tid; x < f.n_peers * E && x < AFD_MAX_GROUPS; x += blockDim.x) gl_s[x] = ws.peer_counts[x];
  __syncthreads();
  if (tid != 0) return;
  // In place: one group per (entry, expert) with rows, whose rows are
  // contiguous in the entry's dispatch slot (the SwiGLU GEMM reads them
  // there, the down GEMM writes their outputs straight into the entry's
  // return slot), then one shared group per entry with shared rows (read
  // from its shared_x, outputs into its return shared_x).  h / hs rows
  // follow the groups' order.
  int tiles1 = 0, tiles2 = 0, units1 = 0, units2 = 0, ng = 0, hrow = 0, ntiles = 0;
  const int mt1 = (inter + 63) / 64, mt2 = (hidden + 127) / 128;
  for (int i = 0; i < f.n_peers; i++)
    for (int e = 0, lr0 = 0; e < E; lr0 += gl_s[i * E + e], e++) {
      const int rows = gl_s[i * E + e];
      if (!rows) continue;
      const int nt = (rows + bn - 1) / bn;
      GemmGroup a{rows, window_row(g, f.region[i], f.stage, g.routed_x, lr0, row_bytes), hrow, e, 0,
                  mt1, nt, tiles1, units1, ntiles};
      GemmGroup b{rows, hrow, window_row(g, f.region[i], f.stage, g.routed_x, lr0, row_bytes), e, 0,
                  mt2, nt, tiles2, units2, ntiles};
      plan1->g[ng] = a;
      plan2->g[ng] = b;
      tiles1 += mt1 * nt;
      tiles2 += mt2 * nt;
      units1 += (mt1 + 1) / 2 * nt;
      units2 += (mt2 + 1) / 2 * nt;
      hrow += rows;
      ntiles += nt;
      ng++;
    }
  if (has_shared)
    for (int i = 0; i < f.n_peers; i++) {
      const int rows = ws.peer_shared[i] ? f.sprefix[i + 1] - f.sprefix[i] : 0;
      if (!rows) continue;
      const int nt = (rows + bn - 1) / bn;
      const int mts = (shared_inter + 63) / 64;
      const int wr = window_row(g, f.region[i], f.stage, g.shared_x, 0, row_bytes);
      GemmGroup a{rows, wr, f.sprefix[i], 0, 1, mts, nt, tiles1, units1, ntiles};
      GemmGroup b{rows, f.sprefix[i], wr, 0, 1, mt2, nt, tiles2, units2, ntiles};
      plan1->g[ng] = a;
      plan2->g[ng] = b;
      tiles1 += mts * nt;
      tiles2 += mt2 * nt;
      units1 += (mts + 1) / 2 * nt;
      units2 += (mt2 + 1) / 2 * nt;
      ntiles += nt;
      ng++;
    }
  plan1->ngroups = plan2->ngroups = ng;
  plan1->total_tiles = tiles1;
  plan2->total_tiles = tiles2;
  plan1->total_units = units1;
  plan2->total_units = units2;
  plan1->total_ntiles = plan2->total_ntiles = ntiles;
  plan1->bn = plan2->bn = bn;
  for (int i = 0; i < ntiles; i++) ws.dep[i] = 0;
}


// ---------------------------------------------------------------------------
// Shared row r - N of the step (entries in list order), one warp: copied from
// its slot's shared_x into Xp row r, or zeros for an entry that sent no
// shared rows; when the shared expert reads its rows in place, only the s
// rows of such entries are zeroed here (the combine adds s for every token).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void gather_shared_row(const uint8_t* win, const WinGeom& g, const FanIn& f,
                                                  const DevWS& ws, int r, int N, int row_bytes, int hidden,
                                                  int sh_in_place) {
  const int lane = threadIdx.x & 31;
  const int t = r - N;
  const int i = entry_of_shared(f, t);
  if (sh_in_place) {
    if (!ws.peer_shared[i]) {
      float4* srow = reinterpret_cast<float4*>(ws.s + (int64_t)t * hidden);
      for (int v = lane; v < hidden / 4; v += 32) srow[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  const int nvec = row_bytes / 16;
  uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(ws.xp) + (int64_t)r * row_bytes);
  if (!ws.peer_shared[i]) {
    for (int v = lane; v < nvec; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(slot_ptr(win, g, f.region[i], f.stage) + g.shared_x +
                                                    (int64_t)(t - f.sprefix[i]) * row_bytes);
  for (int v = lane; v < nvec; v += 32) dst[v] = __ldg(src + v);
}

// ---------------------------------------------------------------------------
// a3 gather: Xp[pos] = the row of token perm[pos] / k, read straight from its
// peer slot (the fan-in concatenation is never materialised), then the
// shared rows in concatenation order.  One warp per row, 16-byte vectors:
// small token-form fan-ins (their rows stay in L2; a warp per position
// spreads the copies over many warps) and the grouped form.
// ---------------------------------------------------------------------------
template <bool kDev>
__global__ void __launch_bounds__(kThreads)
k_gather(const uint8_t* win, WinGeom g, const __grid_constant__ FanIn fp, DevWS ws, int k, int row_bytes,
         int hidden, int has_shared, int sh_in_place, uint8_t* ret_headers, int E) {
  grid_dep_wait();
  grid_dep_launch();
  const FanIn& f = step_item<kDev>(fp, ws.item);
  if (read_status(ws.status)) return;
  if (ret_headers) {  // the combine releases the flags: the return headers now, counters zeroed
    for (int i = blockIdx.x; i < f.n_peers; i += gridDim.x) {
      write_return_header(ret_headers, g, f, ws, E, k, i);
      if (threadIdx.x == 0) ws.ret_count[i] = 0;
    }
  }
  const int N = f.grouped ? f.rtotal : f.total * k;
  const int rows = N + (has_shared ? f.stotal : 0);
  const int nvec = row_bytes / 16;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  for (int r = wid; r < rows; r += warps) {
    if (r >= N) {
      gather_shared_row(win, g, f, ws, r, N, row_bytes, hidden, sh_in_place);
      continue;
    }
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(ws.xp) + (int64_t)r * row_bytes);
    int i, local;
    if (f.grouped) {
      // source row r of the entries' concatenation goes to position
      // base[i][e] + (its row within the entry's expert-e group)
      i = entry_of_rows(f, r);
      local = r - f.rprefix[i];
      const int E = f.num_experts;
      const int* gp = ws.gbase + AFD_MAX_PEERS * E + i * E;
      int lo = 0, hi = E - 1;  // the last expert whose first row is <= local (not empty)
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (gp[mid] <= local) lo = mid; else hi = mid - 1;
      }
      int pos = ws.gbase[i * E + lo] + (local - gp[lo]);
      if (!dbg_in_range(ws.dbg, ws.status, AFD_DBG_GATHER_GROUPED, pos, N)) pos = 0;
      dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(ws.xp) + (int64_t)pos * row_bytes);
      if ((threadIdx.x & 31) == 0) {
        ws.perm[pos] = r;
        ws.inv[r] = pos;
      }
    } else {
      int pr = ws.perm[r];
      if (!dbg_in_range(ws.dbg, ws.status, AFD_DBG_GATHER_PERM, pr, N)) pr = 0;
      const int t = pr / k;
      i = entry_of(f, t);
      local = t - f.prefix[i];
    }
    const uint4* src = reinterpret_cast<const uint4*>(slot_ptr(win, g, f.region[i], f.stage) + g.routed_x +
                                                      (int64_t)local * row_bytes);
    for (int v = (threadIdx.x & 31); v < nvec; v += 32) dst[v] = __ldg(src + v);
  }
}

// ---------------------------------------------------------------------------
// a2 + a3 for large token-form fan-ins: the stable permutation and the
// gather in one launch, one CTA per 16-token router block.  While every warp
// loads its two tokens' rows from their slots, the first warp ranks the
// block's partials: position = offsets[e] + base[b][e] (the plan's exclusive
// bases from the router's block histograms) + the rank among the block's
// earlier partials of e (match_any over 32-partial rounds), i.e. a stable
// argsort of the flattened ids; it records perm / inv and the per-peer
// counts.  After one barrier each row goes to its k positions, so every
// token row leaves HBM once (walking the positions instead read each row k
// times, far apart, and L2 kept few of them: 3.2x the rows' bytes came from
// DRAM at the V2-Lite prefill shape).  Then the shared rows, as k_gather.
// ---------------------------------------------------------------------------
constexpr int kRgWarps = kRtTok / 2;  // two tokens per warp

template <bool kDev>
__global__ void __launch_bounds__(kRgWarps * 32)
k_rank_gather(const uint8_t* win, WinGeom g, const __grid_constant__ FanIn fp, DevWS ws, int E, int k,
              const int32_t* __restrict__ base, int row_bytes, int hidden, int has_shared, int sh_in_place) {
  grid_dep_wait();
  grid_dep_launch();
  const FanIn& f = step_item<kDev>(fp, ws.item);
  __shared__ int run_s[256];
  __shared__ int pos_s[kRtTok * 16];  // [token of the block][j], k <= 16
  __shared__ int skip_s;
  if (threadIdx.x == 0) skip_s = read_status(ws.status);
  __syncthreads();  // one decision for the CTA: its loop has barriers
  if (skip_s) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = f.total, N = T * k;
  const int nblocks = (T + kRtTok - 1) / kRtTok;
  const int nvec = row_bytes / 16;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int b = blockIdx.x; b < nblocks; b += gridDim.x) {
    // this warp's two tokens: the first 8 vectors per lane of each row in flight
    const uint4* src[2];
    uint4 buf[2][8];
#pragma unroll
    for (int q = 0; q < 2; q++) {
      const int t = b * kRtTok + 2 * warp + q;
      src[q] = nullptr;
      if (t < T) {
        const int i = entry_of(f, t);
        src[q] = reinterpret_cast<const uint4*>(slot_ptr(win, g, f.region[i], f.stage) + g.routed_x +
                                                (int64_t)(t - f.prefix[i]) * row_bytes);
      }
#pragma unroll
      for (int u = 0; u < 8; u++) {
        const int v = 32 * u + lane;
        buf[q][u] = (src[q] && v < nvec) ? __ldg(src[q] + v) : make_uint4(0, 0, 0, 0);
      }
    }
    if (warp == 0) {
      for (int e = lane; e < E; e += 32) run_s[e] = ws.offsets[e] + base[(int64_t)b * E + e];
      __syncwarp();
      const int f0 = b * kRtTok * k, f1 = min(N, f0 + kRtTok * k);
      for (int g0 = f0; g0 < f1; g0 += 32) {
        const int fi = g0 + lane;
        const bool ok = fi < f1;
        int e = ok ? ws.ids[fi] : -1 - lane;
        if (ok && (e < 0 || e >= E)) {  // cannot come from the router; keep every index in range
          set_error(ws.status, AFD_ERR_SHAPE);
          e = 0;
        }
        const unsigned same = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(same & lt_mask);
        int pos = 0;
        if (ok) pos = run_s[e] + rank;
        __syncwarp();
        if (ok && rank == 0) run_s[e] += __popc(same);
        __syncwarp();
        if (ok) {
          pos_s[fi - f0] = pos;
          ws.perm[pos] = fi;
          ws.inv[fi] = pos;
          atomicAdd(&ws.peer_counts[entry_of(f, fi / k) * E + e], 1);
        }
      }
    }
    __syncthreads();  // the block's positions
#pragma unroll
    for (int q = 0; q < 2; q++) {
      if (!src[q]) continue;
      const int tb = 2 * warp + q;
      for (int v0 = 0; v0 < nvec; v0 += 32 * 8) {
        if (v0 > 0) {  // rows past 256 vectors: the next pass
#pragma unroll
          for (int u = 0; u < 8; u++) {
            const int v = v0 + 32 * u + lane;
            buf[q][u] = v < nvec ? __ldg(src[q] + v) : make_uint4(0, 0, 0, 0);
          }
        }
        for (int j = 0; j < k; j++) {
          int pos = pos_s[tb * k + j];
          if (!dbg_in_range(ws.dbg, ws.status, AFD_DBG_GATHER_INV, pos, N)) pos = 0;
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(ws.xp) + (int64_t)pos * row_bytes);
#pragma unroll
          for (int u = 0; u < 8; u++) {
            const int v = v0 + 32 * u + lane;
            if (v < nvec) dst[v] = buf[q][u];
          }
        }
      }
    }
    __syncthreads();  // run_s and pos_s are free for the next block
  }
  if (has_shared) {
    const int warps = gridDim.x * kRgWarps, wid = blockIdx.x * kRgWarps + warp;
    for (int r = N + wid; r < N + f.stotal; r += warps)
      gather_shared_row(win, g, f, ws, r, N, row_bytes, hidden, sh_in_place);
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
  grid_dep_wait();
  grid_dep_launch();
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
  if (a.layers) {  // the layer of the step was chosen on the device
    const DevLayer& L = a.layers[a.item->layer];
    A = a.wsel == 1 ? (kind ? L.W13s : L.W13) : (kind ? L.Wds : L.Wd);
  }
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
    if (!dbg_in_range(a.dbg, a.status, AFD_DBG_GEMM_OUT, (int64_t)G.out_row0 + r, a.out_rows[kind])) continue;
    const int64_t o = (int64_t)(G.out_row0 + r) * a.ldo[kind] + c;
    if (a.out_fmt[kind] == OUT_F32) {
      reinterpret_cast<float*>(a.out[kind])[o] = v;
    } else if (a.out_fmt[kind] == OUT_Y24) {
      const uint32_t b24 = y24_encode(v);
      reinterpret_cast<uint16_t*>(a.out[kind])[o] = (uint16_t)(b24 >> 8);
      a.out_lo[kind][o] = (uint8_t)(b24 & 0xffu);
    } else {
      reinterpret_cast<__nv_bfloat16*>(a.out[kind])[o] = __float2bfloat16_rn(v);
    }
  }
}

// ---------------------------------------------------------------------------
// a7 combine + split: out[t] = sum_{j ascending} w[t,j] * y[inv[t,j]] + s[t]
// in fp32 (fused multiply-add in j order, then + s), rounded to the
// activation type and written straight into the return slot of t's peer at
// its local row; the route_table row gets the chosen ids.  y and s are fp32
// (the weighted sum may cancel to far less than its terms, so they are
// rounded only once, here).  Deterministic: each output element is reduced
// by one thread in a fixed order.
// ---------------------------------------------------------------------------
template <bool ACT_F32, int kBatch, bool kDev, bool kFlags = false>
__global__ void __launch_bounds__(kThreads)
k_combine(uint8_t* ret, WinGeom g, const __grid_constant__ FanIn fp, DevWS ws, int hidden, int k, int has_shared) {
  // y: fp32 with fp32 activations, else the 24-bit planes (OUT_Y24).
  // kFlags (small fan-ins, one item per warp, every entry with tokens): the
  // gather wrote the return headers; the warp that finishes an entry's last
  // item releases its return flag (a counter per entry), so no return-header
  // kernel follows
  grid_dep_wait();
  grid_dep_launch();
  const FanIn& f = step_item<kDev>(fp, ws.item);
  if (read_status(ws.status)) return;
  // 8 features per lane step: two 16-byte loads of a partial's fp32 row,
  // or 16 bytes of its high plane and 8 of its low plane
  constexpr int kVec = 8;
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const float* __restrict__ y = reinterpret_cast<const float*>(ws.y);
  const uint16_t* __restrict__ y_hi = reinterpret_cast<const uint16_t*>(ws.y);
  const uint8_t* __restrict__ y_lo = ws.y_lo;
  // work item = (token, block of 256 features): a small fan-in still spreads
  // over every SM
  const int nfb = (hidden + 32 * kVec - 1) / (32 * kVec);
  const int64_t items = (int64_t)f.total * nfb;
  for (int64_t it = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items; it += warps) {
    const int t = (int)(it / nfb), fb = (int)(it % nfb);
    const int i = entry_of(f, t);
    const int local = t - f.prefix[i];
    uint8_t* slot = slot_ptr(ret, g, f.region[i], f.stage);
    int my_pos = 0;
    float my_w = 0.0f;
    if (lane < k) {
      my_pos = ws.inv[(int64_t)t * k + lane];
      if (!dbg_in_range(ws.dbg, ws.status, AFD_DBG_COMBINE_INV, my_pos, (int64_t)f.total * k)) my_pos = 0;
      my_w = ws.w[(int64_t)t * k + lane];
      if (fb == 0)
        reinterpret_cast<int32_t*>(slot + g.route_table)[(int64_t)local * k + lane] =
            ws.ids[(int64_t)t * k + lane];
    }
    // every lane takes part in the shuffles; lanes past hidden skip memory
    const int c0 = fb * 32 * kVec + lane * kVec;
    const bool valid = c0 < hidden;
    const int c = valid ? c0 : 0;
    float acc[kVec];
#pragma unroll
    for (int q = 0; q < kVec; q++) acc[q] = 0.0f;
    // rounds of up to kBatch partials: their rows are all loaded before the
    // multiply-adds, which still run in ascending j (8 for small fan-ins,
    // where few warps must keep many loads in flight; 4 for large ones; 1
    // for fp32 activations)
    for (int j0 = 0; j0 < k; j0 += kBatch) {
      uint4 raw[kBatch][2];  // fp32: two 16-byte words; y24: high plane, low plane (8 bytes)
      float wj[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; u++) {
        const int j = j0 + u;
        const int pos = __shfl_sync(0xffffffffu, my_pos, j & 31);
        wj[u] = __shfl_sync(0xffffffffu, my_w, j & 31);
        const bool ld = valid && j < k;
        const int64_t e0 = (int64_t)pos * hidden + c;
        if constexpr (ACT_F32) {
          const uint4* src = reinterpret_cast<const uint4*>(y + e0);
          raw[u][0] = ld ? src[0] : make_uint4(0, 0, 0, 0);
          raw[u][1] = ld ? src[1] : make_uint4(0, 0, 0, 0);
        } else {
          raw[u][0] = ld ? *reinterpret_cast<const uint4*>(y_hi + e0) : make_uint4(0, 0, 0, 0);
          const uint2 l = ld ? *reinterpret_cast<const uint2*>(y_lo + e0) : make_uint2(0, 0);
          raw[u][1] = make_uint4(l.x, l.y, 0, 0);
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; u++) {
        if (j0 + u >= k) break;
        float yv[kVec];
        if constexpr (ACT_F32) {
          const uint32_t w8[kVec] = {raw[u][0].x, raw[u][0].y, raw[u][0].z, raw[u][0].w,
                                     raw[u][1].x, raw[u][1].y, raw[u][1].z, raw[u][1].w};
#pragma unroll
          for (int q = 0; q < kVec; q++) yv[q] = __uint_as_float(w8[q]);
        } else {
          const uint32_t hw[4] = {raw[u][0].x, raw[u][0].y, raw[u][0].z, raw[u][0].w};
          const uint32_t lw[2] = {raw[u][1].x, raw[u][1].y};
#pragma unroll
          for (int q = 0; q < kVec; q++) {
            const uint32_t hi = (q & 1) ? (hw[q >> 1] >> 16) : (hw[q >> 1] & 0xffffu);
            const uint32_t lo = (lw[q >> 2] >> (8 * (q & 3))) & 0xffu;
            yv[q] = y24_decode(hi, lo);
          }
        }
#pragma unroll
        for (int q = 0; q < kVec; q++) acc[q] = __fmaf_rn(wj[u], yv[q], acc[q]);
      }
    }
    if (valid) {  // lanes past hidden write nothing
      if (has_shared) {  // zero rows for peers that sent no shared rows
        const float4* sp = reinterpret_cast<const float4*>(ws.s + (int64_t)t * hidden + c);
        const float4 a = sp[0], b = sp[1];
        acc[0] = __fadd_rn(acc[0], a.x); acc[1] = __fadd_rn(acc[1], a.y);
        acc[2] = __fadd_rn(acc[2], a.z); acc[3] = __fadd_rn(acc[3], a.w);
        acc[4] = __fadd_rn(acc[4], b.x); acc[5] = __fadd_rn(acc[5], b.y);
        acc[6] = __fadd_rn(acc[6], b.z); acc[7] = __fadd_rn(acc[7], b.w);
      }
      if constexpr (ACT_F32) {
        float4* dst = reinterpret_cast<float4*>(slot + g.routed_x + ((int64_t)local * hidden + c) * 4);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      } else {
        uint4 o;
        __nv_bfloat162 p0 = __floats2bfloat162_rn(acc[0], acc[1]);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(acc[2], acc[3]);
        __nv_bfloat162 p2 = __floats2bfloat162_rn(acc[4], acc[5]);
        __nv_bfloat162 p3 = __floats2bfloat162_rn(acc[6], acc[7]);
        o.x = *reinterpret_cast<uint32_t*>(&p0);
        o.y = *reinterpret_cast<uint32_t*>(&p1);
        o.z = *reinterpret_cast<uint32_t*>(&p2);
        o.w = *reinterpret_cast<uint32_t*>(&p3);
        *reinterpret_cast<uint4*>(slot + g.routed_x + ((int64_t)local * hidden + c) * 2) = o;
      }
    }
    if constexpr (kFlags) {
      __threadfence();  // this item's rows (and route-table row) before its count
      __syncwarp();
      if (lane == 0) {
        const int items_i = (f.prefix[i + 1] - f.prefix[i]) * nfb;
        if (atomicAdd(&ws.ret_count[i], 1) == items_i - 1) {
          __threadfence();  // every item of the entry is counted: its payload is out
          st_release_u64(return_flag(ret, g, f, i), ws.cur_seq[i]);
        }
      }
    }
  }
}

// Grouped form, the way back ([RFC]: Async GPU Connector, "Data flow" step 4:
// the Attention side weights and combines): the expert output of every
// received row into its peer's return slot in arrival order (routed_x), and
// the shared expert's outputs (shared_x, rounded to the activation type).
// One warp per row.
template <bool ACT_F32, bool kDev>
__global__ void __launch_bounds__(kThreads)
k_scatter_grouped(uint8_t* ret, WinGeom g, const __grid_constant__ FanIn fp, DevWS ws, int hidden, int has_shared) {
  grid_dep_wait();
  grid_dep_launch();
  const FanIn& f = step_item<kDev>(fp, ws.item);
  if (read_status(ws.status)) return;
  constexpr int kEl = ACT_F32 ? 4 : 2;
  const int row_bytes = hidden * kEl;
  const int rows = f.rtotal + (has_shared ? f.stotal : 0);
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    if (r < f.rtotal) {
      const int i = entry_of_rows(f, r);
      int pos = ws.inv[r];
      if (!dbg_in_range(ws.dbg, ws.status, AFD_DBG_SCATTER_INV, pos, f.rtotal)) pos = 0;
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(ws.y) +
                                                        (int64_t)pos * row_bytes);
      uint4* dst = reinterpret_cast<uint4*>(slot_ptr(ret, g, f.region[i], f.stage) + g.routed_x +
                                            (int64_t)(r - f.rprefix[i]) * row_bytes);
      for (int v = lane; v < row_bytes / 16; v += 32) dst[v] = src[v];
    } else {
      const int t = r - f.rtotal;
      const int i = entry_of_shared(f, t);
      if (!ws.peer_shared[i]) continue;
      const float* src = ws.s + (int64_t)t * hidden;
      uint8_t* dst = slot_ptr(ret, g, f.region[i], f.stage) + g.shared_x +
                     (int64_t)(t - f.sprefix[i]) * row_bytes;
      for (int c = lane * 8; c < hidden; c += 32 * 8) {
        const float4 a = *reinterpret_cast<const float4*>(src + c);
        const float4 b = *reinterpret_cast<const float4*>(src + c + 4);
        if constexpr (ACT_F32) {
          reinterpret_cast<float4*>(dst + (int64_t)c * 4)[0] = a;
          reinterpret_cast<float4*>(dst + (int64_t)c * 4)[1] = b;
        } else {
          __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
          __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
          uint4 o;
          o.x = *reinterpret_cast<uint32_t*>(&p0);
          o.y = *reinterpret_cast<uint32_t*>(&p1);
          o.z = *reinterpret_cast<uint32_t*>(&p2);
          o.w = *reinterpret_cast<uint32_t*>(&p3);
          *reinterpret_cast<uint4*>(dst + (int64_t)c * 2) = o;
        }
      }
    }
  }
}

// return headers, then the return flags (release) = the dispatch seq
template <bool kDev>
__global__ void k_return_header(uint8_t* ret, WinGeom g, const __grid_constant__ FanIn fp, DevWS ws, int E, int k) {
  grid_dep_wait();
  grid_dep_launch();
  const FanIn& f = step_item<kDev>(fp, ws.item);
  if (read_status(ws.status)) return;
  const int i = blockIdx.x;
  if (i >= f.n_peers) return;
  write_return_header(ret, g, f, ws, E, k, i);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    st_release_u64(return_flag(ret, g, f, i), ws.cur_seq[i]);
  }
}

// Unpack: block-local bounded wait on the return flag and header check by
// thread 0, then the block copies its share of the rows.
// thread 0 of the CTA: bounded wait for the return flag of (region, stage)
// to reach expect_seq, then the header checks; the CTA's verdict in *ok
__device__ void unpack_check(const uint8_t* ret, const WinGeom& g, int region, int stage, int E,
                             uint64_t expect_seq, int32_t* status, int64_t timeout_ns,
                             int expect_tokens, int expect_routed, int* ok) {
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
        else if (h[7] != expect_tokens || (expect_routed >= 0 && h[8] != expect_routed))
          e = AFD_ERR_SHAPE;
      }
      if (e > 0) set_error(status, e);
    }
    *ok = (e == 0);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads)
k_unpack(const uint8_t* ret, WinGeom g, int region, int stage, uint4* out, int n, int row_bytes,
         int E, uint64_t expect_seq, int32_t* status, int64_t timeout_ns, int64_t field,
         int expect_tokens, int expect_routed) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int ok;
  unpack_check(ret, g, region, stage, E, expect_seq, status, timeout_ns, expect_tokens, expect_routed, &ok);
  if (!ok) return;
  const uint4* src = reinterpret_cast<const uint4*>(slot_ptr(ret, g, region, stage) + field);
  const int64_t nvec = (int64_t)n * row_bytes / 16;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec;
       v += (int64_t)gridDim.x * blockDim.x)
    out[v] = src[v];
}

// Several peers' unpacks (afd_unpack_splits): CTA row y = entry y, each CTA
// checks its entry's flag and header, then copies its share of the rows.
__global__ void __launch_bounds__(kThreads)
k_unpack_multi(const uint8_t* ret, WinGeom g, int stage, const __grid_constant__ UnpackList ul, int row_bytes,
               int E, int32_t* status, int64_t timeout_ns) {
  grid_dep_wait();
  grid_dep_launch();
  const int e = blockIdx.y;
  if (e >= ul.n) return;
  __shared__ int ok;
  unpack_check(ret, g, ul.region[e], stage, E, ul.seq[e], status, timeout_ns, ul.n_rows[e], -1, &ok);
  if (!ok) return;
  const uint4* src = reinterpret_cast<const uint4*>(slot_ptr(ret, g, ul.region[e], stage) + g.routed_x);
  uint4* out = ul.out[e];
  const int64_t nvec = (int64_t)ul.n_rows[e] * row_bytes / 16;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec;
       v += (int64_t)gridDim.x * blockDim.x)
    out[v] = src[v];
}

// L2 prefetch of a contiguous byte range (weights the next GEMM reads first):
// 64 KB bulk prefetches spread over the grid; returns as soon as they are issued.
__global__ void k_prefetch_l2(const uint8_t* base, int64_t bytes, DevWS ws) {
  grid_dep_wait();
  grid_dep_launch();
  if (!base) {  // the W13 of the layer the device chose for the step in flight
    if (read_status(ws.status)) return;
    const FanIn& f = *ws.item;
    if ((f.grouped ? f.rtotal : f.total) == 0) return;
    base = static_cast<const uint8_t*>(ws.layers[f.layer].W13);
    if (!base) return;
  }
  constexpr int64_t kChunk = 65536;
  const int64_t n = (bytes + kChunk - 1) / kChunk;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t len = min(kChunk, bytes - i * kChunk);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + i * kChunk), "r"((uint32_t)len)
                 : "memory");
  }
}

// Expert weights re-laid for the tensor engines: each 128-row x 64-column
// block (one TMA box, one k-block of one 128-row weight tile) becomes 16
// contiguous KB, ordered [expert][row tile][k-block], so a tile's k-blocks
// stream from HBM as one contiguous run.  Row r of a tile of the gate/up
// weight [E][2I][K] (swiglu) holds inter column 64 t + 16 (r / 32) + r % 16
// of the gate (r / 16 even) or up (odd) rows, the order in which the
// epilogue pairs them; the down weight [E][M][K] keeps its row order (row
// 128 t + r).  Rows and columns past the weight are zero (what the TMA's
// out-of-bounds fill gave on the plain layout).
__global__ void k_tile_weight(const uint16_t* __restrict__ src, uint4* __restrict__ dst, int E, int M, int K,
                              int swiglu, int I, int mtiles) {
  const int nkb = (K + 63) / 64;
  const int64_t total = (int64_t)E * mtiles * nkb * 128 * 8;  // 16-byte pieces
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int piece = (int)(i % 8);
    int64_t r = i / 8;
    const int row = (int)(r % 128);
    r /= 128;
    const int kb = (int)(r % nkb);
    r /= nkb;
    const int t = (int)(r % mtiles);
    const int e = (int)(r / mtiles);
    int srow;
    bool ok;
    if (swiglu) {
      const int j = 4 * t + row / 32;  // 16-column group of the inter dimension
      ok = j < I / 16;
      srow = ((row / 16) & 1) * I + 16 * j + row % 16;
    } else {
      srow = 128 * t + row;
      ok = srow < M;
    }
    uint16_t v[8];
#pragma unroll
    for (int q = 0; q < 8; q++) {
      const int k = 64 * kb + 8 * piece + q;
      v[q] = (ok && k < K) ? src[((int64_t)e * M + srow) * K + k] : (uint16_t)0;
    }
    dst[i] = make_uint4(v[0] | ((uint32_t)v[1] << 16), v[2] | ((uint32_t)v[3] << 16),
                        v[4] | ((uint32_t)v[5] << 16), v[6] | ((uint32_t)v[7] << 16));
  }
}

// The router weight [hidden][E] rearranged for the logits kernels as
// WgQ[E/4 groups][hidden][4 experts] fp32 (experts past E are zero): a lane
// reads the 4 weights of its h for a group of experts with one 16-byte load.
__global__ void k_arrange_wg(const float* Wg, float* WgQ, int hidden, int E) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t n = (int64_t)wgq_groups(E) * hidden * 4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int q = (int)(i & 3);
    const int h = (int)((i >> 2) % hidden);
    const int e = (int)(i / (4 * (int64_t)hidden)) * 4 + q;
    WgQ[i] = e < E ? Wg[(int64_t)h * E + e] : 0.0f;
  }
}

}  // namespace

int router_blocks(int total_tokens) { return (total_tokens + kRtTok - 1) / kRtTok; }

// shared memory of a logits CTA: 8 token rows
size_t router_min_smem_bytes(int hidden, int E, int act_f32) {
  (void)E;
  return (size_t)hidden * kLgTok * (act_f32 ? 4 : 2);
}

namespace {

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
// Canary words (AFD_CFG_CANARY): write the pattern into every guard word of
// a window, or count the words that differ from it.
__global__ void k_canary(uint8_t* win, CanaryGeom cg, int fill, unsigned long long* result) {
  const int64_t per_slot = (int64_t)cg.n * (cg.guard / 4);
  const int64_t flag_words = cg.guard / 4;
  const int64_t total = flag_words + per_slot * cg.nslots;
  for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < total;
       w += (int64_t)gridDim.x * blockDim.x) {
    int64_t off;
    if (w < flag_words) {
      off = cg.flags_bytes - cg.guard + 4 * w;
    } else {
      const int64_t v = w - flag_words;
      const int64_t slot = v / per_slot, r = v % per_slot;
      const int gi = (int)(r / (cg.guard / 4));
      off = cg.flags_bytes + slot * cg.slot_bytes + cg.goff[gi] + 4 * (r % (cg.guard / 4));
    }
    uint32_t* p = reinterpret_cast<uint32_t*>(win + off);
    if (fill) {
      *p = canary_word(off);
    } else if (*p != canary_word(off)) {
      atomicAdd(&result[0], 1ull);
      atomicMin(&result[1], (unsigned long long)off);
    }
  }
}

cudaError_t launch_canary(cudaStream_t stream, uint8_t* win, const CanaryGeom& cg, int fill,
                          unsigned long long* result, int num_sms) {
  k_canary<<<num_sms * 4, kThreads, 0, stream>>>(win, cg, fill, result);
  return cudaGetLastError();
}

cudaError_t launch_pack_payload(const LaunchCtx& lc, const WinGeom& g, uint8_t* win, int region,
                                int stage, const void* rows, int n_rows, const void* xs, int n_shared,
                                int row_bytes) {
  const int64_t work = (int64_t)std::max(n_rows, xs ? n_shared : 0) * row_bytes / 16;
  if (work == 0) return cudaSuccess;
  return launch_k(lc, k_pack_payload, grid_for(work, kThreads * 4, lc.num_sms * 8), kThreads, 0,
                  win, g, region, stage, reinterpret_cast<const uint4*>(rows), n_rows,
                  reinterpret_cast<const uint4*>(xs), n_shared, row_bytes);
}

cudaError_t launch_pack_header(const LaunchCtx& lc, const WinGeom& g, uint8_t* win, int region,
                               int stage, int layer, int n, int with_shared, int num_experts,
                               uint64_t seq, int shutdown, int routed_tokens, const GroupList& gl) {
  return launch_k(lc, k_pack_header, 1, 128, 0, win, g, region, stage, layer, n, with_shared,
                  num_experts, seq, shutdown, routed_tokens, gl);
}

cudaError_t launch_header_check(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                                const FanIn& f, const DevWS& ws, int num_experts, int token_cap,
                                int rows_cap, int has_shared_expert, int64_t timeout_ns,
                                uint32_t go_token) {
  return launch_k(lc, k_header_check, 1, 1024, 0, win, g, f, ws, num_experts, token_cap, rows_cap,
                  has_shared_expert, timeout_ns, go_token);
}

template <typename XS, bool kDev>
static cudaError_t launch_logits_t(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                                   const FanIn& f, const DevWS& ws, int hidden, const float* WgQ,
                                   const float* bias, int E, float* logits) {
  const size_t smem = (size_t)hidden * kLgTok * sizeof(XS);
  cudaError_t err = cudaFuncSetAttribute(k_router_logits<XS, kDev>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  dim3 grid((f.total + kLgTok - 1) / kLgTok, (E + kLgEblk - 1) / kLgEblk);
  return launch_k(lc, k_router_logits<XS, kDev>, grid, kLgWarps * 32, smem, win, g, f, ws, hidden,
                  WgQ, bias, E, logits);
}

// Shared memory of the weight-stationary logits kernel with 4 * epw experts
// per CTA; the ring takes 3 buffers, or 2 when 3 do not fit.  smem = 0: it
// does not fit at all.  (The 2048 bytes held back cover the kernels' static
// shared memory, the step's fan-in included.)
static WsGeom ws_geom(int hidden, int xs_bytes, int epw) {
  constexpr size_t kLimit = 232448 - 2048;
  WsGeom geo{};
  geo.w_bytes = ((size_t)((kWsWarps * epw + 3) / 4) * hidden * 16 + 127) / 128 * 128;
  geo.tile_bytes = (size_t)kWsTok * hidden * xs_bytes;
  for (int ns = 3; ns >= 2; ns--) {
    const size_t total = geo.w_bytes + ns * geo.tile_bytes + 8 * (ns + 1);
    if (total <= kLimit) {
      geo.ns = ns;
      geo.smem = total;
      return geo;
    }
  }
  geo.smem = 0;
  return geo;
}
static_assert(sizeof(FanIn) + 64 <= 2048, "static shared memory of the router kernels");

template <typename XS, int EPW, bool kDev>
static cudaError_t launch_logits_ws(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                                    const FanIn& f, const DevWS& ws, int hidden, const float* WgQ,
                                    const float* bias, int E, float* logits, const WsGeom& geo) {
  cudaError_t err = cudaFuncSetAttribute(k_router_logits_ws<XS, EPW, kDev>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.smem);
  if (err != cudaSuccess) return err;
  const int eblocks = (E + kWsWarps * EPW - 1) / (kWsWarps * EPW);
  const int ntiles = (f.total + kWsTok - 1) / kWsTok;
  // one CTA per SM (the weight block fills most of its shared memory)
  const int gx = std::max(1, std::min(ntiles, lc.num_sms / eblocks));
  return launch_k(lc, k_router_logits_ws<XS, EPW, kDev>, dim3(gx, eblocks), kWsWarps * 32, geo.smem,
                  win, g, f, ws, hidden, WgQ, bias, E, logits, geo);
}

static TwGeom tw_geom(int hidden) {
  constexpr size_t kLimit = 232448 - 2048;
  TwGeom geo{};
  geo.w_bytes = ((size_t)4 * hidden * 16 + 127) / 128 * 128;
  geo.stage_bytes = (size_t)kTwTok * hidden * 2;
  geo.xt_bytes = (tw_rec_offset(hidden) + 127) / 128 * 128;
  const size_t total = geo.w_bytes + geo.stage_bytes + geo.xt_bytes + 16;
  geo.smem = total <= kLimit ? total : 0;
  return geo;
}

template <typename XS, bool kDev>
static cudaError_t launch_logits(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                                 const FanIn& f, const DevWS& ws, int hidden, const float* WgQ,
                                 const float* bias, int E, float* logits, uint32_t go_token,
                                 int64_t go_timeout_ns) {
  if (sizeof(XS) == 2 && E >= 16 && hidden <= 8 * kTw2Chunks * kTwWarps * 32) {
    TwGeom geo = tw_geom(hidden);
    geo.stage_bytes = 0;  // no staging buffer; two record buffers
    geo.smem = geo.w_bytes + 2 * geo.xt_bytes + 16;
    if (geo.smem <= 232448 - 2048) {
      cudaError_t err = cudaFuncSetAttribute(k_router_logits_tw2<kDev>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.smem);
      if (err != cudaSuccess) return err;
      const int eblocks = (E + kTwExperts - 1) / kTwExperts;
      const int ntiles = (f.total + kTwTok - 1) / kTwTok;
      const int gx = std::max(1, std::min(ntiles, lc.num_sms / eblocks));
      return launch_k(lc, k_router_logits_tw2<kDev>, dim3(gx, eblocks), 2 * kTwWarps * 32, geo.smem,
                      win, g, f, ws, hidden, WgQ, bias, E, logits, geo, kDev ? 0u : go_token,
                      go_timeout_ns);
    }
  }
  if (sizeof(XS) == 2 && E >= 16) {
    const TwGeom geo = tw_geom(hidden);
    if (geo.smem) {
      cudaError_t err = cudaFuncSetAttribute(k_router_logits_tw<kDev>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.smem);
      if (err != cudaSuccess) return err;
      const int eblocks = (E + kTwExperts - 1) / kTwExperts;
      const int ntiles = (f.total + kTwTok - 1) / kTwTok;
      const int gx = std::max(1, std::min(ntiles, lc.num_sms / eblocks));
      return launch_k(lc, k_router_logits_tw<kDev>, dim3(gx, eblocks), kTwWarps * 32, geo.smem, win,
                      g, f, ws, hidden, WgQ, bias, E, logits, geo);
    }
  }
  // experts per warp: 4 when there are >= 16 experts, fewer for small E or
  // when the weight block and two token tiles do not fit
  for (int epw = E >= 16 ? 4 : (E >= 8 ? 2 : 1); epw >= 1; epw >>= 1) {
    const WsGeom geo = ws_geom(hidden, (int)sizeof(XS), epw);
    if (!geo.smem) continue;
    if (epw == 4)
      return launch_logits_ws<XS, 4, kDev>(lc, g, win, f, ws, hidden, WgQ, bias, E, logits, geo);
    if (epw == 2)
      return launch_logits_ws<XS, 2, kDev>(lc, g, win, f, ws, hidden, WgQ, bias, E, logits, geo);
    return launch_logits_ws<XS, 1, kDev>(lc, g, win, f, ws, hidden, WgQ, bias, E, logits, geo);
  }
  return launch_logits_t<XS, kDev>(lc, g, win, f, ws, hidden, WgQ, bias, E, logits);
}

static FrGeom fr_geom(int hidden, int E, int epw) {
  FrGeom g{};
  g.C = (E + 15) / 16;
  g.ep = g.C * 16;
  const int wpt = 16 / epw, teams = kFrWarps / wpt, chunk = wpt * 32 * 8;
  auto r128 = [](size_t v) { return (uint32_t)((v + 127) / 128 * 128); };
  g.rec_off = r128((size_t)4 * hidden * 16);  // 4 groups of 4 experts' weights
  g.rec_bytes = r128(tw_rec_offset(chunk));
  g.lb_off = g.rec_off + (uint32_t)teams * 2 * g.rec_bytes;
  g.hist_off = g.lb_off + (uint32_t)(kFrSlots * kFrBlk * g.ep * 4);
  g.bar_off = g.hist_off + (uint32_t)(kFrSlots * g.ep * 4);
  g.smem = g.bar_off + 8u * (1 + kFrSlots + kFrMaxC * kFrSlots);
  return g;
}

// Clusters of the fused router that fit the GPU at once (queried once per
// kernel and cluster shape); clusters beyond it would run in a second wave.
template <int EPW, bool kSpread, bool kDev>
static int fr_max_clusters(const FrGeom& geo, int num_sms) {
  static std::atomic<int> cached[kMaxCachedDevices][kFrMaxC + 1];
  const int d = current_device();
  if (d >= 0) {
    const int c = cached[d][geo.C].load(std::memory_order_relaxed);
    if (c) return c;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(geo.C * std::max(1, num_sms / geo.C)));
  cfg.blockDim = dim3((kFrWarps + 4) * 32);
  cfg.dynamicSmemBytes = geo.smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)geo.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_router_fused<EPW, kSpread, kDev>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = std::max(1, num_sms / geo.C);
  }
  if (d >= 0) cached[d][geo.C].store(n, std::memory_order_relaxed);
  return n;
}

template <int EPW, bool kSpread, bool kDev>
static cudaError_t launch_router_fused(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                                       const FanIn& f, const DevWS& ws, int hidden, const float* WgQ,
                                       const float* bias, int E, int k, int renorm, float scale,
                                       int32_t* hist, uint32_t go_token, int64_t go_timeout_ns) {
  const FrGeom geo = fr_geom(hidden, E, EPW);
  static std::atomic<int> attr_done[kMaxCachedDevices];
  const cudaError_t err = smem_attr_once(k_router_fused<EPW, kSpread, kDev>, 232448 - 2048, attr_done);
  if (err != cudaSuccess) return err;
  constexpr int BPI = kFrWarps * EPW / 16 / 2;
  const int nblocks = (f.total + kFrBlk - 1) / kFrBlk;
  const int ncl = std::max(1, std::min(fr_max_clusters<EPW, kSpread, kDev>(geo, lc.num_sms), (nblocks + BPI - 1) / BPI));
  return launch_k_cluster(lc, k_router_fused<EPW, kSpread, kDev>, dim3((unsigned)(ncl * geo.C)),
                          (kFrWarps + 4) * 32, geo.smem,
                          (unsigned)geo.C, win, g, f, ws, hidden, WgQ, bias, E, k, renorm, scale, hist, geo,
                          kDev ? 0u : go_token, go_timeout_ns);
}

// The fused router covers bf16 activations with hidden <= 2048 and at most
// 128 experts, when the caller takes the block histograms (the allocation-
// free entry point keeps the two-kernel router, whose top-k writes its
// failure sentinel).
static bool fused_router_fits(int hidden, int E, int act_f32, const int32_t* hist) {
  return !act_f32 && hist && E <= kFrMaxC * 16 && hidden <= 2048 &&
         fr_geom(hidden, E, 8).smem <= 232448 - 2048;
}

template <bool kDev>
static cudaError_t launch_router_t(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                                   const FanIn& f, const DevWS& ws, int hidden, int act_f32,
                                   const float* WgQ, const float* bias, int E, int k, int renorm,
                                   float scale, float* logits, int32_t* hist, uint32_t go_token,
                                   int64_t go_timeout_ns) {
  if (fused_router_fits(hidden, E, act_f32, hist)) {
    // small fan-ins (planned by one CTA, no histograms): 4 experts per warp
    // and every block's rows routed across the cluster, since the latency
    // of one tile decides; larger ones: 8 experts per warp (fewer
    // non-multiply instructions per multiply-add) and a block owner that
    // writes the block's histogram.  The same test as the plan's choice.
    if ((int64_t)f.total * k <= kPlanSmallMax)
      return launch_router_fused<4, true, kDev>(lc, g, win, f, ws, hidden, WgQ, bias, E, k, renorm, scale,
                                                hist, go_token, go_timeout_ns);
    return launch_router_fused<8, false, kDev>(lc, g, win, f, ws, hidden, WgQ, bias, E, k, renorm, scale,
                                               hist, go_token, go_timeout_ns);
  }
  cudaError_t err =
      act_f32 ? launch_logits<float, kDev>(lc, g, win, f, ws, hidden, WgQ, bias, E, logits, go_token,
                                           go_timeout_ns)
              : launch_logits<uint16_t, kDev>(lc, g, win, f, ws, hidden, WgQ, bias, E, logits, go_token,
                                              go_timeout_ns);
  if (err != cudaSuccess) return err;
  const int nblocks = router_blocks(f.total);
  return launch_k(lc, k_router_topk<kDev>, nblocks, kRtTok * 32, 0, f, ws, logits, E, k, renorm,
                  scale, hist, nblocks);
}

cudaError_t launch_router(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                          const FanIn& f, const DevWS& ws, int hidden, int act_f32,
                          const float* WgQ, const float* bias, int E, int k, int renorm,
                          float scale, float* logits, int32_t* hist, uint32_t go_token,
                          int64_t timeout_ns) {
  if (f.total == 0) return cudaSuccess;
  // the router's own bound on ws.go: the check's flag waits plus a margin
  const int64_t go_timeout_ns = timeout_ns + 100000000;
  return f.dev ? launch_router_t<true>(lc, g, win, f, ws, hidden, act_f32, WgQ, bias, E, k, renorm,
                                       scale, logits, hist, 0, 0)
               : launch_router_t<false>(lc, g, win, f, ws, hidden, act_f32, WgQ, bias, E, k,
                                        renorm, scale, logits, hist, go_token, go_timeout_ns);
}

template <bool kDev>
static cudaError_t launch_plan_t(const LaunchCtx& lc, const FanIn& f, const DevWS& ws, int E,
                                 int k, int inter, int shared_inter, int hidden, int has_shared,
                                 int bn, GemmPlan* plan1, GemmPlan* plan2, const int32_t* hist,
                                 int32_t* base, const WinGeom& g, int row_bytes, int sh_in_place) {
  if ((int64_t)f.total * k <= kPlanSmallMax) {
    return launch_k(lc, k_plan_small<kDev>, 1, 1024, 0, f, ws, E, k, inter, shared_inter, hidden,
                    has_shared, bn, plan1, plan2, g, row_bytes, sh_in_place);
  }
  // larger fan-ins: counts, offsets, bases and tables here; the ranks with
  // the gather (k_rank_gather)
  (void)hist;
  return launch_k(lc, k_plan_scan<kDev>, 1, kScanWarps * 32, 0, f, ws, E, k, inter, shared_inter,
                  hidden, has_shared, bn, hist, base, plan1, plan2, g, row_bytes, sh_in_place);
}

cudaError_t launch_plan(const LaunchCtx& lc, const FanIn& f, const DevWS& ws, int E, int k,
                        int inter, int shared_inter, int hidden, int has_shared, int bn,
                        GemmPlan* plan1, GemmPlan* plan2, const int32_t* hist, int32_t* base,
                        const WinGeom& g, int row_bytes, int sh_in_place) {
  return f.dev ? launch_plan_t<true>(lc, f, ws, E, k, inter, shared_inter, hidden, has_shared, bn,
                                     plan1, plan2, hist, base, g, row_bytes, sh_in_place)
               : launch_plan_t<false>(lc, f, ws, E, k, inter, shared_inter, hidden, has_shared, bn,
                                      plan1, plan2, hist, base, g, row_bytes, sh_in_place);
}

cudaError_t launch_gather(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                          const FanIn& f, const DevWS& ws, int k, int row_bytes, int hidden,
                          int has_shared, int sh_in_place, uint8_t* ret_headers, int E,
                          const int32_t* base) {
  const int64_t rows = (int64_t)f.total * k + (has_shared ? f.total : 0);
  if (rows == 0) return cudaSuccess;
  if (!f.grouped && (int64_t)f.total * k > kPlanSmallMax) {  // the ranks too (the plan left them)
    const int nblocks = router_blocks(f.total);
    return launch_k(lc, f.dev ? k_rank_gather<true> : k_rank_gather<false>,
                    std::max(1, std::min(nblocks, lc.num_sms * 8)), kRgWarps * 32, 0, win, g, f, ws, E, k,
                    base, row_bytes, hidden, has_shared, sh_in_place);
  }
  return launch_k(lc, f.dev ? k_gather<true> : k_gather<false>,
                  grid_for(rows, kThreads / 32, lc.num_sms * 8), kThreads, 0, win, g, f, ws, k,
                  row_bytes, hidden, has_shared, sh_in_place, ret_headers, E);
}

cudaError_t launch_gemm_simt(const LaunchCtx& lc, const SimtArgs& a, int max_groups) {
  dim3 grid(lc.num_sms * 2, max_groups);
  return launch_k(lc, k_gemm_simt, grid, kThreads, 0, a);
}

cudaError_t launch_combine(const LaunchCtx& lc, const WinGeom& g, uint8_t* ret, const FanIn& f,
                           const DevWS& ws, int hidden, int k, int act_f32, int has_shared, int flags) {
  if (f.total == 0) return cudaSuccess;
  const int64_t items = (int64_t)f.total * ((hidden + 255) / 256);
  const int grid = grid_for(items, kThreads / 32, lc.num_sms * 8);
  const bool small = items < (int64_t)lc.num_sms * 64;
  const bool d = f.dev != 0;
  // y is fp32 (fp32 activations) or 24-bit (bf16) in the token form
  decltype(&k_combine<true, 1, false>) kern = nullptr;
  if (flags)
    kern = act_f32 ? k_combine<true, 1, false, true> : k_combine<false, 8, false, true>;
  else if (act_f32)
    kern = d ? k_combine<true, 1, true> : k_combine<true, 1, false>;
  else
    kern = small ? (d ? k_combine<false, 8, true> : k_combine<false, 8, false>)
                 : (d ? k_combine<false, 4, true> : k_combine<false, 4, false>);
  return launch_k(lc, kern, grid, kThreads, 0, ret, g, f, ws, hidden, k, has_shared);
}

// The combine can release the return flags itself when every warp gets at
// most one item (so counting items is cheap) and every entry has tokens
// (an entry without any would get no item): host-described token-form steps
// of small fan-ins.
bool combine_releases_flags(const LaunchCtx& lc, const FanIn& f, int hidden, int k) {
  if (f.dev || f.grouped || f.total == 0) return false;
  // larger fan-ins rank in the gather (k_rank_gather), so the per-peer
  // counts the return headers carry are final only after it: the
  // return-header kernel writes them
  if ((int64_t)f.total * k > kPlanSmallMax) return false;
  for (int i = 0; i < f.n_peers; i++)
    if (f.prefix[i + 1] == f.prefix[i]) return false;
  const int64_t items = (int64_t)f.total * ((hidden + 255) / 256);
  return items <= (int64_t)lc.num_sms * 8 * (kThreads / 32);
}

cudaError_t launch_return_header(const LaunchCtx& lc, const WinGeom& g, uint8_t* ret,
                                 const uint8_t*, const FanIn& f, const DevWS& ws, int E, int k) {
  return launch_k(lc, f.dev ? k_return_header<true> : k_return_header<false>, f.n_peers, 128, 0,
                  ret, g, f, ws, E, k);
}

cudaError_t launch_pack_multi(const LaunchCtx& lc, const WinGeom& g, uint8_t* win, int stage, int layer,
                              const PackList& pl, int with_shared, int row_bytes, int num_experts) {
  if (pl.n == 0) return cudaSuccess;
  int64_t most = 0;
  for (int e = 0; e < pl.n; e++) most = std::max<int64_t>(most, (int64_t)pl.n_rows[e] * row_bytes / 16);
  const int gx = std::max(1, grid_for(most, kThreads * 4, lc.num_sms * 4));
  cudaError_t err = launch_k(lc, k_pack_payload_multi, dim3((unsigned)gx, (unsigned)pl.n), kThreads, 0, win, g,
                             stage, pl, with_shared, row_bytes);
  if (err != cudaSuccess) return err;
  return launch_k(lc, k_pack_header_multi, pl.n, 128, 0, win, g, stage, layer, pl, with_shared, num_experts);
}

cudaError_t launch_unpack_multi(const LaunchCtx& lc, const WinGeom& g, const uint8_t* ret, int stage,
                                const UnpackList& ul, int row_bytes, int num_experts, int32_t* status,
                                int64_t timeout_ns) {
  if (ul.n == 0) return cudaSuccess;
  int64_t most = 0;
  for (int e = 0; e < ul.n; e++) most = std::max<int64_t>(most, (int64_t)ul.n_rows[e] * row_bytes / 16);
  const int gx = std::max(1, grid_for(most, kThreads * 4, lc.num_sms * 4));
  return launch_k(lc, k_unpack_multi, dim3((unsigned)gx, (unsigned)ul.n), kThreads, 0, ret, g, stage, ul,
                  row_bytes, num_experts, status, timeout_ns);
}

cudaError_t launch_unpack(const LaunchCtx& lc, const WinGeom& g, const uint8_t* ret, int region,
                          int stage, void* out, int n, int row_bytes, int num_experts,
                          uint64_t expect_seq, int32_t* status, int64_t timeout_ns, int64_t field,
                          int expect_tokens, int expect_routed) {
  const int64_t nvec = (int64_t)n * row_bytes / 16;
  return launch_k(lc, k_unpack, grid_for(nvec, kThreads * 4, lc.num_sms * 4), kThreads, 0, ret, g,
                  region, stage, reinterpret_cast<uint4*>(out), n, row_bytes, num_experts,
                  expect_seq, status, timeout_ns, field, expect_tokens, expect_routed);
}

cudaError_t launch_plan_grouped(const LaunchCtx& lc, const FanIn& f, const DevWS& ws, int E,
                                int inter, int shared_inter, int hidden, int has_shared, int bn,
                                GemmPlan* plan1, GemmPlan* plan2, const WinGeom& g, int row_bytes,
                                int in_place, int sh_in_place) {
  return launch_k(lc, f.dev ? k_plan_grouped<true> : k_plan_grouped<false>, 1, 1024, 0, f, ws, E,
                  inter, shared_inter, hidden, has_shared,
                  bn, plan1, plan2, g, row_bytes, in_place, sh_in_place);
}

cudaError_t launch_scatter_grouped(const LaunchCtx& lc, const WinGeom& g, uint8_t* ret,
                                   const FanIn& f, const DevWS& ws, int hidden, int act_f32,
                                   int has_shared) {
  const int64_t rows = (int64_t)f.rtotal + (has_shared ? f.total : 0);
  if (rows == 0) return cudaSuccess;
  const int grid = grid_for(rows, kThreads / 32, lc.num_sms * 8);
  const bool d = f.dev != 0;
  auto kern = act_f32 ? (d ? k_scatter_grouped<true, true> : k_scatter_grouped<true, false>)
                      : (d ? k_scatter_grouped<false, true> : k_scatter_grouped<false, false>);
  return launch_k(lc, kern, grid, kThreads, 0, ret, g, f, ws, hidden, has_shared);
}

cudaError_t launch_prefetch_l2(const LaunchCtx& lc, const void* base, int64_t bytes,
                               const DevWS& ws, int sms) {
  if (bytes <= 0) return cudaSuccess;
  return launch_k(lc, k_prefetch_l2, sms, 32, 0, static_cast<const uint8_t*>(base), bytes, ws);
}

cudaError_t launch_item_head(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                             const PeerList& pl, const DevWS& ws, int num_experts, int token_cap,
                             int rows_cap, int ffn_rank, int ffn_size, int has_shared_expert,
                             int grouped, int tmax, int rmax, int max_layers,
                             int64_t timeout_ns) {
  return launch_k(lc, k_item_head, 1, 1024, 0, win, g, pl, ws, num_experts, token_cap, rows_cap,
                  ffn_rank, ffn_size, has_shared_expert, grouped, tmax, rmax, max_layers,
                  timeout_ns);
}

int tiled_weight_tiles(int M, int swiglu, int I) { return swiglu ? (I / 16 + 3) / 4 : (M + 127) / 128; }

cudaError_t launch_tile_weight(const LaunchCtx& lc, const void* W, void* T, int E, int M, int K, int swiglu,
                               int I) {
  const int mtiles = tiled_weight_tiles(M, swiglu, I);
  const int64_t pieces = (int64_t)E * mtiles * ((K + 63) / 64) * 128 * 8;
  return launch_k(lc, k_tile_weight, grid_for(pieces, kThreads, 4096), kThreads, 0,
                  static_cast<const uint16_t*>(W), static_cast<uint4*>(T), E, M, K, swiglu, I, mtiles);
}

cudaError_t launch_arrange_wg(const LaunchCtx& lc, const float* Wg, float* WgQ, int hidden,
                              int E) {
  return launch_k(lc, k_arrange_wg, grid_for((int64_t)wgq_groups(E) * hidden * 4, kThreads, 1024),
                  kThreads, 0, Wg, WgQ, hidden, E);
}
