// afd_api.cu -- host side of the C ABI declared in include/afd.h: context,
// windows, workspace, TMA descriptors, argument checks and the launch
// sequence of the FFN step.
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>
#include <vector>

#include <algorithm>
#include <cmath>
#include <utility>

#include "afd_internal.cuh"

size_t gemm_tc_smem_bytes();

namespace {

struct LayerW {
  bool set = false;
  const float* Wg = nullptr;
  const float* bias = nullptr;
  const void* W13 = nullptr;
  const void* Wd = nullptr;
  const void* W13s = nullptr;
  const void* Wds = nullptr;
  float* WgQ = nullptr;              // library-owned rearranged router weight
  // library-owned tiled copies for the tensor engines: W13, Wd, W13_s, Wd_s
  void* T[4] = {nullptr, nullptr, nullptr, nullptr};
  size_t T_bytes[4] = {0, 0, 0, 0};
  CUtensorMap tmA1[2];               // SwiGLU projection: routed, shared
  CUtensorMap tmA2[2];               // down projection: routed, shared
};

int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }
int64_t gcd64(int64_t a, int64_t b) {
  while (b) { int64_t t = a % b; a = b; b = t; }
  return a;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_encoder() {
  if (g_encode) return AFD_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return AFD_ERR_CUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return AFD_OK;
}

// bf16 tensor map, 128-byte swizzle, zero fill out of bounds
int encode_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
               const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base),
                        dims, strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    fprintf(stderr, "afd: cuTensorMapEncodeTiled failed (%d), rank %d\n", (int)r, rank);
    return AFD_ERR_CUDA;
  }
  return AFD_OK;
}

// A tiled weight copy [E][tiles][k-blocks][128 rows][64 columns] as a 5-D
// map (column, row, k-block, tile, expert); one box = one 16 KB block, so a
// load's coordinates are (0, 0, k-block, 128-row tile, expert)
int encode_tiled_weight(CUtensorMap* m, const void* T, int E, int tiles, int K) {
  const cuuint64_t nkb = (cuuint64_t)((K + 63) / 64);
  const cuuint64_t dims[5] = {64, 128, nkb, (cuuint64_t)tiles, (cuuint64_t)E};
  const cuuint64_t str[4] = {128, 128 * 128, nkb * 16384, (cuuint64_t)tiles * nkb * 16384};
  const cuuint32_t box[5] = {64, 128, 1, 1, 1};
  return encode_map(m, T, 5, dims, str, box);
}

// [rows][K] token rows, box 64 x box_rows
int encode_rows(CUtensorMap* m, const void* X, int64_t rows, int K, int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)(rows > 0 ? rows : 1)};
  const cuuint64_t str[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  return encode_map(m, X, 2, dims, str, box);
}

int check_dev_ptr(const void* p) {
  if (!p) return AFD_ERR_ARG;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return AFD_ERR_NOT_DEVICE;
  }
  return (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) ? AFD_OK
                                                                              : AFD_ERR_NOT_DEVICE;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// routed rows a slot may carry: routed_cap under token-level dispatch
// (ceil(ceil(token_cap * topk / ffn_size) * multiplier)), else token_cap
int64_t routed_cap_of(const afd_config* c) {
  if (c->ffn_size < 1) return c->token_cap;
  const int64_t even = ((int64_t)c->token_cap * c->topk + c->ffn_size - 1) / c->ffn_size;
  return (int64_t)std::ceil((double)even * (double)c->routed_cap_multiplier);
}

int layout_of(const afd_config* c, afd_layout* L) {
  const int64_t ab = c->act_dtype == AFD_DTYPE_BF16 ? 2 : 4;
  const int64_t row = (int64_t)c->hidden * ab;
  const int64_t a = 256 / gcd64(256, row) * row;
  const int has_shared = c->shared_inter > 0;
  const int64_t rcap = routed_cap_of(c);
  const int64_t rows = std::max<int64_t>(c->token_cap, rcap);
  const int64_t table = std::max<int64_t>((int64_t)c->token_cap * c->topk, c->ffn_size >= 1 ? rcap : 0);
  // AFD_CFG_CANARY: one alignment unit of guard words after every field
  const int64_t gd = (c->flags & AFD_CFG_CANARY) ? a : 0;
  int64_t off = 0;
  L->align = a;
  L->guard = gd;
  L->header = off;
  off += round_up((int64_t)(AFD_HEADER_FIXED_WORDS + c->num_experts) * 4, a) + gd;
  L->route_table = off;
  off += round_up(table * 4, a) + gd;
  L->routed_x = off;
  off += round_up(rows * row, a) + gd;
  L->shared_idx = off;
  if (has_shared) off += round_up((int64_t)c->token_cap * 4, a) + gd;
  L->shared_x = off;
  if (has_shared) off += round_up((int64_t)c->token_cap * row, a) + gd;
  L->slot_bytes = off;
  L->flags_bytes = round_up((int64_t)c->num_peers * c->ring_depth * 8, a) + gd;
  L->window_bytes = L->flags_bytes + (int64_t)c->num_peers * c->ring_depth * off;
  return AFD_OK;
}

int validate_config(const afd_config* c) {
  if (!c) return AFD_ERR_ARG;
  if (c->num_peers < 1 || c->num_peers > AFD_MAX_PEERS || c->ring_depth < 1 || c->ring_depth > AFD_MAX_RING ||
      c->token_cap < 1 || c->max_total_tokens < 0 || c->hidden < 8 || c->num_experts < 1 ||
      c->topk < 1 || (c->ffn_size < 1 && c->topk > c->num_experts) || c->inter < 1 ||
      c->shared_inter < 0 ||
      c->max_layers < 1 || c->routed_cap_multiplier < 1.0f || c->wait_timeout_ns < 0)
    return AFD_ERR_ARG;
  if (c->act_dtype != AFD_DTYPE_F32 && c->act_dtype != AFD_DTYPE_BF16) return AFD_ERR_ARG;
  if (c->flags & ~(AFD_CFG_NO_PDL | AFD_CFG_CANARY | AFD_CFG_SPLIT_GEMMS)) return AFD_ERR_ARG;
  if (c->ffn_size < 0 || c->ffn_size > AFD_MAX_FFN_RANKS || c->ffn_rank < 0 ||
      c->ffn_rank >= std::max(1, c->ffn_size))
    return AFD_ERR_ARG;
  if (c->gemm != AFD_GEMM_TENSOR && c->gemm != AFD_GEMM_SIMT && c->gemm != AFD_GEMM_TENSOR_1CTA)
    return AFD_ERR_ARG;
  const bool tensor = c->gemm != AFD_GEMM_SIMT;
  // kernel coverage: 16-byte rows, <= 256 experts, k <= 16
  if (c->hidden % 8 || c->num_experts > 256 || c->topk > 16) return AFD_ERR_UNSUPPORTED;
  if (c->act_dtype == AFD_DTYPE_F32 && tensor) return AFD_ERR_UNSUPPORTED;
  // tensor-core engine: 16-row gate/up blocks, 32-feature epilogue quadrants
  if (tensor && (c->inter % 16 || c->shared_inter % 16 || c->hidden % 32))
    return AFD_ERR_UNSUPPORTED;
  // the router keeps 16 token rows and a weight ring in shared memory
  if (router_min_smem_bytes(c->hidden, c->num_experts, c->act_dtype == AFD_DTYPE_F32) > 232448)
    return AFD_ERR_UNSUPPORTED;
  const int64_t tmax = c->max_total_tokens ? c->max_total_tokens : (int64_t)c->num_peers * c->token_cap;
  if (tmax * c->topk + tmax > (int64_t)1 << 30) return AFD_ERR_UNSUPPORTED;
  return AFD_OK;
}

}  // namespace

struct afd_ctx {
  afd_config cfg;
  afd_layout L;
  WinGeom geom;
  int device = 0;
  int num_sms = 0;
  cudaStream_t stream = nullptr;
  cudaStream_t side = nullptr;       // L2 weight prefetch beside the small kernels
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  uint8_t* win[2] = {nullptr, nullptr};
  uint8_t* ws_mem = nullptr;
  int64_t ws_bytes = 0;
  DevWS ws;
  GemmPlan* plan1 = nullptr;
  GemmPlan* plan2 = nullptr;
  DevLayer* dlayers = nullptr;       // device copy of every layer's weights (work-item loop)
  CUtensorMap tmXp, tmH, tmHs;        // token boxes of the tensor engine
  CUtensorMap tmXp32, tmH32, tmHs32;  // 32-row boxes (small SM-pair units)
  CUtensorMap tmWin, tmWin32;         // dispatch window as [rows, hidden] (shared rows, and
                                      // the grouped form's rows from one peer, read in place)
  std::vector<LayerW> layers;
  std::vector<uint64_t> last_seq;
  int tmax = 0;
  int act_f32 = 0;
  int64_t launches = 0;
  int last_T = 0;
  int64_t forwards = 0;
  uint32_t go_seq = 0;               // tokens for ws.go, one per host-described routed step
  unsigned long long* canary_result = nullptr;  // AFD_CFG_CANARY: [changed words, first offset]
  int64_t ws_cap[12];
  // stage timing: one set of events per forward, in a ring, so the host
  // reads them after many forwards instead of waiting after each one
  static constexpr int kProfRing = 64;
  bool profiling = false;
  bool events_made = false;
  cudaEvent_t ev[kProfRing][AFD_NUM_STAGES + 1] = {};
  int prof_head = 0;     // set the next forward records into
  int prof_pending = 0;  // recorded sets not yet folded into prof_acc
  double prof_acc[AFD_NUM_STAGES] = {};
  int64_t prof_acc_n = 0;

  // wait for the oldest recorded set and add its stage times to prof_acc
  int fold_oldest() {
    const int idx = (prof_head - prof_pending + kProfRing) % kProfRing;
    if (cudaEventSynchronize(ev[idx][AFD_NUM_STAGES]) != cudaSuccess) return AFD_ERR_CUDA;
    for (int i = 0; i < AFD_NUM_STAGES; i++) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, ev[idx][i], ev[idx][i + 1]) != cudaSuccess) return AFD_ERR_CUDA;
      prof_acc[i] += ms;
    }
    prof_acc_n++;
    prof_pending--;
    return AFD_OK;
  }
  void mark(int i) {
    if (!profiling) return;
    if (i == 0 && prof_pending == kProfRing && fold_oldest()) {
      fprintf(stderr, "afd: stage timing failed; timing switched off\n");
      cudaGetLastError();
      profiling = false;
      return;
    }
    cudaEventRecord(ev[prof_head][i], stream);
    if (i == AFD_NUM_STAGES) {  // a complete set: count it
      prof_head = (prof_head + 1) % kProfRing;
      prof_pending++;
    }
  }

  LaunchCtx lc() { return LaunchCtx{stream, num_sms, &launches, (cfg.flags & AFD_CFG_NO_PDL) ? 0 : 1}; }
  int64_t timeout() const { return cfg.wait_timeout_ns ? cfg.wait_timeout_ns : 1000000000ll; }
};

static CanaryGeom canary_geom(const afd_ctx* c);

static int cuda_fail(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return AFD_OK;
  fprintf(stderr, "afd: %s: %s\n", what, cudaGetErrorString(e));
  return AFD_ERR_CUDA;
}

// the guard regions of a context's windows (AFD_CFG_CANARY)
static CanaryGeom canary_geom(const afd_ctx* c) {
  const afd_layout& L = c->L;
  CanaryGeom cg;
  memset(&cg, 0, sizeof cg);
  cg.flags_bytes = L.flags_bytes;
  cg.slot_bytes = L.slot_bytes;
  cg.guard = L.guard;
  const bool sh = c->cfg.shared_inter > 0;
  // each field's guard ends where the next field (or the slot) begins
  const int64_t ends[5] = {L.route_table, L.routed_x, L.shared_idx, sh ? L.shared_x : 0, L.slot_bytes};
  const int nf = sh ? 5 : 3;
  for (int i = 0; i < nf; i++) cg.goff[i] = (i == nf - 1 ? L.slot_bytes : ends[i]) - L.guard;
  cg.n = nf;
  cg.nslots = c->cfg.num_peers * c->cfg.ring_depth;
  return cg;
}

extern "C" {

const char* afd_strerror(int code) {
  switch (code) {
    case AFD_OK: return "ok";
    case AFD_ERR_ARG: return "invalid argument";
    case AFD_ERR_SHAPE: return "token counts disagree";
    case AFD_ERR_CAPACITY: return "capacity exceeded";
    case AFD_ERR_HEADER: return "bad slot header";
    case AFD_ERR_SEQ: return "sequence number mismatch";
    case AFD_ERR_LAYER: return "layer mismatch or unregistered layer";
    case AFD_ERR_STAGE: return "stage mismatch";
    case AFD_ERR_TIMEOUT: return "device wait timed out";
    case AFD_ERR_SHUTDOWN: return "peer announced shutdown";
    case AFD_ERR_SPLIT_UNEVEN: return "even split does not divide";
    case AFD_ERR_NOT_DEVICE: return "pointer is not device memory";
    case AFD_ERR_CUDA: return "CUDA error";
    case AFD_ERR_UNSUPPORTED: return "unsupported configuration";
    case AFD_ERR_CANARY: return "guard word after a slot field overwritten";
    case AFD_ERR_BOUNDS: return "index out of range (debug build bounds check)";
    default: return "unknown status";
  }
}

int afd_slot_layout(const afd_config* cfg, afd_layout* out) {
  if (!out) return AFD_ERR_ARG;
  const int rc = validate_config(cfg);
  if (rc) return rc;
  return layout_of(cfg, out);
}

int afd_split_sizes(int total, int n_peers, const int* seq_lens, int n_lens, int* sizes) {
  if (n_peers <= 0 || total < 0 || !sizes || n_lens < 0 || (n_lens > 0 && !seq_lens))
    return AFD_ERR_ARG;
  if (n_lens == n_peers) {
    int64_t s = 0;
    for (int i = 0; i < n_peers; i++) {
      if (seq_lens[i] < 0) return AFD_ERR_ARG;
      s += seq_lens[i];
      sizes[i] = seq_lens[i];
    }
    return s == total ? AFD_OK : AFD_ERR_SHAPE;
  }
  if (total % n_peers) return AFD_ERR_SPLIT_UNEVEN;
  for (int i = 0; i < n_peers; i++) sizes[i] = total / n_peers;
  return AFD_OK;
}

void afd_destroy(afd_ctx* ctx) {
  if (!ctx) return;
  cudaSetDevice(ctx->device);
  cudaStreamSynchronize(ctx->stream);
  if (ctx->side) {
    cudaStreamSynchronize(ctx->side);
    cudaStreamDestroy(ctx->side);
  }
  if (ctx->ev_fork) cudaEventDestroy(ctx->ev_fork);
  if (ctx->ev_join) cudaEventDestroy(ctx->ev_join);
  for (auto& l : ctx->layers) {
    cudaFree(l.WgQ);
    for (void* t : l.T) cudaFree(t);
  }
  for (auto& set : ctx->ev)
    for (auto& e : set)
      if (e) cudaEventDestroy(e);
  cudaFree(ctx->win[0]);
  cudaFree(ctx->win[1]);
  cudaFree(ctx->canary_result);
  cudaFree(ctx->ws_mem);
  delete ctx;
}

int afd_create(const afd_config* cfg, void* cuda_stream, afd_ctx** out) {
  if (!out) return AFD_ERR_ARG;
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return AFD_ERR_CUDA;
  }
  afd_ctx* c = new afd_ctx();
  c->cfg = *cfg;
  c->device = dev;
  c->stream = reinterpret_cast<cudaStream_t>(cuda_stream);
  c->act_f32 = cfg->act_dtype == AFD_DTYPE_F32;
  cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev);
  layout_of(cfg, &c->L);
  c->geom = WinGeom{c->L.flags_bytes, c->L.slot_bytes, c->L.header, c->L.route_table,
                    c->L.routed_x, c->L.shared_idx, c->L.shared_x, cfg->ring_depth, cfg->num_peers};
  c->tmax = cfg->max_total_tokens ? cfg->max_total_tokens : cfg->num_peers * cfg->token_cap;
  c->layers.resize(cfg->max_layers);
  if (cfg->gemm == AFD_GEMM_TENSOR) {
    rc = cuda_fail(cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking), "side stream");
    if (!rc) rc = cuda_fail(cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming), "event");
    if (!rc) rc = cuda_fail(cudaEventCreateWithFlags(&c->ev_join, cudaEventDisableTiming), "event");
    if (rc) { afd_destroy(c); return rc; }
  }
  c->last_seq.assign((size_t)cfg->num_peers * cfg->ring_depth, 0);
  for (int d = 0; d < 2; d++) {
    rc = cuda_fail(cudaMalloc(&c->win[d], c->L.window_bytes), "window allocation");
    if (!rc) rc = cuda_fail(cudaMemset(c->win[d], 0, c->L.window_bytes), "window zero");
    if (!rc && c->L.guard)
      rc = cuda_fail(launch_canary(nullptr, c->win[d], canary_geom(c), 1, nullptr, c->num_sms),
                     "canary fill");
    if (rc) { afd_destroy(c); return rc; }
  }
  if (c->L.guard) {
    rc = cuda_fail(cudaMalloc(&c->canary_result, 2 * sizeof(unsigned long long)), "canary result");
    if (!rc) rc = cuda_fail(cudaDeviceSynchronize(), "canary fill");
    if (rc) { afd_destroy(c); return rc; }
  }
  // workspace
  const int64_t Tm = c->tmax, k = cfg->topk, H = cfg->hidden, E = cfg->num_experts;
  const int64_t I = cfg->inter, Is = cfg->shared_inter;
  const int64_t ab = c->act_f32 ? 4 : 2;
  // routed expert outputs y: fp32 in the token form (the combine sums them
  // before the one rounding to the activation type), the activation type in
  // the grouped form (the rows that go back); sized for the wider
  const int64_t yb = 4;
  struct Part { int64_t bytes; } parts[] = {
      {4},                                   // status
      {(int64_t)cfg->num_peers * cfg->ring_depth * 8},  // seen
      {AFD_MAX_PEERS * 8},                   // cur_seq
      {AFD_MAX_PEERS * 4},                   // peer_shared
      {Tm * k * 4}, {Tm * k * 4},            // ids, w
      {E * 4}, {(E + 1) * 4},                // counts, offsets
      {Tm * k * 4}, {Tm * k * 4},            // perm, inv
      {AFD_MAX_PEERS * E * 4},               // peer_counts
      {(Tm * k + Tm) * H * ab},              // xp (routed rows, then shared rows when gathered)
      {Tm * k * I * ab},                     // h
      {Tm * k * H * yb},                     // y
      {Tm * (Is > 0 ? Is : 1) * ab},         // hs
      {Tm * H * 4},                          // s
      {(int64_t)sizeof(GemmPlan)}, {(int64_t)sizeof(GemmPlan)},
      {E * router_blocks((int)Tm) * 4}, {E * router_blocks((int)Tm) * 4},  // hist, base
      {Tm * E * 4},                          // router logits
      {2 * AFD_MAX_PEERS * E * 4},           // grouped-form bases and group-list prefixes
      {(int64_t)sizeof(FanIn)},              // the fan-in of the step in flight
      {AFD_LOOP_WORDS * 4},                  // work-item loop state and log
      {(int64_t)cfg->max_layers * (int64_t)sizeof(DevLayer)},  // per-layer weight table
      {4},                                   // go word (header check -> router)
      {AFD_MAX_PEERS * 4},                   // combine items finished per entry
      {8 * 8},                               // debug build's bounds record
      {(Tm * k + Tm + AFD_MAX_GROUPS + AFD_MAX_PEERS) * 4}};  // token tiles' SwiGLU counters
  const int nparts = sizeof(parts) / sizeof(parts[0]);
  int64_t offs[32], total = 0;
  for (int i = 0; i < nparts; i++) {
    offs[i] = total;
    total += round_up(parts[i].bytes > 0 ? parts[i].bytes : 1, 256);
  }
  rc = cuda_fail(cudaMalloc(&c->ws_mem, total), "workspace allocation");
  if (!rc) rc = cuda_fail(cudaMemset(c->ws_mem, 0, total), "workspace zero");
  if (rc) { afd_destroy(c); return rc; }
  c->ws_bytes = total;
  uint8_t* b = c->ws_mem;
  c->ws.status = reinterpret_cast<int32_t*>(b + offs[0]);
  c->ws.seen = reinterpret_cast<uint64_t*>(b + offs[1]);
  c->ws.cur_seq = reinterpret_cast<uint64_t*>(b + offs[2]);
  c->ws.peer_shared = reinterpret_cast<int32_t*>(b + offs[3]);
  c->ws.ids = reinterpret_cast<int32_t*>(b + offs[4]);
  c->ws.w = reinterpret_cast<float*>(b + offs[5]);
  c->ws.counts = reinterpret_cast<int32_t*>(b + offs[6]);
  c->ws.offsets = reinterpret_cast<int32_t*>(b + offs[7]);
  c->ws.perm = reinterpret_cast<int32_t*>(b + offs[8]);
  c->ws.inv = reinterpret_cast<int32_t*>(b + offs[9]);
  c->ws.peer_counts = reinterpret_cast<int32_t*>(b + offs[10]);
  c->ws.xp = b + offs[11];
  c->ws.h = b + offs[12];
  c->ws.y = b + offs[13];
  // low plane of the 24-bit y after the high plane (2 + 1 of the 4 bytes per element)
  c->ws.y_lo = b + offs[13] + Tm * k * H * 2;
  c->ws.hs = b + offs[14];
  c->ws.s = reinterpret_cast<float*>(b + offs[15]);
  c->ws.hist = reinterpret_cast<int32_t*>(b + offs[18]);
  c->ws.base = reinterpret_cast<int32_t*>(b + offs[19]);
  c->ws.logits = reinterpret_cast<float*>(b + offs[20]);
  c->ws.gbase = reinterpret_cast<int32_t*>(b + offs[21]);
  c->ws.item = reinterpret_cast<FanIn*>(b + offs[22]);
  c->ws.loop = reinterpret_cast<int32_t*>(b + offs[23]);
  c->dlayers = reinterpret_cast<DevLayer*>(b + offs[24]);
  c->ws.layers = c->dlayers;
  c->ws.go = reinterpret_cast<uint32_t*>(b + offs[25]);
  c->ws.ret_count = reinterpret_cast<int32_t*>(b + offs[26]);
  c->ws.dbg = reinterpret_cast<int64_t*>(b + offs[27]);
  c->ws.dep = reinterpret_cast<int32_t*>(b + offs[28]);
  c->plan1 = reinterpret_cast<GemmPlan*>(b + offs[16]);
  c->plan2 = reinterpret_cast<GemmPlan*>(b + offs[17]);
  const int ws_map[12] = {4, 5, 6, 7, 8, 9, 11, 12, 13, 14, 15, 0};
  for (int i = 0; i < 12; i++) c->ws_cap[i] = parts[ws_map[i]].bytes;
  if (cfg->gemm != AFD_GEMM_SIMT) {
    rc = get_encoder();
    // token boxes: 32 rows for one CTA per tile, 128 rows (a CTA's half of a
    // 256-token unit) for the SM-pair engine
    const int box = cfg->gemm == AFD_GEMM_TENSOR ? 128 : 32;
    if (!rc) rc = encode_rows(&c->tmXp, c->ws.xp, Tm * k + Tm, (int)H, box);
    if (!rc) rc = encode_rows(&c->tmH, c->ws.h, Tm * k, (int)I, box);
    if (!rc) rc = encode_rows(&c->tmHs, c->ws.hs, Tm, (int)(Is > 0 ? Is : 64), box);
    if (!rc) rc = encode_rows(&c->tmXp32, c->ws.xp, Tm * k + Tm, (int)H, 32);
    if (!rc) rc = encode_rows(&c->tmH32, c->ws.h, Tm * k, (int)I, 32);
    if (!rc) rc = encode_rows(&c->tmHs32, c->ws.hs, Tm, (int)(Is > 0 ? Is : 64), 32);
    const int64_t win_rows = c->L.window_bytes / (H * ab);
    if (!rc) rc = encode_rows(&c->tmWin, c->win[0], win_rows, (int)H, box);
    if (!rc) rc = encode_rows(&c->tmWin32, c->win[0], win_rows, (int)H, 32);
    if (rc) { afd_destroy(c); return rc; }
  }
  *out = c;
  return AFD_OK;
}

int afd_set_stream(afd_ctx* ctx, void* cuda_stream) {
  if (!ctx) return AFD_ERR_ARG;
  ctx->stream = reinterpret_cast<cudaStream_t>(cuda_stream);
  return AFD_OK;
}

int afd_set_layer(afd_ctx* ctx, int layer, const float* Wg, const float* bias, const void* W13,
                  const void* Wd, const void* W13_s, const void* Wd_s) {
  if (!ctx || layer < 0 || layer >= ctx->cfg.max_layers) return AFD_ERR_ARG;
  const afd_config& c = ctx->cfg;
  const bool has_shared = c.shared_inter > 0;
  // an FFN rank under token-level dispatch never routes: no router weight needed
  if ((!Wg && c.ffn_size < 1) || !W13 || !Wd || (has_shared && (!W13_s || !Wd_s)))
    return AFD_ERR_ARG;
  const void* ptrs[6] = {Wg, bias, W13, Wd, has_shared ? W13_s : nullptr, has_shared ? Wd_s : nullptr};
  for (const void* p : ptrs) {
    if (!p) continue;
    int rc = check_dev_ptr(p);
    if (rc) return rc;
    if (!aligned16(p)) return AFD_ERR_ARG;
  }
  LayerW& L = ctx->layers[layer];
  int rc = AFD_OK;
  // the copies below replace what a forward still in flight may read: no
  // overlap with earlier work on the stream
  LaunchCtx lc = ctx->lc();
  lc.pdl = 0;
  if (Wg) {
    if (!L.WgQ) {
      rc = cuda_fail(cudaMalloc(&L.WgQ, (size_t)wgq_groups(c.num_experts) * c.hidden * 16),
                     "router copy");
      if (rc) return rc;
    }
    rc = cuda_fail(launch_arrange_wg(lc, Wg, L.WgQ, c.hidden, c.num_experts), "router copy");
    if (rc) return rc;
  }
  L.Wg = Wg;
  L.bias = bias;
  L.W13 = W13;
  L.Wd = Wd;
  L.W13s = has_shared ? W13_s : nullptr;
  L.Wds = has_shared ? Wd_s : nullptr;
  if (c.gemm != AFD_GEMM_SIMT) {
    // the tensor engines read tiled copies (one contiguous 16 KB block per
    // TMA box); the caller's buffers are not read after this call returns
    struct Src { const void* W; int E, M, K, swiglu, I; };
    const Src src[4] = {{W13, c.num_experts, 2 * c.inter, c.hidden, 1, c.inter},
                        {Wd, c.num_experts, c.hidden, c.inter, 0, 0},
                        {W13_s, 1, 2 * c.shared_inter, c.hidden, 1, c.shared_inter},
                        {Wd_s, 1, c.hidden, c.shared_inter, 0, 0}};
    CUtensorMap* maps[4] = {&L.tmA1[0], &L.tmA2[0], &L.tmA1[1], &L.tmA2[1]};
    for (int w = 0; w < (has_shared ? 4 : 2) && !rc; w++) {
      const Src& q = src[w];
      const int tiles = tiled_weight_tiles(q.M, q.swiglu, q.I);
      const size_t bytes = (size_t)q.E * tiles * ((q.K + 63) / 64) * 16384;
      if (L.T_bytes[w] != bytes) {
        cudaFree(L.T[w]);
        L.T[w] = nullptr;
        L.T_bytes[w] = 0;
        rc = cuda_fail(cudaMalloc(&L.T[w], bytes), "weight copy");
        if (rc) break;
        L.T_bytes[w] = bytes;
      }
      rc = cuda_fail(launch_tile_weight(lc, q.W, L.T[w], q.E, q.M, q.K, q.swiglu, q.I), "weight copy");
      if (!rc) rc = encode_tiled_weight(maps[w], L.T[w], q.E, tiles, q.K);
    }
    if (!rc && !has_shared) {
      L.tmA1[1] = L.tmA1[0];
      L.tmA2[1] = L.tmA2[0];
    }
    if (!rc) rc = cuda_fail(cudaStreamSynchronize(ctx->stream), "weight copy");
    if (rc) return rc;
    // what the engines (and the decode L2 prefetch) read
    L.W13 = L.T[0];
    L.Wd = L.T[1];
    L.W13s = has_shared ? L.T[2] : nullptr;
    L.Wds = has_shared ? L.T[3] : nullptr;
  }
  // the device table entry, for steps whose layer the device chooses (a
  // pageable source: the copy is staged before the call returns)
  DevLayer d;
  memset(&d, 0, sizeof d);
  d.tmA1[0] = L.tmA1[0];
  d.tmA1[1] = L.tmA1[1];
  d.tmA2[0] = L.tmA2[0];
  d.tmA2[1] = L.tmA2[1];
  d.WgQ = L.WgQ;
  d.bias = L.bias;
  d.W13 = L.W13;
  d.W13s = L.W13s;
  d.Wd = L.Wd;
  d.Wds = L.Wds;
  d.set = 1;
  rc = cuda_fail(cudaMemcpyAsync(ctx->dlayers + layer, &d, sizeof d, cudaMemcpyHostToDevice,
                                 ctx->stream),
                 "layer table");
  if (rc) return rc;
  L.set = true;
  return AFD_OK;
}

static int pack_common(afd_ctx* ctx, int peer, int stage, int layer, const void* x, int n,
                       int with_shared, uint64_t seq, int shutdown) {
  if (!ctx) return AFD_ERR_ARG;
  const afd_config& c = ctx->cfg;
  if (c.ffn_size >= 1 && !shutdown) return AFD_ERR_ARG;  // ranks receive afd_attn_dispatch
  if (peer < 0 || peer >= c.num_peers || stage < 0 || stage >= c.ring_depth || n < 0)
    return AFD_ERR_ARG;
  if (with_shared && c.shared_inter <= 0) return AFD_ERR_ARG;
  if (n > c.token_cap) return AFD_ERR_CAPACITY;
  if (n > 0) {
    const int rc = check_dev_ptr(x);
    if (rc) return rc;
    if (!aligned16(x)) return AFD_ERR_ARG;
  }
  uint64_t& last = ctx->last_seq[(size_t)peer * c.ring_depth + stage];
  if (seq <= last) return AFD_ERR_SEQ;
  const int row_bytes = c.hidden * (ctx->act_f32 ? 4 : 2);
  LaunchCtx lc = ctx->lc();
  GroupList gl;
  memset(&gl, 0, sizeof gl);
  int rc = cuda_fail(launch_pack_payload(lc, ctx->geom, ctx->win[0], peer, stage, x, n,
                                         with_shared ? x : nullptr, n, row_bytes),
                     "pack payload");
  if (!rc)
    rc = cuda_fail(launch_pack_header(lc, ctx->geom, ctx->win[0], peer, stage, layer, n, with_shared,
                                      c.num_experts, seq, shutdown, 0, gl),
                   "pack header");
  if (!rc) last = seq;
  return rc;
}

int afd_pack_grouped(afd_ctx* ctx, int peer, int stage, int layer, const void* rows, int n_rows,
                     const int* group_list, const void* x, int n_tokens, int with_shared,
                     uint64_t seq) {
  if (!ctx || !group_list) return AFD_ERR_ARG;
  const afd_config& c = ctx->cfg;
  if (peer < 0 || peer >= c.num_peers || stage < 0 || stage >= c.ring_depth || n_tokens < 0 ||
      n_rows < 0)
    return AFD_ERR_ARG;
  if (with_shared && c.shared_inter <= 0) return AFD_ERR_ARG;
  // with several ranks a peer's shared rows are its round-robin share:
  // afd_attn_dispatch sends those
  if (with_shared && c.ffn_size > 1) return AFD_ERR_ARG;
  if (n_tokens > c.token_cap || n_rows > routed_cap_of(&c)) return AFD_ERR_CAPACITY;
  GroupList gl;
  memset(&gl, 0, sizeof gl);
  int64_t sum = 0;
  for (int e = 0; e < c.num_experts; e++) {
    if (group_list[e] < 0) return AFD_ERR_ARG;
    gl.n[e] = group_list[e];
    sum += group_list[e];
  }
  if (sum != n_rows) return AFD_ERR_SHAPE;
  for (const auto& pr : {std::make_pair(rows, n_rows), std::make_pair(x, with_shared ? n_tokens : 0)}) {
    if (pr.second <= 0) continue;
    const int rc = check_dev_ptr(pr.first);
    if (rc) return rc;
    if (!aligned16(pr.first)) return AFD_ERR_ARG;
  }
  uint64_t& last = ctx->last_seq[(size_t)peer * c.ring_depth + stage];
  if (seq <= last) return AFD_ERR_SEQ;
  const int row_bytes = c.hidden * (ctx->act_f32 ? 4 : 2);
  LaunchCtx lc = ctx->lc();
  int rc = cuda_fail(launch_pack_payload(lc, ctx->geom, ctx->win[0], peer, stage, rows, n_rows,
                                         with_shared ? x : nullptr, n_tokens, row_bytes),
                     "pack payload");
  if (!rc)
    rc = cuda_fail(launch_pack_header(lc, ctx->geom, ctx->win[0], peer, stage, layer, n_tokens,
                                      with_shared, c.num_experts, seq, 0, n_rows, gl),
                   "pack header");
  if (!rc) last = seq;
  return rc;
}

int afd_pack_slot(afd_ctx* ctx, int peer, int stage, int layer, const void* x, int n_tokens,
                  int with_shared, uint64_t seq) {
  return pack_common(ctx, peer, stage, layer, x, n_tokens, with_shared, seq, 0);
}

int afd_announce_shutdown(afd_ctx* ctx, int peer, int stage, uint64_t seq) {
  return pack_common(ctx, peer, stage, 0, nullptr, 0, 0, seq, 1);
}

// Shared rows of each list entry: its tokens with one FFN rank, its
// round-robin share (tokens ffn_rank, ffn_rank + ffn_size, ...) with several
static void set_shared_rows(FanIn& f, const afd_config& c) {
  f.ffn_size = std::max(1, c.ffn_size);
  f.ffn_rank = c.ffn_size >= 1 ? c.ffn_rank : 0;
  int run = 0;
  for (int i = 0; i < f.n_peers; i++) {
    f.sprefix[i] = run;
    run += rr_rows(f.prefix[i + 1] - f.prefix[i], f.ffn_rank, f.ffn_size);
  }
  f.sprefix[f.n_peers] = run;
  f.stotal = run;
}

// Arguments of a forward: the list entries (slots, each once and in range),
// their token counts (<= token_cap each, total <= the context's capacity)
static int fanin_of(afd_ctx* ctx, int stage, const int* seq_lens, const int* slots, int n_peers,
                    FanIn& f) {
  if (!ctx || !seq_lens || !slots) return AFD_ERR_ARG;
  const afd_config& c = ctx->cfg;
  if (n_peers <= 0 || n_peers > c.num_peers) return AFD_ERR_ARG;
  if (stage < 0 || stage >= c.ring_depth) return AFD_ERR_ARG;
  memset(&f, 0, sizeof f);
  f.n_peers = n_peers;
  f.stage = stage;
  int64_t T = 0;
  for (int i = 0; i < n_peers; i++) {
    if (slots[i] < 0 || slots[i] >= c.num_peers) return AFD_ERR_ARG;
    for (int j = 0; j < i; j++)
      if (slots[j] == slots[i]) return AFD_ERR_ARG;
    if (seq_lens[i] < 0) return AFD_ERR_ARG;
    if (seq_lens[i] > c.token_cap) return AFD_ERR_CAPACITY;
    f.prefix[i] = (int)T;
    f.region[i] = slots[i];
    T += seq_lens[i];
  }
  if (T > ctx->tmax) return AFD_ERR_CAPACITY;
  f.prefix[n_peers] = (int)T;
  f.total = (int)T;
  set_shared_rows(f, c);
  return AFD_OK;
}

static int forward_impl(afd_ctx* ctx, int layer, FanIn& f, const PeerList* dev);

int afd_ffn_forward(afd_ctx* ctx, int layer, int stage, const int* seq_lens, const int* slots,
                    int n_peers) {
  if (ctx && ctx->cfg.ffn_size >= 1) return AFD_ERR_ARG;  // a rank receives grouped rows
  FanIn f;
  const int rc = fanin_of(ctx, stage, seq_lens, slots, n_peers, f);
  if (rc) return rc;
  return forward_impl(ctx, layer, f, nullptr);
}

int afd_ffn_forward_grouped(afd_ctx* ctx, int layer, int stage, const int* n_rows,
                            const int* seq_lens, const int* slots, int n_peers) {
  FanIn f;
  int rc = fanin_of(ctx, stage, seq_lens, slots, n_peers, f);
  if (rc) return rc;
  if (!n_rows) return AFD_ERR_ARG;
  int64_t R = 0;
  const int64_t rows_cap = routed_cap_of(&ctx->cfg);
  for (int i = 0; i < n_peers; i++) {
    if (n_rows[i] < 0) return AFD_ERR_ARG;
    if (n_rows[i] > rows_cap) return AFD_ERR_CAPACITY;
    f.rprefix[i] = (int)R;
    R += n_rows[i];
  }
  if (R > (int64_t)ctx->tmax * ctx->cfg.topk) return AFD_ERR_CAPACITY;
  f.rprefix[n_peers] = (int)R;
  f.rtotal = (int)R;
  f.grouped = 1;
  f.num_experts = ctx->cfg.num_experts;
  return forward_impl(ctx, layer, f, nullptr);
}

// Launch shapes of a work-item loop step over the listed peers: the most
// tokens (and grouped rows) a step may carry; the device fills in the rest.
static int serve_shape(afd_ctx* ctx, const int* slots, int n_peers, int form, PeerList& pl,
                       FanIn& fs) {
  if (!ctx || !slots || (form != AFD_FORM_TOKENS && form != AFD_FORM_GROUPED)) return AFD_ERR_ARG;
  const afd_config& c = ctx->cfg;
  if (form == AFD_FORM_TOKENS && c.ffn_size >= 1) return AFD_ERR_ARG;
  if (n_peers <= 0 || n_peers > c.num_peers) return AFD_ERR_ARG;
  memset(&pl, 0, sizeof pl);
  memset(&fs, 0, sizeof fs);
  pl.n = n_peers;
  for (int i = 0; i < n_peers; i++) {
    if (slots[i] < 0 || slots[i] >= c.num_peers) return AFD_ERR_ARG;
    for (int j = 0; j < i; j++)
      if (slots[j] == slots[i]) return AFD_ERR_ARG;
    pl.slot[i] = slots[i];
    fs.region[i] = slots[i];
  }
  fs.n_peers = n_peers;
  fs.dev = 1;  // the kernels take the step's values from ws.item
  fs.ffn_size = std::max(1, c.ffn_size);
  fs.ffn_rank = c.ffn_size >= 1 ? c.ffn_rank : 0;
  const int64_t cap = (int64_t)n_peers * c.token_cap;
  fs.total = (int)std::min<int64_t>(ctx->tmax, cap);
  fs.prefix[n_peers] = fs.total;
  if (form == AFD_FORM_GROUPED) {
    fs.grouped = 1;
    fs.num_experts = c.num_experts;
    fs.rtotal = (int)std::min<int64_t>((int64_t)ctx->tmax * c.topk, cap);
    fs.rprefix[n_peers] = fs.rtotal;
  }
  return AFD_OK;
}

int afd_ffn_serve(afd_ctx* ctx, const int* slots, int n_peers, int n_items, int form) {
  PeerList pl;
  FanIn fs;
  int rc = serve_shape(ctx, slots, n_peers, form, pl, fs);
  if (rc) return rc;
  if (n_items < 0) return AFD_ERR_ARG;
  for (int it = 0; it < n_items && !rc; it++) {
    FanIn f = fs;
    rc = forward_impl(ctx, -1, f, &pl);
  }
  return rc;
}

struct afd_serve_graph {
  afd_ctx* ctx = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int n_items = 0;
};

int afd_serve_graph_create(afd_ctx* ctx, const int* slots, int n_peers, int n_items, int form,
                           afd_serve_graph** out, int64_t* kernels) {
  if (!out) return AFD_ERR_ARG;
  *out = nullptr;
  PeerList pl;
  FanIn fs;
  int rc = serve_shape(ctx, slots, n_peers, form, pl, fs);
  if (rc) return rc;
  if (n_items <= 0) return AFD_ERR_ARG;
  // captured on a stream of its own (the caller's may be the legacy
  // stream, which cannot be captured); replayed on the context's stream
  cudaStream_t cap = nullptr;
  rc = cuda_fail(cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking), "capture stream");
  if (rc) return rc;
  cudaStream_t user = ctx->stream;
  const bool prof = ctx->profiling;
  ctx->stream = cap;
  ctx->profiling = false;
  const int64_t before = ctx->launches;
  const int64_t fwd = ctx->forwards;
  cudaGraph_t graph = nullptr;
  rc = cuda_fail(cudaStreamBeginCapture(cap, cudaStreamCaptureModeRelaxed), "begin capture");
  if (!rc) {
    int frc = AFD_OK;
    for (int it = 0; it < n_items && !frc; it++) {
      FanIn f = fs;
      frc = forward_impl(ctx, -1, f, &pl);
    }
    rc = cuda_fail(cudaStreamEndCapture(cap, &graph), "end capture");
    if (!rc) rc = frc;
  }
  ctx->stream = user;
  ctx->profiling = prof;
  ctx->forwards = fwd;
  const int64_t captured = ctx->launches - before;
  ctx->launches = before;
  cudaStreamDestroy(cap);
  cudaGraphExec_t exec = nullptr;
  if (!rc) rc = cuda_fail(cudaGraphInstantiate(&exec, graph, 0), "graph instantiate");
  if (rc) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  afd_serve_graph* g = new afd_serve_graph();
  g->ctx = ctx;
  g->graph = graph;
  g->exec = exec;
  g->n_items = n_items;
  if (kernels) *kernels = captured;
  *out = g;
  return AFD_OK;
}

int afd_serve_graph_launch(afd_serve_graph* g) {
  if (!g || !g->ctx) return AFD_ERR_ARG;
  const int rc = cuda_fail(cudaGraphLaunch(g->exec, g->ctx->stream), "graph launch");
  if (!rc) g->ctx->forwards += g->n_items;
  return rc;
}

void afd_serve_graph_destroy(afd_serve_graph* g) {
  if (!g) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
}

int afd_serve_log(afd_ctx* ctx, int32_t* records, int max_records, int* n_records,
                  int64_t* n_served) {
  if (!ctx || !n_records || max_records < 0 || (max_records > 0 && !records)) return AFD_ERR_ARG;
  if (cuda_fail(cudaStreamSynchronize(ctx->stream), "stream sync")) return AFD_ERR_CUDA;
  int32_t w[AFD_LOOP_WORDS];
  if (cuda_fail(cudaMemcpy(w, ctx->ws.loop, sizeof w, cudaMemcpyDeviceToHost), "loop log read"))
    return AFD_ERR_CUDA;
  const int count = w[AFD_LOOP_COUNT];
  if (n_served) *n_served = count;
  const int n = std::min(std::min(max_records, count), AFD_LOOP_LOG_N);
  for (int j = 0; j < n; j++) {  // the last n items, oldest first
    const int idx = (count - n + j) % AFD_LOOP_LOG_N;
    for (int q = 0; q < 4; q++) records[4 * j + q] = w[AFD_LOOP_LOG + 4 * idx + q];
  }
  *n_records = n;
  return AFD_OK;
}

// One FFN step.  dev == nullptr: the host describes it (f, layer).  Else a
// step of the work-item loop over the peers in *dev: the device chooses the
// stage and takes the layer and the counts from the headers; f then holds
// only the launch shapes (the most tokens and rows a step may carry), and
// the weights come from the device layer table.
static int forward_impl(afd_ctx* ctx, int layer, FanIn& f, const PeerList* dev) {
  const afd_config& c = ctx->cfg;
  f.layer = layer;
  const int64_t T = f.total;
  const bool grouped = f.grouped != 0;
  // grouped form from a single peer on a tensor engine: its rows are already
  // grouped by expert in its slot, so the GEMMs read them there and write the
  // outputs into its return slot (no gather, no scatter).  With several peers
  // the per-(peer, expert) groups would be small and each expert's weights
  // read once per peer (measured slower than gathering the peers' rows into
  // one group per expert), so those take the gather and the scatter.
  const bool in_place = grouped && c.gemm != AFD_GEMM_SIMT && f.n_peers == 1;
  // routed rows: T * k partials, or the rows the peers sent already grouped
  const int64_t N = grouped ? f.rtotal : T * c.topk;
  if (!dev && (layer < 0 || layer >= c.max_layers || !ctx->layers[layer].set)) return AFD_ERR_LAYER;
  const LayerW* L = dev ? nullptr : &ctx->layers[layer];
  const int has_shared = c.shared_inter > 0;
  const int ab = ctx->act_f32 ? 4 : 2;
  const int row_bytes = c.hidden * ab;
  // token tile of the grouped GEMMs: 256 rows, or 64 on the SM-pair engine
  // when the experts average <= 48 rows (decode-sized fan-ins), which then
  // runs its deeper narrow ring
  const int bn = c.gemm == AFD_GEMM_TENSOR && N <= 48 * (int64_t)c.num_experts ? 64 : 256;
  // the shared expert reads its rows in place from the slots' shared_x (one
  // group per peer, no copy) when that takes no more GEMM units than the
  // gathered rows: large peers (prefill); with many small peers (decode)
  // each group would stream the shared weights once more, so those rows are
  // gathered.  Steps of the work-item loop (counts unknown here) gather.
  int sh_in_place = 0;
  if (has_shared && !dev && !in_place) {
    int64_t units_ip = 0;
    for (int i = 0; i < f.n_peers; i++) units_ip += (f.sprefix[i + 1] - f.sprefix[i] + bn - 1) / bn;
    sh_in_place = units_ip <= ((int64_t)f.stotal + bn - 1) / bn + 1;
  }
  LaunchCtx lc = ctx->lc();
  const DevWS& ws = ctx->ws;
  // decode-sized fan-ins: the SwiGLU GEMM streams its weights from HBM while
  // the small kernels before it leave HBM idle, so a side stream prefetches
  // the weights of the GEMM's first units (experts in order, 256 rows per
  // unit) into L2 meanwhile; joined at the end of the step.  The fork's event
  // ends the programmatic overlap of the two launches it falls between, and
  // the prefetch's DRAM traffic slows the small kernels' own loads.  Host-
  // described steps fork before the header check (no launch of the step is
  // split) and issue from a few SMs, num_sms / 8, whose copy engines pace the
  // traffic over the small kernels: 95 units (100 MB) from 19 SMs measured
  // 6.33 ms per 26 layers against 6.39 ms for 57 units from every SM forked
  // after the header check (sweep of 57-152 units x 10-152 SMs).  Steps the
  // device describes fork after the item head, whose fan-in they read.
  const bool prefetch = c.gemm == AFD_GEMM_TENSOR && bn == 64 && N > 0;
  int rc = AFD_OK;
  struct Join {  // the main stream waits for the side stream on every way out
    afd_ctx* ctx;
    bool armed = false;
    ~Join() {
      if (armed) cudaStreamWaitEvent(ctx->stream, ctx->ev_join, 0);
    }
  } join{ctx};
  auto fork_prefetch = [&](int units, int sms) -> int {
    const int64_t bytes = (int64_t)units * 256 * c.hidden * 2;
    const int64_t w13 = (int64_t)c.num_experts * 2 * c.inter * c.hidden * 2;
    LaunchCtx side = lc;
    side.stream = ctx->side;
    side.pdl = 0;
    int r = cuda_fail(cudaEventRecord(ctx->ev_fork, ctx->stream), "fork");
    if (!r) r = cuda_fail(cudaStreamWaitEvent(ctx->side, ctx->ev_fork, 0), "fork");
    if (!r) r = cuda_fail(launch_prefetch_l2(side, L ? L->W13 : nullptr, std::min(bytes, w13), ws, sms),
                          "prefetch");
    if (!r) r = cuda_fail(cudaEventRecord(ctx->ev_join, ctx->side), "join");
    if (!r) join.armed = true;
    return r;
  };
  // stage timing marks only for host-described steps
  auto mark = [&](int i) {
    if (!dev) ctx->mark(i);
  };
  if (prefetch && !dev) {
    rc = fork_prefetch(ctx->num_sms * 5 / 8, std::max(1, ctx->num_sms / 8));
    if (rc) return rc;
  }
  mark(0);
  const int rows_cap = (int)routed_cap_of(&c);
  // host-described routed steps: the router starts once the check has the
  // flags (ws.go), not when the check ends
  uint32_t go = 0;
  if (!dev && !grouped) {
    ctx->go_seq = ctx->go_seq % 0x7ffffffeu + 1u;
    go = ctx->go_seq;
  }
  rc = cuda_fail(dev ? launch_item_head(lc, ctx->geom, ctx->win[0], *dev, ws, c.num_experts,
                                        c.token_cap, rows_cap, f.ffn_rank, f.ffn_size, has_shared,
                                        grouped, ctx->tmax, ctx->tmax * c.topk, c.max_layers,
                                        ctx->timeout())
                     : launch_header_check(lc, ctx->geom, ctx->win[0], f, ws, c.num_experts,
                                           c.token_cap, rows_cap, has_shared, ctx->timeout(), go),
                 "header check");
  if (rc) return rc;
  mark(1);
  if (prefetch && dev) {
    rc = fork_prefetch(ctx->num_sms * 3 / 8, ctx->num_sms);
    if (rc) return rc;
  }
  if (!grouped) {  // the grouped form arrives routed
    rc = cuda_fail(launch_router(lc, ctx->geom, ctx->win[0], f, ws, c.hidden, ctx->act_f32,
                                 L ? L->WgQ : nullptr, L ? L->bias : nullptr, c.num_experts, c.topk, c.renorm, c.routed_scaling,
                                 ws.logits, ws.hist, go, ctx->timeout()),
                   "router");
    if (rc) return rc;
  }
  mark(2);
  rc = cuda_fail(grouped ? launch_plan_grouped(lc, f, ws, c.num_experts, c.inter, c.shared_inter,
                                                c.hidden, has_shared, bn, ctx->plan1, ctx->plan2,
                                                ctx->geom, row_bytes, in_place, sh_in_place)
                         : launch_plan(lc, f, ws, c.num_experts, c.topk, c.inter, c.shared_inter,
                                       c.hidden, has_shared, bn, ctx->plan1, ctx->plan2, ws.hist,
                                       ws.base, ctx->geom, row_bytes, sh_in_place),
                 "plan");
  if (rc) return rc;
  mark(3);
  // small host-described token-form steps: the gather writes the return
  // headers and the combine releases the flags (no return-header kernel)
  const bool flags_in_combine = !grouped && combine_releases_flags(lc, f, c.hidden, c.topk);
  if (!in_place) {
    rc = cuda_fail(launch_gather(lc, ctx->geom, ctx->win[0], f, ws, c.topk, row_bytes, c.hidden,
                                 has_shared, sh_in_place, flags_in_combine ? ctx->win[1] : nullptr,
                                 c.num_experts, ws.base),
                   "gather");
    if (rc) return rc;
  }
  mark(4);
  // rows each GEMM output holds: the workspace's (routed, shared) capacity,
  // or the return window's rows when the outputs go there in place
  const int64_t Tcap = ctx->tmax;
  const int64_t win_rows = ctx->L.window_bytes / row_bytes;
  if (N + T > 0) {
    if (c.gemm != AFD_GEMM_SIMT) {
      auto launch = c.gemm == AFD_GEMM_TENSOR ? launch_gemm_tc2 : launch_gemm_tc;
      GemmArgs a1;
      memset(&a1, 0, sizeof a1);
      if (L) {
        a1.tmA[0] = L->tmA1[0];
        a1.tmA[1] = L->tmA1[1];
      } else {
        a1.layers = ws.layers;
        a1.item = ws.item;
        a1.wsel = 1;
      }
      // routed rows: gathered into Xp, or in their slots (grouped form, one
      // peer); shared rows: gathered after them, or in the slots' shared_x
      const bool sh_win = in_place || sh_in_place;
      a1.tmB[0] = in_place ? ctx->tmWin : ctx->tmXp;
      a1.tmBs[0] = in_place ? ctx->tmWin32 : ctx->tmXp32;
      a1.tmB[1] = sh_win ? ctx->tmWin : ctx->tmXp;
      a1.tmBs[1] = sh_win ? ctx->tmWin32 : ctx->tmXp32;
      a1.out[0] = ws.h;
      a1.out[1] = ws.hs;
      a1.out_fmt[0] = a1.out_fmt[1] = OUT_ACT;
      a1.ldo[0] = c.inter;
      a1.ldo[1] = c.shared_inter;
      a1.K[0] = a1.K[1] = c.hidden;
      a1.M[0] = 2 * c.inter;
      a1.M[1] = 2 * c.shared_inter;
      a1.plan = ctx->plan1;
      a1.status = ws.status;
      a1.out_rows[0] = Tcap * c.topk;
      a1.out_rows[1] = Tcap;
      a1.dbg = ws.dbg;
      a1.swiglu = 1;
      a1.bn = bn;
      a1.timeout_ns = ctx->timeout();
      GemmArgs a2;
      memset(&a2, 0, sizeof a2);
      if (L) {
        a2.tmA[0] = L->tmA2[0];
        a2.tmA[1] = L->tmA2[1];
      } else {
        a2.layers = ws.layers;
        a2.item = ws.item;
        a2.wsel = 2;
      }
      a2.tmB[0] = ctx->tmH;
      a2.tmB[1] = ctx->tmHs;
      a2.tmBs[0] = ctx->tmH32;
      a2.tmBs[1] = ctx->tmHs32;
      a2.out[0] = ws.y;
      a2.out[1] = ws.s;
      a2.ldo[0] = a2.ldo[1] = c.hidden;
      // token form: y keeps 24 bits up to the combine, whose weighted sum of
      // a token's k outputs may cancel to far less than each of them (a bf16
      // y would be rounded by up to 2^-9 of itself before that sum); the
      // grouped form returns each row's output in the activation type; the
      // shared output stays fp32
      a2.out_fmt[0] = grouped ? OUT_ACT : OUT_Y24;
      a2.out_lo[0] = ws.y_lo;
      // the shared output in fp32 (as 24-bit planes like y it measured 9 us
      // slower over the V2-Lite prefill GEMMs: two stores per element)
      a2.out_fmt[1] = OUT_F32;
      if (in_place) {  // outputs straight into the return slots (rows = window rows)
        a2.out[0] = a2.out[1] = ctx->win[1];
        a2.out_fmt[1] = OUT_ACT;
      }
      a2.K[0] = c.inter;
      a2.K[1] = c.shared_inter;
      a2.M[0] = a2.M[1] = c.hidden;
      a2.plan = ctx->plan2;
      a2.status = ws.status;
      a2.out_rows[0] = in_place ? win_rows : Tcap * c.topk;
      a2.out_rows[1] = in_place ? win_rows : Tcap;
      a2.dbg = ws.dbg;
      a2.swiglu = 0;
      a2.bn = bn;
      a2.timeout_ns = ctx->timeout();
      if (c.gemm == AFD_GEMM_TENSOR && !(c.flags & AFD_CFG_SPLIT_GEMMS)) {
        // one launch: down units start as soon as their token tile's h rows are stored
        rc = cuda_fail(launch_gemm_tc2_pair(lc, a1, a2, ws.dep), "gemm");
        if (rc) return rc;
        mark(5);
      } else {
        rc = cuda_fail(launch(lc, a1), "gemm1");
        if (rc) return rc;
        mark(5);
        rc = cuda_fail(launch(lc, a2), "gemm2");
        if (rc) return rc;
      }
    } else {
      SimtArgs s1;
      memset(&s1, 0, sizeof s1);
      if (L) {
        s1.A[0] = L->W13;
        s1.A[1] = L->W13s;
      } else {
        s1.layers = ws.layers;
        s1.item = ws.item;
        s1.wsel = 1;
      }
      s1.B[0] = ws.xp;
      s1.B[1] = sh_in_place ? (const void*)ctx->win[0] : ws.xp;  // window rows, or gathered
      s1.ldb[0] = s1.ldb[1] = c.hidden;
      s1.out[0] = ws.h;
      s1.out[1] = ws.hs;
      s1.ldo[0] = c.inter;
      s1.ldo[1] = c.shared_inter;
      s1.out_fmt[0] = s1.out_fmt[1] = ctx->act_f32 ? OUT_F32 : OUT_ACT;
      s1.K[0] = s1.K[1] = c.hidden;
      s1.M[0] = 2 * c.inter;
      s1.M[1] = 2 * c.shared_inter;
      s1.act_f32 = ctx->act_f32;
      s1.swiglu = 1;
      s1.plan = ctx->plan1;
      s1.status = ws.status;
      s1.out_rows[0] = Tcap * c.topk;
      s1.out_rows[1] = Tcap;
      s1.dbg = ws.dbg;
      rc = cuda_fail(launch_gemm_simt(lc, s1, c.num_experts + f.n_peers), "simt gemm1");
      if (rc) return rc;
      mark(5);
      SimtArgs s2 = s1;
      if (L) {
        s2.A[0] = L->Wd;
        s2.A[1] = L->Wds;
      } else {
        s2.wsel = 2;
      }
      s2.B[0] = ws.h;
      s2.B[1] = ws.hs;
      s2.ldb[0] = c.inter;
      s2.ldb[1] = c.shared_inter;
      s2.out[0] = ws.y;
      s2.out[1] = ws.s;
      s2.ldo[0] = s2.ldo[1] = c.hidden;
      s2.out_fmt[0] = ctx->act_f32 ? OUT_F32 : (grouped ? OUT_ACT : OUT_Y24);
      s2.out_lo[0] = ws.y_lo;
      s2.out_fmt[1] = OUT_F32;
      s2.K[0] = c.inter;
      s2.K[1] = c.shared_inter;
      s2.M[0] = s2.M[1] = c.hidden;
      s2.swiglu = 0;
      s2.plan = ctx->plan2;
      rc = cuda_fail(launch_gemm_simt(lc, s2, c.num_experts + f.n_peers), "simt gemm2");
      if (rc) return rc;
    }
  } else {
    mark(5);
  }
  mark(6);
  // the grouped form returns the expert outputs row by row (the Attention
  // side weights and combines); the token form combines here
  rc = cuda_fail(grouped ? (in_place ? cudaSuccess
                                     : launch_scatter_grouped(lc, ctx->geom, ctx->win[1], f, ws,
                                                              c.hidden, ctx->act_f32, has_shared))
                         : launch_combine(lc, ctx->geom, ctx->win[1], f, ws, c.hidden, c.topk,
                                          ctx->act_f32, has_shared, flags_in_combine),
                 grouped ? "scatter" : "combine");
  if (rc) return rc;
  mark(7);
  if (!flags_in_combine) {
    rc = cuda_fail(launch_return_header(lc, ctx->geom, ctx->win[1], ctx->win[0], f, ws, c.num_experts,
                                        c.topk),
                   "return header");
    if (rc) return rc;
  }
  mark(8);
  ctx->last_T = dev ? -1 : (int)T;
  ctx->forwards++;
  return AFD_OK;
}

int afd_pack_slots(afd_ctx* ctx, int n, const int32_t* peers, int stage, int layer,
                   const void* const* x, const int32_t* n_tokens, int with_shared,
                   const uint64_t* seq) {
  if (!ctx || n < 0 || n > AFD_MAX_PEERS || (n > 0 && (!peers || !x || !n_tokens || !seq)))
    return AFD_ERR_ARG;
  const afd_config& c = ctx->cfg;
  if (c.ffn_size >= 1) return AFD_ERR_ARG;  // ranks receive afd_attn_dispatch
  if (stage < 0 || stage >= c.ring_depth) return AFD_ERR_ARG;
  if (with_shared && c.shared_inter <= 0) return AFD_ERR_ARG;
  PackList pl;
  memset(&pl, 0, sizeof pl);
  bool seen[AFD_MAX_PEERS] = {};
  for (int i = 0; i < n; i++) {  // every argument before anything is launched
    const int p = peers[i];
    if (p < 0 || p >= c.num_peers || seen[p] || n_tokens[i] < 0) return AFD_ERR_ARG;
    seen[p] = true;
    if (n_tokens[i] > c.token_cap) return AFD_ERR_CAPACITY;
    if (n_tokens[i] > 0) {
      const int rc = check_dev_ptr(x[i]);
      if (rc) return rc;
      if (!aligned16(x[i])) return AFD_ERR_ARG;
    }
    if (seq[i] <= ctx->last_seq[(size_t)p * c.ring_depth + stage]) return AFD_ERR_SEQ;
    pl.region[i] = p;
    pl.n_rows[i] = n_tokens[i];
    pl.rows[i] = n_tokens[i] > 0 ? static_cast<const uint4*>(x[i]) : nullptr;
    pl.seq[i] = seq[i];
  }
  pl.n = n;
  const int row_bytes = c.hidden * (ctx->act_f32 ? 4 : 2);
  const int rc = cuda_fail(launch_pack_multi(ctx->lc(), ctx->geom, ctx->win[0], stage, layer, pl, with_shared,
                                             row_bytes, c.num_experts),
                           "pack");
  if (!rc)
    for (int i = 0; i < n; i++) ctx->last_seq[(size_t)peers[i] * c.ring_depth + stage] = seq[i];
  return rc;
}

int afd_unpack_splits(afd_ctx* ctx, int n, const int32_t* peers, int stage, void* const* out,
                      const int32_t* n_tokens, const uint64_t* expect_seq) {
  if (!ctx || n < 0 || n > AFD_MAX_PEERS || (n > 0 && (!peers || !out || !n_tokens || !expect_seq)))
    return AFD_ERR_ARG;
  const afd_config& c = ctx->cfg;
  if (stage < 0 || stage >= c.ring_depth) return AFD_ERR_ARG;
  UnpackList ul;
  memset(&ul, 0, sizeof ul);
  for (int i = 0; i < n; i++) {
    const int p = peers[i];
    if (p < 0 || p >= c.num_peers || n_tokens[i] < 0) return AFD_ERR_ARG;
    if (n_tokens[i] > c.token_cap) return AFD_ERR_CAPACITY;
    if (n_tokens[i] > 0) {
      const int rc = check_dev_ptr(out[i]);
      if (rc) return rc;
      if (!aligned16(out[i])) return AFD_ERR_ARG;
    }
    ul.region[i] = p;
    ul.n_rows[i] = n_tokens[i];
    ul.out[i] = n_tokens[i] > 0 ? static_cast<uint4*>(out[i]) : nullptr;
    ul.seq[i] = expect_seq[i];
  }
  ul.n = n;
  const int row_bytes = c.hidden * (ctx->act_f32 ? 4 : 2);
  return cuda_fail(launch_unpack_multi(ctx->lc(), ctx->geom, ctx->win[1], stage, ul, row_bytes, c.num_experts,
                                       ctx->ws.status, ctx->timeout()),
                   "unpack");
}

int afd_unpack_split(afd_ctx* ctx, int peer, int stage, void* out, int n_tokens,
                     uint64_t expect_seq) {
  if (!ctx) return AFD_ERR_ARG;
  const afd_config& c = ctx->cfg;
  if (peer < 0 || peer >= c.num_peers || stage < 0 || stage >= c.ring_depth || n_tokens < 0)
    return AFD_ERR_ARG;
  if (n_tokens > c.token_cap) return AFD_ERR_CAPACITY;
  if (n_tokens > 0) {
    const int rc = check_dev_ptr(out);
    if (rc) return rc;
    if (!aligned16(out)) return AFD_ERR_ARG;
  }
  const int row_bytes = c.hidden * (ctx->act_f32 ? 4 : 2);
  return cuda_fail(launch_unpack(ctx->lc(), ctx->geom, ctx->win[1], peer, stage, out, n_tokens,
                                 row_bytes, c.num_experts, expect_seq, ctx->ws.status,
                                 ctx->timeout(), ctx->geom.routed_x, n_tokens, -1),
                   "unpack");
}

int afd_unpack_grouped(afd_ctx* ctx, int peer, int stage, void* y_out, int n_rows, void* s_out,
                       int n_tokens, uint64_t expect_seq) {
  if (!ctx) return AFD_ERR_ARG;
  const afd_config& c = ctx->cfg;
  if (peer < 0 || peer >= c.num_peers || stage < 0 || stage >= c.ring_depth || n_rows < 0 ||
      n_tokens < 0)
    return AFD_ERR_ARG;
  if (n_rows > routed_cap_of(&c) || n_tokens > c.token_cap) return AFD_ERR_CAPACITY;
  for (const void* p : {y_out, s_out}) {
    if (!p) continue;
    const int rc = check_dev_ptr(p);
    if (rc) return rc;
    if (!aligned16(p)) return AFD_ERR_ARG;
  }
  if ((n_rows && !y_out) || (s_out && c.shared_inter <= 0)) return AFD_ERR_ARG;
  const int row_bytes = c.hidden * (ctx->act_f32 ? 4 : 2);
  // the peer's shared rows at this rank: all its tokens, or its round-robin share
  const int n_shared = rr_rows(n_tokens, c.ffn_size >= 1 ? c.ffn_rank : 0, std::max(1, c.ffn_size));
  int rc = cuda_fail(launch_unpack(ctx->lc(), ctx->geom, ctx->win[1], peer, stage, y_out, n_rows,
                                   row_bytes, c.num_experts, expect_seq, ctx->ws.status,
                                   ctx->timeout(), ctx->geom.routed_x, n_tokens, n_rows),
                     "unpack");
  if (!rc && s_out)
    rc = cuda_fail(launch_unpack(ctx->lc(), ctx->geom, ctx->win[1], peer, stage, s_out, n_shared,
                                 row_bytes, c.num_experts, expect_seq, ctx->ws.status,
                                 ctx->timeout(), ctx->geom.shared_x, n_tokens, n_rows),
                   "unpack");
  return rc;
}

int afd_poll_status(afd_ctx* ctx) {
  if (!ctx) return AFD_ERR_ARG;
  if (cuda_fail(cudaStreamSynchronize(ctx->stream), "stream sync")) return AFD_ERR_CUDA;
  int32_t st = 0;
  if (cuda_fail(cudaMemcpy(&st, ctx->ws.status, 4, cudaMemcpyDeviceToHost), "status read"))
    return AFD_ERR_CUDA;
  if (st && cuda_fail(cudaMemset(ctx->ws.status, 0, 4), "status clear")) return AFD_ERR_CUDA;
  return st;
}

int afd_get_config(afd_ctx* ctx, afd_config* out) {
  if (!ctx || !out) return AFD_ERR_ARG;
  *out = ctx->cfg;
  return AFD_OK;
}

int afd_get_window(afd_ctx* ctx, int direction, void** dev_ptr, int64_t* bytes) {
  if (!ctx || (direction != AFD_DIR_DISPATCH && direction != AFD_DIR_RETURN)) return AFD_ERR_ARG;
  if (dev_ptr) *dev_ptr = ctx->win[direction];
  if (bytes) *bytes = ctx->L.window_bytes;
  return AFD_OK;
}

int afd_get_workspace(afd_ctx* ctx, int which, void** dev_ptr, int64_t* bytes) {
  if (!ctx || which < 0 || which > AFD_WS_STATUS) return AFD_ERR_ARG;
  void* ptrs[12] = {ctx->ws.ids, ctx->ws.w, ctx->ws.counts, ctx->ws.offsets, ctx->ws.perm,
                    ctx->ws.inv, ctx->ws.xp, ctx->ws.h, ctx->ws.y, ctx->ws.hs, ctx->ws.s,
                    ctx->ws.status};
  if (dev_ptr) *dev_ptr = ptrs[which];
  if (bytes) *bytes = ctx->ws_cap[which];
  return AFD_OK;
}

int afd_get_stats(afd_ctx* ctx, afd_stats* out) {
  if (!ctx || !out) return AFD_ERR_ARG;
  out->window_bytes = ctx->L.window_bytes;
  out->workspace_bytes = ctx->ws_bytes;
  out->last_total_tokens = ctx->last_T;
  out->num_sms = ctx->num_sms;
  out->forwards = ctx->forwards;
  return AFD_OK;
}

int afd_last_expert_counts(afd_ctx* ctx, int32_t* counts, int n, int* n_experts) {
  if (!ctx || !counts || n < 1) return AFD_ERR_ARG;
  if (cuda_fail(cudaStreamSynchronize(ctx->stream), "stream sync")) return AFD_ERR_CUDA;
  const int m = std::min(n, ctx->cfg.num_experts);
  if (cuda_fail(cudaMemcpy(counts, ctx->ws.counts, (size_t)m * 4, cudaMemcpyDeviceToHost),
                "expert counts read"))
    return AFD_ERR_CUDA;
  if (n_experts) *n_experts = ctx->cfg.num_experts;
  return AFD_OK;
}

int64_t afd_launch_count(afd_ctx* ctx) { return ctx ? ctx->launches : -1; }

int afd_debug_bounds(afd_ctx* ctx, int32_t* site, int64_t* index, int64_t* limit) {
#ifdef AFD_DEBUG_BOUNDS
  if (!ctx) return AFD_ERR_ARG;
  int64_t rec[4];
  if (cuda_fail(cudaStreamSynchronize(ctx->stream), "stream sync") ||
      cuda_fail(cudaMemcpy(rec, ctx->ws.dbg, sizeof rec, cudaMemcpyDeviceToHost), "bounds record"))
    return AFD_ERR_CUDA;
  if (!rec[0]) return AFD_OK;
  if (site) *site = (int32_t)rec[1];
  if (index) *index = rec[2];
  if (limit) *limit = rec[3];
  return AFD_ERR_BOUNDS;
#else
  (void)ctx; (void)site; (void)index; (void)limit;
  return AFD_ERR_UNSUPPORTED;
#endif
}

int afd_debug_plant(afd_ctx* ctx, int32_t site) {
#ifdef AFD_DEBUG_BOUNDS
  if (!ctx || site < 0 || site >= AFD_DBG_NUM_SITES) return AFD_ERR_ARG;
  const int64_t rec[5] = {0, 0, 0, 0, site};
  if (cuda_fail(cudaStreamSynchronize(ctx->stream), "stream sync") ||
      cuda_fail(cudaMemcpy(ctx->ws.dbg, rec, sizeof rec, cudaMemcpyHostToDevice), "bounds record"))
    return AFD_ERR_CUDA;
  return AFD_OK;
#else
  (void)ctx; (void)site;
  return AFD_ERR_UNSUPPORTED;
#endif
}

int afd_check_canaries(afd_ctx* ctx, int* window, int64_t* offset) {
  if (!ctx || !ctx->L.guard || !ctx->canary_result) return AFD_ERR_ARG;
  if (cuda_fail(cudaStreamSynchronize(ctx->stream), "stream sync")) return AFD_ERR_CUDA;
  const CanaryGeom cg = canary_geom(ctx);
  for (int d = 0; d < 2; d++) {
    const unsigned long long init[2] = {0ull, ~0ull};
    unsigned long long res[2];
    if (cuda_fail(cudaMemcpy(ctx->canary_result, init, sizeof init, cudaMemcpyHostToDevice), "canary") ||
        cuda_fail(launch_canary(ctx->stream, ctx->win[d], cg, 0, ctx->canary_result, ctx->num_sms),
                  "canary check") ||
        cuda_fail(cudaStreamSynchronize(ctx->stream), "canary check") ||
        cuda_fail(cudaMemcpy(res, ctx->canary_result, sizeof res, cudaMemcpyDeviceToHost), "canary"))
      return AFD_ERR_CUDA;
    if (res[0]) {
      if (window) *window = d;
      if (offset) *offset = (int64_t)res[1];
      return AFD_ERR_CANARY;
    }
  }
  return AFD_OK;
}

int afd_profile(afd_ctx* ctx, int enable) {
  if (!ctx) return AFD_ERR_ARG;
  if (enable && !ctx->events_made) {
    for (auto& set : ctx->ev)
      for (auto& e : set)
        if (cuda_fail(cudaEventCreate(&e), "event create")) return AFD_ERR_CUDA;
    ctx->events_made = true;
  }
  ctx->profiling = enable != 0;
  return AFD_OK;
}

int afd_stage_times(afd_ctx* ctx, float* ms, int n, int64_t* forwards) {
  if (!ctx || !ms || n < 0 || n > AFD_NUM_STAGES || !ctx->events_made) return AFD_ERR_ARG;
  while (ctx->prof_pending > 0)
    if (ctx->fold_oldest()) return cuda_fail(cudaGetLastError(), "stage events");
  for (int i = 0; i < n; i++) ms[i] = (float)ctx->prof_acc[i];
  if (forwards) *forwards = ctx->prof_acc_n;
  for (double& a : ctx->prof_acc) a = 0.0;
  ctx->prof_acc_n = 0;
  return AFD_OK;
}

}  // extern "C"
