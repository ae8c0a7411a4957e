// afd_internal.cuh -- structures shared by the host side and the kernels of
// the AFD FFN-side library, plus thin inline-PTX wrappers for sm_103a.
#pragma once

#include <cuda.h>
#include <algorithm>
#include <cstring>
#include <utility>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/afd.h"

#include <atomic>

// Launch settings the launchers cache (a kernel's shared-memory attribute,
// occupancy figures) are per device: a process may hold contexts on several.
constexpr int kMaxCachedDevices = 64;
inline int current_device() {
  int d = 0;
  return cudaGetDevice(&d) == cudaSuccess && d >= 0 && d < kMaxCachedDevices ? d : -1;
}
// the kernel's dynamic shared memory limit raised to `bytes`, once per device
template <typename K>
cudaError_t smem_attr_once(K kernel, int bytes, std::atomic<int>* done /* [kMaxCachedDevices] */) {
  const int d = current_device();
  if (d >= 0 && done[d].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && d >= 0) done[d].store(1, std::memory_order_release);
  return e;
}

#define AFD_MAX_GROUPS 320   // routed experts (<= 256) + one shared group

// ---------------------------------------------------------------------------
// per-forward fan-in description (Data on the wire, step 3: the input is the
// concatenation of the listed peers' rows in list order).  The host
// describes it for afd_ffn_forward and passes it by value to every kernel of
// the step.  In the work-item loop (dev set) the head kernel builds it from
// the slot headers into the workspace (ws.item) and the kernels read it
// there; the host's copy then gives only the launch shapes.
// ---------------------------------------------------------------------------
struct FanIn {
  int n_peers;
  int stage;
  int layer;
  int total;                          // T = sum of seq_lens
  int prefix[AFD_MAX_PEERS + 1];      // exclusive prefix of seq_lens
  int region[AFD_MAX_PEERS];          // peer (window region) of list entry i
  // grouped form (the Attention side routed): the routed rows of entry i
  // are rows [rprefix[i], rprefix[i + 1]) of their concatenation
  int grouped;
  int num_experts;                    // grouped form: E (row placement in the gather)
  int rtotal;
  int rprefix[AFD_MAX_PEERS + 1];
  int dev;                            // 1: the step's values are in ws.item
  // shared rows: entry i's are rows [sprefix[i], sprefix[i + 1]) of their
  // concatenation -- its tokens with one FFN rank, its round-robin share
  // (tokens ffn_rank, ffn_rank + ffn_size, ...) with several
  int ffn_rank, ffn_size;
  int stotal;
  int sprefix[AFD_MAX_PEERS + 1];
};

// how many of the tokens r, r + F, r + 2F, ... are below n
__host__ __device__ inline int rr_rows(int n, int r, int F) {
  return n > r ? (n - r + F - 1) / F : 0;
}

// the listed peers of a work-item loop (the peers of one Attention replica)
struct PeerList {
  int n;
  int slot[AFD_MAX_PEERS];
};

// per-layer weights as the kernels see them when the layer of a step is
// chosen on the device: the TMA maps and plain pointers of every layer,
// one entry per layer in device memory ("layer-select" operators of the
// Async AFD RFC: the address table of every layer plus a device-side index)
struct DevLayer {  // aligned as its tensor maps
  CUtensorMap tmA1[2];    // SwiGLU GEMM weights: routed experts, shared expert
  CUtensorMap tmA2[2];    // down GEMM weights
  const float* WgQ;       // router weight, rearranged
  const float* bias;
  const void* W13;
  const void* W13s;
  const void* Wd;
  const void* Wds;
  int set;
};

// workspace words of the work-item loop
#define AFD_LOOP_ROT 0        // stage the next scan starts at
#define AFD_LOOP_COUNT 1      // items served so far
#define AFD_LOOP_LOG 2        // AFD_LOOP_LOG_N records of 4 words: stage, layer, T, rows
#define AFD_LOOP_LOG_N 64
#define AFD_LOOP_WORDS (AFD_LOOP_LOG + 4 * AFD_LOOP_LOG_N)

// group list carried by value into the header-writing kernel
struct GroupList {
  int32_t n[256];
};

// several peers' slots packed or unpacked in one launch (by value)
struct PackList {
  int n;
  int region[AFD_MAX_PEERS];
  int n_rows[AFD_MAX_PEERS];
  const uint4* rows[AFD_MAX_PEERS];
  uint64_t seq[AFD_MAX_PEERS];
};
struct UnpackList {
  int n;
  int region[AFD_MAX_PEERS];
  int n_rows[AFD_MAX_PEERS];
  uint4* out[AFD_MAX_PEERS];
  uint64_t seq[AFD_MAX_PEERS];  // the flag value each expects
};

// window geometry (both windows share it)
struct WinGeom {
  int64_t flags_bytes, slot_bytes;
  int64_t header, route_table, routed_x, shared_idx, shared_x;
  int ring_depth;
  int num_regions;
};

// Guard regions of a window (AFD_CFG_CANARY): `guard` bytes before
// flags_bytes, and in every slot `guard` bytes at each of the n offsets in
// goff (relative to the slot).  The word at byte offset o of the window
// holds canary_word(o).
struct CanaryGeom {
  int64_t flags_bytes, slot_bytes, guard;
  int64_t goff[5];
  int n, nslots;
};
__host__ __device__ inline uint32_t canary_word(int64_t off) {
  return 0xCA11AFD0u ^ (uint32_t)(off >> 2) ^ ((uint32_t)(off >> 34) << 16);
}
// fill: write the pattern; else count changed words into result[0] and the
// lowest changed offset into result[1] (initialised by the caller)
cudaError_t launch_canary(cudaStream_t stream, uint8_t* win, const CanaryGeom& cg, int fill,
                          unsigned long long* result, int num_sms);

// workspace pointers
struct DevWS {
  int32_t* status;        // [1] sticky first error
  uint64_t* seen;         // [regions * ring] last dispatch flag consumed
  uint64_t* cur_seq;      // [MAX_PEERS] flag value consumed by this forward
  int32_t* peer_shared;   // [MAX_PEERS] 1 if entry i carries shared rows
  int32_t* ids;           // [Tmax * k]
  float* w;               // [Tmax * k]
  int32_t* counts;        // [E]
  int32_t* offsets;       // [E + 1]
  int32_t* perm;          // [Tmax * k]
  int32_t* inv;           // [Tmax * k]
  int32_t* peer_counts;   // [MAX_PEERS * E] (grouped form: the received group lists)
  int32_t* gbase;         // [2 * MAX_PEERS * E] grouped form: row bases, group-list prefixes
  void* xp;               // act [Tmax * k + Tmax, H]
  void* h;                // act [Tmax * k, I]
  void* y;                // routed down-projection outputs [Tmax * k, H]: token form
                          // y24 high plane (u16), grouped form act; fp32 with fp32
                          // activations
  uint8_t* y_lo;          // token form, bf16 activations: y24 low plane (u8) [Tmax * k, H]
  void* hs;               // act [Tmax, Is]
  float* s;               // f32 [Tmax, H]
  int32_t* hist;          // [E, router CTAs] per-CTA expert histograms
  int32_t* base;          // [E, router CTAs] each CTA's first slot in each expert segment
  float* logits;          // [Tmax, E] router logits
  FanIn* item;            // the fan-in of the step in flight
  const DevLayer* layers; // [max_layers] per-layer weights
  int32_t* loop;          // [AFD_LOOP_WORDS] work-item loop state and log
  uint32_t* go;           // [1] the header check's word for the router (AFD_GO_ABORT)
  int32_t* ret_count;     // [MAX_PEERS] combine items finished per entry (return flags)
  int64_t* dbg;           // [8] debug build: failed checks, site, index, limit; [4] planted site
  int32_t* dep;           // [token tiles] SwiGLU epilogue warps done per token tile (one-launch GEMMs)
};

// Debug build (AFD_DEBUG_BOUNDS): index idx, derived from data an earlier
// kernel wrote, must lie in [0, limit) before it is used.  A failure (or a
// planted site, whose bound counts as 0) is recorded once, sets the step's
// status, and returns false: the caller skips the access or uses index 0.
// The release build compiles the check out.
__device__ __forceinline__ bool dbg_in_range(int64_t* dbg, int32_t* status, int site, int64_t idx,
                                             int64_t limit) {
#ifdef AFD_DEBUG_BOUNDS
  if (dbg[4] == site) limit = 0;
  if (idx >= 0 && idx < limit) return true;
  if (atomicAdd(reinterpret_cast<unsigned long long*>(dbg), 1ull) == 0ull) {
    dbg[1] = site;
    dbg[2] = idx;
    dbg[3] = limit;
  }
  atomicCAS(status, 0, AFD_ERR_BOUNDS);
  return false;
#else
  (void)dbg; (void)status; (void)site; (void)idx; (void)limit;
  return true;
#endif
}

// The header check of a host-described step publishes, once every listed
// flag is acquired, the step's go token in ws.go (release); the router's
// CTAs start under programmatic dependent launch, load their gate weights,
// and read the fan-in's rows once they see it (acquire).  Token | ABORT:
// the check found an earlier error or a flag wait ran out; the router then
// does no work (the check reports the error).
#define AFD_GO_ABORT 0x80000000u

// one group of the grouped GEMM: rows of the B operand (tokens) that share
// one weight matrix (an expert, or the shared expert)
struct GemmGroup {
  int rows;      // tokens in the group
  int b_row0;    // first row in the B source
  int out_row0;  // first output row
  int a_idx;     // expert index in the weight tensor
  int kind;      // 0 routed, 1 shared
  int m_tiles;   // 128-row tiles of the weight (M) dimension
  int n_tiles;   // token tiles
  int tile0;     // first linear tile index of the group (one CTA per tile)
  int unit0;     // first pair-tile index (two CTAs, 256 weight rows per unit)
  int nt0;       // first token-tile index over all groups (the same in both plans)
};

struct GemmPlan {
  int ngroups;
  int total_tiles;
  int bn;        // token tile
  int total_units;
  int total_ntiles;
  GemmGroup g[AFD_MAX_GROUPS];
};

// Output formats of the GEMMs.  OUT_Y24 keeps an fp32 result to 24 bits
// (sign, 8 exponent bits, 15 mantissa bits; the low 8 bits rounded off, half
// away from zero) as two planes: the high 16 bits (a bf16 bit pattern, the
// value truncated) and the next 8 bits.  The token form's routed outputs y
// use it: their weighted sum in the combine may cancel to far less than its
// terms, against which a bf16 y (relative rounding 2^-9) is too coarse, and
// 3 bytes per element instead of fp32's 4 cut the combine's reads by a
// quarter (relative rounding 2^-16).
#define OUT_ACT 0
#define OUT_F32 1
#define OUT_Y24 2

// Arguments of the tensor-core grouped GEMM (one launch = one projection).
struct GemmArgs {
  CUtensorMap tmA[2];     // weights: [0] routed experts, [1] shared expert
  CUtensorMap tmB[2];     // token rows: [0] routed source, [1] shared source
                          // (box 64 x 32 rows for the one-CTA engine, 64 x 128
                          // rows for the SM-pair engine)
  CUtensorMap tmBs[2];    // the same sources with 64 x 32 boxes: the SM-pair
                          // engine uses them for units of <= 64 tokens
  void* out[2];           // outputs per kind
  uint8_t* out_lo[2];     // OUT_Y24: the low plane (one byte per element, pitch ldo)
  int64_t ldo[2];         // output row pitch in elements
  int out_fmt[2];         // OUT_ACT (bf16), OUT_F32 or OUT_Y24
  int K[2];               // reduction length per kind
  int M[2];               // weight rows per kind (2I for SwiGLU, H for down)
  const GemmPlan* plan;
  int32_t* status;
  int swiglu;             // 1: gate/up interleaved SwiGLU epilogue
  int bn;                 // the plan's token tile (rows per unit)
  int64_t timeout_ns;
  // layer chosen on the device: tmA is ignored and the weight maps are
  // layers[item->layer].tmA1 (wsel 1) or .tmA2 (wsel 2)
  const DevLayer* layers;
  const FanIn* item;
  int wsel;
  int64_t out_rows[2];    // rows each output holds (checked in the debug build)
  int64_t* dbg;           // the workspace's debug record (DevWS::dbg)
};

// Both projections in one launch of the SM-pair engine: the units of p[0]
// (SwiGLU), then those of p[1] (down), handed to the pairs in the same
// rounds.  A down unit reads the h rows of one token tile of one group, which
// every SwiGLU unit of that tile (one per 256-row weight pair) stores: each of
// the pair's 16 epilogue warps adds 1 to dep[group's nt0 + tile] after its
// stores (release), and the down unit's producers issue its weight loads,
// then wait (acquire, bounded) for m_pairs x 16 before loading the h rows.
// All SwiGLU units precede all down units in every pair's sequence and every
// cluster of the grid is resident at once, so the waits always end.
// nproj 1: p[0] alone, dep unused.
struct GemmPair {
  GemmArgs p[2];
  int32_t* dep;
  int nproj;
};

// SIMT GEMM arguments (fp32 activations, cross-check engine)
struct SimtArgs {
  const void* A[2];       // weights per kind: [E or 1][M][K] row-major
  const void* B[2];       // token rows per kind: [rows][K]
  int64_t ldb[2];
  void* out[2];
  uint8_t* out_lo[2];     // OUT_Y24 low plane
  int64_t ldo[2];
  int out_fmt[2];         // OUT_ACT (the activation type), OUT_F32 or OUT_Y24
  int K[2];
  int M[2];               // SwiGLU: 2I (gate rows then up rows); plain: H
  int act_f32;
  int swiglu;
  const GemmPlan* plan;
  int32_t* status;
  // layer chosen on the device: A is ignored; wsel 1 takes the layer's
  // W13 / W13s, wsel 2 its Wd / Wds
  const DevLayer* layers;
  const FanIn* item;
  int wsel;
  int64_t out_rows[2];    // rows each output holds (checked in the debug build)
  int64_t* dbg;           // the workspace's debug record (DevWS::dbg)
};

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

// fp32 -> 24-bit y (see OUT_Y24): the value's bits rounded at bit 8 (a
// finite value of magnitude within half a unit of the largest rounds to
// infinity, as a bf16 conversion would).  A NaN keeps its quiet bit instead:
// rounding the all-ones payload the tensor cores produce would carry into
// the sign bit and leave -0.
__device__ __forceinline__ uint32_t y24_encode(float v) {
  const uint32_t b = __float_as_uint(v);
  return (b & 0x7fffffffu) > 0x7f800000u ? (b >> 8) | 0x4000u : (b + 0x80u) >> 8;
}
// the two planes back to fp32: high 16 bits, then the low byte, then zero
__device__ __forceinline__ float y24_decode(uint32_t hi16, uint32_t lo8) {
  return __uint_as_float((hi16 << 16) | (lo8 << 8));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// record the first error in the sticky status word
__device__ __forceinline__ void set_error(int32_t* status, int code) {
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ int read_status(const int32_t* status) {
  return *(volatile const int32_t*)status;
}

// Flags are read and written with device scope: every peer of a window
// lives on this GPU (a cross-GPU transport would need system scope).
__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// mbarrier -------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// TMA ------------------------------------------------------------------------
// contiguous bytes global -> shared (both 16-byte aligned, size % 16 == 0)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(tm), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* tm, int c0, int c1,
                                            int c2, int c3, int c4, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
      ::"r"(dst), "l"(tm), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
      : "memory");
}

// tcgen05 -------------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 in, fp32 accumulate)
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Programmatic dependent launch.  Every kernel calls grid_dep_wait() before
// it reads anything an earlier kernel of the stream wrote (a no-op when it
// was launched without the programmatic attribute), then grid_dep_launch()
// so the next kernel's CTAs may be scheduled and run their prologue.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

#endif  // __CUDACC__

// ---------------------------------------------------------------------------
// launchers implemented in the kernel translation units (host side)
// ---------------------------------------------------------------------------
// groups of 4 experts in the rearranged router weight
__host__ __device__ inline int wgq_groups(int E) { return (E + 3) / 4; }

struct LaunchCtx {
  cudaStream_t stream;
  int num_sms;
  int64_t* launches;
  int pdl = 0;  // 1: a launch may start while the previous kernel drains
};

#ifdef __CUDACC__
// Launch with the programmatic-serialisation attribute when lc.pdl is set;
// counts the launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(const LaunchCtx& lc, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                     size_t smem, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = lc.pdl ? 1 : 0;
  ++*lc.launches;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same with thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_k_cluster(const LaunchCtx& lc, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                             size_t smem, unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = lc.pdl ? 2 : 1;
  ++*lc.launches;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
#endif

// routed_x <- rows (n_rows rows); shared_x <- xs and shared_idx = 0..n_shared-1
// when xs is not null
cudaError_t launch_pack_payload(const LaunchCtx& lc, const WinGeom& g, uint8_t* win, int region,
                                int stage, const void* rows, int n_rows, const void* xs, int n_shared,
                                int row_bytes);
// header + flag; routed_tokens and the group list are those of the grouped form
// (0 and all zero for the token form)
cudaError_t launch_pack_header(const LaunchCtx& lc, const WinGeom& g, uint8_t* win, int region,
                               int stage, int layer, int n, int with_shared, int num_experts,
                               uint64_t seq, int shutdown, int routed_tokens, const GroupList& gl);
// host-described step: bounded flag waits and header checks of the listed
// entries, then f is written to ws.item
// rows_cap: routed rows a slot may carry (token_cap, or routed_cap under
// token-level dispatch)
// go_token: 0, or the step's token (1 .. 2^31 - 1) for ws.go
cudaError_t launch_header_check(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                                const FanIn& f, const DevWS& ws, int num_experts,
                                int token_cap, int rows_cap, int has_shared_expert,
                                int64_t timeout_ns, uint32_t go_token);
// device-chosen step: bounded wait for any stage whose listed peers have all
// published, the fan-in built from their headers (token form, or the grouped
// form when grouped is set), the same checks, then ws.item.  tmax / rmax: the
// most tokens / grouped rows a step may carry; max_layers: the layer table's size.
cudaError_t launch_item_head(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                             const PeerList& pl, const DevWS& ws, int num_experts, int token_cap,
                             int rows_cap, int ffn_rank, int ffn_size, int has_shared_expert,
                             int grouped, int tmax, int rmax, int max_layers,
                             int64_t timeout_ns);
// CTAs of the router for T tokens (16 tokens each); sizes the histograms
int router_blocks(int total_tokens);
size_t router_min_smem_bytes(int hidden, int E, int act_f32);
// router: logits [T, E] fp32 (caller's scratch), then top-k / gate weights
// into ws.ids / ws.w and, if hist is not NULL, the per-16-token histograms.
// Without hist (the allocation-free entry point, which has no status poll)
// an error recorded in ws.status makes the top-k write id -1 and a NaN
// weight for every token instead of leaving the outputs unwritten.
cudaError_t launch_router(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                          const FanIn& f, const DevWS& ws, int hidden, int act_f32,
                          const float* WgQ, const float* bias, int E, int k, int renorm,
                          float scale, float* logits, int32_t* hist, uint32_t go_token = 0,
                          int64_t timeout_ns = 0);
// sh_in_place: the shared expert reads its rows in place from the slots'
// shared_x (one group per peer; g, row_bytes give the window rows) instead of
// from the gathered rows after the routed ones
cudaError_t launch_plan(const LaunchCtx& lc, const FanIn& f, const DevWS& ws, int E, int k,
                        int inter, int shared_inter, int hidden, int has_shared, int bn,
                        GemmPlan* plan1, GemmPlan* plan2, const int32_t* hist, int32_t* base,
                        const WinGeom& g, int row_bytes, int sh_in_place);
// ret_headers (not NULL): also write the step's return headers (every word
// but the flag) and zero the entries' item counters (see combine_releases_flags)
// large token-form fan-ins: the stable ranks as well (k_rank_gather, from the
// plan's bases); ret_headers is then unused (the return-header kernel runs)
cudaError_t launch_gather(const LaunchCtx& lc, const WinGeom& g, const uint8_t* win,
                          const FanIn& f, const DevWS& ws, int k, int row_bytes, int hidden,
                          int has_shared, int sh_in_place, uint8_t* ret_headers, int E,
                          const int32_t* base);
cudaError_t launch_gemm_tc(const LaunchCtx& lc, const GemmArgs& a);
cudaError_t launch_gemm_tc2(const LaunchCtx& lc, const GemmArgs& a);
// SwiGLU (a1) and down (a2) projections in one launch (GemmPair); dep: the
// workspace's per-token-tile counters, zeroed by the plan
cudaError_t launch_gemm_tc2_pair(const LaunchCtx& lc, const GemmArgs& a1, const GemmArgs& a2, int32_t* dep);
cudaError_t launch_gemm_simt(const LaunchCtx& lc, const SimtArgs& a, int max_groups);
// flags: the combine releases each entry's return flag after its last item
// (the gather wrote the headers); only where combine_releases_flags holds
cudaError_t launch_combine(const LaunchCtx& lc, const WinGeom& g, uint8_t* ret,
                           const FanIn& f, const DevWS& ws, int hidden, int k, int act_f32,
                           int has_shared, int flags);
bool combine_releases_flags(const LaunchCtx& lc, const FanIn& f, int hidden, int k);
cudaError_t launch_return_header(const LaunchCtx& lc, const WinGeom& g, uint8_t* ret,
                                 const uint8_t* win, const FanIn& f, const DevWS& ws, int E,
                                 int k);
// n rows of the return slot's field; the header must carry expect_tokens
// tokens (and expect_routed routed rows unless it is -1)
cudaError_t launch_pack_multi(const LaunchCtx& lc, const WinGeom& g, uint8_t* win, int stage, int layer,
                              const PackList& pl, int with_shared, int row_bytes, int num_experts);
cudaError_t launch_unpack_multi(const LaunchCtx& lc, const WinGeom& g, const uint8_t* ret, int stage,
                                const UnpackList& ul, int row_bytes, int num_experts, int32_t* status,
                                int64_t timeout_ns);
cudaError_t launch_unpack(const LaunchCtx& lc, const WinGeom& g, const uint8_t* ret, int region,
                          int stage, void* out, int n, int row_bytes, int num_experts,
                          uint64_t expect_seq, int32_t* status, int64_t timeout_ns, int64_t field,
                          int expect_tokens, int expect_routed);
// grouped form: plan from the received group lists; outputs back to the peers
// in_place: one GEMM group per (entry, expert) and per entry's shared rows,
// B rows read from the dispatch window, down-GEMM outputs written into the
// return window (rows given as window rows); else per-expert groups over
// the gathered Xp with a scatter afterwards
cudaError_t launch_plan_grouped(const LaunchCtx& lc, const FanIn& f, const DevWS& ws, int E,
                                int inter, int shared_inter, int hidden, int has_shared, int bn,
                                GemmPlan* plan1, GemmPlan* plan2, const WinGeom& g, int row_bytes,
                                int in_place, int sh_in_place);
cudaError_t launch_scatter_grouped(const LaunchCtx& lc, const WinGeom& g, uint8_t* ret,
                                   const FanIn& f, const DevWS& ws, int hidden, int act_f32,
                                   int has_shared);
// bytes: a multiple of 16 from a 16-byte aligned base; base NULL: the W13
// of the layer in ws.item (nothing when the step has no routed rows); sms:
// the CTAs (one per SM) that issue the 64 KB prefetches, which paces them
cudaError_t launch_prefetch_l2(const LaunchCtx& lc, const void* base, int64_t bytes,
                               const DevWS& ws, int sms);
// 128-row weight tiles of a tensor-engine weight copy, and the copy itself
// ([E][tiles][k-blocks] blocks of 128 x 64 bf16; see k_tile_weight)
int tiled_weight_tiles(int M, int swiglu, int I);
cudaError_t launch_tile_weight(const LaunchCtx& lc, const void* W, void* T, int E, int M, int K, int swiglu,
                               int I);
cudaError_t launch_arrange_wg(const LaunchCtx& lc, const float* Wg, float* WgQ, int hidden,
                                int E);
