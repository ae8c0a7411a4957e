// afd_gemm_tc2.cu -- the grouped expert GEMM on a pair of SMs:
// tcgen05.mma.cta_group::2 (kind::f16, bf16 in, fp32 accumulate in TMEM).
//
// A cluster of two CTAs computes one unit: 256 weight rows x up to 256
// tokens.  CTA r of the pair holds weight rows [128 r, 128 r + 128) of the
// unit (its own 128-row m-tile) and token rows [N/2 r, N/2 (r+1)) of the
// token tile in shared memory; the leader (r = 0) issues the MMAs, which read
// A and B from both CTAs, and each CTA's TMEM receives its 128 weight rows x
// all N tokens.  Per SM and 64-wide k-block the ring takes 16 KB of weights
// and 16 KB of tokens (one CTA alone would take 16 + 32 KB for the same
// MMA work), so six k-blocks fit in flight and each SM fills and reads a
// third less shared memory.  Weights come from the library's tiled copies
// (one contiguous 16 KB block per 128 x 64 box).  Projections and epilogues
// are those of afd_gemm_tc.cu (Async GPU Connector, "Attention gate and FFN
// expert compute": fused_experts gate/up GEMM, SiLU-and-multiply, down GEMM).
//
// Signalling (all waits bounded):
//   full[s]   leader only: one arrive + the bytes of both CTAs' copies (the
//             peer's TMA signals the leader's barrier through its cluster
//             address); the leader's MMA waits on it
//   empty[s]  both CTAs: the leader's MMA commit, multicast to the pair
//   tfull[a]  both CTAs: the leader's commit after a unit's last k-block
//   tempty[a] leader only: every epilogue warp of both CTAs arrives
// Cluster barriers after initialisation and before TMEM release keep every
// remote arrive inside the lifetime of its target.
#include "afd_internal.cuh"

namespace {

constexpr int BM = 128;            // weight rows per CTA
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr int SMALL_BOX_ROWS = 32;
constexpr int SMALL_BOX_BYTES = SMALL_BOX_ROWS * BK * 2;
constexpr int EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + EPI_WARPS * 32;
constexpr int TMEM_COLS = 512;     // two accumulators of 256 columns
constexpr int EPI_PITCH_SWIGLU = 48;
constexpr int EPI_PITCH_BF16 = 80;
constexpr int EPI_BUF_BYTES = 32 * EPI_PITCH_BF16;
constexpr uint64_t kGemmTimeoutNs = 5000000000ull;

// Ring geometry of the two variants: three stages of several adjacent
// 64-wide k-blocks, so a tile takes a half or a third of the barrier round
// trips that one k-block per stage would cost.  Wide: token tiles of up to
// 256 rows (128 per CTA), 2 k-blocks x (16 KB weights + 16 KB tokens) per
// stage; 1 x 6 stages in the same shared memory measured 2.4 % slower over
// the prefill step, 3 x 2 stages 9 % slower.  Narrow, for token tiles of
// <= 64 rows (decode-sized fan-ins, where the weights stream from HBM and the
// tensor pipe idles): 32-row token boxes, 3 k-blocks x (16 KB weights + 4 KB
// tokens) per stage, so every weight row is fetched 384 contiguous bytes at
// a time, which HBM serves measurably faster than 128-byte pieces (2 x 5
// stages measured 0.7 % slower over the decode step).
template <bool kNarrow>
struct Ring {
  static constexpr int BN_HALF = kNarrow ? 32 : 128;   // token rows per CTA
  static constexpr int KPS = kNarrow ? 3 : 2;          // k-blocks per stage
  static constexpr int STAGES = 3;
  static constexpr int B_BYTES = BN_HALF * BK * 2;
  static constexpr int STAGE_BYTES = KPS * (A_BYTES + B_BYTES);
  struct Tail {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int skip;       // this CTA's decision
    int peer_skip;  // the peer's, stored here by the peer
  };
  static constexpr size_t kEpiOffset = ((size_t)STAGES * STAGE_BYTES + sizeof(Tail) + 127) / 128 * 128;
  static constexpr size_t kSmemBytes = 1024 + kEpiOffset + (size_t)EPI_WARPS * EPI_BUF_BYTES;
  static_assert(kEpiOffset % 128 == 0 && EPI_BUF_BYTES % 128 == 0, "epilogue buffers must stay aligned");
  // (plus the static tables of both projections' first units)
  static_assert(kSmemBytes + 2 * AFD_MAX_GROUPS * sizeof(int) <= 232448,
                "over the per-CTA shared memory limit");
  static_assert(STAGE_BYTES % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// address of this CTA's shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void tma2_load_2d(uint32_t dst, const CUtensorMap* tm, int c0, int c1,
                                             uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(tm), "r"(c0), "r"(c1), "r"(bar_cluster)
      : "memory");
}
__device__ __forceinline__ void tma2_load_5d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, int c2,
                                             int c3, int c4, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
      ::"r"(dst), "l"(tm), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar_cluster)
      : "memory");
}
__device__ __forceinline__ void tc2_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p; }"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on the barrier at this offset in every CTA of the pair
__device__ __forceinline__ void tc2_commit_pair(uint32_t bar) {
  const uint16_t mask = 0x3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
      ::"r"(bar), "h"(mask)
      : "memory");
}
__device__ __forceinline__ void tc2_commit_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// kind::f16, D fp32, A and B bf16, K-major; M = 256 across the pair
__device__ __forceinline__ uint32_t idesc_pair(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
}

struct Unit {
  int group, kind, mpair, nt, rows, n_mma;
};

template <bool kNarrow>
// unit0_s: the groups' first unit indices, staged in shared memory (the
// search would otherwise chain one global load per step at every unit)
__device__ __forceinline__ Unit decode_unit(const GemmPlan& p, const int* unit0_s, int ngroups,
                                            int unit) {
  int lo = 0, hi = ngroups - 1;
  while (lo < hi) {  // last group with unit0 <= unit (empty groups share unit0 with the next)
    const int mid = (lo + hi + 1) >> 1;
    if (unit0_s[mid] <= unit) lo = mid; else hi = mid - 1;
  }
  const GemmGroup& G = p.g[lo];
  const int u = unit - G.unit0;
  Unit t;
  t.group = lo;
  t.kind = G.kind;
  if (kNarrow) {
    // decode-sized groups stream their weights from HBM: token tiles vary
    // fastest, so the units sharing a weight tile run on neighbouring
    // clusters and the second read of the tile hits L2
    t.nt = u % G.n_tiles;
    t.mpair = u / G.n_tiles;
  } else {
    // prefill: weight row pairs vary fastest, so the clusters running at
    // once share one token tile (read from HBM once, then from L2)
    const int m_pairs = (G.m_tiles + 1) / 2;
    t.mpair = u % m_pairs;
    t.nt = u / m_pairs;
  }
  t.rows = min(p.bn, G.rows - t.nt * p.bn);
  t.n_mma = (t.rows + 31) & ~31;    // even halves of 16-row multiples
  return t;
}

// The unit a pair takes in round r: rounds of ncl consecutive units.  The
// narrow ring hands a round to the pairs in ascending order in even rounds
// and descending order in odd ones (snake), so with the heaviest units (the
// shared expert's) first in the table the partial last round falls on the
// pairs that drew the lighter ones: 26-layer decode 6.46 -> 6.40 ms.  On the
// wide ring the snake measured slower (prefill 1.479 -> 1.492 ms) and a
// round goes to the pairs in ascending order.
template <bool kNarrow>
__device__ __forceinline__ int round_unit(int r, int cid, int ncl) {
  return r * ncl + ((kNarrow && (r & 1)) ? ncl - 1 - cid : cid);
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         uint64_t deadline, int32_t* status) {
  uint32_t spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++spins & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() > deadline) {
        *abort_flag = 1;
        set_error(status, AFD_ERR_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Wait (acquire, bounded by the kernel's deadline) until a token tile's
// SwiGLU units have all stored their h rows; then order the async proxy (the
// TMA loads that follow) after those generic-proxy stores.
__device__ __forceinline__ bool wait_dep(const int32_t* cnt, int target, volatile int* abort_flag,
                                         uint64_t deadline, int32_t* status) {
  uint32_t spins = 0;
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
    if (v >= target) break;
    if ((++spins & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() > deadline) {
        *abort_flag = 1;
        set_error(status, AFD_ERR_TIMEOUT);
        return false;
      }
    }
    __nanosleep(32);
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

template <bool kNarrow>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
k_gemm_tc2(const __grid_constant__ GemmPair pargs) {
  using R = Ring<kNarrow>;
  constexpr int STAGES = R::STAGES;
  constexpr int STAGE_BYTES = R::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  typename R::Tail* tail = reinterpret_cast<typename R::Tail*>(smem + (size_t)STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int cid = (int)cluster_id_x();
  const int ncl = (int)num_clusters_x();
  const int nproj = pargs.nproj;
  const GemmArgs& args = pargs.p[0];  // status, bn, timeout and layer selection are shared

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; s++) {
      mbar_init(smem_u32(&tail->full[s]), 1);
      mbar_init(smem_u32(&tail->empty[s]), 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(smem_u32(&tail->tfull[b]), 1);
      mbar_init(smem_u32(&tail->tempty[b]), 2 * EPI_WARPS);
    }
    mbar_init(smem_u32(&tail->drain), 1);
    tail->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // TMEM before the dependency wait: a GEMM CTA of an earlier launch never
  // shares this SM (each takes over half its shared memory), so the columns
  // are free; everything up to the wait touches only this CTA's resources
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tail->tmem_base)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  // "this CTA has started": its peer may store into its shared memory once
  // the matching wait below returns (usually at once: both arrived before
  // their dependency waits)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  grid_dep_wait();
  grid_dep_launch();
  // both projections' group tables: the units of p[0], then those of p[1]
  __shared__ int unit0_s[2][AFD_MAX_GROUPS];
  int ngroups[2] = {0, 0}, units[2] = {0, 0};
  for (int ph = 0; ph < nproj; ph++) {
    const GemmPlan& P = *pargs.p[ph].plan;
    ngroups[ph] = min(P.ngroups, AFD_MAX_GROUPS);
    units[ph] = P.total_units;
    for (int i = threadIdx.x; i < ngroups[ph]; i += blockDim.x) unit0_s[ph][i] = P.g[i].unit0;
  }
  if (threadIdx.x == 0) {
    int skip = read_status(args.status);
    for (int ph = 0; ph < nproj; ph++)
      if (kNarrow && pargs.p[ph].plan->bn > 2 * R::BN_HALF && !skip) {  // no room for wider tiles
        set_error(args.status, AFD_ERR_ARG);
        skip = 1;
      }
    tail->skip = skip;
  }
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // the peer has started
  if (threadIdx.x == 0) {
    // the decision goes into the peer's shared memory too, so after the
    // barrier each CTA reads only its own and may leave at once
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(map_to_rank(smem_u32(&tail->peer_skip), rank ^ 1u)),
                 "r"(tail->skip)
                 : "memory");
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers, skip decisions and TMEM columns are in place
  tc_fence_after();
  const int total = units[0] + units[1];
  if (tail->skip || tail->peer_skip || total <= cid) {  // the same decision in both CTAs
    if (warp == 1) {
      __syncwarp();
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tail->tmem_base),
                   "r"(TMEM_COLS));
    }
    return;
  }

  // weight maps per projection: the launch's own, or the device table's
  // entry for the layer the device chose for this step (host-written before
  // any launch)
  const CUtensorMap* tmA_of[2] = {pargs.p[0].tmA, pargs.p[1].tmA};
  for (int ph = 0; ph < nproj; ph++)
    if (pargs.p[ph].layers) {
      const DevLayer& Ld = pargs.p[ph].layers[pargs.p[ph].item->layer];
      tmA_of[ph] = pargs.p[ph].wsel == 1 ? Ld.tmA1 : Ld.tmA2;
    }
  // unit -> (projection, its unit index)
  auto split_unit = [&](int unit, int& ph) { ph = unit >= units[0]; return ph ? unit - units[0] : unit; };
  const uint32_t tmem_base = tail->tmem_base;
  const uint64_t deadline = globaltimer_ns() + kGemmTimeoutNs;
  volatile int* abort_flag = &tail->abort_flag;
  const uint32_t smem_base = smem_u32(smem);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------ TMA producer (both CTAs)
      int s = 0;
      uint32_t sph = 0;
      for (int r = 0;; r++) {
        const int unit = round_unit<kNarrow>(r, cid, ncl);
        if (unit >= total) break;
        int ph;
        const int pu = split_unit(unit, ph);
        const GemmArgs& A = pargs.p[ph];
        const GemmPlan& plan = *A.plan;
        const Unit t = decode_unit<kNarrow>(plan, unit0_s[ph], ngroups[ph], pu);
        const GemmGroup& G = plan.g[t.group];
        const int nkb = (A.K[t.kind] + BK - 1) / BK;
        // a down unit's token rows: the h rows its token tile's SwiGLU
        // units store (every epilogue warp of each of those pairs counts)
        const int32_t* dep = ph == 1 ? pargs.dep + G.nt0 + t.nt : nullptr;
        const int dep_target = ph == 1 ? ((pargs.p[0].plan->g[t.group].m_tiles + 1) / 2) * 2 * EPI_WARPS : 0;
        // one token box per CTA and k-block: 128 rows, or 32 rows when the
        // unit's half fits (decode-sized groups); rows past the half are read
        // but not used by the MMA, past the buffer they are zero-filled
        const int half = t.n_mma / 2;
        const int brow = G.b_row0 + t.nt * plan.bn + (int)rank * half;
        const bool small_box = kNarrow || half <= SMALL_BOX_ROWS;
        const uint32_t b_bytes = small_box ? SMALL_BOX_BYTES : R::B_BYTES;
        const int mt = 2 * t.mpair + (int)rank;
        const CUtensorMap* ta = tmA_of[ph] + t.kind;
        const CUtensorMap* tb = small_box ? &A.tmBs[t.kind] : &A.tmB[t.kind];
        bool ok = true;
        bool dep_ok = dep == nullptr;
        if (dep) {  // usually long done: check once before the weight loads
          int v;
          asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(dep) : "memory");
          dep_ok = v >= dep_target;
          if (dep_ok) asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        for (int kb = 0; kb < nkb; kb += R::KPS) {
          const int cnt = min(R::KPS, nkb - kb);
          if (!wait_bar(smem_u32(&tail->empty[s]), sph ^ 1, abort_flag, deadline, args.status)) { ok = false; break; }
          const uint32_t full_leader = map_to_rank(smem_u32(&tail->full[s]), 0);
          if (rank == 0) mbar_expect_tx(smem_u32(&tail->full[s]), 2 * cnt * (A_BYTES + b_bytes));
          const uint32_t sa = smem_base + s * STAGE_BYTES;
          const uint32_t sb = sa + R::KPS * A_BYTES;
          // weights: the tiled copy's 16 KB blocks (k-block, 128-row tile, expert);
          // they need nothing from the SwiGLU units, so they go first
          for (int j = 0; j < cnt; j++) tma2_load_5d(sa + j * A_BYTES, ta, 0, 0, kb + j, mt, G.a_idx, full_leader);
          if (!dep_ok) {
            if (!wait_dep(dep, dep_target, abort_flag, deadline, args.status)) { ok = false; break; }
            dep_ok = true;
          }
          for (int j = 0; j < cnt; j++) tma2_load_2d(sb + j * R::B_BYTES, tb, (kb + j) * BK, brow, full_leader);
          if (++s == STAGES) { s = 0; sph ^= 1; }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------ MMA issuer (leader CTA)
      int s = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      for (int r = 0; ok; r++) {
        const int unit = round_unit<kNarrow>(r, cid, ncl);
        if (unit >= total) break;
        int uph;
        const int pu = split_unit(unit, uph);
        const Unit t = decode_unit<kNarrow>(*pargs.p[uph].plan, unit0_s[uph], ngroups[uph], pu);
        const int nkb = (pargs.p[uph].K[t.kind] + BK - 1) / BK;
        const uint32_t idesc = idesc_pair(t.n_mma);
        if (!wait_bar(smem_u32(&tail->tempty[acc]), acc_ph ^ 1, abort_flag, deadline, args.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * 256);
        for (int kb = 0; kb < nkb; kb += R::KPS) {
          const int cnt = min(R::KPS, nkb - kb);
          if (!wait_bar(smem_u32(&tail->full[s]), ph, abort_flag, deadline, args.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_base + s * STAGE_BYTES;
          for (int j = 0; j < cnt; j++) {
            const uint64_t adesc = sdesc_sw128(sa + j * A_BYTES);
            const uint64_t bdesc = sdesc_sw128(sa + R::KPS * A_BYTES + j * R::B_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; kk++)
              tc2_mma_f16(d_tmem, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk), idesc,
                          ((kb + j) | kk) != 0);
          }
          tc2_commit_pair(smem_u32(&tail->empty[s]));
          if (++s == STAGES) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        tc2_commit_pair(smem_u32(&tail->tfull[acc]));
        if (++acc == 2) { acc = 0; acc_ph ^= 1; }
      }
      // every issued MMA completes before TMEM is released
      tc2_commit_local(smem_u32(&tail->drain));
      const uint64_t dl = globaltimer_ns() + 100000000ull;
      while (!mbar_try_wait(smem_u32(&tail->drain), 0) && globaltimer_ns() < dl) {}
    }
  } else {
    // ------------------------------ epilogue (warps 2..9, both CTAs)
    const int q = warp & 3;
    const int half_cols = (warp - 2) >> 2;
    uint8_t* ebuf = smem + R::kEpiOffset + (size_t)(warp - 2) * EPI_BUF_BYTES;
    const bool lo = lane < 16;
    const uint32_t tempty_leader[2] = {map_to_rank(smem_u32(&tail->tempty[0]), 0),
                                       map_to_rank(smem_u32(&tail->tempty[1]), 0)};
    int acc = 0;
    uint32_t acc_ph = 0;
    for (int r = 0;; r++) {
      const int unit = round_unit<kNarrow>(r, cid, ncl);
      if (unit >= total) break;
      int uph;
      const int pu = split_unit(unit, uph);
      const GemmArgs& A = pargs.p[uph];
      const GemmPlan& plan = *A.plan;
      const Unit t = decode_unit<kNarrow>(plan, unit0_s[uph], ngroups[uph], pu);
      const GemmGroup& G = plan.g[t.group];
      bool ok = wait_bar(smem_u32(&tail->tfull[acc]), acc_ph, abort_flag, deadline, args.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * 256);
      const int kind = t.kind;
      const int64_t ldo = A.ldo[kind];
      const int64_t row0 = (int64_t)G.out_row0 + (int64_t)t.nt * plan.bn;
      const int mt = 2 * t.mpair + (int)rank;
      const bool rows_ok = dbg_in_range(A.dbg, args.status, AFD_DBG_GEMM_OUT, row0 + t.rows - 1,
                                        A.out_rows[kind]);
      if (A.swiglu) {
        const int col0 = mt * 64 + q * 16;
        const bool cols_ok = col0 + 16 <= A.M[kind] / 2 && rows_ok;
        for (int c0 = half_cols * 32; c0 < t.rows; c0 += 64) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(taddr + (uint32_t)c0, v);
          tmem_ld_wait();
          uint16_t* sb = reinterpret_cast<uint16_t*>(ebuf);
#pragma unroll
          for (int j = 0; j < 16; j++) {
            const float a = __uint_as_float(v[j]), b = __uint_as_float(v[16 + j]);
            const float recv = __shfl_xor_sync(0xffffffffu, lo ? b : a, 16);
            const float g = lo ? a : recv;
            const float u = lo ? recv : b;
            const __nv_bfloat16 hv = __float2bfloat16_rn(silu_f(g) * u);
            const int tok = lo ? j : 16 + j;
            sb[(tok * EPI_PITCH_SWIGLU + (lo ? 0 : 32)) / 2 + (lane & 15)] =
                *reinterpret_cast<const uint16_t*>(&hv);
          }
          __syncwarp();
          const int r = c0 + lane;
          if (r < t.rows && cols_ok) {
            const uint4* src =
                reinterpret_cast<const uint4*>(ebuf + lane * EPI_PITCH_SWIGLU + (lo ? 0 : 32));
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(A.out[kind]) +
                                                  (row0 + r) * ldo + col0);
            dst[0] = src[0];
            dst[1] = src[1];
          }
          __syncwarp();
        }
      } else {
        const int col0 = mt * BM + q * 32;
        const bool cols_ok = col0 + 32 <= A.M[kind] && rows_ok;
        const int fmt = A.out_fmt[kind];
        for (int c0 = half_cols * 32; c0 < t.rows; c0 += 64) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(taddr + (uint32_t)c0, v);
          tmem_ld_wait();
          const int r = c0 + lane;
          if (fmt == OUT_F32) {
            if (cols_ok) {
              float* dst = reinterpret_cast<float*>(A.out[kind]) + (row0 + c0) * ldo + col0 + lane;
#pragma unroll
              for (int c = 0; c < 32; c++)
                if (c0 + c < t.rows) dst[(int64_t)c * ldo] = __uint_as_float(v[c]);
            }
          } else if (fmt == OUT_Y24) {
            // lane = feature: each token row gets 64 contiguous bytes of the
            // high plane and 32 of the low plane per store pair (through
            // shared memory into 16-byte stores measured 9 % slower over
            // the down GEMM: its epilogue competes with the operand traffic)
            if (cols_ok) {
              uint16_t* dh = reinterpret_cast<uint16_t*>(A.out[kind]) + (row0 + c0) * ldo + col0 + lane;
              uint8_t* dl = A.out_lo[kind] + (row0 + c0) * ldo + col0 + lane;
#pragma unroll
              for (int c = 0; c < 32; c++)
                if (c0 + c < t.rows) {
                  const uint32_t b24 = y24_encode(__uint_as_float(v[c]));
                  dh[(int64_t)c * ldo] = (uint16_t)(b24 >> 8);
                  dl[(int64_t)c * ldo] = (uint8_t)(b24 & 0xffu);
                }
            }
          } else {
#pragma unroll
            for (int c = 0; c < 32; c++) {
              const __nv_bfloat16 yv = __float2bfloat16_rn(__uint_as_float(v[c]));
              *reinterpret_cast<uint16_t*>(ebuf + c * EPI_PITCH_BF16 + lane * 2) =
                  *reinterpret_cast<const uint16_t*>(&yv);
            }
            __syncwarp();
            if (r < t.rows && cols_ok) {
              const uint4* src = reinterpret_cast<const uint4*>(ebuf + lane * EPI_PITCH_BF16);
              uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(A.out[kind]) +
                                                    (row0 + r) * ldo + col0);
#pragma unroll
              for (int x = 0; x < 4; x++) dst[x] = src[x];
            }
          }
          __syncwarp();
        }
      }
      if (uph == 0 && pargs.dep) {  // this warp's h rows of the tile are stored (release)
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(pargs.dep + G.nt0 + t.nt, 1);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader[acc]);
      if (++acc == 2) { acc = 0; acc_ph ^= 1; }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote arrive or MMA of the pair is outstanding past this point
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
  }
}

// Cluster slots the GPU holds at once for this kernel (cached): the pair
// launch waits across clusters, so every cluster must be resident together.
template <bool kNarrow>
int max_pairs(int num_sms) {
  static std::atomic<int> cached_dev[kMaxCachedDevices];
  const int d = current_device();
  if (d >= 0) {
    const int c = cached_dev[d].load(std::memory_order_relaxed);
    if (c) return c;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((num_sms / 2) * 2));
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = Ring<kNarrow>::kSmemBytes;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_gemm_tc2<kNarrow>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = 0;
  }
  const int c = n > 0 ? n : -1;
  if (d >= 0) cached_dev[d].store(c, std::memory_order_relaxed);
  return c;
}

template <bool kNarrow>
cudaError_t launch_variant(const LaunchCtx& lc, const GemmPair& a) {
  constexpr size_t smem = Ring<kNarrow>::kSmemBytes;
  static std::atomic<int> attr_done[kMaxCachedDevices];
  const cudaError_t e = smem_attr_once(k_gemm_tc2<kNarrow>, (int)smem, attr_done);
  if (e != cudaSuccess) return e;
  int pairs = lc.num_sms / 2;  // persistent over the unit table
  if (a.nproj == 2) {
    const int m = max_pairs<kNarrow>(lc.num_sms);
    if (m < 1) {  // residency unknown: the two projections as two launches
      GemmPair one;
      memset(&one, 0, sizeof one);
      one.nproj = 1;
      for (int ph = 0; ph < 2; ph++) {
        one.p[0] = a.p[ph];
        const cudaError_t e = launch_k(lc, k_gemm_tc2<kNarrow>, 2 * pairs, NUM_THREADS, smem, one);
        if (e != cudaSuccess) return e;
      }
      return cudaSuccess;
    }
    pairs = std::min(pairs, m);
  }
  return launch_k(lc, k_gemm_tc2<kNarrow>, 2 * pairs, NUM_THREADS, smem, a);
}

}  // namespace

cudaError_t launch_gemm_tc2(const LaunchCtx& lc, const GemmArgs& a) {
  GemmPair p;
  memset(&p, 0, sizeof p);
  p.p[0] = a;
  p.nproj = 1;
  return a.bn <= 2 * Ring<true>::BN_HALF ? launch_variant<true>(lc, p) : launch_variant<false>(lc, p);
}

cudaError_t launch_gemm_tc2_pair(const LaunchCtx& lc, const GemmArgs& a1, const GemmArgs& a2, int32_t* dep) {
  GemmPair p;
  memset(&p, 0, sizeof p);
  p.p[0] = a1;
  p.p[1] = a2;
  p.dep = dep;
  p.nproj = 2;
  return a1.bn <= 2 * Ring<true>::BN_HALF ? launch_variant<true>(lc, p) : launch_variant<false>(lc, p);
}
