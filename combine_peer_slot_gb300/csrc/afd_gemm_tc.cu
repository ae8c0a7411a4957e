// afd_gemm_tc.cu -- grouped expert GEMM on the sm_103a tensor cores
// (tcgen05.mma kind::f16, bf16 in, fp32 accumulate in TMEM), fed by TMA.
//
// Orientation: the weights are the M side (128 rows per tile) and the tokens
// the N side (up to 256 per tile, any multiple of 16), D[m][n] = W[m] . X[n].
// Ragged per-expert token counts then only round N up to 16, and the
// decode-sized groups (a few dozen tokens) stream each weight tile once.
//
// Projections (Async GPU Connector, "Attention gate and FFN expert compute":
// fused_experts = gate/up GEMM, SiLU-and-multiply, down GEMM; Async AFD for
// Prefill on Ascend NPU, "Architecture": W1 with SwiGLU, then W2):
// The weights are read from the library's tiled copies: every 128-row x
// 64-column TMA box is one contiguous 16 KB block, addressed by a 5-D map as
// (0, 0, k-block, 128-row tile, expert).
//  - SwiGLU mode: a tile of W13[e] = [gate rows | up rows] holds 16 gate rows
//    then the 16 matching up rows, four times: 128 rows covering 64
//    intermediate columns.  In TMEM, warp quadrant q holds gate rows in
//    lanes 0-15 and the matching up rows in lanes 16-31; a shuffle pairs
//    them and h = silu(g) * u is written as bf16.
//  - plain mode: y = h . Wd^T with Wd[e] = [hidden, inter], tiles of 128
//    hidden rows in order.
//
// Warp roles (320 threads, one CTA per SM, persistent over the tile table
// built on the device from the expert counts):
//   warp 0  TMA producer (one lane), STAGES-deep smem ring
//   warp 1  TMEM allocator and MMA issuer (one lane)
//   warps 2-9 epilogue: TMEM -> registers -> smem transpose -> 16-byte
//           global stores (lane quadrant = warp % 4, two warps per quadrant
//           take alternate 32-column chunks)
// Two TMEM accumulators (2 x 256 columns) let the epilogue of one tile run
// under the main loop of the next.  Every mbarrier wait is bounded.
#include "afd_internal.cuh"

namespace {

constexpr int BM = 128;
constexpr int BK = 64;             // one 128-byte swizzle atom of bf16
constexpr int BN = 256;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BOX_ROWS = 32;
constexpr int B_BOX_BYTES = B_BOX_ROWS * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;        // two per TMEM lane quadrant
constexpr int NUM_THREADS = 64 + EPI_WARPS * 32;
constexpr int TMEM_COLS = 512;
// per epilogue warp: a 32-token transpose buffer for bf16 outputs, rows
// padded so neither the column writes nor the row reads conflict on banks.
// SwiGLU rows hold 16 values (32 B) at a 48-byte pitch, rows 16-31 shifted by
// 32 B; down-projection rows hold 32 values (64 B) at an 80-byte pitch.
constexpr int EPI_PITCH_SWIGLU = 48;
constexpr int EPI_PITCH_BF16 = 80;
constexpr int EPI_BUF_BYTES = 32 * EPI_PITCH_BF16;
constexpr uint64_t kGemmTimeoutNs = 5000000000ull;

struct SmemTail {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int skip;
};

// layout after the 1024-aligned base: stages | barriers (SmemTail) | epilogue
// buffers at a 128-byte boundary (16-byte vector loads read them)
constexpr size_t kEpiOffset = ((size_t)STAGES * STAGE_BYTES + sizeof(SmemTail) + 127) / 128 * 128;
constexpr size_t kSmemBytes = 1024 + kEpiOffset + (size_t)EPI_WARPS * EPI_BUF_BYTES;
static_assert(kEpiOffset % 128 == 0 && EPI_BUF_BYTES % 128 == 0, "epilogue buffers must stay aligned");
static_assert(kSmemBytes <= 232448, "over the per-CTA shared memory limit");

// shared-memory matrix descriptor: K-major, 128-byte swizzle, rows of 128 B,
// 8-row core groups 1024 B apart (SBO), descriptor version 1
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major,
// N >> 3 at bit 17, M >> 4 at bit 24
__device__ __forceinline__ uint32_t idesc_bf16(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(BM >> 4) << 24);
}

struct Tile {
  int group, kind, mt, nt, rows;   // rows: valid tokens in this tile
};

__device__ __forceinline__ Tile decode_tile(const GemmPlan& p, int tile) {
  int lo = 0, hi = p.ngroups - 1;
  while (lo < hi) {  // last group with tile0 <= tile
    const int mid = (lo + hi + 1) >> 1;
    if (p.g[mid].tile0 <= tile) lo = mid; else hi = mid - 1;
  }
  // skip empty groups sharing the same tile0
  while (lo + 1 < p.ngroups && p.g[lo].m_tiles * p.g[lo].n_tiles == 0) lo++;
  const GemmGroup& G = p.g[lo];
  const int u = tile - G.tile0;
  Tile t;
  t.group = lo;
  t.kind = G.kind;
  t.mt = u % G.m_tiles;
  t.nt = u / G.m_tiles;
  t.rows = min(p.bn, G.rows - t.nt * p.bn);
  return t;
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         uint64_t deadline, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() > deadline) {
        *abort_flag = 1;
        set_error(status, AFD_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// silu(g) = g / (1 + e^-g); the fast divide returns 0 once the denominator
// passes 2^126, which is silu's limit there
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__global__ void __launch_bounds__(NUM_THREADS, 1) k_gemm_tc(const __grid_constant__ GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  SmemTail* tail = reinterpret_cast<SmemTail*>(smem + (size_t)STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const GemmPlan& plan = *args.plan;  // tile table, built by the plan kernel
  grid_dep_wait();
  grid_dep_launch();
  if (threadIdx.x == 0) tail->skip = read_status(args.status);
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; s++) {
      mbar_init(smem_u32(&tail->full[s]), 1);
      mbar_init(smem_u32(&tail->empty[s]), 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(smem_u32(&tail->tfull[b]), 1);
      mbar_init(smem_u32(&tail->tempty[b]), EPI_WARPS);
    }
    mbar_init(smem_u32(&tail->drain), 1);
    tail->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (tail->skip || plan.total_tiles <= (int)blockIdx.x) return;  // uniform for the CTA

  // weight maps: the kernel's own, or the device table's entry for the layer
  // the device chose for this step (host-written before any launch)
  const CUtensorMap* tmA = args.tmA;
  if (args.layers) {
    const DevLayer& Ld = args.layers[args.item->layer];
    tmA = args.wsel == 1 ? Ld.tmA1 : Ld.tmA2;
  }

  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tail->tmem_base)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;
  const int total = plan.total_tiles;
  const uint64_t deadline = globaltimer_ns() + kGemmTimeoutNs;
  volatile int* abort_flag = &tail->abort_flag;
  const uint32_t smem_base = smem_u32(smem);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------ TMA producer
      int s = 0;
      uint32_t ph = 0;
      uint32_t pending = 0;  // stages with a fill issued (for the abort drain)
      uint32_t pend_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const Tile t = decode_tile(plan, tile);
        const GemmGroup& G = plan.g[t.group];
        const int nkb = (args.K[t.kind] + BK - 1) / BK;
        const int nb = (t.rows + B_BOX_ROWS - 1) / B_BOX_ROWS;
        const int brow = G.b_row0 + t.nt * plan.bn;
        const CUtensorMap* ta = tmA + t.kind;
        const CUtensorMap* tb = &args.tmB[t.kind];
        for (int kb = 0; kb < nkb; kb++) {
          if (!wait_bar(smem_u32(&tail->empty[s]), ph ^ 1, abort_flag, deadline, args.status)) { ok = false; break; }
          const uint32_t full = smem_u32(&tail->full[s]);
          const uint32_t sa = smem_base + s * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          mbar_expect_tx(full, A_BYTES + nb * B_BOX_BYTES);
          // weights: the tiled copy's 16 KB block (k-block, 128-row tile, expert)
          tma_load_5d(sa, ta, 0, 0, kb, t.mt, G.a_idx, full);
          for (int q = 0; q < nb; q++)
            tma_load_2d(sb + q * B_BOX_BYTES, tb, kb * BK, brow + q * B_BOX_ROWS, full);
          pending |= 1u << s;
          pend_par = (pend_par & ~(1u << s)) | (ph << s);
          if (++s == STAGES) { s = 0; ph ^= 1; }
        }
      }
      if (!ok) {
        // let every issued copy land before the CTA's shared memory goes away
        const uint64_t dl = globaltimer_ns() + 100000000ull;
        for (int q = 0; q < STAGES; q++)
          if (pending & (1u << q))
            while (!mbar_try_wait(smem_u32(&tail->full[q]), (pend_par >> q) & 1u) && globaltimer_ns() < dl) {}
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------ MMA issuer
      int s = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const Tile t = decode_tile(plan, tile);
        const int nkb = (args.K[t.kind] + BK - 1) / BK;
        const int n_mma = (t.rows + 15) & ~15;
        const uint32_t idesc = idesc_bf16(n_mma);
        if (!wait_bar(smem_u32(&tail->tempty[acc]), acc_ph ^ 1, abort_flag, deadline, args.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < nkb; kb++) {
          if (!wait_bar(smem_u32(&tail->full[s]), ph, abort_flag, deadline, args.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_base + s * STAGE_BYTES;
          const uint64_t adesc = sdesc_sw128(sa);
          const uint64_t bdesc = sdesc_sw128(sa + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; kk++)
            tc_mma_f16(d_tmem, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk), idesc,
                       (kb | kk) != 0);
          tc_commit(smem_u32(&tail->empty[s]));
          if (++s == STAGES) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        tc_commit(smem_u32(&tail->tfull[acc]));
        if (++acc == 2) { acc = 0; acc_ph ^= 1; }
      }
      // all issued MMAs complete before TMEM is released
      tc_commit(smem_u32(&tail->drain));
      const uint64_t dl = globaltimer_ns() + 100000000ull;
      while (!mbar_try_wait(smem_u32(&tail->drain), 0) && globaltimer_ns() < dl) {}
    }
  } else {
    // ------------------------------ epilogue (warps 2..9)
    // warp -> TMEM lane quadrant q = warp % 4 and column half (even or odd
    // 32-column chunks).  Each chunk goes TMEM -> registers -> a per-warp
    // smem transpose -> one token row per lane -> 16-byte global stores.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* ebuf = smem + kEpiOffset + (size_t)(warp - 2) * EPI_BUF_BYTES;
    const bool lo = lane < 16;
    int acc = 0;
    uint32_t acc_ph = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = decode_tile(plan, tile);
      const GemmGroup& G = plan.g[t.group];
      bool ok = wait_bar(smem_u32(&tail->tfull[acc]), acc_ph, abort_flag, deadline, args.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      const int kind = t.kind;
      const int64_t ldo = args.ldo[kind];
      const int64_t row0 = (int64_t)G.out_row0 + (int64_t)t.nt * plan.bn;
      const bool rows_ok = dbg_in_range(args.dbg, args.status, AFD_DBG_GEMM_OUT, row0 + t.rows - 1,
                                        args.out_rows[kind]);
      if (args.swiglu) {
        // lanes 0-15 hold gate rows i = base + lane, lanes 16-31 the up rows
        // of the same i; lane < 16 produces tokens 0-15 of the chunk, lane
        // >= 16 tokens 16-31, after one exchange of 16 values
        const int col0 = t.mt * 64 + q * 16;
        const bool cols_ok = col0 + 16 <= args.M[kind] / 2 && rows_ok;
        for (int c0 = half * 32; c0 < t.rows; c0 += 64) {
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
            const int tok = lo ? j : 16 + j;   // row of the transpose buffer
            sb[(tok * EPI_PITCH_SWIGLU + (lo ? 0 : 32)) / 2 + (lane & 15)] =
                *reinterpret_cast<const uint16_t*>(&hv);
          }
          __syncwarp();
          const int r = c0 + lane;
          if (r < t.rows && cols_ok) {
            const uint4* src =
                reinterpret_cast<const uint4*>(ebuf + lane * EPI_PITCH_SWIGLU + (lo ? 0 : 32));
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(args.out[kind]) +
                                                  (row0 + r) * ldo + col0);
            dst[0] = src[0];
            dst[1] = src[1];
          }
          __syncwarp();
        }
      } else {
        const int col0 = t.mt * BM + q * 32;
        const bool cols_ok = col0 + 32 <= args.M[kind] && rows_ok;
        const int fmt = args.out_fmt[kind];
        for (int c0 = half * 32; c0 < t.rows; c0 += 64) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(taddr + (uint32_t)c0, v);
          tmem_ld_wait();
          const int r = c0 + lane;
          if (fmt == OUT_F32) {
            // lane = feature: each store is 32 consecutive fp32 of one token row
            if (cols_ok) {
              float* dst = reinterpret_cast<float*>(args.out[kind]) + (row0 + c0) * ldo + col0 + lane;
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
              uint16_t* dh = reinterpret_cast<uint16_t*>(args.out[kind]) + (row0 + c0) * ldo + col0 + lane;
              uint8_t* dl = args.out_lo[kind] + (row0 + c0) * ldo + col0 + lane;
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
              uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(args.out[kind]) +
                                                    (row0 + r) * ldo + col0);
#pragma unroll
              for (int x = 0; x < 4; x++) dst[x] = src[x];
            }
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tail->tempty[acc]));
      if (++acc == 2) { acc = 0; acc_ph ^= 1; }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
  }
}

}  // namespace

cudaError_t launch_gemm_tc(const LaunchCtx& lc, const GemmArgs& a) {
  static std::atomic<int> attr_done[kMaxCachedDevices];
  const cudaError_t e = smem_attr_once(k_gemm_tc, (int)kSmemBytes, attr_done);
  if (e != cudaSuccess) return e;
  return launch_k(lc, k_gemm_tc, lc.num_sms, NUM_THREADS, kSmemBytes, a);
}

size_t gemm_tc_smem_bytes() { return kSmemBytes; }
