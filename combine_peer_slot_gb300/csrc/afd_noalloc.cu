// afd_noalloc.cu -- the router step without any device allocation.
//
// Some callers cannot call cudaMalloc: a serving process whose memory pool
// has already reserved the device's free memory (a fresh cudaMalloc fails or
// fragments that pool), or a plugin that must not trigger the device-wide
// synchronisation cudaMalloc/cudaFree can cause.  afd_route_noalloc serves
// them: the caller passes inputs and outputs, and the only scratch the step
// needs -- the rearranged router weight, the router logits and a status
// word -- lives in the file-scope device array below, which every GPU that
// loads this library holds until the process exits.
//
// The array is shared by every call: a call rewrites the router weight
// and clears the status word before the router runs, and calls that overlap
// on the GPU (different streams, no ordering between them) race on it.
// Nothing polls the status word: when a bounded wait inside the router
// gives up, the top-k writes id -1 and a NaN weight for every token, so the
// failure shows in the caller's own outputs.
#include <cstdio>
#include <cstring>
#include <mutex>

#include "afd_internal.cuh"

namespace {

// [rearranged router weight: 4 * ceil(num_experts / 4) * hidden fp32]
// [logits: n_tokens * num_experts fp32][status word]; 256-byte aligned.
static __device__ __align__(256) float
    g_noalloc_scratch[AFD_NOALLOC_MAX_ROUTER_WEIGHTS + AFD_NOALLOC_MAX_LOGITS + 64];

constexpr int kMaxDevices = 64;
// per device: the array's device address, looked up once with that device
// current (two host threads making their first call on one device at once
// both wait for the one lookup)
struct ScratchAddr {
  std::once_flag once;
  float* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
ScratchAddr g_scratch[kMaxDevices];
int64_t g_noalloc_launches = 0;

// In host code the array's name is only a host-side stand-in: its device
// address must be asked for on each device.
int scratch_for_current_device(float** out, int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return AFD_ERR_CUDA;
  }
  ScratchAddr& a = g_scratch[dev];
  std::call_once(a.once, [&a] {
    void* p = nullptr;
    a.err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (a.err == cudaSuccess && !p) a.err = cudaErrorInvalidSymbol;
    if (a.err != cudaSuccess) {
      fprintf(stderr, "afd: cudaGetSymbolAddress failed: %s\n", cudaGetErrorString(a.err));
      cudaGetLastError();
    } else {
      a.ptr = static_cast<float*>(p);
    }
  });
  if (a.err != cudaSuccess) return AFD_ERR_CUDA;
  *out = a.ptr;
  *dev_out = dev;
  return AFD_OK;
}

}  // namespace

extern "C" int afd_route_noalloc(const void* x, int n_tokens, int hidden, int act_dtype,
                                 const float* Wg, const float* bias, int num_experts, int topk,
                                 int renorm, float routed_scaling, int32_t* ids, float* weights,
                                 void* cuda_stream) {
  if (n_tokens < 0 || hidden < 8 || hidden % 8 || num_experts < 1 || num_experts > 256 ||
      topk < 1 || topk > 16 || topk > num_experts ||
      (act_dtype != AFD_DTYPE_F32 && act_dtype != AFD_DTYPE_BF16))
    return AFD_ERR_ARG;
  if ((int64_t)hidden * 4 * wgq_groups(num_experts) > AFD_NOALLOC_MAX_ROUTER_WEIGHTS ||
      (int64_t)n_tokens * num_experts > AFD_NOALLOC_MAX_LOGITS)
    return AFD_ERR_CAPACITY;
  if (n_tokens == 0) return AFD_OK;
  if (!x || !Wg || !ids || !weights || (reinterpret_cast<uintptr_t>(x) & 15)) return AFD_ERR_ARG;
  float* scratch = nullptr;
  int dev = 0;
  int rc = scratch_for_current_device(&scratch, &dev);
  if (rc) return rc;
  float* WgQ = scratch;
  float* logits = scratch + AFD_NOALLOC_MAX_ROUTER_WEIGHTS;
  int32_t* status =
      reinterpret_cast<int32_t*>(scratch + AFD_NOALLOC_MAX_ROUTER_WEIGHTS + AFD_NOALLOC_MAX_LOGITS);
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(cuda_stream);
  LaunchCtx lc{stream, 0, &g_noalloc_launches};
  cudaDeviceGetAttribute(&lc.num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), stream) != cudaSuccess) {
    cudaGetLastError();
    return AFD_ERR_CUDA;
  }
  if (launch_arrange_wg(lc, Wg, WgQ, hidden, num_experts) != cudaSuccess) return AFD_ERR_CUDA;
  // the activations are one contiguous [n_tokens, hidden] block: a single
  // "peer" whose rows start at x
  FanIn f;
  memset(&f, 0, sizeof f);
  f.n_peers = 1;
  f.total = n_tokens;
  f.prefix[1] = n_tokens;
  WinGeom g;
  memset(&g, 0, sizeof g);
  g.ring_depth = 1;
  g.num_regions = 1;
  DevWS ws;
  memset(&ws, 0, sizeof ws);
  ws.status = status;
  ws.ids = ids;
  ws.w = weights;
  if (launch_router(lc, g, static_cast<const uint8_t*>(x), f, ws, hidden,
                    act_dtype == AFD_DTYPE_F32, WgQ, bias, num_experts, topk, renorm,
                    routed_scaling, logits, /*hist=*/nullptr) != cudaSuccess)
    return AFD_ERR_CUDA;
  return AFD_OK;
}
