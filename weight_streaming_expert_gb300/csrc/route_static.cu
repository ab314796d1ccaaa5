// route_static.cu -- routing (router matvec + softmax top-k) for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs while a CUDA graph is
// being captured by someone else, allocators that forbid outside
// allocations, or real-time paths that must not risk an allocation failure
// or an implicit device synchronisation.  moe_route_static serves them: its
// kernel takes its scratch memory (partial logits, the arrival counter, the
// status word) from one fixed array that is part of the library image, so
// the call itself allocates nothing.
//
// The arithmetic is the layer kernel's own (routing.cuh: same matvec units
// and split, same partial-sum order, same top-k), so the routing equals the
// layer's bit for bit; only the hand-off differs: the last unit to finish
// (a device-scope arrival counter, no spin) runs the top-k of every token,
// so no grid-wide residency is needed.
//
// The array is a file-scope __device__ object: every GPU that loads the
// library holds its kNoAllocScratchBytes until the process exits.  All calls
// on a device share it and it keeps the last call's contents, so two calls
// whose work overlaps on the GPU (different streams, no ordering between
// them) race and corrupt each other's results.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.cuh"
#include "moe.h"
#include "routing.cuh"

using namespace wse;

namespace {

// Limits of the allocation-free path (the array is sized for them).
constexpr int kNoAllocMaxTokens = 16;
constexpr size_t kHeaderBytes = 256;  // status word, arrival counter
// partial logits ks x 16 x E: a 152-SM GB300 runs at most 152 units of 8
// experts, ks x E <= 1216, so the layer kernel's split always fits there
constexpr size_t kPartBytes = (size_t)kNoAllocMaxTokens * 1216 * 4;
constexpr size_t kNoAllocScratchBytes = kHeaderBytes + kPartBytes;

static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

struct RouteArgs {
  const __nv_bfloat16* x;
  const __nv_bfloat16* w_router;
  const float* bias;
  int M, H, E, K, ks;
  int32_t* topk_idx;
  float* topk_w;
  int* status;
  unsigned* counter;
  float* part;  // [ks][16][E]
};

template <int KPW>
__global__ void __launch_bounds__(kConsumerWarps * 32) route_kernel(RouteArgs a) {
  __shared__ float4 red[kConsumerWarps * 32];
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const GemvUnit gu = gemv_unit(blockIdx.x, a.ks, a.H, warp);
  uint4 wb[KPW];
  gemv_load_w<KPW>(a.w_router, a.E, a.H, gu, lane, wb);
  const size_t plane = (size_t)kNoAllocMaxTokens * a.E;
  for (int mb = 0; mb * 16 < a.M; ++mb) {
    red[warp * 32 + lane] = gemv_tokens<KPW>(a.x, a.M, a.H, gu, mb, lane, wb);
    __syncthreads();
    if (warp == 0) gemv_store(red, gu, mb, a.M, a.E, plane, a.part, lane);
    __syncthreads();
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(a.counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int m = warp; m < a.M; m += kConsumerWarps) {
    // the lane holding each slot writes its expert id straight to the output
    const float w = topk_dispatch(PlainPlanes{a.part + (size_t)m * a.E, plane}, a.ks, a.bias, a.E, a.K, lane,
                                  a.status, a.topk_idx + m * a.K);
    if (lane < a.K && a.topk_w) a.topk_w[m * a.K + lane] = w;
  }
  if (threadIdx.x == 0) *a.counter = 0u;  // ready for the next call
}

using RouteKernel = void (*)(RouteArgs);
RouteKernel route_kernel_for(int kpw) {
  switch (kpw) {
    case 1: return route_kernel<1>;
    case 2: return route_kernel<2>;
    case 4: return route_kernel<4>;
    case 5: return route_kernel<5>;
    case 8: return route_kernel<8>;
    case 10: return route_kernel<10>;
    case 12: return route_kernel<12>;
    case 16: return route_kernel<16>;
    default: return nullptr;
  }
}

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

int fail(int code, const char* msg) {
  set_last_error_text(msg);  // read back with moe_last_error()
  return code;
}

// Device address of the array on the current device, resolved once per
// device (host code only ever sees a stand-in for the symbol itself).
int scratch_for_device(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device index out of range");
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess || !p) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_route_static(int hidden, int n_experts, int topk, const void* x, const void* w_router,
                     const float* bias, int M, int32_t* topk_idx, float* topk_w,
                     moe_stream_t stream) {
  if (hidden <= 0 || hidden % 256 != 0 || !route_kernel_for(hidden / 256))
    return fail(MOE_ERR_UNSUPPORTED, "hidden must be 256 * {1,2,4,5,8,10,12,16}");
  if (topk < 1 || topk > kMaxTopk) return fail(MOE_ERR_UNSUPPORTED, "topk must be in [1, 32]");
  if (n_experts < topk || n_experts > kMaxExperts)
    return fail(MOE_ERR_UNSUPPORTED, "n_experts must be in [topk, 1024]");
  if (M < 0) return fail(MOE_ERR_INVALID_ARG, "M < 0");
  if (M > kNoAllocMaxTokens)
    return fail(MOE_ERR_UNSUPPORTED, "M exceeds the 16 tokens the static scratch is sized for");
  if (M == 0) return MOE_OK;
  if (!x || !w_router || !topk_idx) return fail(MOE_ERR_INVALID_ARG, "null x/w_router/topk_idx");
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(w_router) & 15u))
    return fail(MOE_ERR_INVALID_ARG, "x and w_router must be 16-byte aligned");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
  int n_sms = 0;
  if ((e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
  void* base = nullptr;
  const int rc = scratch_for_device(dev, &base);
  if (rc != MOE_OK) return rc;

  // the layer kernel's split (same partial sums, so the same routing); a
  // split whose partial logits do not fit the array is refused rather than
  // changed (it would change the summation order)
  const int ks = gemv_split(hidden, n_experts, n_sms);
  if ((size_t)ks * kNoAllocMaxTokens * n_experts * 4 > kPartBytes)
    return fail(MOE_ERR_UNSUPPORTED, "this device's router split needs more partial logits than the static scratch holds");

  uint8_t* b = static_cast<uint8_t*>(base);
  RouteArgs ra{};
  ra.x = static_cast<const __nv_bfloat16*>(x);
  ra.w_router = static_cast<const __nv_bfloat16*>(w_router);
  ra.bias = bias;
  ra.M = M;
  ra.H = hidden;
  ra.E = n_experts;
  ra.K = topk;
  ra.ks = ks;
  ra.topk_idx = topk_idx;
  ra.topk_w = topk_w;
  ra.status = reinterpret_cast<int*>(b);
  ra.counter = reinterpret_cast<unsigned*>(b) + 1;
  ra.part = reinterpret_cast<float*>(b + kHeaderBytes);

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the arrival counter (and the status word) must start at zero
  if ((e = cudaMemsetAsync(b, 0, 8, st)) != cudaSuccess) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
  const dim3 grid(((n_experts + 7) / 8) * ks);
  route_kernel_for(hidden / 256)<<<grid, kConsumerWarps * 32, 0, st>>>(ra);
  if ((e = cudaGetLastError()) != cudaSuccess) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
  return MOE_OK;
}

int moe_route_static_read_status(int* status, moe_stream_t stream) {
  if (!status) return fail(MOE_ERR_INVALID_ARG, "null status");
  if (reinterpret_cast<uintptr_t>(status) & 3u) return fail(MOE_ERR_INVALID_ARG, "status must be 4-byte aligned");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
  void* base = nullptr;
  const int rc = scratch_for_device(dev, &base);
  if (rc != MOE_OK) return rc;
  // the status word is the array's first int (see moe_route_static)
  if ((e = cudaMemcpyAsync(status, base, sizeof(int), cudaMemcpyDefault,
                           reinterpret_cast<cudaStream_t>(stream))) != cudaSuccess)
    return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
  return MOE_OK;
}

}  // extern "C"
