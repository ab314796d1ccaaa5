// route_static.cu -- routing (router GEMV + softmax top-k) for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs while a CUDA graph is
// being captured by someone else, allocators that forbid outside
// allocations, or real-time paths that must not risk an allocation failure
// or an implicit device synchronisation.  moe_route_static serves them: it
// runs the layer's router kernel with its scratch memory (logits, the
// arrival counter, the published compaction) taken from one fixed array that
// is part of the library image, so the call itself allocates nothing.
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

using namespace wse;

namespace {

// Limits of the allocation-free path (the array is sized for them).
constexpr int kNoAllocMaxTokens = 16;
constexpr int kNoAllocMaxPairs = kNoAllocMaxTokens * kMaxTopk;
constexpr size_t kHeaderBytes = 256;  // status, counter, n_groups, n_active
constexpr size_t kLogitsBytes = (size_t)kNoAllocMaxTokens * kMaxExperts * 4;
constexpr size_t kPairBytes = (size_t)kNoAllocMaxPairs * 4;
constexpr size_t kNoAllocScratchBytes = kHeaderBytes + kLogitsBytes + 5 * kPairBytes;

static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

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

// Make sure the kernel may use `bytes` of dynamic shared memory; only ever
// raises the limit (a layer handle may have set its own).
int ensure_smem(RouterKernel k, size_t bytes) {
  if (bytes <= 48 * 1024) return MOE_OK;
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, k);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
  if ((size_t)fa.maxDynamicSharedSizeBytes >= bytes) return MOE_OK;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  return e == cudaSuccess ? MOE_OK : fail(MOE_ERR_CUDA, cudaGetErrorString(e));
}

}  // namespace

extern "C" {

int moe_route_static(int hidden, int n_experts, int topk, const void* x, const void* w_router,
                     const float* bias, int M, int32_t* topk_idx, float* topk_w,
                     moe_stream_t stream) {
  if (hidden <= 0 || hidden % 256 != 0 || !router_kernel_for(hidden / 256))
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
  const RouterKernel k = router_kernel_for(hidden / 256);
  const size_t smem = router_smem_bytes(M, hidden, topk, n_experts);
  void* base = nullptr;
  int rc = scratch_for_device(dev, &base);
  if (rc == MOE_OK) rc = ensure_smem(k, smem);
  if (rc != MOE_OK) return rc;

  uint8_t* b = static_cast<uint8_t*>(base);
  Workspace ws{};
  ws.status = reinterpret_cast<int*>(b);
  ws.router_count = reinterpret_cast<int*>(b) + 1;
  ws.n_groups = reinterpret_cast<int*>(b) + 2;
  ws.n_active = reinterpret_cast<int*>(b) + 3;
  ws.logits = reinterpret_cast<float*>(b + kHeaderBytes);
  uint8_t* pairs = b + kHeaderBytes + kLogitsBytes;
  ws.pair_w = reinterpret_cast<float*>(pairs);
  ws.grp_expert = reinterpret_cast<int*>(pairs + kPairBytes);
  ws.grp_start = reinterpret_cast<int*>(pairs + 2 * kPairBytes);
  ws.grp_cnt = reinterpret_cast<int*>(pairs + 3 * kPairBytes);
  ws.pair_list = reinterpret_cast<int*>(pairs + 4 * kPairBytes);

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the arrival counter (and the status word) must start at zero
  if ((e = cudaMemsetAsync(b, 0, 8, st)) != cudaSuccess) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));

  RouterArgs ra{};
  ra.x = static_cast<const __nv_bfloat16*>(x);
  ra.w_router = static_cast<const __nv_bfloat16*>(w_router);
  ra.bias = bias;
  ra.M = M;
  ra.H = hidden;
  ra.E = n_experts;
  ra.K = topk;
  ra.topk_idx = topk_idx;
  ra.topk_w = topk_w;
  ra.ws = ws;
  const dim3 grid((n_experts + kRouterExpertsPerCta - 1) / kRouterExpertsPerCta);
  k<<<grid, kRouterThreads, smem, st>>>(ra);
  if ((e = cudaGetLastError()) != cudaSuccess) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
  return MOE_OK;
}

}  // extern "C"
