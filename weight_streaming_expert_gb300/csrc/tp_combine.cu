// tp_combine.cu -- the exchange step of a tensor-parallel split of the
// layer: G fp32 partial outputs summed in a fixed order, one bf16 rounding.
//
// Method (page "How Ling-3.0-flash reduces batch 1 decoding latency by 54%
// on 4 Blackwell GPUs", section "PDL: the latency floor of stacked small
// kernels"): the MoE chain ends in an all-reduce of the partial outputs of
// the GPUs that each hold a slice of every expert, and the combine is an
// fp32 sum with a single final cast.  Here each slice's layer call leaves
// its combine unrounded (MOE_FWD_OUT_F32); the parts, gathered side by side,
// are summed in part order and rounded once, so the split layer rounds the
// output exactly as often as the unsplit one.  The order is fixed, so every
// GPU that runs this on the same gathered parts gets the same bits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.cuh"
#include "moe.h"

using namespace wse;

namespace {

constexpr int kThreads = 256;

// One thread per 4 consecutive elements: n_parts 16-byte loads, one 8-byte
// store.  The kernel is a few tens of KB of traffic per call (M x hidden x
// 4 bytes per part), so it is bound by its launch, not by HBM.
__global__ void __launch_bounds__(kThreads) combine_partials_kernel(const float4* __restrict__ parts, int n_parts,
                                                                    size_t n4, uint2* __restrict__ out) {
  const size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x;
  if (i >= n4) return;
  float4 s = __ldg(parts + i);
  for (int p = 1; p < n_parts; ++p) {
    const float4 v = __ldg(parts + (size_t)p * n4 + i);
    s.x += v.x;
    s.y += v.y;
    s.z += v.z;
    s.w += v.w;
  }
  const __nv_bfloat162 lo = __floats2bfloat162_rn(s.x, s.y), hi = __floats2bfloat162_rn(s.z, s.w);
  out[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

}  // namespace

extern "C" {

int moe_combine_partials(const float* parts, int n_parts, size_t n, void* out, moe_stream_t stream) {
  if (!parts || !out) {
    set_last_error_text("null parts/out");
    return MOE_ERR_INVALID_ARG;
  }
  if (n_parts < 1 || n % 4 != 0) {
    set_last_error_text("need n_parts >= 1 and n a multiple of 4");
    return MOE_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(parts) & 15u) || (reinterpret_cast<uintptr_t>(out) & 7u)) {
    set_last_error_text("parts must be 16-byte and out 8-byte aligned");
    return MOE_ERR_INVALID_ARG;
  }
  const char* o = static_cast<const char*>(out);
  const char* p = reinterpret_cast<const char*>(parts);
  if (o < p + (size_t)n_parts * n * 4 && p < o + n * 2) {
    set_last_error_text("out overlaps parts");
    return MOE_ERR_INVALID_ARG;
  }
  if (n == 0) return MOE_OK;
  const size_t n4 = n / 4;
  const unsigned blocks = (unsigned)((n4 + kThreads - 1) / kThreads);
  combine_partials_kernel<<<blocks, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const float4*>(parts), n_parts, n4, static_cast<uint2*>(out));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_error_text(cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // extern "C"
