// kernels.cuh -- argument blocks and launch-side declarations of the layer's
// three forward kernels and the create-time weight re-layout kernels.
#pragma once

#include "common.cuh"

namespace wse {

struct RouterArgs {
  const __nv_bfloat16* x;         // [M][H]
  const __nv_bfloat16* w_router;  // [E][H]
  const float* bias;              // [E] or nullptr
  int M, H, E, K;
  int32_t* topk_idx;              // [M][K] caller output
  float* topk_w;                  // [M][K] caller output or nullptr
  Workspace ws;
};

struct GateUpArgs {
  const uint8_t* w_gate_up;  // packed gate/up tiles, see pack.cu
  const __nv_bfloat16* x;    // [M][H]
  const int32_t* topk_idx;   // [M][K] the router's expert ids
  int M, H, I, K, E;
  int stages;                // ring depth
  uint32_t tile_bytes;       // 8 rows x H x 2
  Workspace ws;
};

struct DownArgs {
  const uint8_t* w_down;     // packed down tiles, see pack.cu
  __nv_bfloat16* out;        // [M][H]
  const int32_t* topk_idx;   // [M][K] the router's expert ids
  int M, H, I, K, E;
  int stages;
  uint32_t tile_bytes;       // 16 rows x I x 2
  Workspace ws;
};

// Router + top-k: grid ceil(E/8) x 256 threads, dynamic smem
// router_smem_bytes(M, H, K, E).  CPL = H/256 (16-byte chunks of a row per lane).
using RouterKernel = void (*)(RouterArgs);
RouterKernel router_kernel_for(int cpl);
size_t router_smem_bytes(int M, int H, int K, int E);

// Gate/up + SwiGLU: grid = #SMs x kExpertThreads.  KPW = H/256.
using GateUpKernel = void (*)(GateUpArgs);
GateUpKernel gateup_kernel_for(int kpw);
size_t gateup_smem_bytes(int stages, uint32_t tile_bytes, int NP, int E);

// Down + combine: grid = #SMs x kDownThreadsPerCta.  KS = I/16.
constexpr int kDownThreadsPerCta = kConsumerWarps * 32;
using DownKernel = void (*)(DownArgs);
DownKernel down_kernel_for(int ks);
size_t down_smem_bytes(int stages, uint32_t tile_bytes, int NP, int E, int H);

// Create-time re-layout (pack.cu).
void pack_gate_up(const __nv_bfloat16* src, __nv_bfloat16* dst, int E, int I, int H,
                  cudaStream_t s);
void pack_down(const __nv_bfloat16* src, __nv_bfloat16* dst, int E, int H, int I, cudaStream_t s);

// Set the calling thread's moe_last_error() text (moe_api.cu).
void set_last_error_text(const char* text);

}  // namespace wse
