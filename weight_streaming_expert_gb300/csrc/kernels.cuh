// kernels.cuh -- argument block and launch-side declarations of the layer
// kernel, the allocation-free routing kernel and the create-time weight
// re-layout.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace wse {

struct LayerArgs {
  const __nv_bfloat16* x;         // [M][H]
  const __nv_bfloat16* w_router;  // [E][H] (caller layout)
  const float* bias;              // [E] or nullptr
  const uint8_t* w_gate_up;       // packed gate/up tiles, see pack.cu
  const uint8_t* w_down;          // packed down tiles, see pack.cu
  const float* s_gu;              // fp8 experts: [E][2I] gate/up row scales (else unused)
  const float* s_d;               // fp8 experts: [E][H] down row scales (else unused)
  __nv_bfloat16* out;             // [M][H] (unused when out_f32 is set)
  float* out_f32;                 // nullptr, or [M][H]: the combine's fp32 sums, not rounded
  int32_t* topk_idx;              // [M][K] caller output
  float* topk_w;                  // [M][K] caller output or nullptr
  int M, H, E, K, I;
  int ks;                         // hidden-dim split of the router matvec
  int gu_stages;                  // gate/up ring depth
  int d_stages;                   // down slots of one super tile (8 cells) each
  uint32_t gu_tile;               // 8 rows x H x 2 bytes
  uint32_t d_tile;                // one down cell: d_spw slabs of 8 rows x I x 2 bytes
  int d_spw;                      // down slabs per cell (a consumer warp's unit; <= 512 / I)
  uint32_t ring_bytes;            // gu_stages*gu_tile + the reduction area
  int trace;                      // record phase timestamps
  int shared;                     // 1: expert E is a shared expert every token passes (weight 1)
  float routed_scale;             // factor on every routed weight
  int sel_only;                   // 1: the bias picks the experts, unbiased logits weigh them
  unsigned long long wait_ns;     // limit of every bounded wait (ns)
  int test_flags;                 // kTestSkipArrival: see below
  Workspace ws;
};

// Test aid: CTA 0 leaves out its arrival at the grid-wide count of reduced
// static gate/up tiles, so every CTA's wait on that count runs out (bounded)
// and the call reports MOE_ERR_DEVICE_TIMEOUT through moe_get_status.
constexpr int kTestSkipArrival = 1;

// The layer kernel: grid = #SMs x kExpertThreads, dynamic shared memory
// layer_smem_bytes(ring_bytes, NP, buckets).  KPW = H/256.
using LayerKernel = void (*)(LayerArgs);
// variant: the instance that handles the layer variants; fp8: the instance
// for E4M3 expert weights (plain layers only); token_blocks: groups of up to
// 8 x token_blocks tokens (1: calls with M <= 8; 2: any call).  nullptr: no
// such instance.
LayerKernel layer_kernel_for(int kpw, bool variant, bool fp8 = false, int token_blocks = 2);
size_t layer_smem_bytes(uint32_t ring_bytes, int NP, int E);
// Bytes of the reduction area that follows the gate/up stages (fp8 with two
// token blocks: two partials per lane).
uint32_t layer_reduction_bytes(bool fp8 = false, int token_blocks = 2);

// Create-time re-layout (pack.cu).
void pack_gate_up(const __nv_bfloat16* src, __nv_bfloat16* dst, int E, int I, int H,
                  cudaStream_t s);
void pack_down(const __nv_bfloat16* src, __nv_bfloat16* dst, int E, int H, int I, cudaStream_t s);
// E4M3 codes: gate/up tiles of 16 rows, down slabs of 16 rows (pack.cu).
void pack_gate_up_fp8(const uint8_t* src, uint8_t* dst, int E, int I, int H, cudaStream_t s);
void pack_down_fp8(const uint8_t* src, uint8_t* dst, int E, int H, int I, cudaStream_t s);

// Set the calling thread's moe_last_error() text (moe_api.cu).
void set_last_error_text(const char* text);

}  // namespace wse
