// gemv_engines.cu -- one expert contraction y = W x for M <= 16 tokens on
// the CUDA cores or on the tensor cores, over the weight layout the layer
// kernel streams, and its C ABI (include/gemv.h): the measurement of where
// the tensor cores start to pay.
//
// Method (page "How Ling-3.0-flash reduces batch 1 decoding latency by 54%
// on 4 Blackwell GPUs"):
//  * "Two kinds of idle": a small-M step is bound by the cold read of the
//    activated expert weights.
//  * "Economics of speculation at batch 1": verifying several tokens reads
//    the same weights as verifying one, so each expert is streamed once for
//    all of its M_e tokens; per weight byte the work is M_e / 2
//    multiply-adds, and which engine does them matters only once M_e is
//    large enough for the arithmetic to catch up with HBM.
//
// GB300 design.  Both engines stream the same 8-row tiles (one contiguous
// block each, fragment order: lane (g, t) owns row g at k = 32q + 8t .. +7
// of chunk q, pack.cu) the same way: one warp per tile, 16 warps per SM,
// each warp with a private two-slot ring of 4 KB stages (8 chunks) in shared
// memory filled by bulk copies on an mbarrier (lane 0 issues; plain loads
// from every warp cannot keep enough bytes in flight to reach the HBM rate:
// measured 29 % of peak).  The tokens sit in shared memory too (padded rows).
// Only the arithmetic differs:
//  * CUDA cores: the tokens are staged as fp32 when they fit (a token then
//    costs two 16-byte shared loads and 8 FMAs per chunk), else as bf16
//    (one load, 8 shifts, 8 FMAs); the lane's 8 weights become fp32 once per
//    chunk (bf16 -> fp32 is a shift) and meet every token in 8 fp32 FMAs,
//    one accumulator per token; the 4 lanes of a row are summed by two
//    shuffles when the tile ends.
//  * Tensor cores: the same 16 bytes are the B operand of two mma.sync
//    m16n8k16 (k-steps 0 and 1), the tokens (8 or 16 rows) the A operand.
// Tokens past M never reach y.  Every wait is bounded: a timeout sets a
// device status word (moe_gemv_get_status) and the warp leaves its loop.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdint>

#include "gemv.h"
#include "kernels.cuh"

namespace wse {
namespace {

constexpr int kGemvWarps = 16;
constexpr int kStageChunks = 8;                        // chunks per stage
constexpr uint32_t kStageBytes = kStageChunks * 512;  // 4 KB
constexpr size_t kRingBytes = (size_t)kGemvWarps * 2 * kStageBytes;
constexpr size_t kSmemLimit = 227 * 1024;
// Token-row padding.  bf16 rows: k * 2 is a multiple of 512 (k % 256 == 0),
// so a 64-byte pad puts rows g and g + 1 in opposite halves of the 32 banks
// and a quarter-warp's 16-byte fragment loads (rows 2p, 2p + 1, 64 bytes
// each) are conflict-free.  fp32 rows are read by broadcast (every lane of a
// quarter-warp in one row): any 16-byte pad will do.
constexpr int kPadBf16 = 64, kPadF32 = 16;

__device__ int g_gemv_status;  // sticky: a bounded wait ran out

struct GemvArgs {
  const uint4* w;  // packed tiles
  const __nv_bfloat16* x;
  float* y;
  int rows, K, M;
};

// Shared-memory token rows: MB rows of K values (bf16, or fp32 when F32),
// each padded (kPadBf16 / kPadF32 bytes); rows past M are zero.
template <bool F32>
__device__ __forceinline__ void stage_tokens(const GemvArgs& a, int MB, uint8_t* xs, int row_bytes) {
  const int per_row = a.K / 8;  // 16-byte chunks of bf16
  for (int i = threadIdx.x; i < MB * per_row; i += blockDim.x) {
    const int m = i / per_row, c = i - m * per_row;
    const uint4 v = m < a.M ? reinterpret_cast<const uint4*>(a.x + (size_t)m * a.K)[c] : make_uint4(0, 0, 0, 0);
    if constexpr (F32) {
      float4* d = reinterpret_cast<float4*>(xs + (size_t)m * row_bytes + 32 * c);
      d[0] = make_float4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y));
      d[1] = make_float4(bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w));
    } else {
      *reinterpret_cast<uint4*>(xs + (size_t)m * row_bytes + 16 * c) = v;
    }
  }
  __syncthreads();
}

// The warp's stages in order: its tiles gw, gw + NW, ..., K/256 stages
// each, through its two ring slots.  Engine::chunk(b, q) consumes one chunk,
// Engine::finish(tile) writes a tile.
template <class Engine>
__device__ __forceinline__ void stream_tiles(const GemvArgs& a, Engine& eng, uint8_t* ring, uint32_t bars) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int gw = blockIdx.x * kGemvWarps + w, NW = gridDim.x * kGemvWarps;
  const int KC = a.K / 32, KS = KC / kStageChunks, n_tiles = a.rows / 8;
  if (gw >= n_tiles) return;
  const int total = (n_tiles - gw + NW - 1) / NW * KS;
  uint8_t* slots = ring + (size_t)w * 2 * kStageBytes;
  const uint32_t slots_u32 = smem_u32(slots), bar = bars + 16u * w;
  const uint64_t pol = l2_evict_first_policy();
  auto issue = [&](int i) {  // stage i of this warp into slot i & 1
    const int ti = gw + NW * (i / KS), j = i - (i / KS) * KS;
    mbar_arrive_expect_tx(bar + 8u * (i & 1), kStageBytes);
    bulk_g2s(slots_u32 + (uint32_t)(i & 1) * kStageBytes, a.w + ((size_t)ti * KC + j * kStageChunks) * 32,
             kStageBytes, bar + 8u * (i & 1), pol);
  };
  if (lane == 0) {
    mbar_init(bar, 1);
    mbar_init(bar + 8, 1);
    fence_mbar_init();
    issue(0);
    if (total > 1) issue(1);
  }
  __syncwarp();
  int q = 0, tile = gw;
  unsigned long long waited = 0;
  for (int i = 0; i < total; ++i) {
    if (!warp_wait(bar + 8u * (i & 1), (uint32_t)(i >> 1) & 1u, &waited)) {
      if (lane == 0) atomicOr(&g_gemv_status, 1);
      break;
    }
    const uint4* st = reinterpret_cast<const uint4*>(slots + (size_t)(i & 1) * kStageBytes) + lane;
#pragma unroll
    for (int c = 0; c < kStageChunks; ++c) eng.chunk(st[32 * c], q + c);
    q += kStageChunks;
    if (q == KC) {
      eng.finish(tile);
      q = 0;
      tile += NW;
    }
    fence_proxy_async_smem();  // this slot's reads before the next copy into it
    __syncwarp();
    if (lane == 0 && i + 2 < total) issue(i + 2);
  }
}

template <int MT, bool F32X>
struct CudaCoreEngine {
  const GemvArgs& a;
  const uint8_t* xs;
  int row_bytes, lane;
  float acc[MT];
  __device__ void chunk(const uint4& b, int q) {
    const float w0 = bf16lo(b.x), w1 = bf16hi(b.x), w2 = bf16lo(b.y), w3 = bf16hi(b.y);
    const float w4 = bf16lo(b.z), w5 = bf16hi(b.z), w6 = bf16lo(b.w), w7 = bf16hi(b.w);
    // token values k = 32q + 8t .. +7
    const uint8_t* xq = xs + (F32X ? 128 * q + 32 * (lane & 3) : 64 * q + 16 * (lane & 3));
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float4 u, v;
      if constexpr (F32X) {
        u = *reinterpret_cast<const float4*>(xq + (size_t)m * row_bytes);
        v = *reinterpret_cast<const float4*>(xq + (size_t)m * row_bytes + 16);
      } else {
        const uint4 h = *reinterpret_cast<const uint4*>(xq + (size_t)m * row_bytes);
        u = make_float4(bf16lo(h.x), bf16hi(h.x), bf16lo(h.y), bf16hi(h.y));
        v = make_float4(bf16lo(h.z), bf16hi(h.z), bf16lo(h.w), bf16hi(h.w));
      }
      float s = acc[m];
      s = fmaf(w0, u.x, s);
      s = fmaf(w1, u.y, s);
      s = fmaf(w2, u.z, s);
      s = fmaf(w3, u.w, s);
      s = fmaf(w4, v.x, s);
      s = fmaf(w5, v.y, s);
      s = fmaf(w6, v.z, s);
      s = fmaf(w7, v.w, s);
      acc[m] = s;
    }
  }
  __device__ void finish(int tile) {
    const int g = lane >> 2;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float v = acc[m];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      if ((lane & 3) == 0 && m < a.M) a.y[(size_t)m * a.rows + tile * 8 + g] = v;
      acc[m] = 0.f;
    }
  }
};

template <int TB>
struct TensorCoreEngine {
  const GemvArgs& a;
  const uint8_t* xs;
  int row_bytes, lane;
  float c0[4], c1[4];
  __device__ void chunk(const uint4& b, int q) {
    const int g = lane >> 2;
    const uint8_t* xq = xs + 64 * q + 16 * (lane & 3);
    const uint4 xa = *reinterpret_cast<const uint4*>(xq + (size_t)g * row_bytes);
    const uint4 xb = TB == 2 ? *reinterpret_cast<const uint4*>(xq + (size_t)(g + 8) * row_bytes) : xa;
    // logical k (2t, 2t+1 | 2t+8, 2t+9) of k-step 0 = physical 8t + (0,1 | 2,3);
    // k-step 1 takes physical 8t + (4,5 | 6,7)
    mma_bf16(c0, xa.x, xb.x, xa.y, xb.y, b.x, b.y);
    mma_bf16(c1, xa.z, xb.z, xa.w, xb.w, b.z, b.w);
  }
  __device__ void finish(int tile) {
    const int g = lane >> 2, n = tile * 8 + 2 * (lane & 3);
    if (g < a.M) {
      a.y[(size_t)g * a.rows + n] = c0[0] + c1[0];
      a.y[(size_t)g * a.rows + n + 1] = c0[1] + c1[1];
    }
    if (TB == 2 && g + 8 < a.M) {
      a.y[(size_t)(g + 8) * a.rows + n] = c0[2] + c1[2];
      a.y[(size_t)(g + 8) * a.rows + n + 1] = c0[3] + c1[3];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) c0[i] = c1[i] = 0.f;
  }
};

// Shared memory: the weight ring (16 warps x 2 x 4 KB), the token rows,
// then the warps' mbarriers (2 each).
template <int MT, bool F32X>
__global__ void __launch_bounds__(kGemvWarps * 32, 1) gemv_cuda_cores(GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int row_bytes = a.K * (F32X ? 4 : 2) + (F32X ? kPadF32 : kPadBf16);
  uint8_t* xs = smem + kRingBytes;
  stage_tokens<F32X>(a, MT, xs, row_bytes);
  CudaCoreEngine<MT, F32X> eng{a, xs, row_bytes, (int)(threadIdx.x & 31)};
#pragma unroll
  for (int m = 0; m < MT; ++m) eng.acc[m] = 0.f;
  stream_tiles(a, eng, smem, smem_u32(xs + (size_t)MT * row_bytes));
}

template <int TB>
__global__ void __launch_bounds__(kGemvWarps * 32, 1) gemv_tensor_cores(GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int row_bytes = a.K * 2 + kPadBf16;
  uint8_t* xs = smem + kRingBytes;
  stage_tokens<false>(a, 8 * TB, xs, row_bytes);
  TensorCoreEngine<TB> eng{a, xs, row_bytes, (int)(threadIdx.x & 31)};
#pragma unroll
  for (int i = 0; i < 4; ++i) eng.c0[i] = eng.c1[i] = 0.f;
  stream_tiles(a, eng, smem, smem_u32(xs + (size_t)8 * TB * row_bytes));
}

using GemvKernel = void (*)(GemvArgs);

template <bool F32X>
GemvKernel cuda_core_kernel(int M) {
  switch (M) {
    case 1: return gemv_cuda_cores<1, F32X>;
    case 2: return gemv_cuda_cores<2, F32X>;
    case 3: return gemv_cuda_cores<3, F32X>;
    case 4: return gemv_cuda_cores<4, F32X>;
    case 5: return gemv_cuda_cores<5, F32X>;
    case 6: return gemv_cuda_cores<6, F32X>;
    case 7: return gemv_cuda_cores<7, F32X>;
    case 8: return gemv_cuda_cores<8, F32X>;
    case 9: return gemv_cuda_cores<9, F32X>;
    case 10: return gemv_cuda_cores<10, F32X>;
    case 11: return gemv_cuda_cores<11, F32X>;
    case 12: return gemv_cuda_cores<12, F32X>;
    case 13: return gemv_cuda_cores<13, F32X>;
    case 14: return gemv_cuda_cores<14, F32X>;
    case 15: return gemv_cuda_cores<15, F32X>;
    case 16: return gemv_cuda_cores<16, F32X>;
    default: return nullptr;
  }
}

void fail(const char* fmt, ...) {
  char buf[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  set_last_error_text(buf);
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool sizes_ok(int rows, int k, int k_step) {
  if (rows < 8 || rows % 8 || k < k_step || k > MOE_GEMV_MAX_K || k % k_step) {
    fail("rows = %d must be a positive multiple of 8 and k = %d a multiple of %d in [%d, %d]", rows, k, k_step,
         k_step, MOE_GEMV_MAX_K);
    return false;
  }
  return true;
}

}  // namespace
}  // namespace wse

using namespace wse;

extern "C" {

int moe_gemv_pack(const void* w, void* packed, int rows, int k, moe_stream_t stream) {
  if (!sizes_ok(rows, k, 32)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(packed)) {
    fail("w and packed must be non-null, 16-byte aligned device pointers");
    return MOE_ERR_INVALID_ARG;
  }
  // the layer's down-weight re-layout, as one "expert" of rows x k
  pack_down(static_cast<const __nv_bfloat16*>(w), static_cast<__nv_bfloat16*>(packed), 1, rows, k,
            reinterpret_cast<cudaStream_t>(stream));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    fail("%s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int moe_gemv(const void* packed, const void* x, float* y, int rows, int k, int M, int engine,
             moe_stream_t stream) {
  if (!sizes_ok(rows, k, 32 * kStageChunks)) return MOE_ERR_INVALID_ARG;
  if (M < 0 || (engine != MOE_GEMV_CUDA_CORES && engine != MOE_GEMV_TENSOR_CORES)) {
    fail("M = %d must be >= 0 and engine = %d one of MOE_GEMV_CUDA_CORES, MOE_GEMV_TENSOR_CORES", M, engine);
    return MOE_ERR_INVALID_ARG;
  }
  if (M > MOE_GEMV_MAX_TOKENS) {
    fail("M = %d exceeds %d", M, MOE_GEMV_MAX_TOKENS);
    return MOE_ERR_UNSUPPORTED;
  }
  if (M == 0) return MOE_OK;
  if (!aligned16(packed) || !aligned16(x) || !y || (reinterpret_cast<uintptr_t>(y) & 3u)) {
    fail("packed and x must be 16-byte aligned and y 4-byte aligned non-null device pointers");
    return MOE_ERR_INVALID_ARG;
  }
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    fail("%s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  GemvArgs ga{reinterpret_cast<const uint4*>(packed), static_cast<const __nv_bfloat16*>(x), y, rows, k, M};
  // ring + token rows + 2 mbarriers per warp; the CUDA cores take fp32
  // token rows when they fit, else bf16
  const size_t bars = (size_t)kGemvWarps * 16;
  const size_t f32 = kRingBytes + (size_t)M * (4 * (size_t)k + kPadF32) + bars;
  GemvKernel kern;
  size_t smem;
  if (engine == MOE_GEMV_CUDA_CORES) {
    const bool fits = f32 <= kSmemLimit;
    kern = fits ? cuda_core_kernel<true>(M) : cuda_core_kernel<false>(M);
    smem = fits ? f32 : kRingBytes + (size_t)M * (2 * (size_t)k + kPadBf16) + bars;
  } else {
    kern = M <= 8 ? gemv_tensor_cores<1> : gemv_tensor_cores<2>;
    smem = kRingBytes + (size_t)(M <= 8 ? 8 : 16) * (2 * (size_t)k + kPadBf16) + bars;
  }
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess) {
    fail("%s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  const int n_tiles = rows / 8;
  const int ctas = (n_tiles + kGemvWarps - 1) / kGemvWarps < sms ? (n_tiles + kGemvWarps - 1) / kGemvWarps : sms;
  kern<<<ctas, kGemvWarps * 32, smem, reinterpret_cast<cudaStream_t>(stream)>>>(ga);
  if ((e = cudaGetLastError()) != cudaSuccess) {
    fail("%s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int moe_gemv_get_status(void) {
  int st = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&st, g_gemv_status, sizeof st);
  if (e != cudaSuccess) {
    fail("%s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  if (st == 0) return MOE_OK;
  const int zero = 0;
  cudaMemcpyToSymbol(g_gemv_status, &zero, sizeof zero);
  fail("a moe_gemv stage wait ran out (status 0x%x)", st);
  return MOE_ERR_DEVICE_TIMEOUT;
}

}  // extern "C"
