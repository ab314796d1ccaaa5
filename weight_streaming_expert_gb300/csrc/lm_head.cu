// lm_head.cu -- the bf16 vocabulary projection of a decode/verify step,
// logits[m][v] = x[m] . W[v] for M <= 16 tokens, as one persistent kernel
// that streams W once, plus its host runtime (include/lm_head.h).
//
// Method (page "How Ling-3.0-flash reduces batch 1 decoding latency by 54%
// on 4 Blackwell GPUs", section "bf16 router gate and lm_head"): at batch 1
// the lm_head is pure bandwidth -- every decode step cold-reads the whole
// projection and has no arithmetic to hide the read behind; in bf16 it reads
// half the bytes of fp32.  The post splits it vocab-parallel over 4 GPUs; a
// vocab-parallel slice is this kernel on fewer rows.
//
// GB300 design.  One CTA per SM: 8 consumer warps and 1 producer warp.  At
// create the weight is re-laid out into tiles of 8 vocabulary rows x H in
// the layer kernel's tensor-core fragment order (pack.cu explains it): one
// contiguous bulk copy per tile (40 KB at H 2560), and a warp's 512-byte
// contiguous shared-memory read hands every lane its m16n8k16 B registers.
// The tiles are split statically over the CTAs: the stream is long and
// uniform (about 130 tiles per SM at 157k x 2560).  The producer stages the
// tiles into a ring of mbarrier-guarded stages, with an L2 evict-first
// policy (the weight is read once per call).  The consumers hold the M
// tokens' A fragments of their eighth of H in registers for the whole call;
// per tile each warp runs its k chunks and a rotating reducer warp sums the
// eight partial 16 x 8 tiles in a fixed order and writes fp32 logits.
// Every wait is bounded: a timeout sets a sticky status bit and the thread
// leaves its loop.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdint>

#include "kernels.cuh"
#include "lm_head.h"

namespace wse {
namespace {

constexpr int kLmThreads = (kConsumerWarps + 1) * 32;  // 8 consumers + the producer warp
constexpr int kLmRedSlots = 8;                           // reduction slots (> ring stages)
constexpr int kLmMaxStages = kLmRedSlots - 1;
constexpr uint32_t kLmBarBytes = 1024;                   // barrier area ahead of the ring
constexpr uint32_t kLmRedBytes = kLmRedSlots * kConsumerWarps * 32 * 16;

struct LmHeadArgs {
  const __nv_bfloat16* x;  // [M][H]
  const uint8_t* w;        // packed tiles
  float* logits;           // [M][V]
  int M, H, V;
  int n_tiles;             // ceil(V / 8)
  int stages;
  uint32_t tile_bytes;     // 8 x H x 2
  int* status;
};

template <int KPW>  // H / 256: 32-wide k chunks per warp
__global__ void __launch_bounds__(kLmThreads, 1) lm_head_kernel(LmHeadArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = a.stages;
  const uint32_t sb = smem_u32(smem);
  auto full = [&](int s) { return sb + 8u * s; };
  auto empty = [&](int s) { return sb + 64u + 8u * s; };
  auto redbar = [&](int r) { return sb + 128u + 8u * r; };
  uint8_t* ring = smem + kLmBarBytes;
  float4* red = reinterpret_cast<float4*>(ring + (size_t)S * a.tile_bytes);
  const int t0 = (int)((long long)a.n_tiles * blockIdx.x / gridDim.x);
  const int t1 = (int)((long long)a.n_tiles * (blockIdx.x + 1) / gridDim.x);
  const int n = t1 - t0;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kConsumerWarps);
    }
    for (int r = 0; r < kLmRedSlots; ++r) mbar_init(redbar(r), kConsumerWarps);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();               // x belongs to this call now
  pdl_launch_dependents();  // the next call's prologue may start as SMs free up
  unsigned long long waited = 0;

  if (warp == kProducerWarp) {
    if (lane != 0) return;
    const uint64_t pol = l2_evict_first_policy();
    for (int j = 0; j < n; ++j) {
      const int s = j % S;
      if (j >= S && !mbar_wait(empty(s), ((j / S) - 1) & 1, &waited)) {
        set_error(a.status, kErrTimeoutEmpty);
        return;
      }
      mbar_arrive_expect_tx(full(s), a.tile_bytes);
      bulk_g2s_chunked(sb + kLmBarBytes + (uint32_t)s * a.tile_bytes, a.w + (size_t)(t0 + j) * a.tile_bytes,
                       a.tile_bytes, full(s), pol);
    }
    return;
  }

  // ---- consumers: A fragments of tokens g4 and g4 + 8 (rows beyond M
  // repeat token 0 and are never stored), this warp's k chunks
  const int g4 = lane >> 2, t4 = lane & 3;
  uint4 xa[KPW], xb[KPW];
  {
    const int m0 = g4 < a.M ? g4 : 0, m1 = g4 + 8 < a.M ? g4 + 8 : 0;
    const uint4* x0 = reinterpret_cast<const uint4*>(a.x + (size_t)m0 * a.H) + t4;
    const uint4* x1 = reinterpret_cast<const uint4*>(a.x + (size_t)m1 * a.H) + t4;
#pragma unroll
    for (int q = 0; q < KPW; ++q) {
      xa[q] = x0[4 * (warp * KPW + q)];
      xb[q] = x1[4 * (warp * KPW + q)];
    }
  }
  for (int j = 0; j < n; ++j) {
    const int s = j % S;
    if (!warp_wait(full(s), (uint32_t)(j / S) & 1u, &waited)) {
      if (lane == 0) set_error(a.status, kErrTimeoutFull);
      break;
    }
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    const uint4* wp = reinterpret_cast<const uint4*>(ring + (size_t)s * a.tile_bytes) + (warp * KPW) * 32 + lane;
#pragma unroll
    for (int q = 0; q < KPW; ++q) {
      const uint4 b = wp[q * 32];
      mma_bf16(c0, xa[q].x, xb[q].x, xa[q].y, xb[q].y, b.x, b.y);
      mma_bf16(c1, xa[q].z, xb[q].z, xa[q].w, xb[q].w, b.z, b.w);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));  // stage free for the producer
    const int slot = j & (kLmRedSlots - 1);
    red[(slot * kConsumerWarps + warp) * 32 + lane] =
        make_float4(c0[0] + c1[0], c0[1] + c1[1], c0[2] + c1[2], c0[3] + c1[3]);
    __syncwarp();
    if (lane == 0) mbar_arrive(redbar(slot));
    if (warp == slot) {  // this tile's reducer (rotates over the warps)
      if (!warp_wait(redbar(slot), (uint32_t)(j >> 3) & 1u, &waited)) {
        if (lane == 0) set_error(a.status, kErrTimeoutReduce);
        break;
      }
      float4 acc = red[(slot * kConsumerWarps) * 32 + lane];
#pragma unroll
      for (int w2 = 1; w2 < kConsumerWarps; ++w2) {
        const float4 v = red[(slot * kConsumerWarps + w2) * 32 + lane];
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      // (acc.x, acc.y): token g4, vocabulary rows v, v + 1; (acc.z, acc.w):
      // token g4 + 8, the same rows
      const int v = (t0 + j) * 8 + 2 * t4;
      if (g4 < a.M) {
        float* o = a.logits + (size_t)g4 * a.V + v;
        if (v < a.V) o[0] = acc.x;
        if (v + 1 < a.V) o[1] = acc.y;
      }
      if (g4 + 8 < a.M) {
        float* o = a.logits + (size_t)(g4 + 8) * a.V + v;
        if (v < a.V) o[0] = acc.z;
        if (v + 1 < a.V) o[1] = acc.w;
      }
    }
  }
}

// Rows [0, V) of W [V][H] into tiles of 8 rows in fragment order; rows of
// the last tile at or beyond V are zero.  16-byte chunk (tile, q, lane) =
// row 8 tile + lane / 4, elements 32 q + 8 (lane % 4) .. + 7.
__global__ void pack_lm_head_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int V, int H) {
  const int KC = H / 32, RC = H / 8;
  const long long total = (long long)((V + 7) / 8) * KC * 32;
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < total;
       c += (long long)gridDim.x * blockDim.x) {
    const int lane = (int)(c & 31);
    const long long r = c >> 5;
    const int q = (int)(r % KC);
    const long long tile = r / KC;
    const long long row = tile * 8 + (lane >> 2);
    dst[c] = row < V ? src[row * RC + 4 * q + (lane & 3)] : make_uint4(0u, 0u, 0u, 0u);
  }
}

using LmKernel = void (*)(LmHeadArgs);

LmKernel lm_kernel_for(int kpw) {
  switch (kpw) {
    case 1: return lm_head_kernel<1>;
    case 2: return lm_head_kernel<2>;
    case 4: return lm_head_kernel<4>;
    case 5: return lm_head_kernel<5>;
    case 8: return lm_head_kernel<8>;
    case 10: return lm_head_kernel<10>;
    case 12: return lm_head_kernel<12>;
    case 16: return lm_head_kernel<16>;
    default: return nullptr;
  }
}

void err(const char* fmt, int a = 0, int b = 0) {
  char buf[256];
  snprintf(buf, sizeof buf, fmt, a, b);
  set_last_error_text(buf);
}

}  // namespace
}  // namespace wse

using namespace wse;

struct moe_lm_head {
  int H = 0, V = 0, n_tiles = 0, n_sms = 0, stages = 0;
  uint32_t tile_bytes = 0;
  size_t smem = 0;
  uint8_t* w = nullptr;
  int* status = nullptr;
  LmKernel kernel = nullptr;
};

static void free_lm(moe_lm_head* h) {
  if (!h) return;
  cudaFree(h->w);
  cudaFree(h->status);
  delete h;
}

extern "C" {

moe_lm_head_t* moe_lm_head_create(int hidden, int vocab, const void* w) {
  if (hidden <= 0 || hidden % 256 != 0 || !lm_kernel_for(hidden / 256)) {
    err("hidden = %d: must be a multiple of 256 with a kernel instance (256..4096)", hidden);
    return nullptr;
  }
  if (vocab <= 0 || vocab > (1 << 24)) {
    err("vocab = %d: must be in 1..16777216", vocab);
    return nullptr;
  }
  if (!w || (reinterpret_cast<uintptr_t>(w) & 15u)) {
    err("w must be a non-null, 16-byte aligned device pointer");
    return nullptr;
  }
  int dev = 0;
  cudaDeviceProp prop{};
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess || (e = cudaGetDeviceProperties(&prop, dev)) != cudaSuccess) {
    cudaGetLastError();
    set_last_error_text(cudaGetErrorString(e));
    return nullptr;
  }
  if (prop.major != 10 || prop.minor != 3) {
    err("device is sm_%d%d; this library is built for sm_103a (GB300)", prop.major, prop.minor);
    return nullptr;
  }
  auto* h = new moe_lm_head;
  h->H = hidden;
  h->V = vocab;
  h->n_tiles = (vocab + 7) / 8;
  h->n_sms = prop.multiProcessorCount;
  h->tile_bytes = 8u * (uint32_t)hidden * 2u;
  const size_t avail = prop.sharedMemPerBlockOptin;
  const size_t fixed = kLmBarBytes + kLmRedBytes;
  const int s = avail > fixed ? (int)((avail - fixed) / h->tile_bytes) : 0;
  h->stages = s < kLmMaxStages ? s : kLmMaxStages;
  if (h->stages < 2) {
    err("hidden = %d: fewer than 2 ring stages fit in shared memory", hidden);
    free_lm(h);
    return nullptr;
  }
  h->smem = fixed + (size_t)h->stages * h->tile_bytes;
  h->kernel = lm_kernel_for(hidden / 256);
  if ((e = cudaFuncSetAttribute(h->kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h->smem)) !=
      cudaSuccess) {
    cudaGetLastError();
    set_last_error_text(cudaGetErrorString(e));
    free_lm(h);
    return nullptr;
  }
  const size_t packed = (size_t)h->n_tiles * h->tile_bytes;
  if (cudaMalloc(&h->w, packed) != cudaSuccess || cudaMalloc(&h->status, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    err("device allocation of the %d-row lm_head weight failed", vocab);
    free_lm(h);
    return nullptr;
  }
  cudaMemset(h->status, 0, sizeof(int));
  // the caller's weight may still be being written by work queued on any
  // stream: wait for the device before the re-layout reads it
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) {
    set_last_error_text(cudaGetErrorString(e));
    free_lm(h);
    return nullptr;
  }
  pack_lm_head_kernel<<<4096, 256>>>(static_cast<const uint4*>(w), reinterpret_cast<uint4*>(h->w), vocab, hidden);
  if ((e = cudaDeviceSynchronize()) != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) {
    set_last_error_text(cudaGetErrorString(e));
    free_lm(h);
    return nullptr;
  }
  return h;
}

int moe_lm_head_forward(moe_lm_head_t* h, const void* x, float* logits, int M, moe_stream_t stream) {
  if (!h) {
    err("null handle");
    return MOE_ERR_INVALID_ARG;
  }
  if (M < 0) {
    err("M = %d < 0", M);
    return MOE_ERR_INVALID_ARG;
  }
  if (M > MOE_LM_HEAD_MAX_TOKENS) {
    err("M = %d exceeds %d", M, MOE_LM_HEAD_MAX_TOKENS);
    return MOE_ERR_UNSUPPORTED;
  }
  if (M == 0) return MOE_OK;
  if (!x || !logits || (reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(logits) & 3u)) {
    err("x must be non-null and 16-byte aligned, logits non-null and 4-byte aligned");
    return MOE_ERR_INVALID_ARG;
  }
  LmHeadArgs la{};
  la.x = static_cast<const __nv_bfloat16*>(x);
  la.w = h->w;
  la.logits = logits;
  la.M = M;
  la.H = h->H;
  la.V = h->V;
  la.n_tiles = h->n_tiles;
  la.stages = h->stages;
  la.tile_bytes = h->tile_bytes;
  la.status = h->status;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c{};
  c.stream = reinterpret_cast<cudaStream_t>(stream);
  c.attrs = attr;
  c.numAttrs = 1;
  c.gridDim = dim3(h->n_tiles < h->n_sms ? h->n_tiles : h->n_sms);
  c.blockDim = dim3(kLmThreads);
  c.dynamicSmemBytes = h->smem;
  const cudaError_t e = cudaLaunchKernelEx(&c, h->kernel, la);
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_last_error_text(cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int moe_lm_head_get_status(moe_lm_head_t* h) {
  if (!h) {
    err("null handle");
    return MOE_ERR_INVALID_ARG;
  }
  int st = 0;
  cudaError_t e;
  if ((e = cudaDeviceSynchronize()) != cudaSuccess ||
      (e = cudaMemcpy(&st, h->status, sizeof st, cudaMemcpyDeviceToHost)) != cudaSuccess) {
    set_last_error_text(cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  if (st == 0) return MOE_OK;
  err("lm_head device wait ran out (status bits 0x%x)", st);
  return MOE_ERR_DEVICE_TIMEOUT;
}

void moe_lm_head_destroy(moe_lm_head_t* h) {
  if (!h) return;
  cudaDeviceSynchronize();
  free_lm(h);
}

}  // extern "C"
