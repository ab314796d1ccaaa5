// router.cu -- router gate matvec + softmax top-k with renormalisation.
//
// Method (page "How Ling-3.0-flash reduces batch 1 decoding latency by 54%
// on 4 Blackwell GPUs"):
//  * "bf16 router gate and lm_head": the gate weight is bf16 and pure
//    bandwidth (2.6 MB per layer at hidden 2560 x 512 experts).
//  * "PDL: the latency floor of stacked small kernels", Figure 7: the gate's
//    weight load does not depend on the producer, so it is issued BEFORE the
//    dependency wait and the cold read flies under the producer's tail; the
//    top-k prefetches its bias the same way.
//
// GB300 design: each warp owns one expert row (H bf16 held in registers,
// 16-byte coalesced loads), so E/8 CTAs of 8 warps read the 2.6 MB once.
// The tokens are staged into shared memory in blocks of 8 with cp.async
// (double-buffered, one round trip per block), and every warp takes its
// dot products from there.  The last CTA to finish (a device-scope arrival
// counter; no spin) runs the top-k: one warp per token, the E logits held
// in registers, k rounds of a two-step redux.sync arg-max (largest value,
// then lowest expert id) with a branch-free rescan of the winning lane.
// The same CTA then builds the token->expert compaction block-wide in
// shared memory and publishes it (compaction.cuh); every CTA of the expert
// kernels loads it with one coalesced read.
#include "compaction.cuh"
#include "kernels.cuh"

namespace wse {

constexpr int kRouterTokBlock = 8;  // tokens staged per shared-memory block

size_t router_smem_bytes(int M, int H, int K, int E) {
  const int rows = M <= kRouterTokBlock ? M : 2 * kRouterTokBlock;
  const size_t stage = (size_t)rows * H * 2;
  const size_t comp = compaction_smem_ints(M * K, E) * 4;  // last CTA, after the tokens
  return stage > comp ? stage : comp;
}

namespace {

// Order-preserving map of a finite float to an unsigned key (larger float ->
// larger key); key 0 is below every finite float and marks "no candidate".
__device__ __forceinline__ uint32_t ordered_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// acc + sum_i w[i]*x[i] over 8 bf16 pairs, fp32.
__device__ __forceinline__ float dot8(const uint4 w, const uint4 x, float acc) {
  acc = fmaf(bf16lo(w.x), bf16lo(x.x), acc);
  acc = fmaf(bf16hi(w.x), bf16hi(x.x), acc);
  acc = fmaf(bf16lo(w.y), bf16lo(x.y), acc);
  acc = fmaf(bf16hi(w.y), bf16hi(x.y), acc);
  acc = fmaf(bf16lo(w.z), bf16lo(x.z), acc);
  acc = fmaf(bf16hi(w.z), bf16hi(x.z), acc);
  acc = fmaf(bf16lo(w.w), bf16lo(x.w), acc);
  acc = fmaf(bf16hi(w.w), bf16hi(x.w), acc);
  return acc;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Stage tokens [8b, 8b+8) of x into shared buffer (b & 1).
__device__ __forceinline__ void stage_tokens(const RouterArgs& a, uint4* xs, int b) {
  const int hc = a.H >> 3;  // 16-byte chunks per token
  const int m0 = b * kRouterTokBlock;
  const int tb = min(kRouterTokBlock, a.M - m0);
  uint4* dst = xs + (size_t)(b & 1) * kRouterTokBlock * hc;
  const uint4* src = reinterpret_cast<const uint4*>(a.x) + (size_t)m0 * hc;
  for (int i = threadIdx.x; i < tb * hc; i += blockDim.x) cp_async16(dst + i, src + i);
  cp_async_commit();
}

// Top-k of token m by one warp; lane l holds the keys of experts l + 32v.
// Round j: the largest remaining value (redux max), then the lowest expert id
// holding it (redux min); lane j keeps result j; the winning lane drops the
// entry and every lane rescans its VPL keys (no divergent loop).  Weights:
// exp(l_j - l_0) normalised over the k chosen = softmax over all E
// renormalised over the k (the full denominator cancels).
template <int VPL>
__device__ void topk_token(const RouterArgs& a, int m, int lane) {
  const float* L = a.ws.logits + (size_t)m * a.E;
  uint32_t key[VPL];
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = v * 32 + lane;
    key[v] = e < a.E ? ordered_key(__ldcg(L + e)) : 0u;
  }
  uint32_t best = 0;
  int bv = 0;
#pragma unroll
  for (int v = 0; v < VPL; ++v)
    if (key[v] > best) { best = key[v]; bv = v; }

  int my_idx = 0;
  float my_val = 0.f;
  for (int j = 0; j < a.K; ++j) {
    const uint32_t top = __reduce_max_sync(0xffffffffu, best);
    const uint32_t cand = (best != 0u && best == top) ? (uint32_t)(bv * 32 + lane) : 0xffffffffu;
    uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    if (win >= (uint32_t)a.E) {  // no candidate left: only a NaN logit pattern can cause it
      if (lane == 0) set_error(a.ws.status, kErrBadIndex);
      win = 0;
    }
    if (lane == j) {
      my_idx = (int)win;
      my_val = key_value(top);
    }
    const bool mine = (int)(win & 31u) == lane;
    uint32_t nb = 0;
    int nv = 0;
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      const uint32_t kv = (mine && v == bv) ? 0u : key[v];
      key[v] = kv;
      if (kv > nb) { nb = kv; nv = v; }
    }
    best = nb;
    bv = nv;
  }
  const float v0 = __shfl_sync(0xffffffffu, my_val, 0);
  const float ex = lane < a.K ? expf(my_val - v0) : 0.f;
  float s = 0.f;
  for (int j = 0; j < a.K; ++j) s += __shfl_sync(0xffffffffu, ex, j);
  if (lane < a.K) {
    const float w = ex / s;
    const int p = m * a.K + lane;
    a.topk_idx[p] = my_idx;
    if (a.topk_w) a.topk_w[p] = w;
    a.ws.pair_w[p] = w;
  }
}

__device__ __forceinline__ void topk_dispatch(const RouterArgs& a, int m, int lane) {
  if (a.E <= 32) topk_token<1>(a, m, lane);
  else if (a.E <= 64) topk_token<2>(a, m, lane);
  else if (a.E <= 128) topk_token<4>(a, m, lane);
  else if (a.E <= 256) topk_token<8>(a, m, lane);
  else if (a.E <= 512) topk_token<16>(a, m, lane);
  else topk_token<32>(a, m, lane);
}

}  // namespace

template <int CPL>
__global__ void __launch_bounds__(kRouterThreads) router_topk_kernel(RouterArgs a) {
  extern __shared__ __align__(16) uint4 xs[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouterExpertsPerCta + warp;
  const bool has_row = e < a.E;

  // Producer-independent: the router row and bias are constant across calls.
  uint4 w[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) w[c] = make_uint4(0, 0, 0, 0);
  if (has_row) {
    const uint4* wr = reinterpret_cast<const uint4*>(a.w_router + (size_t)e * a.H) + lane;
#pragma unroll
    for (int c = 0; c < CPL; ++c) w[c] = __ldg(wr + c * 32);
  }
  const float bias = (has_row && a.bias) ? __ldg(a.bias + e) : 0.f;

  pdl_wait();               // x (and the workspace) now belong to this call
  pdl_launch_dependents();  // the gate/up kernel may start its prologue

  const int hc = a.H >> 3;
  const int nblk = (a.M + kRouterTokBlock - 1) / kRouterTokBlock;
  stage_tokens(a, xs, 0);
  for (int b = 0; b < nblk; ++b) {
    if (b + 1 < nblk) {
      stage_tokens(a, xs, b + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const int m0 = b * kRouterTokBlock;
    const int tb = min(kRouterTokBlock, a.M - m0);
    const uint4* xb = xs + (size_t)(b & 1) * kRouterTokBlock * hc + lane;
    float s[kRouterTokBlock];
#pragma unroll
    for (int t = 0; t < kRouterTokBlock; ++t) s[t] = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
#pragma unroll
      for (int t = 0; t < kRouterTokBlock; ++t)
        if (t < tb) s[t] = dot8(w[c], xb[(size_t)t * hc + c * 32], s[t]);
    }
#pragma unroll
    for (int t = 0; t < kRouterTokBlock; ++t) {
      if (t < tb) {
        float v = s[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0 && has_row) a.ws.logits[(size_t)(m0 + t) * a.E + e] = v + bias;
      }
    }
    __syncthreads();  // the buffer is refilled two blocks later
  }

  // The last CTA to finish runs the top-k.
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(a.ws.router_count, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int m = warp; m < a.M; m += kRouterThreads / 32) topk_dispatch(a, m, lane);
  __syncthreads();  // this CTA's topk_idx writes are visible to it
  // token->expert compaction ("Two fusions and a retune", pair axis), built
  // block-wide in shared memory (reusing the token buffer) and published
  const SmemRouting rt = compact_routing(a.topk_idx, a.M * a.K, a.E, reinterpret_cast<int*>(xs),
                                         a.ws.status);
  publish_routing(rt, a.M * a.K, a.ws);
  if (threadIdx.x == 0) *a.ws.router_count = 0;  // ready for the next call
}

RouterKernel router_kernel_for(int cpl) {
  switch (cpl) {
    case 1: return router_topk_kernel<1>;
    case 2: return router_topk_kernel<2>;
    case 4: return router_topk_kernel<4>;
    case 5: return router_topk_kernel<5>;
    case 8: return router_topk_kernel<8>;
    case 10: return router_topk_kernel<10>;
    case 12: return router_topk_kernel<12>;
    case 16: return router_topk_kernel<16>;
    default: return nullptr;
  }
}

}  // namespace wse
