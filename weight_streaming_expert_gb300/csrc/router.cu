// router.cu -- router gate matvec + softmax top-k + on-device token->expert
// compaction, in one launch.
//
// Method (page "How Ling-3.0-flash reduces batch 1 decoding latency by 54%
// on 4 Blackwell GPUs"):
//  * "bf16 router gate and lm_head": the gate weight is bf16 and pure
//    bandwidth (2.6 MB per layer at hidden 2560 x 512 experts).
//  * "PDL: the latency floor of stacked small kernels", Figure 7: the gate's
//    weight load does not depend on the producer, so it is issued BEFORE the
//    dependency wait and the cold read flies under the producer's tail; the
//    top-k prefetches its bias the same way.
//  * "Two fusions and a retune" (moe_align on the pair axis): the M*k
//    (token, slot) pairs are bucketed by expert with a rank that is stable in
//    pair index, the bucket populations give bucket-ordered offsets and the
//    published total; nothing is read back to the host and the tail beyond
//    the published total is left unwritten.
//
// GB300 design: each warp owns one expert row (H bf16 in registers, 16-byte
// coalesced loads), so E/8 CTAs of 8 warps read the 2.6 MB once.  The last
// CTA to finish (a device-scope counter, no spin) does the top-k (one warp
// per token: k rounds of a two-step redux.sync arg-max over register keys)
// and the compaction (shared-memory histogram, one warp-wide scan, and a
// stable in-bucket rank from __match_any_sync over 32-pair chunks).
#include "kernels.cuh"

namespace wse {

size_t router_smem_bytes(int M, int E, int K) {
  const size_t np = (size_t)M * K;
  return np * 8 + (size_t)E * 12;  // s_idx, s_w [NP]; s_cnt, s_off, s_run [E]
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

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// T tokens starting at m against the register-resident expert row.
template <int CPL, int T>
__device__ __forceinline__ void logits_tokens(const RouterArgs& a, const uint4 (&w)[CPL], int m,
                                              int e, float bias, int lane) {
  const uint4* xr[T];
#pragma unroll
  for (int t = 0; t < T; ++t)
    xr[t] = reinterpret_cast<const uint4*>(a.x + (size_t)(m + t) * a.H) + lane;
  float s[T];
#pragma unroll
  for (int t = 0; t < T; ++t) s[t] = 0.f;
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
#pragma unroll
    for (int t = 0; t < T; ++t) s[t] = dot8(w[c], xr[t][c * 32], s[t]);
  }
#pragma unroll
  for (int t = 0; t < T; ++t) {
    const float v = warp_sum(s[t]);
    if (lane == 0) a.ws.logits[(size_t)(m + t) * a.E + e] = v + bias;
  }
}

// Top-k of token m by one warp.  Lane l holds the keys of experts l, l+32, ...
// Round j selects the largest remaining value with two warp reductions
// (max of the value keys, then min of the expert ids holding it); lane j
// keeps result j.  Weights: exp(l_j - l_0) normalised over
// the k chosen (= softmax over all E renormalised over the k; the full
// denominator cancels).
__device__ void topk_token(const RouterArgs& a, int m, int lane, int* s_idx, float* s_w) {
  const float* L = a.ws.logits + (size_t)m * a.E;
  const int vpl = (a.E + 31) >> 5;
  uint32_t key[32];
#pragma unroll
  for (int v = 0; v < 32; ++v) {
    const int e = v * 32 + lane;
    key[v] = (v < vpl && e < a.E) ? ordered_key(__ldcg(L + e)) : 0u;
  }
  uint32_t taken = 0, bk = 0;
  int bv = -1;
#pragma unroll
  for (int v = 0; v < 32; ++v)
    if (key[v] > bk) { bk = key[v]; bv = v; }

  int my_idx = 0;
  float my_val = 0.f;
  for (int j = 0; j < a.K; ++j) {
    // largest value, then the lowest expert id holding it
    const uint32_t top = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t cand = (bv >= 0 && bk == top) ? (uint32_t)(bv * 32 + lane) : 0xffffffffu;
    uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    if (win >= (uint32_t)a.E) {  // no candidate left: only a NaN logit pattern can cause it
      if (lane == 0) set_error(a.ws.status, kErrBadIndex);
      win = 0;
    }
    if (lane == j) {
      my_idx = (int)win;
      my_val = key_value(top);
    }
    if ((int)(win & 31u) == lane) {
      taken |= 1u << (win >> 5);
      bk = 0;
      bv = -1;
#pragma unroll
      for (int v = 0; v < 32; ++v)
        if (!((taken >> v) & 1u) && key[v] > bk) { bk = key[v]; bv = v; }
    }
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
    s_idx[p] = my_idx;
    s_w[p] = w;
  }
}

}  // namespace

template <int CPL>
__global__ void __launch_bounds__(kRouterThreads) router_topk_compact_kernel(RouterArgs a) {
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

  pdl_wait();                // x (and the workspace) now belong to this call
  pdl_launch_dependents();   // the gate/up kernel may start its prologue

  if (has_row) {
    int m = 0;
    for (; m + 2 <= a.M; m += 2) logits_tokens<CPL, 2>(a, w, m, e, bias, lane);
    for (; m < a.M; ++m) logits_tokens<CPL, 1>(a, w, m, e, bias, lane);
  }

  // Last CTA to finish runs the top-k and the compaction.
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(a.ws.router_count, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  extern __shared__ int4 dyn_smem[];
  const int NP = a.M * a.K;
  int* s_idx = reinterpret_cast<int*>(dyn_smem);
  float* s_w = reinterpret_cast<float*>(s_idx + NP);
  int* s_cnt = reinterpret_cast<int*>(s_w + NP);
  int* s_off = s_cnt + a.E;
  int* s_run = s_off + a.E;

  for (int m = warp; m < a.M; m += kRouterThreads / 32) topk_token(a, m, lane, s_idx, s_w);
  for (int i = threadIdx.x; i < a.E; i += blockDim.x) {
    s_cnt[i] = 0;
    s_run[i] = 0;
  }
  __syncthreads();
  for (int p = threadIdx.x; p < NP; p += blockDim.x) atomicAdd(&s_cnt[s_idx[p]], 1);
  __syncthreads();

  if (warp == 0) {
    // Bucket offsets (pairs), group offsets (<= 16 pairs per group) and the
    // active-expert count: one exclusive scan over experts, lane-contiguous.
    const int E = a.E;
    const int per = (E + 31) >> 5;
    const int e0 = lane * per, e1 = min(E, e0 + per);
    int c_sum = 0, g_sum = 0, a_sum = 0;
    for (int ex = e0; ex < e1; ++ex) {
      const int c = s_cnt[ex];
      c_sum += c;
      g_sum += (c + kGroupTokens - 1) / kGroupTokens;
      a_sum += c > 0;
    }
    int c_inc = c_sum, g_inc = g_sum, a_inc = a_sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int tc = __shfl_up_sync(0xffffffffu, c_inc, o);
      const int tg = __shfl_up_sync(0xffffffffu, g_inc, o);
      const int ta = __shfl_up_sync(0xffffffffu, a_inc, o);
      if (lane >= o) {
        c_inc += tc;
        g_inc += tg;
        a_inc += ta;
      }
    }
    int c_off = c_inc - c_sum, g_off = g_inc - g_sum;
    for (int ex = e0; ex < e1; ++ex) {
      const int c = s_cnt[ex];
      s_off[ex] = c_off;
      for (int q = 0; q * kGroupTokens < c; ++q) {
        const int g = g_off + q;
        a.ws.grp_expert[g] = ex;
        a.ws.grp_start[g] = c_off + q * kGroupTokens;
        a.ws.grp_cnt[g] = min(kGroupTokens, c - q * kGroupTokens);
      }
      c_off += c;
      g_off += (c + kGroupTokens - 1) / kGroupTokens;
    }
    if (lane == 31) {
      *a.ws.n_groups = g_inc;
      *a.ws.n_active = a_inc;
    }
    __syncwarp();
    // Stable placement: position = bucket offset + pairs of the same expert
    // with a smaller pair index.
    for (int base = 0; base < NP; base += 32) {
      const int p = base + lane;
      const bool valid = p < NP;
      const int ex = valid ? s_idx[p] : E + lane;  // sentinel never matches a real expert
      const unsigned same = __match_any_sync(0xffffffffu, ex);
      const int rank = __popc(same & ((1u << lane) - 1u));
      int pos = 0;
      if (valid) pos = s_off[ex] + s_run[ex] + rank;
      __syncwarp();
      if (valid) {
        a.ws.pair_list[pos] = p;
        if (rank == 0) s_run[ex] += __popc(same);
      }
      __syncwarp();
    }
  }
  if (threadIdx.x == 0) *a.ws.router_count = 0;  // ready for the next call
}

RouterKernel router_kernel_for(int cpl) {
  switch (cpl) {
    case 1: return router_topk_compact_kernel<1>;
    case 2: return router_topk_compact_kernel<2>;
    case 4: return router_topk_compact_kernel<4>;
    case 5: return router_topk_compact_kernel<5>;
    case 8: return router_topk_compact_kernel<8>;
    case 10: return router_topk_compact_kernel<10>;
    case 12: return router_topk_compact_kernel<12>;
    case 16: return router_topk_compact_kernel<16>;
    default: return nullptr;
  }
}

}  // namespace wse
