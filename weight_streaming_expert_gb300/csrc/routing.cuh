// routing.cuh -- the router of one call: gate matvec, softmax top-k with
// renormalisation, and the token->expert compaction, as device functions
// shared by the layer kernel and the allocation-free routing kernel.
//
// Method (page "How Ling-3.0-flash reduces batch 1 decoding latency by 54%
// on 4 Blackwell GPUs"):
//  * "bf16 router gate and lm_head": the gate weight is bf16 and pure
//    bandwidth (2.6 MB per layer at hidden 2560 x 512 experts); logits and
//    the softmax are fp32.
//  * "PDL: the latency floor of stacked small kernels", Figure 7: the gate
//    weight does not depend on the producer of x, so its load is issued
//    before the dependency wait.
//  * "Two fusions and a retune" (moe_align on the pair axis): the M*k
//    (token, slot) pairs are bucketed by expert with a stable order inside a
//    bucket, and the bucket offsets never leave the device.
//
// GB300 design.
//  * Gate matvec on the tensor cores: a unit = 8 experts (n8) x 1/ks of the
//    hidden dim; its 8 warps split that slice and every warp runs m16n8k16
//    bf16 MMAs with the tokens as A (16 per pass) and the 8 weight rows as B.
//    The weight keeps the caller's [E][H] layout: inside every 32-wide k
//    chunk the MMA's logical k order is permuted so that lane (g, t) holds
//    physical k = 8t .. 8t+7 of both operands, i.e. ONE 16-byte load per
//    operand row per chunk (the same permutation on A and B leaves every dot
//    product unchanged).  Units write fp32 partial logits; the reader sums
//    the ks partials in a fixed order, so the logits are deterministic.
//    Inside the layer kernel the partial logits live in two buffers used by
//    odd and even calls; a call's units write theirs into the call's buffer
//    and set the same words of the other buffer to an "unwritten" bit
//    pattern (a NaN that no arithmetic produces).  A reader polls the words
//    it needs until none is unwritten, so no grid-wide barrier (and no flag
//    round trip) sits between the matvec and the top-k.
//  * Top-k, one warp per token: the E logits sit in registers (lane l holds
//    experts l + 32v as order-preserving integer keys).  Every lane first
//    lists its two best keys (a max/min tree, then the lowest positions
//    holding them).  A round takes the warp's best list head (redux.sync max
//    of the keys, then redux.sync min of the expert ids holding it: ties --
//    bit-equal logits -- go to the lowest id) and the winning lane shifts
//    its list; a lane that gives both of its keys refills the list with the
//    next two below the last one (rare: it holds three of the winners).
//    Weights: exp(l_j - l_0) over the k chosen, normalised by their sum
//    (= the full softmax renormalised over the k; its denominator cancels).
//  * Compaction from bit masks: an expert is chosen at most once per token,
//    so bit m of mask[e] says "token m chose e".  popc(mask[e]) is the
//    bucket size and popc(mask[e] & (2^m - 1)) the pair's stable rank in its
//    bucket -- every pair is placed independently, no serial pass.
#pragma once

#include "common.cuh"

namespace wse {

// ------------------------------------------------------- gate matvec ---
struct GemvUnit {
  int tile;  // experts [8 tile, 8 tile + 8)
  int kc;    // hidden-dim slice index, 0..ks-1
  int q0;    // first 32-wide k chunk of this warp
  int nq;    // k chunks of this warp
};

__device__ __forceinline__ GemvUnit gemv_unit(int unit, int ks, int H, int warp) {
  GemvUnit u;
  u.tile = unit / ks;
  u.kc = unit - u.tile * ks;
  const int per_unit = (H / 32) / ks;
  u.nq = per_unit / kConsumerWarps;
  u.q0 = u.kc * per_unit + warp * u.nq;
  return u;
}

// B fragments of this warp's slice (rows past E repeat the last row; their
// results are never stored).  KPW = H / 256 >= nq.
template <int KPW>
__device__ __forceinline__ void gemv_load_w(const __nv_bfloat16* __restrict__ w_router, int E, int H,
                                            const GemvUnit& u, int lane, uint4 (&b)[KPW]) {
  const int row = min(u.tile * 8 + (lane >> 2), E - 1);
  const uint4* src = reinterpret_cast<const uint4*>(w_router + (size_t)row * H) + (lane & 3);
#pragma unroll
  for (int q = 0; q < KPW; ++q)
    if (q < u.nq) b[q] = __ldg(src + 4 * (u.q0 + q));
}

// This warp's partial (tokens 16 mb + g, 16 mb + g + 8) x (experts 2t, 2t+1
// of the tile) over its k slice, as (c0, c1, c2, c3) of the m16n8 C tile.
template <int KPW>
__device__ __forceinline__ float4 gemv_tokens(const __nv_bfloat16* __restrict__ x, int M, int H,
                                              const GemvUnit& u, int mb, int lane,
                                              const uint4 (&b)[KPW]) {
  const int g4 = lane >> 2, t4 = lane & 3;
  const int m0 = min(mb * 16 + g4, M - 1), m1 = min(mb * 16 + g4 + 8, M - 1);
  const uint4* x0 = reinterpret_cast<const uint4*>(x + (size_t)m0 * H) + t4;
  const uint4* x1 = reinterpret_cast<const uint4*>(x + (size_t)m1 * H) + t4;
  float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int q = 0; q < KPW; ++q) {
    if (q < u.nq) {
      const uint4 xa = x0[4 * (u.q0 + q)], xb = x1[4 * (u.q0 + q)];
      // logical k (2t, 2t+1 | 2t+8, 2t+9) of step 0 = physical 8t + (0,1 | 2,3);
      // step 1 takes physical 8t + (4,5 | 6,7)
      mma_bf16(c0, xa.x, xb.x, xa.y, xb.y, b[q].x, b[q].y);
      mma_bf16(c1, xa.z, xb.z, xa.w, xb.w, b[q].z, b[q].w);
    }
  }
  return make_float4(c0[0] + c1[0], c0[1] + c1[1], c0[2] + c1[2], c0[3] + c1[3]);
}

// A partial logit that is not written yet (never produced by arithmetic:
// the hardware's NaN results are positive).
constexpr uint32_t kUnwritten = 0xffffffffu;

// One partial logit: a plain store (read after a fence and a counter), or a
// relaxed gpu-scope store (read by other CTAs polling the word).
template <bool kPolled>
__device__ __forceinline__ void put_logit(float* P, size_t i, float v) {
  if constexpr (kPolled)
    asm volatile("st.relaxed.gpu.global.f32 [%0], %1;" ::"l"(P + i), "f"(v) : "memory");
  else
    P[i] = v;
}

// Warp 0 of the unit's CTA: sum the 8 warp partials in warp order and store
// the unit's fp32 partial logits part[kc][m][e] (plane = rows * E floats).
template <bool kPolled = false>
__device__ __forceinline__ void gemv_store(const float4* red, const GemvUnit& u, int mb, int M, int E,
                                           size_t plane, float* __restrict__ part, int lane) {
  float4 s = red[lane];
#pragma unroll
  for (int w = 1; w < kConsumerWarps; ++w) {
    const float4 v = red[w * 32 + lane];
    s.x += v.x;
    s.y += v.y;
    s.z += v.z;
    s.w += v.w;
  }
  const int e = u.tile * 8 + 2 * (lane & 3);
  const int m0 = mb * 16 + (lane >> 2), m1 = m0 + 8;
  float* P = part + (size_t)u.kc * plane;
  if (m0 < M) {
    if (e < E) put_logit<kPolled>(P, (size_t)m0 * E + e, s.x);
    if (e + 1 < E) put_logit<kPolled>(P, (size_t)m0 * E + e + 1, s.y);
  }
  if (m1 < M) {
    if (e < E) put_logit<kPolled>(P, (size_t)m1 * E + e, s.z);
    if (e + 1 < E) put_logit<kPolled>(P, (size_t)m1 * E + e + 1, s.w);
  }
}

// One warp: mark the unit's words of ALL rows (tokens) of the other
// buffer unwritten, ready for the next call (whatever its M).
__device__ __forceinline__ void gemv_clear(const GemvUnit& u, int rows, int E, size_t plane,
                                           float* __restrict__ part, int lane) {
  float* P = part + (size_t)u.kc * plane + u.tile * 8;
  const int n = min(8, E - u.tile * 8);
  for (int i = lane; i < rows * 8; i += 32) {
    const int m = i >> 3, c = i & 7;
    if (c < n) P[(size_t)m * E + c] = __uint_as_float(kUnwritten);
  }
}

// Largest divisor ks of H/256 with ceil(E/8) * ks <= units_max (>= 1).
__host__ __device__ inline int gemv_split(int H, int E, int units_max) {
  const int kpw = H / 256, tiles = (E + 7) / 8;
  int best = 1;
  for (int ks = 1; ks <= kpw; ++ks)
    if (kpw % ks == 0 && tiles * ks <= units_max) best = ks;
  return best;
}

// ------------------------------------------------------------ top-k ----
// Order-preserving map of a float to an unsigned key (larger float ->
// larger key).  Key 0 marks "taken / no expert"; every float maps to >= 1
// (only two NaN encodings share key 1), so a candidate always remains
// while fewer than E experts have been taken.
__device__ __forceinline__ uint32_t ordered_key(float v) {
  const uint32_t u = __float_as_uint(v);
  const uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return k > 1u ? k : 1u;
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// The two best keys of key[0..VPL) strictly below (lk, lv) in the order
// (key desc, position asc), with the lowest positions holding them; a
// missing entry is (0, VPL).  A max/min tree finds the keys (no
// predicates: the dependent chain is short), match masks their positions.
template <int VPL>
__device__ __forceinline__ void top2_below(const uint32_t (&key)[VPL], uint32_t lk, int lv, uint32_t& k1,
                                           int& v1, uint32_t& k2, int& v2) {
  uint32_t kf[VPL];
#pragma unroll
  for (int v = 0; v < VPL; ++v) kf[v] = (key[v] < lk || (key[v] == lk && v > lv)) ? key[v] : 0u;
  uint32_t hi[VPL > 1 ? VPL / 2 : 1], lo[VPL > 1 ? VPL / 2 : 1];
  if constexpr (VPL == 1) {
    hi[0] = kf[0];
    lo[0] = 0u;
  } else {
#pragma unroll
    for (int i = 0; i < VPL / 2; ++i) {
      hi[i] = max(kf[2 * i], kf[2 * i + 1]);
      lo[i] = min(kf[2 * i], kf[2 * i + 1]);
    }
    // merging two (best, second) pairs: best of the bests; second = the
    // better of the losing best and the two seconds
#pragma unroll
    for (int s = 1; s < VPL / 2; s <<= 1) {
#pragma unroll
      for (int i = 0; i + s < VPL / 2; i += 2 * s) {
        const uint32_t h = max(hi[i], hi[i + s]);
        lo[i] = max(min(hi[i], hi[i + s]), max(lo[i], lo[i + s]));
        hi[i] = h;
      }
    }
  }
  k1 = hi[0];
  k2 = lo[0];
  uint32_t m1 = 0u, m2 = 0u;
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    m1 |= (kf[v] == k1 ? 1u : 0u) << v;
    m2 |= (kf[v] == k2 ? 1u : 0u) << v;
  }
  v1 = __ffs(m1) - 1;
  if (k2 == k1) m2 &= m2 - 1u;  // the same key twice: its second position
  v2 = k2 == 0u ? VPL : __ffs(m2) - 1;
}

// Sources of one token's partial logits (ks planes, `plane` words apart).
// sum(): lane l gets the fp32 sum over the planes, in plane order, of the
// logits of experts l + 32 v (0 past E).  one(): the same sum for one expert.
struct PlainPlanes {  // fp32 words, complete before the reader starts
  const float* lg;
  size_t plane;
  template <int VPL>
  __device__ __forceinline__ void sum(int lane, int E, int ks, float (&lv)[VPL], int*) const {
    float l1[VPL];  // planes 0 and 1 in one round trip, further planes one each
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      const int e = v * 32 + lane;
      lv[v] = e < E ? __ldcg(lg + e) : 0.f;
      l1[v] = (ks > 1 && e < E) ? __ldcg(lg + plane + e) : 0.f;
    }
    if (ks > 1) {
#pragma unroll
      for (int v = 0; v < VPL; ++v) lv[v] += l1[v];
    }
    for (int c = 2; c < ks; ++c) {
      float pv[VPL];
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        const int e = v * 32 + lane;
        pv[v] = e < E ? __ldcg(lg + (size_t)c * plane + e) : 0.f;
      }
#pragma unroll
      for (int v = 0; v < VPL; ++v) lv[v] += pv[v];
    }
  }
  __device__ __forceinline__ float one(int e, int ks) const {
    float l = __ldcg(lg + e);
    for (int c = 1; c < ks; ++c) l += __ldcg(lg + (size_t)c * plane + e);
    return l;
  }
};

__device__ __forceinline__ uint32_t ld_relaxed32(const float* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Words written by other CTAs of the same call while this warp reads them:
// every word still unwritten is re-read until none is (bounded: after
// `limit` ns the status gets kErrTimeoutGrid and the call's result is
// undefined).  Planes 0 and 1 are polled together, further planes one each.
struct PolledPlanes {
  const float* lg;
  size_t plane;
  unsigned long long limit;
  template <int VPL>
  __device__ __forceinline__ void poll(const float* P, const float* Q, int lane, int E, uint32_t (&w0)[VPL],
                                       uint32_t (&w1)[VPL], int* status) const {
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      const int e = v * 32 + lane;
      w0[v] = e < E ? ld_relaxed32(P + e) : 0u;
      w1[v] = (Q && e < E) ? ld_relaxed32(Q + e) : 0u;
    }
    unsigned long long t0 = 0ull;
    for (int it = 0;; ++it) {
      bool ok = true;
#pragma unroll
      for (int v = 0; v < VPL; ++v) ok = ok && w0[v] != kUnwritten && w1[v] != kUnwritten;
      if (__all_sync(0xffffffffu, ok)) return;
      if (it == 0) {
        t0 = global_timer_ns();
      } else if (global_timer_ns() - t0 > limit) {
        if (lane == 0) set_error(status, kErrTimeoutGrid);
        return;
      }
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        const int e = v * 32 + lane;
        if (w0[v] == kUnwritten) w0[v] = ld_relaxed32(P + e);
        if (w1[v] == kUnwritten) w1[v] = ld_relaxed32(Q + e);
      }
    }
  }
  template <int VPL>
  __device__ __forceinline__ void sum(int lane, int E, int ks, float (&lv)[VPL], int* status) const {
    uint32_t w0[VPL], w1[VPL];
    poll<VPL>(lg, ks > 1 ? lg + plane : nullptr, lane, E, w0, w1, status);
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      lv[v] = __uint_as_float(w0[v]);  // 0 past E
      if (ks > 1) lv[v] += __uint_as_float(w1[v]);
    }
    for (int c = 2; c < ks; ++c) {
      poll<VPL>(lg + (size_t)c * plane, nullptr, lane, E, w0, w1, status);
#pragma unroll
      for (int v = 0; v < VPL; ++v) lv[v] += __uint_as_float(w0[v]);
    }
  }
  __device__ __forceinline__ float one(int e, int ks) const {  // words already seen written
    float l = __uint_as_float(ld_relaxed32(lg + e));
    for (int c = 1; c < ks; ++c) l += __uint_as_float(ld_relaxed32(lg + (size_t)c * plane + e));
    return l;
  }
};

// Top-k of one token by one warp.  src: the token's partial logits, summed
// in plane order, plus the bias.
// Lane j < K writes slot j's expert id to idx_out[j] (the caller reads them
// after a __syncwarp) and returns slot j's renormalised weight; the other
// lanes return 0.  sel_only: the bias picks the experts only, the weights
// come from the unbiased logits (re-read for the k chosen experts).
template <int VPL, class Src>
__device__ __forceinline__ float topk_token(const Src& src, int ks, const float* __restrict__ bias, int E, int K,
                                            int lane, int* status, int* idx_out, bool sel_only) {
  float lv[VPL], bv_[VPL];
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = v * 32 + lane;
    bv_[v] = (bias && e < E) ? __ldg(bias + e) : 0.f;
  }
  src.template sum<VPL>(lane, E, ks, lv, status);
  uint32_t key[VPL];
#pragma unroll
  for (int v = 0; v < VPL; ++v) {
    const int e = v * 32 + lane;
    if (bias) lv[v] += bv_[v];
    key[v] = e < E ? ordered_key(lv[v]) : 0u;
  }
  uint32_t k1, k2;
  int v1, v2;
  top2_below<VPL>(key, 0xffffffffu, -1, k1, v1, k2, v2);

  uint32_t my_key = 0u, my_win = 0u, top0 = 0u;
  for (int j = 0; j < K; ++j) {
    const uint32_t top = __reduce_max_sync(0xffffffffu, k1);
    const uint32_t cand = (k1 == top) ? (uint32_t)(v1 * 32 + lane) : 0xffffffffu;
    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    top0 = j == 0 ? top : top0;
    my_key = lane == j ? top : my_key;
    my_win = lane == j ? win : my_win;
    const bool mine = (int)(win & 31u) == lane;
    const uint32_t gk = k1;
    const int gv = v1;
    k1 = mine ? k2 : k1;
    v1 = mine ? v2 : v1;
    k2 = mine ? 0u : k2;
    v2 = mine ? VPL : v2;
    if (mine && v1 >= VPL && j + 1 < K) top2_below<VPL>(key, gk, gv, k1, v1, k2, v2);
  }
  if (lane < K) {
    if (my_key == 0u || my_win >= (uint32_t)E) {  // unreachable while K <= E
      set_error(status, kErrBadIndex);
      my_win = 0u;
    }
    idx_out[lane] = (int)my_win;
  }
  // weights: exp(l_j - l_0), normalised by a fixed butterfly sum over the
  // lanes that hold one (lanes >= K add 0)
  float my_val = key_value(my_key), ref_val = key_value(top0);
  if (sel_only && bias) {  // the unbiased logits of the chosen, summed as above
    float l = 0.f;
    if (lane < K) l = src.one((int)my_win, ks);
    my_val = l;
    ref_val = key_value(__reduce_max_sync(0xffffffffu, lane < K ? ordered_key(l) : 0u));
  }
  const float ex = lane < K ? expf(my_val - ref_val) : 0.f;
  float s = ex;
  for (int o = 1; o < K; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return lane < K ? __fdividef(ex, s) : 0.f;
}

template <class Src>
__device__ __forceinline__ float topk_dispatch(const Src& src, int ks, const float* bias, int E, int K, int lane,
                                               int* status, int* idx_out, bool sel_only = false) {
  if (E <= 32) return topk_token<1>(src, ks, bias, E, K, lane, status, idx_out, sel_only);
  if (E <= 64) return topk_token<2>(src, ks, bias, E, K, lane, status, idx_out, sel_only);
  if (E <= 128) return topk_token<4>(src, ks, bias, E, K, lane, status, idx_out, sel_only);
  if (E <= 256) return topk_token<8>(src, ks, bias, E, K, lane, status, idx_out, sel_only);
  if (E <= 512) return topk_token<16>(src, ks, bias, E, K, lane, status, idx_out, sel_only);
  return topk_token<32>(src, ks, bias, E, K, lane, status, idx_out, sel_only);
}

// ------------------------------------------------------- compaction ----
// Shared-memory routing of one call (ints unless noted):
//   mask[E] (u64)  s_off[E]  s_e[NP]  s_w[NP] (float)  pair_list[NP]
//   grp_expert[NP]  grp_start[NP]  grp_cnt[NP]  scal[96]
//   bits[kChunkLevels][kBitWords] (u32)  pre[kBitWords + 1]
// (the compaction comment in the header says how the positions are found).
// bits and pre number the groups without the compaction, for the warp that
// starts the weight copies while the other warps compact: bit e % 32 of
// bits[q][e / 32] says expert e's bucket holds more than 16 q pairs (its
// group q exists) -- the top-k sets it with the atomic OR that adds the
// (16 q + 1)-th member, since each OR returns the members before it and
// exactly one sees 16 q of them; pre[w] counts the groups of the experts
// below 32 w.  Groups run in ascending (expert, q) order, as in the
// compaction.
constexpr int kBitWords = (kMaxExperts + 1 + 31) / 32;  // routed experts + a shared one
constexpr int kChunkLevels = kMaxTokens / kGroupTokens;
static_assert(kMaxTokens % kGroupTokens == 0 && kMaxTokens <= 64, "u64 token masks in 16-token groups");

__host__ __device__ inline size_t routing_smem_bytes(int NP, int E) {
  return (size_t)E * 8 + (size_t)E * 4 + (size_t)NP * 4 * 6 + 96 * 4 + (size_t)kChunkLevels * kBitWords * 4 +
         (kBitWords + 1) * 4;
}

struct SmemRouting {
  unsigned long long* mask;
  int* s_off;
  int* s_e;         // [NP] expert of pair p = token * K + slot
  float* s_w;       // [NP] routing weight of pair p
  int* pair_list;   // [NP] pair id at each sorted position
  int* grp_expert;  // [groups] expert of each group (ascending expert id)
  int* grp_start;   // [groups] first sorted position
  int* grp_cnt;     // [groups] pairs in the group (1..16)
  int* scal;        // [0] groups, [1] distinct experts, [8..88) scan scratch
  unsigned* bits;   // [kChunkLevels][kBitWords] groups that exist, by expert
  int* pre;         // [kBitWords + 1] groups below each word of experts
};

__device__ __forceinline__ SmemRouting routing_carve(uint8_t* base, int NP, int E) {
  SmemRouting r;
  r.mask = reinterpret_cast<unsigned long long*>(base);
  r.s_off = reinterpret_cast<int*>(r.mask + E);
  r.s_e = r.s_off + E;
  r.s_w = reinterpret_cast<float*>(r.s_e + NP);
  r.pair_list = reinterpret_cast<int*>(r.s_w + NP);
  r.grp_expert = r.pair_list + NP;
  r.grp_start = r.grp_expert + NP;
  r.grp_cnt = r.grp_start + NP;
  r.scal = r.grp_cnt + NP;
  r.bits = reinterpret_cast<unsigned*>(r.scal + 96);
  r.pre = reinterpret_cast<int*>(r.bits + kChunkLevels * kBitWords);
  return r;
}

// Add pair (token m, expert e) to the buckets (any thread, any order).
// kNarrow: 32-bit atomics only, a count in s_off[e] (zeroed beforehand;
// the compaction overwrites it) and the mask's 32-bit half -- two atomics
// that serialise less on a hot expert than one 64-bit OR (measured: faster
// from 16 tokens, slower at 6).
template <bool kNarrow = false>
__device__ __forceinline__ void bucket_add(const SmemRouting& r, int e, int m) {
  int before;
  if constexpr (kNarrow) {
    before = atomicAdd(&r.s_off[e], 1);
    atomicOr(reinterpret_cast<unsigned*>(r.mask) + 2 * e + (m >> 5), 1u << (m & 31));
  } else {
    before = __popcll(atomicOr(&r.mask[e], 1ull << m));
  }
  if ((before & (kGroupTokens - 1)) == 0)
    atomicOr(&r.bits[(before / kGroupTokens) * kBitWords + (e >> 5)], 1u << (e & 31));
}

// One warp, after the buckets are complete: pre[] and the group count
// (returned to every lane); levels = chunk levels in use, ceil(M / 16).
// Lane l counts word l (and 32 + l), a five-step scan places them.
__device__ __forceinline__ int count_groups(const SmemRouting& r, int EA, int levels, int lane) {
  const int nw = (EA + 31) / 32;
  int base = 0;
  for (int w0 = 0; w0 < nw; w0 += 32) {  // one pass unless EA > 1024 (a shared expert beside 1024)
    const int w = w0 + lane;
    int c = 0;
    if (w < nw)
      for (int q = 0; q < levels; ++q) c += __popc(r.bits[q * kBitWords + w]);
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (w < nw) r.pre[w] = base + inc - c;
    base += __shfl_sync(0xffffffffu, inc, 31);
  }
  if (lane == 0) r.pre[nw] = base;
  __syncwarp();
  return base;
}

// Position of the n-th (0-based) set bit of a 32-bit word with more than n.
__device__ __forceinline__ int nth_set_bit32(unsigned w, int n) {
  int pos = 0;
#pragma unroll
  for (int b = 16; b >= 1; b >>= 1) {
    const int c = __popc(w & ((1u << b) - 1u));
    if (n >= c) {
      n -= c;
      w >>= b;
      pos += b;
    }
  }
  return pos;
}

// Expert of group g (< the group count; nw words of experts).  `w` is a
// cursor: the word of the previous lookup (start at 0).  The word comes from
// a binary search of pre (lookups with ascending g usually stay in the
// cursor's word), the expert inside it from a binary search of the groups
// below each bit position, in registers.
__device__ __forceinline__ int group_expert(const SmemRouting& r, int g, int levels, int nw, int& w) {
  if (g < r.pre[w]) w = 0;
  if (r.pre[w + 1] <= g) {  // largest w' in (w, nw) with pre[w'] <= g
    int lo = w + 1, hi = nw - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (r.pre[mid] <= g) lo = mid;
      else hi = mid - 1;
    }
    w = lo;
  }
  const int j = g - r.pre[w];
  if (levels == 1) return 32 * w + nth_set_bit32(r.bits[w], j);
  unsigned B[kChunkLevels];
#pragma unroll
  for (int q = 0; q < kChunkLevels; ++q) B[q] = q < levels ? r.bits[q * kBitWords + w] : 0u;
  auto P = [&](int x) {  // groups of the word's experts below bit x
    const unsigned m = (1u << x) - 1u;
    int n = 0;
#pragma unroll
    for (int q = 0; q < kChunkLevels; ++q) n += __popc(B[q] & m);
    return n;
  };
  int b = 0;  // the largest bit b with P(b) <= j: its expert holds group g
#pragma unroll
  for (int step = 16; step >= 1; step >>= 1)
    if (b + step <= 31 && P(b + step) <= j) b += step;
  return 32 * w + b;
}

// Barrier of the nt threads that run a compaction: the whole CTA, or the
// consumer and publisher warps (named barrier 3) while the producer warp
// streams.
__device__ __forceinline__ void routing_sync(int nt) {
  if (nt == (int)blockDim.x)
    __syncthreads();
  else
    asm volatile("bar.sync 3, %0;" ::"r"(nt) : "memory");
}

// Token of pair p: routed pairs p = token * K + slot come first (MK = M * K
// of them), then the shared expert's pairs MK + token.
__device__ __forceinline__ int pair_token(int p, int K, int MK) { return p < MK ? p / K : p - MK; }

// Cooperative over threads tid = 0 .. nt - 1 (the CTA, or the warps that
// routing_sync counts); mask[] and s_e[] complete and visible (a barrier
// before).  Bucket sizes and group counts by a scan over the experts; every
// pair then takes its place independently.  NP pairs (MK routed, see
// pair_token).  Ends with a barrier.
__device__ inline void compact_masks(const SmemRouting& r, int NP, int K, int MK, int E, int tid, int nt) {
  // (pairs << 16) + groups share one int (both <= 2048, no carry)
  const int lane = tid & 31, warp = tid >> 5, nwarps = nt >> 5;
  int* s_wt = r.scal + 8;
  int* s_wa = r.scal + 48;
  const int per = (E + nt - 1) / nt;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int packed = 0, act = 0;
  for (int e = e0; e < e1; ++e) {
    const int c = __popcll(r.mask[e]);
    packed += (c << 16) + (c + kGroupTokens - 1) / kGroupTokens;
    act += c > 0;
  }
  int inc = packed, ainc = act;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    const int ta = __shfl_up_sync(0xffffffffu, ainc, o);
    if (lane >= o) {
      inc += t;
      ainc += ta;
    }
  }
  if (lane == 31) {
    s_wt[warp] = inc;
    s_wa[warp] = ainc;
  }
  routing_sync(nt);
  if (warp == 0) {
    int v = lane < nwarps ? s_wt[lane] : 0;
    int va = lane < nwarps ? s_wa[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, v, o);
      const int ta = __shfl_up_sync(0xffffffffu, va, o);
      if (lane >= o) {
        v += t;
        va += ta;
      }
    }
    if (lane < nwarps) {
      s_wt[lane] = v;
      s_wa[lane] = va;
    }
    if (lane == nwarps - 1) {
      r.scal[0] = v & 0xffff;
      r.scal[1] = va;
    }
  }
  routing_sync(nt);
  {
    const int base = (warp > 0 ? s_wt[warp - 1] : 0) + inc - packed;
    int c_off = base >> 16, g_off = base & 0xffff;
    for (int e = e0; e < e1; ++e) {
      const int c = __popcll(r.mask[e]);
      r.s_off[e] = c_off;
      for (int q = 0; q * kGroupTokens < c; ++q) {
        const int g = g_off + q;
        r.grp_expert[g] = e;
        r.grp_start[g] = c_off + q * kGroupTokens;
        r.grp_cnt[g] = min(kGroupTokens, c - q * kGroupTokens);
      }
      c_off += c;
      g_off += (c + kGroupTokens - 1) / kGroupTokens;
    }
  }
  routing_sync(nt);
  for (int p = tid; p < NP; p += nt) {
    const int e = r.s_e[p], m = pair_token(p, K, MK);
    const int rank = __popcll(r.mask[e] & ((1ull << m) - 1ull));
    r.pair_list[r.s_off[e] + rank] = p;
  }
  routing_sync(nt);
}

// M <= kGroupTokens: every expert's bucket holds at most M <= 16 pairs, so
// it is exactly one group, and the groups are the chosen experts in
// ascending id (the same result as compact_masks).  Worked out on the pair
// axis ("Two fusions and a retune": moe_align compares pairs instead of
// scanning experts): pair p with expert e goes to
//   position = #{q : e_q < e} + #{q < p : e_q = e},
// and the pair of e with the lowest token opens e's group, numbered by the
// group openers with a smaller expert.  Two short loops over the NP pairs
// per thread (the code stays small: it runs once per call, cold), no scan.
// NP pairs (MK routed, see pair_token).  ekey: NP ints of scratch.
// Cooperative over threads t = 0 .. nt - 1 (see routing_sync); mask[] and
// s_e[] complete and visible (a barrier before); scal[0] zero.  Ends with a
// barrier; returns the group count.
__device__ inline int compact_pairs(const SmemRouting& r, int NP, int K, int MK, int* ekey, int t, int nt) {
  for (int p = t; p < NP; p += nt) {
    const int e = r.s_e[p], m = pair_token(p, K, MK);
    ekey[p] = (e << 1) | ((r.mask[e] & ((1ull << m) - 1ull)) == 0ull ? 1 : 0);
  }
  routing_sync(nt);
  for (int p = t; p < NP; p += nt) {
    const int ek = ekey[p], e = ek >> 1;
    int below = 0, open_below = 0, same_before = 0;
    for (int q = 0; q < NP; ++q) {
      const int f = ekey[q];
      const int lt = (f >> 1) < e ? 1 : 0;
      below += lt;
      open_below += lt & f;
      same_before += ((f >> 1) == e && q < p) ? 1 : 0;
    }
    r.pair_list[below + same_before] = p;
    if (ek & 1) {
      r.grp_expert[open_below] = e;
      r.grp_start[open_below] = below;
      r.grp_cnt[open_below] = __popcll(r.mask[e]);
      atomicAdd(&r.scal[0], 1);
    }
  }
  routing_sync(nt);
  const int n_groups = r.scal[0];
  if (t == 0) r.scal[1] = n_groups;
  return n_groups;
}

}  // namespace wse
