// compaction.cuh -- token->expert compaction of one call's routing, built in
// shared memory by every CTA of the expert kernels.
//
// "Two fusions and a retune" (moe_align on the pair axis): the M*k (token,
// slot) pairs are bucketed by expert; each pair's rank inside its bucket is
// stable in pair index; bucket populations give bucket-ordered offsets and
// the published total.  Nothing is read back to the host.
//
// GB300 design: the router's last CTA builds the buckets block-wide in
// shared memory -- a shared-memory histogram, one block-wide scan over the
// experts, a stable rank from __match_any_sync over 32-pair chunks -- and
// publishes them; every CTA of the expert kernels then loads the published
// list into its own shared memory with one coalesced read (load_routing).
#pragma once

#include "common.cuh"

namespace wse {

// Shared-memory layout of the compaction (ints):
//   s_e[NP] s_cnt[E] s_off[E] s_goff[E] s_run[E]
//   grp_expert[NP] grp_start[NP] grp_cnt[NP] pair_list[NP]   + 8 scalars
__host__ __device__ inline size_t compaction_smem_ints(int NP, int E) {
  return (size_t)5 * NP + (size_t)4 * E + 72;
}

struct SmemRouting {
  int* grp_expert;  // [n_groups] expert of each group (ascending expert id)
  int* grp_start;   // [n_groups] first sorted position
  int* grp_cnt;     // [n_groups] pairs in the group (1..16)
  int* pair_list;   // [NP] pair id (token*k + slot) at each sorted position
  int n_groups;
  int n_active;
};

// Cooperative over all threads of the CTA.  topk_idx: [NP] expert ids in
// global memory, final and visible to this CTA.  Returns with the routing in
// shared memory and a __syncthreads() done.
__device__ inline SmemRouting compact_routing(const int32_t* __restrict__ topk_idx, int NP, int E,
                                              int* smem_ints, int* status) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nt >> 5;
  int* s_e = smem_ints;
  int* s_cnt = s_e + NP;
  int* s_off = s_cnt + E;
  int* s_goff = s_off + E;
  int* s_run = s_goff + E;
  SmemRouting r;
  r.grp_expert = s_run + E;
  r.grp_start = r.grp_expert + NP;
  r.grp_cnt = r.grp_start + NP;
  r.pair_list = r.grp_cnt + NP;
  // [0] n_groups, [1] n_active, [8..40) warp pair/group totals, [40..72) warp active totals
  int* s_scal = r.pair_list + NP;

  for (int i = tid; i < E; i += nt) {
    s_cnt[i] = 0;
    s_run[i] = 0;
  }
  for (int p = tid; p < NP; p += nt) {
    int e = __ldcg(topk_idx + p);
    if (e < 0 || e >= E) {
      set_error(status, kErrBadIndex);
      e = 0;
    }
    s_e[p] = e;
  }
  __syncthreads();
  for (int p = tid; p < NP; p += nt) atomicAdd(&s_cnt[s_e[p]], 1);
  __syncthreads();

  // Block-wide exclusive scan over experts of (pairs, groups): both totals
  // are <= NP <= 2048, so they share one int (pairs in bits 16..31, groups in
  // bits 0..15) without carries; active experts are scanned alongside.
  const int per = (E + nt - 1) / nt;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int packed = 0, act = 0;
  for (int e = e0; e < e1; ++e) {
    const int c = s_cnt[e];
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
  int* s_wt = s_scal + 8;   // per-warp packed totals
  int* s_wa = s_scal + 40;  // per-warp active totals
  if (lane == 31) {
    s_wt[warp] = inc;
    s_wa[warp] = ainc;
  }
  __syncthreads();
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
      s_wt[lane] = v;  // inclusive
      s_wa[lane] = va;
    }
    if (lane == nwarps - 1) {
      s_scal[0] = v & 0xffff;  // groups
      s_scal[1] = va;
    }
  }
  __syncthreads();
  {
    int base = (warp > 0 ? s_wt[warp - 1] : 0) + inc - packed;  // exclusive prefix
    int c_off = base >> 16, g_off = base & 0xffff;
    for (int e = e0; e < e1; ++e) {
      const int c = s_cnt[e];
      s_off[e] = c_off;
      s_goff[e] = g_off;
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
  __syncthreads();
  if (warp == 0) {
    // stable placement: pairs of the same expert keep pair-index order
    for (int base = 0; base < NP; base += 32) {
      const int p = base + lane;
      const bool valid = p < NP;
      const int ex = valid ? s_e[p] : E + lane;  // sentinel never matches a real expert
      const unsigned same = __match_any_sync(0xffffffffu, ex);
      const int rank = __popc(same & ((1u << lane) - 1u));
      int pos = 0;
      if (valid) pos = s_off[ex] + s_run[ex] + rank;
      __syncwarp();
      if (valid) {
        r.pair_list[pos] = p;
        if (rank == 0) s_run[ex] += __popc(same);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  r.n_groups = s_scal[0];
  r.n_active = s_scal[1];
  return r;
}

// Publish a shared-memory compaction to the workspace (cooperative).
__device__ inline void publish_routing(const SmemRouting& r, int NP, const Workspace& ws) {
  for (int i = threadIdx.x; i < NP; i += blockDim.x) {
    ws.pair_list[i] = r.pair_list[i];
    if (i < r.n_groups) {
      ws.grp_expert[i] = r.grp_expert[i];
      ws.grp_start[i] = r.grp_start[i];
      ws.grp_cnt[i] = r.grp_cnt[i];
    }
  }
  if (threadIdx.x == 0) {
    *ws.n_groups = r.n_groups;
    *ws.n_active = r.n_active;
  }
}

// Shared-memory layout of a loaded compaction (ints): grp_expert[NP]
// grp_start[NP] grp_cnt[NP] pair_list[NP] + 8 scalars.
__host__ __device__ inline size_t routing_smem_ints(int NP) { return (size_t)4 * NP + 8; }

// Load the published compaction into shared memory (cooperative, one
// coalesced round trip; L2-coherent loads).  Out-of-range values are clamped
// and flagged.  Ends with __syncthreads().
__device__ inline SmemRouting load_routing(const Workspace& ws, int NP, int E, int* smem_ints) {
  SmemRouting r;
  r.grp_expert = smem_ints;
  r.grp_start = r.grp_expert + NP;
  r.grp_cnt = r.grp_start + NP;
  r.pair_list = r.grp_cnt + NP;
  int* s_scal = r.pair_list + NP;
  int ng = __ldcg(ws.n_groups);
  if (ng < 0 || ng > NP) {
    if (threadIdx.x == 0) set_error(ws.status, kErrBadIndex);
    ng = 0;
  }
  for (int i = threadIdx.x; i < NP; i += blockDim.x) {
    int p = __ldcg(ws.pair_list + i);
    if (p < 0 || p >= NP) { set_error(ws.status, kErrBadIndex); p = 0; }
    r.pair_list[i] = p;
    if (i < ng) {
      int e = __ldcg(ws.grp_expert + i), st = __ldcg(ws.grp_start + i), c = __ldcg(ws.grp_cnt + i);
      if (e < 0 || e >= E || c < 1 || c > kGroupTokens || st < 0 || st + c > NP) {
        set_error(ws.status, kErrBadIndex);
        e = 0; st = 0; c = 1;
      }
      r.grp_expert[i] = e;
      r.grp_start[i] = st;
      r.grp_cnt[i] = c;
    }
  }
  if (threadIdx.x == 0) s_scal[0] = ng;
  __syncthreads();
  r.n_groups = s_scal[0];
  r.n_active = 0;
  return r;
}

}  // namespace wse
