// expert_gateup.cu -- fused gate/up GEMV + SwiGLU over the activated experts.
//
// Method (page "How Ling-3.0-flash reduces batch 1 decoding latency by 54%
// on 4 Blackwell GPUs"):
//  * "Two kinds of idle": what is left on the critical path at batch 1 is
//    the cold read of the activated expert weights (~94 MB per layer per
//    step on the post's 4-GPU split) plus the launch floor;
//  * "Economics of speculation at batch 1": verifying several tokens reads
//    the same weights as verifying one -- so each activated expert's [2I, H]
//    weight is streamed from HBM exactly once for all of its tokens;
//  * "Two fusions and a retune" (SwiGLU in the up-GEMM epilogue): silu(gate)
//    * up is folded into the up-projection epilogue, evaluated in float with
//    one final rounding to bf16, and a per-expert row interleave applied at
//    weight load puts each gate row next to its up row in the same output
//    tile (bitwise neutral: every output column is an independent dot).
//
// GB300 design.
//  * Work: the (expert, <=16-token group) list the router published, loaded
//    into shared memory by every CTA (compaction.cuh), times
//    2I/8 tiles of 8 weight rows (4 gate rows interleaved with their 4 up
//    rows) x the full hidden dim (40 KB at H = 2560).  The flat tile range
//    is split evenly over a persistent grid of one CTA per SM; the count is
//    known only on the device, never on the host.
//  * Streaming: one producer thread moves each tile HBM -> shared memory with
//    bulk (TMA) copies into a ring of stages guarded by mbarriers, so up to
//    (stages x 40 KB) per SM are in flight independent of the math warps.
//  * Math: mma.sync m16n8k16 bf16 -> fp32 with the group's tokens as the A
//    operand (m16 = up to 16 tokens) and the 8 weight rows as B (n8).  The
//    eight consumer warps split the hidden (K) dimension; each keeps its
//    slice of the tokens' A fragments in registers for the whole group, so
//    per tile it only reads its 1/8 of the staged weights (one 16-byte
//    shared load per 32 k).  Weights were re-laid out at create so that each
//    lane's 16 bytes ARE its B fragments for two k-steps (conflict-free).
//  * Epilogue: the eight partial 16x8 tiles are summed in a fixed order
//    (deterministic) by a rotating reducer warp, which applies SwiGLU in
//    fp32 and rounds once to bf16.  The accumulator pairs (col 2t, 2t+1)
//    are (gate r, up r) thanks to the interleave, so no data moves.
//  * Every wait is bounded; a timeout sets a sticky error bit and the CTA
//    leaves its loop.
#include "compaction.cuh"
#include "kernels.cuh"

namespace wse {

namespace {

constexpr int kRedSlots = 8;  // == kConsumerWarps; must exceed the ring depth
constexpr size_t kRedOff = 256;
constexpr size_t kRedBytes = (size_t)kRedSlots * kConsumerWarps * 32 * sizeof(float4);
constexpr size_t kRingOff = kRedOff + kRedBytes;
static_assert((2 * kMaxGateUpStages + kRedSlots) * 8 <= kRedOff, "barrier area");
static_assert(kMaxGateUpStages < kRedSlots, "reduction slots must outnumber ring stages");
static_assert(kRingOff % 128 == 0, "ring alignment");

__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

template <int KPW>
__global__ void __launch_bounds__(kExpertThreads, 1) gateup_swiglu_kernel(GateUpArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxGateUpStages;
  uint64_t* redbar = empty + kMaxGateUpStages;
  float4* red = reinterpret_cast<float4*>(smem + kRedOff);
  uint8_t* ring = smem + kRingOff;
  int* comp = reinterpret_cast<int*>(ring + (size_t)a.stages * a.tile_bytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kConsumerWarps);
    }
    for (int r = 0; r < kRedSlots; ++r) mbar_init(smem_u32(&redbar[r]), kConsumerWarps);
    fence_mbar_init();
  }

  // The weights streamed here are chosen by the routing: nothing of the main
  // loop is producer-independent.  Wait for the router, then release the
  // down kernel (its prologue and weight prefetch overlap this kernel).
  pdl_wait();
  pdl_launch_dependents();

  const int NP = a.M * a.K;
  const SmemRouting rt = load_routing(a.ws, NP, a.E, comp);

  const int TPG = (2 * a.I) / kGateUpTileRows;  // tiles per group
  const long long T = (long long)rt.n_groups * TPG;
  const int t0 = (int)(T * blockIdx.x / gridDim.x);
  const int t1 = (int)(T * (blockIdx.x + 1) / gridDim.x);
  const int n = t1 - t0;

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------- producer
    if (lane != 0) return;
    const uint32_t ring_u32 = smem_u32(ring);
    for (int j = 0; j < n; ++j) {
      const int s = j % S;
      unsigned long long waited = 0;
      if (j >= S && !mbar_wait(smem_u32(&empty[s]), ((j / S) - 1) & 1, &waited)) {
        record_timeout(a.ws, 2, kErrTimeoutEmpty, j, S, smem_u32(&empty[s]), waited);
        break;
      }
      const int tile = t0 + j;
      const int g = tile / TPG, tt = tile - g * TPG;
      const int e = rt.grp_expert[g];
      const uint32_t fb = smem_u32(&full[s]);
      mbar_arrive_expect_tx(fb, a.tile_bytes);
      bulk_g2s_chunked(ring_u32 + (uint32_t)s * a.tile_bytes,
                       a.w_gate_up + ((size_t)e * TPG + tt) * a.tile_bytes, a.tile_bytes, fb);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int g4 = lane >> 2, t4 = lane & 3;
  const uint32_t* xw = reinterpret_cast<const uint32_t*>(a.x);
  const int hw = a.H >> 1;  // 32-bit words per token row
  uint32_t af[KPW][2][4];
  int cur_g = -1, start = 0, cnt = 0;
  for (int j = 0; j < n; ++j) {
    const int s = j % S;
    const int tile = t0 + j;
    const int g = tile / TPG, tt = tile - g * TPG;
    if (g != cur_g) {
      // A fragments (tokens x this warp's K slice) of the new group; rows
      // beyond the group's count repeat its first token and are never stored.
      start = rt.grp_start[g];
      cnt = rt.grp_cnt[g];
      const int tok0 = rt.pair_list[start + (g4 < cnt ? g4 : 0)] / a.K;
      const int tok1 = rt.pair_list[start + (g4 + 8 < cnt ? g4 + 8 : 0)] / a.K;
      const uint32_t* x0 = xw + (size_t)tok0 * hw + t4;
      const uint32_t* x1 = xw + (size_t)tok1 * hw + t4;
#pragma unroll
      for (int q = 0; q < KPW; ++q) {
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int kw = (32 * (warp * KPW + q) + 16 * kk) >> 1;
          af[q][kk][0] = x0[kw];
          af[q][kk][1] = x1[kw];
          af[q][kk][2] = x0[kw + 4];
          af[q][kk][3] = x1[kw + 4];
        }
      }
      cur_g = g;
    }
    unsigned long long waited = 0;
    if (!mbar_wait(smem_u32(&full[s]), (j / S) & 1, &waited)) {
      record_timeout(a.ws, 2, kErrTimeoutFull, j, S, smem_u32(&full[s]), waited);
      break;
    }
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    const uint4* wp =
        reinterpret_cast<const uint4*>(ring + (size_t)s * a.tile_bytes) + (warp * KPW) * 32 + lane;
#pragma unroll
    for (int q = 0; q < KPW; ++q) {
      const uint4 b = wp[q * 32];
      mma_bf16(c0, af[q][0][0], af[q][0][1], af[q][0][2], af[q][0][3], b.x, b.y);
      mma_bf16(c1, af[q][1][0], af[q][1][1], af[q][1][2], af[q][1][3], b.z, b.w);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));  // stage free for the producer

    const int slot = j & (kRedSlots - 1);
    red[(slot * kConsumerWarps + warp) * 32 + lane] =
        make_float4(c0[0] + c1[0], c0[1] + c1[1], c0[2] + c1[2], c0[3] + c1[3]);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&redbar[slot]));

    if (warp == slot) {  // reducer of this tile (rotates over the warps)
      if (!mbar_wait(smem_u32(&redbar[slot]), (j >> 3) & 1, &waited)) {
        record_timeout(a.ws, 2, kErrTimeoutReduce, j, S, smem_u32(&redbar[slot]), waited);
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
      // (acc.x, acc.y) = (gate, up) of group token g4, intermediate row
      // 4*tt + t4; (acc.z, acc.w) the same for group token g4 + 8.
      const int r = 4 * tt + t4;
      if (g4 < cnt)
        a.ws.h[(size_t)(start + g4) * a.I + r] = __float2bfloat16_rn(silu(acc.x) * acc.y);
      if (g4 + 8 < cnt)
        a.ws.h[(size_t)(start + g4 + 8) * a.I + r] = __float2bfloat16_rn(silu(acc.z) * acc.w);
    }
  }
}

}  // namespace

size_t gateup_smem_bytes(int stages, uint32_t tile_bytes, int NP, int E) {
  (void)E;
  return kRingOff + (size_t)stages * tile_bytes + routing_smem_ints(NP) * 4;
}

GateUpKernel gateup_kernel_for(int kpw) {
  switch (kpw) {
    case 1: return gateup_swiglu_kernel<1>;
    case 2: return gateup_swiglu_kernel<2>;
    case 4: return gateup_swiglu_kernel<4>;
    case 5: return gateup_swiglu_kernel<5>;
    case 8: return gateup_swiglu_kernel<8>;
    case 10: return gateup_swiglu_kernel<10>;
    case 12: return gateup_swiglu_kernel<12>;
    case 16: return gateup_swiglu_kernel<16>;
    default: return nullptr;
  }
}

}  // namespace wse
