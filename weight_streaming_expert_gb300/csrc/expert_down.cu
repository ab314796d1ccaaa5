// expert_down.cu -- down GEMV over the activated experts with the
// routing-weighted combine fused into its epilogue.
//
// Method (page "How Ling-3.0-flash reduces batch 1 decoding latency by 54%
// on 4 Blackwell GPUs"):
//  * "PDL: the latency floor of stacked small kernels": the MoE chain ends
//    down-GEMM -> combine; the small-M combine is an fp32 sum times a scale
//    with a single final cast (the earlier path rounded twice).  Here the
//    scale is 1 and every output element is one fp32 sum of its token's k
//    weighted expert rows, rounded once.  Producer-independent loads go
//    before the dependency wait: the down weights depend only on the routing
//    (final before this grid can launch), so they are streamed before the
//    wait on the gate/up kernel and fly under its tail.
//  * "Two kinds of idle" / "Economics of speculation at batch 1": each
//    activated expert's [H, I] weight is streamed once for all its tokens.
//
// GB300 design.
//  * Routing: every CTA loads the (expert, <=16-token group) list the router
//    published into its shared memory (compaction.cuh).
//  * Work: (group, 8-row output slab) tiles of 8 rows x I (8 KB at I = 512),
//    in group-major order, split evenly over a persistent one-CTA-per-SM
//    grid.  Weights were re-laid out at create so each lane's 16 bytes are
//    its m16n8k16 B fragments for two k-steps (conflict-free shared loads);
//    the group's tokens are the A operand (m16), their activated rows h held
//    in registers for the whole K = I and the whole group.
//  * Staging: eight warps, each feeding ITSELF through D private stages of a
//    bulk-copy (TMA) ring (warp w takes tiles j = w, w+8, ...; its i-th tile
//    uses stage w + 8 (i mod D)).  A warp issues its first D tiles before the
//    dependency wait and refills a stage with its tile i + D as soon as it
//    has consumed tile i, so eight issuers keep up to 8 D tiles in flight and
//    no producer thread limits the request rate.  With one owner consuming
//    each stage in order, a parity wait can never see a stale phase.
//  * Epilogue: y = w_pair * (W_d h) goes to a per-pair fp32 row.  After its
//    whole range a CTA fences once and adds its tile count to the arrival
//    counter of every 8-row slab it touched.  Slab s is combined by CTA
//    s mod grid (2-3 slabs each at H = 2560): once the counters of all its
//    slabs show every group (a bounded wait), the CTA sums each token's k
//    rows in slot order and writes the output with ONE bf16 rounding.
//    Deterministic: the summation order never depends on scheduling.
#include "compaction.cuh"
#include "kernels.cuh"

namespace wse {

namespace {

constexpr size_t kRingOff = 1024;
constexpr int kDownThreads = kConsumerWarps * 32;
static_assert(kMaxDownStages * 8 + 64 <= kRingOff, "barrier area");
static_assert(kMaxDownStages % kConsumerWarps == 0, "one owner warp per stage");

// tiles t in [t0, t1) with t % SL == s
__device__ __forceinline__ int tiles_in_slab(int t0, int t1, int s, int SL) {
  const int first = t0 + ((s - t0) % SL + SL) % SL;
  return first >= t1 ? 0 : 1 + (t1 - 1 - first) / SL;
}

template <int KP>  // k-step pairs (I / 32)
__global__ void __launch_bounds__(kDownThreads, 1) down_combine_kernel(DownArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  int* s_flag = reinterpret_cast<int*>(full + kMaxDownStages);
  uint8_t* ring = smem + kRingOff;
  int* comp = reinterpret_cast<int*>(ring + (size_t)a.stages * a.tile_bytes);
  const int SL = a.H / kDownTileRows;  // tiles (output slabs) per group
  const int NP = a.M * a.K;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.stages, D = S / kConsumerWarps;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_mbar_init();
  }

  // The routing is final here: the router completed before the gate/up
  // kernel passed its own wait, and this grid was released only after that.
  const SmemRouting rt = load_routing(a.ws, NP, a.E, comp);
  const int n_groups = rt.n_groups;
  const long long T = (long long)n_groups * SL;
  const int t0 = (int)(T * blockIdx.x / gridDim.x);
  const int t1 = (int)(T * (blockIdx.x + 1) / gridDim.x);
  const int n = t1 - t0;
  const int n_mine = n > warp ? (n - warp + kConsumerWarps - 1) / kConsumerWarps : 0;
  const uint32_t ring_u32 = smem_u32(ring);

  // stage this warp's i-th tile into its stage (lane 0 only)
  auto issue = [&](int i) {
    const int j = i * kConsumerWarps + warp;
    const int s = warp + kConsumerWarps * (i % D);
    const int tile = t0 + j;
    const int g = tile / SL, sl = tile - g * SL;
    const uint32_t fb = smem_u32(&full[s]);
    mbar_arrive_expect_tx(fb, a.tile_bytes);
    bulk_g2s(ring_u32 + (uint32_t)s * a.tile_bytes,
             a.w_down + ((size_t)rt.grp_expert[g] * SL + sl) * a.tile_bytes, a.tile_bytes, fb);
  };
  // producer-independent: the first D tiles of every warp, before the wait
  if (lane == 0)
    for (int i = 0; i < D && i < n_mine; ++i) issue(i);

  pdl_wait();               // h (the gate/up output) is complete and visible
  pdl_launch_dependents();  // the next layer's router may prefetch its weights

  const int g4 = lane >> 2, t4 = lane & 3;
  uint32_t af[2 * KP][4];  // A fragments: group tokens x all of K
  int pid0 = -1, pid1 = -1;
  float pw0 = 0.f, pw1 = 0.f;
  int cur_g = -1;
  for (int i = 0; i < n_mine; ++i) {
    const int j = i * kConsumerWarps + warp;
    const int use = i / D, s = warp + kConsumerWarps * (i % D);
    const int tile = t0 + j;
    const int g = tile / SL, sl = tile - g * SL;
    if (g != cur_g) {
      // the group's activated rows, tokens g4 and g4 + 8 (rows past the
      // group's count repeat its first token and are never stored)
      const int start = rt.grp_start[g], cnt = rt.grp_cnt[g];
      const uint32_t* h0 =
          reinterpret_cast<const uint32_t*>(a.ws.h + (size_t)(start + (g4 < cnt ? g4 : 0)) * a.I) + t4;
      const uint32_t* h1 =
          reinterpret_cast<const uint32_t*>(a.ws.h + (size_t)(start + (g4 + 8 < cnt ? g4 + 8 : 0)) * a.I) + t4;
#pragma unroll
      for (int kk = 0; kk < 2 * KP; ++kk) {
        af[kk][0] = h0[kk * 8];
        af[kk][1] = h1[kk * 8];
        af[kk][2] = h0[kk * 8 + 4];
        af[kk][3] = h1[kk * 8 + 4];
      }
      pid0 = g4 < cnt ? rt.pair_list[start + g4] : -1;
      pid1 = g4 + 8 < cnt ? rt.pair_list[start + g4 + 8] : -1;
      pw0 = pid0 >= 0 ? a.ws.pair_w[pid0] : 0.f;
      pw1 = pid1 >= 0 ? a.ws.pair_w[pid1] : 0.f;
      cur_g = g;
    }
    unsigned long long waited = 0;
    if (!mbar_wait(smem_u32(&full[s]), use & 1, &waited)) {
      record_timeout(a.ws, 3, kErrTimeoutFull, j, S, smem_u32(&full[s]), waited);
      break;
    }
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    const uint4* bp = reinterpret_cast<const uint4*>(ring + (size_t)s * a.tile_bytes) + lane;
#pragma unroll
    for (int q = 0; q < KP; ++q) {
      const uint4 b = bp[q * 32];
      mma_bf16(c0, af[2 * q][0], af[2 * q][1], af[2 * q][2], af[2 * q][3], b.x, b.y);
      mma_bf16(c1, af[2 * q + 1][0], af[2 * q + 1][1], af[2 * q + 1][2], af[2 * q + 1][3], b.z, b.w);
    }
    __syncwarp();  // every lane has read the stage
    if (lane == 0 && i + D < n_mine) {
      fence_proxy_async_smem();
      issue(i + D);
    }

    // C: (token g4 | g4 + 8) x (rows 2t, 2t+1 of the slab)
    // y[pair][row] = w_pair * (W_d h_pair)[row]
    const int row = sl * kDownTileRows + 2 * t4;
    if (pid0 >= 0) {
      float* yr = a.ws.y + (size_t)pid0 * a.H + row;
      *reinterpret_cast<float2*>(yr) = make_float2(pw0 * (c0[0] + c1[0]), pw0 * (c0[1] + c1[1]));
    }
    if (pid1 >= 0) {
      float* yr = a.ws.y + (size_t)pid1 * a.H + row;
      *reinterpret_cast<float2*>(yr) = make_float2(pw1 * (c0[2] + c1[2]), pw1 * (c0[3] + c1[3]));
    }
  }

  // ---- end of range: publish every arrival, then combine this CTA's slabs.
  // Slab s is combined by CTA s % gridDim.  Each CTA adds ALL its arrivals
  // before it waits on any slab, so no CTA ever waits on a CTA that waits on
  // it; every CTA of this grid becomes resident (the gate/up kernel it
  // follows never waits on this one), so each wait ends.
  __threadfence();
  __syncthreads();
  const int tid = threadIdx.x;
  for (int s = tid; s < SL; s += kDownThreads) {
    const int c = tiles_in_slab(t0, t1, s, SL);
    if (c > 0) atomicAdd(a.ws.slab_count + s, c);
  }
  const int n_own = SL > (int)blockIdx.x ? (SL - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  if (tid < n_own) {
    int* cnt = a.ws.slab_count + blockIdx.x + tid * gridDim.x;
    const unsigned long long t_start = global_timer_ns();
    for (;;) {
      int v;
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
      if (v == n_groups) break;
      const unsigned long long dt = global_timer_ns() - t_start;
      if (dt > kWaitTimeoutNs) {
        record_timeout(a.ws, 3, kErrTimeoutReduce, (int)blockIdx.x + tid * (int)gridDim.x, S, 0, dt);
        break;
      }
      __nanosleep(32);
    }
    *cnt = 0;  // every arrival is in: ready for the next call
  }
  __syncthreads();
  const int per = a.M * kDownTileRows;
  for (int it = tid; it < n_own * per; it += kDownThreads) {
    const int sl = (int)blockIdx.x + (it / per) * (int)gridDim.x;
    const int m = (it % per) / kDownTileRows;
    const int r = sl * kDownTileRows + (it % kDownTileRows);
    float sum = 0.f;
    for (int k = 0; k < a.K; ++k) sum += __ldcg(a.ws.y + (size_t)(m * a.K + k) * a.H + r);
    a.out[(size_t)m * a.H + r] = __float2bfloat16_rn(sum);
  }
  (void)s_flag;
}

}  // namespace

size_t down_smem_bytes(int stages, uint32_t tile_bytes, int NP, int E, int H) {
  (void)H;
  (void)E;
  return kRingOff + (size_t)stages * tile_bytes + routing_smem_ints(NP) * 4;
}

DownKernel down_kernel_for(int ks) {
  switch (ks) {
    case 8: return down_combine_kernel<4>;    // I = 128
    case 16: return down_combine_kernel<8>;   // I = 256
    case 32: return down_combine_kernel<16>;  // I = 512
    default: return nullptr;
  }
}

}  // namespace wse
