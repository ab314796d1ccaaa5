// expert_down.cu -- down GEMV over the activated experts with the
// routing-weighted combine fused into its epilogue.
//
// Method (page "How Ling-3.0-flash reduces batch 1 decoding latency by 54%
// on 4 Blackwell GPUs"):
//  * "PDL: the latency floor of stacked small kernels": the MoE chain ends
//    down-GEMM -> combine; the small-M combine is an fp32 sum times a scale
//    with a single final cast (the earlier path rounded twice).  Here the
//    scale is 1 and the sum runs over each token's k slots in slot order.
//    Producer-independent loads go before the dependency wait: the down
//    weights depend only on the routing (complete before this grid can
//    launch), so the producer streams them before waiting on the gate/up
//    kernel, and they fly under its tail.
//  * "Two kinds of idle" / "Economics of speculation at batch 1": each
//    activated expert's [H, I] weight is streamed once for all its tokens.
//
// GB300 design.
//  * Work: (group, 16-row output slab) tiles, 16 rows x I (16 KB at I = 512),
//    split evenly over a persistent one-CTA-per-SM grid.  The weights were
//    re-laid out at create so each lane's 16 bytes are its m16n8k16 A
//    fragments (conflict-free shared loads).
//  * One producer thread stages tiles with bulk (TMA) copies into a ring;
//    eight consumer warps each take whole tiles round-robin, holding the
//    group's activated rows h (the B operand, n8 = 8 tokens, two n-tiles for
//    groups of 9..16 tokens) in registers for the whole K = I.
//  * Epilogue: y = w_pair * (W_d h) is written per pair in fp32; a per-slab
//    arrival counter (no spin) elects the last tile of each slab, which sums
//    the k slots of every token in slot order and writes out with ONE bf16
//    rounding.  Deterministic: the order never depends on scheduling.
#include "kernels.cuh"

namespace wse {

namespace {

struct DownMeta {
  int g, sl, start, cnt;
};

constexpr size_t kMetaOff = 2 * kMaxDownStages * 8;
constexpr size_t kRingOff = 1024;
static_assert(kMetaOff + kMaxDownStages * sizeof(DownMeta) <= kRingOff, "meta area");

template <int KS>
__global__ void __launch_bounds__(kExpertThreads, 1) down_combine_kernel(DownArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxDownStages;
  DownMeta* meta = reinterpret_cast<DownMeta*>(smem + kMetaOff);
  uint8_t* ring = smem + kRingOff;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.stages;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int SL = a.H / kDownTileRows;  // tiles (output slabs) per group
  const int NP = a.M * a.K;

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------- producer
    // The routing was published by the router kernel, which completed before
    // the gate/up kernel passed its own wait -- and this grid was released
    // only after that wait.  So the expert ids are final here, before our
    // wait: stream the weights now (L2-coherent loads).
    if (lane == 0) {
      int n_groups = __ldcg(a.ws.n_groups);
      if (n_groups < 0 || n_groups > NP) n_groups = 0;
      const long long T = (long long)n_groups * SL;
      const int t0 = (int)(T * blockIdx.x / gridDim.x);
      const int t1 = (int)(T * (blockIdx.x + 1) / gridDim.x);
      const uint32_t ring_u32 = smem_u32(ring);
      int cg = -1, e = 0, start = 0, cnt = 1;
      for (int j = 0; j < t1 - t0; ++j) {
        const int s = j % S;
        if (j >= S && !mbar_wait(smem_u32(&empty[s]), ((j / S) - 1) & 1)) {
          set_error(a.ws.status, kErrTimeoutEmpty);
          break;
        }
        const int tile = t0 + j;
        const int g = tile / SL, sl = tile - g * SL;
        if (g != cg) {
          e = __ldcg(a.ws.grp_expert + g);
          start = __ldcg(a.ws.grp_start + g);
          cnt = __ldcg(a.ws.grp_cnt + g);
          if (e < 0 || e >= a.E || cnt < 1 || cnt > kGroupTokens || start < 0 || start + cnt > NP) {
            set_error(a.ws.status, kErrBadIndex);
            e = 0; start = 0; cnt = 1;
          }
          cg = g;
        }
        const uint32_t fb = smem_u32(&full[s]);
        asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(fb), "r"(a.tile_bytes)
                     : "memory");
        bulk_g2s_chunked(ring_u32 + (uint32_t)s * a.tile_bytes,
                         a.w_down + ((size_t)e * SL + sl) * a.tile_bytes, a.tile_bytes, fb);
        meta[s] = DownMeta{g, sl, start, cnt};
        mbar_arrive(fb);
      }
      pdl_wait();
      pdl_launch_dependents();
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  pdl_wait();               // h (the gate/up output) is complete and visible
  pdl_launch_dependents();  // the next layer's router may prefetch its weights

  int n_groups = *a.ws.n_groups;
  if (n_groups < 0 || n_groups > NP) n_groups = 0;
  const long long T = (long long)n_groups * SL;
  const int t0 = (int)(T * blockIdx.x / gridDim.x);
  const int t1 = (int)(T * (blockIdx.x + 1) / gridDim.x);
  const int n = t1 - t0;

  const int g4 = lane >> 2, t4 = lane & 3;
  uint32_t hb[2][KS][2];
  int pid[4];
  float pw[4];
  int cur_start = -1;
  for (int j = warp; j < n; j += kConsumerWarps) {
    const int s = j % S;
    if (!mbar_wait(smem_u32(&full[s]), (j / S) & 1)) {
      set_error(a.ws.status, kErrTimeoutFull);
      break;
    }
    const DownMeta md = meta[s];
    if (md.start != cur_start) {
      // B fragments: activated rows of the group's tokens (n = token), all K.
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int i = nt * 8 + g4;
        const int row = md.start + (i < md.cnt ? i : 0);
        const uint32_t* hr = reinterpret_cast<const uint32_t*>(a.ws.h + (size_t)row * a.I) + t4;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          hb[nt][kk][0] = hr[kk * 8];
          hb[nt][kk][1] = hr[kk * 8 + 4];
        }
      }
      // pair ids / weights of this lane's output columns: tokens 2t, 2t+1,
      // 8+2t, 9+2t of the group
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = (q >> 1) * 8 + 2 * t4 + (q & 1);
        pid[q] = -1;
        pw[q] = 0.f;
        if (i < md.cnt) {
          const int p = a.ws.pair_list[md.start + i];
          if (p >= 0 && p < NP) {
            pid[q] = p;
            pw[q] = a.ws.pair_w[p];
          }
        }
      }
      cur_start = md.start;
    }

    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const uint4* ap = reinterpret_cast<const uint4*>(ring + (size_t)s * a.tile_bytes) + lane;
    if (md.cnt > 8) {
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        const uint4 av = ap[kk * 32];
        mma_bf16(acc[0], av.x, av.y, av.z, av.w, hb[0][kk][0], hb[0][kk][1]);
        mma_bf16(acc[1], av.x, av.y, av.z, av.w, hb[1][kk][0], hb[1][kk][1]);
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        const uint4 av = ap[kk * 32];
        mma_bf16(acc[0], av.x, av.y, av.z, av.w, hb[0][kk][0], hb[0][kk][1]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));

    // y[pair][row] = w_pair * (W_d h_pair)[row]; rows sl*16 + g4 and + 8.
    const int row0 = md.sl * kDownTileRows + g4, row1 = row0 + 8;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int q = nt * 2 + c;
        if (pid[q] >= 0) {
          float* yr = a.ws.y + (size_t)pid[q] * a.H;
          yr[row0] = pw[q] * acc[nt][c];
          yr[row1] = pw[q] * acc[nt][c + 2];
        }
      }
    }
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atomicAdd(a.ws.slab_count + md.sl, 1) == n_groups - 1;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      // every group has written its rows of this slab: combine in slot order
      __threadfence();
      for (int idx = lane; idx < a.M * kDownTileRows; idx += 32) {
        const int m = idx / kDownTileRows;
        const int r = md.sl * kDownTileRows + (idx % kDownTileRows);
        float sum = 0.f;
        for (int k = 0; k < a.K; ++k) sum += __ldcg(a.ws.y + (size_t)(m * a.K + k) * a.H + r);
        a.out[(size_t)m * a.H + r] = __float2bfloat16_rn(sum);
      }
      if (lane == 0) a.ws.slab_count[md.sl] = 0;  // ready for the next call
    }
  }
}

}  // namespace

size_t down_smem_bytes(int stages, uint32_t tile_bytes) {
  return kRingOff + (size_t)stages * tile_bytes;
}

DownKernel down_kernel_for(int ks) {
  switch (ks) {
    case 8: return down_combine_kernel<8>;
    case 16: return down_combine_kernel<16>;
    case 32: return down_combine_kernel<32>;
    default: return nullptr;
  }
}

}  // namespace wse
