// layer_kernel.cuh -- one routed-MoE layer call as ONE persistent kernel:
// router matvec -> tagged partial logits -> softmax top-k + compaction -> gate/up
// GEMV with SwiGLU -> down GEMV with the weighted combine.
//
// Method (page "How Ling-3.0-flash reduces batch 1 decoding latency by 54%
// on 4 Blackwell GPUs"):
//  * "Two kinds of idle": at small batch the critical path is the cold read
//    of the activated expert weights plus the launch floor; a routed layer
//    per step reads the router gate (2.6 MB at hidden 2560 x 512 experts)
//    and every activated expert's gate/up and down weights.
//  * "Economics of speculation at batch 1": verifying several tokens reads
//    the same weights as verifying one, so each activated expert is
//    streamed from HBM once for all of its tokens.
//  * "Two fusions and a retune": SwiGLU is folded into the up-projection
//    epilogue (fp32, one rounding to bf16, gate/up rows interleaved at load);
//    the token->expert alignment runs on the device on the pair axis.
//  * "PDL: the latency floor of stacked small kernels": producer-independent
//    loads go before the dependency wait; the small-M combine is an fp32 sum
//    with a single final cast (scale 1 here).
//
// GB300 design.  Grid = one CTA per SM (all resident: every CTA needs most of
// the SM's shared memory), 8 consumer warps, 1 producer warp (stages every
// weight tile) and 1 publisher warp (grid-wide arrivals and waits, so that
// no fence or atomic round trip ever stalls a thread that streams).
//  1. Prologue, before the dependency wait: barriers, the CTA's slice of
//     the router weight into registers.
//  2. Router matvec on the tensor cores (routing.cuh): fp32 partial logits
//     to the call's buffer (odd or even call: the index comes from the
//     arrival count the previous call left), the same words of the other
//     buffer marked unwritten for the next call.  No grid-wide barrier
//     follows: a reader polls the words it needs (bounded) until none is
//     unwritten.
//  3. EVERY CTA computes the top-k of all tokens and the compaction itself
//     (shared memory only): no second launch, no last-CTA hand-off.  The
//     results are bitwise equal in all CTAs (same inputs, same code), so they
//     agree on every position.  With more tokens than a CTA has warps, each
//     token's top-k is found once in the grid and its k slots published as
//     64-bit words that every CTA polls (one token a warp, not several in
//     turn).  With at most 16 tokens every chosen expert is one group and the
//     compaction is worked out on the pair axis (two short loops, no scan).
//  4. Gate/up: (group, 8-row) tiles of 8 weight rows x H, staged by the
//     producer with bulk copies into a ring of mbarrier-guarded stages.
//     The tiles of the first 7/8 of the groups are split statically, the
//     rest are taken one at a time from a global counter, so SMs that stream
//     faster take more (the per-SM rate differs by several per cent).  The producer writes each
//     stage's tile id and signals it before the copy lands, so consumers
//     fetch the group's token rows early.  Eight warps split H; a rotating
//     reducer warp sums their partials in a fixed order and applies SwiGLU.
//  5. Down: (group, 64-output-row) super tiles = 8 slabs of 8 rows x I,
//     one slab per consumer warp, staged the same way (the same producer,
//     the same 7/8 static + dynamic tail split, the same early tile ids).
//     The producer puts the first down super tiles into ring bytes as soon
//     as the gate/up tiles there are consumed for the last time -- HBM does
//     not drain between the two GEMVs.  No grid-wide barrier sits between
//     the GEMVs either: a down tile needs only its own group's h rows.
//     Every CTA's publisher counts it in when its statically split gate/up
//     tiles are reduced, and again when all of them are; a group whose
//     gate/up tiles all lie in the static share is ready once every CTA is
//     counted in the first, any other group once in the second.  The
//     publisher turns the two grid-wide counts into two shared-memory
//     barriers; the producer waits on the one a tile's group needs before it
//     hands the tile id to the consumers (its copy is already in flight).
//     The static down share holds (nearly) only early groups, so in practice
//     nothing waits.
//  6. Combine: the first CTAs (3 output slabs each) sum the k weighted rows
//     of each token in slot order, with ONE bf16 rounding.  Calls of up to 8
//     tokens write each weighted value with the index of the call that wrote
//     it in one 64-bit word, and the combining CTAs poll the values; larger
//     calls wait for a grid-wide count of all CTAs first.
// Every wait is bounded: a timeout sets a sticky status bit, records where,
// and the thread carries on (the call's result is then undefined).
#pragma once

#include "kernels.cuh"
#include "routing.cuh"

namespace wse {

namespace layer_detail {

// shared-memory map (bytes)
constexpr uint32_t kOffFull = 0;      // [8] gate/up stage: data landed (1 arrival + tx)
constexpr uint32_t kOffEmpty = 64;    // [8] gate/up stage: read by the 8 consumer warps
constexpr uint32_t kOffReady = 128;   // [8] gate/up stage: tile id written (1 arrival)
constexpr uint32_t kOffRedBar = 192;  // [8] reduction slot: 8 partials written
constexpr uint32_t kOffDone = 256;    // [1] all consumer warps left the gate/up loop
constexpr uint32_t kOffStatic = 264;  // [1] all consumer warps reduced the static gate/up tiles
constexpr uint32_t kOffLevel1 = 272;  // [1] every CTA's static gate/up tiles reduced (publisher)
constexpr uint32_t kOffLevel2 = 280;  // [1] every CTA's gate/up tiles reduced (publisher)
constexpr uint32_t kOffCall = 288;    // u64: the call's index on the grid counters (1, 2, ...)
constexpr uint32_t kOffCompacted = 296;  // [1] the compaction is in shared memory (1 arrival)
constexpr uint32_t kOffTile = 336;    // [8] int: tile id in each gate/up stage (-1: no more)
constexpr uint32_t kOffDTile = 384;   // [8] int: super-tile id in each down slot (-1: no more)
constexpr uint32_t kOffDFull = 416;   // [8] down slot: data landed (1 arrival + tx)
constexpr uint32_t kOffDEmpty = 480;  // [8] down slot: read by the 8 consumer warps
constexpr uint32_t kOffDReady = 544;  // [8] down slot: super-tile id written (1 arrival)
constexpr uint32_t kOffCells = 608;   // [8][8] int: ring cell of (down slot, consumer warp)
constexpr uint32_t kRingOff = 896;
constexpr int kRedSlots = 8;
constexpr uint32_t kRedBytes = kRedSlots * kConsumerWarps * 32 * 16;
constexpr int kStaticNum = 7, kStaticDen = 8;  // statically split share of the groups
static_assert(kMaxGateUpStages <= 8 && kMaxDownStages <= 8, "barrier map");
static_assert(kOffCall + 8 <= kOffCompacted && kOffCompacted + 8 <= kOffTile && kOffTile + 4 * kMaxGateUpStages <= kOffDTile &&
                  kOffDReady + 8 * kMaxDownStages <= kOffCells &&
                  kOffCells + 4 * kMaxDownStages * kConsumerWarps <= kRingOff,
              "map");
static_assert(kRingOff % 128 == 0, "ring alignment");
static_assert((unsigned long long)(kMaxPairs + kMaxTokens) * (2 * 32 * kMaxDownChunks / kGateUpTileRows) * 1024ull <
                  (1ull << 32),
              "static splits in 32-bit arithmetic (groups x tiles per group x grids of up to 1024 CTAs)");
static_assert(kMaxGateUpStages < kRedSlots, "reduction slots must outnumber ring stages");

struct OneSlab {  // a down cell of one slab, as a compile-time count
  __device__ constexpr operator int() const { return 1; }
};

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Count this CTA in at a grid-wide counter: release fence, then an atomic
// add whose result nobody waits for.
__device__ __forceinline__ void grid_count(unsigned* word) {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], 1;" ::"l"(word) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// A weighted down-projection value with the call index that wrote it: one
// 64-bit relaxed store, so a reader that sees the index sees the value.
__device__ __forceinline__ void put_y(unsigned long long* p, float v, unsigned tag) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(((unsigned long long)tag << 32) | __float_as_uint(v))
               : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void stamp(const LayerArgs& a, int slot) {
  if (a.trace) a.ws.trace[(size_t)blockIdx.x * kTraceSlots + slot] = global_timer_ns();
}

__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Bounded acquire-spin until the count at `word` reaches `target`.
__device__ inline bool grid_wait(const Workspace& ws, const unsigned* word, unsigned long long target,
                                 int phase, unsigned long long limit) {
  const unsigned long long* cnt = reinterpret_cast<const unsigned long long*>(word);
  if (ld_acquire64(cnt) >= target) return true;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
    __nanosleep(32);
    if (ld_acquire64(cnt) >= target) return true;
    const unsigned long long dt = global_timer_ns() - t0;
    if (dt > limit) {
      record_timeout(ws, phase, kErrTimeoutGrid, (int)(target % gridDim.x), 0, 0, dt);
      return false;
    }
  }
}


__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

// First tile of CTA c in a static split of T tiles: floor(T c / grid), in
// 32-bit arithmetic (T <= kMaxPairs x 128 tiles, so T x grid < 2^32).
__device__ __forceinline__ int static_share(int T, unsigned c) { return (int)((unsigned)T * c / gridDim.x); }

}  // namespace layer_detail

// KPW = H / 256: 32-wide k chunks per warp in the gate/up GEMV.  VARIANT:
// the instance that handles the layer variants (shared expert, routed scale,
// selection-only bias); the plain instance compiles none of their code.
// FP8: expert weights as E4M3 codes with fp32 per-row scales -- tiles of 16
// rows (the same bytes as 8 bf16 rows), codes converted to f16 in registers,
// tokens and h converted to f16 per group, the row scales applied in fp32
// after the sums (reducer and down epilogue).
// TB: token blocks of 8 per group.  TB = 2 serves groups of up to 16 tokens
// (any call): the group's tokens are the MMA's A operand (16 rows) and the
// weights B (bf16: the 8-row tile; fp8: each of the tile's two 8-row blocks,
// four MMAs per 16-byte chunk).  TB = 1 serves groups of at most 8 tokens
// (calls with M <= 8) and holds one set of token registers instead of two
// (the two sets are 40 to 128 registers of a 168-register budget): bf16 still
// puts the tokens in A, the same 8 rows in both halves (rows 8..15 of C are
// never stored); fp8 swaps the operands -- the tile's 16 weight rows are A
// and the tokens one n8 B block, two MMAs per chunk.
template <int KPW, bool VARIANT, bool FP8, int TB>
__global__ void __launch_bounds__(kExpertThreads, 1) moe_layer_kernel(LayerArgs a) {
  using namespace layer_detail;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) stamp(a, 19);  // CTA started
  const int S = a.gu_stages;
  constexpr int GU_ROWS = FP8 ? 16 : kGateUpTileRows;  // weight rows per gate/up tile
  constexpr int D_ROWS = FP8 ? 16 : kDownTileRows;     // output rows per down slab
  static_assert(TB == 1 || TB == 2, "token blocks");
  constexpr bool WA = FP8 && TB == 1;                  // the weights are the MMA's A operand
  constexpr bool TWO = TB == 2;                        // a second token set (group rows 8..15)
  constexpr int NB = FP8 && TB == 2 ? 2 : 1;           // float4 partials per lane (gate/up reduction)
  constexpr bool kTaggedRows = TB == 1;                // weighted rows tagged with the call index
  const int NSL = kConsumerWarps, SD = a.d_stages;  // cells per down super tile, down slots
  const int SPW = a.d_spw;                           // down slabs per cell
  const int MK = a.M * a.K;                     // routed pairs (token * K + slot)
  const bool shared = VARIANT && a.shared;
  const int NP = MK + (shared ? a.M : 0);       // + the shared expert's pairs MK + token
  const int EA = a.E + (shared ? 1 : 0);        // buckets: routed experts + the shared one
  const uint32_t sb = smem_u32(smem);
  int* stage_tile = reinterpret_cast<int*>(smem + kOffTile);
  int* dstage_tile = reinterpret_cast<int*>(smem + kOffDTile);
  const uint32_t dsuper = (uint32_t)NSL * a.d_tile;  // bytes of a down super tile
  int* cell_tab = reinterpret_cast<int*>(smem + kOffCells);  // [slot][warp] -> ring cell
  uint8_t* ring = smem + kRingOff;
  const uint32_t ring_u32 = sb + kRingOff;
  float4* red = reinterpret_cast<float4*>(ring + (size_t)S * a.gu_tile);
  const SmemRouting rt = routing_carve(ring + a.ring_bytes, NP, EA);
  auto full = [&](int s) { return sb + kOffFull + 8u * s; };
  auto empty = [&](int s) { return sb + kOffEmpty + 8u * s; };
  auto ready = [&](int s) { return sb + kOffReady + 8u * s; };
  auto redbar = [&](int r) { return sb + kOffRedBar + 8u * r; };
  auto dfull = [&](int d) { return sb + kOffDFull + 8u * d; };
  auto dempty = [&](int d) { return sb + kOffDEmpty + 8u * d; };
  auto dready = [&](int d) { return sb + kOffDReady + 8u * d; };
  const uint32_t done = sb + kOffDone;
  const uint32_t static_bar = sb + kOffStatic;
  const uint32_t level1 = sb + kOffLevel1, level2 = sb + kOffLevel2;
  unsigned long long* call_idx = reinterpret_cast<unsigned long long*>(smem + kOffCall);

  // ---- 1. producer-independent: this CTA's slice of the router weight
  const int units = ((a.E + 7) / 8) * a.ks;
  const int gw = warp < kConsumerWarps ? warp : 0;
  GemvUnit gu = gemv_unit(blockIdx.x, a.ks, a.H, gw);
  uint4 wb[KPW];
  if ((int)blockIdx.x < units && warp < kConsumerWarps) gemv_load_w<KPW>(a.w_router, a.E, a.H, gu, lane, wb);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kConsumerWarps);
      mbar_init(ready(s), 1);
    }
    for (int r = 0; r < kRedSlots; ++r) mbar_init(redbar(r), kConsumerWarps);
    mbar_init(done, kConsumerWarps);
    mbar_init(static_bar, kConsumerWarps);
    mbar_init(level1, 1);
    mbar_init(level2, 1);
    mbar_init(sb + kOffCompacted, 1);
    for (int d = 0; d < SD; ++d) {
      mbar_init(dfull(d), 1);
      mbar_init(dempty(d), kConsumerWarps);
      mbar_init(dready(d), 1);
    }
    fence_mbar_init();
  }
  for (int e = tid; e < EA; e += kExpertThreads) {
    rt.mask[e] = 0ull;
    if constexpr (TB == 2) rt.s_off[e] = 0;  // bucket counts (see bucket_add)
  }
  for (int i = tid; i < kChunkLevels * kBitWords; i += kExpertThreads) rt.bits[i] = 0u;
  for (int p = tid; p < NP; p += kExpertThreads) rt.pair_list[p] = 0;
  if (tid < 2) rt.scal[tid] = 0;

  if (tid == 0) stamp(a, 20);  // prologue done
  pdl_wait();               // x and the workspace belong to this call now
  pdl_launch_dependents();  // the next call's prologue may start as SMs free up
  if (tid == 0) stamp(a, 0);
  if (warp == kPublisherWarp && lane == 0) {
    // the previous call on this workspace is complete: its CTAs' arrivals
    // give this call's index (acquire: nothing of this call moves above it)
    const unsigned long long idx = ld_acquire64(reinterpret_cast<const unsigned long long*>(a.ws.sync + kSyncCount)) /
                                       gridDim.x + 1ull;
    *call_idx = idx;
    if (blockIdx.x == 0) {  // the work counters of the next call (this call's were cleared by the last)
      a.ws.sync[idx & 1ull ? kSyncGateUpNext : kSyncGateUpNextOdd] = 0u;
      a.ws.sync[idx & 1ull ? kSyncDownNext : kSyncDownNextOdd] = 0u;
    }
  }

  // ---- 2. router matvec into this call's buffer of partial logits (no
  // grid-wide barrier after it: the readers poll the words)
  const size_t plane = (size_t)kMaxTokens * a.E;
  __syncthreads();  // the call index is in shared memory
  const bool odd = (*call_idx & 1ull) != 0ull;
  float* part = a.ws.part + (odd ? (size_t)a.ks * plane : 0);
  float* part_next = a.ws.part + (odd ? 0 : (size_t)a.ks * plane);
  for (int unit = blockIdx.x; unit < units; unit += gridDim.x) {
    if (unit != (int)blockIdx.x) {
      gu = gemv_unit(unit, a.ks, a.H, gw);
      if (warp < kConsumerWarps) gemv_load_w<KPW>(a.w_router, a.E, a.H, gu, lane, wb);
    }
    if (warp == kProducerWarp) gemv_clear(gu, kMaxTokens, a.E, plane, part_next, lane);
    for (int mb = 0; mb * 16 < a.M; ++mb) {
      if (warp < kConsumerWarps) red[warp * 32 + lane] = gemv_tokens<KPW>(a.x, a.M, a.H, gu, mb, lane, wb);
      __syncthreads();
      if (warp == 0) gemv_store<true>(red, gu, mb, a.M, a.E, plane, part, lane);
      __syncthreads();
    }
  }
  __syncthreads();
  if (tid == 0) stamp(a, 1);

  // ---- 3. top-k of every token, compaction (every CTA, shared memory only)
  constexpr int kWarps = kExpertThreads / 32;
  bool exchanged = false;
  if constexpr (TB == 2) exchanged = a.M > kWarps;
  if (!exchanged) {  // every CTA finds every token's top-k itself (a token per warp)
    for (int m = warp; m < a.M; m += kWarps) {
      const float w = topk_dispatch(PolledPlanes{part + (size_t)m * a.E, plane, a.wait_ns}, a.ks, a.bias, a.E, a.K,
                                    lane, a.ws.status, rt.s_e + m * a.K, VARIANT && a.sel_only != 0);
      __syncwarp();
      if (lane < a.K) {
        const int p = m * a.K + lane;
        const int idx = rt.s_e[p];
        rt.s_w[p] = VARIANT ? w * a.routed_scale : w;  // the combine's weight; topk_w is unscaled
        bucket_add<TB == 2>(rt, idx, m);
        if (blockIdx.x == 0) {
          a.topk_idx[p] = idx;
          if (a.topk_w) a.topk_w[p] = w;
        }
      }
    }
  } else if constexpr (TB == 2) {
    // more tokens than warps: each token's top-k is found ONCE in the grid
    // (token m by warp m / grid of CTA m mod grid) and published as one
    // 64-bit word per slot; every CTA then polls the M k words (bounded).
    // Taking the tokens in turn on one CTA's warps cost ~3 us per token.
    unsigned long long* xb = a.ws.xtopk + (odd ? (size_t)kMaxTokens * kMaxTopk : 0);
    int* scratch = reinterpret_cast<int*>(red) + warp * kMaxTopk;  // the warp's slot ids
    for (int m = (int)blockIdx.x + (int)gridDim.x * warp; m < a.M; m += (int)gridDim.x * kWarps) {
      const float w = topk_dispatch(PolledPlanes{part + (size_t)m * a.E, plane, a.wait_ns}, a.ks, a.bias, a.E, a.K,
                                    lane, a.ws.status, scratch, VARIANT && a.sel_only != 0);
      __syncwarp();
      if (lane < a.K) {
        const unsigned long long word =
            ((unsigned long long)(unsigned)scratch[lane] << 32) | (unsigned long long)__float_as_uint(w);
        st_relaxed64(xb + m * a.K + lane, word);
      }
      __syncwarp();
    }
    const unsigned long long t0 = global_timer_ns();
    for (int i = tid; i < MK; i += kExpertThreads) {
      unsigned long long word = ld_relaxed64(xb + i);
      while (word == ~0ull) {  // not published yet (bounded)
        if (global_timer_ns() - t0 > a.wait_ns) {
          set_error(a.ws.status, kErrTimeoutGrid);
          word = 0ull;
          break;
        }
        __nanosleep(32);
        word = ld_relaxed64(xb + i);
      }
      const int m = i / a.K, p = i;
      const int idx = (int)(word >> 32);
      const float w = __uint_as_float((unsigned)word);
      rt.s_e[p] = idx;
      rt.s_w[p] = VARIANT ? w * a.routed_scale : w;
      bucket_add<TB == 2>(rt, idx, m);
      if (blockIdx.x == 0) {
        a.topk_idx[p] = idx;
        if (a.topk_w) a.topk_w[p] = w;
      }
    }
  }
  if (shared && tid < a.M) {  // every token's pair with the shared expert, weight 1
    const int p = MK + tid;
    rt.s_e[p] = a.E;
    rt.s_w[p] = 1.0f;
    bucket_add<TB == 2>(rt, a.E, tid);
  }
  __syncthreads();
  if (tid == 0) stamp(a, 12);
  const int TPG = 2 * a.I / GU_ROWS;          // gate/up tiles per group
  const int CL = a.H / (D_ROWS * SPW);        // down cells per group (SPW output slabs each)
  const int SPG = CL / NSL;                   // down super tiles per group
  const int levels = (a.M + kGroupTokens - 1) / kGroupTokens;  // 16-token groups per expert, at most
  // The producer warp does not wait for the compaction: it numbers the
  // groups from the chunk bitmaps and starts the gate/up copies at once,
  // while the other warps compact; the copies' HBM latency hides the
  // compaction.  The two agree on the group order (ascending expert, then
  // chunk).
  // The down phase reuses the ring as cells of SPW slabs (d_tile bytes; a
  // gate/up stage is exactly cps cells, the reduction area behind the
  // stages holds the rest).  Gate/up stage (n_gu + r) mod S is released for
  // the last time r-th (n_gu = this CTA's gate/up tile count; stages it
  // never used come first), the reduction area after all of them.  Listing
  // the cells in that order, down slot u takes list entries 8u .. 8u + 7,
  // one per consumer warp: its first use waits only for the releases that
  // free those cells, and every cell of the ring is used.
  // The producer writes the (slot, warp) -> cell table once, before its
  // first down tile is handed out (the consumers read it after that).
  const int cps = (int)(a.gu_tile / a.d_tile);
  const int gu_cells = S * cps;
  auto slot_rank = [&](int u) -> int {  // release index that frees slot u's last cell (S: reduction area)
    const int p = u * kConsumerWarps + kConsumerWarps - 1;
    return p < gu_cells ? p / cps : S;
  };
  if (warp == kProducerWarp) {
    // ================================================================ producer
    const int n_groups = count_groups(rt, EA, levels, lane);
    if (lane != 0) return;
    stamp(a, 3);
    const int nw = (EA + 31) / 32;
    const int T_gu = n_groups * TPG, T_d = n_groups * SPG;
    const int g_static = n_groups * kStaticNum / kStaticDen;  // as the consumers' (below)
    unsigned long long waited = 0;
    // static share of each phase, then single tiles from the shared tail
    const int Ts = g_static * TPG;
    const int s0 = static_share(Ts, blockIdx.x), s1 = static_share(Ts, blockIdx.x + 1);
    // the fp8 consumers of 16-token groups are bound by their own instructions,
    // not by the copies: for them a static split of every down tile beats the
    // dynamic tail (measured: fp8 M = 16 -2.5 us, 16 Zipf -1.2 us); every
    // other instance keeps the tail (all static cost bf16 M = 6 3.3 us)
    const int Ts2 = FP8 && TB == 2 ? T_d : g_static * SPG;
    const int q0 = static_share(Ts2, blockIdx.x), q1 = static_share(Ts2, blockIdx.x + 1);
    unsigned* next_gu = a.ws.sync + (odd ? kSyncGateUpNextOdd : kSyncGateUpNext);
    const uint64_t wpol = l2_evict_first_policy();  // expert weights: read once per call
    unsigned* next_d = a.ws.sync + (odd ? kSyncDownNextOdd : kSyncDownNext);
    // gate/up tiles of the shared tail are taken one ahead (the atomic's
    // round trip hides behind a tile), starting one tile before the static
    // share ends: a tile taken earlier would be held back from faster SMs.
    // Down tiles of the shared tail are taken only once a slot is free (the
    // slots in flight hide the round trip), so that at the end no CTA holds
    // a tile it cannot start while others have none.
    const int n_s = s1 - s0, n_s2 = q1 - q0;
    int dyn_gu = n_s <= 1 ? Ts + (int)atomicAdd(next_gu, 1u) : 0;
    bool ok = true;
    int level = 0;  // readiness of the h rows seen so far (see the publisher)
    // ---- gate/up tiles
    int j = 0, gu_w = 0, cur_gg = -1, cur_ge = 0;  // group -> expert lookups (ascending groups)
    for (;; ++j) {
      int tile;
      if (j < n_s) {
        tile = s0 + j;
        if (j == n_s - 2) dyn_gu = Ts + (int)atomicAdd(next_gu, 1u);
      } else {
        tile = dyn_gu;
        if (tile < T_gu) dyn_gu = Ts + (int)atomicAdd(next_gu, 1u);
      }
      if (tile >= T_gu) break;
      const int s = j % S;
      if (j >= S && !mbar_wait(empty(s), ((j / S) - 1) & 1, &waited, a.wait_ns)) {
        record_timeout(a.ws, 2, kErrTimeoutEmpty, j, S, empty(s), waited);
        ok = false;
        break;
      }
      stage_tile[s] = tile;
      mbar_arrive(ready(s));
      const int g = tile / TPG, tt = tile - g * TPG;
      if (g != cur_gg) {  // the compaction's table once it exists, the bitmaps before
        cur_gg = g;
        cur_ge = mbar_test_wait(sb + kOffCompacted, 0) ? rt.grp_expert[g] : group_expert(rt, g, levels, nw, gu_w);
      }
      mbar_arrive_expect_tx(full(s), a.gu_tile);
      bulk_g2s_chunked(ring_u32 + (uint32_t)s * a.gu_tile,
                       a.w_gate_up + ((size_t)cur_ge * TPG + tt) * a.gu_tile, a.gu_tile, full(s), wpol);
    }
    const int n_gu = j;
    if (ok) {  // end marker for the consumers
      const int s = j % S;
      if (j >= S && !mbar_wait(empty(s), ((j / S) - 1) & 1, &waited, a.wait_ns)) {
        record_timeout(a.ws, 2, kErrTimeoutEmpty, j, S, empty(s), waited);
        ok = false;
      } else {
        stage_tile[s] = -1;
        mbar_arrive(ready(s));
      }
    }
    stamp(a, 9);
    if (a.trace) a.ws.trace[(size_t)blockIdx.x * kTraceSlots + 11] = (unsigned long long)n_gu;
    // the readiness level the h rows of down group g need
    auto ensure_ready = [&](int g) -> bool {
      const int need = g < g_static ? 1 : 2;
      if (level >= need) return true;
      if (!mbar_wait(need == 1 ? level1 : level2, 0, &waited, a.wait_ns)) {
        record_timeout(a.ws, 3, kErrTimeoutReduce, -5 - need, SD, need == 1 ? level1 : level2, waited);
        return false;
      }
      level = need;
      return true;
    };
    // ---- down super tiles.  Slot u's first use waits until its cells are
    // free: the gate/up stages under them released for the last time (the
    // last S gate/up tiles, in consumption order), and for cells over the
    // reduction area every consumer warp out of the gate/up loop.
    {  // list position p -> cell, by running counters (no division per entry)
      int st = n_gu % S, within = 0;
      for (int p = 0; p < SD * kConsumerWarps; ++p) {
        cell_tab[p] = p >= gu_cells ? p : st * cps + within;
        if (++within == cps) {
          within = 0;
          st = st + 1 == S ? 0 : st + 1;
        }
      }
    }
    int r_done = 0;  // gate/up final releases waited for
    bool red_free = false;
    auto release_until = [&](int rank) -> bool {
      const int upto = rank < S ? rank : S - 1;
      for (; r_done <= upto; ++r_done) {
        const int jf = n_gu - S + r_done;
        if (jf < 0) continue;  // a stage this CTA never used
        const int st = jf % S;
        if (!mbar_wait(empty(st), (jf / S) & 1, &waited, a.wait_ns)) {
          record_timeout(a.ws, 3, kErrTimeoutEmpty, jf, S, empty(st), waited);
          return false;
        }
      }
      if (rank >= S && !red_free) {
        if (!mbar_wait(done, 0, &waited, a.wait_ns)) {
          record_timeout(a.ws, 3, kErrTimeoutEmpty, -1, S, done, waited);
          return false;
        }
        fence_proxy_async_smem();  // the reduction area was last written with ordinary stores
        red_free = true;
      }
      return true;
    };
    int j2 = 0;
    int cur_dg = -1, cur_de = 0;
    // the down tiles take their experts from the compaction: wait for it
    // (it is long done unless this CTA had no gate/up tile at all)
    if (ok && !mbar_wait(sb + kOffCompacted, 0, &waited, a.wait_ns)) {
      record_timeout(a.ws, 3, kErrTimeoutReduce, -9, SD, sb + kOffCompacted, waited);
      ok = false;
    }
    for (; ok; ++j2) {
      const int s = j2 % SD;
      if (j2 < SD) {
        if (!release_until(slot_rank(s))) {
          ok = false;
          break;
        }
      } else if (!mbar_wait(dempty(s), ((j2 / SD) - 1) & 1, &waited, a.wait_ns)) {
        record_timeout(a.ws, 3, kErrTimeoutEmpty, j2, SD, dempty(s), waited);
        ok = false;
        break;
      }
      const int tile = j2 < n_s2 ? q0 + j2 : Ts2 + (int)atomicAdd(next_d, 1u);
      if (tile >= T_d) break;
      // the copy first (weights never depend on h), then the id once the
      // group's h rows are ready
      const int g = tile / SPG, q = tile - g * SPG;
      if (g != cur_dg) {  // the group's expert (the compaction is in place: see below)
        cur_dg = g;
        cur_de = rt.grp_expert[g];
      }
      mbar_arrive_expect_tx(dfull(s), dsuper);
      {  // the 8 slabs are contiguous in global memory; one copy per run of
         // adjacent cells, the runs worked out arithmetically (list positions
         // 8s .. 8s + 7, stage boundaries every cps positions)
        const uint8_t* src = a.w_down + ((size_t)cur_de * CL + (size_t)q * NSL) * a.d_tile;
        int p = s * kConsumerWarps, left = NSL, w0 = 0;
        int r = p / cps, within = p - r * cps;
        while (left > 0) {
          int run, cell;
          if (p >= gu_cells) {
            run = left;
            cell = p;
          } else {
            run = min(left, cps - within);
            cell = ((n_gu + r) % S) * cps + within;
          }
          bulk_g2s_chunked(ring_u32 + (uint32_t)cell * a.d_tile, src + (size_t)w0 * a.d_tile,
                           (uint32_t)run * a.d_tile, dfull(s), wpol);
          p += run;
          w0 += run;
          left -= run;
          ++r;
          within = 0;
        }
      }
      if (!ensure_ready(g)) {
        // the copy just issued lands in a slot no consumer will read: wait
        // for it (bounded) so that no copy is in flight when the CTA exits
        if (!mbar_wait(dfull(s), (uint32_t)(j2 / SD) & 1u, &waited, a.wait_ns))
          record_timeout(a.ws, 3, kErrTimeoutFull, j2, SD, dfull(s), waited);
        ok = false;
        break;
      }
      dstage_tile[s] = tile;
      mbar_arrive(dready(s));
    }
    if (a.trace) a.ws.trace[(size_t)blockIdx.x * kTraceSlots + 16] = (unsigned long long)j2;
    if (ok) {  // end marker (a first use needs no free bytes: only the id is written)
      const int s = j2 % SD;
      if (j2 >= SD && !mbar_wait(dempty(s), ((j2 / SD) - 1) & 1, &waited, a.wait_ns)) {
        record_timeout(a.ws, 3, kErrTimeoutEmpty, j2, SD, dempty(s), waited);
      } else {
        dstage_tile[s] = -1;
        mbar_arrive(dready(s));
      }
    }
    stamp(a, 10);
    return;
  }
  // the consumer and publisher warps (288 threads) compact; the reduction
  // area is free until the gate/up loop: scratch for the pair-axis
  // compaction (small loops: this code runs once per call, with a cold
  // instruction cache, so its size costs more than its arithmetic)
  constexpr int kCompactThreads = kExpertThreads - 32;
  const int ct = warp < kConsumerWarps ? tid : tid - 32;  // 0 .. 287
  const int n_groups = a.M <= kGroupTokens
                           ? compact_pairs(rt, NP, a.K, MK, reinterpret_cast<int*>(red), ct, kCompactThreads)
                           : (compact_masks(rt, NP, a.K, MK, EA, ct, kCompactThreads), rt.scal[0]);
  if (tid == 0) {
    mbar_arrive(sb + kOffCompacted);  // the producer reads grp_expert from here on
    stamp(a, 13);
  }
  if (blockIdx.x == 0) {  // a copy for inspection (moe_read_routing); nothing reads it back
    for (int i = ct; i < NP; i += kCompactThreads) {
      a.ws.pair_list[i] = rt.pair_list[i];
      a.ws.pair_w[i] = rt.s_w[i];
      if (i < n_groups) {
        a.ws.grp_expert[i] = rt.grp_expert[i];
        a.ws.grp_start[i] = rt.grp_start[i];
        a.ws.grp_cnt[i] = rt.grp_cnt[i];
      }
    }
    if (ct == 0) {
      *a.ws.n_groups = n_groups;
      *a.ws.n_active = rt.scal[1];
    }
  }
  // groups [0, g_static) are split statically in both GEMVs: their gate/up
  // tiles are all in the static share, and so are their down tiles
  const int g_static = n_groups * kStaticNum / kStaticDen;
  if (warp == kPublisherWarp) {
    // =============================================================== publisher
    if (lane != 0) return;
    unsigned long long waited = 0;
    const unsigned long long target = *call_idx * gridDim.x;
    // static gate/up tiles reduced here -> counted; every CTA counted -> level 1
    if (!mbar_wait(static_bar, 0, &waited, a.wait_ns)) {
      record_timeout(a.ws, 2, kErrTimeoutReduce, -3, 0, static_bar, waited);
      return;
    }
    if (!(a.test_flags & kTestSkipArrival) || blockIdx.x != 0) grid_count(a.ws.sync + kSyncStaticDone);
    stamp(a, 18);
    if (!grid_wait(a.ws, a.ws.sync + kSyncStaticDone, target, 2, a.wait_ns)) return;
    mbar_arrive(level1);
    stamp(a, 6);
    if constexpr (TB == 2) {
      // every CTA has read the exchanged slots (its routing precedes its
      // static tiles): mark this CTA's share of them unwritten for the
      // next call of this parity
      if (a.M > kExpertThreads / 32) {
        unsigned long long* xb = a.ws.xtopk + (odd ? (size_t)kMaxTokens * kMaxTopk : 0);
        for (int i = (int)blockIdx.x; i < MK; i += (int)gridDim.x)
          st_relaxed64(xb + i, ~0ull);
      }
    }
    // all gate/up tiles reduced here -> counted; every CTA counted -> level 2
    if (!mbar_wait(done, 0, &waited, a.wait_ns)) {
      record_timeout(a.ws, 2, kErrTimeoutReduce, -4, 0, done, waited);
      return;
    }
    grid_count(a.ws.sync + kSyncGateUpDone);
    if (!grid_wait(a.ws, a.ws.sync + kSyncGateUpDone, target, 2, a.wait_ns)) return;
    mbar_arrive(level2);
    stamp(a, 17);
    return;
  }


  // ================================================================ consumers
  const int g4 = lane >> 2, t4 = lane & 3;
  unsigned long long waited = 0;
  {
    // ---- 4. gate/up + SwiGLU
    uint4 xa[KPW], xb[KPW];  // token rows g4 and g4 + 8 of the group: this warp's k chunks
                             // (TB = 1: row g4 only)
    int cur_g = -1, start = 0, cnt = 0;
    // this CTA's statically split tiles come first: after the last of them
    // (or at once if it has none) the warp reports them reduced
    const int Ts = g_static * TPG;
    const int n_static = static_share(Ts, blockIdx.x + 1) - static_share(Ts, blockIdx.x);
    if (n_static == 0 && lane == 0) mbar_arrive(static_bar);
    for (int j = 0;; ++j) {
      const int s = j % S;
      const uint32_t ph = (uint32_t)(j / S) & 1u;
      if (!warp_wait(ready(s), ph, &waited, a.wait_ns)) {
        record_timeout(a.ws, 2, kErrTimeoutFull, j, S, ready(s), waited);
        break;
      }
      const int tile = stage_tile[s];
      if (tile < 0) break;
      const int g = tile / TPG, tt = tile - g * TPG;
      if (g != cur_g) {
        // rows beyond the group's count repeat its first token, never stored
        start = rt.grp_start[g];
        cnt = rt.grp_cnt[g];
        const int p0 = rt.pair_list[start + (g4 < cnt ? g4 : 0)];
        const int p1 = rt.pair_list[start + (g4 + 8 < cnt ? g4 + 8 : 0)];
        const int tok0 = VARIANT ? pair_token(p0, a.K, MK) : p0 / a.K;
        const int tok1 = VARIANT ? pair_token(p1, a.K, MK) : p1 / a.K;
        const uint4* x0 = reinterpret_cast<const uint4*>(a.x + (size_t)tok0 * a.H) + t4;
        const uint4* x1 = reinterpret_cast<const uint4*>(a.x + (size_t)tok1 * a.H) + t4;
#pragma unroll
        for (int q = 0; q < KPW; ++q) {
          xa[q] = x0[4 * (warp * KPW + q)];
          if constexpr (TWO) xb[q] = x1[4 * (warp * KPW + q)];
          if constexpr (FP8) {
            xa[q] = bf16x8_to_f16x8(xa[q]);
            if constexpr (TWO) xb[q] = bf16x8_to_f16x8(xb[q]);
          }
        }
        cur_g = g;
      }
      // fp8 row scales, loaded early by this tile's reducer: weights as A,
      // (gate, up) of intermediate row 8 tt + g4 in (sg.x, su.x); weights as
      // B, rows 8 tt + 2 t4 and + 1 in (sg.x, sg.y) and (su.x, su.y)
      float2 sg = make_float2(1.f, 1.f), su = make_float2(1.f, 1.f);
      if constexpr (FP8) {
        if (warp == (j & (kRedSlots - 1))) {
          const float* sp = a.s_gu + (size_t)rt.grp_expert[g] * 2 * a.I + 8 * tt + (WA ? g4 : 2 * t4);
          if constexpr (WA) {
            sg.x = __ldg(sp);
            su.x = __ldg(sp + a.I);
          } else {
            sg = __ldg(reinterpret_cast<const float2*>(sp));
            su = __ldg(reinterpret_cast<const float2*>(sp + a.I));
          }
        }
      }
      if (!warp_wait(full(s), ph, &waited, a.wait_ns)) {
        record_timeout(a.ws, 2, kErrTimeoutFull, j, S, full(s), waited);
        break;
      }
      if (j == 0 && tid == 0) stamp(a, 4);
      // bf16: c0, c1 = the two k-steps of the one n8 block.  fp8 with weights
      // as A: c0, c1 = the two k-steps; weights as B: c0 = the gate block,
      // c1 = the up block, each over both k-steps
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
      const uint4* wp = reinterpret_cast<const uint4*>(ring + (size_t)s * a.gu_tile) + (warp * KPW) * 32 + lane;
#pragma unroll
      for (int q = 0; q < KPW; ++q) {
        const uint4 b = wp[q * 32];
        if constexpr (WA) {  // b.x, b.y: gate row 8 tt + g4 (8 codes); b.z, b.w: up row 8 tt + g4
          uint32_t g0, g1, g2, g3, u0, u1, u2, u3;
          e4m3x4_to_f16x2(b.x, g0, g1);
          e4m3x4_to_f16x2(b.y, g2, g3);
          e4m3x4_to_f16x2(b.z, u0, u1);
          e4m3x4_to_f16x2(b.w, u2, u3);
          mma_f16(c0, g0, u0, g1, u1, xa[q].x, xa[q].y);
          mma_f16(c1, g2, u2, g3, u3, xa[q].z, xa[q].w);
        } else if constexpr (FP8) {  // the same codes, as the B columns of the gate and up blocks
          uint32_t f0, f1, f2, f3;
          e4m3x4_to_f16x2(b.x, f0, f1);
          e4m3x4_to_f16x2(b.y, f2, f3);
          mma_f16(c0, xa[q].x, xb[q].x, xa[q].y, xb[q].y, f0, f1);
          mma_f16(c0, xa[q].z, xb[q].z, xa[q].w, xb[q].w, f2, f3);
          e4m3x4_to_f16x2(b.z, f0, f1);
          e4m3x4_to_f16x2(b.w, f2, f3);
          mma_f16(c1, xa[q].x, xb[q].x, xa[q].y, xb[q].y, f0, f1);
          mma_f16(c1, xa[q].z, xb[q].z, xa[q].w, xb[q].w, f2, f3);
        } else {
          const uint4 xh = TWO ? xb[q] : xa[q];  // A rows 8..15
          mma_bf16(c0, xa[q].x, xh.x, xa[q].y, xh.y, b.x, b.y);
          mma_bf16(c1, xa[q].z, xh.z, xa[q].w, xh.w, b.z, b.w);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(s));  // stage free for the producer

      const int slot = j & (kRedSlots - 1);
      if constexpr (NB == 2) {
        red[((slot * kConsumerWarps + warp) * 32 + lane) * NB] = make_float4(c0[0], c0[1], c0[2], c0[3]);
        red[((slot * kConsumerWarps + warp) * 32 + lane) * NB + 1] = make_float4(c1[0], c1[1], c1[2], c1[3]);
      } else {
        red[(slot * kConsumerWarps + warp) * 32 + lane] =
            make_float4(c0[0] + c1[0], c0[1] + c1[1], c0[2] + c1[2], c0[3] + c1[3]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(redbar(slot));
      if (warp == slot) {  // this tile's reducer (rotates over the warps)
        if (!warp_wait(redbar(slot), (uint32_t)(j >> 3) & 1u, &waited, a.wait_ns)) {
          record_timeout(a.ws, 2, kErrTimeoutReduce, j, S, redbar(slot), waited);
          break;
        }
        float4 acc[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          acc[b] = red[((slot * kConsumerWarps) * 32 + lane) * NB + b];
#pragma unroll
          for (int w2 = 1; w2 < kConsumerWarps; ++w2) {
            const float4 v = red[((slot * kConsumerWarps + w2) * 32 + lane) * NB + b];
            acc[b].x += v.x;
            acc[b].y += v.y;
            acc[b].z += v.z;
            acc[b].w += v.w;
          }
        }
        // the row scales after the sums, then SwiGLU and ONE bf16 rounding
        if constexpr (WA) {
          // (x, y) = gate of intermediate row 8 tt + g4 for group tokens 2 t4,
          // 2 t4 + 1; (z, w) = up of the same row and tokens
          const int r = 8 * tt + g4, n = 2 * t4;
          const float4 v = acc[0];
          if (n < cnt) a.ws.h[(size_t)(start + n) * a.I + r] = __float2bfloat16_rn(silu(sg.x * v.x) * (su.x * v.z));
          if (n + 1 < cnt)
            a.ws.h[(size_t)(start + n + 1) * a.I + r] = __float2bfloat16_rn(silu(sg.x * v.y) * (su.x * v.w));
        } else if constexpr (FP8) {
          // gate acc[0], up acc[1]: (x, y) = group token g4, intermediate rows
          // 8 tt + 2 t4 and + 1; (z, w) = token g4 + 8
          const int r = 8 * tt + 2 * t4;
          const float4 gt = acc[0], up = acc[1];
          if (g4 < cnt)
            *reinterpret_cast<__nv_bfloat162*>(a.ws.h + (size_t)(start + g4) * a.I + r) = __floats2bfloat162_rn(
                silu(sg.x * gt.x) * (su.x * up.x), silu(sg.y * gt.y) * (su.y * up.y));
          if (g4 + 8 < cnt)
            *reinterpret_cast<__nv_bfloat162*>(a.ws.h + (size_t)(start + g4 + 8) * a.I + r) = __floats2bfloat162_rn(
                silu(sg.x * gt.z) * (su.x * up.z), silu(sg.y * gt.w) * (su.y * up.w));
        } else {
          // (x, y) = (gate, up) of group token g4, intermediate row 4 tt + t4;
          // (z, w) the same for token g4 + 8
          const int r = (GU_ROWS / 2) * tt + t4;
          const float4 v = acc[0];
          if (g4 < cnt) a.ws.h[(size_t)(start + g4) * a.I + r] = __float2bfloat16_rn(silu(v.x) * v.y);
          if (g4 + 8 < cnt) a.ws.h[(size_t)(start + g4 + 8) * a.I + r] = __float2bfloat16_rn(silu(v.z) * v.w);
        }
      }
      if (j == n_static - 1) {  // every static tile of this warp's share is reduced
        __syncwarp();
        if (lane == 0) mbar_arrive(static_bar);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(done);
    if (tid == 0) stamp(a, 5);
  }

  // (this CTA's h rows are all written: the `done` barrier tells the
  // publisher, and the producer holds back each down tile until its group
  // is ready -- the consumers go straight on)

  {
    // ---- 5. down GEMV, weighted rows y[pair] = w_pair * (W_d h_pair);
    // warp w takes cell w of every super tile: SPW consecutive output slabs
    const int kpd = a.I / 32;  // 32-wide k chunks of a down row (<= kMaxDownChunks)
    uint4 ha[kMaxDownChunks], hb[kMaxDownChunks];  // h rows of group tokens g4, g4 + 8 (TB = 1: g4)
    // the pairs this lane stores: weights as A, group tokens 2 t4 and
    // 2 t4 + 1; otherwise tokens g4 and g4 + 8
    int pid[2] = {-1, -1};
    float pw[2] = {0.f, 0.f};
    int cur_g = -1, cur_de = 0;
    // the instances for calls of at most 8 tokens write tagged rows (see the combine)
    const unsigned ytag = (unsigned)*call_idx;
    auto put1 = [&](int p, int col, float v) {  // column col of pair p's weighted row
      if constexpr (kTaggedRows)
        put_y(a.ws.yt + (size_t)p * a.H + col, v, ytag);
      else
        a.ws.y[(size_t)p * a.H + col] = v;
    };
    auto put2 = [&](int p, int col, float v0, float v1) {  // columns col, col + 1
      if constexpr (kTaggedRows) {
        put_y(a.ws.yt + (size_t)p * a.H + col, v0, ytag);
        put_y(a.ws.yt + (size_t)p * a.H + col + 1, v1, ytag);
      } else {
        *reinterpret_cast<float2*>(a.ws.y + (size_t)p * a.H + col) = make_float2(v0, v1);
      }
    };
    for (int j = 0;; ++j) {
      const int s = j % SD;
      const uint32_t ph = (uint32_t)(j / SD) & 1u;
      if (!warp_wait(dready(s), ph, &waited, a.wait_ns)) {
        record_timeout(a.ws, 3, kErrTimeoutFull, j, SD, dready(s), waited);
        break;
      }
      const int tile = dstage_tile[s];
      if (tile < 0) break;
      const int g = tile / SPG;
      const int cl = (tile - g * SPG) * NSL + warp;  // this warp's cell: slabs cl SPW .. cl SPW + SPW - 1
      if (g != cur_g) {
        const int start = rt.grp_start[g], cnt = rt.grp_cnt[g];
        const uint4* h0 =
            reinterpret_cast<const uint4*>(a.ws.h + (size_t)(start + (g4 < cnt ? g4 : 0)) * a.I) + t4;
        const uint4* h1 =
            reinterpret_cast<const uint4*>(a.ws.h + (size_t)(start + (g4 + 8 < cnt ? g4 + 8 : 0)) * a.I) + t4;
#pragma unroll
        for (int q = 0; q < kMaxDownChunks; ++q) {
          if (q < kpd) {
            ha[q] = __ldcg(h0 + 4 * q);  // written by other SMs in this grid: L2, not L1
            if constexpr (TWO) hb[q] = __ldcg(h1 + 4 * q);
            if constexpr (FP8) {
              ha[q] = bf16x8_to_f16x8(ha[q]);
              if constexpr (TWO) hb[q] = bf16x8_to_f16x8(hb[q]);
            }
          }
        }
        if constexpr (FP8) cur_de = rt.grp_expert[g];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int n = WA ? 2 * t4 + i : g4 + 8 * i;
          pid[i] = n < cnt ? rt.pair_list[start + n] : -1;
          pw[i] = pid[i] >= 0 ? rt.s_w[pid[i]] : 0.f;
        }
        cur_g = g;
      }
      // fp8 scales of slab sl's output rows: weights as A, rows 16 sl + g4 and
      // + 8 in (rs.x, rs.y); as B, rows 16 sl + 8 b + 2 t4 and + 1 of block b
      // in (rs.x, rs.y) and (rs.z, rs.w)
      auto row_scales = [&](int sl) -> float4 {
        float4 r = make_float4(1.f, 1.f, 1.f, 1.f);
        if constexpr (WA) {
          const float* sd = a.s_d + (size_t)cur_de * a.H + sl * D_ROWS + g4;
          r.x = __ldg(sd);
          r.y = __ldg(sd + 8);
        } else if constexpr (FP8) {
          const float* sd = a.s_d + (size_t)cur_de * a.H + sl * D_ROWS + 2 * t4;
          const float2 r0 = __ldg(reinterpret_cast<const float2*>(sd));
          const float2 r1 = __ldg(reinterpret_cast<const float2*>(sd + 8));
          r = make_float4(r0.x, r0.y, r1.x, r1.y);
        }
        return r;
      };
      // The cell's NS slabs.  A compile-time 1 (no loop) in every instance but
      // bf16 with TB = 1, whose cells hold SPW slabs (run-time: more than one
      // where I < 512).  A looping copy of this body costs the other
      // instances registers (spills at TB = 2) or, in the fp8 consumers,
      // which are bound by their own instructions, measurable time.
      auto consume_cell = [&](auto ns) -> bool {
        const int NS = ns;
        float4 rs = row_scales(cl * NS);  // the first slab's, while the data lands
        if (!warp_wait(dfull(s), ph, &waited, a.wait_ns)) {
          record_timeout(a.ws, 3, kErrTimeoutFull, j, SD, dfull(s), waited);
          return false;
        }
        if (j == 0 && tid == 0) stamp(a, 14);
        const uint4* bp =
            reinterpret_cast<const uint4*>(ring + (size_t)cell_tab[s * kConsumerWarps + warp] * a.d_tile) + lane;
        for (int u = 0; u < NS; ++u) {
          const int sl = cl * NS + u;
          if (u > 0) rs = row_scales(sl);
          // bf16 and fp8 with weights as A: c0, c1 = the two k-steps; fp8 with
          // weights as B: c0, c1 = the slab's two 8-row blocks
          float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
  #pragma unroll
          for (int q = 0; q < kMaxDownChunks; ++q) {
            if (q < kpd) {
              const uint4 b = bp[(u * kpd + q) * 32];
              if constexpr (WA) {  // b.x, b.y: output row 16 sl + g4; b.z, b.w: row 16 sl + 8 + g4
                uint32_t p0, p1, p2, p3, r0, r1, r2, r3;
                e4m3x4_to_f16x2(b.x, p0, p1);
                e4m3x4_to_f16x2(b.y, p2, p3);
                e4m3x4_to_f16x2(b.z, r0, r1);
                e4m3x4_to_f16x2(b.w, r2, r3);
                mma_f16(c0, p0, r0, p1, r1, ha[q].x, ha[q].y);
                mma_f16(c1, p2, r2, p3, r3, ha[q].z, ha[q].w);
              } else if constexpr (FP8) {  // the same codes, as the B columns of the two blocks
                uint32_t f0, f1, f2, f3;
                e4m3x4_to_f16x2(b.x, f0, f1);
                e4m3x4_to_f16x2(b.y, f2, f3);
                mma_f16(c0, ha[q].x, hb[q].x, ha[q].y, hb[q].y, f0, f1);
                mma_f16(c0, ha[q].z, hb[q].z, ha[q].w, hb[q].w, f2, f3);
                e4m3x4_to_f16x2(b.z, f0, f1);
                e4m3x4_to_f16x2(b.w, f2, f3);
                mma_f16(c1, ha[q].x, hb[q].x, ha[q].y, hb[q].y, f0, f1);
                mma_f16(c1, ha[q].z, hb[q].z, ha[q].w, hb[q].w, f2, f3);
              } else {
                const uint4 hh = TWO ? hb[q] : ha[q];  // A rows 8..15
                mma_bf16(c0, ha[q].x, hh.x, ha[q].y, hh.y, b.x, b.y);
                mma_bf16(c1, ha[q].z, hh.z, ha[q].w, hh.w, b.z, b.w);
              }
            }
          }
          if (u == NS - 1) {
            __syncwarp();  // every lane has read the whole cell
            if (lane == 0) mbar_arrive(dempty(s));
          }
          if constexpr (WA) {
            // c0 + c1: (rows 16 sl + g4 | 16 sl + 8 + g4) x (tokens 2 t4, 2 t4 + 1)
            const int row = sl * D_ROWS + g4;
  #pragma unroll
            for (int i = 0; i < 2; ++i)
              if (pid[i] >= 0) {
                put1(pid[i], row, pw[i] * (rs.x * (c0[i] + c1[i])));
                put1(pid[i], row + 8, pw[i] * (rs.y * (c0[2 + i] + c1[2 + i])));
              }
          } else if constexpr (FP8) {
            // block b: (token g4 | g4 + 8) x (rows 16 sl + 8 b + 2 t4, + 1)
            const int row = sl * D_ROWS + 2 * t4;
  #pragma unroll
            for (int b = 0; b < 2; ++b) {
              const float* v = b ? c1 : c0;
              const float sx = b ? rs.z : rs.x, sy = b ? rs.w : rs.y;
              if (pid[0] >= 0) put2(pid[0], row + 8 * b, pw[0] * (sx * v[0]), pw[0] * (sy * v[1]));
              if (pid[1] >= 0) put2(pid[1], row + 8 * b, pw[1] * (sx * v[2]), pw[1] * (sy * v[3]));
            }
          } else {
            // C: (token g4 | g4 + 8) x (output rows 2 t4, 2 t4 + 1 of the slab)
            const int row = sl * D_ROWS + 2 * t4;
            if (pid[0] >= 0) put2(pid[0], row, pw[0] * (c0[0] + c1[0]), pw[0] * (c0[1] + c1[1]));
            if (pid[1] >= 0) put2(pid[1], row, pw[1] * (c0[2] + c1[2]), pw[1] * (c0[3] + c1[3]));
          }
        }
        return true;
      };
      bool cell_ok;
      if constexpr (FP8 || TWO)
        cell_ok = consume_cell(OneSlab{});
      else
        cell_ok = consume_cell(SPW);
      if (!cell_ok) break;
    }
    if (tid == 0) stamp(a, 7);
  }

  // ---- 6. combine.  Only the first n_own_ctas CTAs combine (3 output
  // slabs each: CTA c owns 3c .. 3c+2): each token's k rows summed in slot
  // order, ONE bf16 rounding.  The other CTAs leave at once, so the next
  // call's CTAs get their SMs (and run their prologue) while the combine
  // runs.  (Three slabs a CTA measured faster than eight: the combine is a
  // latency-bound read of L2, so more CTAs end it sooner, and at hidden 2560
  // about 45 SMs are still left to the next call's prologue.)  Every CTA
  // counts itself in once per call: the next call takes its index from that
  // count.
  // The instances for calls of at most 8 tokens (TB = 1): every weighted
  // row value carries the index of the call that wrote it (one 64-bit
  // store), so an owner polls the values it needs (bounded) and starts as
  // soon as they are there -- no fence, no count round trip after the last
  // row.  The others write plain fp32 rows (half the bytes and stores;
  // measured: at 64 tokens the doubled row traffic cost more than the round
  // trip saves, and the fp8 consumers of 9..16 tokens, bound by their own
  // instructions, lost more to the wider stores than the combine gained)
  // and the owners wait for every CTA's count first.
  const int SLc = a.H / kDownTileRows;  // 8-row output slabs of the combine
  constexpr int kCombineSlabs = 3;
  const int n_own_ctas = min((int)gridDim.x, (SLc + kCombineSlabs - 1) / kCombineSlabs);
  const int own_per = (SLc + n_own_ctas - 1) / n_own_ctas;  // kCombineSlabs unless the grid is small
  const bool owner = (int)blockIdx.x < n_own_ctas;
  if constexpr (kTaggedRows) {
    if (tid == 0) asm volatile("red.relaxed.gpu.global.add.u64 [%0], 1;" ::"l"(a.ws.sync + kSyncCount) : "memory");
    if (!owner) return;
  } else {
    consumers_sync();  // every weighted row of this CTA written
    if (tid == 0) {
      grid_count(a.ws.sync + kSyncCount);
      if (owner) grid_wait(a.ws, a.ws.sync + kSyncCount, *call_idx * gridDim.x, 3, a.wait_ns);
    }
    if (!owner) return;
    consumers_sync();
  }
  if (tid == 0) stamp(a, 15);
  const unsigned ctag = (unsigned)*call_idx;
  const int nthr = kConsumerWarps * 32;
  const int sl0 = (int)blockIdx.x * own_per;
  const int n_own = max(0, min(own_per, SLc - sl0));
  const int per = a.M * kDownTileRows;
  const int KS = a.K + (shared ? 1 : 0);  // the shared slot (pair MK + m) last
  bool waiting_ok = true;
  for (int it = tid; it < n_own * per; it += nthr) {
    const int sl = sl0 + it / per;
    const int m = (it % per) / kDownTileRows;
    const int r = sl * kDownTileRows + (it % kDownTileRows);
    float sum = 0.f;
    if constexpr (!kTaggedRows) {
      const float* yr = a.ws.y + (size_t)m * a.K * a.H + r;
      const float vs = shared ? __ldcg(a.ws.y + (size_t)(MK + m) * a.H + r) : 0.f;  // the shared slot
      for (int k0 = 0; k0 < a.K; k0 += 8) {  // 8 loads in flight, summed in slot order
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = k0 + i < a.K ? __ldcg(yr + (size_t)(k0 + i) * a.H) : 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (k0 + i < a.K) sum += v[i];
      }
      if (shared) sum += vs;  // the shared slot, last
    } else {
      auto pair_of = [&](int j) { return j < a.K ? m * a.K + j : MK + m; };
      for (int k0 = 0; k0 < KS; k0 += 8) {  // 8 values in flight, summed in slot order
        unsigned long long v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          v[i] = k0 + i < KS ? ld_relaxed64(a.ws.yt + (size_t)pair_of(k0 + i) * a.H + r) : ((unsigned long long)ctag << 32);
        bool all = true;
#pragma unroll
        for (int i = 0; i < 8; ++i) all = all && (unsigned)(v[i] >> 32) == ctag;
        if (!all && waiting_ok) {  // not all written yet: poll the missing ones (bounded)
          const unsigned long long t0 = global_timer_ns();
          while (!all) {
            __nanosleep(32);
            all = true;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if ((unsigned)(v[i] >> 32) != ctag) {
                v[i] = ld_relaxed64(a.ws.yt + (size_t)pair_of(k0 + i) * a.H + r);
                all = all && (unsigned)(v[i] >> 32) == ctag;
              }
            if (!all && global_timer_ns() - t0 > a.wait_ns) {
              record_timeout(a.ws, 3, kErrTimeoutGrid, it, 0, 0, global_timer_ns() - t0);
              waiting_ok = false;  // the call's result is undefined; finish without waiting
              break;
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (k0 + i < KS) sum += __uint_as_float((unsigned)v[i]);
      }
    }
    if (a.out_f32)
      a.out_f32[(size_t)m * a.H + r] = sum;  // a partial of a split layer: rounded after the sum of the parts
    else
      a.out[(size_t)m * a.H + r] = __float2bfloat16_rn(sum);
  }
  if (tid == 0) stamp(a, 8);
}

}  // namespace wse
