// common.cuh -- sm_103a building blocks of the layer kernel: mbarrier +
// bulk-copy (TMA) staging, Programmatic Dependent Launch control, the bf16
// tensor-core MMA, and the device workspace of a layer handle.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace wse {

// ------------------------------------------------------------ limits ----
constexpr int kMaxTokens = 64;        // M per forward call
constexpr int kMaxTopk = 32;          // k
constexpr int kMaxExperts = 1024;     // E
constexpr int kMaxPairs = kMaxTokens * kMaxTopk;
constexpr int kGroupTokens = 16;      // pairs per compaction group (one m16 / 2 x n8 tile)
constexpr int kConsumerWarps = 8;
constexpr int kProducerWarp = kConsumerWarps;      // warp 8: stages every weight tile
constexpr int kPublisherWarp = kConsumerWarps + 1; // warp 9: grid-wide arrivals and readiness
constexpr int kExpertThreads = (kConsumerWarps + 2) * 32;
constexpr int kGateUpTileRows = 8;    // 4 gate rows interleaved with their 4 up rows
constexpr int kDownTileRows = 8;      // 8 output rows (n8) x I per down tile
constexpr int kMaxGateUpStages = 7;   // < 8 reduction slots: see the reduction-slot argument
constexpr int kMaxDownStages = 8;     // down slots (ring regions of one 8-slab super tile)
constexpr int kMaxDownChunks = 16;    // 32-wide k chunks of a down row: I <= 512
constexpr uint32_t kBulkChunk = 65536;  // bytes per cp.async.bulk (fewer, larger copies: each
                                        // issue costs the producer shared-memory pipe slots)
constexpr int kTraceSlots = 32;       // per-CTA phase timestamps of a traced call

// Grid-wide synchronisation words (unsigned, 128 bytes apart).  The 64-bit
// counts are never reset: each call adds exactly one arrival per CTA to each
// of them.  A call starts only once the previous call on the same workspace
// has completed (stream order, or the PDL dependency wait), so every CTA
// reads the same kSyncCount at its start: count / grid = calls completed,
// which gives the call's index (1, 2, ...) and every later target.  The two
// work counters come in two sets used by odd and even calls; each call
// clears the other set for the next one.
enum : int {
  kSyncCount = 0,         // 64-bit: arrivals before the combine (one per CTA per call)
  kSyncGateUpNext = 32,   // next gate/up tile of the dynamically shared tail (even calls)
  kSyncDownNext = 64,     // next down super tile of the dynamically shared tail (even calls)
  kSyncStaticDone = 96,   // 64-bit: CTAs whose statically assigned gate/up tiles are reduced
  kSyncGateUpDone = 128,  // 64-bit: CTAs whose gate/up tiles are all reduced
  kSyncGateUpNextOdd = 160,
  kSyncDownNextOdd = 192,
  kSyncWords = 224,
};

// A bounded wait gives up after this long by default (the kernels run for
// microseconds; reaching it means a bug or an SM held by other work, never a
// slow call).  A layer handle can set a shorter limit for its own kernel.
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

// Bits of the sticky device status word.
enum : int {
  kErrTimeoutFull = 1,    // consumer waited too long for a staged tile
  kErrTimeoutEmpty = 2,   // producer waited too long for a free stage
  kErrTimeoutReduce = 4,  // gate/up reducer waited too long for partials
  kErrBadIndex = 8,       // the top-k found no candidate (cannot happen while k <= E)
  kErrTimeoutGrid = 16,   // a grid-wide wait (barrier, h rows, slab arrivals) ran out
};

// Device workspace of one layer handle (all device pointers).
struct Workspace {
  int* status;               // [1] sticky error bits
  unsigned long long* diag;  // [4] first timeout: where, elapsed ns, raw barrier word, thread/grid
  unsigned* sync;            // [kSyncWords] grid-wide counters, see above
  float* part;               // [2][ks][kMaxTokens][E] partial router logits (odd / even calls)
  int* n_groups;             // [1] copy of the call's compaction (inspection only)
  int* n_active;             // [1]
  int* grp_expert;           // [kMaxPairs]
  int* grp_start;            // [kMaxPairs] first sorted position of the group
  int* grp_cnt;              // [kMaxPairs] pairs in the group (1..16)
  int* pair_list;            // [kMaxPairs] pair id (token*k + slot) at each sorted position
  float* pair_w;             // [kMaxPairs] routing weight by pair id
  __nv_bfloat16* h;          // [kMaxPairs][I] SwiGLU rows, sorted-position order
  float* y;                  // [kMaxPairs][H] weighted down-projection rows, by pair id
  unsigned long long* yt;    // [kGroupTokens (k + 1)][H] the same for calls of at most kGroupTokens
                             // tokens: fp32 bits in the low word, the writing call's index (mod 2^32)
                             // in the high word
  unsigned long long* xtopk; // [2][kMaxTokens * kMaxTopk] routed slots of calls with more tokens than
                             // a CTA has warps (odd / even calls): expert id in the high word, weight
                             // bits in the low word, all ones while unwritten
  unsigned long long* trace; // [grid][kTraceSlots] phase timestamps (traced calls)
};

// ------------------------------------------------------------- PTX -----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic Dependent Launch.  wait: block until every prerequisite grid
// has completed and its memory is visible.  launch_dependents: allow the
// next grid in the stream to be scheduled (its own wait still fences on our
// completion).  Both are no-ops for a launch without the PDL attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same with a suspend-time hint: the thread sleeps until the phase
// completes (or the hint elapses) instead of polling, which leaves the
// shared-memory pipe to the warps that work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
constexpr uint32_t kSuspendHintNs = 20000;
// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase with the given parity to complete; false after `limit`
// ns (the caller records an error bit and leaves its loop).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long* waited = nullptr,
                                          unsigned long long limit = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kSuspendHintNs)) return true;
    const unsigned long long dt = global_timer_ns() - t0;
    if (dt > limit) {
      if (waited) *waited = dt;
      return false;
    }
  }
}

// Warp-uniform bounded wait: every lane waits and the lanes agree on the
// outcome by vote, so a timeout never splits the warp before a .aligned
// instruction (mma.sync) or a __syncwarp().
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, unsigned long long* waited,
                                          unsigned long long limit = kWaitTimeoutNs) {
  const bool ok = mbar_wait(bar, parity, waited, limit);
  return __all_sync(0xffffffffu, ok);
}

// Order this thread's earlier generic-proxy shared-memory accesses before its
// later async-proxy (bulk copy) accesses -- needed before refilling a stage
// that was just read with ordinary loads.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bulk (TMA) copy global -> shared, completion counted in bytes on `bar`.
// dst, src and bytes must be multiples of 16.
// L2 policy for data read once per call (the expert weights): evict it
// first, so that what every call re-reads -- the kernel's code, the tokens,
// the router weights, the partial logits, h and y -- stays in L2 while
// hundreds of MB of weights stream past.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s_chunked(uint32_t dst, const uint8_t* src, uint32_t bytes,
                                                 uint32_t bar, uint64_t policy) {
  for (uint32_t off = 0; off < bytes; off += kBulkChunk) {
    uint32_t n = bytes - off < kBulkChunk ? bytes - off : kBulkChunk;
    bulk_g2s(dst + off, src + off, n, bar, policy);
  }
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16x2 (low element first in memory) -> two fp32, exact.
// D = A(16x16, row) * B(16x8, col) + D, f16 inputs, fp32 accumulate (the
// fp8-weight path: codes and activations are exact in f16).
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four E4M3 codes (bytes 0..3 of v) -> two f16x2 in the same element order
// (bytes 0, 1 -> lo; 2, 3 -> hi).  Exact: every E4M3 value is an f16 value.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t v, uint32_t& lo, uint32_t& hi) {
  asm("{ .reg .b16 p, q; mov.b32 {p, q}, %2; cvt.rn.f16x2.e4m3x2 %0, p; cvt.rn.f16x2.e4m3x2 %1, q; }"
      : "=r"(lo), "=r"(hi)
      : "r"(v));
}

// bf16x2 -> f16x2, element order kept; exact for values in f16's normal
// range (bf16's 8-bit significand fits f16's 11).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(__uint_as_float(v & 0xffff0000u)), "f"(__uint_as_float(v << 16)));
  return d;
}
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  return make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ void set_error(int* status, int bits) { atomicOr(status, bits); }

__device__ __forceinline__ unsigned long long mbar_raw(uint32_t bar) {
  unsigned long long v;
  asm volatile("ld.shared.b64 %0, [%1];" : "=l"(v) : "r"(bar) : "memory");
  return v;
}

// Record the first bounded-wait timeout of a call (phase 1 router / 2
// gate-up / 3 down, wait kind = the status bit, CTA, loop index, ring depth)
// and its evidence.
__device__ __forceinline__ void record_timeout(const Workspace& ws, int kernel, int kind, int j,
                                               int stages, uint32_t bar, unsigned long long waited) {
  const unsigned long long where = ((unsigned long long)kernel << 56) |
                                   ((unsigned long long)kind << 48) |
                                   ((unsigned long long)blockIdx.x << 32) |
                                   ((unsigned long long)(stages & 0xffff) << 16) | (unsigned)(j & 0xffff);
  if (atomicCAS(ws.diag, 0ull, where) == 0ull) {
    ws.diag[1] = waited;
    ws.diag[2] = mbar_raw(bar);
    ws.diag[3] = ((unsigned long long)threadIdx.x << 32) | (unsigned)gridDim.x;
  }
  set_error(ws.status, kind);
}

}  // namespace wse
