// moe_api.cu -- host runtime behind include/moe.h: argument checks, weight
// re-layout at create, workspace, the layer kernel's launch (PDL-chained to
// the previous work on the stream), and the per-(handle, M) CUDA graph
// cache.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <string>

#include "kernels.cuh"
#include "moe.h"
#include "routing.cuh"

using namespace wse;

namespace {

thread_local std::string g_last_error;

void set_err(const char* fmt, ...) __attribute__((format(printf, 1, 2)));
void set_err(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side fault injection for tests: MOE_FAULT_INJECT=alloc:N makes the
// N-th device allocation of a moe_create call fail (N >= 1).
struct AllocCounter {
  int fail_at = 0, n = 0;
  AllocCounter() {
    const char* s = std::getenv("MOE_FAULT_INJECT");
    if (s && std::strncmp(s, "alloc:", 6) == 0) fail_at = std::atoi(s + 6);
  }
  cudaError_t alloc(void** p, size_t bytes) {
    ++n;
    if (fail_at > 0 && n == fail_at) {
      *p = nullptr;
      return cudaErrorMemoryAllocation;
    }
    return cudaMalloc(p, bytes);
  }
};

struct GraphEntry {
  cudaGraphExec_t exec = nullptr;
  const void* x = nullptr;
  void* out = nullptr;
  int32_t* idx = nullptr;
  float* tw = nullptr;
  unsigned flags = 0;
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// One launch configuration of the layer kernel: the instance and its
// shared-memory rings, sized for calls of up to max_tokens tokens.
struct LayerPlan {
  LayerKernel kernel = nullptr;
  int max_tokens = 0;
  int d_spw = 1;            // down slabs per cell
  uint32_t tile_d = 0;      // down cell bytes
  int s_gu = 0, s_d = 0;    // gate/up ring depth, down stages
  uint32_t ring_bytes = 0;
  size_t smem_max = 0;      // dynamic shared memory at M = max_tokens
};

}  // namespace

struct moe_layer {
  int H = 0, E = 0, K = 0, I = 0;
  int shared = 0;           // 1: expert E (packed after the routed ones) is a shared expert
  float routed_scale = 1.0f;
  int sel_only = 0;         // the router bias picks the experts only
  int fp8 = 0;              // expert weights are E4M3 codes with per-row scales
  float* sc_gu = nullptr;   // fp8: [E][2I] gate/up row scales
  float* sc_d = nullptr;    // fp8: [E][H] down row scales
  int kp() const { return K + shared; }  // pairs per token
  int ea() const { return E + shared; }  // packed experts
  int dev = 0, n_sms = 0;
  int grid = 0;             // CTAs of a layer launch (all SMs unless moe_set_grid chose fewer)
  unsigned long long wait_ns = kWaitTimeoutNs;  // limit of the kernel's bounded waits
  __nv_bfloat16* w_router = nullptr;
  uint8_t* w_gu = nullptr;  // packed gate/up tiles
  uint8_t* w_d = nullptr;   // packed down tiles
  float* bias = nullptr;
  void* ws_mem = nullptr;
  size_t ws_bytes = 0, weight_bytes = 0, yt_bytes = 0;
  Workspace ws{};
  int ks = 1;               // hidden-dim split of the router matvec
  uint32_t tile_gu = 0;     // gate/up tile bytes
  // plan[0] serves every M, plan[1] calls with M <= 8 (groups of at most 8
  // tokens: one token block -- half the token registers; fp8: half the
  // MMAs and half the reduction area)
  LayerPlan plan[2];
  const LayerPlan& plan_for(int M) const { return M <= plan[1].max_tokens ? plan[1] : plan[0]; }
  std::map<int, GraphEntry> graphs;
  cudaStream_t cap_stream = nullptr;
};

namespace {

void drop_graphs(moe_layer* h);

void free_layer(moe_layer* h) {
  if (!h) return;
  drop_graphs(h);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  cudaFree(h->w_router);
  cudaFree(h->w_gu);
  cudaFree(h->w_d);
  cudaFree(h->sc_gu);
  cudaFree(h->sc_d);
  cudaFree(h->bias);
  cudaFree(h->ws_mem);
  delete h;
}

void drop_graphs(moe_layer* h) {
  for (auto& kv : h->graphs)
    if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
  h->graphs.clear();
}

int cuda_fail(cudaError_t e, const char* what) {
  set_err("%s: %s", what, cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

// Arrival counts from zero, every partial logit of both buffers unwritten
// (the state moe_create leaves).  Only while no kernel of the handle runs.
constexpr size_t kXtopkBytes = 2 * (size_t)kMaxTokens * kMaxTopk * 8;  // the exchanged top-k slots

void restart_counts(moe_layer* h) {
  cudaMemset(h->ws.sync, 0, kSyncWords * 4);
  cudaMemset(h->ws.yt, 0, h->yt_bytes);  // call indices restart at 1: no row may carry an old one
  cudaMemset(h->ws.part, 0xff, 2 * (size_t)h->ks * kMaxTokens * h->E * 4);
  cudaMemset(h->ws.xtopk, 0xff, kXtopkBytes);  // every exchanged slot unwritten
}

// Enqueue the layer kernel.  ev (2 events) brackets it for profiling; the
// records are external event nodes when the stream is being captured.
int launch_layer(moe_layer* h, const void* x, void* out, int32_t* idx, float* tw, int M,
                 cudaStream_t st, bool pdl, bool trace, cudaEvent_t* ev, unsigned flags = 0u) {
  const LayerPlan& pl = h->plan_for(M);
  LayerArgs la{};
  la.x = static_cast<const __nv_bfloat16*>(x);
  la.w_router = h->w_router;
  la.bias = h->bias;
  la.w_gate_up = h->w_gu;
  la.w_down = h->w_d;
  la.s_gu = h->sc_gu;
  la.s_d = h->sc_d;
  const bool f32 = (flags & MOE_FWD_OUT_F32) != 0;
  la.out = f32 ? nullptr : static_cast<__nv_bfloat16*>(out);
  la.out_f32 = f32 ? static_cast<float*>(out) : nullptr;
  la.topk_idx = idx;
  la.topk_w = tw;
  la.M = M; la.H = h->H; la.E = h->E; la.K = h->K; la.I = h->I;
  la.ks = h->ks;
  la.gu_stages = pl.s_gu;
  la.d_stages = pl.s_d;
  la.gu_tile = h->tile_gu;
  la.d_tile = pl.tile_d;
  la.d_spw = pl.d_spw;
  la.ring_bytes = pl.ring_bytes;
  la.trace = trace ? 1 : 0;
  la.shared = h->shared;
  la.routed_scale = h->routed_scale;
  la.sel_only = h->sel_only;
  la.wait_ns = h->wait_ns;
  la.test_flags = (flags & MOE_FWD_TEST_SKIP_ARRIVAL) ? kTestSkipArrival : 0;
  la.ws = h->ws;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c{};
  c.stream = st;
  c.attrs = pdl ? attr : nullptr;
  c.numAttrs = pdl ? 1 : 0;
  c.gridDim = dim3(h->grid);
  c.blockDim = dim3(kExpertThreads);
  c.dynamicSmemBytes = layer_smem_bytes(pl.ring_bytes, M * h->kp(), h->ea());

  cudaError_t e;
  unsigned ev_flags = cudaEventRecordDefault;
  if (ev) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if ((e = cudaStreamIsCapturing(st, &cs)) != cudaSuccess) return cuda_fail(e, "capture status");
    if (cs == cudaStreamCaptureStatusActive) ev_flags = cudaEventRecordExternal;
  }
  if (ev && (e = cudaEventRecordWithFlags(ev[0], st, ev_flags)) != cudaSuccess) return cuda_fail(e, "event record");
  if ((e = cudaLaunchKernelEx(&c, pl.kernel, la)) != cudaSuccess) return cuda_fail(e, "layer kernel launch");
  if (ev && (e = cudaEventRecordWithFlags(ev[1], st, ev_flags)) != cudaSuccess) return cuda_fail(e, "event record");
  return MOE_OK;
}

int check_forward_args(moe_layer* h, const void* x, const void* out, const int32_t* idx, int M,
                       unsigned flags = 0u) {
  if (!h) { set_err("null handle"); return MOE_ERR_INVALID_ARG; }
  if (M < 0) { set_err("M = %d < 0", M); return MOE_ERR_INVALID_ARG; }
  if (M > MOE_MAX_TOKENS) { set_err("M = %d exceeds %d", M, MOE_MAX_TOKENS); return MOE_ERR_UNSUPPORTED; }
  if (M == 0) return MOE_OK;
  if (!x || !out || !idx) { set_err("null x/out/topk_idx"); return MOE_ERR_INVALID_ARG; }
  if (!aligned16(x)) { set_err("x must be 16-byte aligned"); return MOE_ERR_INVALID_ARG; }
  if ((reinterpret_cast<uintptr_t>(out) & ((flags & MOE_FWD_OUT_F32) ? 3u : 1u)) ||
      (reinterpret_cast<uintptr_t>(idx) & 3u)) {
    set_err("out must be 2-byte (fp32 out: 4-byte) and topk_idx 4-byte aligned");
    return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

}  // namespace

void wse::set_last_error_text(const char* text) { g_last_error = text ? text : ""; }

extern "C" {

const char* moe_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"

namespace {

// The create path of moe_create, moe_create_ex and moe_create_fp8: fp8 ->
// w_gate_up / w_down are E4M3 codes with row scales s_gu / s_d (no variants).
moe_layer* create_layer(int hidden, int n_experts, int topk, int inter, const void* w_router,
                        const void* w_gate_up, const void* w_down, const moe_layer_opts_t* opts, const float* s_gu,
                        const float* s_d, bool fp8) {
  g_last_error.clear();
  // ---- argument checks (no CUDA call before these pass) ----
  if (hidden <= 0 || hidden % 256 != 0 || !layer_kernel_for(hidden / 256, false)) {
    set_err("hidden = %d unsupported: need a multiple of 256 with hidden/256 in {1,2,4,5,8,10,12,16}",
            hidden);
    return nullptr;
  }
  if (inter != 128 && inter != 256 && inter != 512) {
    set_err("inter = %d unsupported: need one of {128, 256, 512}", inter);
    return nullptr;
  }
  if (hidden % inter != 0) {
    set_err("hidden = %d is not a multiple of inter = %d (a gate/up tile must be whole down slabs)",
            hidden, inter);
    return nullptr;
  }
  if (topk < 1 || topk > kMaxTopk) { set_err("topk = %d outside [1, %d]", topk, kMaxTopk); return nullptr; }
  if (n_experts < topk || n_experts > kMaxExperts) {
    set_err("n_experts = %d outside [topk, %d]", n_experts, kMaxExperts);
    return nullptr;
  }
  if (!w_router || !w_gate_up || !w_down) { set_err("null weight pointer"); return nullptr; }
  if (!aligned16(w_router) || !aligned16(w_gate_up) || !aligned16(w_down)) {
    set_err("weight pointers must be 16-byte aligned");
    return nullptr;
  }
  const moe_layer_opts_t o = opts ? *opts : moe_layer_opts_t{};
  if ((o.w_shared_gate_up == nullptr) != (o.w_shared_down == nullptr)) {
    set_err("shared expert: give both w_shared_gate_up and w_shared_down, or neither");
    return nullptr;
  }
  if (o.w_shared_gate_up && (!aligned16(o.w_shared_gate_up) || !aligned16(o.w_shared_down))) {
    set_err("shared expert weight pointers must be 16-byte aligned");
    return nullptr;
  }
  const int shared = o.w_shared_gate_up ? 1 : 0;
  if (fp8 && (!s_gu || !s_d || (reinterpret_cast<uintptr_t>(s_gu) & 3u) || (reinterpret_cast<uintptr_t>(s_d) & 3u))) {
    set_err("fp8 experts: the row scales must be non-null, 4-byte aligned device pointers");
    return nullptr;
  }

  // ---- device ----
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { cuda_fail(e, "cudaGetDevice"); return nullptr; }
  cudaDeviceProp prop;
  if ((e = cudaGetDeviceProperties(&prop, dev)) != cudaSuccess) { cuda_fail(e, "device properties"); return nullptr; }
  if (prop.major != 10 || prop.minor != 3) {
    set_err("device %d is sm_%d%d; this library is built for sm_103a (GB300)", dev, prop.major, prop.minor);
    return nullptr;
  }
  cudaFuncAttributes fa;
  const bool variant = o.w_shared_gate_up || o.bias_selection_only || (o.routed_scale > 0.f && o.routed_scale != 1.0f);
  if ((e = cudaFuncGetAttributes(&fa, layer_kernel_for(hidden / 256, variant, fp8))) != cudaSuccess) {
    cuda_fail(e, "kernel image");
    return nullptr;
  }

  moe_layer* h = new moe_layer;
  h->H = hidden; h->E = n_experts; h->K = topk; h->I = inter;
  h->shared = shared;
  h->routed_scale = o.routed_scale > 0.f ? o.routed_scale : 1.0f;
  h->sel_only = o.bias_selection_only ? 1 : 0;
  h->fp8 = fp8 ? 1 : 0;
  h->dev = dev;
  h->n_sms = prop.multiProcessorCount;
  h->grid = h->n_sms;
  h->tile_gu = (uint32_t)(kGateUpTileRows * hidden * 2);
  h->ks = gemv_split(hidden, n_experts, h->n_sms);

  // Rings sized for the largest call of each plan: the gate/up stages plus
  // the reduction area behind them, and the down stages over the same bytes,
  // take what the opt-in shared memory leaves after the routing area (one
  // CTA per SM; deep rings keep enough bytes in flight to cover the loaded
  // HBM latency).  The down phase reuses the ring as slab-sized cells (a
  // gate/up tile is hidden/inter whole slabs of 8 rows x I); a down slot is 8
  // cells, one slab per consumer warp.
  const size_t optin = prop.sharedMemPerBlockOptin;
  for (int i = 0; i < 2; ++i) {
    LayerPlan& pl = h->plan[i];
    const int tb = i == 0 ? 2 : 1;  // token blocks of 8 per group
    pl.kernel = layer_kernel_for(hidden / 256, variant, fp8, tb);
    pl.max_tokens = i == 0 ? kMaxTokens : 8;
    // A down cell (one consumer warp's unit of a super tile) is d_spw
    // consecutive output slabs.  The bf16 instances for M <= 8 take as many
    // as keep it within 8 rows x 512 bf16 (8 KB, whatever inter is: small
    // cells make every copy's fixed cost dominate) while super tiles (8
    // cells) and gate/up stages stay whole; the others take one.
    if (!fp8 && tb == 1)
      while (2 * pl.d_spw * inter <= 512 && hidden % (kDownTileRows * kConsumerWarps * 2 * pl.d_spw) == 0 &&
             hidden % (inter * 2 * pl.d_spw) == 0)
        pl.d_spw *= 2;
    pl.tile_d = (uint32_t)(kDownTileRows * inter * 2 * pl.d_spw);
    const int np_max = pl.max_tokens * h->kp();
    const size_t fixed = layer_smem_bytes(0, np_max, h->ea());
    const size_t avail = optin > fixed ? optin - fixed : 0;
    const size_t red = layer_reduction_bytes(fp8, tb);
    pl.s_gu = avail > red ? (int)std::min<size_t>(kMaxGateUpStages, (avail - red) / h->tile_gu) : 0;
    // Small gate/up tiles (small hidden) can leave the ring short of two
    // down super tiles: it then grows to two where the shared memory allows
    // (cells past the reduction area are down-only, free once the gate/up
    // loop is done, like the reduction area's).
    const size_t dsuper = (size_t)kConsumerWarps * pl.tile_d;
    const size_t ring_gu = (size_t)pl.s_gu * h->tile_gu + red;
    pl.ring_bytes = (uint32_t)(ring_gu < 2 * dsuper && 2 * dsuper <= avail ? 2 * dsuper : ring_gu);
    pl.s_d = (int)std::min<size_t>(kMaxDownStages, pl.ring_bytes / dsuper);
    if (!pl.kernel || pl.s_gu < 2 || pl.s_d < 2) {
      set_err("not enough shared memory for the staging rings");
      free_layer(h);
      return nullptr;
    }
    pl.smem_max = layer_smem_bytes(pl.ring_bytes, np_max, h->ea());
  }

  AllocCounter ac;
  const size_t E = n_experts, H = hidden, I = inter;
  const size_t EA = (size_t)h->ea();  // routed experts, then the shared one
  const size_t wb = fp8 ? 1 : 2;  // bytes per expert weight element
  const size_t b_router = E * H * 2, b_gu = EA * 2 * I * H * wb, b_d = EA * H * I * wb;
  const size_t b_sgu = fp8 ? E * 2 * I * 4 : 0, b_sd = fp8 ? E * H * 4 : 0;
  h->weight_bytes = b_router + b_gu + b_d + b_sgu + b_sd;
  if (ac.alloc((void**)&h->w_router, b_router) != cudaSuccess ||
      ac.alloc((void**)&h->w_gu, b_gu) != cudaSuccess ||
      ac.alloc((void**)&h->w_d, b_d) != cudaSuccess ||
      (fp8 && (ac.alloc((void**)&h->sc_gu, b_sgu) != cudaSuccess ||
               ac.alloc((void**)&h->sc_d, b_sd) != cudaSuccess))) {
    cudaGetLastError();
    set_err("device allocation of %zu weight bytes failed", h->weight_bytes);
    free_layer(h);
    return nullptr;
  }

  // workspace carve-up
  const size_t np = (size_t)kMaxTokens * h->kp();
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
  const size_t o_status = take(4), o_diag = take(32), o_sync = take(kSyncWords * 4);
  const size_t part_bytes = 2 * (size_t)h->ks * kMaxTokens * E * 4;  // odd and even calls
  const size_t o_part = take(part_bytes);
  const size_t o_ng = take(4), o_na = take(4);
  const size_t o_ge = take(np * 4), o_gs = take(np * 4), o_gc = take(np * 4);
  const size_t o_pl = take(np * 4), o_pw = take(np * 4);
  const size_t o_h = take(np * I * 2);
  const size_t o_y = take(np * H * 4);
  const size_t npt = (size_t)kGroupTokens * h->kp();  // tagged rows: calls of at most kGroupTokens tokens
  const size_t o_yt = take(npt * H * 8);
  const size_t o_xt = take(kXtopkBytes);
  const size_t o_tr = take((size_t)h->n_sms * kTraceSlots * 8);
  h->ws_bytes = off;
  if (ac.alloc(&h->ws_mem, h->ws_bytes) != cudaSuccess) {
    cudaGetLastError();
    set_err("device allocation of %zu workspace bytes failed", h->ws_bytes);
    free_layer(h);
    return nullptr;
  }
  uint8_t* base = static_cast<uint8_t*>(h->ws_mem);
  h->ws.status = reinterpret_cast<int*>(base + o_status);
  h->ws.diag = reinterpret_cast<unsigned long long*>(base + o_diag);
  h->ws.sync = reinterpret_cast<unsigned*>(base + o_sync);
  h->ws.part = reinterpret_cast<float*>(base + o_part);
  h->ws.n_groups = reinterpret_cast<int*>(base + o_ng);
  h->ws.n_active = reinterpret_cast<int*>(base + o_na);
  h->ws.grp_expert = reinterpret_cast<int*>(base + o_ge);
  h->ws.grp_start = reinterpret_cast<int*>(base + o_gs);
  h->ws.grp_cnt = reinterpret_cast<int*>(base + o_gc);
  h->ws.pair_list = reinterpret_cast<int*>(base + o_pl);
  h->ws.pair_w = reinterpret_cast<float*>(base + o_pw);
  h->ws.h = reinterpret_cast<__nv_bfloat16*>(base + o_h);
  h->ws.y = reinterpret_cast<float*>(base + o_y);
  h->ws.yt = reinterpret_cast<unsigned long long*>(base + o_yt);
  h->yt_bytes = npt * H * 8;
  h->ws.xtopk = reinterpret_cast<unsigned long long*>(base + o_xt);
  h->ws.trace = reinterpret_cast<unsigned long long*>(base + o_tr);

  // The caller's weights may still be being written by work it queued on
  // any stream (a slice, a cast, a copy): the copies below run on a stream
  // of our own, so wait for everything queued on the device first.
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) {
    cuda_fail(e, "synchronize before reading the weights");
    free_layer(h);
    return nullptr;
  }
  cudaStream_t s = nullptr;
  if ((e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking)) != cudaSuccess) {
    cuda_fail(e, "stream create");
    free_layer(h);
    return nullptr;
  }
  h->cap_stream = s;
  bool ok = cudaMemsetAsync(h->ws_mem, 0, h->ws_bytes, s) == cudaSuccess &&
            cudaMemsetAsync(h->ws.part, 0xff, part_bytes, s) == cudaSuccess &&  // every logit unwritten
            cudaMemsetAsync(h->ws.xtopk, 0xff, kXtopkBytes, s) == cudaSuccess &&  // every slot unwritten
            cudaMemcpyAsync(h->w_router, w_router, b_router, cudaMemcpyDeviceToDevice, s) == cudaSuccess;
  if (ok && fp8) {
    pack_gate_up_fp8(static_cast<const uint8_t*>(w_gate_up), h->w_gu, n_experts, inter, hidden, s);
    pack_down_fp8(static_cast<const uint8_t*>(w_down), h->w_d, n_experts, hidden, inter, s);
    ok = cudaMemcpyAsync(h->sc_gu, s_gu, b_sgu, cudaMemcpyDeviceToDevice, s) == cudaSuccess &&
         cudaMemcpyAsync(h->sc_d, s_d, b_sd, cudaMemcpyDeviceToDevice, s) == cudaSuccess &&
         cudaGetLastError() == cudaSuccess && cudaStreamSynchronize(s) == cudaSuccess;
  } else if (ok) {
    pack_gate_up(static_cast<const __nv_bfloat16*>(w_gate_up), reinterpret_cast<__nv_bfloat16*>(h->w_gu),
                 n_experts, inter, hidden, s);
    pack_down(static_cast<const __nv_bfloat16*>(w_down), reinterpret_cast<__nv_bfloat16*>(h->w_d),
              n_experts, hidden, inter, s);
    if (shared) {  // packed as expert index n_experts
      pack_gate_up(static_cast<const __nv_bfloat16*>(o.w_shared_gate_up),
                   reinterpret_cast<__nv_bfloat16*>(h->w_gu) + E * 2 * I * H, 1, inter, hidden, s);
      pack_down(static_cast<const __nv_bfloat16*>(o.w_shared_down),
                reinterpret_cast<__nv_bfloat16*>(h->w_d) + E * H * I, 1, hidden, inter, s);
    }
    ok = cudaGetLastError() == cudaSuccess && cudaStreamSynchronize(s) == cudaSuccess;
  }
  if (!ok) {
    set_err("weight re-layout failed: %s", cudaGetErrorString(cudaGetLastError()));
    free_layer(h);
    return nullptr;
  }
  // The expert kernels run one CTA per SM with most of its shared memory;
  // asking for the largest carveout up front avoids a reconfiguration of the
  // L1/shared split between launches.  The dynamic shared-memory limit is a
  // property of the kernel function, shared by every handle that launches
  // it: it is set to the device's opt-in maximum, so that a handle created
  // later with a smaller need never lowers it below an earlier handle's.
  e = cudaSuccess;
  for (int i = 0; i < 2 && e == cudaSuccess; ++i)
    if ((e = cudaFuncSetAttribute(h->plan[i].kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)prop.sharedMemPerBlockOptin)) == cudaSuccess)
      e = cudaFuncSetAttribute(h->plan[i].kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) {
    cuda_fail(e, "shared-memory attribute");
    free_layer(h);
    return nullptr;
  }
  return h;
}

}  // namespace

extern "C" {

moe_layer_t* moe_create(int hidden, int n_experts, int topk, int inter, const void* w_router,
                        const void* w_gate_up, const void* w_down) {
  return create_layer(hidden, n_experts, topk, inter, w_router, w_gate_up, w_down, nullptr, nullptr, nullptr, false);
}

moe_layer_t* moe_create_ex(int hidden, int n_experts, int topk, int inter, const void* w_router,
                           const void* w_gate_up, const void* w_down, const moe_layer_opts_t* opts) {
  return create_layer(hidden, n_experts, topk, inter, w_router, w_gate_up, w_down, opts, nullptr, nullptr, false);
}

moe_layer_t* moe_create_fp8(int hidden, int n_experts, int topk, int inter, const void* w_router,
                            const void* q_gate_up, const float* s_gate_up, const void* q_down,
                            const float* s_down) {
  return create_layer(hidden, n_experts, topk, inter, w_router, q_gate_up, q_down, nullptr, s_gate_up, s_down, true);
}


int moe_forward_ex(moe_layer_t* h, const void* x, void* out, int32_t* topk_idx, float* topk_w, int M,
                   moe_stream_t stream, unsigned flags) {
  int rc = check_forward_args(h, x, out, topk_idx, M, flags);
  if (rc != MOE_OK || M == 0) return rc;
  if (topk_w && (reinterpret_cast<uintptr_t>(topk_w) & 3u)) {
    set_err("topk_w must be 4-byte aligned");
    return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool pdl = !(flags & MOE_FWD_NO_PDL);
  const bool trace = (flags & MOE_FWD_TRACE) != 0;
  if (flags & MOE_FWD_GRAPH) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "capture status");
    if (cs == cudaStreamCaptureStatusNone) {
      GraphEntry& ge = h->graphs[M];
      if (!ge.exec || ge.x != x || ge.out != out || ge.idx != topk_idx || ge.tw != topk_w ||
          ge.flags != flags) {
        cudaGraph_t g = nullptr;
        if ((e = cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal)) != cudaSuccess)
          return cuda_fail(e, "begin capture");
        rc = launch_layer(h, x, out, topk_idx, topk_w, M, h->cap_stream, pdl, trace, nullptr, flags);
        e = cudaStreamEndCapture(h->cap_stream, &g);
        if (rc != MOE_OK) { if (g) cudaGraphDestroy(g); return rc; }
        if (e != cudaSuccess) return cuda_fail(e, "end capture");
        if (ge.exec) {
          cudaGraphExecUpdateResultInfo info;
          if (cudaGraphExecUpdate(ge.exec, g, &info) != cudaSuccess) {
            cudaGetLastError();
            cudaGraphExecDestroy(ge.exec);
            ge.exec = nullptr;
          }
        }
        if (!ge.exec && (e = cudaGraphInstantiate(&ge.exec, g, 0)) != cudaSuccess) {
          cudaGraphDestroy(g);
          return cuda_fail(e, "graph instantiate");
        }
        cudaGraphDestroy(g);
        ge.x = x; ge.out = out; ge.idx = topk_idx; ge.tw = topk_w; ge.flags = flags;
      }
      if ((e = cudaGraphLaunch(ge.exec, st)) != cudaSuccess) return cuda_fail(e, "graph launch");
      return MOE_OK;
    }
  }
  return launch_layer(h, x, out, topk_idx, topk_w, M, st, pdl, trace, nullptr, flags);
}

int moe_forward(moe_layer_t* h, const void* x, void* out, int32_t* topk_idx, int M, moe_stream_t stream) {
  return moe_forward_ex(h, x, out, topk_idx, nullptr, M, stream, 0u);
}

int moe_forward_timed(moe_layer_t* h, const void* x, void* out, int32_t* topk_idx, int M,
                      moe_stream_t stream, moe_event_t* ev) {
  int rc = check_forward_args(h, x, out, topk_idx, M);
  if (rc != MOE_OK) return rc;
  if (!ev || !ev[0] || !ev[1]) { set_err("need 2 events"); return MOE_ERR_INVALID_ARG; }
  if (M == 0) return MOE_OK;
  return launch_layer(h, x, out, topk_idx, nullptr, M, reinterpret_cast<cudaStream_t>(stream), false, false,
                      reinterpret_cast<cudaEvent_t*>(ev));
}

int moe_set_router_bias(moe_layer_t* h, const float* bias) {
  if (!h) { set_err("null handle"); return MOE_ERR_INVALID_ARG; }
  cudaError_t e;
  if (!bias) {
    if (h->bias) {
      if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "synchronize");
      cudaFree(h->bias);
      h->bias = nullptr;
    }
    drop_graphs(h);  // captured graphs hold the old pointer
    return MOE_OK;
  }
  if (!h->bias && (e = cudaMalloc((void**)&h->bias, (size_t)h->E * 4)) != cudaSuccess) {
    h->bias = nullptr;
    set_err("bias allocation failed");
    return MOE_ERR_OOM;
  }
  if ((e = cudaMemcpy(h->bias, bias, (size_t)h->E * 4, cudaMemcpyDefault)) != cudaSuccess)
    return cuda_fail(e, "bias copy");
  drop_graphs(h);
  return MOE_OK;
}

int moe_set_wait_limit(moe_layer_t* h, unsigned long long ns) {
  if (!h) { set_err("null handle"); return MOE_ERR_INVALID_ARG; }
  h->wait_ns = ns ? ns : kWaitTimeoutNs;
  drop_graphs(h);  // captured launches hold the old limit
  return MOE_OK;
}

int moe_set_grid(moe_layer_t* h, int ctas) {
  if (!h) { set_err("null handle"); return MOE_ERR_INVALID_ARG; }
  if (ctas < 0 || ctas > h->n_sms) {
    set_err("ctas = %d outside [0, %d] (0: one CTA per SM)", ctas, h->n_sms);
    return MOE_ERR_INVALID_ARG;
  }
  const int g = ctas ? ctas : h->n_sms;
  cudaError_t e;
  int cur = 0;
  if ((e = cudaGetDevice(&cur)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if ((e = cudaSetDevice(h->dev)) != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  // every CTA of the grid must be resident at once: one per SM on an idle
  // device (the instances' occupancy at their largest shared-memory size)
  for (int i = 0; i < 2; ++i) {
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, h->plan[i].kernel, kExpertThreads,
                                                      h->plan[i].smem_max);
    if (e != cudaSuccess || per_sm < 1 || (long long)per_sm * h->n_sms < g) {
      cudaSetDevice(cur);
      if (e != cudaSuccess) return cuda_fail(e, "occupancy");
      set_err("a grid of %d CTAs cannot be resident at once (%d per SM x %d SMs)", g, per_sm, h->n_sms);
      return MOE_ERR_UNSUPPORTED;
    }
  }
  // the call index comes from the arrival count divided by the grid: start
  // the counts again for the new grid (no kernel of this handle runs now)
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) { cudaSetDevice(cur); return cuda_fail(e, "synchronize"); }
  h->grid = g;
  restart_counts(h);
  drop_graphs(h);
  e = cudaDeviceSynchronize();
  cudaSetDevice(cur);
  if (e != cudaSuccess) return cuda_fail(e, "counter reset");
  return MOE_OK;
}

int moe_get_status(moe_layer_t* h) {
  if (!h) { set_err("null handle"); return MOE_ERR_INVALID_ARG; }
  cudaError_t e;
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "synchronize");
  int st = 0;
  unsigned long long dg[4] = {0, 0, 0, 0};
  if ((e = cudaMemcpy(&st, h->ws.status, 4, cudaMemcpyDeviceToHost)) != cudaSuccess ||
      (e = cudaMemcpy(dg, h->ws.diag, sizeof dg, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "status read");
  if (st) {
    cudaMemset(h->ws.status, 0, 4);
    cudaMemset(h->ws.diag, 0, sizeof dg);
    // a wait that gave up may have left the arrival counts between two
    // multiples of the grid: start them again from zero (no kernel runs
    // now), with every partial logit of both buffers unwritten again
    restart_counts(h);
    set_err("device status bits 0x%x (1 stage wait, 2 free-stage wait, 4 reduction wait, 8 no top-k "
            "candidate, 16 grid-wide wait); first timeout: phase %llu kind %llu cta %llu stages %llu "
            "index %llu waited %llu ns barrier 0x%016llx thread %llu grid %llu",
            st, dg[0] >> 56, (dg[0] >> 48) & 0xff, (dg[0] >> 32) & 0xffff, (dg[0] >> 16) & 0xffff,
            dg[0] & 0xffff, dg[1], dg[2], dg[3] >> 32, dg[3] & 0xffffffffull);
    return (st & (kErrTimeoutFull | kErrTimeoutEmpty | kErrTimeoutReduce | kErrTimeoutGrid))
               ? MOE_ERR_DEVICE_TIMEOUT
               : MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int moe_get_info(const moe_layer_t* h, moe_info_t* o) {
  if (!h || !o) { set_err("null argument"); return MOE_ERR_INVALID_ARG; }
  o->hidden = h->H; o->n_experts = h->E; o->topk = h->K; o->inter = h->I;
  o->max_tokens = MOE_MAX_TOKENS;
  o->n_sms = h->n_sms;
  o->grid_ctas = h->grid;
  o->wait_limit_ns = h->wait_ns;
  o->gateup_stages = h->plan[0].s_gu;
  o->down_stages = h->plan[0].s_d;
  o->gateup_tile_bytes = (int)h->tile_gu;
  o->down_tile_bytes = (int)(h->plan[0].tile_d * kConsumerWarps);
  o->weight_bytes = h->weight_bytes;
  o->workspace_bytes = h->ws_bytes;
  o->kernels_per_forward = 1;
  o->router_split = h->ks;
  o->smem_bytes = h->plan[0].smem_max;
  o->shared_expert = h->shared;
  o->routed_scale = h->routed_scale;
  o->bias_selection_only = h->sel_only;
  o->fp8_experts = h->fp8;
  return MOE_OK;
}

int moe_read_routing(moe_layer_t* h, int M, int* n_groups, int* n_active, int32_t* grp_expert,
                     int32_t* grp_start, int32_t* grp_cnt, int32_t* pair_list, float* pair_w, int cap) {
  if (!h || !n_groups || !n_active || M < 0 || M > MOE_MAX_TOKENS) {
    set_err("bad argument");
    return MOE_ERR_INVALID_ARG;
  }
  cudaError_t e;
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "synchronize");
  if ((e = cudaMemcpy(n_groups, h->ws.n_groups, 4, cudaMemcpyDeviceToHost)) != cudaSuccess ||
      (e = cudaMemcpy(n_active, h->ws.n_active, 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "routing read");
  const int ng = *n_groups < cap ? *n_groups : cap;
  const size_t np = (size_t)M * h->kp();
  if (ng > 0 && grp_expert && (e = cudaMemcpy(grp_expert, h->ws.grp_expert, ng * 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "routing read");
  if (ng > 0 && grp_start && (e = cudaMemcpy(grp_start, h->ws.grp_start, ng * 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "routing read");
  if (ng > 0 && grp_cnt && (e = cudaMemcpy(grp_cnt, h->ws.grp_cnt, ng * 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "routing read");
  if (np > 0 && pair_list && (e = cudaMemcpy(pair_list, h->ws.pair_list, np * 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "routing read");
  if (np > 0 && pair_w && (e = cudaMemcpy(pair_w, h->ws.pair_w, np * 4, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "routing read");
  return MOE_OK;
}

int moe_read_trace(moe_layer_t* h, uint64_t* out, int cap) {
  if (!h || !out || cap < 0) { set_err("bad argument"); return -MOE_ERR_INVALID_ARG; }
  const int n = std::min(cap, h->n_sms * kTraceSlots);
  cudaError_t e;
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return -cuda_fail(e, "synchronize");
  if (n > 0 && (e = cudaMemcpy(out, h->ws.trace, (size_t)n * 8, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return -cuda_fail(e, "trace read");
  return n;
}

void moe_destroy(moe_layer_t* h) {
  if (!h) return;
  int cur = 0;
  cudaGetDevice(&cur);
  cudaSetDevice(h->dev);
  cudaDeviceSynchronize();
  free_layer(h);
  cudaSetDevice(cur);
}

}  // extern "C"
