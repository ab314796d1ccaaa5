// moe_oracle.cpp -- CPU oracle for the small-M routed-MoE decode/verify layer.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, single-threaded
// definition of what the layer computes.  Only the test suite, the smoke check
// and the benchmark's CPU-baseline leg may load it.  The GPU library shares
// no code, header, table or helper with it, and never calls it.
//
// Source of the method (cited by page title and section):
//   [LB]  "How Ling-3.0-flash reduces batch 1 decoding latency by 54% on
//          4 Blackwell GPUs" (mirror of the LMSYS post "Chasing the batch-1
//          floor: Ling-3.0-flash speculative decode on Blackwell").
//   Sections used:  "PDL: the latency floor of stacked small kernels"
//   (router chain gate matvec -> top-k; MoE chain up-GEMM -> activation ->
//   down-GEMM -> combine; the combine as an fp32 sum times a scale with a
//   single final cast), "Two fusions and a retune" (SwiGLU = silu(gate)*up
//   evaluated in float with one final rounding; pair-axis bucketing),
//   "bf16 router gate and lm_head" (router weights in bf16; the vocabulary
//   projection as a bf16 matrix-vector product, oracle_lm_head).
//   Layer shape and routing rule (softmax top-k with renormalisation, SwiGLU
//   experts, bf16 inputs, fp32 accumulation) follow the layer definition the
//   post's model uses: a 512-expert routed MoE per layer, hidden 2560.
//
// Readings taken where the pages are silent (each is listed in the design
// notes as well):
//   * accumulation is fp32, in ascending index order, over bf16 inputs
//     converted exactly to fp32;
//   * routing: logits l = x . W_r[e] (+ optional per-expert bias b[e], used
//     only to realise skewed routing), top-k by logit with ties broken toward
//     the lower expert id, weights = full softmax over all experts then
//     renormalised over the chosen k;
//   * the gate/up projections g, u stay fp32; h = bf16(silu(g) * u) with
//     silu(g) = g / (1 + exp(-g)) in fp32, one rounding on the product;
//   * y = W_d h stays fp32; out = bf16(scale * sum_slots w * y), scale = 1,
//     slot order = descending logit;
//   * gate rows are W_gu[e][0:I), up rows are W_gu[e][I:2I);
//   * fp32 -> bf16 is round-to-nearest-even; inputs are finite.
//
// Build: g++ -O2 -ffp-contract=off -fPIC -shared (no FMA contraction, so the
// rounding sequence is the one written here on every host).

#include <cmath>
#include <limits>
#include <cstdint>
#include <cstring>
#include <vector>

extern "C" {

// ---------------------------------------------------------------- bf16 ----

// bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits.
float oracle_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// fp32 -> bf16, round to nearest, ties to even (finite inputs).
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

// ------------------------------------------------------------- router ----

// Router gate matvec ([LB] "bf16 router gate and lm_head"; router chain in
// "PDL: ..."): logits[m][e] = sum_h x[m][h] * W_r[e][h]  (+ bias[e]).
// W_r is stored [n_experts][hidden] (one row per expert).
int oracle_router_logits(int M, int H, int E, const uint16_t* x,
                         const uint16_t* w_router, const float* bias,
                         float* logits) {
  if (M < 0 || H <= 0 || E <= 0 || !x || !w_router || !logits) return 1;
  for (int m = 0; m < M; ++m) {
    for (int e = 0; e < E; ++e) {
      float acc = 0.0f;
      for (int h = 0; h < H; ++h) {
        float xv = oracle_bf16_to_f32(x[(size_t)m * H + h]);
        float wv = oracle_bf16_to_f32(w_router[(size_t)e * H + h]);
        acc = acc + xv * wv;
      }
      if (bias) acc = acc + bias[e];
      logits[(size_t)m * E + e] = acc;
    }
  }
  return 0;
}

// The vocabulary projection of the decode step ("bf16 router gate and
// lm_head": at batch 1 the lm_head is a bf16 matrix-vector product read once
// per step): logits[m][v] = sum_k x[m][k] * W[v][k], fp32, ascending k.
int oracle_lm_head(int M, int H, int V, const uint16_t* x, const uint16_t* w, float* logits) {
  if (M < 0 || H <= 0 || V <= 0 || !x || !w || !logits) return 1;
  for (int m = 0; m < M; ++m) {
    const uint16_t* xr = x + (size_t)m * H;
    for (int v = 0; v < V; ++v) {
      const uint16_t* wr = w + (size_t)v * H;
      float acc = 0.0f;
      for (int k = 0; k < H; ++k) acc = acc + oracle_bf16_to_f32(xr[k]) * oracle_bf16_to_f32(wr[k]);
      logits[(size_t)m * V + v] = acc;
    }
  }
  return 0;
}

// Softmax top-k with renormalisation, one token.
// Selection: the K largest logits, larger first, equal logits -> lower id.
// Weights: p_e = exp(l_e - l_max) / sum_all exp(l_e' - l_max), then
// w_j = p_{idx_j} / sum_{j' < K} p_{idx_j'}.
static void topk_one(int E, int K, const float* l, int32_t* idx, float* w) {
  std::vector<char> taken(E, 0);
  for (int j = 0; j < K; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (best < 0 || l[e] > l[best]) best = e;  // strict '>' keeps lower id on ties
    }
    taken[best] = 1;
    idx[j] = best;
  }
  float lmax = l[idx[0]];
  float z = 0.0f;
  for (int e = 0; e < E; ++e) z = z + std::exp(l[e] - lmax);
  std::vector<float> p(K);
  float s = 0.0f;
  for (int j = 0; j < K; ++j) {
    p[j] = std::exp(l[idx[j]] - lmax) / z;
    s = s + p[j];
  }
  for (int j = 0; j < K; ++j) w[j] = p[j] / s;
}

int oracle_topk_softmax(int M, int E, int K, const float* logits, int32_t* idx,
                        float* w) {
  if (M < 0 || E <= 0 || K <= 0 || K > E || !logits || !idx || !w) return 1;
  for (int m = 0; m < M; ++m)
    topk_one(E, K, logits + (size_t)m * E, idx + (size_t)m * K, w + (size_t)m * K);
  return 0;
}

// Weights for a GIVEN set of K experts (used to score a routing choice made
// elsewhere at a near-tie): same renormalised softmax as above over the set.
int oracle_weights_for_set(int E, int K, const float* logits_row,
                           const int32_t* idx, float* w) {
  if (E <= 0 || K <= 0 || !logits_row || !idx || !w) return 1;
  for (int j = 0; j < K; ++j)
    if (idx[j] < 0 || idx[j] >= E) return 1;
  float lmax = logits_row[idx[0]];
  for (int j = 1; j < K; ++j)
    if (logits_row[idx[j]] > lmax) lmax = logits_row[idx[j]];
  float z = 0.0f;
  for (int e = 0; e < E; ++e) z = z + std::exp(logits_row[e] - lmax);
  std::vector<float> p(K);
  float s = 0.0f;
  for (int j = 0; j < K; ++j) {
    p[j] = std::exp(logits_row[idx[j]] - lmax) / z;
    s = s + p[j];
  }
  for (int j = 0; j < K; ++j) w[j] = p[j] / s;
  return 0;
}

// ------------------------------------------------------------- expert ----

// SwiGLU activation on one (gate, up) pair, as the fused epilogue of
// [LB] "Two fusions and a retune" computes it: silu in float, multiply in
// float, a single rounding of the product to bf16.
uint16_t oracle_swiglu_bf16(float g, float u) {
  float s = g / (1.0f + std::exp(-g));
  return oracle_f32_to_bf16(s * u);
}

// Gate/up projection of one token through one expert, then SwiGLU.
// w_gate_up_e is that expert's [2I][H] block: rows [0,I) gate, [I,2I) up.
// h_out[r] (bf16 bits) for r < I.
int oracle_expert_swiglu(int H, int I, const uint16_t* x_row,
                         const uint16_t* w_gate_up_e, uint16_t* h_out) {
  if (H <= 0 || I <= 0 || !x_row || !w_gate_up_e || !h_out) return 1;
  for (int r = 0; r < I; ++r) {
    float g = 0.0f, u = 0.0f;
    const uint16_t* wg = w_gate_up_e + (size_t)r * H;
    const uint16_t* wu = w_gate_up_e + (size_t)(I + r) * H;
    for (int h = 0; h < H; ++h) {
      float xv = oracle_bf16_to_f32(x_row[h]);
      g = g + xv * oracle_bf16_to_f32(wg[h]);
      u = u + xv * oracle_bf16_to_f32(wu[h]);
    }
    h_out[r] = oracle_swiglu_bf16(g, u);
  }
  return 0;
}

// Down projection of one activated row: y[j] = sum_r h[r] * W_d[j][r].
// w_down_e is that expert's [H][I] block.
int oracle_expert_down(int H, int I, const uint16_t* h_row,
                       const uint16_t* w_down_e, float* y) {
  if (H <= 0 || I <= 0 || !h_row || !w_down_e || !y) return 1;
  for (int j = 0; j < H; ++j) {
    float acc = 0.0f;
    const uint16_t* wd = w_down_e + (size_t)j * I;
    for (int r = 0; r < I; ++r)
      acc = acc + oracle_bf16_to_f32(h_row[r]) * oracle_bf16_to_f32(wd[r]);
    y[j] = acc;
  }
  return 0;
}

// --------------------------------------------------------------- fp8 ----
// Expert weights in fp8 (the post: "once fp8 weights shrink the fixed
// base"): OCP FP8 E4M3 codes with one fp32 scale per output row; the
// dequantized matrix is diag(scale) * decode(codes).

// E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no
// infinities, S.1111.111 is NaN.  Exact value as fp32.
float oracle_e4m3_to_f32(uint8_t v) {
  const int s = v >> 7, e = (v >> 3) & 15, m = v & 7;
  float mag;
  if (e == 15 && m == 7)
    mag = std::numeric_limits<float>::quiet_NaN();
  else if (e == 0)
    mag = std::ldexp((float)m, -9);  // subnormal: (m / 8) * 2^-6
  else
    mag = std::ldexp(1.0f + (float)m / 8.0f, e - 7);
  return s ? -mag : mag;
}

// Gate/up of one token through one fp8 expert (codes [2I][H], scales [2I]):
// g = s[r] * sum_h x[h] * q[r][h], u likewise with row I + r (the row scale
// factored out of the fp32 sum); h = bf16(silu(g) * u).
int oracle_expert_swiglu_fp8(int H, int I, const uint16_t* x_row, const uint8_t* q_gu_e,
                             const float* s_gu_e, uint16_t* h_out) {
  if (H <= 0 || I <= 0 || !x_row || !q_gu_e || !s_gu_e || !h_out) return 1;
  for (int r = 0; r < I; ++r) {
    float g = 0.0f, u = 0.0f;
    const uint8_t* qg = q_gu_e + (size_t)r * H;
    const uint8_t* qu = q_gu_e + (size_t)(I + r) * H;
    for (int h = 0; h < H; ++h) {
      float xv = oracle_bf16_to_f32(x_row[h]);
      g = g + xv * oracle_e4m3_to_f32(qg[h]);
      u = u + xv * oracle_e4m3_to_f32(qu[h]);
    }
    h_out[r] = oracle_swiglu_bf16(s_gu_e[r] * g, s_gu_e[I + r] * u);
  }
  return 0;
}

// Down projection of one activated row through one fp8 expert (codes
// [H][I], scales [H]): y[j] = s[j] * sum_r h[r] * q[j][r].
int oracle_expert_down_fp8(int H, int I, const uint16_t* h_row, const uint8_t* q_d_e, const float* s_d_e,
                           float* y) {
  if (H <= 0 || I <= 0 || !h_row || !q_d_e || !s_d_e || !y) return 1;
  for (int j = 0; j < H; ++j) {
    float acc = 0.0f;
    const uint8_t* qd = q_d_e + (size_t)j * I;
    for (int r = 0; r < I; ++r) acc = acc + oracle_bf16_to_f32(h_row[r]) * oracle_e4m3_to_f32(qd[r]);
    y[j] = s_d_e[j] * acc;
  }
  return 0;
}

// The layer with fp8 expert weights (router bf16, routing and combine as
// oracle_moe_forward): q_gate_up [E][2I][H] + s_gate_up [E][2I],
// q_down [E][H][I] + s_down [E][H].  Outputs as oracle_moe_forward.
int oracle_moe_forward_fp8(int M, int H, int E, int K, int I, const uint16_t* x, const uint16_t* w_router,
                           const float* bias, const uint8_t* q_gate_up, const float* s_gate_up,
                           const uint8_t* q_down, const float* s_down, const int32_t* idx_in,
                           float* logits_out, int32_t* idx_out, float* w_out, float* acc_out, uint16_t* out) {
  if (M < 0 || H <= 0 || E <= 0 || K <= 0 || K > E || I <= 0) return 1;
  if (!x || !w_router || !q_gate_up || !s_gate_up || !q_down || !s_down || !out) return 1;
  if (M == 0) return 0;
  std::vector<float> logits((size_t)M * E);
  std::vector<int32_t> idx((size_t)M * K);
  std::vector<float> w((size_t)M * K);
  if (oracle_router_logits(M, H, E, x, w_router, bias, logits.data())) return 1;
  if (idx_in) {
    for (int m = 0; m < M; ++m) {
      for (int j = 0; j < K; ++j) idx[(size_t)m * K + j] = idx_in[(size_t)m * K + j];
      if (oracle_weights_for_set(E, K, logits.data() + (size_t)m * E, idx.data() + (size_t)m * K,
                                 w.data() + (size_t)m * K))
        return 1;
    }
  } else {
    oracle_topk_softmax(M, E, K, logits.data(), idx.data(), w.data());
  }
  std::vector<uint16_t> hrow(I);
  std::vector<float> y(H), acc(H);
  for (int m = 0; m < M; ++m) {
    const uint16_t* xr = x + (size_t)m * H;
    for (int j = 0; j < H; ++j) acc[j] = 0.0f;
    for (int s = 0; s < K; ++s) {
      const int e = idx[(size_t)m * K + s];
      oracle_expert_swiglu_fp8(H, I, xr, q_gate_up + (size_t)e * 2 * I * H, s_gate_up + (size_t)e * 2 * I,
                               hrow.data());
      oracle_expert_down_fp8(H, I, hrow.data(), q_down + (size_t)e * H * I, s_down + (size_t)e * H, y.data());
      const float ws = w[(size_t)m * K + s];
      for (int j = 0; j < H; ++j) acc[j] = acc[j] + ws * y[j];
    }
    for (int j = 0; j < H; ++j) {
      if (acc_out) acc_out[(size_t)m * H + j] = acc[j];
      out[(size_t)m * H + j] = oracle_f32_to_bf16(acc[j]);
    }
  }
  if (logits_out) std::memcpy(logits_out, logits.data(), logits.size() * 4);
  if (idx_out) std::memcpy(idx_out, idx.data(), idx.size() * 4);
  if (w_out) std::memcpy(w_out, w.data(), w.size() * 4);
  return 0;
}

// -------------------------------------------------------------- layer ----

// The whole layer for M tokens, with the layer variants the post's model
// uses ("Two kinds of idle": a 513-expert decode, i.e. a shared expert fused
// next to the 512 routed ones; "PDL: ...": the combine is an fp32 sum times a
// scale; "the router top-k prefetches its bias").
//   x         [M][H] bf16           w_router  [E][H] bf16
//   bias      [E] fp32 or NULL      w_gate_up [E][2I][H] bf16
//   w_down    [E][H][I] bf16
//   bias_selection_only: 0 -> the bias shifts the logits used for both the
//             selection and the weights; 1 -> it shifts only the selection,
//             the weights are the softmax of the unbiased logits,
//             renormalised over the chosen k.
//   w_shared_gate_up [2I][H], w_shared_down [H][I] bf16, or both NULL: a
//             shared expert every token passes through with weight 1.
//   routed_scale  multiplies every routed weight (1 = none).
//   idx_in    [M][K] or NULL: when given, these experts are used instead of
//             the oracle's own selection and weighted with the oracle's
//             renormalised softmax over that set (near-tie scoring).
// The combine: acc = sum over slots s < K (in order) of (scale * w_s) * y_s,
// then + y_shared; out = bf16(acc), one rounding.
// Outputs (any may be NULL except out):
//   logits [M][E] fp32 (the selection logits), idx [M][K] int32,
//   w [M][K] fp32 (renormalised, unscaled), acc [M][H] fp32 (the combine
//   before the final cast), h [M][K][I] bf16 (routed intermediate rows),
//   out [M][H] bf16.
int oracle_moe_forward_ex(int M, int H, int E, int K, int I, const uint16_t* x,
                          const uint16_t* w_router, const float* bias, int bias_selection_only,
                          const uint16_t* w_gate_up, const uint16_t* w_down,
                          const uint16_t* w_shared_gate_up, const uint16_t* w_shared_down,
                          float routed_scale, const int32_t* idx_in, float* logits_out,
                          int32_t* idx_out, float* w_out, float* acc_out,
                          uint16_t* h_out, uint16_t* out) {
  if (M < 0 || H <= 0 || E <= 0 || K <= 0 || K > E || I <= 0) return 1;
  if (!x || !w_router || !w_gate_up || !w_down || !out) return 1;
  if ((w_shared_gate_up == nullptr) != (w_shared_down == nullptr)) return 1;
  if (M == 0) return 0;
  const bool sel_only = bias_selection_only && bias;
  std::vector<float> logits((size_t)M * E), unbiased;
  std::vector<int32_t> idx((size_t)M * K);
  std::vector<float> w((size_t)M * K);
  if (oracle_router_logits(M, H, E, x, w_router, bias, logits.data())) return 1;
  if (sel_only) {
    unbiased.resize((size_t)M * E);
    if (oracle_router_logits(M, H, E, x, w_router, nullptr, unbiased.data())) return 1;
  }
  const float* wlog = sel_only ? unbiased.data() : logits.data();  // logits the weights come from
  if (idx_in) {
    for (int m = 0; m < M; ++m)
      for (int j = 0; j < K; ++j) idx[(size_t)m * K + j] = idx_in[(size_t)m * K + j];
  } else {
    oracle_topk_softmax(M, E, K, logits.data(), idx.data(), w.data());
  }
  if (idx_in || sel_only) {
    for (int m = 0; m < M; ++m)
      if (oracle_weights_for_set(E, K, wlog + (size_t)m * E, idx.data() + (size_t)m * K,
                                 w.data() + (size_t)m * K))
        return 1;
  }
  std::vector<uint16_t> h(I);
  std::vector<float> y(H);
  std::vector<float> ys(H);
  std::vector<float> acc(H);
  for (int m = 0; m < M; ++m) {
    const uint16_t* xr = x + (size_t)m * H;
    for (int j = 0; j < H; ++j) acc[j] = 0.0f;
    for (int s = 0; s < K; ++s) {
      int e = idx[(size_t)m * K + s];
      oracle_expert_swiglu(H, I, xr, w_gate_up + (size_t)e * 2 * I * H, h.data());
      if (h_out)
        for (int r = 0; r < I; ++r) h_out[((size_t)m * K + s) * I + r] = h[r];
      oracle_expert_down(H, I, h.data(), w_down + (size_t)e * H * I, y.data());
      float ws = routed_scale * w[(size_t)m * K + s];
      for (int j = 0; j < H; ++j) acc[j] = acc[j] + ws * y[j];
    }
    if (w_shared_gate_up) {
      oracle_expert_swiglu(H, I, xr, w_shared_gate_up, h.data());
      oracle_expert_down(H, I, h.data(), w_shared_down, ys.data());
      for (int j = 0; j < H; ++j) acc[j] = acc[j] + ys[j];
    }
    for (int j = 0; j < H; ++j) {
      float v = acc[j];
      if (acc_out) acc_out[(size_t)m * H + j] = v;
      out[(size_t)m * H + j] = oracle_f32_to_bf16(v);
    }
  }
  if (logits_out) std::memcpy(logits_out, logits.data(), logits.size() * 4);
  if (idx_out) std::memcpy(idx_out, idx.data(), idx.size() * 4);
  if (w_out) std::memcpy(w_out, w.data(), w.size() * 4);
  return 0;
}

// The plain layer: no shared expert, scale 1, the bias (if any) on the
// logits for both selection and weights.
int oracle_moe_forward(int M, int H, int E, int K, int I, const uint16_t* x,
                       const uint16_t* w_router, const float* bias,
                       const uint16_t* w_gate_up, const uint16_t* w_down,
                       const int32_t* idx_in, float* logits_out,
                       int32_t* idx_out, float* w_out, float* acc_out,
                       uint16_t* h_out, uint16_t* out) {
  return oracle_moe_forward_ex(M, H, E, K, I, x, w_router, bias, 0, w_gate_up, w_down, nullptr, nullptr,
                               1.0f, idx_in, logits_out, idx_out, w_out, acc_out, h_out, out);
}

}  // extern "C"
