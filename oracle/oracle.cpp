// CPU oracle for the int4 routed-expert MoE layer.
//
// TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, single-threaded
// statement of what the layer computes.  Only the tests, the smoke check and
// the benchmark's CPU-baseline leg may load it.  It shares no code, header,
// table or constant generator with the CUDA library; the two agree because
// both follow the same written definitions below, not because one calls the
// other.
//
// Sources (page title, then section):
//   [P1] "GLM-5.2 on a 32 GB Mac — native MLX port of the Colibri hierarchy"
//        - N1 "GLM-5.2 graph", MoE bullet: sigmoid scores plus correction bias
//          select the experts, the un-biased sigmoid gives the gate weights,
//          true top-8, optional normalisation and routed scale, shared expert
//          in parallel.
//        - N2 "Colibri-compatible quant/container support": per-expert
//          gate/up/down tensors, packed symmetric int4, grouped scales.
//        - "G2 - native GLM-5.2 correctness spine": dequant -> f32
//          multiply-accumulate numerics.
//        - "G2 implementation status": offset-binary Q4 (bias = -8 * scale),
//          lower expert id wins an exact tie, un-biased sigmoid for
//          execution, routed scaling, unweighted shared expert.
//        - "G4 - serial native MTP": RMSNorm squared sums reduced in float64.
//        - N4 "Scheduling and prediction": route the whole batch first, form
//          the stable unique expert union, run each expert over its rows.
//   [P3] "colibri-strix/README.md", "What's implemented": DeepSeek-V3-style
//        sigmoid router (noaux_tc, routed_scaling_factor), shared expert,
//        batch-union MoE.
//   [P4] "Model support - run anything mlx-lm runs", 6.4 "GLM-5.2": RMSNorm
//        with multiplicative weight and double-accumulated reduction,
//        offset-binary int4.
//
// Readings where the pages are silent (each also listed in the design notes):
//   R1  router dot-product order: fixed order stated at router_logit().
//   R2  sigmoid: own exp (Cody-Waite reduction + degree-7 Taylor series),
//       stated at router_exp().
//   R3  group score = sum of the two largest biased scores of the group.
//   R4  experts of unselected groups are excluded (not zero-filled).
//   R5  top-k by biased score descending, exact ties -> lower expert id.
//   R6  w_j = (g_j / sum_j g_j) * routed_scaling_factor, sum in slot order.
//   R7  nibble q in [-8,7] stored as u = q + 8; low nibble = even k.
//   R8  group size 32 along K, fp16 scales.
//   R9  shared expert weight 1, added after the routed sum.
//   R12 plan order: experts ascending, entries (t, j) ascending.
//   R13 RMSNorm: fixed fp64 sum order stated at rmsnorm_row(); the
//       reciprocal root is rounded to fp32 and applied with fp32 products;
//       gamma is multiplicative; normalised activations stay fp32.
//   R22 the other expert formats ([P1] N2: symmetric int4/int8, per-row or
//       grouped scales; G2 status: Q8 applies its scale to the signed
//       two's-complement byte, and a whole-row scale repeated over 32-value
//       groups leaves every dequantised value unchanged): int8 weights one
//       signed byte per element, K bytes per row; per-row scales one fp16 per
//       row.  Stated at dequant_fmt().
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -fno-fast-math -shared -fPIC.
// Contraction must stay off: every fused multiply-add below is written as
// std::fma on purpose, every other product and sum is rounded on its own.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// ---------------------------------------------------------------- numbers --

float bits_to_float(uint32_t u) {
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

uint32_t float_to_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}

// IEEE-754 binary16 -> binary32, exact (every half is a float).
float half_to_float(uint16_t h) {
  const uint32_t sign = (uint32_t)(h >> 15) & 1u;
  const uint32_t expo = (uint32_t)(h >> 10) & 0x1Fu;
  const uint32_t mant = (uint32_t)h & 0x3FFu;
  float mag;
  if (expo == 0) {
    mag = std::ldexp((float)mant, -24);  // subnormal: mant * 2^-24
  } else if (expo == 31) {
    mag = mant ? NAN : INFINITY;
  } else {
    mag = std::ldexp((float)(mant | 0x400u), (int)expo - 25);
  }
  return sign ? -mag : mag;
}

// The stored code u of element k of a packed int4 row (R7 nibble order).
int int4_code(const uint8_t* row_q, int k) {
  const uint8_t byte = row_q[k >> 1];
  return (k & 1) ? (byte >> 4) : (byte & 0xF);
}

// Dequantised weight: (u - 8) * scale, exact in fp32 ([P1] G2 status:
// offset-binary, bias = -8 * scale).  Nibble order R7.
float dequant(const uint8_t* row_q, const uint16_t* row_s, int k) {
  const int u = int4_code(row_q, k);
  const float s = half_to_float(row_s[k / 32]);
  return (float)(u - 8) * s;
}

// Dequantised weight of the other formats (R22): element k of a K-long row
// with weight format fmt (0: packed offset-binary int4 as in dequant(), 1:
// signed int8, one byte per element) and scale group gsz (32: one fp16 scale
// per 32 elements; 0: one fp16 scale for the whole row).  Exact in fp32: q
// has at most 8 significant bits and the scale 11.
float dequant_fmt(const uint8_t* row_q, const uint16_t* row_s, int k, int fmt, int gsz) {
  if (fmt == 0 && gsz == 32) return dequant(row_q, row_s, k);
  int q;
  if (fmt == 1) {
    const uint8_t byte = row_q[k];
    q = byte < 128 ? (int)byte : (int)byte - 256;  // two's complement
  } else {
    q = int4_code(row_q, k) - 8;
  }
  const float s = half_to_float(row_s[gsz == 0 ? 0 : k / gsz]);
  return (float)q * s;
}

// ------------------------------------------------------------------ router --

// R2. Own exponential for the router's sigmoid, defined on t in [-32, 88].
// Method: Cody & Waite argument reduction, t = n*ln2 + r with
// n = rint(t * log2(e)) and r computed against a two-part ln2, then
// exp(r) by its Taylor series to degree 7 (Horner form, fused multiply-adds),
// and exp(t) = exp(r) * 2^n.  Constants are the fp32 roundings of:
//   log2(e); ln2 rounded to 16 significant bits (so n*ln2_hi is exact for
//   |n| < 256) and the fp32 rounding of the remainder ln2 - ln2_hi;
//   1/i! for i = 0..7.
const float kLog2e = 1.44269502162933349609375f;       // fp32(1/ln 2)
const float kLn2Hi = 0.693145751953125f;               // 16-bit ln 2
const float kLn2Lo = 1.428606765330187e-06f;           // fp32(ln2 - ln2_hi)
const float kInvFact[8] = {1.0f, 1.0f, 0.5f, 0.1666666716337204f,
                           0.0416666679084301f, 0.008333333767950535f,
                           0.0013888889225199819f, 0.00019841270113829523f};

float router_exp(float t) {
  const float n = std::nearbyint(t * kLog2e);  // ties to even
  float r = std::fma(-n, kLn2Hi, t);
  r = std::fma(-n, kLn2Lo, r);
  float p = kInvFact[7];
  for (int i = 6; i >= 0; --i) p = std::fma(p, r, kInvFact[i]);
  const int ni = (int)n;  // in [-47, 127] on the domain
  const float two_n = bits_to_float((uint32_t)(ni + 127) << 23);
  return p * two_n;
}

// sigma(z) = 1 / (1 + exp(-z)); saturates to exactly 1 for z > 32 (where
// 1 + exp(-z) rounds to 1 anyway) and to 0 for z < -88.
float router_sigmoid(float z) {
  const float t = -z;
  if (t > 88.0f) return 0.0f;
  if (t < -32.0f) return 1.0f;
  const float e = router_exp(t);
  const float d = 1.0f + e;
  return 1.0f / d;
}

// R1. Router logit = x . w over H (H a multiple of 32), in this fixed order:
// H is cut into 8 equal segments; a segment is read as chunks of 4
// consecutive elements; partial (s, j), j = 0..31, owns the chunks
// j, j+32, j+64, ... of segment s and accumulates their elements in
// ascending index with fused multiply-adds from 0.  The 32 partials of a
// segment are then summed pairwise by halving: for d = 16, 8, 4, 2, 1,
// p[j] = p[j] + p[j + d] for j < d.  The 8 segment sums are summed the same
// way with d = 4, 2, 1.
float router_logit(const float* x, const float* w, int H) {
  const int L = H / 8;
  const int chunks = L / 4;
  float seg[8];
  for (int s = 0; s < 8; ++s) {
    float p[32];
    for (int j = 0; j < 32; ++j) {
      float acc = 0.0f;
      for (int c = j; c < chunks; c += 32) {
        for (int q = 0; q < 4; ++q) {
          const int k = s * L + 4 * c + q;
          acc = std::fma(x[k], w[k], acc);
        }
      }
      p[j] = acc;
    }
    for (int d = 16; d >= 1; d /= 2)
      for (int j = 0; j < d; ++j) p[j] = p[j] + p[j + d];
    seg[s] = p[0];
  }
  for (int d = 4; d >= 1; d /= 2)
    for (int s = 0; s < d; ++s) seg[s] = seg[s] + seg[s + d];
  return seg[0];
}

// a > b in the selection order: larger value first, lower index on a tie.
bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

}  // namespace

extern "C" {

float oracle_router_exp(float t) { return router_exp(t); }
float oracle_router_sigmoid(float z) { return router_sigmoid(z); }
float oracle_half_to_float(uint16_t h) { return half_to_float(h); }
float oracle_dequant(const uint8_t* row_q, const uint16_t* row_s, int k) {
  return dequant(row_q, row_s, k);
}

// logits[t][e] = router_logit(x[t], Wr[e]).
int oracle_router_logits(const float* x, int T, int H, const float* Wr, int E,
                         float* logits) {
  if (H % 32 != 0 || T < 0 || E <= 0) return -1;
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e)
      logits[(size_t)t * E + e] = router_logit(x + (size_t)t * H, Wr + (size_t)e * H, H);
  return 0;
}

// noaux_tc selection for one batch of logits ([P1] N1 MoE bullet and G2
// status; [P3] "What's implemented"; group limits R3/R4; order R5; gates R6).
//   s_e   = sigma(logit_e)              (un-biased score, the gate value)
//   key_e = s_e + bias_e                (selection key)
//   group score = top-2 sum of keys in each of n_group equal groups
//   keep topk_group groups (score desc, lower group on a tie)
//   ids   = top_k experts of the kept groups by key (desc, lower id on tie)
//   w_j   = (s_{id_j} / sum_j s_{id_j}) * rsf
int oracle_select(const float* logits, const float* bias, int T, int E, int k,
                  int n_group, int topk_group, float rsf, int32_t* ids,
                  float* weights) {
  if (n_group <= 0 || E % n_group != 0 || topk_group < 1 || topk_group > n_group)
    return -1;
  const int G = E / n_group;
  if (k < 1 || k > topk_group * G) return -1;
  std::vector<float> s(E), key(E), gscore(n_group);
  std::vector<char> group_kept(n_group), taken(E);
  for (int t = 0; t < T; ++t) {
    const float* lg = logits + (size_t)t * E;
    for (int e = 0; e < E; ++e) {
      s[e] = router_sigmoid(lg[e]);
      key[e] = s[e] + bias[e];
    }
    for (int g = 0; g < n_group; ++g) {
      // two largest keys of the group (values only; ties are irrelevant)
      float a = -INFINITY, b = -INFINITY;
      for (int e = g * G; e < (g + 1) * G; ++e) {
        if (key[e] > a) {
          b = a;
          a = key[e];
        } else if (key[e] > b) {
          b = key[e];
        }
      }
      gscore[g] = (G >= 2) ? a + b : a;
    }
    for (int g = 0; g < n_group; ++g) group_kept[g] = 0;
    for (int r = 0; r < topk_group; ++r) {
      int best = -1;
      for (int g = 0; g < n_group; ++g) {
        if (group_kept[g]) continue;
        if (best < 0 || ranks_before(gscore[g], g, gscore[best], best)) best = g;
      }
      group_kept[best] = 1;
    }
    for (int e = 0; e < E; ++e) taken[e] = 0;
    float sum = 0.0f;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e] || !group_kept[e / G]) continue;
        if (best < 0 || ranks_before(key[e], e, key[best], best)) best = e;
      }
      taken[best] = 1;
      ids[(size_t)t * k + j] = best;
      sum = sum + s[best];
    }
    for (int j = 0; j < k; ++j) {
      const float g = s[ids[(size_t)t * k + j]];
      const float q = g / sum;
      weights[(size_t)t * k + j] = q * rsf;
    }
  }
  return 0;
}

// Routing plan ([P1] N4 first bullet and G3 status "stable row/rank batch
// union"; order R12).  counts[e] = #entries routed to e; offsets = exclusive
// prefix sum (offsets[E] = T*k); perm lists entry indices i = t*k + j grouped
// by expert ascending, and inside an expert by i ascending; active lists the
// experts with count > 0 ascending.
int oracle_plan(const int32_t* ids, int T, int k, int E, int32_t* counts,
                int32_t* offsets, int32_t* perm, int32_t* active,
                int32_t* n_active) {
  const int N = T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int i = 0; i < N; ++i) {
    if (ids[i] < 0 || ids[i] >= E) return -1;
    counts[ids[i]] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int pos = 0;
  for (int e = 0; e < E; ++e)
    for (int i = 0; i < N; ++i)
      if (ids[i] == e) perm[pos++] = i;
  int na = 0;
  for (int e = 0; e < E; ++e)
    if (counts[e] > 0) active[na++] = e;
  *n_active = na;
  return 0;
}

// RMSNorm of one row (R13; [P1] G4: float64 squared sums; [P4] 6.4:
// multiplicative weight, double-accumulated reduction).  The fp64 sum of
// squares uses the same fixed order as router_logit (8 segments x 32
// partials over chunks of 4, fused multiply-adds, pairwise halving); then
//   r  = 1 / sqrt(ss / H + eps)        (fp64, each step rounded)
//   rf = (float)r                      (the pages keep only the reduction in
//                                       double; the scaling is fp32)
//   out_k = (h_k * rf) * gamma_k       (two fp32 products, each rounded)
void rmsnorm_row(const float* h, int H, const float* gamma, double eps, float* out) {
  const int L = H / 8;
  const int chunks = L / 4;
  double seg[8];
  for (int s = 0; s < 8; ++s) {
    double p[32];
    for (int j = 0; j < 32; ++j) {
      double acc = 0.0;
      for (int c = j; c < chunks; c += 32)
        for (int q = 0; q < 4; ++q) {
          const double v = (double)h[s * L + 4 * c + q];
          acc = std::fma(v, v, acc);
        }
      p[j] = acc;
    }
    for (int d = 16; d >= 1; d /= 2)
      for (int j = 0; j < d; ++j) p[j] = p[j] + p[j + d];
    seg[s] = p[0];
  }
  for (int d = 4; d >= 1; d /= 2)
    for (int s = 0; s < d; ++s) seg[s] = seg[s] + seg[s + d];
  const double mean = seg[0] / (double)H;
  const double r = 1.0 / std::sqrt(mean + eps);
  const float rf = (float)r;
  for (int k = 0; k < H; ++k) {
    const float v = h[k] * rf;
    out[k] = gamma ? v * gamma[k] : v;
  }
}

int oracle_rmsnorm(const float* h, int T, int H, const float* gamma, double eps,
                   float* out) {
  if (H % 32 != 0) return -1;
  for (int t = 0; t < T; ++t)
    rmsnorm_row(h + (size_t)t * H, H, gamma, eps, out + (size_t)t * H);
  return 0;
}

}  // extern "C"

namespace {

// One expert's SwiGLU on one token ([P1] N2 and G2: dequant -> f32 MAC;
// [P3] Metal section "routed-expert SwiGLU").  Acc is float (the pages'
// numerics) or double (used only to bound the fp32 oracle's own error).
//   g_i = sum_k Wg[i,k] x_k,  u_i = sum_k Wu[i,k] x_k        (k ascending)
//   h_i = silu(g_i) * u_i,    silu(z) = z / (1 + exp(-z))
//   o_r = sum_i Wd[r,i] h_i                                   (i ascending)
// Weight format fmt and scale group gsz as in dequant_fmt() (R22): a row
// holds K / 2 (int4) or K (int8) bytes and K / 32 or 1 scales.
template <typename Acc>
void expert_swiglu(const float* x, int H, int I, int fmt, int gsz, const uint8_t* gq,
                   const uint16_t* gs, const uint8_t* uq, const uint16_t* us,
                   const uint8_t* dq, const uint16_t* ds, Acc* out) {
  const size_t qh = fmt == 1 ? (size_t)H : (size_t)H / 2;
  const size_t qi = fmt == 1 ? (size_t)I : (size_t)I / 2;
  const size_t sh = gsz == 0 ? 1 : (size_t)H / 32;
  const size_t si = gsz == 0 ? 1 : (size_t)I / 32;
  std::vector<Acc> h(I);
  for (int i = 0; i < I; ++i) {
    const uint8_t* gr = gq + (size_t)i * qh;
    const uint16_t* gsr = gs + (size_t)i * sh;
    const uint8_t* ur = uq + (size_t)i * qh;
    const uint16_t* usr = us + (size_t)i * sh;
    Acc g = 0, u = 0;
    for (int k = 0; k < H; ++k) {
      g = g + (Acc)dequant_fmt(gr, gsr, k, fmt, gsz) * (Acc)x[k];
      u = u + (Acc)dequant_fmt(ur, usr, k, fmt, gsz) * (Acc)x[k];
    }
    const Acc silu = g / ((Acc)1 + std::exp(-g));
    h[i] = silu * u;
  }
  for (int r = 0; r < H; ++r) {
    const uint8_t* dr = dq + (size_t)r * qi;
    const uint16_t* dsr = ds + (size_t)r * si;
    Acc o = 0;
    for (int i = 0; i < I; ++i) o = o + (Acc)dequant_fmt(dr, dsr, i, fmt, gsz) * h[i];
    out[r] = o;
  }
}

bool fmt_ok(int fmt, int gsz) { return (fmt == 0 || fmt == 1) && (gsz == 32 || gsz == 0); }

}  // namespace

extern "C" {

float oracle_dequant_fmt(const uint8_t* row_q, const uint16_t* row_s, int k, int fmt,
                         int gsz) {
  return dequant_fmt(row_q, row_s, k, fmt, gsz);
}

// One expert of any format (R22) on one token, fp32 (prec=0) or fp64 (prec=1).
int oracle_expert_fmt(const float* x, int H, int I, int fmt, int gsz, const uint8_t* gq,
                      const uint16_t* gs, const uint8_t* uq, const uint16_t* us,
                      const uint8_t* dq, const uint16_t* ds, int prec, double* out) {
  if (H % 32 != 0 || I % 32 != 0 || !fmt_ok(fmt, gsz)) return -1;
  if (prec == 0) {
    std::vector<float> o(H);
    expert_swiglu<float>(x, H, I, fmt, gsz, gq, gs, uq, us, dq, ds, o.data());
    for (int r = 0; r < H; ++r) out[r] = o[r];
  } else {
    expert_swiglu<double>(x, H, I, fmt, gsz, gq, gs, uq, us, dq, ds, out);
  }
  return 0;
}

// One grouped-int4 expert on one token, fp32 (prec=0) or fp64 (prec=1)
// accumulation.
int oracle_expert(const float* x, int H, int I, const uint8_t* gq,
                  const uint16_t* gs, const uint8_t* uq, const uint16_t* us,
                  const uint8_t* dq, const uint16_t* ds, int prec, double* out) {
  return oracle_expert_fmt(x, H, I, 0, 32, gq, gs, uq, us, dq, ds, prec, out);
}

struct oracle_layer {
  int hidden, inter, n_experts, top_k, n_group, topk_group;
  float rsf;
  int n_shared, shared_inter;
  const float* router_w;  // [E][H]
  const float* router_b;  // [E]
  // per-expert pointer tables (entries of unselected experts may be NULL)
  const uint8_t* const* gate_q;
  const uint16_t* const* gate_s;
  const uint8_t* const* up_q;
  const uint16_t* const* up_s;
  const uint8_t* const* down_q;
  const uint16_t* const* down_s;
  const uint8_t* sh_gate_q;
  const uint16_t* sh_gate_s;
  const uint8_t* sh_up_q;
  const uint16_t* sh_up_s;
  const uint8_t* sh_down_q;
  const uint16_t* sh_down_s;
  int wfmt;  // weight format of every expert (R22): 0 int4, 1 int8
  int gsz;   // scale group: 32, or 0 for one scale per row
};

// One expert of the layer's format.
static int layer_expert(const oracle_layer* L, const float* x, int I, const uint8_t* gq,
                 const uint16_t* gs, const uint8_t* uq, const uint16_t* us, const uint8_t* dq,
                 const uint16_t* ds, int prec, double* out) {
  return oracle_expert_fmt(x, L->hidden, I, L->wfmt, L->gsz, gq, gs, uq, us, dq, ds, prec, out);
}

// Whole layer on T tokens ([P1] N1 MoE bullet, N4, G2 status; [P3]).
//   x_hat = rmsnorm(x) when gamma_or_null/eps given (eps > 0), else x
//   route x_hat -> ids, w
//   y_t   = resid_t + ( sum_j w_tj * E_{ids_tj}(x_hat_t)  +  S(x_hat_t) )
// with the routed sum taken in slot order j = 0..k-1, then the shared expert
// added, then the residual (if any).  fp32 (prec=0) or fp64 (prec=1) experts.
int oracle_moe_forward(const oracle_layer* L, const float* x, int T, double eps,
                       const float* gamma, const float* resid, int prec,
                       int32_t* ids_out, float* w_out, float* logits_out,
                       float* y) {
  const int H = L->hidden, E = L->n_experts, k = L->top_k;
  std::vector<float> xh((size_t)T * H);
  if (eps > 0) {
    if (oracle_rmsnorm(x, T, H, gamma, eps, xh.data())) return -1;
  } else {
    std::memcpy(xh.data(), x, sizeof(float) * (size_t)T * H);
  }
  std::vector<float> logits((size_t)T * E);
  if (oracle_router_logits(xh.data(), T, H, L->router_w, E, logits.data())) return -1;
  if (logits_out) std::memcpy(logits_out, logits.data(), sizeof(float) * logits.size());
  if (oracle_select(logits.data(), L->router_b, T, E, k, L->n_group, L->topk_group,
                    L->rsf, ids_out, w_out))
    return -2;
  std::vector<double> o(H), acc(H);
  for (int t = 0; t < T; ++t) {
    const float* xt = xh.data() + (size_t)t * H;
    std::vector<float> accf(H, 0.0f);
    std::vector<double> accd(H, 0.0);
    for (int j = 0; j < k; ++j) {
      const int e = ids_out[(size_t)t * k + j];
      const float wj = w_out[(size_t)t * k + j];
      if (!L->gate_q[e] || !L->gate_s[e] || !L->up_q[e] || !L->up_s[e] ||
          !L->down_q[e] || !L->down_s[e])
        return -3;  // caller did not supply a selected expert
      if (layer_expert(L, xt, L->inter, L->gate_q[e], L->gate_s[e], L->up_q[e], L->up_s[e],
                       L->down_q[e], L->down_s[e], prec, o.data()))
        return -4;
      for (int r = 0; r < H; ++r) {
        if (prec == 0)
          accf[r] = accf[r] + wj * (float)o[r];
        else
          accd[r] = accd[r] + (double)wj * o[r];
      }
    }
    if (L->n_shared > 0) {
      if (layer_expert(L, xt, L->shared_inter, L->sh_gate_q, L->sh_gate_s, L->sh_up_q,
                       L->sh_up_s, L->sh_down_q, L->sh_down_s, prec, o.data()))
        return -4;
      for (int r = 0; r < H; ++r) {
        if (prec == 0)
          accf[r] = accf[r] + (float)o[r];
        else
          accd[r] = accd[r] + o[r];
      }
    }
    for (int r = 0; r < H; ++r) {
      const float base = resid ? resid[(size_t)t * H + r] : 0.0f;
      const float v = prec == 0 ? accf[r] : (float)accd[r];
      y[(size_t)t * H + r] = resid ? base + v : v;
    }
  }
  return 0;
}

}  // extern "C"
