// Oracle for one sparse Mixture-of-Experts layer's forward pass.
//
// TEST INFRASTRUCTURE ONLY. This is a plain, slow CPU statement of what the
// layer computes, on one thread (the whole-layer forward can also split its
// token list over std::threads that run the same per-token code). Only the test suite, the smoke check
// and the benchmark's CPU-baseline leg may load it; the product library never
// does, and this file shares no code, header, table or helper with it.
//
// Every floating-point sum is accumulated in double in index order; values are
// rounded to fp32 (or bf16) only where the layer's outputs are defined in that
// type. Sources (the pages describing the "Colibri" MoE engine):
//   [OV]  "Colibri 项目概述" (trdm.cn/news/527833): §2.1 the four atomic steps
//         (routing linear+softmax, top-k with renormalised gates, dispatch by
//         expert id, per-expert FFN then weighted merge); §3.1 the expert
//         matrices w1 (gate), w3 (up), w2 (down); §3.3 dispatch grouping.
//   [GG]  "Colibri 是什么" (wzjinhao.cn/news/17934): §3.2 gating network
//         gates = softmax(x·w_gate + b_gate) with max-subtraction; §2.3 only
//         the experts that received tokens are run.
//   [EN]  "Colibri 不是一只蜂鸟" (discosf.com/news/4731160): §4.2 the
//         dispatcher's counting sort over expert ids (histogram, offsets,
//         groups in scan order).
//   [EM]  "Colibri 一个被低估的轻量级MoE推理引擎" (mhpn.cn/news/2221639):
//         §2.3 scatter into per-expert slots and copy back in token order.
//   [DD]  "一只蜂鸟如何喂饱九头大象" (wth2jhl.online, Colibri deep dive):
//         §7.3 group-wise int4 weights preferred over per-row.
//
// Readings where the pages are silent or garbled (each is also listed in the
// design notes): selection ranks logits, ties go to the lower expert index and
// slots are in descending order; the bias enters the logits before both
// selection and softmax; no capacity limit, every assignment is computed; the
// SwiGLU FFN has no biases, silu(z) = z / (1 + e^-z); within an expert group
// rows keep token order (the counting sort is stable); int4 is a signed
// two's-complement nibble (low nibble = even reduction index) times a bf16
// scale shared by 128 consecutive reduction indices of one output row; MX
// weights are OCP E4M3 bytes or E2M1 nibbles (low nibble = even index) times
// an E8M0 power of two shared by 32 consecutive reduction indices.
//
// Parity status: selection, gates, dispatch, the dense FFN special cases, the
// int4 decode and the bf16 rounding are pinned by the CPU tests; end-to-end
// values beyond those special cases are "parity unpinned" (the pages print no
// worked example).

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

enum DType { DT_F32 = 0, DT_BF16 = 1, DT_I4G128 = 2, DT_MXFP8 = 3, DT_MXFP4 = 4 };
constexpr int kGroup = 128;   // int4 scale group along the reduction index
constexpr int kMxBlock = 32;  // MX scale block along the reduction index

// OCP Microscaling (MX) element and scale formats, decoded exactly from their
// definitions (the block-scaled weight formats of the model families in
// [DD]'s table):
//   E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
//         subnormal (2^-6 * m/8); S.1111.111 is NaN; no infinities.
//   E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is
//         subnormal (m/2); values 0, 0.5, 1, 1.5, 2, 3, 4, 6.
//   E8M0: the block scale 2^(s - 127); s = 255 is NaN.
double e4m3_value(uint8_t b) {
  const int sgn = b >> 7, e = (b >> 3) & 15, m = b & 7;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  const double mag = e == 0 ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return sgn ? -mag : mag;
}
double e2m1_value(uint8_t nib) {
  const int sgn = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
  const double mag = e == 0 ? m / 2.0 : std::ldexp(1.0 + m / 2.0, e - 1);
  return sgn ? -mag : mag;
}
double e8m0_value(uint8_t s) {
  if (s == 255) return std::numeric_limits<double>::quiet_NaN();
  return std::ldexp(1.0, static_cast<int>(s) - 127);
}

// bf16 is the upper half of an IEEE binary32: widening is a 16-bit shift.
float bf16_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

// binary32 -> bf16, round to nearest, ties to even (NaN stays NaN).
uint16_t float_to_bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
    return static_cast<uint16_t>((u >> 16) | 0x0040u);
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return static_cast<uint16_t>(u >> 16);
}

// One element of an activation-typed row-major matrix (f32 or bf16 bits).
double act_at(const void* base, int dt, size_t idx) {
  if (dt == DT_F32) return static_cast<const float*>(base)[idx];
  return bf16_to_float(static_cast<const uint16_t*>(base)[idx]);
}

// A weight matrix [rows][cols] of one expert, row-major, reduction index
// contiguous (the nn.Linear "[out][in]" layout).
struct WeightView {
  const void* data;      // f32 / bf16 / e4m3 elements, or packed int4 / e2m1 bytes
  const void* scale;     // int4: bf16 [rows][cols/128]; MX: E8M0 bytes [rows][cols/32]
  int dt;
  size_t cols;
  // Decoded element, exactly: for int4, w = q * s with |q| <= 8 and an 8-bit
  // significand in s, which is exact in binary32 (and in double); for MX,
  // w = element * 2^(s - 127), exact in double.
  double at(size_t r, size_t c) const {
    if (dt == DT_F32) return static_cast<const float*>(data)[r * cols + c];
    if (dt == DT_BF16)
      return bf16_to_float(static_cast<const uint16_t*>(data)[r * cols + c]);
    if (dt == DT_MXFP8 || dt == DT_MXFP4) {
      const uint8_t s = static_cast<const uint8_t*>(scale)[r * (cols / kMxBlock) + c / kMxBlock];
      double v;
      if (dt == DT_MXFP8) {
        v = e4m3_value(static_cast<const uint8_t*>(data)[r * cols + c]);
      } else {
        const uint8_t byte = static_cast<const uint8_t*>(data)[r * (cols / 2) + c / 2];
        v = e2m1_value((c & 1) ? (byte >> 4) : (byte & 0x0f));
      }
      return v * e8m0_value(s);
    }
    const uint8_t byte = static_cast<const uint8_t*>(data)[r * (cols / 2) + c / 2];
    const int nib = (c & 1) ? (byte >> 4) : (byte & 0x0f);
    const int q = nib >= 8 ? nib - 16 : nib;
    const float s =
        bf16_to_float(static_cast<const uint16_t*>(scale)[r * (cols / kGroup) + c / kGroup]);
    return static_cast<double>(static_cast<float>(q) * s);
  }
};

WeightView expert_view(const void* w, const void* s, int dt, int e, size_t rows,
                       size_t cols) {
  WeightView v;
  v.dt = dt;
  v.cols = cols;
  v.scale = nullptr;
  const size_t n = rows * cols;
  if (dt == DT_F32) {
    v.data = static_cast<const float*>(w) + e * n;
  } else if (dt == DT_BF16) {
    v.data = static_cast<const uint16_t*>(w) + e * n;
  } else if (dt == DT_MXFP8) {
    v.data = static_cast<const uint8_t*>(w) + e * n;
    v.scale = static_cast<const uint8_t*>(s) + e * (n / kMxBlock);
  } else if (dt == DT_MXFP4) {
    v.data = static_cast<const uint8_t*>(w) + e * (n / 2);
    v.scale = static_cast<const uint8_t*>(s) + e * (n / kMxBlock);
  } else {
    v.data = static_cast<const uint8_t*>(w) + e * (n / 2);
    v.scale = static_cast<const uint16_t*>(s) + e * (n / kGroup);
  }
  return v;
}

// Router logits of one token ([GG] §3.2: x·w_gate + b_gate): the dot product
// is summed in double in index order and rounded once to fp32; the bias is
// then added in fp32.
void token_logits(const void* x, int act_dt, const void* w_r, const float* b_r,
                  int t, int d, int E, float* out) {
  for (int e = 0; e < E; ++e) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i)
      acc += act_at(x, act_dt, static_cast<size_t>(t) * d + i) *
             act_at(w_r, act_dt, static_cast<size_t>(e) * d + i);
    float l = static_cast<float>(acc);
    if (b_r) l = l + b_r[e];
    out[e] = l;
  }
}

// Top-k by rank ([OV] §2.1 "Top-k Selection"): rank(e) counts the experts
// that beat e (a larger logit, or an equal logit at a lower index). Expert e
// is selected iff rank(e) < k and goes to slot rank(e). Gates are the softmax
// over all E renormalised over the k selected, which is
// exp(l_j - l_max) / sum_{j' selected} exp(l_j' - l_max), computed in double
// ([GG] §3.2 max-subtraction) and rounded to fp32. gap = l_(k) - l_(k+1)
// (+inf when k == E); inner = smallest gap between adjacent selected slots.
void select_one(const float* l, int E, int k, int32_t* idx, float* w,
                float* gap, float* inner) {
  std::vector<int> by_rank(E, -1);
  for (int e = 0; e < E; ++e) {
    int rank = 0;
    for (int o = 0; o < E; ++o)
      if (l[o] > l[e] || (l[o] == l[e] && o < e)) ++rank;
    by_rank[rank] = e;
  }
  const double m = l[by_rank[0]];
  double denom = 0.0;
  for (int j = 0; j < k; ++j) denom += std::exp(static_cast<double>(l[by_rank[j]]) - m);
  for (int j = 0; j < k; ++j) {
    idx[j] = by_rank[j];
    w[j] = static_cast<float>(std::exp(static_cast<double>(l[by_rank[j]]) - m) / denom);
  }
  if (gap) {
    *gap = (k == E) ? std::numeric_limits<float>::infinity()
                    : l[by_rank[k - 1]] - l[by_rank[k]];
  }
  if (inner) {
    float g = std::numeric_limits<float>::infinity();
    for (int j = 0; j + 1 < k; ++j) {
      const float dj = l[by_rank[j]] - l[by_rank[j + 1]];
      if (dj < g) g = dj;
    }
    *inner = g;
  }
}

// SwiGLU expert FFN of one input row ([OV] §2.1 "Sparse Forward", §3.1 w1/w3/
// w2): a = x·Wg^T, u = x·Wu^T, h = silu(a) * u, y = h·Wd^T, all in double.
void ffn_row(const void* x_rows, int act_dt, size_t row, int d, int f,
             const WeightView& wg, const WeightView& wu, const WeightView& wd,
             std::vector<double>& h, double* y) {
  h.assign(f, 0.0);
  for (int n = 0; n < f; ++n) {
    double a = 0.0, u = 0.0;
    for (int i = 0; i < d; ++i) {
      const double xi = act_at(x_rows, act_dt, row * d + i);
      a += xi * wg.at(n, i);
      u += xi * wu.at(n, i);
    }
    h[n] = a / (1.0 + std::exp(-a)) * u;
  }
  for (int o = 0; o < d; ++o) {
    double acc = 0.0;
    for (int n = 0; n < f; ++n) acc += h[n] * wd.at(o, n);
    y[o] = acc;
  }
}

bool bad_dims(int T, int d, int E, int k) {
  return T < 0 || d <= 0 || E <= 0 || k <= 0 || k > E;
}

// The layer for list positions [i0, i1) of the token list: route and select
// the token's k experts, then y[t] = sum_j g_j * FFN_{e_j}(x[t]) in double
// with j ascending ([OV] section 2.1: routing, top-k, per-expert FFN, weighted
// merge). Writes only the rows of its own positions. Returns -1 on a token
// index outside [0, T).
struct ForwardArgs {
  const void *x, *w_r, *w_gate, *w_up, *w_down, *s_gate, *s_up, *s_down;
  const float* b_r;
  int act_dt, T, d, E, k, w_dt, f;
  const int32_t* tokens;
  double* y_f64;
  void* y_out;
  int32_t* topk_idx;
  float* topk_w;
  float* gap;
};

int forward_range(const ForwardArgs& A, int i0, int i1) {
  const int d = A.d, k = A.k, f = A.f;
  std::vector<float> l(A.E);
  std::vector<int32_t> idx(k);
  std::vector<float> g(k);
  std::vector<double> yt(d), ye(d), h;
  for (int i = i0; i < i1; ++i) {
    const int t = A.tokens ? A.tokens[i] : i;
    if (t < 0 || t >= A.T) return -1;
    token_logits(A.x, A.act_dt, A.w_r, A.b_r, t, d, A.E, l.data());
    float gp = 0.f;
    select_one(l.data(), A.E, k, idx.data(), g.data(), &gp, nullptr);
    for (int o = 0; o < d; ++o) yt[o] = 0.0;
    for (int j = 0; j < k; ++j) {
      const int e = idx[j];
      const WeightView wg = expert_view(A.w_gate, A.s_gate, A.w_dt, e, f, d);
      const WeightView wu = expert_view(A.w_up, A.s_up, A.w_dt, e, f, d);
      const WeightView wd = expert_view(A.w_down, A.s_down, A.w_dt, e, d, f);
      ffn_row(A.x, A.act_dt, t, d, f, wg, wu, wd, h, ye.data());
      for (int o = 0; o < d; ++o) yt[o] += static_cast<double>(g[j]) * ye[o];
    }
    for (int o = 0; o < d; ++o) {
      const size_t q = static_cast<size_t>(i) * d + o;
      if (A.y_f64) A.y_f64[q] = yt[o];
      if (A.y_out) {
        const float v = static_cast<float>(yt[o]);
        if (A.act_dt == DT_F32) static_cast<float*>(A.y_out)[q] = v;
        else static_cast<uint16_t*>(A.y_out)[q] = float_to_bf16_rne(v);
      }
    }
    if (A.topk_idx)
      for (int j = 0; j < k; ++j) A.topk_idx[static_cast<size_t>(i) * k + j] = idx[j];
    if (A.topk_w)
      for (int j = 0; j < k; ++j) A.topk_w[static_cast<size_t>(i) * k + j] = g[j];
    if (A.gap) A.gap[i] = gp;
  }
  return 0;
}

}  // namespace

extern "C" {

int oracle_version(void) { return 1; }

float oracle_bf16_to_float(uint16_t b) { return bf16_to_float(b); }
uint16_t oracle_float_to_bf16(float f) { return float_to_bf16_rne(f); }

// One E4M3 / E2M1 / E8M0 code, decoded (for the MX pins).
double oracle_mx_element(int w_dt, int code) {
  if (w_dt == DT_MXFP8) return e4m3_value(static_cast<uint8_t>(code));
  if (w_dt == DT_MXFP4) return e2m1_value(static_cast<uint8_t>(code & 15));
  return e8m0_value(static_cast<uint8_t>(code));
}

// Decoded weight element (for the int4 and MX pins).
double oracle_weight_at(const void* w, const void* s, int w_dt, int e, int rows,
                        int cols, int r, int c) {
  return expert_view(w, s, w_dt, e, rows, cols).at(r, c);
}

// logits [T][E] in fp32.
int oracle_router_logits(const void* x, int act_dt, const void* w_r,
                         const float* b_r, int T, int d, int E, float* logits) {
  if (bad_dims(T, d, E, 1) || !x || !w_r || !logits) return -1;
  for (int t = 0; t < T; ++t)
    token_logits(x, act_dt, w_r, b_r, t, d, E, logits + static_cast<size_t>(t) * E);
  return 0;
}

// Selection + gates from given fp32 logits [T][E].
int oracle_select_topk(const float* logits, int T, int E, int k,
                       int32_t* topk_idx, float* topk_w, float* gap,
                       float* inner_gap) {
  if (bad_dims(T, 1, E, k) || !logits || !topk_idx || !topk_w) return -1;
  for (int t = 0; t < T; ++t)
    select_one(logits + static_cast<size_t>(t) * E, E, k, topk_idx + static_cast<size_t>(t) * k,
               topk_w + static_cast<size_t>(t) * k, gap ? gap + t : nullptr,
               inner_gap ? inner_gap + t : nullptr);
  return 0;
}

// Dispatch ([EN] §4.2 counting sort; [OV] §3.3 grouping by expert): counts,
// exclusive offsets [E+1], and a stable scatter of the T*k assignments taken
// in (t, j) order: row = offsets[e] + (number of earlier assignments to e).
// Returns -1 on an out-of-range expert id.
int oracle_dispatch(const int32_t* topk_idx, int T, int k, int E, int32_t* counts,
                    int32_t* offsets, int32_t* row_token, int32_t* assign_row) {
  if (bad_dims(T, 1, E, k) || !topk_idx || !counts || !offsets) return -1;
  const size_t n = static_cast<size_t>(T) * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (size_t a = 0; a < n; ++a) {
    const int e = topk_idx[a];
    if (e < 0 || e >= E) return -1;
    counts[e] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int32_t> next(offsets, offsets + E);
  for (size_t a = 0; a < n; ++a) {
    const int e = topk_idx[a];
    const int32_t row = next[e]++;
    if (row_token) row_token[row] = static_cast<int32_t>(a / k);
    if (assign_row) assign_row[a] = row;
  }
  return 0;
}

// FFN of expert e on n_rows input rows x_rows [n_rows][d] (act dtype);
// y_rows [n_rows][d] in double. Weights in the canonical layouts:
// gate/up [E][f][d], down [E][d][f] (int4: bytes [..][cols/2] plus bf16
// scales [..][cols/128]).
int oracle_expert_ffn(const void* x_rows, int act_dt, int n_rows, const void* w_gate,
                      const void* w_up, const void* w_down, const void* s_gate,
                      const void* s_up, const void* s_down, int w_dt, int e, int d,
                      int f, double* y_rows) {
  if (n_rows < 0 || d <= 0 || f <= 0 || e < 0 || !y_rows) return -1;
  if (w_dt == DT_I4G128 && (d % kGroup || f % kGroup)) return -1;
  if ((w_dt == DT_MXFP8 || w_dt == DT_MXFP4) && (d % kMxBlock || f % kMxBlock)) return -1;
  const WeightView wg = expert_view(w_gate, s_gate, w_dt, e, f, d);
  const WeightView wu = expert_view(w_up, s_up, w_dt, e, f, d);
  const WeightView wd = expert_view(w_down, s_down, w_dt, e, d, f);
  std::vector<double> h;
  for (int r = 0; r < n_rows; ++r)
    ffn_row(x_rows, act_dt, r, d, f, wg, wu, wd, h, y_rows + static_cast<size_t>(r) * d);
  return 0;
}

// Weighted merge back to token order ([OV] §2.1, [EM] §2.3):
// y[t] = sum_{j ascending} g[t][j] * y_perm[assign_row[t*k+j]], in double.
// y_out (nullable) receives y rounded to the output dtype (fp32, or fp32 then
// bf16 by round-to-nearest-even).
int oracle_combine(const float* y_perm, const int32_t* assign_row, const float* topk_w,
                   int T, int k, int d, int out_dt, double* y_f64, void* y_out) {
  if (T < 0 || k <= 0 || d <= 0 || !y_perm || !assign_row || !topk_w) return -1;
  for (int t = 0; t < T; ++t) {
    for (int o = 0; o < d; ++o) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) {
        const size_t a = static_cast<size_t>(t) * k + j;
        acc += static_cast<double>(topk_w[a]) *
               y_perm[static_cast<size_t>(assign_row[a]) * d + o];
      }
      const size_t i = static_cast<size_t>(t) * d + o;
      if (y_f64) y_f64[i] = acc;
      if (y_out) {
        const float v = static_cast<float>(acc);
        if (out_dt == DT_F32) static_cast<float*>(y_out)[i] = v;
        else static_cast<uint16_t*>(y_out)[i] = float_to_bf16_rne(v);
      }
    }
  }
  return 0;
}

// The same layer with the token list split into n_threads contiguous ranges,
// one std::thread each. Every token is computed by the same code as in the
// single-threaded call and written to its own rows, so the outputs are
// bit-identical to it for any n_threads (n_threads <= 1 runs on the calling
// thread).
int oracle_moe_forward_mt(const void* x, int act_dt, int T, int d, const void* w_r,
                          const float* b_r, int E, int k, const void* w_gate,
                          const void* w_up, const void* w_down, const void* s_gate,
                          const void* s_up, const void* s_down, int w_dt, int f,
                          const int32_t* tokens, int n_tokens, double* y_f64,
                          void* y_out, int32_t* topk_idx, float* topk_w, float* gap,
                          int n_threads) {
  if (bad_dims(T, d, E, k) || f <= 0 || !x || !w_r) return -1;
  if (tokens && n_tokens < 0) return -1;
  const int n = tokens ? n_tokens : T;
  const ForwardArgs A{x,      w_r,    w_gate, w_up, w_down, s_gate, s_up, s_down, b_r,
                      act_dt, T,      d,      E,    k,      w_dt,   f,    tokens, y_f64,
                      y_out,  topk_idx, topk_w, gap};
  int nt = n_threads < 1 ? 1 : n_threads;
  if (nt > n) nt = n > 0 ? n : 1;
  if (nt == 1) return forward_range(A, 0, n);
  std::vector<int> rc(nt, 0);
  std::vector<std::thread> pool;
  pool.reserve(nt);
  for (int w = 0; w < nt; ++w) {
    const int i0 = static_cast<int>(static_cast<long>(n) * w / nt);
    const int i1 = static_cast<int>(static_cast<long>(n) * (w + 1) / nt);
    pool.emplace_back([&A, &rc, w, i0, i1] { rc[w] = forward_range(A, i0, i1); });
  }
  for (auto& th : pool) th.join();
  for (int r : rc)
    if (r != 0) return r;
  return 0;
}

// Whole layer for the listed tokens (all T when tokens == NULL): route, select,
// then y[t] = sum_j g_j * FFN_{e_j}(x[t]). Outputs are per listed token:
// y_f64 [n][d] (nullable), y_out [n][d] in the act dtype (nullable),
// topk_idx/topk_w [n][k] and gap [n] (nullable).
int oracle_moe_forward(const void* x, int act_dt, int T, int d, const void* w_r,
                       const float* b_r, int E, int k, const void* w_gate,
                       const void* w_up, const void* w_down, const void* s_gate,
                       const void* s_up, const void* s_down, int w_dt, int f,
                       const int32_t* tokens, int n_tokens, double* y_f64,
                       void* y_out, int32_t* topk_idx, float* topk_w, float* gap) {
  return oracle_moe_forward_mt(x, act_dt, T, d, w_r, b_r, E, k, w_gate, w_up, w_down,
                               s_gate, s_up, s_down, w_dt, f, tokens, n_tokens, y_f64,
                               y_out, topk_idx, topk_w, gap, 1);
}

}  // extern "C"
