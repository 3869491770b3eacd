// A1: router linear + softmax + top-k + renormalised gates.
//
// Gating is softmax(x·W_r^T + b) over the E experts (wzjinhao.cn "Colibri
// 是什么", section 3.2); the k largest are kept and their gates renormalised
// (overview page trdm.cn, section 2.1 "Top-k Selection"); the router hands on
// only k ids and k scores per token (discosf.com page, section 2.1).
//
// E <= 32: one fused kernel, one block per token. Its warps split the
// reduction index (a single warp per token leaves the GPU latency-bound at
// decode batch sizes), the partial sums meet in shared memory in fixed warp
// order, and the selection runs warp-per-token: lane e holds the logit of
// expert e in a register and ranks it against the others,
// rank(e) = #{e' : l[e'] > l[e] or (l[e'] == l[e] and e' < e)}.
// E > 32: logits are too many for one warp's registers and W_r too large to
// re-read per token, so a tiled kernel (tensor cores for bf16, CUDA cores for
// fp32) first writes partial dot products over token x expert x
// reduction-slice tiles (fixed slice order, no atomics),
// then a warp-per-token kernel sums the slices, keeps E/32 logits per lane in
// registers and takes k+1 rounds of warp arg-max (larger value, then lower
// index) for the top-k and the k-th/(k+1)-th gap.
//
// Logits are fp32 dot products (bf16 inputs widened exactly) plus the bias in
// fp32. Gates use expf with max-subtraction (same page, section 3.2).
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace coli {
namespace {

constexpr int kWarps = 8;
// bf16 batches of at least this many tokens take the one-launch tiled router
constexpr int kTiledMinTokens = 1024;

COLI_DEV void load8(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

COLI_DEV void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x);
  v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
  v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z);
  v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
}

COLI_DEV bool beats(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// A NaN logit (e.g. from an overflowed input row) would compare false both
// ways and break the ranking; it is ranked as -inf instead, and the token's
// data error is latched.
COLI_DEV float rankable(float v, int* status) {
  if (v != v) {
    latch_error(status, kErrDevice);
    return -INFINITY;
  }
  return v;
}

// Value of the lane that holds `rank` (exactly one lane does).
COLI_DEV float from_rank(int my_rank, float my_val, int rank) {
  const unsigned m = __ballot_sync(0xffffffffu, my_rank == rank);
  return __shfl_sync(0xffffffffu, my_val, __ffs(m) - 1);
}

template <typename TA, int EMAX>
__global__ void __launch_bounds__(kWarps * 32)
    k_route_fused(const TA* __restrict__ x, const TA* __restrict__ w, const float* __restrict__ b,
                  int T, int d, int E, int k, int32_t* __restrict__ topk_idx,
                  float* __restrict__ topk_w, float* __restrict__ gap, int* status) {
  // one block per token: the 8 warps take interleaved 8-wide slices of the
  // reduction index, then warp 0 adds the 8 partial sums in warp order
  __shared__ float part[kWarps][EMAX];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x;
  float acc[EMAX];
#pragma unroll
  for (int e = 0; e < EMAX; ++e) acc[e] = 0.f;
  const TA* xr = x + static_cast<size_t>(t) * d;
  // unrolled so the loads of several slices are in flight at once (less for
  // many experts, whose accumulators already take the registers)
  constexpr int kUnroll = EMAX <= 8 ? 4 : (EMAX <= 16 ? 2 : 1);
#pragma unroll kUnroll
  for (int i = (warp * 32 + lane) * 8; i < d; i += kWarps * 256) {
    float xv[8];
    load8(xr + i, xv);
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
      if (e < E) {
        float wv[8];
        load8(w + static_cast<size_t>(e) * d + i, wv);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[e] = fmaf(xv[j], wv[j], acc[e]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < EMAX; ++e) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
  }
  if (lane == 0) {
#pragma unroll
    for (int e = 0; e < EMAX; ++e) part[warp][e] = acc[e];
  }
  __syncthreads();
  if (warp != 0) return;
  // lane e owns expert e
  const bool mine = lane < E;
  float le = -INFINITY;
  if (mine) {
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) v += part[i][lane];
    le = rankable((b != nullptr) ? v + b[lane] : v, status);
  }
  int rank = 0;
  for (int e = 0; e < E; ++e) {
    const float o = __shfl_sync(0xffffffffu, le, e);
    if (beats(o, e, le, lane)) ++rank;
  }
  if (!mine) rank = 1 << 20;
  const float m = from_rank(rank, le, 0);
  const bool sel = mine && rank < k;
  const float ex = sel ? expf(le - m) : 0.f;
  float den = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  if (sel) {
    topk_idx[static_cast<size_t>(t) * k + rank] = lane;
    topk_w[static_cast<size_t>(t) * k + rank] = ex / den;
  }
  if (gap != nullptr) {
    float g = INFINITY;
    if (k < E) g = from_rank(rank, le, k - 1) - from_rank(rank, le, k);
    if (lane == 0) gap[t] = g;
  }
}

// ---- E > 32 ---------------------------------------------------------------------
constexpr int kTT = 16;   // tokens per tile
constexpr int kTE = 64;   // experts per tile
constexpr int kKS = 512;  // reduction slice per CTA
constexpr int kKC = 32;   // reduction chunk staged in shared memory

template <typename TA>
__global__ void __launch_bounds__(128)
    k_route_partial(const TA* __restrict__ x, const TA* __restrict__ w, int T, int d, int E,
                    float* __restrict__ part) {
  __shared__ float xs[kTT][kKC + 1];
  __shared__ float ws[kTE][kKC + 1];
  const int t0 = blockIdx.x * kTT, e0 = blockIdx.y * kTE, k0 = blockIdx.z * kKS;
  const int k1 = min(d, k0 + kKS);
  const int tid = threadIdx.x;
  const int tp = tid >> 4;   // tokens 2tp, 2tp+1
  const int eq = tid & 15;   // experts 4eq..4eq+3
  float acc[2][4] = {};
  for (int kk = k0; kk < k1; kk += kKC) {
    for (int i = tid; i < kTT * kKC; i += 128) {
      const int r = i / kKC, c = i % kKC, t = t0 + r;
      xs[r][c] = (t < T) ? to_f32(x[static_cast<size_t>(t) * d + kk + c]) : 0.f;
    }
    for (int i = tid; i < kTE * kKC; i += 128) {
      const int r = i / kKC, c = i % kKC, e = e0 + r;
      ws[r][c] = (e < E) ? to_f32(w[static_cast<size_t>(e) * d + kk + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < kKC; ++c) {
      const float xa = xs[2 * tp][c], xb = xs[2 * tp + 1][c];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float wv = ws[4 * eq + j][c];
        acc[0][j] = fmaf(xa, wv, acc[0][j]);
        acc[1][j] = fmaf(xb, wv, acc[1][j]);
      }
    }
    __syncthreads();
  }
  float* dst = part + static_cast<size_t>(blockIdx.z) * T * E;
#pragma unroll
  for (int a = 0; a < 2; ++a) {
    const int t = t0 + 2 * tp + a;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + 4 * eq + j;
      if (e < E) dst[static_cast<size_t>(t) * E + e] = acc[a][j];
    }
  }
}

// Tensor-core logits for bf16 inputs: a block of 4 warps takes 16 tokens x
// 64 experts over one 512-wide reduction slice with mma.sync m16n8k16
// (tokens are M, experts N; warp w owns experts 16w..16w+15). Four 32-index
// steps of loads are issued before any is used, so 8 KiB per warp are in
// flight (the slice is latency-bound otherwise); the four warps read the
// same token rows, which L1 serves after the first. Products of bf16 values
// are exact in fp32; to keep the sum at fp32 round-to-nearest accuracy
// whatever the tensor core's internal adder does, every 32-index step goes
// into a zeroed accumulator that is added to the running sum with an FADD.
// Same partial-slice output as k_route_partial.
constexpr int kTcTok = 16, kTcExp = 64;

__global__ void __launch_bounds__(128)
    k_route_partial_tc(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w,
                       int T, int d, int E, float* __restrict__ part) {
  constexpr int U = 4;
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * kTcTok;
  const int e0 = blockIdx.y * kTcExp + 16 * warp;
  const int k0 = blockIdx.z * kKS, k1 = min(d, k0 + kKS);
  const __nv_bfloat16* xr0 = (t0 + g < T) ? x + static_cast<size_t>(t0 + g) * d + q * 8 : nullptr;
  const __nv_bfloat16* xr8 =
      (t0 + g + 8 < T) ? x + static_cast<size_t>(t0 + g + 8) * d + q * 8 : nullptr;
  const __nv_bfloat16* wr[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int e = e0 + 8 * j + g;
    wr[j] = e < E ? w + static_cast<size_t>(e) * d + q * 8 : nullptr;
  }
  float acc[2][4] = {};
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int k = k0; k < k1; k += 32 * U) {
    uint4 a[U], a8[U], b[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int kk = k + 32 * u;
      const bool in = kk < k1;
      a[u] = (in && xr0) ? *reinterpret_cast<const uint4*>(xr0 + kk) : z;
      a8[u] = (in && xr8) ? *reinterpret_cast<const uint4*>(xr8 + kk) : z;
#pragma unroll
      for (int j = 0; j < 2; ++j)
        b[u][j] = (in && wr[j]) ? *reinterpret_cast<const uint4*>(wr[j] + kk) : z;
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float t[4] = {0.f, 0.f, 0.f, 0.f};
        mma_bf16_16816(t, a[u].x, a8[u].x, a[u].y, a8[u].y, b[u][j].x, b[u][j].y);
        mma_bf16_16816(t, a[u].z, a8[u].z, a[u].w, a8[u].w, b[u][j].z, b[u][j].w);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[j][c] += t[c];
      }
  }
  float* dst = part + static_cast<size_t>(blockIdx.z) * T * E;
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int t = t0 + g + ((c & 2) ? 8 : 0);
      const int e = e0 + 8 * j + 2 * q + (c & 1);
      if (t < T && e < E) dst[static_cast<size_t>(t) * E + e] = acc[j][c];
    }
}

// Order-preserving integer key of a float: a larger float gets a larger key
// (-0 is folded into +0 first, so the two compare equal as floats do). Key 0
// is below every float, including -inf.
COLI_DEV uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v + 0.f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
COLI_DEV float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// One warp, one token: lane holds the logits of experts lane + 32 i (-inf
// past E). k+1 rounds of warp arg-max (larger value, then lower index) give
// the top-k in descending order and the k-th/(k+1)-th gap. A round is one
// warp max over the order keys and one warp min over the indices of the
// lanes that hold that key. The gates are exp(l_j - l_max) / sum_j'
// exp(l_j' - l_max), summed with j ascending.
template <int PER_LANE>
COLI_DEV void select_token(const float (&l)[PER_LANE], int E, int k, int t,
                           int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                           float* __restrict__ gap) {
  const int lane = threadIdx.x & 31;
  uint32_t key[PER_LANE];
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) key[i] = (lane + 32 * i < E) ? order_key(l[i]) : 0u;
  float sel_val[8];
  int sel_idx[8];
  float kth = 0.f, next = INFINITY;  // l_(k) and l_(k+1)
  const int rounds = min(k + 1, E);
#pragma unroll
  for (int r = 0; r < 9; ++r) {
    if (r < 8) {
      sel_val[r] = -INFINITY;
      sel_idx[r] = 0;
    }
    if (r < rounds) {
      // this lane's best remaining key (lower slot = lower index on ties)
      uint32_t best = 0u;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < PER_LANE; ++i)
        if (key[i] > best) {
          best = key[i];
          bi = lane + 32 * i;
        }
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, best);
      const uint32_t cand = (best == kmax && best != 0u) ? static_cast<uint32_t>(bi) : 0xffffffffu;
      const int win = static_cast<int>(__reduce_min_sync(0xffffffffu, cand));
      if ((win & 31) == lane) {
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i)
          if (i == (win >> 5)) key[i] = 0u;  // taken
      }
      const float v = key_value(kmax);
      if (r < 8) {
        sel_val[r] = v;
        sel_idx[r] = win;
      }
      if (r == k - 1) kth = v;
      if (r == k) next = v;
    }
  }
  if (gap != nullptr && lane == 0) gap[t] = (k < E) ? kth - next : INFINITY;
  const float best0 = sel_val[0];
  float den = 0.f, mine = 0.f;
  int id = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < k) {
      const float ex = expf(sel_val[j] - best0);
      den += ex;
      if (j == lane) {
        mine = ex;
        id = sel_idx[j];
      }
    }
  if (lane < k) {
    topk_idx[static_cast<size_t>(t) * k + lane] = id;
    topk_w[static_cast<size_t>(t) * k + lane] = mine / den;
  }
}

// Blocks of kSelWarps warps, one token per warp: a few hundred tokens still
// spread over most SMs. Each expert's logit is the slice sum in slice order;
// the slices are the outer loop, so a lane has its PER_LANE loads of a slice
// in flight together.
constexpr int kSelWarps = 2;

template <int PER_LANE>
__global__ void __launch_bounds__(kSelWarps * 32)
    k_route_select(const float* __restrict__ part, int slices, const float* __restrict__ b,
                   int T, int E, int k, int32_t* __restrict__ topk_idx,
                   float* __restrict__ topk_w, float* __restrict__ gap, int* status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kSelWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  float l[PER_LANE];
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) l[i] = 0.f;
  const float* row = part + static_cast<size_t>(t) * E + lane;
  for (int s = 0; s < slices; ++s) {
    const float* ps = row + static_cast<size_t>(s) * T * E;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i)
      if (lane + 32 * i < E) l[i] += ps[32 * i];
  }
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) {
    const int e = lane + 32 * i;
    float v = -INFINITY;
    if (e < E) {
      v = l[i];
      if (b != nullptr) v += b[e];
      v = rankable(v, status);
    }
    l[i] = v;
  }
  select_token<PER_LANE>(l, E, k, t, topk_idx, topk_w, gap);
}

// ---- bf16, many tokens: one launch ------------------------------------------------
// A block takes 32 tokens and all E experts. Its 8 warps compute the logits
// with mma.sync m16n8k16 (tokens M, experts N, both m-tiles of the block per
// warp so each W_r fragment feeds two MMAs): with NT = ceil(E/8) expert
// tiles, warp w takes expert tiles w % G, w % G + G, ... (G = 8 / ks groups)
// over the ks-th part w / G of the reduction (ks = 8 / NT splits when NT < 8,
// so small E still keeps all warps busy). Every 32-index step goes into a
// zeroed accumulator that is then added with an FADD (fp32 sum of 32-term
// partials, as in the two-launch path), four steps in flight on four running
// sums. Partial logits meet in shared memory, summed over the reduction
// parts in fixed order, plus the bias; then each warp selects for 4 tokens.
constexpr int kTok = 32;

__global__ void __launch_bounds__(256)
    k_route_tc(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w,
               const float* __restrict__ b, int T, int d, int E, int k, int ks,
               int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
               float* __restrict__ gap, int* status) {
  extern __shared__ float sl[];  // [ks][kTok][E] partial logits
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int t0 = blockIdx.x * kTok;
  const int NT = (E + 7) / 8;
  const int G = 8 / ks;
  const int grp = warp % G, kp = warp / G;
  const int steps = d / 32;
  const int s0 = steps * kp / ks, s1 = steps * (kp + 1) / ks;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  // The block's token rows are its only DRAM stream and its warps walk them
  // together a few steps ahead: bring them all into L2 at once (one bulk
  // prefetch per row) so the loads below wait on L2, not on DRAM.
  if (threadIdx.x < kTok && t0 + threadIdx.x < T) {
    const __nv_bfloat16* row = x + static_cast<size_t>(t0 + threadIdx.x) * d;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(row),
                 "r"(static_cast<uint32_t>(d * 2))
                 : "memory");
  }
  const __nv_bfloat16* xr[2][2];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = t0 + 16 * m + g + 8 * h;
      xr[m][h] = t < T ? x + static_cast<size_t>(t) * d + q * 8 : nullptr;
    }
  for (int nt = grp; nt < NT; nt += G) {
    const int e = nt * 8 + g;
    const __nv_bfloat16* wr = e < E ? w + static_cast<size_t>(e) * d + q * 8 : nullptr;
    constexpr int U = 4;
    float acc[U][2][4];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[u][m][c] = 0.f;
    for (int s = s0; s < s1; s += U) {
      uint4 a[U][2][2], bw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const bool in = s + u < s1;
        const int kk = (s + u) * 32;
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int h = 0; h < 2; ++h)
            a[u][m][h] = (in && xr[m][h]) ? *reinterpret_cast<const uint4*>(xr[m][h] + kk) : z;
        bw[u] = (in && wr) ? *reinterpret_cast<const uint4*>(wr + kk) : z;
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          float t4[4] = {0.f, 0.f, 0.f, 0.f};
          mma_bf16_16816(t4, a[u][m][0].x, a[u][m][1].x, a[u][m][0].y, a[u][m][1].y, bw[u].x,
                         bw[u].y);
          mma_bf16_16816(t4, a[u][m][0].z, a[u][m][1].z, a[u][m][0].w, a[u][m][1].w, bw[u].z,
                         bw[u].w);
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[u][m][c] += t4[c];
        }
    }
    // (sum0 + sum1) + (sum2 + sum3), then the block's shared partial table
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float v = (acc[0][m][c] + acc[1][m][c]) + (acc[2][m][c] + acc[3][m][c]);
        const int tl = 16 * m + g + ((c & 2) ? 8 : 0);
        const int ee = nt * 8 + 2 * q + (c & 1);
        if (ee < E) sl[(static_cast<size_t>(kp) * kTok + tl) * E + ee] = v;
      }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kTok * E; i += blockDim.x) {
    float v = 0.f;
    for (int p = 0; p < ks; ++p) v += sl[static_cast<size_t>(p) * kTok * E + i];
    if (b != nullptr) v += b[i % E];
    sl[i] = v;
  }
  __syncthreads();
#define COLI_SELECT_TOKENS(PL)                                                    \
  for (int j = 0; j < kTok / 8; ++j) {                                            \
    const int tl = warp * (kTok / 8) + j, t = t0 + tl;                            \
    if (t >= T) break;                                                            \
    float l[PL];                                                                  \
    _Pragma("unroll") for (int i = 0; i < PL; ++i) {                              \
      const int e = lane + 32 * i;                                                \
      l[i] = e < E ? rankable(sl[tl * E + e], status) : -INFINITY;               \
    }                                                                             \
    select_token<PL>(l, E, k, t, topk_idx, topk_w, gap);                          \
  }
  if (E <= 32) {
    COLI_SELECT_TOKENS(1)
  } else if (E <= 64) {
    COLI_SELECT_TOKENS(2)
  } else if (E <= 128) {
    COLI_SELECT_TOKENS(4)
  } else {
    COLI_SELECT_TOKENS(8)
  }
#undef COLI_SELECT_TOKENS
}

// ---- bf16, many tokens, E > 32: one launch, pipelined -------------------------------
// A block takes 64 tokens and all E experts. The reduction runs in chunks of
// KC indices: 256 threads copy the chunk's token rows and W_r rows into a
// 3-stage shared-memory ring with 16-byte cp.async (rows past T or E are
// zero-filled), row pitch KC*2 + 64 bytes so the fragment loads of a
// quarter-warp hit 8 distinct bank groups. Warp w owns expert tiles w, w+8,
// w+16, w+24 (8 experts each) for all four 16-token tiles; each 64 indices
// go into a fresh mma.sync accumulator (zero input) that is added to the
// running sum with an FADD, so the tensor core never carries a sum across
// more than 64 products. The ring is then reused for the [64][E]
// logit table, plus the bias, and each warp selects for 8 tokens.
constexpr int kBigTok = 64;
constexpr int kBigStages = 3;

COLI_DEV void cp_async16_zfill(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}

template <int KC>
constexpr int big_pitch() { return KC * 2 + 64; }

template <int KC>
size_t big_smem_bytes(int E) {
  const size_t ring = static_cast<size_t>(kBigStages) * (kBigTok + ((E + 7) / 8) * 8) *
                      big_pitch<KC>();
  const size_t table = static_cast<size_t>(kBigTok) * E * sizeof(float);
  return ring > table ? ring : table;
}

template <int KC>
__global__ void __launch_bounds__(256, 1)
    k_route_tc_big(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w,
                   const float* __restrict__ b, int T, int d, int E, int k,
                   int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                   float* __restrict__ gap, int* status) {
  extern __shared__ __align__(16) uint8_t rsm[];
  constexpr int P = big_pitch<KC>();
  constexpr int CH = KC / 8;  // 16-byte pieces per row and chunk
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int t0 = blockIdx.x * kBigTok;
  const int NT = (E + 7) / 8, Ep = NT * 8;
  const int rows = kBigTok + Ep;  // token rows, then expert rows, per stage
  const uint32_t base = smem_u32(rsm);
  const uint32_t stage_bytes = static_cast<uint32_t>(rows) * P;
  const int chunks = d / KC;

  // this thread's copies of a chunk: fixed (row, piece) pairs, so the source
  // pointers and shared offsets are computed once; a chunk moves them by KC
  constexpr int kMaxPieces = (kBigTok + (KC == 128 ? 128 : 256)) * CH / 256;
  const __nv_bfloat16* src0[kMaxPieces];
  uint32_t dst0[kMaxPieces];
  uint32_t valid_mask = 0, live_mask = 0;
#pragma unroll
  for (int u = 0; u < kMaxPieces; ++u) {
    const int i = threadIdx.x + 256 * u;
    const int r = i / CH, piece = i % CH;
    const bool live = r < rows;
    const bool tok = r < kBigTok;
    const int src_row = tok ? t0 + r : r - kBigTok;
    const bool valid = live && (tok ? src_row < T : src_row < E);
    src0[u] = (tok ? x : w) + (valid ? static_cast<size_t>(src_row) * d : 0) + piece * 8;
    dst0[u] = r * P + piece * 16;
    if (valid) valid_mask |= 1u << u;
    if (live) live_mask |= 1u << u;
  }
  auto issue = [&](int c) {
    if (c < chunks) {
      const uint32_t sb = base + (c % kBigStages) * stage_bytes;
#pragma unroll
      for (int u = 0; u < kMaxPieces; ++u)
        if (live_mask & (1u << u))
          cp_async16_zfill(sb + dst0[u], src0[u] + c * KC, (valid_mask >> u) & 1u);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int c = 0; c < kBigStages - 1; ++c) issue(c);

  float acc[4][4][4];  // [expert tile slot][token tile][c]
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[j][m][c] = 0.f;

  for (int c = 0; c < chunks; ++c) {
    cp_async_wait<kBigStages - 2>();  // chunk c has landed (this thread's copies)
    __syncthreads();                  // ... and everyone's; the slot of chunk c-1 is free
    issue(c + kBigStages - 1);
    const uint32_t sb = base + (c % kBigStages) * stage_bytes;
    // 64 indices (two 32-index steps, four MMAs) per fresh accumulator
#pragma unroll
    for (int st = 0; st < KC / 32; st += 2) {
      uint4 a[2][4][2];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int h = 0; h < 2; ++h)
            a[u][m][h] = lds128(sb + (16 * m + g + 8 * h) * P + (st + u) * 64 + q * 16);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int nt = warp + 8 * j;
        if (nt < NT) {
          uint4 bw[2];
#pragma unroll
          for (int u = 0; u < 2; ++u)
            bw[u] = lds128(sb + (kBigTok + nt * 8 + g) * P + (st + u) * 64 + q * 16);
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            float t4[4];
            mma_bf16_16816_z(t4, a[0][m][0].x, a[0][m][1].x, a[0][m][0].y, a[0][m][1].y,
                             bw[0].x, bw[0].y);
            mma_bf16_16816(t4, a[0][m][0].z, a[0][m][1].z, a[0][m][0].w, a[0][m][1].w, bw[0].z,
                           bw[0].w);
            mma_bf16_16816(t4, a[1][m][0].x, a[1][m][1].x, a[1][m][0].y, a[1][m][1].y, bw[1].x,
                           bw[1].y);
            mma_bf16_16816(t4, a[1][m][0].z, a[1][m][1].z, a[1][m][0].w, a[1][m][1].w, bw[1].z,
                           bw[1].w);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) acc[j][m][cc] += t4[cc];
          }
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // the ring becomes the logit table
  float* lt = reinterpret_cast<float*>(rsm);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int nt = warp + 8 * j;
    if (nt >= NT) continue;
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int tl = 16 * m + g + ((cc & 2) ? 8 : 0);
        const int e = nt * 8 + 2 * q + (cc & 1);
        if (e < E) lt[tl * E + e] = acc[j][m][cc] + (b != nullptr ? b[e] : 0.f);
      }
  }
  __syncthreads();
#define COLI_SELECT_BIG(PL)                                                       \
  for (int jt = 0; jt < kBigTok / 8; ++jt) {                                      \
    const int tl = warp * (kBigTok / 8) + jt, t = t0 + tl;                        \
    if (t >= T) break;                                                            \
    float l[PL];                                                                  \
    _Pragma("unroll") for (int i = 0; i < PL; ++i) {                              \
      const int e = lane + 32 * i;                                                \
      l[i] = e < E ? rankable(lt[tl * E + e], status) : -INFINITY;               \
    }                                                                             \
    select_token<PL>(l, E, k, t, topk_idx, topk_w, gap);                          \
  }
  if (E <= 64) {
    COLI_SELECT_BIG(2)
  } else if (E <= 128) {
    COLI_SELECT_BIG(4)
  } else {
    COLI_SELECT_BIG(8)
  }
#undef COLI_SELECT_BIG
}

// ---- bf16, many tokens, 32 < E <= 128: tensor cores with tensor memory ----------------
// A CTA takes 128 tokens (the MMA's M, one tensor-memory lane each) and all E
// experts (N = E rounded up to 16). TMA brings 64-index chunks of the token
// rows and of W_r (128-byte swizzle) into a 6-stage ring, so a CTA keeps up
// to 144 KiB of loads in flight and one wave of CTAs streams x at HBM speed.
// One thread issues tcgen05.mma; every chunk goes into a fresh accumulator
// (one of four tensor-memory buffers), and the thread of each token adds the
// chunk's E partial sums into its fp32 running logits in chunk order, so the
// tensor core never carries a sum across more than 64 products. That thread
// then adds the bias and selects the token's top-k from its registers (k+1
// rounds of arg-max: larger value, then lower index), with the gates and the
// k-th/(k+1)-th gap as in select_token.
constexpr int kGTok = 128;    // tokens per CTA
constexpr int kGK = 64;       // reduction indices per chunk
constexpr int kGStages = 6;
constexpr int kGBufs = 4;     // tensor-memory partial buffers
constexpr int kGThreads = 192;  // warps: 0 TMA, 1 MMA, 2-5 tokens

template <int EMAX>
constexpr size_t g_smem_bytes() {
  return 1024 + kGStages * (kGTok * kGK * 2 + EMAX * kGK * 2) + 256;
}

struct __align__(8) GCtrl {
  uint64_t full[kGStages], empty[kGStages], dfull[kGBufs], dempty[kGBufs];
  uint32_t tmem_base;
  int abort;
};

template <int EMAX>
__global__ void __launch_bounds__(kGThreads, 1)
    k_route_tcg(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                const float* __restrict__ b, int T, int d, int E, int k,
                int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                float* __restrict__ gap, int* status) {
  constexpr int XB = kGTok * kGK * 2, WB = EMAX * kGK * 2;
  constexpr uint32_t kCols = kGBufs * EMAX;  // 256 or 512 tensor-memory columns
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sx = smem_u32(base), sw = sx + kGStages * XB;
  GCtrl& C = *reinterpret_cast<GCtrl*>(base + kGStages * (XB + WB));
  volatile int* abort = &C.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t deadline = global_timer_ns() + kWaitTimeoutNs;
  const int t0 = blockIdx.x * kGTok;
  const int Ep = (E + 15) & ~15;
  const int chunks = d / kGK;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(smem_u32(&C.full[s]), 1);
      mbar_init(smem_u32(&C.empty[s]), 1);
    }
    for (int s = 0; s < kGBufs; ++s) {
      mbar_init(smem_u32(&C.dfull[s]), 1);
      mbar_init(smem_u32(&C.dempty[s]), 4);
    }
    C.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  } else if (warp == 1) {
    tmem_alloc(smem_u32(&C.tmem_base), kCols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = C.tmem_base;

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer
      const uint32_t bytes = XB + static_cast<uint32_t>(Ep) * kGK * 2;
      int stage = 0;
      uint32_t phase = 0;
      for (int c = 0; c < chunks; ++c) {
        if (!wait_bar(smem_u32(&C.empty[stage]), phase ^ 1u, deadline, abort)) break;
        const uint32_t fb = smem_u32(&C.full[stage]);
        mbar_arrive_expect_tx(fb, bytes);
        tma_load_2d(sx + stage * XB, &map_x, fb, c * kGK, t0);
        tma_load_2d(sw + stage * WB, &map_w, fb, c * kGK, 0);
        if (++stage == kGStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer: one fresh accumulator per chunk
      const uint32_t idesc = idesc_bf16(kGTok, Ep);
      int stage = 0;
      uint32_t phase = 0;
      for (int c = 0; c < chunks; ++c) {
        const int buf = c % kGBufs;
        if (!wait_bar(smem_u32(&C.dempty[buf]), ((c / kGBufs) & 1) ^ 1u, deadline, abort)) break;
        if (!wait_bar(smem_u32(&C.full[stage]), phase, deadline, abort)) break;
        tc_fence_after();
        const uint32_t a0 = sx + stage * XB, b0 = sw + stage * WB;
#pragma unroll
        for (int kk = 0; kk < kGK / 16; ++kk)
          umma_ss(tmem + buf * EMAX, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc,
                  kk != 0 ? 1u : 0u);
        umma_commit(smem_u32(&C.empty[stage]));
        umma_commit(smem_u32(&C.dfull[buf]));
        if (++stage == kGStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {  // ---- tokens: warps 2..5, lane 32*(warp%4) + lane = token t0 + that
    const int q = warp & 3;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * q) << 16);
    float acc[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) acc[e] = 0.f;
    bool ok = true;
    for (int c = 0; c < chunks; ++c) {
      const int buf = c % kGBufs;
      // warp-uniform verdict: tcgen05.ld below is warp-collective
      if (!__all_sync(0xffffffffu, wait_bar(smem_u32(&C.dfull[buf]), (c / kGBufs) & 1,
                                            deadline, abort))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < EMAX / 32; ++cc) {
        if (32 * cc < Ep) {
          uint32_t v[32];
          tmem_ld32(tlane + buf * EMAX + 32 * cc, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[32 * cc + i] += __uint_as_float(v[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&C.dempty[buf]));
    }
    const int t = t0 + 32 * q + lane;
    if (ok && t < T) {
      uint32_t key[EMAX];
#pragma unroll
      for (int e = 0; e < EMAX; ++e)
        key[e] = e < E ? order_key(rankable(acc[e] + (b != nullptr ? b[e] : 0.f), status)) : 0u;
      float sel_val[8];
      int sel_idx[8];
      float kth = 0.f, next = INFINITY;  // l_(k) and l_(k+1)
      const int rounds = min(k + 1, E);
#pragma unroll
      for (int r = 0; r < 9; ++r) {
        if (r < 8) {
          sel_val[r] = -INFINITY;
          sel_idx[r] = 0;
        }
        if (r < rounds) {
          uint32_t best = 0u;
          int bi = 0;
#pragma unroll
          for (int e = 0; e < EMAX; ++e)
            if (key[e] > best) {  // strictly greater: the lower index wins ties
              best = key[e];
              bi = e;
            }
#pragma unroll
          for (int e = 0; e < EMAX; ++e)
            if (e == bi) key[e] = 0u;  // taken
          const float v = key_value(best);
          if (r < 8) {
            sel_val[r] = v;
            sel_idx[r] = bi;
          }
          if (r == k - 1) kth = v;
          if (r == k) next = v;
        }
      }
      if (gap != nullptr) gap[t] = (k < E) ? kth - next : INFINITY;
      float ex[8], den = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < k) {
          ex[j] = expf(sel_val[j] - sel_val[0]);
          den += ex[j];
        }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < k) {
          topk_idx[static_cast<size_t>(t) * k + j] = sel_idx[j];
          topk_w[static_cast<size_t>(t) * k + j] = ex[j] / den;
        }
    }
  }

  __syncthreads();
  if (*abort) {
    if (threadIdx.x == 0) {
      latch_error(status, kErrTimeout);
      const uint64_t s0 = global_timer_ns();  // let copies in flight land
      while (global_timer_ns() - s0 < 1000000ull) {
      }
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

int slices_for(int d) { return (d + kKS - 1) / kKS; }

}  // namespace

size_t route_scratch_bytes(int T, int d, int E) {
  if (E <= 32 || T <= 0) return 0;
  // (bf16 batches of kTiledMinTokens or more need none; the size does not
  // depend on the dtype, so callers may always pass this much)
  const size_t n = static_cast<size_t>(slices_for(d)) * T * E * sizeof(float);
  return (n + 255) & ~static_cast<size_t>(255);
}

cudaError_t launch_route(const void* x, const void* w_r, const float* b_r, int T, int d, int E,
                         int k, int act, int32_t* topk_idx, float* topk_w, float* gap,
                         void* scratch, cudaStream_t st, int* status, int* n_launches) {
  if (T == 0) return cudaSuccess;
  const dim3 block(kWarps * 32);
  const dim3 grid((T + kWarps - 1) / kWarps);
  if (act == DT_BF16 && T >= kTiledMinTokens && E > 32 && E <= 128 && E % 16 == 0) {
    // many tokens, up to 128 experts: one launch on the 5th-generation tensor cores
    int dev = 0;
    cudaGetDevice(&dev);
    static bool attr_set[2][128] = {};  // per kernel and device: more than 48 KiB of smem
    CUtensorMap mx, mw;
    cudaError_t e = encode_tmap_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, T, d, kGK, kGTok,
                                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (e == cudaSuccess)
      e = encode_tmap_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_r, E, d, kGK, E,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    const int which = E <= 64 ? 0 : 1;
    const size_t smem = which == 0 ? g_smem_bytes<64>() : g_smem_bytes<128>();
    if (dev >= 0 && dev < 128 && !attr_set[which][dev]) {
      e = which == 0 ? cudaFuncSetAttribute(k_route_tcg<64>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(smem))
                     : cudaFuncSetAttribute(k_route_tcg<128>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      attr_set[which][dev] = true;
    }
    const unsigned grid_t = static_cast<unsigned>((T + kGTok - 1) / kGTok);
    if (which == 0)
      k_route_tcg<64><<<grid_t, kGThreads, smem, st>>>(mx, mw, b_r, T, d, E, k, topk_idx,
                                                       topk_w, gap, status);
    else
      k_route_tcg<128><<<grid_t, kGThreads, smem, st>>>(mx, mw, b_r, T, d, E, k, topk_idx,
                                                        topk_w, gap, status);
    if (n_launches) *n_launches += 1;
    return cudaGetLastError();
  }
  if (act == DT_BF16 && T >= kTiledMinTokens && E > 32) {
    // many tokens, many experts: one launch, 64 tokens per block, pipelined
    int dev = 0;
    cudaGetDevice(&dev);
    static bool attr_set[2][128] = {};  // per kernel and device: more than 48 KiB of smem
    if (d % 128 == 0 && E <= 128) {
      const size_t smem = big_smem_bytes<128>(E);
      if (dev >= 0 && dev < 128 && !attr_set[0][dev]) {
        const cudaError_t e = cudaFuncSetAttribute(
            k_route_tc_big<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
            static_cast<int>(big_smem_bytes<128>(128)));
        if (e != cudaSuccess) return e;
        attr_set[0][dev] = true;
      }
      k_route_tc_big<128><<<(T + kBigTok - 1) / kBigTok, 256, smem, st>>>(
          static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w_r), b_r, T,
          d, E, k, topk_idx, topk_w, gap, status);
    } else {
      const size_t smem = big_smem_bytes<64>(E);
      if (dev >= 0 && dev < 128 && !attr_set[1][dev]) {
        const cudaError_t e = cudaFuncSetAttribute(
            k_route_tc_big<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
            static_cast<int>(big_smem_bytes<64>(256)));
        if (e != cudaSuccess) return e;
        attr_set[1][dev] = true;
      }
      k_route_tc_big<64><<<(T + kBigTok - 1) / kBigTok, 256, smem, st>>>(
          static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w_r), b_r, T,
          d, E, k, topk_idx, topk_w, gap, status);
    }
    if (n_launches) *n_launches += 1;
    return cudaGetLastError();
  }
  if (act == DT_BF16 && T >= kTiledMinTokens) {
    // many tokens, E <= 32: one launch, 32 tokens per block, logits on the tensor cores
    const int NT = (E + 7) / 8;
    const int ks = NT >= 8 ? 1 : 8 / NT;
    const size_t smem = static_cast<size_t>(ks) * kTok * E * sizeof(float);
    k_route_tc<<<(T + kTok - 1) / kTok, 256, smem, st>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w_r), b_r, T, d,
        E, k, ks, topk_idx, topk_w, gap, status);
    if (n_launches) *n_launches += 1;
    return cudaGetLastError();
  }
  if (E <= 32) {
#define COLI_ROUTE_FUSED(TA, EM)                                                             \
  k_route_fused<TA, EM><<<T, block, 0, st>>>(static_cast<const TA*>(x),                 \
                                               static_cast<const TA*>(w_r), b_r, T, d, E, k, \
                                               topk_idx, topk_w, gap, status)
    if (act == DT_F32) {
      if (E <= 8) COLI_ROUTE_FUSED(float, 8);
      else if (E <= 16) COLI_ROUTE_FUSED(float, 16);
      else COLI_ROUTE_FUSED(float, 32);
    } else {
      if (E <= 8) COLI_ROUTE_FUSED(__nv_bfloat16, 8);
      else if (E <= 16) COLI_ROUTE_FUSED(__nv_bfloat16, 16);
      else COLI_ROUTE_FUSED(__nv_bfloat16, 32);
    }
#undef COLI_ROUTE_FUSED
    if (n_launches) *n_launches += 1;
    return cudaGetLastError();
  }
  float* part = static_cast<float*>(scratch);
  const int S = slices_for(d);
  const dim3 pgrid((T + kTT - 1) / kTT, (E + kTE - 1) / kTE, S);
  if (act == DT_F32) {
    k_route_partial<float><<<pgrid, 128, 0, st>>>(static_cast<const float*>(x),
                                                   static_cast<const float*>(w_r), T, d, E, part);
  } else {
    const dim3 tgrid((T + kTcTok - 1) / kTcTok, (E + kTcExp - 1) / kTcExp, S);
    k_route_partial_tc<<<tgrid, 128, 0, st>>>(static_cast<const __nv_bfloat16*>(x),
                                               static_cast<const __nv_bfloat16*>(w_r), T, d, E,
                                               part);
  }
  const dim3 sblock(kSelWarps * 32), sgrid((T + kSelWarps - 1) / kSelWarps);
  if (E <= 64)
    k_route_select<2><<<sgrid, sblock, 0, st>>>(part, S, b_r, T, E, k, topk_idx, topk_w, gap,
                                                status);
  else if (E <= 128)
    k_route_select<4><<<sgrid, sblock, 0, st>>>(part, S, b_r, T, E, k, topk_idx, topk_w, gap,
                                                status);
  else
    k_route_select<8><<<sgrid, sblock, 0, st>>>(part, S, b_r, T, E, k, topk_idx, topk_w, gap,
                                                status);
  if (n_launches) *n_launches += 2;
  return cudaGetLastError();
}

}  // namespace coli
