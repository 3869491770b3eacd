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

namespace coli {
namespace {

constexpr int kWarps = 8;

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

template <int PER_LANE>
__global__ void __launch_bounds__(kWarps * 32)
    k_route_select(const float* __restrict__ part, int slices, const float* __restrict__ b,
                   int T, int E, int k, int32_t* __restrict__ topk_idx,
                   float* __restrict__ topk_w, float* __restrict__ gap, int* status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  float l[PER_LANE];
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) {
    const int e = lane + 32 * i;
    float v = -INFINITY;
    if (e < E) {
      v = 0.f;
      for (int s = 0; s < slices; ++s) v += part[(static_cast<size_t>(s) * T + t) * E + e];
      if (b != nullptr) v += b[e];
      v = rankable(v, status);
    }
    l[i] = v;
  }
  unsigned taken = 0;  // bit i: slot i of this lane already selected
  float best0 = 0.f, prev = 0.f, den = 0.f;
  float sel_val[8];
  int sel_idx[8];
  const int rounds = min(k + 1, E);
  for (int r = 0; r < rounds; ++r) {
    float bv = -INFINITY;
    int bi = 1 << 30;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !(taken & (1u << i)) && beats(l[i], e, bv, bi)) {
        bv = l[i];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (beats(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (r < k) {
      sel_val[r] = bv;
      sel_idx[r] = bi;
    }
    if (r == 0) best0 = bv;
    if (r == k - 1) prev = bv;
    if (r == k && gap != nullptr && lane == 0) gap[t] = prev - bv;
  }
  if (k == E && gap != nullptr && lane == 0) gap[t] = INFINITY;
  // gates: exp(l_j - l_max) / sum_j' exp(l_j' - l_max), j ascending
  for (int j = 0; j < k; ++j) den += expf(sel_val[j] - best0);
  if (lane < k) {
    float v = 0.f;
    int id = 0;
    for (int j = 0; j < k; ++j)
      if (j == lane) {
        v = sel_val[j];
        id = sel_idx[j];
      }
    topk_idx[static_cast<size_t>(t) * k + lane] = id;
    topk_w[static_cast<size_t>(t) * k + lane] = expf(v - best0) / den;
  }
}

int slices_for(int d) { return (d + kKS - 1) / kKS; }

}  // namespace

size_t route_scratch_bytes(int T, int d, int E) {
  if (E <= 32 || T <= 0) return 0;
  const size_t n = static_cast<size_t>(slices_for(d)) * T * E * sizeof(float);
  return (n + 255) & ~static_cast<size_t>(255);
}

cudaError_t launch_route(const void* x, const void* w_r, const float* b_r, int T, int d, int E,
                         int k, int act, int32_t* topk_idx, float* topk_w, float* gap,
                         void* scratch, cudaStream_t st, int* status, int* n_launches) {
  if (T == 0) return cudaSuccess;
  const dim3 block(kWarps * 32);
  const dim3 grid((T + kWarps - 1) / kWarps);
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
  if (E <= 64)
    k_route_select<2><<<grid, block, 0, st>>>(part, S, b_r, T, E, k, topk_idx, topk_w, gap,
                                              status);
  else if (E <= 128)
    k_route_select<4><<<grid, block, 0, st>>>(part, S, b_r, T, E, k, topk_idx, topk_w, gap,
                                              status);
  else
    k_route_select<8><<<grid, block, 0, st>>>(part, S, b_r, T, E, k, topk_idx, topk_w, gap,
                                              status);
  if (n_launches) *n_launches += 2;
  return cudaGetLastError();
}

}  // namespace coli
