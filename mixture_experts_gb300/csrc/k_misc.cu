// A4 combine, the fp32 expert FFN, split-slice reduction, create-time weight
// repacking and the bounded-wait self-test.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace coli {
namespace {

// ---- A4: gate-weighted merge back to token order -----------------------------
// y[t] = sum_{j ascending} g[t][j] * (sum_{s ascending} part[s][row]), row =
// assign_row[t*k+j]: the overview page's weighted merge (trdm.cn section 2.1)
// and the copy back in token order of the mhpn.cn page (section 2.3). A
// gather, so no atomics and a fixed summation order. A row outside
// [0, n_rows) (an assignment the dispatch skipped, or bad caller data) adds
// nothing and latches COLI_EDEVICE; it is never read.
// A block takes one token and a 1024-column slab, a thread one float4 column:
// the k row indices and gates are loaded first, then the k rows of every
// slice (all loads of a slice in flight together), each row summed over the
// slices in order, then merged with j ascending.
template <bool BF16_OUT>
__global__ void __launch_bounds__(256)
    k_combine(const float* __restrict__ part, int splits, size_t part_stride,
              const int32_t* __restrict__ assign_row, const float* __restrict__ topk_w, int T,
              int k, int d, int n_rows, void* __restrict__ y, int* status) {
  const int t = blockIdx.x;
  const int d4 = d / 4;
  const int c = blockIdx.y * blockDim.x + threadIdx.x;
  if (c >= d4) return;
  constexpr int KMAX = 8;
  int row[KMAX];
  float g[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    row[j] = -1;
    g[j] = 0.f;
    if (j < k) {
      const size_t a = static_cast<size_t>(t) * k + j;
      const int r = assign_row[a];
      g[j] = topk_w[a];
      if (r >= 0 && r < n_rows) row[j] = r;
      else if (c == 0) latch_error(status, kErrDevice);
    }
  }
  float4 v[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j)
    v[j] = row[j] >= 0 ? reinterpret_cast<const float4*>(part)[static_cast<size_t>(row[j]) * d4 + c]
                       : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 1; s < splits; ++s) {
    const float4* ps = reinterpret_cast<const float4*>(part + s * part_stride);
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (row[j] >= 0) {
        const float4 w = ps[static_cast<size_t>(row[j]) * d4 + c];
        v[j].x += w.x;
        v[j].y += w.y;
        v[j].z += w.z;
        v[j].w += w.w;
      }
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < KMAX; ++j)
    if (row[j] >= 0) {
      acc.x = fmaf(g[j], v[j].x, acc.x);
      acc.y = fmaf(g[j], v[j].y, acc.y);
      acc.z = fmaf(g[j], v[j].z, acc.z);
      acc.w = fmaf(g[j], v[j].w, acc.w);
    }
  if (BF16_OUT) {
    uint2 o;
    o.x = pack_bf16x2(acc.x, acc.y);
    o.y = pack_bf16x2(acc.z, acc.w);
    reinterpret_cast<uint2*>(y)[static_cast<size_t>(t) * d4 + c] = o;
  } else {
    reinterpret_cast<float4*>(y)[static_cast<size_t>(t) * d4 + c] = acc;
  }
}

// The same merge from bf16 rows: a thread takes 8 consecutive columns of one
// token (16 bytes of each of its k rows, all loads issued before the sums),
// so a 256-thread block covers 2048 columns. Sums in fp32, j ascending.
template <bool BF16_OUT>
__global__ void __launch_bounds__(256)
    k_combine_bf16(const uint4* __restrict__ y_perm, const int32_t* __restrict__ assign_row,
                   const float* __restrict__ topk_w, int T, int k, int d, int n_rows,
                   void* __restrict__ y, int* status) {
  const int d8 = d / 8;
  const long gid = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x;
  if (gid >= static_cast<long>(T) * d8) return;
  const int t = static_cast<int>(gid / d8), c = static_cast<int>(gid % d8);
  constexpr int KMAX = 8;
  uint4 v[KMAX];
  float g[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    v[j] = make_uint4(0u, 0u, 0u, 0u);
    g[j] = 0.f;
    if (j < k) {
      const size_t a = static_cast<size_t>(t) * k + j;
      const int row = assign_row[a];
      if (row >= 0 && row < n_rows) {
        g[j] = topk_w[a];
        v[j] = y_perm[static_cast<size_t>(row) * d8 + c];
      } else {
        latch_error(status, kErrDevice);
      }
    }
  }
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    if (j < k) {
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(g[j], bf16_lo(w[i]), acc[2 * i]);
        acc[2 * i + 1] = fmaf(g[j], bf16_hi(w[i]), acc[2 * i + 1]);
      }
    }
  }
  if (BF16_OUT) {
    reinterpret_cast<uint4*>(y)[gid] =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                   pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  } else {
    float4* dst = reinterpret_cast<float4*>(y) + 2 * gid;
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

__global__ void __launch_bounds__(256)
    k_reduce_splits(const float* __restrict__ part, int splits, size_t part_stride, size_t n4,
                    float* __restrict__ out) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float4 v = reinterpret_cast<const float4*>(part)[i];
    for (int s = 1; s < splits; ++s) {
      const float4 w = reinterpret_cast<const float4*>(part + s * part_stride)[i];
      v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
    }
    reinterpret_cast<float4*>(out)[i] = v;
  }
}

// ---- A3 in fp32 (CUDA cores; tensor cores would round to tf32) ---------------
COLI_DEV int expert_of_row(const int32_t* __restrict__ offsets, int E, int r) {
  int lo = 0, hi = E;  // offsets[lo] <= r < offsets[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (offsets[mid] <= r) lo = mid;
    else hi = mid;
  }
  return lo;
}

COLI_DEV float dot4(const float4 a, const float4 b, float acc) {
  acc = fmaf(a.x, b.x, acc);
  acc = fmaf(a.y, b.y, acc);
  acc = fmaf(a.z, b.z, acc);
  return fmaf(a.w, b.w, acc);
}

// One warp per (row, 8 features): lanes split the reduction index.
__global__ void __launch_bounds__(256)
    k_f32_gateup(const float* __restrict__ w_gu, const float* __restrict__ x,
                 const int32_t* __restrict__ offsets, int n_rows, int E, int d, int f,
                 float* __restrict__ H) {
  const int lane = threadIdx.x & 31;
  const long wid = blockIdx.x * 8L + (threadIdx.x >> 5);
  const int per_row = f / 8;
  if (wid >= static_cast<long>(n_rows) * per_row) return;
  const int r = static_cast<int>(wid / per_row), n0 = static_cast<int>(wid % per_row) * 8;
  const int e = expert_of_row(offsets, E, r);
  const float* xr = x + static_cast<size_t>(r) * d;
  const size_t gb = static_cast<size_t>(e) * 2 * f + 128 * (n0 / 64) + (n0 % 64);
  float g[8] = {}, u[8] = {};
  for (int i = lane * 4; i < d; i += 128) {
    const float4 xv = *reinterpret_cast<const float4*>(xr + i);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      g[j] = dot4(xv, *reinterpret_cast<const float4*>(w_gu + (gb + j) * d + i), g[j]);
      u[j] = dot4(xv, *reinterpret_cast<const float4*>(w_gu + (gb + 64 + j) * d + i), u[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      g[j] += __shfl_xor_sync(0xffffffffu, g[j], off);
      u[j] += __shfl_xor_sync(0xffffffffu, u[j], off);
    }
  if (lane < 8) {
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j == lane) {
        a = g[j];
        b = u[j];
      }
    H[static_cast<size_t>(r) * f + n0 + lane] = a / (1.f + expf(-a)) * b;
  }
}

__global__ void __launch_bounds__(256)
    k_f32_down(const float* __restrict__ w_dn, const float* __restrict__ H,
               const int32_t* __restrict__ offsets, int n_rows, int E, int d, int f,
               float* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const long wid = blockIdx.x * 8L + (threadIdx.x >> 5);
  const int per_row = d / 8;
  if (wid >= static_cast<long>(n_rows) * per_row) return;
  const int r = static_cast<int>(wid / per_row), o0 = static_cast<int>(wid % per_row) * 8;
  const int e = expert_of_row(offsets, E, r);
  const float* hr = H + static_cast<size_t>(r) * f;
  const size_t ob = static_cast<size_t>(e) * d + o0;
  float acc[8] = {};
  for (int i = lane * 4; i < f; i += 128) {
    const float4 hv = *reinterpret_cast<const float4*>(hr + i);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      acc[j] = dot4(hv, *reinterpret_cast<const float4*>(w_dn + (ob + j) * f + i), acc[j]);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], off);
  if (lane < 8) {
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j == lane) a = acc[j];
    y[static_cast<size_t>(r) * d + o0 + lane] = a;
  }
}

// ---- weight repacking (create time) -------------------------------------------
// Canonical int4 word: nibble p holds index p (p = 0..7, low nibble first).
// Kernel order: even indices 0,2,4,6 in nibbles 0..3, odd 1,3,5,7 in 4..7.
COLI_DEV uint32_t reorder_nibbles(uint32_t w) {
  uint32_t r = 0;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const uint32_t nib = (w >> (4 * p)) & 0xFu;
    const int dst = (p & 1) ? 4 + (p >> 1) : (p >> 1);
    r |= nib << (4 * dst);
  }
  return r;
}

// Copies rows (as 32-bit words) into the kernel layout. Gate/up mode: dst row
// R of expert e holds gate row 64*(R/128) + R%128 when R%128 < 64, else the
// up row 64*(R/128) + R%128 - 64. Down mode: identity.
__global__ void __launch_bounds__(256)
    k_repack(const uint32_t* __restrict__ src_a, const uint32_t* __restrict__ src_b,
             int src_rows_per_e, int dst_rows_per_e, int words_per_row, int E, bool interleave,
             bool nibbles, uint32_t* __restrict__ dst) {
  const long total = static_cast<long>(E) * dst_rows_per_e;
  for (long R = blockIdx.x; R < total; R += gridDim.x) {
    const int e = static_cast<int>(R / dst_rows_per_e), rr = static_cast<int>(R % dst_rows_per_e);
    const uint32_t* src;
    if (interleave) {
      const int blk = rr / 128, off = rr % 128;
      const int srow = 64 * blk + (off < 64 ? off : off - 64);
      src = (off < 64 ? src_a : src_b) +
            (static_cast<size_t>(e) * src_rows_per_e + srow) * words_per_row;
    } else {
      src = src_a + (static_cast<size_t>(e) * src_rows_per_e + rr) * words_per_row;
    }
    uint32_t* out = dst + static_cast<size_t>(R) * words_per_row;
    for (int i = threadIdx.x; i < words_per_row; i += blockDim.x)
      out[i] = nibbles ? reorder_nibbles(src[i]) : src[i];
  }
}

// Scale rows (bf16, [rows][groups]) follow the same row map; copied as u16.
__global__ void __launch_bounds__(256)
    k_repack_scales(const uint16_t* __restrict__ src_a, const uint16_t* __restrict__ src_b,
                    int src_rows_per_e, int dst_rows_per_e, int groups, int E, bool interleave,
                    uint16_t* __restrict__ dst) {
  const long total = static_cast<long>(E) * dst_rows_per_e * groups;
  for (long i = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const long R = i / groups;
    const int g = static_cast<int>(i % groups);
    const int e = static_cast<int>(R / dst_rows_per_e), rr = static_cast<int>(R % dst_rows_per_e);
    const uint16_t* src;
    int srow = rr;
    if (interleave) {
      const int blk = rr / 128, off = rr % 128;
      srow = 64 * blk + (off < 64 ? off : off - 64);
      src = off < 64 ? src_a : src_b;
    } else {
      src = src_a;
    }
    dst[i] = src[(static_cast<size_t>(e) * src_rows_per_e + srow) * groups + g];
  }
}

// ---- bounded-wait self-test --------------------------------------------------------
__global__ void k_selftest_wait(int spin_limit, int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing arrives: phase 0 never completes
    bool done = false;
    for (int i = 0; i < spin_limit && !done; ++i) done = mbar_try_wait(smem_u32(&bar), 0);
    if (!done) latch_error(status, kErrTimeout);
  }
}

}  // namespace

cudaError_t launch_combine(const float* y_part, int splits, size_t part_stride,
                           const int32_t* assign_row, const float* topk_w, int T, int k, int d,
                           int out_dt, void* y, cudaStream_t st, int* status) {
  if (T == 0) return cudaSuccess;
  const int d4 = d / 4;
  const int threads = d4 >= 256 ? 256 : ((d4 + 31) / 32) * 32;
  const dim3 grid(T, (d4 + threads - 1) / threads);
  const int n_rows = T * k;  // assign_row maps the T*k assignments onto rows [0, T*k)
  if (out_dt == DT_BF16)
    k_combine<true><<<grid, threads, 0, st>>>(y_part, splits, part_stride, assign_row, topk_w,
                                              T, k, d, n_rows, y, status);
  else
    k_combine<false><<<grid, threads, 0, st>>>(y_part, splits, part_stride, assign_row, topk_w,
                                               T, k, d, n_rows, y, status);
  return cudaGetLastError();
}

cudaError_t launch_combine_bf16(const __nv_bfloat16* y_perm, const int32_t* assign_row,
                                const float* topk_w, int T, int k, int d, int out_dt, void* y,
                                cudaStream_t st, int* status) {
  if (T == 0) return cudaSuccess;
  const long n = static_cast<long>(T) * (d / 8);
  const unsigned grid = static_cast<unsigned>((n + 255) / 256);
  const int n_rows = T * k;
  if (out_dt == DT_BF16)
    k_combine_bf16<true><<<grid, 256, 0, st>>>(reinterpret_cast<const uint4*>(y_perm),
                                               assign_row, topk_w, T, k, d, n_rows, y, status);
  else
    k_combine_bf16<false><<<grid, 256, 0, st>>>(reinterpret_cast<const uint4*>(y_perm),
                                                assign_row, topk_w, T, k, d, n_rows, y, status);
  return cudaGetLastError();
}

cudaError_t launch_reduce_splits(const float* y_part, int splits, size_t part_stride, int n_rows,
                                 int d, float* y_perm, cudaStream_t st) {
  const size_t n4 = static_cast<size_t>(n_rows) * d / 4;
  if (n4 == 0) return cudaSuccess;
  size_t grid = (n4 + 255) / 256;
  if (grid > 8192) grid = 8192;
  k_reduce_splits<<<static_cast<unsigned>(grid), 256, 0, st>>>(y_part, splits, part_stride, n4,
                                                                 y_perm);
  return cudaGetLastError();
}

cudaError_t launch_f32_ffn(const float* w_gu, const float* w_dn, const float* x_perm,
                           const int32_t* offsets, int n_rows, int E, int d, int f, float* H,
                           float* y_perm, cudaStream_t st, int* n_launches) {
  if (n_rows == 0) return cudaSuccess;
  const long w1 = static_cast<long>(n_rows) * (f / 8);
  k_f32_gateup<<<static_cast<unsigned>((w1 + 7) / 8), 256, 0, st>>>(w_gu, x_perm, offsets,
                                                                      n_rows, E, d, f, H);
  const long w2 = static_cast<long>(n_rows) * (d / 8);
  k_f32_down<<<static_cast<unsigned>((w2 + 7) / 8), 256, 0, st>>>(w_dn, H, offsets, n_rows, E,
                                                                    d, f, y_perm);
  if (n_launches) *n_launches += 2;
  return cudaGetLastError();
}

cudaError_t launch_repack(const void* src_gate, const void* src_up, const void* src_down,
                          const void* sg, const void* su, const void* sd, int wdt, int E, int d,
                          int f, void* dst_gu, void* dst_sgu, void* dst_dn, void* dst_sdn,
                          cudaStream_t st) {
  const bool i4 = wdt == DT_I4G128;
  const int esize4 = wdt == DT_F32 ? 4 : 2;  // bytes per element x 2 for int4 handled below
  const int gu_words = i4 ? d / 8 : d * esize4 / 4;
  const int dn_words = i4 ? f / 8 : f * esize4 / 4;
  const unsigned grid = 4096;
  k_repack<<<grid, 256, 0, st>>>(static_cast<const uint32_t*>(src_gate),
                                 static_cast<const uint32_t*>(src_up), f, 2 * f, gu_words, E, true,
                                 i4, static_cast<uint32_t*>(dst_gu));
  k_repack<<<grid, 256, 0, st>>>(static_cast<const uint32_t*>(src_down), nullptr, d, d, dn_words,
                                 E, false, i4, static_cast<uint32_t*>(dst_dn));
  if (i4) {
    k_repack_scales<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(sg),
                                          static_cast<const uint16_t*>(su), f, 2 * f, d / 128, E,
                                          true, static_cast<uint16_t*>(dst_sgu));
    k_repack_scales<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(sd), nullptr, d, d,
                                          f / 128, E, false, static_cast<uint16_t*>(dst_sdn));
  }
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(int spin_limit, int* status, cudaStream_t st) {
  k_selftest_wait<<<1, 32, 0, st>>>(spin_limit, status);
  return cudaGetLastError();
}

}  // namespace coli
