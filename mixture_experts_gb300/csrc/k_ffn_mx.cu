// A3, decode path for block-scaled experts: OCP Microscaling (MX) weights,
// E4M3 bytes (MXFP8) or E2M1 nibbles (MXFP4), each 32 consecutive reduction
// indices of a row sharing one E8M0 scale 2^(s - 127). The deep-dive page's
// model-family table lists engines that run native MXFP4 and FP8 weights;
// here they are the expert weights of the decode (weight-streaming) path.
//
// Every E4M3 and E2M1 value is exact in fp16, and the hardware converts two
// codes to an fp16 pair in one instruction (cvt.rn.f16x2.e4m3x2 /
// .e2m1x2), so the weights feed fp16 mma.sync m16n8k16 (swap-AB as in the
// bf16/int4 decode kernels: weight rows are M, the <= 16 token rows N) with
// the activations converted to fp16 once per forward. The two MMAs of one
// 32-index block go into a fresh accumulator that is multiplied by the
// block's scale in fp32 (a power of two: exact) and added to the running
// sum, so w = element * 2^(s - 127) is used exactly.
//
// Layout (made at create): gate/up rows interleaved in blocks of 64 as in the
// other paths; within every 128 reduction indices of a row the bytes are
// reordered so lane q of a quad finds the 8 indices 32b + 8q .. 32b + 8q + 7
// of the four blocks b contiguous (32 bytes for E4M3, 16 for E2M1). Scale
// bytes keep the canonical [rows][K/32] order (four per 128-index step).
// Weights are loaded straight into registers with streaming loads (several
// steps in flight, no shared memory, so L1 keeps the activation rows).
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace coli {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRowsPerPass = 16;  // token rows per weight pass (two 8-token tiles)

template <int FMT>
constexpr int kLaneStep = FMT == 8 ? 32 : 16;  // bytes of one row per lane and 128-index step

COLI_DEV void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                      uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

COLI_DEV void mma_f16_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

COLI_DEV uint32_t word4(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// fp32 -> fp16, round to nearest even; a value beyond the fp16 range is
// saturated and latches a data error (it never becomes inf).
COLI_DEV __half to_f16_checked(float v, int* status) {
  if (fabsf(v) > 65504.f) {
    latch_error(status, kErrDevice);
    v = copysignf(65504.f, v);
  }
  return __float2half_rn(v);
}

// Two E8M0 codes (a 16-bit half of a scale word) -> their fp32 values
// 2^(s - 127), exactly (the hardware conversion handles s = 0 and s = 255).
COLI_DEV void e8m0x2_f32(uint32_t word, int half, float& lo, float& hi) {
  uint32_t b;
  asm("cvt.rn.bf16x2.ue8m0x2 %0, %1;"
      : "=r"(b)
      : "h"(static_cast<unsigned short>(half ? (word >> 16) : (word & 0xffffu))));
  lo = __uint_as_float(b << 16);
  hi = __uint_as_float(b & 0xffff0000u);
}

// One warp: two 16-row weight tiles (rows r, r + 8 of each per lane) x NT
// 8-token tiles. A step is two MX blocks (64 indices) for E4M3, four (128)
// for E2M1: 16 bytes per row and lane, loaded straight into registers with
// streaming loads, U steps in flight. wrow[m][h]: the lane's first byte of
// row (m, h); srow[m][h]: the row's scale words (4 blocks per word);
// xrow[n]: fp16 activations of this lane's token row of tile n, offset by 8q
// (nullptr for padding rows). Blocks run over [blk0, blk1) (multiples of the
// step's block count).
template <int FMT, int NT>
COLI_DEV void mx_mainloop(const uint8_t* const (&wrow)[2][2], const uint32_t* const (&srow)[2][2],
                          const __half* const (&xrow)[NT], int blk0, int blk1,
                          float (&acc)[2][NT][4]) {
  constexpr int BPS = FMT == 8 ? 2 : 4;  // blocks per step
  constexpr int U = NT == 1 ? 2 : 1;     // steps of loads in flight
  const int st0 = blk0 / BPS, st1 = blk1 / BPS;
  // byte offset of step t within a row segment: E4M3 chunk t/2 (128 bytes
  // per 128 indices), half t%2; E2M1 chunk t (64 bytes)
  auto wofs = [](int t) -> size_t {
    return FMT == 8 ? static_cast<size_t>(t >> 1) * 128 + (t & 1) * 16 : static_cast<size_t>(t) * 64;
  };
  auto process = [&](int t, const uint4 (&wv)[2][2]) {
    uint32_t sw[2][2];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int h = 0; h < 2; ++h) sw[m][h] = srow[m][h][FMT == 8 ? (t >> 1) : t];
#pragma unroll
    for (int bb = 0; bb < BPS; bb += 2) {
      // scales of blocks bb, bb+1 of the step (both in one 16-bit half)
      const int half = FMT == 8 ? (t & 1) : (bb >> 1);
      float sc[2][2][2];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h) e8m0x2_f32(sw[m][h], half, sc[m][h][0], sc[m][h][1]);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int b = bb + u;               // block within the step
        const int blk = t * BPS + b;        // block within the row
        uint4 bx[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n)
          bx[n] = xrow[n] ? ldg_keep(xrow[n] + blk * 32) : make_uint4(0u, 0u, 0u, 0u);
        uint32_t f[2][2][4];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if constexpr (FMT == 8) e4m3x8_f16(word4(wv[m][h], 2 * b), word4(wv[m][h], 2 * b + 1), f[m][h]);
            else e2m1x8_f16(word4(wv[m][h], b), f[m][h]);
          }
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            float tt[4];
            mma_f16_z(tt, f[m][0][0], f[m][1][0], f[m][0][1], f[m][1][1], bx[n].x, bx[n].y);
            mma_f16(tt, f[m][0][2], f[m][1][2], f[m][0][3], f[m][1][3], bx[n].z, bx[n].w);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              acc[m][n][c] = fmaf(sc[m][c >> 1][u], tt[c], acc[m][n][c]);
          }
      }
    }
  };
  int t = st0;
  for (; t + U <= st1; t += U) {
    uint4 wv[U][2][2];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h) wv[u][m][h] = ldg_stream(wrow[m][h] + wofs(t + u));
#pragma unroll
    for (int u = 0; u < U; ++u) process(t + u, wv[u]);
  }
  for (; t < st1; ++t) {
    uint4 wv[2][2];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int h = 0; h < 2; ++h) wv[m][h] = ldg_stream(wrow[m][h] + wofs(t));
    process(t, wv);
  }
}

struct MxArgs {
  const uint8_t* w;          // repacked weights (gate/up or down)
  const uint8_t* s;          // E8M0 scales [weight rows][K/32]
  const uint8_t* const* wtab;  // residency tier: expert e's weights at wtab[e], or nullptr
  const uint8_t* const* stab;  // ... and its scales at stab[e]
  const __half* x;           // fp16 activations: [T][K] through row_token, or [rows][K]
  const int32_t* row_token;  // non-null: row r reads x[row_token[r]]
  const int32_t* offsets;    // [E+1]
  int E, K;                  // experts, reduction length
  int rows_per_expert;       // weight rows per expert (2f or d)
  int f, d, splits;
  __half* H;                 // gate/up output [rows][f] (fp16)
  float* y_part;             // down output [splits][rows][d]
  size_t part_stride;
  int* status;
};

template <int FMT>
COLI_DEV size_t mx_row_bytes(int K) {
  return FMT == 8 ? static_cast<size_t>(K) : static_cast<size_t>(K) / 2;
}

template <int FMT, int NT>
COLI_DEV void mx_gateup_chunk(const MxArgs& A, const int32_t* tok, int e, int n0, int row0,
                              int nrows) {
  const int lane = threadIdx.x & 31, r = lane >> 2, q = lane & 3;
  const size_t rb = mx_row_bytes<FMT>(A.K);
  const int sw = A.K / 128;  // scale words per row
  const size_t gin = 128 * (n0 / 64) + (n0 % 64);  // row within the expert
  const size_t e0 = static_cast<size_t>(e) * A.rows_per_expert;
  const uint8_t* wbase = A.wtab ? A.wtab[e] : A.w + e0 * rb;
  const uint32_t* sbase = reinterpret_cast<const uint32_t*>(A.stab ? A.stab[e] : A.s + e0 * sw * 4);
  const uint8_t* wrow[2][2];
  const uint32_t* srow[2][2];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const size_t row = gin + 64 * m + r + 8 * h;
      wrow[m][h] = wbase + row * rb + q * kLaneStep<FMT>;
      srow[m][h] = sbase + row * sw;
    }
  const __half* xrow[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int j = 8 * n + r;
    const size_t src = static_cast<size_t>(tok ? tok[row0 + j] : row0 + j);
    xrow[n] = j < nrows ? A.x + src * A.K + q * 8 : nullptr;
  }
  float acc[2][NT][4];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[m][n][c] = 0.f;
  mx_mainloop<FMT, NT>(wrow, srow, xrow, 0, A.K / 32, acc);
  // acc[0] = gate, acc[1] = up: features r, r+8; tokens 2q, 2q+1 of each tile
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = 8 * n + 2 * q + (c & 1);
      if (j >= nrows) continue;
      const int feat = n0 + r + ((c & 2) ? 8 : 0);
      const float a = acc[0][n][c], u = acc[1][n][c];
      A.H[static_cast<size_t>(row0 + j) * A.f + feat] =
          to_f16_checked(a / (1.f + expf(-a)) * u, A.status);
    }
}

template <int FMT, int NT>
COLI_DEV void mx_down_chunk(const MxArgs& A, int e, int o0, int split, int row0, int nrows) {
  const int lane = threadIdx.x & 31, r = lane >> 2, q = lane & 3;
  const size_t rb = mx_row_bytes<FMT>(A.K);
  const int sw = A.K / 128;
  const size_t e0 = static_cast<size_t>(e) * A.rows_per_expert;
  const uint8_t* wbase = A.wtab ? A.wtab[e] : A.w + e0 * rb;
  const uint32_t* sbase = reinterpret_cast<const uint32_t*>(A.stab ? A.stab[e] : A.s + e0 * sw * 4);
  const uint8_t* wrow[2][2];
  const uint32_t* srow[2][2];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const size_t row = static_cast<size_t>(o0) + 16 * m + r + 8 * h;  // within the expert
      wrow[m][h] = wbase + row * rb + q * kLaneStep<FMT>;
      srow[m][h] = sbase + row * sw;
    }
  const __half* xrow[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int j = 8 * n + r;
    xrow[n] = j < nrows ? A.x + static_cast<size_t>(row0 + j) * A.K + q * 8 : nullptr;
  }
  float acc[2][NT][4];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[m][n][c] = 0.f;
  // slices split the row's 128-index chunks (so any step size divides them)
  const int chunks = A.K / 128;
  const int c0 = static_cast<int>(static_cast<long>(chunks) * split / A.splits);
  const int c1 = static_cast<int>(static_cast<long>(chunks) * (split + 1) / A.splits);
  mx_mainloop<FMT, NT>(wrow, srow, xrow, 4 * c0, 4 * c1, acc);
  float* out = A.y_part + static_cast<size_t>(split) * A.part_stride;
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = 8 * n + 2 * q + (c & 1);
        if (j >= nrows) continue;
        const int o = o0 + 16 * m + r + ((c & 2) ? 8 : 0);
        out[static_cast<size_t>(row0 + j) * A.d + o] = acc[m][n][c];
      }
}

// Persistent warps over items (expert, 16 features); consecutive items share
// the expert so a block's warps re-read the same activation rows from L1.
template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) k_mx_gateup(const MxArgs A) {
  const int W = gridDim.x * kWarps;
  const int per_e = A.f / 16;
  const int items = A.E * per_e;
  for (int it = blockIdx.x * kWarps + (threadIdx.x >> 5); it < items; it += W) {
    const int e = it / per_e, n0 = (it % per_e) * 16;
    const int r0 = A.offsets[e], r1 = A.offsets[e + 1];
    for (int row0 = r0; row0 < r1; row0 += kMaxRowsPerPass) {
      const int nrows = min(kMaxRowsPerPass, r1 - row0);
      if (nrows <= 8) mx_gateup_chunk<FMT, 1>(A, A.row_token, e, n0, row0, nrows);
      else mx_gateup_chunk<FMT, 2>(A, A.row_token, e, n0, row0, nrows);
    }
  }
}

// Items (slice, expert, 32 outputs); the slice is outermost so neighbouring
// warps read the same part of H.
template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) k_mx_down(const MxArgs A) {
  const int W = gridDim.x * kWarps;
  const int per_e = A.d / 32;
  const int per_split = A.E * per_e;
  const int items = per_split * A.splits;
  for (int it = blockIdx.x * kWarps + (threadIdx.x >> 5); it < items; it += W) {
    const int split = it / per_split, rem = it % per_split;
    const int e = rem / per_e, o0 = (rem % per_e) * 32;
    const int r0 = A.offsets[e], r1 = A.offsets[e + 1];
    for (int row0 = r0; row0 < r1; row0 += kMaxRowsPerPass) {
      const int nrows = min(kMaxRowsPerPass, r1 - row0);
      if (nrows <= 8) mx_down_chunk<FMT, 1>(A, e, o0, split, row0, nrows);
      else mx_down_chunk<FMT, 2>(A, e, o0, split, row0, nrows);
    }
  }
}

// bf16 -> fp16 rows (activations of the MX path), saturating and latching a
// data error beyond the fp16 range.
__global__ void __launch_bounds__(256)
    k_bf16_to_f16(const uint4* __restrict__ in, size_t n8, uint4* __restrict__ out, int* status) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 v = in[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half lo = to_f16_checked(bf16_lo(w[k]), status);
      const __half hi = to_f16_checked(bf16_hi(w[k]), status);
      o[k] = static_cast<uint32_t>(__half_as_ushort(lo)) |
             (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
    }
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Create-time reorder of one MX weight row set: within every 128 reduction
// indices, lane q's 8 indices of the four 32-index blocks become contiguous.
// E4M3: unit = 8 bytes, source unit (b, q) -> destination unit (q, b);
// E2M1: unit = 4 bytes, the same 4 x 4 transpose. Rows follow the gate/up
// interleave (gate row 64*(R/128) + R%128 for R%128 < 64, else the up row).
__global__ void __launch_bounds__(256)
    k_repack_mx(const uint8_t* __restrict__ src_a, const uint8_t* __restrict__ src_b,
                int src_rows_per_e, int dst_rows_per_e, int row_bytes, int unit, int E,
                bool interleave, uint8_t* __restrict__ dst) {
  const long total = static_cast<long>(E) * dst_rows_per_e;
  const int chunk = 16 * unit;  // bytes of 128 indices
  for (long R = blockIdx.x; R < total; R += gridDim.x) {
    const int e = static_cast<int>(R / dst_rows_per_e), rr = static_cast<int>(R % dst_rows_per_e);
    const uint8_t* src;
    if (interleave) {
      const int blk = rr / 128, off = rr % 128;
      const int srow = 64 * blk + (off < 64 ? off : off - 64);
      src = (off < 64 ? src_a : src_b) + (static_cast<size_t>(e) * src_rows_per_e + srow) * row_bytes;
    } else {
      src = src_a + (static_cast<size_t>(e) * src_rows_per_e + rr) * row_bytes;
    }
    uint8_t* out = dst + static_cast<size_t>(R) * row_bytes;
    for (int i = threadIdx.x; i < row_bytes; i += blockDim.x) {
      const int c = i / chunk, w = i % chunk;  // destination byte w of chunk c
      const int du = w / unit, j = w % unit;   // destination unit = (q, b)
      const int q = du / 4, b = du % 4;
      out[i] = src[c * chunk + (4 * b + q) * unit + j];
    }
  }
}

// Scale bytes follow the same row order (no reorder within a row).
__global__ void __launch_bounds__(256)
    k_repack_rows_u8(const uint8_t* __restrict__ src_a, const uint8_t* __restrict__ src_b,
                     int src_rows_per_e, int dst_rows_per_e, int row_bytes, int E,
                     bool interleave, uint8_t* __restrict__ dst) {
  const long total = static_cast<long>(E) * dst_rows_per_e * row_bytes;
  for (long i = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const long R = i / row_bytes;
    const int c = static_cast<int>(i % row_bytes);
    const int e = static_cast<int>(R / dst_rows_per_e), rr = static_cast<int>(R % dst_rows_per_e);
    const uint8_t* src = src_a;
    int srow = rr;
    if (interleave) {
      const int blk = rr / 128, off = rr % 128;
      srow = 64 * blk + (off < 64 ? off : off - 64);
      src = off < 64 ? src_a : src_b;
    }
    dst[i] = src[(static_cast<size_t>(e) * src_rows_per_e + srow) * row_bytes + c];
  }
}

// Flags weights outside the prefill converters' fast conversion: E4M3 NaN
// codes (any byte whose low seven bits are all ones) and scale bytes above
// 142 (scales beyond 2^15, NaN included).
__global__ void __launch_bounds__(256)
    k_mx_scan(const uint4* __restrict__ w, size_t w_vec, const uint4* __restrict__ s,
              size_t s_vec, int* flag) {
  bool hit = false;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < w_vec;
       i += stride) {
    const uint4 v = w[i];
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) hit |= (((x[j] & 0x7f7f7f7fu) + 0x01010101u) & 0x80808080u) != 0u;
  }
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < s_vec;
       i += stride) {
    const uint4 v = s[i];
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) hit |= __vcmpgtu4(x[j], 0x8e8e8e8eu) != 0u;
  }
  if (__any_sync(0xffffffffu, hit) && (threadIdx.x & 31) == 0) *flag = 1;
}

}  // namespace

int mx_blocks_per_sm(int wdt) {
  int b = 0;
  const cudaError_t e =
      wdt == DT_MXFP8
          ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_mx_gateup<8>, kThreads, 0)
          : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_mx_gateup<4>, kThreads, 0);
  if (e != cudaSuccess) b = 1;
  return b < 1 ? 1 : b;
}

cudaError_t launch_to_f16(const void* x_bf16, size_t n, void* x_f16, cudaStream_t st,
                          int* status) {
  const size_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  size_t grid = (n8 + 255) / 256;
  if (grid > 4096) grid = 4096;
  k_bf16_to_f16<<<static_cast<unsigned>(grid), 256, 0, st>>>(static_cast<const uint4*>(x_bf16),
                                                             n8, static_cast<uint4*>(x_f16),
                                                             status);
  return cudaGetLastError();
}

cudaError_t launch_mx_gateup(const FfnWeights& w, const void* x16, const int32_t* row_token,
                             const int32_t* offsets, int E, int d, int f, void* H16, int grid,
                             cudaStream_t st, int* status) {
  MxArgs A{};
  A.w = static_cast<const uint8_t*>(w.w_gu);
  A.s = static_cast<const uint8_t*>(w.s_gu_u8);
  A.wtab = w.tab_gu;
  A.stab = w.tab_sgu;
  A.x = static_cast<const __half*>(x16);
  A.row_token = row_token;
  A.offsets = offsets;
  A.E = E;
  A.K = d;
  A.rows_per_expert = 2 * f;
  A.f = f;
  A.d = d;
  A.splits = 1;
  A.H = static_cast<__half*>(H16);
  A.status = status;
  if (w.wdt == DT_MXFP8) k_mx_gateup<8><<<grid, kThreads, 0, st>>>(A);
  else k_mx_gateup<4><<<grid, kThreads, 0, st>>>(A);
  return cudaGetLastError();
}

cudaError_t launch_mx_down(const FfnWeights& w, const void* H16, const int32_t* offsets, int E,
                           int d, int f, int splits, float* y_part, size_t part_stride, int grid,
                           cudaStream_t st, int* status) {
  MxArgs A{};
  A.w = static_cast<const uint8_t*>(w.w_dn);
  A.s = static_cast<const uint8_t*>(w.s_dn_u8);
  A.wtab = w.tab_dn;
  A.stab = w.tab_sdn;
  A.x = static_cast<const __half*>(H16);
  A.offsets = offsets;
  A.E = E;
  A.K = f;
  A.rows_per_expert = d;
  A.f = f;
  A.d = d;
  A.splits = splits;
  A.y_part = y_part;
  A.part_stride = part_stride;
  A.status = status;
  if (w.wdt == DT_MXFP8) k_mx_down<8><<<grid, kThreads, 0, st>>>(A);
  else k_mx_down<4><<<grid, kThreads, 0, st>>>(A);
  return cudaGetLastError();
}

cudaError_t launch_repack_mx(const void* src_gate, const void* src_up, const void* src_down,
                             const void* sg, const void* su, const void* sd, int wdt, int E,
                             int d, int f, void* dst_gu, void* dst_sgu, void* dst_dn,
                             void* dst_sdn, cudaStream_t st) {
  const int unit = wdt == DT_MXFP8 ? 8 : 4;
  const int gu_bytes = wdt == DT_MXFP8 ? d : d / 2;
  const int dn_bytes = wdt == DT_MXFP8 ? f : f / 2;
  const unsigned grid = 4096;
  k_repack_mx<<<grid, 256, 0, st>>>(static_cast<const uint8_t*>(src_gate),
                                    static_cast<const uint8_t*>(src_up), f, 2 * f, gu_bytes, unit,
                                    E, true, static_cast<uint8_t*>(dst_gu));
  k_repack_mx<<<grid, 256, 0, st>>>(static_cast<const uint8_t*>(src_down), nullptr, d, d,
                                    dn_bytes, unit, E, false, static_cast<uint8_t*>(dst_dn));
  k_repack_rows_u8<<<grid, 256, 0, st>>>(static_cast<const uint8_t*>(sg),
                                         static_cast<const uint8_t*>(su), f, 2 * f, d / 32, E,
                                         true, static_cast<uint8_t*>(dst_sgu));
  k_repack_rows_u8<<<grid, 256, 0, st>>>(static_cast<const uint8_t*>(sd), nullptr, d, d, f / 32,
                                         E, false, static_cast<uint8_t*>(dst_sdn));
  return cudaGetLastError();
}

cudaError_t launch_mx_scan(const void* w, size_t w_bytes, const void* s, size_t s_bytes, int wdt,
                           int* flag, cudaStream_t st) {
  // E2M1 has no NaN code: only the scales are scanned
  const size_t wv = wdt == DT_MXFP8 ? w_bytes / 16 : 0, sv = s_bytes / 16;
  k_mx_scan<<<1024, 256, 0, st>>>(static_cast<const uint4*>(w), wv,
                                  static_cast<const uint4*>(s), sv, flag);
  return cudaGetLastError();
}

}  // namespace coli
