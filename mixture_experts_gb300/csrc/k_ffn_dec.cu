// A3, decode path: per-expert SwiGLU FFN for groups of a few rows.
//
// With a handful of tokens per expert the FFN is bound by streaming each
// active expert's weights once (the "sparse GEMM" of the overview page,
// trdm.cn section 3.3, measured there as a fraction of memory bandwidth;
// batch-union — each expert read once however many tokens chose it — from
// the wth2jhl.online deep dive, section 4.3). Experts with no rows are never
// read (wzjinhao.cn section 2.3).
//
// Design (swap-AB): the weight rows are the M side of a warp-level
// m16n8k16 bf16 tensor-core MMA and the (<= 32) token rows of the expert are
// the N side, so every weight byte is loaded exactly once, straight from HBM
// into registers with 16-byte streaming loads, and used as the A fragment
// without passing through shared memory. The reduction index is permuted
// consistently on both operands (a dot product does not depend on the order
// of its terms): in every 32-wide step, lane q = lane % 4 owns the 8
// contiguous indices 8q..8q+7 of its two rows, which feed the k-slots
// {2q, 2q+1, 2q+8, 2q+9} of two MMAs; the token fragment is loaded with the
// same 16-byte pattern from the activations.
//
// int4 experts: a step is one 128-wide scale group and lane q owns indices
// 32q..32q+31 (16 bytes). The weights were reordered at create so each 32-bit
// word holds 8 consecutive indices with even ones in the low half-word; one
// LOP3 per pair turns two nibbles into bf16 (136 + q), an HSUB2 removes the
// 136, and the group's partial sums are scaled by the row's bf16 scale in
// fp32: sum_g s_g * sum_{i in g} q_i x_i, i.e. exactly w = q * s.
//
// Gate and up tiles of the same 16 features are processed by one warp so
// silu(gate) * up is applied in registers (h is rounded to bf16 for the down
// projection). The down projection splits its reduction into `splits`
// slices when there are too few (expert, 32-row) items to fill the GPU; the
// slices are summed in fixed order later (no float atomics).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace coli {
namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerBlock = kThreads / 32;
template <bool INT4>
constexpr int kMaxRowsPerPass = INT4 ? 16 : 32;  // token rows per weight pass

// int4: per-warp cp.async ring, kRing steps of 4 x 16 bytes per lane
constexpr int kRing = 3;
constexpr int kRingStep = 4 * 32 * 16;  // 2 KiB per warp and step
constexpr size_t kI4Smem = static_cast<size_t>(kThreads / 32) * kRing * kRingStep;
extern __shared__ __align__(16) uint8_t dec_smem[];

COLI_DEV uint4 zero4() { return make_uint4(0u, 0u, 0u, 0u); }

// acc[m][n] += A(tile m) x B(n) over one 8-index chunk held as bf16 uint4s:
// ar/ar8 rows r and r+8 of tile m, b the token fragment.
template <int NT>
COLI_DEV void mma_chunk(float (&acc)[2][NT][4], const uint4 (&ar)[2], const uint4 (&ar8)[2],
                        const uint4 (&b)[NT]) {
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      mma_bf16_16816(acc[m][n], ar[m].x, ar8[m].x, ar[m].y, ar8[m].y, b[n].x, b[n].y);
      mma_bf16_16816(acc[m][n], ar[m].z, ar8[m].z, ar[m].w, ar8[m].w, b[n].z, b[n].w);
    }
}

// One warp: two 16-row weight tiles x NT 8-token tiles over steps [s0, s1).
// wrow[m][h]: byte pointer to row (r + 8h) of tile m, already offset by this
// lane's 16-byte column; a step advances 64 bytes. xrow[n]: byte pointer to
// this lane's token row of tile n (offset by the lane's column), nullptr for
// padding rows. srow[m][h]: int4 scales of the same rows (one per step).
template <bool INT4, int NT>
COLI_DEV void mainloop(const uint8_t* const (&wrow)[2][2], const __nv_bfloat16* const (&srow)[2][2],
                       const uint8_t* const (&xrow)[NT], int s0, int s1,
                       float (&acc)[2][NT][4], const float* const (&xs)[NT][2]) {
  if constexpr (!INT4) {
    // loads in flight per lane: U * (4 + NT) x 16 bytes
    constexpr int U = NT == 1 ? 4 : (NT == 2 ? 2 : 1);
    int s = s0;
    for (; s + U <= s1; s += U) {
      uint4 a[U][2][2], b[U][NT];
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int h = 0; h < 2; ++h) a[u][m][h] = ldg_stream(wrow[m][h] + (s + u) * 64);
#pragma unroll
        for (int n = 0; n < NT; ++n)
          b[u][n] = xrow[n] ? ldg_keep(xrow[n] + (s + u) * 64) : zero4();
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint4 ar[2] = {a[u][0][0], a[u][1][0]};
        const uint4 ar8[2] = {a[u][0][1], a[u][1][1]};
        mma_chunk<NT>(acc, ar, ar8, b[u]);
      }
    }
    for (; s < s1; ++s) {
      uint4 ar[2], ar8[2], b[NT];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        ar[m] = ldg_stream(wrow[m][0] + s * 64);
        ar8[m] = ldg_stream(wrow[m][1] + s * 64);
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) b[n] = xrow[n] ? ldg_keep(xrow[n] + s * 64) : zero4();
      mma_chunk<NT>(acc, ar, ar8, b);
    }
  } else {
    // A step is one 128-index group. Three things keep a warp's step short:
    //  - weights: the lane's four 16-byte fragments travel through a
    //    lane-private cp.async ring in shared memory, kRing - 1 steps ahead
    //    (many bytes in flight without holding registers); chunk j of every
    //    lane is contiguous, so the 16-byte accesses are conflict-free;
    //  - activations: the next step's fragments are loaded into registers
    //    while this step computes, so the L1/L2 latency is hidden;
    //  - arithmetic: one LOP3 per weight pair (values 136 + q); the offset
    //    136 * sum(x) of each token and group comes from a table made once
    //    per forward (k_group_sums), so the tensor pipe only does the
    //    weight MMAs (legacy MMA issue rate is what bounds this loop).
    // The lane's x fragment is 64 bytes (32 consecutive indices) at byte
    // offset 256*s + 64*q; the ring is sized to leave most of L1 to it.
    const int lane = threadIdx.x & 31;
    const uint32_t ring = smem_u32(dec_smem) + (threadIdx.x >> 5) * kRing * kRingStep + lane * 16;
    auto issue = [&](int step, int slot) {
      if (step < s1) {
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int h = 0; h < 2; ++h)
            cp_async16(ring + slot * kRingStep + (2 * m + h) * 512, wrow[m][h] + step * 64);
      }
      cp_async_commit();
    };
#pragma unroll
    for (int i = 0; i < kRing - 1; ++i) issue(s0 + i, i);
    // activations one step ahead when a single token tile leaves room for
    // the extra registers; with two tiles they are loaded at the step start
    constexpr bool kAhead = NT == 1;
    uint4 bx[NT][4];
    if (kAhead) {
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int v = 0; v < 4; ++v)
          bx[n][v] = xrow[n] ? ldg_keep(xrow[n] + s0 * 256 + v * 16) : zero4();
    }
    int slot = 0;
    for (int s = s0; s < s1; ++s) {
      issue(s + kRing - 1, slot == 0 ? kRing - 1 : slot - 1);
      float sc[2][2];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h) sc[m][h] = __bfloat162float(srow[m][h][s]);
      cp_async_wait<kRing - 1>();  // this lane's copies of step s have landed
      uint4 a[2][2];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int h = 0; h < 2; ++h) a[m][h] = lds128(ring + slot * kRingStep + (2 * m + h) * 512);
      slot = slot + 1 == kRing ? 0 : slot + 1;
      uint4 cx[NT][4];  // this step's activations
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          if (kAhead) {  // take them, and request the next step's
            cx[n][v] = bx[n][v];
            if (s + 1 < s1)
              bx[n][v] = xrow[n] ? ldg_keep(xrow[n] + (s + 1) * 256 + v * 16) : zero4();
          } else {
            cx[n][v] = xrow[n] ? ldg_keep(xrow[n] + s * 256 + v * 16) : zero4();
          }
        }
      float g[2][NT][4], corr[NT][2];
#pragma unroll
      for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int c = 0; c < 4; ++c) g[0][n][c] = g[1][n][c] = 0.f;
#pragma unroll
        for (int t = 0; t < 2; ++t) corr[n][t] = xs[n][t] ? xs[n][t][s] : 0.f;  // 136 sum x
      }
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        uint4 bv[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) bv[n] = cx[n][v];
        const uint4 ar[2] = {dequant136(word_of(a[0][0], v)), dequant136(word_of(a[1][0], v))};
        const uint4 ar8[2] = {dequant136(word_of(a[0][1], v)), dequant136(word_of(a[1][1], v))};
        mma_chunk<NT>(g, ar, ar8, bv);
      }
      // sum q x = sum (136 + q) x - 136 sum x, times the row's scale
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int c = 0; c < 4; ++c)
            acc[m][n][c] = fmaf(sc[m][c >> 1], g[m][n][c] - corr[n][c & 1], acc[m][n][c]);
    }
    cp_async_wait<0>();  // no copy of this lane outlives the chunk
  }
}

struct DecArgs {
  const float* xsum;             // int4: 136 * per-group sums of the activation rows
  const uint8_t* w;              // gate/up or down weights (bytes)
  const __nv_bfloat16* s;        // int4 scales or nullptr
  const uint8_t* const* wtab;    // residency tier: expert e's weights at wtab[e], or nullptr
  const uint8_t* const* stab;    // ... and its int4 scales at stab[e]
  const __nv_bfloat16* x;        // activations [rows][K] (x_perm or H), or x [T][K]
  const int32_t* row_token;      // non-null: row r reads x[row_token[r]] (and its xsum row)
  const int32_t* offsets;        // [E+1]
  int E, K;                      // experts, reduction length
  int rows_per_expert;           // weight rows per expert (2f or d)
  int f;                         // features (gate/up)
  int d;                         // outputs (down)
  int splits;                    // reduction slices (down)
  __nv_bfloat16* H;              // gate/up output [rows][f]
  float* y_part;                 // down output [splits][rows][d]
  size_t part_stride;            // elements between slices
};

// Byte offset of the lane's 16-byte column within a row at step 0.
template <bool INT4>
COLI_DEV size_t row_bytes(int K) {
  return INT4 ? static_cast<size_t>(K) / 2 : static_cast<size_t>(K) * 2;
}

template <bool INT4, int NT>
COLI_DEV void gateup_chunk(const DecArgs& A, const int32_t* tok, int e, int n0, int row0,
                          int nrows) {
  const int lane = threadIdx.x & 31, r = lane >> 2, q = lane & 3;
  const size_t rb = row_bytes<INT4>(A.K);
  const int gs = A.K / 128;
  // interleaved rows: gate feature n -> 128*(n/64) + n%64, up -> +64
  const size_t gin = 128 * (n0 / 64) + (n0 % 64);  // row within the expert
  const uint8_t* wbase = A.wtab ? A.wtab[e] : A.w + static_cast<size_t>(e) * A.rows_per_expert * rb;
  const __nv_bfloat16* sbase =
      !INT4 ? nullptr
            : (A.stab ? reinterpret_cast<const __nv_bfloat16*>(A.stab[e])
                      : A.s + static_cast<size_t>(e) * A.rows_per_expert * gs);
  const uint8_t* wrow[2][2];
  const __nv_bfloat16* srow[2][2];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const size_t row = gin + 64 * m + r + 8 * h;
      wrow[m][h] = wbase + row * rb + q * 16;
      srow[m][h] = INT4 ? sbase + row * gs : nullptr;
    }
  // activation row of token column j: the permuted row, or the token's row of
  // x when the rows are gathered here (the dispatch then copies nothing)
  auto src_row = [&](int j) -> size_t {
    return static_cast<size_t>(tok ? tok[row0 + j] : row0 + j);
  };
  const uint8_t* xrow[NT];
  const int xlane = INT4 ? q * 64 : q * 16;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int j = 8 * n + r;
    xrow[n] = j < nrows ? reinterpret_cast<const uint8_t*>(A.x + src_row(j) * A.K) + xlane
                        : nullptr;
  }
  float acc[2][NT][4];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[m][n][c] = 0.f;
  const int steps = INT4 ? A.K / 128 : A.K / 32;
  const float* xs[NT][2];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int j = 8 * n + 2 * q + t;  // the accumulator columns this lane holds
      xs[n][t] = (INT4 && j < nrows) ? A.xsum + src_row(j) * gs : nullptr;
    }
  mainloop<INT4, NT>(wrow, srow, xrow, 0, steps, acc, xs);
  // acc[0] = gate, acc[1] = up: rows (features) r, r+8; columns (tokens) 2q, 2q+1
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = 8 * n + 2 * q + (c & 1);
      if (j >= nrows) continue;
      const int feat = n0 + r + ((c & 2) ? 8 : 0);
      const float a = acc[0][n][c], u = acc[1][n][c];
      const float hval = a / (1.f + expf(-a)) * u;
      A.H[static_cast<size_t>(row0 + j) * A.f + feat] = __float2bfloat16_rn(hval);
    }
}

template <bool INT4, int NT>
COLI_DEV void down_chunk(const DecArgs& A, int e, int o0, int split, int row0, int nrows) {
  const int lane = threadIdx.x & 31, r = lane >> 2, q = lane & 3;
  const size_t rb = row_bytes<INT4>(A.K);
  const int gs = A.K / 128;
  const uint8_t* wbase = A.wtab ? A.wtab[e] : A.w + static_cast<size_t>(e) * A.rows_per_expert * rb;
  const __nv_bfloat16* sbase =
      !INT4 ? nullptr
            : (A.stab ? reinterpret_cast<const __nv_bfloat16*>(A.stab[e])
                      : A.s + static_cast<size_t>(e) * A.rows_per_expert * gs);
  const uint8_t* wrow[2][2];
  const __nv_bfloat16* srow[2][2];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const size_t row = static_cast<size_t>(o0) + 16 * m + r + 8 * h;  // within the expert
      wrow[m][h] = wbase + row * rb + q * 16;
      srow[m][h] = INT4 ? sbase + row * gs : nullptr;
    }
  const uint8_t* xrow[NT];
  const int xlane = INT4 ? q * 64 : q * 16;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int j = 8 * n + r;
    xrow[n] = j < nrows ? reinterpret_cast<const uint8_t*>(A.x + static_cast<size_t>(row0 + j) * A.K) + xlane
                        : nullptr;
  }
  float acc[2][NT][4];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[m][n][c] = 0.f;
  const int steps = INT4 ? A.K / 128 : A.K / 32;
  const int s0 = static_cast<int>(static_cast<long>(steps) * split / A.splits);
  const int s1 = static_cast<int>(static_cast<long>(steps) * (split + 1) / A.splits);
  const float* xs[NT][2];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int j = 8 * n + 2 * q + t;  // the accumulator columns this lane holds
      xs[n][t] = (INT4 && j < nrows) ? A.xsum + static_cast<size_t>(row0 + j) * gs : nullptr;
    }
  mainloop<INT4, NT>(wrow, srow, xrow, s0, s1, acc, xs);
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

// bf16: the expert offsets (and, for a decode-sized batch, the row -> token
// map) are copied into shared memory once per block, so no item starts with a
// dependent global load. Returns the row -> token map to use (the copy, the
// global one, or nullptr). The int4 kernels declare no static shared memory:
// their blocks fill the 48 KiB weight ring exactly, and any more would move
// the SM's shared-memory carve-out up a step and shrink the L1 that holds
// their activations (measured: 10% slower).
constexpr int kMaxE = 256;
constexpr int kTokStage = 2048;
COLI_DEV const int32_t* stage_maps(const DecArgs& A, int* s_off, int* s_tok) {
  for (int i = threadIdx.x; i <= A.E; i += blockDim.x) s_off[i] = A.offsets[i];
  const int n_rows = A.offsets[A.E];
  const bool tok = s_tok != nullptr && A.row_token != nullptr && n_rows <= kTokStage;
  if (tok)
    for (int i = threadIdx.x; i < n_rows; i += blockDim.x) s_tok[i] = A.row_token[i];
  __syncthreads();
  return tok ? s_tok : A.row_token;
}

// Persistent: warp w of the grid takes items w, w + W, w + 2W, ...; an item
// is (expert, 16 features); consecutive items share the expert so the warps
// of a block re-read the same activation rows from L1.
template <bool INT4>
__global__ void __launch_bounds__(kThreads, 2) k_dec_gateup(const DecArgs A) {
  const int32_t* off = A.offsets;
  const int32_t* tok = A.row_token;
  if constexpr (!INT4) {
    __shared__ int s_off[kMaxE + 1], s_tok[kTokStage];
    tok = stage_maps(A, s_off, s_tok);
    off = s_off;
  }
  const int W = gridDim.x * kWarpsPerBlock;
  const int per_e = A.f / 16;
  const int items = A.E * per_e;
  for (int it = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); it < items; it += W) {
    const int e = it / per_e, n0 = (it % per_e) * 16;
    const int r0 = off[e], r1 = off[e + 1];
    for (int row0 = r0; row0 < r1; row0 += kMaxRowsPerPass<INT4>) {
      const int nrows = min(kMaxRowsPerPass<INT4>, r1 - row0);
      switch ((nrows + 7) / 8) {
        case 1: gateup_chunk<INT4, 1>(A, tok, e, n0, row0, nrows); break;
        case 2: gateup_chunk<INT4, 2>(A, tok, e, n0, row0, nrows); break;
        case 3: if constexpr (!INT4) gateup_chunk<INT4, 3>(A, tok, e, n0, row0, nrows); break;
        default: if constexpr (!INT4) gateup_chunk<INT4, 4>(A, tok, e, n0, row0, nrows); break;
      }
    }
  }
}

// Item = (slice, expert, 32 outputs); the slice is outermost so neighbouring
// warps read the same part of H.
template <bool INT4>
__global__ void __launch_bounds__(kThreads, 2) k_dec_down(const DecArgs A) {
  const int32_t* off = A.offsets;
  if constexpr (!INT4) {
    __shared__ int s_off[kMaxE + 1];
    stage_maps(A, s_off, nullptr);
    off = s_off;
  }
  const int W = gridDim.x * kWarpsPerBlock;
  const int per_e = A.d / 32;
  const int per_split = A.E * per_e;
  const int items = per_split * A.splits;
  for (int it = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); it < items; it += W) {
    const int split = it / per_split, rem = it % per_split;
    const int e = rem / per_e, o0 = (rem % per_e) * 32;
    const int r0 = off[e], r1 = off[e + 1];
    for (int row0 = r0; row0 < r1; row0 += kMaxRowsPerPass<INT4>) {
      const int nrows = min(kMaxRowsPerPass<INT4>, r1 - row0);
      switch ((nrows + 7) / 8) {
        case 1: down_chunk<INT4, 1>(A, e, o0, split, row0, nrows); break;
        case 2: down_chunk<INT4, 2>(A, e, o0, split, row0, nrows); break;
        case 3: if constexpr (!INT4) down_chunk<INT4, 3>(A, e, o0, split, row0, nrows); break;
        default: if constexpr (!INT4) down_chunk<INT4, 4>(A, e, o0, split, row0, nrows); break;
      }
    }
  }
}

// out[r][g] = 136 * sum of the 128 activations of group g of row r (fp32,
// fixed order: 4 per lane, then a butterfly), one warp per (row, group).
__global__ void __launch_bounds__(256)
    k_group_sums(const __nv_bfloat16* __restrict__ rows, int n_rows, int K,
                 float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int groups = K / 128;
  const long total = static_cast<long>(n_rows) * groups;
  for (long w = blockIdx.x * 8L + (threadIdx.x >> 5); w < total; w += gridDim.x * 8L) {
    const long r = w / groups;
    const int g = static_cast<int>(w % groups);
    const uint2 v = *reinterpret_cast<const uint2*>(rows + r * K + g * 128 + lane * 4);
    float sum = (bf16_lo(v.x) + bf16_hi(v.x)) + (bf16_lo(v.y) + bf16_hi(v.y));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) out[w] = 136.f * sum;
  }
}

}  // namespace

cudaError_t launch_group_sums(const __nv_bfloat16* rows, int n_rows, int K, float* out,
                              cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  const long warps = static_cast<long>(n_rows) * (K / 128);
  long grid = (warps + 7) / 8;
  if (grid > 4096) grid = 4096;
  k_group_sums<<<static_cast<unsigned>(grid), 256, 0, st>>>(rows, n_rows, K, out);
  return cudaGetLastError();
}

int dec_blocks_per_sm() {
  // the int4 kernels hold their weight ring in dynamic shared memory
  cudaFuncSetAttribute(k_dec_gateup<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(kI4Smem));
  cudaFuncSetAttribute(k_dec_down<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(kI4Smem));
  int a = 0, b = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, k_dec_gateup<false>, kThreads, 0) !=
      cudaSuccess)
    a = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_dec_gateup<true>, kThreads, kI4Smem) !=
      cudaSuccess)
    b = 1;
  int c = a < b ? a : b;
  return c < 1 ? 1 : c;
}

int dec_down_splits(int n_rows, int E, int d, int steps, int n_warps, int max_splits) {
  // Items (expert, 32 outputs, slice) are dealt round-robin to the warps, so
  // the slowest warp does ceil(items / warps) of them: pick the fewest
  // slices that keep that within 5% of the mean (or the best balance), with
  // at least 8 reduction steps per slice.
  const int active = n_rows < E ? n_rows : E;  // at most this many non-empty experts
  if (active <= 0 || max_splits <= 1) return 1;
  const long per = static_cast<long>(active) * (d / 32);
  int best = 1;
  double best_eff = 0.0;
  for (int s = 1; s <= max_splits && steps / s >= 8; ++s) {
    const long items = per * s;
    if (items < n_warps && s < max_splits) {
      // fewer items than warps: every extra slice adds parallelism
      const double eff = static_cast<double>(items) / n_warps;
      if (eff > best_eff) { best_eff = eff; best = s; }
      continue;
    }
    const long rounds = (items + n_warps - 1) / n_warps;
    const double eff = static_cast<double>(items) / (static_cast<double>(rounds) * n_warps);
    if (eff >= 0.95) return s;
    if (eff > best_eff + 1e-9) { best_eff = eff; best = s; }
  }
  return best;
}

cudaError_t launch_dec_gateup(const FfnWeights& w, const __nv_bfloat16* x,
                              const int32_t* row_token, const int32_t* offsets, int E, int d,
                              int f, __nv_bfloat16* H, const float* xsum, int grid,
                              cudaStream_t st) {
  DecArgs A{};
  A.xsum = xsum;
  A.w = static_cast<const uint8_t*>(w.w_gu);
  A.s = w.s_gu;
  A.wtab = w.tab_gu;
  A.stab = w.tab_sgu;
  A.x = x;
  A.row_token = row_token;
  A.offsets = offsets;
  A.E = E;
  A.K = d;
  A.rows_per_expert = 2 * f;
  A.f = f;
  A.d = d;
  A.splits = 1;
  A.H = H;
  if (w.wdt == DT_I4G128) k_dec_gateup<true><<<grid, kThreads, kI4Smem, st>>>(A);
  else k_dec_gateup<false><<<grid, kThreads, 0, st>>>(A);
  return cudaGetLastError();
}

cudaError_t launch_dec_down(const FfnWeights& w, const __nv_bfloat16* H, const int32_t* offsets,
                            int E, int d, int f, int splits, float* y_part, size_t part_stride,
                            const float* hsum, int grid, cudaStream_t st) {
  DecArgs A{};
  A.xsum = hsum;
  A.w = static_cast<const uint8_t*>(w.w_dn);
  A.s = w.s_dn;
  A.wtab = w.tab_dn;
  A.stab = w.tab_sdn;
  A.x = H;
  A.offsets = offsets;
  A.E = E;
  A.K = f;
  A.rows_per_expert = d;
  A.f = f;
  A.d = d;
  A.splits = splits;
  A.y_part = y_part;
  A.part_stride = part_stride;
  if (w.wdt == DT_I4G128) k_dec_down<true><<<grid, kThreads, kI4Smem, st>>>(A);
  else k_dec_down<false><<<grid, kThreads, 0, st>>>(A);
  return cudaGetLastError();
}

}  // namespace coli
