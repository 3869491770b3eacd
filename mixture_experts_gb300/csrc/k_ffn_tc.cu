// A3, prefill path: grouped expert GEMM on the 5th-generation tensor cores,
// bf16 expert weights (int4 and MX experts: k_ffn_tcq.cu, which dequantises
// the weights into tensor memory).
//
// For groups of hundreds of rows per expert the FFN is a dense contraction
// (per expert: rows x d x 2f for gate/up, rows x f x d for down), so it runs
// on tcgen05: TMA copies 128x64 activation tiles and 256x64 weight tiles
// (128-byte swizzle) into a 4-stage shared-memory ring, one thread issues
// tcgen05.mma (M=128, N=256, K=16, bf16 in, fp32 accumulate) into a tensor
// memory accumulator, and four epilogue warps read the accumulator back with
// tcgen05.ld. The accumulator is double-buffered in TMEM (2 x 256 of the 512
// columns) so the epilogue of one tile overlaps the main loop of the next.
//
// Grouping (the per-expert GEMM fed by the token-to-expert map and expert
// offsets of the trdm.cn overview page, section 3.3): each CTA derives the
// tile list from the device-side offsets — expert e contributes
// ceil(rows_e / 128) row tiles x (N / 256) column tiles, experts without rows
// contribute none (their weights are never read: wzjinhao.cn page,
// section 2.3) — and walks it with a static stride of gridDim.x, consecutive
// tiles sharing the weight tile so the L2 serves the other row tiles. Row
// tiles that run past an expert's rows are computed but not stored (an output
// row depends on its own input row only, so whatever those rows hold — the
// next expert's rows, or stale workspace past the last group — never reaches
// a stored value); rows past the end of the buffer are zero-filled by TMA.
//
// Gate/up epilogue: the weights are interleaved in 64-row blocks (gate rows,
// then the matching up rows), so accumulator columns c and c + 64 of each
// 128-column half are gate and up of the same feature; h = silu(gate) * up is
// written as bf16. Down epilogue: fp32 rows of y_perm.
//
// Every mbarrier wait is bounded by one kernel-wide deadline; a CTA that
// reaches it latches COLI_ETIMEOUT, unwinds all roles, waits briefly for
// copies in flight, frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace coli {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int A_BYTES = BM * BK * 2;  // 16 KiB
constexpr int B_BYTES = BN * BK * 2;  // 32 KiB
constexpr int TMEM_COLS = 512;
constexpr int kMaxE = 256;
constexpr int STAGES = 4;
constexpr int kThreads = 192;  // warps: 0 TMA, 1 MMA (+ TMEM alloc), 2-5 epilogue
constexpr int kStageBytes = A_BYTES + B_BYTES;

// bf16 x bf16 -> fp32, A and B K-major, M = 128, N = 256.
constexpr uint32_t kIdesc = idesc_bf16(BM, BN);

struct __align__(8) Ctrl {
  uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2];
  uint32_t tmem_base;
  int abort;
  int tile_off[kMaxE + 1];  // first tile of expert e
  int row_off[kMaxE + 1];   // first row of expert e (the offsets)
};

constexpr size_t kSmem = 1024 + STAGES * kStageBytes + sizeof(Ctrl);

struct Tile {
  int e, nt, mt;
};

COLI_DEV Tile decode_tile(const Ctrl& C, int E, int n_tiles_n, int t) {
  int lo = 0, hi = E;  // tile_off[lo] <= t < tile_off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (C.tile_off[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int rows = C.row_off[lo + 1] - C.row_off[lo];
  const int mts = (rows + BM - 1) / BM;
  const int local = t - C.tile_off[lo];
  return Tile{lo, local / mts, local % mts};
}

// EPI 0: gate/up + SwiGLU -> bf16 H [rows][N/2]; EPI 1: fp32 out [rows][N];
// EPI 2: bf16 out [rows][N].
template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
              const int32_t* __restrict__ offsets, int E, int K, int N, void* __restrict__ out,
              int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sa = smem_u32(base);
  const uint32_t sb = sa + STAGES * A_BYTES;
  Ctrl& C = *reinterpret_cast<Ctrl*>(base + STAGES * kStageBytes);
  volatile int* abort = &C.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t deadline = global_timer_ns() + kWaitTimeoutNs;
  const int n_tiles_n = (N + BN - 1) / BN;
  const int kblocks = K / BK;

  // tile table from the expert offsets (warp 0), barriers (thread 0),
  // tensor memory (warp 1)
  if (warp == 0) {
    int mts[kMaxE / 32], sum = 0;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
      const int e = lane * (kMaxE / 32) + i;
      int m = 0;
      if (e < E) {
        const int r0 = offsets[e], r1 = offsets[e + 1];
        C.row_off[e] = r0;
        if (e == E - 1) C.row_off[E] = r1;
        m = ((r1 - r0 + BM - 1) / BM) * n_tiles_n;
      }
      mts[i] = m;
      sum += m;
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
      const int e = lane * (kMaxE / 32) + i;
      if (e < E) C.tile_off[e] = run;
      run += mts[i];
    }
    if (lane == 31) C.tile_off[E] = incl;  // all tiles
    if (lane == 0) {
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(smem_u32(&C.full[s]), 1);
        mbar_init(smem_u32(&C.empty[s]), 1);
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(smem_u32(&C.tfull[a]), 1);
        mbar_init(smem_u32(&C.tempty[a]), 4);
      }
      C.abort = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
  } else if (warp == 1) {
    tmem_alloc(smem_u32(&C.tmem_base), TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = C.tmem_base;
  const int total = C.tile_off[E];

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < total && !*abort; t += gridDim.x) {
        const Tile tl = decode_tile(C, E, n_tiles_n, t);
        const int a_row = C.row_off[tl.e] + tl.mt * BM;
        const int b_row = tl.e * N + tl.nt * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          // a free slot: the MMA of its last use has completed
          if (!wait_bar(smem_u32(&C.empty[stage]), phase ^ 1u, deadline, abort)) break;
          const uint32_t fb = smem_u32(&C.full[stage]);
          mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
          tma_load_2d(sa + stage * A_BYTES, &map_a, fb, kb * BK, a_row);
          tma_load_2d(sb + stage * B_BYTES, &map_b, fb, kb * BK, b_row);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer
      int stage = 0, local = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < total && !*abort; t += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!wait_bar(smem_u32(&C.tempty[acc]), acc_phase ^ 1u, deadline, abort)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bar(smem_u32(&C.full[stage]), phase, deadline, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sa + stage * A_BYTES, b0 = sb + stage * B_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_ss(d_tmem, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), kIdesc,
                    (kb | k) != 0 ? 1u : 0u);
          umma_commit(smem_u32(&C.empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&C.tfull[acc]));
      }
    }
  } else if (warp < 6) {  // ---- epilogue: warps 2..5, TMEM lanes 32*(warp%4) ..
    const int qw = warp & 3;
    const int r = qw * 32 + lane;
    int local = 0;
    for (int t = blockIdx.x; t < total && !*abort; t += gridDim.x, ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      // warp-uniform verdict: tcgen05.ld below is warp-collective
      if (!__all_sync(0xffffffffu, wait_bar(smem_u32(&C.tfull[acc]), acc_phase, deadline, abort)))
        break;
      tc_fence_after();
      const Tile tl = decode_tile(C, E, n_tiles_n, t);
      const int row = C.row_off[tl.e] + tl.mt * BM + r;
      const bool valid = row < C.row_off[tl.e + 1];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(qw * 32) << 16) + acc * BN;
      if constexpr (EPI == 0) {
        const int F = N / 2;  // features
        __nv_bfloat16* H = static_cast<__nv_bfloat16*>(out);
#pragma unroll 1
        for (int ci = 0; ci < 4; ++ci) {
          const int c = (ci & 1) + (ci >> 1) * 4;  // gate chunks 0, 1, 4, 5
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c * 32, g);
          tmem_ld32(taddr + (c + 2) * 32, u);
          const int feat = tl.nt * 128 + (c & 1) * 32 + (c >> 2) * 64;
          if (valid && feat < F) {
            uint32_t packed[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float a0 = __uint_as_float(g[2 * j]), a1 = __uint_as_float(g[2 * j + 1]);
              const float u0 = __uint_as_float(u[2 * j]), u1 = __uint_as_float(u[2 * j + 1]);
              packed[j] = pack_bf16x2(a0 / (1.f + expf(-a0)) * u0, a1 / (1.f + expf(-a1)) * u1);
            }
            uint4* dst = reinterpret_cast<uint4*>(H + static_cast<size_t>(row) * F + feat);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                                  packed[4 * v + 3]);
          }
        }
      } else if constexpr (EPI == 1) {
        float* Y = static_cast<float*>(out);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(taddr + c * 32, v);
          const int col = tl.nt * BN + c * 32;
          if (valid && col < N) {
            uint4* dst = reinterpret_cast<uint4*>(Y + static_cast<size_t>(row) * N + col);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          }
        }
      } else {  // EPI 2: bf16 out (round to nearest even)
        __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(out);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(taddr + c * 32, v);
          const int col = tl.nt * BN + c * 32;
          if (valid && col < N) {
            uint32_t p[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              p[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            uint4* dst = reinterpret_cast<uint4*>(Y + static_cast<size_t>(row) * N + col);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&C.tempty[acc]));
    }
  }

  __syncthreads();
  if (*abort) {
    if (threadIdx.x == 0) {
      latch_error(status, kErrTimeout);
      const uint64_t t0 = global_timer_ns();  // let copies in flight land
      while (global_timer_ns() - t0 < 1000000ull) {
      }
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---- CTA-pair kernel (bf16 weights) ------------------------------------------------
// A pair of CTAs (a cluster of two, one per SM) computes a 256-row x 256-column
// tile with cta_group::2 MMAs issued by the first CTA: each CTA loads its own
// 128 activation rows and half (128 rows) of the weight tile into its shared
// memory, and the tensor cores of the pair read both halves, so a CTA moves
// 32 KiB per 64-deep stage instead of 48 KiB for the same MMA work. Each
// CTA's tensor memory receives its 128 rows of the accumulator and its own
// four epilogue warps drain them. The first CTA's barriers count the pair's
// TMA bytes and both CTAs' epilogue arrivals; its MMA commits arrive on the
// matching barriers of both CTAs.
constexpr int PAIR_STAGES = 6;
constexpr int BH_BYTES = (BN / 2) * BK * 2;  // 16 KiB: a CTA's half of the weight tile
constexpr uint32_t kIdescPair = idesc_bf16(2 * BM, BN);

struct __align__(8) CtrlPair {
  uint64_t full[PAIR_STAGES], empty[PAIR_STAGES], tfull[2], tempty[2];
  uint32_t tmem_base;
  int abort;
  int tile_off[kMaxE + 1];
  int row_off[kMaxE + 1];
};

// 16 KiB of headroom after the weight stages: every operand read of the MMAs
// stays inside this CTA's allocation whatever the stage.
constexpr int kPairGuard = 16384;
constexpr size_t kPairSmem =
    1024 + PAIR_STAGES * (A_BYTES + BH_BYTES) + kPairGuard + sizeof(CtrlPair);

// Tile t of the pair grid: expert, 256-column tile, 256-row tile.
COLI_DEV Tile decode_pair_tile(const CtrlPair& C, int E, int t) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (C.tile_off[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int rows = C.row_off[lo + 1] - C.row_off[lo];
  const int mts = (rows + 2 * BM - 1) / (2 * BM);
  const int local = t - C.tile_off[lo];
  return Tile{lo, local / mts, local % mts};
}

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    k_tc_gemm_pair(const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_b, const int32_t* __restrict__ offsets,
                   int E, int K, int N, void* __restrict__ out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sa = smem_u32(base);
  const uint32_t sb = sa + PAIR_STAGES * A_BYTES;
  CtrlPair& C =
      *reinterpret_cast<CtrlPair*>(base + PAIR_STAGES * (A_BYTES + BH_BYTES) + kPairGuard);
  volatile int* abort = &C.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool first = rank == 0;
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const uint64_t deadline = global_timer_ns() + kWaitTimeoutNs;
  const int n_tiles_n = (N + BN - 1) / BN;
  const int kblocks = K / BK;

  if (warp == 0) {
    int mts[kMaxE / 32], sum = 0;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
      const int e = lane * (kMaxE / 32) + i;
      int m = 0;
      if (e < E) {
        const int r0 = offsets[e], r1 = offsets[e + 1];
        C.row_off[e] = r0;
        if (e == E - 1) C.row_off[E] = r1;
        m = ((r1 - r0 + 2 * BM - 1) / (2 * BM)) * n_tiles_n;
      }
      mts[i] = m;
      sum += m;
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
      const int e = lane * (kMaxE / 32) + i;
      if (e < E) C.tile_off[e] = run;
      run += mts[i];
    }
    if (lane == 31) C.tile_off[E] = incl;
    if (lane == 0) {
      for (int st = 0; st < PAIR_STAGES; ++st) {
        mbar_init(smem_u32(&C.full[st]), 1);
        mbar_init(smem_u32(&C.empty[st]), 1);
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(smem_u32(&C.tfull[a]), 1);
        mbar_init(smem_u32(&C.tempty[a]), 8);  // four epilogue warps in each CTA
      }
      C.abort = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
  } else if (warp == 1) {
    tmem_alloc_pair(smem_u32(&C.tmem_base), TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before anything arrives on them
  tc_fence_after();
  const uint32_t tmem = C.tmem_base;
  const int total = C.tile_off[E];

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer (both CTAs): own rows, own half of B
      int stage = 0;
      uint32_t phase = 0;
      for (int t = pair; t < total && !*abort; t += n_pairs) {
        const Tile tl = decode_pair_tile(C, E, t);
        const int a_row = C.row_off[tl.e] + tl.mt * 2 * BM + static_cast<int>(rank) * BM;
        const int b_row = tl.e * N + tl.nt * BN + static_cast<int>(rank) * (BN / 2);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bar_cluster(smem_u32(&C.empty[stage]), phase ^ 1u, deadline, abort)) break;
          const uint32_t fb = smem_u32(&C.full[stage]);
          if (first) mbar_arrive_expect_tx(fb, 2 * (A_BYTES + BH_BYTES));
          const uint32_t fb0 = map_shared(fb, 0);
          tma_load_2d_pair(sa + stage * A_BYTES, &map_a, fb0, kb * BK, a_row);
          tma_load_2d_pair(sb + stage * BH_BYTES, &map_b, fb0, kb * BK, b_row);
          if (++stage == PAIR_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && first) {  // ---- MMA issuer (first CTA of the pair)
      int stage = 0, local = 0;
      uint32_t phase = 0;
      for (int t = pair; t < total && !*abort; t += n_pairs, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!wait_bar_cluster(smem_u32(&C.tempty[acc]), acc_phase ^ 1u, deadline, abort)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bar_cluster(smem_u32(&C.full[stage]), phase, deadline, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sa + stage * A_BYTES, b0 = sb + stage * BH_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_ss_pair(d_tmem, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), kIdescPair,
                         (kb | k) != 0 ? 1u : 0u);
          umma_commit_pair(smem_u32(&C.empty[stage]));
          if (++stage == PAIR_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(smem_u32(&C.tfull[acc]));
      }
    }
  } else {  // ---- epilogue (both CTAs): warps 2..5, this CTA's 128 rows
    const int qw = warp & 3;
    const int r = qw * 32 + lane;
    int local = 0;
    for (int t = pair; t < total && !*abort; t += n_pairs, ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!__all_sync(0xffffffffu,
                      wait_bar_cluster(smem_u32(&C.tfull[acc]), acc_phase, deadline, abort)))
        break;
      tc_fence_after();
      const Tile tl = decode_pair_tile(C, E, t);
      const int row = C.row_off[tl.e] + tl.mt * 2 * BM + static_cast<int>(rank) * BM + r;
      const bool valid = row < C.row_off[tl.e + 1];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(qw * 32) << 16) + acc * BN;
      if constexpr (EPI == 0) {
        const int F = N / 2;
        __nv_bfloat16* H = static_cast<__nv_bfloat16*>(out);
#pragma unroll 1
        for (int ci = 0; ci < 4; ++ci) {
          const int c = (ci & 1) + (ci >> 1) * 4;
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c * 32, g);
          tmem_ld32(taddr + (c + 2) * 32, u);
          const int feat = tl.nt * 128 + (c & 1) * 32 + (c >> 2) * 64;
          if (valid && feat < F) {
            uint32_t packed[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float a0 = __uint_as_float(g[2 * j]), a1 = __uint_as_float(g[2 * j + 1]);
              const float u0 = __uint_as_float(u[2 * j]), u1 = __uint_as_float(u[2 * j + 1]);
              packed[j] = pack_bf16x2(a0 / (1.f + expf(-a0)) * u0, a1 / (1.f + expf(-a1)) * u1);
            }
            uint4* dst = reinterpret_cast<uint4*>(H + static_cast<size_t>(row) * F + feat);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                                  packed[4 * v + 3]);
          }
        }
      } else if constexpr (EPI == 1) {
        float* Y = static_cast<float*>(out);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(taddr + c * 32, v);
          const int col = tl.nt * BN + c * 32;
          if (valid && col < N) {
            uint4* dst = reinterpret_cast<uint4*>(Y + static_cast<size_t>(row) * N + col);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          }
        }
      } else {
        __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(out);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(taddr + c * 32, v);
          const int col = tl.nt * BN + c * 32;
          if (valid && col < N) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            uint4* dst = reinterpret_cast<uint4*>(Y + static_cast<size_t>(row) * N + col);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_shared(smem_u32(&C.tempty[acc]), 0));
    }
  }

  __syncthreads();
  if (*abort) {
    if (threadIdx.x == 0) {
      latch_error(status, kErrTimeout);
      const uint64_t t0 = global_timer_ns();  // let copies in flight land
      while (global_timer_ns() - t0 < 1000000ull) {
      }
    }
    __syncthreads();
  }
  cluster_sync();  // neither CTA frees tensor memory or exits while the pair still works
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

// 2-D bf16 [rows][cols] row-major, box [box_rows][64], 128-byte swizzle.
cudaError_t make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, int box_rows) {
  return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, rows, cols, BK, box_rows,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

cudaError_t encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* ptr,
                           uint64_t rows, uint64_t cols, int box_cols, int box_rows,
                           CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * static_cast<cuuint64_t>(elem_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

struct TcPlan {
  CUtensorMap map_wgu, map_wdn, map_xperm, map_h;
  bool pair;           // CTA-pair kernel with half-height weight maps
  QPlan* q = nullptr;  // int4 / MX weights: the tensor-memory-operand kernel
  int E, d, f, grid;
};

bool tc_supported(int wdt, int d, int f) {
  if (encode_fn() == nullptr) return false;
  if (wdt == DT_BF16) return d % 64 == 0 && f % 64 == 0;
  return tcq_supported(wdt, d, f);
}

template <int EPI>
static cudaError_t set_smem() {
  return cudaFuncSetAttribute(k_tc_gemm<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kSmem));
}

cudaError_t tc_plan_create(TcPlan** plan, int wdt, const void* w_gu, const void* w_dn,
                           const void* s_gu, const void* s_dn, int E, int d, int f, int max_rows,
                           const void* x_perm, const void* H, bool mx_general) {
  *plan = nullptr;
  TcPlan* p = new TcPlan();
  p->E = E;
  p->d = d;
  p->f = f;
  cudaError_t e;
  if (wdt != DT_BF16) {
    e = tcq_plan_create(&p->q, wdt, w_gu, w_dn, s_gu, s_dn, E, d, f, max_rows, x_perm, H,
                        mx_general);
    if (e != cudaSuccess) {
      delete p;
      return e;
    }
    *plan = p;
    return cudaSuccess;
  }
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
    delete p;
    return e;
  }
  // each CTA of a pair loads 128 of the 256 weight rows of a tile
  p->pair = sms >= 2;
  p->grid = p->pair ? sms & ~1 : sms;  // whole pairs
  const int box = p->pair ? BN / 2 : BN;
  e = make_map(&p->map_wgu, w_gu, static_cast<uint64_t>(E) * 2 * f, d, box);
  if (e == cudaSuccess) e = make_map(&p->map_wdn, w_dn, static_cast<uint64_t>(E) * d, f, box);
  if (e == cudaSuccess) e = set_smem<0>();
  if (e == cudaSuccess) e = set_smem<1>();
  if (e == cudaSuccess) e = set_smem<2>();
  for (auto fn : {k_tc_gemm_pair<0>, k_tc_gemm_pair<1>, k_tc_gemm_pair<2>})
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kPairSmem));
  if (e == cudaSuccess) e = make_map(&p->map_xperm, x_perm, static_cast<uint64_t>(max_rows), d, BM);
  if (e == cudaSuccess) e = make_map(&p->map_h, H, static_cast<uint64_t>(max_rows), f, BM);
  if (e != cudaSuccess) {
    delete p;
    return e;
  }
  *plan = p;
  return cudaSuccess;
}

void tc_plan_destroy(TcPlan* plan) {
  if (plan && plan->q) tcq_plan_destroy(plan->q);
  delete plan;
}

template <int EPI>
static void launch(const TcPlan* p, const CUtensorMap& map_a, const CUtensorMap& map_b,
                   const int32_t* offsets, int K, int N, void* out, cudaStream_t st,
                   int* status) {
  if (p->pair)
    k_tc_gemm_pair<EPI><<<p->grid, 192, kPairSmem, st>>>(map_a, map_b, offsets, p->E, K, N, out,
                                                         status);
  else
    k_tc_gemm<EPI><<<p->grid, kThreads, kSmem, st>>>(map_a, map_b, offsets, p->E, K, N, out,
                                                     status);
}

cudaError_t launch_tc_gateup(TcPlan* p, const void* x_perm, bool own_x_perm,
                             const int32_t* offsets, void* H, int n_rows, cudaStream_t st,
                             int* status) {
  if (p->q) return launch_tcq_gateup(p->q, x_perm, own_x_perm, offsets, H, n_rows, st, status);
  if (n_rows == 0) return cudaSuccess;
  CUtensorMap map_a;
  if (own_x_perm) {
    map_a = p->map_xperm;
  } else {
    const cudaError_t e = make_map(&map_a, x_perm, static_cast<uint64_t>(n_rows), p->d, BM);
    if (e != cudaSuccess) return e;
  }
  launch<0>(p, map_a, p->map_wgu, offsets, p->d, 2 * p->f, H, st, status);
  return cudaGetLastError();
}

cudaError_t launch_tc_down(TcPlan* p, const void* H, const int32_t* offsets, void* y_perm,
                           bool bf16_out, int n_rows, cudaStream_t st, int* status) {
  (void)H;  // always the plan's H buffer, mapped at create
  if (p->q) return launch_tcq_down(p->q, offsets, y_perm, bf16_out, n_rows, st, status);
  if (n_rows == 0) return cudaSuccess;
  if (bf16_out)
    launch<2>(p, p->map_h, p->map_wdn, offsets, p->f, p->d, y_perm, st, status);
  else
    launch<1>(p, p->map_h, p->map_wdn, offsets, p->f, p->d, y_perm, st, status);
  return cudaGetLastError();
}

}  // namespace coli
