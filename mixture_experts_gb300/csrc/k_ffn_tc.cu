// A3, prefill path: grouped expert GEMM on the 5th-generation tensor cores,
// bf16 expert weights (int4 and MX experts: k_ffn_tcq.cu, which dequantises
// the weights into tensor memory).
//
// For groups of hundreds of rows per expert the FFN is a dense contraction
// (per expert: rows x d x 2f for gate/up, rows x f x d for down), so it runs
// on tcgen05 with CTA pairs: TMA copies 64-deep slices of the weight tile and
// the token rows (128-byte swizzle) into a 6-stage shared-memory ring of each
// CTA, the pair's first CTA issues tcgen05.mma.cta_group::2 (bf16 in, fp32
// accumulate) into tensor memory, and four epilogue warps per CTA read the
// accumulator back with tcgen05.ld. The accumulator is double-buffered in
// tensor memory (2 x 256 of the 512 columns) so the epilogue of one tile
// overlaps the main loop of the next.
//
// Grouping (the per-expert GEMM fed by the token-to-expert map and expert
// offsets of the trdm.cn overview page, section 3.3): each CTA derives the
// tile list from the device-side offsets — expert e contributes
// ceil(2f or d / 256) weight tiles x ceil(rows_e / 256) token tiles, experts
// without rows contribute none (their weights are never read: wzjinhao.cn
// page, section 2.3) — and walks it with a static stride, consecutive tiles
// sharing the weight tile so the L2 serves the other token tiles. Token
// columns past an expert's rows are computed but not stored (an output row
// depends on its own input row only); rows past the end of the buffer are
// zero-filled by TMA.
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
constexpr int TMEM_COLS = 512;
constexpr int kMaxE = 256;

struct Tile {
  int e, nt, mt;  // expert, weight tile, token tile
};

// ---- CTA-pair kernel (bf16 weights) ------------------------------------------------
// A pair of CTAs (a cluster of two, one per SM) computes a tile of 256 weight
// rows x up to 256 token rows with cta_group::2 MMAs issued by the first CTA.
// The weights are the A operand (M = 256: each CTA loads its 128 rows) and
// the activations the B operand (N = the tile's token rows rounded up to 16:
// each CTA loads half of them), so a CTA moves 32 KiB per 64-deep stage and
// an expert's last, partial token tile costs what it holds (with 256-row
// token tiles the ragged tails were 16-18% extra MMA work on the
// mixtral_prefill and skewed workloads). Each CTA's tensor memory receives
// the accumulator rows of its 128 weight rows (D[weight row][token]) and its
// own four epilogue warps drain them. The first CTA's barriers count the
// pair's TMA bytes and both CTAs' epilogue arrivals; its MMA commits arrive
// on the matching barriers of both CTAs.
//
// Gate/up: a CTA's 128 weight rows are one interleaved block (gate rows of 64
// features, then their up rows), so lanes 0-63 hold gate rows and 64-127 the
// matching up rows. The warps of quarters q and q + 2 pair up: for each
// 32-token chunk each hands the other half of its values through a small
// shared-memory buffer (an mbarrier per pair and buffer, bounded waits), the
// gate warp finishes the chunk's first 16 tokens and the up warp the last 16,
// and h = silu(gate) * up goes to H [token][feature]. (Loading the weight
// rows in 16-row boxes so that gate and up of a feature share a warp took
// eight TMA copies per stage and slowed the gate/up GEMM by 25%.) Down: lane =
// output column. A store instruction writes 32 consecutive columns of a
// token row.
constexpr int PAIR_STAGES = 6;
constexpr int WH_BYTES = BM * BK * 2;        // 16 KiB: a CTA's 128 weight rows
constexpr int XH_BYTES = (BN / 2) * BK * 2;  // 16 KiB: a CTA's half of the 256 token rows
constexpr int XCH_BYTES = 4 * 2 * 16 * 32 * 4;  // gate/up hand-over: [quarter][buffer][16][32] fp32

struct __align__(8) CtrlPair {
  uint64_t full[PAIR_STAGES], empty[PAIR_STAGES], tfull[2], tempty[2], xbar[2][2];
  uint32_t tmem_base;
  int abort;
  int tile_off[kMaxE + 1];
  int row_off[kMaxE + 1];
};

constexpr size_t kPairSmem =
    1024 + PAIR_STAGES * (WH_BYTES + XH_BYTES) + XCH_BYTES + sizeof(CtrlPair);

// Tile t of the pair grid: expert, 256-row weight tile, 256-row token tile.
COLI_DEV Tile decode_pair_tile(const CtrlPair& C, int E, int t) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (C.tile_off[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int rows = C.row_off[lo + 1] - C.row_off[lo];
  const int mts = (rows + BN - 1) / BN;
  const int local = t - C.tile_off[lo];
  return Tile{lo, local / mts, local % mts};
}

// Token rows of a tile rounded up to 16 (the MMA's N).
COLI_DEV int pair_tile_n(const CtrlPair& C, const Tile& tl) {
  const int rows = min(BN, C.row_off[tl.e + 1] - C.row_off[tl.e] - tl.mt * BN);
  return (rows + 15) & ~15;
}

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    k_tc_gemm_pair(const __grid_constant__ CUtensorMap map_x,
                   const __grid_constant__ CUtensorMap map_w, const int32_t* __restrict__ offsets,
                   int E, int K, int N, void* __restrict__ out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sw = smem_u32(base);                // weight stages (A)
  const uint32_t sx = sw + PAIR_STAGES * WH_BYTES;  // activation stages (B)
  float* xch = reinterpret_cast<float*>(base + PAIR_STAGES * (WH_BYTES + XH_BYTES));
  CtrlPair& C =
      *reinterpret_cast<CtrlPair*>(base + PAIR_STAGES * (WH_BYTES + XH_BYTES) + XCH_BYTES);
  volatile int* abort = &C.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool first = rank == 0;
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const uint64_t deadline = global_timer_ns() + kWaitTimeoutNs;
  const int n_wt = (N + BN - 1) / BN;  // 256-row weight tiles per expert
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
        m = ((r1 - r0 + BN - 1) / BN) * n_wt;
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
        for (int b = 0; b < 2; ++b) mbar_init(smem_u32(&C.xbar[a][b]), 2);  // a warp pair
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
    if (lane == 0) {  // ---- TMA producer (both CTAs): own weight rows, own half of the tokens
      int stage = 0;
      uint32_t phase = 0;
      for (int t = pair; t < total && !*abort; t += n_pairs) {
        const Tile tl = decode_pair_tile(C, E, t);
        const int w_row = tl.e * N + tl.nt * BN + static_cast<int>(rank) * BM;
        const int x_row = C.row_off[tl.e] + tl.mt * BN +
                          static_cast<int>(rank) * (pair_tile_n(C, tl) / 2);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bar_cluster(smem_u32(&C.empty[stage]), phase ^ 1u, deadline, abort)) break;
          const uint32_t fb = smem_u32(&C.full[stage]);
          if (first) mbar_arrive_expect_tx(fb, 2 * (WH_BYTES + XH_BYTES));
          const uint32_t fb0 = map_shared(fb, 0);
          tma_load_2d_pair(sw + stage * WH_BYTES, &map_w, fb0, kb * BK, w_row);
          tma_load_2d_pair(sx + stage * XH_BYTES, &map_x, fb0, kb * BK, x_row);
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
        const uint32_t idesc = idesc_bf16(2 * BM, pair_tile_n(C, decode_pair_tile(C, E, t)));
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bar_cluster(smem_u32(&C.full[stage]), phase, deadline, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sw + stage * WH_BYTES, b0 = sx + stage * XH_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_ss_pair(d_tmem, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), idesc,
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
  } else {  // ---- epilogue (both CTAs): warps 2..5, lanes 32*(warp%4) .. of this CTA's rows
    const int q = warp & 3;
    int local = 0;
    uint32_t xseq = 0;   // gate/up hand-overs so far (the pair's buffers alternate)
    bool xfail = false;  // a hand-over wait gave up
    for (int t = pair; t < total && !*abort; t += n_pairs, ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!__all_sync(0xffffffffu,
                      wait_bar_cluster(smem_u32(&C.tfull[acc]), acc_phase, deadline, abort)))
        break;
      tc_fence_after();
      const Tile tl = decode_pair_tile(C, E, t);
      const int tok0 = C.row_off[tl.e] + tl.mt * BN;
      const int tok_end = C.row_off[tl.e + 1];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + acc * BN;
      if constexpr (EPI == 0) {
        const int F = N / 2;
        __nv_bfloat16* H = static_cast<__nv_bfloat16*>(out);
        const bool up = q >= 2;
        const int pq = q & 1;  // pair: gate quarter pq, up quarter pq + 2
        const int blk = 2 * tl.nt + static_cast<int>(rank);
        const int feat = blk * 64 + 32 * pq + lane;
        if (blk * 64 < F) {  // this CTA's block lies inside the expert's rows
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            const int t0 = tok0 + 32 * c;
            if (t0 >= tok_end) break;
            uint32_t v[32];
            tmem_ld32(taddr + 32 * c, v);
            // hand the partner what it finishes: the gate warp's values of
            // tokens 16..31, the up warp's of tokens 0..15
            const int b = xseq & 1;
            const uint32_t xph = (xseq >> 1) & 1u;
            ++xseq;
            float* mine = xch + ((q * 2 + b) * 16) * 32;
            const float* theirs = xch + (((q ^ 2) * 2 + b) * 16) * 32;
#pragma unroll
            for (int j = 0; j < 16; ++j) mine[j * 32 + lane] = __uint_as_float(v[up ? j : 16 + j]);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&C.xbar[pq][b]));
            if (!__all_sync(0xffffffffu,
                            wait_bar(smem_u32(&C.xbar[pq][b]), xph, deadline, abort))) {
              xfail = true;
              break;
            }
            // (silu with the fast exponential and division: h is rounded to
            // bf16, far coarser than their few-ulp error)
            const int tb = t0 + (up ? 16 : 0);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float other = theirs[j * 32 + lane];
              const float g = up ? other : __uint_as_float(v[j]);
              const float u = up ? __uint_as_float(v[16 + j]) : other;
              if (tb + j < tok_end)
                H[static_cast<size_t>(tb + j) * F + feat] =
                    __float2bfloat16_rn(__fdividef(g, 1.f + __expf(-g)) * u);
            }
          }
          if (xfail) break;
        }
      } else {
        const int col = tl.nt * BN + static_cast<int>(rank) * BM + 32 * q + lane;
        if (col - lane < N) {  // this warp's 32 columns lie inside the output
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            const int t0 = tok0 + 32 * c;
            if (t0 >= tok_end) break;
            uint32_t v[32];
            tmem_ld32(taddr + 32 * c, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (t0 + j >= tok_end) break;
              const size_t at = static_cast<size_t>(t0 + j) * N + col;
              if constexpr (EPI == 1) static_cast<float*>(out)[at] = __uint_as_float(v[j]);
              else
                static_cast<__nv_bfloat16*>(out)[at] =
                    __float2bfloat16_rn(__uint_as_float(v[j]));
            }
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
  QPlan* q = nullptr;  // int4 / MX weights: the tensor-memory-operand kernel
  int E, d, f, grid;
};

bool tc_supported(int wdt, int d, int f) {
  if (encode_fn() == nullptr) return false;
  if (wdt != DT_BF16) return tcq_supported(wdt, d, f);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  return d % 64 == 0 && f % 64 == 0 && sms >= 2;  // CTA pairs
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
  p->grid = sms & ~1;  // whole pairs
  // a CTA's 128 weight rows; token rows in a CTA's half of 256
  e = make_map(&p->map_wgu, w_gu, static_cast<uint64_t>(E) * 2 * f, d, BM);
  if (e == cudaSuccess) e = make_map(&p->map_wdn, w_dn, static_cast<uint64_t>(E) * d, f, BM);
  for (auto fn : {k_tc_gemm_pair<0>, k_tc_gemm_pair<1>, k_tc_gemm_pair<2>})
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kPairSmem));
  if (e == cudaSuccess)
    e = make_map(&p->map_xperm, x_perm, static_cast<uint64_t>(max_rows), d, BN / 2);
  if (e == cudaSuccess) e = make_map(&p->map_h, H, static_cast<uint64_t>(max_rows), f, BN / 2);
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
static void launch(const TcPlan* p, const CUtensorMap& map_x, const CUtensorMap& map_w,
                   const int32_t* offsets, int K, int N, void* out, cudaStream_t st,
                   int* status) {
  k_tc_gemm_pair<EPI><<<p->grid, 192, kPairSmem, st>>>(map_x, map_w, offsets, p->E, K, N, out,
                                                       status);
}

cudaError_t launch_tc_gateup(TcPlan* p, const void* x_perm, bool own_x_perm,
                             const int32_t* offsets, void* H, int n_rows, cudaStream_t st,
                             int* status) {
  if (p->q) return launch_tcq_gateup(p->q, x_perm, own_x_perm, offsets, H, n_rows, st, status);
  if (n_rows == 0) return cudaSuccess;
  CUtensorMap map_x;
  if (own_x_perm) {
    map_x = p->map_xperm;
  } else {
    const cudaError_t e = make_map(&map_x, x_perm, static_cast<uint64_t>(n_rows), p->d, BN / 2);
    if (e != cudaSuccess) return e;
  }
  launch<0>(p, map_x, p->map_wgu, offsets, p->d, 2 * p->f, H, st, status);
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
