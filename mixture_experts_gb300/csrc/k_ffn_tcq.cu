// A3, prefill path for quantised experts (int4 groups of 128 with bf16
// scales; MXFP8 and MXFP4 with an E8M0 scale per 32): a grouped GEMM on the
// 5th-generation tensor cores with the weights as the tensor-memory operand.
//
// The expert weights arrive quantised, so every weight has to become bf16
// before the tensor core can multiply it, and that conversion, not the MMA,
// is what the kernel is built around. A tile is 128 weight rows x 256 token
// rows. Eight converter warps (two per lane quarter, alternate stages) turn
// the tile's 128 weight rows of each 64-index stage into bf16 pairs in
// registers and write them straight into tensor memory (tcgen05.st), where
// tcgen05.mma reads them as its A operand;
// TMA brings the 256 activation rows (bf16, 128-byte swizzle) into shared
// memory as the B operand; the fp32 accumulator D[weight row][token] takes
// 256 tensor-memory columns beside four 32-column A stages. Per stage the
// converters produce 8192 weights for 2.1 M multiply-adds (half the weights
// per MMA of a tile with 256 weight rows) and the converted operand never
// passes through shared memory.
//
// Raw weights come by TMA in slots of 128 bytes of every weight row (128-byte
// swizzle): one slot holds 256 reduction indices of int4 or E2M1 codes (four
// stages) or 128 of E4M3 codes (two). The MX bytes keep the decode layout:
// within each 128-index step the 8-index unit 4b + u (block b, quarter u) is
// stored at unit position 4u + b, so a stage's blocks 2h and 2h + 1 arrive as
// one 16-byte (E4M3) or 8-byte (E2M1) piece per quarter u whose halves are
// the stage's units u and 4 + u.
//
// Conversion. int4: 136 + q from the nibble (one LOP3 per pair), minus 136
// (exact), times the group scale: q * s rounded once to bf16. MX: every
// element is exact in bf16 (an E4M3 or E2M1 value times a
// power of two) unless the product leaves bf16's range. The hardware turns
// two codes into an fp16 pair; moving the fp16 exponent field into the low
// bits of the bf16 one gives the element times 2^-112 exactly (fp16 holds
// these values as normals, and the dropped mantissa bits are zero), and one
// bf16 multiply by 2^(s - 15) applies the block scale exactly. That factor is
// a bf16 normal for s <= 142 (scales up to 2^15); weights with larger scales,
// NaN scales or E4M3 NaN codes are converted through fp32 instead (one flag
// per layer, found when the layer is created).
//
// Grouping follows the bf16 kernel: each CTA derives the tile list from the
// device-side expert offsets (experts without rows contribute no tiles, so
// their weights are never read) and walks it with a stride of gridDim.x,
// consecutive tiles sharing a weight tile. An expert's last token tile runs
// its MMAs with N = its rows rounded up to 16, so a ragged tail costs what
// it holds; token columns past the expert's rows are not stored, and rows
// past the activation buffer are zero-filled by TMA.
//
// Epilogues (eight warps, two per lane quarter, 128 accumulator columns
// each: with one accumulator in tensor memory the next tile's MMAs wait for
// them). Gate/up: the weights are interleaved in blocks of 64 rows (gate
// rows of 64 features, then their up rows) and a tile is one block; the
// converters put the gate row of feature 16q + l in lane 32q + l and its up
// row in lane 32q + 16 + l, so each epilogue warp holds both halves of its 16
// features and one lane shuffle pairs them; h = silu(gate) * up goes to H
// [token][feature] in bf16. Down: lane = output column; y_perm rows in fp32
// or bf16. A store instruction writes 16 or 32 consecutive columns of a
// token row.
//
// Every mbarrier wait is bounded by one kernel-wide deadline; a CTA that
// reaches it latches COLI_ETIMEOUT, unwinds all roles, waits briefly for
// copies in flight, frees its tensor memory and returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace coli {

struct QPlan {
  CUtensorMap map_x, map_h, map_wgu, map_wdn;  // activations x_perm / H; raw weights
  const void *s_gu, *s_dn;                     // scales
  int wdt, E, d, f, grid, general;
};

namespace {

constexpr int TM = 128;                   // weight rows per tile (A rows, tensor-memory lanes)
constexpr int TN = 256;                   // token rows per tile (B rows, the MMA's N)
constexpr int BK = 64;                    // reduction indices per stage
constexpr int STAGES = 4;
constexpr int XB_BYTES = TN * BK * 2;     // 32 KiB of activations per stage
constexpr int RAW_ROW = 128;              // raw weight bytes per row and slot
constexpr int SLOT_BYTES = TM * RAW_ROW;  // 16 KiB
constexpr int SLOTS = 3;
constexpr int D_COL = 0;                  // accumulator: 256 fp32 columns
constexpr int A_COL = 256;                // A stages: BK / 2 columns of bf16 pairs each
constexpr int TMEM_COLS = 512;
constexpr int kEpiWarps = 8;             // two per lane quarter, half the columns each
constexpr int kConvWarps = 8;            // two per lane quarter, alternate stages
constexpr int kThreads = 32 * (2 + kEpiWarps + kConvWarps);  // 0 TMA, 1 MMA, epilogue, converters
constexpr int kConv0 = 2 + kEpiWarps;     // first converter warp
constexpr int kMaxE = 256;

// stages per raw slot: 128 bytes of a row are 128 E4M3 codes or 256 4-bit ones
template <int WQ>
constexpr int kSubs = WQ == DT_MXFP8 ? 2 : 4;

struct __align__(8) Ctrl {
  uint64_t full[STAGES], empty[STAGES], rawfull[SLOTS], rawempty[SLOTS], tfull, tempty;
  uint32_t tmem_base;
  int abort;
  int tile_off[kMaxE + 1];  // first tile of expert e
  int row_off[kMaxE + 1];   // first token row of expert e (the offsets)
};

constexpr size_t kSmem = 1024 + STAGES * XB_BYTES + SLOTS * SLOT_BYTES + sizeof(Ctrl);

struct QArgs {
  const void* scales;  // int4: bf16 [weight rows][K/128]; MX: E8M0 bytes [weight rows][K/32]
  int total_rows;      // weight rows in the tensor (E x rows per expert)
  int general;         // MX: convert through fp32 (NaN codes or scales beyond 2^15 present)
};

struct Tile {
  int e, wt, mt;  // expert, weight tile, token tile
};

COLI_DEV Tile decode_tile(const Ctrl& C, int E, int t) {
  int lo = 0, hi = E;  // tile_off[lo] <= t < tile_off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (C.tile_off[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int rows = C.row_off[lo + 1] - C.row_off[lo];
  const int mts = (rows + TN - 1) / TN;
  const int local = t - C.tile_off[lo];
  return Tile{lo, local / mts, local % mts};
}

// Row of the tile's 128 weight rows held in tensor-memory lane 32q + l.
template <int EPI>
COLI_DEV int lane_row(int q, int l) {
  if constexpr (EPI == 0) return l < 16 ? 16 * q + l : 64 + 16 * q + (l - 16);
  return 32 * q + l;
}

// One weight row's scales for raw slot `slot`, as two words: int4: the bf16
// pairs (s, s) of the slot's two 128-index groups; MXFP8: the slot's four
// E8M0 bytes; MXFP4: its eight. Zero past the tensor or the row.
template <int WQ>
COLI_DEV void slot_scales(const QArgs& q, int row, int K, int slot, uint32_t (&s)[2]) {
  s[0] = s[1] = 0u;
  if (row >= q.total_rows) return;
  if constexpr (WQ == DT_I4G128) {
    const int G = K / 128;
    const unsigned short* p =
        static_cast<const unsigned short*>(q.scales) + static_cast<size_t>(row) * G;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int g = 2 * slot + i;
      if (g < G) {
        const uint32_t v = __ldg(p + g);
        s[i] = v | (v << 16);
      }
    }
  } else {
    const int W = K / 128;  // scale words per row
    const uint32_t* p = reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(q.scales) +
                                                          static_cast<size_t>(row) * (K / 32));
    constexpr int NW = WQ == DT_MXFP8 ? 1 : 2;
#pragma unroll
    for (int i = 0; i < NW; ++i)
      if (NW * slot + i < W) s[i] = __ldg(p + NW * slot + i);
  }
}

// 2^(s - 127) in fp32 (s = 255: NaN).
COLI_DEV float e8m0_f32(uint32_t s) {
  if (s == 255u) return __uint_as_float(0x7fc00000u);
  return s == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(s << 23);
}

// Four fp16 pairs of one MX unit times the block scale 2^(s - 127) -> bf16
// pairs o[0..3].
template <bool GENERAL>
COLI_DEV void mx_unit(const uint32_t (&f)[4], uint32_t s, uint32_t* o) {
  if constexpr (!GENERAL) {
    const uint32_t fac = ((s + 112u) << 7) * 0x00010001u;  // bf16 pair (2^(s-15), 2^(s-15))
#pragma unroll
    for (int p = 0; p < 4; ++p)
      o[p] = fma_bf16x2(((f[p] & 0x7fff7fffu) >> 3) | (f[p] & 0x80008000u), fac, 0x80008000u);
  } else {
    const float sc = e8m0_f32(s);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&f[p]));
      o[p] = pack_bf16x2(v.x * sc, v.y * sc);
    }
  }
}

// One converter thread: stage `sub` of the raw slot row at `rowp` (raw row
// rr of the tile, 128-byte swizzled: 16-byte chunk c at chunk c ^ (rr % 8))
// -> 32 bf16 pairs, reduction indices 2i and 2i + 1 of the stage in o[i].
template <int WQ, bool GENERAL>
COLI_DEV void convert_stage(uint32_t rowp, int rr, int sub, const uint32_t (&sc)[2],
                            uint32_t (&o)[32]) {
  if constexpr (WQ == DT_I4G128) {
    // 32 bytes = 64 indices; words hold indices 8w..8w+7, pairs by nib_pair136
    constexpr uint32_t kOne = 0x3f803f80u, kMinus136 = 0xc308c308u, kMinusZero = 0x80008000u;
    const uint32_t s2 = sc[sub >> 1];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const uint4 v = lds128(rowp + (((2 * sub + cc) ^ (rr & 7)) << 4));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w = word_of(v, i);
#pragma unroll
        for (int p = 0; p < 4; ++p)
          o[16 * cc + 4 * i + p] =
              fma_bf16x2(fma_bf16x2(nib_pair136(w, p), kOne, kMinus136), s2, kMinusZero);
      }
    }
  } else if constexpr (WQ == DT_MXFP8) {
    const int h = sub;  // half of the slot's 128-index step
    const uint32_t s0 = (sc[0] >> (16 * h)) & 0xffu, s1 = (sc[0] >> (16 * h + 8)) & 0xffu;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint4 v = lds128(rowp + (((2 * u + h) ^ (rr & 7)) << 4));
      uint32_t f0[4], f1[4];
      e4m3x8_f16(v.x, v.y, f0);  // unit u of block 2h
      e4m3x8_f16(v.z, v.w, f1);  // unit u of block 2h + 1
      mx_unit<GENERAL>(f0, s0, &o[4 * u]);
      mx_unit<GENERAL>(f1, s1, &o[16 + 4 * u]);
    }
  } else {  // DT_MXFP4: two 128-index steps per slot
    const int step = sub >> 1, h = sub & 1;
    const uint32_t w = sc[step];
    const uint32_t s0 = (w >> (16 * h)) & 0xffu, s1 = (w >> (16 * h + 8)) & 0xffu;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint2 v = lds64(rowp + (((4 * step + u) ^ (rr & 7)) << 4) + 8 * h);
      uint32_t f0[4], f1[4];
      e2m1x8_f16(v.x, f0);
      e2m1x8_f16(v.y, f1);
      mx_unit<GENERAL>(f0, s0, &o[4 * u]);
      mx_unit<GENERAL>(f1, s1, &o[16 + 4 * u]);
    }
  }
}

// EPI 0: gate/up + SwiGLU -> bf16 H [rows][N/2]; EPI 1: fp32 out [rows][N];
// EPI 2: bf16 out [rows][N]. map_w: the raw weight bytes [E*N][row bytes],
// box 128 rows x 128 bytes; map_x: bf16 activations [rows][K], box 256 x 64.
template <int EPI, int WQ>
__global__ void __launch_bounds__(kThreads, 1)
    k_tcq_gemm(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
               const int32_t* __restrict__ offsets, int E, int K, int N, void* __restrict__ out,
               QArgs qa, int* status) {
  constexpr int SUBS = kSubs<WQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sx = smem_u32(base);
  const uint32_t sraw = sx + STAGES * XB_BYTES;
  Ctrl& C = *reinterpret_cast<Ctrl*>(base + STAGES * XB_BYTES + SLOTS * SLOT_BYTES);
  volatile int* abort = &C.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t deadline = global_timer_ns() + kWaitTimeoutNs;
  const int n_wt = N / TM;  // weight tiles per expert
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
        m = ((r1 - r0 + TN - 1) / TN) * n_wt;
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
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(smem_u32(&C.full[s]), 5);  // the producer's expect_tx + four converter warps
        mbar_init(smem_u32(&C.empty[s]), 1);
      }
      for (int s = 0; s < SLOTS; ++s) {
        mbar_init(smem_u32(&C.rawfull[s]), 1);
        mbar_init(smem_u32(&C.rawempty[s]), kConvWarps);
      }
      mbar_init(smem_u32(&C.tfull), 1);
      mbar_init(smem_u32(&C.tempty), kEpiWarps);
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
    if (lane == 0) {  // ---- TMA producer: raw weight slots and activation stages
      int stage = 0, slot = 0;
      uint32_t phase = 0, sphase = 0;
      for (int t = blockIdx.x; t < total && !*abort; t += gridDim.x) {
        const Tile tl = decode_tile(C, E, t);
        const int w_row = tl.e * N + tl.wt * TM;
        const int x_row = C.row_off[tl.e] + tl.mt * TN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (kb % SUBS == 0) {
            if (!wait_bar(smem_u32(&C.rawempty[slot]), sphase ^ 1u, deadline, abort)) break;
            const uint32_t rb = smem_u32(&C.rawfull[slot]);
            mbar_arrive_expect_tx(rb, SLOT_BYTES);
            tma_load_2d(sraw + slot * SLOT_BYTES, &map_w, rb, (kb / SUBS) * RAW_ROW, w_row);
            if (++slot == SLOTS) {
              slot = 0;
              sphase ^= 1u;
            }
          }
          if (!wait_bar(smem_u32(&C.empty[stage]), phase ^ 1u, deadline, abort)) break;
          const uint32_t fb = smem_u32(&C.full[stage]);
          mbar_arrive_expect_tx(fb, XB_BYTES);
          tma_load_2d(sx + stage * XB_BYTES, &map_x, fb, kb * BK, x_row);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer: D (+)= A[tmem] x B[smem]^T
      int stage = 0, local = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < total && !*abort; t += gridDim.x, ++local) {
        if (!wait_bar(smem_u32(&C.tempty), (local & 1) ^ 1u, deadline, abort)) break;
        tc_fence_after();
        // the MMA's N covers the tile's token rows, rounded up to 16: an
        // expert's last, partial tile costs what it holds
        const Tile tl = decode_tile(C, E, t);
        const int rows = min(TN, C.row_off[tl.e + 1] - C.row_off[tl.e] - tl.mt * TN);
        const uint32_t idesc = idesc_bf16(TM, (rows + 15) & ~15);
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bar(smem_u32(&C.full[stage]), phase, deadline, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = tmem + A_COL + stage * (BK / 2);
          const uint32_t b0 = sx + stage * XB_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_ts(tmem + D_COL, a0 + k * 8, sw128_desc(b0 + k * 32), idesc,
                    (kb | k) != 0 ? 1u : 0u);
          umma_commit(smem_u32(&C.empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&C.tfull));
      }
    }
  } else if (warp < kConv0) {  // ---- epilogue: lanes 32*(warp%4) .., columns of one half
    const int q = warp & 3;
    const int c0 = ((warp - 2) >> 2) * (TN / 64);  // first 32-column chunk of this warp's half
    const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + D_COL;
    int local = 0;
    for (int t = blockIdx.x; t < total && !*abort; t += gridDim.x, ++local) {
      // warp-uniform verdict: tcgen05.ld below is warp-collective
      if (!__all_sync(0xffffffffu, wait_bar(smem_u32(&C.tfull), local & 1, deadline, abort)))
        break;
      tc_fence_after();
      const Tile tl = decode_tile(C, E, t);
      const int tok0 = C.row_off[tl.e] + tl.mt * TN;
      const int tok_end = C.row_off[tl.e + 1];
      if constexpr (EPI == 0) {
        const int F = N / 2;
        __nv_bfloat16* H = static_cast<__nv_bfloat16*>(out);
        const bool up = lane >= 16;
        const int feat = tl.wt * (TM / 2) + 16 * q + (lane & 15);
#pragma unroll 1
        for (int c = c0; c < c0 + TN / 64; ++c) {
          const int t0 = tok0 + 32 * c;
          if (t0 >= tok_end) break;
          uint32_t v[32];
          tmem_ld32(taddr + 32 * c, v);
          // gate lanes finish tokens 0..15 of the chunk, up lanes 16..31
          // (silu with the fast exponential and division: h is rounded to
          // bf16, far coarser than their few-ulp error)
          const int tb = t0 + (up ? 16 : 0);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, up ? v[j] : v[16 + j], 16);
            const float g = __uint_as_float(up ? recv : v[j]);
            const float u = __uint_as_float(up ? v[16 + j] : recv);
            if (tb + j < tok_end)
              H[static_cast<size_t>(tb + j) * F + feat] =
                  __float2bfloat16_rn(__fdividef(g, 1.f + __expf(-g)) * u);
          }
        }
      } else {
        const int col = tl.wt * TM + 32 * q + lane;
#pragma unroll 1
        for (int c = c0; c < c0 + TN / 64; ++c) {
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
              static_cast<__nv_bfloat16*>(out)[at] = __float2bfloat16_rn(__uint_as_float(v[j]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&C.tempty));
    }
  } else {  // ---- converters: the last eight warps, weights -> bf16 A operand in tensor memory
    // two warps per lane quarter take alternate stages, so one's conversion
    // overlaps the other's tensor-memory store and barrier round trip
    const int q = warp & 3;
    const int g = (warp - kConv0) >> 2;  // stage parity this warp converts
    const int rr = lane_row<EPI>(q, lane);
    const uint32_t a_lane = tmem + (static_cast<uint32_t>(32 * q) << 16) + A_COL;
    int stage = 0, slot = 0;
    uint32_t phase = 0, sphase = 0;
    for (int t = blockIdx.x; t < total && !*abort; t += gridDim.x) {
      const Tile tl = decode_tile(C, E, t);
      const int row = tl.e * N + tl.wt * TM + rr;
      // this slot's scales, and the next slot's requested a slot ahead
      uint32_t sc[2], scn[2];
      slot_scales<WQ>(qa, row, K, 0, sc);
      slot_scales<WQ>(qa, row, K, 1, scn);
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        const int sub = kb % SUBS;
        const bool last = sub == SUBS - 1 || kb == kblocks - 1;  // the slot's last stage
        if (sub == 0 && kb > 0) {
          sc[0] = scn[0];
          sc[1] = scn[1];
          slot_scales<WQ>(qa, row, K, kb / SUBS + 1, scn);
        }
        if ((stage & 1) == g) {
          // the A stage is free once the MMA that read it completed; the raw
          // slot holds this stage's weights
          if (!__all_sync(0xffffffffu,
                          wait_bar(smem_u32(&C.empty[stage]), phase ^ 1u, deadline, abort) &&
                              wait_bar(smem_u32(&C.rawfull[slot]), sphase, deadline, abort))) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t o[32];
          const uint32_t rowp = sraw + slot * SLOT_BYTES + rr * RAW_ROW;
          if (qa.general) convert_stage<WQ, true>(rowp, rr, sub, sc, o);
          else convert_stage<WQ, false>(rowp, rr, sub, sc, o);
          tmem_st32(a_lane + stage * (BK / 2), o);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&C.full[stage]));
        } else if (last) {
          // a slot whose stages are all the other warp's: its release below
          // must still come after the slot's data arrived (so it counts for
          // this fill of the buffer, not the previous one)
          if (!__all_sync(0xffffffffu,
                          wait_bar(smem_u32(&C.rawfull[slot]), sphase, deadline, abort))) {
            ok = false;
            break;
          }
        }
        if (last) {
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&C.rawempty[slot]));
          if (++slot == SLOTS) {
            slot = 0;
            sphase ^= 1u;
          }
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
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

template <int EPI, int WQ>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(k_tcq_gemm<EPI, WQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kSmem));
}

template <int WQ>
cudaError_t set_smem_all() {
  cudaError_t e = set_smem<0, WQ>();
  if (e == cudaSuccess) e = set_smem<1, WQ>();
  if (e == cudaSuccess) e = set_smem<2, WQ>();
  return e;
}

template <int EPI, int WQ>
void launch_one(const QPlan* p, const CUtensorMap& map_x, const CUtensorMap& map_w,
                const int32_t* offsets, int K, int N, void* out, const QArgs& qa,
                cudaStream_t st, int* status) {
  k_tcq_gemm<EPI, WQ><<<p->grid, kThreads, kSmem, st>>>(map_x, map_w, offsets, p->E, K, N, out,
                                                        qa, status);
}

template <int EPI>
void launch_fmt(const QPlan* p, const CUtensorMap& map_x, const CUtensorMap& map_w,
                const int32_t* offsets, int K, int N, void* out, const QArgs& qa,
                cudaStream_t st, int* status) {
  if (p->wdt == DT_I4G128)
    launch_one<EPI, DT_I4G128>(p, map_x, map_w, offsets, K, N, out, qa, st, status);
  else if (p->wdt == DT_MXFP8)
    launch_one<EPI, DT_MXFP8>(p, map_x, map_w, offsets, K, N, out, qa, st, status);
  else
    launch_one<EPI, DT_MXFP4>(p, map_x, map_w, offsets, K, N, out, qa, st, status);
}

// bf16 [rows][cols], box 256 rows x 64 columns, 128-byte swizzle.
cudaError_t map_act(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols) {
  return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, rows, cols, BK, TN,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

// raw weight bytes [rows][row_bytes], box 128 rows x 128 bytes, 128-byte swizzle.
cudaError_t map_raw(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t row_bytes) {
  return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, ptr, rows, row_bytes, RAW_ROW, TM,
                        CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

bool tcq_supported(int wdt, int d, int f) {
  if (wdt != DT_I4G128 && wdt != DT_MXFP8 && wdt != DT_MXFP4) return false;
  // a weight row must fill the 128-byte box: 4-bit rows need K >= 256
  const int min_k = wdt == DT_MXFP8 ? 128 : 256;
  return d % 128 == 0 && f % 128 == 0 && d >= min_k && f >= min_k;
}

cudaError_t tcq_plan_create(QPlan** plan, int wdt, const void* w_gu, const void* w_dn,
                            const void* s_gu, const void* s_dn, int E, int d, int f,
                            int max_rows, const void* x_perm, const void* H, bool general) {
  *plan = nullptr;
  QPlan* p = new QPlan();
  p->wdt = wdt;
  p->E = E;
  p->d = d;
  p->f = f;
  p->s_gu = s_gu;
  p->s_dn = s_dn;
  p->general = general ? 1 : 0;
  int dev = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&p->grid, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
    delete p;
    return e;
  }
  const uint64_t per_byte = wdt == DT_MXFP8 ? 1 : 2;  // elements per byte
  e = map_raw(&p->map_wgu, w_gu, static_cast<uint64_t>(E) * 2 * f, d / per_byte);
  if (e == cudaSuccess) e = map_raw(&p->map_wdn, w_dn, static_cast<uint64_t>(E) * d, f / per_byte);
  if (e == cudaSuccess) e = map_act(&p->map_x, x_perm, static_cast<uint64_t>(max_rows), d);
  if (e == cudaSuccess) e = map_act(&p->map_h, H, static_cast<uint64_t>(max_rows), f);
  if (e == cudaSuccess)
    e = wdt == DT_I4G128 ? set_smem_all<DT_I4G128>()
                         : (wdt == DT_MXFP8 ? set_smem_all<DT_MXFP8>() : set_smem_all<DT_MXFP4>());
  if (e != cudaSuccess) {
    delete p;
    return e;
  }
  *plan = p;
  return cudaSuccess;
}

void tcq_plan_destroy(QPlan* plan) { delete plan; }

cudaError_t launch_tcq_gateup(QPlan* p, const void* x_perm, bool own_x_perm,
                              const int32_t* offsets, void* H, int n_rows, cudaStream_t st,
                              int* status) {
  if (n_rows == 0) return cudaSuccess;
  CUtensorMap map_x;
  if (own_x_perm) {
    map_x = p->map_x;
  } else {
    const cudaError_t e = map_act(&map_x, x_perm, static_cast<uint64_t>(n_rows), p->d);
    if (e != cudaSuccess) return e;
  }
  const QArgs qa{p->s_gu, p->E * 2 * p->f, p->general};
  launch_fmt<0>(p, map_x, p->map_wgu, offsets, p->d, 2 * p->f, H, qa, st, status);
  return cudaGetLastError();
}

cudaError_t launch_tcq_down(QPlan* p, const int32_t* offsets, void* y_perm, bool bf16_out,
                            int n_rows, cudaStream_t st, int* status) {
  if (n_rows == 0) return cudaSuccess;
  const QArgs qa{p->s_dn, p->E * p->d, p->general};
  if (bf16_out)
    launch_fmt<2>(p, p->map_h, p->map_wdn, offsets, p->f, p->d, y_perm, qa, st, status);
  else
    launch_fmt<1>(p, p->map_h, p->map_wdn, offsets, p->f, p->d, y_perm, qa, st, status);
  return cudaGetLastError();
}

}  // namespace coli
