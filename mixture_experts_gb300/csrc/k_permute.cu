// A2: dispatch — expert histogram, exclusive prefix, stable scatter, row copy.
//
// The counting sort of the discosf.com page (section 4.2: per-expert counts,
// offsets, groups of token indices) and the overview page's two-phase
// dispatch (trdm.cn, section 3.3: token-to-expert map plus per-expert
// offsets), kept entirely on the GPU. Assignments are taken in (token, slot)
// order; an assignment to expert e lands in row
//   offsets[e] + #{earlier assignments to e},
// so rows of one expert keep token order and every output is unique.
//
// Counts use shared-memory atomics (order-free, exact). Ranks never do:
// within a warp they come from __match_any_sync + popc of the lower lanes,
// across the warps of a tile from a per-expert prefix over warp order, and
// across tiles/blocks from running per-expert bases. Small batches
// (T*k <= kFusedMax) run in one block with no global scratch; larger ones
// use count / scan / scatter kernels with a [blocks][E] scratch table.
#include "common.cuh"
#include "internal.h"

namespace coli {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kFusedMax = 16384;  // assignments handled by the single-block kernel
constexpr int kChunk = 2048;      // assignments per block in the multi-block kernels
constexpr int kMaxE = 256;

COLI_DEV unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive scan of v over threads 0..255 (256-thread prefix of the block);
// every thread of the block must call it. Returns the exclusive prefix and
// writes the total to *total.
COLI_DEV int scan256(int v, int* sh /* >= 9 ints */, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  int x = (tid < kMaxE) ? v : 0;
  int inc = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += y;
  }
  if (tid < kMaxE && lane == 31) sh[w] = inc;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int i = 0; i < kMaxE / 32; ++i) {
      const int c = sh[i];
      sh[i] = run;
      run += c;
    }
    sh[8] = run;
  }
  __syncthreads();
  const int ex = (tid < kMaxE) ? sh[w] + inc - x : 0;
  *total = sh[8];
  __syncthreads();
  return ex;
}

// Stable scatter of assignments [a0, a1) given per-expert running bases in
// shared memory (base[e] = first free row of expert e for this range).
COLI_DEV void scatter_range(const int32_t* __restrict__ topk_idx, int a0, int a1, int E, int k,
                            int* base, int (*wcnt)[kMaxE], int* tot,
                            int32_t* __restrict__ row_token, int32_t* __restrict__ assign_row) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  for (int t0 = a0; t0 < a1; t0 += kThreads) {
    for (int i = tid; i < kWarps * E; i += kThreads) wcnt[i / E][i % E] = 0;
    __syncthreads();
    const int a = t0 + tid;
    int e = -1;
    if (a < a1) {
      const int v = topk_idx[a];
      if (v >= 0 && v < E) e = v;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lanemask_lt());
    if (e >= 0 && lane == __ffs(peers) - 1) wcnt[w][e] = __popc(peers);
    __syncthreads();
    if (tid < E) {
      int p = 0;
      for (int i = 0; i < kWarps; ++i) {
        const int c = wcnt[i][tid];
        wcnt[i][tid] = p;
        p += c;
      }
      tot[tid] = p;
    }
    __syncthreads();
    if (e >= 0) {
      const int row = base[e] + wcnt[w][e] + rank;
      row_token[row] = a / k;
      assign_row[a] = row;
    } else if (a < a1) {
      assign_row[a] = -1;  // skipped (bad id): a later combine adds nothing for it
    }
    __syncthreads();
    if (tid < E) base[tid] += tot[tid];
    __syncthreads();
  }
}

COLI_DEV void count_range(const int32_t* __restrict__ topk_idx, int a0, int a1, int E, int* hist,
                          int* status) {
  for (int a = a0 + threadIdx.x; a < a1; a += kThreads) {
    const int e = topk_idx[a];
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else latch_error(status, kErrDevice);
  }
}

__global__ void __launch_bounds__(kThreads)
    k_perm_fused(const int32_t* __restrict__ topk_idx, int n, int E, int k,
                 int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                 int32_t* __restrict__ row_token, int32_t* __restrict__ assign_row, int* status) {
  __shared__ int hist[kMaxE], base[kMaxE], tot[kMaxE], sh[9];
  __shared__ int wcnt[kWarps][kMaxE];
  const int tid = threadIdx.x;
  if (tid < kMaxE) hist[tid] = 0;
  __syncthreads();
  count_range(topk_idx, 0, n, E, hist, status);
  __syncthreads();
  int total;
  const int c = (tid < E) ? hist[tid] : 0;
  const int ex = scan256(c, sh, &total);
  if (tid < E) {
    counts[tid] = c;
    offsets[tid] = ex;
    base[tid] = ex;
  }
  if (tid == 0) offsets[E] = total;
  __syncthreads();
  scatter_range(topk_idx, 0, n, E, k, base, wcnt, tot, row_token, assign_row);
}

__global__ void __launch_bounds__(kThreads)
    k_perm_count(const int32_t* __restrict__ topk_idx, int n, int E,
                 int32_t* __restrict__ block_counts, int* status) {
  __shared__ int hist[kMaxE];
  const int tid = threadIdx.x;
  if (tid < kMaxE) hist[tid] = 0;
  __syncthreads();
  const int a0 = blockIdx.x * kChunk, a1 = min(n, a0 + kChunk);
  count_range(topk_idx, a0, a1, E, hist, status);
  __syncthreads();
  if (tid < E) block_counts[static_cast<size_t>(blockIdx.x) * E + tid] = hist[tid];
}

// One block: per-expert totals and offsets; block_counts[b][e] becomes the
// first row of expert e for block b.
__global__ void __launch_bounds__(kThreads)
    k_perm_scan(int32_t* __restrict__ block_counts, int nb, int E, int32_t* __restrict__ counts,
                int32_t* __restrict__ offsets) {
  __shared__ int sh[9];
  const int tid = threadIdx.x;
  int run = 0;
  if (tid < E) {
    for (int b = 0; b < nb; ++b) {
      int32_t* p = block_counts + static_cast<size_t>(b) * E + tid;
      const int c = *p;
      *p = run;
      run += c;
    }
  }
  int total;
  const int ex = scan256(tid < E ? run : 0, sh, &total);
  if (tid < E) {
    counts[tid] = run;
    offsets[tid] = ex;
    for (int b = 0; b < nb; ++b) block_counts[static_cast<size_t>(b) * E + tid] += ex;
  }
  if (tid == 0) offsets[E] = total;
}

__global__ void __launch_bounds__(kThreads)
    k_perm_scatter(const int32_t* __restrict__ topk_idx, int n, int E, int k,
                   const int32_t* __restrict__ block_base, int32_t* __restrict__ row_token,
                   int32_t* __restrict__ assign_row) {
  __shared__ int base[kMaxE], tot[kMaxE];
  __shared__ int wcnt[kWarps][kMaxE];
  const int tid = threadIdx.x;
  if (tid < E) base[tid] = block_base[static_cast<size_t>(blockIdx.x) * E + tid];
  __syncthreads();
  const int a0 = blockIdx.x * kChunk, a1 = min(n, a0 + kChunk);
  scatter_range(topk_idx, a0, a1, E, k, base, wcnt, tot, row_token, assign_row);
}

// x_perm[r] = x[row_token[r]], one warp per row, 16-byte vectors. Each token
// row is read k times, far apart in time (rows are in expert order), while
// the T*k-row copy streams through L2: the reads carry an L2 evict-last
// policy and the writes evict-first, so x stays in L2 and is read from DRAM
// about once.
__global__ void __launch_bounds__(256)
    k_gather_rows(const uint4* __restrict__ x, const int32_t* __restrict__ row_token, int n_rows,
                  int T, int vec_per_row, uint4* __restrict__ x_perm, int* status) {
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * 8;
  uint64_t keep, stream;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(stream));
  for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < n_rows; r += warps) {
    const int t = row_token[r];
    if (t < 0 || t >= T) {
      if (lane == 0) latch_error(status, kErrDevice);
      continue;
    }
    const uint4* src = x + static_cast<size_t>(t) * vec_per_row;
    uint4* dst = x_perm + static_cast<size_t>(r) * vec_per_row;
    // up to 8 vectors per lane in flight: all loads of a batch, then its stores
    constexpr int kBatch = 8;
    for (int v0 = 0; v0 < vec_per_row; v0 += 32 * kBatch) {
      uint4 u[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int v = v0 + 32 * b + lane;
        if (v < vec_per_row)
          asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                       : "=r"(u[b].x), "=r"(u[b].y), "=r"(u[b].z), "=r"(u[b].w)
                       : "l"(src + v), "l"(keep));
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int v = v0 + 32 * b + lane;
        if (v < vec_per_row)
          asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(dst + v),
                       "r"(u[b].x), "r"(u[b].y), "r"(u[b].z), "r"(u[b].w), "l"(stream)
                       : "memory");
      }
    }
  }
}

}  // namespace

size_t permute_scratch_bytes(int T, int k, int E) {
  const long n = static_cast<long>(T) * k;
  if (n <= kFusedMax) return 0;
  const size_t nb = static_cast<size_t>((n + kChunk - 1) / kChunk);
  return (nb * E * sizeof(int32_t) + 255) & ~static_cast<size_t>(255);
}

cudaError_t launch_permute(const int32_t* topk_idx, const void* x, int T, int d, int E, int k,
                           int act, int32_t* counts, int32_t* offsets, int32_t* row_token,
                           int32_t* assign_row, void* x_perm, void* scratch, cudaStream_t st,
                           int* status, int* n_launches) {
  const int n = T * k;
  int launches = 0;
  if (n <= kFusedMax) {
    k_perm_fused<<<1, kThreads, 0, st>>>(topk_idx, n, E, k, counts, offsets, row_token,
                                         assign_row, status);
    launches = 1;
  } else {
    const int nb = (n + kChunk - 1) / kChunk;
    int32_t* table = static_cast<int32_t*>(scratch);
    k_perm_count<<<nb, kThreads, 0, st>>>(topk_idx, n, E, table, status);
    k_perm_scan<<<1, kThreads, 0, st>>>(table, nb, E, counts, offsets);
    k_perm_scatter<<<nb, kThreads, 0, st>>>(topk_idx, n, E, k, table, row_token, assign_row);
    launches = 3;
  }
  if (x_perm != nullptr && n > 0) {
    const int esize = (act == DT_F32) ? 4 : 2;
    const int vec = d * esize / 16;
    int grid = (n + 7) / 8;
    if (grid > 4096) grid = 4096;
    k_gather_rows<<<grid, 256, 0, st>>>(static_cast<const uint4*>(x), row_token, n, T, vec,
                                        static_cast<uint4*>(x_perm), status);
    launches += 1;
  }
  if (n_launches) *n_launches += launches;
  return cudaGetLastError();
}

}  // namespace coli
