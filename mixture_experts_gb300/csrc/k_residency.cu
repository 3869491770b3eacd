// Expert residency tier: all experts live in pinned host memory (Grace
// LPDDR on a GB300 node, reached from the GPU over NVLink-C2C) and a hot set
// of S of them also lives in HBM slots. The deep-dive page (wth2jhl.online,
// sections 3.1 and 4.2) describes the tiers, a hot set picked from routing
// history and a bounded look-ahead prefetch; its section 8.1 notes that
// placement does not change the results.
//
// Here the decode kernels address every expert through a per-expert pointer
// table, so an expert in a slot is read from HBM and any other one is
// streamed straight from host memory over C2C. After each forward a
// one-block policy kernel updates each expert's routing score
// (score = 0.75 * score + rows this forward), ranks the experts by score
// (ties: lower index), and promotes at most P of the top-S experts that are
// not resident, most popular first, into the slots of resident experts that
// left the top S (least popular first; empty slots first of all). It
// repoints the tables and writes a copy list that a grid-wide copy kernel
// then executes (host -> slot). Everything runs on the forward's stream: the
// next forward's FFN sees the new tables only after the copies, and nothing
// synchronises the host or allocates.
#include "common.cuh"
#include "internal.h"

namespace coli {
namespace {

constexpr int kMaxE = 256;

__global__ void __launch_bounds__(kMaxE)
    k_residency_policy(const int32_t* __restrict__ counts, int E, int S, int P, ResidencyState R) {
  __shared__ float sc[kMaxE];
  __shared__ int by_rank[kMaxE];
  const int e = threadIdx.x;
  if (e < E) {
    const float v = 0.75f * R.score[e] + static_cast<float>(counts[e]);
    R.score[e] = v;
    sc[e] = v;
  }
  __syncthreads();
  if (e < E) {
    int rank = 0;
    for (int o = 0; o < E; ++o)
      if (sc[o] > sc[e] || (sc[o] == sc[e] && o < e)) ++rank;
    by_rank[rank] = e;
  }
  __syncthreads();
  if (e != 0) return;
  // one thread walks the ranking: promotions from the top, victims from the
  // bottom (slots whose expert fell out of the top S), empty slots first
  int n = 0;
  int victim_pos = E - 1;
  int empty = 0;
  for (int r = 0; r < S && r < E && n < P; ++r) {
    const int x = by_rank[r];
    if (R.slot_of[x] >= 0) continue;           // already resident
    int slot = -1;
    while (empty < S && slot < 0) {            // an unused slot
      if (R.expert_in[empty] < 0) slot = empty;
      ++empty;
    }
    while (slot < 0 && victim_pos >= S) {      // a resident expert outside the top S
      const int v = by_rank[victim_pos--];
      if (R.slot_of[v] >= 0) {
        slot = R.slot_of[v];
        R.slot_of[v] = -1;
        R.tab_gu[v] = R.host_gu + static_cast<size_t>(v) * R.gu_bytes;
        R.tab_dn[v] = R.host_dn + static_cast<size_t>(v) * R.dn_bytes;
        R.tab_sgu[v] = R.host_sgu + static_cast<size_t>(v) * R.sgu_bytes;
        R.tab_sdn[v] = R.host_sdn + static_cast<size_t>(v) * R.sdn_bytes;
      }
    }
    if (slot < 0) break;                       // every slot holds a top-S expert
    R.slot_of[x] = slot;
    R.expert_in[slot] = x;
    R.tab_gu[x] = R.slot_gu + static_cast<size_t>(slot) * R.gu_bytes;
    R.tab_dn[x] = R.slot_dn + static_cast<size_t>(slot) * R.dn_bytes;
    R.tab_sgu[x] = R.slot_sgu + static_cast<size_t>(slot) * R.sgu_bytes;
    R.tab_sdn[x] = R.slot_sdn + static_cast<size_t>(slot) * R.sdn_bytes;
    R.copy_list[2 * n] = x;
    R.copy_list[2 * n + 1] = slot;
    ++n;
  }
  *R.n_copy = n;
  *R.promotions += n;
}

// Copies the listed experts (gate/up, down and their scales) host -> slot,
// 16 bytes per thread and step over the concatenated ranges.
__global__ void __launch_bounds__(256) k_residency_copy(ResidencyState R) {
  const int n = *R.n_copy;
  const size_t parts[4] = {R.gu_bytes, R.dn_bytes, R.sgu_bytes, R.sdn_bytes};
  const size_t per_expert = (parts[0] + parts[1] + parts[2] + parts[3]) / 16;
  const size_t total = per_expert * n;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(i / per_expert);
    size_t off = (i % per_expert) * 16;
    const int x = R.copy_list[2 * j], slot = R.copy_list[2 * j + 1];
    const uint8_t* src;
    uint8_t* dst;
    if (off < parts[0]) {
      src = R.host_gu + static_cast<size_t>(x) * parts[0] + off;
      dst = R.slot_gu + static_cast<size_t>(slot) * parts[0] + off;
    } else if ((off -= parts[0]) < parts[1]) {
      src = R.host_dn + static_cast<size_t>(x) * parts[1] + off;
      dst = R.slot_dn + static_cast<size_t>(slot) * parts[1] + off;
    } else if ((off -= parts[1]) < parts[2]) {
      src = R.host_sgu + static_cast<size_t>(x) * parts[2] + off;
      dst = R.slot_sgu + static_cast<size_t>(slot) * parts[2] + off;
    } else {
      off -= parts[2];
      src = R.host_sdn + static_cast<size_t>(x) * parts[3] + off;
      dst = R.slot_sdn + static_cast<size_t>(slot) * parts[3] + off;
    }
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
}

}  // namespace

cudaError_t launch_residency_update(const int32_t* counts, int E, int S, int P,
                                    const ResidencyState& R, int grid, cudaStream_t st) {
  if (P <= 0) return cudaSuccess;
  k_residency_policy<<<1, kMaxE, 0, st>>>(counts, E, S, P, R);
  k_residency_copy<<<grid, 256, 0, st>>>(R);
  return cudaGetLastError();
}

}  // namespace coli
