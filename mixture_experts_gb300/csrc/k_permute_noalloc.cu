// coli_permute_noalloc: the dispatch stage for callers that cannot allocate
// device memory.
//
// coli_permute needs a small [blocks][E] table of device scratch once a
// batch has more than 16384 (token, expert) assignments, and leaves it to the
// caller to provide it. Some callers have no way to do that at the point of
// the call: a plugin running inside a host program whose device memory pool
// belongs to that program, or a real-time loop that is not allowed to
// allocate after start-up. This entry point takes the same inputs and
// outputs but keeps its scratch in a fixed array that lives in this library's
// device image, so it calls no cudaMalloc, no cudaFree and no allocating
// library routine.
#include <stdio.h>

#include <mutex>

#include "../../include/coli_moe.h"
#include "internal.h"

namespace {

// The scratch area: COLI_PERMUTE_STATIC_SCRATCH_BYTES of device memory that
// every GPU loading the library keeps until the process exits. All calls
// share it; the count kernel writes every table entry before the scan and
// scatter kernels read it, so nothing has to be cleared between calls. Two
// calls whose kernels overlap on a GPU would overwrite each other's table.
static __device__ __align__(256) int32_t g_permute_scratch[COLI_PERMUTE_STATIC_SCRATCH_BYTES / 4];

// The array's name in host code is only a host-side stand-in; kernels need
// its device address, taken once per device with that device current.
int scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return COLI_ECUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess || p == nullptr) return COLI_ECUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return COLI_OK;
}

int reject(int code, const char* msg) { return coli::record_error(code, msg); }

}  // namespace

extern "C" {

int coli_permute_noalloc(const int32_t* topk_idx, const void* x, int32_t T, int32_t d, int32_t E,
                         int32_t k, int32_t act, int32_t* counts, int32_t* offsets,
                         int32_t* row_token, int32_t* assign_row, void* x_perm, void* stream) {
  if (T < 0 || d <= 0 || d % 64 || E < 1 || E > 256 || k < 1 || k > E ||
      static_cast<long>(T) * k > (1L << 24)) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "bad sizes T=%d d=%d E=%d k=%d: need T >= 0, d a positive multiple of 64, "
             "1 <= E <= 256, 1 <= k <= E and T*k <= 16777216",
             T, d, E, k);
    return reject(COLI_EINVAL, msg);
  }
  if (act != COLI_F32 && act != COLI_BF16) return reject(COLI_EINVAL, "bad act dtype");
  const size_t need = coli::permute_scratch_bytes(T, k, E);
  if (need > COLI_PERMUTE_STATIC_SCRATCH_BYTES) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "T*k=%ld with E=%d needs %zu bytes of scratch, more than the %d-byte static "
             "area; call coli_permute with caller-provided scratch instead",
             static_cast<long>(T) * k, E, need, COLI_PERMUTE_STATIC_SCRATCH_BYTES);
    return reject(COLI_EINVAL, msg);
  }
  if (!topk_idx || !counts || !offsets || !row_token || !assign_row)
    return reject(COLI_EINVAL, "topk_idx, counts, offsets, row_token, assign_row must be set");
  if (x_perm != nullptr &&
      (x == nullptr || (reinterpret_cast<uintptr_t>(x) & 15u) ||
       (reinterpret_cast<uintptr_t>(x_perm) & 15u)))
    return reject(COLI_EINVAL, "x and x_perm must be set and 16-byte aligned");
  // every call resolves the address (only the first call on a device does
  // the lookup), even when this batch needs no scratch
  void* scratch = nullptr;
  if (scratch_address(&scratch) != COLI_OK)
    return reject(COLI_ECUDA, "cudaGetSymbolAddress of the static scratch area failed");
  const cudaError_t e = coli::launch_permute(
      topk_idx, x, T, d, E, k, act, counts, offsets, row_token, assign_row, x_perm, scratch,
      static_cast<cudaStream_t>(stream), coli::device_status_ptr(), nullptr);
  if (e != cudaSuccess) return reject(COLI_ECUDA, cudaGetErrorString(e));
  return COLI_OK;
}

}  // extern "C"
