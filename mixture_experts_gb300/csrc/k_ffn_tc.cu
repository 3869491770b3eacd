// A3, prefill path: TMA + tcgen05/TMEM grouped GEMM (placeholder until the
// kernel lands; tc_supported() reports false so the decode kernels run).
#include "internal.h"

namespace coli {

struct TcPlan {};

bool tc_supported(int, int) { return false; }

cudaError_t tc_plan_create(TcPlan** plan, const void*, const void*, int, int, int, int) {
  *plan = nullptr;
  return cudaErrorNotSupported;
}

void tc_plan_destroy(TcPlan* plan) { delete plan; }

cudaError_t launch_tc_gateup(TcPlan*, const void*, const int32_t*, void*, int, cudaStream_t,
                             int*) {
  return cudaErrorNotSupported;
}

cudaError_t launch_tc_down(TcPlan*, const void*, const int32_t*, float*, int, cudaStream_t, int*) {
  return cudaErrorNotSupported;
}

}  // namespace coli
