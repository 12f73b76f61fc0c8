// q4mm_tc.cu — tensor-core path (not built yet: every entry reports unsupported).
#include "q4mm_internal.h"

namespace q4 {
bool tc_kernel_built() { return false; }
TcPlan tc_plan(const Weight*, int64_t, int, bool) { return TcPlan{1, 1, 16}; }
size_t tc_partial_bytes(const Weight*, const TcPlan&, int64_t) { return 0; }
size_t tc_xop_bytes(const Weight*, const TcPlan&, int64_t) { return 0; }
int tc_launch_count(const TcPlan&, int64_t) { return 0; }
int launch_tc(const Weight*, const float*, int64_t, float*, int32_t*, float*, const TcPlan&,
              const Workspace&, cudaStream_t) {
  return Q4_ERR_UNSUPPORTED;
}
}  // namespace q4
