// attn_bwd.cu -- placeholder until the backward kernels land.
#include <cuda.h>
#include "common.cuh"
namespace ccg {
int bwd_kv_tile_rows(int D) { return D == 128 ? 128 : 64; }
int bwd_q_tile_rows(int) { return 128; }
int bwd_map_rows(int which, int D) { return which < 4 ? 128 : bwd_kv_tile_rows(D); }
cudaError_t launch_attn_bwd(const CUtensorMap*, const WorkItem*, const WorkItem*, const PlanHeader*,
                            const int32_t*, const int32_t*, const float*, const float*, void*, void*,
                            void*, int32_t*, int, int, int, int, int64_t, int, float, int, int, int*,
                            cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace ccg
