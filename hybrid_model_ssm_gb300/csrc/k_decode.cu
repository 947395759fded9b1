// Instantiations of the decode-step kernel (non-flush and flush steps).
#include "rssm_launch.cuh"

namespace rssm {
cudaError_t launch_decode(const Params& p, int grid, size_t smem, cudaStream_t st, int N, int dtype, int rf) {
  if (rf == kDelta) return launch_delta(kDecode, p, grid, smem, st, N, dtype);
  return dtype == 0 ? dispatch_n<kDecode, float>(p, grid, smem, st, N, rf)
                    : dispatch_n<kDecode, __nv_bfloat16>(p, grid, smem, st, N, rf);
}
}  // namespace rssm
