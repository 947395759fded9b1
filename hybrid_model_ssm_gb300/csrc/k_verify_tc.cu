// Instantiations of the tensor-core verify kernel (bf16 inputs, FP32 checkpoint;
// N in {64, 128}; P in {32, 64, 128}, so that 128 rows hold whole heads).
#include "rssm_launch.cuh"
#include "rssm_verify_tc.cuh"

namespace rssm {

template <int N, int P>
static cudaError_t launch_tc_one(const TcParams& p, const CUtensorMap& tmap, int grid, size_t smem, cudaStream_t st) {
  auto kern = verify_tc_kernel<N, P>;
  static bool attr_set = false;  // one GPU per process: set the opt-in size once
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p, tmap);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_verify_tc(const TcParams& p, const CUtensorMap& tmap, int grid, size_t smem, cudaStream_t st,
                             int N, int P) {
  if (N == 128) {
    if (P == 64) return launch_tc_one<128, 64>(p, tmap, grid, smem, st);
    if (P == 128) return launch_tc_one<128, 128>(p, tmap, grid, smem, st);
    if (P == 32) return launch_tc_one<128, 32>(p, tmap, grid, smem, st);
  } else if (N == 64) {
    if (P == 64) return launch_tc_one<64, 64>(p, tmap, grid, smem, st);
    if (P == 128) return launch_tc_one<64, 128>(p, tmap, grid, smem, st);
    if (P == 32) return launch_tc_one<64, 32>(p, tmap, grid, smem, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace rssm
