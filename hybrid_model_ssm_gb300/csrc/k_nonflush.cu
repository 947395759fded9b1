// k_nonflush.cu - instantiations of the warp-per-head non-flush decode step.
#include "rssm_launch.cuh"
#include "rssm_nonflush.cuh"

namespace rssm {

template <int N, typename TIn, int RF>
cudaError_t launch_nf_one(const Params& p, const NfStage& sg, int grid, int warps, size_t smem, cudaStream_t st) {
  auto kern = nonflush_kernel<N, TIn, RF>;
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
  cfg.blockDim = dim3(warps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p, sg);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename TIn>
cudaError_t nf_dispatch(const Params& p, const NfStage& sg, int grid, int warps, size_t smem, cudaStream_t st, int N,
                        int rf) {
  if (N == 64) {
    if (rf == kRfE4m3) return launch_nf_one<64, TIn, kRfE4m3>(p, sg, grid, warps, smem, st);
    if (rf == kRfE2m1) return launch_nf_one<64, TIn, kRfE2m1>(p, sg, grid, warps, smem, st);
    if (rf == kCkF16) return launch_nf_one<64, TIn, kCkF16>(p, sg, grid, warps, smem, st);
  } else if (N == 128) {
    if (rf == kRfE4m3) return launch_nf_one<128, TIn, kRfE4m3>(p, sg, grid, warps, smem, st);
    if (rf == kRfE2m1) return launch_nf_one<128, TIn, kRfE2m1>(p, sg, grid, warps, smem, st);
    if (rf == kCkF16) return launch_nf_one<128, TIn, kCkF16>(p, sg, grid, warps, smem, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_nonflush(const Params& p, const NfStage& sg, int grid, int warps, size_t smem, cudaStream_t st,
                            int N, int dtype, int rf) {
  return dtype == 0 ? nf_dispatch<float>(p, sg, grid, warps, smem, st, N, rf)
                    : nf_dispatch<__nv_bfloat16>(p, sg, grid, warps, smem, st, N, rf);
}

}  // namespace rssm
