// Split-KV combine kernel ("用 TileLang 编写高性能 DeepSeek MLA 内核…", section
// Combine Kernel), launched after the split kernel when the split kernel does not
// combine itself.  Sequences with one split were finished by the split kernel and
// are skipped.  Grid (b, ceil(h / 32), 4): one CTA per sequence, 32-row group and
// quarter of the 512 columns; 4 warps of 32 columns each (combine_block).
#include <stdint.h>

#include "combine.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

constexpr int kWarps = 4;

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
combine_kernel(FwdArgs a) {
  // launched with programmatic stream serialisation: the split kernel's partials
  // are read only once it has completed
  sm100::grid_dependency_wait();
  sm100::launch_dependents();
  const int seq = blockIdx.x;
  const int s0 = a.num_splits[seq];
  const int n = a.num_splits[seq + 1] - s0;
  if (n <= 1) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ uint4 tile[kWarps][32][4];  // [warp][row][16-B piece, swizzled]
  combine_block<T>(a, seq, s0, n, blockIdx.y * 32, 32 * blockIdx.z + kCombineChunks * warp, tile[warp], lane);
}

}  // namespace

cudaError_t launch_combine(const FwdArgs &a, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.b, (a.h + 31) / 32, 4);
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // e4m3 inputs give bf16 outputs
  return a.dtype == MLA_DTYPE_FP16 ? cudaLaunchKernelEx(&cfg, combine_kernel<__half>, a)
                                   : cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16>, a);
}

}  // namespace mla
