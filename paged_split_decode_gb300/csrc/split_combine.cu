// split_combine.cu -- launches the split-combine kernel of the balanced and
// fixed split modes right behind the decode kernel, with programmatic
// dependent launch so that its CTAs are scheduled while the decode grid drains.
#include "launch.h"

namespace pd {

cudaError_t launch_split_combine(int D, const DecodeParams& p, int n_units, int dim_chunks, int batch,
                                 int threads, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n_units), static_cast<unsigned>(dim_chunks),
                     static_cast<unsigned>(p.hg));
  const bool wide = batch > 4, big = wide && threads > 256;
  cfg.blockDim = dim3(big ? 512 : 256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (D == 128)
    e = big    ? cudaLaunchKernelEx(&cfg, split_combine_kernel<128, 8, 512>, p)
        : wide ? cudaLaunchKernelEx(&cfg, split_combine_kernel<128, 8, 256>, p)
               : cudaLaunchKernelEx(&cfg, split_combine_kernel<128, 4, 256>, p);
  else
    e = big    ? cudaLaunchKernelEx(&cfg, split_combine_kernel<256, 8, 512>, p)
        : wide ? cudaLaunchKernelEx(&cfg, split_combine_kernel<256, 8, 256>, p)
               : cudaLaunchKernelEx(&cfg, split_combine_kernel<256, 4, 256>, p);
  if (e != cudaSuccess) return e;
  return cudaPeekAtLastError();
}

}  // namespace pd
