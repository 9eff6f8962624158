// combine.cu -- the split-K combine on its own: merges S fp32 (m, l, O)
// partials per row into one fp16 row (the combine step of the per-head split
// decode in opengfx1030/vllm-rdna pull request #33, "Purpose").
//   M = max_s m_s, w_s = exp(m_s - M) (0 for an empty chunk, m_s = -inf),
//   out = sum_s w_s O_s / sum_s w_s l_s, zeros when every chunk is empty.
// One thread per (row, 8 output dims); partials are read in split order, so
// the result does not depend on scheduling.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "pdecode.h"
#include "ptx.cuh"

namespace pd {
namespace {

constexpr float kLog2eF = 1.4426950408889634f;

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ m,
                                                      const float* __restrict__ l,
                                                      const float* __restrict__ o, int rows, int S,
                                                      int D, __half* __restrict__ out) {
  const int dch = D / 8;
  const long long item = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (item >= static_cast<long long>(rows) * dch) return;
  const int r = static_cast<int>(item / dch), dc = static_cast<int>(item % dch);
  const float* mr = m + static_cast<long long>(r) * S;
  const float* lr = l + static_cast<long long>(r) * S;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, mr[s]);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float L = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const float ms = mr[s];
      const float w = (ms == -INFINITY) ? 0.f : ex2((ms - M) * kLog2eF);
      L += w * lr[s];
      const float4* src =
          reinterpret_cast<const float4*>(o + (static_cast<long long>(r) * S + s) * D + dc * 8);
      const float4 a = src[0], b = src[1];
      acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
      acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
    }
  }
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  uint4 v;
  v.x = pack_half2(acc[0] * inv, acc[1] * inv);
  v.y = pack_half2(acc[2] * inv, acc[3] * inv);
  v.z = pack_half2(acc[4] * inv, acc[5] * inv);
  v.w = pack_half2(acc[6] * inv, acc[7] * inv);
  *reinterpret_cast<uint4*>(out + static_cast<long long>(r) * D + dc * 8) = v;
}

}  // namespace
}  // namespace pd

extern "C" pd_status decode_paged_combine(const float* part_m, const float* part_l,
                                          const float* part_o, int rows, int num_splits, int D,
                                          void* out, void* stream) {
  if (rows < 0 || num_splits < 1 || D < 8 || D > 1024 || D % 8 != 0) return PD_ERR_SHAPE;
  if (rows == 0) return PD_OK;
  if (!part_m || !part_l || !part_o || !out) return PD_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(part_o) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u) ||
      (reinterpret_cast<uintptr_t>(part_m) & 3u) || (reinterpret_cast<uintptr_t>(part_l) & 3u))
    return PD_ERR_ALIGN;
  const long long items = static_cast<long long>(rows) * (D / 8);
  const int threads = 256;
  const long long blocks = (items + threads - 1) / threads;
  if (blocks > 0x7fffffffll) return PD_ERR_UNSUPPORTED;
  pd::combine_kernel<<<static_cast<unsigned>(blocks), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      part_m, part_l, part_o, rows, num_splits, D, static_cast<__half*>(out));
  return cudaPeekAtLastError() == cudaSuccess ? PD_OK : PD_ERR_CUDA;
}
