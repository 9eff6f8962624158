// kv_writer.cu -- the paged KV-cache writer: stores the K and V rows of new
// tokens at their cache slots, the layout the decode reads (the writer-layout
// cell of the "Test Plan" in opengfx1030/vllm-rdna pull request #33).
//
// Token t goes to block slot / block_size, offset slot % block_size of
// [num_blocks, block_size, Hkv, D]; its Hkv*D elements are contiguous in both
// the input [T, Hkv, D] and the cache, so the copy is a stream of 16-byte
// input vectors (8 values) per token. fp16 and bfloat16 caches get the input
// bits as they are (the input has the cache's type); fp8 and int8 caches get
// the code nearest to the IEEE fp32 quotient
// x / scale: cvt.rn.satfinite to e4m3 (ties to even, +-448 at most, NaN ->
// 0x7F), or round-to-nearest-even to an integer clamped to [-127, 127]
// (NaN -> 0).
//
// Memory-bound: a grid-stride loop over (token, vector) items, K and V of an
// item together, sized to a few resident blocks per SM.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pdecode.h"

namespace pd {
namespace {

constexpr int kWriterThreads = 256;
constexpr int kWriterBlocksPerSm = 8;

__device__ __forceinline__ uint32_t e4m3x2_of(float lo, float hi) {
  uint16_t r;
  // the first source lands in the upper byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t i8_of(float t) {
  int c = __float2int_rn(t);  // NaN -> 0; beyond int range saturates
  c = max(-127, min(127, c));
  return static_cast<uint32_t>(c) & 0xffu;
}

template <int KV>
__device__ __forceinline__ void store_row8(void* cache, long long elem, uint4 x, float scale) {
  if constexpr (KV == PD_KV_F16) {
    *reinterpret_cast<uint4*>(static_cast<__half*>(cache) + elem) = x;
  } else {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      f[2 * i] = __fdiv_rn(p.x, scale);
      f[2 * i + 1] = __fdiv_rn(p.y, scale);
    }
    uint2 o;
    if constexpr (KV == PD_KV_FP8_E4M3) {
      o.x = e4m3x2_of(f[0], f[1]) | (e4m3x2_of(f[2], f[3]) << 16);
      o.y = e4m3x2_of(f[4], f[5]) | (e4m3x2_of(f[6], f[7]) << 16);
    } else {
      o.x = i8_of(f[0]) | (i8_of(f[1]) << 8) | (i8_of(f[2]) << 16) | (i8_of(f[3]) << 24);
      o.y = i8_of(f[4]) | (i8_of(f[5]) << 8) | (i8_of(f[6]) << 16) | (i8_of(f[7]) << 24);
    }
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(cache) + elem) = o;
  }
}

template <int KV>
__global__ void __launch_bounds__(kWriterThreads) kv_writer_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int64_t* __restrict__ slot_mapping, long long items, int vecs_per_token,
    long long slots, int block_size, void* __restrict__ k_cache, void* __restrict__ v_cache,
    float k_scale, float v_scale, uint32_t* error_flag) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long it = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; it < items;
       it += stride) {
    const long long t = it / vecs_per_token;
    const int vec = static_cast<int>(it - t * vecs_per_token);
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;  // padding token
    if (slot >= slots) {
      if (error_flag && vec == 0) atomicOr(error_flag, PD_DEVERR_SLOT);
      continue;
    }
    const long long blk = slot / block_size, off = slot - blk * block_size;
    const long long elem =
        ((blk * block_size + off) * vecs_per_token + vec) * 8;  // first element of the vector
    const uint4 kx = __ldcs(k_new + it), vx = __ldcs(v_new + it);
    store_row8<KV>(k_cache, elem, kx, k_scale);
    store_row8<KV>(v_cache, elem, vx, v_scale);
  }
}

}  // namespace
}  // namespace pd

extern "C" pd_status write_kv_cache(const void* k_new, const void* v_new,
                                    const int64_t* slot_mapping, int num_tokens, void* k_cache,
                                    void* v_cache, const pd_dims* dims, uint32_t* error_flag,
                                    void* stream) {
  if (!dims) return PD_ERR_NULL;
  const pd_dims& d = *dims;
  if (num_tokens < 0 || d.Hkv < 1 || d.D < 8 || d.D % 8 != 0 || d.block_size < 1 ||
      d.num_blocks < 0)
    return PD_ERR_SHAPE;
  if (d.kv_dtype != PD_KV_F16 && d.kv_dtype != PD_KV_FP8_E4M3 && d.kv_dtype != PD_KV_INT8 &&
      d.kv_dtype != PD_KV_BF16)
    return PD_ERR_DTYPE;
  const long long row = static_cast<long long>(d.Hkv) * d.D;
  if (row / 8 > 0x7fffffffll) return PD_ERR_SHAPE;
  if (num_tokens == 0) return PD_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PD_ERR_NULL;
  const bool two_byte = d.kv_dtype == PD_KV_F16 || d.kv_dtype == PD_KV_BF16;
  const uintptr_t cache_align = two_byte ? 15u : 7u;
  if ((reinterpret_cast<uintptr_t>(k_new) & 15u) || (reinterpret_cast<uintptr_t>(v_new) & 15u) ||
      (reinterpret_cast<uintptr_t>(k_cache) & cache_align) ||
      (reinterpret_cast<uintptr_t>(v_cache) & cache_align) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PD_ERR_ALIGN;
  const int vecs = static_cast<int>(row / 8);
  const long long items = static_cast<long long>(num_tokens) * vecs;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return PD_ERR_CUDA;
  const long long want = (items + pd::kWriterThreads - 1) / pd::kWriterThreads;
  const long long cap = static_cast<long long>(sms) * pd::kWriterBlocksPerSm;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  const long long slots = static_cast<long long>(d.num_blocks) * d.block_size;
  auto s = static_cast<cudaStream_t>(stream);
  const auto* kn = static_cast<const uint4*>(k_new);
  const auto* vn = static_cast<const uint4*>(v_new);
  switch (d.kv_dtype) {
    case PD_KV_F16:
    case PD_KV_BF16:  // 16-bit caches: the input bits as they are
      pd::kv_writer_kernel<PD_KV_F16><<<grid, pd::kWriterThreads, 0, s>>>(
          kn, vn, slot_mapping, items, vecs, slots, d.block_size, k_cache, v_cache, 1.f, 1.f,
          error_flag);
      break;
    case PD_KV_FP8_E4M3:
      pd::kv_writer_kernel<PD_KV_FP8_E4M3><<<grid, pd::kWriterThreads, 0, s>>>(
          kn, vn, slot_mapping, items, vecs, slots, d.block_size, k_cache, v_cache, d.k_scale,
          d.v_scale, error_flag);
      break;
    default:
      pd::kv_writer_kernel<PD_KV_INT8><<<grid, pd::kWriterThreads, 0, s>>>(
          kn, vn, slot_mapping, items, vecs, slots, d.block_size, k_cache, v_cache, d.k_scale,
          d.v_scale, error_flag);
      break;
  }
  return cudaGetLastError() == cudaSuccess ? PD_OK : PD_ERR_CUDA;
}
