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
// Memory-bound: one warp per token in a grid-stride loop, lanes over the
// token's 16-byte vectors (K and V together), a few resident blocks per SM. The quotient is the
// correctly rounded fp32 x / scale, formed from the reciprocal r = RN(1/scale)
// by one residual correction, two elements at a time with the packed f32x2
// multiply and fused multiply-add (Markstein's theorem: with r the correctly
// rounded reciprocal and q0 = RN(x r) within an ulp of x / scale, the residual
// e = x - q0 scale is exact under FMA and RN(q0 + e r) is the correctly
// rounded quotient, for quotients away from the underflow range); the host
// takes the plain division when the scale is outside [2^-100, 2^100].
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pdecode.h"

namespace pd {
namespace {

// Eight resident blocks of 256 threads per SM for the quantising writers (the
// register budget is held to 32 per thread for it): measured 38.0 -> 35.7 us
// (fp8 cache) and 39.3 -> 35.4 us (int8) for 32768 tokens against five blocks
// at 47 registers. The 16-bit copy keeps its own register count (held to 32
// it measured 46.5 -> 49.7 us).
constexpr int kWriterThreads = 256;
constexpr int kWriterBlocksPerSm = 8;

__device__ __forceinline__ uint32_t e4m3x2_of(float lo, float hi) {
  uint16_t r;
  // the first source lands in the upper byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Code of an int8 cache: the quotient clamped to [-127, 127] (NaN -> 0) and
// rounded to the nearest integer, ties to even, by adding 1.5 * 2^23: the sum's
// low mantissa bits then hold the integer in two's complement. Returns the
// float whose low byte is the code.
__device__ __forceinline__ uint32_t i8_bits(float t) {
  t = (t == t) ? fminf(fmaxf(t, -127.f), 127.f) : 0.f;
  return __float_as_uint(t + 12582912.f);
}

// Two fp32 values in one 64-bit register (low word = first), for the packed
// f32x2 arithmetic of sm_100-class GPUs.
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
  return static_cast<unsigned long long>(__float_as_uint(lo)) |
         (static_cast<unsigned long long>(__float_as_uint(hi)) << 32);
}
__device__ __forceinline__ float f2_lo(unsigned long long v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f2_hi(unsigned long long v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Correctly rounded quotients x / s of a pair (see the header): q0 = RN(x r),
// e = x - q0 s (exact under FMA), q1 = RN(q0 + e r), as packed f32x2
// operations; ns = -s. q1 is kept unless it is zero or NaN: then q0 is the
// quotient (x = +-0, whose sign q1 can lose, or x infinite, where the
// residual is NaN; a NaN x gives NaN either way). `fast` = 0 takes the plain
// correctly rounded division (scales outside [2^-100, 2^100]).
__device__ __forceinline__ float2 quot2(float2 x, float s, unsigned long long r2, unsigned long long ns2,
                                        bool fast) {
  if (!fast) return make_float2(__fdiv_rn(x.x, s), __fdiv_rn(x.y, s));
  const unsigned long long xx = f2_pack(x.x, x.y);
  const unsigned long long q0 = f2_mul(xx, r2);
  const unsigned long long e = f2_fma(q0, ns2, xx);
  const unsigned long long q1 = f2_fma(e, r2, q0);
  const float a = f2_lo(q1), b = f2_hi(q1);
  return make_float2(fabsf(a) > 0.f ? a : f2_lo(q0), fabsf(b) > 0.f ? b : f2_hi(q0));
}

// Minimum / maximum that return NaN when either input is NaN.
__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float min_nan(float a, float b) {
  float d;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
// int8 code of a quotient t: max(t, -127) (NaN kept), then the conversion's
// own rounding to the nearest integer (ties to even), saturation at 127 and
// NaN -> 0. The code is in the low byte.
__device__ __forceinline__ uint32_t i8_code(float t) {
  uint32_t d;
  asm("cvt.rni.sat.s8.f32 %0, %1;" : "=r"(d) : "f"(max_nan(t, -127.f)));
  return d;
}
// int8 codes of a pair on the fast path: x is first held to [-b, b]
// (b = 128 |scale|; NaN kept), which changes no code (every quotient beyond
// +-127.5 saturates) and keeps the residual finite, so the plain residual
// quotient q1 is the correctly rounded one (the sign of a zero quotient does
// not matter for an integer code).
__device__ __forceinline__ uint32_t i8_pair_fast(float2 x, float b, unsigned long long r2,
                                                 unsigned long long ns2) {
  const unsigned long long xx = f2_pack(min_nan(max_nan(x.x, -b), b), min_nan(max_nan(x.y, -b), b));
  const unsigned long long q0 = f2_mul(xx, r2);
  const unsigned long long e = f2_fma(q0, ns2, xx);
  const unsigned long long q1 = f2_fma(e, r2, q0);
  return __byte_perm(i8_code(f2_lo(q1)), i8_code(f2_hi(q1)), 0x0040);
}

// BIN: the new tokens are bfloat16 (fp16 otherwise); both widen to fp32 exactly.
template <int KV, bool BIN>
__device__ __forceinline__ void store_row8(void* cache, long long elem, uint4 x, float scale, float rcp,
                                           bool fast) {
  if constexpr (KV == PD_KV_F16) {
    *reinterpret_cast<uint4*>(static_cast<__half*>(cache) + elem) = x;
  } else {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    const unsigned long long r2 = f2_pack(rcp, rcp), ns2 = f2_pack(-scale, -scale);
    if (KV == PD_KV_INT8 && fast) {
      const float b = 128.f * fabsf(scale);
      uint32_t c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 p = BIN ? make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u))
                             : __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        c[i] = i8_pair_fast(p, b, r2, ns2);
      }
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(cache) + elem) =
          make_uint2(__byte_perm(c[0], c[1], 0x5410), __byte_perm(c[2], c[3], 0x5410));
      return;
    }
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 p = BIN ? make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u))
                           : __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      const float2 q = quot2(p, scale, r2, ns2, fast);
      f[2 * i] = q.x;
      f[2 * i + 1] = q.y;
    }
    uint2 o;
    if constexpr (KV == PD_KV_FP8_E4M3) {
      o.x = e4m3x2_of(f[0], f[1]) | (e4m3x2_of(f[2], f[3]) << 16);
      o.y = e4m3x2_of(f[4], f[5]) | (e4m3x2_of(f[6], f[7]) << 16);
    } else {
      // low bytes of four sums -> one word (prmt selects bytes 0 of each)
      o.x = __byte_perm(__byte_perm(i8_bits(f[0]), i8_bits(f[1]), 0x0040),
                        __byte_perm(i8_bits(f[2]), i8_bits(f[3]), 0x0040), 0x5410);
      o.y = __byte_perm(__byte_perm(i8_bits(f[4]), i8_bits(f[5]), 0x0040),
                        __byte_perm(i8_bits(f[6]), i8_bits(f[7]), 0x0040), 0x5410);
    }
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(cache) + elem) = o;
  }
}

template <int KV, bool BIN>
__global__ void __launch_bounds__(kWriterThreads, KV == PD_KV_F16 ? 1 : kWriterBlocksPerSm) kv_writer_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int64_t* __restrict__ slot_mapping, long long num_tokens, int vecs_per_token,
    long long slots, void* __restrict__ k_cache, void* __restrict__ v_cache, float k_scale,
    float v_scale, float k_rcp, float v_rcp, int fast, uint32_t* error_flag) {
  // one warp per token (grid-stride over tokens), lanes over its 16-byte input
  // vectors; cache row = slot (block slot / bs, offset slot % bs of the
  // [num_blocks, bs, Hkv, D] cache is row slot of [num_blocks * bs, Hkv, D])
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (kWriterThreads / 32);
  for (long long t = static_cast<long long>(blockIdx.x) * (kWriterThreads / 32) + (threadIdx.x >> 5);
       t < num_tokens; t += warps) {
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;  // padding token
    if (slot >= slots) {
      if (error_flag && lane == 0) atomicOr(error_flag, PD_DEVERR_SLOT);
      continue;
    }
    const uint4* kin = k_new + t * vecs_per_token;
    const uint4* vin = v_new + t * vecs_per_token;
    const long long base = static_cast<long long>(slot) * vecs_per_token;
#pragma unroll 4
    for (int v = lane; v < vecs_per_token; v += 32) {
      const uint4 kx = __ldcs(kin + v), vx = __ldcs(vin + v);
      store_row8<KV, BIN>(k_cache, (base + v) * 8, kx, k_scale, k_rcp, fast != 0);
      store_row8<KV, BIN>(v_cache, (base + v) * 8, vx, v_scale, v_rcp, fast != 0);
    }
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
      d.kv_dtype != PD_KV_BF16 && d.kv_dtype != PD_KV_FP8_E4M3_BF16 && d.kv_dtype != PD_KV_INT8_BF16)
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
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return PD_ERR_CUDA;
  const long long want = (static_cast<long long>(num_tokens) + pd::kWriterThreads / 32 - 1) / (pd::kWriterThreads / 32);
  const long long cap = static_cast<long long>(sms) * pd::kWriterBlocksPerSm;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  const long long slots = static_cast<long long>(d.num_blocks) * d.block_size;
  auto s = static_cast<cudaStream_t>(stream);
  // residual-corrected division for scales whose reciprocal and quotients stay
  // in the normal range; the plain correctly rounded division otherwise
  auto moderate = [](float x) { const float a = x < 0 ? -x : x; return a >= 0x1p-100f && a <= 0x1p100f; };
  const int fast = moderate(d.k_scale) && moderate(d.v_scale) ? 1 : 0;
  const float k_rcp = fast ? 1.f / d.k_scale : 0.f, v_rcp = fast ? 1.f / d.v_scale : 0.f;
  const auto* kn = static_cast<const uint4*>(k_new);
  const auto* vn = static_cast<const uint4*>(v_new);
  switch (d.kv_dtype) {
    case PD_KV_F16:
    case PD_KV_BF16:  // 16-bit caches: the input bits as they are
      pd::kv_writer_kernel<PD_KV_F16, false><<<grid, pd::kWriterThreads, 0, s>>>(
          kn, vn, slot_mapping, static_cast<long long>(num_tokens), vecs, slots, k_cache, v_cache, 1.f, 1.f, 1.f, 1.f, 0,
          error_flag);
      break;
    case PD_KV_FP8_E4M3:
      pd::kv_writer_kernel<PD_KV_FP8_E4M3, false><<<grid, pd::kWriterThreads, 0, s>>>(
          kn, vn, slot_mapping, static_cast<long long>(num_tokens), vecs, slots, k_cache, v_cache, d.k_scale,
          d.v_scale, k_rcp, v_rcp, fast, error_flag);
      break;
    case PD_KV_FP8_E4M3_BF16:
      pd::kv_writer_kernel<PD_KV_FP8_E4M3, true><<<grid, pd::kWriterThreads, 0, s>>>(
          kn, vn, slot_mapping, static_cast<long long>(num_tokens), vecs, slots, k_cache, v_cache, d.k_scale,
          d.v_scale, k_rcp, v_rcp, fast, error_flag);
      break;
    case PD_KV_INT8_BF16:
      pd::kv_writer_kernel<PD_KV_INT8, true><<<grid, pd::kWriterThreads, 0, s>>>(
          kn, vn, slot_mapping, static_cast<long long>(num_tokens), vecs, slots, k_cache, v_cache, d.k_scale,
          d.v_scale, k_rcp, v_rcp, fast, error_flag);
      break;
    default:
      pd::kv_writer_kernel<PD_KV_INT8, false><<<grid, pd::kWriterThreads, 0, s>>>(
          kn, vn, slot_mapping, static_cast<long long>(num_tokens), vecs, slots, k_cache, v_cache, d.k_scale,
          d.v_scale, k_rcp, v_rcp, fast, error_flag);
      break;
  }
  return cudaPeekAtLastError() == cudaSuccess ? PD_OK : PD_ERR_CUDA;
}
