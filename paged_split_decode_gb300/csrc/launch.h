// launch.h -- internal interface between the host layer and the kernel
// instantiation units (one translation unit per head size and KV dtype, so
// they compile in parallel).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "decode_kernel.cuh"

namespace pd {

struct KernelShape {
  int threads;      // threads per CTA
  int smem_bytes;   // dynamic shared memory per CTA
  int rows_padded;  // RP: query rows per unit rounded up to the row-tile size
  int ctas_per_sm;  // resident CTAs per SM the configuration is sized for
  int heads;        // KV heads per tile (the TMA box's head extent)
  int unit_cost;    // balanced split: virtual tiles charged to every unit start
  int fixed_pieces; // 1: a piece has a large fixed cost (set-up, pipeline refill, epilogue), so
                    // an automatic plan over few units takes the fixed split (one piece per CTA)
  int max_clusters[17];  // [S]: clusters of S CTAs the device runs at once (0: no cluster merge)
};

// Returns false when no instantiation covers (D, kv kind, nt, grouped):
// grouped = 1 asks for the head-group tiles (KernelShape::heads KV heads per
// tile, Hkv a multiple of four), grouped = 0 for per-head tiles.
bool kernel_shape(int D, int kv, int nt, int grouped, KernelShape* out);

// Launch the instantiation for (D, kv kind, nt, grouped) on `grid` CTAs.
cudaError_t launch_decode(int D, int kv, int nt, int grouped, const CUtensorMap& tk,
                          const CUtensorMap& tv, const DecodeParams& p, int grid,
                          cudaStream_t stream);

// Split combine behind a decode launch (split_combine.cu); each split unit's
// output dims are spread over dim_chunks CTAs per head (a divisor of D / 4);
// batch > 4 selects the kernel that loads eight pieces' partials at a time
// (else four), and with it threads > 256 its 512-thread form.
cudaError_t launch_split_combine(int D, const DecodeParams& p, int n_units, int dim_chunks, int batch,
                                 int threads, cudaStream_t stream);

// Per-dtype/head-size entry points defined in decode_*.cu.
bool shape_f16_d128(int nt, int grouped, KernelShape* out);
bool shape_f16_d256(int nt, int grouped, KernelShape* out);
bool shape_fp8_d128(int nt, int grouped, KernelShape* out);
bool shape_fp8_d256(int nt, int grouped, KernelShape* out);
bool shape_i8_d128(int nt, int grouped, KernelShape* out);
bool shape_i8_d256(int nt, int grouped, KernelShape* out);
bool shape_fp8q_d128(int nt, int grouped, KernelShape* out);  // bfloat16 q and out
bool shape_fp8q_d256(int nt, int grouped, KernelShape* out);
bool shape_i8q_d128(int nt, int grouped, KernelShape* out);
bool shape_i8q_d256(int nt, int grouped, KernelShape* out);
bool shape_bf16_d128(int nt, int grouped, KernelShape* out);
bool shape_bf16_d256(int nt, int grouped, KernelShape* out);
cudaError_t launch_f16_d128(int nt, int grouped, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, int,
                            cudaStream_t);
cudaError_t launch_f16_d256(int nt, int grouped, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, int,
                            cudaStream_t);
cudaError_t launch_fp8_d128(int nt, int grouped, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, int,
                            cudaStream_t);
cudaError_t launch_fp8_d256(int nt, int grouped, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, int,
                            cudaStream_t);
cudaError_t launch_i8_d128(int nt, int grouped, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, int,
                           cudaStream_t);
cudaError_t launch_i8_d256(int nt, int grouped, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, int,
                           cudaStream_t);
cudaError_t launch_fp8q_d128(int nt, int grouped, const CUtensorMap&, const CUtensorMap&, const DecodeParams&,
                             int, cudaStream_t);
cudaError_t launch_fp8q_d256(int nt, int grouped, const CUtensorMap&, const CUtensorMap&, const DecodeParams&,
                             int, cudaStream_t);
cudaError_t launch_i8q_d128(int nt, int grouped, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, int,
                            cudaStream_t);
cudaError_t launch_i8q_d256(int nt, int grouped, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, int,
                            cudaStream_t);
cudaError_t launch_bf16_d128(int nt, int grouped, const CUtensorMap&, const CUtensorMap&,
                             const DecodeParams&, int, cudaStream_t);
cudaError_t launch_bf16_d256(int nt, int grouped, const CUtensorMap&, const CUtensorMap&,
                             const DecodeParams&, int, cudaStream_t);

// Identity of the CUDA context current on the calling thread: a number the
// driver never hands out twice in one process (the primary context made after
// a cudaDeviceReset gets a new one), or 0 when no context is current or the
// driver cannot tell. Per-device set-up (a kernel's shared-memory opt-in, a
// device symbol's address) is keyed on it, so it is redone after a reset.
unsigned long long current_context_id();

// Runs `setup` once per CUDA context for the calling thread's current device:
// `done` holds, per device ordinal (< 64), the id of the context that last
// completed it. Returns setup's error, or cudaSuccess.
template <class F>
cudaError_t once_per_context(unsigned long long (&done)[64], F setup) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const unsigned long long ctx = current_context_id();
  if (ctx != 0 && __atomic_load_n(&done[dev], __ATOMIC_ACQUIRE) == ctx) return cudaSuccess;
  e = setup();
  if (e != cudaSuccess) return e;
  __atomic_store_n(&done[dev], ctx, __ATOMIC_RELEASE);
  return cudaSuccess;
}

// Largest thread-block cluster of a cluster-merged split: 16 CTAs, beyond the
// portable 8 (each kernel opts in with cudaFuncAttributeNonPortableClusterSizeAllowed).
constexpr int kMaxCluster = 16;

// A kernel's per-context attributes: its dynamic shared memory opt-in and
// clusters of up to kMaxCluster CTAs.
template <class Kern>
cudaError_t set_kernel_attributes(Kern kernel, int smem) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

// Clusters of c CTAs (2 <= c <= kMaxCluster) of `kernel` (threads and dynamic
// shared memory per CTA as given) that the device runs at once
// (cudaOccupancyMaxActiveClusters), found once per context: counts[c], 0 for
// c < 2 or when the query fails (then no cluster merge is planned).
template <class Kern>
void max_active_clusters(Kern kernel, int threads, int smem, unsigned long long (&ctx_done)[64],
                         int (&cache)[64][kMaxCluster + 1], int (&counts)[kMaxCluster + 1]) {
  for (int c = 0; c <= kMaxCluster; ++c) counts[c] = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return;
  const cudaError_t e = once_per_context(ctx_done, [&] {
    cudaError_t r = set_kernel_attributes(kernel, smem);
    if (r != cudaSuccess) return r;
    for (int c = 2; c <= kMaxCluster; ++c) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(c * 64), 1, 1);
      cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
      cfg.dynamicSmemBytes = static_cast<size_t>(smem);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(c);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();  // the query's own failure: no cluster merge
        n = 0;
      }
      cache[dev][c] = n;
    }
    return cudaSuccess;
  });
  if (e != cudaSuccess) return;
  for (int c = 0; c <= kMaxCluster; ++c) counts[c] = cache[dev][c];
}

// Launch with programmatic dependent launch: the kernel's CTAs may be
// scheduled while the preceding grid in the stream drains; the kernel waits
// (griddepcontrol.wait) before its first global memory access.
// With cluster > 1 the grid (a multiple of it) runs as clusters of that many
// CTAs.
template <class Kern, class... Args>
cudaError_t launch_pdl(Kern kernel, int grid, int threads, int smem, cudaStream_t stream, int cluster,
                       const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) return e;
  return cudaPeekAtLastError();  // the error stays visible to the caller
}

// Launch one configuration; sets the shared-memory opt-in once per context.
template <class Cfg>
cudaError_t launch_cfg(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, int grid,
                       cudaStream_t stream) {
  static unsigned long long attr_ctx[64] = {};
  cudaError_t e = once_per_context(attr_ctx, [] {
    return set_kernel_attributes(decode_paged_kernel<Cfg>, Cfg::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_paged_kernel<Cfg>, grid, Cfg::kThreads, Cfg::kSmemBytes, stream, p.cluster, tk, tv, p);
}

// Largest ring (stage count, capped at 32) whose shared-memory plan lets
// MINB CTAs share one SM's 228 KiB (1 KiB of it reserved per CTA; at most
// 227 KiB for one CTA).
constexpr int smem_limit(int minb) { return minb == 1 ? 227 * 1024 : 228 * 1024 / minb - 1024; }
// The stage count is a multiple of KG (see Cfg).
template <int D, int KV, int NT, int KG, int MINB, int DS, int HG, int RG, int NS = 32>
constexpr int ring_stages() {
  if constexpr (NS <= KG)
    return KG;
  else if constexpr (NS % KG != 0)
    return ring_stages<D, KV, NT, KG, MINB, DS, HG, RG, NS - 1>();
  else if constexpr (Cfg<D, KV, NT, KG, NS, MINB, DS, HG, RG>::kSmemBytes <= smem_limit(MINB))
    return NS;
  else
    return ring_stages<D, KV, NT, KG, MINB, DS, HG, RG, NS - 1>();
}
template <int D, int KV, int NT, int KG, int MINB, int DS = (NT == 1 ? 1 : 2), int HG = 1,
          int RG = ((NT == 4 && DS == 2) ? 2 : 1)>
using CfgFor =
    Cfg<D, KV, NT, KG, ring_stages<D, KV, NT, KG, MINB, DS, HG, RG>(), MINB, DS, HG, RG>;

template <class Cfg>
bool shape_of(KernelShape* out) {
  out->threads = Cfg::kThreads;
  out->smem_bytes = Cfg::kSmemBytes;
  out->rows_padded = Cfg::RP;
  out->ctas_per_sm = Cfg::kMinBlocks;
  out->heads = Cfg::HG;
  // a piece's epilogue (partial rows) and the pipeline turn it causes, as
  // 16-key tiles: ranges that take on a second unit get that many fewer
  // (measured on GB300, D=256 GQA 6:1 L=4096, 0 -> 4 tiles: B=8 28.8 -> 28.5
  // us, e4m3 B=32 54.9 -> 54.2 us, L=32768 B=1 30.2 -> 30.0 us, B=32 86.1 ->
  // 86.0 us; 12 tiles slowed B=32 to 87.2 us)
  out->unit_cost = 4;
  out->fixed_pieces = 0;
  static unsigned long long ctx_done[64] = {};
  static int cache[64][kMaxCluster + 1] = {};
  max_active_clusters(decode_paged_kernel<Cfg>, Cfg::kThreads, Cfg::kSmemBytes, ctx_done, cache, out->max_clusters);
  return true;
}

}  // namespace pd
