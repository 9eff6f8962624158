// pdecode_api.cu -- host side of libpdecode: argument validation, the split
// plan, TMA descriptors for the paged caches, and launches on the caller's
// stream. The C ABI is declared in include/pdecode.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <atomic>
#include <mutex>

#include "launch.h"
#include "pdecode.h"

namespace pd {

bool kernel_shape(int D, int kv, int nt, int grouped, KernelShape* out) {
  if (kv == kKvBf16)
    return D == 128 ? shape_bf16_d128(nt, grouped, out)
                    : D == 256 && shape_bf16_d256(nt, grouped, out);
  if (kv == kKvFp8Bq)
    return D == 128 ? shape_fp8q_d128(nt, grouped, out) : D == 256 && shape_fp8q_d256(nt, grouped, out);
  if (kv == kKvInt8Bq)
    return D == 128 ? shape_i8q_d128(nt, grouped, out) : D == 256 && shape_i8q_d256(nt, grouped, out);
  if (D == 128)
    return kv == kKvFp8 ? shape_fp8_d128(nt, grouped, out) : kv == kKvInt8 ? shape_i8_d128(nt, grouped, out)
                                                                      : shape_f16_d128(nt, grouped, out);
  if (D == 256)
    return kv == kKvFp8 ? shape_fp8_d256(nt, grouped, out) : kv == kKvInt8 ? shape_i8_d256(nt, grouped, out)
                                                                      : shape_f16_d256(nt, grouped, out);
  return false;
}

cudaError_t launch_decode(int D, int kv, int nt, int grouped, const CUtensorMap& tk,
                          const CUtensorMap& tv, const DecodeParams& p, int grid, cudaStream_t s) {
  if (kv == kKvBf16)
    return D == 128 ? launch_bf16_d128(nt, grouped, tk, tv, p, grid, s)
                    : launch_bf16_d256(nt, grouped, tk, tv, p, grid, s);
  if (kv == kKvFp8Bq)
    return D == 128 ? launch_fp8q_d128(nt, grouped, tk, tv, p, grid, s)
                    : launch_fp8q_d256(nt, grouped, tk, tv, p, grid, s);
  if (kv == kKvInt8Bq)
    return D == 128 ? launch_i8q_d128(nt, grouped, tk, tv, p, grid, s)
                    : launch_i8q_d256(nt, grouped, tk, tv, p, grid, s);
  if (D == 128)
    return kv == kKvFp8 ? launch_fp8_d128(nt, grouped, tk, tv, p, grid, s)
           : kv == kKvInt8 ? launch_i8_d128(nt, grouped, tk, tv, p, grid, s)
                           : launch_f16_d128(nt, grouped, tk, tv, p, grid, s);
  return kv == kKvFp8 ? launch_fp8_d256(nt, grouped, tk, tv, p, grid, s)
         : kv == kKvInt8 ? launch_i8_d256(nt, grouped, tk, tv, p, grid, s)
                         : launch_f16_d256(nt, grouped, tk, tv, p, grid, s);
}

namespace {

constexpr unsigned long long kTimeoutNs = 2000000000ull;  // 2 s per pipeline wait (default)
std::atomic<unsigned long long> g_wait_limit_ns{kTimeoutNs};
std::atomic<int> g_inject{0};

// Resolved work decomposition of one call.
struct Plan {
  int splits;       // 0 = balanced, >= 1 fixed
  int grid;         // CTAs launched
  int nt;           // row tiles per head
  int hg;           // KV heads per tile
  long long slots;  // partial slots in the workspace
  long long n_merge; // units the split combine visits
  long long units;  // B * Hkv / hg work units
  int rows_padded;
  int unit_cost;    // balanced split: virtual tiles per unit start
  int cluster;      // > 1: the fixed split's pieces of a unit form a cluster that merges them
  int sms;          // SMs of the device the plan was made for
  size_t off_ml, off_o, bytes;  // workspace layout
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Caches of one-byte codes (e4m3fn or int8, with an fp16 or a bfloat16 q).
bool byte_kind(int kv) {
  return kv == PD_KV_FP8_E4M3 || kv == PD_KV_INT8 || kv == PD_KV_FP8_E4M3_BF16 || kv == PD_KV_INT8_BF16;
}
// q and out (and a writer's new tokens) in bfloat16.
bool bf16_io(int kv) { return kv == PD_KV_BF16 || kv == PD_KV_FP8_E4M3_BF16 || kv == PD_KV_INT8_BF16; }

pd_status check_dims(const pd_dims* d, int qlen) {
  if (!d) return PD_ERR_NULL;
  if (d->B < 0 || d->Hq < 1 || d->Hkv < 1 || d->D < 1 || d->block_size < 1 || d->num_blocks < 0 ||
      d->max_blocks_per_seq < 0 || qlen < 1)
    return PD_ERR_SHAPE;
  if (d->Hq % d->Hkv != 0) return PD_ERR_SHAPE;
  if (d->kv_dtype != PD_KV_F16 && d->kv_dtype != PD_KV_BF16 && !byte_kind(d->kv_dtype))
    return PD_ERR_DTYPE;
  if (byte_kind(d->kv_dtype) && (!std::isfinite(d->k_scale) || !std::isfinite(d->v_scale)))
    return PD_ERR_SHAPE;
  if (d->D != 128 && d->D != 256) return PD_ERR_UNSUPPORTED;
  if (d->block_size % kTileKeys != 0) return PD_ERR_UNSUPPORTED;
  if (qlen > 8) return PD_ERR_UNSUPPORTED;
  const int R = d->Hq / d->Hkv * qlen;
  if (R > 32) return PD_ERR_UNSUPPORTED;
  // 32-bit index headroom: tiles, keys and cache rows
  const long long cap_keys = static_cast<long long>(d->max_blocks_per_seq) * d->block_size;
  if (cap_keys > (1ll << 30)) return PD_ERR_UNSUPPORTED;
  if (static_cast<long long>(d->B) * d->Hkv * (cap_keys / kTileKeys + 1 + 64) > (1ll << 31) - 1)
    return PD_ERR_UNSUPPORTED;
  if (static_cast<long long>(d->num_blocks) * d->block_size > (1ll << 31) - 1) return PD_ERR_UNSUPPORTED;
  if (static_cast<long long>(d->B) * qlen * d->Hq > (1ll << 31) - 1) return PD_ERR_UNSUPPORTED;
  return PD_OK;
}

int device_sm_count(int sm_count) {
  if (sm_count > 0) return sm_count;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Automatic split (num_splits = 0): balanced over every resident CTA slot,
// except when the units are few (<= a quarter of the CTA slots) and either
// their work is small (at most 24 visible tiles per CTA slot, from the table
// capacity and the window: latency-bound, where each piece's fixed cost and
// the combine's fan-in dominate) or the kernel's pieces carry a large fixed
// cost (the tensor-memory kernels, KernelShape::fixed_pieces): then a fixed
// split of each unit into
// floor(0.84 CTA slots / units) chunks, one per CTA, which leaves about a
// sixth of the SMs idle but gives every CTA one piece. Measured on GB300
// (D=256 GQA 6:1, L=4096): B = 1 / 2 / 3 12.9 / 16.1 / 19.2 -> 12.0 / 15.0 /
// 18.0 us; windowed L=32768 B = 1 / 2 12.8 / 15.8 -> 12.0 / 14.9 us; qlen=3
// e4m3 verify B=8 39.8 -> 36.0 us; shapes with more work per CTA (B >= 8 at
// L=4096, L=32768 without a window) stay balanced: there the two splits are
// within ~2 % or the fixed one loses (B=16: +1.0 us, 2 x 2048 tiles: +0.5). The
// workspace is sized for the balanced split in either case (the fixed split
// needs fewer slots), so pd_workspace_bytes does not depend on the window.
pd_status make_plan(const pd_dims* d, int qlen, int num_splits, int sm_count, Plan* pl, int window = 0) {
  pd_status st = check_dims(d, qlen);
  if (st != PD_OK) return st;
  if (num_splits < 0) return PD_ERR_SHAPE;
  const int sms = device_sm_count(sm_count);
  if (sms <= 0) return PD_ERR_CUDA;
  pl->sms = sms;
  const int R = d->Hq / d->Hkv * qlen;
  pl->nt = (R + 7) / 8;
  KernelShape ks;
  // tiles of several KV heads read the cache contiguously; they serve the
  // single-row-tile shapes whose head count is a multiple of four (the
  // instantiation chooses how many heads a tile holds: 2 or 4)
  const bool grouped = pl->nt == 1 && d->Hkv % 4 == 0;
  if (!(grouped && kernel_shape(d->D, d->kv_dtype, pl->nt, 1, &ks)) &&
      !kernel_shape(d->D, d->kv_dtype, pl->nt, 0, &ks))
    return PD_ERR_UNSUPPORTED;
  pl->hg = ks.heads;
  pl->rows_padded = ks.rows_padded;
  pl->unit_cost = ks.unit_cost;
  pl->units = static_cast<long long>(d->B) * (d->Hkv / pl->hg);
  int splits = num_splits;
  if (splits == 0 && d->B > kMaxAutoB) splits = 1;  // plenty of units: one piece each
  const int ctas = sms * ks.ctas_per_sm;  // persistent grid: every resident CTA slot
  const bool automatic = splits == 0;
  if (automatic && pl->units > 0 && pl->units <= ctas / 4) {
    const long long cap_keys = static_cast<long long>(d->max_blocks_per_seq) * d->block_size;
    const long long vis_keys = window > 0 ? std::min<long long>(cap_keys, window + qlen + kTileKeys) : cap_keys;
    const long long tiles = pl->units * (vis_keys / kTileKeys + 1);
    if (tiles <= 24ll * ctas || ks.fixed_pieces)
      splits = static_cast<int>(std::max<long long>(1, (ctas * 27 / 32) / pl->units));
  }
  pl->splits = splits;
  if (splits == 0) {
    pl->grid = ctas;
    pl->slots = 2ll * ctas;  // a CTA's range holds at most two split pieces
    pl->n_merge = pl->units;
  } else {
    const long long pieces = pl->units * splits;
    pl->grid = static_cast<int>(pieces < ctas ? (pieces > 0 ? pieces : 1) : ctas);
    pl->slots = splits > 1 ? pieces : 0;
    pl->n_merge = splits > 1 ? pl->units : 0;
  }
  // an automatic plan sizes its workspace for the balanced split, whichever
  // split it chose (so the size does not depend on the window)
  const long long ws_slots = automatic && d->B <= kMaxAutoB ? 2ll * ctas : pl->slots;
  if (pl->slots == 0 && ws_slots == 0) {
    pl->off_ml = pl->off_o = pl->bytes = 0;
  } else {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t ml = up(static_cast<size_t>(ws_slots) * pl->rows_padded * 2 * 4);
    const size_t o = static_cast<size_t>(ws_slots) * pl->rows_padded * d->D * 4;
    pl->off_ml = 0;
    pl->off_o = ml;
    pl->bytes = ml + o;
  }
  // A fixed split of at most kMaxCluster pieces per unit, one CTA each, on a kernel
  // that merges a unit's pieces inside its thread-block cluster (distributed
  // shared memory), when the device runs every unit's cluster at once: no
  // split-combine launch. (The workspace keeps the size computed above, so it
  // does not depend on the device's cluster occupancy.)
  pl->cluster = 0;
  if (splits >= 2 && splits <= kMaxCluster && pl->units * splits == pl->grid &&
      ks.max_clusters[splits] >= pl->units) {
    pl->cluster = splits;
    pl->n_merge = 0;
  }
  return PD_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

// cuCtxGetCurrent and cuCtxGetId through the runtime's driver entry points.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

namespace {

// 3-D map over a paged cache viewed as [num_blocks*block_size][Hkv][D]:
// box = one 128-byte row slab x one head x 16 keys, 128B swizzle.
// Box: 128 bytes of D x hg heads x 16 keys, 128-byte swizzled.
bool encode_cache_map(CUtensorMap* m, const void* base, const pd_dims* d, int hg) {
  auto fn = encode_fn();
  if (!fn) return false;
  const bool byte = byte_kind(d->kv_dtype);
  const cuuint64_t elem = byte ? 1 : 2;
  const cuuint64_t rows = static_cast<cuuint64_t>(d->num_blocks) * d->block_size;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d->D), static_cast<cuuint64_t>(d->Hkv),
                        rows > 0 ? rows : 1};
  cuuint64_t strides[2] = {d->D * elem, static_cast<cuuint64_t>(d->Hkv) * d->D * elem};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elem), static_cast<cuuint32_t>(hg),
                       static_cast<cuuint32_t>(kTileKeys)};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType type = byte ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : d->kv_dtype == PD_KV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = fn(m, type, 3,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace
}  // namespace pd

using namespace pd;

extern "C" {

void pd_set_wait_limit_ns(unsigned long long ns) {
  g_wait_limit_ns.store(ns ? ns : kTimeoutNs, std::memory_order_relaxed);
}

void pd_set_fault_injection(int mode) { g_inject.store(mode == 1 ? 1 : 0, std::memory_order_relaxed); }

const char* pd_status_str(pd_status s) {
  switch (s) {
    case PD_OK: return "ok";
    case PD_ERR_NULL: return "a required pointer is NULL";
    case PD_ERR_SHAPE: return "inconsistent or out-of-range sizes";
    case PD_ERR_DTYPE: return "unknown KV dtype";
    case PD_ERR_UNSUPPORTED: return "shape not implemented by these kernels";
    case PD_ERR_ALIGN: return "pointer not 16-byte aligned";
    case PD_ERR_WORKSPACE: return "workspace missing or too small";
    case PD_ERR_CUDA: return "CUDA runtime error";
  }
  return "unknown status";
}

size_t pd_workspace_bytes(const pd_dims* dims, int qlen, int num_splits, int sm_count) {
  Plan pl;
  if (make_plan(dims, qlen, num_splits, sm_count, &pl) != PD_OK) return 0;
  return pl.bytes;
}

int pd_grid_ctas(const pd_dims* dims, int qlen, int num_splits, int sm_count) {
  Plan pl;
  if (make_plan(dims, qlen, num_splits, sm_count, &pl) != PD_OK) return 0;
  return pl.grid;
}

}  // extern "C"

namespace {

// decode_paged and decode_paged_varlen: q_start null means B sequences of qlen
// query tokens each (total_q = B * qlen); otherwise sequence b owns rows
// [q_start[b], q_start[b+1]) of q and out, at most qlen of them.
pd_status decode_impl(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_start,
                      int total_q, float scale, int window, int qlen, int num_splits, void* out,
                      const pd_dims* dims, void* workspace, size_t workspace_bytes,
                      uint32_t* error_flag, void* stream) {
  pd_status st = check_dims(dims, qlen);
  if (st != PD_OK) return st;
  if (num_splits < 0 || !std::isfinite(scale)) return PD_ERR_SHAPE;
  if (total_q < 0 || static_cast<long long>(total_q) * dims->Hq > (1ll << 31) - 1)
    return q_start ? PD_ERR_SHAPE : PD_ERR_UNSUPPORTED;
  if (dims->B == 0 || total_q == 0) return PD_OK;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out) return PD_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(q_start) & 3u) || (reinterpret_cast<uintptr_t>(error_flag) & 3u))
    return PD_ERR_ALIGN;
  if (dims->num_blocks == 0) return PD_ERR_SHAPE;
  Plan pl;
  st = make_plan(dims, qlen, num_splits, 0, &pl, window);
  if (st != PD_OK) return st;
  if (pl.bytes > 0) {
    if (!workspace || workspace_bytes < pl.bytes) return PD_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PD_ERR_ALIGN;
  }

  CUtensorMap tk, tv;
  if (!encode_cache_map(&tk, k_cache, dims, pl.hg) || !encode_cache_map(&tv, v_cache, dims, pl.hg))
    return PD_ERR_CUDA;

  const bool fp8 = byte_kind(dims->kv_dtype);  // scaled codes
  DecodeParams p;
  p.q = static_cast<const __half*>(q);
  p.out = static_cast<__half*>(out);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.q_start = q_start;
  p.total_q = total_q;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.n_merge = static_cast<int>(pl.n_merge);
  p.decode_grid = pl.grid;
  p.rows_padded = pl.rows_padded;
  p.ws_ml = pl.bytes ? reinterpret_cast<float*>(ws + pl.off_ml) : nullptr;
  p.ws_o = pl.bytes ? reinterpret_cast<float*>(ws + pl.off_o) : nullptr;
  p.error_flag = error_flag;
  p.B = dims->B;
  p.qlen = qlen;
  p.Hq = dims->Hq;
  p.Hkv = dims->Hkv;
  p.G = dims->Hq / dims->Hkv;
  p.R = p.G * qlen;
  p.hg = pl.hg;
  p.hgn = dims->Hkv / pl.hg;
  p.rows_head = pl.rows_padded / pl.hg;
  p.max_blocks = dims->max_blocks_per_seq;
  p.block_size = dims->block_size;
  p.num_blocks = dims->num_blocks;
  p.tiles_per_block = dims->block_size / kTileKeys;
  p.window = window > 0 ? window : 0;
  p.num_splits = pl.splits;
  p.unit_cost = pl.unit_cost;
  const double ks = fp8 ? static_cast<double>(dims->k_scale) : 1.0;
  p.sl2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634 * ks);
  p.out_scale = fp8 ? dims->v_scale : 1.0f;
  p.out_bf16 = bf16_io(dims->kv_dtype) ? 1 : 0;
  p.timeout_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  p.inject = g_inject.load(std::memory_order_relaxed);
  p.cluster = pl.cluster;

  cudaError_t e = launch_decode(dims->D, dims->kv_dtype, pl.nt, pl.hg > 1 ? 1 : 0, tk, tv, p, pl.grid,
                                static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess && pl.n_merge > 0) {
    // pieces per split unit: about grid / units + 1 (balanced) or S (fixed);
    // many pieces -> spread a unit's dims over CTAs so threads can share pieces,
    // but keep the combine grid within one CTA per SM: those CTAs are resident
    // beside the decode grid and do their pre-wait work (the unit's piece
    // layout) while it runs, where CTAs beyond that start only as decode CTAs
    // exit and add that work to the tail (measured on GB300, D=256 GQA 6:1:
    // B = 2 / 3 / 8 15.0 / 17.6 / 28.9 -> 13.9 / 16.7 / 28.6 us, e4m3 B = 32
    // 54.1 -> 52.5, L = 32768 B = 2 47.2 -> 45.8, windowed B = 2 14.7 ->
    // 13.7; D=128 (28,4) ragged 86.5 -> 87.0; B = 1 and B = 32 unchanged)
    const long long per_unit = pl.splits == 0 ? pl.grid / (pl.units > 0 ? pl.units : 1) + 1 : pl.splits;
    int chunks = per_unit >= 16 ? dims->D / 8 : per_unit >= 4 ? dims->D / 32 : 1;
    while (chunks > 1 && pl.n_merge * chunks * pl.hg > pl.sms) chunks >>= 1;
    // units of more than four pieces: the combine that loads eight pieces'
    // partials at a time (one L2 round trip for up to eight), else the one
    // of four, which needs fewer registers (measured on GB300, D=256 GQA 6:1:
    // e4m3 B = 32 52.3 -> 50.8 us, B = 8 28.2 -> 27.9, B = 3 16.6 -> 16.4 with
    // eight; the headline's ~3.4 pieces per unit 0.3 us slower with eight)
    const int batch = per_unit > 4 ? 8 : 4;
    // a CTA's items (row, 4 dims) beyond 256: the batch-8 kernel's 512-thread
    // form gives each thread one item (e4m3 / int8 B = 32: 384 items)
    const long long items = static_cast<long long>(p.R) * (dims->D / chunks / 4);
    const int threads = items > 256 ? 512 : 256;
    e = launch_split_combine(dims->D, p, static_cast<int>(pl.n_merge), chunks, batch, threads,
                             static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? PD_OK : PD_ERR_CUDA;
}

}  // namespace

extern "C" {

pd_status decode_paged(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_table, const int32_t* seq_lens, float scale,
                       int window, int qlen, int num_splits, void* out, const pd_dims* dims,
                       void* workspace, size_t workspace_bytes, uint32_t* error_flag,
                       void* stream) {
  if (!dims) return PD_ERR_NULL;
  const long long total = static_cast<long long>(dims->B) * (qlen > 0 ? qlen : 0);
  if (total > (1ll << 31) - 1) return PD_ERR_UNSUPPORTED;
  return decode_impl(q, k_cache, v_cache, block_table, seq_lens, nullptr, static_cast<int>(total),
                     scale, window, qlen, num_splits, out, dims, workspace, workspace_bytes,
                     error_flag, stream);
}

pd_status decode_paged_varlen(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_table, const int32_t* seq_lens,
                              const int32_t* query_start_loc, int num_query_tokens, int max_qlen,
                              float scale, int window, int num_splits, void* out,
                              const pd_dims* dims, void* workspace, size_t workspace_bytes,
                              uint32_t* error_flag, void* stream) {
  if (!dims) return PD_ERR_NULL;
  if (dims->B > 0 && num_query_tokens > 0 && !query_start_loc) return PD_ERR_NULL;
  return decode_impl(q, k_cache, v_cache, block_table, seq_lens, query_start_loc,
                     num_query_tokens, scale, window, max_qlen, num_splits, out, dims, workspace,
                     workspace_bytes, error_flag, stream);
}

}  // extern "C"
