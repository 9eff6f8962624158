// decode_i8_d256.cu -- instantiations of the decode kernel for int8 KV, D=256.
// NT = row tiles of 8 query rows per KV head (rows per head = Hq/Hkv * qlen
// <= 8*NT); KG = key groups (consumer warps per row tile). Per-head tiles
// (HG = 1): two CTAs share each SM, so two producers keep the SM's TMA
// traffic flowing. Head-group tiles (C1H, NT = 1, Hkv a multiple of 4): a
// tile holds 16 keys of HG consecutive KV heads -- one contiguous run of the
// cache per key -- and one CTA per SM holds a deep ring of them; each head has
// its own consumer warps (DS of them splitting D). The ring takes as many
// stages as the shared memory allows. The head-group shapes are the ones that
// measured fastest on GB300.
#include "launch.h"

namespace pd {
namespace {
constexpr int kD = 256;
// The shapes for caches of this kind, with an fp16 q (kKv = kKvInt8) or a
// bfloat16 q and out (kKvInt8Bq).
template <int kKv>
struct Shapes {
  using C1 = CfgFor<kD, kKv, 1, 2, 2>;
  using C2 = CfgFor<kD, kKv, 2, 1, 2, 1, 1, 2>;
  using C3 = CfgFor<kD, kKv, 3, 1, 2, 1, 1, 3>;
  using C4 = CfgFor<kD, kKv, 4, 1, 2, 1, 1, 4>;
  using C1H = CfgFor<kD, kKv, 1, 1, 1, 1, 4>;

  static bool shape(int nt, int grouped, KernelShape* out) {
    if (grouped) return nt == 1 && shape_of<C1H>(out);
    switch (nt) {
      case 1: return shape_of<C1>(out);
      case 2: return shape_of<C2>(out);
      case 3: return shape_of<C3>(out);
      case 4: return shape_of<C4>(out);
      default: return false;
    }
  }

  static cudaError_t launch(int nt, int grouped, const CUtensorMap& tk, const CUtensorMap& tv,
                            const DecodeParams& p, int grid, cudaStream_t s) {
    if (grouped) return nt == 1 ? launch_cfg<C1H>(tk, tv, p, grid, s) : cudaErrorInvalidValue;
    switch (nt) {
      case 1: return launch_cfg<C1>(tk, tv, p, grid, s);
      case 2: return launch_cfg<C2>(tk, tv, p, grid, s);
      case 3: return launch_cfg<C3>(tk, tv, p, grid, s);
      case 4: return launch_cfg<C4>(tk, tv, p, grid, s);
      default: return cudaErrorInvalidValue;
    }
  }
};
}  // namespace

bool shape_i8_d256(int nt, int grouped, KernelShape* out) {
  return Shapes<kKvInt8>::shape(nt, grouped, out);
}
bool shape_i8q_d256(int nt, int grouped, KernelShape* out) {
  return Shapes<kKvInt8Bq>::shape(nt, grouped, out);
}
cudaError_t launch_i8_d256(int nt, int grouped, const CUtensorMap& tk, const CUtensorMap& tv,
                          const DecodeParams& p, int grid, cudaStream_t s) {
  return Shapes<kKvInt8>::launch(nt, grouped, tk, tv, p, grid, s);
}
cudaError_t launch_i8q_d256(int nt, int grouped, const CUtensorMap& tk, const CUtensorMap& tv,
                           const DecodeParams& p, int grid, cudaStream_t s) {
  return Shapes<kKvInt8Bq>::launch(nt, grouped, tk, tv, p, grid, s);
}

}  // namespace pd
