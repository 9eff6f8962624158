// decode_i8_d256.cu -- instantiations of the decode kernel for int8 KV, D=256.
// NT = row tiles of 8 query rows per KV head (rows per head = Hq/Hkv * qlen
// <= 8*NT); KG = key groups (consumer warps per row tile). Per-head tiles
// (HG = 1): two CTAs share each SM, so two producers keep the SM's TMA
// traffic flowing. Head-group tiles (C1H, NT = 1, Hkv a multiple of 4): a
// tile holds 16 keys of HG consecutive KV heads -- one contiguous run of the
// cache per key -- and one CTA per SM holds a deep ring of them; each head has
// its own consumer warps (DS of them splitting D). The ring takes as many
// stages as the shared memory allows. The head-group shapes are the ones that
// measured fastest on GB300. Units of 9 to 32 query rows per KV head (two to
// four row tiles) run on the tensor-memory kernel of decode_tci8.cuh instead:
// the int8 codes are widened exactly to fp16 operands of tcgen05.mma
// kind::f16.
#include "decode_tci8.cuh"

namespace pd {
namespace {
constexpr int kD = 256;
// The shapes for caches of this kind, with an fp16 q (kKv = kKvInt8) or a
// bfloat16 q and out (kKvInt8Bq).
template <int kKv>
struct Shapes {
  using C1 = CfgFor<kD, kKv, 1, 2, 2>;
  // two to four row tiles: the tensor-core (tcgen05) kernel, one softmax
  // warpgroup per row tile
  template <int NG>
  using TC = Tci8<kD, q_is_bf16(kKv), NG>;
  using C1H = CfgFor<kD, kKv, 1, 1, 1, 1, 4>;

  static bool shape(int nt, int grouped, KernelShape* out) {
    if (grouped) return nt == 1 && shape_of<C1H>(out);
    switch (nt) {
      case 1: return shape_of<C1>(out);
      case 2: return shape_tci8<TC<2>>(nt, out);
      case 3: return shape_tci8<TC<3>>(nt, out);
      case 4: return shape_tci8<TC<4>>(nt, out);
      default: return false;
    }
  }

  static cudaError_t launch(int nt, int grouped, const CUtensorMap& tk, const CUtensorMap& tv,
                            const DecodeParams& p, int grid, cudaStream_t s) {
    if (grouped) return nt == 1 ? launch_cfg<C1H>(tk, tv, p, grid, s) : cudaErrorInvalidValue;
    switch (nt) {
      case 1: return launch_cfg<C1>(tk, tv, p, grid, s);
      case 2: return launch_tci8<TC<2>>(tk, tv, p, grid, s);
      case 3: return launch_tci8<TC<3>>(tk, tv, p, grid, s);
      case 4: return launch_tci8<TC<4>>(tk, tv, p, grid, s);
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
