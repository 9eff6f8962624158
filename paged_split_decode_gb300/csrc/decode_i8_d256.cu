// decode_i8_d256.cu -- instantiations of the decode kernel for int8 KV, D=256.
// NT = row tiles of 8 query rows (rows per unit = Hq/Hkv * qlen <= 8*NT);
// KG = key groups (consumer warps per row tile); two CTAs share each SM, so
// two producers keep the SM's TMA traffic flowing; the ring takes as many
// stages as half an SM's shared memory allows.
#include "launch.h"

namespace pd {
namespace {
constexpr int kKv = kKvInt8;
constexpr int kD = 256;
using C1 = CfgFor<kD, kKv, 1, 2, 2>;
using C2 = CfgFor<kD, kKv, 2, 1, 2>;
using C3 = CfgFor<kD, kKv, 3, 1, 2>;
using C4 = CfgFor<kD, kKv, 4, 1, 2>;
}  // namespace

bool shape_i8_d256(int nt, KernelShape* out) {
  switch (nt) {
    case 1: return shape_of<C1>(out);
    case 2: return shape_of<C2>(out);
    case 3: return shape_of<C3>(out);
    case 4: return shape_of<C4>(out);
    default: return false;
  }
}

cudaError_t launch_i8_d256(int nt, const CUtensorMap& tk, const CUtensorMap& tv,
                            const DecodeParams& p, int grid, cudaStream_t s) {
  switch (nt) {
    case 1: return launch_cfg<C1>(tk, tv, p, grid, s);
    case 2: return launch_cfg<C2>(tk, tv, p, grid, s);
    case 3: return launch_cfg<C3>(tk, tv, p, grid, s);
    case 4: return launch_cfg<C4>(tk, tv, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pd
