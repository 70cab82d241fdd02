// The shapes the tcgen05 kernels serve.
#include "ssd_internal.h"

namespace ssd {

// The tensor-core kernels serve bf16 io with head dim 64 and state 128: Mamba-2
// with chunk 64 (the 130M and 2.7B layer shapes), and MIMO with a power-of-two
// rank R <= 64 (any chunk; they cut the fused sequence into chunks of 64
// positions, 64 / R steps, which changes nothing but the summation order).
// Everything else runs on the CUDA-core kernels.  Their (chunk, head) items
// are indexed with 32-bit integers.
Dims tc_dims(const Dims& d) {
  Dims f = d;
  if (d.variant != kMimo) return f;
  int rs = 0;
  while ((1 << rs) < d.R) ++rs;
  f.rs = rs;
  f.T = d.T * d.R;
  f.L = 64;
  f.nc = (f.T + 63) / 64;
  f.R = 1;
  f.LR = 64;
  f.G = d.H;
  f.hpg = 1;
  return f;
}

bool tc_forward_supported(const Dims& d) {
  if (!d.bf16 || d.P != 64 || d.N != 128) return false;
  if (d.variant == kMamba2) {
    if (d.L != 64) return false;
  } else if (d.variant == kMimo) {
    if (d.R > 64 || (d.R & (d.R - 1)) != 0 || (long long)d.T * d.R > 0x3fffffffll) return false;
  } else {
    return false;
  }
  const Dims f = tc_dims(d);
  return (long long)f.b * f.nc * f.H < (1ll << 31) && f.b <= 65535 && f.G <= 65535;
}
bool tc_backward_supported(const Dims& d) { return tc_forward_supported(d); }

}  // namespace ssd
