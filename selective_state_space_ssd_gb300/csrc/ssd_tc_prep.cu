// The shapes the tcgen05 kernels serve.
#include "ssd_internal.h"

namespace ssd {

// The tensor-core kernels serve Mamba-2 with bf16 io, chunk 64, head dim 64
// and state 128 (the 130M and 2.7B layer shapes); everything else runs on the
// CUDA-core kernels.  Their (chunk, head) items are indexed with 32-bit integers.
bool tc_forward_supported(const Dims& d) {
  return d.variant == kMamba2 && d.bf16 && d.L == 64 && d.P == 64 && d.N == 128 &&
         (long long)d.b * d.nc * d.H < (1ll << 31) && d.b <= 65535 && d.G <= 65535;
}
bool tc_backward_supported(const Dims& d) { return tc_forward_supported(d); }

}  // namespace ssd
