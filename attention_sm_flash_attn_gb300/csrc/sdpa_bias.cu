// sdpa_bias.cu -- the attention kernels that add an additive bias (a mask
// array) to the scores, instantiated in a translation unit of their own so that
// they compile in parallel with the others (sdpa_api.cu).  The host side of the
// bias (validation, strides) is in sdpa_api.cu.
#include "sdpa_launch.cuh"

namespace gbsdpa_host {

int launch_bias_variant(bool bf16, int mode, int D, int Dv, const AttnParams& p, long long items,
                        cudaStream_t stream, DeviceState* st) {
  return bf16 ? launch_variant<true, true>(mode, D, Dv, p, items, stream, st)
              : launch_variant<false, true>(mode, D, Dv, p, items, stream, st);
}

int resident_bias_variant(bool bf16, int mode, int D, int Dv, DeviceState* st) {
  return bf16 ? resident_variant<true, true>(mode, D, Dv, st)
              : resident_variant<false, true>(mode, D, Dv, st);
}

}  // namespace gbsdpa_host
