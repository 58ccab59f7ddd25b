// k_decode_c42.cu -- instantiations of the persistent decode kernel
// (decode_dev.cuh) for packed rows of up to 4 (gate/up) and 2 (down)
// 16-byte chunks per lane.
#include "decode_dev.cuh"

namespace moe {

dec::DecodeFn decode_pick_c42(int T) { return dec::pick_m<4, 2>(T); }

}  // namespace moe
