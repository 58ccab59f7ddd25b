// k_decode_c11.cu -- instantiations of the persistent decode kernel
// (decode_dev.cuh) for packed rows of up to 1 (gate/up) and 1 (down)
// 16-byte chunks per lane.
#include "decode_dev.cuh"

namespace moe {

dec::DecodeFn decode_pick_c11(int T) { return dec::pick_m<1, 1>(T); }

}  // namespace moe
