// k_decode_c21.cu -- instantiations of the persistent decode kernel
// (decode_dev.cuh) for packed rows of up to 2 (gate/up) and 1 (down)
// 16-byte chunks per lane.
#include "decode_dev.cuh"

namespace moe {

dec::DecodeFn decode_pick_c21(int T) { return dec::pick_m<2, 1>(T); }

}  // namespace moe
