// k_decode.cu -- launch of the persistent single-kernel decode layer
// (decode_dev.cuh): the instantiation that covers the layer's sizes, its
// cooperative grid and the launch itself.
#include "decode_dev.cuh"

namespace moe {

namespace {

using dec::DecodeFn;

int cpl_need(int kdim) { return (kdim / 32 + 31) / 32; }  // 16-byte chunks per lane of one packed row

// The smallest instantiated (gate/up, down) chunk counts covering D and I;
// nullptr when none does (I above 2048 or D above 6144).
DecodeFn pick(const LayerArgs &a) {
    const int cg = cpl_need(a.D), cd = cpl_need(a.I);
    if (a.T < 1 || a.T > kSmallT) return nullptr;
    if (cg <= 1 && cd <= 1) return decode_pick_c11(a.T);
    if (cg <= 2 && cd <= 1) return decode_pick_c21(a.T);
    if (cg <= 4 && cd <= 2) return decode_pick_c42(a.T);
    if (cg <= 6 && cd <= 2) return decode_pick_c62(a.T);
    return nullptr;
}

int mch_of(int T) { return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : T <= 8 ? 8 : 16; }

size_t smem_of(const LayerArgs &a) { return (size_t)mch_of(a.T) * (a.D > a.I ? a.D : a.I); }

}  // namespace

cudaError_t decode_grid(const LayerArgs &a, int num_sms, int *grid) {
    *grid = 0;
    DecodeFn fn = pick(a);
    if (!fn || !stream_supported(a.D, a.I) || a.K * a.T > 256) return cudaSuccess;
    int coop = 0, dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (ce != cudaSuccess || !coop) return ce;
    // the attribute belongs to the instantiation, which handles of other sizes
    // share: set it to the largest tile any of them can need
    const size_t smem = smem_of(a);
    ce = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, mch_of(a.T) * kMaxDim);
    if (ce != cudaSuccess) return ce;
    int occ = 0;
    ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, 256, smem);
    if (ce != cudaSuccess) return ce;
    occ = occ > 2 ? 2 : occ;
    // the quantiser CTAs are the last T; they must not be fewer than T
    if (occ >= 1 && num_sms * occ >= a.T) *grid = num_sms * occ;
    return cudaSuccess;
}

cudaError_t launch_decode_layer(const LayerArgs &a, int grid, cudaStream_t s) {
    DecodeFn fn = pick(a);
    if (!fn || grid < 1) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem_of(a);
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    // the kernel waits (griddepcontrol.wait) before it reads anything the
    // previous kernel in the stream writes, so it may start early
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, fn, a);
}

}  // namespace moe
