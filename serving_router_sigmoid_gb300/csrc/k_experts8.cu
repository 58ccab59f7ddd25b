// k_experts8.cu -- the int8-weight instantiations of the row-per-warp expert
// kernels (experts_dev.cuh): the layer's experts stored as per-row int8
// (reader.mx "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型" §05 quantize_rows, §12
// matmul_q_idot: int8 weights x int8 activations, exact integer dot).  A
// separate translation unit so the two weight widths compile in parallel.
#include "experts_dev.cuh"

namespace moe {

namespace {

int cpl8_for(int n) {  // 16-byte chunks per lane for a row of n int8 values
    const int ch = (n + 511) / 512;
    return ch <= 2 ? 2 : ch <= 4 ? 4 : ch <= 8 ? 8 : ch <= 12 ? 12 : 16;
}

int mch8_index(int mch) { return mch <= 1 ? 0 : mch <= 2 ? 1 : mch <= 4 ? 2 : 3; }

#define MOE_CPL8_SWITCH(cpl, EXPR_T)                       \
    switch (cpl) {                                          \
        case 2: { constexpr int C = 2; EXPR_T; } break;     \
        case 4: { constexpr int C = 4; EXPR_T; } break;     \
        case 8: { constexpr int C = 8; EXPR_T; } break;     \
        case 12: { constexpr int C = 12; EXPR_T; } break;   \
        default: { constexpr int C = 16; EXPR_T; } break;   \
    }

#define MOE_MCH8_SWITCH(mch, EXPR_M)                       \
    switch (mch8_index(mch)) {                             \
        case 0: { constexpr int M_ = 1; EXPR_M; } break;   \
        case 1: { constexpr int M_ = 2; EXPR_M; } break;   \
        case 2: { constexpr int M_ = 4; EXPR_M; } break;   \
        default: { constexpr int M_ = 8; EXPR_M; } break;  \
    }

}  // namespace

cudaError_t launch_gateup8(const LayerArgs &a, int mch, int grid, cudaStream_t s) {
    const int cpl = cpl8_for(a.D);
    MOE_MCH8_SWITCH(mch, MOE_CPL8_SWITCH(cpl, (gateup_kernel<C, M_, 8><<<grid, 256, 0, s>>>(a))))
    return cudaGetLastError();
}

cudaError_t launch_down8(const LayerArgs &a, int mch, int grid, bool fused, cudaStream_t s) {
    const int cpl = cpl8_for(a.I);
    const size_t smem = (size_t)(1 << mch8_index(mch)) * a.I;
    if (fused) {
        MOE_MCH8_SWITCH(mch, MOE_CPL8_SWITCH(cpl, (down_kernel<C, M_, true, 8><<<grid, 256, smem, s>>>(a))))
    } else {
        MOE_MCH8_SWITCH(mch, MOE_CPL8_SWITCH(cpl, (down_kernel<C, M_, false, 8><<<grid, 256, smem, s>>>(a))))
    }
    return cudaGetLastError();
}

// Grid sizes of the int8 instantiations: resident CTAs per SM x SMs.
cudaError_t prepare_expert_kernels8(int D, int I, int num_sms, int grid_gu[4], int grid_dn[4]) {
    const int cg = cpl8_for(D), cd = cpl8_for(I);
    for (int mi = 0; mi < 4; ++mi) {
        const int mch = 1 << mi;
        void *fg = nullptr, *fd = nullptr, *fdf = nullptr;
        MOE_MCH8_SWITCH(mch, MOE_CPL8_SWITCH(cg, (fg = (void *)gateup_kernel<C, M_, 8>)))
        MOE_MCH8_SWITCH(mch, MOE_CPL8_SWITCH(cd, (fd = (void *)down_kernel<C, M_, false, 8>)))
        MOE_MCH8_SWITCH(mch, MOE_CPL8_SWITCH(cd, (fdf = (void *)down_kernel<C, M_, true, 8>)))
        const int smem = mch * I, smem_max = mch * kMaxDim;
        cudaError_t ce;
        if ((ce = cudaFuncSetAttribute(fd, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max)) != cudaSuccess)
            return ce;
        if ((ce = cudaFuncSetAttribute(fdf, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max)) != cudaSuccess)
            return ce;
        int og = 0, od = 0;
        if ((ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&og, fg, 256, 0)) != cudaSuccess) return ce;
        if ((ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&od, fd, 256, smem)) != cudaSuccess) return ce;
        og = og < 1 ? 1 : (og > 8 ? 8 : og);
        od = od < 1 ? 1 : (od > 8 ? 8 : od);
        grid_gu[mi] = og * num_sms;
        grid_dn[mi] = od * num_sms;
    }
    return cudaSuccess;
}

}  // namespace moe
