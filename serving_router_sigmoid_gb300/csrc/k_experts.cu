// k_experts.cu -- the int4 instantiations of the row-per-warp expert kernels
// (experts_dev.cuh), the ordered slot reduction, RMSNorm for the residual
// block, and the per-row int4 and int8 weight packers.
//
// Sources: reader.mx "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型" §11 (weighted
// add into the token's output), §04 (rmsnorm with double accumulation), §06
// (int4 packer), §05 (quantize_rows: per-row int8 weights); besthub.dev
// "Running 744B MoE on 25GB RAM" §06, §11.
#include "experts_dev.cuh"

namespace moe {

// ---------------------------------------------------------------- reduce

// out[t] = (resid[t] +) sum_k w[t,k] * y[t,k] + y[t,shared], slots in order
// (slots adaptive top-p dropped are skipped).
// Every slot's value is loaded before the first add (K <= KB: the register
// arrays hold KB routed slots, so a layer with a small K keeps the
// occupancy high enough for the loads in flight this HBM-bound step needs).
template <int KB>
__global__ void __launch_bounds__(256) reduce_kernel(LayerArgs a) {
    const int t = blockIdx.y;
    const int o = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (o >= a.D) return;
    const int K = a.K, S = a.S, D = a.D;
    const float *pt = a.part + (size_t)t * S * D + o;
    float4 y[KB + 1];
    float wk[KB];
    bool kept[KB];  // a slot top-p dropped has no expert output
#pragma unroll
    for (int k = 0; k <= KB; ++k) {
        if (k < S) y[k] = *reinterpret_cast<const float4 *>(pt + (size_t)k * D);
        if (k < K && k < KB) {
            wk[k] = a.wts[t * K + k];
            kept[k] = a.idx[t * K + k] != kDroppedSel;
        }
    }
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.resid) r = *reinterpret_cast<const float4 *>(a.resid + (size_t)t * D + o);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < KB; ++k) {
        if (k < K && kept[k]) {
            acc.x = __fadd_rn(acc.x, __fmul_rn(wk[k], y[k].x));
            acc.y = __fadd_rn(acc.y, __fmul_rn(wk[k], y[k].y));
            acc.z = __fadd_rn(acc.z, __fmul_rn(wk[k], y[k].z));
            acc.w = __fadd_rn(acc.w, __fmul_rn(wk[k], y[k].w));
        }
    }
    if (a.n_shared) {
#pragma unroll
        for (int k = 0; k <= KB; ++k) {
            if (k == K) {
                acc.x = __fadd_rn(acc.x, y[k].x);
                acc.y = __fadd_rn(acc.y, y[k].y);
                acc.z = __fadd_rn(acc.z, y[k].z);
                acc.w = __fadd_rn(acc.w, y[k].w);
            }
        }
    }
    if (a.resid) {
        acc.x = __fadd_rn(r.x, acc.x);
        acc.y = __fadd_rn(r.y, acc.y);
        acc.z = __fadd_rn(r.z, acc.z);
        acc.w = __fadd_rn(r.w, acc.w);
    }
    *reinterpret_cast<float4 *>(a.out + (size_t)t * D + o) = acc;
}

// --------------------------------------------------------------- rmsnorm

// reader.mx article §04: ms = sum x^2 in double; r = 1/sqrtf((float)(ms/D)+eps);
// out = x*r*w in fp32.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float *__restrict__ x, const float *__restrict__ w,
                                                      float eps, float *__restrict__ out, int D) {
    __shared__ double red[32];
    __shared__ float s_r;
    const float *row = x + (size_t)blockIdx.x * D;
    double ms = 0.0;
    for (int i = threadIdx.x; i < D; i += blockDim.x) ms += (double)row[i] * (double)row[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ms += __shfl_xor_sync(0xffffffffu, ms, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ms;
    __syncthreads();
    if (threadIdx.x < 32) {
        double v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (threadIdx.x == 0) s_r = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn((float)(v / D), eps)));
    }
    __syncthreads();
    const float r = s_r;
    for (int i = threadIdx.x; i < D; i += blockDim.x)
        out[(size_t)blockIdx.x * D + i] = __fmul_rn(__fmul_rn(row[i], r), w[i]);
}

// ------------------------------------------------------------------ pack

// reader.mx article §06: s = max(amax/7, 1e-8); v = nearest integer of w/s
// (IEEE division, ties to even) clamped to [-8, 7]; byte j = (v[2j]+8) |
// (v[2j+1]+8) << 4; odd rows pad the last high nibble with 8.
__global__ void __launch_bounds__(256) pack_int4_kernel(const float *__restrict__ w, uint8_t *__restrict__ q4,
                                                        float *__restrict__ scale, long long I) {
    __shared__ float red[32];
    const long long o = blockIdx.x;
    const float *row = w + o * I;
    float amax = 0.f;
    for (long long i = threadIdx.x; i < I; i += blockDim.x) amax = fmaxf(amax, fabsf(row[i]));
    amax = block_max_nonneg(amax, red);
    float s = __fdiv_rn(amax, 7.f);
    if (s < 1e-8f) s = 1e-8f;
    const long long nb = (I + 1) >> 1;
    for (long long j = threadIdx.x; j < nb; j += blockDim.x) {
        int v0 = __float2int_rn(__fdiv_rn(row[2 * j], s));
        v0 = min(7, max(-8, v0));
        int v1 = 0;
        if (2 * j + 1 < I) {
            v1 = __float2int_rn(__fdiv_rn(row[2 * j + 1], s));
            v1 = min(7, max(-8, v1));
        }
        q4[o * nb + j] = (uint8_t)((v0 + 8) | ((v1 + 8) << 4));
    }
    if (threadIdx.x == 0) scale[o] = s;
}

// reader.mx article §05 quantize_rows with bits = 8: s = max(amax/127, 1e-8);
// v = nearest integer of w/s (IEEE division, ties to even) clamped to
// [-128, 127], one int8 per value, natural order.
__global__ void __launch_bounds__(256) pack_int8_kernel(const float *__restrict__ w, int8_t *__restrict__ q8,
                                                        float *__restrict__ scale, long long I) {
    __shared__ float red[32];
    const long long o = blockIdx.x;
    const float *row = w + o * I;
    float amax = 0.f;
    for (long long i = threadIdx.x; i < I; i += blockDim.x) amax = fmaxf(amax, fabsf(row[i]));
    amax = block_max_nonneg(amax, red);
    float s = __fdiv_rn(amax, 127.f);
    if (s < 1e-8f) s = 1e-8f;
    for (long long i = threadIdx.x; i < I; i += blockDim.x)
        q8[o * I + i] = (int8_t)min(127, max(-128, __float2int_rn(__fdiv_rn(row[i], s))));
    if (threadIdx.x == 0) scale[o] = s;
}

// ---------------------------------------------------------- launchers

int mch_index(int mch) { return mch <= 1 ? 0 : mch <= 2 ? 1 : mch <= 4 ? 2 : 3; }

static int cpl_for(int n) {  // chunks per lane for a row of n int4 values
    const int ch = (n + 1023) / 1024;
    return ch <= 1 ? 1 : ch <= 2 ? 2 : ch <= 4 ? 4 : ch <= 6 ? 6 : 8;
}

template <int CPL, int MCH>
static void *gateup_ptr() { return (void *)gateup_kernel<CPL, MCH, 4>; }
template <int CPL, int MCH, bool F>
static void *down_ptr() { return (void *)down_kernel<CPL, MCH, F, 4>; }

#define MOE_CPL_SWITCH(cpl, MCH, EXPR_T)                 \
    switch (cpl) {                                        \
        case 1: { constexpr int C = 1; EXPR_T; } break;   \
        case 2: { constexpr int C = 2; EXPR_T; } break;   \
        case 4: { constexpr int C = 4; EXPR_T; } break;   \
        case 6: { constexpr int C = 6; EXPR_T; } break;   \
        default: { constexpr int C = 8; EXPR_T; } break;  \
    }

#define MOE_MCH_SWITCH(mch, EXPR_M)                       \
    switch (mch_index(mch)) {                             \
        case 0: { constexpr int M_ = 1; EXPR_M; } break;  \
        case 1: { constexpr int M_ = 2; EXPR_M; } break;  \
        case 2: { constexpr int M_ = 4; EXPR_M; } break;  \
        default: { constexpr int M_ = 8; EXPR_M; } break; \
    }

cudaError_t launch_gateup(const LayerArgs &a, int mch, int grid, cudaStream_t s) {
    if (a.wbits == 8) return launch_gateup8(a, mch, grid, s);
    const int cpl = cpl_for(a.D);
    MOE_MCH_SWITCH(mch, MOE_CPL_SWITCH(cpl, M_, (gateup_kernel<C, M_, 4><<<grid, 256, 0, s>>>(a))))
    return cudaGetLastError();
}

cudaError_t launch_down(const LayerArgs &a, int mch, int grid, bool fused, cudaStream_t s) {
    if (a.wbits == 8) return launch_down8(a, mch, grid, fused, s);
    const int cpl = cpl_for(a.I);
    const size_t smem = (size_t)(1 << mch_index(mch)) * a.I;
    if (fused) {
        MOE_MCH_SWITCH(mch, MOE_CPL_SWITCH(cpl, M_, (down_kernel<C, M_, true, 4><<<grid, 256, smem, s>>>(a))))
    } else {
        MOE_MCH_SWITCH(mch, MOE_CPL_SWITCH(cpl, M_, (down_kernel<C, M_, false, 4><<<grid, 256, smem, s>>>(a))))
    }
    return cudaGetLastError();
}

cudaError_t launch_reduce(const LayerArgs &a, cudaStream_t s) {
    dim3 grid((a.D / 4 + 255) / 256, a.T);
    if (a.K <= 4)
        reduce_kernel<4><<<grid, 256, 0, s>>>(a);
    else if (a.K <= 8)
        reduce_kernel<8><<<grid, 256, 0, s>>>(a);
    else
        reduce_kernel<kMaxK><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const float *x, const float *w, float eps, float *out, int T, int D, cudaStream_t s) {
    rmsnorm_kernel<<<T, 256, 0, s>>>(x, w, eps, out, D);
    return cudaGetLastError();
}

cudaError_t launch_pack_int4(const float *w, uint8_t *q4, float *scale, int64_t O, int64_t I, cudaStream_t s) {
    // one CTA per row; rows beyond the 2^31-1 grid limit go in further launches
    const int64_t step = 0x7fffffff;
    for (int64_t o0 = 0; o0 < O; o0 += step) {
        const int64_t n = (O - o0) < step ? (O - o0) : step;
        pack_int4_kernel<<<(unsigned)n, 256, 0, s>>>(w + o0 * I, q4 + o0 * ((I + 1) / 2), scale + o0, I);
        cudaError_t ce = cudaGetLastError();
        if (ce != cudaSuccess) return ce;
    }
    return cudaSuccess;
}

cudaError_t launch_pack_int8(const float *w, int8_t *q8, float *scale, int64_t O, int64_t I, cudaStream_t s) {
    const int64_t step = 0x7fffffff;
    for (int64_t o0 = 0; o0 < O; o0 += step) {
        const int64_t n = (O - o0) < step ? (O - o0) : step;
        pack_int8_kernel<<<(unsigned)n, 256, 0, s>>>(w + o0 * I, q8 + o0 * I, scale + o0, I);
        cudaError_t ce = cudaGetLastError();
        if (ce != cudaSuccess) return ce;
    }
    return cudaSuccess;
}

// Grid sizes: resident CTAs per SM (occupancy) x SMs, for every MCH variant.
cudaError_t prepare_expert_kernels(int D, int I, int num_sms, int grid_gu[4], int grid_dn[4]) {
    const int cg = cpl_for(D), cd = cpl_for(I);
    for (int mi = 0; mi < 4; ++mi) {
        const int mch = 1 << mi;
        void *fg = nullptr, *fd = nullptr, *fdf = nullptr;
        MOE_MCH_SWITCH(mch, MOE_CPL_SWITCH(cg, M_, (fg = gateup_ptr<C, M_>())))
        MOE_MCH_SWITCH(mch, MOE_CPL_SWITCH(cd, M_, (fd = down_ptr<C, M_, false>())))
        MOE_MCH_SWITCH(mch, MOE_CPL_SWITCH(cd, M_, (fdf = down_ptr<C, M_, true>())))
        const int smem = mch * I;
        // the attribute belongs to the instantiation, which layers of other
        // sizes share: set it to the largest tile any of them can need
        const int smem_max = mch * kMaxDim;
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
