// k_experts.cu -- the expert kernels of the routed-MoE layer: fused int4
// gate/up + SiLU*up, down projection with the expert-output scatter, the
// ordered slot reduction, and RMSNorm for the residual block.
//
// Sources: reader.mx "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型" §11 (SwiGLU
// expert: gate/up, siluf(g)*u, down, weighted add into the token's output),
// §12 (int8 activations x int4 weights with an exact integer dot, then the
// activation and row scales), §04 (siluf, rmsnorm with double accumulation);
// besthub.dev "Running 744B MoE on 25GB RAM" §11, §12.
//
// Decode-sized batches stream each union expert's packed rows once: every
// warp owns whole output rows, reads them with 16-byte streaming loads (no L1
// allocation) and multiplies them against the int8 activations of all rows
// routed to that expert.  Offset nibbles n = v + 8 go straight into dp4a;
// sum((n-8) x) = sum(n x) - 8 sum(x) restores the signed dot exactly.
#include "layer_args.cuh"

namespace moe {

// Contiguous share [beg, end) of n_items for this CTA, so consecutive items
// of a CTA mostly belong to the same expert.
__device__ __forceinline__ void item_range(int n_items, int &beg, int &end) {
    beg = (int)(((long long)blockIdx.x * n_items) / gridDim.x);
    end = (int)(((long long)(blockIdx.x + 1) * n_items) / gridDim.x);
}

// ------------------------------------------------------------- gate / up

// Item = (union entry u, block of rpi_gu gate/up output rows).  Each warp
// takes rpi_gu/8 rows.  For each chunk of up to MCH token rows of the expert
// it computes the int32 gate and up dots, h = silu(g)*u in fp32, stores h and
// raises the row's max|h| (bit pattern of a non-negative float, so an
// integer atomicMax is exact and order-independent).
template <int CPL, int MCH>
__global__ void __launch_bounds__(256) gateup_kernel(LayerArgs a) {
    __shared__ unsigned s_amax[MCH];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = a.D, I = a.I, S = a.S;
    const int nch = D >> 5;         // 16-byte weight chunks per row
    const size_t rowb = (size_t)(D >> 1);
    const int rpw = a.rpi_gu >> 3;  // rows per warp
    int beg, end;
    item_range(a.meta->n_gu_items, beg, end);

    for (int item = beg; item < end; ++item) {
        const int u = item / a.nb_gu, b = item - u * a.nb_gu;
        const int e = a.meta->uexp[u], r0 = a.meta->ubeg[u], M = a.meta->ubeg[u + 1] - r0;
        const DevExpert ex = a.experts[e];
        for (int m0 = 0; m0 < M; m0 += MCH) {
            const int mc = min(MCH, M - m0);
            int tk[MCH], xsm[MCH], ent[MCH];
            float sxv[MCH];
#pragma unroll
            for (int m = 0; m < MCH; ++m) {
                if (m < mc) {
                    ent[m] = a.rows[r0 + m0 + m];
                    tk[m] = ent[m] / S;
                    xsm[m] = a.xsum[tk[m]];
                    sxv[m] = a.sx[tk[m]];
                } else {
                    ent[m] = tk[m] = xsm[m] = 0;
                    sxv[m] = 0.f;
                }
            }
            __syncthreads();
            if (threadIdx.x < MCH) s_amax[threadIdx.x] = 0u;
            __syncthreads();

            for (int j = 0; j < rpw; ++j) {
                const int o = b * a.rpi_gu + warp * rpw + j;
                if (o >= I) break;
                const uint8_t *grow = ex.gq + (size_t)o * rowb;
                const uint8_t *urow = ex.uq + (size_t)o * rowb;
                int4 gw[CPL], uw[CPL];
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    const int ch = lane + 32 * c;
                    if (ch < nch) {
                        gw[c] = ld_stream16(grow + (size_t)ch * 16);
                        uw[c] = ld_stream16(urow + (size_t)ch * 16);
                    }
                }
                int ag[MCH], au[MCH];
#pragma unroll
                for (int m = 0; m < MCH; ++m) ag[m] = au[m] = 0;
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    const int ch = lane + 32 * c;
                    if (ch < nch) {
#pragma unroll
                        for (int m = 0; m < MCH; ++m) {
                            if (m < mc) {
                                const int4 *xp = reinterpret_cast<const int4 *>(a.xq + (size_t)tk[m] * D + (size_t)ch * 32);
                                const int4 x0 = __ldg(xp), x1 = __ldg(xp + 1);
                                int g = ag[m], q = au[m];
                                g = dot_word((uint32_t)gw[c].x, x0.x, x0.y, g);
                                q = dot_word((uint32_t)uw[c].x, x0.x, x0.y, q);
                                g = dot_word((uint32_t)gw[c].y, x0.z, x0.w, g);
                                q = dot_word((uint32_t)uw[c].y, x0.z, x0.w, q);
                                g = dot_word((uint32_t)gw[c].z, x1.x, x1.y, g);
                                q = dot_word((uint32_t)uw[c].z, x1.x, x1.y, q);
                                g = dot_word((uint32_t)gw[c].w, x1.z, x1.w, g);
                                q = dot_word((uint32_t)uw[c].w, x1.z, x1.w, q);
                                ag[m] = g;
                                au[m] = q;
                            }
                        }
                    }
                }
                // every lane gets every row's sums; lane m finishes row m
                int myg = 0, myu = 0, myxs = 0, myent = 0;
                float mysx = 0.f;
#pragma unroll
                for (int m = 0; m < MCH; ++m) {
                    if (m < mc) {
                        const int g = warp_sum_i(ag[m]);
                        const int q = warp_sum_i(au[m]);
                        if (lane == m) {
                            myg = g; myu = q; myxs = xsm[m]; mysx = sxv[m]; myent = ent[m];
                        }
                    }
                }
                if (lane < mc) {
                    const int gi = myg - 8 * myxs, ui = myu - 8 * myxs;
                    const float gf = __fmul_rn(__fmul_rn((float)gi, mysx), __ldg(ex.gs + o));
                    const float uf = __fmul_rn(__fmul_rn((float)ui, mysx), __ldg(ex.us + o));
                    const float hv = __fmul_rn(silu_f(gf), uf);
                    const int r = r0 + m0 + lane;
                    a.h[(size_t)r * I + o] = hv;
                    atomicMax(&s_amax[lane], __float_as_uint(fabsf(hv)));
                    if (a.dbg.gate_acc) a.dbg.gate_acc[(size_t)myent * I + o] = gi;
                    if (a.dbg.up_acc) a.dbg.up_acc[(size_t)myent * I + o] = ui;
                }
            }
            __syncthreads();
            if (threadIdx.x < mc) atomicMax(a.hamax + r0 + m0 + threadIdx.x, s_amax[threadIdx.x]);
        }
    }
}

// ------------------------------------------------------------------ down

// Item = (union entry u, block of rpi_dn output rows of D).  The CTA first
// requantises the expert's h rows to int8 (qrow_i8 with the row amax from
// the gate/up pass) into shared memory in the even/odd layout, then each warp
// streams rpi_dn/8 down rows.  y = ((float)acc * sh) * sd[o] goes to
// part[entry, o].  With FUSED the last CTA to finish a row block (arrival
// counter, no waiting) sums that block's slots for every token.
template <int CPL, int MCH, bool FUSED>
__global__ void __launch_bounds__(256) down_kernel(LayerArgs a) {
    extern __shared__ __align__(16) int8_t hq_s[];  // [MCH][I]
    __shared__ int s_hsum[MCH];
    __shared__ float s_sh[MCH];
    __shared__ int s_ent[MCH];
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = a.D, I = a.I;
    const int nch = I >> 5;
    const size_t rowb = (size_t)(I >> 1);
    const int rpw = a.rpi_dn >> 3;
    int beg, end;
    item_range(a.meta->n_dn_items, beg, end);
    int staged_u = -1, staged_m0 = -1;

    for (int item = beg; item < end; ++item) {
        const int u = item / a.nb_dn, b = item - u * a.nb_dn;
        const int e = a.meta->uexp[u], r0 = a.meta->ubeg[u], M = a.meta->ubeg[u + 1] - r0;
        const DevExpert ex = a.experts[e];
        for (int m0 = 0; m0 < M; m0 += MCH) {
            const int mc = min(MCH, M - m0);
            if (u != staged_u || m0 != staged_m0) {
                __syncthreads();
                if (threadIdx.x < MCH) s_hsum[threadIdx.x] = 0;
                if (threadIdx.x < mc) {
                    const int r = r0 + m0 + threadIdx.x;
                    float s, inv;
                    act_scale(__uint_as_float(__ldcg(a.hamax + r)), s, inv);
                    s_sh[threadIdx.x] = s;
                    s_ent[threadIdx.x] = a.rows[r];
                }
                __syncthreads();
                for (int m = 0; m < mc; ++m) {
                    const int r = r0 + m0 + m;
                    float s, inv;
                    act_scale(__uint_as_float(__ldcg(a.hamax + r)), s, inv);
                    int sum = 0;
                    for (int g = threadIdx.x; g < (I >> 3); g += blockDim.x) {
                        const float *hp = a.h + (size_t)r * I + 8 * g;
                        const float4 v0 = ld_cg_f4(hp), v1 = ld_cg_f4(hp + 4);
                        const int q0 = quant_i8(v0.x, inv), q1 = quant_i8(v0.y, inv), q2 = quant_i8(v0.z, inv),
                                  q3 = quant_i8(v0.w, inv), q4 = quant_i8(v1.x, inv), q5 = quant_i8(v1.y, inv),
                                  q6 = quant_i8(v1.z, inv), q7 = quant_i8(v1.w, inv);
                        sum += q0 + q1 + q2 + q3 + q4 + q5 + q6 + q7;
                        const uint32_t ev = (q0 & 255) | ((q2 & 255) << 8) | ((q4 & 255) << 16) | ((uint32_t)(q6 & 255) << 24);
                        const uint32_t od = (q1 & 255) | ((q3 & 255) << 8) | ((q5 & 255) << 16) | ((uint32_t)(q7 & 255) << 24);
                        *reinterpret_cast<uint2 *>(hq_s + (size_t)m * I + 8 * g) = make_uint2(ev, od);
                        if (a.dbg.hq && b == 0) {
                            const uint32_t n0 = (q0 & 255) | ((q1 & 255) << 8) | ((q2 & 255) << 16) | ((uint32_t)(q3 & 255) << 24);
                            const uint32_t n1 = (q4 & 255) | ((q5 & 255) << 8) | ((q6 & 255) << 16) | ((uint32_t)(q7 & 255) << 24);
                            *reinterpret_cast<uint2 *>(a.dbg.hq + (size_t)s_ent[m] * I + 8 * g) = make_uint2(n0, n1);
                        }
                    }
                    sum = warp_sum_i(sum);
                    if (lane == 0) atomicAdd(&s_hsum[m], sum);
                }
                if (a.dbg.sh && b == 0 && threadIdx.x < mc) a.dbg.sh[s_ent[threadIdx.x]] = s_sh[threadIdx.x];
                __syncthreads();
                staged_u = u;
                staged_m0 = m0;
            }

            for (int j = 0; j < rpw; ++j) {
                const int o = b * a.rpi_dn + warp * rpw + j;
                if (o >= D) break;
                const uint8_t *drow = ex.dq + (size_t)o * rowb;
                int4 dw[CPL];
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    const int ch = lane + 32 * c;
                    if (ch < nch) dw[c] = ld_stream16(drow + (size_t)ch * 16);
                }
                int ad[MCH];
#pragma unroll
                for (int m = 0; m < MCH; ++m) ad[m] = 0;
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    const int ch = lane + 32 * c;
                    if (ch < nch) {
#pragma unroll
                        for (int m = 0; m < MCH; ++m) {
                            if (m < mc) {
                                const int4 *hp = reinterpret_cast<const int4 *>(hq_s + (size_t)m * I + (size_t)ch * 32);
                                const int4 x0 = hp[0], x1 = hp[1];
                                int v = ad[m];
                                v = dot_word((uint32_t)dw[c].x, x0.x, x0.y, v);
                                v = dot_word((uint32_t)dw[c].y, x0.z, x0.w, v);
                                v = dot_word((uint32_t)dw[c].z, x1.x, x1.y, v);
                                v = dot_word((uint32_t)dw[c].w, x1.z, x1.w, v);
                                ad[m] = v;
                            }
                        }
                    }
                }
                int myd = 0;
#pragma unroll
                for (int m = 0; m < MCH; ++m) {
                    if (m < mc) {
                        const int v = warp_sum_i(ad[m]);
                        if (lane == m) myd = v;
                    }
                }
                if (lane < mc) {
                    const int di = myd - 8 * s_hsum[lane];
                    const float y = __fmul_rn(__fmul_rn((float)di, s_sh[lane]), __ldg(ex.ds + o));
                    const int en = s_ent[lane];
                    a.part[(size_t)en * D + o] = y;
                    if (a.dbg.down_acc) a.dbg.down_acc[(size_t)en * D + o] = di;
                }
            }
        }

        if (FUSED) {
            // every token's slots of row block b are complete once all
            // n_union items of that block have arrived
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) s_last = (atomicAdd(a.dn_cnt + b, 1) == a.meta->n_union - 1);
            __syncthreads();
            if (s_last) {
                __threadfence();
                const int o0 = b * a.rpi_dn, K = a.K, S = a.S;
                const int nrow = min(a.rpi_dn, D - o0);
                for (int i = threadIdx.x; i < a.T * nrow; i += blockDim.x) {
                    const int t = i / nrow, o = o0 + (i - t * nrow);
                    const float *pt = a.part + (size_t)t * S * D + o;
                    float acc = 0.f;
                    for (int k = 0; k < K; ++k)  // a slot top-p dropped has no expert output
                        if (__ldcg(a.idx + t * K + k) != kDroppedSel)
                            acc = __fadd_rn(acc, __fmul_rn(__ldcg(a.wts + t * K + k), __ldcg(pt + (size_t)k * D)));
                    if (a.n_shared) acc = __fadd_rn(acc, __ldcg(pt + (size_t)K * D));
                    if (a.resid) acc = __fadd_rn(__ldcg(a.resid + (size_t)t * D + o), acc);
                    a.out[(size_t)t * D + o] = acc;
                }
                if (threadIdx.x == 0) a.dn_cnt[b] = 0;
            }
        }
    }
}

// ---------------------------------------------------------------- reduce

// out[t] = (resid[t] +) sum_k w[t,k] * y[t,k] + y[t,shared], slots in order
// (slots adaptive top-p dropped are skipped).
// Every slot's value is loaded before the first add (K <= kMaxK).
__global__ void __launch_bounds__(256) reduce_kernel(LayerArgs a) {
    const int t = blockIdx.y;
    const int o = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (o >= a.D) return;
    const int K = a.K, S = a.S, D = a.D;
    const float *pt = a.part + (size_t)t * S * D + o;
    float4 y[kMaxK + 1];
    float wk[kMaxK];
    bool kept[kMaxK];  // a slot top-p dropped has no expert output
#pragma unroll
    for (int k = 0; k <= kMaxK; ++k) {
        if (k < S) y[k] = *reinterpret_cast<const float4 *>(pt + (size_t)k * D);
        if (k < K && k < kMaxK) {
            wk[k] = a.wts[t * K + k];
            kept[k] = a.idx[t * K + k] != kDroppedSel;
        }
    }
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.resid) r = *reinterpret_cast<const float4 *>(a.resid + (size_t)t * D + o);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
        if (k < K && kept[k]) {
            acc.x = __fadd_rn(acc.x, __fmul_rn(wk[k], y[k].x));
            acc.y = __fadd_rn(acc.y, __fmul_rn(wk[k], y[k].y));
            acc.z = __fadd_rn(acc.z, __fmul_rn(wk[k], y[k].z));
            acc.w = __fadd_rn(acc.w, __fmul_rn(wk[k], y[k].w));
        }
    }
    if (a.n_shared) {
#pragma unroll
        for (int k = 0; k <= kMaxK; ++k) {
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

// ---------------------------------------------------------- launchers

int mch_index(int mch) { return mch <= 1 ? 0 : mch <= 2 ? 1 : mch <= 4 ? 2 : 3; }

static int cpl_for(int n) {  // chunks per lane for a row of n int4 values
    const int ch = (n + 1023) / 1024;
    return ch <= 1 ? 1 : ch <= 2 ? 2 : ch <= 4 ? 4 : ch <= 6 ? 6 : 8;
}

template <int CPL, int MCH>
static void *gateup_ptr() { return (void *)gateup_kernel<CPL, MCH>; }
template <int CPL, int MCH, bool F>
static void *down_ptr() { return (void *)down_kernel<CPL, MCH, F>; }

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
    const int cpl = cpl_for(a.D);
    MOE_MCH_SWITCH(mch, MOE_CPL_SWITCH(cpl, M_, (gateup_kernel<C, M_><<<grid, 256, 0, s>>>(a))))
    return cudaGetLastError();
}

cudaError_t launch_down(const LayerArgs &a, int mch, int grid, bool fused, cudaStream_t s) {
    const int cpl = cpl_for(a.I);
    const size_t smem = (size_t)(1 << mch_index(mch)) * a.I;
    if (fused) {
        MOE_MCH_SWITCH(mch, MOE_CPL_SWITCH(cpl, M_, (down_kernel<C, M_, true><<<grid, 256, smem, s>>>(a))))
    } else {
        MOE_MCH_SWITCH(mch, MOE_CPL_SWITCH(cpl, M_, (down_kernel<C, M_, false><<<grid, 256, smem, s>>>(a))))
    }
    return cudaGetLastError();
}

cudaError_t launch_reduce(const LayerArgs &a, cudaStream_t s) {
    dim3 grid((a.D / 4 + 255) / 256, a.T);
    reduce_kernel<<<grid, 256, 0, s>>>(a);
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
