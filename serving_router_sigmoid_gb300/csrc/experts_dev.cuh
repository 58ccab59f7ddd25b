// experts_dev.cuh -- the row-per-warp expert kernels (fused gate/up +
// SiLU*up, down with the expert-output scatter) for int4 and int8 weights.
// Internal: instantiated by k_experts.cu (int4) and k_experts8.cu (int8).
//
// Sources: reader.mx "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型" §11 (SwiGLU
// expert: gate/up, siluf(g)*u, down, weighted add into the token's output),
// §12 (int8 activations x int4 weights, or int8 weights (fmt 1,
// matmul_q_idot), with an exact integer dot, then the activation and row
// scales), §05 (per-row int8 weights); besthub.dev "Running 744B MoE on 25GB
// RAM" §11, §12.
//
// Every warp owns whole output rows, reads them with 16-byte streaming loads
// (no L1 allocation) and multiplies them against the int8 activations of all
// rows routed to that expert.  int4 (WB = 4): offset nibbles n = v + 8 go
// straight into dp4a; sum((n-8) x) = sum(n x) - 8 sum(x) restores the signed
// dot exactly.  int8 (WB = 8): the weight bytes are signed already; a byte
// permute regroups each 8-group into its even and odd elements, the order in
// which the activations are stored, and dp4a takes them as they are.
#pragma once

#include "layer_args.cuh"

namespace moe {

// One 16-byte chunk of an int8 weight row (elements 16c .. 16c+15, natural
// order) against the same 16 activations stored as two even/odd 8-groups:
// acc + sum_i w_i x_i, exact.
__device__ __forceinline__ int dot_chunk8(const int4 &w, const int4 &x, int acc) {
    const uint32_t wx = (uint32_t)w.x, wy = (uint32_t)w.y, wz = (uint32_t)w.z, ww = (uint32_t)w.w;
    acc = __dp4a((int)__byte_perm(wx, wy, 0x6420), x.x, acc);  // elements 0, 2, 4, 6
    acc = __dp4a((int)__byte_perm(wx, wy, 0x7531), x.y, acc);  // elements 1, 3, 5, 7
    acc = __dp4a((int)__byte_perm(wz, ww, 0x6420), x.z, acc);  // elements 8, 10, 12, 14
    acc = __dp4a((int)__byte_perm(wz, ww, 0x7531), x.w, acc);  // elements 9, 11, 13, 15
    return acc;
}

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
template <int CPL, int MCH, int WB>
__global__ void __launch_bounds__(256) gateup_kernel(LayerArgs a) {
    __shared__ unsigned s_amax[MCH];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = a.D, I = a.I, S = a.S;
    const int nch = WB == 4 ? D >> 5 : D >> 4;  // 16-byte weight chunks per row
    const size_t rowb = (size_t)(WB == 4 ? D >> 1 : D);
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
                                if (WB == 4) {
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
                                } else {
                                    const int4 x0 = __ldg(reinterpret_cast<const int4 *>(a.xq + (size_t)tk[m] * D) + ch);
                                    ag[m] = dot_chunk8(gw[c], x0, ag[m]);
                                    au[m] = dot_chunk8(uw[c], x0, au[m]);
                                }
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
                    const int off = WB == 4 ? 8 * myxs : 0;  // offset nibbles: sum((n-8)x) = sum(nx) - 8 sum(x)
                    const int gi = myg - off, ui = myu - off;
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
template <int CPL, int MCH, bool FUSED, int WB>
__global__ void __launch_bounds__(256) down_kernel(LayerArgs a) {
    extern __shared__ __align__(16) int8_t hq_s[];  // [MCH][I]
    __shared__ int s_hsum[MCH];
    __shared__ float s_sh[MCH];
    __shared__ int s_ent[MCH];
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = a.D, I = a.I;
    const int nch = WB == 4 ? I >> 5 : I >> 4;  // 16-byte weight chunks per row
    const size_t rowb = (size_t)(WB == 4 ? I >> 1 : I);
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
                                if (WB == 4) {
                                    const int4 *hp = reinterpret_cast<const int4 *>(hq_s + (size_t)m * I + (size_t)ch * 32);
                                    const int4 x0 = hp[0], x1 = hp[1];
                                    int v = ad[m];
                                    v = dot_word((uint32_t)dw[c].x, x0.x, x0.y, v);
                                    v = dot_word((uint32_t)dw[c].y, x0.z, x0.w, v);
                                    v = dot_word((uint32_t)dw[c].z, x1.x, x1.y, v);
                                    v = dot_word((uint32_t)dw[c].w, x1.z, x1.w, v);
                                    ad[m] = v;
                                } else {
                                    const int4 x0 = reinterpret_cast<const int4 *>(hq_s + (size_t)m * I)[ch];
                                    ad[m] = dot_chunk8(dw[c], x0, ad[m]);
                                }
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
                    const int di = WB == 4 ? myd - 8 * s_hsum[lane] : myd;
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

}  // namespace moe
