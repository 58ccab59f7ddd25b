// k_router.cu -- activation quantiser, sigmoid+bias top-K router and the
// token -> expert permutation (expert union) of the routed-MoE layer.
//
// Sources: reader.mx "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型" §11 (router:
// sigmoid(logit)+bias picks top-K, weight = plain sigmoid * routed_scale;
// batch union so each expert is read once) and §12 (qrow_i8 per-row int8
// quantiser); besthub.dev "Running 744B MoE on 25GB RAM" §11, §12.
#include <cfloat>
#include <climits>

#include "layer_args.cuh"

namespace moe {

// ------------------------------------------------------------------ scans

// Exclusive scan of n <= 2*blockDim.x ints (shared memory in/out, distinct
// arrays).  wtot: shared int[33].  Returns the total to every thread.
__device__ int block_excl_scan(const int *in, int *out, int n, int *wtot) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int i0 = 2 * tid, i1 = 2 * tid + 1;
    const int v0 = i0 < n ? in[i0] : 0, v1 = i1 < n ? in[i1] : 0;
    const int s = v0 + v1;
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    __syncthreads();
    if (lane == 31) wtot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int wv = lane < nw ? wtot[lane] : 0;
        int wi = wv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < nw) wtot[lane] = wi - wv;
        if (lane == 31) wtot[32] = wi;
    }
    __syncthreads();
    const int base = wtot[warp] + incl - s;
    if (i0 < n) out[i0] = base;
    if (i1 < n) out[i1] = base + v0;
    const int total = wtot[32];
    __syncthreads();
    return total;
}

// ---------------------------------------------------------------- quantiser

// One token row, whole block (256 threads): writes the even/odd permuted int8
// row, its scale and the sum of its codes (used by the offset-nibble dot
// product).  D % 8 == 0, D <= 8192, 16-byte aligned rows.  Each thread owns up
// to four 8-element groups, loaded once into registers before any use.
__device__ void quant_token_perm(const float *__restrict__ xrow, int D, int8_t *__restrict__ xq_row,
                                 float *sx_out, int32_t *xsum_out, int8_t *nat_row) {
    __shared__ float red_f[32];
    __shared__ int red_i[32];
    constexpr int G = kMaxDim / (8 * 256);
    const int ng = D >> 3;
    float4 v[2 * G];
#pragma unroll
    for (int k = 0; k < G; ++k) {
        const int g = threadIdx.x + 256 * k;
        if (g < ng) {
            v[2 * k] = __ldg(reinterpret_cast<const float4 *>(xrow + 8 * g));
            v[2 * k + 1] = __ldg(reinterpret_cast<const float4 *>(xrow + 8 * g + 4));
        } else {
            v[2 * k] = v[2 * k + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 2 * G; ++k)
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[k].x), fabsf(v[k].y)), fmaxf(fabsf(v[k].z), fabsf(v[k].w))));
    amax = block_max_nonneg(amax, red_f);
    float s, inv;
    act_scale(amax, s, inv);
    int sum = 0;
#pragma unroll
    for (int k = 0; k < G; ++k) {
        const int g = threadIdx.x + 256 * k;
        if (g >= ng) continue;
        const float4 a = v[2 * k], b = v[2 * k + 1];
        const int q0 = quant_i8(a.x, inv), q1 = quant_i8(a.y, inv), q2 = quant_i8(a.z, inv),
                  q3 = quant_i8(a.w, inv), q4 = quant_i8(b.x, inv), q5 = quant_i8(b.y, inv),
                  q6 = quant_i8(b.z, inv), q7 = quant_i8(b.w, inv);
        sum += q0 + q1 + q2 + q3 + q4 + q5 + q6 + q7;
        const uint32_t ev = (q0 & 255) | ((q2 & 255) << 8) | ((q4 & 255) << 16) | ((uint32_t)(q6 & 255) << 24);
        const uint32_t od = (q1 & 255) | ((q3 & 255) << 8) | ((q5 & 255) << 16) | ((uint32_t)(q7 & 255) << 24);
        *reinterpret_cast<uint2 *>(xq_row + 8 * g) = make_uint2(ev, od);
        if (nat_row) {
            const uint32_t n0 = (q0 & 255) | ((q1 & 255) << 8) | ((q2 & 255) << 16) | ((uint32_t)(q3 & 255) << 24);
            const uint32_t n1 = (q4 & 255) | ((q5 & 255) << 8) | ((q6 & 255) << 16) | ((uint32_t)(q7 & 255) << 24);
            *reinterpret_cast<uint2 *>(nat_row + 8 * g) = make_uint2(n0, n1);
        }
    }
    sum = block_sum_i(sum, red_i);
    if (threadIdx.x == 0) {
        *sx_out = s;
        *xsum_out = sum;
    }
}

__global__ void __launch_bounds__(256) quant_perm_kernel(LayerArgs a) {
    const int t = blockIdx.x;
    quant_token_perm(a.x + (size_t)t * a.D, a.D, a.xq + (size_t)t * a.D, a.sx + t, a.xsum + t,
                     a.dbg.xq ? a.dbg.xq + (size_t)t * a.D : nullptr);
}

// Natural-order quantiser for the public moe_quant_act_int8: any D, any alignment.
__global__ void __launch_bounds__(256) quant_natural_kernel(const float *__restrict__ x, int8_t *__restrict__ xq,
                                                            float *__restrict__ sx, int D) {
    __shared__ float red_f[32];
    const float *row = x + (size_t)blockIdx.x * D;
    float amax = 0.f;
    for (int i = threadIdx.x; i < D; i += blockDim.x) amax = fmaxf(amax, fabsf(row[i]));
    amax = block_max_nonneg(amax, red_f);
    float s, inv;
    act_scale(amax, s, inv);
    for (int i = threadIdx.x; i < D; i += blockDim.x) xq[(size_t)blockIdx.x * D + i] = (int8_t)quant_i8(row[i], inv);
    if (threadIdx.x == 0) sx[blockIdx.x] = s;
}

// ------------------------------------------------------------------ top-K

// sigmoid / selection score of one expert, fp32 IEEE as on the pages.
__device__ __forceinline__ void score(float logit, float b, float &p, float &c) {
    p = __fdiv_rn(1.f, __fadd_rn(1.f, expf(-logit)));
    c = __fadd_rn(p, b);
}

// Order-preserving map of a float onto uint32 (for non-NaN values): larger
// float <=> larger key, equal floats <=> equal keys.
__device__ __forceinline__ uint32_t order_key(float v) {
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Greedy top-K of one token by one warp.  Lane l holds experts l + 32 j.
// Each round takes the largest c among the experts not yet taken; an exact
// tie goes to the lower expert index (the pages' strict '>' ascending scan).
// A round is one warp max over the order keys and one warp min over the
// indices of the lanes that hold that key.  NaN scores never win.
template <int EPL>
__device__ void select_topk(const float (&c)[EPL], const float (&p)[EPL], int E, int K, float scale,
                            int32_t *idx_out, float *w_out, int *s_idx_out, int32_t *err) {
    const int lane = threadIdx.x & 31;
    uint32_t key[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) key[j] = (lane + 32 * j < E && !(c[j] != c[j])) ? order_key(c[j]) : 0u;
    uint32_t taken = 0;
    for (int k = 0; k < K; ++k) {
        // lane-local best: largest key, lowest index on a tie (ascending j)
        uint32_t bk = 0;
        int bj = -1;
#pragma unroll
        for (int j = 0; j < EPL; ++j)
            if (!((taken >> j) & 1u) && key[j] > bk) {
                bk = key[j];
                bj = j;
            }
        const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
        int bi;
        if (wk == 0u) {
            // no finite score left (non-finite input): lowest free index, weight 0
            int cand = INT_MAX;
#pragma unroll
            for (int j = EPL - 1; j >= 0; --j)
                if (!((taken >> j) & 1u) && lane + 32 * j < E) cand = lane + 32 * j;
            bi = __reduce_min_sync(0xffffffffu, cand);
            if (lane == 0 && err) atomicOr(err, kErrNoSelection);
        } else {
            bi = __reduce_min_sync(0xffffffffu, (bk == wk && bj >= 0) ? lane + 32 * bj : INT_MAX);
        }
        const int owner = bi & 31, oj = bi >> 5;
        float pv = 0.f;
#pragma unroll
        for (int j = 0; j < EPL; ++j)
            if (j == oj) pv = p[j];
        pv = __shfl_sync(0xffffffffu, pv, owner);
        if (wk == 0u) pv = 0.f;
        if (lane == owner) taken |= 1u << oj;
        if (lane == 0) {
            idx_out[k] = bi;
            w_out[k] = __fmul_rn(pv, scale);
            if (s_idx_out) s_idx_out[k] = bi;
        }
    }
}

// ------------------------------------------------------- routing tables

// Builds the union tables of a batch from its n = T*K selections (shared
// memory, (token, slot) order), n <= blockDim.x.  Thread i ranks selection i
// by (expert, i): that rank is its row in the expert-grouped order (stable:
// rows of one expert keep (token, slot) order).  The first selection of each
// expert also ranks its expert among the distinct ones, which gives the
// union position (ascending expert id) and the expert's first row.
__device__ void build_routing_small(const LayerArgs &a, const int *s_idx, int T) {
    __shared__ int s_first[kSmallT * kMaxK];
    __shared__ int s_nu;
    const int K = a.K, S = a.S, n = T * K, tid = threadIdx.x;
    int e = -1, less = 0;
    bool first = true;
    if (tid < n) {
        e = s_idx[tid];
        for (int j = 0; j < n; ++j) {
            const int ej = s_idx[j];
            less += ej < e;
            if (ej == e && j < tid) {
                ++less;
                first = false;
            }
        }
        a.rows[less] = (tid / K) * S + (tid % K);
        s_first[tid] = first;
    }
    if (tid == 0) s_nu = 0;
    __syncthreads();
    if (tid < n && first) {
        int upos = 0;
        for (int j = 0; j < n; ++j) upos += s_first[j] && s_idx[j] < e;
        a.meta->uexp[upos] = e;
        a.meta->ubeg[upos] = less;
        atomicAdd(&s_nu, 1);
    }
    __syncthreads();
    if (tid == 0) {
        const int n_routed = s_nu;
        int nu = n_routed;
        a.meta->ubeg[n_routed] = n;
        if (a.n_shared) {
            a.meta->uexp[n_routed] = a.E;
            a.meta->ubeg[n_routed + 1] = n + T;
            nu += 1;
        }
        a.meta->n_union = nu;
        a.meta->n_gu_items = nu * a.nb_gu;
        a.meta->n_dn_items = nu * a.nb_dn;
    }
    if (a.n_shared)
        for (int t = tid; t < T; t += blockDim.x) a.rows[n + t] = t * S + K;
}

// --------------------------------------------------- small-batch router

// T <= kSmallT.  CTAs [0, ceil(E/2)) compute the logits of two experts each
// (four warps per expert, each a quarter of D);
// CTAs [ceil(E/2), ceil(E/2)+T) quantise one token each.  The last CTA to
// finish (arrival counter, no waiting) runs top-K and builds the union.
template <int EPL>
__global__ void __launch_bounds__(256) router_small_kernel(LayerArgs a) {
    __shared__ float red[8][kSmallT];
    __shared__ int s_idx[kSmallT * kMaxK];
    __shared__ int s_last;
    const int T = a.T, D = a.D, E = a.E;
    const int n_lcta = (E + 1) >> 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if ((int)blockIdx.x >= n_lcta) {
        const int t = blockIdx.x - n_lcta;
        quant_token_perm(a.x + (size_t)t * D, D, a.xq + (size_t)t * D, a.sx + t, a.xsum + t,
                         a.dbg.xq ? a.dbg.xq + (size_t)t * D : nullptr);
        if (t == 0)
            for (int i = tid; i < T * a.S; i += blockDim.x) a.hamax[i] = 0u;
    } else {
        // warp = (expert, quarter of D); all of the warp's router weights are
        // loaded before any use so the CTA has its whole 2 x 24 KB in flight
        const int e = blockIdx.x * 2 + (warp >> 2), q = warp & 3;
        const int L4 = D >> 4;  // float4 per quarter row
        float4 w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int c = j * 32 + lane;
            w[j] = (e < E && c < L4) ? __ldg(reinterpret_cast<const float4 *>(a.Wr + (size_t)e * D) + q * L4 + c)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int t = 0; t < T; ++t) {
            const float4 *xr = reinterpret_cast<const float4 *>(a.x + (size_t)t * D) + q * L4;
            float v = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int c = j * 32 + lane;
                if (c < L4) {
                    const float4 xv = __ldg(xr + c);
                    v = fmaf(w[j].x, xv.x, v);
                    v = fmaf(w[j].y, xv.y, v);
                    v = fmaf(w[j].z, xv.z, v);
                    v = fmaf(w[j].w, xv.w, v);
                }
            }
            v = warp_sum_f(v);
            if (lane == 0) red[warp][t] = v;
        }
        __syncthreads();
        if (tid < 2 * kSmallT) {
            const int which = tid / kSmallT, t = tid % kSmallT, e2 = blockIdx.x * 2 + which;
            if (t < T && e2 < E) {
                const int w0 = which * 4;
                const float l = ((red[w0][t] + red[w0 + 1][t]) + red[w0 + 2][t]) + red[w0 + 3][t];
                a.logits[t * E + e2] = l;
                __threadfence();  // the writer makes its logit visible before the arrival
            }
        }
    }

    // arrival: the last CTA finishes the routing (the quantiser CTAs' outputs
    // are read by later kernels only, so they need no fence here)
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&a.meta->counter, 1) == (int)gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int t = warp; t < T; t += 8) {
        float c[EPL], p[EPL];
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int e = lane + 32 * j;
            if (e < E) {
                score(__ldcg(a.logits + t * E + e), __ldg(a.bias + e), p[j], c[j]);
            } else {
                p[j] = 0.f;
                c[j] = -INFINITY;
            }
        }
        select_topk<EPL>(c, p, E, a.K, a.routed_scale, a.idx + t * a.K, a.wts + t * a.K,
                         s_idx + t * a.K, a.err);
    }
    __syncthreads();
    build_routing_small(a, s_idx, T);
    if (tid == 0) a.meta->counter = 0;
}

// ------------------------------------------------------- tiled router

// 16 tokens per CTA, all E experts; logits stay in shared memory.  Used by
// moe_router_topk and by the layer for T > kSmallT.
template <int EPL>
__global__ void __launch_bounds__(256) router_tile_kernel(const float *__restrict__ x, const float *__restrict__ Wr,
                                                          const float *__restrict__ bias, int T, int D, int E, int K,
                                                          float scale, int32_t *__restrict__ idx,
                                                          float *__restrict__ w, int32_t *err) {
    extern __shared__ __align__(16) float sm[];
    const int wstride = ((E * 33) + 3) & ~3;
    float *Wc = sm;                 // [E][33]
    float *Xc = Wc + wstride;       // [32][16]
    float *Lg = Xc + 32 * 16;       // [16][E]
    const int t0 = blockIdx.x * 16, nt = min(16, T - t0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int e0 = tid, e1 = tid + 256;
    float acc0[16], acc1[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) acc0[t] = acc1[t] = 0.f;

    for (int d0 = 0; d0 < D; d0 += 32) {
        const int n4 = min(32, D - d0) >> 2;
        __syncthreads();
        for (int i = tid; i < E * n4; i += 256) {
            const int e = i / n4, j = i - e * n4;
            const float4 v = __ldg(reinterpret_cast<const float4 *>(Wr + (size_t)e * D + d0) + j);
            float *dst = Wc + e * 33 + 4 * j;
            dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
        }
        for (int i = tid; i < 16 * n4; i += 256) {
            const int t = i / n4, j = i - t * n4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < nt) v = __ldg(reinterpret_cast<const float4 *>(x + (size_t)(t0 + t) * D + d0) + j);
            Xc[(4 * j + 0) * 16 + t] = v.x;
            Xc[(4 * j + 1) * 16 + t] = v.y;
            Xc[(4 * j + 2) * 16 + t] = v.z;
            Xc[(4 * j + 3) * 16 + t] = v.w;
        }
        __syncthreads();
        const int dl = n4 * 4;
        for (int d = 0; d < dl; ++d) {
            const float4 *xr = reinterpret_cast<const float4 *>(Xc + d * 16);
            const float4 xa = xr[0], xb = xr[1], xc = xr[2], xd = xr[3];
            const float xv[16] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w,
                                  xc.x, xc.y, xc.z, xc.w, xd.x, xd.y, xd.z, xd.w};
            if (e0 < E) {
                const float wv = Wc[e0 * 33 + d];
#pragma unroll
                for (int t = 0; t < 16; ++t) acc0[t] = fmaf(wv, xv[t], acc0[t]);
            }
            if (EPL > 8 && e1 < E) {
                const float wv = Wc[e1 * 33 + d];
#pragma unroll
                for (int t = 0; t < 16; ++t) acc1[t] = fmaf(wv, xv[t], acc1[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        if (t < nt) {
            if (e0 < E) Lg[t * E + e0] = acc0[t];
            if (EPL > 8 && e1 < E) Lg[t * E + e1] = acc1[t];
        }
    }
    __syncthreads();
    for (int t = warp; t < nt; t += 8) {
        float c[EPL], p[EPL];
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int e = lane + 32 * j;
            if (e < E) {
                score(Lg[t * E + e], __ldg(bias + e), p[j], c[j]);
            } else {
                p[j] = 0.f;
                c[j] = -INFINITY;
            }
        }
        select_topk<EPL>(c, p, E, K, scale, idx + (size_t)(t0 + t) * K, w + (size_t)(t0 + t) * K, nullptr, err);
    }
}

// ------------------------------------------------- large-batch permute

// One CTA of 1024 threads.  Stable counting sort of the T*K selections by
// expert with per-warp histograms (deterministic, no atomics on global
// memory), then the union tables.  Also clears the h amax words.
__global__ void __launch_bounds__(1024) permute_large_kernel(LayerArgs a) {
    extern __shared__ int hist[];  // [32][E]
    __shared__ int tot[kMaxE], base[kMaxE], flg[kMaxE], upos[kMaxE], wtot[33];
    const int E = a.E, K = a.K, S = a.S, T = a.T, n = T * K;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < 32 * E; i += blockDim.x) hist[i] = 0;
    for (int i = tid; i < T * S; i += blockDim.x) a.hamax[i] = 0u;
    __syncthreads();
    const int L = (((n + 31) / 32) + 31) & ~31;  // per-warp slice, a multiple of 32
    const int beg = warp * L, end = min(n, beg + L);
    const unsigned lt = (1u << lane) - 1u;
    for (int g = beg; g < end; g += 32) {
        const int i = g + lane;
        const bool v = i < end;
        int e = v ? a.idx[i] : -1;
        if (v && (e < 0 || e >= E)) { e = 0; atomicOr(a.err, kErrRouteCount); }
        const unsigned m = __match_any_sync(0xffffffffu, e);
        if (v && __popc(m & lt) == 0) hist[warp * E + e] += __popc(m);
        __syncwarp();
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < 32; ++w) {
            const int c = hist[w * E + e];
            hist[w * E + e] = run;
            run += c;
        }
        tot[e] = run;
        flg[e] = run > 0;
    }
    __syncthreads();
    block_excl_scan(tot, base, E, wtot);
    const int n_routed = block_excl_scan(flg, upos, E, wtot);
    for (int e = tid; e < E; e += blockDim.x)
        if (tot[e] > 0) {
            a.meta->uexp[upos[e]] = e;
            a.meta->ubeg[upos[e]] = base[e];
        }
    if (tid == 0) {
        int nu = n_routed;
        a.meta->ubeg[n_routed] = n;
        if (a.n_shared) {
            a.meta->uexp[n_routed] = E;
            a.meta->ubeg[n_routed + 1] = n + T;
            nu += 1;
        }
        a.meta->n_union = nu;
        a.meta->n_gu_items = nu * a.nb_gu;
        a.meta->n_dn_items = nu * a.nb_dn;
    }
    for (int i = tid; i < 32 * E; i += blockDim.x) hist[i] += base[i % E];
    __syncthreads();
    for (int g = beg; g < end; g += 32) {
        const int i = g + lane;
        const bool v = i < end;
        int e = v ? a.idx[i] : -1;
        if (v && (e < 0 || e >= E)) e = 0;
        const unsigned m = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(m & lt);
        if (v) a.rows[hist[warp * E + e] + rank] = (i / K) * S + (i % K);
        __syncwarp();
        if (v && rank == 0) hist[warp * E + e] += __popc(m);
        __syncwarp();
    }
    if (a.n_shared)
        for (int t = tid; t < T; t += blockDim.x) a.rows[n + t] = t * S + K;
}

// ---------------------------------------------------------- launchers

static int epl_for(int E) { return E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : E <= 256 ? 8 : 16; }

cudaError_t launch_router_small(const LayerArgs &a, cudaStream_t s) {
    const int grid = (a.E + 1) / 2 + a.T;
    switch (epl_for(a.E)) {
        case 1: router_small_kernel<1><<<grid, 256, 0, s>>>(a); break;
        case 2: router_small_kernel<2><<<grid, 256, 0, s>>>(a); break;
        case 4: router_small_kernel<4><<<grid, 256, 0, s>>>(a); break;
        case 8: router_small_kernel<8><<<grid, 256, 0, s>>>(a); break;
        default: router_small_kernel<16><<<grid, 256, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_quant_perm(const LayerArgs &a, cudaStream_t s) {
    quant_perm_kernel<<<a.T, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_quant_natural(const float *x, int8_t *xq, float *sx, int T, int D, cudaStream_t s) {
    quant_natural_kernel<<<T, 256, 0, s>>>(x, xq, sx, D);
    return cudaGetLastError();
}

template <int EPL>
static cudaError_t launch_tile_t(const float *x, const float *Wr, const float *bias, int T, int D, int E, int K,
                                 float scale, int32_t *idx, float *w, int32_t *err, cudaStream_t s) {
    const size_t smem = sizeof(float) * ((((size_t)E * 33) + 3) / 4 * 4 + 32 * 16 + 16 * (size_t)E);
    cudaError_t ce = cudaFuncSetAttribute(router_tile_kernel<EPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)smem);
    if (ce != cudaSuccess) return ce;
    router_tile_kernel<EPL><<<(T + 15) / 16, 256, smem, s>>>(x, Wr, bias, T, D, E, K, scale, idx, w, err);
    return cudaGetLastError();
}

cudaError_t launch_router_tile(const float *x, const float *Wr, const float *bias, int T, int D, int E, int K,
                               float scale, int32_t *idx, float *w, int32_t *err, cudaStream_t s) {
    switch (epl_for(E)) {
        case 1: return launch_tile_t<1>(x, Wr, bias, T, D, E, K, scale, idx, w, err, s);
        case 2: return launch_tile_t<2>(x, Wr, bias, T, D, E, K, scale, idx, w, err, s);
        case 4: return launch_tile_t<4>(x, Wr, bias, T, D, E, K, scale, idx, w, err, s);
        case 8: return launch_tile_t<8>(x, Wr, bias, T, D, E, K, scale, idx, w, err, s);
        default: return launch_tile_t<16>(x, Wr, bias, T, D, E, K, scale, idx, w, err, s);
    }
}

cudaError_t launch_permute(const LayerArgs &a, cudaStream_t s) {
    const size_t smem = sizeof(int) * 32 * (size_t)a.E;
    cudaError_t ce = cudaFuncSetAttribute(permute_large_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)smem);
    if (ce != cudaSuccess) return ce;
    permute_large_kernel<<<1, 1024, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
