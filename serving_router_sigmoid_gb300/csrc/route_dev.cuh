// route_dev.cuh -- device building blocks of the router and the activation
// quantiser: one-token int8 quantiser (even/odd layout), sigmoid+bias
// scores and the warp top-K.  Internal.
//
// Sources: reader.mx "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型" §11 (router:
// sigmoid(logit)+bias picks top-K, weight = plain sigmoid * routed_scale) and
// §12 (qrow_i8 per-row int8 quantiser); besthub.dev "Running 744B MoE on 25GB
// RAM" §11, §12.
#pragma once

#include <cfloat>
#include <climits>

#include "layer_args.cuh"

namespace moe {

// ---------------------------------------------------------------- quantiser

// One token row, whole block (256 threads): writes the even/odd permuted int8
// row, its scale and the sum of its codes (used by the offset-nibble dot
// product).  D % 8 == 0, D <= 8192, 16-byte aligned rows.  Each thread owns up
// to four 8-element groups, loaded once into registers before any use.
// Outputs (each may be null): xq_row / sx_out / xsum_out global; nat_row the
// natural-order codes.
__device__ __forceinline__ void quant_token_perm(const float *__restrict__ xrow, int D, int8_t *__restrict__ xq_row,
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
        if (xq_row) *reinterpret_cast<uint2 *>(xq_row + 8 * g) = make_uint2(ev, od);
        if (nat_row) {
            const uint32_t n0 = (q0 & 255) | ((q1 & 255) << 8) | ((q2 & 255) << 16) | ((uint32_t)(q3 & 255) << 24);
            const uint32_t n1 = (q4 & 255) | ((q5 & 255) << 8) | ((q6 & 255) << 16) | ((uint32_t)(q7 & 255) << 24);
            *reinterpret_cast<uint2 *>(nat_row + 8 * g) = make_uint2(n0, n1);
        }
    }
    sum = block_sum_i(sum, red_i);
    if (threadIdx.x == 0) {
        if (sx_out) *sx_out = s;
        if (xsum_out) *xsum_out = sum;
    }
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

// Adaptive expert top-p (aimsg.uk "低配电脑也能跑GLM 5.2" --topp; reader.mx
// §11 runs the union over the first keff selections of each token): keff is
// the length of the shortest prefix of the K selections, in selection order,
// whose routing weights reach top_p times the sum of all K (fp32 sums left to
// right, the bound one fp32 product), at least 1; top_p outside (0, 1) keeps
// all K.  w(j) returns the weight of selection j.  Every caller evaluates the
// same sums in the same order, so the decision is the same everywhere.
template <typename W>
__device__ __forceinline__ int topp_keff(W w, int K, float top_p) {
    if (!(top_p > 0.f && top_p < 1.f)) return K;
    float total = 0.f;
    for (int j = 0; j < K; ++j) total = __fadd_rn(total, w(j));
    const float bound = __fmul_rn(top_p, total);
    float run = 0.f;
    for (int j = 0; j < K; ++j) {
        run = __fadd_rn(run, w(j));
        if (run >= bound) return j + 1;
    }
    return K;
}

// Greedy top-K of one token by one warp.  Lane l holds experts l + 32 j.
// Each round takes the largest c among the experts not yet taken; an exact
// tie goes to the lower expert index (the pages' strict '>' ascending scan).
// A round is one warp max over the order keys and one warp min over the
// indices of the lanes that hold that key.  NaN scores never win.  With
// top_p in (0, 1) the selections past keff (topp_keff) are dropped: id
// kDroppedSel, weight 0.
template <int EPL>
__device__ __forceinline__ void select_topk(const float (&c)[EPL], const float (&p)[EPL], int E, int K, float scale,
                            int32_t *idx_out, float *w_out, int *s_idx_out, int32_t *err, float top_p = 0.f) {
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
    if (lane == 0 && top_p > 0.f && top_p < 1.f) {
        const int keff = topp_keff([&](int j) { return w_out[j]; }, K, top_p);
        for (int k = keff; k < K; ++k) {
            idx_out[k] = kDroppedSel;
            w_out[k] = 0.f;
            if (s_idx_out) s_idx_out[k] = kDroppedSel;
        }
    }
}

// ------------------------------------------------- parallel top-K (whole CTA)

// Composite selection key of expert e: a larger score c first, the lower
// expert index on an exact tie (the pages' strict '>' ascending scan), NaN
// scores below every number (key 0 in the high word), experts e >= E below
// everything.  Sorting these keys in descending order gives exactly the
// order in which select_topk picks.  Bits 0..15 are free for a payload.
__device__ __forceinline__ unsigned long long sel_key(float c, int e, int E) {
    if (e >= E) return 0ull;
    const uint32_t k = (c != c) ? 0u : order_key(c);
    return ((unsigned long long)k << 32) | ((uint32_t)(0xFFFFu - (uint32_t)e) << 16);
}

// Descending bitonic sort of 32*NPL keys held by one warp (element i =
// lane + 32*s in v[s]).
template <int NPL>
__device__ __forceinline__ void warp_sort_desc(unsigned long long (&v)[NPL]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32 * NPL; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            unsigned long long o[NPL];
#pragma unroll
            for (int s = 0; s < NPL; ++s) o[s] = j < 32 ? __shfl_xor_sync(0xffffffffu, v[s], j) : v[s ^ (j >> 5)];
#pragma unroll
            for (int s = 0; s < NPL; ++s) {
                const int i = lane + 32 * s;
                const bool keep_max = ((i & j) == 0) == ((i & k) == 0);
                const unsigned long long mx = v[s] > o[s] ? v[s] : o[s], mn = v[s] > o[s] ? o[s] : v[s];
                v[s] = keep_max ? mx : mn;
            }
        }
    }
}

// Top-K of T <= kSmallT tokens by a whole CTA (8 warps, 256 threads), in
// groups of four tokens: every warp sorts its slice of the experts (32 per
// warp for E <= 256, else 64) for each token of the group and keeps its best
// K (K <= 16) with their sigmoids; then warp g merges the 8 lists of token g.
// Every logit of the group is loaded before any sort.  Selection order and
// weights are those of select_topk: weight = sigmoid(logit) * scale, 0 (with
// kErrNoSelection) for a pick whose score is NaN; with top_p in (0, 1) the
// picks past keff are dropped (id kDroppedSel, weight 0).  logits: [T][E] (read
// through L2; with POLL the slots are published as data and the CTA reloads
// them, bounded, until none holds kLogitEmpty).  scratch: shared [4][8][kMaxK]
// keys, pscr: shared [4][8][kMaxK] sigmoids.  Outputs [T][K]: idx/w (shared or
// global), or with packed != null one word (expert << 32 | weight bits) per
// selection, stored as a single relaxed 64-bit write.  err may be null.
template <bool POLL>
__device__ __forceinline__ void topk_small_cta(const float *logits, const float *__restrict__ bias, int T, int E,
                                               int K, float scale, int32_t *idx, float *w,
                                               unsigned long long *packed, int32_t *err,
                                               unsigned long long (*scratch)[8][kMaxK], float (*pscr)[8][kMaxK],
                                               float top_p = 0.f) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool one = E <= 256;  // one expert per lane (else two)
    float bsum[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const int e = one ? warp * 32 + lane : warp * 64 + lane + 32 * s;
        bsum[s] = (e < E && (s == 0 || !one)) ? __ldg(bias + e) : 0.f;
    }
    for (int t0 = 0; t0 < T; t0 += 4) {
        const int ng = T - t0 < 4 ? T - t0 : 4;
        float lg[4][2];
        const unsigned long long t_begin = POLL ? global_ns() : 0ull;
        for (;;) {
            bool miss = false;
#pragma unroll
            for (int g = 0; g < 4; ++g)
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    const int e = one ? warp * 32 + lane : warp * 64 + lane + 32 * s;
                    const float *src = logits + (size_t)(t0 + g) * E + e;
                    const bool valid = g < ng && e < E && (s == 0 || !one);
                    uint32_t bits = 0u;
                    if (valid) bits = POLL ? ld_relaxed_u32(src) : __float_as_uint(__ldcg(src));
                    miss |= POLL && bits == kLogitEmpty;
                    lg[g][s] = __uint_as_float(bits);
                }
            if (!POLL || !__syncthreads_or(miss)) break;
            const bool late = threadIdx.x == 0 && global_ns() - t_begin > kWaitNs;
            if (__syncthreads_or(late)) {
                if (threadIdx.x == 0 && err) atomicOr(err, kErrSyncTimeout);
                break;
            }
            __nanosleep(64);
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            if (g >= ng) break;
            float p[2], c[2];
            unsigned long long v[2];
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const int e = one ? warp * 32 + lane : warp * 64 + lane + 32 * s;
                p[s] = c[s] = 0.f;
                if (e < E) score(lg[g][s], bsum[s], p[s], c[s]);
                v[s] = sel_key(c[s], e, E);
            }
            // position of each key in the warp's slice travels in bits 0..7
            // (below the expert bits, so it never decides the order)
            int src;
            if (one) {
                unsigned long long u[1] = {v[0] | (uint32_t)lane};
                warp_sort_desc<1>(u);
                v[0] = u[0];
            } else {
                v[0] |= (uint32_t)lane;
                v[1] |= (uint32_t)(lane + 32);
                warp_sort_desc<2>(v);
            }
            src = (int)(v[0] & 0xFFu);
            const float p0 = __shfl_sync(0xffffffffu, p[0], src & 31);
            const float p1 = __shfl_sync(0xffffffffu, p[1], src & 31);
            if (lane < K) {  // K <= 16: the best K are in lanes 0..K-1
                scratch[g][warp][lane] = v[0] & ~0xFFull;
                pscr[g][warp][lane] = src < 32 ? p0 : p1;
            }
        }
        __syncthreads();
        if (warp < ng) {
            const int t = t0 + warp;
            unsigned long long v[4];
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const int i = lane + 32 * s, src = i / K, k = i - src * K;
                v[s] = (i < 8 * K) ? (scratch[warp][src][k] | (uint32_t)i) : 0ull;
            }
            if (K <= 8) {
                unsigned long long u[2] = {v[0], v[1]};
                warp_sort_desc<2>(u);
                v[0] = u[0];
            } else {
                warp_sort_desc<4>(v);
            }
            // the best K are in lanes 0..K-1, in selection order
            const unsigned long long key = v[0];
            const int i = (int)(key & 0xFFu);
            int e = (int)(0xFFFFu - (uint32_t)((key >> 16) & 0xFFFFu));
            const bool nan_pick = (key >> 32) == 0ull;
            float wv = (lane < K && !nan_pick) ? __fmul_rn(pscr[warp][i / K][i % K], scale) : 0.f;
            // adaptive top-p: every lane evaluates keff over the K weights
            const int keff = topp_keff([&](int j) { return __shfl_sync(0xffffffffu, wv, j); }, K, top_p);
            if (lane >= keff) {
                e = kDroppedSel;
                wv = 0.f;
            }
            if (lane < K) {
                if (packed) {
                    st_relaxed_u64(packed + t * K + lane, ((unsigned long long)(uint32_t)e << 32) | __float_as_uint(wv));
                } else {
                    idx[t * K + lane] = e;
                    w[t * K + lane] = wv;
                }
                if (nan_pick && err) atomicOr(err, kErrNoSelection);
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------ router logits

// Logits of one expert for tokens 0..T-1 (T <= kSmallT), by a whole CTA of 256
// threads: warp w sums the w-th eighth of the row (each lane one fmaf chain
// over its float4 chunks, then a warp tree) and thread t < T adds the eight
// partials in warp order.  Every router of decode-sized batches uses this
// arithmetic, so their logits agree bit for bit.  D % 32 == 0, D <= kMaxDim.
// logits_request issues the loads of the expert's router row (and, with X0,
// of token 0's activations) so that they can be queued ahead of other
// traffic; logits_finish multiplies.  NW float4 slots per lane cover
// D <= 1024 * NW.  red: shared [8][kSmallT].  Thread t < T receives the
// logit of token t.
template <int NW, bool X0>
struct WrRegs {
    float4 w[NW];
    float4 x0[X0 ? NW : 1];
};

template <int NW, bool X0>
__device__ __forceinline__ void logits_request(WrRegs<NW, X0> &r, const float *__restrict__ wrow,
                                               const float *__restrict__ x, int D) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L8 = D >> 5;  // float4 per eighth of a row
    const float4 *wr = reinterpret_cast<const float4 *>(wrow) + warp * L8;
    const float4 *xr = reinterpret_cast<const float4 *>(x) + warp * L8;
#pragma unroll
    for (int j = 0; j < NW; ++j) {
        const int c = j * 32 + lane;
        r.w[j] = c < L8 ? __ldg(wr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (X0) r.x0[j] = c < L8 ? __ldg(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

template <int NW, bool X0>
__device__ __forceinline__ float logits_finish(const WrRegs<NW, X0> &r, const float *__restrict__ x, int T, int D,
                                               float (*red)[kSmallT]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L8 = D >> 5;
    for (int t = 0; t < T; ++t) {
        const float4 *xr = reinterpret_cast<const float4 *>(x + (size_t)t * D) + warp * L8;
        float v = 0.f;
#pragma unroll
        for (int j = 0; j < NW; ++j) {
            const int c = j * 32 + lane;
            if (c < L8) {
                const float4 xv = (X0 && t == 0) ? r.x0[X0 ? j : 0] : __ldg(xr + c);
                v = fmaf(r.w[j].x, xv.x, v);
                v = fmaf(r.w[j].y, xv.y, v);
                v = fmaf(r.w[j].z, xv.z, v);
                v = fmaf(r.w[j].w, xv.w, v);
            }
        }
        v = warp_sum_f(v);
        if (lane == 0) red[warp][t] = v;
    }
    __syncthreads();
    float l = 0.f;
    if ((int)threadIdx.x < T) {
        l = red[0][threadIdx.x];
#pragma unroll
        for (int w8 = 1; w8 < 8; ++w8) l = __fadd_rn(l, red[w8][threadIdx.x]);
    }
    __syncthreads();
    return l;
}

// Loads only the router row into r.w (logits_request without the
// activations: weights may be requested before the previous kernel in the
// stream, which writes the activations, has finished).
template <int NW, bool X0>
__device__ __forceinline__ void logits_request_w(WrRegs<NW, X0> &r, const float *__restrict__ wrow, int D) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L8 = D >> 5;
    const float4 *wr = reinterpret_cast<const float4 *>(wrow) + warp * L8;
#pragma unroll
    for (int j = 0; j < NW; ++j) {
        const int c = j * 32 + lane;
        r.w[j] = c < L8 ? __ldg(wr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Loads only token 0's activations into r.x0, in logits_request's layout (for
// a CTA that computes no logit but quantises token 0 from registers).
template <int NW>
__device__ __forceinline__ void x0_request(WrRegs<NW, true> &r, const float *__restrict__ x, int D) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L8 = D >> 5;
    const float4 *xr = reinterpret_cast<const float4 *>(x) + warp * L8;
#pragma unroll
    for (int j = 0; j < NW; ++j) {
        const int c = j * 32 + lane;
        r.x0[j] = c < L8 ? __ldg(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Token 0 quantised from the registers of logits_request / x0_request, with
// the arithmetic of quant_token_perm (absmax / 127 scale, round to nearest
// even; the max and the integer code sum do not depend on the order), into
// the two-plane tile with its scale and code sum; xq_row / sx_out / xsum_out
// / nat_row (each may be null) receive the global rows.  Thread (w, lane)
// holds float4 number w * D/32 + 32 j + lane of the row: elements 4f..4f+3,
// the low or high half of 8-group f/2, i.e. two bytes of its even word and
// two of its odd word in the permuted layout.  All threads call it.
template <int NW>
__device__ __forceinline__ void quant_x0_tile(const WrRegs<NW, true> &r, int D, int8_t *tile, float *tile_sx,
                                              int *tile_xsum, int8_t *xq_row, float *sx_out, int32_t *xsum_out,
                                              int8_t *nat_row) {
    __shared__ float red_f[32];
    __shared__ int red_i[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L8 = D >> 5;
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < NW; ++j) {
        const float4 v = r.x0[j];  // zero beyond the row
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    amax = block_max_nonneg(amax, red_f);
    float s, inv;
    act_scale(amax, s, inv);
    int sum = 0;
#pragma unroll
    for (int j = 0; j < NW; ++j) {
        const int c = j * 32 + lane;
        if (c >= L8) continue;
        const int f = warp * L8 + c;
        const float4 v = r.x0[j];
        const int q0 = quant_i8(v.x, inv), q1 = quant_i8(v.y, inv), q2 = quant_i8(v.z, inv),
                  q3 = quant_i8(v.w, inv);
        sum += q0 + q1 + q2 + q3;
        const int byte = 8 * (f >> 1) + 2 * (f & 1);  // even half-word; the odd one 4 bytes on
        const uint16_t ev = (uint16_t)((q0 & 255) | ((q2 & 255) << 8));
        const uint16_t od = (uint16_t)((q1 & 255) | ((q3 & 255) << 8));
        *reinterpret_cast<uint16_t *>(plane_byte(tile, D, 0, byte)) = ev;
        *reinterpret_cast<uint16_t *>(plane_byte(tile, D, 0, byte + 4)) = od;
        if (xq_row) {
            *reinterpret_cast<uint16_t *>(xq_row + byte) = ev;
            *reinterpret_cast<uint16_t *>(xq_row + byte + 4) = od;
        }
        if (nat_row)
            *reinterpret_cast<uint32_t *>(nat_row + 4 * f) =
                (q0 & 255) | ((q1 & 255) << 8) | ((q2 & 255) << 16) | ((uint32_t)(q3 & 255) << 24);
    }
    sum = block_sum_i(sum, red_i);
    if (threadIdx.x == 0) {
        *tile_sx = s;
        *tile_xsum = sum;
        if (sx_out) *sx_out = s;
        if (xsum_out) *xsum_out = sum;
    }
}

__device__ __forceinline__ float expert_logits_cta(const float *__restrict__ wrow, const float *__restrict__ x,
                                                   int T, int D, float (*red)[kSmallT]) {
    WrRegs<kMaxDim / 1024, false> r;
    logits_request(r, wrow, x, D);
    return logits_finish(r, x, T, D, red);
}

}  // namespace moe
