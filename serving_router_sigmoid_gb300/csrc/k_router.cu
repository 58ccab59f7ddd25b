// k_router.cu -- activation quantiser, sigmoid+bias top-K router and the
// token -> expert permutation (expert union) of the routed-MoE layer.
//
// Sources: reader.mx "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型" §11 (router:
// sigmoid(logit)+bias picks top-K, weight = plain sigmoid * routed_scale;
// batch union so each expert is read once) and §12 (qrow_i8 per-row int8
// quantiser); besthub.dev "Running 744B MoE on 25GB RAM" §11, §12.
#include "route_dev.cuh"

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

// ------------------------------------------------------- routing tables

// Builds the union tables of a batch from its n = T*K selections (shared
// memory, (token, slot) order), n <= blockDim.x.  Thread i ranks selection i
// by (expert, i): that rank is its row in the expert-grouped order (stable:
// rows of one expert keep (token, slot) order).  The first selection of each
// expert also ranks its expert among the distinct ones, which gives the
// union position (ascending expert id) and the expert's first row.
// Selections that adaptive top-p dropped (kDroppedSel) take no row; the
// shared expert's rows follow the kept ones.
__device__ void build_routing_small(const LayerArgs &a, const int *s_idx, int T) {
    __shared__ int s_first[kSmallT * kMaxK];
    __shared__ int s_nu;
    const int K = a.K, S = a.S, tid = threadIdx.x;
    int e = -1, less = 0;
    bool first = false;
    if (tid < T * K) {
        e = s_idx[tid];
        if (e != kDroppedSel) {
            first = true;
            for (int j = 0; j < T * K; ++j) {
                const int ej = s_idx[j];
                if (ej == kDroppedSel) continue;
                less += ej < e;
                if (ej == e && j < tid) {
                    ++less;
                    first = false;
                }
            }
            a.rows[less] = (tid / K) * S + (tid % K);
        }
        s_first[tid] = first;
    }
    if (tid == 0) s_nu = 0;
    const int n = __syncthreads_count(tid < T * K && e != kDroppedSel);  // kept selections
    if (tid < T * K && first) {
        int upos = 0;
        for (int j = 0; j < T * K; ++j) upos += s_first[j] && s_idx[j] < e;
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

// T <= kSmallT.  CTA e < E computes the logits of expert e (expert_logits_cta);
// CTAs [E, E+T) quantise one token each.  The last CTA to
// finish (arrival counter, no waiting) runs top-K (topk_small_cta) and builds
// the union.
__global__ void __launch_bounds__(256) router_small_kernel(LayerArgs a) {
    __shared__ float red[8][kSmallT];
    __shared__ unsigned long long tk[4][8][kMaxK];
    __shared__ float tkp[4][8][kMaxK];
    __shared__ int s_idx[kSmallT * kMaxK];
    __shared__ int s_last;
    const int T = a.T, D = a.D, E = a.E;
    const int tid = threadIdx.x;

    if ((int)blockIdx.x >= E) {
        const int t = blockIdx.x - E;
        quant_token_perm(a.x + (size_t)t * D, D, a.xq + (size_t)t * D, a.sx + t, a.xsum + t,
                         a.dbg.xq ? a.dbg.xq + (size_t)t * D : nullptr);
        if (t == 0)
            for (int i = tid; i < T * a.S; i += blockDim.x) a.hamax[i] = 0u;
    } else {
        const int e = blockIdx.x;
        const float l = expert_logits_cta(a.Wr + (size_t)e * D, a.x, T, D, red);
        if (tid < T) {
            a.logits[tid * E + e] = l;
            __threadfence();  // the writer makes its logit visible before the arrival
        }
    }

    // arrival: the last CTA finishes the routing (the quantiser CTAs' outputs
    // are read by later kernels only, so they need no fence here)
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&a.meta->counter, 1) == (int)gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    topk_small_cta<false>(a.logits, a.bias, T, E, a.K, a.routed_scale, s_idx, a.wts, nullptr, a.err, tk, tkp,
                          a.top_p);
    for (int i = tid; i < T * a.K; i += blockDim.x) a.idx[i] = s_idx[i];
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

// ------------------------------------------------ large-batch router (2 kernels)

// Logits of a large batch as a register-tiled fp32 GEMM: CTA tile 128 tokens
// x 128 experts, K in chunks of 32 through a 4-stage cp.async ring (rows kept
// d-contiguous, so no transpose on the way in), 256 threads each
// accumulating 8 tokens x 8 experts (rows ty + 16 i, columns tx + 16 j, which
// keeps the shared-memory reads conflict-free) with one fmaf chain per output
// in ascending d: per 4 d, 16 16-byte shared loads feed 256 fmaf.  One CTA
// per SM.  K is split into gridDim.z contiguous ranges of whole chunks (at T
// = 2048 the 32 tiles x 9 ranges make two waves of the 152 SMs); range z
// writes its partial logits to logits + z T E and the select kernel adds the
// partials in z order.  D % 32 == 0; rows past T or E read zeros.
constexpr int kRLM = 128, kRLK = 32, kRLStages = 4, kRLPitch = kRLK + 4;  // floats per staged row
constexpr size_t kRLStageFloats = 2 * (size_t)kRLM * kRLPitch;
constexpr size_t kRLSmemBytes = kRLStages * kRLStageFloats * sizeof(float);

__device__ __forceinline__ void rl_cp_async16(float *smem, const float *gmem, bool valid) {
    // src-size 0 fills the 16 bytes with zeros (gmem stays a valid address)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem), "r"(valid ? 16 : 0)
                 : "memory");
}

__global__ void __launch_bounds__(256, 1) router_logits_kernel(const float *__restrict__ x, const float *__restrict__ Wr,
                                                               int T, int D, int E, float *__restrict__ logits) {
    extern __shared__ __align__(16) float rls[];  // [kRLStages][2][kRLM][kRLPitch]
    const int nch = D / kRLK, z = blockIdx.z, nz = gridDim.z;
    const int cb = (int)((long long)z * nch / nz), ce = (int)((long long)(z + 1) * nch / nz), n_c = ce - cb;
    logits += (size_t)z * T * E;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.x * kRLM, n0 = blockIdx.y * kRLM;
    // copy q = tid + 256 i of a stage: operand q / 512 (x, Wr), row (q / 4) % 128, 16-byte segment q % 4
    auto load_stage = [&](int stage, int chunk) {
        float *st = rls + (size_t)stage * kRLStageFloats;
#pragma unroll
        for (int i = 0; i < kRLK / 4; ++i) {
            const int q = tid + 256 * i, op = q / (kRLM * (kRLK / 4)), row = (q / (kRLK / 4)) % kRLM,
                      seg = q % (kRLK / 4);
            const int g = (op == 0 ? m0 : n0) + row, lim = op == 0 ? T : E;
            const float *src = (op == 0 ? x : Wr) + (size_t)(g < lim ? g : lim - 1) * D + chunk * kRLK + seg * 4;
            rl_cp_async16(st + (size_t)op * kRLM * kRLPitch + row * kRLPitch + seg * 4, src, g < lim);
        }
    };
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
#pragma unroll
    for (int s = 0; s < kRLStages - 1; ++s) {
        if (s < n_c) load_stage(s, cb + s);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    for (int c = 0; c < n_c; ++c) {
        // chunk c has landed (every later group may still be in flight), and
        // every thread is done with chunk c - 1, whose stage is refilled now
        asm volatile("cp.async.wait_group %0;" ::"n"(kRLStages - 2) : "memory");
        __syncthreads();
        if (c + kRLStages - 1 < n_c) load_stage((c + kRLStages - 1) % kRLStages, cb + c + kRLStages - 1);
        asm volatile("cp.async.commit_group;" ::: "memory");
        const float *As = rls + (size_t)(c % kRLStages) * kRLStageFloats, *Bs = As + kRLM * kRLPitch;
#pragma unroll
        for (int kk = 0; kk < kRLK; kk += 4) {
            float4 av[8], bv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) av[i] = *reinterpret_cast<const float4 *>(As + (ty + 16 * i) * kRLPitch + kk);
#pragma unroll
            for (int j = 0; j < 8; ++j) bv[j] = *reinterpret_cast<const float4 *>(Bs + (tx + 16 * j) * kRLPitch + kk);
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float v = acc[i][j];
                    v = fmaf(av[i].x, bv[j].x, v);
                    v = fmaf(av[i].y, bv[j].y, v);
                    v = fmaf(av[i].z, bv[j].z, v);
                    v = fmaf(av[i].w, bv[j].w, v);
                    acc[i][j] = v;
                }
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int t = m0 + ty + 16 * i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = n0 + tx + 16 * j;
            if (e < E) logits[(size_t)t * E + e] = acc[i][j];
        }
    }
}

// Top-K of a large batch from its logits (the sum of nz partial buffers in
// order): one warp per token (select_topk).
template <int EPL>
__global__ void __launch_bounds__(256) router_select_kernel(const float *__restrict__ logits, int nz,
                                                            const float *__restrict__ bias, int T, int E, int K,
                                                            float scale, float top_p, int32_t *__restrict__ idx,
                                                            float *__restrict__ w, int32_t *err) {
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= T) return;
    float c[EPL], p[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        const int e = lane + 32 * j;
        if (e < E) {
            float l = __ldg(logits + (size_t)t * E + e);
            for (int z = 1; z < nz; ++z) l = __fadd_rn(l, __ldg(logits + ((size_t)z * T + t) * E + e));
            score(l, __ldg(bias + e), p[j], c[j]);
        } else {
            p[j] = 0.f;
            c[j] = -INFINITY;
        }
    }
    select_topk<EPL>(c, p, E, K, scale, idx + (size_t)t * K, w + (size_t)t * K, nullptr, err, top_p);
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
    // the warp's selections kPB steps of 32 at a time, all loads of a batch
    // issued before the first is used; e = -1 for none or a dropped one
    constexpr int kPB = 16;
    auto load_batch = [&](int g0, int (&ev)[kPB]) {
#pragma unroll
        for (int j = 0; j < kPB; ++j) {
            const int i = g0 + 32 * j + lane;
            ev[j] = i < end ? __ldg(a.idx + i) : kDroppedSel;
        }
    };
    for (int g0 = beg; g0 < end; g0 += 32 * kPB) {
        int ev[kPB];
        load_batch(g0, ev);
#pragma unroll
        for (int j = 0; j < kPB; ++j) {
            int e = ev[j];
            const bool kept = e != kDroppedSel;  // a selection top-p dropped takes no row
            if (kept && (e < 0 || e >= E)) { e = 0; atomicOr(a.err, kErrRouteCount); }
            if (!kept) e = -1;
            const unsigned m = __match_any_sync(0xffffffffu, e);
            if (kept && __popc(m & lt) == 0) hist[warp * E + e] += __popc(m);
            __syncwarp();
        }
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
    const int n_kept = block_excl_scan(tot, base, E, wtot);
    const int n_routed = block_excl_scan(flg, upos, E, wtot);
    for (int e = tid; e < E; e += blockDim.x)
        if (tot[e] > 0) {
            a.meta->uexp[upos[e]] = e;
            a.meta->ubeg[upos[e]] = base[e];
        }
    if (tid == 0) {
        int nu = n_routed;
        a.meta->ubeg[n_routed] = n_kept;
        if (a.n_shared) {
            a.meta->uexp[n_routed] = E;
            a.meta->ubeg[n_routed + 1] = n_kept + T;
            nu += 1;
        }
        a.meta->n_union = nu;
        a.meta->n_gu_items = nu * a.nb_gu;
        a.meta->n_dn_items = nu * a.nb_dn;
    }
    for (int i = tid; i < 32 * E; i += blockDim.x) hist[i] += base[i % E];
    __syncthreads();
    for (int g0 = beg; g0 < end; g0 += 32 * kPB) {
        int ev[kPB];
        load_batch(g0, ev);
#pragma unroll
        for (int j = 0; j < kPB; ++j) {
            const int i = g0 + 32 * j + lane;
            int e = ev[j];
            const bool kept = e != kDroppedSel;
            if (kept && (e < 0 || e >= E)) e = 0;
            if (!kept) e = -1;
            const unsigned m = __match_any_sync(0xffffffffu, e);
            const int rank = __popc(m & lt);
            if (kept) a.rows[hist[warp * E + e] + rank] = (i / K) * S + (i % K);
            __syncwarp();
            if (kept && rank == 0) hist[warp * E + e] += __popc(m);
            __syncwarp();
        }
    }
    if (a.n_shared)
        for (int t = tid; t < T; t += blockDim.x) a.rows[n_kept + t] = t * S + K;
}

// ---------------------------------------------------------- launchers

static int epl_for(int E) { return E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : E <= 256 ? 8 : 16; }

cudaError_t launch_router_small(const LayerArgs &a, cudaStream_t s) {
    router_small_kernel<<<a.E + a.T, 256, 0, s>>>(a);
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

template <int EPL>
static cudaError_t launch_select_t(const float *logits, int nz, const float *bias, int T, int E, int K, float scale,
                                   float top_p, int32_t *idx, float *w, int32_t *err, cudaStream_t s) {
    router_select_kernel<EPL><<<(T + 7) / 8, 256, 0, s>>>(logits, nz, bias, T, E, K, scale, top_p, idx, w, err);
    return cudaGetLastError();
}

cudaError_t launch_router_gemm(const float *x, const float *Wr, const float *bias, int T, int D, int E, int K,
                               float scale, float top_p, float *logits, int32_t *idx, float *w, int32_t *err,
                               cudaStream_t s) {
    const int nz = D / kRLK < router_splits(T) ? D / kRLK : router_splits(T);
    cudaError_t ce = cudaFuncSetAttribute(router_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)kRLSmemBytes);
    if (ce != cudaSuccess) return ce;
    router_logits_kernel<<<dim3((T + kRLM - 1) / kRLM, (E + kRLM - 1) / kRLM, nz), 256, kRLSmemBytes, s>>>(
        x, Wr, T, D, E, logits);
    ce = cudaGetLastError();
    if (ce != cudaSuccess) return ce;
    switch (epl_for(E)) {
        case 1: return launch_select_t<1>(logits, nz, bias, T, E, K, scale, top_p, idx, w, err, s);
        case 2: return launch_select_t<2>(logits, nz, bias, T, E, K, scale, top_p, idx, w, err, s);
        case 4: return launch_select_t<4>(logits, nz, bias, T, E, K, scale, top_p, idx, w, err, s);
        case 8: return launch_select_t<8>(logits, nz, bias, T, E, K, scale, top_p, idx, w, err, s);
        default: return launch_select_t<16>(logits, nz, bias, T, E, K, scale, top_p, idx, w, err, s);
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
