// k_grouped.cu -- tensor-core grouped GEMMs of the routed-MoE layer for
// batches where each union expert sees many tokens (prefill).
//
// Sources: reader.mx "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型" §11 (batch union:
// every expert's weights are read once and applied to all rows routed to it;
// SwiGLU expert) and §12 (int8 activations x int4 weights, exact integer dot,
// then activation and row scales); besthub.dev "Running 744B MoE on 25GB
// RAM" §11, §12.
//
// Design (GB300): exact int32 tensor-core MMAs (mma.sync m16n8k32, signed
// int8 activations x unsigned nibble codes; sum((n-8)x) = sum(nx) - 8 sum(x)
// restores the signed int4 weights).  A CTA tile is 64 token rows of one
// union expert x 128 weight rows (64 gate rows with the same 64 up rows, or
// 128 down rows), K in chunks of 128 through a 4-stage cp.async pipeline.
// Inside an MMA the K order is permuted identically on both operands: a
// packed weight word (one 8-element group) gives its low nibbles (elements
// 0,2,4,6) and high nibbles (1,3,5,7), which meet the two words of the
// even/odd activation layout; lane (g, t) of k-step j works on group 4t + j
// of the 128-element chunk.  Tiles are ordered (expert, weight block, token
// block) so the token blocks of one weight block run back to back and share
// it through L2.  A persistent grid walks the tiles.
#include <cuda_fp16.h>

#include "layer_args.cuh"

namespace moe {

namespace {

constexpr int kBM = 64;            // token rows per tile
constexpr int kBN = 128;           // weight rows per tile
constexpr int kBK = 128;           // K elements per stage (64 packed bytes per weight row)
constexpr int kStages = 4;
constexpr int kApitch = kBK + 16;  // smem bytes per activation row (no bank conflicts)
constexpr int kBpitch = kBK / 2;   // smem bytes per weight row

enum GemmKind { kGU = 0, kDN = 1 };

struct StageSmem {
    int8_t A[kBM * kApitch];
    uint8_t B[kBN * kBpitch];
};

constexpr size_t kSmemStages = sizeof(StageSmem) * kStages;
// per-tile tables after the stages: tok/ent/xsum [kBM] int, sx [kBM] float,
// scales [kBN] float, amax [kBM] uint, m-block prefix [kMaxE + 2] int
constexpr size_t kSmemTotal = kSmemStages + 4 * (4 * kBM + kBN) + 4 * kBM + 4 * (kMaxE + 2);

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// D[16x8] += A[16x32] (s8) * B[32x8] (u8), int32 accumulate.
__device__ __forceinline__ void mma_s8u8(int (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.u8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word_of(const int4 (&v)[2], int i) {
    const int4 &q = v[i >> 2];
    const int r = i & 3;
    return (uint32_t)(r == 0 ? q.x : r == 1 ? q.y : r == 2 ? q.z : q.w);
}

__device__ __forceinline__ uint32_t word_of1(const int4 &q, int r) {
    return (uint32_t)(r == 0 ? q.x : r == 1 ? q.y : r == 2 ? q.z : q.w);
}

}  // namespace

// KIND = kGU: A = int8 activations of the expert's tokens (gathered from xq by
//   token), B = 64 gate rows + the same 64 up rows; epilogue h = silu(g) * u
//   per (token row, output row), max|h| per row.
// KIND = kDN: A = requantised h rows of the expert (contiguous grouped rows),
//   B = 128 down rows; epilogue y = (acc*sh)*sd into part[entry].
template <int KIND>
__global__ void __launch_bounds__(256) grouped_gemm_kernel(LayerArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    StageSmem *st = reinterpret_cast<StageSmem *>(smem);
    int *s_src = reinterpret_cast<int *>(smem + kSmemStages);  // A source row (token or grouped row)
    int *s_ent = s_src + kBM;
    int *s_xsum = s_ent + kBM;
    float *s_sx = reinterpret_cast<float *>(s_xsum + kBM);
    float *s_sc = s_sx + kBM;                                   // [kBN] weight row scales
    unsigned *s_amax = reinterpret_cast<unsigned *>(s_sc + kBN);
    int *s_mbeg = reinterpret_cast<int *>(s_amax + kBM);        // [n_union + 1]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tg = lane & 3;
    const int wm = warp >> 2, wn = warp & 3;  // 2 x 4 warps: 32 token rows x 32 weight rows each
    const int S = a.S;
    const int kdim = KIND == kGU ? a.D : a.I;
    const int rowb = kdim >> 1;
    const int nbe = KIND == kGU ? a.I / (kBN / 2) : a.D / kBN;  // weight blocks per expert
    const int nks = kdim / kBK;                                 // K stages per tile
    const int nu = a.meta->n_union;

    // token blocks per union entry, prefix in shared memory
    if (warp == 0) {
        int run = 0;
        for (int u0 = 0; u0 < nu; u0 += 32) {
            const int u = u0 + lane;
            const int mbk = u < nu ? (a.meta->ubeg[u + 1] - a.meta->ubeg[u] + kBM - 1) / kBM : 0;
            int incl = mbk;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (u < nu) s_mbeg[u] = run + incl - mbk;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) s_mbeg[nu] = run;
    }
    __syncthreads();
    const int n_tiles = s_mbeg[nu] * nbe;

    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        // ---- decode (expert, weight block, token block)
        int lo = 0, hi = nu - 1;
        while (lo < hi) {  // last u with s_mbeg[u] * nbe <= tile
            const int mid = (lo + hi + 1) >> 1;
            if (s_mbeg[mid] * nbe <= tile) lo = mid; else hi = mid - 1;
        }
        const int u = lo;
        const int mbu = s_mbeg[u + 1] - s_mbeg[u];
        const int local = tile - s_mbeg[u] * nbe;
        const int nb = local / mbu, mb = local - nb * mbu;
        const int r0 = a.meta->ubeg[u];
        const int M = a.meta->ubeg[u + 1] - r0;
        const int mrow0 = mb * kBM;                 // first token row of the tile inside the expert
        const int valid = min(kBM, M - mrow0);
        const DevExpert ex = a.experts[a.meta->uexp[u]];

        __syncthreads();  // the previous tile's epilogue is done with the tables
        if (tid < kBM) {
            const int m = tid < valid ? tid : 0;    // padding rows repeat a real row
            const int r = r0 + mrow0 + m;
            const int ent = a.rows[r];
            s_ent[tid] = ent;
            if (KIND == kGU) {
                const int t = ent / S;
                s_src[tid] = t;
                s_xsum[tid] = a.xsum[t];
                s_sx[tid] = a.sx[t];
            } else {
                s_src[tid] = r;
                s_xsum[tid] = a.hsum[r];
                s_sx[tid] = a.shq[r];
            }
            s_amax[tid] = 0u;
        }
        if (tid < kBN) {
            if (KIND == kGU)
                s_sc[tid] = tid < 64 ? __ldg(ex.gs + nb * 64 + tid) : __ldg(ex.us + nb * 64 + tid - 64);
            else
                s_sc[tid] = __ldg(ex.ds + nb * kBN + tid);
        }
        __syncthreads();

        // ---- K loop: 4-stage cp.async pipeline
        const int8_t *Asrc = KIND == kGU ? a.xq : a.hq;
        auto load_stage = [&](int ks) {
            StageSmem &S_ = st[ks % kStages];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int c = tid + 256 * i;
                const int row = c >> 3, c16 = c & 7;  // 64 rows x 8 chunks of 16 B
                cp_async16(S_.A + row * kApitch + c16 * 16,
                           Asrc + (size_t)s_src[row] * kdim + (size_t)ks * kBK + c16 * 16);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int c = tid + 256 * i;
                const int row = c >> 2, q = c & 3;    // 128 rows x 4 chunks of 16 B
                const uint8_t *wrow;
                if (KIND == kGU)
                    wrow = row < 64 ? ex.gq + (size_t)(nb * 64 + row) * rowb
                                    : ex.uq + (size_t)(nb * 64 + row - 64) * rowb;
                else
                    wrow = ex.dq + (size_t)(nb * kBN + row) * rowb;
                cp_async16(S_.B + row * kBpitch + q * 16, wrow + (size_t)ks * (kBK / 2) + q * 16);
            }
        };

        int acc[2][4][4];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0;

#pragma unroll
        for (int p = 0; p < kStages - 1; ++p) {
            if (p < nks) load_stage(p);
            cp_async_commit();
        }
        for (int ks = 0; ks < nks; ++ks) {
            cp_async_wait<kStages - 2>();
            __syncthreads();  // stage ks visible to all; stage ks-1 fully consumed
            if (ks + kStages - 1 < nks) load_stage(ks + kStages - 1);
            cp_async_commit();
            const StageSmem &S_ = st[ks % kStages];
            int4 xa[2][2], xb[2][2], wb[4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const int row = wm * 32 + mt * 16 + g;
                const int4 *pa = reinterpret_cast<const int4 *>(S_.A + row * kApitch + 32 * tg);
                const int4 *pb = reinterpret_cast<const int4 *>(S_.A + (row + 8) * kApitch + 32 * tg);
                xa[mt][0] = pa[0];
                xa[mt][1] = pa[1];
                xb[mt][0] = pb[0];
                xb[mt][1] = pb[1];
            }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int row = KIND == kGU ? ((nt < 2 ? 0 : 64) + wn * 16 + (nt & 1) * 8 + g) : (wn * 32 + nt * 8 + g);
                wb[nt] = *reinterpret_cast<const int4 *>(S_.B + row * kBpitch + 16 * tg);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const uint32_t w = word_of1(wb[nt], j);
                    const uint32_t lo4 = w & 0x0F0F0F0Fu, hi4 = (w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt)
                        mma_s8u8(acc[mt][nt], word_of(xa[mt], 2 * j), word_of(xb[mt], 2 * j),
                                 word_of(xa[mt], 2 * j + 1), word_of(xb[mt], 2 * j + 1), lo4, hi4);
                }
            }
        }
        cp_async_wait<0>();

        // ---- epilogue
        if (KIND == kGU) {
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int m = wm * 32 + mt * 16 + g + 8 * half;
                    float mx = 0.f;
#pragma unroll
                    for (int np = 0; np < 2; ++np) {
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            const int i = 2 * half + cc;
                            const int ol = wn * 16 + np * 8 + 2 * tg + cc;  // 0..63
                            if (m < valid) {
                                const int gi = acc[mt][np][i] - 8 * s_xsum[m];
                                const int ui = acc[mt][np + 2][i] - 8 * s_xsum[m];
                                const float gf = __fmul_rn(__fmul_rn((float)gi, s_sx[m]), s_sc[ol]);
                                const float uf = __fmul_rn(__fmul_rn((float)ui, s_sx[m]), s_sc[64 + ol]);
                                const float hv = __fmul_rn(silu_f(gf), uf);
                                const int o = nb * 64 + ol;
                                a.h[(size_t)(r0 + mrow0 + m) * a.I + o] = hv;
                                mx = fmaxf(mx, fabsf(hv));
                                if (a.dbg.gate_acc) a.dbg.gate_acc[(size_t)s_ent[m] * a.I + o] = gi;
                                if (a.dbg.up_acc) a.dbg.up_acc[(size_t)s_ent[m] * a.I + o] = ui;
                            }
                        }
                    }
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    if (tg == 0 && m < valid) atomicMax(&s_amax[m], __float_as_uint(mx));
                }
            }
            __syncthreads();
            if (tid < valid) atomicMax(a.hamax + r0 + mrow0 + tid, s_amax[tid]);
        } else {
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int m = wm * 32 + mt * 16 + g + 8 * (i >> 1);
                        const int ol = wn * 32 + nt * 8 + 2 * tg + (i & 1);
                        if (m < valid) {
                            const int di = acc[mt][nt][i] - 8 * s_xsum[m];
                            const float y = __fmul_rn(__fmul_rn((float)di, s_sx[m]), s_sc[ol]);
                            const int o = nb * kBN + ol;
                            a.part[(size_t)s_ent[m] * a.D + o] = y;
                            if (a.dbg.down_acc) a.dbg.down_acc[(size_t)s_ent[m] * a.D + o] = di;
                        }
                    }
                }
            }
        }
    }
}

// Requantise every grouped h row to int8 (the activation quantiser of [A] §12
// with the row max|h| of the gate/up pass) in the even/odd lane layout, with
// the row code sum and scale.  kRQ grouped rows per CTA, every row's loads of
// a pass issued before the first is used (a CTA per row left each thread one
// row's loads in flight).
constexpr int kRQ = 4;
__global__ void __launch_bounds__(256) requant_h_kernel(LayerArgs a) {
    __shared__ int red_i[kRQ][8];
    // grouped rows of this batch: T*S, fewer when adaptive top-p dropped selections
    const int n_rows = a.meta->ubeg[a.meta->n_union];
    const int I = a.I, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = blockIdx.x * kRQ;
    if (r0 >= n_rows) return;
    float sc[kRQ], inv[kRQ];
    int sum[kRQ], ent[kRQ];
#pragma unroll
    for (int j = 0; j < kRQ; ++j) {
        const bool ok = r0 + j < n_rows;
        act_scale(ok ? __uint_as_float(a.hamax[r0 + j]) : 0.f, sc[j], inv[j]);
        ent[j] = ok ? a.rows[r0 + j] : 0;
        sum[j] = 0;
    }
    for (int gi = threadIdx.x; gi < (I >> 3); gi += blockDim.x) {
        float4 v0[kRQ], v1[kRQ];
#pragma unroll
        for (int j = 0; j < kRQ; ++j) {
            if (r0 + j < n_rows) {
                const float *hp = a.h + (size_t)(r0 + j) * I + 8 * gi;
                v0[j] = *reinterpret_cast<const float4 *>(hp);
                v1[j] = *reinterpret_cast<const float4 *>(hp + 4);
            }
        }
#pragma unroll
        for (int j = 0; j < kRQ; ++j) {
            if (r0 + j >= n_rows) continue;
            const int r = r0 + j;
            const float iv = inv[j];
            const int q0 = quant_i8(v0[j].x, iv), q1 = quant_i8(v0[j].y, iv), q2 = quant_i8(v0[j].z, iv),
                      q3 = quant_i8(v0[j].w, iv), q4 = quant_i8(v1[j].x, iv), q5 = quant_i8(v1[j].y, iv),
                      q6 = quant_i8(v1[j].z, iv), q7 = quant_i8(v1[j].w, iv);
            sum[j] += q0 + q1 + q2 + q3 + q4 + q5 + q6 + q7;
            const uint32_t ev = (q0 & 255) | ((q2 & 255) << 8) | ((q4 & 255) << 16) | ((uint32_t)(q6 & 255) << 24);
            const uint32_t od = (q1 & 255) | ((q3 & 255) << 8) | ((q5 & 255) << 16) | ((uint32_t)(q7 & 255) << 24);
            *reinterpret_cast<uint2 *>(a.hq + (size_t)r * I + 8 * gi) = make_uint2(ev, od);
            if (a.xf) {  // the tcgen05 GEMM's operand: the same codes as f16 integers, same order
                auto h2 = [](int lo, int hi) {
                    return (uint32_t)__half_as_ushort(__int2half_rn(lo)) | ((uint32_t)__half_as_ushort(__int2half_rn(hi)) << 16);
                };
                *reinterpret_cast<uint4 *>(a.xf + (size_t)r * I + 8 * gi) =
                    make_uint4(h2(q0, q2), h2(q4, q6), h2(q1, q3), h2(q5, q7));
            }
            if (a.dbg.hq) {
                const uint32_t n0 = (q0 & 255) | ((q1 & 255) << 8) | ((q2 & 255) << 16) | ((uint32_t)(q3 & 255) << 24);
                const uint32_t n1 = (q4 & 255) | ((q5 & 255) << 8) | ((q6 & 255) << 16) | ((uint32_t)(q7 & 255) << 24);
                *reinterpret_cast<uint2 *>(a.dbg.hq + (size_t)ent[j] * I + 8 * gi) = make_uint2(n0, n1);
            }
        }
    }
    // the rows' code sums: warp sums, then thread j adds row j's
#pragma unroll
    for (int j = 0; j < kRQ; ++j) {
        const int w = warp_sum_i(sum[j]);
        if (lane == 0) red_i[j][warp] = w;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kRQ; ++j) {
        if ((int)threadIdx.x == j && r0 + j < n_rows) {
            int t = 0;
            for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red_i[j][w];
            a.hsum[r0 + j] = t;
            a.shq[r0 + j] = sc[j];
            if (a.dbg.sh) a.dbg.sh[ent[j]] = sc[j];
        }
    }
}

// ------------------------------------------------------------- launchers

bool grouped_supported(int D, int I) { return D % kBK == 0 && I % kBK == 0 && I % 64 == 0 && D % kBN == 0; }

size_t grouped_smem_bytes() { return kSmemTotal; }

template <int KIND>
static cudaError_t launch_g(const LayerArgs &a, int num_sms, cudaStream_t s) {
    auto fn = grouped_gemm_kernel<KIND>;
    cudaError_t ce = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemTotal);
    if (ce != cudaSuccess) return ce;
    int occ = 1;
    ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, 256, kSmemTotal);
    if (ce != cudaSuccess) return ce;
    occ = occ < 1 ? 1 : (occ > 4 ? 4 : occ);
    fn<<<num_sms * occ, 256, kSmemTotal, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_grouped_gateup(const LayerArgs &a, int num_sms, cudaStream_t s) {
    return launch_g<kGU>(a, num_sms, s);
}

cudaError_t launch_requant_h(const LayerArgs &a, cudaStream_t s) {
    requant_h_kernel<<<(a.T * a.S + kRQ - 1) / kRQ, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_grouped_down(const LayerArgs &a, int num_sms, cudaStream_t s) {
    return launch_g<kDN>(a, num_sms, s);
}

}  // namespace moe
