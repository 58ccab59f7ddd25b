// k_stream.cu -- HBM-streaming expert kernels for decode-sized batches
// (at most 16 tokens per union expert).
//
// Sources: reader.mx "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型" §11 (SwiGLU
// expert on the batch's expert union, each expert's weights read once; h =
// siluf(gate)*up; down; weighted add) and §12 (int8 activations x int4
// weights, exact integer dot, then activation and row scales); besthub.dev
// "Running 744B MoE on 25GB RAM" §11, §12.
//
// Design (GB300): every CTA owns a contiguous range of row groups (a gate row
// with the same up row, or two down rows, of one union expert), so the union
// experts are streamed once, spread evenly over all SMs.  Warps take the
// CTA's groups round-robin and keep one packed row in flight ahead of the one
// they multiply: the 16-byte streaming loads (no L1 allocation) of the next
// unit are issued before the current one is computed.
// The activations of the current expert live in shared memory in the even/odd
// nibble-lane layout, staged once per expert the CTA meets (one CTA-wide
// barrier pair per expert boundary).  Offset nibbles go straight into dp4a
// (sum((n-8)x) = sum(nx) - 8 sum(x)), a warp reduction finishes each row.
#include "stream_dev.cuh"

namespace moe {

// Work list of one CTA: a contiguous range [p0, p1) of row groups over all
// union experts (gate/up: row pairs, each = a gate unit then an up unit;
// down: pairs of rows, each one unit).  Warp w takes groups p0 + w + 8i.
template <int KIND, int CPL, int MCH>
__global__ void __launch_bounds__(256) stream_kernel(LayerArgs a) {
    constexpr int UPG = KIND == kGateUp ? 2 : 1;        // units per row group
    constexpr int RPG = UnitShape<KIND, CPL>::kRows;          // output rows per row group
    extern __shared__ __align__(16) int8_t xs[];         // [MCH][kdim] even/odd int8 activations
    __shared__ int s_ent[MCH], s_xsum[MCH];
    __shared__ float s_sx[MCH];
    __shared__ int s_hpart[8][MCH];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.S;
    const int kdim = KIND == kGateUp ? a.D : a.I;
    const int rows_out = KIND == kGateUp ? a.I : a.D;
    const int rowb = kdim >> 1, nch = rowb >> 4;
    const int gpe = rows_out / RPG;  // row groups per expert
    const int n_groups = a.meta->n_union * gpe;
    const int p0 = (int)(((long long)blockIdx.x * n_groups) / gridDim.x);
    const int p1 = (int)(((long long)(blockIdx.x + 1) * n_groups) / gridDim.x);
    if (p0 >= p1) return;

    // unit j of this warp: group p0 + warp + 8*(j / UPG), matrix j % UPG
    const int n_my_groups = p1 - p0 > warp ? (p1 - p0 - warp + 7) / 8 : 0;
    const int n_my = n_my_groups * UPG;
    int ex_u = -1;
    DevExpert ex{};
    auto unit_src = [&](int j, const uint8_t *&mat, const float *&sc, int &o) {
        const int p = p0 + warp + 8 * (j / UPG), u = p / gpe;
        if (u != ex_u) {
            ex_u = u;
            ex = a.experts[a.meta->uexp[u]];
        }
        o = (p - u * gpe) * RPG;
        if (KIND == kGateUp) {
            mat = (j % UPG == 0) ? ex.gq : ex.uq;
            sc = (j % UPG == 0) ? ex.gs : ex.us;
        } else {
            mat = ex.dq;
            sc = ex.ds;
        }
    };
    UnitRegs<KIND, CPL> A, B;
    if (n_my > 0) {
        const uint8_t *mat;
        const float *sc;
        int o;
        unit_src(0, mat, sc, o);
        load_unit<KIND, CPL>(A, mat, sc, o, rowb, nch, lane);
    }

    float amax_run = 0.f;  // lane m: max|h| of token row m of the staged expert (gate/up)
    int hsum = 0;          // lane m: sum of the requantised h row m (down)
    int held_g = 0;        // lane m: gate sum waiting for its up row
    float held_gs = 0.f;   // that gate row's scale
    int r0 = 0, M = 0, j = 0;
    const int ua = p0 / gpe, ub = (p1 - 1) / gpe;
    for (int ue = ua; ue <= ub; ++ue) {
        // ---- stage the activations of union entry ue (every warp, every boundary)
        if (KIND == kGateUp && ue > ua && lane < M) atomicMax(a.hamax + r0 + lane, __float_as_uint(amax_run));
        __syncthreads();
        r0 = a.meta->ubeg[ue];
        M = a.meta->ubeg[ue + 1] - r0;
        if (M > MCH) {
            if (threadIdx.x == 0) atomicOr(a.err, kErrTooManyRows);
            M = MCH;
        }
        if (threadIdx.x < M) s_ent[threadIdx.x] = a.rows[r0 + threadIdx.x];
        __syncthreads();
        if (KIND == kGateUp) {
            if (threadIdx.x < M) {
                const int t = s_ent[threadIdx.x] / S;
                s_xsum[threadIdx.x] = a.xsum[t];
                s_sx[threadIdx.x] = a.sx[t];
            }
            const int n16 = kdim >> 4;
            for (int i = threadIdx.x; i < M * n16; i += blockDim.x) {
                const int m = i / n16, c = i - m * n16;
                *reinterpret_cast<int4 *>(plane_byte(xs, kdim, m, 16 * c)) =
                    __ldg(reinterpret_cast<const int4 *>(a.xq + (size_t)(s_ent[m] / S) * kdim) + c);
            }
        } else {
            const int n8 = kdim >> 3;
            const bool first_block = p0 <= ue * gpe;  // this CTA owns the expert's first rows
            for (int m = 0; m < M; ++m) {
                float s, inv;
                act_scale(__uint_as_float(__ldcg(a.hamax + r0 + m)), s, inv);
                if (threadIdx.x == 0) s_sx[m] = s;
                int sum = 0;
                for (int gi = threadIdx.x; gi < n8; gi += blockDim.x) {
                    const float *hp = a.h + (size_t)(r0 + m) * kdim + 8 * gi;
                    const float4 v0 = ld_cg_f4(hp), v1 = ld_cg_f4(hp + 4);
                    const int q0 = quant_i8(v0.x, inv), q1 = quant_i8(v0.y, inv), q2 = quant_i8(v0.z, inv),
                              q3 = quant_i8(v0.w, inv), q4 = quant_i8(v1.x, inv), q5 = quant_i8(v1.y, inv),
                              q6 = quant_i8(v1.z, inv), q7 = quant_i8(v1.w, inv);
                    sum += q0 + q1 + q2 + q3 + q4 + q5 + q6 + q7;
                    const uint32_t ev = (q0 & 255) | ((q2 & 255) << 8) | ((q4 & 255) << 16) | ((uint32_t)(q6 & 255) << 24);
                    const uint32_t od = (q1 & 255) | ((q3 & 255) << 8) | ((q5 & 255) << 16) | ((uint32_t)(q7 & 255) << 24);
                    *reinterpret_cast<uint2 *>(plane_byte(xs, kdim, m, 8 * gi)) = make_uint2(ev, od);
                    if (a.dbg.hq && first_block) {
                        const uint32_t n0 = (q0 & 255) | ((q1 & 255) << 8) | ((q2 & 255) << 16) | ((uint32_t)(q3 & 255) << 24);
                        const uint32_t n1 = (q4 & 255) | ((q5 & 255) << 8) | ((q6 & 255) << 16) | ((uint32_t)(q7 & 255) << 24);
                        *reinterpret_cast<uint2 *>(a.dbg.hq + (size_t)s_ent[m] * kdim + 8 * gi) = make_uint2(n0, n1);
                    }
                }
                sum = warp_sum_i(sum);
                if (lane == 0) s_hpart[warp][m] = sum;
            }
            if (a.dbg.sh && first_block && threadIdx.x < M) a.dbg.sh[s_ent[threadIdx.x]] = s_sx[threadIdx.x];
        }
        __syncthreads();
        if (KIND == kDown) {
            hsum = 0;
            if (lane < M)
#pragma unroll
                for (int w = 0; w < 8; ++w) hsum += s_hpart[w][lane];
        }
        amax_run = 0.f;

        // ---- this warp's units whose group belongs to union entry ue.  Two
        // register sets alternate: the next unit streams into one while the
        // other is multiplied.
        const int g_end = min(p1, (ue + 1) * gpe);  // groups of ue end here
        auto in_seg = [&](int jj) { return jj < n_my && p0 + warp + 8 * (jj / UPG) < g_end; };
        auto prefetch = [&](UnitRegs<KIND, CPL> &R, int jj) {
            if (jj < n_my) {
                const uint8_t *mat;
                const float *sc;
                int o;
                unit_src(jj, mat, sc, o);
                load_unit<KIND, CPL>(R, mat, sc, o, rowb, nch, lane);
            }
        };
        auto process = [&](const UnitRegs<KIND, CPL> &R, int jj) {
            const int p = p0 + warp + 8 * (jj / UPG);
            const int o0 = (p - ue * gpe) * RPG;
            if (KIND == kGateUp) {
                int acc[MCH];
#pragma unroll
                for (int m = 0; m < MCH; ++m) acc[m] = 0;
                dot_rows<CPL, MCH>(acc, R.w[0], xs, kdim, M, nch, lane);
                const int mine = lane_sum<MCH>(acc, M, lane);
                if (jj % UPG == 0) {
                    held_g = mine;
                    held_gs = R.s[0];
                } else if (lane < M) {
                    const int gi = held_g - 8 * s_xsum[lane], ui = mine - 8 * s_xsum[lane];
                    const float gf = __fmul_rn(__fmul_rn((float)gi, s_sx[lane]), held_gs);
                    const float uf = __fmul_rn(__fmul_rn((float)ui, s_sx[lane]), R.s[0]);
                    const float hv = __fmul_rn(silu_f(gf), uf);
                    a.h[(size_t)(r0 + lane) * a.I + o0] = hv;
                    amax_run = fmaxf(amax_run, fabsf(hv));
                    if (a.dbg.gate_acc) a.dbg.gate_acc[(size_t)s_ent[lane] * a.I + o0] = gi;
                    if (a.dbg.up_acc) a.dbg.up_acc[(size_t)s_ent[lane] * a.I + o0] = ui;
                }
            } else {
#pragma unroll
                for (int rr = 0; rr < RPG; ++rr) {
                    int acc[MCH];
#pragma unroll
                    for (int m = 0; m < MCH; ++m) acc[m] = 0;
                    dot_rows<CPL, MCH>(acc, R.w[rr], xs, kdim, M, nch, lane);
                    const int mine = lane_sum<MCH>(acc, M, lane);
                    if (lane < M) {
                        const int o = o0 + rr;
                        const int di = mine - 8 * hsum;
                        const float y = __fmul_rn(__fmul_rn((float)di, s_sx[lane]), R.s[rr]);
                        a.part[(size_t)s_ent[lane] * a.D + o] = y;
                        if (a.dbg.down_acc) a.dbg.down_acc[(size_t)s_ent[lane] * a.D + o] = di;
                    }
                }
            }
        };
        while (in_seg(j)) {
            prefetch(B, j + 1);
            process(A, j);
            ++j;
            if (!in_seg(j)) {
                A = B;  // the pipeline continues in A across the expert boundary
                break;
            }
            prefetch(A, j + 1);
            process(B, j);
            ++j;
        }
    }
    if (KIND == kGateUp && lane < M) atomicMax(a.hamax + r0 + lane, __float_as_uint(amax_run));
}

// ------------------------------------------------------------- launchers

static int mch_for(int T) { return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : T <= 8 ? 8 : 16; }
static int cpl_of(int kdim) {
    const int c = (kdim / 32 + 31) / 32;  // 16-byte chunks per lane of one packed row
    return c <= 1 ? 1 : c <= 2 ? 2 : c <= 4 ? 4 : c <= 6 ? 6 : 8;
}

bool stream_supported(int D, int I) { return D % 32 == 0 && I % 32 == 0 && D % 4 == 0; }

template <int KIND, int CPL, int MCH>
static cudaError_t launch_t(const LayerArgs &a, int num_sms, cudaStream_t s) {
    const int kdim = KIND == kGateUp ? a.D : a.I;
    const size_t smem = (size_t)MCH * kdim;
    auto fn = stream_kernel<KIND, CPL, MCH>;
    cudaError_t ce = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (ce != cudaSuccess) return ce;
    int occ = 1;
    ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, 256, smem);
    if (ce != cudaSuccess) return ce;
    occ = occ < 1 ? 1 : (occ > 4 ? 4 : occ);
    fn<<<num_sms * occ, 256, smem, s>>>(a);
    return cudaGetLastError();
}

template <int KIND, int CPL>
static cudaError_t launch_m(const LayerArgs &a, int num_sms, cudaStream_t s) {
    switch (mch_for(a.T)) {
        case 1: return launch_t<KIND, CPL, 1>(a, num_sms, s);
        case 2: return launch_t<KIND, CPL, 2>(a, num_sms, s);
        case 4: return launch_t<KIND, CPL, 4>(a, num_sms, s);
        case 8: return launch_t<KIND, CPL, 8>(a, num_sms, s);
        default: return launch_t<KIND, CPL, 16>(a, num_sms, s);
    }
}

template <int KIND>
static cudaError_t launch_k(const LayerArgs &a, int num_sms, cudaStream_t s) {
    switch (cpl_of(KIND == kGateUp ? a.D : a.I)) {
        case 1: return launch_m<KIND, 1>(a, num_sms, s);
        case 2: return launch_m<KIND, 2>(a, num_sms, s);
        case 4: return launch_m<KIND, 4>(a, num_sms, s);
        case 6: return launch_m<KIND, 6>(a, num_sms, s);
        default: return launch_m<KIND, 8>(a, num_sms, s);
    }
}

cudaError_t launch_gateup_stream(const LayerArgs &a, int num_sms, cudaStream_t s) {
    return launch_k<kGateUp>(a, num_sms, s);
}

cudaError_t launch_down_stream(const LayerArgs &a, int num_sms, cudaStream_t s) {
    return launch_k<kDown>(a, num_sms, s);
}

}  // namespace moe
