// decode_dev.cuh -- the routed-MoE layer for decode-sized batches (1 to 16
// tokens) as one persistent kernel: activation quantiser, sigmoid+bias top-K
// router, expert union, fused gate/up, down and the ordered weighted sum.
//
// Sources: reader.mx "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型" §11 (router:
// sigmoid(logit)+bias picks top-K, weight = plain sigmoid * routed_scale;
// the batch union so each expert's weights are read once; SwiGLU expert
// h = siluf(gate)*up, down, weighted add, shared expert added) and §12 (int8
// per-row activations x int4 weights with an exact integer dot, then the
// activation and row scales); besthub.dev "Running 744B MoE on 25GB RAM"
// §11, §12.
//
// Design (GB300).  At decode sizes the layer reads ~19 MB per union expert
// and does almost no arithmetic: it is one long weight stream, and every
// kernel boundary costs a ramp-up and a tail of several microseconds.  So the
// whole layer is one cooperative launch with every CTA resident (2 per SM),
// moving through three phases that hand data over through L2:
//   1. CTA b < E computes the logits of experts b, b + G, ... (its router
//      row is requested first: everything downstream waits on the logits)
//      and publishes each as data (the slot itself is the flag).  At one
//      token every CTA quantises the token into its own tile from the
//      registers the router loads brought; for T > 1 the last T CTAs
//      quantise one token each (arrival counter).  At one token every CTA
//      also streams its slice of the shared expert's gate/up, which needs
//      no routing (a router CTA requests those rows once its logits are
//      out).  Meanwhile CTA G-1-t polls token t's logits, selects its top-K
//      and publishes the selections as data.
//   2. Every CTA polls the published selections and builds the union
//      tables itself, in shared memory; then it streams its contiguous
//      slice of the routed experts' gate/up rows (for T > 1 with the shared
//      expert's; slices weighted by measured per-group costs; h to L2).
//   3. A grid-wide arrival barrier; each CTA arrives, then requests its
//      first down rows, then waits.  The CTA stages the h rows of the
//      entries in its slice (max|h| of each row by a block reduction of the
//      loaded values, then the int8 codes) and streams their down rows into
//      per-slot partial outputs; at one token the CTAs form one run per
//      union entry.  An arrival counter per block of 64 output rows sums the
//      rows written; the CTA that completes a block adds that block's slots
//      in the fixed slot order (shared expert last), so the result does not
//      depend on which CTA arrives when.
// Every wait is bounded (one second of %globaltimer): on time-out the kernel
// sets kErrSyncTimeout in the error word and runs on to its end, so nothing
// hangs and the stream stays usable.  The counters and hand-over buffers
// come in two sets used by alternate launches (DecodeState): each launch
// restores the set the previous one used, so no CTA waits at the end.
#pragma once

#include <type_traits>

#include "route_dev.cuh"
#include "stream_dev.cuh"

namespace moe {
namespace dec {

constexpr int kMaxContrib = 128;                       // reduce-block arrivals listed per CTA
constexpr int kTabEntries = kMaxK + 1;                 // union entries of one token (pointers kept in shared memory)

// Thread 0 records phase stamp k of this CTA when tracing is on.
__device__ __forceinline__ void stamp(const LayerArgs &a, int k) {
    if (a.trace && threadIdx.x == 0 && (long long)(blockIdx.x + 1) * kTraceStamps <= a.trace_n)
        a.trace[(size_t)blockIdx.x * kTraceStamps + k] = global_ns();
}

// All threads: the CTA's global writes so far become visible device-wide,
// then *cnt += 1.
__device__ __forceinline__ void cta_arrive(int *cnt) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(cnt, 1);
    }
}

// All threads: wait (bounded) until *cnt >= target; afterwards everything the
// arriving CTAs wrote before arriving is visible to every thread of the CTA.
__device__ __forceinline__ void cta_wait(const int *cnt, int target, int32_t *err) {
    if (threadIdx.x == 0) {
        if (ld_acquire(cnt) < target) {
            const unsigned long long t0 = global_ns();
            while (ld_acquire(cnt) < target) {
                if (global_ns() - t0 > kWaitNs) {
                    atomicOr(err, kErrSyncTimeout);
                    break;
                }
                __nanosleep(32);
            }
        }
        __threadfence();
    }
    __syncthreads();
}

// Shared-memory state of one CTA (besides the activation tile).
struct DecodeSmem {
    int ent[kSmallT];                 // entry ids (t*S + slot) of the staged expert's rows
    int xsum[kSmallT];                // code sums of those activation rows
    float sx[kSmallT];                // their scales
    int hpart[8][kSmallT];            // per-warp partial code sums of requantised h rows
    float red[8][kSmallT];            // per-warp partial logits
    int idx[kSmallT * kMaxK];         // top-K selections, (token, slot) order
    float w[kSmallT * kMaxK];         // their routing weights
    int first[kSmallT * kMaxK];       // selection is its expert's first
    int rows[kSmallT * (kMaxK + 1)];  // entry ids grouped by union entry
    int uexp[kSmallT * kMaxK + 1];    // union entry -> expert (shared expert = E, last)
    int ubeg[kSmallT * kMaxK + 2];    // union entry -> first grouped row
    int sh_uexp[1];                   // one-entry view of the shared expert
    int sh_ubeg[2];
    DevExpert uexd[kTabEntries];      // one token: the union entries' expert pointers
    int nu;                           // routed union entries
    int nblk;                         // reduce blocks this CTA completed
    unsigned int epoch;               // the launch's epoch (DecodeState)
    int slice[4];                     // this CTA's routed gate/up and down group ranges
    int blk_list[kMaxRedBlk];          // reduce blocks this CTA completed
    int ncontrib;                      // (block, rows) contributions listed
    int2 contrib[kMaxContrib];
    unsigned long long tk[4][8][kMaxK];  // top-K candidates (topk_small_cta)
    float tkp[4][8][kMaxK];              // their sigmoids
};

template <int KIND>
__device__ __forceinline__ int units_of_warp(int p0, int p1, int warp) {
    constexpr int UPG = KIND == kGateUp ? 2 : 1;
    return p1 - p0 > warp ? ((p1 - p0 - warp + 7) / 8) * UPG : 0;
}

// Requests unit j of this warp (group p0 + warp + 8*(j / UPG) of the union
// view, matrix j % UPG) into R.  ex_u/ex cache the current expert's pointers,
// read from tab[entry] when the CTA holds them in shared memory, else from
// the global expert table.
template <int KIND, int CPL>
__device__ __forceinline__ void request(UnitRegs<KIND, CPL> &R, const LayerArgs &a, const int *uexp, int gpe,
                                        int p0, int n_my, int j, int &ex_u, DevExpert &ex,
                                        const DevExpert *tab = nullptr) {
    constexpr int UPG = KIND == kGateUp ? 2 : 1, RPG = UnitShape<KIND, CPL>::kRows;
    if (j >= n_my) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kdim = KIND == kGateUp ? a.D : a.I;
    const int rowb = kdim >> 1, nch = rowb >> 4;
    const int p = p0 + warp + 8 * (j / UPG), u = p / gpe;
    if (u != ex_u) {
        ex_u = u;
        ex = tab ? tab[u] : a.experts[uexp[u]];
    }
    const int o = (p - u * gpe) * RPG;
    const uint8_t *mat;
    const float *sc;
    if (KIND == kGateUp) {
        mat = (j % UPG == 0) ? ex.gq : ex.uq;
        sc = (j % UPG == 0) ? ex.gs : ex.us;
    } else {
        mat = ex.dq;
        sc = ex.ds;
    }
    load_unit<KIND, CPL>(R, mat, sc, o, rowb, nch, lane);
}

// Requests the first two units of the warp's share of groups [p0, p1).
template <int KIND, int CPL>
__device__ __forceinline__ void prime(UnitRegs<KIND, CPL> &A, UnitRegs<KIND, CPL> &B, const LayerArgs &a,
                                      const int *uexp, int gpe, int p0, int p1, int &ex_u, DevExpert &ex,
                                      const DevExpert *tab = nullptr) {
    const int n_my = units_of_warp<KIND>(p0, p1, threadIdx.x >> 5);
    ex_u = -1;
    request<KIND, CPL>(A, a, uexp, gpe, p0, n_my, 0, ex_u, ex, tab);
    request<KIND, CPL>(B, a, uexp, gpe, p0, n_my, 1, ex_u, ex, tab);
}

// Streams row groups [p0, p1) of a union view (gate/up: a gate row with the
// same up row; down: two rows) through the CTA's eight warps; A and B hold
// the warp's first two units (prime).  Per union entry the CTA stages the
// activations (gate/up: the quantised tokens; down: h requantised from L2)
// in the two-plane layout, then each warp multiplies its units while the
// next one is in flight.  Must be called by all threads with the same range.
// At one token, hset (when not null) receives the h values as data (each
// value its own flag) and the down staging reads them from there.
template <int KIND, int CPL, int MCH>
__device__ __forceinline__ void stream_phase(const LayerArgs &a, DecodeSmem &sm, int8_t *xs, const int *uexp,
                                             const int *ubeg, int p0, int p1, UnitRegs<KIND, CPL> &A,
                                             UnitRegs<KIND, CPL> &B, int &ex_u, DevExpert &ex, float *hset,
                                             const DevExpert *tab = nullptr) {
    constexpr int UPG = KIND == kGateUp ? 2 : 1, RPG = UnitShape<KIND, CPL>::kRows;
    // at one token every gate/up entry multiplies the same row (token 0),
    // staged once in xs / sm.sx[0] / sm.xsum[0] by the caller
    constexpr bool kFixedX = KIND == kGateUp && MCH == 1;
    if (p0 >= p1) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.S;
    const int kdim = KIND == kGateUp ? a.D : a.I;
    const int rows_out = KIND == kGateUp ? a.I : a.D;
    const int nch = (kdim >> 1) >> 4;
    const int gpe = rows_out / RPG;
    const int n_my = units_of_warp<KIND>(p0, p1, warp);

    if constexpr (kFixedX) {
        // one token: one row per entry and nothing staged per entry, so
        // each warp runs straight through the entries of its units, with no
        // block barrier between entries (a group is a gate row and the same
        // up row)
        int held_g = 0;
        float held_gs = 0.f;
        auto process1 = [&](const UnitRegs<KIND, CPL> &R, int jj) {
            const int p = p0 + warp + 8 * (jj / UPG), ue = p / gpe, o0 = p - ue * gpe;
            int acc[1] = {0};
            dot_rows<CPL, 1>(acc, R.w[0], xs, kdim, 1, nch, lane);
            const int mine = lane_sum<1>(acc, 1, lane);
            if (jj % UPG == 0) {
                held_g = mine;
                held_gs = R.s[0];
            } else if (lane == 0) {
                const int r0 = ubeg[ue];
                const int gi = held_g - 8 * sm.xsum[0], ui = mine - 8 * sm.xsum[0];
                const float gf = __fmul_rn(__fmul_rn((float)gi, sm.sx[0]), held_gs);
                const float uf = __fmul_rn(__fmul_rn((float)ui, sm.sx[0]), R.s[0]);
                const float hv = __fmul_rn(silu_f(gf), uf);
                if (hset) {  // published as data: the down CTAs poll it
                    const uint32_t bits = __float_as_uint(hv);
                    st_relaxed_u32(hset + (size_t)r0 * a.I + o0, bits == kHEmpty ? 0x7FFFFFFFu : bits);
                } else {
                    a.h[(size_t)r0 * a.I + o0] = hv;
                }
                if (a.dbg.gate_acc) a.dbg.gate_acc[(size_t)sm.rows[r0] * a.I + o0] = gi;
                if (a.dbg.up_acc) a.dbg.up_acc[(size_t)sm.rows[r0] * a.I + o0] = ui;
            }
        };
        for (int j = 0; j < n_my;) {
            process1(A, j);
            request<KIND, CPL>(A, a, uexp, gpe, p0, n_my, j + 2, ex_u, ex, tab);
            if (++j >= n_my) break;
            process1(B, j);
            request<KIND, CPL>(B, a, uexp, gpe, p0, n_my, j + 2, ex_u, ex, tab);
            ++j;
        }
        return;
    }

    int hsum = 0;          // lane m: code sum of the requantised h row m (down)
    int held_g = 0;        // lane m: gate sum waiting for its up row
    float held_gs = 0.f;   // that gate row's scale
    int r0 = 0, M = 0, j = 0;
    bool flip = false;     // the next unit is in B
    const int ua = p0 / gpe, ub = (p1 - 1) / gpe;
    for (int ue = ua; ue <= ub; ++ue) {
        __syncthreads();
        r0 = ubeg[ue];
        M = ubeg[ue + 1] - r0;
        if (M > MCH) {
            if (threadIdx.x == 0) atomicOr(a.err, kErrTooManyRows);
            M = MCH;
        }
        if (threadIdx.x < M) sm.ent[threadIdx.x] = sm.rows[r0 + threadIdx.x];
        __syncthreads();
        if (KIND == kGateUp) {  // (one token took the path above)
            if (threadIdx.x < M) {
                const int t = sm.ent[threadIdx.x] / S;
                sm.xsum[threadIdx.x] = __ldcg(a.xsum + t);
                sm.sx[threadIdx.x] = __ldcg(a.sx + t);
            }
            const int n16 = kdim >> 4;
            for (int i = threadIdx.x; i < M * n16; i += blockDim.x) {
                const int m = i / n16, c = i - m * n16;
                *reinterpret_cast<int4 *>(plane_byte(xs, kdim, m, 16 * c)) =
                    __ldcg(reinterpret_cast<const int4 *>(a.xq + (size_t)(sm.ent[m] / S) * kdim) + c);
            }
        } else {
            // the entry's h rows, one 8-group per thread (the down chunk
            // counts instantiated give I <= 2048 = 8 * blockDim): max|h| of
            // the row by a block reduction of the loaded values, then the
            // scale, the codes and their sum
            static_assert(KIND != kDown || CPL <= 2, "one 8-group of an h row per thread");
            const int n8 = kdim >> 3, gi = threadIdx.x;
            const bool first_block = p0 <= ue * gpe;  // this CTA owns the entry's first rows
            for (int m = 0; m < M; ++m) {
                float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
                if (gi < n8) {
                    if (MCH == 1 && hset) {
                        // one token: the h values are their own flags (the
                        // gate/up CTAs write them with no fence or counter);
                        // this thread's 8 are read until none is still empty
                        const float *hp = hset + (size_t)(r0 + m) * kdim + 8 * gi;
                        const unsigned long long t0 = global_ns();
                        for (;;) {
                            const uint4 w0 = ld_relaxed_v4(hp), w1 = ld_relaxed_v4(hp + 4);
                            v0 = make_float4(__uint_as_float(w0.x), __uint_as_float(w0.y), __uint_as_float(w0.z),
                                             __uint_as_float(w0.w));
                            v1 = make_float4(__uint_as_float(w1.x), __uint_as_float(w1.y), __uint_as_float(w1.z),
                                             __uint_as_float(w1.w));
                            const bool empty = w0.x == kHEmpty || w0.y == kHEmpty || w0.z == kHEmpty ||
                                               w0.w == kHEmpty || w1.x == kHEmpty || w1.y == kHEmpty ||
                                               w1.z == kHEmpty || w1.w == kHEmpty;
                            if (!empty) break;
                            if (global_ns() - t0 > kWaitNs) {
                                atomicOr(a.err, kErrSyncTimeout);
                                break;
                            }
                            __nanosleep(32);
                        }
                    } else {
                        const float *hp = a.h + (size_t)(r0 + m) * kdim + 8 * gi;
                        v0 = ld_cg_f4(hp);
                        v1 = ld_cg_f4(hp + 4);
                    }
                }
                float amax = fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                                   fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w))));
                amax = block_max_nonneg(amax, &sm.red[0][0]);
                float s, inv;
                act_scale(amax, s, inv);
                if (threadIdx.x == 0) sm.sx[m] = s;
                if (a.dbg.sh && first_block && threadIdx.x == m) a.dbg.sh[sm.ent[m]] = s;
                int sum = 0;
                if (gi < n8) {
                    const int q0 = quant_i8(v0.x, inv), q1 = quant_i8(v0.y, inv), q2 = quant_i8(v0.z, inv),
                              q3 = quant_i8(v0.w, inv), q4 = quant_i8(v1.x, inv), q5 = quant_i8(v1.y, inv),
                              q6 = quant_i8(v1.z, inv), q7 = quant_i8(v1.w, inv);
                    sum = q0 + q1 + q2 + q3 + q4 + q5 + q6 + q7;
                    const uint32_t ev = (q0 & 255) | ((q2 & 255) << 8) | ((q4 & 255) << 16) | ((uint32_t)(q6 & 255) << 24);
                    const uint32_t od = (q1 & 255) | ((q3 & 255) << 8) | ((q5 & 255) << 16) | ((uint32_t)(q7 & 255) << 24);
                    *reinterpret_cast<uint2 *>(plane_byte(xs, kdim, m, 8 * gi)) = make_uint2(ev, od);
                    if (a.dbg.hq && first_block) {
                        const uint32_t n0 = (q0 & 255) | ((q1 & 255) << 8) | ((q2 & 255) << 16) | ((uint32_t)(q3 & 255) << 24);
                        const uint32_t n1 = (q4 & 255) | ((q5 & 255) << 8) | ((q6 & 255) << 16) | ((uint32_t)(q7 & 255) << 24);
                        *reinterpret_cast<uint2 *>(a.dbg.hq + (size_t)sm.ent[m] * kdim + 8 * gi) = make_uint2(n0, n1);
                    }
                }
                sum = warp_sum_i(sum);
                if (lane == 0) sm.hpart[warp][m] = sum;
            }
        }
        __syncthreads();
        if (KIND == kDown) {
            hsum = 0;
            if (lane < M)
#pragma unroll
                for (int w = 0; w < 8; ++w) hsum += sm.hpart[w][lane];
        }

        const int g_end = min(p1, (ue + 1) * gpe);  // groups of entry ue end here
        auto in_seg = [&](int jj) { return jj < n_my && p0 + warp + 8 * (jj / UPG) < g_end; };
        // the loops are compiled for MM token rows: 1, 2 or the batch's
        // widest entry, the smallest that holds this entry's M (an expert
        // that one or two tokens chose does not pay for the widest entry)
        auto process = [&](auto mm, const UnitRegs<KIND, CPL> &R, int jj) {
            constexpr int MM = decltype(mm)::value;
            const int p = p0 + warp + 8 * (jj / UPG);
            const int o0 = (p - ue * gpe) * RPG;
            if (KIND == kGateUp) {
                int acc[MM];
#pragma unroll
                for (int m = 0; m < MM; ++m) acc[m] = 0;
                dot_rows<CPL, MM>(acc, R.w[0], xs, kdim, M, nch, lane);
                const int mine = lane_sum<MM>(acc, M, lane);
                if (jj % UPG == 0) {
                    held_g = mine;
                    held_gs = R.s[0];
                } else if (lane < M) {
                    const int gi = held_g - 8 * sm.xsum[lane], ui = mine - 8 * sm.xsum[lane];
                    const float gf = __fmul_rn(__fmul_rn((float)gi, sm.sx[lane]), held_gs);
                    const float uf = __fmul_rn(__fmul_rn((float)ui, sm.sx[lane]), R.s[0]);
                    const float hv = __fmul_rn(silu_f(gf), uf);
                    a.h[(size_t)(r0 + lane) * a.I + o0] = hv;
                    if (a.dbg.gate_acc) a.dbg.gate_acc[(size_t)sm.ent[lane] * a.I + o0] = gi;
                    if (a.dbg.up_acc) a.dbg.up_acc[(size_t)sm.ent[lane] * a.I + o0] = ui;
                }
            } else {
#pragma unroll
                // the unit's RPG rows are consecutive outputs: at one token,
                // with 4 of them (16-byte aligned: o0 is a multiple of 4),
                // one 16-byte store (wider batches keep their registers)
                constexpr bool kY4 = MCH == 1 && RPG == 4;
                float yv[RPG];
#pragma unroll
                for (int rr = 0; rr < RPG; ++rr) {
                    int acc[MM];
#pragma unroll
                    for (int m = 0; m < MM; ++m) acc[m] = 0;
                    dot_rows<CPL, MM>(acc, R.w[rr], xs, kdim, M, nch, lane);
                    const int mine = lane_sum<MM>(acc, M, lane);
                    yv[rr] = 0.f;
                    if (lane < M) {
                        const int o = o0 + rr;
                        const int di = mine - 8 * hsum;
                        yv[rr] = __fmul_rn(__fmul_rn((float)di, sm.sx[lane]), R.s[rr]);
                        if (!kY4) a.part[(size_t)sm.ent[lane] * a.D + o] = yv[rr];
                        if (a.dbg.down_acc) a.dbg.down_acc[(size_t)sm.ent[lane] * a.D + o] = di;
                    }
                }
                if (kY4 && lane < M)
                    *reinterpret_cast<float4 *>(a.part + (size_t)sm.ent[lane] * a.D + o0) =
                        make_float4(yv[0], yv[RPG > 1 ? 1 : 0], yv[RPG > 2 ? 2 : 0], yv[RPG > 3 ? 3 : 0]);
            }
        };
        // X holds unit j, Y unit j + 1; each processed set is refilled with
        // the unit two ahead.  Returns true when the next unit is in Y.
        auto run = [&](auto mm, UnitRegs<KIND, CPL> &X, UnitRegs<KIND, CPL> &Y) -> bool {
            while (in_seg(j)) {
                process(mm, X, j);
                request<KIND, CPL>(X, a, uexp, gpe, p0, n_my, j + 2, ex_u, ex, tab);
                ++j;
                if (!in_seg(j)) return true;
                process(mm, Y, j);
                request<KIND, CPL>(Y, a, uexp, gpe, p0, n_my, j + 2, ex_u, ex, tab);
                ++j;
            }
            return false;
        };
        auto run_m = [&](UnitRegs<KIND, CPL> &X, UnitRegs<KIND, CPL> &Y) -> bool {
            using C1 = std::integral_constant<int, 1>;
            using C2 = std::integral_constant<int, MCH < 2 ? MCH : 2>;
            using CW = std::integral_constant<int, MCH>;
            if (MCH == 1 || M <= 1) return run(C1{}, X, Y);
            if (MCH == 2 || M <= 2) return run(C2{}, X, Y);
            return run(CW{}, X, Y);
        };
        flip = flip ? !run_m(B, A) : run_m(A, B);
    }
}

// Contiguous slices of the row groups of entries [0, n) (gpe groups each)
// weighted by cost.  The cost of a group of an entry chosen by M tokens is
// its measured time on this part in units of ~0.05 us (per-CTA phase traces
// of an 8-token verify batch, CTAs whose slice lies in one entry): the loops
// of one or two token rows cost about the weight stream (6, 7); wider loops
// (compiled for the batch's widest entry, see stream_phase) cost a base plus
// a per-token share, larger for the down rows (7 + 3 M) than for the
// gate/up pairs (6 + 2 M).  CTA b gets the groups whose cumulative cost
// falls in [b W / G, (b+1) W / G); every CTA evaluates the same monotone
// map, so the slices tile the groups exactly.
template <int KIND>
__device__ __forceinline__ long long group_cost(const int *ubeg, int u) {
    const int M = ubeg[u + 1] - ubeg[u];
    return M <= 1 ? 6 : M <= 2 ? 7 : KIND == kGateUp ? 6 + 2 * M : 7 + 3 * M;
}
// Each entry's first group also carries the cost of staging that entry's
// token rows (one round trip for the quantised tokens of a gate/up entry,
// about one per h row of a down entry): a CTA whose slice starts k entries
// pays k stagings more.
template <int KIND>
__device__ __forceinline__ long long entry_cost(const int *ubeg, int u) {
    const int M = ubeg[u + 1] - ubeg[u];
    return KIND == kGateUp ? 28 : 20 * M;
}
template <int KIND>
__device__ __forceinline__ int group_at_cost(const int *ubeg, int n, int gpe, long long c) {
    long long pre = 0;
    for (int u = 0; u < n; ++u) {
        const long long w = group_cost<KIND>(ubeg, u), ce = entry_cost<KIND>(ubeg, u), span = ce + (long long)gpe * w;
        if (c < pre + span) return u * gpe + (c - pre < ce ? 0 : (int)((c - pre - ce) / w));
        pre += span;
    }
    return n * gpe;
}
template <int KIND>
__device__ __forceinline__ void cost_slice(const int *ubeg, int n, int gpe, int b, int G, int &p0, int &p1) {
    long long W = 0;
    for (int u = 0; u < n; ++u) W += entry_cost<KIND>(ubeg, u) + (long long)gpe * group_cost<KIND>(ubeg, u);
    p0 = group_at_cost<KIND>(ubeg, n, gpe, (long long)b * W / G);
    p1 = group_at_cost<KIND>(ubeg, n, gpe, (long long)(b + 1) * W / G);
}

// The union tables of the batch from its T*K selections in sm.idx ((token,
// slot) order), built in shared memory by the whole CTA (T*K <= blockDim).
// Thread i ranks selection i by (expert, i): that rank is its row in the
// expert-grouped order (rows of one expert keep (token, slot) order).  The
// first selection of each expert also ranks its expert among the distinct
// ones: the union is in ascending expert id, the shared expert last.
// Selections that adaptive top-p dropped (kDroppedSel) take no row; the
// shared expert's rows follow the kept ones.  Returns the kept count.
__device__ __forceinline__ int build_union(DecodeSmem &sm, int T, int K, int S, int E, int n_shared) {
    const int n = T * K, tid = threadIdx.x;
    int e = -1, less = 0;
    bool first = false;
    if (tid == 0) sm.nu = 0;
    if (tid < n) {
        e = sm.idx[tid];
        if (e != kDroppedSel) {
            first = true;
            for (int j = 0; j < n; ++j) {
                const int ej = sm.idx[j];
                if (ej == kDroppedSel) continue;
                less += ej < e;
                if (ej == e && j < tid) {
                    ++less;
                    first = false;
                }
            }
            sm.rows[less] = (tid / K) * S + (tid % K);
        }
        sm.first[tid] = first;
    }
    const int n_kept = __syncthreads_count(tid < n && e != kDroppedSel);
    if (tid < n && first) {
        int upos = 0;
        for (int j = 0; j < n; ++j) upos += sm.first[j] && sm.idx[j] < e;
        sm.uexp[upos] = e;
        sm.ubeg[upos] = less;
        atomicAdd(&sm.nu, 1);
    }
    if (n_shared && tid < T) sm.rows[n_kept + tid] = tid * S + K;
    __syncthreads();
    if (tid == 0) {
        const int nr = sm.nu;
        sm.ubeg[nr] = n_kept;
        if (n_shared) {
            sm.uexp[nr] = E;
            sm.ubeg[nr + 1] = n_kept + T;
        }
    }
    __syncthreads();
    return n_kept;
}

template <int CPLG, int CPLD, int MCH>
__global__ void __launch_bounds__(256, 2) decode_layer_kernel(LayerArgs a) {
    extern __shared__ __align__(16) int8_t xs[];  // [MCH][max(D, I)] activation tile
    __shared__ DecodeSmem sm;
    const int tid = threadIdx.x;
    const int b = blockIdx.x, G = gridDim.x;
    const int T = a.T, D = a.D, I = a.I, E = a.E, K = a.K, S = a.S, n_sel = T * K;

    // one-entry view of the shared expert: grouped rows [n_sel, n_sel + T)
    if (tid < T) sm.rows[n_sel + tid] = tid * S + K;
    if (tid == 0) {
        sm.sh_uexp[0] = E;
        sm.sh_ubeg[0] = n_sel;
        sm.sh_ubeg[1] = n_sel + T;
    }
    __syncthreads();

    // Weights first: the router rows, then the first rows of the shared
    // expert, which need no routing.  They depend on nothing the previous
    // kernel in the stream writes, so they are requested before waiting for
    // it (launched with programmatic stream serialisation, this grid may
    // start while that one drains).
    WrRegs<CPLG, MCH == 1> wr;  // D <= 1024 * CPLG; at one token also token 0's activations
    if (b < E) logits_request_w(wr, a.Wr + (size_t)b * D, D);
    int ex_u = -1;
    DevExpert ex{};
    UnitRegs<kGateUp, CPLG> A, B;
    // (one token: the shared expert's gate/up streams here, within the
    // routing's latency; more tokens: it is compute bound in the wide dot
    // loops and would hold up the union, so it joins the routed entries'
    // cost-weighted slices instead)
    // (with adaptive top-p the shared rows follow the kept selections, whose
    // count the routing decides: the shared expert then joins the slices)
    const bool sh_early = MCH == 1 && a.n_shared && !(a.top_p > 0.f && a.top_p < 1.f);
    const int sp0 = sh_early ? (int)((long long)b * I / G) : 0;
    const int sp1 = sh_early ? (int)((long long)(b + 1) * I / G) : 0;
    // (a router CTA requests them once its logits are out, so that the router
    // rows have HBM to themselves at the start)
    if (b >= E) prime<kGateUp, CPLG>(A, B, a, sm.sh_uexp, I, sp0, sp1, ex_u, ex);
    // everything the previous kernel wrote (the activations, the decode
    // state) is read from here on
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) sm.epoch = ld_relaxed_u32(&a.dstate->epoch);
    __syncthreads();
    stamp(a, 0);
    // this launch's set of counters and hand-over buffers; the other set
    // (the previous launch's) is restored for the next launch, a share per CTA
    const int par = (int)(sm.epoch & 1u);
    FusedSync *sy = &a.dstate->set[par];
    float *const dlog = a.dlog + (size_t)par * kSmallT * E;
    unsigned long long *const dsel = a.dsel + (size_t)par * kSmallT * K;
    // one token with the hand-over buffer: the h rows, each value its own
    // flag, instead of a grid barrier after gate/up (null: the barrier)
    float *const hset = MCH == 1 && a.dh ? a.dh + (size_t)par * S * I : nullptr;
    // (then the CTA counts itself as having read the epoch; CTA 0 advances
    // it once all have)
    if (hset && tid == 0) atomicAdd(&sy->gu_cnt, 1);
    {
        FusedSync *so = &a.dstate->set[par ^ 1];
        float *const olog = a.dlog + (size_t)(par ^ 1) * kSmallT * E;
        unsigned long long *const osel = a.dsel + (size_t)(par ^ 1) * kSmallT * K;
        const int stride = G * blockDim.x;
        for (int i = b * blockDim.x + tid; i < kSmallT * E; i += stride) st_relaxed_u32(olog + i, kLogitEmpty);
        for (int i = b * blockDim.x + tid; i < kSmallT * K; i += stride) st_relaxed_u64(osel + i, kSelEmpty);
        for (int i = b * blockDim.x + tid; i < kMaxRedBlk; i += stride) so->blk[i] = 0;
        // (every launch, whatever its batch: the next launch may be a
        // one-token one, which polls that set's h values)
        if (a.dh) {
            float *const oh = a.dh + (size_t)(par ^ 1) * S * I;
            for (int i = b * blockDim.x + tid; i < S * I; i += stride) st_relaxed_u32(oh + i, kHEmpty);
        }
        if (b == 0 && tid == 0) {
            so->quant_cnt = 0;
            so->gu_cnt = 0;
        }
    }

    // ---- phase 1.  The router logits (everything downstream waits on
    // them); at one token every CTA also holds token 0's activations.
    if constexpr (MCH == 1) x0_request(wr, a.x, D);

    // router logits of experts b, b + G, ... (the arithmetic of the
    // four-kernel router), published as data: the slot itself is the flag
    if (b < E) {
        for (int e = b; e < E; e += G) {
            if (e != b) logits_request(wr, a.Wr + (size_t)e * D, a.x, D);
            const float l = logits_finish(wr, a.x, T, D, sm.red);
            if (tid < T) {
                const uint32_t bits = __float_as_uint(l);
                st_relaxed_u32(dlog + tid * E + e, bits == kLogitEmpty ? 0x7FFFFFFFu : bits);
            }
        }
        prime<kGateUp, CPLG>(A, B, a, sm.sh_uexp, I, sp0, sp1, ex_u, ex);
    }
    stamp(a, 1);

    // quantiser.  At one token every CTA quantises token 0 into its own tile
    // from the registers the router loads left (the last CTA also writes the
    // global row: the debug outputs).  Else the last T CTAs, one token each,
    // write the global rows the staged tiles are read from.
    const int tq = G - 1 - b;
    if constexpr (MCH == 1) {
        quant_x0_tile(wr, D, xs, &sm.sx[0], &sm.xsum[0], tq == 0 ? a.xq : nullptr, tq == 0 ? a.sx : nullptr,
                      tq == 0 ? a.xsum : nullptr, tq == 0 ? a.dbg.xq : nullptr);
    } else if (tq < T) {
        quant_token_perm(a.x + (size_t)tq * D, D, a.xq + (size_t)tq * D, a.sx + tq, a.xsum + tq,
                         a.dbg.xq ? a.dbg.xq + (size_t)tq * D : nullptr);
        cta_arrive(&sy->quant_cnt);
    }

    // top-K: CTA G-1-t selects token t's experts (topk_small_cta, the
    // routine of the four-kernel router) as soon as its logits are in, and
    // publishes them as data, while the other CTAs stream the shared expert
    if (tq < T)
        topk_small_cta<true>(dlog + (size_t)tq * E, a.bias, 1, E, K, a.routed_scale, nullptr, nullptr,
                             dsel + (size_t)tq * K, a.err, sm.tk, sm.tkp, a.top_p);

    // shared expert gate/up, once the quantised tokens are in
    if (MCH > 1) cta_wait(&sy->quant_cnt, T, a.err);
    stamp(a, 2);
    stream_phase<kGateUp, CPLG, MCH>(a, sm, xs, sm.sh_uexp, sm.sh_ubeg, sp0, sp1, A, B, ex_u, ex, hset);
    stamp(a, 3);

    // ---- phase 2: every CTA reads the published selections (bounded wait;
    // an entry still empty at the time-out becomes expert 0 with weight 0)
    // and builds the union itself
    {
        const unsigned long long t_begin = global_ns();
        for (;;) {
            bool miss = false;
            for (int i = tid; i < n_sel; i += blockDim.x) {
                const unsigned long long v = ld_relaxed_u64(dsel + i);
                const int e = (int)(v >> 32);
                miss |= v == kSelEmpty;
                sm.idx[i] = v == kSelEmpty ? 0 : e == kDroppedSel ? kDroppedSel : (e >= 0 && e < E) ? e : 0;
                sm.w[i] = v == kSelEmpty ? 0.f : __uint_as_float((uint32_t)v);
            }
            if (!__syncthreads_or(miss)) break;
            const bool late = tid == 0 && global_ns() - t_begin > kWaitNs;
            if (__syncthreads_or(late)) {
                if (tid == 0) atomicOr(a.err, kErrSyncTimeout);
                break;
            }
            __nanosleep(64);
        }
    }
    stamp(a, 4);
    const int n_kept = build_union(sm, T, K, S, E, a.n_shared);
    stamp(a, 5);
    const int n_r = sm.nu, n_u = n_r + a.n_shared;
    // one token: the union entries' expert pointers go to shared memory, so
    // that no warp's first request of an entry waits on a global load of them
    const DevExpert *const tab = MCH == 1 ? sm.uexd : nullptr;
    if (MCH == 1) {
        if (tid < n_u) sm.uexd[tid] = a.experts[sm.uexp[tid]];
        __syncthreads();
    }
    if (b == 0) {  // the tables for the debug entry point and other readers
        for (int i = tid; i < n_sel; i += blockDim.x) {
            a.idx[i] = sm.idx[i];
            a.wts[i] = sm.w[i];
        }
        for (int i = tid; i < n_kept + a.n_shared * T; i += blockDim.x) a.rows[i] = sm.rows[i];
        for (int i = tid; i < n_u; i += blockDim.x) a.meta->uexp[i] = sm.uexp[i];
        for (int i = tid; i <= n_u; i += blockDim.x) a.meta->ubeg[i] = sm.ubeg[i];
        if (tid == 0) {
            a.meta->n_union = n_u;
            a.meta->n_gu_items = n_u * a.nb_gu;
            a.meta->n_dn_items = n_u * a.nb_dn;
        }
    }

    // routed experts' gate/up (with the shared expert's for T > 1) and all
    // entries' down: contiguous slices of (entry, row group)
    constexpr int RPD = UnitShape<kDown, CPLD>::kRows;  // down rows per group
    const int gpd = D / RPD;
    int rp0, rp1, dp0, dp1;
    if (MCH == 1) {  // one token: every group costs the same, an even split
        // (the shared expert's gate/up ran in phase 1 unless adaptive top-p
        // moved it here)
        const long long Nr = (long long)(sh_early ? n_r : n_u) * I, Nd = (long long)n_u * gpd;
        rp0 = (int)(b * Nr / G);
        rp1 = (int)((b + 1) * Nr / G);
        if (G >= n_u) {
            // down: the CTAs split into one run per entry (entry u gets CTAs
            // [u G / n_u, (u+1) G / n_u)), so that no CTA stages the h of two
            // entries; each run splits its entry's groups evenly
            const int u = (int)(((long long)b * n_u + n_u - 1) / G);  // first u with (u+1) G / n_u > b
            const int c0 = (int)((long long)u * G / n_u), c1 = (int)((long long)(u + 1) * G / n_u);
            const int j = b - c0, c = c1 - c0;
            dp0 = u * gpd + (int)((long long)j * gpd / c);
            dp1 = u * gpd + (int)((long long)(j + 1) * gpd / c);
        } else {
            dp0 = (int)(b * Nd / G);
            dp1 = (int)((b + 1) * Nd / G);
        }
    } else {
        if (tid == 0) {
            cost_slice<kGateUp>(sm.ubeg, n_u, I, b, G, sm.slice[0], sm.slice[1]);
            cost_slice<kDown>(sm.ubeg, n_u, gpd, b, G, sm.slice[2], sm.slice[3]);
        }
        __syncthreads();
        rp0 = sm.slice[0];
        rp1 = sm.slice[1];
        dp0 = sm.slice[2];
        dp1 = sm.slice[3];
    }
    prime<kGateUp, CPLG>(A, B, a, sm.uexp, I, rp0, rp1, ex_u, ex, tab);
    stream_phase<kGateUp, CPLG, MCH>(a, sm, xs, sm.uexp, sm.ubeg, rp0, rp1, A, B, ex_u, ex, hset, tab);
    stamp(a, 6);

    // ---- phase 3.  More tokens: the CTA arrives, requests its first down
    // rows, then waits for every h row (arrival first: its fence would
    // otherwise wait for these loads too).  One token: no barrier; the CTA
    // requests its first down rows and its staging reads the entry's h rows
    // until every value is there.
    UnitRegs<kDown, CPLD> A2, B2;
    if (hset) {
        prime<kDown, CPLD>(A2, B2, a, sm.uexp, gpd, dp0, dp1, ex_u, ex, tab);
    } else {
        cta_arrive(&sy->gu_cnt);
        prime<kDown, CPLD>(A2, B2, a, sm.uexp, gpd, dp0, dp1, ex_u, ex);
        cta_wait(&sy->gu_cnt, G + a.wait_extra, a.err);
        // every CTA has read the epoch (before it arrived): advance it
        if (b == 0 && tid == 0) st_relaxed_u32(&a.dstate->epoch, sm.epoch + 1u);
    }
    stamp(a, 7);
    stream_phase<kDown, CPLD, MCH>(a, sm, xs, sm.uexp, sm.ubeg, dp0, dp1, A2, B2, ex_u, ex, hset, tab);
    stamp(a, 8);
    // the next kernel in the stream may launch once every CTA is here: its
    // prologue (weight requests) overlaps this grid's reduce and exit
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // rows written per reduce block; the CTA whose rows complete a block
    // (n_u entries x its rows) reduces it.  Thread 0 lists the (block, rows)
    // contributions of this CTA, and one thread per contribution arrives, so
    // the arrivals travel to L2 together.
    __syncthreads();
    if (tid == 0) {
        __threadfence();  // this CTA's partial rows are visible before any arrival
        int nc = 0;
        sm.nblk = 0;
        if (dp0 < dp1) {
            for (int u = dp0 / gpd; u <= (dp1 - 1) / gpd; ++u) {
                const int lo = RPD * (max(dp0, u * gpd) - u * gpd), hi = RPD * (min(dp1, (u + 1) * gpd) - u * gpd);
                for (int bb = lo / kRedRows; bb * kRedRows < hi; ++bb) {
                    const int b_lo = bb * kRedRows, b_hi = min(D, b_lo + kRedRows);
                    const int cnt = min(hi, b_hi) - max(lo, b_lo);
                    if (nc < kMaxContrib) {
                        sm.contrib[nc++] = make_int2(bb, cnt);
                    } else if (atomicAdd(&sy->blk[bb], cnt) + cnt == n_u * (b_hi - b_lo)) {
                        sm.blk_list[atomicAdd(&sm.nblk, 1)] = bb;  // beyond the list: arrive here
                    }
                }
            }
        }
        sm.ncontrib = nc;
    }
    __syncthreads();
    if (tid < sm.ncontrib) {
        const int bb = sm.contrib[tid].x, cnt = sm.contrib[tid].y;
        const int rows = min(D, (bb + 1) * kRedRows) - bb * kRedRows;
        if (atomicAdd(&sy->blk[bb], cnt) + cnt == n_u * rows) {
            __threadfence();  // every other contribution to the block is visible from here on
            sm.blk_list[atomicAdd(&sm.nblk, 1)] = bb;
        }
    }
    if (tid == 0) __threadfence();
    __syncthreads();
    // reduce the completed blocks: one (block, token, 4 rows) task per
    // thread, every slot loaded before the ordered sum
    {
        const int n4 = kRedRows / 4, nt = sm.nblk * T * n4;
        for (int q = tid; q < nt; q += blockDim.x) {
            const int blk = q / (T * n4), rem = q - blk * T * n4, t = rem / n4;
            const int o = sm.blk_list[blk] * kRedRows + 4 * (rem - t * n4);
            if (o >= D) continue;
            const float *pt = a.part + (size_t)t * S * D + o;
            float4 y[kMaxK + 1];
#pragma unroll
            for (int k = 0; k <= kMaxK; ++k)
                if (k < S) y[k] = ld_cg_f4(pt + (size_t)k * D);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kMaxK; ++k) {
                if (k < K && sm.idx[t * K + k] != kDroppedSel) {  // a dropped slot has no expert output
                    const float wk = sm.w[t * K + k];
                    acc.x = __fadd_rn(acc.x, __fmul_rn(wk, y[k].x));
                    acc.y = __fadd_rn(acc.y, __fmul_rn(wk, y[k].y));
                    acc.z = __fadd_rn(acc.z, __fmul_rn(wk, y[k].z));
                    acc.w = __fadd_rn(acc.w, __fmul_rn(wk, y[k].w));
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
                const float4 r = *reinterpret_cast<const float4 *>(a.resid + (size_t)t * D + o);
                acc.x = __fadd_rn(r.x, acc.x);
                acc.y = __fadd_rn(r.y, acc.y);
                acc.z = __fadd_rn(r.z, acc.z);
                acc.w = __fadd_rn(r.w, acc.w);
            }
            *reinterpret_cast<float4 *>(a.out + (size_t)t * D + o) = acc;
        }
    }

    // one token: every CTA has read the epoch (each counted itself after
    // reading it) before CTA 0 advances it (bounded; the test hook's extra
    // arrival makes this wait run out)
    if (hset && b == 0 && tid == 0) {
        const int target = G + a.wait_extra;
        if (ld_acquire(&sy->gu_cnt) < target) {
            const unsigned long long t0 = global_ns();
            while (ld_acquire(&sy->gu_cnt) < target) {
                if (global_ns() - t0 > kWaitNs) {
                    atomicOr(a.err, kErrSyncTimeout);
                    break;
                }
                __nanosleep(64);
            }
        }
        st_relaxed_u32(&a.dstate->epoch, sm.epoch + 1u);
    }

    stamp(a, 9);
}

using DecodeFn = void (*)(LayerArgs);

// The kernel for T tokens at chunk counts (CPLG, CPLD): instantiated by one
// translation unit per (CPLG, CPLD) pair so they compile in parallel.
template <int CPLG, int CPLD>
DecodeFn pick_m(int T) {
    if (T <= 1) return decode_layer_kernel<CPLG, CPLD, 1>;
    if (T <= 2) return decode_layer_kernel<CPLG, CPLD, 2>;
    if (T <= 4) return decode_layer_kernel<CPLG, CPLD, 4>;
    if (T <= 8) return decode_layer_kernel<CPLG, CPLD, 8>;
    return decode_layer_kernel<CPLG, CPLD, 16>;
}

}  // namespace dec

// One per instantiated pair (k_decode_c*.cu).
dec::DecodeFn decode_pick_c11(int T);
dec::DecodeFn decode_pick_c21(int T);
dec::DecodeFn decode_pick_c42(int T);
dec::DecodeFn decode_pick_c62(int T);

}  // namespace moe
