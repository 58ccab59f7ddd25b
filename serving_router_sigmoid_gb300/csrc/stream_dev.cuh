// stream_dev.cuh -- device building blocks of the HBM-streaming expert
// GEMVs (decode-sized batches): register units of packed int4 rows, the
// two-plane shared-memory activation layout and the offset-nibble dp4a dot.
// Internal.
//
// Sources: reader.mx "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型" §12 (int8
// activations x int4 weights, exact integer dot, scales applied after);
// besthub.dev "Running 744B MoE on 25GB RAM" §12.
#pragma once

#include "layer_args.cuh"

namespace moe {

enum Kind { kGateUp = 0, kDown = 1 };

// A unit is what one warp multiplies between two pipeline steps: one packed
// row (gate or up) for gate/up; for down, as many rows as keep about 2 KB per
// unit in flight (4 rows of up to 1 KB, 2 of up to 2 KB, else 1).  A warp
// keeps one unit in flight while it multiplies another, so the unit size sets
// the bytes in flight.
template <int KIND, int CPL>
struct UnitShape {
    static constexpr int kRows = KIND == kGateUp ? 1 : (CPL <= 2 ? 4 : CPL <= 4 ? 2 : 1);
};

template <int KIND, int CPL>
struct UnitRegs {
    int4 w[UnitShape<KIND, CPL>::kRows][CPL];
    float s[UnitShape<KIND, CPL>::kRows];
};

template <int KIND, int CPL>
__device__ __forceinline__ void load_unit(UnitRegs<KIND, CPL> &r, const uint8_t *mat, const float *scale, int o,
                                          int rowb, int nch, int lane) {
#pragma unroll
    for (int rr = 0; rr < UnitShape<KIND, CPL>::kRows; ++rr) {
        const uint8_t *row = mat + (size_t)(o + rr) * rowb;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int ch = lane + 32 * c;
            if (ch < nch) r.w[rr][c] = ld_stream16(row + (size_t)ch * 16);
        }
        r.s[rr] = __ldg(scale + o + rr);
    }
}

// acc[m] += dot(row, x_m) over this lane's chunks (offset nibbles, even/odd x).
template <int CPL, int MCH>
__device__ __forceinline__ void dot_rows(int (&acc)[MCH], const int4 (&w)[CPL], const int8_t *xs, int kdim, int M,
                                         int nch, int lane) {
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int ch = lane + 32 * c;
        if (ch < nch) {
#pragma unroll
            for (int m = 0; m < MCH; ++m) {
                if (m < M) {
                    const int4 *pa = reinterpret_cast<const int4 *>(xs + (size_t)m * kdim);
                    const int4 x0 = pa[ch], x1 = pa[(kdim >> 5) + ch];
                    int v = acc[m];
                    v = dot_word((uint32_t)w[c].x, x0.x, x0.y, v);
                    v = dot_word((uint32_t)w[c].y, x0.z, x0.w, v);
                    v = dot_word((uint32_t)w[c].z, x1.x, x1.y, v);
                    v = dot_word((uint32_t)w[c].w, x1.z, x1.w, v);
                    acc[m] = v;
                }
            }
        }
    }
}

// Warp sums of acc[0..M); lane m receives the sum of token row m.
template <int MCH>
__device__ __forceinline__ int lane_sum(const int (&acc)[MCH], int M, int lane) {
    int mine = 0;
#pragma unroll
    for (int m = 0; m < MCH; ++m) {
        if (m < M) {
            const int v = warp_sum_i(acc[m]);
            if (lane == m) mine = v;
        }
    }
    return mine;
}

}  // namespace moe
