// layer_args.cuh -- kernel argument block shared by the layer kernels and the
// host launch code.  Internal.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {

struct LayerArgs {
    int D, I, E, K, S, n_shared, T;
    float routed_scale;
    float top_p;         // adaptive expert top-p in (0, 1); other values: plain top-K
    int wbits;           // expert weight width: 4 (packed int4 rows) or 8 (int8 rows)
    const float *x;      // [T, D] fp32 layer input (post-norm activations)
    const float *Wr;     // [E, D]
    const float *bias;   // [E]
    const DevExpert *experts;  // [E + n_shared]
    int8_t *xq;          // [Tmax, D] int8, even/odd permuted 8-groups
    float *sx;           // [Tmax]
    int32_t *xsum;       // [Tmax] sum of xq over the row
    float *logits;       // [router_splits(Tmax), max(kSmallT, Tmax), E] (partials of the large-batch router)
    int32_t *idx;        // [Tmax, K]
    float *wts;          // [Tmax, K]
    int32_t *rows;       // [Tmax * S] entry ids (t*S + slot) grouped by union expert
    RouteMeta *meta;
    float *h;            // [Tmax * S, I] fp32 SwiGLU output, by grouped row
    uint32_t *hamax;     // [Tmax * S] bits of max|h| per grouped row
    float *part;         // [Tmax * S, D] expert outputs y by entry id
    int8_t *hq;          // [Tmax * S, I] requantised h (even/odd layout), by grouped row
    uint16_t *xf;        // [Tmax * S, max(D, I)] f16 activation operand rows of the tcgen05 GEMMs, by grouped row
                         // (gate/up: the token's codes, D per row; down: the requantised h, I per row), or null
    int32_t *hsum;       // [Tmax * S] code sums of hq rows
    float *shq;          // [Tmax * S] scales of hq rows
    int32_t *dn_cnt;     // [nb_dn] arrival counters of the fused reduce
    DecodeState *dstate;  // counters of the persistent decode kernel (two sets)
    // hand-over buffers of the persistent decode kernel, one per set of
    // counters; a set is empty (logits / selections) when its launch starts
    float *dlog;                 // [2][kSmallT, E] logits, kLogitEmpty until written
    unsigned long long *dsel;    // [2][kSmallT, K] packed selections, kSelEmpty until written
    float *dh;                   // [2][S, I] h rows of a one-token launch, kHEmpty until written
    unsigned long long *trace;  // [trace_n] phase stamps of that kernel, or null
    int trace_n;
    float *out;          // [T, D]
    const float *resid;  // [T, D] or null: out = resid + MoE
    int32_t *err;
    int nb_gu, rpi_gu;   // gate/up: row blocks per expert, rows per block
    int nb_dn, rpi_dn;   // down: row blocks per expert, rows per block
    int wait_extra;      // test hook: arrivals the decode kernel's grid barrier waits for beyond G
    const CUtensorMap *wmaps;  // [3 (E + n_shared)] TMA maps of the packed gate, up, down rows, or null
    DebugPtrs dbg;
};

// Host launchers (defined in the .cu files).
cudaError_t launch_router_small(const LayerArgs &a, cudaStream_t s);
cudaError_t launch_quant_perm(const LayerArgs &a, cudaStream_t s);
cudaError_t launch_router_tile(const float *x, const float *Wr, const float *bias, int T, int D,
                               int E, int K, float scale, int32_t *idx, float *w, int32_t *err,
                               cudaStream_t s);
cudaError_t launch_permute(const LayerArgs &a, cudaStream_t s);
// Large-batch router through a logits buffer [T, E]: tiled fp32 GEMM, then
// one warp per token for the top-K.
cudaError_t launch_router_gemm(const float *x, const float *Wr, const float *bias, int T, int D, int E, int K,
                               float scale, float top_p, float *logits, int32_t *idx, float *w, int32_t *err,
                               cudaStream_t s);
cudaError_t launch_gateup(const LayerArgs &a, int mch, int grid, cudaStream_t s);
cudaError_t launch_down(const LayerArgs &a, int mch, int grid, bool fused_reduce, cudaStream_t s);
cudaError_t launch_reduce(const LayerArgs &a, cudaStream_t s);
cudaError_t launch_rmsnorm(const float *x, const float *w, float eps, float *out, int T, int D,
                           cudaStream_t s);
cudaError_t launch_quant_natural(const float *x, int8_t *xq, float *sx, int T, int D,
                                 cudaStream_t s);
cudaError_t launch_pack_int4(const float *w, uint8_t *q4, float *scale, int64_t O, int64_t I,
                             cudaStream_t s);
cudaError_t launch_pack_int8(const float *w, int8_t *q8, float *scale, int64_t O, int64_t I, cudaStream_t s);
// int8-weight experts (row-per-warp kernels; the layer's only path for them)
cudaError_t launch_gateup8(const LayerArgs &a, int mch, int grid, cudaStream_t s);
cudaError_t launch_down8(const LayerArgs &a, int mch, int grid, bool fused, cudaStream_t s);
cudaError_t prepare_expert_kernels8(int D, int I, int num_sms, int grid_gu[4], int grid_dn[4]);
// FP8 E4M3 matrix with 128 x 128 block scales -> packed int4 + row scales.
cudaError_t launch_fp8_to_int4(const uint8_t *w8, const float *scale_inv, uint8_t *q4, float *scale, int64_t O,
                               int64_t I, cudaStream_t s);
cudaError_t launch_gateup_stream(const LayerArgs &a, int grid, cudaStream_t s);
cudaError_t launch_down_stream(const LayerArgs &a, int grid, cudaStream_t s);
bool stream_supported(int D, int I);
// Persistent single-kernel layer for T <= kSmallT (cooperative launch).
// decode_grid: CTAs of the launch for this T (0 if the kernel cannot run).
cudaError_t decode_grid(const LayerArgs &a, int num_sms, int *grid);
cudaError_t launch_decode_layer(const LayerArgs &a, int grid, cudaStream_t s);
cudaError_t launch_grouped_gateup(const LayerArgs &a, int num_sms, cudaStream_t s);
cudaError_t launch_requant_h(const LayerArgs &a, cudaStream_t s);
cudaError_t launch_grouped_down(const LayerArgs &a, int num_sms, cudaStream_t s);
bool grouped_supported(int D, int I);
// Tensor-core (tcgen05, f16-exact) expert GEMMs of large batches.  Their
// activation operand is the f16 row buffer xf, read through TMA tensor maps
// (gate/up: rows of D columns; down: rows of I columns), encoded once per
// workspace.
struct UmmaMaps {
    CUtensorMap gu, dn;
};
bool umma_supported(int D, int I);
cudaError_t umma_encode_maps(void *xf, int rows, int D, int I, UmmaMaps *maps);
// Host: the weight maps of an expert table (host copy of the device table).
cudaError_t umma_encode_weight_maps(const DevExpert *tab, int ne, int D, int I, CUtensorMap *maps);
cudaError_t launch_act_rows_f16(const LayerArgs &a, cudaStream_t s);
cudaError_t launch_umma_gateup(const LayerArgs &a, const UmmaMaps &maps, int num_sms, cudaStream_t s);
cudaError_t launch_umma_down(const LayerArgs &a, const UmmaMaps &maps, int num_sms, cudaStream_t s);
// Occupancy-derived grid sizes and kernel attributes (call once per device).
cudaError_t prepare_expert_kernels(int D, int I, int num_sms, int grid_gu[4], int grid_dn[4]);
int mch_index(int mch);

}  // namespace moe
