// common.cuh -- shared device helpers and internal structures of the
// routed-MoE layer library (sm_103a).  Internal: not part of the C ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/moe_int4.h"

namespace moe {

constexpr int kMaxE = 512;        // routed experts per layer
constexpr int kMaxK = 16;         // experts per token
constexpr int kSmallT = 16;       // token count served by the fused small-batch router
constexpr int kMaxDim = 8192;     // D and I upper bound (GEMV chunks per lane <= 8)
constexpr int kRouterSplitK = 9;  // partial logit buffers of the large-batch router (K split), at most
// K ranges of the large-batch router at T tokens: 9 from 128 tokens on (the
// 128 x 128 tiles alone would leave most SMs idle), else 4 (which keeps the
// partial buffers of a small batch small)
inline constexpr int router_splits(long long T) { return T >= 128 ? kRouterSplitK : 4; }

// Device error word bits (moe_layer_device_status).
constexpr int kErrNoSelection = 1;   // a token had no finite selection score left
constexpr int kErrRouteCount = 2;    // routing table inconsistent
constexpr int kErrTooManyRows = 8;   // an expert had more rows than the streaming tile
constexpr int kErrSyncTimeout = 16;  // a wait of the persistent decode kernel ran out of time

// Expert id of a selection that adaptive top-p dropped (no expert: its slot
// is skipped by the union and the weighted sum).
constexpr int kDroppedSel = -1;

struct DevExpert {
    const uint8_t *gq, *uq, *dq;
    const float *gs, *us, *ds;
};

// Routing tables built on the device for one forward.  Union entry u covers
// rows [ubeg[u], ubeg[u+1]) of `rows`; the shared expert (if any) is the last
// entry with id E.
struct RouteMeta {
    int n_union;
    int n_gu_items;
    int n_dn_items;
    int counter;  // last-CTA counter of the small-batch router (reset by that CTA)
    int uexp[kMaxE + 1];
    int ubeg[kMaxE + 2];
};

// Arrival counters of the persistent decode kernel.  There are two sets, and
// with them two sets of its hand-over buffers: launch n uses set n % 2 (the
// parity of `epoch`, which CTA 0 advances once every CTA has read it) and
// restores set (n + 1) % 2, which launch n - 1 used, for launch n + 1.  So no
// CTA has to wait at the end of a launch for all others to finish before
// the state can be cleared.
constexpr int kRedRows = 64;                    // output rows per reduce block
constexpr int kMaxRedBlk = kMaxDim / kRedRows;  // reduce blocks of the largest D
struct FusedSync {
    int quant_cnt;         // quantiser CTAs finished
    int gu_cnt;            // CTAs finished with gate/up
    int blk[kMaxRedBlk];   // down rows written per reduce block
};
struct DecodeState {
    unsigned int epoch;    // launches so far (its parity selects the set)
    FusedSync set[2];
};

// Phase time stamps of the persistent decode kernel (moe_layer_set_trace):
// per CTA, %globaltimer at kernel start, after the router/quantiser roles,
// after the quantiser wait, after the shared expert's gate/up, after the
// router wait, after top-K + union, after the routed gate/up, after the
// gate/up barrier, after the down rows, at the end.
constexpr int kTraceStamps = 10;

struct DebugPtrs {
    int8_t *xq;
    int32_t *gate_acc, *up_acc;
    int8_t *hq;
    float *sh;
    int32_t *down_acc;
};

// ------------------------------------------------------------------ helpers

// Sentinels of the decode kernel's data-as-flag hand-overs: a logit slot or a
// packed selection that has not been written yet.  0xFFFFFFFF is a NaN that
// arithmetic never produces (it yields the canonical 0x7FFFFFFF).
constexpr uint32_t kLogitEmpty = 0xFFFFFFFFu;
constexpr unsigned long long kSelEmpty = 0xFFFFFFFFFFFFFFFFull;
constexpr uint32_t kHEmpty = 0xFFFFFFFFu;  // an h value not yet written (one-token decode launches)
constexpr unsigned long long kWaitNs = 1000000000ull;  // bound of every wait: 1 s

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Coherent (L2) loads and stores for values other CTAs of the same grid poll.
__device__ __forceinline__ uint32_t ld_relaxed_u32(const void *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const void *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint4 ld_relaxed_v4(const void *p) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u32(void *p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_u64(void *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Block-wide max of non-negative floats; every thread gets the result.
// `red` must hold blockDim.x/32 floats.
__device__ __forceinline__ float block_max_nonneg(float v, float *red) {
    v = warp_max_f(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = lane < nw ? red[lane] : 0.f;
    r = warp_max_f(r);
    return r;
}

__device__ __forceinline__ int block_sum_i(int v, int *red) {
    v = warp_sum_i(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    int r = lane < nw ? red[lane] : 0;
    r = warp_sum_i(r);
    return r;
}

// Streaming 16-byte load of read-once weights: no L1 allocation.
__device__ __forceinline__ int4 ld_stream16(const void *p) {
    int4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16-byte load through L2 only (data written earlier in the same grid by other CTAs).
__device__ __forceinline__ float4 ld_cg_f4(const float *p) { return __ldcg(reinterpret_cast<const float4 *>(p)); }

// Per-row int8 quantisation scale: s = max(amax/127, 1e-12), inv = 1/s, both
// IEEE-rounded (reader.mx article §12, qrow_i8).
__device__ __forceinline__ void act_scale(float amax, float &s, float &inv) {
    s = __fdiv_rn(amax, 127.f);
    if (s < 1e-12f) s = 1e-12f;
    inv = __fdiv_rn(1.f, s);
}

__device__ __forceinline__ int quant_i8(float v, float inv) { return __float2int_rn(__fmul_rn(v, inv)); }

// Byte position of element i (0..7) of an 8-group in the even/odd lane
// layout used by the int4 GEMV kernels: [x0 x2 x4 x6 | x1 x3 x5 x7].  With
// that layout the low nibbles of a packed weight word (elements 0,2,4,6) meet
// the first activation word and the high nibbles the second.
__device__ __forceinline__ int perm8(int i) { return (i & 1) ? 4 + (i >> 1) : (i >> 1); }

// Sum over the 8 nibble-offset products of one packed weight word against the
// permuted activations: returns acc + sum_i nibble_i * x_i (nibbles unsigned,
// 0..15); the caller subtracts 8 * sum(x) once per row.
__device__ __forceinline__ int dot_word(uint32_t w, int xe, int xo, int acc) {
    const int lo = static_cast<int>(w & 0x0F0F0F0Fu);
    const int hi = static_cast<int>((w >> 4) & 0x0F0F0F0Fu);
    acc = __dp4a(lo, xe, acc);
    acc = __dp4a(hi, xo, acc);
    return acc;
}

// Shared-memory activations: row m holds the even/odd int8 row split in two
// planes, plane A = the first 16 bytes of every 32-byte chunk (activation
// groups 4c, 4c+1), plane B = the last 16 (groups 4c+2, 4c+3), so that the
// 16-byte reads of a warp are contiguous (no bank conflicts).
__device__ __forceinline__ int8_t *plane_byte(int8_t *xs, int kdim, int m, int byte) {
    const int ch = byte >> 5, in = byte & 31;
    return xs + (size_t)m * kdim + (in >= 16 ? (kdim >> 1) : 0) + ch * 16 + (in & 15);
}

__device__ __forceinline__ float silu_f(float g) { return __fdiv_rn(g, __fadd_rn(1.f, expf(-g))); }

}  // namespace moe
