// k_umma.cu -- the expert GEMMs of large batches (prefill) on the fifth-
// generation tensor cores: tcgen05.mma kind::f16 with the int4 weights and
// int8 activations carried exactly as f16 and fp32 accumulators in TMEM.
//
// Sources: reader.mx "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型" §11 (each union
// expert's SwiGLU over the tokens routed to it: h = siluf(gate)*up, then
// down) and §12 (int8 activations x int4 weights, an exact integer dot, then
// the activation and row scales); besthub.dev "Running 744B MoE on 25GB RAM"
// §11, §12.
//
// Exactness.  sm_103a has no int8 kind of tcgen05.mma.  The weights are the
// integers n - 8 in [-8, 7] and the activations integers in [-127, 127], all
// exact in f16; every product is an integer of magnitude <= 1016 and every
// partial sum of a row stays below 6144 * 1016 < 2^24, so fp32 accumulation
// of these products is exact and the accumulator equals the int32 dot.
//
// Design (GB300).  D[weight rows x tokens] = W[rows x K] . X[tokens x K]^T:
// the weight rows are the MMA's M side (128 per tile) and the tokens of one
// union entry its N side (up to 128 per tile, padded to 16), so small experts
// waste at most 15 token columns.  For gate/up the 128 rows are 64 gate rows
// interleaved with the same 64 up rows, so one lane shuffle pairs g and u in
// the epilogue.  K runs in stages of 64.
//  - The activation operand is not converted here: a small kernel before the
//    GEMM writes every grouped row of the batch (gate/up: the token's int8
//    codes; down: the requantised h codes) as f16 integers, once, and one
//    producer thread moves each stage's token tile into shared memory with
//    TMA tile loads (boxes of 32 rows x 64 f16 = 128 bytes per row, 128-byte
//    swizzle: the K-major layout the MMA reads).  Rows past the tile's tokens
//    belong to the next entry (or lie past the tensor and read as zeros):
//    their accumulator columns are computed and ignored.
//  - One CTA per SM, 26 warps: 4 epilogue warps (TMEM lanes 0..127), two
//    groups of 8 converter warps (even and odd stages), 1 MMA warp, 4 weight
//    load warps, 1 activation TMA warp.
//  - The load warps copy the weight rows of 4 stages at a time into a
//    4-slot raw ring with 16-byte cp.async (32 rows per warp, 8 lanes per
//    128-byte row, so every warp instruction is fully coalesced); each
//    lane's copies arrive on the slot's barrier when they land.  Converter
//    thread c of a group owns one fixed 16-byte chunk of each of its stages,
//    expands it to f16 (a byte permute into 0x64xx patterns and one f16x2
//    subtraction per pair) and stores it into TMEM (the MMA's A operand); its
//    warp then arrives on the stage's barrier.  The packed weight nibbles come
//    out in the order e0 e2 e4 e6 e1 e3 e5 e7 of each 8-group, which is
//    exactly the even/odd order in which the activation rows are stored, so
//    both operands see the same permutation of K.
//  - The MMA thread waits for a stage's weights (converter barrier) and its
//    token tile (TMA transaction barrier), issues four K=16 MMAs and commits
//    them to the stage's "empty" barrier; after a tile's last stage to an
//    accumulator barrier.  Two 128-column TMEM accumulators let the epilogue
//    of one tile overlap the MMAs of the next.
//  - Epilogue: tcgen05.ld 32 columns at a time; gate/up: h = silu(g)*u, max|h|
//    per token row; down: y = (acc*sh)*sd into the per-slot partial rows.
// Every barrier wait is bounded (one second of %globaltimer); a time-out sets
// kErrSyncTimeout and an abort flag every role polls, the MMA thread drains
// its outstanding MMAs (bounded), the copy issuers wait (bounded) for their
// copies in flight, and the TMEM is freed before the CTA exits.
#include <cuda.h>
#include <cuda_fp16.h>

#include "layer_args.cuh"

namespace moe {

namespace {

constexpr int kGU = 0, kDN = 1;
constexpr int kThreads = 832;             // 26 warps
constexpr int kConv0 = 128;               // first converter thread: two groups of 8 warps
constexpr int kMmaWarp = 20;
constexpr int kLoadWarp0 = 21;            // four weight load warps
constexpr int kLoadWarps = 4;
constexpr int kTmaWarp = 25;              // activation tiles
constexpr int kBKs = 64;                  // K elements per stage
constexpr int kTok = 128;                 // token columns per tile at most
constexpr int kBoxRows = 32;              // token rows per TMA box
constexpr int kSt = 6;                    // operand stages (weights in TMEM, activations in shared memory)
constexpr int kRA = 4;                    // weight raw ring: slots of up to 4 stages (128 bytes per row)
constexpr uint32_t kBF16 = kTok * 128;    // 128 tokens x 64 f16
constexpr uint32_t kARowPitch = 144;      // raw weight row pitch: 128 bytes + 16 of padding
// raw weight row r sits at r * pitch (+64 for the second 64-row half), so the
// 16-byte reads of 8 consecutive tile rows fall in 8 different bank groups
__device__ __forceinline__ uint32_t raw_row_off(int r) { return (uint32_t)r * kARowPitch + (r >= 64 ? 64u : 0u); }
constexpr uint32_t kARaw = 128 * kARowPitch + 64;  // 128 rows x up to 4 stages of 64 int4
constexpr uint32_t kOffB = 0;
constexpr uint32_t kOffRA = kOffB + kSt * kBF16;
constexpr uint32_t kDyn = kOffRA + kRA * kARaw;  // 170 KB
constexpr size_t kSmemBytes = kDyn + 1024;       // + alignment to 1024 bytes
constexpr uint32_t kTmemCols = 512;       // accumulators [0, 256), weight stages [256, 256 + 32 kSt)
constexpr uint32_t kTmemA = 2 * kTok;     // first weight-stage column
constexpr uint32_t kAcolStage = 32;       // columns per weight stage: 64 f16 as 32 pairs
static_assert(kTmemA + kSt * kAcolStage <= kTmemCols, "TMEM columns");

struct UmmaSmem {
    uint64_t full[kSt], bfull[kSt], empty[kSt], acc_full[2], acc_empty[2], drain;
    uint64_t raw_full[kRA], raw_empty[kRA];
    uint32_t tmem;
    int abort;
    int tp[kMaxE + 2];        // tiles before each union entry
    int tok_r[2][kTok];       // per accumulator: grouped row of each token column
    int tok_e[2][kTok];       //   its entry id (token * S + slot)
    float tok_s[2][kTok];     //   its activation scale
    float red[4][kTok];       // max|h| per token column, per epilogue warp
};

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mb_init(uint64_t *b, int n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n));
}
__device__ __forceinline__ void mb_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mb_try(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// The same test with a suspend-time hint: a thread whose phase is not yet
// complete sleeps in the barrier unit (up to about 0.1 ms) instead of spinning.
__device__ __forceinline__ bool mb_try_sleep(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity), "r"(100000u)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase with this parity; false on abort or time-out.
__device__ __forceinline__ bool mb_wait(uint64_t *b, uint32_t parity, volatile int *abort, int32_t *err) {
    if (mb_try(b, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mb_try_sleep(b, parity)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > kWaitNs) {
            *abort = 1;
            atomicOr(err, kErrSyncTimeout);
            return false;
        }
    }
}

// Named barrier 1 over the 128 epilogue threads; returns the OR of p over
// them, so a decision to leave the loop is the same in every thread.
__device__ __forceinline__ bool epi_bar_or(bool p) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.or.pred po, 1, 128, pi;\n selp.u32 %0, 1, 0, po;\n}"
        : "=r"(r)
        : "r"((uint32_t)p)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void mb_expect_tx(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
// The barrier receives one arrival once every cp.async this thread issued
// before has landed (noinc: the arrival counts toward the initial count).
__device__ __forceinline__ void cp_async_arrive(uint64_t *b) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(su32(b)) : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// tcgen05 shared-memory descriptor: K-major, 128-byte swizzle, 8-row atoms
// 1024 bytes apart; the atom base is 1024-byte aligned and the start address
// steps 32 bytes per K=16 slice inside the 128-byte rows.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor of kind::f16: f16 A and B, K-major, fp32 D, M = 128.
__device__ __forceinline__ uint32_t idesc_f16(int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// One packed int4 word (8 weights of an 8-group) -> 16 bytes of f16 (n - 8)
// in the order e0 e2 e4 e6 e1 e3 e5 e7.
__device__ __forceinline__ uint4 w4_to_f16(uint32_t w) {
    const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu, m = 0x64646464u, k = 0x64086408u;
    return make_uint4(hsub2(__byte_perm(lo, m, 0x4140), k), hsub2(__byte_perm(lo, m, 0x4342), k),
                      hsub2(__byte_perm(hi, m, 0x4140), k), hsub2(__byte_perm(hi, m, 0x4342), k));
}
// TMA tile load of a 2D f16 tensor (box of the map) into shared memory,
// completing on the barrier's transaction count.  c0 = element column (a
// multiple of 64 here: 128-byte aligned), c1 = row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(su32(bar))
        : "memory");
}

struct Tile {
    int u, wb, r0, nvalid, npad;
};

__device__ __forceinline__ Tile tile_of(const LayerArgs &a, const UmmaSmem &sm, int nu, int nwb, int t) {
    int lo = 0, hi = nu - 1;
    while (lo < hi) {  // last entry with tp[u] <= t
        const int mid = (lo + hi + 1) >> 1;
        if (sm.tp[mid] <= t) lo = mid; else hi = mid - 1;
    }
    Tile x;
    x.u = lo;
    const int beg = a.meta->ubeg[lo], M = a.meta->ubeg[lo + 1] - beg;
    const int ntb = (M + kTok - 1) / kTok, local = t - sm.tp[lo];
    x.wb = local / ntb;
    const int tb = local - x.wb * ntb;
    x.r0 = beg + tb * kTok;
    x.nvalid = min(kTok, M - tb * kTok);
    x.npad = (x.nvalid + 15) & ~15;
    return x;
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1) umma_gemm_kernel(const __grid_constant__ CUtensorMap xmap, LayerArgs a) {
    extern __shared__ uint8_t dyn_raw[];
    __shared__ UmmaSmem sm;
    uint8_t *dyn = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = su32(dyn);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x, G = gridDim.x, S = a.S;
    const int kdim = KIND == kGU ? a.D : a.I;
    const int rowb = kdim >> 1;
    const int nwb = KIND == kGU ? a.I / 64 : a.D / 128;  // weight blocks per expert
    const int kst = kdim / kBKs;                          // stages per tile
    const int ch = kst % 4 == 0 ? 4 : kst % 2 == 0 ? 2 : 1;  // stages per weight copy (slot of the raw ring)
    const int nu = a.meta->n_union;
    volatile int *abort = &sm.abort;

    if (tid == 0) {
        int run = 0;
        for (int u = 0; u < nu; ++u) {
            sm.tp[u] = run;
            run += nwb * ((a.meta->ubeg[u + 1] - a.meta->ubeg[u] + kTok - 1) / kTok);
        }
        sm.tp[nu] = run;
        sm.abort = 0;
        for (int s = 0; s < kSt; ++s) {
            mb_init(&sm.full[s], 8);   // the 8 converter warps of the stage's group
            mb_init(&sm.bfull[s], 1);  // the TMA issuer's arrival, plus the tile's bytes
            mb_init(&sm.empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mb_init(&sm.acc_full[s], 1);
            mb_init(&sm.acc_empty[s], 4);
        }
        mb_init(&sm.drain, 1);
        for (int s = 0; s < kRA; ++s) {
            mb_init(&sm.raw_full[s], 32 * kLoadWarps);
            mb_init(&sm.raw_empty[s], ch == 1 ? 8 : 16);  // the warps of every group that converts from the slot
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&sm.tmem)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = sm.tmem;
    const int n_tiles = sm.tp[nu];
    const int n_my = b < n_tiles ? (n_tiles - b + G - 1) / G : 0;
    const int n_stages = n_my * kst;

    if (tid >= kConv0 && tid < kConv0 + 512) {
        // ------------------------------------------------------ converters
        const int grp = (tid - kConv0) >> 8;      // this group converts stages i = grp (mod 2)
        const int ct = (tid - kConv0) & 255;
        // the warp writes its TMEM lane quarter (warp % 4); tile row
        // m = 32 * quarter + lane, 16-byte half ah = converter warp / 4; raw
        // row ra holds tile row m (gate/up rows interleave: m = 2i gate, 2i+1 up)
        const int cw = ct >> 5, m = 32 * (warp & 3) + lane, ah = cw >> 2;
        const int ra = KIND == kGU ? ((m & 1) * 64 + (m >> 1)) : m;
        const int lch = ch == 4 ? 2 : ch == 2 ? 1 : 0;
        int fs = grp, use3 = 0;  // TMEM stage slot (i % kSt) and its use (i / kSt)
        for (int i = grp; i < n_stages; i += 2) {
            const int q = i >> lch, within = i & (ch - 1), rs = q & (kRA - 1);
            bool ok = true;
            if (within < 2) ok = mb_wait(&sm.raw_full[rs], (uint32_t)((q / kRA) & 1), abort, a.err);
            if (ok && i >= kSt) ok = mb_wait(&sm.empty[fs], (uint32_t)((use3 - 1) & 1), abort, a.err);
            if (__any_sync(0xffffffffu, !ok)) break;  // the whole warp leaves together
            // 4 packed words -> 16 f16 pairs of tile row m, to TMEM
            const uint4 w = *reinterpret_cast<const uint4 *>(dyn + kOffRA + (uint32_t)rs * kARaw + raw_row_off(ra) +
                                                             within * 32 + ah * 16);
            if (within + 2 >= ch) {  // this group's last stage of the slot: one arrival per warp
                __syncwarp();
                if (lane == 0) mb_arrive(&sm.raw_empty[rs]);
            }
            const uint4 p0 = w4_to_f16(w.x), p1 = w4_to_f16(w.y), p2 = w4_to_f16(w.z), p3 = w4_to_f16(w.w);
            const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + kTmemA + (uint32_t)fs * kAcolStage +
                                (uint32_t)ah * 16;
            asm volatile(
                "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(ta),
                "r"(p0.x), "r"(p0.y), "r"(p0.z), "r"(p0.w), "r"(p1.x), "r"(p1.y), "r"(p1.z), "r"(p1.w), "r"(p2.x),
                "r"(p2.y), "r"(p2.z), "r"(p2.w), "r"(p3.x), "r"(p3.y), "r"(p3.z), "r"(p3.w)
                : "memory");
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mb_arrive(&sm.full[fs]);
            fs += 2;
            if (fs >= kSt) { fs -= kSt; ++use3; }
        }
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------------- MMA
        if (lane == 0) {
            for (int ti = 0; ti < n_my && !*abort; ++ti) {
                const Tile x = tile_of(a, sm, nu, nwb, b + ti * G);
                const uint32_t idesc = idesc_f16(x.npad);
                const int buf = ti & 1;
                if (ti >= 2 && !mb_wait(&sm.acc_empty[buf], (uint32_t)(((ti >> 1) - 1) & 1), abort, a.err)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t dt = tmem + (uint32_t)(buf * kTok);
                bool ok = true;
                for (int ks = 0; ks < kst; ++ks) {
                    const int i = ti * kst + ks, fs = i % kSt;
                    const uint32_t ph = (uint32_t)((i / kSt) & 1);
                    if (!mb_wait(&sm.full[fs], ph, abort, a.err) || !mb_wait(&sm.bfull[fs], ph, abort, a.err)) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t at = tmem + kTmemA + (uint32_t)fs * kAcolStage, b0 = sbase + kOffB + (uint32_t)fs * kBF16;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t acc = (ks | kk) != 0 ? 1u : 0u;
                        asm volatile(
                            "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                            " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(dt),
                            "r"(at + kk * 8), "l"(desc_sw128(b0 + kk * 32)), "r"(idesc), "r"(acc));
                    }
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                     su32(&sm.empty[fs]))
                                 : "memory");
                }
                if (!ok) break;
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                 su32(&sm.acc_full[buf]))
                             : "memory");
            }
            // every MMA issued by this thread has finished before the TMEM is freed
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             su32(&sm.drain))
                         : "memory");
            const unsigned long long t0 = global_ns();
            while (!mb_try(&sm.drain, 0u))
                if (global_ns() - t0 > kWaitNs) {
                    atomicOr(a.err, kErrSyncTimeout);
                    break;
                }
        }
        __syncwarp();
    } else if (warp == kTmaWarp) {
        // -------------------------------------------- activation tiles (TMA)
        if (lane == 0) {
            int issued = 0, t_ti = -1, nbox = 0, r0 = 0;
            for (int i = 0; i < n_stages && !*abort; ++i) {
                const int ti = i / kst, ks = i - ti * kst, fs = i % kSt;
                if (ti != t_ti) {
                    t_ti = ti;
                    const Tile x = tile_of(a, sm, nu, nwb, b + ti * G);
                    nbox = (x.npad + kBoxRows - 1) / kBoxRows;
                    r0 = x.r0;
                }
                // the slot is free once the MMAs that read it have completed
                if (i >= kSt && !mb_wait(&sm.empty[fs], (uint32_t)(((i / kSt) - 1) & 1), abort, a.err)) break;
                mb_expect_tx(&sm.bfull[fs], (uint32_t)nbox * kBoxRows * 128u);
                const uint32_t dst = sbase + kOffB + (uint32_t)fs * kBF16;
                for (int bx = 0; bx < nbox; ++bx)
                    tma_load_2d(dst + (uint32_t)bx * kBoxRows * 128u, &xmap, ks * kBKs, r0 + kBoxRows * bx, &sm.bfull[fs]);
                issued = i + 1;
            }
            // tiles still in flight land before the CTA may leave (bounded)
            const unsigned long long t0 = global_ns();
            for (int i = issued - kSt < 0 ? 0 : issued - kSt; i < issued; ++i)
                while (!mb_try(&sm.bfull[i % kSt], (uint32_t)((i / kSt) & 1)))
                    if (global_ns() - t0 > kWaitNs) {
                        atomicOr(a.err, kErrSyncTimeout);
                        break;
                    }
        }
        __syncwarp();
    } else if (warp >= kLoadWarp0 && warp < kLoadWarp0 + kLoadWarps) {
        // ------------------------------------------------------ weight loads
        // slot q of the raw ring: 128 weight rows x ch stages (ch * 32 bytes
        // per row), kRA slots ahead of the converters; load warp w copies rows
        // 32w .. 32w+31, lane l the 16-byte pieces l, l + 32, ... of them
        // (row = piece / 8, column piece % 8)
        const int lw = warp - kLoadWarp0;
        const int n_q = n_stages / ch;
        int l_ti = -1, issued = 0;
        const uint8_t *r0p = nullptr, *r1p = nullptr;  // first rows of the two 64-row halves
        for (int q = 0; q < n_q; ++q) {
            const int rs = q % kRA;
            if (q >= kRA && !mb_wait(&sm.raw_empty[rs], (uint32_t)(((q / kRA) - 1) & 1), abort, a.err)) break;
            const int i0 = q * ch, ti = i0 / kst, ks0 = i0 - ti * kst;
            if (ti != l_ti) {
                l_ti = ti;
                const Tile x = tile_of(a, sm, nu, nwb, b + ti * G);
                const DevExpert ex = a.experts[a.meta->uexp[x.u]];
                if (KIND == kGU) {
                    r0p = ex.gq + (size_t)(x.wb * 64) * rowb;
                    r1p = ex.uq + (size_t)(x.wb * 64) * rowb;
                } else {
                    r0p = ex.dq + (size_t)(x.wb * 128) * rowb;
                    r1p = r0p + (size_t)64 * rowb;
                }
            }
            const uint32_t dst = sbase + kOffRA + (uint32_t)rs * kARaw;
            const int pcs = 2 * ch;  // 16-byte pieces per row in this slot
#pragma unroll
            for (int p = lane; p < 32 * 8; p += 32) {
                const int row = 32 * lw + (p >> 3), col = p & 7;
                if (col < pcs) {
                    const uint8_t *src = (row < 64 ? r0p + (size_t)row * rowb : r1p + (size_t)(row - 64) * rowb) +
                                         ks0 * 32 + col * 16;
                    cp_async16(dst + raw_row_off(row) + col * 16, src, 16u);
                }
            }
            cp_async_arrive(&sm.raw_full[rs]);
            issued = q + 1;
        }
        // copies still in flight land before the CTA may leave (bounded)
        const unsigned long long t0 = global_ns();
        for (int q = issued - kRA < 0 ? 0 : issued - kRA; q < issued; ++q)
            while (!mb_try(&sm.raw_full[q % kRA], (uint32_t)((q / kRA) & 1)))
                if (global_ns() - t0 > kWaitNs) {
                    atomicOr(a.err, kErrSyncTimeout);
                    break;
                }
    } else if (warp < 4) {
        // ------------------------------------------------------ epilogue
        for (int ti = 0; ti < n_my; ++ti) {
            const Tile x = tile_of(a, sm, nu, nwb, b + ti * G);
            const int buf = ti & 1;
            const DevExpert ex = a.experts[a.meta->uexp[x.u]];
            if (tid < x.nvalid) {
                const int r = x.r0 + tid, e = a.rows[r];
                sm.tok_r[buf][tid] = r;
                sm.tok_e[buf][tid] = e;
                sm.tok_s[buf][tid] = KIND == kGU ? a.sx[e / S] : a.shq[r];
            }
            if (epi_bar_or(*abort != 0)) break;
            const bool got = mb_wait(&sm.acc_full[buf], (uint32_t)((ti >> 1) & 1), abort, a.err);
            if (epi_bar_or(!got)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(buf * kTok);
            int o;
            float s_a = 0.f, s_b = 0.f;
            if (KIND == kGU) {
                o = x.wb * 64 + warp * 16 + (lane >> 1);
                s_a = __ldg(ex.gs + o);
                s_b = __ldg(ex.us + o);
            } else {
                o = x.wb * 128 + warp * 32 + lane;
                s_a = __ldg(ex.ds + o);
            }
            for (int c0 = 0; c0 < x.npad; c0 += 32) {
                uint32_t v[32];
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                    "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                    : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                      "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                      "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
                      "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
                      "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                    : "r"(ta + (uint32_t)c0));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = c0 + jj;
                    const float acc = __uint_as_float(v[jj]);
                    if (KIND == kGU) {
                        const float up = __shfl_xor_sync(0xffffffffu, acc, 1);
                        float hv = 0.f;
                        if (j < x.nvalid && (lane & 1) == 0) {
                            const int gi = __float2int_rn(acc), ui = __float2int_rn(up);
                            const float sx = sm.tok_s[buf][j];
                            const float gf = __fmul_rn(__fmul_rn((float)gi, sx), s_a);
                            const float uf = __fmul_rn(__fmul_rn((float)ui, sx), s_b);
                            hv = __fmul_rn(silu_f(gf), uf);
                            a.h[(size_t)sm.tok_r[buf][j] * a.I + o] = hv;
                            if (a.dbg.gate_acc) a.dbg.gate_acc[(size_t)sm.tok_e[buf][j] * a.I + o] = gi;
                            if (a.dbg.up_acc) a.dbg.up_acc[(size_t)sm.tok_e[buf][j] * a.I + o] = ui;
                        }
                        float mx = fabsf(hv);
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                        if (lane == 0 && j < kTok) sm.red[warp][j] = mx;
                    } else if (j < x.nvalid) {
                        const int di = __float2int_rn(acc);
                        const float y = __fmul_rn(__fmul_rn((float)di, sm.tok_s[buf][j]), s_a);
                        a.part[(size_t)sm.tok_e[buf][j] * a.D + o] = y;
                        if (a.dbg.down_acc) a.dbg.down_acc[(size_t)sm.tok_e[buf][j] * a.D + o] = di;
                    }
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mb_arrive(&sm.acc_empty[buf]);
            if (KIND == kGU) {
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (tid < x.nvalid) {
                    const float m = fmaxf(fmaxf(sm.red[0][tid], sm.red[1][tid]), fmaxf(sm.red[2][tid], sm.red[3][tid]));
                    atomicMax(a.hamax + x.r0 + tid, __float_as_uint(m));
                }
            }
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == kMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

// The activation operand of the gate/up GEMM: grouped row r = the int8 codes
// of its token (even/odd order kept) as f16 integers (exact).
__global__ void __launch_bounds__(256) act_rows_f16_kernel(const int8_t *__restrict__ xq,
                                                           const int32_t *__restrict__ rows, const RouteMeta *meta,
                                                           int S, int D, __half *__restrict__ xf) {
    const int r = blockIdx.x;
    // grouped rows of this batch: T*S, fewer when adaptive top-p dropped selections
    if (r >= meta->ubeg[meta->n_union]) return;
    const int tok = rows[r] / S;
    const int8_t *src = xq + (size_t)tok * D;
    __half *dst = xf + (size_t)r * D;
    for (int g = threadIdx.x; g < (D >> 3); g += blockDim.x) {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(src + 8 * g));
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t word = k < 2 ? v.x : v.y, sh = 16 * (k & 1);
            const int lo = (int)(int8_t)((word >> sh) & 0xFFu), hi = (int)(int8_t)((word >> (sh + 8)) & 0xFFu);
            o[k] = (uint32_t)__half_as_ushort(__int2half_rn(lo)) | ((uint32_t)__half_as_ushort(__int2half_rn(hi)) << 16);
        }
        *reinterpret_cast<uint4 *>(dst + 8 * g) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <int KIND>
cudaError_t launch_u(const LayerArgs &a, const CUtensorMap &map, int num_sms, cudaStream_t s) {
    auto fn = umma_gemm_kernel<KIND>;
    cudaError_t ce = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (ce != cudaSuccess) return ce;
    fn<<<num_sms, kThreads, kSmemBytes, s>>>(map, a);
    return cudaGetLastError();
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library).
cudaError_t encode_fn(EncodeTiledFn *out) {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        cudaError_t ce = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (ce != cudaSuccess) return ce;
        if (q != cudaDriverEntryPointSuccess || !p) return cudaErrorNotSupported;
        fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    *out = fn;
    return cudaSuccess;
}

// Map of a row-major f16 matrix [rows, cols] (16-byte aligned base, cols a
// multiple of 64): boxes of kBoxRows rows x 64 columns (128 bytes), 128-byte
// swizzle; rows past the matrix read as zeros.
cudaError_t encode_rows_f16(void *base, int rows, int cols, CUtensorMap *map) {
    EncodeTiledFn fn = nullptr;
    cudaError_t ce = encode_fn(&fn);
    if (ce != cudaSuccess) return ce;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBKs, (cuuint32_t)kBoxRows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

bool umma_supported(int D, int I) { return D % 128 == 0 && I % 64 == 0 && D <= kMaxDim && I <= kMaxDim; }

cudaError_t umma_encode_maps(void *xf, int rows, int D, int I, UmmaMaps *maps) {
    if ((reinterpret_cast<uintptr_t>(xf) & 15u) || rows < 1) return cudaErrorInvalidValue;
    cudaError_t ce = encode_rows_f16(xf, rows, D, &maps->gu);
    if (ce == cudaSuccess) ce = encode_rows_f16(xf, rows, I, &maps->dn);
    return ce;
}

cudaError_t launch_act_rows_f16(const LayerArgs &a, cudaStream_t s) {
    act_rows_f16_kernel<<<a.T * a.S, 256, 0, s>>>(a.xq, a.rows, a.meta, a.S, a.D, reinterpret_cast<__half *>(a.xf));
    return cudaGetLastError();
}

cudaError_t launch_umma_gateup(const LayerArgs &a, const UmmaMaps &maps, int num_sms, cudaStream_t s) {
    return launch_u<kGU>(a, maps.gu, num_sms, s);
}

cudaError_t launch_umma_down(const LayerArgs &a, const UmmaMaps &maps, int num_sms, cudaStream_t s) {
    return launch_u<kDN>(a, maps.dn, num_sms, s);
}

}  // namespace moe
