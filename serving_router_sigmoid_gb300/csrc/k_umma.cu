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
// Design (GB300).  D[tokens x weight rows] = X[tokens x K] . W[rows x K]^T:
// the tokens of one union entry are the MMA's M side (128 per tile, rows past
// the entry's tokens computed and ignored) and 256 weight rows its N side
// (gate/up: 128 gate rows then the same 128 up rows; down: 256 output rows).
// On this part one M=128, K=16 tcgen05.mma costs about 125 cycles whatever its
// N up to 256 (measured back to back from one thread), so only N = 256 runs
// the tensor cores at their dense rate: the wide weight side goes on N.  K
// runs in stages of 64.
//  - The activation operand is not converted here: a small kernel before the
//    GEMM writes every grouped row of the batch (gate/up: the token's int8
//    codes; down: the requantised h codes) as f16 integers, once, and one
//    producer thread moves each stage's 128-token tile into shared memory
//    with TMA tile loads (boxes of 32 rows x 64 f16 = 128 bytes per row,
//    128-byte swizzle: the K-major layout the MMA reads).
//  - Packed weights, two ways.  With per-expert tensor maps (built with the
//    layer handle) one producer thread moves each stage's 256 rows x 32
//    packed bytes into a 5-stage ring by TMA (boxes of 128 rows).  Without
//    them (the allocation-free entry point) the converter threads load
//    their packed bytes straight from global memory into registers, kPD
//    stages ahead and across tile boundaries (a warp: 16 rows x 32 bytes,
//    whole sectors).
//  - A converter thread owns one weight row of every stage (TMA path: all
//    32 packed bytes, 8 warps; register path: one 16-byte half, 16 warps).
//    Once the stage's f16 slot is free it expands its bytes to f16
//    (a byte permute into 0x64xx patterns and one f16x2 subtraction per
//    pair) and stores the 16-byte results into the stage's
//    128-byte-swizzled K-major weight tile in shared memory (the MMA's B
//    operand); after a proxy fence its warp arrives on the stage's barrier
//    (and releases the TMA ring slot it read: generic reads of memory the
//    async proxy rewrites).  The packed weight nibbles come out in the order
//    e0 e2 e4 e6 e1 e3 e5 e7 of each 8-group, which is exactly the even/odd
//    order in which the activation rows are stored, so both operands see
//    the same permutation of K.
//  - One CTA per SM.  Warps 0..3 are the epilogue (TMEM lanes 0..127 = the
//    tile's tokens); with the TMA weight path the MMA issuer and both TMA
//    issuers share the first scheduler (warp % 4 == 0) with epilogue warp 0
//    only, and the 8 converters the other three, because the MMA issuer
//    runs a stage only when it gets issue slots (moving the converters off
//    its scheduler took gate/up at prefill 2048 from 1.53 to 1.45 ms).
//  - The MMA thread waits for a stage's weights (converter barrier) and its
//    token tile (TMA transaction barrier), issues four M=128, N=256, K=16 MMAs
//    (descriptors formed once per stage, +32 bytes per K=16 slice) and
//    commits them to the "empty" barriers of the stage's weight slot (3
//    slots) and token slot (5 slots: the TMA loads are the slower ones);
//    after a tile's last stage to an accumulator barrier.  Two 256-column
//    TMEM accumulators (all 512 columns) let the epilogue of one tile
//    overlap the MMAs of the next.
//  - Shared memory: 5 token stages (80 KB), 3 f16 weight stages (96 KB) and,
//    with TMA weights, 5 packed stages (40 KB).  The register-load path keeps
//    the CTA at most 196 KB, which leaves the L1 a 60 KB share of the SM's
//    256 KB for its loads in flight (the same kernel with 32 KB more shared
//    memory, unused, ran 1.2x slower).
//  - What bounds it (ncu, gate/up at prefill 2048): the tensor pipe is
//    active ~50% of the time, the LSU data pipe ~50% (the f16 weight stores
//    and their bank conflicts with the tensor core's operand reads), issue
//    ~50%; deeper rings (4 f16 weight stages, 6-8 packed stages) changed
//    nothing, the scheduler that runs the MMA issuer did.
//  - Epilogue: thread m of the 128 holds token m's whole row of the tile:
//    gate/up: 16 gate and the matching 16 up columns at a time,
//    h = silu(g)*u written as contiguous 128-byte runs, max|h| of the token
//    kept in a register; down: y = (acc*sh)*sd into the token's per-slot
//    partial row.
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
constexpr int kBKs = 64;                  // K elements per stage
constexpr int kTok = 128;                 // token rows per tile (the MMA's M)
constexpr int kWN = 256;                  // weight rows per tile (the MMA's N)
constexpr int kBoxRows = 32;              // token rows per TMA box
constexpr uint32_t kXF16 = kTok * 128;    // 128 tokens x 64 f16
constexpr uint32_t kWF16 = kWN * 128;     // 256 weight rows x 64 f16
constexpr uint32_t kRawB = kWN * 32;      // 256 weight rows x 64 packed int4
constexpr int kPD = 4;                    // weight stages each converter thread has in flight (registers)
constexpr uint32_t kTmemCols = 2 * kWN;   // two accumulators of 256 columns
// Stage rings in shared memory: f16 token tiles (TMA), f16 weight tiles
// (converted) and, when the packed weights arrive by TMA (WTMA, one more
// warp issues them), their packed tiles; else the converter threads load the
// packed weights into registers.
template <bool WTMA>
struct Cfg {
    // warps: 0..3 epilogue (TMEM lane quadrants); WTMA: the MMA issuer, the
    // token tile and weight tile TMA issuers on the first sub-partition
    // (warp % 4 == 0), the 8 converters on sub-partitions 1..3, so that the
    // MMA issuer shares its scheduler with no converter work
    static constexpr int kThreads = WTMA ? 480 : 704;  // 15 or 22 warps
    static constexpr int kConv = WTMA ? 8 : 16;        // converter warps
    static constexpr int kMmaWarp = WTMA ? 4 : 20;
    static constexpr int kTmaWarp = WTMA ? 8 : 21;     // token tiles
    static constexpr int kWTmaWarp = WTMA ? 12 : -1;   // packed weight tiles
    // converter index of a warp (0..15), or -1
    __device__ static int conv_of(int w) {
        if (!WTMA) return w >= 4 && w < 20 ? w - 4 : -1;
        if (w < 5 || w > 14 || (w & 3) == 0) return -1;
        return ((w >> 2) - 1) * 3 + (w & 3) - 1;
    }
    static constexpr int kStX = 5;
    static constexpr int kStW = 3;
    static constexpr int kRW = WTMA ? 5 : 0;
    static constexpr uint32_t kOffX = 0;
    static constexpr uint32_t kOffW = kOffX + kStX * kXF16;
    static constexpr uint32_t kOffR = kOffW + kStW * kWF16;
    static constexpr uint32_t kDyn = kOffR + kRW * kRawB;
    static constexpr size_t kSmemBytes = kDyn + 1024;  // + alignment to 1024 bytes
};
constexpr int kStMax = 8;                 // barrier slots of the largest ring

struct UmmaSmem {
    uint64_t full[kStMax], empty_w[kStMax], bfull[kStMax], empty_x[kStMax], acc_full[2], acc_empty[2], drain;
    uint64_t raw_full[kStMax], raw_empty[kStMax];
    uint32_t tmem;
    int abort;
    int tp[kMaxE + 2];        // tiles before each union entry
    float wsc[2][kWN];        // per accumulator: the row scales of the tile's weight rows
};

// Loads into registers need the L1 (its share of the SM's 256 KB is what
// shared memory leaves): 176 KB leaves 60 KB, and the same kernel with 32 KB
// more shared memory, unused, ran 1.2x slower.  TMA loads do not.
static_assert(Cfg<false>::kSmemBytes + sizeof(UmmaSmem) <= 196 * 1024, "keep the L1 share the weight loads need");
static_assert(Cfg<true>::kSmemBytes + sizeof(UmmaSmem) <= 227 * 1024, "shared memory of one CTA");

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

// One 32-byte store of 8 fp32 values (32-byte aligned p): a thread writes a
// whole sector of its row, so the epilogue's scattered row stores take half
// the instructions of 16-byte ones.
__device__ __forceinline__ void st_global_v8(float *p, const float *v) {
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(v[0]), "f"(v[1]),
                 "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                 : "memory");
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
// 16 bytes of packed weights straight into registers (read once per CTA:
// no L1 allocation).
__device__ __forceinline__ uint4 ld_weights16(const uint8_t *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// tcgen05 shared-memory descriptor: K-major, 128-byte swizzle, 8-row atoms
// 1024 bytes apart; the atom base is 1024-byte aligned and the start address
// steps 32 bytes per K=16 slice inside the 128-byte rows.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Byte offset of 16-byte chunk c (K positions 8c..8c+7) of row r in a
// 128-byte-swizzled K-major tile (8-row atoms of 1024 bytes; the chunk index
// is XORed with the row within the atom), the layout TMA's 128-byte swizzle
// writes and desc_sw128 describes.
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
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

// 16 consecutive 32-bit TMEM columns of this warp's 32 lanes (one per lane).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}

// 32 consecutive 32-bit TMEM columns of this warp's 32 lanes (one per lane).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
          "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}

struct Tile {
    int u, wb, r0, nvalid;
};

// Tile t: union entry u, weight block wb (256 rows), token block (128 rows);
// the token blocks of one weight block are consecutive.
__device__ __forceinline__ Tile tile_of(const LayerArgs &a, const UmmaSmem &sm, int nu, int t) {
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
    return x;
}

template <int KIND, bool WTMA>
__global__ void __launch_bounds__(Cfg<WTMA>::kThreads, 1)
    umma_gemm_kernel(const __grid_constant__ CUtensorMap xmap, LayerArgs a) {
    constexpr int kStX = Cfg<WTMA>::kStX, kStW = Cfg<WTMA>::kStW, kRW = Cfg<WTMA>::kRW;
    constexpr int kMmaWarp = Cfg<WTMA>::kMmaWarp, kTmaWarp = Cfg<WTMA>::kTmaWarp, kWTmaWarp = Cfg<WTMA>::kWTmaWarp;
    constexpr uint32_t kOffX = Cfg<WTMA>::kOffX, kOffW = Cfg<WTMA>::kOffW, kOffR = Cfg<WTMA>::kOffR;
    static_assert(kStX <= kStMax && kStW <= kStMax && kRW <= kStMax, "barrier slots");
    extern __shared__ uint8_t dyn_raw[];
    __shared__ UmmaSmem sm;
    uint8_t *dyn = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = su32(dyn);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x, G = gridDim.x, S = a.S;
    const int kdim = KIND == kGU ? a.D : a.I;
    const int rowb = kdim >> 1;
    const int nwb = KIND == kGU ? a.I / (kWN / 2) : a.D / kWN;  // weight blocks per expert
    const int kst = kdim / kBKs;                                // stages per tile
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
        for (int s = 0; s < kStW; ++s) {
            mb_init(&sm.full[s], Cfg<WTMA>::kConv);  // the converter warps
            mb_init(&sm.empty_w[s], 1);
        }
        for (int s = 0; s < kStX; ++s) {
            mb_init(&sm.bfull[s], 1);  // the TMA issuer's arrival, plus the tile's bytes
            mb_init(&sm.empty_x[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mb_init(&sm.acc_full[s], 1);
            mb_init(&sm.acc_empty[s], 4);
        }
        mb_init(&sm.drain, 1);
        for (int s = 0; s < kRW; ++s) {
            mb_init(&sm.raw_full[s], 1);    // the weight TMA issuer's arrival, plus the tile's bytes
            mb_init(&sm.raw_empty[s], Cfg<WTMA>::kConv);  // the converter warps
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

    const int cw = Cfg<WTMA>::conv_of(warp);
    if (WTMA && cw >= 0) {
        // ------------------------------------ converters (weights by TMA)
        // thread: weight row n = 32 * cw + lane of the tile, its 32 packed
        // bytes (a warp reads 1 KB of the ring slot, contiguous; its 16-byte
        // stores of 8 consecutive rows hit 8 different bank groups).  The
        // ring slot is written by the async
        // proxy (TMA) and read here by the generic one, so it is released
        // only after the proxy fence that also publishes the f16 tile.
        const int n = 32 * cw + lane;
        int fs = 0, fph = 0, rs = 0, rph = 0;  // weight tile and ring slots, use parities
        for (int i = 0; i < n_stages; ++i) {
            bool ok = mb_wait(&sm.raw_full[rs], (uint32_t)rph, abort, a.err);
            if (__any_sync(0xffffffffu, !ok)) break;  // the whole warp leaves together
            const uint8_t *rp = dyn + kOffR + (uint32_t)rs * kRawB + (uint32_t)n * 32u;
            const uint4 w = *reinterpret_cast<const uint4 *>(rp), v = *reinterpret_cast<const uint4 *>(rp + 16);
            ok = i < kStW || mb_wait(&sm.empty_w[fs], (uint32_t)(fph ^ 1), abort, a.err);
            if (__any_sync(0xffffffffu, !ok)) break;
            uint8_t *wt = dyn + kOffW + (uint32_t)fs * kWF16;
            *reinterpret_cast<uint4 *>(wt + sw_off(n, 0)) = w4_to_f16(w.x);
            *reinterpret_cast<uint4 *>(wt + sw_off(n, 1)) = w4_to_f16(w.y);
            *reinterpret_cast<uint4 *>(wt + sw_off(n, 2)) = w4_to_f16(w.z);
            *reinterpret_cast<uint4 *>(wt + sw_off(n, 3)) = w4_to_f16(w.w);
            *reinterpret_cast<uint4 *>(wt + sw_off(n, 4)) = w4_to_f16(v.x);
            *reinterpret_cast<uint4 *>(wt + sw_off(n, 5)) = w4_to_f16(v.y);
            *reinterpret_cast<uint4 *>(wt + sw_off(n, 6)) = w4_to_f16(v.z);
            *reinterpret_cast<uint4 *>(wt + sw_off(n, 7)) = w4_to_f16(v.w);
            // the slot read and the tile written, both ordered before the
            // async proxy's next accesses (the TMA refill, the MMA)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                mb_arrive(&sm.raw_empty[rs]);
                mb_arrive(&sm.full[fs]);
            }
            if (++rs == kRW) { rs = 0; rph ^= 1; }
            if (++fs == kStW) { fs = 0; fph ^= 1; }
        }
    } else if (!WTMA && cw >= 0) {
        // ------------------------------------------------------ converters
        // thread: weight row n = 16 * cw + lane / 2 of the tile (a warp reads
        // 16 whole 32-byte row pieces per stage), 16-byte half hf = lane % 2
        // of the stage's 32 packed bytes; the loads run kPD stages ahead in
        // registers, across tile boundaries
        const int n = 16 * cw + (lane >> 1), hf = lane & 1;
        int l_i = 0, l_ti = 0, l_ks = 0;  // the next stage to load and its tile / K stage
        const uint8_t *src = nullptr;     // this thread's row piece in the tile l_ti
        auto load_next = [&](uint4 &dst) {
            if (l_i >= n_stages) return;
            if (l_ks == 0) {
                const Tile x = tile_of(a, sm, nu, b + l_ti * G);
                const DevExpert ex = a.experts[a.meta->uexp[x.u]];
                if (KIND == kGU)
                    src = n < 128 ? ex.gq + (size_t)(x.wb * 128 + n) * rowb : ex.uq + (size_t)(x.wb * 128 + n - 128) * rowb;
                else
                    src = ex.dq + (size_t)(x.wb * 256 + n) * rowb;
                src += hf * 16;
            }
            dst = ld_weights16(src + l_ks * 32);
            ++l_i;
            if (++l_ks == kst) { l_ks = 0; ++l_ti; }
        };
        uint4 pre[kPD];
#pragma unroll
        for (int k = 0; k < kPD; ++k) load_next(pre[k]);
        int fs = 0, fph = 0;  // stage slot i % kStW and its use parity
        bool run = true;
        for (int i0 = 0; i0 < n_stages && run; i0 += kPD) {
#pragma unroll
            for (int k = 0; k < kPD; ++k) {
                const int i = i0 + k;
                if (i >= n_stages) break;
                const uint4 w = pre[k];
                load_next(pre[k]);
                const bool ok = i < kStW || mb_wait(&sm.empty_w[fs], (uint32_t)(fph ^ 1), abort, a.err);
                if (__any_sync(0xffffffffu, !ok)) {  // the whole warp leaves together
                    run = false;
                    break;
                }
                uint8_t *wt = dyn + kOffW + (uint32_t)fs * kWF16;
                *reinterpret_cast<uint4 *>(wt + sw_off(n, 4 * hf + 0)) = w4_to_f16(w.x);
                *reinterpret_cast<uint4 *>(wt + sw_off(n, 4 * hf + 1)) = w4_to_f16(w.y);
                *reinterpret_cast<uint4 *>(wt + sw_off(n, 4 * hf + 2)) = w4_to_f16(w.z);
                *reinterpret_cast<uint4 *>(wt + sw_off(n, 4 * hf + 3)) = w4_to_f16(w.w);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // to the MMA's proxy
                __syncwarp();
                if (lane == 0) mb_arrive(&sm.full[fs]);
                if (++fs == kStW) { fs = 0; fph ^= 1; }
            }
        }
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | ((uint32_t)(kWN >> 3) << 17) | ((uint32_t)(kTok >> 4) << 24);
            int fs = 0, fph = 0, xs = 0, xph = 0;  // weight and token stage slots, use parities
            for (int ti = 0; ti < n_my && !*abort; ++ti) {
                const int buf = ti & 1;
                if (ti >= 2 && !mb_wait(&sm.acc_empty[buf], (uint32_t)(((ti >> 1) - 1) & 1), abort, a.err)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t dt = tmem + (uint32_t)(buf * kWN);
                bool ok = true;
                for (int ks = 0; ks < kst; ++ks) {
                    if (!mb_wait(&sm.full[fs], (uint32_t)fph, abort, a.err) ||
                        !mb_wait(&sm.bfull[xs], (uint32_t)xph, abort, a.err)) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint64_t dx = desc_sw128(sbase + kOffX + (uint32_t)xs * kXF16);
                    const uint64_t dw = desc_sw128(sbase + kOffW + (uint32_t)fs * kWF16);
                    const uint32_t acc = ks != 0 ? 1u : 0u;
                    // four K=16 slices: the descriptors' start address steps 32 bytes (2 units)
                    asm volatile(
                        "{\n .reg .pred p, q;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 q, 1, 0;\n"
                        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
                        " tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %3, q;\n"
                        " tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %3, q;\n"
                        " tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %3, q;\n}" ::"r"(dt),
                        "l"(dx), "l"(dw), "r"(idesc), "r"(acc), "l"(dx + 2), "l"(dw + 2), "l"(dx + 4), "l"(dw + 4),
                        "l"(dx + 6), "l"(dw + 6));
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                     su32(&sm.empty_w[fs]))
                                 : "memory");
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                     su32(&sm.empty_x[xs]))
                                 : "memory");
                    if (++fs == kStW) { fs = 0; fph ^= 1; }
                    if (++xs == kStX) { xs = 0; xph ^= 1; }
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
            int issued = 0, t_ti = -1, r0 = 0, fs = 0, fph = 0;
            for (int i = 0; i < n_stages && !*abort; ++i) {
                const int ti = i / kst, ks = i - ti * kst;
                if (ti != t_ti) {
                    t_ti = ti;
                    r0 = tile_of(a, sm, nu, b + ti * G).r0;
                }
                // the slot is free once the MMAs that read it have completed
                if (i >= kStX && !mb_wait(&sm.empty_x[fs], (uint32_t)(fph ^ 1), abort, a.err)) break;
                mb_expect_tx(&sm.bfull[fs], kXF16);
                const uint32_t dst = sbase + kOffX + (uint32_t)fs * kXF16;
#pragma unroll
                for (int bx = 0; bx < kTok / kBoxRows; ++bx)
                    tma_load_2d(dst + (uint32_t)bx * kBoxRows * 128u, &xmap, ks * kBKs, r0 + kBoxRows * bx, &sm.bfull[fs]);
                issued = i + 1;
                if (++fs == kStX) { fs = 0; fph ^= 1; }
            }
            // tiles still in flight land before the CTA may leave (bounded)
            const unsigned long long t0 = global_ns();
            for (int i = issued - kStX < 0 ? 0 : issued - kStX; i < issued; ++i)
                while (!mb_try(&sm.bfull[i % kStX], (uint32_t)((i / kStX) & 1)))
                    if (global_ns() - t0 > kWaitNs) {
                        atomicOr(a.err, kErrSyncTimeout);
                        break;
                    }
        }
        __syncwarp();
    } else if (WTMA && warp == kWTmaWarp) {
        // ------------------------------------------ packed weight tiles (TMA)
        // each stage: the tile's 256 rows x 32 bytes, two boxes of 128 rows
        // (gate/up: the gate rows, then the same rows of up; down: 256 rows)
        if (lane == 0) {
            int issued = 0, t_ti = -1, y0 = 0, y1 = 0, rs = 0, rph = 0;
            const CUtensorMap *m0 = nullptr, *m1 = nullptr;
            for (int i = 0; i < n_stages && !*abort; ++i) {
                const int ti = i / kst, ks = i - ti * kst;
                if (ti != t_ti) {
                    t_ti = ti;
                    const Tile x = tile_of(a, sm, nu, b + ti * G);
                    const int e = a.meta->uexp[x.u];
                    if (KIND == kGU) {
                        m0 = a.wmaps + 3 * e;
                        m1 = m0 + 1;
                        y0 = y1 = x.wb * 128;
                    } else {
                        m0 = m1 = a.wmaps + 3 * e + 2;
                        y0 = x.wb * 256;
                        y1 = y0 + 128;
                    }
                }
                // the slot is free once every converter warp has read it
                if (i >= kRW && !mb_wait(&sm.raw_empty[rs], (uint32_t)(rph ^ 1), abort, a.err)) break;
                mb_expect_tx(&sm.raw_full[rs], kRawB);
                const uint32_t dst = sbase + kOffR + (uint32_t)rs * kRawB;
                tma_load_2d(dst, m0, ks * 32, y0, &sm.raw_full[rs]);
                tma_load_2d(dst + kRawB / 2, m1, ks * 32, y1, &sm.raw_full[rs]);
                issued = i + 1;
                if (++rs == kRW) { rs = 0; rph ^= 1; }
            }
            // tiles still in flight land before the CTA may leave (bounded)
            const unsigned long long t0 = global_ns();
            for (int i = issued - kRW < 0 ? 0 : issued - kRW; i < issued; ++i)
                while (!mb_try(&sm.raw_full[i % kRW], (uint32_t)((i / kRW) & 1)))
                    if (global_ns() - t0 > kWaitNs) {
                        atomicOr(a.err, kErrSyncTimeout);
                        break;
                    }
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------ epilogue
        // thread m = token row m of the tile (TMEM lane m)
        const int m = tid;
        for (int ti = 0; ti < n_my; ++ti) {
            const Tile x = tile_of(a, sm, nu, b + ti * G);
            const int buf = ti & 1;
            const DevExpert ex = a.experts[a.meta->uexp[x.u]];
            // the tile's 256 weight-row scales (gate/up: gate then up)
            for (int j = tid; j < kWN; j += 128)
                sm.wsc[buf][j] = KIND == kGU ? __ldg((j < 128 ? ex.gs : ex.us) + x.wb * 128 + (j & 127))
                                             : __ldg(ex.ds + x.wb * 256 + j);
            const bool valid = m < x.nvalid;
            const int r = x.r0 + m;
            const int e = valid ? a.rows[r] : 0;
            const float ts = valid ? (KIND == kGU ? a.sx[e / S] : a.shq[r]) : 0.f;
            if (epi_bar_or(*abort != 0)) break;  // also orders the scale stores before their reads
            const bool got = mb_wait(&sm.acc_full[buf], (uint32_t)((ti >> 1) & 1), abort, a.err);
            if (epi_bar_or(!got)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(buf * kWN);
            float hmax = 0.f;
            if (KIND == kGU) {
                // 16 gate columns and the matching 16 up columns at a time
                for (int c = 0; c < 8; ++c) {
                    uint32_t v[16], u[16];
                    tmem_ld16(ta + (uint32_t)(16 * c), v);
                    tmem_ld16(ta + (uint32_t)(128 + 16 * c), u);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                    if (!valid) continue;
                    const int o0 = x.wb * 128 + 16 * c;
                    float hv[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int gi = __float2int_rn(__uint_as_float(v[jj])), ui = __float2int_rn(__uint_as_float(u[jj]));
                        const float gf = __fmul_rn(__fmul_rn((float)gi, ts), sm.wsc[buf][16 * c + jj]);
                        const float uf = __fmul_rn(__fmul_rn((float)ui, ts), sm.wsc[buf][128 + 16 * c + jj]);
                        hv[jj] = __fmul_rn(silu_f(gf), uf);
                        hmax = fmaxf(hmax, fabsf(hv[jj]));
                        if (a.dbg.gate_acc) a.dbg.gate_acc[(size_t)e * a.I + o0 + jj] = gi;
                        if (a.dbg.up_acc) a.dbg.up_acc[(size_t)e * a.I + o0 + jj] = ui;
                    }
                    float *hp = a.h + (size_t)r * a.I + o0;
#pragma unroll
                    for (int q = 0; q < 2; ++q) st_global_v8(hp + 8 * q, hv + 8 * q);
                }
            } else {
                for (int c = 0; c < 8; ++c) {
                    uint32_t v[32];
                    tmem_ld32(ta + (uint32_t)(32 * c), v);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                    if (!valid) continue;
                    const int o0 = x.wb * 256 + 32 * c;
                    float yv[32];
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        const int di = __float2int_rn(__uint_as_float(v[jj]));
                        yv[jj] = __fmul_rn(__fmul_rn((float)di, ts), sm.wsc[buf][32 * c + jj]);
                        if (a.dbg.down_acc) a.dbg.down_acc[(size_t)e * a.D + o0 + jj] = di;
                    }
                    float *yp = a.part + (size_t)e * a.D + o0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) st_global_v8(yp + 8 * q, yv + 8 * q);
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mb_arrive(&sm.acc_empty[buf]);
            if (KIND == kGU && valid) atomicMax(a.hamax + r, __float_as_uint(hmax));
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == kMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

// The activation operand of the gate/up GEMM: grouped row r = the int8 codes
// of its token (even/odd order kept) as f16 integers (exact).  kAR grouped
// rows per CTA, each pass's loads of every row issued before the first is
// converted.
constexpr int kAR = 4;
__global__ void __launch_bounds__(256) act_rows_f16_kernel(const int8_t *__restrict__ xq,
                                                           const int32_t *__restrict__ rows, const RouteMeta *meta,
                                                           int S, int D, __half *__restrict__ xf) {
    // grouped rows of this batch: T*S, fewer when adaptive top-p dropped selections
    const int n_rows = meta->ubeg[meta->n_union];
    const int r0 = blockIdx.x * kAR;
    if (r0 >= n_rows) return;
    int tok[kAR];
#pragma unroll
    for (int j = 0; j < kAR; ++j) tok[j] = r0 + j < n_rows ? rows[r0 + j] / S : 0;
    for (int g = threadIdx.x; g < (D >> 3); g += blockDim.x) {
        uint2 v[kAR];
#pragma unroll
        for (int j = 0; j < kAR; ++j)
            if (r0 + j < n_rows) v[j] = __ldg(reinterpret_cast<const uint2 *>(xq + (size_t)tok[j] * D + 8 * g));
#pragma unroll
        for (int j = 0; j < kAR; ++j) {
            if (r0 + j >= n_rows) continue;
            uint32_t o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t word = k < 2 ? v[j].x : v[j].y, sh = 16 * (k & 1);
                const int lo = (int)(int8_t)((word >> sh) & 0xFFu), hi = (int)(int8_t)((word >> (sh + 8)) & 0xFFu);
                o[k] = (uint32_t)__half_as_ushort(__int2half_rn(lo)) | ((uint32_t)__half_as_ushort(__int2half_rn(hi)) << 16);
            }
            *reinterpret_cast<uint4 *>(xf + (size_t)(r0 + j) * D + 8 * g) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

template <int KIND, bool WTMA>
cudaError_t launch_u(const LayerArgs &a, const CUtensorMap &map, int num_sms, cudaStream_t s) {
    auto fn = umma_gemm_kernel<KIND, WTMA>;
    constexpr size_t smem = Cfg<WTMA>::kSmemBytes;
    cudaError_t ce = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (ce != cudaSuccess) return ce;
    fn<<<num_sms, Cfg<WTMA>::kThreads, smem, s>>>(map, a);
    return cudaGetLastError();
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).
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

// gate/up tiles take 128 gate and 128 up rows, down tiles 256 output rows
bool umma_supported(int D, int I) { return D % 256 == 0 && I % 128 == 0 && D <= kMaxDim && I <= kMaxDim; }

cudaError_t umma_encode_maps(void *xf, int rows, int D, int I, UmmaMaps *maps) {
    if ((reinterpret_cast<uintptr_t>(xf) & 15u) || rows < 1) return cudaErrorInvalidValue;
    cudaError_t ce = encode_rows_f16(xf, rows, D, &maps->gu);
    if (ce == cudaSuccess) ce = encode_rows_f16(xf, rows, I, &maps->dn);
    return ce;
}

cudaError_t launch_act_rows_f16(const LayerArgs &a, cudaStream_t s) {
    act_rows_f16_kernel<<<(a.T * a.S + kAR - 1) / kAR, 256, 0, s>>>(a.xq, a.rows, a.meta, a.S, a.D,
                                                                   reinterpret_cast<__half *>(a.xf));
    return cudaGetLastError();
}

cudaError_t launch_umma_gateup(const LayerArgs &a, const UmmaMaps &maps, int num_sms, cudaStream_t s) {
    return a.wmaps ? launch_u<kGU, true>(a, maps.gu, num_sms, s) : launch_u<kGU, false>(a, maps.gu, num_sms, s);
}

cudaError_t launch_umma_down(const LayerArgs &a, const UmmaMaps &maps, int num_sms, cudaStream_t s) {
    return a.wmaps ? launch_u<kDN, true>(a, maps.dn, num_sms, s) : launch_u<kDN, false>(a, maps.dn, num_sms, s);
}

// The packed weight tiles of every expert of the table: per expert three
// maps (gate, up, down) of uint8 rows, boxes of 32 bytes x 128 rows, no
// swizzle (the converters read 32-byte row pieces), 256-byte L2 promotion.
cudaError_t umma_encode_weight_maps(const DevExpert *tab, int ne, int D, int I, CUtensorMap *maps) {
    EncodeTiledFn fn = nullptr;
    cudaError_t ce = encode_fn(&fn);
    if (ce != cudaSuccess) return ce;
    auto enc = [&](const uint8_t *base, int rows, int rowb, CUtensorMap *m) {
        if (!base || (reinterpret_cast<uintptr_t>(base) & 15u)) return false;
        const cuuint64_t dims[2] = {(cuuint64_t)rowb, (cuuint64_t)rows};
        const cuuint64_t strides[1] = {(cuuint64_t)rowb};
        const cuuint32_t box[2] = {32u, 128u};
        const cuuint32_t estr[2] = {1, 1};
        return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    for (int e = 0; e < ne; ++e)
        if (!enc(tab[e].gq, I, D / 2, &maps[3 * e]) || !enc(tab[e].uq, I, D / 2, &maps[3 * e + 1]) ||
            !enc(tab[e].dq, D, I / 2, &maps[3 * e + 2]))
            return cudaErrorInvalidValue;
    return cudaSuccess;
}

}  // namespace moe
