// k_fp8.cu -- the checkpoint converter's step on the GPU: an FP8 E4M3 weight
// matrix with one fp32 scale_inv per 128 x 128 block, dequantised and packed
// to the int4 layout with one fp32 scale per row, in one pass over HBM.
//
// Sources: reader.mx "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型" §02 (the
// checkpoint config: quant_method fp8, fmt e4m3, weight_block_size
// [128, 128]) and §06 从 FP8 到 int4 (FP8 block-scale decoding: the bytes
// widened to fp32 times the block's scale_inv; then the per-row int4 packer:
// s = max(amax / 7, 1e-8), nearest integer of w / s with ties to even, clamped
// to [-8, 7], stored +8 as nibbles, element 2j low); besthub.dev "Running 744B
// MoE on 25GB RAM" §06.
//
// Design (GB300).  The step is HBM-bound: 1 byte read and half a byte written
// per weight.  One warp owns one row at a time.  The amax pass issues all of a
// lane's 16-byte loads of the row at once (rows of up to 8192 codes) and keeps
// nothing but the running maximum; the packing pass walks the row's chunks
// again, one at a time, from L1, so the code and the register footprint stay
// small (an unrolled packing pass overflowed the instruction cache and halved
// the occupancy) and no fp32 copy of the matrix exists.  A 16-byte chunk lies
// inside one 128-column block, so each chunk needs one scale.  E4M3 is
// sign-magnitude with a monotone encoding, so the largest |value| of a chunk
// is the one of its largest 7-bit magnitude code, and (rounding being
// monotone) the chunk's largest |w| is that value times the block scale: the
// amax pass costs a few byte-max instructions per chunk.  The widening uses
// the hardware e4m3x2 -> f16x2 conversion (exact: every E4M3 value is an f16
// value), then f16 -> f32 (exact).  The packer's division is replaced, where
// that provably gives the same code, by a product with the row's reciprocal
// (nibble2_fast, two codes per packed f32x2 instruction); a chunk with a
// quotient near a tie is redone exactly.  Rows that are not a multiple of 16
// codes, longer than 8192 or unaligned take a plain per-element path with the
// packer's arithmetic.
#include "layer_args.cuh"

namespace moe {

namespace {

constexpr int kWarpsPerCta = 8;
constexpr int kMaxCpl = 16;  // 16-byte chunks per lane: rows of up to 32 * 16 * 16 = 8192 codes

// Two E4M3 codes (low byte -> .x) widened to fp32, exactly.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two) {
    uint32_t h;
    asm("{\n .reg .b16 lo;\n cvt.u16.u32 lo, %1;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n}" : "=r"(h) : "r"(two));
    float2 r;
    asm("{\n .reg .f16 a, b;\n mov.b32 {a, b}, %2;\n cvt.f32.f16 %0, a;\n cvt.f32.f16 %1, b;\n}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(h));
    return r;
}

// The packer's code of one dequantised value: nearest integer of w / s (IEEE
// division, ties to even), clamped to [-8, 7], plus 8.
__device__ __forceinline__ uint32_t nibble_of(float w, float s) {
    const int v = __float2int_rn(__fdiv_rn(w, s));
    return (uint32_t)(min(7, max(-8, v)) + 8);
}

// Two fp32 lanes in one 64-bit register pair (.x low), and the packed
// two-lane IEEE operations of sm_100 and later: each lane is rounded to
// nearest exactly as the scalar operation would round it.
__device__ __forceinline__ unsigned long long f32x2_of(float lo, float hi) {
    return ((unsigned long long)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ unsigned long long mul_f32x2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long add_f32x2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long sub_f32x2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// The packer's code without the division, where that provably gives the
// same result.  With inv = fl(1/s) and g = fl(sc * inv), y = fl(v * g) differs
// from the packer's quotient fl(fl(v * sc) / s) by at most five roundings of
// relative size 2^-24 of a quotient whose magnitude is at most 7 (|w| <= amax,
// s >= amax/7 rounded): less than 2^-18.  So when y lies farther than 2^-17
// from every half-integer, both round to the same integer.  Rounding y to an
// integer: adding M = 1.5 * 2^23 + 8 rounds at integer granularity with ties
// to even (M is even) and leaves 8 + nearest(y) in the low four bits of the
// sum (|nearest(y)| <= 7, so no borrow or carry leaves the nibble).  `near`
// is set when y lies within 2^-17 of a half-integer: the caller then forms
// the quotient exactly as the packer does.
// Here for the two codes of v at once: returns the two sums z (lane x in
// the low word), whose low bytes are 8 + nearest(y) (0..15: the nibbles);
// rmax collects max |y - nearest(y)|.  g2 and m2 hold g and M in both lanes.
__device__ __forceinline__ unsigned long long nibble2_fast(float2 v, unsigned long long g2, unsigned long long m2,
                                                           float &rmax) {
    const unsigned long long y = mul_f32x2(f32x2_of(v.x, v.y), g2);
    const unsigned long long z = add_f32x2(y, m2);
    const unsigned long long r = sub_f32x2(y, sub_f32x2(z, m2));  // y - nearest(y), exact
    rmax = fmaxf(rmax, fmaxf(fabsf(__uint_as_float((uint32_t)r)), fabsf(__uint_as_float((uint32_t)(r >> 32)))));
    return z;
}

// Packed bytes of one 16-code chunk (4 words, element 2j low nibble).  Per
// word, the four sums' low bytes are gathered into one word [n0 n1 n2 n3]
// (byte permutes); q | q >> 4 then holds n0 | n1 << 4 in byte 0 and
// n2 | n3 << 4 in byte 2, and a last permute joins two words' bytes 0 and 2.
// near is set when a quotient lies within 2^-17 of a half-integer.
__device__ __forceinline__ uint2 pack_chunk_fast(uint4 c, float g, bool &near) {
    constexpr float kM = 12582920.f;  // 1.5 * 2^23 + 8 (nibble2_fast)
    const unsigned long long g2 = f32x2_of(g, g), m2 = f32x2_of(kM, kM);
    float rmax = 0.f;
    auto word = [&](uint32_t w) {
        const unsigned long long za = nibble2_fast(e4m3x2_to_f32x2(w & 0xFFFFu), g2, m2, rmax);
        const unsigned long long zb = nibble2_fast(e4m3x2_to_f32x2(w >> 16), g2, m2, rmax);
        const uint32_t q = __byte_perm(__byte_perm((uint32_t)za, (uint32_t)(za >> 32), 0x0040),
                                       __byte_perm((uint32_t)zb, (uint32_t)(zb >> 32), 0x0040), 0x5410);
        return q | (q >> 4);
    };
    const uint32_t t0 = word(c.x), t1 = word(c.y), t2 = word(c.z), t3 = word(c.w);
    near = rmax >= 0.5f - 7.62939453125e-06f;
    return make_uint2(__byte_perm(t0, t1, 0x6420), __byte_perm(t2, t3, 0x6420));
}

// The packer's arithmetic for a whole chunk (rare: a quotient near a tie).
__device__ __noinline__ uint2 pack_chunk_exact(uint4 c, float sc, float s) {
    uint32_t out[2] = {0u, 0u};
    const uint32_t wd[4] = {c.x, c.y, c.z, c.w};
    for (int q = 0; q < 8; ++q) {
        const float2 v = e4m3x2_to_f32x2((wd[q >> 1] >> (16 * (q & 1))) & 0xFFFFu);
        const uint32_t pair = nibble_of(__fmul_rn(v.x, sc), s) | (nibble_of(__fmul_rn(v.y, sc), s) << 4);
        out[q >> 2] |= pair << (8 * (q & 3));
    }
    return make_uint2(out[0], out[1]);
}

// Largest magnitude code (0..127) among the 16 codes of a chunk.
__device__ __forceinline__ uint32_t max_mag_code(uint4 c) {
    const uint32_t m = 0x7F7F7F7Fu;
    uint32_t v = __vmaxu4(__vmaxu4(c.x & m, c.y & m), __vmaxu4(c.z & m, c.w & m));
    v = __vmaxu4(v, v >> 16);
    v = __vmaxu4(v, v >> 8);
    return v & 0xFFu;
}

__device__ __forceinline__ float row_scale(float amax) {
    float s = __fdiv_rn(amax, 7.f);
    return s < 1e-8f ? 1e-8f : s;
}

// Rows of I = 16 * nch codes (nch <= 32 * CPL), 16-byte aligned rows.  The
// amax pass issues all of a lane's 16-byte loads of the row at once (they
// stay in L1); the packing pass reloads one chunk at a time, which keeps the
// loop small and the registers few.
template <int CPL>
__global__ void __launch_bounds__(32 * kWarpsPerCta) fp8_to_int4_kernel(const uint8_t *__restrict__ w8,
                                                                         const float *__restrict__ si,
                                                                         uint8_t *__restrict__ q4,
                                                                         float *__restrict__ scale, long long O,
                                                                         int I) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nch = I >> 4, nbi = (I + 127) >> 7;
    const long long stride = (long long)gridDim.x * kWarpsPerCta;
    for (long long o = (long long)blockIdx.x * kWarpsPerCta + warp; o < O; o += stride) {
        const uint4 *row = reinterpret_cast<const uint4 *>(w8 + o * I);
        const float *srow = si + (o >> 7) * nbi;
        uint4 raw[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            const int c = lane + 32 * j;
            raw[j] = c < nch ? __ldg(row + c) : make_uint4(0u, 0u, 0u, 0u);
        }
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            const int c = lane + 32 * j;
            const float sc = c < nch ? __ldg(srow + (c >> 3)) : 0.f;
            const float v = e4m3x2_to_f32x2(max_mag_code(raw[j])).x;
            amax = fmaxf(amax, fabsf(__fmul_rn(v, sc)));
        }
        amax = warp_max_f(amax);
        const float s = row_scale(amax);
        if (lane == 0) scale[o] = s;
        const float inv = __fdiv_rn(1.f, s);
        uint2 *qrow = reinterpret_cast<uint2 *>(q4 + o * (I >> 1));
#pragma unroll 1
        for (int c = lane; c < nch; c += 32) {
            const uint4 cv = __ldg(row + c);
            const float sc = __ldg(srow + (c >> 3));
            bool near = false;
            uint2 pk = pack_chunk_fast(cv, __fmul_rn(sc, inv), near);
            if (near) pk = pack_chunk_exact(cv, sc, s);
            qrow[c] = pk;
        }
    }
}

// Any shape and alignment: per element, reading the row twice.
__global__ void __launch_bounds__(32 * kWarpsPerCta) fp8_to_int4_any_kernel(const uint8_t *__restrict__ w8,
                                                                             const float *__restrict__ si,
                                                                             uint8_t *__restrict__ q4,
                                                                             float *__restrict__ scale, long long O,
                                                                             long long I) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long nbi = (I + 127) >> 7, nb = (I + 1) >> 1;
    const long long stride = (long long)gridDim.x * kWarpsPerCta;
    for (long long o = (long long)blockIdx.x * kWarpsPerCta + warp; o < O; o += stride) {
        const uint8_t *row = w8 + o * I;
        const float *srow = si + (o >> 7) * nbi;
        float amax = 0.f;
        for (long long i = lane; i < I; i += 32)
            amax = fmaxf(amax, fabsf(__fmul_rn(e4m3x2_to_f32x2(row[i]).x, __ldg(srow + (i >> 7)))));
        amax = warp_max_f(amax);
        const float s = row_scale(amax);
        if (lane == 0) scale[o] = s;
        for (long long j = lane; j < nb; j += 32) {
            const long long i = 2 * j;
            const uint32_t lo = nibble_of(__fmul_rn(e4m3x2_to_f32x2(row[i]).x, __ldg(srow + (i >> 7))), s);
            const uint32_t hi =
                i + 1 < I ? nibble_of(__fmul_rn(e4m3x2_to_f32x2(row[i + 1]).x, __ldg(srow + ((i + 1) >> 7))), s)
                          : 8u;
            q4[o * nb + j] = (uint8_t)(lo | (hi << 4));
        }
    }
}

template <int CPL>
cudaError_t launch_fast(const uint8_t *w8, const float *si, uint8_t *q4, float *scale, int64_t O, int64_t I,
                        int grid, cudaStream_t s) {
    fp8_to_int4_kernel<CPL><<<grid, 32 * kWarpsPerCta, 0, s>>>(w8, si, q4, scale, O, (int)I);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fp8_to_int4(const uint8_t *w8, const float *si, uint8_t *q4, float *scale, int64_t O, int64_t I,
                               cudaStream_t s) {
    int dev = 0, nsm = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (ce != cudaSuccess) return ce;
    // a persistent grid: rows are handed out by a grid-stride loop
    const int64_t ctas = (O + kWarpsPerCta - 1) / kWarpsPerCta;
    const int per_sm = 8;
    const int grid = (int)(ctas < (int64_t)nsm * per_sm ? ctas : (int64_t)nsm * per_sm);
    const bool fast = I > 0 && I % 16 == 0 && I <= 512 * kMaxCpl &&
                      (reinterpret_cast<uintptr_t>(w8) & 15u) == 0 && (reinterpret_cast<uintptr_t>(q4) & 7u) == 0;
    if (fast) {
        const int64_t cpl = (I / 16 + 31) / 32;
        if (cpl <= 4) return launch_fast<4>(w8, si, q4, scale, O, I, grid, s);
        if (cpl <= 8) return launch_fast<8>(w8, si, q4, scale, O, I, grid, s);
        if (cpl <= 12) return launch_fast<12>(w8, si, q4, scale, O, I, grid, s);
        return launch_fast<16>(w8, si, q4, scale, O, I, grid, s);
    }
    fp8_to_int4_any_kernel<<<grid, 32 * kWarpsPerCta, 0, s>>>(w8, si, q4, scale, O, I);
    return cudaGetLastError();
}

}  // namespace moe
