/*
 * moe_oracle.h -- plain, slow CPU oracle for one GLM-5.2 routed-MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * library under serving_router_sigmoid_gb300/.
 *
 * Sources (the only authority on what the layer computes):
 *   [A] reader.mx, "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型":
 *       §02 model config (FP8 e4m3 checkpoint, 128 x 128 weight blocks),
 *       §04 手写的基础数学 (rmsnorm, siluf, layer order),
 *       §05 先用 400 行验证流式思路 (per-row int8 weights, quantize_rows),
 *       §06 从 FP8 到 int4 (FP8 block-scale decoding, per-row int4 packer,
 *           nibble layout, worked example),
 *       §11 MoE 路由与专家执行 (sigmoid+bias top-K router, expert union over the
 *           first keff[s] selections of each token, SwiGLU),
 *       §12 AVX2 整数 kernel (per-row int8 activation quantiser, integer dot).
 *   [B] besthub.dev, "Running 744B MoE on 25GB RAM: Int4, Disk Streaming & MLA
 *       Compression", §06, §11, §12 (summaries of the same steps).
 *   [C] aimsg.uk, "低配电脑也能跑GLM 5.2", 使用方法 item 4 (--topp, adaptive
 *       expert top-p) and 性能数据 (--topp 0.7).
 *
 * Precision: the pages fix fp32 arithmetic (float, expf, lrintf); the oracle
 * follows it.  Integer dot products are exact int32.  The router's double
 * twin (orc_router_gap_f64) only measures the top-K selection margin.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* One expert: gate/up are [I, ceil(D/2)] packed int4 + [I] fp32 row scales,
 * down is [D, ceil(I/2)] packed int4 + [D] fp32 row scales; in an int8-weight
 * layer (weight_bits 8) gate/up are [I, D] int8 and down [D, I] int8 (the
 * pointers then point at int8 codes). */
typedef struct {
    const uint8_t *gq, *uq, *dq;
    const float *gs, *us, *ds;
} OrcExpert;

/* One layer.  experts has E + n_shared entries; the shared expert (if any)
 * is entry E.  Entries of experts no token selects may be NULL. */
typedef struct {
    int D, I, E, K, n_shared;
    float routed_scale;
    const float *Wr;   /* [E, D] fp32 router weight, out-major */
    const float *bias; /* [E] fp32 correction bias */
    const OrcExpert *experts;
    float top_p;       /* adaptive expert top-p in (0, 1); 0 or >= 1: plain top-K */
    int weight_bits;   /* 4 (packed int4, the default; 0 also means 4) or 8 (int8 rows [O, I]) */
} OrcLayer;

/* Optional per-(token, slot) intermediates; every pointer may be NULL.
 * slot s in [0, K) is the s-th selected expert, slot K the shared expert.
 * S = K + n_shared. */
typedef struct {
    int32_t *idx;      /* [T, K] selected experts, selection order */
    float *w;          /* [T, K] routing weights (after routed_scale) */
    int8_t *xq;        /* [T, D] int8 activations, natural order */
    float *sx;         /* [T] activation scales */
    int32_t *gate_acc; /* [T, S, I] */
    int32_t *up_acc;   /* [T, S, I] */
    int8_t *hq;        /* [T, S, I] */
    float *sh;         /* [T, S] */
    int32_t *down_acc; /* [T, S, D] */
    float *y;          /* [T, S, D] expert outputs before the routing weight */
    int32_t *uniq;     /* [E] union of routed experts, first-appearance order */
    int32_t *n_uniq;   /* [1] */
} OrcDebug;

int   orc_version(void);
void  orc_set_threads(int n);
int   orc_max_threads(void);

void  orc_pack_int4(const float *w, uint8_t *q4, float *scale, int64_t O, int64_t I);
void  orc_unpack_int4(const uint8_t *q4, int8_t *v, int64_t O, int64_t I);
/* FP8 E4M3 weights with one fp32 scale_inv per 128 x 128 block (the
 * checkpoint format, [A] §06): decode one byte; dequantise a matrix
 * w8 [O, I] with scale_inv [ceil(O/128), ceil(I/128)] to fp32; or dequantise
 * and pack to int4 in one call (q4 / scale as orc_pack_int4). */
float orc_fp8_e4m3_decode(uint8_t b);
void  orc_fp8_block_dequant(const uint8_t *w8, const float *scale_inv, float *w, int64_t O, int64_t I);
void  orc_fp8_block_to_int4(const uint8_t *w8, const float *scale_inv, uint8_t *q4, float *scale, int64_t O,
                            int64_t I);
float orc_qrow_i8(const float *x, int8_t *q, int64_t n);
void  orc_quant_act(const float *x, int8_t *xq, float *sx, int64_t T, int64_t D);
int32_t orc_dot_i4_i8(const uint8_t *q4row, const int8_t *x, int64_t n);
/* Per-row symmetric quantisation to `bits` (2..8) stored one value per int8
 * ([A] §05 quantize_rows) and the int8 x int8 dot ([A] §12 dot_i8i8). */
void  orc_quantize_rows(const float *w, int8_t *q, float *scale, int64_t O, int64_t I, int bits);
int32_t orc_dot_i8_i8(const int8_t *w, const int8_t *x, int64_t n);
void  orc_router(const float *x, const float *Wr, const float *bias, int T, int D, int E,
                 int K, float routed_scale, int32_t *idx, float *w, float *p_out);
void  orc_router_gap_f64(const float *x, const float *Wr, const float *bias, int T, int D,
                         int E, int K, double *gap);
int   orc_topp_keff(const float *w, int K, float top_p);
int   orc_union(const int32_t *idx, int T, int K, int E, int32_t *uniq);
void  orc_rmsnorm(const float *x, const float *w, float *out, int D, float eps);
int   orc_layer_forward(const OrcLayer *L, const float *x, int T, float *out, OrcDebug *dbg);
int   orc_block_forward(const OrcLayer *L, float *x, const float *norm_w, float eps, int T);

#ifdef __cplusplus
}
#endif
#endif
