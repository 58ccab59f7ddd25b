/*
 * moe_int4.h -- C ABI of a GB300 (sm_103a) routed-MoE layer library.
 *
 * The library computes one GLM-5.2 (glm_moe_dsa) routed-MoE layer forward:
 * a sigmoid router with correction bias choosing top-K of E experts with
 * weights sigmoid(logit) * routed_scale, SwiGLU experts stored as packed int4
 * with one fp32 scale per row, applied to activations quantised per row to
 * int8, a batch-wide union of experts so each expert's weights are read once,
 * and an always-on shared expert.
 *
 * Sources (page title, section):
 *   reader.mx, "惊呆了！25GB 内存上运行 GLM 5.2 744B 模型":
 *     §02 模型与硬件 (model config: hidden 6144, 256 experts, top-8, 1 shared
 *         expert, moe_intermediate 2048, sigmoid scoring, routed_scaling_factor 2.5),
 *     §04 手写的基础数学 (rmsnorm with double accumulation; siluf; layer order),
 *     §06 从 FP8 到 int4 (per-row int4 packing and nibble layout),
 *     §11 MoE 路由与专家执行 (router, expert union, SwiGLU and weighted add),
 *     §12 AVX2 整数 kernel (per-row int8 activation quantiser, integer dot).
 *   besthub.dev, "Running 744B MoE on 25GB RAM: Int4, Disk Streaming & MLA
 *     Compression", §06, §11, §12 (the same steps summarised).
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers unless the parameter says "host".
 *   - Every call is asynchronous on `stream` (0 = legacy default stream); it
 *     only validates arguments on the host and enqueues kernels.  No call
 *     allocates, frees or synchronises, except moe_layer_create / _destroy
 *     and moe_layer_device_status (which synchronises `stream`).
 *   - Return value: MOE_OK (0) or a negative MOE_ERR_* code.  On error nothing
 *     was enqueued unless the code is MOE_ERR_CUDA (a launch failed); the text
 *     of the last error on the calling thread is in moe_last_error().
 *   - There is no CPU fallback: a missing GPU or a failed launch is an error.
 *   - Non-finite inputs (NaN / Inf) are outside the contract; the kernels stay
 *     memory-safe on them but the results are unspecified.
 */
#ifndef MOE_INT4_H
#define MOE_INT4_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1) /* NULL or misaligned pointer, bad handle, bad scalar */
#define MOE_ERR_SHAPE (-2)       /* unsupported or mismatched sizes, n_tokens > max_tokens */
#define MOE_ERR_CUDA (-3)        /* a CUDA call or kernel launch failed */
#define MOE_ERR_NOMEM (-4)       /* device allocation failed (create only) */
#define MOE_ERR_DEVICE (-5)      /* a kernel flagged an inconsistency (moe_layer_device_status) */

/* Library version, (major << 16) | minor. */
int moe_version(void);

/* Text of the last error returned on the calling thread ("" if none).  The
 * string is owned by the library and valid until the next call on the thread. */
const char *moe_last_error(void);

/*
 * Per-row int4 packing of a weight matrix.
 * reader.mx article §06 (C packer / Python converter); besthub.dev §06.
 *   w     [O, I] fp32, row-major (any alignment)
 *   q4    [O, (I+1)/2] uint8 out: byte j of row o holds element 2j in its low
 *         nibble and element 2j+1 in its high nibble, each stored as value+8;
 *         an odd I pads the last high nibble with 8 (value 0)
 *   scale [O] fp32 out: s = max(amax_row / 7, 1e-8)
 * value = nearest integer of w/s (IEEE division, ties to even), clamped to
 * [-8, 7].  Byte-exact with the packer described on the pages.
 * Errors: INVALID_ARG for NULL pointers, SHAPE for O < 0, I < 0 or O*I >= 2^62.
 */
int moe_pack_int4(const float *w, uint8_t *q4, float *scale, int64_t O, int64_t I,
                  cudaStream_t stream);

/*
 * Per-row int8 weights (the int8-weight expert format).
 * reader.mx article §05 (quantize_rows with bits = 8) and §12 (fmt 1:
 * matmul_q_idot, int8 weights x int8 activations).
 *   w     [O, I] fp32, row-major (any alignment)
 *   q8    [O, I] int8 out, natural order
 *   scale [O] fp32 out: s = max(amax_row / 127, 1e-8)
 * value = nearest integer of w/s (IEEE division, ties to even), clamped to
 * [-128, 127].  Byte-exact with the quantiser described on the pages.
 * Errors: INVALID_ARG for NULL pointers, SHAPE for O < 0, I < 0 or O*I >= 2^62.
 */
int moe_pack_int8(const float *w, int8_t *q8, float *scale, int64_t O, int64_t I, cudaStream_t stream);

/*
 * The checkpoint converter's step: an FP8 weight matrix to the packed int4
 * layout.  reader.mx article §02 (checkpoint config: fmt e4m3,
 * weight_block_size [128, 128]) and §06 (FP8 block-scale decoding, then the
 * per-row int4 packer); besthub.dev §06.
 *   w8        [O, I] uint8 FP8 E4M3 codes, row-major ("fn" variant: sign,
 *             4 exponent bits with bias 7, 3 mantissa bits, no infinities)
 *   scale_inv [ceil(O/128), ceil(I/128)] fp32, row-major: the factor of the
 *             128 x 128 block that holds element (o, i)
 *   q4, scale as moe_pack_int4 (outputs)
 * Computes w = e4m3(w8[o, i]) * scale_inv[o/128][i/128] (one fp32 product)
 * and packs w exactly as moe_pack_int4 does: byte-exact with packing the
 * dequantised fp32 matrix, without ever forming it (one read of w8, one write
 * of q4).  Fastest when I % 16 == 0, I <= 8192, w8 16-byte and q4 8-byte
 * aligned; any shape and alignment is accepted.  The NaN codes (0x7F, 0xFF)
 * are outside the contract.
 * Errors: INVALID_ARG for NULL pointers, SHAPE for O < 0, I < 0 or O*I >= 2^62.
 */
int moe_fp8_block_to_int4(const uint8_t *w8, const float *scale_inv, uint8_t *q4, float *scale, int64_t O,
                          int64_t I, cudaStream_t stream);

/*
 * Per-token int8 activation quantiser.
 * reader.mx article §12 (qrow_i8); besthub.dev §12.
 *   x  [n_tokens, D] fp32 row-major;  xq [n_tokens, D] int8 out (natural
 *   element order);  sx [n_tokens] fp32 out.
 * s = max(amax_row / 127, 1e-12); inv = 1/s; xq = nearest integer of x*inv
 * (ties to even).  Bit-exact with the quantiser described on the pages.
 * Errors: INVALID_ARG for NULL pointers, SHAPE for n_tokens < 0 or D < 1.
 */
int moe_quant_act_int8(const float *x, int8_t *xq, float *sx, int n_tokens, int D,
                       cudaStream_t stream);

/*
 * Sigmoid router with correction bias and greedy top-K.
 * reader.mx article §11 (sigmoid(logit)+bias selects, the weight is the plain
 * sigmoid); §02 config (scoring_func sigmoid, routed_scaling_factor 2.5).
 *   x    [n_tokens, D] fp32 (the fp32 post-norm activations, not int8)
 *   Wr   [E, D] fp32 router weight, out-major;  bias [E] fp32
 *   idx  [n_tokens, K] int32 out, in selection order (descending
 *        sigmoid(logit)+bias; an exact tie goes to the lower expert index)
 *   w    [n_tokens, K] fp32 out: sigmoid(logit[idx]) * routed_scale (not
 *        renormalised)
 * Logits are accumulated in fp32 (order differs from a sequential loop by
 * rounding only).  1 <= K <= 16, K <= E <= 512, D % 4 == 0, x and Wr 16-byte
 * aligned.  Errors: INVALID_ARG, SHAPE.
 */
int moe_router_topk(const float *x, const float *Wr, const float *bias, int n_tokens, int D,
                    int E, int K, float routed_scale, int32_t *idx, float *w,
                    cudaStream_t stream);

/* Layer description (host struct, copied by create). */
typedef struct {
    int D;              /* hidden size (6144 for GLM-5.2); D % 32 == 0, D <= 8192 */
    int I;              /* expert intermediate size (2048); I % 32 == 0, I <= 8192 */
    int E;              /* routed experts (256); 1 <= E <= 512 */
    int K;              /* experts per token (8); 1 <= K <= min(E, 16) */
    int n_shared;       /* 0 or 1 always-on shared experts, same I as routed */
    float routed_scale; /* routed_scaling_factor (2.5) */
    int max_tokens;     /* largest n_tokens any forward will pass; >= 1 */
    float top_p;        /* adaptive expert top-p (aimsg.uk article, --topp; reader.mx
                         * article §11 runs the union over each token's first keff
                         * selections).  In (0, 1): each token keeps the shortest
                         * prefix of its K selections, in selection order, whose
                         * weights reach top_p times the sum of all K (fp32 sums in
                         * order, at least one), with unchanged weights; the others
                         * are dropped (no expert read, no term in the sum; in
                         * moe_layer_debug their idx is -1 and w 0).  0 (or any value
                         * outside (0, 1)): plain top-K.  NaN: INVALID_ARG. */
    int weight_bits;    /* expert weight width: 4 (packed int4, moe_pack_int4; 0 also
                         * means 4) or 8 (per-row int8, moe_pack_int8: reader.mx
                         * article §05 quantize_rows, §12 int8 x int8 dot).  int8
                         * layers run the row-per-warp expert kernels at every batch
                         * size (neither the single decode kernel nor the tensor-core
                         * GEMMs). */
} MoeLayerDesc;

/* One expert's packed weights (device pointers, as moe_pack_int4 writes them):
 * gate_q/up_q [I, D/2] uint8, gate_s/up_s [I] fp32, down_q [D, I/2] uint8,
 * down_s [D] fp32.  Every pointer 16-byte aligned.  With weight_bits 8 (as
 * moe_pack_int8 writes them): gate_q/up_q [I, D] int8, down_q [D, I] int8. */
typedef struct {
    const uint8_t *gate_q, *up_q, *down_q;
    const float *gate_s, *up_s, *down_s;
} MoeExpertW;

/*
 * Create a layer handle.
 *   desc     host: layer sizes;  Wr [E, D] fp32, bias [E] fp32 (device)
 *   experts  host array of E + n_shared entries; entry E is the shared expert
 *   handle_out host: receives the handle
 * Ownership: Wr, bias and every expert buffer stay owned by the caller and
 * must outlive the handle (they are borrowed, never copied or freed).  The
 * handle owns a device workspace sized for desc->max_tokens (about
 * max_tokens * (K+1) * (4*I + 4*D) bytes plus small tables) and a device copy
 * of the expert pointer table.  Uses the current CUDA device.
 * Errors: INVALID_ARG, SHAPE, NOMEM, CUDA.
 */
int moe_layer_create(const MoeLayerDesc *desc, const float *Wr, const float *bias,
                     const MoeExpertW *experts, void **handle_out);

/* Release a handle and its workspace (synchronises the device first).
 * NULL is accepted.  Errors: CUDA. */
int moe_layer_destroy(void *handle);

/*
 * One routed-MoE layer forward.
 * reader.mx article §11 and §12; besthub.dev §11, §12.
 *   x   [n_tokens, D] fp32;  out [n_tokens, D] fp32 out (may not alias x)
 * out[t] = sum_k w[t,k] * y_k(t) + y_shared(t), summed in slot order, where
 * y_e(t) = down_e( hq ) * scales, h = silu(gate_e(xq)) * up_e(xq) requantised
 * per row to int8, and every dot product is an exact int32 accumulation of
 * int4 weights with int8 activations; scales are applied as
 * ((float)acc * s_act) * s_row.  The workspace makes one handle usable by one
 * stream at a time.  0 <= n_tokens <= max_tokens.  The launch sequence has no
 * host synchronisation and may be captured in a CUDA graph.
 * Errors: INVALID_ARG, SHAPE, CUDA.
 */
int moe_layer_forward(void *handle, const float *x, int n_tokens, float *out,
                      cudaStream_t stream);

/*
 * The same layer forward on host buffers (the pages' engine takes its
 * activations from host memory; the pages have no separate entry point for
 * it): enqueues on `stream`, in this order, the copy of x to the handle's
 * device staging rows, moe_layer_forward, and the copy of the result back to
 * out; returns before they finish (synchronise the stream before reading
 * out).
 *   x_host   host [n_tokens, D] fp32;  out_host host [n_tokens, D] fp32 out
 *   Page-locked host memory lets the copies run asynchronously; with
 *   pageable memory CUDA performs them synchronously.  At decode sizes
 *   (n_tokens <= 16) a page-locked, device-addressable, 16-byte aligned
 *   out_host receives the output rows directly from the kernel's stores, and
 *   no copy back is enqueued.  The staging rows are part of the handle (one
 *   forward at a time per handle, as for moe_layer_forward);
 *   0 <= n_tokens <= max_tokens.
 * Errors: INVALID_ARG, SHAPE, CUDA.
 */
int moe_layer_forward_host(void *handle, const float *x_host, int n_tokens, float *out_host,
                           cudaStream_t stream);

/*
 * Residual MoE block of a layer stack: x <- x + MoE(RMSNorm(x)).
 * reader.mx article §04 (rmsnorm: mean of squares in double, r = 1/sqrtf(ms/D
 * + eps), x*r*w; layer order norm -> MoE -> residual add).
 *   x_inout [n_tokens, D] fp32, updated in place;  norm_w [D] fp32;  eps > 0.
 * Errors: INVALID_ARG, SHAPE, CUDA.
 */
int moe_block_forward(void *handle, float *x_inout, const float *norm_w, float eps,
                      int n_tokens, cudaStream_t stream);

/* Intermediates of one forward, for parity checks.  Every pointer is a device
 * pointer and may be NULL (not written).  S = K + n_shared; slot s < K is the
 * s-th selected expert, slot K the shared expert. */
typedef struct {
    int32_t *idx;      /* [T, K] */
    float *w;          /* [T, K] */
    int8_t *xq;        /* [T, D] natural order */
    float *sx;         /* [T] */
    int32_t *gate_acc; /* [T, S, I] int32 gate dot products */
    int32_t *up_acc;   /* [T, S, I] */
    int8_t *hq;        /* [T, S, I] requantised h, natural order */
    float *sh;         /* [T, S] */
    int32_t *down_acc; /* [T, S, D] */
    int32_t *union_experts; /* [E + 1] routed union (ascending id) then the shared id E */
    int32_t *n_union;  /* [1] entries written to union_experts */
} MoeDebugOut;

/*
 * Same as moe_layer_forward and also writes the requested intermediates.
 * `out` may be NULL.  Errors: as moe_layer_forward.
 */
int moe_layer_debug(void *handle, const float *x, int n_tokens, float *out,
                    const MoeDebugOut *dbg_host, cudaStream_t stream);

/*
 * Synchronise `stream`, then read and clear the handle's device error word
 * (set by a kernel that met an input outside the contract, e.g. a token with
 * no finite selection score, or a wait of the persistent decode kernel that
 * ran out of time, flag value 16; the handle's arrival counters are then cleared).  *status_out (host) receives 0 or the flag bits.
 * Returns MOE_OK, or MOE_ERR_DEVICE when a flag was set.
 */
int moe_layer_device_status(void *handle, cudaStream_t stream, int *status_out);

/* Kernel identifiers for moe_layer_set_probe. */
#define MOE_PROBE_NONE 0
#define MOE_PROBE_GATE_UP 1
#define MOE_PROBE_DOWN 2
#define MOE_PROBE_ROUTER 3

/*
 * Timing probe: while set, every forward records `begin` on its stream just
 * before the kernel `which` and `end` just after it (as external event-record
 * nodes under stream capture).  which = MOE_PROBE_NONE clears it.  When a
 * decode-sized batch runs as the single persistent kernel (see
 * MOE_OPT_DECODE_SINGLE_KERNEL) every probe id brackets that kernel.  The
 * events are owned by the caller.  Errors: INVALID_ARG.
 */
int moe_layer_set_probe(void *handle, int which, cudaEvent_t begin, cudaEvent_t end);

/* Options of a handle (moe_layer_set_option / moe_layer_get_option). */
/* 1 (default): batches of 1..16 tokens run the whole layer as one persistent
 * kernel (cooperative launch, every CTA resident; its phases hand over through
 * arrival counters with bounded waits); 0: as a sequence of four kernels
 * (router + quantiser + union, gate/up, down, ordered reduce).  Both give
 * bit-identical outputs.  The single kernel needs cooperative launch support,
 * I <= 2048 and D <= 8192; otherwise the four-kernel sequence runs. */
#define MOE_OPT_DECODE_SINGLE_KERNEL 1
/* read-only: 1 when the single-kernel path can run for this handle */
#define MOE_OPT_DECODE_SINGLE_KERNEL_AVAILABLE 2
/* 1 (default): batches of more than 16 tokens run their expert GEMMs on the
 * tcgen05 tensor cores (kind::f16 with the int4 / int8 values carried exactly,
 * fp32 accumulation, which is exact for these sizes; the activation tiles
 * arrive by TMA from f16 operand rows the library writes once per batch); 0:
 * on the legacy integer MMA (mma.sync s8 x u8).  Both give bit-identical
 * int32 dot products.  Needs D % 256 == 0 and I % 128 == 0. */
#define MOE_OPT_TCGEN05_GEMM 3
/* read-only: 1 when the tcgen05 expert GEMMs can run for this handle (tile-
 * aligned sizes, max_tokens > 16, and the TMA tensor maps of their activation
 * operand encoded at create); otherwise batches above 16 tokens run on the
 * legacy integer MMA whatever MOE_OPT_TCGEN05_GEMM says. */
#define MOE_OPT_TCGEN05_GEMM_AVAILABLE 5
/* 1 (default): the tcgen05 GEMMs bring the packed weight rows in by TMA,
 * through tensor maps of every expert's gate, up and down rows that the
 * handle encodes at create (3 x 128 bytes per expert, device memory owned by
 * the handle); 0: the converter threads load them into registers.  Both give
 * bit-identical results.  Reading it returns 0 when the maps could not be
 * made (e.g. a weight row not 16-byte aligned): the register loads then run. */
#define MOE_OPT_TCGEN05_TMA_WEIGHTS 6
/* Test hook of the failure path, 0 (default) or 1: with 1 the persistent
 * decode kernel's grid barrier (after gate/up) waits for one arrival more
 * than there are CTAs, so that bounded wait runs out (one second) and the
 * launch sets the flag value 16 in the error word, which moe_layer_device_status
 * reports (clearing the handle's counters); the kernel then runs to its end
 * and its output is still the full result.  Used by the tests to exercise
 * time-out detection without a GPU fault. */
#define MOE_OPT_DECODE_TEST_WAIT_TIMEOUT 4

/*
 * Set / read a handle option (host).  Not part of the pages' interface: these
 * select between two equivalent launch plans of the same computation (or
 * turn on the test hook above).
 * Errors: INVALID_ARG (bad handle, unknown option, value out of range).
 */
int moe_layer_set_option(void *handle, int option, int value);
int moe_layer_get_option(void *handle, int option, int *value_out);

/*
 * Phase trace of the persistent decode kernel (a tracing aid; the pages have
 * no counterpart).  While set, every launch of that kernel writes, for CTA b,
 * 10 %globaltimer stamps (ns) to stamps_dev[10*b .. 10*b+9] as long as
 * 10*(b+1) <= n_stamps: kernel start, router/quantiser roles done, quantised
 * tokens in, shared expert gate/up done, all logits in, top-K + union done,
 * routed gate/up done, gate/up barrier passed, down rows done, end.
 * stamps_dev: device, 8-byte aligned, owned by the caller; NULL / 0 clears.
 * Errors: INVALID_ARG.
 */
int moe_layer_set_trace(void *handle, uint64_t *stamps_dev, int n_stamps);

/* Bytes of device workspace a handle with this description owns (host). */
int moe_layer_workspace_bytes(const MoeLayerDesc *desc, size_t *bytes_out);

/*
 * Allocation-free variant of moe_layer_forward.  The pages have no
 * counterpart: this entry point exists for callers that must not allocate
 * device memory -- e.g. a host framework or plugin host whose allocator owns
 * every byte of the GPU, a runtime with a fixed, pre-planned memory budget, or
 * a latency-critical loop where cudaMalloc (which can synchronise the device)
 * is not allowed.  It takes no handle and calls no cudaMalloc, cudaFree or
 * other allocating routine.  It runs the same kernels with the same launch
 * plan as moe_layer_forward (the single persistent kernel up to 16 tokens,
 * the tcgen05 expert GEMMs above), so its output equals that of a handle of
 * the same layer bit for bit.
 *   desc        host: layer sizes (max_tokens is ignored)
 *   Wr, bias    device: as for moe_layer_create
 *   experts_dev DEVICE array of E + n_shared MoeExpertW (entry E = shared
 *               expert), owned by the caller, 16-byte aligned.  As for
 *               moe_layer_create, no pointer in it may be NULL and every
 *               gate_q / up_q / down_q must be 16-byte aligned; this call
 *               cannot read the device table to check that, so the caller
 *               must (the Python binding checks it before copying the table).
 *   x, out      device [n_tokens, D] fp32, 16-byte aligned, out != x
 * The workspace is one static device array of 8 MiB (every GPU that loads the
 * library holds it until the process exits); its first 256 bytes hold the
 * error word, the rest bounds the batch: a batch whose workspace
 * (moe_layer_workspace_bytes with max_tokens = n_tokens) exceeds
 * 8 MiB - 256 B is rejected with MOE_ERR_SHAPE and a message naming the
 * limit.  For the GLM-5.2 layer (D 6144, I 2048, E 256, K 8, one shared
 * expert) that is at most 18 tokens per call.
 * The first call on a device, with that device current, resolves the array's
 * device address (cudaGetSymbolAddress), reads the SM count and sets the
 * kernels' attributes for this layer shape (kept for later calls, up to 8
 * shapes per device); make that first call before any stream capture.  A
 * set-up that failed is tried again by the next call.  Every call shares the
 * one array and keeps the previous call's contents (the routing tables and
 * counters are cleared at the start of each call): calls that overlap on the
 * GPU -- on two streams, or two threads, at once -- race and must not be
 * issued.
 * Device-side flags (the same bits moe_layer_device_status reports) collect
 * in the array's error word across calls until moe_layer_static_status
 * reads and clears them.
 * Errors: INVALID_ARG, SHAPE, CUDA.
 */
int moe_layer_forward_static(const MoeLayerDesc *desc, const float *Wr, const float *bias,
                             const MoeExpertW *experts_dev, const float *x, int n_tokens, float *out,
                             cudaStream_t stream);

/*
 * Error flags of the allocation-free entry point on the current device (no
 * counterpart on the pages; it allocates nothing either).  Synchronises
 * `stream`, then reads and clears the static workspace's error word, which
 * collects the device-side flags of every moe_layer_forward_static call on
 * this device since the last read (e.g. a token with no finite selection
 * score, flag value 1; a bounded wait that ran out of time, flag value 16).
 * *status_out (host) receives 0 or the flag bits.
 * Returns MOE_OK, MOE_ERR_DEVICE when a flag was set, or INVALID_ARG / CUDA.
 */
int moe_layer_static_status(cudaStream_t stream, int *status_out);

#ifdef __cplusplus
}
#endif
#endif /* MOE_INT4_H */
