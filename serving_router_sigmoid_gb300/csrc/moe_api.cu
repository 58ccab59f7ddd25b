// moe_api.cu -- the C ABI of the routed-MoE layer library: argument
// validation, the handle with its device workspace, and the launch sequence of
// one layer forward.  Every compute step runs in this library's kernels.
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <functional>
#include <mutex>
#include <new>

#include "layer_args.cuh"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t ce, const char *what) {
    return fail(MOE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(ce), cudaGetErrorName(ce));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr uint32_t kMagic = 0x4d6f4534u;  // handle tag

struct Handle {
    uint32_t magic;
    int device;
    MoeLayerDesc d;
    int S;
    const float *Wr, *bias;
    moe::DevExpert *experts;  // device table [E + n_shared]
    // workspace
    void *ws;
    size_t ws_bytes;
    int8_t *xq;
    float *sx;
    int32_t *xsum;
    float *logits;
    int32_t *idx;
    float *wts;
    int32_t *rows;
    moe::RouteMeta *meta;
    float *h;
    uint32_t *hamax;
    float *part;
    int8_t *hq;
    uint16_t *xf;  // f16 operand rows of the tcgen05 GEMMs
    moe::UmmaMaps maps;  // their TMA tensor maps
    bool maps_ok;
    CUtensorMap *wmaps;  // device [3 (E + n_shared)]: TMA maps of the packed expert rows, or null
    bool tma_weights;    // MOE_OPT_TCGEN05_TMA_WEIGHTS
    int32_t *hsum;
    float *shq;
    int32_t *dn_cnt;
    moe::DecodeState *dstate;
    float *dlog;
    unsigned long long *dsel;
    float *dh;  // [2][S, I] one-token h hand-over of the decode kernel (own allocation; null: grid barrier)
    int32_t *err;
    float *xnorm;  // [Tmax, D] RMSNorm output of moe_block_forward; input staging of moe_layer_forward_host
    float *xout;   // [Tmax, D] output staging of moe_layer_forward_host (own allocation)
    int nb_gu, rpi_gu, nb_dn, rpi_dn;
    int grid_gu[4], grid_dn[4];
    int num_sms;
    bool stream_ok;  // shapes and alignment the streaming kernels cover
    bool single_kernel;  // decode batches run the persistent single-kernel layer
    bool tcgen05_gemm;   // larger batches run the tcgen05 expert GEMMs
    int test_wait_extra;  // MOE_OPT_DECODE_TEST_WAIT_TIMEOUT
    int wbits;            // expert weight width: 4 or 8
    int dec_grid[moe::kSmallT + 1];  // its grid per token count (0: not available)
    int probe_which;
    cudaEvent_t probe_begin, probe_end;
    unsigned long long *trace;  // phase stamps of the persistent decode kernel
    int trace_n;
};

constexpr int kRpiGu = 16;  // gate/up rows per item: 2 per warp
constexpr int kRpiDn = 32;  // down rows per item: 4 per warp

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace layout; returns the total and fills offsets when h != nullptr.
size_t layout(const MoeLayerDesc &d, Handle *h) {
    const size_t T = (size_t)d.max_tokens, S = (size_t)d.K + d.n_shared;
    const size_t D = d.D, I = d.I, E = d.E, K = d.K;
    const size_t nb_dn = (D + 15) / 16;  // arrival counters: enough for 16-row tiles
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    const size_t o_xq = take(T * D);
    const size_t o_sx = take(4 * T);
    const size_t o_xsum = take(4 * T);
    const size_t o_logits =
        take(4 * moe::router_splits((long long)T) * (T > (size_t)moe::kSmallT ? T : (size_t)moe::kSmallT) * E);
    const size_t o_idx = take(4 * T * K);
    const size_t o_wts = take(4 * T * K);
    const size_t o_rows = take(4 * T * S);
    const size_t o_meta = take(sizeof(moe::RouteMeta));
    const size_t o_h = take(4 * T * S * I);
    const size_t o_hamax = take(4 * T * S);
    const size_t o_part = take(4 * T * S * D);
    const size_t o_hq = take(T * S * I);
    // the tcgen05 GEMMs' f16 operand rows: only batches above the decode sizes use them
    const size_t o_xf = take(T > (size_t)moe::kSmallT ? 2 * T * S * (D > I ? D : I) : 0);
    const size_t o_hsum = take(4 * T * S);
    const size_t o_shq = take(4 * T * S);
    const size_t o_cnt = take(4 * nb_dn);
    const size_t o_sync = take(sizeof(moe::DecodeState));
    const size_t o_dlog = take(2 * 4 * moe::kSmallT * E);
    const size_t o_dsel = take(2 * 8 * moe::kSmallT * K);
    const size_t o_err = take(4);
    const size_t o_xn = take(4 * T * D);
    if (h) {
        char *b = static_cast<char *>(h->ws);
        h->xq = reinterpret_cast<int8_t *>(b + o_xq);
        h->sx = reinterpret_cast<float *>(b + o_sx);
        h->xsum = reinterpret_cast<int32_t *>(b + o_xsum);
        h->logits = reinterpret_cast<float *>(b + o_logits);
        h->idx = reinterpret_cast<int32_t *>(b + o_idx);
        h->wts = reinterpret_cast<float *>(b + o_wts);
        h->rows = reinterpret_cast<int32_t *>(b + o_rows);
        h->meta = reinterpret_cast<moe::RouteMeta *>(b + o_meta);
        h->h = reinterpret_cast<float *>(b + o_h);
        h->hamax = reinterpret_cast<uint32_t *>(b + o_hamax);
        h->part = reinterpret_cast<float *>(b + o_part);
        h->hq = reinterpret_cast<int8_t *>(b + o_hq);
        h->xf = reinterpret_cast<uint16_t *>(b + o_xf);
        h->hsum = reinterpret_cast<int32_t *>(b + o_hsum);
        h->shq = reinterpret_cast<float *>(b + o_shq);
        h->dn_cnt = reinterpret_cast<int32_t *>(b + o_cnt);
        h->dstate = reinterpret_cast<moe::DecodeState *>(b + o_sync);
        h->dlog = reinterpret_cast<float *>(b + o_dlog);
        h->dsel = reinterpret_cast<unsigned long long *>(b + o_dsel);
        h->err = reinterpret_cast<int32_t *>(b + o_err);
        h->xnorm = reinterpret_cast<float *>(b + o_xn);
    }
    return off;
}

int check_desc(const MoeLayerDesc *d) {
    if (!d) return fail(MOE_ERR_INVALID_ARG, "desc is NULL");
    if (d->D < 32 || d->D > moe::kMaxDim || d->D % 32)
        return fail(MOE_ERR_SHAPE, "D=%d: need 32 <= D <= %d and D %% 32 == 0", d->D, moe::kMaxDim);
    if (d->I < 32 || d->I > moe::kMaxDim || d->I % 32)
        return fail(MOE_ERR_SHAPE, "I=%d: need 32 <= I <= %d and I %% 32 == 0", d->I, moe::kMaxDim);
    if (d->E < 1 || d->E > moe::kMaxE) return fail(MOE_ERR_SHAPE, "E=%d: need 1 <= E <= %d", d->E, moe::kMaxE);
    if (d->K < 1 || d->K > moe::kMaxK || d->K > d->E)
        return fail(MOE_ERR_SHAPE, "K=%d: need 1 <= K <= min(E, %d)", d->K, moe::kMaxK);
    if (d->n_shared < 0 || d->n_shared > 1) return fail(MOE_ERR_SHAPE, "n_shared=%d: need 0 or 1", d->n_shared);
    if (d->max_tokens < 1 || d->max_tokens > (1 << 20))
        return fail(MOE_ERR_SHAPE, "max_tokens=%d: need 1 <= max_tokens <= 2^20", d->max_tokens);
    if (!(d->routed_scale == d->routed_scale)) return fail(MOE_ERR_INVALID_ARG, "routed_scale is NaN");
    if (!(d->top_p == d->top_p)) return fail(MOE_ERR_INVALID_ARG, "top_p is NaN");
    if (d->weight_bits != 0 && d->weight_bits != 4 && d->weight_bits != 8)
        return fail(MOE_ERR_SHAPE, "weight_bits=%d: need 4 (or 0) or 8", d->weight_bits);
    return MOE_OK;
}

Handle *as_handle(void *p) {
    Handle *h = static_cast<Handle *>(p);
    if (!h || h->magic != kMagic) return nullptr;
    return h;
}

cudaError_t record(cudaEvent_t ev, cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    cudaError_t ce = cudaStreamIsCapturing(s, &st);
    if (ce != cudaSuccess) return ce;
    if (st == cudaStreamCaptureStatusActive) return cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
    return cudaEventRecord(ev, s);
}

// The state the persistent decode kernel expects at launch (and restores at
// its end): zero counters and max|h| words, empty logit and selection slots.
cudaError_t reset_decode_state(const Handle *h, cudaStream_t s) {
    cudaError_t ce = cudaMemsetAsync(h->dstate, 0, sizeof(moe::DecodeState), s);
    if (ce == cudaSuccess) ce = cudaMemsetAsync(h->dlog, 0xFF, 2 * 4 * moe::kSmallT * (size_t)h->d.E, s);
    if (ce == cudaSuccess) ce = cudaMemsetAsync(h->dsel, 0xFF, 2 * 8 * moe::kSmallT * (size_t)h->d.K, s);
    if (ce == cudaSuccess && h->dh) ce = cudaMemsetAsync(h->dh, 0xFF, 2 * 4 * (size_t)h->S * h->d.I, s);
    return ce;
}

// Grids of the persistent decode kernel for T = 1..kSmallT (0 where it
// cannot run: unsupported shape or no cooperative launch).
cudaError_t prepare_decode(Handle *h) {
    moe::LayerArgs a;
    std::memset(&a, 0, sizeof a);
    a.D = h->d.D; a.I = h->d.I; a.E = h->d.E; a.K = h->d.K; a.S = h->S; a.n_shared = h->d.n_shared;
    h->dec_grid[0] = 0;
    for (int T = 1; T <= moe::kSmallT; ++T) {
        a.T = T;
        h->dec_grid[T] = 0;
        if (T > h->d.max_tokens || h->wbits != 4) continue;  // the single kernel streams int4 rows only
        cudaError_t ce = moe::decode_grid(a, h->num_sms, &h->dec_grid[T]);
        if (ce != cudaSuccess) return ce;
    }
    h->single_kernel = true;
    h->tcgen05_gemm = true;
    return cudaSuccess;
}

// The launch sequence of one forward.  x is the layer input (already
// normalised for a block), out/resid as in LayerArgs.
int run_layer(Handle *h, const float *x, int T, float *out, const float *resid, const moe::DebugPtrs &dbg,
              cudaStream_t s) {
    moe::LayerArgs a;
    std::memset(&a, 0, sizeof a);
    a.D = h->d.D; a.I = h->d.I; a.E = h->d.E; a.K = h->d.K; a.S = h->S; a.n_shared = h->d.n_shared; a.T = T;
    a.routed_scale = h->d.routed_scale;
    a.top_p = h->d.top_p;
    a.wbits = h->wbits;
    a.x = x; a.Wr = h->Wr; a.bias = h->bias; a.experts = h->experts;
    a.xq = h->xq; a.sx = h->sx; a.xsum = h->xsum; a.logits = h->logits; a.idx = h->idx; a.wts = h->wts;
    a.rows = h->rows; a.meta = h->meta; a.h = h->h; a.hamax = h->hamax; a.part = h->part; a.dn_cnt = h->dn_cnt;
    a.hq = h->hq; a.hsum = h->hsum; a.shq = h->shq; a.dstate = h->dstate;
    a.dlog = h->dlog; a.dsel = h->dsel; a.dh = h->dh;
    a.trace = h->trace; a.trace_n = h->trace_n;
    a.out = out; a.resid = resid; a.err = h->err;
    a.nb_gu = h->nb_gu; a.rpi_gu = h->rpi_gu; a.nb_dn = h->nb_dn; a.rpi_dn = h->rpi_dn;
    a.wait_extra = h->test_wait_extra;
    a.wmaps = h->tma_weights ? h->wmaps : nullptr;
    a.dbg = dbg;
    const int mch = T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8;
    const int mi = moe::mch_index(mch);
    const bool small = T <= moe::kSmallT;
    cudaError_t ce;

    // decode-sized batches: the whole layer as one persistent kernel (every
    // probe id brackets it)
    if (small && h->single_kernel && h->dec_grid[T] > 0) {
        if (h->probe_which != MOE_PROBE_NONE && (ce = record(h->probe_begin, s)) != cudaSuccess)
            return cuda_fail(ce, "probe record");
        if ((ce = moe::launch_decode_layer(a, h->dec_grid[T], s)) != cudaSuccess)
            return cuda_fail(ce, "decode layer launch");
        if (h->probe_which != MOE_PROBE_NONE && (ce = record(h->probe_end, s)) != cudaSuccess)
            return cuda_fail(ce, "probe record");
        return MOE_OK;
    }

    if (h->probe_which == MOE_PROBE_ROUTER && (ce = record(h->probe_begin, s)) != cudaSuccess)
        return cuda_fail(ce, "probe record");
    if (small) {
        if ((ce = moe::launch_router_small(a, s)) != cudaSuccess) return cuda_fail(ce, "router_small launch");
    } else {
        if ((ce = moe::launch_quant_perm(a, s)) != cudaSuccess) return cuda_fail(ce, "quant launch");
        if ((ce = moe::launch_router_gemm(x, h->Wr, h->bias, T, a.D, a.E, a.K, a.routed_scale, a.top_p, h->logits,
                                          h->idx, h->wts, h->err, s)) != cudaSuccess)
            return cuda_fail(ce, "router_tile launch");
        if ((ce = moe::launch_permute(a, s)) != cudaSuccess) return cuda_fail(ce, "permute launch");
    }
    if (h->probe_which == MOE_PROBE_ROUTER && (ce = record(h->probe_end, s)) != cudaSuccess)
        return cuda_fail(ce, "probe record");

    // larger batches with tile-aligned shapes: tensor-core grouped GEMMs
    // (tcgen05 with f16-exact operands; the legacy integer MMA on request)
    // (int8 weights run the row-per-warp kernels at every batch size)
    const bool umma = h->wbits == 4 && h->tcgen05_gemm && h->maps_ok && moe::umma_supported(a.D, a.I);
    if (!small && h->wbits == 4 && (umma || moe::grouped_supported(a.D, a.I))) {
        if (umma) {
            a.xf = h->xf;
            if ((ce = moe::launch_act_rows_f16(a, s)) != cudaSuccess) return cuda_fail(ce, "operand rows launch");
        }
        if (h->probe_which == MOE_PROBE_GATE_UP && (ce = record(h->probe_begin, s)) != cudaSuccess)
            return cuda_fail(ce, "probe record");
        ce = umma ? moe::launch_umma_gateup(a, h->maps, h->num_sms, s) : moe::launch_grouped_gateup(a, h->num_sms, s);
        if (ce != cudaSuccess) return cuda_fail(ce, "gateup launch");
        if (h->probe_which == MOE_PROBE_GATE_UP && (ce = record(h->probe_end, s)) != cudaSuccess)
            return cuda_fail(ce, "probe record");
        if (h->probe_which == MOE_PROBE_DOWN && (ce = record(h->probe_begin, s)) != cudaSuccess)
            return cuda_fail(ce, "probe record");
        if ((ce = moe::launch_requant_h(a, s)) != cudaSuccess) return cuda_fail(ce, "requant launch");
        ce = umma ? moe::launch_umma_down(a, h->maps, h->num_sms, s) : moe::launch_grouped_down(a, h->num_sms, s);
        if (ce != cudaSuccess) return cuda_fail(ce, "down launch");
        if ((ce = moe::launch_reduce(a, s)) != cudaSuccess) return cuda_fail(ce, "reduce launch");
        if (h->probe_which == MOE_PROBE_DOWN && (ce = record(h->probe_end, s)) != cudaSuccess)
            return cuda_fail(ce, "probe record");
        return MOE_OK;
    }

    // decode-sized batches stream the experts through register-pipelined
    // warps; shapes the grouped tiles do not cover use the row-per-warp dp4a
    // kernels
    const bool stream = small && h->stream_ok;
    if (h->probe_which == MOE_PROBE_GATE_UP && (ce = record(h->probe_begin, s)) != cudaSuccess)
        return cuda_fail(ce, "probe record");
    ce = stream ? moe::launch_gateup_stream(a, h->num_sms, s) : moe::launch_gateup(a, mch, h->grid_gu[mi], s);
    if (ce != cudaSuccess) return cuda_fail(ce, "gateup launch");
    if (h->probe_which == MOE_PROBE_GATE_UP && (ce = record(h->probe_end, s)) != cudaSuccess)
        return cuda_fail(ce, "probe record");

    if (h->probe_which == MOE_PROBE_DOWN && (ce = record(h->probe_begin, s)) != cudaSuccess)
        return cuda_fail(ce, "probe record");
    ce = stream ? moe::launch_down_stream(a, h->num_sms, s) : moe::launch_down(a, mch, h->grid_dn[mi], small, s);
    if (ce != cudaSuccess) return cuda_fail(ce, "down launch");
    if ((stream || !small) && (ce = moe::launch_reduce(a, s)) != cudaSuccess) return cuda_fail(ce, "reduce launch");
    if (h->probe_which == MOE_PROBE_DOWN && (ce = record(h->probe_end, s)) != cudaSuccess)
        return cuda_fail(ce, "probe record");
    return MOE_OK;
}

int check_forward(Handle *h, const float *x, int T, const float *out) {
    if (!h) return fail(MOE_ERR_INVALID_ARG, "invalid handle");
    if (T < 0 || T > h->d.max_tokens)
        return fail(MOE_ERR_SHAPE, "n_tokens=%d outside [0, max_tokens=%d]", T, h->d.max_tokens);
    if (T == 0) return MOE_OK;
    if (!x || !out) return fail(MOE_ERR_INVALID_ARG, "x or out is NULL");
    if (!aligned16(x) || !aligned16(out)) return fail(MOE_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
    int dev = -1;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaGetDevice");
    if (dev != h->device) return fail(MOE_ERR_INVALID_ARG, "current device %d is not the handle's device %d", dev, h->device);
    return MOE_OK;
}

}  // namespace

extern "C" {

int moe_version(void) { return (1 << 16) | 0; }

const char *moe_last_error(void) { return g_err; }

int moe_pack_int4(const float *w, uint8_t *q4, float *scale, int64_t O, int64_t I, cudaStream_t stream) {
    if (O < 0 || I < 0) return fail(MOE_ERR_SHAPE, "O=%lld I=%lld must be >= 0", (long long)O, (long long)I);
    if (O == 0) return MOE_OK;
    if (I > 0 && O > ((int64_t)1 << 62) / I) return fail(MOE_ERR_SHAPE, "O*I too large");
    if (!w || !q4 || !scale) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
    cudaError_t ce = moe::launch_pack_int4(w, q4, scale, O, I, stream);
    return ce == cudaSuccess ? MOE_OK : cuda_fail(ce, "pack_int4 launch");
}

int moe_fp8_block_to_int4(const uint8_t *w8, const float *scale_inv, uint8_t *q4, float *scale, int64_t O,
                          int64_t I, cudaStream_t stream) {
    if (O < 0 || I < 0) return fail(MOE_ERR_SHAPE, "O=%lld I=%lld must be >= 0", (long long)O, (long long)I);
    if (O == 0) return MOE_OK;
    if (I > 0 && O > ((int64_t)1 << 62) / I) return fail(MOE_ERR_SHAPE, "O*I too large");
    if (!w8 || !scale_inv || !q4 || !scale) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
    cudaError_t ce = moe::launch_fp8_to_int4(w8, scale_inv, q4, scale, O, I, stream);
    return ce == cudaSuccess ? MOE_OK : cuda_fail(ce, "fp8_to_int4 launch");
}

int moe_pack_int8(const float *w, int8_t *q8, float *scale, int64_t O, int64_t I, cudaStream_t stream) {
    if (O < 0 || I < 0) return fail(MOE_ERR_SHAPE, "O=%lld I=%lld must be >= 0", (long long)O, (long long)I);
    if (O == 0) return MOE_OK;
    if (I > 0 && O > ((int64_t)1 << 62) / I) return fail(MOE_ERR_SHAPE, "O*I too large");
    if (!w || !q8 || !scale) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
    cudaError_t ce = moe::launch_pack_int8(w, q8, scale, O, I, stream);
    return ce == cudaSuccess ? MOE_OK : cuda_fail(ce, "pack_int8 launch");
}

int moe_quant_act_int8(const float *x, int8_t *xq, float *sx, int n_tokens, int D, cudaStream_t stream) {
    if (n_tokens < 0 || D < 1) return fail(MOE_ERR_SHAPE, "n_tokens=%d D=%d", n_tokens, D);
    if (n_tokens == 0) return MOE_OK;
    if (!x || !xq || !sx) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
    cudaError_t ce = moe::launch_quant_natural(x, xq, sx, n_tokens, D, stream);
    return ce == cudaSuccess ? MOE_OK : cuda_fail(ce, "quant launch");
}

int moe_router_topk(const float *x, const float *Wr, const float *bias, int n_tokens, int D, int E, int K,
                    float routed_scale, int32_t *idx, float *w, cudaStream_t stream) {
    if (n_tokens < 0 || D < 4 || D % 4 || E < 1 || E > moe::kMaxE || K < 1 || K > moe::kMaxK || K > E)
        return fail(MOE_ERR_SHAPE, "n_tokens=%d D=%d E=%d K=%d", n_tokens, D, E, K);
    if (n_tokens == 0) return MOE_OK;
    if (!x || !Wr || !bias || !idx || !w) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(x) || !aligned16(Wr)) return fail(MOE_ERR_INVALID_ARG, "x and Wr must be 16-byte aligned");
    cudaError_t ce = moe::launch_router_tile(x, Wr, bias, n_tokens, D, E, K, routed_scale, idx, w, nullptr, stream);
    return ce == cudaSuccess ? MOE_OK : cuda_fail(ce, "router launch");
}

int moe_layer_workspace_bytes(const MoeLayerDesc *desc, size_t *bytes_out) {
    int rc = check_desc(desc);
    if (rc) return rc;
    if (!bytes_out) return fail(MOE_ERR_INVALID_ARG, "bytes_out is NULL");
    *bytes_out = layout(*desc, nullptr);
    return MOE_OK;
}

int moe_layer_create(const MoeLayerDesc *desc, const float *Wr, const float *bias, const MoeExpertW *experts,
                     void **handle_out) {
    int rc = check_desc(desc);
    if (rc) return rc;
    if (!Wr || !bias || !experts || !handle_out) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(Wr)) return fail(MOE_ERR_INVALID_ARG, "Wr must be 16-byte aligned");
    const int ne = desc->E + desc->n_shared;
    for (int e = 0; e < ne; ++e) {
        const MoeExpertW &x = experts[e];
        if (!x.gate_q || !x.up_q || !x.down_q || !x.gate_s || !x.up_s || !x.down_s)
            return fail(MOE_ERR_INVALID_ARG, "expert %d has a NULL pointer", e);
        if (!aligned16(x.gate_q) || !aligned16(x.up_q) || !aligned16(x.down_q))
            return fail(MOE_ERR_INVALID_ARG, "expert %d weights must be 16-byte aligned", e);
    }
    *handle_out = nullptr;
    Handle *h = new (std::nothrow) Handle();
    if (!h) return fail(MOE_ERR_NOMEM, "host allocation failed");
    std::memset(h, 0, sizeof *h);
    h->d = *desc;
    h->S = desc->K + desc->n_shared;
    h->Wr = Wr;
    h->bias = bias;
    h->rpi_gu = kRpiGu;
    h->nb_gu = (desc->I + kRpiGu - 1) / kRpiGu;
    h->rpi_dn = kRpiDn;
    h->nb_dn = (desc->D + kRpiDn - 1) / kRpiDn;
    cudaError_t ce;
    int nsm = 0;
    if ((ce = cudaGetDevice(&h->device)) != cudaSuccess ||
        (ce = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, h->device)) != cudaSuccess) {
        delete h;
        return cuda_fail(ce, "device query");
    }
    h->num_sms = nsm;
    h->wbits = desc->weight_bits == 8 ? 8 : 4;
    h->stream_ok = h->wbits == 4 && moe::stream_supported(desc->D, desc->I);
    if ((ce = h->wbits == 8 ? moe::prepare_expert_kernels8(desc->D, desc->I, nsm, h->grid_gu, h->grid_dn)
                            : moe::prepare_expert_kernels(desc->D, desc->I, nsm, h->grid_gu, h->grid_dn)) !=
            cudaSuccess ||
        (ce = prepare_decode(h)) != cudaSuccess) {
        delete h;
        return cuda_fail(ce, "kernel attributes");
    }
    h->ws_bytes = layout(*desc, nullptr);
    if ((ce = cudaMalloc(&h->ws, h->ws_bytes)) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return fail(MOE_ERR_NOMEM, "workspace of %zu bytes: %s", h->ws_bytes, cudaGetErrorString(ce));
    }
    layout(*desc, h);
    h->maps_ok = h->wbits == 4 && moe::umma_supported(desc->D, desc->I) &&
                 moe::umma_encode_maps(h->xf, desc->max_tokens * h->S, desc->D, desc->I, &h->maps) == cudaSuccess;
    if ((ce = cudaMalloc(&h->experts, sizeof(moe::DevExpert) * ne)) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(h->ws);
        delete h;
        return fail(MOE_ERR_NOMEM, "expert table: %s", cudaGetErrorString(ce));
    }
    moe::DevExpert *tab = new (std::nothrow) moe::DevExpert[ne];
    if (!tab) {
        cudaFree(h->ws);
        cudaFree(h->experts);
        delete h;
        return fail(MOE_ERR_NOMEM, "host allocation failed");
    }
    for (int e = 0; e < ne; ++e)
        tab[e] = moe::DevExpert{experts[e].gate_q, experts[e].up_q, experts[e].down_q,
                                experts[e].gate_s, experts[e].up_s, experts[e].down_s};
    ce = cudaMemcpy(h->experts, tab, sizeof(moe::DevExpert) * ne, cudaMemcpyHostToDevice);
    // TMA maps of the packed rows for the tcgen05 GEMMs (without them, or if
    // a row start is not 16-byte aligned, those GEMMs load the rows into
    // registers instead)
    if (ce == cudaSuccess && h->maps_ok) {
        CUtensorMap *hm = new (std::nothrow) CUtensorMap[3 * (size_t)ne];
        if (hm && moe::umma_encode_weight_maps(tab, ne, desc->D, desc->I, hm) == cudaSuccess &&
            cudaMalloc(&h->wmaps, sizeof(CUtensorMap) * 3 * (size_t)ne) == cudaSuccess) {
            ce = cudaMemcpy(h->wmaps, hm, sizeof(CUtensorMap) * 3 * (size_t)ne, cudaMemcpyHostToDevice);
        } else {
            cudaGetLastError();
            h->wmaps = nullptr;
        }
        delete[] hm;
    }
    delete[] tab;
    if (ce == cudaSuccess) ce = cudaMemset(h->ws, 0, h->ws_bytes);
    // the one-token h hand-over (its own allocation, so that the workspace
    // size, which the allocation-free entry point shares, does not change)
    if (ce == cudaSuccess) ce = cudaMalloc(&h->dh, 2 * 4 * (size_t)h->S * desc->I);
    if (ce == cudaSuccess) ce = cudaMalloc(&h->xout, 4 * (size_t)desc->max_tokens * desc->D);
    if (ce == cudaSuccess) ce = reset_decode_state(h, 0);
    if (ce == cudaSuccess) ce = cudaDeviceSynchronize();
    if (ce != cudaSuccess) {
        cudaFree(h->ws);
        cudaFree(h->experts);
        cudaFree(h->wmaps);
        cudaFree(h->dh);
        cudaFree(h->xout);
        delete h;
        return cuda_fail(ce, "handle initialisation");
    }
    h->tma_weights = true;
    h->magic = kMagic;
    *handle_out = h;
    return MOE_OK;
}

int moe_layer_destroy(void *handle) {
    if (!handle) return MOE_OK;
    Handle *h = as_handle(handle);
    if (!h) return fail(MOE_ERR_INVALID_ARG, "invalid handle");
    cudaError_t ce = cudaDeviceSynchronize();
    cudaFree(h->ws);
    cudaFree(h->experts);
    cudaFree(h->wmaps);
    cudaFree(h->dh);
    cudaFree(h->xout);
    h->magic = 0;
    delete h;
    return ce == cudaSuccess ? MOE_OK : cuda_fail(ce, "destroy");
}

int moe_layer_forward(void *handle, const float *x, int n_tokens, float *out, cudaStream_t stream) {
    Handle *h = as_handle(handle);
    int rc = check_forward(h, x, n_tokens, out);
    if (rc || n_tokens == 0) return rc;
    if (x == out) return fail(MOE_ERR_INVALID_ARG, "out may not alias x");
    return run_layer(h, x, n_tokens, out, nullptr, moe::DebugPtrs{}, stream);
}

int moe_layer_forward_host(void *handle, const float *x_host, int n_tokens, float *out_host,
                           cudaStream_t stream) {
    Handle *h = as_handle(handle);
    if (!h) return fail(MOE_ERR_INVALID_ARG, "invalid handle");
    if (n_tokens < 0 || n_tokens > h->d.max_tokens)
        return fail(MOE_ERR_SHAPE, "n_tokens=%d outside [0, max_tokens=%d]", n_tokens, h->d.max_tokens);
    if (n_tokens == 0) return MOE_OK;
    if (!x_host || !out_host) return fail(MOE_ERR_INVALID_ARG, "x_host or out_host is NULL");
    if (!h->xout) return fail(MOE_ERR_INVALID_ARG, "handle has no staging rows");
    int rc = check_forward(h, h->xnorm, n_tokens, h->xout);
    if (rc) return rc;
    const size_t bytes = sizeof(float) * (size_t)n_tokens * h->d.D;
    // decode sizes: a page-locked out_host that the device can address takes
    // the output rows straight from the kernel's stores (no copy after the
    // forward); otherwise the rows are staged in the handle and copied back
    float *out_dev = nullptr;
    if (n_tokens <= moe::kSmallT) {
        cudaPointerAttributes pa;
        if (cudaPointerGetAttributes(&pa, out_host) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
            pa.devicePointer && aligned16(pa.devicePointer))
            out_dev = static_cast<float *>(pa.devicePointer);
        else
            (void)cudaGetLastError();  // a pageable pointer is not an error here
    }
    cudaError_t ce = cudaMemcpyAsync(h->xnorm, x_host, bytes, cudaMemcpyHostToDevice, stream);
    if (ce != cudaSuccess) return cuda_fail(ce, "copy of x to the device");
    rc = run_layer(h, h->xnorm, n_tokens, out_dev ? out_dev : h->xout, nullptr, moe::DebugPtrs{}, stream);
    if (rc || out_dev) return rc;
    ce = cudaMemcpyAsync(out_host, h->xout, bytes, cudaMemcpyDeviceToHost, stream);
    if (ce != cudaSuccess) return cuda_fail(ce, "copy of out to the host");
    return MOE_OK;
}

int moe_block_forward(void *handle, float *x_inout, const float *norm_w, float eps, int n_tokens,
                      cudaStream_t stream) {
    Handle *h = as_handle(handle);
    int rc = check_forward(h, x_inout, n_tokens, x_inout);
    if (rc || n_tokens == 0) return rc;
    if (!norm_w) return fail(MOE_ERR_INVALID_ARG, "norm_w is NULL");
    if (!(eps >= 0.f)) return fail(MOE_ERR_INVALID_ARG, "eps must be >= 0");
    cudaError_t ce = moe::launch_rmsnorm(x_inout, norm_w, eps, h->xnorm, n_tokens, h->d.D, stream);
    if (ce != cudaSuccess) return cuda_fail(ce, "rmsnorm launch");
    return run_layer(h, h->xnorm, n_tokens, x_inout, x_inout, moe::DebugPtrs{}, stream);
}

int moe_layer_debug(void *handle, const float *x, int n_tokens, float *out, const MoeDebugOut *dbg,
                    cudaStream_t stream) {
    Handle *h = as_handle(handle);
    if (!h) return fail(MOE_ERR_INVALID_ARG, "invalid handle");
    if (!dbg) return fail(MOE_ERR_INVALID_ARG, "dbg is NULL");
    float *o = out ? out : h->xnorm;  // scratch output when the caller does not want it
    int rc = check_forward(h, x, n_tokens, o);
    if (rc || n_tokens == 0) return rc;
    moe::DebugPtrs p{dbg->xq, dbg->gate_acc, dbg->up_acc, dbg->hq, dbg->sh, dbg->down_acc};
    rc = run_layer(h, x, n_tokens, o, nullptr, p, stream);
    if (rc) return rc;
    cudaError_t ce = cudaSuccess;
    const size_t TK = (size_t)n_tokens * h->d.K;
    if (dbg->idx && ce == cudaSuccess) ce = cudaMemcpyAsync(dbg->idx, h->idx, 4 * TK, cudaMemcpyDeviceToDevice, stream);
    if (dbg->w && ce == cudaSuccess) ce = cudaMemcpyAsync(dbg->w, h->wts, 4 * TK, cudaMemcpyDeviceToDevice, stream);
    if (dbg->sx && ce == cudaSuccess)
        ce = cudaMemcpyAsync(dbg->sx, h->sx, 4 * (size_t)n_tokens, cudaMemcpyDeviceToDevice, stream);
    if (dbg->union_experts && ce == cudaSuccess)
        ce = cudaMemcpyAsync(dbg->union_experts, h->meta->uexp, 4 * (size_t)(h->d.E + 1), cudaMemcpyDeviceToDevice,
                             stream);
    if (dbg->n_union && ce == cudaSuccess)
        ce = cudaMemcpyAsync(dbg->n_union, &h->meta->n_union, 4, cudaMemcpyDeviceToDevice, stream);
    return ce == cudaSuccess ? MOE_OK : cuda_fail(ce, "debug copies");
}

int moe_layer_device_status(void *handle, cudaStream_t stream, int *status_out) {
    Handle *h = as_handle(handle);
    if (!h || !status_out) return fail(MOE_ERR_INVALID_ARG, "invalid handle or NULL status_out");
    int v = 0;
    cudaError_t ce = cudaStreamSynchronize(stream);
    if (ce == cudaSuccess) ce = cudaMemcpy(&v, h->err, 4, cudaMemcpyDeviceToHost);
    if (ce == cudaSuccess) ce = cudaMemset(h->err, 0, 4);
    // a wait that ran out of time may leave the decode kernel's state behind
    if (ce == cudaSuccess && (v & moe::kErrSyncTimeout)) ce = reset_decode_state(h, stream);
    if (ce == cudaSuccess && (v & moe::kErrSyncTimeout)) ce = cudaStreamSynchronize(stream);
    if (ce != cudaSuccess) return cuda_fail(ce, "device status");
    *status_out = v;
    return v ? fail(MOE_ERR_DEVICE, "device error flags 0x%x", v) : MOE_OK;
}

int moe_layer_set_option(void *handle, int option, int value) {
    Handle *h = as_handle(handle);
    if (!h) return fail(MOE_ERR_INVALID_ARG, "invalid handle");
    switch (option) {
        case MOE_OPT_DECODE_SINGLE_KERNEL:
            if (value != 0 && value != 1) return fail(MOE_ERR_INVALID_ARG, "value %d: need 0 or 1", value);
            h->single_kernel = value != 0;
            return MOE_OK;
        case MOE_OPT_TCGEN05_GEMM:
            if (value != 0 && value != 1) return fail(MOE_ERR_INVALID_ARG, "value %d: need 0 or 1", value);
            h->tcgen05_gemm = value != 0;
            return MOE_OK;
        case MOE_OPT_DECODE_TEST_WAIT_TIMEOUT:
            if (value != 0 && value != 1) return fail(MOE_ERR_INVALID_ARG, "value %d: need 0 or 1", value);
            h->test_wait_extra = value;
            return MOE_OK;
        case MOE_OPT_TCGEN05_TMA_WEIGHTS:
            if (value != 0 && value != 1) return fail(MOE_ERR_INVALID_ARG, "value %d: need 0 or 1", value);
            h->tma_weights = value != 0;
            return MOE_OK;
        default:
            return fail(MOE_ERR_INVALID_ARG, "unknown option %d", option);
    }
}

int moe_layer_get_option(void *handle, int option, int *value_out) {
    Handle *h = as_handle(handle);
    if (!h || !value_out) return fail(MOE_ERR_INVALID_ARG, "invalid handle or NULL value_out");
    switch (option) {
        case MOE_OPT_DECODE_SINGLE_KERNEL:
            *value_out = h->single_kernel ? 1 : 0;
            return MOE_OK;
        case MOE_OPT_TCGEN05_GEMM:
            *value_out = h->tcgen05_gemm ? 1 : 0;
            return MOE_OK;
        case MOE_OPT_DECODE_TEST_WAIT_TIMEOUT:
            *value_out = h->test_wait_extra;
            return MOE_OK;
        case MOE_OPT_TCGEN05_GEMM_AVAILABLE:
            *value_out = h->maps_ok && moe::umma_supported(h->d.D, h->d.I) ? 1 : 0;
            return MOE_OK;
        case MOE_OPT_TCGEN05_TMA_WEIGHTS:
            *value_out = h->tma_weights && h->wmaps ? 1 : 0;
            return MOE_OK;
        case MOE_OPT_DECODE_SINGLE_KERNEL_AVAILABLE: {
            int any = 0;
            for (int T = 1; T <= moe::kSmallT; ++T) any |= h->dec_grid[T] > 0;
            *value_out = any;
            return MOE_OK;
        }
        default:
            return fail(MOE_ERR_INVALID_ARG, "unknown option %d", option);
    }
}

int moe_layer_set_trace(void *handle, uint64_t *stamps_dev, int n_stamps) {
    Handle *h = as_handle(handle);
    if (!h) return fail(MOE_ERR_INVALID_ARG, "invalid handle");
    if (n_stamps < 0 || (n_stamps > 0 && !stamps_dev)) return fail(MOE_ERR_INVALID_ARG, "bad trace buffer");
    if (stamps_dev && (reinterpret_cast<uintptr_t>(stamps_dev) & 7u))
        return fail(MOE_ERR_INVALID_ARG, "trace buffer must be 8-byte aligned");
    h->trace = n_stamps > 0 ? reinterpret_cast<unsigned long long *>(stamps_dev) : nullptr;
    h->trace_n = n_stamps;
    return MOE_OK;
}

int moe_layer_set_probe(void *handle, int which, cudaEvent_t begin, cudaEvent_t end) {
    Handle *h = as_handle(handle);
    if (!h) return fail(MOE_ERR_INVALID_ARG, "invalid handle");
    if (which < MOE_PROBE_NONE || which > MOE_PROBE_ROUTER) return fail(MOE_ERR_INVALID_ARG, "bad probe id %d", which);
    if (which != MOE_PROBE_NONE && (!begin || !end)) return fail(MOE_ERR_INVALID_ARG, "NULL event");
    h->probe_which = which;
    h->probe_begin = begin;
    h->probe_end = end;
    return MOE_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free forward.  The workspace of this entry point is a file-scope
// device array instead of cudaMalloc'ed memory; every GPU that loads the
// library holds it until the process exits.  Host code cannot pass the
// array's name to a kernel (on the host it only stands for the symbol), so
// its device address is looked up once per device with cudaGetSymbolAddress.
// The first 256 bytes hold the error word, at a fixed place so that
// moe_layer_static_status finds it whatever the last call's sizes were; the
// layer workspace follows.
namespace {

constexpr size_t kStaticScratchBytes = (size_t)8 << 20;  // 8 MiB
constexpr size_t kStaticErrBytes = 256;                  // error word (+ padding)
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// The caller's device table of MoeExpertW is read by the kernels as
// moe::DevExpert: both must have the same layout.
static_assert(sizeof(MoeExpertW) == sizeof(moe::DevExpert), "expert table layout");
static_assert(offsetof(MoeExpertW, gate_q) == offsetof(moe::DevExpert, gq), "expert table layout");
static_assert(offsetof(MoeExpertW, up_q) == offsetof(moe::DevExpert, uq), "expert table layout");
static_assert(offsetof(MoeExpertW, down_q) == offsetof(moe::DevExpert, dq), "expert table layout");
static_assert(offsetof(MoeExpertW, gate_s) == offsetof(moe::DevExpert, gs), "expert table layout");
static_assert(offsetof(MoeExpertW, up_s) == offsetof(moe::DevExpert, us), "expert table layout");
static_assert(offsetof(MoeExpertW, down_s) == offsetof(moe::DevExpert, ds), "expert table layout");

constexpr int kMaxDevices = 64;
constexpr int kStaticPlans = 8;  // launch plans kept per device (distinct layer shapes)

// Grids of one layer shape, as moe_layer_create computes them.
struct StaticPlan {
    bool used;
    int D, I, E, K, n_shared, wbits;
    int grid_gu[4], grid_dn[4];
    int dec_grid[moe::kSmallT + 1];
};

struct StaticDeviceState {
    bool ready;     // scratch address and SM count resolved
    void *scratch;  // device address of g_static_scratch on this device
    int num_sms;
    int next;       // plan slot replaced next when all are used
    StaticPlan plans[kStaticPlans];
};
std::mutex g_static_mu;
StaticDeviceState g_static_dev[kMaxDevices];

// With the device current and g_static_mu held: resolve the scratch address
// and the SM count once per device.  A failure is not remembered, so a later
// call tries again.  No allocation happens here.
cudaError_t static_ready(StaticDeviceState &st, int dev) {
    if (st.ready) return cudaSuccess;
    void *p = nullptr;
    int nsm = 0;
    cudaError_t ce = cudaGetSymbolAddress(&p, g_static_scratch);
    if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (ce != cudaSuccess) {
        cudaGetLastError();
        return ce;
    }
    st.scratch = p;
    st.num_sms = nsm;
    st.ready = true;
    return cudaSuccess;
}

// With g_static_mu held: the launch plan of this layer shape, computed (kernel
// attributes, occupancy) on its first use and kept for later calls.
cudaError_t static_plan(StaticDeviceState &st, const MoeLayerDesc &d, int dev, const StaticPlan **out) {
    for (int i = 0; i < kStaticPlans; ++i) {
        const StaticPlan &p = st.plans[i];
        if (p.used && p.D == d.D && p.I == d.I && p.E == d.E && p.K == d.K && p.n_shared == d.n_shared &&
            p.wbits == (d.weight_bits == 8 ? 8 : 4)) {
            *out = &p;
            return cudaSuccess;
        }
    }
    Handle tmp;
    std::memset(&tmp, 0, sizeof tmp);
    tmp.device = dev;
    tmp.d = d;
    tmp.d.max_tokens = moe::kSmallT;  // decode grids for every decode-sized batch
    tmp.S = d.K + d.n_shared;
    tmp.num_sms = st.num_sms;
    tmp.wbits = d.weight_bits == 8 ? 8 : 4;
    cudaError_t ce = tmp.wbits == 8 ? moe::prepare_expert_kernels8(d.D, d.I, st.num_sms, tmp.grid_gu, tmp.grid_dn)
                                    : moe::prepare_expert_kernels(d.D, d.I, st.num_sms, tmp.grid_gu, tmp.grid_dn);
    if (ce == cudaSuccess) ce = prepare_decode(&tmp);
    if (ce != cudaSuccess) return ce;
    StaticPlan &p = st.plans[st.next];
    st.next = (st.next + 1) % kStaticPlans;
    p.used = true;
    p.D = d.D; p.I = d.I; p.E = d.E; p.K = d.K; p.n_shared = d.n_shared; p.wbits = tmp.wbits;
    std::memcpy(p.grid_gu, tmp.grid_gu, sizeof p.grid_gu);
    std::memcpy(p.grid_dn, tmp.grid_dn, sizeof p.grid_dn);
    std::memcpy(p.dec_grid, tmp.dec_grid, sizeof p.dec_grid);
    *out = &p;
    return cudaSuccess;
}

}  // namespace

extern "C" int moe_layer_forward_static(const MoeLayerDesc *desc, const float *Wr, const float *bias,
                                        const MoeExpertW *experts_dev, const float *x, int n_tokens, float *out,
                                        cudaStream_t stream) {
    int rc = check_desc(desc);
    if (rc) return rc;
    if (n_tokens < 0) return fail(MOE_ERR_SHAPE, "n_tokens=%d must be >= 0", n_tokens);
    if (n_tokens == 0) return MOE_OK;
    MoeLayerDesc d = *desc;
    d.max_tokens = n_tokens;
    const size_t need = layout(d, nullptr);
    if (need > kStaticScratchBytes - kStaticErrBytes)
        return fail(MOE_ERR_SHAPE,
                    "n_tokens=%d needs %zu bytes of workspace; the static workspace holds %zu bytes "
                    "(use moe_layer_create/moe_layer_forward for larger batches)",
                    n_tokens, need, kStaticScratchBytes - kStaticErrBytes);
    if (!Wr || !bias || !experts_dev || !x || !out) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(Wr) || !aligned16(x) || !aligned16(out) || !aligned16(experts_dev))
        return fail(MOE_ERR_INVALID_ARG, "Wr, x, out and experts_dev must be 16-byte aligned");
    if (x == out) return fail(MOE_ERR_INVALID_ARG, "out may not alias x");
    int dev = -1;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_INVALID_ARG, "device %d out of range", dev);

    // a handle that lives on the stack and points into the static workspace
    Handle h;
    std::memset(&h, 0, sizeof h);
    {
        std::lock_guard<std::mutex> lk(g_static_mu);
        StaticDeviceState &st = g_static_dev[dev];
        if ((ce = static_ready(st, dev)) != cudaSuccess) return cuda_fail(ce, "static workspace set-up");
        const StaticPlan *plan = nullptr;
        if ((ce = static_plan(st, d, dev, &plan)) != cudaSuccess) return cuda_fail(ce, "kernel attributes");
        h.ws = static_cast<char *>(st.scratch) + kStaticErrBytes;
        h.num_sms = st.num_sms;
        std::memcpy(h.grid_gu, plan->grid_gu, sizeof h.grid_gu);
        std::memcpy(h.grid_dn, plan->grid_dn, sizeof h.grid_dn);
        std::memcpy(h.dec_grid, plan->dec_grid, sizeof h.dec_grid);
        h.err = static_cast<int32_t *>(st.scratch);
    }
    h.magic = kMagic;
    h.device = dev;
    h.d = d;
    h.S = d.K + d.n_shared;
    h.Wr = Wr;
    h.bias = bias;
    h.experts = reinterpret_cast<moe::DevExpert *>(const_cast<MoeExpertW *>(experts_dev));
    h.ws_bytes = need;
    int32_t *err = h.err;
    layout(d, &h);
    h.err = err;  // the fixed error word, not the layout's
    h.maps_ok = h.wbits == 4 && n_tokens > moe::kSmallT && moe::umma_supported(d.D, d.I) &&
                moe::umma_encode_maps(h.xf, n_tokens * (d.K + d.n_shared), d.D, d.I, &h.maps) == cudaSuccess;
    h.rpi_gu = kRpiGu;
    h.nb_gu = (d.I + kRpiGu - 1) / kRpiGu;
    h.rpi_dn = kRpiDn;
    h.nb_dn = (d.D + kRpiDn - 1) / kRpiDn;
    h.wbits = d.weight_bits == 8 ? 8 : 4;
    h.stream_ok = h.wbits == 4 && moe::stream_supported(d.D, d.I);
    h.single_kernel = true;
    h.tcgen05_gemm = true;
    // the arrival counters and routing tables must start at zero (their place
    // moves with the sizes); everything else is written before it is read.
    // The error word keeps its flags until moe_layer_static_status reads them.
    if ((ce = cudaMemsetAsync(h.meta, 0, sizeof(moe::RouteMeta), stream)) != cudaSuccess ||
        (ce = cudaMemsetAsync(h.dn_cnt, 0, 4 * (size_t)((d.D + 15) / 16), stream)) != cudaSuccess ||
        (ce = reset_decode_state(&h, stream)) != cudaSuccess)
        return cuda_fail(ce, "static workspace clear");
    return run_layer(&h, x, n_tokens, out, nullptr, moe::DebugPtrs{}, stream);
}

extern "C" int moe_layer_static_status(cudaStream_t stream, int *status_out) {
    if (!status_out) return fail(MOE_ERR_INVALID_ARG, "status_out is NULL");
    int dev = -1;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_INVALID_ARG, "device %d out of range", dev);
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_static_mu);
        StaticDeviceState &st = g_static_dev[dev];
        if ((ce = static_ready(st, dev)) != cudaSuccess) return cuda_fail(ce, "static workspace set-up");
        scratch = st.scratch;
    }
    int v = 0;
    ce = cudaStreamSynchronize(stream);
    if (ce == cudaSuccess) ce = cudaMemcpy(&v, scratch, 4, cudaMemcpyDeviceToHost);
    if (ce == cudaSuccess) ce = cudaMemsetAsync(scratch, 0, 4, stream);
    if (ce == cudaSuccess) ce = cudaStreamSynchronize(stream);
    if (ce != cudaSuccess) return cuda_fail(ce, "static status");
    *status_out = v;
    return v ? fail(MOE_ERR_DEVICE, "device error flags 0x%x", v) : MOE_OK;
}
