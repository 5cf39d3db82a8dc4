// kivi_api.cu -- the C ABI of libkivi (declared in include/kivi.h): argument
// validation, host-side cache bookkeeping and kernel launches.
//
// Bookkeeping follows the residual-window scheme of "4.4 KV Cache
// quantization", section 3.2 and "KIVI: A Tuning-Free Asymmetric 2bit
// Quantization for KV Cache", "The streaming complication": after the N_s
// sink tokens ("09 -- KV Cache Quantization", "Anti-patterns": kept fp16) the
// cache holds n_quant quantised tokens (a multiple of R, so key groups stay
// aligned to the first token after the sink) followed by 1..R fp16 residual
// tokens.  Appending T tokens to a state with r residual tokens makes
// n = r + T; the last ((n - 1) mod R) + 1 of them stay fp16 and the rest are
// quantised.  A full residual is therefore flushed lazily, when the next token
// arrives, which makes a prefill of T tokens identical to T single-token
// appends.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "kivi_internal.cuh"

using namespace kivi;

namespace {

// NVTX range around a C-ABI call (header-only NVTX 3: a no-op unless a
// profiler is attached), so a timeline shows which call issued which kernels.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

int64_t pairs_of(const kivi_params *p) { return (int64_t)p->batch * p->num_kv_heads; }

int check_params(const kivi_params *p)
{
    if (!p)
        return KIVI_ERR_INVALID_ARG;
    if (p->reserved != 0 || p->batch <= 0 || p->num_q_heads <= 0 || p->num_kv_heads <= 0 ||
        p->head_dim <= 0 || p->group <= 0 || p->residual <= 0 || p->capacity_tokens < 0 ||
        p->sink_tokens < 0)
        return KIVI_ERR_INVALID_ARG;
    if ((p->meta != KIVI_META_FP32 && p->meta != KIVI_META_FP16) || p->sink_tokens > kMaxSink ||
        (p->flush != KIVI_FLUSH_WINDOW && p->flush != KIVI_FLUSH_GROUP))
        return KIVI_ERR_UNSUPPORTED;
    if (p->num_q_heads % p->num_kv_heads != 0 || p->capacity_tokens % p->residual != 0)
        return KIVI_ERR_INVALID_ARG;
    if (p->bits == 8) {
        // FP8 KV: one byte per element, 32-token records, per-tensor scales
        if (p->fp8_format != KIVI_FP8_E4M3 && p->fp8_format != KIVI_FP8_E5M2)
            return KIVI_ERR_INVALID_ARG;
        if (!(p->fp8_k_scale > 0.0f) || !(p->fp8_v_scale > 0.0f) ||
            !std::isfinite(p->fp8_k_scale) || !std::isfinite(p->fp8_v_scale))
            return KIVI_ERR_INVALID_ARG;
        if (p->group != 32 || p->meta != KIVI_META_FP32)
            return KIVI_ERR_UNSUPPORTED;
    } else if (p->fp8_format != KIVI_FP8_NONE) {
        return KIVI_ERR_INVALID_ARG;
    }
    if (p->bits != 2 && p->bits != 4 && p->bits != 8)
        return KIVI_ERR_UNSUPPORTED;
    if (p->head_dim != kHeadDim)
        return KIVI_ERR_UNSUPPORTED;
    if (p->group != 16 && p->group != 32 && p->group != 64 && p->group != 128)
        return KIVI_ERR_UNSUPPORTED;
    if (p->head_dim % p->group != 0 || p->residual % p->group != 0)
        return KIVI_ERR_UNSUPPORTED;
    if (p->num_q_heads / p->num_kv_heads > kMaxGroupQ)
        return KIVI_ERR_UNSUPPORTED;
    const int64_t pairs = pairs_of(p);
    if (pairs > 65535)
        return KIVI_ERR_UNSUPPORTED;
    // largest buffer: pairs * cap * d * 4 bytes (fp32 metadata, G = 16 worst case
    // is below the fp16 residual-free code buffers) must stay far from overflow
    if (p->capacity_tokens > ((int64_t)1 << 40) / pairs)
        return KIVI_ERR_UNSUPPORTED;
    return KIVI_OK;
}

// Bytes of one key-group record: Ks, Kz (fp32 [d] each) and, per token, key
// and value code rows plus the value scale and zero point of each group.
int64_t record_bytes(const kivi_params *p)
{
    const int64_t d = p->head_dim, G = p->group, rb = d * p->bits / 8;
    if (p->bits == 8)
        return 64 * d;                      // FP8: 32 tokens of key bytes, then value bytes
    const int64_t w = p->meta == KIVI_META_FP16 ? 2 : 4;   // bytes per scale / zero point
    return 2 * w * d + G * (2 * rb + 2 * w * (d / G));
}

int fp16_rows(const kivi_params *p) { return p->sink_tokens + p->residual; }

size_t buffer_bytes(const kivi_params *p, int which)
{
    const int64_t P = pairs_of(p), cap = p->capacity_tokens, d = p->head_dim, G = p->group;
    switch (which) {
    case 0: return (size_t)(P * (cap / G) * record_bytes(p));
    case 1:
    case 2: return (size_t)(P * fp16_rows(p) * d * 2);
    default: return 0;
    }
}

const void *buffer_ptr(const kivi_cache *c, int which)
{
    switch (which) {
    case 0: return c->history;
    case 1: return c->k_fp16;
    case 2: return c->v_fp16;
    default: return nullptr;
    }
}

int check_buffers(const kivi_cache *c)
{
    for (int w = 0; w < 3; ++w) {
        const void *ptr = buffer_ptr(c, w);
        if (buffer_bytes(&c->p, w) > 0 && !ptr)
            return KIVI_ERR_INVALID_ARG;
        if (!aligned16(ptr))
            return KIVI_ERR_INVALID_ARG;
    }
    return KIVI_OK;
}

int check_cache(const kivi_cache *c)
{
    if (!c)
        return KIVI_ERR_INVALID_ARG;
    int st = check_params(&c->p);
    if (st != KIVI_OK)
        return st;
    st = check_buffers(c);
    if (st != KIVI_OK)
        return st;
    const int R = c->p.residual;
    const int64_t unit = c->p.flush == KIVI_FLUSH_GROUP ? c->p.group : R;
    if (c->reserved != 0 || c->resid_head < 0 || c->resid_head >= R ||
        (c->p.flush == KIVI_FLUSH_WINDOW && c->resid_head != 0))
        return KIVI_ERR_INVALID_ARG;
    if (c->n_quant < 0 || c->n_quant > c->p.capacity_tokens || c->n_quant % unit != 0 ||
        c->n_resid < 0 || c->n_resid > R || (c->n_quant > 0 && c->n_resid == 0) ||
        c->n_sink < 0 || c->n_sink > c->p.sink_tokens ||
        (c->n_sink < c->p.sink_tokens && c->n_quant + c->n_resid > 0))
        return KIVI_ERR_INVALID_ARG;
    return KIVI_OK;
}

int32_t max_splits(const kivi_params *p)
{
    const int64_t pairs = pairs_of(p);
    const int64_t chunks = (p->capacity_tokens + kChunk - 1) / kChunk;
    int64_t s = (kSplitBlocksCap + pairs - 1) / pairs;
    if (s > chunks)
        s = chunks;
    if (s < 1)
        s = 1;
    return (int32_t)s;
}

// Workspace: [256-byte header: status word][per-pair block counters, rounded
// up to 256 bytes][partials for S + 1 per query row: o, then m, then l].  The
// header and the counters must be zero before first use; the kernels leave
// the counters at zero again.
size_t counters_bytes(const kivi_params *p) { return ((size_t)pairs_of(p) * 4 + 255) / 256 * 256; }

size_t workspace_bytes(const kivi_params *p)
{
    const int64_t rows = (int64_t)p->batch * p->num_q_heads;
    return kWorkspaceHeader + counters_bytes(p) +
           (size_t)rows * (size_t)(max_splits(p) + 1) * (size_t)(p->head_dim + 2) * 4;
}

struct WsView {
    unsigned *status;
    unsigned *counters;
    float *m, *l, *o;
};

WsView ws_view(const kivi_cache *c, void *ws, int32_t S)
{
    const int64_t rows = (int64_t)c->p.batch * c->p.num_q_heads;
    char *base = static_cast<char *>(ws);
    WsView v;
    v.status = reinterpret_cast<unsigned *>(base);
    v.counters = reinterpret_cast<unsigned *>(base + kWorkspaceHeader);
    // o first: it starts 256-byte aligned and its rows are whole float4s
    v.o = reinterpret_cast<float *>(base + kWorkspaceHeader + counters_bytes(&c->p));
    v.m = v.o + rows * (S + 1) * c->p.head_dim;
    v.l = v.m + rows * (S + 1);
    return v;
}

// Enqueue the split kernel; with out set it also merges the partials (the
// last block of each pair), otherwise it only writes them.
int enqueue_decode(kivi_cache *c, const void *q, void *out, float softmax_scale, int32_t S,
                   void *workspace, cudaStream_t stream, int poison_first_copy = 0)
{
    if (!(softmax_scale > 0.0f) || !std::isfinite(softmax_scale))
        softmax_scale = 1.0f / std::sqrt((float)c->p.head_dim);
    const WsView w = ws_view(c, workspace, S);
    DecodeArgs a;
    a.hist = static_cast<const uint8_t *>(c->history);
    a.kr = static_cast<const __half *>(c->k_fp16);
    a.vr = static_cast<const __half *>(c->v_fp16);
    a.q = static_cast<const __half *>(q);
    a.ws_m = w.m;
    a.ws_l = w.l;
    a.ws_o = w.o;
    a.status = w.status;
    a.counters = w.counters;
    a.out = static_cast<__half *>(out);
    a.cap = c->p.capacity_tokens;
    a.n_quant = c->n_quant;
    a.n_fp16 = c->n_sink + c->n_resid;     // the sink rows, then the residual ring
    a.n_sink = c->n_sink;
    a.Ns = c->p.sink_tokens;
    a.R = c->p.residual;
    a.head = c->resid_head;
    a.rows = fp16_rows(&c->p);
    a.Hkv = c->p.num_kv_heads;
    a.g = c->p.num_q_heads / c->p.num_kv_heads;
    a.S = S;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.fp8_k_scale = c->p.fp8_k_scale;
    a.fp8_v_scale = c->p.fp8_v_scale;
    a.poison_first_copy = poison_first_copy;
    const cudaError_t e = c->p.bits == 8
        ? launch_decode_fp8(c->p.fp8_format, a, (int)pairs_of(&c->p), stream, nullptr)
        : launch_decode_partial(c->p.bits, c->p.group, c->p.meta, a, (int)pairs_of(&c->p), stream);
    if (e != cudaSuccess)
        return KIVI_ERR_CUDA;
    c->kernel_launches += 1;
    return KIVI_OK;
}

cudaError_t fp8_blocks_per_sm(const kivi_cache *c, int *per_sm)
{
    DecodeArgs dummy{};
    dummy.g = c->p.num_q_heads / c->p.num_kv_heads;
    return launch_decode_fp8(c->p.fp8_format, dummy, 0, nullptr, per_sm);
}

// Split count for a request (0 = automatic), within the workspace's
// kivi_decode_max_splits and, when fit_cap > 0, within fit_cap as well (the
// count the allocation-free entry point's fixed scratch can hold): an
// explicit request above either limit is KIVI_ERR_WORKSPACE, the automatic
// count is clamped to both.
int resolve_splits(const kivi_cache *c, int32_t requested, int32_t *out, int64_t fit_cap = 0)
{
    const int64_t chunks = (c->n_quant + kChunk - 1) / kChunk;
    const int64_t limit = chunks > 0 ? chunks : 1;
    int64_t cap = max_splits(&c->p);
    if (fit_cap > 0 && fit_cap < cap)
        cap = fit_cap;
    int64_t S;
    if (requested < 0)
        return KIVI_ERR_INVALID_ARG;
    if (requested > 0) {
        S = requested < limit ? requested : limit;
        if (S > cap)
            return KIVI_ERR_WORKSPACE;
    } else {
        // the blocks the GPU holds at once: SMs x resident blocks per SM
        int dev = 0, sms = 0, per_sm = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            (c->p.bits == 8
                 ? fp8_blocks_per_sm(c, &per_sm)
                 : decode_blocks_per_sm(c->p.bits, c->p.group, c->p.meta,
                                        c->p.num_q_heads / c->p.num_kv_heads, &per_sm)) != cudaSuccess)
            return KIVI_ERR_CUDA;
        // Every (pair, split) block is one CTA; ceil(blocks / resident)
        // waves run, and a block's time is a fixed start-up and merge cost
        // plus its chunks (a block streams at about the same rate whether or
        // not its wave is full: its copies in flight set its rate).  Take the
        // split count with the smallest waves x (overhead + chunks per block),
        // the overhead worth 12 chunks (measured on GB300: one block of the
        // 8B layer costs ~16 us fixed and ~1.4 us per 128-token chunk).
        const int64_t pairs = pairs_of(&c->p);
        const int64_t resident = (int64_t)(per_sm > 0 ? per_sm : 1) * sms;
        const int64_t smax = std::min<int64_t>(cap, limit);
        constexpr int64_t kBlockOverheadChunks = 12;
        S = 1;
        int64_t best = INT64_MAX;
        for (int64_t s = 1; s <= smax; ++s) {
            const int64_t waves = (pairs * s + resident - 1) / resident;
            const int64_t cost = waves * (kBlockOverheadChunks + (chunks + s - 1) / s);
            if (cost < best) {
                best = cost;
                S = s;
            }
        }
    }
    if (S > limit)
        S = limit;
    if (S < 1)
        S = 1;
    *out = (int32_t)S;
    return KIVI_OK;
}

int check_decode_io(const kivi_cache *c, const void *ws, size_t ws_bytes)
{
    if (!ws || !aligned16(ws))
        return KIVI_ERR_INVALID_ARG;
    if (ws_bytes < workspace_bytes(&c->p))
        return KIVI_ERR_WORKSPACE;
    if (c->n_sink + c->n_quant + c->n_resid == 0)
        return KIVI_ERR_EMPTY;
    return KIVI_OK;
}

}  // namespace

extern "C" {

int kivi_params_validate(const kivi_params *p) { return check_params(p); }

size_t kivi_cache_buffer_bytes(const kivi_params *p, int which)
{
    if (check_params(p) != KIVI_OK || which < 0 || which > 2)
        return 0;
    return buffer_bytes(p, which);
}

size_t kivi_history_record_bytes(const kivi_params *p)
{
    if (check_params(p) != KIVI_OK)
        return 0;
    return (size_t)record_bytes(p);
}

int kivi_cache_init(kivi_cache *c, const kivi_params *p, void *history, void *k_fp16,
                    void *v_fp16)
{
    if (!c)
        return KIVI_ERR_INVALID_ARG;
    int st = check_params(p);
    if (st != KIVI_OK)
        return st;
    kivi_cache t;
    std::memset(&t, 0, sizeof(t));
    t.p = *p;
    t.history = history;
    t.k_fp16 = k_fp16;
    t.v_fp16 = v_fp16;
    st = check_buffers(&t);
    if (st != KIVI_OK)
        return st;
    *c = t;
    return KIVI_OK;
}

int kivi_cache_reset(kivi_cache *c)
{
    int st = check_cache(c);
    if (st != KIVI_OK)
        return st;
    c->n_quant = 0;
    c->n_resid = 0;
    c->n_sink = 0;
    c->resid_head = 0;
    return KIVI_OK;
}

int kivi_quantize_prefill(kivi_cache *c, const void *k, const void *v, int64_t T, int layout,
                          kivi_stream_t stream)
{
    NvtxRange nvtx_range("kivi_quantize_prefill");
    int st = check_cache(c);
    if (st != KIVI_OK)
        return st;
    if (T < 0 || (layout != KIVI_LAYOUT_BHTD && layout != KIVI_LAYOUT_BTHD))
        return KIVI_ERR_INVALID_ARG;
    if (T == 0)
        return KIVI_OK;
    if (!k || !v || !aligned16(k) || !aligned16(v))
        return KIVI_ERR_INVALID_ARG;

    const kivi_params &p = c->p;
    const int R = p.residual, G = p.group, d = p.head_dim;
    // "09 -- KV Cache Quantization", "Anti-patterns": the first N_s tokens of
    // the sequence fill the fp16 sink rows and are never quantised; only the
    // tokens after them enter the residual / quantised stream.
    const int64_t take = std::min<int64_t>(T, p.sink_tokens - c->n_sink);
    const int64_t Tq = T - take;
    const int64_t n = c->n_resid + Tq;
    int64_t r_new, nq_new;
    if (p.flush == KIVI_FLUSH_GROUP) {
        // the oldest G tokens leave the window whenever it is over-full
        const int64_t f = n > R ? (n - R + G - 1) / G : 0;
        nq_new = f * G;
        r_new = n - nq_new;
    } else {
        r_new = Tq > 0 ? ((n - 1) % R) + 1 : c->n_resid;
        nq_new = Tq > 0 ? n - r_new : 0;
    }
    if (c->n_quant + nq_new > p.capacity_tokens)
        return KIVI_ERR_CAPACITY;
    if (nq_new / G > 0x7fffffff)
        return KIVI_ERR_UNSUPPORTED;

    int64_t sb, sh, stt;
    if (layout == KIVI_LAYOUT_BHTD) {
        sb = (int64_t)p.num_kv_heads * T * d;
        sh = T * d;
        stt = d;
    } else {
        sb = T * p.num_kv_heads * d;
        sh = d;
        stt = (int64_t)p.num_kv_heads * d;
    }
    const int pairs = (int)pairs_of(&p);
    const int rows = fp16_rows(&p);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint64_t launches = 0;

    auto copy_rows = [&](int64_t src_tok0, int dst_row0, int ring, int slot0, int ntok) {
        ResidArgs a;
        a.k_in = static_cast<const __half *>(k);
        a.v_in = static_cast<const __half *>(v);
        a.in_sb = sb;
        a.in_sh = sh;
        a.in_st = stt;
        a.k_res = static_cast<__half *>(c->k_fp16);
        a.v_res = static_cast<__half *>(c->v_fp16);
        a.rows = rows;
        a.Hkv = p.num_kv_heads;
        a.src_tok0 = src_tok0;
        a.dst_row0 = dst_row0;
        a.ring = ring;
        a.slot0 = slot0;
        a.ntok = ntok;
        ++launches;
        return launch_residual_copy(a, pairs, s) == cudaSuccess;
    };

    if (take > 0 && !copy_rows(0, c->n_sink, 0, 0, (int)take))
        return KIVI_ERR_CUDA;
    if (nq_new > 0) {
        QuantArgs a;
        a.k_in = static_cast<const __half *>(k);
        a.v_in = static_cast<const __half *>(v);
        a.in_sb = sb;
        a.in_sh = sh;
        a.in_st = stt;
        a.skip = take;
        a.k_res = static_cast<const __half *>(c->k_fp16);
        a.v_res = static_cast<const __half *>(c->v_fp16);
        a.rows = rows;
        a.Ns = p.sink_tokens;
        a.R = R;
        a.head = c->resid_head;
        a.n_old = c->n_resid;
        a.Hkv = p.num_kv_heads;
        a.n_quant = c->n_quant;
        a.nq_new = nq_new;
        a.cap = p.capacity_tokens;
        a.hist = static_cast<uint8_t *>(c->history);
        a.fp8_k_scale = p.fp8_k_scale;
        a.fp8_v_scale = p.fp8_v_scale;
        a.v8 = aligned32(k) && aligned32(v) && aligned32(c->k_fp16) && aligned32(c->v_fp16);
        const cudaError_t e = p.bits == 8 ? launch_quantize_fp8(p.fp8_format, a, pairs, s)
                                          : launch_quantize(p.bits, G, p.meta, a, pairs, s);
        if (e != cudaSuccess)
            return KIVI_ERR_CUDA;
        ++launches;
    }
    if (Tq > 0) {
        // The new residual is the last r_new tokens of the concatenation
        // [old residual, new tokens]; concatenation token u lives in ring
        // slot (head + u) mod R, so kept old tokens stay where they are and
        // kept new tokens go to their own slots.  The quantise kernel above
        // has already read the flushed old tokens on the same stream.
        const int64_t first = std::max<int64_t>(nq_new, c->n_resid);   // first kept new token
        const int kept_new = (int)(n - first);
        if (kept_new > 0 &&
            !copy_rows(take + (first - c->n_resid), p.sink_tokens, R,
                       (int)((c->resid_head + first) % R), kept_new))
            return KIVI_ERR_CUDA;
    }
    c->n_sink += (int32_t)take;
    c->n_quant += nq_new;
    c->n_resid = (int32_t)r_new;
    c->resid_head = (int32_t)((c->resid_head + nq_new) % R);
    c->kernel_launches += launches;
    return KIVI_OK;
}

int kivi_append_token(kivi_cache *c, const void *k_new, const void *v_new, kivi_stream_t stream)
{
    return kivi_quantize_prefill(c, k_new, v_new, 1, KIVI_LAYOUT_BHTD, stream);
}

int32_t kivi_decode_max_splits(const kivi_params *p)
{
    if (check_params(p) != KIVI_OK)
        return 0;
    return max_splits(p);
}

size_t kivi_decode_workspace_bytes(const kivi_params *p)
{
    if (check_params(p) != KIVI_OK)
        return 0;
    return workspace_bytes(p);
}

int32_t kivi_decode_num_splits(const kivi_cache *c, int32_t requested)
{
    int st = check_cache(c);
    if (st != KIVI_OK)
        return st;
    int32_t S = 0;
    st = resolve_splits(c, requested, &S);
    return st != KIVI_OK ? st : S;
}

int kivi_decode_partial(kivi_cache *c, const void *q, float softmax_scale, int32_t num_splits,
                        void *workspace, size_t ws_bytes, kivi_stream_t stream)
{
    NvtxRange nvtx_range("kivi_decode_partial");
    int st = check_cache(c);
    if (st != KIVI_OK)
        return st;
    if (!q || !aligned16(q))
        return KIVI_ERR_INVALID_ARG;
    st = check_decode_io(c, workspace, ws_bytes);
    if (st != KIVI_OK)
        return st;
    int32_t S = 0;
    st = resolve_splits(c, num_splits, &S);
    if (st != KIVI_OK)
        return st;
    return enqueue_decode(c, q, nullptr, softmax_scale, S, workspace,
                          reinterpret_cast<cudaStream_t>(stream));
}

int kivi_decode_combine(kivi_cache *c, void *out, int32_t num_splits, const void *workspace,
                        size_t ws_bytes, kivi_stream_t stream)
{
    NvtxRange nvtx_range("kivi_decode_combine");
    int st = check_cache(c);
    if (st != KIVI_OK)
        return st;
    if (!out || !aligned16(out))
        return KIVI_ERR_INVALID_ARG;
    st = check_decode_io(c, workspace, ws_bytes);
    if (st != KIVI_OK)
        return st;
    int32_t S = 0;
    st = resolve_splits(c, num_splits, &S);
    if (st != KIVI_OK)
        return st;
    const WsView w = ws_view(c, const_cast<void *>(workspace), S);
    CombineArgs a;
    a.ws_m = w.m;
    a.ws_l = w.l;
    a.ws_o = w.o;
    a.out = static_cast<__half *>(out);
    a.S = S;
    const int rows = c->p.batch * c->p.num_q_heads;
    if (launch_decode_combine(a, rows, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KIVI_ERR_CUDA;
    c->kernel_launches += 1;
    return KIVI_OK;
}

int kivi_decode_attention(kivi_cache *c, const void *q, void *out, float softmax_scale,
                          int32_t num_splits, void *workspace, size_t ws_bytes,
                          kivi_stream_t stream)
{
    NvtxRange nvtx_range("kivi_decode_attention");
    int st = check_cache(c);
    if (st != KIVI_OK)
        return st;
    if (!q || !aligned16(q))
        return KIVI_ERR_INVALID_ARG;
    if (!out || !aligned16(out))
        return KIVI_ERR_INVALID_ARG;
    int32_t S = 0;
    st = check_decode_io(c, workspace, ws_bytes);
    if (st != KIVI_OK)
        return st;
    st = resolve_splits(c, num_splits, &S);
    if (st != KIVI_OK)
        return st;
    return enqueue_decode(c, q, out, softmax_scale, S, workspace,
                          reinterpret_cast<cudaStream_t>(stream));
}

int kivi_test_decode_wait_timeout(kivi_cache *c, const void *q, void *out, void *workspace,
                                  size_t ws_bytes, kivi_stream_t stream)
{
    int st = check_cache(c);
    if (st != KIVI_OK)
        return st;
    if (c->p.bits == 8 || c->p.group < 32 || c->n_quant == 0)
        return KIVI_ERR_UNSUPPORTED;
    if (!q || !aligned16(q) || !out || !aligned16(out))
        return KIVI_ERR_INVALID_ARG;
    st = check_decode_io(c, workspace, ws_bytes);
    if (st != KIVI_OK)
        return st;
    int32_t S = 0;
    st = resolve_splits(c, 0, &S);
    if (st != KIVI_OK)
        return st;
    return enqueue_decode(c, q, out, 0.0f, S, workspace, reinterpret_cast<cudaStream_t>(stream),
                          1);
}

double kivi_kv_bytes(int64_t L, int64_t B, int64_t T, int64_t H_kv, int64_t d,
                     double bytes_per_elem)
{
    return 2.0 * (double)L * (double)B * (double)T * (double)H_kv * (double)d * bytes_per_elem;
}

const char *kivi_status_string(int status)
{
    switch (status) {
    case KIVI_OK: return "ok";
    case KIVI_ERR_INVALID_ARG: return "invalid argument";
    case KIVI_ERR_UNSUPPORTED: return "parameters not supported by this library";
    case KIVI_ERR_CAPACITY: return "quantised history would exceed capacity_tokens";
    case KIVI_ERR_WORKSPACE: return "decode workspace too small for the split count";
    case KIVI_ERR_CUDA: return "CUDA launch or runtime call failed";
    case KIVI_ERR_EMPTY: return "decode on an empty cache";
    default: return "unknown status";
    }
}

int kivi_abi_version(void) { return KIVI_ABI_VERSION; }
size_t kivi_sizeof_params(void) { return sizeof(kivi_params); }
size_t kivi_sizeof_cache(void) { return sizeof(kivi_cache); }

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free decode (kivi_decode_attention_static).
//
// Some callers cannot allocate device memory at the point where they decode:
// code that runs inside a host framework whose memory pool owns the whole
// device, or a latency-critical serving loop where cudaMalloc (which may
// synchronise the device) is not acceptable.  For them this entry point takes
// its split-K scratch from a fixed array compiled into the library instead of
// a caller-provided workspace.  The array is kStaticScratchBytes per GPU;
// every GPU that loads the library holds it until the process exits.
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;   // 8 MiB
constexpr int kStaticMaxDevices = 64;

// Host code must not pass this name to a kernel: on the host it is only a
// stand-in for the device symbol.  Its device address comes from
// cudaGetSymbolAddress in static_scratch_address below.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void *g_scratch_address[kStaticMaxDevices];

// Device address of the scratch array on the current device; looked up once
// per device, with that device current, on its first use.
int static_scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return KIVI_ERR_CUDA;
    if (dev < 0 || dev >= kStaticMaxDevices)
        return KIVI_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_address[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p)
            return KIVI_ERR_CUDA;
        g_scratch_address[dev] = p;
    }
    *out = g_scratch_address[dev];
    return KIVI_OK;
}

}  // namespace

extern "C" size_t kivi_decode_static_scratch_bytes(void) { return kStaticScratchBytes; }

extern "C" int kivi_decode_attention_static(kivi_cache *c, const void *q, void *out,
                                            float softmax_scale, int32_t num_splits,
                                            kivi_stream_t stream)
{
    NvtxRange nvtx_range("kivi_decode_attention_static");
    int st = check_cache(c);
    if (st != KIVI_OK)
        return st;
    if (!q || !aligned16(q) || !out || !aligned16(out) || num_splits < 0)
        return KIVI_ERR_INVALID_ARG;
    if (c->n_sink + c->n_quant + c->n_resid == 0)
        return KIVI_ERR_EMPTY;
    // Splits the array holds: S + 1 partials per query row after the header
    // and the counters.  Reject before touching the GPU when not even one
    // split per pair fits.
    const int64_t rows = (int64_t)c->p.batch * c->p.num_q_heads;
    const size_t fixed = kWorkspaceHeader + counters_bytes(&c->p);
    const size_t per_split = (size_t)rows * (size_t)(c->p.head_dim + 2) * 4;
    const int64_t fit = fixed >= kStaticScratchBytes
                            ? 0 : (int64_t)((kStaticScratchBytes - fixed) / per_split) - 1;
    if (fit < 1)
        return KIVI_ERR_WORKSPACE;
    int32_t S = 0;
    st = resolve_splits(c, num_splits, &S, fit);
    if (st != KIVI_OK)
        return st;
    void *ws = nullptr;
    st = static_scratch_address(&ws);
    if (st != KIVI_OK)
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The status word and the per-pair counters must start at zero; the
    // partials are fully rewritten by every call.
    if (cudaMemsetAsync(ws, 0, fixed, s) != cudaSuccess)
        return KIVI_ERR_CUDA;
    return enqueue_decode(c, q, out, softmax_scale, S, ws, s);
}

extern "C" int kivi_decode_static_status(uint32_t *out, kivi_stream_t stream)
{
    if (!out)
        return KIVI_ERR_INVALID_ARG;
    void *ws = nullptr;
    int st = static_scratch_address(&ws);
    if (st != KIVI_OK)
        return st;
    // the status word is the first 4 bytes of the array (the workspace
    // header); copying it allocates nothing
    if (cudaMemcpyAsync(out, ws, sizeof(uint32_t), cudaMemcpyDefault,
                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KIVI_ERR_CUDA;
    return KIVI_OK;
}
