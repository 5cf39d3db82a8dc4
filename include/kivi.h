/*
 * kivi.h -- C ABI of libkivi: KIVI-style asymmetric low-bit KV-cache
 * quantisation and decode attention on one GB300 GPU (sm_103a).
 *
 * What the library computes, by source page and section:
 *
 *  - Key cache quantised per channel: for each (batch, kv-head) pair, each
 *    channel of each run of G consecutive tokens gets its own scale and zero
 *    point ("4.4 KV Cache quantization", section 3.1 "Two tensors, two
 *    groupings"; "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV
 *    Cache", "Quantize along the axis that hides the outliers").
 *  - Value cache quantised per token: each run of G channels of one token gets
 *    its own scale and zero point (same sections).
 *  - Asymmetric min/max quantiser, fp32: s = max((max - min) / (2^b - 1), 1e-8),
 *    z = round(-min / s), q = clamp(round(x / s) + z, 0, 2^b - 1), rounding
 *    half to even ("KV Cache INT4 Quantization for 1M+ Token Context
 *    Windows", section 2).
 *  - b = 2 or 4 bit codes, packed four or two per byte ("KV Cache
 *    Quantization (KIVI & FP4)", section 4; the INT4 page, section 2).
 *  - The newest tokens stay in an fp16 residual window of R tokens that is
 *    quantised in one batch once it is full ("4.4 KV Cache quantization",
 *    section 3.2; "KIVI: ...", "The streaming complication").
 *  - Optionally the first N_s tokens of every sequence are never quantised
 *    ("09 -- KV Cache Quantization", "Anti-patterns": do not quantise the
 *    attention-sink tokens; preserve-first-N).
 *  - Decode attention o = softmax(q K^T * tau) V over the sink tokens, the
 *    quantised history and the fp16 residual, dequantising inside the
 *    attention kernel ("09 -- KV Cache Quantization", "Per-channel vs
 *    per-token in the actual attention kernel" -- the dequantisation must be
 *    fused into the tile loop; "4.4 KV Cache quantization", section 2,
 *    P = softmax(QK^T / sqrt d)).  Grouped query attention: query head h_q
 *    reads kv head h_q / (Hq / Hkv) ("KV Cache Quantization (KIVI & FP4)",
 *    section 1).
 *
 * Conventions for every function:
 *  - Ownership: the caller allocates and frees every device buffer (for
 *    example with PyTorch).  The library never allocates or frees device
 *    memory.  Its only global state is the fixed scratch array that
 *    kivi_decode_attention_static uses (see there); every other function
 *    works on caller memory only.
 *  - Device pointers must be 16-byte aligned, else KIVI_ERR_INVALID_ARG.
 *  - Calls are asynchronous on the given stream (NULL = legacy default
 *    stream).  The host-side bookkeeping (n_sink, n_quant, n_resid) is
 *    updated when the work is enqueued and never needs a device read-back.
 *  - Everything is validated before anything is launched; on any error the
 *    cache is left unchanged.  No function aborts or traps on the device.
 *  - A kivi_cache is not thread-safe; use one host thread per cache object.
 *
 * Layout of one cache (P = batch * num_kv_heads pairs, pair index
 * p = b * num_kv_heads + h, cap = capacity_tokens, d = head_dim, b = bits,
 * RB = d * b / 8 code bytes per token row, VG = d / G value groups per token):
 *
 *    which 0  history  the quantised tokens as key-group records: pair p's
 *                      record j (its tokens jG .. jG + G - 1) starts at byte
 *                      (p * cap / G + j) * kivi_history_record_bytes(p):
 *                        Ks[d] | Kz[d] |
 *                        G / SL sub-slices of SL = min(G, 32) tokens, each
 *                          Kc[SL][RB]  key codes, LSB first along channels
 *                          Vc[SL][RB]  value codes, LSB first along the
 *                                      stored channel order below
 *                          Vs[SL][VG] | Vz[SL][VG]
 *                      scales and zero points in fp32 (KIVI_META_FP32) or
 *                      fp16 (KIVI_META_FP16).  Record bytes = 8 d + G (2 RB +
 *                      8 VG) with fp32 -- 128 per token at 2-bit G = 32, 160
 *                      at 4-bit G = 64 -- and 4 d + G (2 RB + 4 VG) with fp16
 *                      (96 per token at 2-bit G = 32).  With bits = 8 a
 *                      record is 32 tokens: Kc[32][d] fp8 | Vc[32][d] fp8
 *                      (64 d bytes, 256 per token).
 *    which 1  k_fp16   fp16 [P][N_s + R][d]: N_s sink rows, then the R
 *                      residual slots (a ring, see kivi_cache)
 *    which 2  v_fp16   fp16 [P][N_s + R][d]
 *
 * Stored value channel order: channel c of value group j = c / G, at
 * u = c mod G, is stored at position (d/8) r + (G/8) j + e with r = u / (G/8)
 * and e = u mod (G/8), so that the runs of G/8 channels with the same r of
 * all groups sit side by side (one word per token for the decode's per-lane
 * loads).  When such a run is shorter than a byte (2-bit G = 16) the order is
 * the natural one.  The pages fix only the grouping axes and the codes per
 * byte; the record layout and this order are this library's storage format.
 *
 * Zero points are integer-valued, not clamped to the code range, and a zero
 * point of zero is stored as +0.
 */
#ifndef KIVI_H
#define KIVI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KIVI_ABI_VERSION 2

/* Same type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st *kivi_stream_t;

enum kivi_status {
    KIVI_OK = 0,
    KIVI_ERR_INVALID_ARG = -1,  /* null/misaligned pointer, bad size or state  */
    KIVI_ERR_UNSUPPORTED = -2,  /* parameters outside what the kernels support */
    KIVI_ERR_CAPACITY = -3,     /* quantised history would exceed capacity     */
    KIVI_ERR_WORKSPACE = -4,    /* decode workspace too small                  */
    KIVI_ERR_CUDA = -5,         /* a CUDA launch or runtime call failed        */
    KIVI_ERR_EMPTY = -6         /* decode on a cache holding no tokens         */
};

/* Input layouts of the fp16 K/V handed to kivi_quantize_prefill (row = token,
 * column = channel, "4.4 KV Cache quantization", section 3.1). */
enum kivi_layout {
    KIVI_LAYOUT_BHTD = 0,       /* [B][Hkv][T][d] */
    KIVI_LAYOUT_BTHD = 1        /* [B][T][Hkv][d] */
};

/* Scale / zero-point storage of the quantised history. */
enum kivi_meta {
    KIVI_META_FP32 = 0,         /* fp32 scale and integer-valued fp32 zero point */
    KIVI_META_FP16 = 1          /* fp16 scale and zero point ("09 -- KV Cache
                                   Quantization", "KIVI -- the reference paper"):
                                   s is rounded up to binary16 and kept at least
                                   2^-24 and |min| / 2048, so |z| <= 2048 is an
                                   exact binary16 integer */
};

/* Residual flush policy: what happens when a token arrives at a full window
 * of R fp16 tokens. */
enum kivi_flush {
    KIVI_FLUSH_WINDOW = 0,      /* all R tokens are quantised in one batch ("4.4 KV
                                   Cache quantization", section 3.2) */
    KIVI_FLUSH_GROUP = 1        /* only the oldest G tokens -- one key group -- are
                                   quantised ("KIVI: ...", "The streaming
                                   complication": a completed group is frozen as
                                   the window slides); the window then slides in
                                   steps of G and holds R - G + 1 .. R tokens.
                                   Values follow the same counter. */
};

/* FP8 KV ("09 -- KV Cache Quantization", "The lazy default: FP8 KV"; "4.4 KV
 * Cache quantization", section 4.2: FP8 still needs a scale): with bits = 8
 * every flushed element is stored as fp8(x / scale) -- x / scale in fp32,
 * rounded to the nearest value of the format (ties to even) and saturated to
 * its largest finite value -- with one scale per tensor for K and one for V
 * (1.0 when uncalibrated).  The window, sink and flush rules are those of the
 * integer codes. */
enum kivi_fp8_format {
    KIVI_FP8_NONE = 0,          /* bits 2 / 4: KIVI integer codes            */
    KIVI_FP8_E4M3 = 1,          /* 4 exponent bits, 3 mantissa bits, max 448  */
    KIVI_FP8_E5M2 = 2           /* 5 exponent bits, 2 mantissa bits, max 57344 */
};

/* Problem parameters.  Supported by this library:
 *   bits in {2, 4} (KIVI codes) or 8 (FP8 KV: fp8_format E4M3 or E5M2,
 *   G = 32, positive finite scales, meta KIVI_META_FP32); head_dim = 128;
 *   group G in {16, 32, 64, 128};
 *   residual R a positive multiple of G; num_q_heads a multiple of
 *   num_kv_heads with a query group Hq/Hkv of 1..8; batch * num_kv_heads
 *   <= 65535; capacity_tokens >= 0 and a multiple of R; sink_tokens 0..256
 *   (0 = plain KIVI); meta KIVI_META_FP32 or KIVI_META_FP16; flush
 *   KIVI_FLUSH_WINDOW or KIVI_FLUSH_GROUP.
 *   Anything else valid in principle returns KIVI_ERR_UNSUPPORTED; nonsense
 *   (non-positive sizes, Hq % Hkv != 0, capacity % R != 0, sink_tokens < 0)
 *   returns KIVI_ERR_INVALID_ARG. */
typedef struct kivi_params {
    int32_t bits;             /* b: 2 or 4                                     */
    int32_t group;            /* G: tokens per key group = channels per value group */
    int32_t residual;         /* R: fp16 residual window length in tokens       */
    int32_t batch;            /* B                                              */
    int32_t num_q_heads;      /* Hq                                             */
    int32_t num_kv_heads;     /* Hkv                                            */
    int32_t head_dim;         /* d                                              */
    int32_t sink_tokens;      /* N_s: first tokens of every sequence kept fp16  */
    int64_t capacity_tokens;  /* max quantised tokens per pair                  */
    int32_t meta;             /* enum kivi_meta                                 */
    int32_t flush;            /* enum kivi_flush                                */
    int32_t fp8_format;       /* enum kivi_fp8_format (bits 8 only)             */
    float fp8_k_scale;        /* bits 8: per-tensor key scale                   */
    float fp8_v_scale;        /* bits 8: per-tensor value scale                 */
    int32_t reserved;         /* must be 0                                      */
} kivi_params;

/* One layer's cache: the three caller-owned device buffers (layout above)
 * plus host-side bookkeeping.  State: n_sink sink tokens (0..N_s; below N_s
 * only while the sequence is shorter than N_s), then n_quant quantised tokens
 * (a multiple of R with KIVI_FLUSH_WINDOW, of G with KIVI_FLUSH_GROUP)
 * followed by n_resid residual tokens (1..R whenever a token follows the
 * sink).  The residual slots form a ring: the oldest residual token is in
 * slot resid_head, the i-th oldest in slot (resid_head + i) mod R (always 0
 * with KIVI_FLUSH_WINDOW).  kernel_launches counts the kernels this library
 * enqueued on behalf of the cache (informational). */
typedef struct kivi_cache {
    kivi_params p;
    void *history;
    void *k_fp16;
    void *v_fp16;
    int64_t n_quant;
    int32_t n_resid;
    int32_t n_sink;
    int32_t resid_head;
    int32_t reserved;         /* 0 */
    uint64_t kernel_launches;
} kivi_cache;

/* KIVI_OK if the parameters are supported, else the status the other calls
 * would return for them.  Host only. */
int kivi_params_validate(const kivi_params *p);

/* Bytes of buffer `which` (0..2, table above) for these parameters; 0 if the
 * parameters are not supported or `which` is out of range.  Host only. */
size_t kivi_cache_buffer_bytes(const kivi_params *p, int which);

/* Bytes of one key-group record of the history buffer; 0 if unsupported. */
size_t kivi_history_record_bytes(const kivi_params *p);

/* Bind a cache to caller-allocated buffers and set n_sink = n_quant =
 * n_resid = 0.  Buffer contents need not be initialised.  Host only; no CUDA
 * call. */
int kivi_cache_init(kivi_cache *c, const kivi_params *p, void *history, void *k_fp16,
                    void *v_fp16);

/* Forget all tokens (n_sink = n_quant = n_resid = resid_head = 0).  Host
 * only. */
int kivi_cache_reset(kivi_cache *c);

/* Append T tokens of fp16 keys and values (device pointers, layout `layout`,
 * B and Hkv as in the parameters) -- the streaming quantisation pass after a
 * prefill ("KV Cache Quantization (KIVI & FP4)", section 6).  While the sink
 * holds fewer than N_s tokens, the first new tokens fill it (kept fp16).  The
 * tokens after them follow the current residual; of those n = n_resid + T'
 * tokens the last ((n - 1) mod R) + 1 (KIVI_FLUSH_WINDOW), or the last
 * n - G ceil((n - R) / G) when n > R (KIVI_FLUSH_GROUP), stay in the fp16
 * residual and the rest are quantised (keys in groups of G tokens counted
 * from the first token after the sink, values per token) and appended to the
 * history.  T = 0 is a
 * no-op.  A call may be made on a non-empty cache (chunked prefill); the
 * result is bit-identical to feeding the same tokens one at a time through
 * kivi_append_token.
 * Errors: KIVI_ERR_CAPACITY if n_quant would exceed capacity_tokens.
 * Reads k, v and the old residual; the caller must keep k, v alive until the
 * stream reaches this work. */
int kivi_quantize_prefill(kivi_cache *c, const void *k, const void *v, int64_t T,
                          int layout, kivi_stream_t stream);

/* One decode step's token: k_new, v_new fp16 [B][Hkv][d] (device).  If the
 * residual is full (n_resid == R), its R tokens (KIVI_FLUSH_WINDOW: "once
 * enough new tokens accumulate, they are quantized in a batch", "4.4 KV Cache
 * quantization", section 3.2) or its oldest G tokens (KIVI_FLUSH_GROUP) are
 * first quantised into the history; then the token is stored in the
 * residual.  Exactly kivi_quantize_prefill with T = 1. */
int kivi_append_token(kivi_cache *c, const void *k_new, const void *v_new,
                      kivi_stream_t stream);

/* Largest split count (token-axis partitions per pair) any decode on a cache
 * with these parameters may use, and the workspace bytes that count needs:
 * a 256-byte header (a status word the kernels OR error bits into), one
 * 32-bit counter per (batch, kv-head) pair rounded up to 256 bytes, and
 * B*Hq*(max_splits + 1)*(d + 2) fp32 partials (one per split, and one more
 * that holds the fp16 rows for G = 16 and stays empty otherwise).  Zero the whole workspace once when allocating it;
 * the kernels leave the counters at zero again.  Host only; 0 for
 * unsupported parameters. */
int32_t kivi_decode_max_splits(const kivi_params *p);
size_t kivi_decode_workspace_bytes(const kivi_params *p);

/* Split count a decode on this cache's current state would use for the
 * requested count: a positive request is clamped to one split per 128
 * quantised tokens (at least 1) and must then not exceed
 * kivi_decode_max_splits (else KIVI_ERR_WORKSPACE); 0 = automatic: the
 * count with the smallest waves x (fixed cost + chunks per block), waves
 * being the (pair, split) blocks over the blocks the GPU holds at once,
 * within the same limits.  Negative status on error.  Host only apart from
 * reading the SM count and the kernel's resident blocks per SM for 0. */
int32_t kivi_decode_num_splits(const kivi_cache *c, int32_t requested);

/* Decode attention for one new query per head: q fp16 [B][Hq][d] -> out fp16
 * [B][Hq][d].  softmax_scale <= 0 selects 1/sqrt(d).  Work is split along the
 * token axis into num_splits ranges per pair (flash-decoding), one block
 * each; the fp16 rows (sink and residual) are dealt to the pair's blocks in
 * 16-token tiles (tile s, s + num_splits, ... to block s); each block
 * keeps a running max and sum and writes (m, l, unnormalised o) to the
 * workspace, and the last block of each pair to finish merges them into out
 * (one kernel launch).
 * Errors: KIVI_ERR_EMPTY on an empty cache, KIVI_ERR_WORKSPACE if ws_bytes
 * is below kivi_decode_workspace_bytes or num_splits exceeds
 * kivi_decode_max_splits.  Never changes the cache state.  Calls that share
 * one workspace must not overlap on the GPU. */
int kivi_decode_attention(kivi_cache *c, const void *q, void *out, float softmax_scale,
                          int32_t num_splits, void *workspace, size_t ws_bytes,
                          kivi_stream_t stream);

/* kivi_decode_attention in two launches: kivi_decode_partial writes the
 * S + 1 partials per query row only, kivi_decode_combine merges them into
 * out.  Both must be given the same resolved split count
 * (kivi_decode_num_splits) and the same workspace; the result equals the
 * one-launch call's. */
int kivi_decode_partial(kivi_cache *c, const void *q, float softmax_scale,
                        int32_t num_splits, void *workspace, size_t ws_bytes,
                        kivi_stream_t stream);
int kivi_decode_combine(kivi_cache *c, void *out, int32_t num_splits,
                        const void *workspace, size_t ws_bytes, kivi_stream_t stream);

/* Allocation-free variant of kivi_decode_attention, for callers that cannot
 * allocate device memory where they decode (for example code running inside
 * a host framework whose memory pool owns the device, or a latency-critical
 * loop where cudaMalloc, which may synchronise the device, is not allowed).
 * The pages have no counterpart; this is a packaging choice of the library.
 *
 * Same arguments and results as kivi_decode_attention minus the workspace:
 * the split-K scratch lives in one array of kivi_decode_static_scratch_bytes()
 * bytes (8 MiB) compiled into the library, held by every GPU that loads the
 * library until the process exits.  The call allocates nothing: no cudaMalloc,
 * cudaFree or allocating library routine.
 *  - The first call on a device looks up the array's device address with that
 *    device current (cudaGetSymbolAddress); make that first call before any
 *    stream capture on the device.
 *  - Every call on a device shares the one array.  Each call zeroes the
 *    status word and rewrites every partial it reads, but calls whose work
 *    overlaps on the GPU (other streams, or other threads) race on the array:
 *    serialise them.
 *  - Needs 256 + 4*B*Hkv (rounded up to 256) + B*Hq*(S + 1)*(d + 2)*4 bytes
 *    for S splits.  An explicit num_splits
 *    that does not fit, or a problem where even one split per pair does not
 *    fit, returns KIVI_ERR_WORKSPACE before anything is launched; with
 *    num_splits = 0 the automatic count is clamped to what fits. */
int kivi_decode_attention_static(kivi_cache *c, const void *q, void *out,
                                 float softmax_scale, int32_t num_splits,
                                 kivi_stream_t stream);
size_t kivi_decode_static_scratch_bytes(void);

/* Error bits the kernels of the last kivi_decode_attention_static call on
 * the current device set (0 = none; 1 = a bounded wait inside the decode
 * gave up and the output is not valid): the first word of the fixed scratch
 * array, copied into *out (host or device memory) on `stream`.  Read it
 * after that stream has reached the copy.  Allocates nothing.  Like the
 * decode itself it looks up the array's address on first use on a device. */
int kivi_decode_static_status(uint32_t *out, kivi_stream_t stream);

/* KV-cache bytes M_KV = 2 * L * B * T * H_kv * d * b, b in bytes per element
 * ("4.4 KV Cache quantization", section 1).  Host only. */
double kivi_kv_bytes(int64_t L, int64_t B, int64_t T, int64_t H_kv, int64_t d,
                     double bytes_per_elem);

/* Error bit of the decode status word (the first word of a workspace or of
 * the fixed scratch array): a bounded wait of a decode kernel on its copies
 * gave up, so that call's output is not valid.  The word is sticky: the
 * kernels only OR bits into it. */
#define KIVI_STATUS_WAIT_TIMEOUT 1u

/* Test hook for the failure path of the decode's bounded waits: exactly
 * kivi_decode_attention with the automatic split count, except that the
 * first bulk copy of warp 0 of the block (split 0, pair 0) is armed for 16
 * bytes more than it brings.  That warp's wait therefore gives up after its
 * bound (about 2 s); the block writes empty partials for its rows, takes its
 * merge ticket and exits, every other block runs as usual, and no copy is
 * left in flight.  The call returns KIVI_OK; afterwards the status word
 * holds KIVI_STATUS_WAIT_TIMEOUT, the rows of pair 0 are not valid, every
 * other row equals kivi_decode_attention's with the same split count, and
 * the context stays usable.  KIVI_ERR_UNSUPPORTED unless the cache uses the
 * tensor-core decode (b in {2, 4}, G >= 32) and holds quantised tokens. */
int kivi_test_decode_wait_timeout(kivi_cache *c, const void *q, void *out,
                                  void *workspace, size_t ws_bytes, kivi_stream_t stream);

/* Static description of a status code. */
const char *kivi_status_string(int status);

/* ABI self-description, so that bindings can check their struct mirrors. */
int kivi_abi_version(void);
size_t kivi_sizeof_params(void);
size_t kivi_sizeof_cache(void);

#ifdef __cplusplus
}
#endif
#endif /* KIVI_H */
