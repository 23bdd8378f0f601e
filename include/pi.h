/*
 * pi.h -- C ABI of the predictor-guided, neuron-aware sparse FFN for
 * single-token decode in ReLU-family LLMs (library: libpi_sparse_ffn.so).
 *
 * The method (PowerInfer summary page, gptget.net, arXiv 2312.12456; sections
 * "核心创新" core innovation and "方法详解" method detail): per decode token an
 * online activation predictor marks the FFN neurons expected to fire, and
 * neuron-aware sparse operators compute only those neurons -- the rows of the
 * up/gate projections and the matching rows of the down projection.  Hot
 * neurons, found by offline profiling ("关键结果" key results: ~26% of neurons
 * carry 80% of the firings), are stored first.  Supported activations: ReLU,
 * ReGLU and squared ReLU (PowerInfer README translation, gittoolsai.com,
 * "常见问题解答" FAQ item 2).  Weights may be fp16, fp32 or INT4 Q4_0 (same
 * README, "量化" quantization).
 *
 * Conventions for every entry point:
 *  - The caller owns every buffer.  Pointers documented "device" must be CUDA
 *    device memory (or managed memory) of the current device; "host" pointers
 *    are ordinary host memory.  The library allocates nothing and keeps no
 *    pointer after a call returns.
 *  - Device work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and is asynchronous: no entry point except
 *    pi_sync_status() waits for the GPU.  Active counts stay on the device.
 *  - Arguments are validated on the host before anything is launched; on any
 *    error nothing is enqueued and the status says why.  Conditions that only
 *    the GPU can see (an active list longer than its capacity, a neuron index
 *    out of range, a bounded device-side wait that gave up) set bits in an
 *    error word inside the workspace; pi_sync_status() reports and clears them.
 *    No kernel traps or asserts.
 *  - Layouts are row-major.  FFN matrices are neuron-major: row j of w_up,
 *    w_gate and w_down belongs to neuron j and holds d_model values (so
 *    w_down is the transpose of the usual fc2 / down_proj weight).
 *  - Activations x, y, residual are fp32 [batch][d_model].  Accumulation is
 *    fp32 throughout.
 *  - Neuron indices are positions in the storage order (after any hot-first
 *    permutation), int32, ascending.
 */
#ifndef PI_SPARSE_FFN_H
#define PI_SPARSE_FFN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PI_API __attribute__((visibility("default")))
#else
#define PI_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PI_OK = 0,
    PI_ERR_NULL = 1,      /* a required pointer is NULL                              */
    PI_ERR_SHAPE = 2,     /* a size is out of range or breaks a divisibility rule    */
    PI_ERR_DTYPE = 3,     /* unsupported storage type or type combination            */
    PI_ERR_ALIGN = 4,     /* a pointer is not aligned as documented                  */
    PI_ERR_CAPACITY = 5,  /* device: an active list exceeded its capacity            */
    PI_ERR_CUDA = 6,      /* a CUDA launch or runtime call failed                    */
    PI_ERR_TIMEOUT = 7,   /* device: a bounded wait gave up                          */
    PI_ERR_WORKSPACE = 8, /* workspace missing or smaller than required              */
    PI_ERR_ALIAS = 9,     /* an output overlaps an input it may not overlap          */
    PI_ERR_INDEX = 10     /* a neuron index out of range (device), or a host neuron
                             order that is not a permutation (pi_shard_neurons)     */
} pi_status;

typedef enum { PI_F32 = 0, PI_F16 = 1, PI_Q4_0 = 2 } pi_dtype;
typedef enum { PI_ACT_RELU = 0, PI_ACT_RELU2 = 1 } pi_act;

typedef void *pi_stream; /* cudaStream_t */

#define PI_MAX_BATCH 8
#define PI_MAX_D_MODEL 16384
#define PI_MAX_RANK 2048

/*
 * One FFN layer with its activation predictor.  All pointers are device
 * pointers owned by the caller, 16-byte aligned unless stated.
 *
 *   non-gated (gated = 0):  z_j = w_up[j].x + b_act[j],   a_j = act(z_j)
 *   gated (ReGLU, gated = 1): z_j = w_gate[j].x + b_act[j], a_j = act(z_j) * (w_up[j].x)
 *   output:                  y = sum_j a_j * w_down[j] + b_down (+ residual)
 *   act = ReLU, max(z, 0), or squared ReLU, max(z, 0)^2.
 *
 *   predictor (d -> rank, ReLU, rank -> d_ff; the pages give its purpose, not
 *   its form, and this low-rank form is the reading taken):
 *     h_k = max(p1[k].x, 0),  logit_j = p2[j].h + p_bias[j],  neuron j is
 *     predicted active when j < dense_prefix or logit_j > threshold.
 *
 * Storage:
 *   wtype PI_F32 / PI_F16: w_up, w_gate, w_down are [d_ff][d_model].
 *   wtype PI_Q4_0: each matrix is one blob of pi_q4_0_bytes(d_ff, d_model)
 *     bytes: all 4-bit codes first ([d_ff][d_model/2] bytes; in each block of 32
 *     weights, weight e < 16 is the low nibble of code byte e and weight
 *     e >= 16 the high nibble of byte e-16), then all scales
 *     ([d_ff][d_model/32] binary16).  Weight = scale * (code - 8).
 *   ptype PI_F32 / PI_F16: p1 is [rank][d_model], p2 is [d_ff][rank].
 *   b_act [d_ff], b_down [d_model], p_bias [d_ff]: fp32, 4-byte aligned, may
 *     each be NULL (= zero).  w_gate is NULL unless gated.
 * Limits: 8 <= d_model <= PI_MAX_D_MODEL and d_model % 8 == 0 (% 256 for
 *   Q4_0); 1 <= d_ff < 2^26 (< 2^23 for calls that run the predictor);
 *   8 <= rank <= PI_MAX_RANK, rank % 8 == 0 (only checked by calls that run
 *   the predictor).
 */
typedef struct pi_ffn_desc_s {
    int32_t d_model;
    int32_t d_ff;
    int32_t rank;
    int32_t gated;   /* 0 or 1 */
    int32_t act;     /* pi_act */
    int32_t wtype;   /* pi_dtype of w_up / w_gate / w_down */
    int32_t ptype;   /* pi_dtype of p1 / p2: PI_F32 or PI_F16 */
    float threshold;
    const void *w_up;
    const void *w_gate;
    const void *w_down;
    const float *b_act;
    const float *b_down;
    const void *p1;
    const void *p2;
    const float *p_bias;
    /* Optional (NULL: none): the layer the caller runs next on the same stream.
     * A scheduling hint that the current kernels do not use: asking L2 for
     * that layer's predictor P1 during this layer's sparse FFN phase was
     * measured slower on GB300 (the rows did not reach the next layer's SMs
     * faster, and the request took HBM time from this layer's tail).  The
     * library never reads *next. */
    const struct pi_ffn_desc_s *next;
    /* Always-on prefix: neurons [0, dense_prefix) of the storage order are
     * active at every step whatever the predictor says, and their rows of p2
     * and p_bias are not read by the one-kernel layer step.  With the
     * hot-first order (pi_hot_first_perm) these are the neurons an offline
     * profile found to fire most often -- the pages' hot neurons, which the
     * method keeps on the fast device (PowerInfer summary page, "方法详解"
     * method detail) -- so the predictor only decides the cold tail.
     * 0 <= dense_prefix <= d_ff; 0 = none. */
    int32_t dense_prefix;
} pi_ffn_desc;

/* Human-readable name of a status code (static string, never NULL). */
PI_API const char *pi_status_str(int32_t status);

/*
 * Bytes of workspace that pi_predict, pi_sparse_ffn, pi_ffn_layer and
 * pi_dense_ffn need for this layer shape at this batch size (0 when the
 * descriptor is invalid).  The workspace is device memory, 256-byte aligned,
 * and must be zero-filled once before its first use; after that the calls
 * keep it consistent themselves.  One workspace serves any sequence of calls
 * on the same stream for descriptors of the same d_model, d_ff, rank and a
 * batch no larger than the one it was sized for; calls that overlap in time
 * (other streams) need separate workspaces.  After a call that reported
 * PI_ERR_TIMEOUT the workspace must be zero-filled again before its next use.
 * Bytes 4..7 of the workspace (a uint32) may be set by the caller: the number
 * of polls after which a wait of one CTA on others (a grid barrier, the work
 * queue) gives up; 0, the zero-filled default, means about 4 million polls
 * (seconds).  A smaller value makes a lost wait fail faster.
 */
PI_API size_t pi_workspace_bytes(const pi_ffn_desc *desc, int32_t batch);

/* Workspace bytes for pi_compact over n mask entries (same rules as above). */
PI_API size_t pi_compact_workspace_bytes(int32_t n);

/*
 * Active-index compaction: idx[0..count) = ascending positions j < n with
 * mask[j] != 0, count = their number.  This is the step that turns a
 * predicted activity mask into the neuron list the sparse operators walk.
 *   mask  device uint8 [n] (any alignment); n >= 1.
 *   idx   device int32 [cap], 4-byte aligned; count device int32 [1].
 *   When more than cap entries are set, the first cap are written, *count =
 *   cap, and PI_ERR_CAPACITY is raised in the workspace error word.
 * Bit-exact: the result is unique.
 */
PI_API pi_status pi_compact(const uint8_t *mask, int32_t n, int32_t *idx, int32_t *count, int32_t cap,
                     void *ws, size_t ws_bytes, pi_stream stream);

/*
 * Predictor: for every token b of the batch, logit[b][j] = p2[j].h_b + p_bias[j]
 * with h_b = max(p1.x_b, 0); a neuron is active when logit > threshold for at
 * least one token of the batch (the union of the per-token masks); idx /
 * *n_active receive the compacted ascending active list as in pi_compact.
 *   x       device fp32 [batch][d_model], 1 <= batch <= PI_MAX_BATCH.
 *   logits  device fp32 [batch][d_ff] or NULL.   mask device uint8 [d_ff] or NULL.
 *   idx     device int32 [cap]; n_active device int32 [1]; cap >= 1.
 */
PI_API pi_status pi_predict(const pi_ffn_desc *desc, const float *x, int32_t batch, float *logits,
                     uint8_t *mask, int32_t *idx, int32_t *n_active, int32_t cap, void *ws,
                     size_t ws_bytes, pi_stream stream);

/*
 * Neuron-aware sparse FFN over a given active list: for each token b,
 *   y[b] = sum_{k < n} a_{b, idx[k]} * w_down[idx[k]] + b_down + residual[b],
 * where a is the layer's activation (see pi_ffn_desc).  Only the listed rows of
 * w_up / w_gate / w_down are read.  Neurons not listed contribute nothing.
 *   idx       device int32 [*n_active], ascending, each in [0, d_ff) (an index
 *             outside is skipped and raises PI_ERR_INDEX in the error word).
 *   n_active  device int32 [1], read on the device (0 <= n <= d_ff).
 *   residual  device fp32 [batch][d_model] or NULL; it may equal y.
 *   y         device fp32 [batch][d_model]; must not overlap x.
 * batch 1 runs on CUDA cores; batch 2..8 (wtype F16 or Q4_0) runs the union
 * rows through tensor cores.
 */
PI_API pi_status pi_sparse_ffn(const pi_ffn_desc *desc, const float *x, int32_t batch, const int32_t *idx,
                        const int32_t *n_active, const float *residual, float *y, void *ws,
                        size_t ws_bytes, pi_stream stream);

/*
 * One decode step of the layer: pi_predict followed by pi_sparse_ffn on the
 * predicted (union) active list, enqueued as back-to-back kernels that may
 * overlap their weight prefetch with the previous kernel.
 *   idx / n_active  device int32 [d_ff] / [1] receiving the active list, or
 *                   NULL to keep it inside the workspace.
 *   other arguments as in pi_sparse_ffn.
 * At batch 1 (for the shapes it supports) the whole step is one kernel of one
 * CTA per SM whose CTAs synchronise across the grid, so it needs all of them
 * resident at once.  If other streams or processes hold SMs long enough, its
 * bounded waits give up: PI_ERR_TIMEOUT from pi_sync_status, and y is not
 * valid.  With idx / n_active NULL the FFN rows are spread over the CTAs
 * dynamically (for d_ff up to 509 x the number of SMs; wider layers take the
 * next path); otherwise the ascending list is also written, which costs one
 * more grid-wide synchronisation.  Every predicted neuron is computed in both
 * cases.
 */
PI_API pi_status pi_ffn_layer(const pi_ffn_desc *desc, const float *x, int32_t batch, const float *residual,
                       float *y, int32_t *idx, int32_t *n_active, void *ws, size_t ws_bytes,
                       pi_stream stream);

/*
 * The next layer of a stack whose layers feed each other (one decode token
 * through consecutive FFN layers): the layer-to-layer glue of pi_rms_residual
 * and then pi_ffn_layer, fused.  Per token b,
 *   v = x_prev[b] + y_prev[b],  x[b] = v / sqrt(mean(v^2))  (0 when v = 0),
 *   y[b] = FFN of this layer at x[b] (no residual),
 * with x[b] also written out (the next glue step needs it).  For the shapes
 * where pi_ffn_layer runs one kernel at batch 1, the glue is part of that
 * kernel: every CTA rescales the whole vector itself, after the previous
 * layer's kernel has finished, so no launch sits between two layers.  Other
 * shapes run pi_rms_residual's kernel first.  The stack's input glue follows
 * the reading of "output plus residual as the next layer's input" taken for
 * the OPT-175B-shaped stack (weightless RMS rescale of the sum).
 *   x_prev, y_prev  device fp32 [batch][d_model], 16-byte aligned.
 *   x, y            device fp32 [batch][d_model]; neither may overlap x_prev
 *                   or y_prev, and y may not overlap x (PI_ERR_ALIAS).
 *   idx, n_active, ws, ws_bytes: as in pi_ffn_layer.
 */
PI_API pi_status pi_ffn_layer_chain(const pi_ffn_desc *desc, const float *x_prev, const float *y_prev, int32_t batch,
                                    float *x, float *y, int32_t *idx, int32_t *n_active, void *ws, size_t ws_bytes,
                                    pi_stream stream);

/* Dense FFN (every neuron), through the same operators; the all-active
 * special case used as a check and as the dense baseline. */
PI_API pi_status pi_dense_ffn(const pi_ffn_desc *desc, const float *x, int32_t batch, const float *residual,
                       float *y, void *ws, size_t ws_bytes, pi_stream stream);

/* Bytes of a Q4_0 blob for a [rows][cols] matrix (0 unless cols % 32 == 0). */
PI_API size_t pi_q4_0_bytes(int64_t rows, int64_t cols);

/*
 * Quantise a [rows][cols] matrix to a Q4_0 blob (layout in pi_ffn_desc).  Per
 * block of 32 weights: a = the weight of largest magnitude (the first on
 * ties); scale = binary16(a / -8) (+0 when a == 0); code = clamp(floor(w /
 * scale + 8.5), 0, 15), computed in binary32 (8 when the scale is 0).
 *   src  device, src_type PI_F32 or PI_F16, 16-byte aligned; dst device
 *        [pi_q4_0_bytes(rows, cols)], 16-byte aligned; cols % 32 == 0.
 */
PI_API pi_status pi_quantize_q4_0(const void *src, int32_t src_type, int64_t rows, int64_t cols, void *dst,
                           pi_stream stream);

/*
 * The same quantiser on the host (synchronous, needs no GPU), for offline
 * conversion of checkpoints: byte for byte what pi_quantize_q4_0 writes for
 * fp32 input.
 *   src  host fp32 [rows][cols], row-major; cols % 32 == 0 (else PI_ERR_SHAPE).
 *   dst  host buffer of pi_q4_0_bytes(rows, cols) bytes, not overlapping src
 *        (else PI_ERR_ALIAS).
 */
PI_API pi_status pi_quantize_q4_0_host(const float *src, int64_t rows, int64_t cols, void *dst);

/*
 * Offline activation profiling (PowerInfer summary, "方法详解": hot neurons
 * are found by analysing the activation distribution offline): for each of
 * the T tokens of X (device fp32 [T][d_model]), counts[j] += 1 when the
 * pre-activation feeding act() (fc1, or gate when gated) is > 0.  counts is
 * device int32 [d_ff] and is accumulated into, not cleared.
 */
PI_API pi_status pi_fire_counts(const pi_ffn_desc *desc, const float *X, int32_t T, int32_t *counts,
                         pi_stream stream);

/*
 * Hot-first neuron order from firing counts (host, synchronous): perm[p] is
 * the original neuron stored at position p -- neurons sorted by count, highest
 * first, ties in ascending neuron order.  counts and perm are host int32 [n].
 */
PI_API pi_status pi_hot_first_perm(const int32_t *counts, int32_t n, int32_t *perm);

/*
 * Row permutation: dst row i = src row perm[i], for a [rows][row_bytes] byte
 * matrix (device, non-overlapping; perm device int32 [rows] with entries in
 * [0, rows); an entry outside that range leaves its destination row
 * unwritten).  Applies a neuron order to w_up / w_gate / w_down / p2
 * (rows = d_ff) and to the per-neuron vectors b_act / p_bias (row_bytes = 4).
 * Q4_0 blobs are permuted before quantisation, or as their two sections (codes
 * rows of d_model/2 bytes, then scale rows of d_model/16 bytes) separately.
 */
PI_API pi_status pi_permute_rows(const void *src, void *dst, int64_t rows, int64_t row_bytes,
                          const int32_t *perm, pi_stream stream);

/*
 * Row gather between matrices of different heights: dst row i = src row idx[i]
 * for i < dst_rows.  src device [src_rows][row_bytes], dst device
 * [dst_rows][row_bytes], non-overlapping; idx device int32 [dst_rows], each
 * entry in [0, src_rows) (an entry outside leaves its destination row
 * unwritten).  Builds the rows of one neuron shard (pi_shard_neurons) of every
 * per-neuron array of a layer.  PI_ERR_SHAPE for a non-positive size,
 * PI_ERR_ALIGN for a misaligned idx, PI_ERR_ALIAS when src and dst overlap.
 */
PI_API pi_status pi_gather_rows(const void *src, int64_t src_rows, void *dst, int64_t dst_rows, int64_t row_bytes,
                         const int32_t *idx, pi_stream stream);

/*
 * Neuron sharding of one layer over `shards` devices (host, synchronous).
 * Neurons are independent in the sparse operator -- each one's rows of
 * w_up / w_gate / w_down, its bias, its predictor row of p2 and p_bias -- so a
 * layer splits by neuron, as the pages split one FFN between a GPU (hot
 * neurons) and a CPU (cold neurons) and add the two parts (PowerInfer README
 * translation, gittoolsai.com, "摘要" abstract and "推理" inference).  p1 is
 * replicated: every shard computes h itself.  The order (normally the
 * hot-first order of pi_hot_first_perm, so that every shard gets an equal
 * share of the frequently active neurons) is dealt round-robin: shard s gets
 * order[s], order[s + shards], ...
 * order host int32 [n], a permutation of 0..n-1 (else PI_ERR_INDEX); out host
 * int32 with room for ceil(n / shards) entries; *count receives the shard's
 * size.  Each shard runs the layer on its rows and yields a partial y; the
 * layer output is the sum of the partials (one all-reduce of batch x d_model
 * fp32 per layer), with b_down and the residual given to one shard only.
 * PI_ERR_SHAPE unless 1 <= shards <= n and 0 <= shard < shards.
 */
PI_API pi_status pi_shard_neurons(const int32_t *order, int32_t n, int32_t shards, int32_t shard, int32_t *out,
                           int32_t *count);

/*
 * Layer-to-layer glue of a stack of FFN layers whose output feeds the next
 * layer's input: v = x + y, x_next = v / sqrt(mean(v^2)) per token (0 when
 * v = 0).  x, y, x_next device fp32 [batch][d_model]; x_next may equal x or y.
 */
PI_API pi_status pi_rms_residual(const float *x, const float *y, int32_t batch, int32_t d_model, float *x_next,
                          pi_stream stream);

/*
 * Wait for `stream`, then read and clear the device error word of `ws` (a
 * workspace of any of the calls above).  Returns PI_OK, or the first of
 * PI_ERR_TIMEOUT, PI_ERR_CAPACITY, PI_ERR_INDEX that was raised since the last
 * call, or PI_ERR_CUDA when the stream itself reports an error.
 */
PI_API pi_status pi_sync_status(void *ws, size_t ws_bytes, pi_stream stream);

/*
 * pi_ffn_layer at batch 1 without a caller-provided workspace, for callers
 * that cannot allocate device memory (code in a host callback or an allocator
 * hook, plugins whose host forbids cudaMalloc, threads that must not risk the
 * device-wide synchronisation cudaMalloc / cudaFree can cause).  This entry
 * point is an engineering addition with no counterpart in the method's pages.
 *
 * Scratch space is a fixed file-scope device array of 1088 KiB inside the
 * library, present on every GPU that loads it until the process exits.  Limits:
 * d_ff <= 65536 and rank <= PI_MAX_RANK; larger layers return PI_ERR_SHAPE.
 * Every call looks up the array's device address on the current device (no
 * allocation); the first call on a device may load the library's device code,
 * so make it before any stream capture.  Nothing is allocated by any call.
 *
 * All calls share the array and it keeps the last call's contents.  Each call
 * first clears the error word, and zero-fills the part of the array the layer
 * uses when d_model, d_ff, rank, wtype or ptype differ from the previous
 * call's on that device or when the previous call's bounded wait gave up, so
 * layers of different shapes may alternate and a timeout needs no action from
 * the caller.  Calls that overlap on the GPU (other streams or unordered host
 * threads) race on the array and give wrong results.
 *   x, residual, y, idx, n_active: as in pi_ffn_layer with batch 1 (idx and
 *   n_active may both be NULL).
 *   status_out: device int32 [1] or NULL; receives the device error bits of
 *   this call when it completes (0 = none; 1 = a bounded device wait gave up;
 *   2 = active list over capacity; 4 = a neuron index out of range).
 */
PI_API pi_status pi_ffn_layer_static(const pi_ffn_desc *desc, const float *x, const float *residual, float *y,
                                     int32_t *idx, int32_t *n_active, int32_t *status_out, pi_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* PI_SPARSE_FFN_H */
