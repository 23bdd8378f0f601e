// extern "C" entry points of the sparse-FFN library: host-side validation,
// workspace layout and kernel sequencing.  Declarations and the contract of
// each call are in include/pi.h.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <numeric>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "internal.h"
#include "pi.h"

namespace pi {

// Row gather of aux.cu (declared here rather than in internal.h, which the
// fused kernels include).
cudaError_t launch_gather_rows(const void *src, int64_t src_rows, void *dst, int64_t dst_rows, int64_t row_bytes,
                               const int *idx, cudaStream_t s);

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

WsLayout ws_layout(int d_model, int d_ff, int rank, int batch)
{
    WsLayout L{};
    size_t o = 0;
    L.ctrl = o;
    o += sizeof(WsCtrl);
    L.status = o;  // epoch-tagged status words of the scan kernels
    o = align256(o + (size_t)((d_ff + 31) / 32) * 8);
    L.fcount = o;  // plain per-CTA counts of the one-kernel layer step (its own region)
    o = align256(o + (size_t)1024 * 4);
    L.h = o;
    o = align256(o + (size_t)batch * (size_t)rank * 4);
    L.idx = o;
    o = align256(o + (size_t)d_ff * 4);
    L.nact = o;
    o = align256(o + 16);
    L.candb = o;
    if (batch == 1) o = align256(o + (size_t)d_ff * 4);
    L.qent = o;
    if (batch == 1) o = align256(o + (size_t)d_ff * 8);
    L.act = L.xf = L.uctl = L.zbuf = L.ucnt = L.xfh = L.umask = o;
    if (batch > 1) {
        const size_t tiles = ((size_t)d_ff + 15) / 16;
        const size_t gemm_tiles = ((size_t)(d_ff > rank ? d_ff : rank) + 15) / 16;  // FFN up or predictor
        L.act = o;
        o = align256(o + tiles * 512);
        L.xf = o;
        o = align256(o + (((size_t)d_model + 31) / 32) * 1024);
        L.uctl = o;
        o = align256(o + 96);
        L.zbuf = o;
        o = align256(o + gemm_tiles * 1024);
        L.ucnt = o;
        o = align256(o + gemm_tiles * 4);
        L.xfh = o;
        o = align256(o + (((size_t)(rank > 0 ? rank : 0) + 31) / 32) * 1024);
        L.umask = o;
        o = align256(o + (size_t)d_ff);
    }
    L.total = o;
    return L;
}

size_t compact_ws_bytes(int n) { return align256(sizeof(WsCtrl) + (size_t)((n + 31) / 32) * 8); }

int sm_count()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (cache[dev] == 0) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = v > 0 ? v : 1;
    }
    return cache[dev];
}

}  // namespace pi

using namespace pi;

namespace {

inline bool al(const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// A named NVTX range around the host side of an entry point (the enqueue), so
// profilers can attribute the kernels each call launches; costs a pointer
// check when no tool is attached.
struct Nvtx {
    explicit Nvtx(const char *name) { nvtxRangePushA(name); }
    ~Nvtx() { nvtxRangePop(); }
};

inline bool overlap(const void *a, size_t an, const void *b, size_t bn)
{
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + bn && y < x + an;
}

inline pi_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PI_OK : PI_ERR_CUDA; }

// Checks of the FFN part (ffn) and / or the predictor part (pred) of a desc.
pi_status check_desc(const pi_ffn_desc *D, bool ffn, bool pred)
{
    if (!D) return PI_ERR_NULL;
    if (D->d_model < 8 || D->d_model > PI_MAX_D_MODEL || D->d_model % 8) return PI_ERR_SHAPE;
    if (D->d_ff < 1 || D->d_ff >= (1 << 26)) return PI_ERR_SHAPE;
    if (D->gated != 0 && D->gated != 1) return PI_ERR_SHAPE;
    if (D->act != PI_ACT_RELU && D->act != PI_ACT_RELU2) return PI_ERR_SHAPE;
    if (ffn) {
        if (D->wtype != PI_F32 && D->wtype != PI_F16 && D->wtype != PI_Q4_0) return PI_ERR_DTYPE;
        if (D->wtype == PI_Q4_0 && D->d_model % 256) return PI_ERR_SHAPE;
        if (!D->w_up || !D->w_down || (D->gated && !D->w_gate)) return PI_ERR_NULL;
        if (!al(D->w_up, 16) || !al(D->w_down, 16) || (D->gated && !al(D->w_gate, 16))) return PI_ERR_ALIGN;
        if ((D->b_act && !al(D->b_act, 4)) || (D->b_down && !al(D->b_down, 16))) return PI_ERR_ALIGN;
    }
    if (pred) {
        if (D->ptype != PI_F32 && D->ptype != PI_F16) return PI_ERR_DTYPE;
        if (D->rank < 8 || D->rank > PI_MAX_RANK || D->rank % 8) return PI_ERR_SHAPE;
        if (D->d_ff >= (1 << 23)) return PI_ERR_SHAPE;
        if (D->dense_prefix < 0 || D->dense_prefix > D->d_ff) return PI_ERR_SHAPE;
        if (!D->p1 || !D->p2) return PI_ERR_NULL;
        if (!al(D->p1, 16) || !al(D->p2, 16) || (D->p_bias && !al(D->p_bias, 4))) return PI_ERR_ALIGN;
    }
    return PI_OK;
}

pi_status check_ws(void *ws, size_t ws_bytes, size_t need)
{
    if (!ws) return PI_ERR_WORKSPACE;
    if (!al(ws, 256)) return PI_ERR_ALIGN;
    if (ws_bytes < need) return PI_ERR_WORKSPACE;
    return PI_OK;
}

pi_status check_io(const pi_ffn_desc *D, const float *x, int32_t B, const float *residual, const float *y)
{
    if (B < 1 || B > PI_MAX_BATCH) return PI_ERR_SHAPE;
    if (!x || !y) return PI_ERR_NULL;
    if (!al(x, 16) || !al(y, 16) || (residual && !al(residual, 16))) return PI_ERR_ALIGN;
    const size_t nb = (size_t)B * D->d_model * sizeof(float);
    if (overlap(x, nb, y, nb)) return PI_ERR_ALIAS;
    if (residual && residual != y && overlap(residual, nb, y, nb)) return PI_ERR_ALIAS;
    if (B > 1 && D->wtype == PI_F32) return PI_ERR_DTYPE;
    return PI_OK;
}

template <typename T>
T *at(void *ws, size_t off) { return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off); }

pi_status enqueue_predict(const pi_ffn_desc *D, const float *x, int32_t B, float *logits, uint8_t *mask, int32_t *idx,
                          int32_t *n_active, int32_t cap, void *ws, float *y_init, const float *residual,
                          cudaStream_t s)
{
    const WsLayout L = ws_layout(D->d_model, D->d_ff, D->rank, B);
    if (B > 1 && D->ptype == PI_F16) {
        // several tokens: both predictor contractions on tensor cores, then one scan
        UnionPredArgs a{};
        a.p1 = D->p1;
        a.p2 = D->p2;
        a.p_bias = D->p_bias;
        a.tau = D->threshold;
        a.x = x;
        a.B = B;
        a.d = D->d_model;
        a.r = D->rank;
        a.F = D->d_ff;
        a.h = at<float>(ws, L.h);
        a.logits = logits;
        a.mask = mask ? mask : at<uint8_t>(ws, L.umask);
        a.xf_x = at<uint32_t>(ws, L.xf);
        a.xf_h = at<uint32_t>(ws, L.xfh);
        a.uexp_x = at<int>(ws, L.uctl);
        a.amax = at<unsigned>(ws, L.uctl + 32);
        a.uexp_h = at<int>(ws, L.uctl + 64);
        a.zbuf = at<float>(ws, L.zbuf);
        a.ucnt = at<unsigned>(ws, L.ucnt);
        a.ctrl = at<WsCtrl>(ws, L.ctrl);
        a.prefix = D->dense_prefix;
        if (launch_pred_union(a, s) != cudaSuccess) return PI_ERR_CUDA;
        if (launch_compact(a.mask, D->d_ff, idx, n_active, cap, a.ctrl, at<unsigned long long>(ws, L.status), s) !=
            cudaSuccess)
            return PI_ERR_CUDA;
        if (y_init && launch_init_y(y_init, D->b_down, residual, B, D->d_model, nullptr, nullptr, 0, s) != cudaSuccess)
            return PI_ERR_CUDA;
        return PI_OK;
    }
    float *h = at<float>(ws, L.h);
    const size_t p2_bytes = (size_t)D->d_ff * D->rank * (D->ptype == PI_F16 ? 2 : 4);
    cudaError_t e = launch_pred_hidden(D->ptype, D->p1, x, B, D->d_model, D->rank, h, D->p2, p2_bytes, D->p_bias,
                                       D->b_act, D->d_ff, s);
    if (e != cudaSuccess) return PI_ERR_CUDA;
    PredParams p{};
    p.p2 = D->p2;
    p.p_bias = D->p_bias;
    p.h = h;
    p.B = B;
    p.r = D->rank;
    p.F = D->d_ff;
    p.tau = D->threshold;
    p.prefix = D->dense_prefix;
    p.logits = logits;
    p.mask = mask;
    p.idx = idx;
    p.n_active = n_active;
    p.cap = cap;
    p.ctrl = at<WsCtrl>(ws, L.ctrl);
    p.status = at<unsigned long long>(ws, L.status);
    p.y = y_init;
    p.residual = residual;
    p.b_down = D->b_down;
    p.d = D->d_model;
    return cuda_status(launch_pred_logits(D->ptype, p, s));
}

pi_status enqueue_sparse(const pi_ffn_desc *D, const float *x, int32_t B, const int32_t *idx,
                         const int32_t *n_active, float *y, void *ws, cudaStream_t s, bool xf_ready = false)
{
    const WsLayout L = ws_layout(D->d_model, D->d_ff, D->rank, B);
    SparseParams p{};
    p.w_act = static_cast<const uint8_t *>(D->gated ? D->w_gate : D->w_up);
    p.w_up = static_cast<const uint8_t *>(D->gated ? D->w_up : nullptr);
    p.w_down = static_cast<const uint8_t *>(D->w_down);
    p.b_act = D->b_act;
    p.x = x;
    p.idx = idx;
    p.n_active = n_active;
    p.y = y;
    p.ctrl = at<WsCtrl>(ws, L.ctrl);
    if (B > 1) {
        p.act_ws = at<float>(ws, L.act);
        p.xf = at<uint32_t>(ws, L.xf);
        p.uexp = at<int>(ws, L.uctl);
        p.amax = at<unsigned>(ws, L.uctl + 32);
        p.zbuf = at<float>(ws, L.zbuf);
        p.ucnt = at<unsigned>(ws, L.ucnt);
        p.xf_ready = xf_ready ? 1 : 0;
    }
    p.d = D->d_model;
    p.F = D->d_ff;
    p.act = D->act;
    p.B = B;
    const cudaError_t e = B == 1 ? launch_sparse_b1(D->wtype, D->gated, p, s)
                                 : launch_sparse_union(D->wtype, D->gated, p, s);
    return cuda_status(e);
}

}  // namespace

extern "C" {

const char *pi_status_str(int32_t st)
{
    switch (st) {
    case PI_OK: return "ok";
    case PI_ERR_NULL: return "required pointer is NULL";
    case PI_ERR_SHAPE: return "size out of range or not divisible as required";
    case PI_ERR_DTYPE: return "unsupported storage type";
    case PI_ERR_ALIGN: return "pointer not aligned as required";
    case PI_ERR_CAPACITY: return "active list exceeded its capacity";
    case PI_ERR_CUDA: return "CUDA error";
    case PI_ERR_TIMEOUT: return "bounded device wait gave up";
    case PI_ERR_WORKSPACE: return "workspace missing or too small";
    case PI_ERR_ALIAS: return "output overlaps an input";
    case PI_ERR_INDEX: return "neuron index out of range";
    default: return "unknown status";
    }
}

size_t pi_workspace_bytes(const pi_ffn_desc *desc, int32_t batch)
{
    if (!desc || batch < 1 || batch > PI_MAX_BATCH) return 0;
    if (desc->d_model < 8 || desc->d_ff < 1 || desc->rank < 0) return 0;
    return ws_layout(desc->d_model, desc->d_ff, desc->rank, batch).total;
}

size_t pi_compact_workspace_bytes(int32_t n) { return n < 1 ? 0 : compact_ws_bytes(n); }

pi_status pi_compact(const uint8_t *mask, int32_t n, int32_t *idx, int32_t *count, int32_t cap, void *ws,
                     size_t ws_bytes, pi_stream stream)
{
    Nvtx nv("pi_compact");
    if (!mask || !idx || !count) return PI_ERR_NULL;
    if (n < 1 || cap < 1) return PI_ERR_SHAPE;
    if (!al(idx, 4) || !al(count, 4)) return PI_ERR_ALIGN;
    pi_status st = check_ws(ws, ws_bytes, compact_ws_bytes(n));
    if (st != PI_OK) return st;
    return cuda_status(launch_compact(mask, n, idx, count, cap, at<WsCtrl>(ws, 0),
                                      at<unsigned long long>(ws, sizeof(WsCtrl)), (cudaStream_t)stream));
}

pi_status pi_predict(const pi_ffn_desc *desc, const float *x, int32_t batch, float *logits, uint8_t *mask,
                     int32_t *idx, int32_t *n_active, int32_t cap, void *ws, size_t ws_bytes, pi_stream stream)
{
    Nvtx nv("pi_predict");
    pi_status st = check_desc(desc, false, true);
    if (st != PI_OK) return st;
    if (batch < 1 || batch > PI_MAX_BATCH || cap < 1) return PI_ERR_SHAPE;
    if (!x || !idx || !n_active) return PI_ERR_NULL;
    if (!al(x, 16) || (logits && !al(logits, 4)) || !al(idx, 4) || !al(n_active, 4)) return PI_ERR_ALIGN;
    st = check_ws(ws, ws_bytes, ws_layout(desc->d_model, desc->d_ff, desc->rank, batch).total);
    if (st != PI_OK) return st;
    return enqueue_predict(desc, x, batch, logits, mask, idx, n_active, cap, ws, nullptr, nullptr,
                           (cudaStream_t)stream);
}

pi_status pi_sparse_ffn(const pi_ffn_desc *desc, const float *x, int32_t batch, const int32_t *idx,
                        const int32_t *n_active, const float *residual, float *y, void *ws, size_t ws_bytes,
                        pi_stream stream)
{
    Nvtx nv("pi_sparse_ffn");
    pi_status st = check_desc(desc, true, false);
    if (st != PI_OK) return st;
    st = check_io(desc, x, batch, residual, y);
    if (st != PI_OK) return st;
    if (!idx || !n_active) return PI_ERR_NULL;
    if (!al(idx, 4) || !al(n_active, 4)) return PI_ERR_ALIGN;
    st = check_ws(ws, ws_bytes, ws_layout(desc->d_model, desc->d_ff, desc->rank, batch).total);
    if (st != PI_OK) return st;
    const cudaStream_t s = (cudaStream_t)stream;
    if (launch_init_y(y, desc->b_down, residual, batch, desc->d_model, nullptr, nullptr, 0, s) != cudaSuccess)
        return PI_ERR_CUDA;
    return enqueue_sparse(desc, x, batch, idx, n_active, y, ws, s);
}

}  // extern "C"

namespace {

// pi_ffn_layer, and with x_prev / y_prev given its chained form: the input is
// then x = (x_prev + y_prev) / rms(x_prev + y_prev), written to x (the one-
// kernel step computes it in its prologue; other shapes run the glue kernel
// first).
pi_status ffn_layer(const pi_ffn_desc *desc, const float *x, const float *x_prev, const float *y_prev, int32_t batch,
                    const float *residual, float *y, int32_t *idx, int32_t *n_active, void *ws, size_t ws_bytes,
                    cudaStream_t s)
{
    pi_status st = check_desc(desc, true, true);
    if (st != PI_OK) return st;
    st = check_io(desc, x, batch, residual, y);
    if (st != PI_OK) return st;
    if ((idx == nullptr) != (n_active == nullptr)) return PI_ERR_NULL;
    if ((idx && !al(idx, 4)) || (n_active && !al(n_active, 4))) return PI_ERR_ALIGN;
    const WsLayout L = ws_layout(desc->d_model, desc->d_ff, desc->rank, batch);
    st = check_ws(ws, ws_bytes, L.total);
    if (st != PI_OK) return st;
    const bool chained = x_prev != nullptr;
    if (chained) {
        const size_t nb = (size_t)batch * desc->d_model * sizeof(float);
        if (!y_prev) return PI_ERR_NULL;
        if (!al(x_prev, 16) || !al(y_prev, 16)) return PI_ERR_ALIGN;
        if (overlap(x, nb, x_prev, nb) || overlap(x, nb, y_prev, nb) || overlap(y, nb, x_prev, nb) ||
            overlap(y, nb, y_prev, nb))
            return PI_ERR_ALIAS;
    }
    if (batch == 1 &&
        fused_layer_supported(desc->wtype, desc->ptype, desc->d_model, desc->d_ff, desc->rank, desc->dense_prefix)) {
        // one kernel per token: predictor, scan and sparse FFN without kernel boundaries
        LayerB1Args a{};
        a.wtype = desc->wtype;
        a.ptype = desc->ptype;
        a.gated = desc->gated;
        a.act = desc->act;
        a.p1 = desc->p1;
        a.p2 = desc->p2;
        a.p_bias = desc->p_bias;
        a.tau = desc->threshold;
        a.r = desc->rank;
        a.w_up = desc->w_up;
        a.w_gate = desc->w_gate;
        a.w_down = desc->w_down;
        a.b_act = desc->b_act;
        a.b_down = desc->b_down;
        a.x = x;
        a.x_prev = chained ? x_prev : nullptr;
        a.y_prev = chained ? y_prev : nullptr;
        a.x_out = chained ? const_cast<float *>(x) : nullptr;
        a.residual = residual;
        a.y = y;
        a.idx_out = idx;
        a.n_active = n_active;
        a.cand = at<int32_t>(ws, L.idx);
        a.cand_bias = at<float>(ws, L.candb);
        a.qent = at<unsigned long long>(ws, L.qent);
        a.h = at<float>(ws, L.h);
        a.status = at<unsigned>(ws, L.fcount);
        a.ctrl = at<WsCtrl>(ws, L.ctrl);
        a.d = desc->d_model;
        a.F = desc->d_ff;
        a.prefix = desc->dense_prefix;
        return cuda_status(launch_layer_b1(a, s));
    }
    if (chained && launch_rms_residual(x_prev, y_prev, batch, desc->d_model, const_cast<float *>(x), s) != cudaSuccess)
        return PI_ERR_CUDA;
    if (!idx) {
        idx = at<int32_t>(ws, L.idx);
        n_active = at<int32_t>(ws, L.nact);
    }
    st = enqueue_predict(desc, x, batch, nullptr, nullptr, idx, n_active, desc->d_ff, ws, y, residual, s);
    if (st != PI_OK) return st;
    // the tensor-core predictor left x's fp16 fragments in the workspace (fp16 layout)
    const bool xf_ready = batch > 1 && desc->ptype == PI_F16 && desc->wtype == PI_F16;
    return enqueue_sparse(desc, x, batch, idx, n_active, y, ws, s, xf_ready);
}

}  // namespace

extern "C" {

pi_status pi_ffn_layer(const pi_ffn_desc *desc, const float *x, int32_t batch, const float *residual, float *y,
                       int32_t *idx, int32_t *n_active, void *ws, size_t ws_bytes, pi_stream stream)
{
    Nvtx nv("pi_ffn_layer");
    return ffn_layer(desc, x, nullptr, nullptr, batch, residual, y, idx, n_active, ws, ws_bytes, (cudaStream_t)stream);
}

pi_status pi_ffn_layer_chain(const pi_ffn_desc *desc, const float *x_prev, const float *y_prev, int32_t batch, float *x,
                             float *y, int32_t *idx, int32_t *n_active, void *ws, size_t ws_bytes, pi_stream stream)
{
    Nvtx nv("pi_ffn_layer_chain");
    if (!x_prev || !y_prev) return PI_ERR_NULL;
    return ffn_layer(desc, x, x_prev, y_prev, batch, nullptr, y, idx, n_active, ws, ws_bytes, (cudaStream_t)stream);
}

pi_status pi_dense_ffn(const pi_ffn_desc *desc, const float *x, int32_t batch, const float *residual, float *y,
                       void *ws, size_t ws_bytes, pi_stream stream)
{
    Nvtx nv("pi_dense_ffn");
    pi_status st = check_desc(desc, true, false);
    if (st != PI_OK) return st;
    st = check_io(desc, x, batch, residual, y);
    if (st != PI_OK) return st;
    const WsLayout L = ws_layout(desc->d_model, desc->d_ff, desc->rank, batch);
    st = check_ws(ws, ws_bytes, L.total);
    if (st != PI_OK) return st;
    const cudaStream_t s = (cudaStream_t)stream;
    int32_t *idx = at<int32_t>(ws, L.idx);
    int32_t *n = at<int32_t>(ws, L.nact);
    if (launch_init_y(y, desc->b_down, residual, batch, desc->d_model, idx, n, desc->d_ff, s) != cudaSuccess)
        return PI_ERR_CUDA;
    return enqueue_sparse(desc, x, batch, idx, n, y, ws, s);
}

size_t pi_q4_0_bytes(int64_t rows, int64_t cols)
{
    if (rows < 1 || cols < 32 || cols % 32) return 0;
    return (size_t)rows * (size_t)(cols / 2) + (size_t)rows * (size_t)(cols / 32) * 2;
}

pi_status pi_quantize_q4_0(const void *src, int32_t src_type, int64_t rows, int64_t cols, void *dst,
                           pi_stream stream)
{
    Nvtx nv("pi_quantize_q4_0");
    if (!src || !dst) return PI_ERR_NULL;
    if (src_type != PI_F32 && src_type != PI_F16) return PI_ERR_DTYPE;
    if (rows < 1 || cols < 32 || cols % 32) return PI_ERR_SHAPE;
    if (!al(src, 16) || !al(dst, 16)) return PI_ERR_ALIGN;
    const size_t nsrc = (size_t)rows * cols * (src_type == PI_F32 ? 4 : 2);
    if (overlap(src, nsrc, dst, pi_q4_0_bytes(rows, cols))) return PI_ERR_ALIAS;
    return cuda_status(launch_quantize_q4_0(src, src_type, rows, cols, dst, (cudaStream_t)stream));
}

// binary32 -> binary16, round to nearest, ties to even (IEEE 754 conversion,
// written from the format definitions): normal results by integer rounding of
// the 23-bit significand to 10 bits, subnormal results by rounding |f| * 2^24
// to an integer (exact scaling, then the FP environment's ties-to-even).
static uint16_t host_f32_to_f16(float f)
{
    uint32_t x;
    std::memcpy(&x, &f, 4);
    const uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    const uint32_t ax = x & 0x7fffffffu;
    if (ax > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);  // NaN
    if (ax >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u);  // >= 65520 rounds to infinity
    if (ax < 0x38800000u) {                                     // below 2^-14: subnormal or zero
        const float m = std::nearbyint(std::fabs(f) * 16777216.0f);  // |f| * 2^24, exact
        return (uint16_t)(sign | (uint16_t)m);                  // m == 1024 is the smallest normal
    }
    const uint32_t e = (ax >> 23) - 127 + 15, mant = ax & 0x7fffffu;
    uint32_t h = (e << 10) | (mant >> 13);
    const uint32_t rest = mant & 0x1fffu;
    if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) ++h;   // carries into the exponent as it should
    return (uint16_t)(sign | h);
}

static float host_f16_to_f32(uint16_t h)
{
    const uint32_t e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
    float v;
    if (e == 0) v = std::ldexp((float)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = std::ldexp((float)(m | 0x400u), (int)e - 25);
    return (h & 0x8000u) ? -v : v;
}

pi_status pi_quantize_q4_0_host(const float *src, int64_t rows, int64_t cols, void *dst)
{
    Nvtx nv("pi_quantize_q4_0_host");
    if (!src || !dst) return PI_ERR_NULL;
    if (rows < 1 || cols < 32 || cols % 32) return PI_ERR_SHAPE;
    if (overlap(src, (size_t)rows * cols * 4, dst, pi_q4_0_bytes(rows, cols))) return PI_ERR_ALIAS;
    uint8_t *codes = static_cast<uint8_t *>(dst);
    uint8_t *scales = codes + (size_t)rows * (size_t)(cols / 2);
    const int64_t nb = cols / 32;
    for (int64_t j = 0; j < rows; ++j) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *w = src + j * cols + b * 32;
            float amax = w[0];  // the first weight of largest magnitude
            for (int e = 1; e < 32; ++e)
                if (std::fabs(w[e]) > std::fabs(amax)) amax = w[e];
            const float s32 = amax / -8.0f;
            const uint16_t s16 = s32 == 0.0f ? (uint16_t)0 : host_f32_to_f16(s32);
            const float sc = host_f16_to_f32(s16);
            uint8_t q[32];
            for (int e = 0; e < 32; ++e) {
                int qi = 8;
                if (sc != 0.0f) {
                    volatile float t = w[e] / sc;  // binary32 quotient, then binary32 sum
                    const float fl = std::floor(t + 8.5f);
                    qi = fl < 0.0f ? 0 : (fl > 15.0f ? 15 : (int)fl);
                }
                q[e] = (uint8_t)qi;
            }
            uint8_t *cb = codes + j * (cols / 2) + b * 16;
            for (int e = 0; e < 16; ++e) cb[e] = (uint8_t)(q[e] | (q[e + 16] << 4));
            std::memcpy(scales + 2 * (size_t)(j * nb + b), &s16, 2);  // little-endian binary16
        }
    }
    return PI_OK;
}

pi_status pi_fire_counts(const pi_ffn_desc *desc, const float *X, int32_t T, int32_t *counts, pi_stream stream)
{
    Nvtx nv("pi_fire_counts");
    pi_status st = check_desc(desc, true, false);
    if (st != PI_OK) return st;
    if (desc->wtype == PI_Q4_0) return PI_ERR_DTYPE;
    if (!X || !counts) return PI_ERR_NULL;
    if (T < 1) return PI_ERR_SHAPE;
    if (!al(X, 4) || !al(counts, 4)) return PI_ERR_ALIGN;
    const void *w = desc->gated ? desc->w_gate : desc->w_up;
    return cuda_status(launch_fire_counts(desc->wtype, w, desc->b_act, X, T, desc->d_model, desc->d_ff, counts,
                                          (cudaStream_t)stream));
}

pi_status pi_hot_first_perm(const int32_t *counts, int32_t n, int32_t *perm)
{
    if (!counts || !perm) return PI_ERR_NULL;
    if (n < 1) return PI_ERR_SHAPE;
    std::vector<int32_t> order((size_t)n);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [counts](int32_t a, int32_t b) { return counts[a] > counts[b]; });
    std::copy(order.begin(), order.end(), perm);
    return PI_OK;
}

pi_status pi_permute_rows(const void *src, void *dst, int64_t rows, int64_t row_bytes, const int32_t *perm,
                          pi_stream stream)
{
    Nvtx nv("pi_permute_rows");
    if (!src || !dst || !perm) return PI_ERR_NULL;
    if (rows < 1 || row_bytes < 1) return PI_ERR_SHAPE;
    if (!al(perm, 4)) return PI_ERR_ALIGN;
    if (overlap(src, (size_t)(rows * row_bytes), dst, (size_t)(rows * row_bytes))) return PI_ERR_ALIAS;
    return cuda_status(launch_permute_rows(src, dst, rows, row_bytes, perm, (cudaStream_t)stream));
}

pi_status pi_gather_rows(const void *src, int64_t src_rows, void *dst, int64_t dst_rows, int64_t row_bytes,
                         const int32_t *idx, pi_stream stream)
{
    Nvtx nv("pi_gather_rows");
    if (!src || !dst || !idx) return PI_ERR_NULL;
    if (src_rows < 1 || dst_rows < 1 || row_bytes < 1) return PI_ERR_SHAPE;
    if (!al(idx, 4)) return PI_ERR_ALIGN;
    if (overlap(src, (size_t)(src_rows * row_bytes), dst, (size_t)(dst_rows * row_bytes))) return PI_ERR_ALIAS;
    return cuda_status(launch_gather_rows(src, src_rows, dst, dst_rows, row_bytes, idx, (cudaStream_t)stream));
}

pi_status pi_shard_neurons(const int32_t *order, int32_t n, int32_t shards, int32_t shard, int32_t *out,
                           int32_t *count)
{
    if (!order || !out || !count) return PI_ERR_NULL;
    if (n < 1 || shards < 1 || shard < 0 || shard >= shards || shards > n) return PI_ERR_SHAPE;
    std::vector<uint8_t> seen((size_t)n, 0);
    for (int32_t p = 0; p < n; ++p) {
        const int32_t j = order[p];
        if (j < 0 || j >= n || seen[(size_t)j]) return PI_ERR_INDEX;
        seen[(size_t)j] = 1;
    }
    int32_t c = 0;
    for (int32_t p = shard; p < n; p += shards) out[c++] = order[p];
    *count = c;
    return PI_OK;
}

pi_status pi_rms_residual(const float *x, const float *y, int32_t batch, int32_t d_model, float *x_next,
                          pi_stream stream)
{
    Nvtx nv("pi_rms_residual");
    if (!x || !y || !x_next) return PI_ERR_NULL;
    if (batch < 1 || d_model < 1) return PI_ERR_SHAPE;
    if (!al(x, 4) || !al(y, 4) || !al(x_next, 4)) return PI_ERR_ALIGN;
    return cuda_status(launch_rms_residual(x, y, batch, d_model, x_next, (cudaStream_t)stream));
}

pi_status pi_sync_status(void *ws, size_t ws_bytes, pi_stream stream)
{
    Nvtx nv("pi_sync_status");
    if (!ws) return PI_ERR_WORKSPACE;
    if (ws_bytes < sizeof(WsCtrl)) return PI_ERR_WORKSPACE;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return PI_ERR_CUDA;
    unsigned err = 0;
    if (cudaMemcpy(&err, ws, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess) return PI_ERR_CUDA;
    if (err) {
        const unsigned zero = 0;
        if (cudaMemcpy(ws, &zero, sizeof(unsigned), cudaMemcpyHostToDevice) != cudaSuccess) return PI_ERR_CUDA;
    }
    if (err & ERR_TIMEOUT) return PI_ERR_TIMEOUT;
    if (err & ERR_CAPACITY) return PI_ERR_CAPACITY;
    if (err & ERR_INDEX) return PI_ERR_INDEX;
    return PI_OK;
}

}  // extern "C"
