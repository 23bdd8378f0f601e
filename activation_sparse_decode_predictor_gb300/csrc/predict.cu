// Activation predictor and active-index compaction.
//
// The predictor marks, per decode token, the FFN neurons expected to fire
// (PowerInfer summary page, "核心创新" core innovation: an adaptive predictor
// predicts the activated neurons so that unnecessary computation is skipped).
// Its form here is the low-rank MLP d -> r -> d_ff with a hidden ReLU:
//   h = max(P1 x, 0),  logit = P2 h + p_bias,  active = logit > threshold,
// and a batch of tokens shares the union of their active sets.
//
// Kernels:
//   k_pred_hidden  h = max(P1 x, 0): one warp per P1 row, x staged in shared
//                  memory, 16-byte streaming loads, shuffle reduction.
//   k_pred_logits  logit rows of P2 (one warp per row, two rows in flight),
//                  threshold and union, warp-ballot mask words, then a
//                  single-pass decoupled look-back scan across tiles (Merrill &
//                  Garland, "Single-pass Parallel Prefix Scan with Decoupled
//                  Look-back", 2016) that writes the ascending active list.
//   k_compact      the same scan over a caller-given byte mask.
// Both scan kernels take their logical tile from a ticket counter, so a tile
// only ever waits on tiles that started before it; every wait is bounded.
#include "internal.h"

namespace pi {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <typename PT>
__device__ __forceinline__ float dot_chunk(uint4 w, const float *x);
template <>
__device__ __forceinline__ float dot_chunk<__half>(uint4 w, const float *x) { return dot8_f16(w, x); }
template <>
__device__ __forceinline__ float dot_chunk<float>(uint4 w, const float *x) { return dot4_f32(w, x); }

// ---------------------------------------------------------------------------------
// h[b][k] = max(P1[k] . x[b], 0)
template <typename PT>
__global__ void __launch_bounds__(kThreads) k_pred_hidden(const PT *__restrict__ p1, const float *__restrict__ x,
                                                          int B, int d, int r, float *__restrict__ h)
{
    extern __shared__ __align__(16) float xs[];  // [d]
    constexpr int EPC = 16 / sizeof(PT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kWarps + warp;
    const int nch = d / EPC;
    const uint4 *wrow = reinterpret_cast<const uint4 *>(p1 + (size_t)row * d);

    // The predictor weights do not depend on the previous kernel: pull this
    // CTA's rows towards L2 while that kernel is still running.
    if (lane == 0 && row < r) prefetch_l2(wrow, (uint32_t)(d * sizeof(PT)));
    pdl_wait();
    pdl_trigger();

    for (int b = 0; b < B; ++b) {
        const float4 *xb = reinterpret_cast<const float4 *>(x + (size_t)b * d);
        for (int i = threadIdx.x; i < d / 4; i += kThreads) reinterpret_cast<float4 *>(xs)[i] = xb[i];
        __syncthreads();
        if (row < r) {
            float acc = 0.f;
            for (int c0 = lane; c0 < nch; c0 += 32 * 4) {
                uint4 w[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (c0 + 32 * u < nch) w[u] = ld_stream(wrow + c0 + 32 * u);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (c0 + 32 * u < nch) acc += dot_chunk<PT>(w[u], xs + (c0 + 32 * u) * EPC);
            }
            acc = warp_sum(acc);
            if (lane == 0) h[(size_t)b * r + row] = fmaxf(acc, 0.f);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------------
// Decoupled look-back.  Tile status word: high 32 bits = (epoch << 2) | flag
// (flag 1: tile aggregate, 2: inclusive prefix), low 32 bits = the value.
__device__ __forceinline__ unsigned long long pack_status(unsigned epoch, unsigned flag, unsigned v)
{
    return ((unsigned long long)(((epoch & 0x3fffffffu) << 2) | flag) << 32) | v;
}

// Returns the exclusive prefix of `tile` (number of active entries in tiles
// before it) and publishes this tile's inclusive prefix.  Single thread.
__device__ unsigned lookback(unsigned long long *status, int tile, unsigned count, unsigned epoch, unsigned *err)
{
    if (tile == 0) {
        st_volatile_u64(&status[0], pack_status(epoch, 2u, count));
        return 0u;
    }
    st_volatile_u64(&status[tile], pack_status(epoch, 1u, count));
    unsigned excl = 0;
    int p = tile - 1;
    long long spins = 0;
    while (p >= 0) {
        const unsigned long long s = ld_volatile_u64(&status[p]);
        const unsigned tag = (unsigned)(s >> 32);
        const unsigned flag = tag & 3u;
        if ((tag >> 2) == (epoch & 0x3fffffffu) && flag != 0u) {
            excl += (unsigned)s;
            if (flag == 2u) break;
            --p;
        } else {
            if (++spins > kSpinLimit) {
                atomicOr(err, ERR_TIMEOUT);
                break;
            }
            __nanosleep(32);
        }
    }
    st_volatile_u64(&status[tile], pack_status(epoch, 2u, excl + count));
    return excl;
}

struct ScanSmem {
    unsigned words[32];
    unsigned wpre[32];
    unsigned tile, epoch, base;
};

// Given this tile's mask words (smem), find its offset and write its entries
// of the ascending active list; the last tile writes the total.  All threads.
__device__ void scan_emit(ScanSmem &sm, int ntiles, int tile_start, int nw, int *idx, int *n_active, int cap,
                          WsCtrl *ctrl, unsigned long long *status)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = (int)sm.tile;
    if (warp == 0) {
        const unsigned c = lane < nw ? __popc(sm.words[lane]) : 0u;
        unsigned inc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned t = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += t;
        }
        if (lane < nw) sm.wpre[lane] = inc - c;
        const unsigned total = __shfl_sync(0xffffffffu, inc, 31);
        if (lane == 0) {
            const unsigned base = lookback(status, tile, total, sm.epoch, &ctrl->err);
            sm.base = base;
            if (tile == ntiles - 1) {
                unsigned all = base + total;
                if (all > (unsigned)cap) {
                    atomicOr(&ctrl->err, ERR_CAPACITY);
                    all = (unsigned)cap;
                }
                *n_active = (int)all;
            }
        }
    }
    __syncthreads();
    const unsigned base = sm.base;
    for (int wd = warp; wd < nw; wd += kWarps) {
        const unsigned bits = sm.words[wd];
        if ((bits >> lane) & 1u) {
            const unsigned pos = base + sm.wpre[wd] + __popc(bits & ((1u << lane) - 1u));
            if (pos < (unsigned)cap) idx[pos] = tile_start + wd * 32 + lane;
        }
    }
}

// The last CTA of a launch to finish resets the ticket counters and moves the
// epoch on, so the next launch starts from a clean scan state.
__device__ __forceinline__ void scan_finish(WsCtrl *ctrl, int ntiles, unsigned epoch)
{
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned d = atomicAdd(&ctrl->done, 1u);
        if (d == (unsigned)ntiles - 1u) {
            ctrl->ticket = 0u;
            ctrl->done = 0u;
            __threadfence();
            atomicExch(&ctrl->epoch, epoch + 1u);
        }
    }
}

__device__ __forceinline__ void scan_start(ScanSmem &sm, WsCtrl *ctrl)
{
    if (threadIdx.x == 0) {
        sm.tile = atomicAdd(&ctrl->ticket, 1u);
        sm.epoch = *reinterpret_cast<volatile unsigned *>(&ctrl->epoch);
    }
}

// ---------------------------------------------------------------------------------
template <typename PT, int NB>
__global__ void __launch_bounds__(kThreads) k_pred_logits(PredParams p)
{
    extern __shared__ __align__(16) float dsm[];
    __shared__ ScanSmem sm;
    constexpr int EPC = 16 / sizeof(PT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nch = p.r / EPC;
    const size_t rowbytes = (size_t)p.r * sizeof(PT);
    float *hs = dsm;                          // [B][r]
    float *lg = dsm + (size_t)p.B * p.r;      // [NB][tile_rows]
    const PT *p2 = static_cast<const PT *>(p.p2);

    // Prologue, independent of the predecessor: prefetch the P2 rows of tile
    // blockIdx.x into L2 (each warp a contiguous eighth).  Tickets hand tiles
    // out in start order, so this is the tile this CTA gets, or close to it.
    {
        const int r0 = blockIdx.x * p.tile_rows;
        const int r1 = min(r0 + p.tile_rows, p.F);
        if (r0 < r1 && lane == 0) {
            const size_t bytes = (size_t)(r1 - r0) * rowbytes;
            const size_t piece = ((bytes + kWarps - 1) / kWarps + 15) & ~(size_t)15;
            const size_t off = (size_t)warp * piece;
            if (off < bytes) {
                const size_t len = min(piece, bytes - off);
                prefetch_l2(reinterpret_cast<const uint8_t *>(p2 + (size_t)r0 * p.r) + off, (uint32_t)len);
            }
        }
    }
    pdl_wait();
    pdl_trigger();
    scan_start(sm, p.ctrl);
    {
        const float4 *h4 = reinterpret_cast<const float4 *>(p.h);
        for (int i = threadIdx.x; i < p.B * p.r / 4; i += kThreads) reinterpret_cast<float4 *>(hs)[i] = h4[i];
    }
    __syncthreads();
    const int tile = (int)sm.tile;
    const int tile_start = tile * p.tile_rows;
    const int nrows = min(p.tile_rows, p.F - tile_start);

    for (int rr = warp; rr < nrows; rr += 2 * kWarps) {
        const int ra = rr, rb = rr + kWarps;
        const bool hasb = rb < nrows;
        const uint4 *wa = reinterpret_cast<const uint4 *>(p2 + (size_t)(tile_start + ra) * p.r);
        const uint4 *wb = reinterpret_cast<const uint4 *>(p2 + (size_t)(tile_start + (hasb ? rb : ra)) * p.r);
        float acc_a[NB], acc_b[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) acc_a[b] = acc_b[b] = 0.f;
        for (int c0 = lane; c0 < nch; c0 += 32 * 4) {
            uint4 va[4], vb[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + 32 * u;
                if (c < nch) {
                    va[u] = ld_stream(wa + c);
                    vb[u] = ld_stream(wb + c);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + 32 * u;
                if (c < nch) {
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        if (b < p.B) {
                            acc_a[b] += dot_chunk<PT>(va[u], hs + (size_t)b * p.r + c * EPC);
                            acc_b[b] += dot_chunk<PT>(vb[u], hs + (size_t)b * p.r + c * EPC);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (b < p.B) {
                const float sa = warp_sum(acc_a[b]);
                const float sb = warp_sum(acc_b[b]);
                if (lane == 0) {
                    const int ja = tile_start + ra, jb = tile_start + rb;
                    const float la = sa + (p.p_bias ? p.p_bias[ja] : 0.f);
                    lg[b * p.tile_rows + ra] = la;
                    if (p.logits) p.logits[(size_t)b * p.F + ja] = la;
                    if (hasb) {
                        const float lb = sb + (p.p_bias ? p.p_bias[jb] : 0.f);
                        lg[b * p.tile_rows + rb] = lb;
                        if (p.logits) p.logits[(size_t)b * p.F + jb] = lb;
                    }
                }
            }
        }
    }
    __syncthreads();

    // threshold + union -> mask words
    const int nw = (nrows + 31) >> 5;
    for (int wd = warp; wd < nw; wd += kWarps) {
        const int row = wd * 32 + lane;
        bool on = false;
        if (row < nrows) {
#pragma unroll
            for (int b = 0; b < NB; ++b)
                if (b < p.B) on = on || (lg[b * p.tile_rows + row] > p.tau);
            if (p.mask) p.mask[tile_start + row] = on ? 1 : 0;
        }
        const unsigned bits = __ballot_sync(0xffffffffu, on);
        if (lane == 0) sm.words[wd] = bits;
    }
    __syncthreads();
    scan_emit(sm, p.ntiles, tile_start, nw, p.idx, p.n_active, p.cap, p.ctrl, p.status);

    // Initialise the FFN output (b_down + residual) for the sparse kernel that
    // follows: this tile's share of the B*d values.
    if (p.y) {
        const int nvec = p.B * p.d / 4;
        const int v0 = (int)((long long)nvec * tile / p.ntiles);
        const int v1 = (int)((long long)nvec * (tile + 1) / p.ntiles);
        float4 *y4 = reinterpret_cast<float4 *>(p.y);
        for (int v = v0 + threadIdx.x; v < v1; v += kThreads) {
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
            if (p.b_down) o = reinterpret_cast<const float4 *>(p.b_down)[v % (p.d / 4)];
            if (p.residual) {
                const float4 rz = reinterpret_cast<const float4 *>(p.residual)[v];
                o.x += rz.x;
                o.y += rz.y;
                o.z += rz.z;
                o.w += rz.w;
            }
            y4[v] = o;
        }
    }
    scan_finish(p.ctrl, p.ntiles, sm.epoch);
}

// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) k_compact(const uint8_t *__restrict__ mask, int n, int *idx, int *count,
                                                      int cap, WsCtrl *ctrl, unsigned long long *status, int ntiles,
                                                      int tile_rows)
{
    __shared__ ScanSmem sm;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    scan_start(sm, ctrl);
    __syncthreads();
    const int tile_start = (int)sm.tile * tile_rows;
    const int nrows = min(tile_rows, n - tile_start);
    const int nw = (nrows + 31) >> 5;
    for (int wd = warp; wd < nw; wd += kWarps) {
        const int row = wd * 32 + lane;
        const bool on = row < nrows && mask[tile_start + row] != 0;
        const unsigned bits = __ballot_sync(0xffffffffu, on);
        if (lane == 0) sm.words[wd] = bits;
    }
    __syncthreads();
    scan_emit(sm, ntiles, tile_start, nw, idx, count, cap, ctrl, status);
    scan_finish(ctrl, ntiles, sm.epoch);
}

}  // namespace

// ---------------------------------------------------------------------------------
cudaError_t launch_pred_hidden(int ptype, const void *p1, const float *x, int B, int d, int r, float *h,
                               cudaStream_t s)
{
    const dim3 grid((r + kWarps - 1) / kWarps);
    const size_t smem = (size_t)d * sizeof(float);
    if (ptype == 1) {
        auto k = k_pred_hidden<__half>;
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        return launch_pdl(k, grid, dim3(kThreads), smem, s, static_cast<const __half *>(p1), x, B, d, r, h);
    }
    auto k = k_pred_hidden<float>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return launch_pdl(k, grid, dim3(kThreads), smem, s, static_cast<const float *>(p1), x, B, d, r, h);
}

template <typename PT>
static cudaError_t pred_logits_nb(const PredParams &p, cudaStream_t s)
{
    const size_t smem = ((size_t)p.B * p.r + (size_t)8 * p.tile_rows) * sizeof(float);
    void (*k)(PredParams);
    if (p.B <= 1)
        k = k_pred_logits<PT, 1>;
    else if (p.B <= 2)
        k = k_pred_logits<PT, 2>;
    else if (p.B <= 4)
        k = k_pred_logits<PT, 4>;
    else
        k = k_pred_logits<PT, 8>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return launch_pdl(k, dim3(p.ntiles), dim3(kThreads), smem, s, p);
}

cudaError_t launch_pred_logits(int ptype, const PredParams &p, cudaStream_t s)
{
    return ptype == 1 ? pred_logits_nb<__half>(p, s) : pred_logits_nb<float>(p, s);
}

cudaError_t launch_compact(const uint8_t *mask, int n, int *idx, int *count, int cap, WsCtrl *ctrl,
                           unsigned long long *status, cudaStream_t s)
{
    const ScanGeom g = scan_geom(n);
    return launch_pdl(k_compact, dim3(g.ntiles), dim3(kThreads), 0, s, mask, n, idx, count, cap, ctrl, status,
                      g.ntiles, g.tile_rows);
}

}  // namespace pi
