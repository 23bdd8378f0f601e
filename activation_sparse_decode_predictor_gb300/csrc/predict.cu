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
//   k_pred_logits  logit rows of P2 (one warp per row, four rows in flight),
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
// Small per-neuron vectors (p_bias, b_act): pull into L2 in 16-byte-aligned
// pieces, split over the CTAs of the grid.
__device__ __forceinline__ void prefetch_vec_l2(const float *v, int n)
{
    if (!v || n <= 0) return;
    const uintptr_t a0 = ((uintptr_t)v + 15) & ~(uintptr_t)15;
    const uintptr_t a1 = ((uintptr_t)(v + n)) & ~(uintptr_t)15;
    if (a1 <= a0) return;
    const size_t bytes = a1 - a0;
    const size_t per = ((bytes + gridDim.x - 1) / gridDim.x + 15) & ~(size_t)15;
    const size_t off = (size_t)blockIdx.x * per;
    if (off < bytes) prefetch_l2(reinterpret_cast<const void *>(a0 + off), (uint32_t)min(per, bytes - off));
}

template <typename PT>
__global__ void __launch_bounds__(kThreads) k_pred_hidden(const PT *__restrict__ p1, const float *__restrict__ x,
                                                          int B, int d, int r, float *__restrict__ h,
                                                          const uint8_t *__restrict__ p2, size_t p2_bytes,
                                                          const float *p_bias, const float *b_act, int F)
{
    extern __shared__ __align__(16) float xs[];  // [d]
    constexpr int EPC = 16 / sizeof(PT);
    constexpr int U = 8;  // 16-byte loads in flight per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kWarps + warp;
    const int nch = d / EPC;
    const uint4 *wrow = reinterpret_cast<const uint4 *>(p1 + (size_t)row * d);

    // The predictor weights do not depend on the previous kernel: pull this
    // CTA's P1 rows and a 1/grid slice of P2 towards L2 while that kernel is
    // still running, so both predictor GEMVs later read L2.
    if (lane == 0) {
        if (row < r) prefetch_l2(wrow, (uint32_t)(d * sizeof(PT)));
        const size_t per_cta = ((p2_bytes + gridDim.x - 1) / gridDim.x + 15) & ~(size_t)15;
        const size_t piece = ((per_cta + kWarps - 1) / kWarps + 15) & ~(size_t)15;
        const size_t off = (size_t)blockIdx.x * per_cta + (size_t)warp * piece;
        if (off < p2_bytes) prefetch_l2(p2 + off, (uint32_t)min(piece, p2_bytes - off));
        // the per-neuron biases the logit kernel and the sparse FFN will read
        if (warp == 0) prefetch_vec_l2(p_bias, F);
        if (warp == 1) prefetch_vec_l2(b_act, F);
    }
    pdl_wait();
    pdl_trigger();

    for (int b = 0; b < B; ++b) {
        const float4 *xb = reinterpret_cast<const float4 *>(x + (size_t)b * d);
        for (int i = threadIdx.x; i < d / 4; i += kThreads) reinterpret_cast<float4 *>(xs)[i] = xb[i];
        __syncthreads();
        if (row < r) {
            float acc = 0.f;
            for (int c0 = lane; c0 < nch; c0 += 32 * U) {
                uint4 w[U];
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (c0 + 32 * u < nch) w[u] = ld_stream(wrow + c0 + 32 * u);
#pragma unroll
                for (int u = 0; u < U; ++u)
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
// before it) and publishes this tile's inclusive prefix.  Called by all 32
// lanes of one warp: each pass reads a window of 32 predecessor status words
// at once, so a tile resolves its prefix in about tile/32 L2 round trips even
// when every tile finishes at the same moment.
__device__ unsigned lookback_warp(unsigned long long *status, int tile, unsigned count, unsigned epoch, unsigned *err)
{
    const int lane = threadIdx.x & 31;
    const unsigned ep = epoch & 0x3fffffffu;
    if (tile == 0) {
        if (lane == 0) st_volatile_u64(&status[0], pack_status(epoch, 2u, count));
        return 0u;
    }
    if (lane == 0) st_volatile_u64(&status[tile], pack_status(epoch, 1u, count));
    unsigned excl = 0;
    int base = tile - 1;
    long long spins = 0;
    for (;;) {
        const int p = base - lane;
        unsigned flag = 2u, val = 0u;  // before tile 0: an empty inclusive prefix
        if (p >= 0) {
            const unsigned long long s = ld_volatile_u64(&status[p]);
            const unsigned tag = (unsigned)(s >> 32);
            flag = (tag >> 2) == ep ? (tag & 3u) : 0u;
            val = (unsigned)s;
        }
        if (__any_sync(0xffffffffu, flag == 0u)) {
            if (++spins > kSpinLimit) {
                if (lane == 0) atomicOr(err, ERR_TIMEOUT);
                break;
            }
            __nanosleep(32);
            continue;
        }
        const unsigned pm = __ballot_sync(0xffffffffu, flag == 2u);
        const int first = pm ? __ffs(pm) - 1 : 31;
        unsigned v = lane <= first ? val : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        excl += v;
        if (pm) break;
        base -= 32;
    }
    if (lane == 0) st_volatile_u64(&status[tile], pack_status(epoch, 2u, excl + count));
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
        const unsigned base = lookback_warp(status, tile, total, sm.epoch, &ctrl->err);
        if (lane == 0) {
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

__device__ __forceinline__ void scan_start(ScanSmem &sm, WsCtrl *ctrl, int ntiles)
{
    if (threadIdx.x == 0) {
        unsigned t = atomicAdd(&ctrl->ticket, 1u);
        if (t >= (unsigned)ntiles) {  // a workspace that was not zero-filled: stay in bounds, report it
            atomicOr(&ctrl->err, ERR_TIMEOUT);
            t %= (unsigned)ntiles;
        }
        sm.tile = t;
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
    float *hs = dsm;                          // [B][r]
    float *lg = dsm + (size_t)p.B * p.r;      // [NB][tile_rows]
    float *pb = lg + (size_t)NB * p.tile_rows; // [tile_rows]
    const PT *p2 = static_cast<const PT *>(p.p2);

    // P2 was pulled towards L2 by the hidden-layer kernel's prologue.
    pdl_wait();
    pdl_trigger();
    scan_start(sm, p.ctrl, p.ntiles);
    {
        const float4 *h4 = reinterpret_cast<const float4 *>(p.h);
        for (int i = threadIdx.x; i < p.B * p.r / 4; i += kThreads) reinterpret_cast<float4 *>(hs)[i] = h4[i];
    }
    __syncthreads();
    const int tile = (int)sm.tile;
    const int tile_start = tile * p.tile_rows;
    const int nrows = min(p.tile_rows, p.F - tile_start);
    for (int i = threadIdx.x; i < nrows; i += kThreads) pb[i] = p.p_bias ? p.p_bias[tile_start + i] : 0.f;
    __syncthreads();

    constexpr int RW = 4;  // rows in flight per warp
    for (int rr = warp; rr < nrows; rr += RW * kWarps) {
        const uint4 *wp[RW];
        bool ok[RW];
#pragma unroll
        for (int i = 0; i < RW; ++i) {
            const int row = rr + i * kWarps;
            ok[i] = row < nrows;
            wp[i] = reinterpret_cast<const uint4 *>(p2 + (size_t)(tile_start + (ok[i] ? row : rr)) * p.r);
        }
        float acc[RW][NB];
#pragma unroll
        for (int i = 0; i < RW; ++i)
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[i][b] = 0.f;
        for (int c0 = lane; c0 < nch; c0 += 32 * 4) {
            uint4 v[RW][4];
#pragma unroll
            for (int i = 0; i < RW; ++i)
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = c0 + 32 * u;
                    if (ok[i] && c < nch) v[i][u] = ld_stream(wp[i] + c);
                }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + 32 * u;
                if (c < nch) {
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        if (b < p.B) {
                            const float *hb = hs + (size_t)b * p.r + c * EPC;
#pragma unroll
                            for (int i = 0; i < RW; ++i)
                                if (ok[i]) acc[i][b] += dot_chunk<PT>(v[i][u], hb);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < RW; ++i) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b < p.B) {
                    const float sum = warp_sum(acc[i][b]);
                    const int row = rr + i * kWarps;
                    if (lane == 0 && ok[i]) {
                        const int j = tile_start + row;
                        const float l = sum + pb[row];
                        lg[b * p.tile_rows + row] = l;
                        if (p.logits) p.logits[(size_t)b * p.F + j] = l;
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
    scan_start(sm, ctrl, ntiles);
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
                               const void *p2, size_t p2_bytes, const float *p_bias, const float *b_act, int F,
                               cudaStream_t s)
{
    const dim3 grid((r + kWarps - 1) / kWarps);
    const size_t smem = (size_t)d * sizeof(float);
    if (ptype == 1) {
        auto k = k_pred_hidden<__half>;
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        return launch_pdl(k, grid, dim3(kThreads), smem, s, static_cast<const __half *>(p1), x, B, d, r, h,
                          static_cast<const uint8_t *>(p2), p2_bytes, p_bias, b_act, F);
    }
    auto k = k_pred_hidden<float>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return launch_pdl(k, grid, dim3(kThreads), smem, s, static_cast<const float *>(p1), x, B, d, r, h,
                      static_cast<const uint8_t *>(p2), p2_bytes, p_bias, b_act, F);
}

template <typename PT>
static cudaError_t pred_logits_nb(const PredParams &p, cudaStream_t s)
{
    const size_t smem = ((size_t)p.B * p.r + (size_t)9 * p.tile_rows) * sizeof(float);
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
