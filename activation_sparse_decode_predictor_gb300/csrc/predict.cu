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
//   k_pred_logits  one CTA per SM over a balanced contiguous neuron range:
//                  logit rows of P2 (one warp per row, four rows in flight,
//                  P2 already pulled into L2 by k_pred_hidden), threshold and
//                  union, warp-ballot mask words, then a single-pass scan
//                  across CTAs (each publishes its count and sums those of
//                  the CTAs before it) that writes the ascending active list.
//   k_compact      the same scan over a caller-given byte mask.
// Every cross-CTA wait is bounded.
#include <algorithm>

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
// Cross-CTA scan.  CTA c owns the contiguous neuron range [c*F/G, (c+1)*F/G)
// and G never exceeds the number of SMs, so every CTA of the grid is resident
// at once.  Each CTA publishes its active count in a status word tagged with
// the launch's epoch, then sums the counts of all CTAs before it, read in one
// parallel pass (G <= #SMs words) and re-polled, with a bound, only where a
// predecessor has not published yet.  The last CTA to finish moves the epoch
// on, so stale words of earlier launches are never mistaken for current ones.
__device__ __forceinline__ unsigned long long pack_status(unsigned epoch, unsigned v)
{
    return ((unsigned long long)(((epoch & 0x7fffffffu) << 1) | 1u) << 32) | v;
}

template <int NT>
__device__ __forceinline__ unsigned block_sum(unsigned v, unsigned *red)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    unsigned t = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) t += red[w];
    return t;
}

template <int NT>
__device__ unsigned sum_before(unsigned long long *status, int c, unsigned count, unsigned epoch, unsigned *err,
                               unsigned *red)
{
    const unsigned want = ((epoch & 0x7fffffffu) << 1) | 1u;
    if (threadIdx.x == 0) st_volatile_u64(&status[c], pack_status(epoch, count));
    unsigned part = 0;
    for (int i = threadIdx.x; i < c; i += NT) {
        unsigned long long s = ld_volatile_u64(&status[i]);
        long long spins = 0;
        while ((unsigned)(s >> 32) != want) {
            if (++spins > kSpinLimit) {
                atomicOr(err, ERR_TIMEOUT);
                s = 0;
                break;
            }
            __nanosleep(32);
            s = ld_volatile_u64(&status[i]);
        }
        part += (unsigned)s;
    }
    return block_sum<NT>(part, red);
}

// Exclusive prefix of popc(words[0..nw)) into wpre; returns the total.
template <int NT>
__device__ unsigned scan_words(const unsigned *words, unsigned *wpre, int nw, unsigned *red)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per = (nw + NT - 1) / NT;
    const int w0 = threadIdx.x * per, w1 = min(nw, w0 + per);
    unsigned mine = 0;
    for (int w = w0; w < w1; ++w) mine += __popc(words[w]);
    unsigned inc = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    __syncthreads();
    if (lane == 31) red[warp] = inc;
    __syncthreads();
    unsigned before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        if (w < warp) before += red[w];
        total += red[w];
    }
    unsigned run = before + inc - mine;
    for (int w = w0; w < w1; ++w) {
        wpre[w] = run;
        run += __popc(words[w]);
    }
    __syncthreads();
    return total;
}

// Write this CTA's entries of the ascending active list.
template <int NT>
__device__ void emit_idx(const unsigned *words, const unsigned *wpre, int nw, int row0, unsigned base, int *idx,
                         int cap)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int wd = warp; wd < nw; wd += NT / 32) {
        const unsigned bits = words[wd];
        if ((bits >> lane) & 1u) {
            const unsigned pos = base + wpre[wd] + __popc(bits & ((1u << lane) - 1u));
            if (pos < (unsigned)cap) idx[pos] = row0 + wd * 32 + lane;
        }
    }
}

__device__ __forceinline__ void scan_finish(WsCtrl *ctrl, int G, unsigned epoch)
{
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned d = atomicAdd(&ctrl->done, 1u);
        if (d == (unsigned)G - 1u) {
            ctrl->done = 0u;
            __threadfence();
            atomicExch(&ctrl->epoch, epoch + 1u);
        }
    }
}

__device__ __forceinline__ void write_total(int c, int G, unsigned base, unsigned count, int *n_active, int cap,
                                            unsigned *err)
{
    if (threadIdx.x == 0 && c == G - 1) {
        unsigned all = base + count;
        if (all > (unsigned)cap) {
            atomicOr(err, ERR_CAPACITY);
            all = (unsigned)cap;
        }
        *n_active = (int)all;
    }
}

constexpr int kLThreads = 512;          // logit kernel: 16 warps per CTA, one CTA per SM
constexpr int kLWarps = kLThreads / 32;
constexpr int kChunk = 1024;            // rows per logits chunk held in shared memory

// ---------------------------------------------------------------------------------
template <typename PT, int NB>
__global__ void __launch_bounds__(kLThreads, 1) k_pred_logits(PredParams p)
{
    extern __shared__ __align__(16) float dsm[];
    __shared__ unsigned red[kLWarps];
    __shared__ unsigned s_epoch;
    constexpr int EPC = 16 / sizeof(PT);
    constexpr int RW = 4;  // rows in flight per warp
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, G = gridDim.x;
    const int r0 = (int)((long long)p.F * c / G);
    const int R = (int)((long long)p.F * (c + 1) / G) - r0;
    const int nw = (R + 31) >> 5;
    const int nch = p.r / EPC;
    float *hs = dsm;                                   // [B][r]
    float *lg = hs + (size_t)p.B * p.r;                // [NB][kChunk]
    float *pb = lg + (size_t)NB * kChunk;              // [kChunk]
    unsigned *words = reinterpret_cast<unsigned *>(pb + kChunk);  // [nw]
    unsigned *wpre = words + nw;                                  // [nw]
    const PT *p2 = static_cast<const PT *>(p.p2);

    // Prologue, independent of the predecessor: the first chunk's biases.
    for (int i = threadIdx.x; i < min(R, kChunk); i += kLThreads) pb[i] = p.p_bias ? p.p_bias[r0 + i] : 0.f;
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) s_epoch = *reinterpret_cast<volatile unsigned *>(&p.ctrl->epoch);
    {
        const float4 *h4 = reinterpret_cast<const float4 *>(p.h);
        for (int i = threadIdx.x; i < p.B * p.r / 4; i += kLThreads) reinterpret_cast<float4 *>(hs)[i] = h4[i];
    }
    __syncthreads();

    for (int ch0 = 0; ch0 < R; ch0 += kChunk) {
        const int cn = min(kChunk, R - ch0);
        if (ch0 > 0) {
            for (int i = threadIdx.x; i < cn; i += kLThreads) pb[i] = p.p_bias ? p.p_bias[r0 + ch0 + i] : 0.f;
            __syncthreads();
        }
        for (int rr = warp; rr < cn; rr += RW * kLWarps) {
            const uint4 *wp[RW];
            bool ok[RW];
#pragma unroll
            for (int i = 0; i < RW; ++i) {
                const int row = rr + i * kLWarps;
                ok[i] = row < cn;
                wp[i] = reinterpret_cast<const uint4 *>(p2 + (size_t)(r0 + ch0 + (ok[i] ? row : rr)) * p.r);
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
                        const int cc = c0 + 32 * u;
                        if (ok[i] && cc < nch) v[i][u] = ld_stream(wp[i] + cc);
                    }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int cc = c0 + 32 * u;
                    if (cc < nch) {
#pragma unroll
                        for (int b = 0; b < NB; ++b) {
                            if (b < p.B) {
                                const float *hb = hs + (size_t)b * p.r + cc * EPC;
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
                        const int row = rr + i * kLWarps;
                        if (lane == 0 && ok[i]) {
                            const float l = sum + pb[row];
                            lg[b * kChunk + row] = l;
                            if (p.logits) p.logits[(size_t)b * p.F + r0 + ch0 + row] = l;
                        }
                    }
                }
            }
        }
        __syncthreads();
        // threshold + union -> this chunk's mask words
        for (int wd = warp; wd < (cn + 31) / 32; wd += kLWarps) {
            const int row = wd * 32 + lane;
            bool on = false;
            if (row < cn) {
#pragma unroll
                for (int b = 0; b < NB; ++b)
                    if (b < p.B) on = on || (lg[b * kChunk + row] > p.tau);
                on = on || r0 + ch0 + row < p.prefix;  // always-on prefix
                if (p.mask) p.mask[r0 + ch0 + row] = on ? 1 : 0;
            }
            const unsigned bits = __ballot_sync(0xffffffffu, on);
            if (lane == 0) words[ch0 / 32 + wd] = bits;
        }
        __syncthreads();
    }

    const unsigned epoch = s_epoch;
    const unsigned count = scan_words<kLThreads>(words, wpre, nw, red);
    const unsigned base = sum_before<kLThreads>(p.status, c, count, epoch, &p.ctrl->err, red);
    write_total(c, G, base, count, p.n_active, p.cap, &p.ctrl->err);
    emit_idx<kLThreads>(words, wpre, nw, r0, base, p.idx, p.cap);

    // Initialise the FFN output (b_down + residual) for the sparse kernel that
    // follows: this CTA's share of the B*d values.
    if (p.y) {
        const int nvec = p.B * p.d / 4;
        const int v0 = (int)((long long)nvec * c / G);
        const int v1 = (int)((long long)nvec * (c + 1) / G);
        float4 *y4 = reinterpret_cast<float4 *>(p.y);
        for (int v = v0 + threadIdx.x; v < v1; v += kLThreads) {
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
    scan_finish(p.ctrl, G, epoch);
}

// ---------------------------------------------------------------------------------
constexpr int kCThreads = 256;

__global__ void __launch_bounds__(kCThreads, 1) k_compact(const uint8_t *__restrict__ mask, int n, int *idx,
                                                          int *count_out, int cap, WsCtrl *ctrl,
                                                          unsigned long long *status)
{
    extern __shared__ __align__(16) unsigned cw[];
    __shared__ unsigned red[kCThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, G = gridDim.x;
    const int r0 = (int)((long long)n * c / G);
    const int R = (int)((long long)n * (c + 1) / G) - r0;
    const int nw = (R + 31) >> 5;
    unsigned *words = cw, *wpre = cw + nw;
    pdl_wait();
    pdl_trigger();
    const unsigned epoch = *reinterpret_cast<volatile unsigned *>(&ctrl->epoch);
    for (int wd = warp; wd < nw; wd += kCThreads / 32) {
        const int row = wd * 32 + lane;
        const bool on = row < R && mask[r0 + row] != 0;
        const unsigned bits = __ballot_sync(0xffffffffu, on);
        if (lane == 0) words[wd] = bits;
    }
    __syncthreads();
    const unsigned cnt = scan_words<kCThreads>(words, wpre, nw, red);
    const unsigned base = sum_before<kCThreads>(status, c, cnt, epoch, &ctrl->err, red);
    write_total(c, G, base, cnt, count_out, cap, &ctrl->err);
    emit_idx<kCThreads>(words, wpre, nw, r0, base, idx, cap);
    scan_finish(ctrl, G, epoch);
}

// The same compaction for masks of at most 64 Ki entries in one CTA.  Warp w owns
// bytes [2048 w, 2048 w + 2048) as 16 rounds of 128 bytes (lane l: bytes 4l..4l+3
// of the round), all loaded up front.  The warp totals are scanned across the
// block; then, round by round, a shuffle scan of the lanes' counts gives each
// lane its output slots, so a round's indices leave as one contiguous run.  No
// cross-CTA wait at all.
constexpr int kSmallThreads = 1024;
constexpr int kSmallMax = 2048 * (kSmallThreads / 32);  // capacity of the kernel
constexpr int kSmallUse = 8192;  // used up to here: beyond, the multi-CTA scan measured faster (GB300)

__global__ void __launch_bounds__(kSmallThreads, 1) k_compact_small(const uint8_t *__restrict__ mask, int n, int *idx,
                                                                    int *count_out, int cap, unsigned *err)
{
    __shared__ unsigned wsum[kSmallThreads / 32];
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned nib[16];  // per round: bit e set if byte 4 lane + e of the round is non-zero
    unsigned mine = 0;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const int o = 2048 * warp + 128 * r + 4 * lane;
        unsigned w = 0;
        if (o + 4 <= n) {
            w = *reinterpret_cast<const unsigned *>(mask + o);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (o + e < n) w |= (unsigned)mask[o + e] << (8 * e);
        }
        nib[r] = ((w & 0xffu) ? 1u : 0u) | ((w & 0xff00u) ? 2u : 0u) | ((w & 0xff0000u) ? 4u : 0u) |
                 ((w & 0xff000000u) ? 8u : 0u);
        mine += __popc(nib[r]);
    }
    unsigned tot = mine;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (lane == 0) wsum[warp] = tot;
    __syncthreads();
    if (warp == 0) {
        const unsigned x = wsum[lane];
        unsigned xi = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, xi, o);
            if (lane >= o) xi += y;
        }
        wsum[lane] = xi - x;  // exclusive over warps
        if (lane == 31) {
            unsigned all = xi;
            if (all > (unsigned)cap) {
                atomicOr(err, ERR_CAPACITY);
                all = (unsigned)cap;
            }
            *count_out = (int)all;
        }
    }
    __syncthreads();
    unsigned base = wsum[warp];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const unsigned c = __popc(nib[r]);
        unsigned incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        unsigned pos = base + incl - c;
        const int b0 = 2048 * warp + 128 * r + 4 * lane;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if ((nib[r] >> e) & 1u) {
                if (pos < (unsigned)cap) idx[pos] = b0 + e;
                ++pos;
            }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
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

// One CTA per SM (never more CTAs than SMs, so all are resident together),
// and never more CTAs than 32-neuron words.
int scan_grid(int n) { return std::max(1, std::min(sm_count(), (n + 31) / 32)); }

template <typename PT>
static cudaError_t pred_logits_nb(const PredParams &p, cudaStream_t s)
{
    const int G = scan_grid(p.F);
    const int nw = ((p.F + G - 1) / G + 31) / 32 + 1;
    const size_t smem = ((size_t)p.B * p.r + (size_t)9 * kChunk) * sizeof(float) + (size_t)2 * nw * sizeof(unsigned);
    void (*k)(PredParams);
    if (p.B <= 1)
        k = k_pred_logits<PT, 1>;
    else if (p.B <= 2)
        k = k_pred_logits<PT, 2>;
    else if (p.B <= 4)
        k = k_pred_logits<PT, 4>;
    else
        k = k_pred_logits<PT, 8>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(G), dim3(kLThreads), smem, s, p);
}

cudaError_t launch_pred_logits(int ptype, const PredParams &p, cudaStream_t s)
{
    return ptype == 1 ? pred_logits_nb<__half>(p, s) : pred_logits_nb<float>(p, s);
}

cudaError_t launch_compact(const uint8_t *mask, int n, int *idx, int *count, int cap, WsCtrl *ctrl,
                           unsigned long long *status, cudaStream_t s)
{
    if (n <= kSmallUse && n <= kSmallMax && ((uintptr_t)mask & 3) == 0)
        return launch_pdl(k_compact_small, dim3(1), dim3(kSmallThreads), 0, s, mask, n, idx, count, cap, &ctrl->err);
    const int G = scan_grid(n);
    const int nw = ((n + G - 1) / G + 31) / 32 + 1;
    const size_t smem = (size_t)2 * nw * sizeof(unsigned);
    cudaError_t e = cudaFuncSetAttribute(k_compact, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_compact, dim3(G), dim3(kCThreads), smem, s, mask, n, idx, count, cap, ctrl, status);
}

}  // namespace pi
