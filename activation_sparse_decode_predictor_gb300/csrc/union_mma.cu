// Batched decode (2..8 tokens) through one sparse FFN layer, on tensor cores.
//
// With several tokens in flight the active rows are the union of the tokens'
// predicted sets and every token is computed on every union row (PowerInfer
// summary page, "技术贡献" technical contributions: neuron-aware sparse
// operators; the batch case turns the gather-GEMV into a small dense
// contraction over the gathered rows).  For the union list idx[0..n):
//   z[k][b]  = W_act[idx_k] . x_b  (and u[k][b] = W_up[idx_k] . x_b, ReGLU)
//   a[k][b]  = act(z + b_act[idx_k]) (times u)
//   y_b     += sum_k a[k][b] * W_down[idx_k]
// Both contractions run on mma.sync m16n8k16 (fp16 in, fp32 accumulate).
//
// Precision.  The fp32 operands x and a are each split into two fp16 terms
// (hi = fp16(v), lo = fp16(v - hi)) after a per-token power-of-two scaling that
// puts the token's largest magnitude in [2^10, 2^11); the hi and lo terms are
// separate columns of the n8 operand, so products carry about 22 bits of the
// fp32 operand.  fp16 weights enter exactly.  Q4_0 up-projection weights enter
// as the exact integers q - 8 with the block scale applied in fp32 after each
// 32-wide block; Q4_0 down-projection weights are dequantised to fp16 in
// registers (scale * (q - 8), one rounding, relative error <= 2^-11).
//
// Kernels (one stream, chained with programmatic dependent launch):
//   k_union_prep  x -> fp16 hi/lo fragments in mma B-operand order, exponents.
//   k_union_up    persistent, one CTA per SM.  Work unit = 16 union rows x one
//                 chunk of d_model of one matrix; units are ordered chunk-major
//                 and dealt out to CTAs in contiguous ranges (balanced to one
//                 unit).  A producer warp streams the 16 rows of each unit into a
//                 shared-memory ring with 1-D bulk copies; consumer warp w takes
//                 units w, w+8, ...  Partial sums of a tile are added into a
//                 per-tile buffer; the warp that completes a tile applies the
//                 activation and writes a in the down kernel's fragment order.
//   k_union_down  persistent.  Work unit = 16 union rows x one column block of
//                 W_down; CTAs take contiguous ranges, each consumer warp owns a
//                 fixed column slice of the block and accumulates in registers,
//                 then adds its slice into y with vector atomics when the column
//                 block changes.
#include <cuda_fp16.h>

#include "ffn_rows.cuh"
#include "internal.h"
#include "pi.h"

namespace pi {

namespace {

constexpr int kUW = 8;                   // consumer warps
constexpr int kUThreads = kUW * 32 + 32; // + producer warp
constexpr int kUMaxStages = 32;
constexpr size_t kHdrU = 2048;           // mbarriers + the producer's neuron-id table
static_assert(2 * kUMaxStages * 8 + 2 * 128 * 4 <= kHdrU, "header region too small");
constexpr size_t kSmemBudget = 225 * 1024;
constexpr int kScaleExp = 10;            // scaled operands have their maximum in [2^10, 2^11)
constexpr int kBatchJobs = 8;            // producer reads idx for 8 jobs (128 rows) at a time

// Up-projection chunks (elements of d_model per unit) and shared-memory rows.
constexpr int kKsF16 = 512;
constexpr int kKsQ4 = 1024;
constexpr int kRsF16Up = kKsF16 * 2 + 64;  // 1088: 16-byte row reads of 8 lanes hit distinct banks
constexpr int kRsQ4 = 528;                 // 512 code bytes + 16: 32-bit row reads conflict-free
constexpr int kSsQ4 = 80;                  // 64 scale bytes + 16
// Down-projection column blocks.
constexpr int kCwF16 = 512;
constexpr int kCwQ4 = 1024;
constexpr int kRsF16Dn = kCwF16 * 2 + 16;  // 1040: ldmatrix rows hit distinct banks

constexpr uint32_t up_stage_bytes(bool q4) { return q4 ? 16u * (kRsQ4 + kSsQ4) : 16u * kRsF16Up; }
constexpr uint32_t dn_stage_bytes(bool q4) { return q4 ? 16u * (kRsQ4 + kSsQ4) : 16u * kRsF16Dn; }

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t pack_h2(__half lo, __half hi)
{
    return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// fp32 v -> (hi, lo) fp16 with hi + lo = v to about 22 bits.
__device__ __forceinline__ void split_f16(float v, __half &hi, __half &lo)
{
    hi = __float2half_rn(v);
    lo = __float2half_rn(v - __half2float(hi));
}

// Exponent e with max * 2^-e in [2^10, 2^11) (0 for an all-zero or non-finite maximum).
__device__ __forceinline__ int scale_exp(float mx)
{
    if (!(mx > 0.f) || !isfinite(mx)) return 0;
    int e = ilogbf(mx) - kScaleExp;
    return e < -120 ? -120 : (e > 120 ? 120 : e);
}

// Nibble pairs of a 32-bit word -> fp16x2 of (q - 8): 0x6400 | q is the fp16 1024 + q.
__device__ __forceinline__ uint32_t q4_pair(uint32_t w)
{
    const uint32_t v = (w & 0x000F000Fu) | 0x64006400u;
    const __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&v), __half2half2(__ushort_as_half(0x6408)));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// Position along d_model of half h of register r of lane-quad t in step s of the
// B-operand fragment (must match how the up kernel reads its weight rows).
//   fp16: lane t reads 8 consecutive weights 32s + 8t .. +7 of a row; register r
//         holds weights 2r, 2r+1 of those.
//   Q4_0: lane t reads code bytes 4t..4t+3 of block s; register r takes nibble
//         (r & 1) of bytes 4t + (r >> 1) (half 0) and 4t + (r >> 1) + 2 (half 1);
//         byte e of a block holds element e (low nibble) and e + 16 (high).
__device__ __forceinline__ int frag_k(bool q4, int s, int t, int r, int h)
{
    if (q4) return 32 * s + 4 * t + (r >> 1) + 2 * h + 16 * (r & 1);
    return 32 * s + 8 * t + 2 * r + h;
}

// ------------------------------------------------------------------------------------
// x -> xf[step][group][lane][4] (fp16x2).  Group layout: B <= 4: one group, column
// g < 4 is hi of token g, column g >= 4 lo of token g - 4.  B > 4: group 0 hi,
// group 1 lo, column g = token g.  Columns of absent tokens are zero.
__global__ void __launch_bounds__(256) k_union_prep(const float *__restrict__ x, int B, int d, int q4,
                                                     uint32_t *__restrict__ xf, int *__restrict__ uexp,
                                                     unsigned *__restrict__ amax)
{
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    const int NG = B > 4 ? 2 : 1;
    __shared__ float red[8];
    float m = 0.f;
    const bool live = b < B;
    if (live)
        for (int i = threadIdx.x; i < d; i += blockDim.x) m = fmaxf(m, fabsf(x[(size_t)b * d + i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
    const int e = live ? scale_exp(m) : 0;
    if (threadIdx.x == 0) {
        uexp[b] = e;
        amax[b] = 0u;
    }
    if (NG == 1 && b >= 4) return;  // those columns hold the lo terms of tokens 0..3
    const int ghi = b, glo = NG == 1 ? b + 4 : b;
    const int grp_lo = NG == 1 ? 0 : 1;
    const int steps = (d + 31) / 32;
    for (int v = threadIdx.x; v < steps * 16; v += blockDim.x) {
        const int s = v >> 4, t = (v >> 2) & 3, r = v & 3;
        __half hi[2], lo[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int k = frag_k(q4 != 0, s, t, r, h);
            const float xv = (live && k < d) ? ldexpf(x[(size_t)b * d + k], -e) : 0.f;
            split_f16(xv, hi[h], lo[h]);
        }
        xf[(((size_t)s * NG + 0) * 32 + ghi * 4 + t) * 4 + r] = pack_h2(hi[0], hi[1]);
        xf[(((size_t)s * NG + grp_lo) * 32 + glo * 4 + t) * 4 + r] = pack_h2(lo[0], lo[1]);
    }
}

// ------------------------------------------------------------------------------------
// Producer warp shared by the up and down kernels: job j of the CTA's range copies
// the 16 rows idx[16 * tile(j) + r] (rows past n repeat row n - 1, whose values are
// finite and are multiplied by zero or discarded) into stage j % nstages.  The
// neuron ids are read one batch of 8 jobs ahead so that their latency overlaps
// the copies of the batch before.
template <typename JobTile, typename JobBytes, typename CopyRow>
__device__ void produce_rows(const SparseParams &p, int n, int cnt, long long u0, int nstages, uint64_t *full,
                             uint64_t *empty, int *tab, JobTile job_tile, JobBytes job_bytes, CopyRow copy_row)
{
    constexpr int kNone = -2147483647 - 1;  // no job at this position
    const int lane = threadIdx.x & 31;
    unsigned *err = &p.ctrl->err;
    auto fetch = [&](int jb, int (&out)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int v = lane + 32 * i;
            const int jj = jb + (v >> 4);
            out[i] = kNone;
            if (jj < cnt) {
                int row = 16 * job_tile(u0 + jj) + (v & 15);
                row = row < n ? row : n - 1;
                out[i] = __ldcg(p.idx + row);
            }
        }
    };
    auto store = [&](int buf, const int (&in)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int j = in[i];
            if (j == kNone) {
                j = 0;
            } else if (j < 0 || j >= p.F) {
                atomicOr(err, ERR_INDEX);
                j = 0;
            }
            tab[buf * 128 + lane + 32 * i] = j;
        }
    };
    int pre[4];
    fetch(0, pre);
    store(0, pre);
    __syncwarp();
    bool failed = false;
    int j = 0;
    for (int jb = 0; jb < cnt && !failed; jb += kBatchJobs) {
        const int buf = (jb / kBatchJobs) & 1;
        fetch(jb + kBatchJobs, pre);
        const int je = min(cnt, jb + kBatchJobs);
        for (j = jb; j < je; ++j) {
            const int s = j % nstages;
            if (j >= nstages) {
                bool ok = true;
                if (lane == 0) ok = mbar_wait(&empty[s], (unsigned)((j / nstages) - 1) & 1u, err);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    failed = true;
                    break;
                }
            }
            if (lane == 0) mbar_arrive_expect_tx(&full[s], 16u * job_bytes(u0 + j));
            __syncwarp();
            if (lane < 16) copy_row(u0 + j, s, lane, tab[buf * 128 + (j - jb) * 16 + lane], &full[s]);
        }
        __syncwarp();
        store(buf ^ 1, pre);
        __syncwarp();
    }
    if (failed && lane == 0) {
        // never leave the CTA with bulk copies in flight into its shared memory
        for (int s = 0; s < nstages && s < j; ++s) {
            const int last = s + ((j - 1 - s) / nstages) * nstages;
            mbar_wait(&full[s], (unsigned)(last / nstages) & 1u, err);
        }
    }
}

// ------------------------------------------------------------------------------------
template <int WT, bool GATED, int NG>
__global__ void __launch_bounds__(kUThreads, 1) k_union_up(SparseParams p, int nstages)
{
    constexpr bool Q4 = WT == PI_Q4_0;
    constexpr int KS = Q4 ? kKsQ4 : kKsF16;   // elements of d_model per unit
    constexpr int M = GATED ? 2 : 1;          // matrices per row tile
    constexpr uint32_t SB = up_stage_bytes(Q4);
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kUMaxStages;
    int *tab = reinterpret_cast<int *>(empty + kUMaxStages);  // [2][128]
    uint8_t *stages = smem + kHdrU;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = p.d, F = p.F;
    unsigned *err = &p.ctrl->err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();

    int n = __ldcg(p.n_active);
    n = n < 0 ? 0 : (n > F ? F : n);
    const int T = (n + 15) >> 4;
    const int C = (d + KS - 1) / KS;
    const long long per = (long long)T * M;
    const long long U = per * C;
    const int G = gridDim.x;
    const long long u0 = U * blockIdx.x / G, u1 = U * (blockIdx.x + 1) / G;
    const int cnt = (int)(u1 - u0);
    if (cnt <= 0) return;

    if (warp == kUW) {
        auto job_tile = [&](long long u) { return (int)((u % per) / M); };
        auto job_bytes = [&](long long u) {
            const int len = min(KS, d - (int)(u / per) * KS);
            return Q4 ? (uint32_t)(len / 2 + len / 16) : (uint32_t)len * 2u;
        };
        auto copy_row = [&](long long u, int s, int r, int jn, uint64_t *bar) {
            const int c = (int)(u / per);
            const int m = (int)(u % M);
            const int k0 = c * KS, len = min(KS, d - k0);
            const uint8_t *W = (GATED && m == 1) ? p.w_up : p.w_act;
            uint8_t *st = stages + (size_t)s * SB;
            if constexpr (Q4) {
                bulk_g2s(st + r * kRsQ4, W + (size_t)jn * (d / 2) + k0 / 2, (uint32_t)(len / 2), bar);
                bulk_g2s(st + 16 * kRsQ4 + r * kSsQ4, W + (size_t)F * (d / 2) + (size_t)jn * (d / 16) + k0 / 16,
                         (uint32_t)(len / 16), bar);
            } else {
                bulk_g2s(st + r * kRsF16Up, W + ((size_t)jn * d + k0) * 2, (uint32_t)len * 2u, bar);
            }
        };
        produce_rows(p, n, cnt, u0, nstages, full, empty, tab, job_tile, job_bytes, copy_row);
        return;
    }

    // ---------------------------------- consumer warps ----------------------------------
    const int g = lane >> 2, t = lane & 3;
    // exponents of the two tokens whose sums this lane adds (tokens 2t, 2t+1)
    const int tk0 = 2 * t;
    const float sc0 = tk0 < 8 ? ldexpf(1.f, __ldcg(p.uexp + tk0)) : 0.f;
    const float sc1 = tk0 + 1 < 8 ? ldexpf(1.f, __ldcg(p.uexp + tk0 + 1)) : 0.f;
    const int B = p.B;

    for (int jj = warp; jj < cnt; jj += kUW) {
        const int s = jj % nstages;
        const long long u = u0 + jj;
        const int c = (int)(u / per);
        const int tile = (int)((u % per) / M);
        const int m = (int)(u % M);
        if (!mbar_wait(&full[s], (unsigned)(jj / nstages) & 1u, err)) break;
        const uint8_t *st = stages + (size_t)s * SB;
        const int k0 = c * KS, len = min(KS, d - k0);
        float acc[NG][4];
#pragma unroll
        for (int q = 0; q < NG; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
        const uint8_t *xfp = reinterpret_cast<const uint8_t *>(p.xf) + ((size_t)(k0 / 32) * NG * 32 + lane) * 16;
        if constexpr (!Q4) {
            const int nsteps = (len + 31) / 32;
            const uint8_t *ra = st + g * kRsF16Up + 16 * t;
            const uint8_t *rb = ra + 8 * kRsF16Up;
#pragma unroll 4
            for (int q = 0; q < nsteps; ++q) {
                uint4 a0 = *reinterpret_cast<const uint4 *>(ra + q * 64);
                uint4 a1 = *reinterpret_cast<const uint4 *>(rb + q * 64);
                if (q * 32 + 8 * t >= len) a0 = a1 = make_uint4(0u, 0u, 0u, 0u);  // ragged end of d_model
#pragma unroll
                for (int gr = 0; gr < NG; ++gr) {
                    const uint4 bx = ldg_nc_v4(xfp + ((size_t)q * NG + gr) * 512);
                    mma16816(acc[gr], a0.x, a1.x, a0.y, a1.y, bx.x, bx.y);
                    mma16816(acc[gr], a0.z, a1.z, a0.w, a1.w, bx.z, bx.w);
                }
            }
        } else {
            const int nsteps = len / 32;
            const uint8_t *ca = st + g * kRsQ4 + 4 * t;
            const uint8_t *cb = ca + 8 * kRsQ4;
            const __half *sa = reinterpret_cast<const __half *>(st + 16 * kRsQ4 + g * kSsQ4);
            const __half *sb = reinterpret_cast<const __half *>(st + 16 * kRsQ4 + (g + 8) * kSsQ4);
#pragma unroll 4
            for (int q = 0; q < nsteps; ++q) {
                const uint32_t w0 = *reinterpret_cast<const uint32_t *>(ca + q * 16);
                const uint32_t w1 = *reinterpret_cast<const uint32_t *>(cb + q * 16);
                const float s0 = __half2float(sa[q]), s1 = __half2float(sb[q]);
                const uint32_t p0 = q4_pair(w0), p1 = q4_pair(w0 >> 4), p2 = q4_pair(w0 >> 8), p3 = q4_pair(w0 >> 12);
                const uint32_t r0 = q4_pair(w1), r1 = q4_pair(w1 >> 4), r2 = q4_pair(w1 >> 8), r3 = q4_pair(w1 >> 12);
#pragma unroll
                for (int gr = 0; gr < NG; ++gr) {
                    const uint4 bx = ldg_nc_v4(xfp + ((size_t)q * NG + gr) * 512);
                    float tmp[4] = {0.f, 0.f, 0.f, 0.f};
                    mma16816(tmp, p0, r0, p1, r1, bx.x, bx.y);
                    mma16816(tmp, p2, r2, p3, r3, bx.z, bx.w);
                    acc[gr][0] = fmaf(s0, tmp[0], acc[gr][0]);
                    acc[gr][1] = fmaf(s0, tmp[1], acc[gr][1]);
                    acc[gr][2] = fmaf(s1, tmp[2], acc[gr][2]);
                    acc[gr][3] = fmaf(s1, tmp[3], acc[gr][3]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);

        // hi + lo columns -> this lane's sums for tokens 2t, 2t+1 (lanes t < 2 when NG == 1)
        float z[4];
        bool has;
        if constexpr (NG == 1) {
#pragma unroll
            for (int i = 0; i < 4; ++i) z[i] = acc[0][i] + __shfl_xor_sync(0xffffffffu, acc[0][i], 2);
            has = t < 2;
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) z[i] = acc[0][i] + acc[1][i];
            has = true;
        }
        float *zb = p.zbuf + ((size_t)tile * 2 + m) * 128;
        if (has) {
            atomicAdd(reinterpret_cast<float2 *>(zb + g * 8 + tk0), make_float2(z[0] * sc0, z[1] * sc1));
            atomicAdd(reinterpret_cast<float2 *>(zb + (g + 8) * 8 + tk0), make_float2(z[2] * sc0, z[3] * sc1));
        }
        __threadfence();
        __syncwarp();
        unsigned old = 0;
        if (lane == 0) old = atomicAdd(p.ucnt + tile, 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old != (unsigned)(C * M - 1)) continue;

        // ---- this warp completed the tile: activation, fragment-order store, reset ----
        __threadfence();
        const int row = lane >> 1, tb = 4 * (lane & 1);
        float *z0p = p.zbuf + ((size_t)tile * 2 + 0) * 128 + row * 8 + tb;
        float *z1p = p.zbuf + ((size_t)tile * 2 + 1) * 128 + row * 8 + tb;
        const float4 zg = __ldcg(reinterpret_cast<const float4 *>(z0p));
        float4 zu = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (GATED) zu = __ldcg(reinterpret_cast<const float4 *>(z1p));
        __stcg(reinterpret_cast<float4 *>(z0p), make_float4(0.f, 0.f, 0.f, 0.f));
        if constexpr (GATED) __stcg(reinterpret_cast<float4 *>(z1p), make_float4(0.f, 0.f, 0.f, 0.f));
        const int k = 16 * tile + row;
        bool valid = k < n;
        float bias = 0.f;
        if (valid) {
            // an out-of-range neuron id (flagged by the producer, which copied row 0
            // in its place) contributes nothing
            const int jn = __ldcg(p.idx + k);
            valid = jn >= 0 && jn < F;
            if (valid && p.b_act) bias = p.b_act[jn];
        }
        const float zgv[4] = {zg.x, zg.y, zg.z, zg.w};
        const float zuv[4] = {zu.x, zu.y, zu.z, zu.w};
        float mx[4];
        const int tq = (row & 7) >> 1, jx = (row & 1) + 2 * (row >> 3);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float a = 0.f;
            if (valid && tb + i < B) {
                a = activate(p.act, zgv[i] + bias);
                if constexpr (GATED) a *= zuv[i];
            }
            p.act_ws[(((size_t)tile * 4 + tq) * 8 + tb + i) * 4 + jx] = a;
            mx[i] = fabsf(a);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int o = 2; o < 32; o <<= 1) mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], o));
        if (lane < 2)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (mx[i] > 0.f) atomicMax(p.amax + tb + i, __float_as_uint(mx[i]));
        if (lane == 0) p.ucnt[tile] = 0u;
    }
}

// ------------------------------------------------------------------------------------
template <int WT, int NG>
__global__ void __launch_bounds__(kUThreads, 1) k_union_down(SparseParams p, int nstages)
{
    constexpr bool Q4 = WT == PI_Q4_0;
    constexpr int CW = Q4 ? kCwQ4 : kCwF16;   // columns of a block
    constexpr int IT = Q4 ? 8 : 4;            // 16-column tiles per warp
    constexpr int WC = IT * 16;               // columns per warp
    constexpr uint32_t SB = dn_stage_bytes(Q4);
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kUMaxStages;
    int *tab = reinterpret_cast<int *>(empty + kUMaxStages);
    uint8_t *stages = smem + kHdrU;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = p.d, F = p.F;
    unsigned *err = &p.ctrl->err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kUW);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_trigger();

    // idx and n_active were complete before the up kernel passed its own wait,
    // and the weights are constant, so the producer starts before the wait.
    int n = __ldcg(p.n_active);
    n = n < 0 ? 0 : (n > F ? F : n);
    const int T = (n + 15) >> 4;
    const int NCB = (d + CW - 1) / CW;
    const long long U = (long long)NCB * T;
    const int G = gridDim.x;
    const long long u0 = U * blockIdx.x / G, u1 = U * (blockIdx.x + 1) / G;
    const int cnt = (int)(u1 - u0);
    if (cnt <= 0) return;

    if (warp == kUW) {
        auto job_tile = [&](long long u) { return (int)(u % T); };
        auto job_bytes = [&](long long u) {
            const int nc = min(CW, d - (int)(u / T) * CW);
            return Q4 ? (uint32_t)(nc / 2 + nc / 16) : (uint32_t)nc * 2u;
        };
        auto copy_row = [&](long long u, int s, int r, int jn, uint64_t *bar) {
            const int cb = (int)(u / T);
            const int c0 = cb * CW, nc = min(CW, d - c0);
            uint8_t *st = stages + (size_t)s * SB;
            if constexpr (Q4) {
                bulk_g2s(st + r * kRsQ4, p.w_down + (size_t)jn * (d / 2) + c0 / 2, (uint32_t)(nc / 2), bar);
                bulk_g2s(st + 16 * kRsQ4 + r * kSsQ4,
                         p.w_down + (size_t)F * (d / 2) + (size_t)jn * (d / 16) + c0 / 16, (uint32_t)(nc / 16), bar);
            } else {
                bulk_g2s(st + r * kRsF16Dn, p.w_down + ((size_t)jn * d + c0) * 2, (uint32_t)nc * 2u, bar);
            }
        };
        produce_rows(p, n, cnt, u0, nstages, full, empty, tab, job_tile, job_bytes, copy_row);
        return;
    }

    // ---------------------------------- consumer warps ----------------------------------
    pdl_wait();  // activations and their maxima come from the up kernel
    const int g = lane >> 2, t = lane & 3;
    // the activations of token b were scaled by 2^-e_b (e_b from the largest |a|)
    const int tokB = NG == 1 ? (g & 3) : g;  // token of this lane's B-operand column
    const float inv = ldexpf(1.f, -scale_exp(__uint_as_float(__ldcg(p.amax + tokB))));
    const float sc0 = ldexpf(1.f, scale_exp(__uint_as_float(__ldcg(p.amax + 2 * t))));
    const float sc1 = ldexpf(1.f, scale_exp(__uint_as_float(__ldcg(p.amax + 2 * t + 1))));
    float *fb = reinterpret_cast<float *>(stages + (size_t)nstages * SB) + (size_t)warp * 8 * WC;
    const int B = p.B;

    float acc[IT][NG][4];
    auto zero_acc = [&]() {
#pragma unroll
        for (int i = 0; i < IT; ++i)
#pragma unroll
            for (int q = 0; q < NG; ++q) acc[i][q][0] = acc[i][q][1] = acc[i][q][2] = acc[i][q][3] = 0.f;
    };
    // Adds this warp's slice of column block cb into y (through shared memory, so
    // that the atomics are 16-byte vectors).
    auto flush = [&](int cb) {
        const int c0 = cb * CW + warp * WC;
#pragma unroll
        for (int i = 0; i < IT; ++i) {
            float v[4];
            if constexpr (NG == 1) {
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = acc[i][0][e] + __shfl_xor_sync(0xffffffffu, acc[i][0][e], 2);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = acc[i][0][e] + acc[i][1][e];
            }
            if (NG == 2 || t < 2) {
                int col0, col1;  // columns of rows g and g + 8 of tile i within the warp slice
                if constexpr (Q4) {
                    const int h = i >> 2, mm = i & 3;
                    col0 = 64 * h + 32 * (g >> 2) + 4 * (g & 3) + mm;
                    col1 = col0 + 16;
                } else {
                    col0 = 16 * i + g;
                    col1 = col0 + 8;
                }
                fb[(2 * t) * WC + col0] = v[0] * sc0;
                fb[(2 * t + 1) * WC + col0] = v[1] * sc1;
                fb[(2 * t) * WC + col1] = v[2] * sc0;
                fb[(2 * t + 1) * WC + col1] = v[3] * sc1;
            }
        }
        __syncwarp();
        for (int e = lane; e < B * (WC / 4); e += 32) {
            const int tok = e / (WC / 4), c4 = e % (WC / 4);
            const int col = c0 + 4 * c4;
            if (col < d)
                atomicAdd(reinterpret_cast<float4 *>(p.y + (size_t)tok * d + col),
                          *reinterpret_cast<const float4 *>(fb + tok * WC + 4 * c4));
        }
        __syncwarp();
    };

    zero_acc();
    int cur = -1;
    for (int jj = 0; jj < cnt; ++jj) {
        const int s = jj % nstages;
        const long long u = u0 + jj;
        const int cb = (int)(u / T), tile = (int)(u % T);
        if (cb != cur) {
            if (cur >= 0) {
                flush(cur);
                zero_acc();
            }
            cur = cb;
        }
        if (!mbar_wait(&full[s], (unsigned)(jj / nstages) & 1u, err)) {
            cur = -1;
            break;
        }
        const uint8_t *st = stages + (size_t)s * SB;
        const bool live = cb * CW + warp * WC < d;
        if (live) {
            // B operand: a[k][tok] for k = 2t, 2t+1, 2t+8, 2t+9 of this tile, split hi/lo
            const float4 av = __ldcg(reinterpret_cast<const float4 *>(p.act_ws) + ((size_t)tile * 4 + t) * 8 + tokB);
            __half h0, h1, h2, h3, l0, l1, l2, l3;
            split_f16(av.x * inv, h0, l0);
            split_f16(av.y * inv, h1, l1);
            split_f16(av.z * inv, h2, l2);
            split_f16(av.w * inv, h3, l3);
            uint32_t bf[NG][2];
            if constexpr (NG == 1) {
                const bool lo = g >= 4;
                bf[0][0] = lo ? pack_h2(l0, l1) : pack_h2(h0, h1);
                bf[0][1] = lo ? pack_h2(l2, l3) : pack_h2(h2, h3);
            } else {
                bf[0][0] = pack_h2(h0, h1);
                bf[0][1] = pack_h2(h2, h3);
                bf[NG - 1][0] = pack_h2(l0, l1);
                bf[NG - 1][1] = pack_h2(l2, l3);
            }
            if constexpr (!Q4) {
                // ldmatrix.trans: lane l addresses row (l & 7) + 8 * (l >> 4) of the
                // stage, columns 16 i + 8 * ((l >> 3) & 1) of the warp slice
                const int mq = lane >> 3, rr = lane & 7;
                const uint32_t base = smem_u32(st) + (uint32_t)((rr + 8 * (mq >> 1)) * kRsF16Dn) +
                                      (uint32_t)((warp * WC + 8 * (mq & 1)) * 2);
#pragma unroll
                for (int i = 0; i < IT; ++i) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_trans(base + 32u * i, a0, a1, a2, a3);
#pragma unroll
                    for (int q = 0; q < NG; ++q) mma16816(acc[i][q], a0, a1, a2, a3, bf[q][0], bf[q][1]);
                }
            } else {
                const uint8_t *codes = st + 64 * warp + 4 * g;
                const uint8_t *scl = st + 16 * kRsQ4;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t wa = *reinterpret_cast<const uint32_t *>(codes + (2 * t) * kRsQ4 + 32 * h);
                    const uint32_t wb = *reinterpret_cast<const uint32_t *>(codes + (2 * t + 1) * kRsQ4 + 32 * h);
                    const uint32_t wc = *reinterpret_cast<const uint32_t *>(codes + (2 * t + 8) * kRsQ4 + 32 * h);
                    const uint32_t wd = *reinterpret_cast<const uint32_t *>(codes + (2 * t + 9) * kRsQ4 + 32 * h);
                    const int blk = 4 * warp + 2 * h + (g >> 2);
                    const __half2 sA = __halves2half2(*reinterpret_cast<const __half *>(scl + (2 * t) * kSsQ4 + 2 * blk),
                                                      *reinterpret_cast<const __half *>(scl + (2 * t + 1) * kSsQ4 + 2 * blk));
                    const __half2 sB = __halves2half2(*reinterpret_cast<const __half *>(scl + (2 * t + 8) * kSsQ4 + 2 * blk),
                                                      *reinterpret_cast<const __half *>(scl + (2 * t + 9) * kSsQ4 + 2 * blk));
                    const uint32_t x01 = __byte_perm(wa, wb, 0x5410), y01 = __byte_perm(wa, wb, 0x7632);
                    const uint32_t x89 = __byte_perm(wc, wd, 0x5410), y89 = __byte_perm(wc, wd, 0x7632);
#pragma unroll
                    for (int mm = 0; mm < 4; ++mm) {
                        const uint32_t v01 = (mm < 2 ? x01 : y01) >> (8 * (mm & 1));
                        const uint32_t v89 = (mm < 2 ? x89 : y89) >> (8 * (mm & 1));
                        uint32_t a[4];
                        const uint32_t q0 = q4_pair(v01), q1 = q4_pair(v01 >> 4);
                        const uint32_t q2 = q4_pair(v89), q3 = q4_pair(v89 >> 4);
                        const __half2 d0 = __hmul2(*reinterpret_cast<const __half2 *>(&q0), sA);
                        const __half2 d1 = __hmul2(*reinterpret_cast<const __half2 *>(&q1), sA);
                        const __half2 d2 = __hmul2(*reinterpret_cast<const __half2 *>(&q2), sB);
                        const __half2 d3 = __hmul2(*reinterpret_cast<const __half2 *>(&q3), sB);
                        a[0] = *reinterpret_cast<const uint32_t *>(&d0);
                        a[1] = *reinterpret_cast<const uint32_t *>(&d1);
                        a[2] = *reinterpret_cast<const uint32_t *>(&d2);
                        a[3] = *reinterpret_cast<const uint32_t *>(&d3);
#pragma unroll
                        for (int q = 0; q < NG; ++q)
                            mma16816(acc[4 * h + mm][q], a[0], a[1], a[2], a[3], bf[q][0], bf[q][1]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (cur >= 0 && cur * CW + warp * WC < d) flush(cur);
}

template <typename K>
cudaError_t set_smem(K kern, size_t bytes)
{
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int WT, bool GATED, int NG>
cudaError_t launch_up(const SparseParams &p, cudaStream_t s)
{
    constexpr uint32_t SB = up_stage_bytes(WT == PI_Q4_0);
    const size_t fit = (kSmemBudget - kHdrU) / SB;
    const int ns = (int)(fit < (size_t)kUMaxStages ? fit : (size_t)kUMaxStages);
    const size_t smem = kHdrU + (size_t)ns * SB;
    static bool once = false;
    if (!once) {
        cudaError_t e = set_smem(k_union_up<WT, GATED, NG>, smem);
        if (e != cudaSuccess) return e;
        once = true;
    }
    return launch_pdl(k_union_up<WT, GATED, NG>, dim3(sm_count()), dim3(kUThreads), smem, s, p, ns);
}

template <int WT, int NG>
cudaError_t launch_down(const SparseParams &p, cudaStream_t s)
{
    constexpr bool Q4 = WT == PI_Q4_0;
    constexpr uint32_t SB = dn_stage_bytes(Q4);
    constexpr size_t fbytes = (size_t)kUW * 8 * (Q4 ? 128 : 64) * 4;
    const size_t fit = (kSmemBudget - kHdrU - fbytes) / SB;
    const int ns = (int)(fit < (size_t)kUMaxStages ? fit : (size_t)kUMaxStages);
    const size_t smem = kHdrU + (size_t)ns * SB + fbytes;
    static bool once = false;
    if (!once) {
        cudaError_t e = set_smem(k_union_down<WT, NG>, smem);
        if (e != cudaSuccess) return e;
        once = true;
    }
    return launch_pdl(k_union_down<WT, NG>, dim3(sm_count()), dim3(kUThreads), smem, s, p, ns);
}

template <int WT>
cudaError_t launch_union_wt(int gated, const SparseParams &p, cudaStream_t s)
{
    cudaError_t e;
    if (p.B > 4)
        e = gated ? launch_up<WT, true, 2>(p, s) : launch_up<WT, false, 2>(p, s);
    else
        e = gated ? launch_up<WT, true, 1>(p, s) : launch_up<WT, false, 1>(p, s);
    if (e != cudaSuccess) return e;
    return p.B > 4 ? launch_down<WT, 2>(p, s) : launch_down<WT, 1>(p, s);
}

}  // namespace

cudaError_t launch_sparse_union(int wtype, int gated, const SparseParams &p, cudaStream_t s)
{
    if (wtype != PI_F16 && wtype != PI_Q4_0) return cudaErrorNotSupported;
    if (p.B < 2 || p.B > 8) return cudaErrorInvalidValue;
    cudaError_t e = launch_pdl(k_union_prep, dim3(8), dim3(256), 0, s, p.x, p.B, p.d, wtype == PI_Q4_0 ? 1 : 0,
                               p.xf, p.uexp, p.amax);
    if (e != cudaSuccess) return e;
    return wtype == PI_Q4_0 ? launch_union_wt<PI_Q4_0>(gated, p, s) : launch_union_wt<PI_F16>(gated, p, s);
}

}  // namespace pi
