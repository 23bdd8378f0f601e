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
// Data movement.  Rows are gathered by a producer warp with 1-D bulk (TMA)
// copies, one per row piece, into a shared-memory ring.  A bulk copy costs a
// roughly fixed issue time (about 45 ns per copy per SM measured on GB300), so
// pieces are kept at 2-4 KB: smaller pieces cap the stream well below HBM
// bandwidth whatever the format.
//
// Kernels (one stream, chained with programmatic dependent launch):
//   k_union_prep  x -> fp16 hi/lo fragments in mma B-operand order, exponents.
//   k_union_up    persistent, one CTA per SM.  Work unit = 16 union rows x one
//                 chunk of d_model (2048 fp16 weights; 4096 Q4_0 weights at
//                 2-4 tokens, 2048 at 5-8 tokens: up_ks) of one
//                 matrix; units are ordered chunk-major and dealt out to CTAs in
//                 contiguous ranges.  The 8 consumer warps split each unit's
//                 chunk and leave their partial sums in one of 4 shared-memory
//                 slots (mbarrier-tracked); a dedicated reducing warp sums the
//                 slots and adds them into per-tile buffers, batching up to 4
//                 units per memory fence, so no consumer ever waits on global
//                 atomics; the unit that completes a tile has the reducing warp
//                 apply the activation and write a in the down kernel's
//                 fragment order.
//   k_union_down  persistent.  Work unit = 16 union rows x a 2048-column block
//                 of W_down (+ the tile's activations); CTAs take contiguous
//                 ranges, each consumer warp owns 256 columns of the block and
//                 accumulates in registers, then adds its slice into y with
//                 vector atomics when the column block changes.
// With more than 4 tokens the hi and lo operand terms go through two mma into
// the same accumulator (the n8 columns are the 8 tokens); with up to 4 tokens
// they are separate columns of one mma.
#include <cuda_fp16.h>

#include "ffn_rows.cuh"
#include "internal.h"
#include "pi.h"

namespace pi {

namespace {

constexpr int kUW = 8;                   // consumer warps
constexpr int kUThreads = kUW * 32 + 32; // + producer warp (down kernel)
constexpr int kUpThreads = kUThreads + 32; // + reducing warp (up kernel)
constexpr int kUMaxStages = 32;
constexpr size_t kHdrU = 2048;           // mbarriers + the producer's neuron-id table
static_assert(2 * kUMaxStages * 8 + 2 * 128 * 4 <= kHdrU, "header region too small");
constexpr size_t kSmemBudget = 225 * 1024;
constexpr int kScaleExp = 10;            // scaled operands have their maximum in [2^10, 2^11)
constexpr int kBatchJobs = 8;            // producer reads idx for 8 jobs (128 rows) at a time
constexpr int kSlots = 4;                // up kernel: partial-sum slots in flight
constexpr int kEpiFfn = 0, kEpiHidden = 1, kEpiLogits = 2;  // up kernel epilogues

// Up-projection chunks (weights of d_model per unit) and shared-memory row strides.
constexpr int kKsF16 = 2048;
constexpr int kKsQ4 = 4096;
// Unit width of the up kernel: Q4_0 at 5-8 tokens (two operand groups) takes
// 2048-weight units so that each warp's x fragments of a unit (8 steps x 2
// groups x 16 bytes per lane) stay in registers across the units of a chunk.
__host__ __device__ constexpr int up_ks(bool q4, int ng) { return q4 ? (ng == 2 ? 2048 : kKsQ4) : kKsF16; }
// Down-projection column blocks.
constexpr int kCw = 2048;                  // columns per block (4 KB fp16 row pieces)
constexpr int kWc = kCw / kUW;             // 256 columns per consumer warp
constexpr int kIt = kWc / 16;              // 16 sixteen-column tiles per warp
constexpr int kRsF16Dn = kCw * 2 + 16;     // 4112: ldmatrix rows hit distinct banks
constexpr int kRsQ4Dn = kCw / 2 + 16;      // 1040: 32-bit reads of rows 2t.. conflict-free
constexpr int kSsQ4Dn = kCw / 16 + 16;     // 144
constexpr int kFlushCols = 64;             // columns per pass of the down kernel's flush
constexpr uint32_t kTileAct = 512;         // activations of one 16-row tile: [8 tokens][4][4] fp32

__host__ __device__ constexpr uint32_t dn_act_off(bool q4) { return q4 ? 16u * (kRsQ4Dn + kSsQ4Dn) : 16u * kRsF16Dn; }
__host__ __device__ constexpr uint32_t dn_stage_bytes(bool q4) { return dn_act_off(q4) + kTileAct; }

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

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

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
constexpr int kPrepSplit = 16;  // CTAs per token

__global__ void __launch_bounds__(256) k_union_prep(const float *__restrict__ x, int B, int d, int q4,
                                                     uint32_t *__restrict__ xf, int *__restrict__ uexp,
                                                     unsigned *__restrict__ amax)
{
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x, part = blockIdx.y;
    const int NG = B > 4 ? 2 : 1;
    __shared__ float red[8];
    float m = 0.f;
    const bool live = b < B;
    if (live) {
        const float4 *xb = reinterpret_cast<const float4 *>(x + (size_t)b * d);
#pragma unroll 8
        for (int i = threadIdx.x; i < d / 4; i += blockDim.x) {
            const float4 v = xb[i];
            m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
    const int e = live ? scale_exp(m) : 0;
    if (threadIdx.x == 0 && part == 0) {
        uexp[b] = e;
        amax[b] = 0u;
    }
    if (NG == 1 && b >= 4) return;  // those columns hold the lo terms of tokens 0..3
    const int ghi = b, glo = NG == 1 ? b + 4 : b;
    const int grp_lo = NG == 1 ? 0 : 1;
    const int steps = (d + 31) / 32;
    const int v0 = steps * 16 * part / kPrepSplit, v1 = steps * 16 * (part + 1) / kPrepSplit;
    for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
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
// Producer warp shared by the up and down kernels.  Job j of the CTA's range
// copies the 16 rows idx[16 * tile(j) + r] (rows past n repeat row n - 1, whose
// values are finite and are multiplied by zero or discarded) into stage
// j % nstages: lane r < 16 issues row r's bulk copies after lane 0 has set the
// stage's expected byte count.  The neuron ids are read one batch of 8 jobs
// ahead so their latency overlaps the copies of the batch before.  The first
// `pre` jobs are issued before the programmatic-launch wait (weights and ids
// only, their bytes announced with expect_tx and no arrival); after the wait,
// late(j, s) copies late_bytes of data that the previous kernel produced, and
// the stage's single arrival follows.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

template <typename JobTile, typename JobBytes, typename Issue, typename Late>
__device__ void produce_rows(const SparseParams &p, int n, int cnt, int nstages, int pre, uint32_t late_bytes,
                             uint64_t *full, uint64_t *empty, int *tab, JobTile job_tile, JobBytes job_bytes,
                             Issue issue, Late late)
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
                int row = 16 * job_tile(jj) + (v & 15);
                row = row < n ? row : n - 1;
                out[i] = p.idx ? __ldcg(p.idx + row) : row;
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
    pre = min(pre, cnt);
    auto release_pre = [&]() {
        pdl_wait();
        for (int jj = 0; jj < pre; ++jj) {
            if (lane == 0) mbar_arrive_expect_tx(&full[jj % nstages], late_bytes);
            __syncwarp();
            late(jj, jj % nstages);
        }
    };
    int pref[4];
    fetch(0, pref);
    store(0, pref);
    __syncwarp();
    bool failed = false;
    int j = 0;
    if (pre == 0) release_pre();
    for (int jb = 0; jb < cnt && !failed; jb += kBatchJobs) {
        const int buf = (jb / kBatchJobs) & 1;
        fetch(jb + kBatchJobs, pref);
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
            const bool early = j < pre;
            if (lane == 0) {
                if (early)
                    mbar_expect_tx(&full[s], job_bytes(j));
                else
                    mbar_arrive_expect_tx(&full[s], job_bytes(j) + late_bytes);
            }
            __syncwarp();
            issue(j, s, tab + buf * 128 + (j - jb) * 16);
            if (!early) late(j, s);
            if (j == pre - 1) release_pre();
        }
        __syncwarp();
        store(buf ^ 1, pref);
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
template <int WT, bool GATED, int NG, int EPI>
__global__ void __launch_bounds__(kUpThreads, 1) k_union_up(SparseParams p, int nstages, int rs, int ss, uint32_t SB)
{
    constexpr bool Q4 = WT == PI_Q4_0;
    constexpr int KS = up_ks(Q4, NG);         // weights of d_model per unit
    constexpr int SPW = KS / 32 / kUW;        // 32-wide steps per warp and unit
    constexpr int M = GATED ? 2 : 1;          // matrices per row tile
    // rs, ss: row strides of a stage (code / fp16 rows; Q4_0 scale rows), SB: stage bytes
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kUMaxStages;
    int *tab = reinterpret_cast<int *>(empty + kUMaxStages);  // [2][128]
    uint8_t *stages = smem + kHdrU;
    float *red = reinterpret_cast<float *>(stages + (size_t)nstages * SB);  // [kSlots][8 warps][16 rows][8 tokens]
    __shared__ __align__(8) uint64_t rdy[kSlots];  // all 256 consumer lanes wrote their partial sums
    __shared__ __align__(8) uint64_t fre[kSlots];  // the unit's reducing warp has read the slot
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = p.d, F = p.F;
    unsigned *err = &p.ctrl->err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kUW);
        }
        for (int b = 0; b < kSlots; ++b) {
            mbar_init(&rdy[b], kUW * 32);
            mbar_init(&fre[b], 32);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();

    int n = p.n_active ? __ldcg(p.n_active) : F;  // no list: every row of W, in order
    n = n < 0 ? 0 : (n > F ? F : n);
    const int T = (n + 15) >> 4;
    const int C = (d + KS - 1) / KS;
    const int per = T * M;                    // units per chunk
    const long long U = (long long)per * C;
    const int G = gridDim.x;
    const int u0 = (int)(U * blockIdx.x / G), u1 = (int)(U * (blockIdx.x + 1) / G);
    const int cnt = u1 - u0;
    if (cnt <= 0) return;

    if (warp == kUW + 1) {
        // ---------------------------- reducing warp ----------------------------
        const int rrow = lane >> 1, rtb = 4 * (lane & 1);  // row and first token of this lane
        float rsc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) rsc[i] = ldexpf(1.f, __ldcg(p.uexp + rtb + i));
        const int B = p.B;
        float mx[4] = {0.f, 0.f, 0.f, 0.f};  // largest |a| per token (FFN epilogue)
        // Epilogue of one finished 16-row tile for this lane's row and 4 tokens:
        //   FFN:    a = act(z + b) (* u) -> activation fragments of the down kernel;
        //   hidden: h = max(z, 0) -> h[token][row];
        //   logits: l = z + p_bias -> logits (optional), union over tokens of l > tau -> mask.
        auto epilogue = [&](int tile, float4 zg, float4 zu, float bias, bool valid) {
            const int k = 16 * tile + rrow;
            const float zgv[4] = {zg.x, zg.y, zg.z, zg.w};
            const float zuv[4] = {zu.x, zu.y, zu.z, zu.w};
            if constexpr (EPI == kEpiFfn) {
                const int tq = (rrow & 7) >> 1, jx = (rrow & 1) + 2 * (rrow >> 3);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float a = 0.f;
                    if (valid && rtb + i < B) {
                        a = activate(p.act, zgv[i] + bias);
                        if constexpr (GATED) a *= zuv[i];
                    }
                    p.act_ws[(((size_t)tile * 8 + rtb + i) * 4 + tq) * 4 + jx] = a;
                    mx[i] = fmaxf(mx[i], fabsf(a));
                }
            } else if constexpr (EPI == kEpiHidden) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (valid && rtb + i < B) p.out_h[(size_t)(rtb + i) * F + k] = fmaxf(zgv[i], 0.f);
            } else {
                bool on = false;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (valid && rtb + i < B) {
                        const float l = zgv[i] + bias;
                        if (p.out_logits) p.out_logits[(size_t)(rtb + i) * F + k] = l;
                        on = on || l > p.tau;
                    }
                const int other = __shfl_xor_sync(0xffffffffu, on ? 1 : 0, 1);  // the row's other 4 tokens
                on = on || other != 0 || k < p.prefix;  // always-on prefix
                if (valid && rtb == 0) p.out_mask[k] = on ? 1 : 0;
            }
        };
        for (int jn = 0; jn < cnt;) {
            int nb = 0;
            for (; nb < kSlots && jn + nb < cnt; ++nb) {
                const int jj = jn + nb;
                const unsigned par = (unsigned)(jj / kSlots) & 1u;
                if (nb == 0 ? !mbar_wait(&rdy[jj % kSlots], par, err) : !mbar_test_wait(&rdy[jj % kSlots], par)) break;
            }
            if (nb == 0) break;  // gave up (error raised)
            // neuron ids and biases of this lane's row in every tile of the batch, issued
            // now so their latency hides behind the atomics and the fence below
            int jid[kSlots];
            float bias[kSlots];
            const float *bvec = EPI == kEpiFfn ? p.b_act : (EPI == kEpiLogits ? p.p_bias : nullptr);
#pragma unroll
            for (int b = 0; b < kSlots; ++b) {
                const int k = 16 * (((u0 + jn + b) % per) / M) + rrow;
                jid[b] = (b < nb && k < n) ? (p.idx ? __ldcg(p.idx + k) : k) : -1;
            }
#pragma unroll
            for (int b = 0; b < kSlots; ++b)
                bias[b] = (jid[b] >= 0 && jid[b] < F && bvec) ? __ldg(bvec + jid[b]) : 0.f;
#pragma unroll
            for (int b = 0; b < kSlots; ++b) {
                if (b >= nb) break;
                const int jj = jn + b, u = u0 + jj;
                const float *rb = red + (size_t)(jj % kSlots) * (kUW * 128);
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (NG == 2 || rtb == 0) {
#pragma unroll
                    for (int w = 0; w < kUW; ++w) {
                        const float4 pz = *reinterpret_cast<const float4 *>(rb + w * 128 + rrow * 8 + rtb);
                        v.x += pz.x;
                        v.y += pz.y;
                        v.z += pz.z;
                        v.w += pz.w;
                    }
                    v.x *= rsc[0];
                    v.y *= rsc[1];
                    v.z *= rsc[2];
                    v.w *= rsc[3];
                }
                mbar_arrive(&fre[jj % kSlots]);
                const int tile = (u % per) / M;
                if (C * M == 1) {
                    // one unit is the whole tile: no partial sums to combine
                    epilogue(tile, v, make_float4(0.f, 0.f, 0.f, 0.f), bias[b], jid[b] >= 0 && jid[b] < F);
                } else if (NG == 2 || rtb == 0) {
                    atomicAdd(reinterpret_cast<float4 *>(p.zbuf + ((size_t)tile * 2 + u % M) * 128 + rrow * 8 + rtb), v);
                }
            }
            if (C * M > 1) {
                fence_acq_rel_gpu();
                __syncwarp();
                unsigned old = 0;
                if (lane < nb) old = atomicAdd(p.ucnt + ((u0 + jn + lane) % per) / M, 1u);
                const unsigned last = __ballot_sync(0xffffffffu, lane < nb && old == (unsigned)(C * M - 1));
                if (last) {
                    // ---- tiles completed by this batch: epilogue, then reset their buffers ----
                    fence_acq_rel_gpu();
                    float4 zg[kSlots], zu[kSlots];
#pragma unroll
                    for (int b = 0; b < kSlots; ++b) {
                        zg[b] = zu[b] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if ((last >> b) & 1u) {
                            const float *zt = p.zbuf + (size_t)(((u0 + jn + b) % per) / M) * 256 + rrow * 8 + rtb;
                            zg[b] = __ldcg(reinterpret_cast<const float4 *>(zt));
                            if constexpr (GATED) zu[b] = __ldcg(reinterpret_cast<const float4 *>(zt + 128));
                        }
                    }
#pragma unroll
                    for (int b = 0; b < kSlots; ++b) {
                        if (!((last >> b) & 1u)) continue;
                        const int tile = ((u0 + jn + b) % per) / M;
                        float *zt = p.zbuf + (size_t)tile * 256 + rrow * 8 + rtb;
                        __stcg(reinterpret_cast<float4 *>(zt), make_float4(0.f, 0.f, 0.f, 0.f));
                        if constexpr (GATED) __stcg(reinterpret_cast<float4 *>(zt + 128), make_float4(0.f, 0.f, 0.f, 0.f));
                        // an out-of-range neuron id (flagged by the producer, which copied
                        // row 0 in its place) contributes nothing
                        epilogue(tile, zg[b], zu[b], bias[b], jid[b] >= 0 && jid[b] < F);
                        if (lane == b) p.ucnt[tile] = 0u;
                    }
                }
            }
            jn += nb;
        }
        if constexpr (EPI == kEpiFfn) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int o = 2; o < 32; o <<= 1) mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], o));
            if (lane < 2)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (mx[i] > 0.f) atomicMax(p.amax + rtb + i, __float_as_uint(mx[i]));
        }
        return;
    }

    if (warp == kUW) {
        const unsigned long long pol = evict_first_policy();
        auto job_tile = [&](int jj) { return ((u0 + jj) % per) / M; };
        auto job_bytes = [&](int jj) {
            const int len = min(KS, d - ((u0 + jj) / per) * KS);
            return 16u * (Q4 ? (uint32_t)(len / 2 + len / 16) : (uint32_t)len * 2u);
        };
        auto issue = [&](int jj, int s, const int *rows) {
            if (lane >= 16) return;
            const int u = u0 + jj;
            const int c = u / per, m = u % M;
            const int k0 = c * KS, len = min(KS, d - k0);
            const uint8_t *W = (GATED && m == 1) ? p.w_up : p.w_act;
            uint8_t *st = stages + (size_t)s * SB;
            const size_t jn = (size_t)rows[lane];
            if constexpr (Q4) {
                bulk_g2s_once(st + lane * rs, W + jn * (d / 2) + k0 / 2, (uint32_t)(len / 2), &full[s], pol);
                bulk_g2s_once(st + 16 * rs + lane * ss, W + (size_t)F * (d / 2) + jn * (d / 16) + k0 / 16,
                              (uint32_t)(len / 16), &full[s], pol);
            } else {
                bulk_g2s_once(st + lane * rs, W + (jn * d + k0) * 2, (uint32_t)len * 2u, &full[s], pol);
            }
        };
        produce_rows(p, n, cnt, nstages, 0, 0u, full, empty, tab, job_tile, job_bytes, issue, [](int, int) {});
        return;
    }

    // ---------------------------------- consumer warps ----------------------------------
    const int g = lane >> 2, t = lane & 3;
    constexpr bool XREG = SPW * NG <= 16;  // x fragments held in registers (every unit width chosen above)
    uint4 xr[XREG ? SPW : 1][NG];
    int xc = -1;
    for (int jj = 0; jj < cnt; ++jj) {
        const int s = jj % nstages;
        const int u = u0 + jj;
        const int c = u / per;
        const int q0 = warp * SPW;
        if constexpr (XREG) {
            // this warp's x fragments for chunk c: loaded before the stage wait, and kept
            // while consecutive units share the chunk (units are ordered chunk-major)
            if (c != xc) {
                const int nq = (min(KS, d - c * KS) + 31) / 32;
                const uint8_t *xfc = reinterpret_cast<const uint8_t *>(p.xf) + ((size_t)(c * KS / 32) * NG * 32 + lane) * 16;
#pragma unroll
                for (int i = 0; i < SPW; ++i)
#pragma unroll
                    for (int gr = 0; gr < NG; ++gr)
                        xr[i][gr] = q0 + i < nq ? ldg_nc_v4(xfc + ((size_t)(q0 + i) * NG + gr) * 512)
                                                : make_uint4(0u, 0u, 0u, 0u);
                xc = c;
            }
        }
        if (!mbar_wait(&full[s], (unsigned)(jj / nstages) & 1u, err)) break;
        const uint8_t *st = stages + (size_t)s * SB;
        const int k0 = c * KS, len = min(KS, d - k0);
        float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};  // two mma chains
        const int q1 = min(q0 + SPW, (len + 31) / 32);
        const uint8_t *xfp = reinterpret_cast<const uint8_t *>(p.xf) + ((size_t)(k0 / 32) * NG * 32 + lane) * 16;
        if constexpr (!Q4) {
            const uint8_t *ra = st + g * rs + 16 * t;
            const uint8_t *rb = ra + 8 * rs;
#pragma unroll
            for (int i = 0; i < SPW; ++i) {
                const int q = q0 + i;
                if (q < q1) {
                    uint4 a0 = *reinterpret_cast<const uint4 *>(ra + q * 64);
                    uint4 a1 = *reinterpret_cast<const uint4 *>(rb + q * 64);
                    if (q * 32 + 8 * t >= len) a0 = a1 = make_uint4(0u, 0u, 0u, 0u);  // ragged end of d_model
#pragma unroll
                    for (int gr = 0; gr < NG; ++gr) {  // NG == 2: hi then lo terms into the same sums
                        const uint4 bx = xr[i][gr];
                        mma16816(acc, a0.x, a1.x, a0.y, a1.y, bx.x, bx.y);
                        mma16816(acc2, a0.z, a1.z, a0.w, a1.w, bx.z, bx.w);
                    }
                }
            }
        } else {
            const uint8_t *ca = st + g * rs + 4 * t;
            const uint8_t *cb = ca + 8 * rs;
            const __half *sa = reinterpret_cast<const __half *>(st + 16 * rs + g * ss);
            const __half *sb = reinterpret_cast<const __half *>(st + 16 * rs + (g + 8) * ss);
#pragma unroll
            for (int i = 0; i < SPW; ++i) {
                const int q = q0 + i;
                if (q >= q1) break;
                const uint32_t w0 = *reinterpret_cast<const uint32_t *>(ca + q * 16);
                const uint32_t w1 = *reinterpret_cast<const uint32_t *>(cb + q * 16);
                const float s0 = __half2float(sa[q]), s1 = __half2float(sb[q]);
                const uint32_t p0 = q4_pair(w0), p1 = q4_pair(w0 >> 4), p2 = q4_pair(w0 >> 8), p3 = q4_pair(w0 >> 12);
                const uint32_t r0 = q4_pair(w1), r1 = q4_pair(w1 >> 4), r2 = q4_pair(w1 >> 8), r3 = q4_pair(w1 >> 12);
#pragma unroll
                for (int gr = 0; gr < NG; ++gr) {
                    uint4 bx;
                    if constexpr (XREG)
                        bx = xr[i][gr];
                    else
                        bx = ldg_nc_v4(xfp + ((size_t)q * NG + gr) * 512);
                    float tmp[4] = {0.f, 0.f, 0.f, 0.f};
                    mma16816(tmp, p0, r0, p1, r1, bx.x, bx.y);
                    mma16816(tmp, p2, r2, p3, r3, bx.z, bx.w);
                    float *ac = (gr & 1) ? acc2 : acc;
                    ac[0] = fmaf(s0, tmp[0], ac[0]);
                    ac[1] = fmaf(s0, tmp[1], ac[1]);
                    ac[2] = fmaf(s1, tmp[2], ac[2]);
                    ac[3] = fmaf(s1, tmp[3], ac[3]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);

        // -> this warp's partial sums for tokens 2t, 2t+1 (NG == 1: hi + lo columns, lanes t < 2)
        float z[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            z[i] = acc[i] + acc2[i];
            if constexpr (NG == 1) z[i] += __shfl_xor_sync(0xffffffffu, z[i], 2);
        }
        const int sl = jj % kSlots, use = jj / kSlots;
        float *rb = red + (size_t)sl * (kUW * 128);
        if (use > 0 && !mbar_wait(&fre[sl], (unsigned)(use - 1) & 1u, err)) break;
        if (NG == 2 || t < 2) {
            *reinterpret_cast<float2 *>(rb + warp * 128 + g * 8 + 2 * t) = make_float2(z[0], z[1]);
            *reinterpret_cast<float2 *>(rb + warp * 128 + (g + 8) * 8 + 2 * t) = make_float2(z[2], z[3]);
        }
        mbar_arrive(&rdy[sl]);
    }
}

template <int WT, int NG>
__global__ void __launch_bounds__(kUThreads, 1) k_union_down(SparseParams p, int nstages)
{
    constexpr bool Q4 = WT == PI_Q4_0;
    constexpr int CW = kCw;                   // columns of a block
    constexpr int IT = kIt;                   // 16-column tiles per warp
    constexpr int WC = kWc;                   // columns per warp
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
        const unsigned long long pol = evict_first_policy();
        auto job_tile = [&](int jj) { return (int)((u0 + jj) % T); };
        auto job_bytes = [&](int jj) {
            const int nc = min(CW, d - (int)((u0 + jj) / T) * CW);
            return 16u * (Q4 ? (uint32_t)(nc / 2 + nc / 16) : (uint32_t)nc * 2u);
        };
        auto issue = [&](int jj, int s, const int *rows) {
            if (lane >= 16) return;
            const long long u = u0 + jj;
            const int c0 = (int)(u / T) * CW, nc = min(CW, d - c0);
            uint8_t *st = stages + (size_t)s * SB;
            const size_t jn = (size_t)rows[lane];
            if constexpr (Q4) {
                bulk_g2s_once(st + lane * kRsQ4Dn, p.w_down + jn * (d / 2) + c0 / 2, (uint32_t)(nc / 2), &full[s], pol);
                bulk_g2s_once(st + 16 * kRsQ4Dn + lane * kSsQ4Dn, p.w_down + (size_t)F * (d / 2) + jn * (d / 16) + c0 / 16,
                              (uint32_t)(nc / 16), &full[s], pol);
            } else {
                bulk_g2s_once(st + lane * kRsF16Dn, p.w_down + (jn * d + c0) * 2, (uint32_t)nc * 2u, &full[s], pol);
            }
        };
        // the tile's activations (written by the up kernel), one 512-byte copy
        auto late = [&](int jj, int s) {
            if (lane != 16) return;
            const int tile = (int)((u0 + jj) % T);
            bulk_g2s(stages + (size_t)s * SB + dn_act_off(Q4),
                     reinterpret_cast<const uint8_t *>(p.act_ws) + (size_t)tile * kTileAct, kTileAct, &full[s]);
        };
        produce_rows(p, n, cnt, nstages, nstages, kTileAct, full, empty, tab, job_tile, job_bytes, issue, late);
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
    float *fb = reinterpret_cast<float *>(stages + (size_t)nstages * SB) + (size_t)warp * 8 * kFlushCols;
    const int B = p.B;

    float acc[IT][4];
    auto zero_acc = [&]() {
#pragma unroll
        for (int i = 0; i < IT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    };
    // Adds this warp's slice of column block cb into y (through shared memory, so
    // that the atomics are 16-byte vectors).
    auto flush = [&](int cb) {
        const int c0 = cb * CW + warp * WC;
#pragma unroll
        for (int ps = 0; ps < WC / kFlushCols; ++ps) {
            // pass ps: the tiles whose columns fall in [64 ps, 64 ps + 64) of the warp slice
#pragma unroll
            for (int i = ps * 4; i < ps * 4 + 4; ++i) {
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    v[e] = acc[i][e];
                    if constexpr (NG == 1) v[e] += __shfl_xor_sync(0xffffffffu, v[e], 2);
                }
                if (NG == 2 || t < 2) {
                    int col0, col1;  // columns of rows g and g + 8 of tile i, within the pass
                    if constexpr (Q4) {
                        col0 = 32 * (g >> 2) + 4 * (g & 3) + (i & 3);
                        col1 = col0 + 16;
                    } else {
                        col0 = 16 * (i & 3) + g;
                        col1 = col0 + 8;
                    }
                    fb[(2 * t) * kFlushCols + col0] = v[0] * sc0;
                    fb[(2 * t + 1) * kFlushCols + col0] = v[1] * sc1;
                    fb[(2 * t) * kFlushCols + col1] = v[2] * sc0;
                    fb[(2 * t + 1) * kFlushCols + col1] = v[3] * sc1;
                }
            }
            __syncwarp();
            for (int e = lane; e < B * (kFlushCols / 4); e += 32) {
                const int tok = e / (kFlushCols / 4), c4 = e % (kFlushCols / 4);
                const int col = c0 + ps * kFlushCols + 4 * c4;
                if (col < d)
                    atomicAdd(reinterpret_cast<float4 *>(p.y + (size_t)tok * d + col),
                              *reinterpret_cast<const float4 *>(fb + tok * kFlushCols + 4 * c4));
            }
            __syncwarp();
        }
    };

    zero_acc();
    int cur = -1;
    for (int jj = 0; jj < cnt; ++jj) {
        const int s = jj % nstages;
        const long long u = u0 + jj;
        const int cb = (int)(u / T);
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
            const float4 av = *reinterpret_cast<const float4 *>(st + dn_act_off(Q4) + (tokB * 4 + t) * 16);
            __half h0, h1, h2, h3, l0, l1, l2, l3;
            split_f16(av.x * inv, h0, l0);
            split_f16(av.y * inv, h1, l1);
            split_f16(av.z * inv, h2, l2);
            split_f16(av.w * inv, h3, l3);
            uint32_t bf[NG][2];  // NG == 2: [0] hi terms, [1] lo terms, both into the same sums
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
                    for (int q = 0; q < NG; ++q) mma16816(acc[i], a0, a1, a2, a3, bf[q][0], bf[q][1]);
                }
            } else {
                const uint8_t *codes = st + (WC / 2) * warp + 4 * g;
                const uint8_t *scl = st + 16 * kRsQ4Dn;
#pragma unroll
                for (int h = 0; h < WC / 64; ++h) {
                    const uint32_t wa = *reinterpret_cast<const uint32_t *>(codes + (2 * t) * kRsQ4Dn + 32 * h);
                    const uint32_t wb = *reinterpret_cast<const uint32_t *>(codes + (2 * t + 1) * kRsQ4Dn + 32 * h);
                    const uint32_t wc = *reinterpret_cast<const uint32_t *>(codes + (2 * t + 8) * kRsQ4Dn + 32 * h);
                    const uint32_t wd = *reinterpret_cast<const uint32_t *>(codes + (2 * t + 9) * kRsQ4Dn + 32 * h);
                    const int blk = (WC / 32) * warp + 2 * h + (g >> 2);
                    const __half2 sA = __halves2half2(*reinterpret_cast<const __half *>(scl + (2 * t) * kSsQ4Dn + 2 * blk),
                                                      *reinterpret_cast<const __half *>(scl + (2 * t + 1) * kSsQ4Dn + 2 * blk));
                    const __half2 sB = __halves2half2(*reinterpret_cast<const __half *>(scl + (2 * t + 8) * kSsQ4Dn + 2 * blk),
                                                      *reinterpret_cast<const __half *>(scl + (2 * t + 9) * kSsQ4Dn + 2 * blk));
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
                            mma16816(acc[4 * h + mm], a[0], a[1], a[2], a[3], bf[q][0], bf[q][1]);
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

template <int WT, bool GATED, int NG, int EPI = kEpiFfn>
cudaError_t launch_up(const SparseParams &p, cudaStream_t s)
{
    // stages sized by the widest chunk this contraction has (its K may be far below KS)
    constexpr bool Q4 = WT == PI_Q4_0;
    constexpr int KS = up_ks(Q4, NG);
    const int kse = p.d < KS ? p.d : KS;
    int rs, ss;
    if (Q4) {
        rs = kse / 2 + 16;   // kse % 256 == 0: rows 16 bytes past a 128-byte multiple
        ss = kse / 16 + 16;
    } else {
        rs = (kse * 2 + 127) / 128 * 128 + 64;  // 64 bytes past a 128-byte multiple
        ss = 0;
    }
    const uint32_t SB = 16u * (uint32_t)(rs + ss);
    constexpr size_t rbytes = (size_t)kSlots * kUW * 128 * 4;  // the partial-sum slots
    const size_t fit = (kSmemBudget - kHdrU - rbytes) / SB;
    const int ns = (int)(fit < (size_t)kUMaxStages ? fit : (size_t)kUMaxStages);
    const size_t smem = kHdrU + (size_t)ns * SB + rbytes;
    static bool once = false;
    if (!once) {
        // the largest request any shape makes
        cudaError_t e = set_smem(k_union_up<WT, GATED, NG, EPI>, kSmemBudget);
        if (e != cudaSuccess) return e;
        once = true;
    }
    return launch_pdl(k_union_up<WT, GATED, NG, EPI>, dim3(sm_count()), dim3(kUpThreads), smem, s, p, ns, rs, ss, SB);
}

template <int WT, int NG>
cudaError_t launch_down(const SparseParams &p, cudaStream_t s)
{
    constexpr bool Q4 = WT == PI_Q4_0;
    constexpr uint32_t SB = dn_stage_bytes(Q4);
    constexpr size_t fbytes = (size_t)kUW * 8 * kFlushCols * 4;
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
    if (!p.xf_ready) {
        const cudaError_t e = launch_pdl(k_union_prep, dim3(8, kPrepSplit), dim3(256), 0, s, p.x, p.B, p.d,
                                         wtype == PI_Q4_0 ? 1 : 0, p.xf, p.uexp, p.amax);
        if (e != cudaSuccess) return e;
    }
    return wtype == PI_Q4_0 ? launch_union_wt<PI_Q4_0>(gated, p, s) : launch_union_wt<PI_F16>(gated, p, s);
}

cudaError_t launch_pred_union(const UnionPredArgs &a, cudaStream_t s)
{
    if (a.B < 2 || a.B > 8) return cudaErrorInvalidValue;
    // x -> fragments (these also serve the FFN's up projection, which is told to skip its own)
    cudaError_t e = launch_pdl(k_union_prep, dim3(8, kPrepSplit), dim3(256), 0, s, a.x, a.B, a.d, 0, a.xf_x, a.uexp_x,
                               a.amax);
    if (e != cudaSuccess) return e;
    SparseParams q{};
    q.ctrl = a.ctrl;
    q.zbuf = a.zbuf;
    q.ucnt = a.ucnt;
    q.B = a.B;
    q.act = 0;
    // h = max(P1 x, 0): every row of P1 against the tokens
    q.w_act = static_cast<const uint8_t *>(a.p1);
    q.xf = a.xf_x;
    q.uexp = a.uexp_x;
    q.d = a.d;
    q.F = a.r;
    q.out_h = a.h;
    e = a.B > 4 ? launch_up<PI_F16, false, 2, kEpiHidden>(q, s) : launch_up<PI_F16, false, 1, kEpiHidden>(q, s);
    if (e != cudaSuccess) return e;
    e = launch_pdl(k_union_prep, dim3(8, kPrepSplit), dim3(256), 0, s, a.h, a.B, a.r, 0, a.xf_h, a.uexp_h, a.amax);
    if (e != cudaSuccess) return e;
    // logits = P2 h + p_bias, union over tokens of logit > tau -> mask
    q.w_act = static_cast<const uint8_t *>(a.p2);
    q.xf = a.xf_h;
    q.uexp = a.uexp_h;
    q.d = a.r;
    q.F = a.F;
    q.out_h = nullptr;
    q.p_bias = a.p_bias;
    q.tau = a.tau;
    q.prefix = a.prefix;
    q.out_logits = a.logits;
    q.out_mask = a.mask;
    return a.B > 4 ? launch_up<PI_F16, false, 2, kEpiLogits>(q, s) : launch_up<PI_F16, false, 1, kEpiLogits>(q, s);
}

}  // namespace pi
