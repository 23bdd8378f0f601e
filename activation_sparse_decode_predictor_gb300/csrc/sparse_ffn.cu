// Neuron-aware sparse FFN for one decode token (batch 1).
//
// For the ascending active list idx[0..n): a_k = act(W_act[idx_k] . x + b) (times
// W_up[idx_k] . x for ReGLU) and y += sum_k a_k * W_down[idx_k].  Only listed
// rows are read (PowerInfer summary page, "技术贡献" technical contributions:
// neuron-level sparse matrix operators; "方法详解" method detail: the sparse
// operator works directly at neuron granularity).
//
// GB300 design: a persistent grid of one CTA per SM.  Each CTA owns a
// contiguous slice of the active list.  One producer thread streams whole
// neuron rows (contiguous 8-48 KB) from HBM into a ring of shared-memory
// stages with 1-D bulk (TMA) copies completing on mbarriers; eight consumer
// warps compute.  Each thread owns fixed 16-byte column chunks of d_model, so
// x and the partial output stay in registers.  An "up" job (the gate/up rows
// of one neuron) ends in a CTA reduction that yields a_k; the producer then
// fetches that neuron's down row only when a_k != 0 (a zero activation
// contributes exactly nothing), interleaving those "down" jobs with later up
// jobs so HBM never idles.  The CTA's partial y is added to global y with
// 16-byte vector atomics at the end.
#include "ffn_rows.cuh"
#include "internal.h"

namespace pi {

namespace {

constexpr int kNCW = 8;                 // consumer warps
constexpr int kNCT = kNCW * 32;         // consumer threads
constexpr int kThreads = kNCT + 32;     // + producer warp
constexpr int kMaxStages = 24;
constexpr int kSeg = 512;               // rows per segment (bounds the per-row smem tables)
constexpr size_t kHdr = 16384;          // barriers, job table, per-row tables (see layout below)
constexpr int kJobUp = 1, kJobDown = 2, kJobEnd = 3;

struct RowTables {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    int4 job[kMaxStages];               // kind, row-in-segment, neuron, 0
    float red[2][kNCW][2];
    int j[kSeg];                        // neuron of each row of the segment
    float bias[kSeg];                   // b_act of each row
    float a[kSeg];                      // activation of each row
    int state[kSeg];                    // 0 pending, 1 zero, 2 non-zero
};
static_assert(sizeof(RowTables) <= kHdr, "header region too small");

template <int WT, bool GATED, int CH>
__global__ void __launch_bounds__(kThreads, 1) k_sparse_b1(SparseParams p, int nstages, uint32_t stage_bytes)
{
    constexpr int EPC = Fmt<WT>::EPC;
    extern __shared__ __align__(128) uint8_t smem[];
    RowTables &T = *reinterpret_cast<RowTables *>(smem);
    uint8_t *stages = smem + kHdr;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = p.d, F = p.F;
    const uint32_t R = row_slot_bytes(WT, d);
    const int nch = d / EPC;
    unsigned *err = &p.ctrl->err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            mbar_init(&T.full[s], 1);
            mbar_init(&T.empty[s], kNCW);
        }
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < kSeg; i += kThreads) T.state[i] = 0;
    __syncthreads();

    pdl_wait();
    pdl_trigger();

    int n = *p.n_active;
    n = n < 0 ? 0 : (n > F ? F : n);
    const int G = gridDim.x;
    const int k0 = (int)((long long)n * blockIdx.x / G);
    const int k1 = (int)((long long)n * (blockIdx.x + 1) / G);
    const int cnt = k1 - k0;
    if (cnt == 0) return;

    if (warp == kNCW) {
        // ------------------------------ producer warp ------------------------------
        int q = 0;  // jobs issued so far (all segments)
        const unsigned long long pol = evict_first_policy();
        bool failed = false;
        for (int seg = 0; seg < cnt && !failed; seg += kSeg) {
            const int sn = min(kSeg, cnt - seg);
            for (int i = lane; i < sn; i += 32) T.j[i] = p.idx[k0 + seg + i];
            __syncwarp();
            if (lane == 0) {
                volatile int *state = T.state;
                int up = 0, ds = 0;
                for (;;) {
                    int kind, i = 0, j = 0;
                    if (ds < up && state[ds] != 0) {
                        const int stt = state[ds];
                        state[ds] = 0;
                        i = ds++;
                        if (stt == 1) continue;  // a == 0: the down row is not needed
                        kind = kJobDown;
                        j = T.j[i];
                    } else if (up < sn) {
                        i = up++;
                        j = T.j[i];
                        if (j < 0 || j >= F) {
                            atomicOr(err, ERR_INDEX);
                            T.a[i] = 0.f;
                            state[i] = 1;
                            continue;
                        }
                        kind = kJobUp;
                    } else if (ds < sn) {
                        // every up job is out; wait for the consumers to finish one
                        long long spins = 0;
                        while (state[ds] == 0 && ++spins < kSpinLimit) __nanosleep(64);
                        if (state[ds] == 0) {
                            atomicOr(err, ERR_TIMEOUT);
                            failed = true;
                            kind = kJobEnd;
                        } else {
                            continue;
                        }
                    } else {
                        kind = kJobEnd;
                    }
                    const int s = q % nstages;
                    if (q >= nstages && !mbar_wait(&T.empty[s], (unsigned)((q / nstages) - 1) & 1u, err)) {
                        failed = true;
                        break;
                    }
                    T.job[s] = make_int4(kind, i, j, 0);
                    uint8_t *st = stages + (size_t)s * stage_bytes;
                    if (kind == kJobUp) {
                        mbar_arrive_expect_tx(&T.full[s], GATED ? 2u * R : R);
                        copy_row<WT>(st, p.w_act, j, d, F, &T.full[s], pol);
                        if constexpr (GATED) copy_row<WT>(st + R, p.w_up, j, d, F, &T.full[s], pol);
                    } else if (kind == kJobDown) {
                        mbar_arrive_expect_tx(&T.full[s], R);
                        copy_row<WT>(st, p.w_down, j, d, F, &T.full[s], pol);
                    } else {
                        mbar_arrive(&T.full[s]);
                    }
                    ++q;
                    if (kind == kJobEnd) break;
                }
            }
            q = __shfl_sync(0xffffffffu, q, 0);
            failed = __shfl_sync(0xffffffffu, failed, 0);
            __syncwarp();
            named_bar_sync(2, kThreads);  // segment boundary: tables are reused
        }
        if (failed && lane == 0) {
            // never leave the CTA with bulk copies in flight into its shared memory
            for (int s = 0; s < nstages && s < q; ++s) {
                const int last = s + ((q - 1 - s) / nstages) * nstages;  // last job issued on stage s
                mbar_wait(&T.full[s], (unsigned)(last / nstages) & 1u, err);
            }
        }
        return;
    }

    // -------------------------------- consumer warps ----------------------------------
    const int t = threadIdx.x;
    float xr[CH][EPC];
    float acc[CH][EPC];
#pragma unroll
    for (int u = 0; u < CH; ++u) {
        const int c = t + kNCT * u;
#pragma unroll
        for (int e = 0; e < EPC; e += 4) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c < nch) v = *reinterpret_cast<const float4 *>(p.x + (size_t)c * EPC + e);
            xr[u][e] = v.x;
            xr[u][e + 1] = v.y;
            xr[u][e + 2] = v.z;
            xr[u][e + 3] = v.w;
            acc[u][e] = acc[u][e + 1] = acc[u][e + 2] = acc[u][e + 3] = 0.f;
        }
    }
    bool any = false, failed = false;
    int q = 0, ub = 0;
    for (int seg = 0; seg < cnt; seg += kSeg) {
        const int sn = min(kSeg, cnt - seg);
        if (warp == 0) {
            for (int i = lane; i < sn; i += 32) {
                const int j = p.idx[k0 + seg + i];
                T.bias[i] = (p.b_act && j >= 0 && j < F) ? p.b_act[j] : 0.f;
            }
            __syncwarp();
        }
        while (!failed) {
            const int s = q % nstages;
            if (!mbar_wait(&T.full[s], (unsigned)(q / nstages) & 1u, err)) {
                failed = true;
                break;
            }
            const int4 job = T.job[s];
            if (job.x == kJobEnd) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&T.empty[s]);
                ++q;
                break;
            }
            const uint8_t *st = stages + (size_t)s * stage_bytes;
            if (job.x == kJobUp) {
                float pa = 0.f, pu = 0.f;
#pragma unroll
                for (int u = 0; u < CH; ++u) {
                    const int c = t + kNCT * u;
                    if (c < nch) {
                        pa += chunk_dot<WT>(st, c, d, xr[u]);
                        if constexpr (GATED) pu += chunk_dot<WT>(st + R, c, d, xr[u]);
                    }
                }
                pa = warp_sum(pa);
                if constexpr (GATED) pu = warp_sum(pu);
                if (lane == 0) {
                    T.red[ub & 1][warp][0] = pa;
                    T.red[ub & 1][warp][1] = pu;
                }
                named_bar_sync(1, kNCT);
                if (t == 0) {
                    float z = 0.f, uu = 0.f;
#pragma unroll
                    for (int w = 0; w < kNCW; ++w) {
                        z += T.red[ub & 1][w][0];
                        uu += T.red[ub & 1][w][1];
                    }
                    float a = activate(p.act, z + T.bias[job.y]);
                    if constexpr (GATED) a *= uu;
                    T.a[job.y] = a;
                    __threadfence_block();
                    *reinterpret_cast<volatile int *>(&T.state[job.y]) = (a != 0.f) ? 2 : 1;
                }
                ++ub;
            } else {
                const float a = T.a[job.y];
#pragma unroll
                for (int u = 0; u < CH; ++u) {
                    const int c = t + kNCT * u;
                    if (c < nch) chunk_axpy<WT>(st, c, d, a, acc[u]);
                }
                any = true;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&T.empty[s]);
            ++q;
        }
        named_bar_sync(2, kThreads);
        if (failed) break;
    }
    if (!any) return;
    // CTA partial -> global y (16-byte vector atomics)
#pragma unroll
    for (int u = 0; u < CH; ++u) {
        const int c = t + kNCT * u;
        if (c < nch) {
#pragma unroll
            for (int e = 0; e < EPC; e += 4)
                atomicAdd(reinterpret_cast<float4 *>(p.y + (size_t)c * EPC + e),
                          make_float4(acc[u][e], acc[u][e + 1], acc[u][e + 2], acc[u][e + 3]));
        }
    }
}

template <int WT, bool GATED>
cudaError_t launch_ch(const SparseParams &p, cudaStream_t s)
{
    constexpr int EPC = Fmt<WT>::EPC;
    const int nch = p.d / EPC;
    const int need = (nch + kNCT - 1) / kNCT;
    const uint32_t R = row_slot_bytes(WT, p.d);
    const uint32_t stage_bytes = ((GATED ? 2u : 1u) * R + 127u) & ~127u;
    const size_t budget = 200 * 1024;
    int ns = (int)((budget - kHdr) / stage_bytes);
    ns = ns > kMaxStages ? kMaxStages : ns;
    if (ns < 2) return cudaErrorInvalidValue;
    const size_t smem = kHdr + (size_t)ns * stage_bytes;
    void (*k)(SparseParams, int, uint32_t);
    if (need <= 1)
        k = k_sparse_b1<WT, GATED, 1>;
    else if (need <= 2)
        k = k_sparse_b1<WT, GATED, 2>;
    else if (need <= 4)
        k = k_sparse_b1<WT, GATED, 4>;
    else if (need <= 8)
        k = k_sparse_b1<WT, GATED, 8>;
    else if constexpr (WT == 0)
        k = k_sparse_b1<WT, GATED, 16>;
    else
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(sm_count()), dim3(kThreads), smem, s, p, ns, stage_bytes);
}

}  // namespace

cudaError_t launch_sparse_b1(int wtype, int gated, const SparseParams &p, cudaStream_t s)
{
    switch (wtype * 2 + (gated ? 1 : 0)) {
    case 0: return launch_ch<0, false>(p, s);
    case 1: return launch_ch<0, true>(p, s);
    case 2: return launch_ch<1, false>(p, s);
    case 3: return launch_ch<1, true>(p, s);
    case 4: return launch_ch<2, false>(p, s);
    case 5: return launch_ch<2, true>(p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pi
