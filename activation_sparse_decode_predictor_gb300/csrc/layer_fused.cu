// One decode token through one FFN layer in a single kernel (batch 1): the
// predictor, the active-neuron scan and the neuron-aware sparse FFN, without
// kernel boundaries between them.
//
// Method (PowerInfer summary page, "核心创新" core innovation and "方法详解"
// method detail): an online predictor marks the neurons expected to fire and
// neuron-aware sparse operators compute only those neurons.  Predictor form,
// as in predict.cu: h = max(P1 x, 0), logit = P2 h + p_bias, active when
// logit > threshold.  FFN as in sparse_ffn.cu.  Optionally the first H
// neurons (the hot-first order's always-on prefix) are active at every step:
// the predictor then covers only the tail [H, F) and no P2 row of the prefix
// is read.
//
// GB300 design.  One CTA per SM (all CTAs resident together), 1 producer warp
// + 8 consumer warps (12 for rows of 12 Ki fp16 columns or more).  The producer
// thread streams every byte the CTA needs through one ring of shared-memory
// stages with 1-D bulk copies completing on mbarriers, in job order:
//   P1 jobs      consecutive rows of this CTA's share of the predictor's P1,
//   P2 jobs      8 rows of P2 each (12 in the 12-warp variant when a stage
//                holds them), for this CTA's contiguous neuron range,
//   FFN jobs     up/gate rows of this CTA's share of the active neurons, and
//                the down row of each neuron whose activation is non-zero.
// Every weight copy carries an L2 evict-first policy: a decode step reads each
// weight byte once, and those lines must not push out what is read again
// (activations, the queue, the control block).  On entry,
// before the programmatic-dependent-launch wait, the producer fills the ring
// with P1 and P2 rows (they do not depend on the previous kernel).  The
// consumers:
//   0. (chained input) rescale the previous layer's x + y themselves: every CTA
//      sums the squares of the whole vector in the same order, so all CTAs hold
//      the same x, and writes its slice of x out;
//   1. compute their P1 rows -> h slice -> global; grid barrier A; load h;
//   2. compute the logits of their neuron range, threshold, ballot, write the
//      range's active neurons (with their biases) to a candidate list and the
//      count to a status word; grid barrier B; read all counts: the prefix
//      gives this range's place in the ascending active list and the total n;
//   3. take their prefix slice and the balanced share [n*c/G, n*(c+1)/G) of the
//      tail's active list, look each entry up in the candidate lists and hand
//      the neuron ids to the producer (an mbarrier), which asks L2 for all
//      their rows at once and then runs the FFN jobs as sparse_ffn.cu does; the
//      CTA's partial output goes to y with 16-byte vector atomics.
// Steps 2-3 above are the ordered mode, used when the caller asks for the
// ascending active list.  Without that request (queue mode) there is no
// barrier B: each CTA keeps its prefix slice and the first kOwn active neurons
// of its own range (its producer starts on them at once, with no global round
// trip), appends the rest to a shared work queue (one 8-byte entry {launch
// tag, neuron} per neuron) and counts itself done; producers then take kQTake
// queue slots per atomic, claiming a batch only while the CTA's share table
// has room for all of it, and stop when the queue is drained and every CTA has
// published.  The host picks queue mode only when the share tables of all
// CTAs together hold every neuron, so no claimed row is ever dropped.
// The grid barriers are counter barriers: one thread per CTA arrives with a
// release add on a 64-bit counter that is never reset and polls it (acquire,
// bounded) until it reaches a target derived from a per-launch sequence
// number, so no arrival ever has to reset anything.  Every wait is bounded.
// A barrier that gives up is seen by every consumer thread after the next CTA
// barrier (a flag in shared memory), stage waits before warp-wide shuffles are
// decided for the whole warp, and a failed launch publishes nothing, still
// arrives at every grid barrier and drains its copies before it returns.
#include <algorithm>

#include "ffn_rows.cuh"
#include "internal.h"

namespace pi {

namespace {

// Consumer warps: 8, or 12 for the widest rows.  With 8 warps and x of
// d_model >= 12 Ki fp16 columns each consumer thread holds 6-8 chunks of x and
// the per-row dot products run out of independent work; 12 warps take 4-6
// chunks each (measured on the OPT-175B shape: 52.3 -> 51.0 us per layer;
// narrower rows are slower with 12, so they keep 8).
constexpr int kNCW8 = 8;
constexpr int kMaxNCW = 12;
constexpr int kMaxStages = 24;
constexpr int kMaxShare = 512;     // FFN rows per CTA (share of the active list)
constexpr int kMaxRange = 512;     // neurons per CTA range (P2 rows)
constexpr int kMaxG = 1024;
constexpr int kMaxRank = 2048;
constexpr int kGroup = 8;          // P2 rows per job (12 in the 12-warp variant when a stage holds them)
constexpr int kMaxP1 = 8;          // P1 rows per job
constexpr int kMaxP1R = 16;        // P1 rows per CTA (rank / #SMs)
constexpr int kUpRing = 32;        // FFN up rows in flight (> ring stages)
constexpr int kQTake = 4;          // work-queue slots taken per atomic
constexpr int kOwn = 4;            // queue mode: active neurons a CTA keeps from its own range
constexpr int kJobP1 = 1, kJobP2 = 2, kJobUp = 3, kJobDown = 4, kJobEnd = 5;

struct Tables {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t share_ready;
    int4 job[kMaxStages];
    float redp[kMaxP1R][kMaxNCW];
    float redu[kUpRing][kMaxNCW][2];
    int upcnt[kUpRing];
    unsigned long long seq;
    int share_n;
    int count, total;
    unsigned qbase;     // queue mode: the queue slot of the range's k-th active neuron is qbase + k
    int wsum[kMaxNCW];
    float ssq[kMaxNCW];  // chained input: per-warp sums of squares of x_prev + y_prev
    unsigned words[kMaxRange / 32 + 1];
    unsigned wpre[kMaxRange / 32 + 1];
    float lg[kMaxRange];
    float pb[kMaxRange];
    float ba[kMaxRange];
    alignas(16) float hs[kMaxRank];
    int pref[kMaxG];
    int j[kMaxShare];
    float bias[kMaxShare];
    float a[kMaxShare];
    int state[kMaxShare];
    int fail;           // a wait of this CTA gave up: read by every consumer after the next CTA barrier
};
constexpr size_t kHdr = (sizeof(Tables) + 1023) & ~(size_t)1023;

__device__ __forceinline__ int ld_cg_int(const int *p)
{
    int v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_cg_f32(const float *p)
{
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned ld_volatile_u32(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid barrier, called by one thread per CTA after the CTA's own writes (a CTA
// barrier before the call makes the other threads' writes part of this
// thread's release).  Arrivals add to a 64-bit counter that is never reset;
// the barrier is passed when the counter reaches `target` (a multiple of the
// grid size derived from the launch sequence number).  Returns false on
// timeout.
__device__ bool grid_barrier(unsigned long long *ctr, unsigned long long target, bool wait, const WsCtrl *ctrl,
                             unsigned *err)
{
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(ctr) : "memory");
    if (!wait) return false;
    // the first polls do not depend on the control block's limit (a barrier of
    // a healthy launch passes within them); the limit bounds the rest
    for (int i = 0; i < 64; ++i) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
        if ((long long)(v - target) >= 0) return true;
    }
    const long long limit = poll_limit(ctrl);
    for (long long i = 64; i < limit; ++i) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
        if ((long long)(v - target) >= 0) return true;
        __nanosleep(32);
    }
    atomicOr(err, ERR_TIMEOUT);
    return false;
}

template <typename PT>
__device__ __forceinline__ float dot16(uint4 w, const float *x);
template <>
__device__ __forceinline__ float dot16<__half>(uint4 w, const float *x) { return dot8_f16(w, x); }
template <>
__device__ __forceinline__ float dot16<float>(uint4 w, const float *x) { return dot4_f32(w, x); }

struct FusedParams {
    const uint8_t *p1, *p2;
    const float *p_bias;
    const uint8_t *w_act, *w_up, *w_down;
    const float *b_act, *b_down;
    const float *x, *residual;
    const float *x_prev, *y_prev;  // chained input (or null): x = (x_prev + y_prev) / rms(x_prev + y_prev)
    float *x_out;        // chained input: x is also written here
    float *y;
    int *idx_out;        // ordered active list, or null
    int *n_active;       // or null
    int *cand;           // [F] candidate lists (each CTA writes inside its range)
    float *cand_bias;    // [F] b_act of each candidate
    unsigned long long *qent;  // [F] work-queue entries: (launch sequence + 1) << 32 | neuron
    float *h;            // [rank]
    unsigned *status;    // [G] active count of each CTA's range
    WsCtrl *ctrl;
    int d, F, r, act;
    int queue;
    int prefix;          // neurons [0, prefix) always active; the predictor covers [prefix, F)
    float tau;
};

// Default: one CTA per SM with a deep ring.  With PI_FUSED_COLOCATE, narrow
// layers (at most 16 columns of x per consumer thread) are instead compiled for
// two resident CTAs per SM (a register cap that keeps two CTAs' 18 warps within
// each SM sub-partition's register file) with a shallow ring, so the next
// layer's CTA starts its predictor loads while this one works.
#ifndef PI_FUSED_COLOCATE
#define PI_FUSED_COLOCATE 0
#endif
__host__ __device__ constexpr bool colocate(int epc, int ch) { return PI_FUSED_COLOCATE && epc * ch <= 16; }

// Registers: each SM sub-partition's 16 Ki registers hold the warps placed on
// it.  8 consumer warps + the producer put 3 warps on one sub-partition (at
// most 170 registers a thread); 12 + 1 put 4 there, so that variant declares a
// 512-thread bound, which caps it at 128 registers (it launches 416 threads).
template <int WT, typename PT, bool GATED, int CH, int NCW, int KG>
__global__ void __launch_bounds__(NCW == kNCW8 ? kNCW8 * 32 + 32 : 512, colocate(Fmt<WT>::EPC, CH) ? 2 : 1)
    k_layer_b1(FusedParams p, int nstages, uint32_t stage_bytes)
{
    static_assert(NCW == kNCW8 || NCW == kMaxNCW, "8 or 12 consumer warps");
    static_assert(KG == kGroup || (KG == 12 && NCW == kMaxNCW), "P2 jobs of 8 rows, or 12 with 12 warps");
    constexpr int kNCW = NCW;
    constexpr int kNCT = kNCW * 32;
    constexpr int kThreads = kNCT + 32;
    constexpr int EPC = Fmt<WT>::EPC;                // weight elements per 16-byte chunk
    constexpr int PSEG = EPC * (int)sizeof(PT) / 16; // P1 chunks covering one weight chunk's columns
    constexpr int PEPC = 16 / (int)sizeof(PT);       // predictor elements per 16-byte chunk
    static_assert(PSEG >= 1, "predictor chunk wider than a weight chunk");
    extern __shared__ __align__(128) uint8_t smem[];
    Tables &T = *reinterpret_cast<Tables *>(smem);
    uint8_t *stages = smem + kHdr;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, G = gridDim.x;
    const int d = p.d, F = p.F, r = p.r;
    const uint32_t R = row_slot_bytes(WT, d);
    const int nch = d / EPC;
    unsigned *err = &p.ctrl->err;
    const int hk0 = (int)((long long)r * c / G), hk1 = (int)((long long)r * (c + 1) / G);
    // always-on prefix [0, H): this CTA's slice [pf0, pf0 + npf) of it; the
    // predicted tail [H, F) is split into the CTAs' contiguous neuron ranges
    const int H = p.prefix;
    const int pf0 = (int)((long long)H * c / G), npf = (int)((long long)H * (c + 1) / G) - pf0;
    const int j0 = H + (int)((long long)(F - H) * c / G), j1 = H + (int)((long long)(F - H) * (c + 1) / G);
    const int nP1r = hk1 - hk0, nR = j1 - j0;
    const uint32_t p1row = (uint32_t)d * sizeof(PT), p2row = (uint32_t)r * sizeof(PT);
    const int rp1 = max(1, min(kMaxP1, (int)(stage_bytes / p1row)));  // P1 rows per job
    const int nP1 = (nP1r + rp1 - 1) / rp1;
    const int nP2 = (nR + KG - 1) / KG;
    // No ordered active list requested: the FFN rows come from a shared work
    // queue that every CTA feeds with its range's active neurons, so there is
    // no second grid barrier, no prefix scan and no share lookup, and idle CTAs
    // take rows from busy ones.
    const bool qmode = p.queue != 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            mbar_init(&T.full[s], 1);
            mbar_init(&T.empty[s], kNCW);
        }
        mbar_init(&T.share_ready, 1);
        fence_mbar_init();
    }
    if (threadIdx.x == 0) T.fail = 0;
    for (int i = threadIdx.x; i < kMaxShare; i += kThreads) T.state[i] = 0;
    for (int i = threadIdx.x; i < kUpRing; i += kThreads) T.upcnt[i] = 0;
    for (int i = threadIdx.x; i < nR; i += kThreads) {  // layer constants: no need to wait
        T.pb[i] = p.p_bias ? p.p_bias[j0 + i] : 0.f;
        T.ba[i] = p.b_act ? p.b_act[j0 + i] : 0.f;
    }
    __syncthreads();

    if (warp == kNCW) {
        // ================================ producer =================================
        // The producer reads nothing the previous kernel writes (weights only),
        // so it lets the next kernel launch at once; the consumers do so after
        // their wait.  The next layer's CTA can then start its own predictor
        // loads on this SM while this CTA is still working.
        pdl_trigger();
        if (lane == 0) {
            const unsigned long long pol = evict_first_policy();
            int q = 0;
            bool failed = false;
            auto acquire = [&](int qq) -> bool {
                const int s = qq % nstages;
                return qq < nstages || mbar_wait(&T.empty[s], (unsigned)((qq / nstages) - 1) & 1u, err);
            };
            for (int i = 0; i < nP1 + nP2; ++i) {
                if (!acquire(q)) {
                    failed = true;
                    break;
                }
                const int s = q % nstages;
                uint8_t *st = stages + (size_t)s * stage_bytes;
                if (i < nP1) {
                    const int k0 = hk0 + i * rp1, k1 = min(k0 + rp1, hk1);
                    const uint32_t bytes = (uint32_t)(k1 - k0) * p1row;
                    T.job[s] = make_int4(kJobP1, k0, k1, 0);
                    mbar_arrive_expect_tx(&T.full[s], bytes);
                    bulk_g2s_once(st, p.p1 + (size_t)k0 * p1row, bytes, &T.full[s], pol);
                } else {
                    const int g0 = j0 + (i - nP1) * KG, g1 = min(g0 + KG, j1);
                    const uint32_t bytes = (uint32_t)(g1 - g0) * p2row;
                    T.job[s] = make_int4(kJobP2, g0, g1, 0);
                    mbar_arrive_expect_tx(&T.full[s], bytes);
                    bulk_g2s_once(st, p.p2 + (size_t)g0 * p2row, bytes, &T.full[s], pol);
                }
                ++q;
            }
            // FFN jobs, once the consumers have found this CTA's share: with an
            // ordered active list requested, its slice of that list; otherwise
            // (queue mode) the first active neurons of its own range, then rows
            // from the shared work queue
            if (!failed && !mbar_wait(&T.share_ready, 0u, err)) failed = true;
            int sn = failed ? 0 : T.share_n;
#ifndef PI_FUSED_PREFETCH_DOWN
#define PI_FUSED_PREFETCH_DOWN 0
#endif
            // all the share's rows towards L2 at once (fp16 / fp32 rows: measured
            // faster with it; Q4_0 rows: faster without it)
            for (int i = 0; i < (WT == 2 ? 0 : sn); ++i) {
                const int j = T.j[i];
                if (j < 0 || j >= F) continue;
                prefetch_l2(p.w_act + (size_t)j * R, R);
                if constexpr (GATED) prefetch_l2(p.w_up + (size_t)j * R, R);
                if (PI_FUSED_PREFETCH_DOWN) prefetch_l2(p.w_down + (size_t)j * R, R);
            }
            volatile int *state = T.state;
            int up = 0, ds = 0;
            bool exhausted = !qmode;  // queue mode: more rows may still be published
            int pend = -1, pk = 0;    // queue batch taken: slots [pend + pk, pend + kQTake) not read yet
            long long qspins = 0;
            const unsigned par = (unsigned)T.seq & 1u, tag = (unsigned)T.seq + 1u;
            while (!failed) {
                int kind, i = 0, j = 0;
                if (ds < up && state[ds] != 0) {
                    const int stt = state[ds];
                    i = ds++;
                    if (stt == 1) continue;
                    kind = kJobDown;
                    j = T.j[i];
                } else if (up >= sn && !exhausted) {
                    // take kQTake queue slots with one atomic; read the batch's
                    // remaining slots together; a slot is ready once its tag is
                    // this launch's; a slot at or past the final tail ends the queue
                    if (pend < 0) {
                        if (sn + kQTake > kMaxShare) {
                            exhausted = true;
                            continue;
                        }
                        pend = (int)atomicAdd(&p.ctrl->q_head[par], (unsigned)kQTake);
                        pk = 0;
                        qspins = 0;
                    }
                    unsigned long long ev[kQTake];
#pragma unroll
                    for (int k = 0; k < kQTake; ++k) {
                        const int slot = pend + pk + k;
                        ev[k] = 0ull;
                        if (pk + k < kQTake && slot < F)
                            asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(ev[k]) : "l"(p.qent + slot) : "memory");
                    }
                    int took = 0;
#pragma unroll
                    for (int k = 0; k < kQTake; ++k) {
                        if (took != k || pk + k >= kQTake || sn >= kMaxShare) break;
                        if ((unsigned)(ev[k] >> 32) != tag) break;
                        T.j[sn++] = (int)(unsigned)(ev[k] & 0xffffffffull);
                        ++took;
                    }
                    pk += took;
                    if (pk == kQTake || sn >= kMaxShare) {
                        pend = -1;
                        continue;
                    }
                    if (took > 0) {
                        qspins = 0;
                        continue;  // issue those rows' jobs before looking again
                    }
                    if (ld_acquire_u32(&p.ctrl->q_done[par]) == (unsigned)G &&
                        (unsigned)(pend + pk) >= ld_acquire_u32(&p.ctrl->q_tail[par])) {
                        exhausted = true;  // every CTA has published: the tail is final
                        pend = -1;
                        continue;
                    }
                    if (++qspins < kSpinLimit) {
                        __nanosleep(32);
                        continue;
                    }
                    atomicOr(err, ERR_TIMEOUT);
                    failed = true;
                    kind = kJobEnd;
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
                if (!acquire(q)) {
                    failed = true;
                    break;
                }
                const int s = q % nstages;
                uint8_t *st = stages + (size_t)s * stage_bytes;
                T.job[s] = make_int4(kind, i, j, 0);
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
            if (failed) {  // never leave bulk copies in flight into this CTA's shared memory
                for (int s = 0; s < nstages && s < q; ++s) {
                    const int last = s + ((q - 1 - s) / nstages) * nstages;
                    mbar_wait(&T.full[s], (unsigned)(last / nstages) & 1u, err);
                }
            }
        }
        return;
    }

    // ================================= consumers ===================================
    const int t = threadIdx.x;
    pdl_wait();
    pdl_trigger();
    if (t == 0) T.seq = ld_volatile_u32(&p.ctrl->bar_seq);

    // this thread's float4 of y = b_down + residual (at most one per thread:
    // d/4/G <= 16384/4/#SMs < 256), loads issued now, stored after phase 1
    int yv = -1;
    float4 yval = make_float4(0.f, 0.f, 0.f, 0.f);
    {
        const int nvec = d / 4;
        const int v0 = (int)((long long)nvec * c / G), v1 = (int)((long long)nvec * (c + 1) / G);
        if (v0 + t < v1) {
            yv = v0 + t;
            if (p.b_down) yval = reinterpret_cast<const float4 *>(p.b_down)[yv];
            if (p.residual) {
                const float4 rz = reinterpret_cast<const float4 *>(p.residual)[yv];
                yval.x += rz.x;
                yval.y += rz.y;
                yval.z += rz.z;
                yval.w += rz.w;
            }
        }
    }
    float xr[CH][EPC];
    float acc[CH][EPC];
    if (!p.x_prev) {
#pragma unroll
        for (int u = 0; u < CH; ++u) {
            const int cc = t + kNCT * u;
#pragma unroll
            for (int e = 0; e < EPC; e += 4) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (cc < nch) v = *reinterpret_cast<const float4 *>(p.x + (size_t)cc * EPC + e);
                xr[u][e] = v.x;
                xr[u][e + 1] = v.y;
                xr[u][e + 2] = v.z;
                xr[u][e + 3] = v.w;
                acc[u][e] = acc[u][e + 1] = acc[u][e + 2] = acc[u][e + 3] = 0.f;
            }
        }
    } else {
        // the layer-to-layer glue of a stack, done by every CTA for the whole
        // vector in the same order (so all CTAs hold the same x): v = x_prev +
        // y_prev, x = v / sqrt(mean(v^2)) (0 when v = 0).  Phase 1 runs on v
        // while the sum of squares is reduced (h = max(P1 v, 0) / rms, as P1 is
        // linear and rms > 0), and x itself is formed after it; this CTA's
        // slice of x also goes to x_out
        float ss = 0.f;
#pragma unroll
        for (int u = 0; u < CH; ++u) {
            const int cc = t + kNCT * u;
#pragma unroll
            for (int e = 0; e < EPC; e += 4) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (cc < nch) {
                    const float4 a = *reinterpret_cast<const float4 *>(p.x_prev + (size_t)cc * EPC + e);
                    const float4 b = *reinterpret_cast<const float4 *>(p.y_prev + (size_t)cc * EPC + e);
                    v = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
                }
                xr[u][e] = v.x;
                xr[u][e + 1] = v.y;
                xr[u][e + 2] = v.z;
                xr[u][e + 3] = v.w;
                ss = fmaf(v.x, v.x, ss);
                ss = fmaf(v.y, v.y, ss);
                ss = fmaf(v.z, v.z, ss);
                ss = fmaf(v.w, v.w, ss);
                acc[u][e] = acc[u][e + 1] = acc[u][e + 2] = acc[u][e + 3] = 0.f;
            }
        }
        ss = warp_sum(ss);
        if (lane == 0) T.ssq[warp] = ss;  // read after phase 1's CTA barrier
    }
    bool ok = true;
    int q = 0;

    auto release = [&](int s) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&T.empty[s]);
    };

    // ---- 1. hidden layer: this CTA's P1 rows, rp1 rows per job ----
    for (int i = 0; i < nP1 && ok; ++i, ++q) {
        const int s = q % nstages;
        if (!mbar_wait_warp(&T.full[s], (unsigned)(q / nstages) & 1u, err)) {
            ok = false;
            T.fail = 1;
            break;
        }
        const uint8_t *st = stages + (size_t)s * stage_bytes;
        const int4 job = T.job[s];
        for (int k = 0; k < job.z - job.y; ++k) {
            float part = 0.f;
#pragma unroll
            for (int u = 0; u < CH; ++u) {
                const int cc = t + kNCT * u;
                if (cc < nch) {
#pragma unroll
                    for (int g = 0; g < PSEG; ++g)
                        part += dot16<PT>(*reinterpret_cast<const uint4 *>(st + (size_t)k * p1row +
                                                                             ((size_t)cc * PSEG + g) * 16),
                                          &xr[u][g * PEPC]);
                }
            }
            part = warp_sum(part);
            if (lane == 0) T.redp[job.y - hk0 + k][warp] = part;
        }
        release(s);
    }
    named_bar_sync(1, kNCT);
    // chained input: 1 / rms of v (the per-warp sums of squares were written
    // before phase 1); h and x are scaled by it, x_out gets this CTA's slice
    float xs = 1.f;
    if (p.x_prev) {
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kNCW; ++w) tot += T.ssq[w];
        const float rms = sqrtf(tot / (float)d);
        xs = rms > 0.f ? 1.f / rms : 0.f;
    }
    if (t < nP1r) {
        float z = 0.f;
#pragma unroll
        for (int w = 0; w < kNCW; ++w) z += T.redp[t][w];
        p.h[hk0 + t] = fmaxf(z, 0.f) * xs;
    }
    if (p.x_prev) {
#pragma unroll
        for (int u = 0; u < CH; ++u)
#pragma unroll
            for (int e = 0; e < EPC; ++e) xr[u][e] *= xs;
        const int nvec = d / 4;
        const int v0 = (int)((long long)nvec * c / G), v1 = (int)((long long)nvec * (c + 1) / G);
        if (v0 + t < v1) {
            const float4 a = reinterpret_cast<const float4 *>(p.x_prev)[v0 + t];
            const float4 b = reinterpret_cast<const float4 *>(p.y_prev)[v0 + t];
            reinterpret_cast<float4 *>(p.x_out)[v0 + t] =
                make_float4((a.x + b.x) * xs, (a.y + b.y) * xs, (a.z + b.z) * xs, (a.w + b.w) * xs);
        }
    }
    // y = b_down + residual for this CTA's share (loaded right after the
    // wait, stored here; ordered before every CTA's atomics by barrier A)
    if (yv >= 0) reinterpret_cast<float4 *>(p.y)[yv] = yval;
    // grid barrier A: every CTA's h slice and y initialisation are out
    named_bar_sync(1, kNCT);
    const unsigned long long base = (2ull * T.seq) * (unsigned long long)G;
    const unsigned qpar = (unsigned)T.seq & 1u;
    if (t == 0 && c == 0) {
        // this launch's work-queue counters start from zero (nobody touches them
        // before grid barrier A; the previous launch used the other set)
        p.ctrl->q_head[qpar] = 0u;
        p.ctrl->q_tail[qpar] = 0u;
        p.ctrl->q_done[qpar] = 0u;
    }
    if (t == 0) {
        if (!grid_barrier(&p.ctrl->bar_ctr, base + (unsigned long long)G, ok, p.ctrl, err)) T.fail = 1;
        // every CTA has read this launch's sequence number: move it on (also
        // after a failure, so the sequence stays in step with the counter)
        if (c == 0) atomicAdd(&p.ctrl->bar_seq, 1u);
    }
    named_bar_sync(1, kNCT);
    if (*reinterpret_cast<volatile int *>(&T.fail)) ok = false;  // the same decision in every consumer thread
    for (int k = t; k < r; k += kNCT) T.hs[k] = ld_cg_f32(p.h + k);
    named_bar_sync(1, kNCT);
    // this lane's slices of h for the P2 rows, kept in registers (the first
    // kHreg chunks per lane; wider ranks read the rest from shared memory)
    constexpr int kHreg = 4;
    float hreg[kHreg][PEPC];
    const int nc2 = r / PEPC;
#pragma unroll
    for (int u = 0; u < kHreg; ++u)
#pragma unroll
        for (int e = 0; e < PEPC; ++e) hreg[u][e] = (lane + 32 * u < nc2) ? T.hs[(lane + 32 * u) * PEPC + e] : 0.f;

    // ---- 2. logits of this CTA's neuron range: each warp takes whole P2 jobs
    //         (up to KG rows) round-robin, keeps all rows in flight, and reduces
    //         them with one transposed butterfly (9 shuffles for 8 rows; 6 more
    //         for rows 8-11 of a 12-row job) ----
    {
        static_assert(kGroup == 8, "butterfly below reduces 8 rows (and a second one 4 more)");
        // Rounds of m <= #stages jobs, one per warp, with a consumer barrier
        // between rounds: a stage's previous job is then always released
        // before anyone waits on its next one, so a parity wait never looks
        // two phases ahead (it could not tell them apart).
        const int q0 = q;
        const int mr = min(kNCW, nstages);
        for (int i0 = 0; i0 < nP2; i0 += mr) {  // uniform trip count: every warp meets every barrier
            if (i0 > 0) named_bar_sync(1, kNCT);
            const int i = i0 + warp;
            if (!ok || warp >= mr || i >= nP2) continue;
            const int qq = q0 + i;
            const int s = qq % nstages;
            if (!mbar_wait_warp(&T.full[s], (unsigned)(qq / nstages) & 1u, err)) {
                ok = false;
                T.fail = 1;
                continue;
            }
            const uint8_t *st = stages + (size_t)s * stage_bytes;
            const int4 job = T.job[s];
            const int nrow = job.z - job.y;
            // All KG rows, branch-free, so their loads and FMA chains
            // interleave: rows past nrow read stage bytes that are in bounds
            // (a stage holds KG rows) and are discarded; chunks past the row
            // end load zeros.
            float v[KG];
#pragma unroll
            for (int rr = 0; rr < KG; ++rr) v[rr] = 0.f;
#pragma unroll
            for (int u = 0; u < kHreg; ++u) {
                const bool in = lane + 32 * u < nc2;
#pragma unroll
                for (int rr = 0; rr < KG; ++rr) {
                    uint4 w = make_uint4(0u, 0u, 0u, 0u);
                    if (in) w = *reinterpret_cast<const uint4 *>(st + (size_t)rr * p2row + (size_t)(lane + 32 * u) * 16);
                    v[rr] += dot16<PT>(w, hreg[u]);
                }
            }
            for (int cc = lane + 32 * kHreg; cc < nc2; cc += 32) {  // ranks above 32*kHreg*PEPC
#pragma unroll
                for (int rr = 0; rr < KG; ++rr)
                    v[rr] += dot16<PT>(*reinterpret_cast<const uint4 *>(st + (size_t)rr * p2row + (size_t)cc * 16),
                                       &T.hs[cc * PEPC]);
            }
            // lanes exchange halves of their row set: after the three steps
            // lane l holds row 4*b4 + 2*b3 + b2 (bits of l) summed over the 8
            // lanes sharing those bits; two more steps finish the sum
#pragma unroll
            for (int m = 16, n = kGroup / 2; m >= 4; m >>= 1, n >>= 1) {
                const bool upper = (lane & m) != 0;
#pragma unroll
                for (int k = 0; k < n; ++k) {
                    const float send = upper ? v[k] : v[k + n];
                    const float keep = upper ? v[k + n] : v[k];
                    v[k] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                }
            }
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
            const int rr = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
            if ((lane & 3) == 0 && rr < nrow) T.lg[job.y + rr - j0] = v[0] + T.pb[job.y + rr - j0];
            if constexpr (KG == 12) {
                // rows 8..11: the same exchange over bits 4 and 3 (lane l then
                // holds row 8 + 2*b4 + b3), then three steps finish the sum
#pragma unroll
                for (int m = 16, n = 2; m >= 8; m >>= 1, n >>= 1) {
                    const bool upper = (lane & m) != 0;
#pragma unroll
                    for (int k = 0; k < n; ++k) {
                        const float send = upper ? v[8 + k] : v[8 + k + n];
                        const float keep = upper ? v[8 + k + n] : v[8 + k];
                        v[8 + k] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                    }
                }
                v[8] += __shfl_xor_sync(0xffffffffu, v[8], 4);
                v[8] += __shfl_xor_sync(0xffffffffu, v[8], 2);
                v[8] += __shfl_xor_sync(0xffffffffu, v[8], 1);
                const int r4 = 8 + ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
                if ((lane & 7) == 0 && r4 < nrow) T.lg[job.y + r4 - j0] = v[8] + T.pb[job.y + r4 - j0];
            }
            // the stage's empty barrier counts one arrival per consumer warp:
            // this warp consumed it alone, so it arrives for all of them
            __syncwarp();
            if (lane == 0) mbar_arrive_cnt(&T.empty[s], kNCW);
        }
        q = q0 + nP2;
    }
    named_bar_sync(1, kNCT);
    if (*reinterpret_cast<volatile int *>(&T.fail)) ok = false;
    // after a failure no neuron is published (the logits are not valid)
    const int nw = (nR + 31) >> 5;
    for (int wd = warp; wd < nw; wd += kNCW) {
        const int row = wd * 32 + lane;
        const bool on = ok && row < nR && T.lg[row] > p.tau;
        const unsigned bits = __ballot_sync(0xffffffffu, on);
        if (lane == 0) T.words[wd] = bits;
    }
    named_bar_sync(1, kNCT);
    if (t < 32) {  // prefix of the range's words (nw <= 17)
        const unsigned cw = t < nw ? (unsigned)__popc(T.words[t]) : 0u;
        unsigned inc = cw;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned v = __shfl_up_sync(0xffffffffu, inc, o);
            if (t >= o) inc += v;
        }
        if (t < nw) T.wpre[t] = inc - cw;
        if (t == 31) T.count = (int)inc;
    }
    named_bar_sync(1, kNCT);
    if (qmode) {
        // keep the range's first kOwn active neurons and hand them to the
        // producer; publish the rest as queue entries, count the CTA as
        // published (release), and arrive at barrier B without waiting
        const int own = min(T.count, kOwn);
        for (int wd = warp; wd < nw; wd += kNCW) {
            const unsigned bits = T.words[wd];
            if ((bits >> lane) & 1u) {
                const int k = (int)T.wpre[wd] + __popc(bits & ((1u << lane) - 1u));
                if (k < own) T.j[npf + k] = j0 + wd * 32 + lane;
            }
        }
        for (int i = t; i < npf; i += kNCT) T.j[i] = pf0 + i;  // the prefix slice first
        named_bar_sync(1, kNCT);
        if (t == 0) {
            T.share_n = ok ? npf + own : 0;
            mbar_arrive(&T.share_ready);
            // queue slots for the range's k-th active neuron, k >= own: qbase + k
            T.qbase = T.count > own ? atomicAdd(&p.ctrl->q_tail[qpar], (unsigned)(T.count - own)) - (unsigned)own : 0u;
        }
        named_bar_sync(1, kNCT);
        const unsigned tag = (unsigned)T.seq + 1u;
        for (int wd = warp; wd < nw; wd += kNCW) {
            const unsigned bits = T.words[wd];
            const int k = (int)T.wpre[wd] + __popc(bits & ((1u << lane) - 1u));
            if (((bits >> lane) & 1u) && k >= own) {
                const int pos = (int)(T.qbase + (unsigned)k);
                // tag and neuron in one 8-byte word: a reader that sees the tag sees the neuron
                const unsigned long long e = ((unsigned long long)tag << 32) | (unsigned)(j0 + wd * 32 + lane);
                asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p.qent + pos), "l"(e) : "memory");
            }
        }
        named_bar_sync(1, kNCT);
        if (t == 0) {
            // the release covers the q_tail reservation above; each entry carries
            // its own launch tag, so readers need no ordering for the entries
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&p.ctrl->q_done[qpar]) : "memory");
            asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(&p.ctrl->bar_ctr) : "memory");
        }
    } else {
    // candidate list of this range: ascending active neurons and their biases
    for (int wd = warp; wd < nw; wd += kNCW) {
        const unsigned bits = T.words[wd];
        if ((bits >> lane) & 1u) {
            const int pos = j0 + (int)T.wpre[wd] + __popc(bits & ((1u << lane) - 1u));
            p.cand[pos] = j0 + wd * 32 + lane;
            p.cand_bias[pos] = T.ba[wd * 32 + lane];
        }
    }
    named_bar_sync(1, kNCT);
    if (t == 0) {
        p.status[c] = (unsigned)T.count;
        if (!grid_barrier(&p.ctrl->bar_ctr, base + 2ull * (unsigned long long)G, ok, p.ctrl, err)) T.fail = 1;
    }
    named_bar_sync(1, kNCT);
    if (*reinterpret_cast<volatile int *>(&T.fail)) ok = false;
    // every range's count -> exclusive prefix and total
    for (int i = t; i < G; i += kNCT) T.pref[i] = (int)ld_cg_int(reinterpret_cast<const int *>(p.status) + i);
    named_bar_sync(1, kNCT);
    {
        const int per = (G + kNCT - 1) / kNCT;
        const int i0 = min(G, t * per), i1 = min(G, i0 + per);
        int mine = 0;
        for (int i = i0; i < i1; ++i) mine += T.pref[i];
        int inc = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        if (lane == 31) T.wsum[warp] = inc;
        named_bar_sync(1, kNCT);
        int before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kNCW; ++w) {
            if (w < warp) before += T.wsum[w];
            total += T.wsum[w];
        }
        int run = before + inc - mine;
        for (int i = i0; i < i1; ++i) {
            const int v = T.pref[i];
            T.pref[i] = run;
            run += v;
        }
        if (t == 0) {
            T.total = total;
            if (c == G - 1 && p.n_active && ok) *p.n_active = H + total;
        }
    }
    named_bar_sync(1, kNCT);
    // after a failure the counts are not this launch's: no list, no share
    const int n = ok ? T.total : 0;
    if (p.idx_out && ok) {  // the prefix slice and this range's part of the ordered active list
        for (int i = t; i < npf; i += kNCT) p.idx_out[pf0 + i] = pf0 + i;
        for (int i = t; i < T.count; i += kNCT) p.idx_out[H + T.pref[c] + i] = p.cand[j0 + i];
    }
    // this CTA's share: its prefix slice, then its balanced share of the tail's list
    const int k0 = (int)((long long)n * c / G), k1 = (int)((long long)n * (c + 1) / G);
    const int sn = ok ? npf + min(k1 - k0, kMaxShare - npf) : 0;
    for (int i = t; i < npf && ok; i += kNCT) {
        T.j[i] = pf0 + i;
        T.bias[i] = p.b_act ? p.b_act[pf0 + i] : 0.f;
    }
    for (int i = t; i < sn - npf; i += kNCT) {
        const int k = k0 + i;
        int lo = 0, hi = G - 1;  // last range whose prefix <= k
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (T.pref[mid] <= k) lo = mid; else hi = mid - 1;
        }
        const int at = H + (int)((long long)(F - H) * lo / G) + (k - T.pref[lo]);
        T.j[npf + i] = ld_cg_int(p.cand + at);
        T.bias[npf + i] = ld_cg_f32(p.cand_bias + at);
    }
    named_bar_sync(1, kNCT);
    if (t == 0) {
        T.share_n = sn;
        mbar_arrive(&T.share_ready);
    }
    }  // ordered-list mode

    // ---- 3. the sparse FFN over this CTA's share ----
    bool any = false;
    while (ok) {
        const int s = q % nstages;
        if (!mbar_wait(&T.full[s], (unsigned)(q / nstages) & 1u, err)) break;
        const int4 job = T.job[s];
        if (job.x == kJobEnd) {
            release(s);
            ++q;
            break;
        }
        const uint8_t *st = stages + (size_t)s * stage_bytes;
        bool two = false;  // this pass also took the next job (an up row that has landed)
        int s2 = 0;
        if (job.x == kJobUp) {
            // 12-warp variant: the next job too, when it is an up row whose
            // data has already landed; both rows go through one dot pass and
            // one round of reductions, which halves the fixed cost per row.
            // (The test looks one use ahead on that stage, as the next wait
            // would.  Measured: faster with 12 warps, slower with 8.)
            int4 job2 = make_int4(0, 0, 0, 0);
            if constexpr (kNCW == kMaxNCW) {
                const int q2 = q + 1;
                s2 = q2 % nstages;
                if (__all_sync(0xffffffffu, mbar_test_wait(&T.full[s2], (unsigned)(q2 / nstages) & 1u)))
                    job2 = T.job[s2];
            }
            two = job2.x == kJobUp;
            const uint8_t *st2 = stages + (size_t)s2 * stage_bytes;
            // the row's bias: from the share table, or (queue mode) from b_act,
            // loaded now and used by the warp that finishes the row
            float bj = 0.f, bj2 = 0.f;
            if (lane == 0) {
                bj = qmode ? (p.b_act ? __ldg(p.b_act + job.z) : 0.f) : T.bias[job.y];
                if (two) bj2 = qmode ? (p.b_act ? __ldg(p.b_act + job2.z) : 0.f) : T.bias[job2.y];
            }
            float pa = 0.f, pu = 0.f, pa2 = 0.f, pu2 = 0.f;
#pragma unroll
            for (int u = 0; u < CH; ++u) {
                const int cc = t + kNCT * u;
                if (cc < nch) {
                    pa += chunk_dot<WT>(st, cc, d, xr[u]);
                    if constexpr (GATED) pu += chunk_dot<WT>(st + R, cc, d, xr[u]);
                    if (two) {
                        pa2 += chunk_dot<WT>(st2, cc, d, xr[u]);
                        if constexpr (GATED) pu2 += chunk_dot<WT>(st2 + R, cc, d, xr[u]);
                    }
                }
            }
            pa = warp_sum(pa);
            if constexpr (GATED) pu = warp_sum(pu);
            if (two) {
                pa2 = warp_sum(pa2);
                if constexpr (GATED) pu2 = warp_sum(pu2);
            }
            // the last warp to contribute to a row finishes it: no CTA barrier
            auto finish = [&](const int4 &jb, float va, float vu, float b) {
                const int e = jb.y & (kUpRing - 1);
                T.redu[e][warp][0] = va;
                T.redu[e][warp][1] = vu;
                __threadfence_block();
                if (atomicAdd(&T.upcnt[e], 1) == kNCW - 1) {
                    __threadfence_block();
                    float z = 0.f, uu = 0.f;
#pragma unroll
                    for (int w = 0; w < kNCW; ++w) {
                        z += T.redu[e][w][0];
                        uu += T.redu[e][w][1];
                    }
                    T.upcnt[e] = 0;
                    float a = activate(p.act, z + b);
                    if constexpr (GATED) a *= uu;
                    T.a[jb.y] = a;
                    __threadfence_block();
                    *reinterpret_cast<volatile int *>(&T.state[jb.y]) = (a != 0.f) ? 2 : 1;
                }
            };
            if (lane == 0) {
                finish(job, pa, pu, bj);
                if (two) finish(job2, pa2, pu2, bj2);
            }
        } else {
            const float a = T.a[job.y];
#pragma unroll
            for (int u = 0; u < CH; ++u) {
                const int cc = t + kNCT * u;
                if (cc < nch) chunk_axpy<WT>(st, cc, d, a, acc[u]);
            }
            any = true;
        }
        release(s);
        ++q;
        if (two) {
            release(s2);
            ++q;
        }
    }
    if (!any) return;
    // every CTA adds into all of y: odd CTAs go through their chunks in the
    // opposite order, so that CTAs finishing together queue on fewer of the
    // same lines of y
    auto add = [&](int u, int e) {
        const int cc = t + kNCT * u;
        if (cc < nch)
            atomicAdd(reinterpret_cast<float4 *>(p.y + (size_t)cc * EPC + e),
                      make_float4(acc[u][e], acc[u][e + 1], acc[u][e + 2], acc[u][e + 3]));
    };
    if ((c & 1) == 0) {
#pragma unroll
        for (int u = 0; u < CH; ++u)
#pragma unroll
            for (int e = 0; e < EPC; e += 4) add(u, e);
    } else {
#pragma unroll
        for (int u = CH - 1; u >= 0; --u)
#pragma unroll
            for (int e = EPC - 4; e >= 0; e -= 4) add(u, e);
    }
}

template <int WT, typename PT, bool GATED, int CH, int NCW, int KG = kGroup>
cudaError_t launch_t(const FusedParams &p, int G, int ns, uint32_t stage_bytes, cudaStream_t s)
{
    auto k = k_layer_b1<WT, PT, GATED, CH, NCW, KG>;
    const size_t smem = kHdr + (size_t)ns * stage_bytes;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // all of the unified L1/shared storage as shared memory, so that two CTAs
    // (this layer's and the next one's) fit on an SM
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(G), dim3(NCW * 32 + 32), smem, s, p, ns, stage_bytes);
}

int chunks_per_thread(int wtype, int d, int ncw)
{
    const int epc = wtype == 0 ? 4 : (wtype == 1 ? 8 : 32);
    return (d / epc + ncw * 32 - 1) / (ncw * 32);
}

// kg12: a stage holds 12 P2 rows (then the 12-warp variant takes P2 jobs of
// 12 rows: half as many bytes again in flight in the logits phase, with 12
// warps to take them)
template <int WT, typename PT, bool GATED>
cudaError_t launch_ch(const FusedParams &p, int d, bool kg12, int G, int ns, uint32_t sb, cudaStream_t s)
{
    const int need = chunks_per_thread(WT, d, kNCW8);
    if constexpr (WT != 2) {
        if (need >= 6) {  // the widest rows: 12 consumer warps, 4-6 chunks a thread
            const int need12 = chunks_per_thread(WT, d, kMaxNCW);
            if (need12 <= 4)
                return kg12 ? launch_t<WT, PT, GATED, 4, kMaxNCW, 12>(p, G, ns, sb, s)
                            : launch_t<WT, PT, GATED, 4, kMaxNCW>(p, G, ns, sb, s);
            if (need12 <= 6)
                return kg12 ? launch_t<WT, PT, GATED, 6, kMaxNCW, 12>(p, G, ns, sb, s)
                            : launch_t<WT, PT, GATED, 6, kMaxNCW>(p, G, ns, sb, s);
        }
    }
    if (need <= 1) return launch_t<WT, PT, GATED, 1, kNCW8>(p, G, ns, sb, s);
    if (need <= 2) return launch_t<WT, PT, GATED, 2, kNCW8>(p, G, ns, sb, s);
    if constexpr (WT != 2) {
        if (need <= 3) return launch_t<WT, PT, GATED, 3, kNCW8>(p, G, ns, sb, s);
        if (need <= 4) return launch_t<WT, PT, GATED, 4, kNCW8>(p, G, ns, sb, s);
        if (need <= 6) return launch_t<WT, PT, GATED, 6, kNCW8>(p, G, ns, sb, s);
        if (need <= 8) return launch_t<WT, PT, GATED, 8, kNCW8>(p, G, ns, sb, s);
    }
    return cudaErrorNotSupported;
}

}  // namespace

bool fused_layer_supported(int wtype, int ptype, int d, int F, int r, int prefix)
{
    const int G = sm_count();
    // a CTA's share table holds its prefix slice and its share of the tail's list
    if ((prefix + G - 1) / G + (F - prefix + G - 1) / G > kMaxShare) return false;
    if (G > kMaxG || r > kMaxRank || (r + G - 1) / G > kMaxP1R) return false;
    if ((d / 4 + G - 1) / G > kNCW8 * 32) return false;  // y initialisation: one float4 per consumer thread
    if (!((wtype == 1 && ptype == 1) || (wtype == 2 && ptype == 1) || (wtype == 0 && ptype == 0))) return false;
    if ((F + G - 1) / G > kMaxRange) return false;
    return chunks_per_thread(wtype, d, kNCW8) <= (wtype == 2 ? 2 : 8);
}

cudaError_t launch_layer_b1(const LayerB1Args &a, cudaStream_t s)
{
    const int G = sm_count();
    FusedParams p{};
    p.p1 = static_cast<const uint8_t *>(a.p1);
    p.p2 = static_cast<const uint8_t *>(a.p2);
    p.p_bias = a.p_bias;
    p.w_act = static_cast<const uint8_t *>(a.gated ? a.w_gate : a.w_up);
    p.w_up = static_cast<const uint8_t *>(a.gated ? a.w_up : nullptr);
    p.w_down = static_cast<const uint8_t *>(a.w_down);
    p.b_act = a.b_act;
    p.b_down = a.b_down;
    p.x = a.x;
    p.residual = a.residual;
    p.x_prev = a.x_prev;
    p.y_prev = a.y_prev;
    p.x_out = a.x_out;
    p.y = a.y;
    p.idx_out = a.idx_out;
    p.n_active = a.n_active;
    p.cand = a.cand;
    p.cand_bias = a.cand_bias;
    p.qent = a.qent;
    p.h = a.h;
    p.status = a.status;
    p.ctrl = a.ctrl;
    p.d = a.d;
    p.F = a.F;
    p.r = a.r;
    p.act = a.act;
    p.tau = a.tau;
    p.queue = (!a.idx_out && !a.n_active && (long long)a.F <= (long long)(kMaxShare - kQTake + 1) * G) ? 1 : 0;
    p.prefix = a.prefix;
    const int esz = a.ptype == 1 ? 2 : 4;
    const uint32_t R = row_slot_bytes(a.wtype, a.d);
    uint32_t sb = std::max<uint32_t>({(uint32_t)a.d * esz, (uint32_t)kGroup * a.r * esz, (a.gated ? 2u : 1u) * R});
    const bool kg12 = 12u * (uint32_t)a.r * esz <= std::max<uint32_t>((uint32_t)a.d * esz, (a.gated ? 2u : 1u) * R);
    sb = (sb + 127u) & ~127u;
    const int need = chunks_per_thread(a.wtype, a.d, kNCW8);
    const int epc = a.wtype == 0 ? 4 : (a.wtype == 1 ? 8 : 32);
    const size_t budget = (size_t)(colocate(epc, need) ? 110 : 226) * 1024;
    int ns = (int)((budget - kHdr) / sb);
    ns = std::max(2, std::min(ns, kMaxStages));
    if (kHdr + (size_t)ns * sb > 227 * 1024) return cudaErrorNotSupported;
    switch (a.wtype * 2 + (a.gated ? 1 : 0)) {
    case 0: return launch_ch<0, float, false>(p, a.d, kg12, G, ns, sb, s);
    case 1: return launch_ch<0, float, true>(p, a.d, kg12, G, ns, sb, s);
    case 2: return launch_ch<1, __half, false>(p, a.d, kg12, G, ns, sb, s);
    case 3: return launch_ch<1, __half, true>(p, a.d, kg12, G, ns, sb, s);
    case 4: return launch_ch<2, __half, false>(p, a.d, kg12, G, ns, sb, s);
    case 5: return launch_ch<2, __half, true>(p, a.d, kg12, G, ns, sb, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pi
