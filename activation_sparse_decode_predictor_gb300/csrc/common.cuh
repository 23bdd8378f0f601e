// Shared device helpers of the sparse-FFN library: inline PTX for programmatic
// dependent launch, L2 bulk prefetch, mbarriers and 1-D bulk (TMA) copies, plus
// the workspace control block.  sm_103a only.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pi {

// Error bits of the device error word (first word of every workspace).
enum : unsigned { ERR_TIMEOUT = 1u, ERR_CAPACITY = 2u, ERR_INDEX = 4u };

// Upper bound on polls of any device-side wait before it gives up, sets
// ERR_TIMEOUT and returns.  Each poll backs off with __nanosleep, so a lost
// wake-up costs well under a second instead of hanging the GPU.
constexpr long long kSpinLimit = 1ll << 22;

// First 256 bytes of a workspace.
struct WsCtrl {
    unsigned err;           // ERR_* bits, cleared by pi_sync_status
    unsigned poll_limit;    // polls of a cross-CTA wait before it gives up (0: kSpinLimit)
    unsigned done;          // scan: CTAs finished in the running launch
    unsigned epoch;         // scan: launch generation, tags the CTA status words
    unsigned long long bar_ctr;  // one-kernel layer step: grid-barrier arrivals (never reset)
    unsigned bar_seq;            // one-kernel layer step: launches completed (moves barrier targets)
    unsigned q_head[2];          // one-kernel layer step, work queue (by launch parity): rows taken
    unsigned q_tail[2];          //   rows reserved by publishing CTAs
    unsigned q_done[2];          //   CTAs that have published all their rows
    unsigned pad[51];
};
static_assert(sizeof(WsCtrl) == 256, "control block is 256 bytes");

// ---- programmatic dependent launch ------------------------------------------------
// Every kernel waits for its predecessor before touching anything the
// predecessor may write, and only then lets its own dependent start; so at most
// two adjacent kernels of a stream ever run at once, and only the part of a
// kernel before pdl_wait() (weight prefetch, barrier set-up) overlaps.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- L2 prefetch of a contiguous range (16-byte aligned start, size % 16 == 0) ------
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---- loads ------------------------------------------------------------------------
// Streaming 16-byte load: read once, do not keep in L1.
__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ unsigned long long ld_volatile_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.volatile.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_volatile_u64(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.volatile.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---- 16-byte weight chunks ----------------------------------------------------------
// fp16: 8 weights; fp32: 4 weights.  dot with fp32 activations (fp32 FMA).
__device__ __forceinline__ float2 h2f(unsigned u)
{
    __half2 h = *reinterpret_cast<__half2 *>(&u);
    return __half22float2(h);
}

// Two accumulator chains of four: a consumer warp has few neighbours on its
// SM sub-partition to hide FMA latency behind, so a chain of 8 dependent FMAs
// per chunk left it waiting.
__device__ __forceinline__ float dot8_f16(uint4 w, const float *x)
{
    float2 a = h2f(w.x), b = h2f(w.y), c = h2f(w.z), d = h2f(w.w);
    float s0 = a.x * x[0], s1 = a.y * x[1];
    s0 = fmaf(b.x, x[2], s0);
    s1 = fmaf(b.y, x[3], s1);
    s0 = fmaf(c.x, x[4], s0);
    s1 = fmaf(c.y, x[5], s1);
    s0 = fmaf(d.x, x[6], s0);
    s1 = fmaf(d.y, x[7], s1);
    return s0 + s1;
}

__device__ __forceinline__ float dot4_f32(uint4 w, const float *x)
{
    float s = __uint_as_float(w.x) * x[0];
    s = fmaf(__uint_as_float(w.y), x[1], s);
    s = fmaf(__uint_as_float(w.z), x[2], s);
    s = fmaf(__uint_as_float(w.w), x[3], s);
    return s;
}

// ---- mbarrier + bulk copy (shared::cta addresses as 32-bit) --------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}

// `count` arrivals at once (a stage consumed by one warp on behalf of all).
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t *bar, uint32_t count)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
                 "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: the thread sleeps in hardware until the
// phase completes or about `ns` nanoseconds pass, instead of spinning on the
// shared-memory pipe that the computing warps need.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, unsigned parity, uint32_t ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

#ifndef PI_MBAR_WAIT_MODE
#define PI_MBAR_WAIT_MODE 0
#endif
#ifndef PI_MBAR_SUSPEND_NS
#define PI_MBAR_SUSPEND_NS 10000u
#endif

// Poll limit of the cross-CTA waits of a launch: the control block's setting,
// or kSpinLimit when it is 0.
__device__ __forceinline__ long long poll_limit(const WsCtrl *c)
{
    const unsigned v = *reinterpret_cast<const volatile unsigned *>(&c->poll_limit);
    return v ? (long long)v : kSpinLimit;
}

// Bounded wait for the phase with the given parity to complete (a bounded
// number of polls, well under a second in total), then it raises
// ERR_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity, unsigned *err)
{
#if PI_MBAR_WAIT_MODE == 0
    for (int i = 0; i < (1 << 16); ++i)
        if (mbar_try_wait_sleep(bar, parity, PI_MBAR_SUSPEND_NS)) return true;
#elif PI_MBAR_WAIT_MODE == 1
    for (long long i = 0; i < kSpinLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
#else
    for (long long i = 0; i < kSpinLimit; ++i) {
        if (mbar_test_wait(bar, parity)) return true;
        __nanosleep(32);
    }
#endif
    atomicOr(err, ERR_TIMEOUT);
    return false;
}

// 1-D bulk copy global -> shared (own CTA), completion counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// mbar_wait by all 32 lanes of a warp with one answer for the warp: true only
// when every lane saw the phase complete, so that no lane leaves a loop of
// warp-wide shuffles that the others stay in.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, unsigned parity, unsigned *err)
{
    const bool got = mbar_wait(bar, parity, err);
    return __all_sync(0xffffffffu, got);
}

// L2 evict-first policy for weights that one decode step reads once, so their
// lines leave L2 before data that is read again (activations, the work queue,
// the control block).  Made
// once per issuing thread: createpolicy is an instruction of its own, and a
// producer that made it before every copy paid for it on each one.
__device__ __forceinline__ unsigned long long evict_first_policy()
{
    unsigned long long pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// bulk_g2s with an L2 cache policy from evict_first_policy().
__device__ __forceinline__ void bulk_g2s_once(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              unsigned long long pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace pi
