// Device helpers shared by the sparse-FFN kernels: 16-byte weight chunks of one
// neuron row held in shared memory (fp32, fp16 or one Q4_0 block), their dot
// product with fp32 activations, their axpy into fp32 accumulators, and the
// bulk copies that bring one neuron row into a stage slot.
#pragma once

#include "common.cuh"

namespace pi {

// Weight storage: 0 fp32 (4/chunk), 1 fp16 (8/chunk), 2 Q4_0 (32/chunk = one block).
template <int WT>
struct Fmt {
    static constexpr int EPC = WT == 0 ? 4 : (WT == 1 ? 8 : 32);
};

// Bytes of one matrix row in a stage slot; Q4_0 = codes then scales.
__host__ __device__ inline uint32_t row_slot_bytes(int wt, int d)
{
    return wt == 0 ? (uint32_t)d * 4u : (wt == 1 ? (uint32_t)d * 2u : (uint32_t)(d / 2 + d / 16));
}

template <int WT>
__device__ __forceinline__ float chunk_dot(const uint8_t *slot, int c, int d, const float *x)
{
    if constexpr (WT == 0) {
        return dot4_f32(*reinterpret_cast<const uint4 *>(slot + c * 16), x);
    } else if constexpr (WT == 1) {
        return dot8_f16(*reinterpret_cast<const uint4 *>(slot + c * 16), x);
    } else {
        const uint4 q = *reinterpret_cast<const uint4 *>(slot + c * 16);
        const float sc = __half2float(*reinterpret_cast<const __half *>(slot + d / 2 + c * 2));
        const unsigned w[4] = {q.x, q.y, q.z, q.w};
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
                const unsigned byte = (w[k] >> (8 * bb)) & 0xffu;
                const int e = 4 * k + bb;
                s = fmaf((float)((int)(byte & 15u) - 8), x[e], s);
                s = fmaf((float)((int)(byte >> 4) - 8), x[e + 16], s);
            }
        }
        return s * sc;
    }
}

template <int WT>
__device__ __forceinline__ void chunk_axpy(const uint8_t *slot, int c, int d, float a, float *acc)
{
    if constexpr (WT == 0) {
        const uint4 w = *reinterpret_cast<const uint4 *>(slot + c * 16);
        acc[0] = fmaf(a, __uint_as_float(w.x), acc[0]);
        acc[1] = fmaf(a, __uint_as_float(w.y), acc[1]);
        acc[2] = fmaf(a, __uint_as_float(w.z), acc[2]);
        acc[3] = fmaf(a, __uint_as_float(w.w), acc[3]);
    } else if constexpr (WT == 1) {
        const uint4 w = *reinterpret_cast<const uint4 *>(slot + c * 16);
        const unsigned u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = h2f(u[k]);
            acc[2 * k] = fmaf(a, f.x, acc[2 * k]);
            acc[2 * k + 1] = fmaf(a, f.y, acc[2 * k + 1]);
        }
    } else {
        const uint4 q = *reinterpret_cast<const uint4 *>(slot + c * 16);
        const float as = a * __half2float(*reinterpret_cast<const __half *>(slot + d / 2 + c * 2));
        const unsigned w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
                const unsigned byte = (w[k] >> (8 * bb)) & 0xffu;
                const int e = 4 * k + bb;
                acc[e] = fmaf(as, (float)((int)(byte & 15u) - 8), acc[e]);
                acc[e + 16] = fmaf(as, (float)((int)(byte >> 4) - 8), acc[e + 16]);
            }
        }
    }
}

// Issue the bulk copies of one matrix row of neuron j into a stage slot, with
// the L2 policy `pol` (evict_first_policy(): each row is read once per step).
template <int WT>
__device__ __forceinline__ void copy_row(uint8_t *slot, const uint8_t *base, int j, int d, int F, uint64_t *bar,
                                         unsigned long long pol)
{
    if constexpr (WT == 2) {
        const size_t cb = (size_t)d / 2, sb = (size_t)d / 16;
        bulk_g2s_once(slot, base + (size_t)j * cb, (uint32_t)cb, bar, pol);
        bulk_g2s_once(slot + cb, base + (size_t)F * cb + (size_t)j * sb, (uint32_t)sb, bar, pol);
    } else {
        const size_t rb = (size_t)d * (WT == 0 ? 4 : 2);
        bulk_g2s_once(slot, base + (size_t)j * rb, (uint32_t)rb, bar, pol);
    }
}

__device__ __forceinline__ float activate(int act, float z)
{
    const float r = fmaxf(z, 0.f);
    return act == 1 ? r * r : r;
}

}  // namespace pi
