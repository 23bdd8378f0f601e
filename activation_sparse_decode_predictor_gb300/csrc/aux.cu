// Small kernels around the sparse FFN: output initialisation, Q4_0
// quantisation, offline firing-count profiling, row permutation and the
// layer-to-layer glue of an FFN stack.
#include "internal.h"

namespace pi {

namespace {

// y = b_down + residual (either may be absent); optionally idx = 0..count-1, *n = count.
__global__ void k_init_y(float *__restrict__ y, const float *__restrict__ b_down, const float *residual, int B, int d,
                         int *iota_idx, int *iota_n, int iota_count)
{
    pdl_wait();
    pdl_trigger();
    const int nvec = B * d / 4;
    const int stride = gridDim.x * blockDim.x;
    for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        if (b_down) o = reinterpret_cast<const float4 *>(b_down)[v % (d / 4)];
        if (residual) {
            const float4 r = reinterpret_cast<const float4 *>(residual)[v];
            o.x += r.x;
            o.y += r.y;
            o.z += r.z;
            o.w += r.w;
        }
        reinterpret_cast<float4 *>(y)[v] = o;
    }
    if (iota_idx) {
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < iota_count; i += stride) iota_idx[i] = i;
        if (blockIdx.x == 0 && threadIdx.x == 0) *iota_n = iota_count;
    }
}

// Q4_0 quantiser, one thread per block of 32 weights (definition in pi.h).
template <typename ST>
__device__ __forceinline__ float load_w(const ST *p);
template <>
__device__ __forceinline__ float load_w<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float load_w<__half>(const __half *p) { return __half2float(*p); }

template <typename ST>
__global__ void k_quantize_q4_0(const ST *__restrict__ src, int64_t rows, int64_t cols, uint8_t *__restrict__ dst)
{
    const int64_t nblk_row = cols / 32;
    const int64_t nblk = rows * nblk_row;
    uint8_t *codes = dst;
    __half *scales = reinterpret_cast<__half *>(dst + rows * (cols / 2));
    for (int64_t blk = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; blk < nblk;
         blk += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = blk / nblk_row, b = blk % nblk_row;
        const ST *w = src + j * cols + b * 32;
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = load_w<ST>(w + e);
        float amax = v[0];
#pragma unroll
        for (int e = 1; e < 32; ++e)
            if (fabsf(v[e]) > fabsf(amax)) amax = v[e];
        const float s32 = __fdiv_rn(amax, -8.0f);
        const __half s16 = s32 == 0.0f ? __float2half_rn(0.0f) : __float2half_rn(s32);
        const float s = __half2float(s16);
        uint8_t q[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            int qi = 8;
            if (s != 0.0f) {
                const float fl = floorf(__fadd_rn(__fdiv_rn(v[e], s), 8.5f));
                qi = fl < 0.0f ? 0 : (fl > 15.0f ? 15 : (int)fl);
            }
            q[e] = (uint8_t)qi;
        }
        uint8_t *cb = codes + j * (cols / 2) + b * 16;
#pragma unroll
        for (int e = 0; e < 16; ++e) cb[e] = (uint8_t)(q[e] | (q[e + 16] << 4));
        scales[j * nblk_row + b] = s16;
    }
}

// Offline profiling: counts[j] += #{t : W[j] . X[t] + b[j] > 0}.  A plain
// shared-memory tiled product (64 neurons x 64 tokens per CTA, 4x4 per thread).
template <typename WT_>
__global__ void __launch_bounds__(256) k_fire_counts(const WT_ *__restrict__ w, const float *__restrict__ bias,
                                                     const float *__restrict__ X, int T, int d, int F,
                                                     int *__restrict__ counts)
{
    __shared__ float Ws[64][33];
    __shared__ float Xs[64][33];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int row0 = blockIdx.x * 64, tok0 = blockIdx.y * 64;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < d; k0 += 32) {
        for (int e = threadIdx.x; e < 64 * 32; e += 256) {
            const int rr = e >> 5, kk = e & 31;
            const int row = row0 + rr, tok = tok0 + rr, k = k0 + kk;
            Ws[rr][kk] = (row < F && k < d) ? load_w<WT_>(w + (size_t)row * d + k) : 0.f;
            Xs[rr][kk] = (tok < T && k < d) ? X[(size_t)tok * d + k] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < 32; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = Ws[ty * 4 + i][kk];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Xs[tx * 4 + j][kk];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = row0 + ty * 4 + i;
        if (row >= F) continue;
        const float bj = bias ? bias[row] : 0.f;
        int c = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int tok = tok0 + tx * 4 + j;
            if (tok < T && acc[i][j] + bj > 0.f) ++c;
        }
        if (c) atomicAdd(&counts[row], c);
    }
}

// dst row i = src row idx[i] for i < dst_rows; an entry outside [0, src_rows)
// leaves its destination row unwritten.
__global__ void k_gather_rows16(const uint4 *__restrict__ src, int64_t src_rows, uint4 *__restrict__ dst,
                                int64_t dst_rows, int64_t vec_per_row, const int *__restrict__ idx)
{
    const int64_t total = dst_rows * vec_per_row;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = e / vec_per_row, v = e % vec_per_row;
        const int r = idx[i];
        if (r < 0 || r >= src_rows) continue;
        dst[e] = src[(int64_t)r * vec_per_row + v];
    }
}

__global__ void k_gather_rows1(const uint8_t *__restrict__ src, int64_t src_rows, uint8_t *__restrict__ dst,
                               int64_t dst_rows, int64_t row_bytes, const int *__restrict__ idx)
{
    const int64_t total = dst_rows * row_bytes;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = e / row_bytes, v = e % row_bytes;
        const int r = idx[i];
        if (r < 0 || r >= src_rows) continue;
        dst[e] = src[(int64_t)r * row_bytes + v];
    }
}

// x_next = v / sqrt(mean(v^2)), v = x + y; one CTA per token.
__global__ void __launch_bounds__(256) k_rms_residual(const float *x, const float *y, int d, float *out)
{
    __shared__ float part[8];
    pdl_wait();
    pdl_trigger();
    const size_t off = (size_t)blockIdx.x * d;
    float ss = 0.f;
    for (int i = threadIdx.x; i < d; i += 256) {
        const float v = x[off + i] + y[off + i];
        ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += part[w];
    const float rms = sqrtf(tot / (float)d);
    __syncthreads();
    for (int i = threadIdx.x; i < d; i += 256) {
        const float v = x[off + i] + y[off + i];
        out[off + i] = rms > 0.f ? v / rms : 0.f;
    }
}

// The same for 16-byte aligned rows with d % 4 == 0 and d <= 16384: 1024 threads,
// each holding up to four float4 of v in registers across the sum and the write,
// so a token costs one memory round trip instead of two strided passes.
constexpr int kRmsThreads = 1024;
constexpr int kRmsVec = 4;

__global__ void __launch_bounds__(kRmsThreads) k_rms_residual4(const float4 *x, const float4 *y, int d4, float4 *out)
{
    __shared__ float part[kRmsThreads / 32];
    pdl_wait();
    pdl_trigger();
    const size_t off = (size_t)blockIdx.x * d4;
    float4 v[kRmsVec];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < kRmsVec; ++k) {
        const int i = threadIdx.x + kRmsThreads * k;
        v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < d4) {
            const float4 a = x[off + i], b = y[off + i];
            v[k] = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
        }
        ss = fmaf(v[k].x, v[k].x, ss);
        ss = fmaf(v[k].y, v[k].y, ss);
        ss = fmaf(v[k].z, v[k].z, ss);
        ss = fmaf(v[k].w, v[k].w, ss);
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kRmsThreads / 32; ++w) tot += part[w];
    const float rms = sqrtf(tot / (float)(4 * d4));
#pragma unroll
    for (int k = 0; k < kRmsVec; ++k) {
        const int i = threadIdx.x + kRmsThreads * k;
        if (i < d4)
            out[off + i] = rms > 0.f ? make_float4(v[k].x / rms, v[k].y / rms, v[k].z / rms, v[k].w / rms)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

int grid_for(int64_t work, int threads)
{
    int64_t g = (work + threads - 1) / threads;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (g > cap) g = cap;
    return g < 1 ? 1 : (int)g;
}

}  // namespace

cudaError_t launch_init_y(float *y, const float *b_down, const float *residual, int B, int d, int *iota_idx,
                          int *iota_n, int iota_count, cudaStream_t s)
{
    const int64_t work = (int64_t)B * d / 4 > iota_count ? (int64_t)B * d / 4 : iota_count;
    return launch_pdl(k_init_y, dim3(grid_for(work, 256)), dim3(256), 0, s, y, b_down, residual, B, d, iota_idx,
                      iota_n, iota_count);
}

cudaError_t launch_quantize_q4_0(const void *src, int src_type, int64_t rows, int64_t cols, void *dst, cudaStream_t s)
{
    const int64_t nblk = rows * (cols / 32);
    const int g = grid_for(nblk, 128);
    if (src_type == 1)
        k_quantize_q4_0<__half><<<g, 128, 0, s>>>(static_cast<const __half *>(src), rows, cols,
                                                   static_cast<uint8_t *>(dst));
    else
        k_quantize_q4_0<float><<<g, 128, 0, s>>>(static_cast<const float *>(src), rows, cols,
                                                  static_cast<uint8_t *>(dst));
    return cudaGetLastError();
}

cudaError_t launch_fire_counts(int wtype, const void *w, const float *b, const float *X, int T, int d, int F,
                               int *counts, cudaStream_t s)
{
    const dim3 grid((F + 63) / 64, (T + 63) / 64);
    if (wtype == 1)
        k_fire_counts<__half><<<grid, 256, 0, s>>>(static_cast<const __half *>(w), b, X, T, d, F, counts);
    else
        k_fire_counts<float><<<grid, 256, 0, s>>>(static_cast<const float *>(w), b, X, T, d, F, counts);
    return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void *src, int64_t src_rows, void *dst, int64_t dst_rows, int64_t row_bytes,
                               const int *idx, cudaStream_t s)
{
    const bool vec = row_bytes % 16 == 0 && ((uintptr_t)src & 15) == 0 && ((uintptr_t)dst & 15) == 0;
    if (vec) {
        const int64_t vpr = row_bytes / 16;
        k_gather_rows16<<<grid_for(dst_rows * vpr, 256), 256, 0, s>>>(
            static_cast<const uint4 *>(src), src_rows, static_cast<uint4 *>(dst), dst_rows, vpr, idx);
    } else {
        k_gather_rows1<<<grid_for(dst_rows * row_bytes, 256), 256, 0, s>>>(
            static_cast<const uint8_t *>(src), src_rows, static_cast<uint8_t *>(dst), dst_rows, row_bytes, idx);
    }
    return cudaGetLastError();
}

cudaError_t launch_permute_rows(const void *src, void *dst, int64_t rows, int64_t row_bytes, const int *perm,
                                cudaStream_t s)
{
    return launch_gather_rows(src, rows, dst, rows, row_bytes, perm, s);
}

cudaError_t launch_rms_residual(const float *x, const float *y, int B, int d, float *out, cudaStream_t s)
{
    const bool vec = d % 4 == 0 && d <= 4 * kRmsVec * kRmsThreads && (((uintptr_t)x | (uintptr_t)y | (uintptr_t)out) & 15) == 0;
    if (vec)
        return launch_pdl(k_rms_residual4, dim3(B), dim3(kRmsThreads), 0, s, reinterpret_cast<const float4 *>(x),
                          reinterpret_cast<const float4 *>(y), d / 4, reinterpret_cast<float4 *>(out));
    return launch_pdl(k_rms_residual, dim3(B), dim3(256), 0, s, x, y, d, out);
}

}  // namespace pi
