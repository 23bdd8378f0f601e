// Allocation-free variant of the one-token layer step (pi_ffn_layer at
// batch 1), for callers that cannot allocate device memory themselves -- for
// example code running inside a host callback or a custom allocator hook,
// a plugin whose host application forbids cudaMalloc, or any thread that
// must not synchronise the device, which cudaMalloc and cudaFree may do.
//
// Its workspace is one file-scope device array of fixed size.  The array lives
// on every GPU that loads the library, from module load until the process
// exits.  Host code may not hand the array's name to a kernel (on the host it
// is only a stand-in symbol), so every call looks up the array's device
// address with cudaGetSymbolAddress while the caller's device is current (no
// allocation; looking it up each time keeps a cudaDeviceReset between calls
// harmless).  The first call on a device may load the library's device code,
// so it should come before any stream capture.  No call allocates: no
// cudaMalloc, no cudaFree, no allocating library routine.
//
// All calls on a device share the array and leave their contents in it.  A
// small kernel at the start of each call prepares it: it clears the error word,
// and it zero-fills the whole region the layer uses when the layer's shape or
// storage types differ from the previous call's on that device, or when the
// previous call left a timeout in the error word (a wait that gave up can
// leave the barrier and queue state out of step).  Two calls that overlap on
// the GPU (different streams, or different host threads without ordering)
// race on the array and give wrong results.
#include <mutex>

#include "internal.h"
#include "pi.h"

namespace {

// Largest layer this entry point accepts: d_ff <= 65536, rank <= 2048, one
// token.  ws_layout() of that shape needs 256 + 16 KiB + 4 KiB + 8 KiB +
// 256 KiB + 256 bytes + 256 KiB + 512 KiB, rounded up here to 1088 KiB.
constexpr size_t kStaticWsBytes = 1088 * 1024;
constexpr int kStaticMaxDff = 65536;

__device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

struct LastShape {
    bool valid;
    int d_model, d_ff, rank, wtype, ptype;
};
std::mutex g_mu;
LastShape g_last[64] = {};

// One block: read the error word the previous call left, then clear the error
// word, or zero-fill the first n16 16-byte words when asked to (reset) or when
// that word holds a timeout.
__global__ void k_static_prepare(uint4 *ws, size_t n16, int reset)
{
    __shared__ int wipe;
    if (threadIdx.x == 0) {
        const unsigned prev = *reinterpret_cast<volatile unsigned *>(ws);
        wipe = reset || (prev & pi::ERR_TIMEOUT) != 0u;
    }
    __syncthreads();
    if (!wipe) {
        if (threadIdx.x == 0) *reinterpret_cast<unsigned *>(ws) = 0u;
        return;
    }
    for (size_t i = threadIdx.x; i < n16; i += blockDim.x) ws[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Device address of g_static_ws on the current device, and the device ordinal.
pi_status static_ws(void **out, int *dev_out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PI_ERR_CUDA;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return PI_ERR_CUDA;
    *out = p;
    *dev_out = dev;
    return PI_OK;
}

}  // namespace

extern "C" PI_API pi_status pi_ffn_layer_static(const pi_ffn_desc *desc, const float *x, const float *residual,
                                                float *y, int32_t *idx, int32_t *n_active, int32_t *status_out,
                                                pi_stream stream)
{
    if (!desc) return PI_ERR_NULL;
    if (desc->d_model < 8 || desc->d_ff < 1 || desc->rank < 0) return PI_ERR_SHAPE;
    if (desc->d_ff > kStaticMaxDff || desc->rank > PI_MAX_RANK) return PI_ERR_SHAPE;
    const pi::WsLayout L = pi::ws_layout(desc->d_model, desc->d_ff, desc->rank, 1);
    if (L.total > kStaticWsBytes) return PI_ERR_SHAPE;
    if (status_out && ((uintptr_t)status_out & 3)) return PI_ERR_ALIGN;
    void *ws = nullptr;
    int dev = 0;
    pi_status st = static_ws(&ws, &dev);
    if (st != PI_OK) return st;
    const cudaStream_t s = (cudaStream_t)stream;
    int reset = 0;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        LastShape &ls = g_last[dev];
        const LastShape now = {true, desc->d_model, desc->d_ff, desc->rank, desc->wtype, desc->ptype};
        reset = !(ls.valid && ls.d_model == now.d_model && ls.d_ff == now.d_ff && ls.rank == now.rank &&
                  ls.wtype == now.wtype && ls.ptype == now.ptype);
        ls = now;
    }
    k_static_prepare<<<1, 1024, 0, s>>>(static_cast<uint4 *>(ws), L.total / 16, reset);
    if (cudaGetLastError() != cudaSuccess) return PI_ERR_CUDA;
    st = pi_ffn_layer(desc, x, 1, residual, y, idx, n_active, ws, L.total, stream);
    if (st != PI_OK) return st;
    if (status_out &&
        cudaMemcpyAsync(status_out, ws, sizeof(unsigned), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return PI_ERR_CUDA;
    return PI_OK;
}
