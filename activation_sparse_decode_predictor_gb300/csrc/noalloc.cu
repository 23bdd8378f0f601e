// Allocation-free variant of the one-token layer step (pi_ffn_layer at
// batch 1), for callers that cannot allocate device memory themselves -- for
// example code running inside a host callback or a custom allocator hook,
// a plugin whose host application forbids cudaMalloc, or any thread that
// must not synchronise the device, which cudaMalloc and cudaFree may do.
//
// Its workspace is one file-scope device array of fixed size.  The array lives
// on every GPU that loads the library, from module load until the process
// exits.  Host code may not hand the array's name to a kernel (on the host it
// is only a stand-in symbol), so the first call on each device looks up the
// array's device address with cudaGetSymbolAddress while that device is
// current, and caches it.  That first call should therefore come before any
// stream capture.  The call allocates nothing: no cudaMalloc, no cudaFree, no
// allocating library routine.
//
// All calls on a device share the array and leave their contents in it.  The
// scan state in it keeps itself consistent from call to call; the error word
// is cleared at the start of each call.  Two calls that overlap on the GPU
// (different streams, or different host threads without ordering) race on the
// array and give wrong results.
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

std::mutex g_mu;
void *g_addr[64] = {nullptr};

// Device address of g_static_ws on the current device (looked up once).
pi_status static_ws(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PI_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return PI_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return PI_OK;
}

}  // namespace

extern "C" PI_API pi_status pi_ffn_layer_static(const pi_ffn_desc *desc, const float *x, const float *residual,
                                                float *y, int32_t *idx, int32_t *n_active, int32_t *status_out,
                                                pi_stream stream)
{
    if (!desc) return PI_ERR_NULL;
    if (desc->d_ff > kStaticMaxDff || desc->rank > PI_MAX_RANK) return PI_ERR_SHAPE;
    const pi::WsLayout L = pi::ws_layout(desc->d_model, desc->d_ff, desc->rank, 1);
    if (L.total > kStaticWsBytes) return PI_ERR_SHAPE;
    if (status_out && ((uintptr_t)status_out & 3)) return PI_ERR_ALIGN;
    void *ws = nullptr;
    pi_status st = static_ws(&ws);
    if (st != PI_OK) return st;
    const cudaStream_t s = (cudaStream_t)stream;
    // a fresh error word for this call; the scan state stays as the last call left it
    if (cudaMemsetAsync(ws, 0, sizeof(unsigned), s) != cudaSuccess) return PI_ERR_CUDA;
    st = pi_ffn_layer(desc, x, 1, residual, y, idx, n_active, ws, L.total, stream);
    if (st != PI_OK) return st;
    if (status_out &&
        cudaMemcpyAsync(status_out, ws, sizeof(unsigned), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return PI_ERR_CUDA;
    return PI_OK;
}
