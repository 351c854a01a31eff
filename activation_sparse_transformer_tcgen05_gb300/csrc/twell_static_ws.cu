// twell_static_ws.cu — the forward pass for callers that cannot allocate
// device memory.
//
// twell_ffn_fwd needs a caller-provided workspace. Some callers have no way to
// provide one: a host framework that owns all device memory and gives plugins
// no allocator, or a latency-critical decode loop where a cudaMalloc/cudaFree
// would synchronise the device and stall every other stream. For them the
// library keeps one file-scope device array of TWELL_STATIC_WS_BYTES and runs
// the unchanged twell_ffn_fwd on it. Nothing is allocated, at set-up or later.
//
// The array is a __device__ symbol. In host code its name is only a host-side
// stand-in, not a device address (a kernel handed it would fault, or on
// systems where the GPU can read host memory silently use the wrong memory).
// The device address is therefore looked up with cudaGetSymbolAddress, once
// per device, with that device current, on the first call made on it. The
// cached address belongs to the device's current context: after a
// cudaDeviceReset the module may load at another address, so a process that
// resets a device must not call this entry point on it again.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/twell.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[TWELL_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_ws_ptr[kMaxDevices] = {nullptr};

// Device address of g_static_ws on the current device (set up on first use).
twell_status static_ws_address(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();  // leave no pending error for the next, unrelated call
        return TWELL_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_ws_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) {
            (void)cudaGetLastError();
            return TWELL_ERR_CUDA;
        }
        g_ws_ptr[dev] = p;
    }
    *out = g_ws_ptr[dev];
    return TWELL_OK;
}

}  // namespace

extern "C" twell_status twell_ffn_fwd_static_ws(const uint16_t* x, const uint16_t* W_up, const uint16_t* W_gate,
                                                const float* b, const uint16_t* W_down, int M, int d, int F, int T,
                                                const twell_buf* h_out, uint16_t* y, int32_t* status, void* stream)
{
    if (!h_out || M <= 0 || d <= 0 || F <= 0 || T <= 0) return TWELL_ERR_INVALID_ARG;
    // The smallest workspace the forward accepts: the gated layout, or the ReLU
    // layout at its smallest staging capacity (32 entries per row and 256-column
    // block). twell_ffn_fwd then takes the largest staging the array holds.
    const size_t need = W_gate ? twell_workspace_bytes(TWELL_OP_GATED_FWD, M, d, F, T, h_out->cap_slots)
                               : twell_fwd_workspace_bytes(M, d, F, T, h_out->cap_slots, 32);
    if (need == 0) return TWELL_ERR_INVALID_ARG;
    if (need > (size_t)TWELL_STATIC_WS_BYTES) return TWELL_ERR_WORKSPACE;  // problem too large for the array
    void* ws = nullptr;
    const twell_status st = static_ws_address(&ws);
    if (st != TWELL_OK) return st;
    // Every byte the forward reads from its workspace it has written earlier in
    // the same call, so the array needs no clearing between calls.
    return twell_ffn_fwd(x, W_up, W_gate, b, W_down, M, d, F, T, h_out, y, ws, (size_t)TWELL_STATIC_WS_BYTES,
                         status, stream);
}
