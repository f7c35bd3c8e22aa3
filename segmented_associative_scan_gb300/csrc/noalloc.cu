// GAE with a built-in look-back workspace, for callers that cannot allocate device
// memory: for example a plugin that a host framework hands only its input and output
// buffers (the framework plans every byte of device memory up front), or a training
// loop running under a fixed memory budget where a cudaMalloc could fail or stall the
// device. The caller still owns the inputs and outputs; the library owns one static
// array, defined below, that every GPU loading the library holds until the process
// exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/rlca.h"
#include "launch.cuh"

namespace {

// Fixed scratch: a 256-byte look-back header plus 32 bytes per tile, for at most
// RLCA_NOALLOC_MAX_TILES tiles (1 MiB + 256 bytes).
constexpr size_t kScratchBytes =
    (size_t)rlca::kWsHeaderBytes + (size_t)RLCA_NOALLOC_MAX_TILES * rlca::kTileStateBytes;
static __device__ __align__(256) unsigned char g_gae_scratch[kScratchBytes];

// Host-side device addresses of g_gae_scratch, one per device, as last set up.
std::mutex g_setup_mutex;
void *g_scratch_addr[rlca::kMaxDevices] = {};

// Address of the scratch on the current device. Host code only holds a stand-in for the
// symbol, so its device address is looked up with the device current, on every call
// (cheap): after cudaDeviceReset the module is loaded again and the array may move.
// Whenever the address is new (first use on this device, or the array moved), the whole
// array is zeroed, synchronously, before it is used.
void *scratch_on_current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= rlca::kMaxDevices) {
        (void)cudaGetLastError();
        return nullptr;
    }
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_gae_scratch) != cudaSuccess || !ptr) {
        (void)cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_addr[dev] != ptr) {
        if (cudaMemset(ptr, 0, kScratchBytes) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        g_scratch_addr[dev] = ptr;
    }
    return ptr;
}

// Runs after every argument check, right before the look-back launch, on its stream.
// The array keeps the previous call's contents. Tile states carry a launch epoch and
// need no clearing; the tile and finish counters and the timeout record must start at
// zero, so clear them (bytes 4..15 of the header; the epoch at byte 0 stays).
cudaError_t clear_header(void *scratch, cudaStream_t stream)
{
    return cudaMemsetAsync(static_cast<unsigned char *>(scratch) + 4, 0, 12, stream);
}

}  // namespace

extern "C" int rlca_gae_noalloc(const float *reward, const float *value,
                                const uint8_t *terminated, const uint8_t *truncated,
                                const float *trunc_value, const float *bootstrap, float gamma,
                                float lambda, int64_t N, int64_t T, int64_t ld,
                                float *advantages, float *returns, void *stream)
{
    // Rows that fit one tile, rows numerous enough to fill the GPU one CTA per row, and
    // every malformed shape go to rlca_gae unchanged: its path uses no workspace, and it
    // returns its own error codes.
    if (N <= 0 || T <= rlca::kTile || T > RLCA_MAX_T || ld < T || !rlca::lookback_pays(N))
        return rlca_gae(reward, value, terminated, truncated, trunc_value, bootstrap, gamma,
                        lambda, N, T, ld, advantages, returns, stream);
    // Look-back path: rlca_gae_ex's checks against a workspace of the array's size (more
    // than RLCA_NOALLOC_MAX_TILES tiles: RLCA_ERR_WORKSPACE), then the header cleared on
    // the stream and the launch. A call that fails a check enqueues nothing.
    void *scratch = scratch_on_current_device();
    if (!scratch) return RLCA_ERR_LAUNCH;
    return rlca::gae_on_library_workspace(reward, value, terminated, truncated, trunc_value,
                                          bootstrap, gamma, lambda, N, T, ld, advantages,
                                          returns, scratch, kScratchBytes, clear_header,
                                          stream);
}
