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
#include "kernels.cuh"

namespace {

// Fixed scratch: a 256-byte look-back header plus 32 bytes per tile, for at most
// RLCA_NOALLOC_MAX_TILES tiles (1 MiB + 256 bytes). Zero at module load.
constexpr size_t kScratchBytes =
    (size_t)rlca::kWsHeaderBytes + (size_t)RLCA_NOALLOC_MAX_TILES * rlca::kTileStateBytes;
static __device__ __align__(256) unsigned char g_gae_scratch[kScratchBytes];

// Host-side device addresses of g_gae_scratch, one per device, found at set-up.
constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Address of the scratch on the current device, setting it up on first use: the symbol's
// device address is looked up with that device current and the array is zeroed once.
void *scratch_on_current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_gae_scratch) != cudaSuccess || !ptr) return nullptr;
        if (cudaMemset(ptr, 0, kScratchBytes) != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = ptr;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" int rlca_gae_noalloc(const float *reward, const float *value,
                                const uint8_t *terminated, const uint8_t *truncated,
                                const float *trunc_value, const float *bootstrap, float gamma,
                                float lambda, int64_t N, int64_t T, int64_t ld,
                                float *advantages, float *returns, void *stream)
{
    const size_t need = rlca_workspace_bytes(N, T);
    if (need > kScratchBytes) return RLCA_ERR_WORKSPACE;  // more than RLCA_NOALLOC_MAX_TILES
    if (need == 0)  // rows fit one tile: no scratch involved
        return rlca_gae(reward, value, terminated, truncated, trunc_value, bootstrap, gamma,
                        lambda, N, T, ld, advantages, returns, stream);
    void *scratch = scratch_on_current_device();
    if (!scratch) return RLCA_ERR_LAUNCH;
    // The array keeps the previous call's contents. Tile states carry a launch epoch and
    // need no clearing; the tile and finish counters and the timeout record must start
    // at zero, so clear them (bytes 4..15 of the header; the epoch at byte 0 stays).
    if (cudaMemsetAsync(static_cast<unsigned char *>(scratch) + 4, 0, 12,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return RLCA_ERR_LAUNCH;
    return rlca_gae_ex(reward, value, terminated, truncated, trunc_value, bootstrap, gamma,
                       lambda, N, T, ld, advantages, returns, scratch, kScratchBytes, stream);
}
