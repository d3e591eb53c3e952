// noalloc.cu -- csa2_index_score_noalloc: the indexer entry point for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or ask a caching allocator for a buffer) at the
// point where they score: an inference server that carves all device memory into fixed
// pools at start-up and forbids later allocations, a plug-in running inside a framework
// that owns the device allocator, or a real-time decode loop that must not take the
// allocator's locks or risk an out-of-memory error mid-step.  This entry point needs no
// workspace argument: its scratch (the indexer's per-row tile counters) lives in a
// file-scope __device__ array that every GPU loading the library holds until the process
// exits.  It calls no cudaMalloc, cudaFree or allocating library routine; it clears the
// counters it uses with cudaMemsetAsync on the caller's stream in each call, so a call
// that timed out cannot leave stale counts behind.
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

#include "../../include/csa2.h"

namespace {

// 65,536 words (256 KB): two counters per query row of the tensor-core indexer, so
// requests of up to 32,768 query rows fit.
constexpr size_t kScratchWords = 65536;
static __device__ __align__(256) uint32_t g_index_scratch[kScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];
bool g_scratch_ready[kMaxDevices];

// Device address of the scratch array on the current device.  The host-side name of a
// __device__ array is only a stand-in, so the address is looked up once per device, with
// that device current, and cached.
csa2_status scratch_for_current_device(void **ptr)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CSA2_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return CSA2_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ready[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_index_scratch) != cudaSuccess || p == nullptr)
            return CSA2_ERR_CUDA;
        g_scratch_ptr[dev] = p;
        g_scratch_ready[dev] = true;
    }
    *ptr = g_scratch_ptr[dev];
    return CSA2_OK;
}

} // namespace

extern "C" {

csa2_status csa2_index_score_noalloc(const csa2_index_args *a, float *scores, int32_t *row_len,
                                     uint32_t *d_status, csa2_stream stream)
{
    const size_t need = csa2_index_score_workspace_size(a);
    if (need > kScratchWords * sizeof(uint32_t)) return CSA2_ERR_WORKSPACE;
    void *ws = nullptr;
    if (need) {
        const csa2_status st = scratch_for_current_device(&ws);
        if (st != CSA2_OK) return st;
    }
    if (need && cudaMemsetAsync(ws, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return CSA2_ERR_CUDA;        // counters start from zero whatever an earlier call left
    return csa2_index_score(a, scores, row_len, ws, need, d_status, stream);
}

} // extern "C"
