// kda_chunk_fwd_noalloc: the forward pass for callers that cannot allocate
// device memory. Some callers cannot call cudaMalloc (or a caching allocator
// on top of it): code that runs inside an allocator's own hooks, processes
// whose device memory is entirely reserved up front by an arena they do not
// control, or latency-critical paths where an allocation's implicit device
// synchronisation is not acceptable. This variant takes its workspace from a
// fixed, library-owned device array instead of from the caller.
//
// The array is a file-scope __device__ object, so every GPU that loads the
// library holds it until the process exits. Host code may not use the array's
// name as a pointer (on the host it is only a stand-in for the symbol): the
// device address is looked up once per device with cudaGetSymbolAddress, with
// that device current, on the first call made on it.
#include <atomic>
#include <string>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// The scratch's device address on the current device (looked up on the first call made there).
kda_status scratch_address(void** ws) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        kda::set_last_error((std::string("cudaGetDevice: ") + cudaGetErrorString(e)).c_str());
        return KDA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        kda::set_last_error("device index beyond the no-allocation table");
        return KDA_ERR_UNSUPPORTED;
    }
    *ws = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!*ws) {
        e = cudaGetSymbolAddress(ws, g_noalloc_scratch);
        if (e != cudaSuccess || !*ws) {
            kda::set_last_error((std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e)).c_str());
            return KDA_ERR_CUDA;
        }
        g_scratch_addr[dev].store(*ws, std::memory_order_release);
    }
    return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_noalloc_device_status(const kda_problem* p, kda_stream_t stream, int32_t* word) {
    void* ws = nullptr;
    const kda_status st = scratch_address(&ws);
    if (st != KDA_OK) return st;
    return kda_device_status(p, ws, (size_t)KDA_NOALLOC_SCRATCH_BYTES, stream, word);
}

extern "C" kda_status kda_chunk_fwd_noalloc(const kda_problem* p, void* o, float* ht,
                                             kda_stream_t stream) {
    if (!p) {
        kda::set_last_error("problem is NULL");
        return KDA_ERR_INVALID_ARG;
    }
    if (p->save_policy != 0) {
        kda::set_last_error("the no-allocation forward has no saved buffer: use save_policy 0");
        return KDA_ERR_INVALID_ARG;
    }
    const size_t need = kda_workspace_size(p, 0);
    if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) {
        kda::set_last_error(("forward workspace of " + std::to_string(need) +
                             " bytes exceeds the no-allocation scratch of " +
                             std::to_string((size_t)KDA_NOALLOC_SCRATCH_BYTES) + " bytes")
                                .c_str());
        return KDA_ERR_WORKSPACE;
    }
    void* ws = nullptr;
    const kda_status st = scratch_address(&ws);
    if (st != KDA_OK) return st;
    // Nothing in the scratch must start at zero: the forward writes every word
    // it reads (chunk table, then the chunk intermediates) within the call.
    return kda_chunk_fwd(p, o, ht, nullptr, ws, (size_t)KDA_NOALLOC_SCRATCH_BYTES, stream);
}
