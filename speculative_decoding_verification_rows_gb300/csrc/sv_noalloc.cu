// sv_noalloc.cu -- sv_verify_chain_noalloc: the uniform-layout verify with its
// scratch in a static device array instead of a caller workspace.
//
// Some callers cannot allocate device memory at the point where they verify:
// code running while a CUDA graph is being captured (cudaMalloc is refused
// during a global-mode capture), serving runtimes that reserve all device
// memory in a pool at start-up and forbid allocations on the decode path
// (an allocation can stall the device and fragment the pool), and plugins
// embedded in a host engine that owns all memory and gives them none.  This
// entry point needs nothing from them but inputs and outputs.
//
// The array is fixed at kNoAllocScratchBytes (32 MiB) and stays resident on
// every GPU that loads this library until the process exits.  Each call
// rewrites every scratch word it later reads (its first kernel resets the
// counters), so leftovers of an earlier call do no harm -- but all calls
// share the one array, so calls whose work overlaps on the GPU (two streams,
// or two host threads) race and must be serialised by the caller.
#include <atomic>

#include <cuda_runtime.h>

#include "sv.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 128;
// Device address of the array, per device.  Host threads making their first
// calls at the same time may both look it up; they store the same address,
// and the atomic makes the store and the loads well defined.
std::atomic<void*> g_scratch_addr[kMaxDevices];

}  // namespace

extern "C" sv_status_t sv_verify_chain_noalloc(const void* target_logits, const void* draft_logits, sv_dtype_t dt,
                                               int n_req, int K, int vocab, const int32_t* draft_tokens,
                                               const int32_t* verify_len, sv_sampling_t sp, uint64_t seed,
                                               int32_t* accept_len, int32_t* out_tokens, int32_t* num_emitted,
                                               int32_t* row_status, sv_stream_t stream)
{
    const size_t need = sv_workspace_size(n_req, K, vocab);
    if (need > kNoAllocScratchBytes) return SV_ERR_UNSUPPORTED;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
    void* scratch = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (scratch == nullptr) {
        // The array's name is a host-side stand-in; the device address comes
        // from the runtime, once per device, with that device current.
        if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess || scratch == nullptr)
            return SV_ERR_CUDA;
        g_scratch_addr[dev].store(scratch, std::memory_order_release);
    }
    return sv_verify_chain(target_logits, draft_logits, dt, n_req, K, vocab, draft_tokens, verify_len, sp, seed,
                           accept_len, out_tokens, num_emitted, row_status, scratch, kNoAllocScratchBytes, stream);
}
