// cpa_no_alloc.cu -- chunked_prefill_attention_no_alloc: the attention call
// for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc and have no spare device buffer to lend
// as workspace: a plugin running inside a host application that owns every
// byte of device memory through its own pool, or a serving loop that must not
// call cudaMalloc / cudaFree on its hot path because those calls can
// synchronise the device and stall the other streams.  For them the split-KV
// partials live in one file-scope __device__ array of fixed size instead of a
// caller-provided workspace.  This call allocates nothing: no cudaMalloc, no
// cudaFree, no allocating library routine.
//
// Costs and rules of the static array:
//   * every GPU that loads this library holds CPA_NO_ALLOC_WORKSPACE_BYTES of
//     device memory for it until the process exits;
//   * a batch whose split-KV partials need more than that is rejected with
//     CPA_ERR_WORKSPACE, before anything is launched;
//   * every call on a device shares the one array and it keeps the last
//     call's contents; nothing in it needs to start at zero (each launch
//     writes every partial before it reads it);
//   * calls that overlap on the GPU (for example on two streams at once)
//     race on the array and may give wrong results: serialise them;
//   * the first call on a device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and caches it; make
//     that first call before any stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/cpa.h"

namespace {

constexpr int kMaxDevices = 64;

// The scratch memory itself.  In host code this name is only a host-side
// handle, never a device address: kernels get the address looked up below.
static __device__ __align__(256) unsigned char g_no_alloc_ws[CPA_NO_ALLOC_WORKSPACE_BYTES];

std::mutex g_no_alloc_mutex;
void *g_no_alloc_ptr[kMaxDevices] = {};

// Device address of g_no_alloc_ws on the current device (looked up once per
// device), or nullptr on failure.
void *no_alloc_workspace() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_no_alloc_mutex);
    if (!g_no_alloc_ptr[dev]) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_no_alloc_ws);
        if (e != cudaSuccess || ptr == nullptr) return nullptr;
        g_no_alloc_ptr[dev] = ptr;
    }
    return g_no_alloc_ptr[dev];
}

}  // namespace

extern "C" cpa_status chunked_prefill_attention_no_alloc(const cpa_batch *batch, const cpa_params *params,
                                                         const void *q, const void *k_new, const void *v_new,
                                                         void *k_cache, void *v_cache, void *out, float *lse,
                                                         void *stream) {
    // 0 for an invalid batch too: chunked_prefill_attention reports that error
    cpa_params p = params ? *params : cpa_params{};
    size_t need = params ? chunked_prefill_workspace_size(batch, &p) : 0;
    if (need > (size_t)CPA_NO_ALLOC_WORKSPACE_BYTES) {
        // without tail pieces, whose partials are an optimisation
        p.flags &= ~CPA_FLAG_TAIL_SPLIT;
        need = chunked_prefill_workspace_size(batch, &p);
    }
    if (need > (size_t)CPA_NO_ALLOC_WORKSPACE_BYTES) return CPA_ERR_WORKSPACE;
    void *ws = no_alloc_workspace();
    if (ws == nullptr) return CPA_ERR_CUDA;
    return chunked_prefill_attention(batch, params ? &p : nullptr, q, k_new, v_new, k_cache, v_cache, out, lse, ws,
                                     (size_t)CPA_NO_ALLOC_WORKSPACE_BYTES, stream);
}
