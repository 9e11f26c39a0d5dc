// gdr_chunk_fwd_noalloc: the chunked prefill for callers that cannot allocate
// device memory themselves.
//
// Some callers have no way to obtain a workspace: code that runs while a
// serving engine has already handed all device memory to its own arena and
// forbids further cudaMalloc calls, plugin hosts that expose no allocator to
// the plugin, or latency-critical loops where cudaMalloc's implicit device
// synchronisation is not acceptable.  This entry point takes the same inputs
// and outputs as gdr_chunk_fwd but uses a fixed scratch array compiled into
// the library instead of a caller-provided workspace.
//
// The scratch array is a file-scope __device__ array of kStaticWorkspaceBytes.
// Every GPU that loads this library holds it until the process exits.  In host
// code its name is only a host-side stand-in, so its device address is looked
// up with cudaGetSymbolAddress on every call, in the context current on the
// calling thread.  The address belongs to that context, not to the device
// index: after cudaDeviceReset, or with another context current on the same
// device, the array lives at a new address, and a cached pointer would send
// the kernels to memory that is no longer mapped.  The lookup is a host-side
// table read once the library's device code is loaded in the context.
#include <cstdio>

#include "gdr.h"
#include "launch.h"

namespace gdr {
namespace {

constexpr size_t kStaticWorkspaceBytes = (size_t)GDR_NOALLOC_WORKSPACE_BYTES;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

// Device address of the scratch array in the current context.
int static_workspace(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess || p == nullptr)
        return set_last_error(GDR_ERR_LAUNCH, "cudaGetSymbolAddress of the static workspace failed: %s",
                              cudaGetErrorString(e));
    *out = p;
    return GDR_OK;
}

}  // namespace
}  // namespace gdr

extern "C" int gdr_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                     const float* gk, const void* beta, const float* initial_state,
                                     const int32_t* cu_seqlens, int N, int64_t T_total, int Hk, int Hv,
                                     int K, int V, float scale, int dtype, int flags, void* o,
                                     float* final_state, gdr_stream_t stream) {
    size_t need = 0;
    const int gate_kind = g ? GDR_GATE_SCALAR : GDR_GATE_CHANNEL;
    if (int rc = gdr_chunk_workspace_size(N, T_total, Hk, Hv, K, V, gate_kind, dtype, flags, &need)) return rc;
    if (need > gdr::kStaticWorkspaceBytes)
        return gdr::set_last_error(GDR_ERR_WORKSPACE,
                                   "gdr_chunk_fwd_noalloc: this problem needs %zu bytes of scratch but the "
                                   "library's static scratch holds %zu; use gdr_chunk_fwd with a workspace",
                                   need, gdr::kStaticWorkspaceBytes);
    void* ws = nullptr;
    if (N > 0 && T_total > 0)
        if (int rc = gdr::static_workspace(&ws)) return rc;
    return gdr_chunk_fwd(q, k, v, g, gk, beta, initial_state, cu_seqlens, N, T_total, Hk, Hv, K, V, scale,
                         dtype, flags, o, final_state, ws, gdr::kStaticWorkspaceBytes, stream);
}
