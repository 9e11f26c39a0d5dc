// Internal host-side launch interface between the C ABI (api.cu) and the
// kernel translation units.  Not installed; the public contract is gdr.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdr {

struct RecurrentArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const void* beta;
    void* pool;
    const int32_t* state_indices;
    const int32_t* cu_seqlens;
    void* o;
    void* ibuf;
    int N, Hk, Hv, K, V, steps, num_slots;
    int64_t T;
    int dtype, pool_dtype, flags;
    float scale;
    // gates formed in the kernel from raw projections (gdr_recurrent_fwd_gated):
    // g = -exp(A_log) softplus(ga + dt_bias), beta = beta_mul sigmoid(gb);
    // ga == nullptr means g / beta are given
    const void* ga = nullptr;
    const void* gb = nullptr;
    const float* A_log = nullptr;
    const float* dt_bias = nullptr;
    float beta_mul = 1.f;
    // gated RMSNorm epilogue (gdr_recurrent_fwd_norm): o <- rmsnorm(o) * weight
    // * sigmoid(gate) per value row; norm_weight == nullptr means none
    const float* norm_weight = nullptr;
    const void* norm_gate = nullptr;
    float norm_eps = 0.f;
};

// Enqueue the recurrent decode / verify kernel.  Returns a cudaError_t.
cudaError_t launch_recurrent(const RecurrentArgs& a, cudaStream_t stream);

struct ChunkArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* gk;
    const void* beta;
    const float* initial_state;
    const int32_t* cu_seqlens;
    void* o;
    float* final_state;
    int N;
    int64_t T;
    int Hk, Hv, K, V, dtype, flags;
    float scale;
    void* workspace;
    size_t ws_bytes;
};

// Workspace layout of the chunked prefill (byte offsets, 256-aligned).
struct ChunkWorkspace {
    int64_t max_chunks;
    size_t off_meta;      // int: [0] = chunk count
    size_t off_offsets;   // int [N+1]: first global chunk of each sequence
    size_t off_table;     // int4 [max_chunks]: (seq, start token, length, -)
    size_t off_qn, off_kn;  // normalised q / k (GDR_QK_L2NORM), input dtype
    size_t off_w, off_u, off_kd, off_qd;   // fp32 [T, Hv, K|V]
    size_t off_p;         // fp32 [max_chunks, Hv, 64, 64]
    size_t off_dl;        // fp32 [max_chunks, Hv, K]
    size_t off_h;         // fp32 [max_chunks, Hv, V, K]
    size_t off_vn;        // fp32 [T, Hv, V]
    size_t off_order;     // int [N]: sequences by decreasing length
    size_t off_blobs;     // tensor-core path operand images
    bool tc;              // tensor-core path (bf16, K = V = 128 or 64)
    // tensor-core path, at most kLocalMetaSeqs sequences and no scan: the
    // metadata kernel is not launched; the prep kernel forms the metadata
    bool local_meta;
    // chunk-parallel scan (GDR_CHUNK_SCAN on the tensor-core path)
    int seg_chunks;       // segment length G in chunks; 0 = scan off
    int64_t max_segs;     // segment capacity: ceil(max_chunks / G) + N
    size_t off_segs;      // int4 [max_segs]: (seq, first chunk in seq, chunks, last?)
    size_t off_segoff;    // int [N+1]: first segment of each sequence
    size_t off_mt;        // fp32 [max_segs, Hv, K, K]: segment transition P
    size_t off_bs;        // fp32 [max_segs, Hv, V, K]: segment offset B, then start state
    size_t total;
};

// Segment length (chunks, >= 1) of the chunk-parallel scan for N sequences
// of T tokens in all and Hv value heads.
int chunk_scan_segment(int N, int64_t T, int Hv);

ChunkWorkspace chunk_workspace_layout(int N, int64_t T, int Hk, int Hv, int K, int V, int gate_kind,
                                      int dtype, int flags);

cudaError_t launch_chunk(const ChunkArgs& a, cudaStream_t stream);

// Calls with at most this many sequences (and no chunk-parallel scan) have
// their chunk metadata formed inside the tensor-core prep kernel.
constexpr int kLocalMetaSeqs = 64;

// Tensor-core chunked prefill (bf16, K = V = 128 or 64): blob bytes and launcher.
size_t chunk_tc_blob_bytes(int64_t max_chunks, int Hk, int Hv, bool channel_gate);
cudaError_t launch_chunk_tc(const ChunkArgs& a, const ChunkWorkspace& w, char* ws, const void* q, const void* k,
                            cudaStream_t stream);

struct GatingArgs {
    const void* a;
    const float* dt_bias;
    const float* A_log;
    const void* b;
    float* g;
    void* beta;
    int64_t T;
    int Hv, dtype, flags;
};

cudaError_t launch_gating(const GatingArgs& a, cudaStream_t stream);

// Record a formatted message for gdr_last_error() on this thread; returns code.
int set_last_error(int code, const char* fmt, ...);

// Device error word (set by bounded device waits that give up).
unsigned int* device_error_word();

// Launch `kernel` so that it may start while the previous kernel in `stream`
// is still running (programmatic dependent launch): the kernel must execute
// griddepcontrol.wait before it reads anything that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Scoped per-kernel timing (active only after gdr_profile_enable(1)): records
// an event on `s` at construction and at destruction, so declare it right
// before a launch inside its own block.
class KernelTimer {
  public:
    KernelTimer(const char* name, cudaStream_t s);
    ~KernelTimer();
    KernelTimer(const KernelTimer&) = delete;
    KernelTimer& operator=(const KernelTimer&) = delete;

  private:
    const char* name_;
    cudaStream_t stream_;
    void* a_;
};

}  // namespace gdr
