// C ABI of libgdr.so: argument checks, workspace sizing, launch sequencing on
// the caller's stream, error reporting.  The contract is documented in
// include/gdr.h.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "common.cuh"
#include "gdr.h"
#include "launch.h"

namespace gdr {

static __device__ unsigned int g_error_word;     // bounded device waits that gave up
static __device__ unsigned int g_validate_word;  // GDR_VALIDATE findings

unsigned int* device_error_word() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    return static_cast<unsigned int*>(p);
}

namespace {

thread_local char t_last_error[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
    return code;
}

int ok() {
    t_last_error[0] = '\0';
    return GDR_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The kernels are built for sm_103a only.
int check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(GDR_ERR_LAUNCH, "cudaGetDevice failed");
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
        return fail(GDR_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only",
                    dev, major, minor);
    return GDR_OK;
}

int launch_status(cudaError_t e, const char* what) {
    if (e != cudaSuccess) return fail(GDR_ERR_LAUNCH, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

// ---- GDR_VALIDATE: device-side content checks (synchronising) -------------
enum : unsigned {
    V_CU_BAD = 1u,        // cu[0] != 0, decreasing, or cu[N] != T
    V_EMPTY_SEQ = 2u,     // empty sequence where not allowed
    V_GATE_BAD = 4u,      // gate not finite or > 0
    V_SLOT_RANGE = 8u,    // slot >= num_slots
    V_SLOT_DUP = 16u,     // a valid slot used twice
    V_STEPS = 32u,        // L_b > steps with intermediate states
};

__global__ void validate_kernel(const int32_t* cu, int N, int64_t T, int allow_empty,
                                const float* gate, int64_t gate_n, const int32_t* idx,
                                int num_slots, int steps) {
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nth = (int64_t)gridDim.x * blockDim.x;
    unsigned bad = 0;
    for (int64_t b = tid; b < N; b += nth) {
        const int lo = cu[b], hi = cu[b + 1];
        if (hi < lo) bad |= V_CU_BAD;
        if (!allow_empty && hi == lo) bad |= V_EMPTY_SEQ;
        if (idx) {
            const int s = idx[b];
            if (s >= num_slots) bad |= V_SLOT_RANGE;
            if (s >= 0 && steps > 0 && hi - lo > steps) bad |= V_STEPS;
            if (s >= 0)
                for (int j = 0; j < b; ++j)
                    if (idx[j] == s) bad |= V_SLOT_DUP;
        }
    }
    if (tid == 0 && (cu[0] != 0 || cu[N] != T)) bad |= V_CU_BAD;
    for (int64_t i = tid; i < gate_n; i += nth) {
        const float x = gate[i];
        if (!(x <= 0.f) || isinf(x)) bad |= V_GATE_BAD;
    }
    if (bad) atomicOr(&g_validate_word, bad);
}

int run_validation(cudaStream_t stream, const int32_t* cu, int N, int64_t T, bool allow_empty,
                   const float* gate, int64_t gate_n, const int32_t* idx, int num_slots, int steps) {
    void* wp = nullptr;
    if (cudaGetSymbolAddress(&wp, g_validate_word) != cudaSuccess)
        return fail(GDR_ERR_LAUNCH, "validation word unavailable");
    cudaMemsetAsync(wp, 0, sizeof(unsigned), stream);
    validate_kernel<<<304, 256, 0, stream>>>(cu, N, T, allow_empty ? 1 : 0, gate, gate_n, idx,
                                             num_slots, steps);
    unsigned word = 0;
    cudaMemcpyAsync(&word, wp, sizeof(unsigned), cudaMemcpyDeviceToHost, stream);
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(GDR_ERR_LAUNCH, "validation: %s", cudaGetErrorString(e));
    if (word)
        return fail(GDR_ERR_VALIDATION,
                    "input validation failed (0x%x):%s%s%s%s%s%s", word,
                    (word & V_CU_BAD) ? " cu_seqlens malformed;" : "",
                    (word & V_EMPTY_SEQ) ? " empty sequence;" : "",
                    (word & V_GATE_BAD) ? " gate not finite or > 0;" : "",
                    (word & V_SLOT_RANGE) ? " state index >= num_slots;" : "",
                    (word & V_SLOT_DUP) ? " duplicate state index;" : "",
                    (word & V_STEPS) ? " sequence longer than steps;" : "");
    return GDR_OK;
}

int check_common(int N, int64_t T, int Hk, int Hv, int K, int V, int dtype) {
    if (N < 0 || T < 0) return fail(GDR_ERR_INVALID_ARG, "negative N (%d) or T_total (%lld)", N, (long long)T);
    if (Hk <= 0 || Hv <= 0 || Hv % Hk != 0)
        return fail(GDR_ERR_INVALID_ARG, "Hv (%d) must be a positive multiple of Hk (%d)", Hv, Hk);
    if (Hv > 65535) return fail(GDR_ERR_UNSUPPORTED, "Hv (%d) above 65535", Hv);
    if (dtype != GDR_BF16 && dtype != GDR_F32) return fail(GDR_ERR_UNSUPPORTED, "dtype %d", dtype);
    if (K != V || (K != 64 && K != 128))
        return fail(GDR_ERR_UNSUPPORTED, "K (%d) and V (%d) must be equal and 64 or 128", K, V);
    return GDR_OK;
}

}  // namespace

int set_last_error(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
    return code;
}

}  // namespace gdr

using namespace gdr;

extern "C" {

int gdr_version(void) { return 100; }

const char* gdr_last_error(void) { return t_last_error; }

int gdr_chunk_workspace_size(int N, int64_t T_total, int Hk, int Hv, int K, int V, int gate_kind,
                             int dtype, int flags, size_t* bytes) {
    if (!bytes) return fail(GDR_ERR_INVALID_ARG, "bytes is NULL");
    if (int rc = check_common(N, T_total, Hk, Hv, K, V, dtype)) return rc;
    if (gate_kind != GDR_GATE_SCALAR && gate_kind != GDR_GATE_CHANNEL)
        return fail(GDR_ERR_INVALID_ARG, "gate_kind %d", gate_kind);
    *bytes = chunk_workspace_layout(N, T_total, Hk, Hv, K, V, gate_kind, dtype, flags).total;
    return ok();
}

int gdr_chunk_fwd(const void* q, const void* k, const void* v, const float* g, const float* gk,
                  const void* beta, const float* initial_state, const int32_t* cu_seqlens, int N,
                  int64_t T_total, int Hk, int Hv, int K, int V, float scale, int dtype, int flags,
                  void* o, float* final_state, void* workspace, size_t ws_bytes,
                  gdr_stream_t stream) {
    if (int rc = check_common(N, T_total, Hk, Hv, K, V, dtype)) return rc;
    if (flags & ~(GDR_QK_L2NORM | GDR_VALIDATE | GDR_CHUNK_SCAN))
        return fail(GDR_ERR_INVALID_ARG, "unsupported flags 0x%x for gdr_chunk_fwd", flags);
    if ((g == nullptr) == (gk == nullptr))
        return fail(GDR_ERR_INVALID_ARG, "exactly one of g / gk must be given");
    if (T_total > 0 && N == 0) return fail(GDR_ERR_INVALID_ARG, "T_total > 0 with N == 0");
    if (N == 0 || T_total == 0) {
        if (N > 0 && final_state) {
            // no tokens: the final state is the initial state (or zeros)
            cudaError_t e = initial_state
                ? cudaMemcpyAsync(final_state, initial_state, sizeof(float) * (size_t)N * Hv * V * K,
                                  cudaMemcpyDeviceToDevice, (cudaStream_t)stream)
                : cudaMemsetAsync(final_state, 0, sizeof(float) * (size_t)N * Hv * V * K,
                                  (cudaStream_t)stream);
            return launch_status(e, "empty prefill");
        }
        return ok();
    }
    if (!q || !k || !v || !beta || !cu_seqlens || !o || !workspace)
        return fail(GDR_ERR_INVALID_ARG, "null pointer argument");
    const void* ptrs[] = {q, k, v, g, gk, beta, initial_state, o, final_state};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(GDR_ERR_INVALID_ARG, "pointer %p not 16-byte aligned", p);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(GDR_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    const ChunkWorkspace w = chunk_workspace_layout(N, T_total, Hk, Hv, K, V, g ? 0 : 1, dtype, flags);
    if (w.tc && N > 65535) return fail(GDR_ERR_UNSUPPORTED, "N (%d) above 65535 sequences per call", N);
    if (w.seg_chunks > 0 && w.max_segs > 65535)
        return fail(GDR_ERR_UNSUPPORTED, "GDR_CHUNK_SCAN: segment capacity %lld above 65535", (long long)w.max_segs);
    if (ws_bytes < w.total)
        return fail(GDR_ERR_WORKSPACE, "workspace %zu bytes < required %zu", ws_bytes, w.total);
    if (w.max_chunks > 0x7fffffffLL) return fail(GDR_ERR_UNSUPPORTED, "too many chunks");
    if (int rc = check_device()) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    if (flags & GDR_VALIDATE) {
        const float* gate = g ? g : gk;
        const int64_t gate_n = T_total * Hv * (g ? 1 : K);
        if (int rc = run_validation(s, cu_seqlens, N, T_total, false, gate, gate_n, nullptr, 0, 0))
            return rc;
    }
    ChunkArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.gk = gk; a.beta = beta;
    a.initial_state = initial_state; a.cu_seqlens = cu_seqlens; a.o = o; a.final_state = final_state;
    a.N = N; a.T = T_total; a.Hk = Hk; a.Hv = Hv; a.K = K; a.V = V; a.dtype = dtype;
    a.flags = flags & ~GDR_VALIDATE; a.scale = scale; a.workspace = workspace; a.ws_bytes = ws_bytes;
    return launch_status(launch_chunk(a, s), "gdr_chunk_fwd launch");
}

// Shared by gdr_recurrent_fwd and gdr_recurrent_fwd_gated: `rg` carries the
// raw gate projections of the fused variant (g and beta are then null).
struct RawGates {
    const void* a;
    const void* b;
    const float* A_log;
    const float* dt_bias;
};

struct OutNorm {
    const float* weight;
    const void* gate;
    float eps;
};

static int recurrent_impl(const void* q, const void* k, const void* v, const float* g, const void* beta,
                          const RawGates* rg, const OutNorm* on, void* state_pool, int pool_dtype, int num_slots,
                          const int32_t* state_indices, const int32_t* cu_seqlens, int N, int64_t T_total, int Hk,
                          int Hv, int K, int V, float scale, int dtype, int flags, void* o, void* intermediate_states,
                          int steps, gdr_stream_t stream, const char* who) {
    if (int rc = check_common(N, T_total, Hk, Hv, K, V, dtype)) return rc;
    if (pool_dtype != GDR_BF16 && pool_dtype != GDR_F32)
        return fail(GDR_ERR_UNSUPPORTED, "pool_dtype %d", pool_dtype);
    const int allowed = rg ? (GDR_QK_L2NORM | GDR_COMMIT | GDR_VALIDATE | GDR_NEG_EIGVAL)
                           : (GDR_QK_L2NORM | GDR_COMMIT | GDR_VALIDATE | GDR_CHANNEL_GATE);
    if (flags & ~allowed) return fail(GDR_ERR_INVALID_ARG, "unsupported flags 0x%x for %s", flags, who);
    if (N == 0) return ok();
    if (num_slots <= 0) return fail(GDR_ERR_INVALID_ARG, "num_slots must be positive");
    if (intermediate_states && steps <= 0)
        return fail(GDR_ERR_INVALID_ARG, "steps must be positive with intermediate_states");
    if (!state_pool || !state_indices || !cu_seqlens)
        return fail(GDR_ERR_INVALID_ARG, "null pointer argument");
    if (T_total > 0 && (!q || !k || !v || !o)) return fail(GDR_ERR_INVALID_ARG, "null pointer argument");
    if (T_total > 0 && !rg && (!g || !beta)) return fail(GDR_ERR_INVALID_ARG, "null pointer argument");
    if (rg && (!rg->A_log || !rg->dt_bias || (T_total > 0 && (!rg->a || !rg->b))))
        return fail(GDR_ERR_INVALID_ARG, "null pointer argument");
    if (on && (!on->weight || (T_total > 0 && !on->gate))) return fail(GDR_ERR_INVALID_ARG, "null pointer argument");
    if (on && !(on->eps >= 0.f)) return fail(GDR_ERR_INVALID_ARG, "eps must be >= 0");
    const void* ptrs[] = {q, k, v, g, beta, state_pool, o, intermediate_states};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(GDR_ERR_INVALID_ARG, "pointer %p not 16-byte aligned", p);
    if (N > 0x7fffffff / 2) return fail(GDR_ERR_UNSUPPORTED, "N too large");
    if (int rc = check_device()) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    if (flags & GDR_VALIDATE) {
        // formed gates are <= 0 and finite for finite projections: only the given ones are checked
        const int64_t gate_n = rg ? 0 : T_total * Hv * ((flags & GDR_CHANNEL_GATE) ? K : 1);
        if (int rc = run_validation(s, cu_seqlens, N, T_total, true, g, gate_n, state_indices,
                                    num_slots, intermediate_states ? steps : 0))
            return rc;
    }
    if (T_total == 0) return ok();  // nothing to compute; a commit would rewrite the same bits
    RecurrentArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.pool = state_pool;
    a.state_indices = state_indices; a.cu_seqlens = cu_seqlens; a.o = o; a.ibuf = intermediate_states;
    a.N = N; a.Hk = Hk; a.Hv = Hv; a.K = K; a.V = V; a.steps = intermediate_states ? steps : 0;
    a.num_slots = num_slots;
    a.T = T_total;
    a.dtype = dtype; a.pool_dtype = pool_dtype; a.flags = flags & ~(GDR_VALIDATE | GDR_NEG_EIGVAL); a.scale = scale;
    if (rg) {
        a.ga = rg->a; a.gb = rg->b; a.A_log = rg->A_log; a.dt_bias = rg->dt_bias;
        a.beta_mul = (flags & GDR_NEG_EIGVAL) ? 2.f : 1.f;
    }
    if (on) {
        a.norm_weight = on->weight; a.norm_gate = on->gate; a.norm_eps = on->eps;
    }
    return launch_status(launch_recurrent(a, s), who);
}

int gdr_recurrent_fwd(const void* q, const void* k, const void* v, const float* g, const void* beta,
                      void* state_pool, int pool_dtype, int num_slots, const int32_t* state_indices,
                      const int32_t* cu_seqlens, int N, int64_t T_total, int Hk, int Hv, int K, int V,
                      float scale, int dtype, int flags, void* o, void* intermediate_states, int steps,
                      gdr_stream_t stream) {
    return recurrent_impl(q, k, v, g, beta, nullptr, nullptr, state_pool, pool_dtype, num_slots, state_indices,
                          cu_seqlens, N, T_total, Hk, Hv, K, V, scale, dtype, flags, o, intermediate_states, steps,
                          stream, "gdr_recurrent_fwd");
}

int gdr_recurrent_fwd_norm(const void* q, const void* k, const void* v, const float* g, const void* beta,
                           void* state_pool, int pool_dtype, int num_slots, const int32_t* state_indices,
                           const int32_t* cu_seqlens, int N, int64_t T_total, int Hk, int Hv, int K, int V,
                           float scale, int dtype, int flags, const float* norm_weight, const void* norm_gate,
                           float eps, void* o, void* intermediate_states, int steps, gdr_stream_t stream) {
    const OutNorm on{norm_weight, norm_gate, eps};
    return recurrent_impl(q, k, v, g, beta, nullptr, &on, state_pool, pool_dtype, num_slots, state_indices,
                          cu_seqlens, N, T_total, Hk, Hv, K, V, scale, dtype, flags, o, intermediate_states, steps,
                          stream, "gdr_recurrent_fwd_norm");
}

int gdr_recurrent_fwd_gated(const void* q, const void* k, const void* v, const void* a, const void* b,
                            const float* A_log, const float* dt_bias, void* state_pool, int pool_dtype,
                            int num_slots, const int32_t* state_indices, const int32_t* cu_seqlens, int N,
                            int64_t T_total, int Hk, int Hv, int K, int V, float scale, int dtype, int flags,
                            void* o, void* intermediate_states, int steps, gdr_stream_t stream) {
    const RawGates rg{a, b, A_log, dt_bias};
    return recurrent_impl(q, k, v, nullptr, nullptr, &rg, nullptr, state_pool, pool_dtype, num_slots, state_indices,
                          cu_seqlens, N, T_total, Hk, Hv, K, V, scale, dtype, flags, o, intermediate_states, steps,
                          stream, "gdr_recurrent_fwd_gated");
}

int gdr_gating_fwd(const void* a, const float* dt_bias, const float* A_log, const void* b, int64_t T,
                   int Hv, int dtype, int flags, float* g, void* beta, gdr_stream_t stream) {
    if (T < 0 || Hv <= 0) return fail(GDR_ERR_INVALID_ARG, "bad T (%lld) or Hv (%d)", (long long)T, Hv);
    if (dtype != GDR_BF16 && dtype != GDR_F32) return fail(GDR_ERR_UNSUPPORTED, "dtype %d", dtype);
    if (flags & ~GDR_NEG_EIGVAL) return fail(GDR_ERR_INVALID_ARG, "unsupported flags 0x%x", flags);
    if (T == 0) return ok();
    if (!a || !dt_bias || !A_log || !b || !g || !beta) return fail(GDR_ERR_INVALID_ARG, "null pointer argument");
    if (int rc = check_device()) return rc;
    GatingArgs ga{};
    ga.a = a; ga.dt_bias = dt_bias; ga.A_log = A_log; ga.b = b; ga.g = g; ga.beta = beta;
    ga.T = T; ga.Hv = Hv; ga.dtype = dtype; ga.flags = flags;
    return launch_status(launch_gating(ga, (cudaStream_t)stream), "gdr_gating_fwd launch");
}

int gdr_get_device_status(gdr_stream_t stream, int* word) {
    unsigned int* p = device_error_word();
    if (!p) return fail(GDR_ERR_LAUNCH, "error word unavailable");
    unsigned int host = 0;
    cudaError_t e = cudaMemcpyAsync(&host, p, sizeof(host), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, sizeof(host), (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return fail(GDR_ERR_LAUNCH, "device status: %s", cudaGetErrorString(e));
    if (word) *word = (int)host;
    if (host) return fail(GDR_ERR_DEVICE_TIMEOUT, "device error word 0x%x", host);
    return ok();
}

}  // extern "C"
