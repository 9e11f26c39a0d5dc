// Recurrent decode / multi-step verify over a slot-indexed state pool.
//
// Design (FlashQLA PR #1, core decode-kernel and paged-verify commits, read
// for what they compute; the H100 tiling is not reused):
//   * one CTA per (sequence b, value-head h, block of BV value rows);
//   * the fp32 state rows live in registers for the whole sequence: a warp
//     owns 16 consecutive rows, lane l holds K/32 consecutive key channels of
//     each row, so a row is one coalesced 512-byte (fp32) read;
//   * per token the two state-vector products S k and S q are reduced for all
//     16 rows at once with a halving butterfly (31 shuffles instead of 160);
//   * o_t = scale * S_t q_t is formed as scale * (a S_{t-1} q + n_t (k . q)),
//     which is S_t q_t with the rank-1 term expanded;
//   * the state stays V-major end to end (pool, intermediate states), so every
//     store is a coalesced row write (the same page measured a K-major
//     transpose store of the final state at ~0.4 TB/s).
// No tensor cores: every step is a matrix-vector product (M = 1).
#include "common.cuh"
#include "launch.h"

namespace gdr {
namespace {

constexpr int kRowsPerWarp = 16;
constexpr int kLptMax = 1024;  // sequences ranked in shared memory


struct RecParams {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const void* beta;
    void* pool;
    const int32_t* idx;
    const int32_t* cu;
    void* o;
    void* ibuf;
    int Hk, Hv, steps, flags, num_slots;
    int lpt;  // multi-token batch of at most kLptMax sequences: longest first
    int64_t T;
    float scale;
    const void* ga;  // raw gate projections (kGate == 2)
    const void* gb;
    const float* A_log;
    const float* dt_bias;
    float beta_mul;
    const float* nw;  // gated RMSNorm epilogue: weight [V], gate [T, Hv, V], eps
    const void* nz;
    float neps;
};

// The sequence of rank r in longest-first order (ties by index; padding and
// out-of-range slots last, as zero-length), for the CTA's NT threads.  Every
// CTA of a multi-token call ranks the (at most kLptMax) sequences itself: the
// lengths are bucketed (0..63, longer ones share bucket 63), the bucket of
// rank r found from the bucket counts, then its sequence by a block-wide
// count in index order.  Costs one coalesced pass over cu_seqlens and the
// slot indices.
template <int NT>
__device__ int lpt_sequence(const RecParams& p, int N, int r) {
    __shared__ int hist[64];
    __shared__ unsigned char key[kLptMax];
    __shared__ int wsum[NT / 32];
    __shared__ int sel_bucket, sel_off, sel;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < 64; i += NT) hist[i] = 0;
    if (tid == 0) sel = -1;
    __syncthreads();
    for (int j = tid; j < N; j += NT) {
        const int slot = p.idx[j];
        const int64_t lo = max(p.cu[j], 0), hi = min((int64_t)p.cu[j + 1], p.T);
        const int len = (slot < 0 || slot >= p.num_slots || hi <= lo) ? 0 : (int)min(hi - lo, (int64_t)63);
        key[j] = (unsigned char)len;
        atomicAdd(&hist[len], 1);
    }
    __syncthreads();
    if (tid == 0) {
        int acc = 0, bk = 0, off = 0;
        for (int k = 63; k >= 0; --k) {
            if (r < acc + hist[k]) { bk = k; off = r - acc; break; }
            acc += hist[k];
        }
        sel_bucket = bk;
        sel_off = off;
    }
    __syncthreads();
    const int bk = sel_bucket;
    int off = sel_off;
    for (int base = 0; base < N; base += NT) {
        const int j = base + tid;
        const bool f = j < N && key[j] == bk;
        const unsigned m = __ballot_sync(0xffffffffu, f);
        if (lane == 0) wsum[warp] = __popc(m);
        __syncthreads();
        int pre = 0, tot = 0;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) {
            pre += w < warp ? wsum[w] : 0;
            tot += wsum[w];
        }
        pre += __popc(m & ((1u << lane) - 1u));
        if (f && pre == off) sel = j;
        off -= tot;
        __syncthreads();
        if (sel >= 0) break;  // uniform: read after the barrier
    }
    return sel;
}

// kMode & 3: 0 scalar log-decay g [T, Hv]; 1 per-key-channel g [T, Hv, K];
// 2 gates formed from raw projections (FlashQLA in-kernel gating commit).
// kMode & 4: gated RMSNorm output epilogue, o <- rmsnorm(o) * w * sigmoid(z)
// over each value row (tokenspeed PR #834, fused gated-norm commit); the CTA
// then owns the whole row (BV = V) and sums the squares across its warps.

// At most 128 registers per thread: four 128-thread (two 256-thread) CTAs per
// SM keep enough rows in flight (the per-token loop is latency-bound).
template <typename InT, typename PoolT, int K, int BV, int kMode>
__global__ void __launch_bounds__(BV / kRowsPerWarp * 32, BV == 64 ? 4 : BV == 128 ? 2 : 1)
recurrent_kernel(RecParams p) {
    constexpr int kGate = kMode & 3;
    constexpr bool kNorm = (kMode & 4) != 0;
    constexpr int kWarps = BV / kRowsPerWarp;
    __shared__ float ssq[2][kWarps];  // per-warp sums of squares, by token parity
    constexpr int KPT = K / 32;  // key channels per lane
    // Work unit (sequence b, head h, value block zb).  Multi-token calls take
    // the sequences longest first, sequence-major, so that the long ones do not
    // form the tail of the grid.
    int b = blockIdx.x, h = blockIdx.y, zb = blockIdx.z;
    if (p.lpt) {
        const int units = gridDim.y * gridDim.z;
        const int lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        const int r = lin / units, u = lin - r * units;
        h = u / gridDim.z;
        zb = u - h * gridDim.z;
        b = lpt_sequence<BV / kRowsPerWarp * 32>(p, gridDim.x, r);
        if (b < 0) return;
    }
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int slot = p.idx[b];
    if (slot < 0 || slot >= p.num_slots) return;  // padding (or out of range): untouched
    // token range clamped to [0, T) so a malformed cu_seqlens cannot index out of bounds
    const int bos = max(p.cu[b], 0), eos = (int)min((int64_t)p.cu[b + 1], p.T);
    const int kh = h / (p.Hv / p.Hk);
    const int V = gridDim.z * BV;
    const int v0 = zb * BV + warp * kRowsPerWarp;

    const InT* __restrict__ qp = static_cast<const InT*>(p.q);
    const InT* __restrict__ kp = static_cast<const InT*>(p.k);
    const InT* __restrict__ vp = static_cast<const InT*>(p.v);
    const InT* __restrict__ bp = static_cast<const InT*>(p.beta);
    InT* __restrict__ op = static_cast<InT*>(p.o);
    PoolT* pool = static_cast<PoolT*>(p.pool);

    PoolT* srow = pool + (((size_t)slot * p.Hv + h) * V + v0) * K + lane * KPT;
    float s[kRowsPerWarp][KPT];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) Vec<PoolT, KPT>::load(srow + (size_t)r * K, s[r]);

    // Per-token inputs of token t + 1 are loaded while token t is processed, so
    // their global-load latency is hidden behind the reductions of the current token.
    constexpr bool chan = kGate == 1;  // GDR_CHANNEL_GATE: g is [T, Hv, K]
    constexpr bool raw = kGate == 2;   // g and beta from raw projections
    const InT* __restrict__ gap = static_cast<const InT*>(p.ga);
    const InT* __restrict__ gbp = static_cast<const InT*>(p.gb);
    const float negA = raw ? -expf(p.A_log[h]) : 0.f, dtb = raw ? p.dt_bias[h] : 0.f;
    float kn[KPT], qn[KPT], gcn[KPT], gn = 0.f, bn = 0.f, vn = 0.f, zn = 0.f, an = 0.f, bbn = 0.f;
    const InT* __restrict__ nzp = static_cast<const InT*>(p.nz);
    const float nwv = kNorm ? p.nw[v0 + (lane & 15)] : 0.f;
    int par = 0;
    auto load_token = [&](int t) {
        Vec<InT, KPT>::load(kp + ((size_t)t * p.Hk + kh) * K + lane * KPT, kn);
        Vec<InT, KPT>::load(qp + ((size_t)t * p.Hk + kh) * K + lane * KPT, qn);
        if (chan) Vec<float, KPT>::load(p.g + ((size_t)t * p.Hv + h) * K + lane * KPT, gcn);
        else if (!raw) gn = p.g[(size_t)t * p.Hv + h];
        if (!raw) bn = to_f(bp[(size_t)t * p.Hv + h]);
        if (raw) {  // raw projections of the gates
            an = to_f(gap[(size_t)t * p.Hv + h]);
            bbn = to_f(gbp[(size_t)t * p.Hv + h]);
        }
        vn = to_f(vp[((size_t)t * p.Hv + h) * V + v0 + (lane & 15)]);
        if (kNorm) zn = to_f(nzp[((size_t)t * p.Hv + h) * V + v0 + (lane & 15)]);
    };
    // raw projections: the decay and beta of the next token are formed at the
    // end of the current one, once its loads have landed, off the next token's
    // dependency chain (every lane forms them; no exchange)
    float ra = 1.f, rb = 0.f;
    auto form_gates = [&]() {
        const float x = an + dtb;  // softplus, threshold 20, as gdr_gating_fwd
        ra = __expf(negA * (x > 20.f ? x : log1pf(expf(x))));
        rb = p.beta_mul / (1.f + expf(-bbn));
    };
    if (bos < eos) load_token(bos);
    if (raw && bos < eos) form_gates();
#pragma unroll 1
    for (int t = bos; t < eos; ++t) {
        float kk[KPT], qq[KPT], ac[KPT];
#pragma unroll
        for (int c = 0; c < KPT; ++c) { kk[c] = kn[c]; qq[c] = qn[c]; ac[c] = chan ? __expf(gcn[c]) : 1.f; }
        float a, bt;
        if (raw) {
            a = ra;
            bt = rb;
        } else {
            a = chan ? 1.f : __expf(gn);
            bt = bn;
        }
        const float vv = vn, zz = zn;
        if (t + 1 < eos) load_token(t + 1);
        if (p.flags & 1) {  // GDR_QK_L2NORM
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int c = 0; c < KPT; ++c) { sk += kk[c] * kk[c]; sq += qq[c] * qq[c]; }
            const float ik = rsqrtf(warp_sum(sk) + 1e-6f), iq = rsqrtf(warp_sum(sq) + 1e-6f);
#pragma unroll
            for (int c = 0; c < KPT; ++c) { kk[c] *= ik; qq[c] *= iq; }
        }

        // decayed products: scalar gate S~ = a S (a applied after the reduction);
        // channel gate S~ = S diag(ac), i.e. S~ k = S (ac o k), S~ q = S (ac o q)
        float ka[KPT], qa[KPT], da[KPT];
#pragma unroll
        for (int c = 0; c < KPT; ++c) {
            ka[c] = chan ? kk[c] * ac[c] : kk[c];
            qa[c] = chan ? qq[c] * ac[c] : qq[c];
            da[c] = chan ? ac[c] : a;
        }
        float x[32];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            float dk = 0.f, dq = 0.f;
#pragma unroll
            for (int c = 0; c < KPT; ++c) { dk += s[r][c] * ka[c]; dq += s[r][c] * qa[c]; }
            x[r] = dk;
            x[r + kRowsPerWarp] = dq;
        }
        float kq = 0.f;
#pragma unroll
        for (int c = 0; c < KPT; ++c) kq += kk[c] * qq[c];
        kq = warp_sum(kq);
        // lane r < 16 now holds (S k)_r, lane 16 + r holds (S q)_r (before the
        // scalar decay a; channel decays are already inside)
        const float red = reduce32_to_lane(x, lane);
        const float n_mine = bt * (vv - a * red);  // valid on lanes < 16
        const float n_row = __shfl_sync(0xffffffffu, n_mine, lane & 15);
        if (kNorm) {
            const float o = lane >= kRowsPerWarp ? p.scale * (a * red + n_row * kq) : 0.f;
            const float ss = warp_sum(o * o);
            if (lane == 0) ssq[par][warp] = ss;
            __syncthreads();
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) tot += ssq[par][w];
            par ^= 1;
            const float rinv = rsqrtf(tot / (float)V + p.neps);
            if (lane >= kRowsPerWarp)
                op[((size_t)t * p.Hv + h) * V + v0 + (lane - kRowsPerWarp)] =
                    from_f<InT>(o * rinv * nwv / (1.f + __expf(-zz)));
        } else if (lane >= kRowsPerWarp) {
            const float o = p.scale * (a * red + n_row * kq);
            op[((size_t)t * p.Hv + h) * V + v0 + (lane - kRowsPerWarp)] = from_f<InT>(o);
        }
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const float nr = __shfl_sync(0xffffffffu, n_mine, r);
#pragma unroll
            for (int c = 0; c < KPT; ++c) s[r][c] = fmaf(da[c], s[r][c], nr * kk[c]);
        }
        if (p.ibuf && t - bos < p.steps) {
            PoolT* irow = static_cast<PoolT*>(p.ibuf) +
                          ((((size_t)b * p.steps + (t - bos)) * p.Hv + h) * V + v0) * K + lane * KPT;
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) Vec<PoolT, KPT>::store(irow + (size_t)r * K, s[r]);
        }
        if (raw && t + 1 < eos) form_gates();  // token t + 1's raw values were loaded at the top
    }
    if (p.flags & 4) {  // GDR_COMMIT
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) Vec<PoolT, KPT>::store(srow + (size_t)r * K, s[r]);
    }
}

template <typename InT, typename PoolT, int K, int kGate>
cudaError_t launch_k(const RecParams& p, int N, int V, cudaStream_t stream) {
    if (kGate != 2 && p.nw) {  // gated-norm epilogue: one CTA per (sequence, head), BV = V = K
        KernelTimer kt("recurrent", stream);
        recurrent_kernel<InT, PoolT, K, K, kGate | 4><<<dim3(N, p.Hv, 1), K / kRowsPerWarp * 32, 0, stream>>>(p);
        return cudaGetLastError();
    }
    // V-column split: 64-row blocks (128 threads) measured best on GB300 for
    // both single-token decode (6.50 vs 6.42 TB/s at 128 rows) and 12-token
    // verify (4.42 vs 4.10 TB/s); 32-row blocks when there are few sequences.
    const long units = (long)N * p.Hv;
    int bv = 64;
    if (V < 64 || units < 256) bv = 32;
#ifdef GDR_REC_BV
    if (GDR_REC_BV <= V) bv = GDR_REC_BV;  // fixed split for tuning builds
#endif
    dim3 grid(N, p.Hv, V / bv);
    KernelTimer kt("recurrent", stream);
    switch (bv) {
        case 128:
            recurrent_kernel<InT, PoolT, K, 128, kGate><<<grid, 256, 0, stream>>>(p);
            break;
        case 64:
            recurrent_kernel<InT, PoolT, K, 64, kGate><<<grid, 128, 0, stream>>>(p);
            break;
        default:
            recurrent_kernel<InT, PoolT, K, 32, kGate><<<grid, 64, 0, stream>>>(p);
            break;
    }
    return cudaGetLastError();
}

template <typename InT, typename PoolT>
cudaError_t launch_kt(const RecParams& p, int N, int K, int V, cudaStream_t stream) {
    const int mode = p.ga ? 2 : (p.flags & 0x10) ? 1 : 0;  // raw gates / GDR_CHANNEL_GATE / scalar
    if (K == 128) {
        if (mode == 2) return launch_k<InT, PoolT, 128, 2>(p, N, V, stream);
        return mode ? launch_k<InT, PoolT, 128, 1>(p, N, V, stream) : launch_k<InT, PoolT, 128, 0>(p, N, V, stream);
    }
    if (mode == 2) return launch_k<InT, PoolT, 64, 2>(p, N, V, stream);
    return mode ? launch_k<InT, PoolT, 64, 1>(p, N, V, stream) : launch_k<InT, PoolT, 64, 0>(p, N, V, stream);
}

}  // namespace

cudaError_t launch_recurrent(const RecurrentArgs& a, cudaStream_t stream) {
    RecParams p;
    p.q = a.q; p.k = a.k; p.v = a.v; p.g = a.g; p.beta = a.beta;
    p.pool = a.pool; p.idx = a.state_indices; p.cu = a.cu_seqlens;
    p.o = a.o; p.ibuf = a.ibuf;
    p.Hk = a.Hk; p.Hv = a.Hv; p.steps = a.steps; p.flags = a.flags; p.scale = a.scale;
    p.num_slots = a.num_slots;
    p.lpt = a.T > a.N && a.N <= kLptMax;
    p.T = a.T;
    p.ga = a.ga; p.gb = a.gb; p.A_log = a.A_log; p.dt_bias = a.dt_bias; p.beta_mul = a.beta_mul;
    p.nw = a.norm_weight; p.nz = a.norm_gate; p.neps = a.norm_eps;
    const bool in_bf16 = a.dtype == 0, pool_bf16 = a.pool_dtype == 0;
    if (in_bf16 && pool_bf16) return launch_kt<__nv_bfloat16, __nv_bfloat16>(p, a.N, a.K, a.V, stream);
    if (in_bf16) return launch_kt<__nv_bfloat16, float>(p, a.N, a.K, a.V, stream);
    if (pool_bf16) return launch_kt<float, __nv_bfloat16>(p, a.N, a.K, a.V, stream);
    return launch_kt<float, float>(p, a.N, a.K, a.V, stream);
}

}  // namespace gdr
