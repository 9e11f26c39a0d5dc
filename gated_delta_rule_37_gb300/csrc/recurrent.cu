// Recurrent decode / multi-step verify over a slot-indexed state pool.
//
// Design (FlashQLA PR #1, core decode-kernel and paged-verify commits, read
// for what they compute; the H100 tiling is not reused):
//   * one CTA per (sequence b, value-head h, block of BV value rows);
//   * the fp32 state rows live in registers for the whole sequence: a warp
//     owns 16 consecutive rows, lane l holds K/32 consecutive key channels of
//     each row, so a row is one coalesced 512-byte (fp32) read;
//   * the lane's state channels are held as fp32x2 register pairs, so the two
//     state-vector products S k and S q and the rank-1 update run as packed
//     FMAs (Blackwell's f32x2 pipe: half the instructions of scalar FMAs);
//   * per token the products are reduced for all 16 rows at once with a
//     halving butterfly (31 shuffles instead of 160); the upper half-warp
//     takes k and q in swapped roles, so the first halving step needs no
//     select;
//   * multi-token calls (verify) stage each window of up to 16 tokens' inputs
//     in shared memory with one wave of loads per CTA, and do the per-token
//     work that does not touch the state (l2 normalisation, k . q, decays,
//     beta) once per CTA; single-token calls (decode) read their inputs
//     straight from global memory;
//   * o_t = scale * S_t q_t is formed as scale * (a S_{t-1} q + n_t (k . q)),
//     which is S_t q_t with the rank-1 term expanded;
//   * the state stays V-major end to end (pool, intermediate states), so every
//     store is a coalesced row write (the same page measured a K-major
//     transpose store of the final state at ~0.4 TB/s).
// No tensor cores: every step is a matrix-vector product (M = 1).
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace gdr {
namespace {

constexpr int kRowsPerWarp = 16;
constexpr int kLptMax = 1024;  // sequences ranked in shared memory
constexpr int kWin = 16;       // tokens whose inputs are staged in shared memory at once

// Dynamic shared memory of the staged (multi-token) input path, in bytes.
template <int K, int BV, int kMode>
constexpr unsigned stage_bytes() {
    return sizeof(float) * kWin * (2 * K + BV + ((kMode & 4) ? BV : 0) + ((kMode & 3) == 1 ? K : 0) + 4);
}

// N consecutive floats of shared memory (N = 2 or 4, 8- or 16-byte aligned)
template <int N> __device__ __forceinline__ void lds(const float* p, float* out) {
    if constexpr (N == 4) {
        const float4 t = *reinterpret_cast<const float4*>(p);
        out[0] = t.x; out[1] = t.y; out[2] = t.z; out[3] = t.w;
    } else {
        const float2 t = *reinterpret_cast<const float2*>(p);
        out[0] = t.x; out[1] = t.y;
    }
}


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
    int lpt;     // multi-token batch of at most kLptMax sequences: longest first
    int pf_stride;  // with lpt: CTAs resident at once (L2 warming of the next unit), 0 = off
    int staged;  // multi-token batch: inputs staged in shared memory by window
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

// The sequences of ranks r and r2 in longest-first order (ties by index;
// padding and out-of-range slots last, as zero-length), for the CTA's NT
// threads; r2 < 0 asks for none (-1 returned).  Every CTA of a multi-token
// call ranks the (at most kLptMax) sequences itself: the lengths are bucketed
// (0..63, longer ones share bucket 63), the bucket of each rank is found from
// the bucket counts (one warp per rank, two buckets per lane, a prefix sum
// over the lanes), then its sequence by a block-wide count in index order.
// Costs one coalesced pass over cu_seqlens and the slot indices.
template <int NT>
__device__ int2 lpt_sequences(const RecParams& p, int N, int r, int r2) {
    static_assert(NT >= 64, "two warps search the two ranks");
    __shared__ int hist[64];
    __shared__ unsigned char key[kLptMax];
    __shared__ int wsum[2][NT / 32];
    __shared__ int sel_bucket[2], sel_off[2], sel[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < 64; i += NT) hist[i] = 0;
    if (tid < 2) sel[tid] = -1;
    __syncthreads();
    for (int j = tid; j < N; j += NT) {
        const int slot = p.idx[j];
        const int64_t lo = max(p.cu[j], 0), hi = min((int64_t)p.cu[j + 1], p.T);
        const int len = (slot < 0 || slot >= p.num_slots || hi <= lo) ? 0 : (int)min(hi - lo, (int64_t)63);
        key[j] = (unsigned char)len;
        atomicAdd(&hist[len], 1);
    }
    __syncthreads();
    if (warp < 2) {
        // lane l covers buckets 63 - 2l and 62 - 2l: a prefix sum over the lanes
        // counts the sequences in longer buckets, and the one lane whose span
        // holds the rank names the bucket and the offset in it
        const int rr = warp ? r2 : r;
        const int h0 = hist[63 - 2 * lane], h1 = hist[62 - 2 * lane];
        int incl = h0 + h1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int before = incl - h0 - h1;
        const bool hit = rr >= before && rr < incl;
        if (hit) {
            const bool first = rr < before + h0;
            sel_bucket[warp] = first ? 63 - 2 * lane : 62 - 2 * lane;
            sel_off[warp] = first ? rr - before : rr - before - h0;
        }
        if (__ballot_sync(0xffffffffu, hit) == 0u && lane == 0) {  // no such rank (r2 < 0)
            sel_bucket[warp] = -1;
            sel_off[warp] = 0;
        }
    }
    __syncthreads();
    const int bk0 = sel_bucket[0], bk1 = sel_bucket[1];
    int off0 = sel_off[0], off1 = sel_off[1];
    for (int base = 0; base < N; base += NT) {
        const int j = base + tid;
        const bool f0 = j < N && key[j] == bk0, f1 = j < N && key[j] == bk1;
        const unsigned m0 = __ballot_sync(0xffffffffu, f0), m1 = __ballot_sync(0xffffffffu, f1);
        if (lane == 0) {
            wsum[0][warp] = __popc(m0);
            wsum[1][warp] = __popc(m1);
        }
        __syncthreads();
        int pre0 = 0, tot0 = 0, pre1 = 0, tot1 = 0;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) {
            pre0 += w < warp ? wsum[0][w] : 0;
            tot0 += wsum[0][w];
            pre1 += w < warp ? wsum[1][w] : 0;
            tot1 += wsum[1][w];
        }
        const unsigned below = (1u << lane) - 1u;
        if (f0 && pre0 + __popc(m0 & below) == off0) sel[0] = j;
        if (f1 && pre1 + __popc(m1 & below) == off1) sel[1] = j;
        off0 -= tot0;
        off1 -= tot1;
        __syncthreads();
        if (sel[0] >= 0 && (bk1 < 0 || sel[1] >= 0)) break;  // uniform: read after the barrier
    }
    return make_int2(sel[0], sel[1]);
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
    // With pf_stride (the CTAs resident at once), the CTA also names the unit
    // that its slot of the GPU will most likely run next, lin + pf_stride, and
    // warms L2 with that unit's state slab and first input rows.
    int b = blockIdx.x, h = blockIdx.y, zb = blockIdx.z;
    int pb = -1, ph = 0, pzb = 0;  // the next unit on this slot (pb < 0: none)
    if (p.lpt) {
        const int units = gridDim.y * gridDim.z;
        const int lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        const int r = lin / units, u = lin - r * units;
        h = u / gridDim.z;
        zb = u - h * gridDim.z;
        const int lin2 = lin + p.pf_stride;
        const bool pf = p.pf_stride > 0 && lin2 < (int)gridDim.x * units;
        const int r2 = pf ? lin2 / units : -1;
        const int2 bb = lpt_sequences<BV / kRowsPerWarp * 32>(p, gridDim.x, r, r2);
        b = bb.x;
        if (pf && bb.y >= 0) {
            const int u2 = lin2 - r2 * units;
            pb = bb.y;
            ph = u2 / gridDim.z;
            pzb = u2 - ph * gridDim.z;
        }
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
    // s2[r][i] = (S[r][2i], S[r][2i + 1]): two neighbouring channels per
    // register pair, so the products and the update run as packed fp32x2 FMAs
    constexpr int KP = KPT / 2;
    float2 s2[kRowsPerWarp][KP];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        float t[KPT];
        Vec<PoolT, KPT>::load(srow + (size_t)r * K, t);
#pragma unroll
        for (int i = 0; i < KP; ++i) s2[r][i] = make_float2(t[2 * i], t[2 * i + 1]);
    }
    auto row = [&](int r, float* t) {
#pragma unroll
        for (int i = 0; i < KP; ++i) { t[2 * i] = s2[r][i].x; t[2 * i + 1] = s2[r][i].y; }
    };

    constexpr bool chan = kGate == 1;  // GDR_CHANNEL_GATE: g is [T, Hv, K]
    constexpr bool raw = kGate == 2;   // g and beta from raw projections
    constexpr int NT = kWarps * 32;
    const InT* __restrict__ gap = static_cast<const InT*>(p.ga);
    const InT* __restrict__ gbp = static_cast<const InT*>(p.gb);
    const InT* __restrict__ nzp = static_cast<const InT*>(p.nz);
    const float nwv = kNorm ? p.nw[v0 + (lane & 15)] : 0.f;
    const int tid = threadIdx.x;
    const bool up = lane >= 16;

    // decay a (scalar gates; 1 for channel gates) and beta of token t
    auto gates = [&](int t, float& a, float& bt) {
        const size_t th = (size_t)t * p.Hv + h;
        a = 1.f;
        if (raw) {  // softplus (threshold 20) and sigmoid, as gdr_gating_fwd
            const float x = to_f(gap[th]) + p.dt_bias[h];
            a = __expf(-expf(p.A_log[h]) * (x > 20.f ? x : log1pf(expf(x))));
            bt = p.beta_mul / (1.f + expf(-to_f(gbp[th])));
        } else {
            if (!chan) a = __expf(p.g[th]);
            bt = to_f(bp[th]);
        }
    };
    // warp-collective: l2-normalise q and k in place (GDR_QK_L2NORM), return k.q
    auto norm_kq = [&](float* kk, float* qq) {
        if (p.flags & 1) {
            float s1 = 0.f, s2q = 0.f;
#pragma unroll
            for (int c = 0; c < KPT; ++c) { s1 += kk[c] * kk[c]; s2q += qq[c] * qq[c]; }
            const float ik = rsqrtf(warp_sum(s1) + 1e-6f), iq = rsqrtf(warp_sum(s2q) + 1e-6f);
#pragma unroll
            for (int c = 0; c < KPT; ++c) { kk[c] *= ik; qq[c] *= iq; }
        }
        float kq = 0.f;
#pragma unroll
        for (int c = 0; c < KPT; ++c) kq += kk[c] * qq[c];
        return warp_sum(kq);
    };

    // One token on the register-resident state.  kk: the lane's k channels;
    // uu / ww: k / q for lanes < 16 and q / k for lanes >= 16 (the upper
    // half-warp takes them in swapped roles, so that the first halving step of
    // the reduction pairs x[r] with the partner's x[16 + r] and needs no
    // select); ac: exp of the channel log-decays.
    int par = 0;
    auto step = [&](int t, const float* kk, const float* uu, const float* ww, const float* ac, float a, float bt,
                    float kq, float vv, float zz) {
        // decayed products: scalar gate S~ = a S (a applied after the reduction);
        // channel gate S~ = S diag(ac), i.e. S~ k = S (ac o k), S~ q = S (ac o q)
        float2 u2[KP], w2[KP], da2[KP], kk2[KP];
#pragma unroll
        for (int i = 0; i < KP; ++i) {
            u2[i] = make_float2(uu[2 * i], uu[2 * i + 1]);
            w2[i] = make_float2(ww[2 * i], ww[2 * i + 1]);
            kk2[i] = make_float2(kk[2 * i], kk[2 * i + 1]);
            if (chan) {
                da2[i] = make_float2(ac[2 * i], ac[2 * i + 1]);
                u2[i] = __fmul2_rn(u2[i], da2[i]);
                w2[i] = __fmul2_rn(w2[i], da2[i]);
            } else {
                da2[i] = make_float2(a, a);
            }
        }
        float x[32];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            float2 du = __fmul2_rn(s2[r][0], u2[0]), dw = __fmul2_rn(s2[r][0], w2[0]);
#pragma unroll
            for (int i = 1; i < KP; ++i) {
                du = __ffma2_rn(s2[r][i], u2[i], du);
                dw = __ffma2_rn(s2[r][i], w2[i], dw);
            }
            x[r] = du.x + du.y;
            x[16 + r] = dw.x + dw.y;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] += __shfl_xor_sync(0xffffffffu, x[i + 16], 16);
        // lane r < 16 now holds (S k)_r, lane 16 + r holds (S q)_r (before the
        // scalar decay a; channel decays are already inside)
        const float red = reduce16_to_lane(x, lane);
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
            const float2 n2 = make_float2(nr, nr);
#pragma unroll
            for (int i = 0; i < KP; ++i) s2[r][i] = __ffma2_rn(da2[i], s2[r][i], __fmul2_rn(n2, kk2[i]));
        }
        if (p.ibuf && t - bos < p.steps) {
            PoolT* irow = static_cast<PoolT*>(p.ibuf) +
                          ((((size_t)b * p.steps + (t - bos)) * p.Hv + h) * V + v0) * K + lane * KPT;
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                float t2[KPT];
                row(r, t2);
                Vec<PoolT, KPT>::store_cs(irow + (size_t)r * K, t2);  // never read back here
            }
        }
    };

    if (p.staged) {
        // Multi-token calls: the inputs of up to kWin tokens are staged in
        // shared memory, in fp32, by the whole CTA at once, so every load of a
        // window is in flight together (with the state loads, for the first
        // window), and the per-token work that does not depend on the state
        // (l2 normalisation, k.q, the decays and beta) is done once per CTA
        // rather than once per warp.  Layout (dynamic shared memory, floats):
        // q rows [kWin][K], k rows [kWin][K], v slice [kWin][BV], norm-gate
        // slice [kWin][BV] (kNorm), exp'd channel decays [kWin][K] (chan),
        // per token {decay, beta, k.q, -} [kWin][4].
        extern __shared__ __align__(16) float dsm[];
        float* sq = dsm;
        float* sk = sq + kWin * K;
        float* sv = sk + kWin * K;
        float* sz = sv + kWin * BV;
        float* sg = sz + (kNorm ? kWin * BV : 0);
        float* stok = sg + (chan ? kWin * K : 0);
        const float* ub = up ? sq : sk;
        const float* wb = up ? sk : sq;
#pragma unroll 1
        for (int t0 = bos; t0 < eos; t0 += kWin) {
            const int n = min(kWin, eos - t0);
            if (t0 > bos) __syncthreads();  // the previous window has been read
            constexpr int E = 16 / sizeof(InT);  // elements per 16-byte piece
            constexpr int PR = K / E, PV = BV / E;
#pragma unroll
            for (int it = 0; it < (kWin * PR + NT - 1) / NT; ++it) {
                const int i = it * NT + tid, j = i / PR, c = (i - j * PR) * E;
                if (j < n) {
                    const size_t off = ((size_t)(t0 + j) * p.Hk + kh) * K + c;
                    float a[E], bq[E];
                    Vec<InT, E>::load(kp + off, a);
                    Vec<InT, E>::load(qp + off, bq);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        sk[j * K + c + e] = a[e];
                        sq[j * K + c + e] = bq[e];
                    }
                }
            }
#pragma unroll
            for (int it = 0; it < (kWin * PV + NT - 1) / NT; ++it) {
                const int i = it * NT + tid, j = i / PV, c = (i - j * PV) * E;
                if (j < n) {
                    const size_t off = ((size_t)(t0 + j) * p.Hv + h) * V + zb * BV + c;
                    float a[E], z[E];
                    Vec<InT, E>::load(vp + off, a);
                    if (kNorm) Vec<InT, E>::load(nzp + off, z);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        sv[j * BV + c + e] = a[e];
                        if (kNorm) sz[j * BV + c + e] = z[e];
                    }
                }
            }
            if (chan) {
#pragma unroll
                for (int it = 0; it < (kWin * K / 4 + NT - 1) / NT; ++it) {
                    const int i = it * NT + tid, j = i / (K / 4), c = (i - j * (K / 4)) * 4;
                    if (j < n) {
                        float gc[4];
                        Vec<float, 4>::load(p.g + ((size_t)(t0 + j) * p.Hv + h) * K + c, gc);
#pragma unroll
                        for (int e = 0; e < 4; ++e) sg[j * K + c + e] = __expf(gc[e]);
                    }
                }
            }
            if (tid < n) {
                float a, bt;
                gates(t0 + tid, a, bt);
                stok[4 * tid] = a;
                stok[4 * tid + 1] = bt;
            }
            __syncthreads();
            for (int j = warp; j < n; j += kWarps) {  // one warp per token
                float kk[KPT], qq[KPT];
                lds<KPT>(sk + j * K + lane * KPT, kk);
                lds<KPT>(sq + j * K + lane * KPT, qq);
                const float kq = norm_kq(kk, qq);
                if (p.flags & 1) {
#pragma unroll
                    for (int c = 0; c < KPT; ++c) {
                        sk[j * K + lane * KPT + c] = kk[c];
                        sq[j * K + lane * KPT + c] = qq[c];
                    }
                }
                if (lane == 0) stok[4 * j + 2] = kq;
            }
            __syncthreads();
            if (t0 == bos && pb >= 0 && warp == kWarps - 1) {
                // warm L2 for the next unit on this slot of the GPU: its state
                // slab, and the k, q rows and v slice of its first window
                const int s2 = p.idx[pb];
                if (s2 >= 0 && s2 < p.num_slots) {
                    const int bos2 = max(p.cu[pb], 0), eos2 = (int)min((int64_t)p.cu[pb + 1], p.T);
                    const int n2 = min(kWin, eos2 - bos2), kh2 = ph / (p.Hv / p.Hk);
                    if (lane == 0)
                        tc::prefetch_l2(pool + (((size_t)s2 * p.Hv + ph) * V + pzb * BV) * K,
                                        (uint32_t)(BV * K * sizeof(PoolT)));
                    for (int e = lane - 1; e >= 0 && e < 3 * n2; e += 31) {
                        const int i = e / 3, w = e - 3 * i;
                        const size_t t2 = (size_t)(bos2 + i);
                        if (w == 0) tc::prefetch_l2(kp + (t2 * p.Hk + kh2) * K, (uint32_t)(K * sizeof(InT)));
                        else if (w == 1) tc::prefetch_l2(qp + (t2 * p.Hk + kh2) * K, (uint32_t)(K * sizeof(InT)));
                        else tc::prefetch_l2(vp + (t2 * p.Hv + ph) * V + pzb * BV, (uint32_t)(BV * sizeof(InT)));
                    }
                }
            }
#pragma unroll 1
            for (int j = 0; j < n; ++j) {
                float kk[KPT], uu[KPT], ww[KPT], ac[KPT];
                lds<KPT>(sk + j * K + lane * KPT, kk);
                lds<KPT>(ub + j * K + lane * KPT, uu);
                lds<KPT>(wb + j * K + lane * KPT, ww);
                if (chan) lds<KPT>(sg + j * K + lane * KPT, ac);
                const float4 tk = *reinterpret_cast<const float4*>(stok + 4 * j);
                const int vr = warp * kRowsPerWarp + (lane & 15);
                step(t0 + j, kk, uu, ww, ac, tk.x, tk.y, tk.z, sv[j * BV + vr], kNorm ? sz[j * BV + vr] : 0.f);
            }
        }
    } else {
        // Single-token calls (decode): every warp reads its token's inputs
        // straight from global memory, with no shared-memory round trip.
#pragma unroll 1
        for (int t = bos; t < eos; ++t) {
            float kk[KPT], qq[KPT], uu[KPT], ww[KPT], ac[KPT];
            Vec<InT, KPT>::load(kp + ((size_t)t * p.Hk + kh) * K + lane * KPT, kk);
            Vec<InT, KPT>::load(qp + ((size_t)t * p.Hk + kh) * K + lane * KPT, qq);
            if (chan) {
                Vec<float, KPT>::load(p.g + ((size_t)t * p.Hv + h) * K + lane * KPT, ac);
#pragma unroll
                for (int c = 0; c < KPT; ++c) ac[c] = __expf(ac[c]);
            }
            const size_t vo = ((size_t)t * p.Hv + h) * V + v0 + (lane & 15);
            const float vv = to_f(vp[vo]);
            const float zz = kNorm ? to_f(nzp[vo]) : 0.f;
            float a, bt;
            gates(t, a, bt);
            const float kq = norm_kq(kk, qq);
#pragma unroll
            for (int c = 0; c < KPT; ++c) {
                uu[c] = up ? qq[c] : kk[c];
                ww[c] = up ? kk[c] : qq[c];
            }
            step(t, kk, uu, ww, ac, a, bt, kq, vv, zz);
        }
    }
    if (p.flags & 4) {  // GDR_COMMIT
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            float t2[KPT];
            row(r, t2);
            Vec<PoolT, KPT>::store(srow + (size_t)r * K, t2);
        }
    }
}

// One instantiation on `grid`.  Multi-token calls in longest-first order also
// get the number of CTAs resident at once (occupancy x SMs), which names the
// unit each CTA warms L2 for.
template <typename InT, typename PoolT, int K, int BV, int kMode>
cudaError_t launch_one(RecParams p, dim3 grid, int sms, cudaStream_t stream) {
    constexpr int threads = BV / kRowsPerWarp * 32;
    const unsigned smem = p.staged ? stage_bytes<K, BV, kMode>() : 0;
    p.pf_stride = 0;
    if (p.lpt && sms > 0) {
        static const int per_sm = [] {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, recurrent_kernel<InT, PoolT, K, BV, kMode>, threads,
                                                              stage_bytes<K, BV, kMode>()) != cudaSuccess)
                n = 0;
            return n;
        }();
        p.pf_stride = per_sm * sms;
    }
    recurrent_kernel<InT, PoolT, K, BV, kMode><<<grid, threads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <typename InT, typename PoolT, int K, int kGate>
cudaError_t launch_k(const RecParams& p, int N, int V, cudaStream_t stream) {
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 0;
    KernelTimer kt("recurrent", stream);
    if (kGate != 2 && p.nw)  // gated-norm epilogue: one CTA per (sequence, head), BV = V = K
        return launch_one<InT, PoolT, K, K, kGate | 4>(p, dim3(N, p.Hv, 1), sms, stream);
    // V-column split.  Single-token decode: 64-row blocks (128 threads)
    // measured best on GB300 (6.50 vs 6.42 TB/s at 128 rows).  Multi-token
    // calls: 128-row blocks (256 threads), since one CTA then stages a window's
    // q, k rows and per-token scalars for twice the rows (verify 0.098 vs
    // 0.103 ms), as long as the units fill every SM with two such CTAs.
    // 32-row blocks when there are few sequences.
    const long units = (long)N * p.Hv;
    int bv = 64;
    if (V < 64 || units < 256) bv = 32;
    else if (p.staged && V % 128 == 0 && sms > 0 && units >= 2L * sms) bv = 128;
#ifdef GDR_REC_BV
    if (GDR_REC_BV <= V) bv = GDR_REC_BV;  // fixed split for tuning builds
#endif
    const dim3 grid(N, p.Hv, V / bv);
    switch (bv) {
        case 128: return launch_one<InT, PoolT, K, 128, kGate>(p, grid, sms, stream);
        case 64: return launch_one<InT, PoolT, K, 64, kGate>(p, grid, sms, stream);
        default: return launch_one<InT, PoolT, K, 32, kGate>(p, grid, sms, stream);
    }
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
    p.staged = a.T > a.N;
    p.pf_stride = 0;
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
