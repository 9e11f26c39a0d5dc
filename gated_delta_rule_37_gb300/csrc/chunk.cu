// Chunked (WY) prefill of the gated delta rule, 64-token chunks.
//
// Steps (each one kernel; the chunk restarts at every sequence start and the
// last chunk of a sequence may be partial):
//   meta   per-sequence chunk offsets and a chunk table, built on the device
//          from cu_seqlens (the host never reads cu_seqlens);
//   prep   optional q/k l2 normalisation into the workspace;
//   intra  per (chunk, value-head): in-chunk gate cumsum gam, the strictly
//          lower A_ij = beta_i sum_c k_i[c] e^{gam_i[c]-gam_j[c]} k_j[c], the
//          unit-lower-triangular inverse Tm = (I + A)^{-1}, the WY factors
//          W = Tm diag(beta) (K o e^{Gam}) and U = Tm diag(beta) V, the
//          decayed keys Kd_j = k_j o e^{gam_L - gam_j}, the decayed queries
//          Qd_i = q_i o e^{gam_i}, the chunk decay e^{gam_L} and the masked
//          attention P_ij = sum_c q_i[c] e^{gam_i[c]-gam_j[c]} k_j[c] (j <= i);
//   state  per (sequence, value-head, block of value rows), serial over the
//          sequence's chunks: store S0 (the chunk's initial state), deltas
//          Nn = U - W S0^T, then S <- S0 diag(e^{gam_L}) + Nn^T Kd
//          (attention-gym PR #344's inter-chunk state kernel, "two dots per
//          chunk");
//   out    per (chunk, value-head): O = scale (Qd S0^T + P Nn).
// Every exponential is of gam_i - gam_j with i >= j or of gam_i itself, all
// <= 0, so any finite gate <= 0 stays finite (cuLA PR #113 review).
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "launch.h"

#include <type_traits>

namespace gdr {

static inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Segment length of the chunk-parallel scan, from a cost model fitted to
// GB300 measurements (microseconds; N sequences of the mean length, 152 SMs,
// one chain or scan CTA per SM).  For S segments of G = ceil(nc / S) chunks:
// the summary pass runs S offsets (the first one from h0, with its output) and
// S - 2 transitions of 4 Hv N CTAs each, the output pass S - 1 segments, the
// scan S - 2 products of a 64 KB transition per CTA:
//   G * (1.51 waves(4 Hv N (2 S - 2)) + 1.75 waves(4 Hv N (S - 1)))
//     + 1.45 (S - 2) waves(32 Hv N) + 10.
// Returns the G of the cheapest S in 2..64 with G >= 4 (ceil(nc / 2) for
// sequences under 8 chunks).  The one pass costs about 1.6 us * nc *
// waves(4 Hv N): the scan pays only while 12 Hv N is well under the SM count.
int chunk_scan_segment(int N, int64_t T, int Hv) {
    constexpr double kSMs = 152.0;
    if (N <= 0 || T <= 0) return 1;
    const double nc = std::ceil((double)T / kChunk / N);
    auto waves = [&](double ctas) { return std::ceil(ctas / kSMs); };
    const double u = 4.0 * Hv * N;
    double best = 1e300;
    int best_g = (int)std::max(1.0, std::ceil(nc / 2));
    for (int S = 2; S <= 64; ++S) {
        const double G = std::ceil(nc / S);
        if (G < 4) break;
        const double segs = std::ceil(nc / G);
        const double t = G * (1.51 * waves(u * (2 * segs - 2)) + 1.75 * waves(u * (segs - 1))) +
                         1.45 * (segs - 2) * waves(32.0 * Hv * N) + 10.0;
        if (t < best) { best = t; best_g = (int)G; }
    }
    return best_g;
}

ChunkWorkspace chunk_workspace_layout(int N, int64_t T, int Hk, int Hv, int K, int V, int gate_kind,
                                      int dtype, int flags) {
    ChunkWorkspace w{};
    w.max_chunks = (T + kChunk - 1) / kChunk + N;
    const size_t esz = dtype == 0 ? 2 : 4;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
    w.off_meta = take(16);
    w.off_offsets = take(sizeof(int) * (size_t)(N + 1));
    w.off_table = take(16 * (size_t)w.max_chunks);
    const bool l2 = flags & 1;
    w.off_qn = take(l2 ? esz * (size_t)T * Hk * K : 0);
    w.off_kn = take(l2 ? esz * (size_t)T * Hk * K : 0);
    w.off_order = take(sizeof(int) * (size_t)(N + 1));
    // bf16 inputs take the tensor-core path (a 64-channel head runs on its
    // 128-channel tiles with the upper half zero); fp32 inputs the CUDA cores
    w.tc = dtype == 0 && K == V && (K == 128 || K == 64);
    if (w.tc) {
        // tensor-core path: pre-swizzled per-chunk operand images only
        w.off_blobs = take(chunk_tc_blob_bytes(w.max_chunks, Hk, Hv, gate_kind == 1));
        // GDR_CHUNK_SCAN (>= 1): 128-channel heads only (the flag is ignored otherwise)
        w.seg_chunks = ((flags & 0x20) && K == 128) ? chunk_scan_segment(N, T, Hv) : 0;
        w.local_meta = w.seg_chunks == 0 && N <= kLocalMetaSeqs;
        if (w.seg_chunks > 0) {
            w.max_segs = (w.max_chunks + w.seg_chunks - 1) / w.seg_chunks + N;
            w.off_segs = take(16 * (size_t)w.max_segs);
            w.off_segoff = take(sizeof(int) * (size_t)(N + 1));
            w.off_mt = take(4 * (size_t)w.max_segs * Hv * K * K);
            w.off_bs = take(4 * (size_t)w.max_segs * Hv * V * K);
        }
        w.total = off;
        return w;
    }
    w.off_w = take(4 * (size_t)T * Hv * K);
    w.off_u = take(4 * (size_t)T * Hv * V);
    w.off_kd = take(4 * (size_t)T * Hv * K);
    w.off_qd = take(4 * (size_t)T * Hv * K);
    w.off_p = take(4 * (size_t)w.max_chunks * Hv * kChunk * kChunk);
    w.off_dl = take(4 * (size_t)w.max_chunks * Hv * K);
    w.off_h = take(4 * (size_t)w.max_chunks * Hv * V * K);
    w.off_vn = take(4 * (size_t)T * Hv * V);
    w.total = off;
    return w;
}

namespace {

// ---------------------------------------------------------------------------
// meta: chunk offsets and table (one CTA)
// ---------------------------------------------------------------------------
// A malformed cu_seqlens (cu[0] != 0, a decreasing entry, cu[N] != T) makes
// the chunk count 0 and meta[1] = 0, so the later kernels touch no memory.
// Below kMetaSmemSeqs sequences the offsets also go to shared memory and the
// chunk table is written with one thread per chunk (its sequence found by
// binary search over the offsets), so one long sequence does not leave its
// table to a single thread; beyond, one thread per sequence writes its chunks.
// Also writes order[]: sequence indices by decreasing length (ties by index),
// the longest-first launch order of the per-sequence kernels (N <= 4096;
// identity beyond).
// With G > 0 (chunk-parallel scan) it also cuts every sequence into segments
// of G chunks (the last one shorter): segs[] = (sequence, first chunk within
// the sequence, chunk count, 1 if it is the sequence's last segment),
// segoff[b] = first segment of sequence b, meta[2] = the segment count.
constexpr int kMetaSmemSeqs = 4096;
__global__ void __launch_bounds__(1024) chunk_meta_kernel(const int32_t* __restrict__ cu, int N,
                                                          int64_t T, int* __restrict__ meta,
                                                          int* __restrict__ offsets,
                                                          int4* __restrict__ table, int* __restrict__ order,
                                                          int G, int4* __restrict__ segs,
                                                          int* __restrict__ segoff) {
    __shared__ int warp_sum[32];
    __shared__ int seg_sum[32];
    __shared__ int s_off[kMetaSmemSeqs + 1];
    __shared__ int bad;
    // the next kernel, if launched as a dependent, may start its prologue now
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) bad = (cu[0] != 0 || (int64_t)cu[N] != T);
    __syncthreads();
    const int per = (N + blockDim.x - 1) / blockDim.x;
    const int b0 = min(N, tid * per), b1 = min(N, b0 + per);
    int cnt = 0;
    for (int b = b0; b < b1; ++b) {
        if (cu[b + 1] < cu[b]) bad = 1;
        cnt += (cu[b + 1] - cu[b] + kChunk - 1) / kChunk;
    }
    // block-wide exclusive scan of the per-thread chunk counts
    int incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) warp_sum[wid] = incl;
    __syncthreads();
    if (bad) {
        if (tid == 0) { meta[0] = 0; meta[1] = 0; meta[2] = 0; }
        return;
    }
    if (wid == 0) {
        int v = warp_sum[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += y;
        }
        warp_sum[lane] = v;
    }
    __syncthreads();
    int c = incl - cnt + (wid > 0 ? warp_sum[wid - 1] : 0);
    if (tid == 0) {
        meta[0] = warp_sum[31];
        meta[1] = 1;
        offsets[N] = warp_sum[31];
    }
    if (N < kMetaSmemSeqs) {
        // offsets into shared memory, then the chunk table with one thread per
        // chunk (its sequence by binary search over the offsets)
        for (int b = b0; b < b1; ++b) {
            offsets[b] = c;
            s_off[b] = c;
            c += (cu[b + 1] - cu[b] + kChunk - 1) / kChunk;
        }
        if (tid == 0) s_off[N] = warp_sum[31];
        __syncthreads();
        const int total = warp_sum[31];
        for (int ci = tid; ci < total; ci += blockDim.x) {
            int lo = 0, hi = N - 1;  // the last sequence whose first chunk is <= ci
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_off[mid] <= ci) lo = mid;
                else hi = mid - 1;
            }
            const int bos = cu[lo], len = cu[lo + 1] - bos, s = (ci - s_off[lo]) * kChunk;
            table[ci] = make_int4(lo, bos + s, min(kChunk, len - s), 0);
        }
    } else {
        for (int b = b0; b < b1; ++b) {
            offsets[b] = c;
            const int bos = cu[b], len = cu[b + 1] - bos;
            for (int s = 0; s < len; s += kChunk, ++c)
                table[c] = make_int4(b, bos + s, min(kChunk, len - s), 0);
        }
    }
    if (G > 0) {
        // the same block-wide exclusive scan over the per-thread segment counts
        int scnt = 0;
        for (int b = b0; b < b1; ++b) {
            const int nc = (cu[b + 1] - cu[b] + kChunk - 1) / kChunk;
            scnt += (nc + G - 1) / G;
        }
        int sincl = scnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, sincl, off);
            if (lane >= off) sincl += y;
        }
        if (lane == 31) seg_sum[wid] = sincl;
        __syncthreads();
        if (wid == 0) {
            int v = seg_sum[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += y;
            }
            seg_sum[lane] = v;
        }
        __syncthreads();
        int sg = sincl - scnt + (wid > 0 ? seg_sum[wid - 1] : 0);
        if (tid == 0) {
            meta[2] = seg_sum[31];
            segoff[N] = seg_sum[31];
        }
        for (int b = b0; b < b1; ++b) {
            segoff[b] = sg;
            const int nc = (cu[b + 1] - cu[b] + kChunk - 1) / kChunk;
            for (int s = 0; s < nc; s += G, ++sg) segs[sg] = make_int4(b, s, min(G, nc - s), s + G >= nc);
        }
    }
    for (int b = tid; b < N; b += blockDim.x) {
        const int lb = cu[b + 1] - cu[b];
        int rank = b;
        if (N <= 4096) {
            rank = 0;
            for (int j = 0; j < N; ++j) {
                const int lj = cu[j + 1] - cu[j];
                rank += (lj > lb) || (lj == lb && j < b);
            }
        }
        order[rank] = b;
    }
}

// ---------------------------------------------------------------------------
// prep: row-wise l2 normalisation, one warp per row of K elements
// ---------------------------------------------------------------------------
template <typename T, int K>
__global__ void l2norm_kernel(const T* __restrict__ x, T* __restrict__ y, int64_t rows) {
    constexpr int KPT = K / 32;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    float v[KPT];
    Vec<T, KPT>::load(x + row * K + lane * KPT, v);
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < KPT; ++c) ss += v[c] * v[c];
    const float inv = rsqrtf(warp_sum(ss) + 1e-6f);
#pragma unroll
    for (int c = 0; c < KPT; ++c) v[c] *= inv;
    Vec<T, KPT>::store(y + row * K + lane * KPT, v);
}

struct ChunkParams {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* gk;
    const void* beta;
    const float* h0;
    void* o;
    float* hT;
    const int* meta;
    const int* offsets;
    const int4* table;
    float* W;
    float* U;
    float* Kd;
    float* Qd;
    float* P;
    float* dL;
    float* H;
    float* Vn;
    const int32_t* cu;
    int Hk, Hv;
    float scale;
};

// ---------------------------------------------------------------------------
// intra: per (chunk, value-head), fp32 SIMT
// ---------------------------------------------------------------------------
template <typename InT, int K>
__global__ void __launch_bounds__(256) chunk_intra_kernel(ChunkParams p) {
    constexpr int C = kChunk;
    constexpr int LD = K + 1;  // padded row stride (floats)
    extern __shared__ float sm[];
    float* Ks = sm;                 // [C][LD]
    float* Qs = Ks + C * LD;        // [C][LD]
    float* Gs = Qs + C * LD;        // [C][LD]  gate cumsum (per channel)
    float* Vs = Gs + C * LD;        // [C][LD]
    float* Am = Vs + C * LD;        // [C][C+1]
    float* Tm = Am + C * (C + 1);   // [C][C+1]
    float* Bs = Tm + C * (C + 1);   // [C]

    const int chunk = blockIdx.x;
    if (chunk >= p.meta[0]) return;
    const int h = blockIdx.y;
    const int4 info = p.table[chunk];
    const int start = info.y, L = info.z;
    const int kh = h / (p.Hv / p.Hk);
    const int tid = threadIdx.x;
    const InT* qp = static_cast<const InT*>(p.q);
    const InT* kp = static_cast<const InT*>(p.k);
    const InT* vp = static_cast<const InT*>(p.v);
    const InT* bp = static_cast<const InT*>(p.beta);

    for (int e = tid; e < C * K; e += blockDim.x) {
        const int i = e / K, c = e % K;
        float kv = 0.f, qv = 0.f, vv = 0.f, gv = 0.f;
        if (i < L) {
            const size_t t = (size_t)start + i;
            kv = to_f(kp[(t * p.Hk + kh) * K + c]);
            qv = to_f(qp[(t * p.Hk + kh) * K + c]);
            vv = to_f(vp[(t * p.Hv + h) * K + c]);  // V == K
            gv = p.gk ? p.gk[(t * p.Hv + h) * K + c] : p.g[t * p.Hv + h];
        }
        Ks[i * LD + c] = kv;
        Qs[i * LD + c] = qv;
        Vs[i * LD + c] = vv;
        Gs[i * LD + c] = gv;
    }
    for (int i = tid; i < C; i += blockDim.x)
        Bs[i] = i < L ? to_f(bp[((size_t)start + i) * p.Hv + h]) : 0.f;
    __syncthreads();
    // in-chunk inclusive cumsum, sequential in token order per channel
    for (int c = tid; c < K; c += blockDim.x) {
        float acc = 0.f;
        for (int i = 0; i < L; ++i) { acc += Gs[i * LD + c]; Gs[i * LD + c] = acc; }
    }
    __syncthreads();
    // A (strictly lower) and P (lower incl. diagonal)
    for (int e = tid; e < C * C; e += blockDim.x) {
        const int i = e / C, j = e % C;
        float a = 0.f, pp = 0.f;
        if (j <= i && i < L) {
            for (int c = 0; c < K; ++c) {
                const float d = __expf(Gs[i * LD + c] - Gs[j * LD + c]);
                const float kj = Ks[j * LD + c] * d;
                a = fmaf(Ks[i * LD + c], kj, a);
                pp = fmaf(Qs[i * LD + c], kj, pp);
            }
        }
        Am[i * (C + 1) + j] = (j < i) ? Bs[i] * a : 0.f;
        p.P[(((size_t)chunk * p.Hv + h) * C + i) * C + j] = (j <= i) ? pp : 0.f;
    }
    __syncthreads();
    // Tm = (I + A)^{-1}: column j by forward substitution (rows >= L stay 0)
    for (int j = tid; j < C; j += blockDim.x) {
        for (int i = 0; i < C; ++i) {
            float x = 0.f;
            if (i < L && i >= j) {
                x = (i == j) ? 1.f : 0.f;
                for (int m = j; m < i; ++m) x = fmaf(-Am[i * (C + 1) + m], Tm[m * (C + 1) + j], x);
            }
            Tm[i * (C + 1) + j] = x;
        }
    }
    __syncthreads();
    // W, U, Kd, Qd rows (only i < L are stored)
    const float* gl = Gs + (L - 1) * LD;
    for (int e = tid; e < L * K; e += blockDim.x) {
        const int i = e / K, c = e % K;
        float w = 0.f, u = 0.f;
        for (int j = 0; j <= i; ++j) {
            const float tb = Tm[i * (C + 1) + j] * Bs[j];
            w = fmaf(tb * __expf(Gs[j * LD + c]), Ks[j * LD + c], w);
            u = fmaf(tb, Vs[j * LD + c], u);
        }
        const size_t row = ((size_t)start + i) * p.Hv + h;
        p.W[row * K + c] = w;
        p.U[row * K + c] = u;
        p.Kd[row * K + c] = Ks[i * LD + c] * __expf(gl[c] - Gs[i * LD + c]);
        p.Qd[row * K + c] = Qs[i * LD + c] * __expf(Gs[i * LD + c]);
    }
    for (int c = tid; c < K; c += blockDim.x) p.dL[((size_t)chunk * p.Hv + h) * K + c] = __expf(gl[c]);
}

// ---------------------------------------------------------------------------
// state: per (sequence, value-head, block of BV value rows), serial in chunks
// ---------------------------------------------------------------------------
template <int K, int BV>
__global__ void __launch_bounds__(256) chunk_state_kernel(ChunkParams p) {
    constexpr int C = kChunk;
    constexpr int LD = K + 1;
    extern __shared__ float sm[];
    float* S = sm;                   // [BV][LD]
    float* Ws = S + BV * LD;         // [C][LD]
    float* Kds = Ws + C * LD;        // [C][LD]
    float* Us = Kds + C * LD;        // [C][BV+1]
    float* dls = Us + C * (BV + 1);  // [K]
    const int b = blockIdx.x, h = blockIdx.y;
    const int V = gridDim.z * BV;
    const int v0 = blockIdx.z * BV;
    const int tid = threadIdx.x;
    if (!p.meta[1]) return;  // malformed cu_seqlens: nothing is touched
    const int bos = p.cu[b], eos = p.cu[b + 1];
    const int c0 = p.offsets[b];

    for (int e = tid; e < BV * K; e += blockDim.x) {
        const int r = e / K, c = e % K;
        S[r * LD + c] = p.h0 ? p.h0[(((size_t)b * p.Hv + h) * V + v0 + r) * K + c] : 0.f;
    }
    int ci = 0;
    for (int cs = bos; cs < eos; cs += C, ++ci) {
        const int L = min(C, eos - cs);
        const size_t chunk = (size_t)c0 + ci;
        __syncthreads();
        for (int e = tid; e < BV * K; e += blockDim.x) {
            const int r = e / K, c = e % K;
            p.H[(((chunk * p.Hv + h) * V) + v0 + r) * K + c] = S[r * LD + c];
        }
        for (int e = tid; e < C * K; e += blockDim.x) {
            const int i = e / K, c = e % K;
            const size_t row = ((size_t)cs + i) * p.Hv + h;
            Ws[i * LD + c] = i < L ? p.W[row * K + c] : 0.f;
            Kds[i * LD + c] = i < L ? p.Kd[row * K + c] : 0.f;
        }
        for (int e = tid; e < C * BV; e += blockDim.x) {
            const int i = e / BV, r = e % BV;
            Us[i * (BV + 1) + r] = i < L ? p.U[(((size_t)cs + i) * p.Hv + h) * V + v0 + r] : 0.f;
        }
        for (int c = tid; c < K; c += blockDim.x) dls[c] = p.dL[(chunk * p.Hv + h) * K + c];
        __syncthreads();
        // deltas Nn[i][r] = U[i][r] - sum_c W[i][c] S[r][c]   (kept in Us)
        for (int e = tid; e < C * BV; e += blockDim.x) {
            const int i = e / BV, r = e % BV;
            float acc = Us[i * (BV + 1) + r];
            for (int c = 0; c < K; ++c) acc = fmaf(-Ws[i * LD + c], S[r * LD + c], acc);
            Us[i * (BV + 1) + r] = i < L ? acc : 0.f;
            if (i < L) p.Vn[(((size_t)cs + i) * p.Hv + h) * V + v0 + r] = acc;
        }
        __syncthreads();
        // S[r][c] = e^{gam_L[c]} S[r][c] + sum_i Nn[i][r] Kd[i][c]
        for (int e = tid; e < BV * K; e += blockDim.x) {
            const int r = e / K, c = e % K;
            float acc = dls[c] * S[r * LD + c];
            for (int i = 0; i < L; ++i) acc = fmaf(Us[i * (BV + 1) + r], Kds[i * LD + c], acc);
            S[r * LD + c] = acc;
        }
    }
    __syncthreads();
    if (p.hT)
        for (int e = tid; e < BV * K; e += blockDim.x) {
            const int r = e / K, c = e % K;
            p.hT[(((size_t)b * p.Hv + h) * V + v0 + r) * K + c] = S[r * LD + c];
        }
}

// ---------------------------------------------------------------------------
// out: per (chunk, value-head):  O = scale (Qd S0^T + P Nn)
// ---------------------------------------------------------------------------
template <typename InT, int K>
__global__ void __launch_bounds__(256) chunk_out_kernel(ChunkParams p) {
    constexpr int C = kChunk;
    constexpr int LD = K + 1;
    constexpr int V = K;
    extern __shared__ float sm[];
    float* Qs = sm;               // [C][LD]
    float* Hs = Qs + C * LD;      // [V][LD]
    float* Ns = Hs + V * LD;      // [C][LD]
    float* Ps = Ns + C * LD;      // [C][C+1]
    const int chunk = blockIdx.x;
    if (chunk >= p.meta[0]) return;
    const int h = blockIdx.y;
    const int4 info = p.table[chunk];
    const int start = info.y, L = info.z;
    const int tid = threadIdx.x;
    for (int e = tid; e < C * K; e += blockDim.x) {
        const int i = e / K, c = e % K;
        const size_t row = ((size_t)start + i) * p.Hv + h;
        Qs[i * LD + c] = i < L ? p.Qd[row * K + c] : 0.f;
        Ns[i * LD + c] = i < L ? p.Vn[row * V + c] : 0.f;
    }
    for (int e = tid; e < V * K; e += blockDim.x) {
        const int r = e / K, c = e % K;
        Hs[r * LD + c] = p.H[(((size_t)chunk * p.Hv + h) * V + r) * K + c];
    }
    for (int e = tid; e < C * C; e += blockDim.x) {
        const int i = e / C, j = e % C;
        Ps[i * (C + 1) + j] = p.P[(((size_t)chunk * p.Hv + h) * C + i) * C + j];
    }
    __syncthreads();
    InT* op = static_cast<InT*>(p.o);
    for (int e = tid; e < L * V; e += blockDim.x) {
        const int i = e / V, r = e % V;
        float acc = 0.f;
        for (int c = 0; c < K; ++c) acc = fmaf(Qs[i * LD + c], Hs[r * LD + c], acc);
        for (int j = 0; j <= i; ++j) acc = fmaf(Ps[i * (C + 1) + j], Ns[j * LD + r], acc);
        op[(((size_t)start + i) * p.Hv + h) * V + r] = from_f<InT>(p.scale * acc);
    }
}

template <typename InT, int K>
cudaError_t launch_chunk_t(const ChunkArgs& a, cudaStream_t stream) {
    constexpr int C = kChunk;
    constexpr int LD = K + 1;
    const ChunkWorkspace w = chunk_workspace_layout(a.N, a.T, a.Hk, a.Hv, a.K, a.V, a.gk ? 1 : 0, a.dtype, a.flags);
    char* ws = static_cast<char*>(a.workspace);
    ChunkParams p{};
    p.q = a.q; p.k = a.k; p.v = a.v; p.g = a.g; p.gk = a.gk; p.beta = a.beta;
    p.h0 = a.initial_state; p.o = a.o; p.hT = a.final_state; p.cu = a.cu_seqlens;
    p.meta = reinterpret_cast<int*>(ws + w.off_meta);
    p.offsets = reinterpret_cast<int*>(ws + w.off_offsets);
    p.table = reinterpret_cast<int4*>(ws + w.off_table);
    p.W = reinterpret_cast<float*>(ws + w.off_w);
    p.U = reinterpret_cast<float*>(ws + w.off_u);
    p.Kd = reinterpret_cast<float*>(ws + w.off_kd);
    p.Qd = reinterpret_cast<float*>(ws + w.off_qd);
    p.P = reinterpret_cast<float*>(ws + w.off_p);
    p.dL = reinterpret_cast<float*>(ws + w.off_dl);
    p.H = reinterpret_cast<float*>(ws + w.off_h);
    p.Vn = reinterpret_cast<float*>(ws + w.off_vn);
    p.Hk = a.Hk; p.Hv = a.Hv; p.scale = a.scale;

    if (!w.local_meta) {
        KernelTimer kt("chunk_meta", stream);
        chunk_meta_kernel<<<1, 1024, 0, stream>>>(a.cu_seqlens, a.N, a.T, reinterpret_cast<int*>(ws + w.off_meta),
                                                  reinterpret_cast<int*>(ws + w.off_offsets),
                                                  reinterpret_cast<int4*>(ws + w.off_table),
                                                  reinterpret_cast<int*>(ws + w.off_order), w.seg_chunks,
                                                  reinterpret_cast<int4*>(ws + w.off_segs),
                                                  reinterpret_cast<int*>(ws + w.off_segoff));
    }
    if (a.flags & 1) {
        const int64_t rows = a.T * a.Hk;
        const unsigned blocks = (unsigned)((rows + 7) / 8);
        InT* qn = reinterpret_cast<InT*>(ws + w.off_qn);
        InT* kn = reinterpret_cast<InT*>(ws + w.off_kn);
        KernelTimer kt("qk_l2norm", stream);
        l2norm_kernel<InT, K><<<blocks, 256, 0, stream>>>(static_cast<const InT*>(a.q), qn, rows);
        l2norm_kernel<InT, K><<<blocks, 256, 0, stream>>>(static_cast<const InT*>(a.k), kn, rows);
        p.q = qn;
        p.k = kn;
    }
    if constexpr (std::is_same<InT, __nv_bfloat16>::value) {
        return launch_chunk_tc(a, w, ws, p.q, p.k, stream);  // every bf16 shape is a tensor-core shape
    } else {
        const size_t sm_intra = sizeof(float) * (4 * C * LD + 2 * C * (C + 1) + C);
        cudaFuncSetAttribute(chunk_intra_kernel<InT, K>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_intra);
        {
            KernelTimer kt("chunk_intra", stream);
            chunk_intra_kernel<InT, K><<<dim3((unsigned)w.max_chunks, a.Hv), 256, sm_intra, stream>>>(p);
        }

        constexpr int BV = 32;
        const size_t sm_state = sizeof(float) * (BV * LD + 2 * C * LD + C * (BV + 1) + K);
        cudaFuncSetAttribute(chunk_state_kernel<K, BV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_state);
        {
            KernelTimer kt("chunk_state", stream);
            chunk_state_kernel<K, BV><<<dim3(a.N, a.Hv, a.V / BV), 256, sm_state, stream>>>(p);
        }

        const size_t sm_out = sizeof(float) * ((2 * C + K) * LD + C * (C + 1));
        cudaFuncSetAttribute(chunk_out_kernel<InT, K>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_out);
        {
            KernelTimer kt("chunk_out", stream);
            chunk_out_kernel<InT, K><<<dim3((unsigned)w.max_chunks, a.Hv), 256, sm_out, stream>>>(p);
        }
        return cudaGetLastError();
    }
}

}  // namespace

cudaError_t launch_chunk(const ChunkArgs& a, cudaStream_t stream) {
    if (a.dtype == 0) {
        if (a.K == 128) return launch_chunk_t<__nv_bfloat16, 128>(a, stream);
        return launch_chunk_t<__nv_bfloat16, 64>(a, stream);
    }
    if (a.K == 128) return launch_chunk_t<float, 128>(a, stream);
    return launch_chunk_t<float, 64>(a, stream);
}

}  // namespace gdr
