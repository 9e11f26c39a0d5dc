// Chunked prefill on the Blackwell tensor cores (bf16 inputs, K = V = 128, or 64 as zero-padded 128-channel tiles).
//
// Two kernels after the chunk metadata (three with the chunk-parallel scan):
//
//  prep  (persistent CTAs walking the (chunk, value-head) items, fully parallel)
//        gam = in-chunk cumsum of the gate; G = K K^T and Q K^T on tcgen05
//        (exact bf16 products, fp32 accumulation); A_ij = beta_i e^{gam_i-gam_j}
//        G_ij (j < i); Tm = (I + A)^{-1} by a blocked forward substitution in
//        fp32; W = Tm diag(beta e^{gam}) K and U = Tm diag(beta) V on tcgen05
//        with Tm split into bf16 hi + lo (K, V exact); the masked attention
//        P_ij = e^{gam_i-gam_j} (q_i . k_j) (j <= i), the decayed queries
//        e^{gam_i} q_i and the decay factors.  Results are written as
//        pre-swizzled operand images ("blobs") so the chain kernel stages them
//        with single 1-D bulk copies.
//        Per-key-channel gates (KDA) have a prep kernel of their own
//        (chunk_prep_kda_kernel, two 256-thread CTAs per SM): A and P from
//        products with the decays folded into both operands around a pivot on
//        tcgen05 (one pivot at the chunk's first token while no channel decays
//        by more than 2^64 over the chunk; otherwise pairs across the halves
//        of 2h-token blocks, each factor <= 1, and pairs inside 4-token blocks
//        on the CUDA cores), W = Tm diag(beta) (K o e^{Gam}) with a 3-term
//        split, and the decayed keys Kd = K o e^{gam_L - Gam} as hi/lo.
//
//  chain (one CTA per value-head x 32-column block of V x sequence, serial
//        over the sequence's chunks; attention-gym PR #344's inter-chunk state
//        recurrence with the output fused in):
//          N  = U - W S0^T            3-term split (W hi/lo x S hi/lo)
//          O  = Qd S0^T + P N         (output)
//          S  = e^{gam_L} S0 + K^T (f o N)     2-term split
//        All M = 128: W_hi and Qd are stacked into one A operand (so is W_lo
//        with P), so the product that forms N forms the output's Qd S0^T too.
//        Warp roles (512 threads): warp 0 stages chunk blobs with
//        cp.async.bulk into a two-deep ring; warp 2 owns the TMEM allocation;
//        warps 4-11 hold the fp32 state S^T (row k in TMEM lane k, 16 of the 32
//        columns per thread), turn the N accumulator into the split operands,
//        and one lane each of warps 4, 5 and 6 issues the tcgen05.mma groups as
//        soon as their operands are published (a single thread issues about
//        one MMA per 60 cycles, so the work is split three ways); warps 14 and
//        15 drain the output accumulator (double-buffered in TMEM) to bf16
//        rows of o.
//        With the chunk-parallel scan the chain runs per segment of G chunks:
//        a summary pass (the first segment of each sequence from h0 with its
//        output; the other segments from zero, their offsets B, and the middle
//        ones from the identity with U = 0, their transitions P), then
//        chunk_seg_scan_kernel composes the start states, then an output pass
//        runs every later segment from its start state.
//
// Every exponential is of gam_i - gam_j with i >= j or of gam_i, all <= 0:
// any finite gate <= 0 keeps every operand finite (cuLA PR #113 review).
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace gdr {
namespace {

constexpr int C = kChunk;  // 64
constexpr int D = 128;     // K = V
constexpr int BV = 32;     // value columns per chain CTA
constexpr int NVB = D / BV;
constexpr int LDA = C + 1;  // padded fp32 row stride for the 64 x 64 solve

// Blob sizes (bytes)
constexpr uint32_t kTile64x128 = C * D * 2;       // 16 KB bf16 [64][128]
constexpr uint32_t kTile64x64 = C * C * 2;        // 8 KB bf16 [64][64]
constexpr uint32_t kUBlock = C * BV * 4;          // 8 KB fp32 [64][32]
constexpr uint32_t kRec = 1024;                   // rowf[64], colf[128]
constexpr uint32_t kXwBytes = 2 * kTile64x128;    // 32 KB stacked [W_hi ; Qd]
constexpr uint32_t kYwBytes = 3 * C * 128;        // 24 KB stacked [W_lo ; P] without its last 8 KB

struct TcParams {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* gk;
    const void* beta;
    const float* h0;
    void* o;
    float* hT;
    const int32_t* cu;
    // chunk metadata: [0] chunk count, [1] 1 if cu_seqlens is well formed,
    // [2] segment count; per-sequence first chunk; chunk table; sequences by
    // decreasing length.  Written by the metadata kernel, or, with local_meta,
    // by CTA 0 of the prep kernel (which then forms its own item map and
    // leaves the table unwritten).
    int* meta;
    int* offsets;
    const int4* table;
    int* order;
    int local_meta;
    int64_t T;
    unsigned char* Xw;   // [chunk][Hv][32 KB]: k128 128 rows = [W_hi ; Qd]
    unsigned char* Ub;   // [chunk][Hv][NVB][8 KB]
    unsigned char* Yw;   // [chunk][Hv][24 KB]: k128 128 rows = [W_lo ; P] (column block 1: W_lo only)
    unsigned char* Kb;   // scalar gate: [chunk][Hk][16 KB]; channel gate: [chunk][Hv][2][16 KB]
    unsigned char* Rb;   // [chunk][Hv][1 KB]
    unsigned int* err;
    int N, Hk, Hv;
    float scale;
    // chunk-parallel scan: mode 0 = one chain CTA runs a whole sequence;
    // 1 = segment summaries: the first segment of a sequence from h0 with its
    // output (end state into Bs, or the final state), the others from zero
    // without output (offset into Bs) and, for the middle ones, from the
    // identity with U = 0 (transition into Mt); 2 = every later segment from
    // its scanned start state in Bs, with output
    int mode;
    const int4* segs;    // (sequence, first chunk in sequence, chunks, last?)
    const int* segoff;   // [N + 1] first segment of each sequence
    float* Mt;           // [segment][Hv][128][128]: Mt[m][k] = P[m][k]
    float* Bs;           // [segment][Hv][128 (v)][128 (k)]
};

__device__ __forceinline__ void raise_error(const TcParams& p, unsigned code) {
    atomicOr(p.err, code);
}

// ---------------------------------------------------------------------------
// Chunk metadata of a call with at most kLocalMetaSeqs sequences, formed by
// each prep CTA in shared memory instead of by the metadata kernel (one launch
// fewer ahead of the prep): cu_seqlens and the first chunk of every sequence.
// A malformed cu_seqlens (cu[0] != 0, a decreasing entry, cu[N] != T) gives
// no chunks.  CTA 0 also writes what the chain kernel reads: the chunk count
// and validity, the per-sequence first chunks and the longest-first order
// (ties by index).
// ---------------------------------------------------------------------------
struct LocalMeta {
    int total;  // chunks of the call (0: malformed cu_seqlens)
    int valid;  // cu_seqlens well formed
    int pad[2];
    int cu[kLocalMetaSeqs + 1];
    int off[kLocalMetaSeqs + 1];
};

template <int NT>
__device__ void local_meta_build(const TcParams& p, LocalMeta& m, int tid) {
    static_assert(NT > kLocalMetaSeqs, "one thread per cu_seqlens entry");
    if (tid <= p.N) m.cu[tid] = p.cu[tid];
    __syncthreads();
    if (tid == 0) {
        bool bad = m.cu[0] != 0 || (int64_t)m.cu[p.N] != p.T;
        int c = 0;
        for (int b = 0; b < p.N; ++b) {
            const int len = m.cu[b + 1] - m.cu[b];
            bad = bad || len < 0;
            m.off[b] = c;
            c += len > 0 ? (len + C - 1) / C : 0;
        }
        m.off[p.N] = c;
        m.total = bad ? 0 : c;
        m.valid = bad ? 0 : 1;
        if (blockIdx.x == 0) {
            p.meta[0] = m.total;
            p.meta[1] = bad ? 0 : 1;
            p.meta[2] = 0;
        }
    }
    __syncthreads();
    if (blockIdx.x == 0 && m.valid) {
        if (tid <= p.N) p.offsets[tid] = m.off[tid];
        if (tid < p.N) {
            const int lb = m.cu[tid + 1] - m.cu[tid];
            int rank = 0;
            for (int j = 0; j < p.N; ++j) {
                const int lj = m.cu[j + 1] - m.cu[j];
                rank += (lj > lb) || (lj == lb && j < tid);
            }
            p.order[rank] = tid;
        }
    }
}

// (first token, length) of chunk ci: from the chunk table, or with local
// metadata from the sequence found by binary search over the first chunks.
__device__ __forceinline__ int2 chunk_rows(const TcParams& p, const LocalMeta& m, int ci) {
    if (!p.local_meta) {
        const int4 e = p.table[ci];
        return make_int2(e.y, e.z);
    }
    int lo = 0, hi = p.N - 1;  // the last sequence whose first chunk is <= ci
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (m.off[mid] <= ci) lo = mid;
        else hi = mid - 1;
    }
    const int start = m.cu[lo] + (ci - m.off[lo]) * C;
    return make_int2(start, min(C, m.cu[lo + 1] - start));
}

// ---------------------------------------------------------------------------
// Inverse of a 64 x 64 unit-lower-triangular matrix (I + A), A strictly lower,
// fp32, 256 threads, by recursive doubling over 16 x 16 blocks:
//   1. the four diagonal blocks X_b = (I + A_bb)^{-1}, one column per thread,
//      right-looking (after x_m is final it is subtracted from every later
//      row, so the dependent chain is 16 steps long, not 120);
//   2. the 32 x 32 halves: T_{2p+1,2p} = -X_{2p+1} (A_{2p+1,2p} X_{2p});
//   3. the lower-left 32 x 32 block: T_10 = -B_1 (A_10 B_0) with B_0, B_1 the
//      two 32 x 32 inverses from step 2.
// Each product is one pass over shared memory with a small register tile per
// thread.  Every entry of Tm is written (zeros above the diagonal) and visible
// to every thread on return.  Z holds 1024 floats of scratch.  Threads from 256
// on only take part in the barriers.
// ---------------------------------------------------------------------------
template <int NT>
__device__ void solve_unit_lower(const float* __restrict__ A, float* __restrict__ Tm, float* __restrict__ Z,
                                 int tid) {
    static_assert(NT == 256 || NT == 512, "solve_unit_lower runs on 256 of 256 or 512 threads");
    const bool act = NT == 256 || tid < 256;
    if (tid < 64) {
        const int r0 = 16 * (tid >> 4), c = tid & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < 15; ++m) {
#pragma unroll
            for (int r = m + 1; r < 16; ++r) x[r] = fmaf(-A[(r0 + r) * LDA + r0 + m], x[m], x[r]);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Tm[(r0 + r) * LDA + r0 + c] = x[r];
    } else if (act) {
        // zeros in the six blocks above the block diagonal
        for (int e = tid - 64; e < 6 * 256; e += 192) {
            const int blk = e >> 8, r = (e >> 4) & 15, c = e & 15;
            const int bi = blk < 3 ? 0 : blk < 5 ? 1 : 2;
            const int bj = blk < 3 ? blk + 1 : blk < 5 ? blk - 1 : 3;
            Tm[(16 * bi + r) * LDA + 16 * bj + c] = 0.f;
        }
    }
    __syncthreads();
    // step 2: pair p = tid / 128; thread: row i, columns j0, j0 + 1 of a 16 x 16 block
    {
        const int p = (tid >> 7) & 1, e = tid & 127, i = e >> 3, j0 = 2 * (e & 7);
        const int r0 = 32 * p, r1 = r0 + 16;
        if (act) {
            float y0 = 0.f, y1 = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float a = A[(r1 + i) * LDA + r0 + m];
                y0 = fmaf(a, Tm[(r0 + m) * LDA + r0 + j0], y0);
                y1 = fmaf(a, Tm[(r0 + m) * LDA + r0 + j0 + 1], y1);
            }
            Z[p * 256 + i * 16 + j0] = y0;
            Z[p * 256 + i * 16 + j0 + 1] = y1;
        }
        __syncthreads();
        if (act) {
            float t0 = 0.f, t1 = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float x = Tm[(r1 + i) * LDA + r1 + m];
                t0 = fmaf(x, Z[p * 256 + m * 16 + j0], t0);
                t1 = fmaf(x, Z[p * 256 + m * 16 + j0 + 1], t1);
            }
            Tm[(r1 + i) * LDA + r0 + j0] = -t0;
            Tm[(r1 + i) * LDA + r0 + j0 + 1] = -t1;
        }
    }
    __syncthreads();
    // step 3: 2 x 2 tile per thread, rows 2 ti, 2 ti + 1 and columns 2 tj, 2 tj + 1
    {
        const int ti = (tid >> 4) & 15, tj = tid & 15, i0 = 2 * ti, j0 = 2 * tj;
        if (act) {
            float y00 = 0.f, y01 = 0.f, y10 = 0.f, y11 = 0.f;
#pragma unroll 8
            for (int m = 0; m < 32; ++m) {
                const float a0 = A[(32 + i0) * LDA + m], a1 = A[(33 + i0) * LDA + m];
                const float b0 = Tm[m * LDA + j0], b1 = Tm[m * LDA + j0 + 1];
                y00 = fmaf(a0, b0, y00);
                y01 = fmaf(a0, b1, y01);
                y10 = fmaf(a1, b0, y10);
                y11 = fmaf(a1, b1, y11);
            }
            Z[i0 * 32 + j0] = y00;
            Z[i0 * 32 + j0 + 1] = y01;
            Z[(i0 + 1) * 32 + j0] = y10;
            Z[(i0 + 1) * 32 + j0 + 1] = y11;
        }
        __syncthreads();
        if (act) {
            float t00 = 0.f, t01 = 0.f, t10 = 0.f, t11 = 0.f;
#pragma unroll 8
            for (int m = 0; m < 32; ++m) {
                const float x0 = Tm[(32 + i0) * LDA + 32 + m], x1 = Tm[(33 + i0) * LDA + 32 + m];
                const float z0 = Z[m * 32 + j0], z1 = Z[m * 32 + j0 + 1];
                t00 = fmaf(x0, z0, t00);
                t01 = fmaf(x0, z1, t01);
                t10 = fmaf(x1, z0, t10);
                t11 = fmaf(x1, z1, t11);
            }
            Tm[(32 + i0) * LDA + j0] = -t00;
            Tm[(32 + i0) * LDA + j0 + 1] = -t01;
            Tm[(33 + i0) * LDA + j0] = -t10;
            Tm[(33 + i0) * LDA + j0 + 1] = -t11;
        }
    }
    __syncthreads();  // Tm complete before any thread reads it
}

// The 8 per-channel values of one 16-byte operand chunk (channels 8 ch ..
// 8 ch + 7 of a row of fp32 gates) as two 16-byte shared loads: scalar loads
// at this 32-byte lane stride would hit each bank eight times over.
__device__ __forceinline__ void ld8(const float* p, float (&f)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// Stage 64 token rows [64][128] bf16 into rows [row0, row0 + 64) of a k128
// smem tile of `rows` rows, with cp.async (all 16-byte pieces in flight at
// once).  Rows >= L and the 16-byte pieces of a row beyond the first nch
// (channels >= 8 nch: a 64-channel head) are zero-filled.
template <int NT>
__device__ __forceinline__ void stage_rows_async(unsigned char* tile, int rows, int row0, const __nv_bfloat16* src,
                                                 size_t row_stride, int L, int nch, int tid) {
    for (int e = tid; e < C * 16; e += NT) {
        const int row = e >> 4, ch = e & 15;
        const bool ok = row < L && ch < nch;
        const __nv_bfloat16* g = src + (size_t)(row < L ? row : 0) * row_stride + (ch < nch ? ch : 0) * 8;
        const uint32_t dst = tc::smem_u32(tile + tc::chunk_k128(row0 + row, ch, rows));
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(g), "r"(ok ? 16 : 0)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// prep kernel (256 threads)
// ---------------------------------------------------------------------------
// Shared memory.  X stacks K (rows 0..63) and Q (rows 64..127) as one M = 128
// operand, so K K^T and Q K^T come from one group of MMAs.  Dead regions are
// reused: the Q rows of X hold T' hi / lo and the fp32 A matrix holds T'' hi /
// lo once the solve has finished.
// 256 threads, two CTAs per SM.
constexpr int kPrepThreads = 256;
constexpr uint32_t kXcb = 2 * C * 128;  // column-block stride of X (128 rows x 128 B)

struct PrepSmem {
    static constexpr uint32_t kX = 0;                         // [K; Q] 128 x 128 bf16 (32 KB)
    static constexpr uint32_t kV = kX + 2 * kTile64x128;      // V tile 64 x 128 (16 KB)
    static constexpr uint32_t kA = kV + kTile64x128;          // fp32 [64][65]
    static constexpr uint32_t kT1h = kX + C * 128;            // Q rows, column block 0
    static constexpr uint32_t kT1l = kX + kXcb + C * 128;     // Q rows, column block 1
    static constexpr uint32_t kT2h = kA;
    static constexpr uint32_t kT2l = kA + kTile64x64;
    static constexpr uint32_t kTm = (kA + C * LDA * 4 + 1023) & ~1023u;  // fp32 [64][65]
    static constexpr uint32_t kZ = kTm + C * LDA * 4;                   // fp32 [1024]
    static constexpr uint32_t kGam = (kZ + 4 * 256 * 4 + 1023) & ~1023u;  // fp32 [64] gate cumsum
    static constexpr uint32_t kBeta = kGam + C * 4;
    static constexpr uint32_t kBar = kBeta + C * 4;
    static constexpr uint32_t kMeta = kBar + 64;          // LocalMeta
    // W lo image staging (W hi is staged over Tm), so that the next item's K, Q
    // rows need not wait for the bulk copies of this item's images
    static constexpr uint32_t kWl = (kMeta + sizeof(LocalMeta) + 1023) & ~1023u;
    static constexpr uint32_t kTotal = kWl + kTile64x128 + 1024;  // + alignment slack
    static_assert(kT2l + kTile64x64 <= kTm, "T'' tiles overlap Tm");
    static_assert(kTile64x128 <= C * LDA * 4 && kTm % 1024 == 0, "W hi image over Tm");
    static_assert(kTotal <= 113 * 1024, "two CTAs per SM");
};

// Every kernel here takes the channel count of K and V in global memory as
// kDk (128, or 64).  The kernels always work on 128-channel tiles; with 64
// channels the upper half of every staged row is zero, so every product,
// image and state entry beyond channel 64 is zero, and the chain runs only
// the value blocks below 64.
template <int kDk>
__global__ void __launch_bounds__(kPrepThreads, 2) chunk_prep_kernel(TcParams p) {
    static_assert(kDk == 128 || kDk == 64, "K = V = 128 or 64");
    using S = PrepSmem;
    constexpr int NT = kPrepThreads;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // Persistent: CTA x takes items x, x + gridDim.x, ... (item = chunk * Hv + h)
    // and warms L2 with the next item's rows while it computes the current one.
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = warp & 3, hf = warp >> 2;  // TMEM lane quadrant, column half
    const int grp = p.Hv / p.Hk;
    const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(p.q);
    const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(p.k);
    const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(p.v);
    const __nv_bfloat16* bp = static_cast<const __nv_bfloat16*>(p.beta);

    float* As = reinterpret_cast<float*>(sm + S::kA);
    float* Tm = reinterpret_cast<float*>(sm + S::kTm);
    float* Z = reinterpret_cast<float*>(sm + S::kZ);
    float* gam = reinterpret_cast<float*>(sm + S::kGam);
    float* bet = reinterpret_cast<float*>(sm + S::kBeta);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S::kBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S::kBar + 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + S::kBar + 24);
    const uint32_t bar0 = tc::smem_u32(&bars[0]);
    const uint32_t barWU = tc::smem_u32(&bars[1]);  // W and U products: two issuers

    if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_slot), 256);
    if (tid == 0) {
        tc::mbar_init(bar0, 1);
        tc::mbar_init(barWU, 2);
        *abort_flag = 0;
        tc::mbar_fence_init();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    uint32_t ph0 = 0;  // parity of the next completion of bar0
    uint32_t phWU = 0;
    tc::grid_dep_wait();    // the chunk table comes from the metadata kernel
    tc::grid_dep_launch();  // the chain kernel may start its prologue on free SMs
    LocalMeta& lm = *reinterpret_cast<LocalMeta*>(sm + S::kMeta);
    if (p.local_meta) local_meta_build<NT>(p, lm, tid);
    const int nitems = (p.local_meta ? lm.total : p.meta[0]) * p.Hv;

    for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
        const int chunk = item / p.Hv, h = item - chunk * p.Hv;
        const int2 info = chunk_rows(p, lm, chunk);
        const int start = info.x, L = info.y;
        const int kh = h / grp;

        // ---- stage K, Q (as X) and V rows (cp.async), gates, beta -------------------
        stage_rows_async<NT>(sm + S::kX, 2 * C, 0, kp + ((size_t)start * p.Hk + kh) * kDk, (size_t)p.Hk * kDk, L,
                             kDk / 8, tid);
        stage_rows_async<NT>(sm + S::kX, 2 * C, C, qp + ((size_t)start * p.Hk + kh) * kDk, (size_t)p.Hk * kDk, L,
                             kDk / 8, tid);
        // the previous item's U image (over V and A; bulk group before its W image)
        if (tid == 0) tc::bulk_wait_read_1();
        __syncthreads();
        stage_rows_async<NT>(sm + S::kV, C, 0, vp + ((size_t)start * p.Hv + h) * kDk, (size_t)p.Hv * kDk, L,
                             kDk / 8, tid);
        asm volatile("cp.async.commit_group;" ::: "memory");
        {
            const int nxt = item + (int)gridDim.x;
            if (nxt < nitems) {
                const int nc = nxt / p.Hv, nh = nxt - nc * p.Hv;
                const int2 ni = chunk_rows(p, lm, nc);
                const int r = tid & 63, which = tid >> 6;
                const size_t tok = (size_t)ni.x + r;
                if (r < ni.y) {
                    if (which == 0) tc::prefetch_l2(kp + (tok * p.Hk + nh / grp) * kDk, kDk * 2);
                    else if (which == 1) tc::prefetch_l2(qp + (tok * p.Hk + nh / grp) * kDk, kDk * 2);
                    else if (which == 2) tc::prefetch_l2(vp + (tok * p.Hv + nh) * kDk, kDk * 2);
                }
                if (tid == 255) tc::prefetch_l2_span(p.g + (size_t)ni.x * p.Hv, (size_t)ni.y * p.Hv * 4);
                if (tid == 254) tc::prefetch_l2_span(bp + (size_t)ni.x * p.Hv, (size_t)ni.y * p.Hv * 2);
            }
        }
        if (tid < C) bet[tid] = tid < L ? to_f(bp[((size_t)start + tid) * p.Hv + h]) : 0.f;
        if (warp < 2) {
            // scalar gate: inclusive scan over 64 tokens with two warps
            float x = tid < L ? __ldg(p.g + ((size_t)start + tid) * p.Hv + h) : 0.f;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            gam[tid] = x;
        }
        __syncthreads();
        if (warp == 1) gam[tid] += gam[31];
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        tc::fence_proxy_async();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
        const uint32_t sX = tc::smem_u32(sm + S::kX), sV = tc::smem_u32(sm + S::kV);
        const float* gl = gam + (L - 1);

        // ---- [K K^T ; Q K^T] on the tensor cores (scalar gate), one M = 128 group ------
        if (tid == 0) {
            constexpr uint32_t id = tc::idesc_bf16(128, 64, false, false);
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t off = (ks >> 2) * kXcb + (ks & 3) * 32;
                tc::mma_bf16(tmem, tc::smem_desc(sX + off, 16, 1024, tc::kSwizzle128),
                             tc::smem_desc(sX + off, 16, 1024, tc::kSwizzle128), id, ks > 0);
            }
            tc::mma_commit(bar0);
        }
        __syncwarp();

        // ---- while that runs: Qd blob, K / Kd blob, decay record ------------------------
        {
            unsigned char* Qdst = p.Xw + ((size_t)chunk * p.Hv + h) * kXwBytes;  // rows 64..127
            for (int e = tid; e < C * 16; e += NT) {
                const int i = e >> 4, ch = e & 15;
                const uint4 raw = *reinterpret_cast<const uint4*>(sm + S::kX + tc::chunk_k128(C + i, ch, 2 * C));
                const __nv_bfloat16* qv = reinterpret_cast<const __nv_bfloat16*>(&raw);
                uint32_t w4[4];
                const float eg = __expf(gam[i]);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    w4[u] = tc::pack_bf16(__bfloat162float(qv[2 * u]) * eg, __bfloat162float(qv[2 * u + 1]) * eg);
                *reinterpret_cast<uint4*>(Qdst + tc::chunk_k128(C + i, ch, 2 * C)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
            if (h % grp == 0) {  // K rows of X, both column blocks -> a [64][128] k128 image
                unsigned char* Kdst = p.Kb + ((size_t)chunk * p.Hk + kh) * kTile64x128;
                for (int e = tid; e < (int)(kTile64x128 / 16); e += NT) {
                    const int cb = e >> 9, r = e & 511;
                    reinterpret_cast<uint4*>(Kdst)[e] = reinterpret_cast<const uint4*>(sm + S::kX + cb * kXcb)[r];
                }
            }
            float* rec = reinterpret_cast<float*>(p.Rb + ((size_t)chunk * p.Hv + h) * kRec);
            if (tid < C) rec[tid] = tid < L ? __expf(gl[0] - gam[tid]) : 0.f;
            if (tid < D) rec[64 + tid] = __expf(gl[0]);
        }

        // ---- A (strictly lower) and P (lower incl. diagonal) -------------------------
        unsigned char* Pdst = p.Yw + ((size_t)chunk * p.Hv + h) * kYwBytes;  // rows 64..127 of column block 0
        {
            if (!tc::mbar_wait(bar0, ph0, abort_flag)) { *abort_flag = 1; raise_error(p, 1u); }
            ph0 ^= 1u;
            tc::fence_after();
            // thread: accumulator row r = 32 q + lane (rows < 64: K K^T, >= 64: Q K^T),
            // columns [32 hf, 32 hf + 32)
            const int r = 32 * q + lane, i = r & 63;
            // all shared-memory reads first (gam, beta), then the arithmetic, then
            // the stores: As may alias gam as far as the compiler knows, and an
            // interleaved load / store order would serialise the 32 elements
            float gj[32];
#pragma unroll
            for (int jj = 0; jj < 32; jj += 4) {
                const float4 g4 = *reinterpret_cast<const float4*>(gam + 32 * hf + jj);
                gj[jj] = g4.x; gj[jj + 1] = g4.y; gj[jj + 2] = g4.z; gj[jj + 3] = g4.w;
            }
            const float gi = gam[i], bi = bet[i];
            float gv[32];
            tc::tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 32 * hf, gv);
            if (r < C) {
                const float sc = i < L ? bi : 0.f;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = 32 * hf + jj;
                    gv[jj] = j < i ? sc * __expf(gi - gj[jj]) * gv[jj] : 0.f;
                }
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) As[i * LDA + 32 * hf + jj] = gv[jj];
            } else {
                uint32_t pk[16];
                const float sc = i < L ? 1.f : 0.f;
#pragma unroll
                for (int jj = 0; jj < 32; jj += 2) {
                    const int j = 32 * hf + jj;
                    const float p0 = j <= i ? sc * __expf(gi - gj[jj]) * gv[jj] : 0.f;
                    const float p1 = j + 1 <= i ? sc * __expf(gi - gj[jj + 1]) * gv[jj + 1] : 0.f;
                    pk[jj >> 1] = tc::pack_bf16(p0, p1);
                }
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    *reinterpret_cast<uint4*>(Pdst + tc::chunk_k128(C + i, 4 * hf + cc, 2 * C)) =
                        make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
            }
        }
        if (tid == 0) tc::bulk_wait_read();  // the previous item's W images (over Tm and kWl)
        tc::fence_before();
        __syncthreads();

        // ---- Tm = (I + A)^{-1} -----------------------------------------------------------
        solve_unit_lower<NT>(As, Tm, Z, tid);

        // ---- split operands: T' = Tm diag(beta e^{gam}) (scalar gate) or Tm diag(beta);
        //      T'' = Tm diag(beta).  Written over the dead Q rows of X and the A matrix.
        for (int e = tid; e < C * 8; e += NT) {
            const int i = e >> 3, ch = e & 7;
            uint32_t h1[4], l1[4], h2[4], l2[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = ch * 8 + 2 * u;
                const float t0 = Tm[i * LDA + j] * bet[j], t1 = Tm[i * LDA + j + 1] * bet[j + 1];
                tc::split2(t0 * __expf(gam[j]), t1 * __expf(gam[j + 1]), h1[u], l1[u]);
                tc::split2(t0, t1, h2[u], l2[u]);
            }
            const uint32_t off = tc::chunk_k128(i, ch, C);
            *reinterpret_cast<uint4*>(sm + S::kT1h + off) = make_uint4(h1[0], h1[1], h1[2], h1[3]);
            *reinterpret_cast<uint4*>(sm + S::kT1l + off) = make_uint4(l1[0], l1[1], l1[2], l1[3]);
            *reinterpret_cast<uint4*>(sm + S::kT2h + off) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
            *reinterpret_cast<uint4*>(sm + S::kT2l + off) = make_uint4(l2[0], l2[1], l2[2], l2[3]);
        }
        tc::fence_proxy_async();
        __syncthreads();

        // ---- W = T' K (lane 0 of warp 0), U = T'' V (lane 0 of warp 1) ----------------------
        if (warp < 2 && lane == 0) {
            tc::fence_after();
            constexpr uint32_t id = tc::idesc_bf16(64, 128, false, true);
            const uint32_t t1h = tc::smem_u32(sm + S::kT1h), t1l = tc::smem_u32(sm + S::kT1l);
            const uint32_t t2h = tc::smem_u32(sm + S::kT2h), t2l = tc::smem_u32(sm + S::kT2l);
            // B operands read MN-major: K rows of X (atom stride kXcb), V / Kg (atom stride 8 KB)
            auto mm = [&](uint32_t dcol, uint32_t a, uint32_t b, uint32_t atom, bool first) {
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tmem + dcol, tc::smem_desc(a + ks * 32, 16, 1024, tc::kSwizzle128),
                                 tc::smem_desc(b + ks * 2048, atom, 1024, tc::kSwizzle128), id, (first && ks == 0) ? 0u : 1u);
            };
            if (warp == 0) {
                mm(0, t1h, sX, kXcb, true);
                mm(0, t1l, sX, kXcb, false);
            } else {
                mm(128, t2h, sV, C * 128, true);
                mm(128, t2l, sV, C * 128, false);
            }
            tc::mma_commit(barWU);
        }
        __syncwarp();

        // ---- W, U out of TMEM into their blobs: row i = 16 q + lane (lane < 16);
        //      warp: columns [64 hf, 64 hf + 64) of W and of U.  The images are staged in
        //      shared memory left dead by the finished MMAs (W hi / lo as 64-row k128
        //      tiles over Tm and in their own region, U value-major over V and A) and
        //      written with bulk copies, so every global write is a contiguous run: U's
        //      first, then W's.  The next item stages its K and Q rows at once, waits
        //      for U's copy before its V rows and for W's before its solve. ------------
        if (!tc::mbar_wait(barWU, phWU, abort_flag)) { *abort_flag = 1; raise_error(p, 1u); }
        phWU ^= 1u;
        tc::fence_after();
        {
            const int i = 16 * q + (lane & 15);
            const uint32_t lrow = tmem + ((uint32_t)(32 * q) << 16);
            unsigned char* sWh = sm + S::kTm;           // [64][128] k128, column-block stride 8 KB
            unsigned char* sWl = sm + S::kWl;
            float* sU = reinterpret_cast<float*>(sm + S::kV);  // 4 x [32 v][64 i]
            constexpr int kBlocks = 2;  // 32-column blocks of W and of U per warp
            for (int q2 = 0; q2 < kBlocks; ++q2) {
                const int cb = kBlocks * hf + q2;  // 32-column block of W and of U
                float wv[32], uv[32];
                tc::tmem_ld32(lrow + 32 * cb, wv);
                tc::tmem_ld32(lrow + 128 + 32 * cb, uv);
                if (lane < 16) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t hw[4], lw[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) tc::split2(wv[8 * cc + 2 * u], wv[8 * cc + 2 * u + 1], hw[u], lw[u]);
                        const uint32_t off = tc::chunk_k128(i, 4 * cb + cc, C);
                        *reinterpret_cast<uint4*>(sWh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        *reinterpret_cast<uint4*>(sWl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    }
                    // U block cb value-major [32 v][64 i]: the chain's thread for row i
                    // then reads a conflict-free column of shared memory
                    float* ublk = sU + cb * (C * BV) + i;
#pragma unroll
                    for (int v = 0; v < BV; ++v) ublk[v * C] = uv[v];
                }
            }
            tc::fence_proxy_async();
            __syncthreads();
            if (tid == 0) {
                unsigned char* Xd = p.Xw + ((size_t)chunk * p.Hv + h) * kXwBytes;  // rows 0..63 of each column block
                unsigned char* Yd = p.Yw + ((size_t)chunk * p.Hv + h) * kYwBytes;
                const uint32_t half = kTile64x128 / 2;  // one 64-row column block
                tc::bulk_s2g(p.Ub + ((size_t)chunk * p.Hv + h) * NVB * kUBlock, tc::smem_u32(sU), NVB * kUBlock);
                tc::bulk_commit();
                tc::bulk_s2g(Xd, tc::smem_u32(sWh), half);
                tc::bulk_s2g(Xd + 2 * half, tc::smem_u32(sWh) + half, half);
                tc::bulk_s2g(Yd, tc::smem_u32(sWl), half);
                tc::bulk_s2g(Yd + 2 * half, tc::smem_u32(sWl) + half, half);
                tc::bulk_commit();
            }
        }
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
    }  // item loop
    if (tid == 0) tc::bulk_wait_all();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
// prep kernel with per-key-channel gates (KDA): 256 threads, two CTAs per SM
// ---------------------------------------------------------------------------
// The same outputs as the scalar-gate prep (W_hi / Qd, W_lo / P, U, the decayed
// keys Kd as hi / lo, the decay record), for gates gk [T, Hv, K].
//   * The in-chunk cumsum is kept in log2 units, Gam2 = log2(e) Gam, so every
//     decay factor is one ex2 of a difference that is <= 0.
//   * Thread (t0 = tid / 8, g = tid % 8) owns tokens t0 and t0 + 32 and, of
//     each, the 16-byte operand chunks g and g + 8 (channels 8g .. 8g + 7 and
//     64 + 8g .. 64 + 8g + 7).  It holds their Gam2 in registers for the whole
//     item; only the rows of the pivots (tokens 4, 8, ..., 60), of the first
//     and of the last token stay in shared memory.
//   * A_ij = beta_i sum_c k_i[c] k_j[c] e^{Gam_i[c] - Gam_j[c]} (j < i) and
//     P_ij = sum_c q_i[c] k_j[c] e^{Gam_i[c] - Gam_j[c]} (j <= i).  While no
//     channel decays by more than 2^64 over the chunk (every chunk of slowly
//     decaying gates), one pivot at the first token serves every pair:
//     e^{Gam_i - Gam_j} = e^{Gam_i - Gam_0} e^{Gam_0 - Gam_j}, the left factor
//     <= 1 and the right one >= 1, both inside [2^-64, 2^64], so each stays in
//     the normal range and its hi / lo split keeps its relative accuracy.
//     One stacked product [K L hi ; Q L hi] [K R hi | K R lo] (N = 128) and
//     one K L lo x K R hi (N = 64) then give all of A and P.  Otherwise, pairs
//     in different halves of a block of 2h tokens (h = 32, 16, 8, 4) go through
//     the tensor cores around the pivot p = first token of the upper half:
//     e^{Gam_i - Gam_j} = e^{Gam_i - Gam_p} e^{Gam_p - Gam_j}, both factors <= 1,
//     folded into the left (k_i, q_i) and right (k_j) operands.  A takes three
//     split products (K_l hi x R hi, K_l hi x R lo, K_l lo x R hi; fp32
//     accuracy for the solve), P two (Q_l hi x R hi + Q_l hi x R lo: P is
//     stored in bf16 and only feeds the output).  Each level's accumulators
//     alternate between two TMEM column sets, so the read-out of one level
//     runs while the next level's products are in flight.  Pairs inside a
//     4-token block are formed on the CUDA cores (a warp takes two blocks, a
//     lane one block and 8 channels).
//   * W = Tm diag(beta) (K o e^{Gam}) with a 3-term split, U = Tm diag(beta) V
//     with a 2-term split, as for the scalar gate.
// Shared memory stays under 113 KB, so two CTAs share an SM and one CTA's
// waits (tensor-core round trips, barriers) are filled by the other's work.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The two bf16 of a packed word as fp32 (element 0 in the low half).
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// a - b on the fp32x2 pipe
__device__ __forceinline__ float2 sub2(float2 a, float2 b) { return __ffma2_rn(b, make_float2(-1.f, -1.f), a); }
// x = hi + lo with hi = bf16(x), lo = bf16(x - hi), two values at once
__device__ __forceinline__ void split2x(float2 x, uint32_t& hi, uint32_t& lo) {
    hi = tc::pack_bf16(x.x, x.y);
    const float2 l = sub2(x, unpack_bf16x2(hi));
    lo = tc::pack_bf16(l.x, l.y);
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kKdaThreads = 256;
constexpr float kSinglePivotSpan2 = 64.f;  // log2 units: factors within [2^-64, 2^64]

struct KdaSmem {
    static constexpr uint32_t kX = 0;                         // [K ; Q] 128 x 128 bf16 (32 KB)
    static constexpr uint32_t kOps = 2 * kTile64x128;         // 40 KB work region
    static constexpr uint32_t kLh = kOps;                     // [K_l hi ; Q_l hi] 64 x 128 (16 KB)
    static constexpr uint32_t kLl = kLh + kTile64x128;        // K_l lo 32 x 128 (8 KB)
    static constexpr uint32_t kRh = kLl + kTile64x128 / 2;    // R hi 32 x 128
    static constexpr uint32_t kRl = kRh + kTile64x128 / 2;    // R lo 32 x 128
    static constexpr uint32_t kOpsEnd = kRl + kTile64x128 / 2;
    static constexpr uint32_t kGt = kOps;                     // fp32 [64][128] Gam2 scratch (cumsum, 4-token pairs)
    static constexpr uint32_t kTm = kOps;                     // fp32 [64][65] after the A / P products
    static constexpr uint32_t kZ = kTm + C * LDA * 4;         // fp32 [1024]
    static constexpr uint32_t kV = kOps + 24576;              // V 64 x 128 (16 KB), loaded after the products
    static constexpr uint32_t kA = kOpsEnd;                   // fp32 [64][65]
    static constexpr uint32_t kT2h = kA, kT2l = kA + kTile64x64;  // T'' hi / lo over A after the solve
    static constexpr uint32_t kP = (kA + C * LDA * 4 + 1023) & ~1023u;  // P bf16 64 x 64 (8 KB)
    static constexpr uint32_t kPiv = kP + kTile64x64;         // fp32 [16][128]: Gam2 of tokens 4, 8, .., 60 and L - 1
    static constexpr uint32_t kBeta = kPiv + 16 * D * 4;
    static constexpr uint32_t kBar = kBeta + C * 4;
    static constexpr uint32_t kMeta = kBar + 64;              // LocalMeta
    static constexpr uint32_t kG0 = (kMeta + sizeof(LocalMeta) + 15) & ~15u;  // fp32 [128]: Gam2 of token 0
    static constexpr uint32_t kTotal = kG0 + D * 4 + 1024;    // + alignment slack
    // single-pivot operands: [K L hi ; Q L hi] over A (column block 0) and P + pivot rows
    // (column block 1), [K R hi ; K R lo] over the work region, K L lo over the work
    // region's tail (column block 0) and the query rows of X (column block 1)
    static constexpr uint32_t kSgA1 = kP;
    static constexpr uint32_t kSgB = kOps;
    static constexpr uint32_t kSgLl0 = kOps + 2 * kTile64x128;
    static constexpr uint32_t kSgLl1 = kX + C * 128;
    static_assert(kTile64x128 <= C * LDA * 4, "A column block 0 (128 rows x 128 B) in the A region");
    static_assert(kSgA1 + kTile64x128 == kBeta, "A column block 1 over P and the pivot rows");
    static_assert(kSgB + 2 * kTile64x128 == kSgLl0, "B column blocks ahead of K L lo");
    static_assert(kSgLl0 + kTile64x128 / 2 == kOpsEnd, "K L lo column block 0 at the work region's tail");
    static_assert((kA | kSgA1 | kSgB | kSgLl0 | kSgLl1) % 1024 == 0, "128-byte swizzled tiles on 1 KB boundaries");
    static_assert(kGt + C * D * 4 <= kOpsEnd, "Gam2 scratch beyond the work region");
    static_assert(kZ + 4096 <= kV, "Z overlaps V");
    static_assert(kV + kTile64x128 == kOpsEnd, "V at the end of the work region");
    static_assert(kT2l + kTile64x64 <= kA + C * LDA * 4, "T'' beyond A");
    static_assert(kTotal <= 113 * 1024, "two CTAs per SM");
};

template <int kDk>
__global__ void __launch_bounds__(kKdaThreads, 2) chunk_prep_kda_kernel(TcParams p) {
    static_assert(kDk == 128 || kDk == 64, "K = V = 128 or 64");
    using S = KdaSmem;
    constexpr int NT = kKdaThreads;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = tid >> 3, g = tid & 7;  // tokens t0, t0 + 32; operand chunks g, g + 8
    const int grp = p.Hv / p.Hk;
    const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(p.q);
    const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(p.k);
    const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(p.v);
    const __nv_bfloat16* bp = static_cast<const __nv_bfloat16*>(p.beta);

    float* As = reinterpret_cast<float*>(sm + S::kA);
    float* Tm = reinterpret_cast<float*>(sm + S::kTm);
    float* Z = reinterpret_cast<float*>(sm + S::kZ);
    float* gt = reinterpret_cast<float*>(sm + S::kGt);
    float* piv = reinterpret_cast<float*>(sm + S::kPiv);
    float* g0 = reinterpret_cast<float*>(sm + S::kG0);
    float* bet = reinterpret_cast<float*>(sm + S::kBeta);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S::kBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S::kBar + 24);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + S::kBar + 32);
    const uint32_t barL[2] = {tc::smem_u32(&bars[0]), tc::smem_u32(&bars[1])};
    const uint32_t barW = tc::smem_u32(&bars[2]);

    if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_slot), 256);
    if (tid == 0) {
        tc::mbar_init(barL[0], 3);
        tc::mbar_init(barL[1], 3);
        tc::mbar_init(barW, 2);
        *abort_flag = 0;
        tc::mbar_fence_init();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    uint32_t phW = 0;
    tc::grid_dep_wait();    // the chunk table comes from the metadata kernel
    tc::grid_dep_launch();  // the chain kernel may start its prologue on free SMs
    LocalMeta& lm = *reinterpret_cast<LocalMeta*>(sm + S::kMeta);
    if (p.local_meta) local_meta_build<NT>(p, lm, tid);
    const int nitems = (p.local_meta ? lm.total : p.meta[0]) * p.Hv;
    const uint32_t sX = tc::smem_u32(sm + S::kX);

    for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
        const int chunk = item / p.Hv, h = item - chunk * p.Hv;
        const int2 info = chunk_rows(p, lm, chunk);
        const int start = info.x, L = info.y;
        const int kh = h / grp;

        // ---- stage K, Q rows and the gate rows (cp.async); zero A and P; beta; warm L2
        //      for the next item ----------------------------------------------------------
        stage_rows_async<NT>(sm + S::kX, 2 * C, 0, kp + ((size_t)start * p.Hk + kh) * kDk, (size_t)p.Hk * kDk, L,
                             kDk / 8, tid);
        stage_rows_async<NT>(sm + S::kX, 2 * C, C, qp + ((size_t)start * p.Hk + kh) * kDk, (size_t)p.Hk * kDk, L,
                             kDk / 8, tid);
        // the previous item's U image (bulk group before its W image) sits in the scratch
        if (tid == 0) tc::bulk_wait_read_1();
        __syncthreads();
        {
            // gk rows [64][128] fp32 into the scratch (rows >= L and channels
            // >= dk zero-filled: a zero log-decay on a zero channel)
            const float* src = p.gk + ((size_t)start * p.Hv + h) * kDk;
            for (int e = tid; e < C * (D / 4); e += NT) {
                const int row = e >> 5, pc = e & 31;
                const bool ok = row < L && 4 * pc < kDk;
                const float* gsrc = src + (size_t)(row < L ? row : 0) * p.Hv * kDk + (4 * pc < kDk ? 4 * pc : 0);
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                             :: "r"(tc::smem_u32(gt + row * D + 4 * pc)), "l"(gsrc), "r"(ok ? 16 : 0) : "memory");
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        {
            const int nxt = item + (int)gridDim.x;
            if (nxt < nitems) {
                const int nc = nxt / p.Hv, nh = nxt - nc * p.Hv;
                const int2 ni = chunk_rows(p, lm, nc);
                const int r = tid & 63, which = tid >> 6;
                const size_t tok = (size_t)ni.x + r;
                if (r < ni.y) {
                    if (which == 0) tc::prefetch_l2(kp + (tok * p.Hk + nh / grp) * kDk, kDk * 2);
                    else if (which == 1) tc::prefetch_l2(qp + (tok * p.Hk + nh / grp) * kDk, kDk * 2);
                    else if (which == 2) tc::prefetch_l2(vp + (tok * p.Hv + nh) * kDk, kDk * 2);
                    else tc::prefetch_l2(p.gk + (tok * p.Hv + nh) * kDk, kDk * 4);
                }
                if (tid == 0) tc::prefetch_l2_span(bp + (size_t)ni.x * p.Hv, (size_t)ni.y * p.Hv * 2);
            }
        }
        // (A needs no clearing: the solve reads its strict lower triangle, all of
        // which the products write)
        if (tid < C) bet[tid] = tid < L ? to_f(bp[((size_t)start + tid) * p.Hv + h]) : 0.f;
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        if (tid == 0) tc::bulk_wait_read();  // the previous item's W image (over A, P and the pivot rows)
        __syncthreads();

        // ---- per-channel cumsum in place, log2 units: thread (channel c, half hf) scans
        //      32 tokens ----------------------------------------------------------------
        {
            const int c = tid & (D - 1), hf = tid >> 7;
            float x[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) x[u] = gt[(32 * hf + u) * D + c];
#pragma unroll
            for (int u = 1; u < 32; ++u) x[u] += x[u - 1];
            if (hf == 0) piv[c] = x[31];  // the first half's total, read by the second half
            __syncthreads();
            const float off = hf ? piv[c] : 0.f;
#pragma unroll
            for (int u = 0; u < 32; ++u) gt[(32 * hf + u) * D + c] = (x[u] + off) * kLog2e;
        }
        __syncthreads();
        // One pivot at the chunk's first token serves every pair while no channel
        // decays by more than 2^kSinglePivotSpan2 over the chunk: the factors
        // e^{Gam_i - Gam_0} <= 1 and e^{Gam_0 - Gam_j} >= 1 then stay well inside the
        // normal range, and each is split hi / lo relative to its own size.
        const bool single = __syncthreads_and(tid >= D || gt[tid] - gt[(L - 1) * D + tid] <= kSinglePivotSpan2) != 0;
        // pivot rows (tokens 4, 8, .., 60; the pivot levels only) and the last token's
        // row; token 0's row; this thread's Gam2
        for (int e = single ? 15 * D + tid : tid; e < 16 * D; e += NT) {
            const int r = e >> 7, tok = r < 15 ? 4 * (r + 1) : L - 1;
            piv[e] = gt[tok * D + (e & (D - 1))];
        }
        if (tid < D) g0[tid] = gt[tid];
        float G[2][16];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const float* src = gt + (t0 + 32 * u) * D + 8 * (g + 8 * cc);
                const float4 a = *reinterpret_cast<const float4*>(src), b = *reinterpret_cast<const float4*>(src + 4);
                G[u][8 * cc + 0] = a.x; G[u][8 * cc + 1] = a.y; G[u][8 * cc + 2] = a.z; G[u][8 * cc + 3] = a.w;
                G[u][8 * cc + 4] = b.x; G[u][8 * cc + 5] = b.y; G[u][8 * cc + 6] = b.z; G[u][8 * cc + 7] = b.w;
            }
        __syncthreads();

        // ---- Qd = Q o e^{Gam} and Kd = K o e^{Gam_L - Gam} (hi / lo) straight to their blobs ----
        {
            unsigned char* Qdst = p.Xw + ((size_t)chunk * p.Hv + h) * kXwBytes;
            unsigned char* Kdst = p.Kb + ((size_t)chunk * p.Hv + h) * 2 * kTile64x128;
            const float* gL = piv + 15 * D;
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int t = t0 + 32 * u, ch = g + 8 * cc;
                    const uint4 qr = *reinterpret_cast<const uint4*>(sm + S::kX + tc::chunk_k128(C + t, ch, 2 * C));
                    const uint4 kr = *reinterpret_cast<const uint4*>(sm + S::kX + tc::chunk_k128(t, ch, 2 * C));
                    const __nv_bfloat16* qv = reinterpret_cast<const __nv_bfloat16*>(&qr);
                    const __nv_bfloat16* kv = reinterpret_cast<const __nv_bfloat16*>(&kr);
                    float l8[8];
                    ld8(gL + 8 * ch, l8);
                    uint32_t qw[4], hw[4], lw[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float* gg = &G[u][8 * cc + 2 * e];
                        qw[e] = tc::pack_bf16(__bfloat162float(qv[2 * e]) * ex2(gg[0]),
                                              __bfloat162float(qv[2 * e + 1]) * ex2(gg[1]));
                        tc::split2(__bfloat162float(kv[2 * e]) * ex2(l8[2 * e] - gg[0]),
                                   __bfloat162float(kv[2 * e + 1]) * ex2(l8[2 * e + 1] - gg[1]), hw[e], lw[e]);
                    }
                    *reinterpret_cast<uint4*>(Qdst + tc::chunk_k128(C + t, ch, 2 * C)) = make_uint4(qw[0], qw[1], qw[2], qw[3]);
                    const uint32_t off = tc::chunk_k128(t, ch, C);
                    *reinterpret_cast<uint4*>(Kdst + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4*>(Kdst + kTile64x128 + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            float* rec = reinterpret_cast<float*>(p.Rb + ((size_t)chunk * p.Hv + h) * kRec);
            if (tid < C) rec[tid] = tid < L ? 1.f : 0.f;
            if (tid < D) rec[64 + tid] = ex2(gL[tid]);
        }

        // ---- A and P across the halves of 2h-token blocks (h = 32, 16, 8, 4) on tcgen05 ----
        constexpr uint32_t idL = tc::idesc_bf16(64, 32, false, false);
        // build level lev's operands: this thread's tokens are left (upper half) or
        // right (lower half) of their block; the 4 tokens of a warp always agree
        auto build = [&](int lev) {
            const int sh = 5 - lev, hh = 1 << sh;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = t0 + 32 * u;
                const int B = t >> (sh + 1), up = (t >> sh) & 1, pv = (2 * B + 1) << sh;
                const int idx = (B << sh) + (t & (hh - 1));
                const float* gp = piv + ((pv >> 2) - 1) * D;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int ch = g + 8 * cc;
                    float p8[8];
                    ld8(gp + 8 * ch, p8);
                    float2 f[4];
                    if (up) {  // e^{Gam_t - Gam_p}, t >= p
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 d = sub2(make_float2(G[u][8 * cc + 2 * e], G[u][8 * cc + 2 * e + 1]),
                                                  make_float2(p8[2 * e], p8[2 * e + 1]));
                            f[e] = make_float2(ex2(d.x), ex2(d.y));
                        }
                    } else {  // e^{Gam_p - Gam_t}, t < p
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 d = sub2(make_float2(p8[2 * e], p8[2 * e + 1]),
                                                  make_float2(G[u][8 * cc + 2 * e], G[u][8 * cc + 2 * e + 1]));
                            f[e] = make_float2(ex2(d.x), ex2(d.y));
                        }
                    }
                    const uint4 kr = *reinterpret_cast<const uint4*>(sm + S::kX + tc::chunk_k128(t, ch, 2 * C));
                    const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w};
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) split2x(__fmul2_rn(unpack_bf16x2(kw[e]), f[e]), hw[e], lw[e]);
                    if (up) {
                        *reinterpret_cast<uint4*>(sm + S::kLh + tc::chunk_k128(idx, ch, C)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        *reinterpret_cast<uint4*>(sm + S::kLl + tc::chunk_k128(idx, ch, 32)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                        const uint4 qr = *reinterpret_cast<const uint4*>(sm + S::kX + tc::chunk_k128(C + t, ch, 2 * C));
                        const uint32_t qw4[4] = {qr.x, qr.y, qr.z, qr.w};
                        uint32_t qw[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 x = __fmul2_rn(unpack_bf16x2(qw4[e]), f[e]);
                            qw[e] = tc::pack_bf16(x.x, x.y);
                        }
                        *reinterpret_cast<uint4*>(sm + S::kLh + tc::chunk_k128(32 + idx, ch, C)) = make_uint4(qw[0], qw[1], qw[2], qw[3]);
                    } else {
                        const uint32_t off = tc::chunk_k128(idx, ch, 32);
                        *reinterpret_cast<uint4*>(sm + S::kRh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        *reinterpret_cast<uint4*>(sm + S::kRl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    }
                }
            }
            tc::fence_proxy_async();
            tc::fence_before();
            __syncthreads();
            tc::fence_after();
        };
        // three issuers, one split product each, into columns 96 (lev % 2) + 32 w.
        // K_l lo is a 32-row tile: the M = 64 product also reads the 32 rows after
        // it (real memory), which land in accumulator rows that are not read.
        auto issue = [&](int lev) {
            // issuers: warps 3, 1 and 4, which skip the read-outs of levels 1..3
            const int role = warp == 3 ? 0 : warp == 1 ? 1 : warp == 4 ? 2 : -1;
            if (role >= 0 && lane == 0) {
                const uint32_t la = tc::smem_u32(sm + (role == 2 ? S::kLl : S::kLh));
                const uint32_t astr = role == 2 ? 32 * 128 : C * 128;
                const uint32_t rb = tc::smem_u32(sm + (role == 1 ? S::kRl : S::kRh));
                const uint32_t d = tmem + 96 * (lev & 1) + 32 * role;
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_bf16(d, tc::smem_desc(la + (ks >> 2) * astr + (ks & 3) * 32, 16, 1024, tc::kSwizzle128),
                                 tc::smem_desc(rb + (ks >> 2) * (32 * 128) + (ks & 3) * 32, 16, 1024, tc::kSwizzle128),
                                 idL, ks > 0);
                tc::mma_commit(barL[lev & 1]);
            }
            __syncwarp();
        };
        // level lev's accumulator: row r = 16 (w % 4) + lane (lane < 16), rows 0..31 A
        // (left token keys), 32..63 P (left token queries); warps w and w + 4 take
        // the right columns n < 16 and n >= 16.  Column n pairs with row r when both
        // fall in the same block of 2h tokens.
        auto wait_level = [&](int lev) {
            if (!tc::mbar_wait(barL[lev & 1], (lev >> 1) & 1, abort_flag)) { *abort_flag = 1; raise_error(p, 1u); }
            tc::fence_after();
        };
        auto readout = [&](int lev) {
            const int sh = 5 - lev, hh = 1 << sh;
            const int q = warp & 3, nh = warp >> 2;
            // below h = 32 a warp's rows (one half of the left tokens) pair only
            // with the right columns of one half: the other warp of the quadrant
            // has nothing to read
            if (hh < 32 && (q & 1) != nh) return;
            const uint32_t a = tmem + ((uint32_t)(32 * q) << 16) + 96 * (lev & 1) + 16 * nh;
            float d[48];
            tc::tmem_ld16x3(a, a + 32, a + 64, d);
            const int r = 16 * q + lane, idx = r & 31, B = idx >> sh;
            const int i = (2 * B + 1) * hh + (idx & (hh - 1));
            if (lane < 16) {
                if (q < 2) {
                    const float bi = bet[i];
#pragma unroll
                    for (int n2 = 0; n2 < 16; ++n2) {
                        const int n = 16 * nh + n2;
                        if ((n >> sh) == B) As[i * LDA + 2 * hh * B + (n & (hh - 1))] = bi * (d[n2] + d[16 + n2] + d[32 + n2]);
                    }
                } else {
#pragma unroll
                    for (int n2 = 0; n2 < 16; ++n2) {
                        const int n = 16 * nh + n2;
                        if ((n >> sh) == B)
                            *reinterpret_cast<__nv_bfloat16*>(sm + S::kP + tc::off_k128(i, 2 * hh * B + (n & (hh - 1)), C)) =
                                __float2bfloat16_rn(d[n2] + d[16 + n2]);
                    }
                }
            }
        };
        if (!single) {
            // P entries above the diagonal are never written on this path
            for (int e = tid; e < (int)(kTile64x64 / 16); e += NT)
                reinterpret_cast<uint4*>(sm + S::kP)[e] = make_uint4(0u, 0u, 0u, 0u);
            build(0);
            issue(0);
            wait_level(0);
            build(1);
            issue(1);
            readout(0);
            wait_level(1);
            build(2);
            issue(2);
            readout(1);
            wait_level(2);
            build(3);
            issue(3);
            readout(2);
            wait_level(3);
            readout(3);

            // ---- pairs inside a 4-token block: warp w has the blocks at tokens 4w and
            //      4w + 32.  Lane (u, o): block u, channels 8o .. 8o + 7; it forms the 6
            //      pairs i > j (A and P) and the 4 diagonal P entries over its 8 channels,
            //      and the 16 partial sums are reduced over the 16 lanes of the block
            //      (transposed, so lane o ends with sum o). --------------------------------
            {
    #pragma unroll
                for (int u = 0; u < 2; ++u)
    #pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        float* dst = gt + (t0 + 32 * u) * D + 8 * (g + 8 * cc);
                        *reinterpret_cast<float4*>(dst) = make_float4(G[u][8 * cc], G[u][8 * cc + 1], G[u][8 * cc + 2], G[u][8 * cc + 3]);
                        *reinterpret_cast<float4*>(dst + 4) = make_float4(G[u][8 * cc + 4], G[u][8 * cc + 5], G[u][8 * cc + 6], G[u][8 * cc + 7]);
                    }
                __syncwarp();
                const int o = lane & 15, tb = 4 * warp + 32 * (lane >> 4);
                float v[16];
                {
                    uint4 kr[4], qr[4];
    #pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        kr[a] = *reinterpret_cast<const uint4*>(sm + S::kX + tc::chunk_k128(tb + a, o, 2 * C));
                        qr[a] = *reinterpret_cast<const uint4*>(sm + S::kX + tc::chunk_k128(C + tb + a, o, 2 * C));
                    }
                    // diagonal: P_aa = q_a . k_a
    #pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        const __nv_bfloat16* kv = reinterpret_cast<const __nv_bfloat16*>(&kr[a]);
                        const __nv_bfloat16* qv = reinterpret_cast<const __nv_bfloat16*>(&qr[a]);
                        float acc = 0.f;
    #pragma unroll
                        for (int e = 0; e < 8; ++e) acc = fmaf(__bfloat162float(qv[e]), __bfloat162float(kv[e]), acc);
                        v[12 + a] = acc;
                    }
                    // pairs (1,0) (2,0) (3,0) (2,1) (3,1) (3,2): A in v[0..5], P in v[6..11]
    #pragma unroll
                    for (int m = 0; m < 6; ++m) {
                        const int i = m < 3 ? m + 1 : (m < 5 ? m - 1 : 3), j = m < 3 ? 0 : (m < 5 ? 1 : 2);
                        float gi[8], gj[8];
                        ld8(gt + (tb + i) * D + 8 * o, gi);
                        ld8(gt + (tb + j) * D + 8 * o, gj);
                        const __nv_bfloat16* ki = reinterpret_cast<const __nv_bfloat16*>(&kr[i]);
                        const __nv_bfloat16* qi = reinterpret_cast<const __nv_bfloat16*>(&qr[i]);
                        const __nv_bfloat16* kj = reinterpret_cast<const __nv_bfloat16*>(&kr[j]);
                        float sa = 0.f, sp = 0.f;
    #pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float kd = __bfloat162float(kj[e]) * ex2(gi[e] - gj[e]);
                            sa = fmaf(__bfloat162float(ki[e]), kd, sa);
                            sp = fmaf(__bfloat162float(qi[e]), kd, sp);
                        }
                        v[m] = sa;
                        v[6 + m] = sp;
                    }
                }
                // transposed reduction over the 16 lanes of the block: lane o ends with sum o
    #pragma unroll
                for (int k = 8; k >= 1; k >>= 1) {
                    const bool upper = (lane & k) != 0;
    #pragma unroll
                    for (int e = 0; e < k; ++e) {
                        const float send = upper ? v[e] : v[e + k];
                        const float keep = upper ? v[e + k] : v[e];
                        v[e] = keep + __shfl_xor_sync(0xffffffffu, send, k);
                    }
                }
                {
                    const int m = o < 6 ? o : (o < 12 ? o - 6 : 0);
                    const int i = tb + (o >= 12 ? o - 12 : (m < 3 ? m + 1 : (m < 5 ? m - 1 : 3)));
                    const int j = o >= 12 ? i : tb + (m < 3 ? 0 : (m < 5 ? 1 : 2));
                    if (o < 6) As[i * LDA + j] = bet[i] * v[0];
                    else *reinterpret_cast<__nv_bfloat16*>(sm + S::kP + tc::off_k128(i, j, C)) = __float2bfloat16_rn(v[0]);
                }
            }
        } else {
            // ---- one pivot at the chunk's first token: every pair from one stacked product.
            //      Left L_i = e^{Gam_i - Gam_0} <= 1: [K L hi ; Q L hi] (128 rows) and K L lo;
            //      right R_j = e^{Gam_0 - Gam_j} >= 1: [K R hi ; K R lo] (128 rows).
            //      A_ij = beta_i (KL_hi KR_hi + KL_hi KR_lo + KL_lo KR_hi)_ij for j < i and
            //      P_ij = (QL_hi KR_hi + QL_hi KR_lo)_ij for j <= i. ----------------------------
            __syncthreads();  // the key images have read the pivot rows, which the operands overwrite
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = t0 + 32 * u;
                // cc = 0 first: its query chunk is where cc = 1 puts K L lo (same thread, same address)
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int ch = g + 8 * cc, c8 = ch & 7;
                    float z8[8];
                    ld8(g0 + 8 * ch, z8);
                    const uint4 kr = *reinterpret_cast<const uint4*>(sm + S::kX + tc::chunk_k128(t, ch, 2 * C));
                    const uint4 qr = *reinterpret_cast<const uint4*>(sm + S::kX + tc::chunk_k128(C + t, ch, 2 * C));
                    const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w}, qw4[4] = {qr.x, qr.y, qr.z, qr.w};
                    uint32_t lh[4], ll[4], rh[4], rl[4], qh[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 d = sub2(make_float2(G[u][8 * cc + 2 * e], G[u][8 * cc + 2 * e + 1]),
                                              make_float2(z8[2 * e], z8[2 * e + 1]));  // Gam_t - Gam_0 <= 0
                        const float2 fl = make_float2(ex2(d.x), ex2(d.y));
                        const float2 fr = make_float2(ex2(-d.x), ex2(-d.y));
                        const float2 kf = unpack_bf16x2(kw[e]);
                        split2x(__fmul2_rn(kf, fl), lh[e], ll[e]);
                        split2x(__fmul2_rn(kf, fr), rh[e], rl[e]);
                        const float2 x = __fmul2_rn(unpack_bf16x2(qw4[e]), fl);
                        qh[e] = tc::pack_bf16(x.x, x.y);
                    }
                    unsigned char* a_blk = sm + (cc ? S::kSgA1 : S::kA);
                    unsigned char* b_blk = sm + S::kSgB + cc * kTile64x128;
                    unsigned char* l_blk = sm + (cc ? S::kSgLl1 : S::kSgLl0);
                    *reinterpret_cast<uint4*>(a_blk + tc::chunk_k128(t, c8, 2 * C)) = make_uint4(lh[0], lh[1], lh[2], lh[3]);
                    *reinterpret_cast<uint4*>(a_blk + tc::chunk_k128(C + t, c8, 2 * C)) = make_uint4(qh[0], qh[1], qh[2], qh[3]);
                    *reinterpret_cast<uint4*>(b_blk + tc::chunk_k128(t, c8, 2 * C)) = make_uint4(rh[0], rh[1], rh[2], rh[3]);
                    *reinterpret_cast<uint4*>(b_blk + tc::chunk_k128(C + t, c8, 2 * C)) = make_uint4(rl[0], rl[1], rl[2], rl[3]);
                    *reinterpret_cast<uint4*>(l_blk + tc::chunk_k128(t, c8, C)) = make_uint4(ll[0], ll[1], ll[2], ll[3]);
                }
            }
            tc::fence_proxy_async();
            tc::fence_before();
            __syncthreads();
            tc::fence_after();
            // [K L hi ; Q L hi] [K R hi | K R lo] (N = 128) into columns 0..127 (lane 0 of
            // warp 3); [K L lo ; -] K R hi (N = 64) into columns 128..191 (lane 0 of warp 1).
            // The K L lo operand reads 128 rows: rows 64..127 are the tiles after it (real
            // memory) and land in accumulator rows that are not read.
            if (lane == 0 && (warp == 3 || warp == 1)) {
                const bool lo = warp == 1;
                const uint32_t idS = lo ? tc::idesc_bf16(128, 64, false, false) : tc::idesc_bf16(128, 128, false, false);
                const uint32_t d = tmem + (lo ? 128 : 0);
                const uint32_t a0 = tc::smem_u32(sm + (lo ? S::kSgLl0 : S::kA));
                const uint32_t a1 = tc::smem_u32(sm + (lo ? S::kSgLl1 : S::kSgA1));
                const uint32_t b0 = tc::smem_u32(sm + S::kSgB);
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kin = (ks & 3) * 32;
                    tc::mma_bf16(d, tc::smem_desc(((ks >> 2) ? a1 : a0) + kin, 16, 1024, tc::kSwizzle128),
                                 tc::smem_desc(b0 + (ks >> 2) * kTile64x128 + kin, 16, 1024, tc::kSwizzle128), idS,
                                 ks > 0);
                }
                tc::mma_commit(barW);
            }
            __syncwarp();
            if (!tc::mbar_wait(barW, phW, abort_flag)) { *abort_flag = 1; raise_error(p, 1u); }
            phW ^= 1u;
            tc::fence_after();
            // read-out: TMEM lane r = accumulator row r (rows 0..63 A, 64..127 P); warps w and
            // w + 4 take the columns j < 32 and j >= 32
            {
                const int q = warp & 3, nh = warp >> 2;
                const int i = 32 * (q & 1) + lane;
                const float bi = bet[i];
#pragma unroll
                for (int hh2 = 0; hh2 < 2; ++hh2) {
                    const int j0 = 32 * nh + 16 * hh2;
                    const uint32_t a = tmem + ((uint32_t)(32 * q) << 16) + j0;
                    float d[48];
                    tc::tmem_ld16x3(a, a + 64, a + 128, d);
                    if (q < 2) {
#pragma unroll
                        for (int n2 = 0; n2 < 16; ++n2)
                            if (j0 + n2 < i) As[i * LDA + j0 + n2] = bi * (d[n2] + d[16 + n2] + d[32 + n2]);
                    } else {
#pragma unroll
                        for (int n2 = 0; n2 < 16; n2 += 2) {
                            const int j = j0 + n2;
                            const float p0 = j <= i ? d[n2] + d[16 + n2] : 0.f;
                            const float p1 = j + 1 <= i ? d[n2 + 1] + d[17 + n2] : 0.f;
                            *reinterpret_cast<uint32_t*>(sm + S::kP + tc::off_k128(i, j, C)) = tc::pack_bf16(p0, p1);
                        }
                    }
                }
            }
        }
        tc::fence_proxy_async();  // P is read by a bulk copy
        __syncthreads();

        // ---- P to its blob; K o e^{Gam} as hi / lo over X (hi over the dead Q rows, lo
        //      in place), the gates read back from the scratch ------------------------------
        if (tid == 0) {
            unsigned char* Pd = p.Yw + ((size_t)chunk * p.Hv + h) * kYwBytes + kTile64x64;  // rows 64..127 of column block 0
            tc::bulk_s2g(Pd, tc::smem_u32(sm + S::kP), kTile64x64);
            tc::bulk_commit();
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int t = t0 + 32 * u, ch = g + 8 * cc;
                const uint32_t off = tc::chunk_k128(t, ch, 2 * C);
                const uint4 kr = *reinterpret_cast<const uint4*>(sm + S::kX + off);
                const __nv_bfloat16* kv = reinterpret_cast<const __nv_bfloat16*>(&kr);
                float g8[8];
                if (single) {  // the scratch holds the right operand now; this thread's Gam2 is in G
#pragma unroll
                    for (int e = 0; e < 8; ++e) g8[e] = G[u][8 * cc + e];
                } else {
                    ld8(gt + t * D + 8 * ch, g8);
                }
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    tc::split2(__bfloat162float(kv[2 * e]) * ex2(g8[2 * e]), __bfloat162float(kv[2 * e + 1]) * ex2(g8[2 * e + 1]),
                               hw[e], lw[e]);
                *reinterpret_cast<uint4*>(sm + S::kX + tc::chunk_k128(C + t, ch, 2 * C)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(sm + S::kX + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
        __syncthreads();
        // V rows (cp.async) over the dead scratch, waited for after the solve
        stage_rows_async<NT>(sm + S::kV, C, 0, vp + ((size_t)start * p.Hv + h) * kDk, (size_t)p.Hv * kDk, L,
                             kDk / 8, tid);
        asm volatile("cp.async.commit_group;" ::: "memory");

        // ---- Tm = (I + A)^{-1}; T'' = Tm diag(beta) as hi / lo over A ---------------
        solve_unit_lower<NT>(As, Tm, Z, tid);
        for (int e = tid; e < C * 8; e += NT) {
            const int i = e >> 3, ch = e & 7;
            uint32_t h2[4], l2[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = ch * 8 + 2 * u;
                tc::split2(Tm[i * LDA + j] * bet[j], Tm[i * LDA + j + 1] * bet[j + 1], h2[u], l2[u]);
            }
            const uint32_t off = tc::chunk_k128(i, ch, C);
            *reinterpret_cast<uint4*>(sm + S::kT2h + off) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
            *reinterpret_cast<uint4*>(sm + S::kT2l + off) = make_uint4(l2[0], l2[1], l2[2], l2[3]);
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        if (tid == 0) tc::bulk_wait_read();  // the P image, whose tile the W image staging reuses
        tc::fence_proxy_async();
        __syncthreads();

        // ---- W = T'' (K o e^Gam) (3 terms, lane 0 of warp 0), U = T'' V (2 terms, lane 0
        //      of warp 1) ------------------------------------------------------------------
        if (warp < 2 && lane == 0) {
            tc::fence_after();
            constexpr uint32_t id = tc::idesc_bf16(64, 128, false, true);
            const uint32_t t2h = tc::smem_u32(sm + S::kT2h), t2l = tc::smem_u32(sm + S::kT2l);
            const uint32_t kgh = sX + C * 128, kgl = sX, sV = tc::smem_u32(sm + S::kV);
            auto mm = [&](uint32_t dcol, uint32_t a, uint32_t b, uint32_t atom, bool first) {
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_bf16(tmem + dcol, tc::smem_desc(a + ks * 32, 16, 1024, tc::kSwizzle128),
                                 tc::smem_desc(b + ks * 2048, atom, 1024, tc::kSwizzle128), id, (first && ks == 0) ? 0u : 1u);
            };
            if (warp == 0) {
                mm(0, t2h, kgh, kXcb, true);
                mm(0, t2h, kgl, kXcb, false);
                mm(0, t2l, kgh, kXcb, false);
            } else {
                mm(128, t2h, sV, C * 128, true);
                mm(128, t2l, sV, C * 128, false);
            }
            tc::mma_commit(barW);
        }
        __syncwarp();
        if (!tc::mbar_wait(barW, phW, abort_flag)) { *abort_flag = 1; raise_error(p, 1u); }
        phW ^= 1u;
        tc::fence_after();
        // ---- W, U out of TMEM (row i = 16 q + lane, lane < 16; warp: two 32-column
        //      blocks of W and of U), staged as blob images (W hi over A, W lo over P
        //      and the pivot rows, U over the work region) and written with bulk
        //      copies: U's first, then W's.  The next item waits for U's to have read
        //      the work region before its gate rows land there, and for W's before
        //      its cumsum; its K and Q rows go into X at once. -----------------------
        {
            const int q = warp & 3, hf = warp >> 2;
            const int i = 16 * q + (lane & 15);
            const uint32_t lrow = tmem + ((uint32_t)(32 * q) << 16);
            unsigned char* sWh = sm + S::kA;
            unsigned char* sWl = sm + S::kP;
            float* sU = reinterpret_cast<float*>(sm + S::kOps);
            for (int q2 = 0; q2 < 2; ++q2) {
                const int cb = 2 * hf + q2;
                float wv[32], uv[32];
                tc::tmem_ld32(lrow + 32 * cb, wv);
                tc::tmem_ld32(lrow + 128 + 32 * cb, uv);
                if (lane < 16) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t hw[4], lw[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) tc::split2(wv[8 * cc + 2 * u], wv[8 * cc + 2 * u + 1], hw[u], lw[u]);
                        const uint32_t off = tc::chunk_k128(i, 4 * cb + cc, C);
                        *reinterpret_cast<uint4*>(sWh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        *reinterpret_cast<uint4*>(sWl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    }
                    float* ublk = sU + cb * (C * BV) + i;
#pragma unroll
                    for (int v = 0; v < BV; ++v) ublk[v * C] = uv[v];
                }
            }
            tc::fence_proxy_async();
            __syncthreads();
            if (tid == 0) {
                unsigned char* Xd = p.Xw + ((size_t)chunk * p.Hv + h) * kXwBytes;
                unsigned char* Yd = p.Yw + ((size_t)chunk * p.Hv + h) * kYwBytes;
                const uint32_t half = kTile64x128 / 2;
                tc::bulk_s2g(p.Ub + ((size_t)chunk * p.Hv + h) * NVB * kUBlock, tc::smem_u32(sU), NVB * kUBlock);
                tc::bulk_commit();
                tc::bulk_s2g(Xd, tc::smem_u32(sWh), half);
                tc::bulk_s2g(Xd + 2 * half, tc::smem_u32(sWh) + half, half);
                tc::bulk_s2g(Yd, tc::smem_u32(sWl), half);
                tc::bulk_s2g(Yd + 2 * half, tc::smem_u32(sWl) + half, half);
                tc::bulk_commit();
            }
        }
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
    }  // item loop
    if (tid == 0) tc::bulk_wait_all();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
// chain kernel
// ---------------------------------------------------------------------------
template <bool kKDA>
struct ChainSmem {
    static constexpr uint32_t kKtBytes = kKDA ? 2 * kTile64x128 : kTile64x128;
    // one pipeline stage
    static constexpr uint32_t kXW = 0;                     // [W_hi ; Qd]   k128, 128 rows (32 KB)
    static constexpr uint32_t kYW = kXW + kXwBytes;        // [W_lo ; P | U] k128, 128 rows (32 KB)
    static constexpr uint32_t kU = kYW + kYwBytes;         // U fp32 [64][32] in the last 8 KB of YW
    static constexpr uint32_t kKt = kYW + 2 * kTile64x128;
    static constexpr uint32_t kRec_ = kKt + kKtBytes;
    static constexpr uint32_t kStage = kRec_ + kRec;
    static constexpr uint32_t kStageTx = kStage;  // bytes landed per stage
    // resident tiles
    static constexpr uint32_t kSh = 2 * kStage;              // S^T hi [128][32] mn64
    static constexpr uint32_t kSl = kSh + D * BV * 2;        // S^T lo (the next atom: [S_hi | S_lo])
    static constexpr uint32_t kNh = kSl + D * BV * 2;        // N' hi [64][32] mn64
    static constexpr uint32_t kNl = kNh + C * BV * 2;        // N' lo
    // N (bf16) for the output: two buffers by chunk parity with a scalar gate;
    // with per-channel gates the row factor is 1, so the output reads N'_hi
    static constexpr int kNBuf = kKDA ? 0 : 2;
    static constexpr uint32_t kN = kNl + C * BV * 2;
    static constexpr uint32_t kBar = kN + kNBuf * C * BV * 2;
    static constexpr uint32_t kTotal = kBar + 256 + 1024;
    static_assert(kTotal <= 232448, "chain shared memory above the 227 KB opt-in limit");
};

enum ChainBar {
    kFull0 = 0, kFull1, kEmpty0, kEmpty1, kD1Full, kD2Full, kOFull0, kOFull1, kOFree0, kOFree1,
    kDrainA, kDrainB, kDrainC, kSPub0, kSPub1, kNPub0, kNPub1, kNumBars
};
// pairs indexed by chunk (or stage) parity: the second of each is the first + 1
static_assert(kFull1 == kFull0 + 1 && kEmpty1 == kEmpty0 + 1 && kOFull1 == kOFull0 + 1 && kOFree1 == kOFree0 + 1 &&
                  kSPub1 == kSPub0 + 1 && kNPub1 == kNPub0 + 1,
              "barrier pairs indexed by parity must be adjacent");
static_assert(8 * kNumBars + 16 <= 256, "barriers, TMEM slot and abort flag fit the 256-byte barrier area");
// Arrival counts: the N accumulator is committed by issuers A and B, a stage is
// released by all three issuers, everything else by one arrival.
__device__ __forceinline__ uint32_t chain_bar_count(int i) {
    return i == kD1Full ? 2u : (i == kEmpty0 || i == kEmpty1) ? 3u : 1u;
}

template <bool kKDA, int kDk>
__global__ void __launch_bounds__(512, 1) chunk_chain_kernel(TcParams p) {
    static_assert(kDk == 128 || kDk == 64, "K = V = 128 or 64");
    using S = ChainSmem<kKDA>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S::kBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S::kBar + 8 * kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + S::kBar + 8 * kNumBars + 8);
    auto bar = [&](int i) { return tc::smem_u32(&bars[i]); };

    // prologue (touches no memory the earlier kernels write), then wait for them
    if (warp == 2) tc::tmem_alloc(tc::smem_u32(tmem_slot), 256);
    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) tc::mbar_init(bar(i), chain_bar_count(i));
        *abort_flag = 0;
        tc::mbar_fence_init();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    tc::grid_dep_wait();
    if (!p.meta[1]) {  // malformed cu_seqlens
        tc::fence_before();
        __syncthreads();
        if (warp == 2) tc::tmem_dealloc(tmem, 256);
        return;
    }
    // Work unit: a whole sequence (mode 0) or one segment of G chunks of it
    // (modes 1 and 2; the summary pass runs two CTA sets, the transition from
    // the identity with U = 0 and the offset from zero).
    // value blocks of the head that carry data: 4, or 2 for a 64-channel head
    // (the operand images keep 4 U blocks per (chunk, head) either way)
    constexpr int nvb = kDk / BV;
    const int hx = blockIdx.x % (p.Hv * nvb);
    const bool transition = p.mode == 1 && blockIdx.x >= p.Hv * nvb;
    const int h = hx / nvb, vb = hx % nvb, v0 = vb * BV;
    int b, nc, c0, cs0 = 0, sg = 0;
    bool last = true;
    if (p.mode == 0) {
        b = p.order[blockIdx.y];
        nc = (p.cu[b + 1] - p.cu[b] + C - 1) / C;
        c0 = p.offsets[b];
    } else {
        sg = blockIdx.y;
        bool idle = sg >= p.meta[2];  // beyond this call's segment count
        if (!idle) {
            const int4 e = p.segs[sg];
            b = e.x; cs0 = e.y; nc = e.z; last = e.w != 0;
            c0 = p.offsets[b] + cs0;
            // the first segment of a sequence runs from h0 in the summary pass
            // (the true chain: output and end state); no transition is formed for
            // it or for the last one, and the output pass skips it
            idle = p.mode == 1 ? (transition && (cs0 == 0 || last)) : cs0 == 0;
        }
        if (idle) {
            tc::fence_before();
            __syncthreads();
            if (warp == 2) tc::tmem_dealloc(tmem, 256);
            return;
        }
    }
    const bool first = cs0 == 0;
    const bool outputs = p.mode != 1 || first;  // transitions are never first
    const int bos = p.cu[b] + cs0 * C, eos = p.cu[b + 1];
    const int kh = h / (p.Hv / p.Hk);
    // Accumulators (fp32 TMEM columns).  The hi and lo split terms of the state
    // (or of N') sit side by side along N, so one N = 64 MMA forms two split
    // products; columns v and 32 + v are summed when read.
    //   D1[2] (M=128, 64 columns, double-buffered): rows 0..63 = W_hi S^T (part
    //         of the N accumulator), rows 64..127 = Qd S^T + P N (the output)
    //   D1b   (M=128, 32 columns): rows 0..63 = W_lo S_hi^T
    //   D2    (M=128, 64 columns): K^T [N'_hi | N'_lo]
    const uint32_t tD1 = tmem, tD1b = tmem + 128, tD2 = tmem + 192;
    const uint32_t base = tc::smem_u32(sm);
    auto fail = [&]() {
        *abort_flag = 1;
        raise_error(p, 2u);
    };

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            for (int c = 0; c < nc && !*abort_flag; ++c) {
                const int s = c & 1;
                if (c >= 2 && !tc::mbar_wait(bar(kEmpty0 + s), ((c >> 1) - 1) & 1, abort_flag)) { fail(); break; }
                const size_t gc = (size_t)c0 + c;
                const uint32_t st = base + s * S::kStage;
                const uint32_t fb = bar(kFull0 + s);
                tc::mbar_arrive_tx(fb, S::kStageTx);
                tc::bulk_g2s(st + S::kXW, p.Xw + (gc * p.Hv + h) * kXwBytes, kXwBytes, fb);
                tc::bulk_g2s(st + S::kYW, p.Yw + (gc * p.Hv + h) * kYwBytes, kYwBytes, fb);
                tc::bulk_g2s(st + S::kU, p.Ub + ((gc * p.Hv + h) * NVB + vb) * kUBlock, kUBlock, fb);
                if (kKDA) tc::bulk_g2s(st + S::kKt, p.Kb + (gc * p.Hv + h) * 2 * kTile64x128, 2 * kTile64x128, fb);
                else tc::bulk_g2s(st + S::kKt, p.Kb + (gc * p.Hk + kh) * kTile64x128, kTile64x128, fb);
                tc::bulk_g2s(st + S::kRec_, p.Rb + (gc * p.Hv + h) * kRec, kRec, fb);
                if (c + 2 < nc) {  // warm L2 with the blobs of chunk c + 2
                    const size_t g2 = gc + 2;
                    tc::prefetch_l2(p.Xw + (g2 * p.Hv + h) * kXwBytes, kXwBytes);
                    tc::prefetch_l2(p.Yw + (g2 * p.Hv + h) * kYwBytes, kYwBytes);
                    tc::prefetch_l2(p.Ub + ((g2 * p.Hv + h) * NVB + vb) * kUBlock, kUBlock);
                    if (kKDA) tc::prefetch_l2(p.Kb + (g2 * p.Hv + h) * 2 * kTile64x128, 2 * kTile64x128);
                    else tc::prefetch_l2(p.Kb + (g2 * p.Hk + kh) * kTile64x128, kTile64x128);
                    tc::prefetch_l2(p.Rb + (g2 * p.Hv + h) * kRec, kRec);
                }
            }
            // drain: wait for the copies of the last (up to) two stages to land
            for (int c = (nc > 2 ? nc - 2 : 0); c < nc; ++c)
                tc::mbar_wait_copies(bar(kFull0 + (c & 1)), (c >> 1) & 1);
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------ state group ------------------------------
        // Eight warps: warp w owns TMEM lane quadrant w % 4 (rows k of S^T) and
        // the 16-column half hf of the block's 32 value columns; the N
        // accumulator rows 0..63 sit in quadrants 0 and 1.  After each named
        // barrier that publishes operand tiles, one lane of warps 4, 5 and 6
        // issues the MMAs that read them (a single thread issues about one
        // tcgen05.mma per 60 cycles, so the work is split):
        //   A (warp 4): D1 = [W_hi ; Qd] [S_hi | S_lo], later D2 = K^T [N'_hi | N'_lo]
        //   B (warp 5): D1b = [W_lo ; P] S_hi
        //   C (warp 6): D1 rows 64..127 += P N (after N is published)
        // Rows of a stacked operand that a product does not need land in
        // accumulator rows nobody reads (or that are dead at that time).
        // Descriptors are built once per tile; a k-step adds its byte offset / 16
        // to the start-address field (tiles sit below 256 KB, so no carry).
        const int q = warp & 3, hf = (warp - 4) >> 2;
        const int t = 32 * q + lane;            // TMEM lane = row k of S^T
        const bool isA = warp == 4 && lane == 0, isB = warp == 5 && lane == 0, isC = warp == 6 && lane == 0;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const bool nrow = q < 2;                // owns row i = t of the N accumulator
        const int i = t;
        const int vh = 16 * hf;                 // first column of this thread's half
        const uint32_t idA = tc::idesc_bf16(128, 2 * BV, false, true);   // [W_hi;Qd] [S_hi|S_lo]
        const uint32_t idB = tc::idesc_bf16(128, BV, false, true);       // [W_lo;P] S_hi, [.;P] N
        const uint32_t id2w = tc::idesc_bf16(128, 2 * BV, true, true);   // K^T [N'_hi|N'_lo]
        const uint32_t id2n = tc::idesc_bf16(128, BV, true, true);       // Kd_lo^T N'_hi
        auto dk128 = [](uint32_t a) { return tc::smem_desc(a, 16, 1024, tc::kSwizzle128); };
        auto dmn128 = [](uint32_t a) { return tc::smem_desc(a, C * 128, 1024, tc::kSwizzle128); };
        auto dmn64 = [](uint32_t a, uint32_t atom) { return tc::smem_desc(a, atom, 512, tc::kSwizzle64); };
        constexpr uint32_t a128[8] = {0, 2, 4, 6, (2 * C * 128) >> 4, ((2 * C * 128) >> 4) + 2,
                                      ((2 * C * 128) >> 4) + 4, ((2 * C * 128) >> 4) + 6};  // 128-row k128, K = 128
        constexpr uint32_t a64[4] = {0, 2, 4, 6};                  // 128-row k128, K = 64 (column block 0)
        constexpr uint32_t amn[4] = {0, 128, 256, 384};            // MN-major A: 2 x 8-row groups per step
        float Sreg[16];
        if (p.mode == 2) {  // scanned start state of the segment
#pragma unroll
            for (int v = 0; v < 16; ++v) Sreg[v] = p.Bs[(((size_t)sg * p.Hv + h) * D + v0 + vh + v) * D + t];
        } else if (transition) {  // identity: column v0 + vh + v of I
#pragma unroll
            for (int v = 0; v < 16; ++v) Sreg[v] = (v0 + vh + v == t) ? 1.f : 0.f;
        } else if (p.h0 && first) {
#pragma unroll
            for (int v = 0; v < 16; ++v)
                Sreg[v] = t < kDk ? p.h0[(((size_t)b * p.Hv + h) * kDk + v0 + vh + v) * kDk + t] : 0.f;
        } else {
#pragma unroll
            for (int v = 0; v < 16; ++v) Sreg[v] = 0.f;
        }
        unsigned char* sSh = sm + S::kSh;
        unsigned char* sSl = sm + S::kSl;
        bool issued = false;
        bool staged = false;  // this chunk's stage was seen landed during the last update product
        bool drained = false;  // (issuer A) this chunk's output buffer was seen drained then too
        for (int c = 0; c < nc; ++c) {
            const int s = c & 1, ob = c & 1;
            const unsigned char* stg = sm + s * S::kStage;
            const uint32_t st = base + s * S::kStage;
            if (!staged && !tc::mbar_wait(bar(kFull0 + s), (c >> 1) & 1, abort_flag)) fail();  // keep going: every named barrier is reached by all threads
            // S^T rows (hi, lo) into the MMA operand tiles.  Their readers (the N
            // products of chunk c - 1) finished before the last state update.
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) split2x(make_float2(Sreg[8 * cc + 2 * u], Sreg[8 * cc + 2 * u + 1]), hw[u], lw[u]);
                const uint32_t off = tc::chunk_mn64(t, 2 * hf + cc);
                *reinterpret_cast<uint4*>(sSh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(sSl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            tc::fence_proxy_async();
            tc::fence_before();
            tc::bar_sync(1, 256);
            if (!kKDA && tid == 128) tc::mbar_arrive(bar(kSPub0 + s));  // S published: the output warps may drain chunk c - 1
            if (isA) {
                // the output rows of D1[ob] were drained (chunk c - 2) before reuse
                if (c >= 2 && !drained && !tc::mbar_wait(bar(kOFree0 + ob), ((c >> 1) - 1) & 1, abort_flag)) fail();
                tc::fence_after();
                tc::mma_ksteps<8>(tD1 + 64 * ob, dk128(st + S::kXW), a128, dmn64(base + S::kSh, D * BV * 2), 64, idA, true);
                tc::mma_commit(bar(kD1Full));
                issued = true;
            } else if (isB) {
                // rows 64..127 of the second column block are not part of the blob;
                // the accumulator rows they reach are not read
                tc::fence_after();
                tc::mma_ksteps<8>(tD1b, dk128(st + S::kYW), a128, dmn64(base + S::kSh, 512), 64, idB, true);
                tc::mma_commit(bar(kD1Full));
                tc::mma_commit(bar(kEmpty0 + s));
                issued = true;
            }
            const float* rec = reinterpret_cast<const float*>(stg + S::kRec_);
            const float colf = rec[64 + t];
            const float rowf = nrow ? rec[i] : 0.f;
            float uv[16];
            if (nrow) {
                const float* ucol = reinterpret_cast<const float*>(stg + S::kU) + (size_t)vh * C + i;
#pragma unroll
                for (int v = 0; v < 16; ++v) uv[v] = transition ? 0.f : ucol[(size_t)v * C];  // transition: U = 0
            }
            // the output's N tile was last read by the output product of chunk c - 2
            // (scalar gate) or c - 1 (per-channel gates: N'_hi) (waited for here, while
            // the N product runs)
            if (S::kNBuf == 2) {
                if (c >= 2 && !tc::mbar_wait(bar(kOFull0 + ob), ((c - 2) >> 1) & 1, abort_flag)) fail();
            } else {
                if (c >= 1 && !tc::mbar_wait(bar(kOFull0 + ((c - 1) & 1)), ((c - 1) >> 1) & 1, abort_flag)) fail();
            }
            // N = U - W S^T  ->  N' = rowf * N (hi, lo), N (bf16).  Rows past the chunk
            // end come out exactly zero: the prep's U and W rows there are zero (beta
            // is zero there, so are those rows of (I + A)^{-1} diag(beta)).
            if (!tc::mbar_wait(bar(kD1Full), c & 1, abort_flag)) fail();  // keep going: every named barrier is reached by all threads
            tc::fence_after();
            float ws[16];  // (W S^T) for this thread's row and 16 columns
            if (nrow) {  // quadrants 0 and 1 (warp-uniform)
                float dv[48];
                tc::tmem_ld16x3(tD1 + 64 * ob + lane_base + vh, tD1 + 64 * ob + lane_base + BV + vh,
                                tD1b + lane_base + vh, dv);
#pragma unroll
                for (int v = 0; v < 16; v += 2) {  // on the fp32x2 pipe
                    const float2 w2 = __fadd2_rn(__fadd2_rn(make_float2(dv[v], dv[v + 1]), make_float2(dv[16 + v], dv[17 + v])),
                                                 make_float2(dv[32 + v], dv[33 + v]));
                    ws[v] = w2.x;
                    ws[v + 1] = w2.y;
                }
            }
            const uint32_t nbuf = (uint32_t)ob * (C * BV * 2);  // scalar gate: the output's N buffer
            if (nrow) {
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t hw[4], lw[4], nw[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int v = 8 * cc + 2 * u;
                        const float2 nn = sub2(make_float2(uv[v], uv[v + 1]), make_float2(ws[v], ws[v + 1]));
                        if (kKDA) {
                            // the row factor is 1 on the chunk's rows (and the rows past
                            // its end are zero), so N' = N and N'_hi is the output's N
                            split2x(nn, hw[u], lw[u]);
                        } else {
                            split2x(__fmul2_rn(nn, make_float2(rowf, rowf)), hw[u], lw[u]);
                            nw[u] = tc::pack_bf16(nn.x, nn.y);
                        }
                    }
                    const uint32_t off = tc::chunk_mn64(i, 2 * hf + cc);
                    *reinterpret_cast<uint4*>(sm + S::kNh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4*>(sm + S::kNl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    if (!kKDA) *reinterpret_cast<uint4*>(sm + S::kN + nbuf + off) = make_uint4(nw[0], nw[1], nw[2], nw[3]);
                }
            }
            tc::fence_proxy_async();
            tc::fence_before();
            tc::bar_sync(1, 256);
            if (kKDA && tid == 128) tc::mbar_arrive(bar(kNPub0 + s));  // N published: the output warps may drain chunk c - 1
            if (isA) {
                tc::fence_after();
                tc::mma_ksteps<4>(tD2, dmn128(st + S::kKt), amn, dmn64(base + S::kNh, C * BV * 2), 64, id2w, true);
                if (kKDA)
                    tc::mma_ksteps<4>(tD2, dmn128(st + S::kKt + kTile64x128), amn, dmn64(base + S::kNh, 512), 64, id2n, false);
                tc::mma_commit(bar(kD2Full));
                tc::mma_commit(bar(kEmpty0 + s));
            } else if (isC) {
                if (!outputs) {  // segment summary: no output, so no P N product
                    tc::mbar_arrive(bar(kOFull0 + ob));
                    tc::mbar_arrive(bar(kEmpty0 + s));
                } else {
                    tc::fence_after();
                    tc::mma_ksteps<4>(tD1 + 64 * ob, dk128(st + S::kYW), a64,
                                      dmn64(base + (kKDA ? S::kNh : S::kN + nbuf), 512), 64, idB, false);
                    tc::mma_commit(bar(kOFull0 + ob));
                    tc::mma_commit(bar(kEmpty0 + s));
                    issued = true;
                }
            }
            // while the update product runs: has the next chunk's stage landed (and,
            // for issuer A, its output buffer been drained)?
            staged = c + 1 < nc && tc::mbar_test(bar(kFull0 + (s ^ 1)), ((c + 1) >> 1) & 1);
            drained = isA && c >= 1 && c + 1 < nc && tc::mbar_test(bar(kOFree0 + (ob ^ 1)), (((c + 1) >> 1) - 1) & 1);
            // S^T <- colf * S^T + dS^T  (hi and lo halves of the accumulator summed)
            if (!tc::mbar_wait(bar(kD2Full), c & 1, abort_flag)) fail();  // keep going: every named barrier is reached by all threads
            tc::fence_after();
            {
                float dv[32];
                tc::tmem_ld16x2(tD2 + lane_base + vh, tD2 + lane_base + BV + vh, dv);
#pragma unroll
                for (int v = 0; v < 16; v += 2) {  // on the fp32x2 pipe
                    const float2 s2 = __ffma2_rn(make_float2(colf, colf), make_float2(Sreg[v], Sreg[v + 1]),
                                                 __fadd2_rn(make_float2(dv[v], dv[v + 1]), make_float2(dv[16 + v], dv[17 + v])));
                    Sreg[v] = s2.x;
                    Sreg[v + 1] = s2.y;
                }
            }
            // (the next thread synchronisation, the barrier that publishes S, is
            // preceded by its own tcgen05 fence)
        }
        if (issued) {  // every MMA this thread issued finished before the CTA leaves
            const int dr = isA ? kDrainA : isB ? kDrainB : kDrainC;
            tc::mma_commit(bar(dr));
            tc::mbar_wait(bar(dr), 0, abort_flag);
        }
        if (p.mode == 1 && !(first && last) && !*abort_flag) {  // segment summary (or the true end of a first segment)
            float* dst = (transition ? p.Mt : p.Bs) + (((size_t)sg * p.Hv + h) * D + v0 + vh) * D + t;
#pragma unroll
            for (int v = 0; v < 16; ++v) dst[(size_t)v * D] = Sreg[v];
        } else if (p.hT && last && !*abort_flag) {
            if (t < kDk) {
#pragma unroll
                for (int v = 0; v < 16; ++v) p.hT[(((size_t)b * p.Hv + h) * kDk + v0 + vh + v) * kDk + t] = Sreg[v];
            }
        }
    } else if (warp >= 12) {
        // ------------------------------ output warps ------------------------------
        // The output rows 64..127 of D1 sit in lane quadrants 2 and 3: warps 14
        // and 15 drain them; warps 12 and 13 only take part in the barriers.
        const int q = warp & 3;
        const bool drain = q >= 2;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const int i = 32 * (q - 2) + lane;
        __nv_bfloat16* op = static_cast<__nv_bfloat16*>(p.o);
        for (int c = 0; c < nc; ++c) {
            const int ob = c & 1;
            if (!tc::mbar_wait(bar(kOFull0 + ob), (c >> 1) & 1, abort_flag)) fail();
            // Drain when the state warps idle rather than beside their state update
            // and S store: with a scalar gate once the next chunk's S is published
            // (the N product runs; varlen prefill chain 90 -> 87 us), with
            // per-channel gates once its N is published (the update product runs;
            // 0.846 -> 0.838 ms; the N-product window measured slower there).  Two
            // barriers by chunk parity: the state group cannot publish chunk c + 3
            // before this chunk is drained (its N product waits for kOFree).
            if (!kKDA && c + 1 < nc && !tc::mbar_wait(bar(kSPub0 + ((c + 1) & 1)), ((c + 1) >> 1) & 1, abort_flag))
                fail();
            if (kKDA && c + 1 < nc && !tc::mbar_wait(bar(kNPub0 + ((c + 1) & 1)), ((c + 1) >> 1) & 1, abort_flag))
                fail();
            tc::fence_after();
            if (drain && outputs) {
                float ov[BV], ld[2 * BV];
                tc::tmem_ld64(tD1 + 64 * ob + lane_base, ld);
#pragma unroll
                for (int v = 0; v < BV; ++v) ov[v] = ld[v] + ld[BV + v];
                const int cs = bos + c * C;
                if (cs + i < eos) {
                    uint4* dst = reinterpret_cast<uint4*>(op + ((size_t)(cs + i) * p.Hv + h) * kDk + v0);
#pragma unroll
                    for (int u = 0; u < BV / 8; ++u)
                        dst[u] = make_uint4(tc::pack_bf16(p.scale * ov[8 * u], p.scale * ov[8 * u + 1]),
                                            tc::pack_bf16(p.scale * ov[8 * u + 2], p.scale * ov[8 * u + 3]),
                                            tc::pack_bf16(p.scale * ov[8 * u + 4], p.scale * ov[8 * u + 5]),
                                            tc::pack_bf16(p.scale * ov[8 * u + 6], p.scale * ov[8 * u + 7]));
                }
            }
            tc::fence_before();
            tc::bar_sync(2, 128);
            if (tid == 384) {
                tc::mbar_arrive(bar(kOFree0 + ob));
            }
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 2) tc::tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
// segment scan (chunk-parallel mode)
// ---------------------------------------------------------------------------
// The state map of a run of chunks is affine in its start state: with S in
// the [V][K] layout, S_end = S_start P + B, P the run from the identity with
// U = 0 and B the run from zero.  The summary pass ran the first segment of
// every sequence from h0 (its true end state E_0 is in B_0) and wrote P_j, B_j
// for the others (no P for the last one).  This kernel composes, in fp32,
//   S_start(1) = E_0,   S_start(j + 1) = S_start(j) P_j + B_j,
// writing S_start(j) over B_j (B_j has been copied in first).  One CTA per
// (value head, 4 value rows, sequence) of 512 threads: thread (k, mg) forms
// the partial product over m in [32 mg, 32 mg + 32) for the 4 rows of column
// k (four warps per scheduler hide the shared-memory latency), group 0 adds
// the partials and keeps the rows in registers; the rows sit transposed in
// shared memory for the next product.  P_j and the CTA's rows of B_j stream
// through a three-deep ring of shared-memory buffers, each filled by two 1-D
// bulk copies on its mbarrier two steps ahead.
constexpr int kScanRows = 4;
constexpr int kScanGroups = 4;
constexpr int kScanThreads = D * kScanGroups;
constexpr int kScanRing = 3;
constexpr uint32_t kScanP = D * D * 4;            // one P buffer
constexpr uint32_t kScanB = kScanRows * D * 4;    // one B buffer (the CTA's rows)
constexpr uint32_t kScanSmem = kScanRing * (kScanP + kScanB);

__global__ void __launch_bounds__(kScanThreads) chunk_seg_scan_kernel(TcParams p) {
    extern __shared__ float4 scan_smem[];
    float* Ps = reinterpret_cast<float*>(scan_smem);
    float* Bsm = Ps + kScanRing * D * D;
    __shared__ float4 Xs[D];                    // [k] -> rows 0..3
    __shared__ float4 red[kScanGroups - 1][D];  // partials of groups 1..3
    __shared__ __align__(8) uint64_t full[kScanRing];
    __shared__ int abort_flag;
    const int tid = threadIdx.x, k = tid & (D - 1), mg = tid >> 7;
    const int h = blockIdx.x / (D / kScanRows), r0 = (blockIdx.x % (D / kScanRows)) * kScanRows;
    const int b = blockIdx.y;
    if (tid == 0) {
        for (int i = 0; i < kScanRing; ++i) tc::mbar_init(tc::smem_u32(&full[i]), 1);
        abort_flag = 0;
        tc::mbar_fence_init();
    }
    __syncthreads();
    tc::grid_dep_wait();    // the segment summaries come from the chain kernel
    tc::grid_dep_launch();  // the output pass may start its prologue
    if (!p.meta[1]) return;
    const int sg0 = p.segoff[b], ns = p.segoff[b + 1] - sg0;
    auto bptr = [&](int j) { return p.Bs + ((size_t)(sg0 + j) * p.Hv + h) * D * D + (size_t)r0 * D; };
    if (ns == 0) {  // no chunks: the final state is the start state
        if (p.hT && mg == 0) {
#pragma unroll
            for (int r = 0; r < 4; ++r)
                p.hT[(((size_t)b * p.Hv + h) * D + r0 + r) * D + k] =
                    p.h0 ? p.h0[(((size_t)b * p.Hv + h) * D + r0 + r) * D + k] : 0.f;
        }
        return;
    }
    if (ns == 1) return;  // the summary pass ran the whole sequence
    // step t = 0 .. ns - 2 writes the start state of segment t + 1 and, for
    // t <= ns - 3, forms the next one from P_{t+1} and B_{t+1}
    float x[4];
    if (mg == 0) {
#pragma unroll
        for (int r = 0; r < 4; ++r) x[r] = bptr(0)[(size_t)r * D + k];  // E_0
        Xs[k] = make_float4(x[0], x[1], x[2], x[3]);
    }
    auto stage = [&](int t) {
        if (tid == 0 && t <= ns - 3) {
            const uint32_t fb = tc::smem_u32(&full[t % kScanRing]);
            tc::mbar_arrive_tx(fb, kScanP + kScanB);
            tc::bulk_g2s(tc::smem_u32(Ps + (t % kScanRing) * D * D),
                         p.Mt + ((size_t)(sg0 + t + 1) * p.Hv + h) * D * D, kScanP, fb);
            tc::bulk_g2s(tc::smem_u32(Bsm + (t % kScanRing) * kScanRows * D), bptr(t + 1), kScanB, fb);
        }
    };
    stage(0);
    stage(1);
    for (int t = 0; t <= ns - 2; ++t) {
        stage(t + 2);  // into the buffers read two steps ago (released by the barrier that ended that step)
        const bool more = t <= ns - 3;
        if (more && !tc::mbar_wait(tc::smem_u32(&full[t % kScanRing]), (t / kScanRing) & 1, &abort_flag)) {
            abort_flag = 1;
            atomicOr(p.err, 2u);
        }
        __syncthreads();  // P, B of segment t + 1 and its start state are visible
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (mg == 0) {
            // the start state of segment t + 1, over its B (copied in above)
            float* bj = bptr(t + 1) + k;
#pragma unroll
            for (int r = 0; r < 4; ++r) bj[(size_t)r * D] = x[r];
            if (more) {
                const float* bs = Bsm + (t % kScanRing) * kScanRows * D + k;
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[r] = bs[r * D];
            }
        }
        if (!more) break;
        const float* P = Ps + (t % kScanRing) * D * D + k;
        float acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
        for (int m = 32 * mg; m < 32 * mg + 32; m += 2) {
            const float p0 = P[m * D], p1 = P[(m + 1) * D];
            const float4 x0 = Xs[m], x1 = Xs[m + 1];
            acc[0] = fmaf(x0.x, p0, acc[0]);
            acc[1] = fmaf(x0.y, p0, acc[1]);
            acc[2] = fmaf(x0.z, p0, acc[2]);
            acc[3] = fmaf(x0.w, p0, acc[3]);
            acc2[0] = fmaf(x1.x, p1, acc2[0]);
            acc2[1] = fmaf(x1.y, p1, acc2[1]);
            acc2[2] = fmaf(x1.z, p1, acc2[2]);
            acc2[3] = fmaf(x1.w, p1, acc2[3]);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[r] += acc2[r];
        if (mg > 0) red[mg - 1][k] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        __syncthreads();  // partials written; every read of the old start state, P and B is done
        if (mg == 0) {
#pragma unroll
            for (int g2 = 0; g2 < kScanGroups - 1; ++g2) {
                const float4 tt = red[g2][k];
                acc[0] += tt.x;
                acc[1] += tt.y;
                acc[2] += tt.z;
                acc[3] += tt.w;
            }
            Xs[k] = make_float4(acc[0], acc[1], acc[2], acc[3]);
#pragma unroll
            for (int r = 0; r < 4; ++r) x[r] = acc[r];
        }
    }
    // no copy may still be writing shared memory when the CTA exits (they are
    // all waited for above unless a wait gave up): the last use of each slot
    if (tid == 0) {
        const int last_t = ns - 3;  // last step with copies
        for (int t = (last_t - kScanRing + 1 > 0 ? last_t - kScanRing + 1 : 0); t <= last_t; ++t)
            tc::mbar_wait_copies(tc::smem_u32(&full[t % kScanRing]), (t / kScanRing) & 1);
    }
}

}  // namespace

size_t chunk_tc_blob_bytes(int64_t max_chunks, int Hk, int Hv, bool kda) {
    const size_t mc = (size_t)max_chunks;
    size_t n = mc * Hv * kXwBytes;              // [W_hi ; Qd]
    n += mc * Hv * NVB * kUBlock;               // U
    n += mc * Hv * kYwBytes;                    // [W_lo ; P]
    n += kda ? mc * Hv * 2 * kTile64x128 : mc * Hk * kTile64x128;  // K / Kd
    n += mc * Hv * kRec;                        // records
    return n;
}

// Persistent prep grid: one CTA per resident slot (SMs x CTAs per SM), never
// more than the item capacity (chunk capacity x value heads).
static unsigned prep_grid(size_t items, int per_sm) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        sms = 148;
    const size_t slots = (size_t)sms * per_sm;
    return (unsigned)(items < slots ? items : slots);
}

cudaError_t launch_chunk_tc(const ChunkArgs& a, const ChunkWorkspace& w, char* ws, const void* q, const void* k,
                            cudaStream_t stream) {
    const bool kda = a.gk != nullptr;
    TcParams p{};
    p.q = q; p.k = k; p.v = a.v; p.g = a.g; p.gk = a.gk; p.beta = a.beta;
    p.h0 = a.initial_state; p.o = a.o; p.hT = a.final_state; p.cu = a.cu_seqlens;
    p.meta = reinterpret_cast<int*>(ws + w.off_meta);
    p.offsets = reinterpret_cast<int*>(ws + w.off_offsets);
    p.table = reinterpret_cast<const int4*>(ws + w.off_table);
    p.order = reinterpret_cast<int*>(ws + w.off_order);
    p.local_meta = w.local_meta ? 1 : 0;
    p.T = a.T;
    const size_t mc = (size_t)w.max_chunks;
    unsigned char* blob = reinterpret_cast<unsigned char*>(ws + w.off_blobs);
    p.Xw = blob; blob += mc * a.Hv * kXwBytes;
    p.Ub = blob; blob += mc * a.Hv * NVB * kUBlock;
    p.Yw = blob; blob += mc * a.Hv * kYwBytes;
    p.Kb = blob; blob += kda ? mc * a.Hv * 2 * kTile64x128 : mc * a.Hk * kTile64x128;
    p.Rb = blob;
    p.err = device_error_word();
    p.N = a.N; p.Hk = a.Hk; p.Hv = a.Hv; p.scale = a.scale;
    const unsigned nvb = (unsigned)(a.K / BV);  // value blocks per head in the chain

    if (w.seg_chunks > 0) {
        p.segs = reinterpret_cast<const int4*>(ws + w.off_segs);
        p.segoff = reinterpret_cast<const int*>(ws + w.off_segoff);
        p.Mt = reinterpret_cast<float*>(ws + w.off_mt);
        p.Bs = reinterpret_cast<float*>(ws + w.off_bs);
    }
    auto run = [&](auto prep_kernel, auto chain_kernel, int smp, int smc, int prep_per_sm, int prep_nt) -> cudaError_t {
        cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smp);
        cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smc);
        {
            KernelTimer kt("chunk_prep", stream);
            const cudaError_t e = launch_dependent(prep_kernel, dim3(prep_grid(mc * a.Hv, prep_per_sm)),
                                                   dim3(prep_nt), (size_t)smp, stream, p);
            if (e != cudaSuccess) return e;
        }
        if (w.seg_chunks == 0) {
            p.mode = 0;
            KernelTimer kt("chunk_chain", stream);
            return launch_dependent(chain_kernel, dim3(a.Hv * nvb, a.N), dim3(512), (size_t)smc, stream, p);
        }
        const unsigned segs = (unsigned)w.max_segs;
        {
            p.mode = 1;  // segment transitions and offsets
            KernelTimer kt("chunk_chain_summary", stream);
            const cudaError_t e = launch_dependent(chain_kernel, dim3(2 * a.Hv * nvb, segs), dim3(512), (size_t)smc,
                                                   stream, p);
            if (e != cudaSuccess) return e;
        }
        {
            cudaFuncSetAttribute(chunk_seg_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScanSmem);
            KernelTimer kt("chunk_seg_scan", stream);
            const cudaError_t e = launch_dependent(chunk_seg_scan_kernel, dim3(a.Hv * (D / kScanRows), a.N),
                                                   dim3(kScanThreads), (size_t)kScanSmem, stream, p);
            if (e != cudaSuccess) return e;
        }
        p.mode = 2;  // segments from their start states, with the output
        KernelTimer kt("chunk_chain", stream);
        return launch_dependent(chain_kernel, dim3(a.Hv * nvb, segs), dim3(512), (size_t)smc, stream, p);
    };
    const bool half = a.K == 64;
    const cudaError_t e =
        kda ? run(half ? chunk_prep_kda_kernel<64> : chunk_prep_kda_kernel<128>,
                  half ? chunk_chain_kernel<true, 64> : chunk_chain_kernel<true, 128>, (int)KdaSmem::kTotal,
                  ChainSmem<true>::kTotal, 2, kKdaThreads)
            : run(half ? chunk_prep_kernel<64> : chunk_prep_kernel<128>,
                  half ? chunk_chain_kernel<false, 64> : chunk_chain_kernel<false, 128>, (int)PrepSmem::kTotal,
                  ChainSmem<false>::kTotal, 2, kPrepThreads);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gdr
