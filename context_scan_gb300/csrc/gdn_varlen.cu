// gdn_varlen.cu -- packed sequences cut into pieces for the tcgen05 chains: the plan (on the
// device, from the checked lengths) and the scan over each sequence's piece summaries.
//
// One chain per (sequence, head) leaves the longest sequence setting the time while most SMs
// idle. As for the fixed-length batch ("RFC: HyperParallel Linear Attention Context Parallel",
// section 2.2: per-piece affine summaries composed by an exclusive scan; "Context Parallelism
// in ART", section 08), a sequence of n chunks is cut into k pieces of about n / k chunks: the
// first phase runs piece 0's forward from the sequence's initial state beside the summaries
// of pieces 1 .. k-2, the scan composes those from the state piece 0 ends in, and the second
// phase runs the forwards of pieces 1 .. k-1 from the scanned states. The lengths live on the
// device, so the plan is made there, by one CTA, before the chains run; the chain grids are
// launched with a bound on their entries and the chains past the plan's count return at once.
//
// The plan: the smallest piece length X (at least kMinPiece chunks) at which both phases fit
// in one wave -- with k_s = ceil(n_s / X), A = sum over the cut sequences of k_s - 1 entries in
// each phase and one entry, in either phase, per sequence left whole; an entry is H chains --
// and, among those X, the one with the shortest two phases and scan (2 X chunk times, plus the
// scan's steps, which run in sequence for each sequence, and the fixed cost of a second phase
// and the plan), taken when that beats the longest sequence run whole; otherwise every
// sequence runs whole (as before).
// The pieces of a sequence are ceil(n_s / k_s) chunks each, the last one the rest; a sequence
// left whole runs in the first phase while it has room, else in the second.
#include <climits>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kPlanThreads = 256;
constexpr int kMinPiece = 8;      // chunks: shorter pieces spend more on the scan than they save
// the fixed cost of a cut, in chunk times: the second phase's ramp (prologue, first loads and a
// pipeline to fill, about 20 us against a chunk's 2.5), the plan, the scan and the launches
constexpr int kCutChunks = 14;
constexpr int kStepChunks = 1;    // one step of a sequence's scan, in chunk times

__device__ __forceinline__ void put_entry(int* tab, int e, int seq, int chunk0, int nch, int start,
                                          int end, int ms) {
    int* t = tab + kPieceFields * e;
    t[PF_SEQ] = seq;
    t[PF_CHUNK0] = chunk0;
    t[PF_NCHUNKS] = nch;
    t[PF_START] = start;
    t[PF_END] = end;
    t[PF_MS] = ms;
    t[6] = 0;
    t[7] = 0;
}

// block-wide exclusive prefix sum (in thread order)
__device__ long long block_excl(long long x, long long* buf) {
    const int t = threadIdx.x;
    __syncthreads();
    buf[t] = x;
    __syncthreads();
    for (int off = 1; off < kPlanThreads; off <<= 1) {
        const long long y = t >= off ? buf[t - off] : 0;
        __syncthreads();
        buf[t] += y;
        __syncthreads();
    }
    return buf[t] - x;
}

__device__ __forceinline__ long long warp_sum(long long x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}
__device__ __forceinline__ int warp_max(int x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
}

__global__ void __launch_bounds__(kPlanThreads) piece_plan_kernel(const int* __restrict__ cc, int nseq,
                                                                  int H, int sms, int e_max,
                                                                  PiecePlan pl) {
    __shared__ long long buf[kPlanThreads];
    __shared__ int nsh[kPlanThreads];              // the lengths, when a cut is possible
    __shared__ long long best_cost[kPlanThreads / 32];
    __shared__ int best_x[kPlanThreads / 32], wmax[kPlanThreads / 32];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int cap = sms / H;   // chains of one phase, in (sequence or piece) entries of H chains
    // a cut needs every sequence's chains in one wave, so then there is a thread per sequence
    const bool may_cut = nseq <= cap && nseq <= kPlanThreads;
    int maxn = 0;
    for (int s = t; s < nseq; s += kPlanThreads) maxn = max(maxn, cc[s + 1] - cc[s]);
    maxn = warp_max(maxn);
    if (lane == 0) wmax[warp] = maxn;
    if (may_cut && t < nseq) nsh[t] = cc[t + 1] - cc[t];
    __syncthreads();
    for (int w = 0; w < kPlanThreads / 32; ++w) maxn = max(maxn, wmax[w]);
    // candidate piece lengths X = kMinPiece, growing by an eighth, below maxn; warp w costs
    // every eighth of them: with k_s = ceil(n_s / X), A = the pieces past the first ones of the
    // cut sequences (entries in each phase), U = the sequences left whole (one entry in either
    // phase), both phases within `cap` entries; the time 2 X + the scan's steps (which run in
    // sequence for each sequence) + the fixed cost of a cut, in chunk times
    long long my_cost = maxn;   // the sequences run whole
    int my_x = maxn;
    if (may_cut && maxn >= 2 * kMinPiece) {
        int i = 0;
        for (int x = kMinPiece; x < maxn; x += max(1, x / 8), ++i) {
            if (i % (kPlanThreads / 32) != warp) continue;
            long long A = 0, U = 0;
            int steps = 0;
            for (int s = lane; s < nseq; s += 32) {
                const int n = nsh[s];
                const int k = n > 0 ? (n + x - 1) / x : 1;
                A += k > 1 ? k - 1 : 0;
                U += k == 1 ? 1 : 0;
                steps = max(steps, k - 2);
            }
            A = warp_sum(A);
            U = warp_sum(U);
            steps = warp_max(steps);
            const bool fits = A <= cap && 2 * A + U <= 2LL * cap && A <= e_max;
            const long long cost = 2LL * x + (long long)kStepChunks * steps + kCutChunks;
            if (fits && cost < my_cost) {
                my_cost = cost;
                my_x = x;
            }
        }
    }
    if (lane == 0) {
        best_cost[warp] = my_cost;
        best_x[warp] = my_x;
    }
    __syncthreads();
    int X = maxn;
    long long bc = maxn;
    for (int w = 0; w < kPlanThreads / 32; ++w)
        if (best_cost[w] < bc || (best_cost[w] == bc && best_x[w] < X)) {
            bc = best_cost[w];
            X = best_x[w];
        }
    if (X < 1) X = 1;
    if (X >= maxn || !may_cut) {
        // nothing cut: every sequence whole, in the first phase
        for (int s = t; s < nseq; s += kPlanThreads) {
            put_entry(pl.tab1f, s, s, 0, INT_MAX / kChunk, -1, -1, -1);
            pl.seqinfo[3 * s] = 1;
            pl.seqinfo[3 * s + 1] = 0;
            pl.seqinfo[3 * s + 2] = 0;
        }
        if (t == 0) {
            pl.counts[0] = nseq;
            pl.counts[1] = 0;
            pl.counts[2] = 0;
            pl.counts[3] = maxn;
        }
        return;
    }
    // a thread per sequence: its pieces, the slots of their states and summaries, and, for a
    // sequence left whole, the phase it runs in (the first while that has room)
    const bool mine = t < nseq;
    const int n = mine ? nsh[t] : 0;
    const int k = mine ? (n > 0 ? (n + X - 1) / X : 1) : 0;
    const long long sig = block_excl(k > 1 ? k - 1 : 0, buf);   // state slots (and phase-2 entries)
    const long long mu = block_excl(k > 2 ? k - 2 : 0, buf);    // summary slots
    const long long u = block_excl(mine && k == 1 ? 1 : 0, buf);   // rank among whole ones
    // the totals: the last thread's exclusive sum plus its own
    __shared__ long long tot[3];
    if (t == kPlanThreads - 1) {
        tot[0] = sig + (k > 1 ? k - 1 : 0);
        tot[1] = mu + (k > 2 ? k - 2 : 0);
        tot[2] = u + (mine && k == 1 ? 1 : 0);
    }
    __syncthreads();
    const long long A = tot[0], U = tot[2];
    const long long room1 = cap - A;   // whole sequences in the first phase
    if (mine) {
        const int s = t;
        const int xs = k > 1 ? (n + k - 1) / k : n;   // chunks of each piece but the last
        if (k == 1) {
            if (u < room1) {
                put_entry(pl.tab1f, s, s, 0, INT_MAX / kChunk, -1, -1, -1);
            } else {   // in the second phase, after the cut sequences' pieces
                put_entry(pl.tab1f, s, -1, 0, 0, -2, -2, -1);   // (no chain here)
                put_entry(pl.tab2, (int)(A + u - room1), s, 0, INT_MAX / kChunk, -1, -1, -1);
            }
        } else {
            // piece 0 from the sequence's initial state; it ends in the state entering piece 1
            put_entry(pl.tab1f, s, s, 0, xs, -1, (int)sig, -1);
            for (int p = 1; p <= k - 2; ++p)   // the summaries of the middle pieces
                put_entry(pl.tab1s, (int)mu + p - 1, s, p * xs, xs, -2, -2, (int)mu + p - 1);
            for (int p = 1; p <= k - 1; ++p)   // the forwards of pieces 1 .. k-1 from their states
                put_entry(pl.tab2, (int)sig + p - 1, s, p * xs, p == k - 1 ? n - p * xs : xs,
                          (int)sig + p - 1, p == k - 1 ? -1 : -2, -1);
        }
        pl.seqinfo[3 * s] = k;
        pl.seqinfo[3 * s + 1] = (int)sig;
        pl.seqinfo[3 * s + 2] = (int)mu;
    }
    if (t == 0) {
        pl.counts[0] = nseq;
        pl.counts[1] = (int)tot[1];
        pl.counts[2] = (int)(A + (U > room1 ? U - room1 : 0));
        pl.counts[3] = X;
    }
}

// The scan of one sequence's pieces on one 16-column tile of the state (one CTA per sequence,
// head and tile; 512 threads): the state entering piece 1 (written by piece 0's forward), then
// H_{p+1} = M_p H_p + S_p for p = 1 .. k-2, each written to its slot. fp32 CUDA cores. The
// product's inner dimension is split over four thread groups of 128 (a 4 x 4 register tile
// each, rows 4 rb .., columns 4 cb ..), whose partial sums meet in shared memory; M_p sits in
// shared memory whole (rows padded to 129 floats: the column reads are conflict-free) and the
// next step's M is loaded into registers while a step computes.
constexpr int kScanThreads = 512;
constexpr int kScanCols = 16;
constexpr int kMp = 129;   // row pitch of the staged M
constexpr int kRp = 20;    // row pitch of the partial sums (float4 stores without conflicts)
constexpr int kScanSmem = (128 * kScanCols + 128 * kMp) * 4;
static_assert(4 * 128 * kRp <= 128 * kMp, "the partial sums fit where M was staged");

__global__ void __launch_bounds__(kScanThreads, 1) piece_scan_kernel(const int* __restrict__ seqinfo,
                                                                     int H,
                                                                     const float* __restrict__ M,
                                                                     const float* __restrict__ S,
                                                                     float* __restrict__ states) {
    const int s = blockIdx.x, h = blockIdx.y, c0 = blockIdx.z * kScanCols;
    const int k = seqinfo[3 * s], sig = seqinfo[3 * s + 1], mu = seqinfo[3 * s + 2];
    if (k < 3) return;
    extern __shared__ __align__(16) float smem[];
    float* Hs = smem;                      // [128][16]: the state tile
    float* Ms = smem + 128 * kScanCols;    // [128][kMp]: M_p; afterwards the partial sums
    const int t = threadIdx.x;
    const int kg = t >> 7, rb = (t & 127) >> 2, cb = t & 3;   // the product's thread roles
    const int mr = t & 127, mq = t >> 7;                      // staging: row mr, columns 32 mq ..
    const int orow = t >> 2, ocol = 4 * (t & 3);              // the output element's row, columns
    const long long kv = 128LL * 128;
    auto slot_of = [&](int p) { return (long long)(mu + p - 1) * H + h; };
    float4 m4[8];
    auto load_m = [&](int p) {
        const float4* src = reinterpret_cast<const float4*>(M + slot_of(p) * kv + mr * 128 + 32 * mq);
#pragma unroll
        for (int q = 0; q < 8; ++q) m4[q] = src[q];
    };
    auto load_s = [&](int p) {
        return *reinterpret_cast<const float4*>(S + slot_of(p) * kv + orow * 128 + c0 + ocol);
    };
    *reinterpret_cast<float4*>(Hs + orow * kScanCols + ocol) = *reinterpret_cast<const float4*>(
        states + ((long long)sig * H + h) * kv + orow * 128 + c0 + ocol);
    load_m(1);
    float4 s4 = load_s(1);
    for (int p = 1; p <= k - 2; ++p) {
        __syncthreads();   // the previous step's partial sums are read (and Hs is complete)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float* d = Ms + mr * kMp + 32 * mq + 4 * q;
            d[0] = m4[q].x;
            d[1] = m4[q].y;
            d[2] = m4[q].z;
            d[3] = m4[q].w;
        }
        __syncthreads();
        float4 s4n = s4;
        if (p + 1 <= k - 2) {   // the next step's operands, in flight while this one computes
            load_m(p + 1);
            s4n = load_s(p + 1);
        }
        float acc[4][4] = {};
        const float* mrow = Ms + 4 * rb * kMp + 32 * kg;
        const float* hrow = Hs + 32 * kg * kScanCols + 4 * cb;
#pragma unroll 8
        for (int j = 0; j < 32; ++j) {
            const float4 hv = *reinterpret_cast<const float4*>(hrow + j * kScanCols);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float m = mrow[i * kMp + j];
                acc[i][0] = fmaf(m, hv.x, acc[i][0]);
                acc[i][1] = fmaf(m, hv.y, acc[i][1]);
                acc[i][2] = fmaf(m, hv.z, acc[i][2]);
                acc[i][3] = fmaf(m, hv.w, acc[i][3]);
            }
        }
        __syncthreads();   // every read of M_p and H_p is done
        float* red = Ms + kg * 128 * kRp;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            *reinterpret_cast<float4*>(red + (4 * rb + i) * kRp + 4 * cb) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        __syncthreads();
        float4 o = s4;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const float4 v = *reinterpret_cast<const float4*>(Ms + g * 128 * kRp + orow * kRp + ocol);
            o.x += v.x;
            o.y += v.y;
            o.z += v.z;
            o.w += v.w;
        }
        *reinterpret_cast<float4*>(Hs + orow * kScanCols + ocol) = o;
        *reinterpret_cast<float4*>(states + ((long long)(sig + p) * H + h) * kv + orow * 128 + c0 +
                                   ocol) = o;
        s4 = s4n;
    }
}

}  // namespace

bool pieces_possible(int T, int nseq, int H, int sms) {
    return (long long)nseq * H <= sms && (long long)T >= 2LL * kMinPiece * kChunk;
}

cudaError_t launch_piece_plan(const int* cu_chunks, int nseq, int H, int sms, int e_max,
                              const PiecePlan& pl, cudaStream_t s) {
    piece_plan_kernel<<<1, kPlanThreads, 0, s>>>(cu_chunks, nseq, H, sms, e_max, pl);
    return cudaGetLastError();
}

cudaError_t launch_piece_scan(const int* seqinfo, int nseq, int H, const float* M, const float* S,
                              float* states, cudaStream_t s) {
    if (nseq < 1 || H < 1 || H > 65535) return cudaErrorInvalidValue;
    const cudaError_t e =
        cudaFuncSetAttribute(piece_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmem);
    if (e != cudaSuccess) return e;
    piece_scan_kernel<<<dim3((unsigned)nseq, (unsigned)H, 128 / kScanCols), kScanThreads, kScanSmem,
                        s>>>(seqinfo, H, M, S, states);
    return cudaGetLastError();
}

}  // namespace gdn
