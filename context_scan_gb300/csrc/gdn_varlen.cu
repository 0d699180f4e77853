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
// device, so the plan is made there, by the block that checks them, right after the check and
// before the WY tiles and the chains; the chain grids are launched with a bound on their
// entries and the chains past the plan's count return at once.
//
// The plan: among the piece lengths X (kMinPiece chunks, then each an eighth longer) at which
// both phases fit in one wave -- with k_s = ceil(n_s / X), A = sum over the cut sequences of
// k_s - 1 entries in each phase and one entry, in either phase, per sequence left whole; an
// entry is H chains -- the one with the shortest two phases and scan (2 X chunk times, plus
// the scan's steps, which run in sequence for each sequence, and the fixed cost of a cut),
// taken when that beats the longest sequence run whole; otherwise every sequence runs whole.
// The pieces of a sequence are ceil(n_s / k_s) chunks each, the last one the rest; a sequence
// left whole runs in the first phase while it has room, else in the second.
#include <algorithm>
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

__device__ __forceinline__ int warp_max(int x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
}

// The plan (one CTA of kPlanThreads, after the length check): cc = the checked chunk offsets,
// written by this block, read through L2.
__device__ void plan_body(const int* cc, int nseq, int H, int sms, int e_max, const PiecePlan& pl) {
    __shared__ int nsh[kPlanThreads];   // the lengths in chunks, when a cut is possible
    __shared__ unsigned long long wbest[kPlanThreads / 32];
    __shared__ int wmax[kPlanThreads / 32];
    __shared__ int wsum[4][kPlanThreads / 32];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int cap = sms / H;   // chains of one phase, in (sequence or piece) entries of H chains
    // a cut needs every sequence's chains in one wave, so then there is a thread per sequence
    const bool may_cut = nseq <= cap && nseq <= kPlanThreads;
    int maxn = 0;
    for (int s = t; s < nseq; s += kPlanThreads) maxn = max(maxn, __ldcg(cc + s + 1) - __ldcg(cc + s));
    maxn = warp_max(maxn);
    if (lane == 0) wmax[warp] = maxn;
    if (may_cut && t < nseq) nsh[t] = __ldcg(cc + t + 1) - __ldcg(cc + t);
    __syncthreads();
    for (int w = 0; w < kPlanThreads / 32; ++w) maxn = max(maxn, wmax[w]);
    // candidate piece lengths X_0 = kMinPiece, X_{i+1} = X_i + max(1, X_i / 8), below maxn (at
    // most ~130 of them for any length that fits an int): thread t costs X_t. With
    // k_s = ceil(n_s / X), A = the pieces past the first ones of the cut sequences (entries in
    // each phase), U = the sequences left whole (one entry in either phase), both phases
    // within `cap` entries; the time 2 X + the scan's steps (which run in sequence for each
    // sequence) + the fixed cost of a cut, in chunk times. Key: (time, X), the smallest wins;
    // running the sequences whole costs maxn.
    unsigned long long best = ((unsigned long long)maxn << 32) | (unsigned)maxn;
    if (may_cut && maxn >= 2 * kMinPiece) {
        int x = kMinPiece;
        for (int i = 0; i < t && x < maxn; ++i) x += max(1, x / 8);
        if (x < maxn) {
            long long A = 0, U = 0;
            int steps = 0;
            for (int s = 0; s < nseq; ++s) {
                const int n = nsh[s];
                const int k = n > 0 ? (n + x - 1) / x : 1;
                A += k - 1;
                U += k == 1 ? 1 : 0;
                steps = max(steps, k - 2);
            }
            const bool fits = A <= cap && 2 * A + U <= 2LL * cap && A <= e_max;
            const long long cost = 2LL * x + (long long)kStepChunks * steps + kCutChunks;
            if (fits && cost < maxn) best = ((unsigned long long)cost << 32) | (unsigned)x;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
        best = o < best ? o : best;
    }
    if (lane == 0) wbest[warp] = best;
    __syncthreads();
    for (int w = 0; w < kPlanThreads / 32; ++w) best = wbest[w] < best ? wbest[w] : best;
    const int X = max(1, (int)(best & 0xffffffffu));
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
            pl.counts[4] = 0;
        }
        return;
    }
    // a thread per sequence: its pieces, the slots of their states and summaries, and, for a
    // sequence left whole, the phase it runs in (the first while that has room). Four
    // exclusive prefix sums in thread order (warp scans, then the warps' totals): the first
    // state slot (and second-phase entry), the first summary slot, the rank among the whole
    // sequences and the rank among the sequences the scan visits (k >= 3).
    const bool mine = t < nseq;
    const int n = mine ? nsh[t] : 0;
    const int k = mine ? (n > 0 ? (n + X - 1) / X : 1) : 0;
    int v[4] = {k > 1 ? k - 1 : 0, k > 2 ? k - 2 : 0, mine && k == 1 ? 1 : 0, k > 2 ? 1 : 0};
    int in[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int y = __shfl_up_sync(0xffffffffu, in[q], off);
            if (lane >= off) in[q] += y;
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int q = 0; q < 4; ++q) wsum[q][warp] = in[q];
    }
    __syncthreads();
    int tot[4] = {0, 0, 0, 0};
    for (int w = 0; w < kPlanThreads / 32; ++w) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (w == warp) in[q] += tot[q] - v[q];   // inclusive -> exclusive, plus the warps before
            tot[q] += wsum[q][w];
        }
    }
    const int sig = in[0], mu = in[1], u = in[2];
    const int A = tot[0], NM = tot[1], U = tot[2];
    const int room1 = cap - A;   // whole sequences in the first phase
    if (mine) {
        const int s = t;
        const int xs = k > 1 ? (n + k - 1) / k : n;   // chunks of each piece but the last
        if (k == 1) {
            if (u < room1) {
                put_entry(pl.tab1f, s, s, 0, INT_MAX / kChunk, -1, -1, -1);
            } else {   // in the second phase, after the cut sequences' pieces
                put_entry(pl.tab1f, s, -1, 0, 0, -2, -2, -1);   // (no chain here)
                put_entry(pl.tab2, A + u - room1, s, 0, INT_MAX / kChunk, -1, -1, -1);
            }
        } else {
            // piece 0 from the sequence's initial state; it ends in the state entering piece 1
            put_entry(pl.tab1f, s, s, 0, xs, -1, sig, -1);
            for (int p = 1; p <= k - 2; ++p)   // the summaries of the middle pieces
                put_entry(pl.tab1s, mu + p - 1, s, p * xs, xs, -2, -2, mu + p - 1);
            for (int p = 1; p <= k - 1; ++p)   // the forwards of pieces 1 .. k-1 from their states
                put_entry(pl.tab2, sig + p - 1, s, p * xs, p == k - 1 ? n - p * xs : xs,
                          sig + p - 1, p == k - 1 ? -1 : -2, -1);
        }
        pl.seqinfo[3 * s] = k;
        pl.seqinfo[3 * s + 1] = sig;
        pl.seqinfo[3 * s + 2] = mu;
        if (k > 2) pl.seqinfo[3 * nseq + in[3]] = s;   // the scan's job list
    }
    if (t == 0) {
        pl.counts[0] = nseq;
        pl.counts[1] = NM;
        pl.counts[2] = A + (U > room1 ? U - room1 : 0);
        pl.counts[3] = X;
        pl.counts[4] = tot[3];
    }
}

// The length check in one block: each thread checks and sums a contiguous run of sequences, a
// block scan turns the per-thread chunk counts into the run's first chunk index. With PLAN,
// the plan follows in the same block.
constexpr unsigned kTagVarlen = 201;   // detail word of a rejected cu_seqlens

template <bool PLAN>
__global__ void __launch_bounds__(kPlanThreads) varlen_meta_kernel(
    const int* __restrict__ cu_in, int nseq, int T, int* cu_out, int* cu_chunks, DeviceError* err,
    int H, int sms, int e_max, PiecePlan pl) {
    __shared__ long long part[kPlanThreads];
    const int t = threadIdx.x;
    const int per = (nseq + kPlanThreads - 1) / kPlanThreads;
    const int s0 = min(nseq, t * per), s1 = min(nseq, s0 + per);
    bool bad = t == 0 && (cu_in[0] != 0 || cu_in[nseq] != T);
    long long acc = 0;
    for (int s = s0; s < s1; ++s) {
        const long long len = (long long)cu_in[s + 1] - cu_in[s];
        bad |= len < 0;
        acc += (len + kChunk - 1) / kChunk;
    }
    bad = __syncthreads_or(bad);
    part[t] = acc;
    __syncthreads();
    for (int off = 1; off < kPlanThreads; off <<= 1) {   // inclusive scan
        const long long x = t >= off ? part[t - off] : 0;
        __syncthreads();
        part[t] += x;
        __syncthreads();
    }
    long long run = part[t] - acc;
    for (int s = s0; s < s1; ++s) {
        cu_out[s] = bad ? 0 : cu_in[s];
        cu_chunks[s] = bad ? 0 : (int)run;
        run += ((long long)cu_in[s + 1] - cu_in[s] + kChunk - 1) / kChunk;
    }
    if (t == 0) {
        cu_out[nseq] = bad ? 0 : T;
        cu_chunks[nseq] = bad ? 0 : (int)part[kPlanThreads - 1];
        if (bad && err && atomicCAS(&err->code, 0u, (unsigned)GDN_ERR_INVALID_ARG) == 0u)
            atomicExch(&err->detail, kTagVarlen);
    }
    if constexpr (PLAN) {
        __syncthreads();   // the chunk offsets are complete
        plan_body(cu_chunks, nseq, H, sms, e_max, pl);
    }
}

// The scan of one sequence's pieces on one 16-column tile of the state (a task: a tile, a head
// and a job -- a sequence cut into three pieces or more, from the plan's job list; at most one
// CTA of 512 threads per SM, each taking every gridDim.x-th task, so that the whole grid is
// resident at once and its programmatic dependent launches right away): the state entering
// piece 1 (written by piece 0's forward), then H_{p+1} = M_p H_p + S_p for p = 1 .. k-2, each
// written to its slot. fp32 CUDA cores. The
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

__device__ __forceinline__ void scan_task(const int* __restrict__ seqinfo, int nseq, int H,
                                          const float* __restrict__ M, const float* __restrict__ S,
                                          float* __restrict__ states, int task) {
    constexpr int tiles = 128 / kScanCols;
    const int c0 = (task % tiles) * kScanCols, h = (task / tiles) % H, job = task / (tiles * H);
    const int s = seqinfo[3 * nseq + job];
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

__global__ void __launch_bounds__(kScanThreads, 1) piece_scan_kernel(const int* __restrict__ seqinfo,
                                                                     const int* __restrict__ counts,
                                                                     int nseq, int H,
                                                                     const float* __restrict__ M,
                                                                     const float* __restrict__ S,
                                                                     float* __restrict__ states) {
    // launched as the summary grid's programmatic dependent: every CTA waits for the first
    // phase, so this grid completes after it
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int tasks = counts[4] * H * (128 / kScanCols);
    for (int task = blockIdx.x; task < tasks; task += gridDim.x) {
        scan_task(seqinfo, nseq, H, M, S, states, task);
        __syncthreads();   // shared memory is free for the next task
    }
    // the second phase's chains may launch once every CTA is here (they wait for this grid
    // before they read a state): they are placed on a GPU the scan has left, not on the SMs it
    // leaves idle while it runs (placed there, a few of them ran ~10 % slower, measured)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace

bool pieces_possible(int T, int nseq, int H, int sms) {
    return (long long)nseq * H <= sms && (long long)T >= 2LL * kMinPiece * kChunk;
}

cudaError_t launch_varlen_meta(const int* cu_in, int nseq, int T, int* cu_out, int* cu_chunks,
                               DeviceError* err, cudaStream_t s) {
    if (!cu_in || !cu_out || !cu_chunks || nseq < 1) return cudaErrorInvalidValue;
    varlen_meta_kernel<false><<<1, kPlanThreads, 0, s>>>(cu_in, nseq, T, cu_out, cu_chunks, err, 1, 1,
                                                         1, PiecePlan{});
    return cudaGetLastError();
}

cudaError_t launch_varlen_meta_plan(const int* cu_in, int nseq, int T, int* cu_out, int* cu_chunks,
                                    DeviceError* err, int H, int sms, int e_max,
                                    const PiecePlan& pl, cudaStream_t s) {
    if (!cu_in || !cu_out || !cu_chunks || nseq < 1 || H < 1) return cudaErrorInvalidValue;
    varlen_meta_kernel<true><<<1, kPlanThreads, 0, s>>>(cu_in, nseq, T, cu_out, cu_chunks, err, H,
                                                        sms, e_max, pl);
    return cudaGetLastError();
}

cudaError_t launch_piece_scan(const PiecePlan& pl, int nseq, int H, int e_max, int sms,
                              const float* M, const float* S, float* states, cudaStream_t s) {
    if (nseq < 1 || H < 1 || e_max < 1 || sms < 1) return cudaErrorInvalidValue;
    // a sequence the scan visits has two entries or more among the e_max
    const long long tasks = (long long)std::max(1, std::min(nseq, e_max / 2)) * H * (128 / kScanCols);
    const cudaError_t e =
        cudaFuncSetAttribute(piece_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)std::min<long long>(tasks, sms));
    cfg.blockDim = dim3(kScanThreads);
    cfg.dynamicSmemBytes = kScanSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, piece_scan_kernel, (const int*)pl.seqinfo,
                              (const int*)pl.counts, nseq, H, M, S, states);
}

}  // namespace gdn
