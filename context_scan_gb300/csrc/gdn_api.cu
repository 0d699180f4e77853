// gdn_api.cu -- the C ABI (include/gdn.h): argument validation, workspace layout and the
// launch sequence on the caller's stream. No allocation, no synchronisation (except
// gdn_check_device_error), no CPU fallback.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <cmath>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

using gdn::ChainParams;

constexpr size_t kHeaderBytes = 256;   // device error word, then the WY queue counter
constexpr size_t kQueueOffset = 64;    // the WY queue counter's offset in the header
// the last piece's WY tiles are formed beside the first phase when they take at least this
// many waves of the WY kernel's CTAs (six per SM) on the whole GPU, and the first phase leaves
// at least this many SMs idle in its last wave
constexpr int kTailMinWaves = 1;
constexpr int kTailMinIdle = 8;
constexpr size_t kAlign = 256;
constexpr int kMaxSub = 8;             // pieces per segment (segmented forward)
constexpr int kMinPieceChunks = 8;     // shortest piece, in chunks
constexpr int kMaxUnevenPieces = 16;   // unequal pieces (one wave per phase): at most this many
constexpr unsigned kSelftestTag = 0x5E;   // detail word of the self-test's timeout

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// How the segmented forward cuts each sequence: P pieces; piece 0 has `first` chunks and the
// others `rest` each (first == rest: equal pieces, whose starts include every segment start).
struct PiecePlan {
    int P, first, rest;
};

struct WsLayout {
    size_t off_wy, off_M, off_S, off_Hp, total;
    int pieces;
    PiecePlan plan;
};

// Shapes that take the tcgen05 kernels (which also need the per-chunk WY tiles).
bool tc_shape(const gdn_problem& p) {
    return p.in_dtype == GDN_DTYPE_BF16 && p.K == 128 && p.V == 128 && !p.gate_k;
}

// Per-channel gates at bf16 inputs: the chains read every chunk's A diag(beta) and C, formed
// beforehand.
bool kda_prep_shape(const gdn_problem& p) { return p.in_dtype == GDN_DTYPE_BF16 && p.gate_k; }

// bytes of per-chunk factors the chains read, per chunk and head
size_t chunk_factor_bytes(const gdn_problem& p) {
    return tc_shape(p) ? (size_t)gdn::kWyPairBytes
                       : (kda_prep_shape(p) ? 2u * 64u * 64u * sizeof(float) : 0u);
}

// Device properties asked on every call, looked up once per device (a call on a short
// problem would otherwise spend a visible part of its time in these queries).
constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];
std::atomic<int> g_cc[kMaxDevices];   // 10 * major + minor, 0 until known

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    int sms = (dev >= 0 && dev < kMaxDevices) ? g_sms[dev].load(std::memory_order_relaxed) : 0;
    if (sms > 0) return sms;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) g_sms[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

// Pieces per sequence for the segmented forward. Piece 0's forward runs from h0 beside the
// summaries of pieces 1..P-2; an in-order scan gives the state entering every piece; pieces
// 1..P-1 then run their forward. Each phase launches B*H*(P-1) chains, one per SM at a time.
// Costs in chunk times (a summary chunk costs kSumRatio of a forward chunk, a scan step about
// three):
//  - equal pieces, P = nseg * {1, 2, 4, 8} (segment starts are piece starts, pieces of at
//    least 8 chunks): 2 * waves(B*H*(P-1)) * chunks / P + 3 * (P - 2);
//  - tcgen05 path only, when both phases fit in one wave (B*H*(P-1) <= SMs): piece 0 of L0
//    chunks and pieces 1..P-1 of x chunks, x = chunks / (P - 1 + kSumRatio), so that piece 0's
//    forward and the summaries end together: max(L0, kSumRatio x) + x + 3 * (P - 2). The
//    forward kernels then write the states entering the segments as they pass them.
// Without a device to size the waves it stays at nseg equal pieces. kSumRatio is the measured
// per-chunk time of the first phase's summary chains over its forward chain (per-CTA clock
// stamps at B2 H32 T32K: 2.46 against 2.51 us).
constexpr double kSumRatio = 0.98;

PiecePlan plan_pieces(const gdn_problem& p, int nseg) {
    const int chunks = p.T / gdn::kChunk;   // a multiple of nseg (checked)
    PiecePlan best{nseg, chunks / nseg, chunks / nseg};
    if (p.T <= 0) return best;
    const int sms = sm_count();
    if (sms < 1) return best;
    const double bh = (double)p.B * p.H;
    auto cost_equal = [&](int P) {
        const double waves = std::ceil(bh * (P > 1 ? P - 1 : 1) / sms);
        const double phases = P > 1 ? 2.0 : 1.0;
        return phases * waves * ((double)chunks / P) + 3.0 * (P > 2 ? P - 2 : 0);
    };
    double best_cost = cost_equal(nseg);
    for (int nsub = 2; nsub <= kMaxSub; nsub *= 2) {
        const int P = nseg * nsub;
        if ((chunks / nseg) % nsub != 0 || chunks / P < kMinPieceChunks) break;
        const double c = cost_equal(P);
        if (c < best_cost) {
            best_cost = c;
            best = PiecePlan{P, chunks / P, chunks / P};
        }
    }
    if (tc_shape(p) && gdn::tc_runtime_ok()) {
        for (int P = 3; P <= kMaxUnevenPieces && bh * (P - 1) <= sms; ++P) {
            int x = (int)std::ceil(chunks / (P - 1 + kSumRatio));
            if (chunks - (P - 1) * x < 1) x = (chunks - 1) / (P - 1);
            const int first = chunks - (P - 1) * x;
            if (x < kMinPieceChunks || first < 1) break;
            const double c = std::max((double)first, kSumRatio * x) + x + 3.0 * (P - 2);
            if (c < best_cost) {
                best_cost = c;
                best = PiecePlan{P, first, x};
            }
        }
    }
    return best;
}

// [header | WY tiles (tcgen05 shapes) | M | S | Hp], each region 256-byte aligned: M, S hold
// the summaries of pieces 1..P-2 and Hp the state entering each piece (indexed by piece)
WsLayout layout(const gdn_problem& p, int nseg) {
    WsLayout w{};
    const size_t bh = (size_t)p.B * p.H;
    w.plan = plan_pieces(p, nseg);
    w.pieces = w.plan.P;
    w.off_wy = kHeaderBytes;
    const size_t wy_bytes = bh * (size_t)(p.T / gdn::kChunk) * chunk_factor_bytes(p);
    w.off_M = w.off_wy + round_up(wy_bytes);
    const size_t P = (size_t)w.pieces;
    const size_t m_bytes = P >= 3 ? round_up(sizeof(float) * P * bh * p.K * p.K) : 0;
    const size_t s_bytes = P >= 3 ? round_up(sizeof(float) * P * bh * p.K * p.V) : 0;
    const size_t h_bytes = P >= 2 ? round_up(sizeof(float) * P * bh * p.K * p.V) : 0;
    w.off_S = w.off_M + m_bytes;
    w.off_Hp = w.off_S + s_bytes;
    w.total = w.off_Hp + h_bytes;
    return w;
}

bool misaligned(const void* ptr) { return ptr && (reinterpret_cast<uintptr_t>(ptr) & 15u); }

gdn_status check_problem(const gdn_problem* p, int nseg) {
    if (!p) return GDN_ERR_INVALID_ARG;
    if (p->B < 1 || p->H < 1 || p->T < 0) return GDN_ERR_INVALID_ARG;
    if (nseg < 1) return GDN_ERR_INVALID_ARG;
    if (p->chunk != gdn::kChunk) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (p->decay_first != 0 && p->decay_first != 1) return GDN_ERR_INVALID_ARG;
    if (p->gate_k != 0 && p->gate_k != 1) return GDN_ERR_INVALID_ARG;
    if (p->K != p->V || (p->K != 64 && p->K != 128)) return GDN_ERR_UNSUPPORTED_SHAPE;
    if ((p->in_dtype != GDN_DTYPE_F32 && p->in_dtype != GDN_DTYPE_BF16) ||
        (p->out_dtype != GDN_DTYPE_F32 && p->out_dtype != GDN_DTYPE_BF16))
        return GDN_ERR_UNSUPPORTED_DTYPE;
    if (p->T % (gdn::kChunk * nseg) != 0) return GDN_ERR_UNSUPPORTED_SHAPE;
    const long long elems = (long long)p->B * p->T * p->H * p->K;
    if (elems >= (1LL << 40)) return GDN_ERR_UNSUPPORTED_SHAPE;
    if ((long long)p->B * p->H * nseg >= (1LL << 31)) return GDN_ERR_UNSUPPORTED_SHAPE;
    return GDN_OK;
}

gdn_status check_device() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
    int cc = (dev >= 0 && dev < kMaxDevices) ? g_cc[dev].load(std::memory_order_relaxed) : 0;
    if (cc == 0) {
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return GDN_ERR_CUDA;
        cc = 10 * major + minor;
        if (dev >= 0 && dev < kMaxDevices) g_cc[dev].store(cc, std::memory_order_relaxed);
    }
    return cc == 103 ? GDN_OK : GDN_ERR_DEVICE;
}

gdn_status check_workspace(const gdn_problem* p, int nseg, const void* ws, size_t ws_bytes) {
    if (!ws || ws_bytes < layout(*p, nseg).total) return GDN_ERR_WORKSPACE;
    if (misaligned(ws)) return GDN_ERR_MISALIGNED;
    return GDN_OK;
}

gdn_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

cudaError_t mark(void* const* events, int i, cudaStream_t s) {
    if (!events || !events[i]) return cudaSuccess;
    return cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), s);
}

ChainParams base_params(const gdn_problem* p, void* ws) {
    ChainParams c{};
    c.B = p->B;
    c.T = p->T;
    c.H = p->H;
    c.K = p->K;
    c.V = p->V;
    c.in_bf16 = p->in_dtype == GDN_DTYPE_BF16;
    c.out_bf16 = p->out_dtype == GDN_DTYPE_BF16;
    c.decay_first = p->decay_first;
    c.gate_k = p->gate_k;
    c.err = reinterpret_cast<gdn::DeviceError*>(ws);
    return c;
}

bool use_tc(const ChainParams& c) { return c.T > 0 && gdn::tc_supported(c); }

// The tcgen05 chains read every chunk's WY tiles from the workspace: form them first (one
// launch for all chunks of the problem). Nothing to do on the CUDA-core path.
cudaError_t prepare(ChainParams& c, const gdn_problem* p, void* ws, cudaStream_t s) {
    c.wy = reinterpret_cast<char*>(ws) + layout(*p, 1).off_wy;
    if (use_tc(c)) return gdn::launch_tc_wy(c, s);
    if (kda_prep_shape(*p) && p->T > 0) return gdn::launch_kda_prep(c, s);
    return cudaSuccess;
}

cudaError_t run_forward(const ChainParams& c, cudaStream_t s) {
    return use_tc(c) ? gdn::launch_tc_forward(c, s) : gdn::launch_simt_forward(c, s);
}

cudaError_t run_summary(const ChainParams& c, cudaStream_t s) {
    return use_tc(c) ? gdn::launch_tc_summary(c, s) : gdn::launch_simt_summary(c, s);
}

// The segmented forward on validated arguments (also gdn_chunk_fwd, nseg = 1): each sequence
// is cut into P pieces (plan_pieces). Stage events: 0 before the WY tiles, 1 before the first
// phase (which includes the last piece's WY tiles when they are formed beside it), 2 before the
// scan, 3 before the second phase, 4 at the end.
gdn_status run_segmented(const gdn_problem* p, int nseg, const void* q, const void* k,
                         const void* v, const void* g, const void* beta, const float* h0, void* o,
                         float* h_final, float* H_in_out, void* workspace, cudaStream_t s,
                         void* const* events) {
    const WsLayout w = layout(*p, nseg);
    const int P = w.pieces, nsub = P / nseg;
    // equal pieces whose starts include every segment start: the scan writes H_in_out;
    // otherwise (pieces of unequal length, or an unequal plan whose pieces came out equal but
    // do not divide the segments) the forwards write it as they pass the segment starts
    const bool equal = w.plan.first == w.plan.rest && P % nseg == 0;
    const int BH = p->B * p->H;
    char* wsb = reinterpret_cast<char*>(workspace);
    if (mark(events, 0, s) != cudaSuccess || mark(events, 1, s) != cudaSuccess ||
        mark(events, 2, s) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (p->T == 0) {
        // nothing to process: every segment starts from h0 and h_final = h0 (or zeros)
        if (H_in_out && gdn::launch_scan(nullptr, nullptr, h0, nullptr, H_in_out, nullptr, 0, nseg,
                                         1, BH, p->K, p->V, s) != cudaSuccess)
            return GDN_ERR_CUDA;
        if (mark(events, 3, s) != cudaSuccess) return GDN_ERR_CUDA;
        if (h_final && gdn::launch_scan(nullptr, nullptr, h0, nullptr, h_final, nullptr, 0, 1, 1, BH,
                                        p->K, p->V, s) != cudaSuccess)
            return GDN_ERR_CUDA;
        return from_cuda(mark(events, 4, s));
    }
    float* M = reinterpret_cast<float*>(wsb + w.off_M);
    float* S = reinterpret_cast<float*>(wsb + w.off_S);
    float* Hp = reinterpret_cast<float*>(wsb + w.off_Hp);
    const long long hstride = (long long)BH * p->K * p->V;
    auto chain = [&]() {
        ChainParams c = base_params(p, workspace);
        c.q = q;
        c.k = k;
        c.v = v;
        c.g = g;
        c.beta = beta;
        c.o = o;
        c.seg_len = w.plan.rest * gdn::kChunk;
        c.first_chunks = w.plan.first;
        c.nseg_total = P;
        if (!equal) {
            c.H_seg = H_in_out;
            c.seg_chunks = p->T / gdn::kChunk / nseg;
        }
        return c;
    };
    // 0. the WY tiles (tcgen05 path only): of every chunk; or, when the first phase's chains
    //    leave SMs free (in its only wave, or in its last), of pieces 0..P-2 only -- the last
    //    piece's are formed on those SMs beside the chains (a programmatic dependent of the
    //    first phase that hands its chunks out from a counter), since only the second phase
    //    reads them
    if (mark(events, 0, s) != cudaSuccess) return GDN_ERR_CUDA;
    ChainParams cw = chain();
    const int nchunks = p->T / gdn::kChunk;
    const int last_lo = P >= 2 ? w.plan.first + (P - 2) * w.plan.rest : nchunks;
    const int sms = sm_count();
    // SMs the first phase leaves idle in its last wave (all of its chains when they fit one)
    const long long chains1 = (long long)BH * (P - 1);
    const long long idle1 = sms > 0 && chains1 % sms != 0 ? sms - chains1 % sms : 0;
    const bool tail_beside = use_tc(cw) && P >= 2 && idle1 >= kTailMinIdle &&
                             (long long)BH * (nchunks - last_lo) >= 6LL * kTailMinWaves * sms;
    cw.wy_lo = 0;
    cw.wy_cnt = tail_beside ? last_lo : 0;
    unsigned* queue = reinterpret_cast<unsigned*>(wsb + kQueueOffset);
    cw.wy_queue_reset = tail_beside ? queue : nullptr;   // zeroed by the first WY launch
    cudaError_t e = prepare(cw, p, workspace, s);
    cw.wy_queue_reset = nullptr;
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    // 1. piece 0's forward from h0, which hands its final state to piece 1, beside the
    //    summaries of pieces 1..P-2 (one grid on the tensor-core path; otherwise the summaries
    //    are launched as the forward's programmatic dependent, so they start at once on the
    //    SMs it leaves free)
    if (mark(events, 1, s) != cudaSuccess) return GDN_ERR_CUDA;
    ChainParams f0 = chain();
    f0.wy = cw.wy;
    f0.h_start = h0;
    f0.seg_first = 0;
    f0.nseg_run = 1;
    f0.h_final = P == 1 ? h_final : nullptr;
    f0.h_out = P > 1 ? Hp : nullptr;
    f0.h_out_seg_stride = hstride;
    if (P >= 3) {
        ChainParams cs = chain();
        cs.wy = cw.wy;
        cs.M = M;
        cs.S = S;
        cs.seg_first = 1;
        cs.nseg_run = P - 2;
        if (tail_beside) {
            e = gdn::launch_tc_phase1(f0, cs, s);
        } else {
            cs.launch_dependent = 1;
            e = run_forward(f0, s);
            if (e == cudaSuccess) e = run_summary(cs, s);
        }
    } else {
        e = run_forward(f0, s);
    }
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    if (tail_beside) {
        ChainParams ct = cw;
        ct.wy_lo = last_lo;
        ct.wy_cnt = nchunks - last_lo;
        ct.wy_queue = queue;
        ct.launch_dependent = 1;
        if (gdn::launch_tc_wy(ct, s) != cudaSuccess) return GDN_ERR_CUDA;
    }
    // 2. the state entering every piece (and every segment)
    if (mark(events, 2, s) != cudaSuccess) return GDN_ERR_CUDA;
    if (P >= 2)
        e = gdn::launch_scan(M, S, Hp + hstride, Hp, equal ? H_in_out : nullptr, h0, 1, P,
                             equal ? nsub : 1, BH, p->K, p->V, s,
                             reinterpret_cast<gdn::DeviceError*>(workspace));
    else if (H_in_out)
        e = gdn::launch_scan(nullptr, nullptr, h0, nullptr, H_in_out, nullptr, 0, 1, 1, BH, p->K, p->V, s);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    // 3. pieces 1..P-1 from the scanned states
    if (mark(events, 3, s) != cudaSuccess) return GDN_ERR_CUDA;
    if (P >= 2) {
        ChainParams cf = chain();
        cf.wy = cw.wy;
        cf.h_start = Hp;
        cf.h_start_seg_stride = hstride;
        cf.h_final = h_final;
        cf.seg_first = 1;
        cf.nseg_run = P - 1;
        if ((e = run_forward(cf, s)) != cudaSuccess) return GDN_ERR_CUDA;
    }
    return from_cuda(mark(events, 4, s));
}


// ---- varlen: [header | WY tiles (tcgen05 shapes), [H][T/64 + nseq] | checked cu_seqlens |
//      cu_chunks | (tcgen05 shapes) the piece plan: tab1f, tab1s, tab2, counts, seqinfo |
//      piece states | piece summaries M, S], each region 256-byte aligned. T/64 + nseq bounds the
//      chunks of any split of T tokens into nseq sequences, and e_max = kPieceSmBound / H the
//      pieces past the first ones on any device, so the layout needs no host copy of the
//      lengths.
constexpr int kPieceSmBound = 256;
struct VarlenLayout {
    size_t off_wy, off_cu, off_cc, off_t1f, off_t1s, off_t2, off_cnt, off_si, off_st, off_m, off_s,
        total;
    int chunk_bound, e_max;
    bool pieces;
};

VarlenLayout varlen_layout(const gdn_problem& p, int nseq) {
    VarlenLayout w{};
    w.chunk_bound = p.T / gdn::kChunk + nseq;
    w.off_wy = kHeaderBytes;
    const size_t wy_bytes = (size_t)p.H * (size_t)w.chunk_bound * chunk_factor_bytes(p);
    w.off_cu = w.off_wy + round_up(wy_bytes);
    w.off_cc = w.off_cu + round_up(sizeof(int) * ((size_t)nseq + 1));
    w.total = w.off_cc + round_up(sizeof(int) * ((size_t)nseq + 1));
    w.pieces = tc_shape(p) && !p.gate_k;
    if (w.pieces) {
        const size_t ent = sizeof(int) * gdn::kPieceFields;
        const size_t kv = (size_t)p.K * p.V, kk = (size_t)p.K * p.K;
        w.e_max = std::max(1, kPieceSmBound / p.H);
        w.off_t1f = w.total;
        w.off_t1s = w.off_t1f + round_up(ent * (size_t)nseq);
        w.off_t2 = w.off_t1s + round_up(ent * (size_t)w.e_max);
        w.off_cnt = w.off_t2 + round_up(ent * (size_t)w.e_max);
        w.off_si = w.off_cnt + round_up(sizeof(int) * 8);
        w.off_st = w.off_si + round_up(sizeof(int) * 4 * (size_t)nseq);
        w.off_m = w.off_st + round_up(sizeof(float) * (size_t)w.e_max * p.H * kv);
        w.off_s = w.off_m + round_up(sizeof(float) * (size_t)w.e_max * p.H * kk);
        w.total = w.off_s + round_up(sizeof(float) * (size_t)w.e_max * p.H * kv);
    }
    return w;
}

gdn_status check_varlen(const gdn_problem* p, int nseq) {
    if (!p) return GDN_ERR_INVALID_ARG;
    if (p->B != 1 || p->H < 1 || p->T < 0 || nseq < 1) return GDN_ERR_INVALID_ARG;
    if (p->chunk != gdn::kChunk) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (p->decay_first != 0 && p->decay_first != 1) return GDN_ERR_INVALID_ARG;
    if (p->gate_k != 0 && p->gate_k != 1) return GDN_ERR_INVALID_ARG;
    if (p->K != p->V || (p->K != 64 && p->K != 128)) return GDN_ERR_UNSUPPORTED_SHAPE;
    if ((p->in_dtype != GDN_DTYPE_F32 && p->in_dtype != GDN_DTYPE_BF16) ||
        (p->out_dtype != GDN_DTYPE_F32 && p->out_dtype != GDN_DTYPE_BF16))
        return GDN_ERR_UNSUPPORTED_DTYPE;
    if ((long long)p->T * p->H * p->K >= (1LL << 40)) return GDN_ERR_UNSUPPORTED_SHAPE;
    if ((long long)p->T + 64LL * ((long long)nseq + 1) >= (1LL << 31)) return GDN_ERR_UNSUPPORTED_SHAPE;
    if ((long long)nseq * p->H >= (1LL << 31) ||
        (long long)p->H * (p->T / gdn::kChunk + nseq) >= (1LL << 31))
        return GDN_ERR_UNSUPPORTED_SHAPE;
    return GDN_OK;
}

// ---- backward: [the forward's / summary's workspace (header first) | o scratch | Hc | Dc | M |
//      S | dS | dH_in (P + 1 slots)], each region 256-byte aligned, P the most pieces
//      bwd_pieces gives on any device. Hc and Dc hold the state entering and the state gradient
//      leaving every chunk ([T/64][B][H][K][V] fp32).
struct BwdLayout {
    size_t off_o, off_hc, off_dc, off_m, off_s, off_ds, off_dh, total;
};

// Pieces of the backward's state-gradient chains. Each (b, h, piece, column tile) is one chain
// and runs one CTA per SM. When the chains of whole sequences fit in one wave, one pass from dht
// gives the gradient leaving every chunk and dh0 (P = 1); otherwise P is the largest power of two
// dividing the chunk count with B*H*tiles*P chains per wave: a first pass gives each piece's
// dS_local, the reverse scan over the piece summaries the gradient leaving each piece, and a
// second pass the gradient leaving every chunk. `sms` is the SM count (capped at
// kBwdSmBound, which sizes the workspace for any device).
constexpr int kBwdSmBound = 256;
int bwd_pieces(const gdn_problem& p, int sms) {
    const int nch = p.T / gdn::kChunk;
    const long long chains =
        (long long)p.B * p.H * (p.V / gdn::state_grad_tile(p.in_dtype == GDN_DTYPE_BF16));
    sms = std::min(sms, kBwdSmBound);
    int P = 1;
    while (nch > 0 && nch % (2 * P) == 0 && chains * 2 * P <= sms) P *= 2;
    return P;
}

BwdLayout bwd_layout(const gdn_problem& p, int nseg_api) {
    (void)nseg_api;   // the backward's own piece count sizes the per-piece arrays
    const int nseg = bwd_pieces(p, kBwdSmBound);
    BwdLayout w{};
    const int nch = p.T / gdn::kChunk;
    const size_t head = std::max(layout(p, nch > 0 ? nch : 1).total, layout(p, 1).total);
    const size_t bh = (size_t)p.B * p.H, kv = (size_t)p.K * p.V, kk = (size_t)p.K * p.K;
    const size_t osz = p.out_dtype == GDN_DTYPE_BF16 ? 2 : 4;
    w.off_o = round_up(head);
    w.off_hc = w.off_o + round_up((size_t)p.B * p.T * p.H * p.V * osz);
    w.off_dc = w.off_hc + round_up(sizeof(float) * nch * bh * kv);
    w.off_m = w.off_dc + round_up(sizeof(float) * nch * bh * kv);
    w.off_s = w.off_m + round_up(sizeof(float) * nseg * bh * kk);
    w.off_ds = w.off_s + round_up(sizeof(float) * nseg * bh * kv);
    w.off_dh = w.off_ds + round_up(sizeof(float) * nseg * bh * kv);
    w.total = w.off_dh + round_up(sizeof(float) * (nseg + 1) * bh * kv);
    return w;
}

gdn_status check_bwd(const gdn_problem* p, int nseg) {
    gdn_status st = check_problem(p, nseg);
    if (st != GDN_OK) return st;
    if (p->gate_k) return GDN_ERR_UNSUPPORTED_SHAPE;
    if ((long long)p->B * p->H * nseg * (p->V / 32) >= (1LL << 31) ||
        (long long)p->B * p->H * (p->T / gdn::kChunk) >= (1LL << 31))
        return GDN_ERR_UNSUPPORTED_SHAPE;
    return GDN_OK;
}

}  // namespace

extern "C" {

size_t gdn_workspace_bytes(const gdn_problem* p, int nseg) {
    if (check_problem(p, nseg) != GDN_OK) return 0;
    return layout(*p, nseg).total;
}

int gdn_segmented_pieces(const gdn_problem* p, int nseg) {
    if (check_problem(p, nseg) != GDN_OK) return 0;
    return plan_pieces(*p, nseg).P;
}

gdn_status gdn_chunk_fwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                         const void* g, const void* beta, const float* h0, void* o,
                         float* h_final, void* workspace, size_t workspace_bytes,
                         void* stream) {
    gdn_status st = check_problem(p, 1);
    if (st != GDN_OK) return st;
    if (p->T > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_INVALID_ARG;
    if ((st = check_workspace(p, 1, workspace, workspace_bytes)) != GDN_OK) return st;
    for (const void* ptr : {q, k, v, g, beta, (const void*)h0, (const void*)o,
                            (const void*)h_final})
        if (misaligned(ptr)) return GDN_ERR_MISALIGNED;
    if ((st = check_device()) != GDN_OK) return st;
    return run_segmented(p, 1, q, k, v, g, beta, h0, o, h_final, nullptr, workspace,
                         reinterpret_cast<cudaStream_t>(stream), nullptr);
}

int gdn_segmented_plan(const gdn_problem* p, int nseg, int* first_chunks, int* rest_chunks) {
    if (first_chunks) *first_chunks = 0;
    if (rest_chunks) *rest_chunks = 0;
    if (check_problem(p, nseg) != GDN_OK) return 0;
    const PiecePlan plan = plan_pieces(*p, nseg);
    if (first_chunks) *first_chunks = plan.first;
    if (rest_chunks) *rest_chunks = plan.rest;
    return plan.P;
}

gdn_status gdn_segment_fwd(const gdn_problem* p, int nseg, const void* q, const void* k,
                           const void* v, const void* g, const void* beta, const float* H_in,
                           void* o, float* h_final, void* workspace, size_t workspace_bytes,
                           void* stream) {
    gdn_status st = check_problem(p, nseg);
    if (st != GDN_OK) return st;
    if (p->T > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_INVALID_ARG;
    if ((st = check_workspace(p, 1, workspace, workspace_bytes)) != GDN_OK) return st;
    for (const void* ptr : {q, k, v, g, beta, (const void*)H_in, (const void*)o,
                            (const void*)h_final})
        if (misaligned(ptr)) return GDN_ERR_MISALIGNED;
    if ((st = check_device()) != GDN_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int BH = p->B * p->H;
    if (p->T == 0) {
        // no tokens: the state leaving the last segment is the state entering it
        if (!h_final) return GDN_OK;
        const float* last = H_in ? H_in + (long long)(nseg - 1) * BH * p->K * p->V : nullptr;
        return from_cuda(gdn::launch_scan(nullptr, nullptr, last, nullptr, h_final, nullptr, 0, 1,
                                          1, BH, p->K, p->V, s));
    }
    ChainParams c = base_params(p, workspace);
    c.q = q;
    c.k = k;
    c.v = v;
    c.g = g;
    c.beta = beta;
    c.o = o;
    c.h_start = H_in;
    c.h_start_seg_stride = (long long)BH * p->K * p->V;
    c.h_final = h_final;
    c.seg_len = p->T / nseg;
    c.seg_first = 0;
    c.nseg_run = nseg;
    c.nseg_total = nseg;
    cudaError_t e = prepare(c, p, workspace, s);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    return from_cuda(run_forward(c, s));
}

gdn_status gdn_segment_summary(const gdn_problem* p, int nseg, const void* k, const void* v,
                               const void* g, const void* beta, float* M, float* S,
                               void* workspace, size_t workspace_bytes, void* stream) {
    gdn_status st = check_problem(p, nseg);
    if (st != GDN_OK) return st;
    if (!M || !S) return GDN_ERR_INVALID_ARG;
    if (p->T > 0 && (!k || !v || !g || !beta)) return GDN_ERR_INVALID_ARG;
    if ((st = check_workspace(p, 1, workspace, workspace_bytes)) != GDN_OK) return st;
    for (const void* ptr : {k, v, g, beta, (const void*)M, (const void*)S})
        if (misaligned(ptr)) return GDN_ERR_MISALIGNED;
    if ((st = check_device()) != GDN_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ChainParams c = base_params(p, workspace);
    c.k = k;
    c.v = v;
    c.g = g;
    c.beta = beta;
    c.M = M;
    c.S = S;
    c.seg_len = p->T / nseg;
    c.nseg_run = nseg;
    c.nseg_total = nseg;
    if (p->T == 0) return from_cuda(run_summary(c, s));
    cudaError_t e = prepare(c, p, workspace, s);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    return from_cuda(run_summary(c, s));
}

gdn_status gdn_summary_scan(const gdn_problem* p, int nseg, const float* M, const float* S,
                            const float* h0, float* H_in, void* stream) {
    if (!p || nseg < 1 || p->B < 1 || p->H < 1) return GDN_ERR_INVALID_ARG;
    if (p->K != p->V || (p->K != 64 && p->K != 128)) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (!H_in || (nseg > 1 && (!M || !S))) return GDN_ERR_INVALID_ARG;
    if ((long long)p->B * p->H >= (1LL << 31)) return GDN_ERR_UNSUPPORTED_SHAPE;
    for (const void* ptr : {(const void*)M, (const void*)S, (const void*)h0, (const void*)H_in})
        if (misaligned(ptr)) return GDN_ERR_MISALIGNED;
    gdn_status st = check_device();
    if (st != GDN_OK) return st;
    return from_cuda(gdn::launch_scan(nseg > 1 ? M : nullptr, nseg > 1 ? S : nullptr, h0, nullptr,
                                      H_in, nullptr, 0, nseg, 1, p->B * p->H, p->K, p->V,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

gdn_status gdn_segmented_fwd(const gdn_problem* p, int nseg, const void* q, const void* k,
                             const void* v, const void* g, const void* beta, const float* h0,
                             void* o, float* h_final, float* H_in_out, void* workspace,
                             size_t workspace_bytes, void* stream) {
    return gdn_segmented_fwd_timed(p, nseg, q, k, v, g, beta, h0, o, h_final, H_in_out,
                                   workspace, workspace_bytes, stream, nullptr);
}

gdn_status gdn_segmented_fwd_timed(const gdn_problem* p, int nseg, const void* q,
                                   const void* k, const void* v, const void* g,
                                   const void* beta, const float* h0, void* o, float* h_final,
                                   float* H_in_out, void* workspace, size_t workspace_bytes,
                                   void* stream, void* const* stage_events) {
    gdn_status st = check_problem(p, nseg);
    if (st != GDN_OK) return st;
    if (p->T > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_INVALID_ARG;
    if ((st = check_workspace(p, nseg, workspace, workspace_bytes)) != GDN_OK) return st;
    for (const void* ptr : {q, k, v, g, beta, (const void*)h0, (const void*)o,
                            (const void*)h_final, (const void*)H_in_out})
        if (misaligned(ptr)) return GDN_ERR_MISALIGNED;
    if ((st = check_device()) != GDN_OK) return st;
    return run_segmented(p, nseg, q, k, v, g, beta, h0, o, h_final, H_in_out, workspace,
                         reinterpret_cast<cudaStream_t>(stream), stage_events);
}

size_t gdn_varlen_workspace_bytes(const gdn_problem* p, int nseq) {
    if (check_varlen(p, nseq) != GDN_OK) return 0;
    return varlen_layout(*p, nseq).total;
}

gdn_status gdn_varlen_fwd(const gdn_problem* p, int nseq, const int* cu_seqlens, const void* q,
                          const void* k, const void* v, const void* g, const void* beta,
                          const float* h0, void* o, float* h_final, void* workspace,
                          size_t workspace_bytes, void* stream) {
    return gdn_varlen_fwd_timed(p, nseq, cu_seqlens, q, k, v, g, beta, h0, o, h_final, workspace,
                                workspace_bytes, stream, nullptr);
}

gdn_status gdn_varlen_fwd_timed(const gdn_problem* p, int nseq, const int* cu_seqlens,
                                const void* q, const void* k, const void* v, const void* g,
                                const void* beta, const float* h0, void* o, float* h_final,
                                void* workspace, size_t workspace_bytes, void* stream,
                                void* const* stage_events) {
    gdn_status st = check_varlen(p, nseq);
    if (st != GDN_OK) return st;
    if (!cu_seqlens) return GDN_ERR_INVALID_ARG;
    if (p->T > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_INVALID_ARG;
    const VarlenLayout w = varlen_layout(*p, nseq);
    if (!workspace || workspace_bytes < w.total) return GDN_ERR_WORKSPACE;
    for (const void* ptr : {(const void*)workspace, (const void*)cu_seqlens, q, k, v, g, beta,
                            (const void*)h0, (const void*)o, (const void*)h_final})
        if (misaligned(ptr)) return GDN_ERR_MISALIGNED;
    if ((st = check_device()) != GDN_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char* wsb = reinterpret_cast<char*>(workspace);
    int* cu = reinterpret_cast<int*>(wsb + w.off_cu);
    int* cc = reinterpret_cast<int*>(wsb + w.off_cc);
    ChainParams c = base_params(p, workspace);
    c.B = nseq;   // one chain per (sequence, head), or per piece below
    c.q = q;
    c.k = k;
    c.v = v;
    c.g = g;
    c.beta = beta;
    c.o = o;
    c.h_start = h0;
    c.h_final = h_final;
    c.seg_first = 0;
    c.nseg_run = 1;
    c.nseg_total = 1;
    c.cu_seqlens = cu;
    c.cu_chunks = cc;
    c.total_chunks = w.chunk_bound;
    c.wy = wsb + w.off_wy;
    const bool tc = use_tc(c) && p->T >= gdn::kChunk;   // (a tensor map box holds 64 tokens)
    const int sms = std::min(sm_count(), kPieceSmBound);
    const bool pieces = tc && w.pieces && gdn::pieces_possible(p->T, nseq, p->H, sms);
    // long sequences cut into pieces for the tcgen05 chains (gdn_varlen.cu): the plan's tables
    gdn::PiecePlan pl{};
    if (pieces) {
        pl.tab1f = reinterpret_cast<int*>(wsb + w.off_t1f);
        pl.tab1s = reinterpret_cast<int*>(wsb + w.off_t1s);
        pl.tab2 = reinterpret_cast<int*>(wsb + w.off_t2);
        pl.counts = reinterpret_cast<int*>(wsb + w.off_cnt);
        pl.seqinfo = reinterpret_cast<int*>(wsb + w.off_si);
    }
    // the chains read the checked copy of the lengths, never the caller's array; the plan, when
    // a cut is possible, is made in the same block right after the check
    if (mark(stage_events, 0, s) != cudaSuccess) return GDN_ERR_CUDA;
    gdn::DeviceError* derr = reinterpret_cast<gdn::DeviceError*>(workspace);
    if ((pieces ? gdn::launch_varlen_meta_plan(cu_seqlens, nseq, p->T, cu, cc, derr, p->H, sms,
                                               w.e_max, pl, s)
                : gdn::launch_varlen_meta(cu_seqlens, nseq, p->T, cu, cc, derr, s)) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (tc && gdn::launch_tc_wy(c, s) != cudaSuccess) return GDN_ERR_CUDA;
    if (kda_prep_shape(*p) && p->T > 0 && gdn::launch_kda_prep(c, s) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (!pieces) {
        if (mark(stage_events, 1, s) != cudaSuccess || mark(stage_events, 2, s) != cudaSuccess ||
            mark(stage_events, 3, s) != cudaSuccess)
            return GDN_ERR_CUDA;
        if ((tc ? gdn::launch_tc_forward(c, s) : gdn::launch_simt_forward(c, s)) != cudaSuccess)
            return GDN_ERR_CUDA;
        return from_cuda(mark(stage_events, 4, s));
    }
    float* states = reinterpret_cast<float*>(wsb + w.off_st);
    float* Mp = reinterpret_cast<float*>(wsb + w.off_m);
    float* Sp = reinterpret_cast<float*>(wsb + w.off_s);
    c.piece_states = states;
    // 1. piece 0 of every sequence (the whole sequence when it is not cut) beside the summaries
    //    of the middle pieces, launched as its programmatic dependent
    if (mark(stage_events, 1, s) != cudaSuccess) return GDN_ERR_CUDA;
    ChainParams f1 = c;
    f1.piece_tab = pl.tab1f;
    f1.piece_n = pl.counts;
    // (the plan keeps each phase within sms / H entries: the summaries and the second phase's
    // entries are at most that many)
    const int phase_entries = std::max(1, std::min(w.e_max, sms / p->H));
    ChainParams s1 = c;
    s1.B = phase_entries;
    s1.piece_tab = pl.tab1s;
    s1.piece_n = pl.counts + 1;
    s1.M = Mp;
    s1.S = Sp;
    s1.h_start = nullptr;
    s1.h_final = nullptr;
    s1.launch_dependent = 1;
    if (gdn::launch_tc_forward(f1, s) != cudaSuccess || gdn::launch_tc_summary(s1, s) != cudaSuccess)
        return GDN_ERR_CUDA;
    // 2. the states entering pieces 2 .. k-1 of every cut sequence (the summary grid's
    //    programmatic dependent)
    if (mark(stage_events, 2, s) != cudaSuccess) return GDN_ERR_CUDA;
    if (gdn::launch_piece_scan(pl, nseq, p->H, w.e_max, sms, Mp, Sp, states, s) != cudaSuccess)
        return GDN_ERR_CUDA;
    // 3. pieces 1 .. k-1 from their states (the scan's programmatic dependent: its chains set
    //    up while the scan runs and wait for it before they read a state)
    if (mark(stage_events, 3, s) != cudaSuccess) return GDN_ERR_CUDA;
    ChainParams f2 = c;
    f2.B = phase_entries;
    f2.piece_tab = pl.tab2;
    f2.piece_n = pl.counts + 2;
    f2.launch_dependent = 1;
    if (gdn::launch_tc_forward(f2, s) != cudaSuccess) return GDN_ERR_CUDA;
    return from_cuda(mark(stage_events, 4, s));
}

gdn_status gdn_state_grad_summary(const gdn_problem* p, int nseg, const void* q, const void* k,
                                  const void* g, const void* beta, const void* dO,
                                  const float* dH_end, float* dS, void* stream) {
    gdn_status st = check_problem(p, nseg);
    if (st != GDN_OK) return st;
    if (p->gate_k) return GDN_ERR_UNSUPPORTED_SHAPE;
    // one CTA per (b, h, segment, 32-column tile) on a one-dimensional grid
    if ((long long)p->B * p->H * nseg * (p->V / 32) >= (1LL << 31)) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (!dS) return GDN_ERR_INVALID_ARG;
    if (p->T > 0 && (!q || !k || !g || !beta || !dO)) return GDN_ERR_INVALID_ARG;
    for (const void* ptr : {q, k, g, beta, dO, (const void*)dH_end, (const void*)dS})
        if (misaligned(ptr)) return GDN_ERR_MISALIGNED;
    if ((st = check_device()) != GDN_OK) return st;
    gdn::StateGradParams c{};
    c.q = q;
    c.k = k;
    c.g = g;
    c.beta = beta;
    c.dO = dO;
    c.dH_end = dH_end;
    c.dS = dS;
    c.B = p->B;
    c.T = p->T;
    c.H = p->H;
    c.K = p->K;
    c.V = p->V;
    c.seg_len = p->T / nseg;
    c.nseg = nseg;
    c.in_bf16 = p->in_dtype == GDN_DTYPE_BF16;
    c.do_bf16 = p->out_dtype == GDN_DTYPE_BF16;
    c.decay_first = p->decay_first;
    return from_cuda(gdn::launch_state_grad(c, reinterpret_cast<cudaStream_t>(stream)));
}

gdn_status gdn_state_grad_scan(const gdn_problem* p, int nseg, const float* M, const float* dS,
                               const float* dht, float* dH_in, void* stream) {
    if (!p || nseg < 1 || p->B < 1 || p->H < 1) return GDN_ERR_INVALID_ARG;
    if (p->K != p->V || (p->K != 64 && p->K != 128)) return GDN_ERR_UNSUPPORTED_SHAPE;
    if (!M || !dS || !dH_in) return GDN_ERR_INVALID_ARG;
    if ((long long)p->B * p->H >= (1LL << 31)) return GDN_ERR_UNSUPPORTED_SHAPE;
    for (const void* ptr : {(const void*)M, (const void*)dS, (const void*)dht, (const void*)dH_in})
        if (misaligned(ptr)) return GDN_ERR_MISALIGNED;
    gdn_status st = check_device();
    if (st != GDN_OK) return st;
    return from_cuda(gdn::launch_state_grad_scan(M, dS, dht, dH_in, nseg, p->B * p->H, p->K, p->V,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

size_t gdn_chunk_bwd_workspace_bytes(const gdn_problem* p, int nseg) {
    if (check_bwd(p, nseg) != GDN_OK) return 0;
    return bwd_layout(*p, nseg).total;
}

gdn_status gdn_chunk_bwd(const gdn_problem* p, int nseg, const void* q, const void* k,
                         const void* v, const void* g, const void* beta, const float* h0,
                         const void* dO, const float* dht, float* dq, float* dk, float* dv,
                         float* dg, float* dbeta, float* dh0, void* workspace,
                         size_t workspace_bytes, void* stream) {
    return gdn_chunk_bwd_timed(p, nseg, q, k, v, g, beta, h0, dO, dht, dq, dk, dv, dg, dbeta,
                               dh0, workspace, workspace_bytes, stream, nullptr);
}

gdn_status gdn_chunk_bwd_timed(const gdn_problem* p, int nseg, const void* q, const void* k,
                               const void* v, const void* g, const void* beta, const float* h0,
                               const void* dO, const float* dht, float* dq, float* dk, float* dv,
                               float* dg, float* dbeta, float* dh0, void* workspace,
                               size_t workspace_bytes, void* stream, void* const* stage_events) {
    void* const* ev = stage_events;
    gdn_status st = check_bwd(p, nseg);
    if (st != GDN_OK) return st;
    if (p->T > 0 && (!q || !k || !v || !g || !beta || !dO || !dq || !dk || !dv || !dg || !dbeta))
        return GDN_ERR_INVALID_ARG;
    const BwdLayout w = bwd_layout(*p, nseg);
    if (!workspace || workspace_bytes < w.total) return GDN_ERR_WORKSPACE;
    for (const void* ptr : {(const void*)workspace, q, k, v, g, beta, (const void*)h0, dO, (const void*)dht,
                            (const void*)dq, (const void*)dk, (const void*)dv, (const void*)dg,
                            (const void*)dbeta, (const void*)dh0})
        if (misaligned(ptr)) return GDN_ERR_MISALIGNED;
    if ((st = check_device()) != GDN_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int BH = p->B * p->H;
    const long long kv = (long long)BH * p->K * p->V;
    if (p->T == 0) {   // dh0 = dht (or zeros)
        if (dh0 && gdn::launch_scan(nullptr, nullptr, dht, nullptr, dh0, nullptr, 0, 1, 1, BH,
                                    p->K, p->V, s) != cudaSuccess)
            return GDN_ERR_CUDA;
        return GDN_OK;
    }
    char* wsb = reinterpret_cast<char*>(workspace);
    float* Hc = reinterpret_cast<float*>(wsb + w.off_hc);
    float* Dc = reinterpret_cast<float*>(wsb + w.off_dc);
    float* M = reinterpret_cast<float*>(wsb + w.off_m);
    float* S = reinterpret_cast<float*>(wsb + w.off_s);
    float* dS = reinterpret_cast<float*>(wsb + w.off_ds);
    float* dH = reinterpret_cast<float*>(wsb + w.off_dh);   // [P + 1]: entering piece s; dht last
    const int nch = p->T / gdn::kChunk;
    // 1. the state entering every chunk: the forward with one segment per chunk (its output is
    //    recomputed into scratch and not used)
    if (mark(ev, 0, s) != cudaSuccess) return GDN_ERR_CUDA;
    st = run_segmented(p, nch, q, k, v, g, beta, h0, wsb + w.off_o, nullptr, Hc, workspace, s,
                       nullptr);
    if (st != GDN_OK) return st;
    if (mark(ev, 1, s) != cudaSuccess) return GDN_ERR_CUDA;
    // 2-4. the gradient leaving every chunk (Dc) and dh0 (RFC 6.4.3: dS_local per piece, the
    //      reverse scan dH_in = M^T dH_out + dS_local, then each piece's chunks again)
    const int P = bwd_pieces(*p, sm_count());
    gdn::StateGradParams sg{};
    sg.q = q;
    sg.k = k;
    sg.g = g;
    sg.beta = beta;
    sg.dO = dO;
    sg.B = p->B;
    sg.T = p->T;
    sg.H = p->H;
    sg.K = p->K;
    sg.V = p->V;
    sg.in_bf16 = p->in_dtype == GDN_DTYPE_BF16;
    sg.do_bf16 = p->out_dtype == GDN_DTYPE_BF16;
    sg.decay_first = p->decay_first;
    // on the tensor-core path the forward above left every chunk's WY tiles in the workspace:
    // the state-gradient chains take A diag(beta exp(Gx)) from them instead of inverting
    if (tc_shape(*p) && gdn::tc_runtime_ok()) sg.wy = wsb + layout(*p, 1).off_wy;
    if (P == 1) {
        // the chains of whole sequences fill at most one wave: one pass from dht (no summaries;
        // the stage events of the summaries and of the second pass mark empty stages)
        sg.seg_len = p->T;
        sg.nseg = 1;
        sg.dH_end = dht;
        sg.dS = dh0 ? dh0 : dS;
        sg.D_chunks = Dc;
        if (mark(ev, 2, s) != cudaSuccess || gdn::launch_state_grad(sg, s) != cudaSuccess ||
            mark(ev, 3, s) != cudaSuccess ||
            mark(ev, 4, s) != cudaSuccess)
            return GDN_ERR_CUDA;
    } else {
        // the pieces' summaries M (their linear parts carry the state gradient backwards)
        ChainParams c = base_params(p, workspace);
        c.k = k;
        c.v = v;
        c.g = g;
        c.beta = beta;
        c.M = M;
        c.S = S;
        c.seg_len = p->T / P;
        c.nseg_run = P;
        c.nseg_total = P;
        if (prepare(c, p, workspace, s) != cudaSuccess || run_summary(c, s) != cudaSuccess)
            return GDN_ERR_CUDA;
        // dS_local of every piece, and the reverse scan to the gradient entering every piece;
        // dH[P] = dht
        sg.seg_len = p->T / P;
        sg.nseg = P;
        sg.dS = dS;
        if (mark(ev, 2, s) != cudaSuccess || gdn::launch_state_grad(sg, s) != cudaSuccess)
            return GDN_ERR_CUDA;
        if (gdn::launch_scan(nullptr, nullptr, dht, nullptr, dH + P * kv, nullptr, 0, 1, 1, BH,
                             p->K, p->V, s) != cudaSuccess ||
            gdn::launch_state_grad_scan(M, dS, dht, dH, P, BH, p->K, p->V, s) != cudaSuccess)
            return GDN_ERR_CUDA;
        if (dh0 && cudaMemcpyAsync(dh0, dH, sizeof(float) * kv, cudaMemcpyDeviceToDevice, s) !=
                       cudaSuccess)
            return GDN_ERR_CUDA;
        // each piece's chunks again from the gradient leaving it, recording the gradient on
        // the state leaving every chunk (RFC 6.4.3 backward_state)
        sg.dH_end = dH + kv;
        sg.D_chunks = Dc;
        if (mark(ev, 3, s) != cudaSuccess || gdn::launch_state_grad(sg, s) != cudaSuccess ||
            mark(ev, 4, s) != cudaSuccess)
            return GDN_ERR_CUDA;
    }
    // 5. every chunk's gradients (RFC 6.4.3 backward_finish)
    gdn::ChunkGradParams cg{};
    cg.q = q;
    cg.k = k;
    cg.v = v;
    cg.g = g;
    cg.beta = beta;
    cg.dO = dO;
    cg.Hc = Hc;
    cg.Dc = Dc;
    cg.dq = dq;
    cg.dk = dk;
    cg.dv = dv;
    cg.dg = dg;
    cg.dbeta = dbeta;
    cg.B = p->B;
    cg.T = p->T;
    cg.H = p->H;
    cg.K = p->K;
    cg.V = p->V;
    cg.in_bf16 = p->in_dtype == GDN_DTYPE_BF16;
    cg.do_bf16 = p->out_dtype == GDN_DTYPE_BF16;
    cg.decay_first = p->decay_first;
    if (gdn::launch_chunk_grad(cg, s) != cudaSuccess || mark(ev, 5, s) != cudaSuccess)
        return GDN_ERR_CUDA;
    return GDN_OK;
}

const char* gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "ok";
        case GDN_ERR_INVALID_ARG: return "invalid argument";
        case GDN_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case GDN_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
        case GDN_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
        case GDN_ERR_WORKSPACE: return "workspace missing or too small";
        case GDN_ERR_CUDA: return "CUDA error";
        case GDN_ERR_TIMEOUT: return "a kernel's bounded wait ran out";
        case GDN_ERR_DEVICE: return "current device is not an sm_103 GPU";
    }
    return "unknown status";
}

gdn_status gdn_selftest_wait_timeout(void* workspace, long long limit_cycles, void* stream) {
    if (!workspace) return GDN_ERR_WORKSPACE;
    if (limit_cycles < 1 || limit_cycles > (1LL << 32)) return GDN_ERR_INVALID_ARG;
    if (misaligned(workspace)) return GDN_ERR_MISALIGNED;
    gdn_status st = check_device();
    if (st != GDN_OK) return st;
    return from_cuda(gdn::launch_wait_selftest(reinterpret_cast<gdn::DeviceError*>(workspace),
                                                limit_cycles, kSelftestTag,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

gdn_status gdn_check_device_error(void* workspace, void* stream, unsigned* detail) {
    if (detail) *detail = 0;
    if (!workspace) return GDN_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    gdn::DeviceError host{};
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaMemcpyAsync(&host, workspace, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
    if (host.code == 0) return GDN_OK;
    if (detail) *detail = host.detail;
    if (cudaMemsetAsync(workspace, 0, sizeof(host), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (host.code == GDN_ERR_TIMEOUT || host.code == GDN_ERR_INVALID_ARG)
        return static_cast<gdn_status>(host.code);
    return GDN_ERR_CUDA;
}

}  // extern "C"
