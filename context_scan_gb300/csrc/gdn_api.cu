// gdn_api.cu -- the C ABI (include/gdn.h): argument validation, workspace layout and the
// launch sequence on the caller's stream. No allocation, no synchronisation (except
// gdn_check_device_error), no CPU fallback.
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

using gdn::ChainParams;

constexpr size_t kHeaderBytes = 256;   // device error word lives here
constexpr size_t kAlign = 256;
constexpr int kMaxSub = 2;             // summary sub-segments per segment (segmented forward)

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct WsLayout {
    size_t off_wy, off_M, off_S, off_Hin, total;
};

// Shapes that take the tcgen05 kernels (which also need the per-chunk WY tiles).
bool tc_shape(const gdn_problem& p) {
    return p.in_dtype == GDN_DTYPE_BF16 && p.K == 128 && p.V == 128;
}

// [header | WY tiles (tcgen05 shapes) | M | S | H_in (nseg > 1)]; M and S hold up to
// kMaxSub sub-segment summaries per segment
WsLayout layout(const gdn_problem& p, int nseg) {
    WsLayout w{};
    const size_t bh = (size_t)p.B * p.H;
    w.off_wy = kHeaderBytes;
    const size_t wy_bytes = tc_shape(p) ? bh * (size_t)(p.T / gdn::kChunk) * 16384u : 0;
    w.off_M = w.off_wy + round_up(wy_bytes);
    if (nseg <= 1) {
        w.total = w.off_M;
        return w;
    }
    w.off_S = w.off_M + round_up(sizeof(float) * kMaxSub * nseg * bh * p.K * p.K);
    w.off_Hin = w.off_S + round_up(sizeof(float) * kMaxSub * nseg * bh * p.K * p.V);
    w.total = w.off_Hin + round_up(sizeof(float) * nseg * bh * p.K * p.V);
    return w;
}

bool misaligned(const void* ptr) { return ptr && (reinterpret_cast<uintptr_t>(ptr) & 15u); }

gdn_status check_problem(const gdn_problem* p, int nseg) {
    if (!p) return GDN_ERR_INVALID_ARG;
    if (p->B < 1 || p->H < 1 || p->T < 0) return GDN_ERR_INVALID_ARG;
    if (nseg < 1) return GDN_ERR_INVALID_ARG;
    if (p->chunk != gdn::kChunk) return GDN_ERR_UNSUPPORTED_SHAPE;
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
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (major != 10 || minor != 3) return GDN_ERR_DEVICE;
    return GDN_OK;
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
    c.err = reinterpret_cast<gdn::DeviceError*>(ws);
    return c;
}

bool use_tc(const ChainParams& c) { return c.T > 0 && gdn::tc_supported(c); }

// Sub-segments per segment for the segmented forward's summaries. The summary launch has
// one CTA per (b, h, segment) and a CTA per SM; when B*H*(nseg-1) CTAs fill the last wave
// poorly, splitting every segment in two (composed again by the scan) balances the waves.
// Kept at 1 unless the split raises the wave efficiency and the halves keep >= 16 chunks.
int summary_split(const ChainParams& c, int nseg) {
    if (!use_tc(c) || nseg < 2) return 1;
    const int chunks = c.T / nseg / gdn::kChunk;
    if (chunks % 2 != 0 || chunks / 2 < 16) return 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return 1;
    const double units = (double)c.B * c.H * (nseg - 1);
    auto eff = [&](double u) { return u / (std::ceil(u / sms) * sms); };
    return eff(2.0 * units) > eff(units) + 0.05 ? 2 : 1;
}

// The tcgen05 chains read every chunk's WY tiles from the workspace: form them first (one
// launch for all chunks of the problem). Nothing to do on the CUDA-core path.
cudaError_t prepare(ChainParams& c, const gdn_problem* p, void* ws, cudaStream_t s) {
    c.wy = reinterpret_cast<char*>(ws) + layout(*p, 1).off_wy;
    return use_tc(c) ? gdn::launch_tc_wy(c, s) : cudaSuccess;
}

cudaError_t run_forward(const ChainParams& c, cudaStream_t s) {
    return use_tc(c) ? gdn::launch_tc_forward(c, s) : gdn::launch_simt_forward(c, s);
}

cudaError_t run_summary(const ChainParams& c, cudaStream_t s) {
    return use_tc(c) ? gdn::launch_tc_summary(c, s) : gdn::launch_simt_summary(c, s);
}

}  // namespace

extern "C" {

size_t gdn_workspace_bytes(const gdn_problem* p, int nseg) {
    if (check_problem(p, nseg) != GDN_OK) return 0;
    return layout(*p, nseg).total;
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
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ChainParams c = base_params(p, workspace);
    c.q = q;
    c.k = k;
    c.v = v;
    c.g = g;
    c.beta = beta;
    c.h_start = h0;
    c.h_start_seg_stride = 0;
    c.o = o;
    c.h_final = h_final;
    c.seg_len = p->T;
    c.nseg_run = 1;
    c.nseg_total = 1;
    if (p->T == 0) {
        // nothing to process: h_final = h0 (or zeros)
        if (!h_final) return GDN_OK;
        return from_cuda(gdn::launch_scan(nullptr, nullptr, h0, h_final, 1, p->B * p->H, p->K,
                                          p->V, s));
    }
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
    return from_cuda(gdn::launch_scan(M, S, h0, H_in, nseg, p->B * p->H, p->K, p->V,
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
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const WsLayout w = layout(*p, nseg);
    char* wsb = reinterpret_cast<char*>(workspace);
    const int BH = p->B * p->H;

    if (nseg == 1) {
        if (mark(stage_events, 0, s) != cudaSuccess || mark(stage_events, 1, s) != cudaSuccess ||
            mark(stage_events, 2, s) != cudaSuccess)
            return GDN_ERR_CUDA;
        if (H_in_out) {
            cudaError_t e = gdn::launch_scan(nullptr, nullptr, h0, H_in_out, 1, BH, p->K, p->V, s);
            if (e != cudaSuccess) return GDN_ERR_CUDA;
        }
        if (mark(stage_events, 3, s) != cudaSuccess) return GDN_ERR_CUDA;
        st = gdn_chunk_fwd(p, q, k, v, g, beta, h0, o, h_final, workspace, workspace_bytes,
                           stream);
        if (st != GDN_OK) return st;
        return from_cuda(mark(stage_events, 4, s));
    }
    float* M = reinterpret_cast<float*>(wsb + w.off_M);
    float* S = reinterpret_cast<float*>(wsb + w.off_S);
    float* H_in = H_in_out ? H_in_out : reinterpret_cast<float*>(wsb + w.off_Hin);

    // 0. the WY tiles of every chunk (tcgen05 path only)
    if (mark(stage_events, 0, s) != cudaSuccess) return GDN_ERR_CUDA;
    ChainParams cw = base_params(p, workspace);
    cw.k = k;
    cw.g = g;
    cw.beta = beta;
    cw.seg_len = p->T / nseg;
    cudaError_t e = prepare(cw, p, workspace, s);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    // 1. summaries of segments 0..nseg-2 (the last segment's summary feeds nothing), each
    //    as nsub sub-segment summaries
    const int nsub = summary_split(cw, nseg);
    ChainParams cs = base_params(p, workspace);
    cs.wy = cw.wy;
    cs.k = k;
    cs.v = v;
    cs.g = g;
    cs.beta = beta;
    cs.M = M;
    cs.S = S;
    cs.seg_len = p->T / nseg / nsub;
    cs.nseg_run = (nseg - 1) * nsub;
    cs.nseg_total = nseg * nsub;
    if (mark(stage_events, 1, s) != cudaSuccess) return GDN_ERR_CUDA;
    e = run_summary(cs, s);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    // 2. exclusive in-order scan of the summaries
    if (mark(stage_events, 2, s) != cudaSuccess) return GDN_ERR_CUDA;
    e = gdn::launch_scan(M, S, h0, H_in, nseg, BH, p->K, p->V, s, nsub);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    if (mark(stage_events, 3, s) != cudaSuccess) return GDN_ERR_CUDA;
    // 3. every segment's forward from its scanned state
    ChainParams cf = base_params(p, workspace);
    cf.wy = cw.wy;
    cf.q = q;
    cf.k = k;
    cf.v = v;
    cf.g = g;
    cf.beta = beta;
    cf.h_start = H_in;
    cf.h_start_seg_stride = (long long)BH * p->K * p->V;
    cf.o = o;
    cf.h_final = h_final;
    cf.seg_len = p->T / nseg;
    cf.nseg_run = nseg;
    cf.nseg_total = nseg;
    e = run_forward(cf, s);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    return from_cuda(mark(stage_events, 4, s));
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
    return host.code == GDN_ERR_TIMEOUT ? GDN_ERR_TIMEOUT : GDN_ERR_CUDA;
}

}  // extern "C"
