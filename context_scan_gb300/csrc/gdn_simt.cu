// gdn_simt.cu -- fp32 CUDA-core kernels: the chunked forward, the segment summary and the
// exclusive summary scan.
//
// These run every problem whose inputs are fp32 (exact fp32 arithmetic, no tensor cores:
// the tensor cores' fp32 path would round operands to tf32) and bf16 problems with
// K == V == 64. Each CTA owns one chain (b, h, segment) and a tile of CT state columns;
// the columns of the state are independent, so tiles of one chain never communicate.
//
// Per chunk of 64 tokens (chunk equations of "Context Parallelism in ART", section 08,
// "First parallelize within a GPU", with the un-decayed read of "RFC: HyperParallel Linear
// Attention Context Parallel", section 2.1):
//   G_i  = inclusive cumsum of g inside the chunk, Gx_i = G_i - g_i
//   L    = diag(beta) P,  P[i,j] = exp(Gx_i - G_j) k_i.k_j  (j < i)
//   A    = (I + L)^{-1}                 -- blocked: 16x16 diagonal blocks by forward
//                                          substitution, then block forward substitution
//   R    = A diag(beta) (V - diag(exp(Gx)) K H)      (= U - W H of the WY form)
//   O    = diag(exp(G)) Q H + C R,  C[i,j] = exp(G_i - G_j) q_i.k_j  (j <= i)
//   H   <- exp(G_last) H + sum_j exp(G_last - G_j) k_j R_j
// The summary runs the same chunk step on the augmented K x (K+V) state [M | S], started
// from [I | 0] with value vectors [0 | v_t] (RFC section 2.2: S is the state reached from
// H_in = 0; M the linear part). Exponents are always differences of cumulative gates
// (never exp(-G)), so wide gate spreads cannot overflow.
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float load_in(const void* base, long long idx, int bf16) {
    if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
    return reinterpret_cast<const float*>(base)[idx];
}

__device__ __forceinline__ void store_out(void* base, long long idx, float x, int bf16) {
    if (bf16)
        reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(x);
    else
        reinterpret_cast<float*>(base)[idx] = x;
}

template <int KD, int CT, bool SUMMARY, bool GATEK>
struct SimtSmem {
    static constexpr int KP = KD + 1;  // padded row of k / q
    static constexpr int LP = 65;      // padded row of the 64x64 matrices
    static constexpr int off_k = 0;
    static constexpr int off_q = off_k + 64 * KP;
    static constexpr int off_v = off_q + (SUMMARY ? 0 : 64 * KP);
    static constexpr int off_h = off_v + 64 * CT;
    static constexpr int off_l = off_h + KD * CT;
    static constexpr int off_a = off_l + 64 * LP;
    static constexpr int off_c = off_a + 64 * LP;
    static constexpr int off_y = off_c + (SUMMARY ? 0 : 64 * LP);
    static constexpr int off_r = off_y + 64 * CT;
    static constexpr int off_s = off_r + 64 * CT;  // scalars: 6 x 64
    // per-channel gates: the chunk's cumulative gates G [64][KP] and a [64][KP] scratch
    static constexpr int off_gk = off_s + 6 * 64;
    static constexpr int off_ek = off_gk + (GATEK ? 64 * KP : 0);
    static constexpr int total = off_ek + (GATEK ? 64 * KP : 0);
    static constexpr size_t bytes = sizeof(float) * total;
};

// GATEK: per-channel gates ("KDA Chunk Backward -- TPU/Pallas Kernel Design", section 1.2):
// g is [B,T,H,K] and every quantity above takes the channel's own cumulative gate, e.g.
// P[i,j] = sum_l k_il k_jl exp(Gx_il - G_jl), the state rows decay by exp(G_last,l).
template <int KD, int CT, bool SUMMARY, bool GATEK>
__global__ void __launch_bounds__(kThreads) simt_chain_kernel(ChainParams p) {
    // a forward grid lets a grid launched as its programmatic dependent start right away
    if (!SUMMARY) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    using L = SimtSmem<KD, CT, SUMMARY, GATEK>;
    extern __shared__ float sm[];
    float* ks = sm + L::off_k;
    float* qs = sm + L::off_q;
    float* vs = sm + L::off_v;
    float* Hs = sm + L::off_h;
    float* Ls = sm + L::off_l;
    float* As = sm + L::off_a;
    float* Cs = sm + L::off_c;
    float* Ys = sm + L::off_y;
    float* Rs = sm + L::off_r;
    float* gam = sm + L::off_s;
    float* gx = gam + 64;
    float* bet = gx + 64;
    float* dk = bet + 64;   // exp(G_last - G_j)
    float* eq = dk + 64;    // exp(G_i)
    float* ekr = eq + 64;   // exp(Gx_i)
    float* Gk = sm + L::off_gk;   // per-channel cumulative gates [i][l] (GATEK)
    float* Ek = sm + L::off_ek;   // per-channel scaled keys [i][l] (GATEK)
    constexpr int KP = L::KP, LP = L::LP;

    const int tid = threadIdx.x;
    const int chain = blockIdx.x;
    const int seg = p.seg_first + chain % p.nseg_run;
    const int bh = chain / p.nseg_run;
    const int b = bh / p.H, h = bh % p.H;
    const int c0 = blockIdx.y * CT;   // first state column of this tile
    const int V = p.V, H = p.H, T = p.T;

    // ---- initial state tile
    for (int e = tid; e < KD * CT; e += kThreads) {
        const int l = e / CT, c = e % CT;
        float x = 0.f;
        if (SUMMARY) {
            x = (c0 + c == l) ? 1.f : 0.f;   // [I | 0]
        } else if (p.h_start) {
            x = p.h_start[(long long)seg * p.h_start_seg_stride +
                          ((long long)bh * KD + l) * V + c0 + c];
        }
        Hs[e] = x;
    }

    // tokens of this chain: a segment of the fixed-length batch, or a whole varlen sequence
    // whose last chunk may be partial (its padding tokens load as zeros with g = beta = 0,
    // which leaves the state untouched, and their outputs are not stored)
    const long long row_base = p.cu_seqlens ? (long long)p.cu_seqlens[b]
                                            : (long long)b * T + (long long)seg * p.seg_len;
    const int seq_tokens = p.cu_seqlens ? p.cu_seqlens[b + 1] - p.cu_seqlens[b] : p.seg_len;
    const int n_chunks = (seq_tokens + kChunk - 1) / kChunk;
    for (int ch = 0; ch < n_chunks; ++ch) {
        const int t0 = ch * kChunk;   // first token of the chunk inside the chain
        // ---- (1) load the chunk
        for (int e = tid; e < 64 * KD; e += kThreads) {
            const int i = e / KD, l = e % KD;
            const long long row = (row_base + t0 + i) * H + h;
            const bool in = t0 + i < seq_tokens;
            ks[i * KP + l] = in ? load_in(p.k, row * KD + l, p.in_bf16) : 0.f;
            if (!SUMMARY) qs[i * KP + l] = in ? load_in(p.q, row * KD + l, p.in_bf16) : 0.f;
        }
        for (int e = tid; e < 64 * CT; e += kThreads) {
            const int i = e / CT, c = e % CT;
            const long long row = (row_base + t0 + i) * H + h;
            const int gc = c0 + c;
            float x = 0.f;
            if (t0 + i < seq_tokens) {
                if (SUMMARY)
                    x = (gc < KD) ? 0.f : load_in(p.v, row * V + (gc - KD), p.in_bf16);
                else
                    x = load_in(p.v, row * V + gc, p.in_bf16);
            }
            vs[e] = x;
        }
        if (tid < 64) {
            const long long row = (row_base + t0 + tid) * H + h;
            const bool in = t0 + tid < seq_tokens;
            if (!GATEK) gx[tid] = in ? load_in(p.g, row, p.in_bf16) : 0.f;   // raw gate for now
            bet[tid] = in ? load_in(p.beta, row, p.in_bf16) : 0.f;
        }
        if (GATEK)
            for (int e = tid; e < 64 * KD; e += kThreads) {
                const int i = e / KD, l = e % KD;
                const long long row = (row_base + t0 + i) * H + h;
                Gk[i * KP + l] = (t0 + i < seq_tokens) ? load_in(p.g, row * KD + l, p.in_bf16) : 0.f;
            }
        __syncthreads();
        if (GATEK) {
            // ---- (2') per-channel inclusive cumsum down the chunk (one thread per channel)
            if (tid < KD) {
                float acc = 0.f;
                for (int i = 0; i < 64; ++i) {
                    acc += Gk[i * KP + tid];
                    Gk[i * KP + tid] = acc;
                }
            }
            __syncthreads();
            // read-side gate of token i, channel l: G_il, or the exclusive G_(i-1)l
            auto gread = [&](int i, int l) {
                return p.decay_first ? Gk[i * KP + l] : (i > 0 ? Gk[(i - 1) * KP + l] : 0.f);
            };
            // ---- (3') L = diag(beta) P and C with per-channel decays; clear A. Every
            //      exponent is a difference G_i - G_j with j <= i, so it is never positive.
            for (int e = tid; e < 64 * 64; e += kThreads) {
                const int i = e / 64, j = e % 64;
                float lv = 0.f, cv = 0.f;
                if (j < i) {
                    float d = 0.f;
#pragma unroll 4
                    for (int l = 0; l < KD; ++l)
                        d = fmaf(ks[i * KP + l] * ks[j * KP + l], __expf(gread(i, l) - Gk[j * KP + l]), d);
                    lv = bet[i] * d;
                }
                if (!SUMMARY && j <= i) {
                    float d = 0.f;
#pragma unroll 4
                    for (int l = 0; l < KD; ++l)
                        d = fmaf(qs[i * KP + l] * ks[j * KP + l], __expf(Gk[i * KP + l] - Gk[j * KP + l]), d);
                    cv = d;
                }
                Ls[i * LP + j] = lv;
                if (!SUMMARY) Cs[i * LP + j] = cv;
                As[i * LP + j] = 0.f;
            }
            // scaled keys of the read, k_il exp(Gread_il)
            for (int e = tid; e < 64 * KD; e += kThreads) {
                const int i = e / KD, l = e % KD;
                Ek[i * KP + l] = ks[i * KP + l] * __expf(gread(i, l));
            }
            __syncthreads();
        }
        // ---- (2) gate cumsum inside the chunk (one warp; two gates per lane)
        if (!GATEK && tid < 32) {
            const float a0 = gx[2 * tid], a1 = gx[2 * tid + 1];
            float s = a0 + a1;
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, s, off);
                if (tid >= off) s += o;
            }
            const float excl = s - (a0 + a1);
            gam[2 * tid] = excl + a0;
            gam[2 * tid + 1] = excl + a0 + a1;
            // read-side gate: Gx_i = G_i - g_i, or G_i when the read sees the decayed state
            gx[2 * tid] = p.decay_first ? excl + a0 : excl;
            gx[2 * tid + 1] = p.decay_first ? excl + a0 + a1 : excl + a0;
        }
        __syncthreads();
        const float glast = GATEK ? 0.f : gam[63];
        if (!GATEK && tid < 64) {
            dk[tid] = expf(glast - gam[tid]);
            eq[tid] = expf(gam[tid]);
            ekr[tid] = expf(gx[tid]);
        }
        // ---- (3) L = diag(beta) P and C; clear A
        for (int e = tid; e < (GATEK ? 0 : 64 * 64); e += kThreads) {
            const int i = e / 64, j = e % 64;
            float lv = 0.f, cv = 0.f;
            if (j < i) {
                float d = 0.f;
#pragma unroll 8
                for (int l = 0; l < KD; ++l) d = fmaf(ks[i * KP + l], ks[j * KP + l], d);
                lv = bet[i] * expf(gx[i] - gam[j]) * d;
            }
            if (!SUMMARY && j <= i) {
                float d = 0.f;
#pragma unroll 8
                for (int l = 0; l < KD; ++l) d = fmaf(qs[i * KP + l], ks[j * KP + l], d);
                cv = expf(gam[i] - gam[j]) * d;
            }
            Ls[i * LP + j] = lv;
            if (!SUMMARY) Cs[i * LP + j] = cv;
            As[i * LP + j] = 0.f;
        }
        __syncthreads();
        // ---- (4a) inverses of the four 16x16 diagonal blocks of I + L
        if (tid < 64) {
            const int base = (tid / 16) * 16, c = tid % 16;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int r = 1; r < 16; ++r) {
                float a = 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) a = fmaf(Ls[(base + r) * LP + base + m], x[m], a);
                if (r > c) x[r] = -a;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) As[(base + r) * LP + base + c] = x[r];
        }
        __syncthreads();
        // ---- (4b) block forward substitution: X_IJ = -inv(T_II) * sum_{m=J}^{I-1} L_Im X_mJ
        {
            float* Yb = Ys;   // scratch, 3 blocks of 16x16 (Ys is free until step 5)
            const int r = tid / 16, c = tid % 16;
            for (int I = 1; I < 4; ++I) {
                for (int J = 0; J < I; ++J) {
                    float a = 0.f;
                    for (int m = J; m < I; ++m) {
#pragma unroll
                        for (int l = 0; l < 16; ++l)
                            a = fmaf(Ls[(16 * I + r) * LP + 16 * m + l],
                                     As[(16 * m + l) * LP + 16 * J + c], a);
                    }
                    Yb[J * 256 + r * 16 + c] = a;
                }
                __syncthreads();
                for (int J = 0; J < I; ++J) {
                    float a = 0.f;
#pragma unroll
                    for (int l = 0; l < 16; ++l)
                        a = fmaf(As[(16 * I + r) * LP + 16 * I + l], Yb[J * 256 + l * 16 + c], a);
                    As[(16 * I + r) * LP + 16 * J + c] = -a;
                }
                __syncthreads();
            }
        }
        // ---- (5) Y = diag(beta) (V - diag(exp(Gx)) K H)
        for (int e = tid; e < 64 * CT; e += kThreads) {
            const int i = e / CT, c = e % CT;
            float a = 0.f;
#pragma unroll 8
            for (int l = 0; l < KD; ++l) a = fmaf(GATEK ? Ek[i * KP + l] : ks[i * KP + l], Hs[l * CT + c], a);
            Ys[e] = bet[i] * (vs[e] - (GATEK ? a : ekr[i] * a));
        }
        __syncthreads();
        // ---- (6) R = A Y
        for (int e = tid; e < 64 * CT; e += kThreads) {
            const int i = e / CT, c = e % CT;
            float a = 0.f;
            for (int j = 0; j <= i; ++j) a = fmaf(As[i * LP + j], Ys[j * CT + c], a);
            Rs[e] = a;
        }
        __syncthreads();
        // ---- (7) O = diag(exp(G)) Q H + C R (per channel: Q scaled by exp(G_il) in place)
        if (!SUMMARY && GATEK) {
            for (int e = tid; e < 64 * KD; e += kThreads) {
                const int i = e / KD, l = e % KD;
                qs[i * KP + l] *= __expf(Gk[i * KP + l]);
            }
            __syncthreads();
        }
        if (!SUMMARY) {
            for (int e = tid; e < 64 * CT; e += kThreads) {
                const int i = e / CT, c = e % CT;
                float a = 0.f;
#pragma unroll 8
                for (int l = 0; l < KD; ++l) a = fmaf(qs[i * KP + l], Hs[l * CT + c], a);
                float bsum = 0.f;
                for (int j = 0; j <= i; ++j) bsum = fmaf(Cs[i * LP + j], Rs[j * CT + c], bsum);
                const long long row = (row_base + t0 + i) * H + h;
                if (t0 + i < seq_tokens)
                    store_out(p.o, row * V + c0 + c, GATEK ? a + bsum : fmaf(eq[i], a, bsum), p.out_bf16);
            }
            __syncthreads();
        }
        // ---- (8) H <- exp(G_last) H + sum_j exp(G_last - G_j) k_j R_j (per channel: row l
        //      decays by exp(G_last,l), the keys by exp(G_last,l - G_jl))
        if (GATEK) {
            for (int e = tid; e < 64 * KD; e += kThreads) {
                const int j = e / KD, l = e % KD;
                Ek[j * KP + l] = ks[j * KP + l] * __expf(Gk[63 * KP + l] - Gk[j * KP + l]);
            }
            __syncthreads();
        }
        const float dlast = expf(glast);
        for (int e = tid; e < KD * CT; e += kThreads) {
            const int l = e / CT, c = e % CT;
            float a = 0.f;
#pragma unroll 8
            for (int j = 0; j < 64; ++j)
                a = fmaf(GATEK ? Ek[j * KP + l] : dk[j] * ks[j * KP + l], Rs[j * CT + c], a);
            Hs[e] = fmaf(GATEK ? __expf(Gk[63 * KP + l]) : dlast, Hs[e], a);
        }
        __syncthreads();
    }

    // ---- write the chain's final state
    if (SUMMARY) {
        const long long base = (long long)seg * p.B * H + bh;
        for (int e = tid; e < KD * CT; e += kThreads) {
            const int l = e / CT, c = e % CT;
            const int gc = c0 + c;
            if (gc < KD)
                p.M[(base * KD + l) * KD + gc] = Hs[e];
            else
                p.S[(base * KD + l) * V + (gc - KD)] = Hs[e];
        }
    } else {
        if (p.h_final && seg == p.nseg_total - 1)
            for (int e = tid; e < KD * CT; e += kThreads) {
                const int l = e / CT, c = e % CT;
                p.h_final[((long long)bh * KD + l) * V + c0 + c] = Hs[e];
            }
        if (p.h_out)   // the state entering the next segment
            for (int e = tid; e < KD * CT; e += kThreads) {
                const int l = e / CT, c = e % CT;
                p.h_out[(seg + 1) * p.h_out_seg_stride + ((long long)bh * KD + l) * V + c0 + c] = Hs[e];
            }
    }
    // a summary grid launched as a programmatic dependent completes after its primary grid
    if (SUMMARY) asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int KD, bool SUMMARY, bool GATEK>
cudaError_t launch_chain_g(const ChainParams& p, cudaStream_t s) {
    constexpr int CT = 32;
    using L = SimtSmem<KD, CT, SUMMARY, GATEK>;
    auto kern = simt_chain_kernel<KD, CT, SUMMARY, GATEK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::bytes);
    if (e != cudaSuccess) return e;
    const int ncols = SUMMARY ? KD + p.V : p.V;
    dim3 grid((unsigned)(p.B * p.H * p.nseg_run), (unsigned)(ncols / CT));
    if (!p.launch_dependent) {
        kern<<<grid, kThreads, L::bytes, s>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int KD, bool SUMMARY>
cudaError_t launch_chain(const ChainParams& p, cudaStream_t s) {
    // per-channel gates at bf16 inputs: the sub-block normalised chains with their products on
    // the tensor cores (gdn_kda_mma.cu)
    if (p.gate_k && p.in_bf16) return launch_kda_mma_chain(p, SUMMARY, s);
    return p.gate_k ? launch_chain_g<KD, SUMMARY, true>(p, s) : launch_chain_g<KD, SUMMARY, false>(p, s);
}

// In-order scan over consecutive pieces of each sequence, fp32, one CTA per (head, 32-column
// tile); the serial dependency runs over pieces inside the CTA: the state entering piece
// p_first is given (h_first, or zero), and the state entering piece p+1 is M[p] H + S[p]
// (the affine summary of piece p applied to the state entering it). Each step stages M[p] in
// shared memory (rows padded to KD + 4 floats) and every thread accumulates a 4 x 4 block of
// the product in registers, four terms of the sum at a time. The states entering pieces
// p_first+1 .. P-1 go to Hp, those entering every nsub-th piece (segment starts) to H_seg.
template <int KD>
__global__ void __launch_bounds__(KD * 2)
scan_kernel(const float* __restrict__ M, const float* __restrict__ S,
            const float* __restrict__ h_first, float* __restrict__ Hp, float* __restrict__ H_seg,
            const float* __restrict__ h_seg0, int p_first, int P, int nsub, int BH, int V) {
    constexpr int CT = 32, NT = KD * 2, MP = KD + 4;
    extern __shared__ float4 sm4[];
    float* Ms = reinterpret_cast<float*>(sm4);   // KD x MP
    float* Hc = Ms + KD * MP;                    // KD x CT, the current state's column tile
    const int bh = blockIdx.x, c0 = blockIdx.y * CT, tid = threadIdx.x;
    const int ri = tid >> 3, ci = tid & 7;       // rows 4ri..4ri+3, columns 4ci..4ci+3
    // state tile <-> global [.][BH][KD][V]
    auto put = [&](float* dst, long long slot) {
        const long long hb = (slot * BH + bh) * KD;
        for (int e = tid; e < KD * CT / 4; e += NT) {
            const int l = e / (CT / 4), c4 = e % (CT / 4);
            *reinterpret_cast<float4*>(dst + (hb + l) * V + c0 + 4 * c4) =
                *reinterpret_cast<const float4*>(Hc + l * CT + 4 * c4);
        }
    };
    if (H_seg && p_first > 0)   // the state entering the first segment
        for (int e = tid; e < KD * CT / 4; e += NT) {
            const int l = e / (CT / 4), c4 = e % (CT / 4);
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (h_seg0) x = *reinterpret_cast<const float4*>(h_seg0 + ((long long)bh * KD + l) * V + c0 + 4 * c4);
            *reinterpret_cast<float4*>(H_seg + ((long long)bh * KD + l) * V + c0 + 4 * c4) = x;
        }
    for (int e = tid; e < KD * CT / 4; e += NT) {
        const int l = e / (CT / 4), c4 = e % (CT / 4);
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (h_first) x = *reinterpret_cast<const float4*>(h_first + ((long long)bh * KD + l) * V + c0 + 4 * c4);
        *reinterpret_cast<float4*>(Hc + l * CT + 4 * c4) = x;
    }
    __syncthreads();
    for (int p = p_first; p < P; ++p) {
        // Hc holds the state entering piece p
        if (Hp && p > p_first) put(Hp, p);
        if (H_seg && p % nsub == 0) put(H_seg, p / nsub);
        if (p == P - 1 || !M) continue;   // no summaries: every piece starts from the same state
        const float* Mg = M + ((long long)p * BH + bh) * KD * KD;
        const float* Sg = S + ((long long)p * BH + bh) * KD * V;
        // all of this thread's loads of M in flight at once (the trip count is a constant)
#pragma unroll
        for (int e = tid; e < KD * KD / 4; e += NT) {
            const int i = e / (KD / 4), l4 = e % (KD / 4);
            *reinterpret_cast<float4*>(Ms + i * MP + 4 * l4) =
                __ldg(reinterpret_cast<const float4*>(Mg + (long long)i * KD + 4 * l4));
        }
        float acc[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float4 x = __ldg(reinterpret_cast<const float4*>(
                Sg + (long long)(4 * ri + r) * V + c0 + 4 * ci));
            acc[r][0] = x.x;
            acc[r][1] = x.y;
            acc[r][2] = x.z;
            acc[r][3] = x.w;
        }
        __syncthreads();
#pragma unroll 2
        for (int l = 0; l < KD; l += 4) {
            float4 m[4], hv[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) m[r] = *reinterpret_cast<const float4*>(Ms + (4 * ri + r) * MP + l);
#pragma unroll
            for (int q = 0; q < 4; ++q) hv[q] = *reinterpret_cast<const float4*>(Hc + (l + q) * CT + 4 * ci);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float mr[4] = {m[r].x, m[r].y, m[r].z, m[r].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[r][0] = fmaf(mr[q], hv[q].x, acc[r][0]);
                    acc[r][1] = fmaf(mr[q], hv[q].y, acc[r][1]);
                    acc[r][2] = fmaf(mr[q], hv[q].z, acc[r][2]);
                    acc[r][3] = fmaf(mr[q], hv[q].w, acc[r][3]);
                }
            }
        }
        __syncthreads();   // every read of Hc and Ms is done
#pragma unroll
        for (int r = 0; r < 4; ++r)
            *reinterpret_cast<float4*>(Hc + (4 * ri + r) * CT + 4 * ci) =
                make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
        __syncthreads();
    }
}

template <int KD>
cudaError_t launch_scan_k(const float* M, const float* S, const float* h_first, float* Hp,
                          float* H_seg, const float* h_seg0, int p_first, int P, int nsub, int BH,
                          int V, cudaStream_t s) {
    const size_t smem = sizeof(float) * ((size_t)KD * (KD + 4) + (size_t)KD * 32);
    cudaError_t e = cudaFuncSetAttribute(scan_kernel<KD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)BH, (unsigned)(V / 32));
    scan_kernel<KD><<<grid, KD * 2, smem, s>>>(M, S, h_first, Hp, H_seg, h_seg0, p_first, P, nsub,
                                                BH, V);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_forward(const ChainParams& p, cudaStream_t s) {
    return p.K == 128 ? launch_chain<128, false>(p, s) : launch_chain<64, false>(p, s);
}

cudaError_t launch_simt_summary(const ChainParams& p, cudaStream_t s) {
    return p.K == 128 ? launch_chain<128, true>(p, s) : launch_chain<64, true>(p, s);
}

cudaError_t launch_scan(const float* M, const float* S, const float* h_first, float* Hp,
                        float* H_seg, const float* h_seg0, int p_first, int P, int nsub, int BH,
                        int K, int V, cudaStream_t s, DeviceError* err) {
    if (nsub < 1 || p_first < 0 || P <= p_first) return cudaErrorInvalidValue;
    if (err && tc_scan_supported(M, S, p_first, P, K, V))
        return launch_tc_scan(M, S, h_first, Hp, H_seg, h_seg0, p_first, P, nsub, BH, err, s);
    if (K == 128) return launch_scan_k<128>(M, S, h_first, Hp, H_seg, h_seg0, p_first, P, nsub, BH, V, s);
    if (K == 64) return launch_scan_k<64>(M, S, h_first, Hp, H_seg, h_seg0, p_first, P, nsub, BH, V, s);
    return cudaErrorInvalidValue;
}

}  // namespace gdn
