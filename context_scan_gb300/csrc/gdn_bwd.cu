// gdn_bwd.cu -- the state-gradient path of the backward pass: per-segment state-gradient
// summaries and their reverse scan ("RFC: HyperParallel Linear Attention Context Parallel",
// section 6.4.3: the summary step yields dS_local, then dH_in = M^T dH_out + dS_local).
//
// The gradient on the state runs backwards through the transposed token transitions. A
// chunk of 64 tokens maps its entering state H to R = U - W H, O = Qd H + C R and
// H' = exp(G_last) H + Kd^T R (the chunk equations of "Context Parallelism in ART",
// section 08, "First parallelize within a GPU", with the read of the RFC's section 2.1),
// so with D' = dL/dH' and dO the chunk's output gradient,
//   dR = Kd D' + C^T dO                      (64 x V)
//   D  = exp(G_last) D' + Qd^T dO - W^T dR   (K x V, the gradient on the entering state)
// with W^T dR = K^T diag(beta exp(Gx)) (A^T dR), A = (I + diag(beta) P)^{-1}. The state
// gradient's columns are independent, like the state's: each CTA owns one chain (b, h,
// segment) and a tile of CT columns, walks the segment's chunks from the last to the first
// and writes D at the segment's start. fp32 on the CUDA cores; exponents are differences of
// cumulative gates, never exp(-G).
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float ld(const void* base, long long idx, int bf16) {
    if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
    return reinterpret_cast<const float*>(base)[idx];
}

template <int KD, int CT>
struct BwdSmem {
    static constexpr int KP = KD + 1;   // padded rows of k / q
    static constexpr int LP = 65;       // padded rows of the 64 x 64 matrices
    static constexpr int off_k = 0;
    static constexpr int off_q = off_k + 64 * KP;
    static constexpr int off_do = off_q + 64 * KP;
    static constexpr int off_d = off_do + 64 * CT;
    static constexpr int off_l = off_d + KD * CT;
    static constexpr int off_a = off_l + 64 * LP;
    static constexpr int off_c = off_a + 64 * LP;
    static constexpr int off_z = off_c + 64 * LP;
    static constexpr int off_r = off_z + 64 * CT;
    static constexpr int off_s = off_r + 64 * CT;   // scalars: 6 x 64
    static constexpr int total = off_s + 6 * 64;
    static constexpr size_t bytes = sizeof(float) * total;
};

template <int KD, int CT>
__global__ void __launch_bounds__(kThreads) state_grad_kernel(StateGradParams p) {
    using L = BwdSmem<KD, CT>;
    extern __shared__ float sm[];
    float* ks = sm + L::off_k;
    float* qs = sm + L::off_q;
    float* dos = sm + L::off_do;
    float* Ds = sm + L::off_d;
    float* Ls = sm + L::off_l;
    float* As = sm + L::off_a;
    float* Cs = sm + L::off_c;
    float* Zs = sm + L::off_z;
    float* Rs = sm + L::off_r;
    float* gam = sm + L::off_s;   // inclusive cumulative gate G_i
    float* gx = gam + 64;         // read-side gate (exclusive Gx_i, or G_i for the decayed read)
    float* bet = gx + 64;
    float* dk = bet + 64;         // exp(G_last - G_j)
    float* eq = dk + 64;          // exp(G_i)
    float* ekr = eq + 64;         // beta_i exp(Gx_i)
    constexpr int KP = L::KP, LP = L::LP;

    const int tid = threadIdx.x;
    const int seg = blockIdx.x % p.nseg;
    const int bh = blockIdx.x / p.nseg;
    const int b = bh / p.H, h = bh % p.H;
    const int c0 = blockIdx.y * CT;
    const int V = p.V, H = p.H;
    const long long head = (long long)seg * p.B * H + bh;   // [seg][b][h] index

    for (int e = tid; e < KD * CT; e += kThreads) {
        const int l = e / CT, c = e % CT;
        Ds[e] = p.dH_end ? p.dH_end[(head * KD + l) * V + c0 + c] : 0.f;
    }

    const long long row0 = (long long)b * p.T + (long long)seg * p.seg_len;
    for (int ch = p.seg_len / kChunk - 1; ch >= 0; --ch) {
        const long long r0 = row0 + (long long)ch * kChunk;
        // ---- (1) load k, q, the dO tile, g, beta
        for (int e = tid; e < 64 * KD; e += kThreads) {
            const int i = e / KD, l = e % KD;
            const long long row = (r0 + i) * H + h;
            ks[i * KP + l] = ld(p.k, row * KD + l, p.in_bf16);
            qs[i * KP + l] = ld(p.q, row * KD + l, p.in_bf16);
        }
        for (int e = tid; e < 64 * CT; e += kThreads) {
            const int i = e / CT, c = e % CT;
            dos[e] = ld(p.dO, ((r0 + i) * H + h) * V + c0 + c, p.do_bf16);
        }
        if (tid < 64) {
            const long long row = (r0 + tid) * H + h;
            gx[tid] = ld(p.g, row, p.in_bf16);   // raw gate until the cumsum
            bet[tid] = ld(p.beta, row, p.in_bf16);
        }
        __syncthreads();
        // ---- (2) inclusive / read-side cumulative gates (one warp, two tokens per lane)
        if (tid < 32) {
            const float a0 = gx[2 * tid], a1 = gx[2 * tid + 1];
            float s = a0 + a1;
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, s, off);
                if (tid >= off) s += o;
            }
            const float excl = s - (a0 + a1);
            gam[2 * tid] = excl + a0;
            gam[2 * tid + 1] = excl + a0 + a1;
            gx[2 * tid] = p.decay_first ? excl + a0 : excl;
            gx[2 * tid + 1] = p.decay_first ? excl + a0 + a1 : excl + a0;
        }
        __syncthreads();
        const float glast = gam[63];
        if (tid < 64) {
            dk[tid] = expf(glast - gam[tid]);
            eq[tid] = expf(gam[tid]);
            ekr[tid] = bet[tid] * expf(gx[tid]);
        }
        // ---- (3) L = diag(beta) P (j < i) and C (j <= i); clear A
        for (int e = tid; e < 64 * 64; e += kThreads) {
            const int i = e / 64, j = e % 64;
            float lv = 0.f, cv = 0.f;
            if (j <= i) {
                float dkk = 0.f, dqk = 0.f;
#pragma unroll 8
                for (int l = 0; l < KD; ++l) {
                    const float kj = ks[j * KP + l];
                    dkk = fmaf(ks[i * KP + l], kj, dkk);
                    dqk = fmaf(qs[i * KP + l], kj, dqk);
                }
                if (j < i) lv = bet[i] * expf(gx[i] - gam[j]) * dkk;
                cv = expf(gam[i] - gam[j]) * dqk;
            }
            Ls[i * LP + j] = lv;
            Cs[i * LP + j] = cv;
            As[i * LP + j] = 0.f;
        }
        __syncthreads();
        // ---- (4a) inverses of the four 16 x 16 diagonal blocks of I + L (forward substitution)
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
        // ---- (4b) off-diagonal blocks: A_IJ = -inv(T_II) sum_{m=J}^{I-1} L_Im A_mJ
        {
            float* Yb = Zs;   // 3 blocks of 16 x 16 scratch (Zs is free until step 6)
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
        // ---- (5) dR = Kd D' + C^T dO
        for (int e = tid; e < 64 * CT; e += kThreads) {
            const int j = e / CT, c = e % CT;
            float a = 0.f;
#pragma unroll 8
            for (int l = 0; l < KD; ++l) a = fmaf(ks[j * KP + l], Ds[l * CT + c], a);
            float t = 0.f;
            for (int i = j; i < 64; ++i) t = fmaf(Cs[i * LP + j], dos[i * CT + c], t);
            Rs[e] = fmaf(dk[j], a, t);
        }
        __syncthreads();
        // ---- (6) Z = diag(beta exp(Gx)) A^T dR
        for (int e = tid; e < 64 * CT; e += kThreads) {
            const int j = e / CT, c = e % CT;
            float a = 0.f;
            for (int i = j; i < 64; ++i) a = fmaf(As[i * LP + j], Rs[i * CT + c], a);
            Zs[e] = ekr[j] * a;
        }
        __syncthreads();
        // ---- (7) D = exp(G_last) D' + Qd^T dO - K^T Z
        const float dlast = expf(glast);
        for (int e = tid; e < KD * CT; e += kThreads) {
            const int l = e / CT, c = e % CT;
            float a = 0.f;
#pragma unroll 8
            for (int i = 0; i < 64; ++i)
                a = fmaf(eq[i] * qs[i * KP + l], dos[i * CT + c], fmaf(-ks[i * KP + l], Zs[i * CT + c], a));
            Ds[e] = fmaf(dlast, Ds[e], a);
        }
        __syncthreads();
    }

    for (int e = tid; e < KD * CT; e += kThreads) {
        const int l = e / CT, c = e % CT;
        p.dS[(head * KD + l) * V + c0 + c] = Ds[e];
    }
}

// Reverse scan over segments: dH_in[s] = M[s]^T dH_in[s+1] + dS[s], dH_in[nseg] = dht (or
// zero). One CTA per (head, 32-column tile); M[s] is staged in shared memory and every
// thread accumulates a 4 x 4 block of the product.
template <int KD>
__global__ void __launch_bounds__(KD * 2)
state_grad_scan_kernel(const float* __restrict__ M, const float* __restrict__ dS,
                       const float* __restrict__ dht, float* __restrict__ dH_in, int nseg, int BH,
                       int V) {
    constexpr int CT = 32, NT = KD * 2, MP = KD + 4;
    extern __shared__ float4 sm4[];
    float* Ms = reinterpret_cast<float*>(sm4);   // KD x MP
    float* Gs = Ms + KD * MP;                    // KD x CT, the gradient entering from above
    const int tid = threadIdx.x;
    const int bh = blockIdx.x, c0 = blockIdx.y * CT;
    // thread -> rows i0..i0+3, columns j0..j0+3 of the KD x CT output tile
    const int i0 = (tid / (CT / 4)) * 4, j0 = (tid % (CT / 4)) * 4;
    static_assert((KD / 4) * (CT / 4) == NT, "one 4 x 4 block per thread");
    for (int e = tid; e < KD * CT; e += NT) {
        const int l = e / CT, c = e % CT;
        Gs[e] = dht ? dht[((long long)bh * KD + l) * V + c0 + c] : 0.f;
    }
    for (int s = nseg - 1; s >= 0; --s) {
        const long long hs = (long long)s * BH + bh;
        const float* Mp = M + hs * KD * KD;
        for (int e = tid; e < KD * KD / 4; e += NT) {
            const int r = (4 * e) / KD, c = (4 * e) % KD;
            *reinterpret_cast<float4*>(&Ms[r * MP + c]) = reinterpret_cast<const float4*>(Mp)[e];
        }
        __syncthreads();
        float acc[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                acc[a][c] = dS[(hs * KD + i0 + a) * V + c0 + j0 + c];
        for (int m = 0; m < KD; ++m) {
            const float4 mr = *reinterpret_cast<const float4*>(&Ms[m * MP + i0]);   // M[m][i0..]
            const float4 gr = *reinterpret_cast<const float4*>(&Gs[m * CT + j0]);
            const float mv[4] = {mr.x, mr.y, mr.z, mr.w}, gv[4] = {gr.x, gr.y, gr.z, gr.w};
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(mv[a], gv[c], acc[a][c]);
        }
        __syncthreads();   // every thread has read Gs and Ms
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const float4 out = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
            *reinterpret_cast<float4*>(&Gs[(i0 + a) * CT + j0]) = out;
            *reinterpret_cast<float4*>(&dH_in[(hs * KD + i0 + a) * V + c0 + j0]) = out;
        }
        __syncthreads();
    }
}

template <int KD>
cudaError_t launch_state_grad_k(const StateGradParams& p, cudaStream_t s) {
    constexpr int CT = 32;
    using L = BwdSmem<KD, CT>;
    auto kern = state_grad_kernel<KD, CT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::bytes);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.B * p.H * p.nseg), (unsigned)(p.V / CT));
    kern<<<grid, kThreads, L::bytes, s>>>(p);
    return cudaGetLastError();
}

template <int KD>
cudaError_t launch_state_grad_scan_k(const float* M, const float* dS, const float* dht,
                                     float* dH_in, int nseg, int BH, int V, cudaStream_t s) {
    constexpr int CT = 32;
    const size_t bytes = sizeof(float) * (KD * (KD + 4) + KD * CT);
    auto kern = state_grad_scan_kernel<KD>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)BH, (unsigned)(V / CT)), KD * 2, bytes, s>>>(M, dS, dht, dH_in, nseg,
                                                                      BH, V);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_state_grad(const StateGradParams& p, cudaStream_t s) {
    return p.K == 64 ? launch_state_grad_k<64>(p, s) : launch_state_grad_k<128>(p, s);
}

cudaError_t launch_state_grad_scan(const float* M, const float* dS, const float* dht,
                                   float* dH_in, int nseg, int BH, int K, int V, cudaStream_t s) {
    return K == 64 ? launch_state_grad_scan_k<64>(M, dS, dht, dH_in, nseg, BH, V, s)
                   : launch_state_grad_scan_k<128>(M, dS, dht, dH_in, nseg, BH, V, s);
}

}  // namespace gdn
