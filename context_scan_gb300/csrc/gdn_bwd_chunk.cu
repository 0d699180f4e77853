// gdn_bwd_chunk.cu -- the per-chunk gradients of the backward pass: dq, dk, dv, dg, dbeta
// ("RFC: HyperParallel Linear Attention Context Parallel", section 6.4.3: after the state
// gradients are known at every chunk boundary, "backward_state + backward_finish" give
// dQ, dK, dV, dg, dbeta; "KDA Chunk Backward -- TPU/Pallas Kernel Design", section 2).
//
// With the state H entering a chunk and the gradient D' on the state leaving it, a chunk's
// gradients depend on nothing else, so every (b, h, chunk) is one independent CTA. The
// equations are the vector-Jacobian products of the chunk forward ("Context Parallelism in
// ART", section 08, "First parallelize within a GPU", with the read of the RFC's section
// 2.1), each line of the forward taken backwards:
//   forward:  P[i,j] = e^(Gx_i - G_j) k_i.k_j (j < i), A = (I + diag(beta) P)^-1,
//             Kr = e^Gx k, U = A diag(beta) V, W = A diag(beta) Kr, R = U - W H,
//             C[i,j] = e^(G_i - G_j) q_i.k_j (j <= i), Qd = e^G q, Kd = e^(Gn - G) k
//   backward: dR = Kd D' + C^T dO,  dC = tril(dO R^T),  dQd = dO H^T,  dKd = R D'^T,
//             dW = -dR H^T,  X = A^T dR,  Y = A^T dW,  dv = beta X,  dKr = beta Y,
//             dA = dR (beta V)^T + dW (beta Kr)^T,  dL = -tril(A^T dA A^T, -1),
//             dbeta = rowsum(X . V) + rowsum(Y . Kr) + rowsum(dL . P),
//             S = beta dL . e^(Gx_i - G_j):  dk = S k + S^T k,
//             S' = dC . e^(G_i - G_j):  dq = S' k,  dk += S'^T q,
//             dq += e^G dQd,  dk += e^(Gn - G) dKd + e^Gx dKr,
//   and the gate terms of P, C, Qd, Kd, Kr and e^Gn summed per token into dG (through G) and
//   dGx (through the read-side gate), then dg = reverse cumulative sum of dG + dGx, minus dGx
//   when the read sees the un-decayed state (Gx = G - g).
// fp32 on the CUDA cores. V is walked in tiles of 16 columns: the products that contract over
// V (dC, dA, dQd, dKd, dW) accumulate across the tiles -- the last three in registers -- and
// the products that produce V-wide results (R, dR, X, dv) are finished tile by tile.
// Exponents are differences of cumulative gates (or G, Gx themselves, which are <= 0).
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kCgThreads = 256;
constexpr int kCT = 16;   // V columns per tile

__device__ __forceinline__ float ldv(const void* base, long long idx, int bf16) {
    if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
    return reinterpret_cast<const float*>(base)[idx];
}
__device__ __forceinline__ float4 l4(const float* p) { return *reinterpret_cast<const float4*>(p); }
// Sum over the 16 lanes of a half-warp, in a fixed order (every lane gets the sum). All sums of
// the kernel are taken in a fixed order, so its results do not vary from run to run.
__device__ __forceinline__ float half_sum(float x) {
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

template <int KD>
struct CgSmem {
    static constexpr int P64 = 68;          // row pitch of the 64 x 64 matrices
    static constexpr int KP = KD + 4;       // row pitch of the 64 x KD matrices and of H^T tiles
    static constexpr int CTP = kCT + 4;     // row pitch of the 64 x 16 tiles
    static constexpr int k = 0;                          // k       [64][KP]
    static constexpr int a = k + 64 * KP;                // A       [64][P64]
    static constexpr int c = a + 64 * P64;               // C, then S'
    static constexpr int p = c + 64 * P64;               // P
    static constexpr int dc = p + 64 * P64;              // dC
    static constexpr int da = dc + 64 * P64;             // dA, then dL, then S
    static constexpr int w = da + 64 * P64;              // W, then dW  [64][KP]
    static constexpr int t = w + 64 * KP;                // tile region (see below)
    // tile region: v, dO, R, dR [64][CTP] and H^T, D'^T [kCT][KP]; before the tile loop q
    // [64][KP] (then the inverse's scratch), after it A^T dA [64][P64], then q again
    static constexpr int t_v = t, t_do = t_v + 64 * CTP, t_r = t_do + 64 * CTP,
                         t_dr = t_r + 64 * CTP, t_h = t_dr + 64 * CTP, t_d = t_h + kCT * KP;
    static constexpr int tile_end = t_d + kCT * KP;
    static constexpr int s = (tile_end > t + 64 * KP ? tile_end : t + 64 * KP);
    // per-token scalars
    enum { G = 0, GX, EG, EGX, DKF, BET, EKR, DG, DGX, DBETA, RED, NS };
    static constexpr int total = s + NS * 64;
    static constexpr size_t bytes = sizeof(float) * total;
    static_assert(64 * P64 <= tile_end - t || 64 * P64 <= 64 * KP, "A^T dA fits the tile region");
};

template <int KD>
__global__ void __launch_bounds__(kCgThreads) chunk_grad_kernel(ChunkGradParams p) {
    using L = CgSmem<KD>;
    constexpr int KP = L::KP, P64 = L::P64, CTP = L::CTP;
    constexpr int CW = KD / 16;   // columns of a thread's 4 x CW block of a 64 x KD matrix
    extern __shared__ float4 smv[];
    float* sm = reinterpret_cast<float*>(smv);
    float* ks = sm + L::k;
    float* As = sm + L::a;
    float* Cs = sm + L::c;
    float* Ps = sm + L::p;
    float* dCs = sm + L::dc;
    float* dAs = sm + L::da;
    float* Ws = sm + L::w;
    float* sc = sm + L::s;
    float* G = sc + 64 * L::G;
    float* Gx = sc + 64 * L::GX;
    float* eG = sc + 64 * L::EG;
    float* eGx = sc + 64 * L::EGX;
    float* dkf = sc + 64 * L::DKF;
    float* bet = sc + 64 * L::BET;
    float* ekr = sc + 64 * L::EKR;
    float* dG = sc + 64 * L::DG;
    float* dGx = sc + 64 * L::DGX;
    float* dbs = sc + 64 * L::DBETA;
    float* red = sc + 64 * L::RED;

    const int tid = threadIdx.x, lane = tid & 31;
    const int nch = p.T / kChunk;
    const int c = blockIdx.x % nch;
    const int bh = blockIdx.x / nch;
    const int b = bh / p.H, h = bh % p.H;
    const int H = p.H, V = p.V;
    const long long row0 = (long long)b * p.T + (long long)c * kChunk;   // flattened (b, t)
    const long long st0 = ((long long)c * p.B * H + bh) * KD * V;        // Hc / Dc offset

    // ---- (1) k, and q into the tile region; the gates and beta
    float* qs = sm + L::t;
    for (int e = tid; e < 64 * KD; e += kCgThreads) {
        const int i = e / KD, l = e % KD;
        const long long idx = ((row0 + i) * H + h) * KD + l;
        ks[i * KP + l] = ldv(p.k, idx, p.in_bf16);
        qs[i * KP + l] = ldv(p.q, idx, p.in_bf16);
    }
    if (tid < 64) {
        const long long row = (row0 + tid) * H + h;
        Gx[tid] = ldv(p.g, row, p.in_bf16);   // raw gate until the cumsum
        bet[tid] = ldv(p.beta, row, p.in_bf16);
        dG[tid] = 0.f;
        dGx[tid] = 0.f;
        dbs[tid] = 0.f;
        red[tid] = 0.f;
    }
    __syncthreads();
    if (tid < 32) {   // inclusive and read-side cumulative gates, two tokens per lane
        const float a0 = Gx[2 * lane], a1 = Gx[2 * lane + 1];
        float s = a0 + a1;
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += o;
        }
        const float excl = s - (a0 + a1);
        G[2 * lane] = excl + a0;
        G[2 * lane + 1] = excl + a0 + a1;
        Gx[2 * lane] = p.decay_first ? excl + a0 : excl;
        Gx[2 * lane + 1] = p.decay_first ? excl + a0 + a1 : excl + a0;
    }
    __syncthreads();
    const float Gn = G[63];
    if (tid < 64) {
        eG[tid] = expf(G[tid]);
        eGx[tid] = expf(Gx[tid]);
        dkf[tid] = expf(Gn - G[tid]);
        ekr[tid] = bet[tid] * expf(Gx[tid]);
    }
    // ---- (2) P = e^(Gx_i - G_j) k_i.k_j (j < i), C = e^(G_i - G_j) q_i.k_j (j <= i); A = 0
    {
        const int i0 = (tid >> 4) * 4, j0 = (tid & 15) * 4;
        float kk[4][4] = {}, qk[4][4] = {};
        if (j0 <= i0 + 3) {
#pragma unroll 2
            for (int l = 0; l < KD; l += 4) {
                float4 ki[4], qi[4], kj[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    ki[r] = l4(&ks[(i0 + r) * KP + l]);
                    qi[r] = l4(&qs[(i0 + r) * KP + l]);
                    kj[r] = l4(&ks[(j0 + r) * KP + l]);
                }
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int s2 = 0; s2 < 4; ++s2) {
                        kk[r][s2] += ki[r].x * kj[s2].x + ki[r].y * kj[s2].y + ki[r].z * kj[s2].z + ki[r].w * kj[s2].w;
                        qk[r][s2] += qi[r].x * kj[s2].x + qi[r].y * kj[s2].y + qi[r].z * kj[s2].z + qi[r].w * kj[s2].w;
                    }
            }
        }
        __syncthreads();   // the gates' exponentials are in place
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = i0 + r;
            float pv[4], cv[4];
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2) {
                const int j = j0 + s2;
                pv[s2] = (j < i) ? expf(Gx[i] - G[j]) * kk[r][s2] : 0.f;
                cv[s2] = (j <= i) ? expf(G[i] - G[j]) * qk[r][s2] : 0.f;
            }
            *reinterpret_cast<float4*>(&Ps[i * P64 + j0]) = make_float4(pv[0], pv[1], pv[2], pv[3]);
            *reinterpret_cast<float4*>(&Cs[i * P64 + j0]) = make_float4(cv[0], cv[1], cv[2], cv[3]);
            *reinterpret_cast<float4*>(&As[i * P64 + j0]) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(&dCs[i * P64 + j0]) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(&dAs[i * P64 + j0]) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    __syncthreads();
    // ---- (3) A = (I + L)^-1, L = diag(beta) P: the four 16 x 16 diagonal blocks by forward
    //      substitution (a column per thread), then the blocks below them by block rounds
    if (tid < 64) {
        const int base = (tid / 16) * 16, cc = tid % 16;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == cc) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
            float a = 0.f;
#pragma unroll
            for (int m = 0; m < r; ++m) a = fmaf(bet[base + r] * Ps[(base + r) * P64 + base + m], x[m], a);
            if (r > cc) x[r] = -a;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) As[(base + r) * P64 + base + cc] = x[r];
    }
    __syncthreads();
    {
        float* Yb = qs;   // 3 blocks of 16 x 16 scratch (q is reloaded at the end)
        const int r = tid / 16, cc = tid % 16;
        for (int I = 1; I < 4; ++I) {
            for (int J = 0; J < I; ++J) {
                float a = 0.f;
                for (int m = J; m < I; ++m) {
#pragma unroll
                    for (int l = 0; l < 16; ++l)
                        a = fmaf(bet[16 * I + r] * Ps[(16 * I + r) * P64 + 16 * m + l],
                                 As[(16 * m + l) * P64 + 16 * J + cc], a);
                }
                Yb[J * 256 + r * 16 + cc] = a;
            }
            __syncthreads();
            for (int J = 0; J < I; ++J) {
                float a = 0.f;
#pragma unroll
                for (int l = 0; l < 16; ++l)
                    a = fmaf(As[(16 * I + r) * P64 + 16 * I + l], Yb[J * 256 + l * 16 + cc], a);
                As[(16 * I + r) * P64 + 16 * J + cc] = -a;
            }
            __syncthreads();
        }
    }
    // ---- (4) W = A diag(beta e^Gx) K, a 4 x CW block per thread
    const int i0 = (tid >> 4) * 4, l0 = (tid & 15) * CW;
    {
        float acc[4][CW] = {};
        for (int j = 0; j < i0 + 4; ++j) {   // A[i][j] = 0 for j > i
            const float e = ekr[j];
            float kv[CW];
#pragma unroll
            for (int w = 0; w < CW; w += 4) {
                const float4 t4 = l4(&ks[j * KP + l0 + w]);
                kv[w] = e * t4.x, kv[w + 1] = e * t4.y, kv[w + 2] = e * t4.z, kv[w + 3] = e * t4.w;
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float a = As[(i0 + r) * P64 + j];
#pragma unroll
                for (int w = 0; w < CW; ++w) acc[r][w] = fmaf(a, kv[w], acc[r][w]);
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int w = 0; w < CW; w += 4)
                *reinterpret_cast<float4*>(&Ws[(i0 + r) * KP + l0 + w]) =
                    make_float4(acc[r][w], acc[r][w + 1], acc[r][w + 2], acc[r][w + 3]);
    }
    __syncthreads();

    // ---- (5) the V tiles
    float* vt = sm + L::t_v;
    float* dot = sm + L::t_do;
    float* Rt = sm + L::t_r;
    float* dRt = sm + L::t_dr;
    float* Ht = sm + L::t_h;   // H^T tile [kCT][KP]
    float* Dt = sm + L::t_d;   // D'^T tile [kCT][KP]
    float dQd[4][CW] = {}, dKd[4][CW] = {}, dW[4][CW] = {};
    float deg = 0.f;   // this thread's share of <D', H>
    float xv = 0.f;    // this thread's share of rowsum(X . V) for row rr
    const int rr = tid >> 2, cc4 = (tid & 3) * 4;   // a 1 x 4 block of a 64 x 16 tile
    for (int c0 = 0; c0 < V; c0 += kCT) {
        for (int e = tid; e < 64 * kCT; e += kCgThreads) {
            const int i = e / kCT, cc = e % kCT;
            const long long idx = ((row0 + i) * H + h) * V + c0 + cc;
            vt[i * CTP + cc] = ldv(p.v, idx, p.in_bf16);
            dot[i * CTP + cc] = ldv(p.dO, idx, p.do_bf16);
        }
        for (int e = tid; e < KD * kCT; e += kCgThreads) {
            const int l = e / kCT, cc = e % kCT;
            const long long idx = st0 + (long long)l * V + c0 + cc;
            const float hv = p.Hc[idx], dv = p.Dc[idx];
            Ht[cc * KP + l] = hv;
            Dt[cc * KP + l] = dv;
            deg = fmaf(hv, dv, deg);
        }
        __syncthreads();
        // R = A diag(beta) V - W H and dR = Kd D' + C^T dO (row rr, columns cc4..cc4+3)
        {
            float r4[4] = {}, d4[4] = {};
            for (int j = 0; j <= rr; ++j) {
                const float a = As[rr * P64 + j] * bet[j];
                const float4 v4 = l4(&vt[j * CTP + cc4]);
                r4[0] = fmaf(a, v4.x, r4[0]), r4[1] = fmaf(a, v4.y, r4[1]);
                r4[2] = fmaf(a, v4.z, r4[2]), r4[3] = fmaf(a, v4.w, r4[3]);
            }
            for (int l = 0; l < KD; l += 4) {
                const float4 wv = l4(&Ws[rr * KP + l]), kv = l4(&ks[rr * KP + l]);
                const float wa[4] = {wv.x, wv.y, wv.z, wv.w}, ka[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int s2 = 0; s2 < 4; ++s2) {
                        r4[s2] = fmaf(-wa[u], Ht[(cc4 + s2) * KP + l + u], r4[s2]);
                        d4[s2] = fmaf(ka[u], Dt[(cc4 + s2) * KP + l + u], d4[s2]);
                    }
            }
            const float f = dkf[rr];
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2) d4[s2] *= f;
            for (int i = rr; i < 64; ++i) {   // C[i][j] = 0 for j > i
                const float cv = Cs[i * P64 + rr];
                const float4 o4 = l4(&dot[i * CTP + cc4]);
                d4[0] = fmaf(cv, o4.x, d4[0]), d4[1] = fmaf(cv, o4.y, d4[1]);
                d4[2] = fmaf(cv, o4.z, d4[2]), d4[3] = fmaf(cv, o4.w, d4[3]);
            }
            *reinterpret_cast<float4*>(&Rt[rr * CTP + cc4]) = make_float4(r4[0], r4[1], r4[2], r4[3]);
            *reinterpret_cast<float4*>(&dRt[rr * CTP + cc4]) = make_float4(d4[0], d4[1], d4[2], d4[3]);
        }
        __syncthreads();
        // dQd += dO H^T, dKd += R D'^T, dW -= dR H^T (4 x CW blocks, contracting the tile's 16
        // columns)
#pragma unroll 4
        for (int cc = 0; cc < kCT; ++cc) {
            float ov[4], rv[4], drv[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                ov[r] = dot[(i0 + r) * CTP + cc];
                rv[r] = Rt[(i0 + r) * CTP + cc];
                drv[r] = dRt[(i0 + r) * CTP + cc];
            }
            float hv[CW], dv[CW];
#pragma unroll
            for (int w = 0; w < CW; w += 4) {
                const float4 h4 = l4(&Ht[cc * KP + l0 + w]), e4 = l4(&Dt[cc * KP + l0 + w]);
                hv[w] = h4.x, hv[w + 1] = h4.y, hv[w + 2] = h4.z, hv[w + 3] = h4.w;
                dv[w] = e4.x, dv[w + 1] = e4.y, dv[w + 2] = e4.z, dv[w + 3] = e4.w;
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int w = 0; w < CW; ++w) {
                    dQd[r][w] = fmaf(ov[r], hv[w], dQd[r][w]);
                    dKd[r][w] = fmaf(rv[r], dv[w], dKd[r][w]);
                    dW[r][w] = fmaf(-drv[r], hv[w], dW[r][w]);
                }
        }
        // dC += dO R^T and dA += dR (diag(beta) V)^T (4 x 4 blocks)
        {
            const int a0 = (tid >> 4) * 4, b0 = (tid & 15) * 4;
            float dc[4][4] = {}, dav[4][4] = {};
#pragma unroll
            for (int cc = 0; cc < kCT; cc += 4) {
                float4 o4[4], dr4[4], r4[4], v4[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    o4[r] = l4(&dot[(a0 + r) * CTP + cc]);
                    dr4[r] = l4(&dRt[(a0 + r) * CTP + cc]);
                    r4[r] = l4(&Rt[(b0 + r) * CTP + cc]);
                    v4[r] = l4(&vt[(b0 + r) * CTP + cc]);
                }
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int s2 = 0; s2 < 4; ++s2) {
                        dc[r][s2] += o4[r].x * r4[s2].x + o4[r].y * r4[s2].y + o4[r].z * r4[s2].z + o4[r].w * r4[s2].w;
                        dav[r][s2] += dr4[r].x * v4[s2].x + dr4[r].y * v4[s2].y + dr4[r].z * v4[s2].z + dr4[r].w * v4[s2].w;
                    }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float4* pc = reinterpret_cast<float4*>(&dCs[(a0 + r) * P64 + b0]);
                float4* pa = reinterpret_cast<float4*>(&dAs[(a0 + r) * P64 + b0]);
                float4 x = *pc, y = *pa;
                x.x += dc[r][0], x.y += dc[r][1], x.z += dc[r][2], x.w += dc[r][3];
                y.x += dav[r][0] * bet[b0], y.y += dav[r][1] * bet[b0 + 1];
                y.z += dav[r][2] * bet[b0 + 2], y.w += dav[r][3] * bet[b0 + 3];
                *pc = x;
                *pa = y;
            }
        }
        // X = A^T dR: dv = beta X, dbeta += rowsum(X . V)
        {
            float x4[4] = {};
            for (int i = rr; i < 64; ++i) {   // A[i][j] = 0 for j > i
                const float a = As[i * P64 + rr];
                const float4 d4 = l4(&dRt[i * CTP + cc4]);
                x4[0] = fmaf(a, d4.x, x4[0]), x4[1] = fmaf(a, d4.y, x4[1]);
                x4[2] = fmaf(a, d4.z, x4[2]), x4[3] = fmaf(a, d4.w, x4[3]);
            }
            const float be = bet[rr];
            const float4 v4 = l4(&vt[rr * CTP + cc4]);
            float* out = p.dv + ((row0 + rr) * H + h) * V + c0 + cc4;
            out[0] = be * x4[0], out[1] = be * x4[1], out[2] = be * x4[2], out[3] = be * x4[3];
            xv += x4[0] * v4.x + x4[1] * v4.y + x4[2] * v4.z + x4[3] * v4.w;
        }
        __syncthreads();
    }
    // <D', H> over the whole state: one partial per warp (red[0..7]); rowsum(X . V) over the
    // four threads of a row
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) deg += __shfl_xor_sync(0xffffffffu, deg, off);
    if (lane == 0) red[tid >> 5] = deg;
    xv += __shfl_xor_sync(0xffffffffu, xv, 1);
    xv += __shfl_xor_sync(0xffffffffu, xv, 2);
    if ((tid & 3) == 0) dbs[rr] += xv;
    // ---- (6) dW into shared memory (W is no longer needed)
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int w = 0; w < CW; w += 4)
            *reinterpret_cast<float4*>(&Ws[(i0 + r) * KP + l0 + w]) =
                make_float4(dW[r][w], dW[r][w + 1], dW[r][w + 2], dW[r][w + 3]);
    __syncthreads();
    // ---- (7) Y = A^T dW: dKr = beta Y enters dk as e^Gx dKr; dbeta += rowsum(Y . Kr);
    //      dGx += rowsum(dKr . Kr)
    float dkacc[4][CW];
    {
        float y[4][CW] = {};
        for (int i = i0; i < 64; ++i) {   // rows j = i0.. of A^T need A[i][j], i >= j
            float dwv[CW];
#pragma unroll
            for (int w = 0; w < CW; w += 4) {
                const float4 t4 = l4(&Ws[i * KP + l0 + w]);
                dwv[w] = t4.x, dwv[w + 1] = t4.y, dwv[w + 2] = t4.z, dwv[w + 3] = t4.w;
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float a = (i >= i0 + r) ? As[i * P64 + i0 + r] : 0.f;
#pragma unroll
                for (int w = 0; w < CW; ++w) y[r][w] = fmaf(a, dwv[w], y[r][w]);
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int j = i0 + r;
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < CW; ++w) {
                s = fmaf(y[r][w], ks[j * KP + l0 + w], s);
                dkacc[r][w] = ekr[j] * y[r][w];   // e^Gx beta Y = e^Gx dKr
            }
            // Y . Kr = e^Gx (Y . k); dKr . Kr = beta e^Gx (Y . k)
            s = half_sum(s);
            if ((tid & 15) == 0) {
                dbs[j] += eGx[j] * s;
                dGx[j] += ekr[j] * s;
            }
        }
    }
    // ---- (8) dA += dW (diag(beta e^Gx) K)^T (4 x 4 blocks)
    {
        const int a0 = (tid >> 4) * 4, b0 = (tid & 15) * 4;
        float acc[4][4] = {};
#pragma unroll 2
        for (int l = 0; l < KD; l += 4) {
            float4 w4[4], k4[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                w4[r] = l4(&Ws[(a0 + r) * KP + l]);
                k4[r] = l4(&ks[(b0 + r) * KP + l]);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int s2 = 0; s2 < 4; ++s2)
                    acc[r][s2] += w4[r].x * k4[s2].x + w4[r].y * k4[s2].y + w4[r].z * k4[s2].z + w4[r].w * k4[s2].w;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            float4* pa = reinterpret_cast<float4*>(&dAs[(a0 + r) * P64 + b0]);
            float4 y = *pa;
            y.x += acc[r][0] * ekr[b0], y.y += acc[r][1] * ekr[b0 + 1];
            y.z += acc[r][2] * ekr[b0 + 2], y.w += acc[r][3] * ekr[b0 + 3];
            *pa = y;
        }
    }
    __syncthreads();
    // ---- (9) T1 = A^T dA (into the tile region), then dL = -tril(T1 A^T, -1) over dA
    float* T1 = sm + L::t;
    {
        const int a0 = (tid >> 4) * 4, b0 = (tid & 15) * 4;
        float acc[4][4] = {};
        for (int i = a0; i < 64; ++i) {   // A[i][j] = 0 for j > i
            const float4 d4 = l4(&dAs[i * P64 + b0]);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float a = (i >= a0 + r) ? As[i * P64 + a0 + r] : 0.f;
                acc[r][0] = fmaf(a, d4.x, acc[r][0]), acc[r][1] = fmaf(a, d4.y, acc[r][1]);
                acc[r][2] = fmaf(a, d4.z, acc[r][2]), acc[r][3] = fmaf(a, d4.w, acc[r][3]);
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
            *reinterpret_cast<float4*>(&T1[(a0 + r) * P64 + b0]) =
                make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
    }
    __syncthreads();
    {
        const int a0 = (tid >> 4) * 4, b0 = (tid & 15) * 4;   // dL rows j = a0.., columns m = b0..
        float acc[4][4] = {};
        for (int n = 0; n < b0 + 4; ++n) {   // A[m][n] = 0 for n > m
            float tv[4], av[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) tv[r] = T1[(a0 + r) * P64 + n];
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2) av[s2] = As[(b0 + s2) * P64 + n];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int s2 = 0; s2 < 4; ++s2) acc[r][s2] = fmaf(tv[r], av[s2], acc[r][s2]);
        }
        __syncthreads();   // every thread has read dA's rows through T1 ... and T1 is complete
        // dL, then its terms: dbeta += rowsum(dL . P); dP = beta dL; t = dP . P:
        // dGx_i += rowsum(t), dG_j -= colsum(t); S = dP . e^(Gx_i - G_j) over dA
        float rsb[4] = {}, rsg[4] = {}, csg[4] = {};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int j = a0 + r;
            float sv[4];
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2) {
                const int m = b0 + s2;
                const float dl = (m < j) ? -acc[r][s2] : 0.f;
                const float pv = Ps[j * P64 + m];
                const float dp = bet[j] * dl;
                rsb[r] = fmaf(dl, pv, rsb[r]);
                rsg[r] = fmaf(dp, pv, rsg[r]);
                csg[s2] = fmaf(dp, pv, csg[s2]);
                sv[s2] = (m < j) ? dp * expf(Gx[j] - G[m]) : 0.f;
            }
            *reinterpret_cast<float4*>(&dAs[j * P64 + b0]) = make_float4(sv[0], sv[1], sv[2], sv[3]);
        }
        // dC's terms: t' = dC . C (j <= i): dG_i += rowsum(t'), dG_j -= colsum(t');
        // S' = dC . e^(G_i - G_j) over dC
        float rsc[4] = {}, csc[4] = {};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = a0 + r;
            float sv[4];
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2) {
                const int j = b0 + s2;
                const float dc = (j <= i) ? dCs[i * P64 + j] : 0.f;
                const float t = dc * Cs[i * P64 + j];
                rsc[r] += t;
                csc[s2] += t;
                sv[s2] = (j <= i) ? dc * expf(G[i] - G[j]) : 0.f;
            }
            *reinterpret_cast<float4*>(&dCs[i * P64 + b0]) = make_float4(sv[0], sv[1], sv[2], sv[3]);
        }
        // row sums over the 16 threads of a row block (one half-warp); column sums through
        // shared memory (T1 is dead), one partial per row block
        float* part = sm + L::t;   // [16][64]
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float b = half_sum(rsb[r]), g = half_sum(rsg[r]), c = half_sum(rsc[r]);
            if ((tid & 15) == 0) {
                dbs[a0 + r] += b;
                dGx[a0 + r] += g;
                dG[a0 + r] += c;
            }
            part[(tid >> 4) * 64 + b0 + r] = -csg[r] - csc[r];
        }
    }
    __syncthreads();
    if (tid < 64) {
        float a = 0.f;
#pragma unroll
        for (int g = 0; g < 16; ++g) a += sm[L::t + g * 64 + tid];
        dG[tid] += a;
    }
    __syncthreads();
    // ---- (10) q back into the tile region (T1 is dead)
    for (int e = tid; e < 64 * KD; e += kCgThreads) {
        const int i = e / KD, l = e % KD;
        qs[i * KP + l] = ldv(p.q, ((row0 + i) * H + h) * KD + l, p.in_bf16);
    }
    __syncthreads();
    // ---- (11) dq = S' k + e^G dQd;  dk = S k + S^T k + S'^T q + e^(Gn - G) dKd + e^Gx dKr;
    //      gate terms of Qd and Kd
    {
        float dq[4][CW] = {}, dk[4][CW] = {};
        for (int j = 0; j < 64; ++j) {
            float kv[CW], qv[CW];
#pragma unroll
            for (int w = 0; w < CW; w += 4) {
                const float4 k4 = l4(&ks[j * KP + l0 + w]), q4 = l4(&qs[j * KP + l0 + w]);
                kv[w] = k4.x, kv[w + 1] = k4.y, kv[w + 2] = k4.z, kv[w + 3] = k4.w;
                qv[w] = q4.x, qv[w + 1] = q4.y, qv[w + 2] = q4.z, qv[w + 3] = q4.w;
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = i0 + r;
                const float s1 = dCs[i * P64 + j];                        // S'[i][j]
                const float s2 = dAs[i * P64 + j] + dAs[j * P64 + i];     // S[i][j] + S[j][i]
                const float s3 = dCs[j * P64 + i];                        // S'[j][i]
#pragma unroll
                for (int w = 0; w < CW; ++w) {
                    dq[r][w] = fmaf(s1, kv[w], dq[r][w]);
                    dk[r][w] = fmaf(s2, kv[w], fmaf(s3, qv[w], dk[r][w]));
                }
            }
        }
        float tg[4] = {}, tk[4] = {};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = i0 + r;
            const float eg = eG[i], f = dkf[i];
            float* oq = p.dq + ((row0 + i) * H + h) * KD + l0;
            float* ok = p.dk + ((row0 + i) * H + h) * KD + l0;
#pragma unroll
            for (int w = 0; w < CW; ++w) {
                const float qd = eg * qs[i * KP + l0 + w];   // Qd
                const float kd = f * ks[i * KP + l0 + w];    // Kd
                tg[r] = fmaf(dQd[r][w], qd, tg[r]);
                tk[r] = fmaf(dKd[r][w], kd, tk[r]);
                oq[w] = fmaf(eg, dQd[r][w], dq[r][w]);
                ok[w] = fmaf(f, dKd[r][w], dk[r][w]) + dkacc[r][w];
            }
        }
        float tks = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float t = half_sum(tg[r] - tk[r]);
            tks += tk[r];
            if ((tid & 15) == 0) dG[i0 + r] += t;
        }
        tks = half_sum(tks);   // this row block's share of sum(dKd . Kd), part of dGn
        if ((tid & 15) == 0) red[16 + (tid >> 4)] = tks;
    }
    __syncthreads();
    // ---- (12) dg = reverse cumulative sum of dG + dGx (+ dGn at the last token), minus dGx for
    //      the read before the decay; dbeta
    if (tid < 32) {
        float tk = 0.f, hd = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) tk += red[16 + i];
#pragma unroll
        for (int i = 0; i < 8; ++i) hd += red[i];
        const float dGn = tk + expf(Gn) * hd;
        // lane owns tokens 2 lane, 2 lane + 1; reverse cumulative sum over 64 tokens
        float a0 = dG[2 * lane] + dGx[2 * lane];
        float a1 = dG[2 * lane + 1] + dGx[2 * lane + 1] + (lane == 31 ? dGn : 0.f);
        float s = a0 + a1;   // inclusive suffix sum from the right
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_down_sync(0xffffffffu, s, off);
            if (lane + off < 32) s += o;
        }
        const float suf1 = s - a0;   // sum over tokens 2 lane + 1 ..
        const float suf0 = s;        // sum over tokens 2 lane ..
        const float g0 = suf0 - (p.decay_first ? 0.f : dGx[2 * lane]);
        const float g1 = suf1 - (p.decay_first ? 0.f : dGx[2 * lane + 1]);
        const long long r0i = (row0 + 2 * lane) * H + h;
        p.dg[r0i] = g0;
        p.dg[r0i + H] = g1;
        p.dbeta[r0i] = dbs[2 * lane];
        p.dbeta[r0i + H] = dbs[2 * lane + 1];
    }
}

template <int KD>
cudaError_t launch_chunk_grad_k(const ChunkGradParams& p, cudaStream_t s) {
    using L = CgSmem<KD>;
    auto kern = chunk_grad_kernel<KD>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::bytes);
    if (e != cudaSuccess) return e;
    const long long nblk = (long long)p.B * p.H * (p.T / kChunk);
    if (nblk == 0) return cudaSuccess;
    kern<<<(unsigned)nblk, kCgThreads, L::bytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_grad(const ChunkGradParams& p, cudaStream_t s) {
    // bf16 inputs: the tensor-core products (tf32 operands keep the bf16 bar); fp32 inputs keep
    // fp32 products on the CUDA cores
    if (p.in_bf16) return launch_chunk_grad_mma(p, s);
    return p.K == 64 ? launch_chunk_grad_k<64>(p, s) : launch_chunk_grad_k<128>(p, s);
}

}  // namespace gdn
