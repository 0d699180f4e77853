// gdn_bwd_chunk_mma.cu -- the per-chunk gradients of the backward pass (dq, dk, dv, dg, dbeta)
// with their products on the tensor cores, for bf16 inputs.
//
// The same computation, in the same order and with the same names, as chunk_grad_kernel
// (gdn_bwd_chunk.cu; "RFC: HyperParallel Linear Attention Context Parallel", section 6.4.3,
// backward_state + backward_finish; the chunk equations of "Context Parallelism in ART",
// section 08, taken backwards): every (b, h, chunk) is one independent CTA that starts from
// the chunk's inputs, the state H entering it and the gradient D' on the state leaving it.
// Every product -- K K^T, Q K^T, W, R, dR, dQd, dKd, dW, dC, dA, A^T dR, A^T dW, A^T dA and its
// product with A^T, dq and dk from the score gradients -- is a sum of warp-level m16n8k8 MMAs
// (tf32 operands rounded to nearest, fp32 accumulation) whose fragments are read straight from
// the fp32 matrices in shared memory; the triangular inverse, the gates, the masks and the
// per-token sums stay on the CUDA cores. Row pitches of 4 mod 32 words make the fragment
// reads of a row-major operand free of bank conflicts.
//
// Warp tiles (8 warps): 64 x 64 products 16 x 32 per warp, 64 x K products 32 x 32 (K = 128)
// or 16 x 32 (K = 64), the 64 x 16 products of one V tile 16 x 8. dQd, dKd, dW, dC and dA
// accumulate in registers over the V tiles. Every per-token sum is taken in a fixed order
// (shuffles within a warp, per-warp partials summed in order), so the results do not vary
// from run to run.
#include <cuda_bf16.h>

#include "gdn_internal.h"
#include "gdn_warp_mma.cuh"

namespace gdn {
namespace {

constexpr int kMgThreads = 256;
constexpr int kMT = 16;   // V columns per tile

__device__ __forceinline__ float ldin(const void* base, long long idx, int bf16) {
    if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
    return reinterpret_cast<const float*>(base)[idx];
}
// 16-byte asynchronous copies global -> shared (both addresses 16-byte aligned)
__device__ __forceinline__ void cp16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait_prior() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
template <int KD>
struct MgSmem {
    static constexpr int P64 = 68;          // row pitch of the 64 x 64 matrices
    static constexpr int KP = KD + 4;       // row pitch of the 64 x KD matrices and H^T tiles
    static constexpr int CTP = kMT + 4;     // row pitch of the 64 x 16 fp32 tiles (R, dR, dO)
    static constexpr int HP = kMT + 8;      // row pitch of the K x 16 tiles of H and D'
    static constexpr int VPB = kMT + 8;     // row pitch (bf16 elements) of the 64 x 16 bf16 tiles
    static constexpr int k = 0;                          // k       [64][KP]
    static constexpr int a = k + 64 * KP;                // A       [64][P64]
    static constexpr int c = a + 64 * P64;               // C, then S'
    static constexpr int p = c + 64 * P64;               // P
    static constexpr int da = p + 64 * P64;              // dA, then S
    static constexpr int w = da + 64 * P64;              // W, then dW  [64][KP]
    static constexpr int t = w + 64 * KP;                // tile region (see below)
    // tile region: q before the tile loop (then the inverse's scratch); during it two buffers
    // of the tile's inputs as copied -- H and D' [KD][HP] fp32, v [64][VPB] bf16, dO [64][CTP]
    // fp32 or [64][VPB] bf16 -- and R, dR [64][CTP]; A^T dA [64][P64] after it, then q again
    static constexpr int BUF = 2 * KD * HP + 64 * VPB / 2 + 64 * CTP;   // floats per buffer
    static constexpr int t_buf = t, t_r = t_buf + 2 * BUF, t_dr = t_r + 64 * CTP;
    static constexpr int tile_end = t_dr + 64 * CTP;
    static constexpr int s = (tile_end > t + 64 * KP ? tile_end : t + 64 * KP);
    enum { G = 0, GX, EG, EGX, DKF, BET, EKR, DG, DGX, DBETA, RED, NS };
    static constexpr int part = s + NS * 64;             // per-warp partial sums [12][64]
    static constexpr int total = part + 12 * 64;
    static constexpr size_t bytes = sizeof(float) * total;
    static_assert(64 * P64 <= tile_end - t || 64 * P64 <= 64 * KP, "A^T dA fits the tile region");
    static_assert(bytes <= 232448, "shared memory budget");
};

template <int KD, bool DOB>   // DOB: dO in bf16 (the output dtype)
__global__ void __launch_bounds__(kMgThreads, 1) chunk_grad_mma_kernel(ChunkGradParams p) {
    using L = MgSmem<KD>;
    constexpr int KP = L::KP, P64 = L::P64, CTP = L::CTP, HP = L::HP, VPB = L::VPB;
    // 64 x K warp tiles: 32 x 32 at K = 128 (column groups of 32: 4), 16 x 32 at K = 64 (2)
    constexpr int MTK = KD == 128 ? 2 : 1;
    constexpr int NCG = KD / 32;
    extern __shared__ float4 smv[];
    float* sm = reinterpret_cast<float*>(smv);
    float* ks = sm + L::k;
    float* As = sm + L::a;
    float* Cs = sm + L::c;
    float* Ps = sm + L::p;
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
    float* part = sm + L::part;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g4 = lane >> 2, t4 = lane & 3;
    const int nch = p.T / kChunk;
    const int c = blockIdx.x % nch;
    const int bh = blockIdx.x / nch;
    const int b = bh / p.H, h = bh % p.H;
    const int H = p.H, V = p.V;
    const long long row0 = (long long)b * p.T + (long long)c * kChunk;   // flattened (b, t)
    const long long st0 = ((long long)c * p.B * H + bh) * KD * V;        // Hc / Dc offset
    // warp tiles: 64 x 64 outputs, 64 x K outputs, one V tile's 64 x 16 outputs
    const int m64 = 16 * (warp & 3), n64 = 32 * (warp >> 2), cg64 = warp >> 2;
    const int mK = KD == 128 ? 32 * (warp & 1) : 16 * (warp & 3);
    const int nK = KD == 128 ? 32 * (warp >> 1) : 32 * (warp >> 2);
    const int cgK = KD == 128 ? (warp >> 1) : (warp >> 2);
    const int mV = 16 * (warp & 3), nV = 8 * (warp >> 2);

    // ---- (1) k, and q into the tile region (bf16, eight per 16-byte load, every load of a
    //      thread in flight before the first store); the gates and beta
    float* qs = sm + L::t;
    constexpr int NKV = 64 * KD / 8 / kMgThreads;
    auto load_rows = [&](const void* src, float* dst) {
        uint4 u[NKV];
#pragma unroll
        for (int n = 0; n < NKV; ++n) {
            const int e = tid + n * kMgThreads, i = e / (KD / 8), l8 = 8 * (e % (KD / 8));
            u[n] = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(src) +
                                                    ((row0 + i) * H + h) * KD + l8);
        }
#pragma unroll
        for (int n = 0; n < NKV; ++n) {
            const int e = tid + n * kMgThreads, i = e / (KD / 8), l8 = 8 * (e % (KD / 8));
            float* d = dst + i * KP + l8;
            *reinterpret_cast<float4*>(d) =
                make_float4(__uint_as_float(u[n].x << 16), __uint_as_float(u[n].x & 0xFFFF0000u),
                            __uint_as_float(u[n].y << 16), __uint_as_float(u[n].y & 0xFFFF0000u));
            *reinterpret_cast<float4*>(d + 4) =
                make_float4(__uint_as_float(u[n].z << 16), __uint_as_float(u[n].z & 0xFFFF0000u),
                            __uint_as_float(u[n].w << 16), __uint_as_float(u[n].w & 0xFFFF0000u));
        }
    };
    load_rows(p.k, ks);
    load_rows(p.q, qs);
    if (tid < 64) {
        const long long row = (row0 + tid) * H + h;
        Gx[tid] = ldin(p.g, row, p.in_bf16);   // raw gate until the cumsum
        bet[tid] = ldin(p.beta, row, p.in_bf16);
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
        float sq[1][4][4] = {}, sk[1][4][4] = {};
        wtile<1, 4>(sq, m64, n64, KD, lane, [&](int r, int l) { return qs[r * KP + l]; },
                    [&](int l, int j) { return ks[j * KP + l]; });
        wtile<1, 4>(sk, m64, n64, KD, lane, [&](int r, int l) { return ks[r * KP + l]; },
                    [&](int l, int j) { return ks[j * KP + l]; });
        __syncthreads();   // the gates' exponentials are in place
        wtile_each<1, 4>(sq, m64, n64, lane, [&](int i, int j, float& v) {
            Cs[i * P64 + j] = (j <= i) ? expf(G[i] - G[j]) * v : 0.f;
        });
        wtile_each<1, 4>(sk, m64, n64, lane, [&](int i, int j, float& v) {
            Ps[i * P64 + j] = (j < i) ? expf(Gx[i] - G[j]) * v : 0.f;
            As[i * P64 + j] = 0.f;
        });
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
    // ---- (4) W = A diag(beta e^Gx) K
    {
        float wacc[MTK][4][4] = {};
        wtile<MTK, 4>(wacc, mK, nK, 64, lane, [&](int i, int j) { return As[i * P64 + j] * ekr[j]; },
                      [&](int j, int l) { return ks[j * KP + l]; });
        wtile_each<MTK, 4>(wacc, mK, nK, lane, [&](int i, int l, float& v) { Ws[i * KP + l] = v; });
    }
    __syncthreads();

    // ---- (5) the V tiles, each copied into shared memory while the one before it computes
    float* Rt = sm + L::t_r;
    float* dRt = sm + L::t_dr;
    auto buf_h = [&](int bb) { return sm + L::t_buf + bb * L::BUF; };            // H [KD][HP]
    auto buf_d = [&](int bb) { return buf_h(bb) + KD * HP; };                     // D' [KD][HP]
    auto buf_v = [&](int bb) {                                                    // v [64][VPB]
        return reinterpret_cast<__nv_bfloat16*>(buf_h(bb) + 2 * KD * HP);
    };
    auto buf_o = [&](int bb) { return buf_h(bb) + 2 * KD * HP + 64 * VPB / 2; };  // dO
    auto issue_tile = [&](int c0, int bb) {
        float* hb = buf_h(bb);
        float* db = buf_d(bb);
        for (int e = tid; e < KD * (kMT / 4); e += kMgThreads) {
            const int l = e / (kMT / 4), q4 = 4 * (e % (kMT / 4));
            const long long g0 = st0 + (long long)l * V + c0 + q4;
            cp16(hb + l * HP + q4, p.Hc + g0);
            cp16(db + l * HP + q4, p.Dc + g0);
        }
        __nv_bfloat16* vb = buf_v(bb);
        for (int e = tid; e < 64 * (kMT / 8); e += kMgThreads) {
            const int j = e / (kMT / 8), q8 = 8 * (e % (kMT / 8));
            cp16(vb + j * VPB + q8,
                 reinterpret_cast<const __nv_bfloat16*>(p.v) + ((row0 + j) * H + h) * V + c0 + q8);
        }
        if (DOB) {
            __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(buf_o(bb));
            for (int e = tid; e < 64 * (kMT / 8); e += kMgThreads) {
                const int j = e / (kMT / 8), q8 = 8 * (e % (kMT / 8));
                cp16(ob + j * VPB + q8,
                     reinterpret_cast<const __nv_bfloat16*>(p.dO) + ((row0 + j) * H + h) * V + c0 + q8);
            }
        } else {
            float* ob = buf_o(bb);
            for (int e = tid; e < 64 * (kMT / 4); e += kMgThreads) {
                const int j = e / (kMT / 4), q4 = 4 * (e % (kMT / 4));
                cp16(ob + j * CTP + q4,
                     reinterpret_cast<const float*>(p.dO) + ((row0 + j) * H + h) * V + c0 + q4);
            }
        }
        cp_commit();
    };
    float dQd[MTK][4][4] = {}, dKd[MTK][4][4] = {}, dRH[MTK][4][4] = {};   // dW = -dR H^T
    float dCa[1][4][4] = {}, dAa[1][4][4] = {};
    float deg = 0.f;                  // this thread's share of <D', H>
    float xv0 = 0.f, xv1 = 0.f;       // rowsum(X . V) over this thread's columns, rows mV + g4, + 8
    issue_tile(0, 0);
#pragma unroll 1
    for (int c0 = 0; c0 < V; c0 += kMT) {
        const int bb = (c0 / kMT) & 1;
        if (c0 + kMT < V) issue_tile(c0 + kMT, bb ^ 1);
        else cp_commit();   // an empty group keeps "all but the newest" meaning this tile
        cp_wait_prior();
        __syncthreads();
        const float* Hn = buf_h(bb);
        const float* Dn = buf_d(bb);
        const __nv_bfloat16* vbt = buf_v(bb);
        const float* obf = buf_o(bb);
        const __nv_bfloat16* obh = reinterpret_cast<const __nv_bfloat16*>(buf_o(bb));
        auto vt = [&](int j, int cc) { return __bfloat162float(vbt[j * VPB + cc]); };
        auto dot = [&](int j, int cc) {
            return DOB ? __bfloat162float(obh[j * VPB + cc]) : obf[j * CTP + cc];
        };
        for (int e = tid; e < KD * kMT; e += kMgThreads) {
            const int l = e / kMT, cc = e % kMT;
            deg = fmaf(Hn[l * HP + cc], Dn[l * HP + cc], deg);
        }
        // R = A diag(beta) V - W H and dR = Kd D' + C^T dO on this tile's 16 columns
        {
            float r[1][1][4] = {}, d[1][1][4] = {};
            wtile<1, 1>(r, mV, nV, 64, lane, [&](int i, int j) { return As[i * P64 + j] * bet[j]; },
                        [&](int j, int cc) { return vt(j, cc); });
            wtile<1, 1>(r, mV, nV, KD, lane, [&](int i, int l) { return -Ws[i * KP + l]; },
                        [&](int l, int cc) { return Hn[l * HP + cc]; });
            wtile<1, 1>(d, mV, nV, KD, lane, [&](int i, int l) { return dkf[i] * ks[i * KP + l]; },
                        [&](int l, int cc) { return Dn[l * HP + cc]; });
            wtile<1, 1>(d, mV, nV, 64, lane, [&](int i, int j) { return Cs[j * P64 + i]; },
                        [&](int j, int cc) { return dot(j, cc); });
            wtile_each<1, 1>(r, mV, nV, lane, [&](int i, int cc, float& v) { Rt[i * CTP + cc] = v; });
            wtile_each<1, 1>(d, mV, nV, lane, [&](int i, int cc, float& v) { dRt[i * CTP + cc] = v; });
        }
        __syncthreads();
        // dQd += dO H^T, dKd += R D'^T, dR H^T (= -dW), contracting the tile's 16 columns
        wtile<MTK, 4>(dQd, mK, nK, kMT, lane, [&](int i, int cc) { return dot(i, cc); },
                      [&](int cc, int l) { return Hn[l * HP + cc]; });
        wtile<MTK, 4>(dKd, mK, nK, kMT, lane, [&](int i, int cc) { return Rt[i * CTP + cc]; },
                      [&](int cc, int l) { return Dn[l * HP + cc]; });
        wtile<MTK, 4>(dRH, mK, nK, kMT, lane, [&](int i, int cc) { return dRt[i * CTP + cc]; },
                      [&](int cc, int l) { return Hn[l * HP + cc]; });
        // dC += dO R^T and dA += dR (diag(beta) V)^T
        wtile<1, 4>(dCa, m64, n64, kMT, lane, [&](int i, int cc) { return dot(i, cc); },
                    [&](int cc, int j) { return Rt[j * CTP + cc]; });
        wtile<1, 4>(dAa, m64, n64, kMT, lane, [&](int i, int cc) { return dRt[i * CTP + cc]; },
                    [&](int cc, int j) { return bet[j] * vt(j, cc); });
        // X = A^T dR: dv = beta X, rowsum(X . V)
        {
            float x[1][1][4] = {};
            wtile<1, 1>(x, mV, nV, 64, lane, [&](int j, int i) { return As[i * P64 + j]; },
                        [&](int i, int cc) { return dRt[i * CTP + cc]; });
            const int j0 = mV + g4, cc = nV + 2 * t4;
            const float b0 = bet[j0], b1 = bet[j0 + 8];
            *reinterpret_cast<float2*>(p.dv + ((row0 + j0) * H + h) * V + c0 + cc) =
                make_float2(b0 * x[0][0][0], b0 * x[0][0][1]);
            *reinterpret_cast<float2*>(p.dv + ((row0 + j0 + 8) * H + h) * V + c0 + cc) =
                make_float2(b1 * x[0][0][2], b1 * x[0][0][3]);
            xv0 += x[0][0][0] * vt(j0, cc) + x[0][0][1] * vt(j0, cc + 1);
            xv1 += x[0][0][2] * vt(j0 + 8, cc) + x[0][0][3] * vt(j0 + 8, cc + 1);
        }
        __syncthreads();
    }
    // ---- (6) dW into shared memory (W is no longer needed); the per-token sums so far
    wtile_each<MTK, 4>(dRH, mK, nK, lane, [&](int i, int l, float& v) { Ws[i * KP + l] = -v; });
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) deg += __shfl_xor_sync(0xffffffffu, deg, off);
    if (lane == 0) red[warp] = deg;   // <D', H>: one partial per warp
    xv0 = quad_sum(xv0);
    xv1 = quad_sum(xv1);
    if (t4 == 0) {
        part[(warp >> 2) * 64 + mV + g4] = xv0;
        part[(warp >> 2) * 64 + mV + g4 + 8] = xv1;
    }
    __syncthreads();
    if (tid < 64) dbs[tid] += part[tid] + part[64 + tid];
    __syncthreads();
    // ---- (7) Y = A^T dW: dKr = beta Y enters dk as e^Gx dKr; dbeta += rowsum(Y . Kr);
    //      dGx += rowsum(dKr . Kr)
    float dkacc[MTK][4][4] = {};
    wtile<MTK, 4>(dkacc, mK, nK, 64, lane, [&](int j, int i) { return As[i * P64 + j]; },
                  [&](int i, int l) { return Ws[i * KP + l]; });
    {
        float rs[MTK][2] = {};
#pragma unroll
        for (int mt = 0; mt < MTK; ++mt)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = mK + 16 * mt + g4 + 8 * (e >> 1), l = nK + 8 * nt + 2 * t4 + (e & 1);
                    rs[mt][e >> 1] = fmaf(dkacc[mt][nt][e], ks[j * KP + l], rs[mt][e >> 1]);
                    dkacc[mt][nt][e] *= ekr[j];   // e^Gx beta Y = e^Gx dKr
                }
#pragma unroll
        for (int mt = 0; mt < MTK; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float s = quad_sum(rs[mt][hh]);
                if (t4 == 0) part[cgK * 64 + mK + 16 * mt + g4 + 8 * hh] = s;
            }
    }
    __syncthreads();
    if (tid < 64) {
        float s = 0.f;   // Y . Kr = e^Gx (Y . k); dKr . Kr = beta e^Gx (Y . k)
#pragma unroll
        for (int q = 0; q < NCG; ++q) s += part[q * 64 + tid];
        dbs[tid] += eGx[tid] * s;
        dGx[tid] += ekr[tid] * s;
    }
    // ---- (8) dA += dW (diag(beta e^Gx) K)^T, then dA into shared memory
    wtile<1, 4>(dAa, m64, n64, KD, lane, [&](int i, int l) { return Ws[i * KP + l]; },
                [&](int l, int j) { return ekr[j] * ks[j * KP + l]; });
    wtile_each<1, 4>(dAa, m64, n64, lane, [&](int i, int j, float& v) { dAs[i * P64 + j] = v; });
    __syncthreads();
    // ---- (9) T1 = A^T dA (into the tile region), then dL = -tril(T1 A^T, -1)
    float* T1 = sm + L::t;
    {
        float t1[1][4][4] = {};
        wtile<1, 4>(t1, m64, n64, 64, lane, [&](int a, int i) { return As[i * P64 + a]; },
                    [&](int i, int bb) { return dAs[i * P64 + bb]; });
        wtile_each<1, 4>(t1, m64, n64, lane, [&](int a, int bb, float& v) { T1[a * P64 + bb] = v; });
    }
    __syncthreads();
    {
        float tl[1][4][4] = {};
        wtile<1, 4>(tl, m64, n64, 64, lane, [&](int j, int n) { return T1[j * P64 + n]; },
                    [&](int n, int m) { return As[m * P64 + n]; });
        // dL and its terms: dbeta += rowsum(dL . P); dP = beta dL; t = dP . P: dGx_j += rowsum(t),
        // dG_m -= colsum(t); S = dP . e^(Gx_j - G_m) over dA. dC's terms: t' = dC . C (m <= j):
        // dG_j += rowsum(t'), dG_m -= colsum(t'); S' = dC . e^(G_j - G_m) over C
        float rsb[2] = {}, rsg[2] = {}, rsc[2] = {}, cs[4][2] = {};
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = m64 + g4 + 8 * (e >> 1), m = n64 + 8 * nt + 2 * t4 + (e & 1);
                const float dl = (m < j) ? -tl[0][nt][e] : 0.f;
                const float pv = Ps[j * P64 + m];
                const float dp = bet[j] * dl;
                rsb[e >> 1] = fmaf(dl, pv, rsb[e >> 1]);
                rsg[e >> 1] = fmaf(dp, pv, rsg[e >> 1]);
                dAs[j * P64 + m] = (m < j) ? dp * expf(Gx[j] - G[m]) : 0.f;
                const float dc = (m <= j) ? dCa[0][nt][e] : 0.f;
                const float tc = dc * Cs[j * P64 + m];
                rsc[e >> 1] += tc;
                cs[nt][e & 1] += fmaf(dp, pv, tc);
                Cs[j * P64 + m] = (m <= j) ? dc * expf(G[j] - G[m]) : 0.f;
            }
        // rows: the four lanes of a row, then the two column groups through shared memory;
        // columns: the eight lanes of a column, then the four row groups
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const float b2 = quad_sum(rsb[hh]), g2 = quad_sum(rsg[hh]), c2 = quad_sum(rsc[hh]);
            if (t4 == 0) {
                const int j = m64 + g4 + 8 * hh;
                part[(0 + cg64) * 64 + j] = b2;
                part[(2 + cg64) * 64 + j] = g2;
                part[(4 + cg64) * 64 + j] = c2;
            }
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float s = col_sum(cs[nt][u]);
                if (g4 == 0) part[(6 + (warp & 3)) * 64 + n64 + 8 * nt + 2 * t4 + u] = s;
            }
    }
    __syncthreads();
    if (tid < 64) {
        dbs[tid] += part[tid] + part[64 + tid];
        dGx[tid] += part[128 + tid] + part[192 + tid];
        dG[tid] += (part[256 + tid] + part[320 + tid]) -
                   (((part[384 + tid] + part[448 + tid]) + part[512 + tid]) + part[576 + tid]);
    }
    __syncthreads();
    // ---- (10) q back into the tile region (T1 is dead)
    load_rows(p.q, qs);
    __syncthreads();
    // ---- (11) dq = S' K + e^G dQd;  dk = S K + S^T K + S'^T Q + e^(Gn - G) dKd + e^Gx dKr;
    //      the gate terms of Qd and Kd
    {
        float tg[MTK][2] = {}, tk[MTK][2] = {};
#pragma unroll
        for (int mt = 0; mt < MTK; ++mt)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = mK + 16 * mt + g4 + 8 * (e >> 1), l = nK + 8 * nt + 2 * t4 + (e & 1);
                    const float eg = eG[i], f = dkf[i];
                    tg[mt][e >> 1] = fmaf(dQd[mt][nt][e], eg * qs[i * KP + l], tg[mt][e >> 1]);
                    tk[mt][e >> 1] = fmaf(dKd[mt][nt][e], f * ks[i * KP + l], tk[mt][e >> 1]);
                    dQd[mt][nt][e] *= eg;                                  // dq starts at e^G dQd
                    dKd[mt][nt][e] = fmaf(f, dKd[mt][nt][e], dkacc[mt][nt][e]);   // dk at ...
                }
        wtile<MTK, 4>(dQd, mK, nK, 64, lane, [&](int i, int j) { return Cs[i * P64 + j]; },
                      [&](int j, int l) { return ks[j * KP + l]; });
        wtile<MTK, 4>(dKd, mK, nK, 64, lane,
                      [&](int i, int j) { return dAs[i * P64 + j] + dAs[j * P64 + i]; },
                      [&](int j, int l) { return ks[j * KP + l]; });
        wtile<MTK, 4>(dKd, mK, nK, 64, lane, [&](int i, int j) { return Cs[j * P64 + i]; },
                      [&](int j, int l) { return qs[j * KP + l]; });
#pragma unroll
        for (int mt = 0; mt < MTK; ++mt)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int i = mK + 16 * mt + g4 + 8 * hh, l = nK + 8 * nt + 2 * t4;
                    const long long o = ((row0 + i) * H + h) * KD + l;
                    *reinterpret_cast<float2*>(p.dq + o) =
                        make_float2(dQd[mt][nt][2 * hh], dQd[mt][nt][2 * hh + 1]);
                    *reinterpret_cast<float2*>(p.dk + o) =
                        make_float2(dKd[mt][nt][2 * hh], dKd[mt][nt][2 * hh + 1]);
                }
        float tks = 0.f;
#pragma unroll
        for (int mt = 0; mt < MTK; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float d = quad_sum(tg[mt][hh] - tk[mt][hh]);
                tks += tk[mt][hh];
                if (t4 == 0) part[cgK * 64 + mK + 16 * mt + g4 + 8 * hh] = d;
            }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) tks += __shfl_xor_sync(0xffffffffu, tks, off);
        if (lane == 0) red[16 + warp] = tks;   // this warp's share of sum(dKd . Kd), part of dGn
    }
    __syncthreads();
    if (tid < 64) {
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < NCG; ++q) s += part[q * 64 + tid];
        dG[tid] += s;
    }
    __syncthreads();
    // ---- (12) dg = reverse cumulative sum of dG + dGx (+ dGn at the last token), minus dGx for
    //      the read before the decay; dbeta
    if (tid < 32) {
        float tk = 0.f, hd = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) tk += red[16 + i];
#pragma unroll
        for (int i = 0; i < 8; ++i) hd += red[i];
        const float dGn = tk + expf(Gn) * hd;
        float a0 = dG[2 * lane] + dGx[2 * lane];
        float a1 = dG[2 * lane + 1] + dGx[2 * lane + 1] + (lane == 31 ? dGn : 0.f);
        float s = a0 + a1;   // inclusive suffix sum from the right
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_down_sync(0xffffffffu, s, off);
            if (lane + off < 32) s += o;
        }
        const float suf1 = s - a0;
        const float suf0 = s;
        const float g0 = suf0 - (p.decay_first ? 0.f : dGx[2 * lane]);
        const float g1 = suf1 - (p.decay_first ? 0.f : dGx[2 * lane + 1]);
        const long long r0i = (row0 + 2 * lane) * H + h;
        p.dg[r0i] = g0;
        p.dg[r0i + H] = g1;
        p.dbeta[r0i] = dbs[2 * lane];
        p.dbeta[r0i + H] = dbs[2 * lane + 1];
    }
}

template <int KD, bool DOB>
cudaError_t launch_k(const ChunkGradParams& p, cudaStream_t s) {
    using L = MgSmem<KD>;
    auto kern = chunk_grad_mma_kernel<KD, DOB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::bytes);
    if (e != cudaSuccess) return e;
    const long long nblk = (long long)p.B * p.H * (p.T / kChunk);
    if (nblk == 0) return cudaSuccess;
    kern<<<(unsigned)nblk, kMgThreads, L::bytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_grad_mma(const ChunkGradParams& p, cudaStream_t s) {
    if (!p.in_bf16) return cudaErrorInvalidValue;   // the v tiles are copied as bf16
    if (p.K == 64) return p.do_bf16 ? launch_k<64, true>(p, s) : launch_k<64, false>(p, s);
    return p.do_bf16 ? launch_k<128, true>(p, s) : launch_k<128, false>(p, s);
}

}  // namespace gdn
