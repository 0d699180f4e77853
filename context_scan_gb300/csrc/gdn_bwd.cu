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
// and writes D at the segment's start. Exponents are differences of cumulative gates, never
// exp(-G). Two instances: fp32 on the CUDA cores (fp32 inputs), and with the products -- L, C,
// dR, A^T dR and the update of D -- as warp-level tensor-core tiles (tf32 operands, fp32
// accumulation; bf16 inputs), whose fragments are read from shared memory at row pitches that
// keep them free of bank conflicts.
#include <cuda_bf16.h>

#include "gdn_internal.h"
#include "gdn_warp_mma.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float ld(const void* base, long long idx, int bf16) {
    if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
    return reinterpret_cast<const float*>(base)[idx];
}

// A prefetched element as loaded: fp32 bits, or the 16 bits of a bf16 in the high half -- the
// conversion waits until the value is stored, so that the loads of the next chunk stay in
// flight while the current one computes.
__device__ __forceinline__ uint32_t ld_bits(const void* base, long long idx, int bf16) {
    if (bf16) return (uint32_t)reinterpret_cast<const unsigned short*>(base)[idx];
    return __float_as_uint(reinterpret_cast<const float*>(base)[idx]);
}
__device__ __forceinline__ float from_bits(uint32_t x, int bf16) {
    return __uint_as_float(bf16 ? x << 16 : x);
}

template <int KD, int CT, bool MMA>
struct BwdSmem {
    static constexpr int TP = 68;       // padded rows of the transposed k / q ([l][i]) and of
                                        // the 64 x 64 matrices (float4-aligned)
    // row pitch of the CT-column tiles: the tensor-core instance reads them as MMA fragments,
    // which a pitch of 8 mod 32 words keeps free of bank conflicts
    static constexpr int DP = MMA ? CT + 8 : CT;
    static constexpr int KRQ = MMA ? 0 : 64 * KD;       // the row copies only the FFMA loops use
    static constexpr int off_kr = 0;                    // k  [64][KD]  (row i = token)
    static constexpr int off_qr = off_kr + KRQ;         // q  [64][KD]
    static constexpr int off_kt = off_qr + KRQ;         // k^T [KD][TP]
    static constexpr int off_qt = off_kt + KD * TP;     // q^T [KD][TP]
    static constexpr int off_do = off_qt + KD * TP;     // dO tile [64][DP]
    static constexpr int off_d = off_do + 64 * DP;      // D tile  [KD][DP]
    static constexpr int off_l = off_d + KD * DP;       // L = diag(beta) P  [64][TP]
    static constexpr int off_a = off_l + 64 * TP;       // A                 [64][TP]
    static constexpr int off_c = off_a + 64 * TP;       // C                 [64][TP]
    static constexpr int off_z = off_c + 64 * TP;       // Z tile [64][DP]
    static constexpr int off_r = off_z + 64 * DP;       // dR tile [64][DP]
    static constexpr int off_s = off_r + 64 * DP;       // scalars: 6 x 64
    static constexpr int total = off_s + 6 * 64;
    static constexpr size_t bytes = sizeof(float) * total;
    static_assert(bytes <= 232448, "shared memory budget");
};

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

// Every large product below gives each thread a 4 x 4 (or 4 x 2) block of the result in
// registers and reads its operands as float4 / float2 rows of shared memory, so the loop
// does 8-16 FMAs per shared-memory load (a thread per output reads two operands per FMA).
template <int KD, int CT, bool MMA>
__global__ void __launch_bounds__(kThreads) state_grad_kernel(StateGradParams p) {
    static_assert(kThreads == 256 && (CT == 32 || (MMA && CT == 64)),
                  "thread blocking assumes 256 threads; CT = 32, or 64 for the tensor-core instance");
    using L = BwdSmem<KD, CT, MMA>;
    constexpr int DP = L::DP;
    extern __shared__ float4 smv[];
    float* sm = reinterpret_cast<float*>(smv);
    float* kr = sm + L::off_kr;
    float* qr = sm + L::off_qr;
    float* kt = sm + L::off_kt;
    float* qt = sm + L::off_qt;
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
    constexpr int TP = L::TP;

    // one-dimensional grid, the column tile varying fastest: a chain's tiles are launched side
    // by side and L2 serves the k, q, g, beta reads that they repeat
    const int tid = threadIdx.x;
    const int ntiles = p.V / CT;
    const int chain = blockIdx.x / ntiles;
    const int seg = chain % p.nseg;
    const int bh = chain / p.nseg;
    const int b = bh / p.H, h = bh % p.H;
    const int c0 = (blockIdx.x % ntiles) * CT;
    const int V = p.V, H = p.H;
    const long long head = (long long)seg * p.B * H + bh;   // [seg][b][h] index

    for (int e = tid; e < KD * CT; e += kThreads) {
        const int l = e / CT, c = e % CT;
        Ds[l * DP + c] = p.dH_end ? p.dH_end[(head * KD + l) * V + c0 + c] : 0.f;
    }

    // The next chunk's k, q, dO, g and beta are loaded into registers while the current
    // chunk computes. Each thread owns NKQ (token quad, key channel) items of k and q -- the
    // four tokens of a quad land in one float4 of the transposed copies, so those stores are
    // free of bank conflicts -- and ND elements of the dO tile.
    constexpr int NKQ = 16 * KD / kThreads, ND = 64 * CT / kThreads;
    uint32_t pk[NKQ][4], pq[NKQ][4], pd[ND], pg = 0u, pb = 0u;
    uint4 pa[2];   // (with the WY tiles) this thread's 16-byte pieces of A diag(beta 2^Gx)
    const long long row0 = (long long)b * p.T + (long long)seg * p.seg_len;
    const bool use_wy = MMA && p.wy != nullptr;
    const uint8_t* wy_head = use_wy ? reinterpret_cast<const uint8_t*>(p.wy) +
                                          ((long long)bh * (p.T / kChunk) +
                                           (long long)seg * (p.seg_len / kChunk)) * kWyPairBytes +
                                          kWyTileBytes
                                    : nullptr;

    auto prefetch = [&](int ch) {
        const long long r0 = row0 + (long long)ch * kChunk;
#pragma unroll
        for (int n = 0; n < NKQ; ++n) {
            const int e = tid + n * kThreads, l = e % KD, i4 = (e / KD) * 4;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const long long idx = ((r0 + i4 + r) * H + h) * KD + l;
                pk[n][r] = ld_bits(p.k, idx, p.in_bf16);
                pq[n][r] = ld_bits(p.q, idx, p.in_bf16);
            }
        }
#pragma unroll
        for (int n = 0; n < ND; ++n) {
            const int e = tid + n * kThreads, i = e / CT, c = e % CT;
            pd[n] = ld_bits(p.dO, ((r0 + i) * H + h) * V + c0 + c, p.do_bf16);
        }
        if (tid < 64) {
            const long long row = (r0 + tid) * H + h;
            pg = ld_bits(p.g, row, p.in_bf16);
            pb = ld_bits(p.beta, row, p.in_bf16);
        }
        if (use_wy) {
            const uint4* t = reinterpret_cast<const uint4*>(wy_head + (long long)ch * kWyPairBytes);
            pa[0] = t[tid];
            if (tid + kThreads < kWyTileBytes / 16) pa[1] = t[tid + kThreads];
        }
    };
    const int n_chunks = p.seg_len / kChunk;
    if (use_wy)   // A's entries above its diagonal blocks, which the tiles do not carry
        for (int e = tid; e < 64 * 64; e += kThreads) {
            const int i = e >> 6, j = e & 63;
            if (j >= 16 * ((i >> 4) + 1)) As[i * TP + j] = 0.f;
        }
    if (n_chunks > 0) prefetch(n_chunks - 1);
    for (int ch = n_chunks - 1; ch >= 0; --ch) {
        // ---- (1) the prefetched chunk into shared memory: k, q (row and transposed copies),
        //      the dO tile, g, beta; then start loading the chunk before it
#pragma unroll
        for (int n = 0; n < NKQ; ++n) {
            const int e = tid + n * kThreads, l = e % KD, i4 = (e / KD) * 4;
            float kv4[4], qv4[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                kv4[r] = from_bits(pk[n][r], p.in_bf16);
                qv4[r] = from_bits(pq[n][r], p.in_bf16);
            }
            if constexpr (!MMA) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    kr[(i4 + r) * KD + l] = kv4[r];
                    qr[(i4 + r) * KD + l] = qv4[r];
                }
            }
            st4(&kt[l * TP + i4], make_float4(kv4[0], kv4[1], kv4[2], kv4[3]));
            st4(&qt[l * TP + i4], make_float4(qv4[0], qv4[1], qv4[2], qv4[3]));
        }
#pragma unroll
        for (int n = 0; n < ND; ++n) {
            const int e = tid + n * kThreads;
            dos[(e / CT) * DP + e % CT] = from_bits(pd[n], p.do_bf16);
        }
        if (tid < 64) {
            gx[tid] = from_bits(pg, p.in_bf16);   // raw gate until the cumsum
            bet[tid] = from_bits(pb, p.in_bf16);
        }
        if (use_wy) {
            // A diag(beta 2^Gx) from its bf16 tile (its 320 nonzero 16-byte pieces): piece e
            // lies in slab s, half hh, row group R, core row e % 8 -- row 8 R + e % 8, columns
            // 8 (2 s + hh) .. + 7; the entries above the diagonal blocks were zeroed before the
            // first chunk
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int e = tid + r * kThreads;
                if (e >= kWyTileBytes / 16) break;
                const int o = 16 * e;
                int sl = 0;
#pragma unroll
                for (int q = 1; q < 4; ++q) sl += o >= wy_slab0(q);
                const int o1 = o - wy_slab0(sl), hh = o1 >= wy_slab_lbo(sl) ? 1 : 0;
                const int o2 = o1 - hh * wy_slab_lbo(sl);
                const int row = 8 * (2 * sl + (o2 >> 7)) + (e & 7), cb = 8 * (2 * sl + hh);
                const uint32_t w4[4] = {pa[r].x, pa[r].y, pa[r].z, pa[r].w};
                float* dst = As + row * TP + cb;
                st4(dst, make_float4(__uint_as_float(w4[0] << 16), __uint_as_float(w4[0] & 0xFFFF0000u),
                                     __uint_as_float(w4[1] << 16), __uint_as_float(w4[1] & 0xFFFF0000u)));
                st4(dst + 4, make_float4(__uint_as_float(w4[2] << 16), __uint_as_float(w4[2] & 0xFFFF0000u),
                                         __uint_as_float(w4[3] << 16), __uint_as_float(w4[3] & 0xFFFF0000u)));
            }
        }
        __syncthreads();
        if (ch > 0) prefetch(ch - 1);
        // the gradient on the state leaving this chunk (D' before the chunk's own update)
        if (p.D_chunks) {
            const long long cg = (long long)seg * (p.seg_len / kChunk) + ch;   // chunk index
            float* dst = p.D_chunks + (cg * p.B * H + bh) * KD * V + c0;
            for (int e = tid; e < KD * CT; e += kThreads) {
                const int l = e / CT, c = e % CT;
                dst[(long long)l * V + c] = Ds[l * DP + c];
            }
        }
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
        if constexpr (MMA) {
            const int warp = tid >> 5, lane = tid & 31;
            const int m64 = 16 * (warp & 3), n64 = 32 * (warp >> 2);   // 16 x 32 per warp
            float sq[1][4][4] = {}, sk[1][4][4] = {};
            wtile<1, 4>(sq, m64, n64, KD, lane, [&](int i, int l) { return qt[l * TP + i]; },
                        [&](int l, int j) { return kt[l * TP + j]; });
            if (!use_wy) {
                wtile<1, 4>(sk, m64, n64, KD, lane, [&](int i, int l) { return kt[l * TP + i]; },
                            [&](int l, int j) { return kt[l * TP + j]; });
                wtile_each<1, 4>(sk, m64, n64, lane, [&](int i, int j, float& v) {
                    Ls[i * TP + j] = (j < i) ? bet[i] * __expf(gx[i] - gam[j]) * v : 0.f;
                    As[i * TP + j] = 0.f;
                });
            }
            wtile_each<1, 4>(sq, m64, n64, lane, [&](int i, int j, float& v) {
                Cs[i * TP + j] = (j <= i) ? __expf(gam[i] - gam[j]) * v : 0.f;
            });
        } else {
            const int i0 = (tid / 16) * 4, j0 = (tid % 16) * 4;
            float kk[4][4] = {}, qk[4][4] = {};
            if (j0 <= i0 + 3) {   // blocks wholly above the diagonal stay zero
#pragma unroll 4
                for (int l = 0; l < KD; ++l) {
                    const float4 a = ld4(&kt[l * TP + i0]), qa = ld4(&qt[l * TP + i0]);
                    const float4 bb = ld4(&kt[l * TP + j0]);
                    const float av[4] = {a.x, a.y, a.z, a.w}, qv[4] = {qa.x, qa.y, qa.z, qa.w};
                    const float bv[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            kk[r][c] = fmaf(av[r], bv[c], kk[r][c]);
                            qk[r][c] = fmaf(qv[r], bv[c], qk[r][c]);
                        }
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = i0 + r;
                float lv[4], cv[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int j = j0 + c;
                    lv[c] = (j < i) ? bet[i] * expf(gx[i] - gam[j]) * kk[r][c] : 0.f;
                    cv[c] = (j <= i) ? expf(gam[i] - gam[j]) * qk[r][c] : 0.f;
                }
                st4(&Ls[i * TP + j0], make_float4(lv[0], lv[1], lv[2], lv[3]));
                st4(&Cs[i * TP + j0], make_float4(cv[0], cv[1], cv[2], cv[3]));
                st4(&As[i * TP + j0], make_float4(0.f, 0.f, 0.f, 0.f));
            }
        }
        __syncthreads();
        // ---- (4a) inverses of the four 16 x 16 diagonal blocks of I + L (forward substitution)
        //      (with the WY tiles, A diag(beta exp(Gx)) came with the chunk: steps 4a, 4b skipped)
        if (!use_wy && tid < 64) {
            const int base = (tid / 16) * 16, c = tid % 16;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int r = 1; r < 16; ++r) {
                float a = 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) a = fmaf(Ls[(base + r) * TP + base + m], x[m], a);
                if (r > c) x[r] = -a;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) As[(base + r) * TP + base + c] = x[r];
        }
        __syncthreads();
        // ---- (4b) off-diagonal blocks: A_IJ = -inv(T_II) sum_{m=J}^{I-1} L_Im A_mJ
        if (!use_wy) {
            float* Yb = Zs;   // 3 blocks of 16 x 16 scratch (Zs is free until step 6)
            const int r = tid / 16, c = tid % 16;
            for (int I = 1; I < 4; ++I) {
                for (int J = 0; J < I; ++J) {
                    float a = 0.f;
                    for (int m = J; m < I; ++m) {
#pragma unroll
                        for (int l = 0; l < 16; ++l)
                            a = fmaf(Ls[(16 * I + r) * TP + 16 * m + l],
                                     As[(16 * m + l) * TP + 16 * J + c], a);
                    }
                    Yb[J * 256 + r * 16 + c] = a;
                }
                __syncthreads();
                for (int J = 0; J < I; ++J) {
                    float a = 0.f;
#pragma unroll
                    for (int l = 0; l < 16; ++l)
                        a = fmaf(As[(16 * I + r) * TP + 16 * I + l], Yb[J * 256 + l * 16 + c], a);
                    As[(16 * I + r) * TP + 16 * J + c] = -a;
                }
                __syncthreads();
            }
        }
        if constexpr (MMA) {
            // 8 warps: four row groups by two column halves of the CT-column tile
            constexpr int NT = CT / 16;
            const int warp = tid >> 5, lane = tid & 31;
            const int mr = 16 * (warp & 3), nr = (CT / 2) * (warp >> 2);   // 64 x CT: 16 x CT/2 per warp
            // ---- (5) dR = Kd D' + C^T dO
            {
                float d[1][NT][4] = {};
                wtile<1, NT>(d, mr, nr, KD, lane, [&](int i, int l) { return dk[i] * kt[l * TP + i]; },
                             [&](int l, int c) { return Ds[l * DP + c]; });
                wtile<1, NT>(d, mr, nr, 64, lane, [&](int i, int j) { return Cs[j * TP + i]; },
                             [&](int j, int c) { return dos[j * DP + c]; });
                wtile_each<1, NT>(d, mr, nr, lane, [&](int i, int c, float& v) { Rs[i * DP + c] = v; });
            }
            __syncthreads();
            // ---- (6) Z = diag(beta exp(Gx)) A^T dR
            {
                float z[1][NT][4] = {};
                wtile<1, NT>(z, mr, nr, 64, lane, [&](int j, int i) { return As[i * TP + j]; },
                             [&](int i, int c) { return Rs[i * DP + c]; });
                // (the WY tile is A diag(beta exp(Gx)) already)
                wtile_each<1, NT>(z, mr, nr, lane,
                                  [&](int j, int c, float& v) { Zs[j * DP + c] = (use_wy ? 1.f : ekr[j]) * v; });
            }
            __syncthreads();
            // ---- (7) D = exp(G_last) D' + Qd^T dO - K^T Z: K x CT, (16 K / 64) x CT/2 per warp
            {
                constexpr int MT = KD / 64;
                const int ml = 16 * MT * (warp & 3), nl = (CT / 2) * (warp >> 2);
                float a[MT][NT][4] = {};
                wtile<MT, NT>(a, ml, nl, 64, lane, [&](int l, int i) { return eq[i] * qt[l * TP + i]; },
                              [&](int i, int c) { return dos[i * DP + c]; });
                wtile<MT, NT>(a, ml, nl, 64, lane, [&](int l, int i) { return -kt[l * TP + i]; },
                              [&](int i, int c) { return Zs[i * DP + c]; });
                const float dlast = expf(glast);
                wtile_each<MT, NT>(a, ml, nl, lane, [&](int l, int c, float& v) {
                    float* dp = &Ds[l * DP + c];
                    *dp = fmaf(dlast, *dp, v);
                });
            }
        } else {
            // ---- (5) dR = Kd D' + C^T dO, one 4 x 2 block (rows j0.., columns cc..) per thread
            const int j0 = (tid / 16) * 4, cc = (tid % 16) * 2;
            {
                float a[4][2] = {}, t[4][2] = {};
#pragma unroll 4
                for (int l = 0; l < KD; ++l) {
                    const float4 kv = ld4(&kt[l * TP + j0]);
                    const float2 dv = *reinterpret_cast<const float2*>(&Ds[l * CT + cc]);
                    const float k4[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        a[r][0] = fmaf(k4[r], dv.x, a[r][0]);
                        a[r][1] = fmaf(k4[r], dv.y, a[r][1]);
                    }
                }
                for (int i = j0; i < 64; ++i) {   // C[i][j] = 0 for j > i
                    const float4 cv = ld4(&Cs[i * TP + j0]);
                    const float2 ov = *reinterpret_cast<const float2*>(&dos[i * CT + cc]);
                    const float c4[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        t[r][0] = fmaf(c4[r], ov.x, t[r][0]);
                        t[r][1] = fmaf(c4[r], ov.y, t[r][1]);
                    }
                }
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    *reinterpret_cast<float2*>(&Rs[(j0 + r) * CT + cc]) =
                        make_float2(fmaf(dk[j0 + r], a[r][0], t[r][0]), fmaf(dk[j0 + r], a[r][1], t[r][1]));
            }
            __syncthreads();
            // ---- (6) Z = diag(beta exp(Gx)) A^T dR (same blocking)
            {
                float a[4][2] = {};
                for (int i = j0; i < 64; ++i) {   // A[i][j] = 0 for j > i
                    const float4 av = ld4(&As[i * TP + j0]);
                    const float2 rv = *reinterpret_cast<const float2*>(&Rs[i * CT + cc]);
                    const float a4[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        a[r][0] = fmaf(a4[r], rv.x, a[r][0]);
                        a[r][1] = fmaf(a4[r], rv.y, a[r][1]);
                    }
                }
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    *reinterpret_cast<float2*>(&Zs[(j0 + r) * CT + cc]) =
                        make_float2(ekr[j0 + r] * a[r][0], ekr[j0 + r] * a[r][1]);
            }
            __syncthreads();
            // ---- (7) D = exp(G_last) D' + Qd^T dO - K^T Z, one 4 x CW block (rows l0..) per thread
            {
                constexpr int CW = KD * CT / (kThreads * 4);   // 4 columns at K = 128, 2 at K = 64
                const int l0 = (tid / (CT / CW)) * 4, d0 = (tid % (CT / CW)) * CW;
                float a[4][CW] = {};
#pragma unroll 4
                for (int i = 0; i < 64; ++i) {
                    const float e = eq[i];
                    const float4 qv = ld4(&qr[i * KD + l0]), kv = ld4(&kr[i * KD + l0]);
                    float o4[CW], z4[CW];
                    if constexpr (CW == 4) {
                        const float4 ov = ld4(&dos[i * CT + d0]), zv = ld4(&Zs[i * CT + d0]);
                        o4[0] = ov.x, o4[1] = ov.y, o4[2] = ov.z, o4[3] = ov.w;
                        z4[0] = zv.x, z4[1] = zv.y, z4[2] = zv.z, z4[3] = zv.w;
                    } else {
#pragma unroll
                        for (int c = 0; c < CW; ++c) {
                            o4[c] = dos[i * CT + d0 + c];
                            z4[c] = Zs[i * CT + d0 + c];
                        }
                    }
                    const float q4[4] = {e * qv.x, e * qv.y, e * qv.z, e * qv.w};
                    const float k4[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int c = 0; c < CW; ++c)
                            a[r][c] = fmaf(q4[r], o4[c], fmaf(-k4[r], z4[c], a[r][c]));
                }
                const float dlast = expf(glast);
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < CW; ++c) {
                        float* dp = &Ds[(l0 + r) * CT + d0 + c];
                        *dp = fmaf(dlast, *dp, a[r][c]);
                    }
            }
        }
        __syncthreads();
    }

    for (int e = tid; e < KD * CT; e += kThreads) {
        const int l = e / CT, c = e % CT;
        p.dS[(head * KD + l) * V + c0 + c] = Ds[l * DP + c];
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

template <int KD, int CT, bool MMA>
cudaError_t launch_state_grad_kv(const StateGradParams& p, cudaStream_t s) {
    using L = BwdSmem<KD, CT, MMA>;
    auto kern = state_grad_kernel<KD, CT, MMA>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::bytes);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.B * p.H * p.nseg * (p.V / CT)));
    kern<<<grid, kThreads, L::bytes, s>>>(p);
    return cudaGetLastError();
}

template <int KD>
cudaError_t launch_state_grad_k(const StateGradParams& p, cudaStream_t s) {
    // bf16 inputs: the tensor-core products (tf32 operands keep the bf16 bar) on 64-column
    // tiles; fp32 inputs keep fp32 products on the CUDA cores, 32-column tiles
    if (p.in_bf16) return launch_state_grad_kv<KD, state_grad_tile(1), true>(p, s);
    return launch_state_grad_kv<KD, state_grad_tile(0), false>(p, s);
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
