// gdn_kda_mma.cu -- the chunked forward and the segment summary with per-channel gates
// ("KDA Chunk Backward -- TPU/Pallas Kernel Design", section 1.2: g is [B,T,H,K] and every
// key channel decays by its own gate) for bf16 inputs, with the products on the warp-level
// tensor cores.
//
// The chunk step is the one of the CUDA-core chains (gdn_simt.cu, GATEK), per channel l:
//   G_il the inclusive cumulative gate in the chunk, Gr_il the read-side one (G_(i-1)l, or G_il
//   when the read sees the decayed state)
//   L[i,j] = beta_i sum_l k_il k_jl e^(Gr_il - G_jl) (j < i),  A = (I + L)^-1
//   C[i,j] = sum_l q_il k_jl e^(G_il - G_jl) (j <= i)
//   R = A diag(beta) (V - (K . e^Gr) H),  O = (Q . e^G) H + C R
//   H <- diag(e^G_last) H + (K . e^(G_last - G))^T R
// L and C by sub-block normalisation (the page's section 3.7): the 64 tokens are four blocks of
// 16; block row I of L and C is the product of the row block's scaled keys (queries)
// k_il e^(Gr_il - ref_l) against the chunk's keys scaled k_jl e^(ref_l - G_jl), with ref the
// cumulative gate just before block I (zero for the first). Both factors are at most 1 for every
// entry left of the diagonal block (G only decreases), so those are plain products of bounded
// operands; inside the diagonal block the second factor grows with the block's own gate spread,
// and a block whose spread exceeds kSpreadMax (any channel) is formed entry by entry with the
// exponential of each difference instead. Every other factor is a difference with j <= i or
// G_last - G_j, so never above 1. All products are sums of m16n8k8 tf32 MMAs (fp32
// accumulation) whose fragments are read from fp32 shared memory -- the scaled operands are
// formed as the fragments are read; the inverse stays on the CUDA cores.
//
// L, C and A depend only on the chunk's keys, queries and gates, so kda_prep_kernel forms them
// once per chunk, fully parallel (one CTA per chunk), and writes A diag(beta) and C (fp32) to
// the workspace. The chains -- one CTA per (b, h, segment) and tile of CT state columns, as the
// CUDA-core chains -- load them with the chunk's other inputs, scale the chunk's keys and
// queries once (K . e^Gr for the read, K . e^(G_last - G) for the update, Q . e^G for the
// output), and run the four products that carry the state:
//   R = A diag(beta) (V - (K . e^Gr) H),  O = (Q . e^G) H + C R,
//   H <- diag(e^G_last) H + (K . e^(G_last - G))^T R.
#include <cuda_bf16.h>

#include "gdn_internal.h"
#include "gdn_warp_mma.cuh"

namespace gdn {
namespace {

constexpr int kKdaThreads = 256;
constexpr int kKdaCT = 64;
// largest exponent a diagonal block's scaled keys may carry (e^80 ~ 5.5e34, far inside fp32)
constexpr float kSpreadMax = 80.f;

__device__ __forceinline__ float kin(const void* base, long long idx, int bf16) {
    if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
    return reinterpret_cast<const float*>(base)[idx];
}
__device__ __forceinline__ void kout(void* base, long long idx, float x, int bf16) {
    if (bf16)
        reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(x);
    else
        reinterpret_cast<float*>(base)[idx] = x;
}
// eight bf16 to fp32 in shared memory (two 16-byte stores)
__device__ __forceinline__ void put8(float* dst, uint4 u) {
    *reinterpret_cast<float4*>(dst) =
        make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                    __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
    *reinterpret_cast<float4*>(dst + 4) =
        make_float4(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xFFFF0000u),
                    __uint_as_float(u.w << 16), __uint_as_float(u.w & 0xFFFF0000u));
}

// ---- the per-chunk factors: A diag(beta) and C -------------------------------------------
template <int KD>
struct PrepSmem {
    static constexpr int KPB = KD + 8;  // row pitch (bf16 elements) of k and q: 4 mod 32 words
    static constexpr int KP = KD + 4;   // row pitch of G (4 mod 32 words)
    static constexpr int LP = 68;       // row pitch of the 64 x 64 matrices
    // k and q as bf16 (as loaded); once L and C are formed, A [64][LP] and the inverse's
    // scratch (3 x 256) take their place
    static constexpr int KQ = 64 * KPB;   // floats of the k and q rows together
    static constexpr int KQSZ = KQ > 64 * LP + 3 * 256 ? KQ : 64 * LP + 3 * 256;
    static constexpr int kq = 0;
    static constexpr int gk = kq + KQSZ;               // cumulative gates G [64][KP]
    static constexpr int l = gk + 64 * KP;             // L [64][LP]
    static constexpr int c = l + 64 * LP;              // C [64][LP]
    static constexpr int bet = c + 64 * LP;            // beta [64]
    static constexpr int ref = bet + 64;               // block references [4][KD]
    static constexpr int total = ref + 4 * KD;
    static constexpr size_t bytes = sizeof(float) * total;
    // two CTAs per SM
    static_assert(2 * (bytes + 1024) <= 233472, "shared memory budget: two CTAs per SM");
};

// One CTA per chunk: the chunk's per-channel cumulative gates, L and C by sub-block
// normalisation (a diagonal block whose gate spread is too wide to factor entry by entry),
// A = (I + L)^-1 by 16 x 16 diagonal inverses and block substitution, then A diag(beta) and C
// to out[chunk] ([2][64][64] fp32). Chunks are numbered (b*H + h)*(T/64) + n for the batch, or
// h*total_chunks + cu_chunks[b] + n for packed sequences (tokens past a sequence's end load as
// zeros with g = beta = 0).
template <int KD>
__global__ void __launch_bounds__(kKdaThreads, 2) kda_prep_kernel(ChainParams p, float* out) {
    using L = PrepSmem<KD>;
    constexpr int KP = L::KP, LP = L::LP, KPB = L::KPB;
    extern __shared__ float4 smv[];
    float* sm = reinterpret_cast<float*>(smv);
    unsigned short* kb16 = reinterpret_cast<unsigned short*>(sm + L::kq);
    unsigned short* qb16 = kb16 + 64 * KPB;
    auto kf = [&](int i, int l) { return __uint_as_float((uint32_t)kb16[i * KPB + l] << 16); };
    auto qf = [&](int i, int l) { return __uint_as_float((uint32_t)qb16[i * KPB + l] << 16); };
    float* Gk = sm + L::gk;
    float* Ls = sm + L::l;
    float* Cs = sm + L::c;
    float* As = sm + L::kq;          // (once L and C are formed)
    float* Yb = As + 64 * LP;        // the inverse's scratch
    float* bet = sm + L::bet;
    float* ref = sm + L::ref;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long ch = blockIdx.x;
    int h, valid = 64;
    long long row0;
    if (!p.cu_seqlens) {
        const int nchunks = p.T / kChunk;
        const long long bh = ch / nchunks;
        h = (int)(bh % p.H);
        row0 = (bh / p.H) * p.T + (ch % nchunks) * kChunk;
    } else {
        h = (int)(ch / p.total_chunks);
        const int cc = (int)(ch % p.total_chunks);
        if (cc >= p.cu_chunks[p.B]) return;   // past the last chunk (the grid holds a bound)
        int lo = 0, hi = p.B;   // the sequence s with cu_chunks[s] <= cc < cu_chunks[s+1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.cu_chunks[mid] <= cc) lo = mid; else hi = mid;
        }
        const int t0 = p.cu_seqlens[lo] + kChunk * (cc - p.cu_chunks[lo]);
        row0 = t0;
        valid = min(kChunk, p.cu_seqlens[lo + 1] - t0);
    }
    const int H = p.H;
    // ---- (1) k, q, g (8 bf16 per 16-byte load) and beta
    {
        const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(p.k);
        const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(p.q);
        const __nv_bfloat16* gb = reinterpret_cast<const __nv_bfloat16*>(p.g);
        constexpr int NKV = 64 * KD / 8 / kKdaThreads;
        uint4 uk[NKV], uq[NKV], ug[NKV];
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int n = 0; n < NKV; ++n) {
            const int e = tid + n * kKdaThreads, i = e / (KD / 8), l8 = 8 * (e % (KD / 8));
            const bool in = i < valid;
            const long long o = ((row0 + i) * H + h) * KD + l8;
            uk[n] = in ? *reinterpret_cast<const uint4*>(kb + o) : zero;
            uq[n] = in && p.q ? *reinterpret_cast<const uint4*>(qb + o) : zero;
            ug[n] = in ? *reinterpret_cast<const uint4*>(gb + o) : zero;
        }
        const float bt = (tid < 64 && tid < valid) ? kin(p.beta, (row0 + tid) * H + h, 1) : 0.f;
#pragma unroll
        for (int n = 0; n < NKV; ++n) {
            const int e = tid + n * kKdaThreads, i = e / (KD / 8), l8 = 8 * (e % (KD / 8));
            *reinterpret_cast<uint4*>(kb16 + i * KPB + l8) = uk[n];
            *reinterpret_cast<uint4*>(qb16 + i * KPB + l8) = uq[n];
            put8(Gk + i * KP + l8, ug[n]);
        }
        if (tid < 64) bet[tid] = bt;
    }
    __syncthreads();
    // ---- (2) per-channel inclusive cumsum down the chunk, the block references, and whether
    //      a diagonal block's spread is too wide to factor
    bool wide[4] = {false, false, false, false};
    if (tid < KD) {
        float acc = 0.f;
        for (int i = 0; i < 64; ++i) {
            acc += Gk[i * KP + tid];
            Gk[i * KP + tid] = acc;
        }
#pragma unroll
        for (int I = 0; I < 4; ++I) {
            const float rI = I == 0 ? 0.f : Gk[(16 * I - 1) * KP + tid];
            ref[I * KD + tid] = rI;
            wide[I] = rI - Gk[(16 * I + 15) * KP + tid] > kSpreadMax;
        }
    }
    bool exact[4];
#pragma unroll
    for (int I = 0; I < 4; ++I) exact[I] = __syncthreads_or(wide[I]) != 0;   // also a barrier
    auto gread = [&](int i, int l) {
        return p.decay_first ? Gk[i * KP + l] : (i > 0 ? Gk[(i - 1) * KP + l] : 0.f);
    };
    // ---- (3) L and C by blocks of 16 rows: warp w forms block row w >> 1 of L (w even) or of
    //      C (w odd) against all 64 columns, then masks it
    {
        const int I = warp >> 1, prod = warp & 1;
        const float* rf = ref + I * KD;
        float acc[1][8][4] = {};
        auto fb = [&](int l, int j) {   // the chunk's keys against reference I
            return kf(j, l) * __expf(fminf(rf[l] - Gk[j * KP + l], kSpreadMax));
        };
        if (prod == 0)
            wtile<1, 8>(acc, 16 * I, 0, KD, lane,
                        [&](int i, int l) { return kf(i, l) * __expf(gread(i, l) - rf[l]); }, fb);
        else
            wtile<1, 8>(acc, 16 * I, 0, KD, lane,
                        [&](int i, int l) { return qf(i, l) * __expf(Gk[i * KP + l] - rf[l]); }, fb);
        if (prod == 0) {
            wtile_each<1, 8>(acc, 16 * I, 0, lane, [&](int i, int j, float& v) {
                Ls[i * LP + j] = (j < i) ? bet[i] * v : 0.f;
            });
        } else {
            wtile_each<1, 8>(acc, 16 * I, 0, lane, [&](int i, int j, float& v) {
                Cs[i * LP + j] = (j <= i) ? v : 0.f;
            });
        }
    }
    __syncthreads();
    // a diagonal block whose gates spread too far: its entries one by one, each decay the
    // exponential of one difference with j <= i
    if (exact[0] || exact[1] || exact[2] || exact[3]) {
#pragma unroll 1
        for (int I = 0; I < 4; ++I) {
            if (!exact[I]) continue;
            for (int e = tid; e < 256; e += kKdaThreads) {
                const int i = 16 * I + e / 16, j = 16 * I + e % 16;
                float lv = 0.f, cv = 0.f;
                if (j < i) {
                    for (int l = 0; l < KD; ++l)
                        lv = fmaf(kf(i, l) * kf(j, l), __expf(gread(i, l) - Gk[j * KP + l]), lv);
                    lv *= bet[i];
                }
                if (j <= i)
                    for (int l = 0; l < KD; ++l)
                        cv = fmaf(qf(i, l) * kf(j, l), __expf(Gk[i * KP + l] - Gk[j * KP + l]), cv);
                Ls[i * LP + j] = lv;
                Cs[i * LP + j] = cv;
            }
        }
        __syncthreads();
    }
    // ---- (4a) inverses of the four 16x16 diagonal blocks of I + L (A takes q's place; the
    //      rest of A starts at zero)
    for (int e = tid; e < 64 * 64; e += kKdaThreads) As[(e >> 6) * LP + (e & 63)] = 0.f;
    __syncthreads();
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
        const int r = tid / 16, c = tid % 16;
        for (int I = 1; I < 4; ++I) {
            for (int J = 0; J < I; ++J) {
                float a = 0.f;
                for (int m = J; m < I; ++m) {
#pragma unroll
                    for (int l = 0; l < 16; ++l)
                        a = fmaf(Ls[(16 * I + r) * LP + 16 * m + l], As[(16 * m + l) * LP + 16 * J + c], a);
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
    // ---- (5) A diag(beta) and C out, four consecutive floats per store
    float* dst = out + ch * (2 * 64 * 64);
    for (int e = tid; e < 64 * 16; e += kKdaThreads) {
        const int i = e >> 4, j4 = 4 * (e & 15);
        const float* a = As + i * LP + j4;
        *reinterpret_cast<float4*>(dst + i * 64 + j4) =
            make_float4(a[0] * bet[j4], a[1] * bet[j4 + 1], a[2] * bet[j4 + 2], a[3] * bet[j4 + 3]);
        *reinterpret_cast<float4*>(dst + 4096 + i * 64 + j4) = *reinterpret_cast<const float4*>(Cs + i * LP + j4);
    }
}

template <int KD, int CT, bool SUMMARY>
struct KdaSmem {
    static constexpr int KP = KD + 4;   // row pitch of k, q, G (4 mod 32 words)
    static constexpr int LP = 68;       // row pitch of the 64 x 64 matrices
    static constexpr int VP = CT + 8;   // row pitch of the 64 x CT tiles and of the state tile
    static constexpr int k = 0;                                // k [64][KP]
    static constexpr int q = k + 64 * KP;                      // q [64][KP] (forward)
    static constexpr int gk = q + (SUMMARY ? 0 : 64 * KP);     // cumulative gates G [64][KP]
    static constexpr int v = gk + 64 * KP;                     // V tile, then Y [64][VP]
    static constexpr int hs = v + 64 * VP;                     // state tile [KD][VP]
    static constexpr int a = hs + KD * VP;                     // A diag(beta) [64][LP]
    static constexpr int c = a + 64 * LP;                      // C [64][LP] (forward)
    static constexpr int r = c + (SUMMARY ? 0 : 64 * LP);      // R [64][VP]
    static constexpr int eg = r + 64 * VP;                     // e^(G_last) [KD]
    static constexpr int total = eg + KD;
    static constexpr size_t bytes = sizeof(float) * total;
    static_assert(bytes <= 232448, "shared memory budget");
};

template <int KD, int CT, bool SUMMARY>
__global__ void __launch_bounds__(kKdaThreads, 1) kda_chain_mma_kernel(ChainParams p) {
    // a forward grid lets a grid launched as its programmatic dependent start right away
    if (!SUMMARY) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    using L = KdaSmem<KD, CT, SUMMARY>;
    constexpr int KP = L::KP, LP = L::LP, VP = L::VP;
    constexpr int NT = CT / 16;   // 8-column fragments of a warp's half of a CT-column tile
    extern __shared__ float4 smv[];
    float* sm = reinterpret_cast<float*>(smv);
    float* ks = sm + L::k;
    float* qs = sm + L::q;
    float* Gk = sm + L::gk;
    float* vs = sm + L::v;
    float* Hs = sm + L::hs;
    float* As = sm + L::a;
    float* Cs = sm + L::c;
    float* Rs = sm + L::r;
    float* eg = sm + L::eg;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chain = blockIdx.x;
    const int seg = p.seg_first + chain % p.nseg_run;
    const int bh = chain / p.nseg_run;
    const int b = bh / p.H, h = bh % p.H;
    const int c0 = blockIdx.y * CT;   // first state column of this tile
    const int V = p.V, H = p.H, T = p.T;
    // warp tiles: 64 x CT outputs 16 x CT/2 per warp, KD x CT outputs (16 KD/64) x CT/2
    const int mr = 16 * (warp & 3), nr = (CT / 2) * (warp >> 2);
    constexpr int MTH = KD / 64;
    const int mh = 16 * MTH * (warp & 3);

    // ---- initial state tile
    for (int e = tid; e < KD * CT; e += kKdaThreads) {
        const int l = e / CT, c = e % CT;
        float x = 0.f;
        if (SUMMARY) {
            x = (c0 + c == l) ? 1.f : 0.f;   // [I | 0]
        } else if (p.h_start) {
            x = p.h_start[(long long)seg * p.h_start_seg_stride + ((long long)bh * KD + l) * V + c0 + c];
        }
        Hs[l * VP + c] = x;
    }

    // tokens of this chain: a segment of the fixed-length batch, or a whole varlen sequence
    // whose last chunk may be partial (its padding tokens load as zeros with g = beta = 0,
    // which leaves the state untouched, and their outputs are not stored)
    const long long row_base = p.cu_seqlens ? (long long)p.cu_seqlens[b]
                                            : (long long)b * T + (long long)seg * p.seg_len;
    const int seq_tokens = p.cu_seqlens ? p.cu_seqlens[b + 1] - p.cu_seqlens[b] : p.seg_len;
    const int n_chunks = (seq_tokens + kChunk - 1) / kChunk;
    // this chain's chunks' A diag(beta) and C, as kda_prep_kernel numbers them
    const float* prep = reinterpret_cast<const float*>(p.wy) +
                        (p.cu_seqlens ? (long long)h * p.total_chunks + p.cu_chunks[b]
                                      : (long long)bh * (T / kChunk) + (long long)seg * (p.seg_len / kChunk)) *
                            (2 * 64 * 64);
    // the read-side gate of token i, channel l
    auto gread = [&](int i, int l) {
        return p.decay_first ? Gk[i * KP + l] : (i > 0 ? Gk[(i - 1) * KP + l] : 0.f);
    };
    // The next chunk's k, q, g (8 bf16 of a row per 16-byte load), V tile and beta are loaded
    // into registers while the current chunk computes.
    constexpr int NKV = 64 * KD / 8 / kKdaThreads, NVV = 64 * CT / 8 / kKdaThreads;
    static_assert(NKV * 8 * kKdaThreads == 64 * KD && NVV * 8 * kKdaThreads == 64 * CT, "load split");
    const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(p.k);
    const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(p.q);
    const __nv_bfloat16* gb = reinterpret_cast<const __nv_bfloat16*>(p.g);
    const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(p.v);
    uint4 pk[NKV], pq[NKV], pg[NKV], pv[NVV];
    float4 pa[4], pc[4];   // A diag(beta) and C: four 16-byte pieces each
    auto prefetch = [&](int chn) {
        const int tn = chn * kChunk;
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
        const float4* pf = reinterpret_cast<const float4*>(prep + (long long)chn * (2 * 64 * 64));
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            pa[n] = pf[tid + n * kKdaThreads];
            if (!SUMMARY) pc[n] = pf[1024 + tid + n * kKdaThreads];
        }
#pragma unroll
        for (int n = 0; n < NKV; ++n) {
            const int e = tid + n * kKdaThreads, i = e / (KD / 8), l8 = 8 * (e % (KD / 8));
            const bool in = tn + i < seq_tokens;
            const long long o = ((row_base + tn + i) * H + h) * KD + l8;
            pk[n] = in ? *reinterpret_cast<const uint4*>(kb + o) : zero;
            if (!SUMMARY) pq[n] = in ? *reinterpret_cast<const uint4*>(qb + o) : zero;
            pg[n] = in ? *reinterpret_cast<const uint4*>(gb + o) : zero;
        }
#pragma unroll
        for (int n = 0; n < NVV; ++n) {
            const int e = tid + n * kKdaThreads, i = e / (CT / 8), c8 = 8 * (e % (CT / 8));
            const int gc = c0 + c8;
            const bool in = tn + i < seq_tokens && (!SUMMARY || gc >= KD);
            const long long o = ((row_base + tn + i) * H + h) * V + (SUMMARY ? gc - KD : gc);
            pv[n] = in ? *reinterpret_cast<const uint4*>(vb + o) : zero;
        }
    };
    if (n_chunks > 0) prefetch(0);
#pragma unroll 1
    for (int ch = 0; ch < n_chunks; ++ch) {
        const int t0 = ch * kChunk;
        // ---- (1) the chunk into shared memory: k, q, the per-channel gates, the V tile, beta;
        //      then start loading the next one
#pragma unroll
        for (int n = 0; n < NKV; ++n) {
            const int e = tid + n * kKdaThreads, i = e / (KD / 8), l8 = 8 * (e % (KD / 8));
            put8(ks + i * KP + l8, pk[n]);
            if (!SUMMARY) put8(qs + i * KP + l8, pq[n]);
            put8(Gk + i * KP + l8, pg[n]);
        }
#pragma unroll
        for (int n = 0; n < NVV; ++n) {
            const int e = tid + n * kKdaThreads, i = e / (CT / 8), c8 = 8 * (e % (CT / 8));
            put8(vs + i * VP + c8, pv[n]);
        }
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const int e = tid + n * kKdaThreads, i = e >> 4, j4 = 4 * (e & 15);
            *reinterpret_cast<float4*>(As + i * LP + j4) = pa[n];
            if (!SUMMARY) *reinterpret_cast<float4*>(Cs + i * LP + j4) = pc[n];
        }
        __syncthreads();
        if (ch + 1 < n_chunks) prefetch(ch + 1);
        // ---- (2) per-channel inclusive cumsum down the chunk (one thread per channel)
        if (tid < KD) {
            float acc = 0.f;
            for (int i = 0; i < 64; ++i) {
                acc += Gk[i * KP + tid];
                Gk[i * KP + tid] = acc;
            }
            eg[tid] = __expf(acc);
        }
        __syncthreads();
        // ---- (3) the chunk's scaled operands, once: K . e^Gr (for the read) over G, K .
        //      e^(G_last - G) (for the update) over k, Q . e^G (for the output) over q; every
        //      exponent is a difference with the earlier token first, or G itself, so at most 0
        {
            constexpr int NE = 64 * KD / kKdaThreads;
            float kr[NE], kl[NE], qg[NE];
#pragma unroll
            for (int n = 0; n < NE; ++n) {
                const int e = tid + n * kKdaThreads, i = e / KD, l = e % KD;
                const float kv = ks[i * KP + l], G = Gk[i * KP + l];
                kr[n] = kv * __expf(gread(i, l));
                kl[n] = kv * __expf(Gk[63 * KP + l] - G);
                qg[n] = SUMMARY ? 0.f : qs[i * KP + l] * __expf(G);
            }
            __syncthreads();
#pragma unroll
            for (int n = 0; n < NE; ++n) {
                const int e = tid + n * kKdaThreads, i = e / KD, l = e % KD;
                Gk[i * KP + l] = kr[n];
                ks[i * KP + l] = kl[n];
                if (!SUMMARY) qs[i * KP + l] = qg[n];
            }
        }
        __syncthreads();
        // ---- (5) Y = V - (K . e^Gr) H, over the V tile
        {
            float acc[1][NT][4] = {};
            wtile<1, NT>(acc, mr, nr, KD, lane, [&](int i, int l) { return Gk[i * KP + l]; },
                         [&](int l, int c) { return Hs[l * VP + c]; });
            wtile_each<1, NT>(acc, mr, nr, lane, [&](int i, int c, float& v) {
                vs[i * VP + c] = vs[i * VP + c] - v;
            });
        }
        __syncthreads();
        // ---- (6) R = A diag(beta) Y
        {
            float acc[1][NT][4] = {};
            wtile<1, NT>(acc, mr, nr, 64, lane, [&](int i, int j) { return As[i * LP + j]; },
                         [&](int j, int c) { return vs[j * VP + c]; });
            wtile_each<1, NT>(acc, mr, nr, lane, [&](int i, int c, float& v) { Rs[i * VP + c] = v; });
        }
        __syncthreads();
        // ---- (7) O = (Q . e^G) H + C R
        if (!SUMMARY) {
            float acc[1][NT][4] = {};
            wtile<1, NT>(acc, mr, nr, KD, lane, [&](int i, int l) { return qs[i * KP + l]; },
                         [&](int l, int c) { return Hs[l * VP + c]; });
            wtile<1, NT>(acc, mr, nr, 64, lane, [&](int i, int j) { return Cs[i * LP + j]; },
                         [&](int j, int c) { return Rs[j * VP + c]; });
            wtile_each<1, NT>(acc, mr, nr, lane, [&](int i, int c, float& v) {
                if (t0 + i < seq_tokens) {
                    const long long row = (row_base + t0 + i) * H + h;
                    kout(p.o, row * V + c0 + c, v, p.out_bf16);
                }
            });
            __syncthreads();   // every read of H is done before the update below
        }
        // ---- (8) H <- diag(e^G_last) H + (K . e^(G_last - G))^T R
        {
            float acc[MTH][NT][4] = {};
            wtile<MTH, NT>(acc, mh, nr, 64, lane, [&](int l, int j) { return ks[j * KP + l]; },
                           [&](int j, int c) { return Rs[j * VP + c]; });
            wtile_each<MTH, NT>(acc, mh, nr, lane, [&](int l, int c, float& v) {
                Hs[l * VP + c] = fmaf(eg[l], Hs[l * VP + c], v);
            });
        }
        __syncthreads();
    }

    // ---- write the chain's final state
    if (SUMMARY) {
        const long long base = (long long)seg * p.B * H + bh;
        for (int e = tid; e < KD * CT; e += kKdaThreads) {
            const int l = e / CT, c = e % CT;
            const int gc = c0 + c;
            if (gc < KD)
                p.M[(base * KD + l) * KD + gc] = Hs[l * VP + c];
            else
                p.S[(base * KD + l) * V + (gc - KD)] = Hs[l * VP + c];
        }
    } else {
        if (p.h_final && seg == p.nseg_total - 1)
            for (int e = tid; e < KD * CT; e += kKdaThreads) {
                const int l = e / CT, c = e % CT;
                p.h_final[((long long)bh * KD + l) * V + c0 + c] = Hs[l * VP + c];
            }
        if (p.h_out)   // the state entering the next segment
            for (int e = tid; e < KD * CT; e += kKdaThreads) {
                const int l = e / CT, c = e % CT;
                p.h_out[(seg + 1) * p.h_out_seg_stride + ((long long)bh * KD + l) * V + c0 + c] = Hs[l * VP + c];
            }
    }
    // a summary grid launched as a programmatic dependent completes after its primary grid
    if (SUMMARY) asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int KD, bool SUMMARY>
cudaError_t launch_kda(const ChainParams& p, cudaStream_t s) {
    constexpr int CT = kKdaCT;
    using L = KdaSmem<KD, CT, SUMMARY>;
    auto kern = kda_chain_mma_kernel<KD, CT, SUMMARY>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::bytes);
    if (e != cudaSuccess) return e;
    const int ncols = SUMMARY ? KD + p.V : p.V;
    dim3 grid((unsigned)(p.B * p.H * p.nseg_run), (unsigned)(ncols / CT));
    if (!p.launch_dependent) {
        kern<<<grid, kKdaThreads, L::bytes, s>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kKdaThreads);
    cfg.dynamicSmemBytes = L::bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int KD>
cudaError_t launch_prep(const ChainParams& p, cudaStream_t s) {
    using L = PrepSmem<KD>;
    auto kern = kda_prep_kernel<KD>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::bytes);
    if (e != cudaSuccess) return e;
    const long long nblk = p.cu_seqlens ? (long long)p.H * p.total_chunks
                                        : (long long)p.B * p.H * (p.T / kChunk);
    if (nblk == 0) return cudaSuccess;
    if (nblk >= (1LL << 31)) return cudaErrorInvalidValue;
    kern<<<(unsigned)nblk, kKdaThreads, L::bytes, s>>>(p, reinterpret_cast<float*>(p.wy));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kda_prep(const ChainParams& p, cudaStream_t s) {
    if (!p.gate_k || !p.in_bf16 || !p.wy) return cudaErrorInvalidValue;
    return p.K == 64 ? launch_prep<64>(p, s) : launch_prep<128>(p, s);
}

cudaError_t launch_kda_mma_chain(const ChainParams& p, bool summary, cudaStream_t s) {
    if (!p.gate_k || !p.in_bf16 || !p.wy) return cudaErrorInvalidValue;
    if (p.K == 64) return summary ? launch_kda<64, true>(p, s) : launch_kda<64, false>(p, s);
    return summary ? launch_kda<128, true>(p, s) : launch_kda<128, false>(p, s);
}

}  // namespace gdn
