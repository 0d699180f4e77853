// gdn_wy.cu -- the per-chunk WY factors for the tcgen05 chain kernels (bf16, K == V == 128).
//
// For every 64-token chunk of every (b, h) this kernel forms, independently of all other
// chunks (it needs only the chunk's keys and gates),
//   L  = diag(beta) P,  P[i,j] = 2^(Gx_i - G_j) k_i.k_j  (j < i),  A = (I + L)^-1
//   A_beta = A diag(beta)          (so that U = A_beta V)
//   A_gam  = A diag(beta 2^Gx)     (so that W = A_gam K)
// ("Context Parallelism in ART", section 08, the per-chunk WY representation; gates in log2
// units, G the inclusive and Gx the exclusive cumulative sum of g within the chunk). The two
// factors are written as bf16 64 x 64 tiles in exactly the byte image the chain kernels use
// as tcgen05 operands: K-major rows of 128 bytes with the 128-byte swizzle. A chain then loads
// a chunk's pair with one bulk copy instead of inverting on its critical path, and the
// inverse is computed once per chunk rather than once per chain that walks the chunk.
//
// One CTA of four warps per chunk: K K^T on mma.sync (bf16, fp32 accumulate), L from the
// accumulators, the four 16 x 16 diagonal blocks of the inverse by forward substitution
// (one block per warp; rows in registers, shuffles), three rounds of block forward
// substitution on mma.sync (tf32), then the scaled bf16 tiles leave through one bulk store.
// The k tile, L and the output tiles share one 16 KB buffer (each is dead before the next
// is written), so six CTAs fit on an SM and hide each other's latencies; the kernel has no
// waits.
#include "gdn_tc_common.cuh"

namespace gdn {
namespace {

constexpr int kWyThreads = 128;
constexpr int kWyD = 128;          // K
constexpr float kWyLog2e = 1.4426950408889634f;

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t WY_K = 0;        // K tile bf16: [khalf 2][64 rows x 128 B], 128-byte swizzle;
constexpr uint32_t WY_L = 0;        // then L fp32 64 x 64 (sw64) once K K^T is in registers;
constexpr uint32_t WY_OUT = 0;      // then the two bf16 output tiles once the rounds are done
constexpr uint32_t WY_A = 16384;    // A fp32 64 x 64 (sw64)
constexpr uint32_t WY_Y = 32768;    // per-warp 16 x 8 fp32 scratch of the block rounds
constexpr uint32_t WY_SC = 34816;   // Gx, G, beta, beta 2^Gx: [4][64] fp32
constexpr uint32_t WY_END = 35840;
constexpr uint32_t kWySmem = WY_END + 1024;

struct WyParams {
    const void* k;
    const void* g;
    const void* beta;
    uint8_t* wy;        // [B*H][T/64][2][8192 B]
    int T, H;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D = A B + D, m16n8k16, bf16 in, fp32 accumulate
__device__ __forceinline__ void mma_m16n8k16_bf16(float* d, const uint32_t* a, const uint32_t* b) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__global__ void __launch_bounds__(kWyThreads, 6) wy_kernel(const WyParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    float* Lm = reinterpret_cast<float*>(sm + WY_L);
    float* Am = reinterpret_cast<float*>(sm + WY_A);
    float* sc = reinterpret_cast<float*>(sm + WY_SC);
    const float* Gx = sc;
    const float* G = sc + 64;
    const float* bet = sc + 128;
    const float* bekr = sc + 192;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nchunks = p.T / 64;
    const long long ch = blockIdx.x;                  // (b*H + h) * nchunks + n
    const int n = (int)(ch % nchunks);
    const long long bh = ch / nchunks;
    const int b = (int)(bh / p.H), h = (int)(bh % p.H);
    const long long row0 = (long long)b * p.T + (long long)n * 64;   // flattened (b, t)

    // ---- K tile: 64 rows of 256 bytes, half a row per 16 lanes (coalesced), stored in two
    //      64-feature halves with the 128-byte swizzle
    {
        const uint4* kg = reinterpret_cast<const uint4*>(p.k);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int e = tid + kWyThreads * r, row = e >> 4, c16 = e & 15;
            const uint4 x = __ldg(kg + ((row0 + row) * p.H + h) * (kWyD / 8) + c16);
            *reinterpret_cast<uint4*>(sm + WY_K + (c16 >> 3) * 8192 + sw128(row, c16 & 7)) = x;
        }
    }
    // ---- gates: cumulative sums in log2 units (first warp, two tokens per lane)
    if (warp == 0) {
        const long long i0 = (row0 + 2 * lane) * p.H + h;
        const float g0 = bf16_at(p.g, i0) * kWyLog2e, g1 = bf16_at(p.g, i0 + p.H) * kWyLog2e;
        const float b0 = bf16_at(p.beta, i0), b1 = bf16_at(p.beta, i0 + p.H);
        float sum = g0 + g1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, sum, off);
            if (lane >= off) sum += o;
        }
        const float excl = sum - (g0 + g1);
        sc[2 * lane] = excl;               // Gx
        sc[2 * lane + 1] = excl + g0;
        sc[64 + 2 * lane] = excl + g0;     // G
        sc[64 + 2 * lane + 1] = excl + g0 + g1;
        sc[128 + 2 * lane] = b0;           // beta
        sc[128 + 2 * lane + 1] = b1;
        sc[192 + 2 * lane] = b0 * ex2(excl);        // beta 2^Gx
        sc[192 + 2 * lane + 1] = b1 * ex2(excl + g0);
    }
    __syncthreads();

    // ---- K K^T for rows 16w..16w+15 (warp w), column tiles of 8 up to the diagonal block,
    //      then L = diag(beta) (2^(Gx_i - G_j) k_i.k_j) below the diagonal, straight from the
    //      accumulators
    {
        float d[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
        const int lrow = lane & 7, lsel = lane >> 3;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t kt = base + WY_K + (ks >> 2) * 8192;
            const int c0 = (ks & 3) * 2;
            uint32_t a[4];
            // matrices: rows 0-7 / 8-15 of the block at k 0-7, then the same rows at k 8-15
            ldsm_x4(kt + sw128(16 * warp + lrow + 8 * (lsel & 1), c0 + (lsel >> 1)), a);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                if (np > warp) continue;   // both column tiles lie above the diagonal block
                uint32_t bb[4];
                // column tile 2np: key rows 16np..+7 at k 0-7 and 8-15; tile 2np+1: rows +8
                ldsm_x4(kt + sw128(16 * np + lrow + 8 * (lsel >> 1), c0 + (lsel & 1)), bb);
                mma_m16n8k16_bf16(d[2 * np], a, bb);
                mma_m16n8k16_bf16(d[2 * np + 1], a, bb + 2);
            }
        }
        __syncthreads();   // every warp's reads of the k tile are done: L goes over it
        const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            if ((nt >> 1) > warp) continue;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = 16 * warp + gq + 8 * (e >> 1), j = 8 * nt + 2 * tq + (e & 1);
                Lm[sw64(i, j)] = (j < i) ? bet[i] * ex2(Gx[i] - G[j]) * d[nt][e] : 0.f;
            }
        }
    }
    __syncthreads();

    // ---- diagonal 16 x 16 blocks of (I + L)^-1, block w by warp w: lane (r, half) owns
    //      columns 8 half .. 8 half + 7 of row r, X[r] = e_r - sum_{m<r} L[r][m] X[m], with
    //      row m broadcast by shuffles once it is final. Rows are zero beyond their diagonal,
    //      so the updates run over all columns with constant bounds. The blocks above the
    //      diagonal are never written: the rounds never read them and the packing masks them.
    {
        const int bs = 16 * warp, r = lane & 15, half = lane >> 4, src0 = lane & 16;
        float x[8];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) x[cc] = (8 * half + cc == r) ? 1.f : 0.f;
#pragma unroll 1
        for (int m = 0; m < 15; ++m) {
            const float f = (r > m) ? Lm[sw64(bs + r, bs + m)] : 0.f;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const float xm = __shfl_sync(0xffffffffu, x[cc], src0 + m);
                x[cc] = fmaf(-f, xm, x[cc]);
            }
        }
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) Am[sw64(bs + r, bs + 8 * half + cc)] = x[cc];
    }
    __syncthreads();

    // ---- block forward substitution: X_IJ = -X_II sum_{m=J}^{I-1} L_Im X_mJ
    float* Ys = reinterpret_cast<float*>(sm + WY_Y) + warp * 128;
#pragma unroll 1
    for (int I = 1; I < 4; ++I) {
#pragma unroll 1
        for (int tile = warp; tile < 2 * I; tile += 4) {
            const int J = tile >> 1, n0 = 16 * J + 8 * (tile & 1);
            float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
            for (int m = J; m < I; ++m)
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    uint32_t a[4], bb[2];
                    frag_a(Lm, 16 * I, 16 * m + 8 * kk, lane, a);
                    frag_b(Am, 16 * m + 8 * kk, n0, lane, bb);
                    mma_m16n8k8(y, a, bb);
                }
            const int gq = lane >> 2, tq = lane & 3;
            Ys[gq * 8 + 2 * tq] = y[0];
            Ys[gq * 8 + 2 * tq + 1] = y[1];
            Ys[(gq + 8) * 8 + 2 * tq] = y[2];
            Ys[(gq + 8) * 8 + 2 * tq + 1] = y[3];
            __syncwarp();
            float xo[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                uint32_t a[4], bb[2];
                frag_a(Am, 16 * I, 16 * I + 8 * kk, lane, a);
                bb[0] = tf32_bits(Ys[(8 * kk + tq) * 8 + gq]);
                bb[1] = tf32_bits(Ys[(8 * kk + tq + 4) * 8 + gq]);
                mma_m16n8k8(xo, a, bb);
            }
            __syncwarp();
            Am[sw64(16 * I + gq, n0 + 2 * tq)] = -xo[0];
            Am[sw64(16 * I + gq, n0 + 2 * tq + 1)] = -xo[1];
            Am[sw64(16 * I + gq + 8, n0 + 2 * tq)] = -xo[2];
            Am[sw64(16 * I + gq + 8, n0 + 2 * tq + 1)] = -xo[3];
        }
        __syncthreads();
    }

    // ---- A diag(beta) (threads 0..63) and A diag(beta 2^Gx) (64..127) as bf16 K-major rows,
    //      over L's space (the last round's barrier retired every read of L), zero above the
    //      row's diagonal block, then one bulk store of both tiles
    {
        const int i = tid & 63;
        const int jend = (i & ~15) + 16;   // columns of the blocks up to the diagonal one
        const float* scale = (tid < 64) ? bet : bekr;
        uint8_t* tile = sm + WY_OUT + ((tid < 64) ? 0 : 8192);
#pragma unroll 1
        for (int cq = 0; cq < 8; ++cq) {
            float a[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                a[jj] = (8 * cq + jj < jend) ? Am[sw64(i, 8 * cq + jj)] * scale[8 * cq + jj] : 0.f;
            *reinterpret_cast<uint4*>(tile + sw128(i, cq)) =
                make_uint4(pack_bf16(a[0], a[1]), pack_bf16(a[2], a[3]), pack_bf16(a[4], a[5]),
                           pack_bf16(a[6], a[7]));
        }
    }
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {
        uint8_t* dst = p.wy + ch * 16384;
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                     "r"(base + WY_OUT), "r"(16384u)
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        // the shared source must stay valid until the copy has read it
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    }
}

}  // namespace

cudaError_t launch_tc_wy(const ChainParams& c, cudaStream_t s) {
    if (!c.wy) return cudaErrorInvalidValue;
    const long long nblk = (long long)c.B * c.H * (c.T / kChunk);
    if (nblk == 0) return cudaSuccess;
    if (nblk >= (1LL << 31)) return cudaErrorInvalidValue;
    WyParams p{c.k, c.g, c.beta, reinterpret_cast<uint8_t*>(c.wy), c.T, c.H};
    cudaError_t e = cudaFuncSetAttribute(wy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kWySmem);
    if (e != cudaSuccess) return e;
    wy_kernel<<<(unsigned)nblk, kWyThreads, kWySmem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
