// gdn_wy.cu -- the per-chunk WY factors for the tcgen05 chain kernels (bf16, K == V == 128).
//
// For every 64-token chunk of every (b, h) this kernel forms, independently of all other
// chunks (it needs only the chunk's keys and gates),
//   L  = diag(beta) P,  P[i,j] = 2^(Gx_i - G_j) k_i.k_j  (j < i),  A = (I + L)^-1
//   A_beta = A diag(beta)          (so that U = A_beta V)
//   A_gam  = A diag(beta 2^Gx)     (so that W = A_gam K)
// ("Context Parallelism in ART", section 08, the per-chunk WY representation; gates in log2
// units, G the inclusive and Gx the exclusive cumulative sum of g within the chunk). The two
// factors are written as bf16 tcgen05 operands of 8 x 8 core matrices without their zero
// blocks above the diagonal (format at kWyTileBytes in gdn_internal.h): a chain loads a
// chunk's pair with one bulk copy instead of inverting on its critical path, and the inverse
// is computed once per chunk rather than once per chain that walks the chunk. A core is 128
// contiguous bytes, so every store of an mma.sync fragment (a lane's two columns of rows g
// and g + 8) covers whole 128-byte lines.
//
// One CTA of four warps per chunk: the k tile arrives by TMA in the chain kernels' swizzled
// layout; K K^T goes to tensor memory as two tcgen05 groups (bf16, fp32 accumulate) whose A
// operand starts at the tile for columns 0..31 (rows in lanes 0..63) and 64 rows before it for
// columns 32..63 (rows in lanes 64..127), so each warp reads out its own quarter and forms L;
// then the four 16 x 16 diagonal blocks of the inverse by forward substitution (warps 0 and 1,
// a column per lane, L's rows as shared-memory broadcasts), then the blocks below the diagonal
// by two levels of the block-triangular inverse on mma.sync (tf32): 16 -> 32 rows, then
// 32 -> 64. The blocks of L that feed the tensor cores and the inverse itself are kept as tf32
// bit patterns in row-padded layouts (68 and 72 words per row), so that fragments load with
// ldmatrix or plain shared loads at constant offsets; the diagonal blocks of L stay fp32 for
// the substitution. Each block of the inverse is scaled and written to global memory as bf16
// as soon as it is final. Six CTAs share an SM (64
// tensor-memory columns each) and hide each other's latencies; the two waits (the tile,
// K K^T) are bounded.
#include <algorithm>
#include <cstring>

#include "gdn_tc_common.cuh"

namespace gdn {
namespace {

constexpr int kWyThreads = 128;
constexpr float kWyLog2e = 1.4426950408889634f;

constexpr int LS = 68;   // row pitch (words) of L (tf32 below the diagonal blocks)
constexpr int XS = 72;   // row pitch (words) of the tf32 inverse X
// The diagonal 16 x 16 blocks of L (fp32) live in L's rows above the diagonal, at the same
// pitch: block b at rows ld_row(b).., columns ld_col(b).. (blocks 0, 1 in rows 16..31, columns
// 16..47; blocks 2, 3 in rows 32..47, columns 32..63), so that two blocks read or written
// together fall on different banks and X never overlaps them.
__host__ __device__ constexpr int ld_row(int b) { return b < 2 ? 16 : 32; }
__host__ __device__ constexpr int ld_col(int b) { return 16 + 16 * b - (b < 2 ? 0 : 16); }
static_assert(ld_col(0) == 16 && ld_col(1) == 32 && ld_col(2) == 32 && ld_col(3) == 48, "diagonal block map");

// shared-memory map (bytes from a 1024-aligned base). Rows 0..15 of L are never used (the
// first block row has nothing below the diagonal), so the scratch, the scalars and the
// barriers live there; 36 KB per CTA lets six CTAs share an SM. The allocation must also hold
// the K K^T operand windows: an M = 128 MMA reads 128 rows (16 KB) of its A operand per
// feature half, so the first group reads up to 8 KB past the tile's end and the second group
// from 8 KB before its start -- bytes 0 .. 32 KB + 96 in all, whatever else lives there.
constexpr uint32_t WY_K = 8192;     // K tile bf16: [khalf 2][64 rows x 128 B], 128-byte swizzle
constexpr uint32_t WY_LT = 0;       // then L (tf32, 64 x LS, rows 16..63) once K K^T is in TMEM
constexpr uint32_t WY_X = 17408;    // X = (I + L)^-1 (tf32, 64 x XS)
constexpr uint32_t WY_Y = 0;        // per-warp 16 x 8 fp32 scratch of the block rounds
constexpr uint32_t WY_SC = 2048;    // Gx, G, beta, beta 2^Gx: [4][64] fp32
constexpr uint32_t WY_BAR = 3072;   // mbarriers (tile, K K^T), tensor-memory address
constexpr uint32_t WY_CF = 3200;    // column factors 2^(r_J - G_j) of L (fp32 [64])
constexpr uint32_t WY_END = 35840;
constexpr uint32_t kWySmem = WY_END + 1024;   // + alignment slack
constexpr uint32_t kWyTmemCols = 64;
constexpr uint32_t ID_KK = idesc_bf16(128, 32, false, false);   // K K^T, 32 columns per group
static_assert(64 * LS * 4 <= WY_X - WY_LT && 64 * XS * 4 <= WY_END - WY_X, "layout");
static_assert(WY_BAR + 64 <= WY_CF && WY_CF + 256 <= 16 * LS * 4,
              "scratch, scalars and barriers fit in L's unused rows");
static_assert(WY_K + 3 * 8192 + 128 <= WY_END, "the K K^T operand windows stay inside the allocation");

struct WyParams {
    CUtensorMap tm_k;
    const void* g;
    const void* beta;
    uint8_t* wy;        // [B*H][T/64] tile pairs of kWyPairBytes
    int T, H;
    int decay_first;   // read-side gate G (decayed read) instead of Gx
    const int* cu_seqlens;   // varlen: packed sequences (null for the fixed-length batch)
    const int* cu_chunks;
    int nseq, total_chunks;   // varlen: total_chunks bounds the chunks (T/64 + nseq)
    int wy_lo, wy_cnt;        // fixed length: chunks wy_lo .. wy_lo + wy_cnt - 1 of each (b, h)
    unsigned* queue;          // wy_queue_kernel: the next chunk to hand out
    unsigned* queue_reset;    // wy_kernel: a counter to zero for a later wy_queue_kernel launch
    unsigned items;           // chunks the launch covers
    DeviceError* err;
    long long wait_limit;   // SM clock cycles before a wait gives up
};

// 16-byte output piece of row `row`, columns 8 c .. 8 c + 7 of one factor's tile
__device__ __forceinline__ uint4* out_chunk(uint8_t* tile, int row, int c) {
    return reinterpret_cast<uint4*>(tile + wy_piece(row, c));
}

// wait tags recorded in the device error word's detail field
enum : unsigned { WTAG_TILE = 101, WTAG_KK = 102 };

// Per-CTA state of the WY kernels: shared-memory base, barriers and tensor memory.
struct WyCta {
    uint8_t* sm;
    uint32_t base, bar_tile, bar_kk, tmem;
    volatile int* abort_flag;
};

// Barriers and the 64 tensor-memory columns of a WY CTA (every thread calls this once).
__device__ __forceinline__ WyCta wy_setup() {
    extern __shared__ uint8_t smem_raw[];
    WyCta w;
    const uint32_t raw = smem_u32(smem_raw);
    w.base = (raw + 1023u) & ~1023u;
    w.sm = smem_raw + (w.base - raw);
    w.bar_tile = w.base + WY_BAR;
    w.bar_kk = w.base + WY_BAR + 8;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(w.sm + WY_BAR + 16);
    w.abort_flag = reinterpret_cast<volatile int*>(w.sm + WY_BAR + 20);
    if (threadIdx.x == 0) {
        mbar_init(w.bar_tile, 1);
        mbar_init(w.bar_kk, 1);
        *w.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (threadIdx.x < 32) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         w.base + WY_BAR + 16),
                     "r"(kWyTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    w.tmem = *tmem_slot;
    return w;
}

__device__ __forceinline__ void wy_teardown(const WyCta& w) {
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(w.tmem),
                     "r"(kWyTmemCols)
                     : "memory");
    }
}

// One chunk's pair of WY tiles. `ch` numbers the chunks the launch covers; `it` counts the
// chunks this CTA has formed before (the barriers' phase). Every thread of the CTA calls it;
// it ends with every thread past its last read of shared memory.
__device__ __forceinline__ void wy_chunk(const WyParams& p, const WyCta& w, unsigned ch, uint32_t it) {
    uint8_t* sm = w.sm;
    const uint32_t base = w.base, bar_tile = w.bar_tile, bar_kk = w.bar_kk, tmem = w.tmem;
    volatile int* abort_flag = w.abort_flag;
    const uint32_t par = it & 1u;
    uint32_t* Lt = reinterpret_cast<uint32_t*>(sm + WY_LT);
    uint32_t* X = reinterpret_cast<uint32_t*>(sm + WY_X);
    float* Lf = reinterpret_cast<float*>(sm + WY_LT);   // L's words as fp32 (diagonal blocks)
    float* sc = reinterpret_cast<float*>(sm + WY_SC);
    const float* Gx = sc;
    const float* G = sc + 64;
    const float* bet = sc + 128;
    const float* bekr = sc + 192;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int h, valid = 64;                  // valid: tokens of the chunk inside its sequence
    long long row0;                     // flattened (b, t) of the chunk's first token
    long long tile;                     // index of the chunk's tile pair in p.wy
    // (32-bit index arithmetic: a launch covers fewer than 2^31 chunks, and every thread
    // computes these)
    if (!p.cu_seqlens) {
        // chunks wy_lo .. wy_lo + wy_cnt - 1 of every (b, h), the heads fastest: the CTAs of
        // one chunk's heads run together and read neighbouring rows of k, g and beta
        const unsigned nchunks = (unsigned)p.T / 64u;
        const unsigned bn = ch / (unsigned)p.H;
        h = (int)(ch - bn * (unsigned)p.H);
        const unsigned b = bn / (unsigned)p.wy_cnt;
        const int n = p.wy_lo + (int)(bn - b * (unsigned)p.wy_cnt);
        row0 = (long long)b * p.T + (long long)n * 64;
        tile = ((long long)b * p.H + h) * nchunks + n;
    } else {
        // (the heads fastest here too)
        const int c = (int)(ch / (unsigned)p.H);
        h = (int)(ch - (unsigned)c * (unsigned)p.H);
        if (c >= __ldg(p.cu_chunks + p.nseq)) return;   // past the last chunk (the grid holds a bound)
        int lo = 0, hi = p.nseq;   // the sequence s with cu_chunks[s] <= c < cu_chunks[s+1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(p.cu_chunks + mid) <= c) lo = mid; else hi = mid;
        }
        const int n = c - __ldg(p.cu_chunks + lo);
        const int t0 = __ldg(p.cu_seqlens + lo) + 64 * n;
        row0 = t0;
        valid = min(64, __ldg(p.cu_seqlens + lo + 1) - t0);
        tile = (long long)h * p.total_chunks + c;
    }
    uint8_t* out_b = p.wy + tile * kWyPairBytes;   // A diag(beta)
    uint8_t* out_g = out_b + kWyTileBytes;          // A diag(beta 2^Gx)

    // ---- the k tile (two 64-feature halves, 128-byte swizzle) by TMA
    if (tid == 0) {
        mbar_arrive_expect_tx(bar_tile, 16384u);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
            tma_load_3d(base + WY_K + hf * 8192, &p.tm_k, bar_tile, hf * 64, h, (int)row0);
    }
    // ---- gates: cumulative sums in log2 units (two tokens per lane); tokens past the end of a
    //      varlen sequence get g = 0 and beta = 0, which makes them no-ops on the state
    if (warp == 1) {
        const long long i0 = (row0 + 2 * lane) * p.H + h;
        const bool v0 = 2 * lane < valid, v1 = 2 * lane + 1 < valid;
        const float g0 = v0 ? bf16_at(p.g, i0) * kWyLog2e : 0.f;
        const float g1 = v1 ? bf16_at(p.g, i0 + p.H) * kWyLog2e : 0.f;
        const float b0 = v0 ? bf16_at(p.beta, i0) : 0.f, b1 = v1 ? bf16_at(p.beta, i0 + p.H) : 0.f;
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
        // beta 2^Gx (beta 2^G when the read sees the decayed state)
        sc[192 + 2 * lane] = b0 * ex2(p.decay_first ? excl + g0 : excl);
        sc[192 + 2 * lane + 1] = b1 * ex2(p.decay_first ? excl + g0 + g1 : excl + g0);
        // column factors of L below the diagonal blocks: 2^(r_J - G_j), r_J = G at the end of
        // j's 16-token block J (lane 8 J + 7 holds it as its second token); at most 1
        const float rJ = __shfl_sync(0xffffffffu, excl + g0 + g1, 8 * (lane >> 3) + 7);
        float* cf = reinterpret_cast<float*>(sm + WY_CF);
        cf[2 * lane] = ex2(rJ - (excl + g0));
        cf[2 * lane + 1] = ex2(rJ - (excl + g0 + g1));
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- K K^T (M = 128, N = 32 per group, bf16, fp32 accumulate): columns 0..31 with A
    //      starting at the tile (rows in lanes 0..63; lanes 64..127 unused), columns 32..63
    //      with A starting 64 rows before it (rows in lanes 64..127; lanes 0..63 unused), so
    //      each of the four warps reads its own quarter out of tensor memory
    bool issued = false;
    if (tid == 0 && mbar_wait(bar_tile, par, abort_flag, p.wait_limit, p.err, WTAG_TILE)) {
        tc_fence_after();
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16) {
            const uint32_t off = (k16 >> 2) * 8192 + (k16 & 3) * 32;
            mma_ss<ID_KK>(tmem, desc_k(base + WY_K + off), desc_k(base + WY_K + off), k16 > 0);
            mma_ss<ID_KK>(tmem + 32, desc_k(base + WY_K - 8192 + off),
                          desc_k(base + WY_K + 4096 + off), k16 > 0);
        }
        mma_commit(bar_kk);
        issued = true;
    }
    __syncwarp();

    // ---- L = diag(beta) (2^(Gx_i - G_j) k_i.k_j) below the diagonal: warp w has rows
    //      i = 32 (w & 1) + lane and columns 32 (w >> 1) .. + 31 (warp 2's quarter lies above
    //      the diagonal). fp32 for the diagonal 16 x 16 blocks, tf32 for the rest.
    {
        const int i = 32 * (warp & 1) + lane, jb = 32 * (warp >> 1);
        const bool ok = __shfl_sync(0xffffffffu,
                                    (int)mbar_wait(bar_kk, par, abort_flag, p.wait_limit, p.err, WTAG_KK), 0) != 0;
        if (ok && warp != 2) {
            tc_fence_after();
            float kk[32];
            const uint32_t t_row = tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)jb;
            tmem_ld16(t_row, kk);
            tmem_ld16(t_row + 16, kk + 16);
            tmem_wait_ld();
            const float bi = bet[i], gxi = p.decay_first ? G[i] : Gx[i];   // read-side gate
            const int I = i >> 4;
            const float* cf = reinterpret_cast<const float*>(sm + WY_CF);
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {   // the warp's two 16-column blocks J
                const int J = (jb >> 4) + hb;
                const float* kv = kk + 16 * hb;
                if (J < I) {
                    // below the diagonal blocks: 2^(gx_i - G_j) = 2^(gx_i - r_J) 2^(r_J - G_j),
                    // both factors at most 1 (the gates only decay), so no exponential per entry
                    const float rf = bi * ex2(gxi - G[16 * J + 15]);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 c4 = *reinterpret_cast<const float4*>(cf + 16 * J + 4 * q);
                        *reinterpret_cast<uint4*>(Lt + i * LS + 16 * J + 4 * q) =
                            make_uint4(tf32_operand(rf * c4.x * kv[4 * q]), tf32_operand(rf * c4.y * kv[4 * q + 1]),
                                       tf32_operand(rf * c4.z * kv[4 * q + 2]), tf32_operand(rf * c4.w * kv[4 * q + 3]));
                    }
                } else if (J == I) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int j = 16 * J + 4 * q;
                        float v[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            v[e] = (j + e < i) ? bi * ex2(gxi - G[j + e]) * kv[4 * q + e] : 0.f;
                        *reinterpret_cast<float4*>(Lf + (ld_row(I) + (i & 15)) * LS + ld_col(I) + 4 * q) =
                            make_float4(v[0], v[1], v[2], v[3]);
                    }
                }
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    // should a wait have given up, K K^T retires and the tile's copy lands before their memory
    // is reused
    if (tid == 0 && *abort_flag) {
        if (issued) mbar_drain(bar_kk, par, p.wait_limit);
        mbar_drain(bar_tile, par, p.wait_limit);
    }
    __syncthreads();

    // ---- diagonal 16 x 16 blocks of (I + L)^-1 by forward substitution down the columns:
    //      warps 0 and 1 take two blocks each, lane (block, c) computes column c of its block,
    //      X[i][c] = [i == c] - sum_{j<i} L[i][j] X[j][c] (the sum as two interleaved partial
    //      sums), the whole column in registers and L's rows read as broadcasts. The columns go
    //      back over the block's L.
    if (warp < 2) {
        const int blk = 2 * warp + (lane >> 4), c = lane & 15;
        float* lb = Lf + ld_row(blk) * LS + ld_col(blk);
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float a0 = (i == c) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
            for (int j4 = 0; j4 < i; j4 += 4) {
                const float4 l4 = *reinterpret_cast<const float4*>(lb + i * LS + j4);
                a0 = fmaf(-l4.x, x[j4], a0);
                if (j4 + 1 < i) a1 = fmaf(-l4.y, x[j4 + 1], a1);
                if (j4 + 2 < i) a0 = fmaf(-l4.z, x[j4 + 2], a0);
                if (j4 + 3 < i) a1 = fmaf(-l4.w, x[j4 + 3], a1);
            }
            x[i] = a0 + a1;
        }
        __syncwarp();   // every lane of the warp has read its blocks of L
#pragma unroll
        for (int i = 0; i < 16; ++i) lb[i * LS + c] = x[i];
    }
    __syncthreads();
    {
        // every warp: its diagonal block, row r, columns 8 half .. +7 -> X (tf32) and both
        // outputs (one 16-byte chunk per tile)
        const int bs = 16 * warp, r = lane & 15, half = lane >> 4;
        const float* lr = Lf + (ld_row(warp) + r) * LS + ld_col(warp) + 8 * half;
        const float4 xa = *reinterpret_cast<const float4*>(lr);
        const float4 xb = *reinterpret_cast<const float4*>(lr + 4);
        const float x[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
        const int row = bs + r, c0 = bs + 8 * half;
        uint4* xs = reinterpret_cast<uint4*>(X + row * XS + c0);
        xs[0] = make_uint4(tf32_operand(x[0]), tf32_operand(x[1]), tf32_operand(x[2]), tf32_operand(x[3]));
        xs[1] = make_uint4(tf32_operand(x[4]), tf32_operand(x[5]), tf32_operand(x[6]), tf32_operand(x[7]));
        *out_chunk(out_b, row, c0 >> 3) =
            make_uint4(pack_bf16(x[0] * bet[c0], x[1] * bet[c0 + 1]),
                       pack_bf16(x[2] * bet[c0 + 2], x[3] * bet[c0 + 3]),
                       pack_bf16(x[4] * bet[c0 + 4], x[5] * bet[c0 + 5]),
                       pack_bf16(x[6] * bet[c0 + 6], x[7] * bet[c0 + 7]));
        *out_chunk(out_g, row, c0 >> 3) =
            make_uint4(pack_bf16(x[0] * bekr[c0], x[1] * bekr[c0 + 1]),
                       pack_bf16(x[2] * bekr[c0 + 2], x[3] * bekr[c0 + 3]),
                       pack_bf16(x[4] * bekr[c0 + 4], x[5] * bekr[c0 + 5]),
                       pack_bf16(x[6] * bekr[c0 + 6], x[7] * bekr[c0 + 7]));
    }
    __syncthreads();

    // ---- the blocks below the diagonal, by two levels of the block-triangular inverse
    //      [[A, 0], [C, D]]^-1 = [[A^-1, 0], [-D^-1 C A^-1, D^-1]]:
    //      stage 1 (16 -> 32 rows): X_10 = -X_11 L_10 X_00 (warps 0, 1) and
    //        X_32 = -X_33 L_32 X_22 (warps 2, 3), an 8-wide half of the block each;
    //      stage 2 (32 -> 64 rows): the lower-left 32 x 32 block -X_[11] (L_[10] X_[00]) with
    //        X_[00] = [[X_00, 0], [X_10, X_11]] and X_[11] = [[X_22, 0], [X_32, X_33]], one
    //        8-wide column strip per warp (X_01 = 0 leaves warps 2, 3 half the sum).
    //      Fragments of L and of the row-major X blocks by ldmatrix (four 8 x 4-word tiles);
    //      the products Y go through a per-warp scratch to become B operands. Each finished
    //      16 x 8 tile is scaled and written to the outputs as bf16 pairs; stage 1's tiles also
    //      go back to X (tf32) for stage 2.
    const int gq = lane >> 2, tq = lane & 3;
    const uint32_t lt_u = smem_u32(Lt), x_u = smem_u32(X);
    // this lane's ldmatrix row address within a 16 x 8 tile at (r0, c0) of a row-major matrix
    const int lm_r = (lane & 7) + 8 * ((lane >> 3) & 1), lm_c = 4 * (lane >> 4);
    auto ldsm = [&](uint32_t (&a)[4], uint32_t m_u, int pitch, int r0, int c0) {
        const uint32_t addr = m_u + (uint32_t)(((r0 + lm_r) * pitch + c0 + lm_c) * 4);
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                     : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                     : "r"(addr)
                     : "memory");
    };
    // B fragment: X rows k0 + tq (+4), column n0 + gq
    auto ldx_b = [&](uint32_t (&bb)[2], int k0, int n0) {
        const uint32_t* xb = X + (k0 + tq) * XS + n0 + gq;
        bb[0] = xb[0];
        bb[1] = xb[4 * XS];
    };
    // a 16 x 8 accumulator tile through row-major scratch Ys: B fragment rows 8 kk + tq (+4)
    auto put_y = [&](float* Ys, const float (&y)[4]) {
        Ys[gq * 8 + 2 * tq] = y[0];
        Ys[gq * 8 + 2 * tq + 1] = y[1];
        Ys[(gq + 8) * 8 + 2 * tq] = y[2];
        Ys[(gq + 8) * 8 + 2 * tq + 1] = y[3];
    };
    auto get_y = [&](uint32_t (&bb)[2], const float* Ys, int kk) {
        bb[0] = tf32_operand(Ys[(8 * kk + tq) * 8 + gq]);
        bb[1] = tf32_operand(Ys[(8 * kk + tq + 4) * 8 + gq]);
    };
    // X = -z at rows r0, r0 + 8 (r0 = 16 I + gq), columns c0, c0 + 1 (c0 = n0 + 2 tq): both
    // outputs as bf16 pairs, byte 4 tq of the 16-byte piece (row, n0 / 8) -- across the warp
    // one whole core per store
    auto put_out = [&](const float (&z)[4], int r0, int n0) {
        const int c0 = n0 + 2 * tq;
        const float b0 = bet[c0], b1 = bet[c0 + 1], e0 = bekr[c0], e1 = bekr[c0 + 1];
        const int o0 = wy_piece(r0, n0 >> 3) + 4 * tq, o1 = wy_piece(r0 + 8, n0 >> 3) + 4 * tq;
        *reinterpret_cast<uint32_t*>(out_b + o0) = pack_bf16(-z[0] * b0, -z[1] * b1);
        *reinterpret_cast<uint32_t*>(out_b + o1) = pack_bf16(-z[2] * b0, -z[3] * b1);
        *reinterpret_cast<uint32_t*>(out_g + o0) = pack_bf16(-z[0] * e0, -z[1] * e1);
        *reinterpret_cast<uint32_t*>(out_g + o1) = pack_bf16(-z[2] * e0, -z[3] * e1);
    };
    {
        const int Ib = warp < 2 ? 1 : 3, Jb = Ib - 1;
        const int n0 = 16 * Jb + 8 * (warp & 1);
        float* Ys = reinterpret_cast<float*>(sm + WY_Y) + warp * 128;
        float y[4] = {0.f, 0.f, 0.f, 0.f}, z[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t a[4], bb[2];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {   // Y = L_{Ib,Jb} X_{Jb,Jb}
            ldsm(a, lt_u, LS, 16 * Ib, 16 * Jb + 8 * kk);
            ldx_b(bb, 16 * Jb + 8 * kk, n0);
            mma_m16n8k8(y, a, bb);
        }
        put_y(Ys, y);
        __syncwarp();
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {   // Z = X_{Ib,Ib} Y
            ldsm(a, x_u, XS, 16 * Ib, 16 * Ib + 8 * kk);
            get_y(bb, Ys, kk);
            mma_m16n8k8(z, a, bb);
        }
        const int r0 = 16 * Ib + gq, c0 = n0 + 2 * tq;
        *reinterpret_cast<uint2*>(X + r0 * XS + c0) = make_uint2(tf32_operand(-z[0]), tf32_operand(-z[1]));
        *reinterpret_cast<uint2*>(X + (r0 + 8) * XS + c0) = make_uint2(tf32_operand(-z[2]), tf32_operand(-z[3]));
        put_out(z, r0, n0);
    }
    __syncthreads();   // X_10 and X_32 are in X; L_10 (rows 16..31 of L) is dead
    {
        const int Jw = warp >> 1, n0 = 8 * warp;
        // scratch for Y_2, Y_3 in L's rows 16..31 (free after stage 1)
        float* Y2 = reinterpret_cast<float*>(sm + WY_LT + 16 * LS * 4) + warp * 256;
        float* Y3 = Y2 + 128;
        float y2[4] = {0.f, 0.f, 0.f, 0.f}, y3[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t a[4], bb[2];
#pragma unroll
        for (int k8 = 0; k8 < 4; ++k8) {   // Y_I = sum_m L_{I,m} X_{m,Jw}, I = 2, 3
            if (k8 >= 2 * Jw) {
                ldx_b(bb, 8 * k8, n0);
                ldsm(a, lt_u, LS, 32, 8 * k8);
                mma_m16n8k8(y2, a, bb);
                ldsm(a, lt_u, LS, 48, 8 * k8);
                mma_m16n8k8(y3, a, bb);
            }
        }
        put_y(Y2, y2);
        put_y(Y3, y3);
        __syncwarp();
        float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {   // Z_2 = X_22 Y_2
            get_y(bb, Y2, kk);
            ldsm(a, x_u, XS, 32, 32 + 8 * kk);
            mma_m16n8k8(z, a, bb);
        }
        put_out(z, 32 + gq, n0);
#pragma unroll
        for (int e = 0; e < 4; ++e) z[e] = 0.f;
#pragma unroll
        for (int k8 = 0; k8 < 4; ++k8) {   // Z_3 = X_32 Y_2 + X_33 Y_3
            get_y(bb, k8 < 2 ? Y2 : Y3, k8 & 1);
            ldsm(a, x_u, XS, 48, 32 + 8 * k8);
            mma_m16n8k8(z, a, bb);
        }
        put_out(z, 48 + gq, n0);
    }
    // every warp is done with the tile, L and X before the next chunk's copy lands on them
    fence_proxy_async();
    __syncthreads();
}

// One CTA per chunk.
__global__ void __launch_bounds__(kWyThreads, 6) wy_kernel(const __grid_constant__ WyParams p) {
    if (p.queue_reset && blockIdx.x == 0 && threadIdx.x == 0) *p.queue_reset = 0u;
    const WyCta w = wy_setup();
    wy_chunk(p, w, blockIdx.x, 0);
    wy_teardown(w);
}

// Chunks handed out one at a time from p.queue (zeroed before the launch) to a grid of any
// size: launched as the programmatic dependent of a chain grid, the CTAs that fit beside the
// chains start at once and take chunks until none is left, and the rest start as the chains
// finish. Every CTA then waits for the preceding grid, so that what follows in the stream sees
// both grids complete.
__global__ void __launch_bounds__(kWyThreads, 6) wy_queue_kernel(const __grid_constant__ WyParams p) {
    const WyCta w = wy_setup();
    volatile unsigned* slot = reinterpret_cast<volatile unsigned*>(w.sm + WY_BAR + 24);
#pragma unroll 1
    for (uint32_t it = 0;; ++it) {
        if (threadIdx.x == 0) *slot = atomicAdd(p.queue, 1u);
        __syncthreads();
        const unsigned item = *slot;
        const bool stop = item >= p.items || *w.abort_flag;
        __syncthreads();   // every thread has read the slot (and the flag) before either changes
        if (stop) break;
        wy_chunk(p, w, item, it);
    }
    wy_teardown(w);
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// varlen: chunk numbering of the packed sequences (a prefix sum over at most a few thousand
// lengths, one thread)
}  // namespace

cudaError_t launch_tc_wy(const ChainParams& c, cudaStream_t s) {
    if (!c.wy) return cudaErrorInvalidValue;
    const int nchunks = c.T / kChunk;
    const int lo = c.cu_seqlens ? 0 : c.wy_lo;
    const int cnt = c.cu_seqlens ? 0 : (c.wy_cnt > 0 ? c.wy_cnt : nchunks - lo);
    if (!c.cu_seqlens && (lo < 0 || cnt < 0 || lo + cnt > nchunks)) return cudaErrorInvalidValue;
    const long long nblk = c.cu_seqlens ? (long long)c.H * c.total_chunks : (long long)c.B * c.H * cnt;
    if (nblk == 0)
        return c.wy_queue_reset ? cudaMemsetAsync(c.wy_queue_reset, 0, sizeof(unsigned), s)
                                : cudaSuccess;
    if (nblk >= (1LL << 31) || (c.wy_queue && c.cu_seqlens)) return cudaErrorInvalidValue;
    WyParams p;
    memset(&p, 0, sizeof(p));
    if (!make_map(&p.tm_k, c.k, c)) return cudaErrorInvalidValue;
    p.g = c.g;
    p.beta = c.beta;
    p.wy = reinterpret_cast<uint8_t*>(c.wy);
    p.T = c.T;
    p.H = c.H;
    p.decay_first = c.decay_first;
    p.cu_seqlens = c.cu_seqlens;
    p.cu_chunks = c.cu_chunks;
    p.nseq = c.B;
    p.total_chunks = c.total_chunks;
    p.wy_lo = lo;
    p.wy_cnt = cnt;
    p.queue = c.wy_queue;
    p.queue_reset = c.wy_queue_reset;
    p.items = (unsigned)nblk;
    p.err = c.err;
    p.wait_limit = 4000000000LL;   // ~2 s at GB300 clocks
    void (*kern)(WyParams) = c.wy_queue ? wy_queue_kernel : wy_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kWySmem);
    if (e != cudaSuccess) return e;
    if (!c.wy_queue) {
        wy_kernel<<<(unsigned)nblk, kWyThreads, kWySmem, s>>>(p);
        return cudaGetLastError();
    }
    // as many CTAs as the whole GPU holds at once (six per SM), or fewer if there are fewer
    // chunks; optionally launched as the programmatic dependent of the preceding grid
    int sms = 0, dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    const long long grid = std::min<long long>(nblk, 6LL * std::max(sms, 1));
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kWyThreads);
    cfg.dynamicSmemBytes = kWySmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = c.launch_dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, wy_queue_kernel, p);
}

}  // namespace gdn
