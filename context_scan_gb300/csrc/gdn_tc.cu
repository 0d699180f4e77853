// gdn_tc.cu -- tcgen05 tensor-core chain kernels for bf16 inputs with K == V == 128.
//
// One CTA owns one chain: a (b, h, segment) and one 128-column block of the state. The
// forward chain's block is the K x V state itself; a summary chain's block is either the
// M part (state started from I, value vectors 0) or the S part (started from 0, values v)
// of the augmented K x (K+V) summary state (RFC: HyperParallel Linear Attention Context
// Parallel, section 2.2: S is reached from H_in = 0, M is the linear part). The chain walks
// its segment's 64-token chunks in order with the fp32 state kept in tensor memory.
//
// Chunk equations ("Context Parallelism in ART", section 08, "First parallelize within a
// GPU", with the un-decayed read of the RFC's section 2.1), gates in log2 units:
//   G  = inclusive cumsum of g in the chunk, Gx = G - g (exclusive)
//   L  = diag(beta) P,  P[i,j] = 2^(Gx_i - G_j) k_i.k_j (j < i);   A = (I + L)^-1
//   U  = A diag(beta) V,   W = A diag(beta 2^Gx) K
//   R  = U - W H
//   O  = Qd H + C R,   Qd = diag(2^G) Q,   C[i,j] = 2^(G_i - G_j) q_i.k_j (j <= i)
//   H <- 2^(G_last) H + sum_j 2^(G_last - G_j) k_j R_j
// Every contraction is an M = 128 tcgen05.mma with fp32 accumulation in tensor memory; a
// 128-wide dimension (v or k) is put on M, so the products are formed transposed:
//   P1  [K ; Q] K^T        rows 0..63: K K^T, rows 64..127: Q K^T      kind::f16 (bf16)
//   P2  U^T = V^T (A diag(beta))^T                                      kind::f16
//   P3  W^T = K^T (A diag(beta 2^Gx))^T                                 kind::f16
//   S1  R^T = U^T + H^T (-W)^T      A = H^T from tensor memory          kind::tf32
//   S2  O^T = H^T Qd^T              A = H^T from tensor memory          kind::tf32
//   S3  O^T += R^T C^T              A = R^T from tensor memory          kind::tf32
//   S4  H^T += (R^T diag(2^(G_last - G))) K, the decayed R^T held in tensor memory as an
//       unevaluated bf16 sum hi + lo (two MMAs); the master is pre-scaled by 2^G_last.
// The fp32 state and the corrected values R never pass through bf16. Exponents are always
// differences of cumulative gates, never 2^-G. The factors A diag(beta) and A diag(beta 2^Gx),
// A = (I + L)^-1, depend only on the chunk's keys and gates: the WY kernel (gdn_wy.cu) forms
// them for every chunk beforehand, fully parallel, and a chain loads a chunk's pair with one
// bulk copy next to its k/q tiles.
//
// Warp roles: warps 0-3 "state" (tensor-memory lanes 0..127; S1-S4, output, final state),
// warps 4-7 "prep" (P1-P3, gate cumsum, C, Qd, -W), warp 8 "producer" (TMA loads of the
// q/k/v tiles with 128-byte swizzle and bulk copies of the WY tiles into two stages; plain
// loads of the gates). Prep of chunk n+1 runs while the state group works on chunk n. Each
// group issues its own MMAs (commits track the issuing thread's MMAs). Named barriers are
// the non-.aligned form: a group's leader warp diverges around its mbarrier poll, and the
// .aligned form may count a diverged warp's halves as separate arrivals. Every wait on an
// mbarrier is bounded: on expiry the kernel records GDN_ERR_TIMEOUT in the device error
// word, drains what it issued and frees tensor memory.
#include <cstring>

#include "gdn_tc_common.cuh"

namespace gdn {
namespace {

constexpr int kD = 128;        // K == V
constexpr int kC = 64;         // tokens per chunk
constexpr int kThreads = 288;  // 4 state warps + 4 prep warps + 1 producer warp
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

// tensor-memory columns (32-bit cells, 128 lanes)
constexpr uint32_t TM_S = 0;     // [K;Q] K^T, then W^T                       (prep)
constexpr uint32_t TM_U = 64;    // U^T -> R^T, two buffers by chunk parity   (64, 128)
constexpr uint32_t TM_O = 192;   // O^T, two buffers by chunk parity          (192, 256)
constexpr uint32_t TM_RD = 320;  // decayed R^T as packed bf16: hi 320..351, lo 352..383
constexpr uint32_t TM_H = 384;   // state master H^T (128 columns)

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t SM_KQ0 = 0;        // stage 0: [khalf][K rows | Q rows], 2 x 16 KB
constexpr uint32_t SM_KQ1 = 32768;    // stage 1
constexpr uint32_t SM_V = 65536;      // [vhalf][64 rows x 128 B]
constexpr uint32_t SM_W = 81920;      // -W tf32 K-major: [kblock 4][64 rows (i) x 32 (k)]
constexpr uint32_t SM_QT = 114688;    // Qd tf32 K-major: [kblock 4][64 rows (i) x 32 (k)]
constexpr uint32_t SM_C0 = 147456;    // C tf32 K-major: [kblock 2][64 rows (i) x 32 (j)], x2
constexpr uint32_t SM_C1 = 163840;
constexpr uint32_t SM_A0 = 180224;    // stage 0 WY tiles: A diag(beta) | A diag(beta 2^Gx), bf16
constexpr uint32_t SM_A1 = 196608;    // stage 1
constexpr uint32_t SM_SCAL = 212992;  // per-chunk scalars [parity 2][SC_N][64] + gates [stage 2][64]
constexpr uint32_t SM_BAR = 215552;   // mbarriers and flags
constexpr uint32_t SM_END = 215680;
constexpr uint32_t kSmemBytes = SM_END + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

// per-chunk scalar arrays (offsets in units of 64 floats within a parity block)
enum { SC_GAM = 0, SC_DD, SC_EG, SC_MISC, SC_N = 4 };

// mbarrier slots and flags at SM_BAR
constexpr uint32_t B_FULL0 = 0, B_FULL1 = 8, B_EMPTY0 = 16, B_EMPTY1 = 24, B_VEMPTY = 32,
                   B_BARP = 40, B_BARS = 48, B_PREPDONE = 56, B_WFREE = 64, B_UFREE0 = 72,
                   B_UFREE1 = 80, B_TMEM = 88, B_ABORT = 92, B_GO_S = 96, B_GO_P = 100,
                   B_VFULL = 104;

// wait tags recorded in the device error word's detail field
enum : unsigned {
    TAG_FULL = 1, TAG_BARP = 2, TAG_BARS = 3, TAG_EMPTY = 4, TAG_VEMPTY = 5, TAG_PREPDONE = 6,
    TAG_WFREE = 7, TAG_UFREE = 8, TAG_VFULL = 9
};

struct TcParams {
    CUtensorMap tm_q;
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    ChainParams c;
    long long wait_limit;   // SM clock cycles before a wait gives up
};

// 64 token rows of one output column from a 64-column O^T buffer in tensor memory
__device__ __forceinline__ void store_o_rows(const ChainParams& c, uint32_t t_col, long long idx0,
                                             long long tok_stride) {
#pragma unroll 1
    for (int g = 0; g < 4; ++g) {
        float ov[16];
        tmem_ld16(t_col + 16 * g, ov);
        tmem_wait_ld();
        const long long base = idx0 + (long long)(16 * g) * tok_stride;
        if (c.out_bf16) {
            __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(c.o) + base;
#pragma unroll
            for (int j = 0; j < 16; ++j) o[(long long)j * tok_stride] = __float2bfloat16_rn(ov[j]);
        } else {
            float* o = reinterpret_cast<float*>(c.o) + base;
#pragma unroll
            for (int j = 0; j < 16; ++j) o[(long long)j * tok_stride] = ov[j];
        }
    }
}

// ------------------------------------------------------------------------------------
// the chain kernel
// ------------------------------------------------------------------------------------
template <bool SUMMARY>
__global__ void __launch_bounds__(kThreads, 1) tc_chain_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);

    float* scal = reinterpret_cast<float*>(sm + SM_SCAL);              // [parity][SC_N][64]
    float* gates = reinterpret_cast<float*>(sm + SM_SCAL + 2 * SC_N * 256);   // [stage][64]
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sm + SM_BAR + B_TMEM);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + SM_BAR + B_ABORT);
    const uint32_t bar0 = base + SM_BAR;

    const ChainParams& c = p.c;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    int blk = 1;                    // 1: values are v (forward, or the S part); 0: M part
    int chain = blockIdx.x;
    if (SUMMARY) {
        blk = chain & 1;
        chain >>= 1;
    }
    const int seg = chain % c.nseg_run;
    const int bh = chain / c.nseg_run;
    const int b = bh / c.H, h = bh % c.H;
    const int nchunks = c.seg_len / kC;
    const bool need_v = !SUMMARY || blk == 1;
    const long long limit = p.wait_limit;

    if (tid == 0) {
        mbar_init(bar0 + B_FULL0, 2);
        mbar_init(bar0 + B_FULL1, 2);
        mbar_init(bar0 + B_EMPTY0, 1);
        mbar_init(bar0 + B_EMPTY1, 1);
        mbar_init(bar0 + B_VEMPTY, 1);
        mbar_init(bar0 + B_VFULL, 1);
        mbar_init(bar0 + B_BARP, 1);
        mbar_init(bar0 + B_BARS, 1);
        mbar_init(bar0 + B_PREPDONE, 1);
        mbar_init(bar0 + B_WFREE, 1);
        mbar_init(bar0 + B_UFREE0, 1);
        mbar_init(bar0 + B_UFREE1, 1);
        *abort_flag = 0;
        *reinterpret_cast<volatile int*>(sm + SM_BAR + B_GO_S) = 1;
        *reinterpret_cast<volatile int*>(sm + SM_BAR + B_GO_P) = 1;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         bar0 + B_TMEM),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8) {
        // ================================ producer ================================
        // K and Q tiles, the WY tiles and the gates go to a two-stage ring released after
        // S4; the V tile has its own single buffer released after P2, so a chunk's K and Q are
        // never held back by the previous chunk's V. The M part needs only A diag(beta 2^Gx).
        const uint32_t wy_bytes = need_v ? 16384u : 8192u;
        const uint32_t wy_skip = 16384u - wy_bytes;
        const uint32_t tx = 16384u + (SUMMARY ? 0u : 16384u) + wy_bytes;
        const uint8_t* wy_chain = reinterpret_cast<const uint8_t*>(c.wy) +
                                  (((long long)bh * (c.T / kC) + (long long)seg * nchunks) << 14);
        int issued_last[2] = {-1, -1}, v_issued_last = -1;
#pragma unroll 1
        for (int n = 0; n < nchunks; ++n) {
            const int s = n & 1;
            const uint32_t full = bar0 + (s ? B_FULL1 : B_FULL0);
            const int row0 = b * c.T + seg * c.seg_len + n * kC;   // flattened (b, t) row
            // the whole warp polls together (identical values in every lane), so it stays
            // converged and never waits on itself
            if (n >= 2 && !mbar_wait(bar0 + (s ? B_EMPTY1 : B_EMPTY0), ((n >> 1) - 1) & 1,
                                     abort_flag, limit, c.err, TAG_EMPTY))
                break;
            if (lane == 0) {
                mbar_arrive_expect_tx(full, tx);
                const uint32_t kq = base + (s ? SM_KQ1 : SM_KQ0);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    tma_load_3d(kq + hf * 16384, &p.tm_k, full, hf * 64, h, row0);
                    if (!SUMMARY) tma_load_3d(kq + hf * 16384 + 8192, &p.tm_q, full, hf * 64, h, row0);
                }
                bulk_load(base + (s ? SM_A1 : SM_A0) + wy_skip,
                          wy_chain + ((long long)n << 14) + wy_skip, wy_bytes, full);
            }
            if (s) issued_last[1] = n; else issued_last[0] = n;
            float* gs = gates + s * 64;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int i = lane + 32 * e;
                gs[i] = bf16_at(c.g, (long long)(row0 + i) * c.H + h) * kLog2e;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(full);
            if (need_v) {
                if (n >= 1 &&
                    !mbar_wait(bar0 + B_VEMPTY, (n - 1) & 1, abort_flag, limit, c.err, TAG_VEMPTY))
                    break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar0 + B_VFULL, 16384u);
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf)
                        tma_load_3d(base + SM_V + hf * 8192, &p.tm_v, bar0 + B_VFULL, hf * 64, h, row0);
                }
                v_issued_last = n;
            }
        }
        if (*abort_flag && lane == 0) {
            // let every copy this warp issued land before the CTA's memory is released
            if (issued_last[0] >= 0) mbar_drain(bar0 + B_FULL0, (issued_last[0] >> 1) & 1, limit);
            if (issued_last[1] >= 0) mbar_drain(bar0 + B_FULL1, (issued_last[1] >> 1) & 1, limit);
            if (v_issued_last >= 0) mbar_drain(bar0 + B_VFULL, v_issued_last & 1, limit);
        }
    } else if (warp >= 4) {
        // ================================== prep ==================================
        const int pt = tid - 128, pw = warp - 4;
        const uint32_t t_row = tmem + ((uint32_t)(pw * 32) << 16);   // this warp's TMEM lanes
        volatile int* go = reinterpret_cast<volatile int*>(sm + SM_BAR + B_GO_P);
        uint32_t barp_phase = 0;
        bool barp_pending = false;

        // the group's first warp waits (optionally) and publishes a verdict that all read
        // after the named barrier, so a timeout cannot split the group
#define pwait(bar, parity, tag, doit) \
    group_wait<2>(pw == 0, lane == 0, (bar), (parity), (doit), go, abort_flag, limit, c.err, (tag))
#define pmma_wait() \
    (pwait(bar0 + B_BARP, barp_phase, TAG_BARP, true) ? (barp_phase ^= 1u, barp_pending = false, true) : false)

#pragma unroll 1
        for (int n = 0; n < nchunks; ++n) {
            const int s = n & 1;
            const uint32_t kq = base + (s ? SM_KQ1 : SM_KQ0);
            const uint32_t wyt = base + (s ? SM_A1 : SM_A0);
            float* sc = scal + (n & 1) * (SC_N * 64);
            if (!pwait(bar0 + (s ? B_FULL1 : B_FULL0), (n >> 1) & 1, TAG_FULL, true)) break;

            // ---- P1: [K ; Q] K^T -> TM_S; rows 64..127 (Q K^T) give C
            if (!SUMMARY && pt == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_ss(tmem + TM_S, desc_k(kq + off), desc_k(kq + off), ID_P1, ks > 0);
                }
                mma_commit(bar0 + B_BARP);
            }
            // ---- gate cumsum and per-chunk scalars (first prep warp)
            if (pw == 0) {
                const float* gs = gates + s * 64;
                const float g0 = gs[2 * lane], g1 = gs[2 * lane + 1];
                float sum = g0 + g1;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o = __shfl_up_sync(0xffffffffu, sum, off);
                    if (lane >= off) sum += o;
                }
                const float excl = sum - (g0 + g1);
                const float glast = __shfl_sync(0xffffffffu, sum, 31);
                const float G0 = excl + g0, G1 = excl + g0 + g1;
                sc[SC_GAM * 64 + 2 * lane] = G0;
                sc[SC_GAM * 64 + 2 * lane + 1] = G1;
                sc[SC_DD * 64 + 2 * lane] = ex2(glast - G0);
                sc[SC_DD * 64 + 2 * lane + 1] = ex2(glast - G1);
                sc[SC_EG * 64 + 2 * lane] = ex2(G0);
                sc[SC_EG * 64 + 2 * lane + 1] = ex2(G1);
                if (lane == 0) sc[SC_MISC * 64] = ex2(glast);
            }
            __syncwarp();
            if (!SUMMARY) {
                barp_pending = true;
                if (!pmma_wait()) break;   // its barrier also publishes the scalars
                tc_fence_after();
                // C and Qd overwrite what chunk n-2's S3 and chunk n-1's S2 read
                if (!pwait(bar0 + B_WFREE, (n - 1) & 1, TAG_WFREE, n >= 1)) break;
                if (pt >= 64) {
                    // ---- C rows (lanes 64..127), tf32 K-major, 16 columns at a time
                    const float* gam = sc + SC_GAM * 64;
                    const int i = pt & 63;
                    const float gi = gam[i];
                    uint8_t* ctile = sm + ((n & 1) ? SM_C1 : SM_C0);
#pragma unroll 1
                    for (int g = 0; g < 4; ++g) {
                        float sv[16];
                        tmem_ld16(t_row + TM_S + 16 * g, sv);
                        tmem_wait_ld();
                        uint32_t t[16];
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int j = 16 * g + jj;
                            t[jj] = tf32_bits((j <= i) ? ex2(gi - gam[j]) * sv[jj] : 0.f);
                        }
                        // columns 16g..16g+15: tf32 block g >> 1, 16-byte chunks 4(g&1)..+3
                        uint8_t* blkp = ctile + (g >> 1) * 8192;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<uint4*>(blkp + sw128(i, 4 * (g & 1) + q)) =
                                make_uint4(t[4 * q], t[4 * q + 1], t[4 * q + 2], t[4 * q + 3]);
                    }
                } else {
                    // ---- Qd = 2^G_i q_i as tf32 K-major (threads 0..63: row i = pt)
                    const int i = pt;
                    const float egi = sc[SC_EG * 64 + i];
#pragma unroll 1
                    for (int kh = 0; kh < 2; ++kh) {
                        const uint8_t* src = sm + (s ? SM_KQ1 : SM_KQ0) + kh * 16384 + 8192;
#pragma unroll 2
                        for (int cc = 0; cc < 8; ++cc) {
                            const uint4 u = *reinterpret_cast<const uint4*>(src + sw128(i, cc));
                            const uint4 lo4 = make_uint4(
                                tf32_bits(__uint_as_float(u.x << 16) * egi),
                                tf32_bits(__uint_as_float(u.x & 0xFFFF0000u) * egi),
                                tf32_bits(__uint_as_float(u.y << 16) * egi),
                                tf32_bits(__uint_as_float(u.y & 0xFFFF0000u) * egi));
                            const uint4 hi4 = make_uint4(
                                tf32_bits(__uint_as_float(u.z << 16) * egi),
                                tf32_bits(__uint_as_float(u.z & 0xFFFF0000u) * egi),
                                tf32_bits(__uint_as_float(u.w << 16) * egi),
                                tf32_bits(__uint_as_float(u.w & 0xFFFF0000u) * egi));
                            // features 64 kh + 8 cc .. +7: tf32 block 2 kh + cc / 4, chunks
                            // 2 (cc % 4) + {0, 1}
                            uint8_t* dst = sm + SM_QT + (kh * 2 + (cc >> 2)) * 8192;
                            *reinterpret_cast<uint4*>(dst + sw128(i, (2 * cc) & 7)) = lo4;
                            *reinterpret_cast<uint4*>(dst + sw128(i, (2 * cc + 1) & 7)) = hi4;
                        }
                    }
                }
                fence_proxy_async();
                tc_fence_before();
                prep_bar();   // TM_S has been read: P3 may overwrite it
            }
            // ---- P2 (U^T into the parity's U buffer, once chunk n-2's R is retired) and P3
            const uint32_t t_u = tmem + TM_U + (n & 1) * 64;
            if (!pwait(bar0 + ((n & 1) ? B_UFREE1 : B_UFREE0), ((n >> 1) - 1) & 1, TAG_UFREE,
                       n >= 2))
                break;
            if (!pwait(bar0 + B_VFULL, n & 1, TAG_VFULL, need_v)) break;
            if (pt == 0) {
                tc_fence_after();
                if (need_v) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ss(t_u, desc_mn(base + SM_V + ks * 2048, 8192), desc_k(wyt + ks * 32),
                               ID_P23, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(tmem + TM_S, desc_mn(kq + ks * 2048, 16384),
                           desc_k(wyt + 8192 + ks * 32), ID_P23, ks > 0);
                if (need_v) mma_commit(bar0 + B_VEMPTY);
                mma_commit(bar0 + B_BARP);
            }
            __syncwarp();
            barp_pending = true;
            if (!pmma_wait()) break;
            tc_fence_after();
            // ---- -W as a tf32 K-major B operand, once chunk n-1's S1 retired
            {
                if (SUMMARY && !pwait(bar0 + B_WFREE, (n - 1) & 1, TAG_WFREE, n >= 1)) break;
                // thread k holds column k of W^T's rows i: writes element (row i, feature k)
                const int k = pt;
                uint8_t* col = sm + SM_W + (k >> 5) * 8192 + (k & 3) * 4;
                const int qk = (k & 31) >> 2;
#pragma unroll 1
                for (int g = 0; g < 4; ++g) {
                    float w[16];
                    tmem_ld16(t_row + TM_S + 16 * g, w);
                    tmem_wait_ld();
#pragma unroll
                    for (int ii = 0; ii < 16; ++ii)
                        *reinterpret_cast<uint32_t*>(col + sw128(16 * g + ii, qk)) = tf32_bits(-w[ii]);
                }
            }
            fence_proxy_async();
            tc_fence_before();
            prep_bar();
            if (pt == 0) mbar_arrive(bar0 + B_PREPDONE);
        }
        if (*go == 0 && barp_pending && pt == 0) mbar_drain(bar0 + B_BARP, barp_phase, limit);
#undef pmma_wait
#undef pwait
    } else {
        // ================================== state =================================
        const int st = tid;
        const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);
        volatile int* go = reinterpret_cast<volatile int*>(sm + SM_BAR + B_GO_S);
        uint32_t bars_phase = 0;
        bool bars_pending = false;
        const long long bhoff = (long long)bh * kD * kD;
        const long long tok_stride = (long long)c.H * kD;   // elements between two tokens of o

#define swait(bar, parity, tag) \
    group_wait<1>(warp == 0, lane == 0, (bar), (parity), true, go, abort_flag, limit, c.err, (tag))
#define smma_wait() \
    (swait(bar0 + B_BARS, bars_phase, TAG_BARS) ? (bars_phase ^= 1u, bars_pending = false, true) : false)
// o rows of chunk m from that chunk's O buffer: thread v writes column v
#define store_output(m)                                                                          \
    store_o_rows(c, t_row + TM_O + ((m) & 1) * 64,                                               \
                 ((long long)(b * c.T + seg * c.seg_len + (m) * kC) * c.H + h) * kD + st, tok_stride)

        // ---- initial state: row `st` of H^T (= column st of H)
#pragma unroll 1
        for (int g = 0; g < 8; ++g) {
            uint32_t x[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int k = 16 * g + j;
                float v0 = 0.f;
                if (SUMMARY)
                    v0 = (blk == 0 && k == st) ? 1.f : 0.f;
                else if (c.h_start)
                    v0 = c.h_start[seg * c.h_start_seg_stride + bhoff + (long long)k * kD + st];
                x[j] = __float_as_uint(v0);
            }
            tmem_st16(t_row + TM_H + 16 * g, x);
        }
        tmem_wait_st();
        tc_fence_before();
        state_bar();

        int done = 0;   // chunks completed
#pragma unroll 1
        for (int n = 0; n < nchunks; ++n) {
            const int s = n & 1;
            const uint32_t kq = base + (s ? SM_KQ1 : SM_KQ0);
            const uint32_t t_u = tmem + TM_U + (n & 1) * 64;
            const uint32_t t_o = tmem + TM_O + (n & 1) * 64;
            const float* sc = scal + (n & 1) * (SC_N * 64);
            if (!swait(bar0 + B_PREPDONE, n & 1, TAG_PREPDONE)) break;
            // ---- S1: R^T = U^T + H^T (-W)^T ;  S2: O^T = H^T Qd^T  (A = H^T in TMEM)
            if (st == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 16; ++ks)
                    mma_ts_tf32(t_u, tmem + TM_H + ks * 8,
                                desc_k(base + SM_W + (ks >> 2) * 8192 + (ks & 3) * 32), ID_TF,
                                (need_v || ks > 0) ? 1u : 0u);
                if (!SUMMARY) {
#pragma unroll
                    for (int ks = 0; ks < 16; ++ks)
                        mma_ts_tf32(t_o, tmem + TM_H + ks * 8,
                                    desc_k(base + SM_QT + (ks >> 2) * 8192 + (ks & 3) * 32), ID_TF,
                                    ks > 0);
                }
                mma_commit(bar0 + B_WFREE);
                mma_commit(bar0 + B_BARS);
            }
            __syncwarp();
            bars_pending = true;
            // ---- meanwhile: the previous chunk's output
            if (!SUMMARY && n >= 1) {
                tc_fence_after();
                store_output(n - 1);
            }
            if (!smma_wait()) break;
            tc_fence_after();
            // ---- decayed R^T -> packed bf16 hi/lo in TMEM; pre-scale the master by 2^G_last
            {
                const float* dd = sc + SC_DD * 64;
                const uint32_t t_ur = t_row + TM_U + (n & 1) * 64;
#pragma unroll 1
                for (int g = 0; g < 4; ++g) {
                    float r[16];
                    tmem_ld16(t_ur + 16 * g, r);
                    tmem_wait_ld();
                    // packed column q holds the pair (2q, 2q+1) of the 64 tokens j
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float x0 = r[2 * j] * dd[16 * g + 2 * j];
                        const float x1 = r[2 * j + 1] * dd[16 * g + 2 * j + 1];
                        const float h0 = __bfloat162float(__float2bfloat16_rn(x0));
                        const float h1 = __bfloat162float(__float2bfloat16_rn(x1));
                        hi[j] = pack_bf16(h0, h1);
                        lo[j] = pack_bf16(x0 - h0, x1 - h1);
                    }
                    tmem_st8(t_row + TM_RD + 8 * g, hi);
                    tmem_st8(t_row + TM_RD + 32 + 8 * g, lo);
                }
                const float ecl = sc[SC_MISC * 64];
#pragma unroll 1
                for (int g = 0; g < 8; ++g) {
                    float x[16];
                    uint32_t y[16];
                    tmem_ld16(t_row + TM_H + 16 * g, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) y[j] = __float_as_uint(x[j] * ecl);
                    tmem_st16(t_row + TM_H + 16 * g, y);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            state_bar();
            // ---- S3: O^T += R^T C^T (A = R^T in TMEM) ; S4: H^T += (R^T D) K (A = hi, lo in TMEM)
            if (st == 0) {
                tc_fence_after();
                if (!SUMMARY) {
                    const uint32_t cb = base + ((n & 1) ? SM_C1 : SM_C0);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ts_tf32(t_o, t_u + ks * 8, desc_k(cb + (ks >> 2) * 8192 + (ks & 3) * 32),
                                    ID_TF, 1u);
                }
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ts_bf16(tmem + TM_H, tmem + TM_RD + part * 32 + ks * 8,
                                    desc_mn(kq + ks * 2048, 16384), ID_S4, 1u);
                mma_commit(bar0 + (s ? B_EMPTY1 : B_EMPTY0));
                mma_commit(bar0 + ((n & 1) ? B_UFREE1 : B_UFREE0));
                mma_commit(bar0 + B_BARS);
            }
            __syncwarp();
            bars_pending = true;
            if (!smma_wait()) break;
            tc_fence_after();
            done = n + 1;
        }

        if (*go == 0) {
            if (bars_pending && st == 0)   // let an issued MMA group retire before TMEM is freed
                mbar_drain(bar0 + B_BARS, bars_phase, limit);
        } else {
            if (!SUMMARY && done >= 1) store_output(done - 1);
            // ---- the chain's final state: thread v writes column v of H (row v of H^T)
            float* dst = nullptr;
            if (SUMMARY) {
                const long long sb = ((long long)seg * c.B * c.H + bh) * kD * kD;
                dst = (blk == 0 ? c.M : c.S) + sb;
            } else if (c.h_final && seg == c.nseg_total - 1) {
                dst = c.h_final + bhoff;
            }
            if (dst) {
#pragma unroll 1
                for (int g = 0; g < 8; ++g) {
                    float x[16];
                    tmem_ld16(t_row + TM_H + 16 * g, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) dst[(long long)(16 * g + j) * kD + st] = x[j];
                }
            }
        }
#undef store_output
#undef smma_wait
#undef swait
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

// ------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------
template <bool SUMMARY>
cudaError_t launch(const ChainParams& c, cudaStream_t s) {
    if (!c.wy) return cudaErrorInvalidValue;
    TcParams tp;
    memset(&tp, 0, sizeof(tp));
    tp.c = c;
    tp.wait_limit = 4000000000LL;   // ~2 s at GB300 clocks
    if (!make_map(&tp.tm_k, c.k, c)) return cudaErrorInvalidValue;
    if (!SUMMARY && !make_map(&tp.tm_q, c.q, c)) return cudaErrorInvalidValue;
    if (!make_map(&tp.tm_v, c.v, c)) return cudaErrorInvalidValue;
    auto kern = tc_chain_kernel<SUMMARY>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long chains = (long long)c.B * c.H * c.nseg_run * (SUMMARY ? 2 : 1);
    kern<<<(unsigned)chains, kThreads, kSmemBytes, s>>>(tp);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(const ChainParams& p) {
    return p.in_bf16 && p.K == kD && p.V == kD && p.seg_len > 0 && p.seg_len % kC == 0 &&
           encode_fn() != nullptr;
}

cudaError_t launch_tc_forward(const ChainParams& p, cudaStream_t s) { return launch<false>(p, s); }
cudaError_t launch_tc_summary(const ChainParams& p, cudaStream_t s) { return launch<true>(p, s); }

}  // namespace gdn
