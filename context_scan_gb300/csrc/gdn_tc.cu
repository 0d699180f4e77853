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
// The factors A diag(beta) and A diag(beta 2^Gx) depend only on the chunk's keys and gates:
// the WY kernel (gdn_wy.cu) forms them for every chunk beforehand, fully parallel, and a
// chain loads a chunk's pair with one bulk copy.
//
// Scaled state. The master in tensor memory is H_s with H = sigma H_s, where the scalar
// sigma is a function of the gates alone: sigma <- sigma 2^(G_last) after each chunk. The
// decay then never touches the 128 x 128 master: it moves into the scalars of the operands
// (-sigma W, sigma Qd) and of the update (2^(G_last - G_j) / sigma_next). When sigma_next
// would fall below 2^-64 the chunk folds sigma into the master instead (one pass over it)
// and sigma restarts at 1, so no scale factor exceeds 2^64. sigma is tracked as log2.
//
// Every contraction is an M = 128 tcgen05.mma with fp32 accumulation in tensor memory; a
// 128-wide dimension (v or k) is put on M, so the products are formed transposed:
//   P1  [Q ; -] K^T        rows 0..63: Q K^T (rows 64..127 unused)      kind::f16 (bf16)
//   P2  U^T = V^T (A diag(beta))^T                                      kind::f16
//   P3  W^T = K^T (A diag(beta 2^Gx))^T                                 kind::f16
//   S12 [R^T | O^T] = [U^T | 0] + H_s^T [-sigma W ; sigma Qd]^T       kind::tf32, N = 128
//       (A = H_s^T from tensor memory; the summary has no O and runs the R^T half, N = 64)
//   S3  O^T += R^T C^T                     A = R^T from tensor memory   kind::tf32
//   S4  H_s^T += (R^T diag(2^(G_last - G) / sigma_next)) K, the scaled R^T held in tensor
//       memory as an unevaluated bf16 sum hi + lo (two MMAs).
// The fp32 state and the corrected values R never pass through bf16. Exponents are always
// differences of cumulative gates or bounded by the renormalisation.
//
// Warp roles: warps 0-3 "state" (tensor-memory lanes 0..127; S1-S4, final state), warps
// 4-11 "prep" (two warp groups, each covering lanes 0..127: P1-P3, gate cumsum and the
// sigma bookkeeping, C, sigma Qd, -sigma W, and the output rows of chunk n-2; P1 of chunk
// n+1 is issued as soon as chunk n's W^T has been read out of tensor memory), warp 12
// "producer" (TMA loads of the q/k/v tiles with 128-byte swizzle, bulk copies of the WY
// tiles, gates). Rings: k in KST stages (released by S4), q in two (released by prep), WY
// tiles in AST (released by P3), v in one (released by P2). Prep of chunk n+1 runs while the
// state group works on chunk n. Each group issues its own MMAs (commits track the issuing
// thread's MMAs). Named barriers are the non-.aligned form: a group's leader warp diverges
// around its mbarrier poll. Every wait on an mbarrier is bounded: on expiry the kernel
// records GDN_ERR_TIMEOUT in the device error word, drains what it issued and frees tensor
// memory.
#include <cstring>

#include "gdn_tc_common.cuh"

namespace gdn {
namespace {

constexpr int kD = 128;         // K == V
constexpr int kC = 64;          // tokens per chunk
constexpr int kThreads = 416;   // 4 state warps + 8 prep warps + 1 producer warp
constexpr int kPrepThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRenorm = -64.f;   // log2 of the smallest sigma kept without folding

// tensor-memory columns (32-bit cells, 128 lanes)
constexpr uint32_t TM_S = 0;     // Q K^T, then W^T                           (prep)
constexpr uint32_t TM_U = 64;    // two buffers by chunk parity: U^T -> R^T, and in the
                                 // forward O^T right after it (64 + 128 p: R^T | O^T)
constexpr uint32_t TM_RD = 320;  // scaled R^T as packed bf16: hi 320..351, lo 352..383
constexpr uint32_t TM_H = 384;   // state master H_s^T (128 columns)

// Shared-memory map (bytes from a 1024-aligned base). A k, q or v tile is two 64-feature
// halves of 64 rows x 128 bytes (8 KB each, 128-byte swizzle); a WY stage is the tile pair
// A diag(beta) | A diag(beta 2^Gx) (8 KB each).
template <bool SUMMARY>
struct Smem {
    static constexpr int KST = SUMMARY ? 4 : 3;   // k ring stages
    static constexpr int QST = SUMMARY ? 0 : 2;   // q ring stages
    static constexpr int AST = SUMMARY ? 2 : 1;   // WY tile stages
    static constexpr uint32_t K0 = 0;
    static constexpr uint32_t Q0 = K0 + KST * 16384;
    static constexpr uint32_t A0 = Q0 + QST * 16384;
    static constexpr uint32_t V = A0 + AST * 16384;
    // the S12 B operand, tf32 K-major: [kblock 4][-sigma W rows i (64) | sigma Qd rows i (64)]
    // x 32 features (the summary holds only the W rows)
    static constexpr uint32_t WQ_KB = SUMMARY ? 8192 : 16384;   // bytes per kblock
    static constexpr uint32_t W = V + 16384;
    static constexpr uint32_t C0 = W + 4 * WQ_KB;   // C tf32: [kblock 2][64 (i) x 32 (j)], x2
    static constexpr uint32_t SCAL = C0 + (SUMMARY ? 0 : 32768);
    static constexpr uint32_t TU_STRIDE = SUMMARY ? 64 : 128;   // tensor-memory U(+O) buffer pitch
    static constexpr uint32_t GATES = SCAL + 2 * 4 * 256;        // after scalars [parity 2][SC_N][64]
    static constexpr uint32_t BAR = GATES + KST * 256;           // gates [k stage][64]
    static constexpr uint32_t END = BAR + 256;
    static constexpr uint32_t BYTES = END + 1024;                // + alignment slack
    static_assert(BYTES <= 232448, "shared memory budget");
};

// per-chunk scalar arrays (offsets in units of 64 floats within a parity block)
enum { SC_GAM = 0, SC_DD, SC_EG, SC_MISC, SC_N = 4 };
// SC_MISC slots: 0 = fold factor for the master (1 if none), 1 = sigma after the chunk,
// 2 = sigma during the chunk

// mbarrier slots and flags at Smem::BAR
constexpr uint32_t B_KFULL = 0, B_KEMPTY = 32, B_QFULL = 64, B_QEMPTY = 80, B_AFULL = 96,
                   B_AEMPTY = 112, B_VFULL = 128, B_VEMPTY = 136, B_BARP = 144, B_BARS = 152,
                   B_PREPDONE = 160, B_WFREE = 168, B_UFREE = 176, B_TMEM = 192, B_ABORT = 196,
                   B_GO_S = 200, B_GO_P = 204;

// wait tags recorded in the device error word's detail field
enum : unsigned {
    TAG_KFULL = 1, TAG_BARP = 2, TAG_BARS = 3, TAG_KEMPTY = 4, TAG_VEMPTY = 5, TAG_PREPDONE = 6,
    TAG_WFREE = 7, TAG_UFREE = 8, TAG_VFULL = 9, TAG_QFULL = 10, TAG_QEMPTY = 11,
    TAG_AFULL = 12, TAG_AEMPTY = 13
};

struct TcParams {
    CUtensorMap tm_q;
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    ChainParams c;
    long long wait_limit;   // SM clock cycles before a wait gives up
};

// 32 token rows of one output column from a 64-column O^T buffer in tensor memory
__device__ __forceinline__ void store_o_rows32(const ChainParams& c, uint32_t t_col, long long idx0,
                                               long long tok_stride) {
#pragma unroll 1
    for (int g = 0; g < 2; ++g) {
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
// 13 warps are allocated registers as 16: bound them at 65536 / 512 per thread
template <bool SUMMARY>
__global__ void __launch_bounds__(512, 1) tc_chain_kernel(const __grid_constant__ TcParams p) {
    using L = Smem<SUMMARY>;
    constexpr int KST = L::KST, AST = L::AST;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);

    float* scal = reinterpret_cast<float*>(sm + L::SCAL);     // [parity][SC_N][64]
    float* gates = reinterpret_cast<float*>(sm + L::GATES);   // [k stage][64]
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sm + L::BAR + B_TMEM);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::BAR + B_ABORT);
    const uint32_t bar0 = base + L::BAR;

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
    const long long tok_stride = (long long)c.H * kD;   // elements between two tokens of o
    const long long row_seg = (long long)b * c.T + (long long)seg * c.seg_len;   // flattened (b, t)

    if (tid == 0) {
        for (int i = 0; i < KST; ++i) {
            mbar_init(bar0 + B_KFULL + 8 * i, 2);
            mbar_init(bar0 + B_KEMPTY + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar0 + B_QFULL + 8 * i, 1);
            mbar_init(bar0 + B_QEMPTY + 8 * i, 1);
            mbar_init(bar0 + B_AFULL + 8 * i, 1);
            mbar_init(bar0 + B_AEMPTY + 8 * i, 1);
            mbar_init(bar0 + B_UFREE + 8 * i, 1);
        }
        mbar_init(bar0 + B_VFULL, 1);
        mbar_init(bar0 + B_VEMPTY, 1);
        mbar_init(bar0 + B_BARP, 1);
        mbar_init(bar0 + B_BARS, 1);
        mbar_init(bar0 + B_PREPDONE, 1);
        mbar_init(bar0 + B_WFREE, 1);
        *abort_flag = 0;
        *reinterpret_cast<volatile int*>(sm + L::BAR + B_GO_S) = 1;
        *reinterpret_cast<volatile int*>(sm + L::BAR + B_GO_P) = 1;
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

    if (warp == 12) {
        // ================================ producer ================================
        // The whole warp runs the loop (its lanes poll together and stay converged); lane 0
        // issues the copies, every lane loads two gates. The gates of chunk n+1 are loaded
        // into registers while chunk n's copies are in flight.
        const uint32_t wy_bytes = need_v ? 16384u : 8192u;
        const uint32_t wy_skip = 16384u - wy_bytes;
        const uint8_t* wy_chain = reinterpret_cast<const uint8_t*>(c.wy) +
                                  (((long long)bh * (c.T / kC) + (long long)seg * nchunks) << 14);
        int k_last[KST], q_last[2] = {-1, -1}, a_last[2] = {-1, -1}, v_last = -1;
#pragma unroll
        for (int i = 0; i < KST; ++i) k_last[i] = -1;
        float gpre0 = 0.f, gpre1 = 0.f;
        if (nchunks > 0) {
            gpre0 = bf16_at(c.g, (row_seg + lane) * c.H + h) * kLog2e;
            gpre1 = bf16_at(c.g, (row_seg + lane + 32) * c.H + h) * kLog2e;
        }
#pragma unroll 1
        for (int n = 0; n < nchunks; ++n) {
            const long long row0 = row_seg + (long long)n * kC;
            const int ks = n % KST;
            if (n >= KST && !mbar_wait(bar0 + B_KEMPTY + 8 * ks, ((n / KST) - 1) & 1, abort_flag,
                                       limit, c.err, TAG_KEMPTY))
                break;
            if (lane == 0) {
                const uint32_t full = bar0 + B_KFULL + 8 * ks;
                mbar_arrive_expect_tx(full, 16384u);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
                    tma_load_3d(base + L::K0 + ks * 16384 + hf * 8192, &p.tm_k, full, hf * 64, h,
                                (int)row0);
            }
            k_last[ks] = n;
            gates[ks * 64 + lane] = gpre0;
            gates[ks * 64 + lane + 32] = gpre1;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar0 + B_KFULL + 8 * ks);
            if (n + 1 < nchunks) {
                gpre0 = bf16_at(c.g, (row0 + kC + lane) * c.H + h) * kLog2e;
                gpre1 = bf16_at(c.g, (row0 + kC + lane + 32) * c.H + h) * kLog2e;
            }
            if (!SUMMARY) {
                const int qs = n & 1;
                if (n >= 2 && !mbar_wait(bar0 + B_QEMPTY + 8 * qs, ((n >> 1) - 1) & 1, abort_flag,
                                         limit, c.err, TAG_QEMPTY))
                    break;
                if (lane == 0) {
                    const uint32_t full = bar0 + B_QFULL + 8 * qs;
                    mbar_arrive_expect_tx(full, 16384u);
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf)
                        tma_load_3d(base + L::Q0 + qs * 16384 + hf * 8192, &p.tm_q, full, hf * 64,
                                    h, (int)row0);
                }
                q_last[qs] = n;
            }
            {
                const int as = n % AST;
                if (n >= AST && !mbar_wait(bar0 + B_AEMPTY + 8 * as, ((n / AST) - 1) & 1,
                                           abort_flag, limit, c.err, TAG_AEMPTY))
                    break;
                if (lane == 0) {
                    const uint32_t full = bar0 + B_AFULL + 8 * as;
                    mbar_arrive_expect_tx(full, wy_bytes);
                    bulk_load(base + L::A0 + as * 16384 + wy_skip,
                              wy_chain + ((long long)n << 14) + wy_skip, wy_bytes, full);
                }
                a_last[as] = n;
            }
            if (need_v) {
                if (n >= 1 &&
                    !mbar_wait(bar0 + B_VEMPTY, (n - 1) & 1, abort_flag, limit, c.err, TAG_VEMPTY))
                    break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar0 + B_VFULL, 16384u);
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf)
                        tma_load_3d(base + L::V + hf * 8192, &p.tm_v, bar0 + B_VFULL, hf * 64, h,
                                    (int)row0);
                }
                v_last = n;
            }
        }
        if (*abort_flag && lane == 0) {
            // let every copy this warp issued land before the CTA's memory is released
#pragma unroll
            for (int i = 0; i < KST; ++i)
                if (k_last[i] >= 0) mbar_drain(bar0 + B_KFULL + 8 * i, (k_last[i] / KST) & 1, limit);
            for (int i = 0; i < 2; ++i) {
                if (q_last[i] >= 0) mbar_drain(bar0 + B_QFULL + 8 * i, (q_last[i] >> 1) & 1, limit);
                if (a_last[i] >= 0) mbar_drain(bar0 + B_AFULL + 8 * i, (a_last[i] / AST) & 1, limit);
            }
            if (v_last >= 0) mbar_drain(bar0 + B_VFULL, v_last & 1, limit);
        }
    } else if (warp >= 4) {
        // ================================== prep ==================================
        const int pt = tid - 128, pw = warp - 4;
        const int grp = pw >> 2, lq = pw & 3;   // warp group (0, 1); tensor-memory lane quarter
        const uint32_t t_row = tmem + ((uint32_t)(lq * 32) << 16);   // this warp's TMEM lanes
        volatile int* go = reinterpret_cast<volatile int*>(sm + L::BAR + B_GO_P);
        uint32_t barp_phase = 0;
        bool barp_pending = false;
        float lam = 0.f;   // log2 sigma before the current chunk (first prep warp)

        // the group's first warp waits (optionally) and publishes a verdict that all read
        // after the named barrier, so a timeout cannot split the group
#define pwait(bar, parity, tag, doit)                                                          \
    group_wait<2, kPrepThreads>(pw == 0, lane == 0, (bar), (parity), (doit), go, abort_flag, \
                                limit, c.err, (tag))
#define pmma_wait() \
    (pwait(bar0 + B_BARP, barp_phase, TAG_BARP, true) ? (barp_phase ^= 1u, barp_pending = false, true) : false)
// output rows of chunk m from its O^T buffer: lanes v, this warp group's 32 token columns
#define store_output(m)                                                                       \
    store_o_rows32(c, t_row + TM_U + ((m) & 1) * 128 + 64 + 32 * grp,                          \
                   ((row_seg + (long long)(m) * kC + 32 * grp) * c.H + h) * kD + 32 * lq + lane, \
                   tok_stride)

// P1: [Q ; -] K^T -> TM_S for chunk m (k stage m % KST, q stage m & 1); lanes 0..63 hold
// Q K^T. Rows 64..127 of the A operand run into the next buffer and are never read.
#define issue_p1(m)                                                                           \
    do {                                                                                      \
        if (pt == 0) {                                                                        \
            const uint32_t kst1 = base + L::K0 + ((m) % KST) * 16384;                          \
            const uint32_t qst1 = base + L::Q0 + ((m) & 1) * 16384;                            \
            tc_fence_after();                                                                 \
            _Pragma("unroll") for (int k16 = 0; k16 < 8; ++k16) {                             \
                const uint32_t off = (k16 >> 2) * 8192 + (k16 & 3) * 32;                      \
                mma_ss<ID_P1>(tmem + TM_S, desc_k(qst1 + off), desc_k(kst1 + off), k16 > 0); \
            }                                                                                 \
            mma_commit(bar0 + B_BARP);                                                        \
        }                                                                                     \
        __syncwarp();                                                                         \
        barp_pending = true;                                                                  \
    } while (0)

        bool run = true;
        if (!SUMMARY && nchunks > 0) {
            run = pwait(bar0 + B_KFULL, 0, TAG_KFULL, true) && pwait(bar0 + B_QFULL, 0, TAG_QFULL, true);
            if (run) issue_p1(0);
        }
#pragma unroll 1
        for (int n = 0; run && n < nchunks; ++n) {
            const int ks = n % KST, qs = n & 1, as = n % AST;
            const uint32_t kst = base + L::K0 + ks * 16384;
            const uint32_t ast = base + L::A0 + as * 16384;
            const uint32_t t_u = tmem + TM_U + (n & 1) * L::TU_STRIDE;
            float* sc = scal + (n & 1) * (SC_N * 64);
            // chunk n-2 is retired: its scalars, U/R, O and C buffers may be reused
            if (!pwait(bar0 + B_UFREE + 8 * (n & 1), ((n >> 1) - 1) & 1, TAG_UFREE, n >= 2)) break;
            if (SUMMARY && !pwait(bar0 + B_KFULL + 8 * ks, (n / KST) & 1, TAG_KFULL, true)) break;

            // ---- gate cumsum, sigma bookkeeping and per-chunk scalars (first prep warp)
            if (pw == 0) {
                const float* gs = gates + ks * 64;
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
                const bool fold = lam + glast < kRenorm;
                const float lam_next = fold ? 0.f : lam + glast;
                sc[SC_GAM * 64 + 2 * lane] = G0;
                sc[SC_GAM * 64 + 2 * lane + 1] = G1;
                // update scale 2^(G_last - G_j) / sigma_next = 2^(-G_j - lam) unless folded
                sc[SC_DD * 64 + 2 * lane] = fold ? ex2(glast - G0) : ex2(-G0 - lam);
                sc[SC_DD * 64 + 2 * lane + 1] = fold ? ex2(glast - G1) : ex2(-G1 - lam);
                sc[SC_EG * 64 + 2 * lane] = ex2(lam + G0);       // sigma 2^G_i
                sc[SC_EG * 64 + 2 * lane + 1] = ex2(lam + G1);
                if (lane == 0) {
                    sc[SC_MISC * 64] = fold ? ex2(lam + glast) : 1.f;
                    sc[SC_MISC * 64 + 1] = ex2(lam_next);
                    sc[SC_MISC * 64 + 2] = ex2(lam);
                }
                lam = lam_next;
            }
            __syncwarp();
            if (!SUMMARY) {
                if (!pmma_wait()) break;   // P1 of this chunk; its barrier also publishes the scalars
                tc_fence_after();
                // C and sigma Qd overwrite what chunk n-1's S12 read
                if (!pwait(bar0 + B_WFREE, (n - 1) & 1, TAG_WFREE, n >= 1)) break;
                if (lq < 2) {
                    // ---- C rows i = lanes 0..63, this group's 32 columns j, tf32 K-major
                    const float* gam = sc + SC_GAM * 64;
                    const int i = 32 * lq + lane;
                    const float gi = gam[i];
                    uint8_t* ctile = sm + L::C0 + (n & 1) * 16384 + grp * 8192;
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        float sv[16];
                        tmem_ld16(t_row + TM_S + 32 * grp + 16 * hh, sv);
                        tmem_wait_ld();
                        uint32_t t[16];
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int j = 32 * grp + 16 * hh + jj;
                            t[jj] = tf32_bits((j <= i) ? ex2(gi - gam[j]) * sv[jj] : 0.f);
                        }
                        // columns 32 grp + 16 hh ..: tf32 block grp, 16-byte chunks 4 hh ..
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<uint4*>(ctile + sw128(i, 4 * hh + q)) =
                                make_uint4(t[4 * q], t[4 * q + 1], t[4 * q + 2], t[4 * q + 3]);
                    }
                } else {
                    // ---- sigma Qd = sigma 2^G_i q_i as tf32 K-major: row i, feature half kh
                    const int qt = (grp * 2 + (lq - 2)) * 32 + lane;
                    const int i = qt >> 1, kh = qt & 1;
                    const float egi = sc[SC_EG * 64 + i];
                    const uint8_t* src = sm + L::Q0 + qs * 16384 + kh * 8192;
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
                        // features 64 kh + 8 cc .. +7: kblock 2 kh + cc / 4 (rows 64.. of the
                        // S12 operand), chunks 2 (cc % 4) + {0, 1}
                        uint8_t* dst = sm + L::W + (kh * 2 + (cc >> 2)) * L::WQ_KB + 8192;
                        *reinterpret_cast<uint4*>(dst + sw128(i, (2 * cc) & 7)) = lo4;
                        *reinterpret_cast<uint4*>(dst + sw128(i, (2 * cc + 1) & 7)) = hi4;
                    }
                }
                fence_proxy_async();
                tc_fence_before();
                named_bar<2, kPrepThreads>();   // TM_S has been read; the q tile is consumed
                if (pt == 0) mbar_arrive(bar0 + B_QEMPTY + 8 * qs);
            }
            // ---- P2 (U^T into the parity's U buffer) and P3 (W^T into TM_S)
            if (!pwait(bar0 + B_AFULL + 8 * as, (n / AST) & 1, TAG_AFULL, true)) break;
            if (!pwait(bar0 + B_VFULL, n & 1, TAG_VFULL, need_v)) break;
            if (pt == 0) {
                tc_fence_after();
                if (need_v) {
#pragma unroll
                    for (int k16 = 0; k16 < 4; ++k16)
                        mma_ss<ID_P23>(t_u, desc_mn(base + L::V + k16 * 2048, 8192),
                                       desc_k(ast + k16 * 32), k16 > 0);
                }
#pragma unroll
                for (int k16 = 0; k16 < 4; ++k16)
                    mma_ss<ID_P23>(tmem + TM_S, desc_mn(kst + k16 * 2048, 8192),
                                   desc_k(ast + 8192 + k16 * 32), k16 > 0);
                if (need_v) mma_commit(bar0 + B_VEMPTY);
                mma_commit(bar0 + B_AEMPTY + 8 * as);
                mma_commit(bar0 + B_BARP);
            }
            __syncwarp();
            barp_pending = true;
            if (!SUMMARY) {
                // ---- while P2/P3 run: output rows of chunk n-2 (retired above), then zero its
                //      O^T buffer, which S12 of this chunk accumulates into
                tc_fence_after();
                if (n >= 2) store_output(n - 2);
                const uint32_t zero[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u,
                                           0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                tmem_st16(t_row + TM_U + (n & 1) * 128 + 64 + 32 * grp, zero);
                tmem_st16(t_row + TM_U + (n & 1) * 128 + 64 + 32 * grp + 16, zero);
                tmem_wait_st();
            }
            if (!pmma_wait()) break;
            tc_fence_after();
            // ---- -sigma W as rows 0..63 of the S12 B operand, once chunk n-1's S12 retired
            {
                if (SUMMARY && !pwait(bar0 + B_WFREE, (n - 1) & 1, TAG_WFREE, n >= 1)) break;
                const float nsig = -sc[SC_MISC * 64 + 2];
                // lane k of W^T's rows i: writes element (row i, feature k)
                const int k = 32 * lq + lane;
                uint8_t* col = sm + L::W + lq * L::WQ_KB + (k & 3) * 4;
                const int qk = (k & 31) >> 2;
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    float w[16];
                    tmem_ld16(t_row + TM_S + 32 * grp + 16 * hh, w);
                    tmem_wait_ld();
#pragma unroll
                    for (int ii = 0; ii < 16; ++ii)
                        *reinterpret_cast<uint32_t*>(col + sw128(32 * grp + 16 * hh + ii, qk)) =
                            tf32_bits(nsig * w[ii]);
                }
            }
            fence_proxy_async();
            tc_fence_before();
            named_bar<2, kPrepThreads>();
            // ---- TM_S is free again: P1 of the next chunk goes to the tensor pipe now
            if (!SUMMARY && n + 1 < nchunks) {
                const int n1 = n + 1;
                if (!pwait(bar0 + B_KFULL + 8 * (n1 % KST), (n1 / KST) & 1, TAG_KFULL, true)) break;
                if (!pwait(bar0 + B_QFULL + 8 * (n1 & 1), (n1 >> 1) & 1, TAG_QFULL, true)) break;
                issue_p1(n1);
            }
            if (pt == 0) mbar_arrive(bar0 + B_PREPDONE);
        }
#undef issue_p1
        if (*go == 0) {
            if (barp_pending && pt == 0) mbar_drain(bar0 + B_BARP, barp_phase, limit);
        } else if (!SUMMARY) {
            // ---- output rows of the last two chunks
#pragma unroll 1
            for (int m = (nchunks >= 2 ? nchunks - 2 : 0); m < nchunks; ++m) {
                if (!pwait(bar0 + B_UFREE + 8 * (m & 1), (m >> 1) & 1, TAG_UFREE, true)) break;
                tc_fence_after();
                store_output(m);
            }
        }
#undef store_output
#undef pmma_wait
#undef pwait
    } else {
        // ================================== state =================================
        const int st = tid;
        const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);
        volatile int* go = reinterpret_cast<volatile int*>(sm + L::BAR + B_GO_S);
        uint32_t bars_phase = 0;
        bool bars_pending = false;
        const long long bhoff = (long long)bh * kD * kD;
        float sig_next = 1.f;   // sigma after the last completed chunk

#define swait(bar, parity, tag)                                                              \
    group_wait<1, 128>(warp == 0, lane == 0, (bar), (parity), true, go, abort_flag, limit, \
                       c.err, (tag))
#define smma_wait() \
    (swait(bar0 + B_BARS, bars_phase, TAG_BARS) ? (bars_phase ^= 1u, bars_pending = false, true) : false)

        // ---- initial state: row `st` of H^T (= column st of H), sigma = 1
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
        named_bar<1, 128>();

        int done = 0;   // chunks completed
#pragma unroll 1
        for (int n = 0; n < nchunks; ++n) {
            const int ks = n % KST;
            const uint32_t kst = base + L::K0 + ks * 16384;
            const uint32_t t_u = tmem + TM_U + (n & 1) * L::TU_STRIDE;
            const uint32_t t_o = t_u + 64;   // forward only
            const float* sc = scal + (n & 1) * (SC_N * 64);
            if (!swait(bar0 + B_PREPDONE, n & 1, TAG_PREPDONE)) break;
            // ---- S12: [R^T | O^T] = [U^T | 0] + H_s^T [-sigma W ; sigma Qd]^T (forward);
            //      the summary forms only R^T = U^T + H_s^T (-sigma W)^T
            if (st == 0) {
                tc_fence_after();
                if (!SUMMARY) {
#pragma unroll
                    for (int k8 = 0; k8 < 16; ++k8)
                        mma_ts_tf32<ID_TF128>(t_u, tmem + TM_H + k8 * 8,
                                              desc_k(base + L::W + (k8 >> 2) * L::WQ_KB + (k8 & 3) * 32),
                                              1u);
                } else {
#pragma unroll
                    for (int k8 = 0; k8 < 16; ++k8)
                        mma_ts_tf32<ID_TF>(t_u, tmem + TM_H + k8 * 8,
                                           desc_k(base + L::W + (k8 >> 2) * L::WQ_KB + (k8 & 3) * 32),
                                           (need_v || k8 > 0) ? 1u : 0u);
                }
                mma_commit(bar0 + B_WFREE);
                mma_commit(bar0 + B_BARS);
            }
            __syncwarp();
            bars_pending = true;
            const float fold = sc[SC_MISC * 64];
            sig_next = sc[SC_MISC * 64 + 1];
            if (!smma_wait()) break;
            tc_fence_after();
            // ---- scaled R^T -> packed bf16 hi/lo in TMEM (and, rarely, fold sigma into H_s)
            {
                const float* dd = sc + SC_DD * 64;
                const uint32_t t_ur = t_row + TM_U + (n & 1) * L::TU_STRIDE;
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
                if (fold != 1.f) {
#pragma unroll 1
                    for (int g = 0; g < 8; ++g) {
                        float x[16];
                        uint32_t y[16];
                        tmem_ld16(t_row + TM_H + 16 * g, x);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j) y[j] = __float_as_uint(x[j] * fold);
                        tmem_st16(t_row + TM_H + 16 * g, y);
                    }
                }
                tmem_wait_st();
            }
            tc_fence_before();
            named_bar<1, 128>();
            // ---- S3: O^T += R^T C^T (A = R^T in TMEM) ; S4: H_s^T += (R^T D) K (A = hi, lo)
            if (st == 0) {
                tc_fence_after();
                if (!SUMMARY) {
                    const uint32_t cb = base + L::C0 + (n & 1) * 16384;
#pragma unroll
                    for (int k8 = 0; k8 < 8; ++k8)
                        mma_ts_tf32<ID_TF>(t_o, t_u + k8 * 8,
                                           desc_k(cb + (k8 >> 2) * 8192 + (k8 & 3) * 32), 1u);
                }
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int k16 = 0; k16 < 4; ++k16)
                        mma_ts_bf16<ID_S4>(tmem + TM_H, tmem + TM_RD + part * 32 + k16 * 8,
                                           desc_mn(kst + k16 * 2048, 8192), 1u);
                mma_commit(bar0 + B_KEMPTY + 8 * ks);
                mma_commit(bar0 + B_UFREE + 8 * (n & 1));
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
            // ---- the chain's final state H = sigma H_s: thread v writes column v of H
            float* dst = nullptr;
            if (SUMMARY) {
                const long long sb = ((long long)seg * c.B * c.H + bh) * kD * kD;
                dst = (blk == 0 ? c.M : c.S) + sb;
            } else if (c.h_final && seg == c.nseg_total - 1) {
                dst = c.h_final + bhoff;
            }
            if (dst) {
                const float sg = done > 0 ? sig_next : 1.f;
#pragma unroll 1
                for (int g = 0; g < 8; ++g) {
                    float x[16];
                    tmem_ld16(t_row + TM_H + 16 * g, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) dst[(long long)(16 * g + j) * kD + st] = sg * x[j];
                }
            }
        }
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
    constexpr uint32_t bytes = Smem<SUMMARY>::BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
    if (e != cudaSuccess) return e;
    const long long chains = (long long)c.B * c.H * c.nseg_run * (SUMMARY ? 2 : 1);
    kern<<<(unsigned)chains, kThreads, bytes, s>>>(tp);
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
