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
//       (forward: into the parity's O^T buffer, read out and zeroed before S12 runs there)
//   S12 [R^T | O^T] = [U^T | 0] + H_s^T [-sigma W ; sigma Qd]^T       kind::tf32, N = 128
//       (A = H_s^T from tensor memory; the summary has no O and runs the R^T half, N = 64)
//   S3  O^T += R^T C^T                     A = R^T from tensor memory   kind::tf32
//   S4  H_s^T += (R^T diag(2^(G_last - G) / sigma_next)) K, the scaled R^T held in tensor
//       memory as an unevaluated bf16 sum hi + lo (two MMAs).
// The fp32 state and the corrected values R never pass through bf16. Exponents are always
// differences of cumulative gates or bounded by the renormalisation.
//
// Warp roles (forward, 14 warps): warps 0-3 "state" (tensor-memory lanes 0..127: S12, S3,
// S4 issued by thread 0, the pack of R^T, final state); warps 4-11 "prep" (two warp groups,
// each covering lanes 0..127: gate cumsum and the sigma bookkeeping, the output rows of chunk
// n-2, C from Q K^T (the warps of lanes 0..63), sigma Qd, -sigma W); warp 12 issues the prep
// MMAs: P1 of chunk n once the C warps have read chunk n-1's Q K^T out of TM_S, P2 once chunk
// n-2 has retired its U buffer, P3 once the prep warps have stored chunk n-2's output rows
// from the O^T buffer P3 writes; warp 13 "producer" (TMA loads of the q/k/v tiles with
// 128-byte swizzle, bulk copies of the WY tiles, gates). The summary (16 warps) has two
// state groups (M part, S part), one prep group, the MMA warp for P2/P3, the producer, and
// one warp per state group that issues that group's S12 and S4 while the group only packs.
// Rings: k in KST stages (released by S4), q in two (released by prep), WY tiles in AST
// (released by P3), v in one (released by P2). Prep of chunk n+1 runs while the state group
// works on chunk n. Commits track the issuing thread's MMAs. Named barriers are the
// non-.aligned form: a group's leader warp diverges around its mbarrier poll. Every wait on
// an mbarrier is bounded: on expiry the kernel records GDN_ERR_TIMEOUT in the device error
// word, drains what it issued and frees tensor memory.
#include <algorithm>
#include <cstring>

#include "gdn_tc_common.cuh"

namespace gdn {
namespace {

constexpr int kD = 128;         // K == V
constexpr int kC = 64;          // tokens per chunk
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRenorm = -64.f;   // log2 of the smallest sigma kept without folding
// An fp32 value in tensor memory read as a tf32 MMA operand (H_s in S12, R^T in S3) loses its
// low 13 bits: it is truncated toward zero by 2^-11 / m of its magnitude on average (m in
// [1, 2) its mantissa), i.e. by 2^-11 / (2 ln 2) for mantissas spread log-uniformly. The B
// operand of each of those products is scaled by the inverse, so that the products carry no
// systematic bias; what remains is a zero-mean rounding error of at most 2^-11 of the operand.
// (S4 reads the scaled R^T as a bf16 hi + lo pair, which is accurate to 2^-16.)
constexpr float kTruncComp = 1.0f + 3.5222e-4f;

// Warps and tensor memory (32-bit cells, 128 lanes); one CTA per SM. The forward has one
// state warp group and two prep warp groups; a summary CTA carries both blocks of the
// augmented state -- the M part (from I, values 0) and the S part (from 0, values v) -- in
// two state warp groups fed by one prep group, which forms the shared W once per chunk.
template <bool SUMMARY>
struct Cfg {
    static constexpr int NSG = SUMMARY ? 2 : 1;              // state warp groups
    static constexpr int NGRP = SUMMARY ? 1 : 2;             // prep warp groups
    static constexpr int PREP_WARP0 = 4 * NSG;
    static constexpr int PREP_THREADS = 128 * NGRP;
    // one more warp issues the prep group's MMAs (P1 in the forward, P2, P3); in the summary
    // one warp per state group issues that group's MMAs (S12, S4)
    static constexpr int MMA_WARP = 4 * NSG + 4 * NGRP;
    static constexpr int PRODUCER_WARP = MMA_WARP + 1;
    static constexpr int ISSUE_WARP0 = PRODUCER_WARP + 1;
    static constexpr int THREADS = 32 * (ISSUE_WARP0 + (SUMMARY ? NSG : 0));
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TM_S = 0;    // forward: Q K^T; summary: W^T
    static constexpr uint32_t TM_U = 64;   // U^T -> R^T, two buffers by chunk parity; the
                                           // forward keeps W^T, then O^T right after each
                                           // (64 + 128 p)
    static constexpr int NUB = 2;                            // U buffers
    static constexpr uint32_t TU_STRIDE = SUMMARY ? 64 : 128;
    // scaled R^T packed as bf16 pairs, 16 tokens per 16 columns: hi in the first 8, lo in
    // the next 8. The forward keeps R^T for S3 and packs into its own 64 columns (TM_RD);
    // the summary (no S3) packs in place over R^T.
    static constexpr uint32_t TM_RD = 320;
    static constexpr uint32_t TM_RM = 192;   // summary: R^T of the M part (one buffer)
    // state master H_s^T (128 columns) of state group sg: forward 384; summary M 256, S 384
    __host__ __device__ static constexpr uint32_t tm_h(int sg) { return SUMMARY ? 256u + 128u * (uint32_t)sg : 384u; }
};

// Shared-memory map (bytes from a 1024-aligned base). A k, q or v tile is two 64-feature
// halves of 64 rows x 128 bytes (8 KB each, 128-byte swizzle); a WY stage holds the tile pair
// A diag(beta) | A diag(beta 2^Gx) as stored (kWyTileBytes each: the four MMA slabs of each
// factor, no zeros above the diagonal blocks).
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
    static constexpr uint32_t GATES = SCAL + 2 * 4 * 256;        // after scalars [parity 2][SC_N][64]
    static constexpr uint32_t BAR = GATES + KST * 256;           // gates [k stage][64]
    static constexpr uint32_t END = BAR + 512;
    static constexpr uint32_t BYTES = END + 1024;                // + alignment slack
    static_assert(BYTES <= 232448u, "shared memory budget");
};

// per-chunk scalar arrays (offsets in units of 64 floats within a parity block)
enum { SC_GAM = 0, SC_DD, SC_EG, SC_MISC, SC_N = 4 };
// SC_MISC slots: 0 = fold factor for the master (1 if none), 1 = sigma after the chunk,
// 2 = sigma during the chunk

// mbarrier slots and flags at Smem::BAR
constexpr uint32_t B_KFULL = 0, B_KEMPTY = 32, B_QFULL = 64, B_QEMPTY = 80, B_AFULL = 96,
                   B_AEMPTY = 112, B_VFULL = 128, B_VEMPTY = 136, B_BARP = 144, B_BARS = 152,
                   B_PREPDONE = 160, B_WFREE = 168, B_UFREE = 176, B_TMEM = 192, B_ABORT = 196,
                   B_GO_S = 200, B_GO_P = 204, B_BARS1 = 208, B_GO_S1 = 216, B_CDONE = 224,
                   B_WREAD = 232, B_MDRAIN = 240, B_SDRAIN = 248, B_S4 = 256, B_S4B = 264,
                   B_EPIDONE = 272, B_P1DONE = 280;

// wait tags recorded in the device error word's detail field
enum : unsigned {
    TAG_KFULL = 1, TAG_BARP = 2, TAG_BARS = 3, TAG_KEMPTY = 4, TAG_VEMPTY = 5, TAG_PREPDONE = 6,
    TAG_WFREE = 7, TAG_UFREE = 8, TAG_VFULL = 9, TAG_QFULL = 10, TAG_QEMPTY = 11,
    TAG_AFULL = 12, TAG_AEMPTY = 13, TAG_CDONE = 14, TAG_WREAD = 15, TAG_EPIDONE = 16,
    TAG_P1DONE = 17
};

struct TcParams {
    CUtensorMap tm_q;
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    ChainParams c;
    long long wait_limit;   // SM clock cycles before a wait gives up
};

// 32 token rows of one output column from a 64-column O^T buffer in tensor memory; rows from
// `valid` on (past the end of a varlen sequence) are not stored
template <bool OUT_BF16>
__device__ __forceinline__ void store_o_rows32(const ChainParams& c, uint32_t t_col, long long idx0,
                                               long long tok_stride, int valid) {
    float ov2[2][16];
    tmem_ld16(t_col, ov2[0]);
    tmem_ld16(t_col + 16, ov2[1]);
    tmem_wait_ld();
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        const float* ov = ov2[g];
        const long long base = idx0 + (long long)(16 * g) * tok_stride;
        if (OUT_BF16) {
            __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(c.o) + base;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (16 * g + j < valid) o[(long long)j * tok_stride] = __float2bfloat16_rn(ov[j]);
        } else {
            float* o = reinterpret_cast<float*>(c.o) + base;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (16 * g + j < valid) o[(long long)j * tok_stride] = ov[j];
        }
    }
}

// a state group (128 threads) and its issuer warp meet here once per chunk (named barriers 5
// and 6)
__device__ __forceinline__ void pack_bar(int sg) {
    if (sg == 0) named_bar<5, 160>();
    else named_bar<6, 160>();
}

// ------------------------------------------------------------------------------------
// the chain kernel
// ------------------------------------------------------------------------------------
// Registers are allocated to warps in groups of four: 15 or 16 warps count as 16, so at most
// 128 registers per thread.
// VARLEN: the chains are the packed sequences of c.cu_seqlens (forward only); the
// fixed-length instance has none of the end-of-sequence checks.
template <bool SUMMARY, bool VARLEN, bool OUT_BF16>
__device__ __forceinline__ void chain_body(const TcParams& p, const int chain) {
    using L = Smem<SUMMARY>;
    using F = Cfg<SUMMARY>;
    constexpr int KST = L::KST, AST = L::AST, NUB = F::NUB, NSG = F::NSG;
    constexpr uint32_t TM_S = F::TM_S, TM_U = F::TM_U, TM_RD = F::TM_RD;
    constexpr int kPrepThreads = F::PREP_THREADS;
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
    const int seg = c.seg_first + chain % c.nseg_run;
    const int bh = chain / c.nseg_run;
    const int b = bh / c.H, h = bh % c.H;
    // packed sequences cut into pieces: entry b of the piece table (the grid bounds the entries:
    // chains past this plan's count return at once -- in a grid launched as a programmatic
    // dependent, after waiting for its primary like its other chains)
    const int* pent = nullptr;
    if (VARLEN && c.piece_tab) {
        if (b >= __ldg(c.piece_n) || __ldg(c.piece_tab + kPieceFields * b + PF_SEQ) < 0) {
            if (SUMMARY || c.launch_dependent) asm volatile("griddepcontrol.wait;" ::: "memory");
            return;
        }
        pent = c.piece_tab + kPieceFields * b;
    }
    const int vseq = pent ? __ldg(pent + PF_SEQ) : b;         // the packed sequence
    const int vchunk0 = pent ? __ldg(pent + PF_CHUNK0) : 0;   // the piece's first chunk in it
    // tokens of this chain: a segment of the fixed-length batch, or a varlen sequence or piece
    // (whose last chunk may be partial: its padding tokens get g = 0 here and beta = 0 in the
    // WY tiles, which leaves the state untouched, and their outputs are not stored)
    // (fixed length: segment 0 may be longer or shorter than the others, see first_chunks)
    const int seg_chunks0 = c.first_chunks > 0 ? c.first_chunks : c.seg_len / kC;
    const int chunk0 = VARLEN || seg == 0 ? 0 : seg_chunks0 + (seg - 1) * (c.seg_len / kC);
    const int seq_tokens =
        VARLEN ? min(c.cu_seqlens[vseq + 1] - c.cu_seqlens[vseq] - vchunk0 * kC,
                     pent ? __ldg(pent + PF_NCHUNKS) * kC : (1 << 30))
               : (seg == 0 ? seg_chunks0 * kC : c.seg_len);
    const int nchunks = (seq_tokens + kC - 1) / kC;
    constexpr bool need_v = true;   // every CTA forms U (the forward, or the summary's S part)
    const long long limit = p.wait_limit;
    const long long tok_stride = (long long)c.H * kD;   // elements between two tokens of o
    const long long row_seg = VARLEN ? (long long)c.cu_seqlens[vseq] + (long long)vchunk0 * kC
                                     : (long long)b * c.T + (long long)chunk0 * kC;   // flattened (b, t)
    // the state the chain starts from and the one it ends in (null: zero, not kept), and where
    // a summary's M and S go
    const long long kv = (long long)kD * kD;
    const float* hstart = c.h_start ? c.h_start + seg * c.h_start_seg_stride + bh * kv : nullptr;
    float* hend = c.h_final && seg == c.nseg_total - 1 ? c.h_final + bh * kv : nullptr;
    float* msum = SUMMARY ? c.M + ((long long)seg * c.B * c.H + bh) * kv : nullptr;
    float* ssum = SUMMARY ? c.S + ((long long)seg * c.B * c.H + bh) * kv : nullptr;
    if (pent) {
        const int ps = __ldg(pent + PF_START), pe = __ldg(pent + PF_END), pm = __ldg(pent + PF_MS);
        const long long sh = (long long)vseq * c.H + h;   // the sequence's (s, h)
        hstart = ps >= 0 ? c.piece_states + ((long long)ps * c.H + h) * kv
                         : (c.h_start ? c.h_start + sh * kv : nullptr);
        hend = pe >= 0 ? c.piece_states + ((long long)pe * c.H + h) * kv
                       : (pe == -1 && c.h_final ? c.h_final + sh * kv : nullptr);
        if (SUMMARY) {
            msum = c.M + ((long long)pm * c.H + h) * kv;
            ssum = c.S + ((long long)pm * c.H + h) * kv;
        }
    }

    // A forward grid lets a grid launched after it as its programmatic dependent start right
    // away (the summaries that run beside the first piece's forward); a summary grid so
    // launched finishes only after its primary has (see the end of the kernel).
    if (!SUMMARY) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) {
        for (int i = 0; i < KST; ++i) {
            mbar_init(bar0 + B_KFULL + 8 * i, 2);
            mbar_init(bar0 + B_KEMPTY + 8 * i, NSG);   // each state group's S4 reads the k tile
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar0 + B_QFULL + 8 * i, 1);
            mbar_init(bar0 + B_QEMPTY + 8 * i, 1);
            mbar_init(bar0 + B_AFULL + 8 * i, 1);
            mbar_init(bar0 + B_AEMPTY + 8 * i, 1);
            mbar_init(bar0 + B_UFREE + 8 * i, NSG);
        }
        mbar_init(bar0 + B_VFULL, 1);
        mbar_init(bar0 + B_VEMPTY, 1);
        mbar_init(bar0 + B_BARP, 1);
        mbar_init(bar0 + B_BARS, 1);
        mbar_init(bar0 + B_BARS1, 1);
        mbar_init(bar0 + B_PREPDONE, 1);
        mbar_init(bar0 + B_WFREE, NSG);   // each state group's S1 reads -sigma W
        mbar_init(bar0 + B_CDONE, 1);
        mbar_init(bar0 + B_WREAD, 1);
        mbar_init(bar0 + B_MDRAIN, 1);
        mbar_init(bar0 + B_SDRAIN, NSG);   // each state group's last MMAs
        mbar_init(bar0 + B_S4, 1);         // S4 retired (state group 0's issuer)
        mbar_init(bar0 + B_S4B, 1);        // S4 retired (state group 1's issuer)
        mbar_init(bar0 + B_EPIDONE, 1);    // forward: the parity's O^T buffer has been read out
        mbar_init(bar0 + B_P1DONE, 1);     // forward: Q K^T is in TM_S
        *abort_flag = 0;
        *reinterpret_cast<volatile int*>(sm + L::BAR + B_GO_S) = 1;
        *reinterpret_cast<volatile int*>(sm + L::BAR + B_GO_S1) = 1;
        *reinterpret_cast<volatile int*>(sm + L::BAR + B_GO_P) = 1;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         bar0 + B_TMEM),
                     "r"(F::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == F::PRODUCER_WARP) {
        // ================================ producer ================================
        // The whole warp runs the loop (its lanes poll together and stay converged); lane 0
        // issues the copies, every lane loads two gates. The gates of chunk n+1 are loaded
        // into registers while chunk n's copies are in flight.
        // (the M part of a summary needs only the second factor)
        const uint32_t wy_bytes = need_v ? (uint32_t)kWyPairBytes : (uint32_t)kWyTileBytes;
        const uint8_t* wy_chain = reinterpret_cast<const uint8_t*>(c.wy) +
                                  (VARLEN ? (long long)h * c.total_chunks + c.cu_chunks[vseq] + vchunk0
                                          : (long long)bh * (c.T / kC) + chunk0) *
                                      kWyPairBytes;
        int k_last[KST], q_last[2] = {-1, -1}, a_last[2] = {-1, -1}, v_last = -1;
#pragma unroll
        for (int i = 0; i < KST; ++i) k_last[i] = -1;
        float gpre0 = 0.f, gpre1 = 0.f;
        if (nchunks > 0) {
            gpre0 = (!VARLEN || lane < seq_tokens) ? bf16_at(c.g, (row_seg + lane) * c.H + h) * kLog2e : 0.f;
            gpre1 = (!VARLEN || lane + 32 < seq_tokens) ? bf16_at(c.g, (row_seg + lane + 32) * c.H + h) * kLog2e : 0.f;
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
                const int t1 = (n + 1) * kC + lane;   // token index inside the chain
                gpre0 = (!VARLEN || t1 < seq_tokens) ? bf16_at(c.g, (row0 + kC + lane) * c.H + h) * kLog2e : 0.f;
                gpre1 = (!VARLEN || t1 + 32 < seq_tokens) ? bf16_at(c.g, (row0 + kC + lane + 32) * c.H + h) * kLog2e : 0.f;
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
                    const uint32_t skip = (uint32_t)kWyPairBytes - wy_bytes;
                    mbar_arrive_expect_tx(full, wy_bytes);
                    bulk_load(base + L::A0 + as * 16384 + skip,
                              wy_chain + (long long)n * kWyPairBytes + skip, wy_bytes, full);
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
    } else if (warp == F::MMA_WARP) {
        // ============================== prep MMA issue ============================
        // The prep group's tensor-core work, issued from here so that no prep thread stalls
        // behind an MMA issue. Forward, per chunk n: P2 (U^T into the parity's U buffer, once
        // chunk n-2 has retired it), P3 (W^T into TM_S, once the C warps have read Q K^T out of
        // it) and P1 of chunk n+1 ([Q ; -] K^T into TM_S, once the prep group has read W^T out
        // of it). Summary, per chunk n: P2 and P3 once the U buffer is retired and W^T of chunk
        // n-1 has been read out. Lane 0 issues; every wait is bounded.
        if (SUMMARY && lane == 0 && nchunks > 0) {
            auto ok = [&](uint32_t bar, uint32_t parity, unsigned tag) {
                return mbar_wait(bar, parity, abort_flag, limit, c.err, tag);
            };
#pragma unroll 1
            for (int n = 0; n < nchunks; ++n) {
                const int as = n % AST;
                const uint32_t kst = base + L::K0 + (n % KST) * 16384;
                const uint32_t ast = base + L::A0 + as * 16384;
                const uint32_t t_u = tmem + TM_U + (n % NUB) * F::TU_STRIDE;
                const bool run =
                    (n < NUB || ok(bar0 + B_UFREE + 8 * (n % NUB), ((n / NUB) - 1) & 1, TAG_UFREE)) &&
                    (n == 0 || ok(bar0 + B_WREAD, (n - 1) & 1, TAG_WREAD)) &&
                    ok(bar0 + B_KFULL + 8 * (n % KST), (n / KST) & 1, TAG_KFULL) &&
                    ok(bar0 + B_AFULL + 8 * as, (n / AST) & 1, TAG_AFULL) &&
                    ok(bar0 + B_VFULL, n & 1, TAG_VFULL);
                if (!run) break;
                tc_fence_after();
                wy_mma(t_u, base + L::V, ast);
                wy_mma(tmem + TM_S, kst, ast + kWyTileBytes);
                mma_commit(bar0 + B_VEMPTY);
                mma_commit(bar0 + B_AEMPTY + 8 * as);
                mma_commit(bar0 + B_BARP);
            }
            mma_commit(bar0 + B_MDRAIN);
            mbar_drain(bar0 + B_MDRAIN, 0, limit);
        }
        if (!SUMMARY && lane == 0 && nchunks > 0) {
            auto ok = [&](uint32_t bar, uint32_t parity, unsigned tag) {
                return mbar_wait(bar, parity, abort_flag, limit, c.err, tag);
            };
#pragma unroll 1
            for (int n = 0; n < nchunks; ++n) {
                const int as = n % AST;
                const uint32_t kst = base + L::K0 + (n % KST) * 16384;
                const uint32_t qst = base + L::Q0 + (n & 1) * 16384;
                const uint32_t ast = base + L::A0 + as * 16384;
                const uint32_t t_u = tmem + TM_U + (n % NUB) * F::TU_STRIDE;
                // P1: [Q ; -] K^T -> TM_S once the C warps have read chunk n-1's Q K^T out of
                // it; lanes 0..63 hold Q K^T (rows 64..127 of the A operand run into the next
                // buffer and are never read)
                bool run = (n == 0 || ok(bar0 + B_CDONE, (n - 1) & 1, TAG_CDONE)) &&
                           ok(bar0 + B_KFULL + 8 * (n % KST), (n / KST) & 1, TAG_KFULL) &&
                           ok(bar0 + B_QFULL + 8 * (n & 1), (n >> 1) & 1, TAG_QFULL);
                if (!run) break;
                tc_fence_after();
#pragma unroll
                for (int k16 = 0; k16 < 8; ++k16) {
                    const uint32_t off = (k16 >> 2) * 8192 + (k16 & 3) * 32;
                    mma_ss<ID_P1>(tmem + TM_S, desc_k(qst + off), desc_k(kst + off), k16 > 0);
                }
                mma_commit(bar0 + B_P1DONE);
                // P2: U^T into the parity's U buffer once chunk n-2 has retired it
                run = (n < NUB || ok(bar0 + B_UFREE + 8 * (n % NUB), ((n / NUB) - 1) & 1, TAG_UFREE)) &&
                      ok(bar0 + B_AFULL + 8 * as, (n / AST) & 1, TAG_AFULL) &&
                      ok(bar0 + B_VFULL, n & 1, TAG_VFULL);
                if (!run) break;
                tc_fence_after();
                wy_mma(t_u, base + L::V, ast);
                mma_commit(bar0 + B_VEMPTY);
                // P3: W^T into the parity's O^T buffer once the prep group has stored chunk
                // n-2's output rows from it (S12 of chunk n then accumulates O^T there)
                if (!(run = ok(bar0 + B_EPIDONE, n & 1, TAG_EPIDONE))) break;
                tc_fence_after();
                wy_mma(tmem + TM_U + (n & 1) * 128 + 64, kst, ast + kWyTileBytes);
                mma_commit(bar0 + B_AEMPTY + 8 * as);
                mma_commit(bar0 + B_BARP);   // covers P2 as well
            }
            // everything issued here retires before tensor memory is released
            mma_commit(bar0 + B_MDRAIN);
            mbar_drain(bar0 + B_MDRAIN, 0, limit);
        }
        __syncwarp();
    } else if (warp >= F::PREP_WARP0 && warp < F::MMA_WARP) {
        // ================================== prep ==================================
        const int pt = tid - 32 * F::PREP_WARP0, pw = warp - F::PREP_WARP0;
        const int grp = pw >> 2, lq = pw & 3;   // warp group; tensor-memory lane quarter
        constexpr int ECOLS = 64 / F::NGRP;      // W^T / O^T columns per warp group
        const uint32_t t_row = tmem + ((uint32_t)(lq * 32) << 16);   // this warp's TMEM lanes
        volatile int* go = reinterpret_cast<volatile int*>(sm + L::BAR + B_GO_P);
        uint32_t barp_phase = 0;   // one phase of B_BARP per chunk (P3 and P2 retired)
        float lam = 0.f;   // log2 sigma before the current chunk (prep warp pw 2)

        // the group's first warp waits (optionally) and publishes a verdict that all read
        // after the named barrier, so a timeout cannot split the group
#define pwait(bar, parity, tag, doit)                                                          \
    group_wait<2, kPrepThreads>(pw == 0, lane == 0, (bar), (parity), (doit), go, abort_flag, \
                                limit, c.err, (tag))
#define pmma_wait() \
    (pwait(bar0 + B_BARP, barp_phase, TAG_BARP, true) ? (barp_phase ^= 1u, true) : false)
// A warp waits on its own (all lanes poll together; lane 0's verdict is broadcast, so the
// warp stays uniform). If it gives up, the abort flag is up and the group stops at its next
// group wait.
#define warp_wait(bar, parity, abort_flag_, limit_, err_, tag, lane_, ...)                       \
    (__shfl_sync(0xffffffffu,                                                                 \
                 (int)(!(true __VA_OPT__(&& (__VA_ARGS__))) ||                                 \
                       mbar_wait((bar), (parity), (abort_flag_), (limit_), (err_), (tag))),    \
                 0) != 0)
// output rows of chunk m from its O^T buffer: lanes v, this warp group's 32 token columns
#define store_output(m)                                                                       \
    store_o_rows32<OUT_BF16>(c, t_row + TM_U + ((m) & 1) * 128 + 64 + 32 * grp,                \
                   ((row_seg + (long long)(m) * kC + 32 * grp) * c.H + h) * kD + 32 * lq + lane, \
                   tok_stride, VARLEN ? seq_tokens - ((m) * kC + 32 * grp) : 32)


#pragma unroll 1
        for (int n = 0; n < nchunks; ++n) {
            const int ks = n % KST, qs = n & 1;
            float* sc = scal + (n & 1) * (SC_N * 64);
            // chunk n-NUB is retired: its U/R (and in the forward O, C and scalar) buffers may
            // be reused
            if (!pwait(bar0 + B_UFREE + 8 * (n % NUB), ((n / NUB) - 1) & 1, TAG_UFREE, n >= NUB))
                break;
            // ---- gate cumsum, sigma bookkeeping and per-chunk scalars (first prep warp; the
            //      gates arrive with the chunk's k tile)
            // (warp pw 2: warp pw 0 may be busy issuing P2)
            const bool gates_ok =
                pw == 2 && __shfl_sync(0xffffffffu,
                                       (int)mbar_wait(bar0 + B_KFULL + 8 * ks, (n / KST) & 1,
                                                      abort_flag, limit, c.err, TAG_KFULL), 0);
            if (gates_ok) {
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
                // ---- every warp: its share of the output rows of chunk n-2 (retired above) from
                //      the parity's O^T buffer, which the MMA warp's P3 then reuses for W^T
                tc_fence_after();
                if (n >= 2) store_output(n - 2);
                tc_fence_before();
                named_bar<2, kPrepThreads>();   // the scalars are published, the O^T buffer read
                if (pt == 0) mbar_arrive(bar0 + B_EPIDONE);
                if (lq < 2) {
                    // ---- C rows i = lanes 0..63 (warps of lane quarters 0, 1), this group's 32
                    //      columns j, tf32 K-major; once every C warp has read Q K^T out of TM_S,
                    //      the MMA warp issues the next chunk's P1 into it
                    if (warp_wait(bar0 + B_P1DONE, n & 1, abort_flag, limit, c.err, TAG_P1DONE, lane)) {
                        tc_fence_after();
                        const float* gam = sc + SC_GAM * 64;
                        const int i = 32 * lq + lane;
                        const float gi = gam[i];
                        uint8_t* ctile = sm + L::C0 + (n & 1) * 16384 + grp * 8192;
                        float sv2[2][16];
                        tmem_ld16(t_row + TM_S + 32 * grp, sv2[0]);
                        tmem_ld16(t_row + TM_S + 32 * grp + 16, sv2[1]);
                        tmem_wait_ld();
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const float* sv = sv2[hh];
                            uint32_t t[16];
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) {
                                const int j = 32 * grp + 16 * hh + jj;
                                // (S3 reads R^T truncated: C carries kTruncComp)
                                t[jj] = tf32_operand((j <= i) ? ex2(gi - gam[j]) * (sv[jj] * kTruncComp) : 0.f);
                            }
                            // columns 32 grp + 16 hh ..: tf32 block grp, 16-byte chunks 4 hh ..
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                *reinterpret_cast<uint4*>(ctile + sw128(i, 4 * hh + q)) =
                                    make_uint4(t[4 * q], t[4 * q + 1], t[4 * q + 2], t[4 * q + 3]);
                        }
                    }
                    fence_proxy_async();
                    tc_fence_before();
                    named_bar<3, 128>();   // the C warps only
                    if (pt == 0) mbar_arrive(bar0 + B_CDONE);
                    __syncwarp();
                } else {
                    // ---- sigma Qd = sigma 2^G_i q_i as tf32 K-major: row i, feature half kh
                    // (the q tile's arrival is waited for here: P1 is the MMA warp's)
                    if (warp_wait(bar0 + B_WFREE, (n - 1) & 1, abort_flag, limit, c.err, TAG_WFREE,
                                  lane, n >= 1) &&
                        warp_wait(bar0 + B_QFULL + 8 * qs, (n >> 1) & 1, abort_flag, limit, c.err,
                                  TAG_QFULL, lane)) {
                        const int qt = (grp * 2 + (lq - 2)) * 32 + lane;
                        const int i = qt >> 1, kh = qt & 1;
                        const float egi = sc[SC_EG * 64 + i] * kTruncComp;   // S12 reads H_s truncated
                        const uint8_t* src = sm + L::Q0 + qs * 16384 + kh * 8192;
#pragma unroll 2
                        for (int cc = 0; cc < 8; ++cc) {
                            const uint4 u = *reinterpret_cast<const uint4*>(src + sw128(i, cc));
                            const uint4 lo4 = make_uint4(
                                tf32_operand(__uint_as_float(u.x << 16) * egi),
                                tf32_operand(__uint_as_float(u.x & 0xFFFF0000u) * egi),
                                tf32_operand(__uint_as_float(u.y << 16) * egi),
                                tf32_operand(__uint_as_float(u.y & 0xFFFF0000u) * egi));
                            const uint4 hi4 = make_uint4(
                                tf32_operand(__uint_as_float(u.z << 16) * egi),
                                tf32_operand(__uint_as_float(u.z & 0xFFFF0000u) * egi),
                                tf32_operand(__uint_as_float(u.w << 16) * egi),
                                tf32_operand(__uint_as_float(u.w & 0xFFFF0000u) * egi));
                            // features 64 kh + 8 cc .. +7: kblock 2 kh + cc / 4 (rows 64.. of the
                            // S12 operand), chunks 2 (cc % 4) + {0, 1}
                            uint8_t* dst = sm + L::W + (kh * 2 + (cc >> 2)) * L::WQ_KB + 8192;
                            *reinterpret_cast<uint4*>(dst + sw128(i, (2 * cc) & 7)) = lo4;
                            *reinterpret_cast<uint4*>(dst + sw128(i, (2 * cc + 1) & 7)) = hi4;
                        }
                    }
                }
                fence_proxy_async();   // sigma Qd and C are read by the state group's MMAs
            }
            // (the summary's P2 and P3 are the MMA warp's)
            if (!pmma_wait()) break;   // P3 (and P2) done; for the forward also every C and Qd
            tc_fence_after();
            // W^T: in TM_S (summary) or in the parity's O^T buffer (forward)
            const uint32_t t_w = t_row + (SUMMARY ? TM_S : TM_U + (n & 1) * 128 + 64) + ECOLS * grp;
            // ---- -sigma W as rows 0..63 of the S12 B operand, once chunk n-1's S12 retired
            //      (the forward's Qd warps waited for that before the barrier above)
            {
                if (SUMMARY && !pwait(bar0 + B_WFREE, (n - 1) & 1, TAG_WFREE, n >= 1)) break;
                const float nsig = -sc[SC_MISC * 64 + 2] * kTruncComp;   // S12 reads H_s truncated
                // lane k of W^T's rows i: writes element (row i, feature k)
                const int k = 32 * lq + lane;
                uint8_t* col = sm + L::W + lq * L::WQ_KB + (k & 3) * 4;
                const int qk = (k & 31) >> 2;
#pragma unroll 1
                for (int hb = 0; hb < ECOLS; hb += 32) {
                    float w2[2][16];
                    tmem_ld16(t_w + hb, w2[0]);
                    tmem_ld16(t_w + hb + 16, w2[1]);
                    tmem_wait_ld();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const float* w = w2[hh];
#pragma unroll
                        for (int ii = 0; ii < 16; ++ii)
                            *reinterpret_cast<uint32_t*>(
                                col + sw128(ECOLS * grp + hb + 16 * hh + ii, qk)) =
                                tf32_operand(nsig * w[ii]);
                    }
                }
                if (!SUMMARY) {
                    // the forward's S12 accumulates this chunk's O^T from zero here
                    const uint32_t zero[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u,
                                               0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                    tmem_st16(t_w, zero);
                    tmem_st16(t_w + 16, zero);
                    tmem_wait_st();
                }
            }
            fence_proxy_async();
            tc_fence_before();
            named_bar<2, kPrepThreads>();
            // ---- the chunk is ready for the state group; in the forward the q tile is consumed
            //      (P1 and sigma Qd); in the summary TM_S is free again for the next P3
            if (pt == 0) {
                mbar_arrive(bar0 + B_PREPDONE);
                if (!SUMMARY) mbar_arrive(bar0 + B_QEMPTY + 8 * qs);
                else mbar_arrive(bar0 + B_WREAD);
            }
        }
        if (*go == 0) {
            // (the prep MMAs are the MMA warp's, which lets them retire itself)
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
#undef warp_wait
#undef pmma_wait
#undef pwait
    } else if (warp >= F::THREADS / 32) {
        // warps of a wider launch (the forward's CTAs of the combined first-phase grid): idle
    } else if (SUMMARY && warp >= F::ISSUE_WARP0) {
        if constexpr (SUMMARY) {
        // ========================= state MMA issue (summary) =========================
        // One warp per state group issues that group's tensor-core work, so that no thread
        // that packs R^T stalls behind an MMA issue: per chunk n, S12 once the prep group's
        // operands are in place and S4 of chunk n-1 has updated H_s, then S4 once the group
        // has packed R^T (a named barrier with the group). Both sides pass that barrier
        // exactly once per chunk (and once for the initial state) whatever happens, so a
        // wait that gives up cannot strand the other side; after one, nothing more is
        // issued. Lane 0 issues; the warp polls together. (The forward's state group issues
        // its own MMAs: there the prep group, not the state group, sets the pace.)
        const int sg = warp - F::ISSUE_WARP0;
        const bool m_part = SUMMARY && sg == 0;
        const uint32_t tm_h = F::tm_h(sg);
        const uint32_t bar_s = bar0 + (sg == 0 ? B_BARS : B_BARS1);
        const uint32_t bar_4 = bar0 + (sg == 0 ? B_S4 : B_S4B);
        auto wwait = [&](uint32_t bar, uint32_t parity, unsigned tag) {
            const bool r = mbar_wait(bar, parity, abort_flag, limit, c.err, tag);
            return __shfl_sync(0xffffffffu, (int)r, 0) != 0;
        };
        tc_fence_before();
        pack_bar(sg);   // the initial state is in tensor memory
        bool ok = true;
#pragma unroll 1
        for (int n = 0; n < nchunks; ++n) {
            const int ks = n % KST;
            const uint32_t kst = base + L::K0 + ks * 16384;
            const uint32_t tu_col = m_part ? F::TM_RM : TM_U + (n % NUB) * F::TU_STRIDE;
            const uint32_t t_u = tmem + tu_col;
            ok = ok && wwait(bar0 + B_PREPDONE, n & 1, TAG_PREPDONE) &&
                 (n == 0 || wwait(bar_4, (n - 1) & 1, TAG_BARS));
            // ---- S12: R^T = U^T + H_s^T (-sigma W)^T (no U in the M part)
            if (ok && lane == 0) {
                tc_fence_after();
#pragma unroll
                for (int k8 = 0; k8 < 16; ++k8)
                    mma_ts_tf32<ID_TF>(t_u, tmem + tm_h + k8 * 8,
                                       desc_k(base + L::W + (k8 >> 2) * L::WQ_KB + (k8 & 3) * 32),
                                       (!m_part || k8 > 0) ? 1u : 0u);
                mma_commit(bar0 + B_WFREE);
                mma_commit(bar_s);
            }
            __syncwarp();
            pack_bar(sg);   // the group has packed the scaled R^T (in place)
            // ---- S4: H_s^T += (R^T D) K (A = hi, lo in TMEM)
            if (ok && lane == 0) {
                tc_fence_after();
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int k16 = 0; k16 < 4; ++k16)
                        mma_ts_bf16<ID_S4>(tmem + tm_h, tmem + tu_col + 16 * k16 + 8 * part,
                                           desc_mn(kst + k16 * 2048, 8192), 1u);
                mma_commit(bar0 + B_KEMPTY + 8 * ks);
                mma_commit(bar0 + B_UFREE + 8 * (n % NUB));
                mma_commit(bar_4);
            }
            __syncwarp();
        }
        // every MMA issued here retires before the final state is read out or tensor memory
        // is released (the state group waits for this, or drains it)
        if (lane == 0) mma_commit(bar0 + B_SDRAIN);
        __syncwarp();
        }
    } else if constexpr (SUMMARY) {
        // ================================== state =================================
        // summary state group sg: the M part (0) or the S part (1). Per chunk: wait for S12,
        // pack the scaled R^T in place, hand it to the group's issuer warp.
        const int sg = SUMMARY ? (warp >> 2) : 0;
        const int st = tid & 127;                      // = column of H this thread owns
        const uint32_t t_row = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t tm_h = F::tm_h(sg);
        const uint32_t bar_s = bar0 + (sg == 0 ? B_BARS : B_BARS1);
        volatile int* go = reinterpret_cast<volatile int*>(sm + L::BAR + (sg == 0 ? B_GO_S : B_GO_S1));
        const bool m_part = SUMMARY && sg == 0;       // starts from I, no values
        uint32_t bars_phase = 0;
        const long long bhoff = (long long)bh * kD * kD;
        float sig_next = 1.f;   // sigma after the last completed chunk

// each state group synchronises its waits on its own named barrier (1 or 4)
#define swait(bar, parity, tag)                                                                  \
    (sg == 0 ? group_wait<1, 128>(warp == 0, lane == 0, (bar), (parity), true, go, abort_flag,   \
                                  limit, c.err, (tag))                                           \
             : group_wait<4, 128>(warp == 4, lane == 0, (bar), (parity), true, go, abort_flag,   \
                                  limit, c.err, (tag)))

        // ---- initial state: row `st` of H^T (= column st of H), sigma = 1 (a forward grid
        // launched as a programmatic dependent reads it only once its primary has completed)
        if (!SUMMARY && c.launch_dependent) asm volatile("griddepcontrol.wait;" ::: "memory");
#pragma unroll 1
        for (int g = 0; g < 8; ++g) {
            uint32_t x[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int k = 16 * g + j;
                float v0 = 0.f;
                if (SUMMARY)
                    v0 = (m_part && k == st) ? 1.f : 0.f;
                else if (hstart)
                    v0 = hstart[(long long)k * kD + st];
                x[j] = __float_as_uint(v0);
            }
            tmem_st16(t_row + tm_h + 16 * g, x);
        }
        tmem_wait_st();
        tc_fence_before();
        pack_bar(sg);

        bool live = true;   // uniform over the group
        int done = 0;       // chunks completed
#pragma unroll 1
        for (int n = 0; n < nchunks; ++n) {
            // R^T buffer: the summary's M part has its own; otherwise the parity's U buffer
            const uint32_t tu_col = m_part ? F::TM_RM : TM_U + (n % NUB) * F::TU_STRIDE;
            const float* sc = scal + (n & 1) * (SC_N * 64);
            // the chunk's scalars are published with PREPDONE; S12 retires after it
            live = live && swait(bar0 + B_PREPDONE, n & 1, TAG_PREPDONE);
            float fold = 1.f;
            if (live) {
                fold = sc[SC_MISC * 64];
                sig_next = sc[SC_MISC * 64 + 1];
            }
            live = live && swait(bar_s, bars_phase, TAG_BARS);
            bars_phase ^= 1u;
            if (live) {
                tc_fence_after();
                // ---- scaled R^T -> packed bf16 hi/lo in TMEM (and, rarely, fold sigma into H_s)
                const uint32_t rd_col = tu_col;   // packed in place
                {
                    const float* dd = sc + SC_DD * 64;
                    const uint32_t t_ur = t_row + tu_col;
#pragma unroll 1
                    for (int g2 = 0; g2 < 4; g2 += 2) {
                      float r2[2][16];
                      tmem_ld16(t_ur + 16 * g2, r2[0]);
                      tmem_ld16(t_ur + 16 * g2 + 16, r2[1]);
                      tmem_wait_ld();
#pragma unroll
                      for (int gg = 0; gg < 2; ++gg) {
                        const int g = g2 + gg;
                        const float* r = r2[gg];
                        // packed column q holds the pair (2q, 2q+1) of the 64 tokens j
                        uint32_t hi[8], lo[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float2 d2 = *reinterpret_cast<const float2*>(dd + 16 * g + 2 * j);
                            const float x0 = r[2 * j] * d2.x;
                            const float x1 = r[2 * j + 1] * d2.y;
                            // hi = x truncated to bf16 (its top 16 bits), lo = the exact remainder
                            // truncated to bf16: hi + lo is within 2^-16 |x| of x. Integer and
                            // byte-permute operations only, no conversions.
                            const uint32_t b0 = __float_as_uint(x0), b1 = __float_as_uint(x1);
                            hi[j] = __byte_perm(b0, b1, 0x7632);
                            const float l0 = x0 - __uint_as_float(b0 & 0xFFFF0000u);
                            const float l1 = x1 - __uint_as_float(b1 & 0xFFFF0000u);
                            lo[j] = __byte_perm(__float_as_uint(l0), __float_as_uint(l1), 0x7632);
                        }
                        // (in the summary this overwrites the 16 columns just read)
                        tmem_st8(t_row + rd_col + 16 * g, hi);
                        tmem_st8(t_row + rd_col + 16 * g + 8, lo);
                      }
                    }
                    if (fold != 1.f) {
#pragma unroll 1
                        for (int g = 0; g < 8; ++g) {
                            float x[16];
                            uint32_t y[16];
                            tmem_ld16(t_row + tm_h + 16 * g, x);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 16; ++j) y[j] = __float_as_uint(x[j] * fold);
                            tmem_st16(t_row + tm_h + 16 * g, y);
                        }
                    }
                    tmem_wait_st();
                }
                done = n + 1;
            }
            tc_fence_before();
            pack_bar(sg);   // the issuer's S4 reads the packed R^T
        }

        // every MMA the group's issuer issued (the last S4) completes before the final state
        // is read out or tensor memory is released
        const bool drained = live && swait(bar0 + B_SDRAIN, 0, TAG_BARS);
        if (!drained) {
            if (st == 0) mbar_drain(bar0 + B_SDRAIN, 0, limit);
        } else {
            tc_fence_after();
            // ---- the chain's final state H = sigma H_s: thread v writes column v of H
            float* dst = SUMMARY ? (m_part ? msum : ssum) : hend;
            // the forward may also hand its final state to the next segment
            float* dst2 = (!SUMMARY && c.h_out) ? c.h_out + (seg + 1) * c.h_out_seg_stride + bhoff : nullptr;
            if (dst || dst2) {
                const float sgm = done > 0 ? sig_next : 1.f;
#pragma unroll 1
                for (int g = 0; g < 8; ++g) {
                    float x[16];
                    tmem_ld16(t_row + tm_h + 16 * g, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const long long idx = (long long)(16 * g + j) * kD + st;
                        if (dst) dst[idx] = sgm * x[j];
                        if (dst2) dst2[idx] = sgm * x[j];
                    }
                }
            }
        }
#undef swait
    } else {
        // ================================== state =================================
        // state group sg: the forward's only group, or the summary's M part (0) / S part (1)
        const int sg = SUMMARY ? (warp >> 2) : 0;
        const int st = tid & 127;                      // = column of H this thread owns
        const uint32_t t_row = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t tm_h = F::tm_h(sg);
        const uint32_t bar_s = bar0 + (sg == 0 ? B_BARS : B_BARS1);
        volatile int* go = reinterpret_cast<volatile int*>(sm + L::BAR + (sg == 0 ? B_GO_S : B_GO_S1));
        const bool m_part = SUMMARY && sg == 0;       // starts from I, no values
        uint32_t bars_phase = 0;
        bool bars_pending = false;
        uint32_t s4_parity = 0;    // bar_s phase of the last S4 (issuing thread)
        bool s4_pending = false;
        const long long bhoff = (long long)bh * kD * kD;
        float sig_next = 1.f;   // sigma after the last completed chunk

// each state group synchronises on its own named barrier (1 or 4)
#define sbar()                                   \
    do {                                         \
        if (sg == 0) named_bar<1, 128>();        \
        else named_bar<4, 128>();                \
    } while (0)
#define swait(bar, parity, tag)                                                                  \
    (sg == 0 ? group_wait<1, 128>(warp == 0, lane == 0, (bar), (parity), true, go, abort_flag,   \
                                  limit, c.err, (tag))                                           \
             : group_wait<4, 128>(warp == 4, lane == 0, (bar), (parity), true, go, abort_flag,   \
                                  limit, c.err, (tag)))
#define smma_wait() \
    (swait(bar_s, bars_phase, TAG_BARS) ? (bars_phase ^= 1u, bars_pending = false, true) : false)

        // ---- initial state: row `st` of H^T (= column st of H), sigma = 1 (a forward grid
        // launched as a programmatic dependent reads it only once its primary has completed)
        if (!SUMMARY && c.launch_dependent) asm volatile("griddepcontrol.wait;" ::: "memory");
#pragma unroll 1
        for (int g = 0; g < 8; ++g) {
            uint32_t x[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int k = 16 * g + j;
                float v0 = 0.f;
                if (SUMMARY)
                    v0 = (m_part && k == st) ? 1.f : 0.f;
                else if (hstart)
                    v0 = hstart[(long long)k * kD + st];
                x[j] = __float_as_uint(v0);
            }
            tmem_st16(t_row + tm_h + 16 * g, x);
        }
        tmem_wait_st();
        tc_fence_before();
        sbar();

        int done = 0;   // chunks completed
#pragma unroll 1
        for (int n = 0; n < nchunks; ++n) {
            const int ks = n % KST;
            const uint32_t kst = base + L::K0 + ks * 16384;
            // R^T buffer: the summary's M part has its own; otherwise the parity's U buffer
            const uint32_t tu_col = m_part ? F::TM_RM : TM_U + (n % NUB) * F::TU_STRIDE;
            const uint32_t t_u = tmem + tu_col;
            const uint32_t t_o = t_u + 64;   // forward only
            const float* sc = scal + (n & 1) * (SC_N * 64);
            // ---- the state entering this chunk, when an API segment starts here (the pieces
            //      a sequence is cut into need not start at segment starts): H = sigma H_s
            //      once the previous chunk's S4 has retired; thread v writes column v
            if (!VARLEN && c.H_seg && (chunk0 + n) % c.seg_chunks == 0) {
                if (s4_pending && !swait(bar_s, s4_parity, TAG_BARS)) break;
                s4_pending = false;
                tc_fence_after();
                float* dst = c.H_seg + (long long)((chunk0 + n) / c.seg_chunks) * c.B * c.H * kD * kD + bhoff;
#pragma unroll 1
                for (int g = 0; g < 8; ++g) {
                    float x[16];
                    tmem_ld16(t_row + tm_h + 16 * g, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) dst[(long long)(16 * g + j) * kD + st] = sig_next * x[j];
                }
            }
            if (!swait(bar0 + B_PREPDONE, n & 1, TAG_PREPDONE)) break;
            // the previous chunk's S4 has updated H_s (the issuing thread waits; if it gives up
            // it raises the abort flag, issues nothing, and the group stops at its next wait)
            const bool s4_ok = st != 0 || !s4_pending ||
                               mbar_wait(bar_s, s4_parity, abort_flag, limit, c.err, TAG_BARS);
            s4_pending = false;
            // ---- S12: [R^T | O^T] = [U^T | 0] + H_s^T [-sigma W ; sigma Qd]^T (forward);
            //      the summary forms only R^T = U^T + H_s^T (-sigma W)^T (no U in the M part)
            if (st == 0 && s4_ok) {
                tc_fence_after();
                if (!SUMMARY) {
#pragma unroll
                    for (int k8 = 0; k8 < 16; ++k8)
                        mma_ts_tf32<ID_TF128>(t_u, tmem + tm_h + k8 * 8,
                                              desc_k(base + L::W + (k8 >> 2) * L::WQ_KB + (k8 & 3) * 32),
                                              1u);
                } else {
#pragma unroll
                    for (int k8 = 0; k8 < 16; ++k8)
                        mma_ts_tf32<ID_TF>(t_u, tmem + tm_h + k8 * 8,
                                           desc_k(base + L::W + (k8 >> 2) * L::WQ_KB + (k8 & 3) * 32),
                                           (!m_part || k8 > 0) ? 1u : 0u);
                }
                mma_commit(bar0 + B_WFREE);
                mma_commit(bar_s);
            }
            __syncwarp();
            bars_pending = true;
            const float fold = sc[SC_MISC * 64];
            sig_next = sc[SC_MISC * 64 + 1];
            if (!smma_wait()) break;
            tc_fence_after();
            // ---- scaled R^T -> packed bf16 hi/lo in TMEM (and, rarely, fold sigma into H_s)
            const uint32_t rd_col = SUMMARY ? tu_col : TM_RD;
            {
                const float* dd = sc + SC_DD * 64;
                const uint32_t t_ur = t_row + tu_col;
#pragma unroll 1
                for (int g2 = 0; g2 < 4; g2 += 2) {
                  float r2[2][16];
                  tmem_ld16(t_ur + 16 * g2, r2[0]);
                  tmem_ld16(t_ur + 16 * g2 + 16, r2[1]);
                  tmem_wait_ld();
#pragma unroll
                  for (int gg = 0; gg < 2; ++gg) {
                    const int g = g2 + gg;
                    const float* r = r2[gg];
                    // packed column q holds the pair (2q, 2q+1) of the 64 tokens j
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float2 d2 = *reinterpret_cast<const float2*>(dd + 16 * g + 2 * j);
                        const float x0 = r[2 * j] * d2.x;
                        const float x1 = r[2 * j + 1] * d2.y;
                        // hi = x truncated to bf16 (its top 16 bits), lo = the exact remainder
                        // truncated to bf16: hi + lo is within 2^-16 |x| of x. Integer and
                        // byte-permute operations only, no conversions.
                        const uint32_t b0 = __float_as_uint(x0), b1 = __float_as_uint(x1);
                        hi[j] = __byte_perm(b0, b1, 0x7632);
                        const float l0 = x0 - __uint_as_float(b0 & 0xFFFF0000u);
                        const float l1 = x1 - __uint_as_float(b1 & 0xFFFF0000u);
                        lo[j] = __byte_perm(__float_as_uint(l0), __float_as_uint(l1), 0x7632);
                    }
                    // (in the summary this overwrites the 16 columns just read)
                    tmem_st8(t_row + rd_col + 16 * g, hi);
                    tmem_st8(t_row + rd_col + 16 * g + 8, lo);
                  }
                }
                if (fold != 1.f) {
#pragma unroll 1
                    for (int g = 0; g < 8; ++g) {
                        float x[16];
                        uint32_t y[16];
                        tmem_ld16(t_row + tm_h + 16 * g, x);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j) y[j] = __float_as_uint(x[j] * fold);
                        tmem_st16(t_row + tm_h + 16 * g, y);
                    }
                }
                tmem_wait_st();
            }
            // ---- S3 O^T += R^T C^T (A = R^T in TMEM), issued once this warp has packed (the
            //      issuing thread stalls while the tensor pipe takes the MMAs; before the pack
            //      that stall would hold back the pack and with it S4)
            if (st == 0) {
                const uint32_t cb = base + L::C0 + (n & 1) * 16384;
#pragma unroll
                for (int k8 = 0; k8 < 8; ++k8)
                    mma_ts_tf32<ID_TF>(t_o, t_u + k8 * 8,
                                       desc_k(cb + (k8 >> 2) * 8192 + (k8 & 3) * 32), 1u);
            }
            __syncwarp();
            tc_fence_before();
            sbar();
            // ---- S4: H_s^T += (R^T D) K (A = hi, lo in TMEM); its commits also cover S3. Only
            //      the issuing thread waits for it, just before it issues the next chunk's S12
            //      (which reads H_s); the rest of the group goes on to the next chunk.
            if (st == 0) {
                tc_fence_after();
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int k16 = 0; k16 < 4; ++k16)
                        mma_ts_bf16<ID_S4>(tmem + tm_h, tmem + rd_col + 16 * k16 + 8 * part,
                                           desc_mn(kst + k16 * 2048, 8192), 1u);
                mma_commit(bar0 + B_KEMPTY + 8 * ks);
                mma_commit(bar0 + B_UFREE + 8 * (n % NUB));
                mma_commit(bar_s);
            }
            __syncwarp();
            s4_parity = bars_phase;   // the phase S4 completes
            s4_pending = true;
            bars_phase ^= 1u;
            done = n + 1;
        }

        // every MMA this group issued (the last S4) completes before the final state is read
        // out or tensor memory is released
        if (st == 0) mma_commit(bar0 + B_SDRAIN);
        __syncwarp();
        const bool drained = *go != 0 && swait(bar0 + B_SDRAIN, 0, TAG_BARS);
        if (!drained) {
            if (st == 0) mbar_drain(bar0 + B_SDRAIN, 0, limit);
        } else {
            tc_fence_after();
            // ---- the chain's final state H = sigma H_s: thread v writes column v of H
            float* dst = SUMMARY ? (m_part ? msum : ssum) : hend;
            // the forward may also hand its final state to the next segment
            float* dst2 = (!SUMMARY && c.h_out) ? c.h_out + (seg + 1) * c.h_out_seg_stride + bhoff : nullptr;
            if (dst || dst2) {
                const float sgm = done > 0 ? sig_next : 1.f;
#pragma unroll 1
                for (int g = 0; g < 8; ++g) {
                    float x[16];
                    tmem_ld16(t_row + tm_h + 16 * g, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const long long idx = (long long)(16 * g + j) * kD + st;
                        if (dst) dst[idx] = sgm * x[j];
                        if (dst2) dst2[idx] = sgm * x[j];
                    }
                }
            }
        }
#undef sbar
#undef smma_wait
#undef swait
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(F::TMEM_COLS)
                     : "memory");
    // a grid launched as a programmatic dependent completes after its primary grid (a no-op
    // otherwise), so the launches that follow it in the stream see both finished
    if (SUMMARY || c.launch_dependent) asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <bool SUMMARY, bool VARLEN, bool OUT_BF16>
__global__ void __launch_bounds__(512, 1) tc_chain_kernel(const __grid_constant__ TcParams p) {
    chain_body<SUMMARY, VARLEN, OUT_BF16>(p, blockIdx.x);
}

// The first phase of the segmented forward as one grid: CTAs 0 .. nf-1 run the first piece's
// forward, the others the summaries of the pieces beside it. (The two kinds stay in contiguous
// blocks of CTAs: alternated over the grid, they took twice as long, measured at the bench
// workload.) Every CTA lets a programmatic dependent of the grid start at once (on the SMs the
// chains leave free).
struct TcPhase1Params {
    TcParams f;
    TcParams s;
    int nf;
};

template <bool OUT_BF16>
__global__ void __launch_bounds__(512, 1) tc_phase1_kernel(const __grid_constant__ TcPhase1Params p) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if ((int)blockIdx.x < p.nf) chain_body<false, false, OUT_BF16>(p.f, blockIdx.x);
    else chain_body<true, false, false>(p.s, (int)blockIdx.x - p.nf);
}

// ------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------
template <bool SUMMARY>
bool make_params(const ChainParams& c, TcParams* tp) {
    memset(tp, 0, sizeof(*tp));
    tp->c = c;
    tp->wait_limit = 4000000000LL;   // ~2 s at GB300 clocks
    if (!make_map(&tp->tm_k, c.k, c)) return false;
    if (!SUMMARY && !make_map(&tp->tm_q, c.q, c)) return false;
    return make_map(&tp->tm_v, c.v, c);
}

template <bool SUMMARY>
cudaError_t launch(const ChainParams& c, cudaStream_t s) {
    // (a summary over packed sequences: their pieces, from a piece table)
    if (!c.wy || (SUMMARY && c.cu_seqlens && !c.piece_tab)) return cudaErrorInvalidValue;
    TcParams tp;
    if (!make_params<SUMMARY>(c, &tp)) return cudaErrorInvalidValue;
    // one instance per output type and packing, so that each carries only its own store path
    void (*kern)(TcParams) = tc_chain_kernel<SUMMARY, false, false>;
    if constexpr (SUMMARY) {
        if (c.cu_seqlens) kern = tc_chain_kernel<true, true, false>;
    } else {
        if (c.cu_seqlens)
            kern = c.out_bf16 ? tc_chain_kernel<false, true, true> : tc_chain_kernel<false, true, false>;
        else if (c.out_bf16)
            kern = tc_chain_kernel<false, false, true>;
    }
    constexpr uint32_t bytes = Smem<SUMMARY>::BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
    if (e != cudaSuccess) return e;
    const long long chains = (long long)c.B * c.H * c.nseg_run;
    if (!c.launch_dependent) {
        kern<<<(unsigned)chains, Cfg<SUMMARY>::THREADS, bytes, s>>>(tp);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)chains);
    cfg.blockDim = dim3(Cfg<SUMMARY>::THREADS);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tp);
}

cudaError_t launch_phase1(const ChainParams& f, const ChainParams& sm, cudaStream_t s) {
    if (!f.wy || !sm.wy || f.cu_seqlens || sm.cu_seqlens) return cudaErrorInvalidValue;
    TcPhase1Params pp;
    if (!make_params<false>(f, &pp.f) || !make_params<true>(sm, &pp.s)) return cudaErrorInvalidValue;
    const long long nf = (long long)f.B * f.H * f.nseg_run;
    const long long ns = (long long)sm.B * sm.H * sm.nseg_run;
    if (nf + ns >= (1LL << 31)) return cudaErrorInvalidValue;
    pp.nf = (int)nf;
    void (*kern)(TcPhase1Params) = f.out_bf16 ? tc_phase1_kernel<true> : tc_phase1_kernel<false>;
    constexpr uint32_t bytes = std::max(Smem<false>::BYTES, Smem<true>::BYTES);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes);
    if (e != cudaSuccess) return e;
    static_assert(Cfg<false>::THREADS <= Cfg<true>::THREADS, "the summary is the wider CTA");
    kern<<<(unsigned)(nf + ns), Cfg<true>::THREADS, bytes, s>>>(pp);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(const ChainParams& p) {
    return p.in_bf16 && p.K == kD && p.V == kD && !p.gate_k &&
           (p.cu_seqlens || (p.seg_len > 0 && p.seg_len % kC == 0)) && encode_fn() != nullptr;
}

bool tc_runtime_ok() { return encode_fn() != nullptr; }

namespace {
// One CTA waits, the way every chain kernel waits, on an mbarrier that nothing arrives at, with
// a wait limit of `limit` SM cycles: the wait gives up, records GDN_ERR_TIMEOUT with `tag` in
// the device error word and the kernel returns (a check of the failure path; the context
// stays usable).
__global__ void wait_selftest_kernel(DeviceError* err, long long limit, unsigned tag) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x < 32) {   // one warp polls together, as the kernels' leader warps do
        const bool ok = mbar_wait(b, 0, &abort_flag, limit, err, tag);
        if (ok && threadIdx.x == 0) record_error(err, GDN_ERR_CUDA, tag);   // cannot happen
    }
    __syncthreads();
}
}  // namespace

cudaError_t launch_wait_selftest(DeviceError* err, long long limit, unsigned tag, cudaStream_t s) {
    wait_selftest_kernel<<<1, 64, 0, s>>>(err, limit, tag);
    return cudaGetLastError();
}

cudaError_t launch_tc_forward(const ChainParams& p, cudaStream_t s) { return launch<false>(p, s); }
cudaError_t launch_tc_summary(const ChainParams& p, cudaStream_t s) { return launch<true>(p, s); }
cudaError_t launch_tc_phase1(const ChainParams& fwd, const ChainParams& sum, cudaStream_t s) {
    return launch_phase1(fwd, sum, s);
}

}  // namespace gdn
