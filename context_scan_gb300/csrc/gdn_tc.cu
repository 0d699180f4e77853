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
//   O  = diag(2^G) Q H + C R,   C[i,j] = 2^(G_i - G_j) q_i.k_j (j <= i)
//   H <- 2^(G_last) H + sum_j 2^(G_last - G_j) k_j R_j
// Every contraction is issued as an M = 128 tcgen05.mma (kind::f16, bf16 operands, fp32
// accumulation in tensor memory) by putting a 128-wide dimension on M -- the products are
// formed transposed:
//   P1  S^T-free Gram: D[0:128, 0:64]   = [K ; Q] K^T         (rows 0..63 K K^T, 64..127 Q K^T)
//   P2  U^T          = V^T (A diag(beta))^T
//   P3  W^T          = K^T (A diag(beta 2^Gx))^T
//   S1  R^T          = U^T + H^T (-W)^T    (accumulates onto U^T)
//   S2  (Q H)^T      = H^T Q^T
//   S3  (C R)^T      = R^T C^T
//   S4  H^T         += (R^T diag(2^(G_last - G))) K   (state master pre-scaled by 2^G_last)
// S1-S3 are kind::tf32 with the A operand (H^T, R^T) read straight from tensor memory, so
// the fp32 state and the corrected values are never rounded to bf16; S4 feeds the decayed
// R^T as an unevaluated bf16 sum hi + lo (two MMAs). P1-P3 and S4 are kind::f16 (bf16).
// The triangular inverse, gate exponentials and the output combine run on CUDA cores.
// Exponents are always differences of cumulative gates, never 2^-G.
//
// Warps 0-3 ("math") own tensor-memory lanes 0..127 and run the chunk step; warp 4 is the
// producer (TMA loads of the q/k/v tiles, 128-byte swizzle, two stages; plain loads of the
// gates). Every wait on an mbarrier is bounded: on expiry the kernel records
// GDN_ERR_TIMEOUT in the device error word, drains what it issued and frees tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstring>
#include <mutex>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kD = 128;        // K == V
constexpr int kC = 64;         // tokens per chunk
constexpr int kThreads = 160;  // 4 math warps + 1 producer warp
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

// tensor-memory columns (fp32 accumulators, 128 lanes each)
constexpr uint32_t TM_S = 0;     // [K;Q] K^T, then W^T
constexpr uint32_t TM_U0 = 64;   // U^T -> R^T (even chunks)
constexpr uint32_t TM_U1 = 128;  // (odd chunks)
constexpr uint32_t TM_OI = 192;  // H^T Q^T
constexpr uint32_t TM_OA = 256;  // R^T C^T
constexpr uint32_t TM_H = 320;   // state master H^T (128 columns)

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t SM_KQ0 = 0;        // stage 0: [khalf][K rows | Q rows] 2 x 16 KB
constexpr uint32_t SM_KQ1 = 32768;    // stage 1
constexpr uint32_t SM_V = 65536;      // [vhalf][64 rows x 128 B]
constexpr uint32_t SM_W = 81920;      // -W tf32, K-major: [kblock][64 rows (i) x 32 (k)];
                                      // inverse scratch before that
constexpr uint32_t SM_QT = 114688;    // Q tf32, K-major: [kblock][64 rows (i) x 32 (k)]
constexpr uint32_t SM_RD = 147456;    // R^T diag(2^(G_last - G)) as bf16 hi (+0) and lo (+16 KB);
                                      // before that, L (+0) and A (+16 KB) of the inverse, fp32
constexpr uint32_t SM_AB = 180224;    // A diag(beta) bf16: 64 rows (i) x 64 (j)
constexpr uint32_t SM_ABG = 188416;   // A diag(beta 2^Gx) bf16
constexpr uint32_t SM_C = 196608;     // C tf32: [kblock][64 rows (i) x 32 (j)]
constexpr uint32_t SM_SCAL = 212992;  // gates per stage + per-chunk scalars
constexpr uint32_t SM_BAR = 216064;   // mbarriers, tmem base, abort flag
constexpr uint32_t SM_END = 216128;
constexpr uint32_t kSmemBytes = SM_END + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

// 64 x 64 fp32 matrices of the inverse: row-major with the column XOR-swizzled by the row,
// so both row-wise and column-wise walks by a warp hit 32 distinct banks
__device__ __forceinline__ int sw64(int i, int j) { return i * 64 + (j ^ (i & 31)); }

// mbarrier slots (8 bytes each) at SM_BAR
constexpr uint32_t B_FULL0 = 0, B_FULL1 = 8, B_EMPTY0 = 16, B_EMPTY1 = 24, B_VEMPTY = 32,
                   B_MMA = 40, B_TMEM = 48, B_ABORT = 52, B_GO = 56;

// wait tags recorded in the device error word's detail field
enum : unsigned { TAG_FULL = 1, TAG_MMA = 2, TAG_EMPTY = 3, TAG_VEMPTY = 4 };

struct TcParams {
    CUtensorMap tm_q;
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    ChainParams c;
    long long wait_limit;   // SM clock cycles before a wait gives up
};

// ------------------------------------------------------------------------------------
// PTX wrappers
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void record_error(DeviceError* e, unsigned code, unsigned detail) {
    if (e && atomicCAS(&e->code, 0u, code) == 0u) atomicExch(&e->detail, detail);
}

// Bounded wait for the completion of the phase with the given parity. Gives up when the
// CTA's abort flag is raised or after `limit` SM cycles (then records the timeout and
// raises the flag). Returns false if it gave up.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       long long limit, DeviceError* err, unsigned tag) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            record_error(err, GDN_ERR_TIMEOUT, tag);
            *abort_flag = 1;
            return false;
        }
    }
}

// Bounded wait used only while shutting down after an abort: lets copies or MMAs this CTA
// issued retire before its shared and tensor memory are released.
__device__ __noinline__ void mbar_drain(uint32_t bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > limit) return;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void math_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Shared-memory matrix descriptor (sm_100 format): start, leading/stride byte offsets,
// version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// K-major operand, rows of 128 bytes packed in 8-row groups of 1024 bytes
__device__ __forceinline__ uint64_t desc_k(uint32_t saddr) { return sdesc(saddr, 16, 1024); }
// MN-major operand: 64-element blocks along M/N `mn_stride` bytes apart, 8-row groups along
// K 1024 bytes apart
__device__ __forceinline__ uint64_t desc_mn(uint32_t saddr, uint32_t mn_stride) {
    return sdesc(saddr, mn_stride, 1024);
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D.
constexpr uint32_t idesc(int M, int N, bool a_mn, bool b_mn, bool a_neg) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_neg ? 1u : 0u) << 13) |
           ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t ID_P1 = idesc(128, 64, false, false, false);
constexpr uint32_t ID_P23 = idesc(128, 64, true, false, false);
constexpr uint32_t ID_S4 = idesc(128, 128, false, true, false);
// kind::tf32, fp32 D, M = 128, N = 64, A from tensor memory, B K-major (S1, S2, S3)
constexpr uint32_t ID_TF = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(64 >> 3) << 17) |
                           ((uint32_t)(128 >> 4) << 24);

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                    uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(accumulate)
        : "memory");
}

// D (+)= A B with A read from tensor memory (tf32 operands, fp32 accumulation)
__device__ __forceinline__ void mma_ta_tf32(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                            uint32_t id, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ float to_tf32(float x) {
    uint32_t y;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(y) : "f"(x));
    return __uint_as_float(y);
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&t);
}

// Write 8*nchunk consecutive values of one 128-byte row of a 128-byte-swizzled tile,
// starting at 16-byte chunk c0 of the row (rows packed in 8-row groups of 1024 bytes).
template <int NCHUNK>
__device__ __forceinline__ void st_row_sw128(uint8_t* tile, int row, int c0, const float* v) {
    uint8_t* rp = tile + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
    for (int c = 0; c < NCHUNK; ++c) {
        uint4 pk;
        pk.x = pack_bf16(v[8 * c + 0], v[8 * c + 1]);
        pk.y = pack_bf16(v[8 * c + 2], v[8 * c + 3]);
        pk.z = pack_bf16(v[8 * c + 4], v[8 * c + 5]);
        pk.w = pack_bf16(v[8 * c + 6], v[8 * c + 7]);
        *reinterpret_cast<uint4*>(rp + (((c0 + c) ^ (row & 7)) << 4)) = pk;
    }
}

__device__ __forceinline__ float bf16_at(const void* base, long long idx) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
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

    float* gates = reinterpret_cast<float*>(sm + SM_SCAL);   // [stage][g | beta][64]
    float* s_gam = gates + 256;   // G (log2 units)
    float* s_gx = s_gam + 64;     // Gx
    float* s_eg = s_gx + 64;      // 2^G
    float* s_dd = s_eg + 64;      // 2^(G_last - G)
    float* s_bet = s_dd + 64;     // beta
    float* s_bekr = s_bet + 64;   // beta 2^Gx
    float* s_misc = s_bekr + 64;  // [0] = 2^G_last
    float* Ls = reinterpret_cast<float*>(sm + SM_RD);            // inverse only
    float* As = reinterpret_cast<float*>(sm + SM_RD + 16384);    // inverse only
    float* Yscr = reinterpret_cast<float*>(sm + SM_W);           // inverse only
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
        mbar_init(bar0 + B_MMA, 1);
        *abort_flag = 0;
        *reinterpret_cast<volatile int*>(sm + SM_BAR + B_GO) = 1;
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

    if (warp == 4) {
        // ================================ producer ================================
        const uint32_t tx = 16384u + (SUMMARY ? 0u : 16384u) + (need_v ? 16384u : 0u);
        int issued_last[2] = {-1, -1};
        for (int n = 0; n < nchunks; ++n) {
            const int s = n & 1;
            const uint32_t full = bar0 + (s ? B_FULL1 : B_FULL0);
            // lane 0 waits; the warp follows its verdict, so the lanes never diverge
            int ok = 1;
            if (lane == 0) {
                if (n >= 2)
                    ok = mbar_wait(bar0 + (s ? B_EMPTY1 : B_EMPTY0), ((n >> 1) - 1) & 1,
                                   abort_flag, limit, c.err, TAG_EMPTY);
                if (ok && need_v && n >= 1)
                    ok = mbar_wait(bar0 + B_VEMPTY, (n - 1) & 1, abort_flag, limit, c.err,
                                   TAG_VEMPTY);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            const int row0 = b * c.T + seg * c.seg_len + n * kC;   // flattened (b, t) row
            if (lane == 0) {
                mbar_arrive_expect_tx(full, tx);
                const uint32_t kq = base + (s ? SM_KQ1 : SM_KQ0);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    tma_load_3d(kq + hf * 16384, &p.tm_k, full, hf * 64, h, row0);
                    if (!SUMMARY) tma_load_3d(kq + hf * 16384 + 8192, &p.tm_q, full, hf * 64, h, row0);
                    if (need_v) tma_load_3d(base + SM_V + hf * 8192, &p.tm_v, full, hf * 64, h, row0);
                }
            }
            issued_last[s] = n;
            float* gs = gates + s * 128;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int i = lane + 32 * e;
                const long long idx = (long long)(row0 + i) * c.H + h;
                gs[i] = bf16_at(c.g, idx) * kLog2e;
                gs[64 + i] = bf16_at(c.beta, idx);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(full);
        }
        if (*abort_flag && lane == 0) {
            // let every copy this warp issued land before the CTA's memory is released
            for (int s = 0; s < 2; ++s)
                if (issued_last[s] >= 0)
                    mbar_drain(bar0 + (s ? B_FULL1 : B_FULL0), (issued_last[s] >> 1) & 1, limit);
        }
    } else {
        // ================================== math ==================================
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;   // this warp's TMEM lanes
        const uint32_t t_row = tmem + lane_off;
        uint32_t mma_phase = 0;
        bool mma_pending = false;
        const long long bhoff = (long long)bh * kD * kD;

        // ---- initial state: row `tid` of H^T (= column tid of H)
        for (int part = 0; part < 4; ++part) {
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int k = part * 32 + j;
                float v0 = 0.f;
                if (SUMMARY) {
                    v0 = (blk == 0 && k == tid) ? 1.f : 0.f;
                } else if (c.h_start) {
                    v0 = c.h_start[seg * c.h_start_seg_stride + bhoff + (long long)k * kD + tid];
                }
                x[j] = v0;
            }
            tmem_st32(t_row + TM_H + part * 32, x);
        }
        tmem_wait_st();
        tc_fence_before();
        math_bar();

        // Thread 0 waits and publishes a verdict before the named barrier; every math
        // thread then reads the same verdict, so a timeout cannot split the warps.
        volatile int* s_go = reinterpret_cast<volatile int*>(sm + SM_BAR + B_GO);
        auto math_wait = [&](uint32_t bar, uint32_t parity, unsigned tag) -> bool {
            if (tid == 0) {
                const bool ok = mbar_wait(bar, parity, abort_flag, limit, c.err, tag);
                *s_go = (ok && !*abort_flag) ? 1 : 0;
            }
            math_bar();
            return *s_go != 0;
        };
        auto mma_wait = [&]() -> bool {
            const bool ok = math_wait(bar0 + B_MMA, mma_phase, TAG_MMA);
            if (ok) {
                mma_phase ^= 1u;
                mma_pending = false;
            }
            return ok;
        };

        for (int n = 0; n < nchunks; ++n) {
            const int s = n & 1;
            const uint32_t kq = base + (s ? SM_KQ1 : SM_KQ0);
            const uint32_t t_u = tmem + ((n & 1) ? TM_U1 : TM_U0);
            if (!math_wait(bar0 + (s ? B_FULL1 : B_FULL0), (n >> 1) & 1, TAG_FULL)) break;
            // ---- gate cumsum and per-chunk scalars (warp 0)
            if (warp == 0) {
                const float* gs = gates + s * 128;
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
                s_gam[2 * lane] = G0;
                s_gam[2 * lane + 1] = G1;
                s_gx[2 * lane] = excl;
                s_gx[2 * lane + 1] = G0;
                s_eg[2 * lane] = ex2(G0);
                s_eg[2 * lane + 1] = ex2(G1);
                s_dd[2 * lane] = ex2(glast - G0);
                s_dd[2 * lane + 1] = ex2(glast - G1);
                const float b0 = gs[64 + 2 * lane], b1 = gs[64 + 2 * lane + 1];
                s_bet[2 * lane] = b0;
                s_bet[2 * lane + 1] = b1;
                s_bekr[2 * lane] = b0 * ex2(excl);
                s_bekr[2 * lane + 1] = b1 * ex2(G0);
                if (lane == 0) s_misc[0] = ex2(glast);
            }
            math_bar();

            // ---- Q tile -> tf32 K-major copy (B operand of S2): thread = (row i, k half)
            if (!SUMMARY) {
                const int i = tid >> 1, kh = tid & 1;
                const uint8_t* src = sm + (s ? SM_KQ1 : SM_KQ0) + kh * 16384 + 8192 +
                                     (i >> 3) * 1024 + (i & 7) * 128;
                uint8_t* dst = sm + SM_QT + (i >> 3) * 1024 + (i & 7) * 128;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 u = *reinterpret_cast<const uint4*>(src + ((cc ^ (i & 7)) << 4));
                    // 8 bf16 -> 8 fp32 (exact); features k = 64 kh + 8 cc .. + 7
                    const uint4 lo4 = make_uint4(u.x << 16, u.x & 0xFFFF0000u, u.y << 16, u.y & 0xFFFF0000u);
                    const uint4 hi4 = make_uint4(u.z << 16, u.z & 0xFFFF0000u, u.w << 16, u.w & 0xFFFF0000u);
                    const int kb = kh * 2 + (cc >> 2);
                    const int q0 = (2 * cc) & 7, q1 = (2 * cc + 1) & 7;
                    *reinterpret_cast<uint4*>(dst + kb * 8192 + ((q0 ^ (i & 7)) << 4)) = lo4;
                    *reinterpret_cast<uint4*>(dst + kb * 8192 + ((q1 ^ (i & 7)) << 4)) = hi4;
                }
                fence_proxy_async();
            }

            // ---- P1: [K ; Q] K^T -> TM_S
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma(tmem + TM_S, desc_k(kq + off), desc_k(kq + off), ID_P1, ks > 0);
                }
                mma_commit(bar0 + B_MMA);
            }
            mma_pending = true;
            if (!mma_wait()) break;
            tc_fence_after();

            // ---- L rows (lanes 0..63) and C rows (lanes 64..127)
            {
                float srow[64];
                tmem_ld32(t_row + TM_S, srow);
                tmem_ld32(t_row + TM_S + 32, srow + 32);
                tmem_wait_ld();
                if (tid < 64) {
                    const int i = tid;
                    const float gxi = s_gx[i], bi = s_bet[i];
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        Ls[sw64(i, j)] = (j < i) ? bi * ex2(gxi - s_gam[j]) * srow[j] : 0.f;
                } else if (!SUMMARY) {
                    // C row i as tf32, K-major: two 32-wide blocks of 128-byte rows
                    const int i = tid - 64;
                    const float gi = s_gam[i];
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        srow[j] = to_tf32((j <= i) ? ex2(gi - s_gam[j]) * srow[j] : 0.f);
#pragma unroll
                    for (int kb = 0; kb < 2; ++kb) {
                        uint8_t* rp = sm + SM_C + kb * 8192 + (i >> 3) * 1024 + (i & 7) * 128;
#pragma unroll
                        for (int cq = 0; cq < 8; ++cq) {
                            const float* vv = srow + kb * 32 + cq * 4;
                            *reinterpret_cast<uint4*>(rp + ((cq ^ (i & 7)) << 4)) =
                                make_uint4(__float_as_uint(vv[0]), __float_as_uint(vv[1]),
                                           __float_as_uint(vv[2]), __float_as_uint(vv[3]));
                        }
                    }
                }
            }
            tc_fence_before();
            math_bar();

            // ---- A = (I + L)^-1: 16x16 diagonal blocks, then block forward substitution
            if (tid < 64) {
                const int bs = (tid >> 4) * 16, cc = tid & 15;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) x[r] = (r == cc) ? 1.f : 0.f;
#pragma unroll
                for (int r = 1; r < 16; ++r) {
                    float a = 0.f;
#pragma unroll
                    for (int m = 0; m < r; ++m) a = fmaf(Ls[sw64(bs + r, bs + m)], x[m], a);
                    if (r > cc) x[r] = -a;
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) As[sw64(bs + r, bs + cc)] = x[r];
            } else {
                // zero the blocks above the diagonal
                for (int e = tid - 64; e < 6 * 256; e += 64) {
                    const int blkid = e >> 8, w = e & 255;
                    const int I = (blkid < 3) ? 0 : (blkid < 5 ? 1 : 2);
                    const int J = (blkid < 3) ? blkid + 1 : (blkid < 5 ? blkid - 1 : 3);
                    As[sw64(16 * I + (w >> 4), 16 * J + (w & 15))] = 0.f;
                }
            }
            math_bar();
            {
                const int r0 = tid >> 4, cc = tid & 15;
                for (int I = 1; I < 4; ++I) {
                    for (int J = 0; J < I; ++J) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int r = r0 + 8 * e;
                            float a = 0.f;
                            for (int m = J; m < I; ++m) {
#pragma unroll
                                for (int l = 0; l < 16; ++l)
                                    a = fmaf(Ls[sw64(16 * I + r, 16 * m + l)],
                                             As[sw64(16 * m + l, 16 * J + cc)], a);
                            }
                            Yscr[J * 256 + r * 16 + cc] = a;
                        }
                    }
                    math_bar();
                    for (int J = 0; J < I; ++J) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int r = r0 + 8 * e;
                            float a = 0.f;
#pragma unroll
                            for (int l = 0; l < 16; ++l)
                                a = fmaf(As[sw64(16 * I + r, 16 * I + l)], Yscr[J * 256 + l * 16 + cc], a);
                            As[sw64(16 * I + r, 16 * J + cc)] = -a;
                        }
                    }
                    math_bar();
                }
            }
            // ---- A diag(beta) and A diag(beta 2^Gx), bf16, K-major rows
            {
                const int i = tid & 63;
                const float* scale = (tid < 64) ? s_bet : s_bekr;
                float arow[64];
#pragma unroll
                for (int j = 0; j < 64; ++j) arow[j] = As[sw64(i, j)] * scale[j];
                st_row_sw128<8>(sm + ((tid < 64) ? SM_AB : SM_ABG), i, 0, arow);
            }
            fence_proxy_async();
            math_bar();

            // ---- P2: U^T = V^T (A diag beta)^T -> t_u ;  P3: W^T = K^T (A diag(beta 2^Gx))^T -> TM_S
            if (tid == 0) {
                tc_fence_after();
                if (need_v) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma(t_u, desc_mn(base + SM_V + ks * 2048, 8192),
                            desc_k(base + SM_AB + ks * 32), ID_P23, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma(tmem + TM_S, desc_mn(kq + ks * 2048, 16384), desc_k(base + SM_ABG + ks * 32),
                        ID_P23, ks > 0);
                if (need_v) mma_commit(bar0 + B_VEMPTY);
                mma_commit(bar0 + B_MMA);
            }
            mma_pending = true;
            if (!mma_wait()) break;
            tc_fence_after();

            // ---- -W -> tf32, K-major B operand of S1: thread k writes column k of rows i
            {
                float w[64];
                tmem_ld32(t_row + TM_S, w);
                tmem_ld32(t_row + TM_S + 32, w + 32);
                tmem_wait_ld();
                const int k = tid;
                uint8_t* col = sm + SM_W + (k >> 5) * 8192 + (k & 3) * 4;
                const int qk = (k & 31) >> 2;
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    *reinterpret_cast<float*>(col + (i >> 3) * 1024 + (i & 7) * 128 +
                                              ((qk ^ (i & 7)) << 4)) = to_tf32(-w[i]);
            }
            fence_proxy_async();
            tc_fence_before();
            math_bar();

            // ---- S1: R^T = U^T - H^T W^T (onto t_u);  S2: H^T Q^T -> TM_OI
            if (tid == 0) {
                tc_fence_after();
                // A = H^T straight from tensor memory (fp32 master read as tf32)
#pragma unroll
                for (int ks = 0; ks < 16; ++ks)
                    mma_ta_tf32(t_u, tmem + TM_H + ks * 8,
                                desc_k(base + SM_W + (ks >> 2) * 8192 + (ks & 3) * 32), ID_TF,
                                (need_v || ks > 0) ? 1u : 0u);
                if (!SUMMARY) {
#pragma unroll
                    for (int ks = 0; ks < 16; ++ks)
                        mma_ta_tf32(tmem + TM_OI, tmem + TM_H + ks * 8,
                                    desc_k(base + SM_QT + (ks >> 2) * 8192 + (ks & 3) * 32), ID_TF,
                                    ks > 0);
                }
                mma_commit(bar0 + B_MMA);
            }
            mma_pending = true;
            if (!mma_wait()) break;
            tc_fence_after();

            // ---- R^T row v = tid -> bf16 (plain and decayed); pre-scale the master by 2^G_last
            {
                float r[64];
                const uint32_t t_ur = lane_off + ((n & 1) ? TM_U1 : TM_U0);
                tmem_ld32(tmem + t_ur, r);
                tmem_ld32(tmem + t_ur + 32, r + 32);
                tmem_wait_ld();
                // decayed R as an unevaluated bf16 sum hi + lo (R itself stays in TMEM for S3)
                float lo[64];
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const float x = r[j] * s_dd[j];
                    r[j] = __bfloat162float(__float2bfloat16_rn(x));
                    lo[j] = x - r[j];
                }
                st_row_sw128<8>(sm + SM_RD, tid, 0, r);
                st_row_sw128<8>(sm + SM_RD + 16384, tid, 0, lo);
                const float ecl = s_misc[0];
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    float x[32];
                    tmem_ld32(t_row + TM_H + part * 32, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] *= ecl;
                    tmem_st32(t_row + TM_H + part * 32, x);
                }
                tmem_wait_st();
            }
            fence_proxy_async();
            tc_fence_before();
            math_bar();

            // ---- S3: R^T C^T -> TM_OA ;  S4: H^T += R^T diag(2^(G_last - G)) K
            if (tid == 0) {
                tc_fence_after();
                if (!SUMMARY) {
                    // (C R)^T = R^T C^T with R^T read from tensor memory, tf32
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ta_tf32(tmem + TM_OA, t_u + ks * 8,
                                    desc_k(base + SM_C + (ks >> 2) * 8192 + (ks & 3) * 32), ID_TF,
                                    ks > 0);
                }
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma(tmem + TM_H, desc_k(base + SM_RD + part * 16384 + ks * 32),
                            desc_mn(kq + ks * 2048, 16384), ID_S4, 1u);
                mma_commit(bar0 + (s ? B_EMPTY1 : B_EMPTY0));
                mma_commit(bar0 + B_MMA);
            }
            mma_pending = true;
            if (!mma_wait()) break;
            tc_fence_after();

            // ---- output: o_i = 2^G_i (H^T Q^T)[:, i] + (R^T C^T)[:, i]
            if (!SUMMARY) {
                const int row0 = b * c.T + seg * c.seg_len + n * kC;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float oi[32], oa[32];
                    tmem_ld32(t_row + TM_OI + half * 32, oi);
                    tmem_ld32(t_row + TM_OA + half * 32, oa);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int i = half * 32 + j;
                        const float val = fmaf(s_eg[i], oi[j], oa[j]);
                        const long long idx = ((long long)(row0 + i) * c.H + h) * kD + tid;
                        if (c.out_bf16)
                            reinterpret_cast<__nv_bfloat16*>(c.o)[idx] = __float2bfloat16_rn(val);
                        else
                            reinterpret_cast<float*>(c.o)[idx] = val;
                    }
                }
            }
            tc_fence_before();
            math_bar();
        }

        if (*s_go == 0) {
            if (mma_pending && tid == 0)   // let an issued MMA group retire before TMEM is freed
                mbar_drain(bar0 + B_MMA, mma_phase, limit);
        } else {
            // ---- the chain's final state: thread v writes column v of H (row v of H^T)
            float* dst = nullptr;
            if (SUMMARY) {
                const long long sb = ((long long)seg * c.B * c.H + bh) * kD * kD;
                dst = (blk == 0 ? c.M : c.S) + sb;
            } else if (c.h_final && seg == c.nseg_total - 1) {
                dst = c.h_final + bhoff;
            }
            if (dst) {
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    float x[32];
                    tmem_ld32(t_row + TM_H + part * 32, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) dst[(long long)(part * 32 + j) * kD + tid] = x[j];
                }
            }
        }
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
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// [B*T, H, 128] bf16 viewed as a 3-d tensor; box = 64 features x 1 head x 64 tokens
bool make_map(CUtensorMap* m, const void* ptr, const ChainParams& c) {
    auto fn = encode_fn();
    if (!fn || !ptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)c.H, (cuuint64_t)c.B * (cuuint64_t)c.T};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)c.H * kD * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool SUMMARY>
cudaError_t launch(const ChainParams& c, cudaStream_t s) {
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
