// gdn_scan_tc.cu -- the in-order scan over pieces (segment prefix scan) on the tensor cores,
// for K == V == 128.
//
// Per (b, h) the state entering piece p + 1 is H_{p+1} = M_p H_p + S_p, starting from the
// state entering piece p_first ("RFC: HyperParallel Linear Attention Context Parallel",
// section 2.2: compose and the exclusive scan of the affine summaries; "Context Parallelism
// in ART", section 08, "Then parallelize across GPUs"). The same contract as the CUDA-core
// scan_kernel (gdn_simt.cu): the state entering every piece p > p_first is written to Hp[p],
// the state entering every piece p with p % nsub == 0 to H_seg[p / nsub], and H_seg[0] is
// h_seg0 (or zero) when p_first > 0.
//
// One CTA per (b, h) and column tile of the state (32 or 64 columns, so that the grid fits in
// one wave when it can): the step is one M = 128, K = 128 product on tcgen05 (kind::tf32, fp32
// accumulation in tensor memory) with the accumulator preloaded with S_p's tile.
//   A operand: M_p as stored (K-major: row k, 128 features), brought by TMA in four boxes of
//     32 features x 128 rows with the 128-byte swizzle -- exactly the operand layout. The
//     tensor core reads it as tf32, i.e. with its low 13 bits dropped: truncated toward zero
//     by 2^-11 / (2 ln 2) of its magnitude on average for mantissas spread log-uniformly. The
//     B side carries the inverse factor, so the product has no systematic bias; what remains
//     is a zero-mean error of at most 2^-11 per element of M. M_{p+1} is loaded while step p
//     runs.
//   B operand: the state tile transposed (row = state column c, 128 features k), times that
//     factor, as the sum hi + lo of two tf32 operands (hi = the value with its low 13 bits
//     dropped, lo = the exact remainder): two passes, M (H_hi + H_lo), so the state enters the
//     product at fp32 accuracy.
// 128 threads: thread k owns row k of the state tile (tensor-memory lane k); S_{p+1}'s row is
// loaded into registers while step p's product runs. Every wait on an mbarrier is bounded: on
// expiry the kernel records GDN_ERR_TIMEOUT, lets what it issued retire (bounded), frees
// tensor memory and returns.
#include "gdn_tc_common.cuh"

namespace gdn {
namespace {

constexpr int kScThreads = 128;
constexpr float kScTruncComp = 1.0f + 3.5222e-4f;   // 1 + 2^-11 / (2 ln 2)
// shared memory (bytes from a 1024-aligned base)
constexpr uint32_t SC_M0 = 0;            // M_p as loaded, two buffers: [kblock 4][128 rows x 128 B]
constexpr uint32_t SC_MBYTES = 65536;
constexpr uint32_t SC_BHI = 2 * SC_MBYTES;   // state tile^T hi: [kblock 4][NT rows x 128 B], then lo
template <int NT>
struct ScanSmem {
    static constexpr uint32_t BBYTES = 4 * NT * 128;
    static constexpr uint32_t BLO = SC_BHI + BBYTES;
    static constexpr uint32_t BAR = BLO + BBYTES;   // mbarriers: M buffers 0, 1; MMA; flags
    static constexpr uint32_t BYTES = BAR + 64 + 1024;   // + alignment slack
    static_assert(BYTES <= 232448u, "shared memory budget");
};
// kind::tf32, M = 128, N = NT, A and B K-major in shared memory
template <int NT>
struct IdScan {
    static constexpr uint32_t value =
        (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(NT >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
};

enum : unsigned { STAG_M = 301, STAG_MMA = 302 };

struct ScanParams {
    CUtensorMap tm_m;   // M viewed as [P*BH*128 rows, 128 columns] fp32
    const float* S;
    const float* h_first;
    float* Hp;
    float* H_seg;
    const float* h_seg0;
    int p_first, P, nsub, BH;
    DeviceError* err;
    long long wait_limit;
};

template <uint32_t ID>
__device__ __forceinline__ void mma_ss_tf32(uint32_t d_tmem, uint64_t a, uint64_t b,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "n"(ID), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

template <int NT>
__global__ void __launch_bounds__(kScThreads, 1) scan_tc_kernel(const __grid_constant__ ScanParams p) {
    using L = ScanSmem<NT>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    const uint32_t bar_m0 = base + L::BAR, bar_mma = base + L::BAR + 16;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sm + L::BAR + 24);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::BAR + 28);
    volatile int* go = reinterpret_cast<volatile int*>(sm + L::BAR + 32);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, c0 = blockIdx.y * NT;
    const int k = tid;                                   // state row (tensor-memory lane)
    const int nsteps = p.P - 1 - p.p_first;              // products to form (>= 1)
    const long long kv = 128LL * 128;

    auto load_m = [&](int s) {   // M of step s (piece p_first + s) into buffer s & 1
        const uint32_t bar = bar_m0 + 8 * (s & 1);
        const int row0 = ((p.p_first + s) * p.BH + bh) * 128;
        mbar_arrive_expect_tx(bar, SC_MBYTES);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)
            tma_load_2d(base + SC_M0 + (s & 1) * SC_MBYTES + kb * 16384, &p.tm_m, bar, kb * 32, row0);
    };
    if (tid == 0) {
        mbar_init(bar_m0, 1);
        mbar_init(bar_m0 + 8, 1);
        mbar_init(bar_mma, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
        load_m(0);
        if (nsteps > 1) load_m(1);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         base + L::BAR + 24),
                     "r"((uint32_t)NT)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // the state entering the first segment, when the scan starts past it
    if (p.H_seg && p.p_first > 0) {
        const float* src = p.h_seg0 ? p.h_seg0 + ((long long)bh * 128 + k) * 128 + c0 : nullptr;
        float* dst = p.H_seg + ((long long)bh * 128 + k) * 128 + c0;
#pragma unroll
        for (int j = 0; j < NT; j += 4)
            *reinterpret_cast<float4*>(dst + j) =
                src ? __ldg(reinterpret_cast<const float4*>(src + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // row k of the state tile entering piece p_first, and of S_{p_first}
    float h[NT], sv[NT];
    auto load_row = [&](float* dst, const float* src) {
#pragma unroll
        for (int j = 0; j < NT; j += 4) {
            const float4 x = src ? __ldg(reinterpret_cast<const float4*>(src + j))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            dst[j] = x.x, dst[j + 1] = x.y, dst[j + 2] = x.z, dst[j + 3] = x.w;
        }
    };
    auto s_row = [&](int pc) { return p.S + ((long long)pc * p.BH + bh) * kv + (long long)k * 128 + c0; };
    load_row(h, p.h_first ? p.h_first + ((long long)bh * 128 + k) * 128 + c0 : nullptr);
    load_row(sv, s_row(p.p_first));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_row = tmem + ((uint32_t)(32 * warp) << 16);   // this warp's lanes, column 0

    // byte offset of element (row c, feature k) in a [kblock 4][NT rows x 128 B] operand
    const uint32_t b_kb = (uint32_t)(k >> 5) * (NT * 128), b_chunk = (uint32_t)((k & 31) >> 2),
                   b_word = (uint32_t)(k & 3) * 4;
    int issued = 0;     // MMA groups committed
    int loads = nsteps > 1 ? 2 : 1;   // M loads issued
    bool ok = true;
#pragma unroll 1
    for (int s = 0; s <= nsteps; ++s) {
        const int pc = p.p_first + s;   // h is the state entering piece pc
        if (p.Hp && s > 0) {
            float* dst = p.Hp + ((long long)pc * p.BH + bh) * kv + (long long)k * 128 + c0;
#pragma unroll
            for (int j = 0; j < NT; j += 4)
                *reinterpret_cast<float4*>(dst + j) = make_float4(h[j], h[j + 1], h[j + 2], h[j + 3]);
        }
        if (p.H_seg && pc % p.nsub == 0) {
            float* dst = p.H_seg + ((long long)(pc / p.nsub) * p.BH + bh) * kv + (long long)k * 128 + c0;
#pragma unroll
            for (int j = 0; j < NT; j += 4)
                *reinterpret_cast<float4*>(dst + j) = make_float4(h[j], h[j + 1], h[j + 2], h[j + 3]);
        }
        if (s == nsteps) break;
        // ---- B = the state tile transposed (with the compensation factor), hi and lo; the
        //      accumulator <- S_p's tile
#pragma unroll
        for (int c = 0; c < NT; ++c) {
            const uint32_t off = b_kb + sw128(c, b_chunk) + b_word;
            const float x = h[c] * kScTruncComp;
            const float hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
            *reinterpret_cast<float*>(sm + SC_BHI + off) = hi;
            *reinterpret_cast<float*>(sm + L::BLO + off) = x - hi;
        }
#pragma unroll
        for (int j = 0; j < NT; j += 16) tmem_st16(t_row + j, reinterpret_cast<const uint32_t*>(sv + j));
        tmem_wait_st();
        fence_proxy_async();   // the operands written by these threads are read by the MMAs
        tc_fence_before();
        // ---- M_p has landed (the first warp waits; every thread reads its verdict)
        const uint32_t mbuf = SC_M0 + (s & 1) * SC_MBYTES;
        if (!group_wait<1, kScThreads>(warp == 0, lane == 0, bar_m0 + 8 * (s & 1), (s >> 1) & 1,
                                       true, go, abort_flag, p.wait_limit, p.err, STAG_M)) {
            ok = false;
            break;
        }
        // ---- D += M (H_hi + H_lo) (K = 128 in steps of 8)
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int k8 = 0; k8 < 16; ++k8) {
                const uint32_t ao = (k8 >> 2) * 16384 + (k8 & 3) * 32;
                const uint32_t bo = (k8 >> 2) * (NT * 128) + (k8 & 3) * 32;
                mma_ss_tf32<IdScan<NT>::value>(tmem, desc_k(base + mbuf + ao), desc_k(base + SC_BHI + bo), 1u);
                mma_ss_tf32<IdScan<NT>::value>(tmem, desc_k(base + mbuf + ao), desc_k(base + L::BLO + bo), 1u);
            }
            mma_commit(bar_mma);
        }
        __syncwarp();
        ++issued;
        // S of the next step into registers while the product runs
        if (s + 1 < nsteps) load_row(sv, s_row(pc + 1));
        if (!group_wait<1, kScThreads>(warp == 0, lane == 0, bar_mma, (issued - 1) & 1, true, go,
                                       abort_flag, p.wait_limit, p.err, STAG_MMA)) {
            ok = false;
            break;
        }
        tc_fence_after();
        // the MMAs have read M_p's buffer: the load of M_{p+2} can go into it
        if (tid == 0 && s + 2 < nsteps) {
            load_m(s + 2);
            ++loads;
        }
        // ---- row k of the state entering piece pc + 1
#pragma unroll
        for (int j = 0; j < NT; j += 16) tmem_ld16(t_row + j, h + j);
        tmem_wait_ld();
        tc_fence_before();
        __syncthreads();   // every lane read out before the next step's S overwrites it
    }
    // ---- after a wait gave up: let the MMAs and copies this CTA issued retire before its
    //      shared and tensor memory are released
    if (!ok && tid == 0) {
        if (issued > 0) mbar_drain(bar_mma, (issued - 1) & 1, p.wait_limit);
        for (int s = 0; s < loads; ++s) mbar_drain(bar_m0 + 8 * (s & 1), (s >> 1) & 1, p.wait_limit);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"((uint32_t)NT)
                     : "memory");
    }
}

template <int NT>
cudaError_t launch_scan_nt(const ScanParams& sp, cudaStream_t s) {
    using L = ScanSmem<NT>;
    cudaError_t e = cudaFuncSetAttribute(scan_tc_kernel<NT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::BYTES);
    if (e != cudaSuccess) return e;
    scan_tc_kernel<NT><<<dim3((unsigned)sp.BH, 128 / NT), kScThreads, L::BYTES, s>>>(sp);
    return cudaGetLastError();
}

bool make_m_map(CUtensorMap* m, const float* M, int P, int BH) {
    auto fn = encode_fn();
    if (!fn || !M) return false;
    cuuint64_t dims[2] = {128, (cuuint64_t)P * (cuuint64_t)BH * 128};
    cuuint64_t strides[1] = {128 * 4};
    cuuint32_t box[2] = {32, 128};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(M), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_scan_supported(const float* M, const float* S, int p_first, int P, int K, int V) {
    return M && S && K == 128 && V == 128 && P - p_first >= 2 && tc_runtime_ok();
}

cudaError_t launch_tc_scan(const float* M, const float* S, const float* h_first, float* Hp,
                           float* H_seg, const float* h_seg0, int p_first, int P, int nsub, int BH,
                           DeviceError* err, cudaStream_t s) {
    ScanParams sp{};
    if (!make_m_map(&sp.tm_m, M, P, BH)) return cudaErrorInvalidValue;
    sp.S = S;
    sp.h_first = h_first;
    sp.Hp = Hp;
    sp.H_seg = H_seg;
    sp.h_seg0 = h_seg0;
    sp.p_first = p_first;
    sp.P = P;
    sp.nsub = nsub;
    sp.BH = BH;
    sp.err = err;
    sp.wait_limit = 4000000000LL;   // ~2 s at GB300 clocks
    // one CTA per SM (shared memory): 32-column tiles while the grid fits in one wave
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidValue;
    return (long long)BH * 4 <= sms ? launch_scan_nt<32>(sp, s) : launch_scan_nt<64>(sp, s);
}

}  // namespace gdn
