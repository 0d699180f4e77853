// gdn_tc_common.cuh -- device helpers shared by the tcgen05 chain kernels and the WY kernel:
// PTX wrappers (mbarrier, TMA, tcgen05, mma.sync), swizzled tile addressing, and the host
// side tensor-map encoder. Included by one translation unit per kernel family; everything
// here has internal linkage.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "gdn_internal.h"

namespace gdn {
namespace {

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

// As mbar_try_wait, but the hardware may suspend the waiting warp for up to `hint_ns`
// nanoseconds until the phase completes, instead of the warp re-polling and taking issue
// slots from the warps it shares a scheduler with.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity,
                                                      uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void record_error(DeviceError* e, unsigned code, unsigned detail) {
    if (e && atomicCAS(&e->code, 0u, code) == 0u) atomicExch(&e->detail, detail);
}

// Bounded wait for the completion of the phase with the given parity. Gives up when the
// CTA's abort flag is raised or after `limit` SM cycles (then records the timeout and
// raises the flag). Returns false if it gave up. The common case -- the phase has completed
// -- is inlined at every call site; only the polling loop is a call. (With most of the SM's
// shared memory in use, L1 is small and a call's stack traffic can go out to L2: in a kernel
// whose warps hand work to each other every few hundred cycles, that was the largest cost
// of a wait.)
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                            long long limit, DeviceError* err, unsigned tag) {
    const long long t0 = clock64();
    for (;;) {
        // suspended in hardware (up to 20 us per try) rather than re-polling: a polling warp
        // starves the compute warps on its scheduler
        if (mbar_try_wait_suspend(bar, parity, 20000u)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            record_error(err, GDN_ERR_TIMEOUT, tag);
            *abort_flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          long long limit, DeviceError* err, unsigned tag) {
    return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity, abort_flag, limit, err, tag);
}

// Bounded wait used only while shutting down after an abort: lets copies or MMAs this CTA
// issued retire before its shared and tensor memory are released.
__device__ __noinline__ void mbar_drain(uint32_t bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > limit) return;
}

// Named barrier over `N` threads (non-.aligned form: the threads of a warp may arrive
// diverged, e.g. after a leader warp's lane-0 work).
template <int ID, int N>
__device__ __forceinline__ void named_bar() {
    asm volatile("barrier.sync %0, %1;" ::"n"(ID), "n"(N) : "memory");
}

// The first warp of a warp group waits (when `doit`) -- all of its lanes poll together and
// see identical values, so the warp stays converged -- and its lane 0 publishes a verdict
// before the group's named barrier; every thread of the group then reads the same verdict,
// so a timeout can never split the group between a barrier and a break.
template <int ID, int N>
__device__ __forceinline__ bool group_wait(bool leader_warp, bool lane0, uint32_t bar,
                                           uint32_t parity, bool doit, volatile int* go,
                                           volatile int* abort_flag, long long limit,
                                           DeviceError* err, unsigned tag) {
    if (leader_warp) {
        const bool ok = !doit || mbar_wait(bar, parity, abort_flag, limit, err, tag);
        if (lane0) *go = (ok && !*abort_flag) ? 1 : 0;
    }
    named_bar<ID, N>();
    __syncwarp();   // the leader warp diverged around its poll: reconverge before .aligned work
    return *go != 0;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// untiled bulk copy global -> shared, completing on an mbarrier (16-byte aligned, size a
// multiple of 16)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
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
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t tf32_bits(float x) {
    uint32_t y;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(y) : "f"(x));
    return y;
}

// A tf32 MMA operand rounded to nearest (ties away from zero) with one integer add: adding
// half a tf32 unit (bit 12) to the sign-magnitude fp32 pattern carries into the 19 bits the
// MMA reads, and the MMA ignores the low 13 bits, so they need no clearing. Same rounding as
// cvt.rna.tf32.f32, on the integer pipe instead of the conversion pipe.
__device__ __forceinline__ uint32_t tf32_operand(float x) { return __float_as_uint(x) + 0x1000u; }

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
// K-major operand: rows of 128 bytes packed in 8-row groups of 1024 bytes
__device__ __forceinline__ uint64_t desc_k(uint32_t saddr) { return sdesc(saddr, 16, 1024); }
// K-major operand without swizzle: 8-row x 16-byte core matrices `lbo` bytes apart along K,
// 8-row groups `sbo` bytes apart
__device__ __forceinline__ uint64_t desc_kn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}
// MN-major operand: 64-element blocks along M/N `mn_stride` bytes apart, 8-row groups along
// K 1024 bytes apart
__device__ __forceinline__ uint64_t desc_mn(uint32_t saddr, uint32_t mn_stride) {
    return sdesc(saddr, mn_stride, 1024);
}

// Instruction descriptors (dense, fp32 D). kind::f16 with bf16 A and B:
constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t ID_P1 = idesc_bf16(128, 64, false, false);
constexpr uint32_t ID_P23 = idesc_bf16(128, 64, true, false);
constexpr uint32_t ID_WY1 = idesc_bf16(128, 48, true, false);
constexpr uint32_t ID_WY2 = idesc_bf16(128, 32, true, false);
constexpr uint32_t ID_WY3 = idesc_bf16(128, 16, true, false);

constexpr uint32_t ID_S4 = idesc_bf16(128, 128, false, true);   // A from tensor memory
// kind::tf32, M = 128, N = 64, A from tensor memory, B K-major (S1, S2, S3)
constexpr uint32_t ID_TF = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(64 >> 3) << 17) |
                           ((uint32_t)(128 >> 4) << 24);
// kind::tf32, M = 128, N = 128 (the forward's fused R^T | O^T product)
constexpr uint32_t ID_TF128 = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(128 >> 3) << 17) |
                              ((uint32_t)(128 >> 4) << 24);

// The instruction descriptor is an immediate (template argument): the issuing thread then
// spends no instructions moving it into place, which keeps back-to-back MMAs from being
// issue-bound.
template <uint32_t ID>
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "n"(ID), "r"(accumulate)
        : "memory");
}

// D^T = X^T F^T for a WY factor F (format at kWyTileBytes in gdn_internal.h) and a 64-row
// operand X whose transpose is the MN-major A operand at `a` (two 64-feature halves 8192
// bytes apart): four MMAs, the one for columns 16 s .. 16 s + 15 of F over F's rows
// 16 s .. 63 only (N = 64 - 16 s, into accumulator columns 16 s ..); the first initialises
// all 64 columns
__device__ __forceinline__ void wy_mma(uint32_t d_tmem, uint32_t a, uint32_t tile) {
    mma_ss<ID_P23>(d_tmem, desc_mn(a, 8192), desc_kn(tile + wy_slab0(0), wy_slab_lbo(0), 128), 0u);
    mma_ss<ID_WY1>(d_tmem + 16, desc_mn(a + 2048, 8192), desc_kn(tile + wy_slab0(1), wy_slab_lbo(1), 128), 1u);
    mma_ss<ID_WY2>(d_tmem + 32, desc_mn(a + 4096, 8192), desc_kn(tile + wy_slab0(2), wy_slab_lbo(2), 128), 1u);
    mma_ss<ID_WY3>(d_tmem + 48, desc_mn(a + 6144, 8192), desc_kn(tile + wy_slab0(3), wy_slab_lbo(3), 128), 1u);
}

template <uint32_t ID>
__device__ __forceinline__ void mma_ts_tf32(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "n"(ID), "r"(accumulate)
        : "memory");
}

template <uint32_t ID>
__device__ __forceinline__ void mma_ts_bf16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "n"(ID), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Tensor-memory accesses of this thread's lane: 16 or 8 consecutive 32-bit columns. The
// kernel walks wide rows in rolled loops over such groups: each chunk executes its code
// once, so compact loops (rather than fully unrolled rows) keep it in the instruction cache.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
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

// byte address of 16-byte chunk `c` of row `row` in a 128-byte-swizzled tile of 128-byte rows
__device__ __forceinline__ uint32_t sw128(int row, int c) {
    return (row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4);
}

__device__ __forceinline__ float bf16_at(const void* base, long long idx) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
}

// 64 x 64 fp32 matrices of the inverse: row-major with the column XOR-swizzled by the row,
// so both row-wise and column-wise walks by a warp hit 32 distinct banks
__device__ __forceinline__ int sw64(int i, int j) { return i * 64 + (j ^ (i & 31)); }

// D = A B + D on the warp-level tensor path, m16n8k8, tf32 in, fp32 accumulate
__device__ __forceinline__ void mma_m16n8k8(float* d, const uint32_t* a, const uint32_t* b) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// m16n8k8 fragments from swizzled fp32 64x64 matrices (rows r0.., cols c0..)
__device__ __forceinline__ void frag_a(const float* M, int r0, int c0, int lane, uint32_t* a) {
    const int g = lane >> 2, t = lane & 3;
    a[0] = tf32_bits(M[sw64(r0 + g, c0 + t)]);
    a[1] = tf32_bits(M[sw64(r0 + g + 8, c0 + t)]);
    a[2] = tf32_bits(M[sw64(r0 + g, c0 + t + 4)]);
    a[3] = tf32_bits(M[sw64(r0 + g + 8, c0 + t + 4)]);
}
__device__ __forceinline__ void frag_b(const float* M, int r0, int c0, int lane, uint32_t* b) {
    const int g = lane >> 2, t = lane & 3;
    b[0] = tf32_bits(M[sw64(r0 + t, c0 + g)]);
    b[1] = tf32_bits(M[sw64(r0 + t + 4, c0 + g)]);
}

// ------------------------------------------------------------------------------------
// host side: the tensor-map encoder from the driver, looked up once
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

// [B*T, H, 128] bf16 (a packed varlen batch: [T, H, 128]) viewed as a 3-d tensor; box = 64
// features x 1 head x 64 tokens
bool make_map(CUtensorMap* m, const void* ptr, const ChainParams& c) {
    constexpr int kD = 128;
    auto fn = encode_fn();
    if (!fn || !ptr) return false;
    const cuuint64_t rows = c.cu_seqlens ? (cuuint64_t)c.T : (cuuint64_t)c.B * (cuuint64_t)c.T;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)c.H, rows};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)c.H * kD * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace gdn
