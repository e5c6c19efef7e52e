// common.cuh -- shared device helpers of libaqpq (sm_103a).
//
// Inline-PTX wrappers used by the kernels: mbarriers (init / expect-tx /
// bounded try-wait), the bulk copy engine (global -> shared, and shared -> a
// peer CTA's shared memory, completion counted in bytes on an mbarrier),
// per-thread cp.async copies, cluster barriers and addressing, packed fp32
// pair arithmetic, programmatic dependent launch, tcgen05 tensor-core MMAs
// with TMEM accumulators.  Every wait here is bounded
// in wall-clock time: a wait that runs out returns false, and the caller
// records AQ_DEV_TIMEOUT instead of hanging.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "aqpq.h"

namespace aq {

constexpr int kHeadDim = 128;
constexpr int kCodewords = 256;
constexpr int kPage = 16;
// 200 ms: far above any legitimate copy, far below a watchdog.
constexpr unsigned long long kWaitLimitNs = 200ull * 1000ull * 1000ull;
// Longest suspension one mbarrier try-wait asks for (1 ms).
constexpr uint32_t kSuspendHintNs = 1000000u;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrive once and add `bytes` to the transaction count of the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

// Arrive once on `bar` (release: this thread's earlier shared-memory writes
// are visible to whoever waits for the phase).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}

// Test phase `parity` of `bar`; a thread whose phase is still open is
// suspended (up to kSuspendHintNs) until it completes instead of spinning.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// Test phase `parity` of `bar` without suspending.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete; false once `limit_ns` has
// passed.  Limits below 100 us poll without suspending, so that a short limit
// (the host-settable one of the decode kernels, lowered to test the timeout
// path) is honoured.
__device__ __forceinline__ bool mbar_wait_limit(uint64_t *bar, uint32_t parity, unsigned long long limit_ns) {
    const bool poll = limit_ns < 100000ull;
    if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
        if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Wait for phase `parity` of `bar` to complete; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    return mbar_wait_limit(bar, parity, kWaitLimitNs);
}

// Bulk copy `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global to this CTA's shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// TMA tensor copy of one box of a 2-D tensor map (x = innermost element
// coordinate, y = row) to this CTA's shared memory; completion is counted in
// bytes on `bar`.  `map` is the address of a __grid_constant__ kernel
// parameter.  The destination is aligned to the map's swizzle period.
__device__ __forceinline__ void tma_load_2d(void *dst_smem, const void *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 16-byte global -> shared copy through L2 (cp.async.cg): the destination is
// any 16-byte aligned shared address, so a copy can lay rows out in its own
// (swizzled) order.  Completion is tracked per thread.
__device__ __forceinline__ void cp_async_16(uint32_t dst_smem, const void *src_gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src_gmem) : "memory");
}

// Arrive on `bar` once every cp.async this thread has issued so far has
// landed; the arrival is one of the counts the barrier was initialised with.
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// 8-byte streaming load through the non-coherent path, not kept in L1 (data
// that no kernel writes while this one runs).
__device__ __forceinline__ uint2 ldg_stream_v2(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

// 8- / 16-byte loads through the coherent path, not kept in L1 (data that a
// preceding kernel may have written).
__device__ __forceinline__ uint2 ld_global_na_v2(const void *p) {
    uint2 v;
    asm volatile("ld.global.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_global_na_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void flag_status(int32_t *status, int32_t bits) {
    if (status) atomicOr(status, bits);
}

// Internal invariants, checked only in builds with AQ_DEBUG_CHECKS: a failed
// one sets AQ_DEV_INVARIANT in the status word (no trap, no early exit).
#ifdef AQ_DEBUG_CHECKS
#define AQ_DCHECK(status, cond)                                       \
    do {                                                              \
        if (!(cond)) ::aq::flag_status((status), AQ_DEV_INVARIANT);   \
    } while (0)
#else
#define AQ_DCHECK(status, cond) \
    do {                        \
    } while (0)
#endif

__device__ __forceinline__ float2 h2_to_f2(uint32_t u) {
    __half2 h = *reinterpret_cast<__half2 *>(&u);
    return __half22float2(h);
}

// ---- packed fp32 pairs (sm_100-family f32x2 arithmetic) ---------------------
// Each lane of a pair is rounded exactly as the scalar operation would be.
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float2 f2_unpack(unsigned long long v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return make_float2(lo, hi);
}

__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Two fp16 values (one 32-bit word) as a packed fp32 pair.
__device__ __forceinline__ unsigned long long h2_to_f2p(uint32_t u) {
    const float2 f = h2_to_f2(u);
    return f2_pack(f.x, f.y);
}

// 2^x by the hardware approximation (relative error about 2^-22; 2^-inf = 0,
// 2^0 = 1): the softmax weights need no more.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Warp-wide maximum of a float (all 32 lanes take part).
__device__ __forceinline__ float warp_max_f32(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// ---- thread-block cluster helpers ------------------------------------------
// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_u32(uint32_t local_smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem_addr), "r"(rank));
    return r;
}

// Bulk copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from
// this CTA's shared memory to a shared-memory address of the cluster (from
// mapa_u32); the bytes are counted on the destination CTA's mbarrier, given
// as a cluster address.  Writes to the source by the generic proxy must be
// fenced (fence_proxy_async_shared) before the copy is issued.
__device__ __forceinline__ void bulk_s2cluster(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "r"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}

// Asynchronous store into a peer CTA's shared memory; the bytes are counted
// on the peer's mbarrier (complete_tx), which orders them for its waiters.
__device__ __forceinline__ void st_async_f32(uint32_t remote_addr, float v, uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(remote_addr),
        "f"(v), "r"(remote_bar)
        : "memory");
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Programmatic dependent launch: wait until the preceding kernel on the stream
// has completed and its memory is visible (returns at once when this kernel
// was not launched as its dependent); allow the next kernel to start launching.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}


// ---- warp-level tensor-core tiles (small fused contractions) -----------------
// Four 8x8 fp16 matrices from shared memory, transposed: lane l gives the row
// address of row l%8 of matrix l/8 (16 bytes each); register j of lane l then
// holds elements (2(l%4), l/4) and (2(l%4)+1, l/4) of matrix j, i.e. the
// m16n8k16 A fragment of the transposed 16x16 block when the matrices are
// (rows 0-7, cols 0-7), (rows 0-7, cols 8-15), (rows 8-15, cols 0-7),
// (rows 8-15, cols 8-15) of the stored block.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// The same four matrices untransposed: register j of lane l holds elements
// (l/4, 2(l%4)) and (l/4, 2(l%4)+1) of matrix j -- the A fragment when the
// matrices are (rows 0-7, cols 0-7), (rows 8-15, cols 0-7), (rows 0-7,
// cols 8-15), (rows 8-15, cols 8-15) of a row-major 16x16 block.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// d += A(16x16, fp16) * B(16x8, fp16) with fp32 accumulation, warp-wide.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two fp32 values as an fp16 pair (x in the low half) split into a rounded
// high part and the rounded remainder: x = hi + lo to about 22 bits.
__device__ __forceinline__ void f16x2_split(float x, float y, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x, y);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// ---- 5th-generation tensor cores (tcgen05) -----------------------------------
// One CTA (cta_group::1) allocates tensor memory (TMEM) columns, one thread
// issues MMAs whose operands sit in shared memory (described by 64-bit matrix
// descriptors) and whose fp32 accumulator lives in TMEM, and the warps read
// the accumulator back lane by lane.  Warp w of a warpgroup may only touch
// TMEM lanes [32(w%4), 32(w%4)+32).

// Allocate `ncols` (a power of two >= 32) TMEM columns; the base address is
// written to shared memory.  Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Release what tmem_alloc took (same warp, same column count).
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// Order tcgen05 operations around a thread synchronisation (barrier or
// mbarrier wait): `before` on the signalling side, `after` on the waiting side.
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, no swizzle: the operand is a grid of core
// matrices of 8 rows x 16 bytes (rows 16 bytes apart); `lbo` is the byte
// distance between core matrices adjacent along K, `sbo` between core
// matrices adjacent along M (or N).  Bits 46-47 hold the descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
           (static_cast<uint64_t>(sbo >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B fp16, both
// K-major, tile M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n) {
    return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// Instruction descriptor of kind::tf32: fp32 accumulator, A and B tf32 (fp32
// in shared memory, 10 fraction bits used), both K-major, tile M x N.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int m, int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// D[tmem] (+)= A * B^T for one K = 16 step of fp16 operands (kind::f16: A and
// B both fp16, descriptor from idesc_f16_f32); `accumulate` = 0 overwrites D.
__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same for one K = 8 step of tf32 operands (kind::tf32, descriptor from
// idesc_tf32_f32).
__device__ __forceinline__ void umma_tf32(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape); the
// registers are valid after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Three-input maximum (NaN inputs are ignored unless all are NaN).
__device__ __forceinline__ float max3_f32(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Three-input minimum (NaN inputs are ignored unless all are NaN).
__device__ __forceinline__ float min3_f32(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

}  // namespace aq
