// Shared helpers of libmoe.so: status reporting, launch accounting, number
// conversions and the sm_103a PTX wrappers (mbarrier, TMA, tcgen05) the grouped
// GEMMs are built from.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <string>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// host side: status, messages, launch accounting
// ---------------------------------------------------------------------------

int fail(int status, const char* fmt, ...);          // records the message, returns status
int check_launch(const char* what);                    // cudaGetLastError after a launch
void count_launch(uint64_t n = 1);                     // kernels this library launched
int sm_count();                                        // SMs of the current device
int set_smem_limit(const void* kernel, int bytes);     // opt in to > 48 KB dynamic smem
uint64_t wait_limit_ns();                              // pipeline wait limit for the next launches
uint32_t next_splitk_gen();                            // nonzero split-K generation for the next GEMM call

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define MOE_REQUIRE(cond, ...)                                   \
    do {                                                         \
        if (!(cond)) return ::moe::fail(MOE_ERR_INVALID, __VA_ARGS__); \
    } while (0)

// Encode a 2-D bf16/fp16 tensor map: rows x cols (cols contiguous), box
// box_rows x 64 elements (128 bytes, the 128-byte swizzle span).
int make_tmap_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows, int act);
// Encode a plain (unswizzled) 2-D tensor map of any element type: rows x cols
// elements of elem_bytes each, box box_rows x box_cols.
int make_tmap_2d_raw(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t rows,
                     uint64_t cols, uint32_t box_cols, uint32_t box_rows);
// Encode a plain 3-D tensor map: dims d0 (contiguous) x d1 x d2 elements,
// byte strides s1 (between d1 steps) and s2 (between d2 steps), box
// b0 x b1 x b2. Used to fetch two separated halves of a weight tile with one
// copy.
int make_tmap_3d_raw(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t d0,
                     uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2);
// Encode a 5-D bf16/fp16 tensor map with the 128-byte swizzle: dims d[0]
// (contiguous; a box of 64 elements = 128 bytes) to d[4], byte strides st of
// dims 1..4, box b.
int make_tmap_5d(CUtensorMap* map, const void* base, int act, const uint64_t (&d)[5], const uint64_t (&st)[4],
                 const uint32_t (&b)[5]);

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel in the stream is still finishing (its launch and
// CTA set-up overlap that kernel's tail). Every kernel of this library starts
// with pdl_wait(), which blocks until the previous kernel has completed and
// its writes are visible, so the order of the steps is unchanged. Inside a
// captured CUDA graph the dependency becomes a programmatic edge.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ---------------------------------------------------------------------------
// device side
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The 1024-byte aligned start of the dynamic shared memory. Derived from the
// shared array by pointer arithmetic (not through an integer), so the
// compiler keeps the shared address space and emits shared-memory loads and
// stores for everything addressed from it.
__device__ __forceinline__ uint8_t* align1024_shared(uint8_t* base) {
    return base + ((1024u - (smem_u32(base) & 1023u)) & 1023u);
}

// Programmatic dependent launch, device side. pdl_wait: block until the
// kernels this grid depends on have completed and their memory is visible
// (a no-op for a grid launched without the attribute). Called first in every
// kernel, by every thread, before any global memory is touched, so a kernel
// also completes only after its predecessor did. pdl_launch_next: allow the
// next kernel in the stream to be scheduled now rather than when this one's
// CTAs have exited. Only the activation gather calls it (the GEMM after it
// then sets up while the gather runs); triggering early in every kernel
// measured slower on decode-sized layers (fine-grained T=8 72.7 -> 77 us).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void set_err(int32_t* err, int bits) {
    if (err) atomicOr(err, bits);
}

// activation element conversions (ACT = MOE_ACT_BF16 | MOE_ACT_F16)
template <int ACT> struct Act;
template <> struct Act<MOE_ACT_BF16> {
    using T = __nv_bfloat16;
    using T2 = __nv_bfloat162;
    static __device__ __forceinline__ float to_f(T v) { return __bfloat162float(v); }
    static __device__ __forceinline__ T from_f(float v) { return __float2bfloat16_rn(v); }
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        T2 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    static __device__ __forceinline__ float2 unpack2(uint32_t u) {
        T2 v = *reinterpret_cast<T2*>(&u);
        return __bfloat1622float2(v);
    }
};
template <> struct Act<MOE_ACT_F16> {
    using T = __half;
    using T2 = __half2;
    static __device__ __forceinline__ float to_f(T v) { return __half2float(v); }
    static __device__ __forceinline__ T from_f(float v) { return __float2half_rn(v); }
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        T2 v = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    static __device__ __forceinline__ float2 unpack2(uint32_t u) {
        T2 v = *reinterpret_cast<T2*>(&u);
        return __half22float2(v);
    }
};

// ---- mbarrier -------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// The same test, but a thread whose phase is not complete is suspended until
// it completes or hint_ns nanoseconds pass, instead of returning at once: a
// waiting warp then takes no issue slots from the warps that share its
// sub-partition.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
// longest suspension of one try_wait in a bounded wait: how long another
// role's abort can go unnoticed
constexpr uint64_t kWaitSleepNs = 200000ull;

// How long a pipeline wait may last, by default, before the kernel gives up
// (the whole layer at the largest supported size runs in a few
// milliseconds). Each launch carries its own limit (WaitCtx::limit_ns); the
// host takes it from wait_limit_ns().
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// What a bounded wait needs: the CTA's abort flag (raised by whichever role
// gives up first, so the others stop waiting too), the device error word and
// the launch's time limit.
struct WaitCtx {
    volatile int* abort;
    int32_t* err;
    uint64_t limit_ns;
};

// Wait for the phase of `bar` with parity `parity` to complete. Gives up
// (returns false) when the CTA's abort flag is raised by another role, or
// after w.limit_ns, in which case it raises the flag itself and records
// MOE_DEV_ERR_TIMEOUT in the error word.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    const uint32_t sleep = static_cast<uint32_t>(w.limit_ns < kWaitSleepNs ? w.limit_ns : kWaitSleepNs);
    while (true) {
        if (mbar_try_wait_sleep(a, parity, sleep)) return true;
        if (*w.abort) return false;
        if (globaltimer_ns() - t0 > w.limit_ns) {
            *w.abort = 1;
            set_err(w.err, MOE_DEV_ERR_TIMEOUT);
            return false;
        }
    }
}

// Flags in global memory that one CTA raises for another within a launch.
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait until the global flag *f holds v, with the same limit and abort rule
// as mbar_wait. Every calling thread observes the flag itself (acquire), so
// each sees the data released before it.
__device__ __forceinline__ bool flag_wait(const int* f, int v, const WaitCtx& w) {
    if (ld_acquire_gpu(f) == v) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (ld_acquire_gpu(f) == v) return true;
        if (*w.abort) return false;
        if (globaltimer_ns() - t0 > w.limit_ns) {
            *w.abort = 1;
            set_err(w.err, MOE_DEV_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(64);
    }
}

// Bounded wait that ignores the abort flag: used on the way out to let copies
// already in flight land before the CTA exits.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(a, parity, static_cast<uint32_t>(kWaitSleepNs))) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// ---- clusters (CTA pairs) ------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// shared::cluster address of the same shared-memory location in CTA `rank`
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// The same arrival without release semantics, for a signal whose payload the
// thread has already completed by a blocking wait (TMEM written by
// tcgen05.st and waited for with tcgen05.wait::st): a release at cluster
// scope measured 0.3 - 1.4 us per arrival on this path, the relaxed form a
// few cycles.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the two halves of cluster_sync_all, for work between the arrival and the wait
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- cp.async (global -> shared, no register round trip) -----------------------
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// 16 bytes when `full`, else 16 zero bytes (src is not read then, but must be a valid address)
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, bool full) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(full ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// wait until at most N of this thread's committed groups are still in flight
template <int N> __device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---- ldmatrix: 8x8 b16 matrices from shared memory in mma.sync fragment order ----
// Lanes 8i .. 8i + 7 give the row addresses (16-byte aligned) of matrix i;
// lane l receives row l / 4, columns 2 (l % 4) and 2 (l % 4) + 1 of each.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x2(uint32_t (&r)[2], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}

// ---- TMA ------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}
// TMA load of a CTA pair: the data lands in this CTA's shared memory and the
// byte count completes on `bar_cluster`, which may be the peer CTA's barrier
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster)
        : "memory");
}
__device__ __forceinline__ void tma_load_5d_pair(void* dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                                 int32_t c2, int32_t c3, int32_t c4, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar_cluster)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int32_t c0, int32_t c1, int32_t c2,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// make generic-proxy shared-memory writes visible to the async proxy (the
// tensor cores read operands through it)
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- tcgen05 (5th-generation tensor cores, accumulators in TMEM) -----------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, both operands K-major, kind::f16
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// CTA-pair forms: the allocation / release is collective (one warp of each
// peer CTA), the MMA is issued by one thread of the pair, and its commit
// arrives on the barrier at the same offset in each CTA of `mask`
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16: A (M=128 rows x K=16) sits in
// TMEM with row m in lane m and the 16-bit elements (2c, 2c+1) of row m in
// column c, so one K=16 step reads 8 consecutive columns
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// CTA-pair TS form: D[tmem] (+)= A[tmem] * B[smem]^T with M = 256, each CTA
// of the pair holding its 128 rows of A at a_tmem in its own TMEM (layout as
// for tc_mma_ts) and its half of B's rows at the same shared-memory offset;
// issued by one thread of the pair
__device__ __forceinline__ void tc_mma_pair_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive on `bar` once every tcgen05 op this thread issued so far completes
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (taddr.lane + i), columns [taddr.col, taddr.col + 32)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Wait for this thread's TMEM loads and tie the registers of r to the wait:
// tcgen05.ld writes its destination registers asynchronously, and the empty
// asm statements (ordered after the wait, with r as in/out operands) keep the
// compiler from reading or moving r before it.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(r[i]));
}
// 32 lanes x 32 consecutive 32-bit columns from registers: thread i of the
// warp writes lane (taddr.lane + i), columns [taddr.col, taddr.col + 32)
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with the 128-byte swizzle: rows of 128 bytes (64 16-bit elements), 8-row
// groups 1024 bytes apart (stride byte offset), tile base 1024-byte aligned.
// Fields: start address >> 4 (bits 0-13), leading byte offset >> 4 (16-29,
// unused for swizzled K-major), stride byte offset >> 4 (32-45), descriptor
// version 1 (46-47), base offset 0 (49-51), swizzle mode 2 = 128B (61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor of kind::f16 with f32 accumulation, A and B K-major.
// Fields: D format (bits 4-5: 1 = f32), A format (7-9) and B format (10-12):
// 0 = f16, 1 = bf16; N >> 3 (17-22); M >> 4 (24-28).
__host__ __device__ constexpr uint32_t f16_idesc(int act, int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(act == MOE_ACT_BF16 ? 1 : 0) << 7) |
           (static_cast<uint32_t>(act == MOE_ACT_BF16 ? 1 : 0) << 10) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

}  // namespace moe
