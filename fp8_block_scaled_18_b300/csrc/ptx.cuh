// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA tensor loads,
// tcgen05 (TMEM allocation, MMA, commit, loads, fences) and the e4m3
// conversions.  Written from the public PTX ISA description of each
// instruction; every wait here is bounded (see bounded_wait below).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8bs {

// Device status bits (the library's status word; read by fp8bs_sync_status).
enum : unsigned {
    DEVERR_WAIT_TIMEOUT = 1u,   // a pipeline wait gave up
    DEVERR_SELFTEST = 2u        // the debug self-test wait gave up (expected)
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Shared control block of one CTA for bounded waits.
struct WaitCtl {
    volatile int* abort;     // shared memory: set once any wait of the CTA gives up
    unsigned* err;           // device status word
    uint64_t timeout_ns;     // per-wait limit
};

// Wait for the phase of `bar` with the given parity to complete.  Gives up
// when the CTA's abort flag is raised or after ctl.timeout_ns; on its own
// timeout it raises the abort flag and records DEVERR_WAIT_TIMEOUT.
// Returns false when it gave up.
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 0) {
            if (*ctl.abort) return false;
            if (globaltimer_ns() - t0 > ctl.timeout_ns) {
                *ctl.abort = 1;
                atomicOr(ctl.err, DEVERR_WAIT_TIMEOUT);
                return false;
            }
        }
    }
}

// Warp-uniform form of bounded_wait: every lane polls, and the warp proceeds
// only if all lanes saw the phase complete (a lane that gave up makes the
// whole warp give up).  Also reconverges the warp before the .sync.aligned
// tcgen05 instructions that follow a wait.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
    const bool ok = bounded_wait(bar, parity, ctl);
    return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------- thread-block clusters

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared::cluster address of `addr` (a shared::cta address of this CTA)
// in the CTA of the cluster with the given rank.
__device__ __forceinline__ uint32_t mapa_rank(uint32_t addr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
    return d;
}
// All threads of every CTA of the cluster: after barrier initialisation
// (before any CTA touches another's shared memory) and before exit (no CTA
// leaves while a peer may still read or write its shared memory).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ int32_t ld_cluster_s32(uint32_t cluster_addr) {
    int32_t v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
    return v;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t cluster_addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_cluster_v4f32(uint32_t cluster_addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}

// ---------------------------------------------------------------- programmatic dependent launch

// A kernel launched with programmatic stream serialisation may start while
// the previous kernel in its stream is still running.  grid_dependency_wait()
// returns once that kernel has completed and its memory is visible, so it
// must come before the kernel's first global-memory access (read or write)
// and before it claims any resource the previous kernel might still need
// (TMEM).  allow_dependents() lets the next such kernel start its prologue.
// Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled bulk tensor load global -> shared, completion counted in bytes on `bar`.
// c0 is the innermost (contiguous) coordinate in elements, c1 the row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int32_t c0,
                                            int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

// 2-D tiled bulk tensor store shared -> global of one box at (c0, c1);
// elements of the box outside the tensor are not written.  Tracked by the
// executing thread's bulk async-groups (bulk_commit_group / bulk_wait_*).
__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src, int32_t c0, int32_t c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed bulk groups are still
// reading their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until at most N of this thread's committed bulk groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Order this thread's earlier shared-memory writes before later async-proxy
// (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05

// Allocate `ncols` TMEM columns (power of two >= 32) for this CTA; the TMEM
// address is written to shared memory at `dst`.  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
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

// Shared-memory matrix descriptor for a K-major operand tile stored the way
// TMA writes it with 128-byte swizzling: rows of 128 bytes, 8-row groups of
// 1024 bytes.  Fields: start address >> 4 (bits 0-13), leading byte offset
// >> 4 (16-29; unused by swizzled K-major layouts, set to 1), stride byte
// offset >> 4 (32-45) = 1024 B between 8-row groups, descriptor version 1
// (bits 46-47), base offset 0 (tile 1024-byte aligned), swizzle mode 2 =
// 128-byte (bits 61-63).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma.kind::f8f6f4 with fp32 accumulate,
// A = B = e4m3, both K-major, shape M x N (x K = 32).  Bits: D format (4-5) =
// 1 (f32); A format (7-9) = 0 (e4m3); B format (10-12) = 0 (e4m3); A/B
// negate/transpose 0; N >> 3 at bits 17-22; M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Load 16 consecutive fp32 TMEM columns of this warp's 32 lanes as 8
// packed pairs (column 2j in the low half of p[j]) and wait for them.
__device__ __forceinline__ void tmem_ld_x16_pairs(uint32_t taddr, uint64_t (&p)[8]) {
    asm volatile(
        "{\n\t.reg .b32 t<16>;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {t0,t1,t2,t3,t4,t5,t6,t7,t8,t9,t10,t11,t12,t13,t14,t15}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {t0, t1};\n\t"
        "mov.b64 %1, {t2, t3};\n\t"
        "mov.b64 %2, {t4, t5};\n\t"
        "mov.b64 %3, {t6, t7};\n\t"
        "mov.b64 %4, {t8, t9};\n\t"
        "mov.b64 %5, {t10, t11};\n\t"
        "mov.b64 %6, {t12, t13};\n\t"
        "mov.b64 %7, {t14, t15};\n\t"
        "}"
        : "=l"(p[0]), "=l"(p[1]), "=l"(p[2]), "=l"(p[3]), "=l"(p[4]), "=l"(p[5]), "=l"(p[6]), "=l"(p[7])
        : "r"(taddr)
        : "memory");
}

// acc[j] += f2 * cur[j] on packed fp32 pairs (fma.rn.f32x2: two IEEE
// fused multiply-adds) while the next 16 TMEM columns load into nxt; the
// load is waited for before the block ends, so nxt is complete on return.
__device__ __forceinline__ void tmem_ld_x16_pairs_fma(uint32_t taddr_next, uint64_t (&nxt)[8], uint64_t (&acc)[8],
                                                      const uint64_t (&cur)[8], uint64_t f2) {
    asm volatile(
        "{\n\t.reg .b32 t<16>;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {t0,t1,t2,t3,t4,t5,t6,t7,t8,t9,t10,t11,t12,t13,t14,t15}, [%25];\n\t"
        "fma.rn.f32x2 %8, %24, %16, %8;\n\t"
        "fma.rn.f32x2 %9, %24, %17, %9;\n\t"
        "fma.rn.f32x2 %10, %24, %18, %10;\n\t"
        "fma.rn.f32x2 %11, %24, %19, %11;\n\t"
        "fma.rn.f32x2 %12, %24, %20, %12;\n\t"
        "fma.rn.f32x2 %13, %24, %21, %13;\n\t"
        "fma.rn.f32x2 %14, %24, %22, %14;\n\t"
        "fma.rn.f32x2 %15, %24, %23, %15;\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {t0, t1};\n\t"
        "mov.b64 %1, {t2, t3};\n\t"
        "mov.b64 %2, {t4, t5};\n\t"
        "mov.b64 %3, {t6, t7};\n\t"
        "mov.b64 %4, {t8, t9};\n\t"
        "mov.b64 %5, {t10, t11};\n\t"
        "mov.b64 %6, {t12, t13};\n\t"
        "mov.b64 %7, {t14, t15};\n\t"
        "}"
        : "=l"(nxt[0]), "=l"(nxt[1]), "=l"(nxt[2]), "=l"(nxt[3]), "=l"(nxt[4]), "=l"(nxt[5]), "=l"(nxt[6]), "=l"(nxt[7]), "+l"(acc[0]), "+l"(acc[1]), "+l"(acc[2]), "+l"(acc[3]), "+l"(acc[4]), "+l"(acc[5]), "+l"(acc[6]), "+l"(acc[7])
        : "l"(cur[0]), "l"(cur[1]), "l"(cur[2]), "l"(cur[3]), "l"(cur[4]), "l"(cur[5]), "l"(cur[6]), "l"(cur[7]), "l"(f2), "r"(taddr_next)
        : "memory");
}

// acc[j] += f2 * cur[j] on 8 packed fp32 pairs.
__device__ __forceinline__ void fma_pairs(uint64_t (&acc)[8], const uint64_t (&cur)[8], uint64_t f2) {
    asm volatile(
        "fma.rn.f32x2 %0, %16, %8, %0;\n\t"
        "fma.rn.f32x2 %1, %16, %9, %1;\n\t"
        "fma.rn.f32x2 %2, %16, %10, %2;\n\t"
        "fma.rn.f32x2 %3, %16, %11, %3;\n\t"
        "fma.rn.f32x2 %4, %16, %12, %4;\n\t"
        "fma.rn.f32x2 %5, %16, %13, %5;\n\t"
        "fma.rn.f32x2 %6, %16, %14, %6;\n\t"
        "fma.rn.f32x2 %7, %16, %15, %7;\n\t"
        ""
        : "+l"(acc[0]), "+l"(acc[1]), "+l"(acc[2]), "+l"(acc[3]), "+l"(acc[4]), "+l"(acc[5]), "+l"(acc[6]), "+l"(acc[7])
        : "l"(cur[0]), "l"(cur[1]), "l"(cur[2]), "l"(cur[3]), "l"(cur[4]), "l"(cur[5]), "l"(cur[6]), "l"(cur[7]), "l"(f2));
}

// Load 64 consecutive fp32 TMEM columns of this warp's 32 lanes (one
// wait for all the loads) as 32 packed pairs.
__device__ __forceinline__ void tmem_ld_cols_pairs(uint32_t taddr, uint64_t (&p)[32]) {
    asm volatile(
        "{\n\t.reg .b32 t<64>;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t0,t1,t2,t3,t4,t5,t6,t7,t8,t9,t10,t11,t12,t13,t14,t15,t16,t17,t18,t19,t20,t21,t22,t23,t24,t25,t26,t27,t28,t29,t30,t31}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t32,t33,t34,t35,t36,t37,t38,t39,t40,t41,t42,t43,t44,t45,t46,t47,t48,t49,t50,t51,t52,t53,t54,t55,t56,t57,t58,t59,t60,t61,t62,t63}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {t0, t1};\n\t"
        "mov.b64 %1, {t2, t3};\n\t"
        "mov.b64 %2, {t4, t5};\n\t"
        "mov.b64 %3, {t6, t7};\n\t"
        "mov.b64 %4, {t8, t9};\n\t"
        "mov.b64 %5, {t10, t11};\n\t"
        "mov.b64 %6, {t12, t13};\n\t"
        "mov.b64 %7, {t14, t15};\n\t"
        "mov.b64 %8, {t16, t17};\n\t"
        "mov.b64 %9, {t18, t19};\n\t"
        "mov.b64 %10, {t20, t21};\n\t"
        "mov.b64 %11, {t22, t23};\n\t"
        "mov.b64 %12, {t24, t25};\n\t"
        "mov.b64 %13, {t26, t27};\n\t"
        "mov.b64 %14, {t28, t29};\n\t"
        "mov.b64 %15, {t30, t31};\n\t"
        "mov.b64 %16, {t32, t33};\n\t"
        "mov.b64 %17, {t34, t35};\n\t"
        "mov.b64 %18, {t36, t37};\n\t"
        "mov.b64 %19, {t38, t39};\n\t"
        "mov.b64 %20, {t40, t41};\n\t"
        "mov.b64 %21, {t42, t43};\n\t"
        "mov.b64 %22, {t44, t45};\n\t"
        "mov.b64 %23, {t46, t47};\n\t"
        "mov.b64 %24, {t48, t49};\n\t"
        "mov.b64 %25, {t50, t51};\n\t"
        "mov.b64 %26, {t52, t53};\n\t"
        "mov.b64 %27, {t54, t55};\n\t"
        "mov.b64 %28, {t56, t57};\n\t"
        "mov.b64 %29, {t58, t59};\n\t"
        "mov.b64 %30, {t60, t61};\n\t"
        "mov.b64 %31, {t62, t63};\n\t"
        "}"
        : "=l"(p[0]), "=l"(p[1]), "=l"(p[2]), "=l"(p[3]), "=l"(p[4]), "=l"(p[5]), "=l"(p[6]), "=l"(p[7]), "=l"(p[8]), "=l"(p[9]), "=l"(p[10]), "=l"(p[11]), "=l"(p[12]), "=l"(p[13]), "=l"(p[14]), "=l"(p[15]), "=l"(p[16]), "=l"(p[17]), "=l"(p[18]), "=l"(p[19]), "=l"(p[20]), "=l"(p[21]), "=l"(p[22]), "=l"(p[23]), "=l"(p[24]), "=l"(p[25]), "=l"(p[26]), "=l"(p[27]), "=l"(p[28]), "=l"(p[29]), "=l"(p[30]), "=l"(p[31])
        : "r"(taddr + 0u), "r"(taddr + 32u)
        : "memory");
}

// Load 80 consecutive fp32 TMEM columns of this warp's 32 lanes (one
// wait for all the loads) as 40 packed pairs.
__device__ __forceinline__ void tmem_ld_cols_pairs(uint32_t taddr, uint64_t (&p)[40]) {
    asm volatile(
        "{\n\t.reg .b32 t<80>;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t0,t1,t2,t3,t4,t5,t6,t7,t8,t9,t10,t11,t12,t13,t14,t15,t16,t17,t18,t19,t20,t21,t22,t23,t24,t25,t26,t27,t28,t29,t30,t31}, [%40];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t32,t33,t34,t35,t36,t37,t38,t39,t40,t41,t42,t43,t44,t45,t46,t47,t48,t49,t50,t51,t52,t53,t54,t55,t56,t57,t58,t59,t60,t61,t62,t63}, [%41];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {t64,t65,t66,t67,t68,t69,t70,t71,t72,t73,t74,t75,t76,t77,t78,t79}, [%42];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {t0, t1};\n\t"
        "mov.b64 %1, {t2, t3};\n\t"
        "mov.b64 %2, {t4, t5};\n\t"
        "mov.b64 %3, {t6, t7};\n\t"
        "mov.b64 %4, {t8, t9};\n\t"
        "mov.b64 %5, {t10, t11};\n\t"
        "mov.b64 %6, {t12, t13};\n\t"
        "mov.b64 %7, {t14, t15};\n\t"
        "mov.b64 %8, {t16, t17};\n\t"
        "mov.b64 %9, {t18, t19};\n\t"
        "mov.b64 %10, {t20, t21};\n\t"
        "mov.b64 %11, {t22, t23};\n\t"
        "mov.b64 %12, {t24, t25};\n\t"
        "mov.b64 %13, {t26, t27};\n\t"
        "mov.b64 %14, {t28, t29};\n\t"
        "mov.b64 %15, {t30, t31};\n\t"
        "mov.b64 %16, {t32, t33};\n\t"
        "mov.b64 %17, {t34, t35};\n\t"
        "mov.b64 %18, {t36, t37};\n\t"
        "mov.b64 %19, {t38, t39};\n\t"
        "mov.b64 %20, {t40, t41};\n\t"
        "mov.b64 %21, {t42, t43};\n\t"
        "mov.b64 %22, {t44, t45};\n\t"
        "mov.b64 %23, {t46, t47};\n\t"
        "mov.b64 %24, {t48, t49};\n\t"
        "mov.b64 %25, {t50, t51};\n\t"
        "mov.b64 %26, {t52, t53};\n\t"
        "mov.b64 %27, {t54, t55};\n\t"
        "mov.b64 %28, {t56, t57};\n\t"
        "mov.b64 %29, {t58, t59};\n\t"
        "mov.b64 %30, {t60, t61};\n\t"
        "mov.b64 %31, {t62, t63};\n\t"
        "mov.b64 %32, {t64, t65};\n\t"
        "mov.b64 %33, {t66, t67};\n\t"
        "mov.b64 %34, {t68, t69};\n\t"
        "mov.b64 %35, {t70, t71};\n\t"
        "mov.b64 %36, {t72, t73};\n\t"
        "mov.b64 %37, {t74, t75};\n\t"
        "mov.b64 %38, {t76, t77};\n\t"
        "mov.b64 %39, {t78, t79};\n\t"
        "}"
        : "=l"(p[0]), "=l"(p[1]), "=l"(p[2]), "=l"(p[3]), "=l"(p[4]), "=l"(p[5]), "=l"(p[6]), "=l"(p[7]), "=l"(p[8]), "=l"(p[9]), "=l"(p[10]), "=l"(p[11]), "=l"(p[12]), "=l"(p[13]), "=l"(p[14]), "=l"(p[15]), "=l"(p[16]), "=l"(p[17]), "=l"(p[18]), "=l"(p[19]), "=l"(p[20]), "=l"(p[21]), "=l"(p[22]), "=l"(p[23]), "=l"(p[24]), "=l"(p[25]), "=l"(p[26]), "=l"(p[27]), "=l"(p[28]), "=l"(p[29]), "=l"(p[30]), "=l"(p[31]), "=l"(p[32]), "=l"(p[33]), "=l"(p[34]), "=l"(p[35]), "=l"(p[36]), "=l"(p[37]), "=l"(p[38]), "=l"(p[39])
        : "r"(taddr + 0u), "r"(taddr + 32u), "r"(taddr + 64u)
        : "memory");
}

__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float lo_f32(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi_f32(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }

// ---------------------------------------------------------------- e4m3

// Two fp32 -> packed e4m3x2, round to nearest-even, saturating to +-448
// (NaN -> NaN).  Byte 0 of the result encodes `lo`, byte 1 encodes `hi`.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Packed e4m3x2 -> two fp32 (exact: e4m3 is a subset of f16).
__device__ __forceinline__ float2 cvt_e4m3x2_to_f32(uint16_t v) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    __half2 h = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(h);
}

}  // namespace fp8bs
