// hf_ptx.cuh -- inline-PTX building blocks for sm_103a kernels: mbarriers
// with bounded waits, TMA (cp.async.bulk[.tensor]), tcgen05 MMA / TMEM
// access, and the shared-memory and instruction descriptors they take.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "hf_internal.h"

namespace hf {

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before the previous kernel on its stream has
// finished; griddep_wait() blocks until that kernel has completed and its
// memory operations are visible (a no-op without such a dependency), and
// griddep_launch_dependents() lets the next kernel start once every CTA of
// this one has called it or exited.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Shared abort flag + device status word used by every bounded wait of a CTA.
struct WaitCtl {
    volatile uint32_t* abort_flag;   // shared memory, per CTA
    uint32_t* status;                // global: [0] = first error code, [1] = site
    uint64_t limit_ns;
};

// Load with acquire semantics at GPU scope: the writes another CTA made before
// its release (a fence, then the atomic that published them) are visible to
// this thread's later loads.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* ptr)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

__device__ __forceinline__ void report_error(const WaitCtl& w, uint32_t code, uint32_t site)
{
    *w.abort_flag = 1;
    if (atomicCAS(w.status, 0u, code) == 0u) atomicExch(w.status + 1, site);
}

// Waits for the phase with parity `parity` of `bar` to complete.  Gives up
// (returns false) when the CTA's abort flag is raised or after limit_ns, in
// which case it records HF_ERR_TIMEOUT with `site` and raises the flag.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtl& w, uint32_t site)
{
    const uint32_t addr = smem_u32(bar);
    if (mbar_try_wait(addr, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(addr, parity)) return true;
        if ((i & 63u) == 0u) {
            if (*w.abort_flag) return false;
            if (globaltimer_ns() - t0 > w.limit_ns) {
                report_error(w, HF_DEV_ERR_TIMEOUT, site);
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_read_all()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Plain (untiled) bulk copy global -> shared; 16-byte aligned, size % 16 == 0.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Generic-proxy writes to shared memory -> visible to the async proxy
// (tensor core reads of smem operands, TMA stores).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads/stores, fences
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_result, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Warp-wide forms: the whole (converged) warp executes them with the same
// operands and the lane that elect.sync picks (the same lane every time, with
// all 32 lanes active) issues the instruction.  Keeping the issuing warp
// converged lets the operands stay warp-uniform, which keeps the issue rate
// at the tensor core's pace while other warps of the sub-partition compute.
__device__ __forceinline__ void mma_ss_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// A whole K loop of tcgen05.mma (kind::f16, cta_group::1) in one block,
// issued by one elected lane of a converged warp.  A and B are K-major with
// the 128-byte swizzle: 16-element K steps are 32 bytes (2 descriptor units)
// apart inside a 64-element chunk, chunks CH descriptor units apart.  The
// first MMA accumulates into D iff `acc`, the others always.  NK = 4 or 8.
template <int NK, int CH>
__device__ __forceinline__ void mma_ss_kloop_warp(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    static_assert(NK == 4 || NK == 8, "K loop of 4 or 8 steps");
    if (NK == 4) {
        asm volatile(
            "{\n\t.reg .pred e, p, t;\n\t.reg .b64 ra, rb;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "setp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 t, %5, 0;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
            "add.s64 ra, %1, 2;\n\tadd.s64 rb, %2, 2;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
            "add.s64 ra, %1, 4;\n\tadd.s64 rb, %2, 4;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
            "add.s64 ra, %1, 6;\n\tadd.s64 rb, %2, 6;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t}"
            ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(1u)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred e, p, t;\n\t.reg .b64 ra, rb;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "setp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 t, %5, 0;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
            "add.s64 ra, %1, 2;\n\tadd.s64 rb, %2, 2;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
            "add.s64 ra, %1, 4;\n\tadd.s64 rb, %2, 4;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
            "add.s64 ra, %1, 6;\n\tadd.s64 rb, %2, 6;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
            "add.s64 ra, %1, %6;\n\tadd.s64 rb, %2, %6;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
            "add.s64 ra, %1, %7;\n\tadd.s64 rb, %2, %7;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
            "add.s64 ra, %1, %8;\n\tadd.s64 rb, %2, %8;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t"
            "add.s64 ra, %1, %9;\n\tadd.s64 rb, %2, %9;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, t;\n\t}"
            ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(1u), "n"(CH), "n"(CH + 2), "n"(CH + 4), "n"(CH + 6)
            : "memory");
    }
}

// Four tcgen05.mma with A from tensor memory (16 K elements = 8 columns per
// step) and B from shared memory (K steps STEP descriptor units apart), in
// one block, issued by one elected lane of a converged warp.  The first
// accumulates iff `acc`.
template <int STEP>
__device__ __forceinline__ void mma_ts_k4_warp(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b64 rb;\n\t.reg .b32 ra;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 t, %5, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "add.u32 ra, %1, 8;\n\tadd.s64 rb, %2, %6;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
        "add.u32 ra, %1, 16;\n\tadd.s64 rb, %2, %7;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t"
        "add.u32 ra, %1, 24;\n\tadd.s64 rb, %2, %8;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rb, %3, t;\n\t}"
        ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc), "r"(1u), "n"(STEP), "n"(2 * STEP), "n"(3 * STEP)
        : "memory");
}

// One full attention batch of a tile in one block, issued by one elected lane
// of a converged warp, with no other instruction of the thread between the
// MMAs: P V over two slabs (A = P from tensor memory, 8 columns per K step,
// the second slab 32 columns on; B = the two value slabs vd0 / vd1, K steps
// STEP units apart; the first MMA accumulates iff `acc`), then Q K^T into
// `s` (A = q, B = k, eight K
// steps: 2 units apart within a 128-byte chunk, CH units between chunks; the
// first overwrites), and an arrival on `bar_s`.  With `rel`, arrivals on
// `bar_v` once the P V MMAs complete and on `bar_k` once the Q K^T MMAs do.
template <int STEP, int CH>
__device__ __forceinline__ void mma_attn_batch_warp(uint32_t o, uint32_t p_tmem, uint64_t vd0, uint64_t vd1,
                                                    uint32_t idesc_pv, uint32_t acc, uint32_t s, uint64_t q,
                                                    uint64_t k, uint32_t idesc_qk, uint64_t* bar_v, uint64_t* bar_s,
                                                    uint64_t* bar_k, uint32_t rel)
{
    asm volatile(
        "{\n\t.reg .pred e, p, t, z, w;\n\t.reg .b64 ra, rb;\n\t.reg .b32 ta;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %5, 0;\n\tsetp.ne.b32 t, %13, 0;\n\tsetp.ne.b32 z, %13, 1;\n\t"
        "setp.ne.and.b32 w, %21, 0, e;\n\t"
        // P V, first value slab
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n\t"
        "add.u32 ta, %1, 8;\n\tadd.s64 rb, %2, %14;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], rb, %4, t;\n\t"
        "add.u32 ta, %1, 16;\n\tadd.s64 rb, %2, %15;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], rb, %4, t;\n\t"
        "add.u32 ta, %1, 24;\n\tadd.s64 rb, %2, %16;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], rb, %4, t;\n\t"
        // P V, second value slab
        "add.u32 ta, %1, 32;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], %3, %4, t;\n\t"
        "add.u32 ta, %1, 40;\n\tadd.s64 rb, %3, %14;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], rb, %4, t;\n\t"
        "add.u32 ta, %1, 48;\n\tadd.s64 rb, %3, %15;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], rb, %4, t;\n\t"
        "add.u32 ta, %1, 56;\n\tadd.s64 rb, %3, %16;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], rb, %4, t;\n\t"
        "@w tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%10];\n\t"
        // Q K^T
        "@e tcgen05.mma.cta_group::1.kind::f16 [%6], %7, %8, %9, z;\n\t"
        "add.s64 ra, %7, 2;\n\tadd.s64 rb, %8, 2;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%6], ra, rb, %9, t;\n\t"
        "add.s64 ra, %7, 4;\n\tadd.s64 rb, %8, 4;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%6], ra, rb, %9, t;\n\t"
        "add.s64 ra, %7, 6;\n\tadd.s64 rb, %8, 6;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%6], ra, rb, %9, t;\n\t"
        "add.s64 ra, %7, %17;\n\tadd.s64 rb, %8, %17;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%6], ra, rb, %9, t;\n\t"
        "add.s64 ra, %7, %18;\n\tadd.s64 rb, %8, %18;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%6], ra, rb, %9, t;\n\t"
        "add.s64 ra, %7, %19;\n\tadd.s64 rb, %8, %19;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%6], ra, rb, %9, t;\n\t"
        "add.s64 ra, %7, %20;\n\tadd.s64 rb, %8, %20;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%6], ra, rb, %9, t;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%11];\n\t"
        "@w tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%12];\n\t}"
        ::"r"(o), "r"(p_tmem), "l"(vd0), "l"(vd1), "r"(idesc_pv), "r"(acc), "r"(s), "l"(q), "l"(k), "r"(idesc_qk),
          "r"(smem_u32(bar_v)), "r"(smem_u32(bar_s)), "r"(smem_u32(bar_k)), "r"(1u), "n"(STEP), "n"(2 * STEP),
          "n"(3 * STEP), "n"(CH), "n"(CH + 2), "n"(CH + 4), "n"(CH + 6), "r"(rel)
        : "memory");
}

__device__ __forceinline__ void mma_commit_warp(uint64_t* bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

// Arrive (once) on `bar` when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// TMEM address: lane in bits 31..16, column in bits 15..0.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col)
{
    return base + (lane << 16) + col;
}

// 32 lanes x 32 consecutive 32-bit columns -> 32 registers per thread
// (thread i of the warp gets lane (lane_base + i)).  Waits for completion.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 32 lanes x 32 columns store from 32 registers per thread; waits for completion.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// The same load without the wait: several loads can be in flight; call
// tmem_wait_ld() and then reg_dep32() on every destination array before the
// registers are used (reg_dep32 ties later uses to the wait).
__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 32 lanes x 16 columns -> 16 registers per thread, without the wait (see
// tmem_ld32_nw).
__device__ __forceinline__ void tmem_ld16_nw(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void reg_dep16(uint32_t (&r)[16])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
}

// 32 lanes x 8 columns store from 8 registers per thread; no wait.
__device__ __forceinline__ void tmem_st8_nw(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void reg_dep32(uint32_t (&r)[32])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// 32 lanes x 16 columns store from 16 registers per thread; no wait (a later
// tmem_wait_st() or the fence before a thread sync orders it).
__device__ __forceinline__ void tmem_st16_nw(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Packed fp32 pairs and three-input max (sm_100+ instructions)
// ---------------------------------------------------------------------------
// (d0, d1) = (a0 * b0 + c0, a1 * b1 + c1), each rounded to nearest.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0, float c1)
{
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// (d0, d1) = (a0 + b0, a1 + b1), each rounded to nearest.
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// (d0, d1) = (a0 * b0, a1 * b1), each rounded to nearest.
__device__ __forceinline__ void mul2(float& d0, float& d1, float a0, float a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ---------------------------------------------------------------------------
// Descriptors
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor (tcgen05): start address, leading- and
// stride-dimension byte offsets (16-byte units), fixed version bits 46..48 =
// 0b001, swizzle mode in bits 61..63 (2 = 128-byte swizzle).
// For a K-major operand with 128-byte swizzle: rows are 128 B apart, 8-row
// groups SBO = 1024 B apart, LBO unused; advancing K by 16 bf16 within the
// 128-byte row adds 32 B to the start address.
// For an MN-major operand with 128-byte swizzle: each K row holds 64
// consecutive MN elements (128 B); 64-element MN chunks are LBO apart; 8-row
// K groups are SBO = 1024 B apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;   // SWIZZLE_128B
    return d;
}

// Instruction descriptor, kind::f16: D f32, A and B bf16, dense.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   15 A MN-major, 16 B MN-major, 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Byte offset of element (row, col) inside a [rows x 64] bf16 tile stored
// with the 128-byte swizzle (the layout TMA SWIZZLE_128B writes for a box
// whose inner extent is 64 bf16).  Tile base must be 1024-byte aligned.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t col)
{
    return row * 128u + ((((col >> 3) ^ (row & 7u)) & 7u) << 4) + ((col & 7u) << 1);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Pack two floats to bf16x2 (round to nearest even): `lo` in bits 15..0.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// phi(x) = elu(x) + 1 = x + 1 for x > 0, e^x otherwise; e^x as 2^(x log2 e)
// on the special-function unit (ex2.approx), which is several times cheaper
// here than the __expf intrinsic.
__device__ __forceinline__ float phi_elu1(float x)
{
    return x > 0.0f ? x + 1.0f : ex2_approx(x * 1.4426950408889634f);
}

}  // namespace hf
