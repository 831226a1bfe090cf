// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA tensor loads,
// and the tcgen05 (5th-generation tensor core) instructions with TMEM
// accumulators.  Each wrapper is one instruction; the encodings of the shared
// memory matrix descriptor and of the instruction descriptor follow the PTX ISA
// description of tcgen05.mma.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace bigemm {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch: wait until the grids this one depends on
// have completed (their writes visible); let dependent grids start launching.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Kernel entry of the library's launches: wait for the previous grid, then let
// the next one launch at once, so its launch and set-up overlap this grid.
// Safe because every kernel of the library waits before it reads anything the
// grid before it writes (griddepcontrol.wait waits for that grid to finish).
__device__ __forceinline__ void griddep_enter()
{
    griddep_wait();
    griddep_launch_dependents();
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Test the phase; if it is not complete the thread may be suspended until it
// completes or about `hint_ns` pass, whichever comes first.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity,
                                              uint32_t hint_ns = 1000000u)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Wait until the phase of `bar` with the given parity has completed.  Bounded:
// gives up after timeout_ns of wall time (or 2^30 polls), or as soon as another
// warp of the block has raised *abort.  On a timeout it raises *abort and the
// global error word.  Returns true when the phase completed.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t timeout_ns,
                                          volatile int *abort, int *err)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 30); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > timeout_ns) break;
        }
    }
    *abort = 1;
    atomicExch(err, 4 /* BIGEMM_ERR_TIMEOUT */);
    return false;
}

// Warp-converged form: lane 0 waits, every lane of the warp gets the outcome.
// Keeps role warps converged (their other lanes never idle at a CTA barrier
// while one lane works).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity,
                                               uint64_t timeout_ns, volatile int *abort, int *err)
{
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, timeout_ns, abort, err) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// ----------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Bulk tensor stores from shared memory (tile -> global), tracked per thread
// in bulk async-groups.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int c0,
                                             int c1, int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            map),
        "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, const void *src, int c0,
                                             int c1, int c2, int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
            map),
        "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// Element-wise atomic add of a shared-memory box into global memory (fp32
// maps), tracked like a store.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap *map, const void *src, int c0,
                                                  int c1, int c2)
{
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%2, %3, %4}], [%1];" ::"l"(map),
        "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_reduce_add_4d(const CUtensorMap *map, const void *src, int c0,
                                                  int c1, int c2, int c3)
{
    asm volatile(
        "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%2, %3, %4, %5}], [%1];" ::"l"(map),
        "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// 4-byte asynchronous global -> shared copy through L1; a thread's copies
// complete in commit-group order (cp_async_wait<N>: all but the newest N groups)
__device__ __forceinline__ void cp_async4(void *dst_smem, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst_smem)), "l"(src)
                 : "memory");
}
// 16-byte asynchronous global -> shared copy that bypasses L1 (both addresses
// 16-byte aligned)
__device__ __forceinline__ void cp_async16(void *dst_smem, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst_smem)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N committed bulk groups are still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait()
{
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Barrier among `count` threads (a multiple of 32) using hardware barrier `id`.
__device__ __forceinline__ void named_barrier(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2, int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// im2col load of a 4-D channels-last tensor: the pixels from base position
// (c1, c2, c3) = (w, h, n), channels from c0, each read at its position
// shifted by (ow, oh) (a filter tap)
__device__ __forceinline__ void tma_load_im2col_4d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                                   int c0, int c1, int c2, int c3, uint16_t ow,
                                                   uint16_t oh)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.im2col.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2], {%7, %8};" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "h"(ow), "h"(oh)
        : "memory");
}

// ------------------------------------------------------------------- tcgen05
// TMEM allocation: executed by one whole warp; the allocated base address is
// written to shared memory.  ncols is a power of two in [32, 512].
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D(tmem) (+)= A(smem desc) * B(smem desc); accumulate when `accum` != 0.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accum)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
        : "memory");
}

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accum)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives the
// 32 columns of TMEM lane (lane base + i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 form): start address, leading and
// stride byte offsets (all >> 4), the fixed version bit at 46, base offset 0,
// and the swizzle mode in bits 61..63 (0 none, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swz, uint32_t base_offset = 0)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    // matrix base offset (bits 49..51); the kernels keep it 0: starts that are
    // not on a 1024-byte boundary still read the swizzle phase from their
    // address bits
    d |= (uint64_t)(base_offset & 7u) << 49;
    d |= (uint64_t)(swz & 7u) << 61;
    return d;
}

// The two 32-bit halves of a shared-memory descriptor, so that issue loops
// can step the start address with one 32-bit add (start >> 4 sits in the low
// 14 bits; shared memory offsets stay below 2^18, so the field never carries).
__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo)
{
    return ((saddr >> 4) & 0x3FFFu) | (((lbo >> 4) & 0x3FFFu) << 16);
}

__device__ __forceinline__ uint32_t desc_hi(uint32_t sbo, uint32_t swz)
{
    return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | ((swz & 7u) << 29);
}

// tcgen05.mma with the descriptors given as (lo, hi) halves.
template <bool TF32>
__device__ __forceinline__ void umma_lohi(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi,
                                          uint32_t b_lo, uint32_t b_hi, uint32_t idesc,
                                          uint32_t accum)
{
    if (TF32)
        asm volatile(
            "{\n\t.reg .pred p;\n\t.reg .b64 ad, bd;\n\t"
            "mov.b64 ad, {%1, %2};\n\t"
            "mov.b64 bd, {%3, %4};\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], ad, bd, %5, p;\n\t}" ::"r"(d_tmem),
            "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accum)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t.reg .b64 ad, bd;\n\t"
            "mov.b64 ad, {%1, %2};\n\t"
            "mov.b64 bd, {%3, %4};\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p;\n\t}" ::"r"(d_tmem),
            "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accum)
            : "memory");
}

// The four MMAs of one 128-byte K block of K-major, 128-byte swizzled operands
// (the start address advances 32 bytes, 2 in descriptor units, per MMA) in one
// asm block: the first accumulates when `accum_first` != 0, the rest always.
// One issuing thread pays for every instruction between MMAs, so the block
// keeps that to two adds and two register pairings per MMA.
template <bool TF32>
__device__ __forceinline__ void umma4_kmajor(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi,
                                             uint32_t b_lo, uint32_t b_hi, uint32_t idesc,
                                             uint32_t accum_first)
{
    if (TF32)
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t.reg .b64 ad, bd;\n\t.reg .b32 al, bl;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "setp.eq.b32 q, %6, %6;\n\t"
            "mov.b64 ad, {%1, %2};\n\tmov.b64 bd, {%3, %4};\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], ad, bd, %5, p;\n\t"
            "add.u32 al, %1, 2;\n\tadd.u32 bl, %3, 2;\n\t"
            "mov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], ad, bd, %5, q;\n\t"
            "add.u32 al, %1, 4;\n\tadd.u32 bl, %3, 4;\n\t"
            "mov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], ad, bd, %5, q;\n\t"
            "add.u32 al, %1, 6;\n\tadd.u32 bl, %3, 6;\n\t"
            "mov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], ad, bd, %5, q;\n\t}" ::"r"(d_tmem),
            "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accum_first)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t.reg .b64 ad, bd;\n\t.reg .b32 al, bl;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "setp.eq.b32 q, %6, %6;\n\t"
            "mov.b64 ad, {%1, %2};\n\tmov.b64 bd, {%3, %4};\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p;\n\t"
            "add.u32 al, %1, 2;\n\tadd.u32 bl, %3, 2;\n\t"
            "mov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, q;\n\t"
            "add.u32 al, %1, 4;\n\tadd.u32 bl, %3, 4;\n\t"
            "mov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, q;\n\t"
            "add.u32 al, %1, 6;\n\tadd.u32 bl, %3, 6;\n\t"
            "mov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, q;\n\t}" ::"r"(d_tmem),
            "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accum_first)
            : "memory");
}

// ------------------------------------------------------ CTA pairs (cluster of 2)
// The CTA's rank in its cluster.
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of the same shared-memory offset in CTA `rank`
// of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Arrive on an mbarrier given by its shared::cluster address (possibly in the
// peer CTA), with release semantics at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// Every thread of every CTA of the cluster: arrive, then wait for all.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// TMEM allocation for a CTA pair: one warp of each of the two CTAs executes it;
// the same columns are allocated in both CTAs' tensor memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// TMA tensor loads into this CTA's shared memory whose completion is counted
// on an mbarrier of either CTA of the pair (cluster_bar: a shared::cluster
// address).
__device__ __forceinline__ void tma_load_3d_pair(void *dst, const CUtensorMap *map,
                                                 uint32_t cluster_bar, int c0, int c1, int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(cluster_bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d_pair(void *dst, const CUtensorMap *map,
                                                 uint32_t cluster_bar, int c0, int c1, int c2,
                                                 int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(cluster_bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// Arrive once on the mbarrier at the same offset in each CTA of `cta_mask`
// when every tcgen05 operation of the pair issued so far by this thread has
// completed.
__device__ __forceinline__ void umma_commit_pair_mc(uint64_t *bar, uint16_t cta_mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Arrive once on this CTA's mbarrier `bar` when every tcgen05 operation of
// the pair issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// The four MMAs of one 128-byte K block for a CTA pair (M = 256: each CTA's
// 128 rows of A and half of B's N rows at the same shared-memory offsets).
template <bool TF32>
__device__ __forceinline__ void umma4_kmajor_pair(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi,
                                                  uint32_t b_lo, uint32_t b_hi, uint32_t idesc,
                                                  uint32_t accum_first)
{
    if (TF32)
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t.reg .b64 ad, bd;\n\t.reg .b32 al, bl;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "setp.eq.b32 q, %6, %6;\n\t"
            "mov.b64 ad, {%1, %2};\n\tmov.b64 bd, {%3, %4};\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%0], ad, bd, %5, p;\n\t"
            "add.u32 al, %1, 2;\n\tadd.u32 bl, %3, 2;\n\t"
            "mov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%0], ad, bd, %5, q;\n\t"
            "add.u32 al, %1, 4;\n\tadd.u32 bl, %3, 4;\n\t"
            "mov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%0], ad, bd, %5, q;\n\t"
            "add.u32 al, %1, 6;\n\tadd.u32 bl, %3, 6;\n\t"
            "mov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%0], ad, bd, %5, q;\n\t}" ::"r"(d_tmem),
            "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accum_first)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t.reg .b64 ad, bd;\n\t.reg .b32 al, bl;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "setp.eq.b32 q, %6, %6;\n\t"
            "mov.b64 ad, {%1, %2};\n\tmov.b64 bd, {%3, %4};\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], ad, bd, %5, p;\n\t"
            "add.u32 al, %1, 2;\n\tadd.u32 bl, %3, 2;\n\t"
            "mov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], ad, bd, %5, q;\n\t"
            "add.u32 al, %1, 4;\n\tadd.u32 bl, %3, 4;\n\t"
            "mov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], ad, bd, %5, q;\n\t"
            "add.u32 al, %1, 6;\n\tadd.u32 bl, %3, 6;\n\t"
            "mov.b64 ad, {al, %2};\n\tmov.b64 bd, {bl, %4};\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], ad, bd, %5, q;\n\t}" ::"r"(d_tmem),
            "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accum_first)
            : "memory");
}

// Instruction descriptor for kind::f16 / kind::tf32 with an fp32 accumulator:
// operand format (0 f16, 1 bf16, 2 tf32) for A and B, major-ness of A and B
// (0 K-major, 1 MN-major), N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t fmt, uint32_t a_mn, uint32_t b_mn,
                                                  uint32_t M, uint32_t N)
{
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (a_mn << 15) | (b_mn << 16) |
           ((N >> 3) << 17) | ((M >> 4) << 24);
}

}  // namespace bigemm
