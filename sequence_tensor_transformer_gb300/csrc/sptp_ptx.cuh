// Inline-PTX wrappers for sm_103a: mbarriers, TMA, tcgen05 (TMEM + UMMA), and
// the bounded waits every kernel of the library uses.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "sptp_internal.h"

namespace sptp {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Context of a bounded wait: where to report, the CTA-wide abort flag, and
// the time limit.  Once one wait of a CTA gives up, every other wait of that
// CTA sees the abort flag and returns false too, so all roles leave their
// loops and the CTA reaches its teardown.
struct WaitCtx {
    DeviceStatus* status;
    volatile int* abort_flag;  // shared memory
    unsigned long long limit_ns;
};

__device__ __forceinline__ void report_timeout(const WaitCtx& w, int where, int info) {
    *w.abort_flag = 1;
    if (w.status != nullptr && atomicCAS(&w.status->code, 0, -6 /* SPTP_ERR_TIMEOUT */) == 0) {
        w.status->where = where;
        w.status->block = blockIdx.x;
        w.status->info = info;
    }
}

// Waits for the completion of the mbarrier phase with parity `parity`;
// returns false if the wait gave up (timeout or CTA abort).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w, int where,
                                          int info) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*w.abort_flag) return false;
        if (global_timer_ns() - t0 > w.limit_ns) {
            report_timeout(w, where, info);
            return false;
        }
    }
}

// Waits until a global int reaches `target` (acquire); bounded like mbar_wait.
__device__ __forceinline__ bool flag_wait_geq(const int* flag, int target, const WaitCtx& w, int where,
                                              int info) {
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v >= target) return true;
        if (*w.abort_flag) return false;
        if (global_timer_ns() - t0 > w.limit_ns) {
            report_timeout(w, where, info);
            return false;
        }
        __nanosleep(64);
    }
}

// Warp-wide bounded wait until a global int reaches `target`: every lane
// performs its own acquire load of the same word (one transaction, so every
// lane sees the same value and the loop stays warp-uniform), so each lane's
// later reads are ordered after the releasing writes.  Returns false if the
// wait gave up.
__device__ __forceinline__ bool warp_flag_wait_geq(const int* flag, int target, const WaitCtx& w, int where,
                                                   int info) {
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (__all_sync(0xffffffffu, v >= target)) return true;
        if (__any_sync(0xffffffffu, *w.abort_flag != 0)) return false;
        if (__any_sync(0xffffffffu, global_timer_ns() - t0 > w.limit_ns)) {
            if ((threadIdx.x & 31) == 0) report_timeout(w, where, info);
            return false;
        }
        __nanosleep(64);
    }
}

// ---------------------------------------------------------------- bounds-checked builds
// Built with -DSPTP_BOUNDS_CHECK, the kernels check the indices and
// addresses they compute -- decoded tiles, readiness counters, pending-ring
// slots, the cluster shape, TMA box origins, global loads and stores --
// against the buffers they address before using them.  A failed check
// records SPTP_ERR_BOUNDS (-11), the place (kWhereBounds*) and the offending
// value in the status words, raises the CTA's abort flag and skips the
// access; the kernel then leaves through its bounded waits.  In the normal
// build every check is the constant true and compiles to nothing.
#ifdef SPTP_BOUNDS_CHECK
constexpr bool kBoundsChecked = true;
#else
constexpr bool kBoundsChecked = false;
#endif

__device__ __forceinline__ void report_bounds(DeviceStatus* st, volatile int* abort_flag, int where, long long value) {
    if (abort_flag != nullptr) *abort_flag = 1;
    if (st != nullptr && atomicCAS(&st->code, 0, -11 /* SPTP_ERR_BOUNDS */) == 0) {
        st->where = where;
        st->block = blockIdx.x;
        const long long lim = 0x7fffffffll;
        st->info = static_cast<int>(value > lim ? lim : (value < -lim ? -lim : value));
    }
}

// true if ok; in a checked build a false `ok` is recorded and false returned.
__device__ __forceinline__ bool checked(bool ok, DeviceStatus* st, volatile int* abort_flag, int where,
                                        long long value) {
    if constexpr (kBoundsChecked) {
        if (!ok) {
            report_bounds(st, abort_flag, where, value);
            return false;
        }
    }
    return true;
}

// [off, off + n) within [0, limit) (elements or bytes)
__device__ __forceinline__ bool checked_range(long long off, long long n, long long limit, DeviceStatus* st,
                                              volatile int* abort_flag, int where) {
    return checked(off >= 0 && off + n <= limit, st, abort_flag, where, off);
}

// 0 <= i < n
__device__ __forceinline__ bool checked_index(long long i, long long n, DeviceStatus* st, volatile int* abort_flag,
                                              int where) {
    return checked(i >= 0 && i < n, st, abort_flag, where, i);
}

// A TMA box origin: the inner coordinate x aligned to `align` elements (16
// bytes and more) and inside [0, extent_x); the row coordinate inside
// [0, extent_rows) (a box may hang over the end and is zero-filled there).
__device__ __forceinline__ bool checked_tma(int x, int align, int extent_x, long long row, long long extent_rows,
                                            DeviceStatus* st, volatile int* abort_flag) {
    if constexpr (kBoundsChecked) {
        if (x < 0 || x % align != 0 || x >= extent_x) return checked(false, st, abort_flag, kWhereBoundsTma, x);
        if (row < 0 || row >= extent_rows) return checked(false, st, abort_flag, kWhereBoundsTma, row);
    }
    return true;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of the box at (c0 = inner coordinate, c1 = row) into shared
// memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// Bulk (non-tensor) copy of `bytes` (multiple of 16, 16-byte aligned ends)
// from global to this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Orders this thread's earlier generic-proxy accesses before later
// async-proxy (TMA) accesses of shared memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 3-D and 4-D tiled loads for CTA pairs (coordinates innermost first); the
// shared-memory image of a box with trailing extents of 1 is that of the 2-D
// box.
__device__ __forceinline__ void tma_load_3d_pair(void* smem_dst, const CUtensorMap* map, uint32_t mbar_cluster,
                                                 int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar_cluster), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d_pair(void* smem_dst, const CUtensorMap* map, uint32_t mbar_cluster,
                                                 int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4, %5, %6}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar_cluster), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// ---------------------------------------------------------------- tcgen05
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

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulator.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Loads 32 consecutive fp32 columns of the warp's 32 TMEM lanes (one lane per
// thread).
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Loads 16 consecutive fp32 columns of the warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- clusters / CTA pairs
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Full cluster barrier (release/acquire); safe for divergent warps.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier given by its shared::cluster address (own or peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// The same arrive without release semantics: it orders nothing of this
// thread's earlier memory writes (for signals that only order tcgen05 work,
// made complete beforehand by tcgen05.wait and tcgen05.fence).
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// 2-D tiled TMA load into this CTA's shared memory whose completion bytes are
// counted on an mbarrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, uint32_t mbar_cluster,
                                                 int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar_cluster), "r"(c0), "r"(c1)
        : "memory");
}

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

// CTA-pair UMMA issued by the even CTA: A rows come from both CTAs' shared
// memory (M/2 each), B columns from both (N/2 each), D lands in both TMEMs.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// E4M3 x E4M3 -> fp32 CTA-pair UMMA (K = 32 per instruction, 32 bytes of
// each operand row: the same shared-memory layout as a K = 16 bf16 step).
__device__ __forceinline__ void umma_e4m3_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives once, on the mbarrier at this shared offset in every CTA of
// `cta_mask`, when all prior pair UMMAs of this thread have completed.
__device__ __forceinline__ void umma_commit_pair_multicast(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// ---------------------------------------------------------------- cross-CTA publication
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void red_release_add(int* ctr, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(ctr), "r"(v) : "memory");
}

// OR of `v` over the `nthreads` threads that use named barrier `id`.
template <int ID, int NTHREADS>
__device__ __forceinline__ bool named_barrier_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pin, pout;\n\t"
        "setp.ne.u32 pin, %1, 0;\n\t"
        "bar.red.or.pred pout, %2, %3, pin;\n\t"
        "selp.u32 %0, 1, 0, pout;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "n"(ID), "n"(NTHREADS)
        : "memory");
    return r != 0;
}

template <int ID, int NTHREADS>
__device__ __forceinline__ void named_barrier_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(NTHREADS) : "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// 128-byte swizzle: rows of 128 bytes (64 elements), 8-row swizzle atoms
// 1024 bytes apart.  Fields: start address >> 4 (bits 0-13), leading byte
// offset >> 4 (bits 16-29; unused for swizzled K-major, set to 1), stride
// byte offset >> 4 (bits 32-45) = 1024 >> 4, descriptor version 1 (bits
// 46-47), base offset 0 (tiles are 1024-byte aligned), swizzle mode 2 =
// 128-byte (bits 61-63).
__device__ __forceinline__ uint64_t smem_desc_kmajor_sw128(uint32_t smem_addr) {
    uint64_t desc = 0;
    desc |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
    desc |= static_cast<uint64_t>(1u) << 16;
    desc |= static_cast<uint64_t>(1024u >> 4) << 32;
    desc |= static_cast<uint64_t>(1u) << 46;
    desc |= static_cast<uint64_t>(2u) << 61;
    return desc;
}

// Instruction descriptor of kind::f16 with bf16 A/B, fp32 D, both operands
// K-major: D format F32 (bits 4-5 = 1), A format BF16 (bits 7-9 = 1),
// B format BF16 (bits 10-12 = 1), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// The same for kind::f8f6f4 with E4M3 A and B (format code 0 in bits 7-9 and
// 10-12), K-major, fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n) {
    return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

}  // namespace sptp
