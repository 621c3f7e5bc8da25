// sm100.cuh -- inline-PTX building blocks for sm_103a kernels: mbarriers with
// bounded waits, TMA tile loads, tensor-memory (TMEM) allocation/load/store
// and tcgen05 MMAs with their shared-memory and instruction descriptors.
//
// Written from the public PTX ISA description of these instructions.  Every
// wait in here is bounded: a wait that exceeds its time limit records
// ATTN_DEV_TIMEOUT in the kernel's status word, raises the CTA's abort flag
// and returns false, so that the kernel can drain and leave instead of
// spinning forever.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace attn {

// Device status word bits (read by attn_get_device_status).
constexpr unsigned ATTN_DEV_TIMEOUT = 1u;
// A kernel found an input index outside its declared range (a paged-cache
// block id or sequence length) and used a safe substitute instead.
constexpr unsigned ATTN_DEV_BAD_INPUT = 2u;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// Abort / timeout bookkeeping shared by all waits of one CTA.
// ---------------------------------------------------------------------------
struct WaitGuard {
    unsigned* status;       // global device status word
    volatile int* abort;    // CTA-wide abort flag in shared memory
    uint64_t limit_ns;      // per-wait limit
};

__device__ __forceinline__ void record_timeout(const WaitGuard& g, unsigned site) {
    // First failing site in bits 8..15, timeout flag in bit 0.
    atomicCAS(g.status, 0u, ATTN_DEV_TIMEOUT | ((site & 0xffu) << 8));
    atomicOr(g.status, ATTN_DEV_TIMEOUT);
    *g.abort = 1;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return done != 0;
}

// Wait until the phase with the given parity has completed.  Returns false
// (after recording the timeout) if it does not within the guard's limit or if
// another thread of the CTA has already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          const WaitGuard& g, unsigned site) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*g.abort) return false;
        if (global_timer_ns() - t0 > g.limit_ns) {
            record_timeout(g, site);
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) tile loads, completion counted on an mbarrier.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)),
           "r"(c0), "r"(c1) : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)),
           "r"(c0), "r"(c1), "r"(c2) : "memory");
}

// Tiled store shared -> global through a tensor map (bulk-group completion).
// Rows of the box outside the tensor are not written.  Coordinates must not
// be negative.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* src, int c0, int c1,
                                             int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
        :: "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until the shared-memory sources of this thread's bulk groups have been read.
__device__ __forceinline__ void bulk_wait_group_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_group0() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA, tensor core) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Prefetch a tile into L2 through a tensor map (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* m, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 :: "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2) : "memory");
}

// Contiguous bulk copy global -> shared (no tensor map).  dst, src 16-byte
// aligned, bytes a multiple of 16; completion counted on bar.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes),
           "r"(smem_u32(bar)) : "memory");
}

// ---------------------------------------------------------------------------
// Tensor memory
// ---------------------------------------------------------------------------
// Allocate ncols columns (power of two, >= 32); executed by one full warp.
// The TMEM address is written to *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(dst)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// A TMEM address: bits 31..16 lane, bits 15..0 column.  A warp may only touch
// the 32-lane quarter given by (warp id % 4).
__device__ __forceinline__ uint32_t tmem_lane_base(uint32_t tmem, int warp_id) {
    return tmem + ((static_cast<uint32_t>(warp_id & 3) * 32u) << 16);
}

// Load 32 consecutive 32-bit columns of this thread's lane (shape 32x32b).
// The registers are not valid until tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
          "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// Wait for all of this thread's outstanding tcgen05.ld; the "+r" operands tie
// the registers of one load to the wait so no use can be scheduled earlier.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
          "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
          "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
          "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
          "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
          "+r"(r[30]), "+r"(r[31])
        :: "memory");
}

// Empty statement that orders the use of r after a preceding wait.
__device__ __forceinline__ void reg_order(uint32_t (&r)[32]) {
    asm volatile(""
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
          "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
          "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
          "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
          "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
          "+r"(r[30]), "+r"(r[31])
        :: "memory");
}

// Empty statement that orders the use of a 64-register array after a
// preceding wait (the second array of a pair loaded before one wait).
__device__ __forceinline__ void reg_order64(uint32_t (&r)[64]) {
    asm volatile(""
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
          "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
          "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
          "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]),
          "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]),
          "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]),
          "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]),
          "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63])
        :: "memory");
}

// Store 32 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        :: "r"(taddr),
           "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
           "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]),
           "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
           "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
           "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),
           "r"(r[30]), "r"(r[31])
        : "memory");
}

// Load 64 consecutive 32-bit columns of this thread's lane (shape 32x32b);
// valid after tmem_wait_ld64().
__device__ __forceinline__ void tmem_ld32x64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr));
}

// Store 64 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_st32x64(uint32_t taddr, const uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};"
        :: "r"(taddr),
           "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
           "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
           "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
           "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]),
           "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]),
           "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]),
           "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]),
           "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
        : "memory");
}

// Store 16 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
           "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
           "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// 16-lane shapes.  A warp addresses 16 lanes L0 .. L0+15 of its quarter; its
// thread i holds lanes La = L0 + i/4 and Lb = La + 8.  With .16x256b, chunk n
// (8 columns) occupies registers 4n .. 4n+3 = (La, 8n + 2(i%4)), (La, +1),
// (Lb, 8n + 2(i%4)), (Lb, +1).  With .16x128b, chunk n (4 columns) occupies
// registers 2n, 2n+1 = (La, 4n + i%4), (Lb, 4n + i%4).
// 128 columns of 16 lanes; valid after tmem_wait_ld64().
__device__ __forceinline__ void tmem_ld_16x256b_x16(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]),
          "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]),
          "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
          "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]),
          "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]),
          "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr));
}
// 64 columns of 16 lanes; valid after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
// 16 columns of 16 lanes (two 8-column chunks: registers 0-3 chunk 0, 4-7
// chunk 1; within a chunk, registers 0, 1 row L0 + i/4 and 2, 3 row L0 + i/4
// + 8); valid after tmem_wait_ld8().
__device__ __forceinline__ void tmem_ld_16x256b_x2(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld8(uint32_t (&r)[8]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7])
                 :: "memory");
}
__device__ __forceinline__ void tmem_st_16x256b_x2(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x256b.x2.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
           "r"(r[6]), "r"(r[7])
        : "memory");
}

// Store 64 columns of 16 lanes (layout of tmem_ld_16x256b_x8).
__device__ __forceinline__ void tmem_st_16x256b_x8(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        :: "r"(taddr),
           "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
           "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
           "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
           "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
           "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
// Store 64 columns of 16 lanes, two registers per 4-column chunk.
__device__ __forceinline__ void tmem_st_16x128b_x16(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x128b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        :: "r"(taddr),
           "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
           "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
           "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
           "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
           "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
// tmem_wait_ld for a 64-register load.
__device__ __forceinline__ void tmem_wait_ld64(uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
          "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
          "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
          "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
          "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
          "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]),
          "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]),
          "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]),
          "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]),
          "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]),
          "+r"(r[61]), "+r"(r[62]), "+r"(r[63])
        :: "memory");
}

// Add the two bf16 halves of a packed pair to two fp32 accumulators
// (mixed-precision add; no separate unpacking).
__device__ __forceinline__ void add_bf16x2_to_f32(uint32_t pk, float& lo_acc, float& hi_acc) {
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, lo, %0;\n\t"
        "add.rn.f32.bf16 %1, hi, %1;\n\t}"
        : "+f"(lo_acc), "+f"(hi_acc) : "r"(pk));
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05.mma descriptors
// ---------------------------------------------------------------------------
// Instruction descriptor, kind::f16 with bf16 (or, with f16, fp16) A/B and an
// fp32 accumulator:
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16, 0 = f16), 10-12 B
//   format (same), 15 A major (0 = K-major, 1 = MN-major), 16 B major,
//   17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t mma_idesc_bf16_f32(int M, int N, bool a_mn_major,
                                                          bool b_mn_major, bool f16 = false) {
    return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) |
           (static_cast<uint32_t>(a_mn_major) << 15) |
           (static_cast<uint32_t>(b_mn_major) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor with 128-byte swizzling:
//   bits 0-13 start address >> 4, 16-29 leading-dimension byte offset >> 4,
//   32-45 stride-dimension byte offset >> 4, 46-47 version (1),
//   49-51 base offset (0: atoms are 1024-byte aligned), 61-63 layout
//   (2 = 128-byte swizzle).
// K-major operand: rows of 128 bytes, 8-row atoms 1024 bytes apart (SBO); the
//   leading offset is unused while an MMA's K extent stays inside one row.
// MN-major operand: 64 contiguous MN elements per 128-byte row, one row per K
//   index; LBO = distance between 64-element MN blocks, SBO = distance
//   between groups of 8 K rows.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// MMA issue.  The wrappers below are executed by all 32 lanes of a converged
// warp; `leader` (from elect_leader(), taken once) is nonzero in exactly one
// lane, which issues.  Keeping the warp converged keeps the operands
// warp-uniform, and predicating on a stored flag instead of electing per
// instruction matters: elect.sync waits for the warp's queued MMAs to be
// taken by the tensor pipe (measured: about 200 cycles behind a queued group
// of eight), while setp does not.

// Nonzero in exactly one lane of the (converged) calling warp.
__device__ __forceinline__ uint32_t elect_leader() {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, e;\n\t}"
        : "=r"(r) :: "memory");
    return r;
}

// A group of MMAs into one accumulator in one statement; the first MMA
// accumulates only if `accumulate`, the others always.
// SS form: A and B from shared memory (descriptors a[k], b[k]).
__device__ __forceinline__ void mma_bf16_ss_x4(uint32_t d_tmem, const uint64_t (&a)[4],
                                               const uint64_t (&b)[4], uint32_t idesc,
                                               uint32_t accumulate, uint32_t leader) {
    asm volatile(
        "{\n\t.reg .pred e, pa, pt;\n\t"
        "setp.ne.b32 e, %11, 0;\n\t"
        "setp.ne.b32 pa, %10, 0;\n\t"
        "setp.eq.b32 pt, %9, %9;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %9, pa;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %9, pt;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %9, pt;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %9, pt;\n\t}"
        :: "r"(d_tmem), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]),
           "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]),
           "r"(idesc), "r"(accumulate), "r"(leader) : "memory");
}

__device__ __forceinline__ void mma_bf16_ss_x8(uint32_t d_tmem, const uint64_t (&a)[8],
                                               const uint64_t (&b)[8], uint32_t idesc,
                                               uint32_t accumulate, uint32_t leader) {
    asm volatile(
        "{\n\t.reg .pred e, pa, pt;\n\t"
        "setp.ne.b32 e, %19, 0;\n\t"
        "setp.ne.b32 pa, %18, 0;\n\t"
        "setp.eq.b32 pt, %17, %17;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %9, %17, pa;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %10, %17, pt;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %17, pt;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %17, pt;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %17, pt;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %14, %17, pt;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %15, %17, pt;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %16, %17, pt;\n\t}"
        :: "r"(d_tmem), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]),
           "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]),
           "r"(idesc), "r"(accumulate), "r"(leader) : "memory");
}

// TS form: A from tensor memory (addresses a[k]), B from shared memory.
__device__ __forceinline__ void mma_bf16_ts_x8(uint32_t d_tmem, const uint32_t (&a)[8],
                                               const uint64_t (&b)[8], uint32_t idesc,
                                               uint32_t accumulate, uint32_t leader) {
    asm volatile(
        "{\n\t.reg .pred e, pa, pt;\n\t"
        "setp.ne.b32 e, %19, 0;\n\t"
        "setp.ne.b32 pa, %18, 0;\n\t"
        "setp.eq.b32 pt, %17, %17;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %9, %17, pa;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %10, %17, pt;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %11, %17, pt;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %12, %17, pt;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %13, %17, pt;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], %14, %17, pt;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %15, %17, pt;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], %16, %17, pt;\n\t}"
        :: "r"(d_tmem), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]),
           "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]),
           "r"(idesc), "r"(accumulate), "r"(leader) : "memory");
}

// Arrive once on bar when all previously issued tcgen05 async operations of
// the leader lane have completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar, uint32_t leader) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "setp.ne.b32 e, %1, 0;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        :: "r"(smem_u32(bar)), "r"(leader) : "memory");
}

// ---------------------------------------------------------------------------
// Small numeric helpers
// ---------------------------------------------------------------------------
// Packed fp32 pairs (one 64-bit register pair) and the sm_100 f32x2 ops that
// do two fp32 operations per instruction.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Per-warp register budget change (values are multiples of 8); every thread
// of the warp executes it.
template <int N>
__device__ __forceinline__ void regs_increase() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(N));
}
template <int N>
__device__ __forceinline__ void regs_decrease() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(N));
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two floats -> packed bf16x2 (round to nearest even); lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 2^x on the FMA and integer pipes, for x <= 64 (arguments below -126 give
// 2^-126 instead of 0).  Cody-Waite split x = j + f with j = rint(x) (the
// 1.5 * 2^23 rounding trick, exact in fp32 for |x| < 2^22) and
// f in [-1/2, 1/2]; 2^f by a degree-4 polynomial whose maximum relative error
// on [-1/2, 1/2] is minimised (Remez exchange; csrc/fit_exp2_poly.py prints
// the coefficients and the bound, 2.7e-6); 2^j is added to the exponent field.
// Two arguments at a time through the packed f32x2 instructions.
__device__ __forceinline__ void exp2_poly_x2(uint64_t x2, float& y0, float& y1) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    float x0, x1;
    f2_unpack(x2, x0, x1);
    const uint64_t xc = f2_pack(fmaxf(x0, -126.0f), fmaxf(x1, -126.0f));
    const uint64_t t = f2_add(xc, f2_pack(kMagic, kMagic));
    const uint64_t j = f2_add(t, f2_pack(-kMagic, -kMagic));
    const uint64_t f = f2_fma(j, f2_pack(-1.0f, -1.0f), xc);
    uint64_t p = f2_fma(f2_pack(0.009570102207362652f, 0.009570102207362652f), f,
                        f2_pack(0.05591785907745361f, 0.05591785907745361f));
    p = f2_fma(p, f, f2_pack(0.240247443318367f, 0.240247443318367f));
    p = f2_fma(p, f, f2_pack(0.6931217908859253f, 0.6931217908859253f));
    p = f2_fma(p, f, f2_pack(0.9999992847442627f, 0.9999992847442627f));
    float p0, p1, t0, t1;
    f2_unpack(p, p0, p1);
    f2_unpack(t, t0, t1);
    y0 = __int_as_float(__float_as_int(p0) + (__float_as_int(t0) << 23));
    y1 = __int_as_float(__float_as_int(p1) + (__float_as_int(t1) << 23));
}

__device__ __forceinline__ float bf16_lo_to_f32(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi_to_f32(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// fp16 counterparts: two floats -> packed f16x2 (round to nearest even, lo in
// the low half), the halves of a pair -> fp32 (exact), and the mixed-precision
// add of both halves to two fp32 accumulators.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float f16_lo_to_f32(uint32_t x) {
    float f;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}"
        : "=f"(f) : "r"(x));
    return f;
}
__device__ __forceinline__ float f16_hi_to_f32(uint32_t x) {
    float f;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, hi;\n\t}"
        : "=f"(f) : "r"(x));
    return f;
}
__device__ __forceinline__ void add_f16x2_to_f32(uint32_t pk, float& lo_acc, float& hi_acc) {
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.f16 %0, lo, %0;\n\t"
        "add.rn.f32.f16 %1, hi, %1;\n\t}"
        : "+f"(lo_acc), "+f"(hi_acc) : "r"(pk));
}

// The 16-bit I/O element: bf16 (kF16 = false) or fp16.  kMaxPartial bounds a
// thread's partial weight sum on the prefill's fast path so that every weight
// stays finite in the element type: 2^62 for bf16 (fp32's exponent range),
// 2^15 for fp16 (largest finite value 65504).
template <bool kF16>
struct Elem16 {
    static constexpr float kMaxPartial = kF16 ? 0x1p15f : 0x1p62f;
    __device__ static __forceinline__ uint32_t pack(float lo, float hi) {
        if constexpr (kF16) return pack_f16x2(lo, hi);
        else return pack_bf16x2(lo, hi);
    }
    __device__ static __forceinline__ void add2(uint32_t pk, float& lo_acc, float& hi_acc) {
        if constexpr (kF16) add_f16x2_to_f32(pk, lo_acc, hi_acc);
        else add_bf16x2_to_f32(pk, lo_acc, hi_acc);
    }
    __device__ static __forceinline__ float lo(uint32_t x) {
        if constexpr (kF16) return f16_lo_to_f32(x);
        else return bf16_lo_to_f32(x);
    }
    __device__ static __forceinline__ float hi(uint32_t x) {
        if constexpr (kF16) return f16_hi_to_f32(x);
        else return bf16_hi_to_f32(x);
    }
};

}  // namespace attn
