// Inline-PTX building blocks for sm_103a: mbarriers, TMA tensor loads, tcgen05
// (tensor memory allocation, MMA, loads/stores, commits, fences), shared-memory
// matrix descriptors, and bounded waits that report instead of hanging.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"

namespace fa {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// The same test, but a thread whose phase is not complete yet is suspended (it
// issues nothing) until the phase completes or about `hint_ns` nanoseconds pass.
// Waiting warps share issue slots with the warp that feeds the tensor core, so
// they must sleep rather than spin.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

// Everything a bounded wait needs: where to record a failure, the CTA's shared
// abort flag (set by the first wait that gives up, so the other roles stop
// waiting early), and the time limit.
struct Guard {
    int *status;             // device status word: [0] error code, [1] site of first error
    volatile int *abort;     // shared memory, 0 while healthy
    unsigned long long limit_ns;
};

__device__ __forceinline__ bool mbar_wait_slow_body(uint32_t bar, uint32_t parity, const Guard &g,
                                                    int site) {
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
        if (*g.abort) return false;
        if (global_timer_ns() - t0 > g.limit_ns) {
            *g.abort = 1;
            atomicCAS(g.status + 1, 0, site);
            atomicExch(g.status, FA_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __noinline__ inline bool mbar_wait_slow(uint32_t bar, uint32_t parity, const Guard &g,
                                                   int site) {
    return mbar_wait_slow_body(bar, parity, g, site);
}

// Wait until the phase with the given parity of barrier `bar` has completed.
// Returns false (after recording FA_ERR_TIMEOUT, or because another role of this
// CTA already gave up) instead of spinning forever.  The slow path is a called
// function, except with kInline: a kernel whose warpgroups rebalance registers
// (setmaxnreg) cannot share one compiled function across their different
// register budgets, so it inlines the slow path at every wait.
template <bool kInline = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const Guard &g, int site) {
    if (mbar_try_wait(bar, parity)) return true;
    if constexpr (kInline)
        return mbar_wait_slow_body(bar, parity, g, site);
    else
        return mbar_wait_slow(bar, parity, g, site);
}

// The same for all 32 lanes of a warp; the result is warp-uniform, so code after
// it may issue warp-collective (.sync.aligned) instructions.
template <bool kInline = false>
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, const Guard &g,
                                               int site) {
    bool ok = mbar_wait<kInline>(bar, parity, g, site);
    return __all_sync(0xffffffffu, ok);
}

// ----------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// 3-D tiled load (x innermost) into shared memory, completing bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, uint32_t bar, int x,
                                            int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// Plain (untiled) bulk copy global -> shared; size and both addresses 16-byte aligned.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Bulk element-wise fp32 add of shared memory into global memory (async proxy).
__device__ __forceinline__ void bulk_reduce_add_f32(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile(
        "cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(dst),
        "r"(src), "r"(bytes)
        : "memory");
}

// Plain bulk copy shared -> global (async proxy); size and addresses 16-byte aligned.
// Programmatic dependent launch: the next kernel on the stream may start launching
// once every CTA of this grid has signalled (or exited); a kernel launched that way
// waits for the previous grid to complete, and its writes to be visible, here.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Tiled bulk add of a shared-memory box into global memory through a tensor map
// (fp32 elements; rows outside the tensor are skipped).  Completes in a bulk group.
__device__ __forceinline__ void tma_reduce_add_3d(const void *tmap, uint32_t src, int x, int y,
                                                  int z) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%2, %3, %4}], [%1];" ::"l"(tmap),
        "r"(src), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed bulk groups still READ their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Make generic-proxy writes to shared memory visible to the async proxy (TMA, MMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A * B[smem]^T, kind::f16 (bf16 in, fp32 accumulate); A from shared
// memory (SS) or, K-major, from tensor memory (TS).  Every lane of the warp makes
// the call with the same operands and one elected lane issues the instruction:
// warp-uniform issuing code lets the compiler do the descriptor arithmetic on the
// uniform datapath instead of per-lane registers, which matters because the
// issuing warp shares its scheduler with busy softmax/compute warps.
__device__ __forceinline__ void mma_ss_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same two forms for kind::f8f6f4 (8-bit A and B of the type the instruction
// descriptor names, fp32 accumulate); K = 32 elements (32 bytes) per instruction.
__device__ __forceinline__ void mma_ss_elect_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_ts_elect_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation the issuing thread started so
// far is done (one elected lane of the calling warp commits).
__device__ __forceinline__ void tc_commit_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            bar)
        : "memory");
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D, dense.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format (1 = bf16),
//   bit 15 A major (0 = K-major, 1 = MN-major), bit 16 B major, 17-22 N>>3, 24-28 M>>4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major,
                                                      bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4 with e4m3 A and B (format code 0) and fp32
// D, dense, both operands K-major.  Same bit positions as idesc_bf16_f32.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand.
//   bits 0-13 start address >> 4, 16-29 leading-dimension byte offset >> 4,
//   32-45 stride-dimension byte offset >> 4, 46-48 = 0b001 (tcgen05 descriptor),
//   49-51 base offset (0: atoms are 1024-byte aligned), 61-63 swizzle (2 = 128B).
// K-major operand: rows of 128 B (64 bf16 of K), SBO = 1024 (8-row group stride).
// MN-major operand: 128 B runs along M/N, LBO = stride between 64-element MN
// chunks, SBO = stride between groups of 8 K rows.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// A descriptor for an address `byte_off` bytes past the one `d` describes (the
// start-address field is the low word's address >> 4 and never overflows here).
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t byte_off) {
    return d + (uint64_t)(byte_off >> 4);
}

// 32 lanes x 32 consecutive 32-bit columns: lane t of the warp gets row
// (lane base + t), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
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

// Wait for this thread's outstanding tcgen05.ld; the registers of `r` are tied to
// the wait so the compiler cannot use them before it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]),
                   "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]),
                   "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Barrier `id` (1-15; 0 is __syncthreads) over the first `count` threads that
// reach it, a multiple of 32.
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Warpgroup register reallocation: every warp of a warpgroup makes the same call.
// dec returns registers to the CTA's pool; inc waits until the pool can supply
// them, so the targets of all warpgroups must add up to no more than the
// registers the CTA was launched with.
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------ numerics

// Hardware base-2 exponential and logarithm (MUFU), flush-to-zero.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs (sm_100+): one instruction for two independent IEEE fp32
// operations, each rounded to nearest like its scalar form.  Pairs are passed as
// two floats; the moves in and out of the 64-bit register are free when the two
// sit in an aligned register pair.
__device__ __forceinline__ uint64_t f32x2_splat(float a) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(a));
    return r;
}

// (x0, x1) <- (x0, x1) * b + c  with b, c splatted pairs.
__device__ __forceinline__ void fma_f32x2(float &x0, float &x1, uint64_t b, uint64_t c) {
    asm("{\n\t.reg .b64 x;\n\tmov.b64 x, {%0, %1};\n\tfma.rn.f32x2 x, x, %2, %3;\n\t"
        "mov.b64 {%0, %1}, x;\n\t}"
        : "+f"(x0), "+f"(x1)
        : "l"(b), "l"(c));
}

// (x0, x1) <- (x0, x1) * b + (c0, c1)  with b a splatted pair.
__device__ __forceinline__ void fma_f32x2(float &x0, float &x1, uint64_t b, float c0, float c1) {
    asm("{\n\t.reg .b64 x, c;\n\tmov.b64 x, {%0, %1};\n\tmov.b64 c, {%3, %4};\n\t"
        "fma.rn.f32x2 x, x, %2, c;\n\tmov.b64 {%0, %1}, x;\n\t}"
        : "+f"(x0), "+f"(x1)
        : "l"(b), "f"(c0), "f"(c1));
}

// (a0, a1) <- (a0, a1) * (x0, x1).
__device__ __forceinline__ void mul_f32x2(float &a0, float &a1, float x0, float x1) {
    asm("{\n\t.reg .b64 a, x;\n\tmov.b64 a, {%0, %1};\n\tmov.b64 x, {%2, %3};\n\t"
        "mul.rn.f32x2 a, a, x;\n\tmov.b64 {%0, %1}, a;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(x0), "f"(x1));
}

// (a0, a1) <- (a0, a1) + (x0, x1).
__device__ __forceinline__ void add_f32x2(float &a0, float &a1, float x0, float x1) {
    asm("{\n\t.reg .b64 a, x;\n\tmov.b64 a, {%0, %1};\n\tmov.b64 x, {%2, %3};\n\t"
        "add.rn.f32x2 a, a, x;\n\tmov.b64 {%0, %1}, a;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(x0), "f"(x1));
}

// (x0, x1) <- (x0, x1) * b  with b a splatted pair.
__device__ __forceinline__ void mul_f32x2(float &x0, float &x1, uint64_t b) {
    asm("{\n\t.reg .b64 x;\n\tmov.b64 x, {%0, %1};\n\tmul.rn.f32x2 x, x, %2;\n\t"
        "mov.b64 {%0, %1}, x;\n\t}"
        : "+f"(x0), "+f"(x1)
        : "l"(b));
}

// max(a, b, c) in one instruction (sm_100+).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Four fp32 -> four e4m3 bytes (round to nearest even, finite values beyond 448
// saturate); a lands in bits 0-7, b in 8-15, c in 16-23, e in 24-31.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float e) {
    uint16_t lo, hi;
    // cvt.*.e4m3x2 puts its first source operand in the upper byte
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(e), "f"(c));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` lands in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

}  // namespace fa
