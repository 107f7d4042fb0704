// Inline-PTX building blocks for sm_103a: mbarrier, TMA tile loads, tcgen05 MMA
// with TMEM accumulators, TMEM loads/stores, and the shared-memory and instruction
// descriptors tcgen05.mma consumes.  Everything here is written against the PTX ISA
// (tcgen05 family, cp.async.bulk.tensor, mbarrier); no library headers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace jfa {

// Spin-wait limit for every pipeline mbarrier wait in the kernels (nanoseconds of
// %globaltimer).  A correct pipeline never waits longer than one tile's work; the
// limit only turns a logic error into an error status instead of a hang.
#ifndef JFA_WAIT_TIMEOUT_NS
#define JFA_WAIT_TIMEOUT_NS 2000000000ull
#endif
// Limit of the waits with which a role, before its CTA exits, lets its own TMA loads and
// tensor-core products finish (drains).  Those always complete; the limit is kept apart
// from the pipeline's, and never shortened, so that a role that gave up on the pipeline
// still waits for everything it issued before shared memory and TMEM are released.
#ifndef JFA_DRAIN_TIMEOUT_NS
#define JFA_DRAIN_TIMEOUT_NS 2000000000ull
#endif

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
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

// try_wait with a suspend-time hint: a thread whose phase is not complete is parked
// by the hardware until the phase completes or about `hint_ns` pass, instead of
// spinning and taking issue slots from the warps that share its scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false if
// the wait gave up: after JFA_WAIT_TIMEOUT_NS, or as soon as another role of the
// CTA raised *abort_flag.  A drain passes nullptr: it ignores the flag and waits up to
// JFA_DRAIN_TIMEOUT_NS.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                            const volatile int* abort_flag) {
    const uint64_t limit = abort_flag ? JFA_WAIT_TIMEOUT_NS : JFA_DRAIN_TIMEOUT_NS;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (abort_flag && *abort_flag) return false;
        if (globaltimer_ns() - t0 > limit) return false;
    }
}

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, abort_flag);
}

// Drain of a ring of `stages` full barriers (at bar0, 8 bytes apart) after `count` loads
// were issued into it in order, stage i % stages for load i: waits for the last load of
// each stage.
__device__ __forceinline__ void drain_ring(uint32_t bar0, uint32_t count, uint32_t stages) {
    for (uint32_t s = 0; s < stages; ++s)
        if (count > s) {
            const uint32_t last = ((count - 1 - s) / stages) * stages + s;
            mbar_wait_bounded(bar0 + 8u * s, (last / stages) & 1, nullptr);
        }
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of one box into shared memory, completing on `bar` (complete_tx).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later async-proxy
// reads (tcgen05.mma operands, TMA stores and reduces).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D tiled reduce-add of one box from shared memory into global memory (element type and
// swizzle from the tensor map), tracked by the issuing thread's bulk async-groups: close
// the group with bulk_commit, then bulk_wait_read before the box's shared memory is
// written again, and bulk_wait_done before the thread exits.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y)
                 : "memory");
}
// 2-D tiled store of one box from shared memory to global memory, tracked like
// tma_reduce_add_2d.  A store writes every row of the box that lies inside the tensor.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Every committed group of this thread has finished reading its shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Every committed group of this thread has completed.
__device__ __forceinline__ void bulk_wait_done() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------- tcgen05 / TMEM

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
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
// True in exactly one lane of the (converged) warp: the lowest active lane.  Code
// that issues tcgen05 operations under it keeps the surrounding values warp-uniform.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 l;\n\t"
        "elect.sync l|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Element format codes of the kind::f16 instruction descriptor.
enum : uint32_t { kFmtF16 = 0, kFmtBF16 = 1 };

// Instruction descriptor (32 bits) for dense kind::f16 with an fp32
// accumulator: [4,6) D format (1 = f32), [7,10) A format, [10,13) B format,
// bit 15 A is MN-major, bit 16 B is MN-major, [17,23) N>>3, [24,29) M>>4.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t fmt, int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((uint32_t(N) >> 3) << 17) | ((uint32_t(M) >> 4) << 24);
}

// Shared-memory matrix descriptor (64 bits) for a 128-byte-swizzled operand:
// [0,14) start address >> 4, [16,30) leading-dimension byte offset >> 4,
// [32,46) stride-dimension byte offset >> 4, [46,48) = 1 (tcgen05 descriptor
// version), [49,52) base offset = 0 (atoms are 1024-byte aligned), [61,64) layout
// type 2 = SWIZZLE_128B.
//   K-major operand: rows of 128 bytes along K; SBO = 1024 (8-row group stride);
//                    LBO unused.  Advancing K inside the atom adds bytes to start.
//   MN-major operand: 128-byte rows along MN, one row per K index; LBO = stride
//                    between 128-byte MN blocks; SBO = stride between 8-deep K groups.
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= uint64_t((saddr & 0x3FFFFu) >> 4);
    d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
    d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
    d |= uint64_t(1) << 46;
    d |= uint64_t(2) << 61;
    return d;
}

// A shared-memory descriptor split into its 32-bit halves.  The start address lives
// in the low 14 bits (address >> 4), so moving an operand by `bytes` inside shared
// memory is a single 32-bit add of bytes >> 4 to `lo` (addresses stay below 256 KB,
// so the field never overflows).
struct SDesc {
    uint32_t lo, hi;
};
__device__ __forceinline__ SDesc sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    const uint64_t d = make_sdesc_sw128(saddr, lbo, sbo);
    return SDesc{uint32_t(d), uint32_t(d >> 32)};
}

// MMA issue with descriptors given as (lo + byte offset / 16, hi); the offsets are
// compile-time constants in the callers' unrolled loops, so each MMA costs an add or
// two and the instruction itself.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, SDesc a, uint32_t a_off, SDesc b, uint32_t b_off,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
        "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
        "r"(a.lo + (a_off >> 4)), "r"(a.hi), "r"(b.lo + (b_off >> 4)), "r"(b.hi), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, SDesc b, uint32_t b_off, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
        "mov.b64 db, {%2, %3};\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b.lo + (b_off >> 4)), "r"(b.hi), "r"(idesc), "r"(accumulate));
}

// tcgen05.ld 32x32b: thread t of warp w (w = warp index mod 4) reads TMEM lane
// 32*w + t; .xN reads N consecutive 32-bit columns starting at taddr's column.
#define JFA_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                  "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : JFA_R8(0), JFA_R8(8), JFA_R8(16), JFA_R8(24)
        : "r"(taddr));
}
#undef JFA_R8
#define JFA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                  "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        JFA_W8(0), JFA_W8(8), JFA_W8(16), JFA_W8(24)
        : "memory");
}
#undef JFA_W8
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
// 8-column forms of the above (8 registers), for rarely taken paths where registers
// are short.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Wait for outstanding tcgen05.ld, with the destination registers of the load as
// in/out operands: the compiler then cannot schedule any use of them above the wait.
#define JFA_RW8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), \
                   "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : JFA_RW8(0), JFA_RW8(8), JFA_RW8(16), JFA_RW8(24)::"memory");
}
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[8]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : JFA_RW8(0)::"memory");
}
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : JFA_RW8(0), JFA_RW8(8)::"memory");
}
#undef JFA_RW8
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- misc

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Packs a warp's 32 x 32 fp32 chunk (lane = row, raw = the row's 32 values as bits), each
// times `mul`, as bf16 into the warp's 2 KB staging buffer at shared address stg: row r's
// 16-byte piece q at byte 64 r + 16 (q ^ ((r >> 1) & 3)), so that any eight consecutive rows
// cover all 32 banks.  That is also the box layout of a tensor map with 64-byte box rows and
// 64-byte swizzle (16-byte chunks XORed with bits 7-8 of the address; stg 512-byte aligned).
__device__ __forceinline__ void stage_chunk_bf16(uint32_t stg, const uint32_t (&raw)[32], float mul, int lane) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        st_shared_v4(stg + uint32_t(lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4)),
                     pack_bf16x2(__uint_as_float(raw[8 * q + 0]) * mul, __uint_as_float(raw[8 * q + 1]) * mul),
                     pack_bf16x2(__uint_as_float(raw[8 * q + 2]) * mul, __uint_as_float(raw[8 * q + 3]) * mul),
                     pack_bf16x2(__uint_as_float(raw[8 * q + 4]) * mul, __uint_as_float(raw[8 * q + 5]) * mul),
                     pack_bf16x2(__uint_as_float(raw[8 * q + 6]) * mul, __uint_as_float(raw[8 * q + 7]) * mul));
    }
    __syncwarp();
}

// Writes a warp's 32 x 32 fp32 chunk (as stage_chunk_bf16) as bf16 to 32 global rows of 64
// bytes: row r at dst + r * stride (elements; 16-byte aligned), skipped unless bit r of valid
// is set.  The rows go through the staging, so every global store instruction writes eight
// whole 64-byte rows.  Stored straight from registers, each instruction would instead touch
// 32 rows, one 16-byte piece of each: four times the cache-line transactions.
__device__ __forceinline__ void store_chunk_bf16(uint32_t stg, const uint32_t (&raw)[32], float mul, int lane,
                                                 uint32_t valid, __nv_bfloat16* dst, size_t stride) {
    stage_chunk_bf16(stg, raw, mul, lane);
    const int piece = lane & 3;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = (lane >> 2) + 8 * k;
        const uint4 u = ld_shared_v4(stg + uint32_t(r * 64 + ((piece ^ ((r >> 1) & 3)) << 4)));
        if ((valid >> r) & 1u) *reinterpret_cast<uint4*>(dst + size_t(r) * stride + 8 * piece) = u;
    }
    __syncwarp();
}

// Packed dual fp32 arithmetic (fma/add on a pair of floats, one instruction).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// max(a, b, c) in one instruction (three-input max.f32, sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace jfa
