// Device-side building blocks for the sm_103a decode-linear kernels: shared
// memory barriers (mbarrier) with bounded waits, TMA tensor loads, ldmatrix,
// warp-level bf16 MMA and exact e4m3 / bf16 conversions, all as inline PTX.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dl {

// Error bits OR-ed into g_dl_device_error when a bounded wait gives up.
constexpr unsigned kErrConsumerWait = 1u;
constexpr unsigned kErrProducerWait = 2u;
constexpr unsigned kErrDrainWait = 4u;
constexpr unsigned kErrRunWait = 8u;     // split-run hand-over (ticket warp / consumers)

// Every device-side wait gives up after this long (unless a launch asks for
// another limit) and reports an error bit.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Where a bounded wait reports that it gave up (the device error word) and
// how long it waits first.
struct WaitCtl {
    unsigned* word;
    unsigned long long limit_ns;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
                 ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// w.limit_ns, ORs `err_bit` into the device error word and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const WaitCtl& w, unsigned err_bit) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
#pragma unroll 1
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > w.limit_ns) {
            atomicOr(w.word, err_bit);
            return false;
        }
    }
}

// ---------------------------------------------------------------- dependent launch

// Let the next kernel on the stream (launched with programmatic stream
// serialization) start now; it still waits for this grid's completion before
// it touches anything this grid writes.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the previous kernel on the stream has completed and its memory
// operations are visible (returns at once when there is no such kernel).
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

// One box of a one-dimensional tensor map at element c0 (c0 * element size a
// multiple of 16 bytes); elements past the tensor's end arrive as zeros.
__device__ __forceinline__ void tma_load_1d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0) {
    asm volatile(
        "cp.async.bulk.tensor.1d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0)
        : "memory");
}

// Bulk (non-tensor) copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) global -> this CTA's shared memory, counted as transaction bytes
// on the barrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// ---------------------------------------------------------------- shared loads

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, int a, int b, int c, int d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// ---------------------------------------------------------------- MMA

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- warp reductions

__device__ __forceinline__ unsigned warp_max_u32(unsigned v) {
    unsigned r;
    asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
    return r;
}

__device__ __forceinline__ unsigned warp_min_u32(unsigned v) {
    unsigned r;
    asm volatile("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
    return r;
}

// ---------------------------------------------------------------- conversions

// Four e4m3 codes (bytes 0..3 of `four`) to two f16x2: lo = (code0, code1),
// hi = (code2, code3), low byte -> low half.  Exact for every code (E4M3FN
// values are normal f16 numbers or zero; NaN codes become f16 NaN); one
// conversion-pipe instruction per pair.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t"
        ".reg .b16 c0, c1;\n\t"
        "mov.b32 {c0, c1}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, c0;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, c1;\n\t"
        "}"
        : "=r"(lo), "=r"(hi) : "r"(four));
}

// Two fp32 to f16x2 (a -> low half), round to nearest even.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float a, float b) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

// Two e4m3 codes (low byte -> low half) to two bf16, exactly.  e4m3 -> f16 is
// exact (every E4M3FN value is a normal f16 or zero; NaN stays NaN), f16 ->
// f32 is exact, and an f32 holding an e4m3 value has at most 4 significant
// bits, so its upper 16 bits ARE the bf16 encoding: one byte-permute packs
// the two upper halves.  Only the first step uses the conversion pipe.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two_codes) {
    uint32_t out;
    asm("{\n\t"
        ".reg .b16 c, lo, hi;\n\t"
        ".reg .b32 h2;\n\t"
        ".reg .f32 flo, fhi;\n\t"
        "cvt.u16.u32 c, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 h2, c;\n\t"
        "mov.b32 {lo, hi}, h2;\n\t"
        "cvt.f32.f16 flo, lo;\n\t"
        "cvt.f32.f16 fhi, hi;\n\t"
        "prmt.b32 %0, flo, fhi, 0x7632;\n\t"
        "}"
        : "=r"(out) : "r"(two_codes));
    return out;
}

// acc + a.lo * b.lo, then + a.hi * b.hi: bf16 x bf16 products are exact in
// fp32; each step is one fused multiply-add with a single rounding.
__device__ __forceinline__ float fma2_bf16(uint32_t a, uint32_t b, float acc) {
#if defined(DL_SIMT_CONVERT_FMA)
    acc = fmaf(__uint_as_float(a << 16), __uint_as_float(b << 16), acc);
    acc = fmaf(__uint_as_float(a & 0xffff0000u), __uint_as_float(b & 0xffff0000u), acc);
    return acc;
#else
    float d;
    asm("{\n\t"
        ".reg .b16 al, ah, bl, bh;\n\t"
        ".reg .f32 t;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 t, al, bl, %3;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, t;\n\t"
        "}"
        : "=f"(d) : "r"(a), "r"(b), "f"(acc));
    return d;
#endif
}

// acc + a.lo * b.lo, then + a.hi * b.hi for f16 pairs: f16 x f16 products are
// exact in fp32; each step is one fused multiply-add with a single rounding.
__device__ __forceinline__ float fma2_f16(uint32_t a, uint32_t b, float acc) {
    float d;
    asm("{\n\t"
        ".reg .b16 al, ah, bl, bh;\n\t"
        ".reg .f32 t;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 t, al, bl, %3;\n\t"
        "fma.rn.f32.f16 %0, ah, bh, t;\n\t"
        "}"
        : "=f"(d) : "r"(a), "r"(b), "f"(acc));
    return d;
}

// Global loads of 8 / 16 bytes (plain, coherent: the data may have been
// written by the previous kernel on the stream).
__device__ __forceinline__ uint2 ldg64(const void* p) {
    uint2 v;
    asm volatile("ld.global.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ldg128(const void* p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// fp32 -> bf16 bits, round to nearest even (NaN stays NaN).
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float v) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Ticket increment with acquire-release semantics at GPU scope: publishes this
// CTA's partial (ordered before by a CTA barrier) and, for the last arriver,
// makes every earlier contributor's partial visible.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Four floats (16-byte aligned) from L2, bypassing L1.
__device__ __forceinline__ float4 ld_cg_f32x4(const float* p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

// ---------------------------------------------------------------- tcgen05 (5th-gen tensor cores)

// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle (rows of 128 bytes, 8-row groups of 1024 bytes, the layout
// a SWIZZLE_128B tensor copy writes; the group base 1024-byte aligned): start
// address, leading offset (unused for this layout), stride between 8-row
// groups, descriptor version 1, layout type 2 (128-byte swizzle).  A K step
// inside the 128-byte row moves the start address by its byte offset.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3fffu);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of a dense kind::f8f6f4 MMA: fp32 accumulator, A and
// B e4m3, both K-major, M = 128 rows, N columns (a multiple of 16).
__host__ __device__ constexpr uint32_t umma_idesc_e4m3(int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// Tensor-memory allocation by one whole warp: ncols columns (a power of two
// >= 32); the address is written to shared memory at `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(slot), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[taddr] (+)= A . B^T for one K step, issued by a single thread.
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// The mbarrier receives one arrival once every MMA this thread issued before
// has completed (its shared-memory operands read, its results in TMEM).
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar) : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane (the warp reads
// the 32 lanes of its quadrant; taddr carries the quadrant's first lane).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Two fp32 -> two e4m3 codes, round to nearest even, saturating to +-448:
// a in the low byte, b in the high byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

}  // namespace dl
