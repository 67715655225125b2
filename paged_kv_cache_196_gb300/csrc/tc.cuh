// tcgen05 / TMEM / tensor-map TMA helpers (inline PTX for sm_100-family
// parts, built for sm_103a).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace pkv {
namespace tc {

// ------------------------------------------------------------ TMA (tiled)
KV_DEVICE void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

KV_DEVICE void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

KV_DEVICE void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ------------------------------------------------------------ TMEM
// Allocates `cols` tensor-memory columns (a power of two >= 32); the whole
// warp executes it.  The base address is written to *slot (shared memory).
KV_DEVICE void tmem_alloc(uint32_t *slot, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(slot)),
                 "r"(cols)
                 : "memory");
}
KV_DEVICE void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
KV_DEVICE void tmem_dealloc(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
                 : "memory");
}
KV_DEVICE void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
KV_DEVICE void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane.
KV_DEVICE void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
KV_DEVICE void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
// 16 consecutive 32-bit columns of this thread's TMEM lane.
KV_DEVICE void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
KV_DEVICE void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}
KV_DEVICE void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
KV_DEVICE void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------ UMMA
// Shared-memory matrix descriptor, 128-byte swizzle (8-row x 128-byte atoms,
// atoms 1024-byte aligned).  lbo / sbo in bytes.
// Low word: start address (bits 0-13) and leading offset (bits 16-29), both
// in 16-byte units.  Adding k to it moves the start by 16k bytes as long as
// the address field does not carry (shared-memory addresses are below 2^18).
__host__ __device__ constexpr uint32_t smem_desc_sw128_lo(uint32_t saddr, uint32_t lbo) {
    return ((saddr >> 4) & 0x3FFFu) | (((lbo >> 4) & 0x3FFFu) << 16);
}
// High word: stride offset (bits 32-45), descriptor version for this
// architecture family (bit 46), layout 128-byte swizzle (bits 61-63 = 2).
__host__ __device__ constexpr uint32_t smem_desc_sw128_hi(uint32_t sbo) {
    return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}

// Instruction descriptor for kind::f16 with bf16 A/B, fp32 accumulate.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n, bool a_mn_major,
                                                      bool b_mn_major) {
    return (1u << 4)                     // D format: f32
           | (1u << 7)                   // A format: bf16
           | (1u << 10)                  // B format: bf16
           | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Instruction descriptor for kind::f16 with fp16 A/B, fp32 accumulate.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n, bool a_mn_major,
                                                     bool b_mn_major) {
    return (1u << 4)                     // D format: f32; A and B format fields 0: f16
           | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// The eight K16 steps of one 128-deep contraction in one block of PTX, so
// that an MMA costs its two descriptor adds: D = A B^T (D += with acc_first)
// with A and B K-major 128-row tiles in shared memory, each two 64-element
// swizzle atoms 16 KiB apart.  a_lo / b_lo are the tiles' descriptor low
// words and hi their shared high word (smem_desc_sw128_lo / _hi); step kk of
// atom hh starts 16384 hh + 32 kk bytes in.
KV_DEVICE void mma_ss_k128(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                           uint32_t idesc, uint32_t acc_first) {
    asm volatile(
        "{\n\t.reg .pred p, t;\n\t.reg .b32 x, y;\n\t.reg .b64 a, b;\n\t"
        "setp.ne.u32 p, %5, 0;\n\tsetp.eq.u32 t, %5, %5;\n\t"
        "mov.b64 a, {%1, %3};\n\tmov.b64 b, {%2, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, p;\n\t"
        "add.u32 x, %1, 2;\n\tadd.u32 y, %2, 2;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
        "add.u32 x, %1, 4;\n\tadd.u32 y, %2, 4;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
        "add.u32 x, %1, 6;\n\tadd.u32 y, %2, 6;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
        "add.u32 x, %1, 1024;\n\tadd.u32 y, %2, 1024;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
        "add.u32 x, %1, 1026;\n\tadd.u32 y, %2, 1026;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
        "add.u32 x, %1, 1028;\n\tadd.u32 y, %2, 1028;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t"
        "add.u32 x, %1, 1030;\n\tadd.u32 y, %2, 1030;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, t;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(acc_first)
        : "memory");
}
// The same with A in tensor memory: D (+)= A B for 128 K values, A at
// a_tmem (step kk at column offset 8 kk: 16 fp16 values per lane), B an
// MN-major shared-memory operand whose step kk starts 2048 kk bytes in.
KV_DEVICE void mma_ts_k128(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t hi,
                           uint32_t idesc, uint32_t acc_first) {
    asm volatile(
        "{\n\t.reg .pred p, t;\n\t.reg .b32 x, y;\n\t.reg .b64 b;\n\t"
        "setp.ne.u32 p, %5, 0;\n\tsetp.eq.u32 t, %5, %5;\n\t"
        "mov.b64 b, {%2, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %4, p;\n\t"
        "add.u32 x, %1, 8;\n\tadd.u32 y, %2, 128;\n\tmov.b64 b, {y, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %4, t;\n\t"
        "add.u32 x, %1, 16;\n\tadd.u32 y, %2, 256;\n\tmov.b64 b, {y, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %4, t;\n\t"
        "add.u32 x, %1, 24;\n\tadd.u32 y, %2, 384;\n\tmov.b64 b, {y, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %4, t;\n\t"
        "add.u32 x, %1, 32;\n\tadd.u32 y, %2, 512;\n\tmov.b64 b, {y, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %4, t;\n\t"
        "add.u32 x, %1, 40;\n\tadd.u32 y, %2, 640;\n\tmov.b64 b, {y, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %4, t;\n\t"
        "add.u32 x, %1, 48;\n\tadd.u32 y, %2, 768;\n\tmov.b64 b, {y, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %4, t;\n\t"
        "add.u32 x, %1, 56;\n\tadd.u32 y, %2, 896;\n\tmov.b64 b, {y, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [x], b, %4, t;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(hi), "r"(idesc), "r"(acc_first)
        : "memory");
}
// The mbarrier receives one arrival when every tcgen05 operation issued so
// far by this thread has completed.
KV_DEVICE void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

KV_DEVICE void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Packs two floats as bf16 (round to nearest even): lo -> bits 0..15.
KV_DEVICE uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Packs two floats as fp16 (round to nearest even): lo -> bits 0..15.
KV_DEVICE uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two bf16 values (a 32-bit word, low half = lower index) as two fp16 values
// in the same positions.  Exact for magnitudes in [2^-14, 65280]; smaller
// ones become fp16 subnormals (absolute error below 2^-25); larger finite
// ones saturate to +-65504 (callers check the range); NaN stays NaN.
// *mx takes the larger of itself and both magnitudes (NaN is not counted).
KV_DEVICE uint32_t bf16x2_to_f16x2(uint32_t w, float *mx) {
    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
    *mx = fmaxf(*mx, fmaxf(fabsf(lo), fabsf(hi)));
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace tc
}  // namespace pkv
