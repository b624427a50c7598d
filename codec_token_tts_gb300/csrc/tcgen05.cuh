// Helpers shared by the tcgen05 kernels (sm_103a): shared-memory addresses and
// matrix descriptors (128-byte swizzle), bounded mbarrier waits, 2-D TMA tile
// loads, TMEM loads / stores, single-CTA MMA issue and commit.
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace ttsbb {

constexpr unsigned long long TC_TIMEOUT_NS = 1000000000ull;  // bound of every mbarrier wait

__device__ __forceinline__ uint32_t s_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long g_time() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Shared-memory matrix descriptor for a K-major operand stored as 128-byte
// rows in 128-byte-swizzle atoms of 8 rows (1024 B apart): start address >> 4
// at bits 0-13, leading offset 16 B (unused for swizzled K-major), stride
// offset 1024 B >> 4 at bits 32-45, descriptor version 1 at bit 46, layout
// SWIZZLE_128B (2) at bits 61-63.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void tc_mbar_init(uint64_t* b, int n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(s_addr(b)), "r"(n));
}
__device__ __forceinline__ bool tc_mbar_try(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(s_addr(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: false after TIMEOUT_NS or when *abort is set.
__device__ __forceinline__ bool tc_wait(uint64_t* b, uint32_t parity, volatile int* abort) {
    if (tc_mbar_try(b, parity)) return true;
    const unsigned long long t0 = g_time();
    for (uint32_t i = 0;; ++i) {
        if (tc_mbar_try(b, parity)) return true;
        if ((i & 63) == 63) {
            if (*abort) return false;
            if (g_time() - t0 > TC_TIMEOUT_NS) return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            s_addr(dst)),
        "l"(map), "r"(x), "r"(y), "r"(s_addr(bar))
        : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];" ::"r"(s_addr(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(s_addr(bar))
        : "memory");
}

// byte offset of 16-byte piece c of row r in a 128-byte-swizzled chunk
__device__ __forceinline__ uint32_t sw128_off(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// MN-major 128-byte-swizzled operand descriptor with explicit leading / stride offsets
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// 32 lanes x 32 columns of 32 bit from TMEM (no wait: tm_wait_ld before use)
__device__ __forceinline__ void tm_ld32_nw(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tm_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tm_st32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void at_mma(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void at_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(s_addr(bar)) : "memory");
}
// hardware base-2 exponential (approximate, flushes denormals); ex2(-inf) = 0
__device__ __forceinline__ float at_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Host: 2-D bf16 tensor map [rows][K] (K contiguous), box [box_rows][64], 128-byte swizzle,
// cached by (base, rows, K, box rows). False when the driver entry point is missing.
bool tc_make_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows);
// Host: 4-D bf16 tensor map [parts][B][T][C] (C contiguous, C a multiple of 8), box box_c (64 or 32)
// channels x 128 rows of one (part, item), 128- or 64-byte swizzle; out-of-range rows and channels
// read as zeros.
bool tc_make_map_rows(CUtensorMap* m, const void* base, int C, int T, int B, int parts, int box_c);
// Host: 2-D bf16 tensor map [rows][K], box [box_rows][box_k], box_k 64 (128-byte swizzle) or 32
// (64-byte swizzle).
bool tc_make_map_k(CUtensorMap* m, const void* base, int rows, int K, int box_rows, int box_k);

}  // namespace ttsbb
