// Dense Y = X W^T on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// Persistent: one CTA per SM walks the 128-token x 256-feature output tiles
// (tile = blockIdx.x, + gridDim.x, ...). A producer thread loads
// 128-byte-swizzled K-slices of X (128 x 64) and W (256 x 64) with TMA into a
// 4-stage shared-memory ring that runs on across tiles; one thread issues
// tcgen05.mma (M=128, N=256, K=16, bf16 in, fp32 accumulate) into one of two
// TMEM accumulators (2 x 256 columns) and commits each stage back to the
// producer through an mbarrier; sixteen epilogue warps drain the other
// accumulator with tcgen05.ld (four per 32-lane quarter of TMEM = 32 token
// rows, 64 columns each) while the next tile accumulates, applying the same
// fused epilogues as the other linear kernels (fp32 store, residual add,
// SwiGLU over interleaved gate/up columns, logits + argmax, permuted
// audio-head logits).
//
// Every mbarrier wait is bounded; on timeout the CTA raises the error word,
// stops issuing work, waits (bounded) for its copies and MMAs in flight,
// frees TMEM and returns.
#include <algorithm>
#include <mutex>
#include <unordered_map>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

#include <array>
#include "tcgen05.cuh"

namespace ttsbb {

namespace tc {
constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPW = 16;  // epilogue warps: EPW / 4 per TMEM lane quarter, BN / (EPW / 4) columns each
constexpr int OST = 32 * 16 * 4;                       // per epilogue warp: [32 rows][16 fp32] store staging
constexpr int OST_OFF = STAGES * STAGE_BYTES;          // staging buffers, then the barriers
constexpr int BAR_OFF = OST_OFF + EPW * OST;
constexpr int SMEM = BAR_OFF + 256 + 1024;             // + alignment of the dynamic base
constexpr int TMEM_COLS = 2 * BN;  // two accumulators
constexpr int NT = 64 + 32 * EPW;  // warp 0 TMA, warp 1 MMA + TMEM owner, then the epilogue warps
constexpr unsigned long long TIMEOUT_NS = TC_TIMEOUT_NS;
// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A bf16 (7-9 = 1),
// B bf16 (10-12 = 1), both K-major (15, 16 = 0), N >> 3 at 17-22, M >> 4 at 24-28.
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);
}  // namespace tc
static_assert(tc::SMEM <= 232448, "shared memory per CTA");

__device__ __forceinline__ float silu_tc(float x) { return x / (1.f + __expf(-x)); }

// Apply the epilogue to 16 consecutive accumulator columns of one token row.
__device__ __forceinline__ void tc_epilogue16(const Epi& e, int t, int n0, int N, const float* v,
                                              unsigned long long& best) {
    switch (e.mode) {
        case EPI_STORE_F32:
        case EPI_ADD_F32: {
            float* row = reinterpret_cast<float*>(e.out) + (size_t)t * e.ldo + n0;
            if (n0 + 16 <= N) {
#pragma unroll
                for (int j = 0; j < 16; j += 4) {
                    float4 o = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                    if (e.mode == EPI_ADD_F32) {
                        const float4 p = *reinterpret_cast<const float4*>(row + j);
                        o.x += p.x; o.y += p.y; o.z += p.z; o.w += p.w;
                    }
                    *reinterpret_cast<float4*>(row + j) = o;
                }
            } else {
                for (int j = 0; j < 16 && n0 + j < N; ++j) row[j] = (e.mode == EPI_ADD_F32 ? row[j] : 0.f) + v[j];
            }
            break;
        }
        case EPI_STORE_BF16: {
            bf16* row = reinterpret_cast<bf16*>(e.out) + (size_t)t * e.ldo + n0;
            for (int j = 0; j < 16 && n0 + j < N; ++j) row[j] = f2bf(v[j]);
            break;
        }
        case EPI_SWIGLU: {  // columns (2i, 2i+1) = (gate_i, up_i)
            bf16* row = reinterpret_cast<bf16*>(e.out) + (size_t)t * e.ldo + n0 / 2;
            bf16* rlo = e.out_lo ? reinterpret_cast<bf16*>(e.out_lo) + (size_t)t * e.ldo + n0 / 2 : nullptr;
            if (n0 + 16 <= N) {
                uint32_t pk[4], pl[4];
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    const float m0 = silu_tc(v[2 * j]) * v[2 * j + 1];
                    const float m1 = silu_tc(v[2 * j + 2]) * v[2 * j + 3];
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(m0, m1);
                    pk[j / 2] = *reinterpret_cast<uint32_t*>(&h2);
                    __nv_bfloat162 l2 = __halves2bfloat162(f2bf_lo(m0), f2bf_lo(m1));
                    pl[j / 2] = *reinterpret_cast<uint32_t*>(&l2);
                }
                *reinterpret_cast<uint4*>(row) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                if (rlo) *reinterpret_cast<uint4*>(rlo) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
            } else {
                for (int j = 0; 2 * j + 1 < 16 && n0 + 2 * j + 1 < N; ++j) {
                    const float mv = silu_tc(v[2 * j]) * v[2 * j + 1];
                    row[j] = f2bf(mv);
                    if (rlo) rlo[j] = f2bf_lo(mv);
                }
            }
            break;
        }
        case EPI_LOGITS: {
            float* row = e.out ? reinterpret_cast<float*>(e.out) + (size_t)t * e.ldo + n0 : nullptr;
            for (int j = 0; j < 16 && n0 + j < N; ++j) {
                if (row) row[j] = v[j];
                const unsigned long long pk = pack_argmax(v[j], n0 + j);
                best = pk > best ? pk : best;
            }
            break;
        }
        case EPI_LOGITS_PERM: {
            const int b = t / e.perm_rows, s = t % e.perm_rows;
            float* out = reinterpret_cast<float*>(e.out);
            for (int j = 0; j < 16 && n0 + j < N; ++j) {
                const int n = n0 + j, k = n / e.perm_vocab, vv = n % e.perm_vocab;
                out[(((size_t)b * e.perm_groups + k) * e.perm_rows + s) * e.perm_vocab + vv] = v[j];
            }
            break;
        }
        default:
            break;
    }
}

// 16 consecutive fp32 accumulator columns of this thread's TMEM lane (warp-collective)
__device__ __forceinline__ void tc_ld16(uint32_t ta, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(ta));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// Bulk tensor store / reduce-add of a shared-memory box (async proxy), and their group waits.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, const void* src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(x), "r"(y),
                 "r"(s_addr(src))
                 : "memory");
}
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, int x, int y, const void* src) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map),
                 "r"(x), "r"(y), "r"(s_addr(src))
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// With split = 1 the activations come as bf16 high + low parts (tmA, tmAl): the k-loop runs over
// K twice, Y = X_hi W^T + X_lo W^T, the second pass reading the same weight tiles (from L2).
// EPI_STORE_F32 / EPI_ADD_F32 leave through tmO (the fp32 output [T][ldo], boxes of 32 rows x 16
// columns, 64-byte swizzle): each epilogue warp stages its 32 rows x 16 columns in shared memory and
// one lane issues a bulk tensor store (or reduce-add, for the residual), so the stores are full
// coalesced boxes instead of one 16-byte piece per row per instruction. EPI_SWIGLU does the same
// with its 32 rows x 32 bf16 outputs (64 columns of gate/up pairs) through tmO, and the low parts
// through tmOl when the output has them.
__global__ void __launch_bounds__(tc::NT, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAl,
              const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmO,
              const __grid_constant__ CUtensorMap tmOl, int split, int T, int N, int K, const __grid_constant__ Epi e,
              int* err) {
    using namespace tc;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char* sA = smem;
    unsigned char* sB = smem + STAGES * A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
    uint64_t* empty = full + STAGES;
    uint64_t* accf = empty + STAGES;  // [2] accumulator ready (MMA -> epilogue)
    uint64_t* acce = accf + 2;        // [2] accumulator drained (epilogue -> MMA), 4 warp arrivals
    uint64_t* fin = acce + 2;         // every MMA issued by this CTA has completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
    volatile int* abort_s = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int MT = (T + BM - 1) / BM, NTL = (N + BN - 1) / BN, tiles = MT * NTL, KT = K / BK, KT2 = split ? 2 * KT : KT;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc_mbar_init(full + s, 1);
            tc_mbar_init(empty + s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc_mbar_init(accf + i, 1);
            tc_mbar_init(acce + i, EPW);
        }
        tc_mbar_init(fin, 1);
        *abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s_addr(tmem_slot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // barriers and TMEM are set up; activations (and the output) come from upstream kernels
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer: the stage ring runs on across tiles
            uint32_t g = 0;  // k-blocks issued
            for (int tile = blockIdx.x; tile < tiles && !*abort_s; tile += gridDim.x) {
                const int m0 = (tile % MT) * BM, n0 = (tile / MT) * BN;
                for (int kt = 0; kt < KT2; ++kt, ++g) {
                    const int s = g % STAGES, kx = (kt < KT ? kt : kt - KT) * BK;
                    if (g >= STAGES && !tc_wait(empty + s, ((g / STAGES) - 1) & 1, abort_s)) {
                        *abort_s = 1;
                        break;
                    }
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(s_addr(full + s)),
                                 "r"(STAGE_BYTES)
                                 : "memory");
                    tma_load_2d(sA + s * A_BYTES, kt < KT ? &tmA : &tmAl, kx, m0, full + s);
                    tma_load_2d(sB + s * B_BYTES, &tmB, kx, n0, full + s);
                }
            }
            if (*abort_s) {  // let the copies in flight (the last STAGES issued) land before the CTA can exit
                for (uint32_t i = g > (uint32_t)STAGES ? g - STAGES : 0; i < g; ++i) {
                    const unsigned long long t0 = g_time();
                    while (!tc_mbar_try(full + i % STAGES, (i / STAGES) & 1) && g_time() - t0 < TIMEOUT_NS) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------- MMA issuer
            uint32_t g = 0;  // k-blocks consumed
            int it = 0;      // tiles of this CTA
            bool ok = true;
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x, ++it) {
                const int buf = it & 1;
                if (it >= 2 && !tc_wait(acce + buf, ((it >> 1) - 1) & 1, abort_s)) {  // epilogue drained it
                    *abort_s = 1;
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t d = tmem + (uint32_t)(buf * BN);
                for (int kt = 0; kt < KT2; ++kt, ++g) {
                    const int s = g % STAGES;
                    if (!tc_wait(full + s, (g / STAGES) & 1, abort_s)) {
                        *abort_s = 1;
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t a0 = s_addr(sA + s * A_BYTES), b0 = s_addr(sB + s * B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint64_t ad = sw128_desc(a0 + k * 32), bd = sw128_desc(b0 + k * 32);
                        const uint32_t acc = (kt | k) ? 1u : 0u;
                        asm volatile(
                            "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                            " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
                            "l"(ad), "l"(bd), "r"(IDESC), "r"(acc));
                    }
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                        s_addr(empty + s))
                                 : "memory");
                }
                if (!ok) break;
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                    s_addr(accf + buf))
                             : "memory");
            }
            // every MMA issued so far completes before TMEM may be freed
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(s_addr(fin))
                         : "memory");
            const unsigned long long t0 = g_time();
            while (!tc_mbar_try(fin, 0) && g_time() - t0 < TIMEOUT_NS) {
            }
        }
    } else {
        // ---------------- epilogue: warp w reads TMEM lanes 32 * (w % 4) .. of the tile's accumulator,
        // columns [h CW, (h + 1) CW) with h = (w - 2) / 4
        constexpr int CW = BN / (EPW / 4);
        const int q = warp & 3, h = (warp - 2) >> 2;
        const bool tma_out = e.mode == EPI_STORE_F32 || e.mode == EPI_ADD_F32;
        const bool tma_swiglu = e.mode == EPI_SWIGLU;
        const bool tma_bf16 = e.mode == EPI_STORE_BF16;
        unsigned char* ost = smem + OST_OFF + (warp - 2) * OST;
        int it = 0;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++it) {
            const int buf = it & 1;
            if (!tc_wait(accf + buf, (it >> 1) & 1, abort_s) || *abort_s) {
                if (lane == 0 && q == 0) set_err(err, ERR_TIMEOUT);
                *abort_s = 1;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int m0 = (tile % MT) * BM, n0 = (tile / MT) * BN;
            const int t = m0 + q * 32 + lane;
            unsigned long long best = 0ull;
            if (tma_out) {  // fp32 store / residual add through the staged boxes
                for (int c = h * CW; c < (h + 1) * CW; c += 16) {
                    float v[16];
                    tc_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + c), v);
                    if (lane == 0) bulk_wait_read0();  // the previous box has been read out of the staging buffer
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 4; ++k)  // 16-byte piece k of row `lane`, 64-byte swizzle
                        *reinterpret_cast<float4*>(ost + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) =
                            make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0 && n0 + c < N && m0 + q * 32 < T) {
                        if (e.mode == EPI_ADD_F32)
                            tma_reduce_add_2d(&tmO, n0 + c, m0 + q * 32, ost);
                        else
                            tma_store_2d(&tmO, n0 + c, m0 + q * 32, ost);
                        bulk_commit();
                    }
                }
            }
            if (tma_swiglu) {  // 64 gate/up columns -> 32 bf16 outputs per row, staged as one 64-byte row
                uint32_t lo_pk[4][4];
                if (lane == 0) bulk_wait_read0();
                __syncwarp();
#pragma unroll
                for (int k = 0; k < CW / 16; ++k) {
                    float v[16];
                    tc_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + h * CW + 16 * k), v);
                    uint32_t pk[4];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const float m0v = silu_tc(v[4 * jj]) * v[4 * jj + 1];
                        const float m1v = silu_tc(v[4 * jj + 2]) * v[4 * jj + 3];
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(m0v, m1v);
                        pk[jj] = *reinterpret_cast<uint32_t*>(&h2);
                        __nv_bfloat162 l2 = __halves2bfloat162(f2bf_lo(m0v), f2bf_lo(m1v));
                        lo_pk[k][jj] = *reinterpret_cast<uint32_t*>(&l2);
                    }
                    *reinterpret_cast<uint4*>(ost + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                const int xo = (n0 + h * CW) / 2, yo = m0 + q * 32;
                const bool in = n0 + h * CW < N && yo < T;
                if (lane == 0 && in) {
                    tma_store_2d(&tmO, xo, yo, ost);
                    bulk_commit();
                }
                if (e.out_lo) {
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < CW / 16; ++k)
                        *reinterpret_cast<uint4*>(ost + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) =
                            make_uint4(lo_pk[k][0], lo_pk[k][1], lo_pk[k][2], lo_pk[k][3]);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0 && in) {
                        tma_store_2d(&tmOl, xo, yo, ost);
                        bulk_commit();
                    }
                }
            }
            if (tma_bf16) {  // bf16 store: two 16-column chunks per staged 64-byte row, one box per pair
                for (int c = h * CW; c < (h + 1) * CW; c += 32) {
                    float v[32];
                    tc_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + c), v);
                    tc_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + c + 16), v + 16);
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t pk[4];
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * k + 2 * jj], v[8 * k + 2 * jj + 1]);
                            pk[jj] = *reinterpret_cast<uint32_t*>(&h2);
                        }
                        *reinterpret_cast<uint4*>(ost + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0 && n0 + c < N && m0 + q * 32 < T) {
                        tma_store_2d(&tmO, n0 + c, m0 + q * 32, ost);
                        bulk_commit();
                    }
                }
            }
            for (int c = h * CW; c < (h + 1) * CW && !tma_out && !tma_swiglu && !tma_bf16; c += 16) {
                uint32_t r[16];
                const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN + c);
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
                    "[%16];"
                    : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                      "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                      "=r"(r[14]), "=r"(r[15])
                    : "r"(ta));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (t < T && n0 + c < N) {
                    float v[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
                    tc_epilogue16(e, t, n0 + c, N, v, best);
                }
            }
            if (e.mode == EPI_LOGITS && e.amax && t < T && best) atomicMax(e.amax + t, best);
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(s_addr(acce + buf)) : "memory");
        }
        if ((tma_out || tma_swiglu || tma_bf16) && lane == 0) bulk_wait0();  // every bulk store of this warp has completed
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
    }
}

// ---------------------------------------------------------------- decode batches (8 < T <= 256)
// Y = (X_hi + X_lo) W^T for a handful of tokens, weights streamed once. The
// roles swap so the weights fill the 128-row M side: A = a 128-row tile of W,
// B = the tokens' high parts (rows 0..TB-1) stacked on their low parts
// (rows TB..2TB-1), N = 2 TB. TB is at most 128 (N <= 256), so a grid row
// takes one block of up to 128 tokens; a launch over 129..256 tokens has two
// grid rows (or is issued as two launches, one per block). The S CTAs of one
// thread-block cluster split K for one 128-row tile and one token block; each
// sums hi + lo per token into its shared memory. After a cluster barrier,
// CTA r owns the block's tokens [r T / S, (r+1) T / S): every
// CTA pushes each peer's token slice of its partial with one bulk copy into
// that peer's receive buffer (completion on the peer's mbarrier); the owner
// adds the S partials in rank order (deterministic) and applies the epilogue,
// one thread per output feature.
namespace tcd {
constexpr int EPW = 16;  // epilogue warps (EPW / 4 per TMEM lane quarter)
constexpr int BM = 128, BK = 64, STAGES = 4, NT = 64 + 32 * EPW;  // warp 0 TMA, warp 1 MMA, then the epilogue
constexpr int MAXTB = 128;                          // tokens per CTA (one token block)
constexpr int MAXBLK = 4;                           // token blocks per launch (grid y)
constexpr int A_BYTES = BM * BK * 2;                // 16 KB
constexpr int STAGE = A_BYTES + 2 * MAXTB * BK * 2; // 48 KB
constexpr int SMEM = STAGES * STAGE + 1024 + 256;
constexpr int MAXS = 16;
static_assert((2 * MAXTB + MAXS) * BM * 4 <= STAGES * STAGE, "partials and receive buffer must fit the stages");
}  // namespace tcd
constexpr unsigned long long TIMEOUT_NS_TCD = tc::TIMEOUT_NS;

// Address of `local` in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(s_addr(local)), "r"(rank));
    return remote;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Epilogue arguments held in registers (the kernel's Epi lives in local
// memory; stores through its generic pointers would force reloads).
struct TcdOut {
    float* __restrict__ f32;          // STORE / ADD / LOGITS output (LOGITS: may be null)
    bf16* __restrict__ hi;            // SWIGLU output
    bf16* __restrict__ lo;            // SWIGLU low part (may be null)
    unsigned long long* __restrict__ amax;
    int ldo;
    // folded RMSNorm (see Epi): producer outputs (rows of this token block) and consumer scale
    const bf16* __restrict__ ng;
    bf16* __restrict__ ny;
    bf16* __restrict__ nylo;
    float* __restrict__ nss;          // [8][Ttot], absolute token index
    const float* __restrict__ css;    // [8][Ttot] (the scales themselves are preloaded: TcdPre)
    int Ttot, tb0;
};

// 1 / RMS of token tg from the 8 per-tile sums of squares of its 1024 features (fixed order)
__device__ __forceinline__ float tcd_norm_scale(const float* __restrict__ ss, int Ttot, int tg, float eps) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += ss[(size_t)i * Ttot + tg];
    return rsqrtf(s * (1.f / 1024.f) + eps);
}

// Per-token epilogue inputs that do not depend on the product, read by the epilogue warps while
// the MMAs run (one round trip for all of a warp's tokens instead of one or more per token): the
// folded norm's inverse RMS (consumers), the residual slice h[t][n .. n + 3] and the gains
// (EPI_ADD_F32), or the token's position and cache block (EPI_QKROPE). Entry i is token
// t0 + w + i * EPW of the warp; lane i < 8 computes the per-token scalars and broadcasts them.
constexpr int TCD_TPW = tcd::MAXTB / tcd::EPW;  // tokens per epilogue warp at most (one split)
static_assert(TCD_TPW <= 32, "per-token scalars are computed one per lane");
struct TcdPre {
    float rs[TCD_TPW];   // folded-norm scale (1 without a folded norm)
    uint4 pv[TCD_TPW];   // EPI_ADD_F32: the residual float4; EPI_QKROPE: {pos, cache block or -1, valid, 0}
    uint2 gam;           // EPI_ADD_F32 with a norm output: the gains of features n .. n + 3 (bf16)
};
__device__ __forceinline__ void tcd_preload(TcdPre& P, const Epi& e, int t0, int t1, int tb0, int n0, int N, int w,
                                            int lane) {
    const int n = n0 + lane * 4;
    const int ti = t0 + w + lane * tcd::EPW;  // this lane's token (lanes < TCD_TPW)
    float my_rs = 1.f;
    int my_pos = 0, my_phys = -1, my_valid = 0;
    if (lane < TCD_TPW && ti < t1) {
        const int tg = tb0 + ti;
        if (e.nrm_scale_ss) my_rs = tcd_norm_scale(e.nrm_scale_ss, e.nrm_T, tg, e.nrm_eps);
        if (e.mode == EPI_QKROPE) {
            const EpiQk& k = e.qk;
            const int seq = tg / k.tok_per_seq, s = tg - seq * k.tok_per_seq;
            my_valid = s < k.seq_len[seq];
            my_pos = k.seq_start[seq] + s;
            if (my_valid && n0 / HD >= NQ) {  // k / v head: the cache block that receives this token
                const int j = my_pos / KVB;
                my_phys = k.kv.page_table ? k.kv.page_table[(size_t)k.kv.seq_slot[seq] * k.kv.mbps + j] : seq * k.kv.mbps + j;
                if (my_phys < 0) {
                    set_err(k.err, ERR_KV_RANGE);
                    my_phys = -1;
                }
            }
        }
    }
    const bool add = e.mode == EPI_ADD_F32 && n + 4 <= N;
#pragma unroll
    for (int i = 0; i < TCD_TPW; ++i) {
        P.rs[i] = __shfl_sync(0xffffffffu, my_rs, i);
        P.pv[i] = make_uint4((uint32_t)__shfl_sync(0xffffffffu, my_pos, i), (uint32_t)__shfl_sync(0xffffffffu, my_phys, i),
                             (uint32_t)__shfl_sync(0xffffffffu, my_valid, i), 0u);
        const int t = t0 + w + i * tcd::EPW;
        if (add && t < t1) P.pv[i] = *reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(e.out) + (size_t)(tb0 + t) * e.ldo + n);
    }
    P.gam = add && e.nrm_gamma ? *reinterpret_cast<const uint2*>(e.nrm_gamma + n) : make_uint2(0u, 0u);
}

// Rank-order sum of the S partials of token t (local index tl of nt_all), features f .. f + 3:
// this CTA's own (rank r) in red, the peers' in recv.
__device__ __forceinline__ float4 tcd_sum(const float* __restrict__ red, const float* __restrict__ recv, int t, int tl,
                                          int nt_all, uint32_t S, uint32_t r, int f) {
    constexpr int BM = tcd::BM;
    if (S == 1) return *reinterpret_cast<const float4*>(red + (size_t)t * BM + f);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = 0; p0 < (int)S; p0 += 4) {
        float4 x[4];
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
            const int p = min(p0 + pp, (int)S - 1);
            const float* src = p == (int)r ? red + (size_t)t * BM + f : recv + ((size_t)p * nt_all + tl) * BM + f;
            x[pp] = *reinterpret_cast<const float4*>(src);
        }
#pragma unroll
        for (int pp = 0; pp < 4; ++pp)
            if (p0 + pp < (int)S) { v.x += x[pp].x; v.y += x[pp].y; v.z += x[pp].z; v.w += x[pp].w; }
    }
    return v;
}

// Sum, in rank order, the S partials of tokens [t0, t1) (this CTA's own
// partial in `red`, the peers' in `recv`) and apply the epilogue. Epilogue
// warp w (of EPW) takes tokens t0 + w, t0 + w + EPW, ...; lane l takes the four features
// n0 + 4l .. 4l + 3 (vector loads and stores; a gate/up pair stays in one lane).
template <int MODE>
__device__ __forceinline__ void tcd_reduce(const TcdOut o, const TcdPre& P, const float* __restrict__ red,
                                           const float* __restrict__ recv, int t0, int t1, uint32_t S, uint32_t r,
                                           int n0, int N, int w, int lane) {
    const int nt_all = t1 - t0, f = lane * 4, n = n0 + f;
#pragma unroll
    for (int i = 0; i < TCD_TPW; ++i) {
        const int t = t0 + w + i * tcd::EPW;
        if (t >= t1) break;
        const int tl = t - t0;
        float4 v = tcd_sum(red, recv, t, tl, nt_all, S, r, f);
        const size_t row = (size_t)t * o.ldo;
        if (MODE != EPI_ADD_F32 && o.css) {  // the folded RMSNorm of this product's input rows
            const float rs = P.rs[i];
            v.x *= rs; v.y *= rs; v.z *= rs; v.w *= rs;
        }
        if (MODE == EPI_STORE_F32 || MODE == EPI_ADD_F32) {
            float* dst = o.f32 + row + n;
            if (n + 4 <= N) {
                if (MODE == EPI_ADD_F32) {
                    v.x += __uint_as_float(P.pv[i].x); v.y += __uint_as_float(P.pv[i].y);
                    v.z += __uint_as_float(P.pv[i].z); v.w += __uint_as_float(P.pv[i].w);
                }
                *reinterpret_cast<float4*>(dst) = v;
                if (MODE == EPI_ADD_F32 && o.ng) {  // the next norm's input: h * gamma, and this tile's sum of squares
                    const uint2 gr = P.gam;
                    const float g0 = __uint_as_float(gr.x << 16), g1 = __uint_as_float(gr.x & 0xFFFF0000u);
                    const float g2 = __uint_as_float(gr.y << 16), g3 = __uint_as_float(gr.y & 0xFFFF0000u);
                    const float f0 = v.x * g0, f1 = v.y * g1, f2 = v.z * g2, f3 = v.w * g3;
                    __nv_bfloat162 a2 = __floats2bfloat162_rn(f0, f1), b2 = __floats2bfloat162_rn(f2, f3);
                    uint2 hv;
                    hv.x = *reinterpret_cast<uint32_t*>(&a2);
                    hv.y = *reinterpret_cast<uint32_t*>(&b2);
                    *reinterpret_cast<uint2*>(o.ny + (size_t)t * 1024 + n) = hv;
                    __nv_bfloat162 al = __halves2bfloat162(f2bf_lo(f0), f2bf_lo(f1));
                    __nv_bfloat162 bl = __halves2bfloat162(f2bf_lo(f2), f2bf_lo(f3));
                    hv.x = *reinterpret_cast<uint32_t*>(&al);
                    hv.y = *reinterpret_cast<uint32_t*>(&bl);
                    *reinterpret_cast<uint2*>(o.nylo + (size_t)t * 1024 + n) = hv;
                    const float ssp = warp_sum(v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w);
                    if (lane == 0) o.nss[(size_t)(n0 / 128) * o.Ttot + o.tb0 + t] = ssp;
                }
            } else {
                const float vv[4] = {v.x, v.y, v.z, v.w};
                for (int j = 0; j < 4 && n + j < N; ++j) dst[j] = (MODE == EPI_ADD_F32 ? dst[j] : 0.f) + vv[j];
            }
        } else if (MODE == EPI_SWIGLU) {  // features (2i, 2i+1) = (gate_i, up_i)
            if (n + 4 <= N) {
                const float m0 = silu_tc(v.x) * v.y, m1 = silu_tc(v.z) * v.w;
                __nv_bfloat162 h2 = __floats2bfloat162_rn(m0, m1);
                *reinterpret_cast<__nv_bfloat162*>(o.hi + row + n / 2) = h2;
                if (o.lo) *reinterpret_cast<__nv_bfloat162*>(o.lo + row + n / 2) = __halves2bfloat162(f2bf_lo(m0), f2bf_lo(m1));
            } else if (n + 2 <= N) {
                const float m0 = silu_tc(v.x) * v.y;
                o.hi[row + n / 2] = f2bf(m0);
                if (o.lo) o.lo[row + n / 2] = f2bf_lo(m0);
            }
        } else {  // EPI_LOGITS
            const float vv[4] = {v.x, v.y, v.z, v.w};
            unsigned long long best = 0ull;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (n + j < N) {
                    if (o.f32) o.f32[row + n + j] = vv[j];
                    const unsigned long long pk = pack_argmax(vv[j], n + j);
                    best = pk > best ? pk : best;
                }
#pragma unroll
            for (int sh = 16; sh >= 1; sh >>= 1) {
                const unsigned long long x = __shfl_xor_sync(0xffffffffu, best, sh);
                best = x > best ? x : best;
            }
            if (lane == 0 && o.amax && best) atomicMax(o.amax + t, best);
        }
    }
}

// EPI_QKROPE on the decode GEMM: this CTA's 128 features are one head (n0 / 128: q 0..15, k 16..23,
// v 24..31). Per token (warp w takes tokens t0 + w, t0 + w + EPW, ..., lane l features 4l .. 4l + 3)
// the rank-order sum of the partials, then the same arithmetic as the separate q/k norm + RoPE +
// append kernel: the head's RMSNorm (warp sum of squares) and gain, the rotation of dims (i, i + 64)
// by pos * theta^(-2i/128) with the partner dims in lane l ^ 16 (omnivoice-cpp, Qwen3 specifics:
// per-head RMSNorm before RoPE; Qwen3-TTS ncnn port: 1-D half-rotate RoPE); q to q / qf, k and v
// appended to the paged cache. tb0: the block's first token in the launch.
__device__ __forceinline__ void tcd_qkrope(const EpiQk& k, const TcdPre& P, const float* __restrict__ red,
                                           const float* __restrict__ recv, int t0, int t1, uint32_t S, uint32_t r,
                                           int n0, int w, int lane, int tb0, bool scaled) {
    const int nt_all = t1 - t0, f = lane * 4, u = n0 / HD;
    const bool isq = u < NQ;
    const int hh = isq ? u : u - NQ;
    float gmv[4];  // this lane's q or k norm gains
#pragma unroll
    for (int e = 0; e < 4; ++e) gmv[e] = bf2f((isq ? k.qn : k.kn)[lane * 4 + e]);
#pragma unroll
    for (int i = 0; i < TCD_TPW; ++i) {
        const int t = t0 + w + i * tcd::EPW;
        if (t >= t1) break;
        const int tl = t - t0;
        float4 x = tcd_sum(red, recv, t, tl, nt_all, S, r, f);
        const int tg = tb0 + t;
        if (scaled) {  // the folded input RMSNorm of this token
            const float rs = P.rs[i];
            x.x *= rs; x.y *= rs; x.z *= rs; x.w *= rs;
        }
        const int pos = (int)P.pv[i].x, phys = (int)P.pv[i].y;
        const bool valid = P.pv[i].z != 0u;
        // the cache row of a k / v head's valid token (phys < 0: no append)
        bf16* kdst = phys >= 0 ? k.kv.pool + (size_t)phys * 2 * NKV * KVB * HD + (size_t)(pos % KVB) * HD : nullptr;
        if (u >= NQ + NKV) {  // v head: copied into the cache
            if (kdst) {
                __nv_bfloat162 a2 = __floats2bfloat162_rn(x.x, x.y), b2 = __floats2bfloat162_rn(x.z, x.w);
                uint2 o;
                o.x = *reinterpret_cast<uint32_t*>(&a2);
                o.y = *reinterpret_cast<uint32_t*>(&b2);
                *reinterpret_cast<uint2*>(kdst + (size_t)NKV * KVB * HD + (size_t)(u - NQ - NKV) * KVB * HD + f) = o;
            }
            continue;
        }
        if (!isq && !kdst) continue;
        const float ss = warp_sum(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w);
        const float rn = rsqrtf(ss * (1.f / HD) + k.eps);
        float v[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = v[e] * rn * gmv[e];
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pv[e] = __shfl_xor_sync(0xffffffffu, v[e], 16);
        const int i0 = (lane & 15) * 4;
        const float* ct = k.cos_t + (size_t)pos * (HD / 2) + i0;
        const float* st = k.sin_t + (size_t)pos * (HD / 2) + i0;
        float o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float c = valid ? ct[e] : 1.f, sn = valid ? st[e] : 0.f;
            o[e] = (lane < 16) ? (v[e] * c - pv[e] * sn) : (v[e] * c + pv[e] * sn);
        }
        __nv_bfloat162 a2 = __floats2bfloat162_rn(o[0], o[1]), b2 = __floats2bfloat162_rn(o[2], o[3]);
        uint2 wv;
        wv.x = *reinterpret_cast<uint32_t*>(&a2);
        wv.y = *reinterpret_cast<uint32_t*>(&b2);
        if (isq && k.qf) {
            const float4 f4 = valid ? make_float4(o[0], o[1], o[2], o[3]) : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(k.qf + (size_t)tg * NQ * HD + hh * HD + f) = f4;
        } else if (isq) {
            if (!valid) wv = make_uint2(0u, 0u);
            *reinterpret_cast<uint2*>(k.q + (size_t)tg * NQ * HD + hh * HD + f) = wv;
        } else {
            *reinterpret_cast<uint2*>(kdst + (size_t)hh * KVB * HD + f) = wv;
        }
    }
}

__global__ void __launch_bounds__(tcd::NT, 1)
    k_gemm_tcd(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmXh,
               const __grid_constant__ CUtensorMap tmXl, int T, int TB, int tb_base, int N, int K,
               const __grid_constant__ Epi e, int* err) {
    using namespace tcd;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    // a stage holds one weight tile and the token block's high and low tiles: sized by TB, so a
    // small token block leaves room for a second CTA (of the next kernel) on the SM
    const int STG = A_BYTES + 2 * TB * BK * 2;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STG);
    uint64_t* empty = full + STAGES;
    uint64_t* accf = empty + STAGES;
    uint64_t* recvb = accf + 1;  // peers' slices of this CTA's tokens have landed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(recvb + 1);
    volatile int* abort_s = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // over the stages once the MMAs are done: this CTA's partial sums [TB][128], then the
    // receive buffer [S][tokens of this CTA][128]
    float* red = reinterpret_cast<float*>(smem);
    float* recv = red + TB * BM;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t S, r;
    asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(S));
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    const int n0 = (int)(blockIdx.x / S) * BM;
    // this CTA's tokens: [tb0, tb0 + Th), one block of up to MAXTB per grid row
    const int tb0 = tb_base + (int)blockIdx.y * MAXTB, Th = min(T - tb0, MAXTB);
    const int KT = K / BK, kb0 = (int)(r * KT / S), nk = (int)((r + 1) * KT / S) - kb0;
    const uint32_t b_bytes = 2u * TB * BK * 2, ncols = 2u * TB;
    const uint32_t tcols = ncols <= 32 ? 32 : ncols <= 64 ? 64 : ncols <= 128 ? 128 : 256;
    // kind::f16, D f32, A/B bf16 K-major, N = 2 TB, M = 128
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((ncols >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc_mbar_init(full + s, 1);
            tc_mbar_init(empty + s, 1);
        }
        tc_mbar_init(accf, 1);
        tc_mbar_init(recvb, 1);
        *abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s_addr(tmem_slot)),
                     "r"(tcols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;
    pdl_trigger();
    if (!(warp == 0 && lane == 0)) pdl_wait();  // activations (and the output) come from upstream kernels
    // tokens owned by CTA q: [tok(q), tok(q + 1))
    auto tok = [&](uint32_t q) { return (int)(q * (uint32_t)Th / S); };
    const int t0 = tok(r), t1 = tok(r + 1);
    TcdPre pre;

    if (warp == 0) {
        if (lane == 0) {  // TMA producer
            // the weights do not depend on upstream kernels: the first stages' weight tiles are
            // requested before waiting for them, the activation tiles after
            const int pre = nk < STAGES ? nk : STAGES;
            for (int i = 0; i < pre; ++i) {
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(s_addr(full + i)),
                             "r"((uint32_t)A_BYTES + b_bytes)
                             : "memory");
                tma_load_2d(smem + i * STG, &tmW, (kb0 + i) * BK, n0, full + i);
            }
            pdl_wait();
            int issued = 0;
            for (int i = 0; i < nk; ++i) {
                const int s = i % STAGES;
                if (i >= STAGES && !tc_wait(empty + s, ((i / STAGES) - 1) & 1, abort_s)) {
                    *abort_s = 1;
                    break;
                }
                unsigned char* st = smem + s * STG;
                const int kx = (kb0 + i) * BK;
                if (i >= pre) {
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(s_addr(full + s)),
                                 "r"((uint32_t)A_BYTES + b_bytes)
                                 : "memory");
                    tma_load_2d(st, &tmW, kx, n0, full + s);
                }
                tma_load_2d(st + A_BYTES, &tmXh, kx, tb0, full + s);
                tma_load_2d(st + A_BYTES + TB * BK * 2, &tmXl, kx, tb0, full + s);
                ++issued;
            }
            if (*abort_s && issued < pre) issued = pre;  // weight tiles already requested must land too
            if (*abort_s) {
                for (int i = 0; i < issued; ++i) {
                    const unsigned long long t0 = g_time();
                    while (!tc_mbar_try(full + i % STAGES, (i / STAGES) & 1) && g_time() - t0 < TIMEOUT_NS_TCD) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            for (int i = 0; i < nk; ++i) {
                const int s = i % STAGES;
                if (!tc_wait(full + s, (i / STAGES) & 1, abort_s)) {
                    *abort_s = 1;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t a0 = s_addr(smem + s * STG), b0 = a0 + A_BYTES;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    const uint64_t ad = sw128_desc(a0 + k * 32), bd = sw128_desc(b0 + k * 32);
                    const uint32_t acc = (i | k) ? 1u : 0u;
                    asm volatile(
                        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem),
                        "l"(ad), "l"(bd), "r"(idesc), "r"(acc));
                }
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                    s_addr(empty + s))
                             : "memory");
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                s_addr(accf))
                         : "memory");
        }
    } else {
        // partial sums: thread = feature q * 32 + lane; column c < TB is token c's high part, TB + c its low
        // part; the EPW / 4 warps of a lane quarter take 16-column chunks in turn
        const int q = warp & 3, hf = (warp - 2) >> 2, f = q * 32 + lane;
        tcd_preload(pre, e, t0, t1, tb0, n0, N, warp - 2, lane);  // overlaps the MMAs
        const bool ok = tc_wait(accf, 0, abort_s) && !*abort_s;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (ok) {
            for (int c = 16 * hf; c < TB; c += 16 * (EPW / 4)) {
                uint32_t hi[16], lo[16];
                const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c;
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
                    "[%16];"
                    : "=r"(hi[0]), "=r"(hi[1]), "=r"(hi[2]), "=r"(hi[3]), "=r"(hi[4]), "=r"(hi[5]), "=r"(hi[6]),
                      "=r"(hi[7]), "=r"(hi[8]), "=r"(hi[9]), "=r"(hi[10]), "=r"(hi[11]), "=r"(hi[12]), "=r"(hi[13]),
                      "=r"(hi[14]), "=r"(hi[15])
                    : "r"(ta));
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
                    "[%16];"
                    : "=r"(lo[0]), "=r"(lo[1]), "=r"(lo[2]), "=r"(lo[3]), "=r"(lo[4]), "=r"(lo[5]), "=r"(lo[6]),
                      "=r"(lo[7]), "=r"(lo[8]), "=r"(lo[9]), "=r"(lo[10]), "=r"(lo[11]), "=r"(lo[12]), "=r"(lo[13]),
                      "=r"(lo[14]), "=r"(lo[15])
                    : "r"(ta + (uint32_t)TB));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int j = 0; j < 16; ++j) red[(c + j) * BM + f] = __uint_as_float(hi[j]) + __uint_as_float(lo[j]);
            }
        } else if (lane == 0 && q == 0) {
            set_err(err, ERR_TIMEOUT);
        }
    }
    if (threadIdx.x == 0)  // expect the S - 1 peers' slices of this CTA's tokens
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(s_addr(recvb)),
                     "r"((uint32_t)((S - 1) * (t1 - t0) * BM * 4))
                     : "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    cluster_sync_all();  // every CTA's partials are in its shared memory, every receive barrier armed
    if (threadIdx.x == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // partials written by threads -> bulk copy reads
        for (uint32_t q = 0; q < S; ++q) {
            const int a0 = tok(q), a1 = tok(q + 1);
            if (q == r || a1 == a0) continue;
            // my partial of q's tokens -> q's receive slot r
            const uint32_t dst = dsmem_addr(recv + (size_t)r * (a1 - a0) * BM, q);
            const uint32_t bar = dsmem_addr(recvb, q);
            asm volatile(
                "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                "r"(s_addr(red + (size_t)a0 * BM)), "r"((uint32_t)((a1 - a0) * BM * 4)), "r"(bar)
                : "memory");
        }
    }
    if (warp >= 2) {
        const bool got = t1 == t0 || S == 1 || tc_wait(recvb, 0, abort_s);
        if (!got && lane == 0 && warp == 2) set_err(err, ERR_TIMEOUT);
        // this CTA's incoming partials have landed: the peers' copies out of their shared memory are done
        asm volatile("barrier.cluster.arrive;" ::: "memory");
        TcdOut o;
        const size_t orow = (size_t)tb0 * e.ldo;
        o.f32 = e.out ? reinterpret_cast<float*>(e.out) + orow : nullptr;
        o.hi = e.out ? reinterpret_cast<bf16*>(e.out) + orow : nullptr;
        o.lo = e.out_lo ? reinterpret_cast<bf16*>(e.out_lo) + orow : nullptr;
        o.amax = e.amax ? e.amax + tb0 : nullptr;
        o.ldo = e.ldo;
        o.ng = e.nrm_gamma;
        o.ny = e.nrm_y ? e.nrm_y + (size_t)tb0 * 1024 : nullptr;
        o.nylo = e.nrm_ylo ? e.nrm_ylo + (size_t)tb0 * 1024 : nullptr;
        o.nss = e.nrm_ss;
        o.css = e.nrm_scale_ss;
        o.Ttot = e.nrm_T;
        o.tb0 = tb0;
        const int w = warp - 2;
        switch (e.mode) {
            case EPI_QKROPE: tcd_qkrope(e.qk, pre, red, recv, t0, t1, S, r, n0, w, lane, tb0, e.nrm_scale_ss != nullptr);
                break;
            case EPI_STORE_F32: tcd_reduce<EPI_STORE_F32>(o, pre, red, recv, t0, t1, S, r, n0, N, w, lane); break;
            case EPI_ADD_F32: tcd_reduce<EPI_ADD_F32>(o, pre, red, recv, t0, t1, S, r, n0, N, w, lane); break;
            case EPI_SWIGLU: tcd_reduce<EPI_SWIGLU>(o, pre, red, recv, t0, t1, S, r, n0, N, w, lane); break;
            default: tcd_reduce<EPI_LOGITS>(o, pre, red, recv, t0, t1, S, r, n0, N, w, lane); break;
        }
    }
    // exit (and free the SM for the next launch) once every peer has received this CTA's partials,
    // without waiting for the peers' reductions
    if (warp < 2) asm volatile("barrier.cluster.arrive;" ::: "memory");
    asm volatile("barrier.cluster.wait;" ::: "memory");
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tcols));
    }
}

// ---------------------------------------------------------------- bidirectional attention on tcgen05
// Flash attention for the MaskGIT pass (no mask but per-sequence key lengths).
// A CTA takes 64 queries of the two query heads of one KV head: 128 rows
// (rows 0..63 head 2g, 64..127 head 2g+1) of Q, loaded once into shared
// memory in the 128-byte-swizzled K-major layout. Per tile of 128 keys (two
// cache blocks) a producer thread loads K and V [128 keys][128 dims] with TMA
// into a 2-stage ring; the MMA thread computes S = Q K^T into one of two TMEM
// buffers (M = N = K = 128, K-major operands) and, once the softmax warps
// have written P, O += P V into a TMEM accumulator (V read MN-major, as the
// cache stores it). Eight softmax warps, two per row quarter (TMEM lanes),
// each take 64 of a tile's 128 columns: a thread reads its half row into
// registers, the two halves exchange their maxima through shared memory,
// and each writes P = exp2(s - m) as bf16 into its half of one of two
// shared-memory buffers (swizzled, the A operand of P V), keeping its own
// partial row sum. The running max m moves only when a tile's max exceeds it
// by more than 8, and then O (TMEM, each half its 64 columns) and the sums
// are rescaled, so P stays <= 2^8 and the result is exact up to rounding;
// with P double-buffered the softmax of tile j + 1 runs while the tensor
// cores do P V of tile j. Every wait is bounded.
// The precise variant (causal prefill, whose K / V feed every later step)
// carries Q and P as bf16 high + low parts (x = hi + lo to ~2^-17): S = Q_hi
// K^T + Q_lo K^T and O += P_hi V + P_lo V, from fp32 queries. Its tiles fit
// the same 224 KB with one K stage and one (hi + lo) P buffer: the K copy of
// tile j + 1 and its S product overlap the softmax of tile j, which is the
// longer part of a tile.
namespace at {
constexpr int BQ = 64, ROWS = 128, BKV = 128, NT = 320;
constexpr int CHUNK = ROWS * 128;                 // 128 rows x 128 B, 128-byte swizzled
constexpr int TILE = 2 * CHUNK;                   // 128 rows x 128 bf16: two 64-column chunks
template <bool PRECISE>
struct Lay {
    static constexpr int KST = PRECISE ? 1 : 2, VST = 2, NPB = PRECISE ? 1 : 2;  // K, V stages; P buffers
    static constexpr int Q_OFF = 0, QL_OFF = TILE;                               // QL: precise only
    static constexpr int K_OFF = (PRECISE ? 2 : 1) * TILE, V_OFF = K_OFF + KST * TILE, P_OFF = V_OFF + VST * TILE;
    static constexpr int PL_OFF = P_OFF + TILE;                                  // precise only
    static constexpr int BAR_OFF = P_OFF + (PRECISE ? 2 : NPB) * TILE;          // 224 KB of tiles, then barriers
    static constexpr int PM_OFF = BAR_OFF + 256;  // [2 tile parities][2 halves][128 rows] fp32 row maxima
    static constexpr int SMEM = PM_OFF + 2 * 2 * ROWS * 4;  // the tiles start the (1 KB-aligned) dynamic shared memory
};
constexpr int TMEM_COLS = 512;                    // S buffers at 0, 128; O at 256
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(128 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
constexpr uint32_t IDESC_PV = IDESC | (1u << 16);  // B (V) MN-major
// V stage: [cache block i][dims 64c .. 64c+63][64 keys x 128 B]: MN-major atoms of 64 dims x 8 keys,
// 1024 B apart along the keys (stride offset), 8 KB apart along the dims (leading offset)
constexpr uint32_t V_LBO = 8192, V_SBO = 1024;
constexpr unsigned long long TIMEOUT_NS = TC_TIMEOUT_NS;
}  // namespace at
static_assert(at::Lay<false>::SMEM <= 232448 && at::Lay<true>::SMEM <= 232448, "shared memory per CTA");

// Flash attention on tcgen05 for the dense passes: the bidirectional MaskGIT pass (every query sees
// keys < key_len[b]) and the causal prefill (query at position seq_start[b] + s sees keys up to its
// own position, cached keys included).
// grid (ceil(S / 64), 8, B), 320 threads. q [B*S][16][128] bf16 (precise: qf, the same in fp32); pool: K and V tiles [64][128] per
// (block, KV head), [blocks][K, V][8][64][128]; cache block j of sequence b is
// page_table[seq_slot[b] * mbps + j] (j < mbps; an entry below 0 reads as zeros), or b * mbps + j
// without a page table; out [B*S][16][128] bf16 (+ low parts out_lo, value - bf16(value), if given).
struct AttnTcArgs {
    const bf16* q;
    const float* qf;            // precise variant: fp32 queries
    const int32_t* key_len;     // bidirectional: keys per sequence
    const int32_t* seq_start;   // causal: position of query 0 of each sequence (null: 0)
    const int32_t* page_table;  // null: blocks of sequence b at b * mbps
    const int32_t* seq_slot;
    int mbps;
    int causal;
    int S;
    bf16* out;
    bf16* out_lo;
    int* err;
};
template <bool PRECISE>
__global__ void __launch_bounds__(at::NT, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap tmKV, const __grid_constant__ AttnTcArgs A) {
    const int S = A.S;
    bf16* __restrict__ out = A.out;
    int* err = A.err;
    using namespace at;
    using Ly = Lay<PRECISE>;
    constexpr int KST = Ly::KST, VST = Ly::VST, NPB = Ly::NPB;
    extern __shared__ __align__(1024) unsigned char smem[];
    if (s_addr(smem) & 1023u) {  // the swizzled tiles need a 1 KB-aligned base
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) set_err(err, ERR_LAYOUT);
        return;
    }
    uint64_t* k_full = reinterpret_cast<uint64_t*>(smem + Ly::BAR_OFF);  // [KST] K of a tile landed
    uint64_t* k_empty = k_full + 2;        // [KST] S of the tile done (K stage free)
    uint64_t* v_full = k_empty + 2;        // [VST] V of a tile landed
    uint64_t* v_empty = v_full + 2;        // [VST] P V of the tile done (V stage free)
    uint64_t* s_full = v_empty + 2;        // [2] S buffer j & 1 written
    uint64_t* p_full = s_full + 2;         // [2] P buffer j & 1 written (8 softmax-warp arrivals)
    uint64_t* o_done = p_full + 2;         // [2] P V of tile j complete, by j & 1
    uint64_t* fin = o_done + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
    volatile int* abort_s = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* pm = reinterpret_cast<float*>(smem + Ly::PM_OFF);
    const int qt = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            tc_mbar_init(k_full + i, 1);
            tc_mbar_init(k_empty + i, 1);
            tc_mbar_init(v_full + i, 1);
            tc_mbar_init(v_empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc_mbar_init(s_full + i, 1);
            tc_mbar_init(p_full + i, 8);
            tc_mbar_init(o_done + i, 1);
        }
        tc_mbar_init(fin, 1);
        *abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s_addr(tmem_slot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    pdl_wait();  // q and the K / V tiles come from upstream kernels
    pdl_trigger();
    // keys this CTA's queries may see: causal, up to the position of its last query
    const int start = A.causal && A.seq_start ? A.seq_start[b] : 0;
    const int L = A.causal ? start + min(S, (qt + 1) * BQ) : A.key_len[b];
    const int nt = (L + BKV - 1) / BKV;
    const int32_t* pt = A.page_table ? A.page_table + (size_t)A.seq_slot[b] * A.mbps : nullptr;
    // K and V tiles j of one stage: 2 cache blocks x 2 dims chunks of 64 x 64 each
    auto issue_tile = [&](int which, int j) {
        const int st = j % (which ? VST : KST);
        uint64_t* full = which ? v_full : k_full;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(s_addr(full + st)),
                     "r"((uint32_t)(2 * CHUNK))
                     : "memory");
        for (int i = 0; i < 2; ++i) {
            // blocks past the sequence hold masked keys; a block past the table reads as zeros
            const int blk = 2 * j + i;
            const int phys = blk >= A.mbps ? -1 : pt ? pt[blk] : b * A.mbps + blk;
            const int row = ((phys * 2 + which) * NKV + g) * KVB;
            for (int c = 0; c < 2; ++c) {
                // K stage: [dims chunk c][keys 64i ..]; V stage: [cache block i][dims chunk c]
                const int off = which ? i * CHUNK + c * (CHUNK / 2) : c * CHUNK + i * (CHUNK / 2);
                tma_load_2d(smem + (which ? Ly::V_OFF : Ly::K_OFF) + st * TILE + off, &tmKV, c * 64, row, full + st);
            }
        }
    };
    // the first stages are requested by the thread that initialised the barriers, before Q is staged
    const int preK = nt < KST ? nt : KST, preV = nt < VST ? nt : VST;
    if (threadIdx.x == 0) {
        for (int j = 0; j < preK; ++j) issue_tile(0, j);
        for (int j = 0; j < preV; ++j) issue_tile(1, j);
    }
    // Q rows -> shared memory, swizzled (rows past the sequence are zero); all loads first
    {
        constexpr int NQL = (ROWS * 16 + NT - 1) / NT;
        if constexpr (PRECISE) {  // fp32 queries -> high and low bf16 parts
            float4 qv[NQL][2];
#pragma unroll
            for (int k = 0; k < NQL; ++k) {
                const int i = threadIdx.x + k * NT, r = (i >> 4) & (ROWS - 1), pc = i & 15;
                const int sq = qt * BQ + (r & 63), head = 2 * g + (r >> 6);
                qv[k][0] = qv[k][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i < ROWS * 16 && sq < S) {
                    const float4* src = reinterpret_cast<const float4*>(A.qf + (((size_t)b * S + sq) * NQ + head) * HD + pc * 8);
                    qv[k][0] = src[0];
                    qv[k][1] = src[1];
                }
            }
#pragma unroll
            for (int k = 0; k < NQL; ++k) {
                const int i = threadIdx.x + k * NT, r = (i >> 4) & (ROWS - 1), pc = i & 15;
                if (i < ROWS * 16) {
                    const float f[8] = {qv[k][0].x, qv[k][0].y, qv[k][0].z, qv[k][0].w,
                                        qv[k][1].x, qv[k][1].y, qv[k][1].z, qv[k][1].w};
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(f[2 * u], f[2 * u + 1]);
                        const float2 hf = __bfloat1622float2(h2);
                        __nv_bfloat162 l2 = __floats2bfloat162_rn(f[2 * u] - hf.x, f[2 * u + 1] - hf.y);
                        hi[u] = *reinterpret_cast<uint32_t*>(&h2);
                        lo[u] = *reinterpret_cast<uint32_t*>(&l2);
                    }
                    const uint32_t o = (pc >> 3) * CHUNK + sw128_off(r, pc & 7);
                    *reinterpret_cast<uint4*>(smem + Ly::Q_OFF + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(smem + Ly::QL_OFF + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
        } else {
            uint4 qv[NQL];
#pragma unroll
            for (int k = 0; k < NQL; ++k) {
                const int i = threadIdx.x + k * NT, r = (i >> 4) & (ROWS - 1), pc = i & 15;
                const int sq = qt * BQ + (r & 63), head = 2 * g + (r >> 6);
                qv[k] = make_uint4(0u, 0u, 0u, 0u);
                if (i < ROWS * 16 && sq < S)
                    qv[k] = *reinterpret_cast<const uint4*>(A.q + (((size_t)b * S + sq) * NQ + head) * HD + pc * 8);
            }
#pragma unroll
            for (int k = 0; k < NQL; ++k) {
                const int i = threadIdx.x + k * NT, r = (i >> 4) & (ROWS - 1), pc = i & 15;
                if (i < ROWS * 16)
                    *reinterpret_cast<uint4*>(smem + Ly::Q_OFF + (pc >> 3) * CHUNK + sw128_off(r, pc & 7)) = qv[k];
            }
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // Q (generic writes) -> tensor core reads
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane < 2) {  // ---------------- TMA producers: lane 0 K, lane 1 V of each 128-key tile
            const int which = lane, ST = which ? VST : KST;
            uint64_t* full = which ? v_full : k_full;
            uint64_t* empty = which ? v_empty : k_empty;
            int issued = which ? preV : preK;
            for (int j = issued; j < nt; ++j) {
                const int st = j % ST;
                if (!tc_wait(empty + st, ((j / ST) - 1) & 1, abort_s)) {
                    *abort_s = 1;
                    break;
                }
                issue_tile(which, j);
                ++issued;
            }
            if (*abort_s)
                for (int j = issued > ST ? issued - ST : 0; j < issued; ++j) {
                    const unsigned long long t0 = g_time();
                    while (!tc_mbar_try(full + j % ST, (j / ST) & 1) && g_time() - t0 < TIMEOUT_NS) {
                    }
                }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------- MMA issuer
            const uint32_t q0 = s_addr(smem + Ly::Q_OFF), ql0 = s_addr(smem + Ly::QL_OFF);
            auto issue_s = [&](int j) {  // S_j = Q K_j^T into buffer j & 1 (precise: + Q_lo K_j^T)
                const int st = j % KST;
                const uint32_t k0 = s_addr(smem + Ly::K_OFF + st * TILE), d = tmem + (uint32_t)((j & 1) * 128);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (uint32_t)((kk >> 2) * CHUNK + (kk & 3) * 32);
                    at_mma(d, sw128_desc(q0 + off), sw128_desc(k0 + off), IDESC, kk ? 1u : 0u);
                }
                if constexpr (PRECISE) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (uint32_t)((kk >> 2) * CHUNK + (kk & 3) * 32);
                        at_mma(d, sw128_desc(ql0 + off), sw128_desc(k0 + off), IDESC, 1u);
                    }
                }
                at_commit(s_full + (j & 1));
                at_commit(k_empty + st);
            };
            bool ok = nt > 0 && tc_wait(k_full, 0, abort_s);
            if (ok) {
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                issue_s(0);
            }
            for (int j = 0; j < nt && ok; ++j) {
                if (j + 1 < nt) {  // S buffer (j+1) & 1 was read by the softmax of tile j - 1 (p_full waited)
                    if (!tc_wait(k_full + (j + 1) % KST, ((j + 1) / KST) & 1, abort_s)) { ok = false; break; }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    issue_s(j + 1);
                }
                if (!tc_wait(p_full + (j & 1), (j >> 1) & 1, abort_s)) { ok = false; break; }
                if (!tc_wait(v_full + j % VST, (j / VST) & 1, abort_s)) { ok = false; break; }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const int st = j % VST;
                const uint32_t p0 = s_addr(smem + Ly::P_OFF + (j % NPB) * TILE), v0 = s_addr(smem + Ly::V_OFF + st * TILE);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {  // 16 keys per step: P chunk kk >> 2, V block kk >> 2, 8-key groups 2 (kk & 3)
                    const uint64_t ad = sw128_desc(p0 + (uint32_t)((kk >> 2) * CHUNK + (kk & 3) * 32));
                    const uint64_t bd = sw128_desc_mn(v0 + (uint32_t)((kk >> 2) * CHUNK + (kk & 3) * 2048), V_LBO, V_SBO);
                    at_mma(tmem + 256, ad, bd, IDESC_PV, (j | kk) ? 1u : 0u);
                }
                if constexpr (PRECISE) {
                    const uint32_t pl0 = s_addr(smem + Ly::PL_OFF);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = sw128_desc(pl0 + (uint32_t)((kk >> 2) * CHUNK + (kk & 3) * 32));
                        const uint64_t bd = sw128_desc_mn(v0 + (uint32_t)((kk >> 2) * CHUNK + (kk & 3) * 2048), V_LBO, V_SBO);
                        at_mma(tmem + 256, ad, bd, IDESC_PV, 1u);
                    }
                }
                at_commit(o_done + (j & 1));
                at_commit(v_empty + st);
            }
            if (!ok) *abort_s = 1;
            at_commit(fin);
            const unsigned long long t0 = g_time();
            while (!tc_mbar_try(fin, 0) && g_time() - t0 < TIMEOUT_NS) {
            }
        }
    } else {
        // ---------------- softmax + epilogue: thread = row (TMEM lane), half = 64 of the 128 columns
        const int qd = warp & 3, r = qd * 32 + lane, half = (warp - 2) >> 2;
        const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
        const uint32_t cbase = (uint32_t)(half * 64);
        const float sc = rsqrtf((float)HD) * 1.4426950408889634f;
        float m_used = -INFINITY, l = 0.f;
        // keys this row sees: causal, up to its own position
        const int row_lim = A.causal ? start + qt * BQ + (r & 63) + 1 : L;
        // the two warps of a row quarter meet at a named barrier once per tile and twice after the
        // loop; after a failed wait a warp keeps meeting them (skipping the work), so neither can hang
        bool ok = true;
        auto wait_u = [&](uint64_t* bar, uint32_t par) {  // warp-uniform bounded wait
            if (ok) ok = __all_sync(0xffffffffu, tc_wait(bar, par, abort_s));
            if (!ok && lane == 0) *abort_s = 1;
        };
        for (int j = 0; j < nt; ++j) {
            uint32_t v[64];
            float mh = -INFINITY;
            const int kvalid = row_lim - j * BKV - half * 64;  // keys of this half the row may see
            wait_u(s_full + (j & 1), (j >> 1) & 1);
            if (ok) {
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t sb = lane_base + (uint32_t)((j & 1) * 128) + cbase;
                tm_ld32_nw(sb, v);
                tm_ld32_nw(sb + 32, v + 32);
                tm_wait_ld();
                if (kvalid < 64) {
#pragma unroll
                    for (int x = 0; x < 64; ++x)
                        if (x >= kvalid) v[x] = 0xFF800000u;  // -inf
                }
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int x = 0; x < 64; ++x) m4[x & 3] = fmaxf(m4[x & 3], __uint_as_float(v[x]));
                mh = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            }
            // row max over both halves (a half may be fully masked: -inf)
            float* pmj = pm + (j & 1) * 2 * ROWS;
            pmj[half * ROWS + r] = mh;
            asm volatile("bar.sync %0, 64;" ::"r"(1 + qd) : "memory");
            const float mx = fmaxf(pmj[r], pmj[ROWS + r]) * sc;
            if (!ok) continue;
            float alpha = 1.f;
            const bool move = mx > m_used + 8.f;
            if (move) {
                alpha = (m_used == -INFINITY) ? 0.f : at_ex2(m_used - mx);
                m_used = mx;
            }
            // the P buffer of tile j was read by P V of tile j - NPB
            if (j >= NPB) wait_u(o_done + ((j - NPB) & 1), ((j - NPB) >> 1) & 1);
            if (ok && move && j >= 1) {  // rescale this half of O once P V of tile j - 1 is in it
                wait_u(o_done + ((j - 1) & 1), ((j - 1) >> 1) & 1);
                if (ok) {
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    for (int ch = 0; ch < 2; ++ch) {
                        uint32_t o[32];
                        tm_ld32_nw(lane_base + 256 + cbase + ch * 32, o);
                        tm_wait_ld();
#pragma unroll
                        for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
                        tm_st32(lane_base + 256 + cbase + ch * 32, o);
                    }
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                }
            }
            if (!ok) continue;
            l *= alpha;
            float l4[4] = {0.f, 0.f, 0.f, 0.f};
            // this half's keys are key chunk `half` of the P buffer (64 keys = one 128-byte row)
            unsigned char* prow = smem + Ly::P_OFF + (j % NPB) * TILE + half * CHUNK;
            unsigned char* plrow = smem + Ly::PL_OFF + half * CHUNK;  // precise only
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                uint32_t pk[16], pl[16];
#pragma unroll
                for (int x = 0; x < 32; x += 2) {
                    const float p0 = at_ex2(fmaf(__uint_as_float(v[ch * 32 + x]), sc, -m_used));
                    const float p1 = at_ex2(fmaf(__uint_as_float(v[ch * 32 + x + 1]), sc, -m_used));
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                    pk[x >> 1] = *reinterpret_cast<uint32_t*>(&h2);
                    if constexpr (PRECISE) {  // the row sum takes the weights P V applies (hi + lo)
                        const float2 pr = __bfloat1622float2(h2);
                        __nv_bfloat162 l2 = __floats2bfloat162_rn(p0 - pr.x, p1 - pr.y);
                        pl[x >> 1] = *reinterpret_cast<uint32_t*>(&l2);
                        const float2 lr = __bfloat1622float2(l2);
                        l4[(x >> 1) & 3] += (pr.x + lr.x) + (pr.y + lr.y);
                    } else {
                        l4[(x >> 1) & 3] += p0 + p1;
                    }
                }
#pragma unroll
                for (int pp = 0; pp < 4; ++pp) {
                    *reinterpret_cast<uint4*>(prow + sw128_off(r, ch * 4 + pp)) =
                        make_uint4(pk[4 * pp], pk[4 * pp + 1], pk[4 * pp + 2], pk[4 * pp + 3]);
                    if constexpr (PRECISE)
                        *reinterpret_cast<uint4*>(plrow + sw128_off(r, ch * 4 + pp)) =
                            make_uint4(pl[4 * pp], pl[4 * pp + 1], pl[4 * pp + 2], pl[4 * pp + 3]);
                }
            }
            l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P (generic writes) -> tensor core reads
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(s_addr(p_full + (j & 1))) : "memory");
        }
        // row sum over both halves (through the max buffer of parity nt & 1, free once both passed tile nt - 1)
        float* ls = pm + (nt & 1) * 2 * ROWS;
        asm volatile("bar.sync %0, 64;" ::"r"(1 + qd) : "memory");  // both halves done with every max buffer read
        ls[half * ROWS + r] = ok ? l : 0.f;
        asm volatile("bar.sync %0, 64;" ::"r"(1 + qd) : "memory");
        l = ls[r] + ls[ROWS + r];
        if (nt > 0) wait_u(o_done + ((nt - 1) & 1), ((nt - 1) >> 1) & 1);
        if (ok && nt > 0) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int sq = qt * BQ + (r & 63), head = 2 * g + (r >> 6);
            const float inv = l > 0.f ? 1.f / l : 0.f;
            for (int ch = 0; ch < 2; ++ch) {
                uint32_t o[32];
                tm_ld32_nw(lane_base + 256 + cbase + ch * 32, o);
                tm_wait_ld();
                if (sq < S) {
                    const size_t off = (((size_t)b * S + sq) * NQ + head) * HD + cbase + ch * 32;
#pragma unroll
                    for (int x = 0; x < 32; x += 8) {
                        uint32_t w[4], wl[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float f0 = __uint_as_float(o[x + 2 * u]) * inv, f1 = __uint_as_float(o[x + 2 * u + 1]) * inv;
                            __nv_bfloat162 a2 = __floats2bfloat162_rn(f0, f1);
                            w[u] = *reinterpret_cast<uint32_t*>(&a2);
                            const float2 hf = __bfloat1622float2(a2);
                            __nv_bfloat162 l2 = __floats2bfloat162_rn(f0 - hf.x, f1 - hf.y);
                            wl[u] = *reinterpret_cast<uint32_t*>(&l2);
                        }
                        *reinterpret_cast<uint4*>(out + off + x) = make_uint4(w[0], w[1], w[2], w[3]);
                        if (A.out_lo) *reinterpret_cast<uint4*>(A.out_lo + off + x) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                    }
                }
            }
        } else if (lane == 0) {
            set_err(err, ERR_TIMEOUT);
            *abort_s = 1;
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
    }
}

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D bf16 tensor [rows][K] (K contiguous), box [box_rows][64], 128-byte swizzle.
static bool encode_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)tc::BK, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoded maps are cached by (base, rows, K, box rows): weights never move and
// the engine's activation buffers are fixed, so a decode step re-encodes
// nothing. The cache is per process and guarded by a mutex; a full cache
// is cleared (maps are cheap to re-encode).
bool tc_make_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows) {
    struct Key {
        const void* base;
        int rows, K, box;
        bool operator==(const Key& o) const { return base == o.base && rows == o.rows && K == o.K && box == o.box; }
    };
    struct KeyHash {
        size_t operator()(const Key& k) const {
            size_t h = std::hash<const void*>()(k.base);
            h ^= (size_t)k.rows * 0x9E3779B97F4A7C15ull + (size_t)k.K * 0xC2B2AE3D27D4EB4Full + (size_t)k.box;
            return h;
        }
    };
    static std::mutex mu;
    static std::unordered_map<Key, CUtensorMap, KeyHash> cache;
    const Key key{base, rows, K, box_rows};
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *m = it->second;
            return true;
        }
    }
    if (!encode_map(m, base, rows, K, box_rows)) return false;
    std::lock_guard<std::mutex> g(mu);
    if (cache.size() > 4096) cache.clear();
    cache.emplace(key, *m);
    return true;
}

bool gemm_tc_available() { return encode_fn() != nullptr; }

// fp32 (or bf16) output [rows][ld] (first `cols` columns), box of 64-byte rows (16 fp32 / 32 bf16) x
// 32 rows, 64-byte swizzle: the dense GEMM's bulk-store epilogue. Cached like the operand maps.
static bool make_out_map(CUtensorMap* m, const void* base, int rows, int cols, int ld, bool bf16_out = false) {
    struct Key {
        const void* base;
        int rows, cols, ld, bf;
        bool operator==(const Key& o) const {
            return base == o.base && rows == o.rows && cols == o.cols && ld == o.ld && bf == o.bf;
        }
    };
    struct KeyHash {
        size_t operator()(const Key& k) const {
            return std::hash<const void*>()(k.base) ^ ((size_t)k.rows * 0x9E3779B97F4A7C15ull + (size_t)k.cols * 131 + (size_t)k.ld);
        }
    };
    static std::mutex mu;
    static std::unordered_map<Key, CUtensorMap, KeyHash> cache;
    const Key key{base, rows, cols, ld, bf16_out ? 1 : 0};
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *m = it->second;
            return true;
        }
    }
    auto fn = encode_fn();
    const int esz = bf16_out ? 2 : 4;
    if (!fn || (ld * esz) % 16 != 0 || cols > ld || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * esz};
    const cuuint32_t box[2] = {(cuuint32_t)(64 / esz), 32};  // 64-byte rows of the box
    const cuuint32_t es[2] = {1, 1};
    if (fn(m, bf16_out ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base),
           dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> g(mu);
    if (cache.size() > 4096) cache.clear();
    cache.emplace(key, *m);
    return true;
}

// 4-D bf16 tensor [parts][B][T][C] (C contiguous), box box_c (64 or 32) channels x 128 rows of one
// (part, item), 128- or 64-byte swizzle (rows of box_c x 2 bytes); rows and channels outside the
// tensor read as zeros. Not cached.
bool tc_make_map_rows(CUtensorMap* m, const void* base, int C, int T, int B, int parts, int box_c) {
    auto fn = encode_fn();
    if (!fn || C % 8 != 0 || C <= 0 || T <= 0 || B <= 0 || parts <= 0 || (box_c != 64 && box_c != 32)) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)C, (cuuint64_t)T, (cuuint64_t)B, (cuuint64_t)parts};
    const cuuint64_t strides[3] = {(cuuint64_t)C * 2, (cuuint64_t)T * C * 2, (cuuint64_t)B * T * C * 2};
    const cuuint32_t box[4] = {(cuuint32_t)box_c, 128, 1, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, box_c == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 tensor [rows][K] (K contiguous), box [box_rows][box_k] with box_k 64 (128-byte swizzle)
// or 32 (64-byte swizzle). Not cached.
bool tc_make_map_k(CUtensorMap* m, const void* base, int rows, int K, int box_rows, int box_k) {
    auto fn = encode_fn();
    if (!fn || (box_k != 64 && box_k != 32) || K % 8 != 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)box_k, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, box_k == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool PRECISE>
static int launch_attn_tc(const CUtensorMap& mkv, const AttnTcArgs& A, int B, cudaStream_t st) {
    constexpr int SMEM = at::Lay<PRECISE>::SMEM;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_attn_tc<PRECISE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        attr = true;
    }
    dim3 grid((A.S + at::BQ - 1) / at::BQ, NKV, B);
    return launch_pdl(k_attn_tc<PRECISE>, grid, at::NT, SMEM, st, mkv, A) == cudaSuccess ? 1 : 0;
}

// Bidirectional attention of the MaskGIT pass on tcgen05 (no page table: sequence b's blocks at
// b * bps). Returns launches (0 = not available).
int launch_attn_bidir_tc(const bf16* q, const bf16* pool, size_t pool_blocks, int bps, const int32_t* key_len, int B,
                         int S, bf16* out, int* err, cudaStream_t st) {
    if (B <= 0 || S <= 0 || !gemm_tc_available()) return 0;
    const size_t rows = pool_blocks * 2 * NKV * KVB;  // [rows][128]: K and V tiles of every (block, KV head)
    if (rows > (size_t)INT32_MAX) return 0;
    CUtensorMap mkv;
    if (!tc_make_map(&mkv, pool, (int)rows, HD, KVB)) return 0;
    AttnTcArgs A{q, nullptr, key_len, nullptr, nullptr, nullptr, bps, 0, S, out, nullptr, err};
    return launch_attn_tc<false>(mkv, A, B, st);
}

// Causal prefill attention on tcgen05 over the paged cache (one layer's pool of pool_blocks
// blocks): query s of sequence b sits at position seq_start[b] + s. With fp32 queries qf the
// precise variant runs (Q and P as high + low parts), else bf16 q. Returns launches (0 = not available).
int launch_attn_causal_tc(const bf16* q, const float* qf, KVView kv, size_t pool_blocks, const int32_t* seq_start,
                          int B, int S, bf16* out, bf16* out_lo, int* err, cudaStream_t st) {
    if (B <= 0 || S <= 0 || !gemm_tc_available()) return 0;
    const size_t rows = pool_blocks * 2 * NKV * KVB;
    if (rows > (size_t)INT32_MAX) return 0;
    CUtensorMap mkv;
    if (!tc_make_map(&mkv, kv.pool, (int)rows, HD, KVB)) return 0;
    AttnTcArgs A{q, qf, nullptr, seq_start, kv.page_table, kv.seq_slot, kv.mbps, 1, S, out, out_lo, err};
    return qf ? launch_attn_tc<true>(mkv, A, B, st) : launch_attn_tc<false>(mkv, A, B, st);
}

namespace {
constexpr int TCD_CAND[8] = {1, 2, 3, 4, 6, 8, 12, 16};  // cluster sizes (split-K ways)
// Clusters of each candidate size that fit at once (1 CTA per SM), found once per process.
const int* tcd_fit() {
    static const std::array<int, 8> fit = [] {
        std::array<int, 8> f{};
        cudaFuncSetAttribute(k_gemm_tcd, cudaFuncAttributeMaxDynamicSharedMemorySize, tcd::SMEM);
        const bool nonport = cudaFuncSetAttribute(k_gemm_tcd, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
        for (int i = 0; i < 8; ++i) {
            if (TCD_CAND[i] > 8 && !nonport) continue;
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(TCD_CAND[i]);
            q.blockDim = dim3(tcd::NT);
            q.dynamicSmemBytes = tcd::SMEM;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = TCD_CAND[i];
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            q.attrs = qa;
            q.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, k_gemm_tcd, &q) == cudaSuccess) f[i] = n;
        }
        cudaGetLastError();
        return f;
    }();
    return fit.data();
}
// The most CTAs with which `clusters` clusters (one per weight tile and token block) all run in
// one wave, and the cluster size S that gives it; 0 if no size fits.
int tcd_pick(int clusters, int KT, int& S) {
    const int* fit = tcd_fit();
    int best = 0;
    S = 1;
    for (int i = 0; i < 8; ++i)
        if (TCD_CAND[i] <= KT && clusters <= fit[i] && clusters * TCD_CAND[i] > best) {
            best = clusters * TCD_CAND[i];
            S = TCD_CAND[i];
        }
    return best;
}
}  // namespace

bool gemm_tcd_takes(int T, int N, int K) {
    if (T <= 0 || T > tcd::MAXBLK * tcd::MAXTB || N <= 0 || K <= 0 || K % tcd::BK != 0) return false;
    const int blocks = (T + tcd::MAXTB - 1) / tcd::MAXTB;
    if (blocks <= 2) return true;  // one launch over both blocks, or one launch per block
    int S = 1;
    return tcd_pick(((N + tcd::BM - 1) / tcd::BM) * blocks, K / tcd::BK, S) > 0;  // more blocks: one wave, one launch
}

int launch_gemm_tcd(const bf16* X, const bf16* X_lo, const bf16* W, int T, int N, int K, const Epi& e, int* err,
                    cudaStream_t st) {
    if (!X_lo || !gemm_tcd_takes(T, N, K)) return 0;
    if (e.mode != EPI_STORE_F32 && e.mode != EPI_ADD_F32 && e.mode != EPI_SWIGLU && e.mode != EPI_LOGITS &&
        e.mode != EPI_QKROPE)
        return 0;
    if (e.mode == EPI_QKROPE && N != QKV) return 0;
    const int blocks = (T + tcd::MAXTB - 1) / tcd::MAXTB;  // token blocks of up to 128
    const int TB = blocks > 1 ? tcd::MAXTB : (T + 15) / 16 * 16;
    CUtensorMap mw, mh, ml;
    if (!tc_make_map(&mw, W, N, K, tcd::BM) || !tc_make_map(&mh, X, T, K, TB) || !tc_make_map(&ml, X_lo, T, K, TB)) return 0;
    const int tiles = (N + tcd::BM - 1) / tcd::BM, KT = K / tcd::BK;
    int S1 = 1, S2 = 1;
    const int one = tcd_pick(tiles, KT, S1);
    // every token block in one launch when that keeps as many CTAs busy as a launch per block (more
    // than two blocks: whenever it fits one wave, which gemm_tcd_takes checked)
    const bool joint = blocks > 2 || (blocks > 1 && tcd_pick(tiles * blocks, KT, S2) >= one);
    if (blocks > 2) tcd_pick(tiles * blocks, KT, S2);
    auto go = [&](int S, int rows, int tb_base) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(tiles * S, rows);
        cfg.blockDim = dim3(tcd::NT);
        cfg.dynamicSmemBytes = tcd::STAGES * (tcd::A_BYTES + 2 * TB * tcd::BK * 2) + 1024 + 256;
        cfg.stream = st;
        cudaLaunchAttribute at[2];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = S;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, k_gemm_tcd, mw, mh, ml, T, TB, tb_base, N, K, e, err) == cudaSuccess;
    };
    if (joint) return go(S2, blocks, 0) ? 1 : 0;
    int n = 0;
    for (int b = 0; b < blocks; ++b) {
        if (!go(S1, 1, b * tcd::MAXTB)) return n;
        ++n;
    }
    return n;
}


// Y = X W^T on tcgen05. Requires K % 64 == 0, 16-byte aligned X and W rows.
// Returns the number of kernels launched (0 if the shape is not supported).
int launch_gemm_tc(const bf16* X, const bf16* W, int T, int N, int K, const Epi& e, int* err, cudaStream_t st,
                   const bf16* X_lo) {
    if (T <= 0 || N <= 0 || K % tc::BK != 0) return 0;
    CUtensorMap ma, mal, mb, mo, mol;
    if (!tc_make_map(&ma, X, T, K, tc::BM) || !tc_make_map(&mb, W, N, K, tc::BN)) return 0;
    if (X_lo && !tc_make_map(&mal, X_lo, T, K, tc::BM)) return 0;
    if (!X_lo) mal = ma;
    mo = mol = ma;  // unused unless set below
    if (e.mode == EPI_STORE_F32 || e.mode == EPI_ADD_F32) {
        if (!make_out_map(&mo, e.out, T, N, e.ldo)) return 0;
    } else if (e.mode == EPI_STORE_BF16) {
        if (!make_out_map(&mo, e.out, T, N, e.ldo, true)) return 0;
    } else if (e.mode == EPI_SWIGLU) {
        if (N % 2 != 0 || !make_out_map(&mo, e.out, T, N / 2, e.ldo, true)) return 0;
        if (e.out_lo && !make_out_map(&mol, e.out_lo, T, N / 2, e.ldo, true)) return 0;
    }
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::SMEM);
        attr = true;
    }
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    }
    const int tiles = ((N + tc::BN - 1) / tc::BN) * ((T + tc::BM - 1) / tc::BM);
    launch_pdl(k_gemm_tc, std::min(tiles, sms), tc::NT, tc::SMEM, st, ma, mal, mb, mo, mol, X_lo ? 1 : 0, T, N, K, e,
               err);
    return 1;
}

}  // namespace ttsbb
