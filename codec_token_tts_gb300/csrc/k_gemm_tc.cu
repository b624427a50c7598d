// Dense Y = X W^T on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// One CTA computes a 128-token x 256-feature tile: a producer thread loads
// 128-byte-swizzled K-slices of X (128 x 64) and W (256 x 64) with TMA into a
// 4-stage shared-memory ring; one thread issues tcgen05.mma (M=128, N=256,
// K=16, bf16 in, fp32 accumulate) into a TMEM accumulator and commits each
// stage back to the producer through an mbarrier; four epilogue warps read
// the accumulator with tcgen05.ld (each warp owns its 32-lane quarter of
// TMEM = 32 token rows) and apply the same fused epilogues as the other
// linear kernels (fp32 store, residual add, SwiGLU over interleaved gate/up
// columns, logits + argmax, permuted audio-head logits).
//
// Every mbarrier wait is bounded; on timeout the CTA raises the error word,
// stops issuing work, waits (bounded) for its copies in flight, frees TMEM and
// returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace ttsbb {

namespace tc {
constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + 256;
constexpr int TMEM_COLS = 256;
constexpr int NT = 192;  // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2-5 epilogue
constexpr unsigned long long TIMEOUT_NS = 1000000000ull;
// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A bf16 (7-9 = 1),
// B bf16 (10-12 = 1), both K-major (15, 16 = 0), N >> 3 at 17-22, M >> 4 at 24-28.
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);
}  // namespace tc

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
            if (g_time() - t0 > tc::TIMEOUT_NS) return false;
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

__global__ void __launch_bounds__(tc::NT, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int T, int N, int K,
              Epi e, int* err) {
    using namespace tc;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char* sA = smem;
    unsigned char* sB = smem + STAGES * A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* accf = empty + STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
    volatile int* abort_s = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int KT = K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc_mbar_init(full + s, 1);
            tc_mbar_init(empty + s, 1);
        }
        tc_mbar_init(accf, 1);
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

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int kt = 0; kt < KT; ++kt) {
                const int s = kt % STAGES;
                if (kt >= STAGES && !tc_wait(empty + s, ((kt / STAGES) - 1) & 1, abort_s)) {
                    *abort_s = 1;
                    break;
                }
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(s_addr(full + s)),
                             "r"(STAGE_BYTES)
                             : "memory");
                tma_load_2d(sA + s * A_BYTES, &tmA, kt * BK, m0, full + s);
                tma_load_2d(sB + s * B_BYTES, &tmB, kt * BK, n0, full + s);
                ++issued;
            }
            if (*abort_s) {  // let every issued copy land before the CTA can exit
                for (int kt = 0; kt < issued; ++kt) {
                    const unsigned long long t0 = g_time();
                    while (!tc_mbar_try(full + kt % STAGES, (kt / STAGES) & 1) && g_time() - t0 < TIMEOUT_NS) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            bool ok = true;
            for (int kt = 0; kt < KT && ok; ++kt) {
                const int s = kt % STAGES;
                if (!tc_wait(full + s, (kt / STAGES) & 1, abort_s)) {
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
                        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem),
                        "l"(ad), "l"(bd), "r"(IDESC), "r"(acc));
                }
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                    s_addr(empty + s))
                             : "memory");
            }
            // accumulator complete (or abandoned): wake the epilogue either way
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                s_addr(accf))
                         : "memory");
        }
    } else {
        // ---------------- epilogue: warp w reads TMEM lanes 32 * (w % 4) ..
        const int q = warp & 3;
        const bool ok = tc_wait(accf, 0, abort_s) && !*abort_s;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const int t = m0 + q * 32 + lane;
        unsigned long long best = 0ull;
        if (ok) {
            for (int c = 0; c < BN; c += 16) {
                uint32_t r[16];
                const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c;
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
        } else if (lane == 0 && q == 0) {
            set_err(err, ERR_TIMEOUT);
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
static bool make_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows) {
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

bool gemm_tc_available() { return encode_fn() != nullptr; }

// Y = X W^T on tcgen05. Requires K % 64 == 0, 16-byte aligned X and W rows.
// Returns the number of kernels launched (0 if the shape is not supported).
int launch_gemm_tc(const bf16* X, const bf16* W, int T, int N, int K, const Epi& e, int* err, cudaStream_t st) {
    if (T <= 0 || N <= 0 || K % tc::BK != 0) return 0;
    CUtensorMap ma, mb;
    if (!make_map(&ma, X, T, K, tc::BM) || !make_map(&mb, W, N, K, tc::BN)) return 0;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::SMEM);
        attr = true;
    }
    dim3 grid((N + tc::BN - 1) / tc::BN, (T + tc::BM - 1) / tc::BM);
    k_gemm_tc<<<grid, tc::NT, tc::SMEM, st>>>(ma, mb, T, N, K, e, err);
    return 1;
}

}  // namespace ttsbb
