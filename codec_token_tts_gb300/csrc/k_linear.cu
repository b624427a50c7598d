// Linear layers of the backbone step: Y = X W^T (W in PyTorch (out, in) layout)
// with fused epilogues (residual add, SwiGLU over interleaved gate/up rows,
// logits + argmax, permuted audio-head logits).
//   * k_gemv: T <= 8 token rows, weight streaming with 128-bit loads (HBM-bound
//     decode at small batch).
//   * k_gemm_mma: any T, bf16 tensor cores through mma.sync with a cp.async
//     pipeline.
#include "common.cuh"

namespace ttsbb {

__device__ __forceinline__ float silu(float x) { return x / (1.f + __expf(-x)); }

// Store one accumulator element under the single-element epilogues.
__device__ __forceinline__ void epi_one(const Epi& e, int t, int n, float v) {
    switch (e.mode) {
        case EPI_STORE_F32:
            reinterpret_cast<float*>(e.out)[(size_t)t * e.ldo + n] = v;
            break;
        case EPI_STORE_BF16:
            reinterpret_cast<bf16*>(e.out)[(size_t)t * e.ldo + n] = f2bf(v);
            break;
        case EPI_ADD_F32:
            reinterpret_cast<float*>(e.out)[(size_t)t * e.ldo + n] += v;
            break;
        case EPI_LOGITS:
            if (e.out) reinterpret_cast<float*>(e.out)[(size_t)t * e.ldo + n] = v;
            break;
        case EPI_LOGITS_PERM: {
            const int b = t / e.perm_rows, s = t % e.perm_rows;
            const int k = n / e.perm_vocab, v2 = n % e.perm_vocab;
            reinterpret_cast<float*>(e.out)[(((size_t)b * e.perm_groups + k) * e.perm_rows + s) * e.perm_vocab + v2] = v;
            break;
        }
        default:
            break;
    }
}

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int m) {
    uint32_t lo = (uint32_t)v, hi = (uint32_t)(v >> 32);
    lo = __shfl_xor_sync(0xffffffffu, lo, m);
    hi = __shfl_xor_sync(0xffffffffu, hi, m);
    return ((unsigned long long)hi << 32) | lo;
}
__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}

// ---------------------------------------------------------------- GEMV (T <= 8)
// 8 warps; each warp owns ROWS consecutive output rows (features). Lane l
// streams 16-byte chunks l, l+32, ... of each weight row; X sits in shared
// memory. ROWS = 2 keeps a gate/up pair in one warp for the SwiGLU epilogue.
template <int T, int ROWS>
__global__ void __launch_bounds__(256) k_gemv(const bf16* __restrict__ X, const bf16* __restrict__ X_lo,
                                              const bf16* __restrict__ W, int N, int K, Epi e) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    bf16* xs = reinterpret_cast<bf16*>(smem_raw);
    bf16* xl = xs + (size_t)T * K;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // stage X [T][K] (and its low parts)
    const int nchunk = T * K / 8;
    for (int i = tid; i < nchunk; i += 256) {
        reinterpret_cast<uint4*>(xs)[i] = reinterpret_cast<const uint4*>(X)[i];
        if (X_lo) reinterpret_cast<uint4*>(xl)[i] = reinterpret_cast<const uint4*>(X_lo)[i];
    }
    __syncthreads();

    const int row0 = (blockIdx.x * 8 + warp) * ROWS;
    if (row0 >= N) return;
    float acc[ROWS][T];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int t = 0; t < T; ++t) acc[r][t] = 0.f;

    const int kchunks = K / 256;  // 256 elements per warp pass
    constexpr int U = 4;
    for (int c0 = 0; c0 < kchunks; c0 += U) {
        uint4 w[ROWS][U];
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u;
                if (c < kchunks && row0 + r < N)
                    w[r][u] = ldg_nc_v4(W + (size_t)(row0 + r) * K + c * 256 + lane * 8);
                else
                    w[r][u] = make_uint4(0, 0, 0, 0);
            }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + u;
            if (c >= kchunks) break;
#pragma unroll
            for (int t = 0; t < T; ++t) {
                float xf[8];
                unpack8(reinterpret_cast<const uint4*>(xs + (size_t)t * K + c * 256)[lane], xf);
                if (X_lo) {
                    float lf[8];
                    unpack8(reinterpret_cast<const uint4*>(xl + (size_t)t * K + c * 256)[lane], lf);
#pragma unroll
                    for (int j = 0; j < 8; ++j) xf[j] += lf[j];
                }
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    float wf[8];
                    unpack8(w[r][u], wf);
                    float a = acc[r][t];
#pragma unroll
                    for (int j = 0; j < 8; ++j) a = fmaf(wf[j], xf[j], a);
                    acc[r][t] = a;
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int t = 0; t < T; ++t) acc[r][t] = warp_sum(acc[r][t]);

    if (e.mode == EPI_SWIGLU) {
        // rows (2i, 2i+1) = (gate_i, up_i)
        if (lane < T) {
#pragma unroll
            for (int t = 0; t < T; ++t)
                if (t == lane) {
#pragma unroll
                    for (int r = 0; r + 1 < ROWS; r += 2) {
                        const float g = acc[r][t], u = acc[r + 1][t];
                        const float mv = silu(g) * u;
                        reinterpret_cast<bf16*>(e.out)[(size_t)t * e.ldo + (row0 + r) / 2] = f2bf(mv);
                        if (e.out_lo) reinterpret_cast<bf16*>(e.out_lo)[(size_t)t * e.ldo + (row0 + r) / 2] = f2bf_lo(mv);
                    }
                }
        }
        return;
    }
    if (lane < T) {
#pragma unroll
        for (int t = 0; t < T; ++t)
            if (t == lane) {
                unsigned long long best = 0ull;
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    if (row0 + r >= N) continue;
                    epi_one(e, t, row0 + r, acc[r][t]);
                    if (e.mode == EPI_LOGITS) best = umax64(best, pack_argmax(acc[r][t], row0 + r));
                }
                if (e.mode == EPI_LOGITS && e.amax) atomicMax(e.amax + t, best);
            }
    }
}

template <int T>
static void gemv_t(const bf16* X, const bf16* X_lo, const bf16* W, int N, int K, const Epi& e, cudaStream_t st) {
    const size_t smem = (size_t)(X_lo ? 2 : 1) * T * K * sizeof(bf16);
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(k_gemv<T, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * 8 * 3072 * 2);
        attr_set = true;
    }
    const int rows_per_cta = 16;
    k_gemv<T, 2><<<(N + rows_per_cta - 1) / rows_per_cta, 256, smem, st>>>(X, X_lo, W, N, K, e);
}

int launch_gemv(const bf16* X, const bf16* W, int T, int N, int K, const Epi& e, cudaStream_t st, const bf16* X_lo) {
    switch (T) {
        case 1: gemv_t<1>(X, X_lo, W, N, K, e, st); break;
        case 2: gemv_t<2>(X, X_lo, W, N, K, e, st); break;
        case 3: gemv_t<3>(X, X_lo, W, N, K, e, st); break;
        case 4: gemv_t<4>(X, X_lo, W, N, K, e, st); break;
        case 5: gemv_t<5>(X, X_lo, W, N, K, e, st); break;
        case 6: gemv_t<6>(X, X_lo, W, N, K, e, st); break;
        case 7: gemv_t<7>(X, X_lo, W, N, K, e, st); break;
        case 8: gemv_t<8>(X, X_lo, W, N, K, e, st); break;
        default: return 0;
    }
    return 1;
}

// ---------------------------------------------------------------- GEMM (mma.sync)
// Tile 128 tokens x 128 features x 32, 8 warps (4 along tokens x 2 along
// features, 32x64 each), 4-stage cp.async pipeline, padded shared rows (80 B)
// so ldmatrix is conflict-free.
namespace gm {
constexpr int BM = 128, BN = 128, BK = 32, LDS = BK + 8, STAGES = 4;
constexpr int TILE_A = BM * LDS, TILE_B = BN * LDS;
constexpr int SMEM = STAGES * (TILE_A + TILE_B) * 2;
constexpr int SMEM_SPLIT = STAGES * (2 * TILE_A + TILE_B) * 2;
}  // namespace gm

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool pred) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    const int n = pred ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t* r, const void* p) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(s));
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, const uint32_t* b) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// SPLIT: the activations come as bf16 high + low parts; a second MMA per
// k-step adds the low part (weights are read once, so this is free when the
// GEMM streams weights at small T).
template <bool SPLIT>
__global__ void __launch_bounds__(256) k_gemm_mma(const bf16* __restrict__ X, const bf16* __restrict__ X_lo,
                                                  const bf16* __restrict__ W, int T, int N, int K, Epi e) {
    using namespace gm;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    bf16* sA = reinterpret_cast<bf16*>(smem_raw);
    bf16* sB = sA + STAGES * TILE_A;
    bf16* sL = sB + STAGES * TILE_B;  // low parts (SPLIT only)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 1, wn = warp & 1;
    const int n0 = blockIdx.x * BN, t0 = blockIdx.y * BM;
    const int ktiles = K / BK;

    auto load_stage = [&](int stage, int kt) {
        const int k0 = kt * BK;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int c = tid + i * 256;  // 512 chunks: row = c / 4, col = (c % 4) * 8
            const int r = c >> 2, col = (c & 3) * 8;
            const int tr = t0 + r, nr = n0 + r;
            cp_async16(sA + stage * TILE_A + r * LDS + col, X + (size_t)min(tr, T - 1) * K + k0 + col, tr < T);
            cp_async16(sB + stage * TILE_B + r * LDS + col, W + (size_t)min(nr, N - 1) * K + k0 + col, nr < N);
            if (SPLIT)
                cp_async16(sL + stage * TILE_A + r * LDS + col, X_lo + (size_t)min(tr, T - 1) * K + k0 + col, tr < T);
        }
    };

    float acc[2][8][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[i][j][q] = 0.f;

#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < ktiles) load_stage(s, s);
        cp_async_commit();
    }
    for (int kt = 0; kt < ktiles; ++kt) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        const int nk = kt + STAGES - 1;
        if (nk < ktiles) load_stage(nk % STAGES, nk);
        cp_async_commit();
        const bf16* a_s = sA + (kt % STAGES) * TILE_A;
        const bf16* b_s = sB + (kt % STAGES) * TILE_B;
#pragma unroll
        for (int kk = 0; kk < BK; kk += 16) {
            uint32_t af[2][4], bfr[4][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int r = wm * 32 + i * 16 + (lane & 15);
                ldmatrix_x4(af[i], a_s + r * LDS + kk + (lane >> 4) * 8);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = wn * 64 + j * 16 + (lane & 7) + ((lane >> 4) << 3);
                ldmatrix_x4(bfr[j], b_s + r * LDS + kk + ((lane >> 3) & 1) * 8);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    mma16816(acc[i][2 * j], af[i], &bfr[j][0]);
                    mma16816(acc[i][2 * j + 1], af[i], &bfr[j][2]);
                }
            if (SPLIT) {
                const bf16* l_s = sL + (kt % STAGES) * TILE_A;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int r = wm * 32 + i * 16 + (lane & 15);
                    ldmatrix_x4(af[i], l_s + r * LDS + kk + (lane >> 4) * 8);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        mma16816(acc[i][2 * j], af[i], &bfr[j][0]);
                        mma16816(acc[i][2 * j + 1], af[i], &bfr[j][2]);
                    }
            }
        }
    }
    cp_async_wait<0>();

    // epilogue: c0,c1 at (row lane/4, cols 2*(lane%4) + {0,1}); c2,c3 at row + 8
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int t = t0 + wm * 32 + i * 16 + (lane >> 2) + hr * 8;
            unsigned long long best = 0ull;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int n = n0 + wn * 64 + j * 8 + (lane & 3) * 2;
                const float v0 = acc[i][j][hr * 2], v1 = acc[i][j][hr * 2 + 1];
                if (t < T && n < N) {
                    if (e.mode == EPI_SWIGLU) {
                        const float mv = silu(v0) * v1;
                        reinterpret_cast<bf16*>(e.out)[(size_t)t * e.ldo + n / 2] = f2bf(mv);
                        if (e.out_lo) reinterpret_cast<bf16*>(e.out_lo)[(size_t)t * e.ldo + n / 2] = f2bf_lo(mv);
                    } else {
                        epi_one(e, t, n, v0);
                        if (n + 1 < N) epi_one(e, t, n + 1, v1);
                        if (e.mode == EPI_LOGITS) {
                            best = umax64(best, pack_argmax(v0, n));
                            if (n + 1 < N) best = umax64(best, pack_argmax(v1, n + 1));
                        }
                    }
                }
            }
            if (e.mode == EPI_LOGITS && e.amax) {
                best = umax64(best, shfl_xor_u64(best, 1));
                best = umax64(best, shfl_xor_u64(best, 2));
                if ((lane & 3) == 0 && t < T && best) atomicMax(e.amax + t, best);
            }
        }
}

int launch_gemm(const bf16* X, const bf16* W, int T, int N, int K, const Epi& e, cudaStream_t st, const bf16* X_lo,
                int* err) {
    if (T <= 0) return 0;
    if (T <= 8) return launch_gemv(X, W, T, N, K, e, st, X_lo);
    if (!X_lo && gemm_tc_available()) {
        const int n = launch_gemm_tc(X, W, T, N, K, e, err, st);
        if (n) return n;
    }
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(k_gemm_mma<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, gm::SMEM);
        cudaFuncSetAttribute(k_gemm_mma<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, gm::SMEM_SPLIT);
        attr_set = true;
    }
    dim3 grid((N + gm::BN - 1) / gm::BN, (T + gm::BM - 1) / gm::BM);
    if (X_lo)
        k_gemm_mma<true><<<grid, 256, gm::SMEM_SPLIT, st>>>(X, X_lo, W, T, N, K, e);
    else
        k_gemm_mma<false><<<grid, 256, gm::SMEM, st>>>(X, nullptr, W, T, N, K, e);
    return 1;
}

}  // namespace ttsbb
