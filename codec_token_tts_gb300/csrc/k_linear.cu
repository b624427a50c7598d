// Linear layers of the backbone step: Y = X W^T (W in PyTorch (out, in) layout)
// with fused epilogues (residual add, SwiGLU over interleaved gate/up rows,
// logits + argmax, permuted audio-head logits).
//   * k_gemv: T <= 8 token rows, weight streaming with 128-bit loads (HBM-bound
//     decode at small batch).
//   * k_gemm_mma: any T, bf16 tensor cores through mma.sync with a cp.async
//     pipeline.
#include <algorithm>

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
    pdl_wait();  // upstream results are read below
    pdl_trigger();
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
    launch_pdl(k_gemv<T, 2>, (N + rows_per_cta - 1) / rows_per_cta, 256, smem, st, X, X_lo, W, N, K, e);
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
    pdl_wait();  // upstream results are read below
    pdl_trigger();
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

// ---------------------------------------------------------------- split-K GEMM for decode batches
// Y[T][N] = (X + X_lo)[T][K] W[N][K]^T for 8 < T <= 256. CTA (n-tile, k-split)
// owns a 64-feature x KC slice of W and the matching T x KC activations: it
// issues every load of its slice at once (one round trip), computes a
// 64 x T partial on mma.sync (both activation parts), writes it to the
// workspace, and the last CTA to arrive at the n-tile's counter sums the K
// splits in index order and applies the epilogue (deterministic; it also
// re-arms the counter for the next launch). KC = 256 / MT keeps the
// activation chunk at 64 KB whatever T is.
namespace sk {
constexpr int BN = 64, LDS_PAD = 8, MAXT = 256;
}  // namespace sk

template <int MT>  // token tiles of 64; KC = 256 / MT
__global__ void __launch_bounds__(256) k_gemm_splitk(const bf16* __restrict__ X, const bf16* __restrict__ X_lo,
                                                     const bf16* __restrict__ W, int T, int N, int K, Epi e,
                                                     float* __restrict__ part, int* __restrict__ ctr) {
    pdl_wait();  // upstream results are read below
    pdl_trigger();
    using namespace sk;
    constexpr int KC = 256 / MT, LDS = KC + LDS_PAD, TP = MT * 64;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    bf16* sW = reinterpret_cast<bf16*>(smem_raw);  // [64][LDS]
    bf16* sA = sW + BN * LDS;                        // [TP][LDS]
    bf16* sL = sA + TP * LDS;                        // [TP][LDS]
    __shared__ int last_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 1, wn = warp & 1;  // 4 x 2 warps: rows wm*16 (+64 per token tile), cols wn*32
    const int n0 = blockIdx.x * BN, kc0 = blockIdx.y * KC;
    const int KS = gridDim.y;
    constexpr int CPR = KC / 8;  // 16-byte chunks per row

    for (int c = tid; c < BN * CPR; c += 256) {
        const int r = c / CPR, col = (c % CPR) * 8;
        cp_async16(sW + r * LDS + col, W + (size_t)(n0 + r) * K + kc0 + col, true);
    }
    for (int c = tid; c < TP * CPR; c += 256) {
        const int r = c / CPR, col = (c % CPR) * 8;
        const size_t src = (size_t)min(r, T - 1) * K + kc0 + col;
        cp_async16(sA + r * LDS + col, X + src, r < T);
        cp_async16(sL + r * LDS + col, X_lo + src, r < T);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();

    float acc[MT][4][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[mt][j][q] = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < KC; kk += 16) {
        uint32_t bfr[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int r = wn * 32 + j * 16 + (lane & 7) + ((lane >> 4) << 3);
            ldmatrix_x4(bfr[j], sW + r * LDS + kk + ((lane >> 3) & 1) * 8);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            uint32_t af[4], lf[4];
            const int r = mt * 64 + wm * 16 + (lane & 15);
            ldmatrix_x4(af, sA + r * LDS + kk + (lane >> 4) * 8);
            ldmatrix_x4(lf, sL + r * LDS + kk + (lane >> 4) * 8);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                mma16816(acc[mt][2 * j], af, &bfr[j][0]);
                mma16816(acc[mt][2 * j + 1], af, &bfr[j][2]);
                mma16816(acc[mt][2 * j], lf, &bfr[j][0]);
                mma16816(acc[mt][2 * j + 1], lf, &bfr[j][2]);
            }
        }
    }
    // partial tile -> workspace part[ks][t][n]
    float* pk = part + (size_t)blockIdx.y * T * N;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int t = mt * 64 + wm * 16 + (lane >> 2) + hr * 8;
            if (t >= T) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + wn * 32 + j * 8 + (lane & 3) * 2;
                *reinterpret_cast<float2*>(pk + (size_t)t * N + n) = make_float2(acc[mt][j][hr * 2], acc[mt][j][hr * 2 + 1]);
            }
        }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int old = atomicAdd(ctr + blockIdx.x, 1);
        last_s = (old == KS - 1);
        if (last_s) ctr[blockIdx.x] = 0;  // re-arm for the next launch
    }
    __syncthreads();
    if (!last_s) return;
    __threadfence();
    // last CTA: thread -> (t, 4 features); the K splits are summed in index
    // order, four splits' loads in flight at a time; then the epilogue
    for (int idx = tid; idx < T * (BN / 4); idx += 256) {
        const int t = idx / (BN / 4), n = n0 + (idx % (BN / 4)) * 4;
        const float* src = part + (size_t)t * N + n;
        const size_t sstride = (size_t)T * N;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        int s = 0;
        for (; s + 4 <= KS; s += 4) {
            float4 p[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) p[u] = __ldcg(reinterpret_cast<const float4*>(src + (s + u) * sstride));
#pragma unroll
            for (int u = 0; u < 4; ++u) { v.x += p[u].x; v.y += p[u].y; v.z += p[u].z; v.w += p[u].w; }
        }
        for (; s < KS; ++s) {
            const float4 p = __ldcg(reinterpret_cast<const float4*>(src + s * sstride));
            v.x += p.x; v.y += p.y; v.z += p.z; v.w += p.w;
        }
        const float vv[4] = {v.x, v.y, v.z, v.w};
        if (e.mode == EPI_SWIGLU) {
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
                const float mv = silu(vv[u]) * vv[u + 1];
                reinterpret_cast<bf16*>(e.out)[(size_t)t * e.ldo + (n + u) / 2] = f2bf(mv);
                if (e.out_lo) reinterpret_cast<bf16*>(e.out_lo)[(size_t)t * e.ldo + (n + u) / 2] = f2bf_lo(mv);
            }
        } else {
            unsigned long long best = 0ull;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                epi_one(e, t, n + u, vv[u]);
                const unsigned long long pk = pack_argmax(vv[u], n + u);
                best = pk > best ? pk : best;
            }
            if (e.mode == EPI_LOGITS && e.amax) atomicMax(e.amax + t, best);
        }
    }
}

template <int MT>
static constexpr int splitk_smem() {
    return (sk::BN + 2 * MT * 64) * (256 / MT + sk::LDS_PAD) * 2;
}

static int launch_splitk(const bf16* X, const bf16* X_lo, const bf16* W, int T, int N, int K, const Epi& e,
                         const SplitK& w, cudaStream_t st) {
    using namespace sk;
    if (T > MAXT || N % BN != 0 || N / BN > w.n_ctr) return 0;
    const int MT = T <= 64 ? 1 : (T <= 128 ? 2 : 4);
    const int KC = 256 / MT;
    if (K % KC != 0) return 0;
    const int KS = K / KC;
    if ((size_t)KS * T * N > w.part_elems) return 0;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_gemm_splitk<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, splitk_smem<1>());
        cudaFuncSetAttribute(k_gemm_splitk<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, splitk_smem<2>());
        cudaFuncSetAttribute(k_gemm_splitk<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, splitk_smem<4>());
        attr = true;
    }
    dim3 grid(N / BN, KS);
    switch (MT) {
        case 1: launch_pdl(k_gemm_splitk<1>, grid, 256, splitk_smem<1>(), st, X, X_lo, W, T, N, K, e, w.part, w.ctr); break;
        case 2: launch_pdl(k_gemm_splitk<2>, grid, 256, splitk_smem<2>(), st, X, X_lo, W, T, N, K, e, w.part, w.ctr); break;
        default: launch_pdl(k_gemm_splitk<4>, grid, 256, splitk_smem<4>(), st, X, X_lo, W, T, N, K, e, w.part, w.ctr); break;
    }
    return 1;
}

int launch_gemm(const bf16* X, const bf16* W, int T, int N, int K, const Epi& e, cudaStream_t st, const bf16* X_lo,
                int* err, const SplitK* skw) {
    if (T <= 0) return 0;
    if (e.mode == EPI_QKROPE || e.nrm_gamma || e.nrm_scale_ss)  // fused epilogues: the split-K decode GEMM only (else 0)
        return X_lo && T > 8 && gemm_tc_available() ? launch_gemm_tcd(X, X_lo, W, T, N, K, e, err, st) : 0;
    if (T <= 8) return launch_gemv(X, W, T, N, K, e, st, X_lo);
    if (X_lo && gemm_tc_available()) {
        // 128-token blocks (N = 2 x block <= 256 per MMA); 0 if the product does not fit the kernel
        const int n = launch_gemm_tcd(X, X_lo, W, T, N, K, e, err, st);
        if (n) return n;
    }
    if (X_lo && T > 256 && gemm_tc_available()) {
        // split activations beyond 256 tokens (a causal prefill): the dense persistent kernel, two
        // passes over K (high parts, then low parts) into the same accumulator
        const int n = launch_gemm_tc(X, W, T, N, K, e, err, st, X_lo);
        if (n) return n;
    }
    if (X_lo && skw) {
        const int n = launch_splitk(X, X_lo, W, T, N, K, e, *skw, st);
        if (n) return n;
    }
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
        launch_pdl(k_gemm_mma<true>, grid, 256, gm::SMEM_SPLIT, st, X, X_lo, W, T, N, K, e);
    else
        launch_pdl(k_gemm_mma<false>, grid, 256, gm::SMEM, st, X, (const bf16*)nullptr, W, T, N, K, e);
    return 1;
}

}  // namespace ttsbb
