// DAC decoder: frame features -> 24 kHz audio ("omnivoice-cpp
// docs/ARCHITECTURE.md", Audio tokenizer pipeline, Decode; DAC decoder block
// channels; Snake activation; ConvTranspose1d). fc2 (1024 -> 256), conv1
// (256 -> 1024, k 7), five blocks (snake, ConvTranspose1d k 2r stride r, then
// three residual units: snake, Conv1d k 7 dilation 1/3/9, snake, Conv1d k 1,
// add), snake, conv2 (32 -> 1, k 7): 960 samples per frame.
//
// Activations are fp32 [B][C][T]. k_dac_conv computes a 64-channel x
// 128-sample output tile per CTA: input channels in chunks of 16, their
// snake'd input window (128 + (K - 1) d samples, zero outside the sequence:
// the snake of 0 is 0) and the weight slice staged in shared memory. A thread
// owns 4 output channels x two runs of 4 contiguous samples (64 apart); per
// input channel it reads each run's window of 4 + (K - 1) d samples once, as
// 16-byte loads that are contiguous across the warp, and applies every tap
// from registers. Bias and an optional residual (read and written by the same
// thread, so the add can be in place) in the epilogue.
// k_dac_convT is output-stationary: with K = 2 s, output sample o takes input
// samples q / s and q / s - 1 (q = o + p) through taps q mod s and q mod s + s.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "common.cuh"
#include "tcgen05.cuh"
#include "../../include/tts_bb.h"

#define TTS_API extern "C" __attribute__((visibility("default")))

using namespace ttsbb;

namespace dac {
constexpr int RATIOS[5] = {8, 5, 4, 2, 3};
constexpr int CH[6] = {1024, 512, 256, 128, 64, 32};
constexpr int DIL[3] = {1, 3, 9};
constexpr int TO = 128, TOC = 64, ICC = 16, NT = 256, MAXW = TO + 6 * 9 + 2;  // + the last window's 16-byte tail
constexpr int ICC_T = 8, MAXK_T = 16, MAXW_T = TO / 2 + 3;
}  // namespace dac

struct DacBlockW {
    float *alpha, *up_w, *up_b;
    float *a1[3], *w1[3], *b1[3], *a2[3], *w2[3], *b2[3];
    float *alpha_inv, *a1_inv[3], *a2_inv[3];  // 1 / (alpha + 1e-9) (tensor-core path)
};

// One convolution on the tensor-core path: packed weights and their tensor map.
struct DacTcConv {
    bf16* wp = nullptr;
    CUtensorMap map;
    int IC = 0, OC = 0, taps = 0, dil = 1, pad = 0, s = 1, po = 0, N = 0, NTL = 0, Npad = 0;
    int bk = 64;  // channels per K chunk (32 when IC is 32)
};

struct tts_bb_dac {
    cudaStream_t st = nullptr;
    bool tc = false;  // convolutions of conv1 and the blocks on tcgen05
    DacTcConv tc_fc2, tc_conv1, tc_up[5], tc_r1[5][3], tc_r2[5][3];
    int* err = nullptr;    // device error word of the tcgen05 kernels
    int* h_err = nullptr;  // pinned host copy
    int n_sm = 1;
    float *fc2_w = nullptr, *fc2_b = nullptr, *conv1_w = nullptr, *conv1_b = nullptr;
    DacBlockW blk[5] = {};
    float *final_alpha = nullptr, *conv2_w = nullptr, *conv2_b = nullptr, *final_inv = nullptr;
    float *buf[3] = {nullptr, nullptr, nullptr};
    size_t buf_elems = 0;
    std::vector<void*> allocs;
};

namespace {

// snake with the reciprocal 1 / (a + 1e-9) precomputed (the same value the division gives)
__device__ __forceinline__ float dac_snake_inv(float x, float a, float inv) {
    const float s = sinf(a * x);
    return x + inv * s * s;
}

__device__ __forceinline__ float dac_snake(float x, float a) {
    const float s = sinf(a * x);
    return x + (1.f / (a + 1e-9f)) * s * s;
}

// y[b][oc][t] = bias[oc] + sum_ic sum_k w[oc][ic][k] snake(x[b][ic][t + k dil - pad]) (+ res[b][oc][t])
// x element (b, ic, t) at x + b xb + ic xc + t xt. grid (ceil(T_out / 128), ceil(OC / 64), B), 256 threads.
// Thread (ty, tx): channels oc0 + 4 ty + q, samples t0 + 4 tx + 64 h + j (q, j < 4, h < 2).
template <int K, int DIL>
__global__ void __launch_bounds__(dac::NT) k_dac_conv(const float* __restrict__ x, long xb, long xc, long xt,
                                                      const float* __restrict__ alpha, const float* __restrict__ w,
                                                      const float* __restrict__ bias, const float* res, float* y, int IC,
                                                      int OC, int T_in, int T_out, int pad) {
    using namespace dac;
    constexpr int KP = (K + 3) & ~3;                    // taps padded to whole 16-byte rows
    constexpr int NWIN = (4 + (K - 1) * DIL + 3) / 4;   // 16-byte pieces of one run's window
    __shared__ __align__(16) float xs[ICC][MAXW];
    __shared__ __align__(16) float ws[TOC][ICC][KP];
    static_assert(4 * 15 + 64 + 4 * NWIN <= MAXW, "window past the staged row");
    const int t0 = blockIdx.x * TO, oc0 = blockIdx.y * TOC, b = blockIdx.z;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int W = TO + (K - 1) * DIL;
    const float* xbp = x + (size_t)b * xb;
    float acc[4][8];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[q][j] = 0.f;
    for (int ic0 = 0; ic0 < IC; ic0 += ICC) {
        for (int i = tid; i < ICC * MAXW; i += NT) {
            const int c = i / MAXW, tt = i - c * MAXW, ic = ic0 + c, ti = t0 + tt - pad;
            float v = 0.f;
            if (tt < W && ic < IC && ti >= 0 && ti < T_in) {
                v = xbp[(size_t)ic * xc + (size_t)ti * xt];
                if (alpha) v = dac_snake(v, alpha[ic]);
            }
            xs[c][tt] = v;
        }
        for (int i = tid; i < TOC * ICC * KP; i += NT) {
            const int o = i / (ICC * KP), r = i - o * (ICC * KP), c = r / KP, k = r - c * KP;
            const int oc = oc0 + o, ic = ic0 + c;
            ws[o][c][k] = (k < K && oc < OC && ic < IC) ? w[((size_t)oc * IC + ic) * K + k] : 0.f;
        }
        __syncthreads();
#pragma unroll 2
        for (int c = 0; c < ICC; ++c) {
            float wv[4][KP];
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int k4 = 0; k4 < KP; k4 += 4) {
                    const float4 f = *reinterpret_cast<const float4*>(&ws[ty * 4 + q][c][k4]);
                    wv[q][k4] = f.x; wv[q][k4 + 1] = f.y; wv[q][k4 + 2] = f.z; wv[q][k4 + 3] = f.w;
                }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float xv[4 * NWIN];
#pragma unroll
                for (int p4 = 0; p4 < NWIN; ++p4) {
                    const float4 f = *reinterpret_cast<const float4*>(&xs[c][4 * tx + 64 * h + 4 * p4]);
                    xv[4 * p4] = f.x; xv[4 * p4 + 1] = f.y; xv[4 * p4 + 2] = f.z; xv[4 * p4 + 3] = f.w;
                }
#pragma unroll
                for (int k = 0; k < K; ++k)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[q][4 * h + j] = fmaf(wv[q][k], xv[j + k * DIL], acc[q][4 * h + j]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int oc = oc0 + ty * 4 + q;
        if (oc >= OC) continue;
        const float bv = bias[oc];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int t = t0 + 4 * tx + 64 * (j >> 2) + (j & 3);
            if (t >= T_out) continue;
            const size_t o = ((size_t)b * OC + oc) * T_out + t;
            float v = acc[q][j] + bv;
            if (res) v += res[o];
            y[o] = v;
        }
    }
}

// ConvTranspose1d, K = 2 s: y[b][oc][o] = bias[oc] + sum_ic (w[ic][oc][r] snake(x[ic][m]) +
// w[ic][oc][r + s] snake(x[ic][m - 1])), q = o + p, m = q / s, r = q % s (taps outside the input skipped).
// grid (ceil(T_out / 128), ceil(OC / 64), B), 256 threads.
__global__ void __launch_bounds__(dac::NT) k_dac_convT(const float* __restrict__ x, const float* __restrict__ alpha,
                                                       const float* __restrict__ w, const float* __restrict__ bias,
                                                       float* __restrict__ y, int IC, int OC, int T_in, int T_out, int s,
                                                       int p) {
    using namespace dac;
    __shared__ float xs[ICC_T][MAXW_T];
    __shared__ float ws[ICC_T][TOC][MAXK_T];
    const int t0 = blockIdx.x * TO, oc0 = blockIdx.y * TOC, b = blockIdx.z;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int K = 2 * s;
    const int m0 = (t0 + p) / s - 1;                        // first input sample the tile reads
    const int W = (t0 + TO - 1 + p) / s - m0 + 1;           // <= 128 / s + 2
    const float* xbp = x + (size_t)b * IC * T_in;
    float acc[4][8];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[q][j] = 0.f;
    for (int ic0 = 0; ic0 < IC; ic0 += ICC_T) {
        for (int i = tid; i < ICC_T * W; i += NT) {
            const int c = i / W, tt = i - c * W, ic = ic0 + c, ti = m0 + tt;
            float v = 0.f;
            if (ic < IC && ti >= 0 && ti < T_in) v = dac_snake(xbp[(size_t)ic * T_in + ti], alpha[ic]);
            xs[c][tt] = v;
        }
        for (int i = tid; i < ICC_T * TOC * K; i += NT) {
            const int c = i / (TOC * K), r = i - c * (TOC * K), o = r / K, k = r - o * K;
            const int ic = ic0 + c, oc = oc0 + o;
            ws[c][o][k] = (ic < IC && oc < OC) ? w[((size_t)ic * OC + oc) * K + k] : 0.f;
        }
        __syncthreads();
#pragma unroll 2
        for (int c = 0; c < ICC_T; ++c) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int q = t0 + tx + 16 * j + p, m = q / s, r = q - m * s;
                const float x0 = xs[c][m - m0], x1 = xs[c][m - 1 - m0];
#pragma unroll
                for (int qq = 0; qq < 4; ++qq)
                    acc[qq][j] = fmaf(ws[c][ty * 4 + qq][r], x0, fmaf(ws[c][ty * 4 + qq][r + s], x1, acc[qq][j]));
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int oc = oc0 + ty * 4 + q;
        if (oc >= OC) continue;
        const float bv = bias[oc];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int t = t0 + tx + 16 * j;
            if (t < T_out) y[((size_t)b * OC + oc) * T_out + t] = acc[q][j] + bv;
        }
    }
}

// ---------------------------------------------------------------- tensor-core convolutions
// conv1 and every convolution of the blocks as an implicit GEMM on tcgen05:
// D[u][n] = sum_k sum_ic A[u + k dil - pad][ic] W_k[n][ic] over output rows u, where A is the
// convolution's input after its snake, kept time-major ([T][C]) as bf16 high + low parts, so the
// 128 x 64 operand tile of tap k is one TMA box at row u0 + k dil - pad (rows outside the item and
// channels past C read as zeros). A plain convolution has n = oc and writes row u to sample u;
// ConvTranspose1d (K = 2 s) is two taps over input rows u - 1 and u with weights w[ic][oc][ph + s]
// and w[ic][oc][ph], and column n = ph OC + oc writes sample u s + ph - p (q = o + p, m = q / s,
// ph = q mod s: every output phase of input row u is a column of the same product). Activations on
// this path are time-major ([B][T][C]), so each thread's 16 columns are 16 contiguous channels of
// one output sample in every tensor it reads or writes.
// fp32 operands enter as high + low parts (x = hi + lo to ~2^-17): D = A_hi W_hi + A_hi W_lo +
// A_lo W_hi in fp32 (the dropped A_lo W_lo is ~2^-18 of each product).
// Persistent, like the dense GEMM: a TMA thread fills a 3-stage ring with the four tiles of each
// (channel chunk, tap) step (A hi / lo, W hi / lo), one thread issues the step's 12 MMAs (M 128,
// N NTL <= 128, K 16) into one of two TMEM accumulators, and eight epilogue warps (two per TMEM
// lane quarter, half the columns each) drain the other:
// bias, an optional fp32 residual (read and written by the same thread, so in place is allowed),
// the fp32 output, and the next convolution's input: snake of this output as high + low parts.
// The snake's sine is reduced to [-pi/2, pi/2] first (sin^2 has period pi; Cody and Waite's
// two-constant reduction with fused multiply-adds) and then taken by the hardware sine, whose
// absolute error there is ~2^-21. Every wait is bounded.
namespace dig {
constexpr int BM = 128, BK = 64, MAXN = 128, NT = 320, STAGES = 3;  // warps 2-9: epilogue
constexpr int A_BYTES = BM * BK * 2;                   // one part of an A tile (of 64 channels at most)
constexpr int W_BYTES = MAXN * BK * 2;                 // one part of a W tile (NTL rows used)
constexpr int STAGE = 2 * A_BYTES + 2 * W_BYTES;       // A hi, A lo, W hi, W lo
constexpr int BAR_OFF = STAGES * STAGE;
constexpr int MAXOC = 1024;
constexpr int PAR_OFF = BAR_OFF + 256;                 // bias, alpha, 1 / (alpha + 1e-9) per channel
constexpr int SMEM = PAR_OFF + 3 * MAXOC * 4 + 1024;   // + alignment of the dynamic base
constexpr int TMEM_COLS = 2 * MAXN;                    // two accumulators
}  // namespace dig

// snake(x) = x + inv sin^2(a x) with a x reduced by the nearest multiple of pi (pi = PI_HI + PI_LO,
// both floats) before the hardware sine
__device__ __forceinline__ float dac_snake_fast(float x, float a, float inv) {
    constexpr float INV_PI = 0.318309886183790672f, PI_HI = 3.14159274101257324f, PI_LO = -8.74227766e-8f;
    const float y = a * x;
    const float k = rintf(y * INV_PI);
    const float r = fmaf(-k, PI_LO, fmaf(-k, PI_HI, y));
    const float sn = __sinf(r);
    return fmaf(inv * sn, sn, x);
}
static_assert(dig::SMEM <= 232448, "shared memory per CTA");

// K-major operand with 64-byte rows (32 bf16) in 64-byte-swizzle atoms of 8 rows (512 B apart):
// layout SWIZZLE_64B (4) at bits 61-63, otherwise as the 128-byte form
__device__ __forceinline__ uint64_t sw64_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(512 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)4 << 61;
    return d;
}

struct DacIgArgs {
    int IC, OC, T_in, T_out, B;
    int bk;               // channels per K chunk: 64 (128-byte rows) or 32 (64-byte rows, for IC = 32)
    int taps, dil, pad;   // tap k of row u reads input row u + k dil - pad
    int s, po;            // column n: channel n mod OC, output sample u s + n / OC - po
    int U, N, NTL, Npad;  // rows, columns (s OC), columns per tile, rows of one (part, tap) weight block
    const float* bias;    // [OC]
    const float* res;     // [B][T_out][OC] added, or null (may alias y)
    float* y;             // [B][T_out][OC] fp32 output, or null
    bf16* s_out;          // [2][B][T_out][OC] next input: high, low parts of snake(out), or null
    const float* alpha_out;  // that snake's alpha [OC] (null: the output itself)
    const float* alpha_inv;  // 1 / (alpha_out + 1e-9) [OC]
    int* err;
};

__global__ void __launch_bounds__(dig::NT, 1)
    k_dac_igemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                const __grid_constant__ DacIgArgs a) {
    using namespace dig;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
    uint64_t* empty = full + STAGES;
    uint64_t* accf = empty + STAGES;  // [2] accumulator ready (MMA -> epilogue)
    uint64_t* acce = accf + 2;        // [2] accumulator drained (4 epilogue warp arrivals)
    uint64_t* fin = acce + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
    volatile int* abort_s = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* p_bias = reinterpret_cast<float*>(smem + PAR_OFF);
    float* p_alpha = p_bias + MAXOC;
    float* p_inv = p_alpha + MAXOC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int MT = (a.U + BM - 1) / BM, NTT = a.Npad / a.NTL, tiles = MT * NTT * a.B;
    const int bk = a.bk, nch = (a.IC + bk - 1) / bk, KT = nch * a.taps;
    for (int i = threadIdx.x; i < a.OC; i += blockDim.x) {  // OC <= MAXOC (checked on the host)
        p_bias[i] = a.bias[i];
        p_alpha[i] = a.alpha_out ? a.alpha_out[i] : 0.f;
        p_inv[i] = a.alpha_out ? a.alpha_inv[i] : 0.f;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            tc_mbar_init(full + i, 1);
            tc_mbar_init(empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc_mbar_init(accf + i, 1);
            tc_mbar_init(acce + i, 8);
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

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer: the stage ring runs on across tiles
            uint32_t g = 0;
            const uint32_t bytes = (uint32_t)(2 * BM * bk * 2 + 2 * a.NTL * bk * 2);
            for (int tile = blockIdx.x; tile < tiles && !*abort_s; tile += gridDim.x) {
                const int mt = tile % MT, rest = tile / MT, n0 = (rest % NTT) * a.NTL, b = rest / NTT;
                const int u0 = mt * BM;
                for (int kt = 0; kt < KT; ++kt, ++g) {
                    const int st = g % STAGES, c = kt / a.taps, k = kt - c * a.taps;
                    if (g >= STAGES && !tc_wait(empty + st, ((g / STAGES) - 1) & 1, abort_s)) {
                        *abort_s = 1;
                        break;
                    }
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(s_addr(full + st)),
                                 "r"(bytes)
                                 : "memory");
                    unsigned char* sp = smem + st * STAGE;
                    const int row = u0 + k * a.dil - a.pad;
                    tma_load_4d(sp, &tmA, c * bk, row, b, 0, full + st);
                    tma_load_4d(sp + A_BYTES, &tmA, c * bk, row, b, 1, full + st);
                    tma_load_2d(sp + 2 * A_BYTES, &tmW, c * bk, k * a.Npad + n0, full + st);
                    tma_load_2d(sp + 2 * A_BYTES + W_BYTES, &tmW, c * bk, (a.taps + k) * a.Npad + n0, full + st);
                }
            }
            if (*abort_s)  // let the copies in flight land before the CTA can exit
                for (uint32_t i = g > (uint32_t)STAGES ? g - STAGES : 0; i < g; ++i) {
                    const unsigned long long t0 = g_time();
                    while (!tc_mbar_try(full + i % STAGES, (i / STAGES) & 1) && g_time() - t0 < TC_TIMEOUT_NS) {
                    }
                }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------- MMA issuer
            const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(a.NTL >> 3) << 17) |
                                   ((uint32_t)(BM >> 4) << 24);
            uint32_t g = 0;
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x, ++it) {
                const int buf = it & 1;
                if (it >= 2 && !tc_wait(acce + buf, ((it >> 1) - 1) & 1, abort_s)) {
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t d = tmem + (uint32_t)(buf * MAXN);
                for (int kt = 0; kt < KT; ++kt, ++g) {
                    const int st = g % STAGES;
                    if (!tc_wait(full + st, (g / STAGES) & 1, abort_s)) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t ah = s_addr(smem + st * STAGE), al = ah + A_BYTES;
                    const uint32_t wh = ah + 2 * A_BYTES, wl = wh + W_BYTES;
                    if (bk == 64) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t off = (uint32_t)(kk * 32);
                            at_mma(d, sw128_desc(ah + off), sw128_desc(wh + off), idesc, (kt | kk) ? 1u : 0u);
                            at_mma(d, sw128_desc(ah + off), sw128_desc(wl + off), idesc, 1u);
                            at_mma(d, sw128_desc(al + off), sw128_desc(wh + off), idesc, 1u);
                        }
                    } else {  // 32 channels: two K steps in 64-byte rows
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const uint32_t off = (uint32_t)(kk * 32);
                            at_mma(d, sw64_desc(ah + off), sw64_desc(wh + off), idesc, (kt | kk) ? 1u : 0u);
                            at_mma(d, sw64_desc(ah + off), sw64_desc(wl + off), idesc, 1u);
                            at_mma(d, sw64_desc(al + off), sw64_desc(wh + off), idesc, 1u);
                        }
                    }
                    at_commit(empty + st);
                }
                if (!ok) break;
                at_commit(accf + buf);
            }
            if (!ok) *abort_s = 1;
            at_commit(fin);  // every MMA issued completes before TMEM may be freed
            const unsigned long long t0 = g_time();
            while (!tc_mbar_try(fin, 0) && g_time() - t0 < TC_TIMEOUT_NS) {
            }
        }
    } else {
        // ---------------- epilogue: warp w reads TMEM lanes 32 (w % 4) .. (one output row per thread),
        // columns [h NTL / 2, (h + 1) NTL / 2) with h = (w - 2) / 4: two warps per row quarter
        const int q = warp & 3, h = (warp - 2) >> 2;
        int it = 0;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++it) {
            const int buf = it & 1;
            if (!tc_wait(accf + buf, (it >> 1) & 1, abort_s) || *abort_s) {
                if (lane == 0 && q == 0) set_err(a.err, ERR_TIMEOUT);
                *abort_s = 1;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int mt = tile % MT, rest = tile / MT, n0 = (rest % NTT) * a.NTL, b = rest / NTT;
            const int u = mt * BM + q * 32 + lane, half = a.NTL >> 1;
            for (int c0 = h * half; c0 < (h + 1) * half; c0 += 16) {
                uint32_t v[16];
                __syncwarp();  // the TMEM load is warp-collective: converge after the row guard below
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
                    "[%16];"
                    : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                      "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                    : "r"(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * MAXN + c0)));
                tm_wait_ld();
                if (u >= a.U) continue;
                // the 16 columns are channels oc0 .. oc0 + 15 of output phase ph (OC is a multiple of 16)
                const int n = n0 + c0, ph = n / a.OC, oc0 = n - ph * a.OC;
                const int o = u * a.s + ph - a.po;
                if (n >= a.N || o < 0 || o >= a.T_out) continue;
                const size_t row = ((size_t)b * a.T_out + o) * a.OC + oc0;
                float x[16];
                if (a.res) {  // every residual load before any store (y may alias res)
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        const float4 r4 = *reinterpret_cast<const float4*>(a.res + row + j);
                        x[j] = r4.x; x[j + 1] = r4.y; x[j + 2] = r4.z; x[j + 3] = r4.w;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) x[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) x[j] += __uint_as_float(v[j]) + p_bias[oc0 + j];
                if (a.y) {
#pragma unroll
                    for (int j = 0; j < 16; j += 4)
                        *reinterpret_cast<float4*>(a.y + row + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
                }
                if (a.s_out) {
                    if (a.alpha_out) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) x[j] = dac_snake_fast(x[j], p_alpha[oc0 + j], p_inv[oc0 + j]);
                    }
                    bf16* hrow = a.s_out + row;
                    bf16* lrow = hrow + (size_t)a.B * a.T_out * a.OC;
#pragma unroll
                    for (int p8 = 0; p8 < 2; ++p8) {
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int q2 = 0; q2 < 4; ++q2) {
                            const float f0 = x[8 * p8 + 2 * q2], f1 = x[8 * p8 + 2 * q2 + 1];
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(f0, f1);
                            const float2 hf = __bfloat1622float2(h2);
                            __nv_bfloat162 l2 = __floats2bfloat162_rn(f0 - hf.x, f1 - hf.y);
                            hi[q2] = *reinterpret_cast<uint32_t*>(&h2);
                            lo[q2] = *reinterpret_cast<uint32_t*>(&l2);
                        }
                        *reinterpret_cast<uint4*>(hrow + 8 * p8) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4*>(lrow + 8 * p8) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(s_addr(acce + buf)) : "memory");
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
    }
}

__global__ void k_dac_recip(const float* __restrict__ alpha, int n, float* __restrict__ inv) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) inv[i] = 1.f / (alpha[i] + 1e-9f);
}

// x fp32 [n] -> s_out [2][n]: high and low bf16 parts (the time-major features, input of fc2).
__global__ void k_dac_split(const float* __restrict__ x, size_t n, bf16* __restrict__ s_out) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const float v = x[i];
        const bf16 h = __float2bfloat16_rn(v);
        s_out[i] = h;
        s_out[i + n] = __float2bfloat16_rn(v - __bfloat162float(h));
    }
}

// conv2 (32 -> 1, k 7, pad 3) on the snake'd input given as high + low parts, time-major
// [2][B][T][32]: audio[b][t] = bias + sum_k sum_c w[c][k] x[t + k - 3][c]. grid (ceil(T / 256), B),
// 256 threads; the 262-row window (hi + lo summed in fp32) is staged in shared memory.
__global__ void __launch_bounds__(256) k_dac_conv2(const bf16* __restrict__ s_in, const float* __restrict__ w,
                                                   const float* __restrict__ bias, int T, int B,
                                                   float* __restrict__ audio) {
    __shared__ float xs[262][33];
    __shared__ float ws[7][32];
    const int t0 = blockIdx.x * 256, b = blockIdx.y;
    const size_t lo_off = (size_t)B * T * 32;
    for (int i = threadIdx.x; i < 224; i += 256) ws[i % 7][i / 7] = w[i];  // w [1][32][7]
    for (int i = threadIdx.x; i < 262 * 4; i += 256) {  // 16-byte pieces: 8 channels of one row, both parts
        const int r = i >> 2, pc = i & 3, t = t0 - 3 + r;
        uint4 hv = make_uint4(0u, 0u, 0u, 0u), lv = hv;
        if (t >= 0 && t < T) {
            const size_t si = ((size_t)b * T + t) * 32 + pc * 8;
            hv = *reinterpret_cast<const uint4*>(s_in + si);
            lv = *reinterpret_cast<const uint4*>(s_in + si + lo_off);
        }
        const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w}, lw[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            xs[r][pc * 8 + 2 * j] = __uint_as_float(hw[j] << 16) + __uint_as_float(lw[j] << 16);
            xs[r][pc * 8 + 2 * j + 1] = __uint_as_float(hw[j] & 0xFFFF0000u) + __uint_as_float(lw[j] & 0xFFFF0000u);
        }
    }
    __syncthreads();
    const int t = t0 + threadIdx.x;
    if (t >= T) return;
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < 7; ++k)
#pragma unroll
        for (int c = 0; c < 32; ++c) acc = fmaf(ws[k][c], xs[threadIdx.x + k][c], acc);
    audio[(size_t)b * T + t] = acc + bias[0];
}

// Packed weights for k_dac_igemm: out[(part * taps + k) * Npad + n][ic] bf16 (part 0 high, 1 low,
// zero past OC x s columns and IC channels), ICpad columns. transposed = 0: w [OC][IC][taps] (tap k,
// column n = oc); 1: ConvTranspose1d w [IC][OC][2 s] (tap 0 = input u - 1: w[..][ph + s], tap 1 = input
// u: w[..][ph], column n = ph OC + oc).
__global__ void k_dac_pack(const float* __restrict__ w, int transposed, int IC, int OC, int taps, int s, int Npad,
                           int ICpad, bf16* __restrict__ out) {
    const size_t total = (size_t)2 * taps * Npad * ICpad;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int ic = (int)(i % ICpad);
        const size_t rr = i / ICpad;
        const int n = (int)(rr % Npad), k = (int)((rr / Npad) % taps), part = (int)(rr / ((size_t)Npad * taps));
        float v = 0.f;
        if (ic < IC && n < OC * s) {
            if (!transposed) {
                v = w[((size_t)n * IC + ic) * taps + k];
            } else {
                const int ph = n / OC, oc = n - ph * OC;
                v = w[((size_t)ic * OC + oc) * (2 * s) + (k == 0 ? ph + s : ph)];
            }
        }
        const bf16 hi = __float2bfloat16_rn(v);
        out[i] = part == 0 ? hi : __float2bfloat16_rn(v - __bfloat162float(hi));
    }
}

template <typename T>
cudaError_t dalloc_copy(tts_bb_dac* d, T** dst, const void* src, size_t n) {
    void* v = nullptr;
    cudaError_t e = cudaMalloc(&v, n * sizeof(T));
    if (e != cudaSuccess) return e;
    d->allocs.push_back(v);
    *dst = static_cast<T*>(v);
    if (src) e = cudaMemcpyAsync(v, src, n * sizeof(T), cudaMemcpyDefault, d->st);
    return e;
}

// Pack one convolution's weights for the tensor-core path (transposed: ConvTranspose1d with stride s).
bool tc_prepare(tts_bb_dac* d, DacTcConv& c, const float* w, bool transposed, int IC, int OC, int K, int dil, int pad,
                int s) {
    c.IC = IC;
    c.OC = OC;
    c.taps = transposed ? 2 : K;
    c.dil = transposed ? 1 : dil;
    c.pad = transposed ? 1 : pad;
    c.s = transposed ? s : 1;
    c.po = transposed ? (s + 1) / 2 : 0;
    c.N = OC * c.s;
    c.NTL = c.N < dig::MAXN ? c.N : dig::MAXN;
    if (c.NTL % 32 != 0 || c.N % c.NTL != 0 || IC % 8 != 0 || OC % 16 != 0 || OC > dig::MAXOC) return false;
    c.Npad = c.N;
    c.bk = IC == 32 ? 32 : dig::BK;
    const int ICpad = (IC + c.bk - 1) / c.bk * c.bk;
    const size_t n = (size_t)2 * c.taps * c.Npad * ICpad;
    if (dalloc_copy(d, &c.wp, nullptr, n) != cudaSuccess) return false;
    k_dac_pack<<<1024, 256, 0, d->st>>>(w, transposed ? 1 : 0, IC, OC, c.taps, c.s, c.Npad, ICpad, c.wp);
    if (cudaGetLastError() != cudaSuccess) return false;
    return tc_make_map_k(&c.map, c.wp, 2 * c.taps * c.Npad, ICpad, c.NTL, c.bk);
}

// One convolution on the tensor-core path. s_in: its input (after its snake) as [2][B][T_in][IC]
// high / low parts. Outputs: y (fp32 [B][T_out][OC], + res), and s_out = the next convolution's input
// (snake alpha_out of this output, [2][B][T_out][OC]); either may be null. Rows: output samples, or
// input samples 0 .. T_in for ConvTranspose1d (every output phase of a row is a column).
bool tc_conv(tts_bb_dac* d, const DacTcConv& c, const bf16* s_in, int B, int T_in, int T_out, const float* bias,
             const float* res, float* y, bf16* s_out, const float* alpha_out, const float* alpha_inv) {
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_dac_igemm, cudaFuncAttributeMaxDynamicSharedMemorySize, dig::SMEM);
        attr = true;
    }
    CUtensorMap ma;
    if (!tc_make_map_rows(&ma, s_in, c.IC, T_in, B, 2, c.bk)) return false;
    DacIgArgs a{c.IC, c.OC, T_in, T_out, B, c.bk, c.taps, c.dil, c.pad, c.s, c.po, c.s > 1 ? T_in + 1 : T_out,
                c.N, c.NTL, c.Npad, bias, res, y, s_out, alpha_out, alpha_inv, d->err};
    const long tiles = (long)((a.U + dig::BM - 1) / dig::BM) * (c.Npad / c.NTL) * B;
    const int grid = (int)std::min<long>(tiles, d->n_sm);
    k_dac_igemm<<<grid, dig::NT, dig::SMEM, d->st>>>(ma, c.map, a);
    return true;
}

void conv(tts_bb_dac* d, const float* x, long xb, long xc, long xt, const float* alpha, const float* w,
          const float* bias, const float* res, float* y, int B, int IC, int OC, int T_in, int T_out, int K, int dil,
          int pad) {
    dim3 grid((T_out + dac::TO - 1) / dac::TO, (OC + dac::TOC - 1) / dac::TOC, B);
    if (K == 1)
        k_dac_conv<1, 1><<<grid, dac::NT, 0, d->st>>>(x, xb, xc, xt, alpha, w, bias, res, y, IC, OC, T_in, T_out, pad);
    else if (dil == 1)
        k_dac_conv<7, 1><<<grid, dac::NT, 0, d->st>>>(x, xb, xc, xt, alpha, w, bias, res, y, IC, OC, T_in, T_out, pad);
    else if (dil == 3)
        k_dac_conv<7, 3><<<grid, dac::NT, 0, d->st>>>(x, xb, xc, xt, alpha, w, bias, res, y, IC, OC, T_in, T_out, pad);
    else
        k_dac_conv<7, 9><<<grid, dac::NT, 0, d->st>>>(x, xb, xc, xt, alpha, w, bias, res, y, IC, OC, T_in, T_out, pad);
}

}  // namespace

TTS_API void tts_bb_dac_free(tts_bb_dac* d) {
    if (!d) return;
    cudaStreamSynchronize(d->st);
    for (void* p : d->allocs) cudaFree(p);
    if (d->h_err) cudaFreeHost(d->h_err);
    delete d;
}

TTS_API tts_bb_status tts_bb_dac_create(const tts_bb_dac_weights* w, void* stream, tts_bb_dac** out) {
    if (!out) return TTS_BB_E_INVALID;
    *out = nullptr;
    if (!w || !w->fc2_w || !w->fc2_b || !w->conv1_w || !w->conv1_b || !w->final_alpha || !w->conv2_w || !w->conv2_b)
        return TTS_BB_E_INVALID;
    for (int i = 0; i < 5; ++i) {
        const tts_bb_dac_block& bw = w->block[i];
        if (!bw.alpha || !bw.up_w || !bw.up_b) return TTS_BB_E_INVALID;
        for (int j = 0; j < 3; ++j)
            if (!bw.res_alpha1[j] || !bw.res_w1[j] || !bw.res_b1[j] || !bw.res_alpha2[j] || !bw.res_w2[j] ||
                !bw.res_b2[j])
                return TTS_BB_E_INVALID;
    }
    tts_bb_dac* d = new tts_bb_dac();
    d->st = static_cast<cudaStream_t>(stream);
    bool ok = dalloc_copy(d, &d->fc2_w, w->fc2_w, 256 * 1024) == cudaSuccess &&
              dalloc_copy(d, &d->fc2_b, w->fc2_b, 256) == cudaSuccess &&
              dalloc_copy(d, &d->conv1_w, w->conv1_w, (size_t)1024 * 256 * 7) == cudaSuccess &&
              dalloc_copy(d, &d->conv1_b, w->conv1_b, 1024) == cudaSuccess &&
              dalloc_copy(d, &d->final_alpha, w->final_alpha, 32) == cudaSuccess &&
              dalloc_copy(d, &d->conv2_w, w->conv2_w, 32 * 7) == cudaSuccess &&
              dalloc_copy(d, &d->conv2_b, w->conv2_b, 1) == cudaSuccess;
    for (int i = 0; i < 5 && ok; ++i) {
        const int ic = dac::CH[i], oc = dac::CH[i + 1], r = dac::RATIOS[i];
        const tts_bb_dac_block& bw = w->block[i];
        DacBlockW& bd = d->blk[i];
        ok = dalloc_copy(d, &bd.alpha, bw.alpha, ic) == cudaSuccess &&
             dalloc_copy(d, &bd.up_w, bw.up_w, (size_t)ic * oc * 2 * r) == cudaSuccess &&
             dalloc_copy(d, &bd.up_b, bw.up_b, oc) == cudaSuccess;
        for (int j = 0; j < 3 && ok; ++j)
            ok = dalloc_copy(d, &bd.a1[j], bw.res_alpha1[j], oc) == cudaSuccess &&
                 dalloc_copy(d, &bd.w1[j], bw.res_w1[j], (size_t)oc * oc * 7) == cudaSuccess &&
                 dalloc_copy(d, &bd.b1[j], bw.res_b1[j], oc) == cudaSuccess &&
                 dalloc_copy(d, &bd.a2[j], bw.res_alpha2[j], oc) == cudaSuccess &&
                 dalloc_copy(d, &bd.w2[j], bw.res_w2[j], (size_t)oc * oc) == cudaSuccess &&
                 dalloc_copy(d, &bd.b2[j], bw.res_b2[j], oc) == cudaSuccess;
    }
    ok = ok && dalloc_copy(d, &d->err, nullptr, 1) == cudaSuccess &&
         cudaMemsetAsync(d->err, 0, sizeof(int), d->st) == cudaSuccess &&
         cudaMallocHost(reinterpret_cast<void**>(&d->h_err), sizeof(int)) == cudaSuccess;
    // the tensor-core path (TTS_BB_DAC=fp32 keeps every convolution on the CUDA-core kernels)
    const char* ev = std::getenv("TTS_BB_DAC");
    d->tc = ok && gemm_tc_available() && !(ev && std::strcmp(ev, "fp32") == 0);
    {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&d->n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || d->n_sm < 1) d->n_sm = 1;
    }
    if (d->tc) {
        bool t = true;
        auto recip = [&](const float* al, int n, float** inv) {  // 1 / (alpha + 1e-9) per channel
            if (t && dalloc_copy(d, inv, nullptr, n) == cudaSuccess) {
                k_dac_recip<<<(n + 255) / 256, 256, 0, d->st>>>(al, n, *inv);
            } else {
                t = false;
            }
        };
        recip(d->final_alpha, 32, &d->final_inv);
        for (int i = 0; i < 5; ++i) {
            recip(d->blk[i].alpha, dac::CH[i], &d->blk[i].alpha_inv);
            for (int j = 0; j < 3; ++j) {
                recip(d->blk[i].a1[j], dac::CH[i + 1], &d->blk[i].a1_inv[j]);
                recip(d->blk[i].a2[j], dac::CH[i + 1], &d->blk[i].a2_inv[j]);
            }
        }
        t = t && tc_prepare(d, d->tc_fc2, d->fc2_w, false, 1024, 256, 1, 1, 0, 1) &&
            tc_prepare(d, d->tc_conv1, d->conv1_w, false, 256, 1024, 7, 1, 3, 1);
        for (int i = 0; i < 5 && t; ++i) {
            const int ic = dac::CH[i], oc = dac::CH[i + 1], r = dac::RATIOS[i];
            t = tc_prepare(d, d->tc_up[i], d->blk[i].up_w, true, ic, oc, 2 * r, 1, 0, r);
            for (int j = 0; j < 3 && t; ++j)
                t = tc_prepare(d, d->tc_r1[i][j], d->blk[i].w1[j], false, oc, oc, 7, dac::DIL[j], 3 * dac::DIL[j], 1) &&
                    tc_prepare(d, d->tc_r2[i][j], d->blk[i].w2[j], false, oc, oc, 1, 1, 0, 1);
        }
        if (!t) ok = false;
    }
    if (!ok || cudaStreamSynchronize(d->st) != cudaSuccess) {
        tts_bb_dac_free(d);
        return TTS_BB_E_OOM;
    }
    *out = d;
    return TTS_BB_OK;
}

TTS_API tts_bb_status tts_bb_dac_decode(tts_bb_dac* d, int B, int T, const float* features, float* audio) {
    if (!d || B < 1 || T < 1 || !features || !audio) return TTS_BB_E_INVALID;
    if (B > 65535 || (size_t)B * T * 960 > (size_t)INT32_MAX) return TTS_BB_E_INVALID;  // grid z = B
    // largest activation: block 4's output, 32 channels x 960 T samples = 30720 T floats per item
    const size_t need = (size_t)B * T * 30720;
    if (need > d->buf_elems) {
        cudaStreamSynchronize(d->st);
        for (int i = 0; i < 3; ++i)
            if (d->buf[i]) {
                cudaFree(d->buf[i]);
                d->allocs.erase(std::remove(d->allocs.begin(), d->allocs.end(), (void*)d->buf[i]), d->allocs.end());
                d->buf[i] = nullptr;
            }
        d->buf_elems = 0;
        for (int i = 0; i < 3; ++i)
            if (dalloc_copy(d, &d->buf[i], nullptr, need) != cudaSuccess) return TTS_BB_E_OOM;
        d->buf_elems = need;
    }
    float *A = d->buf[0], *Bf = d->buf[1], *Cb = d->buf[2];
    if (d->tc) {
        // tensor-core path: X = A holds the fp32 block activation (residual source, time-major
        // [B][T][C]); Sa / Sb (the other two buffers, 2 x 30720 T bf16 per item each) the next
        // convolution's input
        float* X = A;
        bf16* Sa = reinterpret_cast<bf16*>(Bf);
        bf16* Sb = reinterpret_cast<bf16*>(Cb);
        // the features are time-major already: fc2 is a k = 1 convolution over them
        k_dac_split<<<1024, 256, 0, d->st>>>(features, (size_t)B * T * 1024, Sa);
        bool ok = tc_conv(d, d->tc_fc2, Sa, B, T, T, d->fc2_b, nullptr, nullptr, Sb, nullptr, nullptr);
        std::swap(Sa, Sb);
        ok = ok && tc_conv(d, d->tc_conv1, Sa, B, T, T, d->conv1_b, nullptr, nullptr, Sb, d->blk[0].alpha,
                           d->blk[0].alpha_inv);
        std::swap(Sa, Sb);
        int Tc = T;
        for (int i = 0; i < 5 && ok; ++i) {
            const int r = dac::RATIOS[i], To = Tc * r;
            const DacBlockW& bw = d->blk[i];
            ok = tc_conv(d, d->tc_up[i], Sa, B, Tc, To, bw.up_b, nullptr, X, Sb, bw.a1[0], bw.a1_inv[0]);
            std::swap(Sa, Sb);
            for (int j = 0; j < 3 && ok; ++j) {
                ok = tc_conv(d, d->tc_r1[i][j], Sa, B, To, To, bw.b1[j], nullptr, nullptr, Sb, bw.a2[j], bw.a2_inv[j]);
                std::swap(Sa, Sb);
                // the residual unit's output feeds the next unit, the next block's upsampling, or conv2
                // (after the final snake; the block activation itself is not needed after the last unit)
                const bool last = i == 4 && j == 2;
                const float* next_alpha = j < 2 ? bw.a1[j + 1] : (i < 4 ? d->blk[i + 1].alpha : d->final_alpha);
                const float* next_inv = j < 2 ? bw.a1_inv[j + 1] : (i < 4 ? d->blk[i + 1].alpha_inv : d->final_inv);
                ok = ok && tc_conv(d, d->tc_r2[i][j], Sa, B, To, To, bw.b2[j], X, last ? nullptr : X, Sb, next_alpha,
                                   next_inv);
                std::swap(Sa, Sb);
            }
            Tc = To;
        }
        if (!ok) return TTS_BB_E_CUDA;
        k_dac_conv2<<<dim3((Tc + 255) / 256, B), 256, 0, d->st>>>(Sa, d->conv2_w, d->conv2_b, Tc, B, audio);
        return cudaGetLastError() == cudaSuccess ? TTS_BB_OK : TTS_BB_E_CUDA;
    }
    // fc2 on [B][T][1024] (channel stride 1, time stride 1024) -> A [B][256][T]
    conv(d, features, (long)T * 1024, 1, 1024, nullptr, d->fc2_w, d->fc2_b, nullptr, A, B, 1024, 256, T, T, 1, 1, 0);
    conv(d, A, (long)256 * T, T, 1, nullptr, d->conv1_w, d->conv1_b, nullptr, Bf, B, 256, 1024, T, T, 7, 1, 3);
    float *cur = Bf, *nxt = A;
    int Tc = T;
    for (int i = 0; i < 5; ++i) {
        const int ic = dac::CH[i], oc = dac::CH[i + 1], r = dac::RATIOS[i], To = Tc * r;
        const DacBlockW& bw = d->blk[i];
        {
            dim3 grid((To + dac::TO - 1) / dac::TO, (oc + dac::TOC - 1) / dac::TOC, B);
            k_dac_convT<<<grid, dac::NT, 0, d->st>>>(cur, bw.alpha, bw.up_w, bw.up_b, nxt, ic, oc, Tc, To, r, (r + 1) / 2);
            for (int j = 0; j < 3; ++j) {
                const int dl = dac::DIL[j];
                conv(d, nxt, (long)oc * To, To, 1, bw.a1[j], bw.w1[j], bw.b1[j], nullptr, Cb, B, oc, oc, To, To, 7, dl, 3 * dl);
                conv(d, Cb, (long)oc * To, To, 1, bw.a2[j], bw.w2[j], bw.b2[j], nxt, nxt, B, oc, oc, To, To, 1, 1, 0);
            }
        }
        std::swap(cur, nxt);
        Tc = To;
    }
    conv(d, cur, (long)32 * Tc, Tc, 1, d->final_alpha, d->conv2_w, d->conv2_b, nullptr, audio, B, 32, 1, Tc, Tc, 7, 1, 3);
    return cudaGetLastError() == cudaSuccess ? TTS_BB_OK : TTS_BB_E_CUDA;
}

TTS_API tts_bb_status tts_bb_dac_sync(tts_bb_dac* d) {
    if (!d) return TTS_BB_E_INVALID;
    if (cudaMemcpyAsync(d->h_err, d->err, sizeof(int), cudaMemcpyDeviceToHost, d->st) != cudaSuccess ||
        cudaStreamSynchronize(d->st) != cudaSuccess)
        return TTS_BB_E_CUDA;
    const int v = *d->h_err;
    if (v) {
        cudaMemsetAsync(d->err, 0, sizeof(int), d->st);
        cudaStreamSynchronize(d->st);
        return (v & ERR_TIMEOUT) ? TTS_BB_E_DEVICE_TIMEOUT : TTS_BB_E_CUDA;
    }
    return TTS_BB_OK;
}
