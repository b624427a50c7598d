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
#include <vector>

#include "common.cuh"
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
};

struct tts_bb_dac {
    cudaStream_t st = nullptr;
    float *fc2_w = nullptr, *fc2_b = nullptr, *conv1_w = nullptr, *conv1_b = nullptr;
    DacBlockW blk[5] = {};
    float *final_alpha = nullptr, *conv2_w = nullptr, *conv2_b = nullptr;
    float *buf[3] = {nullptr, nullptr, nullptr};
    size_t buf_elems = 0;
    std::vector<void*> allocs;
};

namespace {

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
    // fc2 on [B][T][1024] (channel stride 1, time stride 1024) -> A [B][256][T]
    conv(d, features, (long)T * 1024, 1, 1024, nullptr, d->fc2_w, d->fc2_b, nullptr, A, B, 1024, 256, T, T, 1, 1, 0);
    conv(d, A, (long)256 * T, T, 1, nullptr, d->conv1_w, d->conv1_b, nullptr, Bf, B, 256, 1024, T, T, 7, 1, 3);
    float *cur = Bf, *nxt = A;
    int Tc = T;
    for (int i = 0; i < 5; ++i) {
        const int ic = dac::CH[i], oc = dac::CH[i + 1], r = dac::RATIOS[i], To = Tc * r;
        const DacBlockW& bw = d->blk[i];
        dim3 grid((To + dac::TO - 1) / dac::TO, (oc + dac::TOC - 1) / dac::TOC, B);
        k_dac_convT<<<grid, dac::NT, 0, d->st>>>(cur, bw.alpha, bw.up_w, bw.up_b, nxt, ic, oc, Tc, To, r, (r + 1) / 2);
        for (int j = 0; j < 3; ++j) {
            const int dl = dac::DIL[j];
            conv(d, nxt, (long)oc * To, To, 1, bw.a1[j], bw.w1[j], bw.b1[j], nullptr, Cb, B, oc, oc, To, To, 7, dl, 3 * dl);
            conv(d, Cb, (long)oc * To, To, 1, bw.a2[j], bw.w2[j], bw.b2[j], nxt, nxt, B, oc, oc, To, To, 1, 1, 0);
        }
        std::swap(cur, nxt);
        Tc = To;
    }
    conv(d, cur, (long)32 * Tc, Tc, 1, d->final_alpha, d->conv2_w, d->conv2_b, nullptr, audio, B, 32, 1, Tc, Tc, 7, 1, 3);
    return cudaGetLastError() == cudaSuccess ? TTS_BB_OK : TTS_BB_E_CUDA;
}
