// Qwen3-TTS codec quantizer lookup: codes -> the [B][512][T] float hidden of
// the codec body ("Qwen3-TTS ncnn port", Codec Decoder split, steps 1-4: the
// 16 codebooks and two projection weights are read, each frame looks up one
// row per codebook, the first (semantic) codebook and the other 15
// (acoustic) codebooks are projected separately and summed).
//
// A frame's result is one product: with s = C_0[code_0] (the semantic row)
// and a = sum_{k>=1} C_k[code_k] (the acoustic rows summed in fp32), the
// output is P_sem s + P_ac a. k_quant_gather writes the row
// X = [s | a_hi | a_lo] (bf16; a = a_hi + a_lo to ~16 mantissa bits, s is
// exact), and the packed weight W = [P_sem | P_ac | P_ac] (out x 3d, built
// once at create) turns that into one bf16 GEMM with fp32 accumulation,
// whose permuted epilogue stores channel-major out[b][o][t] directly. The
// packed width kp is 3d rounded up to 256 columns (the GEMM kernels' k-step
// granularity); the extra columns are zero in both operands.
#include <algorithm>
#include <new>
#include <vector>

#include "common.cuh"
#include "../../include/tts_bb.h"

#define TTS_API extern "C" __attribute__((visibility("default")))

using namespace ttsbb;

struct tts_bb_quantizer {
    int K = 0, n = 0, d = 0, out = 0, kp = 0;
    cudaStream_t st = nullptr;
    bf16* books = nullptr;   // [K][n][d]
    bf16* w = nullptr;       // [out][kp] = [P_sem | P_ac | P_ac | 0]
    bf16* x = nullptr;       // [frames][kp] gathered rows
    size_t x_frames = 0;
    int* err = nullptr;      // device error word (ERR_BAD_ID)
    int* h_err = nullptr;
    std::vector<void*> allocs;
};

namespace {

constexpr int QG_WARPS = 8;  // frames per CTA of the gather (one warp each)

// One warp per frame f = (b, t): lanes take 8-column chunks of the d columns.
// Codes outside 0..n-1 contribute a zero row and raise ERR_BAD_ID.
__global__ void __launch_bounds__(QG_WARPS * 32) k_quant_gather(const int32_t* __restrict__ codes,
                                                                const bf16* __restrict__ books, int K, int n, int d,
                                                                int T, long frames, int kp, bf16* __restrict__ x,
                                                                int* err) {
    pdl_wait();
    pdl_trigger();
    __shared__ int s_code[QG_WARPS][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long f = (long)blockIdx.x * QG_WARPS + warp;
    if (f >= frames) return;  // whole warps leave together
    const int b = (int)(f / T), t = (int)(f % T);
    int my = lane < K ? codes[((size_t)b * K + lane) * T + t] : 0;
    const bool bad = lane < K && (my < 0 || my >= n);
    if (bad) my = -1;
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_err(err, ERR_BAD_ID);
    s_code[warp][lane] = my;
    __syncwarp();
    bf16* xr = x + (size_t)f * kp;
    for (int c = 3 * d + lane * 8; c < kp; c += 32 * 8) *reinterpret_cast<uint4*>(xr + c) = make_uint4(0u, 0u, 0u, 0u);
    for (int c = lane * 8; c < d; c += 32 * 8) {
        const int c0 = s_code[warp][0];
        uint4 s = make_uint4(0u, 0u, 0u, 0u);
        if (c0 >= 0) s = *reinterpret_cast<const uint4*>(books + (size_t)c0 * d + c);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int k = 1; k < K; ++k) {
            const int ck = s_code[warp][k];
            if (ck < 0) continue;
            float v[8];
            unpack8(*reinterpret_cast<const uint4*>(books + ((size_t)k * n + ck) * d + c), v);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] += v[e];
        }
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
            const float2 hf = __bfloat1622float2(h2);
            const __nv_bfloat162 l2 = __floats2bfloat162_rn(acc[2 * e] - hf.x, acc[2 * e + 1] - hf.y);
            hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
            lo[e] = *reinterpret_cast<const uint32_t*>(&l2);
        }
        *reinterpret_cast<uint4*>(xr + c) = s;
        *reinterpret_cast<uint4*>(xr + d + c) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(xr + 2 * d + c) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// W[o][0:d) = P_sem[o], W[o][d:2d) = W[o][2d:3d) = P_ac[o], W[o][3d:kp) = 0
__global__ void k_quant_pack(const bf16* __restrict__ ps, const bf16* __restrict__ pa, int d, int kp,
                             bf16* __restrict__ w) {
    const int o = blockIdx.x;
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        const bf16 a = pa[(size_t)o * d + c];
        w[(size_t)o * kp + c] = ps[(size_t)o * d + c];
        w[(size_t)o * kp + d + c] = a;
        w[(size_t)o * kp + 2 * d + c] = a;
    }
    for (int c = 3 * d + threadIdx.x; c < kp; c += blockDim.x) w[(size_t)o * kp + c] = f2bf(0.f);
}

template <typename T>
cudaError_t qalloc(tts_bb_quantizer* q, T** p, size_t n) {
    void* v = nullptr;
    const cudaError_t e = cudaMalloc(&v, std::max<size_t>(n, 1) * sizeof(T));
    if (e == cudaSuccess) {
        q->allocs.push_back(v);
        *p = static_cast<T*>(v);
    }
    return e;
}

}  // namespace

TTS_API void tts_bb_quantizer_free(tts_bb_quantizer* q) {
    if (!q) return;
    cudaStreamSynchronize(q->st);
    for (void* p : q->allocs) cudaFree(p);
    if (q->h_err) cudaFreeHost(q->h_err);
    delete q;
}

TTS_API tts_bb_status tts_bb_quantizer_create(int n_codebooks, int codebook_size, int dim, int out_dim,
                                              const void* const* codebooks, const void* proj_semantic,
                                              const void* proj_acoustic, void* stream, tts_bb_quantizer** out) {
    if (!out) return TTS_BB_E_INVALID;
    *out = nullptr;
    if (n_codebooks < 2 || n_codebooks > 32 || codebook_size < 1 || dim < 64 || dim > 1024 || dim % 64 ||
        out_dim < 1 || out_dim > 8192 || !codebooks || !proj_semantic || !proj_acoustic)
        return TTS_BB_E_INVALID;
    if ((long long)n_codebooks * codebook_size * dim > (1ll << 34)) return TTS_BB_E_INVALID;
    for (int k = 0; k < n_codebooks; ++k)
        if (!codebooks[k]) return TTS_BB_E_INVALID;
    tts_bb_quantizer* q = new (std::nothrow) tts_bb_quantizer();
    if (!q) return TTS_BB_E_OOM;
    q->K = n_codebooks;
    q->n = codebook_size;
    q->d = dim;
    q->out = out_dim;
    q->kp = (3 * dim + 255) / 256 * 256;
    q->st = static_cast<cudaStream_t>(stream);
    auto bail = [&](tts_bb_status s) {
        tts_bb_quantizer_free(q);
        return s;
    };
    bf16 *ps = nullptr, *pa = nullptr;
    if (qalloc(q, &q->books, (size_t)n_codebooks * codebook_size * dim) != cudaSuccess ||
        qalloc(q, &q->w, (size_t)out_dim * q->kp) != cudaSuccess || qalloc(q, &ps, (size_t)out_dim * dim) != cudaSuccess ||
        qalloc(q, &pa, (size_t)out_dim * dim) != cudaSuccess || qalloc(q, &q->err, 1) != cudaSuccess ||
        cudaMallocHost(&q->h_err, sizeof(int)) != cudaSuccess)
        return bail(TTS_BB_E_OOM);
    const size_t book = (size_t)codebook_size * dim * sizeof(bf16), proj = (size_t)out_dim * dim * sizeof(bf16);
    for (int k = 0; k < n_codebooks; ++k)
        if (cudaMemcpyAsync(q->books + (size_t)k * codebook_size * dim, codebooks[k], book, cudaMemcpyDefault, q->st) !=
            cudaSuccess)
            return bail(TTS_BB_E_CUDA);
    if (cudaMemcpyAsync(ps, proj_semantic, proj, cudaMemcpyDefault, q->st) != cudaSuccess ||
        cudaMemcpyAsync(pa, proj_acoustic, proj, cudaMemcpyDefault, q->st) != cudaSuccess)
        return bail(TTS_BB_E_CUDA);
    k_quant_pack<<<out_dim, 128, 0, q->st>>>(ps, pa, dim, q->kp, q->w);
    cudaMemsetAsync(q->err, 0, sizeof(int), q->st);
    if (cudaStreamSynchronize(q->st) != cudaSuccess || cudaGetLastError() != cudaSuccess) return bail(TTS_BB_E_CUDA);
    for (bf16* p : {ps, pa}) {  // the unpacked copies are no longer needed
        cudaFree(p);
        q->allocs.erase(std::remove(q->allocs.begin(), q->allocs.end(), (void*)p), q->allocs.end());
    }
    *out = q;
    return TTS_BB_OK;
}

TTS_API tts_bb_status tts_bb_quantizer_decode(tts_bb_quantizer* q, int B, int T, const int32_t* codes, float* out) {
    if (!q || B < 1 || T < 1 || !codes || !out) return TTS_BB_E_INVALID;
    const size_t frames = (size_t)B * T;
    if (frames > (size_t)INT32_MAX / 4) return TTS_BB_E_INVALID;
    if (frames > q->x_frames) {
        cudaStreamSynchronize(q->st);
        if (q->x) {
            cudaFree(q->x);
            q->allocs.erase(std::remove(q->allocs.begin(), q->allocs.end(), (void*)q->x), q->allocs.end());
            q->x = nullptr;
            q->x_frames = 0;
        }
        if (qalloc(q, &q->x, frames * q->kp) != cudaSuccess) return TTS_BB_E_OOM;
        q->x_frames = frames;
    }
    launch_pdl(k_quant_gather, (unsigned)((frames + QG_WARPS - 1) / QG_WARPS), QG_WARPS * 32, 0, q->st, codes,
               (const bf16*)q->books, q->K, q->n, q->d, T, (long)frames, q->kp, q->x, q->err);
    // out[b][o][t]: the permuted epilogue with groups = channels and one value per group
    Epi e{};
    e.mode = EPI_LOGITS_PERM;
    e.out = out;
    e.perm_rows = T;
    e.perm_vocab = 1;
    e.perm_groups = q->out;
    if (!launch_gemm(q->x, q->w, (int)frames, q->out, q->kp, e, q->st, nullptr, q->err)) return TTS_BB_E_UNSUPPORTED;
    return cudaGetLastError() == cudaSuccess ? TTS_BB_OK : TTS_BB_E_CUDA;
}

TTS_API tts_bb_status tts_bb_quantizer_sync(tts_bb_quantizer* q) {
    if (!q) return TTS_BB_E_INVALID;
    if (cudaMemcpyAsync(q->h_err, q->err, sizeof(int), cudaMemcpyDeviceToHost, q->st) != cudaSuccess ||
        cudaStreamSynchronize(q->st) != cudaSuccess)
        return TTS_BB_E_CUDA;
    const int v = *q->h_err;
    if (v) {
        cudaMemsetAsync(q->err, 0, sizeof(int), q->st);
        cudaStreamSynchronize(q->st);
        if (v & ERR_BAD_ID) return TTS_BB_E_BAD_ID;
        return TTS_BB_E_CUDA;
    }
    return TTS_BB_OK;
}
