// RVQ codec decode: codes -> 1024-d frame features ("omnivoice-cpp
// docs/ARCHITECTURE.md", Audio tokenizer pipeline, Decode, and RVQ codec:
// for each codebook k the frame's code selects a 64-d embedding row, which
// project_out (1024 x 64 weight, 1024 bias) maps to the output, summed over k).
//
// The eight lookups and projections of a frame form one product: the frame's
// gathered rows concatenated along k, X = [e_0 | e_1 | ... | e_7] (K d =
// 512 columns), times W = [W_0 | W_1 | ... | W_7] (1024 x 512, built once
// when the handle is created), plus the summed biases. k_rvq_gather writes X
// (bf16, as stored) and initialises the output rows with the bias sum; the
// tcgen05 GEMM then adds X W^T in fp32.
#include <algorithm>
#include <vector>

#include "common.cuh"
#include "../../include/tts_bb.h"

#define TTS_API extern "C" __attribute__((visibility("default")))

using namespace ttsbb;

struct tts_bb_rvq {
    int K = 0, n = 0, d = 0, out = 0;
    cudaStream_t st = nullptr;
    bf16* embed = nullptr;   // [K][n][d]
    bf16* w = nullptr;       // [out][K d]
    float* bias = nullptr;   // [out], sum over k
    bf16* x = nullptr;       // [frames][K d] gathered rows
    size_t x_frames = 0;
    int* err = nullptr;      // device error word (ERR_BAD_ID)
    int* h_err = nullptr;
    std::vector<void*> allocs;
};

namespace {

// grid frames, 128 threads: row f = (b, t) of X and of the output
__global__ void k_rvq_gather(const int32_t* __restrict__ codes, const bf16* __restrict__ embed,
                             const float* __restrict__ bias, int K, int n, int d, int out_dim, int T,
                             bf16* __restrict__ x, float* __restrict__ out, int* err) {
    pdl_wait();
    pdl_trigger();
    const long f = blockIdx.x;
    const int b = (int)(f / T), t = (int)(f % T);
    for (int i = threadIdx.x; i < K * d; i += blockDim.x) {
        const int k = i / d, c = i - k * d;
        const int code = codes[((size_t)b * K + k) * T + t];
        bf16 v = f2bf(0.f);
        if (code >= 0 && code < n) v = embed[((size_t)k * n + code) * d + c];
        else if (c == 0) set_err(err, ERR_BAD_ID);
        x[f * K * d + i] = v;
    }
    for (int o = threadIdx.x; o < out_dim; o += blockDim.x) out[f * out_dim + o] = bias[o];
}

// W[o][k d + c] = proj_w[k][o][c]; bias[o] = sum_k proj_b[k][o] (in k order)
__global__ void k_rvq_pack(const bf16* __restrict__ wk, const bf16* __restrict__ bk, int k, int K, int d, int out_dim,
                           bf16* __restrict__ w, float* __restrict__ bias) {
    const int o = blockIdx.x;
    for (int c = threadIdx.x; c < d; c += blockDim.x) w[(size_t)o * K * d + k * d + c] = wk[(size_t)o * d + c];
    if (threadIdx.x == 0) bias[o] = (k == 0 ? 0.f : bias[o]) + bf2f(bk[o]);
}

template <typename T>
cudaError_t ralloc(tts_bb_rvq* r, T** p, size_t n) {
    void* v = nullptr;
    const cudaError_t e = cudaMalloc(&v, std::max<size_t>(n, 1) * sizeof(T));
    if (e == cudaSuccess) {
        r->allocs.push_back(v);
        *p = static_cast<T*>(v);
    }
    return e;
}

}  // namespace

TTS_API void tts_bb_rvq_free(tts_bb_rvq* r) {
    if (!r) return;
    cudaStreamSynchronize(r->st);
    for (void* p : r->allocs) cudaFree(p);
    if (r->h_err) cudaFreeHost(r->h_err);
    delete r;
}

TTS_API tts_bb_status tts_bb_rvq_create(int n_codebooks, int codebook_size, int dim, int out_dim,
                                        const void* const* embed, const void* const* proj_w,
                                        const void* const* proj_b, void* stream, tts_bb_rvq** out) {
    if (!out) return TTS_BB_E_INVALID;
    *out = nullptr;
    if (n_codebooks < 1 || n_codebooks > 64 || codebook_size < 1 || dim < 8 || dim % 8 || out_dim < 1 ||
        (n_codebooks * dim) % 64 || !embed || !proj_w || !proj_b)
        return TTS_BB_E_INVALID;
    for (int k = 0; k < n_codebooks; ++k)
        if (!embed[k] || !proj_w[k] || !proj_b[k]) return TTS_BB_E_INVALID;
    tts_bb_rvq* r = new tts_bb_rvq();
    r->K = n_codebooks;
    r->n = codebook_size;
    r->d = dim;
    r->out = out_dim;
    r->st = static_cast<cudaStream_t>(stream);
    auto bail = [&](tts_bb_status s) {
        tts_bb_rvq_free(r);
        return s;
    };
    if (ralloc(r, &r->embed, (size_t)n_codebooks * codebook_size * dim) != cudaSuccess ||
        ralloc(r, &r->w, (size_t)out_dim * n_codebooks * dim) != cudaSuccess ||
        ralloc(r, &r->bias, (size_t)out_dim) != cudaSuccess || ralloc(r, &r->err, 1) != cudaSuccess ||
        cudaMallocHost(&r->h_err, sizeof(int)) != cudaSuccess)
        return bail(TTS_BB_E_OOM);
    for (int k = 0; k < n_codebooks; ++k) {
        if (cudaMemcpyAsync(r->embed + (size_t)k * codebook_size * dim, embed[k],
                            (size_t)codebook_size * dim * sizeof(bf16), cudaMemcpyDefault, r->st) != cudaSuccess)
            return bail(TTS_BB_E_CUDA);
        k_rvq_pack<<<out_dim, 64, 0, r->st>>>(static_cast<const bf16*>(proj_w[k]), static_cast<const bf16*>(proj_b[k]),
                                               k, n_codebooks, dim, out_dim, r->w, r->bias);
    }
    cudaMemsetAsync(r->err, 0, sizeof(int), r->st);
    if (cudaStreamSynchronize(r->st) != cudaSuccess || cudaGetLastError() != cudaSuccess) return bail(TTS_BB_E_CUDA);
    if (!gemm_tc_available()) return bail(TTS_BB_E_UNSUPPORTED);
    *out = r;
    return TTS_BB_OK;
}

TTS_API tts_bb_status tts_bb_rvq_decode(tts_bb_rvq* r, int B, int T, const int32_t* codes, float* out) {
    if (!r || B < 1 || T < 1 || !codes || !out) return TTS_BB_E_INVALID;
    const size_t frames = (size_t)B * T;
    if (frames > (size_t)INT32_MAX / 2) return TTS_BB_E_INVALID;
    if (frames > r->x_frames) {
        cudaStreamSynchronize(r->st);
        if (r->x) {
            cudaFree(r->x);
            r->allocs.erase(std::remove(r->allocs.begin(), r->allocs.end(), (void*)r->x), r->allocs.end());
            r->x = nullptr;
            r->x_frames = 0;
        }
        if (ralloc(r, &r->x, frames * r->K * r->d) != cudaSuccess) return TTS_BB_E_OOM;
        r->x_frames = frames;
    }
    launch_pdl(k_rvq_gather, (unsigned)frames, 128, 0, r->st, codes, (const bf16*)r->embed, (const float*)r->bias,
               r->K, r->n, r->d, r->out, T, r->x, out, r->err);
    Epi e{};
    e.mode = EPI_ADD_F32;
    e.out = out;
    e.ldo = r->out;
    if (!launch_gemm(r->x, r->w, (int)frames, r->out, r->K * r->d, e, r->st, nullptr, r->err))
        return TTS_BB_E_UNSUPPORTED;
    return cudaGetLastError() == cudaSuccess ? TTS_BB_OK : TTS_BB_E_CUDA;
}

TTS_API tts_bb_status tts_bb_rvq_sync(tts_bb_rvq* r) {
    if (!r) return TTS_BB_E_INVALID;
    if (cudaMemcpyAsync(r->h_err, r->err, sizeof(int), cudaMemcpyDeviceToHost, r->st) != cudaSuccess ||
        cudaStreamSynchronize(r->st) != cudaSuccess)
        return TTS_BB_E_CUDA;
    const int v = *r->h_err;
    if (v) {
        cudaMemsetAsync(r->err, 0, sizeof(int), r->st);
        cudaStreamSynchronize(r->st);
        if (v & ERR_BAD_ID) return TTS_BB_E_BAD_ID;
        return TTS_BB_E_CUDA;
    }
    return TTS_BB_OK;
}
