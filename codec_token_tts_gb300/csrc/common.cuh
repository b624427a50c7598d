// Shared device helpers and kernel launch declarations of the tts_bb engine.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace ttsbb {

typedef __nv_bfloat16 bf16;

constexpr int HID = 1024;      // hidden size
constexpr int HD = 128;        // head dim
constexpr int NQ = 16;         // query heads
constexpr int NKV = 8;         // kv heads
constexpr int QKV = (NQ + 2 * NKV) * HD;  // 4096 fused projection rows
constexpr int KVB = 64;        // tokens per KV block

// Device error word bits.
enum : int { ERR_BAD_ID = 1, ERR_TIMEOUT = 2, ERR_KV_RANGE = 4, ERR_LAYOUT = 8 };

__device__ __forceinline__ void set_err(int* err, int bit) {
    if (err) atomicOr(err, bit);
}

__device__ __forceinline__ float bf2f(bf16 x) { return __bfloat162float(x); }
__device__ __forceinline__ bf16 f2bf(float x) { return __float2bfloat16_rn(x); }
// Low bf16 part of a value whose high part is f2bf(x): hi + lo carries ~16 mantissa bits.
__device__ __forceinline__ bf16 f2bf_lo(float x) { return __float2bfloat16_rn(x - __bfloat162float(__float2bfloat16_rn(x))); }

// 8 bf16 packed in a uint4 -> 8 floats
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Argmax packing: (order-preserving float bits << 32) | (~index), so a 64-bit
// max picks the largest value and, among equal values, the lowest index.
__device__ __forceinline__ unsigned long long pack_argmax(float v, int idx) {
    uint32_t u = __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

// ---------------------------------------------------------------- epilogues
enum EpiMode : int {
    EPI_STORE_F32 = 0,   // out_f32[t*ldo + n] = acc
    EPI_STORE_BF16 = 1,  // out_bf16[t*ldo + n] = acc
    EPI_ADD_F32 = 2,     // out_f32[t*ldo + n] += acc (residual)
    EPI_SWIGLU = 3,      // rows interleaved gate/up: out_bf16[t*ldo + n/2] = silu(g)*u
    EPI_LOGITS = 4,      // out_f32 (optional) + packed argmax per row (optional)
    EPI_LOGITS_PERM = 5, // OmniVoice audio heads: out[((b*G + k)*R + s)*V + v]
    EPI_QKROPE = 6       // the QKV product: q/k RMSNorm + RoPE, q out, k and v appended (decode GEMM only)
};

// Paged KV cache of one layer. Block of (seq, j): page_table[seq_slot[seq]*mbps + j] or, when
// page_table is null, seq*mbps + j.
struct KVView {
    bf16* pool;            // layer base: [blocks][2][8][64][128]
    const int32_t* page_table;
    const int32_t* seq_slot;
    int mbps;              // blocks per slot row of the page table
};

// EPI_QKROPE arguments: token t belongs to sequence t / tok_per_seq at position seq_start[seq] +
// t % tok_per_seq, valid when t % tok_per_seq < seq_len[seq]; q -> q (bf16) or qf (fp32, when
// non-null) [T][16][128], k and v -> the paged cache kv.
struct EpiQk {
    const bf16* qn;
    const bf16* kn;
    const float* cos_t;
    const float* sin_t;
    float eps;
    bf16* q;
    float* qf;
    KVView kv;
    const int32_t* seq_start;
    const int32_t* seq_len;
    int tok_per_seq;
    int* err;
};

struct Epi {
    int mode;
    void* out;
    int ldo;
    unsigned long long* amax;  // EPI_LOGITS: [T] packed argmax
    int perm_rows;             // EPI_LOGITS_PERM: rows per batch (R)
    int perm_vocab;            // V
    int perm_groups;           // G
    void* out_lo;              // EPI_SWIGLU: optional bf16 low part (value - bf16(value))
    EpiQk qk;                  // EPI_QKROPE
    // RMSNorm folded into the decode GEMM (split-K kernel only). Producer (EPI_ADD_F32): besides h,
    // write the next norm's input h * gamma as bf16 high + low parts (nrm_y, nrm_ylo, [T][1024]) and
    // this 128-feature tile's sum of squares of h per token (nrm_ss[tile][T]). Consumer: scale each
    // token row of the product by rsqrt(sum over the 8 tiles of nrm_scale_ss[tile][T] / 1024 + eps).
    const bf16* nrm_gamma;
    bf16* nrm_y;
    bf16* nrm_ylo;
    float* nrm_ss;
    const float* nrm_scale_ss;
    float nrm_eps;
    int nrm_T;
};

// ---------------------------------------------------------------- programmatic dependent launch
// Kernels of the step chain are launched with programmatic stream
// serialization: a kernel may be dispatched while its predecessor finishes,
// runs only setup that reads no upstream results, then waits in pdl_wait()
// until the predecessor has completed and its writes are visible. pdl_trigger()
// lets the next kernel of the chain be dispatched early (it launches only once
// every CTA of this grid is running). Both are no-ops without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- kernels
struct TableSet {
    const bf16* tab[16];
    int rows[16];
    int n;
};

// h[t] = embeds[t] (optional) + sum_k E_k[ids[t][k]] (ids[t][k] == -1 skipped)
int launch_embed_codebooks(const TableSet& ts, const int32_t* ids, const bf16* embeds,
                            float* h, int T, int* err, cudaStream_t st);
// OmniVoice hybrid embedding; tokens t = b*S + s
int launch_embed_omnivoice(const bf16* text, int text_vocab, const bf16* audio, int n_cb, int vocab,
                            const int32_t* ids, const uint8_t* mask, float* h, int B, int S, int* err,
                            cudaStream_t st);
// y[t] = bf16(rmsnorm(h[src(t)]) * gamma); src(t) = (t / per) * stride + offset + t % per,
// or, when last_len != nullptr, src(t) = t * stride + last_len[t] - 1. y_lo (optional) gets the
// low bf16 parts, value - bf16(value).
int launch_rmsnorm(const float* h, const bf16* gamma, bf16* y, int T, float eps, int per, int stride,
                    int offset, const int32_t* last_len, cudaStream_t st, bf16* y_lo = nullptr);
// Y = X W^T with epilogue; X [T][K] bf16, W [N][K] bf16. T small (<= 8).
// X_lo (optional): low bf16 parts of the activations; the products use X + X_lo.
int launch_gemv(const bf16* X, const bf16* W, int T, int N, int K, const Epi& e, cudaStream_t st,
                const bf16* X_lo = nullptr);
// Y = X W^T with epilogue, tensor cores, any T.
// Split-K workspace for the small-batch GEMM: fp32 partial tiles and one
// arrival counter per 64-feature tile (zero between launches).
struct SplitK {
    float* part;
    size_t part_elems;
    int* ctr;
    int n_ctr;
};
// T <= 8: the matrix-vector kernel. Split activations (X_lo): the swap-AB cluster split-K tcgen05
// kernel (k_gemm_tc.cu) for up to two 128-token blocks, and for three or four when one launch of
// them fits one wave (gemm_tcd_takes); beyond that the dense persistent tcgen05 kernel with two
// passes over K. Plain bf16 activations with T > 8: the dense tcgen05 kernel. Without tcgen05
// the mma.sync kernels (split-K with a workspace, else tiled with a second MMA per k-step).
// Fused epilogues (q/k norm + RoPE + append, folded norms) run on the split-K tcgen05 kernel only.
int launch_gemm(const bf16* X, const bf16* W, int T, int N, int K, const Epi& e, cudaStream_t st,
                const bf16* X_lo = nullptr, int* err = nullptr, const SplitK* sk = nullptr);
// Dense persistent tcgen05 GEMM; with X_lo the activations are bf16 high + low parts (two passes over K).
int launch_gemm_tc(const bf16* X, const bf16* W, int T, int N, int K, const Epi& e, int* err, cudaStream_t st,
                   const bf16* X_lo = nullptr);
int launch_gemm_tcd(const bf16* X, const bf16* X_lo, const bf16* W, int T, int N, int K, const Epi& e, int* err,
                    cudaStream_t st);
// Whether launch_gemm_tcd takes a [T x K] x [N x K]^T product (up to four 128-token blocks).
bool gemm_tcd_takes(int T, int N, int K);
bool gemm_tc_available();
// MaskGIT greedy update (k_maskgit.cu): two launches
int launch_maskgit_update(const float* logits, int n_items, int K, int T, int V, int S_log, int cond_pos0,
                          int uncond_pos0, int32_t* ids, int S_ids, int cond_ids_pos0, int uncond_ids_pos0,
                          int mask_id, float cfg, float penalty, int n_unmask, unsigned long long* keys, int32_t* pred,
                          cudaStream_t st);
int mg_max_vocab();
int launch_attn_bidir_tc(const bf16* q, const bf16* pool, size_t pool_blocks, int bps, const int32_t* key_len, int B,
                         int S, bf16* out, int* err, cudaStream_t st);

// Per-token q/k RMSNorm + RoPE; q -> qout [T][16][128] bf16; k, v -> paged pool.
// Token t belongs to sequence t / tok_per_seq at position seq_start[seq] + t % tok_per_seq,
// valid when t % tok_per_seq < seq_len[seq].
// qout_f (optional): the queries as fp32 [T][16][128] instead of bf16 in qout. qkv_bf (optional):
// the QKV rows as bf16 [T][4096], read instead of the fp32 qkv.
int launch_qk_norm_rope_append(const float* qkv, const bf16* qn, const bf16* kn, const float* cos_t,
                                const float* sin_t, float eps, bf16* qout, KVView kv, const int32_t* seq_start,
                                const int32_t* seq_len, int tok_per_seq, int T, int* err, cudaStream_t st,
                                float* qout_f = nullptr, const bf16* qkv_bf = nullptr);
// Decode attention, one query per sequence: split-K flash decode + combine; for max_len <=
// ATTN_SHORT_CTX one warp per (query, KV head) over the whole context, no combine.
// qf (optional): fp32 queries [B][16][128], read instead of the bf16 q.
// tps > 1: B = sequences x tps queries of a short causal prefill (query b is token b % tps of
// sequence b / tps, seq_len gives each sequence's valid tokens).
constexpr int ATTN_SHORT_CTX = 32;
int launch_attn_decode(const bf16* q, KVView kv, const int32_t* seq_start, int B, int max_len,
                        float* part, bf16* out, int max_splits, cudaStream_t st, bf16* out_lo = nullptr,
                        const float* qf = nullptr, int tps = 1, const int32_t* seq_len = nullptr);
// Prefill / bidirectional attention over the paged view, tensor cores.
// causal: query at position p sees keys <= p; else keys < key_len[seq].
// out_lo (optional): low bf16 parts of the output, value - bf16(value).
int launch_attn_prefill(const bf16* q, KVView kv, const int32_t* seq_start, const int32_t* seq_len,
                         const int32_t* key_len, int causal, int B, int S, bf16* out, cudaStream_t st,
                         bf16* out_lo = nullptr);
// Causal prefill attention on tcgen05 over one layer's paged pool (pool_blocks blocks): query s of
// sequence b at position seq_start[b] + s sees keys 0 .. that position; out_lo (optional) low parts.
// With fp32 queries qf (non-null) Q and P enter the products as bf16 high + low parts; else bf16 q.
int launch_attn_causal_tc(const bf16* q, const float* qf, KVView kv, size_t pool_blocks, const int32_t* seq_start,
                          int B, int S, bf16* out, bf16* out_lo, int* err, cudaStream_t st);
// out[b * stride] = unpacked argmax
int launch_argmax_finalize(const unsigned long long* amax, int32_t* out, int stride, int B, cudaStream_t st);

}  // namespace ttsbb
