// Row-wise kernels of the backbone step: codebook gather-sum, OmniVoice hybrid
// embedding, RMSNorm, per-head q/k RMSNorm + half-rotate RoPE + paged KV
// append, argmax unpacking.
#include "common.cuh"

namespace ttsbb {

// ---------------------------------------------------------------- a1 gather-sum
// Sum of codebook embeddings into the fp32 residual (Qwen3-TTS ncnn port, model
// structure: the 16 embeddings of a frame are added to form the next input).
// One CTA per token, 128 threads x 8 elements. Out-of-table ids are skipped
// and flagged; -1 means "no token from this codebook".
__global__ void __launch_bounds__(128) k_embed_codebooks(TableSet ts, const int32_t* __restrict__ ids,
                                                         const bf16* __restrict__ embeds,
                                                         float* __restrict__ h, int* err) {
    pdl_wait();  // upstream results are read below
    pdl_trigger();
    const int t = blockIdx.x;
    const int c = threadIdx.x * 8;
    float acc[8];
    if (embeds) {
        unpack8(*reinterpret_cast<const uint4*>(embeds + (size_t)t * HID + c), acc);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    }
    if (ids) {
        for (int k = 0; k < ts.n; ++k) {
            const int id = __ldg(ids + (size_t)t * ts.n + k);
            if (id == -1) continue;
            if (id < -1 || id >= ts.rows[k]) {
                if (threadIdx.x == 0) set_err(err, ERR_BAD_ID);
                continue;
            }
            float f[8];
            unpack8(ldg_nc_v4(ts.tab[k] + (size_t)id * HID + c), f);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += f[i];
        }
    }
    float4* o = reinterpret_cast<float4*>(h + (size_t)t * HID + c);
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

int launch_embed_codebooks(const TableSet& ts, const int32_t* ids, const bf16* embeds, float* h, int T,
                            int* err, cudaStream_t st) {
    if (T <= 0) return 0;
    launch_pdl(k_embed_codebooks, T, 128, 0, st, ts, ids, embeds, h, err);
    return 1;
}

// OmniVoice hybrid embedding (omnivoice-cpp ARCHITECTURE.md, Component
// architecture): audio positions take sum_k audio[id_k + vocab*k], text
// positions take text[id_0]. ids [B][n_cb][S].
__global__ void __launch_bounds__(128) k_embed_omnivoice(const bf16* __restrict__ text, int text_vocab,
                                                         const bf16* __restrict__ audio, int n_cb, int vocab,
                                                         const int32_t* __restrict__ ids,
                                                         const uint8_t* __restrict__ mask,
                                                         float* __restrict__ h, int S, int* err) {
    pdl_wait();  // upstream results are read below
    pdl_trigger();
    const int t = blockIdx.x;
    const int b = t / S, s = t % S;
    const int c = threadIdx.x * 8;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    if (mask[t]) {
        for (int k = 0; k < n_cb; ++k) {
            const int id = __ldg(ids + ((size_t)b * n_cb + k) * S + s);
            if (id < 0 || id >= vocab) {
                if (threadIdx.x == 0) set_err(err, ERR_BAD_ID);
                continue;
            }
            float f[8];
            unpack8(ldg_nc_v4(audio + ((size_t)id + (size_t)vocab * k) * HID + c), f);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += f[i];
        }
    } else {
        const int id = __ldg(ids + (size_t)b * n_cb * S + s);
        if (id < 0 || id >= text_vocab) {
            if (threadIdx.x == 0) set_err(err, ERR_BAD_ID);
        } else {
            unpack8(ldg_nc_v4(text + (size_t)id * HID + c), acc);
        }
    }
    float4* o = reinterpret_cast<float4*>(h + (size_t)t * HID + c);
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

int launch_embed_omnivoice(const bf16* text, int text_vocab, const bf16* audio, int n_cb, int vocab,
                            const int32_t* ids, const uint8_t* mask, float* h, int B, int S, int* err,
                            cudaStream_t st) {
    if (B * S <= 0) return 0;
    launch_pdl(k_embed_omnivoice, B * S, 128, 0, st, text, text_vocab, audio, n_cb, vocab, ids, mask, h, S, err);
    return 1;
}

// ---------------------------------------------------------------- a2/a7/a10 RMSNorm
// y = h * rsqrt(mean(h^2) + eps) * gamma; fp32 residual in, bf16 out. One warp per row.
__global__ void __launch_bounds__(256) k_rmsnorm(const float* __restrict__ h, const bf16* __restrict__ gamma,
                                                 bf16* __restrict__ y, int T, float eps, int per, int stride,
                                                 int offset, const int32_t* __restrict__ last_len,
                                                 bf16* __restrict__ y_lo) {
    pdl_wait();  // upstream results are read below
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    size_t src;
    if (last_len) src = (size_t)t * stride + last_len[t] - 1;
    else src = (size_t)(t / per) * stride + offset + (t % per);
    const float4* row = reinterpret_cast<const float4*>(h + src * HID);
    float4 v[8];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[i] = row[i * 32 + lane];
        ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
    }
    ss = warp_sum(ss);
    const float r = rsqrtf(ss * (1.f / HID) + eps);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = (i * 32 + lane) * 4;
        const uint2 gr = *reinterpret_cast<const uint2*>(gamma + e);
        const float g0 = __uint_as_float(gr.x << 16), g1 = __uint_as_float(gr.x & 0xFFFF0000u);
        const float g2 = __uint_as_float(gr.y << 16), g3 = __uint_as_float(gr.y & 0xFFFF0000u);
        const float f0 = v[i].x * r * g0, f1 = v[i].y * r * g1, f2 = v[i].z * r * g2, f3 = v[i].w * r * g3;
        __nv_bfloat162 a = __floats2bfloat162_rn(f0, f1);
        __nv_bfloat162 b = __floats2bfloat162_rn(f2, f3);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t*>(&a);
        o.y = *reinterpret_cast<uint32_t*>(&b);
        *reinterpret_cast<uint2*>(y + (size_t)t * HID + e) = o;
        if (y_lo) {
            __nv_bfloat162 al = __halves2bfloat162(f2bf_lo(f0), f2bf_lo(f1));
            __nv_bfloat162 bl = __halves2bfloat162(f2bf_lo(f2), f2bf_lo(f3));
            o.x = *reinterpret_cast<uint32_t*>(&al);
            o.y = *reinterpret_cast<uint32_t*>(&bl);
            *reinterpret_cast<uint2*>(y_lo + (size_t)t * HID + e) = o;
        }
    }
}

int launch_rmsnorm(const float* h, const bf16* gamma, bf16* y, int T, float eps, int per, int stride, int offset,
                    const int32_t* last_len, cudaStream_t st, bf16* y_lo) {
    if (T <= 0) return 0;
    launch_pdl(k_rmsnorm, (T + 7) / 8, 256, 0, st, h, gamma, y, T, eps, per, stride, offset, last_len, y_lo);
    return 1;
}

// ---------------------------------------------------------------- a4 q/k norm + RoPE + KV append
// Per token: 16 q heads, 8 k heads, 8 v heads = 32 units over 8 warps. Lane l
// holds head elements 4l..4l+3; the RoPE partner of element i (< 64) is i + 64,
// held by lane l ^ 16. q/k: RMSNorm over the head (gain q_norm / k_norm) then
// rotate pairs (i, i+64) by pos * theta^(-2i/128) (omnivoice-cpp, Qwen3
// specifics: per-head RMSNorm before RoPE; Qwen3-TTS ncnn port, mRoPE
// conclusion: 1-D half-rotate RoPE). The cos/sin table is computed on the host.
// 4 consecutive QKV values from fp32 or bf16 rows
__device__ __forceinline__ float4 qkv_load4(const float* __restrict__ f, const bf16* __restrict__ b, size_t i) {
    if (b) {
        const uint2 u = *reinterpret_cast<const uint2*>(b + i);
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                           __uint_as_float(u.y & 0xFFFF0000u));
    }
    return *reinterpret_cast<const float4*>(f + i);
}

__global__ void __launch_bounds__(256) k_qk_norm_rope_append(
    const float* __restrict__ qkv, const bf16* __restrict__ qkv_bf, const bf16* __restrict__ qn, const bf16* __restrict__ kn,
    const float* __restrict__ cos_t, const float* __restrict__ sin_t, float eps, bf16* __restrict__ qout,
    KVView kv, const int32_t* __restrict__ seq_start, const int32_t* __restrict__ seq_len, int tok_per_seq,
    int* err, float* __restrict__ qout_f) {
    pdl_wait();  // upstream results are read below
    pdl_trigger();
    const int t = blockIdx.x;
    const int seq = t / tok_per_seq, s = t % tok_per_seq;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool valid = s < seq_len[seq];
    const int pos = seq_start[seq] + s;
    bf16* kdst = nullptr;
    bf16* vdst = nullptr;
    if (valid) {
        const int j = pos / KVB;
        const int phys = kv.page_table ? kv.page_table[(size_t)kv.seq_slot[seq] * kv.mbps + j]
                                       : seq * kv.mbps + j;
        if (phys < 0) {
            if (threadIdx.x == 0) set_err(err, ERR_KV_RANGE);
        } else {
            kdst = kv.pool + (size_t)phys * 2 * NKV * KVB * HD + (size_t)(pos % KVB) * HD;
            vdst = kdst + (size_t)NKV * KVB * HD;
        }
    }
    const size_t row = (size_t)t * QKV;
    const int i0 = (lane & 15) * 4;  // frequency index of this lane's first element
    for (int u = warp; u < 32; u += 8) {
        if (u >= 24) {  // v head: copy
            const int g = u - 24;
            if (!kdst) continue;
            const float4 x = qkv_load4(qkv, qkv_bf, row + NQ * HD + NKV * HD + g * HD + lane * 4);
            __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y), b = __floats2bfloat162_rn(x.z, x.w);
            uint2 o;
            o.x = *reinterpret_cast<uint32_t*>(&a);
            o.y = *reinterpret_cast<uint32_t*>(&b);
            *reinterpret_cast<uint2*>(vdst + (size_t)g * KVB * HD + lane * 4) = o;
            continue;
        }
        const bool isq = u < 16;
        const int hh = isq ? u : u - 16;
        if (!isq && !kdst) continue;
        const size_t src = row + (isq ? hh * HD : NQ * HD + hh * HD);
        float4 x = qkv_load4(qkv, qkv_bf, src + lane * 4);
        float ss = warp_sum(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w);
        const float r = rsqrtf(ss * (1.f / HD) + eps);
        const bf16* gm = isq ? qn : kn;
        float v[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = v[e] * r * bf2f(gm[lane * 4 + e]);
        float p[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) p[e] = __shfl_xor_sync(0xffffffffu, v[e], 16);
        float o[4];
        const float* ct = cos_t + (size_t)pos * (HD / 2) + i0;
        const float* st = sin_t + (size_t)pos * (HD / 2) + i0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float c = valid ? ct[e] : 1.f, sn = valid ? st[e] : 0.f;
            o[e] = (lane < 16) ? (v[e] * c - p[e] * sn) : (v[e] * c + p[e] * sn);
        }
        __nv_bfloat162 a = __floats2bfloat162_rn(o[0], o[1]), b = __floats2bfloat162_rn(o[2], o[3]);
        uint2 w;
        w.x = *reinterpret_cast<uint32_t*>(&a);
        w.y = *reinterpret_cast<uint32_t*>(&b);
        if (isq && qout_f) {  // fp32 queries (decode and tcgen05 causal prefill attention read them unrounded)
            const float4 f4 = valid ? make_float4(o[0], o[1], o[2], o[3]) : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(qout_f + (size_t)t * NQ * HD + hh * HD + lane * 4) = f4;
        } else if (isq) {
            if (!valid) w = make_uint2(0u, 0u);
            *reinterpret_cast<uint2*>(qout + (size_t)t * NQ * HD + hh * HD + lane * 4) = w;
        } else {
            *reinterpret_cast<uint2*>(kdst + (size_t)hh * KVB * HD + lane * 4) = w;
        }
    }
}

int launch_qk_norm_rope_append(const float* qkv, const bf16* qn, const bf16* kn, const float* cos_t,
                                const float* sin_t, float eps, bf16* qout, KVView kv, const int32_t* seq_start,
                                const int32_t* seq_len, int tok_per_seq, int T, int* err, cudaStream_t st,
                                float* qout_f, const bf16* qkv_bf) {
    if (T <= 0) return 0;
    launch_pdl(k_qk_norm_rope_append, T, 256, 0, st, qkv, qkv_bf, qn, kn, cos_t, sin_t, eps, qout, kv, seq_start, seq_len,
                                             tok_per_seq, err, qout_f);
    return 1;
}

// ---------------------------------------------------------------- argmax
__global__ void k_argmax_finalize(const unsigned long long* __restrict__ amax, int32_t* out, int stride, int B) {
    pdl_wait();  // upstream results are read below
    pdl_trigger();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) out[(size_t)b * stride] = (int32_t)(0xFFFFFFFFu - (uint32_t)(amax[b] & 0xFFFFFFFFull));
}

int launch_argmax_finalize(const unsigned long long* amax, int32_t* out, int stride, int B, cudaStream_t st) {
    if (B <= 0) return 0;
    launch_pdl(k_argmax_finalize, (B + 127) / 128, 128, 0, st, amax, out, stride, B);
    return 1;
}

}  // namespace ttsbb
