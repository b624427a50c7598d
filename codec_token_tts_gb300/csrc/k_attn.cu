// GQA attention over the paged KV cache (16 query heads, 8 KV heads of 128:
// query head h reads KV head h/2, scale 1/sqrt(128), softmax in fp32).
//   * Decode (query length 1; Qwen3-TTS ncnn port, single-token SDPA and host
//     attention): split-K flash decode. One CTA per (sequence, KV head,
//     split) reads each K/V block once for both of its query heads; warp-
//     shuffle online softmax; a combine kernel merges the splits in a fixed
//     order (deterministic, no float atomics).
//   * Prefill / bidirectional pass (omnivoice-cpp MaskGIT decoder: no KV cache,
//     non-causal attention): flash attention on bf16 tensor cores (mma.sync),
//     one CTA per (sequence, KV head, 64-query tile) covering both query heads.
#include "common.cuh"

namespace ttsbb {

constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ const bf16* kv_tile(const KVView& kv, int seq, int j, int which, int g) {
    const int phys = kv.page_table ? kv.page_table[(size_t)kv.seq_slot[seq] * kv.mbps + j] : seq * kv.mbps + j;
    return kv.pool + (((size_t)phys * 2 + which) * NKV + g) * (size_t)KVB * HD;
}

// ---------------------------------------------------------------- decode
// One warp's 16 keys, rows row0 .. row0 + 15 of a cache block whose first key is kbase (K tile kb,
// V tile vb): the scores of both query heads (lane l holds head elements 4l .. 4l + 3), then the
// online-softmax update of each head's running max m, sum l and output o. Keys >= L are masked.
__device__ __forceinline__ void attn_warp_keys16(const float (&q0)[4], const float (&q1)[4], const bf16* kb, const bf16* vb,
                                                 int kbase, int row0, int L, int lane, float& m0, float& m1, float& l0,
                                                 float& l1, float (&o0)[4], float (&o1)[4]) {
    const int key0 = kbase + row0;
    float d[32];  // d[h*16 + kk]
    uint2 kr[16], vr[16];
    // K of the 16 keys now; their V rows (16 x 256 B: one 128-byte line per lane) are
    // prefetched into L2 and read after the scores, so fewer registers are live across the loads
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
        const bool ok = key0 + kk < L;
        kr[kk] = ok ? *reinterpret_cast<const uint2*>(kb + (size_t)(row0 + kk) * HD + lane * 4) : make_uint2(0u, 0u);
    }
    if (key0 + (lane >> 1) < L)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(vb + (size_t)(row0 + (lane >> 1)) * HD + (lane & 1) * 64));
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
        const float k0 = __uint_as_float(kr[kk].x << 16), k1 = __uint_as_float(kr[kk].x & 0xFFFF0000u);
        const float k2 = __uint_as_float(kr[kk].y << 16), k3 = __uint_as_float(kr[kk].y & 0xFFFF0000u);
        d[kk] = q0[0] * k0 + q0[1] * k1 + q0[2] * k2 + q0[3] * k3;
        d[16 + kk] = q1[0] * k0 + q1[1] * k1 + q1[2] * k2 + q1[3] * k3;
    }
    // transpose-reduce: afterwards lane i holds the full dot of index i (head i/16, key i%16)
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = upper ? d[i] : d[i + s];
            const float recv = __shfl_xor_sync(0xffffffffu, send, s);
            d[i] = (upper ? d[i + s] : d[i]) + recv;
        }
    }
    const int mykey = key0 + (lane & 15);
    const float score = (mykey < L) ? d[0] : -INFINITY;
    float mx = score;
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float mx0 = __shfl_sync(0xffffffffu, mx, 0), mx1 = __shfl_sync(0xffffffffu, mx, 16);
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float mine_m = (lane < 16) ? mn0 : mn1;
    const float p = (mine_m == -INFINITY) ? 0.f : exp2f(score - mine_m);
    float ps = p;
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    const float ps0 = __shfl_sync(0xffffffffu, ps, 0), ps1 = __shfl_sync(0xffffffffu, ps, 16);
    const float a0 = (mn0 == -INFINITY) ? 1.f : exp2f(m0 - mn0);
    const float a1 = (mn1 == -INFINITY) ? 1.f : exp2f(m1 - mn1);
    l0 = l0 * a0 + ps0;
    l1 = l1 * a1 + ps1;
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int e = 0; e < 4; ++e) { o0[e] *= a0; o1[e] *= a1; }
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
        const bool ok = key0 + kk < L;
        vr[kk] = ok ? *reinterpret_cast<const uint2*>(vb + (size_t)(row0 + kk) * HD + lane * 4) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
        const float p0 = __shfl_sync(0xffffffffu, p, kk), p1 = __shfl_sync(0xffffffffu, p, 16 + kk);
        {
            const float v0 = __uint_as_float(vr[kk].x << 16), v1 = __uint_as_float(vr[kk].x & 0xFFFF0000u);
            const float v2 = __uint_as_float(vr[kk].y << 16), v3 = __uint_as_float(vr[kk].y & 0xFFFF0000u);
            o0[0] += p0 * v0; o0[1] += p0 * v1; o0[2] += p0 * v2; o0[3] += p0 * v3;
            o1[0] += p1 * v0; o1[1] += p1 * v1; o1[2] += p1 * v2; o1[3] += p1 * v3;
        }
    }
}

// Query heads 2g and 2g + 1 of query b, elements 4 lane .. 4 lane + 3, scaled by log2(e) / sqrt(128)
// (fp32 queries qf if given, else the bf16 rows of q).
__device__ __forceinline__ void attn_load_q(const bf16* __restrict__ q, const float* __restrict__ qf, int b, int g, int lane,
                                            float (&q0)[4], float (&q1)[4]) {
    const float sc = rsqrtf((float)HD) * LOG2E;
    if (qf) {
        const float4 a = *reinterpret_cast<const float4*>(qf + ((size_t)b * NQ + 2 * g) * HD + lane * 4);
        const float4 c = *reinterpret_cast<const float4*>(qf + ((size_t)b * NQ + 2 * g + 1) * HD + lane * 4);
        q0[0] = a.x * sc; q0[1] = a.y * sc; q0[2] = a.z * sc; q0[3] = a.w * sc;
        q1[0] = c.x * sc; q1[1] = c.y * sc; q1[2] = c.z * sc; q1[3] = c.w * sc;
    } else {
        const bf16* qp = q + ((size_t)b * NQ + 2 * g) * HD + lane * 4;
        const uint2 a = *reinterpret_cast<const uint2*>(qp);
        const uint2 c = *reinterpret_cast<const uint2*>(qp + HD);
        q0[0] = __uint_as_float(a.x << 16) * sc; q0[1] = __uint_as_float(a.x & 0xFFFF0000u) * sc;
        q0[2] = __uint_as_float(a.y << 16) * sc; q0[3] = __uint_as_float(a.y & 0xFFFF0000u) * sc;
        q1[0] = __uint_as_float(c.x << 16) * sc; q1[1] = __uint_as_float(c.x & 0xFFFF0000u) * sc;
        q1[2] = __uint_as_float(c.y << 16) * sc; q1[3] = __uint_as_float(c.y & 0xFFFF0000u) * sc;
    }
}

// grid (n_splits, 8, B), 128 threads. Warp w takes keys 16w..16w+15 of every
// block of the split; lane l holds head elements 4l..4l+3 of both query heads.
// With one split the CTA writes the normalised output itself (what the
// combine would compute: its weight for a single split is exactly 1).
// Query b (grid z) is token b % tps of sequence b / tps: with tps = 1 one decode token per
// sequence; with tps > 1 a short causal prefill, query s at position seq_start + s seeing keys up
// to its own position (a padding token, s >= seq_len, sees the sequence's valid keys only).
__global__ void __launch_bounds__(128) k_attn_decode(const bf16* __restrict__ q, KVView kv,
                                                     const int32_t* __restrict__ seq_start, int bps,
                                                     int n_splits, float* __restrict__ part,
                                                     bf16* __restrict__ out, bf16* __restrict__ out_lo,
                                                     const float* __restrict__ qf, int tps,
                                                     const int32_t* __restrict__ seq_len) {
    pdl_wait();  // upstream results are read below
    pdl_trigger();
    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seq = b / tps, s_tok = b - seq * tps;
    // keys incl. the token just appended (decode), or up to this query's position (short prefill)
    const int L = tps == 1 ? seq_start[seq] + 1 : seq_start[seq] + min(s_tok + 1, seq_len[seq]);
    const int nblk = (L + KVB - 1) / KVB;
    const int blk0 = split * bps, blk1 = min(nblk, blk0 + bps);

    float q0[4], q1[4];
    attn_load_q(q, qf, b, g, lane, q0, q1);
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o0[4] = {0.f, 0.f, 0.f, 0.f}, o1[4] = {0.f, 0.f, 0.f, 0.f};

    for (int j = blk0; j < blk1; ++j) {
        const bf16* kb = kv_tile(kv, seq, j, 0, g);
        const bf16* vb = kv_tile(kv, seq, j, 1, g);
        attn_warp_keys16(q0, q1, kb, vb, j * KVB, warp * 16, L, lane, m0, m1, l0, l1, o0, o1);
    }
    // merge the 4 warps of the CTA
    __shared__ float sm_ml[4][4];
    __shared__ float sm_o[4][2][HD];
    if (lane == 0) { sm_ml[warp][0] = m0; sm_ml[warp][1] = l0; sm_ml[warp][2] = m1; sm_ml[warp][3] = l1; }
#pragma unroll
    for (int e = 0; e < 4; ++e) { sm_o[warp][0][lane * 4 + e] = o0[e]; sm_o[warp][1][lane * 4 + e] = o1[e]; }
    __syncthreads();
    // thread t: head t / 64, elements (t % 64) * 2, +1
    const int hh = threadIdx.x >> 6, e0 = (threadIdx.x & 63) * 2;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_ml[w][hh * 2]);
    float l = 0.f, a = 0.f, c = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float mw = sm_ml[w][hh * 2];
        const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
        l += sm_ml[w][hh * 2 + 1] * f;
        a += sm_o[w][hh][e0] * f;
        c += sm_o[w][hh][e0 + 1] * f;
    }
    if (n_splits == 1) {
        const size_t o = ((size_t)b * NQ + 2 * g + hh) * HD + e0;
        const float r0 = l > 0.f ? a / l : 0.f, r1 = l > 0.f ? c / l : 0.f;
        out[o] = f2bf(r0);
        out[o + 1] = f2bf(r1);
        if (out_lo) {
            out_lo[o] = f2bf_lo(r0);
            out_lo[o + 1] = f2bf_lo(r1);
        }
        return;
    }
    // part layout per (b, head, split): [HD] o, then m, l
    float* dst = part + (((size_t)b * NQ + 2 * g + hh) * n_splits + split) * (HD + 2);
    dst[e0] = a;
    dst[e0 + 1] = c;
    if ((threadIdx.x & 63) == 0) { dst[HD] = M; dst[HD + 1] = l; }
}

// Decode attention for contexts that fit two 16-key rounds (max_len <= ATTN_SHORT_CTX, e.g. the
// Code Predictor's 16 positions): one warp per (query, KV head) pair takes the keys in rounds of
// 16 (the split kernel's per-warp step, continued with the online softmax) and writes the
// normalised output; no warp idles on keys past the end. Queries as in k_attn_decode.
// grid ceil(B * 8 / 4), 128 threads; warp w of CTA c takes pair 4c + w = b * 8 + g.
__global__ void __launch_bounds__(128) k_attn_decode_short(const bf16* __restrict__ q, KVView kv,
                                                           const int32_t* __restrict__ seq_start, int npairs,
                                                           bf16* __restrict__ out, bf16* __restrict__ out_lo,
                                                           const float* __restrict__ qf, int tps,
                                                           const int32_t* __restrict__ seq_len) {
    pdl_wait();  // upstream results are read below
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = blockIdx.x * 4 + warp;
    if (pair >= npairs) return;
    const int b = pair / NKV, g = pair - b * NKV;
    const int seq = b / tps, s_tok = b - seq * tps;
    const int L = tps == 1 ? seq_start[seq] + 1 : seq_start[seq] + min(s_tok + 1, seq_len[seq]);
    float q0[4], q1[4];
    attn_load_q(q, qf, b, g, lane, q0, q1);
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o0[4] = {0.f, 0.f, 0.f, 0.f}, o1[4] = {0.f, 0.f, 0.f, 0.f};
    if (L > 0) {
        const bf16* kb = kv_tile(kv, seq, 0, 0, g);
        const bf16* vb = kv_tile(kv, seq, 0, 1, g);
        for (int row0 = 0; row0 < L && row0 < KVB; row0 += 16)
            attn_warp_keys16(q0, q1, kb, vb, 0, row0, L, lane, m0, m1, l0, l1, o0, o1);
    }
    const size_t o = ((size_t)b * NQ + 2 * g) * HD + lane * 4;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float r0 = l0 > 0.f ? o0[e] / l0 : 0.f, r1 = l1 > 0.f ? o1[e] / l1 : 0.f;
        out[o + e] = f2bf(r0);
        out[o + HD + e] = f2bf(r1);
        if (out_lo) {
            out_lo[o + e] = f2bf_lo(r0);
            out_lo[o + HD + e] = f2bf_lo(r1);
        }
    }
}

// grid B*16, 128 threads: merge the splits of one (sequence, head) in split order.
__global__ void __launch_bounds__(128) k_attn_combine(const float* __restrict__ part, int n_splits,
                                                      bf16* __restrict__ out, bf16* __restrict__ out_lo) {
    pdl_wait();  // upstream results are read below
    pdl_trigger();
    const int bh = blockIdx.x, d = threadIdx.x;
    const float* p = part + (size_t)bh * n_splits * (HD + 2);
    float M = -INFINITY;
    for (int s = 0; s < n_splits; ++s) M = fmaxf(M, p[s * (HD + 2) + HD]);
    float l = 0.f, o = 0.f;
    for (int s = 0; s < n_splits; ++s) {
        const float ms = p[s * (HD + 2) + HD];
        const float f = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
        l += p[s * (HD + 2) + HD + 1] * f;
        o += p[s * (HD + 2) + d] * f;
    }
    const float r = l > 0.f ? o / l : 0.f;
    out[(size_t)bh * HD + d] = f2bf(r);
    if (out_lo) out_lo[(size_t)bh * HD + d] = f2bf_lo(r);
}

int launch_attn_decode(const bf16* q, KVView kv, const int32_t* seq_start, int B, int max_len, float* part,
                        bf16* out, int max_splits, cudaStream_t st, bf16* out_lo, const float* qf, int tps,
                        const int32_t* seq_len) {
    if (tps < 1 || (tps > 1 && !seq_len)) return 0;
    if (B <= 0) return 0;
    if (max_len <= ATTN_SHORT_CTX) {
        const int npairs = B * NKV;
        launch_pdl(k_attn_decode_short, (npairs + 3) / 4, 128, 0, st, q, kv, seq_start, npairs, out, out_lo, qf, tps,
                   seq_len);
        return 1;
    }
    const int nblk = (max_len + KVB - 1) / KVB;
    // ~32 CTAs per SM (several waves): the block scheduler balances ragged sequence lengths
    // (splits past a sequence's end exit at once); measured better than one wave of 8 per SM
    int splits = (32 * 152 + B * NKV - 1) / (B * NKV);
    splits = max(1, min(splits, min(nblk, max_splits)));
    const int bps = (nblk + splits - 1) / splits;
    splits = (nblk + bps - 1) / bps;
    launch_pdl(k_attn_decode, dim3(splits, NKV, B), 128, 0, st, q, kv, seq_start, bps, splits, part, out, out_lo, qf,
               tps, seq_len);
    if (splits == 1) return 1;
    launch_pdl(k_attn_combine, B * NQ, 128, 0, st, part, splits, out, out_lo);
    return 2;
}

// ---------------------------------------------------------------- prefill / bidirectional
namespace fa {
constexpr int BQ = 64, LDS = HD + 8;  // padded rows: 272 B, conflict-free ldmatrix
constexpr int Q_ELEMS = 2 * BQ * LDS, KV_ELEMS = KVB * LDS;
constexpr int SMEM = (Q_ELEMS + 4 * KV_ELEMS) * 2;
}  // namespace fa

__device__ __forceinline__ void cp_async16z(void* smem, const void* gmem, bool pred) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(pred ? 16 : 0));
}
__device__ __forceinline__ void ldsm_x4(uint32_t* r, const void* p) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(s));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t* r, const void* p) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(s));
}
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

// grid (ceil(S/64), 8, B), 256 threads. Warps 0-3: query head 2g, warps 4-7:
// head 2g+1; each warp 16 query rows.
__global__ void __launch_bounds__(256) k_attn_prefill(const bf16* __restrict__ q, KVView kv,
                                                      const int32_t* __restrict__ seq_start,
                                                      const int32_t* __restrict__ seq_len,
                                                      const int32_t* __restrict__ key_len, int causal, int S,
                                                      bf16* __restrict__ out, bf16* __restrict__ out_lo) {
    pdl_wait();  // upstream results are read below
    pdl_trigger();
    using namespace fa;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    bf16* sQ = reinterpret_cast<bf16*>(smem_raw);
    bf16* sK = sQ + Q_ELEMS;          // [2][KVB][LDS]
    bf16* sV = sK + 2 * KV_ELEMS;     // [2][KVB][LDS]
    const int qt = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int start = seq_start[b];
    const int len = causal ? seq_len[b] : S;
    const int kv_end = causal ? min(start + len, start + (qt + 1) * BQ) : key_len[b];
    if (qt * BQ >= S) return;
    const int ntiles = (kv_end + KVB - 1) / KVB;

    // Q: rows r = hsel*64 + i, token b*S + qt*64 + i, head 2g + hsel
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = tid + i * 256;          // 2048 chunks of 16 B
        const int r = c >> 4, col = (c & 15) * 8;
        const int hsel = r >> 6, s = qt * BQ + (r & 63);
        const bool ok = s < S;
        const bf16* src = q + ((size_t)(b * S + (ok ? s : 0)) * NQ + 2 * g + hsel) * HD + col;
        cp_async16z(sQ + r * LDS + col, src, ok);
    }
    auto load_kv = [&](int buf, int j) {
        const bf16* kb = kv_tile(kv, b, j, 0, g);
        const bf16* vb = kv_tile(kv, b, j, 1, g);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = tid + i * 256;      // 1024 chunks per operand
            const int r = c >> 4, col = (c & 15) * 8;
            const bool ok = j * KVB + r < kv_end;
            cp_async16z(sK + buf * KV_ELEMS + r * LDS + col, kb + (size_t)r * HD + col, ok);
            cp_async16z(sV + buf * KV_ELEMS + r * LDS + col, vb + (size_t)r * HD + col, ok);
        }
    };
    load_kv(0, 0);
    asm volatile("cp.async.commit_group;");

    const int hsel = warp >> 2, wr = (warp & 3) * 16;
    const int row_a = qt * BQ + wr + (lane >> 2);         // query index within sequence (rows g, g+8)
    const int qpos0 = start + row_a, qpos1 = qpos0 + 8;
    const float sc = rsqrtf((float)HD) * LOG2E;

    uint32_t qf[8][4];
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[i][e] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

    for (int j = 0; j < ntiles; ++j) {
        if (j + 1 < ntiles) load_kv((j + 1) & 1, j + 1);
        asm volatile("cp.async.commit_group;");
        asm volatile("cp.async.wait_group 1;");
        __syncthreads();
        if (j == 0) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                ldsm_x4(qf[kk], sQ + (hsel * BQ + wr + (lane & 15)) * LDS + kk * 16 + (lane >> 4) * 8);
        }
        const bf16* kS = sK + (j & 1) * KV_ELEMS;
        const bf16* vS = sV + (j & 1) * KV_ELEMS;
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
            for (int n2 = 0; n2 < 4; ++n2) {
                uint32_t bfr[4];
                const int r = n2 * 16 + (lane & 7) + ((lane >> 4) << 3);
                ldsm_x4(bfr, kS + r * LDS + kk * 16 + ((lane >> 3) & 1) * 8);
                mma_bf16(s[2 * n2], qf[kk], bfr[0], bfr[1]);
                mma_bf16(s[2 * n2 + 1], qf[kk], bfr[2], bfr[3]);
            }
        }
        // mask + online softmax (base 2)
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kp = j * KVB + n * 8 + (lane & 3) * 2 + (e & 1);
                const int qp = (e < 2) ? qpos0 : qpos1;
                const bool ok = kp < kv_end && (!causal || kp <= qp);
                const float v = ok ? s[n][e] * sc : -INFINITY;
                s[n][e] = v;
                mx[e >> 1] = fmaxf(mx[e >> 1], v);
            }
        float alpha[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
            const float mn = fmaxf(mrow[r], mx[r]);
            alpha[r] = (mn == -INFINITY) ? 1.f : exp2f(mrow[r] - mn);
            mrow[r] = mn;
        }
        float ls[2] = {0.f, 0.f};
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float m = mrow[e >> 1];
                // rounded to bf16 here, as P V will use it: the row sum then matches the weights applied
                const float p = bf2f(f2bf((m == -INFINITY) ? 0.f : exp2f(s[n][e] - m)));
                s[n][e] = p;
                ls[e >> 1] += p;
            }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            ls[r] += __shfl_xor_sync(0xffffffffu, ls[r], 1);
            ls[r] += __shfl_xor_sync(0xffffffffu, ls[r], 2);
            lrow[r] = lrow[r] * alpha[r] + ls[r];
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            o[i][0] *= alpha[0]; o[i][1] *= alpha[0];
            o[i][2] *= alpha[1]; o[i][3] *= alpha[1];
        }
        // O += P V
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t pa[4];
            pa[0] = pack_bf2(s[2 * kk][0], s[2 * kk][1]);
            pa[1] = pack_bf2(s[2 * kk][2], s[2 * kk][3]);
            pa[2] = pack_bf2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            pa[3] = pack_bf2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
            for (int d2 = 0; d2 < 8; ++d2) {
                uint32_t vf[4];
                const int r = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                ldsm_x4_t(vf, vS + r * LDS + d2 * 16 + (lane >> 4) * 8);
                mma_bf16(o[2 * d2], pa, vf[0], vf[1]);
                mma_bf16(o[2 * d2 + 1], pa, vf[2], vf[3]);
            }
        }
        __syncthreads();
    }
    asm volatile("cp.async.wait_group 0;");
    // write O / l
    const float inv0 = lrow[0] > 0.f ? 1.f / lrow[0] : 0.f, inv1 = lrow[1] > 0.f ? 1.f / lrow[1] : 0.f;
    const int h = 2 * g + hsel;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int s_idx = row_a + r * 8;
        if (s_idx >= S) continue;
        const size_t off = ((size_t)(b * S + s_idx) * NQ + h) * HD;
        const float inv = r ? inv1 : inv0;
#pragma unroll
        for (int d8 = 0; d8 < 16; ++d8) {
            const int d = d8 * 8 + (lane & 3) * 2;
            const float v0 = o[d8][2 * r] * inv, v1 = o[d8][2 * r + 1] * inv;
            const uint32_t hi = pack_bf2(v0, v1);
            *reinterpret_cast<uint32_t*>(out + off + d) = hi;
            if (out_lo) {  // low parts: value - bf16(value)
                const float2 hf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hi));
                *reinterpret_cast<uint32_t*>(out_lo + off + d) = pack_bf2(v0 - hf.x, v1 - hf.y);
            }
        }
    }
}

int launch_attn_prefill(const bf16* q, KVView kv, const int32_t* seq_start, const int32_t* seq_len,
                         const int32_t* key_len, int causal, int B, int S, bf16* out, cudaStream_t st,
                         bf16* out_lo) {
    if (B <= 0 || S <= 0) return 0;
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(k_attn_prefill, cudaFuncAttributeMaxDynamicSharedMemorySize, fa::SMEM);
        attr_set = true;
    }
    dim3 grid((S + fa::BQ - 1) / fa::BQ, NKV, B);
    launch_pdl(k_attn_prefill, grid, 256, fa::SMEM, st, q, kv, seq_start, seq_len, key_len, causal, S, out, out_lo);
    return 1;
}

}  // namespace ttsbb
