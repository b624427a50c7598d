// Persistent decode step for small batch (B <= 4): the whole 28-layer step —
// codebook gather-sum, RMSNorm, QKV, q/k-norm + RoPE + KV append, GQA
// attention over the paged cache, o_proj + residual, RMSNorm, gate/up +
// SwiGLU, down + residual, final norm, codec head + argmax — in one
// cooperative launch with one CTA per SM.
//
// At batch 1 the step is a stream of 0.89 GB of weights that no activation
// gates: each CTA owns a fixed row slice of every matrix, and a producer warp
// copies those slices (cp.async.bulk, completion on mbarriers) into a
// shared-memory ring, running ahead of the consumers by up to the ring size.
// The eight consumer warps wait on the ring and on grid barriers only where
// the data flow needs them (after QKV, after attention, after o_proj, after
// gate/up, after down). Every wait is bounded: on timeout the kernel raises
// the error word and an abort flag, stops waiting and runs to its end.
#include "mega.cuh"

namespace ttsbb {

namespace mk {
constexpr int NCW = 8;                  // consumer warps
constexpr int NCT = NCW * 32;           // consumer threads
constexpr int NT = NCT + 32;            // + one producer warp
constexpr int RING = 176 * 1024;        // weight ring bytes
constexpr int NSLOT = 16;               // chunks in flight at most
constexpr int CHUNK = 32 * 1024;        // bytes per chunk (whole rows)
constexpr int XS_BYTES = MAXB * 3072 * 4;   // fp32 activations
constexpr int MAXSPLIT = 64;            // cache blocks per sequence (4096 tokens)
constexpr int NSTAMP = 16;              // trace stamps per layer
constexpr int ATT_FLOATS = (NCW * (2 * HD + 4) + 2 * HD) > (MAXB * NQ * MAXSPLIT) ? (NCW * (2 * HD + 4) + 2 * HD)
                                                                                    : (MAXB * NQ * MAXSPLIT);
constexpr int SMEM = RING + XS_BYTES + ATT_FLOATS * 4 + 2 * NSLOT * 8 + 64;
constexpr unsigned long long TIMEOUT_NS = 2000000000ull;  // 2 s per wait
}  // namespace mk

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long gtime() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* b, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     su32(dst)),
                 "l"(src), "r"(bytes), "r"(su32(bar))
                 : "memory");
}
__device__ __forceinline__ void named_sync() { asm volatile("bar.sync 1, %0;" ::"n"(mk::NCT) : "memory"); }

// Bounded mbarrier wait; false on timeout or when another CTA aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, const MegaArgs& a) {
    if (mbar_try(b, parity)) return true;
    const unsigned long long t0 = gtime();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try(b, parity)) return true;
        if ((i & 63) == 63) {
            if (*reinterpret_cast<volatile int*>(a.abort_flag)) return false;
            if (gtime() - t0 > mk::TIMEOUT_NS) {
                set_err(a.err, ERR_TIMEOUT);
                atomicExch(a.abort_flag, 1);
                return false;
            }
        }
    }
}

// Grid barrier among the consumer threads of all CTAs (the producer warps do
// not take part). Counter is monotonic; barrier k waits for base + k * G arrivals.
// After a timeout (or another CTA's abort) it stops waiting: consumers never
// leave early, so every named barrier of the CTA still completes, and with the
// abort flag set every later wait returns at once — the kernel finishes with
// the error word raised and garbage outputs.
__device__ __forceinline__ void grid_sync(const MegaArgs& a, int& k) {
    named_sync();
    if (threadIdx.x == 0) {
        ++k;
        const unsigned long long target = a.bar_base + (unsigned long long)k * gridDim.x;
        __threadfence();
        atomicAdd(a.bar, 1ull);
        const unsigned long long t0 = gtime();
        for (uint32_t i = 0;; ++i) {
            const unsigned long long v = *reinterpret_cast<volatile unsigned long long*>(a.bar);
            if (v >= target) break;
            if ((i & 31) == 31) {
                if (*reinterpret_cast<volatile int*>(a.abort_flag)) break;
                if (gtime() - t0 > mk::TIMEOUT_NS) {
                    set_err(a.err, ERR_TIMEOUT);
                    atomicExch(a.abort_flag, 1);
                    break;
                }
            }
        }
        __threadfence();
    }
    named_sync();
}

// ---------------------------------------------------------------- schedule
// Op o of layer l (o = 0 QKV, 1 O, 2 gate/up, 3 down) or the head (l = n_layers).
struct OpDesc {
    const bf16* W;
    int N, K;
};
__device__ __forceinline__ OpDesc op_desc(const MegaArgs& a, int l, int o) {
    if (l == a.n_layers) return {a.head, a.head_rows, HID};
    const MegaLayer& L = a.L[l];
    switch (o) {
        case 0: return {L.wqkv, QKV, HID};
        case 1: return {L.wo, HID, NQ * HD};
        case 2: return {L.wgu, 2 * a.ffn, HID};
        default: return {L.wd, HID, a.ffn};
    }
}
// Row slice [r0, r1) of CTA c, split in pairs so gate/up rows stay together.
__device__ __forceinline__ void cta_rows(int N, int c, int G, int& r0, int& r1) {
    const long pairs = N / 2;
    r0 = (int)(pairs * c / G) * 2;
    r1 = (int)(pairs * (c + 1) / G) * 2;
}
__device__ __forceinline__ int rows_per_chunk(int K) {
    int r = mk::CHUNK / (K * 2);
    r &= ~1;
    return r < 2 ? 2 : (r > 16 ? 16 : r);
}

// Ring position bookkeeping shared by producer and consumers (same sequence).
struct Ring {
    unsigned long long head = 0;
    uint32_t k = 0;  // chunk counter
    __device__ __forceinline__ uint32_t place(uint32_t bytes) {
        uint32_t p = (uint32_t)(head % mk::RING);
        if (p + bytes > (uint32_t)mk::RING) {
            head += mk::RING - p;
            p = 0;
        }
        head += bytes;
        return p;
    }
};

// ---------------------------------------------------------------- consumer pieces
// xs[b][0..1023] = bf16(rmsnorm(src[b]) * gamma); warp b does row b.
__device__ __forceinline__ void stage_norm(const MegaArgs& a, const float* src, const bf16* gamma, float* xs) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < a.B) {
        const float4* row = reinterpret_cast<const float4*>(src + (size_t)warp * HID);
        float4 v[8];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[i] = __ldcg(row + i * 32 + lane);
            ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
        }
        ss = warp_sum(ss);
        const float r = rsqrtf(ss * (1.f / HID) + a.eps);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = (i * 32 + lane) * 4;
            const uint2 gr = *reinterpret_cast<const uint2*>(gamma + e);
            *reinterpret_cast<float4*>(xs + (size_t)warp * HID + e) =
                make_float4(v[i].x * r * __uint_as_float(gr.x << 16), v[i].y * r * __uint_as_float(gr.x & 0xFFFF0000u),
                            v[i].z * r * __uint_as_float(gr.y << 16), v[i].w * r * __uint_as_float(gr.y & 0xFFFF0000u));
        }
    }
}

// Layer-0 input: h[b] = embeds[b] + sum_k E_k[ids[b][k]] computed by every CTA
// (into smem as fp32 in place of the residual read); CTA 0 also stores it.
__device__ __forceinline__ void stage_embed(const MegaArgs& a, float* hs) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < a.B) {
        const int b = warp;
        for (int c = lane * 8; c < HID; c += 256) {
            float acc[8];
            if (a.embeds) {
                unpack8(*reinterpret_cast<const uint4*>(a.embeds + (size_t)b * HID + c), acc);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.f;
            }
            if (a.ids) {
                for (int k = 0; k < a.tabs.n; ++k) {
                    const int id = a.ids[b * a.tabs.n + k];
                    if (id == -1) continue;
                    if (id < -1 || id >= a.tabs.rows[k]) {
                        if (blockIdx.x == 0 && c == 0) set_err(a.err, ERR_BAD_ID);
                        continue;
                    }
                    float f[8];
                    unpack8(*reinterpret_cast<const uint4*>(a.tabs.tab[k] + (size_t)id * HID + c), f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] += f[i];
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) hs[b * HID + c + i] = acc[i];
            if (blockIdx.x == 0) {
                float4* o = reinterpret_cast<float4*>(a.h + (size_t)b * HID + c);
                o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            }
        }
    }
}

// Consume this CTA's chunks of one op: y[b][row] = sum_k W[row][k] x[b][k].
// Warp w takes rows 2w and 2w+1 of each chunk (a gate/up pair for SwiGLU).
template <int B>
__device__ __forceinline__ void consume_op(const MegaArgs& a, int l, int o, Ring& ring, unsigned char* ring_mem,
                                           uint64_t* full, uint64_t* empty, const float* xs) {
    const OpDesc d = op_desc(a, l, o);
    int r0, r1;
    cta_rows(d.N, blockIdx.x, gridDim.x, r0, r1);
    const int rpc = rows_per_chunk(d.K);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nv = d.K / 256;  // 16-byte vectors per lane per row
    const bool is_head = (l == a.n_layers);
    for (int rc = r0; rc < r1; rc += rpc) {
        const int nr = min(rpc, r1 - rc);
        const uint32_t bytes = (uint32_t)nr * d.K * 2;
        const uint32_t p = ring.place(bytes);
        const uint32_t slot = ring.k % mk::NSLOT, par = (ring.k / mk::NSLOT) & 1;
        ring.k++;
        if (a.trace && threadIdx.x == 0) {  // time spent waiting for this chunk's weights
            const unsigned long long t0 = gtime();
            mbar_wait(full + slot, par, a);
            a.trace[((size_t)blockIdx.x * a.n_layers + (l < a.n_layers ? l : a.n_layers - 1)) * mk::NSTAMP + 15] +=
                gtime() - t0;
        }
        mbar_wait(full + slot, par, a);  // on abort: compute on whatever is there
        const bf16* wc = reinterpret_cast<const bf16*>(ring_mem + p);
        float acc[2][B];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
#pragma unroll
            for (int b = 0; b < B; ++b) acc[rr][b] = 0.f;
        const int lr0 = 2 * warp;
        if (lr0 < nr) {
            for (int i = 0; i < nv; ++i) {
                const int col = (i * 32 + lane) * 8;
                float xf[B][8];
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    const float4 x0 = *reinterpret_cast<const float4*>(xs + b * d.K + col);
                    const float4 x1 = *reinterpret_cast<const float4*>(xs + b * d.K + col + 4);
                    xf[b][0] = x0.x; xf[b][1] = x0.y; xf[b][2] = x0.z; xf[b][3] = x0.w;
                    xf[b][4] = x1.x; xf[b][5] = x1.y; xf[b][6] = x1.z; xf[b][7] = x1.w;
                }
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    if (lr0 + rr >= nr) break;
                    float wf[8];
                    unpack8(*reinterpret_cast<const uint4*>(wc + (size_t)(lr0 + rr) * d.K + col), wf);
#pragma unroll
                    for (int b = 0; b < B; ++b) {
                        float s = acc[rr][b];
#pragma unroll
                        for (int j = 0; j < 8; ++j) s = fmaf(wf[j], xf[b][j], s);
                        acc[rr][b] = s;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + slot);
        if (lr0 < nr) {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int b = 0; b < B; ++b) acc[rr][b] = warp_sum(acc[rr][b]);
            if (lane < B) {
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    if (b != lane) continue;
                    const int row = rc + lr0;
                    if (is_head) {
                        unsigned long long best = 0ull;
#pragma unroll
                        for (int rr = 0; rr < 2; ++rr) {
                            if (lr0 + rr >= nr) break;
                            if (a.logits) a.logits[(size_t)b * a.head_rows + row + rr] = acc[rr][b];
                            const unsigned long long pk = pack_argmax(acc[rr][b], row + rr);
                            best = pk > best ? pk : best;
                        }
                        if (a.argmax_out) atomicMax(a.amax + b, best);
                    } else if (o == 0) {
                        a.qkv[(size_t)b * QKV + row] = acc[0][b];
                        if (lr0 + 1 < nr) a.qkv[(size_t)b * QKV + row + 1] = acc[1][b];
                    } else if (o == 2) {
                        const float g = acc[0][b], u = acc[1][b];
                        a.m[(size_t)b * a.ffn + row / 2] = g / (1.f + __expf(-g)) * u;
                    } else {  // o_proj / down: residual add (each row has one owner)
                        float* hr = a.h + (size_t)b * HID + row;
                        hr[0] = __ldcg(hr) + acc[0][b];
                        if (lr0 + 1 < nr) hr[1] = __ldcg(hr + 1) + acc[1][b];
                    }
                }
            }
        }
    }
}

// q/k RMSNorm + RoPE of one head held 4 elements per lane (partner lane ^ 16).
__device__ __forceinline__ void norm_rope4(float* v, const bf16* gamma, int pos, const MegaArgs& a, int lane) {
    float ss = warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]);
    const float r = rsqrtf(ss * (1.f / HD) + a.eps);
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = v[e] * r * bf2f(gamma[lane * 4 + e]);
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = __shfl_xor_sync(0xffffffffu, v[e], 16);
    const int i0 = (lane & 15) * 4;
    const float* ct = a.cos_t + (size_t)pos * (HD / 2) + i0;
    const float* st = a.sin_t + (size_t)pos * (HD / 2) + i0;
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = (lane < 16) ? (v[e] * ct[e] - p[e] * st[e]) : (v[e] * ct[e] + p[e] * st[e]);
}

// One attention unit: sequence b, KV head g, cache block j. Writes the block's
// softmax partial (o[128], running max, running sum) for query heads 2g, 2g+1.
// The unit that owns the last block also appends the new token's K/V.
__device__ __forceinline__ void attn_unit(const MegaArgs& a, int l, int b, int g, int j, float* att, bool stamp) {
#define USTAMP(i)                                                                                 \
    do {                                                                                          \
        if (stamp && a.trace && threadIdx.x == 0)                                                 \
            a.trace[((size_t)blockIdx.x * a.n_layers + l) * mk::NSTAMP + (i)] = gtime();         \
    } while (0)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pos = a.pos[b], L = pos + 1;
    const int nblk = (L + KVB - 1) / KVB;
    const float* row = a.qkv + (size_t)b * QKV;
    float* sq = att + mk::NCW * (2 * HD + 4);  // [2][HD] scaled queries
    const int phys = __ldcg(a.page_table + (size_t)a.slot[b] * a.mbps + j);
    bf16* kb = a.pool + (size_t)l * a.layer_elems + ((size_t)phys * 2 * NKV + g) * KVB * HD;
    bf16* vb = kb + (size_t)NKV * KVB * HD;
    if (warp < 2) {
        float v[4];
        const float4 x = __ldcg(reinterpret_cast<const float4*>(row + (2 * g + warp) * HD + lane * 4));
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
        norm_rope4(v, a.L[l].qn, pos, a, lane);
        const float sc = rsqrtf((float)HD) * 1.4426950408889634f;
#pragma unroll
        for (int e = 0; e < 4; ++e) sq[warp * HD + lane * 4 + e] = v[e] * sc;
    } else if (warp == 2 && j == nblk - 1) {
        float v[4];
        const float4 x = __ldcg(reinterpret_cast<const float4*>(row + NQ * HD + g * HD + lane * 4));
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
        norm_rope4(v, a.L[l].kn, pos, a, lane);
        __nv_bfloat162 p0 = __floats2bfloat162_rn(v[0], v[1]), p1 = __floats2bfloat162_rn(v[2], v[3]);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t*>(&p0);
        o.y = *reinterpret_cast<uint32_t*>(&p1);
        *reinterpret_cast<uint2*>(kb + (size_t)(pos % KVB) * HD + lane * 4) = o;
    } else if (warp == 3 && j == nblk - 1) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(row + NQ * HD + NKV * HD + g * HD + lane * 4));
        __nv_bfloat162 p0 = __floats2bfloat162_rn(x.x, x.y), p1 = __floats2bfloat162_rn(x.z, x.w);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t*>(&p0);
        o.y = *reinterpret_cast<uint32_t*>(&p1);
        *reinterpret_cast<uint2*>(vb + (size_t)(pos % KVB) * HD + lane * 4) = o;
    }
    named_sync();
    USTAMP(12);
    // warp w: keys 8w..8w+7 of the block
    float q0[4], q1[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) { q0[e] = sq[lane * 4 + e]; q1[e] = sq[HD + lane * 4 + e]; }
    const int key0 = j * KVB + warp * 8;
    float d[16];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint2 kr = make_uint2(0u, 0u);
        if (key0 + kk < L) kr = __ldcg(reinterpret_cast<const uint2*>(kb + (size_t)(warp * 8 + kk) * HD + lane * 4));
        const float k0 = __uint_as_float(kr.x << 16), k1 = __uint_as_float(kr.x & 0xFFFF0000u);
        const float k2 = __uint_as_float(kr.y << 16), k3 = __uint_as_float(kr.y & 0xFFFF0000u);
        d[kk] = q0[0] * k0 + q0[1] * k1 + q0[2] * k2 + q0[3] * k3;
        d[8 + kk] = q1[0] * k0 + q1[1] * k1 + q1[2] * k2 + q1[3] * k3;
    }
    // transpose-reduce over the 16 lanes of each half, then across halves:
    // lane i ends with the dot of index i & 15 (head (i & 15) / 8, key i & 7)
#pragma unroll
    for (int s = 8; s >= 1; s >>= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = upper ? d[i] : d[i + s];
            const float recv = __shfl_xor_sync(0xffffffffu, send, s);
            d[i] = (upper ? d[i + s] : d[i]) + recv;
        }
    }
    d[0] += __shfl_xor_sync(0xffffffffu, d[0], 16);
    const int idx = lane & 15, hh = idx >> 3, kk = idx & 7;
    const float score = (key0 + kk < L) ? d[0] : -INFINITY;
    float mx = score;
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    const float p = (mx == -INFINITY) ? 0.f : exp2f(score - mx);
    float ps = p;
    ps += __shfl_xor_sync(0xffffffffu, ps, 1);
    ps += __shfl_xor_sync(0xffffffffu, ps, 2);
    ps += __shfl_xor_sync(0xffffffffu, ps, 4);
    const float m0 = __shfl_sync(0xffffffffu, mx, 0), m1 = __shfl_sync(0xffffffffu, mx, 8);
    const float l0 = __shfl_sync(0xffffffffu, ps, 0), l1 = __shfl_sync(0xffffffffu, ps, 8);
    (void)hh;
    float o0[4] = {0.f, 0.f, 0.f, 0.f}, o1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k2 = 0; k2 < 8; ++k2) {
        const float p0 = __shfl_sync(0xffffffffu, p, k2), p1 = __shfl_sync(0xffffffffu, p, 8 + k2);
        if (key0 + k2 < L) {
            const uint2 vr = __ldcg(reinterpret_cast<const uint2*>(vb + (size_t)(warp * 8 + k2) * HD + lane * 4));
            const float v0 = __uint_as_float(vr.x << 16), v1 = __uint_as_float(vr.x & 0xFFFF0000u);
            const float v2 = __uint_as_float(vr.y << 16), v3 = __uint_as_float(vr.y & 0xFFFF0000u);
            o0[0] += p0 * v0; o0[1] += p0 * v1; o0[2] += p0 * v2; o0[3] += p0 * v3;
            o1[0] += p1 * v0; o1[1] += p1 * v1; o1[2] += p1 * v2; o1[3] += p1 * v3;
        }
    }
    USTAMP(13);
    float* wml = att + warp * (2 * HD + 4);
    if (lane == 0) { wml[2 * HD] = m0; wml[2 * HD + 1] = l0; wml[2 * HD + 2] = m1; wml[2 * HD + 3] = l1; }
#pragma unroll
    for (int e = 0; e < 4; ++e) { wml[lane * 4 + e] = o0[e]; wml[HD + lane * 4 + e] = o1[e]; }
    named_sync();
    // merge the 8 warps: thread t -> head t / 128, element t % 128
    {
        const int t = threadIdx.x, h2 = t >> 7, e = t & 127;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < mk::NCW; ++w) M = fmaxf(M, att[w * (2 * HD + 4) + 2 * HD + 2 * h2]);
        float lsum = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < mk::NCW; ++w) {
            const float* ww = att + w * (2 * HD + 4);
            const float mw = ww[2 * HD + 2 * h2];
            const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
            lsum += ww[2 * HD + 2 * h2 + 1] * f;
            acc += ww[h2 * HD + e] * f;
        }
        float* dst = a.part + (((size_t)b * NQ + 2 * g + h2) * a.nblk_max + j) * PART_STRIDE;
        dst[e] = acc;
        if (e == 0) { dst[HD] = M; dst[HD + 1] = lsum; }
    }
    named_sync();
    USTAMP(14);
#undef USTAMP
}

// xs[b][h*128 + d] = merge of the block partials of (b, h), in block order.
// First the per-block weights w_j = 2^(m_j - M) / sum_j l_j 2^(m_j - M) go to
// shared memory (one thread per (b, h)); then every thread combines float4
// slices with all block loads issued before any is used.
__device__ __forceinline__ void stage_attn_out(const MegaArgs& a, float* xs, float* wsm) {
    const int nb_max = a.nblk_max;
    for (int t = threadIdx.x; t < a.B * NQ; t += mk::NCT) {
        const int b = t / NQ, h = t % NQ;
        const int nblk = (a.pos[b] + 1 + KVB - 1) / KVB;
        const float* p = a.part + ((size_t)b * NQ + h) * nb_max * PART_STRIDE;
        float M = -INFINITY;
        for (int j = 0; j < nblk; ++j) M = fmaxf(M, __ldcg(p + j * PART_STRIDE + HD));
        float lsum = 0.f;
        for (int j = 0; j < nblk; ++j) {
            const float mj = __ldcg(p + j * PART_STRIDE + HD);
            const float f = (mj == -INFINITY) ? 0.f : exp2f(mj - M);
            wsm[t * mk::MAXSPLIT + j] = f;
            lsum += __ldcg(p + j * PART_STRIDE + HD + 1) * f;
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        for (int j = 0; j < nblk; ++j) wsm[t * mk::MAXSPLIT + j] *= inv;
    }
    named_sync();
    for (int t = threadIdx.x; t < a.B * NQ * (HD / 4); t += mk::NCT) {
        const int bh = t / (HD / 4), e4 = t % (HD / 4);
        const int b = bh / NQ;
        const int nblk = (a.pos[b] + 1 + KVB - 1) / KVB;
        const float4* p = reinterpret_cast<const float4*>(a.part + (size_t)bh * nb_max * PART_STRIDE);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j0 = 0; j0 < nblk; j0 += 8) {
            float4 v[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                if (j0 + jj < nblk) v[jj] = __ldcg(reinterpret_cast<const float4*>(
                                        reinterpret_cast<const float*>(p) + (size_t)(j0 + jj) * PART_STRIDE) + e4);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                if (j0 + jj < nblk) {
                    const float w = wsm[bh * mk::MAXSPLIT + j0 + jj];
                    acc.x += w * v[jj].x; acc.y += w * v[jj].y; acc.z += w * v[jj].z; acc.w += w * v[jj].w;
                }
        }
        *reinterpret_cast<float4*>(xs + (size_t)bh * HD + e4 * 4) = acc;
    }
}

// ---------------------------------------------------------------- the kernel
template <int B>
__global__ void __launch_bounds__(mk::NT, 1) k_decode_mega(const __grid_constant__ MegaArgs a) {
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* ring_mem = smem;
    float* xs = reinterpret_cast<float*>(smem + mk::RING);
    float* att = reinterpret_cast<float*>(smem + mk::RING + mk::XS_BYTES);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + mk::RING + mk::XS_BYTES + mk::ATT_FLOATS * 4);
    uint64_t* empty = full + mk::NSLOT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < mk::NSLOT; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, mk::NCW);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == mk::NCW) {
        // ------------------------------------------------ producer: weight stream
        if (lane == 0) {
            Ring ring;
            unsigned long long ends[mk::NSLOT];
            unsigned long long tail = 0;
            uint32_t consumed = 0;
            bool ok = true;
            for (int l = 0; l <= a.n_layers && ok; ++l) {
                const int nops = (l == a.n_layers) ? (a.head ? 1 : 0) : 4;
                for (int o = 0; o < nops && ok; ++o) {
                    const OpDesc d = op_desc(a, l, o);
                    int r0, r1;
                    cta_rows(d.N, blockIdx.x, gridDim.x, r0, r1);
                    const int rpc = rows_per_chunk(d.K);
                    for (int rc = r0; rc < r1 && ok; rc += rpc) {
                        const int nr = min(rpc, r1 - rc);
                        const uint32_t bytes = (uint32_t)nr * d.K * 2;
                        const uint32_t k = ring.k;
                        const unsigned long long h0 = ring.head;
                        const uint32_t p = ring.place(bytes);
                        // free ring space and the slot: wait for the oldest chunks in order
                        while (ok && (k - consumed >= (uint32_t)mk::NSLOT || ring.head - tail > (unsigned long long)mk::RING)) {
                            const uint32_t s = consumed % mk::NSLOT;
                            ok = mbar_wait(empty + s, (consumed / mk::NSLOT) & 1, a);
                            if (ok) { tail = ends[s]; ++consumed; }
                        }
                        (void)h0;
                        if (!ok) break;
                        const uint32_t slot = k % mk::NSLOT;
                        ends[slot] = ring.head;
                        ring.k++;
                        mbar_expect_tx(full + slot, bytes);
                        bulk_g2s(ring_mem + p, d.W + (size_t)rc * d.K, bytes, full + slot);
                    }
                }
            }
            // drain: wait for every copy still in flight before leaving
            while (consumed < ring.k) {
                const uint32_t s = consumed % mk::NSLOT;
                if (ok) {
                    if (!mbar_wait(empty + s, (consumed / mk::NSLOT) & 1, a)) ok = false;
                } else {
                    // aborted: wait (bounded) for the copy itself to land
                    const unsigned long long t0 = gtime();
                    while (!mbar_try(full + s, (consumed / mk::NSLOT) & 1) && gtime() - t0 < mk::TIMEOUT_NS) {
                    }
                }
                ++consumed;
            }
        }
        return;
    }

    // ---------------------------------------------------- consumers
    Ring ring;
    int bk = 0;  // grid barriers passed
#define STAMP(i)                                                                                  \
    do {                                                                                          \
        if (a.trace && threadIdx.x == 0)                                                          \
            a.trace[((size_t)blockIdx.x * a.n_layers + l) * mk::NSTAMP + (i)] = gtime();         \
    } while (0)
    // per-step prologue (CTA 0): page-table entries for new blocks, argmax reset
    if (blockIdx.x == 0 && threadIdx.x < a.n_upd) const_cast<int32_t*>(a.page_table)[a.upd_idx[threadIdx.x]] = a.upd_val[threadIdx.x];
    if (blockIdx.x == 0 && threadIdx.x < B) a.amax[threadIdx.x] = 0ull;
    for (int l = 0; l < a.n_layers; ++l) {
        STAMP(0);
        // ---- QKV
        if (l == 0) {
            // embedding sum -> global h (CTA 0) and every CTA's normed input
            float* hrow = xs + B * 1024;  // scratch after the input rows
            stage_embed(a, hrow);
            named_sync();
            // norm from the smem copy
            if (warp < B) {
                float ss = 0.f;
                for (int c = lane; c < HID; c += 32) ss += hrow[warp * HID + c] * hrow[warp * HID + c];
                ss = warp_sum(ss);
                const float r = rsqrtf(ss * (1.f / HID) + a.eps);
                for (int c = lane; c < HID; c += 32)
                    xs[warp * HID + c] = hrow[warp * HID + c] * r * bf2f(a.L[0].in_norm[c]);
            }
        } else {
            stage_norm(a, a.h, a.L[l].in_norm, xs);
        }
        named_sync();
        consume_op<B>(a, l, 0, ring, ring_mem, full, empty, xs);
        STAMP(1);
        grid_sync(a, bk);
        STAMP(2);
        // ---- attention units (b, g, block j)
        {
            int u = 0;
            for (int b = 0; b < B; ++b) {
                const int nblk = (a.pos[b] + 1 + KVB - 1) / KVB;
                for (int g = 0; g < NKV; ++g)
                    for (int j = 0; j < nblk; ++j, ++u)
                        if (u % (int)gridDim.x == (int)blockIdx.x) attn_unit(a, l, b, g, j, att, u < (int)gridDim.x);
            }
        }
        STAMP(3);
        grid_sync(a, bk);
        STAMP(4);
        // ---- o_proj + residual
        stage_attn_out(a, xs, att);
        named_sync();
        STAMP(5);
        consume_op<B>(a, l, 1, ring, ring_mem, full, empty, xs);
        STAMP(6);
        grid_sync(a, bk);
        STAMP(7);
        // ---- gate/up + SwiGLU
        stage_norm(a, a.h, a.L[l].post_norm, xs);
        named_sync();
        consume_op<B>(a, l, 2, ring, ring_mem, full, empty, xs);
        STAMP(8);
        grid_sync(a, bk);
        STAMP(9);
        // ---- down + residual
        for (int t = threadIdx.x; t < B * a.ffn / 4; t += mk::NCT)
            reinterpret_cast<float4*>(xs)[t] = __ldcg(reinterpret_cast<const float4*>(a.m) + t);
        named_sync();
        consume_op<B>(a, l, 3, ring, ring_mem, full, empty, xs);
        STAMP(10);
        grid_sync(a, bk);
        STAMP(11);
    }
#undef STAMP
    // ---- final norm + head + argmax
    if (a.head) {
        stage_norm(a, a.h, a.final_norm, xs);
        named_sync();
        consume_op<B>(a, a.n_layers, 0, ring, ring_mem, full, empty, xs);
        if (a.argmax_out) {
            grid_sync(a, bk);
            if (blockIdx.x == 0 && threadIdx.x < B)
                a.argmax_out[(size_t)threadIdx.x * a.argmax_stride] =
                    (int32_t)(0xFFFFFFFFu - (uint32_t)(a.amax[threadIdx.x] & 0xFFFFFFFFull));
        }
    }
}

// Number of grid barriers one launch performs (the host advances the counter base by this x G).
int mega_barriers(int n_layers, bool head, bool argmax) { return 5 * n_layers + ((head && argmax) ? 1 : 0); }

int mega_smem_bytes() { return mk::SMEM; }

template <int B>
static cudaError_t launch_b(const MegaArgs& a, int grid, cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_decode_mega<B>, cudaFuncAttributeMaxDynamicSharedMemorySize, mk::SMEM);
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(mk::NT);
    cfg.dynamicSmemBytes = mk::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_decode_mega<B>, a);
}

cudaError_t launch_decode_mega(const MegaArgs& a, int grid, cudaStream_t st) {
    switch (a.B) {
        case 1: return launch_b<1>(a, grid, st);
        case 2: return launch_b<2>(a, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

// Largest grid the cooperative launch accepts (one CTA per SM is the design).
int mega_max_grid() {
    int dev = 0, sms = 0, per = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(k_decode_mega<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, mk::SMEM);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_decode_mega<1>, mk::NT, mk::SMEM);
    return per >= 1 ? sms : 0;
}

}  // namespace ttsbb
