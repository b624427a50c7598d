// Persistent small-batch decode step (B <= 2) with flag-in-data exchanges.
//
// One cooperative launch, one CTA per SM, runs the whole 28-layer step. Each
// CTA owns fixed row slices of every weight matrix; a producer warp streams
// them (cp.async.bulk + mbarriers) into a shared-memory ring that runs ahead
// of the eight consumer warps. Between the dependent phases of a layer the
// CTAs exchange vectors through global memory in 8-byte words that carry the
// value and an epoch tag together: a reader polls the words it needs until
// every tag shows the current epoch, so one exchange costs one write-to-read
// latency instead of a grid barrier plus a read round trip. Per layer:
//   h (all rows)  -> norm -> QKV rows          -> q/k/v words
//   q/k/v of one KV head group -> attention unit (one cache block) -> partial words
//   all partials  -> merge -> o_proj rows       -> own residual rows -> h words
//   h (all rows)  -> norm -> gate/up rows       -> SwiGLU words
//   SwiGLU (all)  -> down rows                  -> own residual rows -> h words
// Exchange buffers alternate by layer parity; epochs grow monotonically across
// launches (the host passes the base), so stale words never match. Each CTA
// keeps its own residual rows on chip. Every wait is bounded (timeout_ns): on
// timeout the kernel raises the error word and a shared abort flag, after
// which all waits return at once and the kernel runs to its end.
#include "mega.cuh"

namespace ttsbb {

namespace ll {
constexpr int NCW = 8;
constexpr int NCT = NCW * 32;
constexpr int NT = NCT + 32;
constexpr int RING = 176 * 1024;
constexpr int NSLOT = 16;
constexpr int CHUNK = 34 * 1024;             // ring chunk budget: 16 padded rows of K = 1024
constexpr int ROW_PAD = 32;                  // bytes after each weight row in the ring (conflict-free fragment loads)
constexpr int XF_BYTES = mk::MAXB * 3072 * 2 * 2;  // staged activations: bf16 high + low part per value
constexpr int OWN_MAX = 32;                 // own residual rows per CTA (>= ceil(1024 / G) rounded to pairs)
constexpr int MAXSPLIT = 64;                // cache blocks per sequence (4096 tokens)
constexpr int ATT_UNIT = NCW * (2 * HD + 4) + 2 * HD;
constexpr int ATT_MERGE = 2 * mk::MAXB * NQ * MAXSPLIT;
constexpr int ATT_FLOATS = ATT_UNIT > ATT_MERGE ? ATT_UNIT : ATT_MERGE;
constexpr int PART_FLOATS = NCW * 64 * mk::MAXB;  // per-warp partial sums of one op ([KS][64 rows][B])
constexpr int SMEM = RING + XF_BYTES + mk::MAXB * OWN_MAX * 4 + ATT_FLOATS * 4 + PART_FLOATS * 4 + 2 * NSLOT * 8 + 64;
}  // namespace ll

// ---------------------------------------------------------------- small PTX helpers
__device__ __forceinline__ uint32_t l_su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long l_time() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void l_mbar_init(uint64_t* b, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(l_su32(b)), "r"(count));
}
__device__ __forceinline__ bool l_mbar_try(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(l_su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Non-blocking test of a phase (cheaper than try_wait when it has completed).
__device__ __forceinline__ bool l_mbar_test(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(l_su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void l_named_sync() { asm volatile("bar.sync 1, %0;" ::"n"(ll::NCT) : "memory"); }

__device__ __forceinline__ bool l_aborted(const MegaArgs& a) { return *reinterpret_cast<volatile int*>(a.abort_flag) != 0; }
__device__ __forceinline__ void l_raise(const MegaArgs& a) {
    set_err(a.err, ERR_TIMEOUT);
    atomicExch(a.abort_flag, 1);
}

// try_wait with a suspend-time hint: the thread sleeps in hardware until the
// phase completes or the hint (ns) elapses, leaving issue slots to the consumers.
__device__ __forceinline__ bool l_mbar_try_sleep(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(l_su32(b)), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}
// Producer-side bounded wait (sleeping between checks).
__device__ __forceinline__ bool l_mbar_wait_sleep(uint64_t* b, uint32_t parity, const MegaArgs& a) {
    if (l_mbar_try(b, parity)) return true;
    const unsigned long long t0 = l_time();
    for (;;) {
        if (l_mbar_try_sleep(b, parity)) return true;
        if (l_aborted(a)) return false;
        if (l_time() - t0 > a.timeout_ns) { l_raise(a); return false; }
    }
}
__device__ __forceinline__ bool l_mbar_wait(uint64_t* b, uint32_t parity, const MegaArgs& a) {
    if (l_mbar_test(b, parity)) return true;
    const unsigned long long t0 = l_time();
    for (uint32_t i = 0;; ++i) {
        if (l_mbar_try(b, parity)) return true;
        if ((i & 63) == 63) {
            if (l_aborted(a)) return false;
            if (l_time() - t0 > a.timeout_ns) { l_raise(a); return false; }
        }
    }
}

// 8-byte exchange word: low 32 bits the float, high 32 bits the epoch.
__device__ __forceinline__ void ll_put(unsigned long long* p, float v, uint32_t ep) {
    const unsigned long long w = ((unsigned long long)ep << 32) | (unsigned long long)__float_as_uint(v);
    asm volatile("st.global.cg.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ unsigned long long ll_ld(const unsigned long long* p) {
    unsigned long long w;
    asm volatile("ld.global.cg.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}
__device__ __forceinline__ void ll_ld2(const unsigned long long* p, unsigned long long& w0, unsigned long long& w1) {
    asm volatile("ld.global.cg.v2.u64 {%0, %1}, [%2];" : "=l"(w0), "=l"(w1) : "l"(p) : "memory");
}
// Wait until words w[0..n) (loaded from p[0..n)) all carry epoch ep: the
// caller issues every load first, so one exchange costs one round trip;
// stale words are reloaded individually (bounded).
template <int N>
__device__ __forceinline__ void ll_settle(unsigned long long (&w)[N], const unsigned long long* const (&p)[N], uint32_t ep,
                                          const MegaArgs& a) {
    bool ok = true;
#pragma unroll
    for (int i = 0; i < N; ++i) ok &= (uint32_t)(w[i] >> 32) == ep;
    if (ok) return;
    // Reissue every stale word each round (one round trip per check; the
    // whole exchange is a few KB per CTA, so the L2 request rate stays low).
    const unsigned long long t0 = l_time();
    for (uint32_t it = 0;; ++it) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            if ((uint32_t)(w[i] >> 32) != ep) w[i] = ll_ld(p[i]);
        ok = true;
#pragma unroll
        for (int i = 0; i < N; ++i) ok &= (uint32_t)(w[i] >> 32) == ep;
        if (ok) return;
        if ((it & 15) == 15) {
            if (l_aborted(a)) return;
            if (l_time() - t0 > a.timeout_ns) { l_raise(a); return; }
        }
    }
}
// ll_settle with the address of word i computed by addr(i) instead of stored.
template <int N, typename Addr>
__device__ __forceinline__ void ll_settle_f(unsigned long long (&w)[N], Addr addr, uint32_t ep, const MegaArgs& a) {
    bool ok = true;
#pragma unroll
    for (int i = 0; i < N; ++i) ok &= (uint32_t)(w[i] >> 32) == ep;
    if (ok) return;
    const unsigned long long t0 = l_time();
    for (uint32_t it = 0;; ++it) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            if ((uint32_t)(w[i] >> 32) != ep) w[i] = ll_ld(addr(i));
        ok = true;
#pragma unroll
        for (int i = 0; i < N; ++i) ok &= (uint32_t)(w[i] >> 32) == ep;
        if (ok) return;
        if ((it & 15) == 15) {
            if (l_aborted(a)) return;
            if (l_time() - t0 > a.timeout_ns) { l_raise(a); return; }
        }
    }
}
__device__ __forceinline__ float ll_val(unsigned long long w) { return __uint_as_float((uint32_t)w); }

// ---------------------------------------------------------------- schedule (same as the producer)
struct LOp {
    const bf16* W;
    int N, K;
};
__device__ __forceinline__ LOp l_op(const MegaArgs& a, int l, int o) {
    if (l == a.n_layers) return {a.head, a.head_rows, HID};
    const MegaLayer& L = a.L[l];
    switch (o) {
        case 0: return {L.wqkv, QKV, HID};
        case 1: return {L.wo, HID, NQ * HD};
        case 2: return {L.wgu, 2 * a.ffn, HID};
        default: return {L.wd, HID, a.ffn};
    }
}
__device__ __forceinline__ void l_rows(int N, int c, int G, int& r0, int& r1) {
    const unsigned pairs = (unsigned)N / 2;  // pairs * (c + 1) < 2^32 for every shape here
    r0 = (int)(pairs * (unsigned)c / (unsigned)G) * 2;
    r1 = (int)(pairs * (unsigned)(c + 1) / (unsigned)G) * 2;
}
// weight rows per ring chunk for a K-column matrix (even, 2..16), rows padded by ROW_PAD
__host__ __device__ constexpr int l_rpc(int K) {
    return ((ll::CHUNK / (K * 2 + ll::ROW_PAD)) & ~1) < 2 ? 2
         : (((ll::CHUNK / (K * 2 + ll::ROW_PAD)) & ~1) > 16 ? 16 : ((ll::CHUNK / (K * 2 + ll::ROW_PAD)) & ~1));
}
struct LRing {
    unsigned long long head = 0;  // bytes placed so far, including skipped ring tails
    uint32_t pos = 0;             // offset of the next placement in the ring
    uint32_t k = 0;               // chunks placed so far
    __device__ __forceinline__ uint32_t place(uint32_t bytes) {
        if (pos + bytes > (uint32_t)ll::RING) {
            head += ll::RING - pos;
            pos = 0;
        }
        const uint32_t p = pos;
        pos += bytes;
        head += bytes;
        return p;
    }
};

// Exchange buffers inside MegaArgs::xbuf (unsigned long long words):
//   h : [2][XR][MAXB][HID]   q/k/v : [2][MAXB][QKV]   m : [2][XR][MAXB][3072]
//   part : [2][XR][MAXB][16][nblk_max][132]
// Every CTA reads all of h, m and the attention partials, so their writers
// store XR copies and CTA c reads copy c % XR: fewer readers per L2 line, and
// a shorter exchange.
struct XBufs {
    unsigned long long *h, *q, *m, *p;
};
__device__ __forceinline__ XBufs l_bufs(const MegaArgs& a) {
    XBufs x;
    x.h = a.xbuf;
    x.q = x.h + 2 * LL_XR * mk::MAXB * HID;
    x.m = x.q + 2 * mk::MAXB * QKV;
    x.p = x.m + 2 * LL_XR * mk::MAXB * 3072;
    return x;
}
constexpr size_t XH_REP = (size_t)mk::MAXB * HID, XM_REP = (size_t)mk::MAXB * 3072;
// h version v: base of the copies, and the copy this CTA reads
__device__ __forceinline__ unsigned long long* xh_base(const XBufs& X, int v) { return X.h + (size_t)(v & 1) * LL_XR * XH_REP; }
__device__ __forceinline__ unsigned long long* xh_mine(const XBufs& X, int v) { return xh_base(X, v) + (blockIdx.x % LL_XR) * XH_REP; }
__device__ __forceinline__ unsigned long long* xm_base(const XBufs& X, int l) { return X.m + (size_t)(l & 1) * LL_XR * XM_REP; }
__device__ __forceinline__ unsigned long long* xm_mine(const XBufs& X, int l) { return xm_base(X, l) + (blockIdx.x % LL_XR) * XM_REP; }
__device__ __forceinline__ size_t xp_rep(const MegaArgs& a) { return (size_t)mk::MAXB * NQ * a.nblk_max * PART_STRIDE; }
__device__ __forceinline__ unsigned long long* xp_base(const MegaArgs& a, const XBufs& X, int l) {
    return X.p + (size_t)(l & 1) * LL_XRP * xp_rep(a);
}

// Epoch of each exchange: h version v (0 = layer-0 input, 2l+1 after o_proj, 2l+2 after down).
__device__ __forceinline__ uint32_t ep_h(const MegaArgs& a, int v) { return a.ep_base + 3u * (uint32_t)v; }
__device__ __forceinline__ uint32_t ep_q(const MegaArgs& a, int l) { return a.ep_base + 6u * (uint32_t)l + 1u; }
__device__ __forceinline__ uint32_t ep_p(const MegaArgs& a, int l) { return a.ep_base + 6u * (uint32_t)l + 2u; }
__device__ __forceinline__ uint32_t ep_m(const MegaArgs& a, int l) { return a.ep_base + 6u * (uint32_t)l + 4u; }

// ---------------------------------------------------------------- consumer pieces
// Staged activations for the tensor-core matrix-vector products: value x of
// token b, column k of a K-column operand is kept as x ~= hi + lo (two bf16,
// so the products keep ~16 mantissa bits) in the column order of the mma
// fragments: 16-column step, lane quad (4 columns), part (hi, lo), element.
__device__ __forceinline__ int xf_idx(int K, int b, int k, int part) {
    return b * K * 2 + (k >> 4) * 32 + ((k >> 2) & 3) * 8 + part * 4 + (k & 3);
}
__device__ __forceinline__ uint32_t xf_split2(float v0, float v1, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
    lo = *reinterpret_cast<const uint32_t*>(&l);
    return *reinterpret_cast<const uint32_t*>(&h);
}
// columns k, k+1 (k even)
__device__ __forceinline__ void xf_put2(bf16* xf, int K, int b, int k, float v0, float v1) {
    uint32_t lo;
    const uint32_t hi = xf_split2(v0, v1, lo);
    *reinterpret_cast<uint32_t*>(xf + xf_idx(K, b, k, 0)) = hi;
    *reinterpret_cast<uint32_t*>(xf + xf_idx(K, b, k, 1)) = lo;
}
// columns k..k+3 (k a multiple of 4)
__device__ __forceinline__ void xf_put4(bf16* xf, int K, int b, int k, float v0, float v1, float v2, float v3) {
    uint2 hi, lo;
    hi.x = xf_split2(v0, v1, lo.x);
    hi.y = xf_split2(v2, v3, lo.y);
    *reinterpret_cast<uint2*>(xf + xf_idx(K, b, k, 0)) = hi;
    *reinterpret_cast<uint2*>(xf + xf_idx(K, b, k, 1)) = lo;
}

// xf[b][k] = rmsnorm(h_v[b]) * gamma (staged), h read from the exchange words of version v.
template <int B>
__device__ __forceinline__ void l_stage_norm(const MegaArgs& a, const unsigned long long* hx, uint32_t ep,
                                             const bf16* gamma, bf16* xf, float* red) {
    const int t = threadIdx.x;
    // the gains do not depend on the exchange: their loads go first
    const uint32_t g0 = __ldg(reinterpret_cast<const unsigned int*>(gamma + 2 * t));
    const uint32_t g1 = __ldg(reinterpret_cast<const unsigned int*>(gamma + 512 + 2 * t));
    // thread t: elements 2t, 2t+1 and 512+2t, 512+2t+1 of each token row, so
    // a warp's 16-byte loads cover 512 contiguous bytes (all loads issued before any check)
    unsigned long long w[B * 4];
#pragma unroll
    for (int b = 0; b < B; ++b) {
        ll_ld2(hx + (size_t)b * HID + 2 * t, w[b * 4], w[b * 4 + 1]);
        ll_ld2(hx + (size_t)b * HID + 512 + 2 * t, w[b * 4 + 2], w[b * 4 + 3]);
    }
    ll_settle_f(w, [&](int i) { return hx + (size_t)(i >> 2) * HID + ((i & 2) ? 512 : 0) + 2 * t + (i & 1); }, ep, a);
    const float g4[4] = {__uint_as_float(g0 << 16), __uint_as_float(g0 & 0xFFFF0000u),
                         __uint_as_float(g1 << 16), __uint_as_float(g1 & 0xFFFF0000u)};
    float v[B][4];
#pragma unroll
    for (int b = 0; b < B; ++b) {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            v[b][e] = ll_val(w[b * 4 + e]);
            ss += v[b][e] * v[b][e];
        }
        ss = warp_sum(ss);
        if ((t & 31) == 0) red[b * ll::NCW + (t >> 5)] = ss;
    }
    l_named_sync();
#pragma unroll
    for (int b = 0; b < B; ++b) {
        float ss = 0.f;
#pragma unroll
        for (int wi = 0; wi < ll::NCW; ++wi) ss += red[b * ll::NCW + wi];
        const float r = rsqrtf(ss * (1.f / HID) + a.eps);
        xf_put2(xf, HID, b, 2 * t, v[b][0] * g4[0] * r, v[b][1] * g4[1] * r);
        xf_put2(xf, HID, b, 512 + 2 * t, v[b][2] * g4[2] * r, v[b][3] * g4[3] * r);
    }
}

__device__ __forceinline__ void l_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                      uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The k-loop of l_consume: the warp's NK column steps over TT tiles (TT and
// LASTHI fixed at compile time, so the loads carry no branch and schedule
// freely). LASTHI = the last tile's rows 8..15 hold rows of the slice (else
// they are zero and not loaded).
template <int B, int MAXT, int NK, int TT, bool LASTHI>
__device__ __forceinline__ void l_mma_loop(float (&d)[MAXT][2][4], const int (&ra)[MAXT][2], const unsigned char* ring_mem,
                                           const bf16* xb, uint32_t bmask) {
    static_assert(NK % 2 == 0 && TT <= MAXT, "column steps per warp must be even");
#pragma unroll
    for (int tt = 0; tt < MAXT; ++tt)
#pragma unroll
        for (int q = 0; q < 2; ++q) d[tt][q][0] = d[tt][q][1] = d[tt][q][2] = d[tt][q][3] = 0.f;
#pragma unroll 4
    for (int s = 0; s < NK; ++s) {
        uint2 bv = *reinterpret_cast<const uint2*>(xb + s * 32);
        bv.x &= bmask;
        bv.y &= bmask;
#pragma unroll
        for (int tt = 0; tt < TT; ++tt) {
            const uint2 lo = *reinterpret_cast<const uint2*>(ring_mem + ra[tt][0] + s * 32);
            const uint2 hi = (LASTHI || tt + 1 < TT) ? *reinterpret_cast<const uint2*>(ring_mem + ra[tt][1] + s * 32)
                                                    : make_uint2(0u, 0u);
            l_mma(d[tt][s & 1], lo.x, hi.x, lo.y, hi.y, bv.x, bv.y);
        }
    }
}
template <int B, int MAXT, int NK, int TT>
__device__ __forceinline__ void l_mma_dispatch(float (&d)[MAXT][2][4], const int (&ra)[MAXT][2], const unsigned char* ring_mem,
                                               const bf16* xb, uint32_t bmask, int T, bool lasthi) {
    if constexpr (TT <= MAXT) {
        if (T == TT) {
            if (lasthi) l_mma_loop<B, MAXT, NK, TT, true>(d, ra, ring_mem, xb, bmask);
            else l_mma_loop<B, MAXT, NK, TT, false>(d, ra, ring_mem, xb, bmask);
        } else {
            l_mma_dispatch<B, MAXT, NK, TT + 1>(d, ra, ring_mem, xb, bmask, T, lasthi);
        }
    }
}

// Consume this CTA's chunks of one op: rows r0..r1 of a K-column matrix,
// results to `sink(b, row, v_row, true, v_row+1, r0)` per even row.
// Tensor cores (m16n8k16, bf16 in, fp32 accumulate): the rows form 16-row
// tiles (A, from the ring, rows padded so fragment loads are conflict-free);
// the staged activations are the B operand, column 2b the high and 2b+1 the
// low part of token b. Columns are permuted consistently in A and B so each
// thread's fragment is one 8-byte load: within every 16 columns, the four
// k-slots of lane quad t are the columns 4t..4t+3. Warp w takes columns
// [w K/8, (w+1) K/8) of every tile; its partial sums go to `part` and, after a
// barrier, threads add the eight partials of each row pair in order and call
// the sink. Callers put a barrier between consecutive calls (the partial
// buffer is reused).
constexpr int MAXC = 4;        // chunks per op per CTA: holds for grids >= 96 CTAs (gate/up 6144 rows: <= 64 rows = 4 chunks)
constexpr int PART_ROWS = 64;  // most rows of one op in one CTA (grids >= 96 CTAs, N <= 6144)
template <int B, int K, int MAXT, typename Sink>
__device__ __forceinline__ void l_consume(const MegaArgs& a, int l, int2 rows, LRing& ring, unsigned char* ring_mem,
                                          uint64_t* full, uint64_t* empty, const bf16* xf, float* part, int stamp,
                                          Sink sink) {
    // MAXT = most 16-row tiles of this op in one CTA (grids >= LL_MIN_GRID)
    constexpr int RPC = l_rpc(K), RS = K * 2 + ll::ROW_PAD, NK = K / ll::NCW / 16;
    static_assert(MAXT * 16 <= PART_ROWS, "tiles exceed the partial buffer");
    static_assert(K % (ll::NCW * 16) == 0, "columns must split into 16-column steps per warp");
    // rows = this CTA's slice [r0, r1) of the op (l_rows); K is the op's column count (the host checks both)
    const int r0 = rows.x, R = rows.y - rows.x, T = (R + 15) >> 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tq = lane & 3;
    // ring chunks of this op, in the producer's order
    uint32_t off[MAXC] = {0u, 0u, 0u, 0u};
    const uint32_t slot0 = ring.k;
    int nc = 0;
    for (int rc = 0; rc < R && nc < MAXC; rc += RPC, ++nc) {
        const uint32_t p = ring.place((uint32_t)min(RPC, R - rc) * RS);
#pragma unroll
        for (int c = 0; c < MAXC; ++c)
            if (c == nc) off[c] = p;
        ring.k++;
    }
    // ring byte offsets of this thread's A rows (16 t + g and 16 t + g + 8); rows past the
    // slice read row R - 1 instead (their results are dropped), so the loads need no branch
    int ra[MAXT][2];
#pragma unroll
    for (int tt = 0; tt < MAXT; ++tt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = min(16 * tt + g + 8 * h, R - 1), c = i / RPC, rin = i - c * RPC;
            const uint32_t base = c == 0 ? off[0] : c == 1 ? off[1] : c == 2 ? off[2] : off[3];
            ra[tt][h] = (int)(base + (uint32_t)rin * RS) + (warp * NK * 16 + tq * 4) * 2;
        }
    for (int c = 0; c < nc; ++c) l_mbar_wait(full + (slot0 + c) % ll::NSLOT, ((slot0 + c) / ll::NSLOT) & 1, a);
    // profiling stamps of this op (slot base `stamp`): +0 ring waits done, +1+w warp w's products done, +9 sink done
    if (stamp >= 0 && a.trace && threadIdx.x == 0) a.trace[((size_t)blockIdx.x * a.n_layers + l) * TRACE_STRIDE + stamp] = l_time();
    // two accumulator sets per tile (even / odd column steps) halve the mma dependency chain
    float d[MAXT][2][4];
    // B fragment: lanes g < 2B carry token g / 2 (high part for even g, low for odd); the others
    // load a valid address and are masked to zero
    const int gb = min(g, 2 * B - 1);
    const bf16* xb = xf + (gb >> 1) * K * 2 + (gb & 1) * 4 + tq * 8 + warp * NK * 32;
    const uint32_t bmask = g < 2 * B ? 0xffffffffu : 0u;
#pragma unroll
    for (int tt = 0; tt < MAXT; ++tt)
#pragma unroll
        for (int q = 0; q < 2; ++q) d[tt][q][0] = d[tt][q][1] = d[tt][q][2] = d[tt][q][3] = 0.f;
    // tile count and whether the last tile's rows 8..15 hold rows of the slice, chosen once
    l_mma_dispatch<B, MAXT, NK, 1>(d, ra, ring_mem, xb, bmask, T, R > 16 * (T - 1) + 8);
    // thread (g, tq < B) holds rows 16 t + g (d0 + d1) and 16 t + g + 8 (d2 + d3) of token tq
    if (tq < B) {
#pragma unroll
        for (int tt = 0; tt < MAXT; ++tt) {
            const int i = 16 * tt + g;
            if (i < R) part[(warp * PART_ROWS + i) * B + tq] = (d[tt][0][0] + d[tt][0][1]) + (d[tt][1][0] + d[tt][1][1]);
            if (i + 8 < R) part[(warp * PART_ROWS + i + 8) * B + tq] = (d[tt][0][2] + d[tt][0][3]) + (d[tt][1][2] + d[tt][1][3]);
        }
    }
    __syncwarp();
    if (stamp >= 0 && a.trace && lane == 0)
        a.trace[((size_t)blockIdx.x * a.n_layers + l) * TRACE_STRIDE + stamp + 1 + warp] = l_time();
    if (lane == 0)
        for (int c = 0; c < nc; ++c)
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(l_su32(empty + (slot0 + c) % ll::NSLOT)) : "memory");
    l_named_sync();
    for (int i = threadIdx.x; i < (R / 2) * B; i += ll::NCT) {
        const int pr = i / B, b = i - pr * B, row = 2 * pr;
        float v0 = 0.f, v1 = 0.f;
#pragma unroll
        for (int k = 0; k < ll::NCW; ++k) {
            v0 += part[(k * PART_ROWS + row) * B + b];
            v1 += part[(k * PART_ROWS + row + 1) * B + b];
        }
        sink(b, r0 + row, v0, true, v1, r0);
    }
    if (stamp >= 0 && a.trace && threadIdx.x == 0) a.trace[((size_t)blockIdx.x * a.n_layers + l) * TRACE_STRIDE + stamp + 9] = l_time();
}

// q/k RMSNorm + RoPE of one head, 4 elements per lane (RoPE partner lane ^ 16);
// g4 = the lane's 4 gains, c4 / s4 = its 4 cos / sin table entries.
__device__ __forceinline__ void l_norm_rope4(float* v, const float* g4, const float4& c4, const float4& s4,
                                             const MegaArgs& a, int lane) {
    const float ss = warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]);
    const float r = rsqrtf(ss * (1.f / HD) + a.eps);
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = v[e] * r * g4[e];
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = __shfl_xor_sync(0xffffffffu, v[e], 16);
    const float ct[4] = {c4.x, c4.y, c4.z, c4.w}, st[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = (lane < 16) ? (v[e] * ct[e] - p[e] * st[e]) : (v[e] * ct[e] + p[e] * st[e]);
}
__device__ __forceinline__ void l_gain4(const bf16* gamma, int lane, float* g4) {
    const uint2 u = *reinterpret_cast<const uint2*>(gamma + lane * 4);
    g4[0] = __uint_as_float(u.x << 16); g4[1] = __uint_as_float(u.x & 0xFFFF0000u);
    g4[2] = __uint_as_float(u.y << 16); g4[3] = __uint_as_float(u.y & 0xFFFF0000u);
}

// Request the K and V tiles of this CTA's attention units (unit u = (b, g, block j),
// CTA c runs u = c, c + G, ...) at layer l into L2, ahead of the layer that reads them.
__device__ __forceinline__ void l_prefetch_kv(const MegaArgs& a, int l, int B, int nblk0, int nblk1) {
    const int units_b0 = NKV * nblk0, n_units = units_b0 + NKV * nblk1;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        int b = 0, r = u;
        if (B > 1 && r >= units_b0) { b = 1; r -= units_b0; }
        const int nblk = b == 0 ? nblk0 : nblk1;
        const int g = r / nblk, j = r - g * nblk;
        const int phys = j == nblk - 1 ? a.last_phys[b] : __ldcg(a.page_table + (size_t)a.slot[b] * a.mbps + j);
        const bf16* kb = a.pool + (size_t)l * a.layer_elems + ((size_t)phys * 2 * NKV + g) * KVB * HD;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(kb), "r"(KVB * HD * 2) : "memory");
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(kb + (size_t)NKV * KVB * HD), "r"(KVB * HD * 2)
                     : "memory");
    }
}

// Attention unit (b, g, block j): K/V of the block's old keys are loaded
// before the q/k/v words are polled; the owner of the last block also appends
// the new token. Writes the block's softmax partial words for heads 2g, 2g+1.
__device__ __forceinline__ void l_attn_unit(const MegaArgs& a, const XBufs& X, int l, int b, int g, int j, float* att) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (a.trace && threadIdx.x == 0) a.trace[((size_t)blockIdx.x * a.n_layers + l) * TRACE_STRIDE + 62] = l_time();
    const int pos = a.pos[b], L = pos + 1;
    const int nblk = (L + KVB - 1) / KVB;
    const bool last = (j == nblk - 1);
    const int phys = last ? a.last_phys[b] : __ldcg(a.page_table + (size_t)a.slot[b] * a.mbps + j);
    bf16* kb = a.pool + (size_t)l * a.layer_elems + ((size_t)phys * 2 * NKV + g) * KVB * HD;
    bf16* vb = kb + (size_t)NKV * KVB * HD;
    // old keys of this warp (keys 8w..8w+7 of the block), loaded ahead of the q/k/v exchange
    const int key0 = j * KVB + warp * 8;
    uint2 kr[8], vr[8];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const bool ok = key0 + kk < pos;  // the new token (position pos) comes from the exchange
        kr[kk] = ok ? __ldcg(reinterpret_cast<const uint2*>(kb + (size_t)(warp * 8 + kk) * HD + lane * 4)) : make_uint2(0u, 0u);
        vr[kk] = ok ? __ldcg(reinterpret_cast<const uint2*>(vb + (size_t)(warp * 8 + kk) * HD + lane * 4)) : make_uint2(0u, 0u);
    }
    float* sq = att + ll::NCW * (2 * HD + 4);  // [2][HD] scaled queries
    const unsigned long long* qx = X.q + ((size_t)(l & 1) * mk::MAXB + b) * QKV;
    const uint32_t eq = ep_q(a, l);
    __shared__ uint2 newk[HD / 4], newv[HD / 4];
    // inputs that do not depend on the exchange: gains and this position's RoPE entries
    float g4[4];
    l_gain4(warp < 2 ? a.L[l].qn : a.L[l].kn, lane, g4);
    const float4 c4 = *reinterpret_cast<const float4*>(a.cos_t + (size_t)pos * (HD / 2) + (lane & 15) * 4);
    const float4 s4 = *reinterpret_cast<const float4*>(a.sin_t + (size_t)pos * (HD / 2) + (lane & 15) * 4);
    auto poll4 = [&](const unsigned long long* src, float* v) {
        unsigned long long w[4];
        const unsigned long long* p[4] = {src, src + 1, src + 2, src + 3};
        ll_ld2(src, w[0], w[1]);
        ll_ld2(src + 2, w[2], w[3]);
        ll_settle(w, p, eq, a);
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = ll_val(w[e]);
    };
    if (warp < 2) {
        float v[4];
        poll4(qx + (2 * g + warp) * HD + lane * 4, v);
        l_norm_rope4(v, g4, c4, s4, a, lane);
        const float sc = rsqrtf((float)HD) * 1.4426950408889634f;
#pragma unroll
        for (int e = 0; e < 4; ++e) sq[warp * HD + lane * 4 + e] = v[e] * sc;
    } else if (warp == 2 && last) {
        float v[4];
        poll4(qx + NQ * HD + g * HD + lane * 4, v);
        l_norm_rope4(v, g4, c4, s4, a, lane);
        __nv_bfloat162 p0 = __floats2bfloat162_rn(v[0], v[1]), p1 = __floats2bfloat162_rn(v[2], v[3]);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t*>(&p0);
        o.y = *reinterpret_cast<uint32_t*>(&p1);
        *reinterpret_cast<uint2*>(kb + (size_t)(pos % KVB) * HD + lane * 4) = o;
        newk[lane] = o;
    } else if (warp == 3 && last) {
        float v[4];
        poll4(qx + NQ * HD + NKV * HD + g * HD + lane * 4, v);
        __nv_bfloat162 p0 = __floats2bfloat162_rn(v[0], v[1]), p1 = __floats2bfloat162_rn(v[2], v[3]);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t*>(&p0);
        o.y = *reinterpret_cast<uint32_t*>(&p1);
        *reinterpret_cast<uint2*>(vb + (size_t)(pos % KVB) * HD + lane * 4) = o;
        newv[lane] = o;
    }
    l_named_sync();
    if (a.trace && threadIdx.x == 0) a.trace[((size_t)blockIdx.x * a.n_layers + l) * TRACE_STRIDE + 60] = l_time();
    if (last && key0 <= pos && pos < key0 + 8) {  // this warp holds the new token's slot
        kr[pos - key0] = newk[lane];
        vr[pos - key0] = newv[lane];
    }
    float q0[4], q1[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) { q0[e] = sq[lane * 4 + e]; q1[e] = sq[HD + lane * 4 + e]; }
    float d[16];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const float k0 = __uint_as_float(kr[kk].x << 16), k1 = __uint_as_float(kr[kk].x & 0xFFFF0000u);
        const float k2 = __uint_as_float(kr[kk].y << 16), k3 = __uint_as_float(kr[kk].y & 0xFFFF0000u);
        d[kk] = q0[0] * k0 + q0[1] * k1 + q0[2] * k2 + q0[3] * k3;
        d[8 + kk] = q1[0] * k0 + q1[1] * k1 + q1[2] * k2 + q1[3] * k3;
    }
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
    const int kk0 = lane & 7;
    const float score = (key0 + kk0 < L) ? d[0] : -INFINITY;
    float mx = score;
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    const float pr = (mx == -INFINITY) ? 0.f : exp2f(score - mx);
    float ps = pr;
    ps += __shfl_xor_sync(0xffffffffu, ps, 1);
    ps += __shfl_xor_sync(0xffffffffu, ps, 2);
    ps += __shfl_xor_sync(0xffffffffu, ps, 4);
    const float m0 = __shfl_sync(0xffffffffu, mx, 0), m1 = __shfl_sync(0xffffffffu, mx, 8);
    const float l0 = __shfl_sync(0xffffffffu, ps, 0), l1 = __shfl_sync(0xffffffffu, ps, 8);
    float o0[4] = {0.f, 0.f, 0.f, 0.f}, o1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k2 = 0; k2 < 8; ++k2) {
        const float p0 = __shfl_sync(0xffffffffu, pr, k2), p1 = __shfl_sync(0xffffffffu, pr, 8 + k2);
        const float v0 = __uint_as_float(vr[k2].x << 16), v1 = __uint_as_float(vr[k2].x & 0xFFFF0000u);
        const float v2 = __uint_as_float(vr[k2].y << 16), v3 = __uint_as_float(vr[k2].y & 0xFFFF0000u);
        o0[0] += p0 * v0; o0[1] += p0 * v1; o0[2] += p0 * v2; o0[3] += p0 * v3;
        o1[0] += p1 * v0; o1[1] += p1 * v1; o1[2] += p1 * v2; o1[3] += p1 * v3;
    }
    float* wml = att + warp * (2 * HD + 4);
    if (lane == 0) { wml[2 * HD] = m0; wml[2 * HD + 1] = l0; wml[2 * HD + 2] = m1; wml[2 * HD + 3] = l1; }
#pragma unroll
    for (int e = 0; e < 4; ++e) { wml[lane * 4 + e] = o0[e]; wml[HD + lane * 4 + e] = o1[e]; }
    l_named_sync();
    {
        const int t = threadIdx.x, h2 = t >> 7, e = t & 127;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < ll::NCW; ++w) M = fmaxf(M, att[w * (2 * HD + 4) + 2 * HD + 2 * h2]);
        float lsum = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < ll::NCW; ++w) {
            const float* ww = att + w * (2 * HD + 4);
            const float mw = ww[2 * HD + 2 * h2];
            const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
            lsum += ww[2 * HD + 2 * h2 + 1] * f;
            acc += ww[h2 * HD + e] * f;
        }
        if (a.trace && threadIdx.x == 0) a.trace[((size_t)blockIdx.x * a.n_layers + l) * TRACE_STRIDE + 61] = l_time();
        unsigned long long* dst = xp_base(a, X, l) + (((size_t)b * NQ + 2 * g + h2) * a.nblk_max + j) * PART_STRIDE;
        const uint32_t ep = ep_p(a, l);
        const size_t rs = xp_rep(a);
#pragma unroll
        for (int rep = 0; rep < LL_XRP; ++rep) {
            ll_put(dst + rep * rs + e, acc, ep);
            if (e == 0) { ll_put(dst + rep * rs + HD, M, ep); ll_put(dst + rep * rs + HD + 1, lsum, ep); }
        }
    }
    l_named_sync();
}

// xf[b][h*128 + e] (staged) = merge of the block partial words of (b, h) in block order.
// Thread t owns E outputs of one (b, h), as E/4 groups of 4 spaced HD/(E/4)
// apart (so a warp's loads stay contiguous); per round it loads, for J
// blocks at once, each block's running max / sum and its outputs, waits
// once, and folds them in (online, block order kept).
template <int B>
__device__ __forceinline__ void l_stage_attn(const MegaArgs& a, const XBufs& X, int l, bf16* xf) {
    constexpr int E = B * NQ * HD / ll::NCT;  // outputs per thread
    constexpr int G4 = E / 4, GS = HD / G4;   // groups of 4 outputs, their spacing
    constexpr int J = B == 1 ? 3 : 2;         // cache blocks per poll round
    constexpr int W = 2 + E;                  // words per block
    constexpr int TPH = HD / E;               // threads per (b, h)
    const uint32_t ep = ep_p(a, l);
    const int t = threadIdx.x, bh = t / TPH, e0 = (t - bh * TPH) * 4, b = bh / NQ;
    const unsigned long long* base =
        xp_base(a, X, l) + (blockIdx.x % LL_XRP) * xp_rep(a) + (size_t)bh * a.nblk_max * PART_STRIDE;
    const int nblk = (a.pos[b] + 1 + KVB - 1) / KVB;
    float M = -INFINITY, lsum = 0.f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    for (int j0 = 0; j0 < nblk; j0 += J) {
        unsigned long long w[J * W];
        auto addr = [&](int i) {
            const int jj = i / W, k = i - jj * W;
            const unsigned long long* rec = base + (size_t)min(j0 + jj, nblk - 1) * PART_STRIDE;
            return k < 2 ? rec + HD + k : rec + e0 + ((k - 2) >> 2) * GS + ((k - 2) & 3);
        };
#pragma unroll
        for (int jj = 0; jj < J; ++jj) {
            const unsigned long long* rec = base + (size_t)min(j0 + jj, nblk - 1) * PART_STRIDE;
            ll_ld2(rec + HD, w[jj * W], w[jj * W + 1]);
#pragma unroll
            for (int g = 0; g < G4; ++g) {
                ll_ld2(rec + e0 + g * GS, w[jj * W + 2 + 4 * g], w[jj * W + 3 + 4 * g]);
                ll_ld2(rec + e0 + g * GS + 2, w[jj * W + 4 + 4 * g], w[jj * W + 5 + 4 * g]);
            }
        }
        ll_settle_f(w, addr, ep, a);
#pragma unroll
        for (int jj = 0; jj < J; ++jj) {
            if (j0 + jj >= nblk) break;
            const float mj = ll_val(w[jj * W]), lj = ll_val(w[jj * W + 1]);
            const float Mn = fmaxf(M, mj);
            const float fo = (M == -INFINITY) ? 0.f : exp2f(M - Mn);
            const float fj = (mj == -INFINITY) ? 0.f : exp2f(mj - Mn);
            lsum = lsum * fo + lj * fj;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = acc[e] * fo + ll_val(w[jj * W + 2 + e]) * fj;
            M = Mn;
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
    for (int g = 0; g < G4; ++g)
        xf_put4(xf, NQ * HD, b, (bh - b * NQ) * HD + e0 + g * GS, acc[4 * g] * inv, acc[4 * g + 1] * inv,
                acc[4 * g + 2] * inv, acc[4 * g + 3] * inv);
}

// ---------------------------------------------------------------- the kernel
template <int B>
__global__ void __launch_bounds__(ll::NT, 1) k_decode_ll(const __grid_constant__ MegaArgs a) {
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* ring_mem = smem;
    bf16* xf = reinterpret_cast<bf16*>(smem + ll::RING);     // staged activations of the current op
    float* hown = reinterpret_cast<float*>(smem + ll::RING + ll::XF_BYTES);  // [B][OWN_MAX]
    float* att = hown + mk::MAXB * ll::OWN_MAX;
    float* part = att + ll::ATT_FLOATS;
    uint64_t* full = reinterpret_cast<uint64_t*>(part + ll::PART_FLOATS);
    uint64_t* empty = full + ll::NSLOT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < ll::NSLOT; ++i) {
            l_mbar_init(full + i, 1);
            l_mbar_init(empty + i, ll::NCW);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == ll::NCW) {
        // ------------------------------------------------ producer: weight stream
        if (lane == 0) {
            LRing ring;
            unsigned long long ends[ll::NSLOT];
            unsigned long long tail = 0;
            uint32_t consumed = 0;
            bool ok = true;
            for (int l = 0; l <= a.n_layers && ok; ++l) {
                const int nops = (l == a.n_layers) ? (a.head ? 1 : 0) : 4;
                for (int o = 0; o < nops && ok; ++o) {
                    const LOp d = l_op(a, l, o);
                    int r0, r1;
                    l_rows(d.N, blockIdx.x, gridDim.x, r0, r1);
                    // this CTA's rows of the same op one layer ahead (the head after the last layer)
                    // -> L2, so HBM keeps streaming while the ring is full and ring copies hit L2
                    if ((a.l2_prefetch & 1) && (l + 1 < a.n_layers || (l + 1 == a.n_layers && a.head && o == 0))) {
                        const LOp nx = l_op(a, l + 1, o);
                        int p0, p1;
                        l_rows(nx.N, blockIdx.x, gridDim.x, p0, p1);
                        const char* src = reinterpret_cast<const char*>(nx.W + (size_t)p0 * nx.K);
                        const uint32_t total = (uint32_t)(p1 - p0) * (uint32_t)nx.K * 2u;
                        for (uint32_t off = 0; off < total; off += 16384u)
                            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src + off),
                                         "r"(min(16384u, total - off))
                                         : "memory");
                    }
                    const int rpc = l_rpc(d.K);
                    const uint32_t rs = (uint32_t)d.K * 2 + ll::ROW_PAD;  // ring row stride
                    for (int rc = r0; rc < r1 && ok; rc += rpc) {
                        const int nr = min(rpc, r1 - rc);
                        const uint32_t bytes = (uint32_t)nr * d.K * 2;
                        const uint32_t k = ring.k;
                        const uint32_t p = ring.place((uint32_t)nr * rs);
                        while (ok && (k - consumed >= (uint32_t)ll::NSLOT ||
                                      ring.head - tail > (unsigned long long)ll::RING)) {
                            const uint32_t s = consumed % ll::NSLOT;
                            ok = l_mbar_wait_sleep(empty + s, (consumed / ll::NSLOT) & 1, a);
                            if (ok) { tail = ends[s]; ++consumed; }
                        }
                        if (!ok) break;
                        const uint32_t slot = k % ll::NSLOT;
                        if (a.trace && rc == r0 && l < a.n_layers && (o == 2 || o == 3))  // issue time of the op's first chunk
                            a.trace[((size_t)blockIdx.x * a.n_layers + l) * TRACE_STRIDE + 11 + o] = l_time();
                        ends[slot] = ring.head;
                        ring.k++;
                        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(l_su32(full + slot)),
                                     "r"(bytes)
                                     : "memory");
                        for (int i = 0; i < nr; ++i)  // one copy per row: rows land ROW_PAD bytes apart
                            asm volatile(
                                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                                    l_su32(ring_mem + p + (uint32_t)i * rs)),
                                "l"(d.W + (size_t)(rc + i) * d.K), "r"((uint32_t)d.K * 2), "r"(l_su32(full + slot))
                                : "memory");
                    }
                }
            }
            while (consumed < ring.k) {  // every copy must land before the CTA leaves
                const uint32_t s = consumed % ll::NSLOT;
                if (ok) {
                    if (!l_mbar_wait_sleep(empty + s, (consumed / ll::NSLOT) & 1, a)) ok = false;
                } else {
                    const unsigned long long t0 = l_time();
                    while (!l_mbar_try(full + s, (consumed / ll::NSLOT) & 1) && l_time() - t0 < a.timeout_ns) {
                    }
                }
                ++consumed;
            }
        }
        return;
    }

    // ---------------------------------------------------- consumers
    const XBufs X = l_bufs(a);
    LRing ring;
    int own0, own1;
    l_rows(HID, blockIdx.x, gridDim.x, own0, own1);
    // this CTA's row slices of every op (the same for all layers)
    int2 rows_qkv, rows_o, rows_gu, rows_d, rows_head;
    l_rows(QKV, blockIdx.x, gridDim.x, rows_qkv.x, rows_qkv.y);
    l_rows(HID, blockIdx.x, gridDim.x, rows_o.x, rows_o.y);
    l_rows(2 * 3072, blockIdx.x, gridDim.x, rows_gu.x, rows_gu.y);
    rows_d = rows_o;
    l_rows(a.head_rows, blockIdx.x, gridDim.x, rows_head.x, rows_head.y);
    const int nblk0 = (a.pos[0] + 1 + KVB - 1) / KVB;
    const int nblk1 = B > 1 ? (a.pos[B > 1 ? 1 : 0] + 1 + KVB - 1) / KVB : 0;
    const int units_b0 = NKV * nblk0;
    const int n_units = units_b0 + NKV * nblk1;
    const int t = threadIdx.x;
#define LSTAMP(i)                                                                                 \
    do {                                                                                          \
        if (a.trace && t == 0) a.trace[((size_t)blockIdx.x * a.n_layers + l) * TRACE_STRIDE + (i)] = l_time(); \
    } while (0)

    // page-table entries of blocks opened by this step (read by later launches)
    if (blockIdx.x == 0 && t < a.n_upd) const_cast<int32_t*>(a.page_table)[a.upd_idx[t]] = a.upd_val[t];
    if (t == 0 && (a.l2_prefetch & 2) && n_units > (int)blockIdx.x) l_prefetch_kv(a, 0, B, nblk0, nblk1);
    // layer-0 input: every CTA sums the embeddings itself (fp32 in the attention
    // scratch); own rows are kept
    float* xs = att;
    for (int b = 0; b < B; ++b) {
        for (int c = t * 4; c < HID; c += ll::NCT * 4) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            if (a.embeds) {
                const uint2 u = *reinterpret_cast<const uint2*>(a.embeds + (size_t)b * HID + c);
                acc[0] = __uint_as_float(u.x << 16); acc[1] = __uint_as_float(u.x & 0xFFFF0000u);
                acc[2] = __uint_as_float(u.y << 16); acc[3] = __uint_as_float(u.y & 0xFFFF0000u);
            }
            if (a.ids) {
                for (int k = 0; k < a.tabs.n; ++k) {
                    const int id = a.ids[b * a.tabs.n + k];
                    if (id == -1) continue;
                    if (id < -1 || id >= a.tabs.rows[k]) {
                        if (blockIdx.x == 0 && c == 0) set_err(a.err, ERR_BAD_ID);
                        continue;
                    }
                    const uint2 u = *reinterpret_cast<const uint2*>(a.tabs.tab[k] + (size_t)id * HID + c);
                    acc[0] += __uint_as_float(u.x << 16); acc[1] += __uint_as_float(u.x & 0xFFFF0000u);
                    acc[2] += __uint_as_float(u.y << 16); acc[3] += __uint_as_float(u.y & 0xFFFF0000u);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                xs[b * HID + c + e] = acc[e];
                if (c + e >= own0 && c + e < own1) hown[b * ll::OWN_MAX + (c + e - own0)] = acc[e];
            }
        }
    }
    l_named_sync();
    // norm of the layer-0 input straight from shared memory
    {
        float* red = part;
        for (int b = 0; b < B; ++b) {
            float ss = 0.f;
            for (int c = t; c < HID; c += ll::NCT) ss += xs[b * HID + c] * xs[b * HID + c];
            ss = warp_sum(ss);
            if (lane == 0) red[b * ll::NCW + warp] = ss;
        }
        l_named_sync();
        for (int b = 0; b < B; ++b) {
            float ss = 0.f;
#pragma unroll
            for (int w = 0; w < ll::NCW; ++w) ss += red[b * ll::NCW + w];
            const float r = rsqrtf(ss * (1.f / HID) + a.eps);
            for (int c = 2 * t; c < HID; c += 2 * ll::NCT)
                xf_put2(xf, HID, b, c, xs[b * HID + c] * r * bf2f(a.L[0].in_norm[c]),
                        xs[b * HID + c + 1] * r * bf2f(a.L[0].in_norm[c + 1]));
        }
    }
    l_named_sync();

    for (int l = 0; l < a.n_layers; ++l) {
        LSTAMP(0);
        if (t == 0 && (a.l2_prefetch & 2) && l + 1 < a.n_layers && n_units > (int)blockIdx.x)
            l_prefetch_kv(a, l + 1, B, nblk0, nblk1);
        if (a.trace && t == 0 && l == 0) {
            uint32_t smid;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
            a.trace[(size_t)blockIdx.x * a.n_layers * TRACE_STRIDE + 12] = smid;
        }
        if (l > 0) {
            l_stage_norm<B>(a, xh_mine(X, 2 * l), ep_h(a, 2 * l), a.L[l].in_norm, xf, att);
            l_named_sync();
        }
        LSTAMP(1);
        // ---- QKV rows -> q/k/v words
        {
            unsigned long long* qx = X.q + (size_t)(l & 1) * mk::MAXB * QKV;
            const uint32_t eq = ep_q(a, l);
            l_consume<B, HID, (QKV + LL_MIN_GRID - 1) / LL_MIN_GRID / 16 + 1>(a, l, rows_qkv, ring, ring_mem, full, empty, xf, part, 40,
                         [&](int b, int row, float v0, bool two, float v1, int) {
                             ll_put(qx + (size_t)b * QKV + row, v0, eq);
                             if (two) ll_put(qx + (size_t)b * QKV + row + 1, v1, eq);
                         });
        }
        LSTAMP(2);
        // ---- attention units: unit u = (b, g, j) in order; CTA c takes u = c, c + G, ...
        for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
            int b = 0, r = u;
            if (B > 1 && r >= units_b0) { b = 1; r -= units_b0; }
            const int nblk = b == 0 ? nblk0 : nblk1;
            const int g = r / nblk, j = r - g * nblk;
            l_attn_unit(a, X, l, b, g, j, att);
            if (a.trace && t == 0) a.trace[((size_t)blockIdx.x * a.n_layers + l) * TRACE_STRIDE + 15] += 1;
        }
        LSTAMP(3);
        // ---- merge + o_proj + residual (own rows) -> h words (version 2l+1)
        l_stage_attn<B>(a, X, l, xf);
        l_named_sync();
        LSTAMP(4);
        l_consume<B, NQ * HD, 1>(a, l, rows_o, ring, ring_mem, full, empty, xf, part, 50,
                     [&](int b, int row, float v0, bool two, float v1, int r0) {
                         hown[b * ll::OWN_MAX + row - r0] += v0;
                         if (two) hown[b * ll::OWN_MAX + row + 1 - r0] += v1;
                     });
        l_named_sync();
        if (!(a.debug_stall && l == 0 && blockIdx.x == 0)) {  // (test hook: withhold CTA 0's words once)
            unsigned long long* hx = xh_base(X, 2 * l + 1);
            const uint32_t eh = ep_h(a, 2 * l + 1);
            const int n = B * (own1 - own0);
            for (int i = t; i < LL_XR * n; i += ll::NCT) {
                const int rep = i / n, k = i - rep * n, b = k / (own1 - own0), r = k - b * (own1 - own0);
                ll_put(hx + rep * XH_REP + (size_t)b * HID + own0 + r, hown[b * ll::OWN_MAX + r], eh);
            }
        }
        LSTAMP(5);
        // ---- gate/up + SwiGLU -> m words
        l_stage_norm<B>(a, xh_mine(X, 2 * l + 1), ep_h(a, 2 * l + 1), a.L[l].post_norm, xf, att);
        l_named_sync();
        LSTAMP(6);
        {
            unsigned long long* mx = xm_base(X, l);
            const uint32_t em = ep_m(a, l);
            l_consume<B, HID, 4>(a, l, rows_gu, ring, ring_mem, full, empty, xf, part, 20,
                         [&](int b, int row, float g, bool, float u, int) {
                             const float m = g / (1.f + __expf(-g)) * u;
#pragma unroll
                             for (int rep = 0; rep < LL_XR; ++rep) ll_put(mx + rep * XM_REP + (size_t)b * 3072 + row / 2, m, em);
                         });
        }
        LSTAMP(7);
        // ---- down + residual (own rows) -> h words (version 2l+2)
        {
            const unsigned long long* mx = xm_mine(X, l);
            const uint32_t em = ep_m(a, l);
            // thread t: values 512k + 2t, 512k + 2t + 1 (k < 6) of each row, so a warp's
            // 16-byte loads cover 512 contiguous bytes; all loads first
            unsigned long long w[B * 12];
#pragma unroll
            for (int b = 0; b < B; ++b)
#pragma unroll
                for (int k = 0; k < 6; ++k) ll_ld2(mx + (size_t)b * 3072 + 512 * k + 2 * t, w[b * 12 + 2 * k], w[b * 12 + 2 * k + 1]);
            ll_settle_f(w, [&](int i) { return mx + (size_t)(i / 12) * 3072 + 512 * ((i % 12) >> 1) + 2 * t + (i & 1); }, em, a);
#pragma unroll
            for (int b = 0; b < B; ++b)
#pragma unroll
                for (int k = 0; k < 6; ++k)
                    xf_put2(xf, 3072, b, 512 * k + 2 * t, ll_val(w[b * 12 + 2 * k]), ll_val(w[b * 12 + 2 * k + 1]));
        }
        l_named_sync();
        LSTAMP(8);
        l_consume<B, 3072, 1>(a, l, rows_d, ring, ring_mem, full, empty, xf, part, 30,
                     [&](int b, int row, float v0, bool two, float v1, int r0) {
                         hown[b * ll::OWN_MAX + row - r0] += v0;
                         if (two) hown[b * ll::OWN_MAX + row + 1 - r0] += v1;
                     });
        l_named_sync();
        {
            unsigned long long* hx = xh_base(X, 2 * l + 2);
            const uint32_t eh = ep_h(a, 2 * l + 2);
            const int n = B * (own1 - own0);
            for (int i = t; i < LL_XR * n; i += ll::NCT) {
                const int rep = i / n, k = i - rep * n, b = k / (own1 - own0), r = k - b * (own1 - own0);
                ll_put(hx + rep * XH_REP + (size_t)b * HID + own0 + r, hown[b * ll::OWN_MAX + r], eh);
                if (l == a.n_layers - 1 && rep == 0) a.h[(size_t)b * HID + own0 + r] = hown[b * ll::OWN_MAX + r];
            }
        }
        LSTAMP(9);
    }
#undef LSTAMP
    // ---- final norm + head + argmax
    if (a.head) {
        const int vl = 2 * a.n_layers;
        l_stage_norm<B>(a, xh_mine(X, vl), ep_h(a, vl), a.final_norm, xf, att);
        l_named_sync();
        __shared__ unsigned long long best_s[mk::MAXB];
        if (t < B) best_s[t] = 0ull;
        l_named_sync();
        l_consume<B, HID, 4>(a, a.n_layers, rows_head, ring, ring_mem, full, empty, xf, part, -1,
                     [&](int b, int row, float v0, bool two, float v1, int) {
                         if (a.logits) {
                             a.logits[(size_t)b * a.head_rows + row] = v0;
                             if (two) a.logits[(size_t)b * a.head_rows + row + 1] = v1;
                         }
                         unsigned long long pk = pack_argmax(v0, row);
                         if (two) {
                             const unsigned long long p1 = pack_argmax(v1, row + 1);
                             pk = p1 > pk ? p1 : pk;
                         }
                         atomicMax(best_s + b, pk);
                     });
        l_named_sync();
        if (a.argmax_out) {
            __shared__ int last_s;
            if (t == 0) {
                for (int b = 0; b < B; ++b) atomicMax(a.amax + b, best_s[b]);
                __threadfence();
                const unsigned int old = atomicAdd(a.done, 1u);
                last_s = (old == gridDim.x - 1);
            }
            l_named_sync();
            if (last_s && t < B) {
                __threadfence();
                const unsigned long long best = atomicExch(a.amax + t, 0ull);  // read and re-arm for the next step
                a.argmax_out[(size_t)t * a.argmax_stride] = (int32_t)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
            }
            if (last_s && t == 0) atomicExch(a.done, 0u);
        }
    }
}

int ll_smem_bytes() { return ll::SMEM; }
static_assert((3072 * 2 + LL_MIN_GRID - 1) / LL_MIN_GRID <= l_rpc(HID) * MAXC, "gate/up slice exceeds MAXC chunks");
static_assert((3072 * 2 + LL_MIN_GRID - 1) / LL_MIN_GRID * (2 * HID + ll::ROW_PAD) <= ll::RING, "gate/up slice exceeds the ring");
static_assert(l_rpc(HID) == 16 && l_rpc(NQ * HD) == 8 && l_rpc(3072) == 4, "ring chunk shapes");
// tile counts at the call sites: o_proj and down slices fit one tile, gate/up and the head four
static_assert((HID / 2 + LL_MIN_GRID - 1) / LL_MIN_GRID * 2 <= 16 && (3072 + LL_MIN_GRID - 1) / LL_MIN_GRID * 2 <= 64,
              "op slices exceed their tile counts");
static_assert((3072 * 2 + LL_MIN_GRID - 1) / LL_MIN_GRID <= PART_ROWS && PART_ROWS * mk::MAXB * ll::NCW <= ll::PART_FLOATS,
              "one op's rows exceed the partial buffer");
uint32_t ll_epochs_per_launch(int n_layers) { return 6u * (uint32_t)n_layers + 8u; }

template <int B>
static cudaError_t ll_launch_b(const MegaArgs& a, int grid, cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_decode_ll<B>, cudaFuncAttributeMaxDynamicSharedMemorySize, ll::SMEM);
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(ll::NT);
    cfg.dynamicSmemBytes = ll::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_decode_ll<B>, a);
}

cudaError_t launch_decode_ll(const MegaArgs& a, int grid, cudaStream_t st) {
    switch (a.B) {
        case 1: return ll_launch_b<1>(a, grid, st);
        case 2: return ll_launch_b<2>(a, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

int ll_max_grid() {
    int dev = 0, sms = 0, per = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(k_decode_ll<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, ll::SMEM);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_decode_ll<1>, ll::NT, ll::SMEM);
    // one op's chunks must fit the ring and MAXC at once, own residual rows must fit OWN_MAX
    if (per < 1 || sms < LL_MIN_GRID || (HID / 2 + sms - 1) / sms * 2 > ll::OWN_MAX) return 0;
    return sms;
}

}  // namespace ttsbb
