// MaskGIT greedy update of one refinement step, on the device ("omnivoice-cpp
// docs/ARCHITECTURE.md", MaskGIT decoder; class and position temperatures 0).
//
// k_mg_score — one warp per target cell (item i, codebook k, position t):
//   z = c + s (c - u) over the audio vocabulary (float32, one rounding per
//   operation: no fused multiply-add, so the argmax is reproducible), its
//   log-sum-exp, pred = argmax over the ids other than the mask id (lowest
//   id on ties), score = z[pred] - lse - k * penalty. A cell whose current
//   id is not the mask id gets key 0 (never taken); a masked cell gets the
//   unique key (order(score) << 32) | (2^32 - 1 - flat), flat = k T + t, so
//   a larger key is a higher score, then a lower flat index.
// k_mg_select — one CTA per item: the n = min(n_unmask, masked cells)
//   largest keys are found by a most-significant-digit radix select (8 bits
//   per pass, counts in shared memory, the keys read from shared memory) and
//   their cells take pred in both the conditional and the unconditional id rows.
#include "common.cuh"

namespace ttsbb {

namespace mg {
constexpr int MAXV_LANE = 33;  // vocabulary up to 32 * 33 = 1056 ids
constexpr int SELECT_NT = 1024;
constexpr int SELECT_SMEM = 160 * 1024;        // keys staged in shared memory up to 20480 cells per item
constexpr int SELECT_CAND = 1024;              // boundary-bin keys finished by one warp
// a logits row staged in shared memory: the 16-byte chunks covering it, up to 3 floats of lead-in
constexpr int ROWF = 32 * MAXV_LANE + 4;       // floats per staged row (a multiple of 4)
constexpr int MAXQ = (ROWF / 4 + 31) / 32;     // 16-byte chunks per lane
constexpr int SCORE_WARPS = 1, SCORE_NT = 32 * SCORE_WARPS;  // one-warp CTAs: measured fastest of 1, 2, 4, 8
constexpr int SCORE_SMEM = SCORE_WARPS * 2 * ROWF * 4;  // per warp its (cond, uncond) rows
}  // namespace mg

__device__ __forceinline__ unsigned long long mg_key(float score, int flat) {
    if (!(score == score)) return 0ull;  // NaN: never taken
    const uint32_t b = __float_as_uint(score);
    const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)flat);
}

// The conditional and unconditional logits rows of a cell (item i, codebook k, position t).
__device__ __forceinline__ void mg_rows(const float* logits, long cell, long KT, int T, int V, int S_log, int n_items,
                                        int K, int cond_pos0, int uncond_pos0, const float*& c, const float*& u) {
    const int i = (int)(cell / KT), r = (int)(cell % KT), k = r / T, t = r % T;
    c = logits + (((size_t)i * K + k) * S_log + cond_pos0 + t) * V;
    u = logits + (((size_t)(n_items + i) * K + k) * S_log + uncond_pos0 + t) * V;
}

// One row of V floats starting at any 4-byte boundary (V = 1025): the warp copies the 16-byte
// chunks that cover it (aligned asynchronous copies, all in flight at once) to dst, where element
// v sits at v + lead-in. A chunk that holds a byte of the row lies in the row's own memory page, so
// the few floats read past either end of a row are never out of a mapping.
__device__ __forceinline__ void mg_stage_row(const float* row, int V, float* dst, int lane) {
    const float4* r4 = reinterpret_cast<const float4*>(reinterpret_cast<uintptr_t>(row) & ~(uintptr_t)15);
    const int nq = ((int)((reinterpret_cast<uintptr_t>(row) & 15) >> 2) + V + 3) >> 2;
#pragma unroll
    for (int j = 0; j < mg::MAXQ; ++j) {
        const int q = lane + 32 * j;
        if (q < nq)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst + 4 * q)),
                         "l"(r4 + q)
                         : "memory");
    }
}
__device__ __forceinline__ int mg_lead(const float* row) { return (int)((reinterpret_cast<uintptr_t>(row) & 15) >> 2); }

// grid ceil(n_items K T / SCORE_WARPS), SCORE_NT threads, mg::SCORE_SMEM bytes of shared memory:
// one warp per cell, small CTAs so that many are resident per SM (24, by shared memory) and their
// loads and arithmetic interleave.
__global__ void __launch_bounds__(mg::SCORE_NT) k_mg_score(const float* __restrict__ logits, int n_items, int K, int T, int V,
                                                           int S_log, int cond_pos0, int uncond_pos0,
                                                           const int32_t* __restrict__ ids, int S_ids, int cond_ids_pos0,
                                                           int mask_id, float cfg, float penalty,
                                                           unsigned long long* __restrict__ keys, int32_t* __restrict__ pred) {
    pdl_wait();  // the logits come from the pass
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long KT = (long)K * T;
    const long cell = (long)blockIdx.x * mg::SCORE_WARPS + warp;
    if (cell >= (long)n_items * KT) return;
    const int r = (int)(cell % KT), i = (int)(cell / KT), k = r / T, t = r % T;
    const float *c, *u;
    mg_rows(logits, cell, KT, T, V, S_log, n_items, K, cond_pos0, uncond_pos0, c, u);
    extern __shared__ float4 mg_smem[];
    float* sc = reinterpret_cast<float*>(mg_smem) + warp * 2 * mg::ROWF;
    float* su = sc + mg::ROWF;
    // global -> shared without registers: every 16-byte copy of the lane in flight at once
    mg_stage_row(c, V, sc, lane);
    mg_stage_row(u, V, su, lane);
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
    const int shc = mg_lead(c), shu = mg_lead(u);
    // z = c + s (c - u), one rounding per operation, kept in registers; pass 1: max and argmax,
    // pass 2: sum of exp(z - max) (the hardware exponential: relative error ~1e-7 per term)
    float z[mg::MAXV_LANE];
    float mx = -INFINITY, best = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int j = 0; j < mg::MAXV_LANE; ++j) {
        const int v = lane + 32 * j;
        z[j] = -INFINITY;
        if (v < V) {
            const float cz = sc[v + shc];
            z[j] = __fadd_rn(cz, __fmul_rn(cfg, __fsub_rn(cz, su[v + shu])));
            mx = fmaxf(mx, z[j]);
            const bool better = v != mask_id && (z[j] > best || bi == 0x7FFFFFFF);  // v grows with j
            best = better ? z[j] : best;
            bi = better ? v : bi;
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ob > best || (ob == best && oi < bi)) {
            best = ob;
            bi = oi;
        }
    }
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < mg::MAXV_LANE; ++j) sum += __expf(z[j] - mx);  // z = -inf past the row: 0
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) {
        const float lse = mx + logf(sum);
        const float score = (best - lse) - (float)k * penalty;
        const int cur = ids[((size_t)i * K + k) * S_ids + cond_ids_pos0 + t];
        keys[cell] = cur == mask_id ? mg_key(score, r) : 0ull;
        pred[cell] = bi;
    }
}

// One warp picks the digit of the rem-th largest key from a 256-bin histogram: lane l holds digits
// 255 - 8l .. 248 - 8l (descending). Returns the digit, the rank left within its bin and the bin's
// count, the same in every lane.
__device__ __forceinline__ void mg_pick_digit(const int* hist, int rem, int lane, int& sel, int& rem_out, int& cnt) {
    int cq[8], tot = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        cq[q] = hist[255 - 8 * lane - q];
        tot += cq[q];
    }
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int excl = incl - tot;
    const unsigned bal = __ballot_sync(0xffffffffu, excl < rem && rem <= incl);
    const int src = __ffs(bal) - 1;
    int d = 0, rr = 0, c = 0;
    if (lane == src) {
        int cum = excl;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (cum + cq[q] >= rem) {
                d = 255 - 8 * lane - q;
                rr = rem - cum;
                c = cq[q];
                break;
            }
            cum += cq[q];
        }
    }
    sel = __shfl_sync(0xffffffffu, d, src);
    rem_out = __shfl_sync(0xffffffffu, rr, src);
    cnt = __shfl_sync(0xffffffffu, c, src);
}

// grid n_items, 1024 threads; staged: the item's K T keys are copied once into (dynamic) shared
// memory and the radix passes read them there. The whole CTA runs the passes while the boundary
// bin is large; once it holds at most SELECT_CAND keys, they are gathered into a list and warp 0
// takes the remaining digits alone (no CTA barriers), with the same digit choices.
__global__ void __launch_bounds__(mg::SELECT_NT) k_mg_select(const unsigned long long* __restrict__ keys,
                                                             const int32_t* __restrict__ pred, int n_items, int K,
                                                             int T, int n_unmask, int32_t* __restrict__ ids, int S_ids,
                                                             int cond_ids_pos0, int uncond_ids_pos0, int staged) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ unsigned long long mg_keys[];
    __shared__ int hist[256];
    __shared__ int s_cnt[mg::SELECT_NT / 32];
    __shared__ unsigned long long cand[mg::SELECT_CAND];
    __shared__ int s_sel, s_rem, s_bin, s_nc;
    __shared__ unsigned long long s_thr;
    const int i = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int KT = K * T;
    const unsigned long long* kg = keys + (size_t)i * KT;
    const unsigned long long* kp = staged ? mg_keys : kg;
    // masked cells of this item (and the keys staged)
    int cnt = 0;
#pragma unroll 4
    for (int j = tid; j < KT; j += mg::SELECT_NT) {
        const unsigned long long key = kg[j];
        if (staged) mg_keys[j] = key;
        cnt += key != 0ull;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (lane == 0) s_cnt[warp] = cnt;
    __syncthreads();
    if (tid == 0) {
        int tot = 0;
        for (int w = 0; w < mg::SELECT_NT / 32; ++w) tot += s_cnt[w];
        s_rem = min(n_unmask, tot);
        s_nc = 0;
    }
    __syncthreads();
    int rem = s_rem;
    if (rem <= 0) return;
    unsigned long long prefix = 0ull, pmask = 0ull;
    int sh = 56;
    for (; sh >= 0; sh -= 8) {
        if (tid < 256) hist[tid] = 0;
        __syncthreads();
        // early digits are shared by most keys (scores of similar size): lanes with the same digit add
        // once per warp, so a bin takes one shared-memory atomic per warp instead of one per key
        for (int j0 = 0; j0 < KT; j0 += mg::SELECT_NT) {
            const int j = j0 + tid;
            int bin = -1;
            if (j < KT) {
                const unsigned long long key = kp[j];
                if (key != 0ull && (key & pmask) == prefix) bin = (int)((key >> sh) & 255ull);
            }
            const unsigned same = __match_any_sync(0xffffffffu, bin);
            if (bin >= 0 && lane == __ffs(same) - 1) atomicAdd(&hist[bin], __popc(same));
        }
        __syncthreads();
        if (warp == 0) {
            int d, rr, c;
            mg_pick_digit(hist, rem, lane, d, rr, c);
            if (lane == 0) {
                s_sel = d;
                s_rem = rr;
                s_bin = c;
            }
        }
        __syncthreads();
        prefix |= (unsigned long long)s_sel << sh;
        pmask |= 255ull << sh;
        rem = s_rem;
        const int bin = s_bin;
        __syncthreads();
        if (sh > 0 && bin <= mg::SELECT_CAND) break;  // few keys left in the boundary bin
    }
    if (sh > 0) {  // gather the boundary bin's keys; warp 0 takes the lower digits
        for (int j = tid; j < KT; j += mg::SELECT_NT) {
            const unsigned long long key = kp[j];
            if (key != 0ull && (key & pmask) == prefix) cand[atomicAdd(&s_nc, 1)] = key;
        }
        __syncthreads();
        if (warp == 0) {
            const int nc = s_nc;
            for (int sh2 = sh - 8; sh2 >= 0; sh2 -= 8) {
#pragma unroll
                for (int q = 0; q < 8; ++q) hist[lane * 8 + q] = 0;
                __syncwarp();
                for (int j = lane; j < nc; j += 32) {
                    const unsigned long long key = cand[j];
                    if ((key & pmask) == prefix) atomicAdd(&hist[(int)((key >> sh2) & 255ull)], 1);
                }
                __syncwarp();
                int d, rr, c;
                mg_pick_digit(hist, rem, lane, d, rr, c);
                __syncwarp();
                prefix |= (unsigned long long)d << sh2;
                pmask |= 255ull << sh2;
                rem = rr;
            }
            if (lane == 0) s_thr = prefix;
        }
        __syncthreads();
        prefix = s_thr;
    }
    // keys are unique: exactly the n largest are >= the n-th largest (prefix)
    const int32_t* pp = pred + (size_t)i * KT;
    for (int j = tid; j < KT; j += mg::SELECT_NT) {
        const unsigned long long key = kp[j];
        if (key != 0ull && key >= prefix) {
            const int k = j / T, t = j - k * T, p = pp[j];
            ids[((size_t)i * K + k) * S_ids + cond_ids_pos0 + t] = p;
            ids[((size_t)(n_items + i) * K + k) * S_ids + uncond_ids_pos0 + t] = p;
        }
    }
}

int mg_max_vocab() { return 32 * mg::MAXV_LANE; }

int launch_maskgit_update(const float* logits, int n_items, int K, int T, int V, int S_log, int cond_pos0,
                          int uncond_pos0, int32_t* ids, int S_ids, int cond_ids_pos0, int uncond_ids_pos0,
                          int mask_id, float cfg, float penalty, int n_unmask, unsigned long long* keys, int32_t* pred,
                          cudaStream_t st) {
    const long cells = (long)n_items * K * T;
    if (cells <= 0) return 0;
    static const bool attr = [] {
        cudaFuncSetAttribute(k_mg_select, cudaFuncAttributeMaxDynamicSharedMemorySize, mg::SELECT_SMEM);
        return true;
    }();
    (void)attr;
    launch_pdl(k_mg_score, (unsigned)((cells + mg::SCORE_WARPS - 1) / mg::SCORE_WARPS), mg::SCORE_NT, mg::SCORE_SMEM, st,
               logits, n_items, K, T, V, S_log, cond_pos0, uncond_pos0, (const int32_t*)ids, S_ids, cond_ids_pos0, mask_id,
               cfg, penalty, keys, pred);
    const int staged = (long)K * T * 8 <= mg::SELECT_SMEM;
    launch_pdl(k_mg_select, n_items, mg::SELECT_NT, staged ? K * T * 8 : 0, st, (const unsigned long long*)keys,
               (const int32_t*)pred, n_items, K, T, n_unmask, ids, S_ids, cond_ids_pos0, uncond_ids_pos0, staged);
    return 2;
}

}  // namespace ttsbb
