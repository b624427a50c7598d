// Host engine and C ABI (include/tts_bb.h): weight ownership, the paged KV
// block pool and page tables, per-call validation, and the layer schedule of
// the backbone step (Talker / Code-Predictor prefill and decode, MaskGIT pass).
#include <algorithm>
#include <climits>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "common.cuh"
#include "mega.cuh"
#include "../../include/tts_bb.h"

using namespace ttsbb;

#define TTS_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr int MAX_B = 256;        // sequences per call (per-call arrays travel as kernel parameters)
constexpr int MAX_UPD = 1024;     // page-table updates per setup launch
constexpr int MAX_SPLITS = 64;    // decode attention splits

// Per-call sequence description and page-table updates, passed by value.
struct SetupArgs {
    int B;
    int n_upd;
    int clear_amax;
    int32_t slot[MAX_B];
    int32_t start[MAX_B];
    int32_t len[MAX_B];
    int32_t key_len[MAX_B];
    int32_t upd_idx[MAX_UPD];
    int32_t upd_val[MAX_UPD];
};

__global__ void k_setup(SetupArgs a, int32_t* seq_slot, int32_t* seq_start, int32_t* seq_len, int32_t* key_len,
                        int32_t* page_table, unsigned long long* amax) {
    pdl_wait();  // upstream results are read below
    pdl_trigger();
    for (int i = threadIdx.x; i < a.B; i += blockDim.x) {
        seq_slot[i] = a.slot[i];
        seq_start[i] = a.start[i];
        seq_len[i] = a.len[i];
        key_len[i] = a.key_len[i];
        if (a.clear_amax) amax[i] = 0ull;
    }
    for (int i = threadIdx.x; i < a.n_upd; i += blockDim.x) page_table[a.upd_idx[i]] = a.upd_val[i];
}

// Per-call state of a decode step replayed from a CUDA graph: the setup
// arguments and the caller's pointers, refreshed by one host-to-device copy
// before each replay, so every captured launch keeps fixed parameters.
struct StepBlock {
    SetupArgs a;
    const int32_t* ids;      // [B][n_codebooks] or null
    const bf16* embeds;      // [B][HID] or null
    float* logits_out;       // [B][head_rows] or null
    int32_t* argmax_out;     // stride argmax_stride, or null
    int argmax_stride;
    float* hidden_out;       // [B][HID] or null
};

// Graph-step setup: block 0 does k_setup's work from the step block; block b
// copies token b's ids / embeddings into the engine's fixed input buffers.
__global__ void k_step_setup(const StepBlock* __restrict__ sb, int n_cb, int32_t* seq_slot, int32_t* seq_start,
                             int32_t* seq_len, int32_t* key_len, int32_t* page_table, unsigned long long* amax,
                             int32_t* ids_buf, bf16* emb_buf) {
    pdl_wait();  // upstream results are read below
    pdl_trigger();
    const SetupArgs& a = sb->a;
    const int b = blockIdx.x;
    if (b == 0) {
        for (int i = threadIdx.x; i < a.B; i += blockDim.x) {
            seq_slot[i] = a.slot[i];
            seq_start[i] = a.start[i];
            seq_len[i] = a.len[i];
            key_len[i] = a.key_len[i];
            if (a.clear_amax) amax[i] = 0ull;
        }
        for (int i = threadIdx.x; i < a.n_upd; i += blockDim.x) page_table[a.upd_idx[i]] = a.upd_val[i];
    }
    if (b < a.B) {
        if (ids_buf && sb->ids)
            for (int k = threadIdx.x; k < n_cb; k += blockDim.x) ids_buf[b * n_cb + k] = sb->ids[(size_t)b * n_cb + k];
        if (emb_buf && sb->embeds)
            for (int i = threadIdx.x; i < HID; i += blockDim.x) emb_buf[(size_t)b * HID + i] = sb->embeds[(size_t)b * HID + i];
    }
}

// Graph-step outputs: block b copies token b's logits, argmax and final hidden
// state to the caller's pointers from the step block.
__global__ void k_step_publish(const StepBlock* __restrict__ sb, const float* logits, int rows,
                               const unsigned long long* amax, const float* hid) {
    pdl_wait();  // upstream results are read below
    pdl_trigger();
    const int b = blockIdx.x;
    if (logits && sb->logits_out)
        for (int i = threadIdx.x; i < rows; i += blockDim.x) sb->logits_out[(size_t)b * rows + i] = logits[(size_t)b * rows + i];
    if (amax && sb->argmax_out && threadIdx.x == 0)
        sb->argmax_out[(size_t)b * sb->argmax_stride] = (int32_t)(0xFFFFFFFFu - (uint32_t)(amax[b] & 0xFFFFFFFFull));
    if (hid && sb->hidden_out)
        for (int i = threadIdx.x; i < HID; i += blockDim.x) sb->hidden_out[(size_t)b * HID + i] = hid[(size_t)b * HID + i];
}

// Frame loop, between the Talker step and the Code Predictor (Qwen3-TTS ncnn port, model
// structure): row b of the Code Predictor's 2-token prefill gets the Talker's final-normed
// hidden state (bf16) at position 0 and zero at position 1, whose ids carry code 0 alone; the id
// rows of the 14 decode calls start at -1 (each call's argmax fills the next call's column).
// grid B, 256 threads.
__global__ void k_frame_prep(const float* __restrict__ hid, const bf16* __restrict__ gamma, float eps,
                             const int32_t* __restrict__ code0, bf16* __restrict__ cp_emb, int32_t* __restrict__ cp_ids,
                             int32_t* __restrict__ steps, int B) {
    const int b = blockIdx.x, t = threadIdx.x;
    __shared__ float red[8];
    const float* x = hid + (size_t)b * HID;
    float v[4], ss = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        v[e] = x[t + 256 * e];
        ss += v[e] * v[e];
    }
    ss = warp_sum(ss);
    if ((t & 31) == 0) red[t >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[w];
    const float r = rsqrtf(tot * (1.f / HID) + eps);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int c = t + 256 * e;
        cp_emb[(size_t)b * 2 * HID + c] = f2bf(v[e] * r * bf2f(gamma[c]));
        cp_emb[(size_t)b * 2 * HID + HID + c] = f2bf(0.f);
    }
    if (t < 32) cp_ids[(size_t)b * 32 + t] = t == 16 ? code0[b] : -1;
    for (int i = t; i < 15 * 16; i += 256) steps[((size_t)(i >> 4) * B + b) * 16 + (i & 15)] = -1;
}

// codes[b] = [code 0, codes 1..14 from the decode calls' id rows, code 15 already in place]
__global__ void k_frame_collect(const int32_t* __restrict__ code0, const int32_t* __restrict__ steps,
                                int32_t* __restrict__ codes, int B) {
    const int b = blockIdx.x, j = threadIdx.x;
    if (j == 0) codes[(size_t)b * 16] = code0[b];
    else if (j < 15) codes[(size_t)b * 16 + j] = steps[((size_t)j * B + b) * 16 + j];
}

__global__ void k_kv_copy(bf16* pool, const int32_t* page_table, int slot, int mbps, int pos0, int n, bf16* k,
                          bf16* v, int to_pool, int n_blocks, int* err) {
    // one CTA per token, 256 threads: 8 kv heads x 128 elements, 4 per thread for K and V
    const int t = blockIdx.x;
    const int pos = pos0 + t;
    const int phys = page_table[(size_t)slot * mbps + pos / KVB];
    if (phys < 0 || phys >= n_blocks) {  // no block behind this position: report, touch nothing
        if (threadIdx.x == 0) set_err(err, ERR_KV_RANGE);
        return;
    }
    for (int e = threadIdx.x; e < NKV * HD; e += blockDim.x) {
        const int g = e / HD, d = e % HD;
        const size_t pk = (((size_t)phys * 2 + 0) * NKV + g) * KVB * HD + (size_t)(pos % KVB) * HD + d;
        const size_t pv = pk + (size_t)NKV * KVB * HD;
        const size_t io = (size_t)t * NKV * HD + e;
        if (to_pool) {
            pool[pk] = k[io];
            pool[pv] = v[io];
        } else {
            k[io] = pool[pk];
            v[io] = pool[pv];
        }
    }
}

struct LayerW {
    bf16 *in_norm, *wqkv, *qn, *kn, *wo, *post_norm, *wgu, *wd;
};

}  // namespace

struct tts_bb {
    tts_bb_config cfg;
    cudaStream_t st = nullptr;
    int dev = 0;
    std::vector<void*> allocs;
    std::vector<LayerW> L;
    TableSet tabs{};
    bf16* text = nullptr;
    bf16* audio = nullptr;
    bf16* final_norm = nullptr;
    bf16* heads[TTS_BB_MAX_HEADS] = {};
    float* cos_t = nullptr;
    float* sin_t = nullptr;
    int rope_len = 0;
    // KV
    bf16* pool = nullptr;
    size_t layer_elems = 0;   // elements per layer of the pool
    int kv_blocks = 0, mbps = 0;
    int32_t* d_page_table = nullptr;
    std::vector<int32_t> page_table;
    std::vector<int> slot_len;
    std::vector<int> free_blocks;
    // scratch
    int T_cap = 0;
    float* h = nullptr;
    bf16* y = nullptr;
    float* qkv = nullptr;
    bf16* q = nullptr;
    float* qf = nullptr;                // decode: fp32 queries for the decode attention
    float* nss = nullptr;               // decode: per-tile sums of squares of the folded RMSNorms [8][T]
    bool launch_missing = false;        // a fused GEMM epilogue had no kernel to run on
    bf16* ao = nullptr;
    bf16* m = nullptr;
    bf16 *y_lo = nullptr, *ao_lo = nullptr, *m_lo = nullptr;  // low bf16 parts (decode)
    SplitK sk{};                        // split-K workspace of the decode-batch GEMM
    float* part = nullptr;
    unsigned long long* amax = nullptr;
    int32_t *seq_slot = nullptr, *seq_start = nullptr, *seq_len = nullptr, *key_len = nullptr;
    bf16* mg_pool = nullptr;
    bool attn_bidir_tc = false;
    bool attn_causal_tc = false;        // causal prefill of 64 or more positions per sequence on tcgen05
    bool fuse_qk = false;               // q/k norm + RoPE + KV append in the decode GEMM's QKV epilogue
    bool fold_norm = false;             // decode batches: the RMSNorms folded into the decode GEMMs' epilogues
    bool short_prefill_attn = false;    // causal prefills of <= 8 positions per sequence on the decode attention
    int32_t* hx_ids = nullptr;  // tts_bb_decode_step_host: device copies of the caller's host ids and argmax
    int32_t* hx_am = nullptr;
    float* hx_logits = nullptr;
    // frame-loop scratch (on the Code Predictor's handle): Talker hidden, code 0, prefill input,
    // prefill ids, and the id rows of the 14 decode calls
    float* fr_hid = nullptr;
    int32_t* fr_code0 = nullptr;
    bf16* fr_emb = nullptr;
    int32_t* fr_ids = nullptr;
    int32_t* fr_steps = nullptr;
    int fr_cap = 0;
    unsigned long long* mg_keys = nullptr;  // MaskGIT update scratch: a key and a prediction per cell
    int32_t* mg_pred = nullptr;
    size_t mg_cells = 0;
    int l2_prefetch = 3;         // persistent step, L2 prefetch one layer ahead: bit 0 weight rows, bit 1 attention K/V
    size_t mg_pool_blocks = 0;
    int* err = nullptr;
    int* h_err = nullptr;
    std::string last_error;
    uint64_t launches = 0;
    SetupArgs* setup = nullptr;  // host staging (large struct)
    // per-kernel timing (tts_bb_profile): events around every launch, by kernel kind
    bool prof_on = false;
    struct ProfRec { int kind; cudaEvent_t a, b; double bytes; double flops; };
    std::vector<ProfRec> prof;
    std::vector<cudaEvent_t> ev_pool;
    std::string prof_json;
    // persistent small-batch decode step
    int mega_grid = 0;                 // 0 = not available on this device
    int* mega_abort = nullptr;
    unsigned long long* ll_xbuf = nullptr;   // exchange words
    unsigned long long* ll_amax = nullptr;   // [MAXB], re-armed by the kernel
    unsigned int* ll_done = nullptr;
    uint32_t ep_base = 1;
    MegaArgs* mega = nullptr;          // per-handle constant fields filled at create
    unsigned long long* mega_trace = nullptr;   // phase stamps while profiling
    std::vector<double> phase_us;      // summed per-phase mean-over-CTA durations over traced layers
    std::vector<double> phase_max_us;  // summed per-phase max-over-CTA durations
    long phase_n = 0;                  // traced layers
    double unit_split[2] = {0, 0};
    long unit_split_n[2] = {0, 0};
    double ring_wait[2] = {0, 0};      // persistent step: weight-ring waits inside gate/up and down
    long ring_wait_n = 0;
    // multi-kernel decode steps replayed from CUDA graphs
    static constexpr int RING = 8;
    bool graphs_on = false;
    StepBlock* d_step = nullptr;       // device step block (read by the captured setup / publish)
    StepBlock* h_ring = nullptr;       // pinned staging, RING entries
    cudaEvent_t ring_ev[RING] = {};
    bool ring_used[RING] = {};
    int ring_i = 0;
    int32_t* ids_buf = nullptr;        // [max_batch][n_codebooks]
    bf16* emb_buf = nullptr;           // [max_batch][HID]
    float* logits_buf = nullptr;       // [max_batch][head_rows]
    struct DecodeGraph {
        int key[7];
        int seen = 0;                  // calls with this key (the first runs eagerly)
        cudaGraphExec_t exec = nullptr;
        uint64_t n_kernels = 0;
        bool bad = false;              // capture failed: stay eager
    };
    std::vector<DecodeGraph> graphs;
    // failure-handling test hooks (tts_bb_debug_fault, TTS_BB_FAIL_ALLOC_AT)
    unsigned long n_allocs = 0;
    unsigned long long wait_limit_ns = 2000000000ull;
    int stall_next = 0;
};

namespace {

tts_bb_status fail(tts_bb* h, tts_bb_status s, const char* fmt, ...) __attribute__((format(printf, 3, 4)));
tts_bb_status fail(tts_bb* h, tts_bb_status s, const char* fmt, ...) {
    if (h) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        h->last_error = buf;
    }
    return s;
}

tts_bb_status cuda_fail(tts_bb* h, cudaError_t e, const char* what) {
    return fail(h, e == cudaErrorMemoryAllocation ? TTS_BB_E_OOM : TTS_BB_E_CUDA, "%s: %s", what,
                cudaGetErrorString(e));
}

// TTS_BB_FAIL_ALLOC_AT=n: the n-th device allocation of a handle fails (test hook).
inline bool alloc_fault(tts_bb* h) {
    const char* v = std::getenv("TTS_BB_FAIL_ALLOC_AT");
    const long at = v ? std::atol(v) : 0L;
    return at > 0 && (long)++h->n_allocs == at;
}

template <typename T>
cudaError_t dalloc(tts_bb* h, T** p, size_t n) {
    if (alloc_fault(h)) return cudaErrorMemoryAllocation;
    void* v = nullptr;
    const cudaError_t e = cudaMalloc(&v, std::max<size_t>(n, 1) * sizeof(T));
    if (e == cudaSuccess) {
        h->allocs.push_back(v);
        *p = reinterpret_cast<T*>(v);
    }
    return e;
}

constexpr int MAX_CFG_LEN = 1 << 20;

bool cfg_supported(const tts_bb_config& c, std::string& why) {
    if (c.hidden != HID || c.n_q_heads != NQ || c.n_kv_heads != NKV || c.head_dim != HD) {
        why = "kernels are built for hidden 1024, 16 q / 8 kv heads of 128";
        return false;
    }
    if (c.ffn % 256 != 0 || c.ffn <= 0 || c.ffn > 3072) {
        why = "ffn must be a positive multiple of 256, at most 3072";
        return false;
    }
    if (c.max_ctx > MAX_CFG_LEN || c.max_tokens > MAX_CFG_LEN || c.max_slots > MAX_CFG_LEN) {
        why = "max_ctx, max_tokens and max_slots are limited to 2^20";  // host tables scale with them
        return false;
    }
    return true;
}

tts_bb_status check_launch(tts_bb* h, const char* what) {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(h, e, what);
    return TTS_BB_OK;
}

// Read (and clear) the device error word; synchronises the stream.
tts_bb_status read_err(tts_bb* h) {
    cudaError_t e = cudaMemcpyAsync(h->h_err, h->err, sizeof(int), cudaMemcpyDeviceToHost, h->st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->st);
    if (e != cudaSuccess) return cuda_fail(h, e, "stream");
    const int v = *h->h_err;
    if (v) {
        cudaMemsetAsync(h->err, 0, sizeof(int), h->st);
        if ((v & ERR_TIMEOUT) && h->mega_abort) {  // re-arm the persistent step after an abort
            cudaMemsetAsync(h->mega_abort, 0, sizeof(int), h->st);
            cudaMemsetAsync(h->ll_amax, 0, mk::MAXB * sizeof(unsigned long long), h->st);
            cudaMemsetAsync(h->ll_done, 0, sizeof(unsigned int), h->st);
        }
        cudaStreamSynchronize(h->st);
        if (v & ERR_TIMEOUT) return fail(h, TTS_BB_E_DEVICE_TIMEOUT, "a device-side wait timed out");
        if (v & ERR_BAD_ID) return fail(h, TTS_BB_E_BAD_ID, "a token id was outside its table (skipped)");
        if (v & ERR_KV_RANGE) return fail(h, TTS_BB_E_INVALID, "a KV position had no block");
        if (v & ERR_LAYOUT) return fail(h, TTS_BB_E_CUDA, "a kernel's shared memory was not 1 KB aligned");
    }
    return TTS_BB_OK;
}

tts_bb_status finish(tts_bb* h) {
    tts_bb_status s = check_launch(h, "kernel launch");
    if (s != TTS_BB_OK) return s;
    if (h->launch_missing) {
        h->launch_missing = false;
        return fail(h, TTS_BB_E_CUDA, "a fused decode-GEMM epilogue could not be launched");
    }
    if (h->cfg.sync_errors) return read_err(h);
    return TTS_BB_OK;
}

enum Kind { K_SETUP, K_EMBED, K_RMSNORM, K_GEMV, K_GEMM, K_QKROPE, K_ATTN_DECODE, K_ATTN_PREFILL, K_ARGMAX,
            K_KVCOPY, K_MEGA, K_GEMM_TC, K_GEMM_TCD, K_ATTN_BIDIR_TC, K_MG_UPDATE, K_FRAME, K_ATTN_CAUSAL_TC,
            K_ATTN_DECODE_SHORT, K_NKINDS };
const char* kind_name[K_NKINDS] = {"setup", "embed_gather", "rmsnorm", "gemv", "gemm_mma_split", "qk_norm_rope_append",
                                   "attn_decode", "attn_prefill", "argmax", "kv_copy", "decode_step_persistent",
                                   "gemm_tcgen05", "gemm_tcgen05_decode", "attn_bidir_tcgen05", "maskgit_update", "frame_glue",
                                   "attn_causal_tcgen05", "attn_decode_short"};

cudaEvent_t prof_event(tts_bb* h) {
    if (!h->ev_pool.empty()) {
        cudaEvent_t e = h->ev_pool.back();
        h->ev_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Brackets the launches of one engine step with CUDA events when profiling is on,
// and counts the kernels launched. bytes / flops: algorithmic work of the launch.
struct Launch {
    tts_bb* h;
    int kind;
    double bytes, flops;
    cudaEvent_t a = nullptr;
    Launch(tts_bb* h_, int kind_, double bytes_ = 0, double flops_ = 0) : h(h_), kind(kind_), bytes(bytes_), flops(flops_) {
        if (h->prof_on) {
            a = prof_event(h);
            cudaEventRecord(a, h->st);
        }
    }
    void operator+=(int n) { h->launches += n; }
    ~Launch() {
        if (a) {
            cudaEvent_t b = prof_event(h);
            cudaEventRecord(b, h->st);
            h->prof.push_back({kind, a, b, bytes, flops});
        }
    }
};

double gemm_bytes(int T, int N, int K, int out_bytes) {
    return 2.0 * N * K + 2.0 * T * K + (double)out_bytes * T * N;
}

// Scratch for T tokens (grows on demand; only between calls).
tts_bb_status ensure_scratch(tts_bb* h, int T) {
    if (T <= h->T_cap) return TTS_BB_OK;
    if (h->h) {
        cudaStreamSynchronize(h->st);
        void* olds[] = {h->h, h->y, h->qkv, h->q, h->qf, h->ao, h->m, h->y_lo, h->ao_lo, h->m_lo, h->nss};
        for (void* p : olds) {
            cudaFree(p);
            h->allocs.erase(std::remove(h->allocs.begin(), h->allocs.end(), p), h->allocs.end());
        }
    }
    cudaError_t e;
    if ((e = dalloc(h, &h->h, (size_t)T * HID)) != cudaSuccess ||
        (e = dalloc(h, &h->y, (size_t)T * HID)) != cudaSuccess ||
        (e = dalloc(h, &h->qkv, (size_t)T * QKV)) != cudaSuccess ||
        (e = dalloc(h, &h->q, (size_t)T * NQ * HD)) != cudaSuccess ||
        (e = dalloc(h, &h->qf, (size_t)T * NQ * HD)) != cudaSuccess ||
        (e = dalloc(h, &h->ao, (size_t)T * NQ * HD)) != cudaSuccess ||
        (e = dalloc(h, &h->m, (size_t)T * h->cfg.ffn)) != cudaSuccess ||
        (e = dalloc(h, &h->y_lo, (size_t)T * HID)) != cudaSuccess ||
        (e = dalloc(h, &h->ao_lo, (size_t)T * NQ * HD)) != cudaSuccess ||
        (e = dalloc(h, &h->m_lo, (size_t)T * h->cfg.ffn)) != cudaSuccess ||
        (e = dalloc(h, &h->nss, (size_t)8 * T)) != cudaSuccess) {
        h->T_cap = 0;
        h->h = nullptr;
        return cuda_fail(h, e, "scratch allocation");
    }
    h->T_cap = T;
    return TTS_BB_OK;
}

void launch_setup(tts_bb* h, SetupArgs& a) {
    Launch L(h, K_SETUP);
    launch_pdl(k_setup, 1, 256, 0, h->st, a, h->seq_slot, h->seq_start, h->seq_len, h->key_len, h->d_page_table, h->amax);
    L += 1;
}

// The layer schedule shared by every mode. T tokens laid out as B sequences x
// tok_per_seq positions; mode: 0 decode (query length 1), 1 causal prefill,
// 2 bidirectional pass.
// Returns true when the decode step folded its RMSNorms into the GEMM epilogues: the final norm's
// input (h * gamma, high + low parts) and sums of squares are then in y / y_lo / nss for run_head.
bool run_layers(tts_bb* h, int B, int tok_per_seq, int mode, int max_len, KVView kv_base, size_t layer_stride,
                double kv_read_bytes = 0, double attn_flops = 0) {
    const tts_bb_config& c = h->cfg;
    const int T = B * tok_per_seq;
    // decode batches on the split-K decode GEMM: each RMSNorm after the first is folded into the
    // GEMMs around it (the residual-add epilogue writes h * gamma and per-tile sums of squares; the
    // next product scales its rows by the inverse RMS)
    const bool fold = mode == 0 && h->fold_norm && T > 8 && T <= 256;
    // the bidirectional pass keeps K / V in its own pool (no page table), which the tcgen05 kernel reads by TMA
    const bool bidir_tc = mode == 2 && h->attn_bidir_tc;
    // a causal prefill of a full 64-query tile per sequence or more runs on tcgen05 from fp32
    // queries (shorter ones stay on the mma.sync kernel)
    const bool causal_tc = mode == 1 && h->attn_causal_tc && tok_per_seq >= 64;
    // a causal prefill of at most 8 positions per sequence (the Code Predictor's 2-token call) runs
    // on the decode attention kernel, one query per token, from fp32 queries
    const bool short_prefill = mode == 1 && !causal_tc && tok_per_seq <= 8 && h->short_prefill_attn;
    for (int l = 0; l < c.n_layers; ++l) {
        const LayerW& w = h->L[l];
        KVView kv = kv_base;
        kv.pool = kv_base.pool + (size_t)l * layer_stride;
        // decode and causal prefill carry GEMM inputs as bf16 high + low parts (the
        // prefill writes the K/V that every later step reads); the bidirectional
        // pass, tensor-bound, uses plain bf16
        const bool split = mode != 2;
        // the kernel launch_gemm picks for an N x K product
        auto gk_of = [&](int N, int K) {
            return T <= 8 ? K_GEMV : (split && (T <= 256 || gemm_tcd_takes(T, N, K)) ? K_GEMM_TCD : K_GEMM_TC);
        };
        const int gk = gk_of(QKV, HID), gk_o = gk_of(HID, NQ * HD), gk_gu = gk_of(2 * c.ffn, HID), gk_d = gk_of(HID, c.ffn);
        bf16* ylo = split ? h->y_lo : nullptr;
        bf16* aolo = split ? h->ao_lo : nullptr;
        bf16* mlo = split ? h->m_lo : nullptr;
        const SplitK* skp = split && h->sk.part ? &h->sk : nullptr;
        const double norm_bytes = T * (4.0 + 2.0) * HID + 2.0 * HID;
        auto need = [&](int n) {  // a folded epilogue must run on the decode GEMM
            if (fold && !n) h->launch_missing = true;
            return n;
        };
        auto scale_in = [&](Epi& ee) {  // consumer of a folded norm
            ee.nrm_scale_ss = h->nss;
            ee.nrm_eps = c.rms_eps;
            ee.nrm_T = T;
        };
        auto norm_out = [&](Epi& ee, const bf16* gamma) {  // producer of the next folded norm's input
            ee.nrm_gamma = gamma;
            ee.nrm_y = h->y;
            ee.nrm_ylo = h->y_lo;
            ee.nrm_ss = h->nss;
            ee.nrm_eps = c.rms_eps;
            ee.nrm_T = T;
        };
        if (!fold || l == 0) {
            Launch L(h, K_RMSNORM, norm_bytes);
            L += launch_rmsnorm(h->h, w.in_norm, h->y, T, c.rms_eps, 1, 1, 0, nullptr, h->st, ylo);
        }
        Epi e{};
        float* qf_out = mode == 0 || causal_tc || short_prefill ? h->qf : nullptr;
        int fused = 0;
        if (gk == K_GEMM_TCD && h->fuse_qk) {
            // the split-K decode GEMM applies q/k norm + RoPE and appends k, v in its epilogue
            e.mode = EPI_QKROPE;
            e.qk = EpiQk{w.qn, w.kn, h->cos_t, h->sin_t, c.rms_eps, h->q, qf_out, kv, h->seq_start, h->seq_len,
                         tok_per_seq, h->err};
            if (fold && l > 0) scale_in(e);
            Launch L(h, gk, gemm_bytes(T, QKV, HID, 2), 2.0 * T * QKV * HID);
            fused = launch_gemm(h->y, w.wqkv, T, QKV, HID, e, h->st, ylo, h->err, skp);
            L += fused;
            e = Epi{};
        }
        if (!fused) {
            // the bidirectional pass (bf16 operands throughout) keeps its QKV rows in bf16
            bf16* qkv_bf = mode == 2 && gk == K_GEMM_TC ? reinterpret_cast<bf16*>(h->qkv) : nullptr;
            e.mode = qkv_bf ? EPI_STORE_BF16 : EPI_STORE_F32; e.out = h->qkv; e.ldo = QKV;
            if (fold && l > 0) scale_in(e);
            { Launch L(h, gk, gemm_bytes(T, QKV, HID, qkv_bf ? 2 : 4), 2.0 * T * QKV * HID); L += need(launch_gemm(h->y, w.wqkv, T, QKV, HID, e, h->st, ylo, h->err, skp)); }
            { Launch L(h, K_QKROPE, T * ((qkv_bf ? 2.0 : 4.0) * QKV + 2.0 * QKV));
              L += launch_qk_norm_rope_append(h->qkv, w.qn, w.kn, h->cos_t, h->sin_t, c.rms_eps, h->q, kv,
                                              h->seq_start, h->seq_len, tok_per_seq, T, h->err, h->st, qf_out, qkv_bf); }
        }
        if (bidir_tc) {
            Launch L(h, K_ATTN_BIDIR_TC, 0, attn_flops);
            L += launch_attn_bidir_tc(h->q, kv.pool, h->mg_pool_blocks, kv.mbps, h->key_len, B, tok_per_seq, h->ao, h->err, h->st);
        } else if (mode == 0) {
            Launch L(h, max_len <= ATTN_SHORT_CTX ? K_ATTN_DECODE_SHORT : K_ATTN_DECODE, kv_read_bytes + T * (2.0 * NQ * HD * 2),
                     4.0 * NQ * HD * (kv_read_bytes / (2.0 * NKV * HD * 2)));
            L += launch_attn_decode(h->q, kv, h->seq_start, B, max_len, h->part, h->ao, MAX_SPLITS, h->st, aolo, h->qf);
        } else if (short_prefill) {
            Launch L(h, c.max_ctx <= ATTN_SHORT_CTX ? K_ATTN_DECODE_SHORT : K_ATTN_DECODE, 0, attn_flops);
            const int nb = std::max(c.max_batch, 1);
            L += launch_attn_decode(h->q, kv, h->seq_start, T, c.max_ctx, h->part, h->ao, std::max(1, nb * MAX_SPLITS / T),
                                    h->st, aolo, h->qf, tok_per_seq, h->seq_len);
        } else if (causal_tc) {
            Launch L(h, K_ATTN_CAUSAL_TC, 0, attn_flops);
            L += launch_attn_causal_tc(h->q, h->qf, kv, (size_t)h->kv_blocks, h->seq_start, B, tok_per_seq, h->ao, aolo,
                                       h->err, h->st);
        } else {
            Launch L(h, K_ATTN_PREFILL, 0, attn_flops);
            L += launch_attn_prefill(h->q, kv, h->seq_start, h->seq_len, h->key_len, mode == 1, B, tok_per_seq, h->ao, h->st,
                                     aolo);
        }
        e = Epi{};
        e.mode = EPI_ADD_F32; e.out = h->h; e.ldo = HID;
        if (fold) norm_out(e, w.post_norm);
        { Launch L(h, gk_o, gemm_bytes(T, HID, NQ * HD, 8), 2.0 * T * HID * NQ * HD); L += need(launch_gemm(h->ao, w.wo, T, HID, NQ * HD, e, h->st, aolo, h->err, skp)); }
        if (!fold) { Launch L(h, K_RMSNORM, norm_bytes); L += launch_rmsnorm(h->h, w.post_norm, h->y, T, c.rms_eps, 1, 1, 0, nullptr, h->st, ylo); }
        e = Epi{};
        e.mode = EPI_SWIGLU; e.out = h->m; e.ldo = c.ffn; e.out_lo = mlo;
        if (fold) scale_in(e);
        { Launch L(h, gk_gu, gemm_bytes(T, 2 * c.ffn, HID, 1), 2.0 * T * 2 * c.ffn * HID); L += need(launch_gemm(h->y, w.wgu, T, 2 * c.ffn, HID, e, h->st, ylo, h->err, skp)); }
        e = Epi{};
        e.mode = EPI_ADD_F32; e.out = h->h; e.ldo = HID;
        if (fold) norm_out(e, l + 1 < c.n_layers ? h->L[l + 1].in_norm : h->final_norm);
        { Launch L(h, gk_d, gemm_bytes(T, HID, c.ffn, 8), 2.0 * T * HID * c.ffn); L += need(launch_gemm(h->m, w.wd, T, HID, c.ffn, e, h->st, mlo, h->err, skp)); }
    }
    return fold;
}

// Final norm of B selected rows + head GEMM with logits / argmax.
// folded: the decode layers left the final norm's input (h * gamma, high + low parts) and sums of
// squares in y / y_lo / nss, so the head scales its rows instead of running the norm.
void run_head(tts_bb* h, int B, int per_seq, int head_idx, bool last_of_seq, float* logits_out, int32_t* argmax_out,
              int argmax_stride, bool split = false, bool finalize = true, bool folded = false) {
    const tts_bb_config& c = h->cfg;
    bf16* ylo = split ? h->y_lo : nullptr;
    if (!folded) {
        Launch L(h, K_RMSNORM, B * 6.0 * HID + 2.0 * HID);
        L += launch_rmsnorm(h->h, h->final_norm, h->y, B, c.rms_eps, 1, per_seq, 0, last_of_seq ? h->seq_len : nullptr, h->st, ylo);
    }
    Epi e{};
    e.mode = EPI_LOGITS; e.out = logits_out; e.ldo = c.head_rows; e.amax = argmax_out ? h->amax : nullptr;
    if (folded) {
        e.nrm_scale_ss = h->nss;
        e.nrm_eps = c.rms_eps;
        e.nrm_T = B;
    }
    const int gk = B <= 8 ? K_GEMV : (split && (B <= 256 || gemm_tcd_takes(B, c.head_rows, HID)) ? K_GEMM_TCD : K_GEMM_TC);
    { Launch L(h, gk, gemm_bytes(B, c.head_rows, HID, logits_out ? 4 : 0), 2.0 * B * c.head_rows * HID);
      const int n = launch_gemm(h->y, h->heads[head_idx], B, c.head_rows, HID, e, h->st, ylo, h->err,
                                split && h->sk.part ? &h->sk : nullptr);
      if (folded && !n) h->launch_missing = true;
      L += n; }
    if (argmax_out && finalize) { Launch L(h, K_ARGMAX); L += launch_argmax_finalize(h->amax, argmax_out, argmax_stride, B, h->st); }
}

bool slots_ok(tts_bb* h, int B, const int32_t* slots) {
    if (!slots) return false;
    std::vector<char> seen(h->cfg.max_slots, 0);
    for (int b = 0; b < B; ++b) {
        if (slots[b] < 0 || slots[b] >= h->cfg.max_slots || seen[slots[b]]) return false;
        seen[slots[b]] = 1;
    }
    return true;
}

// Reserve the blocks that growing each slot to new_len[b] needs; all or nothing.
tts_bb_status grow_slots(tts_bb* h, int B, const int32_t* slots, const int* new_len, SetupArgs& a) {
    int need = 0;
    for (int b = 0; b < B; ++b) {
        const int have = (h->slot_len[slots[b]] + KVB - 1) / KVB;
        const int want = (new_len[b] + KVB - 1) / KVB;
        need += std::max(0, want - have);
    }
    if (need > (int)h->free_blocks.size())
        return fail(h, TTS_BB_E_OOM, "KV block pool exhausted: need %d blocks, %zu free", need, h->free_blocks.size());
    a.n_upd = 0;
    std::vector<std::pair<int, int>> upd;
    for (int b = 0; b < B; ++b) {
        const int s = slots[b];
        const int have = (h->slot_len[s] + KVB - 1) / KVB;
        const int want = (new_len[b] + KVB - 1) / KVB;
        for (int j = have; j < want; ++j) {
            const int blk = h->free_blocks.back();
            h->free_blocks.pop_back();
            h->page_table[(size_t)s * h->mbps + j] = blk;
            upd.push_back({s * h->mbps + j, blk});
        }
    }
    // updates beyond what one setup launch carries go in extra launches first
    size_t i = 0;
    while (upd.size() - i > (size_t)MAX_UPD) {
        SetupArgs* ex = new SetupArgs();
        ex->B = 0;
        ex->n_upd = MAX_UPD;
        for (int k = 0; k < MAX_UPD; ++k, ++i) { ex->upd_idx[k] = upd[i].first; ex->upd_val[k] = upd[i].second; }
        launch_setup(h, *ex);
        delete ex;
    }
    for (; i < upd.size(); ++i) {
        a.upd_idx[a.n_upd] = upd[i].first;
        a.upd_val[a.n_upd] = upd[i].second;
        a.n_upd++;
    }
    return TTS_BB_OK;
}

// Enqueue the multi-kernel decode step of the captured graph for this call's
// shape (B, head, which inputs and outputs), capturing it on the key's second
// call (the first runs eagerly, so every launcher's one-time setup has run).
// Per-call state travels in the step block; returns false to run eagerly.
bool decode_step_graph(tts_bb* h, int B, int head_idx, const int32_t* ids, const void* embeds, float* logits_out,
                       int32_t* argmax_out, int argmax_stride, float* hidden_out, const SetupArgs& a,
                       tts_bb_status& st) {
    const tts_bb_config& c = h->cfg;
    const bool want_head = head_idx >= 0 && (logits_out || argmax_out);
    const int key[7] = {B, want_head ? head_idx : -1, ids != nullptr, embeds != nullptr, logits_out != nullptr,
                        argmax_out != nullptr, hidden_out != nullptr};
    tts_bb::DecodeGraph* g = nullptr;
    for (auto& x : h->graphs)
        if (std::memcmp(x.key, key, sizeof key) == 0) g = &x;
    if (!g) {
        h->graphs.emplace_back();
        g = &h->graphs.back();
        std::memcpy(g->key, key, sizeof key);
    }
    if (g->bad || g->seen++ == 0) return false;
    // stage this call's state: wait until the ring entry's previous copy has been consumed
    const int i = h->ring_i;
    h->ring_i = (i + 1) % tts_bb::RING;
    if (h->ring_used[i]) cudaEventSynchronize(h->ring_ev[i]);
    StepBlock& sb = h->h_ring[i];
    std::memcpy(&sb.a, &a, sizeof(SetupArgs));
    sb.ids = ids;
    sb.embeds = reinterpret_cast<const bf16*>(embeds);
    sb.logits_out = logits_out;
    sb.argmax_out = argmax_out;
    sb.argmax_stride = argmax_stride;
    sb.hidden_out = hidden_out;
    if (!g->exec) {
        const uint64_t before = h->launches;
        cudaGraph_t graph = nullptr;
        bool ok = cudaStreamBeginCapture(h->st, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
        if (ok) {
            launch_pdl(k_step_setup, B, 256, 0, h->st, h->d_step, c.n_codebooks, h->seq_slot, h->seq_start, h->seq_len,
                                                h->key_len, h->d_page_table, h->amax, ids ? h->ids_buf : nullptr,
                                                embeds ? h->emb_buf : nullptr);
            h->launches += 1;
            h->launches += launch_embed_codebooks(h->tabs, ids ? h->ids_buf : nullptr, embeds ? h->emb_buf : nullptr,
                                                  h->h, B, h->err, h->st);
            KVView kv{h->pool, h->d_page_table, h->seq_slot, h->mbps};
            const bool folded = run_layers(h, B, 1, 0, c.max_ctx, kv, h->layer_elems, 0);  // attention grid sized for max_ctx
            if (want_head)
                run_head(h, B, 1, head_idx, false, logits_out ? h->logits_buf : nullptr, argmax_out, 1, true, false,
                         folded);
            launch_pdl(k_step_publish, B, 256, 0, h->st, h->d_step, want_head && logits_out ? h->logits_buf : nullptr,
                                                  c.head_rows, want_head && argmax_out ? h->amax : nullptr,
                                                  hidden_out ? h->h : nullptr);
            h->launches += 1;
            ok = cudaStreamEndCapture(h->st, &graph) == cudaSuccess && graph;
        }
        if (ok) ok = cudaGraphInstantiate(&g->exec, graph, 0) == cudaSuccess;
        if (graph) cudaGraphDestroy(graph);
        g->n_kernels = h->launches - before;
        h->launches = before;
        if (!ok) {
            cudaGetLastError();
            g->bad = true;
            g->exec = nullptr;
            return false;
        }
    }
    cudaError_t e = cudaMemcpyAsync(h->d_step, &sb, sizeof(StepBlock), cudaMemcpyHostToDevice, h->st);
    if (e == cudaSuccess) e = cudaEventRecord(h->ring_ev[i], h->st);
    h->ring_used[i] = true;
    if (e == cudaSuccess) e = cudaGraphLaunch(g->exec, h->st);
    if (e != cudaSuccess) {
        st = cuda_fail(h, e, "decode step graph");
        return true;
    }
    h->launches += g->n_kernels;
    st = finish(h);
    return true;
}

}  // namespace

// ============================================================== C ABI
TTS_API void tts_bb_default_config(tts_bb_config* c) {
    if (!c) return;
    std::memset(c, 0, sizeof *c);
    c->n_layers = 28;
    c->hidden = 1024;
    c->n_q_heads = 16;
    c->n_kv_heads = 8;
    c->head_dim = 128;
    c->ffn = 3072;
    c->rms_eps = 1e-6f;
    c->rope_theta = 1e6f;
    c->n_codebooks = 16;
    c->codebook_rows[0] = 3072;
    for (int k = 1; k < 16; ++k) c->codebook_rows[k] = 2048;
    c->n_heads = 1;
    c->head_rows = 3072;
    c->max_slots = 64;
    c->max_ctx = 4096;
    c->max_batch = 64;
    c->max_tokens = 4096;
    c->sync_errors = 1;
}

TTS_API const char* tts_bb_version(void) { return "0.1.0 (sm_103a)"; }

TTS_API const char* tts_bb_last_error(const tts_bb* h) { return h ? h->last_error.c_str() : "null handle"; }

TTS_API uint64_t tts_bb_launch_count(const tts_bb* h) { return h ? h->launches : 0; }

TTS_API tts_bb_status tts_bb_debug_fault(tts_bb* h, int what, int64_t arg) {
    if (!h) return TTS_BB_E_INVALID;
    switch (what) {
        case TTS_BB_DEBUG_WAIT_LIMIT_NS:
            if (arg < 1000000 || arg > 10000000000LL) return fail(h, TTS_BB_E_INVALID, "wait limit %lld ns outside 1e6..1e10", (long long)arg);
            h->wait_limit_ns = (unsigned long long)arg;
            return TTS_BB_OK;
        case TTS_BB_DEBUG_STALL_NEXT_STEP:
            h->stall_next = 1;
            return TTS_BB_OK;
        default:
            return fail(h, TTS_BB_E_INVALID, "unknown debug hook %d", what);
    }
}

TTS_API void tts_bb_free(tts_bb* h) {
    if (!h) return;
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(h->dev);
    if (h->st) cudaStreamSynchronize(h->st);
    else cudaDeviceSynchronize();
    for (auto& g : h->graphs)
        if (g.exec) cudaGraphExecDestroy(g.exec);
    for (int i = 0; i < tts_bb::RING; ++i)
        if (h->ring_ev[i]) cudaEventDestroy(h->ring_ev[i]);
    if (h->h_ring) cudaFreeHost(h->h_ring);
    for (void* p : h->allocs) cudaFree(p);
    if (h->h_err) cudaFreeHost(h->h_err);
    for (auto& r : h->prof) { cudaEventDestroy(r.a); cudaEventDestroy(r.b); }
    for (cudaEvent_t e : h->ev_pool) cudaEventDestroy(e);
    delete h->setup;
    delete h->mega;
    cudaSetDevice(cur);
    delete h;
}

// The body of tts_bb_create; `made` holds the handle once it exists, so a
// host allocation failure (std::bad_alloc) can free it at the C boundary.
static tts_bb_status create_impl(const tts_bb_config* cfg, const tts_bb_weights* w, void* stream, tts_bb** out,
                                 tts_bb*& made) {
    if (out) *out = nullptr;
    if (!cfg || !w || !out) return TTS_BB_E_INVALID;
    const tts_bb_config& c = *cfg;
    if (c.n_layers < 0 || c.n_layers > 256 || c.max_batch <= 0 || c.max_batch > MAX_B || c.max_tokens < 0 ||
        c.max_slots < 0 || c.max_ctx < 0 || c.n_codebooks < 0 || c.n_codebooks > TTS_BB_MAX_CODEBOOKS ||
        c.n_heads < 0 || c.n_heads > TTS_BB_MAX_HEADS || (c.n_heads > 0 && c.head_rows <= 0) || !(c.rms_eps > 0.f) ||
        !(c.rope_theta > 1.f) || (c.max_slots > 0 && c.max_ctx <= 0) || c.kv_blocks < 0)
        return TTS_BB_E_INVALID;
    std::string why;
    if (!cfg_supported(c, why)) return TTS_BB_E_UNSUPPORTED;
    if ((c.n_layers > 0 && !w->layer) || !w->final_norm) return TTS_BB_E_INVALID;
    for (int k = 0; k < c.n_codebooks; ++k)
        if (!w->codebook[k] || c.codebook_rows[k] <= 0) return TTS_BB_E_INVALID;
    const bool omni = c.text_vocab > 0 || c.audio_codebooks > 0;
    if (omni && (c.text_vocab <= 0 || c.audio_codebooks <= 0 || c.audio_vocab <= 0 || !w->text_table ||
                 !w->audio_table))
        return TTS_BB_E_INVALID;
    const int n_head_mats = omni ? (c.n_heads > 0 ? 1 : 0) : c.n_heads;
    for (int j = 0; j < n_head_mats; ++j)
        if (!w->head[j]) return TTS_BB_E_INVALID;
    for (int l = 0; l < c.n_layers; ++l)
        for (int r = 0; r < TTS_BB_LAYER_TENSORS; ++r)
            if (!w->layer[l * TTS_BB_LAYER_TENSORS + r]) return TTS_BB_E_INVALID;

    tts_bb* h = new tts_bb();
    made = h;
    h->cfg = c;
    h->st = reinterpret_cast<cudaStream_t>(stream);
    cudaGetDevice(&h->dev);
    h->setup = new SetupArgs();
    auto bail = [&](tts_bb_status s) {
        tts_bb_free(h);
        return s;
    };
    cudaError_t e;
    const size_t H = HID, F = c.ffn;
    // weights: one allocation per tensor family
    auto copy = [&](bf16* dst, const void* src, size_t n) {
        return cudaMemcpy(dst, src, n * sizeof(bf16), cudaMemcpyDefault);
    };
    h->L.resize(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
        const void* const* t = w->layer + (size_t)l * TTS_BB_LAYER_TENSORS;
        LayerW& lw = h->L[l];
        bf16* blk = nullptr;
        const size_t n = 3 * H + 2 * HD + (size_t)QKV * H + H * NQ * HD + 2 * F * H + H * F;
        if ((e = dalloc(h, &blk, n)) != cudaSuccess) return bail(TTS_BB_E_OOM);
        lw.in_norm = blk;
        lw.post_norm = lw.in_norm + H;
        lw.qn = lw.post_norm + H;
        lw.kn = lw.qn + HD;
        lw.wqkv = lw.kn + HD + H;  // keep 16-byte alignment
        lw.wo = lw.wqkv + (size_t)QKV * H;
        lw.wgu = lw.wo + H * NQ * HD;
        lw.wd = lw.wgu + 2 * F * H;
        if ((e = copy(lw.in_norm, t[TTS_BB_W_IN_NORM], H)) != cudaSuccess ||
            (e = copy(lw.post_norm, t[TTS_BB_W_POST_NORM], H)) != cudaSuccess ||
            (e = copy(lw.qn, t[TTS_BB_W_Q_NORM], HD)) != cudaSuccess ||
            (e = copy(lw.kn, t[TTS_BB_W_K_NORM], HD)) != cudaSuccess ||
            (e = copy(lw.wqkv, t[TTS_BB_W_Q], (size_t)NQ * HD * H)) != cudaSuccess ||
            (e = copy(lw.wqkv + (size_t)NQ * HD * H, t[TTS_BB_W_K], (size_t)NKV * HD * H)) != cudaSuccess ||
            (e = copy(lw.wqkv + (size_t)(NQ + NKV) * HD * H, t[TTS_BB_W_V], (size_t)NKV * HD * H)) != cudaSuccess ||
            (e = copy(lw.wo, t[TTS_BB_W_O], H * NQ * HD)) != cudaSuccess ||
            (e = copy(lw.wd, t[TTS_BB_W_DOWN], H * F)) != cudaSuccess)
            return bail(cuda_fail(h, e, "weight copy"));
        // gate/up interleaved by row: row 2i = gate_i, row 2i+1 = up_i
        if ((e = cudaMemcpy2D(lw.wgu, 2 * H * sizeof(bf16), t[TTS_BB_W_GATE], H * sizeof(bf16), H * sizeof(bf16), F,
                              cudaMemcpyDefault)) != cudaSuccess ||
            (e = cudaMemcpy2D(lw.wgu + H, 2 * H * sizeof(bf16), t[TTS_BB_W_UP], H * sizeof(bf16), H * sizeof(bf16), F,
                              cudaMemcpyDefault)) != cudaSuccess)
            return bail(cuda_fail(h, e, "weight copy"));
    }
    h->tabs.n = c.n_codebooks;
    for (int k = 0; k < c.n_codebooks; ++k) {
        bf16* p = nullptr;
        if ((e = dalloc(h, &p, (size_t)c.codebook_rows[k] * H)) != cudaSuccess) return bail(TTS_BB_E_OOM);
        if ((e = copy(p, w->codebook[k], (size_t)c.codebook_rows[k] * H)) != cudaSuccess)
            return bail(cuda_fail(h, e, "table copy"));
        h->tabs.tab[k] = p;
        h->tabs.rows[k] = c.codebook_rows[k];
    }
    if (omni) {
        if ((e = dalloc(h, &h->text, (size_t)c.text_vocab * H)) != cudaSuccess ||
            (e = dalloc(h, &h->audio, (size_t)c.audio_codebooks * c.audio_vocab * H)) != cudaSuccess)
            return bail(TTS_BB_E_OOM);
        if ((e = copy(h->text, w->text_table, (size_t)c.text_vocab * H)) != cudaSuccess ||
            (e = copy(h->audio, w->audio_table, (size_t)c.audio_codebooks * c.audio_vocab * H)) != cudaSuccess)
            return bail(cuda_fail(h, e, "table copy"));
    }
    if ((e = dalloc(h, &h->final_norm, H)) != cudaSuccess) return bail(TTS_BB_E_OOM);
    if ((e = copy(h->final_norm, w->final_norm, H)) != cudaSuccess) return bail(cuda_fail(h, e, "norm copy"));
    for (int j = 0; j < n_head_mats; ++j) {
        const size_t rows = omni ? (size_t)c.n_heads * c.head_rows : (size_t)c.head_rows;
        if ((e = dalloc(h, &h->heads[j], rows * H)) != cudaSuccess) return bail(TTS_BB_E_OOM);
        if ((e = copy(h->heads[j], w->head[j], rows * H)) != cudaSuccess) return bail(cuda_fail(h, e, "head copy"));
    }
    // RoPE tables, computed in double on the host: angle = pos * theta^(-2i/128)
    h->rope_len = std::max(std::max(c.max_ctx, c.max_tokens), 1);
    {
        std::vector<float> ct((size_t)h->rope_len * (HD / 2)), sn((size_t)h->rope_len * (HD / 2));
        for (int p = 0; p < h->rope_len; ++p)
            for (int i = 0; i < HD / 2; ++i) {
                const double inv = std::pow((double)c.rope_theta, -2.0 * i / HD);
                const double a = (double)p * inv;
                ct[(size_t)p * (HD / 2) + i] = (float)std::cos(a);
                sn[(size_t)p * (HD / 2) + i] = (float)std::sin(a);
            }
        if ((e = dalloc(h, &h->cos_t, ct.size())) != cudaSuccess || (e = dalloc(h, &h->sin_t, sn.size())) != cudaSuccess)
            return bail(TTS_BB_E_OOM);
        cudaMemcpy(h->cos_t, ct.data(), ct.size() * sizeof(float), cudaMemcpyHostToDevice);
        cudaMemcpy(h->sin_t, sn.data(), sn.size() * sizeof(float), cudaMemcpyHostToDevice);
    }
    // KV pool [layer][block][K|V][8][64][128]
    if (c.max_slots > 0) {
        h->mbps = (c.max_ctx + KVB - 1) / KVB;
        long long nblk = c.kv_blocks > 0 ? (long long)c.kv_blocks : (long long)c.max_slots * h->mbps;
        if (const char* cap = std::getenv("TTS_BB_MAX_BLOCKS")) {
            const long long v = std::atoll(cap);
            if (v > 0) nblk = std::min(nblk, v);
        }
        if (nblk > INT32_MAX) return bail(TTS_BB_E_UNSUPPORTED);  // physical block ids are int32
        h->kv_blocks = (int)nblk;
        h->layer_elems = (size_t)h->kv_blocks * 2 * NKV * KVB * HD;
        if ((e = dalloc(h, &h->pool, h->layer_elems * c.n_layers)) != cudaSuccess) return bail(TTS_BB_E_OOM);
        if ((e = dalloc(h, &h->d_page_table, (size_t)c.max_slots * h->mbps)) != cudaSuccess) return bail(TTS_BB_E_OOM);
        h->page_table.assign((size_t)c.max_slots * h->mbps, -1);
        cudaMemcpy(h->d_page_table, h->page_table.data(), h->page_table.size() * sizeof(int32_t),
                   cudaMemcpyHostToDevice);
        h->slot_len.assign(c.max_slots, 0);
        h->free_blocks.resize(h->kv_blocks);
        for (int i = 0; i < h->kv_blocks; ++i) h->free_blocks[i] = h->kv_blocks - 1 - i;  // pop_back gives 0, 1, ...
    }
    const int nb = std::max(c.max_batch, 1);
    if ((e = dalloc(h, &h->part, (size_t)nb * NQ * MAX_SPLITS * (HD + 2))) != cudaSuccess ||
        (e = dalloc(h, &h->amax, (size_t)std::max(nb, c.max_tokens))) != cudaSuccess ||
        (e = dalloc(h, &h->seq_slot, MAX_B)) != cudaSuccess || (e = dalloc(h, &h->seq_start, MAX_B)) != cudaSuccess ||
        (e = dalloc(h, &h->seq_len, MAX_B)) != cudaSuccess || (e = dalloc(h, &h->key_len, MAX_B)) != cudaSuccess ||
        (e = dalloc(h, &h->err, 1)) != cudaSuccess)
        return bail(TTS_BB_E_OOM);
    if ((e = cudaMallocHost(&h->h_err, sizeof(int))) != cudaSuccess) return bail(TTS_BB_E_OOM);
    if (c.max_batch > 8) {  // K splits x N, largest over the decode GEMMs, for K slices of 256 / token-tiles
        const int mt = c.max_batch <= 64 ? 1 : (c.max_batch <= 128 ? 2 : 4);
        const size_t ks_n = std::max(std::max((size_t)(HID * mt / 256) * 2 * c.ffn, (size_t)(NQ * HD * mt / 256) * HID),
                                     std::max((size_t)(c.ffn * mt / 256) * HID, (size_t)(HID * mt / 256) * QKV));
        h->sk.part_elems = std::max(ks_n, (size_t)(HID * mt / 256) * std::max(c.head_rows, 1)) * c.max_batch;
        h->sk.n_ctr = 256;
        if ((e = dalloc(h, &h->sk.part, h->sk.part_elems)) != cudaSuccess || (e = dalloc(h, &h->sk.ctr, 256)) != cudaSuccess)
            return bail(TTS_BB_E_OOM);
        cudaMemset(h->sk.ctr, 0, 256 * sizeof(int));
    }
    {
        const char* av = std::getenv("TTS_BB_BIDIR_ATTN");  // "mma": the mma.sync flash kernel for the bidirectional pass
        h->attn_bidir_tc = gemm_tc_available() && !(av && std::strcmp(av, "mma") == 0);
        const char* pv = std::getenv("TTS_BB_PREFILL_ATTN");  // "mma": the mma.sync flash kernel for the causal prefill
        h->attn_causal_tc = gemm_tc_available() && !(pv && std::strcmp(pv, "mma") == 0);
        const char* fq = std::getenv("TTS_BB_QKV_EPILOGUE");  // "separate": the q/k norm + RoPE + append kernel
        h->fuse_qk = gemm_tc_available() && !(fq && std::strcmp(fq, "separate") == 0);
        const char* fnm = std::getenv("TTS_BB_NORM_FOLD");  // "off": the RMSNorm kernels in decode batches
        h->fold_norm = gemm_tc_available() && !(fnm && std::strcmp(fnm, "off") == 0);
        h->short_prefill_attn = !(pv && std::strcmp(pv, "mma") == 0);  // TTS_BB_PREFILL_ATTN=mma: every prefill on mma.sync
    }
    if (c.max_slots > 0) {  // graph-replayed decode steps: step block, staging ring, fixed input / output buffers
        const char* gv = std::getenv("TTS_BB_GRAPHS");
        h->graphs_on = !(gv && std::strcmp(gv, "0") == 0);
        if ((e = dalloc(h, &h->d_step, 1)) != cudaSuccess ||
            (e = dalloc(h, &h->ids_buf, (size_t)c.max_batch * std::max(c.n_codebooks, 1))) != cudaSuccess ||
            (e = dalloc(h, &h->emb_buf, (size_t)c.max_batch * HID)) != cudaSuccess ||
            (e = dalloc(h, &h->logits_buf, (size_t)c.max_batch * std::max(c.head_rows, 1))) != cudaSuccess ||
            cudaMallocHost(&h->h_ring, tts_bb::RING * sizeof(StepBlock)) != cudaSuccess)
            return bail(TTS_BB_E_OOM);
        for (int i = 0; i < tts_bb::RING; ++i)
            if (cudaEventCreateWithFlags(&h->ring_ev[i], cudaEventDisableTiming) != cudaSuccess) return bail(TTS_BB_E_CUDA);
    }
    cudaMemset(h->err, 0, sizeof(int));
    tts_bb_status s = ensure_scratch(h, std::max(nb, std::max(c.max_tokens, 1)));
    if (s != TTS_BB_OK) return bail(s);
    // persistent decode step: abort flag, exchange words, argmax words, constant arguments
    if (c.max_slots > 0 && c.n_layers >= 1 && c.n_layers <= mk::MAXL && c.max_ctx <= 64 * KVB && c.ffn == 3072 && (c.n_heads == 0 || (c.head_rows % 2 == 0 && c.head_rows <= 6144)) && c.text_vocab == 0) {
        h->mega_grid = ll_max_grid();
        cudaGetLastError();
        // 128 CTAs split every matrix evenly (QKV 32, o_proj / down 8, gate/up 48, head 24 rows per CTA),
        // so no CTA carries an extra row pair into the critical path: measured faster than all 152 SMs
        // (2040 vs 1911 tokens/s at batch 1) and than every grid from 96 to 144 tried.
        if (h->mega_grid >= 128) h->mega_grid = 128;
        if (const char* pf = std::getenv("TTS_BB_L2_PREFETCH")) h->l2_prefetch = std::atoi(pf) & 3;
        if (const char* g = std::getenv("TTS_BB_DECODE_CTAS"))  // tuning knob: CTAs of the persistent step
            h->mega_grid = std::max(std::min(ll_max_grid(), LL_MIN_GRID), std::min(ll_max_grid(), std::atoi(g)));
        if (h->mega_grid > 0) {
            const size_t xw = ll_xbuf_words(h->mbps);
            if ((e = dalloc(h, &h->mega_abort, 1)) != cudaSuccess ||
                (e = dalloc(h, &h->ll_xbuf, xw)) != cudaSuccess || (e = dalloc(h, &h->ll_amax, mk::MAXB)) != cudaSuccess ||
                (e = dalloc(h, &h->ll_done, 1)) != cudaSuccess)
                return bail(TTS_BB_E_OOM);
            cudaMemset(h->mega_abort, 0, sizeof(int));
            cudaMemset(h->ll_xbuf, 0, xw * sizeof(unsigned long long));
            cudaMemset(h->ll_amax, 0, mk::MAXB * sizeof(unsigned long long));
            cudaMemset(h->ll_done, 0, sizeof(unsigned int));
            MegaArgs* ma = new MegaArgs();
            std::memset(ma, 0, sizeof *ma);
            for (int l = 0; l < c.n_layers; ++l) {
                const LayerW& lw = h->L[l];
                ma->L[l] = {lw.in_norm, lw.wqkv, lw.qn, lw.kn, lw.wo, lw.post_norm, lw.wgu, lw.wd};
            }
            ma->tabs = h->tabs;
            ma->final_norm = h->final_norm;
            ma->head_rows = c.head_rows;
            ma->pool = h->pool;
            ma->layer_elems = h->layer_elems;
            ma->page_table = h->d_page_table;
            ma->mbps = h->mbps;
            ma->h = h->h;
            ma->qkv = h->qkv;
            ma->nblk_max = h->mbps;
            ma->amax = h->ll_amax;
            ma->abort_flag = h->mega_abort;
            ma->xbuf = h->ll_xbuf;
            ma->done = h->ll_done;
            ma->err = h->err;
            ma->cos_t = h->cos_t;
            ma->sin_t = h->sin_t;
            ma->eps = c.rms_eps;
            ma->n_layers = c.n_layers;
            ma->ffn = c.ffn;
            h->mega = ma;
        }
    }
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return bail(cuda_fail(h, e, "create"));
    *out = h;
    return TTS_BB_OK;
}

TTS_API tts_bb_status tts_bb_create(const tts_bb_config* cfg, const tts_bb_weights* w, void* stream, tts_bb** out) {
    tts_bb* made = nullptr;
    try {
        return create_impl(cfg, w, stream, out, made);
    } catch (const std::bad_alloc&) {  // no exception crosses the C boundary
        if (made) tts_bb_free(made);
        if (out) *out = nullptr;
        return TTS_BB_E_OOM;
    }
}

TTS_API int tts_bb_slot_len(const tts_bb* h, int slot) {
    if (!h || slot < 0 || slot >= h->cfg.max_slots) return -1;
    return h->slot_len[slot];
}

TTS_API tts_bb_status tts_bb_truncate(tts_bb* h, int slot, int len) {
    if (!h) return TTS_BB_E_INVALID;
    if (slot < 0 || slot >= h->cfg.max_slots) return fail(h, TTS_BB_E_INVALID, "slot %d out of range", slot);
    if (len < 0 || len > h->slot_len[slot]) return fail(h, TTS_BB_E_INVALID, "truncate length %d invalid", len);
    const int keep = (len + KVB - 1) / KVB, have = (h->slot_len[slot] + KVB - 1) / KVB;
    for (int j = keep; j < have; ++j) {
        int32_t& e = h->page_table[(size_t)slot * h->mbps + j];
        h->free_blocks.push_back(e);
        e = -1;
    }
    h->slot_len[slot] = len;
    // the device copy of freed entries is not cleared: freed blocks are only
    // reachable again after a new append rewrites the entry.
    return TTS_BB_OK;
}

TTS_API tts_bb_status tts_bb_release(tts_bb* h, int slot) { return tts_bb_truncate(h, slot, 0); }

TTS_API tts_bb_status tts_bb_sync(tts_bb* h) {
    if (!h) return TTS_BB_E_INVALID;
    return read_err(h);
}

TTS_API tts_bb_status tts_bb_decode_step(tts_bb* h, int B, const int32_t* slots, const int32_t* kv_lens,
                                         const int32_t* ids, int head_idx, float* logits_out, int32_t* argmax_out,
                                         const tts_bb_opts* opts) {
    if (!h) return TTS_BB_E_INVALID;
    const tts_bb_config& c = h->cfg;
    if (c.max_slots <= 0) return fail(h, TTS_BB_E_UNSUPPORTED, "handle has no KV cache");
    if (B <= 0 || B > c.max_batch) return fail(h, TTS_BB_E_INVALID, "B=%d outside 1..%d", B, c.max_batch);
    if (!slots_ok(h, B, slots)) return fail(h, TTS_BB_E_INVALID, "slots must be distinct and in range");
    if (!kv_lens) return fail(h, TTS_BB_E_INVALID, "kv_lens is NULL");
    const void* embeds = opts ? opts->embeds : nullptr;
    if (!ids && !embeds) return fail(h, TTS_BB_E_INVALID, "need ids or embeds");
    if (ids && c.n_codebooks == 0) return fail(h, TTS_BB_E_INVALID, "handle has no codebook tables");
    if (head_idx >= c.n_heads || head_idx < -1) return fail(h, TTS_BB_E_INVALID, "head_idx %d out of range", head_idx);
    if (head_idx < 0 && (logits_out || argmax_out)) return fail(h, TTS_BB_E_INVALID, "outputs need a head");
    std::vector<int> nl(B);
    for (int b = 0; b < B; ++b) {
        if (kv_lens[b] != h->slot_len[slots[b]])
            return fail(h, TTS_BB_E_INVALID, "kv_lens[%d]=%d but slot %d holds %d tokens", b, kv_lens[b], slots[b],
                        h->slot_len[slots[b]]);
        if (kv_lens[b] + 1 > c.max_ctx) return fail(h, TTS_BB_E_INVALID, "slot %d would exceed max_ctx", slots[b]);
        nl[b] = kv_lens[b] + 1;
    }
    SetupArgs& a = *h->setup;
    a.B = B;
    a.clear_amax = argmax_out != nullptr;
    tts_bb_status s = grow_slots(h, B, slots, nl.data(), a);
    if (s != TTS_BB_OK) return s;
    for (int b = 0; b < B; ++b) {
        a.slot[b] = slots[b];
        a.start[b] = kv_lens[b];
        a.len[b] = 1;
        a.key_len[b] = nl[b];
        h->slot_len[slots[b]] = nl[b];
    }
    const char* path = std::getenv("TTS_BB_DECODE_PATH");
    const bool want_head = head_idx >= 0 && (logits_out || argmax_out);
    if (h->mega && B <= mk::MAXB && !(path && std::strcmp(path, "multi") == 0)) {
        MegaArgs ma = *h->mega;
        ma.ids = ids;
        ma.embeds = reinterpret_cast<const bf16*>(embeds);
        ma.head = want_head ? h->heads[head_idx] : nullptr;
        ma.logits = want_head ? logits_out : nullptr;
        ma.argmax_out = want_head ? argmax_out : nullptr;
        ma.argmax_stride = opts && opts->argmax_stride ? opts->argmax_stride : 1;
        ma.B = B;
        for (int b = 0; b < B; ++b) {
            ma.slot[b] = slots[b];
            ma.pos[b] = kv_lens[b];
        }
        ma.n_upd = a.n_upd;
        for (int i = 0; i < a.n_upd; ++i) {
            ma.upd_idx[i] = a.upd_idx[i];
            ma.upd_val[i] = a.upd_val[i];
        }
        ma.ep_base = h->ep_base;
        ma.timeout_ns = h->wait_limit_ns;
        ma.debug_stall = h->stall_next;
        ma.l2_prefetch = h->l2_prefetch;
        h->stall_next = 0;
        for (int b = 0; b < B; ++b) ma.last_phys[b] = h->page_table[(size_t)slots[b] * h->mbps + kv_lens[b] / KVB];
        ma.trace = nullptr;
        if (h->prof_on) {
            if (!h->mega_trace &&
                dalloc(h, &h->mega_trace, (size_t)h->mega_grid * mk::MAXL * TRACE_STRIDE) != cudaSuccess)
                return fail(h, TTS_BB_E_OOM, "trace buffer");
            if (h->phase_n == 0)
                cudaMemsetAsync(h->mega_trace, 0, (size_t)h->mega_grid * mk::MAXL * TRACE_STRIDE * 8, h->st);
            ma.trace = h->mega_trace;
        }
        double kvb = 0;
        for (int b = 0; b < B; ++b) kvb += (double)nl[b] * 2 * NKV * HD * 2 * c.n_layers;
        const double wbytes = (double)c.n_layers * 2.0 * HID * (QKV + NQ * HD + 3.0 * c.ffn) +
                              (ma.head ? 2.0 * c.head_rows * HID : 0);
        {
            Launch L(h, K_MEGA, wbytes + kvb, 2.0 * B * wbytes / 2);
            const cudaError_t e = launch_decode_ll(ma, h->mega_grid, h->st);
            if (e != cudaSuccess) return cuda_fail(h, e, "persistent decode step launch");
            L += 1;
        }
        h->ep_base += ll_epochs_per_launch(c.n_layers);
        if (ma.trace) {  // fold this launch's phase stamps into the profile (synchronises)
            const int NS = TRACE_STRIDE, NP = 10, G = h->mega_grid, NL = c.n_layers;
            std::vector<unsigned long long> st((size_t)G * NL * NS, 0ull);
            cudaMemcpyAsync(st.data(), h->mega_trace, st.size() * 8, cudaMemcpyDeviceToHost, h->st);
            cudaStreamSynchronize(h->st);
            if (h->phase_us.empty()) { h->phase_us.assign(NP, 0.0); h->phase_max_us.assign(NP, 0.0); }
            for (int l = 0; l < NL; ++l)
                for (int i = 0; i < NP; ++i) {
                    if (i == NP - 1 && l + 1 >= NL) continue;
                    double sum = 0, mx = 0;
                    for (int g = 0; g < G; ++g) {
                        const unsigned long long* r = &st[((size_t)g * NL + l) * NS];
                        const unsigned long long nxt = (i == NP - 1) ? st[((size_t)g * NL + l + 1) * NS] : r[i + 1];
                        const double d = (double)(nxt - r[i]) * 1e-3;
                        sum += d;
                        mx = d > mx ? d : mx;
                    }
                    h->phase_us[i] += sum / G;
                    h->phase_max_us[i] += mx;
                }
            // ring waits inside gate/up (stamps 6 -> 20) and down (8 -> 30)
            for (int l = 0; l < NL; ++l)
                for (int g = 0; g < G; ++g) {
                    const unsigned long long* r = &st[((size_t)g * NL + l) * NS];
                    if (!r[20] || !r[30]) continue;
                    h->ring_wait[0] += (r[20] - r[6]) * 1e-3;
                    h->ring_wait[1] += (r[30] - r[8]) * 1e-3;
                    h->ring_wait_n++;
                }
            // attention-unit phase (stamps 2 -> 3) split by whether the CTA ran a unit
            for (int l = 0; l < NL; ++l)
                for (int g = 0; g < G; ++g) {
                    const unsigned long long* r = &st[((size_t)g * NL + l) * NS];
                    const int k = r[15] ? 1 : 0;
                    h->unit_split[k] += (r[3] - r[2]) * 1e-3;
                    h->unit_split_n[k]++;
                }
            h->phase_n += NL;
            if (const char* dump = std::getenv("TTS_BB_TRACE_DUMP")) {  // raw stamps of the latest launch
                if (FILE* f = std::fopen(dump, "wb")) {
                    std::fwrite(st.data(), 8, st.size(), f);
                    std::fclose(f);
                }
            }
            cudaMemsetAsync(h->mega_trace, 0, st.size() * 8, h->st);
        }
        if (opts && opts->hidden_out)
            cudaMemcpyAsync(opts->hidden_out, h->h, (size_t)B * HID * sizeof(float), cudaMemcpyDeviceToDevice, h->st);
        return finish(h);
    }
    if (h->graphs_on && !h->prof_on) {
        tts_bb_status gs = TTS_BB_OK;
        if (decode_step_graph(h, B, head_idx, ids, embeds, logits_out, argmax_out,
                              opts && opts->argmax_stride ? opts->argmax_stride : 1, opts ? opts->hidden_out : nullptr, a,
                              gs))
            return gs;
    }
    launch_setup(h, a);
    {
        Launch L(h, K_EMBED, B * (4.0 * HID + (ids ? 2.0 * HID * c.n_codebooks : 0) + (embeds ? 2.0 * HID : 0)));
        L += launch_embed_codebooks(h->tabs, ids, reinterpret_cast<const bf16*>(embeds), h->h, B, h->err, h->st);
    }
    KVView kv{h->pool, h->d_page_table, h->seq_slot, h->mbps};
    double kv_bytes = 0;
    for (int b = 0; b < B; ++b) kv_bytes += (double)nl[b] * 2 * NKV * HD * 2;
    // attention splits are sized for max_ctx here as in the graph-replayed step, so a step's
    // summation order (and result) does not depend on which of the two ran
    const bool folded = run_layers(h, B, 1, 0, c.max_ctx, kv, h->layer_elems, kv_bytes);
    if (opts && opts->hidden_out)
        cudaMemcpyAsync(opts->hidden_out, h->h, (size_t)B * HID * sizeof(float), cudaMemcpyDeviceToDevice, h->st);
    if (head_idx >= 0 && (logits_out || argmax_out))
        run_head(h, B, 1, head_idx, false, logits_out, argmax_out, opts && opts->argmax_stride ? opts->argmax_stride : 1,
                 true, true, folded);
    return finish(h);
}

TTS_API tts_bb_status tts_bb_prefill(tts_bb* h, int B, int S, const int32_t* slots, const int32_t* lens,
                                     const int32_t* ids, int head_idx, float* logits_out, int32_t* argmax_out,
                                     const tts_bb_opts* opts) {
    if (!h) return TTS_BB_E_INVALID;
    const tts_bb_config& c = h->cfg;
    if (c.max_slots <= 0) return fail(h, TTS_BB_E_UNSUPPORTED, "handle has no KV cache");
    if (B <= 0 || B > c.max_batch || S <= 0 || (long)B * S > std::max(c.max_tokens, c.max_batch))
        return fail(h, TTS_BB_E_INVALID, "B=%d S=%d outside the configured sizes", B, S);
    if (!slots_ok(h, B, slots)) return fail(h, TTS_BB_E_INVALID, "slots must be distinct and in range");
    if (!lens) return fail(h, TTS_BB_E_INVALID, "lens is NULL");
    const void* embeds = opts ? opts->embeds : nullptr;
    if (!ids && !embeds) return fail(h, TTS_BB_E_INVALID, "need ids or embeds");
    if (ids && c.n_codebooks == 0) return fail(h, TTS_BB_E_INVALID, "handle has no codebook tables");
    if (head_idx >= c.n_heads || head_idx < -1) return fail(h, TTS_BB_E_INVALID, "head_idx %d out of range", head_idx);
    if (head_idx < 0 && (logits_out || argmax_out)) return fail(h, TTS_BB_E_INVALID, "outputs need a head");
    std::vector<int> nl(B);
    for (int b = 0; b < B; ++b) {
        if (lens[b] < 1 || lens[b] > S) return fail(h, TTS_BB_E_INVALID, "lens[%d]=%d outside 1..%d", b, lens[b], S);
        nl[b] = h->slot_len[slots[b]] + lens[b];
        if (nl[b] > c.max_ctx) return fail(h, TTS_BB_E_INVALID, "slot %d would exceed max_ctx", slots[b]);
    }
    SetupArgs& a = *h->setup;
    a.B = B;
    a.clear_amax = argmax_out != nullptr;
    tts_bb_status s = grow_slots(h, B, slots, nl.data(), a);
    if (s != TTS_BB_OK) return s;
    for (int b = 0; b < B; ++b) {
        a.slot[b] = slots[b];
        a.start[b] = h->slot_len[slots[b]];
        a.len[b] = lens[b];
        a.key_len[b] = nl[b];
        h->slot_len[slots[b]] = nl[b];
    }
    launch_setup(h, a);
    const int T = B * S;
    {
        Launch L(h, K_EMBED, T * (4.0 * HID + (ids ? 2.0 * HID * c.n_codebooks : 0) + (embeds ? 2.0 * HID : 0)));
        L += launch_embed_codebooks(h->tabs, ids, reinterpret_cast<const bf16*>(embeds), h->h, T, h->err, h->st);
    }
    KVView kv{h->pool, h->d_page_table, h->seq_slot, h->mbps};
    double aflops = 0;   // causal: query j of a row sees start + j + 1 keys
    for (int b = 0; b < B; ++b)
        aflops += 4.0 * NQ * HD * ((double)lens[b] * a.start[b] + 0.5 * (double)lens[b] * (lens[b] + 1));
    run_layers(h, B, S, 1, 0, kv, h->layer_elems, 0, aflops);
    if (opts && opts->hidden_out)
        cudaMemcpyAsync(opts->hidden_out, h->h, (size_t)T * HID * sizeof(float), cudaMemcpyDeviceToDevice, h->st);
    if (head_idx >= 0 && (logits_out || argmax_out))
        run_head(h, B, S, head_idx, true, logits_out, argmax_out, opts && opts->argmax_stride ? opts->argmax_stride : 1, true);
    return finish(h);
}

TTS_API tts_bb_status tts_bb_maskgit_pass(tts_bb* h, int B, int S, const int32_t* ids, const uint8_t* audio_mask,
                                          const int32_t* key_lens, int audio_start, float* logits_out,
                                          const tts_bb_opts* opts) {
    if (!h) return TTS_BB_E_INVALID;
    const tts_bb_config& c = h->cfg;
    if (!h->text || !h->audio) return fail(h, TTS_BB_E_UNSUPPORTED, "handle has no text/audio tables");
    if (B <= 0 || B > c.max_batch || S <= 0 || (long)B * S > c.max_tokens)
        return fail(h, TTS_BB_E_INVALID, "B=%d S=%d outside the configured sizes", B, S);
    if (S > h->rope_len) return fail(h, TTS_BB_E_INVALID, "S=%d beyond the RoPE table", S);
    if (!ids || !audio_mask) return fail(h, TTS_BB_E_INVALID, "ids and audio_mask are required");
    if (audio_start < 0 || audio_start >= S) return fail(h, TTS_BB_E_INVALID, "audio_start %d outside 0..S-1", audio_start);
    if (logits_out && c.n_heads <= 0) return fail(h, TTS_BB_E_INVALID, "handle has no audio heads");
    if (key_lens)
        for (int b = 0; b < B; ++b)
            if (key_lens[b] < 1 || key_lens[b] > S) return fail(h, TTS_BB_E_INVALID, "key_lens[%d] outside 1..S", b);
    const int bps = (S + KVB - 1) / KVB;
    const size_t need_blocks = (size_t)B * bps;
    if (need_blocks > h->mg_pool_blocks) {
        if (h->mg_pool) {
            cudaStreamSynchronize(h->st);
            cudaFree(h->mg_pool);
            h->allocs.erase(std::remove(h->allocs.begin(), h->allocs.end(), (void*)h->mg_pool), h->allocs.end());
            h->mg_pool = nullptr;
            h->mg_pool_blocks = 0;
        }
        cudaError_t e = dalloc(h, &h->mg_pool, need_blocks * 2 * NKV * KVB * HD);
        if (e != cudaSuccess) return cuda_fail(h, e, "MaskGIT scratch");
        // keys past a sequence's end are masked (probability 0) but still multiplied: keep them finite
        e = cudaMemsetAsync(h->mg_pool, 0, need_blocks * 2 * NKV * KVB * HD * sizeof(bf16), h->st);
        if (e != cudaSuccess) return cuda_fail(h, e, "MaskGIT scratch");
        h->mg_pool_blocks = need_blocks;
    }
    SetupArgs& a = *h->setup;
    a.B = B;
    a.n_upd = 0;
    a.clear_amax = 0;
    for (int b = 0; b < B; ++b) {
        a.slot[b] = b;
        a.start[b] = 0;
        a.len[b] = S;
        a.key_len[b] = key_lens ? key_lens[b] : S;
    }
    launch_setup(h, a);
    {
        Launch L(h, K_EMBED);
        L += launch_embed_omnivoice(h->text, c.text_vocab, h->audio, c.audio_codebooks, c.audio_vocab, ids, audio_mask,
                                    h->h, B, S, h->err, h->st);
    }
    KVView kv{h->mg_pool, nullptr, h->seq_slot, bps};
    double aflops = 0;
    for (int b = 0; b < B; ++b) aflops += 4.0 * NQ * HD * (double)S * a.key_len[b];
    run_layers(h, B, S, 2, 0, kv, 0, 0, aflops);
    if (opts && opts->hidden_out)
        cudaMemcpyAsync(opts->hidden_out, h->h, (size_t)B * S * HID * sizeof(float), cudaMemcpyDeviceToDevice, h->st);
    if (logits_out) {
        const int Sa = S - audio_start;
        { Launch L(h, K_RMSNORM, B * Sa * 6.0 * HID);
          L += launch_rmsnorm(h->h, h->final_norm, h->y, B * Sa, c.rms_eps, Sa, S, audio_start, nullptr, h->st); }
        Epi e{};
        e.mode = EPI_LOGITS_PERM; e.out = logits_out; e.perm_rows = Sa; e.perm_vocab = c.head_rows;
        e.perm_groups = c.n_heads;
        const int N = c.n_heads * c.head_rows;
        Launch L(h, B * Sa <= 8 ? K_GEMV : K_GEMM_TC, gemm_bytes(B * Sa, N, HID, 4), 2.0 * B * Sa * N * HID);
        L += launch_gemm(h->y, h->heads[0], B * Sa, N, HID, e, h->st, nullptr, h->err);
    }
    return finish(h);
}

TTS_API tts_bb_status tts_bb_decode_step_host(tts_bb* h, int B, const int32_t* slots, const int32_t* kv_lens,
                                              const int32_t* ids, int head_idx, int32_t* argmax_out,
                                              float* logits_out) {
    if (!h) return TTS_BB_E_INVALID;
    const tts_bb_config& c = h->cfg;
    if (!ids || c.n_codebooks <= 0) return fail(h, TTS_BB_E_INVALID, "decode_step_host needs host ids and codebook tables");
    if (B <= 0 || B > c.max_batch) return fail(h, TTS_BB_E_INVALID, "B=%d outside 1..%d", B, c.max_batch);
    const int rows = std::max(c.head_rows, 1);
    if (!h->hx_ids) {
        cudaError_t e = dalloc(h, &h->hx_ids, (size_t)c.max_batch * c.n_codebooks);
        if (e == cudaSuccess) e = dalloc(h, &h->hx_am, (size_t)c.max_batch);
        if (e == cudaSuccess) e = dalloc(h, &h->hx_logits, (size_t)c.max_batch * rows);
        if (e != cudaSuccess) return cuda_fail(h, e, "host-buffer staging");
    }
    cudaError_t e = cudaMemcpyAsync(h->hx_ids, ids, (size_t)B * c.n_codebooks * sizeof(int32_t), cudaMemcpyHostToDevice,
                                    h->st);
    if (e != cudaSuccess) return cuda_fail(h, e, "ids copy");
    const bool sync_errors = h->cfg.sync_errors;
    h->cfg.sync_errors = 0;  // one synchronisation at the end, below
    const tts_bb_status st = tts_bb_decode_step(h, B, slots, kv_lens, h->hx_ids, head_idx,
                                                logits_out ? h->hx_logits : nullptr, argmax_out ? h->hx_am : nullptr,
                                                nullptr);
    h->cfg.sync_errors = sync_errors;
    if (st != TTS_BB_OK) return st;
    if (argmax_out &&
        (e = cudaMemcpyAsync(argmax_out, h->hx_am, (size_t)B * sizeof(int32_t), cudaMemcpyDeviceToHost, h->st)) != cudaSuccess)
        return cuda_fail(h, e, "argmax copy");
    if (logits_out && (e = cudaMemcpyAsync(logits_out, h->hx_logits, (size_t)B * rows * sizeof(float),
                                           cudaMemcpyDeviceToHost, h->st)) != cudaSuccess)
        return cuda_fail(h, e, "logits copy");
    return read_err(h);  // the error word's copy and the one stream synchronisation
}

TTS_API tts_bb_status tts_bb_frame_step(tts_bb* talker, tts_bb* cp, int B, const int32_t* slots,
                                        const int32_t* kv_lens, int32_t* codes, float* talker_logits) {
    if (!talker || !cp) return TTS_BB_E_INVALID;
    const tts_bb_config &tc = talker->cfg, &cc = cp->cfg;
    if (talker->st != cp->st) return fail(cp, TTS_BB_E_INVALID, "frame_step: both handles must share one stream");
    if (tc.n_codebooks != 16 || cc.n_codebooks != 16 || tc.n_heads < 1 || cc.n_heads < 15)
        return fail(cp, TTS_BB_E_INVALID, "frame_step: needs 16 codebooks, a Talker head and 15 predictor heads");
    if (B < 1 || B > cc.max_slots || B > cc.max_batch || 2 * B > cc.max_tokens || cc.max_ctx < 16)
        return fail(cp, TTS_BB_E_INVALID, "frame_step: B=%d does not fit the Code Predictor handle", B);
    if (!codes || !slots || !kv_lens) return fail(talker, TTS_BB_E_INVALID, "frame_step: NULL codes, slots or kv_lens");
    if (B > cp->fr_cap) {
        cudaStreamSynchronize(cp->st);
        for (void* p : {(void*)cp->fr_hid, (void*)cp->fr_code0, (void*)cp->fr_emb, (void*)cp->fr_ids, (void*)cp->fr_steps})
            if (p) {
                cudaFree(p);
                cp->allocs.erase(std::remove(cp->allocs.begin(), cp->allocs.end(), p), cp->allocs.end());
            }
        cp->fr_hid = nullptr;
        cp->fr_code0 = nullptr;
        cp->fr_emb = nullptr;
        cp->fr_ids = nullptr;
        cp->fr_steps = nullptr;
        cp->fr_cap = 0;
        cudaError_t e = dalloc(cp, &cp->fr_hid, (size_t)B * HID);
        if (e == cudaSuccess) e = dalloc(cp, &cp->fr_code0, (size_t)B);
        if (e == cudaSuccess) e = dalloc(cp, &cp->fr_emb, (size_t)B * 2 * HID);
        if (e == cudaSuccess) e = dalloc(cp, &cp->fr_ids, (size_t)B * 32);
        if (e == cudaSuccess) e = dalloc(cp, &cp->fr_steps, (size_t)15 * B * 16);
        if (e != cudaSuccess) return cuda_fail(cp, e, "frame-loop scratch");
        cp->fr_cap = B;
    }
    std::vector<int32_t> cps(B), len2(B, 2), lens(B);
    for (int b = 0; b < B; ++b) {
        cps[b] = b;
        if (cp->slot_len[b]) tts_bb_release(cp, b);  // a frame left behind by a failed call
    }
    // Talker: this frame's 16 codes at the next position -> code 0 and the hidden state
    tts_bb_opts to{};
    to.hidden_out = cp->fr_hid;
    tts_bb_status st = tts_bb_decode_step(talker, B, slots, kv_lens, codes, 0, talker_logits, cp->fr_code0, &to);
    if (st != TTS_BB_OK) return st;
    {
        Launch L(cp, K_FRAME);
        k_frame_prep<<<B, 256, 0, cp->st>>>(cp->fr_hid, talker->final_norm, tc.rms_eps, cp->fr_code0, cp->fr_emb,
                                            cp->fr_ids, cp->fr_steps, B);
        L += 1;
    }
    // Code Predictor: 2-token prefill (head 0 -> code 1), then calls 1..14 (head j -> code j + 1)
    tts_bb_opts po{};
    po.embeds = cp->fr_emb;
    po.argmax_stride = 16;
    st = tts_bb_prefill(cp, B, 2, cps.data(), len2.data(), cp->fr_ids, 0, nullptr, cp->fr_steps + (size_t)1 * B * 16 + 1,
                        &po);
    for (int j = 1; j < 15 && st == TTS_BB_OK; ++j) {
        for (int b = 0; b < B; ++b) lens[b] = j + 1;
        tts_bb_opts dopt{};
        dopt.argmax_stride = 16;
        int32_t* dst = j < 14 ? cp->fr_steps + (size_t)(j + 1) * B * 16 + (j + 1) : codes + 15;
        st = tts_bb_decode_step(cp, B, cps.data(), lens.data(), cp->fr_steps + (size_t)j * B * 16, j, nullptr, dst,
                                &dopt);
    }
    if (st == TTS_BB_OK) {
        Launch L(cp, K_FRAME);
        k_frame_collect<<<B, 32, 0, cp->st>>>(cp->fr_code0, cp->fr_steps, codes, B);
        L += 1;
        st = finish(cp);
    }
    for (int b = 0; b < B; ++b) tts_bb_release(cp, b);
    return st;
}

TTS_API tts_bb_status tts_bb_maskgit_update(tts_bb* h, int n_items, int T, const float* logits, int S_logits,
                                            int cond_pos0, int uncond_pos0, int32_t* ids, int S_ids,
                                            int cond_ids_pos0, int uncond_ids_pos0, int n_unmask, float cfg_scale,
                                            float layer_penalty) {
    if (!h) return TTS_BB_E_INVALID;
    const tts_bb_config& c = h->cfg;
    if (c.n_heads <= 0 || c.head_rows < 2 || c.head_rows > mg_max_vocab())
        return fail(h, TTS_BB_E_INVALID, "maskgit_update needs audio heads of 2..%d ids", mg_max_vocab());
    if (n_items < 1 || T < 1 || n_unmask < 0 || !logits || !ids)
        return fail(h, TTS_BB_E_INVALID, "maskgit_update: bad sizes or NULL buffers");
    if (cond_pos0 < 0 || uncond_pos0 < 0 || (long long)cond_pos0 + T > S_logits || (long long)uncond_pos0 + T > S_logits)
        return fail(h, TTS_BB_E_INVALID, "maskgit_update: logits windows outside S_logits=%d", S_logits);
    if (cond_ids_pos0 < 0 || uncond_ids_pos0 < 0 || (long long)cond_ids_pos0 + T > S_ids ||
        (long long)uncond_ids_pos0 + T > S_ids)
        return fail(h, TTS_BB_E_INVALID, "maskgit_update: id windows outside S_ids=%d", S_ids);
    const size_t cells = (size_t)n_items * c.n_heads * T;
    if (cells > (size_t)INT32_MAX / 2) return fail(h, TTS_BB_E_INVALID, "maskgit_update: too many cells");
    if (cells > h->mg_cells) {
        cudaStreamSynchronize(h->st);
        for (void* p : {(void*)h->mg_keys, (void*)h->mg_pred})
            if (p) {
                cudaFree(p);
                h->allocs.erase(std::remove(h->allocs.begin(), h->allocs.end(), p), h->allocs.end());
            }
        h->mg_keys = nullptr;
        h->mg_pred = nullptr;
        h->mg_cells = 0;
        cudaError_t e = dalloc(h, &h->mg_keys, cells);
        if (e == cudaSuccess) e = dalloc(h, &h->mg_pred, cells);
        if (e != cudaSuccess) return cuda_fail(h, e, "MaskGIT update scratch");
        h->mg_cells = cells;
    }
    {
        Launch L(h, K_MG_UPDATE, (double)cells * 2.0 * c.head_rows * 4.0);
        L += launch_maskgit_update(logits, n_items, c.n_heads, T, c.head_rows, S_logits, cond_pos0, uncond_pos0, ids,
                                   S_ids, cond_ids_pos0, uncond_ids_pos0, c.head_rows - 1, cfg_scale, layer_penalty,
                                   n_unmask, h->mg_keys, h->mg_pred, h->st);
    }
    return finish(h);
}

TTS_API tts_bb_status tts_bb_maskgit_schedule(int num_step, int n_total, double t_shift, int32_t* counts) {
    if (num_step < 1 || n_total < 0 || !(t_shift > 0.0) || !counts) return TTS_BB_E_INVALID;
    auto tp = [&](int i) {
        const double t = (double)i / (double)num_step;
        return t_shift * t / (t_shift * t + (1.0 - t));
    };
    for (int i = 0; i < num_step; ++i) counts[i] = (int32_t)std::ceil((double)n_total * (tp(i + 1) - tp(i)));
    return TTS_BB_OK;
}

TTS_API tts_bb_status tts_bb_debug_kv_read(tts_bb* h, int layer, int slot, int pos0, int n, void* k_out, void* v_out) {
    if (!h) return TTS_BB_E_INVALID;
    if (h->cfg.max_slots <= 0 || layer < 0 || layer >= h->cfg.n_layers || slot < 0 || slot >= h->cfg.max_slots ||
        pos0 < 0 || n < 0 || (long long)pos0 + n > h->slot_len[slot] || !k_out || !v_out)
        return fail(h, TTS_BB_E_INVALID, "debug_kv_read: bad arguments");
    if (n == 0) return TTS_BB_OK;
    {
        Launch L(h, K_KVCOPY);
        k_kv_copy<<<n, 256, 0, h->st>>>(h->pool + (size_t)layer * h->layer_elems, h->d_page_table, slot, h->mbps, pos0, n,
                                        reinterpret_cast<bf16*>(k_out), reinterpret_cast<bf16*>(v_out), 0, h->kv_blocks,
                                        h->err);
        L += 1;
    }
    return finish(h);
}

TTS_API tts_bb_status tts_bb_debug_kv_write(tts_bb* h, int layer, int slot, int pos0, int n, const void* k,
                                           const void* v) {
    if (!h) return TTS_BB_E_INVALID;
    if (h->cfg.max_slots <= 0 || layer < 0 || layer >= h->cfg.n_layers || slot < 0 || slot >= h->cfg.max_slots ||
        pos0 < 0 || n < 0 || pos0 > h->slot_len[slot] || (long long)pos0 + n > h->cfg.max_ctx || !k || !v)
        return fail(h, TTS_BB_E_INVALID, "debug_kv_write: bad arguments");
    if (n == 0) return TTS_BB_OK;
    const int new_len = std::max(h->slot_len[slot], pos0 + n);
    SetupArgs& a = *h->setup;
    a.B = 0;
    a.clear_amax = 0;
    int32_t s1[1] = {slot};
    int nl[1] = {new_len};
    tts_bb_status s = grow_slots(h, 1, s1, nl, a);
    if (s != TTS_BB_OK) return s;
    h->slot_len[slot] = new_len;
    launch_setup(h, a);
    {
        Launch L(h, K_KVCOPY);
        k_kv_copy<<<n, 256, 0, h->st>>>(h->pool + (size_t)layer * h->layer_elems, h->d_page_table, slot, h->mbps, pos0, n,
                                        const_cast<bf16*>(reinterpret_cast<const bf16*>(k)),
                                        const_cast<bf16*>(reinterpret_cast<const bf16*>(v)), 1, h->kv_blocks, h->err);
        L += 1;
    }
    return finish(h);
}

TTS_API tts_bb_status tts_bb_profile(tts_bb* h, int on) {
    if (!h) return TTS_BB_E_INVALID;
    cudaStreamSynchronize(h->st);
    for (auto& r : h->prof) {
        h->ev_pool.push_back(r.a);
        h->ev_pool.push_back(r.b);
    }
    h->prof.clear();
    h->phase_us.clear();
    h->phase_max_us.clear();
    h->phase_n = 0;
    h->unit_split[0] = h->unit_split[1] = 0;
    h->unit_split_n[0] = h->unit_split_n[1] = 0;
    h->ring_wait[0] = h->ring_wait[1] = 0;
    h->ring_wait_n = 0;
    h->prof_on = on != 0;
    return TTS_BB_OK;
}

TTS_API const char* tts_bb_profile_report(tts_bb* h) {
    if (!h) return "{}";
    cudaStreamSynchronize(h->st);
    double ms[K_NKINDS] = {}, bytes[K_NKINDS] = {}, flops[K_NKINDS] = {};
    long n[K_NKINDS] = {};
    for (const auto& r : h->prof) {
        float t = 0.f;
        if (cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess) ms[r.kind] += t;
        bytes[r.kind] += r.bytes;
        flops[r.kind] += r.flops;
        n[r.kind]++;
    }
    std::string j = "{\"kernels\": [";
    bool first = true;
    for (int k = 0; k < K_NKINDS; ++k) {
        if (!n[k]) continue;
        char buf[320];
        snprintf(buf, sizeof buf, "%s{\"kind\": \"%s\", \"launches\": %ld, \"ms\": %.6f, \"bytes\": %.0f, \"flops\": %.0f}",
                 first ? "" : ", ", kind_name[k], n[k], ms[k], bytes[k], flops[k]);
        j += buf;
        first = false;
    }
    j += "]";
    if (h->phase_n > 0) {
        static const char* names[10] = {"wait_h_norm", "qkv", "attention_units", "wait_partials_merge", "o_proj",
                                        "wait_h_norm2", "gate_up_swiglu", "wait_m", "down", "to_next_layer"};
        j += ", \"persistent_phases_us_per_layer\": {";
        for (int i = 0; i < 10; ++i) {
            char buf[160];
            snprintf(buf, sizeof buf, "%s\"%s\": {\"mean\": %.3f, \"max\": %.3f}", i ? ", " : "", names[i],
                     h->phase_us[i] / h->phase_n, h->phase_max_us[i] / h->phase_n);
            j += buf;
        }
        j += "}";
        if (h->unit_split_n[0] + h->unit_split_n[1]) {
            char buf[200];
            snprintf(buf, sizeof buf, ", \"attention_phase_us\": {\"ctas_without_unit\": %.3f, \"ctas_with_units\": %.3f, \"share_with\": %.3f}",
                     h->unit_split_n[0] ? h->unit_split[0] / h->unit_split_n[0] : 0.0,
                     h->unit_split_n[1] ? h->unit_split[1] / h->unit_split_n[1] : 0.0,
                     (double)h->unit_split_n[1] / (h->unit_split_n[0] + h->unit_split_n[1]));
            j += buf;
        }
        if (h->ring_wait_n) {
            char buf[160];
            snprintf(buf, sizeof buf, ", \"ring_wait_us\": {\"gate_up\": %.3f, \"down\": %.3f}",
                     h->ring_wait[0] / h->ring_wait_n, h->ring_wait[1] / h->ring_wait_n);
            j += buf;
        }
    }
    j += "}";
    h->prof_json = j;
    return h->prof_json.c_str();
}
