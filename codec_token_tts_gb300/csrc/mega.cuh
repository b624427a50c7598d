// Persistent small-batch decode step (k_decode_ll.cu): argument block and launch API.
#pragma once
#include "common.cuh"

namespace ttsbb {

namespace mk {
constexpr int MAXB = 2;    // largest batch the persistent step runs (fp32 activations in shared memory)
constexpr int MAXL = 32;   // layers
}  // namespace mk

// Attention partial record per (sequence, head, cache block): 128 outputs,
// running max, running sum, padding to keep records 16-byte aligned.
constexpr int PART_STRIDE = HD + 4;

struct MegaLayer {
    const bf16 *in_norm, *wqkv, *qn, *kn, *wo, *post_norm, *wgu, *wd;
};

// Everything one launch needs, passed by value (about 2.5 KB).
struct MegaArgs {
    MegaLayer L[mk::MAXL];
    TableSet tabs;
    const int32_t* ids;        // [B][n_codebooks] or null
    const bf16* embeds;        // [B][HID] or null
    const bf16* final_norm;
    const bf16* head;          // [head_rows][HID] or null
    int head_rows;
    float* logits;             // [B][head_rows] or null
    int32_t* argmax_out;       // or null
    int argmax_stride;
    bf16* pool;
    size_t layer_elems;
    const int32_t* page_table;
    int mbps;
    int slot[mk::MAXB];
    int pos[mk::MAXB];
    int n_upd;
    int upd_idx[mk::MAXB];
    int upd_val[mk::MAXB];
    float* h;                  // [B][HID] residual (fp32)
    float* qkv;                // [B][QKV]
    int nblk_max;
    unsigned long long* amax;  // [B]
    int* abort_flag;
    int* err;
    const float* cos_t;
    const float* sin_t;
    float eps;
    int B, n_layers, ffn;
    unsigned long long* trace; // optional: [grid][n_layers][TRACE_STRIDE] globaltimer stamps of CTA phases
    // flag-in-data exchange (k_decode_ll.cu)
    unsigned long long* xbuf;  // exchange words (value | epoch << 32), zero-initialised
    uint32_t ep_base;          // first epoch of this launch (grows by ll_epochs_per_launch)
    int last_phys[mk::MAXB];   // physical block holding each sequence's new token
    unsigned int* done;        // CTAs finished with the head (last one publishes the argmax)
    unsigned long long timeout_ns;  // bound of every wait (exchange polls, ring slots)
    int debug_stall;           // test hook: CTA 0 withholds one exchange, so every wait runs out
    int l2_prefetch;           // bit 0: next-layer weight rows into L2 (producer); bit 1: next-layer K/V of the attention units
};

// Launch one decode step on `grid` CTAs (cooperative: all co-resident or an error).
cudaError_t launch_decode_ll(const MegaArgs& a, int grid, cudaStream_t st);
int ll_max_grid();
constexpr int LL_MIN_GRID = 96;   // smallest grid whose per-CTA op slices fit the weight ring
constexpr int TRACE_STRIDE = 64;  // profiling stamps per (CTA, layer)
// Replicas of the h and SwiGLU exchange vectors and of the attention partials (readers spread over
// them, writers store every copy). Measured at batch 1 on 128 CTAs (tokens/s, h/SwiGLU : partials):
// 1:1 2001, 2:2 2072, 4:4 2091, 4:2 2092, 8:8 2027, 16:8 2036, 16:16 1994.
constexpr int LL_XR = 4;
constexpr int LL_XRP = 4;
uint32_t ll_epochs_per_launch(int n_layers);
// Exchange words the flag-in-data step needs for mbps cache blocks per sequence.
inline size_t ll_xbuf_words(int mbps) {
    return 2ull * mk::MAXB * (LL_XR * HID + QKV + LL_XR * 3072) + 2ull * LL_XRP * mk::MAXB * NQ * (size_t)mbps * PART_STRIDE;
}

}  // namespace ttsbb
