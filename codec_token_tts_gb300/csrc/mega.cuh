// Persistent small-batch decode step (k_decode_mega.cu): argument block and launch API.
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
    float* m;                  // [B][ffn] SwiGLU output (fp32)
    float* part;               // [B][16][nblk_max][PART_STRIDE]
    int nblk_max;
    unsigned long long* amax;  // [B]
    unsigned long long* bar;   // grid barrier counter (monotonic)
    unsigned long long bar_base;
    int* abort_flag;
    int* err;
    const float* cos_t;
    const float* sin_t;
    float eps;
    int B, n_layers, ffn;
    unsigned long long* trace; // optional: [grid][n_layers][12] globaltimer stamps of CTA phases
};

// Launch one decode step on `grid` CTAs (cooperative: all co-resident or an error).
cudaError_t launch_decode_mega(const MegaArgs& a, int grid, cudaStream_t st);
// Grid barriers one launch performs; the host advances MegaArgs::bar_base by this times grid.
int mega_barriers(int n_layers, bool head, bool argmax);
// Largest cooperative grid (one CTA per SM), 0 if the kernel cannot run here.
int mega_max_grid();

}  // namespace ttsbb
