/*
 * tts_bb.h — C ABI of the GB300 (sm_103a) engine for the forward step of the
 * Qwen3-0.6B-shaped backbone that drives codec-token speech generation.
 *
 * The backbone (28 layers, hidden 1024, 16 query / 8 KV heads of 128, SwiGLU
 * 3072, RMSNorm eps 1e-6, q/k RMSNorm before half-rotate RoPE theta 1e6) is the
 * one described on "omnivoice-cpp docs/ARCHITECTURE.md" (GGUF layout;
 * Component architecture, Qwen3 specifics) and "Qwen3-TTS ncnn port"
 * (Tencent/ncnn discussion 6877; model structure, Talker and Code Predictor;
 * single-token SDPA and host attention; mRoPE conclusion).
 *
 * Conventions follow the public C99 ABI of omnivoice-cpp (Public API and ABI
 * guarantee): an opaque handle, a default-initialiser for the config struct,
 * a negative status enum, caller-owned outputs, a version string. The header
 * is plain C99; the library exports only tts_bb_* symbols.
 *
 * Pointers. Unless a parameter says otherwise:
 *   - "device" arrays are CUDA device pointers (e.g. torch CUDA tensors) on
 *     the device that was current at tts_bb_create; they must stay valid
 *     until the work enqueued on the handle's stream has finished;
 *   - "host" arrays are ordinary CPU memory read before the call returns.
 * All compute calls are asynchronous on the handle's stream. Host-side
 * argument errors return before anything is enqueued and change no state.
 * Device-side errors (an out-of-range id) are latched in a device error word:
 * with config.sync_errors = 1 every call ends by reading it (one stream
 * synchronisation); with 0 the caller reads it with tts_bb_sync().
 * A handle is not thread-safe: one host thread at a time.
 */
#ifndef TTS_BB_H
#define TTS_BB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TTS_BB_VERSION_MAJOR 0
#define TTS_BB_VERSION_MINOR 1
#define TTS_BB_VERSION_PATCH 0

#define TTS_BB_MAX_CODEBOOKS 16
#define TTS_BB_MAX_HEADS 16
#define TTS_BB_KV_BLOCK 64

typedef struct tts_bb tts_bb; /* opaque engine handle */

typedef enum {
    TTS_BB_OK = 0,
    TTS_BB_E_INVALID = -1,         /* bad argument; nothing was enqueued */
    TTS_BB_E_UNSUPPORTED = -2,     /* valid C, a shape the kernels are not built for */
    TTS_BB_E_CUDA = -3,            /* a CUDA runtime call failed */
    TTS_BB_E_OOM = -4,             /* device memory or KV blocks exhausted */
    TTS_BB_E_DEVICE_TIMEOUT = -5,  /* a bounded device-side wait ran out */
    TTS_BB_E_BAD_ID = -6,          /* a token id was out of its table (it was skipped) */
    TTS_BB_E_NOT_IMPLEMENTED = -7
} tts_bb_status;

/* Backbone and engine shape. Field names follow the Code Predictor config of
 * "rightkit-qts 0.2.0" (Mode API: hidden_size, n_layers, heads, kv heads,
 * intermediate_size, head_dim, rms_norm_eps, rope_theta, vocab_size). */
typedef struct {
    int n_layers;          /* 28 Talker / OmniVoice, 5 Code Predictor */
    int hidden;            /* 1024 (the only value the kernels support) */
    int n_q_heads;         /* 16 */
    int n_kv_heads;        /* 8 */
    int head_dim;          /* 128 */
    int ffn;               /* 3072 */
    float rms_eps;         /* 1e-6 */
    float rope_theta;      /* 1e6 */
    /* Input embedding: the codebook tables E_0..E_{n_codebooks-1} are summed
     * (Qwen3-TTS ncnn port, model structure: the 16 embeddings of a frame are
     * added to form the next Talker input). */
    int n_codebooks;
    int codebook_rows[TTS_BB_MAX_CODEBOOKS];
    /* OmniVoice hybrid input (omnivoice-cpp, Component architecture): a text
     * table of text_vocab rows and an audio table of audio_codebooks *
     * audio_vocab rows. 0 = absent. */
    int text_vocab;
    int audio_codebooks;
    int audio_vocab;
    /* Output heads: n_heads bf16 matrices of [head_rows][hidden] (Talker 1 x
     * 3072, Code Predictor 15 x 2048). For OmniVoice set n_heads = audio_codebooks
     * and head_rows = audio_vocab: one [n_heads*head_rows][hidden] matrix
     * (audio_heads) is passed in head[0]. 0 heads = hidden-state only. */
    int n_heads;
    int head_rows;
    /* KV cache: paged, TTS_BB_KV_BLOCK tokens per block. */
    int max_slots;         /* concurrent sequences (stream slots), at most 2^20 */
    int max_ctx;           /* longest sequence, tokens, at most 2^20 */
    int kv_blocks;         /* physical blocks; 0 = max_slots * ceil(max_ctx / 64) */
    int max_batch;         /* largest B of one call (scratch sizing) */
    int max_tokens;        /* largest B*S of one prefill / MaskGIT call, at most 2^20 */
    int sync_errors;       /* 1 = each call synchronises to report device errors */
} tts_bb_config;

/* Per-layer tensor roles (PyTorch (out, in) row-major, bf16). */
enum {
    TTS_BB_W_IN_NORM = 0,  /* [hidden]           input_layernorm */
    TTS_BB_W_Q,            /* [heads*128][hidden] q_proj */
    TTS_BB_W_K,            /* [kv*128][hidden]   k_proj */
    TTS_BB_W_V,            /* [kv*128][hidden]   v_proj */
    TTS_BB_W_Q_NORM,       /* [128]              q_norm */
    TTS_BB_W_K_NORM,       /* [128]              k_norm */
    TTS_BB_W_O,            /* [hidden][heads*128] o_proj */
    TTS_BB_W_POST_NORM,    /* [hidden]           post_attention_layernorm */
    TTS_BB_W_GATE,         /* [ffn][hidden]      gate_proj */
    TTS_BB_W_UP,           /* [ffn][hidden]      up_proj */
    TTS_BB_W_DOWN,         /* [hidden][ffn]      down_proj */
    TTS_BB_LAYER_TENSORS
};

/* Weight pointers, bf16 bit patterns. Host or device memory (anything
 * cudaMemcpy with cudaMemcpyDefault accepts). tts_bb_create copies them into
 * engine-owned device memory (fusing q/k/v and interleaving gate/up), so the
 * caller may free its copies once tts_bb_create has returned. */
typedef struct {
    const void* codebook[TTS_BB_MAX_CODEBOOKS]; /* [codebook_rows[k]][hidden] */
    const void* text_table;                     /* [text_vocab][hidden] or NULL */
    const void* audio_table;                    /* [audio_codebooks*audio_vocab][hidden] or NULL */
    const void* const* layer;                   /* n_layers * TTS_BB_LAYER_TENSORS pointers */
    const void* final_norm;                     /* [hidden] */
    const void* head[TTS_BB_MAX_HEADS];         /* [head_rows][hidden] each */
} tts_bb_weights;

/* Optional per-call inputs and outputs. NULL options = all defaults. */
typedef struct {
    /* device bf16 [tokens][hidden], added to the codebook sum (the Code
     * Predictor's Talker-hidden row, or a plain embedding input). */
    const void* embeds;
    /* device fp32 [tokens][hidden]: the residual after the last layer, before
     * the final norm. */
    float* hidden_out;
    /* element stride between consecutive rows of argmax_out (0 = 1): lets a
     * Talker / Code-Predictor loop write codes straight into the next frame's
     * id matrix. */
    int argmax_stride;
} tts_bb_opts;

/* Fill *cfg with the Qwen3-TTS Talker shape: 28 layers, 16 codebooks
 * (E_0 3072 rows, E_1..E_15 2048 rows), one 3072-row head, 64 slots, 4096 ctx. */
void tts_bb_default_config(tts_bb_config* cfg);

/* Create an engine on the current CUDA device; `stream` is a cudaStream_t
 * (NULL = the legacy default stream) on which every call of the handle runs.
 * Allocates the weights, the KV block pool and scratch. Returns
 * TTS_BB_E_INVALID for a bad config, TTS_BB_E_UNSUPPORTED for a shape the
 * kernels are not built for (or max_slots, max_ctx, max_tokens above 2^20),
 * TTS_BB_E_OOM when device or host memory runs out. No exception leaves the
 * call. */
tts_bb_status tts_bb_create(const tts_bb_config* cfg, const tts_bb_weights* w,
                            void* stream, tts_bb** out);

/* Wait for the handle's work and free everything it owns. NULL is a no-op. */
void tts_bb_free(tts_bb* h);

/* Causal prefill (Qwen3-TTS ncnn port: prompt prefill fills the per-layer
 * KV cache). Sequence b appends lens[b] tokens (1..S) to slot slots[b],
 * starting at the slot's current length, so a prefill can extend a cache.
 *   B, S      batch and padded length; B*S <= max_tokens, B <= max_batch
 *   slots     host int32 [B], distinct, in [0, max_slots)
 *   lens      host int32 [B], 1..S
 *   ids       device int32 [B][S][n_codebooks]; -1 = no token from that
 *             codebook at that position; NULL = embeddings only
 *   head_idx  head applied to the last valid position of each row (-1 = none)
 *   logits_out device fp32 [B][head_rows] or NULL
 *   argmax_out device int32 [B] (stride opts->argmax_stride) or NULL; the
 *             lowest index wins a tie
 *   opts->embeds     [B][S][hidden]; opts->hidden_out [B][S][hidden]
 * An out-of-table id is skipped and reported as TTS_BB_E_BAD_ID. */
tts_bb_status tts_bb_prefill(tts_bb* h, int B, int S, const int32_t* slots, const int32_t* lens,
                             const int32_t* ids, int head_idx, float* logits_out,
                             int32_t* argmax_out, const tts_bb_opts* opts);

/* One decode step, query length 1, for B sequences (Qwen3-TTS ncnn port,
 * single-token SDPA and host attention: RoPE, KV append and GQA attention over
 * the cache for a query of length 1).
 *   slots    host int32 [B], distinct
 *   kv_lens  host int32 [B]: tokens already cached in each slot; must equal
 *            the engine's length for the slot (TTS_BB_E_INVALID otherwise).
 *            The new token is written at position kv_lens[b] and attention
 *            covers kv_lens[b] + 1 tokens.
 *   ids      device int32 [B][n_codebooks] (-1 = absent) or NULL
 *   logits_out / argmax_out as in tts_bb_prefill, one row per sequence
 *   opts->embeds [B][hidden]; opts->hidden_out [B][hidden] */
tts_bb_status tts_bb_decode_step(tts_bb* h, int B, const int32_t* slots, const int32_t* kv_lens,
                                 const int32_t* ids, int head_idx, float* logits_out,
                                 int32_t* argmax_out, const tts_bb_opts* opts);

/* tts_bb_decode_step with HOST buffers, for a caller that keeps its ids and
 * reads each step's tokens on the host (a streaming loop): copies ids (host
 * int32 [B][n_codebooks], pinned for an asynchronous copy) to the device, runs
 * the step, copies argmax_out (host int32 [B] or NULL) and logits_out (host
 * fp32 [B][head_rows] or NULL) back, and returns once they have landed (one
 * stream synchronisation, which also reads the device error word). Other
 * arguments and errors as in tts_bb_decode_step. Device staging for max_batch
 * rows is allocated on the first call. */
tts_bb_status tts_bb_decode_step_host(tts_bb* h, int B, const int32_t* slots, const int32_t* kv_lens,
                                      const int32_t* ids, int head_idx, int32_t* argmax_out, float* logits_out);

/* One full bidirectional MaskGIT pass without a KV cache (omnivoice-cpp,
 * MaskGIT decoder: every step is a full prefill with non-causal attention;
 * Component architecture: hybrid text/audio embedding and audio heads;
 * Inner-loop optimisations: logits only over the audio window).
 *   ids         device int32 [B][audio_codebooks][S] (text id on every row at
 *               text positions, audio codes 0..audio_vocab-1 at audio positions)
 *   audio_mask  device uint8 [B][S], 1 = audio position
 *   key_lens    host int32 [B] (keys >= key_lens[b] are padding) or NULL = S
 *   audio_start first position of the audio window, 0 <= audio_start < S
 *   logits_out  device fp32 [B][n_heads][S - audio_start][head_rows]:
 *               logits[b][k][s][v] = final_norm(x[b][audio_start+s]) . W[k*head_rows + v]
 *   opts->hidden_out [B][S][hidden]
 * Requires a handle with text and audio tables; B*S <= max_tokens. */
tts_bb_status tts_bb_maskgit_pass(tts_bb* h, int B, int S, const int32_t* ids,
                                  const uint8_t* audio_mask, const int32_t* key_lens,
                                  int audio_start, float* logits_out, const tts_bb_opts* opts);

/* One frame of the Talker -> Code Predictor loop (Qwen3-TTS ncnn port, model
 * structure: the Talker predicts codebook 0 of each frame, the Code Predictor
 * the other 15 in 15 autoregressive steps, and the frame's 16 embeddings
 * summed are the Talker's next input), for B streams at once, greedy:
 *   1. the Talker decodes `codes` (this frame's input, [B][16], -1 = absent)
 *      at position kv_lens[b] of slot slots[b] (as tts_bb_decode_step), head 0
 *      -> code 0, and its last-layer hidden state;
 *   2. the Code Predictor runs a 2-token prefill in its slots 0..B-1: position
 *      0 = the Talker hidden state after the Talker's final norm (bf16),
 *      position 1 = E_0[code 0]; head 0 -> code 1; then calls j = 1..14 feed
 *      E_j[code j] at position j + 1, head j -> code j + 1; its slots are
 *      released afterwards;
 *   3. codes[b] = the frame's 16 codes (the next frame's input).
 *   talker, cp     handles on the same stream; cp has 16 codebooks (the
 *                  Talker's tables), >= 15 heads, B <= max_slots, max_batch,
 *                  2 B <= max_tokens, max_ctx >= 16
 *   slots, kv_lens host int32 [B] for the Talker, as in tts_bb_decode_step
 *   codes          device int32 [B][16], read then overwritten
 *   talker_logits  device fp32 [B][Talker head_rows] or NULL
 * Everything runs on the shared stream (about 2 + 16 launches and, for B > 2,
 * graph replays); scratch is allocated on the first call that needs more.
 * Errors as in tts_bb_decode_step / tts_bb_prefill (status of the first call
 * that failed); TTS_BB_E_INVALID for handles that do not fit. */
tts_bb_status tts_bb_frame_step(tts_bb* talker, tts_bb* cp, int B, const int32_t* slots,
                                const int32_t* kv_lens, int32_t* codes, float* talker_logits);

/* Greedy token update of one MaskGIT refinement step on the device
 * (omnivoice-cpp, MaskGIT decoder, class and position temperatures 0). The
 * batch of a pass holds n_items conditional rows (0..n_items-1) followed by
 * their n_items unconditional rows (n_items..2 n_items-1). For every target
 * cell (item i, codebook k < n_heads, position t < T):
 *   z     = c + cfg_scale (c - u), float32, c the conditional and u the
 *           unconditional logits of the cell (one rounding per operation)
 *   pred  = argmax of z over the ids other than the mask id (head_rows - 1),
 *           lowest id on ties
 *   score = z[pred] - logsumexp(z over all head_rows ids) - k layer_penalty
 * Cells whose current id (conditional row) is not the mask id are kept. Of
 * the masked cells of each item, the min(n_unmask, masked) with the highest
 * score (ties: lowest k T + t) take pred, written to the conditional and the
 * unconditional rows.
 *   logits  device fp32 [2 n_items][n_heads][S_logits][head_rows] (the
 *           maskgit_pass output); the cell's logits sit at position
 *           cond_pos0 + t (conditional rows) and uncond_pos0 + t
 *           (unconditional rows)
 *   ids     device int32 [2 n_items][n_heads][S_ids], updated in place at
 *           positions cond_ids_pos0 + t and uncond_ids_pos0 + t
 *   cfg_scale 2.0 and layer_penalty 5.0 on the page.
 * Two kernel launches on the handle's stream; the scratch (12 bytes per cell)
 * is allocated on the first call that needs more. TTS_BB_E_INVALID for
 * windows outside their tensors, n_items < 1, T < 1, n_unmask < 0 or a
 * handle without audio heads (or with more than 1056 ids per head). */
tts_bb_status tts_bb_maskgit_update(tts_bb* h, int n_items, int T, const float* logits, int S_logits,
                                    int cond_pos0, int uncond_pos0, int32_t* ids, int S_ids,
                                    int cond_ids_pos0, int uncond_ids_pos0, int n_unmask,
                                    float cfg_scale, float layer_penalty);

/* Cells newly unmasked at each of num_step MaskGIT steps, host only:
 * counts[i] = ceil(n_total (t'[i+1] - t'[i])) with t[i] = i / num_step
 * shifted by t' = s t / (s t + (1 - t)), s = t_shift (0.1 on the page, whose
 * time-step function is not printed: this shift is a reading). The counts sum
 * to at least n_total. TTS_BB_E_INVALID for num_step < 1, n_total < 0,
 * t_shift <= 0 or a NULL counts. */
tts_bb_status tts_bb_maskgit_schedule(int num_step, int n_total, double t_shift, int32_t* counts);

/* RVQ codec decode (omnivoice-cpp, Audio tokenizer pipeline, Decode, and RVQ
 * codec): codes of K codebooks -> out_dim frame features,
 *   out[b][t] = sum_k ( embed_k[codes[b][k][t]] . proj_w_k^T + proj_b_k )
 * with embed_k [codebook_size][dim] (codebook.embed), proj_w_k [out_dim][dim]
 * (project_out.weight) and proj_b_k [out_dim] (project_out.bias), all device
 * bf16 pointers, K of each; the OmniVoice codec has K = 8, 1024 x 64 tables and
 * out_dim 1024. tts_bb_rvq_create copies them (the caller may free its copies)
 * and returns TTS_BB_E_INVALID for NULL pointers or sizes outside
 * 1 <= K <= 64, dim a multiple of 8 with K * dim a multiple of 64,
 * TTS_BB_E_OOM, TTS_BB_E_UNSUPPORTED without tcgen05 tensor maps. */
typedef struct tts_bb_rvq tts_bb_rvq;
tts_bb_status tts_bb_rvq_create(int n_codebooks, int codebook_size, int dim, int out_dim,
                                const void* const* embed, const void* const* proj_w,
                                const void* const* proj_b, void* stream, tts_bb_rvq** out);
/* codes device int32 [B][K][T]; out device fp32 [B][T][out_dim]. Asynchronous
 * on the handle's stream (a gather kernel and one GEMM); a code outside
 * 0..codebook_size-1 contributes nothing and is reported by tts_bb_rvq_sync as
 * TTS_BB_E_BAD_ID. Scratch (K * dim bf16 per frame) grows on the first call
 * that needs more. */
tts_bb_status tts_bb_rvq_decode(tts_bb_rvq* r, int B, int T, const int32_t* codes, float* out);
/* Wait for the handle's work; returns (and clears) a latched device error. */
tts_bb_status tts_bb_rvq_sync(tts_bb_rvq* r);
/* Wait and free. NULL is a no-op. */
void tts_bb_rvq_free(tts_bb_rvq* r);

/* Qwen3-TTS codec quantizer lookup (Qwen3-TTS ncnn port, Codec Decoder split,
 * steps 1-4): the frame's 16 codes -> the 512-channel float hidden that the
 * codec body reads,
 *   out[b][o][t] = P_sem[o] . C_0[codes[b][0][t]]
 *                + P_ac[o] . sum_{k=1..K-1} C_k[codes[b][k][t]]
 * i.e. the first (semantic) codebook through its own projection and the
 * other K-1 (acoustic) codebooks summed through the second projection.
 *   codebooks     K device bf16 pointers, each [codebook_size][dim]
 *   proj_semantic device bf16 [out_dim][dim]; proj_acoustic the same
 * (the page: 16 codebooks of 2048 entries, out_dim 512; it does not print the
 * codebook width, so dim is a parameter; the projections are bias-free).
 * tts_bb_quantizer_create copies them (the caller may free its copies) and
 * returns TTS_BB_E_INVALID for NULL pointers or sizes outside 2 <= K <= 32,
 * dim a multiple of 64 in 64..1024, 1 <= out_dim <= 8192; TTS_BB_E_OOM. */
typedef struct tts_bb_quantizer tts_bb_quantizer;
tts_bb_status tts_bb_quantizer_create(int n_codebooks, int codebook_size, int dim, int out_dim,
                                      const void* const* codebooks, const void* proj_semantic,
                                      const void* proj_acoustic, void* stream, tts_bb_quantizer** out);
/* codes device int32 [B][K][T]; out device fp32 [B][out_dim][T] (channel-major,
 * the [1, 512, T] layout the page feeds to the codec body). Asynchronous on the
 * handle's stream (a gather kernel and one GEMM); the acoustic sum is carried
 * as bf16 high + low parts, so the result keeps fp32-level accuracy over the
 * bf16 tables. A code outside 0..codebook_size-1 contributes nothing and is
 * reported by tts_bb_quantizer_sync as TTS_BB_E_BAD_ID. Scratch (3 * dim bf16
 * per frame, rounded up to 256) grows on the first call that needs more. */
tts_bb_status tts_bb_quantizer_decode(tts_bb_quantizer* q, int B, int T, const int32_t* codes, float* out);
/* Wait for the handle's work; returns (and clears) a latched device error. */
tts_bb_status tts_bb_quantizer_sync(tts_bb_quantizer* q);
/* Wait and free. NULL is a no-op. */
void tts_bb_quantizer_free(tts_bb_quantizer* q);

/* DAC decoder: frame features -> 24 kHz audio (omnivoice-cpp, Audio tokenizer
 * pipeline, Decode; DAC decoder block channels; Snake activation;
 * ConvTranspose1d): fc2 Linear 1024 -> 256, conv1 (256 -> 1024, k 7, pad 3),
 * five blocks with ratios r = 8, 5, 4, 2, 3 and channels 1024 -> 512 -> 256 ->
 * 128 -> 64 -> 32 (snake; ConvTranspose1d k 2r, stride r, padding ceil(r/2),
 * output_padding r % 2; three residual units with dilations 1, 3, 9: snake,
 * Conv1d k 7 pad 3d, snake, Conv1d k 1, add), snake, conv2 (32 -> 1, k 7,
 * pad 3). Snake: y = x + sin(alpha x)^2 / (alpha + 1e-9), alpha per channel.
 * Every convolution and the Linear have a bias. All weights are device fp32
 * in PyTorch layouts; tts_bb_dac_create copies them. */
typedef struct {
    const float* alpha;          /* [IC] snake before the upsampling convolution */
    const float* up_w;           /* [IC][OC][2r] ConvTranspose1d weight */
    const float* up_b;           /* [OC] */
    const float* res_alpha1[3];  /* [OC] */
    const float* res_w1[3];      /* [OC][OC][7] */
    const float* res_b1[3];      /* [OC] */
    const float* res_alpha2[3];  /* [OC] */
    const float* res_w2[3];      /* [OC][OC][1] */
    const float* res_b2[3];      /* [OC] */
} tts_bb_dac_block;
typedef struct {
    const float* fc2_w;          /* [256][1024] */
    const float* fc2_b;          /* [256] */
    const float* conv1_w;        /* [1024][256][7] */
    const float* conv1_b;        /* [1024] */
    tts_bb_dac_block block[5];
    const float* final_alpha;    /* [32] */
    const float* conv2_w;        /* [1][32][7] */
    const float* conv2_b;        /* [1] */
} tts_bb_dac_weights;
typedef struct tts_bb_dac tts_bb_dac;
/* TTS_BB_E_INVALID for a NULL pointer, TTS_BB_E_OOM when memory runs out. */
tts_bb_status tts_bb_dac_create(const tts_bb_dac_weights* w, void* stream, tts_bb_dac** out);
/* features device fp32 [B][T][1024] (the RVQ decode output); audio device fp32
 * [B][960 T]. Asynchronous on the handle's stream; three activation buffers of
 * 30720 T floats per item are allocated on the first call that needs more.
 * fc2, conv1 and every convolution of the five blocks run on the tensor cores
 * (39 launches) with fp32 operands split into bf16 high + low parts (three
 * products per pair, fp32 accumulation) and time-major activations; conv2 runs
 * in fp32 on the CUDA cores. Environment TTS_BB_DAC=fp32 at create: every
 * convolution in fp32 on the CUDA cores, channel-major (38 launches).
 * TTS_BB_E_INVALID for NULL buffers, B < 1 or B > 65535, T < 1, or B x 960 T
 * above 2^31 - 1 samples. */
tts_bb_status tts_bb_dac_decode(tts_bb_dac* d, int B, int T, const float* features, float* audio);
/* Wait for the handle's work; returns (and clears) a latched device error
 * (TTS_BB_E_DEVICE_TIMEOUT: a bounded wait of a tensor-core kernel ran out). */
tts_bb_status tts_bb_dac_sync(tts_bb_dac* d);
/* Wait and free. NULL is a no-op. */
void tts_bb_dac_free(tts_bb_dac* d);

/* Return the slot's KV blocks to the pool; its length becomes 0. */
tts_bb_status tts_bb_release(tts_bb* h, int slot);

/* Shorten a slot to `len` tokens (0 <= len <= current length); blocks past
 * the new end go back to the pool. Positions >= len are rewritten by the next
 * prefill or decode step. */
tts_bb_status tts_bb_truncate(tts_bb* h, int slot, int len);

/* Current cached length of a slot, or -1 for a bad handle or slot. */
int tts_bb_slot_len(const tts_bb* h, int slot);

/* Wait for the handle's stream and report (then clear) any latched device error. */
tts_bb_status tts_bb_sync(tts_bb* h);

/* Text of the last error on this handle (empty string if none). */
const char* tts_bb_last_error(const tts_bb* h);

/* "MAJOR.MINOR.PATCH (sm_103a)". */
const char* tts_bb_version(void);

/* Test hooks: read or write n tokens of one layer's cache of one slot,
 * positions pos0..pos0+n-1, through the page table.
 *   k, v  device bf16 [n][n_kv_heads][head_dim] (keys after q/k-norm and RoPE)
 * tts_bb_debug_kv_write extends the slot to pos0+n if it was shorter
 * (allocating blocks); pos0 must not exceed the current length. */
tts_bb_status tts_bb_debug_kv_read(tts_bb* h, int layer, int slot, int pos0, int n,
                                   void* k_out, void* v_out);
tts_bb_status tts_bb_debug_kv_write(tts_bb* h, int layer, int slot, int pos0, int n,
                                    const void* k, const void* v);

/* Test hooks for failure handling (no counterpart on the pages): they force
 * device-side waits to run out without faulting the GPU.
 *   what = TTS_BB_DEBUG_WAIT_LIMIT_NS: every wait of the persistent decode
 *          step (exchange polls, weight-ring slots) gives up after arg ns
 *          (default 2e9; arg in 1e6 .. 1e10, else TTS_BB_E_INVALID).
 *   what = TTS_BB_DEBUG_STALL_NEXT_STEP: the next persistent decode step
 *          (batch <= 2) withholds one CTA's exchange words, so every CTA's
 *          wait runs out; that step returns TTS_BB_E_DEVICE_TIMEOUT (its
 *          outputs are undefined) and the handle stays usable. arg unused.
 * Returns TTS_BB_E_INVALID for a null handle or an unknown `what`. The
 * environment variable TTS_BB_FAIL_ALLOC_AT=n makes the n-th device
 * allocation of a handle being created fail (creation returns TTS_BB_E_OOM). */
enum { TTS_BB_DEBUG_WAIT_LIMIT_NS = 1, TTS_BB_DEBUG_STALL_NEXT_STEP = 2 };
tts_bb_status tts_bb_debug_fault(tts_bb* h, int what, int64_t arg);

/* Number of kernel launches the handle has enqueued since creation (a
 * counter kept on the host; lets a caller count launches in a timed region). */
uint64_t tts_bb_launch_count(const tts_bb* h);

/* Per-kernel timing. tts_bb_profile(h, 1) clears the record and brackets
 * every later kernel launch of the handle with CUDA events on its stream;
 * tts_bb_profile(h, 0) stops. tts_bb_profile_report waits for the stream and
 * returns a JSON summary {"kernels": [{"kind", "launches", "ms", "bytes",
 * "flops"}]}: per kernel kind, the launches, their summed event time and
 * their algorithmic bytes and flops. The string stays valid until the next
 * report or tts_bb_free. The events add a little time between launches, so
 * time a clean run without profiling. */
tts_bb_status tts_bb_profile(tts_bb* h, int on);
const char* tts_bb_profile_report(tts_bb* h);

/* Decode attention that allocates nothing (the pages have no counterpart: it
 * exists for callers of this library that may not call cudaMalloc — a plug-in
 * whose host framework owns every device allocation, or a real-time audio
 * thread that must not block in the allocator).
 *
 * It runs the same GQA decode attention kernels as tts_bb_decode_step on the
 * caller's own buffers (split-K flash decode; for max_position < 32 one warp
 * per query and KV head, which writes no partials); the split partials go to
 * a fixed array in device memory that is part of the library (TTS_BB_STATIC_ATTN_MAX_B x 16 heads x
 * TTS_BB_STATIC_ATTN_MAX_SPLITS x 130 floats = 4.26 MB, held by every GPU that
 * loads the library until the process exits). No cudaMalloc or cudaFree, no
 * allocating library call.
 *   q           device bf16 [B][16][128]: queries after q-norm and RoPE
 *   kv_pool     device bf16 blocks [n][2][8][64][128]: block p holds K then V
 *               of 64 positions for the 8 KV heads (the engine's pool layout)
 *   page_table  device int32 [B][blocks_per_seq]: physical block of each
 *               64-token block of sequence b
 *   positions   device int32 [B]: position of the query token of sequence b;
 *               its K/V must already be in the pool, attention covers
 *               positions 0..positions[b]. Values outside 0..max_position
 *               are clamped into that range on the device before any read
 *               (so no access leaves the caller's page-table rows); the
 *               output of such a sequence is then not meaningful
 *   max_position the largest value in positions (host int)
 *   out         device bf16 [B][16][128]
 *   stream      cudaStream_t (NULL = legacy default stream)
 * Returns TTS_BB_E_INVALID for NULL pointers, B outside
 * 1..TTS_BB_STATIC_ATTN_MAX_B or a max_position the page table cannot hold;
 * TTS_BB_E_CUDA if a CUDA error is already pending when the call starts (it
 * is left pending, not cleared) or a launch fails. The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current. Every call shares the
 * array and overwrites all the partials it reads, so nothing needs clearing
 * between calls; calls that overlap on the GPU (other streams, other host
 * threads) race on it and must be serialised by the caller. */
#define TTS_BB_STATIC_ATTN_MAX_B 64
#define TTS_BB_STATIC_ATTN_MAX_SPLITS 8
tts_bb_status tts_bb_gqa_decode_attention_static(const void* q, const void* kv_pool, const int32_t* page_table,
                                                 int blocks_per_seq, const int32_t* positions, int B,
                                                 int max_position, void* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* TTS_BB_H */
