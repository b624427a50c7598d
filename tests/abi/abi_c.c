/* Plain C99 consumer of include/tts_bb.h: built with -std=c99 -Wall -Werror
 * -pedantic and run without a GPU. It calls every entry point through an
 * early-return path (NULL handle or invalid arguments), so it checks that the
 * header is valid C99 and that every declared symbol links and returns the
 * documented status without touching a device. */
#include <stdio.h>
#include <string.h>
#include "tts_bb.h"

#define EXPECT(cond)                                              \
    do {                                                          \
        if (!(cond)) {                                            \
            fprintf(stderr, "FAILED: %s (line %d)\n", #cond, __LINE__); \
            return 1;                                             \
        }                                                         \
    } while (0)

int main(void) {
    tts_bb_config cfg;
    tts_bb_weights w;
    tts_bb_opts o;
    tts_bb* h = NULL;
    int32_t slots[1] = {0}, lens[1] = {1};
    char k[16], v[16];
    memset(&w, 0, sizeof w);
    memset(&o, 0, sizeof o);
    tts_bb_default_config(&cfg);
    EXPECT(cfg.n_layers == 28 && cfg.hidden == 1024 && cfg.n_q_heads == 16 && cfg.n_kv_heads == 8);
    EXPECT(cfg.head_dim == 128 && cfg.ffn == 3072 && cfg.n_codebooks == 16 && cfg.head_rows == 3072);
    EXPECT(strncmp(tts_bb_version(), "0.1.0", 5) == 0);
    EXPECT(tts_bb_create(NULL, &w, NULL, &h) == TTS_BB_E_INVALID && h == NULL);
    EXPECT(tts_bb_create(&cfg, NULL, NULL, &h) == TTS_BB_E_INVALID);
    EXPECT(tts_bb_create(&cfg, &w, NULL, NULL) == TTS_BB_E_INVALID);
    cfg.hidden = 2048;
    EXPECT(tts_bb_create(&cfg, &w, NULL, &h) == TTS_BB_E_UNSUPPORTED);
    tts_bb_default_config(&cfg);
    EXPECT(tts_bb_create(&cfg, &w, NULL, &h) == TTS_BB_E_INVALID); /* NULL weight pointers */
    EXPECT(tts_bb_prefill(NULL, 1, 1, slots, lens, NULL, -1, NULL, NULL, &o) == TTS_BB_E_INVALID);
    EXPECT(tts_bb_decode_step(NULL, 1, slots, lens, NULL, -1, NULL, NULL, NULL) == TTS_BB_E_INVALID);
    EXPECT(tts_bb_maskgit_pass(NULL, 1, 1, NULL, NULL, NULL, 0, NULL, NULL) == TTS_BB_E_INVALID);
    EXPECT(tts_bb_release(NULL, 0) == TTS_BB_E_INVALID);
    EXPECT(tts_bb_truncate(NULL, 0, 0) == TTS_BB_E_INVALID);
    EXPECT(tts_bb_slot_len(NULL, 0) == -1);
    EXPECT(tts_bb_sync(NULL) == TTS_BB_E_INVALID);
    EXPECT(tts_bb_debug_kv_read(NULL, 0, 0, 0, 1, k, v) == TTS_BB_E_INVALID);
    EXPECT(tts_bb_debug_kv_write(NULL, 0, 0, 0, 1, k, v) == TTS_BB_E_INVALID);
    EXPECT(tts_bb_launch_count(NULL) == 0);
    EXPECT(tts_bb_profile(NULL, 1) == TTS_BB_E_INVALID);
    EXPECT(strcmp(tts_bb_profile_report(NULL), "{}") == 0);
    EXPECT(strlen(tts_bb_last_error(NULL)) > 0);
    EXPECT(tts_bb_gqa_decode_attention_static(NULL, NULL, NULL, 1, NULL, 1, 0, NULL, NULL) == TTS_BB_E_INVALID);
    EXPECT(tts_bb_gqa_decode_attention_static(k, k, slots, 1, slots, TTS_BB_STATIC_ATTN_MAX_B + 1, 0, v, NULL) ==
           TTS_BB_E_INVALID);
    EXPECT(tts_bb_frame_step(NULL, NULL, 1, NULL, NULL, NULL, NULL) == TTS_BB_E_INVALID);
    EXPECT(tts_bb_decode_step_host(NULL, 1, NULL, NULL, NULL, 0, NULL, NULL) == TTS_BB_E_INVALID);
    {
        tts_bb_rvq* r = NULL;
        EXPECT(tts_bb_rvq_create(8, 1024, 64, 1024, NULL, NULL, NULL, NULL, &r) == TTS_BB_E_INVALID && r == NULL);
        EXPECT(tts_bb_rvq_decode(NULL, 1, 1, NULL, NULL) == TTS_BB_E_INVALID);
        EXPECT(tts_bb_rvq_sync(NULL) == TTS_BB_E_INVALID);
        tts_bb_rvq_free(NULL);
        tts_bb_quantizer* qz = NULL;
        EXPECT(tts_bb_quantizer_create(16, 2048, 256, 512, NULL, NULL, NULL, NULL, &qz) == TTS_BB_E_INVALID && qz == NULL);
        EXPECT(tts_bb_quantizer_decode(NULL, 1, 1, NULL, NULL) == TTS_BB_E_INVALID);
        EXPECT(tts_bb_quantizer_sync(NULL) == TTS_BB_E_INVALID);
        tts_bb_quantizer_free(NULL);
    }
    {
        tts_bb_dac* d = NULL;
        tts_bb_dac_weights dw;
        memset(&dw, 0, sizeof(dw));
        EXPECT(tts_bb_dac_create(&dw, NULL, &d) == TTS_BB_E_INVALID && d == NULL);
        EXPECT(tts_bb_dac_decode(NULL, 1, 1, NULL, NULL) == TTS_BB_E_INVALID);
        EXPECT(tts_bb_dac_sync(NULL) == TTS_BB_E_INVALID);
        tts_bb_dac_free(NULL);
    }
    EXPECT(tts_bb_maskgit_update(NULL, 1, 1, NULL, 1, 0, 0, NULL, 1, 0, 0, 1, 2.0f, 5.0f) == TTS_BB_E_INVALID);
    {
        int32_t counts[32];
        int32_t sum = 0;
        int i;
        EXPECT(tts_bb_maskgit_schedule(32, 6144, 0.1, counts) == TTS_BB_OK);
        for (i = 0; i < 32; ++i) sum += counts[i];
        EXPECT(sum >= 6144 && sum < 6144 + 32 && counts[0] < counts[31]);
        EXPECT(tts_bb_maskgit_schedule(0, 10, 0.1, counts) == TTS_BB_E_INVALID);
    }
    tts_bb_free(NULL);
    printf("abi_c: ok\n");
    return 0;
}
