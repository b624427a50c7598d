"""Plain, slow, float64 CPU oracle of the codec-token TTS backbone forward step.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import, call or
execute this package: only the test suite, the smoke check and the benchmark's
CPU-baseline leg use it. It shares no code with the CUDA engine; both sides
only read the same seeded bf16 bit patterns from the ``synth`` module.

Sources (page title, section):
  * "omnivoice-cpp docs/ARCHITECTURE.md" — GGUF layout (backbone shape, eps,
    rope base), Component architecture (hybrid embedding, audio heads,
    Qwen3 specifics: q/k norm before RoPE, SwiGLU, GQA 2:1), MaskGIT decoder
    (no KV cache, bidirectional full pass).
  * "Qwen3-TTS ncnn port" (Tencent/ncnn discussion 6877) — model structure
    (Talker 28 layers / 3072-way codebook-0 logits, Code Predictor 5 layers,
    15 autoregressive steps, 16 embeddings summed into the next Talker input),
    single-token SDPA and host attention (half-rotate RoPE, per-layer KV cache,
    GQA), mRoPE conclusion (t == h == w collapses to 1-D RoPE).
  * "rightkit-qts 0.2.0" (docs.rs) — Mode API (Code Predictor config fields,
    identity input projection for 0.6B, talker-wide embeddings), Synthetic
    tests (cached / recompute equivalence).
  * "omnivoice-cpp docs/ARCHITECTURE.md", MaskGIT decoder — the greedy token
    update of one refinement step (maskgit_update.py); Audio tokenizer
    pipeline and RVQ codec — the decode of codes to frame features (rvq.py);
    DAC decoder block channels, Snake activation, ConvTranspose1d — the
    decoder from frame features to audio (dac.py).

Every function computes its plain definition in float64; matrix products use
numpy's ``@``. No blocking, fusion or reordering beyond the definitions.
"""
from .backbone import *  # noqa: F401,F403
from .loops import *  # noqa: F401,F403
from .maskgit_update import *  # noqa: F401,F403
from .rvq import *  # noqa: F401,F403
from .dac import *  # noqa: F401,F403
