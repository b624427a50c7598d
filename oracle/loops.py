"""Oracle drivers for the step loops around the backbone.

Test infrastructure only. These follow the generation protocols on the pages:
  * Talker frame loop (Qwen3-TTS ncnn port, model structure: the Talker
    predicts codebook 0 from 3072-way logits; the 16 embeddings of a frame are
    summed into the next Talker input; greedy mode is used for exact alignment).
  * Code Predictor inner loop (same page: 15 autoregressive steps produce
    codebooks 1..15 from the Talker hidden state; rightkit-qts Mode API:
    identity input projection for 0.6B, talker-wide embeddings).
  * MaskGIT full bidirectional pass (omnivoice-cpp ARCHITECTURE.md, MaskGIT
    decoder and Component architecture).
  * The Talker -> Code Predictor frame loop (Qwen3-TTS ncnn port, model
    structure: 16 codes per frame, their embeddings summed into the next
    Talker input).

All drivers support teacher forcing: pass the id stream to replay and the
driver uses it instead of its own argmax, so a GPU run and the oracle see
identical inputs at every step.
"""
from __future__ import annotations

from typing import List, Optional

import numpy as np

from .backbone import Backbone, KVCache, argmax_first, codebook_embed_sum, omnivoice_embed

__all__ = ["talker_prefill", "talker_decode_steps", "code_predictor_frame", "code_predictor_frames",
           "maskgit_pass", "one_layer_run", "cp_position_ids", "talker_cp_frames"]


def talker_prefill(m: Backbone, ids: np.ndarray, cache: KVCache):
    """Prefill positions 0..P-1 with summed codebook embeddings.

    Returns (hidden[P, H] after the last layer, last-position logits, argmax).
    """
    x = codebook_embed_sum(ids, m.codebooks)
    L0 = len(cache)
    h = m.forward_cached(x, np.arange(L0, L0 + x.shape[0]), cache)
    logits = m.head_logits(h[-1:], 0)[0]
    return h, logits, int(argmax_first(logits))


def talker_decode_steps(m: Backbone, cache: KVCache, first_id0: int, rest_ids: np.ndarray,
                        forced_id0: Optional[np.ndarray] = None):
    """Greedy Talker decode: step t feeds ids [id0_t, rest_ids[t]] at position len(cache).

    id0_0 = first_id0 (argmax of the prefill); id0_{t+1} = argmax of step t,
    or forced_id0[t+1] under teacher forcing. Returns per-step hidden, logits,
    argmax and the id rows that were fed.
    """
    n = rest_ids.shape[0]
    hid, logit, am, fed = [], [], [], []
    id0 = first_id0
    for t in range(n):
        if forced_id0 is not None:
            id0 = int(forced_id0[t])
        row = np.concatenate([[id0], rest_ids[t]]).astype(np.int32)[None, :]
        x = codebook_embed_sum(row, m.codebooks)
        p = len(cache)
        h = m.forward_cached(x, [p], cache)
        lg = m.head_logits(h, 0)[0]
        a = int(argmax_first(lg))
        hid.append(h[0]); logit.append(lg); am.append(a); fed.append(row[0])
        id0 = a
    return np.array(hid), np.array(logit), np.array(am, np.int32), np.array(fed, np.int32)


def cp_position_ids(n_cb: int, j: int, code: int) -> np.ndarray:
    """Id row for a Code Predictor position that feeds codebook j alone (-1 elsewhere)."""
    row = -np.ones(n_cb, dtype=np.int32)
    row[j] = code
    return row


def code_predictor_frame(m: Backbone, talker_hidden: np.ndarray, code0: int,
                         forced: Optional[np.ndarray] = None):
    """One frame of the Code Predictor: codes 1..15 from the Talker hidden state.

    Reading of the step structure (the pages give the 15-step loop, not the
    positions): position 0 holds the Talker hidden state (identity input
    projection for the 0.6B model), position 1 the embedding E_0[code0]. The
    first call is a 2-token causal prefill whose last row goes through head 0
    to give code 1; call j (1..14) feeds E_j[code_j] at position j+1 and head j
    gives code j+1. The Code Predictor has its own final norm.
    ``forced`` (15 ints) replays codes 1..15 as the next inputs.
    Returns (codes[15], logits[15, rows], hidden[15, H]).
    """
    n_cb = len(m.codebooks)
    cache = m.new_cache()
    x0 = np.asarray(talker_hidden, np.float64)[None, :]
    x1 = codebook_embed_sum(cp_position_ids(n_cb, 0, code0)[None, :], m.codebooks)
    h = m.forward_cached(np.concatenate([x0, x1]), [0, 1], cache)
    codes, logits, hidden = [], [], []
    lg = m.head_logits(h[-1:], 0)[0]
    codes.append(int(argmax_first(lg))); logits.append(lg); hidden.append(h[-1])
    for j in range(1, 15):
        prev = int(forced[j - 1]) if forced is not None else codes[-1]
        x = codebook_embed_sum(cp_position_ids(n_cb, j, prev)[None, :], m.codebooks)
        h = m.forward_cached(x, [j + 1], cache)
        lg = m.head_logits(h, j)[0]
        codes.append(int(argmax_first(lg))); logits.append(lg); hidden.append(h[0])
    return np.array(codes, np.int32), np.array(logits), np.array(hidden)


def code_predictor_frames(m: Backbone, talker_hidden: np.ndarray, code0: np.ndarray,
                          forced: Optional[np.ndarray] = None):
    """code_predictor_frame for F independent frames at once (same steps; the
    row-wise projections of the frames share one matrix product).
    talker_hidden[F, H], code0[F], forced[F, 15] or None.
    Returns (codes[F, 15], logits[F, 15, rows])."""
    F = len(code0)
    n_cb = len(m.codebooks)
    caches = [m.new_cache() for _ in range(F)]
    xs = []
    for f in range(F):
        x1 = codebook_embed_sum(cp_position_ids(n_cb, 0, int(code0[f]))[None, :], m.codebooks)
        xs.append(np.concatenate([np.asarray(talker_hidden[f], np.float64)[None, :], x1]))
    hs = m.forward_cached_multi(xs, caches)
    last = np.stack([h[-1] for h in hs])
    lg = m.head_logits(last, 0)
    codes = [argmax_first(lg)]
    logits = [lg]
    for j in range(1, 15):
        prev = forced[:, j - 1] if forced is not None else codes[-1]
        xs = [codebook_embed_sum(cp_position_ids(n_cb, j, int(prev[f]))[None, :], m.codebooks) for f in range(F)]
        hs = m.forward_cached_multi(xs, caches)
        lg = m.head_logits(np.concatenate(hs), j)
        codes.append(argmax_first(lg))
        logits.append(lg)
    return np.stack(codes, axis=1).astype(np.int32), np.stack(logits, axis=1)


def talker_cp_frames(talker: Backbone, cp: Backbone, cache: KVCache, first_codes: np.ndarray, n_frames: int,
                     forced: Optional[np.ndarray] = None):
    """The frame loop of the three-network protocol (Qwen3-TTS ncnn port, model
    structure): per frame the Talker takes the sum of the previous frame's 16
    codebook embeddings at its next position and predicts codebook 0 with the
    3072-way head; the Code Predictor, with fresh state every frame, takes the
    Talker's hidden state and code 0 and predicts codebooks 1..15; the frame's
    16 codes are the next frame's Talker input.

    Reading: the hidden state handed to the Code Predictor is the Talker's
    last-layer output after its final norm (the vector its codec head reads).
    first_codes[16]: the input of frame 0. forced[n_frames, 16] replays codes
    (teacher forcing) as the next inputs. Returns (codes [n_frames, 16], Talker
    logits [n_frames, rows], Code Predictor logits [n_frames, 15, rows],
    hidden handed over [n_frames, H]).
    """
    codes_in = np.asarray(first_codes, np.int32)
    out_codes, t_logits, c_logits, handed = [], [], [], []
    for f in range(n_frames):
        x = codebook_embed_sum(codes_in[None, :], talker.codebooks)
        h = talker.forward_cached(x, [len(cache)], cache)
        lg = talker.head_logits(h, 0)[0]
        code0 = int(forced[f, 0]) if forced is not None else int(argmax_first(lg))
        hidden = talker.final_norm(h)[0]
        cp_codes, cp_lg, _ = code_predictor_frame(cp, hidden, code0, None if forced is None else forced[f, 1:])
        frame = np.concatenate([[code0], cp_codes]).astype(np.int32)
        if forced is not None:
            frame = np.asarray(forced[f], np.int32)
        out_codes.append(np.concatenate([[int(argmax_first(lg))], cp_codes]).astype(np.int32))
        t_logits.append(lg)
        c_logits.append(cp_lg)
        handed.append(hidden)
        codes_in = frame
    return np.array(out_codes), np.array(t_logits), np.array(c_logits), np.array(handed)


def maskgit_pass(m: Backbone, ids: np.ndarray, audio_mask: np.ndarray, audio_start: int,
                 rows: Optional[List[int]] = None, key_lens: Optional[np.ndarray] = None):
    """One MaskGIT refinement pass: hybrid embedding, 28 bidirectional layers,
    audio heads over the audio window [audio_start, S) only (the T_audio output
    narrowing of omnivoice-cpp ARCHITECTURE.md, Inner-loop optimisations).

    Returns (logits[len(rows), 8, S - audio_start, 1025], hidden[len(rows), S, H]).
    """
    B, K, S = ids.shape
    rows = list(range(B)) if rows is None else list(rows)
    x = omnivoice_embed(ids[rows], audio_mask[rows], m.text_table, m.audio_table,
                        m.s.audio_vocab)
    outs, hids = [], []
    for i, b in enumerate(rows):
        kl = None if key_lens is None else int(key_lens[b])
        h = m.forward_bidirectional(x[i], kl)
        hids.append(h)
        outs.append(m.audio_logits(h[None, audio_start:])[0])
    return np.array(outs), np.array(hids)


def one_layer_run(m: Backbone, X: np.ndarray, n_prefill: int):
    """Single-layer config: prefill rows 0..n_prefill-1 of X, then decode the
    remaining rows one at a time with the KV cache. Returns the hidden state
    after the layer for every row (prefill rows, then decode rows)."""
    cache = m.new_cache()
    hp = m.forward_cached(X[:n_prefill], np.arange(n_prefill), cache)
    hd = [m.forward_cached(X[t:t + 1], [t], cache)[0] for t in range(n_prefill, X.shape[0])]
    return hp, np.array(hd)
