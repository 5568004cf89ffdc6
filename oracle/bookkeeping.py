"""Oracle of the post-verify bookkeeping step (commit of the emitted tokens).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the CUDA library or its
binding.

What it restates. "Accélérer Sonar grâce à la spéculation", §Planification
MTP pour un jeton unique: after the draft tokens are accepted, the target's
input tokens are shifted and a kernel inserts the next target tokens into
their slots, so that no CPU synchronisation is needed to learn the accepted
length before the next step. "Speculative Decoding : accélérer l'inférence
des LLM", §Principe et garanties mathématiques: one verification pass emits
between 1 and gamma + 1 tokens (the accepted draft tokens, then the target's
own token).

Readings (the pages fix no layout):
  * Each request b has a token buffer token_buf[b, :max_len] and a length
    seq_lens[b]; its history is token_buf[b, :seq_lens[b]].
  * A verification result (out_tokens[b], n = out_num_accepted[b]) emits the
    n + 1 tokens out_tokens[b, 0..n]; they are appended at seq_lens[b].
  * If they do not all fit in max_len, the ones that fit are appended and the
    request is flagged TRUNCATED.
  * n < 0 (a request the verifier rejected as invalid), n > gamma, a negative
    emitted token, or a length outside [0, max_len] leaves the request as it
    is and flags it BAD.
  * next_input[b] is the last token of the history after the commit (the
    input of the next draft step), -1 if the history is empty.

This is a plain loop over requests and tokens; no batching or reordering.
"""
from __future__ import annotations

import numpy as np

STATUS_BAD = 0x1        # same bit as SV_STATUS_BAD_REQUEST
STATUS_TRUNCATED = 0x4  # same bit as SV_STATUS_TRUNCATED


def commit(out_tokens, out_num_accepted, token_buf, seq_lens, max_len):
    """Returns (token_buf, seq_lens, next_input, status) as new arrays."""
    out_tokens = np.asarray(out_tokens, dtype=np.int32)
    n_acc = np.asarray(out_num_accepted, dtype=np.int32)
    buf = np.array(token_buf, dtype=np.int32, copy=True)
    lens = np.array(seq_lens, dtype=np.int32, copy=True)
    B, G1 = out_tokens.shape
    gamma = G1 - 1
    nxt = np.full(B, -1, dtype=np.int32)
    status = 0
    for b in range(B):
        n = int(n_acc[b])
        L = int(lens[b])
        bad = n < 0 or n > gamma or L < 0 or L > max_len
        if not bad:
            for j in range(n + 1):
                if out_tokens[b, j] < 0:
                    bad = True
        if bad:
            status |= STATUS_BAD
            nxt[b] = -1
            continue
        emitted = n + 1
        room = max_len - L
        c = min(emitted, room)
        for j in range(c):
            buf[b, L + j] = out_tokens[b, j]
        if c < emitted:
            status |= STATUS_TRUNCATED
        lens[b] = L + c
        nxt[b] = buf[b, L + c - 1] if L + c > 0 else -1
    return buf, lens, nxt, status
