"""Oracle of the n-gram (prompt lookup) draft proposer.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the CUDA library or its
binding.

What it restates. "Speculative Decoding : accélérer l'inférence des LLM",
§N-gram lookup et variantes sans modèle: look in the context for the last
sequence of n tokens and propose, as draft tokens, the tokens that followed
it; no model, no training. The same page's §Mise en œuvre dans vLLM shows the
knobs: num_speculative_tokens (gamma), prompt_lookup_min = 2,
prompt_lookup_max = 5.

Readings (the page leaves these open):
  * The context is the request's whole history h = token_buf[b, :L] (prompt
    and generated tokens alike).
  * n is tried from n_max down to n_min; the first (longest) n for which the
    query h[L-n:L] occurs earlier wins. "Earlier" means a start j with
    j + n <= L - 1, so that at least one token follows the occurrence.
  * Among several earlier occurrences, the latest (largest j) is taken.
  * The proposal is h[j+n : j+n+k] with k = min(gamma, L - (j + n)): it stops
    at the end of the history. No match for any n: k = 0.
  * Outputs: draft_tokens[b, :k] = the proposal, draft_tokens[b, k:] = -1,
    num_draft[b] = k. A length outside [0, max_len] gives k = 0 and flags
    the request BAD.

Plain loops, brute force: every n, every j, every element compared.
"""
from __future__ import annotations

import numpy as np

STATUS_BAD = 0x1


def propose_one(hist, gamma, n_min, n_max):
    """(proposal list, n used or 0) for one history (a Python list)."""
    L = len(hist)
    for n in range(n_max, n_min - 1, -1):
        if L < n + 1:
            continue
        query = hist[L - n:L]
        best = -1
        for j in range(0, L - n):  # j + n <= L - 1
            if hist[j:j + n] == query:
                best = j  # keeps the latest
        if best >= 0:
            k = min(gamma, L - (best + n))
            return hist[best + n:best + n + k], n
    return [], 0


def propose(token_buf, seq_lens, gamma, n_min=2, n_max=5):
    """Returns (draft_tokens [B, gamma] int32, num_draft [B] int32, status)."""
    buf = np.asarray(token_buf, dtype=np.int32)
    lens = np.asarray(seq_lens, dtype=np.int32)
    B, max_len = buf.shape
    out = np.full((B, gamma), -1, dtype=np.int32)
    num = np.zeros(B, dtype=np.int32)
    status = 0
    for b in range(B):
        L = int(lens[b])
        if L < 0 or L > max_len:
            status |= STATUS_BAD
            continue
        prop, _ = propose_one([int(x) for x in buf[b, :L]], gamma, n_min, n_max)
        out[b, :len(prop)] = prop
        num[b] = len(prop)
    return out, num, status
