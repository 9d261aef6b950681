"""Helpers of the end-to-end parity tests: the oracle's Markov chain with teacher forcing
at counted near ties, and the exclusion masks of verify decisions.  Host-side numpy only;
the arithmetic itself is the oracle's."""
import numpy as np

import oracle

RTOL = ATOL = 2e-3
DECISION_EPS = 1e-5


def near_tie_gap(top):
    """Biased-logit gap below which the two sides may pick different tokens: the logit
    tolerance on both entries, with headroom."""
    return 4.0 * (ATOL + RTOL * abs(top))


def chain_forced(logits, w1, w2, prev, gpu_tokens, lens=None):
    """The oracle's chain run position by position on its own logits.  Where the GPU's
    draft token differs, the oracle's top-2 gap there must be within the near-tie gap
    (else the test fails); the oracle then continues from the GPU's token.  Returns the
    oracle's biased logits, its (forced) tokens, the near-tie positions (gap within the
    rule, whether or not the GPU flipped) and the flips."""
    B, k, V = logits.shape
    z = np.empty(logits.shape, np.float32)
    toks = np.empty((B, k), np.int32)
    near = flips = 0
    p = np.asarray(prev, np.int32).copy()
    for i in range(k):
        g = oracle.greedy_sample(np.ascontiguousarray(logits[:, i:i + 1, :]), w1, w2, p)
        z[:, i] = g["z"][:, 0]
        t = g["draft_tokens"][:, 0].copy()
        for b in range(B):
            if lens is not None and i >= lens[b]:
                continue
            top = float(g["q_max"][b, 0])
            if g["top2_gap"][b, 0] <= near_tie_gap(top):
                near += 1
            if gpu_tokens[b, i] != t[b]:
                zz = g["z"][b, 0].astype(np.float64)
                assert top - zz[gpu_tokens[b, i]] <= near_tie_gap(top), (b, i)
                flips += 1
                t[b] = gpu_tokens[b, i]
        toks[:, i] = t
        p = t
    return {"z": z, "tokens": toks, "near_tie": near, "flip": flips}


def decision_mask(ref, window=DECISION_EPS):
    """(accept-window, draw-margin) exclusion masks over requests, from the oracle's own
    diagnostics: an accept test with |u - p/q| < window, or a Gumbel-max draw whose gap to
    the runner-up is below the oracle's binary32 error bound."""
    am = np.nan_to_num(ref["accept_margin"], nan=1.0)
    sm = np.nan_to_num(ref["sample_margin"], nan=1.0)
    return np.any(am < window, axis=1), sm < 0.0
