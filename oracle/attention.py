"""Decode attention over a (de)quantised cache, fp64, dense two-pass softmax.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

o = softmax(q K_hat^T / sqrt(d)) V_hat -- [HeadQ] 2.1 (keys are read through
the logits q^T k / sqrt(d)) and 2.2 (values through the p-weighted sum
sum_j p_j v_j). Grouped-query attention maps query head h to KV head
h // (H_q / H_kv). No split-K or online softmax is reproduced here: the
library's chunked evaluation must agree with this plain definition.

``qkqv_scores`` writes the sketched-key score in the form the decode kernel
evaluates it, <q_rot, nu c[idx]> + rho sqrt(pi/2)/m <S q_rot, sigma>, all
over sqrt(d) ([TQ-stats] "Main contribution 1": QJL gives an unbiased
estimate of the residual's inner product). It is algebraically the same as
<q, k_hat>/sqrt(d); the tests check the two agree.
"""

import math

import numpy as np

from . import turboquant as tq


def softmax(s: np.ndarray, axis: int = -1) -> np.ndarray:
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - np.max(s, axis=axis, keepdims=True))
    return e / np.sum(e, axis=axis, keepdims=True)


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """Single head: q [d], K [N, d], V [N, d] -> (o [d], p [N])."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[0]
    s = (np.asarray(K, dtype=np.float64) @ q) / math.sqrt(d)
    p = softmax(s)
    return p @ np.asarray(V, dtype=np.float64), p


def attend_gqa(Q: np.ndarray, K: np.ndarray, V: np.ndarray, lengths=None):
    """Q [B, Hq, d], K/V [B, Hkv, N, d] -> o [B, Hq, d] (fp64).

    ``lengths[b]`` limits sequence b to its first lengths[b] tokens.
    """
    B, Hq, d = Q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, d))
    for b in range(B):
        n = K.shape[2] if lengths is None else int(lengths[b])
        for h in range(Hq):
            out[b, h], _ = attend(Q[b, h], K[b, h // G, :n], V[b, h // G, :n])
    return out


def qkqv_scores(q: np.ndarray, enc_k: "tq.Encoded", params: "tq.Params") -> np.ndarray:
    """Scores of one query against sketched, rotated keys, in the rotated domain."""
    d = params.d
    q = np.asarray(q, dtype=np.float64)
    q_rot = params.rotate(q[None, :])[0]
    c = params.codebook(enc_k.role.bits).centroids32.astype(np.float64)
    base = enc_k.norm.astype(np.float64) * (c[enc_k.idx] @ q_rot)
    s_q = params.S.astype(np.float64) @ q_rot
    sig = np.where(enc_k.signs, 1.0, -1.0)
    m = params.S.shape[0]
    corr = enc_k.rnorm.astype(np.float64) * (tq.SQRT_HALF_PI / m) * (sig @ s_q)
    return (base + corr) / math.sqrt(d)
