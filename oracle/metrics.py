"""Quality measures against full precision (fp64).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

* KL(p || p_hat) between the full-precision and the quantised softmax, and the
  top-5 routing recall -- [TQ-stats] "Evaluation metrics" (mechanism proxies);
  "Significance": mean KL is too optimistic, so the worst case is reported too.
* the 6D error frame -- [TQ-stats] "Evaluation metrics": scale (SNR) and
  direction (phi) errors at the key cache, the value cache and the output T.
  The page names the six axes but does not print their formulas; this module
  uses: scale error |(||x_hat|| / ||x||) - 1| and SNR_dB = 10 log10(||x||^2 /
  ||x - x_hat||^2); direction error 1 - cos(x, x_hat) and phi = arccos(cos).
  parity unpinned: these definitions are a reading, not something the pages fix.
"""

import numpy as np


def kl(p: np.ndarray, p_hat: np.ndarray) -> np.ndarray:
    """KL(p || p_hat) along the last axis."""
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(p_hat, dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        terms = np.where(p > 0, p * (np.log(p) - np.log(np.maximum(q, 1e-300))), 0.0)
    return np.sum(terms, axis=-1)


def topk_recall(p: np.ndarray, p_hat: np.ndarray, k: int = 5) -> np.ndarray:
    p = np.asarray(p)
    q = np.asarray(p_hat)
    a = np.argsort(-p, axis=-1, kind="stable")[..., :k]
    b = np.argsort(-q, axis=-1, kind="stable")[..., :k]
    out = np.empty(p.shape[:-1])
    for ix in np.ndindex(*p.shape[:-1]):
        out[ix] = len(set(a[ix].tolist()) & set(b[ix].tolist())) / k
    return out


def six_d(x: np.ndarray, x_hat: np.ndarray) -> dict:
    """Per-vector scale and direction errors along the last axis (parity unpinned)."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(x_hat, dtype=np.float64)
    nx = np.linalg.norm(x, axis=-1)
    ny = np.linalg.norm(y, axis=-1)
    err = np.linalg.norm(x - y, axis=-1)
    cos = np.sum(x * y, axis=-1) / np.maximum(nx * ny, 1e-300)
    cos = np.clip(cos, -1.0, 1.0)
    with np.errstate(divide="ignore"):
        snr = 10.0 * np.log10(nx ** 2 / np.maximum(err ** 2, 1e-300))
    return {"scale_err": np.abs(ny / np.maximum(nx, 1e-300) - 1.0), "snr_db": snr,
            "dir_err": 1.0 - cos, "phi": np.arccos(cos)}


def summarize(v: np.ndarray) -> dict:
    v = np.asarray(v, dtype=np.float64).reshape(-1)
    return {"mean": float(np.mean(v)), "worst": float(np.max(v)), "min": float(np.min(v))}
