"""KIVI-style asymmetric 2-bit grouped quantisation with a full-precision window.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

[KIVI-geometry] "What quantisation error is made of": for a group, the
smallest value is the zero point, the step is the group's range divided by
2^B - 1, each element is rounded to the nearest step, so the error per element
is at most half a step. "Keys": group keys along tokens per channel
(per-channel); "Values": group values along channels per token (per-token);
the ablation flips either axis. "The systems tax": keep the most recent tokens
(up to 128) in full precision and quantise them in groups once enough have
accumulated.

Readings where the page is silent:

* B = 2, group G = 32, window W = 128 (the page's setting).
* zero point and step are stored as float16: z = fp16(min), s = fp16((max-min)/3)
  (the quotient taken in fp64); codes are computed against the stored values:
  code = clamp(round_half_even((x - z) / s), 0, 3), and code = 0 when s = 0.
  Reconstruction is z + s * code.
* tokens enter the window one by one; when it holds W + G tokens, its oldest G
  tokens are quantised as one group and leave it. After N tokens the window
  therefore holds N - nq tokens, nq = G * floor((N - W) / G) for N >= W + G,
  else nq = 0. The window keeps the inputs rounded to bfloat16.
* both K and V use the window (the page applies it to the cache as a whole).

Storage (the library's, see include/tq.h): 2-bit codes of a token occupy
channel i -> bits [2i, 2i+2) of a 2d-bit string; (z, s) pairs are float16.
"""

from dataclasses import dataclass

import numpy as np

BITS = 2
LEVELS = (1 << BITS) - 1


def to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even), returned as float32."""
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounding = 0x7FFF + ((u >> 16) & 1)
    r = ((u + rounding) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def quantize_groups(vals: np.ndarray):
    """Quantise along the last axis (one group per row).

    Returns (z16, s16, codes, t) where t = (x - z)/s in fp64 is the value whose
    rounding decided each code.
    """
    v = np.asarray(vals, dtype=np.float64)
    mn = v.min(axis=-1)
    mx = v.max(axis=-1)
    z16 = mn.astype(np.float16)
    with np.errstate(over="ignore"):  # a step above fp16's largest finite value rounds to inf
        s16 = ((mx - mn) / LEVELS).astype(np.float16)
    z = z16.astype(np.float64)[..., None]
    s = s16.astype(np.float64)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(s > 0, (v - z) / np.where(s > 0, s, 1.0), 0.0)
    codes = np.clip(np.rint(t), 0, LEVELS).astype(np.uint8)
    return z16, s16, codes, t


def dequantize_groups(z16, s16, codes) -> np.ndarray:
    return z16.astype(np.float64)[..., None] + s16.astype(np.float64)[..., None] * codes.astype(np.float64)


def quantized_length(N: int, window: int = 128, group: int = 32) -> int:
    if N < window + group:
        return 0
    return group * ((N - window) // group)


@dataclass
class KiviTensor:
    """One of K or V for one (batch, head): quantised prefix + bf16 window."""
    per_channel: bool     # groups along tokens (True) or along channels (False)
    nq: int
    codes: np.ndarray     # uint8 [nq, d]
    z16: np.ndarray       # per_channel: [nq/G, d]; per_token: [nq, d/G]
    s16: np.ndarray
    t: np.ndarray         # decision values, same shape as codes
    window: np.ndarray    # float32 (bf16 values) [N - nq, d]

    def dequantize(self, group: int = 32) -> np.ndarray:
        nq, d = self.codes.shape
        if nq:
            if self.per_channel:
                c = self.codes.reshape(nq // group, group, d).transpose(0, 2, 1)   # [g, d, G]
                q = dequantize_groups(self.z16, self.s16, c).transpose(0, 2, 1).reshape(nq, d)
            else:
                c = self.codes.reshape(nq, d // group, group)
                q = dequantize_groups(self.z16, self.s16, c).reshape(nq, d)
        else:
            q = np.zeros((0, d))
        return np.concatenate([q, self.window.astype(np.float64)], axis=0)


def quantize_tensor(x: np.ndarray, per_channel: bool, window: int = 128, group: int = 32) -> KiviTensor:
    """x [N, d] (float32 / bf16 values) -> KiviTensor for the state after N appends."""
    x = np.asarray(x, dtype=np.float32)
    N, d = x.shape
    nq = quantized_length(N, window, group)
    xq = x[:nq].astype(np.float64)
    if per_channel:
        g = xq.reshape(nq // group, group, d).transpose(0, 2, 1)        # [ng, d, G]
        z16, s16, codes, t = quantize_groups(g)
        codes = codes.transpose(0, 2, 1).reshape(nq, d)
        t = t.transpose(0, 2, 1).reshape(nq, d)
    else:
        g = xq.reshape(nq, d // group, group)                          # [nq, d/G, G]
        z16, s16, codes, t = quantize_groups(g)
        codes = codes.reshape(nq, d)
        t = t.reshape(nq, d)
    return KiviTensor(per_channel=per_channel, nq=nq, codes=codes, z16=z16, s16=s16, t=t,
                      window=to_bf16(x[nq:]))


def pack2(codes: np.ndarray) -> np.ndarray:
    """[N, d] 2-bit codes -> [N, d/4] bytes, channel i at bits [2i, 2i+2)."""
    codes = np.asarray(codes, dtype=np.uint8)
    N, d = codes.shape
    c = codes.reshape(N, d // 4, 4).astype(np.uint16)
    return (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)).astype(np.uint8)


def unpack2(packed: np.ndarray, d: int) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    N = p.shape[0]
    out = np.stack([(p >> (2 * k)) & 3 for k in range(4)], axis=-1)
    return out.reshape(N, -1)[:, :d]
