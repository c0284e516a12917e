"""Quality of the GPU path against full precision: KL(p || p_hat), top-5 routing
recall, and the scale / direction errors at K, V and the attention output.

"Statistical Inference and Quality Measures of KV Cache Quantisations Inspired by
TurboQuant", technical summary, "Evaluation metrics" (mechanism proxies and the
6D frame; the frame's formulas are a reading, see oracle/metrics.py) and "Main
contribution 2" (at a 4-bit budget the asymmetric KQV split beats QKQV).

Everything quantised here is produced by the CUDA path (append through the C
ABI, tq_dequantize for K_hat / V_hat, tq_decode_attention for the output); the
full-precision reference is fp64 attention over the raw inputs. The table is
printed (visible with pytest -s).
"""

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import metrics as om
from quantised_kv_cache_gb300 import tq
from quantised_kv_cache_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROWS = []


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantised_kv_cache_gb300 import build
    build.build()
    yield
    _write_report()


def _scores(q, K):
    return np.einsum("bhd,bhnd->bhn", q, K) / np.sqrt(q.shape[-1])


def _softmax(s):
    s = s - s.max(axis=-1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=-1, keepdims=True)


def _measure(label, scheme, n, w, key_dist=None, B=1, H=4, N=1024, seed=5, rotation="wht"):
    q, k, v = wl.generate(w, "cpu", seed=seed, key_dist=key_dist, batch=B, heads_kv=H, heads_q=H, seq=N)
    ctx = tq.Context(128, n, scheme, 42, rotation=rotation)
    cache = tq.Cache(ctx, B, H, N)
    tq.tq_append_quantize(ctx.handle, cache, k.to(DEV), v.to(DEV), torch.zeros(B, dtype=torch.int32, device=DEV))
    kh, vh = tq.tq_dequantize(ctx.handle, cache, 0, N)
    seq = torch.full((B,), N, dtype=torch.int32, device=DEV)
    out = tq.tq_decode_attention(ctx.handle, cache, q.to(DEV), seq, max_len=N)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    q64, k64, v64 = (x.double().numpy() for x in (q, k, v))
    kh64, vh64, o = kh.double().cpu().numpy(), vh.double().cpu().numpy(), out.double().cpu().numpy()
    p, ph = _softmax(_scores(q64, k64)), _softmax(_scores(q64, kh64))
    o_full = oatt.attend_gqa(q64, k64, v64)
    row = {"label": label, "scheme": scheme, "n": n,
           "kl": om.summarize(om.kl(p, ph)), "top5": om.summarize(om.topk_recall(p, ph, 5))}
    for name, x, xh in (("K", k64, kh64), ("V", v64, vh64), ("T", o_full, o)):
        d = om.six_d(x, xh)
        row[name] = {key: float(np.mean(val)) for key, val in d.items()}
    ROWS.append(row)
    return row


def _write_report():
    if not ROWS:
        return
    lines = ["| workload | scheme | n | KL mean | KL worst | top-5 mean | top-5 min | K SNR dB | K 1-cos | "
             "V SNR dB | V 1-cos | T SNR dB | T 1-cos |", "|" + "---|" * 13]
    for r in ROWS:
        lines.append(f"| {r['label']} | {r['scheme']} | {r['n']} | {r['kl']['mean']:.2e} | {r['kl']['worst']:.2e} | "
                     f"{r['top5']['mean']:.3f} | {r['top5']['min']:.2f} | {r['K']['snr_db']:.1f} | "
                     f"{r['K']['dir_err']:.2e} | {r['V']['snr_db']:.1f} | {r['V']['dir_err']:.2e} | "
                     f"{r['T']['snr_db']:.1f} | {r['T']['dir_err']:.2e} |")
    text = "\n".join(lines)
    print("\n" + text)


@pytest.mark.parametrize("dist", ["gauss", "lowrank", "student3"])
def test_quality_sweep_improves_with_bits_and_kqv_beats_qkqv(dist):
    w = wl.WORKLOADS[3]
    kl = {}
    for scheme in ("KV", "KQV", "QKQV"):
        for n in (2, 3, 4):
            r = _measure(f"sweep B1 H4 N1024 fp32 keys={dist}", scheme, n, w, key_dist=dist)
            kl[scheme, n] = r["kl"]["mean"]
            assert r["top5"]["mean"] > 0.2
    for scheme in ("KV", "KQV", "QKQV"):
        assert kl[scheme, 4] < kl[scheme, 2], (scheme, dist, kl)
    if dist == "gauss":
        for scheme in ("KV", "KQV", "QKQV"):
            assert kl[scheme, 4] < kl[scheme, 3] < kl[scheme, 2], (scheme, kl)
        # [TQ-stats] "Main contribution 2": at 4 bits the K-heavy split wins on attention
        assert kl["KQV", 4] < kl["QKQV", 4], kl


def test_quality_llama7b_shaped_kqv4():
    # keys with log-normal channel scales and x10 outlier channels: peaked scores, so the
    # quantised keys move the softmax more than on Gaussian keys (reported, loosely bounded)
    r = _measure("Llama-2-7B-shaped sample B2 H8 N2048 bf16", "KQV", 4, wl.WORKLOADS[2], B=2, H=8, N=2048)
    assert r["top5"]["mean"] > 0.5
    assert r["K"]["dir_err"] < 0.01 and r["T"]["dir_err"] < 0.5


@pytest.mark.parametrize("dist", ["gauss", "student3"])
def test_dense_rotation_quality_matches_the_hadamard(dist):
    # [KVQuant++] "Rate-distortion performance": the QR rotation and the Hadamard transform
    # both bring the coordinates to the fitted marginal, so the K / V reconstruction errors
    # (the rate-distortion quantity the page states) agree between them on the same inputs
    # and budget. The attention KL and the output error are reported: over four heads they
    # move with which tokens' errors meet the largest scores, by up to a few times either way
    w = wl.WORKLOADS[3]
    for scheme, n in (("KQV", 4), ("KQV", 3), ("QKQV", 3)):
        r_w = _measure(f"rotation study B1 H4 N1024 fp32 keys={dist}, Walsh-Hadamard", scheme, n, w, key_dist=dist)
        r_d = _measure(f"rotation study B1 H4 N1024 fp32 keys={dist}, dense SO(d)", scheme, n, w, key_dist=dist,
                       rotation="dense")
        for x in ("K", "V"):
            assert abs(r_w[x]["snr_db"] - r_d[x]["snr_db"]) < 0.5, (scheme, n, x, r_w[x], r_d[x])
            assert abs(r_w[x]["dir_err"] - r_d[x]["dir_err"]) < 0.1 * r_w[x]["dir_err"], (scheme, n, x)


def _kl_rows(q, K, Kh):
    """KL(p || p_hat) per query row, q [n, d], K / Kh [N, d]."""
    s, sh = q @ K.T / np.sqrt(128), q @ Kh.T / np.sqrt(128)
    p, ph = _softmax(s), _softmax(sh)
    return om.kl(p, ph)


def test_headq_side_code_cuts_the_kl_of_calibrated_queries():
    # [HeadQ] section 3 on the rank-4 key / query family (config 3 (b)): per KV head, 63
    # queries of the head's query subspace calibrate a rank-4 basis; 64 other queries of the
    # same subspace are evaluated. 2-bit KQV keys through the CUDA path, with and without side
    # codes (everything else equal)
    w = wl.WORKLOADS[3]
    H, N = 4, 1024
    q, k, v = wl.generate(w, "cpu", seed=21, key_dist="lowrank", batch=1, heads_kv=H, heads_q=H * 127, seq=N)
    q64 = q[0].double().numpy().reshape(H, 127, 128)
    k64 = k[0].double().numpy()
    U = np.stack([sc_principal(q64[h, :63]) for h in range(H)]).astype(np.float32)
    kl = {}
    for name, basis in (("base", None), ("side", U)):
        ctx = tq.Context(128, 2, "KQV", 42)
        if basis is not None:
            tq.tq_set_side_basis(ctx.handle, basis)
        cache = tq.Cache(ctx, 1, H, N)
        tq.tq_append_quantize(ctx.handle, cache, k.to(DEV), v.to(DEV), torch.zeros(1, dtype=torch.int32, device=DEV))
        kh, _ = tq.tq_dequantize(ctx.handle, cache, 0, N)
        kh = kh[0].double().cpu().numpy()
        kl[name] = np.concatenate([_kl_rows(q64[h, 63:], k64[h], kh[h]) for h in range(H)])
    print(f"\nHeadQ rank-4 side code, 2-bit KQV keys, rank-4 queries: KL mean {kl['base'].mean():.3e} -> "
          f"{kl['side'].mean():.3e}, worst {kl['base'].max():.3e} -> {kl['side'].max():.3e}")
    assert kl["side"].mean() < 0.05 * kl["base"].mean()


def sc_principal(x, r=4):
    return tq.tq_principal_basis(np.asarray(x, dtype=np.float32), r)


@pytest.mark.parametrize("dist", ["gauss", "lowrank"])
def test_low_rank_residual_correction_reduces_key_error(dist):
    # [KVQuant++] "Core innovation 4": the top-r right singular vectors of the residual
    # K - K_hat (per head, from a first pass without side codes) as the side basis; the key
    # reconstruction error falls, by at least the Eckart-Young share of the energy those
    # directions hold (the page's 11 % / 19 % at rank 4 / 8 are real-model figures)
    w = wl.WORKLOADS[3]
    H, N = 4, 2048
    _, k, v = wl.generate(w, "cpu", seed=23, key_dist=dist, batch=1, heads_kv=H, heads_q=H, seq=N)
    k64 = k[0].double().numpy()
    ctx = tq.Context(128, 3, "KQV", 42)
    cache = tq.Cache(ctx, 1, H, N)
    tq.tq_append_quantize(ctx.handle, cache, k.to(DEV), v.to(DEV), torch.zeros(1, dtype=torch.int32, device=DEV))
    kh0 = tq.tq_dequantize(ctx.handle, cache, 0, N)[0][0].double().cpu().numpy()
    E = k64 - kh0
    for r in (4, 8):
        U = np.stack([sc_principal(E[h], r) for h in range(H)]).astype(np.float32)
        ctx2 = tq.Context(128, 3, "KQV", 42)
        tq.tq_set_side_basis(ctx2.handle, U)
        c2 = tq.Cache(ctx2, 1, H, N)
        tq.tq_append_quantize(ctx2.handle, c2, k.to(DEV), v.to(DEV), torch.zeros(1, dtype=torch.int32, device=DEV))
        kh = tq.tq_dequantize(ctx2.handle, c2, 0, N)[0][0].double().cpu().numpy()
        mse0, mse = np.mean(E ** 2), np.mean((k64 - kh) ** 2)
        share = np.mean([np.sum((E[h] @ U[h].astype(np.float64)) ** 2) / np.sum(E[h] ** 2) for h in range(H)])
        print(f"\nlow-rank correction keys={dist} rank {r}: key MSE {mse0:.4e} -> {mse:.4e} "
              f"({100 * (1 - mse / mse0):.1f} % lower; the basis holds {100 * share:.1f} % of the residual energy)")
        assert mse < mse0 * (1 - 0.9 * share)
