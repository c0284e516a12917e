"""GPU parity of the KIVI-style 2-bit grouped path (all four axis layouts, the
bf16 window and its group flush) against the CPU oracle, through the C ABI."""

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import kivi as okivi
from quantised_kv_cache_gb300 import tq
from quantised_kv_cache_gb300 import workloads as wl

import parity as P

pytestmark = pytest.mark.gpu
DEV = "cuda"
LAYOUTS = [(True, True), (False, False), (False, True), (True, False)]  # (K per-channel, V per-token)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantised_kv_cache_gb300 import build
    build.build()


def _inputs(B, H, N, seed, dtype=torch.bfloat16):
    w = wl.WORKLOADS[5]
    return wl.generate(w, "cpu", seed=seed, batch=B, heads_kv=H, seq=N, dtype=dtype)


def _fill(ctx, cache, k, v, chunks):
    """Append k/v [B,H,N,d] in the given chunk sizes (same for every sequence)."""
    B = k.shape[0]
    t = 0
    for c in chunks:
        lens = torch.full((B,), t, dtype=torch.int32, device=DEV)
        tq.tq_append_quantize(ctx.handle, cache, k[:, :, t:t + c].contiguous().to(DEV),
                              v[:, :, t:t + c].contiguous().to(DEV), lens)
        t += c
    return t


def _check_tensor(cache, which, x, per_channel, B, H, N):
    cap = cache.struct.capacity
    codes = P.kivi_gpu_codes(cache, which, B, H, N)
    z, s = P.kivi_gpu_stats(cache, which, B, H, per_channel)
    ring = P.kivi_gpu_window(cache, which, B, H)
    rep = P.BandReport()
    for b in range(B):
        for h in range(H):
            st = okivi.quantize_tensor(x[b, h].float().numpy(), per_channel)
            nq = st.nq
            gz, gs = z[b, h], s[b, h]
            if per_channel:
                np.testing.assert_array_equal(gz[: nq // 32], st.z16)
                np.testing.assert_array_equal(gs[: nq // 32], st.s16)
            else:
                np.testing.assert_array_equal(gz[:nq], st.z16)
                np.testing.assert_array_equal(gs[:nq], st.s16)
            mism = codes[b, h, :nq] != st.codes
            dist = np.abs(np.abs(st.t - np.floor(st.t)) - 0.5)  # distance to the rounding boundary
            rep.add(mism, dist)
            win = np.stack([ring[b, h, j % 160] for j in range(nq, N)]) if N > nq else np.zeros((0, 128))
            np.testing.assert_array_equal(win, st.window)
    assert rep.ok(), f"{which}: {rep}"


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("chunks", [[300], [100, 1, 1, 60, 33, 105], [159], [160, 1]])
def test_kivi_append_matches_oracle(layout, chunks):
    kpc, vpt = layout
    B, H = 2, 3
    N = sum(chunks)
    q, k, v = _inputs(B, H, N, seed=N + 17 * kpc + 3 * vpt)
    ctx = tq.Context(128, 2, "KIVI", 0, k_per_channel=kpc, v_per_token=vpt)
    cache = tq.Cache(ctx, B, H, 320)
    _fill(ctx, cache, k, v, chunks)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    _check_tensor(cache, "k", k, kpc, B, H, N)
    _check_tensor(cache, "v", v, not vpt, B, H, N)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_kivi_append_of_fp32_inputs_matches_oracle(layout):
    # fp32 inputs take their own load paths (tokens already in the window are bfloat16)
    kpc, vpt = layout
    B, H, chunks = 2, 3, [100, 1, 1, 60, 33, 105]
    N = sum(chunks)
    q, k, v = _inputs(B, H, N, seed=5 + kpc + 2 * vpt, dtype=torch.float32)
    ctx = tq.Context(128, 2, "KIVI", 0, k_per_channel=kpc, v_per_token=vpt)
    cache = tq.Cache(ctx, B, H, 320)
    _fill(ctx, cache, k, v, chunks)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    # the window holds bfloat16, so a token that ends an append inside the window (at or after
    # nq of that append's total) is quantised later from its bfloat16 value
    ke, ve = k.clone(), v.clone()
    t = 0
    for c in chunks:
        lo = max(t, okivi.quantized_length(t + c))
        ke[:, :, lo:t + c] = k[:, :, lo:t + c].to(torch.bfloat16).float()
        ve[:, :, lo:t + c] = v[:, :, lo:t + c].to(torch.bfloat16).float()
        t += c
    _check_tensor(cache, "k", ke, kpc, B, H, N)
    _check_tensor(cache, "v", ve, not vpt, B, H, N)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("G", [1, 4])
def test_kivi_decode_matches_oracle(layout, G):
    kpc, vpt = layout
    B, Hkv = 2, 2
    Hq = G * Hkv
    N = 1000
    lens = [1000, 421]
    _, k, v = _inputs(B, Hkv, N, seed=5 + G)
    q = torch.randn((B, Hq, 128), generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    ctx = tq.Context(128, 2, "KIVI", 0, k_per_channel=kpc, v_per_token=vpt)
    cache = tq.Cache(ctx, B, Hkv, 1024)
    # each sequence holds exactly lens[b] tokens: fill b=1 separately
    _fill(ctx, cache, k, v, [N])
    cache1 = tq.Cache(ctx, B, Hkv, 1024)
    _fill(ctx, cache1, k[:, :, :lens[1]].contiguous(), v[:, :, :lens[1]].contiguous(), [lens[1]])
    for name in cache.tensors:  # splice sequence 1's state from the shorter fill
        t = cache.tensors[name].view(B, -1)
        t[1].copy_(cache1.tensors[name].view(B, -1)[1])
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = tq.tq_decode_attention(ctx.handle, cache, q.to(DEV), seq, max_len=N, splits=3).cpu().numpy()
    for b in range(B):
        Kh = P.kivi_dequant_gpu_state(cache, "k", B, Hkv, lens[b], kpc)[b]
        Vh = P.kivi_dequant_gpu_state(cache, "v", B, Hkv, lens[b], not vpt)[b]
        for h in range(Hq):
            want, _ = oatt.attend(q[b, h].float().numpy(), Kh[h // G], Vh[h // G])
            assert P.rel_l2(out[b, h], want) < 1e-3


@pytest.mark.parametrize("layout", LAYOUTS[:2])
def test_kivi_dequantize_matches_state(layout):
    kpc, vpt = layout
    B, H, N = 1, 2, 260
    _, k, v = _inputs(B, H, N, seed=2)
    ctx = tq.Context(128, 2, "KIVI", 0, k_per_channel=kpc, v_per_token=vpt)
    cache = tq.Cache(ctx, B, H, 288)
    _fill(ctx, cache, k, v, [N])
    seq = torch.tensor([N], dtype=torch.int32, device=DEV)
    kh, vh = tq.tq_dequantize(ctx.handle, cache, 0, N, seq_lens=seq)
    np.testing.assert_allclose(kh.cpu().numpy(), P.kivi_dequant_gpu_state(cache, "k", B, H, N, kpc), rtol=1e-6,
                               atol=1e-6)
    np.testing.assert_allclose(vh.cpu().numpy(), P.kivi_dequant_gpu_state(cache, "v", B, H, N, not vpt),
                               rtol=1e-6, atol=1e-6)


def test_kivi_capacity_error():
    B, H = 1, 1
    _, k, v = _inputs(B, H, 64, seed=1)
    ctx = tq.Context(128, 2, "KIVI", 0)
    cache = tq.Cache(ctx, B, H, 32)
    lens = torch.zeros((B,), dtype=torch.int32, device=DEV)
    tq.tq_append_quantize(ctx.handle, cache, k.to(DEV), v.to(DEV), lens)
    assert tq.tq_get_device_error(ctx.handle) == tq.TQ_ERR_CAPACITY


def _tie_groups(n_groups, seed):
    """fp32 rows of 32 values whose range makes (max - min) / 3 an exact fp16 midpoint (a tie
    of the step's rounding), lands just beside one, or is tiny / huge, mixed with ordinary
    groups: the step must come out as fp16 of the fp64 quotient in every case."""
    g = np.random.default_rng(seed)
    rows = []
    for i in range(n_groups):
        kind = i % 6
        k, e = int(g.integers(1024, 2048)), int(g.integers(-12, 10))
        m = (k + 0.5) * 2.0 ** (e - 10)  # an fp16 midpoint
        lo = np.float32(g.standard_normal() * 2.0 ** e)
        if kind == 0:
            rng_ = 3.0 * m
        elif kind == 1:
            rng_ = 3.0 * m * (1 + 2.0 ** -21)
        elif kind == 2:
            rng_ = 3.0 * m * (1 - 2.0 ** -21)
        elif kind == 3:
            rng_ = 3.0 * 2.0 ** -20 * float(g.uniform(1, 2))  # a quotient below the normal fp16 range
        elif kind == 4:
            rng_ = 3.0 * 70000.0  # a quotient above the largest fp16
        else:
            rng_ = float(np.exp(g.normal()))
        hi = np.float32(np.float64(lo) + rng_)
        row = lo + (hi - lo) * g.uniform(0, 1, 32).astype(np.float32)
        row[0], row[1] = lo, hi
        rows.append(row.astype(np.float32))
    return np.stack(rows)


def test_kivi_step_rounding_ties_match_the_fp64_quotient():
    # V per token: each token is four groups of 32 channels; 800 groups in 200 tokens
    B, H, N = 1, 1, 200 + 128
    x = _tie_groups(4 * N, seed=4).reshape(1, 1, N, 128)
    k = torch.from_numpy(np.random.default_rng(1).standard_normal((B, H, N, 128)).astype(np.float32))
    v = torch.from_numpy(x)
    ctx = tq.Context(128, 2, "KIVI", 0, k_per_channel=True, v_per_token=True)
    cache = tq.Cache(ctx, B, H, 352)
    _fill(ctx, cache, k, v, [N])
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    _check_tensor(cache, "v", v, False, B, H, N)
    # and per channel: the same values laid along tokens (groups of 32 tokens per channel)
    xt = _tie_groups(128 * 10, seed=5).reshape(128, 10, 32).transpose(1, 2, 0).reshape(1, 1, 320, 128)
    N2 = 320 + 128
    k2 = np.concatenate([xt, np.random.default_rng(2).standard_normal((1, 1, 128, 128)).astype(np.float32)], axis=2)
    ctx2 = tq.Context(128, 2, "KIVI", 0, k_per_channel=True, v_per_token=True)
    cache2 = tq.Cache(ctx2, B, H, 480)
    _fill(ctx2, cache2, torch.from_numpy(np.ascontiguousarray(k2)), torch.from_numpy(np.ascontiguousarray(k2)), [N2])
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx2.handle) == 0
    _check_tensor(cache2, "k", torch.from_numpy(np.ascontiguousarray(k2)), True, B, H, N2)
