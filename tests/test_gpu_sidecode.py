"""GPU parity of the rank-r key side codes ([HeadQ] section 3: a logit correction in a
basis of calibration queries; [KVQuant++] "Core innovation 4": a low-rank correction of
the key residual) against the oracle (oracle/sidecode.py), through the C ABI: base codes
and side codes on every append path, decode attention over the corrected keys,
dequantisation, the decode step, and the quality each correction buys."""

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import codebook as ocb
from oracle import sidecode as sc
from oracle import turboquant as otq
from quantised_kv_cache_gb300 import tq
from quantised_kv_cache_gb300 import workloads as wl

import parity as P

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantised_kv_cache_gb300 import build
    build.build()


def _bases(H, rank, seed):
    g = np.random.default_rng(seed)
    return np.stack([np.linalg.qr(g.standard_normal((128, rank)))[0] for _ in range(H)]).astype(np.float32)


def _side(cache, B, H, N, rank):
    cap = cache.struct.capacity
    z = cache.plane("k_side").cpu().numpy().view(np.float16).reshape(B, H, cap, rank)
    return z[:, :, :N].astype(np.float64)


def _check_side_codes(cache, params, k, U, B, H, N, rank):
    """GPU side codes against U^T (k - k_hat) in fp64, k_hat rebuilt from the GPU's base codes:
    equal up to the float16 rounding of the stored value and the float32 arithmetic."""
    rk = params.roles()[0]
    enc, _, _ = P.gpu_encoded(cache, rk, "k", B, H, N)
    kh = otq.decode(enc, params).reshape(B, H, N, 128)
    e = k.double().numpy() - kh
    want = np.einsum("bhnd,hdr->bhnr", e, U.astype(np.float64))
    got = _side(cache, B, H, N, rank)
    tol = np.abs(want) * 2.0 ** -11 + 1e-5 * np.linalg.norm(e, axis=-1, keepdims=True)
    assert np.all(np.abs(got - want) <= tol), float(np.max(np.abs(got - want) - tol))


@pytest.mark.parametrize("scheme,n", [("KQV", 4), ("KQV", 2), ("KV", 3)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", [(2, 3, 400), (2, 4, 1111)], ids=["few", "bulk"])
@pytest.mark.parametrize("rank", [4, 8])
def test_side_codes_on_every_append_path(scheme, n, dtype, shape, rank):
    B, H, N = shape
    w = wl.Workload(87, "side", B, H, H, N, dtype, scheme, n, key_scale_sigma=1.0)
    _, k, v = wl.generate(w, "cpu", seed=5 + rank)
    U = _bases(H, rank, 1)
    ctx = tq.Context(128, n, scheme, 71)
    tq.tq_set_side_basis(ctx.handle, U)
    cache = tq.Cache(ctx, B, H, N)
    assert cache.sizes.plane_bytes[8] == 2 * rank
    tq.tq_append_quantize(ctx.handle, cache, k.to(DEV), v.to(DEV), torch.zeros(B, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    params = otq.make_params(128, n, scheme, 71)
    # the base codes are those of a context without side codes
    rk = params.roles()[0]
    ora = otq.encode(k.float().numpy().reshape(-1, 128), rk, params)
    gpu, _, _ = P.gpu_encoded(cache, rk, "k", B, H, N)
    rep = P.BandReport()
    P.compare_codes(gpu.idx, ora, ocb.lloyd_max(128, rk.bits).bounds32, rep)
    assert rep.ok(), rep
    _check_side_codes(cache, params, k, U, B, H, N, rank)


@pytest.mark.parametrize("scheme,n,G", [("KQV", 4, 1), ("KQV", 2, 4), ("KV", 2, 2)])
def test_side_corrected_decode_and_dequantize_match_the_oracle(scheme, n, G):
    lens = [301, 67, 900]
    B, Hkv = len(lens), 2
    Hq, N, rank = G * Hkv, max(lens), 4
    w = wl.Workload(86, "side", B, Hq, Hkv, N, torch.bfloat16, scheme, n, key_scale_sigma=1.0)
    q, k, v = wl.generate(w, "cpu", seed=9)
    U = _bases(Hkv, rank, 2)
    ctx = tq.Context(128, n, scheme, 72)
    tq.tq_set_side_basis(ctx.handle, U)
    cache = tq.Cache(ctx, B, Hkv, N)
    tq.tq_append_quantize(ctx.handle, cache, k.to(DEV), v.to(DEV), torch.zeros(B, dtype=torch.int32, device=DEV))
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = tq.tq_decode_attention(ctx.handle, cache, q.to(DEV), seq, max_len=N).cpu().numpy()
    kh_gpu, _ = tq.tq_dequantize(ctx.handle, cache, 0, N)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    params = otq.make_params(128, n, scheme, 72)
    rk, rv = params.roles()
    ek, _, _ = P.gpu_encoded(cache, rk, "k", B, Hkv, N)
    ev, _, _ = P.gpu_encoded(cache, rv, "v", B, Hkv, N)
    z = _side(cache, B, Hkv, N, rank)
    Kb = otq.decode(ek, params).reshape(B, Hkv, N, 128)
    Kc = Kb + np.einsum("bhnr,hdr->bhnd", z, U.astype(np.float64))
    Vh = otq.decode(ev, params).reshape(B, Hkv, N, 128)
    assert P.rel_l2(kh_gpu.cpu().numpy(), Kc) < 1e-5
    want = oatt.attend_gqa(q.double().numpy(), Kc, Vh, lengths=lens)
    for b in range(B):
        for h in range(Hq):
            assert P.rel_l2(out[b, h], want[b, h]) < 1e-3, (b, h)


def test_side_codes_decode_step_equals_append_then_decode():
    lens = [0, 15, 300, 1023]
    B, H, cap = len(lens), 3, 1040
    w = wl.Workload(85, "side", B, H, H, 1024, torch.bfloat16, "KQV", 3, key_scale_sigma=1.0)
    q, k, v = wl.generate(w, "cpu", seed=12)
    qs, ks, vs = wl.step_token(w, 1, "cpu", data_seed=12, batch=B, heads_kv=H)
    ctx = tq.Context(128, 3, "KQV", 73)
    tq.tq_set_side_basis(ctx.handle, _bases(H, 8, 3))
    one, two = tq.Cache(ctx, B, H, cap), tq.Cache(ctx, B, H, cap)
    for c in (one, two):
        tq.tq_append_quantize(ctx.handle, c, k.to(DEV), v.to(DEV), torch.zeros(B, dtype=torch.int32, device=DEV))
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    got = tq.tq_decode_step(ctx.handle, one, qs.to(DEV), ks.to(DEV), vs.to(DEV), seq, max_len=cap)
    tq.tq_append_quantize(ctx.handle, two, ks.to(DEV).contiguous(), vs.to(DEV).contiguous(), seq)
    seq1 = torch.tensor([x + 1 for x in lens], dtype=torch.int32, device=DEV)
    want = tq.tq_decode_attention(ctx.handle, two, qs.to(DEV), seq1, max_len=cap)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    assert torch.equal(one.tensors["records"], two.tensors["records"])
    assert torch.equal(got, want)


def test_side_basis_errors():
    ctx = tq.Context(128, 3, "QKQV", 1)
    with pytest.raises(tq.TQError) as e:
        tq.tq_set_side_basis(ctx.handle, _bases(2, 4, 0))
    assert e.value.status == tq.TQ_ERR_STATE  # sketched keys
    ctx = tq.Context(128, 4, "KQV", 1)
    bad = _bases(2, 4, 0) * 1.1
    with pytest.raises(tq.TQError) as e:
        tq.tq_set_side_basis(ctx.handle, bad)
    assert e.value.status == tq.TQ_ERR_ARG  # columns not orthonormal
    tq.tq_set_side_basis(ctx.handle, _bases(2, 4, 0))
    cache = tq.Cache(ctx, 1, 3, 32)  # three KV heads against a two-head basis
    with pytest.raises(tq.TQError) as e:
        tq.tq_append_quantize(ctx.handle, cache, torch.zeros((1, 3, 1, 128), device=DEV),
                              torch.zeros((1, 3, 1, 128), device=DEV), torch.zeros(1, dtype=torch.int32, device=DEV))
    assert e.value.status == tq.TQ_ERR_ARG
    with pytest.raises(tq.TQError) as e:
        tq.tq_set_rotation(ctx.handle, "dense")  # the rotation is chosen before the basis
    assert e.value.status == tq.TQ_ERR_STATE
