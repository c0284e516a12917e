"""GPU parity of the dense SO(d) rotation ([KVQuant++] "Rotation-invariance guarantee",
"Rate-distortion performance": a random QR rotation in place of the Hadamard transform)
against the CPU oracle (oracle/rotation.py), through the C ABI: codes and signs under
the band rule on every append path, dequantisation, decode attention (one query head
and GQA groups), the decode step, and the reconstruction error of both rotations."""

import numpy as np
import pytest
import torch

from oracle import codebook as ocb
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


def _ctx(n, scheme, seed):
    return tq.Context(128, n, scheme, seed, rotation="dense")


def test_context_rotation_matches_the_oracle():
    from oracle import rotation as orot
    M = tq.tq_draw_rotation(42, 128)
    assert np.max(np.abs(M - orot.dense_rotation(42, 128))) < 1e-7
    ctx = tq.Context(128, 2, "KIVI", 1)
    with pytest.raises(tq.TQError) as e:
        tq.tq_set_rotation(ctx.handle, "dense")
    assert e.value.status == tq.TQ_ERR_STATE


@pytest.mark.parametrize("scheme,n", [("KQV", 4), ("KQV", 3), ("KQV", 2), ("QKQV", 4), ("QKQV", 2)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", [(2, 3, 1300), (2, 4, 1111)], ids=["few", "bulk"])
def test_dense_append_codes_match_the_oracle(scheme, n, dtype, shape):
    # "few": the warp-per-vector launch (dense matrix-vector product by shuffles);
    # "bulk": the tensor-core kernel (fp16 hi / lo passes against sqrt(d) M hi / lo)
    B, H, N = shape
    w = wl.Workload(91, "rotation", B, H, H, N, dtype, scheme, n, key_scale_sigma=1.0, outlier_channels=2,
                    outlier_factor=10.0)
    _, k, v = wl.generate(w, "cpu", seed=13 + n)
    k[0, 1, 5] = 0
    ctx = _ctx(n, scheme, 77)
    cache = tq.Cache(ctx, B, H, N)
    tq.tq_append_quantize(ctx.handle, cache, k.to(DEV), v.to(DEV), torch.zeros(B, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    params = otq.make_params(128, n, scheme, 77, rotation="dense")
    for which, x, role in (("k", k, params.roles()[0]), ("v", v, params.roles()[1])):
        ora = otq.encode(x.float().numpy().reshape(-1, 128), role, params)
        gpu, packed, _ = P.gpu_encoded(cache, role, which, B, H, N)
        rep = P.BandReport()
        mism = P.compare_codes(gpu.idx, ora, ocb.lloyd_max(128, role.bits).bounds32, rep)
        assert rep.ok(), f"{which} codes: {rep}"
        # direct sums of squares on both paths (the dense rotation never takes the bulk
        # bf16 kernel, whose norm comes off the rotation)
        np.testing.assert_allclose(gpu.norm, ora.norm, rtol=P.norm_rtol(False), atol=0)
        if role.qjl:
            srep = P.BandReport()
            P.compare_signs(gpu.signs, ora, srep, skip_rows=mism.any(axis=1))
            assert srep.ok(), f"{which} signs: {srep}"
            np.testing.assert_allclose(gpu.rnorm, ora.rnorm, rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("scheme,n", [("KQV", 4), ("QKQV", 3)])
def test_dense_dequantize_matches_the_oracle(scheme, n):
    B, H, N = 2, 2, 40
    w = wl.Workload(90, "rotation", B, H, H, N, torch.float32, scheme, n)
    _, k, v = wl.generate(w, "cpu", seed=3)
    ctx = _ctx(n, scheme, 5)
    cache = tq.Cache(ctx, B, H, N)
    tq.tq_append_quantize(ctx.handle, cache, k.to(DEV), v.to(DEV), torch.zeros(B, dtype=torch.int32, device=DEV))
    kh, vh = tq.tq_dequantize(ctx.handle, cache, 0, N)
    params = otq.make_params(128, n, scheme, 5, rotation="dense")
    for which, got, role in (("k", kh, params.roles()[0]), ("v", vh, params.roles()[1])):
        enc, _, _ = P.gpu_encoded(cache, role, which, B, H, N)
        want = otq.decode(enc, params).reshape(B, H, N, 128)
        assert P.rel_l2(got.cpu().numpy(), want) < 1e-5


@pytest.mark.parametrize("scheme,n,G", [("KQV", 4, 1), ("KQV", 3, 4), ("QKQV", 3, 2), ("KQV", 2, 8)])
def test_dense_decode_attention_matches_the_oracle(scheme, n, G):
    lens = [301, 67, 1500]
    B, Hkv = len(lens), 2
    Hq = G * Hkv
    N = max(lens)
    w = wl.Workload(89, "rotation", B, Hq, Hkv, N, torch.bfloat16, scheme, n, key_scale_sigma=1.0)
    q, k, v = wl.generate(w, "cpu", seed=31 + G)
    ctx = _ctx(n, scheme, 55)
    cache = tq.Cache(ctx, B, Hkv, N)
    tq.tq_append_quantize(ctx.handle, cache, k.to(DEV), v.to(DEV), torch.zeros(B, dtype=torch.int32, device=DEV))
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = tq.tq_decode_attention(ctx.handle, cache, q.to(DEV), seq, max_len=N)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    want = P.oracle_decode_from_cache(cache, otq.make_params(128, n, scheme, 55, rotation="dense"),
                                      q.float().numpy(), lens, B, Hkv, Hq)
    got = out.cpu().numpy()
    for b in range(B):
        for h in range(Hq):
            assert P.rel_l2(got[b, h], want[b, h]) < 1e-3, (b, h)


def test_dense_decode_step_equals_append_then_decode():
    # the step runs as separate append, query preparation and decode kernels for a dense
    # rotation: it must equal the two calls bit for bit
    lens = [0, 15, 300, 1023]
    B, H, cap = len(lens), 3, 1040
    w = wl.Workload(88, "rotation", B, H, H, 1024, torch.bfloat16, "KQV", 4, key_scale_sigma=1.0)
    q, k, v = wl.generate(w, "cpu", seed=12)
    qs, ks, vs = wl.step_token(w, 1, "cpu", data_seed=12, batch=B, heads_kv=H)
    ctx = _ctx(4, "KQV", 64)
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
