"""GPU parity of the decode step (tq_decode_step: append one token per sequence,
then attend over the sequence including it) against the two calls it stands
for and against the CPU oracle, through the C ABI."""

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


def _prefilled(scheme, n, B, Hkv, G, fill, cap, dtype, seed):
    """A context, a cache whose first `fill` slots of every sequence hold quantised
    tokens, and a step's inputs (queries, new keys and values)."""
    w = wl.Workload(96, "test", B, Hkv * G, Hkv, fill, dtype, scheme, n, key_scale_sigma=1.0)
    q, k, v = wl.generate(w, "cpu", seed=seed)
    ctx = tq.Context(128, n, scheme, 300 + seed)
    cache = tq.Cache(ctx, B, Hkv, cap)
    tq.tq_append_quantize(ctx.handle, cache, k.to(DEV), v.to(DEV), torch.zeros(B, dtype=torch.int32, device=DEV))
    qs, ks, vs = wl.step_token(w, seed, "cpu", data_seed=seed)
    ks[0, 0, 0] = 0  # a zero vector among the new tokens
    return ctx, cache, qs, ks, vs


def _clone(ctx, cache):
    c = tq.Cache(ctx, cache.batch, cache.heads_kv, cache.capacity)
    for name, t in cache.tensors.items():
        c.tensors[name].copy_(t)
    return c


def _two_calls(ctx, cache, q, k, v, lens):
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    tq.tq_append_quantize(ctx.handle, cache, k.to(DEV).contiguous(), v.to(DEV).contiguous(), seq)
    seq1 = torch.tensor([min(max(x + 1, 0), cache.capacity) for x in lens], dtype=torch.int32, device=DEV)
    return tq.tq_decode_attention(ctx.handle, cache, q.to(DEV), seq1, max_len=cache.capacity)


CASES = [("KQV", 4, 1), ("KQV", 3, 1), ("KQV", 2, 1), ("KV", 4, 1), ("KV", 2, 1),
         ("QKQV", 3, 1), ("KQV", 4, 2)]  # the last two: the general (append, then decode) path


@pytest.mark.parametrize("scheme,n,G", CASES)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_step_equals_append_then_decode(scheme, n, G, dtype):
    # ragged lengths: an empty sequence, odd and even slots (the value pair row is shared
    # with a token already stored), a block end, a tile end, a long head
    lens = [0, 77, 300, 63, 15, 1200]
    B, Hkv = len(lens), 3
    ctx, ref, q, k, v = _prefilled(scheme, n, B, Hkv, G, 1300, 1301, dtype, seed=5 + n)
    fused = _clone(ctx, ref)
    want = _two_calls(ctx, ref, q, k, v, lens)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    got = tq.tq_decode_step(ctx.handle, fused, q.to(DEV), k.to(DEV), v.to(DEV), seq, max_len=1301)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    assert torch.equal(seq.cpu(), torch.tensor(lens, dtype=torch.int32))  # lengths are the caller's
    for name, t in ref.tensors.items():
        assert torch.equal(t, fused.tensors[name]), name
    diff = (got - want).abs().max().item()
    assert torch.equal(got, want), diff


@pytest.mark.parametrize("scheme,n", [("KQV", 4), ("KQV", 2), ("KV", 3)])
def test_step_matches_the_oracle(scheme, n):
    lens = [0, 1, 64, 65, 700, 333, 128]
    B, H = len(lens), 4
    ctx, cache, q, k, v = _prefilled(scheme, n, B, H, 1, 700, 720, torch.bfloat16, seed=17)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = tq.tq_decode_step(ctx.handle, cache, q.to(DEV), k.to(DEV), v.to(DEV), seq, max_len=720)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    params = otq.make_params(128, n, scheme, 300 + 17)
    # the new tokens' records against the oracle's encoding (boundary-band rule)
    for which, x, role in (("k", k, params.roles()[0]), ("v", v, params.roles()[1])):
        ora = otq.encode(x.float().numpy().reshape(-1, 128), role, params)
        enc, packed, signs = P.gpu_encoded(cache, role, which, B, H, cache.capacity)
        rows = np.array([(b * H + h) * cache.capacity + lens[b] for b in range(B) for h in range(H)])
        gidx = enc.idx[rows]
        rep = P.BandReport()
        mism = P.compare_codes(gidx, ora, ocb.lloyd_max(128, role.bits).bounds32, rep)
        assert rep.ok_out_of_band(), f"{which} codes: {rep}"
        # the step appends through the warp-per-vector encoder: a direct sum of squares
        np.testing.assert_allclose(enc.norm[rows], ora.norm, rtol=P.norm_rtol(False), atol=0)
        if role.qjl:
            srep = P.BandReport()
            P.compare_signs(enc.signs[rows], ora, srep, skip_rows=mism.any(axis=1))
            assert srep.ok_out_of_band(), f"{which} signs: {srep}"
            np.testing.assert_allclose(enc.rnorm[rows], ora.rnorm, rtol=1e-5, atol=1e-7)
    # attention over the lengths plus one, from the GPU's own codes
    lens1 = [x + 1 for x in lens]
    want = P.oracle_decode_from_cache(cache, params, q.float().numpy(), lens1, B, H, H)
    got = out.cpu().numpy()
    for b in range(B):
        for h in range(H):
            assert P.rel_l2(got[b, h], want[b, h]) < 1e-3, (b, h)


@pytest.mark.parametrize("B,lens_of,cap", [(96, lambda b: b % 6, 16), (128, lambda b: 250 + 9 * (b % 7), 320)],
                         ids=["one-tile-heads", "five-tile-heads"])
def test_step_many_heads_per_cta(B, lens_of, cap):
    # B x 8 heads: each persistent CTA appends for several heads. With one-tile heads every
    # last tile is among the first 16 tiles a CTA copies (appended before its ring prologue);
    # with ~34 tiles per CTA some are copied later (appended while the prologue streams)
    H = 8
    lens = [lens_of(b) for b in range(B)]
    ctx, ref, q, k, v = _prefilled("KQV", 4, B, H, 1, cap, cap, torch.bfloat16, seed=23)
    fused = _clone(ctx, ref)
    want = _two_calls(ctx, ref, q, k, v, lens)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    got = tq.tq_decode_step(ctx.handle, fused, q.to(DEV), k.to(DEV), v.to(DEV), seq, max_len=cap)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    for name, t in ref.tensors.items():
        assert torch.equal(t, fused.tensors[name]), name
    assert torch.equal(got, want)


def test_step_heads_spanning_several_ctas():
    # 2 x 2 heads of ~80 tiles: more tiles than CTAs, the last tile's owner appends
    lens = [5000, 4999]
    ctx, ref, q, k, v = _prefilled("KQV", 4, 2, 2, 1, 5001, 5001, torch.bfloat16, seed=29)
    fused = _clone(ctx, ref)
    want = _two_calls(ctx, ref, q, k, v, lens)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    got = tq.tq_decode_step(ctx.handle, fused, q.to(DEV), k.to(DEV), v.to(DEV), seq, max_len=5001)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    for name, t in ref.tensors.items():
        assert torch.equal(t, fused.tensors[name]), name
    assert torch.equal(got, want)


def test_step_full_sequence_reports_capacity():
    # sequence 1 is full: nothing is appended there, the error word is set, and it is
    # attended over its whole capacity; the others step normally
    lens = [10, 32, 31]
    B, H = len(lens), 2
    ctx, ref, q, k, v = _prefilled("KQV", 3, B, H, 1, 32, 32, torch.float32, seed=37)
    fused = _clone(ctx, ref)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    got = tq.tq_decode_step(ctx.handle, fused, q.to(DEV), k.to(DEV), v.to(DEV), seq, max_len=32)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == tq.TQ_ERR_CAPACITY
    want = _two_calls(ctx, ref, q, k, v, lens)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == tq.TQ_ERR_CAPACITY
    for name, t in ref.tensors.items():
        assert torch.equal(t, fused.tensors[name]), name
    assert torch.equal(got, want)


def test_step_argument_errors():
    ctx = tq.Context(128, 4, "KQV", 1)
    cache = tq.Cache(ctx, 1, 2, 32)
    q = torch.zeros((1, 2, 128), device=DEV)
    kv = torch.zeros((1, 2, 128), device=DEV)
    seq = torch.tensor([4], dtype=torch.int32, device=DEV)
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_step(ctx.handle, cache, q, kv, kv, seq, max_len=64)  # max_len > capacity
    assert e.value.status == tq.TQ_ERR_ARG
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_step(ctx.handle, cache, q, kv, kv, seq, max_len=8, workspace=ws)
    assert e.value.status == tq.TQ_ERR_WORKSPACE



@pytest.mark.parametrize("k_per_channel,v_per_token", [(True, True), (False, False)])
@pytest.mark.parametrize("L", [100, 159, 191])
def test_step_kivi_equals_append_then_decode(k_per_channel, v_per_token, L):
    # KIVI takes the general path (a length kernel, the append, the decode). At L = 159 the
    # step's token brings the window to 160 tokens, so the append also quantises a group out
    # of the window
    B, H = 3, 2
    w = wl.WORKLOADS[5]
    q, k, v = wl.generate(w, "cpu", seed=41, batch=B, heads_kv=H, seq=L + 1)
    ctx = tq.Context(128, 2, "KIVI", 9, k_per_channel=k_per_channel, v_per_token=v_per_token)
    ref = tq.Cache(ctx, B, H, 192)
    tq.tq_append_quantize(ctx.handle, ref, k[:, :, :L].contiguous().to(DEV), v[:, :, :L].contiguous().to(DEV),
                          torch.zeros(B, dtype=torch.int32, device=DEV))
    kn, vn = k[:, :, L:].contiguous(), v[:, :, L:].contiguous()
    fused = _clone(ctx, ref)
    want = _two_calls(ctx, ref, q, kn, vn, [L] * B)
    seq = torch.full((B,), L, dtype=torch.int32, device=DEV)
    got = tq.tq_decode_step(ctx.handle, fused, q.to(DEV), kn.to(DEV), vn.to(DEV), seq, max_len=192)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    for name, t in ref.tensors.items():
        assert torch.equal(t, fused.tensors[name]), name
    assert torch.equal(got, want)
