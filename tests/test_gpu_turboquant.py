"""GPU parity of the TurboQuant-style path (append-quantise, dequantise, decode
attention) against the CPU oracle, called through the C ABI."""

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


def _inputs(B, H, N, dtype, seed, dist="gauss", scale_sigma=0.0, outliers=0):
    w = wl.Workload(99, "test", B, H, H, N, dtype, "KQV", 4, key_dist=dist, key_scale_sigma=scale_sigma,
                    outlier_channels=outliers, outlier_factor=10.0)
    return wl.generate(w, "cpu", seed=seed)


def _append(ctx, cache, k, v, start):
    B = k.shape[0]
    lens = torch.full((B,), start, dtype=torch.int32, device=DEV)
    tq.tq_append_quantize(ctx.handle, cache, k.to(DEV), v.to(DEV), lens)


@pytest.mark.parametrize("scheme,n", [("KQV", 4), ("KQV", 3), ("KQV", 2), ("QKQV", 4), ("QKQV", 2),
                                      ("KV", 4), ("KV", 3), ("KV", 2)])
def test_context_parameters_match_the_oracle(scheme, n):
    ctx = tq.Context(128, n, scheme, 42)
    p = tq.tq_export_params(ctx.handle)
    rk, rv = otq.scheme_roles(scheme, n)
    assert (p.k_bits, p.v_bits) == (rk.bits, rv.bits)
    np.testing.assert_array_equal(p.k_centroids, ocb.lloyd_max(128, rk.bits).centroids32)
    np.testing.assert_array_equal(p.k_bounds, ocb.lloyd_max(128, rk.bits).bounds32)
    np.testing.assert_array_equal(p.v_centroids, ocb.lloyd_max(128, rv.bits).centroids32)
    op = otq.make_params(128, n, scheme, 42)
    np.testing.assert_array_equal(p.diag, op.D)
    np.testing.assert_array_equal(p.sketch, op.S)


@pytest.mark.parametrize("scheme,n", [("KQV", 4), ("KQV", 3), ("KQV", 2), ("QKQV", 4), ("QKQV", 3),
                                      ("QKQV", 2), ("KV", 4), ("KV", 2)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(2, 3, 1300), (2, 4, 1111)], ids=["few", "bulk"])
def test_append_codes_bit_exact(scheme, n, dtype, shape):
    # "few": 7800 vectors per tensor, the warp-per-vector single-launch path (at most 8192);
    # "bulk": 8888, above that path's limit, with a ragged last tile. Each call compares about
    # 10^6 codes per tensor, so that the in-band mismatch fraction (bounded by 1e-5 of the
    # codes compared) is a property of a population large enough for one legitimate in-band
    # flip (expected ~2e-6 per code) not to exceed it by itself
    B, H, N = shape
    q, k, v = _inputs(B, H, N, dtype, seed=7 + n, scale_sigma=1.0, outliers=2)
    k[0, 1, 5] = 0  # a zero vector
    v[1, 2, 9] = 0
    ctx = tq.Context(128, n, scheme, 123)
    cache = tq.Cache(ctx, B, H, N + 5)
    _append(ctx, cache, k, v, 0)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    params = otq.make_params(128, n, scheme, 123)
    for which, x, role in (("k", k, params.roles()[0]), ("v", v, params.roles()[1])):
        xr = x.float().numpy().reshape(-1, 128)
        ora = otq.encode(xr, role, params)
        gpu, packed, signs = P.gpu_encoded(cache, role, which, B, H, N)
        rep = P.BandReport()
        code_mism = P.compare_codes(gpu.idx, ora, ocb.lloyd_max(128, role.bits).bounds32, rep)
        assert rep.ok(), f"{which} codes: {rep}"
        # bytes identical wherever the codes are
        same = ~code_mism.any(axis=1)
        np.testing.assert_array_equal(packed[same], otq.pack_codes(ora.idx[same], role.bits))
        rtol = P.norm_rtol(P.bulk_bf16_path(dtype, B * H * N, role))
        np.testing.assert_allclose(gpu.norm, ora.norm, rtol=rtol, atol=0)
        if role.qjl:
            srep = P.BandReport()
            P.compare_signs(gpu.signs, ora, srep, skip_rows=code_mism.any(axis=1))
            assert srep.ok(), f"{which} signs: {srep}"
            np.testing.assert_allclose(gpu.rnorm, ora.rnorm, rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("scheme,n", [("KQV", 4), ("QKQV", 3), ("KV", 2)])
def test_cache_sizes_describe_the_blocked_layout(scheme, n):
    ctx = tq.Context(128, n, scheme, 1)
    s = tq.tq_cache_sizes_get(ctx.handle, 3, 2, 50)
    rk, rv = otq.scheme_roles(scheme, n)
    tok = [rk.bits * 16, 4, 16 if rk.qjl else 0, 4 if rk.qjl else 0,
           rv.bits * 16, 4, 16 if rv.qjl else 0, 4 if rv.qjl else 0,
           0]  # the keys' side-code plane, empty without tq_set_side_basis
    assert list(s.plane_bytes) == tok
    assert list(s.plane_offset) == [16 * sum(tok[:p]) for p in range(9)]
    assert s.block_bytes == 16 * sum(tok) == 16 * s.record_bytes
    assert s.records == 3 * 2 * 4 * s.block_bytes  # ceil(50 / 16) = 4 blocks per sequence-head
    # the sizing calls under their first-specified names give the same answers
    a = tq.tq_cache_bytes(ctx.handle, 3, 2, 50)
    assert bytes(a) == bytes(s)
    for args in [(3, 2, 2, 50, 0), (3, 4, 2, 50, 5), (300, 2, 2, 40, 0)]:
        assert tq.tq_workspace_bytes(ctx.handle, *args) == tq.tq_workspace_size(ctx.handle, *args)


def test_a_token_lands_where_the_layout_says():
    # one token of sequence-head (b=1, h=0) at slot 37 of a capacity-50 cache: block
    # (1 * 2 + 0) * 4 + 37 // 16 = 10, entry 37 % 16 = 5 of each plane
    B, H, cap, t = 2, 2, 50, 37
    ctx = tq.Context(128, 4, "KQV", 3)
    cache = tq.Cache(ctx, B, H, cap)
    g = torch.Generator().manual_seed(4)
    k = torch.randn(B, H, 1, 128, generator=g)
    v = torch.randn(B, H, 1, 128, generator=g)
    tq.tq_append_quantize(ctx.handle, cache, k.to(DEV), v.to(DEV), torch.full((B,), t, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    s = cache.sizes
    raw = cache.tensors["records"].cpu().numpy()
    blk = raw[10 * s.block_bytes:11 * s.block_bytes]
    knorm = blk[s.plane_offset[1] + 5 * 4:s.plane_offset[1] + 6 * 4].view(np.float32)[0]
    vnorm = blk[s.plane_offset[5] + 5 * 4:s.plane_offset[5] + 6 * 4].view(np.float32)[0]
    np.testing.assert_allclose(knorm, float(k[1, 0, 0].double().norm()), rtol=P.norm_rtol(False))
    np.testing.assert_allclose(vnorm, float(v[1, 0, 0].double().norm()), rtol=P.norm_rtol(False))
    # every other entry of the cache is still zero
    raw_other = raw.copy()
    raw_other[10 * s.block_bytes:11 * s.block_bytes] = 0
    for b in range(B):
        for h in range(H):
            if (b, h) != (1, 0):
                blk2 = (b * H + h) * 4 + 2
                raw_other[blk2 * s.block_bytes:(blk2 + 1) * s.block_bytes] = 0
    assert not raw_other.any()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_appends_that_split_a_token_pair_keep_both_halves(dtype):
    # value codes of tokens 2j and 2j+1 share one field per coordinate: an append starting at
    # an odd slot (here 601) must merge its half without touching the earlier token's half.
    # Both calls are above the few-vector limit (the bulk kernels), as is the one-call reference.
    B, H, N, cut = 2, 8, 1200, 601
    _, k, v = _inputs(B, H, N, dtype, seed=21)
    ctx = tq.Context(128, 4, "KQV", 17)
    one = tq.Cache(ctx, B, H, N)
    _append(ctx, one, k, v, 0)
    two = tq.Cache(ctx, B, H, N)
    _append(ctx, two, k[:, :, :cut].contiguous(), v[:, :, :cut].contiguous(), 0)
    _append(ctx, two, k[:, :, cut:].contiguous(), v[:, :, cut:].contiguous(), cut)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    assert torch.equal(one.tensors["records"], two.tensors["records"])


def test_append_writes_only_its_slots_and_reports_capacity():
    B, H = 2, 2
    _, k, v = _inputs(B, H, 10, torch.float32, seed=3)
    ctx = tq.Context(128, 4, "KQV", 5)
    cache = tq.Cache(ctx, B, H, 16)
    lens = torch.tensor([3, 6], dtype=torch.int32, device=DEV)
    tq.tq_append_quantize(ctx.handle, cache, k[:, :, :4].contiguous().to(DEV), v[:, :, :4].contiguous().to(DEV),
                          lens)
    norms = cache.plane("k_norm").cpu().numpy().view(np.float32).reshape(B, H, 16)
    assert np.all(norms[0, :, 3:7] > 0) and np.all(norms[0, :, :3] == 0) and np.all(norms[0, :, 7:] == 0)
    assert np.all(norms[1, :, 6:10] > 0) and np.all(norms[1, :, :6] == 0) and np.all(norms[1, :, 10:] == 0)
    assert tq.tq_get_device_error(ctx.handle) == 0
    # one sequence past capacity: its writes are skipped, the error word is set, the other lands
    before = cache.plane("k_codes").clone()
    lens = torch.tensor([14, 0], dtype=torch.int32, device=DEV)
    tq.tq_append_quantize(ctx.handle, cache, k[:, :, :4].contiguous().to(DEV), v[:, :, :4].contiguous().to(DEV),
                          lens)
    assert tq.tq_get_device_error(ctx.handle) == tq.TQ_ERR_CAPACITY
    assert tq.tq_get_device_error(ctx.handle) == 0  # cleared on read
    after = cache.plane("k_codes").view(B, H, 16, 64).cpu()
    b4 = before.view(B, H, 16, 64).cpu()
    assert torch.equal(after[0, :, 14:], b4[0, :, 14:])  # slots 14, 15 untouched by the rejected append
    assert torch.equal(after[0, :, :14], b4[0, :, :14])


def test_incremental_appends_equal_one_bulk_append():
    B, H, N = 1, 2, 40
    _, k, v = _inputs(B, H, N, torch.bfloat16, seed=11)
    ctx = tq.Context(128, 4, "KQV", 9)
    bulk = tq.Cache(ctx, B, H, N)
    _append(ctx, bulk, k, v, 0)
    inc = tq.Cache(ctx, B, H, N)
    for t in range(N):
        _append(ctx, inc, k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous(), t)
    for name, tens in bulk.tensors.items():
        assert torch.equal(tens, inc.tensors[name]), name


@pytest.mark.parametrize("scheme,n", [("KQV", 4), ("KQV", 2), ("QKQV", 3), ("KV", 3)])
def test_dequantize_matches_oracle_reconstruction(scheme, n):
    B, H, N = 2, 2, 33
    _, k, v = _inputs(B, H, N, torch.float32, seed=21)
    ctx = tq.Context(128, n, scheme, 77)
    cache = tq.Cache(ctx, B, H, N)
    _append(ctx, cache, k, v, 0)
    kh, vh = tq.tq_dequantize(ctx.handle, cache, 4, N)
    params = otq.make_params(128, n, scheme, 77)
    for which, got, role in (("k", kh, params.roles()[0]), ("v", vh, params.roles()[1])):
        enc, _, _ = P.gpu_encoded(cache, role, which, B, H, N)
        want = otq.decode(enc, params).reshape(B, H, N, 128)[:, :, 4:]
        g = got.cpu().numpy()
        assert P.rel_l2(g, want) < 1e-5


@pytest.mark.parametrize("scheme,n", [("KQV", 4), ("KQV", 3), ("KQV", 2), ("QKQV", 4), ("QKQV", 2),
                                      ("KV", 4), ("KV", 2)])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("splits", [0, 1, 5])
def test_decode_attention_matches_oracle(scheme, n, G, splits):
    B, Hkv = 2, 2
    Hq = Hkv * G
    lens = [301, 67]  # ragged, not tile multiples
    N = max(lens)
    w = wl.Workload(98, "test", B, Hq, Hkv, N, torch.bfloat16, scheme, n, key_scale_sigma=1.0)
    q, k, v = wl.generate(w, "cpu", seed=31 + G)
    ctx = tq.Context(128, n, scheme, 55)
    cache = tq.Cache(ctx, B, Hkv, N + 3)
    _append(ctx, cache, k, v, 0)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = tq.tq_decode_attention(ctx.handle, cache, q.to(DEV), seq, max_len=N, splits=splits)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    want = P.oracle_decode_from_cache(cache, otq.make_params(128, n, scheme, 55), q.float().numpy(), lens, B,
                                      Hkv, Hq)
    for b in range(B):
        for h in range(Hq):
            assert P.rel_l2(got[b, h], want[b, h]) < 1e-3, (b, h, P.rel_l2(got[b, h], want[b, h]))


@pytest.mark.parametrize("N", [1, 2, 9, 33])
def test_decode_short_sequences_and_more_splits_than_tokens(N):
    B, H = 1, 2
    q, k, v = _inputs(B, H, N, torch.float32, seed=N)
    ctx = tq.Context(128, 4, "KQV", 1)
    cache = tq.Cache(ctx, B, H, 64)
    _append(ctx, cache, k, v, 0)
    seq = torch.tensor([N], dtype=torch.int32, device=DEV)
    out = tq.tq_decode_attention(ctx.handle, cache, q.to(DEV), seq, max_len=N, splits=8)
    want = P.oracle_decode_from_cache(cache, otq.make_params(128, 4, "KQV", 1), q.float().numpy(), [N], B, H, H)
    assert P.rel_l2(out.cpu().numpy(), want) < 1e-3
    if N == 1:
        # a single token: the output is that token's reconstructed value (the decode
        # accumulates values on fp16 tensor-core operands, hence the attention bound)
        kh, vh = tq.tq_dequantize(ctx.handle, cache, 0, 1)
        assert P.rel_l2(out.cpu().numpy()[0], vh.cpu().numpy()[0, :, 0]) < 1e-3


def test_decode_argument_errors():
    ctx = tq.Context(128, 4, "KQV", 1)
    cache = tq.Cache(ctx, 1, 2, 32)
    q = torch.zeros((1, 6, 128), device=DEV)
    seq = torch.tensor([4], dtype=torch.int32, device=DEV)
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_attention(ctx.handle, cache, q, seq, max_len=4)  # 6 query heads over 2 kv heads: G = 3
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED
    q = torch.zeros((1, 2, 128), device=DEV)
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_attention(ctx.handle, cache, q, seq, max_len=64)  # max_len > capacity
    assert e.value.status == tq.TQ_ERR_ARG
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_attention(ctx.handle, cache, q, seq, max_len=4, workspace=ws)
    assert e.value.status == tq.TQ_ERR_WORKSPACE


def _decode_case(scheme, n, B, H, lens, seed, cap=None):
    N = max(max(lens), 1)
    w = wl.Workload(97, "test", B, H, H, N, torch.bfloat16, scheme, n, key_scale_sigma=1.0)
    q, k, v = wl.generate(w, "cpu", seed=seed)
    ctx = tq.Context(128, n, scheme, 1000 + seed)
    cache = tq.Cache(ctx, B, H, cap or N)
    _append(ctx, cache, k, v, 0)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = tq.tq_decode_attention(ctx.handle, cache, q.to(DEV), seq, max_len=N)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    return ctx, cache, q, out.cpu().numpy()


@pytest.mark.parametrize("scheme,n", [("KQV", 4), ("QKQV", 3), ("KV", 2)])
def test_decode_ragged_lengths_with_empty_sequences(scheme, n):
    # lengths around the 64-token tile: most of the persistent grid's slices are empty
    lens = [0, 1, 64, 65, 700]
    B, H = len(lens), 3
    ctx, cache, q, got = _decode_case(scheme, n, B, H, lens, seed=41)
    params = otq.make_params(128, n, scheme, 1041)
    full = P.oracle_decode_from_cache(cache, params, q.float().numpy(), [max(x, 1) for x in lens], B, H, H)
    for b in range(B):
        for h in range(H):
            if lens[b] == 0:
                assert np.all(got[b, h] == 0.0)
            else:
                assert P.rel_l2(got[b, h], full[b, h]) < 1e-3, (b, h)


def test_decode_heads_spanning_several_slices():
    # 2 x 2 heads x 79 tiles: more tiles than persistent CTAs, so slices cross heads and
    # heads cross slices
    lens = [5000, 4999]
    ctx, cache, q, got = _decode_case("KQV", 4, 2, 2, lens, seed=43)
    want = P.oracle_decode_from_cache(cache, otq.make_params(128, 4, "KQV", 1043), q.float().numpy(), lens, 2, 2, 2)
    for b in range(2):
        for h in range(2):
            assert P.rel_l2(got[b, h], want[b, h]) < 1e-3, (b, h)


def test_decode_large_batch_uses_split_kernel():
    # batches above the persistent kernel's prefix-table size take the split-K kernel
    B, H, N = 260, 1, 48
    lens = [N - (b % 7) for b in range(B)]
    ctx, cache, q, got = _decode_case("KQV", 4, B, H, lens, seed=47, cap=64)
    params = otq.make_params(128, 4, "KQV", 1047)
    want = P.oracle_decode_from_cache(cache, params, q.float().numpy(), lens, B, H, H)
    for b in [0, 1, 100, 259]:
        assert P.rel_l2(got[b, 0], want[b, 0]) < 1e-3, b
