"""GPU tests of the paged cache layout (include/tq.h, "Paged layout"): the records of
each sequence-head live in 16-token blocks of a shared pool, mapped by a block table
("Your KV cache is not a bit problem but a geometry problem", "The systems tax": a
decoding cache grows one token, hence one block, at a time).

Every kernel family is run on a contiguous cache and on a paged one holding the same
tokens behind a shuffled, non-contiguous table with unused pool blocks between them;
the records (gathered back through the table) and the outputs must be identical bit for
bit, and the paged decode is also checked against the oracle directly."""

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


def _table(B, H, cap, seed, spare=7, unmapped_from=None):
    """A shuffled block table over a pool with `spare` extra blocks; entries of blocks at or
    past unmapped_from[b] tokens (when given) are -1."""
    nblk = (cap + 15) // 16
    g = np.random.default_rng(seed)
    pool = B * H * nblk + spare
    perm = g.permutation(pool)[:B * H * nblk].astype(np.int32).reshape(B, H, nblk)
    if unmapped_from is not None:
        for b in range(B):
            first = (unmapped_from[b] + 15) // 16
            perm[b, :, first:] = -1
    return pool, torch.from_numpy(perm).to(DEV)


def _pair(ctx, B, H, cap, seed, **kw):
    pool, table = _table(B, H, cap, seed, **kw)
    return tq.Cache(ctx, B, H, cap), tq.PagedCache(ctx, B, H, cap, pool, table)


def _same_records(a, b):
    assert torch.equal(a.blocks(), b.blocks())


@pytest.mark.parametrize("scheme,n", [("KQV", 4), ("KQV", 3), ("QKQV", 3), ("KV", 2)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("N", [300, 1111], ids=["few", "bulk"])
def test_paged_append_equals_contiguous(scheme, n, dtype, N):
    # "few": 2 x 4 x 300 = 2400 vectors per tensor (warp-per-vector launch); "bulk": 8888
    # (the bulk / tensor-core kernels), appended in two calls that split a token pair
    B, H, cap = 2, 4, N + 21
    w = wl.Workload(95, "paged", B, H, H, N, dtype, scheme, n, key_scale_sigma=1.0)
    _, k, v = wl.generate(w, "cpu", seed=3)
    ctx = tq.Context(128, n, scheme, 61)
    flat, paged = _pair(ctx, B, H, cap, seed=4)
    cut = N // 2 + 1
    for c in (flat, paged):
        tq.tq_append_quantize(ctx.handle, c, k[:, :, :cut].contiguous().to(DEV), v[:, :, :cut].contiguous().to(DEV),
                              torch.zeros(B, dtype=torch.int32, device=DEV))
        tq.tq_append_quantize(ctx.handle, c, k[:, :, cut:].contiguous().to(DEV), v[:, :, cut:].contiguous().to(DEV),
                              torch.full((B,), cut, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    _same_records(flat, paged)
    # and dequantisation reads through the table too
    kf, vf = tq.tq_dequantize(ctx.handle, flat, 0, N)
    kp, vp = tq.tq_dequantize(ctx.handle, paged, 0, N)
    assert torch.equal(kf, kp) and torch.equal(vf, vp)


@pytest.mark.parametrize("scheme,n,G", [("KQV", 4, 1), ("KV", 3, 1), ("KQV", 3, 4), ("KQV", 4, 2),
                                        ("QKQV", 3, 1), ("QKQV", 2, 2), ("KQV", 2, 8)])
def test_paged_decode_equals_contiguous_and_the_oracle(scheme, n, G):
    # ragged lengths (an empty sequence, a partial block, heads spanning several persistent
    # slices); blocks past each sequence's end are unmapped (-1), as a serving cache leaves them
    lens = [0, 5, 700, 2100, 64]
    B, Hkv = len(lens), 2
    Hq = G * Hkv
    cap = 2112
    w = wl.Workload(94, "paged", B, Hq, Hkv, max(lens), torch.bfloat16, scheme, n, key_scale_sigma=1.0)
    q, k, v = wl.generate(w, "cpu", seed=8)
    ctx = tq.Context(128, n, scheme, 62)
    flat, paged = _pair(ctx, B, Hkv, cap, seed=9, unmapped_from=lens)
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    zero = torch.zeros(B, dtype=torch.int32, device=DEV)
    N = max(lens)
    for c in (flat, paged):
        # each sequence gets exactly its own tokens (appends past a length would reach
        # unmapped blocks): one append of the common prefix length per group of sequences
        for b in range(B):
            if lens[b] == 0:
                continue
            kb = torch.zeros((B, Hkv, lens[b], 128), dtype=k.dtype)
            vb = torch.zeros_like(kb)
            kb[b], vb[b] = k[b, :, :lens[b]], v[b, :, :lens[b]]
            start = torch.full((B,), cap, dtype=torch.int32)  # other sequences: past capacity, skipped
            start[b] = 0
            tq.tq_append_quantize(ctx.handle, c, kb.to(DEV), vb.to(DEV), start.to(DEV))
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == tq.TQ_ERR_CAPACITY  # the skipped sequences report it
    _same_records(flat, paged)
    out_f = tq.tq_decode_attention(ctx.handle, flat, q.to(DEV), seq, max_len=N)
    out_p = tq.tq_decode_attention(ctx.handle, paged, q.to(DEV), seq, max_len=N)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    assert torch.equal(out_f, out_p)
    params = otq.make_params(128, n, scheme, 62)
    want = P.oracle_decode_from_cache(paged, params, q.float().numpy(), [max(x, 1) for x in lens], B, Hkv, Hq)
    got = out_p.cpu().numpy()
    for b in range(B):
        for h in range(Hq):
            if lens[b] == 0:
                assert np.all(got[b, h] == 0.0)
            else:
                assert P.rel_l2(got[b, h], want[b, h]) < 1e-3, (b, h)


def test_paged_large_batch_split_kernel():
    # more than 256 sequences: the split-K kernel, whose stages take several blocks per copy
    B, H, N, cap = 260, 1, 100, 112
    lens = [N - (b % 9) for b in range(B)]
    w = wl.Workload(93, "paged", B, H, H, N, torch.bfloat16, "KQV", 4)
    q, k, v = wl.generate(w, "cpu", seed=10)
    ctx = tq.Context(128, 4, "KQV", 63)
    flat, paged = _pair(ctx, B, H, cap, seed=11)
    for c in (flat, paged):
        tq.tq_append_quantize(ctx.handle, c, k.to(DEV), v.to(DEV), torch.zeros(B, dtype=torch.int32, device=DEV))
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out_f = tq.tq_decode_attention(ctx.handle, flat, q.to(DEV), seq, max_len=N, splits=3)
    out_p = tq.tq_decode_attention(ctx.handle, paged, q.to(DEV), seq, max_len=N, splits=3)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    _same_records(flat, paged)
    assert torch.equal(out_f, out_p)


@pytest.mark.parametrize("scheme,n", [("KQV", 4), ("KV", 2), ("QKQV", 3)])
def test_paged_decode_step_equals_contiguous(scheme, n):
    # the fused step appends into the block the table names for slot seq_lens[b], including
    # a block that was unmapped-free until this step (slot 16 j opens block j)
    lens = [0, 15, 16, 300, 1023]
    B, H, cap = len(lens), 3, 1040
    w = wl.Workload(92, "paged", B, H, H, 1024, torch.bfloat16, scheme, n, key_scale_sigma=1.0)
    q, k, v = wl.generate(w, "cpu", seed=12)
    qs, ks, vs = wl.step_token(w, 3, "cpu", data_seed=12, batch=B, heads_kv=H)
    ctx = tq.Context(128, n, scheme, 64)
    flat, paged = _pair(ctx, B, H, cap, seed=13)
    for c in (flat, paged):
        tq.tq_append_quantize(ctx.handle, c, k.to(DEV), v.to(DEV), torch.zeros(B, dtype=torch.int32, device=DEV))
    seq = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out_f = tq.tq_decode_step(ctx.handle, flat, qs.to(DEV), ks.to(DEV), vs.to(DEV), seq, max_len=cap)
    out_p = tq.tq_decode_step(ctx.handle, paged, qs.to(DEV), ks.to(DEV), vs.to(DEV), seq, max_len=cap)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    _same_records(flat, paged)
    assert torch.equal(out_f, out_p)
    # the appended tokens against the oracle's encoding
    params = otq.make_params(128, n, scheme, 64)
    for which, x, role in (("k", ks, params.roles()[0]), ("v", vs, params.roles()[1])):
        ora = otq.encode(x.float().numpy().reshape(-1, 128), role, params)
        enc, _, _ = P.gpu_encoded(paged, role, which, B, H, cap)
        rows = np.array([(b * H + h) * cap + lens[b] for b in range(B) for h in range(H)])
        rep = P.BandReport()
        P.compare_codes(enc.idx[rows], ora, ocb.lloyd_max(128, role.bits).bounds32, rep)
        assert rep.ok_out_of_band(), rep


def test_unmapped_entries_are_reported_not_accessed():
    # an append whose slot falls in an unmapped block writes nothing and reports TQ_ERR_ARG;
    # a decode that reaches one skips the copy and reports the same
    B, H, cap = 2, 2, 64
    ctx = tq.Context(128, 4, "KQV", 65)
    pool, table = _table(B, H, cap, seed=14)
    table[1, 0, 2] = -1       # sequence 1, head 0, tokens 32..47
    table[0, 1, 0] = pool + 5  # past the pool
    paged = tq.PagedCache(ctx, B, H, cap, pool, table)
    g = torch.Generator().manual_seed(15)
    k = torch.randn(B, H, 1, 128, generator=g)
    v = torch.randn(B, H, 1, 128, generator=g)
    before = paged.tensors["records"].clone()
    tq.tq_append_quantize(ctx.handle, paged, k.to(DEV), v.to(DEV), torch.tensor([3, 40], dtype=torch.int32,
                                                                                device=DEV))
    assert tq.tq_get_device_error(ctx.handle) == tq.TQ_ERR_ARG
    after = paged.tensors["records"]
    pool_blocks = after.view(pool, -1)
    changed = (pool_blocks != before.view(pool, -1)).any(dim=1).nonzero().view(-1).tolist()
    # only the two mapped targets were written: (b0, h0, block 0) and (b1, h1, block 2)
    assert sorted(changed) == sorted([int(table[0, 0, 0]), int(table[1, 1, 2])])
    q = torch.randn(B, 2 * H, 128, generator=g).to(DEV)
    out = tq.tq_decode_attention(ctx.handle, paged, q, torch.tensor([4, 41], dtype=torch.int32, device=DEV),
                                 max_len=48)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == tq.TQ_ERR_ARG
    assert out.shape == (B, 2 * H, 128)


def test_kivi_rejects_a_block_table():
    ctx = tq.Context(128, 2, "KIVI", 1)
    cache = tq.Cache(ctx, 1, 1, 64)
    table = torch.zeros((1, 1, 4), dtype=torch.int32, device=DEV)
    cache.struct.block_table = table.data_ptr()
    cache.struct.pool_blocks = 4
    k = torch.zeros((1, 1, 1, 128), device=DEV)
    with pytest.raises(tq.TQError) as e:
        tq.tq_append_quantize(ctx.handle, cache, k, k, torch.zeros(1, dtype=torch.int32, device=DEV))
    assert e.value.status == tq.TQ_ERR_UNSUPPORTED
