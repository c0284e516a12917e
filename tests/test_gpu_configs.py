"""GPU parity at the five workloads' full sizes (in the launch configuration the
benchmark times): every code where the oracle is fast enough, otherwise seeded
samples of vectors and of (batch, head) decode units the oracle computes one
by one."""

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import codebook as ocb
from oracle import kivi as okivi
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


def _fill(ctx, w, cache, k, v):
    z = torch.zeros((w.batch,), dtype=torch.int32, device=DEV)
    tq.tq_append_quantize(ctx.handle, cache, k, v, z)


def _norm_rtol(x, B, H, N, role):
    return P.norm_rtol(P.bulk_bf16_path(x.dtype, B * H * N, role))


def _check_sampled_codes(cache, params, k, v, B, H, N, n_sample, seed, rep=None, srep=None):
    """Compare n_sample random token-heads of K and V with the oracle's encoding
    (the whole cache was written by one append call of B x H x N vectors per tensor).

    Out-of-band mismatches fail at once; the in-band fraction is checked by the
    caller on the reports accumulated over the whole workload."""
    rep = P.BandReport() if rep is None else rep
    srep = P.BandReport() if srep is None else srep
    g = np.random.default_rng(seed)
    sel = g.choice(B * H * N, size=min(n_sample, B * H * N), replace=False)
    b, h, t = sel // (H * N), (sel // N) % H, sel % N
    for which, x, role in (("k", k, params.roles()[0]), ("v", v, params.roles()[1])):
        xs = x[torch.as_tensor(b), torch.as_tensor(h), torch.as_tensor(t)].float().cpu().numpy()
        ora = otq.encode(xs, role, params)
        cap = cache.struct.capacity
        cb = role.bits * 16
        codes = cache.plane(f"{which}_codes").view(B, H, cap, cb)[torch.as_tensor(b), torch.as_tensor(h),
                                                                   torch.as_tensor(t)].cpu().numpy()
        gidx = otq.unpack_codes(codes, role.bits, 128)
        mism = P.compare_codes(gidx, ora, ocb.lloyd_max(128, role.bits).bounds32, rep)
        assert rep.ok_out_of_band(), f"{which}: {rep}"
        norms = cache.plane(f"{which}_norm").view(torch.float32).view(B, H, cap)[torch.as_tensor(b),
                                                                             torch.as_tensor(h),
                                                                             torch.as_tensor(t)].cpu().numpy()
        np.testing.assert_allclose(norms, ora.norm, rtol=_norm_rtol(x, B, H, N, role))
        if role.qjl:
            sg = cache.plane(f"{which}_signs").view(B, H, cap, 16)[torch.as_tensor(b), torch.as_tensor(h),
                                                                  torch.as_tensor(t)].cpu().numpy()
            P.compare_signs(otq.unpack_signs(sg, 128), ora, srep, skip_rows=mism.any(axis=1))
            assert srep.ok_out_of_band(), f"{which} signs: {srep}"
    return rep, srep


def _unit_planes(cache, role, which, Hkv):
    """A role's planes as [batch][kv head][slot] arrays (fetched once; the value codes
    are converted out of the pair-interleaved blocks on the device)."""
    cap = cache.struct.capacity
    cb = role.bits * 16
    out = {"codes": cache.plane(f"{which}_codes").view(-1, Hkv, cap, cb),
           "norm": cache.plane(f"{which}_norm").view(torch.float32).view(-1, Hkv, cap)}
    if role.qjl:
        out["signs"] = cache.plane(f"{which}_signs").view(-1, Hkv, cap, 16)
        out["rnorm"] = cache.plane(f"{which}_rnorm").view(torch.float32).view(-1, Hkv, cap)
    return out


def _check_sampled_decode(cache, params, q, out, lens, B, Hkv, Hq, units, tol=1e-3):
    """Oracle attention (fp64, over the GPU's own codes) for selected (b, kv head) units
    over their full length, for every query head of each unit's group."""
    G = Hq // Hkv
    rk, rv = params.roles()
    planes = {"k": _unit_planes(cache, rk, "k", Hkv), "v": _unit_planes(cache, rv, "v", Hkv)}
    errs = []
    for (b, hk) in units:
        n = int(lens[b])

        def enc(which, role):
            pl = planes[which]
            take = lambda name: pl[name][b, hk, :n].cpu().numpy()
            sg = take("signs") if role.qjl else None
            rn = take("rnorm") if role.qjl else None
            return otq.encoded_from_storage(role, take("norm"), take("codes"), 128, sg, rn)

        Kh = otq.decode(enc("k", rk), params)
        Vh = otq.decode(enc("v", rv), params)
        for g in range(G):
            h = hk * G + g
            want, _ = oatt.attend(q[b, h].float().cpu().numpy(), Kh, Vh)
            err = P.rel_l2(out[b, h].cpu().numpy(), want)
            errs.append(err)
            assert err < tol, (b, h, err)
    return errs


def _units(B, H, count, seed):
    """`count` distinct seeded (batch, kv head) units."""
    g = np.random.default_rng(seed)
    sel = g.choice(B * H, size=min(count, B * H), replace=False)
    return [(int(u) // H, int(u) % H) for u in sel]


def test_config1_single_head_all_codes_and_output():
    w = wl.WORKLOADS[1]
    q, k, v = wl.generate(w, DEV)
    ctx = tq.Context(128, w.bits, w.scheme, 42)
    cache = tq.Cache(ctx, 1, 1, w.seq)
    _fill(ctx, w, cache, k, v)
    params = otq.make_params(128, w.bits, w.scheme, 42)
    rep, srep = _check_sampled_codes(cache, params, k, v, 1, 1, w.seq, w.seq, 0)  # every token
    assert rep.ok() and srep.ok(), (rep, srep)
    lens = torch.full((1,), w.seq, dtype=torch.int32, device=DEV)
    out = tq.tq_decode_attention(ctx.handle, cache, q, lens, w.seq)
    _check_sampled_decode(cache, params, q, out, [w.seq], 1, 1, 1, [(0, 0)])


def test_config2_llama7b_shaped_decode_step():
    # exactly what the benchmark times: 8191 prefilled tokens per sequence-head (one bulk
    # append), then tq_decode_step appends token 8192 and attends over all of them
    w = wl.WORKLOADS[2]
    q, k, v = wl.generate(w, DEV)
    B, H, N = w.batch, w.heads_kv, w.seq
    ctx = tq.Context(128, w.bits, w.scheme, 42)
    cache = tq.Cache(ctx, B, H, N)
    z = torch.zeros((B,), dtype=torch.int32, device=DEV)
    tq.tq_append_quantize(ctx.handle, cache, k[:, :, :-1].contiguous(), v[:, :, :-1].contiguous(), z)
    torch.cuda.synchronize()
    # the same step as two calls, on a copy of the prefilled cache
    two = tq.Cache(ctx, B, H, N)
    two.tensors["records"].copy_(cache.tensors["records"])
    lens_a = torch.full((B,), N - 1, dtype=torch.int32, device=DEV)
    kn, vn = k[:, :, -1:].contiguous(), v[:, :, -1:].contiguous()
    out = tq.tq_decode_step(ctx.handle, cache, q, kn, vn, lens_a, N)
    tq.tq_append_quantize(ctx.handle, two, kn, vn, lens_a)
    lens = torch.full((B,), N, dtype=torch.int32, device=DEV)
    out_two = tq.tq_decode_attention(ctx.handle, two, q, lens, N)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    # the fused step is bit-equal to append + decode (same records, same output)
    assert torch.equal(cache.tensors["records"], two.tensors["records"])
    assert torch.equal(out, out_two)
    params = otq.make_params(128, w.bits, w.scheme, 42)
    # prefilled records: a seeded sample under the band rule (one bulk call of B H (N - 1) vectors)
    rep, srep = _check_sampled_codes(cache, params, k[:, :, :-1], v[:, :, :-1], B, H, N - 1, 20000, 1)
    # the step's appended record of every head, under the same rule
    _check_sampled_codes_slot(cache, params, k, v, w, rep, srep)
    assert rep.ok() and srep.ok(), (rep, srep)
    errs = _check_sampled_decode(cache, params, q, out, [N] * B, B, H, w.heads_q, _units(B, H, 8, 2))
    assert max(errs) < 1e-3


def _check_sampled_codes_slot(cache, params, k, v, w, rep, srep):
    """The last slot of every sequence-head (written by the decode step's warp-per-vector
    encoder) against the oracle's encoding of the same token."""
    B, H, N = w.batch, w.heads_kv, w.seq
    for which, x, role in (("k", k, params.roles()[0]), ("v", v, params.roles()[1])):
        xs = x[:, :, -1].float().cpu().numpy().reshape(-1, 128)
        ora = otq.encode(xs, role, params)
        codes = cache.plane(f"{which}_codes").view(B, H, N, role.bits * 16)[:, :, -1].cpu().numpy()
        mism = P.compare_codes(otq.unpack_codes(codes.reshape(-1, role.bits * 16), role.bits, 128), ora,
                               ocb.lloyd_max(128, role.bits).bounds32, rep)
        assert rep.ok_out_of_band(), rep
        norms = cache.plane(f"{which}_norm").view(torch.float32).view(B, H, N)[:, :, -1].cpu().numpy()
        np.testing.assert_allclose(norms.reshape(-1), ora.norm, rtol=P.norm_rtol(False))
        if role.qjl:
            sg = cache.plane(f"{which}_signs").view(B, H, N, 16)[:, :, -1].cpu().numpy().reshape(-1, 16)
            P.compare_signs(otq.unpack_signs(sg, 128), ora, srep, skip_rows=mism.any(axis=1))
            assert srep.ok_out_of_band(), srep


@pytest.mark.parametrize("dist", ["gauss", "lowrank", "student3"])
@pytest.mark.parametrize("scheme", ["KV", "KQV", "QKQV"])
@pytest.mark.parametrize("n", [2, 3, 4])
def test_config3_scheme_sweep(dist, scheme, n):
    w = wl.WORKLOADS[3]
    q, k, v = wl.generate(w, DEV, key_dist=dist)
    ctx = tq.Context(128, n, scheme, 42)
    cache = tq.Cache(ctx, w.batch, w.heads_kv, w.seq)
    _fill(ctx, w, cache, k, v)
    lens = torch.full((w.batch,), w.seq, dtype=torch.int32, device=DEV)
    out = tq.tq_decode_attention(ctx.handle, cache, q, lens, w.seq)
    torch.cuda.synchronize()
    params = otq.make_params(128, n, scheme, 42)
    rep, srep = _check_sampled_codes(cache, params, k, v, w.batch, w.heads_kv, w.seq, 3000, n)
    assert rep.ok() and srep.ok(), (rep, srep)
    _check_sampled_decode(cache, params, q, out, [w.seq] * w.batch, w.batch, w.heads_kv, w.heads_q,
                          _units(w.batch, w.heads_kv, 4, 3 + n))


def test_config4_gqa_long_context_64_splits():
    w = wl.WORKLOADS[4]
    q, k, v = wl.generate(w, DEV)
    ctx = tq.Context(128, w.bits, w.scheme, 42)
    cache = tq.Cache(ctx, w.batch, w.heads_kv, w.seq)
    _fill(ctx, w, cache, k, v)
    lens = torch.full((w.batch,), w.seq, dtype=torch.int32, device=DEV)
    out = tq.tq_decode_attention(ctx.handle, cache, q, lens, w.seq, splits=w.splits)
    torch.cuda.synchronize()
    params = otq.make_params(128, w.bits, w.scheme, 42)
    rep, srep = _check_sampled_codes(cache, params, k, v, w.batch, w.heads_kv, w.seq, 20000, 4)
    assert rep.ok() and srep.ok(), (rep, srep)
    _check_sampled_decode(cache, params, q, out, [w.seq], w.batch, w.heads_kv, w.heads_q,
                          [(0, h) for h in range(w.heads_kv)])


@pytest.mark.parametrize("layout", [(True, True), (False, False), (False, True), (True, False)])
def test_config5_kivi_layouts(layout):
    w = wl.WORKLOADS[5]
    kpc, vpt = layout
    q, k, v = wl.generate(w, DEV)
    ctx = tq.Context(128, 2, "KIVI", 0, k_per_channel=kpc, v_per_token=vpt)
    cache = tq.Cache(ctx, w.batch, w.heads_kv, w.seq)
    _fill(ctx, w, cache, k, v)
    lens = torch.full((w.batch,), w.seq, dtype=torch.int32, device=DEV)
    out = tq.tq_decode_attention(ctx.handle, cache, q, lens, w.seq).cpu().numpy()
    assert tq.tq_get_device_error(ctx.handle) == 0
    B, H, N = w.batch, w.heads_kv, w.seq
    codes = cache.plane("k_codes")  # noqa: F841 (planes read through the helpers below)
    for (b, h) in _units(B, H, 8, 5):
        for which, x, per_channel in (("k", k, kpc), ("v", v, not vpt)):
            st = okivi.quantize_tensor(x[b, h].float().cpu().numpy(), per_channel)
            gcodes = P.kivi_gpu_codes(cache, which, B, H, N)[b, h, :st.nq]
            rep = P.BandReport()
            rep.add(gcodes != st.codes, np.abs(np.abs(st.t - np.floor(st.t)) - 0.5))
            assert rep.ok(), rep
            z, s = P.kivi_gpu_stats(cache, which, B, H, per_channel)
            nz = st.nq // 32 if per_channel else st.nq
            np.testing.assert_array_equal(z[b, h, :nz], st.z16)
            np.testing.assert_array_equal(s[b, h, :nz], st.s16)
        Kh = P.kivi_dequant_gpu_state(cache, "k", B, H, N, kpc)[b, h]
        Vh = P.kivi_dequant_gpu_state(cache, "v", B, H, N, not vpt)[b, h]
        want, _ = oatt.attend(q[b, h].float().cpu().numpy(), Kh, Vh)
        assert P.rel_l2(out[b, h], want) < 1e-3
