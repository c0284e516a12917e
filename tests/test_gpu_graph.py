"""The library's calls inside CUDA graphs: a decode loop (append one token per sequence,
attend over the sequence including it, advance the lengths) captured once and replayed
gives byte-for-byte the cache and outputs of the same calls issued eagerly, and so does a
captured bulk append followed by a decode. Every call enqueues its kernels on the caller's
stream and nothing else, which is what capture needs."""

import pytest
import torch

from quantised_kv_cache_gb300 import tq
from quantised_kv_cache_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantised_kv_cache_gb300 import build
    build.build()


def _setup(scheme, n, B, Hkv, G, fill, cap, seed):
    w = wl.Workload(97, "graph", B, Hkv * G, Hkv, fill, torch.bfloat16, scheme, n, key_scale_sigma=1.0)
    q, k, v = wl.generate(w, DEV, seed=seed)
    ctx = tq.Context(128, n, scheme, 500 + seed)
    cache = tq.Cache(ctx, B, Hkv, cap, device=DEV)
    tq.tq_append_quantize(ctx.handle, cache, k, v, torch.zeros(B, dtype=torch.int32, device=DEV))
    steps = [wl.step_token(w, s, DEV, data_seed=seed) for s in range(3)]
    return ctx, cache, steps


def _clone(ctx, cache):
    c = tq.Cache(ctx, cache.batch, cache.heads_kv, cache.capacity, device=DEV)
    for name, t in cache.tensors.items():
        c.tensors[name].copy_(t)
    return c


@pytest.mark.parametrize("scheme,n,G", [("KQV", 4, 1), ("KV", 3, 1), ("KQV", 3, 4)])
def test_captured_decode_loop_replays_the_eager_calls(scheme, n, G):
    B, Hkv, fill, cap = 3, 4, 333, 400
    ctx, cache, steps = _setup(scheme, n, B, Hkv, G, fill, cap, seed=3)
    twin = _clone(ctx, cache)
    lens0 = torch.tensor([fill, fill - 100, 0], dtype=torch.int32, device=DEV)
    ws = torch.empty(tq.tq_workspace_size(ctx.handle, B, Hkv * G, Hkv, cap, 0), dtype=torch.uint8, device=DEV)

    # eager: three steps on the twin
    lens_e = lens0.clone()
    outs_e = []
    for q, kn, vn in steps:
        o = torch.empty((B, Hkv * G, 128), dtype=torch.float32, device=DEV)
        tq.tq_decode_step(ctx.handle, twin, q, kn, vn, lens_e, cap, ws, o)
        lens_e += 1
        outs_e.append(o)
    torch.cuda.synchronize()

    # captured: the same three steps (and the length updates) as one graph
    lens_g = lens0.clone()
    outs_g = [torch.empty((B, Hkv * G, 128), dtype=torch.float32, device=DEV) for _ in steps]
    ws_g = torch.empty_like(ws)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for (q, kn, vn), o in zip(steps, outs_g):
                tq.tq_decode_step(ctx.handle, cache, q, kn, vn, lens_g, cap, ws_g, o,
                                  stream=torch.cuda.current_stream())
                lens_g += 1
    torch.cuda.synchronize()
    # capture ran nothing: the cache and lengths are untouched until the replay
    assert torch.equal(lens_g, lens0)
    g.replay()
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    assert torch.equal(lens_g, lens_e)
    for a, b in zip(outs_g, outs_e):
        assert torch.equal(a, b)
    for name in cache.tensors:
        assert torch.equal(cache.tensors[name], twin.tensors[name]), name
    ctx.close()


def test_captured_append_and_decode_replay_the_eager_calls():
    B, Hkv, G, cap = 2, 3, 2, 300
    w = wl.Workload(98, "graph", B, Hkv * G, Hkv, 200, torch.float32, "KQV", 3, key_scale_sigma=1.0)
    q, k, v = wl.generate(w, DEV, seed=8)
    ctx = tq.Context(128, 3, "KQV", 77)
    a, b = tq.Cache(ctx, B, Hkv, cap, device=DEV), tq.Cache(ctx, B, Hkv, cap, device=DEV)
    start = torch.tensor([0, 50], dtype=torch.int32, device=DEV)
    lens = start + 200
    ws = torch.empty(tq.tq_workspace_size(ctx.handle, B, Hkv * G, Hkv, cap, 0), dtype=torch.uint8, device=DEV)
    out_e = torch.empty((B, Hkv * G, 128), dtype=torch.float32, device=DEV)
    tq.tq_append_quantize(ctx.handle, a, k, v, start)
    tq.tq_decode_attention(ctx.handle, a, q, lens, cap, 0, ws, out_e)
    torch.cuda.synchronize()

    out_g = torch.empty_like(out_e)
    ws_g = torch.empty_like(ws)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            s = torch.cuda.current_stream()
            tq.tq_append_quantize(ctx.handle, b, k, v, start, stream=s)
            tq.tq_decode_attention(ctx.handle, b, q, lens, cap, 0, ws_g, out_g, stream=s)
    g.replay()
    g.replay()  # appending the same tokens at the same slots again changes nothing
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    assert torch.equal(out_g, out_e)
    for name in a.tensors:
        assert torch.equal(a.tensors[name], b.tensors[name]), name
    ctx.close()
