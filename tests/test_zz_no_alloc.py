"""The allocation-free decode entry point (tq_decode_attention_static).

It serves callers that cannot allocate device memory themselves -- an
application that owns the whole device-memory budget, a decode loop that must
never enter the CUDA allocator, a runtime without access to cudaMalloc -- by
keeping the decode workspace in a fixed array inside the library. This file is
collected last so that a run stopping at its first failure has already run
every other test; it must also pass alone in a fresh process."""

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantised_kv_cache_gb300 import build
    build.build()


def _rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("scheme,n,G", [("KQV", 4, 1), ("QKQV", 3, 4), ("KIVI", 2, 2)])
def test_static_scratch_decode_matches_the_workspace_entry_point(scheme, n, G):
    from quantised_kv_cache_gb300 import tq
    from quantised_kv_cache_gb300 import workloads as wl

    B, Hkv, N = 2, 2, 700
    Hq = G * Hkv
    w = wl.Workload(97, "no-alloc test", B, Hq, Hkv, N, torch.bfloat16, scheme, n, key_scale_sigma=1.0)
    q, k, v = wl.generate(w, "cpu", seed=77)
    ctx = tq.Context(128, n, scheme, 11)
    cache = tq.Cache(ctx, B, Hkv, 704)
    tq.tq_append_quantize(ctx.handle, cache, k.to(DEV), v.to(DEV), torch.zeros((B,), dtype=torch.int32,
                                                                               device=DEV))
    lens = torch.tensor([N, 515], dtype=torch.int32, device=DEV)
    qd = q.to(DEV)
    want = tq.tq_decode_attention(ctx.handle, cache, qd, lens, N, splits=3).cpu().numpy()
    L = tq.lib()
    for _ in range(2):  # two calls in a row share (and reuse) the one array
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device=DEV)
        st = tq.lib().tq_decode_attention_static(
            ctx.handle, ctypes.byref(cache.struct), ctypes.c_void_p(qd.data_ptr()), tq.TQ_BF16, B, Hq, Hkv,
            ctypes.c_void_p(lens.data_ptr()), N, 3, ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == tq.TQ_OK, L.tq_status_str(st)
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got))
        assert _rel_l2(got, want) < 1e-3
    assert tq.tq_get_device_error(ctx.handle) == 0


def test_static_scratch_rejects_requests_beyond_its_size():
    from quantised_kv_cache_gb300 import tq

    assert tq.tq_static_scratch_bytes() == 8 << 20
    ctx = tq.Context(128, 4, "KQV", 1)
    B, H, cap = 8, 64, 4096
    need = tq.tq_workspace_size(ctx.handle, B, H, H, cap, 1024)
    assert need > tq.tq_static_scratch_bytes()
    # a cache descriptor of those sizes; the call must refuse before touching it
    buf = torch.zeros(1024, dtype=torch.uint8, device=DEV)
    c = tq.tq_cache()
    c.batch, c.heads_kv, c.capacity = B, H, cap
    c.records = buf.data_ptr()
    q = torch.zeros((B, H, 128), dtype=torch.float32, device=DEV)
    lens = torch.full((B,), cap, dtype=torch.int32, device=DEV)
    out = torch.zeros((B, H, 128), dtype=torch.float32, device=DEV)
    st = tq.lib().tq_decode_attention_static(ctx.handle, ctypes.byref(c), ctypes.c_void_p(q.data_ptr()), tq.TQ_F32,
                                             B, H, H, ctypes.c_void_p(lens.data_ptr()), cap, 1024,
                                             ctypes.c_void_p(out.data_ptr()), None)
    assert st == tq.TQ_ERR_WORKSPACE


@pytest.mark.skipif(not torch.cuda.is_available() or torch.cuda.device_count() < 2,
                    reason="needs a second CUDA device")
def test_static_scratch_refuses_a_call_from_another_device():
    # the scratch array is looked up on the current device; a call made while another device
    # is current than the context's is refused before anything is launched
    from quantised_kv_cache_gb300 import tq

    ctx = tq.Context(128, 4, "KQV", 1)
    B, H, cap = 1, 2, 64
    cache = tq.Cache(ctx, B, H, cap, device=torch.device("cuda", 0))
    q = torch.zeros((B, H, 128), dtype=torch.float32, device="cuda:0")
    lens = torch.full((B,), 10, dtype=torch.int32, device="cuda:0")
    out = torch.zeros((B, H, 128), dtype=torch.float32, device="cuda:0")
    with torch.cuda.device(1):
        st = tq.lib().tq_decode_attention_static(ctx.handle, ctypes.byref(cache.struct),
                                                 ctypes.c_void_p(q.data_ptr()), tq.TQ_F32, B, H, H,
                                                 ctypes.c_void_p(lens.data_ptr()), cap, 0,
                                                 ctypes.c_void_p(out.data_ptr()), None)
    assert st == tq.TQ_ERR_ARG
