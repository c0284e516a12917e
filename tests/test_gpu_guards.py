"""Writes stay inside their buffers, and a cache survives a save / restore.

Guard bands: every cache array, the workspace, the output and the decode step's inputs are
carved from larger buffers whose margins hold a known byte pattern; appends on each append path
(few-vector, bulk bf16, fp32 tensor-core, unrotated, KIVI flush and window) filling sequences up
to exactly their capacity, decodes, decode steps and dequantisation must leave every margin
untouched.

Checkpoint: a cache is plain caller-owned device memory plus the context's seeded parameters,
so copying its arrays to the host, rebuilding a context from the same arguments and copying them
back gives bit-identical attention."""

import numpy as np
import pytest
import torch

from quantised_kv_cache_gb300 import tq
from quantised_kv_cache_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 4096
FILL = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantised_kv_cache_gb300 import build
    build.build()


class Guarded:
    """n bytes (as `dtype`) in the middle of a buffer with GUARD-byte margins of FILL."""

    def __init__(self, n_bytes, dtype=torch.uint8):
        self.n = n_bytes
        self.buf = torch.full((GUARD + n_bytes + GUARD,), FILL, dtype=torch.uint8, device=DEV)
        self.inner = self.buf[GUARD:GUARD + n_bytes]
        self.view = self.inner.view(dtype) if n_bytes else self.inner

    def intact(self):
        return bool((self.buf[:GUARD] == FILL).all()) and bool((self.buf[GUARD + self.n:] == FILL).all())


def guarded_copy(t):
    g = Guarded(t.numel() * t.element_size(), t.dtype)
    g.view.copy_(t.reshape(-1))
    return g, g.view.view(t.shape)


class GuardedCache(tq.Cache):
    def __init__(self, ctx, batch, heads_kv, capacity):
        super().__init__(ctx, batch, heads_kv, capacity, device=DEV)
        self.guards = {}
        for name, t in list(self.tensors.items()):
            g = Guarded(t.numel())
            g.inner.zero_()
            self.guards[name] = g
            self.tensors[name] = g.inner
            setattr(self.struct, name, g.inner.data_ptr())

    def intact(self):
        return all(g.intact() for g in self.guards.values())


CASES = [("KQV", 4, torch.bfloat16, 1), ("KQV", 3, torch.float32, 2), ("KV", 3, torch.bfloat16, 1),
         ("QKQV", 2, torch.float32, 2), ("KIVI", 2, torch.bfloat16, 2)]


@pytest.mark.parametrize("scheme,n,dtype,G", CASES)
def test_appends_decodes_and_steps_stay_inside_their_buffers(scheme, n, dtype, G):
    B, H, cap = 3, 4, 1056  # a multiple of the KIVI group (32)
    ctx = tq.Context(128, n, scheme, 11)
    cache = GuardedCache(ctx, B, H, cap)
    w = wl.Workload(90, "guard", B, H * G, H, 1001, dtype, scheme, n, key_scale_sigma=1.0)
    q, k, v = wl.generate(w, DEV, seed=2)
    # a bulk append from zero (8400 vectors per tensor: the bulk paths), then a few-vector append
    # to 1000 tokens, a decode, and decode steps up to exactly the capacity
    kg, kk = guarded_copy(k[:, :, :700].contiguous())
    vg, vv = guarded_copy(v[:, :, :700].contiguous())
    tq.tq_append_quantize(ctx.handle, cache, kk, vv, torch.zeros(B, dtype=torch.int32, device=DEV))
    k2g, k2 = guarded_copy(k[:, :, 700:1000].contiguous())
    v2g, v2 = guarded_copy(v[:, :, 700:1000].contiguous())
    tq.tq_append_quantize(ctx.handle, cache, k2, v2, torch.full((B,), 700, dtype=torch.int32, device=DEV))
    lens_now = torch.full((B,), 1000, dtype=torch.int32, device=DEV)
    ws_bytes = tq.tq_workspace_size(ctx.handle, B, H * G, H, cap, 0)
    wsg = Guarded(ws_bytes)
    outg = Guarded(B * H * G * 128 * 4, torch.float32)
    qg, qq = guarded_copy(q.contiguous())
    tq.tq_decode_attention(ctx.handle, cache, qq, lens_now, cap, 0, wsg.inner, outg.view.view(B, H * G, 128))
    # 56 decode steps fill the sequences to 1056 tokens, the capacity
    kng, kn = guarded_copy(k[:, :, 1000:1001].contiguous())
    vng, vn = guarded_copy(v[:, :, 1000:1001].contiguous())
    for step in range(cap - 1000):
        lens_step = torch.full((B,), 1000 + step, dtype=torch.int32, device=DEV)
        tq.tq_decode_step(ctx.handle, cache, qq, kn, vn, lens_step, cap, wsg.inner, outg.view.view(B, H * G, 128))
    # dequantise the whole capacity into guarded outputs
    khg = Guarded(B * H * cap * 128 * 4, torch.float32)
    vhg = Guarded(B * H * cap * 128 * 4, torch.float32)
    full = torch.full((B,), cap, dtype=torch.int32, device=DEV)
    tq.tq_dequantize(ctx.handle, cache, 0, cap, seq_lens=full, k_out=khg.view.view(B, H, cap, 128),
                     v_out=vhg.view.view(B, H, cap, 128))
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ctx.handle) == 0
    assert cache.intact(), {name: g.intact() for name, g in cache.guards.items()}
    for g in (kg, vg, k2g, v2g, wsg, outg, qg, kng, vng, khg, vhg):
        assert g.intact()
    assert np.isfinite(outg.view.cpu().numpy()).all()
    ctx.close()


@pytest.mark.parametrize("scheme,n", [("KQV", 4), ("QKQV", 3), ("KIVI", 2)])
def test_a_saved_and_restored_cache_decodes_identically(scheme, n):
    B, H, cap = 2, 3, 320
    w = wl.Workload(91, "ckpt", B, H, H, 300, torch.bfloat16, scheme, n, key_scale_sigma=1.0)
    q, k, v = wl.generate(w, DEV, seed=4)
    ctx = tq.Context(128, n, scheme, 21)
    cache = tq.Cache(ctx, B, H, cap, device=DEV)
    tq.tq_append_quantize(ctx.handle, cache, k, v, torch.zeros(B, dtype=torch.int32, device=DEV))
    lens = torch.tensor([300, 123], dtype=torch.int32, device=DEV)
    want = tq.tq_decode_attention(ctx.handle, cache, q, lens, cap).cpu()
    saved = {name: t.cpu().clone() for name, t in cache.tensors.items()}
    ctx.close()
    del cache
    torch.cuda.synchronize()
    ctx2 = tq.Context(128, n, scheme, 21)  # the same arguments draw the same parameters
    restored = tq.Cache(ctx2, B, H, cap, device=DEV)
    for name, t in saved.items():
        restored.tensors[name].copy_(t.to(DEV))
    got = tq.tq_decode_attention(ctx2.handle, restored, q, lens, cap).cpu()
    assert torch.equal(got, want)
    assert tq.tq_get_device_error(ctx2.handle) == 0
    ctx2.close()
