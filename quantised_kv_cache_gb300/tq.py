"""Thin ctypes binding of libtq's C ABI (include/tq.h), same names as the C calls.

Argument marshalling only: every step of quantisation and attention runs in
the CUDA kernels behind the ABI. PyTorch is used for device memory and
streams. If ``_lib/libtq.so`` is missing this module raises at first use --
there is no fallback implementation.
"""

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libtq.so")

TQ_OK = 0
TQ_ERR_ARG = 1
TQ_ERR_UNSUPPORTED = 2
TQ_ERR_CAPACITY = 3
TQ_ERR_CUDA = 4
TQ_ERR_TIMEOUT = 5
TQ_ERR_STATE = 6
TQ_ERR_ALIGN = 7
TQ_ERR_WORKSPACE = 8

TQ_SCHEME_KV = 0
TQ_SCHEME_KQV = 1
TQ_SCHEME_QKQV = 2
TQ_SCHEME_KIVI = 3
SCHEMES = {"KV": TQ_SCHEME_KV, "KQV": TQ_SCHEME_KQV, "QKQV": TQ_SCHEME_QKQV, "KIVI": TQ_SCHEME_KIVI}

TQ_F32 = 0
TQ_BF16 = 1

TQ_ROTATION_WHT = 0
TQ_ROTATION_DENSE = 1
ROTATIONS = {"wht": TQ_ROTATION_WHT, "dense": TQ_ROTATION_DENSE}

_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t


class tq_cache(ctypes.Structure):
    _fields_ = [("batch", _i), ("heads_kv", _i), ("capacity", _i), ("records", _vp),
                ("k_codes", _vp), ("v_codes", _vp),
                ("k_stats", _vp), ("v_stats", _vp), ("k_window", _vp), ("v_window", _vp),
                ("block_table", _vp), ("pool_blocks", _i)]


# the planes of a block of the records array (TQ schemes), in storage order (tq_plane)
RECORD_PLANES = ["k_codes", "k_norm", "k_signs", "k_rnorm", "v_codes", "v_norm", "v_signs", "v_rnorm", "k_side"]
# separately allocated arrays (records for TQ schemes; the KIVI planes)
ARRAYS = ["records", "k_codes", "v_codes", "k_stats", "v_stats", "k_window", "v_window"]
BLOCK_TOKENS = 16


class tq_cache_sizes(ctypes.Structure):
    _fields_ = [("records", _sz), ("block_bytes", _sz), ("plane_offset", _sz * 9), ("plane_bytes", _sz * 9),
                ("k_codes", _sz), ("v_codes", _sz), ("k_stats", _sz), ("v_stats", _sz), ("k_window", _sz),
                ("v_window", _sz), ("record_bytes", _sz)]


_SIGNATURES = {
    "tq_abi_version": (_i, []),
    "tq_status_str": (ctypes.c_char_p, [_i]),
    "tq_init": (_i, [_i, _i, _i, ctypes.c_uint64, ctypes.POINTER(_vp)]),
    "tq_destroy": (None, [_vp]),
    "tq_set_kivi": (_i, [_vp, _i, _i, _i, _i]),
    "tq_set_rotation": (_i, [_vp, _i]),
    "tq_set_side_basis": (_i, [_vp, _i, _i, _vp]),
    "tq_principal_basis": (_i, [_vp, _i, _i, _i, _vp]),
    "tq_draw_rotation": (_i, [ctypes.c_uint64, _i, _vp]),
    "tq_cache_sizes_get": (_i, [_vp, _i, _i, _i, ctypes.POINTER(tq_cache_sizes)]),
    "tq_cache_bytes": (_i, [_vp, _i, _i, _i, ctypes.POINTER(tq_cache_sizes)]),
    "tq_workspace_bytes": (_i, [_vp, _i, _i, _i, _i, _i, ctypes.POINTER(_sz)]),
    "tq_append_quantize": (_i, [_vp, ctypes.POINTER(tq_cache), _vp, _vp, _i, _i, _i, _i, _vp, _vp]),
    "tq_workspace_size": (_i, [_vp, _i, _i, _i, _i, _i, ctypes.POINTER(_sz)]),
    "tq_decode_attention": (_i, [_vp, ctypes.POINTER(tq_cache), _vp, _i, _i, _i, _i, _vp, _i, _i, _vp, _sz,
                                 _vp, _vp]),
    "tq_decode_step": (_i, [_vp, ctypes.POINTER(tq_cache), _vp, _i, _vp, _vp, _i, _i, _i, _i, _vp, _i, _vp, _sz,
                            _vp, _vp]),
    "tq_dequantize": (_i, [_vp, ctypes.POINTER(tq_cache), _i, _i, _i, _i, _vp, _vp, _vp, _vp]),
    "tq_export_params": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "tq_codebook_f64": (_i, [_i, _i, _vp, _vp]),
    "tq_draw_params": (_i, [ctypes.c_uint64, _i, _vp, _vp]),
    "tq_get_device_error": (_i, [_vp, _vp, ctypes.POINTER(_i)]),
    "tq_set_profile_events": (_i, [_vp, _vp, _vp, _vp, _vp]),
    "tq_decode_attention_static": (_i, [_vp, ctypes.POINTER(tq_cache), _vp, _i, _i, _i, _i, _vp, _i, _i, _vp,
                                        _vp]),
    "tq_static_scratch_bytes": (_sz, []),
    "tq_selftest_bounded_wait": (_i, [_vp, ctypes.c_ulonglong, _vp]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load libtq.so (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libtq.so not built at {LIB_PATH}: run "
                               "`python -m quantised_kv_cache_gb300.build` (no CPU fallback exists)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class TQError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = lib().tq_status_str(status).decode()
        super().__init__(f"{what}: {msg} (status {status})" if what else f"{msg} (status {status})")


def check(status: int, what: str = "") -> None:
    if status != TQ_OK:
        raise TQError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return TQ_F32
    if t.dtype == torch.bfloat16:
        return TQ_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


# ----------------------------------------------------------------------------
# same-name wrappers of the C calls
# ----------------------------------------------------------------------------

def tq_abi_version() -> int:
    return lib().tq_abi_version()


def tq_status_str(status: int) -> str:
    return lib().tq_status_str(status).decode()


def tq_init(d: int, bits: int, scheme, seed: int) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    s = SCHEMES[scheme] if isinstance(scheme, str) else int(scheme)
    check(lib().tq_init(d, bits, s, ctypes.c_uint64(seed), ctypes.byref(h)), "tq_init")
    return h


def tq_destroy(ctx) -> None:
    lib().tq_destroy(ctx)


def tq_set_kivi(ctx, group=32, window=128, k_per_channel=True, v_per_token=True) -> None:
    check(lib().tq_set_kivi(ctx, group, window, int(k_per_channel), int(v_per_token)), "tq_set_kivi")


def tq_set_rotation(ctx, rotation="wht") -> None:
    r = ROTATIONS[rotation] if isinstance(rotation, str) else int(rotation)
    check(lib().tq_set_rotation(ctx, r), "tq_set_rotation")


def tq_set_side_basis(ctx, basis: Optional[np.ndarray]) -> None:
    """basis: float [heads_kv][d][rank] with orthonormal columns per head, or None (off)."""
    if basis is None:
        check(lib().tq_set_side_basis(ctx, 0, 0, None), "tq_set_side_basis")
        return
    B = np.ascontiguousarray(basis, dtype=np.float32)
    heads, d, rank = B.shape
    check(lib().tq_set_side_basis(ctx, rank, heads, B.ctypes.data_as(ctypes.c_void_p)), "tq_set_side_basis")


def tq_principal_basis(x: np.ndarray, rank: int) -> np.ndarray:
    """[d][rank] leading principal directions (about the origin) of the rows of x."""
    X = np.ascontiguousarray(x, dtype=np.float32)
    n, d = X.shape
    U = np.zeros((d, rank), np.float32)
    check(lib().tq_principal_basis(X.ctypes.data_as(ctypes.c_void_p), n, d, rank, U.ctypes.data_as(ctypes.c_void_p)),
          "tq_principal_basis")
    return U


def tq_draw_rotation(seed: int, d: int = 128):
    M = np.zeros((d, d), np.float32)
    check(lib().tq_draw_rotation(ctypes.c_uint64(seed), d, M.ctypes.data_as(ctypes.c_void_p)), "tq_draw_rotation")
    return M


def tq_cache_sizes_get(ctx, batch: int, heads_kv: int, capacity: int) -> tq_cache_sizes:
    out = tq_cache_sizes()
    check(lib().tq_cache_sizes_get(ctx, batch, heads_kv, capacity, ctypes.byref(out)), "tq_cache_sizes_get")
    return out


def tq_cache_bytes(ctx, batch: int, heads_kv: int, capacity: int) -> tq_cache_sizes:
    out = tq_cache_sizes()
    check(lib().tq_cache_bytes(ctx, batch, heads_kv, capacity, ctypes.byref(out)), "tq_cache_bytes")
    return out


def tq_append_quantize(ctx, cache: "Cache", k: torch.Tensor, v: torch.Tensor, seq_lens: torch.Tensor,
                       stream=None) -> None:
    B, H, n, d = k.shape
    assert v.shape == k.shape and k.dtype == v.dtype and k.is_contiguous() and v.is_contiguous()
    assert seq_lens.dtype == torch.int32 and seq_lens.is_cuda
    check(lib().tq_append_quantize(ctx, ctypes.byref(cache.struct), _ptr(k), _ptr(v), _dtype_code(k), B, H, n,
                                   _ptr(seq_lens), _stream(stream)), "tq_append_quantize")


def tq_workspace_size(ctx, batch, heads_q, heads_kv, max_len, splits=0) -> int:
    out = _sz()
    check(lib().tq_workspace_size(ctx, batch, heads_q, heads_kv, max_len, splits, ctypes.byref(out)),
          "tq_workspace_size")
    return out.value


def tq_workspace_bytes(ctx, batch, heads_q, heads_kv, max_len, splits=0) -> int:
    out = _sz()
    check(lib().tq_workspace_bytes(ctx, batch, heads_q, heads_kv, max_len, splits, ctypes.byref(out)),
          "tq_workspace_bytes")
    return out.value


def tq_decode_attention(ctx, cache: "Cache", q: torch.Tensor, seq_lens: torch.Tensor, max_len: int,
                        splits: int = 0, workspace: Optional[torch.Tensor] = None,
                        out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    B, Hq, d = q.shape
    assert q.is_contiguous() and seq_lens.dtype == torch.int32
    Hkv = cache.struct.heads_kv
    need = tq_workspace_size(ctx, B, Hq, Hkv, max_len, splits)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    check(lib().tq_decode_attention(ctx, ctypes.byref(cache.struct), _ptr(q), _dtype_code(q), B, Hq, Hkv,
                                    _ptr(seq_lens), max_len, splits, _ptr(workspace), workspace.numel(),
                                    _ptr(out), _stream(stream)), "tq_decode_attention")
    return out


def tq_decode_step(ctx, cache: "Cache", q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                   seq_lens: torch.Tensor, max_len: int, workspace: Optional[torch.Tensor] = None,
                   out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Append k_new / v_new ([batch][heads_kv][d], or [batch][heads_kv][1][d]) at slot
    seq_lens[b], then attend over seq_lens[b] + 1 tokens; seq_lens is not modified."""
    B, Hq, d = q.shape
    assert q.is_contiguous() and k_new.is_contiguous() and v_new.is_contiguous()
    Hkv = cache.struct.heads_kv
    assert k_new.shape == v_new.shape and k_new.dtype == v_new.dtype and k_new.numel() == B * Hkv * d
    assert seq_lens.dtype == torch.int32 and seq_lens.is_cuda
    need = tq_workspace_size(ctx, B, Hq, Hkv, max_len, 0)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    check(lib().tq_decode_step(ctx, ctypes.byref(cache.struct), _ptr(q), _dtype_code(q), _ptr(k_new), _ptr(v_new),
                               _dtype_code(k_new), B, Hq, Hkv, _ptr(seq_lens), max_len, _ptr(workspace),
                               workspace.numel(), _ptr(out), _stream(stream)), "tq_decode_step")
    return out


def tq_decode_attention_static(ctx, cache: "Cache", q: torch.Tensor, seq_lens: torch.Tensor, max_len: int,
                               splits: int = 0, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """tq_decode_attention with the library's built-in scratch array instead of a workspace."""
    B, Hq, d = q.shape
    assert q.is_contiguous() and seq_lens.dtype == torch.int32
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    check(lib().tq_decode_attention_static(ctx, ctypes.byref(cache.struct), _ptr(q), _dtype_code(q), B, Hq,
                                           cache.struct.heads_kv, _ptr(seq_lens), max_len, splits, _ptr(out),
                                           _stream(stream)), "tq_decode_attention_static")
    return out


def tq_static_scratch_bytes() -> int:
    return lib().tq_static_scratch_bytes()


def tq_dequantize(ctx, cache: "Cache", t0: int, t1: int, seq_lens: Optional[torch.Tensor] = None,
                  k_out: Optional[torch.Tensor] = None, v_out: Optional[torch.Tensor] = None, stream=None):
    B, H = cache.struct.batch, cache.struct.heads_kv
    dev = cache.device
    if k_out is None:
        k_out = torch.empty((B, H, t1 - t0, 128), dtype=torch.float32, device=dev)
    if v_out is None:
        v_out = torch.empty((B, H, t1 - t0, 128), dtype=torch.float32, device=dev)
    check(lib().tq_dequantize(ctx, ctypes.byref(cache.struct), B, H, t0, t1, _ptr(seq_lens), _ptr(k_out),
                              _ptr(v_out), _stream(stream)), "tq_dequantize")
    return k_out, v_out


@dataclass
class Params:
    k_bits: int
    k_centroids: "np.ndarray"
    k_bounds: "np.ndarray"
    v_bits: int
    v_centroids: "np.ndarray"
    v_bounds: "np.ndarray"
    diag: "np.ndarray"
    sketch: "np.ndarray"


def tq_export_params(ctx, d: int = 128) -> Params:
    import numpy as np
    kb, vb = _i(), _i()
    kc, kbd, vc, vbd = (np.zeros(16, np.float32) for _ in range(4))
    diag = np.zeros(d, np.int8)
    S = np.zeros((d, d), np.float32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    check(lib().tq_export_params(ctx, ctypes.byref(kb), p(kc), p(kbd), ctypes.byref(vb), p(vc), p(vbd), p(diag),
                                 p(S)), "tq_export_params")
    Lk, Lv = 1 << kb.value, 1 << vb.value
    return Params(kb.value, kc[:Lk], kbd[:Lk - 1], vb.value, vc[:Lv], vbd[:Lv - 1], diag, S)


def tq_codebook_f64(d: int, bits: int):
    import numpy as np
    c = np.zeros(1 << bits)
    b = np.zeros((1 << bits) - 1)
    check(lib().tq_codebook_f64(d, bits, c.ctypes.data_as(ctypes.c_void_p), b.ctypes.data_as(ctypes.c_void_p)),
          "tq_codebook_f64")
    return c, b


def tq_draw_params(seed: int, d: int):
    import numpy as np
    diag = np.zeros(d, np.int8)
    S = np.zeros((d, d), np.float32)
    check(lib().tq_draw_params(ctypes.c_uint64(seed), d, diag.ctypes.data_as(ctypes.c_void_p),
                               S.ctypes.data_as(ctypes.c_void_p)), "tq_draw_params")
    return diag, S


def tq_set_profile_events(ctx, start=None, stop=None, append_start=None, append_stop=None) -> None:
    """Pass torch.cuda.Event objects (created with enable_timing=True, and recorded at
    least once so that torch has created the CUDA event) or None."""
    def h(e):
        if e is None:
            return None
        if not e.cuda_event:
            raise ValueError("event not yet created: record it once before passing it")
        return ctypes.c_void_p(e.cuda_event)
    check(lib().tq_set_profile_events(ctx, h(start), h(stop), h(append_start), h(append_stop)),
          "tq_set_profile_events")


def tq_get_device_error(ctx, stream=None) -> int:
    code = _i()
    check(lib().tq_get_device_error(ctx, _stream(stream), ctypes.byref(code)), "tq_get_device_error")
    return code.value


def tq_selftest_bounded_wait(ctx, budget_ns: int, stream=None) -> None:
    """Enqueue the bounded-wait self-test (a wait that can only run out)."""
    check(lib().tq_selftest_bounded_wait(ctx, budget_ns, _stream(stream)), "tq_selftest_bounded_wait")


# ----------------------------------------------------------------------------
# device-memory plumbing: a context handle and a cache whose planes torch owns
# ----------------------------------------------------------------------------

class Context:
    """Owns one tq_ctx (created on the current CUDA device)."""

    def __init__(self, d: int = 128, bits: int = 4, scheme="KQV", seed: int = 42, *, kivi_group=32,
                 kivi_window=128, k_per_channel=True, v_per_token=True, rotation="wht"):
        self.d, self.bits, self.seed = d, bits, seed
        self.scheme = scheme if isinstance(scheme, str) else [k for k, v in SCHEMES.items() if v == scheme][0]
        self.handle = tq_init(d, bits, self.scheme, seed)
        self.rotation = rotation
        if rotation != "wht":
            tq_set_rotation(self.handle, rotation)
        if self.scheme == "KIVI":
            tq_set_kivi(self.handle, kivi_group, kivi_window, k_per_channel, v_per_token)
            self.kivi = dict(group=kivi_group, window=kivi_window, k_per_channel=k_per_channel,
                             v_per_token=v_per_token)

    def close(self):
        if self.handle is not None:
            tq_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def _as_parameter_(self):
        return self.handle


def _pair_rows_to_records(planes: torch.Tensor, vb: int) -> torch.Tensor:
    """Value codes of [bh][block] planes (8 pair rows of 32*vb bytes each: row j holds
    tokens 2j, 2j+1; coordinate c in field 16 (c mod 8) + c // 8 of 2*vb bits, token 2j in
    the low vb bits) -> per-token code records in the key-record order (code offset n
    holds coordinate 8 ((n >> 1) & 15) + 2 (n >> 5) + (n & 1), vb bits at bit vb n).
    Runs with torch on the planes' device, a few blocks of sequence-heads at a time."""
    dev = planes.device
    bh, nblk = planes.shape[0], planes.shape[1]
    # bit position, inside the block's plane, of (token t, the coordinate at code offset n)
    t = torch.arange(16).view(16, 1)
    n = torch.arange(128).view(1, 128)
    coord = 8 * ((n >> 1) & 15) + 2 * (n >> 5) + (n & 1)
    field = 16 * (coord % 8) + coord // 8
    pos = (t // 2) * (256 * vb) + 2 * vb * field + vb * (t % 2)          # [16, 128]
    byte0, shift = (pos // 8).to(dev), (pos % 8).to(dev)
    byte1 = torch.clamp(byte0 + 1, max=256 * vb - 1)
    # output record bit q (0 .. 128 vb - 1) = bit q % vb of the code at offset q // vb
    q = torch.arange(128 * vb)
    qn, qs = (q // vb).to(dev), (q % vb).to(dev)
    weights = (1 << torch.arange(8, device=dev)).view(1, 1, 1, 8)
    out = torch.empty((bh, nblk * 16, 16 * vb), dtype=torch.uint8, device=dev)
    step = max(1, (1 << 15) // max(1, nblk))  # about 32K blocks (~1 GB of temporaries) per pass
    for r0 in range(0, bh, step):
        a = planes[r0:r0 + step].reshape(-1, 256 * vb).to(torch.int32)    # [rows, plane bytes]
        word = a[:, byte0.view(-1)] | (a[:, byte1.view(-1)] << 8)          # [rows, 16 * 128]
        codes = (word >> shift.view(1, -1)) & ((1 << vb) - 1)
        codes = codes.view(-1, 16, 128)                                    # [rows, token, offset]
        bits = (codes[:, :, qn] >> qs.view(1, 1, -1)) & 1                  # [rows, token, 128 vb]
        packed = (bits.view(-1, 16, 16 * vb, 8) * weights).sum(-1).to(torch.uint8)
        out[r0:r0 + step] = packed.view(-1, nblk * 16, 16 * vb)
    return out


class Cache:
    """A cache's arrays as torch uint8 tensors on `device` (16-byte aligned): for the TQ
    schemes one blocked records array, for KIVI its planes."""

    def __init__(self, ctx: Context, batch: int, heads_kv: int, capacity: int, device="cuda"):
        self.sizes = tq_cache_sizes_get(ctx.handle, batch, heads_kv, capacity)
        self.device = torch.device(device)
        self.batch, self.heads_kv, self.capacity = batch, heads_kv, capacity
        self.tensors = {}
        self.struct = tq_cache()
        self.struct.batch, self.struct.heads_kv, self.struct.capacity = batch, heads_kv, capacity
        self.struct.block_table, self.struct.pool_blocks = None, 0
        for p in ARRAYS:
            n = self._array_bytes(p)
            if n:
                t = torch.zeros(n, dtype=torch.uint8, device=self.device)
                assert t.data_ptr() % 16 == 0
                self.tensors[p] = t
                setattr(self.struct, p, t.data_ptr())
            else:
                setattr(self.struct, p, None)

    def _array_bytes(self, name: str) -> int:
        return getattr(self.sizes, name)

    @property
    def blocks_per_seq(self) -> int:
        return (self.capacity + BLOCK_TOKENS - 1) // BLOCK_TOKENS

    def blocks(self) -> torch.Tensor:
        """The records as [batch * heads_kv][blocks_per_seq][block_bytes] (TQ schemes)."""
        return self.tensors["records"].view(self.batch * self.heads_kv, self.blocks_per_seq, self.sizes.block_bytes)

    def plane(self, name: str) -> torch.Tensor:
        """One plane as a contiguous uint8 tensor over [batch][heads_kv][capacity] token
        slots (a copy gathered out of the blocks for the TQ schemes' record planes)."""
        if "records" not in self.tensors or name not in RECORD_PLANES:
            return self.tensors[name]
        p = RECORD_PLANES.index(name)
        tok = self.sizes.plane_bytes[p]
        if tok == 0:
            raise KeyError(name)
        off = self.sizes.plane_offset[p]
        nblk = self.blocks_per_seq
        bh = self.batch * self.heads_kv
        blocks = self.blocks()
        planes = blocks[:, :, off:off + BLOCK_TOKENS * tok]
        if name == "v_codes":
            return _pair_rows_to_records(planes, tok // 16)[:, :self.capacity].contiguous().view(-1)
        planes = planes.reshape(bh, nblk * BLOCK_TOKENS * tok)
        return planes[:, :self.capacity * tok].contiguous().view(-1)

    @property
    def record_bytes(self) -> int:
        return self.sizes.record_bytes

    def nbytes(self) -> int:
        return sum(t.numel() for t in self.tensors.values())


class PagedCache(Cache):
    """A TQ-scheme cache in the paged layout (include/tq.h, "Paged layout"): `records` is a
    pool of `pool_blocks` 16-token blocks and `block_table` (int32, on the device,
    [batch][heads_kv][ceil(capacity / 16)]) maps each sequence-head's blocks into it; -1
    marks an entry no call may reach. The table is the caller's: change it in place (in
    stream order) to remap blocks."""

    def __init__(self, ctx: Context, batch: int, heads_kv: int, capacity: int, pool_blocks: int,
                 block_table: torch.Tensor, device="cuda"):
        self.pool_blocks = int(pool_blocks)
        super().__init__(ctx, batch, heads_kv, capacity, device)
        nblk = self.blocks_per_seq
        assert block_table.dtype == torch.int32 and block_table.is_contiguous()
        assert tuple(block_table.shape) == (batch, heads_kv, nblk)
        self.block_table = block_table.to(self.device)
        self.struct.block_table = self.block_table.data_ptr()
        self.struct.pool_blocks = self.pool_blocks

    def _array_bytes(self, name: str) -> int:
        if name == "records":
            return self.pool_blocks * self.sizes.block_bytes
        return getattr(self.sizes, name)

    def blocks(self) -> torch.Tensor:
        """The sequence-heads' blocks gathered out of the pool through the table (a copy;
        unmapped entries read as zero blocks)."""
        pool = self.tensors["records"].view(self.pool_blocks, self.sizes.block_bytes)
        idx = self.block_table.view(-1).long()
        out = pool[idx.clamp(min=0)]
        out[idx < 0] = 0
        return out.view(self.batch * self.heads_kv, self.blocks_per_seq, self.sizes.block_bytes)
