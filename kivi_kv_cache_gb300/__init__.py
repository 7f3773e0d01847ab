"""KIVI KV-cache compression on GB300 (sm_103a): Python binding.

Thin ctypes binding of ``libkivi_gb300.so`` (C ABI in ``include/kivi.h``).
Each ``kivi_*`` function here has the name of the C entry point it calls and
only marshals arguments: it passes the device pointers of torch CUDA tensors
and the current CUDA stream, and raises :class:`KiviError` on a non-OK status.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback. If the library has not been built, the first call
raises ``ImportError`` (build it with ``python -m kivi_kv_cache_gb300.build``).

PyTorch supplies device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "KiviError", "KiviStore", "lib", "library_path",
    "kivi_status_string", "kivi_version", "kivi_wait_timeouts", "kivi_flush_count",
    "kivi_flush_keys", "kivi_flush_values", "kivi_flush_kv", "kivi_dequant", "kivi_dequant_kv",
    "kivi_residual_append", "kivi_residual_compact", "kivi_residual_append_kv", "kivi_residual_compact_kv",
    "kivi_fake_quant_keys", "kivi_fake_quant_values", "kivi_fake_quant_kv",
    "kivi_decode_workspace_size", "kivi_decode_workspace", "kivi_decode_workspace_init",
    "kivi_decode_attend", "kivi_decode_attend_noalloc", "KiviCache",
]

# KIVI_GB300_LIB: load the library from another path (e.g. a build with other
# compile-time tuning); the default is the in-tree build.
library_path = os.environ.get("KIVI_GB300_LIB") or os.path.join(os.path.dirname(os.path.abspath(__file__)),
                                                                 "libkivi_gb300.so")

KIVI_AXIS_KEYS = 0
KIVI_AXIS_VALUES = 1

_lock = threading.Lock()
_lib = None


class KiviError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s failed: %s" % (fn, kivi_status_string(status)))


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises ImportError if it was never built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(library_path):
            raise ImportError("libkivi_gb300.so is not built (run `python -m kivi_kv_cache_gb300.build`); "
                              "there is no fallback path")
        L = ctypes.CDLL(library_path)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        IP = ctypes.POINTER(ctypes.c_int)
        sig = {
            "kivi_status_string": ([I], ctypes.c_char_p),
            "kivi_version": ([], I),
            "kivi_wait_timeouts": ([ctypes.POINTER(ctypes.c_uint), I], I),
            "kivi_flush_count": ([I, I, I], I),
            "kivi_flush_keys": ([P, I, I, I, I, I, I, I, P, P, P, I, I, IP, P], I),
            "kivi_flush_values": ([P, I, I, I, I, I, I, I, P, P, P, I, I, IP, P], I),
            "kivi_flush_kv": ([P, P, I, I, I, I, I, I, I, P, P, P, P, P, P, I, I, IP, P], I),
            "kivi_dequant": ([I, P, P, P, I, I, I, I, I, I, P, P], I),
            "kivi_dequant_kv": ([P, P, P, P, P, P, I, I, I, I, I, I, P, P, P], I),
            "kivi_residual_append_kv": ([P, P, I, I, P, P, I, I, I, I, P], I),
            "kivi_residual_compact_kv": ([P, P, I, I, I, I, I, P], I),
            "kivi_residual_append": ([P, I, I, P, I, I, I, I, P], I),
            "kivi_residual_compact": ([P, I, I, I, I, I, P], I),
            "kivi_fake_quant_keys": ([P, I, I, I, I, I, I, I, P, I, IP, P], I),
            "kivi_fake_quant_values": ([P, I, I, I, I, I, I, I, P, I, IP, P], I),
            "kivi_fake_quant_kv": ([P, P, I, I, I, I, I, I, I, P, P, I, IP, P], I),
            "kivi_decode_workspace_size": ([I, I, I, I, I, I], Z),
            "kivi_decode_plan_info": ([I, I, I, I, I, I, I, I, IP], I),
            "kivi_decode_workspace_init": ([P, Z, P], I),
            "kivi_decode_attend": ([P, P, P, P, P, P, P, I, I, P, P, I, I, I, I, I, I, I, I, F, P, P, Z, P], I),
            "kivi_cache_prefill": ([P, P, P, I, I, IP, P], I),
            "kivi_cache_append": ([P, P, P, I, I, IP, P], I),
            "kivi_cache_decode": ([P, P, I, I, I, F, P, P, Z, P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _check(fn: str, status: int):
    if status != 0:
        raise KiviError(fn, status)


def _rows(x, D: int):
    """Head stride (in tokens) of a [BH, S, D] fp16 view with dense token rows."""
    assert x.dim() == 3 and x.shape[2] == D, tuple(x.shape)
    if x.numel() == 0:  # no rows: any head stride of at least S serves
        return x.shape[1]
    assert x.stride(2) == 1 and x.stride(1) == D and x.stride(0) % D == 0, x.stride()
    return x.stride(0) // D


def kivi_status_string(status: int) -> str:
    return lib().kivi_status_string(int(status)).decode()


def kivi_version() -> int:
    return lib().kivi_version()


def kivi_wait_timeouts(reset: bool = False) -> int:
    """Bounded waits on a bulk copy that ran out since the last reset (zero in
    correct operation); synchronizes the device."""
    n = ctypes.c_uint(0)
    _check("kivi_wait_timeouts", lib().kivi_wait_timeouts(ctypes.byref(n), 1 if reset else 0))
    return n.value


def kivi_flush_count(n_res: int, residual_length: int, group_size: int = 32) -> int:
    return lib().kivi_flush_count(n_res, residual_length, group_size)


KIVI_SCALE_F16 = 0x100  # option bit of every `bits` argument: scales stored as fp16
KIVI_DECODE_STORE_READY = 0x200  # decode option: the preceding kernel on the stream does not write the store


class KiviStore:
    """Device buffers of one packed store (keys or values), allocated by torch.

    codes uint8 [BH, s_cap, D*bits/8]; keys: scale f32 (f16 with scale_f16) /
    zero f16 [BH, s_cap/G, D]; values: the same dtypes, [BH, s_cap, D/G].
    """

    def __init__(self, axis: int, BH: int, s_cap: int, D: int = 128, group_size: int = 32,
                 bits: int = 4, device="cuda", scale_f16: bool = False):
        import torch
        assert s_cap % group_size == 0
        self.axis, self.BH, self.s_cap, self.D, self.G, self.bits = axis, BH, s_cap, D, group_size, bits
        self.scale_f16 = scale_f16
        self.codes = torch.zeros((BH, s_cap, D * bits // 8), dtype=torch.uint8, device=device)
        meta = (BH, s_cap // group_size, D) if axis == KIVI_AXIS_KEYS else (BH, s_cap, D // group_size)
        self.scale = torch.zeros(meta, dtype=torch.float16 if scale_f16 else torch.float32, device=device)
        self.zero = torch.zeros(meta, dtype=torch.float16, device=device)

    @property
    def abi_bits(self) -> int:
        """The `bits` argument of the C ABI: the width plus the scale option."""
        return self.bits | (KIVI_SCALE_F16 if self.scale_f16 else 0)

    def nbytes_per_token(self) -> float:
        return (self.codes[0, 0].numel() + (self.scale.numel() * 4 + self.zero.numel() * 2)
                / (self.BH * self.s_cap))


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def _flush(name: str, x, residual_length: int, store: KiviStore, s_off: int, n_tokens, stream):
    S = x.shape[1] if n_tokens is None else n_tokens
    n = ctypes.c_int(0)
    st = getattr(lib(), name)(_ptr(x), x.shape[0], S, _rows(x, store.D), store.D, store.G, store.abi_bits,
                              residual_length, _ptr(store.codes), _ptr(store.scale), _ptr(store.zero),
                              s_off, store.s_cap, ctypes.byref(n), _stream(stream))
    _check(name, st)
    return n.value


def kivi_flush_keys(x, residual_length: int, store: KiviStore, s_off: int = 0, n_tokens=None,
                    stream=None) -> int:
    """Quantize the oldest kivi_flush_count(S, R, G) tokens of x [BH, S, D] fp16
    into the key store at token offset s_off; returns the number flushed."""
    return _flush("kivi_flush_keys", x, residual_length, store, s_off, n_tokens, stream)


def kivi_flush_values(x, residual_length: int, store: KiviStore, s_off: int = 0, n_tokens=None,
                      stream=None) -> int:
    return _flush("kivi_flush_values", x, residual_length, store, s_off, n_tokens, stream)


def kivi_flush_kv(k, v, residual_length: int, kstore: KiviStore, vstore: KiviStore, s_off: int = 0,
                  n_tokens=None, stream=None) -> int:
    """Key and value flush of the same tokens in one launch."""
    S = k.shape[1] if n_tokens is None else n_tokens
    stride = _rows(k, kstore.D)
    assert _rows(v, vstore.D) == stride and v.shape[0] == k.shape[0]
    n = ctypes.c_int(0)
    assert kstore.scale_f16 == vstore.scale_f16
    st = lib().kivi_flush_kv(_ptr(k), _ptr(v), k.shape[0], S, stride, kstore.D, kstore.G, kstore.abi_bits,
                             residual_length, _ptr(kstore.codes), _ptr(kstore.scale), _ptr(kstore.zero),
                             _ptr(vstore.codes), _ptr(vstore.scale), _ptr(vstore.zero), s_off,
                             kstore.s_cap, ctypes.byref(n), _stream(stream))
    _check("kivi_flush_kv", st)
    return n.value


def kivi_dequant(store: KiviStore, S: int, out=None, stream=None):
    """fp16 [BH, S, D] reconstruction of tokens [0, S) of a store."""
    import torch
    if out is None:
        out = torch.empty((store.BH, S, store.D), dtype=torch.float16, device=store.codes.device)
    st = lib().kivi_dequant(store.axis, _ptr(store.codes), _ptr(store.scale), _ptr(store.zero), store.BH,
                            S, store.D, store.G, store.abi_bits, store.s_cap, _ptr(out), _stream(stream))
    _check("kivi_dequant", st)
    return out


def kivi_dequant_kv(kstore: KiviStore, vstore: KiviStore, S: int, kout=None, vout=None, stream=None):
    """Key and value fp16 reconstructions of tokens [0, S) in one launch."""
    assert kstore.scale_f16 == vstore.scale_f16, "one scale storage for both stores"
    import torch
    if kout is None:
        kout = torch.empty((kstore.BH, S, kstore.D), dtype=torch.float16, device=kstore.codes.device)
    if vout is None:
        vout = torch.empty((vstore.BH, S, vstore.D), dtype=torch.float16, device=vstore.codes.device)
    st = lib().kivi_dequant_kv(_ptr(kstore.codes), _ptr(kstore.scale), _ptr(kstore.zero), _ptr(vstore.codes),
                               _ptr(vstore.scale), _ptr(vstore.zero), kstore.BH, S, kstore.D, kstore.G,
                               kstore.abi_bits, kstore.s_cap, _ptr(kout), _ptr(vout), _stream(stream))
    _check("kivi_dequant_kv", st)
    return kout, vout


def kivi_residual_append_kv(ksrc, vsrc, kres, vres, n_res: int, n_new=None, stream=None):
    """Append n_new token rows of K and V behind the n_res live rows of their windows."""
    n = ksrc.shape[1] if n_new is None else n_new
    stride = _rows(ksrc, kres.shape[2])
    assert _rows(vsrc, vres.shape[2]) == stride and kres.shape == vres.shape
    st = lib().kivi_residual_append_kv(_ptr(ksrc), _ptr(vsrc), stride, n, _ptr(kres), _ptr(vres), kres.shape[0],
                                       kres.shape[1], kres.shape[2], n_res, _stream(stream))
    _check("kivi_residual_append_kv", st)
    return n_res + n


def kivi_residual_compact_kv(kres, vres, n_res: int, n_drop: int, stream=None):
    assert kres.shape == vres.shape
    st = lib().kivi_residual_compact_kv(_ptr(kres), _ptr(vres), kres.shape[0], kres.shape[1], kres.shape[2],
                                        n_res, n_drop, _stream(stream))
    _check("kivi_residual_compact_kv", st)
    return n_res - n_drop


def kivi_residual_append(src, res, n_res: int, n_new=None, stream=None):
    """Copy n_new token rows of src [BH, *, D] behind the n_res live rows of res."""
    n = src.shape[1] if n_new is None else n_new
    st = lib().kivi_residual_append(_ptr(src), _rows(src, res.shape[2]), n, _ptr(res), res.shape[0],
                                    res.shape[1], res.shape[2], n_res, _stream(stream))
    _check("kivi_residual_append", st)
    return n_res + n


def kivi_residual_compact(res, n_res: int, n_drop: int, stream=None):
    st = lib().kivi_residual_compact(_ptr(res), res.shape[0], res.shape[1], res.shape[2], n_res, n_drop,
                                     _stream(stream))
    _check("kivi_residual_compact", st)
    return n_res - n_drop


def _fake_quant(fn: str, x, residual_length: int, out, G: int, bits: int, stream):
    import torch
    BH, S, D = x.shape
    if out is None:
        out = torch.empty((BH, S, D), dtype=torch.float16, device=x.device)
    n = ctypes.c_int(-1)
    st = getattr(lib(), fn)(_ptr(x), BH, S, _rows(x, D), D, G, bits, residual_length, _ptr(out), _rows(out, D),
                            ctypes.byref(n), _stream(stream))
    _check(fn, st)
    return out, n.value


def kivi_fake_quant_keys(x, residual_length: int, out=None, G: int = 32, bits: int = 4, stream=None,
                         scale_f16: bool = False):
    """Fake-quantized keys x [BH, S, D] fp16 -> (out, n_quantized); out may be x (in place)."""
    return _fake_quant("kivi_fake_quant_keys", x, residual_length, out, G,
                       bits | (KIVI_SCALE_F16 if scale_f16 else 0), stream)


def kivi_fake_quant_values(x, residual_length: int, out=None, G: int = 32, bits: int = 4, stream=None,
                           scale_f16: bool = False):
    """Fake-quantized values x [BH, S, D] fp16 -> (out, n_quantized); out may be x (in place)."""
    return _fake_quant("kivi_fake_quant_values", x, residual_length, out, G,
                       bits | (KIVI_SCALE_F16 if scale_f16 else 0), stream)


def kivi_fake_quant_kv(k, v, residual_length: int, kout=None, vout=None, G: int = 32, bits: int = 4,
                       stream=None, scale_f16: bool = False):
    """Fake quantization of keys and values of equal geometry -> (kout, vout, n_quantized)."""
    import torch
    BH, S, D = k.shape
    if kout is None:
        kout = torch.empty((BH, S, D), dtype=torch.float16, device=k.device)
    if vout is None:
        vout = torch.empty((BH, S, D), dtype=torch.float16, device=v.device)
    stride = _rows(k, D)
    assert _rows(v, D) == stride and _rows(kout, D) == _rows(vout, D)
    n = ctypes.c_int(-1)
    bits = bits | (KIVI_SCALE_F16 if scale_f16 else 0)
    st = lib().kivi_fake_quant_kv(_ptr(k), _ptr(v), BH, S, stride, D, G, bits, residual_length, _ptr(kout), _ptr(vout),
                                  _rows(kout, D), ctypes.byref(n), _stream(stream))
    _check("kivi_fake_quant_kv", st)
    return kout, vout, n.value


def kivi_decode_workspace_size(B: int, Hq: int, Hkv: int, S_q: int, n_res: int, D: int = 128) -> int:
    return lib().kivi_decode_workspace_size(B, Hq, Hkv, S_q, n_res, D)


def kivi_decode_plan_info(B: int, Hq: int, Hkv: int, S_q: int, n_res: int, D: int = 128, G: int = 32,
                          bits: int = 4, scale_f16: bool = False) -> dict:
    """The split plan kivi_decode_attend takes for these arguments (host only)."""
    info = (ctypes.c_int * 7)()
    st = lib().kivi_decode_plan_info(B, Hq, Hkv, S_q, n_res, D, G, bits | (KIVI_SCALE_F16 if scale_f16 else 0),
                                     ctypes.cast(info, ctypes.POINTER(ctypes.c_int)))
    _check("kivi_decode_plan_info", st)
    keys = ("pair_kernel", "n_split", "tiles_per_warp", "warps_per_cta", "q_sub", "n_tiles", "tiles_per_split")
    return dict(zip(keys, list(info)))


def kivi_decode_workspace_init(workspace, stream=None) -> None:
    """Zero the merge counters of a fresh workspace (once, before its first decode)."""
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("kivi_decode_workspace_init", lib().kivi_decode_workspace_init(_ptr(workspace), nbytes, _stream(stream)))


def kivi_decode_workspace(nbytes: int, device):
    """A decode workspace of nbytes (at least 16), ready for its first call."""
    import torch
    ws = torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)
    kivi_decode_workspace_init(ws)
    return ws


def kivi_decode_attend(q, kstore: KiviStore, vstore: KiviStore, S_q: int, k_res, v_res, n_res: int,
                       Hkv: int, sm_scale: float, out=None, workspace=None, stream=None, store_ready: bool = False):
    """Single-token decode: q [B, Hq, D] fp16 -> out [B, Hq, D] fp32.
    store_ready: KIVI_DECODE_STORE_READY (the kernel before this call on the
    stream does not write the stores)."""
    import torch
    assert kstore.scale_f16 == vstore.scale_f16, "one scale storage for both stores"
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    need = kivi_decode_workspace_size(B, Hq, Hkv, S_q, n_res, D)
    if workspace is None and need > 0:
        workspace = kivi_decode_workspace(need, q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    res_cap = 0
    if k_res is not None:
        res_cap = _rows(k_res, D)  # head stride in tokens: a view into a larger cache works
        assert _rows(v_res, D) == res_cap
    st = lib().kivi_decode_attend(
        _ptr(q), _ptr(kstore.codes), _ptr(kstore.scale), _ptr(kstore.zero),
        _ptr(vstore.codes), _ptr(vstore.scale), _ptr(vstore.zero), S_q, kstore.s_cap,
        _ptr(k_res), _ptr(v_res), n_res, res_cap, B, Hq, Hkv, D, kstore.G,
        kstore.abi_bits | (KIVI_DECODE_STORE_READY if store_ready else 0),
        float(sm_scale), _ptr(out), _ptr(workspace), wbytes, _stream(stream))
    _check("kivi_decode_attend", st)
    return out


_noalloc_fn = None


def kivi_decode_attend_noalloc(q, kstore: KiviStore, vstore: KiviStore, S_q: int, k_res, v_res, n_res: int,
                               Hkv: int, sm_scale: float, out=None, stream=None):
    """The decode of kivi_decode_attend without a workspace argument: the split
    scratch lives in a library-owned 8 MiB device array (for callers that may
    not allocate device memory when they decode). Calls that overlap on the GPU
    race on that array; make the first call on a device before any stream
    capture."""
    assert kstore.scale_f16 == vstore.scale_f16, "one scale storage for both stores"
    global _noalloc_fn
    import torch
    if _noalloc_fn is None:
        fn = lib().kivi_decode_attend_noalloc
        P, I = ctypes.c_void_p, ctypes.c_int
        fn.argtypes = [P, P, P, P, P, P, P, I, I, P, P, I, I, I, I, I, I, I, I, ctypes.c_float, P, P]
        fn.restype = I
        _noalloc_fn = fn
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
    res_cap = 0
    if k_res is not None:
        res_cap = _rows(k_res, D)
        assert _rows(v_res, D) == res_cap
    st = _noalloc_fn(
        _ptr(q), _ptr(kstore.codes), _ptr(kstore.scale), _ptr(kstore.zero),
        _ptr(vstore.codes), _ptr(vstore.scale), _ptr(vstore.zero), S_q, kstore.s_cap,
        _ptr(k_res), _ptr(v_res), n_res, res_cap, B, Hq, Hkv, D, kstore.G, kstore.abi_bits,
        float(sm_scale), _ptr(out), _stream(stream))
    _check("kivi_decode_attend_noalloc", st)
    return out


class _CacheStruct(ctypes.Structure):
    """The C struct kivi_cache (include/kivi.h), field for field."""
    _fields_ = [("BH", ctypes.c_int), ("D", ctypes.c_int), ("group_size", ctypes.c_int), ("bits", ctypes.c_int),
                ("residual_length", ctypes.c_int), ("s_cap", ctypes.c_int), ("res_cap", ctypes.c_int),
                ("kcodes", ctypes.c_void_p), ("kscale", ctypes.c_void_p), ("kzero", ctypes.c_void_p),
                ("vcodes", ctypes.c_void_p), ("vscale", ctypes.c_void_p), ("vzero", ctypes.c_void_p),
                ("k_res", ctypes.c_void_p), ("v_res", ctypes.c_void_p), ("S_q", ctypes.c_int), ("n_res", ctypes.c_int),
                ("store_written", ctypes.c_int), ("res_off", ctypes.c_int)]


class KiviCache:
    """One attention layer's KIVI cache (C struct kivi_cache): packed key and
    value stores of s_cap tokens, fp16 key and value windows of res_cap
    tokens (default residual_length + group_size), and the counters S_q,
    n_res and res_off (the window's first row), which the C calls update.
    torch allocates the buffers."""

    def __init__(self, BH: int, s_cap: int, D: int = 128, group_size: int = 32, bits: int = 4,
                 residual_length: int = 128, res_cap=None, device="cuda", scale_f16: bool = False):
        import torch
        res_cap = residual_length + group_size if res_cap is None else res_cap
        self.kstore = KiviStore(0, BH, s_cap, D, group_size, bits, device=device, scale_f16=scale_f16)
        self.vstore = KiviStore(1, BH, s_cap, D, group_size, bits, device=device, scale_f16=scale_f16)
        self.k_res = torch.zeros((BH, res_cap, D), dtype=torch.float16, device=device)
        self.v_res = torch.zeros_like(self.k_res)
        ks, vs = self.kstore, self.vstore
        self.c = _CacheStruct(BH, D, group_size, ks.abi_bits, residual_length, s_cap, res_cap,
                              ks.codes.data_ptr(), ks.scale.data_ptr(), ks.zero.data_ptr(),
                              vs.codes.data_ptr(), vs.scale.data_ptr(), vs.zero.data_ptr(),
                              self.k_res.data_ptr(), self.v_res.data_ptr(), 0, 0, 0, 0)

    @property
    def S_q(self) -> int:
        return self.c.S_q

    @property
    def n_res(self) -> int:
        return self.c.n_res

    @property
    def res_off(self) -> int:
        return self.c.res_off

    def state(self):
        """The counters (S_q, n_res, res_off, store_written), e.g. to restore
        them after a graph capture."""
        return self.c.S_q, self.c.n_res, self.c.res_off, self.c.store_written

    def set_state(self, S_q: int, n_res: int, res_off: int = 0, store_written: int = 0) -> None:
        self.c.S_q, self.c.n_res, self.c.res_off, self.c.store_written = S_q, n_res, res_off, store_written

    def window(self):
        """Views of the live window rows: (k, v) [BH, n_res, D] fp16."""
        o, n = self.c.res_off, self.c.n_res
        return self.k_res[:, o:o + n], self.v_res[:, o:o + n]

    def prefill(self, k, v, n_tokens=None, stream=None) -> int:
        """kivi_cache_prefill of k, v [BH, S, D] fp16; returns the tokens flushed."""
        S = k.shape[1] if n_tokens is None else n_tokens
        stride = _rows(k, self.c.D)
        assert _rows(v, self.c.D) == stride
        n = ctypes.c_int(0)
        _check("kivi_cache_prefill", lib().kivi_cache_prefill(ctypes.byref(self.c), _ptr(k), _ptr(v), stride, S,
                                                             ctypes.byref(n), _stream(stream)))
        return n.value

    def append(self, k, v, n_new=None, stream=None) -> int:
        """kivi_cache_append of k, v [BH, n, D] fp16; returns the tokens flushed."""
        n_new = k.shape[1] if n_new is None else n_new
        stride = _rows(k, self.c.D)
        assert _rows(v, self.c.D) == stride
        n = ctypes.c_int(0)
        _check("kivi_cache_append", lib().kivi_cache_append(ctypes.byref(self.c), _ptr(k), _ptr(v), stride, n_new,
                                                           ctypes.byref(n), _stream(stream)))
        return n.value

    def decode(self, q, Hkv: int, sm_scale: float, out=None, workspace=None, stream=None):
        """kivi_cache_decode: q [B, Hq, D] fp16 -> out [B, Hq, D] fp32."""
        import torch
        B, Hq, D = q.shape
        if out is None:
            out = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device)
        if workspace is None:
            need = kivi_decode_workspace_size(B, Hq, Hkv, self.c.S_q, self.c.n_res, D)
            workspace = kivi_decode_workspace(need, q.device) if need > 0 else None
        wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _check("kivi_cache_decode", lib().kivi_cache_decode(ctypes.byref(self.c), _ptr(q), B, Hq, Hkv,
                                                           float(sm_scale), _ptr(out), _ptr(workspace), wbytes,
                                                           _stream(stream)))
        return out
