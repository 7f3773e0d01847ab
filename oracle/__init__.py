"""Plain CPU oracle for KIVI flush / dequantize / decode-attend.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The CUDA product path (``kivi_kv_cache_gb300``) never imports it and
shares no code with it.

The arithmetic lives in ``kivi_oracle.c`` (plain C, fp32 steps as separate IEEE
operations, float64 attention); this module only compiles it with gcc and
marshals numpy arrays. fp16 data travels as ``np.float16`` arrays whose bit
patterns are passed straight to the C code.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kivi_oracle.c")
_LIB = os.path.join(_HERE, "libkivi_oracle.so")
_lock = threading.Lock()
_lib = None

# Strict IEEE flags: no contraction into FMA, no fast-math, no excess precision.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-fexcess-precision=standard", "-frounding-math"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libkivi_oracle.so`` (gcc, no GPU)."""
    with _lock:
        stale = (not os.path.exists(_LIB)
                 or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
                 or os.path.getmtime(_LIB) < os.path.getmtime(os.path.join(_HERE, "kivi_oracle.h")))
        if force or stale:
            tmp = _LIB + ".%d.tmp" % os.getpid()
            cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        # KIVI_ORACLE_LIB points the pin tests at a deliberately broken copy of
        # the oracle (tests/test_oracle_mutants.py); normally it is unset.
        path = os.environ.get("KIVI_ORACLE_LIB") or build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.orc_half_to_float.argtypes = [ctypes.c_uint16]
        lib.orc_half_to_float.restype = ctypes.c_float
        lib.orc_float_to_half.argtypes = [ctypes.c_float]
        lib.orc_float_to_half.restype = ctypes.c_uint16
        lib.orc_half_to_float_n.argtypes = [P, P, ctypes.c_long]
        lib.orc_float_to_half_n.argtypes = [P, P, ctypes.c_long]
        lib.orc_flush_count.argtypes = [I, I, I]
        lib.orc_flush_count.restype = I
        lib.orc_quantize_group.argtypes = [P, I, I, P, P, P]
        lib.orc_pack_codes.argtypes = [P, I, I, P]
        lib.orc_unpack_codes.argtypes = [P, I, I, P]
        lib.orc_flush_keys.argtypes = [P, I, I, I, I, I, I, P, P, P, I, I]
        lib.orc_flush_values.argtypes = [P, I, I, I, I, I, I, P, P, P, I, I]
        lib.orc_recon_f32.argtypes = [I, P, P, P, I, I, I, I, I, I, P]
        lib.orc_dequant.argtypes = [I, P, P, P, I, I, I, I, I, I, P]
        lib.orc_residual_append.argtypes = [P, I, I, I, I, P, I, I]
        lib.orc_residual_compact.argtypes = [P, I, I, I, I, I]
        lib.orc_decode_attend.argtypes = [P, P, P, P, P, P, P, I, I, P, P, I, I,
                                          I, I, I, I, I, I, ctypes.c_double, P]
        for name in ("orc_half_to_float_n", "orc_float_to_half_n", "orc_quantize_group",
                     "orc_pack_codes", "orc_unpack_codes", "orc_flush_keys",
                     "orc_flush_values", "orc_recon_f32", "orc_dequant",
                     "orc_residual_append", "orc_residual_compact", "orc_decode_attend"):
            getattr(lib, name).restype = None
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _f16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.float16, a.dtype
    return a


# --------------------------------------------------------------------------
# fp16 conversions
# --------------------------------------------------------------------------

def half_to_float(h: np.ndarray) -> np.ndarray:
    """binary16 -> binary32 by the oracle's own bit-level conversion."""
    h = np.ascontiguousarray(h).view(np.uint16)
    out = np.empty(h.shape, np.float32)
    _load().orc_half_to_float_n(_p(h), _p(out), h.size)
    return out


def float_to_half(f: np.ndarray) -> np.ndarray:
    """binary32 -> binary16 (round to nearest even), returned as np.float16."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, np.uint16)
    _load().orc_float_to_half_n(_p(f), _p(out), f.size)
    return out.view(np.float16)


# --------------------------------------------------------------------------
# quantizer pieces
# --------------------------------------------------------------------------

def flush_count(n_res: int, residual_length: int, group_size: int) -> int:
    return int(_load().orc_flush_count(n_res, residual_length, group_size))


def quantize_group(v, bits: int):
    """One group of fp32 values -> (codes uint8[n], scale f32, zero f32).
    bits may carry SCALE_F16 (the returned scale is then the binary16 one)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    codes = np.empty(v.size, np.uint8)
    s = np.zeros(1, np.float32)
    z = np.zeros(1, np.float32)
    _load().orc_quantize_group(_p(v), v.size, bits, _p(codes), _p(s), _p(z))
    return codes, s[0], z[0]


def pack_codes(codes, bits: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.size * bits // 8, np.uint8)
    _load().orc_pack_codes(_p(codes), codes.size, bits, _p(out))
    return out


def unpack_codes(packed, n: int, bits: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.empty(n, np.uint8)
    _load().orc_unpack_codes(_p(packed), n, bits, _p(out))
    return out


# --------------------------------------------------------------------------
# store
# --------------------------------------------------------------------------

# Option bit of the C oracle's `bits` arguments: scales stored as binary16.
SCALE_F16 = 0x100


class Store:
    """Quantized store for one tensor (keys or values), host numpy arrays.

    codes  uint8   [BH, s_cap, D*bits/8]
    scale  float32 (or float16 with scale_f16) [BH, s_cap/G, D] (keys) or
           [BH, s_cap, D/G] (values)
    zero   float16 same shape as scale
    """

    def __init__(self, axis: int, BH: int, s_cap: int, D: int, G: int, bits: int, scale_f16: bool = False):
        assert s_cap % G == 0
        self.axis, self.BH, self.s_cap, self.D, self.G, self.bits = axis, BH, s_cap, D, G, bits
        self.scale_f16 = scale_f16
        self.codes = np.zeros((BH, s_cap, D * bits // 8), np.uint8)
        meta = (BH, s_cap // G, D) if axis == 0 else (BH, s_cap, D // G)
        self.scale = np.zeros(meta, np.float16 if scale_f16 else np.float32)
        self.zero = np.zeros(meta, np.float16)

    @property
    def c_bits(self) -> int:
        """The `bits` argument of the C oracle: width plus the scale option."""
        return self.bits | (SCALE_F16 if self.scale_f16 else 0)


def flush(axis: int, x, n_flush: int, store: Store, s_off: int = 0, t0: int = 0):
    """Quantize tokens [t0, t0 + n_flush) of x [BH, S, D] fp16 into ``store`` at
    store token offset s_off (x is read with S tokens between heads)."""
    x = _f16(x)
    BH, S, D = x.shape
    assert 0 <= t0 and t0 + n_flush <= S
    fn = _load().orc_flush_keys if axis == 0 else _load().orc_flush_values
    ptr = ctypes.c_void_p(x.ctypes.data + t0 * D * 2)
    fn(ptr, BH, S, n_flush, D, store.G, store.c_bits, _p(store.codes),
       _p(store.scale), _p(store.zero.view(np.uint16)), s_off, store.s_cap)
    return store


def recon_f32(store: Store, S: int) -> np.ndarray:
    out = np.empty((store.BH, S, store.D), np.float32)
    _load().orc_recon_f32(store.axis, _p(store.codes), _p(store.scale),
                          _p(store.zero.view(np.uint16)), store.BH, S, store.D,
                          store.G, store.c_bits, store.s_cap, _p(out))
    return out


def dequant(store: Store, S: int) -> np.ndarray:
    out = np.empty((store.BH, S, store.D), np.uint16)
    _load().orc_dequant(store.axis, _p(store.codes), _p(store.scale),
                        _p(store.zero.view(np.uint16)), store.BH, S, store.D,
                        store.G, store.c_bits, store.s_cap, _p(out))
    return out.view(np.float16)


def residual_append(res, n_res: int, src, n_new: int, src_bh_stride=None):
    res = _f16(res)
    src = _f16(src)
    BH, cap, D = res.shape
    stride = src.shape[1] if src_bh_stride is None else src_bh_stride
    _load().orc_residual_append(_p(res.view(np.uint16)), BH, cap, D, n_res,
                                _p(src.view(np.uint16)), stride, n_new)
    return res


def residual_compact(res, n_res: int, n_drop: int):
    res = _f16(res)
    BH, cap, D = res.shape
    _load().orc_residual_compact(_p(res.view(np.uint16)), BH, cap, D, n_res, n_drop)
    return res


def decode_attend(q, kstore: Store, vstore: Store, S_q: int, k_res, v_res, n_res: int,
                  Hkv: int, sm_scale: float) -> np.ndarray:
    """q [B, Hq, D] fp16; residual [B*Hkv, res_cap, D] fp16 -> out [B, Hq, D] float64."""
    assert kstore.scale_f16 == vstore.scale_f16, "one scale storage for both stores"
    q = _f16(q)
    k_res = _f16(k_res)
    v_res = _f16(v_res)
    B, Hq, D = q.shape
    res_cap = k_res.shape[1]
    out = np.empty((B, Hq, D), np.float64)
    _load().orc_decode_attend(
        _p(q.view(np.uint16)),
        _p(kstore.codes), _p(kstore.scale), _p(kstore.zero.view(np.uint16)),
        _p(vstore.codes), _p(vstore.scale), _p(vstore.zero.view(np.uint16)),
        S_q, kstore.s_cap,
        _p(k_res.view(np.uint16)), _p(v_res.view(np.uint16)), n_res, res_cap,
        B, Hq, Hkv, D, kstore.G, kstore.c_bits, float(sm_scale), _p(out))
    return out
