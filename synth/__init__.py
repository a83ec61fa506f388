"""Seeded synthetic inputs shared by the GPU library's tests and the oracle.

Thin ctypes wrapper over ``synth/jepa_synth.h`` (compiled to
``synth/libjepa_synth.so``). It generates numbers only -- pixels U(-2, 2) and
the enc.* parameter recipe -- and contains none of the encoder's arithmetic.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libjepa_synth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile libjepa_synth.so in place (gcc, contraction off for bit-identical output)."""
    src = os.path.join(_HERE, "synth_capi.c")
    hdr = os.path.join(_HERE, "jepa_synth.h")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(src), os.path.getmtime(hdr))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-shared", "-fPIC", "-o", tmp, src, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        u64, f64, f32, cp = ctypes.c_uint64, ctypes.c_double, ctypes.c_float, ctypes.c_char_p
        L.jsynth_api_splitmix_at.argtypes = [u64, u64]
        L.jsynth_api_splitmix_at.restype = u64
        L.jsynth_api_fnv1a64.argtypes = [cp]
        L.jsynth_api_fnv1a64.restype = u64
        L.jsynth_api_ln.argtypes = [f64]
        L.jsynth_api_ln.restype = f64
        L.jsynth_api_cos2pi.argtypes = [f64]
        L.jsynth_api_cos2pi.restype = f64
        L.jsynth_api_normal.argtypes = [u64, cp, u64]
        L.jsynth_api_normal.restype = f64
        L.jsynth_api_fill.argtypes = [u64, cp, ctypes.c_int, f64, f64, ctypes.c_int, u64, u64, ctypes.c_void_p]
        L.jsynth_api_fill.restype = None
        L.jsynth_api_param.argtypes = [u64, cp, ctypes.c_int, u64, ctypes.c_void_p]
        L.jsynth_api_param.restype = None
        L.jsynth_api_pixels.argtypes = [u64, u64, u64, ctypes.c_void_p]
        L.jsynth_api_pixels.restype = None
        L.jsynth_api_round_bf16.argtypes = [f32]
        L.jsynth_api_round_bf16.restype = f32
        _lib = L
    return _lib


NORMAL, UNIFORM = 0, 1


def pixels(seed: int, shape) -> np.ndarray:
    """Pixels U(-2, 2) of the given shape (element order = C order of `shape`)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    if n:
        lib().jsynth_api_pixels(seed, 0, n, out.ctypes.data)
    return out.reshape(shape)


def param(seed: int, name: str, shape, bf16_matrices: bool) -> np.ndarray:
    """An enc.* parameter tensor following the synthetic init recipe."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    lib().jsynth_api_param(seed, name.encode(), int(bf16_matrices), n, out.ctypes.data)
    return out.reshape(shape)


def fill(seed: int, name: str, kind: int, a: float, b: float, shape, round_bf16=False, first=0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    lib().jsynth_api_fill(seed, name.encode(), kind, a, b, int(round_bf16), first, n, out.ctypes.data)
    return out.reshape(shape)


def splitmix_at(state: int, i: int) -> int:
    return int(lib().jsynth_api_splitmix_at(state, i))


def fnv1a64(name: str) -> int:
    return int(lib().jsynth_api_fnv1a64(name.encode()))


def ln(x: float) -> float:
    return float(lib().jsynth_api_ln(x))


def cos2pi(v: float) -> float:
    return float(lib().jsynth_api_cos2pi(v))


def round_bf16(x: float) -> float:
    return float(lib().jsynth_api_round_bf16(x))
