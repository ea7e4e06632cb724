"""FP64 CPU oracle for SANA-Video linear attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg
may import this package.  The product path never does.

The arithmetic lives in ``lin_attn_oracle.c`` (plain loops, FP64); this module
compiles it with gcc and wraps it with ctypes.  Inputs are the BF16 bit
patterns of Q_rot, K_rot, V (``uint16`` arrays, ``[H, N, D]``) and the FP32
denominators (``[H, N]``); results are FP64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lin_attn_oracle.c")
_LIB = os.path.join(_HERE, "liblin_attn_oracle.so")
CFLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-std=c11"]

_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile the oracle into a shared library (gcc, OpenMP)."""
    cmd = ["gcc", *CFLAGS, *extra_flags, src, "-o", out]
    subprocess.run(cmd, check=True)
    return out


def _stale(lib_path: str, src: str) -> bool:
    return not os.path.exists(lib_path) or os.path.getmtime(lib_path) < os.path.getmtime(src)


def load(lib_path: str | None = None, src: str = _SRC):
    """Load (building first if missing or older than its source) the oracle library."""
    global _lib
    with _lock:
        if lib_path is None:
            if _lib is not None:
                return _lib
            if _stale(_LIB, _SRC):
                build()
            lib = _bind(ctypes.CDLL(_LIB))
            _lib = lib
            return lib
        if _stale(lib_path, src):
            build(src, lib_path)
        return _bind(ctypes.CDLL(lib_path))


def _bind(lib):
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_kv.argtypes = [i64, i64, i64, p, p, p]
    lib.oracle_kv.restype = ctypes.c_int
    lib.oracle_apply_rows.argtypes = [i64, i64, i64, p, p, p, i64, p, p]
    lib.oracle_apply_rows.restype = ctypes.c_int
    lib.oracle_apply_rows_f64den.argtypes = [i64, i64, i64, p, p, p, i64, p, p]
    lib.oracle_apply_rows_f64den.restype = ctypes.c_int
    lib.oracle_forward.argtypes = [i64, i64, i64, p, p, p, p, p]
    lib.oracle_forward.restype = ctypes.c_int
    lib.oracle_bf16_decode.argtypes = [i64, p, p]
    lib.oracle_bf16_decode.restype = None
    lib.oracle_f32_to_bf16.argtypes = [i64, p, p]
    lib.oracle_f32_to_bf16.restype = None
    lib.oracle_producer.argtypes = [i64, i64, i64, p, p, p, p, ctypes.c_double, p, p, p]
    lib.oracle_producer.restype = ctypes.c_int
    lib.oracle_softmax_attention_rows.argtypes = [i64, i64, i64, p, p, p, ctypes.c_double, i64, p, p]
    lib.oracle_softmax_attention_rows.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_num_threads.restype = None
    return lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected BF16 bit patterns as uint16, got {a.dtype}")
    return a


def _f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.float32:
        raise TypeError(f"expected float32, got {a.dtype}")
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _shape3(a: np.ndarray):
    if a.ndim != 3:
        raise ValueError("expected [H, N, D]")
    return a.shape


def num_threads(lib=None) -> int:
    return (lib or load()).oracle_num_threads()


def set_num_threads(n: int, lib=None) -> None:
    (lib or load()).oracle_set_num_threads(int(n))


def bf16_decode(bits, lib=None) -> np.ndarray:
    bits = _u16(bits)
    out = np.empty(bits.shape, np.float64)
    (lib or load()).oracle_bf16_decode(bits.size, _ptr(bits), _ptr(out))
    return out


def f32_to_bf16(values, lib=None) -> np.ndarray:
    """binary32 -> BF16 bit patterns, round to nearest, ties to even."""
    values = _f32(values)
    out = np.empty(values.shape, np.uint16)
    (lib or load()).oracle_f32_to_bf16(values.size, _ptr(values), _ptr(out))
    return out


def producer(q_bits, k_bits, cos, sin, eps=1e-6, lib=None):
    """ReLU + interleaved RoPE + normaliser: (q_rot bits, k_rot bits, den FP64 [H, N])."""
    q_bits, k_bits = _u16(q_bits), _u16(k_bits)
    H, N, D = _shape3(q_bits)
    if k_bits.shape != (H, N, D):
        raise ValueError("q and k shapes differ")
    cos, sin = _f32(cos).reshape(N, D // 2), _f32(sin).reshape(N, D // 2)
    q_rot = np.empty((H, N, D), np.uint16)
    k_rot = np.empty((H, N, D), np.uint16)
    den = np.empty((H, N), np.float64)
    rc = (lib or load()).oracle_producer(H, N, D, _ptr(q_bits), _ptr(k_bits), _ptr(cos), _ptr(sin), float(eps),
                                         _ptr(q_rot), _ptr(k_rot), _ptr(den))
    if rc:
        raise RuntimeError(f"oracle_producer failed ({rc})")
    return q_rot, k_rot, den


def kv(k_bits, v_bits, lib=None) -> np.ndarray:
    """KV[h] = K[h]^T V[h] in FP64: [H, D, D]."""
    k_bits, v_bits = _u16(k_bits), _u16(v_bits)
    H, N, D = _shape3(k_bits)
    if v_bits.shape != (H, N, D):
        raise ValueError("k and v shapes differ")
    out = np.empty((H, D, D), np.float64)
    rc = (lib or load()).oracle_kv(H, N, D, _ptr(k_bits), _ptr(v_bits), _ptr(out))
    if rc:
        raise RuntimeError(f"oracle_kv failed ({rc})")
    return out


def apply_rows(q_bits, kv_f64, den, rows=None, lib=None) -> np.ndarray:
    """Normalised second GEMM for the given flat rows (h*N + n); [len(rows), D].
    den: FP32 denominators (the layer's input) or FP64 ones (from `producer`); each is
    handled by its own C routine (oracle_apply_rows / oracle_apply_rows_f64den)."""
    q_bits = _u16(q_bits)
    H, N, D = _shape3(q_bits)
    kv_f64 = np.ascontiguousarray(kv_f64, dtype=np.float64)
    if kv_f64.shape != (H, D, D):
        raise ValueError("kv shape mismatch")
    den = np.ascontiguousarray(den).reshape(H, N)
    if den.dtype == np.float64:
        fn = (lib or load()).oracle_apply_rows_f64den
    else:
        den = _f32(den)
        fn = (lib or load()).oracle_apply_rows
    if rows is None:
        n_rows, rows_ptr = H * N, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows, rows_ptr = rows.size, _ptr(rows)
    out = np.empty((n_rows, D), np.float64)
    rc = fn(H, N, D, _ptr(q_bits), _ptr(kv_f64), _ptr(den), n_rows, rows_ptr, _ptr(out))
    if rc:
        raise RuntimeError(f"oracle apply failed ({rc})")
    return out


def forward(q_bits, k_bits, v_bits, den, lib=None) -> np.ndarray:
    """out = (Q (K^T V)) / den for every row, FP64 [H, N, D]."""
    q_bits, k_bits, v_bits = _u16(q_bits), _u16(k_bits), _u16(v_bits)
    H, N, D = _shape3(q_bits)
    if k_bits.shape != (H, N, D) or v_bits.shape != (H, N, D):
        raise ValueError("q, k, v shapes differ")
    den = _f32(den).reshape(H, N)
    out = np.empty((H, N, D), np.float64)
    rc = (lib or load()).oracle_forward(H, N, D, _ptr(q_bits), _ptr(k_bits), _ptr(v_bits),
                                        _ptr(den), _ptr(out))
    if rc:
        raise RuntimeError(f"oracle_forward failed ({rc})")
    return out


def softmax_attention_rows(q_bits, k_bits, v_bits, scale=None, rows=None, lib=None) -> np.ndarray:
    """Softmax attention (no mask, default scale 1/sqrt(D)) for flat rows h*N + n: [len, D]."""
    q_bits, k_bits, v_bits = _u16(q_bits), _u16(k_bits), _u16(v_bits)
    H, N, D = _shape3(q_bits)
    if k_bits.shape != (H, N, D) or v_bits.shape != (H, N, D):
        raise ValueError("q, k, v shapes differ")
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    if rows is None:
        n_rows, rows_ptr = H * N, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows, rows_ptr = rows.size, _ptr(rows)
    out = np.empty((n_rows, D), np.float64)
    rc = (lib or load()).oracle_softmax_attention_rows(H, N, D, _ptr(q_bits), _ptr(k_bits), _ptr(v_bits), scale,
                                                       n_rows, rows_ptr, _ptr(out))
    if rc:
        raise RuntimeError(f"oracle_softmax_attention_rows failed ({rc})")
    return out


def torch_inputs_to_numpy(layer: dict):
    """Convert a synth layer dict (torch, any device) to the oracle's numpy inputs."""
    import torch

    def bits(t):
        t = t.detach().to("cpu").contiguous()
        H, N, D = t.shape[1:]
        return t.view(torch.int16).numpy().view(np.uint16).reshape(H, N, D)

    den = layer["den"].detach().to("cpu").contiguous()
    H, N = den.shape[1:3]
    return (bits(layer["q_rot"]), bits(layer["k_rot"]), bits(layer["v"]),
            den.numpy().astype(np.float32, copy=False).reshape(H, N))
