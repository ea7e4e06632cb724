"""Python binding of liblin_attn.so (ctypes).  Argument marshalling only: every step of
the layer runs in the library's CUDA kernels; torch supplies device memory and streams.

Importing this module loads the library and raises ImportError if it has not been built
(``python -c "import __graft_entry__ as g; g.build()"``).  There is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblin_attn.so")

MODE_HIGH, MODE_LOSSLESS = 0, 1
LAYOUT_HND, LAYOUT_NHD = 0, 1
OUT_F32, OUT_BF16 = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_CUDA, ERR_OOM, ERR_TIMEOUT = range(7)

EXPORTS = (
    "lin_attn_create", "lin_attn_destroy", "lin_attn_forward", "lin_attn_forward_layout", "lin_attn_forward_host",
    "lin_attn_debug_kv", "lin_attn_device_status", "lin_attn_kv_plan",
    "lin_attn_set_stage_events", "lin_attn_error_string", "lin_attn_last_error", "lin_attn_version",
    "lin_attn_forward_noalloc", "lin_attn_forward_fused", "lin_attn_anchor_forward", "lin_attn_forward_fused_layout",
    "lin_attn_set_wait_limit", "lin_attn_noalloc_status", "lin_attn_forward_fused_host",
)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first (__graft_entry__.build())")
    lib = ctypes.CDLL(LIB_PATH)
    p, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    sig = {
        "lin_attn_create": ([ctypes.POINTER(p), i32, i64, i32, i32], i32),
        "lin_attn_destroy": ([p], i32),
        "lin_attn_forward": ([p, p, p, p, p, p, i32, i64, i32, p], i32),
        "lin_attn_forward_layout": ([p, p, p, p, p, p, i32, i64, i32, i32, p], i32),
        "lin_attn_forward_host": ([p, p, p, p, p, p, i32, i64, i32, p], i32),
        "lin_attn_debug_kv": ([p, p, p], i32),
        "lin_attn_device_status": ([p, p], i32),
        "lin_attn_kv_plan": ([i32, i64, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)], i32),
        "lin_attn_set_stage_events": ([p, ctypes.POINTER(p), i32], i32),
        "lin_attn_set_wait_limit": ([p, ctypes.c_uint64], i32),
        "lin_attn_error_string": ([i32], ctypes.c_char_p),
        "lin_attn_last_error": ([], ctypes.c_char_p),
        "lin_attn_version": ([], i32),
        "lin_attn_forward_noalloc": ([p, p, p, p, p, i32, i32, i64, i32, i32, p], i32),
        "lin_attn_noalloc_status": ([p], i32),
        "lin_attn_forward_fused": ([p, p, p, p, p, p, p, i32, i64, i32, p], i32),
        "lin_attn_forward_fused_layout": ([p, p, p, p, p, p, p, i32, i64, i32, i32, p], i32),
        "lin_attn_forward_fused_host": ([p, p, p, p, p, p, p, i32, i64, i32, p], i32),
        "lin_attn_anchor_forward": ([p, p, p, p, p, i32, i64, ctypes.c_float, p], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()


class LinAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = lib.lin_attn_last_error().decode()
        super().__init__(f"{where}: {lib.lin_attn_error_string(status).decode()} ({status}): {detail}")


def _check(status: int, where: str):
    if status != OK:
        raise LinAttnError(status, where)


def error_string(status: int) -> str:
    return lib.lin_attn_error_string(status).decode()


def kv_plan(heads: int, n_tokens: int, mode="high"):
    """(chunks, max partials per head) of the KV reduction for this shape and tier."""
    c, m = ctypes.c_int(), ctypes.c_int()
    _check(lib.lin_attn_kv_plan(heads, n_tokens, _mode(mode), ctypes.byref(c), ctypes.byref(m)), "lin_attn_kv_plan")
    return c.value, m.value


def _mode(mode) -> int:
    if mode in ("high", MODE_HIGH):
        return MODE_HIGH
    if mode in ("lossless", MODE_LOSSLESS):
        return MODE_LOSSLESS
    raise ValueError(f"mode must be 'high' or 'lossless', got {mode!r}")


def _out_code(dtype) -> int:
    if dtype == torch.float32:
        return OUT_F32
    if dtype == torch.bfloat16:
        return OUT_BF16
    raise TypeError(f"out dtype must be float32 or bfloat16, got {dtype}")


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def forward_noalloc(q_rot, k_rot, v, normalizer, out, mode="high", stream=None):
    """Layer call that allocates no device memory (library-owned fixed scratch on the
    inputs' device); for callers that cannot allocate.  ``out`` must be given."""
    for name, t in (("q_rot", q_rot), ("k_rot", k_rot), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")
    if q_rot.dim() != 4 or q_rot.shape[0] != 1 or q_rot.shape != k_rot.shape or q_rot.shape != v.shape:
        raise ValueError("q_rot, k_rot, v must share one [1, H, N, D] shape")
    _, H, N, D = q_rot.shape
    if normalizer.dtype != torch.float32 or tuple(normalizer.shape) != (1, H, N, 1) or not normalizer.is_contiguous():
        raise ValueError(f"normalizer must be a contiguous float32 [1, {H}, {N}, 1] tensor")
    if out.shape != q_rot.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous [1, H, N, D] tensor")
    code = _out_code(out.dtype)
    dev = q_rot.device
    for name, t in (("k_rot", k_rot), ("v", v), ("normalizer", normalizer), ("out", out)):
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}; every tensor must be on {dev}")
    # The entry point runs on the calling thread's current device (its scratch, set-up and
    # the stream all belong to it): make that the tensors' device for the call.
    with torch.cuda.device(dev):
        st = lib.lin_attn_forward_noalloc(q_rot.data_ptr(), k_rot.data_ptr(), v.data_ptr(), normalizer.data_ptr(),
                                          out.data_ptr(), code, H, N, D, _mode(mode), _stream_handle(stream, dev))
    _check(st, "lin_attn_forward_noalloc")
    return out


def noalloc_status(device=None, stream=None) -> int:
    """Waits for ``stream`` and returns the status of the no-alloc calls on ``device`` since
    the previous query (OK, or ERR_TIMEOUT if a kernel gave up waiting), clearing it."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        st = lib.lin_attn_noalloc_status(_stream_handle(stream, dev))
    if st not in (OK, ERR_TIMEOUT):
        _check(st, "lin_attn_noalloc_status")
    return st


class LinAttn:
    """One context: scratch for layers of ``heads`` x up to ``max_tokens`` x ``head_dim``."""

    def __init__(self, heads: int, max_tokens: int, head_dim: int, device=None):
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        if dev.type != "cuda":
            raise ValueError("LinAttn needs a CUDA device")
        self.device = torch.device("cuda", dev.index if dev.index is not None else torch.cuda.current_device())
        self.heads, self.max_tokens, self.head_dim = heads, max_tokens, head_dim
        h = ctypes.c_void_p()
        _check(lib.lin_attn_create(ctypes.byref(h), heads, max_tokens, head_dim, self.device.index), "lin_attn_create")
        self._h = h

    # ------------------------------------------------------------------ checks
    def _check_inputs(self, q, k, v, den, want_device, layout="hnd"):
        for name, t in (("q_rot", q), ("k_rot", k), ("v", v)):
            if t.dtype != torch.bfloat16:
                raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
        if den.dtype != torch.float32:
            raise TypeError(f"normalizer must be float32, got {den.dtype}")
        if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
            raise ValueError("q_rot, k_rot, v must share one 4-D shape")
        if layout == "hnd":
            B, H, N, D = q.shape
        elif layout == "nhd":
            B, N, H, D = q.shape
        else:
            raise ValueError(f"layout must be 'hnd' or 'nhd', got {layout!r}")
        if B != 1:
            raise ValueError(f"batch must be 1, got {B}")
        if H != self.heads or D != self.head_dim:
            raise ValueError(f"context is for H={self.heads}, D={self.head_dim}; got H={H}, D={D}")
        if tuple(den.shape) != (1, H, N, 1):
            raise ValueError(f"normalizer must be [1, {H}, {N}, 1], got {tuple(den.shape)}")
        for name, t in (("q_rot", q), ("k_rot", k), ("v", v), ("normalizer", den)):
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
            if t.device != want_device:
                raise ValueError(f"{name} is on {t.device}, expected {want_device}")
        return N

    # ------------------------------------------------------------------ calls
    def forward(self, q_rot, k_rot, v, normalizer, out=None, mode="high", out_dtype=torch.float32, stream=None,
                layout="hnd"):
        """Enqueue one layer call on device tensors and return ``out``.

        layout "hnd": q_rot, k_rot, v and out are [1, H, N, D].
        layout "nhd": q_rot, k_rot, v are [1, N, H, D] (the model's projection layout) and
        out is [1, N, H*D] (any contiguous tensor of that many elements is accepted).
        normalizer is [1, H, N, 1] either way."""
        n = self._check_inputs(q_rot, k_rot, v, normalizer, self.device, layout)
        if out is None:
            shape = q_rot.shape if layout == "hnd" else (1, n, self.heads * self.head_dim)
            out = torch.empty(shape, dtype=out_dtype, device=self.device)
        elif out.numel() != q_rot.numel() or not out.is_contiguous() or out.device != self.device:
            raise ValueError("out must be a contiguous tensor of the inputs' size on the context's device")
        args = (self._h, q_rot.data_ptr(), k_rot.data_ptr(), v.data_ptr(), normalizer.data_ptr(), out.data_ptr(),
                _out_code(out.dtype), n, _mode(mode))
        if layout == "hnd":
            st = lib.lin_attn_forward(*args, _stream_handle(stream, self.device))
        else:
            st = lib.lin_attn_forward_layout(*args, LAYOUT_NHD, _stream_handle(stream, self.device))
        _check(st, "lin_attn_forward")
        return out

    def forward_fused(self, q, k, v, rope_cos, rope_sin, out=None, out_dtype=torch.float32, stream=None,
                      layout="hnd", mode="high"):
        """Layer call from the pre-activation q, k: ReLU, interleaved RoPE (FP32 tables
        [N, D/2]) and the normaliser run inside the kernels (either tier).

        layout "hnd": q, k, v and out are [1, H, N, D].
        layout "nhd": q, k, v are [1, N, H, D] (the model's projection layout) and out is
        [1, N, H*D] (any contiguous tensor of that many elements is accepted)."""
        for name, t in (("q", q), ("k", k), ("v", v)):
            if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.device != self.device:
                raise ValueError(f"{name} must be a contiguous bfloat16 tensor on {self.device}")
        if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape or q.shape[0] != 1:
            raise ValueError("q, k, v must share one 4-D shape with batch 1")
        if layout == "hnd":
            _, H, N, D = q.shape
        elif layout == "nhd":
            _, N, H, D = q.shape
        else:
            raise ValueError(f"layout must be 'hnd' or 'nhd', got {layout!r}")
        if H != self.heads or D != self.head_dim:
            raise ValueError(f"context is for H={self.heads}, D={self.head_dim}; got H={H}, D={D}")
        for name, t in (("rope_cos", rope_cos), ("rope_sin", rope_sin)):
            if t.dtype != torch.float32 or tuple(t.shape) != (N, D // 2) or not t.is_contiguous() \
                    or t.device != self.device:
                raise ValueError(f"{name} must be a contiguous float32 [{N}, {D // 2}] tensor on {self.device}")
        if out is None:
            shape = q.shape if layout == "hnd" else (1, N, H * D)
            out = torch.empty(shape, dtype=out_dtype, device=self.device)
        elif out.numel() != q.numel() or not out.is_contiguous() or out.device != self.device:
            raise ValueError("out must be a contiguous tensor of the inputs' size on the context's device")
        st = lib.lin_attn_forward_fused_layout(self._h, q.data_ptr(), k.data_ptr(), v.data_ptr(), rope_cos.data_ptr(),
                                               rope_sin.data_ptr(), out.data_ptr(), _out_code(out.dtype), N, _mode(mode),
                                               LAYOUT_HND if layout == "hnd" else LAYOUT_NHD,
                                               _stream_handle(stream, self.device))
        _check(st, "lin_attn_forward_fused")
        return out

    def anchor_forward(self, q, k, v, out=None, out_dtype=torch.bfloat16, scale=None, stream=None):
        """Softmax anchor attention (no mask, default scale 1/sqrt(D)) on [1, H, N, D] BF16."""
        for name, t in (("q", q), ("k", k), ("v", v)):
            if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.device != self.device:
                raise ValueError(f"{name} must be a contiguous bfloat16 tensor on {self.device}")
        if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape or q.shape[0] != 1:
            raise ValueError("q, k, v must share one [1, H, N, D] shape")
        _, H, N, D = q.shape
        if H != self.heads or D != self.head_dim:
            raise ValueError(f"context is for H={self.heads}, D={self.head_dim}; got H={H}, D={D}")
        if out is None:
            out = torch.empty(q.shape, dtype=out_dtype, device=self.device)
        elif out.shape != q.shape or not out.is_contiguous() or out.device != self.device:
            raise ValueError("out must be a contiguous [1, H, N, D] tensor on the context's device")
        st = lib.lin_attn_anchor_forward(self._h, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                         _out_code(out.dtype), N, 0.0 if scale is None else float(scale),
                                         _stream_handle(stream, self.device))
        _check(st, "lin_attn_anchor_forward")
        return out

    def forward_host(self, q_rot, k_rot, v, normalizer, out=None, mode="high", out_dtype=torch.float32, stream=None):
        """One layer call on host tensors (pinned for full copy speed); blocks until ``out`` is filled."""
        cpu = torch.device("cpu")
        n = self._check_inputs(q_rot, k_rot, v, normalizer, cpu)
        if out is None:
            out = torch.empty(q_rot.shape, dtype=out_dtype, pin_memory=True)
        elif out.shape != q_rot.shape or not out.is_contiguous() or out.device != cpu:
            raise ValueError("out must be a contiguous [1, H, N, D] host tensor")
        st = lib.lin_attn_forward_host(self._h, q_rot.data_ptr(), k_rot.data_ptr(), v.data_ptr(),
                                       normalizer.data_ptr(), out.data_ptr(), _out_code(out.dtype), n, _mode(mode),
                                       _stream_handle(stream, self.device))
        _check(st, "lin_attn_forward_host")
        return out

    def forward_fused_host(self, q, k, v, rope_cos, rope_sin, out=None, mode="high", out_dtype=torch.float32,
                           stream=None):
        """The fused-producer call (head-major) on host tensors (pinned for full copy speed):
        q, k, v BF16 [1, H, N, D], rope_cos / rope_sin FP32 [N, D/2]; blocks until ``out``
        is filled."""
        cpu = torch.device("cpu")
        for name, t in (("q", q), ("k", k), ("v", v)):
            if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.device != cpu:
                raise ValueError(f"{name} must be a contiguous bfloat16 host tensor")
        if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape or q.shape[0] != 1:
            raise ValueError("q, k, v must share one 4-D shape with batch 1")
        _, H, N, D = q.shape
        if H != self.heads or D != self.head_dim:
            raise ValueError(f"context is for H={self.heads}, D={self.head_dim}; got H={H}, D={D}")
        for name, t in (("rope_cos", rope_cos), ("rope_sin", rope_sin)):
            if t.dtype != torch.float32 or tuple(t.shape) != (N, D // 2) or not t.is_contiguous() or t.device != cpu:
                raise ValueError(f"{name} must be a contiguous float32 [{N}, {D // 2}] host tensor")
        if out is None:
            out = torch.empty(q.shape, dtype=out_dtype, pin_memory=True)
        elif out.shape != q.shape or not out.is_contiguous() or out.device != cpu:
            raise ValueError("out must be a contiguous [1, H, N, D] host tensor")
        st = lib.lin_attn_forward_fused_host(self._h, q.data_ptr(), k.data_ptr(), v.data_ptr(), rope_cos.data_ptr(),
                                             rope_sin.data_ptr(), out.data_ptr(), _out_code(out.dtype), N,
                                             _mode(mode), _stream_handle(stream, self.device))
        _check(st, "lin_attn_forward_fused_host")
        return out

    def debug_kv(self, stream=None):
        """Reduced KV of the last call, FP32 [H, D, D]."""
        kv = torch.empty(self.heads, self.head_dim, self.head_dim, dtype=torch.float32, device=self.device)
        _check(lib.lin_attn_debug_kv(self._h, kv.data_ptr(), _stream_handle(stream, self.device)), "lin_attn_debug_kv")
        return kv

    def device_status(self, stream=None) -> int:
        """Synchronise the stream and return (clearing) the kernels' status word."""
        return lib.lin_attn_device_status(self._h, _stream_handle(stream, self.device))

    def set_wait_limit(self, limit_ns: int):
        """Test hook: barrier-wait limit of the kernels of later calls (0 = the 2 s default)."""
        _check(lib.lin_attn_set_wait_limit(self._h, int(limit_ns)), "lin_attn_set_wait_limit")

    def set_stage_events(self, events):
        """Arm 4 timing events (torch.cuda.Event(enable_timing=True)) for the next forward."""
        if events is None:
            _check(lib.lin_attn_set_stage_events(self._h, None, 0), "lin_attn_set_stage_events")
            return
        for e in events:
            if not e.cuda_event:  # torch creates the CUDA event lazily, on first record
                e.record(torch.cuda.current_stream(self.device))
        arr = (ctypes.c_void_p * 4)(*[e.cuda_event for e in events])
        _check(lib.lin_attn_set_stage_events(self._h, arr, len(events)), "lin_attn_set_stage_events")

    def close(self):
        if getattr(self, "_h", None):
            lib.lin_attn_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
