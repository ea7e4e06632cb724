"""The C-ABI library: it loads, exports every entry point the header declares, and its
host-side argument checks answer without touching a GPU (no compute calls here)."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "lin_attn.h")
LIB = os.path.join(ROOT, "video_diffusion_dit_gb300", "liblin_attn.so")


@pytest.fixture(scope="module")
def la():
    if not os.path.exists(LIB):
        from video_diffusion_dit_gb300 import build
        build.build()
    from video_diffusion_dit_gb300 import lin_attn
    return lin_attn


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lin_attn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("lin_attn_create", "lin_attn_forward", "lin_attn_destroy"):
        assert want in names


def test_library_exports_every_declared_symbol(la):
    lib = ctypes.CDLL(LIB)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in lin_attn.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\b(lin_attn_\w+)\b", out))
    assert exported == set(declared_functions()), "exports and header declarations differ"
    assert set(la.EXPORTS) == set(declared_functions())


def test_header_compiles_as_c():
    src = '#include "lin_attn.h"\nint main(void){ return lin_attn_version() == LIN_ATTN_VERSION ? 0 : 1; }\n'
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I", os.path.dirname(HEADER),
                        "-x", "c", "-"], input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_plain_c_program_links_and_calls_the_library(la, tmp_path):
    # The boundary from C itself (no ctypes): link against the library, call the entry
    # points that need no GPU, and check what they answer.
    src = tmp_path / "abi_client.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "lin_attn.h"
int main(void) {
    if (lin_attn_version() != LIN_ATTN_VERSION) return 10;
    if (strcmp(lin_attn_error_string(LIN_ATTN_OK), lin_attn_error_string(99)) == 0) return 11;
    lin_attn_ctx *ctx = (lin_attn_ctx *)0x1;
    if (lin_attn_create(&ctx, 0, 1000, 112, 0) != LIN_ATTN_ERR_INVALID_ARG) return 12;
    if (ctx != NULL) return 13;
    if (lin_attn_create(&ctx, 20, 1000, 100, 0) != LIN_ATTN_ERR_UNSUPPORTED) return 14;
    if (strstr(lin_attn_last_error(), "head_dim") == NULL) return 15;
    int chunks = 0, segs = 0;
    if (lin_attn_kv_plan(20, 180320, LIN_ATTN_MODE_HIGH, &chunks, &segs) != LIN_ATTN_OK) return 16;
    if (chunks != 152 || segs != 9) return 17;
    if (lin_attn_kv_plan(0, 10, LIN_ATTN_MODE_HIGH, &chunks, &segs) != LIN_ATTN_ERR_INVALID_ARG) return 18;
    if (lin_attn_destroy(NULL) != LIN_ATTN_OK) return 19;
    puts("ok");
    return 0;
}
""")
    exe = tmp_path / "abi_client"
    libdir = os.path.dirname(LIB)
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe),
                        "-L", libdir, "-llin_attn", f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)


def test_version_and_error_strings(la):
    assert la.lib.lin_attn_version() == 100
    for code in range(7):
        assert la.error_string(code) and la.error_string(code) != "unknown status"
    assert la.error_string(99) == "unknown status"


def test_create_rejects_bad_arguments_before_any_cuda_call(la):
    h = ctypes.c_void_p(1234)
    assert la.lib.lin_attn_create(None, 20, 1000, 112, 0) == la.ERR_INVALID_ARG
    assert la.lib.lin_attn_create(ctypes.byref(h), 0, 1000, 112, 0) == la.ERR_INVALID_ARG
    assert not h.value  # *ctx cleared on failure
    assert la.lib.lin_attn_create(ctypes.byref(h), 20, 0, 112, 0) == la.ERR_INVALID_ARG
    assert la.lib.lin_attn_create(ctypes.byref(h), 20, (1 << 30) + 1, 112, 0) == la.ERR_INVALID_ARG
    for d in (0, 8, 24, 100, 144):
        assert la.lib.lin_attn_create(ctypes.byref(h), 20, 1000, d, 0) == la.ERR_UNSUPPORTED
    assert b"head_dim" in la.lib.lin_attn_last_error()


def test_calls_on_null_context_are_rejected(la):
    p = ctypes.c_void_p(16)
    assert la.lib.lin_attn_forward(None, p, p, p, p, p, 0, 10, 0, None) == la.ERR_INVALID_ARG
    assert la.lib.lin_attn_forward_host(None, p, p, p, p, p, 0, 10, 0, None) == la.ERR_INVALID_ARG
    assert la.lib.lin_attn_debug_kv(None, p, None) == la.ERR_INVALID_ARG
    assert la.lib.lin_attn_device_status(None, None) == la.ERR_INVALID_ARG
    assert la.lib.lin_attn_set_stage_events(None, None, 0) == la.ERR_INVALID_ARG
    assert la.lib.lin_attn_destroy(None) == la.OK
    assert la.lib.lin_attn_forward_layout(None, p, p, p, p, p, 0, 10, 0, 0, None) == la.ERR_INVALID_ARG
    assert la.lib.lin_attn_forward_fused(None, p, p, p, p, p, p, 0, 10, 0, None) == la.ERR_INVALID_ARG
    assert la.lib.lin_attn_forward_fused_layout(None, p, p, p, p, p, p, 0, 10, 0, 0, None) == la.ERR_INVALID_ARG
    assert la.lib.lin_attn_anchor_forward(None, p, p, p, p, 0, 10, 0.0, None) == la.ERR_INVALID_ARG
    # Checks that come before any CUDA call, whatever the context.
    assert la.lib.lin_attn_forward_fused_layout(None, p, p, p, p, p, p, 0, 10, 0, 7, None) == la.ERR_INVALID_ARG
    assert b"layout" in la.lib.lin_attn_last_error()
    assert la.lib.lin_attn_forward_fused_layout(None, p, p, p, None, p, p, 0, 10, 0, 0, None) == la.ERR_INVALID_ARG
    assert b"rotation table" in la.lib.lin_attn_last_error()


def test_noalloc_entry_checks_arguments_before_any_cuda_call(la):
    p = ctypes.c_void_p(16)
    f = la.lib.lin_attn_forward_noalloc
    assert f(None, p, p, p, p, 0, 20, 1000, 112, 0, None) == la.ERR_INVALID_ARG
    assert f(p, p, p, p, p, 0, 0, 1000, 112, 0, None) == la.ERR_INVALID_ARG       # heads
    assert f(p, p, p, p, p, 0, 20, 0, 112, 0, None) == la.ERR_INVALID_ARG         # n_tokens
    assert f(p, p, p, p, p, 0, 20, 1000, 100, 0, None) == la.ERR_UNSUPPORTED      # head_dim
    assert f(p, p, p, p, p, 0, 20, 1000, 112, 5, None) == la.ERR_INVALID_ARG      # mode
    assert f(p, p, p, p, p, 9, 20, 1000, 112, 0, None) == la.ERR_INVALID_ARG      # out dtype
    assert b"out_dtype" in la.lib.lin_attn_last_error()


def test_kv_plan_depends_on_shape_and_tier_only(la):
    # The plan fixes the summation order: a pure function of (H, N, tier) that keeps every
    # head within the reduction's 160-partial budget.  k = max(1, min(152 // H, tiles per
    # head, 150)) chunks per head take each head's leading tiles, cut at the same tokens;
    # on long sequences the spare CTAs (152 - k H) share the rest, so a head has k, k + 1
    # or k + 2 partials.  (tests/test_work_split.py checks the partition tile by tile.)
    for H in (1, 2, 12, 20, 32, 64, 151, 152, 153, 4096):
        for N in (1, 63, 64, 65, 256, 1000, 32760, 180320, 262144):
            if H * N >= 2 ** 31:
                continue
            tiles = -(-N // 64)
            for mode in ("high", "lossless"):
                G, segs = la.kv_plan(H, N, mode)
                assert (G, segs) == la.kv_plan(H, N, mode) == la.kv_plan(H, N, "lossless")
                k = max(1, min(152 // H, tiles, 150))
                if k * H >= 152 or k == tiles or G == k * H:  # no spare CTAs, or no tail worth it
                    assert (G, segs) == (k * H, k)
                else:
                    assert k * H < G <= 152 and k < segs <= k + 2
                assert 1 <= segs <= 160
    assert la.kv_plan(20, 180320, "high") == (152, 9)
    assert la.kv_plan(20, 180320, "lossless") == (152, 9)
    assert la.kv_plan(32, 180320, "high") == (152, 6)
    assert la.kv_plan(152, 180320, "high") == (152, 1)
    assert la.kv_plan(20, 32760, "high") == (140, 7)  # 480p: parts too short for a tail
    with pytest.raises(la.LinAttnError):
        la.kv_plan(0, 10, "high")


def test_binding_rejects_wrong_tensors_without_gpu(la):
    import torch
    # The binding's own checks fire before the library is reached.
    obj = la.LinAttn.__new__(la.LinAttn)
    obj.heads, obj.head_dim, obj.max_tokens = 2, 32, 64
    cpu = torch.device("cpu")
    q = torch.zeros(1, 2, 8, 32, dtype=torch.bfloat16)
    den = torch.ones(1, 2, 8, 1)
    assert obj._check_inputs(q, q, q, den, cpu) == 8
    with pytest.raises(TypeError):
        obj._check_inputs(q.float(), q, q, den, cpu)
    with pytest.raises(TypeError):
        obj._check_inputs(q, q, q, den.double(), cpu)
    with pytest.raises(ValueError):
        obj._check_inputs(q.expand(2, 2, 8, 32), q, q, den, cpu)
    with pytest.raises(ValueError):
        obj._check_inputs(q, q, q, torch.ones(1, 2, 8), cpu)
    with pytest.raises(ValueError):
        obj._check_inputs(q.transpose(2, 3).contiguous().transpose(2, 3), q, q, den, cpu)
    with pytest.raises(ValueError):
        obj._check_inputs(torch.zeros(1, 3, 8, 32, dtype=torch.bfloat16), q, q, den, cpu)
    with pytest.raises(ValueError):
        la._mode("fast")
    with pytest.raises(TypeError):
        la._out_code(torch.float16)


def test_binding_rejects_wrong_fused_and_anchor_arguments_without_gpu(la):
    import torch
    # The fused-producer and anchor calls check their tensors before the library is reached.
    obj = la.LinAttn.__new__(la.LinAttn)
    obj.heads, obj.head_dim, obj.max_tokens = 2, 32, 64
    obj.device = torch.device("cpu")
    obj._h = None
    q = torch.zeros(1, 2, 8, 32, dtype=torch.bfloat16)
    cos = torch.zeros(8, 16)
    with pytest.raises(ValueError):  # float32 activations
        obj.forward_fused(q.float(), q, q, cos, cos)
    with pytest.raises(ValueError):  # shapes differ
        obj.forward_fused(q, q[:, :, :4].contiguous(), q, cos, cos)
    with pytest.raises(ValueError):  # unknown layout
        obj.forward_fused(q, q, q, cos, cos, layout="bnhd")
    with pytest.raises(ValueError):  # table rows must match N
        obj.forward_fused(q, q, q, torch.zeros(9, 16), cos)
    with pytest.raises(ValueError):  # tables must be float32
        obj.forward_fused(q, q, q, cos, cos.double())
    with pytest.raises(ValueError):  # token-major input read with the context's H = 2: N = 2, H = 8
        obj.forward_fused(q, q, q, cos, cos, layout="nhd")
    with pytest.raises(ValueError):  # out of the wrong size
        obj.forward_fused(q, q, q, cos, cos, out=torch.zeros(3))
    with pytest.raises(ValueError):  # anchor: head count of another context
        obj.anchor_forward(torch.zeros(1, 3, 8, 32, dtype=torch.bfloat16), *(torch.zeros(1, 3, 8, 32,
                                                                                       dtype=torch.bfloat16),) * 2)
    with pytest.raises(ValueError):  # anchor: non-contiguous
        qt = q.transpose(2, 3).contiguous().transpose(2, 3)
        obj.anchor_forward(qt, q, q)
    with pytest.raises(ValueError):  # anchor: out of the wrong shape
        obj.anchor_forward(q, q, q, out=torch.zeros(1, 2, 8, 16, dtype=torch.bfloat16))
