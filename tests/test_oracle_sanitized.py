"""The oracle's C code under AddressSanitizer and UndefinedBehaviorSanitizer: every entry
point runs on small ragged shapes (one token, head dim 2, rows at both ends of the layer)
in a child process; any out-of-bounds access or undefined operation aborts it."""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

SCRIPT = r'''
import sys
sys.path.insert(0, sys.argv[2])
import numpy as np
import oracle
lib = oracle.load(sys.argv[1])
rng = np.random.default_rng(0)

def bits(shape):
    return (rng.standard_normal(shape).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)

for H, N, D in ((1, 1, 2), (2, 37, 16), (3, 5, 112)):
    q, k, v = bits((H, N, D)), bits((H, N, D)), bits((H, N, D))
    den = rng.random((H, N)).astype(np.float32) + 1.0
    oracle.forward(q, k, v, den, lib=lib)
    kv = oracle.kv(k, v, lib=lib)
    ends = np.array(sorted({0, H * N - 1}), np.int64)
    oracle.apply_rows(q, kv, den, rows=ends, lib=lib)
    oracle.apply_rows(q, kv, den.astype(np.float64) + 2.0 ** -40, rows=ends, lib=lib)
    oracle.apply_rows(q, kv, den.astype(np.float64), lib=lib)
    cos = rng.random((N, D // 2)).astype(np.float32)
    sin = rng.random((N, D // 2)).astype(np.float32)
    oracle.producer(q, k, cos, sin, lib=lib)
    oracle.softmax_attention_rows(q, k, v, rows=ends, lib=lib)
    oracle.bf16_decode(q, lib=lib)
    oracle.f32_to_bf16(rng.standard_normal(17).astype(np.float32), lib=lib)
print("ok")
'''


def test_oracle_is_clean_under_sanitizers(tmp_path):
    asan = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True, text=True).stdout.strip()
    ubsan = subprocess.run(["gcc", "-print-file-name=libubsan.so"], capture_output=True, text=True).stdout.strip()
    if not (os.path.isabs(asan) and os.path.exists(asan) and os.path.isabs(ubsan) and os.path.exists(ubsan)):
        pytest.skip("gcc sanitizer runtimes not installed")
    import oracle
    lib = str(tmp_path / "liblin_attn_oracle_san.so")
    oracle.build(out=lib, extra_flags=("-g", "-fsanitize=address,undefined", "-fno-sanitize-recover=all",
                                       "-fno-omit-frame-pointer"))
    script = tmp_path / "run.py"
    script.write_text(SCRIPT)
    env = dict(os.environ, LD_PRELOAD=f"{asan} {ubsan}", ASAN_OPTIONS="detect_leaks=0", OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, str(script), lib, ROOT], capture_output=True, text=True, env=env,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), (r.returncode, r.stdout[-2000:], r.stderr[-4000:])
