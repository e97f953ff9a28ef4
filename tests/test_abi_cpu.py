"""Host-only checks of the C ABI library: it builds, loads, and exports every
symbol include/q1.h declares.  No compute call is made (no GPU here)."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libpath():
    from bit_affine_quantized_g128_gb300 import build
    return build.build()


def _declared():
    with open(os.path.join(ROOT, "include", "q1.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q1_[a-z_]+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    d = _declared()
    for name in ("q1_pack", "q1_unpack", "q1_dequantize", "q1_qmv", "q1_qmm_narrow", "q1_qmm",
                 "q1_embed_gather", "q1_ffn_fused", "q1_check_symmetric"):
        assert name in d


def test_library_exports_every_declared_symbol(libpath):
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (q1_\w+)", out))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    from bit_affine_quantized_g128_gb300 import q1
    assert sorted(q1.EXPORTED) == _declared()


def test_library_loads_and_host_only_calls_work(libpath):
    import torch  # noqa: F401  (load order: torch's CUDA runtime first)
    lib = ctypes.CDLL(libpath)
    lib.q1_status_string.restype = ctypes.c_char_p
    lib.q1_status_string.argtypes = [ctypes.c_int]
    assert lib.q1_status_string(0) == b"ok"
    assert b"group_size" in lib.q1_status_string(5)
    lib.q1_ffn_workspace_size.restype = ctypes.c_size_t
    lib.q1_ffn_workspace_size.argtypes = [ctypes.c_int64] * 3
    assert lib.q1_ffn_workspace_size(8, 5120, 17408) == 8 * 17408 * 2
    assert lib.q1_ffn_workspace_size(9, 5120, 17408) == 0
    lib.q1_decode_chain_workspace_size.restype = ctypes.c_size_t
    lib.q1_decode_chain_workspace_size.argtypes = [ctypes.c_int64] * 3
    # a and h [M][D] plus the FFN intermediate [M][F_max], bf16, each 256-byte aligned
    assert lib.q1_decode_chain_workspace_size(1, 5120, 17408) == 2 * 10240 + 34816
    assert lib.q1_decode_chain_workspace_size(3, 128, 384) == 2 * 768 + 2304
    assert lib.q1_decode_chain_workspace_size(9, 5120, 17408) == 0
    lib.q1_set_qmm_max_rows(3)
    assert lib.q1_get_qmm_max_rows() == 3
    lib.q1_set_qmm_max_rows(100)
    assert lib.q1_get_qmm_max_rows() == 8
    lib.q1_set_qmm_max_rows(-2)
    assert lib.q1_get_qmm_max_rows() == 0


def test_threshold_env_read_at_load(libpath):
    code = ("import ctypes, torch; l = ctypes.CDLL(%r); print(l.q1_get_qmm_max_rows())" % libpath)
    env = dict(os.environ, Q1_QMM_MAX_ROWS="5")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                         check=True).stdout.strip()
    assert out == "5"
    env.pop("Q1_QMM_MAX_ROWS")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                         check=True).stdout.strip()
    assert out == "8"


def test_binding_raises_without_library(tmp_path):
    # a fresh process: the binding refuses to run without the CUDA library
    code = ("from bit_affine_quantized_g128_gb300 import q1\n"
            "try:\n    q1.load_library(%r)\nexcept RuntimeError as e:\n    print('raised', e)\n"
            % str(tmp_path / "missing.so"))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT,
                         check=True).stdout
    assert out.startswith("raised")
