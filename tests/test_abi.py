"""Host-only checks of the C ABI: the library builds and loads, exports every
symbol include/fa.h declares, and rejects invalid arguments before launching
anything (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_attention_85_gb300 import build, _lib
    build.build()
    return _lib.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "fa_fwd" in names and "fa_bwd" in names
    for n in names:
        assert hasattr(lib, n), n


def test_binding_names_match_header():
    from exact_attention_85_gb300 import _lib
    assert sorted(_lib.EXPORTS) == _declared()


def test_status_strings(lib):
    from exact_attention_85_gb300 import _lib
    for code, name in [(0, b"FA_OK"), (1, b"FA_ERR_INVALID_ARG"), (2, b"FA_ERR_UNSUPPORTED"),
                       (3, b"FA_ERR_WORKSPACE"), (4, b"FA_ERR_CUDA"), (5, b"FA_ERR_TIMEOUT")]:
        assert lib.fa_status_string(code) == name
    assert _lib.FA_ERR_TIMEOUT == 5


FAKE = 1 << 20  # an aligned non-null value; never dereferenced: validation fails first


def _fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, Hq=2, Hkv=1, N=16, d=128, causal=0,
         scale=0.1, dtype=1):
    return lib.fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, dtype, None)


def test_fwd_argument_validation(lib):
    assert _fwd(lib, q=None) == 1
    assert _fwd(lib, lse=None) == 1
    assert _fwd(lib, q=FAKE + 8) == 1          # misaligned
    assert _fwd(lib, N=0) == 1
    assert _fwd(lib, B=-1) == 1
    assert _fwd(lib, Hq=3, Hkv=2) == 1         # Hq % Hkv != 0
    assert _fwd(lib, scale=0.0) == 1
    assert _fwd(lib, scale=float("nan")) == 1
    assert _fwd(lib, dtype=7) == 1
    assert _fwd(lib, d=96) == 2                # unsupported head dim
    assert _fwd(lib, d=256) == 2
    assert _fwd(lib, B=1 << 12, Hq=1 << 10, Hkv=1, N=1 << 12) == 2  # too many elements


def test_bwd_argument_validation(lib):
    ws_need = lib.fa_bwd_workspace_bytes(1, 2, 16, 128)
    assert ws_need == 256 + 2 * 16 * 128 * 4
    args = [FAKE] * 9 + [1, 2, 1, 16, 128, 0, 0.1, 1]
    assert lib.fa_bwd(*args, None, ws_need, None) == 3           # no workspace
    assert lib.fa_bwd(*args, FAKE, ws_need - 1, None) == 3       # too small
    assert lib.fa_bwd(*args, FAKE + 16, ws_need, None) == 3      # not 256-aligned
    bad = [None] + [FAKE] * 8 + [1, 2, 1, 16, 128, 0, 0.1, 1]
    assert lib.fa_bwd(*bad, FAKE, ws_need, None) == 1
    assert lib.fa_bwd(*([FAKE] * 9 + [1, 2, 1, 16, 80, 0, 0.1, 1]), FAKE, 1 << 30, None) == 2


def test_fp8_argument_validation(lib):
    assert lib.fa_hadamard_quant_fp8(None, None, FAKE, FAKE, 4, 128, FAKE, 256, None) == 1
    assert lib.fa_hadamard_quant_fp8(FAKE, None, FAKE, FAKE, 4, 96, FAKE, 256, None) == 2
    assert lib.fa_hadamard_quant_fp8(FAKE, None, FAKE, FAKE, 4, 128, None, 256, None) == 3
    assert lib.fa_hadamard_quant_fp8(FAKE, None, FAKE, FAKE, 0, 128, FAKE, 256, None) == 1
    base = [FAKE] * 8
    assert lib.fa_fwd_fp8(*([None] + base[1:]), 1, 2, 1, 16, 128, 0, 0.1, None) == 1
    assert lib.fa_fwd_fp8(*base, 1, 2, 2, 16, 64 + 1, 0, 0.1, None) == 2
    assert lib.fa_selftest_bounded_wait(0, None) == 1
    assert lib.fa_selftest_bounded_wait(2000000, None) == 1


def test_debug_and_probe_argument_validation(lib):
    lib.fa_probe_exp2.restype = ctypes.c_longlong
    assert lib.fa_probe_exp2(None, 1, 1, None) == -1
    assert lib.fa_probe_exp2(FAKE + 4, 1, 1, None) == -1
    assert lib.fa_probe_exp2(FAKE, 0, 1, None) == -1
    assert lib.fa_probe_exp2(FAKE, 1, 0, None) == -1
    assert lib.fa_probe_exp2(FAKE, 70000, 1, None) == -1
    args = [FAKE] * 5 + [1, 2, 1, 16, 128, 0, 0.1, 1, None]
    assert lib.fa_fwd_f32_out(*([None] + args[1:])) == 1
    assert lib.fa_fwd_f32_out(*(args[:9] + [96] + args[10:])) == 2


def test_product_path_does_not_reference_oracle():
    """The CUDA library and its binding never import, link or call the oracle."""
    pkg = os.path.join(ROOT, "exact_attention_85_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "fa_oracle" not in text and "liboracle" not in text, f


def test_nvtx_ranges_build(tmp_path):
    """The optional NVTX ranges around the entry points compile (FA_NVTX)."""
    from exact_attention_85_gb300 import build
    import subprocess
    src = os.path.join(ROOT, "exact_attention_85_gb300", "csrc", "fa_api.cu")
    cmd = [build._nvcc(), *build.ARCH, *build.FLAGS, "-DFA_NVTX", "-c", src, "-o", str(tmp_path / "fa_api.o")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
