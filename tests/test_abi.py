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
    assert _fwd(lib, B=1 << 16, Hq=2, Hkv=1, N=1 << 16) == 2    # B * N rows beyond 2^31 - 1
    assert _fwd(lib, B=1 << 12, Hq=1 << 12, Hkv=1, N=1 << 16) == 2  # more CTAs than a 1-D grid holds


def test_persistent_forward_needs_32_byte_aligned_output(lib):
    """fa_fwd_persistent stores O rows 32 bytes at a time: an O that is only
    16-byte aligned is refused before anything is launched (fa_fwd itself
    falls back to the one-CTA-per-block kernel for it); the other checks are
    fa_fwd's."""
    def pers(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, Hq=2, Hkv=1, N=16, d=128, causal=0, scale=0.1,
                 dtype=1)
        a.update(kw)
        return lib.fa_fwd_persistent(*a.values(), None)
    assert pers(o=FAKE + 16) == 1
    assert pers(q=None) == 1
    assert pers(d=96) == 2


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


def test_local_and_two_pass_argument_validation(lib):
    fwd = [FAKE] * 5 + [1, 2, 1, 16, 128]
    assert lib.fa_fwd_local(*fwd, 0, 0.1, 1, None) == 1           # window < 1
    assert lib.fa_fwd_local(*fwd, -3, 0.1, 1, None) == 1
    assert lib.fa_fwd_local(*([None] + fwd[1:]), 4, 0.1, 1, None) == 1
    assert lib.fa_fwd_local(*(fwd[:9] + [96]), 4, 0.1, 1, None) == 2
    ws2 = lib.fa_bwd_two_pass_workspace_bytes(1, 2, 16, 128)
    assert ws2 == 256                                             # D only: 32 floats, rounded up
    assert lib.fa_bwd_two_pass_workspace_bytes(0, 2, 16, 128) == 0
    bwd = [FAKE] * 9 + [1, 2, 1, 16, 128]
    assert lib.fa_bwd_two_pass(*bwd, 0, 0.1, 1, None, ws2, None) == 3
    assert lib.fa_bwd_two_pass(*bwd, 0, 0.1, 1, FAKE, ws2 - 1, None) == 3
    assert lib.fa_bwd_two_pass(*([FAKE + 2] + bwd[1:]), 0, 0.1, 1, FAKE, ws2, None) == 1
    assert lib.fa_bwd_two_pass(*bwd, 0, 0.1, 5, FAKE, ws2, None) == 1   # unknown dtype
    ws1 = lib.fa_bwd_workspace_bytes(1, 2, 16, 128)
    assert lib.fa_bwd_local(*bwd, 0, 0.1, 1, 0, FAKE, ws1, None) == 1   # window < 1
    # the deterministic variant needs D only; the atomic one also the dQ accumulator
    assert lib.fa_bwd_local(*bwd, 4, 0.1, 1, 0, FAKE, ws2, None) == 3
    assert lib.fa_bwd_local(*bwd, 4, float("inf"), 1, 1, FAKE, ws2, None) == 1


def test_varlen_argument_validation(lib):
    cu = FAKE
    # (q, k, v, o, lse, cu_seqlens, B, max_seqlen, total, Hq, Hkv, d, causal, window, scale, dtype, stream)
    def fwd(**kw):
        a = dict(q=FAKE, cu=cu, B=2, max_seqlen=16, total=24, Hq=2, Hkv=1, d=128, causal=1, window=0,
                 scale=0.1, dtype=1)
        a.update(kw)
        return lib.fa_fwd_varlen(a["q"], FAKE, FAKE, FAKE, FAKE, a["cu"], a["B"], a["max_seqlen"], a["total"],
                                 a["Hq"], a["Hkv"], a["d"], a["causal"], a["window"], a["scale"], a["dtype"],
                                 None)
    assert fwd(cu=None) == 1
    assert fwd(cu=FAKE + 2) == 1            # offsets not 4-byte aligned
    assert fwd(B=0) == 1
    assert fwd(max_seqlen=0) == 1
    assert fwd(total=0) == 1
    assert fwd(window=-1) == 1
    assert fwd(window=4, causal=0) == 1     # a window needs the causal mask
    assert fwd(Hq=3, Hkv=2) == 1
    assert fwd(d=32) == 2
    assert fwd(max_seqlen=1 << 30, Hq=1 << 9) == 2   # ceil(max_seqlen / 128) * B * Hq CTAs beyond 2^31 - 1
    assert fwd(q=FAKE + 8) == 1
    for det in (0, 1):
        need = lib.fa_bwd_varlen_workspace_bytes(24, 2, 128, det)
        assert need == 256 + (0 if det else 24 * 2 * 128 * 4)
        args = [FAKE] * 9 + [cu, 2, 16, 24, 2, 1, 128, 1, 0, 0.1, 1, det]
        assert lib.fa_bwd_varlen(*args, FAKE, need - 1, None) == 3
        assert lib.fa_bwd_varlen(*args, FAKE + 64, need, None) == 3   # not 256-aligned
        assert lib.fa_bwd_varlen(*(args[:9] + [None] + args[10:]), FAKE, need, None) == 1
    assert lib.fa_bwd_varlen_workspace_bytes(0, 2, 128, 0) == 0


def test_packed_batch_size_limit_counts_packed_rows(lib):
    """A packed batch is sized by its total rows, not by B * max_seqlen: 64
    sequences with one of 32768 rows and 3000 rows in all pass the size check
    (and here stop at the undersized workspace, before any launch); so do
    more than 2^31 elements per tensor."""
    B, max_seqlen, total, Hq, d = 64, 32768, 3000, 16, 128
    assert B * max_seqlen * Hq * d > 2 ** 31                      # the old, dense-shaped count
    need = lib.fa_bwd_varlen_workspace_bytes(total, Hq, d, 0)
    args = [FAKE] * 9 + [FAKE, B, max_seqlen, total, Hq, Hq, d, 1, 0, 0.1, 1, 0]
    assert lib.fa_bwd_varlen(*args, FAKE, need - 256, None) == 3
    # total * Hq * d beyond 2^31 elements is accepted (64-bit offsets): the
    # call gets as far as the workspace check
    big = 2 ** 31 // (Hq * d) + 1
    need_big = lib.fa_bwd_varlen_workspace_bytes(big, Hq, d, 0)
    args_big = [FAKE] * 9 + [FAKE, B, max_seqlen, big, Hq, Hq, d, 1, 0, 0.1, 1, 0]
    assert lib.fa_bwd_varlen(*args_big, FAKE, need_big - 256, None) == 3


def test_packed_batch_wrappers_marshal_arguments(monkeypatch):
    """The public packed-batch wrappers only allocate outputs and pass them on:
    checked on CPU tensors against a stand-in for the binding that records
    its arguments (nothing is launched)."""
    import torch
    import exact_attention_85_gb300 as fa
    from exact_attention_85_gb300 import _lib

    calls = {}
    monkeypatch.setattr(_lib, "fa_fwd_varlen", lambda *a: calls.setdefault("fwd", a))
    monkeypatch.setattr(_lib, "fa_bwd_varlen", lambda *a: calls.setdefault("bwd", a))
    monkeypatch.setattr(_lib, "fa_bwd_varlen_workspace_bytes", lambda total, Hq, d, det: 256 + (0 if det else 99))
    total, Hq, Hkv, d = 10, 4, 2, 64
    q = torch.zeros(total, Hq, d, dtype=torch.bfloat16)
    k = v = torch.zeros(total, Hkv, d, dtype=torch.bfloat16)
    cu = torch.tensor([0, 3, 3, 10], dtype=torch.int32)
    o, lse = fa.attention_fwd_varlen(q, k, v, cu, causal=True, window=5)
    a = calls["fwd"]
    assert a[0] is q and a[3] is o and a[4] is lse and a[5] is cu
    assert o.shape == q.shape and o.dtype == q.dtype and lse.shape == (Hq, total) and lse.dtype == torch.float32
    assert a[6] == 7 and a[7] is True and a[8] == pytest.approx(d ** -0.5) and a[9] == 5   # max_seqlen, causal, scale, window
    dq, dk, dv = fa.attention_bwd_varlen(q, k, v, o, lse, q, cu, causal=False, deterministic=True)
    b = calls["bwd"]
    assert b[6] is dq and b[7] is dk and b[8] is dv and b[9] is cu and b[10] == 7
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape
    assert b[13] is True and b[14].numel() == 256 and b[15] == 0                           # deterministic, workspace, window
    with pytest.raises(ValueError):
        fa.attention_fwd_varlen(q, k, v, cu, causal=False, window=3)


def test_dense_and_fp8_wrappers_marshal_arguments(monkeypatch):
    """The dense and FP8 wrappers pick the entry point the arguments ask for
    and allocate outputs of the right shape and type (CPU tensors, stand-in
    binding, nothing launched)."""
    import torch
    import exact_attention_85_gb300 as fa
    from exact_attention_85_gb300 import _lib

    calls = []
    for name in ("fa_fwd", "fa_fwd_local", "fa_bwd", "fa_bwd_two_pass", "fa_bwd_local", "fa_hadamard_quant_fp8",
                 "fa_fwd_fp8"):
        monkeypatch.setattr(_lib, name, lambda *a, _n=name: calls.append((_n, a)))
    monkeypatch.setattr(_lib, "fa_bwd_workspace_bytes", lambda *a: 1000)
    monkeypatch.setattr(_lib, "fa_bwd_two_pass_workspace_bytes", lambda *a: 300)
    monkeypatch.setattr(_lib, "fa_hadamard_quant_workspace_bytes", lambda *a: 256)
    B, Hq, Hkv, N, d = 2, 4, 2, 8, 128
    q = torch.zeros(B, Hq, N, d, dtype=torch.float16)
    k = v = torch.zeros(B, Hkv, N, d, dtype=torch.float16)
    o, lse = fa.attention_fwd(q, k, v, causal=True)
    assert calls[-1][0] == "fa_fwd" and calls[-1][1][5] is True and calls[-1][1][6] == pytest.approx(d ** -0.5)
    assert o.shape == q.shape and o.dtype == q.dtype and lse.shape == (B, Hq, N) and lse.dtype == torch.float32
    fa.attention_fwd(q, k, v, causal=True, scale=0.5, window=3)
    assert calls[-1][0] == "fa_fwd_local" and calls[-1][1][5:7] == (3, 0.5)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, lse, q, causal=True)
    n, a = calls[-1]
    assert n == "fa_bwd" and a[6] is dq and a[7] is dk and a[8] is dv and a[11].numel() == 1000
    assert dk.shape == k.shape and dv.shape == v.shape
    fa.attention_bwd(q, k, v, o, lse, q, causal=False, deterministic=True)
    assert calls[-1][0] == "fa_bwd_two_pass" and calls[-1][1][11].numel() == 300
    fa.attention_bwd(q, k, v, o, lse, q, causal=True, deterministic=True, window=4)
    assert calls[-1][0] == "fa_bwd_local" and calls[-1][1][9] == 4 and calls[-1][1][11] is True
    with pytest.raises(ValueError):
        fa.attention_bwd(q, k, v, o, lse, q, causal=False, window=4)
    x = torch.zeros(3, 5, d, dtype=torch.bfloat16)
    x8, desc = fa.hadamard_quant_fp8(x)
    assert calls[-1][0] == "fa_hadamard_quant_fp8" and x8.dtype == torch.float8_e4m3fn and x8.shape == x.shape
    assert desc.shape == (1,) and desc.dtype == torch.float32
    q8 = torch.zeros(B, Hq, N, d, dtype=torch.float8_e4m3fn)
    o8, lse8 = fa.attention_fwd_fp8(q8, q8[:, :Hkv], q8[:, :Hkv], desc, desc, desc, causal=True)
    assert calls[-1][0] == "fa_fwd_fp8" and o8.dtype == torch.bfloat16 and o8.shape == q8.shape
    assert lse8.shape == (B, Hq, N)


def test_binding_marshals_shapes_dtypes_and_errors(monkeypatch):
    """The ctypes layer passes pointers, sizes, element-type codes and
    workspace bytes as the header orders them, and turns a status other
    than FA_OK into FAError (stand-in library, CPU tensors, nothing runs)."""
    import torch
    from exact_attention_85_gb300 import _lib

    class Fake:
        def __init__(self):
            self.calls, self.ret = [], 0

        def __getattr__(self, name):
            if name == "fa_status_string":
                return lambda s: b"FA_ERR_UNSUPPORTED" if s == 2 else b"?"
            return lambda *a: (self.calls.append((name, a)), self.ret)[1]

    fake = Fake()
    monkeypatch.setattr(_lib, "load", lambda: fake)
    B, Hq, Hkv, N, d = 2, 6, 3, 40, 64
    q = torch.zeros(B, Hq, N, d, dtype=torch.bfloat16)
    k = v = torch.zeros(B, Hkv, N, d, dtype=torch.bfloat16)
    lse = torch.zeros(B, Hq, N)
    _lib.fa_fwd(q, k, v, q, lse, True, 0.25, stream=7)
    name, a = fake.calls[-1]
    assert name == "fa_fwd" and a[0] == q.data_ptr() and a[4] == lse.data_ptr()
    assert a[5:] == (B, Hq, Hkv, N, d, 1, 0.25, _lib.FA_BF16, 7)
    ws = torch.zeros(300, dtype=torch.int32)
    qh, kh = q.half(), k.half()
    _lib.fa_bwd(qh, kh, kh, qh, lse, qh, qh, kh, kh, False, 0.5, ws, stream=3)
    name, a = fake.calls[-1]
    assert a[9:] == (B, Hq, Hkv, N, d, 0, 0.5, _lib.FA_FP16, ws.data_ptr(), 1200, 3)
    total = 33
    qp = torch.zeros(total, Hq, d, dtype=torch.bfloat16)
    kp = torch.zeros(total, Hkv, d, dtype=torch.bfloat16)
    cu = torch.tensor([0, 10, 33], dtype=torch.int32)
    _lib.fa_bwd_varlen(qp, kp, kp, qp, lse, qp, qp, kp, kp, cu, 23, True, 0.1, True, ws, window=5, stream=1)
    name, a = fake.calls[-1]
    assert a[9] == cu.data_ptr() and a[10:] == (2, 23, total, Hq, Hkv, d, 1, 5, pytest.approx(0.1), _lib.FA_BF16,
                                                1, ws.data_ptr(), 1200, 1)
    x = torch.zeros(5, 7, 128, dtype=torch.bfloat16)
    _lib.fa_hadamard_quant_fp8(x, None, torch.zeros(5, 7, 128, dtype=torch.uint8), torch.zeros(1), ws, stream=2)
    name, a = fake.calls[-1]
    assert a[1] is None and a[4:] == (35, 128, ws.data_ptr(), 1200, 2)
    with pytest.raises(TypeError):
        _lib.fa_fwd(q.float(), k, v, q, lse, True, 0.25, stream=7)
    fake.ret = 2
    with pytest.raises(_lib.FAError) as e:
        _lib.fa_fwd(q, k, v, q, lse, True, 0.25, stream=7)
    assert e.value.status == 2 and "FA_ERR_UNSUPPORTED" in str(e.value)


def test_binding_refuses_wrong_element_types_and_strided_views():
    """The C calls take bare pointers, so the binding checks what it hands
    them: an fp16 tensor to the bf16-only quantiser, an output of another
    type than the inputs, an LSE that is not fp32, or a strided view would
    otherwise be read as something else with no error.  The checks run
    before the library is called, so CPU tensors serve."""
    import torch
    from exact_attention_85_gb300 import _lib
    x16 = torch.zeros(4, 128, dtype=torch.float16)
    x8 = torch.zeros(4, 128, dtype=torch.uint8)
    one = torch.zeros(1)
    ws = torch.zeros(256, dtype=torch.uint8)
    with pytest.raises(TypeError, match="x: element type"):
        _lib.fa_hadamard_quant_fp8(x16, None, x8, one, ws)
    with pytest.raises(TypeError, match="x8: element type"):
        _lib.fa_hadamard_quant_fp8(x16.to(torch.bfloat16), None, x8.float(), one, ws)
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 8)
    with pytest.raises(TypeError, match="o: element type"):
        _lib.fa_fwd(q, q, q, q.half(), lse, True, 0.125)
    with pytest.raises(TypeError, match="lse: element type"):
        _lib.fa_fwd(q, q, q, q.clone(), lse.double(), True, 0.125)
    with pytest.raises(TypeError, match="unsupported element type"):
        _lib.fa_fwd(q.float(), q.float(), q.float(), q.float(), lse, True, 0.125)
    strided = torch.zeros(1, 2, 64, 8, dtype=torch.bfloat16).transpose(2, 3)
    with pytest.raises(ValueError, match="k: tensor must be contiguous"):
        _lib.fa_fwd(q, strided, q, q.clone(), lse, True, 0.125)
    with pytest.raises(TypeError, match="dq: element type"):
        _lib.fa_bwd(q, q, q, q, lse, q, q.float(), q, q, True, 0.125, ws)
    with pytest.raises(TypeError, match="cu_seqlens: element type"):
        p = torch.zeros(8, 2, 64, dtype=torch.bfloat16)
        _lib.fa_fwd_varlen(p, p, p, p.clone(), torch.zeros(2, 8), torch.tensor([0, 8]), 8, True, 0.125)
    with pytest.raises(TypeError, match="o: element type"):
        q8 = torch.zeros(1, 2, 8, 128, dtype=torch.uint8)
        _lib.fa_fwd_fp8(q8, q8, q8, one, one, one, torch.zeros(1, 2, 8, 128), torch.zeros(1, 2, 8), False, 0.1)
