"""The C-ABI library loads on a machine without a GPU, exports every symbol
that include/*.h declares, and rejects bad arguments on the host before any
CUDA call (no compute calls are made here)."""
import ctypes
import glob
import os
import re

import pytest

import weight_quantized_decode_gb300 as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        txt = open(h).read()
        names += re.findall(r"^QMV_API\s+[\w\s\*]+?\b(\w+)\s*\(", txt, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(q.LIB_PATH):
        from weight_quantized_decode_gb300 import build
        build.build()
    return q.lib()


def test_header_declares_the_boundary():
    names = set(_declared())
    for n in ("qmv_q4_0", "qmv_q8_0", "qmv_moe", "qmm_q4_0_prefill", "qmv_device_status", "qmv_q4_0_swiglu",
              "qmv_q4_0_f32", "qmv_q4_0_swiglu_f32", "qmv_q2w", "qmv_q4_0_q8_1", "qmv_quantize_q8_1",
              "qmv_q4_0_q8_1_pre"):
        assert n in names


_CTYPE = {"const void *": ctypes.c_void_p, "void *": ctypes.c_void_p, "float *": ctypes.c_void_p,
          "const float *": ctypes.c_void_p, "const int8_t *": ctypes.c_void_p, "int8_t *": ctypes.c_void_p,
          "const uint16_t *": ctypes.c_void_p, "uint16_t *": ctypes.c_void_p, "const int32_t *": ctypes.c_void_p,
          "int32_t *": ctypes.c_void_p, "uint32_t *": ctypes.c_void_p, "qmv_stream_t": ctypes.c_void_p,
          "int64_t": ctypes.c_int64, "int": ctypes.c_int, "qmv_status": ctypes.c_int}


def _signatures():
    """name -> list of parameter types as written in include/*.h."""
    sigs = {}
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        txt = open(h).read()
        for name, params in re.findall(r"^QMV_API\s+[\w\s\*]+?\b(\w+)\s*\(([^)]*)\)", txt, flags=re.M):
            plist = [] if params.strip() in ("", "void") else [p.strip() for p in params.split(",")]
            # drop the parameter name: the type is everything before the last identifier
            sigs[name] = [re.sub(r"\s*\b\w+$", "", " ".join(p.split())).replace(" *", " *") for p in plist]
    return sigs


def test_binding_signatures_match_the_header(lib):
    # every entry point's ctypes argument list has the header's length and kinds
    # (pointers as void pointers, sizes as int64, flags as int)
    for name, types in _signatures().items():
        f = getattr(lib, name)
        assert f.argtypes is not None, name
        want = [_CTYPE[t] for t in types]
        got = list(f.argtypes)
        assert len(got) == len(want), (name, types, got)
        for t, w, g in zip(types, want, got):
            ok = g == w or (w is ctypes.c_void_p and getattr(g, "_type_", None) is not None)
            assert ok, (name, t, g)


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(q.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(raw, n)]
    assert not missing, missing


def test_version_and_status_strings(lib):
    assert "sm_103a" in q.qmv_version()
    assert q.qmv_status_str(0) == "ok"
    assert q.qmv_status_str(3) == "shape out of range"


FAKE = 1 << 20      # a 16-byte-aligned non-null address; never dereferenced here


@pytest.mark.parametrize("fn", ["qmv_q4_0", "qmv_q8_0", "qmm_q4_0_prefill", "qmv_q4_0_f32", "qmv_q2w",
                                "qmv_q4_0_q8_1", "qmv_q8_0_q8_1"])
def test_host_validation(lib, fn):
    f = getattr(lib, fn)
    assert f(None, FAKE, FAKE, 8, 256, 1, None) == 1          # NULL W
    assert f(FAKE, None, FAKE, 8, 256, 1, None) == 1          # NULL x
    assert f(FAKE, FAKE, None, 8, 256, 1, None) == 1          # NULL y
    assert f(FAKE + 8, FAKE, FAKE, 8, 256, 1, None) == 2      # W not 16-byte aligned
    assert f(FAKE, FAKE + 1, FAKE, 8, 256, 1, None) == 2      # x not 2-byte aligned
    assert f(FAKE, FAKE, FAKE + 2, 8, 256, 1, None) == 2      # y not 4-byte aligned
    assert f(FAKE, FAKE, FAKE, 8, 250, 1, None) == 3          # K % 32 != 0
    assert f(FAKE, FAKE, FAKE, -1, 256, 1, None) == 3
    assert f(FAKE, FAKE, FAKE, 8, -32, 1, None) == 3
    assert f(FAKE, FAKE, FAKE, 8, 256, -1, None) == 3
    assert f(None, None, None, 0, 256, 1, None) == 0          # empty: nothing to do
    assert f(None, None, None, 8, 256, 0, None) == 0
    if fn != "qmm_q4_0_prefill":
        assert f(FAKE, FAKE, FAKE, 8, 256, 9, None) == 3      # decode takes M <= 8
    else:
        assert f(FAKE, FAKE, FAKE, 8, 256, (1 << 24) + 1, None) == 3   # prefill takes M <= 2^24
        assert f(FAKE, FAKE + 2, FAKE, 8, 256, 64, None) == 2          # tensor-copy x: 16-byte aligned
    if fn == "qmv_q4_0_f32":
        assert f(FAKE, FAKE + 2, FAKE, 8, 256, 1, None) == 2  # fp32 x not 4-byte aligned


@pytest.mark.parametrize("fn", ["qmv_q4_0_swiglu", "qmv_q4_0_swiglu_f32"])
def test_host_validation_swiglu(lib, fn):
    f = getattr(lib, fn)
    assert f(None, FAKE, FAKE, FAKE, 8, 256, 1, None) == 1    # NULL gate table
    assert f(FAKE, None, FAKE, FAKE, 8, 256, 1, None) == 1    # NULL up table
    assert f(FAKE, FAKE, None, FAKE, 8, 256, 1, None) == 1    # NULL x
    assert f(FAKE, FAKE, FAKE, None, 8, 256, 1, None) == 1    # NULL y
    assert f(FAKE, FAKE + 8, FAKE, FAKE, 8, 256, 1, None) == 2  # up table misaligned
    assert f(FAKE, FAKE, FAKE + 1, FAKE, 8, 256, 1, None) == 2  # x misaligned
    assert f(FAKE, FAKE, FAKE, FAKE, 8, 256, 9, None) == 3    # M <= 8
    assert f(FAKE, FAKE, FAKE, FAKE, 8, 250, 1, None) == 3    # K % 32
    assert f(FAKE, FAKE, FAKE, FAKE, 1 << 40, 256, 1, None) == 3   # 2N rows overflow the row index range
    assert f(None, None, None, None, 0, 256, 1, None) == 0    # empty
    assert f(None, None, None, None, 8, 256, 0, None) == 0
    if fn.endswith("_f32"):
        assert f(FAKE, FAKE, FAKE + 2, FAKE, 8, 256, 1, None) == 2   # fp32 x not 4-byte aligned


def test_host_validation_q8_0_q8_1_pre(lib):
    f = lib.qmv_q8_0_q8_1_pre
    assert f(None, FAKE, FAKE, FAKE, 8, 256, 1, None) == 1        # NULL W
    assert f(FAKE, None, FAKE, FAKE, 8, 256, 1, None) == 1        # NULL codes
    assert f(FAKE, FAKE, None, FAKE, 8, 256, 1, None) == 1        # NULL scales
    assert f(FAKE, FAKE, FAKE, None, 8, 256, 1, None) == 1        # NULL y
    assert f(FAKE + 8, FAKE, FAKE, FAKE, 8, 256, 1, None) == 2    # W not 16-byte aligned
    assert f(FAKE, FAKE, FAKE + 1, FAKE, 8, 256, 1, None) == 2    # scales not 2-byte aligned
    assert f(FAKE, FAKE, FAKE, FAKE, 8, 250, 1, None) == 3        # K % 32
    assert f(FAKE, FAKE, FAKE, FAKE, 8, 256, 9, None) == 3        # M <= 8
    assert f(None, None, None, None, 0, 256, 1, None) == 0        # empty
    assert f(None, None, None, None, 8, 256, 0, None) == 0


def test_host_validation_quantize_q8_1(lib):
    f = lib.qmv_quantize_q8_1
    assert f(None, FAKE, FAKE, FAKE, 2, 256, None) == 1           # NULL x
    assert f(FAKE, None, FAKE, FAKE, 2, 256, None) == 1           # NULL codes
    assert f(FAKE, FAKE, None, FAKE, 2, 256, None) == 1           # NULL scales
    assert f(FAKE, FAKE, FAKE, None, 2, 256, None) == 1           # NULL sums
    assert f(FAKE + 8, FAKE, FAKE, FAKE, 2, 256, None) == 2       # x not 16-byte aligned
    assert f(FAKE, FAKE + 4, FAKE, FAKE, 2, 256, None) == 2       # codes not 8-byte aligned
    assert f(FAKE, FAKE, FAKE + 1, FAKE, 2, 256, None) == 2       # scales not 2-byte aligned
    assert f(FAKE, FAKE, FAKE, FAKE + 2, 2, 256, None) == 2       # sums not 4-byte aligned
    assert f(FAKE, FAKE, FAKE, FAKE, 2, 48, None) == 3            # K % 32
    assert f(FAKE, FAKE, FAKE, FAKE, -1, 256, None) == 3
    assert f(None, None, None, None, 0, 256, None) == 0           # empty
    assert f(None, None, None, None, 2, 0, None) == 0


def test_host_validation_q8_1_pre(lib):
    f = lib.qmv_q4_0_q8_1_pre
    assert f(None, FAKE, FAKE, FAKE, FAKE, 8, 256, 1, None) == 1     # NULL W
    assert f(FAKE, None, FAKE, FAKE, FAKE, 8, 256, 1, None) == 1     # NULL codes
    assert f(FAKE, FAKE, None, FAKE, FAKE, 8, 256, 1, None) == 1     # NULL scales
    assert f(FAKE, FAKE, FAKE, None, FAKE, 8, 256, 1, None) == 1     # NULL sums
    assert f(FAKE, FAKE, FAKE, FAKE, None, 8, 256, 1, None) == 1     # NULL y
    assert f(FAKE, FAKE, FAKE + 1, FAKE, FAKE, 8, 256, 1, None) == 2  # scales misaligned
    assert f(FAKE, FAKE, FAKE, FAKE + 2, FAKE, 8, 256, 1, None) == 2  # sums misaligned
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 250, 1, None) == 3     # K % 32
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 256, 9, None) == 3     # M <= 8
    assert f(None, None, None, None, None, 0, 256, 1, None) == 0     # empty


def test_host_validation_moe(lib):
    f = lib.qmv_moe
    assert f(FAKE, None, 4, FAKE, FAKE, 8, 256, 2, None) == 1     # NULL index array
    assert f(FAKE, FAKE, 0, FAKE, FAKE, 8, 256, 2, None) == 3     # no experts
    assert f(FAKE, FAKE + 2, 4, FAKE, FAKE, 8, 256, 2, None) == 2  # index array misaligned
    assert f(FAKE, FAKE, 4, FAKE, FAKE, 8, 256, 65, None) == 3    # too many slots
    assert f(FAKE, FAKE, 4, FAKE, FAKE, 8, 200, 2, None) == 3     # K % 32
    assert f(None, None, 4, None, None, 8, 256, 0, None) == 0


def test_no_cpu_path():
    torch = pytest.importorskip("torch")
    W = torch.zeros((4, 144), dtype=torch.uint8)
    x = torch.zeros((1, 256), dtype=torch.float16)
    with pytest.raises(TypeError):
        q.qmv_q4_0(W, x)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    # Without the built library every call raises; nothing falls back to a CPU path.
    monkeypatch.setattr(q, "_lib", None)
    monkeypatch.setattr(q, "LIB_PATH", str(tmp_path / "libqmv.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        q.qmv_version()
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        q.qmv_q4_0_ptr(FAKE, FAKE, FAKE, 8, 256, 1)
