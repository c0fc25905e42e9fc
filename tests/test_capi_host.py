"""Host-side checks of the C ABI that need no GPU: the library builds for sm_103a,
loads, exports every symbol the header declares, and rejects bad arguments
before touching the device."""
import ctypes
import os
import re

import pytest

from gqa_attention_forward_gb300 import binding, build

HEADER = os.path.join(build.INCLUDE, "gqa_attn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w \*]*?\b(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["attn_fwd", "attn_status_str", "attn_last_device_error", "attn_last_cuda_error",
              "attn_version", "attn_test_set_wait_timeout_ns", "attn_test_inject_stall"]:
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in gqa_attn.h but not exported"


def test_status_strings(lib):
    for code, name in binding.STATUS.items():
        s = binding.attn_status_str(code)
        assert s and s != "unknown status", name
    assert binding.attn_status_str(99) == "unknown status"
    assert binding.attn_version() == 0x000100


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails validation first


@pytest.mark.parametrize("args,code", [
    (dict(Hkv=0), 2), (dict(Hq=6, Hkv=4), 2), (dict(N=-1), 2), (dict(B=-2), 2),
    (dict(scale=0.0), 2), (dict(scale=float("inf")), 2), (dict(scale=float("nan")), 2),
    (dict(D=96), 3), (dict(D=256), 3), (dict(dtype=7), 4),
    (dict(q=0), 1), (dict(o=0), 1), (dict(q=FAKE + 8), 5), (dict(v=FAKE + 2), 5),
    (dict(lse=FAKE + 2), 5),
])
def test_argument_errors(lib, args, code):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=4, Hkv=2, N=16, D=128, scale=0.1,
             causal=1, dtype=1)
    a.update(args)
    st = binding.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"],
                          a["N"], a["D"], a["scale"], a["causal"], a["dtype"], None)
    assert st == code, (args, binding.STATUS.get(st))


@pytest.mark.parametrize("empty", [dict(B=0), dict(Hq=0), dict(N=0)])
def test_empty_problem_is_a_no_op(lib, empty):
    a = dict(B=1, Hq=4, Hkv=2, N=16)
    a.update(empty)
    st = binding.attn_fwd(None, None, None, None, None, a["B"], a["Hq"], a["Hkv"], a["N"], 128,
                          0.1, 1, 1, None)
    assert st == 0


def test_no_device_is_reported_without_a_gpu(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this checks the no-device path")
    st = binding.attn_fwd(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 16, 128, 0.1, 1, 1, None)
    assert st == 8  # ATTN_ERR_NODEVICE: validated, then refused before any launch


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        binding.load(str(tmp_path / "libgqa_attn.so"))


def test_oracle_is_not_on_the_product_path():
    pkg = os.path.dirname(binding.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", text, flags=re.M), f
                assert "attn_oracle" not in text, f


def test_ctypes_signature_matches_header(lib):
    assert lib.attn_fwd.restype is ctypes.c_int
    assert len(lib.attn_fwd.argtypes) == 14
    assert lib.attn_fwd_kv.restype is ctypes.c_int
    assert len(lib.attn_fwd_kv.argtypes) == 15


def _kv(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=4, Hkv=2, Nq=16, Nk=48, D=128,
             scale=0.1, causal=1, dtype=1)
    a.update(over)
    return binding.attn_fwd_kv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"],
                               a["Hkv"], a["Nq"], a["Nk"], a["D"], a["scale"], a["causal"],
                               a["dtype"], None)


@pytest.mark.parametrize("args,code", [
    (dict(Nq=49), 2),              # causal: rows 0 .. Nq-Nk-1 would see no key
    (dict(Nk=0), 2),               # queries over no keys
    (dict(Nk=0, causal=0), 2),
    (dict(Nq=-1), 2), (dict(Nk=-3), 2), (dict(Hq=6, Hkv=4), 2),
    (dict(D=80), 3), (dict(dtype=3), 4), (dict(k=0), 1), (dict(o=FAKE + 4), 5),
])
def test_kv_argument_errors(lib, args, code):
    st = _kv(lib, **args)
    assert st == code, (args, binding.STATUS.get(st))


def test_kv_empty_and_non_causal_longer_queries(lib):
    assert _kv(lib, q=None, k=None, v=None, o=None, Nq=0) == 0
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this checks the no-device path")
    # Nq > Nk is fine without the mask, and Nq == Nk is attn_fwd: both pass validation
    assert _kv(lib, Nq=64, Nk=48, causal=0) == 8
    assert _kv(lib, Nq=48, Nk=48) == 8


def test_decode_and_host_entry_points_validate_first(lib):
    """attn_fwd_decode, attn_fwd_decode_noalloc, attn_fwd_host and the workspace query
    reject bad arguments before touching a device; valid ones reach the device check."""
    torch = pytest.importorskip("torch")
    dims = dict(B=1, Hq=8, Hkv=2, Nq=3, Nk=500, D=128)

    def dec(**o):
        a = dict(dims, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, causal=1, ws=None, nbytes=0)
        a.update(o)
        return binding.attn_fwd_decode(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"],
                                       a["Hkv"], a["Nq"], a["Nk"], a["D"], 0.1, a["causal"], 1,
                                       a["ws"], a["nbytes"], None)

    def noalloc(**o):
        a = dict(dims, q=FAKE, causal=1)
        a.update(o)
        return binding.attn_fwd_decode_noalloc(a["q"], FAKE, FAKE, FAKE, None, a["B"], a["Hq"],
                                               a["Hkv"], a["Nq"], a["Nk"], a["D"], 0.1,
                                               a["causal"], 1, None)

    def host(**o):
        a = dict(dims, qh=FAKE, oh=FAKE, lh=None, ld=None)
        a.update(o)
        return binding.attn_fwd_host(a["qh"], FAKE, FAKE, a["oh"], a["lh"], FAKE, FAKE, FAKE, FAKE,
                                     a["ld"], a["B"], a["Hq"], a["Hkv"], a["Nq"], a["Nk"], a["D"],
                                     0.1, 1, 1, None)

    assert dec(Nq=600) == 2            # causal with Nq > Nk
    assert dec(D=96) == 3
    assert dec(q=0) == 1
    assert dec(ws=FAKE + 8, nbytes=1 << 20) == 5   # misaligned workspace
    assert dec(B=0, q=None) == 0       # empty problem
    assert noalloc(Hq=6, Hkv=4) == 2
    assert noalloc(q=FAKE + 2) == 5
    assert host(qh=None) == 1          # missing host input
    assert host(lh=FAKE) == 1          # lse_h without lse_d
    assert host(Nk=0) == 2
    st, nbytes = binding.attn_fwd_decode_workspace(1, 8, 3, 1, 100, 128)
    assert st == 2 and nbytes == 0     # Hq % Hkv != 0
    if not torch.cuda.is_available():
        assert dec() == 8 and noalloc() == 8 and host() == 8
        assert binding.attn_fwd_decode_workspace(1, 8, 2, 1, 100, 128)[0] == 8
