"""The C-ABI library: it loads, exports every symbol the header declares, and rejects bad
arguments on the host before touching a GPU (so these run without one)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
import sparse_causal_attention_swa_b300 as pkg

HEADER = os.path.join(ROOT, "include", "swa_b300.h")


def declared_functions():
    src = open(HEADER, encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?(?:int|size_t|char\s*\*|const char\s*\*|void)\s*\*?\s*"
                                 r"([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("swa_attn_fwd", "strided_attn_fwd", "diff_attn_fwd", "swa_status_string",
              "swa_device_status", "swa_watchdog_selftest"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(pkg.LIBRARY_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings():
    for code in range(0, 9):
        s = pkg.swa_status_string(code)
        assert s and s != "unknown status"
    assert pkg.swa_status_string(99) == "unknown status"


P = 0x10000  # a 16-byte aligned, never dereferenced pointer value
lib = None


@pytest.fixture(scope="module")
def L():
    return pkg.load()


def call_swa(L, q=P, k=P, v=P, out=P, B=1, Hq=2, Hkv=2, N=128, d=64, W=16, scale=0.125):
    return L.swa_attn_fwd(q, k, v, out, B, Hq, Hkv, N, d, W, scale, None)


def test_swa_validation(L):
    assert call_swa(L, q=None) == 1
    assert call_swa(L, out=None) == 1
    assert call_swa(L, B=0) == 2
    assert call_swa(L, N=0) == 2
    assert call_swa(L, W=0) == 2
    assert call_swa(L, Hq=3, Hkv=2) == 2
    assert call_swa(L, d=96) == 4
    assert call_swa(L, d=256) == 4
    assert call_swa(L, scale=0.0) == 7
    assert call_swa(L, scale=float("nan")) == 7
    assert call_swa(L, scale=-1.0) == 7
    assert call_swa(L, k=P + 8) == 3
    assert call_swa(L, out=P + 2) == 3


def test_strided_validation(L):
    f = L.strided_attn_fwd
    assert f(None, P, P, P, 1, 2, 2, 128, 64, 16, 4, 0.125, None) == 1
    assert f(P, P, P, P, 1, 2, 2, 128, 64, 16, 0, 0.125, None) == 2
    assert f(P, P, P, P, 1, 2, 2, 128, 64, 0, 4, 0.125, None) == 2
    assert f(P, P, P, P, 1, 2, 2, 128, 80, 16, 4, 0.125, None) == 4
    assert f(P, P, P, P + 4, 1, 2, 2, 128, 64, 16, 4, 0.125, None) == 3


def test_diff_validation(L):
    f = L.diff_attn_fwd
    assert f(P, P, None, P, P, 0.8, P, 1, 2, 2, 128, 64, 0.125, None) == 1
    assert f(P, P, P, P, P, float("inf"), P, 1, 2, 2, 128, 64, 0.125, None) == 7
    assert f(P, P, P, P, P, 0.8, P, 1, 2, 4, 128, 64, 0.125, None) == 2
    assert f(P, P, P, P, P + 8, 0.8, P, 1, 2, 2, 128, 64, 0.125, None) == 3


def test_noalloc_validation(L):
    f = L.strided_attn_fwd_noalloc
    assert f(None, P, P, P, 1, 2, 2, 128, 64, 16, 4, 0.125, None) == 1
    assert f(P, P, P, P, 1, 2, 2, 128, 64, 16, 0, 0.125, None) == 2
    assert f(P, P, P, P + 4, 1, 2, 2, 128, 64, 16, 4, 0.125, None) == 3
    # a list longer than the fixed capacity is refused on the host, before any launch
    assert f(P, P, P, P, 1, 1, 1, 1 << 22, 64, 256, 1, 0.125, None) == 8


def test_watchdog_selftest_validation(L):
    assert L.swa_watchdog_selftest(0, None) == 7
    assert L.swa_watchdog_selftest(2_000_000, None) == 7


def test_binding_raises_with_status():
    with pytest.raises(pkg.SwaError) as e:
        pkg.swa_attn_fwd(P, P, P, P, 1, 2, 2, 128, 64, 0, 0.125, stream=0)
    assert e.value.code == 2


def test_decode_validation(L):
    f = L.swa_decode_fwd
    n = L.swa_decode_workspace_bytes(2, 8, 300, 128)
    assert n > 0 and n % 4 == 0
    assert L.swa_decode_workspace_bytes(2, 8, 300, 96) == 0
    ok = dict(q=P, kc=P, vc=P, pos=P, out=P, B=2, Hq=8, Hkv=2, W=300, d=128, scale=0.1, ws=P,
              nb=n)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["q"], a["kc"], a["vc"], a["pos"], a["out"], a["B"], a["Hq"], a["Hkv"], a["W"],
                 a["d"], a["scale"], a["ws"], a["nb"], None)

    assert call(pos=None) == 1
    assert call(ws=None) == 1
    assert call(W=0) == 2
    assert call(Hq=8, Hkv=3) == 2
    assert call(Hq=32, Hkv=1) == 4  # more than 16 query heads per KV head
    assert call(d=80) == 4
    assert call(scale=0.0) == 7
    assert call(q=P + 8) == 3
    assert call(pos=P + 2) == 3
    assert call(ws=P + 16) == 3  # the workspace wants 256-byte alignment
    assert call(nb=n - 1) == 8


def test_cache_and_chunk_validation(L):
    assert L.swa_cache_append(P, P, P, P, None, 2, 2, 64, 128, 1, None) == 1
    assert L.swa_cache_append(P, P, P, P, P, 2, 2, 64, 128, 0, None) == 2
    assert L.swa_cache_append(P, P, P, P, P, 2, 2, 64, 96, 1, None) == 4
    g = L.swa_cache_gather
    assert g(P, P, P, None, 2, 2, 64, 128, 100, 63, 80, None) == 1
    assert g(P, P, P, P, 2, 2, 64, 128, 10, 11, 80, None) == 2  # more history than positions
    assert g(P, P, P, P, 2, 2, 64, 128, 100, 65, 80, None) == 2  # more than W slots
    assert g(P, P, P, P, 2, 2, 64, 128, 100, 63, 40, None) == 2  # context shorter than history
    c = L.swa_chunk_fwd
    assert c(P, P, P, None, 1, 4, 2, 16, 100, 128, 32, 0.1, None) == 1
    assert c(P, P, P, P, 1, 4, 2, 101, 100, 128, 32, 0.1, None) == 2  # C > L
    assert c(P, P, P, P, 1, 4, 2, 0, 100, 128, 32, 0.1, None) == 2
    assert c(P, P, P, P, 1, 4, 2, 16, 100, 128, 0, 0.1, None) == 2


def test_lse_global_and_per_head_lambda_validation(L):
    assert L.swa_attn_fwd_lse(P, P, P, P, P + 2, 1, 2, 2, 128, 64, 16, 0.125, None) == 3
    assert L.strided_attn_fwd_lse(P, P, P, P, P + 1, 1, 2, 2, 128, 64, 16, 4, 0.125, None) == 3
    assert L.global_attn_fwd(P, P, P, P, 1, 2, 2, 128, 64, 16, -1, 0.125, None) == 2
    assert L.global_attn_fwd(None, P, P, P, 1, 2, 2, 128, 64, 16, 4, 0.125, None) == 1
    assert L.diff_attn_fwd_heads(P, P, P, P, P, None, P, 1, 2, 2, 128, 64, 0.125, None) == 1
    assert L.diff_attn_fwd_heads(P, P, P, P, P, P + 2, P, 1, 2, 2, 128, 64, 0.125, None) == 3


def test_diff_window_validation(L):
    f = L.diff_swa_attn_fwd
    assert f(P, P, None, P, P, 0.8, None, P, 1, 2, 2, 128, 64, 32, 0.125, None) == 1
    assert f(P, P, P, P, P, 0.8, None, P, 1, 2, 2, 128, 64, 0, 0.125, None) == 2
    assert f(P, P, P, P, P, float("nan"), None, P, 1, 2, 2, 128, 64, 32, 0.125, None) == 7
    assert f(P, P, P, P, P, 0.8, P + 2, P, 1, 2, 2, 128, 64, 32, 0.125, None) == 3
    assert f(P, P, P, P, P + 8, 0.8, None, P, 1, 2, 2, 128, 64, 32, 0.125, None) == 3
    assert f(P, P, P, P, P, 0.8, None, P, 1, 2, 2, 128, 96, 32, 0.125, None) == 4


def test_bwd_validation(L):
    f = L.swa_attn_bwd
    n = L.swa_attn_bwd_workspace_bytes(2, 4, 300)
    assert n >= 2 * 4 * 300 * 4 and n % 256 == 0
    assert L.swa_attn_bwd_workspace_bytes(0, 4, 300) == 0
    ok = dict(q=P, k=P, v=P, out=P, lse=P, g=P, dq=P, dk=P, dv=P, B=2, Hq=4, Hkv=2, N=300, d=64,
              W=50, scale=0.125, ws=P, nb=n)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["q"], a["k"], a["v"], a["out"], a["lse"], a["g"], a["dq"], a["dk"], a["dv"],
                 a["B"], a["Hq"], a["Hkv"], a["N"], a["d"], a["W"], a["scale"], a["ws"], a["nb"],
                 None)

    assert call(lse=None) == 1
    assert call(dv=None) == 1
    assert call(ws=None) == 1
    assert call(W=0) == 2
    assert call(Hq=4, Hkv=3) == 2
    assert call(B=1, Hq=65536, Hkv=1) == 2
    assert call(d=96) == 4
    assert call(scale=float("inf")) == 7
    assert call(dk=P + 8) == 3
    assert call(lse=P + 2) == 3
    assert call(ws=P + 4) == 3
    assert call(nb=n - 1) == 8


@pytest.mark.parametrize("form", ["strided", "global"])
def test_strided_and_global_bwd_validation(L, form):
    f = getattr(L, f"{form}_attn_bwd")
    wsf = getattr(L, f"{form}_attn_bwd_workspace_bytes")
    B, Hq, Hkv, N, d, W, x = 2, 4, 2, 3000, 64, 256, 128 if form == "strided" else 64
    n = wsf(B, Hq, Hkv, N, d, W, x)
    plain = L.swa_attn_bwd_workspace_bytes(B, Hq, N)
    assert n > plain  # delta plus the compact keys' partial sums
    assert wsf(B, Hq, Hkv, N, d, N, x) == plain  # W >= N: no key before any window
    assert wsf(0, Hq, Hkv, N, d, W, x) == 0 and wsf(B, Hq, Hkv, N, 96, W, x) == 0
    if form == "global":
        assert wsf(B, Hq, Hkv, N, d, W, 0) == plain  # no global tokens: the window
    ok = dict(q=P, k=P, v=P, out=P, lse=P, g=P, dq=P, dk=P, dv=P, B=B, Hq=Hq, Hkv=Hkv, N=N, d=d,
              W=W, x=x, scale=0.125, ws=P, nb=n)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["q"], a["k"], a["v"], a["out"], a["lse"], a["g"], a["dq"], a["dk"], a["dv"],
                 a["B"], a["Hq"], a["Hkv"], a["N"], a["d"], a["W"], a["x"], a["scale"], a["ws"],
                 a["nb"], None)

    assert call(dq=None) == 1
    assert call(W=0) == 2
    assert call(x=-1) == 2
    if form == "strided":
        assert call(x=0) == 2
    assert call(d=96) == 4
    assert call(scale=0.0) == 7
    assert call(dv=P + 8) == 3
    assert call(nb=n - 1) == 8
    assert L.global_attn_fwd_lse(P, P, P, P, P, 1, 2, 2, 128, 64, 16, -1, 0.125, None) == 2
    assert L.global_attn_fwd_lse(P, P, P, P, P + 2, 1, 2, 2, 128, 64, 16, 4, 0.125, None) == 3


def test_diff_bwd_validation(L):
    f = L.diff_attn_bwd
    n = L.diff_attn_bwd_workspace_bytes(2, 4, 2, 300, 64)
    assert n == 2 * L.swa_attn_bwd_workspace_bytes(2, 4, 300) + 2 * 2 * 300 * 64 * 4
    assert L.diff_attn_bwd_workspace_bytes(2, 4, 2, 300, 96) == 0
    ok = dict(q1=P, k1=P, q2=P, k2=P, v=P, lam=0.8, lh=None, o1=P, l1=P, o2=P, l2=P, g=P, dq1=P,
              dk1=P, dq2=P, dk2=P, dv=P, dl=None, B=2, Hq=4, Hkv=2, N=300, d=64, W=100,
              scale=0.125, ws=P, nb=n)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["q1"], a["k1"], a["q2"], a["k2"], a["v"], a["lam"], a["lh"], a["o1"], a["l1"],
                 a["o2"], a["l2"], a["g"], a["dq1"], a["dk1"], a["dq2"], a["dk2"], a["dv"], a["dl"],
                 a["B"], a["Hq"], a["Hkv"], a["N"], a["d"], a["W"], a["scale"], a["ws"], a["nb"],
                 None)

    assert call(o2=None) == 1
    assert call(l1=None) == 1
    assert call(dk2=None) == 1
    assert call(W=0) == 2
    assert call(Hq=4, Hkv=3) == 2
    assert call(d=96) == 4
    assert call(lam=float("nan")) == 7
    assert call(scale=-1.0) == 7
    assert call(dq2=P + 8) == 3
    assert call(dl=P + 2) == 3
    assert call(lh=P + 1) == 3
    assert call(nb=n - 1) == 8


def test_header_compiles_and_library_links_from_c(tmp_path):
    """The header is valid C and the library links and answers from a C program."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib_dir = os.path.dirname(pkg.LIBRARY_PATH)
    exe = str(tmp_path / "abi_from_c")
    src = os.path.join(ROOT, "tests", "abi_c", "abi_from_c.c")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        src, "-o", exe, "-L", lib_dir, "-lswa_b300", f"-Wl,-rpath,{lib_dir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr
