"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports exactly the functions include/rca_attn.h declares, and rejects invalid
arguments before touching any pointer or launching anything."""

import ctypes
import os
import re
import shutil
import subprocess

import pytest

from causal_head_attention_gb300 import _native
from causal_head_attention_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rca_attn.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return _native.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rca_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for n in ("rca_attn_fwd", "rca_attn_bwd", "rca_attn_bwd_workspace_size", "rca_stream_status",
              "rca_last_error", "rca_abi_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in rca_attn.h but not exported"
        assert n in _native._SIG, f"{n} has no binding signature"


def test_only_declared_symbols_are_exported(lib):
    """The library is built with hidden visibility: its dynamic symbol table
    holds the calls the header declares and nothing of its internals (which
    would let a second copy of the library, or a host program defining the
    same names, interfere with it)."""
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm (binutils) not installed")
    out = subprocess.run([nm, "-D", "--defined-only", lib._name], capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    linker = {"_init", "_fini", "__bss_start", "_edata", "_end", "__bss_start__", "__bss_end__", "__end__",
              "_bss_end__"}
    assert exported - linker == set(declared_functions())


def test_abi_version(lib):
    v = lib.rca_abi_version()
    assert v >> 16 == 1


FAKE = ctypes.c_void_p(4096)  # never dereferenced: every call below fails validation first
NULL = ctypes.c_void_p(0)


def fwd(lib, q=FAKE, B=1, Hq=2, Hkv=2, T=8, Dh=64, dt=1, out=FAKE, lse=FAKE):
    return lib.rca_attn_fwd(q, FAKE, FAKE, B, Hq, Hkv, T, Dh, out, lse, dt, NULL)


@pytest.mark.parametrize(
    "kw,status,needle",
    [
        (dict(q=NULL), 1, "null"),
        (dict(out=NULL), 1, "null"),
        (dict(T=0), 1, "fully masked"),
        (dict(B=0), 1, ">= 1"),
        (dict(Hq=3, Hkv=2), 1, "Hq % Hkv"),
        (dict(Dh=96), 2, "Dh=96"),
        (dict(Dh=128, dt=0), 2, "Dh=128"),
        (dict(dt=7), 1, "dtype"),
        (dict(q=ctypes.c_void_p(4100)), 1, "aligned"),
    ],
)
def test_fwd_validation(lib, kw, status, needle):
    assert fwd(lib, **kw) == status
    assert needle in lib.rca_last_error().decode()


def test_workspace_size_and_checks(lib):
    n = lib.rca_attn_bwd_workspace_size(4, 16, 16, 2048, 64, 1)
    assert n >= 4 * 2048 * 16 * 64 * 4 + 2 * 4 * 16 * 2048 * 4
    # fp32 storage adds bf16 hi/lo copies of Q, dO, K, V
    n32 = lib.rca_attn_bwd_workspace_size(4, 16, 4, 2048, 64, 0)
    assert n32 >= n + 4 * 2048 * 64 * 2 * 2 * (2 * 16 + 2 * 4) - 4096
    assert lib.rca_attn_bwd_workspace_size(0, 16, 16, 2048, 64, 1) == 0
    assert lib.rca_attn_bwd_workspace_size(1, 4, 8, 16, 64, 1) == 0  # Hkv > Hq
    assert lib.rca_attn_bwd_workspace_size(1, 4, 4, 16, 64, 9) == 0  # unknown dtype
    # too small a workspace is rejected before anything runs
    st = lib.rca_attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 2, 8, 64, 1,
                          ctypes.c_void_p(4096), 16, NULL)
    assert st == 1 and "workspace too small" in lib.rca_last_error().decode()
    st = lib.rca_attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 2, 8, 64, 1,
                          ctypes.c_void_p(4096 + 16), 1 << 30, NULL)
    assert st == 1 and "256-byte" in lib.rca_last_error().decode()


def test_error_text_is_per_thread(lib):
    import threading

    assert fwd(lib, Dh=96) == 2
    seen = {}

    def other():
        seen["msg"] = lib.rca_last_error().decode()

    t = threading.Thread(target=other)
    t.start()
    t.join()
    assert seen["msg"] == ""
    assert "Dh=96" in lib.rca_last_error().decode()


def test_timeout_setter(lib):
    old = lib.rca_set_wait_timeout_ns(5)
    assert lib.rca_set_wait_timeout_ns(old) == 1000000


def decode(lib, q=FAKE, B=2, Hq=4, Hkv=2, Dh=64, page_size=16, max_pages=8, num_pages=20, dt=1, out=FAKE,
           lse=FAKE, ws=ctypes.c_void_p(1 << 20), ws_bytes=1 << 30, table=FAKE):
    return lib.rca_paged_decode(q, FAKE, FAKE, table, FAKE, B, Hq, Hkv, Dh, page_size, max_pages, num_pages,
                                out, lse, dt, ws, ws_bytes, NULL)


@pytest.mark.parametrize(
    "kw,status,needle",
    [
        (dict(q=NULL), 1, "null"),
        (dict(table=NULL), 1, "null"),
        (dict(B=0), 1, ">= 1"),
        (dict(num_pages=0), 1, ">= 1"),
        (dict(Hq=3, Hkv=2), 1, "Hq % Hkv"),
        (dict(Dh=96), 2, "Dh=96"),
        (dict(page_size=12), 1, "power of two"),
        (dict(page_size=1 << 17), 1, "power of two"),
        (dict(B=8193), 2, "at most"),
        (dict(max_pages=1 << 27), 1, "2^30"),
        (dict(dt=7), 1, "dtype"),
        (dict(q=ctypes.c_void_p(4104)), 1, "16-byte"),
        (dict(lse=ctypes.c_void_p(4098)), 1, "4-byte"),
        (dict(ws=NULL), 1, "workspace is null"),
        (dict(ws=ctypes.c_void_p(4096 + 128)), 1, "256-byte"),
        (dict(ws_bytes=64), 1, "too small"),
    ],
)
def test_decode_validation(lib, kw, status, needle):
    assert decode(lib, **kw) == status
    assert needle in lib.rca_last_error().decode()


def test_decode_workspace_size(lib):
    # one chunk of 256 positions per request at most: no partials, minimum size
    assert lib.rca_paged_decode_workspace_size(4, 8, 8, 64, 16, 16, 1) == 256
    # B * Hq * chunks rows of (max, sum) and Dh floats
    n = lib.rca_paged_decode_workspace_size(64, 16, 16, 64, 16, 128, 1)
    assert n >= 64 * 16 * 8 * (64 + 2) * 4 and n % 256 == 0
    assert lib.rca_paged_decode_workspace_size(4, 8, 8, 96, 16, 16, 1) == 0
    assert lib.rca_paged_decode_workspace_size(4, 8, 8, 64, 12, 16, 1) == 0


def mat_fwd(lib, q=FAKE, B=1, Hq=2, Hkv=2, T=8, Dh=64, dt=1, probs=FAKE, ws=ctypes.c_void_p(1 << 20),
            ws_bytes=1 << 30):
    return lib.rca_attn_materialized_fwd(q, FAKE, FAKE, B, Hq, Hkv, T, Dh, FAKE, probs, FAKE, dt, ws, ws_bytes,
                                         NULL)


@pytest.mark.parametrize(
    "kw,status,needle",
    [
        (dict(q=NULL), 1, "null"),
        (dict(probs=NULL), 1, "null"),
        (dict(T=0), 1, "fully masked"),
        (dict(Hq=3, Hkv=2), 1, "Hq % Hkv"),
        (dict(Dh=96), 2, "Dh=96"),
        (dict(T=70000), 1, "too large"),
        (dict(B=64, Hq=64, T=16384), 1, "too large"),
        (dict(probs=ctypes.c_void_p(4100)), 1, "aligned"),
        (dict(ws=NULL), 1, "workspace is null"),
        (dict(ws_bytes=100), 1, "too small"),
    ],
)
def test_materialized_validation(lib, kw, status, needle):
    assert mat_fwd(lib, **kw) == status
    assert needle in lib.rca_last_error().decode()


def test_materialized_bwd_validation(lib):
    st = lib.rca_attn_materialized_bwd(FAKE, FAKE, FAKE, FAKE, NULL, NULL, FAKE, FAKE, FAKE, 1, 2, 2, 8, 64, 1,
                                       ctypes.c_void_p(1 << 20), 1 << 30, NULL)
    assert st == 1 and "null" in lib.rca_last_error().decode()


@pytest.mark.parametrize(
    "kw,needle",
    [
        (dict(probs=NULL), "null"),
        (dict(grad=NULL), "null"),
        (dict(tile=0), "tile must be >= 1"),
        (dict(tile=-128), "tile must be >= 1"),
        (dict(T=0), ">= 1"),
        (dict(T=70000), "too large"),
        (dict(scale=float("nan")), "finite"),
        (dict(grad=ctypes.c_void_p(4100)), "aligned"),
    ],
)
def test_softmax_bwd_tiled_validation(lib, kw, needle):
    a = dict(probs=FAKE, grad=FAKE, extra=NULL, N=2, T=256, tile=128, scale=0.125)
    a.update(kw)
    st = lib.rca_causal_softmax_bwd_tiled(a["probs"], a["grad"], a["extra"], a["N"], a["T"], a["tile"], a["scale"],
                                          NULL)
    assert st == 1
    assert needle in lib.rca_last_error().decode()
    assert "rca_causal_softmax_bwd_tiled" in lib.rca_last_error().decode() or needle != "null"


def test_materialized_workspace_size(lib):
    n = lib.rca_attn_materialized_workspace_size(4, 16, 16, 2048, 64, 1)
    # bf16 storage: dP [B,Hq,T,T] fp32 only
    assert n >= 4 * 16 * 2048 * 2048 * 4
    # fp32 storage adds three bf16 parts of each of Q, K, V, dO
    n32 = lib.rca_attn_materialized_workspace_size(4, 16, 16, 2048, 64, 0)
    assert n32 >= n + 4 * 3 * 4 * 2048 * 16 * 64 * 2
    assert lib.rca_attn_materialized_workspace_size(4, 16, 16, 2048, 96, 1) == 0


def test_qkv_validation(lib):
    assert lib.rca_attn_fwd_qkv(NULL, 1, 8, 2, 2, 64, FAKE, FAKE, 1, NULL) == 1
    assert "null" in lib.rca_last_error().decode()
    assert lib.rca_attn_fwd_qkv(FAKE, 1, 8, 3, 2, 64, FAKE, FAKE, 1, NULL) == 1
    assert "Hq % Hkv" in lib.rca_last_error().decode()
    assert lib.rca_attn_fwd_qkv(ctypes.c_void_p(4104), 1, 8, 2, 2, 64, FAKE, FAKE, 1, NULL) == 1
    assert "aligned" in lib.rca_last_error().decode()
    assert lib.rca_attn_bwd_qkv(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 2, 64, 1, ctypes.c_void_p(1 << 20), 16,
                                NULL) == 1
    assert "too small" in lib.rca_last_error().decode()


def test_varlen_validation(lib):
    WS, WB = ctypes.c_void_p(1 << 20), 1 << 30
    assert lib.rca_attn_fwd_varlen(FAKE, FAKE, FAKE, NULL, 1, 2, 2, 8, 64, FAKE, FAKE, 1, WS, WB, NULL) == 1
    assert "null" in lib.rca_last_error().decode()
    assert lib.rca_attn_fwd_varlen(FAKE, FAKE, FAKE, ctypes.c_void_p(4098), 1, 2, 2, 8, 64, FAKE, FAKE, 1, WS, WB,
                                   NULL) == 1
    assert "4-byte" in lib.rca_last_error().decode()
    assert lib.rca_attn_fwd_varlen(FAKE, FAKE, FAKE, FAKE, 5000, 2, 2, 8, 64, FAKE, FAKE, 1, WS, WB, NULL) == 2
    assert "B <= 4096" in lib.rca_last_error().decode()
    assert lib.rca_attn_fwd_varlen(FAKE, FAKE, FAKE, FAKE, 1, 2, 2, 8, 64, FAKE, FAKE, 1, WS, 64, NULL) == 1
    assert "too small" in lib.rca_last_error().decode()
    assert lib.rca_attn_varlen_workspace_size(4, 16, 16, 2048, 64, 1) > lib.rca_attn_bwd_workspace_size(
        4, 16, 16, 2048, 64, 1)
    assert lib.rca_attn_bwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 2, 0, 64, 1,
                                   ctypes.c_void_p(1 << 20), 1 << 30, NULL) == 1
    assert "fully masked" in lib.rca_last_error().decode()
