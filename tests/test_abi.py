"""The C-ABI library loads and exports what include/jattn.h declares; host-side
argument checks return their error codes without touching a GPU."""
import ctypes
import os
import re

import pytest

from jagged_attention_recsys_gdpa_gb300 import _binding as B
from jagged_attention_recsys_gdpa_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "jattn.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(jattn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("jattn_workspace_size", "jattn_fwd", "jattn_bwd", "jattn_get_status", "jattn_error_string"):
        assert n in names
    assert set(names) == set(B.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def _params(**kw):
    base = dict(B=2, total_q=10, total_kv=10, H=2, D=128, act=0, mask=1, window=0, scale=0.0, norm_by_lkv=0)
    base.update(kw)
    return B.params(**base)


def test_workspace_size_and_validation(lib):
    n = B.workspace_size(_params())
    assert n > 256 and n % 256 == 0
    bad = [
        dict(D=96), dict(D=0), dict(H=0), dict(B=0), dict(total_q=-1), dict(act=4), dict(mask=2), dict(mask=3),
        dict(mask=4), dict(scale=-1.0), dict(scale=float("nan")), dict(act=0, norm_by_lkv=1),
        dict(total_q=1 << 31), dict(B=1 << 31),
        # block masks need a width and do not combine with the window bit
        dict(mask=5, window=0), dict(mask=6, window=4), dict(mask=7, window=4), dict(mask=8, window=4),
    ]
    for kw in bad:
        size = ctypes.c_size_t(0)
        p = _params(**kw)
        assert lib.jattn_workspace_size(ctypes.byref(p), ctypes.byref(size)) == 1, kw
    for ok in (_params(mask=3, window=4), _params(mask=4, window=64), _params(mask=5, window=1)):
        assert B.workspace_size(ok) > 0
    # softmax needs room for Di; pointwise does not
    assert B.workspace_size(_params(total_q=100000)) > B.workspace_size(_params(total_q=100000, act=1))


def test_host_side_errors_before_any_launch(lib):
    p = _params()
    f = 1 << 20  # never dereferenced: every call below must fail on the host first
    big = 1 << 30

    def fwd(q_off=f, kv_off=f, q=f, k=f, v=f, o=f, lse=f, ws=f, ws_bytes=big, pp=p):
        return lib.jattn_fwd(ctypes.byref(pp), q_off, kv_off, q, k, v, o, lse, ws, ws_bytes, None)

    assert fwd(q_off=None) == 1
    assert fwd(q=f + 2) == 4
    assert fwd(ws=None) == 3
    assert fwd(ws=f + 16) == 3
    assert fwd(ws_bytes=64) == 3
    assert fwd(lse=None) == 1
    assert fwd(pp=_params(D=80)) == 1
    pb = _params(D=80)
    assert lib.jattn_bwd(ctypes.byref(pb), *([f] * 11), f, big, None) == 1
    assert lib.jattn_bwd(ctypes.byref(p), f, f, f, f, f, f, f, f, f + 8, f, f, f, big, None) == 4
    assert lib.jattn_bwd(ctypes.byref(p), f, f, f, f, f, None, f, f, f, f, f, f, big, None) == 1


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    f = 1 << 20  # never dereferenced: the size check comes before any device work
    p = _params(B=1, total_q=1 << 30, total_kv=16)
    rc = lib.jattn_fwd_noalloc(ctypes.byref(p), f, f, f, f, f, f, f, None, None)
    assert rc == 8
    assert b"bytes of scratch" in lib.jattn_last_error()


def test_mxfp8_forward_checks_arguments(lib):
    f = 1 << 20  # never dereferenced: every call below must fail on the host first
    big = 1 << 30

    def call(pp=None, q=f, qs=f, k=f, ks=f, v=f, vs=f, o=f, lse=f):
        pp = pp if pp is not None else _params(mask=1)
        return lib.jattn_fwd_mxfp8(ctypes.byref(pp), f, f, q, qs, f, k, ks, v, vs, f, o, lse, f, big, None)

    assert call(pp=_params(act=1, norm_by_lkv=1)) == 1  # softmax only
    assert call(pp=_params(D=64)) == 1                  # D = 128 only
    assert call(lse=None) == 1
    assert call(qs=None) == 1
    assert call(q=f + 8) == 4
    assert call(vs=f + 2) == 4                          # scale words are read 4 bytes at a time
    assert lib.jattn_fwd_mxfp8(ctypes.byref(_params()), f, f, f, f, None, f, f, f, f, f, f, f, f, big, None) == 1


def test_mxfp8_backward_checks_arguments(lib):
    f = 1 << 20  # never dereferenced: every call below must fail on the host first
    big = 1 << 30

    def call(pp=None, q=f, qs=f, k=f, ks=f, v=f, vs=f, o=f, lse=f, do=f, dos=f, dq=f, dk=f, dv=f, qbs=f):
        pp = pp if pp is not None else _params(mask=1)
        return lib.jattn_bwd_mxfp8(ctypes.byref(pp), f, f, q, qs, qbs, k, ks, v, vs, f, o, lse, do, dos, dq, dk, dv,
                                   f, big, None)

    assert call(pp=_params(act=1, norm_by_lkv=1)) == 1  # softmax only
    assert call(pp=_params(D=64)) == 1                  # D = 128 only
    for name in ("lse", "o", "do", "dos", "dq", "dk", "qbs"):
        assert call(**{name: None}) == 1, name
    assert call(do=f + 8) == 4
    assert call(dv=f + 8) == 4
    assert call(dos=f + 2) == 4                         # scale words are read 4 bytes at a time


def test_error_strings(lib):
    for code in range(10):
        assert B.error_string(code) != "unknown error code", code
    assert B.error_string(99) == "unknown error code"


def test_python_api_rejects_block_with_window():
    import jagged_attention_recsys_gdpa_gb300 as J

    with pytest.raises(ValueError):
        J._mask(True, 16, 64)
    assert J._mask(False, 0, 64) == 4 and J._mask(True, 0, 64) == 5
    assert J._width(0, 64) == 64 and J._width(256, 0) == 256


def test_rope_entry_points_check_arguments(lib):
    """Host-side argument checks of the rotary entry points (no launch)."""
    p = _params(D=64)
    ws = ctypes.c_void_p(256)  # never dereferenced: every call below fails its checks first
    fake = ctypes.c_void_p(4096)
    off = ctypes.c_void_p(8192)
    # missing tables, bad row counts, unaligned tables
    for cos, sin, rows, want in ((None, fake, 10, 1), (fake, None, 10, 1), (fake, fake, 0, 1),
                                 (fake, fake, 1 << 31, 1), (ctypes.c_void_p(4100), fake, 10, 4)):
        assert lib.jattn_rope(ctypes.byref(p), off, off, 0, 0, fake, fake, cos, sin, rows, ws, 256, None) == want
        assert lib.jattn_bwd_rope(ctypes.byref(p), off, off, fake, fake, fake, fake, fake, fake, cos, sin, rows, fake,
                                  fake, fake, ws, 1 << 30, None) == want
    # keys / inverse must be 0 or 1; the workspace must hold the status word
    assert lib.jattn_rope(ctypes.byref(p), off, off, 2, 0, fake, fake, fake, fake, 10, ws, 256, None) == 1
    assert lib.jattn_rope(ctypes.byref(p), off, off, 0, 5, fake, fake, fake, fake, 10, ws, 256, None) == 1
    assert lib.jattn_rope(ctypes.byref(p), off, off, 0, 0, fake, fake, fake, fake, 10, ws, 128, None) == 3


def test_bwd_rope_workspace_size(lib):
    p = _params(D=128, total_q=1000, total_kv=1000)
    base = B.workspace_size(p)
    assert B.bwd_rope_workspace_size(p, 4096) == base + 4096 * 128 * 4
    assert B.bwd_rope_workspace_size(p, 3) == base + 1536  # two 3 x 64 fp32 tables
    size = ctypes.c_size_t(0)
    assert lib.jattn_bwd_rope_workspace_size(ctypes.byref(p), 0, ctypes.byref(size)) == 1


def test_mxfp8_entry_checks_arguments(lib):
    """Host-side checks of jattn_mxfp8_quantize (no launch) and the scale-row bound."""
    assert lib.jattn_mxfp8_scale_rows(3, 100) == 100 // 32 + 3
    assert lib.jattn_mxfp8_scale_rows(-1, 5) == 0
    fake, off, ws = ctypes.c_void_p(4096), ctypes.c_void_p(8192), ctypes.c_void_p(256)
    q = lib.jattn_mxfp8_quantize
    assert q(0, 10, 2, 64, off, fake, fake, fake, fake, ws, 512, None) == 1      # B < 1
    assert q(2, 10, 2, 96, off, fake, fake, fake, fake, ws, 512, None) == 1      # D
    assert q(2, 10, 0, 64, off, fake, fake, fake, fake, ws, 512, None) == 1      # H
    assert q(2, 10, 2, 64, None, fake, fake, fake, fake, ws, 512, None) == 1     # offsets
    assert q(2, 10, 2, 64, off, ctypes.c_void_p(4100), fake, fake, fake, ws, 512, None) == 4  # alignment
    assert q(2, 10, 2, 64, off, fake, fake, fake, fake, ws, 256, None) == 3      # workspace too small
    assert q(2, 10, 2, 64, off, fake, fake, fake, fake, ctypes.c_void_p(300), 512, None) == 3  # misaligned


def test_header_is_plain_c_and_links(tmp_path, lib):
    """include/jattn.h compiles as C99 (no C++ in the boundary), and a C
    program links against libjattn.so and calls entry points that need no GPU."""
    import shutil
    import subprocess

    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = tmp_path / "use_jattn.c"
    src.write_text(
        '#include <stdio.h>\n#include "jattn.h"\n'
        "int main(void) {\n"
        "  jattn_params_t p = {2, 100, 100, 4, 128, JATTN_SOFTMAX, JATTN_MASK_CAUSAL, 0, 0.0f, 0};\n"
        "  size_t bytes = 0;\n"
        "  int rc = jattn_workspace_size(&p, &bytes);\n"
        '  printf("%d %zu %s %lld\\n", rc, bytes, jattn_error_string(JATTN_ERR_OFFSETS),\n'
        "         (long long)jattn_mxfp8_scale_rows(3, 100));\n"
        "  return rc;\n}\n"
    )
    exe = tmp_path / "use_jattn"
    libdir = os.path.dirname(B.library_path())
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe),
                        "-L", libdir, "-ljattn", f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    rc, nbytes, rest = out.stdout.split(" ", 2)
    assert rc == "0" and int(nbytes) == B.workspace_size(_params(B=2, total_q=100, total_kv=100, H=4, D=128, mask=1))
    assert rest.strip().endswith(" 6") and "offsets" in rest


def test_short_query_shapes_hold_their_schedule(lib):
    """Pooling-shaped parameters (pointwise, no mask, D = 128, at most 64
    queries per sequence on average) reserve the short-query schedule and gate
    word in the workspace; other shapes do not."""
    pma = dict(B=512, total_q=16384, total_kv=1_600_000, H=8, D=128, act=2, mask=0, norm_by_lkv=1)
    base = B.workspace_size(_params(**pma))
    assert base > B.workspace_size(_params(**{**pma, "mask": 1}))                  # causal: general kernels only
    assert base > B.workspace_size(_params(**{**pma, "total_q": 64 * 512 + 1}))    # longer queries on average
    assert B.workspace_size(_params(**{**pma, "D": 64})) < base
    cross = dict(B=512, total_q=800_000, total_kv=37_000, H=8, D=128, act=1, mask=0, norm_by_lkv=1)
    assert B.workspace_size(_params(**cross)) > B.workspace_size(_params(**{**cross, "total_kv": 128 * 512 + 1}))


def test_short_query_path_rule():
    """bench.py's accounting mirrors the library's rule for the short-query path."""
    from jagged_attention_recsys_gdpa_gb300 import flops

    assert flops.short_query_path(2, 0, 128, [32, 32, 1], [2000, 0, 5])
    assert flops.short_query_path(1, 0, 128, [64, 3], [1, 1])
    assert flops.short_query_path(1, 0, 128, [5, 0], [7, 0])        # no queries and no keys: fine
    assert not flops.short_query_path(0, 0, 128, [32], [100])       # softmax
    assert not flops.short_query_path(1, 1, 128, [32], [100])       # causal
    assert not flops.short_query_path(1, 0, 64, [32], [100])        # D = 64
    assert not flops.short_query_path(1, 0, 128, [65, 1], [10, 10])  # a sequence beyond 64 queries (gate)
    assert not flops.short_query_path(1, 0, 128, [0, 32], [10, 10])  # keys no query sees (gate)
    assert not flops.short_query_path(1, 0, 128, [100, 100], [1, 1])  # average beyond 64
    # cross-attention over short key sequences: the fused backward's cross mode
    assert flops.short_key_path(1, 0, 128, [1000, 300, 0], [16, 128, 40])
    assert not flops.short_key_path(1, 0, 128, [32, 32], [100, 100])   # pooling shape (short queries)
    assert not flops.short_key_path(1, 0, 128, [1000, 300], [129, 5])  # a sequence beyond 128 keys (gate)
    assert not flops.short_key_path(1, 0, 128, [1000, 300], [0, 5])    # queries without keys (gate)
    assert not flops.short_key_path(0, 0, 128, [1000], [16])           # softmax
