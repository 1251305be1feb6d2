"""Host-only checks of the C ABI (no GPU needed): the library loads, exports
every function include/rmsnorm.h declares, and rejects bad arguments on the
host before any CUDA call. Pointers here are never dereferenced: each case
fails validation first.
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from memory_bound_normalization_fwd_gb300 import binding as B
from memory_bound_normalization_fwd_gb300 import build as BUILD

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rmsnorm.h")


@pytest.fixture(scope="module")
def lib():
    BUILD.build()
    return B.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rmsnorm_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert _declared_functions() == sorted(B.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_version_and_strerror(lib):
    assert B.rmsnorm_version() == 1
    for code in B.STATUS:
        assert B.rmsnorm_strerror(code) != "unknown status"
    assert B.rmsnorm_strerror(12345) == "unknown status"


def test_options_struct_layout_matches_header():
    text = open(HEADER).read()
    body = re.search(r"typedef struct rmsnorm_options \{(.*?)\} rmsnorm_options_t;", text, re.S)
    fields = re.findall(r"int(32|64)_t\s+(\w+);", body.group(1))
    assert [n for _, n in fields] == [n for n, _ in B.Options._fields_]
    assert ctypes.sizeof(B.Options) == 48
    body = re.search(r"typedef struct rmsnorm_plan \{(.*?)\} rmsnorm_plan_t;", text, re.S)
    assert [n for n in re.findall(r"int32_t\s+(\w+);", body.group(1))] == \
        [n for n, _ in B.Plan._fields_]


X, W_, Y, R = 0x10000, 0x20000000, 0x30000000, 0x40000000  # never dereferenced


def _call(lib, x=X, w=W_, y=Y, r=R, M=4, N=8, eps=1e-6, off=0.0, dt=0, opts=None):
    return B.rmsnorm_fwd_ex(x, w, y, r, M, N, eps, off, dt, opts, 0)


@pytest.mark.parametrize("kw,code", [
    (dict(dt=3), -3), (dict(dt=-1), -3),
    (dict(M=-1), -2), (dict(N=0), -2), (dict(N=-5), -2), (dict(M=1 << 62, N=4), -2),
    (dict(eps=-1e-6), -4), (dict(eps=float("nan")), -4), (dict(eps=float("inf")), -4),
    (dict(off=float("nan")), -4), (dict(off=float("inf")), -4),
    (dict(w=0), -1), (dict(x=0), -1), (dict(y=0), -1),
    (dict(x=X + 1), -10), (dict(y=Y + 1), -10), (dict(w=W_ + 1), -10), (dict(r=R + 2), -10),
    (dict(y=X + 2), -5),            # y overlaps x without being equal to it
    (dict(r=X + 16), -5),           # rstd inside x
    (dict(r=Y + 8), -5),            # rstd inside y
    (dict(w=Y + 4), -5),            # w inside y
    (dict(x=Y, w=Y + 2), -5),       # in place, w inside x == y
])
def test_validation_errors(lib, kw, code):
    assert _call(lib, **kw) == code
    assert B.rmsnorm_last_error() != ""


def _call_strided(lib, x=X, ldx=8, w=W_, y=Y, ldy=8, r=R, M=4, N=8, opts=None):
    return B.rmsnorm_fwd_strided(x, ldx, w, y, ldy, r, M, N, 1e-6, 0.0, 0, opts, 0)


@pytest.mark.parametrize("kw,code", [
    (dict(ldx=7), -2), (dict(ldy=4), -2), (dict(ldx=-8), -2),
    (dict(ldx=1 << 45, M=1 << 3), -2),            # span beyond 2^48 bytes
    (dict(y=X, ldx=16, ldy=8), -5),                # in place with different strides
    (dict(y=X + 2 * 8, ldx=16, ldy=16), -5),       # interleaved rows: spans overlap
    (dict(r=X + 3 * 16 * 2, ldx=16), -5),          # rstd inside the span of x
    (dict(x=0), -1), (dict(w=X + 1), -10),
])
def test_strided_validation_errors(lib, kw, code):
    assert _call_strided(lib, **kw) == code
    assert B.rmsnorm_last_error() != ""


@pytest.mark.parametrize("kw,code", [
    (dict(x=X + 2), -10), (dict(y=Y + 2), -10), (dict(w=W_ + 2), -10),  # fp32: 4-byte alignment
    (dict(y=X + 4 * 8 * 4 - 4), -5),      # y starts on x's last element
    (dict(w=Y + 4 * 8 * 4 - 4), -5),      # w on y's last element (4-byte elements)
    (dict(r=X + 4 * 8 * 4 - 4), -5),
    (dict(M=1 << 44, N=8), -2),           # 2^46 elements of 4 bytes: 2^48 bytes
])
def test_fp32_validation_uses_four_byte_elements(lib, kw, code):
    assert _call(lib, dt=2, **kw) == code
    assert B.rmsnorm_last_error() != ""


def test_backward_fp32_checks_four_byte_elements(lib):
    call = lambda **k: B.rmsnorm_bwd(k.get("x", X), W_, R, k.get("dy", 0x60000000), k.get("dx", Y),
                                     0x70000000, 4, 8, 0.0, 2, 0x50000000, 1 << 20, None, 0)
    assert call(x=X + 2) == -10            # 2-byte aligned is not enough for fp32
    assert call(dx=X + 4 * 8 * 4 - 4) == -5  # dx starts on x's last 4-byte element
    assert call(dx=Y, dy=Y + 64) == -5       # dy inside dx (4 x 8 x 4 bytes)
    assert call(x=X, dy=0x7) == -10
    assert B.rmsnorm_bwd(X, W_, R, 0x60000000, Y, 0x70000000, 4, 8, 0.0, 3, 0x50000000, 1 << 20,
                         None, 0) == -3


def test_m_zero_is_ok_without_buffers(lib):
    assert _call(lib, x=0, y=0, r=0, M=0) == 0
    assert _call_strided(lib, x=0, y=0, r=0, M=0, ldx=100, ldy=9) == 0


@pytest.mark.parametrize("field,value", [("variant", 6), ("variant", -1), ("max_ctas", -1),
                                         ("stages", 9), ("stages", -1), ("wait_limit_ns", -5),
                                         ("lanes_per_row", -2), ("struct_size", 8),
                                         ("flags", 64), ("cluster_size", 17),
                                         ("cluster_size", -1), ("l2_prefetch", -2),
                                         ("l2_prefetch", 16), ("prewait_prefetch", -2),
                                         ("prewait_prefetch", 16)])
def test_bad_options(lib, field, value):
    o = B.make_options()
    setattr(o, field, value)
    assert _call(lib, opts=o) == -9


def test_bwd_validation_errors(lib):
    ws = 0x50000000
    call = lambda **k: B.rmsnorm_bwd(k.get("x", X), k.get("w", W_), k.get("r", R), k.get("dy", 0x60000000),
                                     k.get("dx", Y), k.get("dw", 0x70000000), k.get("M", 4), k.get("N", 8),
                                     0.0, k.get("dt", 0), k.get("ws", ws), 1 << 20, None, 0)
    assert call(dt=3) == -3
    assert call(M=-1) == -2
    assert call(w=0) == -1
    assert call(dw=0) == -1
    assert call(ws=0) == -1
    assert call(ws=ws + 8) == -10
    assert call(dx=X + 2) == -5          # partial overlap with x
    assert call(dw=W_) == -5             # dw over w
    assert call(r=R + 1) == -10


# ---------------------------------------------------------------- host-buffer forward

@pytest.mark.parametrize("M,N,dt,chunk,want", [
    (0, 512, 0, 0, 0),                                    # slots + rstd of all M rows:
    (10, 512, 0, 0, 10240 + 256),                         # one chunk of all 10 rows: one slot
    (100000, 512, 0, 0, 4 * (4 << 20) + 400128),          # 4096-row chunks (4 MiB), four slots
    (20, 3, 2, 7, 3 * 256 + 256),                         # fp32, 3 chunks of 7 rows: 3 slots
    (14, 3, 2, 7, 2 * 256 + 256),                         # two chunks: two slots
    (5, 1000, 1, 1, 4 * 2048 + 256),                      # one row per chunk
])
def test_host_path_workspace_size(lib, M, N, dt, chunk, want):
    assert B.rmsnorm_fwd_host_workspace_size(M, N, dt, chunk) == want


@pytest.mark.parametrize("args,code", [((4, 8, 5, 0), -3), ((4, 8, 0, -1), -2), ((-1, 8, 0, 0), -2),
                                       ((4, 0, 0, 0), -2)])
def test_host_path_workspace_size_errors(lib, args, code):
    with pytest.raises(B.RMSNormError) as e:
        B.rmsnorm_fwd_host_workspace_size(*args)
    assert e.value.status == code


HX, HY, HR = 0x7F0000000000, 0x7F0010000000, 0x7F0020000000  # "host" addresses, never touched
WS = 0x50000000


def _host_call(lib, x=HX, w=W_, y=HY, r=HR, M=4, N=8, dt=0, chunk=0, ws=WS, nbytes=1 << 20,
               opts=None):
    return B.rmsnorm_fwd_host(x, w, y, r, M, N, 1e-6, 0.0, dt, chunk, ws, nbytes, opts, 0)


@pytest.mark.parametrize("kw,code", [
    (dict(ws=0), -1), (dict(ws=WS + 8), -10), (dict(nbytes=100), -11),
    (dict(ws=W_), -5),                         # workspace over w
    (dict(ws=HX, nbytes=1 << 20), -5),         # workspace over x
    (dict(w=0), -1), (dict(x=0), -1), (dict(dt=7), -3), (dict(chunk=-3), -2),
    (dict(y=HX + 2), -5),                      # y partly over x
    (dict(r=HX + 4), -5),                      # rstd inside x
])
def test_host_path_validation_before_any_cuda_call(lib, kw, code):
    assert _host_call(lib, **kw) == code
    assert B.rmsnorm_last_error() != ""


def test_host_path_m_zero_needs_nothing(lib):
    assert _host_call(lib, x=0, y=0, r=0, M=0, ws=0, nbytes=0) == 0


CONSUMER = r"""
#include "rmsnorm.h"
#include <stdio.h>
#include <string.h>

int main(void) {
    rmsnorm_options_t o;
    int64_t bytes = -1;
    memset(&o, 0, sizeof(o));
    o.struct_size = (int)sizeof(o);
    /* host-side validation only: a null x is refused before any CUDA call */
    int rc = rmsnorm_fwd(NULL, NULL, NULL, NULL, 4, 8, 1e-6f, 0.0f, RMSNORM_DTYPE_BF16, NULL);
    int rc_ex = rmsnorm_fwd_ex(NULL, NULL, NULL, NULL, 4, 8, 1e-6f, 0.0f, RMSNORM_DTYPE_FP16, &o, NULL);
    int rc_ws = rmsnorm_fwd_host_workspace_size(1000, 512, RMSNORM_DTYPE_BF16, 0, &bytes);
    printf("%d %d %d %d %lld|%s|%s\n", rmsnorm_version(), rc, rc_ex, rc_ws, (long long)bytes,
           rmsnorm_strerror(rc), rmsnorm_last_error());
    return 0;
}
"""


@pytest.mark.parametrize("compiler,std", [("gcc", "-std=c99"), ("g++", "-std=c++17")])
def test_plain_c_and_cpp_consumers_compile_link_and_call(lib, tmp_path, compiler, std):
    # The header is the boundary: a C99 (and a C++) program that includes it
    # with warnings as errors, links the shared library and calls host-only
    # entry points gets the same answers as the Python binding.
    import shutil
    import subprocess
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not installed")
    src = tmp_path / ("consumer.c" if compiler == "gcc" else "consumer.cpp")
    src.write_text(CONSUMER)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(B.library_path())
    subprocess.run([compiler, std, "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                    os.path.join(ROOT, "include"), str(src), B.library_path(),
                    f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.strip()
    head, strerr, detail = out.split("|")
    version, rc, rc_ex, rc_ws, nbytes = (int(v) for v in head.split())
    assert version == B.rmsnorm_version()
    assert rc == rc_ex == -1 and strerr == B.rmsnorm_strerror(-1) and detail
    assert rc_ws == 0 and nbytes == B.rmsnorm_fwd_host_workspace_size(1000, 512, B.BF16, 0)


def test_struct_layouts_match_the_header(tmp_path):
    # The binding's ctypes structures mirror rmsnorm_options_t and
    # rmsnorm_plan_t: every field at the header's offset, same total size.
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not installed")
    fields = {"rmsnorm_options_t": B.Options, "rmsnorm_plan_t": B.Plan}
    lines = []
    for cname, cls in fields.items():
        lines.append(f'    printf("{cname} size %zu\\n", sizeof({cname}));')
        for name, _ in cls._fields_:
            lines.append(f'    printf("{cname} {name} %zu\\n", offsetof({cname}, {name}));')
    src = tmp_path / "layout.c"
    src.write_text('#include "rmsnorm.h"\n#include <stddef.h>\n#include <stdio.h>\n'
                   "int main(void) {\n" + "\n".join(lines) + "\n    return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for cname, cls in fields.items():
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for name, _ in cls._fields_:
            assert got[(cname, name)] == getattr(cls, name).offset, (cname, name)
