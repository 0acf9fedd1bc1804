"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function the headers declare, and rejects bad arguments with the
documented status codes before launching anything."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from attention_backward_bwd_gb300 import binding
    return binding.lib()


def declared_functions():
    names = []
    for h in ("attn_bwd.h", "attn_diag.h"):
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_version(lib):
    assert b"sm_103a" in lib.attn_version()


def test_workspace_size_and_layout(lib):
    from attention_backward_bwd_gb300 import binding
    offs, rows = binding.workspace_layout(2, 300, 4, 128)
    assert rows == 2 * 384
    assert offs["lse2"] == 0 and offs["delta"] >= 4 * rows * 4
    assert offs["dqaccum"] >= offs["delta"] + 4 * rows * 4
    assert offs["sem"] >= offs["dqaccum"] + 4 * rows * 128 * 4
    size = binding.workspace_size(2, 300, 4, 128)
    # 4 heads x (rows / 128) query tiles x 4 row quarters of semaphores, 2 work counters
    assert size >= offs["sem"] + (4 * (rows // 128) * 4 + 2) * 4 and size % 256 == 0
    # head dims above 128 lay dQaccum out at width 256
    offs256, _ = binding.workspace_layout(2, 300, 4, 192)
    assert offs256["sem"] >= offs256["dqaccum"] + 4 * rows * 256 * 4
    # varlen: total rows + one padding tile per sequence
    _, vrows = binding.workspace_layout(3, 1000, 4, 64, varlen=True)
    assert vrows == ((1000 + 3 * 128 + 127) // 128) * 128
    assert lib.attn_bwd_workspace_size(0, 10, 1, 64, 0, 0) == 0


class FakeTensor:
    """Just enough of a tensor for the marshalling code: no memory behind it."""

    def __init__(self, shape, ptr=1 << 20, dtype="bf16", strides=None):
        import torch
        self.shape = shape
        self._ptr = ptr
        self.dtype = {"bf16": torch.bfloat16, "fp16": torch.float16, "f32": torch.float32}[dtype]
        if strides is None:
            strides, acc = [], 1
            for n in reversed(shape):
                strides.insert(0, acc)
                acc *= n
        self._strides = strides

    def dim(self):
        return len(self.shape)

    def stride(self, i):
        return self._strides[i]

    def data_ptr(self):
        return self._ptr

    def numel(self):
        n = 1
        for s in self.shape:
            n *= s
        return n


def call_bwd(lib, q, k, v, o, do, ws_bytes=1 << 30, lse_ptr=1 << 21, ws_ptr=1 << 24,
             dtype=None, causal=0, head_dim=None, cu=None):
    from attention_backward_bwd_gb300 import binding as bd
    ds = [bd._desc(t) for t in (q, k, v, o)]
    d_do, d_dq, d_dk, d_dv = bd._desc(do), bd._desc(q), bd._desc(k), bd._desc(v)
    b, sq, hq, d = q.shape
    sk, hk = k.shape[1], k.shape[2]
    dt = bd._dtype_code(q) if dtype is None else dtype
    return lib.attn_bwd(*(ctypes.byref(x) for x in ds), lse_ptr, ctypes.byref(d_do),
                        ctypes.byref(d_dq), ctypes.byref(d_dk), ctypes.byref(d_dv), dt, b, sq, sk,
                        hq, hk, head_dim or d, 0.125, causal, cu, cu, sq, sk, 0, ws_ptr, ws_bytes,
                        None)


def shapes(b=1, sq=64, sk=64, hq=2, hk=2, d=64, dtype="bf16", ptr=1 << 20):
    q = FakeTensor((b, sq, hq, d), ptr, dtype)
    k = FakeTensor((b, sk, hk, d), ptr, dtype)
    return q, k, FakeTensor((b, sk, hk, d), ptr, dtype), FakeTensor((b, sq, hq, d), ptr, dtype), \
        FakeTensor((b, sq, hq, d), ptr, dtype)


@pytest.mark.parametrize("case,code", [
    ("dtype", -1), ("head_dim", -2), ("head_dim_large", -2), ("gqa_ratio", -2), ("align", -4), ("stride", -3),
    ("null", -5), ("workspace_small", -6), ("workspace_align", -6), ("varlen_half", -9),
])
def test_argument_errors(lib, case, code):
    q, k, v, o, do = shapes()
    kw = {}
    if case == "dtype":
        q, k, v, o, do = shapes(dtype="f32")
    elif case == "head_dim":
        q, k, v, o, do = shapes(d=100)  # not a multiple of 8
    elif case == "head_dim_large":
        q, k, v, o, do = shapes(d=264)  # above 256
    elif case == "gqa_ratio":
        q, k, v, o, do = shapes(hq=3, hk=2)
    elif case == "align":
        q, k, v, o, do = shapes(ptr=(1 << 20) + 8)
    elif case == "stride":
        q = FakeTensor((1, 64, 2, 64), strides=[64 * 2 * 64, 2 * 64 + 4, 64, 1])
    elif case == "null":
        q, k, v, o, do = shapes(ptr=0)
    elif case == "workspace_small":
        kw["ws_bytes"] = 1024
    elif case == "workspace_align":
        kw["ws_ptr"] = (1 << 24) + 64
    if case == "varlen_half":
        from attention_backward_bwd_gb300 import binding as bd
        ds = [bd._desc(t) for t in (q, k, v, o)]
        rc = lib.attn_bwd(*(ctypes.byref(x) for x in ds), 1 << 21, ctypes.byref(bd._desc(do)),
                          ctypes.byref(bd._desc(q)), ctypes.byref(bd._desc(k)),
                          ctypes.byref(bd._desc(v)), 1, 1, 64, 64, 2, 2, 64, 0.125, 0, 1 << 22,
                          None, 64, 64, 0, 1 << 24, 1 << 30, None)
    else:
        rc = call_bwd(lib, q, k, v, o, do, **kw)
    assert rc == code, (rc, lib.attn_last_error())
    assert lib.attn_last_error()  # a message is set


def test_too_many_query_rows_is_a_shape_error(lib):
    # 2^26 query rows x 32 heads: the dQ accumulator's row coordinate would pass 2^31
    q, k, v, o, do = shapes(sq=1 << 26, sk=64, hq=32, hk=8)
    assert call_bwd(lib, q, k, v, o, do) == -2
    assert b"too many query rows" in lib.attn_last_error()


def test_error_message_names_the_problem(lib):
    q, k, v, o, do = shapes(hq=3, hk=2)
    assert call_bwd(lib, q, k, v, o, do) == -2
    assert b"h_k" in lib.attn_last_error()


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from attention_backward_bwd_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        binding.lib()


def test_extended_options_argument_errors(lib):
    """attn_bwd_ex / attn_fwd_ex reject window sides below -1, a negative or
    non-finite softcap and stage masks outside 1..7 before launching anything."""
    from attention_backward_bwd_gb300 import binding as bd
    q, k, v, o, do = shapes()
    ds = [bd._desc(t) for t in (q, k, v, o)]
    d_do, d_dq, d_dk, d_dv = bd._desc(do), bd._desc(q), bd._desc(k), bd._desc(v)

    def bwd(left, right, cap, stages):
        opts = bd.AttnOpts(left, right, cap)
        return lib.attn_bwd_ex(*(ctypes.byref(x) for x in ds), 1 << 21, ctypes.byref(d_do),
                               ctypes.byref(d_dq), ctypes.byref(d_dk), ctypes.byref(d_dv), 1, 1,
                               64, 64, 2, 2, 64, 0.125, 0, None, None, 64, 64, 0,
                               ctypes.byref(opts), stages, 1 << 24, 1 << 30, None)

    assert bwd(-2, 0, 0.0, 7) == -9 and b"window" in lib.attn_last_error()
    assert bwd(3, -5, 0.0, 7) == -9
    assert bwd(3, 0, -1.0, 7) == -9 and b"softcap" in lib.attn_last_error()
    assert bwd(3, 0, float("inf"), 7) == -9
    assert bwd(3, 0, 0.0, 0) == -9 and b"stages" in lib.attn_last_error()
    assert bwd(3, 0, 0.0, 8) == -9
    bad = bd.AttnOpts(-3, 0, 0.0)
    rc = lib.attn_fwd_ex(*(ctypes.byref(x) for x in ds), 1 << 21, 1, 1, 64, 64, 2, 2, 64, 0.125,
                         0, None, None, 64, 64, ctypes.byref(bad), None)
    assert rc == -9 and b"window" in lib.attn_last_error()


def declared_signatures():
    """name -> (return kind, [parameter kinds]) for every function in include/."""
    sigs = {}
    for h in ("attn_bwd.h", "attn_diag.h"):
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for ret, name, params in re.findall(
                r"([A-Za-z_][\w \t]*?\**)\s*\b(attn_[a-z0-9_]+)\s*\(([^()]*)\)\s*;", text):
            params = " ".join(params.split())
            kinds = [] if params in ("", "void") else [_c_kind(p) for p in params.split(",")]
            sigs[name] = (_c_kind(ret.strip() + " r"), kinds)
    return sigs


def _c_kind(decl):
    """Kind of a C declaration 'type name' (name may carry an array suffix)."""
    decl = decl.strip()
    typ = re.sub(r"\s*\b\w+\s*(\[\s*\d*\s*\])?$", "", decl)
    if "*" in typ or "[" in decl or typ.endswith("attn_stream_t"):
        return "ptr"
    for key, kind in (("size_t", "size"), ("int64_t", "i64"), ("float", "float"),
                      ("int", "int"), ("void", "void")):
        if re.search(rf"\b{key}\b", typ):
            return kind
    raise AssertionError(f"unclassified C type in {decl!r}")


def _ctypes_kind(t):
    if t is None:
        return "void"
    if t in (ctypes.c_void_p, ctypes.c_char_p) or issubclass(t, ctypes._Pointer):
        return "ptr"
    for c, kind in ((ctypes.c_size_t, "size"), (ctypes.c_int64, "i64"),
                    (ctypes.c_float, "float"), (ctypes.c_int, "int")):
        if t is c:
            return kind
    raise AssertionError(f"unclassified ctypes type {t}")


def test_binding_signatures_match_the_headers(lib):
    """Every argtypes / restype the binding sets agrees with the header's
    declaration in count and kind (pointer, int, float, size_t, int64_t): a
    drift here would pass wrong values through the ABI without any error."""
    sigs = declared_signatures()
    assert set(sigs) == set(declared_functions())
    for name, (ret, params) in sigs.items():
        f = getattr(lib, name)
        got = [_ctypes_kind(t) for t in f.argtypes]
        assert got == params, f"{name}: binding {got} vs header {params}"
        assert _ctypes_kind(f.restype) == ret, f"{name}: restype vs header {ret}"


def test_struct_layouts_match_the_headers(tmp_path):
    """attn_tensor and attn_opts as a C compiler lays them out (sizes and field
    offsets, from a small program built with gcc against include/attn_bwd.h)
    equal the binding's ctypes structures."""
    import shutil
    import subprocess
    from attention_backward_bwd_gb300 import binding
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = {"attn_tensor": ("ptr", "stride_b", "stride_s", "stride_h"),
              "attn_opts": ("window_left", "window_right", "softcap", "seqused_q", "seqused_k")}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "attn_bwd.h"',
             "int main(void) {"]
    for st, fs in fields.items():
        lines.append(f'  printf("{st} size %zu\\n", sizeof({st}));')
        for f in fs:
            lines.append(f'  printf("{st} {f} %zu\\n", offsetof({st}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    c = {tuple(line.split()[:2]): int(line.split()[2]) for line in out.splitlines()}
    for st, cls in (("attn_tensor", binding.AttnTensor), ("attn_opts", binding.AttnOpts)):
        assert c[(st, "size")] == ctypes.sizeof(cls), st
        for f in fields[st]:
            assert c[(st, f)] == getattr(cls, f).offset, f"{st}.{f}"
        assert [n for n, _ in cls._fields_] == list(fields[st])
