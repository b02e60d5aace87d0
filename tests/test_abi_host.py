"""Host-side checks of the C ABI that need no GPU.

The library must build (or be built), load, and export every function that
include/sdpa.h declares.  Argument validation happens on the host before any
launch, so invalid calls are exercised here with pointers that are never
dereferenced: every call below is rejected by a check, none reaches a kernel.
"""
import ctypes
import os
import re

import pytest

import scaled_dot_product_sm_gb300 as sdpa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdpa.h")


@pytest.fixture(scope="module")
def lib():
    sdpa.build()
    return sdpa.load_library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(sdpa_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_exported_list():
    assert header_functions() == sorted(sdpa.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    assert sdpa.exported_symbols() == list(sdpa.EXPORTS)
    for name in header_functions():
        assert hasattr(lib, name)


def test_status_strings(lib):
    for code in range(5):
        s = lib.sdpa_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert lib.sdpa_status_string(99) == b"unknown status"


def _shape(B=1, Hq=2, Hkv=2, L=8, S=8, E=64, Ev=64, dtype=1, mb=1, mh=1):
    return sdpa.Shape(B, Hq, Hkv, L, S, E, Ev, dtype, mb, mh)


FAKE = 1 << 20           # 16-byte aligned; never dereferenced (every call below fails validation)
P = ctypes.c_void_p


def _fwd(lib, shp, q=FAKE, k=FAKE, v=FAKE, mask=None, scale=float("nan"), causal=0, gqa=0, o=FAKE, lse=FAKE):
    return lib.sdpa_forward(ctypes.byref(shp), P(q), P(k), P(v), P(mask), scale, causal, gqa, P(o), P(lse),
                            None, 0, None)


def _bwd(lib, shp, ws=FAKE, wsb=0, scale=float("nan"), gqa=0, dq=FAKE):
    return lib.sdpa_backward(ctypes.byref(shp), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None,
                             scale, 0, gqa, P(dq), P(FAKE), P(FAKE), P(ws), wsb, None)


INVALID, UNSUPPORTED = 1, 2


@pytest.mark.parametrize("kw", [dict(B=0), dict(L=0), dict(S=-1), dict(E=0), dict(Ev=0), dict(dtype=7),
                                dict(Hq=3, Hkv=2)])
def test_forward_rejects_bad_shapes(lib, kw):
    assert _fwd(lib, _shape(**kw), gqa=1) == INVALID


def test_forward_rejects_gqa_without_flag(lib):
    assert _fwd(lib, _shape(Hq=4, Hkv=2), gqa=0) == INVALID


def test_forward_rejects_bad_mask_dims(lib):
    assert _fwd(lib, _shape(B=2, mb=3), mask=FAKE) == INVALID
    assert _fwd(lib, _shape(Hq=2, mh=4), mask=FAKE) == INVALID


@pytest.mark.parametrize("scale", [-1.0, float("inf"), float("-inf")])
def test_forward_rejects_bad_scale(lib, scale):
    assert _fwd(lib, _shape(), scale=scale) == INVALID


def test_forward_rejects_null_and_misaligned(lib):
    assert _fwd(lib, _shape(), q=0) == INVALID
    assert _fwd(lib, _shape(), lse=0) == INVALID
    assert _fwd(lib, _shape(), k=FAKE + 4) == INVALID
    assert _fwd(lib, _shape(), mask=FAKE + 8) == INVALID


def test_forward_rejects_unsupported_sizes(lib):
    assert _fwd(lib, _shape(E=256, Ev=256)) == UNSUPPORTED
    assert _fwd(lib, _shape(E=60)) == UNSUPPORTED          # bf16 widths must be multiples of 8
    # extents past the kernels' 32-bit counters, including ones whose products would overflow int64
    assert _fwd(lib, _shape(B=1 << 40)) == UNSUPPORTED
    assert _fwd(lib, _shape(B=1 << 62, Hq=1 << 62, Hkv=1 << 62)) == UNSUPPORTED
    assert _fwd(lib, _shape(L=1 << 31)) == UNSUPPORTED
    # tensors of 2^56 elements or more: q of 2^59 rows, then a mask of 2^64 elements
    assert _fwd(lib, _shape(B=1 << 20, Hq=1 << 10, Hkv=1, L=1 << 29), gqa=1) == UNSUPPORTED
    big = (1 << 30) - 1
    assert _fwd(lib, _shape(B=4, Hq=4, Hkv=4, L=big, S=big, mb=4, mh=4), mask=FAKE) == UNSUPPORTED


def test_backward_rejects_small_workspace(lib):
    shp = _shape()
    need = lib.sdpa_backward_workspace_bytes(ctypes.byref(shp))
    assert need >= 2 * 8 * 4
    assert _bwd(lib, shp, ws=FAKE, wsb=need - 1) == INVALID
    assert _bwd(lib, shp, ws=0, wsb=need) == INVALID
    assert _bwd(lib, shp, ws=FAKE, wsb=need, dq=0) == INVALID
    assert _bwd(lib, shp, ws=FAKE, wsb=need, scale=-2.0) == INVALID


def test_decode_workspace_and_splits(lib):
    shp = _shape(B=16, Hq=32, Hkv=8, L=1, S=32768, E=128, Ev=128)
    n = lib.sdpa_decode_num_splits(ctypes.byref(shp))
    assert 1 <= n <= 32768 // 64
    for splits in (1, 2, 7):
        ws = lib.sdpa_decode_workspace_bytes(ctypes.byref(shp), splits)
        rows = 16 * 32
        assert ws >= rows * splits * (128 + 1) * 4
    assert lib.sdpa_forward_workspace_bytes(ctypes.byref(shp)) == lib.sdpa_decode_workspace_bytes(
        ctypes.byref(shp), 0)
    # bf16 prefill on the tensor cores: a unit counter (used by padded calls); fp32 and other widths: none
    assert lib.sdpa_forward_workspace_bytes(ctypes.byref(_shape(L=64))) == 256
    assert lib.sdpa_forward_workspace_bytes(ctypes.byref(_shape(L=64, dtype=0))) == 0
    assert lib.sdpa_forward_workspace_bytes(ctypes.byref(_shape(L=64, E=32, Ev=32))) == 0
    # decode rejects a negative split count and a too-small workspace before launching
    st = lib.sdpa_decode(ctypes.byref(shp), P(FAKE), P(FAKE), P(FAKE), None, float("nan"), 1, -1, P(FAKE),
                         P(FAKE), P(FAKE), 1 << 30, None)
    assert st == INVALID
    st = lib.sdpa_decode(ctypes.byref(shp), P(FAKE), P(FAKE), P(FAKE), None, float("nan"), 1, 4, P(FAKE),
                         P(FAKE), P(FAKE), 16, None)
    assert st == INVALID


def test_backward_workspace_size_formula(lib):
    shp = _shape(B=2, Hq=4, Hkv=2, L=100, S=50, E=64, Ev=64, dtype=0)
    # fp32: D only, rounded to 256 bytes
    assert lib.sdpa_backward_workspace_bytes(ctypes.byref(shp)) == (2 * 4 * 100 * 4 + 255) // 256 * 256


def test_binding_requires_cuda_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 4, 8)
    with pytest.raises(ValueError):
        sdpa.sdpa_forward(q, q, q)


def _fwd_opts(lib, shp, opts):
    return lib.sdpa_forward_opts(ctypes.byref(shp), opts, P(FAKE), P(FAKE), P(FAKE), None, float("nan"), 0,
                                 P(FAKE), P(FAKE), None, 0, None)


def test_opts_entry_points_reject_bad_options(lib):
    shp = _shape()
    # options are required by the *_opts calls
    assert _fwd_opts(lib, shp, None) == INVALID
    assert lib.sdpa_backward_opts(ctypes.byref(shp), None, P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                  None, float("nan"), 0, P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1 << 20,
                                  None) == INVALID
    dshp = _shape(L=1)
    assert lib.sdpa_decode_opts(ctypes.byref(dshp), None, P(FAKE), P(FAKE), P(FAKE), None, float("nan"), 0, 0,
                                P(FAKE), P(FAKE), P(FAKE), 1 << 30, None) == INVALID
    # an alignment other than top-left / bottom-right, and misaligned length arrays
    bad_align = sdpa.Options(None, None, 2, -1, 0)
    assert _fwd_opts(lib, shp, ctypes.byref(bad_align)) == INVALID
    mis_q = sdpa.Options(FAKE + 2, None, 0, 0, 0)
    assert _fwd_opts(lib, shp, ctypes.byref(mis_q)) == INVALID
    mis_kv = sdpa.Options(None, FAKE + 1, 1, 0, 4)
    assert _fwd_opts(lib, shp, ctypes.byref(mis_kv)) == INVALID
    # shape errors still come first
    ok = sdpa.Options(None, None, 1, 0, 16)
    assert _fwd_opts(lib, _shape(B=0), ctypes.byref(ok)) == INVALID


def test_binding_band_options():
    b = sdpa.Band(alignment="bottom_right", right_bound=0, left_bound=128)
    o = b.options()
    assert (o.seq_len_q, o.seq_len_kv, o.diagonal_alignment, o.right_bound, o.left_bound) == (None, None, 1, 0, 128)
    o = sdpa.Band().options()
    assert (o.diagonal_alignment, o.right_bound, o.left_bound) == (0, -1, 0)
    with pytest.raises(ValueError):
        sdpa.Band(alignment="center").options()
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):   # lengths must be CUDA int32
        sdpa.Band(seq_len_q=torch.zeros(2, dtype=torch.int32)).options()


def test_decode_paged_rejects_bad_tables(lib):
    shp = _shape(B=2, Hq=4, Hkv=2, L=1, S=100, E=64, Ev=64)

    def call(pg):
        return lib.sdpa_decode_paged(ctypes.byref(shp), None, pg, P(FAKE), P(FAKE), P(FAKE), None, float("nan"), 1,
                                     0, P(FAKE), P(FAKE), P(FAKE), 1 << 30, None)
    assert call(None) == INVALID
    good = dict(page_table_k=FAKE, page_table_v=FAKE, block_size_k=16, block_size_v=16, max_blocks=7,
                num_blocks_k=20, num_blocks_v=20)
    for bad in (dict(block_size_k=12), dict(block_size_v=4), dict(max_blocks=6), dict(page_table_k=FAKE + 2),
                dict(page_table_v=None), dict(num_blocks_k=0), dict(num_blocks_v=1 << 62)):
        pg = sdpa.PagedKV(**{**good, **bad})
        assert call(ctypes.byref(pg)) == INVALID, bad


def test_dropout_options_are_checked(lib):
    shp = _shape()
    for p in (-0.1, 1.0, float("nan")):
        o = sdpa.Options(None, None, 0, 0, 0, p, 1, 0)
        assert _fwd_opts(lib, shp, ctypes.byref(o)) == INVALID, p
    o = sdpa.Options(None, None, 0, 0, 0, 0.1, 1, 1 << 32)   # the offset fills one 32-bit counter word
    assert _fwd_opts(lib, shp, ctypes.byref(o)) == INVALID
    dshp = _shape(L=1)
    o = sdpa.Options(None, None, 1, 0, 0, 0.1, 1, 0)   # the decode takes no dropout
    assert lib.sdpa_decode_opts(ctypes.byref(dshp), ctypes.byref(o), P(FAKE), P(FAKE), P(FAKE), None, float("nan"), 0,
                                0, P(FAKE), P(FAKE), P(FAKE), 1 << 30, None) == INVALID


def test_binding_checks_tensor_shapes_before_launching():
    """The C ABI sees one shape; every tensor that disagrees with it is refused by the binding
    (ValueError) before the library is loaded, so no kernel can run past a buffer."""
    torch = pytest.importorskip("torch")
    bf, f32 = torch.bfloat16, torch.float32
    B, Hq, Hkv, L, S, E = 2, 4, 2, 8, 24, 16

    def t(*shape, dtype=bf):
        return torch.zeros(*shape, dtype=dtype)
    q, k, v = t(B, Hq, L, E), t(B, Hkv, S, E), t(B, Hkv, S, E)
    o, dO, lse = t(B, Hq, L, E), t(B, Hq, L, E), t(B, Hq, L, dtype=f32)
    bad_forward = [
        dict(k=t(B, Hkv, S, E + 16)),            # K width differs from Q's
        dict(v=t(B, Hkv, S + 1, E)),             # V length differs from K's
        dict(v=t(B, Hkv + 1, S, E)),
        dict(k=t(B, Hkv, S, E, dtype=f32)),      # mixed dtypes
        dict(mask=t(1, 1, L, S + 4, dtype=f32)),  # mask wider than S
        dict(mask=t(1, 1, L - 1, S, dtype=f32)),
        dict(mask=t(1, 1, L, S)),                # mask not fp32
        dict(out=t(B, Hq, L + 1, E)),
        dict(out=t(B, Hq, L, E, dtype=f32)),
        dict(lse=t(B, Hq, L)),                   # lse not fp32
        dict(lse=t(B, Hq, L + 1, dtype=f32)),
    ]
    for bad in bad_forward:
        args = dict(q=q, k=k, v=v, mask=None, out=None, lse=None)
        args.update(bad)
        with pytest.raises(ValueError, match="must have shape|must be torch"):
            sdpa.sdpa_forward(args["q"], args["k"], args["v"], args["mask"], out=args["out"], lse=args["lse"],
                              enable_gqa=True)
    for name, bad in (("o", t(B, Hq, L, E + 16)), ("dO", t(B, Hq, L - 1, E)), ("lse", t(B, Hq, L)),
                      ("dq", t(B, Hq, L, E, dtype=f32)), ("dk", t(B, Hq, S, E)), ("dv", t(B, Hkv, S - 1, E))):
        args = dict(o=o, dO=dO, lse=lse, dq=None, dk=None, dv=None)
        args[name] = bad
        with pytest.raises(ValueError, match="must have shape|must be torch"):
            sdpa.sdpa_backward(q, k, v, args["o"], args["dO"], args["lse"], enable_gqa=True, dq=args["dq"],
                               dk=args["dk"], dv=args["dv"])
    qd = t(B, Hq, 1, E)
    with pytest.raises(ValueError, match="must have shape"):
        sdpa.sdpa_decode(qd, k, t(B, Hkv, S - 8, E), enable_gqa=True)
    # consistent shapes get as far as the device check (host tensors are refused, never passed on)
    with pytest.raises(ValueError, match="CUDA device"):
        sdpa.sdpa_forward(q, k, v, t(1, 1, L, S, dtype=f32), enable_gqa=True)
    with pytest.raises(ValueError, match="CUDA device"):
        sdpa.sdpa_backward(q, k, v, o, dO, lse, enable_gqa=True)


def test_binding_checks_paged_and_band_shapes():
    torch = pytest.importorskip("torch")
    bf = torch.bfloat16
    B, Hq, Hkv, E, bs = 2, 4, 2, 16, 16
    q = torch.zeros(B, Hq, 1, E, dtype=bf)
    kc, vc = torch.zeros(10, Hkv, bs, E, dtype=bf), torch.zeros(10, Hkv, bs, E, dtype=bf)
    pt = torch.zeros(B, 4, dtype=torch.int32)
    with pytest.raises(ValueError, match="must have shape"):
        sdpa.sdpa_decode_paged(q, torch.zeros(10, Hkv, bs, E + 16, dtype=bf), vc, pt, pt, 64, enable_gqa=True)
    with pytest.raises(ValueError, match="must have shape"):
        sdpa.sdpa_decode_paged(q, kc, torch.zeros(10, Hkv + 1, bs, E, dtype=bf), pt, pt, 64, enable_gqa=True)
    with pytest.raises(ValueError, match="page tables"):
        sdpa.sdpa_decode_paged(q, kc, vc, torch.zeros(B + 1, 4, dtype=torch.int32), pt, 64, enable_gqa=True)
    with pytest.raises(ValueError, match="must have shape"):
        sdpa.sdpa_decode_paged(q, kc, vc, pt, pt, 64, mask=torch.zeros(1, 1, 1, 63), enable_gqa=True)
    with pytest.raises(ValueError, match="CUDA device"):
        sdpa.sdpa_decode_paged(q, kc, vc, pt, pt, 64, enable_gqa=True)
    # padding lengths: exactly B of them
    with pytest.raises(ValueError, match="B = 2 lengths"):
        sdpa.Band(seq_len_kv=torch.zeros(3, dtype=torch.int32)).options(batch=2)
    with pytest.raises(ValueError, match="B = 2 lengths"):
        sdpa.Band(seq_len_q=torch.zeros(1, 2, dtype=torch.int32)).options(batch=2)


def test_library_and_oracle_share_nothing():
    """The product path (package, kernels, header) never names or imports the oracle, and the
    oracle never imports the package: the two sides of every parity check are independent."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = os.path.join(root, "scaled_dot_product_sm_gb300")
    product = [os.path.join(dp, f) for dp, _, fs in os.walk(pkg) for f in fs
               if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp"))]
    product += [os.path.join(root, "include", f) for f in os.listdir(os.path.join(root, "include"))]
    assert len(product) > 5
    for path in product:
        with open(path, encoding="utf-8") as fh:
            assert not re.search(r"\boracle\b", fh.read()), path
    odir = os.path.join(root, "oracle")
    for f in os.listdir(odir):
        if f.endswith(".py"):
            with open(os.path.join(odir, f), encoding="utf-8") as fh:
                src = fh.read()
            assert "scaled_dot_product_sm_gb300" not in src and "workloads" not in src, f


def test_header_is_plain_c_and_links(tmp_path):
    """include/sdpa.h compiles as strict C11, every declared entry point links against the
    library, and a C caller gets INVALID_ARG back from calls without a shape (nothing reaches
    the GPU)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    sdpa.build()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    libdir = os.path.dirname(sdpa.LIB_PATH)
    names = sdpa.EXPORTS
    src = tmp_path / "caller.c"
    src.write_text("\n".join([
        '#include "sdpa.h"',
        "#include <stdio.h>",
        "typedef void (*any_fn)(void);",
        "static const any_fn entry_points[] = {" + ", ".join(f"(any_fn){n}" for n in names) + "};",
        "int main(void) {",
        "  if (sizeof(entry_points) / sizeof(entry_points[0]) != %d) return 2;" % len(names),
        "  if (sdpa_forward(NULL, NULL, NULL, NULL, NULL, 0.0, 0, 0, NULL, NULL, NULL, 0, NULL)"
        " != SDPA_ERR_INVALID_ARG) return 3;",
        "  if (sdpa_backward(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0.0, 0, 0, NULL, NULL, NULL,"
        " NULL, 0, NULL) != SDPA_ERR_INVALID_ARG) return 4;",
        "  if (sdpa_decode(NULL, NULL, NULL, NULL, NULL, 0.0, 0, 0, NULL, NULL, NULL, 0, NULL)"
        " != SDPA_ERR_INVALID_ARG) return 5;",
        '  printf("%s\\n", sdpa_status_string(SDPA_ERR_INVALID_ARG));',
        "  return 0;",
        "}",
    ]) + "\n")
    exe = tmp_path / "caller"
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                        os.path.join(root, "include"), str(src), "-o", str(exe), "-L", libdir, "-lsdpa_gb300",
                        f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, (run.returncode, run.stderr)
    assert run.stdout.strip() == lib_status_string(1)


def lib_status_string(code):
    return sdpa.load_library().sdpa_status_string(code).decode()
