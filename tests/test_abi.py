"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every
function include/pva.h declares, and rejects host-checkable bad arguments
before touching the device."""
import ctypes
import os
import re

import pytest

from paged_variable_length_gb300 import build, pva

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return pva.load()


def _declared():
    with open(os.path.join(ROOT, "include", "pva.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"PVA_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)))


def test_header_declares_what_the_binding_lists():
    assert _declared() == sorted(pva.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_only_the_abi_is_exported():
    import subprocess

    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True).stdout
    ours = sorted({line.split()[-1] for line in out.splitlines() if " T " in line and "attn_" in line})
    assert ours == _declared()


def test_version_and_status_strings(lib):
    assert pva.abi_version() == 2
    for s in range(7):
        assert pva.status_string(s).startswith(pva.STATUS_NAMES[s])
    assert "unknown" in pva.status_string(99)


def test_structs_match_the_header_layout(tmp_path):
    """Compile a probe against include/pva.h with the host C compiler and compare
    sizes and field offsets with the ctypes mirrors."""
    import subprocess

    fields = [f for f, _ in pva.Config._fields_]
    src = tmp_path / "probe.c"
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"pva.h\"\nint main(void){\n"
                   "printf(\"%zu %zu\\n\", sizeof(pva_config), sizeof(pva_meta));\n"
                   + "".join(f"printf(\"%zu\\n\", offsetof(pva_config, {f}));\n" for f in fields)
                   + "return 0;}\n")
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    vals = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    assert int(vals[0]) == ctypes.sizeof(pva.Config)
    assert int(vals[1]) == ctypes.sizeof(pva.Meta)
    for f, off in zip(fields, vals[2:]):
        assert getattr(pva.Config, f).offset == int(off), f


def _cfg(**kw):
    base = dict(num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16, num_pages=100, max_batch=4,
                max_tokens=16, max_kv_len=1024)
    base.update(kw)
    return pva.make_config(**base)


@pytest.mark.parametrize("bad", [dict(head_dim=96), dict(page_size=24), dict(page_size=256),
                                 dict(num_qo_heads=30), dict(num_qo_heads=64, num_kv_heads=2),
                                 dict(num_kv_heads=12, num_qo_heads=24), dict(num_pages=0),
                                 dict(num_pages=1 << 28)])  # 2^32 slots of 16
def test_unsupported_or_invalid_config_is_rejected_on_the_host(lib, bad):
    cfg = _cfg(**bad)
    assert pva.attn_workspace_size(cfg) == 0
    meta = pva.Meta()
    dummy = ctypes.c_void_p(256)
    st = lib.attn_prepare_metadata(ctypes.byref(cfg), dummy, dummy, dummy, 8, None, 1, 1, 1, dummy, 1 << 20, None,
                                   ctypes.byref(meta))
    assert st in (1, 2)


def test_null_pointers_are_rejected_on_the_host(lib):
    cfg = _cfg()
    meta = pva.Meta()
    dummy = ctypes.c_void_p(256)
    for args in [(None, dummy, dummy), (dummy, None, dummy), (dummy, dummy, None)]:
        st = lib.attn_prepare_metadata(ctypes.byref(cfg), *args, 8, None, 1, 1, 1, dummy, 1 << 20, None,
                                       ctypes.byref(meta))
        assert st == 1
    st = lib.attn_prepare_metadata(ctypes.byref(cfg), dummy, dummy, dummy, 8, None, 1, 1, 1, dummy, 1 << 20, None,
                                   None)
    assert st == 1


def test_empty_batch_needs_no_lengths_or_page_table(lib):
    """batch 0 reads neither array: NULL passes the argument checks and the call stops at the
    next one (a 16-byte workspace is too small: nothing is launched, with or without a
    device), while new tokens claimed for an empty batch are refused."""
    cfg = _cfg()
    meta = pva.Meta()
    dummy = ctypes.c_void_p(256)
    st = lib.attn_prepare_metadata(ctypes.byref(cfg), dummy, None, None, 0, None, 0, 0, 0, dummy, 16, None,
                                   ctypes.byref(meta))
    assert st in (3, 4)  # PVA_ERR_WORKSPACE_TOO_SMALL, or PVA_ERR_CUDA without a device
    st = lib.attn_prepare_metadata(ctypes.byref(cfg), dummy, None, None, 0, None, 0, 3, 0, dummy, 16, None,
                                   ctypes.byref(meta))
    assert st == 1


def test_misaligned_workspace_and_oversized_batch_are_rejected(lib):
    cfg = _cfg()
    meta = pva.Meta()
    dummy = ctypes.c_void_p(256)
    st = lib.attn_prepare_metadata(ctypes.byref(cfg), dummy, dummy, dummy, 8, None, 1, 1, 1, ctypes.c_void_p(264),
                                   1 << 20, None, ctypes.byref(meta))
    assert st == 1
    st = lib.attn_prepare_metadata(ctypes.byref(cfg), dummy, dummy, dummy, 8, None, 5, 1, 1, dummy, 1 << 20, None,
                                   ctypes.byref(meta))
    assert st == 1


def test_forward_requires_a_prepared_meta(lib):
    meta = pva.Meta()
    dummy = ctypes.c_void_p(256)
    assert lib.attn_forward(ctypes.byref(meta), dummy, dummy, dummy, dummy, dummy, dummy, None, None) == 6
    assert lib.attn_store_kvcache(ctypes.byref(meta), dummy, dummy, dummy, dummy, None) == 6
    assert lib.attn_forward(None, dummy, dummy, dummy, dummy, dummy, dummy, None, None) == 6

