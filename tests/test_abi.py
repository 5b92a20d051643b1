"""The C-ABI library loads and exports every entry point include/pkv.h declares; host-side
argument validation rejects bad calls before any CUDA work (no GPU needed)."""

import ctypes
import os
import re

import pytest

from paged_kv_gqa_14_gb300 import _lib
from paged_kv_gqa_14_gb300 import build as B

HEADER = os.path.join(B.ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return _lib.load()


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^PKV_API\s+[\w\s\*]*?\b(pkv_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["pkv_kv_append", "pkv_paged_attention", "pkv_paged_attention_workspace_size",
                     "pkv_get_device_error", "pkv_status_string"]:
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and the binding knows the signature of each
    assert set(declared_functions()) <= set(_lib.SIGNATURES)


def test_only_declared_symbols_are_exported():
    # -fvisibility=hidden: nothing but the C ABI leaks out of the library
    import subprocess

    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert {e for e in exported if e.startswith("pkv_")} == set(declared_functions())


def test_status_strings(lib):
    for code in range(8):
        assert lib.pkv_status_string(code)
    assert lib.pkv_status_string(99) == b"unknown status"
    assert lib.pkv_version() >= 100


def _append(lib, **kw):
    a = dict(q=16, qs=1024, qh=128, k=16, ks=512, kh=128, v=16, vs=512, vh=128, pos=16, slot=16,
             kc=16, vc=16, T=4, hq=8, hkv=4, d=128, nb=10, bs=16, theta=1e6)
    a.update(kw)
    return lib.pkv_kv_append(a["q"], a["qs"], a["qh"], a["k"], a["ks"], a["kh"], a["v"], a["vs"], a["vh"],
                             a["pos"], a["slot"], a["kc"], a["vc"], a["T"], a["hq"], a["hkv"], a["d"],
                             a["nb"], a["bs"], a["theta"], None)


def test_kv_append_host_validation(lib):
    assert _append(lib, d=96) == 5  # head_dim outside the compiled set
    for bs in (0, -16, 4, 12, 24, 256):  # block_size: a power of two from 8 to 128
        assert _append(lib, bs=bs) == 5
    for bs in (8, 16, 32, 64, 128):
        assert _append(lib, bs=bs, T=0) == 0  # accepted (a no-op: no tokens)
    assert _append(lib, nb=1 << 31) == 2  # block ids are int32
    assert _append(lib, hq=6, hkv=4) == 2  # not a multiple
    assert _append(lib, theta=0.0) == 2
    assert _append(lib, T=-1) == 2
    assert _append(lib, T=0) == 0  # no-op
    assert _append(lib, q=None) == 1
    assert _append(lib, q=8) == 4  # 8-byte aligned pointer
    assert _append(lib, qs=1020) == 3  # rows of consecutive tokens overlap
    assert _append(lib, ks=516) == 4  # stride not a multiple of 8 elements


def _attn(lib, **kw):
    a = dict(q=256, qs=1024, qh=128, kc=256, vc=256, nb=10, bs=16, bt=256, bts=8, mb=8, cl=256, qsl=256,
             B=2, out=512, os=1024, oh=128, T=2, hq=8, hkv=4, d=128, scale=0.1, ws=256, wsb=1 << 20)
    a.update(kw)
    return lib.pkv_paged_attention(a["q"], a["qs"], a["qh"], a["kc"], a["vc"], a["nb"], a["bs"], a["bt"],
                                   a["bts"], a["mb"], a["cl"], a["qsl"], a["B"], a["out"], a["os"], a["oh"],
                                   a["T"], a["hq"], a["hkv"], a["d"], a["scale"], a["ws"], a["wsb"], None)


def test_paged_attention_host_validation(lib):
    assert _attn(lib, d=80) == 5
    for bs in (0, 4, 24, 48, 256):
        assert _attn(lib, bs=bs) == 5
    for bs in (8, 16, 32, 64, 128):
        assert _attn(lib, bs=bs, T=0) == 0
    assert _attn(lib, nb=1 << 31) == 2
    assert _attn(lib, hq=12, hkv=3) == 5  # 8 decode warps must split evenly over kv heads
    assert _attn(lib, hq=36, hkv=4) == 5  # group of 9 > 8
    assert _attn(lib, hq=6, hkv=4) == 2
    assert _attn(lib, T=0) == 0
    assert _attn(lib, B=0) == 0
    assert _attn(lib, q=None) == 1
    assert _attn(lib, bts=4) == 3  # block-table row stride shorter than max_blocks_per_seq
    assert _attn(lib, out=264) == 4  # misaligned out
    assert _attn(lib, os=100) == 3  # overlapping out rows


def test_workspace_size_rejects_bad_sizes(lib):
    assert lib.pkv_paged_attention_workspace_size(-1, 1, 8, 4, 128, 8) == 0
    assert lib.pkv_paged_attention_workspace_size(4, 1, 8, 4, 96, 8) == 0


def test_set_decode_ctas(lib):
    assert lib.pkv_set_decode_ctas(-3) == 2
    assert lib.pkv_set_decode_ctas(0) == 0
    assert lib.pkv_set_kernel_events(9, None, None) == 2
    assert lib.pkv_set_kernel_events(0, None, None) == 0


def test_set_overlap(lib):
    assert lib.pkv_set_overlap(2) == 2
    assert lib.pkv_set_overlap(-1) == 2
    assert lib.pkv_set_overlap(0) == 0
    assert lib.pkv_set_overlap(1) == 0


def test_set_fault_injection(lib):
    # the two test-only faults and "off"; any other kind is refused
    for kind in (3, -1, 100):
        assert lib.pkv_set_fault_injection(kind) == 2  # PKV_ERR_SHAPE
    for kind in (1, 2, 0):
        assert lib.pkv_set_fault_injection(kind) == 0


def test_product_path_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load(str(tmp_path / "missing.so"))


def test_library_has_no_cpu_fallback_symbols():
    # the binding only forwards to the C ABI: no oracle import anywhere in the package
    pkg = os.path.dirname(_lib.__file__)
    for f in os.listdir(pkg):
        if f.endswith(".py") and f != "workloads.py":
            src = open(os.path.join(pkg, f)).read()
            assert "import oracle" not in src and "from oracle" not in src, f


def test_ctypes_signature_count_matches_header():
    assert len(declared_functions()) == len([n for n in _lib.SIGNATURES])
    assert ctypes.sizeof(ctypes.c_size_t) == 8


def test_copy_host_validation(lib):
    assert lib.pkv_copy(None, None, 0, None) == 0  # no-op before any check
    assert lib.pkv_copy(None, 256, 64, None) == 1
    assert lib.pkv_copy(256, None, 64, None) == 1
    assert lib.pkv_copy(264, 256, 64, None) == 4  # dst not 16-byte aligned
    assert lib.pkv_copy(256, 256, 60, None) == 4  # size not a multiple of 16



def _attn_ex_args(x, opt_ptr):
    # a valid-looking call; the option checks come before anything touches the GPU
    return [x, 1024, 128, x, x, 10, 16, x, 8, 8, x, x, 2, x, 1024, 128, 2, 8, 4, 128, ctypes.c_float(0.1),
            x, 1 << 20, None, opt_ptr]


def test_attention_options_are_validated_on_the_host(lib):
    x = ctypes.c_void_p(256)
    opt = _lib.AttentionOptions()
    opt.struct_size = ctypes.sizeof(_lib.AttentionOptions) + 4  # another layout
    assert lib.pkv_paged_attention_ex(*_attn_ex_args(x, ctypes.byref(opt))) == 2  # PKV_ERR_SHAPE
    for field, value in [("decode_kernel", 3), ("prefill_kernel", -1), ("overlap", 3), ("decode_ctas", -1),
                         ("decode_ctas", (1 << 16) + 1), ("flags", 4), ("flags", -1)]:
        opt = _lib.AttentionOptions()
        opt.struct_size = ctypes.sizeof(_lib.AttentionOptions)
        setattr(opt, field, value)
        assert lib.pkv_paged_attention_ex(*_attn_ex_args(x, ctypes.byref(opt))) == 2, field
    opt = _lib.AttentionOptions()
    opt.struct_size = ctypes.sizeof(_lib.AttentionOptions)
    opt.side_stream = 16  # a stream without its fork and join events
    assert lib.pkv_paged_attention_ex(*_attn_ex_args(x, ctypes.byref(opt))) == 1  # PKV_ERR_NULL


def test_workspace_size_ex_rejects_bad_decode_grids(lib):
    assert lib.pkv_paged_attention_workspace_size_ex(4, 4, 8, 4, 128, 8, -1) == 0
    assert lib.pkv_paged_attention_workspace_size_ex(4, 4, 8, 4, 128, 8, (1 << 16) + 1) == 0
    assert lib.pkv_paged_attention_workspace_size_ex(4, 4, 8, 4, 96, 8, 7) == 0
