"""The C ABI without a GPU: libpf.so builds for sm_103a, loads, exports every function that
include/pf.h declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pf.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_decode_pf_gb300 import _build
    _build.build()
    import paged_kv_decode_pf_gb300 as pf
    return pf.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^PF_API\s+[\w\s\*]+?\b(pf_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_abi():
    names = set(declared_functions())
    assert {"pf_reshape_and_cache", "pf_paged_attention_decode", "pf_paged_attention_decode_partition",
            "pf_paged_attention_merge", "pf_paged_attention_partition_workspace_size",
            "pf_get_device_error", "pf_status_string"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_only_declared_symbols_are_exported(lib):
    import subprocess
    from paged_kv_decode_pf_gb300 import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert {n for n in exported if n.startswith("pf_")} == set(declared_functions())


def test_status_strings_and_version(lib):
    import paged_kv_decode_pf_gb300 as pf
    for code, name in pf.STATUS_NAMES.items():
        assert lib.pf_status_string(code).decode() == name
    assert re.fullmatch(r"\d+\.\d+\.\d+", pf.version())


def test_workspace_layout_arithmetic(lib):
    import paged_kv_decode_pf_gb300 as pf
    r = lambda x: (x + 255) // 256 * 256
    for S, Hq, D, mx, P in [(4, 32, 128, 131072, 512), (1, 1, 64, 1, 16), (3, 8, 64, 0, 32), (7, 5, 128, 1000, 48)]:
        NP = max(1, -(-mx // P))
        total, oo, om, ol = pf.partition_workspace_layout(S, Hq, D, mx, P)
        assert (oo, om, ol) == (0, r(S * Hq * NP * D * 4), r(S * Hq * NP * D * 4) + r(S * Hq * NP * 4))
        assert total == ol + r(S * Hq * NP * 4)
        assert lib.pf_paged_attention_partition_workspace_size(S, Hq, D, mx, P) == total
    for bad in [(0, 1, 64, 10, 16), (1, 0, 64, 10, 16), (1, 1, 64, -1, 16), (1, 1, 64, 10, 0)]:
        assert pf.partition_workspace_layout(*bad)[0] == 0


def _decode(lib, fn=None, **kw):
    a = dict(q=0x10000, kc=0x20000, vc=0x30000, bt=0x40000, cl=0x50000, S=2, Hq=8, Hkv=2, D=128, bs=16, MB=4,
             NB=64, scale=0.125, out=0x60000)
    a.update(kw)
    fn = lib.pf_paged_attention_decode if fn is None else fn
    return fn(a["q"], a["kc"], a["vc"], a["bt"], a["cl"], a["S"], a["Hq"], a["Hkv"], a["D"], a["bs"], a["MB"],
              a["NB"], a["scale"], a["out"], None)


DECODE_CHECKS = [
    (dict(S=-1), 1), (dict(Hq=0), 1), (dict(Hkv=0), 1), (dict(Hq=6, Hkv=4), 1), (dict(D=0), 1),
    (dict(bs=0), 1), (dict(MB=0), 1), (dict(NB=0), 1), (dict(NB=2 ** 31), 1), (dict(scale=float("inf")), 1),
    (dict(q=None), 1), (dict(q=0x10002), 1), (dict(bt=0x40002), 1), (dict(out=0x60004), 1),
    (dict(D=96), 2), (dict(D=256), 2), (dict(bs=8), 2), (dict(bs=24), 2), (dict(Hq=32, Hkv=2), 2),
    (dict(Hq=6, Hkv=2), 2),
]


@pytest.mark.parametrize("change,want", DECODE_CHECKS)
def test_decode_host_validation(lib, change, want):
    assert _decode(lib, **change) == want


@pytest.mark.parametrize("change,want", DECODE_CHECKS + [(dict(out=None), 1), (dict(out=0x60002), 1)])
def test_decode_bf16_host_validation(lib, change, want):
    """The bf16-output entry checks its arguments as the fp32 one does (its output 16-byte aligned)."""
    assert _decode(lib, fn=lib.pf_paged_attention_decode_bf16, **change) == want
    assert _decode(lib, fn=lib.pf_paged_attention_decode_bf16, S=0, q=None, kc=None, vc=None, bt=None, cl=None,
                   out=None) == 0


def test_zero_sequences_is_a_no_op(lib):
    assert _decode(lib, S=0, q=None, kc=None, vc=None, bt=None, cl=None, out=None) == 0


def test_partition_and_merge_host_validation(lib):
    P = ctypes.c_void_p
    args = [0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 2, 8, 2, 128, 16, 4, 64, ctypes.c_float(0.1)]
    f = lib.pf_paged_attention_decode_partition
    assert f(*args, 0, 64, P(0x70000), 1 << 20, None) == 1          # partition size 0
    assert f(*args, 24, 64, P(0x70000), 1 << 20, None) == 2         # not a multiple of 16
    assert f(*args, 32, -1, P(0x70000), 1 << 20, None) == 1         # negative max length
    assert f(*args, 32, 64, P(0x70000), 16, None) == 1              # workspace too small
    assert f(*args, 32, 64, P(0x70010), 1 << 20, None) == 1         # workspace misaligned
    m = lib.pf_paged_attention_merge
    assert m(P(0x70000), P(0x50000), 2, 8, 96, 32, 64, P(0x60000), None) == 2
    assert m(P(0x70000), P(0x50000), 2, 8, 128, 0, 64, P(0x60000), None) == 1
    assert m(P(0x70010), P(0x50000), 2, 8, 128, 32, 64, P(0x60000), None) == 1
    assert m(None, None, 0, 8, 128, 32, 64, None, None) == 0


def test_append_host_validation(lib):
    f = lib.pf_reshape_and_cache
    ok = [0x10000, 0x20000, 0x30000, 0x40000, 0x50000]
    assert f(*ok, -1, 2, 64, 16, 10, None) == 1
    assert f(*ok, 4, 2, 60, 16, 10, None) == 2                      # head_dim not a multiple of 8
    assert f(*ok, 4, 2, 64, 0, 10, None) == 1
    assert f(0x10008, *ok[1:], 4, 2, 64, 16, 10, None) == 1         # misaligned k
    assert f(*ok[:2], 0x30004, *ok[3:], 4, 2, 64, 16, 10, None) == 1  # misaligned slot_mapping
    assert f(None, None, None, None, None, 0, 2, 64, 16, 10, None) == 0


def test_debug_wait_limits(lib):
    assert lib.pf_debug_bounded_wait(10, None) == 1
    assert lib.pf_debug_bounded_wait(10 ** 11, None) == 1


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    import paged_kv_decode_pf_gb300 as pf
    monkeypatch.setattr(pf, "_LIB", None)
    monkeypatch.setattr(pf, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        pf.lib()


def test_multi_query_host_validation(lib):
    """Both multi-token entry points check their shapes on the host: more than 65 536 query rows per
    kv head, a head_dim outside {64, 128} or a block size not a multiple of 16 launch nothing; the
    tcgen05 form takes head_dim 128 only; no sequence is a no-op (also past 64 rows per kv head,
    where the prompt-chunk kernel would run)."""
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    for name in ("pf_paged_attention_multi_query", "pf_paged_attention_multi_query_tcgen05"):
        f = getattr(lib, name)
        f.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i64, f32, P, P]
        f.restype = ctypes.c_int
        # q, k, v, tables, lengths, S, q_len, Hq, Hkv, D, bs, max_blocks, num_blocks, scale, out, stream
        args = [None] * 5 + [0, 4, 32, 8, 128, 16, 8, 64, 0.088, None, None]
        assert f(*args) == 0                                          # no sequence: nothing to do
        assert f(*(args[:6] + [17] + args[7:])) == 0                  # 4 x 17 = 68 rows: prompt chunk, no sequence
        assert f(*(args[:6] + [16384] + args[7:])) == 0               # 65 536 rows: the limit
        assert f(*(args[:6] + [16385] + args[7:])) == 2               # 65 540 rows per kv head
        assert f(*(args[:9] + [96] + args[10:])) == 2                 # head_dim 96
        assert f(*(args[:10] + [24] + args[11:])) == 2                # block size not a multiple of 16
        assert f(*(args[:6] + [0] + args[7:])) == 1                   # q_len 0
        assert f(*(args[:7] + [30] + args[8:])) == 1                  # Hq not a multiple of Hkv
    assert lib.pf_paged_attention_multi_query(*(args[:9] + [64] + args[10:])) == 0
    assert lib.pf_paged_attention_multi_query_tcgen05(*(args[:9] + [64] + args[10:])) == 2


def test_multi_query_kernel_selector():
    import torch
    import paged_kv_decode_pf_gb300 as pf
    t = torch.zeros(1)
    with pytest.raises(ValueError, match="unknown kernel"):
        pf.paged_attention_multi_query(t, t, t, t, t, kernel="mma")
