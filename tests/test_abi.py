"""The C-ABI library: it loads, exports every symbol include/gbattn.h declares, and its
host-side validation returns the documented status codes (no GPU needed: every case here
is rejected before anything touches the device)."""
import ctypes
import os
import re

import pytest

import streaming_attention_flashattention_gb300 as gb
from streaming_attention_flashattention_gb300 import build as gbbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbattn.h")


@pytest.fixture(scope="module")
def lib():
    gbbuild.build()
    return gb.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_]\w*\s*\*?\s*(attn_\w+)\s*\(", text, re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["attn_fwd", "attn_decode_splitkv", "attn_decode_workspace_size",
              "attn_last_device_error", "attn_status_string", "attn_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"libgbattn.so does not export {n}"
        assert n in gb.EXPORTS, f"binding does not describe {n}"


def test_version_and_status_strings(lib):
    assert gb.attn_version() >= 100
    assert gb.attn_status_string(0) == "ok"
    for code in range(-7, 0):
        s = gb.attn_status_string(code)
        assert s and s != "unknown status"
    assert gb.attn_status_string(-99) == "unknown status"


A = 0x10000      # fake, 16-byte-aligned addresses: every call below is rejected first
B_ = 0x20000
MIS = 0x10008    # 8-byte aligned only


def fwd(lib, q=A, k=A, v=A, o=B_, lse=None, B=1, Hq=2, Hkv=1, Sq=128, Skv=128, d=128,
        scale=0.1, causal=0, dtype=0):
    return lib.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, d, scale, causal, dtype, None)


def test_fwd_argument_validation(lib):
    assert fwd(lib, q=None) == -1
    assert fwd(lib, o=None) == -1
    assert fwd(lib, B=0) == -1
    assert fwd(lib, Sq=0) == -1
    assert fwd(lib, Skv=-3) == -1
    assert fwd(lib, Hq=3, Hkv=2) == -1
    assert fwd(lib, scale=0.0) == -1
    assert fwd(lib, scale=float("nan")) == -1
    assert fwd(lib, causal=2) == -1
    assert fwd(lib, dtype=5) == -1
    assert fwd(lib, d=96) == -2
    assert fwd(lib, d=256) == -2
    assert fwd(lib, causal=1, Sq=200, Skv=100) == -2
    assert fwd(lib, q=MIS) == -3
    assert fwd(lib, lse=MIS) == -3
    assert fwd(lib, B=70000, Hq=70000, Hkv=70000) == -7


def dec(lib, q=A, kc=A, vc=A, lens=A, o=B_, lse=None, B=4, Hq=64, Hkv=8, Lmax=32768, d=128,
        scale=0.1, ns=16, ws=A, wsb=None):
    if wsb is None:
        wsb = lib.attn_decode_workspace_size(B, Hq, Hkv, Lmax, d, ns)
    return lib.attn_decode_splitkv(q, kc, vc, lens, o, lse, B, Hq, Hkv, Lmax, d, scale, ns, ws,
                                   wsb, None)


def test_decode_argument_validation(lib):
    assert dec(lib, kc=None) == -1
    assert dec(lib, lens=None) == -1
    assert dec(lib, B=0) == -1
    assert dec(lib, Hq=63) == -1
    assert dec(lib, ns=-1) == -1
    assert dec(lib, ns=257) == -1
    assert dec(lib, d=80) == -2
    assert dec(lib, q=MIS) == -3
    assert dec(lib, lens=0x10002) == -3
    # the workspace check sizes for the current device's SM count: without a device the
    # call stops there with GBATTN_ERR_CUDA, with one it rejects the missing or short
    # workspace -- before anything is launched either way
    import torch
    want = -6 if torch.cuda.is_available() else -4
    assert dec(lib, ws=None, wsb=0) == want
    assert dec(lib, wsb=16) == want


def test_counted_prefill_argument_checks(lib):
    f = lib.attn_fwd_counted
    cnt = 0x30000
    assert f(A, A, A, B_, None, 1, 2, 1, 128, 128, 128, 0.1, 1, None, None) == -1   # no counter
    assert f(A, A, A, B_, None, 1, 2, 1, 128, 128, 128, 0.1, 1, 0x30002, None) == -3  # misaligned
    assert f(None, A, A, B_, None, 1, 2, 1, 128, 128, 128, 0.1, 1, cnt, None) == -1
    assert f(A, A, A, B_, None, 1, 2, 1, 128, 128, 96, 0.1, 1, cnt, None) == -2     # d
    assert f(A, A, A, B_, None, 1, 2, 1, 256, 128, 128, 0.1, 1, cnt, None) == -2   # causal Sq > Skv
    assert f(A, A, A, B_, None, 1, 3, 2, 128, 128, 128, 0.1, 0, cnt, None) == -1    # Hq % Hkv


def test_workspace_size(lib):
    def ws(B, Hq, Hkv, L, d, ns, nsm=152):
        return gb.attn_decode_workspace_bytes(B, Hq, Hkv, 1, L, d, ns, nsm)

    def expect(B, Hq, Hkv, slots, d):
        # counters (the work queue, then one partial counter per (b, KV head, chunk group);
        # G <= 8 gives one group) rounded to 256, lse partials rounded to 256, O partials
        rows = B * Hq * slots
        counters = ((1 + B * Hkv) * 4 + 255) // 256 * 256
        return counters + ((rows * 4 + 255) // 256) * 256 + rows * d * 4

    # 16 fixed splits x 32 (sequence, KV head) groups = 512 items, 3.37 waves on 152 SMs:
    # each split runs as 2 pieces, so 32 partials per row
    assert ws(4, 64, 8, 32768, 128, 16) == expect(4, 64, 8, 32, 128)
    # automatic: one slot per 4096 keys of capacity ...
    assert ws(16, 64, 8, 131072, 128, 0) == expect(16, 64, 8, 32, 128)
    # ... raised for few (sequence, KV head) groups to the most splits that keep one wave of
    # 152 work items: 8 groups take 152 // 8 = 19, capped by 256 keys per split (4096 / 256)
    assert ws(1, 64, 8, 4096, 128, 0) == expect(1, 64, 8, 16, 128)
    assert ws(1, 64, 8, 65536, 128, 0) == expect(1, 64, 8, 19, 128)
    # 16 groups: 152 // 16 = 9 splits beat one per 4096 keys (8)
    assert ws(2, 64, 8, 32768, 128, 0) == expect(2, 64, 8, 9, 128)
    # 64 groups: 152 // 64 = 2, the same as one per 4096 keys
    assert ws(8, 64, 8, 8192, 128, 0) == expect(8, 64, 8, 2, 128)
    assert ws(2, 32, 2, 100, 64, 1) == expect(2, 32, 2, 1, 64)
    assert ws(1, 1, 1, 1, 128, 0) > 0
    assert ws(0, 64, 8, 10, 128, 0) == 0
    assert ws(1, 64, 8, 10, 96, 0) == 0
    assert ws(1, 64, 8, 10, 128, 300) == 0
    assert ws(1, 64, 8, 10, 128, 0, nsm=0) == 0
    # the automatic floor follows the SM count: 76 SMs give 76 // 8 = 9 splits for 8 groups
    # (16384 keys: one split per 4096 keys would give 4)
    assert ws(1, 64, 8, 16384, 128, 0, nsm=76) == expect(1, 64, 8, 9, 128)
    assert ws(1, 64, 8, 16384, 128, 0, nsm=304) == expect(1, 64, 8, 38, 128)
    # fixed split counts keep their splits; the pieces follow the SM count (512 items are
    # 6.7 waves on 76 SMs: whole splits)
    assert ws(4, 64, 8, 32768, 128, 16, nsm=76) == expect(4, 64, 8, 16, 128)


def test_current_device_workspace_size_needs_a_device(lib):
    import torch
    n = gb.attn_decode_workspace_size(4, 64, 8, 32768, 128, 16)
    if torch.cuda.is_available():
        nsm = torch.cuda.get_device_properties(0).multi_processor_count
        assert n == gb.attn_decode_workspace_bytes(4, 64, 8, 1, 32768, 128, 16, nsm)
    else:
        assert n == 0


def test_profile_case_driver_parses_without_gpu():
    """The profiling driver that the ncu summaries name is importable and parses its
    arguments on a machine without a GPU."""
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "-m", "streaming_attention_flashattention_gb300.profile_case", "--help"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert "multitoken" in r.stdout


def test_host_workspace_size_rejects_invalid_sizes(lib):
    f = gb.attn_fwd_host_workspace_size
    assert f(0, 8, 2, 128, 128, 128) == 0
    assert f(1, 8, 3, 128, 128, 128) == 0          # Hq % Hkv != 0
    assert f(1, 8, 2, 128, 128, 96) == 0           # d not 64 / 128
    assert f(1, 8, 2, 128, 128, 128, 7) == 0       # dtype


def test_positions_argument_validation(lib):
    def pos(q=A, k=A, v=A, o=B_, lse=None, B=1, Hq=2, Hkv=1, Sq=128, Skv=128, d=128, scale=0.1,
            qp=0, kp=0):
        return lib.attn_fwd_positions(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, d, scale, qp, kp,
                                      None)
    assert pos(q=None) == -1
    assert pos(Sq=0) == -1
    assert pos(Hq=3, Hkv=2) == -1
    assert pos(scale=-1.0) == -1
    assert pos(qp=1 << 41) == -1
    assert pos(kp=-(1 << 41)) == -1
    assert pos(d=96) == -2
    assert pos(o=MIS) == -3
    assert pos(B=70000, Hq=70000, Hkv=70000) == -7


def test_merge_argument_validation(lib):
    def mg(oa=A, la=A, ta=0, ob=A, lb=A, tb=0, oo=B_, lo=None, to=1, rows=10, d=128):
        return lib.attn_merge(oa, la, ta, ob, lb, tb, oo, lo, to, rows, d, None)
    assert mg(oa=None) == -1
    assert mg(lb=None) == -1
    assert mg(oo=None) == -1
    assert mg(ta=7) == -1
    assert mg(to=-1) == -1
    assert mg(rows=-1) == -1
    assert mg(d=0) == -1
    assert mg(d=32) == -2
    assert mg(ob=MIS) == -3
    assert mg(la=A + 2) == -3
    assert mg(rows=1 << 41) == -7
    assert mg(rows=0) == 0            # nothing to do, nothing launched
    assert mg(oa=None, ob=None, la=None, lb=None, oo=None, rows=0) == 0


def test_binding_status_constants_match_the_header():
    text = open(HEADER).read()
    enum = dict((n, int(v)) for n, v in re.findall(r"(GBATTN_(?:OK|ERR_\w+))\s*=\s*(-?\d+)", text))
    assert len(enum) == 8
    for name, value in enum.items():
        assert getattr(gb, name) == value, name


def test_decode_host_argument_validation(lib):
    lens_ok = (ctypes.c_int * 2)(5, 7)
    lens_bad = (ctypes.c_int * 2)(5, 9000)

    def dh(q=A, kc=A, vc=A, lens=None, o=B_, B=2, Hq=8, Hkv=1, Lmax=4096, d=128, scale=0.1,
           ns=0, ws=A, wsb=1 << 30):
        lens = lens_ok if lens is None else lens
        return lib.attn_decode_host(q, kc, vc, lens, o, None, B, Hq, Hkv, Lmax, d, scale, ns, ws,
                                    wsb, None)
    assert dh(q=None) == -1
    assert dh(B=0) == -1
    assert dh(Hq=6, Hkv=4) == -1
    assert dh(scale=0.0) == -1
    assert dh(ns=300) == -1
    assert dh(d=80) == -2
    assert dh(lens=lens_bad) == -1            # a length beyond Lmax, seen on the host
    assert gb.load_library().attn_decode_host_workspace_size(0, 8, 1, 4096, 128, 0) == 0
