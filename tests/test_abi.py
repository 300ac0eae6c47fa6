"""Host-side checks of the C ABI (no GPU needed, nothing is launched).

- libkda.so builds, loads and exports every function include/kda.h declares;
- status strings, ABI version, workspace sizing;
- argument validation rejects bad calls before any launch (the pointers used
  here are never dereferenced: every case fails a host-side check first).
"""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_wise_gb300 import build
    build.build()
    import gated_delta_rule_wise_gb300 as kda
    return kda.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("kda_chunk_fwd", "kda_decode_step", "kda_chunk_fwd_workspace_size",
                 "kda_status_string", "kda_chunk_fwd_status"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    from gated_delta_rule_wise_gb300 import library_path
    out = subprocess.run(["nm", "-D", "--defined-only", library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kda_[a-z0-9_]+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in declared_functions():
        assert getattr(lib, n) is not None


def test_header_compiles_as_plain_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "kda.h"\nint main(void){ return kda_abi_version() == KDA_ABI_VERSION ? 0 : 1; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-c", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(tmp_path / "use.o")], check=True)


def test_status_strings_and_version(lib):
    import gated_delta_rule_wise_gb300 as kda
    assert kda.kda_abi_version() == kda.ABI_VERSION
    for code in range(5):
        s = kda.kda_status_string(code)
        assert s.startswith("KDA_")
    assert "unknown" in kda.kda_status_string(99)


def test_workspace_size(lib):
    import gated_delta_rule_wise_gb300 as kda
    ws = kda.kda_chunk_fwd_workspace_size
    assert ws(1, 1, 64, 16, 16, 16, kda.KDA_F32, kda.KDA_ALPHA_CHANNEL) >= 256
    assert ws(1, 32, 131072, 128, 128, 64, kda.KDA_BF16, kda.KDA_ALPHA_CHANNEL) >= 256
    assert ws(1, 1, 64, 24, 16, 16, kda.KDA_F32, kda.KDA_ALPHA_NONE) == 0      # dk unsupported
    assert ws(1, 1, 64, 16, 16, 8, kda.KDA_F32, kda.KDA_ALPHA_NONE) == 0       # C unsupported
    assert ws(-1, 1, 64, 16, 16, 16, kda.KDA_F32, kda.KDA_ALPHA_NONE) == 0     # negative
    assert ws(1, 1, 64, 16, 16, 16, 7, kda.KDA_ALPHA_NONE) == 0                # bad dtype
    assert ws(1, 1, 64, 16, 16, 16, kda.KDA_F32, 9) == 0                       # bad mode
    assert ws(1, 1, 64, 16, 16, 16, kda.KDA_F32, kda.KDA_ALPHA_NONE, 6) == 0   # bad path
    wsx = kda.kda_chunk_fwd_workspace_size
    big = (1, 32, 4096, 128, 128, 64, kda.KDA_BF16, kda.KDA_ALPHA_CHANNEL)
    # both scans of the tensor path read the same per-chunk records
    assert wsx(*big, kda.KDA_PATH_TENSOR_SPLIT_SCAN) == wsx(*big, kda.KDA_PATH_TENSOR)
    assert wsx(*big, kda.KDA_PATH_TENSOR_WIDE_SCAN) == wsx(*big, kda.KDA_PATH_TENSOR)
    assert wsx(1, 2, 64, 64, 64, 64, kda.KDA_BF16, 0, kda.KDA_PATH_TENSOR_WIDE_SCAN) == 0
    assert wsx(*big, kda.KDA_PATH_TENSOR_PIPELINED) == wsx(*big, kda.KDA_PATH_TENSOR)
    assert wsx(1, 2, 64, 64, 64, 64, kda.KDA_BF16, 0, kda.KDA_PATH_TENSOR_PIPELINED) == 0


def test_host_buffer_size(lib):
    """kda_chunk_fwd_host_buffer_size: segments of the sequence (group_heads = 0)
    or head groups; both hold the workspace of one step and two staging slots
    of its inputs and outputs, so each is at least that step's workspace plus
    twice its input bytes; invalid arguments give 0."""
    import gated_delta_rule_wise_gb300 as kda
    hb, ws = kda.kda_chunk_fwd_host_buffer_size, kda.kda_chunk_fwd_workspace_size
    B, H, T, d, C = 1, 32, 131072, 128, 64
    bf, ch = kda.KDA_BF16, kda.KDA_ALPHA_CHANNEL
    per_tok_in = 2 * (2 * d + d) + 4 + 4 * d            # q, k, v bf16, beta, channel log_alpha
    seg_T = -(-T // 16)
    seg_T = -(-seg_T // C) * C                           # a chunk-aligned sixteenth of T
    seg = hb(B, H, T, d, d, C, bf, ch, 0)
    assert seg >= ws(1, B * H, seg_T, d, d, C, bf, ch) + 2 * B * H * seg_T * per_tok_in
    grp = hb(B, H, T, d, d, C, bf, ch, 4)
    assert grp >= ws(1, 4, T, d, d, C, bf, ch) + 2 * 4 * T * per_tok_in
    # a sequence shorter than one chunk still gets one segment of a chunk
    assert hb(1, 2, 40, d, d, C, bf, ch, 0) >= ws(1, 2, C, d, d, C, bf, ch)
    assert hb(-1, H, T, d, d, C, bf, ch, 0) == 0
    assert hb(B, H, T, d, d, C, bf, ch, -1) == 0
    assert hb(B, H, T, 24, 24, C, bf, ch, 0) == 0       # unsupported head size


FAKE = 0x7f0000000000  # 256-byte aligned, never dereferenced by these cases


def _chunk(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, beta=FAKE, la=FAKE, h0=None, o=FAKE, hT=FAKE,
             B=1, H=1, T=64, dk=16, dv=16, C=16, dt=0, am=2, ws=FAKE, wsb=1 << 20, st=None, path=0,
             ev=None, nev=0)
    a.update(kw)
    return lib.kda_chunk_fwd_ex(a["q"], a["k"], a["v"], a["beta"], a["la"], a["h0"], a["o"],
                                a["hT"], a["B"], a["H"], a["T"], a["dk"], a["dv"], a["C"],
                                a["dt"], a["am"], a["ws"], a["wsb"], a["st"], a["path"],
                                a["ev"], a["nev"])


def test_chunk_argument_validation(lib):
    INV, UNS, OK = 1, 2, 0
    assert _chunk(lib, q=None) == INV
    assert _chunk(lib, o=None) == INV
    assert _chunk(lib, k=FAKE + 8) == INV            # misaligned
    assert _chunk(lib, ws=FAKE + 16) == INV          # workspace must be 256-aligned
    assert _chunk(lib, wsb=16) == INV                # workspace too small
    assert _chunk(lib, la=None) == INV               # decay mode needs log_alpha
    assert _chunk(lib, am=0) == INV                  # ... and NONE forbids it
    assert _chunk(lib, dk=48) == UNS
    assert _chunk(lib, dv=256) == UNS
    assert _chunk(lib, C=128) == UNS
    assert _chunk(lib, B=-1) == INV
    assert _chunk(lib, dt=3) == INV
    assert _chunk(lib, B=70000, H=1) == UNS
    assert _chunk(lib, path=2, dt=0) == UNS          # tensor path needs bf16
    assert _chunk(lib, path=3, dt=0) == UNS          # ... both of its scans
    assert _chunk(lib, path=4, dt=0) == UNS
    assert _chunk(lib, path=4, dt=1, dk=64, dv=64, C=64) == UNS   # wide scan: d = 128 only
    assert _chunk(lib, path=5, dt=0) == UNS                       # pipelined: tensor path
    assert _chunk(lib, path=5, dt=1, dk=64, dv=64, C=64) == UNS   # ... at d = 128 only
    assert _chunk(lib, path=6) == INV                # unknown path
    assert _chunk(lib, nev=2) == INV                 # events requested but NULL
    one = (ctypes.c_void_p * 1)(FAKE)
    assert _chunk(lib, ev=one, nev=1) == INV         # fewer events than launches + 1
    assert _chunk(lib, B=0) == OK                    # nothing to do, nothing launched
    assert _chunk(lib, H=0, q=None, k=None, v=None) == OK


def test_decode_argument_validation(lib):
    f = lib.kda_decode_step
    args = lambda **kw: [kw.get(n, d) for n, d in (
        ("q", FAKE), ("k", FAKE), ("v", FAKE), ("beta", FAKE), ("la", FAKE), ("S", FAKE),
        ("o", FAKE), ("N", 4), ("H", 2), ("dk", 128), ("dv", 128), ("dt", 1), ("am", 2),
        ("st", None))]
    assert f(*args(S=None)) == 1
    assert f(*args(S=FAKE + 4)) == 1
    assert f(*args(la=None)) == 1
    assert f(*args(am=0)) == 1
    assert f(*args(dk=100)) == 2
    assert f(*args(N=-3)) == 1
    assert f(*args(N=0)) == 0


def test_launch_queries(lib):
    import gated_delta_rule_wise_gb300 as kda
    assert kda.kda_chunk_fwd_launches(1, 1, 64, 16, 16, 16, kda.KDA_F32, 2) >= 1
    assert kda.kda_chunk_fwd_launches(0, 1, 64, 16, 16, 16, kda.KDA_F32, 2) == 0
    assert kda.kda_chunk_fwd_launches(1, 1, 64, 24, 16, 16, kda.KDA_F32, 2) == -1
    names = kda.kda_chunk_fwd_kernel_names(1, 32, 131072, 128, 128, 64, kda.KDA_BF16, 2)
    assert names and all(n in kda.KERNEL_SOURCES for n in names)
    for n, files in kda.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(ROOT, "gated_delta_rule_wise_gb300", "csrc", f))


def test_tensor_path_is_what_auto_picks_for_bf16_c64(lib):
    import gated_delta_rule_wise_gb300 as kda
    names = kda.kda_chunk_fwd_kernel_names(1, 32, 131072, 128, 128, 64, kda.KDA_BF16,
                                           kda.KDA_ALPHA_CHANNEL)
    assert names == ["kda_prep_kernel", "kda_scan_kernel"]
    assert kda.kda_chunk_fwd_kernel_names(1, 1, 0, 128, 128, 64, kda.KDA_BF16, 2) == ["kda_scan_kernel"]
    assert kda.kda_chunk_fwd_kernel_names(1, 1, 64, 16, 16, 16, kda.KDA_F32, 2) == ["chunk_ffma_kernel"]
    big = kda.kda_chunk_fwd_workspace_size(1, 32, 131072, 128, 128, 64, kda.KDA_BF16, 2)
    # one 98816-byte record per (head, chunk), then its 768 bytes of normaliser
    # sums, then one float32 128 x 128 state per head and 256 bytes of work counters
    assert big == 256 + 32 * 2048 * (98816 + 768) + 32 * 128 * 128 * 4 + 256


def test_pipelined_launch_plan(lib):
    """A pipelined call: up to 16 segments of at least 8 chunks, a prep and a
    scan launch per segment, the one-CTA-per-head scan except for the last
    segment's split scan; one segment below 16 chunks."""
    import gated_delta_rule_wise_gb300 as kda
    P = kda.KDA_PATH_TENSOR_PIPELINED

    def names(T, H=32):
        return kda.kda_chunk_fwd_kernel_names(1, H, T, 128, 128, 64, kda.KDA_BF16, 2, P)
    assert names(131072) == ["kda_prep_kernel", "kda_scan_wide_kernel"] * 15 + \
        ["kda_prep_kernel", "kda_scan_kernel"]                       # 2048 chunks: 16 x 128
    assert names(64 * 131 + 1) == ["kda_prep_kernel", "kda_scan_wide_kernel"] * 14 + \
        ["kda_prep_kernel", "kda_scan_kernel"]                       # 131 chunks: 15 x 9, last 5
    assert names(64 * 15) == ["kda_prep_kernel", "kda_scan_kernel"]  # 15 chunks: one segment
    assert names(64 * 16) == ["kda_prep_kernel", "kda_scan_wide_kernel",
                              "kda_prep_kernel", "kda_scan_kernel"]
    assert names(0) == ["kda_scan_kernel"]                           # empty: h0 -> hT
    assert lib.kda_chunk_fwd_launches(1, 32, 131072, 128, 128, 64, 1, 2, P) == 32


def test_status_and_selftest_validation(lib):
    assert lib.kda_chunk_fwd_status(None, None) == 1
    assert lib.kda_selftest_wait_timeout(FAKE, 256, 0, None) == 1
    assert lib.kda_selftest_wait_timeout(FAKE, 16, 10, None) == 1


def test_rule_argument_checks_before_any_launch(lib):
    """kda_chunk_fwd_rule rejects bad rule / map combinations synchronously,
    before it touches the device (fake pointers, no GPU needed)."""
    def call(rule, maps, h0=None, hT=FAKE):
        return lib.kda_chunk_fwd_rule(FAKE, FAKE, FAKE, None, None, h0, FAKE, hT,
                                      1, 1, 64, 128, 128, 64, 1, 0, rule, maps, FAKE, 1 << 30,
                                      None)
    assert call(3, 0) == 1                      # unknown rule
    assert call(1, 8) == 1                      # unknown map bit
    assert call(2, 2) == 1                      # beta map with a linear rule
    assert call(0, 1 | 4) == 1                  # two maps for q, k
    assert call(0, 4) == 1                      # the feature map belongs to the linear rules
    assert call(2, 4, h0=FAKE, hT=None) == 2    # the normalised rule starts from zero ...
    assert call(2, 4, h0=None, hT=FAKE) == 2    # ... and keeps its state (S, z) internal


def test_ops_fail_loudly_without_the_library(monkeypatch):
    """No fallback: with libkda.so absent every entry point raises."""
    import gated_delta_rule_wise_gb300 as kda
    monkeypatch.setattr(kda, "_lib", None)
    monkeypatch.setattr(kda, "library_path", lambda: "/nonexistent/libkda.so")
    with pytest.raises(RuntimeError, match="missing"):
        kda.kda_chunk_fwd_workspace_size(1, 1, 64, 16, 16, 16, kda.KDA_F32, 2)
    with pytest.raises(RuntimeError, match="missing"):
        kda.load_library()


def test_package_does_not_import_the_oracle():
    """The library path and the oracle share nothing: importing and loading
    the package leaves the oracle unimported."""
    code = ("import sys, gated_delta_rule_wise_gb300 as kda; kda.load_library(); "
            "print('oracle' in sys.modules, 'workloads' in sys.modules)")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    p = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.split()[:2] == ["False", "False"], p.stdout
