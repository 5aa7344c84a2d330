"""The C ABI library: builds, loads, exports every declared symbol, and rejects
bad arguments on the host before touching the GPU (CPU only)."""
import ctypes
import os
import re
import subprocess

import pytest

from exact_io_aware_34_gb300 import build as fa_build
from exact_io_aware_34_gb300 import fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_\s\*]*?\b(fa_[a-z0-9_]+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert names == sorted(fa.EXPORTED), names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fa.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\sT\s(\w+)$", out.stdout, re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings(lib):
    assert fa.fa_status_string(0) == "FA_OK"
    assert fa.fa_status_string(1) == "FA_ERR_INVALID_ARG"
    assert fa.fa_status_string(2) == "FA_ERR_UNSUPPORTED"
    assert fa.fa_status_string(3) == "FA_ERR_CUDA"
    assert fa.fa_status_string(4) == "FA_ERR_TIMEOUT"
    assert fa.fa_status_string(99) == "FA_ERR_UNKNOWN"


# Fake, never-dereferenced device addresses: every case below is rejected by
# the host-side checks before any CUDA call is made.
A = 0x7F0000000000
GAP = 1 << 30


def call(lib, Q=A, K=A + GAP, V=A + 2 * GAP, O=A + 3 * GAP, L=A + 4 * GAP, B=1, H=1, N=128, d=128, scale=0.1):
    return lib.fa_fwd(Q, K, V, O, L, B, H, N, d, ctypes.c_float(scale), None)


@pytest.mark.parametrize("kwargs,expect", [
    (dict(Q=0), fa.FA_ERR_INVALID_ARG),
    (dict(K=0), fa.FA_ERR_INVALID_ARG),
    (dict(V=0), fa.FA_ERR_INVALID_ARG),
    (dict(O=0), fa.FA_ERR_INVALID_ARG),
    (dict(L=0), fa.FA_ERR_INVALID_ARG),
    (dict(N=0), fa.FA_ERR_INVALID_ARG),
    (dict(N=-5), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=0), fa.FA_ERR_INVALID_ARG),
    (dict(B=70000), fa.FA_ERR_INVALID_ARG),
    (dict(H=1 << 16), fa.FA_ERR_INVALID_ARG),
    (dict(B=1024, H=1024, N=4096), fa.FA_ERR_INVALID_ARG),      # B*H*N >= 2^31
    (dict(d=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(Q=A + 8), fa.FA_ERR_INVALID_ARG),                     # not 16-byte aligned
    (dict(O=A + 3 * GAP + 4), fa.FA_ERR_INVALID_ARG),
    (dict(L=A + 4 * GAP + 2), fa.FA_ERR_INVALID_ARG),
    (dict(O=A + 1024), fa.FA_ERR_INVALID_ARG),                  # O overlaps Q
    (dict(L=A + 2 * GAP + 64), fa.FA_ERR_INVALID_ARG),          # LSE overlaps V
    (dict(L=A + 3 * GAP + 128), fa.FA_ERR_INVALID_ARG),         # LSE overlaps O
])
def test_host_side_rejections(lib, kwargs, expect):
    assert call(lib, **kwargs) == expect


def test_fault_hook_rejects_zero_timeout(lib):
    st = lib.fa_fwd_fault_test(A, A + GAP, A + 2 * GAP, A + 3 * GAP, A + 4 * GAP, 1, 1, 128, 128,
                               ctypes.c_float(0.1), 0, 0, None)
    assert st == fa.FA_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(fa, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        fa.load_library(str(tmp_path / "libfa.so"))


def naive_call(lib, ws=A + 6 * GAP, ws_bytes=1 << 40, **kw):
    args = dict(Q=A, K=A + GAP, V=A + 2 * GAP, O=A + 3 * GAP, L=A + 4 * GAP, B=1, H=1, N=128, d=128, scale=0.1)
    args.update(kw)
    return lib.fa_naive_fwd(args["Q"], args["K"], args["V"], args["O"], args["L"], args["B"], args["H"], args["N"],
                            args["d"], ctypes.c_float(args["scale"]), ws, ws_bytes, None)


def test_naive_workspace_size(lib):
    assert fa.fa_naive_workspace_bytes(1, 1, 128) == 128 * 128 * 2
    assert fa.fa_naive_workspace_bytes(2, 3, 100) == 6 * 100 * 128 * 2      # rows padded to 64 elements
    assert fa.fa_naive_workspace_bytes(0, 1, 128) == 0


@pytest.mark.parametrize("kwargs,expect", [
    (dict(ws=0), fa.FA_ERR_INVALID_ARG),
    (dict(ws=A + 6 * GAP + 64), fa.FA_ERR_INVALID_ARG),        # not 128-byte aligned
    (dict(ws_bytes=128 * 128 * 2 - 1), fa.FA_ERR_INVALID_ARG),  # too small
    (dict(ws=A + 2 * GAP), fa.FA_ERR_INVALID_ARG),             # overlaps V
    (dict(Q=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
])
def test_naive_host_side_rejections(lib, kwargs, expect):
    assert naive_call(lib, **kwargs) == expect


# B*H = 65536 heads of one row: past the launches' gridDim.z limit, and inside
# the no-allocation array (65536 rows of 64 bf16 scores = 8 MiB); inputs spaced
# 1 TiB apart so that only the head count is wrong. Rejected before any CUDA call.
BIG_BH = dict(B=2, H=32768, N=1, **{n: (1 << 44) + (i << 40) for i, n in enumerate(("Q", "K", "V", "O", "L"))})


def test_naive_rejects_head_counts_past_the_grid_limit(lib):
    assert naive_call(lib, ws=(1 << 44) + (6 << 40), **BIG_BH) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_naive_workspace_bytes(2, 32768, 1) <= 64 << 20
    st = lib.fa_naive_fwd_noalloc(BIG_BH["Q"], BIG_BH["K"], BIG_BH["V"], BIG_BH["O"], BIG_BH["L"], 2, 32768, 1, 128,
                                  ctypes.c_float(0.1), None)
    assert st == fa.FA_ERR_UNSUPPORTED


def bwd_call(lib, **kw):
    args = dict(Q=A, K=A + GAP, V=A + 2 * GAP, O=A + 3 * GAP, L=A + 4 * GAP, dO=A + 5 * GAP, dQ=A + 6 * GAP,
                dK=A + 7 * GAP, dV=A + 8 * GAP, ws=A + 9 * GAP, ws_bytes=1 << 40, B=1, H=1, N=128, d=128,
                scale=0.1)
    args.update(kw)
    return lib.fa_bwd(args["Q"], args["K"], args["V"], args["O"], args["dO"], args["L"], args["dQ"], args["dK"],
                      args["dV"], args["B"], args["H"], args["N"], args["d"], ctypes.c_float(args["scale"]),
                      args["ws"], args["ws_bytes"], None)


def test_bwd_workspace_size(lib):
    assert fa.fa_bwd_workspace_bytes(1, 1, 128) == 2 * 128 * 4
    assert fa.fa_bwd_workspace_bytes(2, 3, 100) == 2 * 6 * 128 * 4       # rows padded to 128
    assert fa.fa_bwd_workspace_bytes(1, 2, 129) == 2 * 2 * 256 * 4
    assert fa.fa_bwd_workspace_bytes(1, 0, 128) == 0


@pytest.mark.parametrize("kwargs,expect", [
    (dict(dO=0), fa.FA_ERR_INVALID_ARG),
    (dict(dQ=0), fa.FA_ERR_INVALID_ARG),
    (dict(dK=0), fa.FA_ERR_INVALID_ARG),
    (dict(dV=0), fa.FA_ERR_INVALID_ARG),
    (dict(ws=0), fa.FA_ERR_INVALID_ARG),
    (dict(Q=0), fa.FA_ERR_INVALID_ARG),
    (dict(L=0), fa.FA_ERR_INVALID_ARG),
    (dict(dO=A + 5 * GAP + 8), fa.FA_ERR_INVALID_ARG),           # not 16-byte aligned
    (dict(dK=A + 7 * GAP + 4), fa.FA_ERR_INVALID_ARG),
    (dict(ws=A + 9 * GAP + 64), fa.FA_ERR_INVALID_ARG),          # workspace not 128-byte aligned
    (dict(ws_bytes=2 * 128 * 4 - 1), fa.FA_ERR_INVALID_ARG),     # workspace too small
    (dict(dQ=A + 512), fa.FA_ERR_INVALID_ARG),                   # dQ overlaps Q
    (dict(dV=A + 5 * GAP), fa.FA_ERR_INVALID_ARG),               # dV overlaps dO
    (dict(dK=A + 4 * GAP), fa.FA_ERR_INVALID_ARG),               # dK overlaps LSE
    (dict(dK=A + 6 * GAP + 256), fa.FA_ERR_INVALID_ARG),         # dK overlaps dQ
    (dict(ws=A + 8 * GAP), fa.FA_ERR_INVALID_ARG),               # workspace overlaps dV
    (dict(ws=A + 3 * GAP), fa.FA_ERR_INVALID_ARG),               # workspace overlaps O
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(N=0), fa.FA_ERR_INVALID_ARG),
    # 2 * B * H CTAs, past the 1-D grid limit (inputs spaced 1 TiB apart, so
    # that only the size is wrong)
    (dict(B=65535, H=32768, N=1, **{n: (1 << 44) + (i << 40) for i, n in enumerate(("Q", "K", "V", "O", "L"))}),
     fa.FA_ERR_UNSUPPORTED),
])
def test_bwd_host_side_rejections(lib, kwargs, expect):
    assert bwd_call(lib, **kwargs) == expect


def kv_call(lib, **kw):
    args = dict(Q=A, K=A + GAP, V=A + 2 * GAP, O=A + 3 * GAP, L=A + 4 * GAP, B=1, H=8, Hkv=2, Nq=1, Nkv=4096, d=128,
                scale=0.1, splits=4, ws=A + 5 * GAP, ws_bytes=1 << 40)
    args.update(kw)
    return lib.fa_fwd_kv(args["Q"], args["K"], args["V"], args["O"], args["L"], args["B"], args["H"], args["Hkv"],
                         args["Nq"], args["Nkv"], args["d"], ctypes.c_float(args["scale"]), args["splits"], args["ws"],
                         args["ws_bytes"], None)


@pytest.mark.parametrize("sizes,expect", [
    ((0, 1, 128, 128), fa.FA_ERR_INVALID_ARG),
    ((1, 0, 128, 128), fa.FA_ERR_INVALID_ARG),
    ((1, 1, 0, 128), fa.FA_ERR_INVALID_ARG),
    ((65536, 1, 128, 128), fa.FA_ERR_INVALID_ARG),
    ((1024, 1024, 2048, 128), fa.FA_ERR_INVALID_ARG),   # B*H*N >= 2^31
    ((1, 1, 128, 96), fa.FA_ERR_UNSUPPORTED),
])
def test_launch_shape_rejects_sizes(lib, sizes, expect):
    """The shape query checks sizes as fa_fwd does, before asking the device."""
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_launch_shape(*sizes)
    assert e.value.status == expect


def test_kv_workspace_and_splits(lib):
    # 4 splits of 8 query rows (H = 8, N_q = 1) with d = 128: 4 * 8 * 129 floats
    assert fa.fa_fwd_kv_workspace_bytes(1, 8, 2, 1, 4096, 128, 4) == 4 * 8 * 129 * 4
    assert fa.fa_fwd_kv_workspace_bytes(1, 8, 2, 1, 4096, 128, 1) == 0
    assert fa.fa_fwd_kv_workspace_bytes(1, 8, 2, 1, 200, 128, 9) == 2 * 8 * 129 * 4   # capped at 2 key blocks
    assert fa.fa_fwd_kv_workspace_bytes(1, 8, 2, 300, 300, 128, 1) == 0                # the fused kernel: no split
    assert fa.fa_fwd_kv_workspace_bytes(1, 8, 3, 1, 64, 128, 0) == 0                   # 8 % 3 != 0
    assert fa.fa_fwd_kv_num_splits(1, 8, 2, 1, 200, 128) in (1, 2)
    assert fa.fa_fwd_kv_num_splits(1, 8, 3, 1, 64, 128) == 0
    # long query blocks: 3 key ranges of 300 query rows of 8 heads
    assert fa.fa_fwd_kv_workspace_bytes(1, 8, 2, 300, 300, 128, 3) == 3 * 8 * 300 * 129 * 4


def test_kv_long_query_routing(lib):
    """N_q > 128: the fused forward kernel (1 split, no workspace) when its
    CTAs fill the device, else a key split over one wave of short-query CTAs."""
    # 4 * 32 heads * 16 CTAs of 256 query rows = 2048 CTAs: fused
    assert fa.fa_fwd_kv_num_splits(4, 32, 8, 4096, 4096, 128) == 1
    assert fa.fa_fwd_kv_workspace_bytes(4, 32, 8, 4096, 4096, 128, 0) == 0
    # 8 heads * 2 CTAs: 16 fused CTAs; 2 K/V heads * 4 heads * 4 query blocks = 32 short-query tiles
    s = fa.fa_fwd_kv_num_splits(1, 8, 2, 512, 32768, 128)
    assert 2 <= s <= 256
    assert fa.fa_fwd_kv_workspace_bytes(1, 8, 2, 512, 32768, 128, 0) == s * 8 * 512 * 129 * 4
    # one key block: nothing to split, the fused kernel
    assert fa.fa_fwd_kv_num_splits(1, 8, 2, 512, 100, 64) == 1


@pytest.mark.parametrize("kwargs,expect", [
    (dict(Hkv=3), fa.FA_ERR_INVALID_ARG),                        # H not a multiple of H_kv
    (dict(Hkv=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nq=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nkv=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(ws=0), fa.FA_ERR_INVALID_ARG),                         # 4 splits need a workspace
    (dict(ws=A + 5 * GAP + 16), fa.FA_ERR_INVALID_ARG),          # not 128-byte aligned
    (dict(ws_bytes=4 * 8 * 129 * 4 - 1), fa.FA_ERR_INVALID_ARG),  # too small
    (dict(ws=A + 2 * GAP), fa.FA_ERR_INVALID_ARG),               # overlaps V
    (dict(O=A + GAP + 64), fa.FA_ERR_INVALID_ARG),               # O overlaps K
    (dict(L=A + 3 * GAP + 4), fa.FA_ERR_INVALID_ARG),            # LSE overlaps O
    (dict(Q=A + 8), fa.FA_ERR_INVALID_ARG),
    (dict(Nq=300, Nkv=300, splits=2, ws_bytes=2 * 8 * 300 * 129 * 4 - 1), fa.FA_ERR_INVALID_ARG),  # long queries, small
])
def test_kv_host_side_rejections(lib, kwargs, expect):
    assert kv_call(lib, **kwargs) == expect


@pytest.mark.parametrize("kwargs,expect", [
    (dict(Op=0), fa.FA_ERR_INVALID_ARG),
    (dict(P=0), fa.FA_ERR_INVALID_ARG),
    (dict(rows=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(O=A + 8), fa.FA_ERR_INVALID_ARG),                  # misaligned
    (dict(O=A + 256), fa.FA_ERR_INVALID_ARG),                # O overlaps the partial O
    (dict(L=A + 3 * GAP + 64), fa.FA_ERR_INVALID_ARG),       # LSE overlaps O
])
def test_merge_host_side_rejections(lib, kwargs, expect):
    args = dict(Op=A, Lp=A + GAP, O=A + 3 * GAP, L=A + 3 * GAP + (1 << 20), P=4, rows=1000, d=128)
    args.update(kwargs)
    assert lib.fa_merge_partials(args["Op"], args["Lp"], args["O"], args["L"], args["P"], args["rows"], args["d"],
                                 None) == expect


# --- host-buffer forward (fa_fwd_host): checks that fail before any CUDA call -----------
def host_call(lib, **kw):
    args = dict(Q=A, K=A + GAP, V=A + 2 * GAP, O=A + 3 * GAP, L=A + 4 * GAP, B=1, H=4, N=1000, d=128, scale=0.1,
                chunks=0, ws=A + 5 * GAP, ws_bytes=1 << 40)
    args.update(kw)
    return lib.fa_fwd_host(args["Q"], args["K"], args["V"], args["O"], args["L"], args["B"], args["H"], args["N"],
                           args["d"], ctypes.c_float(args["scale"]), args["chunks"], args["ws"], args["ws_bytes"], None)


def test_host_workspace_bytes(lib):
    pad = lambda n: (n + 255) // 256 * 256
    assert fa.fa_fwd_host_workspace_bytes(1, 4, 1000, 128) == 4 * pad(4 * 1000 * 128 * 2) + pad(4 * 1000 * 4)
    assert fa.fa_fwd_host_workspace_bytes(2, 3, 77, 64) == 4 * pad(6 * 77 * 64 * 2) + pad(6 * 77 * 4)
    assert fa.fa_fwd_host_workspace_bytes(1, 4, 1000, 96) == 0
    assert fa.fa_fwd_host_workspace_bytes(0, 4, 1000, 128) == 0


@pytest.mark.parametrize("kwargs,expect", [
    (dict(Q=0), fa.FA_ERR_INVALID_ARG),
    (dict(O=0), fa.FA_ERR_INVALID_ARG),
    (dict(L=0), fa.FA_ERR_INVALID_ARG),
    (dict(N=0), fa.FA_ERR_INVALID_ARG),
    (dict(chunks=-1), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(ws=0), fa.FA_ERR_INVALID_ARG),                                   # no workspace
    (dict(ws=A + 5 * GAP + 128), fa.FA_ERR_INVALID_ARG),                   # not 256-byte aligned
    (dict(ws_bytes=4 * 4 * 1000 * 256 + 16000 - 1), fa.FA_ERR_INVALID_ARG),  # too small
    (dict(O=A + 64), fa.FA_ERR_INVALID_ARG),                                # O overlaps Q
    (dict(L=A + 3 * GAP + 8), fa.FA_ERR_INVALID_ARG),                       # LSE overlaps O
    (dict(ws=A + 2 * GAP), fa.FA_ERR_INVALID_ARG),                          # workspace overlaps V
])
def test_host_side_rejections_host_path(lib, kwargs, expect):
    assert host_call(lib, **kwargs) == expect
