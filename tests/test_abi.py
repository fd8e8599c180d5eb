"""C-ABI checks that need no GPU: the library builds and loads, exports every function the
public headers declare, validates arguments on the host before touching the device, and
computes the exact T5 bucket thresholds."""
import ctypes
import os
import re

import pytest

import attention_relative_position_gb300 as fa
from attention_relative_position_gb300 import _build
from exact_buckets import exact_thresholds

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fa.load()


def _declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(fat_x?attn_\w+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 18
    assert "fat_xattn_fwd" in names and "fat_xattn_bwd" in names
    for n in names:
        assert hasattr(lib, n), n


def test_strerror(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert fa.fat_attn_strerror(code)
    assert "unknown" in fa.fat_attn_strerror(12345)


@pytest.mark.parametrize("nb,md,bidir", [(32, 128, True), (32, 128, False), (64, 1024, True),
                                         (64, 1024, False), (128, 4096, True), (8, 16, True),
                                         (4, 3, True), (256, 100000, True), (16, 20, False)])
def test_thresholds_are_exact(lib, nb, md, bidir):
    nbh = nb // 2 if bidir else nb
    thr, sat = fa.fat_attn_bucket_thresholds(nb, md, bidir)
    want = exact_thresholds(nbh, md)
    assert thr == want
    assert sat == (want[-1] if want else nbh // 2)


def test_threshold_cache_returns_exact_values_after_eviction(lib):
    """The library keeps the thresholds of a few (buckets, distance) pairs; a run over more
    pairs than it keeps, twice, must return the exact values every time (first computation,
    cached copy, recomputation after the entry was replaced)."""
    pairs = [(16 + 2 * (i % 8), 40 + 37 * i, True) for i in range(24)]
    for _ in range(2):
        for nb, md, bidir in pairs:
            thr, sat = fa.fat_attn_bucket_thresholds(nb, md, bidir)
            want = exact_thresholds(nb // 2, md)
            assert thr == want, (nb, md)
            assert sat == (want[-1] if want else nb // 4)


def test_known_saturation_distances(lib):
    # thresholds derived by hand in tests/golden/t5_buckets.txt
    assert fa.fat_attn_bucket_thresholds(32, 128, True) == ([12, 16, 23, 32, 46, 64, 91], 91)
    assert fa.fat_attn_bucket_thresholds(32, 128, False)[1] == 113
    assert fa.fat_attn_bucket_thresholds(64, 1024, True)[1] == 790


@pytest.mark.parametrize("nb,md,bidir", [(7, 128, True), (2, 128, True), (1, 128, False),
                                         (32, 8, True), (32, 16, False), (512, 4096, True)])
def test_bad_bucket_args(lib, nb, md, bidir):
    with pytest.raises(fa.FatAttnError) as e:
        fa.fat_attn_bucket_thresholds(nb, md, bidir)
    assert e.value.code == -3


def _shape(T=256, n=2, maxL=128, H=2, d=64):
    return fa._Shape(T, n, maxL, H, d, None)


FAKE = 1 << 20  # 16-byte aligned non-null host value; never dereferenced on these paths


def _fwd(lib, sh, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, table=None, nb=0, md=0, bidir=1, slopes=None, cu=FAKE,
             causal=0, scale=1.0, out=FAKE, lse=FAKE)
    a.update(kw)
    return lib.fat_attn_fwd(ctypes.byref(sh), a["q"], a["k"], a["v"], a["table"], a["nb"], a["md"],
                            a["bidir"], a["slopes"], a["cu"], a["causal"], a["scale"], a["out"],
                            a["lse"])


def test_fwd_argument_errors(lib):
    assert lib.fat_attn_fwd(None, FAKE, FAKE, FAKE, None, 0, 0, 1, None, FAKE, 0, 1.0, FAKE,
                            FAKE) == -1
    assert _fwd(lib, _shape(), q=None) == -1
    assert _fwd(lib, _shape(), cu=None) == -1
    assert _fwd(lib, _shape(d=96)) == -2
    assert _fwd(lib, _shape(H=0)) == -2
    assert _fwd(lib, _shape(T=-1)) == -2
    assert _fwd(lib, _shape(), q=FAKE + 8) == -2  # misaligned
    assert _fwd(lib, _shape(), table=FAKE, nb=31, md=128, bidir=1) == -3
    assert _fwd(lib, _shape(), table=FAKE, nb=32, md=8, bidir=1) == -3
    # a bucket layout whose in-kernel lookup table would not fit in shared memory
    assert _fwd(lib, _shape(), table=FAKE, nb=256, md=2_000_000, bidir=1) == -5
    # nothing to do: returns before touching the device
    assert _fwd(lib, _shape(T=0, n=0, maxL=0)) == 0


def test_fwd_ws_argument_errors(lib):
    def fwd_ws(sh, ws, wsb, **kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, cu=FAKE, causal=0)
        a.update(kw)
        return lib.fat_attn_fwd_ws(ctypes.byref(sh), a["q"], a["k"], a["v"], None, 0, 0, 1, None,
                                   a["cu"], a["causal"], 1.0, FAKE, FAKE, ws, wsb)
    assert fwd_ws(_shape(), FAKE, 1 << 20, q=None) == -1
    assert fwd_ws(_shape(d=96), FAKE, 1 << 20) == -2
    assert fwd_ws(_shape(), FAKE + 16, 1 << 20) == -2  # the workspace must be 256-byte aligned
    assert fwd_ws(_shape(T=0, n=0, maxL=0), None, 0) == 0  # nothing to do
    # the split needs the device's SM count: without a device no shape has one
    assert lib.fat_attn_fwd_workspace_size(ctypes.byref(_shape(T=16384, n=1, maxL=16384,
                                                               H=12))) == 0
    assert lib.fat_attn_fwd_workspace_size(None) == 0


def test_bwd_argument_errors(lib):
    sh = _shape()
    need = lib.fat_attn_bwd_workspace_size(ctypes.byref(sh))
    T, H, d = 256, 2, 64
    assert need == ((T * H * d * 4 + 255) // 256) * 256 + ((T * H * 4 + 255) // 256) * 256

    def bwd(**kw):
        a = dict(table=None, ws=FAKE, wsb=need, dbias=None, lse=FAKE, d=64)
        a.update(kw)
        s = _shape(d=a["d"])
        return lib.fat_attn_bwd(ctypes.byref(s), FAKE, FAKE, FAKE, a["table"], 32, 128, 1, None,
                                FAKE, 0, 1.0, FAKE, a["lse"], FAKE, a["ws"], a["wsb"], FAKE, FAKE,
                                FAKE, a["dbias"])

    assert bwd(lse=None) == -1
    assert bwd(dbias=FAKE) == -5          # table gradient without a table
    assert bwd(wsb=need - 1) == -2        # workspace too small
    assert bwd(ws=FAKE + 16) == -2        # workspace not 256-byte aligned
    assert bwd(d=80) == -2


def _bwd_table(lib, d, md):
    sh = _shape(d=d)
    need = lib.fat_attn_bwd_workspace_size(ctypes.byref(sh))
    return lib.fat_attn_bwd(ctypes.byref(sh), FAKE, FAKE, FAKE, FAKE, 32, md, 1, None, FAKE, 0,
                            1.0, FAKE, FAKE, FAKE, FAKE, need, FAKE, FAKE, FAKE, FAKE)


def test_lookup_table_limits_rejected(lib):
    # the first bucket layouts (32 buckets, bidirectional) past the table sizes the header
    # states are rejected before anything touches the device
    assert _fwd(lib, _shape(d=64), table=FAKE, nb=32, md=34405, bidir=1) == -5
    assert _fwd(lib, _shape(d=128), table=FAKE, nb=32, md=9437, bidir=1) == -5
    assert _bwd_table(lib, 64, 2662) == -5
    assert _bwd_table(lib, 128, 7591) == -5
    for md, entries in ((34404, 24687), (9436, 8303), (2661, 3083), (7590, 6951)):
        sat = fa.fat_attn_bucket_thresholds(32, md, True)[1]
        assert 2 * sat + 507 == entries


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the no-GPU path")
def test_lookup_table_limits_accepted(lib):
    # the largest layouts pass the host checks; the first CUDA call then fails (no GPU)
    assert _fwd(lib, _shape(d=64), table=FAKE, nb=32, md=34404, bidir=1) == -4
    assert _fwd(lib, _shape(d=128), table=FAKE, nb=32, md=9436, bidir=1) == -4
    assert _bwd_table(lib, 64, 2661) == -4
    assert _bwd_table(lib, 128, 7590) == -4


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the no-GPU path")
def test_valid_call_without_gpu_reports_cuda_error(lib):
    # host validation passes, the first CUDA call fails: an error code, no crash
    assert _fwd(lib, _shape()) == -4


def _xshape(Tq=64, Tk=300, n=2, mq=40, mk=200, Hq=4, Hkv=2, d=64):
    return fa._XShape(Tq, Tk, n, mq, mk, Hq, Hkv, d, None)


def _xfwd(lib, sh, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, table=None, nb=0, md=0, bidir=1, slopes=None, cuq=FAKE,
             cuk=FAKE, causal=0, scale=1.0, out=FAKE, lse=FAKE)
    a.update(kw)
    return lib.fat_xattn_fwd(ctypes.byref(sh), a["q"], a["k"], a["v"], a["table"], a["nb"],
                             a["md"], a["bidir"], a["slopes"], a["cuq"], a["cuk"], a["causal"],
                             a["scale"], a["out"], a["lse"])


def test_xattn_argument_errors(lib):
    assert lib.fat_xattn_fwd(None, FAKE, FAKE, FAKE, None, 0, 0, 1, None, FAKE, FAKE, 0, 1.0,
                             FAKE, FAKE) == -1
    assert _xfwd(lib, _xshape(), cuk=None) == -1
    assert _xfwd(lib, _xshape(Hq=6, Hkv=4)) == -2   # query heads not a multiple of kv heads
    assert _xfwd(lib, _xshape(Hkv=0)) == -2
    assert _xfwd(lib, _xshape(d=96)) == -2
    assert _xfwd(lib, _xshape(), k=FAKE + 4) == -2  # misaligned
    assert _xfwd(lib, _xshape(), table=FAKE, nb=31, md=128, bidir=1) == -3
    assert _xfwd(lib, _xshape(Tq=0, n=0, mq=0)) == 0  # nothing to do
    # split keys: at most 64 splits, and the workspace is required and checked
    sh = _xshape()
    need = lib.fat_xattn_splitkv_workspace_size(ctypes.byref(sh), 4)
    assert need >= 4 * 64 * 4 * 64 * 4
    assert lib.fat_xattn_splitkv_workspace_size(ctypes.byref(sh), 1) == 0
    def split(ns, ws=FAKE, wsb=need):
        return lib.fat_xattn_fwd_splitkv(ctypes.byref(sh), FAKE, FAKE, FAKE, None, 0, 0, 1, None,
                                         FAKE, FAKE, 0, 1.0, ns, ws, wsb, FAKE, FAKE)
    assert split(65) == -5
    assert split(0) == -5
    assert split(4, ws=None) == -1
    assert split(4, wsb=need - 1) == -2
    assert split(4, ws=FAKE + 16) == -2


def test_xattn_bwd_workspace_layout(lib):
    # dQ accumulator, then (grouped heads) dK and dV accumulators, then D, each 256-aligned
    a = lambda b: (b + 255) // 256 * 256  # noqa: E731
    sh = _xshape(Tq=64, Tk=300, Hq=4, Hkv=2, d=64)
    want = a(64 * 4 * 64 * 4) + 2 * a(300 * 2 * 64 * 4) + a(4 * 64 * 4)
    assert lib.fat_xattn_bwd_workspace_size(ctypes.byref(sh)) == want
    sh1 = _xshape(Tq=64, Tk=300, Hq=4, Hkv=4, d=128)
    assert lib.fat_xattn_bwd_workspace_size(ctypes.byref(sh1)) == a(64 * 4 * 128 * 4) + a(4 * 64 * 4)
    assert fa.fat_xattn_bwd_workspace_size(64, 300, 4, 2, 64) == want
    # self-attention is the special case
    s = _shape(T=256, H=2, d=64)
    x = _xshape(Tq=256, Tk=256, Hq=2, Hkv=2, d=64)
    assert lib.fat_attn_bwd_workspace_size(ctypes.byref(s)) == \
        lib.fat_xattn_bwd_workspace_size(ctypes.byref(x))
