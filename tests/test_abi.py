"""The C-ABI library builds, loads and exports what include/fa.h declares, and
rejects bad arguments before touching the GPU (no compute call is made)."""
import ctypes
import itertools
import os
import re
import shutil

import pytest

import io_aware_attention_gb300 as fa
from io_aware_attention_gb300 import _build

HEADER = os.path.join(_build.INCLUDE, "fa.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists(_build.LIB_PATH),
                                reason="neither nvcc nor a built library")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fa.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert declared_functions() == sorted(fa.EXPORTS)


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    for code in range(6):
        s = lib.fa_status_string(code)
        assert s and s != b"unknown status"
    assert lib.fa_status_string(99) == b"unknown status"
    assert fa.version() >= 100


P = 1 << 20  # fake, 16-byte aligned "device" addresses: never dereferenced


def call(lib, q=P, k=2 * P, v=3 * P, o=4 * P, lse=5 * P, B=1, H=1, N=16, d=64, causal=0,
         scale=0.125):
    vp = ctypes.c_void_p
    return lib.fa_fwd(vp(q), vp(k), vp(v), vp(o), vp(lse), B, H, N, d, causal, scale, None)


@pytest.mark.parametrize("kw, status", [
    (dict(q=0), 1), (dict(k=0), 1), (dict(v=0), 1), (dict(o=0), 1), (dict(lse=0), 1),
    (dict(B=0), 1), (dict(H=-1), 1), (dict(N=0), 1), (dict(d=0), 1),
    (dict(causal=2), 1), (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(scale=0.0), 1), (dict(scale=-0.1), 1),
    (dict(d=100), 2), (dict(d=136), 2), (dict(d=4), 2), (dict(d=256), 2),  # head size: multiples of 8 to 128
    (dict(q=P + 8), 2), (dict(o=4 * P + 4), 2), (dict(lse=5 * P + 2), 2),
    (dict(o=P), 1),                       # o aliases q
    (dict(o=3 * P + 16), 1),              # o overlaps the tail of v
    (dict(lse=4 * P + 64), 1),            # lse inside o
    (dict(B=1 << 40, H=1 << 20), 1),      # element count overflows
])
def test_bad_arguments_are_rejected(lib, kw, status):
    assert call(lib, **kw) == status


def test_plain_c_client(lib, tmp_path):
    """The boundary is a C ABI: a C program built with gcc against fa.h alone
    links the library and gets the answers the header promises."""
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    exe = str(tmp_path / "abi_client")
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "abi_client.c")
    libdir = os.path.dirname(_build.LIB_PATH)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", _build.INCLUDE, src, "-o", exe, "-L", libdir,
                    "-l:" + os.path.basename(_build.LIB_PATH), "-Wl,-rpath," + libdir], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "FAIL" not in r.stdout and r.stdout.count("ok ") == 9


def test_device_status_without_a_gpu_is_a_cuda_error(lib):
    """Both status calls report FA_ERR_CUDA, not a crash, when no device can be
    read (this container has none; on a GPU machine they are exercised by
    tests/test_fa_timeout.py)."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    where = ctypes.c_uint32(7)
    assert lib.fa_check_device_status(None, ctypes.byref(where)) == 3
    assert lib.fa_get_device_status(None) == 3


def test_wait_limit_setter(lib):
    assert lib.fa_set_wait_limit_ns(5_000_000) == 0
    assert lib.fa_set_wait_limit_ns(0) == 0  # back to the default


def test_debug_hook_setter(lib):
    assert lib.fa_debug_skip_k_tile(-2) == 1
    assert lib.fa_debug_skip_k_tile(3) == 0
    assert lib.fa_debug_skip_k_tile(-1) == 0


def test_schedule_hook_setter(lib):
    assert lib.fa_debug_set_schedule(-2) == 1
    assert lib.fa_debug_set_schedule(2) == 1
    for order in (0, 1, -1):
        assert lib.fa_debug_set_schedule(order) == 0


def call_decode(lib, q=P, k=2 * P, v=3 * P, o=4 * P, lse=5 * P, B=1, H=1, Nq=1, Nk=64, d=128, causal=0,
                scale=0.125, ws=6 * P, ws_bytes=1 << 20):
    vp = ctypes.c_void_p
    return lib.fa_decode(vp(q), vp(k), vp(v), vp(o), vp(lse), B, H, Nq, Nk, d, causal, scale, vp(ws), ws_bytes,
                         None)


@pytest.mark.parametrize("kw, status", [
    (dict(q=0), 1), (dict(k=0), 1), (dict(o=0), 1), (dict(lse=0), 1),
    (dict(B=0), 1), (dict(Nq=0), 1), (dict(Nk=0), 1), (dict(causal=2), 1), (dict(scale=0.0), 1),
    (dict(causal=1, Nq=4, Nk=3), 1),   # the causal window needs Nq <= Nk
    (dict(d=100), 2), (dict(d=136), 2), (dict(Nq=9), 2),  # head size, more than 8 query rows
    (dict(q=P + 8), 2), (dict(lse=5 * P + 2), 2), (dict(ws=6 * P + 4), 2),
    (dict(o=3 * P + 16), 1),           # o overlaps v
    (dict(B=70000), 1),                # B*H over the grid's 65535
])
def test_bad_decode_arguments_are_rejected(lib, kw, status):
    assert call_decode(lib, **kw) == status


def test_static_decode_checks_arguments_first(lib):
    vp = ctypes.c_void_p
    # bad arguments are refused before any device call
    assert lib.fa_decode_static(vp(0), vp(2 * P), vp(3 * P), vp(4 * P), vp(5 * P), 1, 1, 1, 64, 128, 0, 0.1,
                                None) == 1
    assert lib.fa_decode_static(vp(P), vp(2 * P), vp(3 * P), vp(4 * P), vp(5 * P), 1, 1, 9, 64, 128, 0, 0.1,
                                None) == 2


def test_static_decode_argument_errors_come_before_the_size_check(lib):
    """fa_decode_static gives a call that fa_decode would refuse the same
    status, at sizes whose scratch need exceeds the static array (1000 heads
    of 8 query rows over 4096 keys: at least three splits each, 11.8 MB of
    partial results or more at any occupancy): the scale, alignment and
    overlap checks run before the device is queried and before
    FA_ERR_TOO_LARGE is considered."""
    vp = ctypes.c_void_p
    for wave in (152, 304, 608, 912, 1216):
        splits, _ = fa.debug_decode_plan(1000, 1, 8, 4096, 128, wave)
        assert 1000 * 8 * splits * 129 * 4 > 8 << 20

    def call(q=P, o=4 * P, lse=5 * P, scale=0.1):
        return lib.fa_decode_static(vp(q), vp(2 * P), vp(3 * P), vp(o), vp(lse), 1000, 1, 8, 4096, 128, 0, scale,
                                    None)

    assert call(scale=float("nan")) == 1
    assert call(scale=-1.0) == 1
    assert call(q=P + 8) == 2
    assert call(lse=5 * P + 2) == 2
    assert call(o=3 * P + 16) == 1  # o overlaps v


def test_decode_plan_covers_the_keys_in_whole_rounds(lib):
    """Every split plan cuts the key range into chunks of whole rounds (32
    keys at the least) that cover it exactly once, each at least 4 rounds
    long when the range is split."""
    for BH, Nq, Nk, d, wave in itertools.product((1, 3, 8, 64, 256, 1000, 4096), (1, 2, 4, 8),
                                                  (1, 100, 1000, 4096, 32768, 100000), (40, 64, 96, 128),
                                                  (152, 608, 1216)):
        splits, chunk = fa.debug_decode_plan(BH, 1, Nq, Nk, d, wave)
        assert (splits - 1) * chunk < Nk <= splits * chunk, (BH, Nq, Nk, d, wave)
        assert chunk % 32 == 0
        assert splits == 1 or chunk >= 128


def test_decode_plan_fills_whole_waves(lib):
    """The partial kernel's CTAs take waves of `wave` resident CTAs; a last
    wave of a few CTAs costs a whole chunk while the rest of the GPU idles.
    The decode bench workload (B8 H32, one query row, 32768 keys, d = 128; 4
    CTAs per SM on 152 SMs): 7 chunks a head give 1792 CTAs in 2.95 waves,
    where 5 chunks would give 1280, two waves and 64 CTAs.  At B2 H32, 19
    chunks a head give 1216 CTAs, two waves exactly.  Over many head counts,
    whenever the heads hold two waves of the shortest chunks (4 rounds of 128
    keys), the CTAs fill at least 90% of the waves they take."""
    assert fa.debug_decode_plan(8, 32, 1, 32768, 128, 608) == (7, 4736)
    assert fa.debug_decode_plan(2, 32, 1, 32768, 128, 608) == (19, 1792)
    for BH, Nk, wave in itertools.product(range(1, 1200, 7), (32768, 65536, 100000), (304, 608, 912, 1216)):
        if BH * -(-Nk // 512) < 2 * wave:
            continue
        splits, _ = fa.debug_decode_plan(BH, 1, 1, Nk, 128, wave)
        ctas = BH * splits
        assert ctas / (-(-ctas // wave) * wave) >= 0.9, (BH, Nk, wave, splits)


def test_decode_plan_search_matches_every_split_count(lib):
    """The plan tries a few dozen split counts, not all of them: up to 16,
    and the fullest for 1 to 8 waves.  Against a search over every count
    from 1 to the most the 4-round minimum allows, under the plan's own cost
    (waves x chunk x K and V bytes a key x wave, plus the partial results
    written and read back), the chosen count is within 5% of the best.  The
    counts it does not try are many waves of the shortest chunks; the cost
    does not charge a CTA's fixed start-up and merge work, which those pay
    most.  One query row at d = 128: rounds of 128 keys."""
    rnd, d, nq = 128, 128, 1

    def cost(BH, Nk, wave, s):
        chunk = (-(-Nk // s) + rnd - 1) // rnd * rnd
        splits = -(-Nk // chunk)
        partials = 2.0 * BH * nq * splits * (d + 1) * 4 if splits > 1 else 0.0
        return -(-(BH * splits) // wave) * chunk * 4 * d * wave + partials

    for BH, Nk, wave in itertools.product((1, 3, 8, 31, 64, 100, 256, 301, 777, 1024, 4096), (4096, 32768, 100000),
                                          (152, 456, 608, 1216)):
        splits, chunk = fa.debug_decode_plan(BH, 1, nq, Nk, d, wave)
        best = min(cost(BH, Nk, wave, s) for s in range(1, -(-Nk // (4 * rnd)) + 1))
        assert cost(BH, Nk, wave, splits) <= 1.05 * best, (BH, Nk, wave, splits)


def test_decode_plan_weighs_the_partials(lib):
    """Splitting 1100 heads of 8 query rows over 1024 keys would shorten the
    last wave but write and read back more partial results than it saves:
    the plan keeps one chunk a head."""
    assert fa.debug_decode_plan(11, 100, 8, 1024, 128, 608) == (1, 1024)


def test_decode_plan_argument_checks(lib):
    with pytest.raises(fa.FaError) as e:
        fa.debug_decode_plan(1, 1, 1, 64, 128, 0)  # wave < 1
    assert e.value.code == 1
    with pytest.raises(fa.FaError) as e:
        fa.debug_decode_plan(1, 1, 9, 64, 128, 608)  # more query rows than the kernel takes
    assert e.value.code == 2
    assert lib.fa_debug_decode_plan(1, 1, 1, 64, 128, 608, None, None) == 1


def test_decode_workspace_query_checks_arguments(lib):
    out = ctypes.c_size_t(0)
    assert lib.fa_decode_workspace_bytes(1, 1, 9, 64, 128, 0, ctypes.byref(out)) == 2
    assert lib.fa_decode_workspace_bytes(1, 1, 1, 64, 128, 0, None) == 1


def call_bwd(lib, q=P, k=2 * P, v=3 * P, o=4 * P, lse=5 * P, do=6 * P, dq=7 * P, dk=8 * P, dv=9 * P, B=1, H=1,
             N=16, d=128, causal=0, scale=0.125, ws=10 * P, ws_bytes=1 << 20):
    vp = ctypes.c_void_p
    return lib.fa_bwd(vp(q), vp(k), vp(v), vp(o), vp(lse), vp(do), vp(dq), vp(dk), vp(dv), B, H, N, d, causal,
                      scale, vp(ws), ws_bytes, None)


@pytest.mark.parametrize("kw, status", [
    (dict(q=0), 1), (dict(o=0), 1), (dict(lse=0), 1), (dict(do=0), 1), (dict(dq=0), 1), (dict(dv=0), 1),
    (dict(ws=0), 1), (dict(B=0), 1), (dict(N=0), 1), (dict(causal=2), 1), (dict(scale=0.0), 1),
    (dict(scale=float("nan")), 1),
    (dict(d=100), 2), (dict(d=256), 2), (dict(d=4), 2),  # head size
    (dict(do=6 * P + 8), 2), (dict(dk=8 * P + 2), 2), (dict(lse=5 * P + 2), 2), (dict(ws=10 * P + 4), 2),
    (dict(ws_bytes=64 * 130 * 4 - 16), 1),            # workspace one row short
    (dict(dq=P), 1),                                  # dq aliases q
    (dict(dk=6 * P + 16), 1),                         # dk overlaps dO
    (dict(dv=8 * P + 512), 1),                        # dv overlaps dk
    (dict(ws=9 * P + 256), 1),                        # workspace overlaps dv
    (dict(lse=7 * P + 64), 1),                        # dq overlaps lse
    (dict(B=1 << 40, H=1 << 20), 1),                  # element count overflows
])
def test_bad_bwd_arguments_are_rejected(lib, kw, status):
    assert call_bwd(lib, **kw) == status


def test_bwd_workspace_bytes(lib):
    out = ctypes.c_size_t(0)
    # rows rounded up to 64 per head; two fp32 row vectors and the fp32 dQ accumulator
    assert lib.fa_bwd_workspace_bytes(2, 3, 100, 128, ctypes.byref(out)) == 0
    assert out.value == 2 * 3 * 128 * (128 + 2) * 4
    assert lib.fa_bwd_workspace_bytes(1, 1, 64, 128, ctypes.byref(out)) == 0
    assert out.value == 64 * 130 * 4
    assert lib.fa_bwd_workspace_bytes(1, 1, 64, 64, ctypes.byref(out)) == 0
    assert out.value == 64 * 66 * 4
    assert lib.fa_bwd_workspace_bytes(1, 1, 64, 96, ctypes.byref(out)) == 0  # padded to 128 columns
    assert out.value == 64 * 130 * 4
    assert lib.fa_bwd_workspace_bytes(1, 1, 64, 40, ctypes.byref(out)) == 0  # padded to 64
    assert out.value == 64 * 66 * 4
    assert lib.fa_bwd_workspace_bytes(1, 1, 64, 100, ctypes.byref(out)) == 2
    assert lib.fa_bwd_workspace_bytes(1, 1, 0, 128, ctypes.byref(out)) == 1
    assert lib.fa_bwd_workspace_bytes(1, 1, 64, 128, None) == 1


def call_ew(lib, x=P, bias=2 * P, keep=3 * P, y=4 * P, rows=4, cols=64, p=0.1):
    vp = ctypes.c_void_p
    return lib.fa_bias_gelu_dropout(vp(x), vp(bias), vp(keep), vp(y), rows, cols, p, None)


@pytest.mark.parametrize("kw, status", [
    (dict(x=0), 1), (dict(bias=0), 1), (dict(y=0), 1), (dict(rows=0), 1), (dict(cols=-8), 1),
    (dict(p=1.0), 1), (dict(p=-0.1), 1), (dict(p=float("nan")), 1),
    (dict(cols=60), 2),                                   # cols not a multiple of 8
    (dict(x=P + 8), 2), (dict(y=4 * P + 4), 2), (dict(keep=3 * P + 2), 2),
    (dict(y=P + 64), 1),                                  # y overlaps x
    (dict(keep=4 * P + 16), 1),                           # keep inside y
    (dict(rows=1 << 40, cols=1 << 30), 1),                # element count overflows
])
def test_bad_ew_arguments_are_rejected(lib, kw, status):
    assert call_ew(lib, **kw) == status
