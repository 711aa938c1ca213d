"""The C-ABI boundary without a GPU: the library builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

import fp8_mqa_logits_02_gb300 as fm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8_mqa_logits.h")

OK, INVALID, UNSUPPORTED, MISALIGNED = 0, -1, -2, -3


@pytest.fixture(scope="module")
def lib():
    fm.build()  # the library and its bounds-checking variant
    return fm.lib()


def header_functions():
    text = open(HEADER).read()
    return re.findall(r"FP8MQA_API\s+[\w\s\*]+?\b(fp8_mqa_\w+)\s*\(", text)


def test_header_declares_expected_entry_points():
    names = header_functions()
    assert "fp8_mqa_logits" in names
    assert len(names) == len(set(names)) == len(fm.SIGNATURES)
    assert set(names) == set(fm.SIGNATURES)


@pytest.mark.parametrize("path", [fm.LIB_PATH, fm.DEBUG_LIB_PATH])
def test_library_exports_every_declared_symbol(lib, path):
    handle = ctypes.CDLL(path)
    for name in header_functions():
        assert hasattr(handle, name), name


def test_status_codes_match_header(lib):
    text = open(HEADER).read()
    codes = dict((int(v), k) for k, v in re.findall(r"(FP8MQA_\w+)\s*=\s*(-?\d+)", text))
    assert codes == fm.STATUS
    for code, name in codes.items():
        assert lib.fp8_mqa_logits_strerror(code).decode().startswith(name)


def test_is_supported_truth_table(lib):
    assert fm.is_supported(8192, 8192)
    assert fm.is_supported(0, 0)
    assert fm.is_supported(1, 1)
    assert not fm.is_supported(16, 16, H=64)
    assert not fm.is_supported(16, 16, D=64)
    assert not fm.is_supported(-1, 16)
    assert not fm.is_supported(16, -1)
    assert not fm.is_supported(2 ** 26, 16)       # M*H = 2^31
    assert fm.is_supported(2 ** 26 - 1, 16)
    assert not fm.is_supported(16, 2 ** 31)
    # a device index that does not exist (or, here, no GPU at all) is never supported; a
    # negative index skips the device check
    assert not fm.is_supported(16, 16, device=4096)
    assert fm.is_supported(16, 16, device=-1)


def test_default_split(lib):
    # about 4, 20 or 16 units per SM for many, some or few row blocks; chunks of at least
    # 8 key tiles
    assert fm.default_split(8192, 8192, 152) == 1
    assert fm.default_split(16384, 32000, 152) == 1
    assert fm.default_split(4096, 32768, 152) == 6
    assert fm.default_split(1024, 131072, 152) == 19
    assert fm.default_split(1, 1, 152) == 1
    # at 128 key tiles per SM or fewer, the split with the fewest rounds x (set-up + tiles
    # per unit): one round of units where it fits, whole rows where they already fill it
    assert fm.default_split(64, 256, 152) == 2
    assert fm.default_split(64, 8192, 152) == 16     # 128 units of 4 tiles
    assert fm.default_split(512, 8192, 152) == 2     # 128 units of 32 tiles
    assert fm.default_split(128, 32768, 152) == 9    # 144 units of 29 tiles
    assert fm.default_split(2048, 2048, 152) == 1
    assert fm.default_split(1024, 1024, 152) == 1
    assert fm.default_split(128, 131072, 152) == 19  # 304 units of 54 tiles: two rounds
    assert fm.default_split(256, 65536, 152) == 9
    assert fm.default_split(2048, 8192, 152) == 1
    for M in (1, 7, 100, 5000):
        for N in (1, 129, 4000, 100000):
            s = fm.default_split(M, N, 152)
            assert 1 <= s <= max(1, -(-N // 128))


def _call(lib, M=16, N=16, H=32, D=128, clean=1, split=0, ptrs=None):
    p = ptrs or [0x1000] * 7
    return lib.fp8_mqa_logits(*p, M, N, H, D, clean, split, None)


def test_rejects_before_any_device_work(lib):
    # fake but aligned pointers: validation must fail before they could be dereferenced
    assert _call(lib, H=16) == UNSUPPORTED
    assert _call(lib, D=64) == UNSUPPORTED
    assert _call(lib, M=-1) == INVALID
    assert _call(lib, N=-5) == INVALID
    assert _call(lib, split=-1) == INVALID
    assert _call(lib, clean=2) == INVALID
    for i in range(7):
        ptrs = [0x1000] * 7
        ptrs[i] = None
        assert _call(lib, ptrs=ptrs) == INVALID, i
    for i, align in enumerate([16, 16, 16, 16, 4, 4, 4]):
        ptrs = [0x1000] * 7
        ptrs[i] = 0x1000 + (8 if align == 16 else 2)
        assert _call(lib, ptrs=ptrs) == MISALIGNED, i
    # empty problems are a no-op that never touches the device, even with null pointers
    assert _call(lib, M=0, ptrs=[None] * 7) == OK
    assert _call(lib, N=0, ptrs=[None] * 7) == OK


def test_wait_limit_setter_round_trips(lib):
    prev = fm.set_wait_limit_ns(12345)
    try:
        assert prev == 10 ** 9                      # the default: one second
        assert fm.set_wait_limit_ns(0) == 12345     # 0 restores the default
        assert fm.set_wait_limit_ns(0) == 10 ** 9
    finally:
        fm.set_wait_limit_ns(0)


def test_host_entry_rejects_bad_workspace(lib):
    need = lib.fp8_mqa_logits_host_workspace_bytes(16, 16, 32, 128)
    assert need > 16 * 16 * 4
    assert lib.fp8_mqa_logits_host_workspace_bytes(16, 16, 16, 128) == 0
    p = [0x1000] * 7
    assert lib.fp8_mqa_logits_host(*p, 16, 16, 32, 128, 1, 0, None, need, None) == INVALID
    assert lib.fp8_mqa_logits_host(*p, 16, 16, 32, 128, 1, 0, 0x1010, need, None) == MISALIGNED
    assert lib.fp8_mqa_logits_host(*p, 16, 16, 32, 128, 1, 0, 0x1000, need - 1, None) == INVALID


def test_binding_rejects_cpu_tensors(lib):
    import torch
    q = torch.zeros((4, 32, 128), dtype=torch.float8_e4m3fn)
    k = torch.zeros((8, 128), dtype=torch.float8_e4m3fn)
    with pytest.raises(ValueError, match="CUDA"):
        fm.fp8_mqa_logits(q, k, torch.ones(8), torch.ones(4, 32),
                          torch.zeros(4, dtype=torch.int32), torch.ones(4, dtype=torch.int32))
    with pytest.raises(TypeError):
        fm.fp8_mqa_logits(q.view(torch.uint8), k, torch.ones(8), torch.ones(4, 32),
                          torch.zeros(4, dtype=torch.int32), torch.ones(4, dtype=torch.int32))


def test_topk_rejects_bad_arguments_before_device_work(lib):
    p = 0x1000
    f = lib.fp8_mqa_topk
    assert f(p, 0, 10, 10, 5, p, p, None) == 0                     # no rows: nothing to do
    assert f(p, 4, 10, 10, 0, p, p, None) == -1
    assert f(p, 4, 10, 10, 2049, p, p, None) == -1
    assert f(p, 4, 10, 9, 5, p, p, None) == -1  # ld < N
    assert f(p, -1, 10, 10, 5, p, p, None) == -1
    assert f(None, 4, 10, 10, 5, p, p, None) == -1
    assert f(p, 4, 10, 10, 5, None, p, None) == -1
    assert f(p, 4, (1 << 30) + 1, (1 << 30) + 1, 5, p, p, None) == \
        -2
    assert f(p + 2, 4, 10, 10, 5, p, p, None) == -3
    assert f(p, 4, 10, 10, 5, p, p + 1, None) == -3


def test_topk_ex_rejects_unknown_flags_before_device_work(lib):
    p = 0x1000
    f = lib.fp8_mqa_topk_ex
    assert f(p, 0, 10, 10, None, None, 5, 1, p, p, None) == 0       # no rows: nothing to do
    assert f(p, 4, 10, 10, None, None, 5, 2, p, p, None) == -1      # an unknown flag bit
    assert f(p, 4, 10, 10, None, None, 5, -1, p, p, None) == -1
    assert f(p, 4, 10, 10, p, None, 5, 1, p, p, None) == -1         # ks without ke


def test_windowed_topk_rejects_bad_arguments_before_device_work(lib):
    p = 0x1000
    f = lib.fp8_mqa_topk_windowed
    assert f(p, 0, 10, 10, p, p, 5, p, p, None) == 0               # no rows: nothing to do
    assert f(p, 4, 10, 10, p, None, 5, p, p, None) == -1           # ks without ke
    assert f(p, 4, 10, 10, None, p, 5, p, p, None) == -1           # ke without ks
    assert f(p, 4, 10, 10, p, p, 0, p, p, None) == -1
    assert f(p, 4, 10, 9, p, p, 5, p, p, None) == -1               # ld < N
    assert f(p, 4, 10, 10, p + 2, p, 5, p, p, None) == -3          # ks misaligned
    assert f(p, 4, 10, 10, p, p + 1, 5, p, p, None) == -3          # ke misaligned
