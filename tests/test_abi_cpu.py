"""Host-only checks of the C ABI: the library loads, exports every function the
public headers declare, and rejects bad arguments before touching a device.
No compute call is made (this runs on machines without a GPU)."""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

import pytest

import dense_tiled_gemm_03_gb300 as gt
from dense_tiled_gemm_03_gb300 import build as native_build

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib():
    native_build.build()
    return gt.library()


def declared_functions() -> list[str]:
    names = []
    for header in sorted((ROOT / "include").glob("*.h")):
        text = header.read_text()
        names += re.findall(r"^GEMM_TN_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("gemm_tn", "gemm_tn_ex", "gemm_tn_host", "gemm_tn_status_string", "gemm_tn_last_cuda_error"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_version_status_strings_and_configs(lib):
    assert gt.gemm_tn_version() == 100
    assert gt.gemm_tn_status_string(gt.GEMM_TN_OK) == "GEMM_TN_OK"
    assert gt.gemm_tn_status_string(gt.GEMM_TN_ERR_TIMEOUT) == "GEMM_TN_ERR_TIMEOUT"
    assert gt.gemm_tn_status_string(99) == "GEMM_TN_ERR_UNKNOWN"
    names = [gt.gemm_tn_config_name(i) for i in range(gt.gemm_tn_num_configs())]
    assert names == ["1cta_n256", "1cta_n128", "2cta_n256", "2cta_n128", "2cta_n256_mc", "1cta_n128_splitk",
                     "1cta_decode_splitk", "1cta_n64"]
    assert gt.gemm_tn_config_name(-1) == "invalid"


def test_config_table(lib, monkeypatch):
    monkeypatch.delenv("GEMM_TN_FORCE_CONFIG", raising=False)
    sel = lambda m, n, k: gt.gemm_tn_config_name(gt.gemm_tn_select_config(gt.GEMM_TN_BF16, m, n, k))
    assert sel(128, 16384, 16384) == "1cta_n128"   # skinny: one 128-row block of outputs
    # few 128 x 128 tiles and a long K: K split over a cluster
    assert sel(128, 1024, 4096) == "1cta_n128_splitk"     # 8 tiles x 8 splits
    assert sel(128, 4096, 4096) == "1cta_n128_splitk"     # 32 tiles x 4 splits
    assert sel(64, 2048, 8192) == "1cta_n128_splitk"      # 16 tiles: 4 splits (15 clusters of 8 fit at once)
    assert sel(8, 4096, 4096) == "1cta_decode_splitk"     # <= 32 rows: B on the MMA's M side
    assert sel(33, 4096, 4096) == "1cta_n128_splitk"
    assert sel(256, 256, 256) == "1cta_n64"               # 4 k-blocks: too short to split; 8 tiles of 128 x 64
    assert sel(384, 384, 256) == "1cta_n64"               # 18 tiles of 128 x 64: at most half the SMs
    assert sel(1024, 1024, 256) == "1cta_n128"            # 128 tiles of 128 x 64 would be more than half
    splits = lambda m, n, k: gt.gemm_tn_select_splits(gt.GEMM_TN_F16, m, n, k)
    assert splits(128, 1024, 4096) == 8                   # 8 tiles, 64 k-blocks
    assert splits(64, 2048, 8192) == 4                    # 16 tiles: more than 15 clusters of 8
    assert splits(1024, 1024, 8192) == 2                  # 64 tiles: more than 36 clusters of 4
    assert splits(512, 512, 512) == 0                     # 8 k-blocks: 32 tiles of 128 x 64 in one round
    assert sel(512, 512, 512) == "1cta_n64"
    assert sel(1024, 1024, 1024) == "1cta_n64"            # 16 k-blocks, a 2-way split: 128 tiles of 128 x 64
    assert sel(200, 512, 512) == "1cta_n64"               # 8 k-blocks, 16 tiles of 128 x 64
    assert sel(512, 512, 576) == "1cta_n128_splitk"       # 9 k-blocks at a 4-way split: the split stays
    assert sel(512, 512, 500) == "1cta_n128_splitk"       # K not a multiple of 64: one k-block per copy
    assert sel(128, 1024, 512) == "1cta_n128_splitk"      # one row of tiles (M <= 128): the split stays
    assert splits(256, 256, 960) == 4
    assert splits(256, 256, 1024) == 4                    # 16 k-blocks: 8 splits would leave 2 per CTA
    assert splits(8, 4096, 4096) == 4                     # the decode kernel's split
    assert splits(8, 2048, 512) == 2                      # decode kernel: 4 k-blocks per CTA kept
    assert splits(64, 2048, 512) == 4                     # 128 x 128 split-K kernel: 2 per CTA
    assert splits(256, 256, 256) == 0 and splits(8192, 8192, 8192) == 0 and splits(0, 5, 5) == 0
    assert sel(1024, 2048, 4096) == "1cta_n128"           # 128 tiles: one round of single-CTA tiles
    assert sel(1280, 2048, 4096) == "1cta_n256"           # 160 tiles of 128 x 128, 80 of 128 x 256: one round
    assert sel(2048, 2048, 2048) == "1cta_n256"
    assert sel(2048, 2048, 8192) == "2cta_n256_mc"        # long K: pair tiles stream less per SM
    assert sel(2560, 2560, 1024) == "2cta_n256_mc"        # 200 tiles of 128 x 256: more than one round
    # with GB300's resident clusters (76 pairs, 36 four-CTA clusters):
    assert sel(8192, 8192, 8192) == "2cta_n256"      # 14 rounds of pair tiles vs 15 of multicast tiles
    assert sel(4096, 4096, 4096) == "2cta_n256_mc"   # 4 rounds either way: multicast streams more per SM
    assert sel(3001, 5003, 4097) == "2cta_n256_mc"
    assert gt.gemm_tn_select_config(gt.GEMM_TN_BF16, 0, 5, 5) == -1
    assert gt.gemm_tn_select_config(7, 5, 5, 5) == -1
    monkeypatch.setenv("GEMM_TN_FORCE_CONFIG", "1cta_n128")
    assert sel(8192, 8192, 8192) == "1cta_n128"
    monkeypatch.setenv("GEMM_TN_FORCE_CONFIG", "2")
    assert sel(8192, 8192, 8192) == "2cta_n256"


# Fake, well-separated addresses: validation never dereferences them.
A, B, C = 0x10000000, 0x20000000, 0x30000000


@pytest.mark.parametrize("args,expected", [
    ((5, 4, 4, 4, A, 4, B, 4, C, 4), gt.GEMM_TN_ERR_UNSUPPORTED_DTYPE),
    ((0, -1, 4, 4, A, 4, B, 4, C, 4), gt.GEMM_TN_ERR_INVALID_VALUE),
    ((0, 4, 4, 1 << 31, A, 1 << 31, B, 1 << 31, C, 4), gt.GEMM_TN_ERR_INVALID_VALUE),
    ((0, 4, 4, 4, A, 4, B, 4, None, 4), gt.GEMM_TN_ERR_INVALID_VALUE),      # NULL C
    ((0, 4, 4, 4, None, 4, B, 4, C, 4), gt.GEMM_TN_ERR_INVALID_VALUE),      # NULL A
    ((0, 4, 4, 4, A, 3, B, 4, C, 4), gt.GEMM_TN_ERR_INVALID_VALUE),         # lda < k
    ((0, 4, 4, 4, A, 4, B, 4, C, 3), gt.GEMM_TN_ERR_INVALID_VALUE),         # ldc < n
    ((0, 4, 4, 4, A + 1, 4, B, 4, C, 4), gt.GEMM_TN_ERR_MISALIGNED),
    ((1, 4, 4, 4, A, 4, B, 4, C + 1, 4), gt.GEMM_TN_ERR_MISALIGNED),
    ((0, 4, 4, 4, A, 4, B, 4, A + 8, 4), gt.GEMM_TN_ERR_INVALID_VALUE),     # C overlaps A
    ((0, 4, 4, 4, A, 4, B, 4, B + 30, 4), gt.GEMM_TN_ERR_INVALID_VALUE),    # C overlaps B's last byte
])
def test_validation_rejects_before_any_device_call(lib, args, expected):
    assert gt.gemm_tn_ex(*args, None, None) == expected
    assert gt.gemm_tn_last_error_message() != ""


def test_empty_output_is_a_noop(lib):
    assert gt.gemm_tn_ex(0, 0, 4, 4, None, 4, None, 4, None, 4, None, None) == gt.GEMM_TN_OK
    assert gt.gemm_tn_ex(1, 4, 0, 4, None, 4, None, 4, None, 1, None, None) == gt.GEMM_TN_OK
    assert gt.gemm_tn(1, 0, 0, 0, None, None, None, None) == gt.GEMM_TN_OK


def test_c_adjacent_to_b_is_not_overlap(lib):
    # B spans [B, B + 32) for 4 x 4 fp16; C starting right after it is legal,
    # so validation passes and the call proceeds to the device check.
    rc = gt.gemm_tn_ex(0, 4, 4, 4, A, 4, B, 4, B + 32, 4, None, None)
    assert rc in (gt.GEMM_TN_OK, gt.GEMM_TN_ERR_UNSUPPORTED_DEVICE, gt.GEMM_TN_ERR_CUDA)
    if rc != gt.GEMM_TN_OK:
        assert "C overlaps" not in gt.gemm_tn_last_error_message()


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from dense_tiled_gemm_03_gb300 import _native
    monkeypatch.setattr(_native, "_lib", None)
    monkeypatch.setattr(_native, "LIBRARY_PATH", tmp_path / "libgemm_tn.so")
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _native.library()



def test_split_choice_invariants(lib, monkeypatch):
    """Over a grid of shapes, a split-K choice always has every cluster
    resident at once (GB300 without a device: 76 clusters of 2, 36 of 4, 15 of
    8), at most half the SMs' worth of tiles, and enough k-blocks per CTA (4,
    or 2 in a 4-way split); any other configuration reports no split."""
    monkeypatch.delenv("GEMM_TN_FORCE_CONFIG", raising=False)
    monkeypatch.delenv("GEMM_TN_SPLITK", raising=False)
    resident = {2: 76, 4: 36, 8: 15}
    split_cfgs = {"1cta_n128_splitk", "1cta_decode_splitk"}
    seen = set()
    for m in (1, 8, 32, 33, 128, 200, 256, 512, 1024, 2048):
        for n in (64, 256, 512, 1000, 2048, 4096, 8192):
            for k in (64, 256, 512, 960, 1024, 4096, 16384):
                s = gt.gemm_tn_select_splits(gt.GEMM_TN_BF16, m, n, k)
                cfg = gt.gemm_tn_config_name(gt.gemm_tn_select_config(gt.GEMM_TN_BF16, m, n, k))
                if cfg not in split_cfgs:
                    assert s == 0, (m, n, k, cfg, s)
                    continue
                tiles = -(-m // 128) * -(-n // 128)
                kb = -(-k // 64)
                assert s in resident, (m, n, k, s)
                assert tiles <= resident[s] and 2 * tiles <= 152, (m, n, k, s, tiles)
                min_kb = {2: 4, 4: 4 if m <= 32 else 2, 8: 4}
                assert kb >= min_kb[s] * s, (m, n, k, s, kb)
                seen.add(s)
    assert seen == {2, 4, 8}


def test_split_override_is_reported(lib, monkeypatch):
    monkeypatch.delenv("GEMM_TN_FORCE_CONFIG", raising=False)
    monkeypatch.setenv("GEMM_TN_SPLITK", "2")
    assert gt.gemm_tn_select_splits(gt.GEMM_TN_F16, 128, 1024, 4096) == 2
    monkeypatch.setenv("GEMM_TN_SPLITK", "0")           # off: whole tiles, no split
    assert gt.gemm_tn_select_splits(gt.GEMM_TN_F16, 128, 1024, 4096) == 0
    monkeypatch.delenv("GEMM_TN_SPLITK")
    monkeypatch.setenv("GEMM_TN_FORCE_CONFIG", "1cta_n128_splitk")   # forced: the largest split K allows
    assert gt.gemm_tn_select_splits(gt.GEMM_TN_F16, 4096, 4096, 256) == 4
    assert gt.gemm_tn_select_splits(gt.GEMM_TN_F16, 4096, 4096, 64) == 0


def test_fused_entry_validation(lib):
    ep = gt.GemmTnEpilogue(1.0, 0.0, None, 7, 0)
    assert gt.gemm_tn_fused(0, 4, 4, 4, A, 4, B, 4, C, 4, ep, None, None) == gt.GEMM_TN_ERR_INVALID_VALUE
    assert "activation" in gt.gemm_tn_last_error_message()
    ep = gt.GemmTnEpilogue(1.0, 0.0, None, 0, 5)
    assert gt.gemm_tn_fused(0, 4, 4, 4, A, 4, B, 4, C, 4, ep, None, None) == gt.GEMM_TN_ERR_INVALID_VALUE
    ep = gt.GemmTnEpilogue(1.0, 0.0, None, 0, 1)          # fp32 C must be 4-byte aligned
    assert gt.gemm_tn_fused(0, 4, 4, 4, A, 4, B, 4, C + 2, 4, ep, None, None) == gt.GEMM_TN_ERR_MISALIGNED
    ep = gt.GemmTnEpilogue(1.0, 0.0, A + 2, 0, 0)         # bias must be 4-byte aligned
    assert gt.gemm_tn_fused(0, 4, 4, 4, A, 4, B, 4, C, 4, ep, None, None) == gt.GEMM_TN_ERR_MISALIGNED
    # an fp32 C of 4 x 4 spans 64 bytes: starting 40 bytes before B overlaps it
    ep = gt.GemmTnEpilogue(1.0, 0.0, None, 0, 1)
    assert gt.gemm_tn_fused(0, 4, 4, 4, A, 4, B, 4, B - 40, 4, ep, None, None) == gt.GEMM_TN_ERR_INVALID_VALUE
    assert gt.gemm_tn_fused(0, 4, 4, 4, A, 4, B, 4, C, 4, None, None, None) == gt.GEMM_TN_ERR_INVALID_VALUE
    # an e4m3 C (1-byte elements, any alignment) of 4 x 4 spans 16 bytes:
    # starting 15 bytes before B overlaps it; out_dtype 3 does not exist
    ep = gt.GemmTnEpilogue(1.0, 0.0, None, 0, gt.GEMM_TN_OUT_E4M3)
    assert gt.gemm_tn_fused(0, 4, 4, 4, A, 4, B, 4, B - 15, 4, ep, None, None) == gt.GEMM_TN_ERR_INVALID_VALUE
    assert "overlaps" in gt.gemm_tn_last_error_message()
    assert gt.gemm_tn_fused(0, 4, 4, 4, A, 4, B, 4, C + 1, 3, ep, None, None) == gt.GEMM_TN_ERR_INVALID_VALUE
    ep = gt.GemmTnEpilogue(1.0, 0.0, None, 0, 3)
    assert gt.gemm_tn_fused(0, 4, 4, 4, A, 4, B, 4, C, 4, ep, None, None) == gt.GEMM_TN_ERR_INVALID_VALUE
    assert "output dtype" in gt.gemm_tn_last_error_message()


# flash_attn_fwd (include/flash_attn.h): every argument error is reported
# before any device call. Fake 16-byte-aligned addresses 1 MiB apart; one
# [1, 128, 2, 64] array spans 32 KiB.
QA, KA, VA, OA = 1 << 20, 2 << 20, 3 << 20, 4 << 20


@pytest.mark.parametrize("args, expected", [
    ((2, 1, 128, 2, 64, QA, KA, VA, OA, 0.0, 1), gt.GEMM_TN_ERR_UNSUPPORTED_DTYPE),
    ((0, -1, 128, 2, 64, QA, KA, VA, OA, 0.0, 1), gt.GEMM_TN_ERR_INVALID_VALUE),
    ((0, 1, 128, 2, 32, QA, KA, VA, OA, 0.0, 1), gt.GEMM_TN_ERR_INVALID_VALUE),      # head_dim
    ((0, 1, 128, 2, 256, QA, KA, VA, OA, 0.0, 1), gt.GEMM_TN_ERR_INVALID_VALUE),
    ((0, 1, 128, 2, 64, QA, KA, VA, OA, -0.5, 1), gt.GEMM_TN_ERR_INVALID_VALUE),     # scale
    ((0, 1, 128, 2, 64, QA, KA, VA, OA, float("inf"), 1), gt.GEMM_TN_ERR_INVALID_VALUE),
    ((0, 1, 128, 2, 64, QA, KA, VA, OA, float("nan"), 1), gt.GEMM_TN_ERR_INVALID_VALUE),
    ((0, 1, 128, 2, 64, None, KA, VA, OA, 0.0, 1), gt.GEMM_TN_ERR_INVALID_VALUE),
    ((1, 1, 128, 2, 64, QA, KA, VA, None, 0.0, 0), gt.GEMM_TN_ERR_INVALID_VALUE),
    ((0, 1, 128, 2, 64, QA + 8, KA, VA, OA, 0.0, 1), gt.GEMM_TN_ERR_MISALIGNED),
    ((0, 1, 128, 2, 64, QA, KA, VA, OA + 2, 0.0, 1), gt.GEMM_TN_ERR_MISALIGNED),
    ((0, 1, 128, 2, 64, QA, KA, VA, VA + 32752, 0.0, 1), gt.GEMM_TN_ERR_INVALID_VALUE),   # O overlaps V's end
    ((0, 1, 128, 2, 64, QA, KA, VA, QA - 16, 0.0, 1), gt.GEMM_TN_ERR_INVALID_VALUE),      # O overlaps Q's start
    ((0, 1, 1 << 31, 2, 64, QA, KA, VA, OA, 0.0, 1), gt.GEMM_TN_ERR_INVALID_VALUE),       # seq too long
    ((0, 1 << 20, 1 << 12, 1 << 10, 64, QA, KA, VA, OA, 0.0, 1), gt.GEMM_TN_ERR_INVALID_VALUE),  # grid too large
])
def test_flash_attn_validation_rejects_before_any_device_call(lib, args, expected):
    assert gt.flash_attn_fwd(*args, None, None) == expected
    assert gt.gemm_tn_last_error_message() != ""


def test_flash_attn_empty_sizes_are_noops_and_adjacent_o_is_legal(lib):
    for b, s, h in [(0, 128, 2), (1, 0, 2), (1, 128, 0)]:
        assert gt.flash_attn_fwd(0, b, s, h, 64, None, None, None, None, 0.0, 1, None, None) == gt.GEMM_TN_OK
    # V spans [VA, VA + 32768): O starting right after it passes validation
    rc = gt.flash_attn_fwd(1, 1, 128, 2, 64, QA, KA, VA, VA + 32768, 0.0, 1, None, None)
    assert rc in (gt.GEMM_TN_OK, gt.GEMM_TN_ERR_UNSUPPORTED_DEVICE, gt.GEMM_TN_ERR_CUDA)
    if rc != gt.GEMM_TN_OK:
        assert "overlaps" not in gt.gemm_tn_last_error_message()


def test_multicast_guard_refuses_memory_that_is_not_this_gpus(lib):
    """The multicast configuration may read only device memory of the current
    device: host memory, NULL and unknown addresses are refused (on a machine
    without a GPU every pointer is, since there is no current device)."""
    import numpy as np
    host_a = np.zeros(1 << 16, dtype=np.uint16)
    host_b = np.zeros(1 << 16, dtype=np.uint16)
    assert gt.gemm_tn_multicast_allowed(host_a.ctypes.data, host_b.ctypes.data) == 0
    assert gt.gemm_tn_multicast_allowed(None, None) == 0
    assert gt.gemm_tn_multicast_allowed(A, B) == 0


def test_last_config_after_calls_that_launch_nothing(lib):
    """gemm_tn_last_config reports -1 after a call that launched no GEMM
    kernel: a validation error, an empty problem, or no usable device."""
    assert gt.gemm_tn_ex(5, 4, 4, 4, A, 4, B, 4, C, 4, None, None) == gt.GEMM_TN_ERR_UNSUPPORTED_DTYPE
    assert gt.gemm_tn_last_config() == -1
    assert gt.gemm_tn_ex(0, 0, 4, 4, None, 4, None, 4, None, 4, None, None) == gt.GEMM_TN_OK
    assert gt.gemm_tn_last_config() == -1
    rc = gt.gemm_tn_ex(0, 4, 4, 4, A, 4, B, 4, C, 4, None, None)
    if rc != gt.GEMM_TN_OK:
        assert gt.gemm_tn_last_config() == -1


def test_workspace_pool_queries_without_a_device(lib):
    """Without a usable device there is no workspace pool, and trimming it
    reports an error instead of failing silently."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("checks the no-device answers")
    assert gt.gemm_tn_workspace_pool() is None
    assert gt.gemm_tn_trim_workspace() in (gt.GEMM_TN_ERR_UNSUPPORTED_DEVICE, gt.GEMM_TN_ERR_CUDA)


def test_binding_refuses_a_status_word_it_cannot_hand_to_a_kernel():
    """The kernels write an int through the status pointer: only a contiguous
    int32 tensor on the call's device is passed down."""
    import torch

    from dense_tiled_gemm_03_gb300._native import _status_ptr

    cpu = torch.device("cpu")
    assert _status_ptr(None, cpu) is None
    word = torch.zeros(1, dtype=torch.int32)
    assert _status_ptr(word, cpu) == word.data_ptr()
    with pytest.raises(ValueError):
        _status_ptr(word, torch.device("cuda", 0))                     # host memory for a device call
    with pytest.raises(ValueError):
        _status_ptr(torch.zeros(1, dtype=torch.int64), cpu)             # wrong width
    with pytest.raises(ValueError):
        _status_ptr(torch.zeros(0, dtype=torch.int32), cpu)             # no element
    with pytest.raises(ValueError):
        _status_ptr(torch.zeros(4, dtype=torch.int32)[::2], cpu)        # not contiguous


def test_host_entry_binding_checks_shapes_before_any_device_call():
    """mm_tn_host writes M x N elements into `out`: shapes and dtypes are
    checked before the library (or a device) is touched."""
    import torch

    a = torch.zeros(4, 8, dtype=torch.float16)
    with pytest.raises(ValueError):
        gt.mm_tn_host(a, torch.zeros(5, 7, dtype=torch.float16))        # K differs
    with pytest.raises(TypeError):
        gt.mm_tn_host(a, torch.zeros(5, 8, dtype=torch.bfloat16))       # dtypes differ
    with pytest.raises(ValueError):
        gt.mm_tn_host(a, torch.zeros(5, 8, dtype=torch.float16), out=torch.empty(4, 4, dtype=torch.float16))
    with pytest.raises(ValueError):
        gt.mm_tn_host(a, torch.zeros(5, 8, dtype=torch.float16), out=torch.empty(4, 5, dtype=torch.float32))
    with pytest.raises(ValueError):
        gt.mm_tn_host(a, torch.zeros(5, 8, dtype=torch.float16), out=torch.empty(5, 4, dtype=torch.float16).t())
    with pytest.raises(ValueError):
        gt.mm_tn_host(a[0], torch.zeros(5, 8, dtype=torch.float16))     # not 2-D
