"""The C ABI library builds, loads and exports every symbol fattn.h declares,
and rejects bad arguments on the host (no compute call needs a GPU here)."""
import ctypes
import os
import re

import pytest

import exact_attention_11_gb300 as fa
from exact_attention_11_gb300 import _build

HEADER = os.path.join(_build.INCLUDE, "fattn.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fa_forward", "fa_forward_fp32", "fa_backward", "fa_paged_decode", "fa_status_string",
              "fa_device_status", "fa_release", "fa_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in fattn.h but not exported"
        assert name in fa.EXPORTS, f"{name} has no Python binding"


def test_version_and_status_strings(lib):
    assert lib.fa_version() == 10000
    assert fa.fa_status_string(0) == "ok"
    for code in range(-7, 0):
        assert fa.fa_status_string(code) != "unknown status"


NULL = None
P = 4096  # a 16-byte-aligned fake address: never dereferenced on these paths


@pytest.mark.parametrize("args,expect", [
    ((NULL, P, P, P, NULL, 1, 1, 64, 64, 0.125, 0), -1),      # null q
    ((P, P, P, P, NULL, -1, 1, 64, 64, 0.125, 0), -1),        # negative B
    ((P, P, P, P, NULL, 1, 1, 64, 96, 0.125, 0), -2),         # d not 64/128/256
    ((P, P, P, P, NULL, 1, 1, 64, 512, 0.125, 0), -2),        # d = 512
    ((P, P, P, P, NULL, 1, 1, 64, 64, 0.0, 0), -1),           # scale 0
    ((P, P, P, P, NULL, 1, 1, 64, 64, float("nan"), 0), -1),  # scale NaN
    ((P + 2, P, P, P, NULL, 1, 1, 64, 64, 0.125, 0), -3),     # misaligned q
    ((P, P, P, P, P + 4, 1, 1, 64, 64, 0.125, 0), -3),        # misaligned lse
    ((P, P, P, P, NULL, 0, 1, 64, 64, 0.125, 0), 0),          # empty batch: no-op
    ((P, P, P, P, NULL, 1, 1, 0, 64, 0.125, 0), 0),           # N = 0: no-op
])
def test_forward_argument_checks(lib, args, expect):
    for fn in (lib.fa_forward, lib.fa_forward_f16, lib.fa_forward_fp32):
        assert fn(*args, None) == expect


@pytest.mark.parametrize("args,expect", [
    ((NULL, P, P, P, P, P, 1, 1, 128, 16, 4, 0.1), -1),       # null q
    ((P, P, P, P, P, P, 1, 1, 64, 16, 4, 0.1), -2),           # head_size 64
    ((P, P, P, P, P, P, 1, 1, 128, 32, 4, 0.1), -2),          # block_size 32
    ((P, P, P, P, P, P, 1, 0, 128, 16, 4, 0.1), -1),          # no heads
    ((P, P, P, P, P, P, 1, 1, 128, 16, 0, 0.1), -1),          # no block-table columns
    ((P, P + 8, P, P, P, P, 1, 1, 128, 16, 4, 0.1), -3),      # misaligned k_cache
    ((P, P, P, P, P, P, 0, 1, 128, 16, 4, 0.1), 0),           # no sequences: no-op
])
def test_decode_argument_checks(lib, args, expect):
    assert lib.fa_paged_decode(*args, None) == expect
    # the grouped-head entry point with one key/value head per query head
    S, H = args[6], args[7]
    gargs = args[:8] + (H,) + args[8:]
    assert lib.fa_paged_decode_gqa(*gargs, None) == expect


@pytest.mark.parametrize("impl,H,Hk,expect", [
    (0, 8, 0, -1),     # no key/value heads
    (0, 8, 3, -1),     # does not divide
    (0, 12, 4, 0),     # group of 3: tensor-core kernel
    (0, 24, 4, 0),     # group of 6
    (0, 36, 2, -2),    # group of 18: neither kernel
    (0, 17, 1, -2),    # group of 17
    (0, 40, 2, 0),     # group of 20: CUDA-core kernel (multiple of 4)
    (0, 8, 4, 0),      # group of 2: valid (no sequences: no-op)
    (0, 32, 4, 0),     # group of 8
    (0, 64, 1, 0),     # multi-query
    (1, 12, 4, -2),    # CUDA-core only: group of 3 is not built
    (1, 24, 4, -2),    # group of 6
    (1, 32, 4, 0),     # group of 8
    (1, 64, 1, 0),     # multi-query
    (2, 12, 4, 0),     # tensor-core only: group of 3
    (2, 40, 2, -2),    # group of 20 is not a multiple of 16
    (2, 64, 2, 0),     # group of 32: two slices of 16
    (2, 8, 8, 0),      # group 1 is the one-head decode whatever the choice
])
def test_gqa_decode_group_checks(lib, impl, H, Hk, expect):
    assert lib.fa_decode_gqa_select(impl) == 0
    try:
        assert lib.fa_paged_decode_gqa(P, P, P, P, P, P, 0, H, Hk, 128, 16, 4, 0.1, None) == expect
    finally:
        lib.fa_decode_gqa_select(0)


def test_gqa_select_rejects_unknown(lib):
    assert lib.fa_decode_gqa_select(3) == -1
    assert lib.fa_decode_gqa_select(-1) == -1


W = 1 << 20  # a workspace size larger than any case below needs


@pytest.mark.parametrize("args,expect", [
    ((NULL, P, P, P, P, P, P, P, P, 1, 1, 64, 64, 0.125, 0, P, W), -1),     # null q
    ((P, P, P, P, NULL, P, P, P, P, 1, 1, 64, 64, 0.125, 0, P, W), -1),     # null dout
    ((P, P, P, P, P, NULL, P, P, P, 1, 1, 64, 64, 0.125, 0, P, W), -1),     # null lse
    ((P, P, P, P, P, P, P, P, NULL, 1, 1, 64, 64, 0.125, 0, P, W), -1),     # null dv
    ((P, P, P, P, P, P, P, P, P, 1, 1, 64, 96, 0.125, 0, P, W), -2),        # d not 64/128
    ((P, P, P, P, P, P, P, P, P, 1, 1, 64, 64, -1.0, 0, P, W), -1),         # negative scale
    ((P, P, P, P, P + 2, P, P, P, P, 1, 1, 64, 64, 0.125, 0, P, W), -3),    # misaligned dout
    ((P, P, P, P, P, P, P + 8, P, P, 1, 1, 64, 64, 0.125, 0, P, W), -3),    # misaligned dq
    ((P, P, P, P, P, P, P, P, P, 1, 1, 64, 64, 0.125, 0, NULL, W), -1),     # no workspace
    ((P, P, P, P, P, P, P, P, P, 1, 1, 64, 64, 0.125, 0, P + 4, W), -3),    # misaligned workspace
    ((P, P, P, P, P, P, P, P, P, 1, 1, 64, 64, 0.125, 0, P, 4 * 128 * 66 - 1), -1),  # one byte short
    ((P, P, P, P, P, P, P, P, P, 0, 1, 64, 64, 0.125, 0, NULL, 0), 0),      # empty batch: no-op
    ((P, P, P, P, P, P, P, P, P, 1, 1, 0, 64, 0.125, 0, NULL, 0), 0),       # N = 0: no-op
])
def test_backward_argument_checks(lib, args, expect):
    assert lib.fa_backward(*args, None) == expect


def test_backward_workspace_size(lib):
    # fp32 dQ accumulator over N rounded up to 128, then two vectors per 128-query block
    assert lib.fa_backward_workspace_bytes(2, 3, 100, 128) == 4 * 2 * 3 * 128 * 130
    assert lib.fa_backward_workspace_bytes(1, 1, 64, 64) == 4 * 128 * 66
    assert lib.fa_backward_workspace_bytes(1, 2, 129, 64) == 4 * 2 * 256 * 66
    assert lib.fa_backward_workspace_bytes(-1, 1, 64, 64) == 0
    assert fa.fa_backward_workspace_bytes(0, 4, 64, 64) == 0


@pytest.mark.parametrize("mask,stride,N,expect", [
    (NULL, 0, 64, -1),       # no mask
    (P, -16, 64, -1),        # negative stride
    (P + 8, 0, 64, -3),      # misaligned mask
    (P, 8, 64, -3),          # stride not a multiple of 16
    (P, 0, 40, -2),          # N not a multiple of 16
    (P, 0, 0, 0),            # N = 0: no-op
])
def test_masked_forward_argument_checks(lib, mask, stride, N, expect):
    assert lib.fa_forward_masked(P, P, P, P, NULL, mask, stride, 1, 1, N, 64, 0.125, None) == expect


def test_head_dim_256_is_forward_only(lib):
    """d = 256 is served by fa_forward and fa_forward_f16 only."""
    assert lib.fa_forward_masked(P, P, P, P, NULL, P, 0, 1, 1, 64, 256, 0.1, None) == -2
    assert lib.fa_forward_fp32(P, P, P, P, NULL, 1, 1, 64, 256, 0.1, 0, None) == -2
    assert lib.fa_backward(P, P, P, P, P, P, P, P, P, 1, 1, 64, 256, 0.1, 0, P, 1 << 30,
                           None) == -2
    assert lib.fa_forward(P, P, P, P, NULL, 0, 1, 64, 256, 0.1, 1, None) == 0   # empty: no-op


QW = 4 * 2 * 3          # workspace of fa_quantize_fp8 for B=2, H=3, N <= 128


@pytest.mark.parametrize("args,expect", [
    ((NULL, P, P, NULL, P, P, P, P, P, P, 2, 3, 100, 128, P, QW), -1),    # null q
    ((P, P, P, NULL, P, P, NULL, P, P, P, 2, 3, 100, 128, P, QW), -1),    # null vt8
    ((P, P, P, NULL, P, P, P, P, P, NULL, 2, 3, 100, 128, P, QW), -1),    # null v_scale
    ((P, P, P, NULL, P, P, P, P, P, P, 2, 3, 100, 64, P, QW), -2),        # d = 64
    ((P, P, P, P + 4, P, P, P, P, P, P, 2, 3, 100, 128, P, QW), -3),      # misaligned signs
    ((P, P, P, NULL, P + 8, P, P, P, P, P, 2, 3, 100, 128, P, QW), -3),   # misaligned q8
    ((P, P, P, NULL, P, P, P, P, P, P, 2, 3, 100, 128, NULL, QW), -1),    # no workspace
    ((P, P, P, NULL, P, P, P, P, P, P, 2, 3, 100, 128, P, QW - 1), -1),   # one byte short
    ((P, P, P, NULL, P, P, P, P, P, P, 2, 3, 100, 128, P + 2, QW), -3),   # misaligned workspace
    ((P, P, P, NULL, P, P, P, P, P, P, 300, 300, 100, 128, P, 1 << 40), -2),  # B*H > 65535
    ((P, P, P, NULL, P, P, P, P, P, P, -1, 3, 100, 128, P, QW), -1),      # negative B
    ((P, P, P, NULL, P, P, P, P, P, P, 0, 3, 100, 128, NULL, 0), 0),      # empty: no-op
])
def test_quantize_fp8_argument_checks(lib, args, expect):
    assert lib.fa_quantize_fp8(*args, None) == expect


def test_quantize_fp8_sizes(lib):
    # one fp32 block maximum per 128 rows of V
    assert lib.fa_quantize_fp8_workspace_bytes(2, 3, 100, 128) == 4 * 2 * 3
    assert lib.fa_quantize_fp8_workspace_bytes(2, 3, 129, 128) == 4 * 2 * 3 * 2
    assert lib.fa_quantize_fp8_workspace_bytes(-1, 3, 100, 128) == 0
    assert [lib.fa_fp8_vt_stride(n) for n in (1, 16, 17, 4096, -3)] == [16, 16, 32, 4096, 0]


@pytest.mark.parametrize("args,expect", [
    ((P, P, P, NULL, P, P, P, NULL, 1, 1, 64, 128, 0.1, 0), -1),          # null q_scale
    ((P, P, P, P, P, P, P, NULL, 1, 1, 64, 64, 0.1, 0), -2),              # d = 64
    ((P, P, P + 8, P, P, P, P, NULL, 1, 1, 64, 128, 0.1, 0), -3),         # misaligned vt8
    ((P, P, P, P, P, P, P, NULL, 1, 1, 64, 128, 0.0, 0), -1),             # zero scale
    ((P, P, P, P, P, P, P, NULL, 1, 1, 0, 128, 0.1, 1), 0),               # N = 0: no-op
])
def test_forward_fp8_argument_checks(lib, args, expect):
    assert lib.fa_forward_fp8(*args, None) == expect


def test_valid_call_without_gpu_fails_loudly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = lib.fa_forward(P, P, P, P, None, 1, 1, 64, 64, 0.125, 0, None)
    assert rc == -7  # FA_ERR_NO_DEVICE: never a silent CPU path
    with pytest.raises(fa.FattnError):
        fa.fa_forward(P, P, P, P, None, 1, 1, 64, 64, 0.125, 0, None)
    rc = lib.fa_backward(P, P, P, P, P, P, P, P, P, 1, 1, 64, 64, 0.125, 0, P, W, None)
    assert rc == -7
    assert lib.fa_quantize_fp8(P, P, P, NULL, P, P, P, P, P, P, 1, 1, 64, 128, P, 4, None) == -7
    assert lib.fa_forward_fp8(P, P, P, P, P, P, P, NULL, 1, 1, 64, 128, 0.1, 0, None) == -7


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(fa, "_LIB_PATH", str(tmp_path / "libfattn.so"))
    monkeypatch.setattr(fa, "_lib", None)
    with pytest.raises(RuntimeError, match="not found"):
        fa.load()
