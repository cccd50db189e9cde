"""The FP8 part of the oracle against its pins, and plausible mistakes planted
in copies of it (on the CPU), each of which some pin must catch."""
import importlib.util
import os
import sys
import types

import pytest

import fp8_pins
import oracle.fp8 as fp8

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


@pytest.mark.parametrize("check", fp8_pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_fp8_oracle_pin(check):
    check(fp8)


MUTANTS = [
    ("ties_away_from_zero", "r = np.round(a / quantum) * quantum",
     "r = np.floor(a / quantum + 0.5) * quantum"),
    ("four_mantissa_bits", "(e - 3).astype(np.int64)", "(e - 4).astype(np.int64)"),
    ("no_subnormals", "e = np.maximum(ex - 1, -6)", "e = ex - 1"),
    ("no_saturation", "r = np.minimum(r, E4M3_MAX)", "r = r"),
    ("butterfly_sign", "y = np.stack([a + b, a - b], axis=-2)", "y = np.stack([a + b, b - a], axis=-2)"),
    ("butterfly_halves_swapped", "a, b = z[..., 0, :], z[..., 1, :]",
     "a, b = z[..., 1, :], z[..., 0, :]"),
    ("signs_ignored", "y = _f32(x) * _f32(signs)", "y = _f32(x)"),
    ("rotation_factor_dropped", "(s * _rotation_factor(d)).astype(np.float32) if signs",
     "s if signs"),
    ("scale_from_max_not_amax", "s = _scale_of(np.abs(x32[:, :, sl]).max(axis=(2, 3)))",
     "s = _scale_of(x32[:, :, sl].max(axis=(2, 3)))"),
    ("scale_divides_by_256", "s = amax / np.float32(E4M3_MAX)", "s = amax / np.float32(256.0)"),
    ("blocks_of_64_rows", "BLOCK_ROWS = 128", "BLOCK_ROWS = 64"),
    ("v_rotated_too", "vc, vs = quantize_heads(v)",
     "vc, vs = quantize_heads(v if signs is None else hadamard_rows(v, signs))"),
    ("v_per_block", "vc, vs = quantize_heads(v)\n    return dequantize_rows(qc, qs), dequantize_rows(kc, ks), vc * vs[:, :, None, None].astype(np.float64)",
     "vc, vs = quantize_rows(v)\n    return dequantize_rows(qc, qs), dequantize_rows(kc, ks), dequantize_rows(vc, vs)"),
    ("bound_without_v", "bound[b, h] = (w @ np.abs(vd[b, h])) / l", "bound[b, h] = w.sum(axis=1, keepdims=True) / l * 0.25"),
    ("weight_bound_kernel_specific", "P_ABS = 2.0 ** -10", "P_ABS = 2.0 ** -14"),
    ("weight_bound_relative_too_tight", "P_REL = 2.0 ** -4", "P_REL = 2.0 ** -5"),
    ("sigma_without_third", "var[b, h] = ((w * w / 3.0) @ (vd[b, h] ** 2)) / (l * l)",
     "var[b, h] = ((w * w) @ (vd[b, h] ** 2)) / (l * l) * 9.0"),
]


def _load_variant(src: str, name: str) -> types.ModuleType:
    mod = types.ModuleType(f"fp8_mutant_{name}")
    mod.__file__ = fp8.__file__
    exec(compile(src, f"<fp8 mutant {name}>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_fp8_mutant_is_caught(name, find, repl):
    with open(fp8.__file__) as fh:
        src = fh.read()
    assert src.count(find) == 1, f"mutation site for {name} not unique"
    mod = _load_variant(src.replace(find, repl), name)
    failed = []
    for check in fp8_pins.ALL_CHECKS:
        try:
            check(mod)
        except (AssertionError, ValueError, IndexError):
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
