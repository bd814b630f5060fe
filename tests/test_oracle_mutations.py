"""Planted mistakes in the oracle, each of which one of its pins must catch.

A pin suite that still passes on a wrong oracle pins nothing, so each case
below patches one plausible mistake into `oracle` for the duration of the
test (a wrong rounding rule, a dropped term, a wrong sign or index, a
transposed operand) and requires that a named pin of test_oracle_pins.py
then fails.  The mistakes live only in this file and only on the CPU.  No
GPU.
"""

import importlib.util
import os
import types

import numpy as np

import oracle
from oracle import kivi

_spec = importlib.util.spec_from_file_location("_pins", os.path.join(os.path.dirname(__file__), "test_oracle_pins.py"))
pins = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(pins)


def _numpy_with(**overrides):
    """A stand-in for the numpy module as kivi sees it, with some functions replaced."""
    ns = types.SimpleNamespace(**{k: getattr(np, k) for k in dir(np) if not k.startswith("__")})
    for k, f in overrides.items():
        setattr(ns, k, f)
    return ns


def _patch(monkeypatch, name, fn):
    """Replace an oracle function both where the pins call it and where the oracle does."""
    monkeypatch.setattr(oracle, name, fn, raising=False)
    monkeypatch.setattr(kivi, name, fn)


def _fails(pin, *args):
    try:
        pin(*args)
    except AssertionError:
        return True
    return False


def test_the_pins_pass_on_the_oracle_as_it_is():
    for pin, args in [(pins.test_round_half_even_golden, ()), (pins.test_grid_values_roundtrip_exactly, (2,)),
                      (pins.test_nearest_code_brute_force, (4,)), (pins.test_pack_locations_golden, ()),
                      (pins.test_rope_hand_values_and_relative_position, ()),
                      (pins.test_rope_matches_complex_rotation, ()),
                      (pins.test_attention_all_full_precision_is_textbook, (1,)),
                      (pins.test_attention_query_head_mapping, ()),
                      (pins.test_hadamard_rotate_exact_on_small_integers, ()),
                      (pins.test_dense_sparse_error_bound_and_spike_isolation, ())]:
        assert not _fails(pin, *args), pin.__name__


def test_round_half_up_is_caught(monkeypatch):
    monkeypatch.setattr(kivi, "np", _numpy_with(rint=lambda y: np.floor(y + np.float32(0.5))))
    assert _fails(pins.test_round_half_even_golden)


def test_wrong_scale_is_caught(monkeypatch):
    orig = kivi.quantize_asymmetric

    def scale_over_2b_levels(x, axis, bits):
        c, s, m = orig(x, axis, bits)
        return c, (s * np.float32(2 ** bits - 1) / np.float32(2 ** bits)).astype(np.float32), m

    _patch(monkeypatch, "quantize_asymmetric", scale_over_2b_levels)
    assert _fails(pins.test_grid_values_roundtrip_exactly, 2)


def test_dropped_min_term_is_caught(monkeypatch):
    _patch(monkeypatch, "dequantize", lambda codes, scale, mn: codes.astype(np.float64) * np.asarray(scale, np.float64))
    assert _fails(pins.test_grid_values_roundtrip_exactly, 4)


def test_reflected_codes_are_caught(monkeypatch):
    orig = kivi.quantize_asymmetric

    def reflected(x, axis, bits):
        c, s, m = orig(x, axis, bits)
        return ((2 ** bits - 1) - c).astype(np.uint8), s, m

    _patch(monkeypatch, "quantize_asymmetric", reflected)
    assert _fails(pins.test_nearest_code_brute_force, 2)


def test_transposed_bit_fields_are_caught(monkeypatch):
    def swapped(row, col, bits, rows, cols):
        # the fields of the two channel octets (j) and of the two channels of
        # a pair (e) trade places
        nu = 8 // bits
        mt, h, g = row // 16, (row // 8) % 2, row % 8
        kt, j, q, e = col // 16, (col // 8) % 2, (col % 8) // 2, col % 2
        tau = 2 * (mt % 2) + h
        w = ((mt // 2) * (cols // 16) + kt) * (4 // nu) + tau // nu
        word_byte = ((w // 4) * 32 + 4 * g + q) * 16 + (w % 4) * 4
        bit = 16 * j + 8 * e + bits * (tau % nu)
        return word_byte + bit // 8, bit % 8

    _patch(monkeypatch, "code_location", swapped)
    monkeypatch.setattr(kivi, "_LOC_CACHE", {})
    assert _fails(pins.test_pack_locations_golden)


def test_rope_turning_the_wrong_way_is_caught(monkeypatch):
    orig = kivi.rope_rotate
    _patch(monkeypatch, "rope_rotate",
           lambda x, positions, theta=10000.0: orig(x, -np.asarray(positions, np.int64), theta))
    assert _fails(pins.test_rope_hand_values_and_relative_position)


def test_rope_on_adjacent_channel_pairs_is_caught(monkeypatch):
    orig = kivi.rope_rotate
    # channel 2i <-> slot i, 2i + 1 <-> slot i + 64: the rotation then pairs
    # adjacent channels instead of (i, i + 64)
    perm = np.concatenate([np.arange(0, 128, 2), np.arange(1, 128, 2)])
    inv = np.argsort(perm)

    def adjacent(x, positions, theta=10000.0):
        x = np.asarray(x)
        return orig(x[..., perm], positions, theta)[..., inv]

    _patch(monkeypatch, "rope_rotate", adjacent)
    assert _fails(pins.test_rope_matches_complex_rotation)


def test_missing_softmax_scale_is_caught(monkeypatch):
    orig = kivi.dense_attention
    _patch(monkeypatch, "dense_attention", lambda q, K, V, scale: orig(q, K, V, 1.0))
    assert _fails(pins.test_attention_all_full_precision_is_textbook, 0)


def test_wrong_query_head_mapping_is_caught(monkeypatch):
    orig = kivi.OracleCache.keys_values
    monkeypatch.setattr(kivi.OracleCache, "keys_values", lambda self, s, h: orig(self, s, (h + 1) % self.H))
    assert _fails(pins.test_attention_query_head_mapping)


def test_reversed_hadamard_input_is_caught(monkeypatch):
    orig = kivi.hadamard_rotate
    _patch(monkeypatch, "hadamard_rotate", lambda x: orig(np.asarray(x)[..., ::-1]))
    assert _fails(pins.test_hadamard_rotate_exact_on_small_integers)


def test_smallest_element_as_outlier_is_caught(monkeypatch):
    monkeypatch.setattr(kivi, "np", _numpy_with(argmax=np.argmin))
    assert _fails(pins.test_dense_sparse_error_bound_and_spike_isolation)
