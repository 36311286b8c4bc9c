"""Pins of the oracle's e4m3 decoding (the only arithmetic the FP8 forward's
oracle adds to the plain one): code points fixed by the OCP FP8 E4M3
definition, and every one of the 256 codes against torch's float8_e4m3fn."""
import math

import numpy as np
import pytest
import torch

import oracle


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x38, 1.0), (0xB8, -1.0), (0x40, 2.0), (0x3C, 1.5), (0x7E, 448.0),
    (0xFE, -448.0), (0x08, 2.0 ** -6), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9),
    (0x30, 0.5), (0x77, 240.0)])
def test_code_points_from_the_format_definition(code, value):
    assert oracle.e4m3_to_f64(np.array([code], np.uint8))[0] == value


def test_nan_codes():
    v = oracle.e4m3_to_f64(np.array([0x7F, 0xFF], np.uint8))
    assert np.isnan(v).all()


def test_all_codes_match_torch_float8_e4m3fn():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_to_f64(codes.numpy())
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_tensor_input_keeps_its_shape_and_round_trips():
    x = torch.randn(3, 5, 7)
    q8 = x.to(torch.float8_e4m3fn).view(torch.uint8)
    got = oracle.e4m3_to_f64(q8)
    assert got.shape == (3, 5, 7)
    assert np.array_equal(got, x.to(torch.float8_e4m3fn).double().numpy())


def test_fp8_forward_is_the_plain_forward_of_the_decoded_values():
    g = torch.Generator().manual_seed(0)
    q8, k8, v8 = (torch.randn(1, 2, 9, 4, generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
                  for _ in range(3))
    o, l = oracle.fwd_fp8(q8, k8, v8, 0.5, 0.25, 2.0, 0.3, True)
    o0, l0 = oracle.fwd(oracle.e4m3_to_f64(q8) * 0.5, oracle.e4m3_to_f64(k8) * 0.25,
                        oracle.e4m3_to_f64(v8) * 2.0, 0.3, True)
    assert np.array_equal(o, o0) and np.array_equal(l, l0)
