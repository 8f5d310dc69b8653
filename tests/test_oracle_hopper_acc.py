"""Pins for the limited-precision accumulation emulator (CPU only).

The emulator (oracle/hopper_acc.py) restates the pages' description of H800
FP8 accumulation: right-shift alignment to the larger exponent, about 14
retained bits ("Deepseek - Not For everyone", paragraph 5; dssusan.co.kr post
91437, paragraph 2), and promotion to FP32 at a fixed K interval (dssusan
post, paragraph 3).  It is pinned against closed forms, not against hardware.
"""
import math

import numpy as np

from fp8_fine_grained_amax_gb300 import synth
from oracle import hopper_acc


def test_hand_worked_alignment():
    # 1 + 2^-4 with 4 bits: the grid at exponent 0 is 2^-3, the small addend
    # truncates to zero; with 5 bits the grid is 2^-4 and it survives
    assert hopper_acc.add_aligned(1.0, 0.0625, 4) == 1.0
    assert hopper_acc.add_aligned(1.0, 0.0625, 5) == 1.0625
    # truncation is toward zero, not downward
    assert hopper_acc.add_aligned(1.0, -0.0625, 4) == 1.0
    assert hopper_acc.add_aligned(0.0, -0.0625, 4) == -0.0625
    # the larger operand sets the grid: 3 bits at exponent 2 -> grid 1
    assert hopper_acc.add_aligned(4.75, 1.5, 3) == 5.0
    assert hopper_acc.add_aligned(0.0, 0.0, 14) == 0.0


def test_swamping_closed_form():
    # 1 followed by 4096 additions of 2^-14 with 14 bits: the grid at exponent 0
    # is 2^-13, every addend truncates to zero (exact sum 1.25)
    a = np.concatenate([[1.0], np.full(4096, 2.0 ** -14)])[None, :]
    b = np.ones_like(a)
    assert hopper_acc.limited_acc_dot(a, b, 14)[0] == 1.0
    # promotion every 128 products keeps each block's small addends: the
    # first block holds the 1 (its 127 small addends are lost), the 32 later
    # blocks sum to 128 * 2^-14 exactly, except the last one (1 addend short)
    got = hopper_acc.limited_acc_dot(a, b, 14, n_c=128)[0]
    assert got == np.float32(1.0) + np.float32(4096 - 127) * np.float32(2.0 ** -14)


def test_unlimited_bits_is_the_exact_sum(oracle):
    # decoded E4M3 codes (no scales): products are multiples of 2^-18 below
    # 2^18, so every partial sum of 300 of them is exact in a double; with 53
    # bits the alignment grid is never coarser than 2^-18, nothing is truncated
    # and the emulator returns the exact sum
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 256, (2, 16, 300)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0  # no NaN codes
    a, b = oracle.e4m3_decode(codes[0]), oracle.e4m3_decode(codes[1])
    want = np.array([math.fsum(r) for r in a * b])
    assert np.array_equal(hopper_acc.limited_acc_dot(a, b, 53), want)


def test_promotion_every_product_is_fp32_sequential_sum(oracle):
    # FP8 x FP8 products have at most 8 significant bits, so with 24 bits the
    # partial of a single product is exact and each promotion is one FP32 add
    x = synth.activation(8, 512, seed=9)
    w = synth.weight(8, 512, seed=10)
    qa, sa = oracle.quant_act(x)
    qb, _ = oracle.quant_act(w)
    a = oracle.e4m3_decode(qa)
    b = oracle.e4m3_decode(qb)
    want = np.zeros(8, np.float32)
    for k in range(512):
        want = want + (a[:, k] * b[:, k]).astype(np.float32)
    assert np.array_equal(hopper_acc.limited_acc_dot(a, b, 24, n_c=1), want.astype(np.float64))


def test_promotion_bounds_the_error(oracle):
    # context, with a property that must hold: on K = 4096 FP8 dot products,
    # 14-bit accumulation over the whole K loses far more than 14-bit partial
    # sums promoted to FP32 every 128 products
    K = 4096
    x = synth.activation(64, K, seed=11)
    w = synth.weight(64, K, seed=12)
    a = oracle.e4m3_decode(oracle.quant_act(x)[0])
    b = oracle.e4m3_decode(oracle.quant_act(w)[0])
    exact = np.sum(a * b, axis=1)
    absdot = np.sum(np.abs(a * b), axis=1)
    e_full = np.abs(hopper_acc.limited_acc_dot(a, b, 14) - exact) / absdot
    e_prom = np.abs(hopper_acc.limited_acc_dot(a, b, 14, n_c=128) - exact) / absdot
    assert np.max(e_prom) < np.max(e_full) / 4
    assert np.max(e_prom) < 1e-3
