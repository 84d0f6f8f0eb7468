"""The seeded input generator: determinism, rounding and distribution."""

from __future__ import annotations

import numpy as np

import fa_inputs as fi


def test_splitmix64_reference_values():
    # SplitMix64 with state 0: the first outputs of the published generator
    # (next() adds the golden gamma, then mixes) are these well-known values.
    z = np.array([0, 1, 2], dtype=np.uint64)
    with np.errstate(over="ignore"):
        out = fi._mix64((z + np.uint64(1)) * fi._PHI)
    assert [int(x) for x in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_seed_dependent():
    a = fi.make_custom(1, 2, 33, 8, seed=5)
    b = fi.make_custom(1, 2, 33, 8, seed=5)
    c = fi.make_custom(1, 2, 33, 8, seed=6)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert not np.array_equal(a[0], c[0])


def test_q_k_v_streams_are_consecutive_counters():
    w = fi.AttentionWorkload("t", 1, 1, 4, 8, False, 1.0, 9)
    q, k, v = fi.make_qkv(w)
    z = fi.normal_variates(9, 0, 3 * w.n_elem)
    assert np.array_equal(q.ravel(), fi.round_to_bf16_bits(z[:32]))
    assert np.array_equal(k.ravel(), fi.round_to_bf16_bits(z[32:64]))
    assert np.array_equal(v.ravel(), fi.round_to_bf16_bits(z[64:]))


def test_rows_regenerate_bit_exactly():
    w = fi.WORKLOADS["single_head_L128_d64"]
    q, k, v = fi.make_qkv(w)
    rows = np.array([0, 1, 77, 127])
    qr, kr, vr = fi.make_qkv_rows(w, 0, rows)
    assert np.array_equal(qr, q[0, 0, rows])
    assert np.array_equal(kr, k[0, 0, rows])
    assert np.array_equal(vr, v[0, 0, rows])


def test_odd_start_offsets_match():
    z = fi.normal_variates(3, 0, 101)
    for s in (1, 2, 7, 50):
        assert np.array_equal(fi.normal_variates(3, s, 101 - s), z[s:])
    assert np.array_equal(fi.normal_at(3, np.arange(101, dtype=np.uint64)), z)


def test_bf16_round_to_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -7, -2.5,
                     1.0 + 2 ** -8 + 2 ** -20, 0.0, -0.0, np.inf], dtype=np.float32)
    bits = fi.round_to_bf16_bits(vals)
    back = fi.bf16_bits_to_float32(bits)
    # 1 + 2^-8 is a tie -> even (1.0); 1 + 3*2^-8 is a tie -> even (1 + 2^-6)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.0 + 2 ** -6
    assert back[3] == 1.0 + 2 ** -7 and back[4] == -2.5
    assert back[5] == 1.0 + 2 ** -7   # just above the tie rounds up
    assert back[6] == 0.0 and np.signbit(back[7]) and np.isinf(back[8])
    assert fi.round_to_bf16_bits(np.array([np.nan], np.float32))[0] == 0x7FC0


def test_distribution_moments():
    z = fi.normal_variates(42, 0, 1 << 18)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert abs((z ** 4).mean() - 3.0) < 0.05


def test_workload_table():
    w = fi.WORKLOADS
    assert w["B4_H8_L1024_d64"].flops == 4 * 4 * 8 * 1024 ** 2 * 64
    assert w["B2_H16_L4096_d128_causal"].flops == 2 * 2 * 16 * 4096 ** 2 * 128
    assert w["B1_H32_L16384_d128_causal_qk3"].q_std == 3.0
    assert w["B1_H32_L16384_d128_causal_qk3"].v_std == 1.0
    assert [x.seed for x in w.values()] == [42, 43, 44, 45, 46, 47]


def test_grad_out_follows_v_in_the_same_stream():
    from fa_inputs import (AttentionWorkload, make_grad_out, make_grad_out_rows,
                           normal_variates, round_to_bf16_bits)
    w = AttentionWorkload("t", 2, 3, 50, 8, False, 1.0, 9)
    do = make_grad_out(w)
    n = w.n_elem
    expect = round_to_bf16_bits(normal_variates(9, 3 * n, n)).reshape(do.shape)
    assert np.array_equal(do, expect)
    rows = np.array([0, 7, 49])
    assert np.array_equal(make_grad_out_rows(w, 4, rows), do.reshape(6, 50, 8)[4][rows])
