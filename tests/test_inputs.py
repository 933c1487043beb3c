"""The seeded input generator: deterministic, per-head, bf16-exact."""

import numpy as np
import torch

from flashattention_fa_fwd_gb300.inputs import (WORKLOADS, bf16_bits, head_tensor, make_inputs,
                                                round_to_bf16, sample_rows)


def test_round_to_bf16_matches_torch_rne():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 7,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0, 3.0e38, 1e-39],
                                 dtype=np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(round_to_bf16(x), want)
    bits = bf16_bits(round_to_bf16(x))
    back = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(back, want)


def test_generator_is_deterministic_and_per_head():
    w = WORKLOADS["cross_b2_h8_m1000_n3000_d96_peaked"]
    a = head_tensor(w.wid, 1, 5, 64, w.D, w.sigma_qk, w.dtype)
    b = head_tensor(w.wid, 1, 5, 64, w.D, w.sigma_qk, w.dtype)
    np.testing.assert_array_equal(a, b)
    c = head_tensor(w.wid, 1, 6, 64, w.D, w.sigma_qk, w.dtype)
    assert not np.array_equal(a, c)
    assert np.array_equal(round_to_bf16(a), a)               # bf16-exact
    assert 2.0 < a.std() < 4.0                                # sigma 3


def test_make_inputs_heads_subset_matches_full():
    w = WORKLOADS["f32_single_head_m256_n512_d64"]
    q, k, v = make_inputs(w)
    assert q.shape == (1, 1, 256, 64) and k.shape == (1, 1, 512, 64) and q.dtype == np.float32
    q1, k1, v1 = make_inputs(w, heads=[0])
    np.testing.assert_array_equal(q1[0], q[0, 0])
    np.testing.assert_array_equal(v1[0], v[0, 0])


def test_sample_rows_include_edges():
    r = sample_rows(5, 3, 65536, 256)
    assert r.size == 256 and np.all(np.diff(r) > 0)
    for must in (0, 1, 127, 128, 65535):
        assert must in r
    assert sample_rows(5, 3, 10, 256).tolist() == list(range(10))


def test_workload_flops():
    w = WORKLOADS["causal_b8_h32_s4096_d128"]
    assert abs(w.flops - 1.0995e12) / 1.0995e12 < 1e-3
