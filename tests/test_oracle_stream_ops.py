"""Pins of the stream value rotation ("Speculative Streaming" Eq. 7,
V_tn = V_t e^{i eps n}) and of the ConFu future-token hand-off ("ConFu"
key design 1: the contemplate token of the last accepted node).

* rotation by 0 is the identity; every (re, im) pair keeps its modulus;
* the rotation equals numpy's complex multiplication by exp(1j eps s);
* stream s equals stream 1's rotation applied s times (angles add);
* only stream rows change; node rows and padding are untouched;
* the gather picks row T + last_node of every request.
"""

import numpy as np
import pytest

import oracle


def _vb(seed, B=2, H=3, R=40, d=8):
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.standard_normal((B, H, R, d))


@pytest.mark.parametrize("seed", [0, 1])
def test_rotation_identity_and_modulus(seed):
    vb = _vb(seed)
    n = np.array([5, 9])
    gamma = 3
    same = oracle.rotate_stream_values(vb, n, gamma, 0.0)
    for b in range(2):
        T = n[b]
        for j in range(T):
            for s in range(1, gamma + 1):
                assert np.array_equal(same[b, :, T + j * gamma + s - 1], vb[b, :, j])
    rot = oracle.rotate_stream_values(vb, n, gamma, 0.37)
    for b in range(2):
        T = n[b]
        for j in range(T):
            r = T + j * gamma
            m0 = vb[b, :, j, 0::2] ** 2 + vb[b, :, j, 1::2] ** 2
            m1 = rot[b, :, r, 0::2] ** 2 + rot[b, :, r, 1::2] ** 2
            np.testing.assert_allclose(m0, m1, rtol=1e-12)


def test_rotation_is_complex_multiplication():
    vb = _vb(3)
    n, gamma, eps = np.array([4, 6]), 3, 0.21
    rot = oracle.rotate_stream_values(vb, n, gamma, eps)
    for b in range(2):
        T = n[b]
        for j in range(T):
            z = vb[b, :, j, 0::2] + 1j * vb[b, :, j, 1::2]
            for s in range(1, gamma + 1):
                w = z * np.exp(1j * eps * s)
                r = T + j * gamma + s - 1
                np.testing.assert_allclose(rot[b, :, r, 0::2], w.real, atol=1e-12)
                np.testing.assert_allclose(rot[b, :, r, 1::2], w.imag, atol=1e-12)


def test_rotation_angles_add_and_other_rows_untouched():
    vb = _vb(4)
    n, gamma, eps = np.array([3, 7]), 4, 0.13
    rot = oracle.rotate_stream_values(vb, n, gamma, eps)
    for b in range(2):
        T = n[b]
        for j in range(T):
            # rotate stream 1 by eps again (s - 1) times
            cur = rot[b, :, T + j * gamma].copy()
            for s in range(2, gamma + 1):
                c, sn = np.cos(eps), np.sin(eps)
                re, im = cur[:, 0::2].copy(), cur[:, 1::2].copy()
                cur[:, 0::2], cur[:, 1::2] = re * c - im * sn, re * sn + im * c
                np.testing.assert_allclose(rot[b, :, T + j * gamma + s - 1], cur, atol=1e-12)
        untouched = list(range(T)) + list(range(T * (1 + gamma), vb.shape[2]))
        assert np.array_equal(rot[b][:, untouched], vb[b][:, untouched])


def test_future_gather():
    rng = np.random.Generator(np.random.PCG64(5))
    o = rng.standard_normal((3, 20, 4, 8))
    last = np.array([0, 7, 9])
    f = oracle.future_gather(o, last, 10)
    assert f.shape == (3, 4, 8)
    for b, r in enumerate([10, 17, 19]):
        assert np.array_equal(f[b], o[b, r])
