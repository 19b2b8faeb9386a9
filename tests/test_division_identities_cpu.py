"""Exactness of the multiply-high divisions the kernels use instead of an
integer divide (CPU: the identities themselves, over the kernels' ranges).

token_sort_kernel: t = floor(p / k) as (p * ceil(2^32 / k)) >> 32 for every
pair index p < 2^16 and choice count k <= 2^16.
grouped_gemm_kernel: the scale/zero group of element offset k0 as
umulhi(k0, ceil(2^32 / g)) (32-bit constant) for group sizes g that are
multiples of 32 up to 8192 and offsets up to 2 * 8192."""
import numpy as np


def test_pair_token_division_is_exact():
    p = np.arange(0, 65537, dtype=np.uint64)
    for k in list(range(1, 65)) + [96, 127, 128, 255, 256, 1000, 4096, 65535, 65536]:
        m = np.uint64((2**32 + k - 1) // k)  # fits in 33 bits: 64-bit product below 2^49
        t = (p * m) >> np.uint64(32)
        assert np.array_equal(t, p // np.uint64(k)), k


def test_group_index_division_is_exact():
    k0 = np.arange(0, 2 * 8192 + 64, dtype=np.uint64)
    for g in range(32, 8192 + 1, 32):
        m = (2**32 + g - 1) // g
        assert m < 2**32  # the kernels hold it in 32 bits
        gi = (k0 * np.uint64(m)) >> np.uint64(32)
        assert np.array_equal(gi, k0 // np.uint64(g)), g
