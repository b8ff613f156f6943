"""The 16-bit block format of the partial-logit exchange (tests/exchange_format.py), on
the CPU: its codes fit in 16 bits, its error stays within 2^-15 of the block's largest
magnitude, and the lse it yields stays within the 2e-3 bar on the decode workloads'
logit ranges (the bar that the GPU tests apply to the kernel that uses it)."""
import numpy as np
import pytest

from tests.exchange_format import block16, block16_codes


def _blocks(rng):
    yield np.zeros(64, np.float32)
    yield np.full(64, np.nextafter(np.float32(2.0), np.float32(0.0)), np.float32)   # just below a power of 2
    yield -np.full(64, np.nextafter(np.float32(2.0), np.float32(0.0)), np.float32)
    yield np.array([np.float32(1024.0), -np.float32(1024.0)] + [0.0] * 62, np.float32)
    for mag in (1e-30, 1e-6, 1.0, 17.0, 540.0, 1e6, 1e30):
        yield (rng.standard_normal(64) * mag).astype(np.float32)
    yield (rng.standard_normal(7) * 3.0).astype(np.float32)    # a short block (the last page's keys)


def test_codes_fit_sixteen_bits():
    for x in _blocks(np.random.default_rng(0)):
        k, _ = block16_codes(x)
        assert k.min() >= 1 and k.max() <= 65535, (k.min(), k.max())


def test_error_within_two_to_minus_fifteen_of_the_block_max():
    for x in _blocks(np.random.default_rng(1)):
        _, back = block16_codes(x)
        amax = float(np.abs(x.astype(np.float64)).max())
        err = np.abs(back - x.astype(np.float64)).max()
        assert err <= amax * 2.0 ** -15 * (1 + 2.0 ** -10), (amax, err)
    assert np.array_equal(block16_codes(np.zeros(64, np.float32))[1], np.zeros(64))


def test_blocks_follow_pages():
    """A large value in one page does not coarsen the codes of the next page."""
    x = np.concatenate([np.full(64, 1000.0), np.full(64, 1e-3)])
    back = block16(x)
    assert np.abs(back[64:] - 1e-3).max() <= 1e-3 * 2.0 ** -14


def _lse(z):
    m = z.max()
    return m + np.log(np.exp(z - m).sum())


@pytest.mark.parametrize("sharp,bound", [(1, 1e-4), (8, 2e-3)])
def test_lse_shift_on_decode_logits(sharp, bound):
    """Rows shaped like the decode workloads (N(0,1) query and cache rows, 576 dims, scale
    1/sqrt(576)), also at 8x the scale: the lse of logits with the peer's half in the block
    format stays within `bound` of the exact one, and within the Lipschitz bound
    max_j |logit change| (lse is 1-Lipschitz in the max norm)."""
    rng = np.random.default_rng(7 + sharp)
    scale = sharp / np.sqrt(576.0)
    worst = 0.0
    for _ in range(64):
        n = int(rng.integers(1, 700))
        q = rng.standard_normal(576)
        k = rng.standard_normal((n, 576))
        h0, h1 = np.r_[0:256, 512:544], np.r_[256:512, 544:576]
        s0 = (k[:, h0] @ q[h0]).astype(np.float32).astype(np.float64)
        s1 = (k[:, h1] @ q[h1]).astype(np.float32).astype(np.float64)
        exact = _lse(scale * (s0 + s1))
        model = _lse(scale * (s0 + block16(s1)))
        shift = abs(model - exact)
        assert shift <= scale * np.abs(block16(s1) - s1).max() + 1e-12
        worst = max(worst, shift)
    assert worst < bound, worst


def test_bound_grows_with_the_logit_range():
    """The format's error is relative to a row's largest partial logit: at 32x the decode
    scale (logits of order 90) the worst lse shift is several times that at 8x."""
    rng = np.random.default_rng(11)
    q = rng.standard_normal(576)
    k = rng.standard_normal((640, 576))
    h0, h1 = np.r_[0:256, 512:544], np.r_[256:512, 544:576]
    s0, s1 = k[:, h0] @ q[h0], k[:, h1] @ q[h1]
    shift = {m: abs(_lse(m / 24.0 * (s0 + block16(s1))) - _lse(m / 24.0 * (s0 + s1))) for m in (8, 32)}
    assert shift[32] > 2 * shift[8]
