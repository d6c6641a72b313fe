"""The CPU oracle against its pins (no GPU).  See tests/oracle_pins.py."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as P


@pytest.fixture(scope="module")
def O():
    return oracle.default()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(O, pin):
    pin(O)


def test_quantize_matches_float32_restatement(O):
    """Regression check of the build flags (not a pin): numpy's IEEE float32
    ops restate the Sec. 5 rounding; any fused multiply-add or fast-math in
    the C build shows up here as a flipped quant byte."""
    rng = np.random.default_rng(11)
    x = P.random_block_inputs(rng, 1 << 14)
    q, d = O.quantize_q8(x.reshape(1, -1))
    amax = np.abs(x).max(axis=1)
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        dd = (amax / np.float32(127)).astype(np.float32)
        idv = np.where(amax != 0, np.float32(127) / amax, np.float32(0)).astype(np.float32)
        v = (x * idv[:, None]).astype(np.float32)
        v = (v + np.copysign(np.float32(0.5), x)).astype(np.float32)
        v = np.trunc(v)
        qq = np.where(v >= 127, 127, np.where(v <= -127, -127, np.where(np.isnan(v), 0, v)))
    assert np.array_equal(q.reshape(-1), qq.astype(np.int8).reshape(-1))
    assert np.array_equal(d.reshape(-1).view(np.uint32), dd.view(np.uint32))


def test_oracle_rejects_bad_shapes(O):
    with pytest.raises(ValueError):
        O.quantize_q8(np.zeros(33, dtype=np.float32))
    with pytest.raises(ValueError):
        O.matvec(1, np.zeros((2, 16), np.uint8), np.zeros((2, 1), np.float32), 2, 32,
                 np.zeros(32, np.int8), np.zeros(1, np.float32), r0=1, r1=3)
