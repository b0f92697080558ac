"""The CPU oracle against its pins (closed forms, brute force, a library
routine, central differences and invariants). CPU only."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_threads_do_not_change_results(orc):
    """Row-parallel calls compute each row exactly as a single-threaded call."""
    import numpy as np
    rng = np.random.default_rng(0)
    x = (2 * rng.standard_normal((37, 211))).astype(np.float32)
    labels = rng.integers(0, 211, size=37)
    a = orc.ce_rows(x, 211, labels, threads=1)
    b = orc.ce_rows(x, 211, labels, threads=5)
    assert (a == b).all()
    g1, l1 = orc.ce_grad(x, 211, labels, 0.5, threads=1)
    g2, l2 = orc.ce_grad(x, 211, labels, 0.5, threads=4)
    assert (g1 == g2).all() and (l1 == l2).all()
    assert (orc.argmax(x, 211, threads=1) == orc.argmax(x, 211, threads=3)).all()


def test_rejects_bad_shapes(orc):
    import numpy as np
    x = np.zeros((2, 5), dtype=np.float32)
    with pytest.raises(ValueError):
        orc.ce_rows(x, 6, np.zeros(2, dtype=np.int64))
    with pytest.raises(ValueError):
        orc.argmax(x, 0)
    with pytest.raises(TypeError):
        orc.argmax(x.astype(np.float64), 5)
