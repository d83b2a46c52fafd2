"""The GPU tests' output canaries (tests/_gpu.py Guarded), checked on the
CPU with planted mistakes: a write just outside the output is reported, and
an output element left unwritten stays NaN, so no oracle comparison passes."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_canary_catches_a_write_outside_the_output(dtype):
    from tests import _gpu as g
    for where in (-1, 0):   # just before the output, just after it
        gd = g.Guarded((3, 5), dtype, device="cpu")
        gd.t.fill_(1.0)
        gd.check("clean")                     # writes inside the output are fine
        idx = g.GUARD - 1 if where < 0 else g.GUARD + gd.n
        gd.buf[idx] = 0.5
        with pytest.raises(AssertionError, match="outside"):
            gd.check("planted")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_unwritten_output_is_nan_and_fails_the_comparison(dtype):
    from tests import _gpu as g
    gd = g.Guarded((2, 4, 8), dtype, device="cpu")
    ref = np.zeros((2, 4, 8))
    gd.t[0].fill_(0.0)                        # row 1 left unwritten
    got = gd.t.float().numpy()
    assert np.isnan(got[1]).all() and not np.isnan(got[0]).any()
    with pytest.raises(AssertionError):
        g.compare(got, ref, "planted")
