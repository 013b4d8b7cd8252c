"""The library's host-side learning-rate schedule (nc_lr_schedule) against the
oracle's definition, and its argument checks.  No GPU is needed: the schedule
is host arithmetic in libnc.so.

nanochat speedrun walkthrough (lyylswood.com), section 预搜检: the rate
scales as 1/sqrt(dim); lrm falls linearly to 0 near the end of training.
The library's values are fp32, the oracle's fp64: relative error <= 2e-7.
"""

import numpy as np
import pytest

from oracle import schedule as osched


def test_library_schedule_matches_oracle():
    from pretraining_step_03_b300 import _lib as L
    base = (0.02, 0.2, 0.004)
    for n, f in ((21400, 0.2), (100, 0.2), (7, 1.0), (50, 0.0), (3, 0.5)):
        for s in sorted({0, n // 2, n - 1, min(n - 1, n - round(f * n)), max(0, n - 2)}):
            for d in (1280, 1920):
                got = L.nc_lr_schedule(s, n, f, d, 1280, base)
                ref = osched.learning_rates(s, n, f, d, 1280, base)
                np.testing.assert_allclose(got, ref, rtol=2e-7, atol=0)


@pytest.mark.parametrize("args", [(5, 5, 0.2, 1280, 1280), (-1, 5, 0.2, 1280, 1280),
                                  (0, 0, 0.2, 1280, 1280), (0, 5, 1.5, 1280, 1280),
                                  (0, 5, -0.1, 1280, 1280), (0, 5, 0.2, 0, 1280)])
def test_library_schedule_rejects_bad_arguments(args):
    from pretraining_step_03_b300 import _lib as L
    with pytest.raises(L.NcError):
        L.nc_lr_schedule(*args, (0.02, 0.2, 0.004))
