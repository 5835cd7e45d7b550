"""The FMA-pipe 2^x used optionally by the extend softmax: range reduction
x = j + f (j = round(x) via the 1.5 * 2^23 trick) and a fitted cubic for 2^f.
Its constants are read from the kernel header and its float32 evaluation is
checked against exact 2^x over the range the softmax uses."""
import os
import re

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "radixattention_prefix_shared_gb300", "csrc")


def _constants():
    src = open(os.path.join(CSRC, "common.cuh")).read()
    return [float(re.search(rf"kExp2C{i} = ([0-9.eE+-]+)f;", src).group(1)) for i in (1, 2, 3)]


def test_exp2_polynomial_error_bound():
    import importlib.util
    spec = importlib.util.spec_from_file_location("exp2_fit", os.path.join(CSRC, "exp2_fit.py"))
    fit = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(fit)
    c = _constants()
    x = np.linspace(-125, 8, 400001, dtype=np.float32)
    got = fit.exp2_f32(x, c).astype(np.float64)
    rel = np.abs(got / np.exp2(x.astype(np.float64)) - 1)
    assert rel.max() < 1.1e-4
    # exact at integers (f = 0 gives p = 1), so a lone key still weighs exactly 1
    xi = np.arange(-125, 9, dtype=np.float32)
    assert np.array_equal(fit.exp2_f32(xi, c), np.exp2(xi.astype(np.float64)).astype(np.float32))
