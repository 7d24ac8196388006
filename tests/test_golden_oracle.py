"""The oracle reproduces the stored golden fixtures (regression, CPU only)."""

import glob
import json
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = sorted(glob.glob(os.path.join(os.path.dirname(__file__), "golden", "*.json")))


def load(path):
    with open(path) as f:
        c = json.load(f)
    c["inputs"] = {k: np.asarray(v, dtype=np.float64) for k, v in c["inputs"].items()}
    c["expected"] = {k: np.asarray(v, dtype=np.float64) for k, v in c["expected"].items()}
    return c


@pytest.mark.parametrize("path", GOLDEN, ids=[os.path.basename(p) for p in GOLDEN])
def test_oracle_reproduces_golden(path):
    c = load(path)
    i, e, eps = c["inputs"], c["expected"], c["eps"]
    if c["op"] == "ln":
        got = dict(zip(("y", "mean", "rstd"), O.layer_norm_forward(i["x"], i["gamma"], i["beta"], eps)))
        got.update(zip(("dx", "dgamma", "dbeta"), O.layer_norm_backward(i["dy"], i["x"], i["gamma"], eps)))
    elif c["op"] == "rms":
        got = dict(zip(("y", "rstd"), O.rms_norm_forward(i["x"], i["gamma"], eps)))
        got.update(zip(("dx", "dgamma"), O.rms_norm_backward(i["dy"], i["x"], i["gamma"], eps)))
    elif c["op"] == "fused":
        got = dict(zip(("y", "h", "rstd"),
                       O.fused_add_rms_norm_forward(i["x"], i["residual"], i["gamma"], eps, c["dtype"])))
        got.update(zip(("dh", "dgamma"),
                       O.fused_add_rms_norm_backward_from_h(i["dy"], got["h"], i["gamma"], eps, i["dh_stream"])))
    elif c["op"] == "ln_y":
        got = dict(zip(("dx", "dgamma", "dbeta"),
                       O.layer_norm_backward_from_output(i["dy"], i["y"], i["rstd"], i["gamma"], i["beta"])))
    else:
        assert c["op"] == "rms_y", c["op"]
        got = dict(zip(("dx", "dgamma"), O.rms_norm_backward_from_output(i["dy"], i["y"], i["rstd"], i["gamma"])))
    assert set(got) == set(e)
    for k in e:
        np.testing.assert_allclose(got[k], e[k], rtol=1e-12, atol=1e-12, err_msg=k)


def test_golden_inputs_are_storage_exact():
    for path in GOLDEN:
        c = load(path)
        for k, v in c["inputs"].items():
            dt = "float32" if k == "rstd" else c["dtype"]  # a saved rstd is fp32 whatever the rows are
            assert np.array_equal(O.round_to_dtype(v, dt), v), (path, k)
