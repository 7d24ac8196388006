"""Write the small golden fixtures in this folder from the fp64 oracle.

The pages print no worked example with numbers, so every stored expected
value here comes from ``oracle/`` (and only from it); inputs are drawn from a
seeded numpy generator and rounded to their storage dtype by the oracle's
rounding helpers.  Run from the repository root:

    python tests/golden/make_golden.py
"""

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle as O  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))

# (name, op, N, H, dtype, eps, x offset, x scale)
CASES = [
    ("ln_f32_4x37", "ln", 4, 37, "float32", 1e-5, 0.0, 1.0),
    ("ln_bf16_3x64", "ln", 3, 64, "bfloat16", 1e-5, 0.0, 1.0),
    ("ln_f32_offset_3x40", "ln", 3, 40, "float32", 1e-5, 1000.0, 1e-2),
    ("ln_f32_h1_5x1", "ln", 5, 1, "float32", 1e-5, 0.0, 1.0),
    ("rms_bf16_3x72", "rms", 3, 72, "bfloat16", 1e-5, 0.0, 1.0),
    ("rms_f32_2x9", "rms", 2, 9, "float32", 1e-6, 0.0, 1.0),
    ("fused_bf16_2x48", "fused", 2, 48, "bfloat16", 1e-6, 0.0, 1.0),
    ("fused_f32_3x13", "fused", 3, 13, "float32", 1e-6, 0.0, 1.0),
    ("ln_y_bf16_3x40", "ln_y", 3, 40, "bfloat16", 1e-5, 0.0, 1.0),
    ("rms_y_f32_2x24", "rms_y", 2, 24, "float32", 1e-5, 0.0, 1.0),
]


def _r(a, dt):
    return O.round_to_dtype(np.asarray(a, dtype=np.float64), dt)


def make(name, op, N, H, dt, eps, off, scale, seed):
    rng = np.random.default_rng(seed)
    x = _r(off + scale * rng.standard_normal((N, H)), dt)
    gamma = _r(1.0 + 0.1 * rng.standard_normal(H), dt)
    beta = _r(0.1 * rng.standard_normal(H), dt)
    dy = _r(rng.standard_normal((N, H)), dt)
    res = _r(rng.standard_normal((N, H)), dt)
    stream = _r(rng.standard_normal((N, H)), dt)  # drawn last: the earlier draws keep their values
    case = {"name": name, "op": op, "N": N, "H": H, "dtype": dt, "eps": eps,
            "source": "oracle/norm_oracle.py via tests/golden/make_golden.py",
            "inputs": {"x": x.tolist(), "gamma": gamma.tolist()}}
    exp = {}
    if op == "ln":
        case["inputs"]["beta"] = beta.tolist()
        case["inputs"]["dy"] = dy.tolist()
        y, mean, rstd = O.layer_norm_forward(x, gamma, beta, eps)
        dx, dg, db = O.layer_norm_backward(dy, x, gamma, eps)
        exp.update(y=y, mean=mean, rstd=rstd, dx=dx, dgamma=dg, dbeta=db)
    elif op == "rms":
        case["inputs"]["dy"] = dy.tolist()
        y, rstd = O.rms_norm_forward(x, gamma, eps)
        dx, dg = O.rms_norm_backward(dy, x, gamma, eps)
        exp.update(y=y, rstd=rstd, dx=dx, dgamma=dg)
    elif op == "fused":
        case["inputs"]["residual"] = res.tolist()
        case["inputs"]["dy"] = dy.tolist()
        case["inputs"]["dh_stream"] = stream.tolist()
        y, h, rstd = O.fused_add_rms_norm_forward(x, res, gamma, eps, dt)
        # the backward reads the stored h, and the residual stream's gradient
        dh, dg = O.fused_add_rms_norm_backward_from_h(dy, h, gamma, eps, stream)
        exp.update(y=y, h=h, rstd=rstd, dh=dh, dgamma=dg)
    elif op == "ln_y":
        # the backward from the forward's stored output y and saved fp32 rstd
        y, _, rstd = O.layer_norm_forward(x, gamma, beta, eps)
        y, rstd = _r(y, dt), O.round_to_float32(rstd)
        case["inputs"].update(beta=beta.tolist(), dy=dy.tolist(), y=y.tolist(), rstd=rstd.tolist())
        dx, dg, db = O.layer_norm_backward_from_output(dy, y, rstd, gamma, beta)
        exp.update(dx=dx, dgamma=dg, dbeta=db)
    else:
        y, rstd = O.rms_norm_forward(x, gamma, eps)
        y, rstd = _r(y, dt), O.round_to_float32(rstd)
        case["inputs"].update(dy=dy.tolist(), y=y.tolist(), rstd=rstd.tolist())
        dx, dg = O.rms_norm_backward_from_output(dy, y, rstd, gamma)
        exp.update(dx=dx, dgamma=dg)
    case["expected"] = {k: np.asarray(v).tolist() for k, v in exp.items()}
    return case


def main():
    for i, c in enumerate(CASES):
        case = make(*c, seed=1000 + i)
        with open(os.path.join(HERE, c[0] + ".json"), "w") as f:
            json.dump(case, f, indent=0)
            f.write("\n")
    print(f"wrote {len(CASES)} fixtures")


if __name__ == "__main__":
    main()
