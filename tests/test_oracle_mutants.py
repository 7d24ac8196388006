"""Plant plausible mistakes in copies of the oracle and check the pins catch each.

The mistakes live here, on the CPU, in stand-in functions; the oracle itself
is untouched.  A mutant survives only if every pin in ``oracle_pins`` still
passes with it, and this test fails if any mutant survives.
"""

from types import SimpleNamespace

import numpy as np
import pytest

import oracle
from oracle import norm_oracle as R
from oracle_pins import ALL_PINS


def _ns(**override):
    base = {name: getattr(oracle, name) for name in oracle.__all__}
    base.update(override)
    return SimpleNamespace(**base)


def _ln_fwd(var_div=None, eps_outside=False, gamma_flip=False, mean_div=None):
    def f(x, gamma=None, beta=None, eps=1e-5):
        x = np.asarray(x, dtype=np.float64)
        N, H = x.shape
        g = np.ones(H) if gamma is None else np.asarray(gamma, dtype=np.float64)
        b = np.zeros(H) if beta is None else np.asarray(beta, dtype=np.float64)
        if gamma_flip:
            g = g[::-1]
        mean = x.sum(axis=1) / (mean_div(H) if mean_div else H)
        var = ((x - mean[:, None]) ** 2).sum(axis=1) / (var_div(H) if var_div else H)
        rstd = 1.0 / (np.sqrt(var) + eps) if eps_outside else 1.0 / np.sqrt(var + eps)
        y = (x - mean[:, None]) * rstd[:, None] * g + b
        return y, mean, rstd
    return f


def _ln_bwd(drop_c2=False, sign_c1=1.0, forget_gamma=False, dgamma_no_rstd=False, dbeta_of_g=False):
    def f(dy, x, gamma=None, eps=1e-5):
        dy = np.asarray(dy, dtype=np.float64)
        x = np.asarray(x, dtype=np.float64)
        H = x.shape[1]
        gm = np.ones(H) if gamma is None else np.asarray(gamma, dtype=np.float64)
        mean, var = R.two_pass_stats(x)
        rstd = 1.0 / np.sqrt(var + eps)
        xh = (x - mean[:, None]) * rstd[:, None]
        g = dy if forget_gamma else dy * gm
        c2 = 0.0 if drop_c2 else (g * xh).sum(axis=1)[:, None]
        dx = rstd[:, None] / H * (H * g - sign_c1 * g.sum(axis=1)[:, None] - xh * c2)
        dgamma = (dy * (x - mean[:, None])).sum(axis=0) if dgamma_no_rstd else (dy * xh).sum(axis=0)
        dbeta = g.sum(axis=0) if dbeta_of_g else dy.sum(axis=0)
        return dx, dgamma, dbeta
    return f


def _rms_fwd(subtract_mean=False, no_div=False):
    def f(x, gamma=None, eps=1e-5):
        x = np.asarray(x, dtype=np.float64)
        H = x.shape[1]
        g = np.ones(H) if gamma is None else np.asarray(gamma, dtype=np.float64)
        if subtract_mean:
            x = x - x.mean(axis=1, keepdims=True)
        ms = (x * x).sum(axis=1) / (1 if no_div else H)
        rstd = 1.0 / np.sqrt(ms + eps)
        return x * rstd[:, None] * g, rstd
    return f


def _rms_bwd(c2_no_div=False, wrong_sign=False, dgamma_of_x=False):
    def f(dy, x, gamma=None, eps=1e-5):
        dy = np.asarray(dy, dtype=np.float64)
        x = np.asarray(x, dtype=np.float64)
        H = x.shape[1]
        gm = np.ones(H) if gamma is None else np.asarray(gamma, dtype=np.float64)
        rstd = 1.0 / np.sqrt((x * x).sum(axis=1) / H + eps)
        xh = x * rstd[:, None]
        g = dy * gm
        c2 = (g * xh).sum(axis=1) / (1 if c2_no_div else H)
        dx = rstd[:, None] * (g + (1 if wrong_sign else -1) * xh * c2[:, None])
        dgamma = (dy * (x if dgamma_of_x else xh)).sum(axis=0)
        return dx, dgamma
    return f


def _fused_from_x():
    def f(x, residual, gamma=None, eps=1e-6, h_dtype="float32"):
        x = np.asarray(x, dtype=np.float64)
        h = x + np.asarray(residual, dtype=np.float64)
        y, rstd = R.rms_norm_forward(x, gamma, eps)
        return y, R.round_to_dtype(R.round_to_float32(h), h_dtype), rstd
    return f


def _fused_bwd_half():
    def f(dy, x, residual, gamma=None, eps=1e-6):
        dh, dg = R.rms_norm_backward(dy, np.asarray(x) + np.asarray(residual), gamma, eps)
        return dh, 0.5 * dh, dg
    return f


def _fused_from_h_forgets_stream():
    def f(dy, h, gamma=None, eps=1e-6, dh_stream=None):
        return R.rms_norm_backward(dy, h, gamma, eps)
    return f


def _ln_from_y_forgets_beta():
    def f(dy, y, rstd, gamma=None, beta=None):
        return R.layer_norm_backward_from_output(dy, y, rstd, gamma, None)
    return f


def _rms_from_y_times_gamma():
    def f(dy, y, rstd, gamma=None):
        H = np.asarray(y).shape[1]
        gm = np.ones(H) if gamma is None else np.asarray(gamma, dtype=np.float64)
        return R.rms_norm_backward_from_output(dy, np.asarray(y) * gm * gm, rstd, gamma)
    return f


def _fused_normalises_rounded_h():
    def f(x, residual, gamma=None, eps=1e-6, h_dtype="float32"):
        h = np.asarray(x, dtype=np.float64) + np.asarray(residual, dtype=np.float64)
        h_st = R.round_to_dtype(R.round_to_float32(h), h_dtype)
        y, rstd = R.rms_norm_forward(h_st, gamma, eps)
        return y, h_st, rstd
    return f


def _fused_truncates_h():
    def f(x, residual, gamma=None, eps=1e-6, h_dtype="float32"):
        h = np.asarray(x, dtype=np.float64) + np.asarray(residual, dtype=np.float64)
        y, rstd = R.rms_norm_forward(h, gamma, eps)
        h32 = R.round_to_float32(h)
        return y, (_bf16_truncate(h32) if h_dtype == "bfloat16" else R.round_to_dtype(h32, h_dtype)), rstd
    return f


def _fused_bwd_dgamma_of_x():
    def f(dy, x, residual, gamma=None, eps=1e-6):
        dh, _ = R.rms_norm_backward(dy, np.asarray(x) + np.asarray(residual), gamma, eps)
        _, dg = R.rms_norm_backward(dy, x, gamma, eps)
        return dh, dh.copy(), dg
    return f


def _fused_from_h_subtracts_stream():
    def f(dy, h, gamma=None, eps=1e-6, dh_stream=None):
        dh, dg = R.rms_norm_backward(dy, h, gamma, eps)
        return (dh if dh_stream is None else dh - np.asarray(dh_stream)), dg
    return f


def _ln_from_y(xhat_times_gamma=False, drop_rstd=False):
    def f(dy, y, rstd, gamma=None, beta=None):
        dy = np.asarray(dy, dtype=np.float64)
        y = np.asarray(y, dtype=np.float64)
        H = y.shape[1]
        gm = np.ones(H) if gamma is None else np.asarray(gamma, dtype=np.float64)
        bt = np.zeros(H) if beta is None else np.asarray(beta, dtype=np.float64)
        r = np.ones(y.shape[0]) if drop_rstd else np.asarray(rstd, dtype=np.float64).reshape(-1)
        xh = (y - bt) * gm if xhat_times_gamma else (y - bt) / gm
        g = dy * gm
        dx = r[:, None] / H * (H * g - g.sum(axis=1)[:, None] - xh * (g * xh).sum(axis=1)[:, None])
        return dx, (dy * xh).sum(axis=0), dy.sum(axis=0)
    return f


def _rms_from_y_dgamma_of_y():
    def f(dy, y, rstd, gamma=None):
        dx, _ = R.rms_norm_backward_from_output(dy, y, rstd, gamma)
        return dx, (np.asarray(dy, dtype=np.float64) * np.asarray(y, dtype=np.float64)).sum(axis=0)
    return f


def _merge_wrong(a, b):
    na, ma, m2a = a
    nb, mb, m2b = b
    n = na + nb
    if n == 0:
        return 0.0, 0.0, 0.0
    d = mb - ma
    return n, ma + d * nb / n, m2a + m2b + d * d * n


def _welford_seq_wrong(values):
    count, mean, m2 = 0.0, 0.0, 0.0
    for v in np.asarray(values, dtype=np.float64).ravel():
        count += 1.0
        old = mean
        mean = old + (v - old) / count
        m2 = m2 + (v - old) * (v - old)
    return count, mean, m2


def _bf16_truncate(a):
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    bits = f.view(np.uint32) & np.uint32(0xFFFF0000)
    return bits.view(np.float32).astype(np.float64)


def _f16_truncate(a):
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    with np.errstate(over="ignore"):
        h = f.astype(np.float16).astype(np.float32)
    # step one binary16 unit toward zero wherever nearest rounding went away from zero
    away = np.abs(h) > np.abs(f)
    h = np.where(away, np.nextafter(h.astype(np.float16), np.float16(0)).astype(np.float32), h)
    return h.astype(np.float64)


MUTANTS = {
    "ln_unbiased_variance": dict(layer_norm_forward=_ln_fwd(var_div=lambda H: max(H - 1, 1))),
    "ln_eps_outside_sqrt": dict(layer_norm_forward=_ln_fwd(eps_outside=True)),
    "ln_gamma_reversed": dict(layer_norm_forward=_ln_fwd(gamma_flip=True)),
    "ln_mean_wrong_divisor": dict(layer_norm_forward=_ln_fwd(mean_div=lambda H: H + 1)),
    "ln_bwd_dropped_xhat_term": dict(layer_norm_backward=_ln_bwd(drop_c2=True)),
    "ln_bwd_wrong_sign_sum_g": dict(layer_norm_backward=_ln_bwd(sign_c1=-1.0)),
    "ln_bwd_forgot_gamma": dict(layer_norm_backward=_ln_bwd(forget_gamma=True)),
    "ln_bwd_dgamma_without_rstd": dict(layer_norm_backward=_ln_bwd(dgamma_no_rstd=True)),
    "ln_bwd_dbeta_of_g": dict(layer_norm_backward=_ln_bwd(dbeta_of_g=True)),
    "rms_subtracts_mean": dict(rms_norm_forward=_rms_fwd(subtract_mean=True)),
    "rms_sum_not_mean": dict(rms_norm_forward=_rms_fwd(no_div=True)),
    "rms_bwd_c2_not_divided": dict(rms_norm_backward=_rms_bwd(c2_no_div=True)),
    "rms_bwd_wrong_sign": dict(rms_norm_backward=_rms_bwd(wrong_sign=True)),
    "rms_bwd_dgamma_of_x": dict(rms_norm_backward=_rms_bwd(dgamma_of_x=True)),
    "fused_normalises_x_not_h": dict(fused_add_rms_norm_forward=_fused_from_x()),
    "fused_bwd_halves_dres": dict(fused_add_rms_norm_backward=_fused_bwd_half()),
    "ln_from_output_forgets_beta": dict(layer_norm_backward_from_output=_ln_from_y_forgets_beta()),
    "rms_from_output_multiplies_gamma": dict(rms_norm_backward_from_output=_rms_from_y_times_gamma()),
    "fused_bwd_from_h_forgets_stream": dict(fused_add_rms_norm_backward_from_h=_fused_from_h_forgets_stream()),
    "fused_normalises_rounded_h": dict(fused_add_rms_norm_forward=_fused_normalises_rounded_h()),
    "fused_truncates_h": dict(fused_add_rms_norm_forward=_fused_truncates_h()),
    "fused_bwd_dgamma_of_x": dict(fused_add_rms_norm_backward=_fused_bwd_dgamma_of_x()),
    "fused_bwd_from_h_subtracts_stream": dict(fused_add_rms_norm_backward_from_h=_fused_from_h_subtracts_stream()),
    "ln_from_output_xhat_times_gamma": dict(layer_norm_backward_from_output=_ln_from_y(xhat_times_gamma=True)),
    "ln_from_output_drops_rstd": dict(layer_norm_backward_from_output=_ln_from_y(drop_rstd=True)),
    "rms_from_output_dgamma_of_y": dict(rms_norm_backward_from_output=_rms_from_y_dgamma_of_y()),
    "welford_merge_wrong_weight": dict(welford_merge=_merge_wrong),
    "welford_recurrence_old_mean_twice": dict(welford_sequential=_welford_seq_wrong),
    "bf16_truncates": dict(round_to_bfloat16=_bf16_truncate),
    "f16_truncates": dict(round_to_float16=_f16_truncate),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    ns = _ns(**MUTANTS[name])
    if "welford_merge" in MUTANTS[name] or "welford_sequential" in MUTANTS[name]:
        # welford_tree calls the module-level functions; give the mutant its own tree
        seq, merge = ns.welford_sequential, ns.welford_merge

        def tree(values, cuts):
            values = np.asarray(values, dtype=np.float64).ravel()
            b = [0] + sorted(int(s) for s in cuts) + [values.size]
            acc = (0.0, 0.0, 0.0)
            for lo, hi in zip(b[:-1], b[1:]):
                acc = merge(acc, seq(values[lo:hi]))
            return acc
        ns.welford_tree = tree
    caught = []
    for pin in ALL_PINS:
        try:
            pin(ns)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
