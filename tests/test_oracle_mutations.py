"""Plant plausible mistakes in a private copy of the oracle and check that the
pins in test_oracle.py catch every one of them.

The copy is built from the oracle's source text with one substitution each;
the real oracle module is never modified.
"""
import inspect
import types

import pytest

import oracle.saf_oracle as real
import tests.test_oracle as pins

MUTATIONS = {
    # Eq. 3: wrong index into the relative preference (r[i] instead of r[i-j])
    "relative_index": ("r[np.where(keep, delta, 0)]", "r[np.where(keep, i[:, None] + 0 * delta, 0)]"),
    # Eq. 3: absolute preference indexed by the query instead of the key
    "absolute_index": ("(a[None, :] + r", "(a[i][:, None] + r"),
    # Eq. 3: dropped absolute term
    "dropped_alpha": ("(a[None, :] + r", "(0.0 * a[None, :] + r"),
    # causal mask off by one (diagonal excluded)
    "mask_diagonal": ("keep = delta >= 0", "keep = delta >= 1"),
    # Eq. 5: missing 1/sqrt(d)
    "missing_scale": ("return _row_softmax(_causal_scores(q[rows], k, rows, 1.0 / math.sqrt(d)))",
                      "return _row_softmax(_causal_scores(q[rows], k, rows, 1.0))"),
    "missing_scale_fwd": ("scale = 1.0 / math.sqrt(d)\n    pos = 0", "scale = 1.0\n    pos = 0"),
    # backward: sign error in the softmax Jacobian
    "dS_sign": ("dS = A * (dP - D)", "dS = A * (D - dP)"),
    # backward: D without the A weights
    "D_unweighted": ("D = np.sum(A * dP, axis=1, keepdims=True)", "D = np.sum(dP, axis=1, keepdims=True)"),
    # backward: transposed operand in dK
    "dK_transposed": ("dk += (dS.T @ q[blk]) * scale", "dk += (dS.T @ k[blk]) * scale"),
    # backward: frozen dV with the pattern untransposed
    "frozen_dV_untransposed": ("dv += P.T @ do[blk]", "dv[:len(blk)] += P[:, :len(blk)] @ do[blk]"),
    # pattern gradient: softmax Jacobian without the row term D
    "pattern_no_D": ("dL = P * (G - D)", "dL = P * G"),
    # pattern gradient: diagonal read the wrong way (delta = j instead of i - j)
    "pattern_diag_reversed": ("dr[:i + 1] += dL[t, i::-1]", "dr[:i + 1] += dL[t, :i + 1]"),
    # pattern gradient: dL/dP with V and dO swapped
    "pattern_G_swapped": ("G = do[blk] @ v.T", "G = v[blk] @ do.T"),
    # sampled pattern gradient: D from the values instead of the given output
    "pattern_at_D_from_v": ("D = np.sum(do[b, h] * o[b, h], axis=1)", "D = np.sum(do[b, h] * v[b, h], axis=1)"),
    # sampled pattern gradient: the diagonal's absolute term indexed by the query
    "pattern_at_diag_alpha": ("p = np.exp(a[h, i - x] + r[h, x] - lz[i])", "p = np.exp(a[h, i] + r[h, x] - lz[i])"),
    # sampled pattern gradient: column j's relative term read at the key index
    "pattern_at_col_rho": ("p = np.exp(a[h, j] + r[h, i - j] - lz[i])", "p = np.exp(a[h, j] + r[h, j] - lz[i])"),
    # fitting: relative marginal from the wrong side of the diagonal
    "fit_eta_rel_side": ("np.trace(P, offset=-delta)", "np.trace(P, offset=delta)"),
    # fitting: Eq. 20 without the 1/T
    "fit_grad_no_T": ("return (fa - eta_abs) / T, (fr - eta_rel) / T", "return (fa - eta_abs), (fr - eta_rel) / T"),
    # fitting: Eq. 4 with the relative term's sign flipped
    "fit_loss_sign": ("- np.dot(eta_rel, r)) / T", "+ np.dot(eta_rel, r)) / T"),
    # fitting: start point without the division by the diagonal's length T - delta
    "fit_start_no_length": ("np.log(np.maximum(eta_rel / (T - np.arange(T)), FIT_FLOOR))",
                            "np.log(np.maximum(eta_rel, FIT_FLOOR))"),
    # fitting: r started at zero instead of the diagonal means
    "fit_start_zero": ("np.log(np.maximum(eta_rel / (T - np.arange(T)), FIT_FLOOR))", "np.zeros(T)"),
    # fitting: Adam without the bias correction of its moments
    "fit_adam_no_bias_correction": ("mh = m[k] / (1 - b1 ** t)\n            vh = v[k] / (1 - b2 ** t)",
                                    "mh = m[k]\n            vh = v[k]"),
    # target negentropy: the sum taken over the whole matrix after a flipped log
    "negentropy_sign": ("return float(np.sum(P[pos] * np.log(P[pos]))) / T",
                        "return float(np.sum(P[pos] * np.log(1.0 / P[pos]))) / T"),
    # grouped-query layout: query head mapped to its key/value head by h % g instead of h // g
    "gqa_head_map": ("head_fwd(q[b, h], k[b, h // g], v[b, h // g], a[h], r[h], bool(frozen[h]))",
                     "head_fwd(q[b, h], k[b, h % Hkv], v[b, h % Hkv], a[h], r[h], bool(frozen[h]))"),
    # lse: forgot the max shift
    "lse_no_max": ("return m + np.log(np.sum(np.exp(L - m[:, None]), axis=1))",
                   "return np.log(np.sum(np.exp(L - m[:, None]), axis=1))"),
}

# The regression fixture compares the oracle with values it wrote itself, so it
# would flag any change: it does not count as a pin here.
PIN_TESTS = [(n, f) for n, f in inspect.getmembers(pins, inspect.isfunction)
             if n.startswith("test_") and n != "test_regression_fixture"]


def _mutant(src, old, new, name):
    assert old in src, f"mutation anchor for {name} not found in oracle source"
    mod = types.ModuleType(f"oracle_mutant_{name}")
    exec(compile(src.replace(old, new, 1), mod.__name__, "exec"), mod.__dict__)
    return mod


def _call(fn):
    cases = [()]
    for m in getattr(fn, "pytestmark", []):
        if m.name == "parametrize":
            cases = [(v,) for v in m.args[1]]
    for case in cases:
        fn(*case)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    pytest.importorskip("mpmath")
    src = inspect.getsource(real)
    old, new = MUTATIONS[name]
    mutant = _mutant(src, old, new, name)
    monkeypatch.setattr(pins, "oracle", mutant)
    caught = []
    for tname, fn in PIN_TESTS:
        try:
            _call(fn)
        except Exception:  # an assertion or a shape error both expose the mistake
            caught.append(tname)
    assert caught, f"no pin caught mutation {name}"

