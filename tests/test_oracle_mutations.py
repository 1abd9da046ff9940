"""Planted mistakes in the oracle must each fail at least one oracle pin (no GPU).

Every case below rewrites one line of one oracle function into a plausible
mistake (a dropped term, a wrong sign or index, a transposed operand, a
reversed order), installs the mutant in the oracle module for the duration of
the test, and runs the pins of tests/test_oracle_*.py until one fails.  A
mutant that passes every pin is a hole in the pinning and fails this test.
The mistakes live only in memory, in the oracle, on the CPU; nothing else is
touched.
"""
import inspect
import textwrap

import pytest

import test_oracle_dequant
import test_oracle_ffn
import test_oracle_planner
import test_oracle_routing
from oracle import pw_oracle as O
from oracle import pw_planner as P

_PIN_MODULES = (test_oracle_routing, test_oracle_dequant, test_oracle_ffn, test_oracle_planner)


def _pins():
    """(name, function, kwargs) for every pin, one entry per parameter set."""
    out = []
    for mod in _PIN_MODULES:
        for name, fn in sorted(vars(mod).items()):
            if not name.startswith("test_") or not callable(fn):
                continue
            marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
            if not marks:
                out.append((f"{mod.__name__}.{name}", fn, {}))
                continue
            assert len(marks) == 1, name
            argnames, argvalues = marks[0].args[:2]
            names = [n.strip() for n in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
            for vals in argvalues:
                vals = tuple(vals) if len(names) > 1 else (vals,)
                out.append((f"{mod.__name__}.{name}{vals}", fn, dict(zip(names, vals))))
    return out


PINS = _pins()

# (label, module, function, original text, mistaken text)
MUTATIONS = [
    # routing
    ("top-K off by one", O, "route_topk",
     'idx = np.argsort(-l, axis=1, kind="stable")[:, :K]',
     'idx = np.argsort(-l, axis=1, kind="stable")[:, 1:K + 1]'),
    ("ties go to the higher index", O, "route_topk",
     'idx = np.argsort(-l, axis=1, kind="stable")[:, :K]',
     'idx = (l.shape[1] - 1 - np.argsort(-l[:, ::-1], axis=1, kind="stable"))[:, :K]'),
    ("weights are the logits", O, "route_topk",
     "w = np.take_along_axis(p, idx, axis=1)", "w = np.take_along_axis(l, idx, axis=1)"),
    ("renormalisation dropped", O, "route_topk", "    if renormalize:\n", "    if False:\n"),
    ("softmax normalised over the batch", O, "softmax",
     "return p / p.sum(axis=1, keepdims=True)", "return p / p.sum()"),
    ("router bias subtracted", O, "router_logits",
     "l = l + np.asarray(bias, dtype=np.float64)[None, :]", "l = l - np.asarray(bias, dtype=np.float64)[None, :]"),
    # permutation
    ("bucket order reversed", O, "permute",
     'order = np.argsort(flat, kind="stable")', "order = np.lexsort((-np.arange(flat.size), flat))"),
    ("inv_slot is the permutation, not its inverse", O, "permute",
     "inv_slot[order] = np.arange(T * K, dtype=np.int32)", "inv_slot[:] = order"),
    ("perm_src takes k instead of t", O, "permute",
     "perm_src = (order // K).astype(np.int32)", "perm_src = (order % K).astype(np.int32)"),
    # dequantisation
    ("low bits instead of top bits", O, "code_at_bits",
     "return (code6.astype(np.int64) >> (6 - b))", "return (code6.astype(np.int64) & ((1 << b) - 1))"),
    ("LUT of the wrong row", O, "dequant",
     "return lut[rows, code].astype(np.float64)", "return lut[rows[::-1], code].astype(np.float64)"),
    ("LUT of the next bitwidth", O, "dequant",
     "lut = np.asarray(luts[b - 3])", "lut = np.asarray(luts[min(b - 2, 3)])"),
    ("fp16 page ignored", O, "dequant", "return w16.astype(np.float64)", "return dequant(code6, luts, 6)"),
    # expert FFN
    ("silu sign flipped", O, "silu", "return v / (1.0 + np.exp(-v))", "return v / (1.0 + np.exp(v))"),
    ("gate and up swapped", O, "swiglu_ffn", "return (silu(g) * u) @ Wd.T", "return (silu(u) * g) @ Wd.T"),
    ("activation dropped", O, "swiglu_ffn", "return (silu(g) * u) @ Wd.T", "return (g * u) @ Wd.T"),
    ("down projection transposed", O, "swiglu_ffn", "return (silu(g) * u) @ Wd.T", "return (silu(g) * u) @ Wd"),
    ("up matrix replaced by gate", O, "expert_weights", "for m in range(3)]", "for m in (0, 0, 2)]"),
    ("expert fed unpermuted rows", O, "moe_layer",
     "y_perm[lo:hi] = swiglu_ffn(Wg, Wu, Wd, x[perm_src[lo:hi]])", "y_perm[lo:hi] = swiglu_ffn(Wg, Wu, Wd, x[lo:hi])"),
    # combine
    ("first weight for every k", O, "combine",
     "y += w[:, k:k + 1] * y_perm[slots[:, k]]", "y += w[:, 0:1] * y_perm[slots[:, k]]"),
    ("shared FFN weighted", O, "combine", "y += shared", "y += w.sum(axis=1, keepdims=True) * shared"),
    # stored layouts
    ("plane 0 is the least significant bit", O, "pack_planes",
     "bit = (c >> (5 - p)) & 1", "bit = (c >> p) & 1"),
    ("lane index transposed", O, "_plane_index", "L = 4 * g + t", "L = 4 * t + g"),
    ("bit position inside the word permuted", O, "_plane_index", "q = 8 * k + 4 * h + s", "q = 8 * k + 2 * s + h"),
    ("fp16 register order transposed", O, "_f16_index", "a = rowsel + 2 * colhalf", "a = 2 * rowsel + colhalf"),
    # planner
    ("most damage per byte first", P, "plan_bitwidths",
     "if best_key is None or key < best_key:", "if best_key is None or key > best_key:"),
    ("floors ignored", P, "plan_bitwidths", "if b <= max(level, floors[e]):", "if b <= level:"),
    ("no stages: straight to the last level", P, "plan_bitwidths", "level = LEVELS[stage]", "level = LEVELS[-1]"),
    ("residual ratio inverted", P, "expert_weights",
     "ratio = (float(resid[e]) / float(mass[e])) / (R / M)", "ratio = (float(mass[e]) / float(resid[e])) / (M / R)"),
    ("residual with the squared norm", P, "route_stats",
     "resid[e] += float(w[t, k]) * norms[t]", "resid[e] += float(w[t, k]) * norms[t] ** 2"),
]


def _mutant(mod, fname, old, new):
    src = textwrap.dedent(inspect.getsource(getattr(mod, fname)))
    assert src.count(old) == 1, (fname, old)
    ns = dict(vars(mod))
    exec(compile(src.replace(old, new), f"<mutant of {fname}>", "exec"), ns)
    return ns[fname]


def _first_failing_pin():
    for name, fn, kw in PINS:
        try:
            fn(**kw)
        except Exception:  # an assertion, or the mistake breaking the computation
            return name
    return None


def test_pins_collected():
    assert len(PINS) >= 50
    assert _first_failing_pin() is None  # the unmutated oracle passes every pin


@pytest.mark.parametrize("label,mod,fname,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(label, mod, fname, old, new, monkeypatch):
    monkeypatch.setattr(mod, fname, _mutant(mod, fname, old, new))
    caught = _first_failing_pin()
    assert caught is not None, f"no oracle pin fails when {label} ({fname})"


# Rewrites that change nothing: the harness must not report them as caught
# (a mutant that merely failed to build or run would otherwise count).
EQUIVALENT = [
    (O, "route_topk", 'idx = np.argsort(-l, axis=1, kind="stable")[:, :K]',
     'idx = np.argsort(-l, axis=1, kind="stable")[:, 0:K]'),
    (O, "silu", "return v / (1.0 + np.exp(-v))", "return v / (np.exp(-v) + 1.0)"),
    (O, "pack_planes", "bit = (c >> (5 - p)) & 1", "bit = (c >> (5 - p)) % 2"),
    (O, "combine", "y += shared", "y = y + shared"),
    (P, "plan_bitwidths", "if best_key is None or key < best_key:", "if best_key is None or best_key > key:"),
]


@pytest.mark.parametrize("mod,fname,old,new", EQUIVALENT, ids=[f"{m[1]}:{m[3]}" for m in EQUIVALENT])
def test_equivalent_rewrite_passes_every_pin(mod, fname, old, new, monkeypatch):
    monkeypatch.setattr(mod, fname, _mutant(mod, fname, old, new))
    assert _first_failing_pin() is None
