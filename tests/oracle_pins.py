"""Pins of the CPU oracle: checks against what the definitions and mathematics
fix, none of which re-types the oracle's own formula.

Each pin takes an ``oracle.Oracle`` and raises ``AssertionError`` when the
oracle disagrees. ``tests/test_oracle_pins.py`` runs them on the committed
oracle; ``tests/test_oracle_mutants.py`` runs them on copies of the oracle with
a planted mistake and requires that some pin fails for each.

The definitions pinned are those of the API reference page "gizml:netops"
(Functions: crossEntropyLoss, crossEntropyRows, crossEntropyGrad, argmaxInto,
candidatesInto, splitSumInto; Methods: Tensor.argmax; Constants: TOP_EACH,
CANDIDATE_ROW), and the softmax / log-softmax rows read from the same row
statistics.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.txt")


def _close(a, b, rel=0.0, abs_=0.0, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    both_nan = np.isnan(a) & np.isnan(b)
    same_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        ok = both_nan | same_inf | (np.abs(a - b) <= abs_ + rel * np.abs(b))
    if not ok.all():
        k = int(np.argmin(ok.ravel()))
        raise AssertionError(f"{what}: {a.ravel()[k]!r} != {b.ravel()[k]!r} at flat index {k}")


def _row(values):
    return np.array([values], dtype=np.float32)


# ---------------------------------------------------------------------------
# loss pins


def pin_uniform_rows(orc):
    """All-equal logits: every softmax is 1/V, loss = log V, grad = (1/V - onehot) scale."""
    for V in (1, 2, 3, 1000, 50257, 128256):
        for level in (0.0, -7.5, 1000.0):
            x = np.full((2, V), level, dtype=np.float32)
            labels = np.array([0, V - 1], dtype=np.int64)
            loss = orc.ce_rows(x, V, labels)
            _close(loss, [math.log(V)] * 2, rel=1e-14, abs_=1e-300, what=f"uniform loss V={V}")
            grad, loss2 = orc.ce_grad(x, V, labels, 0.25)
            _close(loss2, loss, rel=0, what="uniform loss from grad call")
            want = np.full((2, V), 0.25 / V)
            want[0, 0] -= 0.25
            want[1, V - 1] -= 0.25
            _close(grad, want, abs_=1e-16, what=f"uniform grad V={V}")


def pin_two_class_closed_form(orc):
    """V = 2: loss = softplus(x_other - x_label); p_label = 1 / (1 + e^d)."""
    for d in (-60.0, -40.0, -20.0, -5.0, -1.0, 0.0, 0.5, 3.0, 30.0):
        x = np.array([[1.0, 1.0 + d], [1.0 + d, 1.0]], dtype=np.float32)
        labels = np.array([0, 1], dtype=np.int64)
        want_loss = math.log1p(math.exp(d)) if d <= 0 else d + math.log1p(math.exp(-d))
        loss = orc.ce_rows(x, 2, labels)
        _close(loss, [want_loss] * 2, rel=1e-13, what=f"two-class loss d={d}")
        sig = 1.0 / (1.0 + math.exp(-d))     # softmax of the other class
        grad, _ = orc.ce_grad(x, 2, labels, 1.0)
        # p_label - 1 cancels in any format: absolute error up to ~1e-16
        _close(grad, [[-sig, sig], [sig, -sig]], rel=1e-13, abs_=2e-16,
               what=f"two-class grad d={d}")


def pin_tiny_loss(orc):
    """Label at the max, the rest far below: loss = log1p(sum e^-gap) ~ 1e-20."""
    x = np.array([[0.0, -60.0, -45.0], [-45.0, 0.0, -90.0]], dtype=np.float32)
    labels = np.array([0, 1], dtype=np.int64)
    want = [math.log1p(math.exp(-60) + math.exp(-45)), math.log1p(math.exp(-45) + math.exp(-90))]
    _close(orc.ce_rows(x, 3, labels), want, rel=1e-12, what="tiny loss")


def _brute_row(xs, label, scale):
    """Definition without the max shift, in pure Python (math.fsum)."""
    e = [math.exp(v) for v in xs]
    s = math.fsum(e)
    loss = -math.log(e[label] / s)
    grad = [(e[j] / s - (1.0 if j == label else 0.0)) * scale for j in range(len(xs))]
    return loss, grad


def pin_bruteforce_tiny(orc):
    """Small rows, |x| <= 4: the unshifted definition summed with math.fsum."""
    rng = np.random.default_rng(1234)
    for V in range(1, 17):
        x = rng.uniform(-4, 4, size=(5, V)).astype(np.float32)
        labels = rng.integers(0, V, size=5).astype(np.int64)
        grad, loss = orc.ce_grad(x, V, labels, 0.125)
        for i in range(5):
            bl, bg = _brute_row([float(v) for v in x[i]], int(labels[i]), 0.125)
            _close(loss[i], bl, rel=1e-12, abs_=1e-15, what=f"brute loss V={V}")
            _close(grad[i], bg, abs_=1e-14, what=f"brute grad V={V}")
        _close(orc.ce_rows(x, V, labels), loss, rel=0, what="ce_rows == ce_grad loss")


def pin_torch_cross_entropy(orc):
    """torch.nn.functional.cross_entropy in f64 on the CPU (a library routine),
    and its autograd gradient."""
    g = torch.Generator().manual_seed(99)
    x32 = (3.0 * torch.randn(16, 50, generator=g)).float()
    labels = torch.randint(0, 50, (16,), generator=g)
    x64 = x32.double().requires_grad_(True)
    ref = torch.nn.functional.cross_entropy(x64, labels, reduction="none")
    scale = 1.0 / 16
    (ref.sum() * scale).backward()
    grad, loss = orc.ce_grad(x32.numpy(), 50, labels.numpy(), scale)
    _close(loss, ref.detach().numpy(), rel=1e-12, what="torch loss rows")
    _close(grad, x64.grad.numpy(), abs_=1e-15, what="torch autograd grad")
    mean_ref = torch.nn.functional.cross_entropy(x32.double(), labels, reduction="mean").item()
    _close(orc.ce_mean(loss), mean_ref, rel=1e-13, what="torch mean")


def pin_central_differences(orc):
    """d loss / d x_j by central differences of the oracle's own loss
    (Richardson-extrapolated, error O(h^4)) equals the oracle's gradient at
    scale 1. Inputs are multiples of 2^-8 so that x +- h is exact in f32."""
    rng = np.random.default_rng(7)
    V = 6
    base = (rng.integers(-512, 512, size=V) / 256.0).astype(np.float32)
    label = 4
    lab = np.array([label], dtype=np.int64)

    def L(v):
        return float(orc.ce_rows(np.asarray([v], dtype=np.float32), V, lab)[0])

    grad, _ = orc.ce_grad(base[None, :].copy(), V, lab, 1.0)
    for j in range(V):
        def D(h):
            xp = base.copy(); xp[j] += h
            xm = base.copy(); xm[j] -= h
            return (L(xp) - L(xm)) / (2 * h)
        h = 2.0 ** -6
        est = (4 * D(h / 2) - D(h)) / 3
        _close(grad[0, j], est, abs_=1e-9, what=f"central difference j={j}")


def pin_grad_invariants(orc):
    """Rows of (softmax - onehot) sum to 0; the label column is (e^-loss - 1) scale."""
    rng = np.random.default_rng(3)
    x = (5.0 * rng.standard_normal((32, 100))).astype(np.float32)
    labels = rng.integers(0, 100, size=32).astype(np.int64)
    scale = 0.75
    grad, loss = orc.ce_grad(x, 100, labels, scale)
    _close(grad.sum(axis=1), np.zeros(32), abs_=1e-14, what="grad row sums")
    lab_col = grad[np.arange(32), labels]
    _close(lab_col, (np.exp(-loss) - 1.0) * scale, abs_=1e-14, what="label column")
    assert (grad[np.arange(100)[None, :] != labels[:, None]] >= 0).all(), "off-label grad < 0"


def pin_shift_invariance(orc):
    """loss(x + c) = loss(x); inputs are multiples of 2^-12 in [-8, 8] so x + 64 is exact."""
    rng = np.random.default_rng(11)
    x = (rng.integers(-8 * 4096, 8 * 4096, size=(8, 300)) / 4096.0).astype(np.float32)
    labels = rng.integers(0, 300, size=8).astype(np.int64)
    a = orc.ce_rows(x, 300, labels)
    for c in (64.0, -64.0):
        _close(orc.ce_rows((x + np.float32(c)).astype(np.float32), 300, labels), a,
               rel=1e-12, what=f"shift {c}")


def pin_mean(orc):
    """Mean of row losses: a known sum, math.fsum on random values, and 0/0 for no rows."""
    _close(orc.ce_mean(np.array([1.0, 2.0, 3.0, 4.0])), 2.5, rel=0, what="mean 1..4")
    rng = np.random.default_rng(5)
    v = rng.uniform(0, 10, size=10001)
    _close(orc.ce_mean(v), math.fsum(v) / v.size, rel=1e-14, what="mean fsum")
    assert math.isnan(orc.ce_mean(np.zeros(0))), "mean of no rows must be NaN"


def pin_nonfinite_rows(orc):
    """NaN, +inf or all -inf rows: the definition's IEEE value is NaN (loss and grad)."""
    nan, inf = float("nan"), float("inf")
    rows = [[1.0, nan, 2.0], [1.0, inf, 2.0], [-inf, -inf, -inf], [nan, nan, nan]]
    x = np.array(rows, dtype=np.float32)
    labels = np.array([0, 0, 1, 2], dtype=np.int64)
    loss = orc.ce_rows(x, 3, labels)
    assert np.isnan(loss).all(), f"non-finite rows must give NaN loss, got {loss}"
    grad, loss2 = orc.ce_grad(x, 3, labels, 1.0)
    assert np.isnan(grad).all() and np.isnan(loss2).all(), "non-finite rows must give NaN grad"
    # -inf entries with a finite max take no probability mass
    x = np.array([[0.0, -inf, 0.0], [0.0, 0.0, -inf]], dtype=np.float32)
    labels = np.array([0, 2], dtype=np.int64)
    grad, loss = orc.ce_grad(x, 3, labels, 2.0)
    _close(loss, [math.log(2), inf], rel=1e-15, what="-inf entries loss")
    _close(grad, [[-1.0, 0.0, 1.0], [1.0, 1.0, -2.0]], abs_=1e-15, what="-inf entries grad")


def pin_bad_label(orc):
    """A label outside [0, vocab): NaN loss; the gradient row is softmax * scale."""
    x = np.array([[0.0, 0.0], [0.0, 0.0]], dtype=np.float32)
    labels = np.array([-1, 2], dtype=np.int64)
    assert np.isnan(orc.ce_rows(x, 2, labels)).all(), "bad label must give NaN loss"
    grad, loss = orc.ce_grad(x, 2, labels, 3.0)
    assert np.isnan(loss).all()
    _close(grad, [[1.5, 1.5], [1.5, 1.5]], abs_=1e-15, what="bad label grad")


def pin_stride_padding(orc):
    """Only the first vocab columns count: padding of NaN or +1e30 changes nothing."""
    rng = np.random.default_rng(17)
    R, V, S = 6, 37, 45
    dense = rng.standard_normal((R, V)).astype(np.float32)
    labels = rng.integers(0, V, size=R).astype(np.int64)
    for pad in (float("nan"), 1e30):
        x = np.full((R, S), pad, dtype=np.float32)
        x[:, :V] = dense
        _close(orc.ce_rows(x, V, labels), orc.ce_rows(dense, V, labels), rel=0, what="padded loss")
        g1, _ = orc.ce_grad(x, V, labels, 1.0)
        g2, _ = orc.ce_grad(dense, V, labels, 1.0)
        _close(g1, g2, rel=0, what="padded grad")
        assert (orc.argmax(x, V) == orc.argmax(dense, V)).all(), "padded argmax"


# ---------------------------------------------------------------------------
# argmax pins


def _brute_argmax(row):
    best, bv = 0, None
    for j, v in enumerate(row):
        if math.isnan(v):
            continue
        if bv is None or v > bv:
            best, bv = j, v
    return best


def pin_argmax_bruteforce(orc):
    """Rows full of ties (small integers): the first of equals; also torch.argmax
    (first maximal index) on the same NaN-free rows."""
    rng = np.random.default_rng(21)
    for V in (1, 2, 3, 7, 16, 33, 40):
        x = rng.integers(0, 5, size=(50, V)).astype(np.float32)
        got = orc.argmax(x, V)
        want = [_brute_argmax([float(v) for v in r]) for r in x]
        assert list(got) == want, f"argmax brute force V={V}"
        assert (got == torch.argmax(torch.from_numpy(x), dim=1).numpy()).all(), "torch.argmax"


def pin_argmax_nan_rules(orc):
    """NaN never wins; a row without a non-NaN value gives 0; -0 == +0."""
    nan, inf = float("nan"), float("inf")
    cases = [([nan, 1.0, nan, 1.0], 1), ([nan, nan], 0), ([nan, -inf], 1), ([-0.0, 0.0], 0),
             ([0.0, -0.0], 0), ([-inf, -inf], 0), ([1.0, inf, inf], 1), ([3.0, nan, 5.0], 2),
             ([nan, 2.0, 1.0], 1)]
    for row, want in cases:
        x = np.array([row], dtype=np.float32)
        got = int(orc.argmax(x, len(row))[0])
        assert got == want, f"argmax {row}: {got} != {want}"


# ---------------------------------------------------------------------------
# golden closed forms


def _parse_golden():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lg, lab, sc, loss, grad, am = [p.strip() for p in line.split("|")]
            env = {"math": math}
            cases.append(dict(
                logits=[float(v) for v in lg.split(",")],
                label=int(lab), scale=float(sc),
                loss=float(eval(loss, env)),
                grad=[float(eval(g, env)) for g in grad.split(",")],
                argmax=int(am)))
    return cases


def pin_golden_closed_forms(orc):
    """tests/golden/closed_forms.txt: hand-derived values of small rows."""
    cases = _parse_golden()
    assert cases, "no golden cases"
    for c in cases:
        x = np.array([c["logits"]], dtype=np.float32)
        V = x.shape[1]
        lab = np.array([c["label"]], dtype=np.int64)
        grad, loss = orc.ce_grad(x, V, lab, c["scale"])
        _close(loss[0], c["loss"], rel=1e-13, abs_=1e-300, what=f"golden loss {c['logits']}")
        _close(orc.ce_rows(x, V, lab)[0], c["loss"], rel=1e-13, abs_=1e-300, what="golden rows")
        _close(grad[0], c["grad"], rel=1e-13, abs_=1e-16, what=f"golden grad {c['logits']}")
        assert int(orc.argmax(x, V)[0]) == c["argmax"], f"golden argmax {c['logits']}"


# ---------------------------------------------------------------------------
# softmax and log-softmax rows


def pin_softmax_closed_forms(orc):
    """Uniform rows: p = 1/V, log p = -log V. Two classes at gap d: p = sigmoid,
    log p = -softplus. A dominant token at a large max: log p = -log1p(e^-gap)."""
    for V in (1, 2, 7, 1000, 50257):
        x = np.full((2, V), 3.5, dtype=np.float32)
        _close(orc.softmax(x, V), np.full((2, V), 1.0 / V), rel=1e-15, what=f"uniform softmax V={V}")
        _close(orc.log_softmax(x, V), np.full((2, V), -math.log(V)), rel=1e-15, abs_=1e-300,
               what=f"uniform log-softmax V={V}")
    for d in (-60.0, -20.0, -1.0, 0.0, 2.0, 30.0):
        x = np.array([[1.0, 1.0 + d]], dtype=np.float32)
        _close(orc.softmax(x, 2), [[1.0 / (1.0 + math.exp(d)), 1.0 / (1.0 + math.exp(-d))]],
               rel=1e-13, abs_=1e-300, what=f"two-class softmax d={d}")
        sp = (lambda z: math.log1p(math.exp(z)) if z <= 0 else z + math.log1p(math.exp(-z)))
        _close(orc.log_softmax(x, 2), [[-sp(d), -sp(-d)]], rel=1e-13, what=f"two-class log-softmax d={d}")
    x = np.array([[100.0, 50.0, 40.0]], dtype=np.float32)
    want0 = -math.log1p(math.exp(-50) + math.exp(-60))
    got = orc.log_softmax(x, 3)
    _close(got[0, 0], want0, rel=1e-12, what="dominant token log p")
    _close(got[0, 1:], [-50 + want0, -60 + want0], rel=1e-14, what="other tokens log p")


def pin_softmax_torch(orc):
    """torch.softmax / torch.log_softmax in f64 on the CPU (library routines)."""
    g = torch.Generator().manual_seed(31)
    x = (4.0 * torch.randn(9, 301, generator=g)).float()
    _close(orc.softmax(x.numpy(), 301), torch.softmax(x.double(), 1).numpy(), abs_=1e-16,
           rel=1e-13, what="torch softmax")
    _close(orc.log_softmax(x.numpy(), 301), torch.log_softmax(x.double(), 1).numpy(), rel=1e-13,
           what="torch log_softmax")


def pin_softmax_invariants(orc):
    """Rows sum to 1; exp(log p) = p; padding past vocab is never read;
    non-finite rows are NaN; -inf entries of a finite row get p = 0, log p = -inf."""
    rng = np.random.default_rng(41)
    R, V, S = 5, 77, 90
    dense = (6 * rng.standard_normal((R, V))).astype(np.float32)
    p = orc.softmax(dense, V)
    _close(p.sum(axis=1), np.ones(R), abs_=1e-14, what="softmax row sums")
    _close(np.exp(orc.log_softmax(dense, V)), p, rel=1e-13, what="exp(log p) = p")
    for pad in (float("nan"), 1e30):
        x = np.full((R, S), pad, dtype=np.float32)
        x[:, :V] = dense
        _close(orc.softmax(x, V), p, rel=0, what="padded softmax")
        _close(orc.log_softmax(x, V), orc.log_softmax(dense, V), rel=0, what="padded log-softmax")
    nan, inf = float("nan"), float("inf")
    bad = np.array([[1.0, nan, 2.0], [1.0, inf, 2.0], [-inf, -inf, -inf]], dtype=np.float32)
    assert np.isnan(orc.softmax(bad, 3)).all() and np.isnan(orc.log_softmax(bad, 3)).all()
    x = np.array([[0.0, -inf, 0.0]], dtype=np.float32)
    _close(orc.softmax(x, 3), [[0.5, 0.0, 0.5]], rel=1e-15, what="-inf softmax")
    _close(orc.log_softmax(x, 3), [[-math.log(2), -inf, -math.log(2)]], rel=1e-15, what="-inf log p")


# ---------------------------------------------------------------------------
# sampling candidates (candidatesInto, TOP_EACH, CANDIDATE_ROW)

_CT, _CK = 256, 4  # threads of a candidates workgroup, values each keeps


def _slots(cand_row):
    """[256, 4, 2] view of one row's candidates: (value, column) per slot."""
    return np.asarray(cand_row, dtype=np.float32).reshape(_CT, _CK, 2)


def _want_cols(V, t, order):
    """The columns t, t + 256, ... below V, in `order` (first 4 kept)."""
    cols = list(range(t, V, _CT))
    cols = cols[::-1] if order == "desc" else cols
    return cols[:_CK]


def pin_candidates_closed_forms(orc):
    """Rows whose candidates follow by hand: x_j = j keeps each thread's last
    four columns, largest first; x_j = -j and a constant row keep its first
    four (equal values: the lower column ranks higher); an all -inf row keeps
    -inf values; NaN is never kept; a slot with no value is (-inf, -1)."""
    inf, nan = float("inf"), float("nan")
    for V in (1, 3, 255, 256, 257, 700, 1024, 1029, 2100):
        up = np.arange(V, dtype=np.float32)[None]
        rows = {
            "increasing": (up, "desc"),
            "decreasing": (-up, "asc"),
            "constant": (np.full((1, V), 2.5, np.float32), "asc"),
            "all -inf": (np.full((1, V), -inf, np.float32), "asc"),
        }
        for name, (x, order) in rows.items():
            sl = _slots(orc.candidates(x, V)[0])
            for t in range(_CT):
                cols = _want_cols(V, t, order)
                for k in range(_CK):
                    if k < len(cols):
                        want = (float(x[0, cols[k]]), float(cols[k]))
                    else:
                        want = (-inf, -1.0)
                    got = (float(sl[t, k, 0]), float(sl[t, k, 1]))
                    assert got == want, f"candidates {name} V={V} thread {t} slot {k}: {got} != {want}"
        # NaN at the even columns: even threads keep nothing, odd ones as the constant row
        x = np.full((1, V), 1.0, np.float32)
        x[0, 0::2] = nan
        sl = _slots(orc.candidates(x, V)[0])
        for t in range(_CT):
            cols = _want_cols(V, t, "asc") if t % 2 else []
            for k in range(_CK):
                want = (1.0, float(cols[k])) if k < len(cols) else (-inf, -1.0)
                got = (float(sl[t, k, 0]), float(sl[t, k, 1]))
                assert got == want, f"candidates NaN V={V} thread {t} slot {k}: {got} != {want}"


def pin_candidates_torch_topk(orc):
    """Rows of distinct values: each thread's slots are torch.topk (a library
    routine) of the values at its columns, in order, with their columns."""
    rng = np.random.default_rng(51)
    for V, S in ((1, 1), (300, 300), (1023, 1030), (5003, 5003)):
        x = np.full((3, S), 1e30, dtype=np.float32)
        x[:, :V] = rng.permutation(3 * V).reshape(3, V).astype(np.float32) * 0.5 - V
        cand = orc.candidates(x, V)
        for i in range(3):
            sl = _slots(cand[i])
            for t in range(_CT):
                vals = torch.from_numpy(x[i, t:V:_CT].copy())
                k = min(_CK, vals.numel())
                if k:
                    tv, ti = torch.topk(vals, k, sorted=True)
                    assert (sl[t, :k, 0] == tv.numpy()).all(), f"topk values V={V} t={t}"
                    assert (sl[t, :k, 1] == (t + _CT * ti.numpy()).astype(np.float32)).all(), \
                        f"topk columns V={V} t={t}"
                assert (sl[t, k:, 0] == -np.inf).all() and (sl[t, k:, 1] == -1).all()


def pin_candidates_invariants(orc):
    """Rows full of ties (small integers) and NaN: every slot is (x[c], c) with
    c = t mod 256; a thread's slots are ordered; it keeps min(4, its non-NaN
    values); the row's four best (value, then the lower column) are all kept,
    and the best is torch.argmax's first maximal index on NaN-free rows."""
    rng = np.random.default_rng(61)
    for V in (5, 300, 1025, 4099):
        x = rng.integers(0, 6, size=(4, V)).astype(np.float32)
        x[1, rng.integers(0, V, size=V // 3)] = np.nan
        cand = orc.candidates(x, V)
        for i in range(4):
            sl = _slots(cand[i])
            kept = set()
            for t in range(_CT):
                real = [(float(v), int(c)) for v, c in sl[t] if c >= 0]
                nn = int(np.count_nonzero(~np.isnan(x[i, t:V:_CT])))
                assert len(real) == min(_CK, nn), f"kept count V={V} t={t}"
                for v, c in real:
                    assert c % _CT == t and x[i, c] == v, f"slot ({v}, {c}) of thread {t}"
                keys = [(-v, c) for v, c in real]
                assert keys == sorted(keys), f"slot order V={V} t={t}"
                kept.update(c for _, c in real)
            order = sorted((-float(x[i, j]), j) for j in range(V) if not math.isnan(x[i, j]))
            assert all(c in kept for _, c in order[:_CK]), f"row top-4 missing V={V}"
            best = min((-float(v), int(c)) for v, c in sl.reshape(-1, 2) if c >= 0)
            if not np.isnan(x[i]).any():
                assert best[1] == int(torch.argmax(torch.from_numpy(x[i]))), "best candidate"


# ---------------------------------------------------------------------------
# split sums (splitSumInto)


def pin_split_sum(orc):
    """Small integers sum exactly in any order; random parts against math.fsum;
    add = 0 never reads y (NaN there changes nothing); one part is a copy."""
    rng = np.random.default_rng(71)
    for splits, total in ((1, 5), (2, 7), (5, 1000), (13, 3)):
        parts = rng.integers(-50, 50, size=(splits, total)).astype(np.float32)
        y = rng.integers(-50, 50, size=total).astype(np.float32)
        want = parts.astype(np.int64).sum(axis=0)
        _close(orc.split_sum(y, parts, add=True), want + y.astype(np.int64), rel=0, what="add")
        _close(orc.split_sum(np.full(total, np.nan, np.float32), parts, add=False), want, rel=0,
               what="no add")
        parts = rng.standard_normal((splits, total)).astype(np.float32) * 1e3
        y = rng.standard_normal(total).astype(np.float32)
        want = [math.fsum([float(y[i])] + [float(v) for v in parts[:, i]]) for i in range(total)]
        _close(orc.split_sum(y, parts, add=True), want, rel=1e-12, abs_=1e-9, what="fsum")
    one = rng.standard_normal((1, 9)).astype(np.float32)
    _close(orc.split_sum(np.zeros(9, np.float32), one, add=False), one[0], rel=0, what="one part")
    assert orc.split_sum(np.zeros(0, np.float32), np.zeros((3, 0), np.float32), add=True).shape == (0,)


# ---------------------------------------------------------------------------
# vocab-sharded rows: slice statistics and their combination


def _random_cuts(rng, V, shards):
    cuts = sorted(rng.choice(np.arange(1, V), size=shards - 1, replace=False).tolist()) if shards > 1 else []
    return [0] + cuts + [V]


def pin_sharded_equals_whole_rows(orc):
    """For any split of the columns, combining the slices' statistics gives
    the whole row's loss (crossEntropyRows), its argmax token and its max;
    rows with NaN, +inf, all -inf, slices all -inf or all NaN, ties across
    slice boundaries and labels out of range included."""
    rng = np.random.default_rng(81)
    nan, inf = float("nan"), float("inf")
    R, V = 14, 97
    x = (4 * rng.standard_normal((R, V))).astype(np.float32)
    x[0, 5] = nan
    x[1, 60] = inf
    x[2, :] = -inf
    x[3, :40] = -inf                   # a slice may be all -inf (masked)
    x[4, :50] = nan                    # a slice may be all NaN
    x[5, :] = 1.0                      # ties everywhere
    x[6, 10] = x[6, 70] = 30.0         # the max twice, in different slices
    x[7, :] = -inf
    x[7, 80] = 2.0                     # one finite value
    x[8, 3] = 60.0                     # the label far below a dominant token
    x[9, :] = x[9, :] - 200.0
    labels = rng.integers(0, V, size=R).astype(np.int64)
    labels[8] = 3                      # a tiny loss: label at the max, the rest far below
    labels[4] = 90                     # a finite label column: only the NaN slice makes the loss NaN
    labels[10] = -1
    labels[11] = V
    whole = orc.ce_rows(x, V, labels)
    arg = orc.argmax(x, V)
    fixed = [[0, 40, V], [0, 50, V], [0, 10, 70, V], [0, 3, 4, V]]   # slices all -inf, all NaN, the max alone
    random_cuts = [_random_cuts(rng, V, shards) for shards in (1, 2, 3, 5, 9) for _ in range(4)]
    for cuts in fixed + random_cuts:
        st = np.stack([orc.ce_stats(x, a, b - a, labels) for a, b in zip(cuts, cuts[1:])])
        comb = orc.ce_stats_combine(st, V, labels)
        _close(comb["loss"], whole, rel=1e-12, abs_=1e-300, what=f"sharded loss {cuts}")
        assert (comb["top"] == arg).all(), f"sharded token {cuts}: {comb['top']} != {arg}"
        fin = ~np.isnan(whole)
        _close(comb["m"][fin], np.nanmax(x[fin], axis=1), rel=0, what="sharded max")


def pin_stats_closed_forms(orc):
    """A constant slice: m = c, t = width - 1, top = its first column; x[label]
    only from the slice that holds the label (0 elsewhere); a slice with a NaN
    has t = NaN; an all -inf slice has m = -inf, t = 0, top = its first column;
    an all-NaN slice has top = -1."""
    nan, inf = float("nan"), float("inf")
    x = np.array([[2.5] * 10, [1.0, nan, 3.0] + [0.0] * 7, [-inf] * 10, [nan] * 10], dtype=np.float32)
    labels = np.array([7, 2, 4, 0], dtype=np.int64)
    st = orc.ce_stats(x, 4, 5, labels)      # columns 4..8
    _close(st[0], [2.5, 4.0, 4.0, 2.5], rel=0, what="constant slice")
    assert st[1][0] == 0.0 and st[1][2] == 4.0 and st[1][3] == 0.0, st[1]   # label 2 is outside
    _close(st[2], [-inf, 0.0, 4.0, -inf], rel=0, what="all -inf slice (its label column is -inf)")
    assert np.isneginf(st[3][0]) and st[3][2] == -1.0, st[3]
    st2 = orc.ce_stats(x, 0, 3, labels)     # columns 0..2 of the NaN row
    assert st2[1][0] == 3.0 and np.isnan(st2[1][1]) and st2[1][2] == 2.0 and st2[1][3] == 3.0, st2[1]
    # two slices of a constant row: T = V - 1, loss = log V
    comb = orc.ce_stats_combine(np.stack([orc.ce_stats(x, 0, 4, labels), orc.ce_stats(x, 4, 6, labels)]), 10,
                                labels)
    _close(comb["t"][0], 9.0, rel=0, what="constant row T")
    _close(comb["loss"][0], math.log(10), rel=1e-15, what="constant row loss")


PINS = [
    pin_uniform_rows, pin_two_class_closed_form, pin_tiny_loss, pin_bruteforce_tiny,
    pin_torch_cross_entropy, pin_central_differences, pin_grad_invariants,
    pin_shift_invariance, pin_mean, pin_nonfinite_rows, pin_bad_label, pin_stride_padding,
    pin_argmax_bruteforce, pin_argmax_nan_rules, pin_golden_closed_forms,
    pin_softmax_closed_forms, pin_softmax_torch, pin_softmax_invariants,
    pin_candidates_closed_forms, pin_candidates_torch_topk, pin_candidates_invariants,
    pin_split_sum, pin_sharded_equals_whole_rows, pin_stats_closed_forms,
]


def failing_pins(orc):
    """Names of the pins that ``orc`` fails (for the mutation test)."""
    bad = []
    for p in PINS:
        try:
            p(orc)
        except Exception:  # a crash or a wrong value both count as caught
            bad.append(p.__name__)
    return bad
