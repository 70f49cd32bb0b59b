"""The tensor-core router's recomputation rule (CPU model): which experts are recomputed in fp32 before
the final selection, and why the selection and its order are then those of the exact logits.

The rule (include/k3moe.h, k3moe_route): the first selection ranks the tensor-core logits (descending,
ties to the lower id); v_k is the k-th selected value. If an unselected expert lies within the margin
below v_k the boundary is tight, and those experts are recomputed together with the selected ones
within the margin above v_k. Every selected expert within the margin of a selected neighbour is
recomputed too. With nothing to recompute the first selection stands; otherwise the experts are
ranked again on the recomputed values and the tensor-core values of the others.

When every tensor-core logit is within delta of the exact one and 2 delta is below the margin, the
final selection equals the exact one, order included. This test checks that claim on adversarial logit
sets (near-ties across the k-th place and inside the selection, exact ties, clusters of the margin's
size) with perturbations up to delta.
"""
import numpy as np

MARGIN = 2e-4


def select(vals, k):
    order = np.lexsort((np.arange(len(vals)), -vals))  # descending value, then the lower id
    return order[:k]


def refine(approx, exact, k, margin=MARGIN):
    sel = select(approx, k)
    vk = approx[sel[-1]]
    unsel = np.ones(len(approx), bool)
    unsel[sel] = False
    below = np.nonzero(unsel & (approx >= vk - margin))[0]
    tight = below.size > 0
    cand = set(below.tolist())
    for i, e in enumerate(sel):
        v = approx[e]
        if (tight and v - vk <= margin) or (i > 0 and approx[sel[i - 1]] - v < margin) or \
                (i + 1 < k and v - approx[sel[i + 1]] < margin):
            cand.add(int(e))
    if not cand:
        return sel, 0
    mixed = approx.copy()
    idx = np.array(sorted(cand))
    mixed[idx] = exact[idx]
    return select(mixed, k), len(cand)


def adversarial_logits(rng, E, k):
    """Logits with structure near the k-th place and inside the top k."""
    ex = rng.standard_normal(E) * 0.05
    top = np.argsort(-ex)[: k + 8]
    kth = ex[top[k - 1]]
    gaps = np.array([0.0, 1e-6, 5e-6, 1e-5, 2e-5, 6e-5, 1e-4, 1.5e-4, 1.99e-4, 2.01e-4, 3e-4])
    # experts just above and below the k-th place, at the gaps above
    for j, e in enumerate(top[k - 4: k + 6]):
        ex[e] = kth + rng.choice([-1, 1]) * rng.choice(gaps)
    # near-ties and exact ties inside the selection
    for j in range(0, k - 6, 3):
        a, b = top[j], top[j + 1]
        ex[b] = ex[a] - rng.choice(gaps)
    # an exact tie straddling the k-th place, sometimes
    if rng.random() < 0.3:
        ex[top[k]] = ex[top[k - 1]]
    return ex


def test_rule_restores_the_exact_selection():
    rng = np.random.default_rng(16)
    E, k, delta = 896, 16, 0.45 * MARGIN  # 2 delta below the margin
    first_wrong = 0
    recomputed = 0
    for _ in range(3000):
        exact = adversarial_logits(rng, E, k)
        approx = exact + rng.uniform(-delta, delta, E)
        want = select(exact, k)
        got, n = refine(approx, exact, k)
        assert np.array_equal(got, want)
        first_wrong += not np.array_equal(select(approx, k), want)
        recomputed += n > 0
    # the cases were hard: the first selection alone was wrong in many of them
    assert first_wrong > 500 and recomputed > first_wrong


def test_nothing_recomputed_when_the_selection_is_well_separated():
    rng = np.random.default_rng(3)
    E, k = 896, 16
    exact = np.arange(E, dtype=np.float64)[rng.permutation(E)] * 1e-3  # all gaps 1e-3 > margin
    approx = exact + rng.uniform(-1e-5, 1e-5, E)
    got, n = refine(approx, exact, k)
    assert n == 0 and np.array_equal(got, select(exact, k))


def test_margin_is_needed():
    """With tensor-core errors above half the margin the rule can fail: the claim's condition matters."""
    rng = np.random.default_rng(5)
    E, k, delta = 896, 16, 3.0 * MARGIN
    fails = 0
    for _ in range(500):
        exact = adversarial_logits(rng, E, k)
        approx = exact + rng.uniform(-delta, delta, E)
        fails += not np.array_equal(refine(approx, exact, k)[0], select(exact, k))
    assert fails > 0
