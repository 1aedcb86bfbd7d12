"""The INT8 epilogue's fast path: exact by an error bound (CPU checks).

The kernels compute a code first with the hardware approximations
(ex2.approx for the exp, rcp.approx for the division) and keep it only when
the value w = SiLU(t)/s_y lies farther from every rounding boundary (a
half-integer) than a bound on |w_fast - w_specified|; otherwise they run the
specified steps.  The bound (|w| (f (1.5e-6 + 2.4e-7 |t|) + 1.2e-6), f an
upper bound of e^-t/(1+e^-t)) is at least twice the first-order error of the
two evaluations when the specified exp is within 1.2e-7 relative, ex2.approx
within 4.8e-7 and rcp.approx within 2.4e-7 (all for |t| <= 80).  These tests
check the exp's bound exhaustively and the decision rule against the oracle
with approximations placed adversarially at the edges of their bounds; the
hardware bounds themselves are checked on the GPU (test_hw_approx.py)."""
import numpy as np

import oracle

F = np.float32
A_SPEC = 1.2e-7      # specified exp, relative
A_EX2 = 4.8e-7       # ex2.approx.ftz.f32, relative (GPU-checked)
R_RCP = 2.4e-7       # rcp.approx.ftz.f32, relative (GPU-checked)
NEG_LOG2E = F(-1.4426950408889634)


def test_spec_exp_error_within_the_assumed_bound():
    """Every float x in [-80, 80] (the fast path's range of -t): the
    specified exp is within A_SPEC relative of the true exp."""
    assert oracle.spec_exp_max_rel_err(-80.0, 80.0) <= A_SPEC


def fast_codes(acc, m_c, inv, z, gamma, rho):
    """The fast path in float32 steps, with ex2 and rcp replaced by the exact
    values times (1 + gamma) and (1 + rho).  Returns (accepted, code)."""
    t = (acc.astype(F) * m_c).astype(F)
    y = (t * NEG_LOG2E).astype(F)
    e = (np.exp2(y.astype(np.float64)) * (1 + gamma)).astype(F)
    d = (F(1) + e).astype(F)
    r = ((1.0 / d.astype(np.float64)) * (1 + rho)).astype(F)
    w = ((t * r).astype(F) * F(inv)).astype(F)
    k = np.rint(w).astype(F)
    dist = (F(0.5) - np.abs((w - k).astype(F))).astype(F)
    f = np.minimum(F(1), (e * F(1.001)).astype(F))
    bound = (np.abs(w).astype(np.float64) * (f.astype(np.float64) * (1.5e-6 + 2.4e-7 * np.abs(t.astype(np.float64)))
                                             + 1.2e-6)).astype(F)
    ok = (np.abs(t) <= 80) & (dist > bound)
    code = np.clip(k + F(z), -128, 127).astype(np.int8)
    return ok, code


def boundary_heavy_samples(rng, count):
    """Accumulators whose pre-activations t = acc m_c follow the layers'
    N(0, 3) spread, half of them moved to the accumulator that puts w
    closest to a half-integer (where a wrong decision would show).  Returns
    (acc, m_c, inv_s_y, moved)."""
    m_c = rng.uniform(2e-5, 3e-3, count).astype(F)
    inv = F(rng.uniform(5.0, 80.0))
    t0 = np.clip(rng.normal(0.0, 3.0, count), -20, 20)
    acc = np.round(t0 / m_c).astype(np.int64)
    t = acc * m_c.astype(np.float64)
    sig = 1 / (1 + np.exp(-t))
    w = t * sig * inv
    half = np.floor(w) + 0.5
    slope = np.maximum(np.abs(sig * (1 + t * (1 - sig))) * inv * m_c, 1e-9)
    moved = rng.random(count) < 0.5
    acc = np.where(moved, acc + np.round((half - w) / slope), acc)
    return np.clip(acc, -2**31, 2**31 - 1).astype(np.int32), m_c, inv, moved


def test_fast_decision_agrees_with_the_oracle_under_adversarial_approximations():
    rng = np.random.default_rng(1)
    total, accepted = 0, 0
    for trial in range(6):
        acc, m_c, inv, moved = boundary_heavy_samples(rng, 400000)
        z = int(rng.integers(-128, 128))
        want = oracle.requant_array(acc, m_c, float(inv), z)
        for gamma in (A_EX2, -A_EX2, 0.0):
            for rho in (R_RCP, -R_RCP):
                ok, code = fast_codes(acc, m_c, inv, z, gamma, rho)
                bad = np.count_nonzero(ok & (code != want))
                assert bad == 0, (trial, gamma, rho, bad)
                total += int((~moved).sum())
                accepted += int((ok & ~moved).sum())
    # Away from the planted boundary cases almost every value takes the fast path.
    assert accepted / total > 0.999, accepted / total


def test_a_bound_without_margin_is_caught():
    """The same check with the bound scaled far down (a dropped term) accepts
    values it must not: the samples do reach the rounding boundaries."""
    rng = np.random.default_rng(2)
    acc, m_c, inv, _ = boundary_heavy_samples(rng, 400000)
    want = oracle.requant_array(acc, m_c, float(inv), 0)
    t = (acc.astype(F) * m_c).astype(F)
    bad = 0
    for gamma, rho in ((A_EX2, R_RCP), (-A_EX2, -R_RCP)):
        y = (t * NEG_LOG2E).astype(F)
        e = (np.exp2(y.astype(np.float64)) * (1 + gamma)).astype(F)
        d = (F(1) + e).astype(F)
        r = ((1.0 / d.astype(np.float64)) * (1 + rho)).astype(F)
        w = ((t * r).astype(F) * F(inv)).astype(F)
        k = np.rint(w).astype(F)
        code = np.clip(k, -128, 127).astype(np.int8)
        bad += np.count_nonzero((np.abs(t) <= 80) & (code != want))
    assert bad > 0
