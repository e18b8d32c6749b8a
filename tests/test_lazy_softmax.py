"""Host check of the online-softmax recurrence the draft decode kernel runs
per 32-token chunk of each page: the running maximum m moves only when a
score leads it by more than 2^5 (then m = max(m, chunk maximum)); the
probabilities are p = 2^(s - (m - 10)) (0 for a masked score, reference 0
while no score has been seen), the accumulators are rescaled by 2^(m_old -
m_new) when m moves.  The recurrence must give the exact softmax-weighted
sum and log-sum-exp, and every p must stay below fp16's largest finite value
(65504), since the kernel rounds p to fp16 for the value-side MMA."""
import numpy as np
import pytest

LAZY = 5.0
FP16_MAX = 65504.0


def lazy_online(scores, values, chunk=32):
    """scores in the log2 domain, shape [n]; values [n, d]; returns (o, lse2, max p)."""
    m, l = -np.inf, 0.0
    o = np.zeros(values.shape[1])
    p_max = 0.0
    for c in range(0, len(scores), chunk):
        s = scores[c:c + chunk]
        v = values[c:c + chunk]
        cm = s.max()
        m_new = max(m, cm) if cm > m + LAZY else m
        corr = 1.0 if (m_new == m) else 2.0 ** (m - m_new)
        ref = 0.0 if m_new == -np.inf else m_new - 10.0
        p = np.where(np.isneginf(s), 0.0, 2.0 ** (s - ref))
        p_max = max(p_max, float(p.max(initial=0.0)))
        l = l * corr + p.sum()
        o = o * corr + p @ v
        m = m_new
    ref = 0.0 if m == -np.inf else m - 10.0
    return o / l, np.log2(l) + ref, p_max


def exact(scores, values):
    w = 2.0 ** (scores - scores.max())
    return (w @ values) / w.sum(), np.log2(w.sum()) + scores.max()


@pytest.mark.parametrize("case", ["random", "rising", "falling", "steps", "masked_head"])
@pytest.mark.parametrize("spread", [1.0, 8.0, 60.0])
def test_lazy_maximum_recurrence(case, spread):
    rng = np.random.default_rng(7)
    n, d = 16 * 256, 8
    s = rng.standard_normal(n) * spread
    if case == "rising":
        s = np.sort(s)
    elif case == "falling":
        s = np.sort(s)[::-1]
    elif case == "steps":     # jumps of just under and just over the threshold
        s = np.repeat(np.arange(n // 32) * (LAZY - 0.01 if spread < 8 else LAZY + 0.01), 32).astype(float)
    elif case == "masked_head":
        s[: n // 3] = -np.inf
    v = rng.standard_normal((n, d))
    o, lse, p_max = lazy_online(s, v)
    ro, rlse = exact(s, v)
    assert np.allclose(o, ro, rtol=1e-12, atol=1e-12)
    assert abs(lse - rlse) <= 1e-12 * max(1.0, abs(rlse))
    assert p_max < FP16_MAX
    assert p_max <= 2.0 ** (10 + LAZY)
