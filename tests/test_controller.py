"""The draft-depth controller (host code behind the C ABI): expected committed
run against its closed form, the observation bookkeeping, the choice against
brute force, and convergence on synthetic acceptance traces.  No GPU."""

import numpy as np
import pytest

import speculative_decode_verification_w4_gb300 as vw4


def expected_run(alphas, depth):
    """sum_{j=0..depth} prod_{i<j} alpha_i, written out term by term."""
    total = 0.0
    for j in range(depth + 1):
        total += float(np.prod(alphas[:j])) if j else 1.0
    return total


def test_fresh_state_reads_one_half_everywhere():
    c = vw4.DepthController(k_max=7)
    for k in range(8):
        t, us = c.expected(k)
        assert t == pytest.approx(2.0 - 0.5 ** k)   # 1 + 1/2 + ... + 1/2^k
        assert us == pytest.approx(1.0)


def test_observe_counts_the_prefix_and_the_first_rejection():
    c = vw4.DepthController(k_max=7, decay=1.0)
    c.observe(4, 2)      # drafts 0, 1 accepted; draft 2 rejected; 3 unknown
    c.observe(3, 3)      # all three accepted
    c.observe(0, 0)      # plain decoding: nothing drafted
    att = list(c.state.att)
    acc = list(c.state.acc)
    assert att[:5] == [2.0, 2.0, 2.0, 0.0, 0.0]
    assert acc[:5] == [2.0, 2.0, 1.0, 0.0, 0.0]


def test_decay_weights_old_observations_down():
    c = vw4.DepthController(k_max=3, decay=0.5)
    c.observe(1, 1)
    c.observe(1, 0)
    assert c.state.att[0] == pytest.approx(1.5)     # 1 * 0.5 + 1
    assert c.state.acc[0] == pytest.approx(0.5)


@pytest.mark.parametrize("seed,k_max", [(s, 7) for s in range(5)] + [(s, 15) for s in range(5, 8)])
def test_expected_and_choice_match_brute_force(seed, k_max):
    g = np.random.default_rng(seed)
    c = vw4.DepthController(k_max=k_max, decay=1.0, draft_us_fixed=float(g.uniform(0, 20)),
                            draft_us_per_token=float(g.uniform(0, 10)),
                            verify_us={w: float(50 + 8 * w + g.uniform(0, 5))
                                       for w in range(1, k_max + 2)})
    for _ in range(200):
        d = int(g.integers(0, k_max + 1))
        c.observe(d, int(g.integers(0, d + 1)))
    alphas = [(c.state.acc[i] + 1.0) / (c.state.att[i] + 2.0) for i in range(k_max + 1)]
    rates = []
    for k in range(k_max + 1):
        t, us = c.expected(k)
        assert t == pytest.approx(expected_run(alphas, k), rel=1e-12)
        cost = c.state.verify_us[k + 1] + (c.state.draft_us_fixed +
                                          k * c.state.draft_us_per_token if k else 0.0)
        assert us == pytest.approx(cost, rel=1e-6)
        rates.append(t / us)
    assert c.choose() == int(np.argmax(rates))   # argmax: first of the maxima


def test_falls_back_to_plain_decoding_when_drafts_are_rejected():
    c = vw4.DepthController(k_max=7, decay=1.0, draft_us_per_token=5.0,
                            verify_us={w: 100.0 + 2.0 * w for w in range(1, 9)})
    for _ in range(100):
        c.observe(3, 0)
    assert c.choose() == 0


def test_drafts_past_eight_when_sixteen_row_verify_is_cheap():
    """Verify widths up to 16 rows: with a flat verify cost and near-certain
    acceptance the deepest depth, 15, wins."""
    c = vw4.DepthController(k_max=15, decay=1.0, draft_us_per_token=1.0,
                            verify_us={w: 100.0 for w in range(1, 17)})
    for _ in range(200):
        c.observe(15, 15)
    assert c.choose() == 15
    t, _ = c.expected(15)
    assert 15.0 < t <= 16.0


def test_drafts_deep_when_verify_width_is_cheap_and_acceptance_high():
    c = vw4.DepthController(k_max=7, decay=1.0, draft_us_per_token=1.0,
                            verify_us={w: 100.0 for w in range(1, 9)})
    for _ in range(100):
        c.observe(7, 7)
    assert c.choose() == 7


def simulate(true_alpha, verify_us, draft_fixed, draft_per, steps, seed):
    """A synthetic acceptance trace driven by the controller's own choices:
    at depth K, draft i is accepted with probability true_alpha[i] given its
    prefix was; the controller sees every committed run."""
    g = np.random.default_rng(seed)
    c = vw4.DepthController(k_max=7, decay=0.995, verify_us=verify_us,
                            draft_us_fixed=draft_fixed, draft_us_per_token=draft_per)
    tokens = us = 0.0
    depths = []
    for step in range(steps):
        explore = step % 10 == 0                 # an exploring step every 10
        k = 7 if explore else c.choose()
        n = 0
        while n < k and g.random() < true_alpha[n]:
            n += 1
        c.observe(k, n)
        if not explore and step >= steps // 2:   # the controller's own steps, settled
            tokens += n + 1
            us += verify_us[k + 1] + (draft_fixed + k * draft_per if k else 0.0)
        depths.append(k)
    return c, tokens / us, depths


def true_rates(true_alpha, verify_us, draft_fixed, draft_per):
    out = []
    for k in range(8):
        t = expected_run(true_alpha, k)
        out.append(t / (verify_us[k + 1] + (draft_fixed + k * draft_per if k else 0.0)))
    return out


@pytest.mark.parametrize("case", [
    # acceptance falls off after three positions; verify cost grows with width
    ([0.85, 0.8, 0.75, 0.1, 0.1, 0.1, 0.1], {w: 60.0 + 6.0 * w for w in range(1, 9)}, 5.0, 4.0),
    # a steep forward cost: wider verify passes cost much more
    ([0.6] * 7, {w: 40.0 * w for w in range(1, 9)}, 2.0, 2.0),
    # a flat forward cost and good drafts
    ([0.9] * 7, {w: 100.0 for w in range(1, 9)}, 1.0, 1.0),
])
def test_converges_on_synthetic_acceptance_traces(case):
    true_alpha, verify_us, draft_fixed, draft_per = case
    best = true_rates(true_alpha, verify_us, draft_fixed, draft_per)
    k_star = int(np.argmax(best))
    c, rate, depths = simulate(true_alpha, verify_us, draft_fixed, draft_per, 3000, 11)
    # after the estimates settle the choice is the best depth (or one within
    # 2 % of its rate), and the throughput of the controller's own steps is
    # close to the optimum
    late = [d for i, d in enumerate(depths[-500:]) if i % 10]
    top = max(best)
    good = {k for k in range(8) if best[k] >= 0.98 * top}
    assert k_star in good
    assert np.mean([d in good for d in late]) > 0.9
    assert rate > 0.9 * top


def test_invalid_arguments():
    c = vw4.DepthController(k_max=3)
    with pytest.raises(vw4.VW4Error):
        c.observe(4, 0)
    with pytest.raises(vw4.VW4Error):
        c.observe(2, 3)
    with pytest.raises(vw4.VW4Error):
        vw4.DepthController(k_max=16)
    c.state.verify_us[2] = 0.0
    with pytest.raises(vw4.VW4Error):
        c.choose()


def test_zero_filled_state_is_rejected_until_init():
    """A zero-filled state is invalid (decay 0, verify costs 0), as the header
    says: choose returns -1 and observe / expected fail; after
    vw4_depth_ctl_init the same struct works."""
    import ctypes
    lib = vw4.load_library()
    st = vw4.DepthCtl()          # ctypes zero-fills
    assert lib.vw4_depth_ctl_choose(ctypes.byref(st)) == -1
    assert lib.vw4_depth_ctl_observe(ctypes.byref(st), 0, 0) == 1
    t, us = ctypes.c_double(), ctypes.c_double()
    assert lib.vw4_depth_ctl_expected(ctypes.byref(st), 0, ctypes.byref(t), ctypes.byref(us)) == 1
    assert lib.vw4_depth_ctl_init(ctypes.byref(st), 3, 1.0) == 0
    assert lib.vw4_depth_ctl_choose(ctypes.byref(st)) in range(4)
    assert lib.vw4_depth_ctl_observe(ctypes.byref(st), 2, 1) == 0
