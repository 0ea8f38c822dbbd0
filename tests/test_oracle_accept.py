"""Pins for the oracle's greedy and sampled acceptance.

Greedy ("VFlash-FM" project page, "How VFlash-FM works" and its worked
cycle): the longest prefix of proposals equal to the target's greedy picks is
accepted and the target's own pick at the first mismatch is appended; the
output must equal autoregressive greedy decoding token for token.

Sampled ("SpecFLASH" README, inference section: the standard speculative
accept/reject rule, lossless): committed tokens must follow the target
distribution exactly.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from serving_sd_verify_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# greedy
# --------------------------------------------------------------------------

def test_worked_cycle_from_the_project_page():
    g = json.load(open(os.path.join(GOLDEN, "worked_cycle.json")))
    T, V = 16, g["vocab"]
    logits = np.zeros((1, T, V))
    for j, t in enumerate(g["target_choice"]):
        logits[0, j, t] = 1.0
    n, c = oracle.accept_greedy(np.array([g["draft"]]), logits)
    assert int(n[0]) == g["expect"]["n_accepted"]
    assert int(c[0]) == g["expect"]["correction"]
    committed = g["draft"][: int(n[0])] + [int(c[0])]
    assert len(committed) == g["expect"]["committed"]
    assert committed[-1] == g["expect"]["next_anchor"]


def test_ties_go_to_lowest_index():
    logits = np.zeros((1, 3, 10))
    logits[0, 0, [3, 7]] = 5.0
    logits[0, 1, [9, 2, 4]] = 1.0
    logits[0, 2, :] = -1.0
    n, c, am = oracle.accept_greedy(np.array([[3, 2]]), logits, return_argmax=True)
    assert am.tolist() == [[3, 2, 0]]
    assert int(n[0]) == 2 and int(c[0]) == 0
    n, c = oracle.accept_greedy(np.array([[7, 2]]), logits)  # 7 ties 3 but loses
    assert int(n[0]) == 0 and int(c[0]) == 3


def test_block_of_one_is_plain_greedy_decode():
    rng = np.random.default_rng(0)
    logits = rng.standard_normal((4, 1, 50))
    n, c = oracle.accept_greedy(np.zeros((4, 0), dtype=np.int32), logits)
    assert n.tolist() == [0] * 4
    assert c.tolist() == [int(np.argmax(logits[b, 0])) for b in range(4)]


def test_all_accepted_gives_bonus_token():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((1, 16, 40))
    am = logits[0].argmax(-1)
    n, c = oracle.accept_greedy(am[None, :15], logits)
    assert int(n[0]) == 15 and int(c[0]) == int(am[15])


@pytest.mark.parametrize("B,V,dtype,sd", [(1, 1000, torch.float32, 2.0),
                                          (4, 5000, torch.bfloat16, 3.0),
                                          (8, 3000, torch.bfloat16, 3.0)])
def test_generator_known_answers(B, V, dtype, sd):
    inp = W.greedy_inputs(B=B, T=16, V=V, dtype=dtype, sd=sd, seed=B)
    n, c, am = oracle.accept_greedy(inp["draft"], inp["logits"], return_argmax=True)
    assert n.tolist() == inp["k"]
    assert c.tolist() == [int(am[b, inp["k"][b]]) for b in range(B)]


def test_workload1_known_answer():
    cfg = W.config(1)
    n, _ = oracle.accept_greedy(cfg["greedy"]["draft"], cfg["greedy"]["logits"])
    assert int(n[0]) == 5


def _toy_lm(prefix, V=12):
    """Deterministic toy language model: logits from a hash of the prefix."""
    h = hash(tuple(prefix)) & 0xFFFFFFFF
    return np.random.default_rng(h).standard_normal(V) * 2.0


def test_greedy_speculation_reproduces_autoregressive_decoding():
    V, T, n_new = 12, 16, 80
    prompt = [1, 5, 7]
    ar = list(prompt)
    while len(ar) < len(prompt) + n_new:
        ar.append(int(np.argmax(_toy_lm(ar, V))))
    rng = np.random.default_rng(7)
    seq = list(prompt)
    cycles, lens = 0, []
    while len(seq) < len(prompt) + n_new:
        # a drafter that is right most of the time, wrong sometimes
        drafts = []
        for j in range(T - 1):
            pos = len(seq) + j
            right = ar[pos] if pos < len(ar) else 0
            drafts.append(right if rng.random() < 0.8 else int(rng.integers(0, V)))
        logits = np.stack([_toy_lm(seq + drafts[:j], V) for j in range(T)])[None]
        n, c = oracle.accept_greedy(np.array([drafts]), logits)
        seq += drafts[: int(n[0])] + [int(c[0])]
        cycles += 1
        lens.append(int(n[0]))
    assert seq[: len(ar)] == ar[: len(seq)]
    assert cycles < n_new          # it did speculate
    assert len(set(lens)) > 1     # accept lengths vary across cycles


# --------------------------------------------------------------------------
# sampled
# --------------------------------------------------------------------------

def _softmax(x, axis=-1):
    z = x - x.max(axis=axis, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=axis, keepdims=True)


def test_p_equal_q_accepts_everything():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((64, 16, 30)) * 2
    q = _softmax(logits)
    drafts = np.array([[rng.choice(30, p=q[b, j]) for j in range(15)] for b in range(64)])
    n, nx, diag = oracle.accept_sample(drafts, q, logits, 1.0, 99, return_diag=True)
    # u < 1 = p/q for every row up to rounding of p vs q
    ratio = oracle.split_diag(diag, 16)["ratio"]
    assert np.all(np.abs(ratio - 1.0) < 1e-12)
    assert n.tolist() == [15] * 64


def test_temperature_scales_the_logits():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((16, 16, 20)) * 2
    tau = 0.6
    q = _softmax(logits / tau)
    drafts = np.array([[rng.choice(20, p=q[b, j]) for j in range(15)] for b in range(16)])
    n, _ = oracle.accept_sample(drafts, q, logits, tau, 5)
    assert n.tolist() == [15] * 16
    n_wrong, _ = oracle.accept_sample(drafts, _softmax(logits), logits, tau, 5)
    assert min(n_wrong.tolist()) < 15


def test_zero_target_prob_rejects_then_draws_from_p():
    V = 8
    logits = np.log(np.array([[0.5, 0.0, 0.25, 0.25, 0, 0, 0, 0]]) + 1e-300)
    logits = np.repeat(logits[None], 2, axis=1).reshape(1, 2, V)
    q = np.zeros((1, 2, V))
    q[0, :, 1] = 1.0  # the drafter is sure of a token the target never picks
    for off in range(50):
        n, nx = oracle.accept_sample(np.array([[1]]), q, logits, 1.0, 11, off)
        assert int(n[0]) == 0
        assert int(nx[0]) in (0, 2, 3)


def _committed_tokens(B, T, V, p_rows, q_rows, seed, offset):
    """Run the rule on B independent copies; return the first two committed tokens."""
    rng = np.random.default_rng(seed)
    logits = np.log(np.broadcast_to(p_rows, (B, T, V)))
    q = np.ascontiguousarray(np.broadcast_to(q_rows, (B, T, V)))
    cq = np.cumsum(q_rows, axis=-1)
    drafts = np.stack([np.searchsorted(cq[j], rng.random(B), side="right")
                       for j in range(T - 1)], axis=1).clip(0, V - 1)
    n, nx = oracle.accept_sample(drafts, q, logits, 1.0, seed, offset)
    first = np.where(n >= 1, drafts[:, 0], nx)
    if T >= 3:
        second = np.where(n >= 2, drafts[:, 1], np.where(n == 1, nx, -1))
    else:
        second = np.where(n == 1, nx, -1)
    return first, second, n


def test_sampled_tokens_follow_target_distribution_chi_square():
    stats = pytest.importorskip("scipy.stats")
    V, T, B = 16, 3, 400_000
    rng = np.random.default_rng(21)
    p_rows = _softmax(rng.standard_normal((T, V)) * 1.5)
    q_rows = _softmax(np.log(p_rows) + rng.standard_normal((T, V)))
    first, second, n = _committed_tokens(B, T, V, p_rows, q_rows, 1234, 0)
    assert 0.2 < (n == 0).mean() < 0.8  # both branches are exercised
    counts = np.bincount(first, minlength=V)
    _, pv = stats.chisquare(counts, B * p_rows[0])
    assert pv > 1e-3, pv
    sel = second >= 0
    counts2 = np.bincount(second[sel], minlength=V)
    _, pv2 = stats.chisquare(counts2, sel.sum() * p_rows[1])
    assert pv2 > 1e-3, pv2


def test_rejection_branch_draws_from_normalised_residual():
    stats = pytest.importorskip("scipy.stats")
    V, T, B = 16, 2, 300_000
    rng = np.random.default_rng(22)
    p_rows = _softmax(rng.standard_normal((T, V)) * 1.5)
    q_rows = _softmax(rng.standard_normal((T, V)) * 1.5)
    first, _, n = _committed_tokens(B, T, V, p_rows, q_rows, 77, 3)
    rej = n == 0
    r = np.maximum(p_rows[0] - q_rows[0], 0.0)
    counts = np.bincount(first[rej], minlength=V)
    exp = rej.sum() * r / r.sum()
    keep = exp > 0
    assert counts[~keep].sum() == 0
    _, pv = stats.chisquare(counts[keep], exp[keep])
    assert pv > 1e-3, pv


def test_sample_diag_reports_the_draw():
    inp = W.sample_inputs(B=3, T=16, V=500, seed=8)
    n, nx, diag = oracle.accept_sample(inp["draft"], inp["q"], inp["logits"], 1.0, 1234,
                                       return_diag=True)
    d = oracle.split_diag(diag, 16)
    for b in range(3):
        assert d["c_prev"][b] <= d["x"][b] < d["c_at"][b]
        assert d["x"][b] == pytest.approx(d["u2"][b] * d["S"][b], rel=1e-15)
        # scanned rows: accepted ones satisfy u < p/q, the stopping one does not
        for j in range(int(n[b])):
            assert d["u"][b, j] < d["ratio"][b, j]
        if n[b] < 15:
            assert not (d["u"][b, n[b]] < d["ratio"][b, n[b]])


def _all_accepted_setup(B, V, seed):
    """p = q on rows 0..T-2 (every proposal accepted), a different p on row T-1."""
    T = 16
    rng = np.random.default_rng(seed)
    p_rows = _softmax(rng.standard_normal((T, V)) * 1.5)
    q_rows = p_rows.copy()
    # the last row must differ from the one before it, or a draw from the
    # wrong row would go unnoticed
    assert np.abs(p_rows[T - 1] - p_rows[T - 2]).sum() > 0.5
    return T, p_rows, q_rows


def test_all_accepted_bonus_follows_last_row_chi_square():
    """With every proposal accepted, the extra token is drawn from p of the last
    row (the standard rule: the target's distribution after the last accepted
    proposal), so its frequencies follow that row and not the one before."""
    stats = pytest.importorskip("scipy.stats")
    V, B = 16, 200_000
    T, p_rows, q_rows = _all_accepted_setup(B, V, 31)
    logits = np.log(np.broadcast_to(p_rows, (B, T, V)))
    q = np.ascontiguousarray(np.broadcast_to(q_rows, (B, T, V)))
    rng = np.random.default_rng(4321)
    cq = np.cumsum(q_rows, axis=-1)
    drafts = np.stack([np.searchsorted(cq[j], rng.random(B), side="right")
                       for j in range(T - 1)], axis=1).clip(0, V - 1)
    n, nx = oracle.accept_sample(drafts, q, logits, 1.0, 4321, 0)
    assert (n == T - 1).all()
    counts = np.bincount(nx, minlength=V)
    _, pv = stats.chisquare(counts, B * p_rows[T - 1])
    assert pv > 1e-3, pv
    # the row before it is clearly rejected by the same test
    _, pv_wrong = stats.chisquare(counts, B * p_rows[T - 2])
    assert pv_wrong < 1e-12, pv_wrong


def test_all_accepted_bonus_uses_last_row_resample_stream():
    """The extra token's uniform is Philox word (row T-1, batch b, stream 1,
    offset), and the token is the inverse CDF of the last row's p at u'·S,
    recomputed here in numpy from the logits."""
    V, B = 40, 64
    T, p_rows, q_rows = _all_accepted_setup(B, V, 32)
    logits = np.log(np.broadcast_to(p_rows, (B, T, V)))
    q = np.ascontiguousarray(np.broadcast_to(q_rows, (B, T, V)))
    rng = np.random.default_rng(5)
    cq = np.cumsum(q_rows, axis=-1)
    drafts = np.stack([np.searchsorted(cq[j], rng.random(B), side="right")
                       for j in range(T - 1)], axis=1).clip(0, V - 1)
    for seed, offset in ((1234, 0), (77, 9)):
        n, nx, diag = oracle.accept_sample(drafts, q, logits, 1.0, seed, offset, return_diag=True)
        d = oracle.split_diag(diag, T)
        assert (n == T - 1).all()
        p_last = _softmax(logits[0, T - 1])
        cdf = np.cumsum(p_last)
        for b in range(B):
            u2 = oracle.uniform(seed, T - 1, b, 1, offset)
            assert d["u2"][b] == u2
            # neither the accept stream of that row nor the row before it
            assert u2 != oracle.uniform(seed, T - 1, b, 0, offset)
            assert u2 != oracle.uniform(seed, T - 2, b, 1, offset)
            x = u2 * cdf[-1]
            want = int(np.searchsorted(cdf, x, side="right"))
            near = np.min(np.abs(cdf - x)) < 1e-12
            assert int(nx[b]) == want or near, (b, int(nx[b]), want)
