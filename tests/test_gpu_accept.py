"""GPU parity of the acceptance kernels and Philox against the fp64 oracle.

Greedy: accept lengths and correction ids bit-exact (argmax compared on the
exact stored values, ties to the lowest index).  Sampled: ids and lengths
bit-exact except where the oracle's own diagnostics show the decision sits
within 1e-6 of a threshold (|u - p/q| < 1e-6, or u'*S within 1e-6*S of a
cumulative-sum boundary).
"""
import numpy as np
import pytest
import torch

import oracle
from serving_sd_verify_gb300 import workloads as W

pytestmark = pytest.mark.gpu

EXCUSE = 1e-6


@pytest.fixture(scope="module")
def S():
    from serving_sd_verify_gb300 import build, sd_verify
    build.build()
    sd_verify.load()
    return sd_verify


def run_greedy(S, draft, logits):
    B, T, V = logits.shape
    dl = logits.cuda()
    dd = draft.to(torch.int32).cuda().contiguous()
    n = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    c = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    ws = S.workspace(S.sd_accept_greedy_workspace_size(B, T, V, S._dt(logits)))
    S.sd_accept_greedy(dd, dl, n, c, ws)
    torch.cuda.synchronize()
    assert counters_zero(ws, 256), "ticket counter not returned to zero"
    return n.cpu().numpy(), c.cpu().numpy()


def counters_zero(ws, nbytes):
    """The acceptance workspaces start with their ticket counters (greedy: the
    first 256 bytes; sampled: 256 bytes, then one per sequence); every completed
    call leaves them at zero."""
    return int(ws[:nbytes].abs().sum()) == 0


@pytest.mark.parametrize("B,T,V,dtype", [
    (1, 16, 1000, torch.float32),
    (1, 16, 152_064, torch.bfloat16),
    (3, 16, 5_001, torch.bfloat16),     # odd V: rows not 16-byte aligned
    (2, 7, 777, torch.float32),
    (20, 16, 3_000, torch.bfloat16),    # more rows than one finisher window
    (5, 1, 4_096, torch.bfloat16),      # block of one = greedy decode
    (4, 3, 13, torch.bfloat16),         # tiny vocab, ragged window
])
def test_greedy_matches_oracle(S, B, T, V, dtype):
    inp = W.greedy_inputs(B=B, T=T, V=V, dtype=dtype, seed=B * 1000 + T)
    n, c = run_greedy(S, inp["draft"], inp["logits"])
    on, oc = oracle.accept_greedy(inp["draft"], inp["logits"])
    assert n.tolist() == on.tolist()
    assert c.tolist() == oc.tolist()
    assert n.tolist() == [min(k, T - 1) for k in inp["k"]]


def test_greedy_ties_lowest_index(S):
    V = 10_000
    lg = torch.zeros(2, 16, V, dtype=torch.bfloat16)
    lg[:, :, [17, 5000, 9999]] = 3.0  # triple tie in every row
    lg[1, 4, 9999] = 3.5
    draft = torch.full((2, 15), 17, dtype=torch.int32)
    n, c = run_greedy(S, draft, lg)
    on, oc = oracle.accept_greedy(draft, lg)
    assert n.tolist() == on.tolist() == [15, 4]
    assert c.tolist() == oc.tolist() == [17, 9999]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_greedy_vector_max_edges(S, dtype):
    """The stream takes each 16-byte vector's maximum first and searches a
    vector for its lowest index only when that maximum is new: rows that are
    all -inf, ties inside one vector and across vectors, a maximum in the
    unaligned head or tail, and rising rows where every vector is new."""
    V = 4_099                                      # odd: rows start unaligned
    T = 8
    lg = torch.randn(1, T, V).to(dtype)
    lg[0, 0] = -float("inf")                       # all -inf: index 0
    lg[0, 1, [1026, 1030, 3001]] = 9.0             # tie inside one vector, and a later one
    lg[0, 2] = torch.arange(V, dtype=torch.float32).to(dtype) / V   # rising (bf16 ties at the top)
    lg[0, 3, 0] = 20.0                             # in the unaligned head
    lg[0, 4, V - 1] = 20.0                         # in the tail
    lg[0, 5] = -float("inf")
    lg[0, 5, [7, 4000]] = -1.0                     # only two ordered values above -inf
    lg[0, 6] = 0.0                                 # all equal: index 0
    draft = torch.zeros((1, T - 1), dtype=torch.int32)
    on, oc, am = oracle.accept_greedy(draft, lg, return_argmax=True)
    assert am[0].tolist()[:7] == [0, 1026, int(am[0, 2]), 0, V - 1, 7, 0]
    for j in range(T):                             # each row as the rejected one
        d = am[0:1, :T - 1].astype(np.int32).copy()
        if j < T - 1:
            d[0, j] = (am[0, j] + 1) % V
        n, c = run_greedy(S, torch.from_numpy(d), lg)
        assert int(n[0]) == j and int(c[0]) == int(am[0, j]), (j, n, c, am[0, j])


def test_greedy_all_accepted_and_worked_cycle(S):
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_cycle.json")))
    lg = torch.zeros(1, 16, g["vocab"], dtype=torch.float32)
    for j, t in enumerate(g["target_choice"]):
        lg[0, j, t] = 1.0
    n, c = run_greedy(S, torch.tensor([g["draft"]], dtype=torch.int32), lg)
    assert int(n[0]) == g["expect"]["n_accepted"] and int(c[0]) == g["expect"]["correction"]


@pytest.mark.parametrize("n", [2, 3])
def test_greedy_full_size_workloads(S, n):
    cfg = W.config(n)
    g = cfg["greedy"]
    got_n, got_c = run_greedy(S, g["draft"], g["logits"])
    on, oc = oracle.accept_greedy(g["draft"], g["logits"])
    assert got_n.tolist() == on.tolist() == g["k"]
    assert got_c.tolist() == oc.tolist()


def test_greedy_workload1(S):
    g = W.config(1)["greedy"]
    got_n, got_c = run_greedy(S, g["draft"], g["logits"])
    on, oc = oracle.accept_greedy(g["draft"], g["logits"])
    assert got_n.tolist() == on.tolist() == [5]
    assert got_c.tolist() == oc.tolist()


def test_greedy_repeated_calls_share_workspace(S):
    inp = W.greedy_inputs(B=2, T=16, V=50_000, seed=5)
    B, T, V = inp["logits"].shape
    ws = S.workspace(S.sd_accept_greedy_workspace_size(B, T, V, S.SD_BF16))
    dl, dd = inp["logits"].cuda(), inp["draft"].cuda()
    on, oc = oracle.accept_greedy(inp["draft"], inp["logits"])
    for _ in range(5):
        n = torch.zeros(B, dtype=torch.int32, device="cuda")
        c = torch.zeros(B, dtype=torch.int32, device="cuda")
        S.sd_accept_greedy(dd, dl, n, c, ws)
        assert n.cpu().tolist() == on.tolist() and c.cpu().tolist() == oc.tolist()


# --------------------------------------------------------------------------
# sampled
# --------------------------------------------------------------------------

def run_sample(S, inp, tau, seed, offset=0, ws=None, path=0):
    """path 1: the two-kernel form; 2: the one-launch form (required); 0: automatic."""
    lg, q, d = inp["logits"], inp["q"], inp["draft"]
    B, T, V = lg.shape
    n = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    nx = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    if ws is None:
        ws = S.workspace(S.sd_accept_sample_workspace_size(B, T, V, S._dt(lg)))
    prev = S.sd_set_sample_path(path)
    try:
        S.sd_accept_sample(d.cuda(), q.cuda(), lg.cuda(), tau, seed, offset, n, nx, ws)
        if path:
            assert S.sd_last_sample_path() == path
    finally:
        S.sd_set_sample_path(prev)
    torch.cuda.synchronize()
    # the counters: the 256-byte header, then two per sequence
    assert counters_zero(ws, 256 + 8 * B), "ticket and barrier counters not returned to zero"
    assert S.sd_fault_word() == 0
    return n.cpu().numpy(), nx.cpu().numpy()


def assert_sample_parity(inp, n, nx, tau, seed, offset=0):
    T = inp["logits"].shape[1]
    on, onx, diag = oracle.accept_sample(inp["draft"], inp["q"], inp["logits"], tau, seed, offset,
                                         return_diag=True)
    d = oracle.split_diag(diag, T)
    excused = 0
    for b in range(len(on)):
        if n[b] != on[b]:
            j = min(n[b], on[b])
            assert abs(d["u"][b, j] - d["ratio"][b, j]) < EXCUSE, (b, n[b], on[b])
            excused += 1
            continue
        if nx[b] != onx[b]:
            # the draw u'.S lies within 1e-6.S of a cumulative-sum boundary of
            # the oracle's id, and the GPU id is the index with positive weight
            # on the other side of that boundary
            S_ = d["S"][b]
            w = _draw_weights(inp, b, int(on[b]), tau, int(d["mode"][b]))
            pos = np.flatnonzero(w > 0)
            allowed = set()
            if abs(d["x"][b] - d["c_prev"][b]) < EXCUSE * S_:
                below = pos[pos < onx[b]]
                if below.size:
                    allowed.add(int(below[-1]))
            if abs(d["x"][b] - d["c_at"][b]) < EXCUSE * S_:
                above = pos[pos > onx[b]]
                if above.size:
                    allowed.add(int(above[0]))
            assert int(nx[b]) in allowed, (b, nx[b], onx[b], sorted(allowed))
            excused += 1
    return on, onx, excused


def _draw_weights(inp, b, n, tau, mode):
    """Weights of the oracle's draw for sequence b at row n, in fp64: the
    residual max(p - q, 0) after a rejection (mode 0), else p."""
    x = inp["logits"][b, n].double().numpy() / tau
    p = np.exp(x - x.max())
    p /= p.sum()
    if mode == 0:
        return np.maximum(p - inp["q"][b, n].double().numpy(), 0.0)
    return p


@pytest.mark.parametrize("B,T,V,tau,dtype", [
    (4, 16, 152_064, 1.0, torch.bfloat16),
    (8, 16, 1_000, 0.7, torch.bfloat16),
    (3, 5, 5_003, 1.3, torch.float32),
    (64, 4, 2_000, 1.0, torch.bfloat16),
    (2, 1, 3_000, 1.0, torch.bfloat16),
    (12, 4, 152_064, 1.0, torch.bfloat16),   # the largest draw chunk (4096 elements)
])
@pytest.mark.parametrize("path", [1, 2])
def test_sample_matches_oracle(S, B, T, V, tau, dtype, path):
    inp = W.sample_inputs(B=B, T=T, V=V, seed=B + V, dtype=dtype)
    for offset in (0, 7):
        n, nx = run_sample(S, inp, tau, 1234, offset, path=path)
        on, onx, exc = assert_sample_parity(inp, n, nx, tau, 1234, offset)
        assert exc <= max(1, B // 20)


@pytest.mark.parametrize("path", [1, 2])
def test_sample_workload5(S, path):
    cfg = W.config(5)
    n, nx = run_sample(S, cfg["sample"], cfg["temperature"], cfg["philox_seed"], path=path)
    on, onx, exc = assert_sample_parity(cfg["sample"], n, nx, cfg["temperature"], cfg["philox_seed"])
    assert exc == 0
    assert (n == on).all() and (nx == onx).all()


@pytest.mark.parametrize("path", [1, 2])
def test_sample_p_equals_q_accepts_all(S, path):
    B, T, V = 6, 16, 4_000
    g = torch.Generator().manual_seed(3)
    lg = (torch.randn(B, T, V, generator=g) * 2).to(torch.bfloat16)
    q = torch.softmax(lg.double(), -1).float()
    draft = torch.multinomial(q[:, :-1].reshape(-1, V).double(), 1, generator=g).reshape(B, T - 1).int()
    inp = {"logits": lg, "q": q, "draft": draft}
    n, nx = run_sample(S, inp, 1.0, 42, path=path)
    on, onx, _ = assert_sample_parity(inp, n, nx, 1.0, 42)
    assert (n >= 14).all()


def test_philox_word_for_word(S):
    n = 1 << 20
    rng = np.random.default_rng(9)
    ctr = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    key = 0x9E3779B97F4A7C15
    out = torch.zeros(n, 4, dtype=torch.int32, device="cuda")
    S.sd_philox4x32_10(torch.from_numpy(ctr.view(np.int32)).cuda(), key, out)
    got = out.cpu().numpy().view(np.uint32)
    want = oracle.philox4x32_10(ctr, np.array([key & 0xFFFFFFFF, key >> 32], dtype=np.uint32))
    assert np.array_equal(got, want)


def test_accept_errors_are_reported_not_launched(S):
    lg = torch.zeros(1, 16, 100, dtype=torch.bfloat16, device="cuda")
    d = torch.zeros(1, 15, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(S.SdError) as e:
        S.sd_accept_greedy(d, lg, n, n, small)
    assert e.value.status == S.SD_ERR_WORKSPACE
    ws = S.workspace(S.sd_accept_sample_workspace_size(1, 16, 100))
    with pytest.raises(S.SdError) as e:
        S.sd_accept_sample(d, lg.float(), lg, 0.0, 1, 0, n, n, ws)
    assert e.value.status == S.SD_ERR_INVALID_ARG
    assert S.sd_fault_word() == 0


@pytest.mark.parametrize("path", [1, 2])
def test_sample_zero_residual_draws_from_p(S, path):
    """q = 2 p (unnormalised, taken as given): a proposal is rejected when
    u >= 1/2, the residual max(p - q, 0) is zero everywhere, and the next token
    is drawn from p, as the oracle does (its draw mode 1)."""
    B, T, V = 16, 4, 20_000
    g = torch.Generator().manual_seed(44)
    lg = (torch.randn(B, T, V, generator=g) * 2).to(torch.bfloat16)
    p = torch.softmax(lg.double(), -1)
    q = (2.0 * p).float()
    draft = torch.multinomial(p[:, :-1].reshape(-1, V), 1, generator=g).reshape(B, T - 1).int()
    inp = {"logits": lg, "q": q, "draft": draft}
    n, nx = run_sample(S, inp, 1.0, 99, path=path)
    on, onx, exc = assert_sample_parity(inp, n, nx, 1.0, 99)
    _, _, diag = oracle.accept_sample(draft, q, lg, 1.0, 99, return_diag=True)
    modes = oracle.split_diag(diag, T)["mode"]
    assert (on < T - 1).any() and (modes[on < T - 1] == 1).all()   # rejections drew from p
    assert exc <= 1


def test_sample_one_launch_is_chosen_where_it_fits(S):
    """The automatic choice takes the one-launch form for the batched workload
    (4 sequences of 16 rows over a 152,064-token vocabulary) and for a single
    sequence, and the two-kernel form where the grid cannot hold it (more
    rows than two CTAs per SM)."""
    for B, T, V, want in [(4, 16, 152_064, 2), (1, 16, 152_064, 2), (32, 16, 2_000, 1)]:
        inp = W.sample_inputs(B=B, T=T, V=V, seed=7 + B)
        n, nx = run_sample(S, inp, 1.0, 5, path=0)
        assert S.sd_last_sample_path() == want, (B, T, V)
        assert_sample_parity(inp, n, nx, 1.0, 5)


def test_sample_one_launch_repeated_calls(S):
    """Back-to-back one-launch calls on one workspace: the barrier counters
    return to zero each time and the draws repeat, also after a call of
    another shape on the same workspace."""
    inp = W.sample_inputs(B=4, T=16, V=152_064, seed=21)
    small = W.sample_inputs(B=2, T=8, V=152_064, seed=22)
    ws = S.workspace(S.sd_accept_sample_workspace_size(4, 16, 152_064))
    first = run_sample(S, inp, 0.8, 77, ws=ws, path=2)
    for _ in range(4):
        again = run_sample(S, inp, 0.8, 77, ws=ws, path=2)
        assert (again[0] == first[0]).all() and (again[1] == first[1]).all()
    n, nx = run_sample(S, small, 1.0, 3, ws=ws, path=2)
    assert_sample_parity(small, n, nx, 1.0, 3)
    assert (run_sample(S, inp, 0.8, 77, ws=ws, path=2)[1] == first[1]).all()
