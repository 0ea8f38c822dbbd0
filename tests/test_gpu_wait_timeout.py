"""Failure detection of the in-kernel barriers, without a GPU fault.

The test hook sd_set_wait_test makes every in-kernel barrier wait for one
arrival more than the grid has -- a flag that nothing sets -- with a 1 ms
limit.  The waits then run out: the call must come back (no hang), set fault
bit 3 (a bounded wait gave up), and leave its counters zero, so that the next
call on the same workspace, with the hook off, is exact against the oracle.
Covered: the tensor-core attention's in-kernel merge of a unit's splits, and
the one-launch sampled rule's grid and sequence barriers.
"""
import numpy as np
import pytest
import torch

from serving_sd_verify_gb300 import workloads as W
from _util import check_attention, oracle_verify_rows, sample_rows

pytestmark = pytest.mark.gpu

WAIT_GAVE_UP = 1 << 3


@pytest.fixture(scope="module")
def S():
    from serving_sd_verify_gb300 import build, sd_verify
    build.build()
    sd_verify.load()
    sd_verify.sd_fault_word()          # start from a clear fault word
    yield sd_verify
    sd_verify.sd_set_wait_test(0, 0)
    sd_verify.sd_set_attention_path(0)
    sd_verify.sd_set_sample_path(0)


def test_attention_merge_wait_gives_up_then_recovers(S):
    B, T, Hq, Hkv = 1, 16, 28, 4
    inp = W.verify_inputs(B=B, T=T, Hq=Hq, Hkv=Hkv, D=128, ctx=[20_000], seed=77)
    q, k, v, ctx = (inp[x].cuda() for x in ("q", "k", "v", "ctx"))
    ws = S.workspace(S.sd_verify_attention_workspace_size(B, T, Hq, Hkv, 128, inp["max_ctx"]))
    out = torch.full((B, T, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    S.sd_set_attention_path(2)
    S.sd_set_wait_test(1, 1_000_000)
    try:
        S.sd_verify_attention(q, k, v, ctx, inp["max_ctx"], out, inp["scale"], ws)
        path, splits = S.sd_last_attention_path()
        torch.cuda.synchronize()
    finally:
        S.sd_set_wait_test(0, 0)
    assert path == 2 and splits > Hkv, "the call must merge several splits per kv head inside the kernel"
    assert S.sd_fault_word() & WAIT_GAVE_UP
    assert int(ws[:256 + 4 * B * Hkv].abs().sum()) == 0, "merge counters not returned to zero"
    # the hook off: the same workspace gives the oracle's result
    out.fill_(float("nan"))
    S.sd_verify_attention(q, k, v, ctx, inp["max_ctx"], out, inp["scale"], ws)
    torch.cuda.synchronize()
    assert S.sd_fault_word() == 0
    rows = sample_rows(B, T, Hq, 48, seed=5)
    want = oracle_verify_rows(inp["q"], inp["k"], inp["v"], inp["ctx"], inp["scale"], rows)
    check_attention(out.cpu().numpy().reshape(B * T * Hq, 128)[rows], want)


def test_sample_barriers_wait_gives_up_then_recovers(S):
    B, T, V = 4, 16, 30_000
    inp = W.sample_inputs(B=B, T=T, V=V, seed=78)
    d, q, lg = inp["draft"].cuda(), inp["q"].cuda(), inp["logits"].cuda()
    ws = S.workspace(S.sd_accept_sample_workspace_size(B, T, V))
    n = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    nx = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    S.sd_set_sample_path(2)
    # the same call on a fresh workspace, hook off: the result to come back to
    S.sd_accept_sample(d, q, lg, 1.0, 55, 0, n, nx, S.workspace(S.sd_accept_sample_workspace_size(B, T, V)))
    want = (n.cpu().tolist(), nx.cpu().tolist())
    S.sd_set_wait_test(1, 1_000_000)
    try:
        S.sd_accept_sample(d, q, lg, 1.0, 55, 0, n, nx, ws)
        assert S.sd_last_sample_path() == 2
        torch.cuda.synchronize()
    finally:
        S.sd_set_wait_test(0, 0)
    assert S.sd_fault_word() & WAIT_GAVE_UP
    assert int(ws[:256 + 8 * B].abs().sum()) == 0, "barrier counters not returned to zero"
    S.sd_accept_sample(d, q, lg, 1.0, 55, 0, n, nx, ws)
    torch.cuda.synchronize()
    S.sd_set_sample_path(0)
    assert S.sd_fault_word() == 0
    assert (n.cpu().tolist(), nx.cpu().tolist()) == want


def test_wait_hook_rejects_nonsense(S):
    with pytest.raises(S.SdError) as e:
        S.sd_set_wait_test(5000, 0)
    assert e.value.status == S.SD_ERR_INVALID_ARG
