"""The greedy acceptance entry point that allocates nothing.

Some hosts cannot give the library a workspace: their own pool allocator owns
all device memory and extensions may not call cudaMalloc, or only the input
and output buffers are at hand.  sd_accept_greedy_noalloc serves them from a
fixed device array the library owns.  This test calls it through the C ABI
twice in a row, on different inputs (the array keeps the previous call's
contents), and checks both results against sd_accept_greedy with an ordinary
caller workspace: accept lengths and correction ids must be identical.
Kept in a file of its own that is collected last.
"""
import ctypes

import pytest
import torch

from serving_sd_verify_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    from serving_sd_verify_gb300 import build, sd_verify
    build.build()
    sd_verify.load()
    return sd_verify


def _with_workspace(S, draft, logits):
    B, T, V = logits.shape
    n = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    c = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    ws = S.workspace(S.sd_accept_greedy_workspace_size(B, T, V, S._dt(logits)))
    S.sd_accept_greedy(draft, logits, n, c, ws)
    torch.cuda.synchronize()
    return n.cpu().tolist(), c.cpu().tolist()


def _no_alloc(S, draft, logits):
    B, T, V = logits.shape
    n = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    c = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    lib = S.load()
    status = lib.sd_accept_greedy_noalloc(
        ctypes.c_void_p(draft.data_ptr()), ctypes.c_void_p(logits.data_ptr()), B, T, V, S._dt(logits),
        ctypes.c_void_p(n.data_ptr()), ctypes.c_void_p(c.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == S.SD_OK, lib.sd_last_error().decode()
    torch.cuda.synchronize()
    return n.cpu().tolist(), c.cpu().tolist()


def test_no_alloc_matches_workspace_entry_point_twice(S):
    cases = [W.greedy_inputs(B=1, T=16, V=152_064, seed=31),          # the 25,119-token step's shape
             W.greedy_inputs(B=8, T=16, V=152_064, seed=32, k=[0, 3, 15, 7, 1, 9, 12, 4])]
    for inp in cases:
        draft, logits = inp["draft"].cuda(), inp["logits"].cuda()
        want = _with_workspace(S, draft, logits)
        got = _no_alloc(S, draft, logits)
        assert got == want
        assert got[0] == [min(k, 15) for k in inp["k"]]
    assert S.sd_fault_word() == 0


def test_no_alloc_rejects_shapes_beyond_its_scratch(S):
    logits = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    lib = S.load()
    # a workspace far beyond the fixed scratch (262,144 rows x 8 bytes of
    # partials, one chunk per row): no launch, a clear status
    status = lib.sd_accept_greedy_noalloc(None, ctypes.c_void_p(logits.data_ptr()), 16384, 16, 1 << 24,
                                          S.SD_BF16, None, None, None)
    assert status == S.SD_ERR_WORKSPACE
    assert b"1 MiB" in lib.sd_last_error()
