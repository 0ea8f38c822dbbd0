"""GPU parity of the SpecFLASH latent compressor against the fp64 oracle.

Tolerance, from the arithmetic: the softmax weights are rounded to bf16
(relative 2^-9 each) before the second product and the output is rounded
once to bf16 (relative 2^-9), so |got - exact| <= 2^-9 (sum_n p_n |F_n|) +
2^-9 |exact|; the test allows twice that, 2^-8 (|exact| + sum_n p_n |F_n|),
which also covers the fp32 accumulation of the scores and of P . F.
"""
import numpy as np
import pytest
import torch

import oracle
from serving_sd_verify_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    from serving_sd_verify_gb300 import build, sd_verify
    build.build()
    sd_verify.load()
    return sd_verify


def run(S, q, f, out=None):
    F, N, d = f.shape
    Cq = q.shape[0]
    ws = S.workspace(S.sd_latent_compress_workspace_size(F, N, Cq, d))
    if out is None:
        out = torch.full((F, Cq, d), 5.0, dtype=torch.bfloat16, device="cuda")
    S.sd_latent_compress(q.cuda() if not q.is_cuda else q, f.cuda() if not f.is_cuda else f, out, ws)
    torch.cuda.synchronize()
    return out


def check(got, q, f, frames=None):
    """got [F', Cq, d] (CPU) against the oracle on the given frames."""
    fr = range(f.shape[0]) if frames is None else frames
    for i, fi in enumerate(fr):
        ref = oracle.latent_compress(q, f[fi])
        mag = oracle.latent_compress(q, f[fi], f[fi].double().abs())
        g = got[i].double().numpy()
        err = np.abs(g - ref)
        tol = 2.0 ** -8 * (np.abs(ref) + mag)
        assert np.isfinite(g).all()
        assert (err <= tol).all(), (fi, err.max(), np.unravel_index(np.argmax(err - tol), err.shape))


@pytest.mark.parametrize("F,N,Cq,d", [
    (2, 576, 64, 256),     # LLaVA-1.5 token count, 64 latents
    (3, 324, 36, 192),     # Qwen2.5-VL token count, 36 latents; d tile partial (3 of 4 chunks)
    (2, 130, 64, 512),     # ragged last feature tile (2 features)
    (1, 700, 17, 320),     # odd query count, 11 feature stages with a ragged one
    (1, 1, 1, 64),         # one feature: the output is that feature
])
def test_matches_oracle(S, F, N, Cq, d):
    q, f = W.latent_inputs(frames=F, N=N, Cq=Cq, d=d, seed=N + Cq)
    got = run(S, q, f).cpu()
    check(got, q, f)
    if N == 1:
        assert torch.equal(got[0, 0], f[0, 0])


def test_strided_features_and_output(S):
    F, N, Cq, d = 3, 300, 64, 256
    q, f = W.latent_inputs(frames=F, N=N, Cq=Cq, d=d, seed=7)
    big = torch.zeros(F, N + 5, d + 64, dtype=torch.bfloat16)
    big[:, :N, :d] = f
    fb = big.cuda()[:, :N, :d]
    obuf = torch.full((F, Cq + 3, d + 32), 9.0, dtype=torch.bfloat16, device="cuda")
    out = obuf[:, :Cq, :d]
    ws = S.workspace(S.sd_latent_compress_workspace_size(F, N, Cq, d))
    S.sd_latent_compress(q.cuda(), fb, out, ws)
    torch.cuda.synchronize()
    check(out.cpu(), q, f)
    ob = obuf.cpu()
    assert (ob[:, Cq:] == 9.0).all() and (ob[:, :, d:] == 9.0).all()


def test_equal_features_return_that_feature(S):
    F, N, Cq, d = 2, 576, 64, 128
    q, f = W.latent_inputs(frames=F, N=N, Cq=Cq, d=d, seed=3)
    f = f[:, :1].expand(F, N, d).contiguous()
    got = run(S, q, f).cpu().double()
    want = f[:, :1].double().expand(F, Cq, d)
    # the weights sum to 1 up to their bf16 rounding (2^-9 each, relative)
    assert (got - want).abs().max() <= 2.0 ** -8 * want.abs().max()


@pytest.mark.parametrize("name,F,N,Cq,d,check_frames", [
    ("llava15_video", 16, 576, 64, 4096, [0, 7, 15]),
    ("qwen25vl_video", 8, 324, 36, 3584, [0, 7]),
])
def test_full_size_sampled_frames(S, name, F, N, Cq, d, check_frames):
    q, f = W.latent_inputs(frames=F, N=N, Cq=Cq, d=d, seed=F)
    out = run(S, q, f)
    out2 = run(S, q, f)
    assert torch.equal(out, out2)        # deterministic
    got = out[check_frames].cpu()
    check(got, q, f, check_frames)
    assert S.sd_fault_word() == 0


def test_argument_errors(S):
    q = torch.zeros(65, 64, dtype=torch.bfloat16, device="cuda")
    f = torch.zeros(1, 10, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, 65, 64, dtype=torch.bfloat16, device="cuda")
    ws = S.workspace(1 << 20)
    with pytest.raises(S.SdError) as e:
        S.sd_latent_compress(q, f, out, ws)                 # 65 queries
    assert e.value.status == S.SD_ERR_INVALID_ARG
    with pytest.raises(S.SdError) as e:
        S.sd_latent_compress(q[:8].float(), f.float(), out[:, :8].float(), ws)
    assert e.value.status == S.SD_ERR_UNSUPPORTED
    f96 = torch.zeros(1, 10, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(S.SdError) as e:                    # d not a multiple of 64
        S.sd_latent_compress(torch.zeros(8, 96, dtype=torch.bfloat16, device="cuda"), f96,
                             torch.zeros(1, 8, 96, dtype=torch.bfloat16, device="cuda"), ws)
    assert e.value.status == S.SD_ERR_INVALID_ARG
    with pytest.raises(S.SdError) as e:
        S.sd_latent_compress(q[:8], f, out[:, :8], S.workspace(64))
    assert e.value.status == S.SD_ERR_WORKSPACE
    assert S.sd_fault_word() == 0
