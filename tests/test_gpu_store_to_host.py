"""sd_store_to_host: a device buffer stored into pinned host memory by the
GPU's cores, after the stream's earlier work.  Checked byte for byte against
the source read back through PyTorch, at sizes from one 16-byte vector to
several MB (ragged against the kernel's grid), ordered after a kernel that
rewrites the source, replayed from a CUDA graph, and refused (nothing
enqueued) for destinations that are not pinned host memory."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    from serving_sd_verify_gb300 import build, sd_verify
    build.build()
    sd_verify.load()
    return sd_verify


@pytest.mark.parametrize("nbytes", [16, 4096 + 16, 229_376 + 256, (3 << 20) + 48])
def test_store_to_host_is_exact_and_ordered(S, nbytes):
    g = torch.Generator(device="cuda").manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda", generator=g)
    dst = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        src.add_(1)                      # a kernel the store must wait for
        S.sd_store_to_host(dst, src, st)
    st.synchronize()
    assert torch.equal(dst, src.cpu())


def test_store_to_host_replays_from_a_cuda_graph(S):
    src = torch.zeros(4096, dtype=torch.int32, device="cuda")
    dst = torch.full((4096,), -1, dtype=torch.int32).pin_memory()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        S.sd_store_to_host(dst, src, st)
        st.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            src.add_(1)
            S.sd_store_to_host(dst, src, st)
    for k in range(1, 4):
        graph.replay()
        torch.cuda.synchronize()
        assert bool((dst == k).all())


def test_store_to_host_refuses_other_destinations(S):
    lib = S.load()
    src = torch.zeros(64, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(64, dtype=torch.uint8)
    device_dst = torch.zeros(64, dtype=torch.uint8, device="cuda")
    pinned = torch.zeros(64, dtype=torch.uint8).pin_memory()
    assert lib.sd_store_to_host(pageable.data_ptr(), src.data_ptr(), 64, None) == S.SD_ERR_INVALID_ARG
    assert lib.sd_store_to_host(device_dst.data_ptr(), src.data_ptr(), 64, None) == S.SD_ERR_INVALID_ARG
    # the source must be device memory
    assert lib.sd_store_to_host(pinned.data_ptr(), pageable.data_ptr(), 64, None) == S.SD_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((pinned == 0).all())
    with pytest.raises(ValueError):
        S.sd_store_to_host(pinned, torch.zeros(32, dtype=torch.uint8, device="cuda"))
