"""CPU checks of the C ABI: the library builds, loads without a GPU, exports
every entry point include/*.h declares, and rejects bad arguments on the host
(status codes, no launch).  No compute call is made here."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def S():
    from serving_sd_verify_gb300 import build, sd_verify
    build.build()
    sd_verify.load()
    return sd_verify


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"(?:^|\n)\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(sd_\w+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("sd_verify_attention", "sd_draft_block_attention", "sd_accept_greedy", "sd_accept_sample"):
        assert n in names


def test_library_exports_every_declared_symbol(S):
    lib = ctypes.CDLL(S.LIB_PATH)
    missing = [n for n in sorted(declared_functions()) if not hasattr(lib, n)]
    assert not missing, missing
    assert set(S.SYMBOLS) == declared_functions()


def test_status_strings_and_version(S):
    lib = S.load()
    assert lib.sd_version() >= 100
    for code, name in enumerate(["SD_OK", "SD_ERR_INVALID_ARG", "SD_ERR_UNSUPPORTED",
                                 "SD_ERR_WORKSPACE", "SD_ERR_CUDA"]):
        assert lib.sd_status_string(code).decode() == name


def test_host_validation_rejects_bad_arguments(S):
    lib = S.load()
    st = S.Strides(100 * 4 * 128, 4 * 128, 128)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    # null q
    r = lib.sd_verify_attention(None, fake, fake, st, fake, 100, fake, 1, 16, 28, 4, 128, 0, 1.0, fake,
                                1 << 30, None)
    assert r == S.SD_ERR_INVALID_ARG
    # T out of range
    r = lib.sd_verify_attention(fake, fake, fake, st, fake, 100, fake, 1, 17, 28, 4, 128, 0, 1.0, fake,
                                1 << 30, None)
    assert r == S.SD_ERR_INVALID_ARG and b"T in [1, 16]" in lib.sd_last_error()
    # Hq not a multiple of Hkv
    r = lib.sd_verify_attention(fake, fake, fake, st, fake, 100, fake, 1, 16, 27, 4, 128, 0, 1.0, fake,
                                1 << 30, None)
    assert r == S.SD_ERR_INVALID_ARG
    # unsupported head dim
    r = lib.sd_verify_attention(fake, fake, fake, st, fake, 100, fake, 1, 16, 28, 4, 96, 0, 1.0, fake,
                                1 << 30, None)
    assert r == S.SD_ERR_UNSUPPORTED
    # misaligned cache stride (bf16, 8 bytes)
    bad = S.Strides(100 * 4 * 128, 4, 128)
    r = lib.sd_verify_attention(fake, fake, fake, bad, fake, 100, fake, 1, 16, 28, 4, 128, 0, 1.0, fake,
                                1 << 30, None)
    assert r == S.SD_ERR_INVALID_ARG
    # drafter without block tensors
    r = lib.sd_draft_block_attention(fake, fake, fake, st, fake, 100, None, None, fake, 1, 16, 28, 4, 128, 0,
                                     1.0, fake, 1 << 30, None)
    assert r == S.SD_ERR_INVALID_ARG
    # greedy: V < 1, null logits
    assert lib.sd_accept_greedy(fake, fake, 1, 16, 0, 0, fake, fake, fake, 1 << 20, None) == S.SD_ERR_INVALID_ARG
    assert lib.sd_accept_greedy(fake, None, 1, 16, 10, 0, fake, fake, fake, 1 << 20, None) == S.SD_ERR_INVALID_ARG
    # sample: temperature must be > 0
    assert lib.sd_accept_sample(fake, fake, fake, 1, 16, 10, 0, 0.0, 1, 0, fake, fake, fake, 1 << 20,
                                None) == S.SD_ERR_INVALID_ARG
    assert lib.sd_accept_sample(fake, fake, fake, 1, 16, 10, 0, float("nan"), 1, 0, fake, fake, fake, 1 << 20,
                                None) == S.SD_ERR_INVALID_ARG
    # philox: negative n
    assert lib.sd_philox4x32_10(fake, 1, fake, -1, None) == S.SD_ERR_INVALID_ARG
    # host store: negative size, null pointer, a size or address off 16 bytes
    # (all refused before any CUDA call); an empty store enqueues nothing
    assert lib.sd_store_to_host(fake, fake, -16, None) == S.SD_ERR_INVALID_ARG
    assert lib.sd_store_to_host(None, fake, 16, None) == S.SD_ERR_INVALID_ARG
    assert lib.sd_store_to_host(fake, fake, 24, None) == S.SD_ERR_INVALID_ARG
    assert lib.sd_store_to_host(ctypes.c_void_p(0x10008), fake, 16, None) == S.SD_ERR_INVALID_ARG
    assert lib.sd_store_to_host(None, None, 0, None) == S.SD_OK


def test_workspace_sizes_are_positive_and_monotone(S):
    a = S.sd_verify_attention_workspace_size(1, 16, 28, 4, 128, 25_119)
    b = S.sd_verify_attention_workspace_size(8, 16, 28, 4, 128, 32_768)
    assert 256 < a <= b
    assert S.sd_draft_block_attention_workspace_size(1, 16, 28, 4, 128, 25_119) > 256
    assert S.sd_accept_greedy_workspace_size(1, 16, 152_064) > 256
    assert S.sd_accept_sample_workspace_size(4, 16, 152_064) > 256
    assert S.sd_verify_attention_workspace_size(1, 17, 28, 4, 128, 100) == 0


def test_tree_calls_take_up_to_64_nodes(S):
    # a tree of up to 64 nodes (the pages' Tree-60); chains stay at 16 slots
    assert S.sd_verify_tree_attention_workspace_size(1, 60, 28, 4, 128, 25_119) > \
        S.sd_verify_tree_attention_workspace_size(1, 16, 28, 4, 128, 25_119) > 256
    assert S.sd_verify_tree_attention_workspace_size(1, 64, 28, 4, 128, 100) > 0
    assert S.sd_verify_tree_attention_workspace_size(1, 65, 28, 4, 128, 100) == 0
    assert S.sd_accept_tree_greedy_workspace_size(2, 64, 152_064) > 256
    assert S.sd_accept_tree_greedy_workspace_size(2, 65, 152_064) == 0
    assert S.sd_accept_greedy_workspace_size(1, 17, 1000) == 0


def test_binding_refuses_cpu_tensors(S):
    import torch
    q = torch.zeros(1, 16, 28, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        S.sd_verify_attention(q, q, q, torch.zeros(1, dtype=torch.int32), 10, q.float(), 1.0,
                              torch.zeros(8, dtype=torch.uint8))


def test_binding_store_to_host_wants_a_pinned_destination(S):
    import torch
    with pytest.raises(ValueError):
        S.sd_store_to_host(torch.zeros(64, dtype=torch.uint8), torch.zeros(64, dtype=torch.uint8))


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    from serving_sd_verify_gb300 import sd_verify
    monkeypatch.setattr(sd_verify, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(sd_verify, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        sd_verify.load()


def test_host_validation_of_the_tree_projector_commit_and_compressor_calls(S):
    lib = S.load()
    st = S.Strides(100 * 4 * 128, 4 * 128, 128)
    fake = ctypes.c_void_p(0x10000)  # 16-byte aligned, never dereferenced
    # tree verify: no tree mask
    r = lib.sd_verify_tree_attention(fake, fake, fake, st, fake, 100, None, fake, 1, 16, 28, 4, 128, 0, 1.0, fake,
                                     1 << 30, None)
    assert r == S.SD_ERR_INVALID_ARG
    # tree greedy: no parents
    r = lib.sd_accept_tree_greedy(fake, None, fake, 1, 16, 100, 0, fake, fake, fake, fake, 1 << 20, None)
    assert r == S.SD_ERR_INVALID_ARG
    # projector: fp32 unsupported, Dout not a multiple of 32, N = 0 is a no-op
    assert lib.sd_project_kv(fake, 64, fake, fake, 4, 64, 64, fake, fake, 64, 1, None) == S.SD_ERR_UNSUPPORTED
    assert lib.sd_project_kv(fake, 64, fake, fake, 4, 64, 48, fake, fake, 64, 0, None) == S.SD_ERR_INVALID_ARG
    assert lib.sd_project_kv(fake, 64, fake, fake, 0, 64, 64, fake, fake, 64, 0, None) == S.SD_OK
    assert lib.sd_last_projector_path() == 0
    # commit-time append: 16 rows of Hd = 8000 do not fit its shared memory
    r = lib.sd_project_kv_commit(fake, 8000, 16 * 8000, fake, fake, 8000, 64, fake, None, fake, 1, 16, fake, fake,
                                 64 * 100, 64, 100, 0, None)
    assert r == S.SD_ERR_UNSUPPORTED
    # commit: T out of range, proposal stride too small for a chain
    r = lib.sd_commit_tokens(fake, 15, None, fake, fake, 1, 17, fake, 1000, None, fake, fake, 64, fake, None, None)
    assert r == S.SD_ERR_INVALID_ARG
    r = lib.sd_commit_tokens(fake, 14, None, fake, fake, 1, 16, fake, 1000, None, fake, fake, 64, fake, None, None)
    assert r == S.SD_ERR_INVALID_ARG
    # tree K/V compaction: a (position, head) row over 512 bytes, a missing path
    big = S.Strides(100 * 512, 512, 512)
    r = lib.sd_compact_tree_kv(fake, fake, big, fake, fake, fake, 1, 16, 100, 1, 512, 0, None)
    assert r == S.SD_ERR_UNSUPPORTED
    r = lib.sd_compact_tree_kv(fake, fake, st, fake, None, fake, 1, 16, 100, 4, 128, 0, None)
    assert r == S.SD_ERR_INVALID_ARG
    # compressor: 65 queries, d not a multiple of 64, fp32, a workspace too small
    ws = S.sd_latent_compress_workspace_size(2, 576, 64, 256)
    assert ws > 0 and S.sd_latent_compress_workspace_size(2, 576, 65, 256) == 0
    assert lib.sd_latent_compress(fake, fake, 256, 576 * 256, 2, 576, 65, 256, fake, 256, 65 * 256, 0, fake, ws,
                                  None) == S.SD_ERR_INVALID_ARG
    assert lib.sd_latent_compress(fake, fake, 96, 576 * 96, 2, 576, 64, 96, fake, 96, 64 * 96, 0, fake, ws,
                                  None) == S.SD_ERR_INVALID_ARG
    assert lib.sd_latent_compress(fake, fake, 256, 576 * 256, 2, 576, 64, 256, fake, 256, 64 * 256, 1, fake, ws,
                                  None) == S.SD_ERR_UNSUPPORTED
    assert lib.sd_latent_compress(fake, fake, 256, 576 * 256, 2, 576, 64, 256, fake, 256, 64 * 256, 0, fake, 64,
                                  None) == S.SD_ERR_WORKSPACE


def test_next_row_workspace_sizes(S):
    assert S.sd_verify_tree_attention_workspace_size(1, 16, 28, 4, 128, 25_119) > 256
    assert S.sd_accept_tree_greedy_workspace_size(1, 16, 152_064) == S.sd_accept_greedy_workspace_size(1, 16, 152_064)
    a = S.sd_latent_compress_workspace_size(16, 576, 64, 4096)
    b = S.sd_latent_compress_workspace_size(32, 576, 64, 4096)
    assert 0 < a < b


def test_path_setters_and_wait_hook_on_the_host(S):
    """The process-wide selectors return the previous setting and fold
    unknown values to automatic; the wait-test hook refuses more than 1024
    extra arrivals and takes (0, 0) back to normal operation.  No launch."""
    lib = S.load()
    prev = lib.sd_set_sample_path(1)
    try:
        assert lib.sd_set_sample_path(2) == 1
        assert lib.sd_set_sample_path(7) == 2      # out of range: automatic
        assert lib.sd_set_sample_path(0) == 0
    finally:
        lib.sd_set_sample_path(prev)
    assert lib.sd_set_wait_test(5000, 0) == S.SD_ERR_INVALID_ARG
    assert lib.sd_set_wait_test(1, 1_000_000) == S.SD_OK
    assert lib.sd_set_wait_test(0, 0) == S.SD_OK


def test_sample_workspace_covers_both_forms(S):
    """The sampled rule's workspace holds the two-kernel form and the one-launch
    form (its records sized for two CTAs per SM), so the call may take either:
    it grows with the batch and never shrinks below the smaller shapes'."""
    lib = S.load()
    sizes = [lib.sd_accept_sample_workspace_size(B, 16, 152_064, S.SD_BF16) for B in (1, 2, 4, 8, 64)]
    assert all(x > 0 for x in sizes) and sizes == sorted(sizes)
