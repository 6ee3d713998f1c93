"""The allocation-free permutation entry point against the block's own permutation.

lmoe_permute_noalloc serves callers that cannot allocate device memory (its scratch is a
fixed array inside the library).  Its outputs must equal, exactly, the offsets / row_of /
tok_of the block's forward call leaves in its workspace for the same top-k ids, on two
calls in a row (the second call reuses the array the first one left behind).  This file is
collected last so that a run stopping at the first failure has run everything else."""
import ctypes

import numpy as np
import pytest
import torch

import workloads

from gpu_util import run, views

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()
    import latent_mixture_experts_router_gb300 as lm
    return lm


def _noalloc_call(lm, idx: torch.Tensor, E: int):
    """One call through the C ABI (ctypes), on the current stream."""
    T, k = idx.shape
    dev = idx.device
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    row_of = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    tok_of = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
    fn = lm.load().lmoe_permute_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    st = fn(idx.data_ptr(), T, k, E, offsets.data_ptr(), row_of.data_ptr(), tok_of.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    assert st == 0, st
    torch.cuda.synchronize()
    return offsets.cpu().numpy(), row_of.cpu().numpy(), tok_of.cpu().numpy()


@pytest.mark.parametrize("shapes", [((300, 32, 4, 0), (77, 8, 2, 1))])
def test_no_alloc_permutation_matches_forward(lm, shapes):
    dev = torch.device("cuda:0")
    for T, E, k, seed in shapes:   # two calls in a row, different sizes and routings
        w = workloads.Workload(f"na{T}", T=T, D=256, L=128, E=E, I=128, k=k, seed=seed)
        inp = workloads.make_inputs(w, dev)
        out, idx, blk, cfg = run(inp)
        v = views(blk, cfg)
        offsets, row_of, tok_of = _noalloc_call(lm, idx, E)
        assert np.array_equal(offsets, v["offsets"])
        assert np.array_equal(row_of, v["row_of"])
        assert np.array_equal(tok_of, v["tok_of"])


@pytest.mark.parametrize("misaligned", [False, True], ids=["aligned", "4-byte-aligned"])
def test_no_alloc_permutation_many_pairs(lm, misaligned):
    # 24000 pairs: several 128-pair chunks per warp segment and a ragged tail; an id array
    # that is only 4-byte aligned takes the scalar loads
    from gpu_util import expected_permutation
    T, k, E = 3000, 8, 64
    g = torch.Generator().manual_seed(11)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    buf = torch.empty(T * k + 1, dtype=torch.int32, device="cuda:0")
    idx = (buf[1:] if misaligned else buf[:-1]).view(T, k)
    idx.copy_(ids.to("cuda:0"))
    assert (idx.data_ptr() % 16 != 0) == misaligned
    counts, offsets_ref, row_ref, tok_ref = expected_permutation(ids.numpy(), E)
    offsets, row_of, tok_of = _noalloc_call(lm, idx, E)
    assert np.array_equal(offsets, offsets_ref)
    assert np.array_equal(row_of, row_ref)
    assert np.array_equal(tok_of, tok_ref)


def test_no_alloc_rejects_sizes_beyond_its_scratch(lm):
    idx = torch.zeros((70000, 1), dtype=torch.int32, device="cuda:0")
    with pytest.raises(lm.LmoeError) as ei:
        from latent_mixture_experts_router_gb300._lib import lmoe_permute_noalloc
        o = torch.empty(9, dtype=torch.int32, device="cuda:0")
        lmoe_permute_noalloc(idx, 8, o, idx, idx.view(-1))
    assert ei.value.status == -2


def test_no_alloc_permutation_at_its_limits(lm):
    # T*k = 65536 pairs over E = 1024 experts: the fixed tile table at full capacity
    from gpu_util import expected_permutation
    T, k, E = 8192, 8, 1024
    g = torch.Generator().manual_seed(12)
    ids = torch.argsort(torch.rand(T, E, generator=g), dim=1)[:, :k].to(torch.int32)
    ids[:64] = torch.arange(k, dtype=torch.int32)      # a crowded expert or two as well
    idx = ids.to("cuda:0")
    counts, offsets_ref, row_ref, tok_ref = expected_permutation(ids.numpy(), E)
    for _ in range(2):
        offsets, row_of, tok_of = _noalloc_call(lm, idx, E)
        assert np.array_equal(offsets, offsets_ref)
        assert np.array_equal(row_of, row_ref)
        assert np.array_equal(tok_of, tok_ref)


def test_no_alloc_refuses_host_memory_before_launching(lm):
    # an output array in (pinned) host memory is not device memory of the current device
    from latent_mixture_experts_router_gb300._lib import lmoe_permute_noalloc
    idx = torch.zeros((4, 2), dtype=torch.int32, device="cuda:0")
    idx[:, 1] = 1
    host = torch.empty(9, dtype=torch.int32).pin_memory()
    row_of = torch.empty((4, 2), dtype=torch.int32, device="cuda:0")
    tok_of = torch.empty(8, dtype=torch.int32, device="cuda:0")
    with pytest.raises(lm.LmoeError) as ei:
        lmoe_permute_noalloc(idx, 8, host, row_of, tok_of)
    assert ei.value.status == -1
