"""Memory-safety checks that stand in for a device sanitiser (no GPU is faulted by any of them).

* Guard bands: every workspace sub-buffer is followed by LMOE_GUARD_BYTES that no call may
  touch.  The workspace is filled with a canary byte, a full-size call of each weight dtype
  (and the NVFP4 decode at T = 1 and 8) runs, and every band must still hold the canary; the
  same call on a zeroed workspace must give bitwise the same output (nothing depends on the
  workspace's initial contents).
* Routing validation: lmoe_validate_routing accepts the routing a real call leaves behind and
  flags (error bit 0x20, LMOE_ERR_ARG) each kind of corruption written into it on purpose:
  a pair's row outside the table, two pairs sharing a row, broken offsets, a tile too tall or
  outside its expert, tile counts beyond the table, a wrong first tile.
* The bounds-checked build (-DLMOE_BOUNDS_CHECKS=1): its forward, which validates the routing
  inside every call, gives bitwise the release library's outputs with an OK status."""
import ctypes
import gc

import numpy as np
import pytest
import torch

import workloads

from gpu_util import make_block, run

pytestmark = pytest.mark.gpu
CANARY = 0xA5


@pytest.fixture(scope="module")
def lm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()
    import latent_mixture_experts_router_gb300 as lm
    yield lm
    gc.collect()
    torch.cuda.empty_cache()


def _bands_intact(lm, cfg, ws, host_io=False):
    g = torch.as_tensor(lm.lmoe_workspace_guards(cfg, host_io=host_io), device=ws.device)
    idx = (g[:, None] + torch.arange(lm.GUARD_BYTES, device=ws.device)[None, :]).reshape(-1)
    bad = (ws[idx] != CANARY).nonzero()
    return bad.numel() == 0, (idx[bad[:8, 0]].tolist() if bad.numel() else [])


@pytest.mark.parametrize("name,T", [("decode_bf16", None), ("prefill_nvfp4", None), ("tiny_fp32", None),
                                    ("decode_nvfp4_hot", 1), ("decode_nvfp4_hot", 8)])
def test_guard_bands_intact_and_initial_contents_irrelevant(lm, name, T):
    # NVFP4 decode at T = 1 (the clear, pre, expert-pair and post kernels) and T = 8 (the chain
    # with the expert pair): their counters start from whatever the workspace holds
    w = workloads.WORKLOADS[name] if T is None else workloads.WORKLOADS[name].with_tokens(T)
    dev = torch.device("cuda:0")
    inp = workloads.make_inputs(w, dev)
    blk = make_block(inp)
    cfg = blk.config(w.T, w.act, "f32")
    ws = blk.workspace(cfg)
    ws.fill_(CANARY)
    out_a, idx_a, _, _ = run(inp, blk=blk)
    out_a = out_a.clone()
    ok, where = _bands_intact(lm, cfg, ws)
    assert ok, f"guard bands written at workspace bytes {where}"
    ws.zero_()
    out_b, idx_b, _, _ = run(inp, blk=blk)
    assert torch.equal(out_a, out_b) and torch.equal(idx_a, idx_b)
    del inp, blk, ws


def test_guard_bands_of_the_host_io_workspace(lm):
    w = workloads.Workload("guard_io", T=70, D=512, L=256, E=8, I=256, k=2, routing="zipf")
    dev = torch.device("cuda:0")
    inp = workloads.make_inputs(w, dev)
    out, _, blk, cfg = run(inp)
    ws = torch.full((lm.lmoe_workspace_size_host_io(cfg),), CANARY, dtype=torch.uint8, device=dev)
    xh = inp.x.cpu().pin_memory()
    oh = torch.empty(w.T, w.D, dtype=torch.float32).pin_memory()
    W = blk.W
    lm.latent_moe_forward_host_io_ex(cfg, xh, W["W_router"], W["W_pool"], W["g_pool"], W["W_gate"], W["W_up"],
                                     W["W_down"], W["g_expert"], W["W_unpool"], W["g_pre"], W["g_post"], w.k, oh, ws,
                                     router_bias=inp.router_bias)
    torch.cuda.synchronize()
    assert torch.equal(oh, out.cpu())
    ok, where = _bands_intact(lm, cfg, ws, host_io=True)
    assert ok, f"guard bands written at workspace bytes {where}"


def _i32(ws, off, n):
    return ws[off:off + 4 * n].view(torch.int32)


@pytest.mark.parametrize("T,E,k,weights", [(300, 16, 4, "bf16"), (600, 4, 2, "bf16"), (40, 32, 8, "nvfp4"),
                                           (2100, 64, 8, "bf16")])
def test_validate_routing_accepts_real_routing_and_flags_corruption(lm, T, E, k, weights):
    w = workloads.Workload(f"val_{T}_{E}", T=T, D=256, L=256, E=E, I=256, k=k, weights=weights, seed=1)
    inp = workloads.make_inputs(w, torch.device("cuda:0"))
    _, _, blk, cfg = run(inp)
    ws = blk._ws
    lay = lm.lmoe_get_workspace_layout(cfg)
    R = T * k
    lm.lmoe_validate_routing(cfg, ws)
    assert lm.lmoe_check_status(cfg, ws) == (0, 0)
    saved = ws.clone()
    row_of = lambda: _i32(ws, lay["row_of"], R)   # noqa: E731
    offsets = lambda: _i32(ws, lay["offsets"], E + 1)   # noqa: E731
    tiles = lambda: _i32(ws, lay["tiles"], 4 * 64)   # noqa: E731  (expert, row0, nrows, ready)
    n_tiles = lambda: _i32(ws, lay["n_tiles"], 1)   # noqa: E731

    def dup_row():
        r = row_of()
        r[1] = r[0]

    def tall_tile():
        t = tiles()
        t[2] = 129

    def tile_outside():
        t = tiles()
        t[1] = t[1] + R

    corruptions = {
        "row_out_of_range": lambda: row_of().__setitem__(5, R + 7),
        "negative_row": lambda: row_of().__setitem__(3, -1),
        "two_pairs_one_row": dup_row,
        "offsets_not_ending_at_R": lambda: offsets().__setitem__(E, R + 1),
        "offsets_decreasing": lambda: offsets().__setitem__(1, offsets()[2].item() + 1),
        "tile_too_tall": tall_tile,
        "tile_outside_its_expert": tile_outside,
        "tile_count_beyond_table": lambda: n_tiles().__setitem__(0, 1 << 20),
        "expert_id_out_of_range": lambda: _i32(ws, lay["topk_idx"], R).__setitem__(0, E),
    }
    for what, corrupt in corruptions.items():
        ws.copy_(saved)
        corrupt()
        lm.lmoe_validate_routing(cfg, ws)
        st, word = lm.lmoe_check_status(cfg, ws)
        assert st == -1 and word & 0x20, what
        ws.copy_(saved)
        lm.lmoe_validate_routing(cfg, ws)
        assert lm.lmoe_check_status(cfg, ws) == (0, 0), what


PAIR_SHAPE = dict(D=512, L=512, E=16, I=2560, k=8)   # the expert pair applies (8 x 20 gate/up tiles)


@pytest.mark.parametrize("weights,routing,T,shape", [("bf16", "uniform", 300, None), ("bf16", "zipf", 600, None),
                                                     ("nvfp4", "hot4", 40, None), ("nvfp4", "uniform", 2100, None),
                                                     ("f32", "uniform", 64, None), ("nvfp4", "hot4", 8, PAIR_SHAPE),
                                                     ("nvfp4", "uniform", 1, PAIR_SHAPE)])
def test_bounds_checked_build_matches_release(lm, weights, routing, T, shape):
    from conftest import build_checked_library
    from latent_mixture_experts_router_gb300 import _lib
    path = build_checked_library()
    chk = ctypes.CDLL(path)
    chk.latent_moe_forward_ex.argtypes = _lib._FWD_ARGS + [ctypes.POINTER(_lib.lmoe_ex)]
    chk.latent_moe_forward_ex.restype = ctypes.c_int
    chk.lmoe_check_status.argtypes = [ctypes.POINTER(_lib.lmoe_config), _lib._P, _lib._P,
                                      ctypes.POINTER(ctypes.c_uint32)]
    chk.lmoe_check_status.restype = ctypes.c_int
    act = "f32" if weights == "f32" else "bf16"
    dims = shape or dict(D=512, L=256, E=16, I=256, k=4)
    w = workloads.Workload(f"chk_{weights}_{T}", T=T, act=act, weights=weights, routing=routing, seed=T % 5, **dims)
    inp = workloads.make_inputs(w, torch.device("cuda:0"))
    ref, idx_ref, blk, cfg = run(inp)
    W = blk.W
    ws = torch.zeros(lm.lmoe_workspace_size(cfg), dtype=torch.uint8, device="cuda:0")
    out = torch.empty_like(ref)
    idx = torch.empty_like(idx_ref)
    keep = []
    args = _lib._fwd_args(cfg, inp.x, W["W_router"], W["W_pool"], W["g_pool"], W["W_gate"], W["W_up"], W["W_down"],
                          W["g_expert"], W["W_unpool"], W["g_pre"], W["g_post"], w.k, out, ws, None, keep)
    ex = _lib.lmoe_ex(_lib._ptr(inp.router_bias), _lib._ptr(inp.forced_idx), idx.data_ptr(), None, None, 0, None,
                      None, None)
    assert chk.latent_moe_forward_ex(*args, ctypes.byref(ex)) == 0
    word = ctypes.c_uint32()
    c = cfg.c()
    st = chk.lmoe_check_status(ctypes.byref(c), ws.data_ptr(), torch.cuda.current_stream().cuda_stream,
                               ctypes.byref(word))
    assert (st, word.value) == (0, 0)
    assert torch.equal(out, ref) and torch.equal(idx, idx_ref)
