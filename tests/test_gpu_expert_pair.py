"""GPU parity of the expert pair: the grouped gate/up and down GEMMs of a few tokens (every M
tile at most 32 rows, gate/up tiles for every SM) as one persistent launch.

* Against the fp64 oracle under the NVFP4 rules, at T = 1 (the single-token path around it),
  ragged T = 3, T = 8 and T = 32 (hot experts; every token on the same k experts: M tiles of
  exactly 32 rows), bf16 and fp32 activations and outputs.
* Against the two separate GEMM launches on the same inputs (lmoe_ex.separate_expert_gemms):
  the same h codes, y and output bit for bit (the pair computes every tile with the same MMAs
  in the same K order and the same epilogues).  lmoe_expert_pair says which calls take it.
* The ready counts left in the tile table: every live M tile counted by all 8 epilogue warps of
  each of its I / 128 gate/up tiles (zero where the separate GEMMs ran).
* Waits that run out end the call with LMOE_ERR_TIMEOUT and leave the context usable."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle.compare import TOL_NVFP4, compare_block

from gpu_util import make_block, run, views

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()
    return torch.device("cuda:0")


# (T, D, L, E, I, k, act, routing): k * I / 128 >= 152 gate/up tiles, L a multiple of 256
SHAPES = [
    (1, 512, 512, 16, 2560, 8, "bf16", "uniform"),
    (3, 512, 768, 16, 1280, 16, "f32", "uniform"),
    (8, 1024, 512, 64, 2560, 8, "bf16", "hot4"),
    (32, 1024, 512, 32, 2560, 8, "bf16", "hot4"),
    (32, 512, 1024, 24, 2560, 8, "bf16", "same"),
    (2, 256, 512, 1024, 1280, 16, "bf16", "uniform"),   # the header's limits: E = 1024, k = 16
]


def _inputs(T, D, L, E, I, k, act, routing, device, seed=7):
    w = workloads.Workload(f"pair_{T}_{D}_{L}_{E}_{I}_{k}_{act}_{routing}", T=T, D=D, L=L, E=E, I=I, k=k,
                           act=act, weights="nvfp4", routing="uniform" if routing == "same" else routing,
                           seed=seed)
    inp = workloads.make_inputs(w, device)
    if routing == "same":   # every token on experts 0 .. k-1: k M tiles of T rows
        inp.forced_idx = torch.arange(k, dtype=torch.int32, device=device).repeat(T, 1).contiguous()
    return w, inp


def _h_codes(lm, blk, cfg, R, I):
    lay = lm.lmoe_get_workspace_layout(cfg)
    return blk._ws[lay["h"]:lay["h"] + R * I // 2].view(R, I // 2).cpu().numpy().copy()


@pytest.mark.parametrize("T,D,L,E,I,k,act,routing", SHAPES)
def test_expert_pair_parity_with_oracle(cuda, T, D, L, E, I, k, act, routing):
    w, inp = _inputs(T, D, L, E, I, k, act, routing, cuda)
    out, idx, blk, cfg = run(inp)
    P = oracle.params_from_inputs(inp)
    x = inp.x.double().cpu().numpy()
    forced = None if inp.forced_idx is None else inp.forced_idx.cpu().numpy()
    tr = oracle.Trace()
    ref = oracle.forward_batched(x, P, k, trace=tr, forced_idx=forced)
    rep = compare_block(out.cpu().numpy(), idx.cpu().numpy(), x, P, k, TOL_NVFP4, tr=tr, ref=ref, forced_idx=forced)
    print(w.name, rep)
    assert rep.ok, str(rep)


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,D,L,E,I,k,act,routing", SHAPES)
def test_expert_pair_matches_separate_gemms(cuda, T, D, L, E, I, k, act, routing, out_dtype):
    import latent_mixture_experts_router_gb300 as lm
    w, inp = _inputs(T, D, L, E, I, k, act, routing, cuda, seed=11)
    blk = make_block(inp)
    path = {"single_token_path": lm.SINGLE_TOKEN_CHAIN} if T == 1 else {}

    def tile_table(cfg, vw):
        n_tiles = int(vw["n_tiles"][0])
        o = lm.lmoe_get_workspace_layout(cfg)["tiles"]
        return blk._ws[o:o + 16 * n_tiles].view(torch.int32).view(n_tiles, 4).cpu().numpy()

    out_s, idx_s, _, cfg = run(inp, blk=blk, out_dtype=out_dtype, separate_expert_gemms=True, **path)
    assert lm.lmoe_expert_pair(cfg)
    out_s = out_s.clone()
    vs = views(blk, cfg)
    R = T * k
    h_s = _h_codes(lm, blk, cfg, R, I)
    # the separate GEMMs leave the ready counts as the table was written: zero
    assert (tile_table(cfg, vs)[:, 3] == 0).all()
    out_p, idx_p, _, _ = run(inp, blk=blk, out_dtype=out_dtype, **path)
    vp = views(blk, cfg)
    h_p = _h_codes(lm, blk, cfg, R, I)
    assert torch.equal(idx_p, idx_s)
    rows = vp["row_of"].reshape(-1)
    assert np.array_equal(h_p[rows], h_s[rows])
    assert np.array_equal(vp["y"][rows], vs["y"][rows])
    assert torch.equal(out_p, out_s)
    # the pair ran: every live M tile counted by the 8 epilogue warps of each of its gate/up tiles
    tiles = tile_table(cfg, vp)
    assert (tiles[:, 3] == 8 * (I // 128)).all(), tiles[:, 3]
    assert (tiles[:, 2] <= 32).all()


@pytest.mark.parametrize("T", [1, 8])
def test_expert_pair_timeout_is_reported_and_context_survives(cuda, T):
    import latent_mixture_experts_router_gb300 as lm
    w, inp = _inputs(T, 512, 512, 16, 2560, 8, "bf16", "uniform", cuda, seed=13)
    blk = make_block(inp)
    path = {"single_token_path": lm.SINGLE_TOKEN_CHAIN} if T == 1 else {}
    ref, _, _, cfg = run(inp, blk=blk, **path)
    ref = ref.clone()
    blk.forward(inp.x, wait_budget_cycles=1, **path)   # every wait gives up at once
    st, word = lm.lmoe_check_status(cfg, blk._ws)
    assert st == -6, (st, hex(word))
    out, _, _, _ = run(inp, blk=blk, **path)
    assert torch.equal(out, ref)


def test_expert_pair_with_stage_events(cuda):
    # stage events keep the pair: the gate_up stage spans both GEMMs, the down stage is empty,
    # and the output is the one without events
    import latent_mixture_experts_router_gb300 as lm
    w, inp = _inputs(8, 1024, 512, 64, 2560, 8, "bf16", "hot4", cuda, seed=17)
    blk = make_block(inp)
    ref, _, _, cfg = run(inp, blk=blk)
    ref = ref.clone()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(lm.NUM_STAGE_EVENTS)]
    out, _, _, _ = run(inp, blk=blk, stage_events=evs)
    assert torch.equal(out, ref)
    g, d = lm.STAGES.index("gate_up"), lm.STAGES.index("down")
    assert evs[g].elapsed_time(evs[g + 1]) > 0
    assert evs[d].elapsed_time(evs[d + 1]) < 0.1 * evs[g].elapsed_time(evs[g + 1])
    n_tiles = int(views(blk, cfg)["n_tiles"][0])
    o = lm.lmoe_get_workspace_layout(cfg)["tiles"]
    tiles = blk._ws[o:o + 16 * n_tiles].view(torch.int32).view(n_tiles, 4).cpu().numpy()
    assert (tiles[:, 3] == 8 * (2560 // 128)).all()
