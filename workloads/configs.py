"""The synthetic workloads of the latent-MoE block and their seeded tensors.

Shapes follow the Muse Spark Open layer: d_model 8192, pooled width 4096,
256 SwiGLU experts of intermediate 4096 (3*4096*4096 = 50.3M parameters per
expert; 256 experts x 62 layers = 799B, the weight budget of the vLLM day-0
post, "Model architecture" table), top-8 routing.  Distributions: x ~ N(0,1);
every W ~ N(0, 1/fan_in); RMSNorm gammas 1 + 0.1*N(0,1) in fp32; eps 1e-6.
x and the gammas are true Gaussians (``rng.gaussian``, Box-Muller, drawn on the
host and copied); the weights use the standardised Irwin-Hall(4) deviate of
``rng.normal`` (variance 1, support +-2*sqrt(3)), drawn on the device with
bit-identical values on any device, so a test can rebuild on the host exactly
the expert slices one token touches.  Nothing here computes any part of the
block.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

from . import rng

# stream ids, one per tensor
S_X, S_WROUTER, S_WPOOL, S_GPOOL, S_WGATE, S_WUP, S_WDOWN, S_GEXP, S_WUNPOOL, S_GPRE, S_GPOST = range(1, 12)
S_ZIPF_PERM, S_HOT_PERM, S_COLD = 12, 13, 14
S_HOT_TOKENS = 100          # + hot expert rank
S_SCALE_OFFSET = 1000       # NVFP4 block-scale codes of tensor s use stream s + 1000


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    D: int
    L: int
    E: int
    I: int
    k: int
    act: str = "bf16"        # dtype of x: "f32" | "bf16"
    weights: str = "bf16"    # "f32" | "bf16" | "nvfp4" (router stays bf16 when nvfp4)
    routing: str = "uniform"  # "uniform" | "zipf" | "hot4"
    eps: float = 1e-6
    seed: int = 0
    zipf_s: float = 1.1
    n_hot: int = 4

    def with_tokens(self, T: int) -> "Workload":
        return Workload(**{**self.__dict__, "T": T, "name": f"{self.name.split('@')[0]}@T{T}"})

    @property
    def R(self) -> int:
        return self.T * self.k


MUSE = dict(D=8192, L=4096, E=256, I=4096, k=8)

WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", T=64, D=512, L=256, E=16, I=512, k=2, act="f32", weights="f32"),
    "decode_bf16": Workload("decode_bf16", T=128, **MUSE),
    "prefill_bf16_zipf": Workload("prefill_bf16_zipf", T=16384, routing="zipf", **MUSE),
    "prefill_nvfp4": Workload("prefill_nvfp4", T=4096, weights="nvfp4", **MUSE),
    "decode_nvfp4_hot": Workload("decode_nvfp4_hot", T=128, weights="nvfp4", routing="hot4", **MUSE),
}
DECODE_SWEEP_T = (1, 8, 32, 128, 512)


# ---------------------------------------------------------------- dense tensors
def _to_dtype(v64: torch.Tensor, dtype: str) -> torch.Tensor:
    v32 = v64.to(torch.float32)          # RNE fp64 -> fp32
    if dtype == "f32":
        return v32
    return v32.to(torch.bfloat16)        # RNE fp32 -> bf16 (same two steps on every device)


def normal_tensor(w: Workload, stream: int, shape, std: float, dtype: str, device="cpu",
                  start: int = 0) -> torch.Tensor:
    n = math.prod(shape)
    return _to_dtype(rng.normal(w.seed, stream, start, n, std, device), dtype).reshape(shape)


def gamma_tensor(w: Workload, stream: int, shape, device="cpu", start: int = 0) -> torch.Tensor:
    n = math.prod(shape)
    z = rng.gaussian(w.seed, stream, start, n, 1.0)
    return (1.0 + z * 0.1).to(torch.float32).reshape(shape).to(device)


def x_tensor(w: Workload, device="cpu", rows=None, first_token: int = 0) -> torch.Tensor:
    """x [T, D] ~ N(0,1) (Box-Muller on the host, rounded fp64 -> fp32 (-> bf16), then copied):
    tokens first_token .. first_token+T-1 of one long seeded sequence; ``rows`` selects a
    subset of tokens instead (same values as in the full tensor)."""
    if rows is None:
        n = w.T * w.D
        out = torch.empty(n, dtype=torch.float32 if w.act == "f32" else torch.bfloat16)
        c = 1 << 22
        for s0 in range(0, n, c):   # converted chunk by chunk (one fp64 chunk live at a time)
            m = min(c, n - s0)
            out[s0:s0 + m] = _to_dtype(rng.gaussian(w.seed, S_X, first_token * w.D + s0, m, 1.0), w.act)
        return out.reshape(w.T, w.D).to(device)
    return torch.stack([_to_dtype(rng.gaussian(w.seed, S_X, int(t) * w.D, w.D, 1.0), w.act)
                        for t in rows]).to(device)


def dense_weight_dtype(w: Workload) -> str:
    return "f32" if w.weights == "f32" else "bf16"


# name -> (stream, per-expert?, rows, cols, fan_in)
def weight_specs(w: Workload):
    return {
        "W_router": (S_WROUTER, False, w.E, w.D, w.D),
        "W_pool": (S_WPOOL, False, w.L, w.D, w.D),
        "W_gate": (S_WGATE, True, w.I, w.L, w.L),
        "W_up": (S_WUP, True, w.I, w.L, w.L),
        "W_down": (S_WDOWN, True, w.L, w.I, w.I),
        "W_unpool": (S_WUNPOOL, False, w.D, w.L, w.L),
    }


def dense_weight(w: Workload, name: str, device="cpu", expert=None) -> torch.Tensor:
    """A dense (f32 or bf16) weight; ``expert`` picks one expert's [rows, cols] slice."""
    stream, per_e, rows, cols, fan_in = weight_specs(w)[name]
    dt = "bf16" if name == "W_router" and w.weights == "nvfp4" else dense_weight_dtype(w)
    std = 1.0 / math.sqrt(fan_in)
    if not per_e:
        return normal_tensor(w, stream, (rows, cols), std, dt, device)
    if expert is not None:
        return normal_tensor(w, stream, (rows, cols), std, dt, device, start=expert * rows * cols)
    return torch.stack([normal_tensor(w, stream, (rows, cols), std, dt, device, start=e * rows * cols)
                        for e in range(w.E)])


def gammas(w: Workload, device="cpu"):
    return {
        "g_pre": gamma_tensor(w, S_GPRE, (w.D,), device),
        "g_pool": gamma_tensor(w, S_GPOOL, (w.L,), device),
        "g_expert": gamma_tensor(w, S_GEXP, (w.E, w.L), device),
        "g_post": gamma_tensor(w, S_GPOST, (w.D,), device),
    }


# ---------------------------------------------------------------- NVFP4 weights
# Packed NVFP4 weights are drawn directly as codes, not by quantising a dense
# draw: sign uniform, E2M1 magnitude index from a fixed normal-like table, block
# scales uniform over the 17 E4M3 codes 0x30..0x40 (0.5 .. 2.0), and one fp32
# tensor scale that makes the dequantised standard deviation 1/sqrt(fan_in).
E2M1_MAG = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
_MAG_P = (0.14, 0.19, 0.17, 0.14, 0.11, 0.14, 0.07, 0.04)
_MAG_CUM16 = tuple(int(round(65536 * sum(_MAG_P[: i + 1]))) for i in range(8))
SCALE_CODE_LO, SCALE_CODE_HI = 0x30, 0x40


def _e4m3_value_for_generator(code: int) -> float:
    e, m = (code >> 3) & 15, code & 7
    return (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)


def nvfp4_tensor_scale(fan_in: int) -> float:
    """fp32 tensor scale so that code * block_scale * s has std 1/sqrt(fan_in)."""
    m2_code = sum(p * v * v for p, v in zip(_MAG_P, E2M1_MAG))
    sc = [_e4m3_value_for_generator(c) for c in range(SCALE_CODE_LO, SCALE_CODE_HI + 1)]
    m2_sc = sum(v * v for v in sc) / len(sc)
    return float(torch.tensor(1.0 / math.sqrt(fan_in * m2_code * m2_sc), dtype=torch.float32))


def nvfp4_weight(w: Workload, name: str, device="cpu", expert=None):
    """Packed NVFP4 weight: (codes u8 [.., rows, cols/2] low nibble = even column,
    scales u8 [.., rows, cols/16] E4M3 codes, tensor scale fp32 [E] or [1])."""
    stream, per_e, rows, cols, fan_in = weight_specs(w)[name]
    assert cols % 16 == 0
    experts = [None] if not per_e else ([expert] if expert is not None else list(range(w.E)))
    codes, scales = [], []
    for e in experts:
        base = 0 if e is None else e * rows * cols
        h = rng.uniform_bits(w.seed, stream, base, rows * cols, device)
        mag16 = h & 0xFFFF
        mag = torch.zeros_like(mag16)
        for c in _MAG_CUM16[:-1]:
            mag += (mag16 >= c).to(torch.int64)
        sign = rng._lsr(h, 63)
        nib = (sign << 3) | mag
        nib = nib.reshape(rows, cols // 2, 2)
        codes.append((nib[..., 0] | (nib[..., 1] << 4)).to(torch.uint8))
        hb = rng.uniform_bits(w.seed, stream + S_SCALE_OFFSET, base // 16, rows * cols // 16, device)
        span = SCALE_CODE_HI - SCALE_CODE_LO + 1
        sc = SCALE_CODE_LO + torch.remainder(rng._lsr(hb, 8), span)
        scales.append(sc.to(torch.uint8).reshape(rows, cols // 16))
    s = nvfp4_tensor_scale(fan_in)
    if per_e and expert is None:
        return torch.stack(codes), torch.stack(scales), torch.full((w.E,), s, dtype=torch.float32, device=device)
    n_s = 1
    return codes[0], scales[0], torch.full((n_s,), s, dtype=torch.float32, device=device)


# ---------------------------------------------------------------- routing inputs
def zipf_bias(w: Workload, device="cpu") -> torch.Tensor:
    """Per-expert logit bias b[pi(r)] = -s*ln(r), r = 1..E, pi a seeded permutation:
    router probability of the rank-r expert then scales as r^-s (Zipf)."""
    perm = rng.permutation(w.seed, S_ZIPF_PERM, w.E)
    b = torch.empty(w.E, dtype=torch.float64)
    for r in range(1, w.E + 1):
        b[perm[r - 1]] = -w.zipf_s * math.log(r)
    return b.to(torch.float32).to(device)


def hot_experts(w: Workload):
    return [int(e) for e in rng.permutation(w.seed, S_HOT_PERM, w.E)[: w.n_hot]]


def forced_routing(w: Workload, device="cpu") -> torch.Tensor:
    """[T, k] int32 expert ids: each of the n_hot hot experts takes ceil(T/2) tokens
    (sampled without replacement); every token's other slots are filled, without
    replacement, uniformly from the cold experts."""
    hot = hot_experts(w)
    take = (w.T + 1) // 2
    chosen = [[] for _ in range(w.T)]
    for r, e in enumerate(hot):
        toks = rng.permutation(w.seed, S_HOT_TOKENS + r, w.T)[:take]
        for t in sorted(int(t) for t in toks):
            chosen[t].append(e)
    cold = [e for e in range(w.E) if e not in hot]
    out = torch.empty(w.T, w.k, dtype=torch.int32)
    for t in range(w.T):
        need = w.k - len(chosen[t])
        h = rng.uniform_bits(w.seed, S_COLD, t * w.E, w.E)
        keys = rng._lsr(h, 2)[cold]
        order = torch.sort(keys, stable=True).indices[:need]
        ids = chosen[t] + [cold[int(i)] for i in order]
        out[t] = torch.tensor(ids, dtype=torch.int32)
    return out.to(device)


@dataclass
class BlockInputs:
    """All inputs of one block call, as torch tensors on one device."""
    w: Workload
    x: torch.Tensor
    W_router: torch.Tensor
    W_pool: object
    W_gate: object
    W_up: object
    W_down: object
    W_unpool: object
    g_pre: torch.Tensor
    g_pool: torch.Tensor
    g_expert: torch.Tensor
    g_post: torch.Tensor
    router_bias: torch.Tensor | None = None
    forced_idx: torch.Tensor | None = None
    extra: dict = field(default_factory=dict)


def make_inputs(w: Workload, device="cpu") -> BlockInputs:
    """Every input of workload ``w`` on ``device`` (NVFP4 weights as (codes, scales, s))."""
    g = gammas(w, device)
    wt = {}
    for name in ("W_pool", "W_gate", "W_up", "W_down", "W_unpool"):
        wt[name] = nvfp4_weight(w, name, device) if w.weights == "nvfp4" else dense_weight(w, name, device)
    return BlockInputs(
        w=w, x=x_tensor(w, device), W_router=dense_weight(w, "W_router", device), **wt, **g,
        router_bias=zipf_bias(w, device) if w.routing == "zipf" else None,
        forced_idx=forced_routing(w, device) if w.routing == "hot4" else None,
    )


def to_device(inp: BlockInputs, device) -> BlockInputs:
    """The same inputs copied to ``device`` (tensors, and the tensors of NVFP4 triples)."""
    import dataclasses

    def mv(v):
        if isinstance(v, tuple):
            return tuple(t.to(device) for t in v)
        return v.to(device) if isinstance(v, torch.Tensor) else v
    return dataclasses.replace(inp, **{f.name: mv(getattr(inp, f.name)) for f in dataclasses.fields(inp)
                                       if f.name not in ("w", "extra")})

