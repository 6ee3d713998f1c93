"""ctypes binding of liblatent_moe.so (include/latent_moe.h), argument marshalling only.

Every function here turns torch tensors into device pointers, calls the C entry
point of the same name, and raises ``LmoeError`` on a non-zero status.  No part
of the block is computed in Python; if the shared library is missing, importing
it fails loudly (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblatent_moe.so")

LMOE_F32, LMOE_BF16, LMOE_NVFP4 = 0, 1, 2
_DT = {"f32": LMOE_F32, "bf16": LMOE_BF16, "nvfp4": LMOE_NVFP4}

STATUS = {0: "LMOE_OK", -1: "LMOE_ERR_ARG", -2: "LMOE_ERR_UNSUPPORTED", -3: "LMOE_ERR_ALIGN",
          -4: "LMOE_ERR_WORKSPACE", -5: "LMOE_ERR_CUDA", -6: "LMOE_ERR_TIMEOUT"}


class LmoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({_lib().lmoe_status_string(status).decode()})")


class lmoe_config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d_model", ctypes.c_int), ("d_latent", ctypes.c_int),
                ("n_experts", ctypes.c_int), ("d_ff", ctypes.c_int), ("top_k", ctypes.c_int),
                ("eps", ctypes.c_float), ("act_dtype", ctypes.c_int), ("weight_dtype", ctypes.c_int),
                ("out_dtype", ctypes.c_int)]


SCALES_ROW_MAJOR, SCALES_BLOCKED = 0, 1   # lmoe_nvfp4_scale_layout


class lmoe_nvfp4_weight(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("tensor_scale", ctypes.c_void_p),
                ("scale_layout", ctypes.c_int)]


class lmoe_ex(ctypes.Structure):
    _fields_ = [("router_bias", ctypes.c_void_p), ("forced_idx", ctypes.c_void_p),
                ("topk_idx_out", ctypes.c_void_p), ("topk_w_out", ctypes.c_void_p),
                ("near_tie_count_out", ctypes.c_void_p), ("wait_budget_cycles", ctypes.c_longlong),
                ("stage_events", ctypes.c_void_p), ("next_norm_gamma", ctypes.c_void_p),
                ("next_norm_out", ctypes.c_void_p), ("single_token_path", ctypes.c_int),
                ("separate_expert_gemms", ctypes.c_int), ("cooperative_launch", ctypes.c_int)]

SINGLE_TOKEN_DEFAULT, SINGLE_TOKEN_KERNEL, SINGLE_TOKEN_CHAIN = 0, 1, 2   # lmoe_ex.single_token_path

STAGES = ["prenorm", "router", "topk", "permute", "pooler", "poolnorm", "gate_up", "down", "combine",
          "unpooler", "postnorm"]
NUM_STAGE_EVENTS = len(STAGES) + 1


_LAYOUT_FIELDS = ["xa", "logits", "topk_idx", "topk_w", "counts", "offsets", "row_of", "tok_of",
                  "tiles", "n_tiles", "p", "ss_p", "xe", "xe_scale", "h", "y", "ss_y", "c", "u",
                  "ss_u", "err", "total"]


_LAYOUT_FIELDS_NVFP4 = ["xq", "xq_scale", "xq_rowscale", "xe_rowscale", "h_scale", "c_scale", "c_rowscale"]


class lmoe_workspace_layout(ctypes.Structure):
    _fields_ = ([(f, ctypes.c_longlong) for f in _LAYOUT_FIELDS + _LAYOUT_FIELDS_NVFP4]
                + [("xa_cols", ctypes.c_int), ("grouped_splits", ctypes.c_longlong)])


_P = ctypes.c_void_p
_FWD_ARGS = [ctypes.POINTER(lmoe_config), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
             ctypes.c_int, _P, _P, ctypes.c_size_t, _P]
_lib_handle = None


def _lib():
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built; run latent_mixture_experts_router_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        L.lmoe_status_string.restype = ctypes.c_char_p
        L.lmoe_status_string.argtypes = [ctypes.c_int]
        for name in ("lmoe_workspace_size", "lmoe_workspace_size_host_io"):
            getattr(L, name).argtypes = [ctypes.POINTER(lmoe_config), ctypes.POINTER(ctypes.c_size_t)]
            getattr(L, name).restype = ctypes.c_int
        L.lmoe_get_workspace_layout.argtypes = [ctypes.POINTER(lmoe_config), ctypes.POINTER(lmoe_workspace_layout)]
        L.lmoe_get_workspace_layout.restype = ctypes.c_int
        L.latent_moe_forward.argtypes = _FWD_ARGS
        L.latent_moe_forward.restype = ctypes.c_int
        L.latent_moe_forward_ex.argtypes = _FWD_ARGS + [ctypes.POINTER(lmoe_ex)]
        L.latent_moe_forward_ex.restype = ctypes.c_int
        L.latent_moe_forward_host_io.argtypes = _FWD_ARGS
        L.latent_moe_forward_host_io.restype = ctypes.c_int
        L.latent_moe_forward_host_io_ex.argtypes = _FWD_ARGS + [ctypes.POINTER(lmoe_ex)]
        L.latent_moe_forward_host_io_ex.restype = ctypes.c_int
        L.lmoe_check_status.argtypes = [ctypes.POINTER(lmoe_config), _P, _P, ctypes.POINTER(ctypes.c_uint32)]
        L.lmoe_check_status.restype = ctypes.c_int
        L.lmoe_wait_selftest.argtypes = [ctypes.POINTER(lmoe_config), _P, ctypes.c_longlong, _P]
        L.lmoe_wait_selftest.restype = ctypes.c_int
        L.lmoe_expert_pair.argtypes = [ctypes.POINTER(lmoe_config), ctypes.POINTER(ctypes.c_int)]
        L.lmoe_expert_pair.restype = ctypes.c_int
        L.lmoe_kernel_launches.restype = ctypes.c_ulonglong
        L.lmoe_kernel_launches.argtypes = []
        _lib_handle = L
    return _lib_handle


def load():
    """Load the shared library (raises ImportError if it is not built)."""
    return _lib()


# ------------------------------------------------------------------ config
@dataclass
class Config:
    T: int
    d_model: int
    d_latent: int
    n_experts: int
    d_ff: int
    top_k: int
    eps: float = 1e-6
    act_dtype: str = "bf16"
    weight_dtype: str = "bf16"
    out_dtype: str = "f32"

    def c(self) -> lmoe_config:
        return lmoe_config(self.T, self.d_model, self.d_latent, self.n_experts, self.d_ff, self.top_k,
                           self.eps, _DT[self.act_dtype], _DT[self.weight_dtype], _DT[self.out_dtype])


def _check(status: int, where: str):
    if status != 0:
        raise LmoeError(status, where)


def _ptr(t) -> int:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _weight_arg(w, keep: list):
    """A dense tensor -> its pointer; an NVFP4 (codes, scales, tensor_scale[, scale_layout])
    tuple -> a pointer to a host lmoe_nvfp4_weight (kept alive in ``keep``).  Without a fourth
    element the scales are declared row-major (which the forward refuses: convert them with
    lmoe_nvfp4_block_scales and pass SCALES_BLOCKED)."""
    if isinstance(w, tuple):
        layout = w[3] if len(w) > 3 else SCALES_ROW_MAJOR
        s = lmoe_nvfp4_weight(_ptr(w[0]), _ptr(w[1]), _ptr(w[2]), int(layout))
        keep.append(s)
        return ctypes.addressof(s)
    return _ptr(w)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def lmoe_workspace_size(cfg: Config) -> int:
    n = ctypes.c_size_t()
    c = cfg.c()
    _check(_lib().lmoe_workspace_size(ctypes.byref(c), ctypes.byref(n)), "lmoe_workspace_size")
    return n.value


def lmoe_workspace_size_host_io(cfg: Config) -> int:
    n = ctypes.c_size_t()
    c = cfg.c()
    _check(_lib().lmoe_workspace_size_host_io(ctypes.byref(c), ctypes.byref(n)), "lmoe_workspace_size_host_io")
    return n.value


def lmoe_expert_pair(cfg: Config) -> bool:
    """Whether a call with ``cfg`` runs the grouped gate/up and down GEMMs as one launch."""
    used = ctypes.c_int()
    c = cfg.c()
    _check(_lib().lmoe_expert_pair(ctypes.byref(c), ctypes.byref(used)), "lmoe_expert_pair")
    return bool(used.value)


def lmoe_get_workspace_layout(cfg: Config) -> dict:
    lay = lmoe_workspace_layout()
    c = cfg.c()
    _check(_lib().lmoe_get_workspace_layout(ctypes.byref(c), ctypes.byref(lay)), "lmoe_get_workspace_layout")
    d = {f: getattr(lay, f) for f in _LAYOUT_FIELDS + _LAYOUT_FIELDS_NVFP4}
    d["xa_cols"] = lay.xa_cols
    d["grouped_splits"] = lay.grouped_splits
    return d


def _fwd_args(cfg, x, W_router, W_pool, g_pool, W_gate, W_up, W_down, g_expert, W_unpool, g_pre,
              g_post, top_k, out, workspace, stream, keep):
    c = cfg.c()
    keep.append(c)
    return [ctypes.byref(c), _ptr(x), _ptr(W_router), _weight_arg(W_pool, keep), _ptr(g_pool),
            _weight_arg(W_gate, keep), _weight_arg(W_up, keep), _weight_arg(W_down, keep), _ptr(g_expert),
            _weight_arg(W_unpool, keep), _ptr(g_pre), _ptr(g_post), int(top_k), _ptr(out),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)]


def latent_moe_forward(cfg, x, W_router, W_pool, g_pool, W_gate, W_up, W_down, g_expert, W_unpool,
                       g_pre, g_post, top_k, out, workspace, stream=None):
    keep = []
    args = _fwd_args(cfg, x, W_router, W_pool, g_pool, W_gate, W_up, W_down, g_expert, W_unpool, g_pre,
                     g_post, top_k, out, workspace, stream, keep)
    _check(_lib().latent_moe_forward(*args), "latent_moe_forward")


def latent_moe_forward_ex(cfg, x, W_router, W_pool, g_pool, W_gate, W_up, W_down, g_expert, W_unpool,
                          g_pre, g_post, top_k, out, workspace, stream=None, router_bias=None,
                          forced_idx=None, topk_idx_out=None, topk_w_out=None, near_tie_count_out=None,
                          wait_budget_cycles=0, stage_events=None, next_norm_gamma=None, next_norm_out=None,
                          single_token_path=0, separate_expert_gemms=False, cooperative_launch=False):
    """``stage_events``: a list of NUM_STAGE_EVENTS torch.cuda.Event(enable_timing=True) or None,
    recorded by the library at the stage boundaries (for per-stage timing; None entries are
    skipped).  ``single_token_path``: with NVFP4 weights and one token, which kernels run
    (SINGLE_TOKEN_DEFAULT, SINGLE_TOKEN_KERNEL or SINGLE_TOKEN_CHAIN; lmoe_ex.single_token_path).
    ``separate_expert_gemms``: gate/up and down as two launches where lmoe_expert_pair() says one.
    ``cooperative_launch``: the single-token persistent kernels launched cooperatively."""
    keep = []
    args = _fwd_args(cfg, x, W_router, W_pool, g_pool, W_gate, W_up, W_down, g_expert, W_unpool, g_pre,
                     g_post, top_k, out, workspace, stream, keep)
    evs = None
    if stage_events is not None:
        assert len(stage_events) == NUM_STAGE_EVENTS
        for e in stage_events:   # torch creates the CUDA event lazily
            if e is not None and e.cuda_event == 0:
                e.record()
        evs = (ctypes.c_void_p * NUM_STAGE_EVENTS)(*[e.cuda_event if e is not None else None
                                                     for e in stage_events])
        keep.append(evs)
    ex = lmoe_ex(_ptr(router_bias), _ptr(forced_idx), _ptr(topk_idx_out), _ptr(topk_w_out),
                 _ptr(near_tie_count_out), int(wait_budget_cycles),
                 ctypes.cast(evs, ctypes.c_void_p) if evs is not None else None,
                 _ptr(next_norm_gamma), _ptr(next_norm_out), int(single_token_path),
                 1 if separate_expert_gemms else 0, 1 if cooperative_launch else 0)
    _check(_lib().latent_moe_forward_ex(*args, ctypes.byref(ex)), "latent_moe_forward_ex")


def latent_moe_forward_host_io(cfg, x_host, W_router, W_pool, g_pool, W_gate, W_up, W_down, g_expert,
                               W_unpool, g_pre, g_post, top_k, out_host, workspace, stream=None):
    keep = []
    args = _fwd_args(cfg, x_host, W_router, W_pool, g_pool, W_gate, W_up, W_down, g_expert, W_unpool,
                     g_pre, g_post, top_k, out_host, workspace, stream, keep)
    _check(_lib().latent_moe_forward_host_io(*args), "latent_moe_forward_host_io")


def latent_moe_forward_host_io_ex(cfg, x_host, W_router, W_pool, g_pool, W_gate, W_up, W_down, g_expert,
                                  W_unpool, g_pre, g_post, top_k, out_host, workspace, stream=None,
                                  router_bias=None, forced_idx=None, single_token_path=0):
    """latent_moe_forward_host_io with the device-resident routing extensions of lmoe_ex."""
    keep = []
    args = _fwd_args(cfg, x_host, W_router, W_pool, g_pool, W_gate, W_up, W_down, g_expert, W_unpool,
                     g_pre, g_post, top_k, out_host, workspace, stream, keep)
    ex = lmoe_ex(_ptr(router_bias), _ptr(forced_idx), None, None, None, 0, None, None, None,
                 int(single_token_path), 0, 0)
    _check(_lib().latent_moe_forward_host_io_ex(*args, ctypes.byref(ex)), "latent_moe_forward_host_io_ex")


def lmoe_check_status(cfg, workspace, stream=None) -> tuple[int, int]:
    """(status, raw error word) of the last calls on ``workspace``; synchronises the stream."""
    c = cfg.c()
    word = ctypes.c_uint32()
    st = _lib().lmoe_check_status(ctypes.byref(c), _ptr(workspace), _stream(stream), ctypes.byref(word))
    return st, word.value


def lmoe_wait_selftest(cfg, workspace, budget_cycles: int, stream=None):
    """Run the wait-timeout diagnostic; lmoe_check_status() then reports the timeout."""
    c = cfg.c()
    _check(_lib().lmoe_wait_selftest(ctypes.byref(c), _ptr(workspace), int(budget_cycles), _stream(stream)),
           "lmoe_wait_selftest")


GUARD_BYTES = 256   # LMOE_GUARD_BYTES


def lmoe_workspace_guards(cfg, host_io: bool = False, lib=None) -> list:
    """Byte offsets of the workspace's guard bands (each GUARD_BYTES long)."""
    L = lib or _lib()
    fn = L.lmoe_workspace_guards
    fn.argtypes = [ctypes.POINTER(lmoe_config), ctypes.c_int, _P, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    fn.restype = ctypes.c_int
    c = cfg.c()
    n = ctypes.c_int()
    _check(fn(ctypes.byref(c), 1 if host_io else 0, None, 0, ctypes.byref(n)), "lmoe_workspace_guards")
    arr = (ctypes.c_longlong * max(n.value, 1))()
    _check(fn(ctypes.byref(c), 1 if host_io else 0, ctypes.cast(arr, _P), n.value, ctypes.byref(n)),
           "lmoe_workspace_guards")
    return list(arr[:n.value])


def lmoe_validate_routing(cfg, workspace, stream=None, lib=None):
    """Check the routing structures the last call left in ``workspace``; a violation shows in
    lmoe_check_status (LMOE_ERR_ARG, bit 0x20 of the error word)."""
    L = lib or _lib()
    fn = L.lmoe_validate_routing
    fn.argtypes = [ctypes.POINTER(lmoe_config), _P, _P]
    fn.restype = ctypes.c_int
    c = cfg.c()
    _check(fn(ctypes.byref(c), _ptr(workspace), _stream(stream)), "lmoe_validate_routing")


def lmoe_kernel_launches() -> int:
    """Kernels the library has launched in this process."""
    return int(_lib().lmoe_kernel_launches())


def lmoe_permute_noalloc(topk_idx, E: int, offsets, row_of, tok_of, stream=None):
    """Expert-contiguous permutation of ``topk_idx`` [T, k] (int32, device) into ``offsets``
    [E+1], ``row_of`` [T, k] and ``tok_of`` [T*k] without any device allocation: the library's
    fixed scratch array is used instead of a workspace (E <= 1024, T*k <= 65536)."""
    L = _lib()
    fn = L.lmoe_permute_noalloc
    fn.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P, _P]
    fn.restype = ctypes.c_int
    T, k = topk_idx.shape
    # the library looks its scratch up for the current device: make the ids' device current
    # and take the stream from it
    with torch.cuda.device(topk_idx.device):
        st = _stream(stream if stream is not None else torch.cuda.current_stream(topk_idx.device))
        _check(fn(_ptr(topk_idx), T, k, int(E), _ptr(offsets), _ptr(row_of), _ptr(tok_of), st),
               "lmoe_permute_noalloc")


def lmoe_quantize_nvfp4(src, codes, scales, s_row=None, row_scale=True, stream=None):
    """NVFP4-quantise the fp32 rows of ``src`` [rows, K] (device) with the block's activation rule."""
    L = _lib()
    fn = L.lmoe_quantize_nvfp4
    fn.argtypes = [_P, ctypes.c_longlong, ctypes.c_int, ctypes.c_int, _P, _P, _P, _P]
    fn.restype = ctypes.c_int
    rows, K = src.shape
    _check(fn(_ptr(src), rows, K, 1 if row_scale else 0, _ptr(codes), _ptr(scales), _ptr(s_row),
              _stream(stream)), "lmoe_quantize_nvfp4")


def lmoe_nvfp4_block_scales(src, K: int, block_rows: int = 128, dst=None, stream=None):
    """Row-major E4M3 scales ``src`` [..., rows, K/16] (uint8, device) -> the block layout the
    NVFP4 GEMMs read, in blocks of ``block_rows`` (128, or 64 for W_gate/W_up) rows; returns a
    flat uint8 tensor unless ``dst`` is given."""
    L = _lib()
    fn = L.lmoe_nvfp4_block_scales
    fn.argtypes = [_P, ctypes.c_longlong, ctypes.c_int, ctypes.c_int, _P, _P]
    fn.restype = ctypes.c_int
    rows = src.numel() // (K // 16)
    if dst is None:
        dst = torch.zeros(rows // block_rows * (K // 64) * 512, dtype=torch.uint8, device=src.device)
    _check(fn(_ptr(src), rows, int(K), int(block_rows), _ptr(dst), _stream(stream)),
           "lmoe_nvfp4_block_scales")
    return dst
