"""The C ABI loads and exports every function include/latent_moe.h declares, and rejects
bad arguments on the host before any launch (no GPU needed for these paths)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lm():
    from conftest import build_library
    build_library()
    import latent_mixture_experts_router_gb300 as lm
    return lm


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:lmoe_status|const char\*)\s+(\w+)\s*\(", src, flags=re.M)
    return names


def test_exports_every_declared_symbol(lm):
    names = declared_functions()
    assert "latent_moe_forward" in names and len(names) >= 8
    lib = ctypes.CDLL(lm.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lm):
    lib = lm.load()
    for s in range(-6, 1):
        assert lib.lmoe_status_string(s)


def test_workspace_sizes_and_layout(lm):
    c = lm.Config(128, 8192, 4096, 256, 4096, 8)
    n = lm.lmoe_workspace_size(c)
    lay = lm.lmoe_get_workspace_layout(c)
    assert lay["total"] == n and lay["xa_cols"] == 2 * 8192
    offs = sorted(v for k, v in lay.items() if k not in ("total", "xa_cols") and v >= 0)
    assert all(o % 256 == 0 for o in offs)
    assert lm.lmoe_workspace_size_host_io(c) > n
    # f32 weights need the bf16 copies and the 3-way router split
    c32 = lm.Config(64, 512, 256, 16, 512, 2, act_dtype="f32", weight_dtype="f32")
    assert lm.lmoe_get_workspace_layout(c32)["xa_cols"] == 3 * 512


def test_expert_pair_rule(lm):
    # host arithmetic: NVFP4, T <= 32 and at least 152 gate/up tiles of 128 columns among
    # max(top_k, T top_k / 128) M tiles (NVFP4 configs have d_latent % 256 == 0)
    muse = dict(d_model=8192, d_latent=4096, n_experts=256, d_ff=4096, top_k=8, weight_dtype="nvfp4")
    for T in (1, 8, 32):
        assert lm.lmoe_expert_pair(lm.Config(T, **muse))
    assert not lm.lmoe_expert_pair(lm.Config(33, **muse))                         # more rows
    assert not lm.lmoe_expert_pair(lm.Config(8, **dict(muse, weight_dtype="bf16")))
    assert not lm.lmoe_expert_pair(lm.Config(1, **dict(muse, d_ff=2304)))         # 8 x 18 = 144
    assert not lm.lmoe_expert_pair(lm.Config(1, **dict(muse, top_k=4, d_ff=4608)))   # 4 x 36
    assert lm.lmoe_expert_pair(lm.Config(1, **dict(muse, top_k=4, d_ff=4864)))   # 4 x 38 = 152
    assert lm.lmoe_expert_pair(lm.Config(3, **dict(muse, top_k=16, d_ff=1280)))   # 16 x 10
    assert not lm.lmoe_expert_pair(lm.Config(2, **dict(muse, top_k=2, d_ff=8192)))   # 2 x 64


@pytest.mark.parametrize("kw,status", [
    (dict(top_k=0), -1), (dict(top_k=17), -1), (dict(n_experts=4, top_k=5), -1),
    (dict(d_model=200), -2), (dict(d_latent=96), -2), (dict(n_experts=2048), -2),
    (dict(T=-1), -1), (dict(eps=-1.0), -1),
])
def test_config_rejected(lm, kw, status):
    base = dict(T=8, d_model=256, d_latent=128, n_experts=8, d_ff=128, top_k=2)
    base.update(kw)
    with pytest.raises(lm.LmoeError) as ei:
        lm.lmoe_workspace_size(lm.Config(**base))
    assert ei.value.status == status


def test_forward_rejects_bad_pointers_without_launching(lm):
    lib = lm.load()
    from latent_mixture_experts_router_gb300._lib import lmoe_config
    c = lm.Config(8, 256, 128, 8, 128, 2).c()
    fake = 1 << 20   # never dereferenced: validation fails first
    args = [ctypes.byref(c)] + [fake] * 11
    # NULL x
    st = lib.latent_moe_forward(ctypes.byref(c), None, *[fake] * 10, 2, fake, fake, 1 << 30, None)
    assert st == -1
    # top_k argument disagreeing with the config
    st = lib.latent_moe_forward(*args, 3, fake, fake, 1 << 30, None)
    assert st == -1
    # misaligned pointer
    st = lib.latent_moe_forward(ctypes.byref(c), fake + 2, *[fake] * 10, 2, fake, fake, 1 << 30, None)
    assert st == -3
    # workspace too small
    st = lib.latent_moe_forward(*args, 2, fake + 4096, fake, 16, None)
    assert st == -4
    assert isinstance(lmoe_config, type)


def test_next_norm_arguments_checked_without_launching(lm):
    # the fused next-layer pre-norm needs both its gamma and its output, 16-byte aligned
    lib = lm.load()
    from latent_mixture_experts_router_gb300._lib import lmoe_ex
    c = lm.Config(8, 256, 128, 8, 128, 2).c()
    fake = 1 << 20   # never dereferenced: validation fails first
    args = [ctypes.byref(c)] + [fake] * 11 + [2, fake, fake, 1 << 30, None]
    only_gamma = lmoe_ex(None, None, None, None, None, 0, None, fake, None)
    assert lib.latent_moe_forward_ex(*args, ctypes.byref(only_gamma)) == -1
    only_out = lmoe_ex(None, None, None, None, None, 0, None, None, fake)
    assert lib.latent_moe_forward_ex(*args, ctypes.byref(only_out)) == -1
    misaligned = lmoe_ex(None, None, None, None, None, 0, None, fake, fake + 4)
    assert lib.latent_moe_forward_ex(*args, ctypes.byref(misaligned)) == -3


def _noalloc_fn(lm):
    fn = lm.load().lmoe_permute_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


@pytest.mark.parametrize("which", range(4))
def test_no_alloc_rejects_misaligned_arrays_without_launching(lm, which):
    # the allocation-free permutation does int32 loads and stores on its four arrays: a
    # pointer that is not 4-byte aligned is refused on the host (no GPU touched)
    fake = [1 << 20, 1 << 21, 1 << 22, 1 << 23]   # never dereferenced
    fake[which] += 2
    idx, offsets, row_of, tok_of = fake
    assert _noalloc_fn(lm)(idx, 8, 2, 16, offsets, row_of, tok_of, None) == -3


@pytest.mark.parametrize("T,k,E,status", [(8, 2, 1025, -2), (32769, 2, 64, -2), (8, 0, 16, -1),
                                          (8, 17, 32, -1), (8, 4, 2, -1)])
def test_no_alloc_rejects_sizes_without_launching(lm, T, k, E, status):
    fake = 1 << 20
    assert _noalloc_fn(lm)(fake, T, k, E, fake, fake, fake, None) == status


@pytest.mark.parametrize("layout,status", [(0, -2), (1, -4)])
def test_nvfp4_scale_layout_is_checked_without_launching(lm, layout, status):
    # row-major scales (the zero value of the field) are refused before any launch; with the
    # block layout declared the call gets as far as the (too small) workspace check
    lib = lm.load()
    from latent_mixture_experts_router_gb300._lib import lmoe_nvfp4_weight
    c = lm.Config(8, 256, 256, 8, 256, 2, weight_dtype="nvfp4").c()
    fake = 1 << 20   # never dereferenced
    ws = [lmoe_nvfp4_weight(fake, fake, fake, layout) for _ in range(5)]
    p = [ctypes.addressof(w) for w in ws]
    st = lib.latent_moe_forward(ctypes.byref(c), fake, fake, p[0], fake, p[1], p[2], p[3], fake, p[4], fake,
                                fake, 2, fake + 4096, fake, 16, None)
    assert st == status


@pytest.mark.parametrize("shape", [(128, 8192, 4096, 256, 4096, 8, "bf16"), (4096, 8192, 4096, 256, 4096, 8, "nvfp4"),
                                   (37, 512, 256, 8, 256, 2, "f32")])
def test_workspace_guard_bands_lie_between_sub_buffers(lm, shape):
    # every band is LMOE_GUARD_BYTES long, inside the workspace, and overlaps none of the
    # public sub-buffers (sized here from the shape)
    T, D, L, E, I, k, wd = shape
    c = lm.Config(T, D, L, E, I, k, act_dtype="f32" if wd == "f32" else "bf16", weight_dtype=wd)
    lay = lm.lmoe_get_workspace_layout(c)
    g = lm.lmoe_workspace_guards(c)
    g_io = lm.lmoe_workspace_guards(c, host_io=True)
    assert len(g) >= 25 and g_io[:len(g)] == g and len(g_io) == len(g) + 2
    assert all(b % 256 == 0 and b + lm.GUARD_BYTES <= lay["total"] for b in g)
    assert max(g_io) + lm.GUARD_BYTES <= lm.lmoe_workspace_size_host_io(c)
    R = T * k
    fp4 = wd == "nvfp4"
    sizes = {"xa": T * lay["xa_cols"] * 2, "logits": T * ((E + 31) // 32 * 32) * 4, "topk_idx": R * 4,
             "topk_w": R * 4, "counts": E * 4, "offsets": (E + 1) * 4, "row_of": R * 4, "tok_of": R * 4,
             "p": T * L * 4, "y": R * L * (2 if fp4 else 4), "u": T * D * 4,
             "xe": R * L // 2 if fp4 else R * L * 2, "h": R * I // 2 if fp4 else R * I * 2,
             "c": T * L // 2 if fp4 else T * L * 2}
    for name, n in sizes.items():
        o = lay[name]
        for b in g:
            assert b + lm.GUARD_BYTES <= o or b >= o + n, (name, o, n, b)


def test_no_process_wide_unique_symbols(lm):
    # A function-local static of a template with external linkage becomes a GNU unique symbol,
    # shared by every copy of the library in a process (the release and the bounds-checked
    # builds): one copy's "attribute already set" flag would then stand for the other's kernels.
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", lm.LIB_PATH], capture_output=True, text=True).stdout
    unique = [ln for ln in out.splitlines() if len(ln.split()) >= 3 and ln.split()[1] == "u"]
    assert unique == [], unique[:5]


def test_binding_structs_match_the_header(lm, tmp_path):
    # every struct the binding passes through the C ABI has the header's size and field offsets
    # (compiled with the host compiler against include/latent_moe.h)
    import shutil
    import subprocess
    from latent_mixture_experts_router_gb300 import _lib
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_inc = "/usr/local/cuda/include"
    if cc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime.h")):
        pytest.skip("no host compiler or CUDA headers")
    structs = {"lmoe_config": _lib.lmoe_config, "lmoe_nvfp4_weight": _lib.lmoe_nvfp4_weight,
               "lmoe_ex": _lib.lmoe_ex, "lmoe_workspace_layout": _lib.lmoe_workspace_layout}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "latent_moe.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'  printf("{name} size %zu\\n", sizeof({name}));')
        for f, _ in cls._fields_:
            lines.append(f'  printf("{name} {f} %zu\\n", offsetof({name}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "abi.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "abi"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o", str(exe)], check=True)
    got = {}
    for ln in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines():
        name, field, val = ln.split()
        got[(name, field)] = int(val)
    for name, cls in structs.items():
        assert got[(name, "size")] == ctypes.sizeof(cls), name
        for f, _ in cls._fields_:
            assert got[(name, f)] == getattr(cls, f).offset, (name, f)
