"""Host-side checks of the C ABI that need no GPU: the library builds, loads,
exports every symbol include/moe.h declares, and rejects bad arguments
before it touches CUDA."""
import ctypes
import os
import re

import pytest

from expert_grouped_gemm_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)


def test_header_declares_and_library_exports_every_symbol(lib):
    decl = declared_symbols()
    assert set(decl) == set(_lib.EXPORTED), decl
    for name in decl:
        assert hasattr(lib, name), name


def _dims(**kw):
    base = dict(T=128, H=256, F=128, E=16, k=4, F_shared=0, dtype="bf16", frozen=False)
    base.update(kw)
    return _lib.make_dims(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(T=0), _lib.MOE_ERR_INVALID_ARG),
    (dict(k=17), _lib.MOE_ERR_INVALID_ARG),
    (dict(E=2048, k=2), _lib.MOE_ERR_UNSUPPORTED),
    (dict(H=100), _lib.MOE_ERR_UNSUPPORTED),
    (dict(F=96), _lib.MOE_ERR_UNSUPPORTED),
    (dict(E=24), _lib.MOE_ERR_UNSUPPORTED),
    (dict(F_shared=-1), _lib.MOE_ERR_INVALID_ARG),
    (dict(H=100, dtype="f32"), _lib.MOE_OK),
    (dict(E=24, k=3, dtype="f32"), _lib.MOE_OK),
])
def test_workspace_size_validation(lib, kw, code):
    d = _dims(**kw)
    n = ctypes.c_size_t(0)
    rc = lib.moe_workspace_size(ctypes.byref(d), ctypes.byref(n))
    assert rc == code, _lib.moe_last_error()
    if code == _lib.MOE_OK:
        assert n.value > 0 and n.value % 256 == 0


def test_workspace_grows_with_tokens(lib):
    a = _lib.moe_workspace_size(_dims(T=128))
    b = _lib.moe_workspace_size(_dims(T=4096))
    assert b > a


def test_workspace_entries_cover_the_size(lib):
    d = _dims(F_shared=64)
    ents = _lib.moe_workspace_entries(d)
    total = _lib.moe_workspace_size(d)
    end = max(o + s for o, s in ents.values())
    assert end == total
    offs = sorted(o for o, _ in ents.values())
    assert all(o % 256 == 0 for o in offs)
    assert {"ab", "h", "y_pair", "pad_off", "x_perm"} <= set(ents)


def _part_bytes(**kw):
    return _lib.moe_workspace_entries(_dims(**kw))["part"][1]


def test_workspace_holds_k_split_partials(lib):
    """The fp32 partial buffer of a K-split GEMM: room for 16 splits of the largest GEMM that
    can have too few tiles for the GPU (up to 256 SMs: at most 128 tiles), and none otherwise."""
    fp = 16 * 4  # splits x bytes per fp32
    # decode-sized: router logits, router dW and both expert forward GEMMs can be split;
    # the largest is the expert gate/up over T*k + 15 min(E, T*k) padded rows
    T, k, H, F, E = 1, 8, 2048, 768, 128
    rdec = T * k + 15 * min(E, T * k)
    assert _part_bytes(T=T, H=H, F=F, E=E, k=k) >= fp * max(rdec * 2 * F, rdec * H, T * E, H * E)
    # training-sized (T=4096): the expert GEMMs have plenty of tiles, the router GEMMs do not
    T = 4096
    assert _part_bytes(T=T, H=H, F=F, E=E, k=k) == (fp * max(T * E, H * E) + 255) // 256 * 256
    # so many router tiles (T=65536 -> 512 x 1) that no GEMM is ever split, except the router dW
    assert _part_bytes(T=65536, H=H, F=F, E=E, k=k) == (fp * H * E + 255) // 256 * 256


FAKE = ctypes.c_void_p(0x10000)   # host-side checks never dereference pointers


def _fwd_args(d, **over):
    args = dict(ws=FAKE, ws_bytes=_lib.moe_workspace_size(d), stream=None, x=FAKE, w_router=FAKE, bias=None,
                w_gate=FAKE, w_up=FAKE, w_down=FAKE, ws_gate=None, ws_up=None, ws_down=None, y=FAKE)
    args.update(over)
    return args


def _call_fwd(lib, d, a):
    return lib.moe_fwd(ctypes.byref(d), a["ws"], a["ws_bytes"], a["stream"], a["x"], a["w_router"], a["bias"],
                       a["w_gate"], a["w_up"], a["w_down"], a["ws_gate"], a["ws_up"], a["ws_down"], a["y"],
                       None, None, None, None, None)


@pytest.mark.parametrize("over,code", [
    (dict(x=None), _lib.MOE_ERR_INVALID_ARG),
    (dict(y=None), _lib.MOE_ERR_INVALID_ARG),
    (dict(w_gate=ctypes.c_void_p(0x10002)), _lib.MOE_ERR_INVALID_ARG),   # misaligned
    (dict(ws=None), _lib.MOE_ERR_WORKSPACE),
    (dict(ws=ctypes.c_void_p(0x10010)), _lib.MOE_ERR_WORKSPACE),          # not 256-aligned
    (dict(ws_bytes=1024), _lib.MOE_ERR_WORKSPACE),
    (dict(ws_gate=FAKE, ws_up=FAKE, ws_down=FAKE), _lib.MOE_ERR_INVALID_ARG),  # shared weights without F_shared
])
def test_fwd_rejects_bad_arguments_before_cuda(lib, over, code):
    d = _dims()
    rc = _call_fwd(lib, d, _fwd_args(d, **over))
    assert rc == code, _lib.moe_last_error()
    assert _lib.moe_last_error()


def test_bwd_and_select_before_fwd_are_state_errors(lib):
    d = _dims()
    ws = ctypes.c_void_p(0x7f0000000000)
    nbytes = _lib.moe_workspace_size(d)
    rc = lib.moe_bwd(ctypes.byref(d), ws, nbytes, None, FAKE, FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None)
    assert rc == _lib.MOE_ERR_STATE, _lib.moe_last_error()
    rc = lib.moe_select_retained(ctypes.byref(d), ws, nbytes, None, FAKE, None, None, None, None)
    assert rc == _lib.MOE_ERR_STATE, _lib.moe_last_error()


def test_frozen_bwd_rejects_gradient_pointers(lib):
    d = _dims(frozen=True)
    nbytes = _lib.moe_workspace_size(d)
    rc = lib.moe_bwd(ctypes.byref(d), FAKE, nbytes, None, FAKE, FAKE, 0, FAKE, FAKE, None, None, None, None, None,
                     None)
    assert rc == _lib.MOE_ERR_INVALID_ARG, _lib.moe_last_error()


def test_full_bwd_requires_gradient_pointers(lib):
    d = _dims()
    nbytes = _lib.moe_workspace_size(d)
    rc = lib.moe_bwd(ctypes.byref(d), FAKE, nbytes, None, FAKE, FAKE, 0, FAKE, None, FAKE, FAKE, FAKE, None, None,
                     None)
    assert rc == _lib.MOE_ERR_INVALID_ARG, _lib.moe_last_error()


def test_cta_pair_variant_compiles():
    """The CTA-pair (cta_group::2) variable-M grouped GEMM, kept as a build option beside
    the default single CTAs, still compiles for sm_103a."""
    import shutil
    import subprocess

    from expert_grouped_gemm_gb300 import build as b

    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = os.path.join(b.CSRC, "gemm_tc.cu")
    os.makedirs(b.BUILD, exist_ok=True)  # in-tree build folder (ignored by git)
    obj = os.path.join(b.BUILD, "gemm_tc_pair_check.o")
    r = subprocess.run([nvcc, *b.ARCH, *b.FLAGS, "-DMOE_VARM_CTAS=2", "-c", src, "-o", obj], capture_output=True,
                       text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    os.remove(obj)


def test_binding_refuses_host_tensors_no_cpu_fallback(lib):
    """Every step of the path runs in the library's kernels: the binding hands only device
    pointers across and refuses host tensors outright instead of computing on the CPU."""
    import torch

    d = _dims()
    T, H, F, E = 128, 256, 128, 16
    bf = torch.bfloat16
    cpu = dict(ws=torch.zeros(_lib.moe_workspace_size(d), dtype=torch.uint8), x=torch.zeros(T, H, dtype=bf),
               w_router=torch.zeros(H, E, dtype=bf), w_gate=torch.zeros(E, H, F, dtype=bf),
               w_up=torch.zeros(E, H, F, dtype=bf), w_down=torch.zeros(E, F, H, dtype=bf),
               y=torch.zeros(T, H, dtype=bf))
    with pytest.raises(ValueError, match="CUDA tensor"):
        _lib.moe_fwd(d, cpu["ws"], cpu["x"], cpu["w_router"], None, cpu["w_gate"], cpu["w_up"], cpu["w_down"],
                     None, None, None, cpu["y"])
    with pytest.raises(ValueError, match="required"):
        _lib._ptr(None, "x")
