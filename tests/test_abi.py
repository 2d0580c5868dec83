"""The C-ABI library loads, exports every symbol include/moe.h declares, and its
host-side argument checks behave.  CPU only: no call here launches a kernel."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")

m = pytest.importorskip("mixture_experts_layer_88_b300")
L = m._lib


def declared_symbols():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", txt)))


def test_header_symbols_exported():
    syms = declared_symbols()
    assert len(syms) >= 13
    lib = ctypes.CDLL(L.LIB_PATH)
    for s in syms:
        assert hasattr(lib, s), s
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r" T (moe_\w+)", out))
    assert set(syms) <= exported
    assert set(L.SYMBOLS) == set(syms)


def test_version_and_status_strings():
    assert "sm_103a" in m.version()
    for code in range(7):
        assert L.lib().moe_status_string(code)


def _cfg(**kw):
    base = dict(T=64, d=256, E=16, K=4, S=1, I=128)
    base.update({k: v for k, v in kw.items() if k in base})
    c = m.make_cfg(**base)
    for k, v in kw.items():
        if k not in base:
            setattr(c, k, v)
    return c


@pytest.mark.parametrize("kw,code", [
    (dict(), 0),
    (dict(K=0), 1), (dict(K=17, E=16), 1), (dict(K=33, E=64), 1), (dict(E=1025), 1),
    (dict(S=65), 1), (dict(T=-1), 1), (dict(d=0), 1), (dict(I=0), 1),
    (dict(d=192), 1),                       # bf16 needs d % 128 == 0
    (dict(I=96), 1),                        # bf16 needs I % 128 == 0
    (dict(score_func=2), 1), (dict(normalize=2), 1),
    (dict(act_dtype=0, wgt_dtype=1), 2),    # mixed pair not built
    (dict(act_dtype=2, wgt_dtype=2), 2),    # e4m3 tokens: not a layer dtype
    (dict(act_dtype=1, wgt_dtype=2), 0),    # FP8 layer: bf16 tokens, e4m3 experts
    (dict(act_dtype=0, wgt_dtype=2), 2),    # fp32 tokens with e4m3 experts: not built
    (dict(act_dtype=1, wgt_dtype=2, d=8320), 1),   # FP8 layers: d, I <= 8192
    (dict(act_dtype=0, wgt_dtype=0, d=96, I=40), 0),   # fp32 takes any d, I
    (dict(T=0), 0),
    # node-limited routing
    (dict(n_groups=4, topk_groups=2), 0),   # 4 groups of 4 experts, K=4 <= 2*4
    (dict(n_groups=4, topk_groups=1), 0),   # K=4 <= 1*4
    (dict(n_groups=8, topk_groups=1), 1),   # K=4 > 1*2 experts
    (dict(n_groups=4, topk_groups=5), 1),   # more kept than groups
    (dict(n_groups=4, topk_groups=0), 1),
    (dict(n_groups=0, topk_groups=2), 1),
    (dict(n_groups=3, topk_groups=1, E=48, K=4), 0),   # groups of 16
    (dict(n_groups=4, topk_groups=1, E=48, K=4), 1),   # groups of 12: not a power of two
    (dict(n_groups=2, topk_groups=1, E=96, K=4), 1),   # groups of 48: not a multiple of 32
    (dict(n_groups=2, topk_groups=1, E=128, K=4), 0),  # groups of 64
    (dict(n_groups=5, topk_groups=2, E=16), 1),        # 16 experts do not split in 5
    (dict(n_groups=64, topk_groups=8, E=1024, K=8), 1),  # more than 32 groups
])
def test_check_cfg(kw, code):
    assert m.check_cfg(_cfg(**kw)) == code


def test_workspace_sizes():
    c = m.make_cfg(8192, 7168, 256, 8, 1, 2048)
    f = m.workspace_size(c, m.MOE_WS_FORWARD)
    # forward scratch holds xp [T*K, d], act [R, I], y [R, d] in bf16
    R = 8192 * 8 + 8192
    assert f >= 2 * (8192 * 8 * 7168 + R * 2048 + R * 7168)
    for w in (m.MOE_WS_ROUTE, m.MOE_WS_DISPATCH, m.MOE_WS_EXPERTS):
        assert 0 < m.workspace_size(c, w) < f
    assert m.workspace_size(_cfg(K=0), m.MOE_WS_FORWARD) == 0


def test_argument_errors_return_before_any_launch():
    c = _cfg()
    lib = L.lib()
    P = None
    # null pointers -> MOE_ERR_INVALID_ARG, synchronously, without touching CUDA
    assert lib.moe_route(ctypes.byref(c), P, P, P, P, P, P, 0, P) == 1
    assert lib.moe_combine(ctypes.byref(c), P, P, P, P, P, P) == 1
    assert lib.moe_update_bias(ctypes.byref(c), P, P, P, P) == 1
    # misaligned bf16 pointer
    assert lib.moe_route(ctypes.byref(c), 8, 16, 16, 16, 16, P, 0, P) == 1
    # workspace too small
    assert lib.moe_route(ctypes.byref(c), 16, 16, 16, 16, 16, 256, 4, P) == 3
    # empty batch is valid and launches nothing
    c0 = _cfg(T=0)
    assert lib.moe_route(ctypes.byref(c0), P, P, P, P, P, P, 0, P) == 0
    assert lib.moe_combine(ctypes.byref(c0), P, P, P, P, P, P) == 0
    assert lib.moe_experts(ctypes.byref(c0), P, P, P, P, P, P, P, P, P, P, 0, P) == 0


def test_prenorm_workspace_and_argument_errors():
    c = m.make_cfg(8192, 7168, 256, 8, 1, 2048)
    f = m.workspace_size(c, m.MOE_WS_FORWARD)
    # the pre-normed forward adds the normalised tokens [T, d] bf16 (the shared
    # experts' input), the weighted centroids [E, d] bf16 and inv_rms [T] fp32
    assert m.workspace_size(c, m.MOE_WS_FORWARD_PRENORM) == \
        f + 8192 * 7168 * 2 + 256 * 7168 * 2 + 8192 * 4
    lib = L.lib()
    P = None
    b = _cfg()
    # eps must be positive; pointers non-null and 16-byte aligned for bf16
    assert lib.moe_rmsnorm(ctypes.byref(b), 16, 16, 0.0, 16, P, P) == 1
    assert lib.moe_rmsnorm(ctypes.byref(b), 16, 16, -1e-6, 16, P, P) == 1
    assert lib.moe_rmsnorm(ctypes.byref(b), P, 16, 1e-6, 16, P, P) == 1
    assert lib.moe_rmsnorm(ctypes.byref(b), 16, 8, 1e-6, 16, P, P) == 1
    assert lib.moe_rmsnorm(ctypes.byref(_cfg(T=0)), P, P, 1e-6, P, P, P) == 0
    args = [16, 16, 1e-6, 16, 16, 16, 16, 16, 16, 256, 256, 256, 16]
    # workspace too small -> MOE_ERR_WORKSPACE before any launch
    assert lib.moe_forward_prenorm(ctypes.byref(b), *args, 256, 64, P) == 3
    # FP8 layers use the FP8 entry point
    f8 = _cfg(wgt_dtype=m.MOE_E4M3)
    assert lib.moe_forward_prenorm(ctypes.byref(f8), *args, 256, 1 << 40, P) == 2
    assert lib.moe_forward_fp8_prenorm(ctypes.byref(b), 16, 16, 1e-6, 16, 16, P, 256, 256,
                                       256, 16, 256, 1 << 40, P) == 1


def test_w8a16_workspace_and_argument_errors():
    c = m.make_cfg(16384, 7168, 256, 8, 1, 2048)
    c.wgt_dtype = m.MOE_E4M3
    # the W8A16 forward uses the bf16 layer's row layout
    v = m.bf16_layout(c)
    assert v.wgt_dtype == m.MOE_BF16 and c.wgt_dtype == m.MOE_E4M3
    assert m.workspace_size(c, m.MOE_WS_FORWARD_W8A16) == m.workspace_size(v, m.MOE_WS_FORWARD)
    assert m.workspace_size(v, m.MOE_WS_FORWARD_W8A16) == 0      # bf16 layers: not an FP8 path
    lib = L.lib()
    P = None
    b = _cfg()
    f8 = _cfg(wgt_dtype=m.MOE_E4M3)
    w = L.Fp8Weights(16, 16, 16, 16, 16, 16, 16, 16)
    # bf16 layers are rejected, missing weights and small workspaces too
    assert lib.moe_forward_w8a16(ctypes.byref(b), 16, 16, 256, ctypes.byref(w), 256, 256, 256,
                                 16, 256, 1 << 40, P) == 1
    assert lib.moe_forward_w8a16(ctypes.byref(f8), 16, 16, 256, None, 256, 256, 256, 16, 256,
                                 1 << 40, P) == 1
    assert lib.moe_forward_w8a16(ctypes.byref(f8), 16, 16, 256, ctypes.byref(w), 256, 256, 256,
                                 16, 256, 64, P) == 3
    assert lib.moe_experts_w8a16(ctypes.byref(f8), 16, 16, 256, ctypes.byref(w), 16, 16, 256, 64,
                                 P) == 3
    assert lib.moe_experts_w8a16(ctypes.byref(_cfg(T=0, wgt_dtype=m.MOE_E4M3)), P, P, P, None, P,
                                 P, P, 0, P) == 0


def test_training_workspace_and_argument_errors():
    c = m.make_cfg(8192, 7168, 256, 8, 1, 2048)
    # backward scratch holds the padded output-gradient rows dy, da, [dgate, dup], du
    rows = 8192 * 8 + 15 * 256 + 8192
    assert m.workspace_size(c, m.MOE_WS_BACKWARD) >= 2 * rows * (7168 + 2048 + 4096 + 7168)
    assert 0 < m.workspace_size(c, m.MOE_WS_FORWARD_TRAIN) < m.workspace_size(c, m.MOE_WS_FORWARD)
    # training is built for bf16 layers only
    f32 = _cfg(act_dtype=m.MOE_F32, wgt_dtype=m.MOE_F32)
    f8 = _cfg(wgt_dtype=m.MOE_E4M3)
    for w in (m.MOE_WS_FORWARD_TRAIN, m.MOE_WS_BACKWARD):
        assert m.workspace_size(f32, w) == 0 and m.workspace_size(f8, w) == 0
    lib = L.lib()
    P = None
    b = _cfg()
    st = L.TrainState(*([256] * 11))
    gr = L.Grads(256, 256, 256, 256, 256, 256)
    fargs = [16, 16, 256, 16, 16, 16, 16]
    assert lib.moe_forward_train(ctypes.byref(f32), *fargs, ctypes.byref(st), 16, 256, 1 << 40,
                                 P) == 2
    assert lib.moe_forward_train(ctypes.byref(b), *fargs, None, 16, 256, 1 << 40, P) == 1
    assert lib.moe_forward_train(ctypes.byref(b), *fargs, ctypes.byref(st), 16, 256, 64, P) == 3
    bargs = [16, 16, 16, 16, 16, 16, 16]
    assert lib.moe_backward(ctypes.byref(f8), *bargs, ctypes.byref(st), ctypes.byref(gr), 256,
                            1 << 40, P) == 2
    assert lib.moe_backward(ctypes.byref(b), *bargs, ctypes.byref(st), None, 256, 1 << 40,
                            P) == 1
    assert lib.moe_backward(ctypes.byref(b), 8, *bargs[1:], ctypes.byref(st), ctypes.byref(gr),
                            256, 1 << 40, P) == 1          # misaligned dout
    assert lib.moe_backward(ctypes.byref(b), *bargs, ctypes.byref(st), ctypes.byref(gr), 256, 64,
                            P) == 3


def test_selftest_limits_checked_before_any_launch():
    lib = L.lib()
    assert lib.moe_selftest_wait_timeout(0, None) == 1
    assert lib.moe_selftest_wait_timeout(2_000_000_000, None) == 1


def test_header_compiles_as_c99_and_links(tmp_path):
    """include/moe.h is plain C: a C99 program compiles against it, links
    libmoe.so and runs the checks that need no GPU."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = os.path.join(root, "tests", "c", "abi_smoke.c")
    exe = str(tmp_path / "abi_smoke")
    libdir = os.path.dirname(L.LIB_PATH)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-I",
                    os.path.join(root, "include"), src, "-L", libdir, "-lmoe",
                    f"-Wl,-rpath,{libdir}", "-o", exe], check=True)
    res = subprocess.run([exe], capture_output=True, text=True)
    assert res.returncode == 0, f"check {res.returncode} failed: {res.stdout}{res.stderr}"
    assert "abi ok" in res.stdout


def test_missing_library_fails_loudly():
    """No CPU fallback: without libmoe.so the loader raises instead of
    returning anything that could run the layer elsewhere."""
    from mixture_experts_layer_88_b300 import _lib
    with pytest.raises(ImportError, match="libmoe.so not built"):
        _lib.load_library(os.path.join(os.path.dirname(_lib.LIB_PATH), "no_such_dir",
                                       "libmoe.so"))
