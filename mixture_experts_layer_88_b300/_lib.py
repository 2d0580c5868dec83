"""ctypes binding of libmoe.so: argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; this module turns
torch tensors into device pointers and the current torch stream into a
cudaStream_t.  If the library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_F32, MOE_BF16, MOE_E4M3 = 0, 1, 2
MOE_SCORE_SIGMOID, MOE_SCORE_SOFTMAX = 0, 1
MOE_WS_ROUTE, MOE_WS_DISPATCH, MOE_WS_EXPERTS, MOE_WS_FORWARD = 0, 1, 2, 3
MOE_WS_FORWARD_PRENORM = 4
MOE_WS_FORWARD_W8A16 = 5
MOE_WS_FORWARD_TRAIN = 6
MOE_WS_BACKWARD = 7

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_TIMEOUT",
          6: "MOE_ERR_DEVICE_BOUNDS"}

# every symbol include/moe.h declares
SYMBOLS = ["moe_workspace_size", "moe_check_cfg", "moe_route", "moe_dispatch", "moe_experts",
           "moe_experts_static",
           "moe_combine", "moe_update_bias", "moe_forward", "moe_fp8_rows", "moe_dispatch_fp8",
           "moe_experts_fp8", "moe_forward_fp8", "moe_rmsnorm", "moe_forward_prenorm",
           "moe_forward_fp8_prenorm", "moe_experts_w8a16", "moe_forward_w8a16",
           "moe_forward_train", "moe_backward",
           "moe_selftest_wait_timeout", "moe_get_status",
           "moe_status_string", "moe_trace_enable", "moe_trace_read", "moe_version"]


class MoeError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


class MoeCfg(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("K", ctypes.c_int32), ("S", ctypes.c_int32), ("I", ctypes.c_int32),
                ("act_dtype", ctypes.c_int32), ("wgt_dtype", ctypes.c_int32),
                ("score_func", ctypes.c_int32), ("normalize", ctypes.c_int32),
                ("add_residual", ctypes.c_int32), ("gamma", ctypes.c_float),
                ("n_groups", ctypes.c_int32), ("topk_groups", ctypes.c_int32)]


class Fp8Weights(ctypes.Structure):
    """moe_fp8_weights_t: e4m3 expert weights and their 128 x 128 block scales."""
    _fields_ = [("w13", ctypes.c_void_p), ("w13_scale", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("w2_scale", ctypes.c_void_p),
                ("ws13", ctypes.c_void_p), ("ws13_scale", ctypes.c_void_p),
                ("ws2", ctypes.c_void_p), ("ws2_scale", ctypes.c_void_p)]


class TrainState(ctypes.Structure):
    """moe_train_state_t: what moe_forward_train keeps for moe_backward."""
    _fields_ = [("idx", ctypes.c_void_p), ("gates", ctypes.c_void_p),
                ("scores", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("perm_tok", ctypes.c_void_p),
                ("pos", ctypes.c_void_p), ("xp", ctypes.c_void_p), ("h", ctypes.c_void_p),
                ("act", ctypes.c_void_p), ("y", ctypes.c_void_p)]


class Grads(ctypes.Structure):
    """moe_grads_t: gradient outputs of moe_backward."""
    _fields_ = [("dx", ctypes.c_void_p), ("dcentroids", ctypes.c_void_p),
                ("dw13", ctypes.c_void_p), ("dw2", ctypes.c_void_p),
                ("dws13", ctypes.c_void_p), ("dws2", ctypes.c_void_p)]


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int32),
                ("total_ms", ctypes.c_float)]


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libmoe.so not built at {path}; run "
                          "`python -m mixture_experts_layer_88_b300.build`")
    lib = ctypes.CDLL(path)
    P, I32, SZ, F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    cfgp = ctypes.POINTER(MoeCfg)
    sig = {
        "moe_workspace_size": (SZ, [cfgp, I32]),
        "moe_check_cfg": (I32, [cfgp]),
        "moe_route": (I32, [cfgp, P, P, P, P, P, P, SZ, P]),
        "moe_dispatch": (I32, [cfgp, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_experts": (I32, [cfgp, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_experts_static": (I32, [cfgp, P, P, P, P, P, P, P, P, P, P]),
        "moe_combine": (I32, [cfgp, P, P, P, P, P, P]),
        "moe_update_bias": (I32, [cfgp, P, P, P, P]),
        "moe_forward": (I32, [cfgp, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_fp8_rows": (I32, [cfgp, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64),
                               ctypes.POINTER(ctypes.c_int64)]),
        "moe_dispatch_fp8": (I32, [cfgp, P, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_experts_fp8": (I32, [cfgp, P, P, P, P, ctypes.POINTER(Fp8Weights), P, P, P, P, SZ,
                                  P]),
        "moe_forward_fp8": (I32, [cfgp, P, P, P, ctypes.POINTER(Fp8Weights), P, P, P, P, P, SZ,
                                  P]),
        "moe_rmsnorm": (I32, [cfgp, P, P, F32, P, P, P]),
        "moe_forward_prenorm": (I32, [cfgp, P, P, F32, P, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_forward_fp8_prenorm": (I32, [cfgp, P, P, F32, P, P, ctypes.POINTER(Fp8Weights), P,
                                          P, P, P, P, SZ, P]),
        "moe_experts_w8a16": (I32, [cfgp, P, P, P, ctypes.POINTER(Fp8Weights), P, P, P, SZ, P]),
        "moe_forward_w8a16": (I32, [cfgp, P, P, P, ctypes.POINTER(Fp8Weights), P, P, P, P, P,
                                    SZ, P]),
        "moe_forward_train": (I32, [cfgp, P, P, P, P, P, P, P, ctypes.POINTER(TrainState), P, P,
                                    SZ, P]),
        "moe_backward": (I32, [cfgp, P, P, P, P, P, P, P, ctypes.POINTER(TrainState),
                               ctypes.POINTER(Grads), P, SZ, P]),
        "moe_selftest_wait_timeout": (I32, [ctypes.c_uint64, P]),
        "moe_get_status": (I32, [P]),
        "moe_status_string": (ctypes.c_char_p, [I32]),
        "moe_trace_enable": (I32, [I32]),
        "moe_trace_read": (I32, [ctypes.POINTER(KernelTime), I32, ctypes.POINTER(I32)]),
        "moe_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_LIB = load_library()   # fails loudly at import when the library is missing


def lib() -> ctypes.CDLL:
    return _LIB


# ----------------------------------------------------------------------------

_DT = {torch.float32: MOE_F32, torch.bfloat16: MOE_BF16}


def make_cfg(T, d, E, K, S, I, dtype=MOE_BF16, score_func=MOE_SCORE_SIGMOID, normalize=1,
             add_residual=1, gamma=1e-3, n_groups=0, topk_groups=0) -> MoeCfg:
    return MoeCfg(T, d, E, K, S, I, dtype, dtype, score_func, normalize, add_residual, gamma,
                  n_groups, topk_groups)


def cfg_from_layer(layer_cfg, T=None) -> MoeCfg:
    """MoeCfg from a moe_inputs.LayerCfg-like object (shape fields only)."""
    dt = {"f32": MOE_F32, "bf16": MOE_BF16, "e4m3": MOE_E4M3}
    c = layer_cfg
    return MoeCfg(c.T if T is None else T, c.d, c.E, c.K, c.S, c.I, dt[c.act], dt[c.wgt],
                  c.score_func, c.normalize, c.add_residual, c.gamma,
                  getattr(c, "n_groups", 0), getattr(c, "topk_groups", 0))


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(code, where):
    if code != 0:
        raise MoeError(code, where)


def workspace_size(cfg: MoeCfg, which: int) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(cfg), which))


def check_cfg(cfg: MoeCfg) -> int:
    return int(lib().moe_check_cfg(ctypes.byref(cfg)))


def alloc_workspace(cfg: MoeCfg, which: int, device="cuda") -> torch.Tensor:
    n = max(256, workspace_size(cfg, which))
    return torch.empty(n, dtype=torch.uint8, device=device)


def route(cfg, x, centroids, bias, idx, gates, ws, stream=None):
    _check(lib().moe_route(ctypes.byref(cfg), _p(x), _p(centroids), _p(bias), _p(idx),
                           _p(gates), _p(ws), ws.numel(), _stream(stream)), "moe_route")


def dispatch(cfg, x, idx, counts, offsets, xp, perm_tok, pos, ws, stream=None):
    _check(lib().moe_dispatch(ctypes.byref(cfg), _p(x), _p(idx), _p(counts), _p(offsets),
                              _p(xp), _p(perm_tok), _p(pos), _p(ws), ws.numel(),
                              _stream(stream)), "moe_dispatch")


def experts(cfg, xp, x, offsets, w13, w2, ws13, ws2, act, y, ws, stream=None):
    _check(lib().moe_experts(ctypes.byref(cfg), _p(xp), _p(x), _p(offsets), _p(w13), _p(w2),
                             _p(ws13), _p(ws2), _p(act), _p(y), _p(ws), ws.numel(),
                             _stream(stream)), "moe_experts")


def experts_static(cfg, xp, x, offsets, w13, w2, ws13, ws2, act, y, stream=None):
    """moe_experts with the library's fixed internal scratch (no workspace)."""
    _check(lib().moe_experts_static(ctypes.byref(cfg), _p(xp), _p(x), _p(offsets), _p(w13),
                                    _p(w2), _p(ws13), _p(ws2), _p(act), _p(y),
                                    _stream(stream)), "moe_experts_static")


def combine(cfg, y, gates, pos, x, out, stream=None):
    _check(lib().moe_combine(ctypes.byref(cfg), _p(y), _p(gates), _p(pos), _p(x), _p(out),
                             _stream(stream)), "moe_combine")


def update_bias(cfg, counts, bias, load_stats=None, stream=None):
    _check(lib().moe_update_bias(ctypes.byref(cfg), _p(counts), _p(bias), _p(load_stats),
                                 _stream(stream)), "moe_update_bias")


def forward(cfg, x, centroids, bias, w13, w2, ws13, ws2, idx, gates, counts, out, ws,
            stream=None):
    _check(lib().moe_forward(ctypes.byref(cfg), _p(x), _p(centroids), _p(bias), _p(w13),
                             _p(w2), _p(ws13), _p(ws2), _p(idx), _p(gates), _p(counts),
                             _p(out), _p(ws), ws.numel(), _stream(stream)), "moe_forward")


def fp8_weights(w: dict) -> Fp8Weights:
    """Fp8Weights from a dict with w13, w13_scale, w2, w2_scale and (when the
    layer has shared experts) ws13, ws13_scale, ws2, ws2_scale tensors."""
    def g(k):
        t = w.get(k)
        return None if t is None or t.numel() == 0 else t.data_ptr()
    return Fp8Weights(g("w13"), g("w13_scale"), g("w2"), g("w2_scale"), g("ws13"),
                      g("ws13_scale"), g("ws2"), g("ws2_scale"))


def fp8_rows(cfg) -> tuple:
    """(rows_in, rows_out, shared_row) of the FP8 row layout."""
    a, b, c = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib().moe_fp8_rows(ctypes.byref(cfg), ctypes.byref(a), ctypes.byref(b),
                              ctypes.byref(c)), "moe_fp8_rows")
    return a.value, b.value, c.value


def dispatch_fp8(cfg, x, idx, counts, offsets, xq, xq_scale, perm_tok, pos, ws, stream=None):
    _check(lib().moe_dispatch_fp8(ctypes.byref(cfg), _p(x), _p(idx), _p(counts), _p(offsets),
                                  _p(xq), _p(xq_scale), _p(perm_tok), _p(pos), _p(ws),
                                  ws.numel(), _stream(stream)), "moe_dispatch_fp8")


def experts_fp8(cfg, xq, xq_scale, offsets, counts, weights: Fp8Weights, act, act_scale, y, ws,
                stream=None):
    _check(lib().moe_experts_fp8(ctypes.byref(cfg), _p(xq), _p(xq_scale), _p(offsets),
                                 _p(counts), ctypes.byref(weights), _p(act), _p(act_scale),
                                 _p(y), _p(ws), ws.numel(), _stream(stream)), "moe_experts_fp8")


def forward_fp8(cfg, x, centroids, bias, weights: Fp8Weights, idx, gates, counts, out, ws,
                stream=None):
    _check(lib().moe_forward_fp8(ctypes.byref(cfg), _p(x), _p(centroids), _p(bias),
                                 ctypes.byref(weights), _p(idx), _p(gates), _p(counts), _p(out),
                                 _p(ws), ws.numel(), _stream(stream)), "moe_forward_fp8")


def rmsnorm(cfg, x, norm_w, eps, xn, inv_rms=None, stream=None):
    _check(lib().moe_rmsnorm(ctypes.byref(cfg), _p(x), _p(norm_w), float(eps), _p(xn),
                             _p(inv_rms), _stream(stream)), "moe_rmsnorm")


def forward_prenorm(cfg, x, norm_w, eps, centroids, bias, w13, w2, ws13, ws2, idx, gates, counts,
                    out, ws, stream=None):
    _check(lib().moe_forward_prenorm(ctypes.byref(cfg), _p(x), _p(norm_w), float(eps),
                                     _p(centroids), _p(bias), _p(w13), _p(w2), _p(ws13),
                                     _p(ws2), _p(idx), _p(gates), _p(counts), _p(out), _p(ws),
                                     ws.numel(), _stream(stream)), "moe_forward_prenorm")


def forward_fp8_prenorm(cfg, x, norm_w, eps, centroids, bias, weights: Fp8Weights, idx, gates,
                        counts, out, ws, stream=None):
    _check(lib().moe_forward_fp8_prenorm(ctypes.byref(cfg), _p(x), _p(norm_w), float(eps),
                                         _p(centroids), _p(bias), ctypes.byref(weights), _p(idx),
                                         _p(gates), _p(counts), _p(out), _p(ws), ws.numel(),
                                         _stream(stream)), "moe_forward_fp8_prenorm")


def bf16_layout(cfg: MoeCfg) -> MoeCfg:
    """The cfg of an FP8 layer's W8A16 path for moe_dispatch / moe_combine
    (the bf16 layer's row layout)."""
    v = MoeCfg()
    ctypes.pointer(v)[0] = cfg
    v.wgt_dtype = MOE_BF16
    return v


def experts_w8a16(cfg, xp, x, offsets, weights: Fp8Weights, act, y, ws, stream=None):
    _check(lib().moe_experts_w8a16(ctypes.byref(cfg), _p(xp), _p(x), _p(offsets),
                                   ctypes.byref(weights), _p(act), _p(y), _p(ws), ws.numel(),
                                   _stream(stream)), "moe_experts_w8a16")


def forward_w8a16(cfg, x, centroids, bias, weights: Fp8Weights, idx, gates, counts, out, ws,
                  stream=None):
    _check(lib().moe_forward_w8a16(ctypes.byref(cfg), _p(x), _p(centroids), _p(bias),
                                   ctypes.byref(weights), _p(idx), _p(gates), _p(counts),
                                   _p(out), _p(ws), ws.numel(), _stream(stream)),
           "moe_forward_w8a16")


TRAIN_KEYS = ("idx", "gates", "scores", "counts", "offsets", "perm_tok", "pos", "xp", "h", "act",
              "y")
GRAD_KEYS = ("dx", "dcentroids", "dw13", "dw2", "dws13", "dws2")


def alloc_train_state(cfg: MoeCfg, device="cuda") -> dict:
    """Device buffers of moe_train_state_t for cfg (bf16 layer)."""
    T, K, E, S, d, I = cfg.T, cfg.K, cfg.E, cfg.S, cfg.d, cfg.I
    R = T * K + S * T
    i32, f32, bf = torch.int32, torch.float32, torch.bfloat16
    return {"idx": torch.empty((T, K), dtype=i32, device=device),
            "gates": torch.empty((T, K), dtype=f32, device=device),
            "scores": torch.empty((T, E), dtype=f32, device=device),
            "counts": torch.empty((E,), dtype=i32, device=device),
            "offsets": torch.empty((E + 1,), dtype=i32, device=device),
            "perm_tok": torch.empty((T * K,), dtype=i32, device=device),
            "pos": torch.empty((T, K), dtype=i32, device=device),
            "xp": torch.empty((T * K, d), dtype=bf, device=device),
            "h": torch.empty((R, 2 * I), dtype=bf, device=device),
            "act": torch.empty((R, I), dtype=bf, device=device),
            "y": torch.empty((R, d), dtype=bf, device=device)}


def alloc_grads(cfg: MoeCfg, device="cuda") -> dict:
    """Gradient buffers of moe_grads_t for cfg (bf16 layer)."""
    T, E, S, d, I = cfg.T, cfg.E, cfg.S, cfg.d, cfg.I
    bf = torch.bfloat16
    return {"dx": torch.empty((T, d), dtype=bf, device=device),
            "dcentroids": torch.empty((E, d), dtype=torch.float32, device=device),
            "dw13": torch.empty((E, 2 * I, d), dtype=bf, device=device),
            "dw2": torch.empty((E, d, I), dtype=bf, device=device),
            "dws13": torch.empty((S, 2 * I, d), dtype=bf, device=device),
            "dws2": torch.empty((S, d, I), dtype=bf, device=device)}


def _struct(cls, keys, bufs):
    def g(k):
        t = bufs.get(k)
        return None if t is None or t.numel() == 0 else t.data_ptr()
    return cls(*[g(k) for k in keys])


def forward_train(cfg, x, centroids, bias, w13, w2, ws13, ws2, state: dict, out, ws,
                  stream=None):
    st = _struct(TrainState, TRAIN_KEYS, state)
    _check(lib().moe_forward_train(ctypes.byref(cfg), _p(x), _p(centroids), _p(bias), _p(w13),
                                   _p(w2), _p(ws13), _p(ws2), ctypes.byref(st), _p(out), _p(ws),
                                   ws.numel(), _stream(stream)), "moe_forward_train")


def backward(cfg, dout, x, centroids, w13, w2, ws13, ws2, state: dict, grads: dict, ws,
             stream=None):
    st = _struct(TrainState, TRAIN_KEYS, state)
    gr = _struct(Grads, GRAD_KEYS, grads)
    _check(lib().moe_backward(ctypes.byref(cfg), _p(dout), _p(x), _p(centroids), _p(w13),
                              _p(w2), _p(ws13), _p(ws2), ctypes.byref(st), ctypes.byref(gr),
                              _p(ws), ws.numel(), _stream(stream)), "moe_backward")


def selftest_wait_timeout(limit_ns: int, stream=None):
    """Runs out one bounded device wait after limit_ns; see include/moe.h."""
    _check(lib().moe_selftest_wait_timeout(int(limit_ns), _stream(stream)),
           "moe_selftest_wait_timeout")


def get_status(stream=None) -> int:
    return int(lib().moe_get_status(_stream(stream)))


def trace_enable(on: bool):
    lib().moe_trace_enable(1 if on else 0)


def trace_read_all(max_kernels: int = 64) -> list:
    """[(name, launches, total_ms)] of every traced kernel since the last read."""
    arr = (KernelTime * max_kernels)()
    n = ctypes.c_int32(0)
    _check(lib().moe_trace_read(arr, max_kernels, ctypes.byref(n)), "moe_trace_read")
    return [(arr[i].name.decode(), int(arr[i].launches), float(arr[i].total_ms))
            for i in range(min(n.value, max_kernels))]


def version() -> str:
    return lib().moe_version().decode()
