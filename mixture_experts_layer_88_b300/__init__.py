"""DeepSeekMoE layer forward and backward for NVIDIA B300 (sm_103a).

The compute runs in libmoe.so (hand-written CUDA behind a C ABI, declared in
include/moe.h); this package only marshals torch tensors into it.
"""
from . import _lib
from ._lib import (MoeCfg, MoeError, make_cfg, cfg_from_layer, workspace_size, check_cfg,
                   alloc_workspace, route, dispatch, experts, combine, update_bias, forward,
                   Fp8Weights, fp8_weights, fp8_rows, dispatch_fp8, experts_fp8, forward_fp8,
                   rmsnorm, forward_prenorm, forward_fp8_prenorm, bf16_layout, experts_w8a16,
                   forward_w8a16, selftest_wait_timeout, MOE_E4M3, MOE_WS_FORWARD_W8A16,
                   get_status, trace_enable, trace_read_all, version, MOE_F32, MOE_BF16,
                   MOE_SCORE_SIGMOID, MOE_SCORE_SOFTMAX, MOE_WS_ROUTE, MOE_WS_DISPATCH,
                   MOE_WS_EXPERTS, MOE_WS_FORWARD, MOE_WS_FORWARD_PRENORM,
                   MOE_WS_FORWARD_TRAIN, MOE_WS_BACKWARD, TrainState, Grads, alloc_train_state,
                   alloc_grads, forward_train, backward)
from .layer import MoeLayer, HostPipeline

__all__ = ["MoeCfg", "MoeError", "MoeLayer", "HostPipeline", "make_cfg", "cfg_from_layer", "workspace_size",
           "check_cfg", "alloc_workspace", "route", "dispatch", "experts", "combine",
           "update_bias", "forward", "Fp8Weights", "fp8_weights", "fp8_rows", "dispatch_fp8",
           "experts_fp8", "forward_fp8", "rmsnorm", "forward_prenorm", "forward_fp8_prenorm",
           "bf16_layout", "experts_w8a16", "forward_w8a16", "selftest_wait_timeout",
           "get_status", "trace_enable", "trace_read_all", "alloc_train_state", "alloc_grads",
           "forward_train", "backward",
           "version"]
