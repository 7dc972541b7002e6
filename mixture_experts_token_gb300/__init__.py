"""Python binding of libmoe_gb300.so, the sm_103a MoE dispatch + expert
library declared in include/moe.h.

The functions here carry the C names and only marshal arguments: tensors
become device pointers, the current torch stream becomes the CUDA stream,
and a non-OK status raises MoeError.  All arithmetic runs in the CUDA
kernels of the library; there is no other code path.  If the library has
not been built (``mixture_experts_token_gb300.build.build()``), every call
raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import c_float, c_int, c_int32, c_int64, c_size_t, c_void_p

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, \
    MOE_ERR_CUDA = range(5)
MOE_DEV_NONFINITE, MOE_DEV_TIMEOUT, MOE_DEV_BAD_INDEX = 1, 2, 4
MOE_DEV_UNALIGNED = 8
MOE_WGRAD_ACCUMULATE, MOE_WGRAD_ROWS16 = 1, 2
MOE_F32, MOE_BF16 = 0, 1
MOE_MODE_FALLBACK_LAYER, MOE_MODE_CAPPED, MOE_MODE_DROPLESS = 0, 1, 2
MOE_WS_PERMUTE, MOE_WS_CHUNKED, MOE_WS_LAYER = 0, 1, 2
MOE_WS_GMM_BACKWARD, MOE_WS_LAYER_BACKWARD = 3, 4


class MoeConfig(ctypes.Structure):
    """moe_config_t."""
    _fields_ = [("T", c_int32), ("H", c_int32), ("E", c_int32),
                ("k", c_int32), ("F", c_int32), ("S", c_int32),
                ("ragged_buffer_factor", c_float), ("n_chunks", c_int32),
                ("dtype", c_int), ("renorm", c_int32),
                ("redundant_slots", c_int32)]

    def with_(self, **kw) -> "MoeConfig":
        c = MoeConfig()
        ctypes.pointer(c)[0] = self
        for key, v in kw.items():
            setattr(c, key, v)
        return c

    def __repr__(self):
        return ("MoeConfig(" + ", ".join(f"{n}={getattr(self, n)}"
                                         for n, _ in self._fields_) + ")")


class MoeLayerInfo(ctypes.Structure):
    """moe_layer_info_t."""
    _fields_ = [("overflow", c_int32), ("n_chunks", c_int32),
                ("capacity", c_int64)]


class MoeRowSegment(ctypes.Structure):
    """moe_row_segment_t."""
    _fields_ = [("group_offsets", c_void_p), ("first_row", c_int32)]


class MoeError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {moe_status_string(status)} ({status})")


_lib = None


def lib():
    """The loaded library (loads it on first use)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "mixture_experts_token_gb300.build.build()")
        handle = ctypes.CDLL(LIB_PATH)
        _declare(handle)
        _lib = handle
    return _lib


def _declare(h):
    P = c_void_p
    cfg = ctypes.POINTER(MoeConfig)
    sig = {
        "moe_router_logits": [cfg, P, P, P, P, P, P],
        "moe_ep_check": [cfg, P, P, P, P, P],
        "moe_ep_dispatch_pack": [cfg, P, P, P, P, P, P, P, P, P],
        "moe_ep_return_map": [cfg, P, P, P, P],
        "moe_ep_localize": [cfg, P, P, c_int32, c_int32, P, P, P],
        "moe_ep_sum_partials": [cfg, c_int32, P, P, P],
        "moe_ep_delocalize": [cfg, P, c_int32, c_int32, P, c_int32, P, P,
                              P],
        "moe_route": [cfg, P, P, P, P, P],
        "moe_check_overflow": [cfg, P, P, P, P, P, P, P, P],
        "moe_permute": [cfg, P, P, c_int32, P, P, P, P, P, P, P, P, P,
                        c_size_t, P],
        "moe_permute_noalloc": [cfg, P, P, c_int32, P, P, P, P, P, P, P, P,
                                P],
        "moe_permute_tables": [cfg, P, c_int32, P, P, P, P, P, P, P, P,
                               c_size_t, P],
        "moe_permute_scatter": [cfg, P, P, P, P, P, P, P, c_size_t, P],
        "moe_gmm_swiglu": [cfg, P, P, P, P, P, P, P, P, P],
        "moe_plan_duplication": [cfg, P, P, P, P, P, P, P],
        "moe_permute_planned": [cfg, P, P, c_int32, P, P, P, P, P, P, P, P,
                                P, P, P, c_size_t, P],
        "moe_gmm_swiglu_mapped": [cfg, c_int32, P, P, P, P, P, P, P, P, P,
                                  P],
        "moe_gmm_gate_up": [cfg, c_int32, P, P, P, P, P, P, P, P],
        "moe_gmm_down": [cfg, c_int32, P, P, P, P, P, P, P],
        "moe_combine": [cfg, P, P, P, P, P],
        "moe_layer_dropless_chunked": [cfg, P, P, P, P, P, P, P, P, c_size_t,
                                       P],
        "moe_layer": [cfg, P, P, P, P, P, P, c_int,
                      ctypes.POINTER(MoeLayerInfo), P, P, c_size_t, P],
        "moe_combine_backward": [cfg, P, P, P, P, P, P, P],
        "moe_route_backward": [cfg, P, P, P, P, P],
        "moe_permute_backward": [cfg, P, P, P, P],
        "moe_gmm_swiglu_saved": [cfg, P, P, P, P, P, P, P, P, P, P, P],
        "moe_gmm_swiglu_backward": [cfg, P, P, P, P, P, P, P, P, P, P, P, P,
                                    P, c_int32, P, P, c_size_t, P],
        "moe_gmm_gate_up_saved": [cfg, c_int32, P, P, P, P, P, P, P, P, P,
                                  P],
        "moe_gmm_down_dgrad": [cfg, c_int32, P, P, P, P, P, P, P, P, P, P],
        "moe_gmm_gate_up_dgrad": [cfg, c_int32, P, P, P, P, P, P, P, P, P],
        "moe_gmm_gate_up_wgrad": [cfg, c_int32, P,
                                  ctypes.POINTER(MoeRowSegment), c_int32,
                                  c_int64, P, P, P, P, P, c_int32, P, P],
        "moe_gmm_down_wgrad": [cfg, c_int32, P,
                               ctypes.POINTER(MoeRowSegment), c_int32,
                               c_int64, P, P, P, c_int32, P, P],
        "moe_regroup_rows": [cfg, c_int32, ctypes.POINTER(MoeRowSegment),
                             c_int32, c_int64, P, P, P, P, P, P, P, P, P, P,
                             P, P, P],
        "moe_combine_backward_rows": [cfg, P, P, P, P, P, P],
        "moe_gmm_down_dgrad_rows": [cfg, c_int32, P, P, P, P, P, P, P, P, P,
                                    P, P, P, P],
        "moe_combine_weight_grad": [cfg, P, P, P, P],
        "moe_layer_backward": [cfg, P, P, P, P, P, P, P, P, P, P, P, c_int,
                               ctypes.POINTER(MoeLayerInfo), P, P, c_size_t,
                               P],
    }
    for name, args in sig.items():
        fn = getattr(h, name)
        fn.argtypes = args
        fn.restype = c_int
    h.moe_layer_graph_create.argtypes = [cfg, P, P, P, P, P, P, P, P,
                                         c_size_t, ctypes.POINTER(P)]
    h.moe_layer_graph_create.restype = c_int
    h.moe_layer_graph_create_traced.argtypes = [cfg, P, P, P, P, P, P, P,
                                                P, c_size_t, P,
                                                ctypes.POINTER(P)]
    h.moe_layer_graph_create_traced.restype = c_int
    h.moe_layer_graph_trace_slots.argtypes = [cfg]
    h.moe_layer_graph_trace_slots.restype = c_int32
    h.moe_layer_graph_launch.argtypes = [P, P]
    h.moe_layer_graph_launch.restype = c_int
    h.moe_layer_graph_overflow_flag.argtypes = [P]
    h.moe_layer_graph_overflow_flag.restype = P
    h.moe_layer_graph_fallback_chunks.argtypes = [P]
    h.moe_layer_graph_fallback_chunks.restype = c_int32
    h.moe_layer_graph_destroy.argtypes = [P]
    h.moe_layer_graph_destroy.restype = None
    h.moe_workspace_bytes.argtypes = [cfg, c_int]
    h.moe_workspace_bytes.restype = c_size_t
    h.moe_validate_config.argtypes = [cfg]
    h.moe_validate_config.restype = c_int
    h.moe_row_dot_parts.argtypes = [cfg]
    h.moe_row_dot_parts.restype = c_int32
    h.moe_capacity_rows.argtypes = [cfg]
    h.moe_capacity_rows.restype = c_int64
    h.moe_chunk_tokens.argtypes = [cfg]
    h.moe_chunk_tokens.restype = c_int32
    h.moe_num_chunks.argtypes = [cfg]
    h.moe_num_chunks.restype = c_int32
    h.moe_gmm_kernel_choice.argtypes = [cfg, c_int32, c_int64]
    h.moe_gmm_kernel_choice.restype = c_int32
    h.moe_test_stall_gemm_producer.argtypes = [c_int64]
    h.moe_test_stall_gemm_producer.restype = None
    h.moe_status_string.argtypes = [c_int]
    h.moe_status_string.restype = ctypes.c_char_p


# ------------------------------------------------------------ marshalling --
def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return c_void_p(t)
    return c_void_p(t.data_ptr())


def _nbytes(t):
    if t is None:
        return 0
    return t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        import torch
        if torch.cuda.is_available():
            return c_void_p(torch.cuda.current_stream().cuda_stream)
        return None
    if isinstance(stream, int):
        return c_void_p(stream)
    return c_void_p(stream.cuda_stream)


def _check(status, where):
    if status != MOE_OK:
        raise MoeError(status, where)


def make_config(T, H, E, k, F, S, factor=2.0, n_chunks=0, dtype="bf16",
                renorm=False, redundant_slots=0) -> MoeConfig:
    return MoeConfig(T, H, E, k, F, S, float(factor), n_chunks,
                     MOE_F32 if dtype in ("f32", "float32") else MOE_BF16,
                     1 if renorm else 0, redundant_slots)


# --------------------------------------------------------- entry points ---
def moe_status_string(status) -> str:
    return lib().moe_status_string(status).decode()


def moe_validate_config(cfg) -> int:
    return lib().moe_validate_config(ctypes.byref(cfg))


def moe_capacity_rows(cfg) -> int:
    return lib().moe_capacity_rows(ctypes.byref(cfg))


def moe_chunk_tokens(cfg) -> int:
    return lib().moe_chunk_tokens(ctypes.byref(cfg))


def moe_num_chunks(cfg) -> int:
    return lib().moe_num_chunks(ctypes.byref(cfg))


def moe_gmm_kernel_choice(cfg, n_groups=0, rows_bound=0) -> int:
    """Bit 1 (value 2): GEMM2 on the CTA-pair kernel; 0: the one-CTA
    kernels (GEMM1 always; bit 0 is never set)."""
    return int(lib().moe_gmm_kernel_choice(ctypes.byref(cfg), n_groups,
                                           rows_bound))


def moe_layer_graph_trace_slots(cfg) -> int:
    return int(lib().moe_layer_graph_trace_slots(ctypes.byref(cfg)))


def moe_test_stall_gemm_producer(fills: int):
    """Tests of failure detection only (see include/moe.h)."""
    lib().moe_test_stall_gemm_producer(fills)


def moe_workspace_bytes(cfg, which) -> int:
    return lib().moe_workspace_bytes(ctypes.byref(cfg), which)


def moe_router_logits(cfg, x, w_router, logit_offset, logits,
                      status_word=None, stream=None):
    _check(lib().moe_router_logits(
        ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(logit_offset),
        _ptr(logits), _ptr(status_word), _stream(stream)),
        "moe_router_logits")


def moe_ep_check(cfg, shard_counts, overflow_flag, required_factor,
                 capacity, stream=None):
    _check(lib().moe_ep_check(ctypes.byref(cfg), _ptr(shard_counts),
                              _ptr(overflow_flag), _ptr(required_factor),
                              _ptr(capacity), _stream(stream)),
           "moe_ep_check")


def moe_ep_dispatch_pack(cfg, x, topk_idx, topk_w, uniq_offsets, uniq_tokens,
                         x_send, send_idx, send_w, stream=None):
    _check(lib().moe_ep_dispatch_pack(
        ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(topk_w),
        _ptr(uniq_offsets), _ptr(uniq_tokens), _ptr(x_send), _ptr(send_idx),
        _ptr(send_w), _stream(stream)), "moe_ep_dispatch_pack")


def moe_ep_return_map(cfg, uniq_offsets, uniq_tokens, row_of_ret,
                      stream=None):
    _check(lib().moe_ep_return_map(ctypes.byref(cfg), _ptr(uniq_offsets),
                                   _ptr(uniq_tokens), _ptr(row_of_ret),
                                   _stream(stream)), "moe_ep_return_map")


def moe_ep_localize(cfg, topk_idx, topk_w, first_expert, n_local, local_idx,
                    local_w, stream=None):
    _check(lib().moe_ep_localize(ctypes.byref(cfg), _ptr(topk_idx),
                                 _ptr(topk_w), first_expert, n_local,
                                 _ptr(local_idx), _ptr(local_w),
                                 _stream(stream)), "moe_ep_localize")


def moe_ep_delocalize(cfg, topk_idx, first_expert, n_local, local_v, v,
                      row_of=None, row_stride=1, stream=None):
    _check(lib().moe_ep_delocalize(ctypes.byref(cfg), _ptr(topk_idx),
                                   first_expert, n_local, _ptr(row_of),
                                   row_stride, _ptr(local_v), _ptr(v),
                                   _stream(stream)), "moe_ep_delocalize")


def moe_ep_sum_partials(cfg, n_parts, parts, y, stream=None):
    _check(lib().moe_ep_sum_partials(ctypes.byref(cfg), n_parts, _ptr(parts),
                                     _ptr(y), _stream(stream)),
           "moe_ep_sum_partials")


def moe_route(cfg, logits, topk_idx, topk_w, status_word=None, stream=None):
    _check(lib().moe_route(ctypes.byref(cfg), _ptr(logits), _ptr(topk_idx),
                           _ptr(topk_w), _ptr(status_word), _stream(stream)),
           "moe_route")


def moe_check_overflow(cfg, topk_idx, expert_counts, expert_offsets,
                       shard_counts, overflow_flag, required_factor, capacity,
                       stream=None):
    _check(lib().moe_check_overflow(
        ctypes.byref(cfg), _ptr(topk_idx), _ptr(expert_counts),
        _ptr(expert_offsets), _ptr(shard_counts), _ptr(overflow_flag),
        _ptr(required_factor), _ptr(capacity), _stream(stream)),
        "moe_check_overflow")


def moe_permute(cfg, x, topk_idx, capped, x_sorted, row_of, sorted_token,
                group_offsets, uniq_offsets, uniq_tokens, expand_idx,
                n_dropped, workspace, stream=None):
    _check(lib().moe_permute(
        ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), 1 if capped else 0,
        _ptr(x_sorted), _ptr(row_of), _ptr(sorted_token),
        _ptr(group_offsets), _ptr(uniq_offsets), _ptr(uniq_tokens),
        _ptr(expand_idx), _ptr(n_dropped), _ptr(workspace),
        _nbytes(workspace), _stream(stream)), "moe_permute")


def moe_permute_tables(cfg, topk_idx, capped, row_of, sorted_token,
                       group_offsets, uniq_offsets, n_dropped, workspace,
                       divert=None, slot_of=None, stream=None):
    """The counting-sort half of moe_permute (moe_permute_planned with
    divert and slot_of); moe_permute_scatter completes it."""
    _check(lib().moe_permute_tables(
        ctypes.byref(cfg), _ptr(topk_idx), 1 if capped else 0, _ptr(divert),
        _ptr(slot_of), _ptr(row_of), _ptr(sorted_token), _ptr(group_offsets),
        _ptr(uniq_offsets), _ptr(n_dropped), _ptr(workspace),
        _nbytes(workspace), _stream(stream)), "moe_permute_tables")


def moe_permute_scatter(cfg, x, row_of, uniq_offsets, x_sorted, uniq_tokens,
                        expand_idx, workspace, stream=None):
    """The row copy of moe_permute, from the tables moe_permute_tables left
    in row_of, uniq_offsets and the workspace."""
    _check(lib().moe_permute_scatter(
        ctypes.byref(cfg), _ptr(x), _ptr(row_of), _ptr(uniq_offsets),
        _ptr(x_sorted), _ptr(uniq_tokens), _ptr(expand_idx), _ptr(workspace),
        _nbytes(workspace), _stream(stream)), "moe_permute_scatter")


def moe_permute_noalloc(cfg, x, topk_idx, capped, x_sorted, row_of,
                        sorted_token, group_offsets, uniq_offsets,
                        uniq_tokens, expand_idx, n_dropped, stream=None):
    """moe_permute with the scratch in the library's fixed device array, for
    callers that cannot allocate device memory (see include/moe.h)."""
    _check(lib().moe_permute_noalloc(
        ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), 1 if capped else 0,
        _ptr(x_sorted), _ptr(row_of), _ptr(sorted_token),
        _ptr(group_offsets), _ptr(uniq_offsets), _ptr(uniq_tokens),
        _ptr(expand_idx), _ptr(n_dropped), _stream(stream)),
        "moe_permute_noalloc")


def moe_gmm_swiglu(cfg, x_sorted, group_offsets, w_gate, w_up, w_down, h,
                   y_sorted, status_word=None, stream=None):
    _check(lib().moe_gmm_swiglu(
        ctypes.byref(cfg), _ptr(x_sorted), _ptr(group_offsets),
        _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(h), _ptr(y_sorted),
        _ptr(status_word), _stream(stream)), "moe_gmm_swiglu")


def moe_gmm_gate_up(cfg, x_sorted, group_offsets, w_gate, w_up, h,
                    status_word=None, stream=None, n_groups=0,
                    group_expert=None):
    _check(lib().moe_gmm_gate_up(
        ctypes.byref(cfg), n_groups, _ptr(group_expert), _ptr(x_sorted),
        _ptr(group_offsets), _ptr(w_gate), _ptr(w_up), _ptr(h),
        _ptr(status_word), _stream(stream)), "moe_gmm_gate_up")


def moe_gmm_down(cfg, h, group_offsets, w_down, y_sorted, status_word=None,
                 stream=None, n_groups=0, group_expert=None):
    _check(lib().moe_gmm_down(
        ctypes.byref(cfg), n_groups, _ptr(group_expert), _ptr(h),
        _ptr(group_offsets), _ptr(w_down), _ptr(y_sorted), _ptr(status_word),
        _stream(stream)), "moe_gmm_down")


def moe_plan_duplication(cfg, expert_counts, divert, slot_of, group_expert,
                         shard_counts_after, overflow_flag_after,
                         stream=None):
    _check(lib().moe_plan_duplication(
        ctypes.byref(cfg), _ptr(expert_counts), _ptr(divert), _ptr(slot_of),
        _ptr(group_expert), _ptr(shard_counts_after),
        _ptr(overflow_flag_after), _stream(stream)), "moe_plan_duplication")


def moe_permute_planned(cfg, x, topk_idx, capped, divert, slot_of, x_sorted,
                        row_of, sorted_token, group_offsets, uniq_offsets,
                        uniq_tokens, expand_idx, n_dropped, workspace,
                        stream=None):
    _check(lib().moe_permute_planned(
        ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), 1 if capped else 0,
        _ptr(divert), _ptr(slot_of), _ptr(x_sorted), _ptr(row_of),
        _ptr(sorted_token), _ptr(group_offsets), _ptr(uniq_offsets),
        _ptr(uniq_tokens), _ptr(expand_idx), _ptr(n_dropped),
        _ptr(workspace), _nbytes(workspace), _stream(stream)),
        "moe_permute_planned")


def moe_gmm_swiglu_mapped(cfg, n_groups, group_expert, x_sorted,
                          group_offsets, w_gate, w_up, w_down, h, y_sorted,
                          status_word=None, stream=None):
    _check(lib().moe_gmm_swiglu_mapped(
        ctypes.byref(cfg), n_groups, _ptr(group_expert), _ptr(x_sorted),
        _ptr(group_offsets), _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(h),
        _ptr(y_sorted), _ptr(status_word), _stream(stream)),
        "moe_gmm_swiglu_mapped")


def moe_combine(cfg, y_sorted, row_of, topk_w, y, stream=None):
    _check(lib().moe_combine(ctypes.byref(cfg), _ptr(y_sorted), _ptr(row_of),
                             _ptr(topk_w), _ptr(y), _stream(stream)),
           "moe_combine")


def moe_layer_dropless_chunked(cfg, x, logits, w_gate, w_up, w_down, y,
                               workspace, status_word=None, stream=None):
    _check(lib().moe_layer_dropless_chunked(
        ctypes.byref(cfg), _ptr(x), _ptr(logits), _ptr(w_gate), _ptr(w_up),
        _ptr(w_down), _ptr(y), _ptr(status_word), _ptr(workspace),
        _nbytes(workspace), _stream(stream)), "moe_layer_dropless_chunked")


def moe_layer(cfg, x, logits, w_gate, w_up, w_down, y, mode, workspace,
              status_word=None, stream=None) -> dict:
    info = MoeLayerInfo()
    _check(lib().moe_layer(
        ctypes.byref(cfg), _ptr(x), _ptr(logits), _ptr(w_gate), _ptr(w_up),
        _ptr(w_down), _ptr(y), mode, ctypes.byref(info), _ptr(status_word),
        _ptr(workspace), _nbytes(workspace), _stream(stream)), "moe_layer")
    return {"overflow": info.overflow, "n_chunks": info.n_chunks,
            "capacity": info.capacity}


# --------------------------------------------------------- backward ------
def moe_combine_backward(cfg, dy, y_sorted, row_of, topk_w, dy_sorted,
                         dtopk_w, stream=None):
    _check(lib().moe_combine_backward(
        ctypes.byref(cfg), _ptr(dy), _ptr(y_sorted), _ptr(row_of),
        _ptr(topk_w), _ptr(dy_sorted), _ptr(dtopk_w), _stream(stream)),
        "moe_combine_backward")


def moe_route_backward(cfg, logits, topk_idx, dtopk_w, dlogits, stream=None):
    _check(lib().moe_route_backward(
        ctypes.byref(cfg), _ptr(logits), _ptr(topk_idx), _ptr(dtopk_w),
        _ptr(dlogits), _stream(stream)), "moe_route_backward")


def moe_permute_backward(cfg, dx_sorted, row_of, dx, stream=None):
    _check(lib().moe_permute_backward(
        ctypes.byref(cfg), _ptr(dx_sorted), _ptr(row_of), _ptr(dx),
        _stream(stream)), "moe_permute_backward")


def moe_gmm_swiglu_saved(cfg, x_sorted, group_offsets, w_gate, w_up, w_down,
                         g, u, h, y_sorted, status_word=None, stream=None):
    _check(lib().moe_gmm_swiglu_saved(
        ctypes.byref(cfg), _ptr(x_sorted), _ptr(group_offsets), _ptr(w_gate),
        _ptr(w_up), _ptr(w_down), _ptr(g), _ptr(u), _ptr(h), _ptr(y_sorted),
        _ptr(status_word), _stream(stream)), "moe_gmm_swiglu_saved")


def moe_gmm_swiglu_backward(cfg, x_sorted, group_offsets, w_gate, w_up,
                            w_down, g, u, h, dy_sorted, dx_sorted, dw_gate,
                            dw_up, dw_down, accumulate, workspace,
                            status_word=None, stream=None):
    _check(lib().moe_gmm_swiglu_backward(
        ctypes.byref(cfg), _ptr(x_sorted), _ptr(group_offsets), _ptr(w_gate),
        _ptr(w_up), _ptr(w_down), _ptr(g), _ptr(u), _ptr(h), _ptr(dy_sorted),
        _ptr(dx_sorted), _ptr(dw_gate), _ptr(dw_up), _ptr(dw_down),
        int(accumulate), _ptr(status_word), _ptr(workspace),
        _nbytes(workspace), _stream(stream)), "moe_gmm_swiglu_backward")


def moe_gmm_gate_up_saved(cfg, x_sorted, group_offsets, w_gate, w_up, g, u,
                          h, status_word=None, stream=None, n_groups=0,
                          group_expert=None):
    _check(lib().moe_gmm_gate_up_saved(
        ctypes.byref(cfg), n_groups, _ptr(group_expert), _ptr(x_sorted), _ptr(group_offsets), _ptr(w_gate),
        _ptr(w_up), _ptr(g), _ptr(u), _ptr(h), _ptr(status_word),
        _stream(stream)), "moe_gmm_gate_up_saved")


def moe_gmm_down_dgrad(cfg, group_offsets, w_down, g, u, dy_sorted, dg, du,
                       status_word=None, stream=None, n_groups=0,
                       group_expert=None):
    _check(lib().moe_gmm_down_dgrad(
        ctypes.byref(cfg), n_groups, _ptr(group_expert), _ptr(group_offsets), _ptr(w_down), _ptr(g),
        _ptr(u), _ptr(dy_sorted), _ptr(dg), _ptr(du), _ptr(status_word),
        _stream(stream)), "moe_gmm_down_dgrad")


def moe_gmm_gate_up_dgrad(cfg, group_offsets, w_gate, w_up, dg, du,
                          dx_sorted, status_word=None, stream=None,
                          n_groups=0, group_expert=None):
    _check(lib().moe_gmm_gate_up_dgrad(
        ctypes.byref(cfg), n_groups, _ptr(group_expert), _ptr(group_offsets), _ptr(w_gate), _ptr(w_up),
        _ptr(dg), _ptr(du), _ptr(dx_sorted), _ptr(status_word),
        _stream(stream)), "moe_gmm_gate_up_dgrad")


def _segments(segments):
    """(group_offsets tensor, first_row) pairs -> moe_row_segment_t[]."""
    arr = (MoeRowSegment * max(len(segments), 1))()
    for i, (off, first) in enumerate(segments):
        arr[i].group_offsets = off if isinstance(off, int) else off.data_ptr()
        arr[i].first_row = int(first)
    return arr


def moe_gmm_gate_up_wgrad(cfg, segments, rows_total, x_sorted, dg, du,
                          dw_gate, dw_up, accumulate, status_word=None,
                          stream=None, n_groups=0, group_expert=None):
    _check(lib().moe_gmm_gate_up_wgrad(
        ctypes.byref(cfg), n_groups, _ptr(group_expert), _segments(segments), len(segments),
        int(rows_total), _ptr(x_sorted), _ptr(dg), _ptr(du), _ptr(dw_gate),
        _ptr(dw_up), int(accumulate), _ptr(status_word), _stream(stream)),
        "moe_gmm_gate_up_wgrad")


def moe_gmm_down_wgrad(cfg, segments, rows_total, h, dy_sorted, dw_down,
                       accumulate, status_word=None, stream=None, n_groups=0,
                       group_expert=None):
    _check(lib().moe_gmm_down_wgrad(
        ctypes.byref(cfg), n_groups, _ptr(group_expert), _segments(segments), len(segments),
        int(rows_total), _ptr(h), _ptr(dy_sorted), _ptr(dw_down),
        int(accumulate), _ptr(status_word), _stream(stream)),
        "moe_gmm_down_wgrad")


def moe_regroup_rows(cfg, segments, rows_out, x_sorted, dg, du, h,
                     dy_sorted, x_out, dg_out, du_out, h_out, dy_out,
                     out_offsets, stream=None, n_groups=0, w_row=None):
    _check(lib().moe_regroup_rows(
        ctypes.byref(cfg), n_groups, _segments(segments), len(segments), int(rows_out),
        _ptr(x_sorted), _ptr(dg), _ptr(du), _ptr(h), _ptr(dy_sorted),
        _ptr(x_out), _ptr(dg_out), _ptr(du_out), _ptr(h_out), _ptr(dy_out),
        _ptr(out_offsets), _ptr(w_row), _stream(stream)), "moe_regroup_rows")


def moe_row_dot_parts(cfg) -> int:
    return int(lib().moe_row_dot_parts(ctypes.byref(cfg)))


def moe_combine_backward_rows(cfg, dy, row_of, topk_w, dy_rows, w_row,
                              stream=None):
    _check(lib().moe_combine_backward_rows(
        ctypes.byref(cfg), _ptr(dy), _ptr(row_of), _ptr(topk_w),
        _ptr(dy_rows), _ptr(w_row), _stream(stream)),
        "moe_combine_backward_rows")


def moe_gmm_down_dgrad_rows(cfg, group_offsets, w_down, g, u, h, dy_rows,
                            w_row, dg, du, row_dot, status_word=None,
                            stream=None, n_groups=0, group_expert=None):
    _check(lib().moe_gmm_down_dgrad_rows(
        ctypes.byref(cfg), n_groups, _ptr(group_expert), _ptr(group_offsets),
        _ptr(w_down), _ptr(g), _ptr(u), _ptr(h), _ptr(dy_rows), _ptr(w_row),
        _ptr(dg), _ptr(du), _ptr(row_dot), _ptr(status_word),
        _stream(stream)), "moe_gmm_down_dgrad_rows")


def moe_combine_weight_grad(cfg, row_of, row_dot, dtopk_w, stream=None):
    _check(lib().moe_combine_weight_grad(
        ctypes.byref(cfg), _ptr(row_of), _ptr(row_dot), _ptr(dtopk_w),
        _stream(stream)), "moe_combine_weight_grad")


def moe_layer_backward(cfg, x, logits, w_gate, w_up, w_down, dy, dx,
                       dlogits, dw_gate, dw_up, dw_down, mode, workspace,
                       status_word=None, stream=None) -> dict:
    info = MoeLayerInfo()
    _check(lib().moe_layer_backward(
        ctypes.byref(cfg), _ptr(x), _ptr(logits), _ptr(w_gate), _ptr(w_up),
        _ptr(w_down), _ptr(dy), _ptr(dx), _ptr(dlogits), _ptr(dw_gate),
        _ptr(dw_up), _ptr(dw_down), mode, ctypes.byref(info),
        _ptr(status_word), _ptr(workspace), _nbytes(workspace),
        _stream(stream)), "moe_layer_backward")
    return {"overflow": info.overflow, "n_chunks": info.n_chunks,
            "capacity": info.capacity}


class MoeLayerGraph:
    """moe_layer_graph_t: the fallback=layer layer as one CUDA graph, bound
    to the tensors given here (they must outlive the graph)."""

    def __init__(self, cfg, x, logits, w_gate, w_up, w_down, y, workspace,
                 status_word=None, trace=None):
        self._h = c_void_p()
        self._keep = (x, logits, w_gate, w_up, w_down, y, workspace,
                      status_word, trace)
        if trace is None:
            _check(lib().moe_layer_graph_create(
                ctypes.byref(cfg), _ptr(x), _ptr(logits), _ptr(w_gate),
                _ptr(w_up), _ptr(w_down), _ptr(y), _ptr(status_word),
                _ptr(workspace), _nbytes(workspace), ctypes.byref(self._h)),
                "moe_layer_graph_create")
        else:
            _check(lib().moe_layer_graph_create_traced(
                ctypes.byref(cfg), _ptr(x), _ptr(logits), _ptr(w_gate),
                _ptr(w_up), _ptr(w_down), _ptr(y), _ptr(status_word),
                _ptr(workspace), _nbytes(workspace), _ptr(trace),
                ctypes.byref(self._h)), "moe_layer_graph_create_traced")

    def launch(self, stream=None):
        _check(lib().moe_layer_graph_launch(self._h, _stream(stream)),
               "moe_layer_graph_launch")

    def overflow_flag_ptr(self) -> int:
        return lib().moe_layer_graph_overflow_flag(self._h)

    def fallback_chunks(self) -> int:
        return lib().moe_layer_graph_fallback_chunks(self._h)

    def close(self):
        if self._h:
            lib().moe_layer_graph_destroy(self._h)
            self._h = c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------- buffer allocation ------
def alloc_step_buffers(cfg, device="cuda"):
    """Device buffers for calling the entry points one by one (torch owns
    the memory; sizes follow include/moe.h)."""
    import torch
    T, H, E, k, F, S = cfg.T, cfg.H, cfg.E, cfg.k, cfg.F, cfg.S
    dt = torch.float32 if cfg.dtype == MOE_F32 else torch.bfloat16
    i32 = dict(dtype=torch.int32, device=device)
    R = T * k
    return {
        "topk_idx": torch.empty((T, k), **i32),
        "topk_w": torch.empty((T, k), dtype=torch.float32, device=device),
        "status": torch.zeros(1, **i32),
        "expert_counts": torch.empty(E, **i32),
        "expert_offsets": torch.empty(E + 1, **i32),
        "shard_counts": torch.empty(S, **i32),
        "overflow_flag": torch.empty(1, **i32),
        "required_factor": torch.empty(1, dtype=torch.float32, device=device),
        "capacity": torch.empty(1, **i32),
        "x_sorted": torch.empty((R, H), dtype=dt, device=device),
        "row_of": torch.empty((T, k), **i32),
        "sorted_token": torch.empty(max(R, 1), **i32),
        "group_offsets": torch.empty(E + S * cfg.redundant_slots + 1, **i32),
        "divert": torch.empty(E, **i32),
        "slot_of": torch.empty(E, **i32),
        "group_expert": torch.empty(E + S * cfg.redundant_slots, **i32),
        "shard_after": torch.empty(S, **i32),
        "flag_after": torch.empty(1, **i32),
        "uniq_offsets": torch.empty(S + 1, **i32),
        "uniq_tokens": torch.empty(max(T * min(k, S), 1), **i32),
        "expand_idx": torch.empty(max(R, 1), **i32),
        "n_dropped": torch.empty(1, **i32),
        "permute_ws": torch.empty(
            max(moe_workspace_bytes(cfg, MOE_WS_PERMUTE), 256),
            dtype=torch.uint8, device=device),
        "h": torch.empty((R, max(F, 1)), dtype=dt, device=device),
        "y_sorted": torch.empty((R, H), dtype=dt, device=device),
        "y": torch.empty((T, H), dtype=dt, device=device),
    }


def layer_workspace(cfg, which=MOE_WS_LAYER, device="cuda"):
    import torch
    n = moe_workspace_bytes(cfg, which)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)
