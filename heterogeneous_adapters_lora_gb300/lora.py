"""Thin Python binding of liblora_gb300 (``include/lora_gb300.h``).

Argument marshalling only: every function forwards to the C entry point of
the same name; all computation runs in the library's CUDA kernels.  Device
memory and streams come from PyTorch.  Importing this module does not load
the library; the first call does, and raises ``RuntimeError`` if it is
missing (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblora_gb300.so")

MAX_SLICES = 8
TILE_ROWS = 16
MOE_W13 = 0
MOE_W2 = 1

STATUS = {
    0: "LORA_OK", 1: "LORA_ERR_INVALID_ARG", 2: "LORA_ERR_INDEX", 3: "LORA_ERR_RANK",
    4: "LORA_ERR_SHAPE", 5: "LORA_ERR_LAYOUT", 6: "LORA_ERR_NOMEM", 7: "LORA_ERR_CUDA",
    8: "LORA_ERR_DEVICE_INDEX", 9: "LORA_ERR_TIMEOUT", 10: "LORA_ERR_CAPACITY",
    11: "LORA_ERR_UNSUPPORTED",
}
CODE = {v: k for k, v in STATUS.items()}

c_i32 = ctypes.c_int32
c_i64 = ctypes.c_int64
c_vp = ctypes.c_void_p
c_size = ctypes.c_size_t


class PoolDesc(ctypes.Structure):
    _fields_ = [("max_loras", c_i32), ("max_rank", c_i32), ("in_dim", c_i32), ("n_slices", c_i32),
                ("out_dims", c_i32 * MAX_SLICES), ("is_lm_head", c_i32), ("num_experts", c_i32),
                ("d_model", c_i32), ("d_mlp", c_i32), ("n_w13_slices", c_i32),
                ("w13_slice_width", c_i32), ("shared_outer", c_i32)]


class Meta(ctypes.Structure):
    _fields_ = [("max_rows", c_i32), ("max_keys", c_i32), ("max_tiles", c_i32), ("max_ltiles", c_i32),
                ("T", c_i32), ("top_k", c_i32), ("n_keys", c_i32), ("mode", c_i32),
                ("sorted", c_vp), ("key_count", c_vp), ("key_offset", c_vp), ("group_key", c_vp),
                ("group_start", c_vp), ("key_group", c_vp), ("tile_group", c_vp),
                ("tile_row0", c_vp), ("tile_keyn", c_vp), ("ltile_row0", c_vp), ("ltile_keyn", c_vp),
                ("ltile_tok0", c_vp), ("stile_row0", c_vp), ("stile_keyn", c_vp), ("counters", c_vp)]


class LoraError(RuntimeError):
    def __init__(self, code, where, cuda_error=None):
        self.code = int(code)
        self.name = STATUS.get(self.code, f"status {code}")
        self.cuda_error = cuda_error
        extra = f" (cudaError {cuda_error})" if cuda_error else ""
        super().__init__(f"{where}: {self.name}{extra}")


_lock = threading.Lock()
_lib = None

EXPORTS = {
    "lora_pool_create": (c_i32, [ctypes.POINTER(PoolDesc), c_vp, ctypes.POINTER(c_vp)]),
    "lora_pool_destroy": (c_i32, [c_vp]),
    "lora_pool_get_desc": (c_i32, [c_vp, ctypes.POINTER(PoolDesc)]),
    "lora_set": (c_i32, [c_vp, c_i32, c_i32, ctypes.c_float, ctypes.POINTER(c_vp), ctypes.POINTER(c_vp),
                         c_i32, c_vp]),
    "lora_set_packed": (c_i32, [c_vp, c_i32, c_i32, ctypes.c_float, c_vp, c_vp, c_vp]),
    "lora_set_moe": (c_i32, [c_vp, c_i32, c_i32, ctypes.c_float, ctypes.POINTER(c_vp),
                             ctypes.POINTER(c_i32), ctypes.POINTER(c_vp), ctypes.POINTER(c_i32), c_i32,
                             c_vp]),
    "lora_reset": (c_i32, [c_vp, c_i32, c_vp]),
    "lora_meta_bytes": (c_size, [c_i32, c_i32]),
    "lora_meta_bind": (c_i32, [ctypes.POINTER(Meta), c_vp, c_size, c_i32, c_i32]),
    "lora_build_meta": (c_i32, [c_vp, c_vp, c_i32, c_vp, c_i32, ctypes.POINTER(Meta), c_vp]),
    "lora_shrink": (c_i32, [c_vp, ctypes.POINTER(Meta), c_vp, c_i64, c_vp, c_vp]),
    "lora_expand": (c_i32, [c_vp, ctypes.POINTER(Meta), c_vp, c_vp, c_i64, c_vp]),
    "lora_workspace_bytes": (c_size, [c_vp, c_i32, c_i32]),
    "lora_workspace_init": (c_i32, [c_vp, c_size, c_vp]),
    "lora_apply_slices": (c_i32, [c_vp, ctypes.POINTER(Meta), c_vp, c_i64, c_vp, c_i64, c_vp, c_size,
                                  c_vp]),
    "lora_apply_slices_static": (c_i32, [c_vp, ctypes.POINTER(Meta), c_vp, c_i64, c_vp, c_i64, c_vp]),
    "lora_static_scratch_bytes": (c_size, []),
    "lora_logits_apply": (c_i32, [c_vp, ctypes.POINTER(Meta), c_vp, c_i64, c_vp, c_i64, c_i32, c_vp, c_vp, c_i64,
                                  c_i32, ctypes.c_float, c_vp, c_size, c_vp]),
    "lora_moe_apply": (c_i32, [c_vp, ctypes.POINTER(Meta), c_i32, c_vp, c_i64, c_vp, c_vp, c_i64, c_vp,
                               c_size, c_vp]),
    "lora_moe_align_padded": (c_i32, [c_vp, ctypes.POINTER(Meta), c_i32, c_i32, c_vp, c_vp, c_vp, c_vp]),
    "lora_moe_apply_blocks": (c_i32, [c_vp, ctypes.POINTER(Meta), c_i32, c_vp, c_i64, c_vp, c_vp, c_i64, c_vp, c_vp,
                                      c_vp, c_i32, c_i32, c_vp]),
    "lora_get_device_status": (c_i32, [c_vp, c_vp]),
    "lora_set_spin_limit": (None, [c_i32]),
    "lora_set_kernel_policy": (None, [c_i32]),
    "lora_kernel_launch_count": (ctypes.c_ulonglong, []),
    "lora_build_meta_apply": (c_i32, [c_vp, c_vp, c_i32, ctypes.POINTER(Meta), c_vp, c_i64, c_vp, c_i64, c_vp, c_size,
                                      c_vp]),
    "lora_last_cuda_error": (c_i32, []),
    "lora_linear_apply": (c_i32, [c_vp, ctypes.POINTER(Meta), c_vp, c_i64, c_vp, c_i64, c_vp, c_vp, c_i64, c_vp, c_size,
                              c_vp]),
    "lora_sink_experts_act": (c_i32, [c_vp, c_i64, c_vp, c_i64, c_i32, c_i32, c_i32, c_vp, c_i64, c_vp]),
    "lora_status_string": (ctypes.c_char_p, [c_i32]),
}


def lib():
    """Load liblora_gb300.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"liblora_gb300.so not found at {LIB_PATH}: run build() first; "
                                   "there is no CPU fallback")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in EXPORTS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _check(code, where):
    if code != 0:
        cuda = int(lib().lora_last_cuda_error()) if code == CODE["LORA_ERR_CUDA"] else None
        raise LoraError(code, where, cuda)


def ptr(obj):
    """Raw address of a torch tensor, numpy array, int or None."""
    if obj is None:
        return None
    if isinstance(obj, int):
        return obj
    if hasattr(obj, "data_ptr"):
        return obj.data_ptr()
    if hasattr(obj, "ctypes"):
        return obj.ctypes.data
    raise TypeError(type(obj))


def stream_ptr(stream=None):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr_array(objs):
    arr = (c_vp * len(objs))(*[ptr(o) for o in objs])
    return arr


# ------------------------------------------------------------------ same-name wrappers


def lora_pool_create(desc: PoolDesc, stream=None):
    h = c_vp()
    _check(lib().lora_pool_create(ctypes.byref(desc), stream_ptr(stream), ctypes.byref(h)),
           "lora_pool_create")
    return h.value


def lora_pool_destroy(pool):
    _check(lib().lora_pool_destroy(pool), "lora_pool_destroy")


def lora_pool_get_desc(pool) -> PoolDesc:
    d = PoolDesc()
    _check(lib().lora_pool_get_desc(pool, ctypes.byref(d)), "lora_pool_get_desc")
    return d


def lora_set(pool, slot, rank, scale, A, B, stream=None):
    _check(lib().lora_set(pool, slot, rank, float(scale), _ptr_array(A), _ptr_array(B), len(A),
                          stream_ptr(stream)), "lora_set")


def lora_set_packed(pool, slot, rank, scale, A, B, stream=None):
    _check(lib().lora_set_packed(pool, slot, rank, float(scale), ptr(A), ptr(B), stream_ptr(stream)),
           "lora_set_packed")


def lora_set_moe(pool, slot, rank, scale, A, a_experts, B, b_experts, stream=None):
    ae = (c_i32 * len(a_experts))(*a_experts)
    be = (c_i32 * len(b_experts))(*b_experts)
    _check(lib().lora_set_moe(pool, slot, rank, float(scale), _ptr_array(A), ae, _ptr_array(B), be,
                              len(A), stream_ptr(stream)), "lora_set_moe")


def lora_reset(pool, slot, stream=None):
    _check(lib().lora_reset(pool, slot, stream_ptr(stream)), "lora_reset")


def lora_meta_bytes(max_rows, max_keys) -> int:
    return int(lib().lora_meta_bytes(max_rows, max_keys))


def lora_meta_bind(meta: Meta, d_buf, nbytes, max_rows, max_keys):
    _check(lib().lora_meta_bind(ctypes.byref(meta), ptr(d_buf), nbytes, max_rows, max_keys),
           "lora_meta_bind")


def lora_build_meta(pool, d_idx, T, d_topk_ids, top_k, meta: Meta, stream=None):
    _check(lib().lora_build_meta(pool, ptr(d_idx), T, ptr(d_topk_ids), top_k, ctypes.byref(meta),
                                 stream_ptr(stream)), "lora_build_meta")


def lora_build_meta_apply(pool, d_idx, T, meta: Meta, x, ldx, y, ldy, ws, ws_bytes, stream=None):
    _check(lib().lora_build_meta_apply(pool, ptr(d_idx), T, ctypes.byref(meta), ptr(x), ldx, ptr(y), ldy, ptr(ws),
                                       ws_bytes, stream_ptr(stream)), "lora_build_meta_apply")


def lora_shrink(pool, meta: Meta, x, ldx, v, stream=None):
    _check(lib().lora_shrink(pool, ctypes.byref(meta), ptr(x), ldx, ptr(v), stream_ptr(stream)),
           "lora_shrink")


def lora_expand(pool, meta: Meta, v, y, ldy, stream=None):
    _check(lib().lora_expand(pool, ctypes.byref(meta), ptr(v), ptr(y), ldy, stream_ptr(stream)),
           "lora_expand")


def lora_workspace_bytes(pool, T, top_k=1) -> int:
    return int(lib().lora_workspace_bytes(pool, T, top_k))


def lora_workspace_init(ws, nbytes, stream=None):
    _check(lib().lora_workspace_init(ptr(ws), nbytes, stream_ptr(stream)), "lora_workspace_init")


def lora_apply_slices(pool, meta: Meta, x, ldx, y, ldy, ws, ws_bytes, stream=None):
    _check(lib().lora_apply_slices(pool, ctypes.byref(meta), ptr(x), ldx, ptr(y), ldy, ptr(ws), ws_bytes,
                                   stream_ptr(stream)), "lora_apply_slices")


def lora_apply_slices_static(pool, meta: Meta, x, ldx, y, ldy, stream=None):
    _check(lib().lora_apply_slices_static(pool, ctypes.byref(meta), ptr(x), ldx, ptr(y), ldy,
                                          stream_ptr(stream)), "lora_apply_slices_static")


def lora_static_scratch_bytes() -> int:
    return int(lib().lora_static_scratch_bytes())


def lora_logits_apply(pool, meta: Meta, hidden, ld_h, logits_in, ld_in, in_cols, mapping, logits_out, ld_out,
                      vocab_size, mup, ws, ws_bytes, stream=None):
    _check(lib().lora_logits_apply(pool, ctypes.byref(meta), ptr(hidden), ld_h, ptr(logits_in), ld_in, in_cols,
                                   ptr(mapping), ptr(logits_out), ld_out, vocab_size, float(mup), ptr(ws),
                                   ws_bytes, stream_ptr(stream)), "lora_logits_apply")


def lora_moe_apply(pool, meta: Meta, which, inp, ld_in, topk_w, out, ld_out, ws, ws_bytes, stream=None):
    _check(lib().lora_moe_apply(pool, ctypes.byref(meta), which, ptr(inp), ld_in, ptr(topk_w), ptr(out),
                                ld_out, ptr(ws), ws_bytes, stream_ptr(stream)), "lora_moe_apply")


def lora_moe_align_padded(pool, meta: Meta, block_m, cap, d_sorted, d_expert, d_npp, stream=None):
    _check(lib().lora_moe_align_padded(pool, ctypes.byref(meta), block_m, cap, ptr(d_sorted), ptr(d_expert),
                                       ptr(d_npp), stream_ptr(stream)), "lora_moe_align_padded")


def lora_moe_apply_blocks(pool, meta: Meta, which, inp, ld_in, topk_w, out, ld_out, d_sorted, d_expert, d_npp,
                          block_m, cap, stream=None):
    _check(lib().lora_moe_apply_blocks(pool, ctypes.byref(meta), which, ptr(inp), ld_in, ptr(topk_w), ptr(out),
                                       ld_out, ptr(d_sorted), ptr(d_expert), ptr(d_npp), block_m, cap,
                                       stream_ptr(stream)), "lora_moe_apply_blocks")


def lora_get_device_status(pool, stream=None) -> int:
    return int(lib().lora_get_device_status(pool, stream_ptr(stream)))


def lora_set_spin_limit(max_polls: int):
    lib().lora_set_spin_limit(int(max_polls))


def lora_set_kernel_policy(policy: int):
    lib().lora_set_kernel_policy(int(policy))


def lora_linear_apply(pool, meta: Meta, x, ldx, W, ldw, bias, y, ldy, ws, ws_bytes, stream=None):
    """Full LoRA linear layer: y = x W^T + bias + delta."""
    _check(lib().lora_linear_apply(pool, ctypes.byref(meta), ptr(x), int(ldx), ptr(W), int(ldw), ptr(bias), ptr(y),
                                   int(ldy), ptr(ws), ws_bytes, stream_ptr(stream)), "lora_linear_apply")


def lora_sink_experts_act(gate_up, ld_gate_up, gammas, ld_gammas, T, n_experts, d_mlp, h, ld_h, stream=None):
    """Inkling sink-expert activation between the w13 and w2 LoRA layers."""
    _check(lib().lora_sink_experts_act(ptr(gate_up), int(ld_gate_up), ptr(gammas), int(ld_gammas), int(T),
                                       int(n_experts), int(d_mlp), ptr(h), int(ld_h), stream_ptr(stream)),
           "lora_sink_experts_act")


def lora_kernel_launch_count() -> int:
    return int(lib().lora_kernel_launch_count())


def lora_last_cuda_error() -> int:
    return int(lib().lora_last_cuda_error())


def lora_status_string(code: int) -> str:
    return lib().lora_status_string(code).decode()
