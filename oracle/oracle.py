"""ctypes wrapper around the C oracle (``lora_oracle.c``) -- test infrastructure.

Every function here only marshals numpy arrays into the C routines and
reshapes their outputs; the arithmetic lives in ``lora_oracle.c``, except the
base product of ``linear``, a float64 numpy matmul (a library primitive).  Parity
status: every routine is pinned by ``tests/test_oracle_pins.py`` (brute force
in fp64, the merged-weight identity, the page invariants and a hand-derived
golden case); none is "parity unpinned".
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading
from types import SimpleNamespace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_LIB = os.path.join(_HERE, "liblora_oracle.so")
_lock = threading.Lock()
_lib = None

_I32P = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_F32P = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_U16P = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_PP = ctypes.POINTER(ctypes.c_void_p)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, OpenMP over independent tokens,
    no FP contraction so every host gives the same bits)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    lib.lo_max_threads.restype = ctypes.c_int
    lib.lo_dense_meta.restype = _I32
    lib.lo_dense_meta.argtypes = [_I32, _I32P, _I32, _I32P, _I32P, _I32P, _I32P, _I32P,
                                  _I32P, _I32P, _I32P, _I32P, _I32P]
    lib.lo_dense_delta.restype = None
    lib.lo_dense_delta.argtypes = [_I32, _I32, _I32, _I32P, _I32, _I32, _I32P, _I32P, _I32P,
                                   _F32P, _U16P, _I64, _PP, _PP, _U16P, _I64, _F32P, _F32P,
                                   ctypes.c_int]
    lib.lo_moe_meta.restype = _I32
    lib.lo_moe_meta.argtypes = [_I32, _I32, _I32, _I32, _I32P, _I32P, _I32P, _I32P, _I32P,
                                _I32P, _I32P, _I32P, _I32P, _I32P, _I32P, _I32P]
    lib.lo_moe_w13.restype = None
    lib.lo_moe_w13.argtypes = [_I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                               _I32P, _I32P, _I32P, _I32P, _F32P, _U16P, _I64, _PP, _PP,
                               _U16P, _I64, _F32P, _F32P, ctypes.c_int]
    lib.lo_moe_align_padded.restype = _I32
    lib.lo_moe_align_padded.argtypes = [_I32, _I32, _I32, _I32, _I32P, _I32P, _I32P, _I32P, _I32, _I32, _I32P,
                                        _I32P, _I32P]
    lib.lo_logits.restype = None
    lib.lo_logits.argtypes = [_I32, _I32, ctypes.c_void_p, _U16P, _I64, _F32P, _I64, ctypes.c_float, _F32P,
                              _I64]
    lib.lo_sink_act.restype = None
    lib.lo_sink_act.argtypes = [_I32, _I32, _I32, _U16P, _I64, _F32P, _I64, _U16P, _I64]
    lib.lo_moe_w2.restype = None
    lib.lo_moe_w2.argtypes = [_I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                              _I32P, _I32P, _F32P, _I32P, _I32P, _F32P, _U16P, _I64,
                              _U16P, _U16P, _U16P, _I64, _F32P, _F32P, ctypes.c_int]
    return lib


@contextlib.contextmanager
def use_library(path):
    """Temporarily route every oracle call to another build of the oracle
    source (the pin tests use this to check that planted mistakes are caught)."""
    global _lib
    with _lock:
        saved = _lib
        _lib = _bind(path)
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def compile_variant(src_text: str, out_path: str) -> str:
    """Compile a (possibly modified) copy of the oracle source with the same flags."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                    "-fPIC", "-shared", src, "-o", out_path, "-lm"], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = _bind(build())
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().lo_max_threads())


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def _ptr_array(arrs):
    ptrs = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    return ctypes.cast(ptrs, _PP)


def dense_meta(idx, L, enabled, rank):
    """Stable sort by slot: returns sorted_tok, counts, segments (see the C file)."""
    lib = _load()
    idx = _c(idx, np.int32)
    T = idx.shape[0]
    enabled, rank = _c(enabled, np.int32), _c(rank, np.int32)
    sorted_tok = np.empty(T, np.int32)
    slot_count = np.empty(L, np.int32)
    seg_slot = np.full(L, -1, np.int32)
    seg_start = np.zeros(L + 1, np.int32)
    slot_seg = np.empty(L, np.int32)
    n_active, n_seg, n_bad = (np.zeros(1, np.int32) for _ in range(3))
    rc = lib.lo_dense_meta(T, idx, L, enabled, rank, sorted_tok, slot_count, seg_slot, seg_start,
                           slot_seg, n_active, n_seg, n_bad)
    assert rc == 0
    S = int(n_seg[0])
    return SimpleNamespace(sorted_tok=sorted_tok, slot_count=slot_count, seg_slot=seg_slot[:S].copy(),
                           seg_start=seg_start[: S + 1].copy(), slot_seg=slot_seg,
                           n_active=int(n_active[0]), n_seg=S, n_bad=int(n_bad[0]))


def dense_delta(case=None, *, x=None, idx=None, A=None, B=None, y_in=None, ranks=None,
                scales=None, enabled=None, out_dims=None, threads: int = 0):
    """Oracle for the dense multi-slice delta.  Returns (y_ref, delta_ref), fp32 [T][sum O]."""
    lib = _load()
    if case is not None:
        x = case.x if x is None else x
        idx = case.idx if idx is None else idx
        A = case.A if A is None else A
        B = case.B if B is None else B
        y_in = case.y0 if y_in is None else y_in
        ranks = case.ranks if ranks is None else ranks
        scales = case.scales if scales is None else scales
        enabled = case.enabled if enabled is None else enabled
        out_dims = case.out_dims if out_dims is None else out_dims
    x = _c(x, np.uint16)
    T, H = x.shape
    A = [_c(a, np.uint16) for a in A]
    B = [_c(b, np.uint16) for b in B]
    L, R = A[0].shape[0], A[0].shape[1]
    out_dims = _c(list(out_dims), np.int32)
    y_in = _c(y_in, np.uint16)
    ldy = y_in.shape[1]
    assert ldy >= int(out_dims.sum())
    y_ref = np.empty((T, ldy), np.float32)
    d_ref = np.empty((T, ldy), np.float32)
    lib.lo_dense_delta(T, H, len(A), out_dims, L, R, _c(idx, np.int32), _c(enabled, np.int32),
                       _c(ranks, np.int32), _c(scales, np.float32), x, H, _ptr_array(A),
                       _ptr_array(B), y_in, ldy, y_ref, d_ref, int(threads))
    return y_ref, d_ref


def moe_meta(topk_ids, idx, L, E, enabled, rank):
    lib = _load()
    topk_ids = _c(topk_ids, np.int32)
    T, K = topk_ids.shape
    NK = L * E
    sorted_pair = np.empty(T * K, np.int32)
    key_count = np.empty(NK, np.int32)
    key_offset = np.empty(NK + 1, np.int32)
    group_key = np.full(NK, -1, np.int32)
    group_start = np.zeros(NK + 1, np.int32)
    n_active, n_groups, n_bad = (np.zeros(1, np.int32) for _ in range(3))
    rc = lib.lo_moe_meta(T, K, E, L, topk_ids, _c(idx, np.int32), _c(enabled, np.int32),
                         _c(rank, np.int32), sorted_pair, key_count, key_offset, group_key,
                         group_start, n_active, n_groups, n_bad)
    assert rc == 0
    G = int(n_groups[0])
    return SimpleNamespace(sorted_pair=sorted_pair, key_count=key_count, key_offset=key_offset,
                           group_key=group_key[:G].copy(), group_start=group_start[: G + 1].copy(),
                           n_active=int(n_active[0]), n_groups=G, n_bad=int(n_bad[0]))


def moe_w13(c, *, ic1_in=None, threads: int = 0, idx=None, enabled=None):
    """Oracle for the w13 MoE-LoRA delta of case ``c``; returns (ic1_ref, delta_ref)."""
    lib = _load()
    ic1_in = _c(c.ic1_0 if ic1_in is None else ic1_in, np.uint16)
    P, ld1 = ic1_in.shape
    out = np.empty((P, ld1), np.float32)
    dl = np.empty((P, ld1), np.float32)
    A13 = [_c(a, np.uint16) for a in c.A13]
    B13 = [_c(b, np.uint16) for b in c.B13]
    lib.lo_moe_w13(c.T, c.K, c.D, c.F13, c.E, c.L, c.R, len(A13), int(c.shared_outer),
                   _c(c.idx if idx is None else idx, np.int32), _c(c.topk_ids, np.int32),
                   _c(c.enabled if enabled is None else enabled, np.int32), _c(c.ranks, np.int32),
                   _c(c.scales, np.float32), _c(c.x, np.uint16), c.D, _ptr_array(A13),
                   _ptr_array(B13), ic1_in, ld1, out, dl, int(threads))
    return out, dl


def moe_w2(c, *, ic3_in=None, threads: int = 0, idx=None, enabled=None):
    """Oracle for the w2 MoE-LoRA delta of case ``c``; returns (ic3_ref, delta_ref)."""
    lib = _load()
    ic3_in = _c(c.ic3_0 if ic3_in is None else ic3_in, np.uint16)
    P, ld3 = ic3_in.shape
    out = np.empty((P, ld3), np.float32)
    dl = np.empty((P, ld3), np.float32)
    lib.lo_moe_w2(c.T, c.K, c.D, c.F, c.E, c.L, c.R, int(c.shared_outer),
                  _c(c.idx if idx is None else idx, np.int32), _c(c.topk_ids, np.int32),
                  _c(c.topk_w, np.float32), _c(c.enabled if enabled is None else enabled, np.int32),
                  _c(c.ranks, np.int32), _c(c.scales, np.float32), _c(c.ic2, np.uint16), c.F,
                  _c(c.A2, np.uint16), _c(c.B2, np.uint16), ic3_in, ld3, out, dl, int(threads))
    return out, dl


def moe_align_padded(topk_ids, idx, L, E, enabled, rank, block_m, cap):
    """Block-padded per-adapter alignment (see lora_oracle.c)."""
    lib = _load()
    topk_ids = _c(topk_ids, np.int32)
    T, K = topk_ids.shape
    sorted_ = np.empty((L, cap), np.int32)
    expert = np.empty((L, cap // block_m), np.int32)
    npp = np.empty(L, np.int32)
    rc = lib.lo_moe_align_padded(T, K, E, L, topk_ids, _c(idx, np.int32), _c(enabled, np.int32),
                                 _c(rank, np.int32), block_m, cap, sorted_, expert, npp)
    assert rc == 0, "capacity"
    return SimpleNamespace(sorted=sorted_, expert=expert, npp=npp)


def logits(logits_in, delta, vocab_size, mapping=None, mup=1.0):
    """lm_head with LoRA: reindex the sharded logits, add the delta (from
    dense_delta), keep the first vocab_size columns, multiply by mup."""
    lib = _load()
    logits_in = _c(logits_in, np.uint16)
    delta = _c(delta, np.float32)
    T = logits_in.shape[0]
    out = np.empty((T, vocab_size), np.float32)
    m = None if mapping is None else _c(mapping, np.int32)
    lib.lo_logits(T, vocab_size, None if m is None else m.ctypes.data, logits_in, logits_in.shape[1], delta,
                  delta.shape[1], float(mup), out, vocab_size)
    return out


def linear(case, W, bias=None, threads: int = 0):
    """Full LoRA linear layer y = x W^T + bias + delta (BaseLinearLayerWithLoRA:
    base output, then the delta of lo_dense_delta added).  The base product of
    the bf16 values is a library matmul in float64; returns float64 [T][O]."""
    from heterogeneous_adapters_lora_gb300.inputs import bf16_bits_to_f32
    x = bf16_bits_to_f32(np.asarray(case.x)).astype(np.float64)
    Wf = bf16_bits_to_f32(np.asarray(W)).astype(np.float64)
    base = x @ Wf.T
    if bias is not None:
        base = base + bf16_bits_to_f32(np.asarray(bias)).astype(np.float64)[None, :]
    _, delta = dense_delta(case, threads=threads)
    return base + delta.astype(np.float64)


def sink_act(gate_up, gammas, n_experts, d_mlp):
    """Inkling sink-expert activation: bf16 bits h[T][n*d_mlp] from bf16 bits
    gate_up[T][2*n*d_mlp] and fp32 gammas[T][n]."""
    lib = _load()
    gate_up = _c(gate_up, np.uint16)
    gammas = _c(gammas, np.float32)
    T = gate_up.shape[0]
    W = n_experts * d_mlp
    assert gate_up.shape[1] >= 2 * W and gammas.shape[1] >= n_experts
    h = np.empty((T, W), np.uint16)
    lib.lo_sink_act(T, n_experts, d_mlp, gate_up, gate_up.shape[1], gammas, gammas.shape[1], h, W)
    return h


__all__ = ["linear", "sink_act", "logits", "moe_align_padded", "build", "use_library", "compile_variant", "source_text", "max_threads", "dense_meta", "dense_delta", "moe_meta", "moe_w13", "moe_w2"]
