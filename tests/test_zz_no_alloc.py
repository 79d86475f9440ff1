"""The allocation-free apply entry point (lora_apply_slices_static).

It serves callers that cannot hand the library a workspace (all device
memory already reserved by another allocator so cudaMalloc would fail,
latency-critical paths that may not block on an allocation, C hosts without
an allocator), by running the persistent split-K kernel on a fixed scratch
array inside the library's device image.  Its result must match the oracle
(twice the delta after two calls in a row on a zero base: the array keeps
the previous call's contents) and lora_apply_slices, within the tolerance
of the other parity tests.  This
file is collected last so a run that stops at the first failure has already
run every other test; it passes alone in a fresh process too.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from heterogeneous_adapters_lora_gb300 import harness as H
from heterogeneous_adapters_lora_gb300 import inputs as gen
from heterogeneous_adapters_lora_gb300 import lora as L
from heterogeneous_adapters_lora_gb300.inputs import bf16_bits_to_f32
from gpu_util import active_mask, assert_delta

pytestmark = pytest.mark.gpu


def _two_calls(run, use_static):
    run.y.copy_(H.to_dev_u16(run.case.y0))
    c = run.case
    for _ in range(2):
        if use_static:
            L.lora_apply_slices_static(run.pool, run.mb.meta, run.x, c.H, run.y, c.out_total)
        else:
            L.lora_apply_slices(run.pool, run.mb.meta, run.x, c.H, run.y, c.out_total, run.ws, run.ws_bytes)
    torch.cuda.synchronize()
    return run.y_host()


@pytest.mark.parametrize("which", ["decode_qkv", "small"])
def test_static_scratch_matches_workspace_entry_point(which):
    if which == "decode_qkv":
        c = gen.decode_qkv()
    else:
        c = gen.dense_case(name="small", T=70, H=1032, out_dims=(136, 264), L=5, R=24, seed=31,
                           ranks=(24, 13, 1, 8, 0), scales=(1.0, 2.0, 0.5, 1.5, 1.0), p_none=0.2)
    run = H.DenseRun(c)
    try:
        run.build_meta()
        y_ws = _two_calls(run, use_static=False)
        y_st = _two_calls(run, use_static=True)
        assert run.status() == 0
    finally:
        run.close()
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert np.array_equal(y_st[~act], c.y0[~act])
    base = bf16_bits_to_f32(c.y0)[act].astype(np.float64)
    d_ws = bf16_bits_to_f32(y_ws)[act] - base
    d_st = bf16_bits_to_f32(y_st)[act] - base
    assert_delta(d_st, d_ws, f"static vs workspace ({which})")
    _, d_ref = oracle.dense_delta(c)
    assert_delta(d_st, 2 * d_ref[act].astype(np.float64), f"static vs oracle ({which})")


def test_static_scratch_rejects_batches_beyond_its_size():
    assert L.lora_static_scratch_bytes() == 8 << 20
    d = L.PoolDesc()
    d.max_loras, d.max_rank, d.in_dim, d.n_slices = 8, 64, 4096, 2
    d.out_dims[0] = d.out_dims[1] = 1024
    pool = L.lora_pool_create(d)
    try:
        T = 8192
        mb = H.MetaBuffer(T, 8)
        idx = torch.zeros(T, dtype=torch.int32, device="cuda")
        L.lora_build_meta(pool, idx, T, None, 1, mb.meta)
        x = torch.zeros((T, 4096), dtype=torch.int16, device="cuda")
        y = torch.zeros((T, 2048), dtype=torch.int16, device="cuda")
        with pytest.raises(L.LoraError) as e:
            L.lora_apply_slices_static(pool, mb.meta, x, 4096, y, 2048)
        assert e.value.code == L.CODE["LORA_ERR_CAPACITY"]
    finally:
        L.lora_pool_destroy(pool)
