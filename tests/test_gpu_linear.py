"""The full LoRA linear layer y = x W^T + bias + delta (vLLM LoRA layer pages,
BaseLinearLayerWithLoRA) through the C ABI against the oracle's merged form."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from heterogeneous_adapters_lora_gb300 import harness as H
from heterogeneous_adapters_lora_gb300 import inputs as gen
from heterogeneous_adapters_lora_gb300 import lora as L
from heterogeneous_adapters_lora_gb300.inputs import bf16_bits_to_f32, f32_to_bf16_bits
from gpu_util import active_mask, assert_delta

pytestmark = pytest.mark.gpu


def _run(c, with_bias):
    rng = np.random.default_rng(c.T)
    bias = f32_to_bf16_bits(rng.normal(0, 0.5, c.out_total).astype(np.float32)) if with_bias else None
    y_ref = oracle.linear(c, c.W, bias)
    run = H.DenseRun(c)
    try:
        run.build_meta()
        d_w = H.to_dev_u16(c.W)
        d_b = H.to_dev_u16(bias) if with_bias else None
        L.lora_linear_apply(run.pool, run.mb.meta, run.x, c.H, d_w, c.H, d_b, run.y, c.out_total, run.ws,
                            run.ws_bytes)
        y = run.y_host()
        assert run.status() == 0
    finally:
        run.close()
    got = bf16_bits_to_f32(y).astype(np.float64)
    assert_delta(got, y_ref, c.name + " full linear")
    # rows without an adapter are the base layer's output alone
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    base = oracle.linear(c, c.W, bias) - oracle.dense_delta(c)[1].astype(np.float64)
    assert_delta(got[~act], base[~act], c.name + " base rows")


@pytest.mark.parametrize("with_bias", [False, True])
def test_linear_tiny(with_bias):
    _run(gen.tiny(), with_bias)


def test_linear_decode_qkv_shapes():
    c = gen.dense_case(name="linear_qkv", T=256, H=4096, out_dims=(4096, 1024, 1024), L=32, R=16, seed=1102,
                       scales=np.full(32, 2.0, np.float32), p_none=0.1, with_W=True, std=0.05)
    _run(c, True)


def test_linear_argument_errors():
    c = gen.tiny()
    run = H.DenseRun(c)
    try:
        run.build_meta()
        d_w = H.to_dev_u16(c.W)
        with pytest.raises(L.LoraError) as e:   # W leading dimension below in_dim
            L.lora_linear_apply(run.pool, run.mb.meta, run.x, c.H, d_w, c.H - 8, None, run.y, c.out_total,
                                run.ws, run.ws_bytes)
        assert e.value.code == L.CODE["LORA_ERR_INVALID_ARG"]
        with pytest.raises(L.LoraError) as e:   # misaligned y
            L.lora_linear_apply(run.pool, run.mb.meta, run.x, c.H, d_w, c.H, None, run.y.data_ptr() + 2,
                                c.out_total, run.ws, run.ws_bytes)
        assert e.value.code == L.CODE["LORA_ERR_INVALID_ARG"]
    finally:
        run.close()
