"""Inkling sink experts (Inkling LoRA PR report, InklingSinkExpertsLinear):
the activation kernel against the oracle, and the whole chain w13 LoRA ->
activation -> w2 LoRA through the C ABI against the oracle chain."""
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


def _ulp_diff(a_bits, b_bits):
    """Distance in bf16 steps between two arrays of bf16 bits (same sign
    ordering via the usual integer mapping)."""
    def key(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + b)
    return np.abs(key(a_bits) - key(b_bits))


@pytest.mark.parametrize("n,d,T,pad", [(2, 1408, 256, 0), (2, 12, 33, 8), (3, 8, 1, 16), (4, 100, 70, 0)])
def test_sink_act_matches_oracle(n, d, T, pad):
    rng = np.random.default_rng(n * 1000 + d + T)
    W = n * d
    gu = f32_to_bf16_bits(rng.normal(0, 2.0, (T, 2 * W + pad)).astype(np.float32))
    gam = rng.uniform(-1.5, 1.5, (T, n + 1)).astype(np.float32)
    h_ref = oracle.sink_act(gu, gam, n, d)
    d_gu = H.to_dev_u16(gu)
    d_g = torch.from_numpy(gam).cuda()
    d_h = torch.full((T, W + pad), -1, dtype=torch.int16, device="cuda")
    L.lora_sink_experts_act(d_gu, 2 * W + pad, d_g, n + 1, T, n, d, d_h, W + pad)
    h = H.from_dev_u16(d_h)
    assert np.all(h[:, W:] == 0xFFFF), "columns past W must be untouched"
    diff = _ulp_diff(h[:, :W], h_ref)
    assert diff.max() <= 1, f"max bf16 step difference {diff.max()}"
    assert (diff > 0).mean() <= 0.01, f"{(diff > 0).mean():.4f} of the values differ"


def test_sink_act_argument_errors():
    x = torch.zeros((4, 32), dtype=torch.int16, device="cuda")
    g = torch.zeros((4, 2), dtype=torch.float32, device="cuda")
    h = torch.zeros((4, 16), dtype=torch.int16, device="cuda")
    bad = [dict(n=2, d=3),                       # W = 6 not a multiple of 8
           dict(ld_gu=24), dict(ld_h=8), dict(ld_g=1), dict(T=-1),
           dict(gu=x.data_ptr() + 2)]            # misaligned
    for kw in bad:
        with pytest.raises(L.LoraError) as e:
            L.lora_sink_experts_act(kw.get("gu", x), kw.get("ld_gu", 32), g, kw.get("ld_g", 2), kw.get("T", 4),
                                    kw.get("n", 2), kw.get("d", 8), h, kw.get("ld_h", 16))
        assert e.value.code == L.CODE["LORA_ERR_INVALID_ARG"], kw
    L.lora_sink_experts_act(x, 32, g, 2, 0, 2, 8, h, 16)  # T = 0: nothing to do


def test_sink_chain_matches_oracle_chain():
    c = gen.sink_case(name="chain", T=96, D=512, n_experts=2, d_mlp=136, L=4, R=16, seed=91)
    W = c.n_experts * c.d_mlp
    # oracle chain: w13 (base + delta, rounded to bf16 as the layer output is) -> act -> w2 delta
    y13_ref, _ = oracle.dense_delta(c.w13)
    h_ref = oracle.sink_act(f32_to_bf16_bits(y13_ref), c.gammas, c.n_experts, c.d_mlp)
    _, d2_ref = oracle.dense_delta(c.w2, x=h_ref)
    run = H.SinkRun(c)
    try:
        run.step()
        y2 = run.r2.y_host()
        assert run.status() == 0
    finally:
        run.close()
    act = active_mask(c.w2.idx, c.w2.L, c.w2.enabled, c.w2.ranks)
    got = bf16_bits_to_f32(y2).astype(np.float64) - bf16_bits_to_f32(c.w2.y0).astype(np.float64)
    assert_delta(got[act], d2_ref[act], "sink chain w2 delta")
    assert np.array_equal(y2[~act], c.w2.y0[~act]), "rows without an adapter keep the base output"
