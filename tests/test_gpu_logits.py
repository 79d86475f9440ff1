"""lm_head with LoRA end to end (reindex of the gathered logits, delta,
vocab slice, muP multiplier) against the oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from heterogeneous_adapters_lora_gb300 import harness as H
from heterogeneous_adapters_lora_gb300 import inputs as gen
from heterogeneous_adapters_lora_gb300 import lora as L
from heterogeneous_adapters_lora_gb300.inputs import bf16_bits_to_f32, f32_to_bf16_bits
from gpu_util import MAX_ABS

pytestmark = pytest.mark.gpu


def _case(vocab_padded, T, seed, p_none=0.2):
    return gen.dense_case(name="lm_head", T=T, H=1024, out_dims=(vocab_padded,), L=3, R=16, seed=seed,
                          scales=np.ones(3, np.float32), p_none=p_none)


@pytest.mark.parametrize("mup", [1.0, 0.125])
@pytest.mark.parametrize("with_map", [False, True])
def test_logits_end_to_end(mup, with_map):
    V, Vp, T = 50000, 50176, 40
    c = _case(Vp, T, seed=61)
    rng = np.random.default_rng(7)
    in_cols = Vp
    base = f32_to_bf16_bits(rng.normal(0, 1, (T, in_cols)).astype(np.float32))
    mapping = rng.permutation(in_cols)[:V].astype(np.int32) if with_map else None
    run = H.DenseRun(c, lm_head=True)
    try:
        run.build_meta()
        d_in = H.to_dev_u16(base)
        d_map = torch.from_numpy(mapping).cuda() if with_map else None
        out = torch.zeros((T, Vp), dtype=torch.int16, device="cuda")
        L.lora_logits_apply(run.pool, run.mb.meta, run.x, c.H, d_in, in_cols, in_cols, d_map, out, Vp, V, mup,
                            run.ws, run.ws_bytes)
        got = bf16_bits_to_f32(H.from_dev_u16(out))[:, :V].astype(np.float64)
        assert run.status() == 0
    finally:
        run.close()
    _, d_ref = oracle.dense_delta(c)
    ref = oracle.logits(base, d_ref, V, mapping=mapping, mup=mup).astype(np.float64)
    err = np.abs(got - ref)
    # two roundings to bf16 (base * mup, then + delta * mup) against one in the oracle
    assert np.all(err <= np.abs(ref) * 2.0 ** -7 + mup * MAX_ABS), err.max()


def test_logits_rejects_vocab_beyond_pool_and_guard():
    c = _case(1024, 8, seed=62)
    run = H.DenseRun(c, lm_head=True)
    try:
        run.build_meta()
        out = torch.zeros((8, 1024), dtype=torch.int16, device="cuda")
        with pytest.raises(L.LoraError) as e:
            L.lora_logits_apply(run.pool, run.mb.meta, run.x, c.H, out, 1024, 1024, None, out, 1024, 1032,
                                1.0, run.ws, run.ws_bytes)
        assert e.value.code == L.CODE["LORA_ERR_SHAPE"]
    finally:
        run.close()
