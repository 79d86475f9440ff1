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


@pytest.fixture(autouse=True, params=[0, 6], ids=["library_gemm", "tcgen05_fused"])
def linear_path(request):
    """Kernel policy 0: cuBLASLt base GEMM + the library's apply; policy 6:
    the tcgen05 GEMM whose accumulator takes the delta."""
    L.lora_set_kernel_policy(request.param)
    yield request.param
    L.lora_set_kernel_policy(0)


def _run(c, with_bias, bias_std=0.5, ldx=None, ldy=None):
    """Run the full linear layer; returns (y as float64 [T][out_total], base of
    the oracle (x W^T + bias, float64), delta of the oracle, active rows)."""
    rng = np.random.default_rng(c.T)
    bias = f32_to_bf16_bits(rng.normal(0, bias_std, c.out_total).astype(np.float32)) if with_bias else None
    y_ref = oracle.linear(c, c.W, bias)
    _, d_ref = oracle.dense_delta(c)
    d_ref = d_ref.astype(np.float64)
    base = y_ref - d_ref
    ldx = c.H if ldx is None else ldx
    ldy = c.out_total if ldy is None else ldy
    run = H.DenseRun(c)
    try:
        run.build_meta()
        x = torch.zeros((c.T, ldx), dtype=torch.int16, device="cuda")
        x[:, :c.H] = run.x
        y = torch.full((c.T, ldy), 0x7fc0, dtype=torch.int16, device="cuda")  # NaN fill: all of y is written
        d_w = H.to_dev_u16(c.W)
        d_b = H.to_dev_u16(bias) if with_bias else None
        L.lora_linear_apply(run.pool, run.mb.meta, x, ldx, d_w, c.H, d_b, y, ldy, run.ws, run.ws_bytes)
        yh = H.from_dev_u16(y)
        assert run.status() == 0
    finally:
        run.close()
    # the padding columns of y are not the layer's: left as they were
    assert np.all(yh[:, c.out_total:] == 0x7fc0)
    got = bf16_bits_to_f32(np.ascontiguousarray(yh[:, :c.out_total])).astype(np.float64)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    # whole output within the delta tolerance, rows without an adapter = base alone
    assert_delta(got, y_ref, c.name + " full linear")
    assert_delta(got[~act], base[~act], c.name + " base rows")
    return got, base, d_ref, act


def _small_base(c, w_std, seed):
    """Replace the case's base weight by one whose output is of the delta's size."""
    rng = np.random.default_rng(seed)
    c.W = f32_to_bf16_bits(rng.normal(0, w_std, (c.out_total, c.H)).astype(np.float32))
    return c


@pytest.mark.parametrize("with_bias", [False, True])
def test_linear_tiny(with_bias):
    _run(gen.tiny(), with_bias)


def test_linear_decode_qkv_shapes():
    c = gen.dense_case(name="linear_qkv", T=256, H=4096, out_dims=(4096, 1024, 1024), L=32, R=16, seed=1102,
                       scales=np.full(32, 2.0, np.float32), p_none=0.1, with_W=True, std=0.05)
    _run(c, True)


@pytest.mark.parametrize("shape", ["tiny", "qkv"])
def test_linear_delta_isolated(shape):
    # The base output x W^T + bias is made about as large as the delta, so the
    # delta y - base (base from the oracle) is checked at the delta tolerance
    # on its own: a delta a few percent wrong fails here, where a large base
    # would hide it in the whole-output norm.  Padded leading dimensions of x
    # and y are exercised at the same time.
    if shape == "tiny":
        c = _small_base(gen.tiny(), 0.002, 3)
        ldx, ldy = c.H + 24, c.out_total + 40
    else:
        c = gen.dense_case(name="linear_qkv_small_base", T=256, H=4096, out_dims=(4096, 1024, 1024), L=32, R=16,
                           seed=1103, scales=np.full(32, 2.0, np.float32), p_none=0.1, with_W=True, std=0.02)
        c = _small_base(c, 0.002, 4)
        ldx, ldy = c.H + 64, c.out_total + 8
    got, base, d_ref, act = _run(c, True, bias_std=0.002, ldx=ldx, ldy=ldy)
    assert np.abs(base[act]).max() < 4 * np.abs(d_ref[act]).max()  # the base does not dominate
    assert_delta(got[act] - base[act], d_ref[act], c.name + " delta alone")


def test_linear_zero_base_is_the_delta():
    # W = 0 and no bias: the layer's output is the delta itself
    c = gen.tiny()
    c.W = np.zeros_like(c.W)
    got, base, d_ref, act = _run(c, False)
    assert np.all(base == 0)
    assert np.all(got[~act] == 0)
    assert_delta(got[act], d_ref[act], "zero base")


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


def _segment_idx(T, lengths_slots):
    idx = np.empty(T, np.int32)
    t = 0
    for n, a in lengths_slots:
        idx[t:t + n] = a
        t += n
    assert t == T
    return idx


def test_linear_prefill_segments_wide_tiles():
    """Prefill-like batch: contiguous runs of one adapter (one run without),
    mixed ranks up to 64, a ragged last tile, and enough tiles for the
    256-wide output tiles of the tensor-core GEMM."""
    T = 2100
    idx = _segment_idx(T, [(300, 0), (517, 1), (129, 2), (200, -1), (411, 3), (64, 5), (279, 6), (200, 7)])
    c = gen.dense_case(name="linear_prefill", T=T, H=512, out_dims=(2560, 2560), L=8, R=64, seed=1201,
                       ranks=(64, 24, 8, 64, 0, 40, 64, 16), scales=(1.0, 0.5, 2.0, 1.0, 1.0, 1.5, 1.0, 0.25),
                       idx=idx, with_W=True)
    c = _small_base(c, 0.004, 5)
    got, base, d_ref, act = _run(c, True, bias_std=0.004)
    assert np.abs(base[act]).max() < 4 * np.abs(d_ref[act]).max()  # the base does not dominate
    assert_delta(got[act] - base[act], d_ref[act], c.name + " delta alone")


def test_linear_many_slots_per_tile():
    """160 slots of rank <= 12 over 300 tokens: up to 128 distinct slots in a
    128-token tile, four slots per delta block, and a hidden size of four K
    blocks (every delta block after the base blocks)."""
    rng = np.random.default_rng(77)
    ranks = rng.choice([12, 5, 0, 8], size=160).astype(np.int32)
    c = gen.dense_case(name="linear_many", T=300, H=256, out_dims=(384, 128), L=160, R=12, seed=1202,
                       ranks=ranks, p_none=0.1, with_W=True)
    c = _small_base(c, 0.0004, 6)
    got, base, d_ref, act = _run(c, True, bias_std=0.0002, ldy=c.out_total + 8)
    assert np.abs(base[act]).max() < 4 * np.abs(d_ref[act]).max()  # the base does not dominate
    assert_delta(got[act] - base[act], d_ref[act], c.name + " delta alone")


def test_linear_rank_above_64_uses_the_library_gemm():
    c = gen.dense_case(name="linear_r72", T=70, H=256, out_dims=(256,), L=3, R=72, seed=1203, with_W=True)
    c = _small_base(c, 0.002, 7)
    got, base, d_ref, act = _run(c, False)
    assert np.abs(base[act]).max() < 4 * np.abs(d_ref[act]).max()  # the base does not dominate
    assert_delta(got[act] - base[act], d_ref[act], c.name + " delta alone")
