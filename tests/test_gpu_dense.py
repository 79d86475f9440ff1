"""Dense LoRA delta on the GPU (lora_apply_slices, lora_shrink, lora_expand)
against the CPU oracle: rel-Frobenius <= 1e-2 and max-abs <= 2e-2 on the
delta, inactive rows bit-identical."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from heterogeneous_adapters_lora_gb300 import harness as H
from heterogeneous_adapters_lora_gb300 import inputs as gen
from heterogeneous_adapters_lora_gb300 import lora as L
from heterogeneous_adapters_lora_gb300.inputs import bf16_bits_to_f32
from gpu_util import active_mask, assert_base_plus_delta, assert_delta, assert_rows_untouched

pytestmark = pytest.mark.gpu


def run_and_check(c, lm_head=False, base_random=False):
    run = H.DenseRun(c, lm_head=lm_head)
    try:
        run.step()
        y = run.y_host()
        assert run.status() == 0
    finally:
        run.close()
    y_ref, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_rows_untouched(y, c.y0, ~act)
    if base_random:
        assert_base_plus_delta(y, c.y0, d_ref, act)
        return None
    return assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], c.name)


def small_case(seed, T=100, H=2504, out_dims=(264, 136), Lk=5, R=24, ranks=(24, 13, 1, 8, 0),
               p_none=0.15, base_y="zero"):
    rng = np.random.default_rng(seed)
    return gen.dense_case(name=f"small{seed}", T=T, H=H, out_dims=out_dims, L=Lk, R=R, seed=seed,
                          ranks=ranks, scales=rng.uniform(0.5, 2.5, Lk).astype(np.float32),
                          p_none=p_none, base_y=base_y)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_small_ragged_multi_tile(seed):
    run_and_check(small_case(seed))


def test_small_random_base():
    run_and_check(small_case(5, base_y="random"), base_random=True)


@pytest.mark.parametrize("T", [1, 2, 17, 33])
def test_tiny_token_counts(T):
    run_and_check(small_case(11, T=T, p_none=0.0))


@pytest.mark.parametrize("T,seed", [(8, 23), (24, 21)])
def test_per_tile_one_item_per_cta(T, seed):
    # fewer rows than 4 per slot and few tiles: the per-tile shrink with one
    # item per CTA; ranks that end inside an 8-rank block, a single rank and
    # rank 0 (the seeds give tokens to slots 0, 1, 2, 3 and 5)
    run_and_check(small_case(seed, T=T, H=3000, out_dims=(264,), Lk=8, R=64,
                             ranks=(64, 40, 57, 1, 24, 33, 16, 0), p_none=0.1))


def test_per_tile_rank_groups_many_items():
    # 512 tokens over 1024 slots: more per-tile items than two waves, so the
    # copy-warp shrink that takes the ranks 16 at a time; ranks that end inside
    # a group (40, 57, 24, 33), a single rank and rank 0
    ranks = tuple((64, 40, 57, 1, 24, 33, 16, 0)[i % 8] for i in range(1024))
    run_and_check(small_case(31, T=512, H=1024, out_dims=(264,), Lk=1024, R=64, ranks=ranks, p_none=0.1))


def test_preset_tiny():
    run_and_check(gen.tiny())


def test_preset_decode_qkv():
    run_and_check(gen.decode_qkv())


def test_preset_decode_qkv_random_base():
    run_and_check(gen.decode_qkv(base_y="random"), base_random=True)


def test_preset_prefill_gate_up():
    run_and_check(gen.prefill_gate_up(permuted=True))


def test_preset_many_adapter_down():
    run_and_check(gen.many_adapter_down())


def test_lm_head_shape():
    c = gen.dense_case(name="lm_head", T=48, H=1024, out_dims=(128256,), L=3, R=16, seed=21,
                       scales=np.ones(3, np.float32), p_none=0.2)
    run_and_check(c, lm_head=True)


def test_all_none_and_rank0_leave_y_bits():
    c = small_case(3, base_y="random")
    c.idx[:] = -1
    run_and_check(c, base_random=True)
    c2 = small_case(4, base_y="random", ranks=(0, 0, 0, 0, 0))
    run_and_check(c2, base_random=True)


def test_reset_slot_gives_zero_delta_and_set_reuses_it():
    c = small_case(6, base_y="random")
    run = H.DenseRun(c)
    try:
        L.lora_reset(run.pool, 0)
        run.step()
        y = run.y_host()
        en = c.enabled.copy()
        en[0] = 0
        y_ref, d_ref = oracle.dense_delta(c, enabled=en)
        act = active_mask(c.idx, c.L, en, c.ranks)
        assert_rows_untouched(y, c.y0, ~act)
        assert_base_plus_delta(y, c.y0, d_ref, act)
        # set it again: slot 0 is back
        H.upload_dense_slot(run.pool, c, 0)
        run.y.copy_(H.to_dev_u16(c.y0))
        run.step()
        y = run.y_host()
        _, d_ref = oracle.dense_delta(c)
        act = active_mask(c.idx, c.L, c.enabled, c.ranks)
        assert_base_plus_delta(y, c.y0, d_ref, act)
    finally:
        run.close()


def test_set_packed_equals_per_slice_set():
    c = small_case(8, out_dims=(64, 128, 64), ranks=(24, 24, 24, 24, 24))
    # one A for all slices, one B split by the slice widths
    for a in range(c.L):
        for j in range(1, 3):
            c.A[j][a] = c.A[0][a]
    run = H.DenseRun(c)
    try:
        for a in range(c.L):
            r = int(c.ranks[a])
            Bw = np.ascontiguousarray(np.concatenate([c.B[j][a, :, :r] for j in range(3)], axis=0))
            L.lora_set_packed(run.pool, a, r, float(c.scales[a]), np.ascontiguousarray(c.A[0][a, :r]), Bw)
        run.step()
        y = run.y_host()
    finally:
        run.close()
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], "packed")


def test_standalone_shrink_expand():
    c = small_case(9)
    run = H.DenseRun(c)
    try:
        run.build_meta()
        v = torch.full((c.n_slices, c.T, c.R), 7.0, dtype=torch.float32, device="cuda")
        L.lora_shrink(run.pool, run.mb.meta, run.x, c.H, v)
        vh = v.cpu().numpy()
        L.lora_expand(run.pool, run.mb.meta, v, run.y, c.out_total)
        y = run.y_host()
    finally:
        run.close()
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    x = bf16_bits_to_f32(c.x).astype(np.float64)
    for j in range(c.n_slices):
        for t in range(c.T):
            a = int(c.idx[t])
            if not act[t]:
                assert np.all(vh[j, t] == 0)
                continue
            r = int(c.ranks[a])
            exact = bf16_bits_to_f32(c.A[j][a, :r]).astype(np.float64) @ x[t]
            assert np.allclose(vh[j, t, :r], exact, rtol=1e-4, atol=1e-5)
            assert np.all(vh[j, t, r:] == 0)
    _, d_ref = oracle.dense_delta(c)
    assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], "shrink+expand")
    assert_rows_untouched(y, c.y0, ~act)


def test_repeated_calls_reuse_workspace():
    """The fused kernel leaves its workspace control words zero: many calls in
    a row each add one delta."""
    c = small_case(12, p_none=0.0)
    run = H.DenseRun(c)
    try:
        run.build_meta()
        for _ in range(5):
            run.apply()
        y = run.y_host()
        assert run.status() == 0
    finally:
        run.close()
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_delta(bf16_bits_to_f32(y)[act], 5 * d_ref[act], "5 calls")


def test_smaller_batch_than_workspace():
    c = small_case(13, T=64)
    run = H.DenseRun(c, max_rows=4096)
    try:
        run.step()
        y = run.y_host()
    finally:
        run.close()
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], "small batch")


def test_cuda_graph_capture_of_meta_and_apply():
    c = gen.decode_qkv()
    run = H.DenseRun(c)
    try:
        s = torch.cuda.Stream()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                run.step()
        run.y.zero_()
        g.replay()
        torch.cuda.synchronize()
        y = run.y_host()
    finally:
        run.close()
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_delta(bf16_bits_to_f32(y)[act], d_ref[act], "graph")


@pytest.mark.parametrize("policy", [0, 3], ids=["fused", "split"])
def test_apply_after_every_slot_reset_leaves_y(policy):
    # Every slot reset: the key-major shrink's CTAs all find rank 0 and leave
    # at once.  They must still let the expand start only after the metadata
    # build is complete, so the expand neither reads the previous build's
    # tile lists nor rewrites y rows the previous apply is still storing.
    # Policy 3 keeps the batch on the split kernels (key-major shrink and the
    # tensor-core expand); 0 takes the fused decode kernel.
    c = gen.decode_qkv()
    L.lora_set_kernel_policy(policy)
    run = H.DenseRun(c)
    try:
        run.step()
        y1 = run.y_host()
        for a in range(c.L):
            L.lora_reset(run.pool, a)
        for _ in range(3):
            run.step()
        y2 = run.y_host()
        assert run.status() == 0
    finally:
        run.close()
        L.lora_set_kernel_policy(0)
    assert np.array_equal(y1, y2)
    _, d_ref = oracle.dense_delta(c)
    act = active_mask(c.idx, c.L, c.enabled, c.ranks)
    assert_delta(bf16_bits_to_f32(y1)[act], d_ref[act], "before reset")
