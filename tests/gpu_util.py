"""Shared helpers of the GPU parity tests (tolerances, tile derivation)."""
import numpy as np

from heterogeneous_adapters_lora_gb300.inputs import bf16_bits_to_f32

# Tolerances of the delta against the fp32 oracle (bf16 inputs, fp32 accumulation).
REL_FROB = 1e-2
MAX_ABS = 2e-2


def delta_errors(d_gpu, d_ref):
    diff = d_gpu.astype(np.float64) - d_ref.astype(np.float64)
    ref = np.linalg.norm(d_ref.astype(np.float64))
    rel = np.linalg.norm(diff) / max(ref, 1e-30)
    return rel, float(np.abs(diff).max()) if diff.size else 0.0


def assert_delta(d_gpu, d_ref, what=""):
    rel, mx = delta_errors(d_gpu, d_ref)
    assert rel <= REL_FROB and mx <= MAX_ABS, f"{what}: rel_frob={rel:.3e} max_abs={mx:.3e}"
    return rel, mx


def assert_rows_untouched(y_gpu_bits, y0_bits, rows):
    assert np.array_equal(y_gpu_bits[rows], y0_bits[rows])


def assert_base_plus_delta(y_gpu_bits, y0_bits, d_ref, rows):
    """With a non-zero base, y_out must equal bf16(y_in + delta) up to one bf16
    ulp of |y_in + delta| plus the delta tolerance."""
    y = bf16_bits_to_f32(y_gpu_bits[rows]).astype(np.float64)
    exact = bf16_bits_to_f32(y0_bits[rows]).astype(np.float64) + d_ref[rows]
    ulp = np.abs(exact) * 2.0 ** -7
    assert np.all(np.abs(y - exact) <= ulp + MAX_ABS)


def tiles_from_groups(group_start, tile_rows=16):
    tg, tr = [], []
    for g in range(len(group_start) - 1):
        for r0 in range(group_start[g], group_start[g + 1], tile_rows):
            tg.append(g)
            tr.append(r0)
    return np.asarray(tg, np.int32), np.asarray(tr, np.int32)


def active_mask(idx, L, enabled, ranks):
    return np.array([bool(0 <= a < L and enabled[a] and ranks[a] > 0) for a in idx], dtype=bool)


def tile_keyn(tg, tr, group_key, group_start, tile_rows=16):
    """(key << 5) | rows of each tile, from the oracle's groups."""
    out = []
    for g, r0 in zip(tg, tr):
        n = min(tile_rows, group_start[g + 1] - r0)
        out.append((int(group_key[g]) << 5) | int(n))
    return np.asarray(out, np.int32)


def long_short_tiles(group_key, group_start, sorted_rows, dense=True, long_min=64, lrows=128, srows=16):
    """Expected long (contiguous-run, 128-row) and short (16-row) tile lists."""
    lt, st = [], []
    for g in range(len(group_start) - 1):
        s0, s1 = int(group_start[g]), int(group_start[g + 1])
        c = s1 - s0
        key = int(group_key[g])
        run = dense and c >= long_min and int(sorted_rows[s1 - 1]) - int(sorted_rows[s0]) == c - 1
        if run:
            for r0 in range(s0, s1, lrows):
                n = min(lrows, s1 - r0)
                lt.append((r0, (key << 8) | n, int(sorted_rows[s0]) + (r0 - s0)))
        else:
            for r0 in range(s0, s1, srows):
                st.append((r0, (key << 5) | min(srows, s1 - r0)))
    return lt, st
