"""Helpers for the oracle pins: fp64 brute force and rounding-error bounds.

These evaluate the closed forms with numpy in float64 on small inputs (a
library matmul per token), to check the fp32 loop oracle against the exact
result within a rigorous fp32 error bound.
"""
import json
import os

import numpy as np

from heterogeneous_adapters_lora_gb300.inputs import (DenseCase, MoECase, bf16_bits_to_f32,
                                                      f32_to_bf16_bits)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
U32 = 2.0 ** -24


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def active(a, L, enabled, ranks):
    return 0 <= a < L and enabled[a] != 0 and ranks[a] > 0


def exact_dense(c: DenseCase):
    """float64 delta and an fp32 error bound per element (sequential fp32 sums:
    |err| <= (H + r + 4) u * scale * |B| |A| |x|)."""
    O = c.out_total
    delta = np.zeros((c.T, O))
    bound = np.zeros((c.T, O))
    x = f64(c.x)
    for t in range(c.T):
        a = int(c.idx[t])
        if not active(a, c.L, c.enabled, c.ranks):
            continue
        r = int(c.ranks[a])
        off = 0
        for j, Oj in enumerate(c.out_dims):
            Aj = f64(c.A[j][a, :r, :])
            Bj = f64(c.B[j][a, :, :r])
            v = Aj @ x[t]
            delta[t, off:off + Oj] = c.scales[a] * (Bj @ v)
            vabs = np.abs(Aj) @ np.abs(x[t])
            bound[t, off:off + Oj] = (c.H + r + 4) * U32 * abs(c.scales[a]) * (np.abs(Bj) @ vabs)
            off += Oj
    return delta, bound + 1e-30


def exact_moe(c: MoECase, which: str):
    P = c.T * c.K
    if which == "w13":
        W = c.n13 * c.F13
    else:
        W = c.D
    delta = np.zeros((P, W))
    bound = np.zeros((P, W))
    x = f64(c.x)
    ic2 = f64(c.ic2)
    for p in range(P):
        t, e = p // c.K, int(c.topk_ids.reshape(-1)[p])
        a = int(c.idx[t])
        if not active(a, c.L, c.enabled, c.ranks):
            continue
        r = int(c.ranks[a])
        if which == "w13":
            for s in range(c.n13):
                ea = 0 if c.shared_outer else e
                As = f64(c.A13[s][a, ea, :r, :])
                Bs = f64(c.B13[s][a, e, :, :r])
                v = As @ x[t]
                sl = slice(s * c.F13, (s + 1) * c.F13)
                delta[p, sl] = c.scales[a] * (Bs @ v)
                bound[p, sl] = (c.D + r + 4) * U32 * abs(c.scales[a]) * (np.abs(Bs) @ (np.abs(As) @ np.abs(x[t])))
        else:
            eb = 0 if c.shared_outer else e
            As = f64(c.A2[a, e, :r, :])
            Bs = f64(c.B2[a, eb, :, :r])
            w = float(c.topk_w.reshape(-1)[p])
            v = As @ ic2[p]
            delta[p] = w * c.scales[a] * (Bs @ v)
            bound[p] = (c.F + r + 6) * U32 * abs(w * c.scales[a]) * (np.abs(Bs) @ (np.abs(As) @ np.abs(ic2[p])))
    return delta, bound + 1e-30


def dense_from_golden(g) -> DenseCase:
    T, H, L, R = g["T"], g["H"], g["L"], g["R"]
    out_dims = tuple(g["out_dims"])
    bits = lambda v: f32_to_bf16_bits(np.asarray(v, np.float32))
    A = [bits(g["A"][j]).reshape(L, R, H) for j in range(len(out_dims))]
    B = [bits(g["B"][j]).reshape(L, out_dims[j], R) for j in range(len(out_dims))]
    ranks = np.asarray(g["ranks"], np.int32)
    return DenseCase("golden", T, H, out_dims, L, R, ranks, np.asarray(g["scales"], np.float32),
                     (ranks > 0).astype(np.int32), np.asarray(g["idx"], np.int32),
                     bits(g["x"]).reshape(T, H), A, B, np.zeros((T, sum(out_dims)), np.uint16))


def moe_from_golden(g) -> MoECase:
    T, K, E, D, F, L, R = (g[k] for k in ("T", "K", "E", "D", "F", "L", "R"))
    bits = lambda v: f32_to_bf16_bits(np.asarray(v, np.float32))
    A13 = [bits(g["A13"][0]).reshape(L, E, R, D)]
    B13 = [bits(g["B13"][0]).reshape(L, E, F, R)]
    ranks = np.full(L, R, np.int32)
    return MoECase("golden", T, K, E, D, F, F, L, R, False, ranks, np.ones(L, np.float32),
                   np.ones(L, np.int32), np.asarray(g["idx"], np.int32),
                   np.asarray(g["topk_ids"], np.int32), np.asarray(g["topk_w"], np.float32),
                   bits(g["x"]).reshape(T, D), bits(g["ic2"]).reshape(T * K, F), A13, B13,
                   bits(g["A2"]).reshape(L, E, R, F), bits(g["B2"]).reshape(L, E, D, R),
                   np.zeros((T * K, F), np.uint16), np.zeros((T * K, D), np.uint16))
