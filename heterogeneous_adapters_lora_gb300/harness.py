"""Device-side plumbing around the C ABI: upload a seeded case into a pool,
allocate metadata/workspace buffers with PyTorch, and call the library.

Nothing here computes any part of the LoRA delta; it only moves the inputs
of ``inputs.DenseCase`` / ``inputs.MoECase`` to the GPU and forwards to the
same-name wrappers of ``lora``.
"""
from __future__ import annotations

import numpy as np
import torch

from . import lora as L


def to_dev_u16(a: np.ndarray, device="cuda") -> torch.Tensor:
    """bf16 bit patterns (uint16) -> int16 device tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device)


def from_dev_u16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


# bf16 bits written into the padding columns of padded rows: a NaN, so a
# kernel that read padding into a product would show it in its output
PAD_BITS = 0x7FC1


def to_dev_u16_padded(a: np.ndarray, pad: int, device="cuda") -> torch.Tensor:
    """[rows][cols] bf16 bits -> device [rows][cols + pad]; pad columns hold PAD_BITS."""
    if pad == 0:
        return to_dev_u16(a, device)
    rows, cols = a.shape
    host = np.full((rows, cols + pad), PAD_BITS, np.uint16)
    host[:, :cols] = a
    return to_dev_u16(host, device)


class MetaBuffer:
    """Caller-owned metadata buffer bound to a ``lora_meta_t``."""

    def __init__(self, max_rows: int, max_keys: int, device="cuda"):
        self.nbytes = L.lora_meta_bytes(max_rows, max_keys)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.meta = L.Meta()
        L.lora_meta_bind(self.meta, self.buf, self.nbytes, max_rows, max_keys)

    def _arr(self, name, n):
        addr = getattr(self.meta, name)
        off = addr - self.buf.data_ptr()
        return self.buf[off:off + 4 * n].view(torch.int32)

    def read(self):
        """Copy the metadata arrays to host numpy (synchronises)."""
        m = self.meta
        cnt = self._arr("counters", 8).cpu().numpy()
        n_active, G, n_bad, NT, NS, NL = (int(v) for v in cnt[:6])
        rows = m.T * m.top_k
        K = m.n_keys
        out = dict(n_active=n_active, n_groups=G, n_bad=n_bad, n_tiles=NT,
                   sorted=self._arr("sorted", rows).cpu().numpy(),
                   key_count=self._arr("key_count", K).cpu().numpy(),
                   key_offset=self._arr("key_offset", K + 1).cpu().numpy(),
                   group_key=self._arr("group_key", G).cpu().numpy(),
                   group_start=self._arr("group_start", G + 1).cpu().numpy(),
                   key_group=self._arr("key_group", K).cpu().numpy(),
                   tile_group=self._arr("tile_group", NT).cpu().numpy(),
                   tile_row0=self._arr("tile_row0", NT).cpu().numpy(),
                   tile_keyn=self._arr("tile_keyn", NT).cpu().numpy(),
                   n_stiles=NS, n_ltiles=NL,
                   stile_row0=self._arr("stile_row0", NS).cpu().numpy(),
                   stile_keyn=self._arr("stile_keyn", NS).cpu().numpy(),
                   ltile_row0=self._arr("ltile_row0", NL).cpu().numpy(),
                   ltile_keyn=self._arr("ltile_keyn", NL).cpu().numpy(),
                   ltile_tok0=self._arr("ltile_tok0", NL).cpu().numpy())
        return out


def dense_desc(case, lm_head: bool = False) -> L.PoolDesc:
    d = L.PoolDesc()
    d.max_loras, d.max_rank, d.in_dim = case.L, case.R, case.H
    d.n_slices = case.n_slices
    for j, o in enumerate(case.out_dims):
        d.out_dims[j] = o
    d.is_lm_head = int(lm_head)
    return d


def moe_desc(case) -> L.PoolDesc:
    d = L.PoolDesc()
    d.max_loras, d.max_rank = case.L, case.R
    d.num_experts, d.d_model, d.d_mlp = case.E, case.D, case.F
    d.n_w13_slices, d.w13_slice_width, d.shared_outer = case.n13, case.F13, int(case.shared_outer)
    return d


def upload_dense_slot(pool, case, a, stream=None):
    r = int(case.ranks[a])
    A = [np.ascontiguousarray(case.A[j][a, :r, :]) for j in range(case.n_slices)]
    B = [np.ascontiguousarray(case.B[j][a, :, :r]) for j in range(case.n_slices)]
    L.lora_set(pool, a, r, float(case.scales[a]), A, B, stream)
    return A, B


def upload_moe_slot(pool, case, a, stream=None):
    r = int(case.ranks[a])
    A = [np.ascontiguousarray(x[a][:, :r, :]) for x in case.A13] + [np.ascontiguousarray(case.A2[a][:, :r, :])]
    B = [np.ascontiguousarray(x[a][:, :, :r]) for x in case.B13] + [np.ascontiguousarray(case.B2[a][:, :, :r])]
    ae = [x.shape[1] for x in case.A13] + [case.A2.shape[1]]
    be = [x.shape[1] for x in case.B13] + [case.B2.shape[1]]
    L.lora_set_moe(pool, a, r, float(case.scales[a]), A, ae, B, be, stream)
    return A, B


class DenseRun:
    """A dense case resident on the GPU: pool, x, y, idx, meta, workspace."""

    def __init__(self, case, device="cuda", lm_head=False, max_rows=None, x_pad=0, y_pad=0):
        self.case = case
        self.pool = L.lora_pool_create(dense_desc(case, lm_head))
        for a in range(case.L):
            if case.ranks[a] > 0 and case.enabled[a]:
                upload_dense_slot(self.pool, case, a)
        # rows of x and y may be wider than the layer (leading dimensions
        # ldx = H + x_pad, ldy = out_total + y_pad)
        self.ldx = case.H + x_pad
        self.ldy = case.out_total + y_pad
        self.x = to_dev_u16_padded(case.x, x_pad, device)
        self.y = to_dev_u16_padded(case.y0, y_pad, device)
        self.idx = torch.from_numpy(case.idx).to(device)
        T = max_rows if max_rows is not None else case.T
        self.mb = MetaBuffer(max(T, 1), case.L, device)
        self.ws_bytes = L.lora_workspace_bytes(self.pool, max(T, 1), 1)
        self.ws = torch.zeros(max(self.ws_bytes, 16), dtype=torch.uint8, device=device)

    def build_meta(self, T=None):
        T = self.case.T if T is None else T
        L.lora_build_meta(self.pool, self.idx, T, None, 1, self.mb.meta)

    def apply(self):
        L.lora_apply_slices(self.pool, self.mb.meta, self.x, self.ldx, self.y, self.ldy, self.ws,
                            self.ws_bytes)

    def step(self):
        self.build_meta()
        self.apply()

    def step_batch(self, T=None):
        """The same step through the single call that builds the metadata and
        applies the layer (lora_build_meta_apply)."""
        T = self.case.T if T is None else T
        L.lora_build_meta_apply(self.pool, self.idx, T, self.mb.meta, self.x, self.ldx, self.y, self.ldy, self.ws,
                                self.ws_bytes)

    def y_full_host(self) -> np.ndarray:
        """All ldy columns of y, padding included."""
        return from_dev_u16(self.y)

    def y_host(self) -> np.ndarray:
        return np.ascontiguousarray(self.y_full_host()[:, :self.case.out_total])

    def status(self) -> int:
        return L.lora_get_device_status(self.pool)

    def close(self):
        if self.pool:
            L.lora_pool_destroy(self.pool)
            self.pool = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MoERun:
    """A MoE case resident on the GPU."""

    def __init__(self, case, device="cuda", in_pad=0, out_pad=0):
        self.case = case
        self.pool = L.lora_pool_create(moe_desc(case))
        for a in range(case.L):
            if case.ranks[a] > 0 and case.enabled[a]:
                upload_moe_slot(self.pool, case, a)
        # rows of the inputs (x, ic2) and outputs (ic1, ic3) may be wider than
        # the layer: ld_in = width + in_pad, ld_out = width + out_pad
        self.in_pad, self.out_pad = in_pad, out_pad
        self.x = to_dev_u16_padded(case.x, in_pad, device)
        self.ic2 = to_dev_u16_padded(case.ic2, in_pad, device)
        self.ic1 = to_dev_u16_padded(case.ic1_0, out_pad, device)
        self.ic3 = to_dev_u16_padded(case.ic3_0, out_pad, device)
        self.idx = torch.from_numpy(case.idx).to(device)
        self.topk = torch.from_numpy(np.ascontiguousarray(case.topk_ids)).to(device)
        self.topk_w = torch.from_numpy(np.ascontiguousarray(case.topk_w).reshape(-1)).to(device)
        rows = case.T * case.K
        self.mb = MetaBuffer(max(rows, 1), case.L * case.E, device)
        self.ws_bytes = L.lora_workspace_bytes(self.pool, max(case.T, 1), case.K)
        self.ws = torch.zeros(max(self.ws_bytes, 16), dtype=torch.uint8, device=device)

    def build_meta(self):
        c = self.case
        L.lora_build_meta(self.pool, self.idx, c.T, self.topk, c.K, self.mb.meta)

    def w13(self):
        c = self.case
        L.lora_moe_apply(self.pool, self.mb.meta, L.MOE_W13, self.x, c.D + self.in_pad, None, self.ic1,
                         c.n13 * c.F13 + self.out_pad, self.ws, self.ws_bytes)

    def w2(self):
        c = self.case
        L.lora_moe_apply(self.pool, self.mb.meta, L.MOE_W2, self.ic2, c.F + self.in_pad, self.topk_w, self.ic3,
                         c.D + self.out_pad, self.ws, self.ws_bytes)

    def ic1_host(self) -> np.ndarray:
        return np.ascontiguousarray(from_dev_u16(self.ic1)[:, :self.case.n13 * self.case.F13])

    def ic3_host(self) -> np.ndarray:
        return np.ascontiguousarray(from_dev_u16(self.ic3)[:, :self.case.D])

    def step(self):
        self.build_meta()
        self.w13()
        self.w2()

    def status(self) -> int:
        return L.lora_get_device_status(self.pool)

    def close(self):
        if self.pool:
            L.lora_pool_destroy(self.pool)
            self.pool = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class SinkRun:
    """An Inkling sink-expert case on the GPU: the w13 and w2 pools, one batch
    metadata (built against the w13 pool: both pools hold the same slots),
    base gate_up, gammas, h and the w2 output."""

    def __init__(self, case, device="cuda"):
        self.case = case
        self.r13 = DenseRun(case.w13, device=device)
        self.r2 = DenseRun(case.w2, device=device)
        W = case.n_experts * case.d_mlp
        self.W = W
        self.gammas = torch.from_numpy(case.gammas).to(device)
        self.h = torch.zeros((case.T, W), dtype=torch.int16, device=device)

    def build_meta(self):
        self.r13.build_meta()

    def apply(self):
        c = self.case
        m = self.r13.mb.meta
        L.lora_apply_slices(self.r13.pool, m, self.r13.x, c.w13.H, self.r13.y, 2 * self.W, self.r13.ws,
                            self.r13.ws_bytes)
        L.lora_sink_experts_act(self.r13.y, 2 * self.W, self.gammas, c.n_experts, c.T, c.n_experts, c.d_mlp,
                                self.h, self.W)
        L.lora_apply_slices(self.r2.pool, m, self.h, self.W, self.r2.y, c.w2.out_total,
                            self.r2.ws, self.r2.ws_bytes)

    def step(self):
        self.build_meta()
        self.apply()

    def status(self) -> int:
        return self.r13.status() | self.r2.status()

    def close(self):
        self.r13.close()
        self.r2.close()


class LinearRun(DenseRun):
    """A dense case with its base weight and bias on the GPU: the full LoRA
    linear layer y = x W^T + bias + delta."""

    def __init__(self, case, bias=None, device="cuda"):
        super().__init__(case, device=device)
        self.W = to_dev_u16(case.W, device)
        self.bias = to_dev_u16(bias, device) if bias is not None else None

    def apply(self):
        c = self.case
        L.lora_linear_apply(self.pool, self.mb.meta, self.x, c.H, self.W, c.H, self.bias, self.y, c.out_total,
                            self.ws, self.ws_bytes)
