"""A resident stack of ternary projections: packed planes in HBM plus one
contiguous arena for each of the step's inputs and outputs, so that a batch-1
decode step is one launch (every activation row quantised and every product
computed by the fused kernel; the two-launch path -- quantise, then multiply --
stays available) and an end-to-end step is one host-to-device and one
device-to-host copy around it.

This is the runtime around the kernels for the layer-by-layer decode of
"Tritium: One Weight Format for Ternary Inference ..." -- Why it does not
scale: a token is 210 independent ternary products; here they are issued as
one persistent launch instead of 210 separate dispatches.
"""
from __future__ import annotations

import torch

from . import (MAX_FUSED_K, ActList, ProjList, QProjList, k_pad, payload_bytes,
               trit_gemm_many, trit_pack, trit_quant_act_many, trit_quant_gemv_many)


class TernaryStack:
    def __init__(self, device="cuda"):
        self.device = torch.device(device)
        self.specs = []        # (name, N, K, M, w_scale)
        self.planes = []
        self.finalized = False

    def add(self, w: torch.Tensor, w_scale: float, M: int = 1, name: str = "") -> int:
        """Pack an int8 ternary matrix [N, K] (host or device) and reserve M
        activation rows for it.  Returns its index."""
        assert not self.finalized
        N, K = w.shape
        wd = w.to(self.device, non_blocking=False)
        planes, err = trit_pack(wd, w_scale)
        torch.cuda.current_stream(self.device).synchronize()
        if int(err.item()) != 0:
            raise ValueError(f"projection {name or len(self.specs)}: non-ternary weights")
        del wd
        self.planes.append(planes)
        self.specs.append((name, N, K, M, float(w_scale)))
        return len(self.specs) - 1

    def twin(self) -> "TernaryStack":
        """A finalized stack over the same planes with arenas of its own: two
        twins let consecutive steps use different activation and output
        buffers, so a step's copies can overlap the next step's products."""
        assert self.finalized
        t = TernaryStack.__new__(TernaryStack)
        t.device = self.device
        t.specs = list(self.specs)
        t.planes = self.planes
        t.finalized = False
        t.finalize()
        return t

    def finalize(self):
        """Allocate the arenas and build the launch lists."""
        dev = self.device
        x_el = sum(M * K for _, N, K, M, _ in self.specs)
        q_el = sum(M * k_pad(K) for _, N, K, M, _ in self.specs)
        m_el = sum(M for _, N, K, M, _ in self.specs)
        y_el = sum(M * N for _, N, K, M, _ in self.specs)
        self.x_arena = torch.zeros(x_el, dtype=torch.float32, device=dev)
        self.q_arena = torch.zeros(q_el + 64, dtype=torch.int8, device=dev)
        self.s_arena = torch.zeros(m_el, dtype=torch.float32, device=dev)
        self.y_arena = torch.zeros(y_el, dtype=torch.int32, device=dev)
        self.f_arena = torch.zeros(y_el, dtype=torch.float32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.x, self.q, self.s, self.y, self.f = [], [], [], [], []
        xo = qo = so = yo = 0
        for _, N, K, M, _ in self.specs:
            self.x.append(self.x_arena[xo:xo + M * K].view(M, K))
            self.q.append(self.q_arena[qo:qo + M * k_pad(K)].view(M, k_pad(K)))
            self.s.append(self.s_arena[so:so + M])
            self.y.append(self.y_arena[yo:yo + M * N].view(M, N))
            self.f.append(self.f_arena[yo:yo + M * N].view(M, N))
            xo += M * K
            qo += M * k_pad(K)   # multiple of 64 bytes: every row stays 16-byte aligned
            so += M
            yo += M * N
        self.acts = ActList([(self.x[i], self.q[i], self.s[i]) for i in range(len(self.specs))])
        self.projs = ProjList([(self.planes[i], self.specs[i][4], self.q[i], self.s[i],
                                self.specs[i][2], self.y[i], self.f[i])
                               for i in range(len(self.specs))])
        self.fusable = all(M == 1 and K <= MAX_FUSED_K for _, N, K, M, _ in self.specs)
        self.qprojs = None
        if self.fusable:
            self.qprojs = QProjList([(self.planes[i], self.specs[i][4], self.x[i], self.q[i],
                                      self.s[i], self.y[i], self.f[i])
                                     for i in range(len(self.specs))])
        self.finalized = True

    # -- one decode step ------------------------------------------------------

    def quantize(self, stream=None):
        trit_quant_act_many(self.acts, self.err, stream)

    def products(self, stream=None):
        trit_gemm_many(self.projs, self.err, stream)

    def fused(self, stream=None):
        """Quantise and multiply every entry in one launch (M = 1 stacks)."""
        trit_quant_gemv_many(self.qprojs, self.err, stream)

    def step(self, stream=None):
        if self.fusable:
            self.fused(stream)
        else:
            self.quantize(stream)
            self.products(stream)

    def step_two_launch(self, stream=None):
        self.quantize(stream)
        self.products(stream)

    # -- sizes ------------------------------------------------------------------

    @property
    def plane_bytes(self) -> int:
        return sum(payload_bytes(N, K) for _, N, K, M, _ in self.specs)

    @property
    def weights(self) -> int:
        return sum(N * K for _, N, K, M, _ in self.specs)

    def product_bytes(self) -> int:
        """Algorithmic bytes of the product launch: every plane byte read once,
        the int8 activations (K_pad per row) and their scales read, y_i32 and
        y_f32 written."""
        b = 0
        for _, N, K, M, _ in self.specs:
            b += payload_bytes(N, K) + M * k_pad(K) + 4 * M + 8 * M * N
        return b

    def fused_bytes(self) -> int:
        """Algorithmic bytes of the fused launch: planes read once, the fp32
        activations read, int8 codes (K_pad per row) and scales written, y_i32
        and y_f32 written."""
        b = 0
        for _, N, K, M, _ in self.specs:
            b += payload_bytes(N, K) + M * (4 * K + k_pad(K) + 4) + 8 * M * N
        return b

    def quant_bytes(self) -> int:
        """fp32 activations read, int8 codes (K_pad per row) and scales written."""
        return sum(M * (4 * K + k_pad(K) + 4) for _, N, K, M, _ in self.specs)
