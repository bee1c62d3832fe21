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


class LayerChain:
    """The dependency-ordered decode of one token through ternary layers: per
    layer four launches, each reading what the one before wrote --
      1. q, k, v from the layer's input row (quantiser fused),
      2. o from q's fp32 output (the attention output's stand-in: attention
         itself is not a ternary product),
      3. gate and up from o's fp32 output (gate also writes the input scale),
      4. the IntMlp codes of relu(a_gate)^2 a_up and the down product.
    This is the per-matvec ordering of a real token ("Tritium ..." -- Why it
    does not scale): every launch waits for the grid before it (programmatic
    stream serialisation) before it reads its input.  Each layer's input row is
    its own buffer (x[layer]); the residual stream and the norms are not part
    of the ternary path.

    weights: per layer, a dict name -> (int8 [N, K] tensor, w_scale) for the
    seven projections q, k, v, o, gate, up, down.

    mlp_form -- the same bits every way:
      "paired": gate/up as one launch that also publishes max|t| partials
        (trit_mlp_gate_up), then the down product forming the IntMlp codes from
        them while it stages its row (trit_mlp_down): 4 launches per layer;
      "split": gate/up, trit_intmlp_quant, the down product of its int8 codes: 5;
      "fused": gate/up, then every CTA of the down product forms the codes it
        needs, max|t| pass included (trit_intmlp_gemv_many): 4."""

    NAMES = ("q", "k", "v", "o", "gate", "up", "down")
    MLP_FORMS = ("paired", "split", "fused")

    def __init__(self, weights, device="cuda", mlp_form: str = "paired"):
        from . import MlpBlockList, MlpProjList, trit_mlp_tmax_bytes
        if mlp_form not in self.MLP_FORMS:
            raise ValueError(f"mlp_form must be one of {self.MLP_FORMS}")
        self.mlp_form = mlp_form
        self.device = torch.device(device)
        dev = self.device
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.layers = []
        self.plane_bytes = 0
        for lw in weights:
            P, S, shape = {}, {}, {}
            for name in self.NAMES:
                w, ws = lw[name]
                planes, err = trit_pack(w.to(dev), ws)
                if int(err.item()) != 0:
                    raise ValueError(f"{name}: non-ternary weights")
                P[name], S[name], shape[name] = planes, float(ws), tuple(w.shape)
                self.plane_bytes += planes.numel()
            Nq, K = shape["q"]
            Nk, Nv = shape["k"][0], shape["v"][0]
            No, Ko = shape["o"]
            Nf, Kg = shape["gate"]
            Nd, Kd = shape["down"]
            if Ko != Nq or Kg != No or Kd != Nf or shape["up"] != shape["gate"]:
                raise ValueError("layer shapes do not chain")
            L = {"P": P, "S": S}
            L["x"] = torch.zeros(K, dtype=torch.float32, device=dev)
            for name, n in (("q", Nq), ("k", Nk), ("v", Nv), ("o", No), ("down", Nd)):
                L["y_" + name] = torch.zeros(n, dtype=torch.int32, device=dev)
                L["f_" + name] = torch.zeros(n, dtype=torch.float32, device=dev)
            L["a_gate"] = torch.zeros(Nf, dtype=torch.int32, device=dev)
            L["a_up"] = torch.zeros(Nf, dtype=torch.int32, device=dev)
            L["s_gu"] = torch.zeros(1, dtype=torch.float32, device=dev)
            # the planes are packed (and the stream synchronised) here, before any
            # launch of the chain: every list may read them ahead of its grid dependency
            L["qkv"] = QProjList([(P[n], S[n], L["x"], None, None, L["y_" + n], L["f_" + n])
                                  for n in ("q", "k", "v")], planes_ready=True)
            L["o"] = QProjList([(P["o"], S["o"], L["f_q"], None, None, L["y_o"], L["f_o"])],
                               planes_ready=True)
            L["gu"] = QProjList([(P["gate"], S["gate"], L["f_o"], None, L["s_gu"], L["a_gate"], None),
                                 (P["up"], S["up"], L["f_o"], None, None, L["a_up"], None)],
                                planes_ready=True)
            L["down"] = MlpProjList([(P["down"], S["down"], L["a_gate"], L["a_up"], L["s_gu"],
                                      S["gate"], S["up"], None, None, L["y_down"], L["f_down"])])
            L["h"] = torch.zeros(k_pad(Kd), dtype=torch.int8, device=dev)
            L["s_h"] = torch.zeros(1, dtype=torch.float32, device=dev)
            L["down_i8"] = ProjList([(P["down"], S["down"], L["h"], L["s_h"], Kd, L["y_down"],
                                      L["f_down"])], planes_ready=True)
            L["tmax"] = torch.zeros(trit_mlp_tmax_bytes(Nf), dtype=torch.uint8, device=dev)
            L["mlp"] = MlpBlockList([(P["gate"], P["up"], P["down"], S["gate"], S["up"], S["down"],
                                      L["f_o"], L["s_gu"], L["a_gate"], L["a_up"], L["tmax"], None,
                                      None, L["y_down"], L["f_down"])], planes_ready=True)
            self.layers.append(L)

    @property
    def x(self):
        return [L["x"] for L in self.layers]

    def step(self, stream=None):
        """One token through every layer: 4 launches per layer (5 for "split")."""
        from . import trit_intmlp_gemv_many, trit_intmlp_quant, trit_mlp_down, trit_mlp_gate_up
        for L in self.layers:
            trit_quant_gemv_many(L["qkv"], self.err, stream)
            trit_quant_gemv_many(L["o"], self.err, stream)
            if self.mlp_form == "paired":
                trit_mlp_gate_up(L["mlp"], self.err, stream)
                trit_mlp_down(L["mlp"], self.err, stream)
                continue
            trit_quant_gemv_many(L["gu"], self.err, stream)
            if self.mlp_form == "fused":
                trit_intmlp_gemv_many(L["down"], self.err, stream)
            else:
                S = L["S"]
                trit_intmlp_quant(L["a_gate"][None, :], L["a_up"][None, :], S["gate"], S["up"],
                                  L["s_gu"], L["h"][None, :], L["s_h"], stream)
                trit_gemm_many(L["down_i8"], self.err, stream)

    @property
    def stages_per_step(self) -> int:
        return 4 * len(self.layers)

    @property
    def launches_per_step(self) -> int:
        return (5 if self.mlp_form == "split" else 4) * len(self.layers)

    def step_bytes(self) -> int:
        """Algorithmic bytes of one token: every plane byte read once; per
        launch its fp32 (or int32) inputs read and int32 + fp32 outputs written."""
        b = self.plane_bytes
        for L in self.layers:
            K = L["x"].numel()
            nq, nk, nv = (L["y_" + n].numel() for n in ("q", "k", "v"))
            no, nf, nd = L["y_o"].numel(), L["a_gate"].numel(), L["y_down"].numel()
            b += 4 * K + 8 * (nq + nk + nv)          # qkv: x read, y + f written
            b += 4 * nq + 8 * no                     # o: q's f read
            b += 4 * no + 4 + 8 * nf                 # gate/up: o's f read, scale, a_gate + a_up
            b += 8 * nf + 4 + 8 * nd                 # down: a_gate + a_up read, scale
        return b
