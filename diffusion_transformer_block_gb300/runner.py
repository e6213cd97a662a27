"""Convenience owner of one library handle plus the caller-side device tensors.

Marshalling only: torch allocates device memory and supplies streams; every step of
the block runs in libkrea_dit.so. Used by the tests, the benchmark and the smoke check.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import torch

from . import (KREA_DIT_BF16, KREA_DIT_FP32, KREA_DIT_FP8_ROW, KREA_DIT_FP8_TENSOR, KREA_DIT_NVFP4,
               krea_dit_block_backward, krea_dit_block_create, krea_dit_block_destroy,
               krea_dit_block_enable_backward, krea_dit_block_forward, krea_dit_block_forward4,
               krea_dit_block_forward8, krea_dit_block_forward_joint, krea_dit_block_workspace,
               krea_dit_graph_destroy, krea_dit_graph_launch, krea_dit_nvfp4_scale_bytes, krea_dit_stack_forward,
               krea_dit_stack_graph_create, krea_dit_timestep_embed, krea_dit_weights4_quantize,
               krea_dit_weights8_quantize, make_config, make_grads, make_temb_weights, make_weights, make_weights4,
               make_weights8)

WEIGHT_KEYS = ("w_qkvg", "w_o", "w_gate", "w_up", "w_down", "norm1_w", "norm2_w", "q_norm_w", "k_norm_w",
               "mod_bias")
TEMB_KEYS = ("w1", "b1", "w2", "b2")
MATRIX_KEYS = ("w_qkvg", "w_o", "w_gate", "w_up", "w_down")
MODES = {"bf16": KREA_DIT_BF16, "fp32": KREA_DIT_FP32, "fp8_tensor": KREA_DIT_FP8_TENSOR, "fp8_row": KREA_DIT_FP8_ROW,
         "nvfp4": KREA_DIT_NVFP4}


class _DevView:
    """Exposes a raw device range through __cuda_array_interface__ for torch.as_tensor."""

    def __init__(self, ptr: int, shape: Sequence[int], typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


class DitBlock:
    """One block handle. ``mode`` is "bf16", "fp32" (the storage / arithmetic mode) or
    "fp8_tensor" / "fp8_row" (bf16 storage, 8-bit GEMMs with tensor-wise / row-wise scales) or "nvfp4"
    (bf16 storage, NVFP4 GEMMs)."""

    def __init__(self, *, max_batch: int, max_seq: int, d: int, n_q: int, n_kv: int, hd: int, F: int,
                 img_h_max: int, img_w_max: int, gate_on: bool = True, mode: str = "bf16", eps: float = 1e-6,
                 rope_base: float = 10000.0, device: str = "cuda:0"):
        self.device = torch.device(device)
        self.mode = mode
        self.mode8 = mode.startswith("fp8")
        self.mode4 = mode == "nvfp4"
        self.dtype = torch.float32 if mode == "fp32" else torch.bfloat16
        self.dims = dict(d=d, n_q=n_q, n_kv=n_kv, hd=hd, F=F, gate_on=gate_on)
        cfg = make_config(max_batch=max_batch, max_seq=max_seq, d_model=d, n_q=n_q, n_kv=n_kv, head_dim=hd, ffn=F,
                          img_h_max=img_h_max, img_w_max=img_w_max, eps=eps, rope_base=rope_base, gate_on=gate_on,
                          mode=MODES[mode])
        with torch.cuda.device(self.device):
            self.handle = krea_dit_block_create(cfg)
        self.w: Dict[str, torch.Tensor] = {}
        self.tw: Dict[str, torch.Tensor] = {}
        self._wstruct = None
        self._twstruct = None
        self.w8: Dict[str, torch.Tensor] = {}
        self._w8struct = None
        self.w4: Dict[str, torch.Tensor] = {}
        self._w4struct = None

    def set_weights(self, w: Dict[str, torch.Tensor], stream=None) -> None:
        """Uploads the weights; in an 8-bit mode also casts the matrices to e4m3 codes."""
        self.w = {k: w[k].to(self.device).contiguous() for k in WEIGHT_KEYS}
        self._wstruct = make_weights(self.w)
        if self.mode8:
            per_row = self.mode == "fp8_row"
            w8: Dict[str, torch.Tensor] = {}
            for k in MATRIX_KEYS:
                m = self.w[k]
                w8[k] = torch.empty(m.shape, device=self.device, dtype=torch.uint8)
                w8["dq_" + k[2:]] = torch.empty(m.shape[0] if per_row else 1, device=self.device, dtype=torch.float32)
            self.w8 = w8
            self._w8struct = make_weights8(w8)
            krea_dit_weights8_quantize(self.handle, self._wstruct, self._w8struct,
                                       stream or torch.cuda.current_stream(self.device))
        if self.mode4:
            w4: Dict[str, torch.Tensor] = {}
            for k in MATRIX_KEYS:
                rows, cols = self.w[k].shape
                w4[k] = torch.empty(rows, cols // 2, device=self.device, dtype=torch.uint8)
                w4["sf_" + k[2:]] = torch.empty(krea_dit_nvfp4_scale_bytes(rows, cols), device=self.device,
                                                dtype=torch.uint8)
                w4["ts_" + k[2:]] = torch.empty(4, device=self.device, dtype=torch.float32)
            self.w4 = w4
            self._w4struct = make_weights4(w4)
            krea_dit_weights4_quantize(self.handle, self._wstruct, self._w4struct,
                                       stream or torch.cuda.current_stream(self.device))

    def set_temb_weights(self, tw: Dict[str, torch.Tensor]) -> None:
        self.tw = {k: tw[k].to(self.device, torch.float32).contiguous() for k in TEMB_KEYS}
        self._twstruct = make_temb_weights(self.tw)

    def timestep_embed(self, t: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        B = t.shape[0]
        if out is None:
            out = torch.empty(B, 6, self.dims["d"], device=self.device, dtype=torch.float32)
        krea_dit_timestep_embed(self.handle, t, B, self._twstruct, out, stream or torch.cuda.current_stream(self.device))
        return out

    def forward(self, x_img: Optional[torch.Tensor], x_txt: Optional[torch.Tensor], B: int, img_h: int, img_w: int,
                n_txt: int, t_emb: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        L = n_txt + img_h * img_w
        if out is None:
            out = torch.empty(B, L, self.dims["d"], device=self.device, dtype=self.dtype)
        xi = x_img if (x_img is not None and img_h * img_w > 0) else None
        xt = x_txt if (x_txt is not None and n_txt > 0) else None
        st = stream or torch.cuda.current_stream(self.device)
        if self.mode8:
            krea_dit_block_forward8(self.handle, xi, xt, B, img_h, img_w, n_txt, t_emb, self._wstruct, self._w8struct,
                                    out, st)
        elif self.mode4:
            krea_dit_block_forward4(self.handle, xi, xt, B, img_h, img_w, n_txt, t_emb, self._wstruct, self._w4struct,
                                    out, st)
        else:
            krea_dit_block_forward(self.handle, xi, xt, B, img_h, img_w, n_txt, t_emb, self._wstruct, out, st)
        return out

    def backward(self, x_img: Optional[torch.Tensor], x_txt: Optional[torch.Tensor], B: int, img_h: int, img_w: int,
                 n_txt: int, t_emb: torch.Tensor, d_out: torch.Tensor, stream=None) -> Dict[str, torch.Tensor]:
        """Gradients of the block (bf16 mode) for the upstream gradient d_out [B, L, d]:
        d_x_txt, d_x_img (bf16) and fp32 d_<weight>, d_mod_bias, d_mod_shared."""
        if not getattr(self, "_bw", False):
            krea_dit_block_enable_backward(self.handle)
            self._bw = True
        dev, d = self.device, self.dims["d"]
        n_img = img_h * img_w
        g: Dict[str, torch.Tensor] = {
            "d_x_txt": torch.empty(B, n_txt, d, device=dev, dtype=self.dtype),
            "d_x_img": torch.empty(B, n_img, d, device=dev, dtype=self.dtype),
            "d_mod_bias": torch.empty(6, d, device=dev, dtype=torch.float32),
            "d_mod_shared": torch.empty(B, 6, d, device=dev, dtype=torch.float32),
        }
        for k in WEIGHT_KEYS:
            if k != "mod_bias":
                g["d_" + k] = torch.empty(self.w[k].shape, device=dev, dtype=torch.float32)
        gs = make_grads({k: (v if v.numel() else None) for k, v in g.items()})
        xi = x_img if (x_img is not None and n_img > 0) else None
        xt = x_txt if (x_txt is not None and n_txt > 0) else None
        krea_dit_block_backward(self.handle, xi, xt, B, img_h, img_w, n_txt, t_emb, self._wstruct, d_out.contiguous(),
                                gs, stream or torch.cuda.current_stream(self.device))
        return g

    def forward_joint(self, x: torch.Tensor, B: int, img_h: int, img_w: int, n_txt: int, t_emb: torch.Tensor,
                      out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """One block on the joint [text; image] sequence x [B, L, d]; ``out`` may be x."""
        if out is None:
            out = torch.empty_like(x)
        krea_dit_block_forward_joint(self.handle, x, B, img_h, img_w, n_txt, t_emb, self._wstruct, out,
                                     stream or torch.cuda.current_stream(self.device))
        return out

    def stack_weights(self, blocks: Sequence[Dict[str, torch.Tensor]]) -> "StackWeights":
        """Device copies of per-block weight dicts, for stack_forward / stack_graph."""
        return StackWeights(blocks, self.device)

    def stack_forward(self, x: torch.Tensor, B: int, img_h: int, img_w: int, n_txt: int, t_emb: torch.Tensor,
                      sw: "StackWeights", stream=None) -> torch.Tensor:
        """Applies the blocks of ``sw`` in turn, in place on x [B, L, d]."""
        krea_dit_stack_forward(self.handle, x, B, img_h, img_w, n_txt, t_emb, sw.structs,
                               stream or torch.cuda.current_stream(self.device))
        return x

    def stack_graph(self, x: torch.Tensor, B: int, img_h: int, img_w: int, n_txt: int, t_emb: torch.Tensor,
                    sw: "StackWeights", stream: torch.cuda.Stream) -> "StackGraph":
        """Captures stack_forward with these buffers into a CUDA graph on ``stream``."""
        g = krea_dit_stack_graph_create(self.handle, x, B, img_h, img_w, n_txt, t_emb, sw.structs, stream)
        return StackGraph(g, (self, x, t_emb, sw))

    def workspace(self, name: str, shape: Sequence[int]) -> torch.Tensor:
        """Copy of a workspace buffer of the last forward, viewed with ``shape``
        (H1 and the DQ_* factors are fp32, the *8 e4m3 codes are returned as uint8, every
        other buffer is in the storage dtype)."""
        ptr, nbytes = krea_dit_block_workspace(self.handle, name)
        if name.startswith("TS_"):
            esz = 4
        elif name.endswith(("8", "4")) or name.startswith("SF_"):
            esz = 1
        elif name == "H1" or name.startswith("DQ_") or self.mode == "fp32":
            esz = 4
        else:
            esz = 2
        n = 1
        for s in shape:
            n *= s
        if n * esz > nbytes:
            raise ValueError(f"{name}: {n * esz} bytes requested, {nbytes} available")
        if n == 0:
            return torch.empty(tuple(shape), device=self.device, dtype=self.dtype)
        view = torch.as_tensor(_DevView(ptr, (n,), {1: "|u1", 2: "<i2", 4: "<f4"}[esz]), device=self.device)
        t = view.clone()
        if esz == 2:
            t = t.view(torch.bfloat16)
        return t.view(tuple(shape))

    def close(self) -> None:
        if getattr(self, "handle", None):
            krea_dit_block_destroy(self.handle)
            self.handle = None

    def __del__(self):  # pragma: no cover - best effort
        try:
            self.close()
        except Exception:
            pass


class StackWeights:
    """Device weights of a stack of blocks (one dict per block, keys as DitBlock.set_weights)."""

    def __init__(self, blocks: Sequence[Dict[str, torch.Tensor]], device: torch.device):
        self.tensors = [{k: w[k].to(device).contiguous() for k in WEIGHT_KEYS} for w in blocks]
        self.structs = [make_weights(w) for w in self.tensors]


class StackGraph:
    """An instantiated stack graph; keeps the buffers it was captured on alive."""

    def __init__(self, graph: int, keep):
        self.graph = graph
        self._keep = keep

    def launch(self, stream=None) -> None:
        krea_dit_graph_launch(self.graph, stream or torch.cuda.current_stream())

    def close(self) -> None:
        if self.graph:
            krea_dit_graph_destroy(self.graph)
            self.graph = None

    def __del__(self):  # pragma: no cover - best effort
        try:
            self.close()
        except Exception:
            pass
