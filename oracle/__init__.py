"""fp64 CPU oracle of the Krea 2 single-stream DiT block forward.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the benchmark's CPU-baseline leg, never by the library. It shares no code
with the CUDA path. Parity pins: every function here is pinned by the CPU tests
(textbook library routines, closed forms, invariants, brute force on tiny
inputs); none is "parity unpinned". ``oracle.gemm8`` adds the block with 8-bit
(e4m3, scaled) GEMM operands, pinned in ``tests/test_oracle_gemm8.py``; ``oracle.backward``
the analytic gradients of the block, pinned in ``tests/test_oracle_backward.py``;
``oracle.nvfp4`` the block with NVFP4 GEMM operands (E2M1 elements, E4M3 scales per 16
elements, a power-of-two tensor scale), pinned in ``tests/test_oracle_nvfp4.py``.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np

from .block import (  # noqa: F401
    apply_rope_2d,
    block_forward,
    gqa_attention,
    modulation,
    round_to_bf16,
    rms_norm,
    rope_angles,
    stack_forward,
    swiglu,
    timestep_embedding,
    timestep_mlp,
    token_positions,
    zero_centred_rms_norm,
)


def mod_shared_for(case) -> np.ndarray:
    """Timestep -> sinusoid -> shared MLP -> mod_shared [B, 6, d] for a seeded case."""
    e = timestep_embedding(case.t)
    return timestep_mlp(e, case.temb["w1"], case.temb["b1"], case.temb["w2"], case.temb["b2"])


def run_case(case, rows: Optional[Sequence[np.ndarray]] = None, *, rope_on: bool = True,
             mod_shared: Optional[np.ndarray] = None, store=None) -> Dict[str, list]:
    """Timestep embedding plus one block forward for a seeded case (duck-typed:
    ``case.cfg`` shapes, ``case.t``, ``case.temb``, ``case.w``, ``case.x_txt``,
    ``case.x_img``)."""
    cfg = case.cfg
    ms = mod_shared_for(case) if mod_shared is None else mod_shared
    return block_forward(
        case.x_txt, case.x_img, (cfg.img_h, cfg.img_w), ms, case.w,
        n_q=cfg.n_q, n_kv=cfg.n_kv, hd=cfg.hd, eps=cfg.eps, rope_base=cfg.rope_base,
        gate_on=cfg.gate_on, rope_on=rope_on, rows=rows, store=store,
    )


def run_stack(case, blocks, *, mod_shared: Optional[np.ndarray] = None, store=None) -> np.ndarray:
    """Timestep embedding plus a stack of blocks for a seeded case; ``blocks`` is a list of
    weight dicts (block 0's is normally ``case.w``). Returns the final joint output."""
    cfg = case.cfg
    ms = mod_shared_for(case) if mod_shared is None else mod_shared
    return stack_forward(
        case.x_txt, case.x_img, (cfg.img_h, cfg.img_w), ms, blocks,
        n_q=cfg.n_q, n_kv=cfg.n_kv, hd=cfg.hd, eps=cfg.eps, rope_base=cfg.rope_base,
        gate_on=cfg.gate_on, store=store,
    )
