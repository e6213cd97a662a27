"""Joint-layout forward, stacks of blocks and their CUDA graph, against the fp64 oracle.

A stack applies blocks in turn to the joint [text; image] sequence, in place, each with
its own weights and mod_bias on the shared timestep modulation. The graph replays the
same launches, so its output must equal the eagerly launched stack bit for bit.

Stack criterion: each block of the path stores its output in the storage dtype, and the
oracle chain with the path's storage rounding (``ref_st``) does the same. A stored output
may land one ulp away from the chain's rounding when its pre-rounding value sits next to a
rounding boundary, and the next block carries that difference through its residual, so
the bound is TOL * RMS(ref) + n_blocks * ulp * |ref|_i. The exact chain's max-abs / RMS is
reported beside it.
"""
import numpy as np
import pytest
import torch

import dit_inputs as di
import oracle
from diffusion_transformer_block_gb300 import KREA_DIT_ERR_INVALID_ARG, KreaDitError
from gpu_helpers import TOL, UNIT_ROUNDOFF, excess, make_block, path_storage, rel_max_err, upload

pytestmark = pytest.mark.gpu

WKEYS = ("w_qkvg", "w_o", "w_gate", "w_up", "w_down", "norm1_w", "norm2_w", "q_norm_w", "k_norm_w", "mod_bias")


def _joint_dev(case, dev):
    return torch.cat([case.dev["x_txt"], case.dev["x_img"]], dim=1).to(dev).contiguous()


def _setup(cfg, n_blocks, x_scale=1.0):
    blocks = di.make_stack(cfg, n_blocks, x_scale=x_scale)
    blk = make_block(cfg)
    t, _, _ = upload(blk, blocks[0])
    ms = blk.timestep_embed(t)
    sw = blk.stack_weights([{k: c.dev[k] for k in WKEYS} for c in blocks])
    x0 = _joint_dev(blocks[0], blk.device)
    return blocks, blk, ms, sw, x0


@pytest.mark.parametrize("name", ["small_a", "tiny", "small_imgonly", "small_txtonly"])
def test_joint_forward_equals_split_forward(name):
    cfg = di.CONFIGS[name]
    case = di.make_case(cfg)
    blk = make_block(cfg)
    try:
        t, x_img, x_txt = upload(blk, case)
        ms = blk.timestep_embed(t)
        ref = blk.forward(x_img, x_txt, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms)
        x = _joint_dev(case, blk.device)
        out = blk.forward_joint(x, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms)
        xin = x.clone()
        blk.forward_joint(xin, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, out=xin)  # in place
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        assert torch.equal(xin, ref)
    finally:
        blk.close()


# x_scale 0.05 shrinks the input so that the blocks' updates dominate the output
@pytest.mark.parametrize("name,n_blocks,gate_on,x_scale", [("small_a", 3, True, 1.0), ("small_b", 2, False, 1.0),
                                                           ("tiny", 2, True, 1.0), ("small_a", 3, True, 0.05),
                                                           ("small_c", 2, True, 0.05)])
def test_stack_graph_matches_eager_and_oracle(name, n_blocks, gate_on, x_scale):
    cfg = di.CONFIGS[name].replace(gate_on=gate_on)
    blocks, blk, ms, sw, x0 = _setup(cfg, n_blocks, x_scale)
    stream = torch.cuda.Stream(blk.device)
    graph = None
    try:
        x_eager = x0.clone()
        blk.stack_forward(x_eager, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, sw)
        torch.cuda.synchronize()
        xg = x0.clone()
        graph = blk.stack_graph(xg, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, sw, stream)
        torch.cuda.synchronize()
        assert torch.equal(xg, x0), "capturing must not run the stack"
        graph.launch(stream)
        stream.synchronize()
        assert torch.equal(xg, x_eager)

        msn = ms.double().cpu().numpy()
        ws = [c.w for c in blocks]
        ref = oracle.run_stack(blocks[0], ws, mod_shared=msn)
        ref_st = oracle.run_stack(blocks[0], ws, mod_shared=msn, store=path_storage(cfg.dtype))
        got = x_eager.double().cpu().numpy()
        tol, ulp = TOL[cfg.dtype], 2 * UNIT_ROUNDOFF[cfg.dtype]
        lit = rel_max_err([got], [ref])
        ex = excess([got], [ref_st], tol, n_blocks * ulp)
        assert ex <= 1.0, f"{name}: stack excess {ex:.3f} (exact-chain max-abs/RMS {lit:.4f})"
        # the stack really moved the sequence (the blocks are not identities)
        assert rel_max_err([x0.double().cpu().numpy()], [ref]) > 2 * tol
    finally:
        if graph is not None:
            graph.close()
        blk.close()


def test_graph_relaunch_applies_the_stack_again():
    cfg = di.CONFIGS["small_a"]
    blocks, blk, ms, sw, x0 = _setup(cfg, 2)
    stream = torch.cuda.Stream(blk.device)
    graph = None
    try:
        twice = x0.clone()
        for _ in range(2):
            blk.stack_forward(twice, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, sw)
        xg = x0.clone()
        torch.cuda.synchronize()
        graph = blk.stack_graph(xg, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, sw, stream)
        graph.launch(stream)
        graph.launch(stream)
        stream.synchronize()
        assert torch.equal(xg, twice)
        # new contents of the captured buffer are picked up by the next launch
        with torch.cuda.stream(stream):
            xg.copy_(x0)
        graph.launch(stream)
        stream.synchronize()
        once = x0.clone()
        blk.stack_forward(once, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, sw)
        torch.cuda.synchronize()
        assert torch.equal(xg, once)
    finally:
        if graph is not None:
            graph.close()
        blk.close()


def test_graph_arguments_are_checked():
    cfg = di.CONFIGS["small_a"]
    blocks, blk, ms, sw, x0 = _setup(cfg, 1)
    stream = torch.cuda.Stream(blk.device)
    try:
        with pytest.raises(KreaDitError) as e:
            blk.stack_graph(x0, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, sw, 0)  # legacy default stream
        assert e.value.status == KREA_DIT_ERR_INVALID_ARG
        with pytest.raises(KreaDitError) as e:  # a shape error surfaces from the capture
            blk.stack_graph(x0, cfg.B + 1, cfg.img_h, cfg.img_w, cfg.n_txt, ms, sw, stream)
        assert e.value.status != 0
        # an empty stack is a graph that leaves x alone
        empty = blk.stack_weights([])
        x = x0.clone()
        g = blk.stack_graph(x, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, empty, stream)
        g.launch(stream)
        stream.synchronize()
        g.close()
        assert torch.equal(x, x0)
        # the handle still works after the failed captures
        y = x0.clone()
        blk.stack_forward(y, cfg.B, cfg.img_h, cfg.img_w, cfg.n_txt, ms, sw)
        torch.cuda.synchronize()
        assert not torch.equal(y, x0)
    finally:
        blk.close()
