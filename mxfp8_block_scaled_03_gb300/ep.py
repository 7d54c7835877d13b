"""Expert parallelism for the MoE layer around the fused MXFP8 expert MLP.

Each rank of a process group owns E / world consecutive experts (rank r: experts
r * E_loc .. (r + 1) * E_loc - 1) and holds only their quantized weights; tokens travel to the
ranks that own their experts and their outputs travel back (page "Efficient MoE training for
biological foundation models", How to run the recipe: the Mixtral-8x7B configuration spreads its
experts over eight GPUs, with the data- and expert-parallel sizes multiplying to the GPU count;
Key technical approaches item 1: tokens are gathered per expert and counted by split_sizes).
All ranks pass routing weights, or none does.

One forward, on every rank of the group:
  1. ``moe_permute`` of the rank's own (token, slot) choices over all E experts.  Because rank
     r's experts are consecutive ids, the sorted rows bound for one rank are one contiguous run.
  2. The per-expert counts travel with one all-to-all ([world, E_loc] int32 each way); their row
     sums become host split sizes (the one host synchronization of the layer: an all-to-all of
     variable sizes needs them on the host).
  3. The sorted token rows (gathered from x_tokens by ``moe_gather_rows``) and their routing
     weights go to their owners with one all-to-all each.
  4. The owner receives, from each source in turn, rows sorted by its local experts.  A stable
     ``moe_permute`` of the received rows by local expert (one slot each) gives the expert-major
     order, the local split sizes and the routing weights in that order; the fused forward
     (``grouped_mlp_fwd_tokens``) gathers the rows in that order inside its activation quantize.
  5. ``moe_gather_rows`` puts the outputs back in the order received, one all-to-all returns
     them to their sources, and ``moe_combine`` sums each token's k expert outputs (the routing
     weight was applied inside ScaledSwiGLU).

Training (``ep_moe_forward_train`` / ``ep_moe_backward``): the forward also saves the owner's
pre-activations and the routing of the call; the backward sends each sorted row's output
gradient (its token's row of d_out: the gradient of the combine) to the owner in the same way,
runs ``grouped_mlp_bwd_tokens`` there (this rank's experts' weight gradients stay on the rank),
and returns dx rows and routing-weight gradients along the forward's path in reverse; each
source sums its tokens' k dx rows (``moe_combine``, the gradient of the token gather) and picks
the routing-weight gradient of each (token, slot).

Every step that touches the rows runs in the library's kernels; the host only computes the
local expert id of each received row from the exchanged counts (world * E_loc numbers).  With
one rank the exchanges are copies and the results equal the single-GPU MoE layer bit for bit.

The compute steps are reached through an ``ops`` object so that the exchange logic can be run
with other implementations of the same operations (``KernelOps`` is the library's).
"""
from __future__ import annotations

import numpy as np


class KernelOps:
    """The compute steps of the layer on the library's CUDA kernels; expert outputs and input
    gradients are bf16 (``y_dtype``)."""

    def __init__(self, mx=None):
        import torch
        if mx is None:
            import mxfp8_block_scaled_03_gb300 as mx
        self.mx = mx
        self.y_dtype = torch.bfloat16
        self.dg_dtype = torch.float32

    def permute(self, experts, gates, E: int):
        split, row_of_slot, token_of_row, gates_sorted, _ = self.mx.moe_permute(experts, gates, E)
        return split, row_of_slot, token_of_row, gates_sorted

    def gather_rows(self, x, index):
        return self.mx.moe_gather_rows(x, index.reshape(-1))

    def expert_mlp(self, x_rows, token_of_row, split, gates_sorted, weights):
        return self.mx.grouped_mlp_fwd_tokens(x_rows, token_of_row, split, gates_sorted, *weights)

    def expert_mlp_train(self, x_rows, token_of_row, split, gates_sorted, weights):
        return self.mx.grouped_mlp_fwd_tokens_train(x_rows, token_of_row, split, gates_sorted, *weights)

    def expert_mlp_bwd(self, x_rows, token_of_row, split, gates_sorted, saved, weights_t, dy_rows):
        dx, dg, dw1, dw2, _ = self.mx.grouped_mlp_bwd_tokens(x_rows, token_of_row, split, gates_sorted, saved,
                                                             *weights_t, dy_rows)
        return dx, dg, dw1, dw2

    def combine(self, y_rows, row_of_slot):
        return self.mx.moe_combine(y_rows, row_of_slot)


def _exchange(out, inp, out_splits, in_splits, group):
    """all_to_all_single along dim 0; 16-bit rows travel as bytes (the exchange is a copy, and
    not every backend moves 16-bit integers)."""
    import torch
    import torch.distributed as dist
    if inp.element_size() == 2:
        out, inp = out.view(torch.uint8), inp.view(torch.uint8)
    dist.all_to_all_single(out, inp, out_splits, in_splits, group=group)


def local_experts_of_received_rows(recv_split: np.ndarray) -> np.ndarray:
    """Local expert id of every received row, in the order received: the rows from source s
    come after those of sources 0 .. s-1, sorted by local expert, recv_split[s, e] of expert e."""
    rs = np.asarray(recv_split, dtype=np.int64)
    world, E_loc = rs.shape
    parts = [np.repeat(np.arange(E_loc, dtype=np.int32), rs[s]) for s in range(world)]
    return np.concatenate(parts) if parts else np.zeros(0, dtype=np.int32)


class EpContext:
    """What the backward needs from a training forward: the routing of this rank's choices and
    of the rows it received, the exchange sizes, the received rows and the saved
    pre-activations of this rank's experts."""

    def __init__(self, **kw):
        self.__dict__.update(kw)


def _dispatch(x_tokens, experts, gates, E, group, ops):
    """Steps 1-3: sort this rank's choices, exchange counts, rows and routing weights, and sort
    the received rows by local expert.  Returns a context (without the forward's outputs)."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    if E % world != 0:
        raise ValueError(f"{E} experts do not divide over {world} ranks")
    if experts.dim() != 2 or experts.dtype != torch.int32 or experts.shape[0] != x_tokens.shape[0]:
        raise ValueError("experts must be int32 [T, k] with T = rows of x_tokens")
    if gates is not None and tuple(gates.shape) != tuple(experts.shape):
        raise ValueError("gates must be [T, k] like experts")
    E_loc = E // world
    T, k = experts.shape
    H = x_tokens.shape[1]
    dev = x_tokens.device

    # 1. sort this rank's choices by expert: the rows bound for rank r are one run
    split, row_of_slot, token_of_row, gates_sorted = ops.permute(experts, gates, E)

    # 2. per-expert counts both ways, row counts on the host (one copy)
    send_split = split.view(world, E_loc).contiguous()
    recv_split = torch.empty_like(send_split)
    dist.all_to_all_single(recv_split, send_split, group=group)
    both = torch.stack([send_split, recv_split]).cpu().numpy()
    send_counts = [int(c) for c in both[0].sum(1)]
    recv_split_h = both[1]
    recv_counts = [int(c) for c in recv_split_h.sum(1)]
    R_recv = sum(recv_counts)

    # 3. rows and routing weights to their owners
    x_send = ops.gather_rows(x_tokens, token_of_row)
    x_recv = torch.empty((R_recv, H), dtype=x_send.dtype, device=dev)
    _exchange(x_recv, x_send, recv_counts, send_counts, group)
    g_recv = None
    if gates_sorted is not None:
        g_recv = torch.empty(R_recv, dtype=gates_sorted.dtype, device=dev)
        _exchange(g_recv, gates_sorted, recv_counts, send_counts, group)

    # the received rows in expert-major order (stable: sources stay in order)
    split_l = ros_l = tor_l = gs_l = None
    if R_recv > 0:
        local_e = torch.from_numpy(local_experts_of_received_rows(recv_split_h)).to(dev)
        split_l, ros_l, tor_l, gs_l = ops.permute(local_e.view(-1, 1),
                                                 None if g_recv is None else g_recv.view(-1, 1), E_loc)
    return EpContext(T=T, k=k, H=H, dev=dev, row_of_slot=row_of_slot, token_of_row=token_of_row,
                     send_counts=send_counts, recv_counts=recv_counts, R_recv=R_recv, x_recv=x_recv,
                     with_gates=gates_sorted is not None, split_l=split_l, ros_l=ros_l, tor_l=tor_l, gs_l=gs_l,
                     saved=None)


def _return_rows(rows_sorted, ctx, group, ops, dtype, width):
    """Rows computed by the owner in expert-major order -> back to their sources, in each
    source's sorted order (steps 4-5 of the forward, and the backward's way home)."""
    import torch
    if ctx.R_recv > 0:
        back = ops.gather_rows(rows_sorted, ctx.ros_l)
    else:
        back = torch.empty((0,) + width, dtype=dtype, device=ctx.dev)
    ret = torch.empty((ctx.T * ctx.k,) + width, dtype=dtype, device=ctx.dev)
    _exchange(ret, back, ctx.send_counts, ctx.recv_counts, group)
    return ret


def ep_moe_forward(x_tokens, experts, gates, weights, E: int, group=None, ops=None):
    """MoE layer forward with the experts spread over the ranks of ``group``.

    x_tokens [T, H] (this rank's tokens), experts int32 [T, k] (global expert ids in [0, E)),
    gates float32 [T, k] or None, weights = (w1_q, w1_sf, w2_q, w2_sf) of this rank's E / world
    experts (the layout ``grouped_mlp_fwd`` takes).  E must be a multiple of the group size.
    Returns out [T, H]: out[t] = sum over t's k slots of expert(slot)(x[t]) scaled by its gate.
    """
    ops = ops or KernelOps()
    ctx = _dispatch(x_tokens, experts, gates, E, group, ops)
    y_sorted = None
    if ctx.R_recv > 0:
        y_sorted = ops.expert_mlp(ctx.x_recv, ctx.tor_l, ctx.split_l, ctx.gs_l, weights)
    y_ret = _return_rows(y_sorted, ctx, group, ops, ops.y_dtype, (ctx.H,))
    return ops.combine(y_ret, ctx.row_of_slot)


def ep_moe_forward_train(x_tokens, experts, gates, weights, E: int, group=None, ops=None):
    """ep_moe_forward that also keeps what ep_moe_backward needs.  Returns (out, ctx)."""
    ops = ops or KernelOps()
    ctx = _dispatch(x_tokens, experts, gates, E, group, ops)
    y_sorted = None
    if ctx.R_recv > 0:
        y_sorted, ctx.saved = ops.expert_mlp_train(ctx.x_recv, ctx.tor_l, ctx.split_l, ctx.gs_l, weights)
    y_ret = _return_rows(y_sorted, ctx, group, ops, ops.y_dtype, (ctx.H,))
    return ops.combine(y_ret, ctx.row_of_slot), ctx


def ep_moe_backward(d_out, ctx, weights_t, group=None, ops=None):
    """Backward of ep_moe_forward_train.

    d_out [T, H] (gradient of this rank's output rows), ctx from the forward, weights_t =
    (w1t_q, w1t_sf, w2t_q, w2t_sf) of this rank's experts quantized along their other axis (the
    layout ``grouped_mlp_bwd`` takes).  Returns (dx [T, H], dgates [T, k] or None, dW1, dW2), the
    weight gradients those of this rank's experts ([E_loc, 2F, H] and [E_loc, H, F]; None when no
    row reached them)."""
    import torch
    ops = ops or KernelOps()
    # the gradient of the combine: each sorted row's output gradient is its token's row of d_out
    dy_send = ops.gather_rows(d_out, ctx.token_of_row)
    dy_recv = torch.empty((ctx.R_recv, ctx.H), dtype=dy_send.dtype, device=ctx.dev)
    _exchange(dy_recv, dy_send, ctx.recv_counts, ctx.send_counts, group)
    dx_sorted = dg_sorted = dw1 = dw2 = None
    if ctx.R_recv > 0:
        dx_sorted, dg_sorted, dw1, dw2 = ops.expert_mlp_bwd(ctx.x_recv, ctx.tor_l, ctx.split_l, ctx.gs_l, ctx.saved,
                                                            weights_t, dy_recv)
    dx_ret = _return_rows(dx_sorted, ctx, group, ops, ops.y_dtype, (ctx.H,))
    dx = ops.combine(dx_ret, ctx.row_of_slot)   # the gradient of the token gather: sum over slots
    dgates = None
    if ctx.with_gates:
        dg_ret = _return_rows(dg_sorted, ctx, group, ops, ops.dg_dtype, ())
        dgates = ops.gather_rows(dg_ret, ctx.row_of_slot).view(ctx.T, ctx.k)
    return dx, dgates, dw1, dw2
