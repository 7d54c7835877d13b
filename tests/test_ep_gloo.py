"""Expert-parallel MoE layer (mxfp8_block_scaled_03_gb300.ep) on CPU: gloo process groups of 1
and 2 ranks, the compute steps done by the oracle; forward, and training forward + backward.

Page "Efficient MoE training for biological foundation models", How to run the recipe (experts
spread over the GPUs, data- and expert-parallel sizes multiplying to the GPU count) and Key
technical approaches item 1 (tokens gathered per expert, counted by split_sizes).

The bar: every rank's output rows equal, bit for bit, the single-process layer (oracle permute,
oracle binary64 expert MLP, oracle combine) on all tokens with all experts, because each row's
expert output depends only on the row and the expert, and the combine sums a token's slots in
the same order.  The backward's dx, routing-weight gradients and (sampled) weight gradients of
each rank's experts equal the single-process backward the same way: an expert's rows reach its
owner in the global (token, slot) order.  This covers the exchange logic (counts, splits, orders,
the regrouping by local expert and the ways back); the CUDA kernels of the same steps are covered
by the GPU tests.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """The layer's compute steps on the oracle (CPU, binary64 expert outputs and gradients).
    For the backward, weights_t = (w1q, w1sf, w2tq, w2tsf, w1tq, w1tsf) of the rank's experts in
    the oracle's layouts, and the weight gradients come back as the entries `dw_entries` (local
    expert, row, column) of dW1 and dW2."""

    def __init__(self, oracle, dw_entries=None):
        import torch
        self.o = oracle
        self.y_dtype = torch.float64
        self.dg_dtype = torch.float64
        self.dw_entries = dw_entries

    def permute(self, experts, gates, E):
        import torch
        split, ros, tor, gs = self.o.moe_permute(experts.numpy(), None if gates is None else gates.numpy(), E)
        return (torch.from_numpy(split), torch.from_numpy(ros), torch.from_numpy(tor),
                None if gs is None else torch.from_numpy(gs))

    def gather_rows(self, x, index):
        return x[index.long()]

    def expert_mlp(self, x_rows, token_of_row, split, gates_sorted, weights):
        import torch
        xs = np.ascontiguousarray(x_rows.numpy().view(np.uint16)[token_of_row.numpy()])
        gs = None if gates_sorted is None else gates_sorted.numpy()
        y, _, _ = self.o.grouped_mlp_rows(xs, split.numpy(), gs, *weights, np.arange(xs.shape[0]),
                                          want_intermediate=False)
        return torch.from_numpy(y)

    def combine(self, y_rows, row_of_slot):
        import torch
        return torch.from_numpy(self.o.moe_combine(y_rows.numpy(), row_of_slot.numpy()))

    def expert_mlp_train(self, x_rows, token_of_row, split, gates_sorted, weights):
        return self.expert_mlp(x_rows, token_of_row, split, gates_sorted, weights), None

    def expert_mlp_bwd(self, x_rows, token_of_row, split, gates_sorted, saved, weights_t, dy_rows):
        import torch
        tor = token_of_row.numpy()
        xs = np.ascontiguousarray(x_rows.numpy().view(np.uint16)[tor])
        dys = np.ascontiguousarray(dy_rows.numpy().view(np.uint16)[tor])
        gs = None if gates_sorted is None else gates_sorted.numpy()
        w1q, w1s, w2tq, w2ts, w1tq, w1ts = weights_t
        dx, dg, _, _ = self.o.grouped_mlp_bwd_rows(xs, split.numpy(), gs, w1q, w1s, w2tq, w2ts, w1tq, w1ts, dys,
                                                   np.arange(xs.shape[0]))
        dw1 = self.o.grouped_mlp_bwd_dw(xs, split.numpy(), gs, w1q, w1s, w2tq, w2ts, dys, 1, self.dw_entries[1])
        dw2 = self.o.grouped_mlp_bwd_dw(xs, split.numpy(), gs, w1q, w1s, w2tq, w2ts, dys, 2, self.dw_entries[2])
        return torch.from_numpy(dx), torch.from_numpy(dg), dw1, dw2


def _problem(case):
    """Tokens, router choices and quantized weights of the whole layer (every rank builds the
    same), and how many tokens each rank holds."""
    sys.path.insert(0, ROOT)
    import oracle
    from mxfp8_block_scaled_03_gb300 import workloads as W
    w = W.moe_workload("tiny")
    T = w.x_tokens.shape[0]
    experts = w.topk_experts.astype(np.int32).copy()
    gates = w.topk_gates.astype(np.float32).copy()
    counts = [T // 2, T - T // 2]
    if case == "uneven":
        counts = [100, T - 100]
    elif case == "one_owner":
        experts = experts % 2          # every choice lands on rank 0's experts (0 and 1)
        experts[:, 1] = 1 - experts[:, 0]
    elif case == "no_gates":
        gates = None
    w1q, w1s = oracle.quantize_rowwise(w.w1)
    w2q, w2s = oracle.quantize_rowwise(w.w2)
    return oracle, w, experts, gates, counts, (w1q, w1s, w2q, w2s)


def _reference(oracle, w, experts, gates, weights):
    split, ros, tor, gs = oracle.moe_permute(experts, gates, w.E)
    xs = np.ascontiguousarray(w.x_tokens[tor])
    y, _, _ = oracle.grouped_mlp_rows(xs, split, gs, *weights, np.arange(xs.shape[0]), want_intermediate=False)
    return oracle.moe_combine(y, ros)


def _worker(rank, world, port, case, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        oracle, w, experts, gates, counts, (w1q, w1s, w2q, w2s) = _problem(case)
        if world == 1:
            counts = [sum(counts)]
        t0 = sum(counts[:rank])
        t1 = t0 + counts[rank]
        E_loc = w.E // world
        F, H = w.F, w.H
        local_w = (w1q[rank * E_loc * 2 * F:(rank + 1) * E_loc * 2 * F], w1s[rank * E_loc * 2 * F:(rank + 1) * E_loc * 2 * F],
                   w2q[rank * E_loc * H:(rank + 1) * E_loc * H], w2s[rank * E_loc * H:(rank + 1) * E_loc * H])
        from mxfp8_block_scaled_03_gb300 import ep
        x_loc = torch.from_numpy(np.ascontiguousarray(w.x_tokens[t0:t1]).view(np.int16))
        ex_loc = torch.from_numpy(np.ascontiguousarray(experts[t0:t1]))
        g_loc = None if gates is None else torch.from_numpy(np.ascontiguousarray(gates[t0:t1]))
        got = ep.ep_moe_forward(x_loc, ex_loc, g_loc, local_w, w.E, ops=OracleOps(oracle)).numpy()
        ref = _reference(oracle, w, experts, gates, (w1q, w1s, w2q, w2s))[t0:t1]
        out[rank] = (got.shape == ref.shape, bool(np.array_equal(got, ref)), float(np.abs(ref).max()))
    finally:
        dist.destroy_process_group()


def _run(world, case):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, case, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return dict(out)


@pytest.mark.parametrize("case", ["even", "uneven", "one_owner", "no_gates"])
def test_ep_two_ranks_matches_single_process_layer(case):
    res = _run(2, case)
    assert set(res) == {0, 1}
    for rank, (shape_ok, equal, mag) in res.items():
        assert shape_ok and mag > 0, (rank, res)
        assert equal, f"rank {rank}: expert-parallel output differs from the single-process layer"


def test_ep_one_rank_is_the_plain_layer():
    res = _run(1, "even")
    assert res[0][0] and res[0][1]


def test_local_expert_ids_follow_the_sources_in_order():
    from mxfp8_block_scaled_03_gb300 import ep
    got = ep.local_experts_of_received_rows(np.array([[2, 0, 1], [0, 3, 1]]))
    assert got.tolist() == [0, 0, 2, 1, 1, 1, 2]
    assert ep.local_experts_of_received_rows(np.zeros((2, 3), dtype=np.int32)).size == 0


def _train_worker(rank, world, port, case, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        oracle, w, experts, gates, counts, (w1q, w1s, w2q, w2s) = _problem(case)
        w2tq, w2ts = oracle.quantize_transposed(w.w2, w.E)
        w1tq, w1ts = oracle.quantize_transposed(w.w1, w.E)
        from mxfp8_block_scaled_03_gb300 import workloads as W
        d_out = W.bf16_bits(np.random.default_rng(5).standard_normal(w.x_tokens.shape).astype(np.float32))
        t0 = sum(counts[:rank])
        t1 = t0 + counts[rank]
        E_loc, F, H = w.E // world, w.F, w.H
        lo, hi = rank * E_loc, (rank + 1) * E_loc
        rng = np.random.default_rng(9)
        ent1 = np.stack([rng.integers(0, E_loc, 40), rng.integers(0, 2 * F, 40), rng.integers(0, H, 40)], 1)
        ent2 = np.stack([rng.integers(0, E_loc, 40), rng.integers(0, H, 40), rng.integers(0, F, 40)], 1)
        ops = OracleOps(oracle, {1: ent1, 2: ent2})
        wl = (w1q[lo * 2 * F:hi * 2 * F], w1s[lo * 2 * F:hi * 2 * F], w2q[lo * H:hi * H], w2s[lo * H:hi * H])
        wt = (wl[0], wl[1], w2tq[lo * F:hi * F], w2ts[lo * F:hi * F], w1tq[lo * H:hi * H], w1ts[lo * H:hi * H])
        from mxfp8_block_scaled_03_gb300 import ep

        def tens(a, view=None):
            a = np.ascontiguousarray(a)
            return torch.from_numpy(a.view(view) if view is not None else a)

        y, ctx = ep.ep_moe_forward_train(tens(w.x_tokens[t0:t1], np.int16), tens(experts[t0:t1]),
                                         None if gates is None else tens(gates[t0:t1]), wl, w.E, ops=ops)
        dx, dg, dw1, dw2 = ep.ep_moe_backward(tens(d_out[t0:t1], np.int16), ctx, wt, ops=ops)

        # the same layer in one process, all experts
        split, ros, tor, gs = oracle.moe_permute(experts, gates, w.E)
        xs = np.ascontiguousarray(w.x_tokens[tor])
        dys = np.ascontiguousarray(d_out[tor])
        y_ref = oracle.moe_combine(oracle.grouped_mlp_rows(xs, split, gs, w1q, w1s, w2q, w2s, np.arange(len(tor)),
                                                           want_intermediate=False)[0], ros)
        dxr, dgr, _, _ = oracle.grouped_mlp_bwd_rows(xs, split, gs, w1q, w1s, w2tq, w2ts, w1tq, w1ts, dys,
                                                     np.arange(len(tor)))
        dx_ref = oracle.moe_combine(dxr, ros)
        g1 = ent1.copy(); g1[:, 0] += lo
        g2 = ent2.copy(); g2[:, 0] += lo
        dw1_ref = oracle.grouped_mlp_bwd_dw(xs, split, gs, w1q, w1s, w2tq, w2ts, dys, 1, g1)
        dw2_ref = oracle.grouped_mlp_bwd_dw(xs, split, gs, w1q, w1s, w2tq, w2ts, dys, 2, g2)
        res = {"y": bool(np.array_equal(y.numpy(), y_ref[t0:t1])),
               "dx": bool(np.array_equal(dx.numpy(), dx_ref[t0:t1])),
               "dx_nonzero": bool(np.abs(dx_ref[t0:t1]).max() > 0)}
        if gates is not None:
            res["dg"] = bool(np.array_equal(dg.numpy(), dgr[ros][t0:t1]))
        if dw1 is None:   # no row reached this rank's experts: the reference gradients are zero
            res["dw"] = not dw1_ref.any() and not dw2_ref.any()
        else:
            res["dw"] = bool(np.array_equal(dw1, dw1_ref) and np.array_equal(dw2, dw2_ref))
        out[rank] = res
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", ["even", "uneven", "one_owner", "no_gates"])
def test_ep_training_two_ranks_matches_single_process_layer(case):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_train_worker, args=(r, 2, port, case, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(600)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = dict(out)
    assert set(res) == {0, 1}
    for rank, r in res.items():
        assert all(r.values()), (rank, r)
