"""Failure detection on the GPU without a fault: every pipeline wait of the GEMM kernels is
bounded, and a wait that runs out records a bit in the workspace error word, raises the abort
flag of its CTA (and of the other CTA of a pair), and lets every role drain and exit.

The test makes the waits run out for real.  MXFP8MOE_WAIT_LIMIT_NS (read by the library at each
call) shortens the pipeline waits to 1 us; the problem has K = 16384, so each tile's
accumulator takes tens of microseconds to arrive and the epilogue's wait for it cannot be met.
Teardown waits for copies and MMAs in flight keep their full 2 s, so no CTA frees TMEM or exits
with work outstanding.  Checked, in a child process per kernel family (CTA pairs, and the
single-CTA kernels):
  - the call itself returns MXFP8_OK (the condition is only visible on the device);
  - mxfp8_check_device_error reports MXFP8_ERR_DEVICE_TIMEOUT with a timeout bit set;
  - the next call on the same workspace, with the normal limit, returns OK, clears the error
    word and reproduces the output of a call made before the timed-out one bit for bit, and
    that output agrees with the oracle on sampled rows.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _child():
    import torch

    import mxfp8_block_scaled_03_gb300 as mx
    import oracle
    from mxfp8_block_scaled_03_gb300 import workloads as W
    from tests import _gpu as G

    os.environ.pop("MXFP8MOE_WAIT_LIMIT_NS", None)
    w = W.custom_moe([200, 312], H=16384, F=256, seed=11)
    x = G.to_dev_bf16(w.x_sorted)
    w1q, w1s, _, _ = mx.mxfp8_quantize(G.to_dev_bf16(w.w1), sf_layout=mx.SF_MMA)
    w2q, w2s, _, _ = mx.mxfp8_quantize(G.to_dev_bf16(w.w2), sf_layout=mx.SF_MMA)
    split = G.to_dev(w.split_sizes)
    gates = G.to_dev(w.gates)
    ws = torch.empty(mx.grouped_mlp_workspace_size(w.R, w.H, w.F, w.E), dtype=torch.uint8, device="cuda")

    y0 = mx.grouped_mlp_fwd(x, split, gates, w1q, w1s, w2q, w2s, workspace=ws)
    st, bits = mx.mxfp8_check_device_error(ws)
    assert st == 0, f"normal call reported {bits:#x}"
    y0 = y0.cpu()

    os.environ["MXFP8MOE_WAIT_LIMIT_NS"] = "1000"
    try:
        mx.grouped_mlp_fwd(x, split, gates, w1q, w1s, w2q, w2s, workspace=ws)   # returns OK: enqueued
        st, bits = mx.mxfp8_check_device_error(ws)
    finally:
        os.environ.pop("MXFP8MOE_WAIT_LIMIT_NS", None)
    assert st == mx.ERR_DEVICE_TIMEOUT, (st, hex(bits))
    assert bits & 0x1F00, hex(bits)
    print(f"timed-out call: status {st}, error bits {bits:#x}", flush=True)

    y1 = mx.grouped_mlp_fwd(x, split, gates, w1q, w1s, w2q, w2s, workspace=ws)
    st, bits = mx.mxfp8_check_device_error(ws)
    assert st == 0 and bits == 0, (st, hex(bits))
    y1 = y1.cpu()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16)), "output after the timed-out call differs"

    rows = np.array([0, 1, 127, 199, 200, 255, 256, 383, 384, 511])
    o1q, o1s = oracle.quantize_rowwise(w.w1)
    o2q, o2s = oracle.quantize_rowwise(w.w2)
    y_ref, _, _ = oracle.grouped_mlp_rows(w.x_sorted, w.split_sizes, w.gates, o1q, o1s, o2q, o2s, rows,
                                          want_intermediate=False)
    rel, mxe = G.y_errors(y1.float().numpy().astype(np.float64)[rows], y_ref)
    assert rel <= G.Y_REL_TOL and mxe <= G.Y_MAX_TOL, (rel, mxe)
    print("timeout path ok", flush=True)


@pytest.mark.parametrize("single_cta", [False, True], ids=["cta_pairs", "single_cta"])
def test_pipeline_wait_timeout_is_reported_and_recovers(single_cta):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from mxfp8_block_scaled_03_gb300 import build_ext
    build_ext.build()
    env = dict(os.environ)
    env.pop("MXFP8MOE_WAIT_LIMIT_NS", None)
    if single_cta:
        env["MXFP8MOE_SINGLE_CTA"] = "1"
    else:
        env.pop("MXFP8MOE_SINGLE_CTA", None)
    r = subprocess.run([sys.executable, os.path.abspath(__file__)], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "timeout path ok" in r.stdout


if __name__ == "__main__":
    _child()
