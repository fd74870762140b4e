"""DecodeStep.run_from_host: the step with inputs in pinned host memory.

Its per-layer copies run on two side streams, overlapping the kernels of the
neighbouring layers; the results must be exactly those of the device-input
step (same kernels, same inputs) and must match the oracle. Captured in a CUDA
graph and replayed too, as the benchmark's end-to-end leg does.
"""
import numpy as np
import pytest
import torch

import workloads
from tests.parity import DeviceWorkload, assert_close, oracle_layer, u16

pytestmark = pytest.mark.gpu


def _host_inputs(dw):
    pin = lambda t: t.cpu().pin_memory()
    host = {"q": pin(dw.q), "k": pin(dw.k), "v": pin(dw.v), "block_tables": pin(dw.block_tables),
            "seq_lens": pin(dw.seq_lens), "positions": pin(dw.positions)}
    dev = {"q": torch.empty_like(dw.q), "k": torch.empty_like(dw.k), "v": torch.empty_like(dw.v),
           "block_tables": dw.block_tables, "seq_lens": dw.seq_lens, "positions": dw.positions}
    return host, dev


@pytest.mark.parametrize("graph", [False, True])
def test_run_from_host_matches_device_step_and_oracle(graph):
    wl = workloads.make("llama1b_b8_l16_u512", seed=3, sentinel=True)
    want_dev = DeviceWorkload(wl)
    want = want_dev.run().cpu().numpy().copy()
    want_dev.step.close()

    dw = DeviceWorkload(wl)  # fresh pool copy: the append runs again on the same bytes
    host, dev = _host_inputs(dw)
    hout = torch.empty(dw.step.out.shape, dtype=torch.float32).pin_memory()
    streams = (torch.cuda.Stream(), torch.cuda.Stream())
    if graph:
        dw.step.run_from_host(host, dev, hout, streams)  # warm-up outside capture
        torch.cuda.synchronize()
        hout.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            dw.step.run_from_host(host, dev, hout, streams)
        g.replay()
    else:
        dw.step.run_from_host(host, dev, hout, streams)
    torch.cuda.synchronize()
    assert dw.step.error_bits() == 0
    got = hout.numpy()
    assert np.array_equal(got, want), "host-input step differs from the device-input step"

    pool_host = u16(wl.pool).reshape(-1).copy()
    q, k, v = u16(wl.q), u16(wl.k), u16(wl.v)
    for layer in range(wl.num_layers):
        _, ref = oracle_layer(pool_host, wl, layer, q[layer], k[layer], v[layer])
        assert_close(got[layer], ref, f"layer {layer}")
    dw.step.close()
