"""Parity at the benchmark's full size and launch configuration: the Kimi-K3 shard pool
(69 layers, 320 slots, H=12, K=V=128, bf16), 64 requests, one decode step over all 69
layers replayed from a CUDA graph exactly as bench.py times it.  The oracle recomputes
sampled (request, layer) pairs one by one from their initial rows; rows of slots no
request uses must not change at all."""
import numpy as np
import pytest
import torch

import bench
import oracle
import recurrent_state_cache_gb300 as rsc
from tests.devio import to_np, widen
from tests.tolerances import max_rel_err, tol

pytestmark = pytest.mark.gpu

LAYERS, P, B, H, K, V = 69, 320, 64, 12, 128, 128
SAMPLE_LAYERS = (0, 37, 68)
SAMPLE_ROWS = (0, 29, 63)


def test_full_size_decode_step_sampled(cuda_dev):
    torch.cuda.set_device(cuda_dev)
    stream = torch.cuda.Stream(device=cuda_dev)
    torch.cuda.set_stream(stream)
    wl = bench.DecodeWorkload(cuda_dev, LAYERS, P, B, H, K, V, rsc.BF16, rsc.BF16, rsc.KDA, seed=0)
    slots = wl.slots.cpu().numpy()
    used = set(int(s) for s in slots)
    unused = [s for s in range(1, P + 1) if s not in used][:4]
    # initial rows of the sampled (layer, slot) pairs and of a few unused slots
    before = {}
    for l in SAMPLE_LAYERS:
        for rrow in SAMPLE_ROWS:
            s = int(slots[rrow])
            before[(l, s)] = (to_np(wl.pool.ssm[l, s]).copy(), to_np(wl.pool.conv[l, s]).copy())
    untouched = {(l, s): (to_np(wl.pool.ssm[l, s]).copy(), to_np(wl.pool.conv[l, s]).copy())
                 for l in SAMPLE_LAYERS for s in unused}
    inputs = {l: (to_np(wl.qkv[l]), to_np(wl.w[l]), to_np(wl.g[l]), to_np(wl.beta[l]))
              for l in SAMPLE_LAYERS}

    graph = bench.graph_of(wl.step, stream)  # the warm-up call inside runs one step
    torch.cuda.synchronize()
    # graph_of ran the step once (warm call); replay once more so two steps have run
    graph.replay()
    torch.cuda.synchronize()
    assert rsc.rsc_get_device_error(wl.pool) == 0

    for l in SAMPLE_LAYERS:
        x, w, g, beta = inputs[l]
        for rrow in SAMPLE_ROWS:
            s = int(slots[rrow])
            ssm0, conv0 = before[(l, s)]
            ref = oracle.Pool(1, 1, H, K, V, oracle.BF16, oracle.BF16, oracle.KDA,
                              np.stack([np.zeros_like(ssm0), ssm0])[None],
                              np.stack([np.zeros_like(conv0), conv0])[None])
            for _ in range(2):  # the same inputs were fed on both steps
                o_ref = oracle.decode_step(ref, 0, [1], x[rrow:rrow + 1], w, g[rrow:rrow + 1],
                                           beta[rrow:rrow + 1])
            assert np.array_equal(to_np(wl.pool.conv[l, s]), ref.conv[0, 1])
            assert max_rel_err(widen(to_np(wl.pool.ssm[l, s])), widen(ref.ssm[0, 1])) <= tol(1, 1)
            assert max_rel_err(widen(to_np(wl.out[l, rrow])), widen(o_ref[0])) <= tol(1, 1)
    for (l, s), (ssm0, conv0) in untouched.items():
        assert np.array_equal(to_np(wl.pool.ssm[l, s]), ssm0)
        assert np.array_equal(to_np(wl.pool.conv[l, s]), conv0)
