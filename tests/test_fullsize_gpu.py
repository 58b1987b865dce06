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


@pytest.mark.parametrize("st", [rsc.BF16, rsc.F32])
def test_full_size_chunked_prefill_13600_with_snapshots(cuda_dev, st):
    """The chunked-prefill workload at full size, in the benchmark's launch configuration:
    one KDA layer, H=12, K=V=128, bf16 io, bf16 state (the tensor-core path) or fp32 state
    (the blocked closed form, at the fp32 bar for states); a 13600-token prompt as calls of
    6144, 6144 and 1312
    tokens through one slot (the first from a fresh state), each followed by an ssm_slot_copy
    of the slot into a fresh snapshot slot; the sequence captured in a CUDA graph and
    replayed.  Every output token, the three snapshots and the final state against the
    oracle's token-by-token run; windows bit-exact; the rest of the pool untouched."""
    from recurrent_state_cache_gb300 import inputs
    from tests.devio import to_dev
    from tests.tolerances import TOL

    torch.cuda.set_device(cuda_dev)
    stream = torch.cuda.Stream(device=cuda_dev)
    torch.cuda.set_stream(stream)
    Hp, Pp, chunks = 12, 6, (6144, 6144, 1312)
    slot, snaps = 1, (2, 3, 4)
    r = inputs.rng(5)
    tc = st == rsc.BF16
    ssm, conv = inputs.pool_arrays(r, 1, Pp, Hp, K, V, st, 1)
    ref = oracle.Pool(1, Pp, Hp, K, V, st, oracle.BF16, oracle.KDA, ssm, conv)
    pool = rsc.SlotPool(1, Pp, Hp, K, V, st, rsc.BF16, rsc.KDA, cuda_dev,
                        ssm=to_dev(ssm, cuda_dev), conv=to_dev(conv, cuda_dev))
    w = inputs.conv_weights(r, Hp, K, V)
    T = sum(chunks)
    x = inputs.projections(r, (T,), Hp, K, V, 1)
    g, beta = inputs.gates(r, (T,), Hp, K, oracle.KDA)
    offs = np.cumsum((0,) + chunks)

    xd, wd, gd, bd = (to_dev(a, cuda_dev) for a in (x, w, g, beta))
    out = torch.empty((T, Hp, V), dtype=torch.bfloat16, device=cuda_dev)
    ws = torch.empty(rsc.kda_prefill_workspace_size(pool, 1, max(chunks)), dtype=torch.uint8,
                     device=cuda_dev)
    slot_d = torch.tensor([slot], dtype=torch.int32, device=cuda_dev)
    snap_d = [torch.tensor([s], dtype=torch.int32, device=cuda_dev) for s in snaps]
    fresh = torch.tensor([0], dtype=torch.uint8, device=cuda_dev)
    cus = [torch.tensor([0, c], dtype=torch.int32, device=cuda_dev) for c in chunks]

    def run():
        for i in range(len(chunks)):
            a, e = int(offs[i]), int(offs[i + 1])
            rsc.kda_prefill_chunk(pool, 0, slot_d, cus[i], xd[a:e], wd, gd[a:e], bd[a:e],
                                  has_initial_state=fresh if i == 0 else None, out=out[a:e],
                                  workspace=ws)
            rsc.ssm_slot_copy(pool, 0, slot_d, snap_d[i])

    # the sequence restarts from a fresh state, so the warm run inside graph_of and the
    # replay leave identical results
    graph = bench.graph_of(run, stream)
    graph.replay()
    torch.cuda.synchronize()
    assert rsc.rsc_get_device_error(pool) == 0

    o_ref = []
    for i, c in enumerate(chunks):
        a, e = int(offs[i]), int(offs[i + 1])
        o_ref.append(oracle.prefill(ref, 0, [slot], np.int32([0, c]), x[a:e], w, g[a:e], beta[a:e],
                                    has_init=np.uint8([0 if i == 0 else 1])))
        oracle.slot_copy(ref, 0, [slot], [snaps[i]])
    o_gpu = widen(to_np(out))
    for i in range(len(chunks)):
        a, e = int(offs[i]), int(offs[i + 1])
        err = max_rel_err(o_gpu[a:e], widen(o_ref[i]), tc=tc)
        assert err <= TOL[1], f"call {i} output max rel err {err}"
    s_gpu, c_gpu = to_np(pool.ssm), to_np(pool.conv)
    assert np.array_equal(c_gpu, ref.conv), "windows differ"
    for s in (slot,) + snaps:
        err = max_rel_err(widen(s_gpu[0, s]), widen(ref.ssm[0, s]), tc=tc)
        assert err <= TOL[st], f"slot {s} state max rel err {err}"
    for s in range(Pp + 1):
        if s not in (slot,) + snaps:
            assert np.array_equal(s_gpu[0, s], ssm[0, s])
