"""The give-up path of a bounded on-chip wait, run on the GPU without a fault or a hang.

A test build of the decode kernel (recurrent_state_cache_gb300._build.build_wait_test)
arms request 0's first state-chunk mbarrier without ever issuing its copy, and shortens the
spin limit: nothing completes that barrier, so every thread of those CTAs runs its bounded
wait out.  The kernel must then set RSC_DEVERR_TIMEOUT, wait (bounded) for the copies it did
issue, and return without storing any row of that state tile, while the other requests of
the same launch are computed normally.  The context stays usable: the next calls through
the library proper are correct."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import recurrent_state_cache_gb300 as rsc
from recurrent_state_cache_gb300 import _build, binding, inputs
from tests.devio import to_dev, to_np, widen
from tests.tolerances import TOL, max_rel_err

pytestmark = pytest.mark.gpu


def test_decode_wait_runs_out_sets_flag_and_next_call_is_clean(cuda_dev):
    L, P, H, K, V, B = 1, 8, 2, 128, 128, 3
    st = rsc.BF16
    r = inputs.rng(41)
    ssm, conv = inputs.pool_arrays(r, L, P, H, K, V, st, st)
    ref = oracle.Pool(L, P, H, K, V, st, st, oracle.KDA, ssm, conv)
    pool = rsc.SlotPool(L, P, H, K, V, st, st, rsc.KDA, cuda_dev, ssm=to_dev(ssm, cuda_dev),
                        conv=to_dev(conv, cuda_dev))
    w = inputs.conv_weights(r, H, K, V)
    slots = np.int32([5, 2, 7])
    x = inputs.projections(r, (B,), H, K, V, st)
    g, beta = inputs.gates(r, (B,), H, K, oracle.KDA)
    args = [to_dev(a, cuda_dev) for a in (slots, x, w, g, beta)]
    out = torch.zeros((B, H, V), dtype=torch.bfloat16, device=cuda_dev)

    test_lib = ctypes.CDLL(_build.build_wait_test())
    vp = ctypes.c_void_p
    test_lib.ssm_pool_create.argtypes = [ctypes.POINTER(binding.PoolDesc), ctypes.POINTER(vp)]
    test_lib.ssm_pool_destroy.argtypes = [vp]
    test_lib.kda_decode_step.argtypes = [vp, ctypes.c_int, vp, ctypes.c_int, vp, vp, vp, vp, vp, vp]
    handle = vp()
    assert test_lib.ssm_pool_create(ctypes.byref(pool.desc), ctypes.byref(handle)) == 0
    stream = torch.cuda.current_stream(cuda_dev)
    try:
        rc = test_lib.kda_decode_step(handle, 0, *(vp(t.data_ptr()) for t in args[:1]), B,
                                      *(vp(t.data_ptr()) for t in args[1:]), vp(out.data_ptr()),
                                      vp(stream.cuda_stream))
        assert rc == 0
        torch.cuda.synchronize()
    finally:
        test_lib.ssm_pool_destroy(handle)

    assert rsc.rsc_get_device_error(pool) == binding.DEVERR_TIMEOUT
    s_gpu = to_np(pool.ssm)
    # request 0: no row of its state stored
    assert np.array_equal(s_gpu[0, slots[0]], ssm[0, slots[0]])
    # requests 1 and 2: computed as usual, against the oracle on their own
    o_ref = oracle.decode_step(ref, 0, slots[1:], x[1:], w, g[1:], beta[1:])
    assert max_rel_err(widen(to_np(out[1:])), widen(o_ref)) <= TOL[st]
    for s in slots[1:]:
        assert max_rel_err(widen(s_gpu[0, s]), widen(ref.ssm[0, s])) <= TOL[st]
        assert np.array_equal(to_np(pool.conv)[0, s], ref.conv[0, s])

    # the context is usable and the library proper is unaffected: a step of two other slots
    nxt = np.int32([1, 3])
    x2 = inputs.projections(r, (2,), H, K, V, st)
    g2, b2 = inputs.gates(r, (2,), H, K, oracle.KDA)
    o2_ref = oracle.decode_step(ref, 0, nxt, x2, w, g2, b2)
    o2 = rsc.kda_decode_step(pool, 0, to_dev(nxt, cuda_dev), to_dev(x2, cuda_dev), args[2],
                             to_dev(g2, cuda_dev), to_dev(b2, cuda_dev))
    assert max_rel_err(widen(to_np(o2)), widen(o2_ref)) <= TOL[st]
    s_gpu = to_np(pool.ssm)
    for s in nxt:
        assert max_rel_err(widen(s_gpu[0, s]), widen(ref.ssm[0, s])) <= TOL[st]
    assert rsc.rsc_get_device_error(pool) == 0
