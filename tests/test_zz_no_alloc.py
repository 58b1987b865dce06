"""kda_prefill_chunk_noalloc, the prefill entry point for callers that cannot allocate
device memory (their HBM is already handed to their own pools, or cudaMalloc's device
synchronisation is not acceptable on their path).  It must give the results of
kda_prefill_chunk with a caller workspace, call after call, on the library's shared
static scratch.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import oracle
import recurrent_state_cache_gb300 as rsc
from recurrent_state_cache_gb300 import binding, inputs
from tests.devio import to_dev, to_np, widen
from tests.tolerances import TOL, max_rel_err

pytestmark = pytest.mark.gpu


def _pools(dev, st, H, K, V, P, seed):
    r = inputs.rng(seed)
    ssm, conv = inputs.pool_arrays(r, 1, P, H, K, V, st, st)
    ref = oracle.Pool(1, P, H, K, V, st, st, oracle.KDA, ssm, conv)
    a = rsc.SlotPool(1, P, H, K, V, st, st, rsc.KDA, dev, ssm=to_dev(ssm, dev), conv=to_dev(conv, dev))
    b = rsc.SlotPool(1, P, H, K, V, st, st, rsc.KDA, dev, ssm=to_dev(ssm, dev), conv=to_dev(conv, dev))
    return r, ref, a, b


@pytest.mark.parametrize("st,K", [
    (rsc.F32, 64),    # blocked path, 2 key channels a lane
    (rsc.F32, 128),   # blocked path, 4 key channels a lane
    (rsc.BF16, 64),   # blocked path of a bf16-state pool
    (rsc.BF16, 128),  # chunkwise tensor-core path: chunk table and operand blocks in the array
])
def test_noalloc_prefill_matches_workspace_prefill_twice(cuda_dev, st, K):
    """Two calls in a row on the shared static scratch (the second continues from the state
    the first left, and meets the first call's leftovers in the array): outputs, states and
    windows equal those of kda_prefill_chunk with a caller workspace, and the oracle's."""
    H, V, P = 2, 128, 6
    r, ref, pool_ws, pool_na = _pools(cuda_dev, st, H, K, V, P, seed=31)
    w_np = inputs.conv_weights(r, H, K, V)
    w = to_dev(w_np, cuda_dev)
    slots_np = np.int32([4, 2])
    slots = to_dev(slots_np, cuda_dev)
    for call in range(2):
        lens = [97, 203] if call == 0 else [1, 130]
        cu = inputs.cu_seqlens(lens)
        T = int(cu[-1])
        x_np = inputs.projections(r, (T,), H, K, V, st)
        g_np, beta_np = inputs.gates(r, (T,), H, K, rsc.KDA)
        hi_np = np.uint8([call, 1])
        o_ref = oracle.prefill(ref, 0, slots_np, cu, x_np, w_np, g_np, beta_np, has_init=hi_np)
        x, g, beta = to_dev(x_np, cuda_dev), to_dev(g_np, cuda_dev), to_dev(beta_np, cuda_dev)
        cu_d, hi = to_dev(cu, cuda_dev), to_dev(hi_np, cuda_dev)
        o_ws = rsc.kda_prefill_chunk(pool_ws, 0, slots, cu_d, x, w, g, beta, has_initial_state=hi)
        o_na = binding.kda_prefill_chunk_noalloc(pool_na, 0, slots, cu_d, x, w, g, beta,
                                                 has_initial_state=hi)
        torch.cuda.synchronize()
        assert max_rel_err(widen(to_np(o_na)), widen(to_np(o_ws))) <= TOL[st]
        assert max_rel_err(widen(to_np(pool_na.ssm)), widen(to_np(pool_ws.ssm))) <= TOL[st]
        assert np.array_equal(to_np(pool_na.conv), to_np(pool_ws.conv))
        tc = st == rsc.BF16 and K == 128  # the chunkwise tensor-core path
        assert max_rel_err(widen(to_np(o_na)), widen(o_ref), tc=tc) <= TOL[st]
        assert max_rel_err(widen(to_np(pool_na.ssm)), widen(ref.ssm), tc=tc) <= TOL[st]
        assert np.array_equal(to_np(pool_na.conv), ref.conv)
        assert rsc.rsc_get_device_error(pool_na) == 0


def test_noalloc_prefill_rejects_sizes_beyond_its_scratch(cuda_dev):
    H, K, V = 12, 128, 128
    pool = rsc.SlotPool(1, 2, H, K, V, rsc.BF16, rsc.BF16, rsc.KDA, cuda_dev)
    T = 4096  # workspace need above the 32 MiB array
    assert rsc.kda_prefill_workspace_size(pool, 1, T) > 32 << 20
    D = pool.D
    x = torch.zeros((T, D), dtype=torch.bfloat16, device=cuda_dev)
    g = torch.zeros((T, H, K), device=cuda_dev)
    beta = torch.zeros((T, H), device=cuda_dev)
    w = torch.zeros((D, 4), device=cuda_dev)
    with pytest.raises(binding.RscError) as e:
        binding.kda_prefill_chunk_noalloc(pool, 0, torch.tensor([1], dtype=torch.int32, device=cuda_dev),
                                          torch.tensor([0, T], dtype=torch.int32, device=cuda_dev),
                                          x, w, g, beta)
    assert e.value.status == binding.RSC_ENOSPACE
