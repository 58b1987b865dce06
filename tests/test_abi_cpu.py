"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every entry
point include/rsc.h declares, and validates arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def rsc():
    from recurrent_state_cache_gb300 import _build, binding
    _build.build()
    return binding


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "rsc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_symbol(rsc):
    declared = _declared_functions()
    assert len(declared) >= 10
    L = rsc.lib()
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(rsc.EXPORTS) == declared


def _desc(rsc, **kw):
    base = dict(num_layers=2, num_slots=5, num_heads=3, head_k=64, head_v=128, conv_kernel=4,
                state_dtype=rsc.BF16, conv_dtype=rsc.BF16, gate=rsc.KDA,
                ssm_base=0x10000, conv_base=0x20000, dev_error=0x30000)
    base.update(kw)
    return rsc.PoolDesc(**base)


def _create(rsc, d):
    h = ctypes.c_void_p()
    rc = rsc.lib().ssm_pool_create(ctypes.byref(d), ctypes.byref(h))
    return rc, h


def test_pool_create_validates_on_host(rsc):
    rc, h = _create(rsc, _desc(rsc))
    assert rc == rsc.RSC_OK and h.value
    assert rsc.lib().ssm_pool_destroy(h) == 0
    cases = [
        (dict(head_k=96), rsc.RSC_EDTYPE), (dict(head_v=32), rsc.RSC_EDTYPE),
        (dict(conv_kernel=3), rsc.RSC_EDTYPE), (dict(state_dtype=7), rsc.RSC_EDTYPE),
        (dict(gate=2), rsc.RSC_EDTYPE), (dict(num_layers=0), rsc.RSC_ERANGE),
        (dict(num_slots=-1), rsc.RSC_ERANGE), (dict(ssm_base=None), rsc.RSC_EINVAL),
        (dict(dev_error=None), rsc.RSC_EINVAL), (dict(conv_base=0x20008), rsc.RSC_EALIGN),
    ]
    for kw, want in cases:
        rc, h = _create(rsc, _desc(rsc, **kw))
        assert rc == want, (kw, rc)
        assert not h.value


def test_calls_reject_bad_arguments_before_launch(rsc):
    rc, h = _create(rsc, _desc(rsc))
    assert rc == 0
    L = rsc.lib()
    p = ctypes.c_void_p(0x40000)
    try:
        # layer out of range, negative batch
        assert L.kda_decode_step(h, 2, p, 1, p, p, p, p, p, None) == rsc.RSC_ERANGE
        assert L.kda_decode_step(h, 0, p, -1, p, p, p, p, p, None) == rsc.RSC_ERANGE
        # batch 0 is a no-op that launches nothing
        assert L.kda_decode_step(h, 0, None, 0, None, None, None, None, None, None) == 0
        # null / misaligned device pointers
        assert L.kda_decode_step(h, 0, p, 1, None, p, p, p, p, None) == rsc.RSC_EINVAL
        assert L.kda_decode_step(h, 0, p, 1, ctypes.c_void_p(0x40008), p, p, p, p,
                                 None) == rsc.RSC_EALIGN
        # the general call: option pairs must be complete, flags known
        O = rsc.DecodeOpts
        ob = lambda *a: ctypes.byref(O(*a))
        assert L.kda_decode_step_ex(h, 0, p, 1, p, p, p, p, p, ob(None, None, None, None, 2),
                                    None) == rsc.RSC_EINVAL
        assert L.kda_decode_step_ex(h, 0, p, 1, p, p, p, p, p, ob(0x40000, None, None, None, 0),
                                    None) == rsc.RSC_EINVAL
        assert L.kda_decode_step_ex(h, 0, p, 1, p, p, p, p, p, ob(None, None, 0x40000, None, 1),
                                    None) == rsc.RSC_EINVAL
        assert L.kda_decode_step_ex(h, 0, p, 1, p, p, p, p, p,
                                    ob(0x40000, 0x40008, None, None, 0), None) == rsc.RSC_EALIGN
        assert L.kda_decode_step_ex(h, 0, p, 1, p, p, p, p, p,
                                    ob(None, None, 0x40000, 0x40002, 0), None) == rsc.RSC_EALIGN
        assert L.kda_decode_step_ex(h, 0, None, 0, None, None, None, None, None,
                                    ob(0x40000, 0x40000, 0x40000, 0x40000, 1), None) == 0
        assert L.kda_decode_step_ex(h, 5, p, 1, p, p, p, p, p, None, None) == rsc.RSC_ERANGE
        # the tracked and gated forms still require their own pointers
        assert L.kda_decode_step_track(h, 0, p, 1, p, p, p, p, p, None, p, None) == rsc.RSC_EINVAL
        assert L.kda_decode_step_gated(h, 0, p, 1, p, p, p, p, p, None, p, None) == rsc.RSC_EINVAL
        # the overlapped form validates the same way
        assert L.kda_decode_step_overlap(h, 2, p, 1, p, p, p, p, p, None) == rsc.RSC_ERANGE
        assert L.kda_decode_step_overlap(h, 0, None, 0, None, None, None, None, None, None) == 0
        assert L.kda_decode_step_overlap(h, 0, p, 1, p, p, None, p, p, None) == rsc.RSC_EINVAL
        assert L.kda_decode_step_overlap(h, 0, p, 1, p, p, p, p, ctypes.c_void_p(0x40004),
                                         None) == rsc.RSC_EALIGN
        # spec: L not a power of two, T > L, bad mode
        assert L.kda_spec_verify_commit(h, 0, 0, p, 1, 3, 6, p, p, p, p, p, p, p, None,
                                        None) == rsc.RSC_ERANGE
        assert L.kda_spec_verify_commit(h, 0, 0, p, 1, 9, 8, p, p, p, p, p, p, p, None,
                                        None) == rsc.RSC_ERANGE
        assert L.kda_spec_verify_commit(h, 0, 5, p, 1, 2, 8, p, p, p, p, p, p, p, None,
                                        None) == rsc.RSC_EINVAL
        assert L.kda_spec_verify_commit(h, 0, 1, p, 1, 2, 8, p, p, None, None, None, None,
                                        None, None, None) == rsc.RSC_EINVAL  # no accept
        # replay: ring too short for T (2 T > depth), depth not a power of two, no rings,
        # misaligned ring array, no ring positions
        R = rsc.ReplayRingsDesc(16, 0x50000, 0x50000, 0x50000, 0x50000, 0x50000, 0x50000)
        rr = ctypes.byref(R)
        assert L.kda_replay_verify_commit(h, rr, 0, 0, p, p, 1, 9, p, p, p, p, p, p, None,
                                          None) == rsc.RSC_ERANGE
        R12 = rsc.ReplayRingsDesc(12, 0x50000, 0x50000, 0x50000, 0x50000, 0x50000, 0x50000)
        assert L.kda_replay_verify_commit(h, ctypes.byref(R12), 0, 0, p, p, 1, 2, p, p, p, p, p,
                                          p, None, None) == rsc.RSC_ERANGE
        assert L.kda_replay_verify_commit(h, None, 0, 0, p, p, 1, 2, p, p, p, p, p, p, None,
                                          None) == rsc.RSC_EINVAL
        Rm = rsc.ReplayRingsDesc(16, 0x50008, 0x50000, 0x50000, 0x50000, 0x50000, 0x50000)
        assert L.kda_replay_verify_commit(h, ctypes.byref(Rm), 0, 0, p, p, 1, 2, p, p, p, p, p,
                                          p, None, None) == rsc.RSC_EALIGN
        assert L.kda_replay_verify_commit(h, rr, 0, 0, p, None, 1, 2, p, p, p, p, p, p, None,
                                          None) == rsc.RSC_EINVAL
        assert L.kda_replay_verify_commit(h, rr, 0, 1, p, p, 1, 2, p, None, None, None, None,
                                          None, None, None) == rsc.RSC_EINVAL  # no accept
        # copy: layer below -1
        assert L.ssm_slot_copy(h, -2, p, p, None, 1, None) == rsc.RSC_ERANGE
        assert L.ssm_slot_copy(h, -1, None, None, None, 0, None) == 0
        # prefill: workspace too small, no sequences
        assert L.kda_prefill_chunk(h, 0, p, p, 1, 100, None, p, p, p, p, p, p, 16,
                                   None) == rsc.RSC_ENOSPACE
        assert L.kda_prefill_chunk(h, 0, p, p, 0, 0, None, p, p, p, p, p, p, 0,
                                   None) == rsc.RSC_ERANGE
        n = ctypes.c_size_t()
        assert L.kda_prefill_workspace_size(h, 1, 100, ctypes.byref(n)) == 0 and n.value > 0
    finally:
        L.ssm_pool_destroy(h)


def test_prefill_workspace_of_the_blocked_form(rsc):
    """Pools outside the tensor-core form (fp32 state, or head_k 64) size their prefill
    workspace as one record per (8-token block, head): floor(T/8) + N blocks, each holding the
    scaled keys and queries [16][K], end-scaled keys [8][K], e^Gamma_end [K], the A / P rows
    [8][16], beta [8] and 8 of padding, and the values [V][8], in fp32."""
    L = rsc.lib()
    for st, K, V in [(rsc.F32, 128, 128), (rsc.F32, 64, 128), (rsc.BF16, 64, 64), (rsc.F32, 128, 64)]:
        rc, h = _create(rsc, _desc(rsc, head_k=K, head_v=V, state_dtype=st))
        assert rc == rsc.RSC_OK
        try:
            rec = 16 * K + 8 * K + K + 8 * 16 + 16 + 8 * V
            for N, T in [(1, 0), (1, 7), (1, 8), (3, 100), (64, 13568)]:
                n = ctypes.c_size_t()
                assert L.kda_prefill_workspace_size(h, N, T, ctypes.byref(n)) == 0
                assert n.value == (T // 8 + N) * 3 * rec * 4, (st, K, V, N, T)
        finally:
            L.ssm_pool_destroy(h)


def test_pool_bytes_agree_with_oracle_layout(rsc):
    import oracle
    for (layers, slots, H, K, V, st, io) in [(69, 80, 12, 128, 128, 1, 1), (48, 1024, 32, 128, 128, 0, 1),
                                             (1, 16, 4, 64, 64, 0, 0)]:
        assert rsc.ssm_pool_bytes(layers, slots, H, K, V, st, io) == \
            oracle.pool_bytes(layers, slots, H, K, V, st, io)


def test_status_strings(rsc):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert rsc.status_string(code) != "unknown status"
    assert rsc.status_string(-99) == "unknown status"
