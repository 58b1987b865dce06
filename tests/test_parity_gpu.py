"""Parity of the CUDA path (through the C ABI) with the CPU oracle on identical seeded
inputs.  Tolerances: max relative error (max |got-ref| / max |ref|) <= 1e-4 with fp32
state and an fp32 tensor, <= 2e-2 when the state or the tensor is bf16 (tests/tolerances);
windows, slot copies and commits bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import recurrent_state_cache_gb300 as rsc
from recurrent_state_cache_gb300 import inputs
from tests.devio import to_dev, to_np, widen
from tests.tolerances import TOL, max_rel_err, tol

pytestmark = pytest.mark.gpu


class Case:
    """One pool held twice: by the oracle (numpy) and on the device (torch)."""

    def __init__(self, dev, seed, L, P, H, K, V, st, io, gate):
        self.r = inputs.rng(seed)
        self.st, self.io, self.gate = st, io, gate
        self.H, self.K, self.V = H, K, V
        ssm, conv = inputs.pool_arrays(self.r, L, P, H, K, V, st, io)
        self.ref = oracle.Pool(L, P, H, K, V, st, io, gate, ssm, conv)
        self.pool = rsc.SlotPool(L, P, H, K, V, st, io, gate, dev,
                                 ssm=to_dev(ssm, dev), conv=to_dev(conv, dev))
        self.w = inputs.conv_weights(self.r, H, K, V)
        self.w_dev = to_dev(self.w, dev)
        self.dev = dev
        self.D = self.pool.D

    def gates(self, lead):
        return inputs.gates(self.r, lead, self.H, self.K, self.gate)

    def proj(self, lead):
        return inputs.projections(self.r, lead, self.H, self.K, self.V, self.io)

    def check_pool(self, tol=None, tc=False):
        tol = TOL[self.st] if tol is None else tol
        s_gpu, c_gpu = to_np(self.pool.ssm), to_np(self.pool.conv)
        assert np.array_equal(c_gpu, self.ref.conv), "conv windows differ"
        err = max_rel_err(widen(s_gpu), widen(self.ref.ssm), tc=tc)
        assert err <= tol, f"state max rel err {err}"
        assert rsc.rsc_get_device_error(self.pool) == 0


def _decode_steps(c, slots, steps):
    slots_d = to_dev(slots, c.dev)
    for _ in range(steps):
        B = len(slots)
        x = c.proj((B,))
        g, beta = c.gates((B,))
        o_ref = oracle.decode_step(c.ref, 0, slots, x, c.w, g, beta)
        o = rsc.kda_decode_step(c.pool, 0, slots_d, to_dev(x, c.dev), c.w_dev, to_dev(g, c.dev),
                                to_dev(beta, c.dev))
        err = max_rel_err(widen(to_np(o)), widen(o_ref))
        assert err <= tol(c.st, c.io), f"output max rel err {err}"
    c.check_pool()


def test_decode_kda_fp32_small_config(cuda_dev):
    """1 KDA layer, fp32, 16-slot pool, 4 random distinct slots, H=4, K=V=64, 8 steps."""
    c = Case(cuda_dev, 0, L=1, P=16, H=4, K=64, V=64, st=0, io=0, gate=rsc.KDA)
    slots = inputs.distinct_slots(c.r, 4, 16)
    _decode_steps(c, slots, 8)


@pytest.mark.parametrize("st,io,gate,H,K,V,B", [
    (1, 1, rsc.KDA, 3, 128, 128, 5),     # Kimi-shaped heads, ragged head count
    (0, 1, rsc.GDN, 2, 128, 128, 3),     # GDN: fp32 state with bf16 io
    (1, 1, rsc.GDN, 2, 64, 128, 1),      # K != V, single request
    (0, 0, rsc.KDA, 1, 128, 64, 7),      # fp32, K != V
    (1, 0, rsc.KDA, 2, 64, 64, 2),       # bf16 state with fp32 io
])
def test_decode_variants(cuda_dev, st, io, gate, H, K, V, B):
    c = Case(cuda_dev, 1, L=2, P=9, H=H, K=K, V=V, st=st, io=io, gate=gate)
    slots = inputs.distinct_slots(c.r, B, 9)
    _decode_steps(c, slots, 3)


@pytest.mark.parametrize("st,io,gate,H,B", [(1, 1, rsc.KDA, 10, 64), (0, 1, rsc.GDN, 32, 20)])
def test_decode_large_batch(cuda_dev, st, io, gate, H, B):
    """More CTAs than the GPU holds at once (several per SM, the headline's regime), plain and
    overlapped launches, against the oracle."""
    c = Case(cuda_dev, 9, L=2, P=B + 4, H=H, K=128, V=128, st=st, io=io, gate=gate)
    slots = inputs.distinct_slots(c.r, B, B + 4)
    slots_d = to_dev(slots, c.dev)
    for layer, overlap in ((0, False), (1, True)):
        x = c.proj((B,))
        g, beta = c.gates((B,))
        o_ref = oracle.decode_step(c.ref, layer, slots, x, c.w, g, beta)
        o = rsc.kda_decode_step(c.pool, layer, slots_d, to_dev(x, c.dev), c.w_dev,
                                to_dev(g, c.dev), to_dev(beta, c.dev), overlap=overlap)
        assert max_rel_err(widen(to_np(o)), widen(o_ref)) <= tol(st, io)
    c.check_pool()


def test_decode_padding_slot_zero_is_legal(cuda_dev):
    c = Case(cuda_dev, 2, L=1, P=4, H=2, K=64, V=64, st=1, io=1, gate=rsc.KDA)
    _decode_steps(c, np.int32([0, 3]), 2)


def test_decode_bad_slot_sets_flag_and_skips_row(cuda_dev):
    c = Case(cuda_dev, 3, L=1, P=4, H=2, K=64, V=64, st=0, io=0, gate=rsc.KDA)
    before_s, before_c = to_np(c.pool.ssm).copy(), to_np(c.pool.conv).copy()
    slots = np.int32([2, 7])  # 7 > P
    x = c.proj((2,))
    g, beta = c.gates((2,))
    rsc.kda_decode_step(c.pool, 0, to_dev(slots, c.dev), to_dev(x, c.dev), c.w_dev,
                        to_dev(g, c.dev), to_dev(beta, c.dev))
    assert rsc.rsc_get_device_error(c.pool) == rsc.binding.DEVERR_SLOT
    assert rsc.rsc_get_device_error(c.pool) == 0  # read clears
    # row 0 (slot 2) was processed; nothing else moved
    s_now, c_now = to_np(c.pool.ssm), to_np(c.pool.conv)
    others = [0, 1, 3, 4]
    assert np.array_equal(s_now[0, others], before_s[0, others])
    assert np.array_equal(c_now[0, others], before_c[0, others])
    o_ref = oracle.decode_step(c.ref, 0, slots[:1], x[:1], c.w, g[:1], beta[:1])
    assert np.array_equal(c_now[0, 2], c.ref.conv[0, 2])
    assert max_rel_err(widen(s_now[0, 2]), widen(c.ref.ssm[0, 2])) <= TOL[0]


@pytest.mark.parametrize("st,io,gate,H,K,V,B", [
    (1, 1, rsc.KDA, 3, 128, 128, 5),
    (0, 1, rsc.GDN, 2, 128, 128, 3),
])
def test_decode_overlap_layer_chain(cuda_dev, st, io, gate, H, K, V, B):
    """kda_decode_step_overlap over a chain of layers on one stream, no synchronisation
    between calls: each layer's qkv is produced by a torch kernel launched right before its
    decode (the input the kernel must wait for), the other layers' decodes are the pending
    work its early state reads overlap.  Against the oracle, and bit-identical to the plain
    launch on a copy of the pool."""
    L, P, steps = 4, 9, 2
    c = Case(cuda_dev, 7, L=L, P=P, H=H, K=K, V=V, st=st, io=io, gate=gate)
    plain = rsc.SlotPool(L, P, H, K, V, st, io, gate, cuda_dev, ssm=c.pool.ssm.clone(),
                         conv=c.pool.conv.clone())
    slots = inputs.distinct_slots(c.r, B, P)
    slots_d = to_dev(slots, c.dev)
    for _ in range(steps):
        xs = [c.proj((B,)) for _ in range(L)]
        gb = [c.gates((B,)) for _ in range(L)]
        src = [to_dev(x, c.dev) for x in xs]
        gd = [(to_dev(g, c.dev), to_dev(b, c.dev)) for g, b in gb]
        torch.cuda.synchronize()
        outs, outs_plain = [], []
        for l in range(L):
            x = torch.zeros_like(src[l])
            torch.mul(src[l], 1, out=x)  # produced by a kernel just before the decode
            outs.append(rsc.kda_decode_step(c.pool, l, slots_d, x, c.w_dev, gd[l][0], gd[l][1],
                                            overlap=True))
        for l in range(L):
            outs_plain.append(rsc.kda_decode_step(plain, l, slots_d, src[l], c.w_dev, gd[l][0],
                                                  gd[l][1]))
        torch.cuda.synchronize()
        for l in range(L):
            o_ref = oracle.decode_step(c.ref, l, slots, xs[l], c.w, gb[l][0], gb[l][1])
            err = max_rel_err(widen(to_np(outs[l])), widen(o_ref))
            assert err <= tol(c.st, c.io), f"layer {l}: output max rel err {err}"
            assert torch.equal(outs[l], outs_plain[l]), f"layer {l}: overlap != plain"
    c.check_pool()
    assert torch.equal(c.pool.ssm, plain.ssm) and torch.equal(c.pool.conv, plain.conv)
    assert rsc.rsc_get_device_error(plain) == 0


@pytest.mark.parametrize("st", [0, 1])
def test_decode_overlap_graph_replayed_back_to_back(cuda_dev, st):
    """Every call overlapped, nothing in between: a CUDA graph of the two layers' decodes (one
    request, one head, so each launch is a single small CTA and nothing but the library's
    own ordering keeps a launch from running ahead) replayed 50 times without
    synchronisation.  Layer 0 of each step follows layer 1 of the step before, whose
    kernel was itself still free to start while layer 0 of that step ran; the early reads
    of layer 0 must still see layer 0's previous write.  Against 51 oracle steps (the
    capture helper runs the graph's calls once before capturing)."""
    import bench
    L, P, H, K, V, B, replays = 2, 3, 1, 128, 128, 1, 50
    c = Case(cuda_dev, 13, L=L, P=P, H=H, K=K, V=V, st=st, io=st, gate=rsc.KDA)
    slots = np.int32([2])
    slots_d = to_dev(slots, c.dev)
    xs = [c.proj((B,)) for _ in range(L)]
    gb = [c.gates((B,)) for _ in range(L)]
    xd = [to_dev(x, c.dev) for x in xs]
    gd = [(to_dev(g, c.dev), to_dev(b, c.dev)) for g, b in gb]
    outs = [torch.empty((B, H, V), dtype=c.pool.io_dtype, device=c.dev) for _ in range(L)]
    stream = torch.cuda.Stream(device=c.dev)

    def step():
        for l in range(L):
            rsc.kda_decode_step(c.pool, l, slots_d, xd[l], c.w_dev, gd[l][0], gd[l][1],
                                out=outs[l], stream=stream, overlap=True)

    graph = bench.graph_of(step, stream)
    with torch.cuda.stream(stream):
        for _ in range(replays):
            graph.replay()
    torch.cuda.synchronize()
    for _ in range(replays + 1):
        o_ref = [oracle.decode_step(c.ref, l, slots, xs[l], c.w, gb[l][0], gb[l][1])
                 for l in range(L)]
    for l in range(L):
        err = max_rel_err(widen(to_np(outs[l])), widen(o_ref[l]))
        assert err <= tol(c.st, c.io), f"layer {l}: output max rel err {err}"
    c.check_pool()


def test_decode_overlap_bad_slot_sets_flag_and_skips_row(cuda_dev):
    """The overlapped launch reads the slot id before waiting for the previous kernel; a bad
    one ends those CTAs before the wait with the error bit set and their rows untouched, and
    the next call on the stream runs normally."""
    c = Case(cuda_dev, 10, L=2, P=4, H=2, K=128, V=128, st=1, io=1, gate=rsc.KDA)
    before_s, before_c = to_np(c.pool.ssm).copy(), to_np(c.pool.conv).copy()
    slots = np.int32([3, 9])  # 9 > P
    x = c.proj((2,))
    g, beta = c.gates((2,))
    rsc.kda_decode_step(c.pool, 0, to_dev(slots, c.dev), to_dev(x, c.dev), c.w_dev,
                        to_dev(g, c.dev), to_dev(beta, c.dev), overlap=True)
    good = np.int32([1, 2])
    x2 = c.proj((2,))
    g2, beta2 = c.gates((2,))
    o2 = rsc.kda_decode_step(c.pool, 1, to_dev(good, c.dev), to_dev(x2, c.dev), c.w_dev,
                             to_dev(g2, c.dev), to_dev(beta2, c.dev), overlap=True)
    assert rsc.rsc_get_device_error(c.pool) == rsc.binding.DEVERR_SLOT
    s_now, c_now = to_np(c.pool.ssm), to_np(c.pool.conv)
    others = [0, 1, 2, 4]
    assert np.array_equal(s_now[0, others], before_s[0, others])
    assert np.array_equal(c_now[0, others], before_c[0, others])
    oracle.decode_step(c.ref, 0, slots[:1], x[:1], c.w, g[:1], beta[:1])
    o2_ref = oracle.decode_step(c.ref, 1, good, x2, c.w, g2, beta2)
    assert max_rel_err(widen(to_np(o2)), widen(o2_ref)) <= tol(1, 1)
    c.check_pool()


# ------------------------------------------------------------------ slot copy

@pytest.mark.parametrize("st,io,layer", [(1, 1, -1), (0, 1, 1), (0, 0, -1)])
def test_slot_copy_bit_exact(cuda_dev, st, io, layer):
    c = Case(cuda_dev, 4, L=3, P=12, H=2, K=128, V=64, st=st, io=io, gate=rsc.KDA)
    perm = c.r.permutation(12) + 1
    src, dst = perm[:4].astype(np.int32), perm[4:8].astype(np.int32)
    mask = np.uint8([1, 0, 1, 1])
    rsc.ssm_slot_copy(c.pool, layer, to_dev(src, c.dev), to_dev(dst, c.dev), to_dev(mask, c.dev))
    oracle.slot_copy(c.ref, layer, src, dst, mask)
    assert np.array_equal(to_np(c.pool.ssm), c.ref.ssm)
    assert np.array_equal(to_np(c.pool.conv), c.ref.conv)


def test_slot_copy_bad_slot_flags(cuda_dev):
    c = Case(cuda_dev, 5, L=1, P=4, H=1, K=64, V=64, st=1, io=1, gate=rsc.KDA)
    before = to_np(c.pool.ssm).copy()
    rsc.ssm_slot_copy(c.pool, 0, to_dev(np.int32([1, 9]), c.dev), to_dev(np.int32([2, 3]), c.dev))
    assert rsc.rsc_get_device_error(c.pool) == rsc.binding.DEVERR_SLOT
    now = to_np(c.pool.ssm)
    assert np.array_equal(now[0, 2], before[0, 1])
    assert np.array_equal(now[0, 3], before[0, 3])


# ------------------------------------------------------------------ spec verify / commit

@pytest.mark.parametrize("st,io,gate,K,V", [(1, 1, rsc.KDA, 128, 128), (0, 0, rsc.KDA, 64, 64),
                                            (0, 1, rsc.GDN, 128, 64)])
def test_spec_verify_and_commit(cuda_dev, st, io, gate, K, V):
    H, B, T, L = 2, 5, 8, 16
    c = Case(cuda_dev, 6, L=1, P=10, H=H, K=K, V=V, st=st, io=io, gate=gate)
    slots = inputs.distinct_slots(c.r, B, 10)
    x = c.proj((B, T))
    g, beta = c.gates((B, T))
    sS_ref, sC_ref, o_ref = oracle.spec_verify(c.ref, 0, slots, T, L, x, c.w, g, beta)
    sdt = rsc.binding.TORCH_DTYPE[st]
    spec_ssm = torch.zeros((B, L, H, V, K), dtype=sdt, device=c.dev)
    spec_conv = torch.zeros((B, L, 3, c.D), dtype=c.pool.io_dtype, device=c.dev)
    before = to_np(c.pool.ssm).copy(), to_np(c.pool.conv).copy()
    slots_d = to_dev(slots, c.dev)
    o = rsc.kda_spec_verify_commit(c.pool, 0, rsc.VERIFY, slots_d, T, L, spec_ssm, spec_conv,
                                   to_dev(x, c.dev), c.w_dev, to_dev(g, c.dev),
                                   to_dev(beta, c.dev))
    assert np.array_equal(to_np(c.pool.ssm), before[0]) and np.array_equal(to_np(c.pool.conv), before[1])
    assert max_rel_err(widen(to_np(o)), widen(o_ref)) <= tol(st, io)
    assert np.array_equal(to_np(spec_conv)[:, :T], sC_ref[:, :T])
    for t in range(T):
        assert max_rel_err(widen(to_np(spec_ssm)[:, t]), widen(sS_ref[:, t])) <= TOL[st], t
    accept = inputs.accept_counts(c.r, B, T)
    rsc.kda_spec_verify_commit(c.pool, 0, rsc.COMMIT, slots_d, T, L, spec_ssm, spec_conv,
                               accept=to_dev(accept, c.dev))
    # commit is a byte gather of the device's own cache entries
    gs, gc = to_np(spec_ssm), to_np(spec_conv)
    now_s, now_c = to_np(c.pool.ssm), to_np(c.pool.conv)
    for b, s in enumerate(slots):
        assert np.array_equal(now_s[0, s], gs[b, accept[b]])
        assert np.array_equal(now_c[0, s], gc[b, accept[b]])
    oracle.spec_commit(c.ref, 0, slots, T, L, sS_ref, sC_ref, accept)
    c.check_pool()


def test_spec_commit_bad_accept_flags(cuda_dev):
    c = Case(cuda_dev, 7, L=1, P=4, H=1, K=64, V=64, st=1, io=1, gate=rsc.KDA)
    B, T, L = 2, 3, 4
    spec_ssm = torch.ones((B, L, 1, 64, 64), dtype=torch.bfloat16, device=c.dev)
    spec_conv = torch.ones((B, L, 3, c.D), dtype=torch.bfloat16, device=c.dev)
    before = to_np(c.pool.ssm).copy()
    rsc.kda_spec_verify_commit(c.pool, 0, rsc.COMMIT, to_dev(np.int32([1, 2]), c.dev), T, L,
                               spec_ssm, spec_conv, accept=to_dev(np.int32([1, 3]), c.dev))
    assert rsc.rsc_get_device_error(c.pool) == rsc.binding.DEVERR_ACCEPT
    now = to_np(c.pool.ssm)
    assert np.array_equal(now[0, 2], before[0, 2])
    assert np.all(widen(now[0, 1]) == 1.0)


# ------------------------------------------------------------------ fused gating

@pytest.mark.parametrize("st,io,gate,K,V", [
    (0, 0, rsc.KDA, 64, 64), (1, 1, rsc.KDA, 128, 128), (0, 1, rsc.GDN, 128, 128),
    (1, 0, rsc.GDN, 64, 128), (1, 1, rsc.KDA, 64, 128),
])
def test_decode_gated_parity(cuda_dev, st, io, gate, K, V):
    """Gates formed in the kernel from raw projections: outputs, states and windows match the
    oracle's gating followed by its decode step, over two steps."""
    H, B = 3, 5
    c = Case(cuda_dev, 34, L=2, P=9, H=H, K=K, V=V, st=st, io=io, gate=gate)
    n = K if gate == rsc.KDA else 1
    slots = inputs.distinct_slots(c.r, B, 9)
    A_log = c.r.normal(0, 0.5, size=(H,)).astype(np.float32)
    dt = c.r.normal(0, 1, size=(H, n)).astype(np.float32)
    dt_dev = to_dev(dt if n > 1 else dt[:, 0].copy(), c.dev)
    for _ in range(2):
        x = c.proj((B,))
        a = c.r.normal(0, 2, size=(B, H, n)).astype(np.float32)
        b = c.r.normal(0, 2, size=(B, H)).astype(np.float32)
        o_ref = oracle.decode_step_gated(c.ref, 1, slots, x, c.w, a, b, A_log, dt)
        a_dev = to_dev(a if n > 1 else a[:, :, 0].copy(), c.dev)
        o = rsc.kda_decode_step_gated(c.pool, 1, to_dev(slots, c.dev), to_dev(x, c.dev), c.w_dev,
                                      a_dev, to_dev(b, c.dev), to_dev(A_log, c.dev), dt_dev)
        assert max_rel_err(widen(to_np(o)), widen(o_ref)) <= tol(st, io)
    c.check_pool()


@pytest.mark.parametrize("st,io,K,V", [(0, 0, 64, 64), (1, 1, 128, 128), (0, 1, 128, 64)])
def test_decode_track_parity(cuda_dev, st, io, K, V):
    """Tracking fused into decode: masked requests' track slots receive the updated state and
    window bit for bit (the same bytes as the active slot), unmasked track slots and all other
    rows match the oracle's decode followed by its masked copy."""
    H, B = 2, 4
    c = Case(cuda_dev, 35, L=2, P=12, H=H, K=K, V=V, st=st, io=io, gate=rsc.KDA)
    slots = np.int32([2, 5, 7, 9])
    track = np.int32([11, 1, 12, 3])
    mask = np.uint8([1, 0, 1, 1])
    x = c.proj((B,))
    g, beta = c.gates((B,))
    o_ref = oracle.decode_step_track(c.ref, 1, slots, x, c.w, g, beta, mask, track)
    o = rsc.kda_decode_step_track(c.pool, 1, to_dev(slots, c.dev), to_dev(x, c.dev), c.w_dev,
                                  to_dev(g, c.dev), to_dev(beta, c.dev), to_dev(mask, c.dev),
                                  to_dev(track, c.dev))
    assert max_rel_err(widen(to_np(o)), widen(o_ref)) <= tol(st, io)
    ssm, conv = to_np(c.pool.ssm), to_np(c.pool.conv)
    for b in range(B):
        if mask[b]:
            assert np.array_equal(ssm[1, track[b]], ssm[1, slots[b]])
            assert np.array_equal(conv[1, track[b]], conv[1, slots[b]])
    c.check_pool()


@pytest.mark.parametrize("st,io,gate,K,V", [(1, 1, rsc.KDA, 128, 128), (0, 0, rsc.GDN, 64, 64)])
def test_decode_ex_gating_tracking_overlap(cuda_dev, st, io, gate, K, V):
    """kda_decode_step_ex with every option at once -- gates formed from raw projections, the
    track copy fused, the overlapped launch -- over a chain of three layers: against the
    oracle's gating followed by its decode and masked track copy, and bit-identical to the
    same options without the overlap on a copy of the pool."""
    H, B, L, P = 2, 4, 3, 12
    c = Case(cuda_dev, 36, L=L, P=P, H=H, K=K, V=V, st=st, io=io, gate=gate)
    plain = rsc.SlotPool(L, P, H, K, V, st, io, gate, cuda_dev, ssm=c.pool.ssm.clone(),
                         conv=c.pool.conv.clone())
    n = K if gate == rsc.KDA else 1
    slots = np.int32([2, 5, 7, 9])
    track = np.int32([11, 1, 12, 3])
    mask = np.uint8([1, 0, 1, 1])
    A_log = c.r.normal(0, 0.5, size=(H,)).astype(np.float32)
    dt = c.r.normal(0, 1, size=(H, n)).astype(np.float32)
    dev = lambda a: to_dev(a, c.dev)
    dt_dev = dev(dt if n > 1 else dt[:, 0].copy())
    xs = [c.proj((B,)) for _ in range(L)]
    raws = [(c.r.normal(0, 2, size=(B, H, n)).astype(np.float32),
             c.r.normal(0, 2, size=(B, H)).astype(np.float32)) for _ in range(L)]
    a_dev = [dev(a if n > 1 else a[:, :, 0].copy()) for a, _ in raws]
    b_dev = [dev(b) for _, b in raws]
    args = dict(A_log=dev(A_log), dt_bias=dt_dev, track_mask=dev(mask), track_slots=dev(track))
    sl = dev(slots)
    torch.cuda.synchronize()
    outs = [rsc.kda_decode_step_ex(c.pool, l, sl, dev(xs[l]), c.w_dev, a_dev[l], b_dev[l],
                                   overlap=True, **args) for l in range(L)]
    outs_plain = [rsc.kda_decode_step_ex(plain, l, sl, dev(xs[l]), c.w_dev, a_dev[l], b_dev[l],
                                         **args) for l in range(L)]
    torch.cuda.synchronize()
    for l in range(L):
        g, beta = oracle.gates_from_raw(c.ref, raws[l][0], raws[l][1], A_log, dt)
        o_ref = oracle.decode_step_track(c.ref, l, slots, xs[l], c.w, g, beta, mask, track)
        assert max_rel_err(widen(to_np(outs[l])), widen(o_ref)) <= tol(st, io), f"layer {l}"
        assert torch.equal(outs[l], outs_plain[l]), f"layer {l}: overlap != plain"
    c.check_pool()
    assert torch.equal(c.pool.ssm, plain.ssm) and torch.equal(c.pool.conv, plain.conv)


def test_allocator_track_plan_and_fused_track_copy(cuda_dev):
    """Host slot management driving the fused track copy: live and ping-pong track slots from
    the allocator, the plan of two steps (lengths crossing the interval), each tracked
    request's snapshot landing in the track slot the plan chose, bit for bit."""
    from recurrent_state_cache_gb300 import binding
    H, K, V, B, P = 2, 64, 64, 3, 16
    c = Case(cuda_dev, 36, L=1, P=P, H=H, K=K, V=V, st=1, io=1, gate=rsc.KDA)
    alloc = binding.SlotAllocator(P)
    live = alloc.acquire(B)
    pairs = alloc.acquire(2 * B).reshape(B, 2)
    nxt = np.zeros(B, np.int32)
    lens = np.int32([255, 256, 511])
    for step in range(2):
        lens = lens + 1  # the token of this step
        mask, track = binding.track_plan(lens, 256, pairs, nxt)
        x = c.proj((B,))
        g, beta = c.gates((B,))
        oracle.decode_step_track(c.ref, 0, live, x, c.w, g, beta, mask, track)
        rsc.kda_decode_step_track(c.pool, 0, to_dev(live, c.dev), to_dev(x, c.dev), c.w_dev,
                                  to_dev(g, c.dev), to_dev(beta, c.dev), to_dev(mask, c.dev),
                                  to_dev(track, c.dev))
        ssm, conv = to_np(c.pool.ssm), to_np(c.pool.conv)
        for bb in range(B):
            if mask[bb]:
                assert np.array_equal(ssm[0, track[bb]], ssm[0, live[bb]])
                assert np.array_equal(conv[0, track[bb]], conv[0, live[bb]])
    # lengths 256 (step 0: request 0) and 512 (step 0: request 2; step 1: none) were tracked
    assert nxt.tolist() == [1, 0, 1]
    c.check_pool()
    alloc.release(np.concatenate([live, pairs.ravel()]))
    assert alloc.free_count() == P


# ------------------------------------------------------------------ ReplaySSM

def _rings_np(rings):
    return {n: to_np(getattr(rings, n)) for n in ("d", "k", "rawv", "rawk", "g", "beta")}


@pytest.mark.parametrize("st,io,gate,K,V,T,depth", [
    (0, 0, rsc.KDA, 64, 64, 5, 16), (1, 1, rsc.KDA, 128, 128, 5, 16),
    (1, 1, rsc.GDN, 128, 128, 5, 16), (0, 1, rsc.KDA, 128, 64, 5, 16),
    (1, 0, rsc.KDA, 64, 128, 5, 16),
    (1, 1, rsc.KDA, 128, 128, 8, 16),   # one full block of eight tokens
    (1, 0, rsc.KDA, 128, 128, 7, 16),   # fp32 io on the tensor-core verify
    (0, 0, rsc.KDA, 128, 128, 11, 32),  # a full block, then three tokens from its end state
    (1, 1, rsc.GDN, 64, 64, 16, 32),    # two full blocks
])
def test_replay_verify_commit_parity(cuda_dev, st, io, gate, K, V, T, depth):
    """Verify: outputs and ring records match the oracle, windows bit-exact, slot untouched;
    commit: the replayed state matches the oracle's replay, windows bit-exact."""
    H, B = 2, 3
    c = Case(cuda_dev, 31, L=2, P=6, H=H, K=K, V=V, st=st, io=io, gate=gate)
    slots = np.int32([5, 2, 4])
    pos = np.int32([0, 9, 14])  # the last request wraps around its ring
    x = c.proj((B, T))
    g, beta = c.gates((B, T))
    rings_ref = oracle.Rings(c.ref, depth)
    sC_ref, o_ref = oracle.replay_verify(c.ref, rings_ref, 1, slots, pos, T, depth, x, c.w, g, beta)
    rings = rsc.ReplayRings(c.pool, depth)
    spec_conv = torch.zeros((B, depth, 3, c.D), dtype=c.pool.io_dtype, device=c.dev)
    before = to_np(c.pool.ssm).copy(), to_np(c.pool.conv).copy()
    slots_d, pos_d = to_dev(slots, c.dev), to_dev(pos, c.dev)
    o = rsc.kda_replay_verify_commit(c.pool, rings, 1, rsc.VERIFY, slots_d, pos_d, T, spec_conv,
                                     to_dev(x, c.dev), c.w_dev, to_dev(g, c.dev), to_dev(beta, c.dev))
    assert np.array_equal(to_np(c.pool.ssm), before[0]) and np.array_equal(to_np(c.pool.conv), before[1])
    assert max_rel_err(widen(to_np(o)), widen(o_ref)) <= tol(st, io)
    assert np.array_equal(to_np(spec_conv)[:, :T], sC_ref[:, :T])
    got = _rings_np(rings)
    for name in ("d", "k", "rawv", "rawk"):
        assert max_rel_err(widen(got[name]), widen(getattr(rings_ref, name))) <= TOL[st], name
    g_ref = rings_ref.g if gate == rsc.KDA else rings_ref.g[..., 0]
    assert np.array_equal(got["g"], g_ref) and np.array_equal(got["beta"], rings_ref.beta)
    assert rsc.rsc_get_device_error(c.pool) == 0
    accept = np.int32([0, T - 1, T // 2])
    rsc.kda_replay_verify_commit(c.pool, rings, 1, rsc.COMMIT, slots_d, pos_d, T, spec_conv,
                                 accept=to_dev(accept, c.dev))
    oracle.replay_commit(c.ref, rings_ref, 1, slots, pos, T, depth, sC_ref, accept)
    c.check_pool()


@pytest.mark.parametrize("st", [0, 1])
def test_replay_commit_lands_on_the_snapshot_commit(cuda_dev, st):
    """On the GPU, the replay path's commit(a) and the snapshot path's commit(a) agree (both
    from the same slot state and inputs): to fp32 rounding with fp32 records, to the bf16 bar
    with bf16 records; windows bit-exact."""
    H, K, V, B, T, depth = 2, 128, 128, 4, 8, 16
    c = Case(cuda_dev, 32, L=1, P=8, H=H, K=K, V=V, st=st, io=st, gate=rsc.KDA)
    c2 = Case(cuda_dev, 32, L=1, P=8, H=H, K=K, V=V, st=st, io=st, gate=rsc.KDA)  # same seed
    slots = to_dev(np.int32([7, 1, 3, 5]), c.dev)
    pos = to_dev(np.int32([3, 8, 15, 0]), c.dev)
    x = c.proj((B, T))
    g, beta = c.gates((B, T))
    accept = to_dev(np.int32([7, 0, 3, 5]), c.dev)
    args = (to_dev(x, c.dev), c.w_dev, to_dev(g, c.dev), to_dev(beta, c.dev))
    rings = rsc.ReplayRings(c.pool, depth)
    sc1 = torch.zeros((B, depth, 3, c.D), dtype=c.pool.io_dtype, device=c.dev)
    rsc.kda_replay_verify_commit(c.pool, rings, 0, rsc.VERIFY, slots, pos, T, sc1, *args)
    rsc.kda_replay_verify_commit(c.pool, rings, 0, rsc.COMMIT, slots, pos, T, sc1, accept=accept)
    ss2 = torch.zeros((B, depth, H, V, K), dtype=c2.pool.ssm.dtype, device=c.dev)
    sc2 = torch.zeros((B, depth, 3, c.D), dtype=c2.pool.io_dtype, device=c.dev)
    rsc.kda_spec_verify_commit(c2.pool, 0, rsc.VERIFY, slots, T, depth, ss2, sc2, *args)
    rsc.kda_spec_verify_commit(c2.pool, 0, rsc.COMMIT, slots, T, depth, ss2, sc2, accept=accept)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(c.pool.conv), to_np(c2.pool.conv))
    bar = 1e-5 if st == 0 else TOL[1]
    assert max_rel_err(widen(to_np(c.pool.ssm)), widen(to_np(c2.pool.ssm))) <= bar
    assert rsc.rsc_get_device_error(c.pool) == 0 and rsc.rsc_get_device_error(c2.pool) == 0


def test_replay_bad_ring_position_flags(cuda_dev):
    c = Case(cuda_dev, 33, L=1, P=4, H=1, K=64, V=64, st=1, io=1, gate=rsc.KDA)
    B, T, depth = 2, 3, 8
    rings = rsc.ReplayRings(c.pool, depth)
    spec_conv = torch.zeros((B, depth, 3, c.D), dtype=c.pool.io_dtype, device=c.dev)
    before = to_np(c.pool.ssm).copy()
    slots = to_dev(np.int32([1, 2]), c.dev)
    rsc.kda_replay_verify_commit(c.pool, rings, 0, rsc.COMMIT, slots, to_dev(np.int32([0, depth]), c.dev),
                                 T, spec_conv, accept=to_dev(np.int32([1, 1]), c.dev))
    assert rsc.rsc_get_device_error(c.pool) == rsc.binding.DEVERR_RING
    assert np.array_equal(to_np(c.pool.ssm)[0, 2], before[0, 2])


# ------------------------------------------------------------------ prefill

@pytest.mark.parametrize("st,io,gate,K,V,lens,init", [
    # blocked path, K = 64 (fp32 and bf16 state, 2 key channels a lane)
    (0, 0, rsc.KDA, 64, 64, [1, 70, 2, 129], [1, 1, 0, 1]),
    (1, 1, rsc.KDA, 64, 128, [65, 3], [1, 0]),
    (1, 0, rsc.GDN, 64, 64, [9, 40], [0, 1]),
    # blocked path, fp32 state, K = 128: whole and ragged 8-token blocks
    (0, 1, rsc.GDN, 128, 128, [200], [1]),
    (0, 0, rsc.KDA, 128, 128, [1, 7, 8, 9, 200], [1, 0, 1, 1, 0]),
    (0, 1, rsc.KDA, 128, 64, [70, 3], [0, 1]),
    (0, 0, rsc.GDN, 128, 64, [33, 16, 2], [1, 1, 0]),
    # chunkwise tensor-core path (bf16 state, K = 128): ragged chunks, fresh / continued
    (1, 1, rsc.KDA, 128, 128, [64, 1, 131], [1, 0, 1]),
    (1, 1, rsc.KDA, 128, 128, [300], [1]),
    (1, 1, rsc.KDA, 128, 64, [200, 7], [1, 1]),
    (1, 0, rsc.GDN, 128, 128, [130, 63], [0, 1]),
])
def test_prefill_parity(cuda_dev, st, io, gate, K, V, lens, init):
    H = 2
    c = Case(cuda_dev, 8, L=2, P=8, H=H, K=K, V=V, st=st, io=io, gate=gate)
    N = len(lens)
    slots = inputs.distinct_slots(c.r, N, 8)
    cu = inputs.cu_seqlens(lens)
    T = int(cu[-1])
    x = c.proj((T,))
    g, beta = c.gates((T,))
    hi = np.uint8(init)
    o_ref = oracle.prefill(c.ref, 1, slots, cu, x, c.w, g, beta, has_init=hi)
    o = rsc.kda_prefill_chunk(c.pool, 1, to_dev(slots, c.dev), to_dev(cu, c.dev),
                              to_dev(x, c.dev), c.w_dev, to_dev(g, c.dev), to_dev(beta, c.dev),
                              has_initial_state=to_dev(hi, c.dev))
    tc = st == 1 and K == 128  # the chunkwise tensor-core path
    assert max_rel_err(widen(to_np(o)), widen(o_ref), tc=tc) <= tol(st, io)
    c.check_pool(tc=tc)


@pytest.mark.parametrize("gate,V", [(rsc.KDA, 128), (rsc.GDN, 64)])
def test_prefill_many_packed_sequences(cuda_dev, gate, V):
    """The tensor-core path over 24 packed sequences: empty ones (fresh and continued), single
    tokens, exact multiples of the 64-token chunk, ragged tails; every output, state and
    window against the oracle (the windows written by the state pass, bit for bit)."""
    H, K = 2, 128
    c = Case(cuda_dev, 14, L=1, P=30, H=H, K=K, V=V, st=1, io=1, gate=gate)
    lens = [0, 1, 64, 0, 2, 3, 128, 65, 17, 0, 191, 64, 1, 5, 250, 63, 0, 33, 129, 2, 70, 3, 0, 96]
    init = [1, 0, 1, 0, 1, 0, 1, 1, 0, 1, 0, 1, 0, 1, 1, 0, 1, 1, 0, 1, 0, 1, 1, 0]
    N = len(lens)
    slots = inputs.distinct_slots(c.r, N, 30)
    cu = inputs.cu_seqlens(lens)
    T = int(cu[-1])
    x = c.proj((T,))
    g, beta = c.gates((T,))
    hi = np.uint8(init)
    o_ref = oracle.prefill(c.ref, 0, slots, cu, x, c.w, g, beta, has_init=hi)
    o = rsc.kda_prefill_chunk(c.pool, 0, to_dev(slots, c.dev), to_dev(cu, c.dev),
                              to_dev(x, c.dev), c.w_dev, to_dev(g, c.dev), to_dev(beta, c.dev),
                              has_initial_state=to_dev(hi, c.dev))
    assert max_rel_err(widen(to_np(o)), widen(o_ref), tc=True) <= TOL[1]
    c.check_pool(tc=True)


@pytest.mark.parametrize("st,K", [(1, 128), (0, 64)])
def test_prefill_call_of_empty_sequences(cuda_dev, st, K):
    """A call whose sequences are all empty (zero tokens): fresh ones get a zero state and
    window, continued ones keep theirs; the rest of the pool is untouched."""
    c = Case(cuda_dev, 15, L=1, P=6, H=2, K=K, V=64, st=st, io=st, gate=rsc.KDA)
    lens, init = [0, 0, 0], [1, 0, 1]
    slots = np.int32([4, 1, 6])
    cu = inputs.cu_seqlens(lens)
    x = c.proj((0,))
    g, beta = c.gates((0,))
    hi = np.uint8(init)
    oracle.prefill(c.ref, 0, slots, cu, x, c.w, g, beta, has_init=hi)
    rsc.kda_prefill_chunk(c.pool, 0, to_dev(slots, c.dev), to_dev(cu, c.dev), to_dev(x, c.dev),
                          c.w_dev, to_dev(g, c.dev), to_dev(beta, c.dev),
                          has_initial_state=to_dev(hi, c.dev))
    c.check_pool(tc=st == 1 and K == 128)


def test_prefill_bad_cu_seqlens_flags(cuda_dev):
    c = Case(cuda_dev, 9, L=1, P=4, H=1, K=64, V=64, st=0, io=0, gate=rsc.KDA)
    x = c.proj((10,))
    g, beta = c.gates((10,))
    before = to_np(c.pool.ssm).copy()
    rsc.kda_prefill_chunk(c.pool, 0, to_dev(np.int32([1]), c.dev), to_dev(np.int32([0, 12]), c.dev),
                          to_dev(x, c.dev), c.w_dev, to_dev(g, c.dev), to_dev(beta, c.dev))
    assert rsc.rsc_get_device_error(c.pool) & rsc.binding.DEVERR_SEQ
    assert np.array_equal(to_np(c.pool.ssm), before)


def test_prefill_kimi_shaped_chunk(cuda_dev):
    """12 heads, K=V=128, bf16: the 1312-token last chunk of the 13600-token prompt
    (20 full 64-token chunks and a ragged 32-token one), continued from a slot state."""
    H, K, V = 12, 128, 128
    c = Case(cuda_dev, 10, L=1, P=3, H=H, K=K, V=V, st=1, io=1, gate=rsc.KDA)
    T = 1312
    x = c.proj((T,))
    g, beta = c.gates((T,))
    cu = np.int32([0, T])
    o_ref = oracle.prefill(c.ref, 0, [2], cu, x, c.w, g, beta)
    o = rsc.kda_prefill_chunk(c.pool, 0, to_dev(np.int32([2]), c.dev), to_dev(cu, c.dev),
                              to_dev(x, c.dev), c.w_dev, to_dev(g, c.dev), to_dev(beta, c.dev))
    assert max_rel_err(widen(to_np(o)), widen(o_ref), tc=True) <= TOL[1]
    c.check_pool(tc=True)


def _strong_gates(c, T, mode):
    """Log-decay gates far beyond the usual draw: a constant -4 per token (a 64-token chunk
    spans 252, a 16-token block 60), -e^3 softplus(N(0,1)) everywhere (every 16-token block
    spans hundreds), or a mix: weak and strong stretches and channels, and full resets."""
    if mode == "const4":
        g, beta = c.gates((T,))
        return np.full_like(g, -4.0), beta
    if mode == "scale20":
        return inputs.gates(c.r, (T,), c.H, c.K, c.gate, scale=float(np.exp(3.0)))
    g, beta = c.gates((T,))
    g = g.copy()
    g[T // 3: 2 * T // 3, ..., : c.K // 2] *= 30.0
    g[c.r.integers(0, T, 4)] = -300.0
    return g, beta


@pytest.mark.parametrize("gate,V,lens,init,mode", [
    (rsc.KDA, 64, [64], [1], "const4"),
    (rsc.KDA, 128, [200, 70], [1, 0], "scale20"),
    (rsc.KDA, 128, [300], [1], "mixed"),
    (rsc.GDN, 128, [130, 63], [0, 1], "scale20"),
    (rsc.GDN, 64, [190], [1], "mixed"),
])
def test_prefill_strong_decay_matches_oracle(cuda_dev, gate, V, lens, init, mode):
    """The tensor-core prefill under decay far beyond the usual draw (the diagonal 16-token
    blocks then run exactly in fp32) against the oracle; no error bit."""
    H, K = 2, 128
    c = Case(cuda_dev, 11, L=1, P=4, H=H, K=K, V=V, st=1, io=1, gate=gate)
    N = len(lens)
    slots = inputs.distinct_slots(c.r, N, 4)
    cu = inputs.cu_seqlens(lens)
    T = int(cu[-1])
    x = c.proj((T,))
    g, beta = _strong_gates(c, T, mode)
    hi = np.uint8(init)
    o_ref = oracle.prefill(c.ref, 0, slots, cu, x, c.w, g, beta, has_init=hi)
    o = rsc.kda_prefill_chunk(c.pool, 0, to_dev(slots, c.dev), to_dev(cu, c.dev),
                              to_dev(x, c.dev), c.w_dev, to_dev(g, c.dev), to_dev(beta, c.dev),
                              has_initial_state=to_dev(hi, c.dev))
    assert max_rel_err(widen(to_np(o)), widen(o_ref), tc=True) <= TOL[1]
    c.check_pool(tc=True)


@pytest.mark.parametrize("gate,V,lens,init,mode", [
    (rsc.KDA, 128, [64, 13], [1, 0], "const4"),
    (rsc.KDA, 128, [200, 70], [1, 0], "scale20"),
    (rsc.KDA, 64, [300], [1], "mixed"),
    (rsc.GDN, 128, [130, 63], [0, 1], "scale20"),
    (rsc.KDA, 128, [77], [1], "grow"),
    (rsc.GDN, 64, [41], [1], "grow"),
])
def test_prefill_blocked_fp32_gates(cuda_dev, gate, V, lens, init, mode):
    """The blocked fp32 prefill under decay far beyond the usual draw, and under a growing
    gate (g = +0.5 per token, about e^4 per 8-token block), against the oracle at the fp32 bar;
    no error bit."""
    H, K = 2, 128
    c = Case(cuda_dev, 16, L=1, P=4, H=H, K=K, V=V, st=0, io=0, gate=gate)
    N = len(lens)
    slots = inputs.distinct_slots(c.r, N, 4)
    cu = inputs.cu_seqlens(lens)
    T = int(cu[-1])
    x = c.proj((T,))
    if mode == "grow":
        g, beta = c.gates((T,))
        g = np.full_like(g, 0.5)
    else:
        g, beta = _strong_gates(c, T, mode)
    hi = np.uint8(init)
    o_ref = oracle.prefill(c.ref, 0, slots, cu, x, c.w, g, beta, has_init=hi)
    o = rsc.kda_prefill_chunk(c.pool, 0, to_dev(slots, c.dev), to_dev(cu, c.dev),
                              to_dev(x, c.dev), c.w_dev, to_dev(g, c.dev), to_dev(beta, c.dev),
                              has_initial_state=to_dev(hi, c.dev))
    assert max_rel_err(widen(to_np(o)), widen(o_ref)) <= TOL[0]
    c.check_pool()


@pytest.mark.parametrize("gate,H,V,N", [(rsc.KDA, 12, 128, 8), (rsc.GDN, 16, 64, 10)])
def test_prefill_blocked_fp32_many_sequences(cuda_dev, gate, H, V, N):
    """Enough sequences x heads for the 32-row tiles of the blocked fp32 prefill (the smaller
    cases above run 8-row tiles); lengths cover empty, single-token, whole and ragged blocks."""
    K = 128
    c = Case(cuda_dev, 17, L=1, P=N + 2, H=H, K=K, V=V, st=0, io=1, gate=gate)
    lens = [0, 1, 8, 23, 64, 5, 17, 40, 9, 3][:N]
    init = [1, 0, 1, 1, 0, 1, 0, 1, 1, 0][:N]
    slots = inputs.distinct_slots(c.r, N, N + 2)
    cu = inputs.cu_seqlens(lens)
    T = int(cu[-1])
    x = c.proj((T,))
    g, beta = c.gates((T,))
    hi = np.uint8(init)
    o_ref = oracle.prefill(c.ref, 0, slots, cu, x, c.w, g, beta, has_init=hi)
    o = rsc.kda_prefill_chunk(c.pool, 0, to_dev(slots, c.dev), to_dev(cu, c.dev),
                              to_dev(x, c.dev), c.w_dev, to_dev(g, c.dev), to_dev(beta, c.dev),
                              has_initial_state=to_dev(hi, c.dev))
    assert max_rel_err(widen(to_np(o)), widen(o_ref)) <= tol(0, 1)
    c.check_pool()


def test_prefill_blocked_fp32_steep_growth_is_flagged(cuda_dev):
    """A growing gate that raises a log gate by more than 80 within an 8-token block (11 per
    token) sets RSC_DEVERR_GATE on the blocked fp32 path."""
    c = Case(cuda_dev, 18, L=1, P=2, H=1, K=128, V=64, st=0, io=0, gate=rsc.KDA)
    T = 16
    x = c.proj((T,))
    _, beta = c.gates((T,))
    g = np.full((T, 1, 128), 11.0, np.float32)
    rsc.kda_prefill_chunk(c.pool, 0, to_dev(np.int32([1]), c.dev), to_dev(np.int32([0, T]), c.dev),
                          to_dev(x, c.dev), c.w_dev, to_dev(g, c.dev), to_dev(beta, c.dev))
    assert rsc.rsc_get_device_error(c.pool) & rsc.binding.DEVERR_GATE


def test_prefill_growing_gate_is_flagged(cuda_dev):
    """A gate that grows the state (g > 0) by more than the tensor-core form represents
    within a chunk sets RSC_DEVERR_GATE; decaying gates never do (tests above)."""
    c = Case(cuda_dev, 12, L=1, P=2, H=1, K=128, V=64, st=1, io=1, gate=rsc.KDA)
    T = 64
    x = c.proj((T,))
    _, beta = c.gates((T,))
    g = np.full((T, 1, 128), 2.0, np.float32)  # grows by 126 over the chunk
    rsc.kda_prefill_chunk(c.pool, 0, to_dev(np.int32([1]), c.dev), to_dev(np.int32([0, T]), c.dev),
                          to_dev(x, c.dev), c.w_dev, to_dev(g, c.dev), to_dev(beta, c.dev))
    assert rsc.rsc_get_device_error(c.pool) & rsc.binding.DEVERR_GATE
