"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test below checks one oracle function against a closed form, a textbook special
case, a library routine, a brute-force unroll on tiny inputs, or numbers printed on the
pages (tests/golden).  They are chosen so that a dropped term, a wrong sign, a wrong
index or a transposed operand in the oracle fails at least one of them.
"""
import json
import os

import numpy as np
import pytest

import oracle
from recurrent_state_cache_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _unit_rows(r, T, K):
    x = r.standard_normal((T, K))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


def _head_case(seed, T, K, V, s0_std=0.3):
    r = np.random.default_rng(seed)
    q = _unit_rows(r, T, K)
    k = _unit_rows(r, T, K)
    v = r.standard_normal((T, V))
    g = -np.logaddexp(0.0, r.standard_normal((T, K)))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal(T)))
    S0 = r.standard_normal((V, K)) * s0_std
    return q, k, v, g, beta, S0


# ----------------------------------------------------------------------- storage dtype

def test_bf16_round_matches_torch_rne():
    torch = pytest.importorskip("torch")
    r = np.random.default_rng(1)
    x = (r.standard_normal(20000) * np.exp(r.uniform(-30, 30, 20000))).astype(np.float32)
    # exact ties (low half == 0x8000) with even and odd kept mantissa
    ties = (np.arange(1, 2001, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties, np.float32([0.0, -0.0, 1e-40, 3.0e38])])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round(x.astype(np.float64))
    assert np.array_equal(got, ref)


# ----------------------------------------------------------------------- short conv

@pytest.mark.parametrize("T", [1, 2, 3, 7])
def test_conv_is_direct_four_tap_filter(T):
    r = np.random.default_rng(2)
    D = 37
    win = r.standard_normal((3, D))
    x = r.standard_normal((T, D))
    w = r.standard_normal((D, 4)).astype(np.float32)
    new_win, y = oracle.conv_sequence(win, x, w)
    ext = np.concatenate([win, x], axis=0)  # oldest first
    for c in range(D):
        ref = np.correlate(ext[:, c], w[c].astype(np.float64), mode="valid")
        np.testing.assert_allclose(y[:, c], ref, rtol=1e-13, atol=1e-13)
    # the window is the last three raw inputs, bit for bit
    assert np.array_equal(new_win, ext[-3:])


# ----------------------------------------------------------------------- delta rule

def test_beta_zero_alpha_one_leaves_state_unchanged():
    q, k, v, _, _, S0 = _head_case(3, T=5, K=8, V=6)
    S, o, _ = oracle.recurrent_head(q, k, v, np.zeros((5, 8)), np.zeros(5), S0)
    assert np.array_equal(S, S0)
    np.testing.assert_allclose(o, q @ S0.T, rtol=1e-14, atol=1e-14)


def test_single_token_from_zero_state():
    q, k, v, g, beta, _ = _head_case(4, T=1, K=8, V=6)
    S, o, d = oracle.recurrent_head(q, k, v, g, beta, np.zeros((6, 8)))
    np.testing.assert_allclose(S, beta[0] * np.outer(v[0], k[0]), rtol=1e-14, atol=1e-15)
    # the output reads the updated state: o = beta (k . q) v
    np.testing.assert_allclose(o[0], beta[0] * (k[0] @ q[0]) * v[0], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(d[0], beta[0] * v[0], rtol=1e-14)


def test_beta_one_writes_value_at_key():
    q, k, v, g, _, S0 = _head_case(5, T=4, K=16, V=12)
    S = S0
    for t in range(4):  # after each token with beta = 1 and |k| = 1: S_new k = v
        S, _, _ = oracle.recurrent_head(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1],
                                        np.ones(1), S)
        np.testing.assert_allclose(S @ k[t], v[t], rtol=1e-12, atol=1e-12)


def _product_unroll(q, k, v, g, beta, S0):
    """S_T = S0 prod_t M_t + sum_t beta_t v_t k_t^T prod_{u>t} M_u with
    M_t = Diag(alpha_t) (I - beta_t k_t k_t^T); o_t = S_t q_t."""
    T, K = k.shape
    M = [np.diag(np.exp(g[t])) @ (np.eye(K) - beta[t] * np.outer(k[t], k[t])) for t in range(T)]
    outs, S_list = [], []
    for t_end in range(1, T + 1):
        acc = S0.copy()
        for t in range(t_end):
            acc = acc @ M[t]
        for t in range(t_end):
            term = beta[t] * np.outer(v[t], k[t])
            for u in range(t + 1, t_end):
                term = term @ M[u]
            acc = acc + term
        S_list.append(acc)
        outs.append(acc @ q[t_end - 1])
    return S_list[-1], np.array(outs)


@pytest.mark.parametrize("seed", [6, 7, 8])
def test_matches_brute_force_product_unroll(seed):
    # V != K so that a transposed state or operand cannot pass
    q, k, v, g, beta, S0 = _head_case(seed, T=6, K=3, V=4)
    S, o, _ = oracle.recurrent_head(q, k, v, g, beta, S0)
    S_ref, o_ref = _product_unroll(q, k, v, g, beta, S0)
    np.testing.assert_allclose(S, S_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)


def test_gdn_with_unit_gate_is_plain_delta_rule():
    # alpha = 1: S <- S (I - beta k k^T) + beta v k^T, the textbook DeltaNet update
    q, k, v, _, beta, S0 = _head_case(9, T=5, K=6, V=5)
    S, _, _ = oracle.recurrent_head(q, k, v, np.zeros((5, 6)), beta, S0)
    ref = S0.copy()
    for t in range(5):
        ref = ref @ (np.eye(6) - beta[t] * np.outer(k[t], k[t])) + beta[t] * np.outer(v[t], k[t])
    np.testing.assert_allclose(S, ref, rtol=1e-12, atol=1e-12)


def test_unrolled_closed_form_of_the_pages():
    # S_m = S_0 Diag(prod_i alpha_i) + sum_j d_j (k_j . prod_{i>j} alpha_i)^T
    q, k, v, g, beta, S0 = _head_case(10, T=9, K=7, V=5)
    S, _, d = oracle.recurrent_head(q, k, v, g, beta, S0)
    G = np.cumsum(g, axis=0)
    ref = S0 * np.exp(G[-1])[None, :]
    for j in range(9):
        ref = ref + np.outer(d[j], k[j] * np.exp(G[-1] - G[j]))
    np.testing.assert_allclose(S, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("T", [8, 11])
def test_block_closed_form_outputs_and_deltas(T):
    # The ReplaySSM verify and the blocked prefill compute each block of up to eight tokens in
    # closed form from the state at the block start S0 (G_t the cumulative log-decay from there):
    #   u_t = S0 (k_t . e^G_t) + sum_{s<t} A[t][s] d_s,  A[t][s] = sum_c k_s k_t e^(G_t - G_s)
    #   d_t = beta_t (v_t - u_t)
    #   o_t = S0 (q_t . e^G_t) + sum_{s<=t} P[t][s] d_s,  P[t][s] = sum_c k_s q_t e^(G_t - G_s)
    # and the state at the block end by the pages' unrolled form.  Blocks chained this way give
    # the recurrence's deltas and outputs.
    q, k, v, g, beta, S0 = _head_case(11, T=T, K=6, V=5)
    S_ref, o_ref, d_ref = oracle.recurrent_head(q, k, v, g, beta, S0)
    S = S0.astype(np.float64).copy()
    d_all, o_all = [], []
    for t0 in range(0, T, 8):
        kb, qb, vb, bb = k[t0:t0 + 8], q[t0:t0 + 8], v[t0:t0 + 8], beta[t0:t0 + 8]
        G = np.cumsum(g[t0:t0 + 8], axis=0)
        n = len(kb)
        d = np.zeros((n, S.shape[0]))
        for t in range(n):
            u = S @ (kb[t] * np.exp(G[t]))
            for s2 in range(t):
                u = u + np.sum(kb[s2] * kb[t] * np.exp(G[t] - G[s2])) * d[s2]
            d[t] = bb[t] * (vb[t] - u)
            o = S @ (qb[t] * np.exp(G[t]))
            for s2 in range(t + 1):
                o = o + np.sum(kb[s2] * qb[t] * np.exp(G[t] - G[s2])) * d[s2]
            d_all.append(d[t])
            o_all.append(o)
        S = S * np.exp(G[-1])[None, :] + sum(np.outer(d[s2], kb[s2] * np.exp(G[-1] - G[s2]))
                                             for s2 in range(n))
    np.testing.assert_allclose(np.array(d_all), d_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(np.array(o_all), o_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(S, S_ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("T,K,V", [(1, 16, 16), (63, 16, 8), (64, 16, 16), (65, 8, 16),
                                   (130, 16, 16), (1312, 32, 32)])
def test_chunkwise_equals_recurrence(T, K, V):
    q, k, v, g, beta, S0 = _head_case(11 + T, T=T, K=K, V=V)
    S_r, o_r, _ = oracle.recurrent_head(q, k, v, g, beta, S0)
    S_c, o_c = oracle.chunkwise_head(q, k, v, g, beta, S0, C=64)
    scale_o = np.max(np.abs(o_r))
    scale_s = np.max(np.abs(S_r))
    assert np.max(np.abs(o_c - o_r)) <= 1e-11 * scale_o
    assert np.max(np.abs(S_c - S_r)) <= 1e-11 * scale_s


@pytest.mark.parametrize("mode", ["const4", "scale20", "mixed"])
def test_chunkwise_equals_recurrence_under_strong_decay(mode):
    """The chunkwise form stays equal to the recurrence when the cumulative log gate of a
    chunk spans hundreds (g = -4 per token: 252 over 64 tokens; g = -e^3 softplus(N(0,1));
    channels and stretches of tokens at very different rates, with full resets)."""
    T, K, V = 200, 16, 8
    q, k, v, g, beta, S0 = _head_case(77, T=T, K=K, V=V)
    r = np.random.default_rng(78)
    if mode == "const4":
        g = np.full((T, K), -4.0)
    elif mode == "scale20":
        g = np.exp(3.0) * g
    else:
        g = g.copy()
        g[70:140, : K // 2] *= 30.0
        g[r.integers(0, T, 5)] = -300.0
    S_r, o_r, _ = oracle.recurrent_head(q, k, v, g, beta, S0)
    S_c, o_c = oracle.chunkwise_head(q, k, v, g, beta, S0, C=64)
    assert np.max(np.abs(o_c - o_r)) <= 1e-11 * np.max(np.abs(o_r))
    assert np.max(np.abs(S_c - S_r)) <= 1e-11 * np.max(np.abs(S_r))


def test_full_decay_token_resets_the_state():
    """alpha = exp(g) -> 0 on token t wipes the state: S_t = beta_t v_t k_t^T and
    o_t = beta_t (k_t . q_t) v_t, whatever came before (the single-token closed form)."""
    T, K, V = 40, 8, 6
    q, k, v, g, beta, S0 = _head_case(79, T=T, K=K, V=V)
    t = 23
    g = g.copy()
    g[t] = -1e4
    S_r, o_r, _ = oracle.recurrent_head(q[: t + 1], k[: t + 1], v[: t + 1], g[: t + 1],
                                       beta[: t + 1], S0)
    np.testing.assert_allclose(S_r, beta[t] * np.outer(v[t], k[t]), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(o_r[t], beta[t] * (k[t] @ q[t]) * v[t], rtol=1e-12, atol=1e-14)
    S_c, o_c = oracle.chunkwise_head(q, k, v, g, beta, S0, C=16)
    S_f, o_f, _ = oracle.recurrent_head(q, k, v, g, beta, S0)
    assert np.max(np.abs(o_c - o_f)) <= 1e-11 * np.max(np.abs(o_f))
    assert np.max(np.abs(S_c - S_f)) <= 1e-11 * np.max(np.abs(S_f))


# ----------------------------------------------------------------------- layer step

def _pool_case(seed, H=2, K=8, V=6, P=5, st=oracle.F32, io=oracle.F32, gate=oracle.KDA):
    r = np.random.default_rng(seed)
    ssm, conv = inputs.pool_arrays(r, 1, P, H, K, V, st, io)
    pool = oracle.Pool(1, P, H, K, V, st, io, gate, ssm, conv)
    w = inputs.conv_weights(r, H, K, V)
    return r, pool, w


def test_layer_split_order_and_output_of_value_channels():
    """S = 0, beta = 1 and identical raw q and k channels: each head's output is
    (|k|^2 / (|k|^2 + eps)) times its conv'd value channels."""
    H, K, V = 3, 8, 5
    r, pool, w = _pool_case(12, H=H, K=K, V=V)
    D = pool.D
    pool.ssm[...] = 0
    w[H * K:2 * H * K] = w[:H * K]                     # same taps for the k block as the q block
    pool.conv[0, 2, :, H * K:2 * H * K] = pool.conv[0, 2, :, :H * K]
    x = r.standard_normal(D).astype(np.float32)
    x[H * K:2 * H * K] = x[:H * K]
    g = np.zeros((1, H, K), np.float32)
    beta = np.ones((1, H), np.float32)
    ext = np.concatenate([pool.conv[0, 2].astype(np.float64), x[None].astype(np.float64)])
    y = np.array([ext[:, c] @ w[c].astype(np.float64) for c in range(D)])
    out = oracle.decode_step(pool, 0, [2], x[None], w, g, beta)
    for h in range(H):
        kk = y[H * K + h * K:H * K + (h + 1) * K]
        ss = kk @ kk
        vv = y[2 * H * K + h * V:2 * H * K + (h + 1) * V]
        np.testing.assert_allclose(out[0, h], ss / (ss + 1e-6) * vv, rtol=1e-6, atol=1e-7)


def test_layer_query_is_normalised_conv_of_q_block():
    """beta = 0, alpha = 1: the state stays and o_h = S_h q_hat with q_hat the L2-normalised
    conv output of head h's q channels (eps = 1e-6)."""
    H, K, V = 2, 8, 6
    r, pool, w = _pool_case(13, H=H, K=K, V=V)
    D = pool.D
    S0 = pool.ssm[0, 3].astype(np.float64).copy()
    x = r.standard_normal(D).astype(np.float32)
    ext = np.concatenate([pool.conv[0, 3].astype(np.float64), x[None].astype(np.float64)])
    y = np.array([ext[:, c] @ w[c].astype(np.float64) for c in range(D)])
    out = oracle.decode_step(pool, 0, [3], x[None], w, np.zeros((1, H, K), np.float32),
                             np.zeros((1, H), np.float32))
    for h in range(H):
        qq = y[h * K:(h + 1) * K]
        qh = qq / np.sqrt(qq @ qq + 1e-6)
        np.testing.assert_allclose(out[0, h], S0[h] @ qh, rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(pool.ssm[0, 3], S0, rtol=1e-7, atol=0)


def test_gdn_gate_is_one_scalar_per_head():
    H, K, V = 2, 8, 6
    r, pool_k, w = _pool_case(14, H=H, K=K, V=V, gate=oracle.KDA)
    pool_g = oracle.Pool(1, 5, H, K, V, oracle.F32, oracle.F32, oracle.GDN,
                         pool_k.ssm, pool_k.conv)
    x = r.standard_normal((1, pool_k.D)).astype(np.float32)
    gh = -np.abs(r.standard_normal((1, H))).astype(np.float32)
    beta = np.full((1, H), 0.7, np.float32)
    o_g = oracle.decode_step(pool_g, 0, [1], x, w, gh, beta)
    o_k = oracle.decode_step(pool_k, 0, [1], x, w, np.repeat(gh[..., None], K, -1), beta)
    assert np.array_equal(o_g, o_k)
    assert np.array_equal(pool_g.ssm, pool_k.ssm)


def test_decode_touches_only_its_slots():
    r, pool, w = _pool_case(15, P=6)
    before_s, before_c = pool.ssm.copy(), pool.conv.copy()
    slots = np.int32([4, 1])
    x = inputs.projections(r, (2,), pool.H, pool.K, pool.V, oracle.F32)
    g, beta = inputs.gates(r, (2,), pool.H, pool.K, oracle.KDA)
    oracle.decode_step(pool, 0, slots, x, w, g, beta)
    untouched = [s for s in range(7) if s not in (1, 4)]
    assert np.array_equal(pool.ssm[0, untouched], before_s[0, untouched])
    assert np.array_equal(pool.conv[0, untouched], before_c[0, untouched])
    # window: rows shift up by one and the new raw input lands in the last row
    for b, s in enumerate(slots):
        assert np.array_equal(pool.conv[0, s, :2], before_c[0, s, 1:])
        assert np.array_equal(pool.conv[0, s, 2], x[b])


def test_bf16_storage_rounds_only_at_store():
    """bf16 decode = fp32-storage decode of the same widened inputs, then bf16 rounding of
    the stored state and output (rounding happens once, at the store)."""
    H, K, V = 2, 8, 6
    r = np.random.default_rng(16)
    ssm, conv = inputs.pool_arrays(r, 1, 4, H, K, V, oracle.BF16, oracle.BF16)
    w = inputs.conv_weights(r, H, K, V)
    x = inputs.projections(r, (2,), H, K, V, oracle.BF16)
    g, beta = inputs.gates(r, (2,), H, K, oracle.KDA)
    pb = oracle.Pool(1, 4, H, K, V, oracle.BF16, oracle.BF16, oracle.KDA, ssm, conv)
    ob = oracle.decode_step(pb, 0, [1, 3], x, w, g, beta)
    # the same step in fp64 storage precision via the head recurrence
    for b, s in enumerate([1, 3]):
        win = oracle.bf16_to_f64(conv[0, s])
        xin = oracle.bf16_to_f64(x[b])
        new_win, y = oracle.conv_sequence(win, xin[None], w)
        assert np.array_equal(oracle.bf16_round(new_win), pb.conv[0, s])
        for h in range(H):
            qq = y[0, h * K:(h + 1) * K]
            kk = y[0, H * K + h * K:H * K + (h + 1) * K]
            vv = y[0, 2 * H * K + h * V:2 * H * K + (h + 1) * V]
            qh, kh = qq / np.sqrt(qq @ qq + 1e-6), kk / np.sqrt(kk @ kk + 1e-6)
            S, o, _ = oracle.recurrent_head(qh[None], kh[None], vv[None], g[b, h][None],
                                            beta[b, h:h + 1], oracle.bf16_to_f64(ssm[0, s, h]))
            assert np.array_equal(oracle.bf16_round(S), pb.ssm[0, s, h])
            assert np.array_equal(oracle.bf16_round(o[0]), ob[b, h])


# ----------------------------------------------------------------------- prefill

def test_prefill_equals_decode_steps():
    """Prefill of T tokens = T decode steps, except that storage rounding happens once at
    the end (fp32 storage: agreement to fp32 rounding)."""
    H, K, V, T = 2, 8, 6, 7
    r, pool, w = _pool_case(17, H=H, K=K, V=V)
    pool2 = oracle.Pool(1, 5, H, K, V, oracle.F32, oracle.F32, oracle.KDA, pool.ssm, pool.conv)
    x = inputs.projections(r, (T,), H, K, V, oracle.F32)
    g, beta = inputs.gates(r, (T,), H, K, oracle.KDA)
    out = oracle.prefill(pool, 0, [2], [0, T], x, w, g, beta)
    outs = [oracle.decode_step(pool2, 0, [2], x[t:t + 1], w, g[t:t + 1], beta[t:t + 1])[0]
            for t in range(T)]
    np.testing.assert_allclose(out, np.stack(outs), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(pool.ssm, pool2.ssm, rtol=1e-5, atol=1e-6)
    assert np.array_equal(pool.conv, pool2.conv)


def test_prefill_fresh_state_and_packed_sequences():
    H, K, V = 2, 8, 6
    r, pool, w = _pool_case(18, H=H, K=K, V=V)
    lens = [5, 2, 9]
    cu = inputs.cu_seqlens(lens)
    x = inputs.projections(r, (cu[-1],), H, K, V, oracle.F32)
    g, beta = inputs.gates(r, (cu[-1],), H, K, oracle.KDA)
    ref = oracle.Pool(1, 5, H, K, V, oracle.F32, oracle.F32, oracle.KDA, pool.ssm, pool.conv)
    out = oracle.prefill(pool, 0, [3, 1, 5], cu, x, w, g, beta, has_init=[1, 0, 1])
    # each sequence alone gives the same result; the fresh one starts from zeros
    ref.ssm[0, 1] = 0
    ref.conv[0, 1] = 0
    for n, s in enumerate([3, 1, 5]):
        a, b = cu[n], cu[n + 1]
        o_n = oracle.prefill(ref, 0, [s], [0, b - a], x[a:b], w, g[a:b], beta[a:b])
        assert np.array_equal(o_n, out[a:b])
    assert np.array_equal(ref.ssm, pool.ssm)
    assert np.array_equal(ref.conv, pool.conv)


# ----------------------------------------------------------------------- copy and spec

def test_slot_copy_bytes_and_mask():
    r, pool, _ = _pool_case(19, P=6, st=oracle.BF16, io=oracle.BF16)
    before_s, before_c = pool.ssm.copy(), pool.conv.copy()
    oracle.slot_copy(pool, -1, [1, 2, 3], [4, 5, 6], mask=[1, 0, 1])
    assert np.array_equal(pool.ssm[:, 4], before_s[:, 1])
    assert np.array_equal(pool.conv[:, 6], before_c[:, 3])
    assert np.array_equal(pool.ssm[:, 5], before_s[:, 5])   # masked out
    assert np.array_equal(pool.ssm[:, :4], before_s[:, :4])


@pytest.mark.parametrize("st", [oracle.F32, oracle.BF16])
def test_spec_commit_equals_accepted_decode_steps(st):
    """COMMIT(a) after VERIFY of T tokens = a+1 decode steps: windows bit-exact; states
    equal up to the storage rounding that decode applies after every step."""
    H, K, V, T, Lc = 2, 8, 6, 5, 8
    r, pool, w = _pool_case(20, H=H, K=K, V=V, st=st, io=st)
    B = 3
    slots = np.int32([5, 2, 4])
    x = inputs.projections(r, (B, T), H, K, V, st)
    g, beta = inputs.gates(r, (B, T), H, K, oracle.KDA)
    accept = np.int32([0, 4, 2])
    ref = oracle.Pool(1, 5, H, K, V, st, st, oracle.KDA, pool.ssm, pool.conv)
    before = pool.ssm.copy(), pool.conv.copy()
    sS, sC, out = oracle.spec_verify(pool, 0, slots, T, Lc, x, w, g, beta)
    assert np.array_equal(pool.ssm, before[0]) and np.array_equal(pool.conv, before[1])
    oracle.spec_commit(pool, 0, slots, T, Lc, sS, sC, accept)
    tol = 1e-6 if st == oracle.F32 else 2e-2
    for b in range(B):
        for t in range(accept[b] + 1):
            o = oracle.decode_step(ref, 0, slots[b:b + 1], x[b, t:t + 1], w, g[b, t:t + 1],
                                   beta[b, t:t + 1])
            err = np.max(np.abs(oracle.to_f64(o[0], st) - oracle.to_f64(out[b, t], st)))
            assert err <= tol * np.max(np.abs(oracle.to_f64(o[0], st)))
        s = slots[b]
        assert np.array_equal(pool.conv[0, s], ref.conv[0, s])
        a, e = oracle.to_f64(pool.ssm[0, s], st), oracle.to_f64(ref.ssm[0, s], st)
        assert np.max(np.abs(a - e)) <= tol * np.max(np.abs(e))


# ----------------------------------------------------------------------- fused gating

def test_softplus_and_sigmoid_closed_forms():
    """softplus(0) = ln 2, softplus(x) - softplus(-x) = x, softplus(x) -> x and -> e^x at the
    ends; sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4, sigmoid(x) + sigmoid(-x) = 1; and softplus'
    = sigmoid (central difference)."""
    assert abs(oracle.softplus(0.0) - np.log(2.0)) < 1e-15
    for x in [-30.0, -3.5, -0.25, 0.7, 4.0, 31.0]:
        assert abs(oracle.softplus(x) - oracle.softplus(-x) - x) < 1e-12 * max(1.0, abs(x))
        assert abs(oracle.sigmoid(x) + oracle.sigmoid(-x) - 1.0) < 1e-15
        h = 1e-5
        slope = (oracle.softplus(x + h) - oracle.softplus(x - h)) / (2 * h)
        assert abs(slope - oracle.sigmoid(x)) < 1e-8
    assert abs(oracle.softplus(60.0) - 60.0) <= 1e-14
    assert abs(oracle.softplus(-60.0) / np.exp(-60.0) - 1.0) < 1e-12
    assert oracle.sigmoid(0.0) == 0.5
    assert abs(oracle.sigmoid(np.log(3.0)) - 0.75) < 1e-15
    assert oracle.sigmoid(-800.0) == 0.0 and oracle.sigmoid(800.0) == 1.0


@pytest.mark.parametrize("gate", [oracle.KDA, oracle.GDN])
def test_gates_from_raw_closed_forms(gate):
    """With a = -dt_bias the softplus argument is 0: g = -exp(A_log) ln 2, so A_log = 0 gives
    alpha = 1/2 and A_log = ln 2 gives alpha = 1/4; b = 0 gives beta = 1/2, b = ln 3 beta = 3/4.
    Each channel's own dt_bias is used (KDA)."""
    H, K = 3, 8
    pool = oracle.Pool(1, 1, H, K, 4, oracle.F32, oracle.F32, gate,
                       np.zeros((1, 2, H, 4, K), np.float32), np.zeros((1, 2, 3, H * (2 * K + 4)), np.float32))
    n = K if gate == oracle.KDA else 1
    r = np.random.default_rng(26)
    dt = r.normal(size=(H, n)).astype(np.float32)
    A_log = np.float32([0.0, np.log(2.0), 0.0])
    a = -dt[None]
    b = np.float32([[0.0, np.log(3.0), -2.0]])
    g, beta = oracle.gates_from_raw(pool, a, b, A_log, dt)
    g = g.reshape(1, H, n)
    np.testing.assert_allclose(np.exp(g[0, 0]), 0.5, rtol=1e-6)
    np.testing.assert_allclose(np.exp(g[0, 1]), 0.25, rtol=1e-6)
    assert abs(beta[0, 0] - 0.5) < 1e-7 and abs(beta[0, 1] - 0.75) < 1e-7
    assert abs(beta[0, 2] - 1.0 / (1.0 + np.exp(2.0))) < 1e-7
    # one channel moved off zero: only its gate changes, by the pinned softplus
    a2 = a.copy()
    a2[0, 2, n - 1] += 1.5
    g2, _ = oracle.gates_from_raw(pool, a2, b, A_log, dt)
    g2 = g2.reshape(1, H, n)
    assert np.array_equal(np.delete(g2.ravel(), 2 * n + n - 1), np.delete(g.ravel(), 2 * n + n - 1))
    assert abs(g2[0, 2, n - 1] - (-oracle.softplus(1.5))) < 1e-6


@pytest.mark.parametrize("gate", [oracle.KDA, oracle.GDN])
def test_gated_decode_is_decode_with_those_gates(gate):
    r, pool, w = _pool_case(27, gate=gate)
    ref = oracle.Pool(1, 5, pool.H, pool.K, pool.V, pool.state_dtype, pool.conv_dtype, gate,
                      pool.ssm.copy(), pool.conv.copy())
    H, K = pool.H, pool.K
    n = K if gate == oracle.KDA else 1
    B = 3
    slots = np.int32([4, 1, 5])
    x = inputs.projections(r, (B,), H, K, pool.V, oracle.F32)
    a = r.normal(size=(B, H, n)).astype(np.float32)
    b = r.normal(size=(B, H)).astype(np.float32)
    A_log = r.normal(size=(H,)).astype(np.float32)
    dt = r.normal(size=(H, n)).astype(np.float32)
    o = oracle.decode_step_gated(pool, 0, slots, x, w, a, b, A_log, dt)
    g, beta = oracle.gates_from_raw(ref, a, b, A_log, dt)
    o2 = oracle.decode_step(ref, 0, slots, x, w, g, beta)
    assert np.array_equal(o, o2) and np.array_equal(pool.ssm, ref.ssm) and np.array_equal(pool.conv, ref.conv)


def test_tracked_decode_copies_updated_rows_only_where_masked():
    """The track copy after a decode step ([p1] mamba_track_interval): masked requests' track
    slots hold the updated state and window byte for byte; unmasked track slots and every other
    row are untouched; the step itself equals the plain decode."""
    r, pool, w = _pool_case(28)
    ref = oracle.Pool(1, 5, pool.H, pool.K, pool.V, pool.state_dtype, pool.conv_dtype, oracle.KDA,
                      pool.ssm.copy(), pool.conv.copy())
    before = pool.ssm.copy(), pool.conv.copy()
    slots, track, mask = np.int32([1, 3]), np.int32([4, 5]), np.uint8([1, 0])
    x = inputs.projections(r, (2,), pool.H, pool.K, pool.V, oracle.F32)
    g, beta = inputs.gates(r, (2,), pool.H, pool.K, oracle.KDA)
    o = oracle.decode_step_track(pool, 0, slots, x, w, g, beta, mask, track)
    o2 = oracle.decode_step(ref, 0, slots, x, w, g, beta)
    assert np.array_equal(o, o2)
    assert np.array_equal(pool.ssm[0, 4], pool.ssm[0, 1]) and np.array_equal(pool.conv[0, 4], pool.conv[0, 1])
    assert np.array_equal(pool.ssm[0, 5], before[0][0, 5]) and np.array_equal(pool.conv[0, 5], before[1][0, 5])
    for s in (0, 1, 2, 3):
        assert np.array_equal(pool.ssm[0, s], ref.ssm[0, s]) and np.array_equal(pool.conv[0, s], ref.conv[0, s])


# ----------------------------------------------------------------------- ReplaySSM

def _replay_case(seed, st, gate=oracle.KDA, depth=16):
    H, K, V, T, Lc = 2, 8, 6, 5, 8
    r, pool, w = _pool_case(seed, H=H, K=K, V=V, st=st, io=st, gate=gate)
    B = 3
    slots = np.int32([5, 2, 4])
    x = inputs.projections(r, (B, T), H, K, V, st)
    g, beta = inputs.gates(r, (B, T), H, K, gate)
    return dict(H=H, K=K, V=V, T=T, Lc=Lc, B=B, pool=pool, w=w, slots=slots, x=x, g=g, beta=beta,
                depth=depth, st=st, gate=gate)


@pytest.mark.parametrize("gate", [oracle.KDA, oracle.GDN])
def test_replay_commit_equals_snapshot_commit(gate):
    """ReplaySSM commit(a) replays tokens 0..a from the slot out of the rings; with fp32 records
    it lands where the snapshot path's commit(a) does (cache entry a), windows bit-exact, and
    verify leaves the slot untouched and gives the snapshot verify's outputs bit for bit."""
    c = _replay_case(21, oracle.F32, gate)
    pool, st = c["pool"], c["st"]
    snap = oracle.Pool(1, 5, c["H"], c["K"], c["V"], st, st, gate, pool.ssm.copy(), pool.conv.copy())
    before = pool.ssm.copy(), pool.conv.copy()
    rings = oracle.Rings(pool, c["depth"])
    pos = np.int32([0, 3, 14])  # the last request wraps around the ring
    accept = np.int32([0, 4, 2])
    sC, out = oracle.replay_verify(pool, rings, 0, c["slots"], pos, c["T"], c["Lc"], c["x"], c["w"],
                                   c["g"], c["beta"])
    assert np.array_equal(pool.ssm, before[0]) and np.array_equal(pool.conv, before[1])
    sS2, sC2, out2 = oracle.spec_verify(snap, 0, c["slots"], c["T"], c["Lc"], c["x"], c["w"],
                                        c["g"], c["beta"])
    assert np.array_equal(out, out2) and np.array_equal(sC, sC2)
    oracle.replay_commit(pool, rings, 0, c["slots"], pos, c["T"], c["Lc"], sC, accept)
    oracle.spec_commit(snap, 0, c["slots"], c["T"], c["Lc"], sS2, sC2, accept)
    assert np.array_equal(pool.conv, snap.conv)
    a, e = oracle.to_f64(pool.ssm, st), oracle.to_f64(snap.ssm, st)
    assert np.max(np.abs(a - e)) <= 1e-6 * np.max(np.abs(e))


def test_replay_records_rebuild_state_by_closed_form():
    """The pages' closed form from the checkpoint and the (d, k, g) records,
    S_m = S_0 Diag(prod_i alpha_i) + sum_j d_j (k_j . prod_{i>j} alpha_i)^T,
    gives the state the snapshot verify stored after m tokens (fp32 records)."""
    c = _replay_case(22, oracle.F32)
    pool, st, H, K, V, T = c["pool"], c["st"], c["H"], c["K"], c["V"], c["T"]
    snap = oracle.Pool(1, 5, H, K, V, st, st, oracle.KDA, pool.ssm.copy(), pool.conv.copy())
    rings = oracle.Rings(pool, c["depth"])
    pos = np.int32([7, 12, 1])
    oracle.replay_verify(pool, rings, 0, c["slots"], pos, T, c["Lc"], c["x"], c["w"], c["g"], c["beta"])
    sS, _, _ = oracle.spec_verify(snap, 0, c["slots"], T, c["Lc"], c["x"], c["w"], c["g"], c["beta"])
    L = c["depth"]
    for b, s in enumerate(c["slots"]):
        S0 = oracle.to_f64(pool.ssm[0, s], st)
        ent = [(pos[b] + t) % L for t in range(T)]
        for m in range(1, T + 1):
            for h in range(H):
                al = np.exp(rings.g[0, s, h, ent[:m]].astype(np.float64))  # [m][K]
                Sm = S0[h] * np.prod(al, axis=0)[None, :]
                for j in range(m):
                    later = np.prod(al[j + 1:], axis=0) if j + 1 < m else np.ones(K)
                    kj = rings.k[0, s, h, ent[j]].astype(np.float64)
                    dj = rings.d[0, s, h, ent[j]].astype(np.float64)
                    Sm = Sm + np.outer(dj, kj * later)
                ref = oracle.to_f64(sS[b, m - 1, h], st)
                assert np.max(np.abs(Sm - ref)) <= 1e-5 * np.max(np.abs(ref)), (b, m, h)


def test_replay_rawk_rawv_are_pre_norm_key_and_conv_value():
    """rawk is the key before its L2 norm (k = rawk / sqrt(|rawk|^2 + eps)), rawv the conv'd
    value channel of the head, g and beta the inputs as given."""
    c = _replay_case(23, oracle.F32)
    pool, H, K, V, T = c["pool"], c["H"], c["K"], c["V"], c["T"]
    rings = oracle.Rings(pool, c["depth"])
    pos = np.int32([2, 2, 2])
    oracle.replay_verify(pool, rings, 0, c["slots"], pos, T, c["Lc"], c["x"], c["w"], c["g"], c["beta"])
    D = pool.D
    for b, s in enumerate(c["slots"]):
        win = oracle.to_f64(pool.conv[0, s], oracle.F32).reshape(3, D)
        _, y = oracle.conv_sequence(win, oracle.to_f64(c["x"][b], oracle.F32), c["w"])
        for t in range(T):
            e = (2 + t) % c["depth"]
            for h in range(H):
                rk = rings.rawk[0, s, h, e].astype(np.float64)
                np.testing.assert_allclose(rk, y[t, H * K + h * K: H * K + (h + 1) * K], rtol=1e-6, atol=1e-7)
                np.testing.assert_allclose(rings.rawv[0, s, h, e], y[t, 2 * H * K + h * V: 2 * H * K + (h + 1) * V],
                                           rtol=1e-6, atol=1e-7)
                kn = rk / np.sqrt(np.sum(rk * rk) + 1e-6)
                np.testing.assert_allclose(rings.k[0, s, h, e], kn, rtol=1e-5, atol=1e-7)
                assert np.array_equal(rings.g[0, s, h, e], c["g"][b, t, h])
                assert rings.beta[0, s, h, e] == c["beta"][b, t, h]


def test_replay_bf16_records_commit_within_tolerance():
    """bf16 records (the pages' storage): commit(a) stays within the bf16 bar of the snapshot
    path's commit(a)."""
    c = _replay_case(24, oracle.BF16)
    pool, st = c["pool"], c["st"]
    snap = oracle.Pool(1, 5, c["H"], c["K"], c["V"], st, st, oracle.KDA, pool.ssm.copy(), pool.conv.copy())
    rings = oracle.Rings(pool, c["depth"])
    pos = np.int32([9, 0, 15])
    accept = np.int32([4, 1, 3])
    sC, _ = oracle.replay_verify(pool, rings, 0, c["slots"], pos, c["T"], c["Lc"], c["x"], c["w"],
                                 c["g"], c["beta"])
    oracle.replay_commit(pool, rings, 0, c["slots"], pos, c["T"], c["Lc"], sC, accept)
    sS2, sC2, _ = oracle.spec_verify(snap, 0, c["slots"], c["T"], c["Lc"], c["x"], c["w"], c["g"], c["beta"])
    oracle.spec_commit(snap, 0, c["slots"], c["T"], c["Lc"], sS2, sC2, accept)
    assert np.array_equal(pool.conv, snap.conv)
    a, e = oracle.to_f64(pool.ssm, st), oracle.to_f64(snap.ssm, st)
    assert np.max(np.abs(a - e)) <= 2e-2 * np.max(np.abs(e))


def test_replay_rejects_short_ring_and_bad_position():
    c = _replay_case(25, oracle.F32, depth=8)  # 2 T = 10 > 8
    rings = oracle.Rings(c["pool"], 8)
    with pytest.raises(ValueError):
        oracle.replay_verify(c["pool"], rings, 0, c["slots"], np.int32([0, 0, 0]), c["T"], c["Lc"],
                             c["x"], c["w"], c["g"], c["beta"])
    c = _replay_case(25, oracle.F32)
    rings = oracle.Rings(c["pool"], 16)
    with pytest.raises(ValueError):
        oracle.replay_verify(c["pool"], rings, 0, c["slots"], np.int32([0, 16, 0]), c["T"], c["Lc"],
                             c["x"], c["w"], c["g"], c["beta"])


# ----------------------------------------------------------------------- pool layout

def test_pool_bytes_reproduce_logged_sizes():
    gold = json.load(open(os.path.join(GOLDEN, "pool_sizes.json")))
    shp = gold["shape"]
    dt = {"f32": oracle.F32, "bf16": oracle.BF16}
    for p in gold["pools"]:
        s, c = oracle.pool_bytes(shp["layers"], p["slots"], shp["H"], shp["K"], shp["V"],
                                 dt[p["state_dtype"]], dt[p["conv_dtype"]])
        assert round(s / 2**30, 2) == p["ssm_gib"], p
        assert round(c / 2**30, 2) == p["conv_gib"], p
    pr = gold["per_request"]
    # one slot of all layers = one row per layer: (slots + 1) rows with slots = 0
    s, c = oracle.pool_bytes(pr["layers"], 0, pr["H"], pr["K"], pr["V"], oracle.BF16, oracle.BF16)
    assert round(s / 2**20, 1) == pr["ssm_mib"]
    assert round(c / 2**20, 2) == pr["conv_mib"]
    assert round((pr["ssm_mib"] + pr["conv_mib"]) * 8, 1) == pr["tp8_total_mib"]
