"""Pins of the float64 oracle to facts the MoDA pages and mathematics fix.

Each test checks the oracle against something other than itself: a library
routine (torch scaled_dot_product_attention / autograd / logsumexp in float64),
brute force on tiny inputs, closed forms, invariants, or the worked index map
printed on the slides.  Together they are chosen so that a dropped term, a
wrong sign, a wrong index or a transposed operand in the oracle fails at least
one of them.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_problem(B, H, Hkv, T, S, d, seed, dtype=np.float64):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, T, d))
    k = rng.standard_normal((B, Hkv, T, d))
    v = rng.standard_normal((B, Hkv, T, d))
    kd = rng.standard_normal((B, Hkv, T, S, d))
    vd = rng.standard_normal((B, Hkv, T, S, d))
    return [x.astype(dtype) for x in (q, k, v, kd, vd)]


def expanded_row_position(i_q, G):
    """t_base(i_q) = floor(i_q / G): the grouped row map of the slides' backup frame."""
    return i_q // G


def flattened_mask(T, S, G):
    """Visibility over the flattened key axis [T sequence keys | T*S depth keys] for the
    G-fold expanded query rows: sequence visible iff floor(i_q/G) >= i_k, depth visible
    iff floor(i_q/G) == floor(j_d/S)  (frame "Backup: grouped indexing", Alg. 1)."""
    iq = torch.arange(T * G)
    pos = expanded_row_position(iq, G)
    seq = pos[:, None] >= torch.arange(T)[None, :]
    dep = pos[:, None] == (torch.arange(T * S) // max(S, 1))[None, :] if S else torch.zeros(T * G, 0, dtype=torch.bool)
    return torch.cat([seq, dep], dim=1)


def flattened_reference(q, k, v, kd, vd, scale=None, requires_grad=False):
    """The joint softmax evaluated by torch SDPA over the flattened key axis, with the
    expanded-row mask above.  Returns (o[B,H,T,d], lse[B,H,T]) as float64 tensors."""
    B, H, T, d = q.shape
    Hkv, S = k.shape[1], kd.shape[3]
    G = H // Hkv
    scale = scale or 1.0 / math.sqrt(d)
    mask = flattened_mask(T, S, G)
    # expanded rows of kv head g: i_q = t*G + hh  (head h = g*G + hh)
    qe = q.reshape(B, Hkv, G, T, d).transpose(2, 3).reshape(B, Hkv, T * G, d)
    kc = torch.cat([k, kd.reshape(B, Hkv, T * S, d)], dim=2)
    vc = torch.cat([v, vd.reshape(B, Hkv, T * S, d)], dim=2)
    oe = F.scaled_dot_product_attention(qe, kc, vc, attn_mask=mask, scale=scale)
    scores = torch.matmul(qe, kc.transpose(-1, -2)) * scale
    lse_e = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1)
    o = oe.reshape(B, Hkv, T, G, d).transpose(2, 3).reshape(B, H, T, d)
    lse = lse_e.reshape(B, Hkv, T, G).transpose(2, 3).reshape(B, H, T)
    return o, lse


def test_oracle_golden_index_map():
    """The slides' worked example: for G=4 the expanded rows 8..15 map to positions 2 and 3."""
    with open(os.path.join(GOLDEN, "grouped_index_map.txt")) as f:
        rows = [line.split() for line in f if line.strip() and not line.startswith("#")]
    assert rows
    for G, r0, r1, pos in rows:
        G, r0, r1 = int(G), int(r0), int(r1)
        want = sorted(int(p) for p in pos.split(","))
        got = sorted(set(int(expanded_row_position(i, G)) for i in range(r0, r1 + 1)))
        assert got == want
        # and the flattened mask gives those rows exactly the depth keys of their own position
        T, S = 5, 3
        m = flattened_mask(T, S, G)
        for i in range(r0, r1 + 1):
            depth_cols = torch.nonzero(m[i, T:]).flatten().tolist()
            p = i // G
            assert depth_cols == list(range(p * S, p * S + S))


@pytest.mark.parametrize("B,H,Hkv,T,d", [(1, 2, 2, 9, 8), (2, 4, 2, 13, 16), (1, 6, 1, 7, 4)])
def test_oracle_no_depth_is_causal_attention(oracle_mod, B, H, Hkv, T, d):
    """H_l empty (S=0): the operator is textbook causal softmax attention (torch SDPA, fp64)."""
    q, k, v, kd, vd = rand_problem(B, H, Hkv, T, 0, d, seed=11)
    o, lse = oracle_mod.forward(q, k, v, kd, vd)
    G = H // Hkv
    tq = torch.from_numpy(q)
    tk = torch.from_numpy(k).repeat_interleave(G, dim=1)
    tv = torch.from_numpy(v).repeat_interleave(G, dim=1)
    ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    np.testing.assert_allclose(o, ref.numpy(), atol=1e-12, rtol=0)
    s = torch.matmul(tq, tk.transpose(-1, -2)) / math.sqrt(d)
    causal = torch.ones(T, T, dtype=torch.bool).tril()
    ref_lse = torch.logsumexp(s.masked_fill(~causal, float("-inf")), dim=-1)
    np.testing.assert_allclose(lse, ref_lse.numpy(), atol=1e-12, rtol=0)


@pytest.mark.parametrize("B,H,Hkv,T,S,d", [(1, 2, 2, 6, 1, 4), (2, 4, 2, 9, 3, 8), (1, 8, 2, 11, 5, 16)])
def test_oracle_matches_flattened_masked_softmax(oracle_mod, B, H, Hkv, T, S, d):
    """The joint operator equals one softmax over the flattened [sequence | depth] key axis
    with the grouped masks of Algorithm 1 (library SDPA + logsumexp in fp64)."""
    q, k, v, kd, vd = rand_problem(B, H, Hkv, T, S, d, seed=5)
    o, lse = oracle_mod.forward(q, k, v, kd, vd)
    ro, rl = flattened_reference(*map(torch.from_numpy, (q, k, v, kd, vd)))
    np.testing.assert_allclose(o, ro.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, rl.numpy(), atol=1e-12, rtol=0)


def test_oracle_constant_values(oracle_mod):
    """All v and vd equal to one vector c: the output is a convex combination, so o = c."""
    q, k, v, kd, vd = rand_problem(2, 4, 2, 10, 3, 8, seed=7)
    c = np.linspace(-2.0, 3.0, 8)
    v[:] = c
    vd[:] = c
    o, _ = oracle_mod.forward(q, k, v, kd, vd)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), atol=1e-13, rtol=0)


def test_oracle_depth_slot_permutation(oracle_mod):
    """Permuting the depth slots of each position leaves o and LSE unchanged."""
    q, k, v, kd, vd = rand_problem(1, 4, 2, 8, 5, 8, seed=3)
    o, lse = oracle_mod.forward(q, k, v, kd, vd)
    rng = np.random.default_rng(1)
    kd2, vd2 = kd.copy(), vd.copy()
    for b in range(kd.shape[0]):
        for g in range(kd.shape[1]):
            for t in range(kd.shape[2]):
                p = rng.permutation(kd.shape[3])
                kd2[b, g, t] = kd[b, g, t, p]
                vd2[b, g, t] = vd[b, g, t, p]
    o2, lse2 = oracle_mod.forward(q, k, v, kd2, vd2)
    np.testing.assert_allclose(o2, o, atol=1e-14, rtol=0)
    np.testing.assert_allclose(lse2, lse, atol=1e-14, rtol=0)


def test_oracle_single_sequence_key_brute_force(oracle_mod):
    """Masking every sequence key but j = t leaves a softmax over {t} and the depth slots,
    checked by an explicit loop with math.exp."""
    B, H, Hkv, T, S, d = 1, 2, 1, 6, 3, 4
    q, k, v, kd, vd = rand_problem(B, H, Hkv, T, S, d, seed=9)
    o, lse = oracle_mod.forward(q, k, v, kd, vd, seq_window=1)
    sc = 1.0 / math.sqrt(d)
    for h in range(H):
        for t in range(T):
            keys = [k[0, 0, t]] + [kd[0, 0, t, i] for i in range(S)]
            vals = [v[0, 0, t]] + [vd[0, 0, t, i] for i in range(S)]
            w = [math.exp(sc * float(np.dot(q[0, h, t], kk))) for kk in keys]
            z = sum(w)
            want = sum(wi * vi for wi, vi in zip(w, vals)) / z
            np.testing.assert_allclose(o[0, h, t], want, atol=1e-13, rtol=0)
            assert abs(lse[0, h, t] - math.log(z)) < 1e-13


def test_oracle_separate_softmaxes_differ(oracle_mod):
    """Two separately normalised softmaxes added together are a different operator."""
    q, k, v, kd, vd = rand_problem(1, 2, 2, 16, 4, 8, seed=2)
    o, _ = oracle_mod.forward(q, k, v, kd, vd)
    tq, tk, tv, tkd, tvd = map(torch.from_numpy, (q, k, v, kd, vd))
    seq = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    sd = torch.softmax(torch.einsum("bhtc,bhtsc->bhts", tq, tkd) / math.sqrt(8), dim=-1)
    dep = torch.einsum("bhts,bhtsc->bhtc", sd, tvd)
    assert np.max(np.abs((seq + dep).numpy() - o)) > 1e-2


def test_oracle_translation_invariance(oracle_mod):
    """Adding one vector c to every k and kd of a kv head shifts each row's scores by a
    constant: o is unchanged, and the gradients obey sum_j dk_j + sum_{t,i} dkd_{t,i} = 0
    per (b, g) and dq unchanged (equivalent to the joint row sum of dS being zero)."""
    q, k, v, kd, vd = rand_problem(2, 4, 2, 7, 3, 6, seed=4)
    dout = np.random.default_rng(8).standard_normal(q.shape)
    o, _ = oracle_mod.forward(q, k, v, kd, vd)
    c = np.random.default_rng(6).standard_normal(6)
    o2, _ = oracle_mod.forward(q, k + c, v, kd + c, vd)
    np.testing.assert_allclose(o2, o, atol=1e-12, rtol=0)
    dq, dk, dv, dkd, dvd = oracle_mod.backward(q, k, v, kd, vd, dout)
    tot = dk.sum(axis=2) + dkd.sum(axis=(2, 3))
    assert np.max(np.abs(tot)) < 1e-10
    dq2 = oracle_mod.backward(q, k + c, v, kd + c, vd, dout)[0]
    np.testing.assert_allclose(dq2, dq, atol=1e-10, rtol=0)


@pytest.mark.parametrize("seq_window", [0, 2])
def test_oracle_backward_finite_differences(oracle_mod, seq_window):
    """Analytic gradients of L = sum(dout * o) against float64 central differences."""
    B, H, Hkv, T, S, d = 1, 4, 2, 5, 3, 4
    x = rand_problem(B, H, Hkv, T, S, d, seed=21)
    dout = np.random.default_rng(22).standard_normal((B, H, T, d))
    grads = oracle_mod.backward(*x, dout, seq_window=seq_window)
    h = 1e-6

    def loss(xs):
        o, _ = oracle_mod.forward(*xs, seq_window=seq_window)
        return float(np.sum(o * dout))

    for which in range(5):
        g = grads[which]
        num = np.zeros_like(g)
        flat = x[which].reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + h
            lp = loss(x)
            flat[i] = old - h
            lm = loss(x)
            flat[i] = old
            num.reshape(-1)[i] = (lp - lm) / (2 * h)
        err = np.max(np.abs(num - g)) / max(np.max(np.abs(g)), 1e-30)
        assert err < 1e-6, (which, err)


def test_oracle_backward_matches_autograd(oracle_mod):
    """Gradients equal torch autograd through the flattened SDPA formulation (fp64)."""
    B, H, Hkv, T, S, d = 2, 8, 2, 9, 4, 8
    x = [torch.from_numpy(a).requires_grad_(True) for a in rand_problem(B, H, Hkv, T, S, d, seed=31)]
    dout = torch.from_numpy(np.random.default_rng(32).standard_normal((B, H, T, d)))
    o, _ = flattened_reference(*x)
    o.backward(dout)
    got = oracle_mod.backward(*[a.detach().numpy() for a in x], dout.numpy())
    for a, g in zip(x, got):
        np.testing.assert_allclose(g, a.grad.numpy(), atol=1e-11, rtol=0)


def test_oracle_sampled_rows_equal_full(oracle_mod):
    """The sampled-row, sampled-position and sampled-key entry points agree with the full ones."""
    B, H, Hkv, T, S, d = 2, 4, 2, 12, 3, 8
    x = rand_problem(B, H, Hkv, T, S, d, seed=41)
    dout = np.random.default_rng(42).standard_normal((B, H, T, d))
    o, lse = oracle_mod.forward(*x)
    rows = np.array([0, 5, 11, 12 * 3 + 7, B * H * T - 1])
    so, sl = oracle_mod.forward(*x, rows=rows)
    np.testing.assert_array_equal(so, o.reshape(-1, d)[rows])
    np.testing.assert_array_equal(sl, lse.reshape(-1)[rows])
    dq, dk, dv, dkd, dvd = oracle_mod.backward(*x, dout)
    pos = np.array([0, 7, T + 3, B * Hkv * T - 1])
    pdq, pdkd, pdvd = oracle_mod.backward_positions(*x, dout, positions=pos)
    G = H // Hkv
    for n, p in enumerate(pos):
        t, bg = p % T, p // T
        b, g = bg // Hkv, bg % Hkv
        np.testing.assert_allclose(pdq[n], dq[b, g * G:(g + 1) * G, t], atol=1e-13, rtol=0)
        np.testing.assert_allclose(pdkd[n], dkd[b, g, t], atol=1e-13, rtol=0)
        np.testing.assert_allclose(pdvd[n], dvd[b, g, t], atol=1e-13, rtol=0)
    keys = np.array([1, T - 1, 2 * T + 4])
    kdk, kdv = oracle_mod.backward_keys(*x, dout, keys=keys)
    np.testing.assert_allclose(kdk, dk.reshape(-1, d)[keys], atol=1e-13, rtol=0)
    np.testing.assert_allclose(kdv, dv.reshape(-1, d)[keys], atol=1e-13, rtol=0)


def test_oracle_reads_storage_types_exactly(oracle_mod):
    """bf16 (as uint16 bits) and fp32 storage are widened exactly: same result as fp64
    arrays holding the same values."""
    x32 = rand_problem(1, 4, 2, 8, 2, 8, seed=51, dtype=np.float32)
    bf = [torch.from_numpy(a).to(torch.bfloat16) for a in x32]
    bits = [b.view(torch.int16).numpy().view(np.uint16) for b in bf]
    wide = [b.to(torch.float64).numpy() for b in bf]
    ob, lb = oracle_mod.forward(*bits)
    ow, lw = oracle_mod.forward(*wide)
    np.testing.assert_array_equal(ob, ow)
    np.testing.assert_array_equal(lb, lw)
    o32, _ = oracle_mod.forward(*x32)
    o64, _ = oracle_mod.forward(*[a.astype(np.float64) for a in x32])
    np.testing.assert_array_equal(o32, o64)


def test_oracle_exp2_form_equivalence():
    """Algorithm 1 writes 2^(S-m); with logits scaled by log2(e) it is the natural-exp
    softmax (frame "Backup: pseudocode needs implementation-level checks")."""
    s = np.random.default_rng(0).standard_normal(37) * 4
    nat = np.exp(s - s.max()) / np.exp(s - s.max()).sum()
    s2 = s * math.log2(math.e)
    base2 = np.exp2(s2 - s2.max()) / np.exp2(s2 - s2.max()).sum()
    np.testing.assert_allclose(base2, nat, rtol=1e-13, atol=0)


# ------------------------------------------------------------------ decode
def test_oracle_decode_is_the_operators_last_row(oracle_mod):
    """A decode step is the newest row of the joint operator: the C++ oracle's row T-1 of
    a full problem whose depth slab at T-1 is the decode step's slots."""
    B, H, Hkv, T, S, d = 2, 6, 2, 37, 5, 16
    q, k, v, kd, vd = rand_problem(B, H, Hkv, T, S, d, seed=71)
    rows = np.array([(b * H + h) * T + T - 1 for b in range(B) for h in range(H)], dtype=np.int64)
    ro, rl = oracle_mod.forward(q, k, v, kd, vd, rows=rows)
    o, lse = oracle_mod.decode(q[:, :, T - 1], k, v, kd[:, :, T - 1], vd[:, :, T - 1])
    np.testing.assert_allclose(o.reshape(B * H, d), ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(B * H), rl, rtol=0, atol=1e-12)


def test_oracle_decode_no_depth_is_single_query_attention(oracle_mod):
    """S = 0: softmax attention of one query over all T cached keys (torch SDPA, float64)."""
    B, H, Hkv, T, d = 1, 4, 2, 23, 8
    rng = np.random.default_rng(72)
    q = rng.standard_normal((B, H, d))
    k = rng.standard_normal((B, Hkv, T, d))
    v = rng.standard_normal((B, Hkv, T, d))
    kd = np.zeros((B, Hkv, 0, d))
    o, lse = oracle_mod.decode(q, k, v, kd, kd)
    G = H // Hkv
    kt = torch.from_numpy(k).repeat_interleave(G, dim=1)
    vt = torch.from_numpy(v).repeat_interleave(G, dim=1)
    qt = torch.from_numpy(q)[:, :, None, :]
    ref = F.scaled_dot_product_attention(qt, kt, vt)[:, :, 0]
    ref_lse = torch.logsumexp(torch.matmul(qt, kt.transpose(-1, -2))[:, :, 0] / math.sqrt(d), dim=-1)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)


def test_oracle_decode_brute_force_and_constant_values(oracle_mod):
    """Tiny case against explicit math.exp loops; constant values give that constant."""
    rng = np.random.default_rng(73)
    q = rng.standard_normal((1, 1, 3))
    k = rng.standard_normal((1, 1, 2, 3))
    v = rng.standard_normal((1, 1, 2, 3))
    kd = rng.standard_normal((1, 1, 2, 3))
    vd = rng.standard_normal((1, 1, 2, 3))
    o, lse = oracle_mod.decode(q, k, v, kd, vd)
    sc = 1 / math.sqrt(3)
    keys = [k[0, 0, 0], k[0, 0, 1], kd[0, 0, 0], kd[0, 0, 1]]
    vals = [v[0, 0, 0], v[0, 0, 1], vd[0, 0, 0], vd[0, 0, 1]]
    w = [math.exp(sc * sum(q[0, 0, c] * kk[c] for c in range(3))) for kk in keys]
    ref = [sum(w[i] * vals[i][c] for i in range(4)) / sum(w) for c in range(3)]
    np.testing.assert_allclose(o[0, 0], ref, rtol=1e-13)
    assert abs(lse[0, 0] - math.log(sum(w))) < 1e-13
    const = np.full_like(v, 2.5)
    oc, _ = oracle_mod.decode(q, k, const, kd, np.full_like(vd, 2.5))
    np.testing.assert_allclose(oc, 2.5, rtol=0, atol=1e-14)


# ------------------------------------------------------------------ depth-KV write path
def test_oracle_depth_store_places_one_slot(oracle_mod):
    """The attention KV becomes exactly one slot; the others are untouched."""
    rng = np.random.default_rng(81)
    k, v = rng.standard_normal((2, 3, 5, 4)), rng.standard_normal((2, 3, 5, 4))
    kd, vd = rng.standard_normal((2, 3, 5, 6, 4)), rng.standard_normal((2, 3, 5, 6, 4))
    nk, nv = oracle_mod.depth_store(k, v, kd, vd, slot=4)
    np.testing.assert_array_equal(nk[:, :, :, 4], k)
    np.testing.assert_array_equal(nv[:, :, :, 4], v)
    others = [s for s in range(6) if s != 4]
    np.testing.assert_array_equal(nk[:, :, :, others], kd[:, :, :, others])
    np.testing.assert_array_equal(nv[:, :, :, others], vd[:, :, :, others])


def test_oracle_depth_project_brute_force(oracle_mod):
    """Projection into a slot against explicit sums on a tiny case; other slots kept."""
    rng = np.random.default_rng(82)
    B, T, Dm, Hkv, S, d = 2, 3, 5, 2, 3, 4
    x = rng.standard_normal((B, T, Dm))
    wk, wv = rng.standard_normal((Dm, Hkv * d)), rng.standard_normal((Dm, Hkv * d))
    kd, vd = rng.standard_normal((B, Hkv, T, S, d)), rng.standard_normal((B, Hkv, T, S, d))
    nk, nv = oracle_mod.depth_project(x, wk, wv, kd, vd, slot=1)
    for b in range(B):
        for g in range(Hkv):
            for t in range(T):
                for c in range(d):
                    ek = sum(x[b, t, m] * wk[m, g * d + c] for m in range(Dm))
                    ev = sum(x[b, t, m] * wv[m, g * d + c] for m in range(Dm))
                    assert abs(nk[b, g, t, 1, c] - ek) < 1e-12 and abs(nv[b, g, t, 1, c] - ev) < 1e-12
    np.testing.assert_array_equal(nk[:, :, :, [0, 2]], kd[:, :, :, [0, 2]])
    np.testing.assert_array_equal(nv[:, :, :, [0, 2]], vd[:, :, :, [0, 2]])


def test_oracle_depth_project_feeds_the_forward(oracle_mod):
    """A slot written by the projection is read by the forward as any other slot: with S = 1
    and the projection of x, the forward equals the forward on a hand-built kd/vd."""
    rng = np.random.default_rng(83)
    B, H, Hkv, T, d, Dm = 1, 2, 1, 4, 4, 3
    q, k, v = rng.standard_normal((B, H, T, d)), rng.standard_normal((B, Hkv, T, d)), rng.standard_normal((B, Hkv, T, d))
    x = rng.standard_normal((B, T, Dm))
    wk, wv = rng.standard_normal((Dm, Hkv * d)), rng.standard_normal((Dm, Hkv * d))
    kd0 = np.zeros((B, Hkv, T, 1, d))
    nk, nv = oracle_mod.depth_project(x, wk, wv, kd0, kd0, slot=0)
    hand_k = np.einsum("btm,mc->btc", x, wk).reshape(B, T, Hkv, d).transpose(0, 2, 1, 3)[:, :, :, None, :]
    hand_v = np.einsum("btm,mc->btc", x, wv).reshape(B, T, Hkv, d).transpose(0, 2, 1, 3)[:, :, :, None, :]
    o1, l1 = oracle_mod.forward(q, k, v, nk, nv)
    o2, l2 = oracle_mod.forward(q, k, v, hand_k, hand_v)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ bounded slot buffer
def test_oracle_sliding_window_keeps_the_newest_in_order(oracle_mod):
    """Marker histories (slot i of kd holds i + position/100, of vd -i): the window of the
    newest W slots, oldest first; W >= L keeps all of them."""
    B, Hkv, T, L, d = 1, 2, 3, 5, 4
    idx = np.arange(L)[None, None, None, :, None] + np.arange(T)[None, None, :, None, None] / 100.0
    kd = np.broadcast_to(idx, (B, Hkv, T, L, d)).copy()
    vd = -kd
    wk, wv = oracle_mod.sliding_window(kd, vd, 3)
    assert wk.shape == (B, Hkv, T, 3, d)
    np.testing.assert_array_equal(np.floor(wk[0, 0, 0, :, 0]), [2, 3, 4])
    np.testing.assert_array_equal(wv, -wk)
    w1k, _ = oracle_mod.sliding_window(kd, vd, 1)
    np.testing.assert_array_equal(np.floor(w1k[..., 0, 0]), 4)
    allk, allv = oracle_mod.sliding_window(kd, vd, 9)
    np.testing.assert_array_equal(allk, kd)
    np.testing.assert_array_equal(allv, vd)


def test_oracle_forward_does_not_depend_on_slot_order(oracle_mod):
    """The joint softmax is a sum over its keys, so permuting a position's slots (keys and
    values together) leaves o and lse unchanged; permuting the keys alone does not."""
    q, k, v, kd, vd = rand_problem(1, 4, 2, 9, 6, 8, seed=91)
    perm = np.array([3, 0, 5, 1, 4, 2])
    o1, l1 = oracle_mod.forward(q, k, v, kd, vd)
    o2, l2 = oracle_mod.forward(q, k, v, kd[:, :, :, perm], vd[:, :, :, perm])
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)
    o3, _ = oracle_mod.forward(q, k, v, kd[:, :, :, perm], vd)
    assert np.max(np.abs(o3 - o1)) > 1e-3


@pytest.mark.parametrize("n_writes", [2, 4, 7, 11])
def test_oracle_ring_buffer_realises_the_window(oracle_mod, n_writes):
    """A ring of C slots written at w mod C and read over its first min(n, C) slots gives
    the forward over the sliding window of the last C writes (brute-force ring, tiny case)."""
    B, H, Hkv, T, d, C = 1, 2, 1, 5, 4, 4
    rng = np.random.default_rng(92 + n_writes)
    q, k, v = (rng.standard_normal(s) for s in ((B, H, T, d), (B, Hkv, T, d), (B, Hkv, T, d)))
    hist_k = rng.standard_normal((B, Hkv, T, n_writes, d))
    hist_v = rng.standard_normal((B, Hkv, T, n_writes, d))
    ring_k = np.full((B, Hkv, T, C, d), 7.0)  # finite junk in slots never written
    ring_v = np.full((B, Hkv, T, C, d), -7.0)
    for w in range(n_writes):
        for b in range(B):
            for g in range(Hkv):
                for t in range(T):
                    ring_k[b, g, t, w % C] = hist_k[b, g, t, w]
                    ring_v[b, g, t, w % C] = hist_v[b, g, t, w]
    n_read = min(n_writes, C)
    o_ring, l_ring = oracle_mod.forward(q, k, v, ring_k[:, :, :, :n_read], ring_v[:, :, :, :n_read])
    o_win, l_win = oracle_mod.forward(q, k, v, *oracle_mod.sliding_window(hist_k, hist_v, C))
    np.testing.assert_allclose(o_ring, o_win, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_ring, l_win, rtol=0, atol=1e-12)
