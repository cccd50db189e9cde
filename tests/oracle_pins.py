"""Checks that pin the float64 oracle to facts outside itself.

Each ``check_*`` function raises AssertionError when the oracle disagrees with
something the pages or the mathematics fix: values worked out by hand from
the definition, a brute-force formula written differently, a library routine
computing the same definition, closed-form special cases, the online-softmax
recurrence of the pages, and the paged-cache layout.  ``test_oracle_pins.py``
runs them on the oracle; ``test_oracle_mutants.py`` runs them on deliberately
broken copies of the oracle to show each plausible mistake is caught.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _expr(s: str) -> float:
    # Fixture expressions only use numbers, + - * /, and ln().
    return float(eval(s, {"__builtins__": {}}, {"ln": math.log}))


def check_hand_examples():
    """Hand-derived examples (tests/golden/hand_examples.json)."""
    with open(os.path.join(GOLDEN, "hand_examples.json")) as f:
        fx = json.load(f)
    for ex in fx["examples"]:
        q = np.array([[_expr(c) for c in r] for r in ex["q"]])[None, None]
        k = np.array([[_expr(c) for c in r] for r in ex["k"]])[None, None]
        v = np.array([[_expr(c) for c in r] for r in ex["v"]])[None, None]
        for mode, causal in (("noncausal", False), ("causal", True)):
            o, lse = oracle.attention_forward(q, k, v, ex["scale"], causal)
            want_o = np.array([[_expr(c) for c in r] for r in ex[mode]["o"]])
            want_lse = np.array([_expr(c) for c in ex[mode]["lse"]])
            np.testing.assert_allclose(o[0, 0], want_o, rtol=0, atol=1e-13,
                                       err_msg=f"{ex['name']} {mode} O")
            np.testing.assert_allclose(lse[0, 0], want_lse, rtol=0, atol=1e-13,
                                       err_msg=f"{ex['name']} {mode} LSE")


def _brute(q, k, v, scale, causal):
    """Attention for one head by direct e^s / sum e^s, no max subtraction,
    pure-Python loops (valid for the small scores used here)."""
    N, d = len(q), len(q[0])
    O = [[0.0] * d for _ in range(N)]
    L = [0.0] * N
    for i in range(N):
        js = range(i + 1) if causal else range(N)
        w = {j: math.exp(scale * math.fsum(q[i][c] * k[j][c] for c in range(d))) for j in js}
        z = math.fsum(w.values())
        for c in range(d):
            O[i][c] = math.fsum(w[j] * v[j][c] for j in js) / z
        L[i] = math.log(z)
    return np.array(O), np.array(L)


def check_brute_force_tiny():
    """Brute force on 4x4 (and a non-square 5x3) single-head problems."""
    r = _rng(11)
    for N, d in ((4, 4), (5, 3), (1, 4)):
        q, k, v = (r.standard_normal((N, d)) for _ in range(3))
        for causal in (False, True):
            scale = 0.7
            o, lse = oracle.attention_forward(q[None, None], k[None, None], v[None, None],
                                              scale, causal)
            bo, bl = _brute(q.tolist(), k.tolist(), v.tolist(), scale, causal)
            np.testing.assert_allclose(o[0, 0], bo, rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(lse[0, 0], bl, rtol=1e-13, atol=1e-14)


def check_library_sdpa():
    """PyTorch's float64 scaled_dot_product_attention on the CPU computes the
    same definition (youngju.dev, section 11); LSE via torch.logsumexp."""
    F = torch.nn.functional
    g = torch.Generator().manual_seed(5)
    for (B, H, N, d, causal) in ((1, 1, 64, 64, False), (2, 3, 77, 64, True),
                                 (1, 2, 130, 128, False), (1, 2, 129, 128, True)):
        q, k, v = (torch.randn(B, H, N, d, generator=g, dtype=torch.float64) for _ in range(3))
        scale = 1.0 / math.sqrt(d)
        o, lse = oracle.attention_forward(q, k, v, scale, causal)
        ref = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
        s = torch.einsum("bhid,bhjd->bhij", q, k) * scale
        if causal:
            s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
        ref_lse = torch.logsumexp(s, dim=-1)
        np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)
        rows = [0, N // 3, N - 1]
        o_r, l_r = oracle.attention_forward_rows(q, k, v, rows, scale, causal)
        np.testing.assert_array_equal(o_r, o[:, :, rows])
        np.testing.assert_array_equal(l_r, lse[:, :, rows])


def check_invariants():
    """Special cases that follow from the definition (eq. (1))."""
    r = _rng(3)
    N, d = 37, 8
    k = r.standard_normal((1, 1, N, d))
    v = r.standard_normal((1, 1, N, d))
    q = r.standard_normal((1, 1, N, d))
    # Rows of P sum to one and are non-negative.
    for causal in (False, True):
        for i in (0, 5, N - 1):
            p = oracle.probs_row(q[0, 0], k[0, 0], i, 0.5, causal)
            assert abs(p.sum() - 1.0) < 1e-14 and (p >= 0).all()
            if causal:
                assert (p[i + 1:] == 0).all()
    # Q = 0: uniform weights -> column mean of V, LSE = ln N (causal: prefix).
    z = np.zeros_like(q)
    o, lse = oracle.attention_forward(z, k, v, 1.0, False)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0].mean(0), (N, d)), atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], np.full(N, math.log(N)), atol=1e-14)
    o, lse = oracle.attention_forward(z, k, v, 1.0, True)
    prefix = np.cumsum(v[0, 0], axis=0) / np.arange(1, N + 1)[:, None]
    np.testing.assert_allclose(o[0, 0], prefix, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], np.log(np.arange(1, N + 1)), atol=1e-14)
    # Identical V rows -> that row, whatever the weights.
    row = r.standard_normal(d)
    o, _ = oracle.attention_forward(q, k, np.broadcast_to(row, (1, 1, N, d)), 0.9, False)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(row, (N, d)), atol=1e-14)
    # Causal row 0 sees only key 0: O_0 = V_0 exactly, LSE_0 = s_00.
    o, lse = oracle.attention_forward(q, k, v, 0.3, True)
    np.testing.assert_array_equal(o[0, 0, 0], v[0, 0, 0])
    assert abs(lse[0, 0, 0] - 0.3 * float(q[0, 0, 0] @ k[0, 0, 0])) < 1e-14
    # Joint permutation of key/value rows leaves non-causal attention unchanged.
    perm = r.permutation(N)
    o1, l1 = oracle.attention_forward(q, k, v, 0.3, False)
    o2, l2 = oracle.attention_forward(q, k[:, :, perm], v[:, :, perm], 0.3, False)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)
    # Shifting every key by u adds scale*q_i.u to row i: O unchanged, LSE shifts.
    u = r.standard_normal(d)
    o3, l3 = oracle.attention_forward(q, k + u, v, 0.3, True)
    o4, l4 = oracle.attention_forward(q, k, v, 0.3, True)
    np.testing.assert_allclose(o3, o4, atol=1e-12)
    np.testing.assert_allclose(l3[0, 0], l4[0, 0] + 0.3 * (q[0, 0] @ u), atol=1e-12)


def check_large_logits():
    """Scores of magnitude ~1e3 overflow exp() unless the row max is
    subtracted first (safe softmax, eq. (1)); the result must stay finite and
    pick the dominant key."""
    N, d = 6, 2
    q = np.zeros((1, 1, N, d)); q[..., 0] = 1.0
    k = np.zeros((1, 1, N, d)); k[0, 0, :, 0] = [-900.0, 200.0, 1000.0, 300.0, -50.0, 999.0]
    v = np.arange(N * d, dtype=np.float64).reshape(1, 1, N, d)
    o, lse = oracle.attention_forward(q, k, v, 1.0, False)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    w = np.exp(k[0, 0, :, 0] - 1000.0)
    np.testing.assert_allclose(o[0, 0, 0], (w[:, None] * v[0, 0]).sum(0) / w.sum(), atol=1e-12)
    np.testing.assert_allclose(lse[0, 0, 0], 1000.0 + math.log(w.sum()), atol=1e-12)


def online_softmax_blockwise(q, k, v, scale, causal, block):
    """Blockwise forward for one head, following the online-softmax updates
    of "Flash Attention" (suniverse77.github.io, section "Online Softmax"):
    eq. (2) for the running max, eq. (3) for the running sum and eq. (4) to
    merge the normalised block output with the running output."""
    N, d = q.shape
    O = np.zeros((N, d)); L = np.zeros(N)
    for i in range(N):
        m_old, l_old, o_old = -np.inf, 0.0, np.zeros(d)
        last = i + 1 if causal else N
        for j0 in range(0, last, block):
            j1 = min(last, j0 + block)
            x = scale * (k[j0:j1] @ q[i])
            m_now = x.max()
            e = np.exp(x - m_now)
            l_now = e.sum()
            o_now = (e @ v[j0:j1]) / l_now
            m_new = max(m_old, m_now)                                   # eq. (2)
            l_new = l_old * np.exp(m_old - m_new) + np.exp(x - m_new).sum()  # eq. (3)
            o_new = (o_old * l_old * np.exp(m_old - m_new)
                     + o_now * l_now * np.exp(m_now - m_new)) / l_new    # eq. (4)
            m_old, l_old, o_old = m_new, l_new, o_new
        O[i], L[i] = o_old, m_old + np.log(l_old)
    return O, L


def check_online_recurrence():
    """The recurrence of eqs. (2)-(4), at any block size, reaches the
    materialised definition: the method is exact."""
    r = _rng(8)
    N, d = 45, 16
    q, k, v = (r.standard_normal((N, d)) for _ in range(3))
    for causal in (False, True):
        o, lse = oracle.attention_forward(q[None, None], k[None, None], v[None, None], 0.25, causal)
        for block in (1, 7, 16, 64):
            bo, bl = online_softmax_blockwise(q, k, v, 0.25, causal, block)
            np.testing.assert_allclose(o[0, 0], bo, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[0, 0], bl, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Paged decode

def k_flat(pb, h, tok, c, H, D, bs, x):
    """Flat element offset of key element c of the token at offset ``tok``
    of physical block pb, head h, in k_cache [nb, H, D/x, bs, x]."""
    return pb * (H * D * bs) + h * (D * bs) + (c // x) * (bs * x) + tok * x + (c % x)


def v_flat(pb, h, tok, c, H, D, bs):
    """Same for value element c in v_cache [nb, H, D, bs]."""
    return pb * (H * D * bs) + h * (D * bs) + c * bs + tok


def check_layout_fixture():
    """The worked layout numbers of the PagedAttention page and hand-derived
    flat offsets (tests/golden/paged_layout.json)."""
    with open(os.path.join(GOLDEN, "paged_layout.json")) as f:
        fx = json.load(f)
    sh = fx["shape"]
    H, D, bs, x = sh["num_heads"], sh["head_size"], sh["block_size"], sh["x"]
    vals = [e["value"] for e in fx["page_numbers"]]
    assert vals[0] == bs * D                      # 16 x 128 elements per block and head
    assert vals[1] == 16 // (2 * 2)               # 16 B over 2 threads of 2-byte elements
    assert vals[2] == 16 // 2 == fx["x_for_2_byte_types"] == x
    assert vals[3] == D * bs // (32 * vals[2])    # 128*16/256
    assert fx["derived_strides"]["kv_block_stride"] == H * D * bs
    assert fx["derived_strides"]["kv_head_stride"] == D * bs == vals[0]
    nb = 16384
    for e in fx["offsets"]:
        args = (e["pb"], e["head"], e["token_in_block"], e["dim"])
        assert k_flat(*args, H, D, bs, x) == e["k_flat"]
        assert v_flat(*args, H, D, bs) == e["v_flat"]
        # numpy's C-order indexing over the page's shapes agrees.
        pb, h, t, c = args
        assert np.ravel_multi_index((pb, h, c // x, t, c % x), (nb, H, D // x, bs, x)) == e["k_flat"]
        assert np.ravel_multi_index((pb, h, c, t), (nb, H, D, bs)) == e["v_flat"]


def _scatter_cache(Ks, Vs, tables, H, D, bs, x, nb):
    """Write each sequence's logical keys/values into flat paged caches."""
    kc = np.zeros(nb * H * D * bs)
    vc = np.zeros(nb * H * D * bs)
    for s, (K, V) in enumerate(zip(Ks, Vs)):
        ctx = K.shape[1]
        for h in range(H):
            for t in range(ctx):
                pb = tables[s][t // bs]
                for c in range(D):
                    kc[k_flat(pb, h, t % bs, c, H, D, bs, x)] = K[h, t, c]
                    vc[v_flat(pb, h, t % bs, c, H, D, bs)] = V[h, t, c]
    return kc.reshape(nb, H, D // x, bs, x), vc.reshape(nb, H, D, bs)


def _decode_case(seed, S=5, H=3, D=16, bs=4, x=8, max_blocks=6):
    r = _rng(seed)
    nb = S * max_blocks + 3
    ctx = [1, bs, bs + 1, max_blocks * bs, 7][:S]
    tables = r.permutation(nb)[:S * max_blocks].reshape(S, max_blocks)
    Ks = [r.standard_normal((H, c, D)) for c in ctx]
    Vs = [r.standard_normal((H, c, D)) for c in ctx]
    q = r.standard_normal((S, H, D))
    kc, vc = _scatter_cache(Ks, Vs, tables, H, D, bs, x, nb)
    return q, kc, vc, tables.astype(np.int32), np.array(ctx, dtype=np.int32), Ks, Vs


def check_decode_matches_gathered_forward():
    """Decode through the block table equals a single-query forward over the
    sequence's contiguous keys and values."""
    q, kc, vc, bt, cl, Ks, Vs = _decode_case(21)
    scale = 0.25
    out, lse = oracle.paged_decode(q, kc, vc, bt, cl, scale)
    for s in range(q.shape[0]):
        c = int(cl[s])
        for h in range(q.shape[1]):
            Q = np.zeros((1, 1, c, q.shape[2])); Q[0, 0, c - 1] = q[s, h]
            o, l = oracle.attention_forward_rows(Q, Ks[s][h][None, None], Vs[s][h][None, None],
                                                 [c - 1], scale, False)
            np.testing.assert_allclose(out[s, h], o[0, 0, 0], atol=1e-13)
            np.testing.assert_allclose(lse[s, h], l[0, 0, 0], atol=1e-13)


def check_decode_one_hot():
    """A key aligned with the query and far larger than the rest selects its
    own value row: the decode gathers the right token for each position."""
    S, H, D, bs, x, mb = 2, 2, 16, 4, 8, 5
    r = _rng(4)
    nb = S * mb
    tables = r.permutation(nb).reshape(S, mb)
    ctx = [17, 9]
    q = np.zeros((S, H, D)); q[:, :, 3] = 1.0
    for s in range(S):
        for target in (0, ctx[s] // 2, ctx[s] - 1):
            Ks = [np.zeros((H, c, D)) for c in ctx]
            Vs = [r.standard_normal((H, c, D)) for c in ctx]
            for h in range(H):
                Ks[s][h, target, 3] = 60.0
            kc, vc = _scatter_cache(Ks, Vs, tables, H, D, bs, x, nb)
            out, lse = oracle.paged_decode(q, kc, vc, tables.astype(np.int32),
                                           np.array(ctx, dtype=np.int32), 1.0)
            for h in range(H):
                np.testing.assert_allclose(out[s, h], Vs[s][h, target], rtol=0, atol=1e-20)


def check_gqa_decode_matches_replicated_heads():
    """Grouped key/value heads ("PagedAttention", data-sketchers.com, section
    "Inputs": the caches have a num_kv_heads axis): the decode with Hk key/value
    heads equals the one-head-per-query decode on caches in which every key/value
    head is repeated for its H/Hk consecutive query heads -- bit for bit, since the
    gathers and sums are the same."""
    for Hk, H in ((2, 8), (1, 4), (3, 3)):
        r = _rng(31 + H)
        S, D, bs, x, mb = 3, 16, 4, 8, 5
        nb = S * mb + 2
        tables = r.permutation(nb)[:S * mb].reshape(S, mb).astype(np.int32)
        ctx = np.array([1, 9, mb * bs], dtype=np.int32)
        q = r.standard_normal((S, H, D))
        kc = r.standard_normal((nb, Hk, D // x, bs, x))
        vc = r.standard_normal((nb, Hk, D, bs))
        G = H // Hk
        out_g, lse_g = oracle.paged_decode(q, kc, vc, tables, ctx, 0.3)
        out_m, lse_m = oracle.paged_decode(q, np.repeat(kc, G, axis=1), np.repeat(vc, G, axis=1),
                                           tables, ctx, 0.3)
        np.testing.assert_array_equal(out_g, out_m)
        np.testing.assert_array_equal(lse_g, lse_m)


def check_gqa_decode_head_groups():
    """Values constant per key/value head (head j holds j + 1 everywhere) make
    every output row equal that constant whatever the probabilities, so query
    head h must read key/value head h // (H / Hk)."""
    S, H, Hk, D, bs, x, mb = 2, 6, 3, 8, 4, 8, 3
    r = _rng(37)
    nb = S * mb
    tables = r.permutation(nb).reshape(S, mb).astype(np.int32)
    ctx = np.array([5, 12], dtype=np.int32)
    q = r.standard_normal((S, H, D))
    kc = r.standard_normal((nb, Hk, D // x, bs, x))
    vc = np.zeros((nb, Hk, D, bs))
    for j in range(Hk):
        vc[:, j] = j + 1.0
    out, _ = oracle.paged_decode(q, kc, vc, tables, ctx, 0.5)
    for h in range(H):
        np.testing.assert_allclose(out[:, h], h // (H // Hk) + 1.0, rtol=0, atol=1e-12)


ALL_CHECKS = [check_hand_examples, check_brute_force_tiny, check_library_sdpa,
              check_invariants, check_large_logits, check_online_recurrence,
              check_layout_fixture, check_decode_matches_gathered_forward,
              check_decode_one_hot, check_gqa_decode_matches_replicated_heads,
              check_gqa_decode_head_groups]
# (the mask checks are appended below, after their definitions)


# --------------------------------------------------------------------------
# Boolean attention mask ("FlashAttention: GPU 메모리 계층을 활용한 어텐션 최적화
# 분석", youngju.dev, section 11.3: attn_mask = tril(ones) as a custom mask)

def check_mask_special_cases():
    """tril(ones) reproduces the causal forward and ones the full forward, bit
    for bit (the same keys in the same order); one visible key per row selects
    its value row exactly with LSE = its score; an all-False row gives O = 0
    and LSE = -inf."""
    r = _rng(41)
    B, H, N, d, scale = 1, 2, 23, 8, 0.4
    q, k, v = (r.standard_normal((B, H, N, d)) for _ in range(3))
    tril = np.tril(np.ones((N, N), dtype=np.uint8))
    o_m, l_m = oracle.attention_forward_masked(q, k, v, tril, scale)
    o_c, l_c = oracle.attention_forward(q, k, v, scale, True)
    np.testing.assert_array_equal(o_m, o_c)
    np.testing.assert_array_equal(l_m, l_c)
    o_m, l_m = oracle.attention_forward_masked(q, k, v, np.ones((N, N), dtype=np.uint8), scale)
    o_f, l_f = oracle.attention_forward(q, k, v, scale, False)
    np.testing.assert_array_equal(o_m, o_f)
    np.testing.assert_array_equal(l_m, l_f)
    pick = r.integers(0, N, size=N)
    one = np.zeros((N, N), dtype=np.uint8)
    one[np.arange(N), pick] = 1
    one[5] = 0                                   # row 5: nothing visible
    o1, l1 = oracle.attention_forward_masked(q, k, v, one, scale)
    for i in range(N):
        if i == 5:
            np.testing.assert_array_equal(o1[:, :, i], 0.0)
            assert np.all(np.isneginf(l1[:, :, i]))
            continue
        np.testing.assert_array_equal(o1[:, :, i], v[:, :, pick[i]])
        np.testing.assert_allclose(l1[:, :, i],
                                   scale * np.einsum("bhc,bhc->bh", q[:, :, i], k[:, :, pick[i]]),
                                   rtol=0, atol=1e-13)


def check_mask_brute_force():
    """Random masks on tiny heads against a pure-Python softmax over the visible
    keys, including a different mask per head."""
    r = _rng(43)
    B, H, N, d, scale = 2, 2, 6, 3, 0.7
    q, k, v = (r.standard_normal((B, H, N, d)) for _ in range(3))
    masks = (r.random((B, H, N, N)) < 0.5).astype(np.uint8)
    masks[0, 1, 2] = 0
    o, lse = oracle.attention_forward_masked(q, k, v, masks, scale)
    for b in range(B):
        for h in range(H):
            for i in range(N):
                vis = [j for j in range(N) if masks[b, h, i, j]]
                if not vis:
                    assert np.all(o[b, h, i] == 0) and np.isneginf(lse[b, h, i])
                    continue
                sc = [scale * sum(q[b, h, i, c] * k[b, h, j, c] for c in range(d)) for j in vis]
                mx = max(sc)
                e = [math.exp(x - mx) for x in sc]
                tot = sum(e)
                for c in range(d):
                    want = sum(e[t] / tot * v[b, h, j, c] for t, j in enumerate(vis))
                    assert abs(o[b, h, i, c] - want) <= 1e-12
                assert abs(lse[b, h, i] - (mx + math.log(tot))) <= 1e-12


# --------------------------------------------------------------------------
# Backward

def check_backward_hand_example():
    """Hand-derived gradients (tests/golden/hand_examples.json)."""
    with open(os.path.join(GOLDEN, "hand_examples.json")) as f:
        fx = json.load(f)
    for ex in fx["backward_examples"]:
        arr = lambda key: np.array([[_expr(c) for c in r] for r in ex[key]])[None, None]
        dq, dk, dv = oracle.attention_backward(arr("q"), arr("k"), arr("v"), arr("dout"),
                                               ex["scale"], False)
        for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
            want = np.array([[_expr(c) for c in r] for r in ex["noncausal"][name]])
            np.testing.assert_allclose(got[0, 0], want, rtol=0, atol=1e-13,
                                       err_msg=f"{ex['name']} {name}")


def check_backward_finite_differences():
    """Central differences of L = sum(O * dO), O from the forward oracle,
    agree with the backward oracle on small heads."""
    r = _rng(17)
    for causal in (False, True):
        N, d, scale = 5, 3, 0.6
        q, k, v, do = (r.standard_normal((1, 1, N, d)) for _ in range(4))
        dq, dk, dv = oracle.attention_backward(q, k, v, do, scale, causal)
        h = 1e-6
        for x, g in ((q, dq), (k, dk), (v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(*x.shape):
                old = x[idx]
                x[idx] = old + h
                lp = (oracle.attention_forward(q, k, v, scale, causal)[0] * do).sum()
                x[idx] = old - h
                lm = (oracle.attention_forward(q, k, v, scale, causal)[0] * do).sum()
                x[idx] = old
                num[idx] = (lp - lm) / (2 * h)
            np.testing.assert_allclose(g, num, rtol=0, atol=1e-7)


def check_backward_library_autograd():
    """PyTorch autograd through float64 scaled_dot_product_attention."""
    F = torch.nn.functional
    g = torch.Generator().manual_seed(23)
    for (B, H, N, d, causal) in ((1, 2, 37, 16, True), (2, 1, 50, 8, False)):
        q, k, v, do = (torch.randn(B, H, N, d, generator=g, dtype=torch.float64) for _ in range(4))
        scale = d ** -0.5
        qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
        o = F.scaled_dot_product_attention(qq, kk, vv, is_causal=causal, scale=scale)
        o.backward(do)
        dq, dk, dv = oracle.attention_backward(q, k, v, do, scale, causal)
        for got, ref in ((dq, qq.grad), (dk, kk.grad), (dv, vv.grad)):
            np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-11)


def check_backward_invariants():
    """Rows of P sum to one and each row of dS sums to zero, so the key
    gradients sum to zero and the value gradients sum to the output
    gradients; identical value rows make dQ and dK vanish; causal row 0 has
    one key, so dQ_0 = 0."""
    r = _rng(29)
    N, d = 33, 6
    q, k, v, do = (r.standard_normal((1, 1, N, d)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.5, causal)
        np.testing.assert_allclose(dk[0, 0].sum(axis=0), np.zeros(d), atol=1e-12)
        np.testing.assert_allclose(dv[0, 0].sum(axis=0), do[0, 0].sum(axis=0), atol=1e-12)
        if causal:
            np.testing.assert_allclose(dq[0, 0, 0], np.zeros(d), atol=1e-15)
    same = np.broadcast_to(r.standard_normal(d), (1, 1, N, d)).copy()
    dq, dk, dv = oracle.attention_backward(q, k, same, do, 0.5, True)
    np.testing.assert_allclose(dq, 0, atol=1e-12)
    np.testing.assert_allclose(dk, 0, atol=1e-12)


ALL_CHECKS += [check_mask_special_cases, check_mask_brute_force]
ALL_CHECKS += [check_backward_hand_example, check_backward_finite_differences,
               check_backward_library_autograd, check_backward_invariants]
