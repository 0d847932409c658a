"""Pins for the oracle's attention (CPU only).

Each test checks ``oracle.attend_rows`` against something other than itself:
closed forms, invariants of exact softmax attention, the dense-mask form of
"llama.cpp 0.9.0 inference boundaries" section 1, or an independent
pure-Python brute force on tiny inputs.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def _rand(seed, shape):
    return np.random.default_rng(seed).standard_normal(shape)


def _pool(seed, R=12, H=2, D=4):
    g = np.random.default_rng(seed)
    return g.standard_normal((R, H, D)), g.standard_normal((R, H, D))


# --- closed forms --------------------------------------------------------------


def test_single_listed_row_returns_that_value_row():
    k, v = _pool(1)
    q = _rand(2, (1, 1, 4, 4))
    rows = np.array([[-1, 7, -1, -5]], dtype=np.int32)
    o, lse = oracle.attend_rows(q, k, v, rows, 0.37)
    for h in range(4):
        np.testing.assert_array_equal(o[0, 0, h], v[7, h // 2])
        assert lse[0, 0, h] == pytest.approx(0.37 * float(q[0, 0, h] @ k[7, h // 2]), rel=1e-15)


def test_zero_query_gives_mean_of_listed_values_and_log_count():
    k, v = _pool(3, R=20)
    q = np.zeros((1, 1, 2, 4))
    rows = np.array([[4, -1, 9, 11, 2, -1]], dtype=np.int32)
    o, lse = oracle.attend_rows(q, k, v, rows, 5.0)
    listed = [4, 9, 11, 2]
    for h in range(2):
        np.testing.assert_allclose(o[0, 0, h], v[listed, h // 1].mean(axis=0), rtol=1e-14, atol=1e-15)
        assert lse[0, 0, h] == pytest.approx(math.log(4), rel=1e-14)


def test_identical_keys_give_mean_of_values():
    k, v = _pool(4, R=10, H=1)
    k[:] = k[0]
    q = _rand(5, (1, 1, 1, 4))
    rows = np.array([[1, 3, 5, 7]], dtype=np.int32)
    o, _ = oracle.attend_rows(q, k, v, rows, 1.0)
    np.testing.assert_allclose(o[0, 0, 0], v[[1, 3, 5, 7], 0].mean(axis=0), rtol=1e-13)


def test_dominant_logit_selects_its_value_row():
    k, v = _pool(6, R=10, H=1)
    q = np.ones((1, 1, 1, 4))
    k[6, 0] = 300.0          # logit 1200 vs O(1) for the others
    rows = np.array([[0, 6, 2, 9]], dtype=np.int32)
    o, _ = oracle.attend_rows(q, k, v, rows, 1.0)
    np.testing.assert_array_equal(o[0, 0, 0], v[6, 0])


def test_two_row_softmax_weight_closed_form():
    # K rows are basis vectors, so the logits are scale*q[0] and scale*q[1]
    D = 4
    k = np.zeros((3, 1, D)); k[0, 0, 0] = 1.0; k[2, 0, 1] = 1.0
    v = np.zeros((3, 1, D)); v[0, 0, 2] = 1.0; v[2, 0, 3] = 1.0
    q = np.array([0.8, -1.3, 0.0, 0.0]).reshape(1, 1, 1, D)
    t = 0.7
    o, lse = oracle.attend_rows(q, k, v, np.array([[2, 0]], dtype=np.int32), t)
    p0 = 1.0 / (1.0 + math.exp(t * (-1.3 - 0.8)))   # weight on pool row 0
    np.testing.assert_allclose(o[0, 0, 0], [0, 0, p0, 1 - p0], rtol=1e-14, atol=1e-16)
    assert lse[0, 0, 0] == pytest.approx(math.log(math.exp(t * 0.8) + math.exp(t * -1.3)), rel=1e-14)


def test_mask_is_additive_and_list_aligned():
    # zero query: weights are exp(mask_j), so O = sum c_j V_j / sum c_j with mask = log c
    k, v = _pool(7, R=9, H=1)
    q = np.zeros((1, 2, 1, 4))
    rows = np.array([[8, 1, 4]], dtype=np.int32)
    c = np.array([[1.0, 2.0, 5.0], [3.0, 0.5, 0.25]])
    mask = np.log(c)[None]
    o, lse = oracle.attend_rows(q, k, v, rows, 1.0, mask=mask)
    for i in range(2):
        want = (c[i, 0] * v[8, 0] + c[i, 1] * v[1, 0] + c[i, 2] * v[4, 0]) / c[i].sum()
        np.testing.assert_allclose(o[0, i, 0], want, rtol=1e-14)
        assert lse[0, i, 0] == pytest.approx(math.log(c[i].sum()), rel=1e-14)


def test_gqa_maps_consecutive_query_heads_to_one_kv_head():
    R, Hkv, D = 6, 2, 4
    k = np.zeros((R, Hkv, D))
    v = np.zeros((R, Hkv, D)); v[:, 0, :] = 1.0; v[:, 1, :] = 2.0
    q = _rand(8, (1, 1, 4, D))
    o, _ = oracle.attend_rows(q, k, v, np.array([[0, 3, 5]], dtype=np.int32), 1.0)
    assert [o[0, 0, h, 0] for h in range(4)] == [1.0, 1.0, 2.0, 2.0]


def test_causal_bottom_right_gives_prefix_means():
    # zero query + causal: query i of Nq sees the first n - Nq + i + 1 list entries
    k, v = _pool(9, R=10, H=1)
    q = np.zeros((1, 3, 1, 4))
    rows = np.array([[9, 2, 7, 0, 5]], dtype=np.int32)
    o, lse = oracle.attend_rows(q, k, v, rows, 1.0, causal=True)
    for i, upto in enumerate([3, 4, 5]):
        np.testing.assert_allclose(o[0, i, 0], v[rows[0, :upto], 0].mean(axis=0), rtol=1e-14)
        assert lse[0, i, 0] == pytest.approx(math.log(upto), rel=1e-14)


def test_kv_len_cuts_the_list_and_causal_uses_it():
    k, v = _pool(10, R=10, H=1)
    q = np.zeros((1, 2, 1, 4))
    rows = np.array([[9, 2, 7, 0, 5, 3]], dtype=np.int32)
    o, _ = oracle.attend_rows(q, k, v, rows, 1.0, causal=True, kv_len=np.array([4]))
    np.testing.assert_allclose(o[0, 0, 0], v[[9, 2, 7], 0].mean(axis=0), rtol=1e-14)
    np.testing.assert_allclose(o[0, 1, 0], v[[9, 2, 7, 0], 0].mean(axis=0), rtol=1e-14)


def test_empty_and_fully_masked_rows_give_zero_and_minus_inf():
    k, v = _pool(11)
    q = _rand(12, (2, 1, 2, 4))
    rows = np.array([[-1, -1, -1], [1, 2, 3]], dtype=np.int32)
    mask = np.zeros((2, 1, 3)); mask[1] = -np.inf
    o, lse = oracle.attend_rows(q, k, v, rows, 1.0, mask=mask)
    assert np.all(o == 0) and np.all(lse == -np.inf)


# --- invariants ------------------------------------------------------------------


def test_permuting_the_list_with_its_mask_leaves_output_unchanged():
    p = synth.random_problem(21, S=2, Nq=2, Hq=4, Hkv=2, D=16, R=40, L=25, with_mask=True)
    q, k, v = (oracle.widen_bf16(a) for a in (p.q, p.k, p.v))
    perm = np.random.default_rng(5).permutation(p.L)
    o1, l1 = oracle.attend_rows(q, k, v, p.kv_rows, p.scale, mask=p.mask)
    o2, l2 = oracle.attend_rows(q, k, v, p.kv_rows[:, perm], p.scale, mask=p.mask[:, :, perm])
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-13)


@pytest.mark.parametrize("poison", [np.nan, 1e30, -np.inf])
def test_unlisted_and_cut_rows_have_no_effect_even_when_poisoned(poison):
    p = synth.random_problem(22, S=2, Nq=1, Hq=4, Hkv=2, D=16, R=50, L=20, kv_len=True)
    q, k, v = (oracle.widen_bf16(a) for a in (p.q, p.k, p.v))
    o1, l1 = oracle.attend_rows(q, k, v, p.kv_rows, p.scale, kv_len=p.kv_len)
    used = set()
    for s in range(p.S):
        used |= {int(r) for r in p.kv_rows[s, :p.kv_len[s]] if r >= 0}
    k2, v2 = k.copy(), v.copy()
    for r in range(p.R):
        if r not in used:
            k2[r] = poison
            v2[r] = poison
    o2, l2 = oracle.attend_rows(q, k2, v2, p.kv_rows, p.scale, kv_len=p.kv_len)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_constant_mask_shift_changes_only_lse():
    p = synth.random_problem(23, S=1, Nq=2, Hq=2, Hkv=1, D=16, R=30, L=12, with_mask=True)
    q, k, v = (oracle.widen_bf16(a) for a in (p.q, p.k, p.v))
    m64 = p.mask.astype(np.float64)
    o1, l1 = oracle.attend_rows(q, k, v, p.kv_rows, p.scale, mask=m64)
    o2, l2 = oracle.attend_rows(q, k, v, p.kv_rows, p.scale, mask=m64 + 3.25)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l2 - l1, 3.25, rtol=1e-12)


def test_minus_inf_mask_equals_padding():
    p = synth.random_problem(24, S=1, Nq=1, Hq=2, Hkv=1, D=16, R=30, L=12, pad_frac=0.0)
    q, k, v = (oracle.widen_bf16(a) for a in (p.q, p.k, p.v))
    mask = np.zeros((1, 1, 12)); mask[0, 0, [2, 5, 6]] = -np.inf
    rows2 = p.kv_rows.copy(); rows2[0, [2, 5, 6]] = -1
    o1, l1 = oracle.attend_rows(q, k, v, p.kv_rows, p.scale, mask=mask)
    o2, l2 = oracle.attend_rows(q, k, v, rows2, p.scale)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# --- the dense-mask formulation (the path the row lists replace) -----------------


@pytest.mark.parametrize("seed,kw", [
    (31, dict()),
    (32, dict(with_mask=True)),
    (33, dict(causal=True, Nq=3)),
    (34, dict(kv_len=True, Nq=2, causal=True)),
    (35, dict(with_mask=True, neg_inf_frac=0.3, Nq=2)),
    (36, dict(Hq=8, Hkv=2, dtype="f16")),
])
def test_rows_form_equals_dense_mask_over_the_whole_pool(seed, kw):
    base = dict(S=2, Nq=1, Hq=4, Hkv=2, D=16, R=64, L=30)
    base.update(kw)
    p = synth.random_problem(seed, **base)
    w = oracle.widen_bf16 if p.dtype == "bf16" else oracle.widen_f16
    q, k, v = w(p.q), w(p.k), w(p.v)
    args = dict(mask=p.mask, causal=p.causal, kv_len=p.kv_len)
    o1, l1 = oracle.attend_rows(q, k, v, p.kv_rows, p.scale, **args)
    o2, l2 = oracle.attend_dense(q, k, v, p.kv_rows, p.scale, **args)
    np.testing.assert_allclose(o1, o2, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-12)


# --- brute force on tiny inputs (independent pure-Python enumeration) -------------


def _brute(q, k, v, rows, scale, mask, causal, kv_len):
    S, Nq, Hq, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv = len(k[0])
    per_group = Hq // Hkv
    res = {}
    for s in range(S):
        n = len(rows[s]) if kv_len is None else kv_len[s]
        for i in range(Nq):
            for h in range(Hq):
                kvh = 0
                while (kvh + 1) * per_group <= h:   # find the KV head by counting groups
                    kvh += 1
                terms = []
                for j, r in enumerate(rows[s]):
                    if j >= n or r < 0:
                        continue
                    if causal and j > n - Nq + i:
                        continue
                    dot = math.fsum(q[s][i][h][d] * k[r][kvh][d] for d in range(D))
                    logit = scale * dot + (0.0 if mask is None else mask[s][i][j])
                    if logit == -math.inf:
                        continue
                    terms.append((math.exp(logit), r))
                if not terms:
                    res[s, i, h] = [0.0] * D
                    continue
                z = math.fsum(t for t, _ in terms)
                res[s, i, h] = [math.fsum(t * v[r][kvh][d] for t, r in terms) / z for d in range(D)]
    return res


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_tiny(seed):
    g = np.random.default_rng(100 + seed)
    S, Nq, Hq, Hkv, D, R, L = 2, 2, 4, 2, 3, 7, 5
    # small dyadic values keep every product exact
    q = g.integers(-4, 5, size=(S, Nq, Hq, D)) / 4.0
    k = g.integers(-4, 5, size=(R, Hkv, D)) / 4.0
    v = g.integers(-8, 9, size=(R, Hkv, D)) / 8.0
    rows = np.stack([g.permutation(R)[:L] for _ in range(S)]).astype(np.int32)
    rows[g.random((S, L)) < 0.25] = -1
    mask = (g.integers(-2, 3, size=(S, Nq, L)) / 2.0) if seed % 2 else None
    if mask is not None:
        mask[0, 0, 1] = -np.inf
    causal = seed >= 3
    kv_len = np.array([L, L - 1]) if seed == 5 else None
    o, _ = oracle.attend_rows(q, k, v, rows, 0.5, mask=mask, causal=causal, kv_len=kv_len)
    ref = _brute(q.tolist(), k.tolist(), v.tolist(), rows.tolist(), 0.5,
                 None if mask is None else mask.tolist(), causal, None if kv_len is None else kv_len.tolist())
    for (s, i, h), want in ref.items():
        np.testing.assert_allclose(o[s, i, h], want, rtol=1e-12, atol=1e-15)


def test_query_rows_subset_matches_full_evaluation():
    p = synth.random_problem(40, S=2, Nq=6, Hq=4, Hkv=2, D=16, R=64, L=40, causal=True, with_mask=True)
    q, k, v = (oracle.widen_bf16(a) for a in (p.q, p.k, p.v))
    o_full, l_full = oracle.attend_rows(q, k, v, p.kv_rows, p.scale, mask=p.mask, causal=True)
    sel = [1, 4, 5]
    o_sub, l_sub = oracle.attend_rows(q[:, sel], k, v, p.kv_rows, p.scale, mask=p.mask, causal=True,
                                      query_rows=sel, n_query=6)
    np.testing.assert_array_equal(o_sub, o_full[:, sel])
    np.testing.assert_array_equal(l_sub, l_full[:, sel])


def test_raw_bits_input_matches_widened_input():
    p = synth.random_problem(41, S=1, Nq=1, Hq=2, Hkv=1, D=16, R=30, L=10)
    q, k, v = (oracle.widen_bf16(a) for a in (p.q, p.k, p.v))
    o1, _ = oracle.attend_rows(q, k, v, p.kv_rows, p.scale)
    o2, _ = oracle.attend_rows(q, p.k, p.v, p.kv_rows, p.scale, kv_format="bf16")
    np.testing.assert_array_equal(o1, o2)
