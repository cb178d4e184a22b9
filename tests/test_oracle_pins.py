"""Pins of the CPU oracle against things other than itself (CPU only).

Each test fixes part of the oracle by a closed form, a hand-solved example,
brute force on tiny inputs, a library routine (torch's fp32->bf16 rounding,
torch's scaled_dot_product_attention, scipy's logsumexp, Python's sorted) or a
figure the pages print. A dropped term, a wrong sign or index, or a transposed
operand in the oracle fails at least one of them.
"""

import ast
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits_of(x_f32):
    return torch.tensor(np.asarray(x_f32, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def to_bits(a):
    """Exact bf16 values -> bits (asserting exactness)."""
    a = np.asarray(a, dtype=np.float64)
    bits = O.f64_to_bf16_bits(a)
    assert np.array_equal(O.bf16_bits_to_f64(bits), a), "value not exactly representable in bf16"
    return bits


# ----------------------------------------------------------------------------- bf16 rounding

def test_rne_matches_torch_on_fp32_values():
    # torch rounds fp32 -> bf16 to nearest-even; on fp32-exact inputs the oracle must agree.
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-38).astype(np.float32),   # fp32 subnormal range
        (rng.standard_normal(20000) * 1e30).astype(np.float32),
        # exact ties: bf16 value + half a bf16 ulp
        (np.float32(1.0) + np.float32(2.0 ** -8) * np.arange(1, 64, 2, dtype=np.float32)),
    ])
    assert np.array_equal(O.f64_to_bf16_bits(x.astype(np.float64)), bf16_bits_of(x))


def test_rne_hand_cases():
    cases = {
        1.0 + 2.0 ** -8: 0x3F80,                 # tie, even neighbour 1.0
        1.0 + 3 * 2.0 ** -8: 0x3F82,             # tie, even neighbour 1 + 2^-6
        1.0 + 2.0 ** -8 + 2.0 ** -40: 0x3F81,    # just above the tie: a detour via fp32 would give 0x3F80
        -(1.0 + 2.0 ** -8 + 2.0 ** -40): 0xBF81,
        2.0 ** -133: 0x0001,                     # smallest bf16 subnormal
        1.5 * 2.0 ** -133: 0x0002,               # subnormal tie -> even
        0.5 * 2.0 ** -133: 0x0000,               # tie between 0 and 2^-133 -> 0
        3.3895313892515355e38: 0x7F7F,           # largest finite bf16
        3.40e38: 0x7F80,                          # rounds past the top -> +inf
        -0.0: 0x8000,
        2.5: 0x4020,
    }
    for x, want in cases.items():
        assert int(O.f64_to_bf16_bits(x)) == want, (x, hex(int(O.f64_to_bf16_bits(x))), hex(want))
    assert int(O.f64_to_bf16_bits(float("nan"))) == 0x7FC0
    assert int(O.f64_to_bf16_bits(float("-inf"))) == 0xFF80


# ----------------------------------------------------------------------------- pooling

def test_pool_hand_cases():
    raw = np.array([[1.0, 2.0], [2.0, 2.0], [3.0, 2.0], [4.0, 2.0],          # mean (2.5, 2)
                    [1.0, 1.0], [1.0, 1.0 + 2 ** -7], [1.0, 1.0], [1.0, 1.0 + 2 ** -7],  # (1, 1+2^-8 -> tie -> 1)
                    [7.0, 7.0], [7.0, 7.0], [7.0, 7.0]])                     # partial block: not pooled
    pooled = O.bf16_bits_to_f64(O.pool_keys(to_bits(raw)))
    assert pooled.shape == (2, 2)
    assert np.array_equal(pooled, [[2.5, 2.0], [1.0, 1.0]])


def test_pool_matches_torch_mean_when_exact():
    # For 4 bf16 values within a 2^15 magnitude ratio the fp32 sum is exact, so
    # torch's (sum/4 in fp32).to(bf16) is the exactly rounded mean.
    g = torch.Generator().manual_seed(3)
    raw = (torch.randn(4096, 128, generator=g) / math.sqrt(128)).to(torch.bfloat16)
    r32 = raw.float().view(-1, 4, 128)
    s32 = ((r32[:, 0] + r32[:, 1]) + r32[:, 2]) + r32[:, 3]
    s64 = r32.double().sum(1)
    exact = (s32.double() == s64).all(dim=1).numpy()
    assert exact.mean() > 0.99
    want = (s32 / 4).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.pool_keys(raw.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(got[exact], want[exact])


def test_pool_empty_and_short_inputs():
    for t in range(4):
        assert O.pool_keys(np.zeros((t, 128), np.uint16)).shape == (0, 128)


def test_pool_constant_block_is_itself():
    rng = np.random.default_rng(5)
    row = to_bits(O.bf16_bits_to_f64(O.f64_to_bf16_bits(rng.standard_normal(128))))
    raw = np.tile(row, (8, 1))
    assert np.array_equal(O.pool_keys(raw), np.tile(row, (2, 1)))


# ----------------------------------------------------------------------------- visibility and budget

def test_dense_limit_is_2051():
    figs = read_page_figures()
    limit = int(figs["dense_limit_tokens"])
    for p in range(0, 4000):
        nb = O.visible_blocks(p)
        sel = O.select_blocks(np.zeros(nb))
        dense = len(sel) == nb
        assert dense == (p <= limit), p
    assert O.DENSE_LIMIT == limit
    # just past the limit: 513 blocks scored, 512 kept
    assert O.visible_blocks(2052) == 513 and len(O.select_blocks(np.zeros(513))) == 512


def test_budget_exact_beyond_limit():
    figs = read_page_figures()
    rng = np.random.default_rng(7)
    for p in list(range(2052, 2200)) + rng.integers(2052, 3_000_000, 200).tolist():
        nb = O.visible_blocks(p)
        sel = O.select_blocks(rng.standard_normal(nb))
        assert len(sel) * O.COMPRESS_RATIO == int(figs["selected_tokens"])
        toks = O.attended_tokens(p, sel)
        assert len(toks) == 2048 + (p % 4) + 1
        assert toks[-1] == p and len(np.unique(toks)) == len(toks)


def test_attended_tokens_membership_definition():
    # t in J  <=>  t <= p and (block(t) selected or t in the query's own block)
    rng = np.random.default_rng(11)
    for p in [0, 1, 3, 4, 5, 37, 2051, 2052, 5000]:
        nb = O.visible_blocks(p)
        sel = np.sort(rng.choice(nb, size=min(nb, 7), replace=False)) if nb else np.zeros(0, np.int64)
        want = [t for t in range(p + 1) if (t // 4) in set(sel.tolist()) or t // 4 >= nb]
        assert O.attended_tokens(p, sel).tolist() == want


# ----------------------------------------------------------------------------- scoring

def test_scores_exact_on_integers():
    rng = np.random.default_rng(13)
    q = rng.integers(-8, 9, 128)
    pk = rng.integers(-8, 9, (50, 128))
    got = O.score_blocks(to_bits(q), to_bits(pk))
    want = [sum(int(a) * int(b) for a, b in zip(q, row)) for row in pk]   # exact integer arithmetic
    assert got.tolist() == want


def test_scores_basis_vectors():
    eye = to_bits(np.eye(128))
    q = to_bits(np.arange(128) - 64.0)
    assert np.array_equal(O.score_blocks(q, eye), np.arange(128) - 64.0)


def _fp32_sums(prods):
    """float32 sums of each row of exact float32 products in three orders: sequential,
    reversed and pairwise (tree)."""
    out = []
    for order in (slice(None), slice(None, None, -1)):
        acc = np.zeros(prods.shape[0], np.float32)
        for d in range(prods.shape[1])[order]:
            acc = (acc + prods[:, d]).astype(np.float32)
        out.append(acc.astype(np.float64))
    pw = prods.copy()
    while pw.shape[1] > 1:
        pw = (pw[:, 0::2] + pw[:, 1::2]).astype(np.float32)
    out.append(pw[:, 0].astype(np.float64))
    return out


def test_score_error_bound_covers_fp32_evaluations():
    # random rows, rows with heavy cancellation and rows of mixed magnitudes: a float32
    # evaluation of q . p (exact bf16 x bf16 products, float32 additions) in each of three
    # orders stays within the bound of the exact score
    rng = np.random.default_rng(61)
    keys = rng.standard_normal((300, 128)).astype(np.float32) / 8
    keys[100:200] *= np.exp2(rng.integers(-20, 20, (100, 128))).astype(np.float32)
    q = rng.standard_normal(128).astype(np.float32)
    kb, qb_ = to_bits(torch.from_numpy(keys).bfloat16().float().numpy()), None
    qv = torch.from_numpy(q).bfloat16().float().numpy()
    keys_v = O.bf16_bits_to_f64(kb)
    # rows 200..299: p_d = +-q_d-ish so the sum nearly cancels
    sign = np.where(rng.random((100, 128)) < 0.5, -1.0, 1.0)
    keys_v[200:] = torch.from_numpy((sign * qv[None, :] * (1 + rng.random((100, 128)) / 64)).astype(np.float32)
                                    ).bfloat16().double().numpy()
    kb = to_bits(keys_v)
    qb_ = to_bits(qv)
    exact = O.score_blocks(qb_, kb)
    bound = O.score_error_bound(qb_, kb)
    prods = (keys_v.astype(np.float32) * qv[None, :]).astype(np.float32)
    assert np.array_equal(prods.astype(np.float64), keys_v * qv[None, :].astype(np.float64))   # exact
    worst = 0.0
    for got in _fp32_sums(prods):
        err = np.abs(got - exact)
        assert np.all(err <= bound)
        worst = max(worst, float(np.max(err / bound)))
    assert worst > 0.0


def test_score_error_bound_is_attained_by_sequential_fp32():
    # One product of 1 followed by 127 products just below half an ulp of 1: a sequential
    # float32 sum rounds every small term away, so its error is 127 x (255/256) 2^-24, within
    # 1.2 % of any bound of the form gamma_128 sum|q p|. The oracle's bound must cover it and
    # may not exceed it by more than 2 %: a bound inflated by a stray factor (u = 2^-23, a
    # wrong n) fails one side or the other.
    q = np.full(128, 2.0 ** -12)
    p = np.full(128, (1 + 127 / 128) * 2.0 ** -13)              # q p = (255/256) 2^-24
    q[0], p[0] = 1.0, 1.0
    qb_, pb = to_bits(q), to_bits(p[None, :])
    exact = O.score_blocks(qb_, pb)
    bound = O.score_error_bound(qb_, pb)
    prods = (p.astype(np.float32) * q.astype(np.float32))[None, :].astype(np.float32)
    seq, rev, tree = _fp32_sums(prods)
    assert seq[0] == 1.0                                          # every small term rounded away
    err = abs(seq[0] - exact[0])
    assert err == 127 * 255 * 2.0 ** -32
    assert err <= bound[0] <= 1.02 * err
    assert abs(rev[0] - exact[0]) <= bound[0] and abs(tree[0] - exact[0]) <= bound[0]
    # the same with a last product of -1: the float32 sum cancels to 0 while the exact score
    # is the 126 lost terms, so only a bound on sum |q p| (not |sum q p|) covers it
    q[127], p[127] = -1.0, 1.0
    qb_, pb = to_bits(q), to_bits(p[None, :])
    exact = O.score_blocks(qb_, pb)
    bound = O.score_error_bound(qb_, pb)
    prods = (p.astype(np.float32) * q.astype(np.float32))[None, :].astype(np.float32)
    seq = _fp32_sums(prods)[0]
    assert seq[0] == 0.0 and exact[0] == 126 * 255 * 2.0 ** -32
    assert abs(seq[0] - exact[0]) <= bound[0]


# ----------------------------------------------------------------------------- top-k

def _brute_force_topk(s, k):
    """The unique k-subset in which every member beats every non-member, where
    a beats b iff s[a] > s[b] or (s[a] == s[b] and a < b)."""
    n = len(s)
    beats = lambda a, b: s[a] > s[b] or (s[a] == s[b] and a < b)
    found = [c for c in itertools.combinations(range(n), k)
             if all(beats(a, b) for a in c for b in range(n) if b not in c)]
    assert len(found) == 1
    return list(found[0])


def test_topk_brute_force_tiny():
    rng = np.random.default_rng(17)
    for n in range(0, 10):
        for trial in range(6):
            s = rng.integers(-2, 3, n).astype(np.float64)          # many duplicates
            if trial == 0:
                s[:] = 1.0                                         # all equal
            for k in range(0, n + 2):
                got = O.select_blocks(s, k).tolist()
                assert got == _brute_force_topk(s, min(k, n)), (s, k)
                srt = sorted(range(n), key=lambda i: (-s[i], i))[: min(k, n)]
                assert got == sorted(srt)


def test_topk_nan_ranks_last_and_kth_score():
    s = np.array([0.5, np.nan, 2.0, 2.0, -1.0])
    assert O.select_blocks(s, 4).tolist() == [0, 2, 3, 4]
    assert O.kth_score(s, 3) == 0.5
    assert O.select_blocks(s, 9).tolist() == [0, 1, 2, 3, 4]


# ----------------------------------------------------------------------------- attention

def _sdpa(q, k, v, mask, n_kv_heads, scale):
    """torch SDPA in fp64 for one query: q [Hq, D], k/v [T, Hkv, D], mask [T] bool."""
    hq = q.shape[0]
    kk = torch.tensor(k).permute(1, 0, 2).repeat_interleave(hq // n_kv_heads, dim=0)   # [Hq, T, D]
    vv = torch.tensor(v).permute(1, 0, 2).repeat_interleave(hq // n_kv_heads, dim=0)
    qq = torch.tensor(q)[:, None, :]                                                  # [Hq, 1, D]
    m = torch.tensor(mask)[None, None, :].expand(hq, 1, -1)
    out = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=m, scale=scale)
    return out[:, 0, :].numpy()


def _rand_case(rng, p, hq, hkv, d, sharp=True):
    s = 1.0 if sharp else 1.0 / math.sqrt(d)
    q = rng.standard_normal((hq, d)) * s
    k = rng.standard_normal((p + 1, hkv, d)) * s
    v = rng.standard_normal((p + 1, hkv, d))
    return q, k, v


def test_dense_regime_equals_causal_sdpa():
    rng = np.random.default_rng(19)
    for p in [0, 1, 2, 3, 4, 9, 100, 2047, 2051]:
        q, k, v = _rand_case(rng, p, 4, 2, 16)
        scores = rng.standard_normal(O.visible_blocks(p))
        sel = O.select_blocks(scores)
        toks = O.attended_tokens(p, sel)
        assert toks.tolist() == list(range(p + 1))
        out, lse = O.attend(q, k, v, toks, 2, 1 / math.sqrt(16))
        ref = _sdpa(q, k, v, np.ones(p + 1, bool), 2, 1 / math.sqrt(16))
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_sparse_regime_equals_masked_sdpa_and_logsumexp():
    from scipy.special import logsumexp
    rng = np.random.default_rng(23)
    for p in [2052, 2055, 3001, 9000]:
        hq, hkv, d = 8, 2, 32
        q, k, v = _rand_case(rng, p, hq, hkv, d)
        sel = O.select_blocks(rng.standard_normal(O.visible_blocks(p)))
        toks = O.attended_tokens(p, sel)
        mask = np.zeros(p + 1, bool)
        mask[toks] = True
        out, lse = O.attend(q, k, v, toks, hkv, 0.125)
        np.testing.assert_allclose(out, _sdpa(q, k, v, mask, hkv, 0.125), rtol=1e-11, atol=1e-12)
        for h in range(hq):
            logits = (k[toks, h // (hq // hkv)] @ q[h]) * 0.125
            assert abs(lse[h] - logsumexp(logits)) < 1e-11


def test_attention_closed_forms():
    rng = np.random.default_rng(29)
    hq, hkv, d = 4, 2, 8
    # p = 0: only the query's own token -> out = V[0] exactly, lse = its logit
    q, k, v = _rand_case(rng, 0, hq, hkv, d)
    out, lse = O.attend(q, k, v, O.attended_tokens(0, []), hkv, 0.5)
    for h in range(hq):
        assert np.array_equal(out[h], v[0, h // 2])
        assert lse[h] == pytest.approx(0.5 * float(k[0, h // 2] @ q[h]), abs=1e-14)
    # constant V rows -> that row; equal keys -> mean of V over J
    p = 5000
    q, k, v = _rand_case(rng, p, hq, hkv, d)
    sel = O.select_blocks(rng.standard_normal(O.visible_blocks(p)))
    toks = O.attended_tokens(p, sel)
    vc = np.broadcast_to(v[0:1], v.shape).copy()
    out, _ = O.attend(q, k, vc, toks, hkv, 0.5)
    np.testing.assert_allclose(out, np.stack([v[0, h // 2] for h in range(hq)]), rtol=1e-13)
    ke = np.broadcast_to(k[0:1], k.shape).copy()
    out, lse = O.attend(q, ke, v, toks, hkv, 0.5)
    np.testing.assert_allclose(out, np.stack([v[toks, h // 2].mean(0) for h in range(hq)]), rtol=1e-12)
    for h in range(hq):
        assert lse[h] == pytest.approx(0.5 * float(k[0, h // 2] @ q[h]) + math.log(len(toks)), rel=1e-12)
    # one dominant key -> its V row
    kd = k.copy()
    t_star = toks[len(toks) // 3]
    kd[t_star] = 200.0 * q[[0, 2]]
    out, _ = O.attend(q[[0, 2]], kd, v, toks, hkv, 1.0)
    np.testing.assert_allclose(out, v[t_star], rtol=1e-9, atol=1e-9)


def test_lse_merge_of_any_partition_equals_unsplit():
    rng = np.random.default_rng(31)
    p = 4099
    hq, hkv, d = 8, 2, 16
    q, k, v = _rand_case(rng, p, hq, hkv, d)
    toks = O.attended_tokens(p, O.select_blocks(rng.standard_normal(O.visible_blocks(p))))
    want_out, want_lse = O.attend(q, k, v, toks, hkv, 0.25)
    for n_parts in [1, 2, 3, 7, 64]:
        perm = rng.permutation(toks)
        cuts = np.sort(rng.choice(np.arange(1, len(toks)), n_parts - 1, replace=False)) if n_parts > 1 else []
        parts = [O.attend_partial(q, k, v, piece, hkv, 0.25) for piece in np.split(perm, cuts)]
        parts.append(O.attend_partial(q, k, v, np.zeros(0, np.int64), hkv, 0.25))   # an empty split
        out, lse = O.lse_merge(parts)
        np.testing.assert_allclose(out, want_out, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse, want_lse, rtol=1e-12, atol=1e-12)


def test_interval_walk_equals_per_query_attention():
    rng = np.random.default_rng(37)
    p = 9000
    hq, hkv, d = 4, 2, 16
    q, k, v = _rand_case(rng, p, hq, hkv, d)
    sel = O.select_blocks(rng.standard_normal(O.visible_blocks(p)))
    want_out, want_lse = O.attend(q, k, v, O.attended_tokens(p, sel), hkv, 0.25)
    for interval in [1000, 4096, 8192, 16384]:
        out, lse = O.interval_walk_query(p, sel, q, k, v, hkv, interval, scale=0.25)
        np.testing.assert_allclose(out, want_out, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse, want_lse, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- golden files

def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = line.split("=", 1)
                vals[key.strip()] = ast.literal_eval(val.strip())
    return vals


def read_page_figures():
    vals = {}
    with open(os.path.join(GOLDEN, "page_figures.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = line.split()
                vals[key] = float(val)
    return vals


def _closed_form(expr):
    return eval(expr, {"__builtins__": {}}, {"e": math.e, "ln": math.log})


def test_tiny_worked_example():
    g = read_golden("tiny_worked_example.txt")
    raw = to_bits(g["raw_idx_k"])
    pooled = O.pool_keys(raw)
    assert O.bf16_bits_to_f64(pooled).tolist() == g["expect_pooled"]
    k = np.stack([g["k_kv0"], g["k_kv1"]], axis=1).astype(np.float64)   # [T, Hkv, D]
    v = np.stack([g["v_kv0"], g["v_kv1"]], axis=1).astype(np.float64)
    r = O.decode_query(g["p"], to_bits(g["q_idx"]), pooled, to_bits(g["q"]), to_bits(k), to_bits(v),
                       g["n_kv_heads"], scale=g["scale"], k_blocks=g["k_blocks"])
    assert r["scores"].tolist() == g["expect_scores"]
    assert r["sel"].tolist() == g["expect_sel"]
    assert r["tokens"].tolist() == g["expect_tokens"]
    want_out = np.array([[_closed_form(x) for x in row] for row in g["expect_out"]])
    want_lse = np.array([_closed_form(x) for x in g["expect_lse"]])
    np.testing.assert_allclose(r["out"], want_out, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(r["lse"], want_lse, rtol=1e-14)


# --------------------------------------------------------------------------- FP8 indexer keys

def _e4m3_table():
    """Every finite non-negative E4M3 value with its mantissa field, from the bit layout:
    exponent field e (bias 7) and mantissa m; e = 0 subnormal (m/8) 2^-6; e = 15, m = 7 NaN."""
    out = {}
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            v = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
            out[v] = m
    vals = sorted(out)
    return np.array(vals), np.array([out[v] for v in vals])


def test_e4m3_table_constants():
    vals, _ = _e4m3_table()
    assert vals.max() == O.E4M3_MAX == 448.0
    assert vals[1] == 2.0 ** -9                     # smallest subnormal
    assert 2.0 ** -6 in vals and vals.size == 127   # 126 non-zero values and zero


def test_e4m3_round_fixed_points_midpoints_and_saturation():
    vals, mant = _e4m3_table()
    for sign in (1.0, -1.0):
        np.testing.assert_array_equal(O.e4m3_round(sign * vals), sign * vals)
    mid = (vals[:-1] + vals[1:]) / 2                # ties: to the even mantissa
    want = np.where(mant[:-1] % 2 == 0, vals[:-1], vals[1:])
    np.testing.assert_array_equal(O.e4m3_round(mid), want)
    eps = np.minimum(np.diff(vals) / 8, 1.0)
    np.testing.assert_array_equal(O.e4m3_round(mid - eps), vals[:-1])
    np.testing.assert_array_equal(O.e4m3_round(mid + eps), vals[1:])
    np.testing.assert_array_equal(O.e4m3_round([449.0, 464.0, 1e9, -1e9]), [448.0, 448.0, 448.0, -448.0])


def test_e4m3_round_is_the_nearest_table_value():
    vals, mant = _e4m3_table()
    rng = np.random.default_rng(41)
    x = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(440.0), 5000)) * rng.choice([-1.0, 1.0], 5000)
    full = np.concatenate([-vals[::-1], vals[1:]])
    for xi, r in zip(x, O.e4m3_round(x)):
        d = np.abs(full - xi)
        assert r == full[np.argmin(d)] or np.isclose(d.min(), np.sort(d)[1])   # ties are pinned above


def test_quantize_pooled_fp8_cases():
    # the largest magnitude maps to 448, an all-zero key to scale 0, every value within half a
    # mantissa step (2^-4 relative) of the key where it is a normal E4M3 value
    rng = np.random.default_rng(43)
    keys = torch.from_numpy(rng.standard_normal((64, 128)).astype(np.float32) / 8).bfloat16().float().numpy()
    keys[5] = 0.0
    bits = to_bits(keys)
    vals, scales = O.quantize_pooled_fp8(bits)
    exact = O.bf16_bits_to_f64(bits)
    assert scales.dtype == np.float32 and scales[5] == 0 and not vals[5].any()
    rows = [r for r in range(64) if r != 5]
    np.testing.assert_array_equal(np.abs(vals[rows]).max(axis=1), 448.0)
    deq = vals[rows] * scales[rows, None].astype(np.float64)
    big = np.abs(exact[rows]) >= 2.0 ** -6 * scales[rows, None] * 1.01
    rel = np.abs(deq - exact[rows])[big] / np.abs(exact[rows])[big]
    assert rel.max() <= 2.0 ** -4 * (1 + 1e-6)


def test_score_blocks_fp8_one_hot_and_linearity():
    q = np.zeros(128, np.float32)
    q[7] = 3.0
    key = np.zeros((2, 128), np.float32)
    key[0, 7] = -0.5
    key[1, 7] = 2.0
    key[1, 9] = 1.0
    vals, scl = O.quantize_pooled_fp8(to_bits(key))
    s = O.score_blocks_fp8(to_bits(q), vals, scl)
    assert s[0] == 3.0 * -448.0 * float(np.float32(0.5) / np.float32(448.0))
    assert s[1] == 3.0 * 448.0 * float(np.float32(2.0) / np.float32(448.0))


def test_score_error_bound_fp8_covers_an_fp32_evaluation():
    # the bound must cover a float32 evaluation of the same score in any summation order:
    # sequential, pairwise and reversed sums of the exact products, then the scale product
    rng = np.random.default_rng(47)
    keys = torch.from_numpy(rng.standard_normal((200, 128)).astype(np.float32) / 8).bfloat16().float().numpy()
    q = torch.from_numpy(rng.standard_normal(128).astype(np.float32)).bfloat16().float().numpy()
    vals, scl = O.quantize_pooled_fp8(to_bits(keys))
    exact = O.score_blocks_fp8(to_bits(q), vals, scl)
    bound = O.score_error_bound_fp8(to_bits(q), vals, scl)
    prods = (vals.astype(np.float32) * q[None, :]).astype(np.float32)     # exact in float32
    assert np.array_equal(prods.astype(np.float64), vals * q[None, :].astype(np.float64))
    for order in (slice(None), slice(None, None, -1)):
        acc = np.zeros(200, np.float32)
        for d in range(128)[order]:
            acc = (acc + prods[:, d]).astype(np.float32)
        got = (acc * scl).astype(np.float32).astype(np.float64)
        assert np.all(np.abs(got - exact) <= bound)
    pw = prods.copy()
    while pw.shape[1] > 1:
        pw = (pw[:, 0::2] + pw[:, 1::2]).astype(np.float32)
    got = (pw[:, 0] * scl).astype(np.float32).astype(np.float64)
    assert np.all(np.abs(got - exact) <= bound)
    assert np.all(bound > 0) and np.all(bound <= 1e-5 * (np.abs(vals) @ np.abs(q)) * scl + 1e-30)


# --------------------------------------------------------------------------- sparse MLA (MQA form)

def _mla_case(n=40, h=8, seed=51):
    rng = np.random.default_rng(seed)
    lat = torch.from_numpy(rng.standard_normal((n, 512)).astype(np.float32) / 8).bfloat16().float().numpy()
    rope = torch.from_numpy(rng.standard_normal((n, 64)).astype(np.float32) / 8).bfloat16().float().numpy()
    q = torch.from_numpy(rng.standard_normal((h, 576)).astype(np.float32)).bfloat16().float().numpy()
    return to_bits(lat), to_bits(rope), to_bits(q)


def test_mla_row_quantisation_groups():
    # each 128-dim group has its own scale: scaling one group by 2^k scales only its scale by
    # 2^k (codes unchanged); every group's largest code is 448; rope passes through exactly
    lat, rope, _ = _mla_case(n=6)
    deq, rp, scl = O.quantize_mla_rows_fp8(lat, rope)
    assert deq.shape == (6, 512) and scl.shape == (6, 4)
    np.testing.assert_array_equal(rp, O.bf16_bits_to_f64(rope))
    lat2 = O.bf16_bits_to_f64(lat).copy()
    lat2[:, 128:256] *= 2.0 ** -5
    deq2, _, scl2 = O.quantize_mla_rows_fp8(to_bits(lat2), rope)
    np.testing.assert_array_equal(scl2[:, 1], scl[:, 1] * np.float32(2.0 ** -5))
    np.testing.assert_array_equal(deq2[:, 128:256], deq[:, 128:256] * 2.0 ** -5)
    np.testing.assert_array_equal(np.delete(deq2, np.s_[128:256], axis=1), np.delete(deq, np.s_[128:256], axis=1))
    codes = deq.reshape(6, 4, 128) / scl.astype(np.float64)[:, :, None]
    np.testing.assert_allclose(np.abs(codes).max(axis=2), 448.0, rtol=0, atol=0)
    exact = O.bf16_bits_to_f64(lat)
    rel = np.abs(deq - exact)[np.abs(exact) > 1e-3] / np.abs(exact)[np.abs(exact) > 1e-3]
    assert rel.max() <= 2.0 ** -4 * (1 + 1e-6)


def test_sparse_mla_attend_vs_sdpa():
    # every head attends the same selected rows (MQA); the value is the latent, the key adds
    # the rotary dims: torch's scaled_dot_product_attention in fp64 on the expanded heads
    lat, rope, qb_ = _mla_case(n=50, h=16)
    latent, rp, _ = O.quantize_mla_rows_fp8(lat, rope)
    rows = np.array([3, 7, 8, 20, 31, 32, 49])
    out, lse = O.sparse_mla_attend(qb_, latent, rp, rows)
    q = torch.from_numpy(O.bf16_bits_to_f64(qb_))[None, :, None, :]
    k = torch.from_numpy(np.concatenate([latent[rows], rp[rows]], axis=1))[None, None].expand(1, 16, -1, -1)
    v = torch.from_numpy(latent[rows])[None, None].expand(1, 16, -1, -1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=1.0 / 24.0)[0, :, 0].numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)
    logits = O.bf16_bits_to_f64(qb_) @ np.concatenate([latent[rows], rp[rows]], axis=1).T / 24.0
    from scipy.special import logsumexp
    np.testing.assert_allclose(lse, logsumexp(logits, axis=1), rtol=1e-13)


def test_sparse_mla_attend_closed_forms_and_merge():
    lat, rope, qb_ = _mla_case(n=30, h=4)
    latent, rp, _ = O.quantize_mla_rows_fp8(lat, rope)
    # one row: every head outputs that row's latent
    out, lse = O.sparse_mla_attend(qb_, latent, rp, [11])
    np.testing.assert_array_equal(out, np.repeat(latent[11][None], 4, axis=0))
    # no rows
    out0, lse0 = O.sparse_mla_attend(qb_, latent, rp, [])
    assert not out0.any() and np.all(np.isneginf(lse0))
    # log-sum-exp merge of two disjoint halves equals the whole
    rows = np.arange(30)
    o1, l1 = O.sparse_mla_attend(qb_, latent, rp, rows[:13])
    o2, l2 = O.sparse_mla_attend(qb_, latent, rp, rows[13:])
    ow, lw = O.sparse_mla_attend(qb_, latent, rp, rows)
    lm = np.logaddexp(l1, l2)
    np.testing.assert_allclose(lm, lw, rtol=1e-14)
    np.testing.assert_allclose(np.exp(l1 - lm)[:, None] * o1 + np.exp(l2 - lm)[:, None] * o2, ow, rtol=1e-12,
                               atol=1e-15)


def test_mla_row_bytes_decode_by_hand():
    # one 656-byte row built by hand: codes 0x38 (1.0), 0x01 (2^-9), 0xFE (-448), 0x00, 0x80
    # (zero), the four group scales 0.5, 2, 0.25, 8, and rope = bf16 1.5 and -3 alternating
    row = np.zeros(656, np.uint8)
    row[0], row[1], row[2], row[3], row[4] = 0x38, 0x01, 0xFE, 0x00, 0x80
    row[128], row[300], row[511] = 0x38, 0x39, 0x40       # 1.0 in group 1, 1.125 in group 2, 2.0 in group 3
    row[512:528] = np.array([0.5, 2.0, 0.25, 8.0], dtype="<f4").view(np.uint8)
    rope = np.array([1.5, -3.0] * 32, dtype=np.float32)
    row[528:] = to_bits(rope).astype("<u2").view(np.uint8)
    lat, rp = O.mla_rows_from_bytes(row[None])
    assert O.MLA_ROW_BYTES == 656 and lat.shape == (1, 512) and rp.shape == (1, 64)
    assert lat[0, 0] == 0.5 and lat[0, 1] == 2.0 ** -10 and lat[0, 2] == -224.0 and lat[0, 3] == 0.0
    assert lat[0, 4] == 0.0 and lat[0, 128] == 2.0 and lat[0, 300] == 1.125 * 0.25 and lat[0, 511] == 16.0
    assert np.count_nonzero(lat) == 6
    np.testing.assert_array_equal(rp[0], rope)
    assert np.isnan(O.e4m3_value(0x7F)) and np.isnan(O.e4m3_value(0xFF))
    vals, _ = _e4m3_table()
    np.testing.assert_array_equal(np.sort(O.e4m3_value(np.arange(0x7F))), vals)      # every finite code


# --------------------------------------------------------------------------- FP8 K/V rows

def test_e4m3_code_by_hand_and_round_trip():
    # codes from the bit layout (sign | exponent field, bias 7 | 3 mantissa bits)
    vals = [1.0, 448.0, -448.0, 2.0 ** -9, 0.0, -0.0, 1.125, 0.5, 2.0 ** -6, 3.5, -0.875 * 2.0 ** -6, 240.0]
    want = [0x38, 0x7E, 0xFE, 0x01, 0x00, 0x80, 0x39, 0x30, 0x08, 0x46, 0x87, 0x77]
    np.testing.assert_array_equal(O.e4m3_code(vals), want)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    np.testing.assert_array_equal(O.e4m3_code(O.e4m3_value(finite)), finite)
    for bad in (1.0625, 449.0, 2.0 ** -10, float("nan"), float("inf")):
        with pytest.raises(ValueError):
            O.e4m3_code([bad])


def _kv_case(t=9, hkv=2, seed=61):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.standard_normal((t, hkv, 256)).astype(np.float32)).bfloat16().float().numpy()
    x[2, hkv - 1] = 0.0                # an all-zero row: both groups scale 0
    x[1, 0, 128:] = 0.0                # one zero group beside a live one
    x[0, hkv - 1, :128] *= 2.0 ** -20  # a group whose quotients are all tiny before scaling
    return x, to_bits(x)


def test_quantize_kv_fp8_scales_are_group_maxima():
    x, bits = _kv_case()
    codes, scales = O.quantize_kv_fp8(bits)
    assert codes.dtype == np.uint8 and codes.shape == (9, 2, 256)
    assert scales.dtype == np.float32 and scales.shape == (9, 2, 2)
    g = x.reshape(9, 2, 2, 128)
    want = (np.abs(g).max(axis=3).astype(np.float32) / np.float32(448.0)).astype(np.float32)
    np.testing.assert_array_equal(scales, want)
    assert scales[2, 1, 0] == scales[2, 1, 1] == 0 and not codes[2, 1].any()
    assert scales[1, 0, 1] == 0 and not codes[1, 0, 128:].any() and scales[1, 0, 0] > 0
    # the largest magnitude of every live group is coded as +-448
    live = scales > 0
    mags = np.abs(O.e4m3_value(codes)).reshape(9, 2, 2, 128).max(axis=3)
    np.testing.assert_array_equal(mags[live], 448.0)


def test_quantize_kv_fp8_codes_are_nearest_table_values():
    # brute force: each code is the table value nearest to the fp32 quotient x / scale
    x, bits = _kv_case(t=3, hkv=1, seed=62)
    codes, scales = O.quantize_kv_fp8(bits)
    vals, _ = _e4m3_table()
    full = np.concatenate([-vals[::-1], vals[1:]])
    g = x.reshape(-1, 128)
    s = scales.reshape(-1)
    got = O.e4m3_value(codes).reshape(-1, 128)
    assert (s == 0).sum() == 3 and not got[s == 0].any()      # token 2 (both groups), token 1 group 1
    for r in np.flatnonzero(s > 0):
        quot = (g[r].astype(np.float32) / s[r]).astype(np.float64)
        for qv, gv in zip(quot, got[r]):
            d = np.abs(full - qv)
            assert gv == full[np.argmin(d)] or np.isclose(d.min(), np.sort(d)[1])


def test_quantize_kv_fp8_groups_are_independent():
    # the groups are dims [0, 128) and [128, 256) of each (token, head) row: scaling one group
    # by 2^-5 scales only its scale, codes unchanged
    x, bits = _kv_case(seed=63)
    codes, scales = O.quantize_kv_fp8(bits)
    y = x.copy()
    y[:, 1, 128:] *= 2.0 ** -5
    codes2, scales2 = O.quantize_kv_fp8(to_bits(y))
    np.testing.assert_array_equal(codes2, codes)
    np.testing.assert_array_equal(scales2[:, 1, 1], scales[:, 1, 1] * np.float32(2.0 ** -5))
    np.testing.assert_array_equal(np.delete(scales2.reshape(9, 4), 3, axis=1), np.delete(scales.reshape(9, 4), 3, axis=1))


def test_dequantize_kv_fp8_by_hand_and_error_bound():
    codes = np.zeros((1, 2, 256), np.uint8)
    codes[0, 0, 0], codes[0, 0, 127], codes[0, 0, 128], codes[0, 1, 255] = 0x38, 0xFE, 0x39, 0x01
    scales = np.array([[[0.5, 4.0], [1.0, 2.0]]], np.float32)
    v = O.dequantize_kv_fp8(codes, scales)
    assert v[0, 0, 0] == 0.5 and v[0, 0, 127] == -224.0 and v[0, 0, 128] == 4.5 and v[0, 1, 255] == 2.0 ** -8
    assert np.count_nonzero(v) == 4
    # half a mantissa step: |deq - x| <= 2^-4 |x| where x / scale is a normal E4M3 value, and
    # the bound is nearly reached somewhere
    x, bits = _kv_case(seed=64)
    c, s = O.quantize_kv_fp8(bits)
    deq = O.dequantize_kv_fp8(c, s)
    sc = np.repeat(s.astype(np.float64), 128, axis=-1)
    big = (np.abs(x) >= 2.0 ** -6 * sc * 1.01) & (x != 0)
    rel = np.abs(deq - x)[big] / np.abs(x)[big]
    assert rel.max() <= 2.0 ** -4 * (1 + 1e-6) and rel.max() > 2.0 ** -4 * 0.9


def test_fp8_kv_rows_rounded_to_bf16_for_the_prefill():
    # the FP8 K/V prefill computes on code x scale rounded once to bf16 (its parity tests compose
    # dequantize_kv_fp8 with f64_to_bf16_bits). With scale 1 (or any power of two) every E4M3
    # value, at most 4 significant bits, is a bf16 value: the rounding is the identity
    rng = np.random.default_rng(66)
    codes = rng.integers(0, 256, (64, 256)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x00
    for sc in (1.0, 2.0 ** -20, 2.0 ** 30):
        x = O.dequantize_kv_fp8(codes, np.full((64, 2), sc, np.float32))
        assert np.array_equal(O.bf16_bits_to_f64(O.f64_to_bf16_bits(x)), x)
    # other scales: half a bf16 step at most, 2^-8 of the magnitude, reached within a few percent
    scales = (2.0 ** rng.uniform(-20, 20, (64, 2))).astype(np.float32)
    x = O.dequantize_kv_fp8(codes, scales)
    r = O.bf16_bits_to_f64(O.f64_to_bf16_bits(x))
    nz = x != 0
    rel = np.abs(r - x)[nz] / np.abs(x)[nz]
    assert rel.max() <= 2.0 ** -8 and rel.max() > 2.0 ** -8 * 0.9
    assert np.array_equal(r == 0, x == 0)


def test_decode_query_on_fp8_kv_closed_forms():
    # identical K rows: every attended token gets the same weight, so each head outputs the mean
    # of the dequantised V rows of its KV head over the attended tokens, and lse = logit + ln n
    rng = np.random.default_rng(65)
    p, hkv, hq = 30, 2, 8
    krow = torch.from_numpy(rng.standard_normal((hkv, 256)).astype(np.float32)).bfloat16().float().numpy()
    k = np.broadcast_to(krow, (p + 1, hkv, 256)).copy()
    vv = torch.from_numpy(rng.standard_normal((p + 1, hkv, 256)).astype(np.float32)).bfloat16().float().numpy()
    kc, ks = O.quantize_kv_fp8(to_bits(k))
    vc, vs = O.quantize_kv_fp8(to_bits(vv))
    kd, vd = O.dequantize_kv_fp8(kc, ks), O.dequantize_kv_fp8(vc, vs)
    q = to_bits(torch.from_numpy(rng.standard_normal((hq, 256)).astype(np.float32)).bfloat16().float().numpy())
    raw = to_bits(torch.from_numpy(rng.standard_normal((p + 1, 128)).astype(np.float32)).bfloat16().float().numpy())
    qi = to_bits(torch.from_numpy(rng.standard_normal(128).astype(np.float32)).bfloat16().float().numpy())
    r = O.decode_query(p, qi, O.pool_keys(raw), q, kd, vd, hkv)
    n = r["tokens"].size
    assert n == p + 1                                # dense: every token up to p
    qf = O.bf16_bits_to_f64(q)
    for h in range(hq):
        kv = h // (hq // hkv)
        np.testing.assert_allclose(r["out"][h], vd[r["tokens"], kv].mean(axis=0), rtol=1e-12, atol=1e-14)
        logit = (kd[0, kv] @ qf[h]) / 16.0
        np.testing.assert_allclose(r["lse"][h], logit + np.log(n), rtol=1e-12)
