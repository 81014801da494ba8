"""Pins of the CPU oracle to facts other than its own formulas (CPU only).

Each pin is chosen so that a plausible slip in the oracle -- a dropped rank,
a wrong shard order, a transposed operand, a wrong owner chunk, an unstable
permutation, a missing gate weight -- fails at least one test here.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle
from workloads import gen


# ---------------------------------------------------------------- formats
def test_widen_known_f16_values():
    bits = np.array([0x3C00, 0xC000, 0x7BFF, 0x0001, 0x3555, 0x0000, 0x8000], dtype=np.uint16)
    want = [1.0, -2.0, 65504.0, 2.0 ** -24, 0.333251953125, 0.0, -0.0]
    got = oracle.widen(bits.view(np.float16), "f16")
    assert got.tolist() == want


def test_widen_known_bf16_values():
    bits = np.array([0x3F80, 0xC000, 0x4049, 0x3E80, 0x0000, 0x7F7F], dtype=np.uint16)
    want = [1.0, -2.0, 3.140625, 0.25, 0.0, 3.3895313892515355e38]
    got = oracle.widen(bits, "bf16")
    assert got.tolist() == want


def test_round_to_bf16_ties_and_random():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1.0);
    # 1 + 3 * 2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6 -> even (1 + 2^-6).
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 1 + 2 ** -8 + 2 ** -20])
    assert oracle.round_to(x, "bf16").tolist() == [1.0, 1 + 2 ** -6, -1.0, 1 + 2 ** -7]
    # independent integer bit-twiddling rounding of the input generator agrees
    r = np.random.default_rng(7).standard_normal(20000).astype(np.float32) * 3
    via_bits = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(r)).astype(np.float64)
    assert np.array_equal(oracle.round_to(r.astype(np.float64), "bf16"), via_bits)


def test_round_to_f16_ties():
    # 1 + 2^-11 is halfway between 1 and 1 + 2^-10 -> 1.0 (even)
    x = np.array([1 + 2 ** -11, 1 + 3 * 2 ** -11, 2049.0, 2051.0])
    assert oracle.round_to(x, "f16").tolist() == [1.0, 1 + 2 ** -9, 2048.0, 2052.0]


# ---------------------------------------------------------------- GEMM
def _brute_gemm(A, B):
    """Exact rational triple loop."""
    M, K = len(A), len(A[0])
    N = len(B[0])
    return [[sum(Fraction(A[i][k]) * Fraction(B[k][j]) for k in range(K)) for j in range(N)]
            for i in range(M)]


def test_gemm_hand_worked_example():
    A = np.array([[1.0, 2.0], [3.0, 4.0]])
    B = np.array([[5.0, 6.0], [7.0, 8.0]])
    assert oracle.gemm(A, B).tolist() == [[19.0, 22.0], [43.0, 50.0]]


def test_gemm_brute_force_exact_on_random_fp16():
    rng = np.random.default_rng(1)
    A = rng.standard_normal((5, 7)).astype(np.float16)
    B = rng.standard_normal((7, 3)).astype(np.float16)
    got = oracle.gemm(oracle.widen(A, "f16"), oracle.widen(B, "f16"))
    want = _brute_gemm(A.astype(np.float64).tolist(), B.astype(np.float64).tolist())
    for i, j in itertools.product(range(5), range(3)):
        # float64 error bound of a 7-term dot product of fp16 values
        assert abs(Fraction(got[i, j]) - want[i][j]) <= Fraction(1, 2 ** 40)


def test_gemm_closed_form_ones():
    M, K, N = 3, 9, 4
    A = np.ones((M, K))
    B = np.array([[k + 1 + j for j in range(N)] for k in range(K)], dtype=np.float64)
    C = oracle.gemm(A, B)
    for j in range(N):
        assert C[0, j] == K * (K + 1) / 2 + j * K


def test_gemm_associativity_and_transpose():
    rng = np.random.default_rng(2)
    A, B, v = rng.standard_normal((6, 5)), rng.standard_normal((5, 4)), rng.standard_normal(4)
    C = oracle.gemm(A, B)
    assert np.allclose(C @ v, A @ (B @ v), rtol=1e-13, atol=1e-13)
    assert np.allclose(oracle.gemm(B.T, A.T), C.T, rtol=1e-13, atol=1e-13)
    with pytest.raises(ValueError):
        oracle.gemm(A, A)


# ---------------------------------------------------------------- AG-GEMM
def _shards_int(seed, R, rows, cols, dtype="f16"):
    return [gen.integers16((seed, r), (rows, cols), -2, 2, dtype) for r in range(R)]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_ag_gemm_brute_force(dtype):
    R, mloc, K, nloc = 3, 2, 5, 2
    xs = _shards_int(11, R, mloc, K, dtype)
    ws = _shards_int(12, R, K, nloc, dtype)
    out = oracle.ag_gemm(xs, ws, dtype)
    for r in range(R):
        for i in range(R * mloc):
            s, li = divmod(i, mloc)
            for j in range(nloc):
                want = sum(float(oracle.widen(xs[s], dtype)[li, k]) *
                           float(oracle.widen(ws[r], dtype)[k, j]) for k in range(K))
                assert out[r][i, j] == want


def test_ag_gemm_identity_weights_return_gathered_x():
    R, mloc, K = 4, 3, 8
    xs = [gen.normal16((5, r), (mloc, K), 1.0, "f16") for r in range(R)]
    ws = [np.zeros((K, K // R * R), np.float16) for _ in range(R)]
    # W1_r = columns [r K/R, (r+1) K/R) of I_K, so Out_r = X[:, those columns]
    eye = np.eye(K, dtype=np.float16)
    ws = [np.ascontiguousarray(eye[:, r * (K // R):(r + 1) * (K // R)]) for r in range(R)]
    out = oracle.ag_gemm(xs, ws, "f16")
    X = np.concatenate([x.astype(np.float64) for x in xs])
    for r in range(R):
        assert np.array_equal(out[r], X[:, r * (K // R):(r + 1) * (K // R)])


def test_ag_gemm_r1_is_plain_gemm_and_shard_order_matters():
    x = gen.normal16(1, (6, 5), 1.0, "f16")
    w = gen.normal16(2, (5, 4), 1.0, "f16")
    assert np.array_equal(oracle.ag_gemm([x], [w], "f16")[0],
                          x.astype(np.float64) @ w.astype(np.float64))
    xs = [gen.normal16((3, r), (2, 5), 1.0, "f16") for r in range(3)]
    a = oracle.ag_gemm(xs, [w] * 3, "f16")[0]
    b = oracle.ag_gemm(xs[::-1], [w] * 3, "f16")[0]
    # reversing the rank order reverses the row blocks of the gathered product
    assert np.array_equal(a[0:2], b[4:6]) and np.array_equal(a[4:6], b[0:2])


def test_ag_gemm_at_matches_full():
    R = 2
    xs = [gen.normal16((8, r), (4, 16), 1.0, "bf16") for r in range(R)]
    ws = [gen.normal16((9, r), (16, 6), 0.02, "bf16") for r in range(R)]
    full = oracle.ag_gemm(xs, ws, "bf16")
    # repeated rows and columns included (the helper widens each one once)
    rows, cols = np.array([0, 7, 3, 7, 0]), np.array([5, 0, 2, 2, 5])
    assert np.allclose(oracle.ag_gemm_at(xs, ws, "bf16", 1, rows, cols),
                       full[1][rows, cols], rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- GEMM-RS
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_gemm_rs_concat_equals_unsplit_gemm(dtype):
    R, M, kloc, N = 4, 8, 3, 5
    As = [gen.normal16((21, r), (M, kloc), 1.0, dtype) for r in range(R)]
    Bs = [gen.normal16((22, r), (kloc, N), 1.0, dtype) for r in range(R)]
    out = oracle.gemm_rs(As, Bs, dtype)
    A = np.concatenate([oracle.widen(a, dtype) for a in As], axis=1)
    B = np.concatenate([oracle.widen(b, dtype) for b in Bs], axis=0)
    full = A @ B
    assert np.allclose(np.concatenate(out), full, rtol=1e-13, atol=1e-13)
    assert [o.shape for o in out] == [(M // R, N)] * R


def test_gemm_rs_brute_force_exact_integers():
    R, M, kloc, N = 2, 4, 3, 2
    As = _shards_int(31, R, M, kloc)
    Bs = _shards_int(32, R, kloc, N)
    out = oracle.gemm_rs(As, Bs, "f16")
    for o in range(R):
        for li in range(M // R):
            i = o * (M // R) + li
            for j in range(N):
                want = sum(int(As[r][i, k]) * int(Bs[r][k, j]) for r in range(R) for k in range(kloc))
                assert out[o][li, j] == want


def test_gemm_rs_identity_blocks_sum_the_shards():
    R, M, N = 3, 6, 4
    As = [gen.normal16((41, r), (M, N), 1.0, "f16") for r in range(R)]
    Bs = [np.eye(N, dtype=np.float16) for _ in range(R)]
    out = oracle.gemm_rs(As, Bs, "f16")
    S = sum(a.astype(np.float64) for a in As)
    for o in range(R):
        assert np.array_equal(out[o], S[o * 2:(o + 1) * 2])


def test_gemm_rs_r1_and_owner_chunks():
    a = gen.normal16(1, (4, 6), 1.0, "f16")
    b = gen.normal16(2, (6, 3), 1.0, "f16")
    assert np.array_equal(oracle.gemm_rs([a], [b], "f16")[0],
                          a.astype(np.float64) @ b.astype(np.float64))
    # rank o must receive rows [o M/R, (o+1) M/R): a one-hot row in A lands in its owner
    R, M, kloc, N = 4, 8, 2, 3
    As = [np.zeros((M, kloc), np.float16) for _ in range(R)]
    As[2][5, 0] = 1.0
    Bs = [np.ones((kloc, N), np.float16) for _ in range(R)]
    out = oracle.gemm_rs(As, Bs, "f16")
    nz = [o for o in range(R) if np.any(out[o])]
    assert nz == [2] and np.array_equal(np.nonzero(out[2])[0], np.array([1, 1, 1]))


def test_gemm_rs_at_matches_full():
    R = 2
    As = [gen.normal16((51, r), (6, 8), 1.0, "f16") for r in range(R)]
    Bs = [gen.normal16((52, r), (8, 5), 0.02, "f16") for r in range(R)]
    full = oracle.gemm_rs(As, Bs, "f16")
    rows, cols = np.array([0, 2, 1, 2, 0]), np.array([4, 0, 3, 3, 4])  # with repeats
    assert np.allclose(oracle.gemm_rs_at(As, Bs, "f16", 1, rows, cols),
                       full[1][rows, cols], rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- routing
@pytest.mark.parametrize("T,E,topk,seed", [(64, 8, 2, 1), (33, 5, 3, 2), (10, 1, 1, 3), (128, 16, 4, 4)])
def test_moe_route_matches_library_sort(T, E, topk, seed):
    ids, _ = gen.routing(seed, T, E, topk)
    counts, offsets, s2r, r2s = oracle.moe_route(ids, E)
    flat = ids.reshape(-1)
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    assert np.array_equal(r2s, np.argsort(flat, kind="stable"))
    assert np.array_equal(s2r[r2s], np.arange(T * topk))
    # grouped order: expert ids along the rows are non-decreasing, slots ascending within one expert
    e_rows = flat[r2s]
    assert np.all(np.diff(e_rows) >= 0)
    for e in range(E):
        seg = r2s[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)


def test_moe_route_hand_example_and_empty_expert():
    ids = np.array([[2, 0], [0, 2], [2, 3]], dtype=np.int32)  # slots 0..5 -> experts 2,0,0,2,2,3
    counts, offsets, s2r, r2s = oracle.moe_route(ids, 5)
    assert counts.tolist() == [2, 0, 3, 1, 0]
    assert offsets.tolist() == [0, 2, 2, 5, 6, 6]
    assert r2s.tolist() == [1, 2, 0, 3, 4, 5]
    assert s2r.tolist() == [2, 0, 1, 3, 4, 5]
    with pytest.raises(ValueError):
        oracle.moe_route(np.array([[7]], dtype=np.int32), 4)


# ---------------------------------------------------------------- MoE layers
def _moe_small(R=2, T=8, H=6, F=4, E=3, topk=2, seed=3, dtype="f16", dist="normal"):
    from workloads import configs
    c = configs.MoE("t", R=R, T=T, H=H, F=F, E=E, topk=topk, dtype=dtype, seed=seed, dist=dist)
    return c, configs.moe_inputs(c)


def test_moe_layer0_single_expert_top1_is_ag_gemm():
    c, d = _moe_small(E=1, topk=1)
    ids = np.zeros((c.T, 1), np.int32)
    h, _ = oracle.moe_layer0(d["x_shards"], d["w1_shards"], ids, 1, "f16")
    ag = oracle.ag_gemm(d["x_shards"], [w[0] for w in d["w1_shards"]], "f16")
    for r in range(c.R):
        assert np.array_equal(h[r], ag[r])


def test_moe_layer0_brute_force_integers():
    c, d = _moe_small(dist="int")
    ids = d["topk_ids"]
    h, (counts, offsets, s2r, r2s) = oracle.moe_layer0(d["x_shards"], d["w1_shards"], ids, c.E, "f16")
    X = np.concatenate(d["x_shards"]).astype(np.int64)
    for r in range(c.R):
        W = d["w1_shards"][r].astype(np.int64)
        for t in range(c.T):
            for k in range(c.topk):
                row = s2r[t * c.topk + k]
                e = ids[t, k]
                want = [sum(int(X[t, i]) * int(W[e, i, j]) for i in range(c.H)) for j in range(W.shape[2])]
                assert h[r][row].tolist() == want


def test_moe_layer0_identical_experts_give_dense_rows():
    c, d = _moe_small(E=4)
    w1 = [np.stack([w[0]] * c.E) for w in d["w1_shards"]]
    h, (_, _, s2r, _) = oracle.moe_layer0(d["x_shards"], w1, d["topk_ids"], c.E, "f16")
    dense = oracle.ag_gemm(d["x_shards"], [w[0] for w in w1], "f16")
    for r in range(c.R):
        for s in range(c.T * c.topk):
            assert np.array_equal(h[r][s2r[s]], dense[r][s // c.topk])


def test_moe_layer1_single_expert_top1_unit_gate_is_gemm_rs():
    c, d = _moe_small(E=1, topk=1, T=8)
    ids = np.zeros((c.T, 1), np.int32)
    g = np.ones((c.T, 1), np.float32)
    out = oracle.moe_layer1(d["h_shards"], d["w2_shards"], ids, g, 1, "f16")
    rs = oracle.gemm_rs(d["h_shards"], [w[0] for w in d["w2_shards"]], "f16")
    for o in range(c.R):
        assert np.allclose(out[o], rs[o], rtol=1e-13, atol=1e-13)


def test_moe_layer1_brute_force_with_gates():
    c, d = _moe_small(dist="int", T=6, R=2, E=3, topk=2)
    ids, g = d["topk_ids"], d["topk_weights"]
    out = oracle.moe_layer1(d["h_shards"], d["w2_shards"], ids, g, c.E, "f16")
    _, _, s2r, _ = oracle.moe_route(ids, c.E)
    for t in range(c.T):
        o, lt = divmod(t, c.T // c.R)
        for j in range(c.H):
            acc = Fraction(0)
            for r in range(c.R):
                for k in range(c.topk):
                    hrow = d["h_shards"][r][s2r[t * c.topk + k]].astype(np.int64)
                    w = d["w2_shards"][r][ids[t, k]].astype(np.int64)
                    dot = sum(int(hrow[i]) * int(w[i, j]) for i in range(hrow.shape[0]))
                    acc += Fraction(float(g[t, k])) * dot
            assert abs(Fraction(out[o][lt, j]) - acc) <= Fraction(1, 2 ** 30)


def test_moe_layer1_identical_experts_gates_sum_to_one_give_dense():
    c, d = _moe_small(E=3, topk=2)
    ids, g = d["topk_ids"], d["topk_weights"]
    w2 = [np.stack([w[0]] * c.E) for w in d["w2_shards"]]
    # H rows of both slots of one token are set equal, so the gate-weighted sum equals one row
    _, _, s2r, _ = oracle.moe_route(ids, c.E)
    hs = []
    for r in range(c.R):
        h = np.array(d["h_shards"][r])
        for t in range(c.T):
            for k in range(1, c.topk):
                h[s2r[t * c.topk + k]] = h[s2r[t * c.topk]]
        hs.append(h)
    out = oracle.moe_layer1(hs, w2, ids, g, c.E, "f16")
    dense_in = [np.stack([hs[r][s2r[t * c.topk]] for t in range(c.T)]) for r in range(c.R)]
    dense = oracle.gemm_rs(dense_in, [w[0] for w in w2], "f16")
    gsum = g.astype(np.float64).sum(axis=1)
    for o in range(c.R):
        lo = o * (c.T // c.R)
        scale = gsum[lo:lo + c.T // c.R, None]
        assert np.allclose(out[o], dense[o] * scale, rtol=1e-12, atol=1e-12)
    assert np.allclose(gsum, 1.0, atol=1e-6)


def test_moe_token_permutation_permutes_outputs():
    c, d = _moe_small(T=8, R=1)
    perm = np.random.default_rng(0).permutation(c.T)
    X = d["x_shards"][0]
    h0, _ = oracle.moe_layer0([X], d["w1_shards"], d["topk_ids"], c.E, "f16")
    y0 = oracle.moe_layer1(h0, d["w2_shards"], d["topk_ids"], d["topk_weights"], c.E, "f16",
                           h_dtype="f64")[0]
    h1, _ = oracle.moe_layer0([X[perm]], d["w1_shards"], d["topk_ids"][perm], c.E, "f16")
    y1 = oracle.moe_layer1(h1, d["w2_shards"], d["topk_ids"][perm], d["topk_weights"][perm],
                           c.E, "f16", h_dtype="f64")[0]
    assert np.allclose(y1, y0[perm], rtol=1e-12, atol=1e-12)


def test_moe_rows_helpers_match_full():
    c, d = _moe_small(T=8, R=2, E=3, topk=2)
    h, _ = oracle.moe_layer0(d["x_shards"], d["w1_shards"], d["topk_ids"], c.E, "f16")
    rows = np.array([0, 5, 15])
    assert np.allclose(oracle.moe_layer0_rows(d["x_shards"], d["w1_shards"], d["topk_ids"], c.E,
                                              "f16", 1, rows), h[1][rows], rtol=1e-14, atol=1e-15)
    y = oracle.moe_layer1(d["h_shards"], d["w2_shards"], d["topk_ids"], d["topk_weights"], c.E, "f16")
    lr = np.array([0, 3, 1, 2, 3])  # every owner row, one twice
    assert np.allclose(oracle.moe_layer1_rows(d["h_shards"], d["w2_shards"], d["topk_ids"],
                                              d["topk_weights"], c.E, "f16", 1, lr),
                       y[1][lr], rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- expert-parallel MoE
def _ep_weights(c, seed=11, dist="normal"):
    """Full expert weights W1 [E, H, F], W2 [E, F, H] and their TP and EP shards."""
    if dist == "int":
        W1 = gen.integers16((seed, 1), (c.E, c.H, c.F), -2, 2, "f16")
        W2 = gen.integers16((seed, 2), (c.E, c.F, c.H), -2, 2, "f16")
    else:
        W1 = gen.normal16((seed, 1), (c.E, c.H, c.F), 0.5, "f16")
        W2 = gen.normal16((seed, 2), (c.E, c.F, c.H), 0.5, "f16")
    fr, el = c.F // c.R, c.E // c.R
    w1_tp = [np.ascontiguousarray(W1[:, :, r * fr:(r + 1) * fr]) for r in range(c.R)]
    w2_tp = [np.ascontiguousarray(W2[:, r * fr:(r + 1) * fr, :]) for r in range(c.R)]
    w1_ep = [np.ascontiguousarray(W1[r * el:(r + 1) * el]) for r in range(c.R)]
    w2_ep = [np.ascontiguousarray(W2[r * el:(r + 1) * el]) for r in range(c.R)]
    return W1, W2, w1_tp, w2_tp, w1_ep, w2_ep


def _eptp_shards(W1, W2, R, tp):
    """Rank r = g tp + t: experts of EP group g, column (W1) / row (W2) block t."""
    E, _, F = W1.shape
    el, fb = E // (R // tp), F // tp
    w1 = [np.ascontiguousarray(W1[(r // tp) * el:(r // tp + 1) * el, :, (r % tp) * fb:(r % tp + 1) * fb])
          for r in range(R)]
    w2 = [np.ascontiguousarray(W2[(r // tp) * el:(r // tp + 1) * el, (r % tp) * fb:(r % tp + 1) * fb, :])
          for r in range(R)]
    return w1, w2


def test_moe_eptp_layer0_does_not_depend_on_the_split():
    # every EP x TP split of the same experts computes the same rows, and tp = R
    # is the tensor-parallel layer0 exactly
    c, d = _moe_small(R=4, T=8, H=6, F=8, E=4, topk=2)
    W1, W2, w1_tp, _, _, _ = _ep_weights(c)
    h_tp, _ = oracle.moe_layer0(d["x_shards"], w1_tp, d["topk_ids"], c.E, "f16")
    for tp in (1, 2, 4):
        w1, _ = _eptp_shards(W1, W2, c.R, tp)
        h, _ = oracle.moe_ep_layer0(d["x_shards"], w1, d["topk_ids"], c.E, "f16", tp=tp)
        assert np.array_equal(h, np.concatenate(h_tp, axis=1)), tp


@pytest.mark.parametrize("tp", [1, 2, 4])
def test_moe_eptp_chain_brute_force_integers(tp):
    # exact rationals per token and slot, for every EP x TP split of R = 4
    c, d = _moe_small(R=4, T=8, H=3, F=8, E=4, topk=2, dist="int")
    W1, W2, _, _, _, _ = _ep_weights(c, dist="int")
    w1, w2 = _eptp_shards(W1, W2, c.R, tp)
    ids, g = d["topk_ids"], d["topk_weights"]
    h, _ = oracle.moe_ep_layer0(d["x_shards"], w1, ids, c.E, "f16", tp=tp)
    y = oracle.moe_ep_layer1(h, w2, ids, g, c.E, "f16", c.R, h_dtype="f64", tp=tp)
    X = np.concatenate(d["x_shards"]).astype(np.int64)
    W1i, W2i = W1.astype(np.int64), W2.astype(np.int64)
    for t in range(c.T):
        o, lt = divmod(t, c.T // c.R)
        for j in range(c.H):
            acc = Fraction(0)
            for k in range(c.topk):
                e = int(ids[t, k])
                hrow = [sum(int(X[t, i]) * int(W1i[e, i, f]) for i in range(c.H)) for f in range(c.F)]
                acc += Fraction(float(g[t, k])) * sum(hrow[f] * int(W2i[e, f, j]) for f in range(c.F))
            assert abs(Fraction(y[o][lt, j]) - acc) <= Fraction(1, 2 ** 30)


def test_moe_ep_layer0_equals_the_tp_column_blocks():
    # the same experts sharded by columns (TP) or by expert (EP) give the same rows
    c, d = _moe_small(R=2, T=8, H=6, F=8, E=4, topk=2)
    _, _, w1_tp, _, w1_ep, _ = _ep_weights(c)
    h_tp, r_tp = oracle.moe_layer0(d["x_shards"], w1_tp, d["topk_ids"], c.E, "f16")
    h_ep, r_ep = oracle.moe_ep_layer0(d["x_shards"], w1_ep, d["topk_ids"], c.E, "f16")
    assert np.array_equal(h_ep, np.concatenate(h_tp, axis=1))
    for a, b in zip(r_tp, r_ep):
        assert np.array_equal(a, b)


def test_moe_ep_layer1_equals_tp_with_row_blocks():
    c, d = _moe_small(R=2, T=8, H=6, F=8, E=4, topk=2)
    _, _, _, w2_tp, _, w2_ep = _ep_weights(c)
    h = gen.normal16((21, 1), (c.T * c.topk, c.F), 1.0, "f16")
    fr = c.F // c.R
    h_tp = [np.ascontiguousarray(h[:, r * fr:(r + 1) * fr]) for r in range(c.R)]
    y_tp = oracle.moe_layer1(h_tp, w2_tp, d["topk_ids"], d["topk_weights"], c.E, "f16")
    y_ep = oracle.moe_ep_layer1(h, w2_ep, d["topk_ids"], d["topk_weights"], c.E, "f16", c.R)
    for o in range(c.R):
        assert np.allclose(y_ep[o], y_tp[o], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("tp", [1, 2])
def test_moe_ep_layer1_rows_match_full(tp):
    c, d = _moe_small(R=2, T=8, H=6, F=8, E=4, topk=2)
    W1, W2, _, _, _, _ = _ep_weights(c)
    _, w2 = _eptp_shards(W1, W2, c.R, tp)
    h = gen.normal16((22, tp), (c.T * c.topk, c.F), 1.0, "f16")
    y = oracle.moe_ep_layer1(h, w2, d["topk_ids"], d["topk_weights"], c.E, "f16", c.R, tp=tp)
    lr = np.array([0, 3, 2])
    for o in range(c.R):
        got = oracle.moe_ep_layer1_rows(h, w2, d["topk_ids"], d["topk_weights"], c.E, "f16", c.R,
                                        o, lr, tp=tp)
        assert np.allclose(got, y[o][lr], rtol=1e-13, atol=1e-14)


def test_moe_ep_chain_brute_force_integers():
    # per token, per slot, in exact rationals: y_t = sum_k g (x_t W1_e) W2_e
    c, d = _moe_small(R=2, T=4, H=3, F=4, E=2, topk=2, dist="int")
    W1, W2, _, _, w1_ep, w2_ep = _ep_weights(c, dist="int")
    ids, g = d["topk_ids"], d["topk_weights"]
    h, _ = oracle.moe_ep_layer0(d["x_shards"], w1_ep, ids, c.E, "f16")
    y = oracle.moe_ep_layer1(h, w2_ep, ids, g, c.E, "f16", c.R, h_dtype="f64")
    X = np.concatenate(d["x_shards"]).astype(np.int64)
    W1i, W2i = W1.astype(np.int64), W2.astype(np.int64)
    for t in range(c.T):
        o, lt = divmod(t, c.T // c.R)
        for j in range(c.H):
            acc = Fraction(0)
            for k in range(c.topk):
                e = int(ids[t, k])
                hrow = [sum(int(X[t, i]) * int(W1i[e, i, f]) for i in range(c.H)) for f in range(c.F)]
                acc += Fraction(float(g[t, k])) * sum(hrow[f] * int(W2i[e, f, j]) for f in range(c.F))
            assert abs(Fraction(y[o][lt, j]) - acc) <= Fraction(1, 2 ** 30)


def test_moe_ep_rank_rows_are_the_owner_experts():
    # rank r's rows are those of experts [r E/R, (r+1) E/R): they come from x . W1 of its own experts
    c, d = _moe_small(R=2, T=8, H=6, F=4, E=4, topk=2)
    W1, _, _, _, w1_ep, _ = _ep_weights(c)
    h, (_, offsets, _, r2s) = oracle.moe_ep_layer0(d["x_shards"], w1_ep, d["topk_ids"], c.E, "f16")
    X = np.concatenate([oracle.widen(x, "f16") for x in d["x_shards"]])
    el = c.E // c.R
    for r in range(c.R):
        for row in range(int(offsets[r * el]), int(offsets[(r + 1) * el])):
            s = int(r2s[row])
            e = int(d["topk_ids"][s // c.topk, s % c.topk])
            assert e // el == r
            assert np.allclose(h[row], X[s // c.topk] @ oracle.widen(W1[e], "f16"), rtol=1e-14)


# ---------------------------------------------------------------- top-k gate
def test_gate_topk_equals_e_is_the_softmax():
    # k = E: every expert chosen, weights = the library softmax of the scores
    from scipy.special import softmax
    g = np.random.default_rng(3)
    L = g.standard_normal((6, 5)).astype(np.float32) * 3
    ids, w = oracle.moe_topk_gate(L, 5)
    for t in range(6):
        want = softmax(L[t].astype(np.float64))
        assert np.allclose(w[t], want[ids[t]], rtol=1e-13, atol=0)
        assert np.all(np.diff(L[t][ids[t]]) <= 0)  # largest first


def test_gate_topk_is_the_renormalised_softmax():
    from scipy.special import softmax
    g = np.random.default_rng(4)
    L = g.standard_normal((20, 16)).astype(np.float32)
    for k in (1, 2, 5):
        ids, w = oracle.moe_topk_gate(L, k)
        for t in range(20):
            full = softmax(L[t].astype(np.float64))
            assert set(ids[t].tolist()) == set(np.argsort(-full, kind="stable")[:k].tolist())
            assert np.allclose(w[t], full[ids[t]] / full[ids[t]].sum(), rtol=1e-13)
        if k == 1:
            assert np.array_equal(ids[:, 0], np.argmax(L, axis=1)) and np.all(w == 1.0)


def test_gate_ties_shift_and_infinities():
    L = np.array([[1, 3, 3, 2],            # tie: lower id first, equal weights
                  [0, 0, 0, 0],            # all equal: ids 0, 1
                  [np.nan, -1, 5, np.inf],  # +inf wins everything
                  [-np.inf] * 4,           # all -inf: lowest ids, uniform
                  [np.nan, np.nan, 2, 2]],  # NaN counts as -inf
                 dtype=np.float32)
    ids, w = oracle.moe_topk_gate(L, 2)
    assert ids.tolist() == [[1, 2], [0, 1], [3, 2], [0, 1], [2, 3]]
    assert w.tolist() == [[0.5, 0.5], [0.5, 0.5], [1.0, 0.0], [0.5, 0.5], [0.5, 0.5]]
    # a constant shift of a token's scores changes nothing (exactly representable shift)
    g = np.random.default_rng(5)
    B = np.round(g.standard_normal((8, 8)) * 64).astype(np.float32) / 64
    i0, w0 = oracle.moe_topk_gate(B, 3)
    i1, w1 = oracle.moe_topk_gate(B + np.float32(8), 3)
    assert np.array_equal(i0, i1) and np.allclose(w0, w1, rtol=1e-14)
    # two chosen scores a, b: w = (1 / (1 + e^(b-a)), e^(b-a) / (1 + e^(b-a)))
    _, w2 = oracle.moe_topk_gate(np.array([[0.0, 1.0, -7.0]], dtype=np.float32), 2)
    e = np.exp(-1.0)
    assert np.allclose(w2[0], [1 / (1 + e), e / (1 + e)], rtol=1e-15)
