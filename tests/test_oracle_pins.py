"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test names what it pins: brute-force sums on tiny inputs, exact rational
arithmetic, closed-form probes, the hand-derived schedule fixture, invariants
the pages fix (own chunk last / first, decomposed equals collective) and a
brute-force search over schedules. A few tests plant a mistake in the oracle
(monkeypatched, on the CPU) and check that a pin catches it.
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import flashoverlap_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ints(rng, shape):
    return rng.integers(-4, 5, size=shape).astype(np.float64)


# --------------------------------------------------------------------------
# Brute force: explicit sums of products in pure Python (tiny inputs).
# --------------------------------------------------------------------------

def _bf_gemm_rs(X, W):
    R = len(X)
    M, K = X[0].shape
    N = W[0].shape[1]
    rows = M // R
    out = []
    for d in range(R):
        y = [[0 for _ in range(N)] for _ in range(rows)]
        for i in range(rows):
            for j in range(N):
                acc = 0
                for r in range(R):
                    for k in range(K):
                        acc += int(X[r][d * rows + i][k]) * int(W[r][k][j])
                y[i][j] = acc
        out.append(np.array(y, dtype=np.float64))
    return out


@pytest.mark.parametrize("R,M,K,N", [(1, 3, 4, 5), (2, 4, 3, 2), (3, 6, 5, 4), (4, 8, 2, 3)])
def test_gemm_rs_matches_brute_force(R, M, K, N):
    rng = np.random.default_rng(R * 100 + M)
    X = [_ints(rng, (M, K)) for _ in range(R)]
    W = [_ints(rng, (K, N)) for _ in range(R)]
    got = oracle.gemm_rs(X, W)
    ref = _bf_gemm_rs(X, W)
    for d in range(R):
        assert np.array_equal(got[d], ref[d])


@pytest.mark.parametrize("R,M,K,N", [(1, 3, 4, 5), (2, 4, 3, 2), (3, 6, 5, 4)])
def test_gemm_ar_matches_brute_force(R, M, K, N):
    rng = np.random.default_rng(R * 31 + M)
    X = [_ints(rng, (M, K)) for _ in range(R)]
    W = [_ints(rng, (K, N)) for _ in range(R)]
    got = oracle.gemm_ar(X, W)
    for q in range(R):
        for i in range(M):
            for j in range(N):
                want = sum(int(X[r][i][k]) * int(W[r][k][j]) for r in range(R) for k in range(K))
                assert got[q][i, j] == want
    # all-reduce = reduce-scatter, then every rank gathers the R shards
    rs = oracle.gemm_rs(X, W)
    for q in range(R):
        assert np.array_equal(got[q], np.concatenate(rs, axis=0))
    assert len(oracle.ar_transfers(R)) == 2 * R * (R - 1)


@pytest.mark.parametrize("R,M,K,N", [(1, 2, 3, 4), (2, 4, 3, 5), (3, 6, 2, 3)])
def test_ag_gemm_matches_brute_force(R, M, K, N):
    rng = np.random.default_rng(7 + R)
    X = [_ints(rng, (M // R, K)) for _ in range(R)]
    W = [_ints(rng, (K, N)) for _ in range(R)]
    Y, G = oracle.ag_gemm(X, W)
    rows = M // R
    for r in range(R):
        for g in range(M):
            src, i = divmod(g, rows)
            for j in range(N):
                want = sum(int(X[src][i][k]) * int(W[r][k][j]) for k in range(K))
                assert Y[r][g, j] == want
    for g in range(M):
        src, i = divmod(g, rows)
        assert np.array_equal(G[g], X[src][i])


@pytest.mark.parametrize("R,T,M,N", [(1, 3, 2, 4), (2, 3, 4, 2), (4, 2, 8, 3)])
def test_dp_grad_rs_matches_brute_force(R, T, M, N):
    rng = np.random.default_rng(11 + R)
    X = [_ints(rng, (T, M)) for _ in range(R)]
    dY = [_ints(rng, (T, N)) for _ in range(R)]
    got = oracle.dp_grad_rs(X, dY)
    rows = M // R
    for d in range(R):
        for i in range(rows):
            for j in range(N):
                want = sum(int(X[r][t][d * rows + i]) * int(dY[r][t][j])
                           for r in range(R) for t in range(T))
                assert got[d][i, j] == want


def test_weight_grads_match_brute_force():
    rng = np.random.default_rng(17)
    X = [_ints(rng, (3, 4)) for _ in range(2)]
    dY = [_ints(rng, (3, 2)) for _ in range(2)]
    got = oracle.weight_grads(X, dY)
    for r in range(2):
        for i in range(4):
            for j in range(2):
                assert got[r][i, j] == sum(int(X[r][t][i]) * int(dY[r][t][j]) for t in range(3))


def test_sampled_rows_equal_full():
    rng = np.random.default_rng(5)
    R, M, K, N = 4, 16, 6, 5
    X = [_ints(rng, (M, K)) for _ in range(R)]
    W = [_ints(rng, (K, N)) for _ in range(R)]
    full = oracle.gemm_rs(X, W)
    for d in range(R):
        assert np.array_equal(oracle.gemm_rs_rows(X, W, d, [0, 3, 1]), full[d][[0, 3, 1]])
    Xa = [_ints(rng, (M // R, K)) for _ in range(R)]
    Y, _ = oracle.ag_gemm(Xa, W)
    for r in range(R):
        assert np.array_equal(oracle.ag_gemm_rows(Xa, W, r, [0, 5, 15]), Y[r][[0, 5, 15]])
    Xd = [_ints(rng, (K, M)) for _ in range(R)]
    dY = [_ints(rng, (K, N)) for _ in range(R)]
    D = oracle.dp_grad_rs(Xd, dY)
    for d in range(R):
        assert np.array_equal(oracle.dp_grad_rs_rows(Xd, dY, d, [2, 0]), D[d][[2, 0]])
    G = oracle.weight_grads(Xd, dY)
    for r in range(R):
        assert np.array_equal(oracle.weight_grads_rows(Xd, dY, r, [3, 0, 15]), G[r][[3, 0, 15]])


# --------------------------------------------------------------------------
# Exact rational arithmetic: the fp64 oracle is within fp64 rounding of the
# exact value for non-integer inputs.
# --------------------------------------------------------------------------

def test_gemm_rs_within_fp64_rounding_of_exact():
    rng = np.random.default_rng(3)
    R, M, K, N = 2, 4, 7, 3
    X = [rng.standard_normal((M, K)) for _ in range(R)]
    W = [rng.standard_normal((K, N)) * 0.02 for _ in range(R)]
    got = oracle.gemm_rs(X, W)
    rows = M // R
    for d in range(R):
        for i in range(rows):
            for j in range(N):
                exact = sum(Fraction(float(X[r][d * rows + i, k])) * Fraction(float(W[r][k, j]))
                            for r in range(R) for k in range(K))
                mag = sum(abs(Fraction(float(X[r][d * rows + i, k])) * Fraction(float(W[r][k, j])))
                          for r in range(R) for k in range(K))
                assert abs(Fraction(got[d][i, j]) - exact) <= mag * Fraction(2 * R * K, 2 ** 52)


# --------------------------------------------------------------------------
# Closed-form probes.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("R", [1, 2, 3, 4, 8])
def test_ag_identity_weight_returns_gather_in_rank_order(R):
    rows, K = 3, 5
    X = [np.arange(rows * K, dtype=np.float64).reshape(rows, K) + 100 * r for r in range(R)]
    W = [np.eye(K) for _ in range(R)]
    Y, G = oracle.ag_gemm(X, W)
    for r in range(R):
        for q in range(R):
            assert np.array_equal(Y[r][q * rows:(q + 1) * rows], X[q])
            assert np.array_equal(G[q * rows:(q + 1) * rows], X[q])


def _pow2_probe(R, M, K, N):
    """X_r = 2^r * E with E one-hot per row (row i -> column i mod K),
    W_r[k, j] = k + 1. Then Y_d[i, j] = (2^R - 1) * (((d*M/R + i) mod K) + 1)."""
    X, W = [], []
    for r in range(R):
        E = np.zeros((M, K))
        E[np.arange(M), np.arange(M) % K] = 1.0
        X.append((2.0 ** r) * E)
        W.append(np.repeat((np.arange(K, dtype=np.float64) + 1)[:, None], N, axis=1))
    rows = M // R
    want = [np.repeat(((((d * rows + np.arange(rows)) % K) + 1) * (2 ** R - 1))[:, None], N, axis=1)
            .astype(np.float64) for d in range(R)]
    return X, W, want


@pytest.mark.parametrize("R", [1, 2, 3, 5, 8])
def test_power_of_two_probe_each_contribution_exactly_once(R):
    X, W, want = _pow2_probe(R, 4 * R, 7, 3)
    for f in (oracle.gemm_rs, oracle.simulate_gemm_rs,
              lambda x, w: oracle.simulate_gemm_rs(x, w, ring=True)):
        got = f(X, W)
        for d in range(R):
            assert np.array_equal(got[d], want[d])


def test_planted_dropped_contribution_is_caught(monkeypatch):
    real = O.reduce_scatter_rows

    def dropped(P):
        return real([np.zeros_like(P[0])] + list(P[1:]))   # rank 0's partial lost

    monkeypatch.setattr(O, "reduce_scatter_rows", dropped)
    X, W, want = _pow2_probe(3, 12, 5, 2)
    got = O.gemm_rs(X, W)
    assert not all(np.array_equal(got[d], want[d]) for d in range(3))


def test_planted_wrong_row_block_is_caught(monkeypatch):
    real = O.reduce_scatter_rows

    def rotated(P):
        out = real(P)
        return out[1:] + out[:1]

    monkeypatch.setattr(O, "reduce_scatter_rows", rotated)
    X, W, want = _pow2_probe(4, 16, 5, 2)
    got = O.gemm_rs(X, W)
    assert not all(np.array_equal(got[d], want[d]) for d in range(4))


def test_planted_transposed_operand_is_caught():
    rng = np.random.default_rng(9)
    X = [_ints(rng, (4, 4)) for _ in range(2)]
    W = [_ints(rng, (4, 4)) for _ in range(2)]
    ref = _bf_gemm_rs(X, W)
    wrong = O.reduce_scatter_rows([X[r] @ W[r].T for r in range(2)])
    assert not all(np.array_equal(wrong[d], ref[d]) for d in range(2))


# --------------------------------------------------------------------------
# Decomposed == collective (integer mode: bit-equal).
# --------------------------------------------------------------------------

@pytest.mark.parametrize("R", [1, 2, 3, 4, 6, 8])
def test_decomposed_rs_equals_collective(R):
    rng = np.random.default_rng(R)
    M, K, N = 2 * R, 5, 3
    X = [_ints(rng, (M, K)) for _ in range(R)]
    W = [_ints(rng, (K, N)) for _ in range(R)]
    ref = oracle.gemm_rs(X, W)
    for ring in (False, True):
        got = oracle.simulate_gemm_rs(X, W, ring=ring)
        for d in range(R):
            assert np.array_equal(got[d], ref[d])
    got = oracle.simulate_gemm_rs(X, W, schedule=oracle.sliced_schedule(R))
    for d in range(R):
        assert np.array_equal(got[d], ref[d])


@pytest.mark.parametrize("R", [1, 2, 3, 4, 8])
def test_decomposed_ag_equals_collective(R):
    rng = np.random.default_rng(20 + R)
    rows, K, N = 2, 4, 3
    X = [_ints(rng, (rows, K)) for _ in range(R)]
    W = [_ints(rng, (K, N)) for _ in range(R)]
    ref, G = oracle.ag_gemm(X, W)
    got, Gr = oracle.simulate_ag_gemm(X, W)
    for r in range(R):
        assert np.array_equal(got[r], ref[r])
        assert np.array_equal(Gr[r], G)


@pytest.mark.parametrize("R", [1, 2, 4, 8])
def test_decomposed_dp_grad_equals_collective(R):
    rng = np.random.default_rng(40 + R)
    T, M, N = 3, 2 * R, 3
    X = [_ints(rng, (T, M)) for _ in range(R)]
    dY = [_ints(rng, (T, N)) for _ in range(R)]
    ref = oracle.dp_grad_rs(X, dY)
    got = oracle.simulate_dp_grad_rs(X, dY)
    for d in range(R):
        assert np.array_equal(got[d], ref[d])


def test_ag_simulator_rejects_use_before_arrival():
    R = 3
    X = [np.ones((1, 2)) for _ in range(R)]
    W = [np.ones((2, 1)) for _ in range(R)]
    bad = oracle.ag_schedule(R).copy()
    bad[:, [1, 2]] = bad[:, [2, 1]]          # consume the 2-hop shard first
    with pytest.raises(AssertionError):
        oracle.simulate_ag_gemm(X, W, schedule=bad)


def test_ring_rs_rejects_schedule_without_own_last():
    R = 3
    X = [np.ones((3, 2)) for _ in range(R)]
    W = [np.ones((2, 1)) for _ in range(R)]
    with pytest.raises(AssertionError):
        oracle.simulate_gemm_rs(X, W, schedule=oracle.sliced_schedule(R), ring=True)


# --------------------------------------------------------------------------
# Schedules: the hand-derived fixture and the invariants the pages fix.
# --------------------------------------------------------------------------

def _read_golden_schedule():
    rs, ag = {}, {}
    with open(os.path.join(GOLDEN, "schedule_r4.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, vals = line.split(":")
            op, r = head.split()
            (rs if op == "rs" else ag)[int(r)] = [int(v) for v in vals.split()]
    return rs, ag


def test_schedules_match_hand_derived_fixture():
    rs, ag = _read_golden_schedule()
    assert oracle.rs_schedule(4).tolist() == [rs[r] for r in range(4)]
    assert oracle.ag_schedule(4).tolist() == [ag[r] for r in range(4)]


@pytest.mark.parametrize("R", list(range(1, 17)))
def test_schedule_invariants(R):
    rs = oracle.rs_schedule(R)
    ag = oracle.ag_schedule(R)
    for r in range(R):
        assert sorted(rs[r].tolist()) == list(range(R))       # (i) permutation
        assert sorted(ag[r].tolist()) == list(range(R))
        assert rs[r, R - 1] == r                               # (ii) own chunk last
        assert ag[r, 0] == r                                   #      own shard first
    for s in range(R):
        assert sorted(rs[:, s].tolist()) == list(range(R))    # (iii) bijection per step
        assert sorted(ag[:, s].tolist()) == list(range(R))
    tr = oracle.rs_transfers(R)
    assert len(tr) == R * (R - 1)                              # (v)
    assert all(step < R - 1 for (_, _, _, step) in tr)        # no send at the last step
    assert len(set((d, c, s) for (_, d, c, s) in tr)) == len(tr)
    ring = oracle.rs_transfers(R, ring=True)
    assert len(ring) == R * (R - 1)
    agt = oracle.ag_transfers(R)
    assert len(agt) == R * (R - 1)
    for (src, dst, shard, s) in agt:                           # ring forwarding feeds step s+1
        assert ag[dst, s + 1] == shard


@pytest.mark.parametrize("R", [2, 3, 4, 5])
def test_dependency_graph_is_acyclic_and_respects_order(R):
    edges = oracle.rs_dependency_edges(R)
    nodes = {(r, s) for r in range(R) for s in range(R)}
    indeg = {n: 0 for n in nodes}
    for a, b in edges:
        indeg[b] += 1
    ready = [n for n in nodes if indeg[n] == 0]
    seen = 0
    adj = {n: [] for n in nodes}
    for a, b in edges:
        adj[a].append(b)
    while ready:
        n = ready.pop()
        seen += 1
        for m in adj[n]:
            indeg[m] -= 1
            if indeg[m] == 0:
                ready.append(m)
    assert seen == len(nodes)
    for (a, b) in edges:
        if a[0] != b[0]:
            assert b[1] > a[1] or b[1] == R - 1                # consumer later in its own order


# --------------------------------------------------------------------------
# Brute force over per-rank orders under the cost model.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("R", [2, 3, 4])
@pytest.mark.parametrize("tx", [0.3, 0.6, 0.9, 1.0])
def test_rank_adaptive_is_optimal_and_tail_free(R, tx):
    tc = 1.0
    ends, last_sends = oracle.brute_force_rs(R, tc, tx)
    ra = oracle.rs_makespan(oracle.rs_schedule(R), tc, tx)
    assert ra == pytest.approx(R * tc)
    assert ends.min() == pytest.approx(R * tc)
    if R > 1:
        assert np.all(ends[last_sends] >= R * tc + tx - 1e-12)
    sl = oracle.rs_makespan(oracle.sliced_schedule(R), tc, tx)
    if R > 1:
        assert sl >= R * tc + tx - 1e-12


def test_own_last_alone_is_not_enough_when_transfers_collide():
    # Two ranks sending to one owner in the same step serialise: with
    # t_x > t_c / 2 such an order is slower although every own chunk is last.
    R, tc, tx = 3, 1.0, 0.9
    orders = np.array([[1, 2, 0], [2, 0, 1], [1, 0, 2]])   # ranks 0 and 2 both send chunk 1 first
    assert all(orders[r, R - 1] == r for r in range(R))
    assert oracle.rs_makespan(orders, tc, tx) > R * tc


def test_vectorised_brute_force_matches_scalar_model():
    R = 3
    perms = list(itertools.permutations(range(R)))
    ends, _ = oracle.brute_force_rs(R, 1.0, 0.7)
    rng = np.random.default_rng(0)
    combos = list(itertools.product(range(len(perms)), repeat=R))
    for i in rng.choice(len(combos), 40, replace=False):
        orders = np.array([perms[q] for q in combos[i]])
        assert ends[i] == pytest.approx(oracle.rs_makespan(orders, 1.0, 0.7))


# --------------------------------------------------------------------------
# Output precision and error measures.
# --------------------------------------------------------------------------

def test_round_bf16_known_values():
    one = 1.0
    ulp = 2.0 ** -7
    assert oracle.round_bf16(np.array([one + ulp / 2]))[0] == one                 # tie -> even
    assert oracle.round_bf16(np.array([one + 1.5 * ulp]))[0] == one + 2 * ulp     # tie -> even
    assert oracle.round_bf16(np.array([one + 0.51 * ulp]))[0] == one + ulp
    assert oracle.round_bf16(np.array([-3.0]))[0] == -3.0
    assert oracle.round_bf16(np.array([0.0]))[0] == 0.0


def test_round_bf16_matches_torch_cast_on_fp32_values():
    g = torch.Generator().manual_seed(0)
    x = torch.randn(100000, generator=g) * 37.0
    want = x.to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(x.to(torch.float64).numpy())
    assert np.array_equal(got, want)


def test_rel_errors_simple_cases():
    ref = np.array([1.0, -2.0, 0.0, 4.0])
    fro, mx, clamped = oracle.rel_errors(ref, ref)
    assert fro == 0.0 and mx == 0.0 and clamped == 1
    got = ref + np.array([0.1, 0.0, 0.0, 0.0])
    fro, mx, _ = oracle.rel_errors(got, ref)
    assert fro == pytest.approx(0.1 / np.sqrt(21.0))
    assert mx == pytest.approx(0.1)
    # the denominator floor: rms(ref) = sqrt(21/4); an error on the zero element
    near0 = ref + np.array([0.0, 0.0, 1e-3, 0.0])
    rms = np.sqrt(21.0 / 4.0)
    assert oracle.rel_errors(near0, ref)[1] == pytest.approx(1e-3 / (1e-3 * rms))
    assert oracle.rel_errors(near0, ref, 1e-2)[1] == pytest.approx(1e-3 / (1e-2 * rms))


# --------------------------------------------------------------------------
# Transfer lists and dependency edges: hand-derived fixture for R = 3 and 4,
# an execution of the message lists on data, and a reachability pin.
# --------------------------------------------------------------------------

def _read_golden_transfers():
    """{(kind, R): [tuples]} from tests/golden/transfers_r3_r4.txt."""
    out = {}
    with open(os.path.join(GOLDEN, "transfers_r3_r4.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, vals = line.split(":")
            parts = head.split()
            kind, R = parts[0], int(parts[1])
            key = (kind, R) if kind != "table" else (kind, R, int(parts[2]))
            out.setdefault(key, []).append(tuple(int(v) for v in vals.split()))
    return out


def _fixture_edges(R):
    return sorted(((a, b), (c, d)) for (a, b, c, d) in _read_golden_transfers()[("edge", R)])


def _ar_fixture_ok(R, fn):
    return sorted(fn(R)) == sorted(_read_golden_transfers()[("ar", R)])


def _edges_fixture_ok(R, fn):
    return sorted(fn(R)) == _fixture_edges(R)


@pytest.mark.parametrize("R", [3, 4])
def test_transfer_lists_match_hand_derived_fixture(R):
    g = _read_golden_transfers()
    assert oracle.rs_schedule(R).tolist() == [list(g[("table", R, r)][0]) for r in range(R)]
    assert sorted(oracle.rs_transfers(R)) == sorted(g[("rs_direct", R)])
    assert sorted(oracle.rs_transfers(R, ring=True)) == sorted(g[("rs_ring", R)])
    assert sorted(oracle.ag_transfers(R)) == sorted(g[("ag", R)])
    assert _ar_fixture_ok(R, oracle.ar_transfers)
    for kind in ("rs_direct", "rs_ring", "ag", "ar"):
        assert len(set(g[(kind, R)])) == len(g[(kind, R)])       # no duplicate message


@pytest.mark.parametrize("R", [3, 4])
def test_dependency_edges_match_hand_derived_fixture(R):
    assert _edges_fixture_ok(R, oracle.rs_dependency_edges)


def _run_ar_messages(P, msgs, sch):
    """Execute an all-reduce message list on data (pure Python bookkeeping).

    Rank r starts with its [M, N] partial P_r. A message (src, dst, c, s) with
    s < R is a reduce-scatter partial: src must compute chunk c at step s, and
    owner dst == c adds rows c of P_src into its shard. A message with s == R
    is the all-gather half: src must be the owner of c, and dst receives the
    finished shard. Returns every rank's [M, N] result, or raises on a message
    that the schedule cannot produce.
    """
    R = len(P)
    rows = P[0].shape[0] // R
    shard = {c: P[c][c * rows:(c + 1) * rows].copy() for c in range(R)}
    got = {(q, c): None for q in range(R) for c in range(R)}
    for (src, dst, c, s) in sorted(msgs, key=lambda m: m[3]):
        if s < R:
            if int(sch[src, s]) != c or dst != c or src == c:
                raise AssertionError(f"bad reduce-scatter message {(src, dst, c, s)}")
            shard[c] = shard[c] + P[src][c * rows:(c + 1) * rows]
        else:
            if src != c or dst == c:
                raise AssertionError(f"bad all-gather message {(src, dst, c, s)}")
            got[(dst, c)] = shard[c].copy()
    for c in range(R):
        got[(c, c)] = shard[c]
    if any(v is None for v in got.values()):
        raise AssertionError("a rank misses a shard")
    return [np.concatenate([got[(q, c)] for c in range(R)], axis=0) for q in range(R)]


@pytest.mark.parametrize("R", [1, 2, 3, 4, 6])
def test_ar_transfers_executed_on_data_give_the_all_reduce(R):
    rng = np.random.default_rng(60 + R)
    M, K, N = 2 * R, 3, 2
    X = [_ints(rng, (M, K)) for _ in range(R)]
    W = [_ints(rng, (K, N)) for _ in range(R)]
    P = [X[r] @ W[r] for r in range(R)]
    got = _run_ar_messages(P, oracle.ar_transfers(R), oracle.rs_schedule(R))
    want = oracle.gemm_ar(X, W)
    for q in range(R):
        assert np.array_equal(got[q], want[q])


def _reaches(edges, a, b):
    adj = {}
    for u, v in edges:
        adj.setdefault(u, []).append(v)
    stack, seen = [a], {a}
    while stack:
        u = stack.pop()
        if u == b:
            return True
        for v in adj.get(u, []):
            if v not in seen:
                seen.add(v)
                stack.append(v)
    return False


def _edges_order_every_contribution_before_owner(R, edges):
    sch = oracle.rs_schedule(R)
    for r in range(R):
        for s in range(R):
            c = int(sch[r, s])
            if c != r and not _reaches(edges, (r, s), (c, R - 1)):
                return False
        for s in range(R - 1):
            if ((r, s), (r, s + 1)) not in edges:
                return False
    return True


@pytest.mark.parametrize("R", [2, 3, 4, 5, 8])
def test_dependency_edges_order_every_contribution_before_the_owners_last_task(R):
    edges = oracle.rs_dependency_edges(R)
    assert _edges_order_every_contribution_before_owner(R, edges)
    # the own-chunk task is the only one that consumes a transfer
    for (a, b) in edges:
        if a[0] != b[0]:
            assert b[1] == R - 1


def test_planted_wrong_all_gather_destination_is_caught(monkeypatch):
    real = O.ar_transfers

    def wrong_chunk(R):
        rs = O.rs_transfers(R)
        return rs + [(c, q, q, R) for c in range(R) for q in range(R) if q != c]

    monkeypatch.setattr(O, "ar_transfers", wrong_chunk)
    for R in (3, 4):
        assert len(O.ar_transfers(R)) == len(real(R))           # the old count pin passes
        assert not _ar_fixture_ok(R, O.ar_transfers)
    R = 3
    P = [np.arange(R * 2 * 2, dtype=np.float64).reshape(R * 2, 2) + r for r in range(R)]
    with pytest.raises(AssertionError):
        _run_ar_messages(P, O.ar_transfers(R), O.rs_schedule(R))


def test_planted_dropped_transfer_edges_are_caught(monkeypatch):
    def program_order_only(R, schedule=None):
        return [((r, s), (r, s + 1)) for r in range(R) for s in range(R - 1)]

    monkeypatch.setattr(O, "rs_dependency_edges", program_order_only)
    for R in (3, 4):
        assert not _edges_fixture_ok(R, O.rs_dependency_edges)
        assert not _edges_order_every_contribution_before_owner(R, O.rs_dependency_edges(R))


def test_planted_wrong_ring_forward_is_caught(monkeypatch):
    real = O.rs_transfers

    def skip_one(R, ring=False, schedule=None):
        out = real(R, ring=ring, schedule=schedule)
        if ring:
            out = [(a, (b + 1) % R, c, s) for (a, b, c, s) in out]   # forward two hops
        return out

    monkeypatch.setattr(O, "rs_transfers", skip_one)
    g = _read_golden_transfers()
    assert sorted(O.rs_transfers(4, ring=True)) != sorted(g[("rs_ring", 4)])


# --------------------------------------------------------------------------
# Flash All-to-All (the Ulysses projection): brute force, a closed-form
# probe, decomposed == collective, the hand-derived message list.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("R,M,K,N", [(1, 2, 3, 4), (2, 4, 3, 6), (3, 6, 2, 3), (4, 8, 3, 8)])
def test_gemm_a2a_matches_brute_force(R, M, K, N):
    rng = np.random.default_rng(70 + R)
    rows = M // R
    X = [_ints(rng, (rows, K)) for _ in range(R)]
    W = [_ints(rng, (K, N)) for _ in range(R)]
    Y = oracle.gemm_a2a(X, W)
    nc = N // R
    for c in range(R):
        assert Y[c].shape == (M, nc)
        for g in range(M):
            r, i = divmod(g, rows)
            for j in range(nc):
                want = sum(int(X[r][i][k]) * int(W[r][k][c * nc + j]) for k in range(K))
                assert Y[c][g, j] == want
        assert np.array_equal(oracle.gemm_a2a_rows(X, W, c, [M - 1, 0]), Y[c][[M - 1, 0]])


@pytest.mark.parametrize("R", [1, 2, 3, 4, 8])
def test_a2a_identity_weight_moves_column_blocks(R):
    # W = I: the projection is X itself, so rank c must hold column block c
    # of every rank's tokens, stacked in rank order.
    rows, K = 3, 2 * R
    X = [np.arange(rows * K, dtype=np.float64).reshape(rows, K) + 1000 * r for r in range(R)]
    W = [np.eye(K) for _ in range(R)]
    for f in (oracle.gemm_a2a, oracle.simulate_gemm_a2a):
        Y = f(X, W)
        for c in range(R):
            for r in range(R):
                assert np.array_equal(Y[c][r * rows:(r + 1) * rows], X[r][:, 2 * c:2 * c + 2])


@pytest.mark.parametrize("R", [1, 2, 3, 4, 6, 8])
def test_decomposed_a2a_equals_collective(R):
    rng = np.random.default_rng(80 + R)
    X = [_ints(rng, (2, 5)) for _ in range(R)]
    W = [_ints(rng, (5, 2 * R)) for _ in range(R)]
    ref = oracle.gemm_a2a(X, W)
    for sch in (None, oracle.sliced_schedule(R)):
        got = oracle.simulate_gemm_a2a(X, W, schedule=sch)
        for c in range(R):
            assert np.array_equal(got[c], ref[c])


def test_a2a_simulator_rejects_a_schedule_that_repeats_a_block():
    R = 3
    X = [np.ones((1, 2)) for _ in range(R)]
    W = [np.ones((2, 3)) for _ in range(R)]
    bad = oracle.rs_schedule(R).copy()
    bad[0, 1] = bad[0, 0]
    with pytest.raises(AssertionError):
        oracle.simulate_gemm_a2a(X, W, schedule=bad)


@pytest.mark.parametrize("R", [3, 4])
def test_a2a_transfers_match_hand_derived_fixture(R):
    g = _read_golden_transfers()
    assert sorted(oracle.a2a_transfers(R)) == sorted(g[("a2a", R)])


@pytest.mark.parametrize("R", list(range(1, 17)))
def test_a2a_transfer_invariants(R):
    tr = oracle.a2a_transfers(R)
    assert len(tr) == R * (R - 1)                                   # every (src, dst != src) once
    assert sorted((a, b) for (a, b, _, _) in tr) == [(a, b) for a in range(R) for b in range(R) if a != b]
    assert all(c == d for (_, d, c, _) in tr)                        # block c goes to rank c
    assert all(s < R - 1 for (_, _, _, s) in tr)                     # the last step sends nothing
    for s in range(R - 1):                                           # one incoming block per rank and step
        assert sorted(d for (_, d, _, st) in tr if st == s) == list(range(R))


def test_planted_swapped_a2a_roles_are_caught(monkeypatch):
    def swapped(P):
        R = len(P)
        nc = P[0].shape[1] // R
        return [np.concatenate([P[c][:, r * nc:(r + 1) * nc] for r in range(R)], axis=0) for c in range(R)]

    monkeypatch.setattr(O, "all_to_all_blocks", swapped)
    R, rows, K = 3, 2, 6
    X = [np.arange(rows * K, dtype=np.float64).reshape(rows, K) + 1000 * r for r in range(R)]
    W = [np.eye(K) for _ in range(R)]
    Y = O.gemm_a2a(X, W)
    ok = all(np.array_equal(Y[c][r * rows:(r + 1) * rows], X[r][:, 2 * c:2 * c + 2])
             for c in range(R) for r in range(R))
    assert not ok


# --------------------------------------------------------------------------
# Query-split attention (the attention core and its row-parallel output
# projection): brute force, closed forms, decomposed == whole.
# --------------------------------------------------------------------------


def _bf_attention(Q, K, V, heads, causal):
    """Pure-Python softmax attention, one query row and one head at a time."""
    T, D = len(Q), len(Q[0])
    d = D // heads
    out = [[0.0] * D for _ in range(T)]
    for h in range(heads):
        for i in range(T):
            keys = range(i + 1) if causal else range(len(K))
            sc = {j: sum(Q[i][h * d + t] * K[j][h * d + t] for t in range(d)) / math.sqrt(d) for j in keys}
            m = max(sc.values())
            w = {j: math.exp(v - m) for j, v in sc.items()}
            z = sum(w.values())
            for t in range(d):
                out[i][h * d + t] = sum(w[j] * V[j][h * d + t] for j in keys) / z
    return np.array(out)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("T,heads,d", [(1, 1, 1), (4, 1, 3), (6, 2, 2), (5, 3, 4)])
def test_attention_matches_brute_force(T, heads, d, causal):
    rng = np.random.default_rng(T * 10 + heads)
    Q, K, V = (rng.standard_normal((T, heads * d)) for _ in range(3))
    got = oracle.attention(Q, K, V, heads, causal)
    assert np.allclose(got, _bf_attention(Q.tolist(), K.tolist(), V.tolist(), heads, causal), rtol=1e-12, atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(1)
    T, heads, d = 7, 2, 3
    K, V = rng.standard_normal((T, heads * d)), rng.standard_normal((T, heads * d))
    Q0 = np.zeros((T, heads * d))
    # zero queries: every score is equal, so each output row is a plain mean
    assert np.allclose(oracle.attention(Q0, K, V, heads, False), np.repeat(V.mean(axis=0, keepdims=True), T, 0))
    prefix = np.cumsum(V, axis=0) / np.arange(1, T + 1)[:, None]
    assert np.allclose(oracle.attention(Q0, K, V, heads, True), prefix)
    # causal: the first query sees only the first key
    Q = rng.standard_normal((T, heads * d))
    assert np.allclose(oracle.attention(Q, K, V, heads, True)[0], V[0])
    # non-causal: permuting keys and values together changes nothing
    perm = rng.permutation(T)
    assert np.allclose(oracle.attention(Q, K[perm], V[perm], heads, False), oracle.attention(Q, K, V, heads, False))


def test_attn_rs_is_attention_then_the_projection_reduce_scattered():
    rng = np.random.default_rng(2)
    R, T, heads, d, H = 2, 4, 1, 2, 3
    Q, K, V = ([rng.standard_normal((T, heads * d)) for _ in range(R)] for _ in range(3))
    Wo = [rng.standard_normal((heads * d, H)) for _ in range(R)]
    Y = oracle.attn_rs(Q, K, V, Wo, heads, True)
    rows = T // R
    for c in range(R):
        for i in range(rows):
            for j in range(H):
                want = 0.0
                for r in range(R):
                    o = _bf_attention(Q[r].tolist(), K[r].tolist(), V[r].tolist(), heads, True)[c * rows + i]
                    want += sum(o[t] * Wo[r][t, j] for t in range(heads * d))
                assert Y[c][i, j] == pytest.approx(want, rel=1e-12, abs=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("R", [1, 2, 3, 4])
def test_query_split_equals_whole_attention(R, causal):
    rng = np.random.default_rng(90 + R)
    T, heads, d, H = 3 * R, 2, 2, 5
    Q, K, V = ([rng.standard_normal((T, heads * d)) for _ in range(R)] for _ in range(3))
    Wo = [rng.standard_normal((heads * d, H)) for _ in range(R)]
    ref = oracle.attn_rs(Q, K, V, Wo, heads, causal)
    for sch in (None, oracle.sliced_schedule(R)):
        got = oracle.simulate_query_split(Q, K, V, Wo, heads, causal, schedule=sch)
        for c in range(R):
            assert np.allclose(got[c], ref[c], rtol=1e-12, atol=1e-12)


def test_planted_attention_mistakes_are_caught(monkeypatch):
    rng = np.random.default_rng(3)
    T, heads, d = 5, 1, 4
    Q, K, V = (rng.standard_normal((T, heads * d)) for _ in range(3))
    want = _bf_attention(Q.tolist(), K.tolist(), V.tolist(), heads, True)
    real_sqrt = np.sqrt

    class NoScale:
        def __getattr__(self, name):
            return (lambda x: 1.0) if name == "sqrt" else getattr(np, name)

    monkeypatch.setattr(O, "np", NoScale())          # the 1/sqrt(d) scale dropped
    assert not np.allclose(O.attention(Q, K, V, heads, True), want)
    monkeypatch.undo()
    assert real_sqrt is np.sqrt

    def off_by_one(Q_, K_, V_, heads_, causal_):
        # a causal mask that also hides the diagonal key (row 0 then sees nothing)
        Qf, Kf, Vf = (np.asarray(a, dtype=np.float64) for a in (Q_, K_, V_))
        S = Qf @ Kf.T / np.sqrt(d)
        S = np.where(np.tril(np.ones((T, T), dtype=bool), -1), S, -1e300)
        P = np.exp(S - S.max(axis=1, keepdims=True))
        return (P / P.sum(axis=1, keepdims=True)) @ Vf

    monkeypatch.setattr(O, "attention", off_by_one)
    assert not np.allclose(O.attention(Q, K, V, heads, True), want)
