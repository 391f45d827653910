"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test ties one oracle function to a closed form, a library routine, an
invariant the pages state, or the independent pure-Python brute force, chosen so
that a dropped term, a wrong sign, a wrong pair index or exponent, or a
transposed operand fails at least one of them.

Source: "Leyline: KV Cache Directives for Agentic Inference", section 2.2
(Delta = |R| - |S|; K_pe_new = R(Delta) K_pe; R(a)R(b) = R(a+b)) and section 2.1
(the directive D = (s_start, s_end, R, m), AMORTIZE splices in place).
"""
import math

import numpy as np
import pytest

import oracle
from oracle import brute

D = 64
THETA = 10000.0


def _rng(seed=0):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------- bf16 ----

def test_bf16_round_matches_torch_on_float32_values():
    """For float32-representable inputs the correctly rounded bf16 is torch's fp32->bf16 conversion."""
    torch = pytest.importorskip("torch")
    r = _rng(1)
    x = np.concatenate([
        r.standard_normal(20000).astype(np.float32),
        (r.standard_normal(2000) * 1e-38).astype(np.float32),  # bf16 subnormal range
        (r.standard_normal(2000) * 1e37).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895e38, -3.3895e38, 1e-45], dtype=np.float32),
    ])
    # exact ties: a bf16 value plus half its spacing
    base = torch.from_numpy(r.standard_normal(4000).astype(np.float32)).to(torch.bfloat16).to(torch.float32).numpy()
    spacing = np.abs(base) * 2.0 ** -7
    spacing = 2.0 ** np.floor(np.log2(np.maximum(spacing, 1e-30)))
    ties = (base + spacing / 2).astype(np.float32)
    x = np.concatenate([x, ties])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_round_closed_forms():
    """Ties go to even; a double just above a tie rounds up (no double rounding through fp32)."""
    one = 0x3F80
    assert oracle.bf16_round([1.0 + 2.0 ** -8])[0] == one  # tie -> even (1.0)
    assert oracle.bf16_round([1.0 + 3 * 2.0 ** -8])[0] == one + 2  # tie -> even (1 + 2^-6)
    assert oracle.bf16_round([1.0 + 2.0 ** -8 + 2.0 ** -40])[0] == one + 1  # above tie -> up
    assert oracle.bf16_round([-(1.0 + 2.0 ** -8 + 2.0 ** -40)])[0] == 0x8000 | (one + 1)
    assert oracle.bf16_round([2.0 ** -133])[0] == 1  # smallest subnormal
    assert oracle.bf16_round([2.0 ** -134])[0] == 0  # half of it: tie -> even (0)
    assert oracle.bf16_round([3.0 * 2.0 ** -134])[0] == 2  # 1.5 steps: tie -> even (2)
    assert oracle.bf16_round([3.5e38])[0] == 0x7F80  # beyond max finite -> inf


def test_bf16_round_matches_bit_pattern_brute_force():
    r = _rng(2)
    x = np.concatenate([r.standard_normal(5000), r.standard_normal(500) * 1e-39,
                        r.standard_normal(500) * 1e38])
    got = oracle.bf16_round(x)
    want = np.array([brute.bf16_round(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, want)


# ----------------------------------------------------------------- RoPE ----

def _complex_rope(v, pos, theta, layout):
    """R(pos) as multiplication of each pair (as a complex number) by exp(i pos theta_j);
    theta_j written as exp(-(2j/d) ln theta), a different expression of theta^(-2j/d)."""
    d = v.shape[0]
    j = np.arange(d // 2)
    th = np.exp(-(2.0 * j / d) * np.log(theta))
    if layout == 0:
        ix, iy = j, j + d // 2
    else:
        ix, iy = 2 * j, 2 * j + 1
    z = (v[ix] + 1j * v[iy]) * np.exp(1j * pos * th)
    out = np.empty(d)
    out[ix] = z.real
    out[iy] = z.imag
    return out


@pytest.mark.parametrize("layout", [0, 1])
def test_rope_matches_complex_exponential(layout):
    r = _rng(3)
    for _ in range(200):
        v = r.standard_normal(D)
        pos = int(r.integers(-(2 ** 17), 2 ** 17))
        got = oracle.rope(v, pos, THETA, layout)
        want = _complex_rope(v, pos, THETA, layout)
        assert np.max(np.abs(got - want)) <= 1e-9 * np.linalg.norm(v)


def test_rope_matches_matrix_exponential_of_generator():
    """R(p) = expm(p A), A the skew generator with A[j+d/2, j] = theta_j (counter-clockwise turn)."""
    scipy_linalg = pytest.importorskip("scipy.linalg")
    j = np.arange(D // 2)
    th = THETA ** (-2.0 * j / D)
    A = np.zeros((D, D))
    A[j + D // 2, j] = th
    A[j, j + D // 2] = -th
    r = _rng(4)
    for p in [1, 2, 3, 7, -5, 31, 50]:
        v = r.standard_normal(D)
        want = scipy_linalg.expm(p * A) @ v
        got = oracle.rope(v, p, THETA)
        assert np.max(np.abs(got - want)) <= 1e-10 * np.linalg.norm(v)


def test_rope_quarter_turn_textbook():
    """Pick theta so that pair 16 turns by exactly pi/2 at position P: (x, y) -> (-y, x)."""
    P = 1000
    theta = (2.0 * P / math.pi) ** 2  # theta_16 = theta^(-1/2) = pi / (2P)
    r = _rng(5)
    v = r.standard_normal(D)
    out = oracle.rope(v, P, theta)
    assert abs(out[16] - (-v[48])) < 1e-12 and abs(out[48] - v[16]) < 1e-12
    # pair 0 always has theta_0 = 1: angle P radians
    c, s = math.cos(P), math.sin(P)
    assert abs(out[0] - (v[0] * c - v[32] * s)) < 1e-12
    assert abs(out[32] - (v[0] * s + v[32] * c)) < 1e-12
    # the same on stored bf16 bands, exactly: rotated values are +-the inputs
    k = oracle.bf16_round(r.standard_normal((50, D)))
    rr = oracle.rerotate(k, 0, P, theta)
    assert np.array_equal(rr[:, 16], k[:, 48] ^ np.uint16(0x8000))
    assert np.array_equal(rr[:, 48], k[:, 16])
    rb = oracle.rotate_bf16only(k, P, theta)
    assert np.array_equal(rb[:, 16], k[:, 48] ^ np.uint16(0x8000))
    assert np.array_equal(rb[:, 48], k[:, 16])


def test_theta_j_exponent():
    assert oracle.theta_j(0, D, THETA) == 1.0
    assert math.isclose(oracle.theta_j(16, D, THETA), 0.01, rel_tol=1e-15)  # 10000^(-1/2)
    assert math.isclose(oracle.theta_j(31, D, THETA), 10000 ** (-31 / 32), rel_tol=1e-15)


def test_rope_closure_and_identity():
    """R(a)R(b) = R(a+b) and R(0) = I (section 2.2)."""
    r = _rng(6)
    for _ in range(200):
        v = r.standard_normal(D)
        a, b = (int(x) for x in r.integers(-(2 ** 17), 2 ** 17, size=2))
        lhs = oracle.rope(oracle.rope(v, a, THETA), b, THETA)
        rhs = oracle.rope(v, a + b, THETA)
        assert np.max(np.abs(lhs - rhs)) <= 1e-10 * np.linalg.norm(v)
        assert np.array_equal(oracle.rope(v, 0, THETA), v)


def test_rope_preserves_half_split_pair_norms():
    r = _rng(7)
    for _ in range(100):
        v = r.standard_normal(D)
        out = oracle.rope(v, int(r.integers(-(2 ** 17), 2 ** 17)), THETA)
        n_in = np.hypot(v[:32], v[32:])
        n_out = np.hypot(out[:32], out[32:])
        assert np.max(np.abs(n_in - n_out)) <= 1e-12 * np.max(n_in)


# ------------------------------------------------------------- rerotate ----

def test_rerotate_identity_when_position_unchanged():
    r = _rng(8)
    k = oracle.bf16_round(r.standard_normal((300, D)))
    t = r.integers(0, 2 ** 17, size=300)
    assert np.array_equal(oracle.rerotate(k, t, t), k)


def test_rerotate_equals_single_rotation_by_delta():
    """Un-rotating by t and rotating by p equals one rotation by p - t (closure), up to fp64 noise."""
    r = _rng(9)
    n = 2000
    k = oracle.bf16_round(r.standard_normal((n, D)))
    t = r.integers(0, 2 ** 17, size=n)
    p = r.integers(0, 2 ** 17, size=n)
    got = oracle.rerotate(k, t, p)
    vals = oracle.bf16_value(k)
    want = np.stack([oracle.bf16_round(oracle.rope(vals[i], int(p[i] - t[i]), THETA)) for i in range(n)])
    diff = np.abs(got.astype(np.int32) - want.astype(np.int32))
    assert np.count_nonzero(diff) <= 5  # near-tie disagreements only
    assert np.all((diff == 0) | (diff == 1))


def test_rerotate_matches_brute_force():
    r = _rng(10)
    for layout in (0, 1):
        k = oracle.bf16_round(r.standard_normal((100, D)))
        t = r.integers(0, 2 ** 17, size=100)
        p = r.integers(0, 2 ** 17, size=100)
        got = oracle.rerotate(k, t, p, THETA, layout)
        want = np.array([brute.rerotate([int(x) for x in k[i]], int(t[i]), int(p[i]), THETA, layout)
                         for i in range(100)], dtype=np.uint16)
        assert np.array_equal(got, want)


def test_rotate_bf16only_identity_and_error_bound():
    r = _rng(11)
    k = oracle.bf16_round(r.standard_normal((500, D)))
    assert np.array_equal(oracle.rotate_bf16only(k, 0), k)
    delta = r.integers(-(2 ** 16), 2 ** 16, size=500)
    got = oracle.bf16_value(oracle.rotate_bf16only(k, delta))
    vals = oracle.bf16_value(k)
    exact = np.stack([oracle.rope(vals[i], int(delta[i]), THETA) for i in range(500)])
    pair_norm = np.hypot(vals[:, :32], vals[:, 32:])
    err = np.abs(got - exact)
    # cos, sin, two products and the sum each carry at most 2^-8 relative rounding
    bound = 5 * 2.0 ** -8 * np.concatenate([pair_norm, pair_norm], axis=1)
    assert np.all(err <= bound)
    assert np.mean(err) > 0  # it is not the exact rotation


# --------------------------------------------------------------- splice ----

def _brute_items(L, dirs):
    items = [("old", t) for t in range(L)]
    for k, (s, e, n) in sorted(enumerate(dirs), key=lambda kv: -kv[1][0]):
        items = items[:s] + [("repl", (k, i)) for i in range(n)] + items[e:]
    return items


def _random_dirs(r, L, k):
    cuts = sorted(int(x) for x in r.integers(0, L + 1, size=2 * k))
    dirs = []
    for i in range(k):
        s, e = cuts[2 * i], cuts[2 * i + 1]
        dirs.append((s, e, int(r.integers(0, 6))))
    # distinct s_start required
    if len({d[0] for d in dirs}) != len(dirs):
        return None
    return dirs


def test_splice_map_matches_list_slicing():
    r = _rng(12)
    checked = 0
    while checked < 400:
        L = int(r.integers(0, 40))
        dirs = _random_dirs(r, L, int(r.integers(1, 4)))
        if dirs is None:
            continue
        newlen, kind, idx, which = oracle.splice_map(L, dirs)
        items = _brute_items(L, dirs)
        assert newlen == len(items) == L + sum(n - (e - s) for s, e, n in dirs)
        for p, (kd, v) in enumerate(items):
            if kd == "old":
                assert kind[p] == 0 and idx[p] == v
            else:
                assert kind[p] == 1 and (which[p], idx[p]) == v
        checked += 1


def test_splice_map_sequential_application():
    """Applying the directives one at a time, left to right with later spans shifted by the
    accumulated Delta, gives the same token list as the composed right-to-left pass."""
    r = _rng(13)
    for _ in range(200):
        L = int(r.integers(1, 60))
        dirs = _random_dirs(r, L, int(r.integers(1, 4)))
        if dirs is None:
            continue
        _, kind, idx, which = oracle.splice_map(L, dirs)
        composed = list(zip(kind.tolist(), idx.tolist(), which.tolist()))
        seq = [(0, t, -1) for t in range(L)]
        shift = 0
        for k in sorted(range(len(dirs)), key=lambda i: dirs[i][0]):
            s, e, n = dirs[k]
            s2, e2 = s + shift, e + shift
            seq = seq[:s2] + [(1, i, k) for i in range(n)] + seq[e2:]
            shift += n - (e - s)
        assert seq == composed


@pytest.mark.parametrize("dirs", [
    [(5, 4, 1)],            # s_start > s_end
    [(0, 11, 0)],           # s_end > L
    [(2, 6, 1), (5, 8, 1)],  # overlap
    [(3, 3, 1), (3, 5, 0)],  # shared s_start
    [(-1, 2, 0)],
])
def test_splice_map_rejects_invalid(dirs):
    with pytest.raises(ValueError):
        oracle.splice_map(10, dirs)


def _tiny_cache(r, layers, L, row):
    return oracle.bf16_round(r.standard_normal((layers, L, row)))


@pytest.mark.parametrize("latent_dim,rope_dim", [(8, 8), (512, 64)])
def test_splice_request_matches_brute_force(latent_dim, rope_dim):
    r = _rng(14)
    row = latent_dim + rope_dim
    cases = [
        (24, [(0, 5, 2)]),            # s_start = 0
        (24, [(10, 24, 3)]),          # s_end = L
        (24, [(7, 7, 4)]),            # pure insertion, Delta > 0
        (24, [(3, 9, 0)]),            # pure deletion
        (24, [(0, 24, 2)]),           # everything replaced
        (30, [(2, 4, 5), (10, 20, 1), (25, 26, 0)]),
        (17, [(16, 17, 1), (1, 2, 0)]),
        (40, [(5, 30, 12)]),
    ]
    n_cases = len(cases) if row < 100 else 3
    for L, dirs in cases[:n_cases]:
        layers = 2
        cache = _tiny_cache(r, layers, L, row)
        repl = [_tiny_cache(r, layers, n, row) for (_, _, n) in dirs]
        got = oracle.splice_request(cache, dirs, repl, latent_dim, THETA)
        for layer in range(layers):
            rows = [[int(x) for x in cache[layer, t]] for t in range(L)]
            bd = [(s, e, [[int(x) for x in repl[k][layer, i]] for i in range(n)])
                  for k, (s, e, n) in enumerate(dirs)]
            want = np.array(brute.splice(rows, bd, latent_dim, THETA), dtype=np.uint16).reshape(-1, row)
            assert np.array_equal(got[layer], want)


def test_splice_request_keeps_latents_prefix_and_repl_bits():
    r = _rng(15)
    layers, L, row = 3, 50, 72
    cache = _tiny_cache(r, layers, L, row)
    dirs = [(10, 30, 4)]
    repl = [_tiny_cache(r, layers, 4, row)]
    out = oracle.splice_request(cache, dirs, repl, 8, THETA)
    assert out.shape == (layers, L - 20 + 4, row)
    assert np.array_equal(out[:, :10], cache[:, :10])          # prefix untouched
    assert np.array_equal(out[:, 10:14], repl[0])              # R copied
    assert np.array_equal(out[:, 14:, :8], cache[:, 30:, :8])  # latents of survivors moved
    # rope band of survivors: norms per pair within bf16 rounding
    a = oracle.bf16_value(out[:, 14:, 8:])
    b = oracle.bf16_value(cache[:, 30:, 8:])
    na = np.hypot(a[..., :32], a[..., 32:])
    nb = np.hypot(b[..., :32], b[..., 32:])
    assert np.all(np.abs(na - nb) <= 2.0 ** -7 * nb + 1e-30)


# ---------------------------------------------------------------- modes ----
# EVICT (KV-streams page: evict without resetting positions) re-indexes survivors but
# keeps their positions; AMORTIZE ("Leyline: KV Cache Directives for Agentic Inference",
# section 2.1) re-encodes them at the new position.

def test_modes_match_brute_force():
    r = _rng(16)
    row, lat = 16, 8
    for _ in range(30):
        L = int(r.integers(5, 40))
        dirs = _random_dirs(r, L, int(r.integers(1, 4)))
        if dirs is None:
            continue
        modes = [int(m) for m in r.choice([0, 2], size=len(dirs))]
        cache = _tiny_cache(r, 1, L, row)
        repl = [_tiny_cache(r, 1, n, row) for (_, _, n) in dirs]
        got = oracle.splice_request(cache, dirs, repl, lat, THETA, 0, modes)
        rows = [[int(x) for x in cache[0, t]] for t in range(L)]
        bd = [(s, e, [[int(x) for x in repl[k][0, i]] for i in range(n)]) for k, (s, e, n) in enumerate(dirs)]
        want = np.array(brute.splice(rows, bd, lat, THETA, 0, modes), dtype=np.uint16).reshape(-1, row)
        assert np.array_equal(got[0], want)


def test_evict_only_is_a_pure_move():
    r = _rng(17)
    cache = _tiny_cache(r, 2, 60, 72)
    dirs = [(5, 20, 3), (30, 31, 0), (40, 40, 2)]
    repl = [_tiny_cache(r, 2, n, 72) for (_, _, n) in dirs]
    out = oracle.splice_request(cache, dirs, repl, 8, THETA, 0, [2, 2, 2])
    _, kind, idx, _ = oracle.splice_map(60, dirs)
    kept = kind == 0
    assert np.array_equal(out[:, kept], cache[:, idx[kept]])
    # with AMORTIZE the same survivors are re-encoded
    out_a = oracle.splice_request(cache, dirs, repl, 8, THETA, 0, [0, 0, 0])
    assert not np.array_equal(out_a[:, kept, 8:], cache[:, idx[kept], 8:])


def test_one_call_equals_calls_one_after_another():
    r = _rng(18)
    for trial in range(20):
        L = 50
        dirs = _random_dirs(r, L, 3)
        if dirs is None:
            continue
        modes = [int(m) for m in r.choice([0, 2], size=3)]
        cache = _tiny_cache(r, 1, L, 24)
        repl = [_tiny_cache(r, 1, n, 24) for (_, _, n) in dirs]
        one = oracle.splice_request(cache, dirs, repl, 8, THETA, 0, modes)
        seq, shift = cache, 0
        for k in sorted(range(3), key=lambda i: dirs[i][0]):
            s, e, n = dirs[k]
            seq = oracle.splice_request(seq, [(s + shift, e + shift, n)], [repl[k]], 8, THETA, 0, [modes[k]])
            shift += n - (e - s)
        # one call rounds a survivor once; one call per directive rounds it up to three
        # times.  Each rounding moves a pair by at most sqrt(2) * 2^-8 of its norm.
        assert one.shape == seq.shape
        assert np.array_equal(one[..., :8], seq[..., :8])
        a, b = oracle.bf16_value(one[..., 8:]), oracle.bf16_value(seq[..., 8:])
        pn = np.hypot(a[..., :8], a[..., 8:])
        pn = np.concatenate([pn, pn], axis=-1)
        assert np.all(np.abs(a - b) <= 4 * np.sqrt(2) * 2.0 ** -8 * pn + 1e-30)


# ---------------------------------------------------------------- heads ----
# GQA/MHA rows ("Leyline: KV Cache Directives for Agentic Inference", section 5: the
# directive abstraction extends to GQA/MHA): the row ends in several RoPE bands, the
# keys of several heads, each re-encoded alone with the same theta_j.

def test_heads_match_brute_force_and_single_band_per_head():
    r = _rng(19)
    lat, d, H = 8, 16, 3
    row = lat + H * d
    for _ in range(10):
        L = int(r.integers(5, 30))
        dirs = _random_dirs(r, L, int(r.integers(1, 3)))
        if dirs is None:
            continue
        modes = [int(m) for m in r.choice([0, 2], size=len(dirs))]
        cache = _tiny_cache(r, 1, L, row)
        repl = [_tiny_cache(r, 1, n, row) for (_, _, n) in dirs]
        got = oracle.splice_request(cache, dirs, repl, lat, THETA, 0, modes, rope_heads=H)
        rows = [[int(x) for x in cache[0, t]] for t in range(L)]
        bd = [(s, e, [[int(x) for x in repl[k][0, i]] for i in range(n)]) for k, (s, e, n) in enumerate(dirs)]
        want = np.array(brute.splice(rows, bd, lat, THETA, 0, modes, rope_heads=H), dtype=np.uint16).reshape(-1, row)
        assert np.array_equal(got[0], want)
        # head h alone, as a single-band row (its band after the copied part), gives the same bits
        for h in range(H):
            sub = np.concatenate([cache[..., :lat], cache[..., lat + h * d: lat + (h + 1) * d]], axis=-1)
            sub_repl = [np.concatenate([x[..., :lat], x[..., lat + h * d: lat + (h + 1) * d]], axis=-1) for x in repl]
            one = oracle.splice_request(sub, dirs, sub_repl, lat, THETA, 0, modes)
            assert np.array_equal(one[..., lat:], got[..., lat + h * d: lat + (h + 1) * d])
