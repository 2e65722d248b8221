"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test names what fixes the expected value: a closed form worked by hand
(derivation in the docstring), an invariant of the written format, a library
routine (numpy / torch converters, numpy sort, numpy matmul), or brute force
(all 65,536 trellis states; a 2^16-state Viterbi search).

The format readings pinned here are those of the design document: format v1,
tile order gb300_v1, mcg multiplier 0x9E3779B1 by default.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import DEFAULT_MCG_MULT as M

# ------------------------------------------------------------ converters


def test_f16_to_double_exhaustive_vs_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.f16_bits_to_f64(bits)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_bf16_to_double_exhaustive_vs_torch():
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = oracle.bf16_bits_to_f64(bits)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def _f32_probe_values():
    rng = np.random.default_rng(11)
    # every fp16 value, the midpoints between neighbours (ties), +-1 ulp of fp32
    # around the midpoints, random fp32 bit patterns and the overflow edge
    h = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (h[:-1] + h[1:]) / 2
    m32 = mids.astype(np.float32)
    near = np.concatenate([m32, np.nextafter(m32, np.float32(np.inf)),
                           np.nextafter(m32, np.float32(0))])
    rnd = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    rnd = rnd[np.isfinite(rnd)]
    edge = np.array([65504, 65519.99, 65520, 65536, 1e30, 2.0**-24, 2.0**-25, 3 * 2.0**-26,
                     2.0**-26, 0.0], dtype=np.float32)
    v = np.concatenate([h.astype(np.float32), near, rnd, edge]).astype(np.float32)
    return np.concatenate([v, -v])


def test_double_to_f16_vs_numpy():
    v = _f32_probe_values()
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    got = np.array([oracle.double_to_f16(float(a)) for a in v], dtype=np.uint16)
    assert (got == ref).all()


def test_double_to_bf16_vs_torch():
    rng = np.random.default_rng(12)
    bits = np.arange(0, 0x7F80, dtype=np.uint32)
    base = (bits << 16).view(np.float32)
    near = np.concatenate([(bits << 16 | 0x8000).view(np.float32),
                           (bits << 16 | 0x7FFF).view(np.float32),
                           (bits << 16 | 0x8001).view(np.float32)])
    rnd = rng.integers(0, 2**32, size=100000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    rnd = rnd[np.isfinite(rnd)]
    v = np.concatenate([base, near, rnd]).astype(np.float32)
    v = np.concatenate([v, -v])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.double_to_bf16(float(a)) for a in v], dtype=np.uint16)
    assert (got == ref).all()


def test_e4m3_vs_torch_on_every_fp16_value():
    """torch.float8_e4m3fn rounds to nearest even; for |v| <= 448 it must agree."""
    bits = np.arange(65536, dtype=np.uint16)
    f = bits.view(np.float16).astype(np.float32)
    ok = np.isfinite(f) & (np.abs(f) <= 448)
    f = f[ok]
    ref = torch.from_numpy(f).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = np.array([oracle.e4m3(float(a)) for a in f])
    assert np.array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))


def test_e4m3_closed_forms():
    # saturating: beyond the largest finite E4M3 value (448 = 1.75 * 2^8)
    for v in (448.0, 449.0, 463.9, 464.0, 480.0, 1e6, math.inf):
        assert oracle.e4m3(v) == 448.0 and oracle.e4m3(-v) == -448.0
    q = 2.0**-9  # least subnormal
    assert oracle.e4m3(q) == q
    assert oracle.e4m3(q / 2) == 0.0           # tie between 0 and q -> even (0)
    assert oracle.e4m3(1.5 * q) == 2 * q       # tie between q and 2q -> even (2q)
    assert oracle.e4m3(1.0 + 1 / 16) == 1.0    # tie in [1,2), ulp 1/8 -> even mantissa 000
    assert oracle.e4m3(1.0 + 3 / 16) == 1.25   # tie -> even mantissa 010
    assert oracle.e4m3(1.84375) == 1.875       # 1.11011b -> 1.111b


# ------------------------------------------------------------ codebook


def test_codebook_closed_form_zero_state():
    """s = 0: x = 0, m = 0x3B603B60, each half is 0x3B60 = 2^-1 * (1 + 864/1024)
    = 0.921875, so v = 1.84375 (exact in fp16); with the E4M3 rule 1.875."""
    assert oracle.f16_to_double(oracle.codebook_f16(0, M)) == 1.84375
    assert oracle.f16_to_double(oracle.weight_f16(0, M, True)) == 1.875
    # any multiplier: the state 0 always hashes to 0
    assert oracle.codebook_f16(0, 12345) == oracle.codebook_f16(0, M)


def test_codebook_closed_form_state_one():
    """s = 1, mult 0x9E3779B1: x = 0x9E3779B1; x & 0x8FFF8FFF = 0x8E3709B1;
    xor 0x3B603B60 -> m = 0xB55732D1.  a = 0x32D1 = 2^-3 (1 + 721/1024)
    = 1745/8192; b = 0xB557 = -2^-2 (1 + 343/1024) = -2734/8192.
    v = -989/8192 = -0.1207275390625 (fp16 bits 0xAFBA).  E4M3: ulp 2^-7 in
    [2^-4, 2^-3), 0.12073/2^-7 = 15.45 -> 15 -> -0.1171875."""
    v = oracle.codebook_f16(1, M)
    assert v == 0xAFBA
    assert oracle.f16_to_double(v) == -989 / 8192
    assert oracle.f16_to_double(oracle.weight_f16(1, M, True)) == -0.1171875


def test_codebook_invariants_all_states():
    """Each fp16 half has exponent field 12..15 (masking keeps exponent bits
    10-11, the xor sets 12-13 and clears 14), so |a|,|b| in [1/8, 2) and
    |v| < 4; no value is NaN/Inf; E4M3 never saturates."""
    vals = np.array([oracle.codebook_f16(s, M) for s in range(65536)], dtype=np.uint16)
    f = oracle.f16_bits_to_f64(vals)
    assert np.isfinite(f).all()
    assert (np.abs(f) < 4).all()
    x = (np.arange(65536, dtype=np.uint64) * M) & 0xFFFFFFFF
    m = (x & 0x8FFF8FFF) ^ 0x3B603B60
    for half in (m & 0xFFFF, m >> 16):
        ex = (half >> 10) & 31
        assert ((ex >= 12) & (ex <= 15)).all()
    # spread: the value distribution is bell shaped around 0 with std ~1
    assert 0.7 < f.std() < 1.6 and abs(f.mean()) < 0.1
    f8 = oracle.f16_bits_to_f64(np.array([oracle.weight_f16(s, M, True) for s in range(0, 65536, 7)],
                                         dtype=np.uint16))
    assert (np.abs(f8) <= 4).all()


def test_tile_positions_bijective_and_hand_values():
    pos = [oracle.tile_position(t) for t in range(256)]
    assert sorted(pos) == [(r, q) for r in range(16) for q in range(16)]
    # t = 64c + 8 r0 + 4 hf + j: row = r0 + 8 (j&1), col = c + 4 (j>>1) + 8 hf
    assert pos[0] == (0, 0)
    assert pos[1] == (8, 0)     # j = 1
    assert pos[2] == (0, 4)     # j = 2
    assert pos[3] == (8, 4)
    assert pos[4] == (0, 8)     # hf = 1
    assert pos[8] == (1, 0)     # r0 = 1
    assert pos[64] == (0, 1)    # c = 1
    assert pos[255] == (15, 15)


def test_state_constant_words_closed_form():
    """All words equal w: the circular stream has period 16, so s_t is w
    rotated right by (t*K mod 16) bits.  Pins bit order and the wrap."""
    rng = np.random.default_rng(3)
    for K in (2, 3, 4):
        for w in rng.integers(0, 65536, size=4):
            words = np.full(16 * K, w, dtype=np.uint16)
            for t in (0, 1, 5, 100, 255):
                r = (t * K) % 16
                expect = ((int(w) >> r) | (int(w) << (16 - r))) & 0xFFFF
                assert oracle.tile_state(words, K, t) == expect


def test_state_shift_register_and_tail_biting():
    """s_{t+1} keeps the top 16-K bits of s_t as its low bits; the last state
    wraps onto the first (circular stream of exactly 256*K bits)."""
    rng = np.random.default_rng(4)
    for K in (2, 3, 4):
        words = rng.integers(0, 65536, size=16 * K, dtype=np.uint16)
        s = [oracle.tile_state(words, K, t) for t in range(256)]
        mask = (1 << (16 - K)) - 1
        for t in range(256):
            assert s[(t + 1) % 256] & mask == s[t] >> K
        # weight 0's state is the first 16 bits of the stream, LSB first
        assert s[0] == int(words[0])


def test_one_state_in_zero_tile_brute_force():
    """Place each of the 65,536 states at bits [0,16) of a zero tile.  Weight 0
    decodes to cb(s); weight 1 (state s >> K) to cb(s >> K); weight 255 wraps
    to state (s << K) & 0xFFFF; every other weight sees state 0 when its
    window misses bits [0,16)."""
    K = 2
    cb = np.array([oracle.codebook_f16(s, M) for s in range(65536)], dtype=np.uint16)
    pos = [oracle.tile_position(t) for t in range(256)]
    rng = np.random.default_rng(5)
    for s in list(range(0, 65536, 97)) + list(rng.integers(0, 65536, size=200)):
        words = np.zeros(16 * K, dtype=np.uint16)
        words[0] = s
        tile = oracle.decode_tile(words, K, M)
        r0, q0 = pos[0]
        r1, q1 = pos[1]
        r255, q255 = pos[255]
        assert tile[q0, r0] == cb[s]
        assert tile[q1, r1] == cb[s >> K]
        assert tile[q255, r255] == cb[(s << K) & 0xFFFF]
        r9, q9 = pos[9]  # window [18, 34) misses the 16 placed bits
        assert tile[q9, r9] == cb[0]


def _viterbi_tailbiting(vals, target, K, start):
    """Minimum squared error over circular state paths with s_0 = start.
    Transition rule written from the format text: s' = (s >> K) | (n << (16-K))."""
    S = 1 << 16
    states = np.arange(S, dtype=np.int64)
    preds = np.stack([((states << K) & 0xFFFF) | p for p in range(1 << K)], axis=1)
    cost = np.full(S, np.inf)
    cost[start] = (vals[start] - target[0]) ** 2
    err = [(vals - target[t]) ** 2 for t in range(len(target))]
    for t in range(1, len(target)):
        cost = cost[preds].min(axis=1) + err[t]
    # close the circle: start must be a successor of the last state
    return cost[preds[start]].min()


@pytest.mark.parametrize("K", [2, 3])
def test_viterbi_round_trip(K):
    """Decode a random tile, then search all 2^16-state trellis paths for the
    decoded values: a zero-error circular path must exist (the decoder is a
    K-bit-shift trellis with 16-bit state and tail-biting), and a perturbed
    target must not be reachable exactly."""
    rng = np.random.default_rng(6 + K)
    words = rng.integers(0, 65536, size=16 * K, dtype=np.uint16)
    tile = oracle.decode_tile(words, K, M)
    pos = [oracle.tile_position(t) for t in range(256)]
    seq = np.array([oracle.f16_to_double(tile[q, r]) for (r, q) in pos])
    vals = oracle.f16_bits_to_f64(np.array([oracle.codebook_f16(s, M) for s in range(65536)],
                                           dtype=np.uint16))
    s0 = oracle.tile_state(words, K, 0)
    assert _viterbi_tailbiting(vals, seq, K, s0) == 0.0
    bad = seq.copy()
    bad[100] += 1e-3
    assert _viterbi_tailbiting(vals, bad, K, s0) > 0.0


def test_hand_encoded_tile_any_width():
    """Encode a random state path that closes on itself by construction (the
    stream bits are the path), for every K, and decode it back."""
    rng = np.random.default_rng(8)
    for K in (2, 3, 4):
        nbits = 256 * K
        bits = rng.integers(0, 2, size=nbits)
        words = np.zeros(16 * K, dtype=np.uint16)
        for p in range(nbits):
            words[p // 16] |= np.uint16(bits[p] << (p % 16))
        for t in (0, 1, 2, 77, 254, 255):
            expect = sum(int(bits[(t * K + b) % nbits]) << b for b in range(16))
            assert oracle.tile_state(words, K, t) == expect


def test_decode_dense_layout_and_side_vectors():
    rng = np.random.default_rng(9)
    K, fin, fout = 3, 32, 48
    codes = rng.integers(0, 65536, size=(fin // 16, fout // 16, 16 * K), dtype=np.uint16)
    dense = oracle.decode_dense(codes, fin, fout, K)
    for i in range(fin // 16):
        for j in range(fout // 16):
            tile = oracle.decode_tile(codes[i, j], K, M)
            assert (dense[16 * i:16 * i + 16, 16 * j:16 * j + 16] == tile).all()
    suh = (1 + 0.1 * rng.standard_normal(fin)).astype(np.float16)
    svh = (1 + 0.1 * rng.standard_normal(fout)).astype(np.float16)
    side = oracle.decode_dense(codes, fin, fout, K, suh=suh.view(np.uint16), svh=svh.view(np.uint16))
    v = dense.view(np.float16).astype(np.float32)
    ref = ((v * suh.astype(np.float32)[:, None]).astype(np.float32)
           * svh.astype(np.float32)[None, :]).astype(np.float16)
    assert (side == ref.view(np.uint16)).all()


# ------------------------------------------------------------ routing


def test_exp_route_accuracy():
    """Within 2 fp32 ulp of exp over [-86, 0]; exact 1 at 0; 0 below -86."""
    xs = np.concatenate([np.linspace(-86, 0, 20001), -np.logspace(-8, 1.9, 2000)]).astype(np.float32)
    for x in xs:
        got = oracle.exp_route(float(x))
        ref = math.exp(float(x))
        ulp = np.spacing(np.float32(ref))
        assert abs(got - ref) <= 2 * ulp, (x, got, ref)
    assert oracle.exp_route(0.0) == 1.0
    assert oracle.exp_route(-86.5) == 0.0 and oracle.exp_route(-math.inf) == 0.0


def test_route_vs_numpy_sort():
    rng = np.random.default_rng(10)
    T, E, k = 64, 288, 8
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[3, 10] = logits[3, 200] = 9.0   # tie -> lower index first
    logits[5, :] = 0.0                     # all tied
    logits[7, 0] = np.nan                  # NaN counts as -inf
    logits[9, :] = -np.inf                 # every logit -inf -> uniform weights
    ids, w, off, pairs = oracle.route(logits, k)
    key = np.where(np.isnan(logits), -np.inf, logits)
    for t in range(T):
        order = np.lexsort((np.arange(E), -key[t]))[:k]
        assert (ids[t] == order).all()
        sel = key[t, order].astype(np.float64)
        if np.isneginf(sel[0]):
            ref = np.full(k, 1.0 / k)
        else:
            ex = np.exp(sel - sel[0])
            ref = ex / ex.sum()
        assert np.allclose(w[t], ref, rtol=1e-6, atol=0)
        assert abs(float(np.float32(w[t]).sum()) - 1.0) <= k * 2**-23
    assert list(ids[3, :2]) == [10, 200]
    assert list(ids[5]) == list(range(k))
    assert 0 not in ids[7] or np.isnan(logits[7]).sum() > E - k
    # segment tables == stable sort by expert (numpy) and bincount prefix
    flat = ids.ravel()
    assert (pairs == np.argsort(flat, kind="stable")).all()
    assert (off == np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))])).all()


def test_route_invariants_zipf():
    from trellis_quantized_moe_exl3_gb300 import synth
    logits = synth.router_logits(5, 512, 288, "zipf")
    ids, w, off, pairs = oracle.route(logits, 8)
    for t in range(512):
        assert len(set(ids[t])) == 8
    assert off[-1] == 512 * 8 and sorted(pairs) == list(range(512 * 8))
    for e in range(288):
        seg = pairs[off[e]:off[e + 1]]
        assert (np.diff(seg) > 0).all() and (ids.ravel()[seg] == e).all()
    counts = np.diff(off)
    assert counts.max() > 5 * counts.mean()   # skewed popularity


# ------------------------------------------------------------ layer


def _small_layer(seed, E=6, H=64, I=32, K=(2, 3, 4), fp8=False, shared=False):
    rng = np.random.default_rng(seed)
    codes, suh, svh = [], [], []
    for p in range(3):
        i, o = (I, H) if p == 2 else (H, I)
        codes.append(rng.integers(0, 65536, size=(E, i // 16, o // 16, 16 * K[p]), dtype=np.uint16))
        suh.append((1 + 0.1 * rng.standard_normal((E, i))).astype(np.float16).view(np.uint16))
        svh.append((1 + 0.1 * rng.standard_normal((E, o))).astype(np.float16).view(np.uint16))
    sw = None
    if shared:
        sw = [rng.standard_normal(((I, H) if p == 2 else (H, I))).astype(np.float16).view(np.uint16)
              for p in range(3)]
    return oracle.Layer(E, H, I, K, codes, suh, svh, fp8_round=fp8, shared_w=sw), codes, suh, svh, sw


@pytest.mark.parametrize("fp8,shared", [(False, False), (True, True)])
def test_layer_vs_numpy_dense_reference(fp8, shared):
    """Oracle layer == numpy matmul on decode_dense weights (fp64)."""
    E, H, I, K, T, k = 6, 64, 32, (2, 3, 4), 5, 2
    L, codes, suh, svh, sw = _small_layer(1, E, H, I, K, fp8, shared)
    rng = np.random.default_rng(2)
    x = rng.standard_normal((T, H)).astype(np.float16).view(np.uint16)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    y = L.forward(x, False, logits, k)
    ids, w, _, _ = oracle.route(logits, k)
    xf = x.view(np.float16).astype(np.float64)
    f = lambda a: a.view(np.float16).astype(np.float64)
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            W = [f(oracle.decode_dense(codes[p][e], *((I, H) if p == 2 else (H, I)), K[p],
                                       fp8_round=fp8)) for p in range(3)]
            g = ((xf[t] * f(suh[0][e])) @ W[0]) * f(svh[0][e])
            u = ((xf[t] * f(suh[1][e])) @ W[1]) * f(svh[1][e])
            h = g / (1 + np.exp(-g)) * u
            ref[t] += float(w[t, j]) * (((h * f(suh[2][e])) @ W[2]) * f(svh[2][e]))
        if shared:
            g = xf[t] @ f(sw[0])
            u = xf[t] @ f(sw[1])
            ref[t] += (g / (1 + np.exp(-g)) * u) @ f(sw[2])
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-9 * np.abs(ref).max())


def test_layer_closed_form_zero_codes():
    """All-zero codes make every weight 1.84375; unit side vectors; top_k = 1
    gives w = 1.  Then g_o = u_o = 1.84375 * sum(x) =: G for every o,
    h = silu(G) * G, and y_o = 1.84375 * I * h for every output o."""
    E, H, I, T = 3, 48, 32, 4
    codes = [np.zeros((E, (I if p == 2 else H) // 16, (H if p == 2 else I) // 16, 32), np.uint16)
             for p in range(3)]
    one = np.uint16(0x3C00)
    suh = [np.full((E, I if p == 2 else H), one, np.uint16) for p in range(3)]
    svh = [np.full((E, H if p == 2 else I), one, np.uint16) for p in range(3)]
    L = oracle.Layer(E, H, I, (2, 2, 2), codes, suh, svh)
    rng = np.random.default_rng(3)
    x = (0.05 * rng.standard_normal((T, H))).astype(np.float16)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    y = L.forward(x.view(np.uint16), False, logits, 1)
    for t in range(T):
        G = 1.84375 * x[t].astype(np.float64).sum()
        h = G / (1 + math.exp(-G)) * G
        assert np.allclose(y[t], 1.84375 * I * h, rtol=1e-13)


def test_rmsnorm_closed_form():
    x = np.full(64, 3.0)
    out = oracle.rmsnorm_row(x, 1e-6)
    assert np.allclose(out, 3.0 / math.sqrt(9.0 + 1e-6), rtol=1e-15)


# ------------------------------------------------------------ Hadamard (format v2)


def _sylvester128():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    return scipy_linalg.hadamard(128).astype(np.float64) / math.sqrt(128.0)


def test_hadamard128_vs_scipy_and_invariants():
    """The 128x128 matrix equals scipy's Sylvester Hadamard matrix divided by
    sqrt(128); it is symmetric, orthogonal (so its own inverse) and maps the
    all-ones vector to sqrt(128) e_0."""
    ref = _sylvester128()
    got = np.array([[oracle.hadamard128_entry(i, j) for j in range(128)] for i in range(128)])
    assert np.allclose(got, ref, rtol=0, atol=1e-16)
    assert np.array_equal(got, got.T)
    assert np.allclose(got @ got, np.eye(128), rtol=0, atol=1e-14)
    ones = got @ np.ones(128)
    assert abs(ones[0] - math.sqrt(128.0)) < 1e-13 and np.abs(ones[1:]).max() < 1e-13


def test_hadamard_blocks_vs_numpy():
    """v . Hb on three 128-blocks equals numpy's block-by-block product with
    the scipy matrix, and preserves the Euclidean norm."""
    ref = _sylvester128()
    v = np.random.default_rng(11).standard_normal(384)
    got = oracle.hadamard_blocks(v)
    want = (v.reshape(3, 128) @ ref).ravel()
    assert np.allclose(got, want, rtol=0, atol=1e-13)
    assert abs(np.linalg.norm(got) - np.linalg.norm(v)) < 1e-12 * np.linalg.norm(v)


@pytest.mark.parametrize("fp8", [False, True])
def test_layer_hadamard_vs_numpy_dense_reference(fp8):
    """Format v2 layer == numpy matmul with the effective weights
    diag(suh) Hb V Hb diag(svh), Hb built from scipy's Sylvester matrix."""
    E, H, I, K, T, k = 4, 256, 128, (2, 3, 4), 3, 2
    _, codes, suh, svh, _ = _small_layer(5, E, H, I, K, fp8, False)
    L = oracle.Layer(E, H, I, K, codes, suh, svh, fp8_round=fp8, hadamard=True)
    rng = np.random.default_rng(6)
    x = rng.standard_normal((T, H)).astype(np.float16).view(np.uint16)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    y = L.forward(x, False, logits, k)
    ids, w, _, _ = oracle.route(logits, k)
    xf = x.view(np.float16).astype(np.float64)
    f = lambda a: a.view(np.float16).astype(np.float64)
    Hs = _sylvester128()
    hb = lambda n: np.kron(np.eye(n // 128), Hs)
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            W = []
            for p in range(3):
                fi, fo = (I, H) if p == 2 else (H, I)
                V = f(oracle.decode_dense(codes[p][e], fi, fo, K[p], fp8_round=fp8))
                W.append(np.diag(f(suh[p][e])) @ hb(fi) @ V @ hb(fo) @ np.diag(f(svh[p][e])))
            g = xf[t] @ W[0]
            u = xf[t] @ W[1]
            h = g / (1 + np.exp(-g)) * u
            ref[t] += float(w[t, j]) * (h @ W[2])
    assert np.allclose(y, ref, rtol=1e-10, atol=1e-9 * np.abs(ref).max())


def test_layer_hadamard_closed_form_zero_codes():
    """Zero codes (every weight c = 1.84375), unit side vectors, top_k = 1.
    The rotation concentrates a constant row on the first entry of each
    128-block (Hb 1 = sqrt(128) e_0 per block), so g_o = u_o = G = 128 c S
    with S = sum_b x[128 b] when o = 0 (mod 128) and 0 otherwise; the down
    input h . Hb is then constant (h_0 / sqrt(128)), and y_o = c I silu(G) G
    when o = 0 (mod 128), 0 otherwise."""
    E, H, I, T = 2, 256, 256, 3
    c = 1.84375
    codes = [np.zeros((E, (I if p == 2 else H) // 16, (H if p == 2 else I) // 16, 32), np.uint16)
             for p in range(3)]
    one = np.uint16(0x3C00)
    suh = [np.full((E, I if p == 2 else H), one, np.uint16) for p in range(3)]
    svh = [np.full((E, H if p == 2 else I), one, np.uint16) for p in range(3)]
    L = oracle.Layer(E, H, I, (2, 2, 2), codes, suh, svh, hadamard=True)
    rng = np.random.default_rng(7)
    x = (0.05 * rng.standard_normal((T, H))).astype(np.float16)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    y = L.forward(x.view(np.uint16), False, logits, 1)
    for t in range(T):
        S = x[t].astype(np.float64)[::128].sum()
        G = 128 * c * S
        want = np.zeros(H)
        want[::128] = c * I * (G / (1 + math.exp(-G))) * G
        assert np.allclose(y[t], want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


# ------------------------------------------------------------ coded shared expert


def test_layer_shared_coded_vs_numpy_dense_reference():
    """A trellis-coded shared expert stored after the routed experts (index E
    of the code arrays) adds expert_E(x) with weight 1 to every token: numpy
    matmul on decode_dense weights (fp64)."""
    E, H, I, K, T, k = 5, 64, 32, (3, 3, 2), 4, 2
    _, codes, suh, svh, _ = _small_layer(8, E + 1, H, I, K, False, False)
    L = oracle.Layer(E, H, I, K, codes, suh, svh, shared_coded=True)
    rng = np.random.default_rng(9)
    x = rng.standard_normal((T, H)).astype(np.float16).view(np.uint16)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    y = L.forward(x, False, logits, k)
    ids, w, _, _ = oracle.route(logits, k)
    assert ids.max() < E
    xf = x.view(np.float16).astype(np.float64)
    f = lambda a: a.view(np.float16).astype(np.float64)

    def expert(e, xt):
        W = [f(oracle.decode_dense(codes[p][e], *((I, H) if p == 2 else (H, I)), K[p]))
             for p in range(3)]
        g = ((xt * f(suh[0][e])) @ W[0]) * f(svh[0][e])
        u = ((xt * f(suh[1][e])) @ W[1]) * f(svh[1][e])
        h = g / (1 + np.exp(-g)) * u
        return ((h * f(suh[2][e])) @ W[2]) * f(svh[2][e])

    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            ref[t] += float(w[t, j]) * expert(ids[t, j], xf[t])
        ref[t] += expert(E, xf[t])
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-9 * np.abs(ref).max())


def test_layer_shared_coded_closed_form_zero_codes():
    """Zero codes for every expert, unit side vectors, top_k = 1: the routed
    expert (weight 1) and the shared one compute the same closed form
    (test_layer_closed_form_zero_codes), so y_o = 2 * 1.84375 * I * h."""
    E, H, I, T = 3, 48, 32, 4
    codes = [np.zeros((E + 1, (I if p == 2 else H) // 16, (H if p == 2 else I) // 16, 32), np.uint16)
             for p in range(3)]
    one = np.uint16(0x3C00)
    suh = [np.full((E + 1, I if p == 2 else H), one, np.uint16) for p in range(3)]
    svh = [np.full((E + 1, H if p == 2 else I), one, np.uint16) for p in range(3)]
    L = oracle.Layer(E, H, I, (2, 2, 2), codes, suh, svh, shared_coded=True)
    rng = np.random.default_rng(3)
    x = (0.05 * rng.standard_normal((T, H))).astype(np.float16)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    y = L.forward(x.view(np.uint16), False, logits, 1)
    for t in range(T):
        G = 1.84375 * x[t].astype(np.float64).sum()
        h = G / (1 + math.exp(-G)) * G
        assert np.allclose(y[t], 2 * 1.84375 * I * h, rtol=1e-13)


# ------------------------------------------------------------ per-expert widths


def _mixed_layer(seed, E, H, I, shared_coded=False):
    """Flat per-projection code arrays, each expert at its own width."""
    rng = np.random.default_rng(seed)
    n = E + int(shared_coded)
    ek = rng.integers(2, 5, size=(n, 3)).astype(np.uint8)
    codes, per = [], []
    for p in range(3):
        fi, fo = (I, H) if p == 2 else (H, I)
        parts = [rng.integers(0, 65536, size=(fi // 16) * (fo // 16) * 16 * int(ek[e, p]),
                              dtype=np.uint16) for e in range(n)]
        per.append(parts)
        codes.append(np.concatenate(parts))
    suh = [(1 + 0.1 * rng.standard_normal((n, I if p == 2 else H))).astype(np.float16).view(np.uint16)
           for p in range(3)]
    svh = [(1 + 0.1 * rng.standard_normal((n, H if p == 2 else I))).astype(np.float16).view(np.uint16)
           for p in range(3)]
    return ek, codes, per, suh, svh


@pytest.mark.parametrize("shared_coded", [False, True])
def test_layer_mixed_widths_vs_numpy_dense_reference(shared_coded):
    """Every expert and projection at its own width (codes back to back):
    numpy matmul on each expert's decode_dense weights at its width."""
    E, H, I, T, k = 5, 64, 32, 4, 2
    ek, codes, per, suh, svh = _mixed_layer(12, E, H, I, shared_coded)
    L = oracle.Layer(E, H, I, (2, 2, 2), codes, suh, svh, shared_coded=shared_coded, expert_K=ek)
    rng = np.random.default_rng(13)
    x = rng.standard_normal((T, H)).astype(np.float16).view(np.uint16)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    y = L.forward(x, False, logits, k)
    ids, w, _, _ = oracle.route(logits, k)
    xf = x.view(np.float16).astype(np.float64)
    f = lambda a: a.view(np.float16).astype(np.float64)

    def expert(e, xt):
        W = [f(oracle.decode_dense(per[p][e].reshape(-1), *((I, H) if p == 2 else (H, I)),
                                   int(ek[e, p]))) for p in range(3)]
        g = ((xt * f(suh[0][e])) @ W[0]) * f(svh[0][e])
        u = ((xt * f(suh[1][e])) @ W[1]) * f(svh[1][e])
        h = g / (1 + np.exp(-g)) * u
        return ((h * f(suh[2][e])) @ W[2]) * f(svh[2][e])

    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            ref[t] += float(w[t, j]) * expert(ids[t, j], xf[t])
        if shared_coded:
            ref[t] += expert(E, xf[t])
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-9 * np.abs(ref).max())


def test_layer_uniform_width_table_equals_plain_layer():
    """A width table that gives every expert the projection's width is the
    plain layout ([E][in/16][out/16][16K], expert e at e times the stride)."""
    E, H, I, K, T, k = 4, 64, 32, (3, 3, 4), 3, 2
    L0, codes, suh, svh, _ = _small_layer(14, E, H, I, K, False, False)
    ek = np.tile(np.array(K, np.uint8), (E, 1))
    L1 = oracle.Layer(E, H, I, (2, 2, 2), [c.reshape(-1) for c in codes], suh, svh, expert_K=ek)
    rng = np.random.default_rng(15)
    x = rng.standard_normal((T, H)).astype(np.float16).view(np.uint16)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    assert np.array_equal(L0.forward(x, False, logits, k), L1.forward(x, False, logits, k))


# ------------------------------------------------------------ FP8 activations (NEXT row 2)


def _torch_quantize_row(a):
    """Independent restatement through torch's float8_e4m3fn conversion."""
    a32 = torch.tensor(np.asarray(a, np.float64), dtype=torch.float32)
    amax = a32.abs().max()
    if float(amax) == 0.0:
        return np.zeros(a32.numel())
    s = amax / torch.tensor(448.0, dtype=torch.float32)
    q = (a32 / s).to(torch.float8_e4m3fn).to(torch.float64)
    return (q * s.to(torch.float64)).numpy()


@pytest.mark.parametrize("scale", [1.0, 1e-3, 37.5])
def test_quantize_row_e4m3_vs_torch(scale):
    """Per-row E4M3 quantisation equals torch's float8_e4m3fn conversion of
    the fp32 quotient a / s, s = fp32(amax / 448), on rows with values down
    in the E4M3 subnormal range."""
    rng = np.random.default_rng(21)
    a = scale * rng.standard_normal(4096) * np.exp(rng.uniform(-8, 0, 4096))
    assert np.array_equal(oracle.quantize_row_e4m3(a), _torch_quantize_row(a))


def test_quantize_row_e4m3_closed_forms():
    """Powers of two below the row maximum quantise without error relative to
    the scale (a_i / s = 448 * 2^-k, exact in E4M3); a zero row stays zero."""
    a = np.array([1.0, -0.5, 0.25, -0.125, 2.0 ** -6, -1.0])
    s = np.float32(1.0) / np.float32(448.0)
    want = np.array([448.0, -224.0, 112.0, -56.0, 7.0, -448.0]) * np.float64(s)
    assert np.array_equal(oracle.quantize_row_e4m3(a), want)
    assert np.array_equal(oracle.quantize_row_e4m3(np.zeros(8)), np.zeros(8))


def test_layer_fp8_activations_vs_numpy_dense_reference():
    """With FP8 activations every projection multiplies the quantised input
    row (after suh): numpy matmul with rows quantised through torch."""
    E, H, I, K, T, k = 5, 64, 32, (4, 4, 4), 3, 2
    L0, codes, suh, svh, _ = _small_layer(22, E, H, I, K, True, False)
    L = oracle.Layer(E, H, I, K, codes, suh, svh, fp8_round=True, act_fp8=True)
    rng = np.random.default_rng(23)
    x = rng.standard_normal((T, H)).astype(np.float16).view(np.uint16)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    y = L.forward(x, False, logits, k)
    ids, w, _, _ = oracle.route(logits, k)
    xf = x.view(np.float16).astype(np.float64)
    f = lambda a: a.view(np.float16).astype(np.float64)
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            W = [f(oracle.decode_dense(codes[p][e], *((I, H) if p == 2 else (H, I)), K[p],
                                       fp8_round=True)) for p in range(3)]
            g = (_torch_quantize_row(xf[t] * f(suh[0][e])) @ W[0]) * f(svh[0][e])
            u = (_torch_quantize_row(xf[t] * f(suh[1][e])) @ W[1]) * f(svh[1][e])
            h = g / (1 + np.exp(-g)) * u
            ref[t] += float(w[t, j]) * ((_torch_quantize_row(h * f(suh[2][e])) @ W[2]) * f(svh[2][e]))
    assert np.allclose(y, ref, rtol=1e-9, atol=1e-9 * np.abs(ref).max())
    # and it differs from the unquantised layer by the E4M3 rounding (~1-4 %)
    y0 = L0.forward(x, False, logits, k)
    rel = np.linalg.norm(y - y0) / np.linalg.norm(y0)
    assert 1e-3 < rel < 0.1
