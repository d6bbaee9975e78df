"""Pins for the oracle's Cassandra split and MoE routing/combine.

Fixed by: the lossless invariant (speculation + verification = every original
bit) over all 65,536 bf16 patterns, the unary code definition, brute-force
Wanda selection and routing on tiny inputs, and the dense-sum identity of a
top-k MoE.
"""
import numpy as np
import pytest

from oracle import cassandra as cs
from oracle import moe, numerics, ternary
from quantized_gemv_unpack_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _small_case(seed=2, N=24, K=256, R=16):
    g = synth.rng(seed)
    W = synth.to_bf16_bits(synth.student_t4(g, (N, K)))
    X, chans = synth.calibration_bf16(g, R, K)
    return W, X


def test_invariant_all_bf16_patterns():
    """Every bf16 bit pattern survives split + merge, both as a kept and as a pruned value."""
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    K = 32
    X = synth.to_bf16_bits(np.ones((2, K), np.float32))
    # kept role: the pattern in column 0, +0 elsewhere (it outscores or ties with a lower column)
    Wk = np.zeros((65536, K), np.uint16)
    Wk[:, 0] = allp
    buf, meta = cs.pack(Wk, X)
    assert meta["keep"][:, 0].all()
    assert np.array_equal(cs.reconstruct(buf, meta), Wk)
    # pruned role: NaN (score +inf) in columns 0..15 fills the kept half, the pattern sits in column 31
    Wp = np.zeros((65536, K), np.uint16)
    Wp[:, :16] = 0x7FC0
    Wp[:, 31] = allp
    buf, meta = cs.pack(Wp, X)
    assert not meta["keep"][:, 31].any()
    assert np.array_equal(cs.reconstruct(buf, meta), Wp)
    # the field-level split is a bijection on all patterns
    S, E, M = numerics.bf16_fields(allp)
    merged = numerics.bf16_from_fields(S, E, ((M >> 4) << 4) | (M & 0xF))
    assert np.array_equal(merged, allp)


def test_bitmap_keeps_half_and_wanda_is_top_half():
    W, X = _small_case()
    N, K = W.shape
    buf, meta = cs.pack(W, X)
    keep = meta["keep"]
    assert (keep.sum(axis=1) == K // 2).all()
    # brute force: Wanda score with explicit loops
    xf = numerics.bf16_bits_to_f64(X)
    c = [sum(float(xf[r, j]) ** 2 for r in range(X.shape[0])) ** 0.5 for j in range(K)]
    wf = numerics.bf16_bits_to_f64(W)
    for n in range(N):
        score = [abs(float(wf[n, j])) * c[j] for j in range(K)]
        order = sorted(range(K), key=lambda j: (-score[j], j))
        assert set(order[: K // 2]) == set(np.flatnonzero(keep[n]))


def test_wanda_uses_activation_norm_not_magnitude_alone():
    # an outlier channel (x20 in calibration) keeps a small weight that magnitude pruning would drop
    K = 64
    Wf = np.full((1, K), 0.01, np.float32)
    Wf[0, 5] = 0.001
    W = synth.to_bf16_bits(Wf)
    X = np.ones((4, K), np.float32)
    X[:, 5] = 20.0
    X[:, 6:] = 0.5                                  # columns 6.. score 0.005 < 0.02 (col 5)
    keep = cs.wanda_keep(W, cs.column_norms(synth.to_bf16_bits(X)))
    assert keep[0, 5]
    # ties (equal scores) keep the lower column: columns 6.. all score the same
    assert keep[0].sum() == K // 2
    assert keep[0, 6:6 + (K // 2 - 6)].all() and not keep[0, 6 + (K // 2 - 6):].any()


def test_unary_code_definition():
    ranks = np.array([0, 2, 1, 0, 5])
    bits = cs.unary_bits(ranks)
    assert "".join(map(str, bits)) == "1" + "001" + "01" + "1" + "000001"
    assert np.array_equal(cs.unary_decode(bits, 5), ranks)
    g = synth.rng(1)
    r = g.integers(0, 12, 3000)
    assert np.array_equal(cs.unary_decode(cs.unary_bits(r), 3000), r)
    words = cs.bits_to_words(cs.unary_bits(r))
    assert np.array_equal(cs.words_to_bits(words)[: len(cs.unary_bits(r))], cs.unary_bits(r))


def test_stream_properties():
    W, X = _small_case(N=40, K=512)
    buf, meta = cs.pack(W, X)
    N, K = W.shape
    Sk, Ek, m_hi, m_lo, pruned = cs.split_values(W, meta["keep"])
    codebook, rank_of, counts = cs.exponent_codebook(Ek)
    # the most frequent exponent gets the one-bit code "1"
    assert codebook[0] == np.argmax(counts) and rank_of[codebook[0]] == 0
    assert list(counts[codebook]) == sorted(counts[codebook], reverse=True)
    bm, sm, stream, rowstart, cb, pr, mlo = cs._sections(buf, meta)
    assert np.array_equal(cb[: meta["n_symbols"]], codebook)
    for n in range(N):
        bits = cs.words_to_bits(stream[rowstart[n]:rowstart[n + 1]])
        ones = np.flatnonzero(bits)
        assert len(ones) == K // 2                   # one codeword per kept value
        assert ones[-1] + 1 == int((rank_of[Ek[n]] + 1).sum())  # total bits = sum(rank + 1); ends in 1
        assert (rowstart[n] % 4) == 0                # rows start 16-byte aligned


def test_draft_truncates_and_zero_pads():
    W, X = _small_case()
    buf, meta = cs.pack(W, X)
    D = cs.draft(buf, meta)
    keep = meta["keep"]
    assert (D[~keep] == 0).all()
    assert np.array_equal(D[keep], W[keep] & np.uint16(0xFFF0))   # low 4 mantissa bits zero-filled
    assert np.array_equal(cs.reconstruct(buf, meta), W)
    assert cs.speculation_bytes(meta) + cs.verification_bytes(meta) <= meta["total"]


def test_worked_example_through_the_split():
    # 0.15625 = 0 01111100 0100000: its high mantissa bits 010 carry the whole value
    v = int("0011111000100000", 2)
    Wf = np.full((1, 32), 0.001, np.float32)
    W = synth.to_bf16_bits(Wf)
    W[0, 3] = v
    X = synth.to_bf16_bits(np.ones((2, 32), np.float32))
    buf, meta = cs.pack(W, X)
    assert meta["keep"][0, 3]
    assert cs.draft(buf, meta)[0, 3] == v
    assert numerics.bf16_bits_to_f64(cs.draft(buf, meta)[0, 3:4])[0] == 0.15625


def test_corrupt_stream_is_rejected():
    W, X = _small_case(N=4, K=128)
    buf, meta = cs.pack(W, X)
    b = bytearray(buf)
    o = meta["offsets"][2]
    b[o:o + 4 * int(meta["stream_words"])] = bytes(4 * int(meta["stream_words"]))  # no codeword ends
    with pytest.raises(ValueError):
        cs.draft(bytes(b), meta)


# ----------------------------------------------------------------------------- MoE

def test_exponent_stats_closed_forms():
    """Entropy and mean unary length of the kept exponents ("Cassandra" 3.3) on distributions
    whose values follow from the definitions: four equally frequent exponents give H = 2 bit and
    ranks 0..3, i.e. codes of 1..4 bits, mean 2.5; counts {2, 1, 1} give H = 1.5 bit and lengths
    1 (twice), 2, 3 (equal counts: smaller exponent first), mean 7/4; one exponent gives H = 0 and
    the one-bit code."""
    from oracle import cassandra as c
    H, L = c.exponent_stats(np.array([120, 121, 122, 123] * 5, dtype=np.uint8))
    assert H == pytest.approx(2.0, abs=1e-12) and L == pytest.approx(2.5, abs=1e-12)
    H, L = c.exponent_stats(np.array([130, 127, 127, 125], dtype=np.uint8))
    assert H == pytest.approx(1.5, abs=1e-12) and L == pytest.approx(1.75, abs=1e-12)
    # which of the two single exponents gets rank 1 does not change the mean, but the order does:
    _, rank_of, _ = c.exponent_codebook(np.array([130, 127, 127, 125], dtype=np.uint8))
    assert (rank_of[127], rank_of[125], rank_of[130]) == (0, 1, 2)
    H, L = c.exponent_stats(np.full(7, 126, dtype=np.uint8))
    assert H == 0.0 and L == 1.0


def test_exponent_stats_source_coding_bound():
    """The unary code of the frequency rank is a prefix code, so its mean length is at least the
    entropy (source coding theorem); for a dyadic geometric distribution p_r = 2^-(r+1) the bound
    is met with equality except for the last symbol, which needs one bit more than the tail."""
    from oracle import cassandra as c
    g = np.random.default_rng(5)
    for _ in range(20):
        E = g.choice(np.arange(110, 140), size=500, p=g.dirichlet(np.ones(30)))
        H, L = c.exponent_stats(E.astype(np.uint8))
        assert L >= H - 1e-12
    counts = [16, 8, 4, 2, 1, 1]                       # p = 1/2, 1/4, 1/8, 1/16, 1/32, 1/32
    E = np.concatenate([np.full(n, 120 + i) for i, n in enumerate(counts)]).astype(np.uint8)
    H, L = c.exponent_stats(E)
    assert H == pytest.approx(1 / 2 + 2 / 4 + 3 / 8 + 4 / 16 + 2 * 5 / 32, abs=1e-12)
    assert L == pytest.approx((16 * 1 + 8 * 2 + 4 * 3 + 2 * 4 + 5 + 6) / 32, abs=1e-12)
    assert L - H == pytest.approx(1 / 32, abs=1e-12)


def test_route_matches_brute_force_and_ties():
    g = synth.rng(8)
    L = synth.router_logits(g, 5, 16)
    L[2, 3] = L[2, 9] = 4.0                                  # a tie at the top
    idx, p = moe.route(L, 4)
    for t in range(5):
        ref = sorted(range(16), key=lambda e: (-float(L[t, e]), e))[:4]
        assert list(idx[t]) == ref
    assert list(idx[2, :2]) == [3, 9]
    assert np.allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    assert (np.diff(p, axis=1) <= 0).all()
    # softmax of the selected logits, written out by hand for one token
    sel = [float(L[0, e]) for e in idx[0]]
    z = [np.exp(v - max(sel)) for v in sel]
    assert np.allclose(p[0], np.array(z) / sum(z), rtol=1e-15)


def test_moe_equals_dense_sum_with_zero_weights():
    g = synth.rng(10)
    E, H, I, topk = 6, 128, 128, 2
    experts = []
    for e in range(E):
        mats = []
        for shape in [(I, H), (I, H), (H, I)]:
            q, _, s16 = ternary.quantize(synth.student_t4(g, shape))
            mats.append(ternary.dequant(q, s16))
        experts.append(mats)
    x = numerics.bf16_bits_to_f64(synth.activations_bf16(g, (1, H)))
    L = synth.router_logits(g, 1, E)
    y, idx, p, parts = moe.moe(x, L, topk, lambda e: experts[e])
    dense = np.zeros(H)
    for e in range(E):
        wg, wu, wd = experts[e]
        gg = wg @ x[0]
        h = gg * (1.0 / (1.0 + np.exp(-gg))) * (wu @ x[0])
        weight = p[0, list(idx[0]).index(e)] if e in idx[0] else 0.0
        dense += weight * (wd @ h)
    assert np.allclose(y[0], dense, rtol=1e-12, atol=1e-14)


def test_silu_closed_forms():
    assert moe.silu(np.array([0.0]))[0] == 0.0
    assert moe.silu(np.array([40.0]))[0] == pytest.approx(40.0, rel=1e-15)
    assert moe.silu(np.array([-1.0]))[0] == pytest.approx(-1.0 / (1.0 + np.e), rel=1e-15)
