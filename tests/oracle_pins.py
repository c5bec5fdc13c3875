"""Checks that pin the CPU oracle to what the pages and the arithmetic fix.

Every function takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch, so the same checks run against the real oracle
(test_oracle_pins.py) and against deliberately broken builds of it
(test_oracle_mutants.py, which shows each planted mistake is caught).

Pins, by source:
  * "Chapter 13 - The QKV + gate matvec family", Figure 13.1: the 2x2 matvec.
  * "Chapter 6 - The kquant family on the reference lane":
      Figure 6.1 (block bytes / bits per element), sections 6.5, 6.6, 6.8
      (byte counts), section 6.3 (hand-packed Q4_K block: scale bytes, the
      sub-block 5 round trip, three dequantized elements), the packing
      equations of section 6.3 (inverted here, checked as a bijection),
      section 6.4 (Q5_K = Q4_K plus a fifth bit; Q6_K codes minus 32 times a
      per-16 int8 scale and an f16 d stored last).
  * IEEE 754 binary16 (the f16 header fields), checked against numpy.
  * Arithmetic facts: one-block brute force (W e_j is column j), single
    rounding of each f32 weight, f64 dot products against numpy's matmul,
    exact scaling by powers of two.
"""
from __future__ import annotations

import numpy as np

import _golden as G

Q4_K, Q5_K, Q6_K = 12, 13, 14


# ---------------------------------------------------------------- helpers
def pack_scale_field(sc, m):
    """Pack eight 6-bit scales and mins into the 12-byte field, following the
    packing equations written out in section 6.3 (the inverse of the
    unpacking rule the oracle implements)."""
    s = np.zeros(12, dtype=np.uint8)
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    return s


def f16_bits(v):
    return int(np.array(v, dtype=np.float16).view(np.uint16))


def q45_block(fmt, d, dmin, sc, m, qs, qh=None):
    bb = 144 if fmt == Q4_K else 176
    b = np.zeros(bb, dtype=np.uint8)
    b[0:2] = np.array([f16_bits(d)], dtype=np.uint16).view(np.uint8)
    b[2:4] = np.array([f16_bits(dmin)], dtype=np.uint16).view(np.uint8)
    b[4:16] = pack_scale_field(sc, m)
    if fmt == Q4_K:
        b[16:144] = qs
    else:
        b[16:48] = qh if qh is not None else 0
        b[48:176] = qs
    return b


def q6_block(d, sc16, ql, qh):
    b = np.zeros(210, dtype=np.uint8)
    b[0:128] = ql
    b[128:192] = qh
    b[192:208] = np.asarray(sc16, dtype=np.int8).view(np.uint8)
    b[208:210] = np.array([f16_bits(d)], dtype=np.uint16).view(np.uint8)
    return b


def worked_block():
    g = G.keyvals("q4k_worked_example.txt")
    b = np.zeros(144, dtype=np.uint8)
    b[0:2] = np.array([int(g["d_bits"], 16)], np.uint16).view(np.uint8)
    b[2:4] = np.array([int(g["dmin_bits"], 16)], np.uint16).view(np.uint8)
    b[4:16] = [int(v, 16) for v in g["scales_hex"].split()]
    b[16 + 0] = int(g["qs_0"], 16)
    b[16 + 32] = int(g["qs_32"], 16)
    return g, b


# ---------------------------------------------------------------- pins
def pin_matvec_2x2(o):
    g = G.keyvals("matvec_2x2.txt")
    W = np.array([G.floats(g["W_row0"]), G.floats(g["W_row1"])], np.float32)
    x = np.array(G.floats(g["x"]), np.float32)
    y, S = o.matvec_f32(W, x)
    assert y[0].tolist() == G.floats(g["y"])
    assert S[0].tolist() == G.floats(g["y"])  # all products positive


def pin_block_geometry(o):
    for name, code, bb, n, bits in G.table("block_geometry.txt"):
        assert o.block_bytes(int(code)) == int(bb), name
        assert o.block_bytes(int(code)) * 8 / int(n) == float(bits), name
    assert o.block_bytes(0) == -1 and o.block_bytes(2) == -1


def pin_byte_counts(o):
    codes = {"Q4_K": Q4_K, "Q5_K": Q5_K, "Q6_K": Q6_K}
    for name, rows, cols, per_row, total, params in G.table(
            "byte_counts.txt"):
        rows, cols = int(rows), int(cols)
        bb = o.block_bytes(codes[name])
        if per_row != "-":
            assert cols // 256 * bb == int(per_row)
        if total != "-":
            assert rows * (cols // 256) * bb == int(total)
        if params != "-":
            assert rows * cols == int(params)


def pin_f16(o):
    g = G.keyvals("q4k_worked_example.txt")
    assert o.f16_to_f32(int(g["d_bits"], 16)) == float(g["d_value"])
    assert o.f16_to_f32(int(g["dmin_bits"], 16)) == float(g["dmin_value"])
    # every binary16 pattern against numpy's own conversion
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([o.f16_to_f32(int(b)) for b in range(0, 65536, 1)],
                   dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def pin_worked_scales(o):
    g, b = worked_block()
    sc, m = G.ints(g["sc"]), G.ints(g["m"])
    for j in range(8):
        assert o.scale_min_k4(b[4:16], j) == (sc[j], m[j]), j
    assert o.scale_min_k4(b[4:16], 5) == (int(g["roundtrip_sc5"]),
                                          int(g["roundtrip_m5"]))
    d, dmin = float(g["d_value"]), float(g["dmin_value"])
    assert [d * sc[j] for j in range(3)] == G.floats(g["eff_scale_0_1_2"])
    assert [dmin * m[j] for j in range(3)] == G.floats(g["eff_min_0_1_2"])
    # the page's packing lines reproduce the printed bytes
    assert list(pack_scale_field(sc, m)) == [
        int(v, 16) for v in g["scales_hex"].split()]


def pin_worked_dequant(o):
    g, b = worked_block()
    out = o.dequant_block(Q4_K, b)
    for key in ("element_0", "element_32", "element_64"):
        idx = int(key.split("_")[1])
        assert out[idx] == np.float32(g[key]), key
    # derived from the same passage: element 96 is the high nibble (3) of
    # qs[32] in sub-block 3, and every zero nibble leaves -dmin*m of its
    # sub-block.
    d, dmin = float(g["d_value"]), float(g["dmin_value"])
    sc, m = G.ints(g["sc"]), G.ints(g["m"])
    assert out[96] == np.float32(d * sc[3] * 3 - dmin * m[3]) == 0.5625
    for e in range(256):
        if e in (0, 32, 64, 96):
            continue
        assert out[e] == np.float32(-dmin * m[e // 32]), e


def pin_scale_bijection(o, n=20000, seed=7):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        sc = rng.integers(0, 64, size=8)
        m = rng.integers(0, 64, size=8)
        s = pack_scale_field(sc, m)
        for j in range(8):
            assert o.scale_min_k4(s, j) == (sc[j], m[j])
    # and every 12-byte field unpacks and re-packs to itself
    for _ in range(n):
        s = rng.integers(0, 256, size=12).astype(np.uint8)
        pairs = [o.scale_min_k4(s, j) for j in range(8)]
        assert list(pack_scale_field([p[0] for p in pairs],
                                     [p[1] for p in pairs])) == list(s)


def _exact_q45(d, dmin, sc, m, codes):
    """Weights in f64 (exact for these magnitudes), rounded once to f32."""
    w = np.array([d * sc[e // 32] * codes[e] - dmin * m[e // 32]
                  for e in range(256)], dtype=np.float64)
    return w.astype(np.float32)


def _q4_codes_to_qs(codes):
    """Place 256 4-bit codes into qs: low nibble of byte 32g+l holds element
    64g+l, high nibble holds 64g+32+l (Figure 6.2 and section 6.2)."""
    qs = np.zeros(128, dtype=np.uint8)
    for g in range(4):
        for l in range(32):
            qs[32 * g + l] = codes[64 * g + l] | (codes[64 * g + 32 + l] << 4)
    return qs


def pin_q4k_single_rounding(o, trials=200, seed=11):
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        d = float(np.float16(rng.uniform(1e-3, 1e-2)))
        dmin = float(np.float16(rng.uniform(1e-3, 1e-2)))
        sc, m = rng.integers(0, 64, 8), rng.integers(0, 64, 8)
        codes = rng.integers(0, 16, 256)
        b = q45_block(Q4_K, d, dmin, sc, m, _q4_codes_to_qs(codes))
        out = o.dequant_block(Q4_K, b)
        ref = _exact_q45(d, dmin, sc, m, codes)
        assert np.array_equal(out.view(np.uint32), ref.view(np.uint32))


def pin_q5k(o, seed=13):
    rng = np.random.default_rng(seed)
    d, dmin = 2.0 ** -5, 2.0 ** -7
    sc, m = rng.integers(0, 64, 8), rng.integers(0, 64, 8)
    qs = rng.integers(0, 256, 128).astype(np.uint8)
    # (1) with every fifth bit clear, Q5_K is the Q4_K block (section 6.4)
    b4 = q45_block(Q4_K, d, dmin, sc, m, qs)
    b5 = q45_block(Q5_K, d, dmin, sc, m, qs, qh=np.zeros(32, np.uint8))
    base = o.dequant_block(Q5_K, b5)
    assert np.array_equal(base, o.dequant_block(Q4_K, b4))
    # (2) all bits set: code 31 everywhere
    b = q45_block(Q5_K, d, dmin, sc, m, np.full(128, 255, np.uint8),
                  qh=np.full(32, 255, np.uint8))
    ref = _exact_q45(d, dmin, sc, m, [31] * 256)
    assert np.array_equal(o.dequant_block(Q5_K, b), ref)
    # (3) one qh bit lifts exactly one weight by 16*d*sc; reading R1 says
    # which one, and the 256 bits cover the 256 weights once each
    seen = set()
    for byte in range(32):
        for bit in range(8):
            qh = np.zeros(32, np.uint8)
            qh[byte] = 1 << bit
            out = o.dequant_block(Q5_K, q45_block(Q5_K, d, dmin, sc, m, qs,
                                                  qh=qh))
            diff = np.nonzero(out != base)[0]
            g, hi = bit // 2, bit % 2
            e = 64 * g + 32 * hi + byte
            assert diff.tolist() == ([e] if sc[e // 32] else []), (byte, bit)
            assert out[e] - base[e] == np.float32(16 * d * sc[e // 32])
            seen.add(e)
    assert seen == set(range(256))


def pin_q6k(o, seed=17):
    rng = np.random.default_rng(seed)
    d = 2.0 ** -5
    sc = np.array([j - 8 if j != 8 else 5 for j in range(16)])  # no zeros
    zero = np.zeros(128, np.uint8), np.zeros(64, np.uint8)
    # (1) all codes 0 -> d*sc*(-32); all codes 63 -> d*sc*31
    base = o.dequant_block(Q6_K, q6_block(d, sc, *zero))
    assert np.array_equal(base, np.array(
        [d * sc[e // 16] * -32 for e in range(256)], np.float32))
    full = o.dequant_block(Q6_K, q6_block(d, sc, np.full(128, 255, np.uint8),
                                          np.full(64, 255, np.uint8)))
    assert np.array_equal(full, np.array(
        [d * sc[e // 16] * 31 for e in range(256)], np.float32))
    # (2) d is the last field: doubling bytes 208..209's value doubles all
    b = q6_block(2 * d, sc, *zero)
    assert np.array_equal(o.dequant_block(Q6_K, b), 2 * base)
    # (3) each ql nibble moves one weight by d*sc, each qh bit pair by 16*d*sc
    # (reading R2 gives the positions); both maps cover all 256 weights
    seen_l, seen_h = set(), set()
    for byte in range(128):
        for nib in range(2):
            ql = np.zeros(128, np.uint8)
            ql[byte] = 1 << (4 * nib)
            out = o.dequant_block(Q6_K, q6_block(d, sc, ql, zero[1]))
            diff = np.nonzero(out != base)[0].tolist()
            h, r = byte // 64, byte % 64
            e = 128 * h + (r % 32) + 32 * (r // 32) + 64 * nib
            assert diff == [e], (byte, nib, diff)
            assert out[e] - base[e] == np.float32(d * sc[e // 16])
            seen_l.add(e)
    for byte in range(64):
        for pair in range(4):
            qh = np.zeros(64, np.uint8)
            qh[byte] = 1 << (2 * pair)
            out = o.dequant_block(Q6_K, q6_block(d, sc, zero[0], qh))
            diff = np.nonzero(out != base)[0].tolist()
            h, l = byte // 32, byte % 32
            e = 128 * h + l + 32 * pair
            assert diff == [e], (byte, pair, diff)
            assert out[e] - base[e] == np.float32(16 * d * sc[e // 16])
            seen_h.add(e)
    assert seen_l == set(range(256)) and seen_h == set(range(256))
    # (4) int8 scales: a one-hot scale leaves only its 16 weights nonzero
    codes_ql = rng.integers(0, 256, 128).astype(np.uint8)
    codes_qh = rng.integers(0, 256, 64).astype(np.uint8)
    for j in range(16):
        one = np.zeros(16, int)
        one[j] = -3
        out = o.dequant_block(Q6_K, q6_block(d, one, codes_ql, codes_qh))
        nz = set(np.nonzero(out)[0].tolist())
        assert nz <= set(range(16 * j, 16 * j + 16)), j


def _random_block(fmt, rng):
    bb = {Q4_K: 144, Q5_K: 176, Q6_K: 210}[fmt]
    b = rng.integers(0, 256, bb).astype(np.uint8)
    if fmt == Q6_K:
        b[208:210] = np.array([f16_bits(rng.uniform(1e-3, 1e-2))],
                              np.uint16).view(np.uint8)
    else:
        b[0:4] = np.array([f16_bits(rng.uniform(1e-3, 1e-2)),
                           f16_bits(rng.uniform(1e-3, 1e-2))],
                          np.uint16).view(np.uint8)
    return b


def pin_one_block_brute_force(o, seed=19):
    """rows=1, cols=256: y for x = e_j is weight j of the block (all j)."""
    rng = np.random.default_rng(seed)
    eye = np.eye(256, dtype=np.float32)
    for fmt in (Q4_K, Q5_K, Q6_K):
        b = _random_block(fmt, rng)
        y, S = o.matvec(fmt, b, 1, 256, eye)
        w = o.dequant_block(fmt, b).astype(np.float64)
        assert np.array_equal(y[:, 0], w)
        assert np.array_equal(S[:, 0], np.abs(w))


def pin_matvec_vs_numpy(o, seed=23):
    """The f64 dot products agree with numpy's matmul of the dequantized
    rows; y(2x) is exactly 2 y(x); a row subset equals the full result."""
    rng = np.random.default_rng(seed)
    for fmt in (Q4_K, Q5_K, Q6_K):
        rows, cols, ntok = 5, 768, 3
        W = np.concatenate([_random_block(fmt, rng)
                            for _ in range(rows * cols // 256)])
        x = rng.standard_normal((ntok, cols)).astype(np.float32)
        y, S = o.matvec(fmt, W, rows, cols, x)
        Wf = o.dequant_rows(fmt, W, cols).astype(np.float64)
        assert Wf.shape == (rows, cols)
        ref = x.astype(np.float64) @ Wf.T
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
        assert np.allclose(S, np.abs(x.astype(np.float64)) @ np.abs(Wf).T,
                           rtol=1e-12)
        y2, _ = o.matvec(fmt, W, rows, cols, 2 * x)
        assert np.array_equal(y2, 2 * y)
        ys, Ss = o.matvec(fmt, W, rows, cols, x, row_idx=[4, 1])
        assert np.array_equal(ys, y[:, [4, 1]])
        # the rows of a matrix are consecutive runs of its blocks
        for i in range(rows):
            blk = W[i * 3 * o.block_bytes(fmt):(i + 1) * 3 * o.block_bytes(fmt)]
            row = np.concatenate([o.dequant_block(
                fmt, blk[k * o.block_bytes(fmt):(k + 1) * o.block_bytes(fmt)])
                for k in range(3)])
            assert np.array_equal(row, Wf[i].astype(np.float32))


ALL_PINS = [
    pin_matvec_2x2, pin_block_geometry, pin_byte_counts, pin_f16,
    pin_worked_scales, pin_worked_dequant, pin_scale_bijection,
    pin_q4k_single_rounding, pin_q5k, pin_q6k, pin_one_block_brute_force,
    pin_matvec_vs_numpy,
]
