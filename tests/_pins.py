"""Pins for the CPU oracle: facts fixed by the format definitions, closed
forms, library routines and brute force -- never the oracle checked against a
retyped copy of itself.

Each pin takes an ``oracle.Oracle`` and the golden codebook and raises
AssertionError on a mismatch.  ``test_oracle_pins`` runs them against the real
oracle; ``test_oracle_mutants`` runs them against deliberately broken builds
of it and requires that some pin fails for each.
"""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# Test-side block construction from named fields (the layout reading: d@0 as
# fp16, scales_h@2 as little-endian u16 holding the 2 high bits of ls_j at bits
# 2j..2j+1, scales_l@4 holding the 4 low bits of ls_j in the low nibble of byte
# j/2 for even j and the high nibble for odd j, qs@8).
# ---------------------------------------------------------------------------
def make_block(d: float, ls, qs) -> np.ndarray:
    b = np.zeros(136, np.uint8)
    b[0:2] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    sh = 0
    for j, v in enumerate(ls):
        sh |= ((int(v) >> 4) & 3) << (2 * j)
    b[2] = sh & 0xFF
    b[3] = sh >> 8
    for j, v in enumerate(ls):
        b[4 + j // 2] |= (int(v) & 0xF) << (4 * (j % 2))
    b[8:] = np.asarray(qs, np.uint8)
    return b


def parse_q8_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "q8_1_closed_forms.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
                cases.append(cur)
            elif key in ("x",):
                cur["x"] = np.array([float(v) for v in vals], np.float32)
            elif key == "q":
                cur["q"] = np.array([int(v) for v in vals], np.int8)
            else:
                cur[key] = float(vals[0])
    return cases


def f16(v) -> int:
    return int(np.float16(np.float32(v)).view(np.uint16))


# ---------------------------------------------------------------------------
# Conversions, against numpy / torch (library routines, RNE).
# ---------------------------------------------------------------------------
def pin_f16_to_f32_all_patterns(orc, kv):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float32)
    got = orc.f16_to_f32(h)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def _f32_probe_values():
    rng = np.random.default_rng(11)
    mags = np.exp2(rng.uniform(-30, 17, 4000)).astype(np.float32)
    vals = mags * np.where(rng.random(4000) < 0.5, -1, 1).astype(np.float32)
    # exact midpoints between neighbouring halves (ties), normal and subnormal
    h = rng.integers(1, 0x7BFF, 2000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    mids = ((lo + hi) / 2).astype(np.float32)
    edge = np.array([0.0, -0.0, 65504, 65519.99, 65520, 1e6, 2**-24, 2**-25, 2**-25 * 1.0001,
                     2**-14, 2**-14 - 2**-25, 6.1e-5, -3.0e-8], np.float32)
    return np.concatenate([vals, mids, -mids, edge])


def pin_f32_to_f16_matches_numpy(orc, kv):
    x = _f32_probe_values()
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = orc.f32_to_f16(x)
    assert np.array_equal(got, ref), np.flatnonzero(got != ref)[:5]


def pin_f32_to_bf16_matches_torch(orc, kv):
    import torch
    rng = np.random.default_rng(12)
    x = (np.exp2(rng.uniform(-140, 120, 4000)) * rng.choice([-1, 1], 4000)).astype(np.float32)
    # ties: bf16 value plus half a quantum
    b = rng.integers(0x0080, 0x7F00, 2000).astype(np.uint32)
    ties = ((b << 16) | 0x8000).astype(np.uint32).view(np.float32)
    x = np.concatenate([x, ties, -ties, np.array([0.0, 3.0e38, 1e-40], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.f32_to_bf16(x)
    assert np.array_equal(got, ref), np.flatnonzero(got != ref)[:5]


# ---------------------------------------------------------------------------
# IQ4_XS decode.
# ---------------------------------------------------------------------------
def pin_kvalues_golden(orc, kv):
    assert orc.kvalues() == kv


def pin_ls_bit_layout(orc, kv):
    rng = np.random.default_rng(13)
    for _ in range(50):
        ls = rng.integers(0, 64, 8)
        blk = make_block(1.0, ls, rng.integers(0, 256, 128))
        assert [orc.ls(blk, j) for j in range(8)] == [int(v) for v in ls]


def pin_ls32_is_zero(orc, kv):
    """ls = 32 everywhere: every sub-block scale d*(ls-32) is 0, so every
    decoded weight and the whole product are exactly 0, whatever d and qs."""
    rng = np.random.default_rng(14)
    blocks = [make_block(float(rng.uniform(1e-3, 4)), [32] * 8, rng.integers(0, 256, 128))
              for _ in range(8)]
    w = np.concatenate(blocks).reshape(2, 4 * 136)
    assert np.all(orc.decode(w, 2, 1024) == 0.0)
    x = rng.standard_normal((3, 1024)).astype(np.float32)
    qs, d_h, _ = orc.quantize_q8_1(x)
    assert np.all(orc.matmul(w, 2, 1024, qs, d_h) == 0.0)


def pin_nibble_positions(orc, kv):
    """Sub-block j with scale 1 (d=1, ls=33), all others scale 0; one qs byte
    set to (b<<4)|a.  Element i of the sub-block is kv[a], element 16+i is
    kv[b]; every other element of it is kv[0]; all other weights are 0."""
    for j in range(8):
        for i in (0, 5, 15):
            a, b = (3 + j + i) % 16, (11 + 2 * j + i) % 16
            if a == b:
                b = (b + 1) % 16
            qs = np.zeros(128, np.uint8)
            qs[16 * j + i] = (b << 4) | a
            ls = [32] * 8
            ls[j] = 33
            w = orc.decode(make_block(1.0, ls, qs).reshape(1, 136), 1, 256)[0]
            exp = np.zeros(256)
            exp[32 * j:32 * j + 32] = kv[0]
            exp[32 * j + i] = kv[a]
            exp[32 * j + 16 + i] = kv[b]
            assert np.array_equal(w, exp), (j, i)


def pin_scale_special_values(orc, kv):
    """d*(ls-32) for hand-checked (d, ls): 0.5*(0-32) = -16, 0.5*(63-32) = 15.5,
    2^-24*(40-32) = 2^-21 (fp16 subnormal d), 65504*(31-32) = -65504."""
    for d, ls, scale in ((0.5, 0, -16.0), (0.5, 63, 15.5), (2.0**-24, 40, 2.0**-21),
                         (65504.0, 31, -65504.0)):
        qs = np.full(128, 0x88, np.uint8)  # nibble 8 everywhere -> kv = 1
        blk = make_block(d, [ls] * 8, qs)
        assert orc.subblock_scale(blk, 3) == scale
        w = orc.decode(blk.reshape(1, 136), 1, 256)[0]
        assert np.all(w == scale * kv[8])


def pin_dequantize_bf16_consistent(orc, kv):
    """bf16 dequant = RNE of the fp32 dequant (torch's float->bfloat16)."""
    import torch
    from iq4_xs_quantized_gb300 import synth
    w = synth.iq4xs_weights(np.random.default_rng(15), 8, 512, 2e-3)
    f32, b16 = orc.dequantize(w, 8, 512, bf16=True)
    ref = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b16, ref)
    assert np.array_equal(f32.astype(np.float64), orc.decode(w, 8, 512))


# ---------------------------------------------------------------------------
# Q8_1.
# ---------------------------------------------------------------------------
def pin_q8_1_golden(orc, kv):
    for c in parse_q8_cases():
        qs, d_h, s_h = orc.quantize_q8_1(c["x"].reshape(1, 32))
        assert np.array_equal(qs[0], c["q"]), c["name"]
        assert int(d_h[0, 0]) == f16(c["d"]), c["name"]
        assert int(s_h[0, 0]) == f16(c["s"]), c["name"]


def pin_q8_1_properties(orc, kv):
    """For any finite block: |q| <= 127, the amax element maps to +-127,
    |x - d*q| <= d/2 (up to one fp32 rounding of x/d), scaling x by 2^k
    leaves q unchanged, and s = d * sum(q) rounded once to fp16."""
    rng = np.random.default_rng(16)
    x = (rng.standard_normal((4, 256)) * np.exp2(rng.integers(-6, 6, (4, 1)))).astype(np.float32)
    qs, d_h, s_h = orc.quantize_q8_1(x)
    xb = x.reshape(4, 8, 32).astype(np.float64)
    qb = qs.reshape(4, 8, 32).astype(np.float64)
    assert np.abs(qb).max() <= 127
    am = np.abs(xb).argmax(axis=2)
    assert np.all(np.abs(np.take_along_axis(qb, am[..., None], 2)) == 127)
    d = np.abs(xb).max(axis=2, keepdims=True).astype(np.float32) / np.float32(127)
    d = d.astype(np.float64)
    assert np.all(np.abs(xb - d * qb) <= d * (0.5 + 1e-6))
    qs2, d2, _ = orc.quantize_q8_1(x * np.float32(8))
    assert np.array_equal(qs2, qs)
    s_ref = (d[..., 0].astype(np.float32) * qb.sum(axis=2).astype(np.float32)).astype(np.float16)
    assert np.array_equal(s_h.reshape(4, 8), s_ref.view(np.uint16))


# ---------------------------------------------------------------------------
# Product.
# ---------------------------------------------------------------------------
def pin_matmul_hand_example(orc, kv):
    vals = {}
    with open(os.path.join(GOLDEN, "matmul_hand_example.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, *v = line.split()
                vals[k] = v
    raw = bytes.fromhex("".join(vals["block_hex"]))
    blk = np.zeros(136, np.uint8)
    blk[:len(raw)] = np.frombuffer(raw, np.uint8)
    x = np.zeros((1, 256), np.float32)
    x[0, 0] = 127
    x[0, 1:16] = 1
    x[0, 16:32] = -1
    qs, d_h, _ = orc.quantize_q8_1(x)
    y = orc.matmul(blk.reshape(1, 136), 1, 256, qs, d_h)
    assert y[0, 0] == float(vals["y"][0])


def pin_matmul_bruteforce_fp64(orc, kv):
    """Oracle product (per-sub-block integer dots, scaled) equals the plain
    fp64 dequantize-then-matmul of the same W and dequantized activations."""
    from iq4_xs_quantized_gb300 import synth
    rng = np.random.default_rng(17)
    N, K, M = 12, 768, 3
    w = synth.iq4xs_weights(rng, N, K, 2e-3)
    x = synth.activations(rng, M, K, outlier_frac=0.02)
    qs, d_h, _ = orc.quantize_q8_1(x)
    W = orc.decode(w, N, K)
    xhat = qs.astype(np.float64) * np.repeat(d_h.view(np.float16).astype(np.float64), 32, axis=1)
    ref = xhat @ W.T
    y = orc.matmul(w, N, K, qs, d_h)
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref))
    y4 = orc.matmul(w, N, K, qs, d_h, nthreads=4)
    assert np.array_equal(y, y4)


def pin_matmul_integer_exact(orc, kv):
    """d = 1 and ls = 33 make every sub-block scale 1; integer activations
    with a +-127 in every block of 32 make every Q8_1 scale 1.  Then y is the
    exact integer product of the codebook values and x (numpy int64 matmul)."""
    rng = np.random.default_rng(18)
    N, K, M = 5, 512, 4
    qs_bytes = rng.integers(0, 256, (N, K // 256, 128)).astype(np.uint8)
    w = np.stack([np.concatenate([make_block(1.0, [33] * 8, qs_bytes[n, b])
                                  for b in range(K // 256)]) for n in range(N)])
    codes = np.zeros((N, K), np.int64)
    kva = np.array(kv, np.int64)
    for n in range(N):
        for b in range(K // 256):
            for j in range(8):
                byt = qs_bytes[n, b, 16 * j:16 * j + 16]
                base = 256 * b + 32 * j
                codes[n, base:base + 16] = kva[byt & 15]
                codes[n, base + 16:base + 32] = kva[byt >> 4]
    x = rng.integers(-126, 127, (M, K)).astype(np.int64)
    x[:, ::32] = 127 * rng.choice([-1, 1], (M, K // 32))
    qs, d_h, _ = orc.quantize_q8_1(x.astype(np.float32))
    assert np.array_equal(qs.astype(np.int64), x)
    y = orc.matmul(w, N, K, qs, d_h)
    assert np.array_equal(y, (x @ codes.T).astype(np.float64))


def pin_all_zero_nibbles(orc, kv):
    """All qs = 0 decodes every weight to kv[0] = -127 times its sub-block
    scale, so y[m] = -127 * sum_j S_j * d_j * sum(q_j) (closed form)."""
    rng = np.random.default_rng(19)
    d = 0.03125
    ls = rng.integers(0, 64, 8)
    blk = make_block(d, ls, np.zeros(128, np.uint8))
    x = rng.standard_normal((2, 256)).astype(np.float32)
    qs, d_h, _ = orc.quantize_q8_1(x)
    S = np.float32(d) * (ls - 32).astype(np.float32)
    dx = d_h.view(np.float16).astype(np.float64)
    sq = qs.reshape(2, 8, 32).astype(np.int64).sum(axis=2)
    exp = -127.0 * (S.astype(np.float64)[None, :] * dx * sq).sum(axis=1)
    y = orc.matmul(blk.reshape(1, 136), 1, 256, qs, d_h)
    assert np.max(np.abs(y[:, 0] - exp)) <= 1e-12 * np.max(np.abs(exp))


def pin_single_activation(orc, kv):
    """x with one nonzero entry v at column k: its block quantizes to q=+-127,
    d = |v|/127, so y[n] = half(d) * (+-127) * w[n, k]."""
    from iq4_xs_quantized_gb300 import synth
    rng = np.random.default_rng(20)
    w = synth.iq4xs_weights(rng, 6, 512, 2e-3)
    W = orc.decode(w, 6, 512)
    for k in (0, 15, 16, 31, 200, 511):
        v = np.float32(-2.75 if k % 2 else 1.5)
        x = np.zeros((1, 512), np.float32)
        x[0, k] = v
        qs, d_h, _ = orc.quantize_q8_1(x)
        dh = float(np.float16(np.float32(abs(v)) / np.float32(127)))
        exp = dh * np.sign(v) * 127 * W[:, k]
        y = orc.matmul(w, 6, 512, qs, d_h)
        assert np.array_equal(y[0], exp), k


def pin_int32_extreme(orc, kv):
    """The largest sub-block dot: all nibbles 0 (kv -127) against q = -127
    gives P = 32*127*127 = 516128, inside int32 and inside fp32's exact range."""
    blk = make_block(1.0, [33] * 8, np.zeros(128, np.uint8))
    x = np.full((1, 256), -5.0, np.float32)
    qs, d_h, _ = orc.quantize_q8_1(x)
    assert orc.subblock_dot(blk.reshape(1, 136), 256, qs, 0, 0, 0, 3) == 516128
    y = orc.matmul(blk.reshape(1, 136), 1, 256, qs, d_h)
    dh = float(np.float16(np.float32(5.0) / np.float32(127)))
    assert y[0, 0] == 8 * 516128 * dh


# ---------------------------------------------------------------------------
# The 32-weight formats Q4_0 (value (q-8)*d) and IQ4_NL (value kv[q]*d), in
# 18-byte blocks (the layout reading: fp16 d at bytes 0-1, nibbles at 2-17;
# element i < 16 is the low nibble of byte 2+i, element 16+i the high one).
# ---------------------------------------------------------------------------
WT_Q4_0, WT_IQ4_NL = 1, 2


def make_b18(d: float, qs) -> np.ndarray:
    b = np.zeros(18, np.uint8)
    b[0:2] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    b[2:] = np.asarray(qs, np.uint8)
    return b


def _nib_value(wtype, kv, nib):
    return nib - 8 if wtype == WT_Q4_0 else kv[nib]


def pin_b18_row_bytes(orc, kv):
    assert orc.row_bytes(WT_Q4_0, 4096) == 4096 // 32 * 18
    assert orc.row_bytes(WT_IQ4_NL, 96) == 3 * 18
    assert orc.row_bytes(WT_Q4_0, 48) == -1
    assert orc.row_bytes(0, 512) == 2 * 136 and orc.row_bytes(0, 96) == -1


def pin_b18_nibble_positions(orc, kv):
    """d = 1; one qs byte (b<<4)|a at position i and a fill byte elsewhere:
    element i decodes to value(a), element 16+i to value(b), every other
    element to the fill nibble's value; Q4_0's value is q-8 (nibble 8 is 0)."""
    for wtype in (WT_Q4_0, WT_IQ4_NL):
        for i in (0, 3, 15):
            a, b = (5 + i) % 16, (12 + 3 * i) % 16
            if a == b:
                b = (b + 1) % 16
            qs = np.full(16, 0x88, np.uint8)
            qs[i] = (b << 4) | a
            blk = make_b18(1.0, qs)
            w = orc.decode_wt(wtype, blk.reshape(1, 18), 1, 32)[0]
            exp = np.full(32, float(_nib_value(wtype, kv, 8)))
            exp[i] = _nib_value(wtype, kv, a)
            exp[16 + i] = _nib_value(wtype, kv, b)
            assert np.array_equal(w, exp), (wtype, i)
            for e in range(32):
                assert orc.b18_code(wtype, blk, e) == exp[e]


def pin_q4_0_values_span_minus8_to_7(orc, kv):
    """Q4_0 nibbles 0..15 decode to -8..7 (the q-8 rule): the sixteen values
    of one block hold each nibble once in the low and once in the high half."""
    qs = (np.arange(16, dtype=np.uint8) | (np.arange(15, -1, -1, dtype=np.uint8) << 4))
    w = orc.decode_wt(WT_Q4_0, make_b18(1.0, qs).reshape(1, 18), 1, 32)[0]
    assert np.array_equal(w[:16], np.arange(-8, 8))
    assert np.array_equal(w[16:], np.arange(7, -9, -1))


def pin_b18_scale_is_d(orc, kv):
    """The block scale is float(d) itself: subnormal, largest and ordinary d."""
    for d in (2.0**-24, 65504.0, 0.375, 1e-3):
        blk = make_b18(d, np.full(16, 0x99, np.uint8))  # nibble 9: Q4_0 1, IQ4_NL 13
        assert orc.b18_scale(blk) == np.float32(np.float16(d))
        w = orc.decode_wt(WT_Q4_0, blk.reshape(1, 18), 1, 32)[0]
        assert np.all(w == float(np.float16(d)) * 1)
        w = orc.decode_wt(WT_IQ4_NL, blk.reshape(1, 18), 1, 32)[0]
        assert np.all(w == float(np.float32(np.float16(d)) * np.float32(kv[9])))


def pin_iq4nl_equals_iq4xs_with_uniform_scale(orc, kv):
    """An IQ4_XS super-block whose eight ls are all L holds the same weights
    as eight IQ4_NL blocks with d' = d*(L-32) (chosen exact in fp16) and the
    same 16 nibble bytes per sub-block: decode and product agree exactly."""
    rng = np.random.default_rng(31)
    N, K, M = 3, 512, 2
    d, L = 0.0078125, 45              # d' = 2^-7 * 13, exact in fp16
    xs_rows, nl_rows = [], []
    for _ in range(N):
        xs_blocks, nl_blocks = [], []
        for _b in range(K // 256):
            qs = rng.integers(0, 256, 128).astype(np.uint8)
            xs_blocks.append(make_block(d, [L] * 8, qs))
            nl_blocks += [make_b18(d * (L - 32), qs[16 * j:16 * j + 16]) for j in range(8)]
        xs_rows.append(np.concatenate(xs_blocks))
        nl_rows.append(np.concatenate(nl_blocks))
    w_xs, w_nl = np.stack(xs_rows), np.stack(nl_rows)
    assert np.array_equal(orc.decode_wt(WT_IQ4_NL, w_nl, N, K), orc.decode(w_xs, N, K))
    x = synth_acts(rng, M, K)
    qs_x, d_h, _ = orc.quantize_q8_1(x)
    assert np.array_equal(orc.matmul_wt(WT_IQ4_NL, w_nl, N, K, qs_x, d_h),
                          orc.matmul(w_xs, N, K, qs_x, d_h))
    assert np.array_equal(orc.matmul_wt(0, w_xs, N, K, qs_x, d_h), orc.matmul(w_xs, N, K, qs_x, d_h))


def synth_acts(rng, M, K):
    return rng.standard_normal((M, K)).astype(np.float32)


def pin_q4_0_integer_exact(orc, kv):
    """d = 1 blocks and integer activations with a +-127 in every block of 32
    (so every Q8_1 scale is 1): y is the exact integer product of the q-8
    values and x (numpy int64 matmul)."""
    rng = np.random.default_rng(32)
    N, K, M = 4, 256, 3
    nib = rng.integers(0, 16, (N, K // 32, 32))
    rows = []
    for n in range(N):
        blocks = []
        for c in range(K // 32):
            qs = (nib[n, c, :16] | (nib[n, c, 16:] << 4)).astype(np.uint8)
            blocks.append(make_b18(1.0, qs))
        rows.append(np.concatenate(blocks))
    w = np.stack(rows)
    codes = (nib.reshape(N, K) - 8).astype(np.int64)
    x = rng.integers(-126, 127, (M, K)).astype(np.int64)
    x[:, 7::32] = 127 * rng.choice([-1, 1], (M, K // 32))
    qs_x, d_h, _ = orc.quantize_q8_1(x.astype(np.float32))
    assert np.array_equal(qs_x.astype(np.int64), x)
    y = orc.matmul_wt(WT_Q4_0, w, N, K, qs_x, d_h)
    assert np.array_equal(y, (x @ codes.T).astype(np.float64))


def pin_q4_0_nibble8_is_zero(orc, kv):
    """Every nibble 8 decodes to 0 under q-8, so the product is exactly 0."""
    rng = np.random.default_rng(33)
    w = np.stack([np.concatenate([make_b18(float(rng.uniform(0.01, 2)), np.full(16, 0x88))
                                  for _ in range(8)]) for _ in range(2)])
    x = synth_acts(rng, 2, 256)
    qs_x, d_h, _ = orc.quantize_q8_1(x)
    assert np.all(orc.matmul_wt(WT_Q4_0, w, 2, 256, qs_x, d_h) == 0.0)


def pin_b18_bruteforce_fp64(orc, kv):
    """Per-block integer dots scaled in fp64 equal the plain fp64
    dequantize-then-matmul of the same W and dequantized activations; the
    fp32 dequantization is exact and its bf16 form is torch's RNE of it."""
    import torch
    from iq4_xs_quantized_gb300 import synth
    rng = np.random.default_rng(34)
    N, K, M = 9, 512, 3
    for wtype in (WT_Q4_0, WT_IQ4_NL):
        w = synth.block32_weights(rng, N, K, 2e-3)
        x = synth.activations(rng, M, K, outlier_frac=0.02)
        qs_x, d_h, _ = orc.quantize_q8_1(x)
        W = orc.decode_wt(wtype, w, N, K)
        xhat = qs_x.astype(np.float64) * np.repeat(d_h.view(np.float16).astype(np.float64), 32, 1)
        ref = xhat @ W.T
        y = orc.matmul_wt(wtype, w, N, K, qs_x, d_h)
        assert np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref))
        assert np.array_equal(y, orc.matmul_wt(wtype, w, N, K, qs_x, d_h, nthreads=3))
        f32, b16 = orc.dequantize_wt(wtype, w, N, K, bf16=True)
        assert np.array_equal(f32.astype(np.float64), W)
        ref16 = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(b16, ref16)


def pin_b18_single_activation(orc, kv):
    """x with one nonzero v at column k: y[n] = half(|v|/127) * sign(v) * 127
    * w[n, k], for both 32-weight formats."""
    from iq4_xs_quantized_gb300 import synth
    rng = np.random.default_rng(35)
    for wtype in (WT_Q4_0, WT_IQ4_NL):
        w = synth.block32_weights(rng, 5, 256, 2e-3)
        W = orc.decode_wt(wtype, w, 5, 256)
        for k in (0, 15, 16, 31, 32, 255):
            v = np.float32(-3.5 if k % 2 else 0.75)
            x = np.zeros((1, 256), np.float32)
            x[0, k] = v
            qs_x, d_h, _ = orc.quantize_q8_1(x)
            dh = float(np.float16(np.float32(abs(v)) / np.float32(127)))
            y = orc.matmul_wt(wtype, w, 5, 256, qs_x, d_h)
            assert np.array_equal(y[0], dh * np.sign(v) * 127 * W[:, k]), (wtype, k)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
